"""Pins of the Qwen3-TTS quantizer-lookup oracle (CPU only).

"Qwen3-TTS ncnn port", Codec Decoder split: codebook 0 (semantic) goes
through one projection, codebooks 1..15 (acoustic) through the other, and the
two are summed into a [B, 512, T] hidden. Closed forms: with one-hot codebook
rows each projection picks one of its columns, so a frame's output channel o
is a known sum of projection entries; integer tables keep every value exact;
a scalar loop over (b, o, t, k, c) restates the definition on a tiny case.
Mutants (the projections swapped between the groups, codebook 0 also summed
into the acoustic group, the output left as [B, T, out], a dropped codebook)
are caught.
"""
import numpy as np
import pytest

import oracle as O

K, N, D, OUT = 16, 10, 6, 7


def _tables(seed=0):
    rng = np.random.default_rng(seed)
    books = [np.eye(N, D)[rng.permutation(N)] * (k + 1) for k in range(K)]  # row r = (k + 1) e_{perm(r)} or 0
    ps = rng.integers(-4, 5, (OUT, D)).astype(np.float64)
    pa = rng.integers(-4, 5, (OUT, D)).astype(np.float64)
    return books, ps, pa


def check_quantizer(fn=O.split_quantizer_decode):
    books, ps, pa = _tables()
    rng = np.random.default_rng(1)
    codes = rng.integers(0, N, (2, K, 5))
    got = fn(codes, books, ps, pa)
    if got.shape != (2, OUT, 5):
        return False
    for b in range(2):
        for t in range(5):
            want = np.zeros(OUT)
            for k in range(K):
                nz = np.nonzero(books[k][codes[b, k, t]])[0]
                if nz.size:  # one-hot row scaled by k + 1 picks column nz of its group's projection
                    want += (k + 1) * (ps if k == 0 else pa)[:, nz[0]]
            if not np.array_equal(got[b, :, t], want):
                return False
    # brute force: scalar loops over the definition on a small random integer case
    r2 = np.random.default_rng(2)
    bk = [r2.integers(-3, 4, (N, D)).astype(np.float64) for _ in range(K)]
    c2 = r2.integers(0, N, (1, K, 3))
    g2 = fn(c2, bk, ps, pa)
    for o in range(OUT):
        for t in range(3):
            s = 0.0
            for c in range(D):
                s += ps[o, c] * bk[0][c2[0, 0, t], c]
                for k in range(1, K):
                    s += pa[o, c] * bk[k][c2[0, k, t], c]
            if g2[0, o, t] != s:
                return False
    return True


def test_quantizer_pins():
    assert check_quantizer()


def _swapped(codes, books, ps, pa):
    return O.split_quantizer_decode(codes, books, pa, ps)


def _semantic_twice(codes, books, ps, pa):
    extra = np.asarray(books[0], np.float64)[np.asarray(codes)[:, 0, :]] @ np.asarray(pa).T
    return O.split_quantizer_decode(codes, books, ps, pa) + extra.transpose(0, 2, 1)


def _frame_major(codes, books, ps, pa):
    y = O.split_quantizer_decode(codes, books, ps, pa)
    return np.ascontiguousarray(y.transpose(0, 2, 1)).reshape(y.shape)


def _dropped_codebook(codes, books, ps, pa):
    return O.split_quantizer_decode(np.asarray(codes)[:, :-1, :], books[:-1], ps, pa)


@pytest.mark.parametrize("mutant", [_swapped, _semantic_twice, _frame_major, _dropped_codebook])
def test_quantizer_mutants_are_caught(mutant):
    assert not check_quantizer(mutant)
