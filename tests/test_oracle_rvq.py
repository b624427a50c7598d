"""Pins of the RVQ-decode oracle (CPU only).

Closed forms from the decode graph ("omnivoice-cpp docs/ARCHITECTURE.md",
RVQ codec): with one-hot embedding rows the projection picks one column of
project_out, so each frame's output is a sum of known columns plus the
biases; a codebook whose table is zero contributes its bias alone; small
integer tables make every value exact. Mutants (a transposed projection, a
dropped bias, the codebook index taken from the wrong axis, a missing
codebook) are caught.
"""
import numpy as np
import pytest

import oracle as O


def _tables(K=3, n=6, d=4, out=5, seed=0):
    rng = np.random.default_rng(seed)
    embed = [np.eye(n, d)[rng.permutation(n)] * (k + 1) for k in range(K)]  # row r = (k+1) e_{perm}
    w = [rng.integers(-4, 5, (out, d)).astype(np.float64) for _ in range(K)]
    b = [rng.integers(-3, 4, out).astype(np.float64) for _ in range(K)]
    return embed, w, b


def check_rvq(fn=O.rvq_decode):
    K, n, d, out = 3, 6, 4, 5
    embed, w, b = _tables(K, n, d, out)
    rng = np.random.default_rng(1)
    codes = rng.integers(0, n, (2, K, 7))
    got = fn(codes, embed, w, b)
    if got.shape != (2, 7, out):
        return False
    for bi in range(2):
        for t in range(7):
            want = np.zeros(out)
            for k in range(K):
                row = embed[k][codes[bi, k, t]]
                nz = np.nonzero(row)[0]
                want += b[k]
                if nz.size:  # one-hot row scaled by k + 1: the projection picks column nz of project_out
                    want += (k + 1) * w[k][:, nz[0]]
            if not np.array_equal(got[bi, t], want):
                return False
    # a zero table leaves the bias alone
    z = [np.zeros_like(e) for e in embed]
    if not np.array_equal(fn(codes, z, w, b)[0, 0], sum(b)):
        return False
    return True


def test_rvq_pins():
    assert check_rvq()


def _transposed(codes, embed, w, b):
    return O.rvq_decode(codes, embed, [np.asarray(x).T.reshape(np.asarray(x).shape) for x in w], b)


def _no_bias(codes, embed, w, b):
    return O.rvq_decode(codes, embed, w, [np.zeros_like(x) for x in b])


def _wrong_axis(codes, embed, w, b):
    return O.rvq_decode(np.ascontiguousarray(np.asarray(codes)[:, ::-1, :]), embed, w, b)


def _missing_codebook(codes, embed, w, b):
    return O.rvq_decode(np.asarray(codes)[:, :-1, :], embed[:-1], w[:-1], b[:-1])


@pytest.mark.parametrize("mutant", [_transposed, _no_bias, _wrong_axis, _missing_codebook])
def test_rvq_mutants_are_caught(mutant):
    assert not check_rvq(mutant)
