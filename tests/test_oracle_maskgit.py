"""Pins of the MaskGIT greedy-update oracle (CPU only).

The update is fixed by the page's steps ("omnivoice-cpp docs/ARCHITECTURE.md",
MaskGIT decoder): CFG combine, log_softmax, mask id -inf, argmax, score =
max log-probability - codebook * penalty, already-unmasked -inf, top-k. Each
check below pins one of those steps with a closed form or a brute-force
recomputation, and the mutants at the end (plausible slips in the oracle)
show that the checks catch them.
"""
import math

import numpy as np
import pytest

import oracle as O

V, MASK = 1025, 1024


def _uniform_case(N=1, K=8, T=5, val=0.25):
    c = np.full((N, K, T, V), val, np.float32)
    return c, c.copy(), np.full((N, K, T), MASK, np.int64)


def check_update(fn=O.maskgit_update):
    # 1. all logits equal: log p = -log V for every real id, pred = 0 (lowest index),
    #    score = -log V - 5 k, so the n best cells are the first n in flat order (codebook 0 first)
    c, u, tok = _uniform_case()
    new, taken, pred, score = fn(c, u, tok, 7, MASK)
    if not np.all(pred == 0):
        return False
    want = -math.log(V) - 5.0 * np.arange(8)[:, None]
    if not np.allclose(score[0], np.broadcast_to(want, (8, 5)), rtol=0, atol=1e-12):
        return False
    flat = taken[0].reshape(-1)
    if not (flat[:7].all() and not flat[7:].any()):
        return False
    if not np.all(new[0].reshape(-1)[:7] == 0) or not np.all(new[0].reshape(-1)[7:] == MASK):
        return False
    # 2. CFG direction: c = e_0, u = 2 e_0 -> z_0 = 1 + 2 (1 - 2) = -1, the rest 0 -> pred = 1
    c = np.zeros((1, 1, 1, V), np.float32)
    u = np.zeros_like(c)
    c[..., 0], u[..., 0] = 1.0, 2.0
    _, _, pred, score = fn(c, u, np.full((1, 1, 1), MASK), 1, MASK)
    if pred[0, 0, 0] != 1:
        return False
    lse = math.log(math.exp(-1.0) + (V - 1))
    if abs(score[0, 0, 0] - (0.0 - lse)) > 1e-12:
        return False
    # 3. the mask id never wins but stays in the normaliser: z[mask] = 10, the rest 0
    c = np.zeros((1, 1, 1, V), np.float32)
    c[..., MASK] = 10.0
    _, _, pred, score = fn(c, c.copy(), np.full((1, 1, 1), MASK), 1, MASK)
    if pred[0, 0, 0] != 0 or abs(score[0, 0, 0] + math.log(math.exp(10.0) + V - 1)) > 1e-12:
        return False
    # 4. unmasked cells keep their ids and score -inf; a step takes min(n, masked) cells
    c, u, tok = _uniform_case(K=2, T=3)
    tok[0, 0, 0], tok[0, 1, 2] = 17, 99
    new, taken, _, score = fn(c, u, tok, 100, MASK)
    if new[0, 0, 0] != 17 or new[0, 1, 2] != 99 or np.isfinite(score[0, 0, 0]) or np.isfinite(score[0, 1, 2]):
        return False
    if taken.sum() != 4 or taken[0, 0, 0] or taken[0, 1, 2]:
        return False
    # 5. brute force on a small random grid: softmax by python loops, top-k by exhaustive order
    rng = np.random.default_rng(5)
    K, T = 3, 4
    c = rng.normal(0, 2, (1, K, T, V)).astype(np.float32)
    u = rng.normal(0, 2, (1, K, T, V)).astype(np.float32)
    tok = np.full((1, K, T), MASK)
    tok[0, 1, 1] = 3
    new, taken, pred, score = fn(c, u, tok, 5, MASK)
    ref = {}
    for k in range(K):
        for t in range(T):
            z = [float(np.float32(c[0, k, t, v]) + np.float32(np.float32(2.0) * np.float32(c[0, k, t, v] - u[0, k, t, v])))
                 for v in range(V)]
            m = max(z)
            lse = m + math.log(sum(math.exp(x - m) for x in z))
            best_v = max(range(V - 1), key=lambda v: (z[v], -v))
            if pred[0, k, t] != best_v:
                return False
            s = z[best_v] - lse - 5.0 * k
            if tok[0, k, t] == MASK:
                if abs(score[0, k, t] - s) > 1e-9:
                    return False
                ref[k * T + t] = s
    chosen = sorted(ref, key=lambda i: (-ref[i], i))[:5]
    if sorted(np.nonzero(taken[0].reshape(-1))[0].tolist()) != sorted(chosen):
        return False
    for i in chosen:
        if new[0].reshape(-1)[i] != pred[0].reshape(-1)[i]:
            return False
    return True


def test_update_pins():
    assert check_update()


def test_schedule_invariants():
    for n_step, n_total in ((32, 6144), (8, 100), (1, 5), (16, 8 * 350)):
        t = O.maskgit_time_steps(n_step, 0.1)
        assert t[0] == 0.0 and t[-1] == 1.0
        assert np.all(np.diff(t) > 0)
        cnt = O.maskgit_schedule(n_step, n_total, 0.1)
        assert len(cnt) == n_step and np.all(cnt >= 1)
        assert n_total <= cnt.sum() < n_total + n_step  # ceil overshoots by < 1 per step
    # shift 1 is the identity warp: uniform counts
    assert np.all(O.maskgit_schedule(8, 800, 1.0) == 100)
    # shift 0.1 unmasks few cells first and many last
    cnt = O.maskgit_schedule(32, 6144, 0.1)
    assert cnt[0] < cnt[-1]


# ---------------------------------------------------------------- planted mistakes
def _wrong_cfg_sign(c, u, tok, n, mask_id, cfg_scale=2.0, layer_penalty=5.0):
    return O.maskgit_update(c, 2 * np.asarray(c, np.float32) - np.asarray(u, np.float32), tok, n, mask_id,
                            cfg_scale, layer_penalty)  # c - s (c - u)


def _mask_before_softmax(c, u, tok, n, mask_id, cfg_scale=2.0, layer_penalty=5.0):
    c = np.array(c, np.float32, copy=True)
    u = np.array(u, np.float32, copy=True)
    c[..., mask_id] = -np.inf
    u[..., mask_id] = -np.inf
    with np.errstate(invalid="ignore"):
        return O.maskgit_update(c, u, tok, n, mask_id, cfg_scale, layer_penalty)


def _penalty_sign(c, u, tok, n, mask_id, cfg_scale=2.0, layer_penalty=5.0):
    return O.maskgit_update(c, u, tok, n, mask_id, cfg_scale, -layer_penalty)


def _ties_to_highest(c, u, tok, n, mask_id, cfg_scale=2.0, layer_penalty=5.0):
    old = O.maskgit_select

    def sel(score, n_unmask):
        flat = score.reshape(-1)
        idx = [i for i in range(flat.size) if np.isfinite(flat[i])]
        idx.sort(key=lambda i: (-flat[i], -i))
        take = np.zeros(flat.shape, bool)
        take[idx[:min(n_unmask, len(idx))]] = True
        return take.reshape(score.shape)

    O.maskgit_update.__globals__["maskgit_select"] = sel
    try:
        return O.maskgit_update(c, u, tok, n, mask_id, cfg_scale, layer_penalty)
    finally:
        O.maskgit_update.__globals__["maskgit_select"] = old


def _no_clamp(c, u, tok, n, mask_id, cfg_scale=2.0, layer_penalty=5.0):
    new, taken, pred, score = O.maskgit_update(c, u, tok, n, mask_id, cfg_scale, layer_penalty)
    for i in range(new.shape[0]):  # top-k over every cell, -inf ones included
        flat = score[i].reshape(-1)
        order = sorted(range(flat.size), key=lambda j: (-flat[j], j))[:n]
        tk = np.zeros(flat.size, bool)
        tk[order] = True
        new[i].reshape(-1)[tk] = pred[i].reshape(-1)[tk]
        taken[i] = tk.reshape(taken[i].shape)
    return new, taken, pred, score


@pytest.mark.parametrize("mutant", [_wrong_cfg_sign, _mask_before_softmax, _penalty_sign, _ties_to_highest,
                                    _no_clamp])
def test_mutants_are_caught(mutant):
    assert not check_update(mutant)
