"""Oracle of the MaskGIT greedy update (one refinement step's token update).

TEST INFRASTRUCTURE ONLY: see the package docstring.

Source: "omnivoice-cpp docs/ARCHITECTURE.md", MaskGIT decoder. Per step, with
class and position temperatures 0 (the greedy, bit-deterministic mode):
  1. CFG combine of the conditional and unconditional logits of each target
     cell: z = c + cfg_scale * (c - u)  (cfg_scale 2.0 by default);
  2. log-probabilities: log_softmax(z) over the audio vocabulary;
  3. the mask id's log-probability is set to -inf;
  4. pred = argmax (lowest index on ties);
  5. score = max log-probability - codebook index * layer_penalty (5.0);
  6. cells already unmasked get score -inf;
  7. the schedule[step] cells with the highest score over the flattened
     [codebook][position] grid take their pred;
  8. the new tokens go to both the conditional and the unconditional rows.
The schedule comes from time steps t_0..t_n on [0, 1] with a shift of 0.1:
count_i = ceil(N_total * (t_{i+1} - t_i)).

Readings where the page leaves a step open (each also listed in the design
notes):
  * z is formed in float32, one rounding per operation (c - u, times the
    scale, plus c), so that the argmax, an integer decided by floating point,
    is taken in the same precision as the kernel's; log_softmax and the score
    are then computed in float64 from those float32 values.
  * top-k ties are broken by the lowest flat index k * T + t.
  * a step never overwrites an unmasked cell: it takes
    min(schedule[step], masked cells) cells.
  * the time steps are t_i = i / n warped by the shift s:
    t' = s t / (1 + (s - 1) t), evaluated as s t / (s t + (1 - t)) (parity
    unpinned: the page does not print the function; only its invariants are
    pinned).
"""
from __future__ import annotations

import math
from typing import Tuple

import numpy as np

__all__ = ["maskgit_time_steps", "maskgit_schedule", "maskgit_cfg_logits", "maskgit_cell_scores",
           "maskgit_select", "maskgit_update"]


def maskgit_time_steps(num_step: int, t_shift: float = 0.1) -> np.ndarray:
    """Time steps t'_0..t'_n on [0, 1], shifted (reading: t' = s t / (1 + (s - 1) t),
    evaluated as s t / (s t + (1 - t)) so that both ends are exact)."""
    t = np.arange(num_step + 1, dtype=np.float64) / num_step
    return t_shift * t / (t_shift * t + (1.0 - t))


def maskgit_schedule(num_step: int, n_total: int, t_shift: float = 0.1) -> np.ndarray:
    """Cells newly unmasked at each step: ceil(N_total * (t'_{i+1} - t'_i))."""
    t = maskgit_time_steps(num_step, t_shift)
    return np.array([math.ceil(n_total * (t[i + 1] - t[i])) for i in range(num_step)], dtype=np.int64)


def maskgit_cfg_logits(c: np.ndarray, u: np.ndarray, cfg_scale: float) -> np.ndarray:
    """Step 1 in float32, one rounding per operation: z = c + s * (c - u)."""
    c32 = np.asarray(c, dtype=np.float32)
    u32 = np.asarray(u, dtype=np.float32)
    d = (c32 - u32).astype(np.float32)
    return (c32 + (np.float32(cfg_scale) * d).astype(np.float32)).astype(np.float32)


def maskgit_cell_scores(c: np.ndarray, u: np.ndarray, tokens: np.ndarray, mask_id: int,
                        cfg_scale: float = 2.0, layer_penalty: float = 5.0) -> Tuple[np.ndarray, np.ndarray]:
    """Steps 1-6 for one item. c, u: [K, T, V] logits; tokens: [K, T] current ids.

    Returns (pred [K, T] int64, score [K, T] float64, -inf where already unmasked).
    """
    z = maskgit_cfg_logits(c, u, cfg_scale).astype(np.float64)       # [K, T, V]
    m = z.max(axis=-1, keepdims=True)
    lse = m + np.log(np.exp(z - m).sum(axis=-1, keepdims=True))
    logp = z - lse                                                      # log_softmax over V
    logp[..., mask_id] = -np.inf
    pred = np.argmax(logp, axis=-1)                                     # first maximum on ties
    best = np.take_along_axis(logp, pred[..., None], axis=-1)[..., 0]
    K = c.shape[0]
    score = best - np.arange(K, dtype=np.float64)[:, None] * layer_penalty
    score = np.where(np.asarray(tokens) == mask_id, score, -np.inf)
    return pred, score


def maskgit_select(score: np.ndarray, n_unmask: int) -> np.ndarray:
    """Step 7: boolean [K, T] of the cells taken: the min(n, masked) highest
    finite scores of the flattened grid, ties to the lowest flat index."""
    flat = score.reshape(-1)
    finite = np.isfinite(flat)
    n = min(int(n_unmask), int(finite.sum()))
    order = sorted(np.nonzero(finite)[0].tolist(), key=lambda i: (-flat[i], i))
    take = np.zeros(flat.shape, dtype=bool)
    take[order[:n]] = True
    return take.reshape(score.shape)


def maskgit_update(cond: np.ndarray, uncond: np.ndarray, tokens: np.ndarray, n_unmask: int, mask_id: int,
                   cfg_scale: float = 2.0, layer_penalty: float = 5.0):
    """One greedy update of every item.

    cond, uncond: [N, K, T, V] logits of the target window; tokens: [N, K, T].
    Returns (new tokens [N, K, T], taken [N, K, T] bool, pred [N, K, T], score [N, K, T]).
    """
    out = np.array(tokens, dtype=np.int64, copy=True)
    N = out.shape[0]
    taken = np.zeros(out.shape, dtype=bool)
    preds = np.zeros(out.shape, dtype=np.int64)
    scores = np.zeros(out.shape, dtype=np.float64)
    for i in range(N):
        pred, score = maskgit_cell_scores(cond[i], uncond[i], out[i], mask_id, cfg_scale, layer_penalty)
        take = maskgit_select(score, n_unmask)
        out[i][take] = pred[take]
        taken[i], preds[i], scores[i] = take, pred, score
    return out, taken, preds, scores
