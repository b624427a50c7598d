"""Oracle of the RVQ codec's decode (codes -> 1024-d frame features).

TEST INFRASTRUCTURE ONLY: see the package docstring.

Source: "omnivoice-cpp docs/ARCHITECTURE.md", Audio tokenizer pipeline
(Decode, TTS path) and RVQ codec (per-codebook tensors and decode graph):
for each of the 8 codebooks k, look up the 64-d embedding row of the frame's
code, project it with project_out (1024 x 64 weight, 1024 bias) and add it
to the frame's output. The per-codebook tensors are codebook.embed
(1024, 64), project_out.weight (1024, 64) and project_out.bias (1024,).

The printed transpose to (B, 1024, T) that follows belongs to the decoder
after this step; the output here is (B, T, 1024).
"""
from __future__ import annotations

from typing import Sequence

import numpy as np

__all__ = ["rvq_decode"]


def rvq_decode(codes: np.ndarray, embed: Sequence[np.ndarray], proj_w: Sequence[np.ndarray],
               proj_b: Sequence[np.ndarray]) -> np.ndarray:
    """codes [B, K, T] int; embed[k] [n_entries, d]; proj_w[k] [out, d]; proj_b[k] [out].

    Returns out [B, T, out] = sum_k (embed[k][codes[:, k, :]] @ proj_w[k].T + proj_b[k]), float64.
    """
    codes = np.asarray(codes)
    B, K, T = codes.shape
    out_dim = np.asarray(proj_w[0]).shape[0]
    out = np.zeros((B, T, out_dim), dtype=np.float64)
    for k in range(K):
        e_k = np.asarray(embed[k], np.float64)[codes[:, k, :]]           # (B, T, d)
        p_k = e_k @ np.asarray(proj_w[k], np.float64).T + np.asarray(proj_b[k], np.float64)
        out += p_k
    return out
