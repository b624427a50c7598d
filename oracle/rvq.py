"""Oracles of the codec quantizer lookups: the OmniVoice RVQ decode (codes ->
1024-d frame features) and the Qwen3-TTS split quantizer (codes -> the
512-channel hidden of its codec body).

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

__all__ = ["rvq_decode", "split_quantizer_decode"]


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


def split_quantizer_decode(codes: np.ndarray, codebooks: Sequence[np.ndarray], proj_semantic: np.ndarray,
                           proj_acoustic: np.ndarray) -> np.ndarray:
    """The Qwen3-TTS codec's quantizer lookup: codes -> the [B, out, T] float hidden.

    Source: "Qwen3-TTS ncnn port", Codec Decoder split, steps 1-4: the 16
    codebooks and two projection weights are read; each frame looks up one
    row per codebook; the first (semantic) codebook and the other 15
    (acoustic) codebooks are projected separately and the two projections
    are summed; the result [B, 512, T] feeds the codec body.

    Readings (the page prints neither the codebook width nor the projection
    form): each projection is a bias-free linear map [out, d] (a 1x1
    convolution), the acoustic group's rows are summed before its projection
    (the same as projecting each row and summing, by linearity), and the
    codebook width d is a parameter.

    codes [B, K, T] int; codebooks[k] [n_k, d]; proj_semantic, proj_acoustic [out, d].
    """
    codes = np.asarray(codes)
    B, K, T = codes.shape
    semantic = np.asarray(codebooks[0], np.float64)[codes[:, 0, :]]                 # (B, T, d)
    acoustic = np.zeros_like(semantic)
    for k in range(1, K):
        acoustic += np.asarray(codebooks[k], np.float64)[codes[:, k, :]]
    y = semantic @ np.asarray(proj_semantic, np.float64).T + acoustic @ np.asarray(proj_acoustic, np.float64).T
    return np.ascontiguousarray(y.transpose(0, 2, 1))                                # (B, out, T)
