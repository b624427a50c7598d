"""Oracle of the codec's DAC decoder (frame features -> 24 kHz audio).

TEST INFRASTRUCTURE ONLY: see the package docstring.

Source: "omnivoice-cpp docs/ARCHITECTURE.md", Audio tokenizer pipeline
(Decode, TTS path), DAC decoder block channels, Snake activation and
ConvTranspose1d via GEMM + col2im_1d:
  features (B, T, 1024) -> transpose (B, 1024, T) -> fc2 Linear 1024 -> 256
  -> conv1 (256 -> 1024, k 7, pad 3)
  -> 5 blocks, ratios r = 8, 5, 4, 2, 3, channels 1024 -> 512 -> 256 -> 128 -> 64 -> 32:
       snake, ConvTranspose1d (IC -> OC, k 2r, stride r, padding ceil(r/2),
       output_padding r % 2), then 3 residual units with dilations 1, 3, 9:
       snake, Conv1d (OC, OC, k 7, dil d, pad 3d), snake, Conv1d (OC, OC, k 1),
       residual add
  -> snake -> conv2 (32 -> 1, k 7, pad 3) -> audio (B, 1, 960 T).
Snake: y = x + 1 / (alpha + 1e-9) * sin(alpha x)^2, alpha per channel.
ConvTranspose1d: PyTorch's definition, output length
(T - 1) s - 2 p + (K - 1) + op + 1 (= s T with these parameters).

Readings: every convolution and the Linear carry a bias (the page's col2im
path adds one when present); the printed chain ends at conv2 (no tanh).
"""
from __future__ import annotations

import math
from typing import Dict, List

import numpy as np

__all__ = ["DAC_RATIOS", "DAC_CHANNELS", "DAC_DILATIONS", "snake", "conv1d", "conv_transpose1d", "dac_decode",
           "dac_shapes"]

DAC_RATIOS = (8, 5, 4, 2, 3)
DAC_CHANNELS = (1024, 512, 256, 128, 64, 32)
DAC_DILATIONS = (1, 3, 9)


def snake(x: np.ndarray, alpha: np.ndarray) -> np.ndarray:
    """x [C, T], alpha [C]: x + 1 / (alpha + 1e-9) * sin(alpha x)^2."""
    a = np.asarray(alpha, np.float64)[:, None]
    return x + (1.0 / (a + 1e-9)) * np.sin(a * x) ** 2


def conv1d(x: np.ndarray, w: np.ndarray, b: np.ndarray, dil: int = 1, pad: int = 0) -> np.ndarray:
    """PyTorch Conv1d (stride 1): x [IC, T], w [OC, IC, K] -> y [OC, T + 2 pad - dil (K - 1)]."""
    IC, T = x.shape
    OC, _, K = w.shape
    xp = np.zeros((IC, T + 2 * pad))
    xp[:, pad:pad + T] = x
    T_out = T + 2 * pad - dil * (K - 1)
    y = np.zeros((OC, T_out)) + np.asarray(b, np.float64)[:, None]
    for k in range(K):
        y += np.asarray(w[:, :, k], np.float64) @ xp[:, k * dil:k * dil + T_out]
    return y


def conv_transpose1d(x: np.ndarray, w: np.ndarray, b: np.ndarray, stride: int, pad: int,
                     out_pad: int) -> np.ndarray:
    """PyTorch ConvTranspose1d: x [IC, T], w [IC, OC, K]. Input sample t adds
    w[:, :, k]^T x[:, t] at output position t stride + k - pad (full output
    cropped by pad on the left, length (T - 1) s - 2 p + (K - 1) + op + 1)."""
    IC, T = x.shape
    _, OC, K = w.shape
    T_out = (T - 1) * stride - 2 * pad + (K - 1) + out_pad + 1
    full = np.zeros((OC, (T - 1) * stride + K + out_pad))
    w = np.asarray(w, np.float64)
    for k in range(K):  # tap k of every input sample t lands at t * stride + k
        full[:, k:k + (T - 1) * stride + 1:stride] += w[:, :, k].T @ x
    y = full[:, pad:pad + T_out]
    return y + np.asarray(b, np.float64)[:, None]


def dac_shapes(T: int) -> List[int]:
    """Sample counts after conv1 and after each block: T, 8T, 40T, 160T, 320T, 960T."""
    out = [T]
    for r in DAC_RATIOS:
        out.append(out[-1] * r)
    return out


def dac_decode(features: np.ndarray, w: Dict) -> np.ndarray:
    """features [B, T, 1024] -> audio [B, 1, 960 T] (float64).

    w: fc2_w [256, 1024], fc2_b [256]; conv1_w [1024, 256, 7], conv1_b [1024];
    blocks[i]: alpha [IC], up_w [IC, OC, 2r], up_b [OC], res[j]: alpha1 [OC],
    w1 [OC, OC, 7], b1 [OC], alpha2 [OC], w2 [OC, OC, 1], b2 [OC];
    final_alpha [32], conv2_w [1, 32, 7], conv2_b [1].
    """
    out = []
    for b in range(features.shape[0]):
        x = np.asarray(features[b], np.float64).T                                 # (1024, T)
        x = np.asarray(w["fc2_w"], np.float64) @ x + np.asarray(w["fc2_b"], np.float64)[:, None]
        x = conv1d(x, w["conv1_w"], w["conv1_b"], 1, 3)
        for i, r in enumerate(DAC_RATIOS):
            blk = w["blocks"][i]
            x = conv_transpose1d(snake(x, blk["alpha"]), blk["up_w"], blk["up_b"], r, math.ceil(r / 2), r % 2)
            for j, d in enumerate(DAC_DILATIONS):
                ru = blk["res"][j]
                y = conv1d(snake(x, ru["alpha1"]), ru["w1"], ru["b1"], d, 3 * d)
                y = conv1d(snake(y, ru["alpha2"]), ru["w2"], ru["b2"], 1, 0)
                x = x + y
        x = conv1d(snake(x, w["final_alpha"]), w["conv2_w"], w["conv2_b"], 1, 3)
        out.append(x)
    return np.array(out)
