"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

This module only draws random numbers and stores them as bf16 bit patterns
(``uint16`` arrays) or integer arrays. It holds none of the backbone's
arithmetic: the oracle upcasts the bit patterns to float64 itself, and the
CUDA path uploads the same bits to the device.

Distributions follow the workloads of the codec-token TTS pages:
linear and embedding weights are bf16(N(0, 0.02)); RMSNorm gains are
bf16(1 + 0.1 N(0, 1)) so that a wrong gain index shows (plain ones would
hide it); codebook ids are uniform within each table; MaskGIT masks follow
a per-row fraction uniform in [0.1, 1.0].
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

__all__ = [
    "ModelShape", "TALKER", "CODE_PREDICTOR", "OMNIVOICE", "ONE_LAYER",
    "rng_for", "bf16_bits", "normal_bf16", "gain_bf16", "model_weights",
    "uniform_ids", "talker_prefill_ids", "maskgit_inputs", "ragged_lengths",
    "kv_values", "block_permutation",
]


@dataclass(frozen=True)
class ModelShape:
    """Shape of one Qwen3-0.6B-style backbone plus its input tables and heads."""
    n_layers: int = 28
    hidden: int = 1024
    n_q_heads: int = 16
    n_kv_heads: int = 8
    head_dim: int = 128
    ffn: int = 3072
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    codebook_rows: tuple = ()          # summed input tables E_0..E_{n-1}
    text_vocab: int = 0                # OmniVoice text table rows (0 = none)
    audio_codebooks: int = 0           # OmniVoice audio table = audio_codebooks * audio_vocab rows
    audio_vocab: int = 0
    n_heads_out: int = 0               # output heads
    head_rows: int = 0                 # rows per head


# Qwen3-TTS Talker: 16 input codebook tables (E_0 has 3072 rows so the
# codebook-0 id fed back from the 3072-way head is always in range), one head.
TALKER = ModelShape(codebook_rows=(3072,) + (2048,) * 15, n_heads_out=1, head_rows=3072)
# Code Predictor: 5 layers, same tables (talker-wide embeddings), 15 heads of 2048.
CODE_PREDICTOR = ModelShape(n_layers=5, codebook_rows=(3072,) + (2048,) * 15,
                            n_heads_out=15, head_rows=2048)
# OmniVoice LM: text table + 8x1025 audio table, audio heads 8200 = 8 x 1025.
OMNIVOICE = ModelShape(text_vocab=151676, audio_codebooks=8, audio_vocab=1025,
                       n_heads_out=8, head_rows=1025)
# One decoder layer fed with embeddings directly, no head.
ONE_LAYER = ModelShape(n_layers=1)


def rng_for(seed: int, name: str) -> np.random.Generator:
    """Independent, reproducible stream per (seed, tensor name)."""
    ss = np.random.SeedSequence([int(seed) & 0xFFFFFFFF, zlib.crc32(name.encode())])
    return np.random.Generator(np.random.PCG64(ss))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); return the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return bf16_bits(x)


def gain_bf16(rng: np.random.Generator, n: int, unit: bool = False) -> np.ndarray:
    if unit:
        return bf16_bits(np.ones(n, np.float32))
    return normal_bf16(rng, (n,), std=0.1, mean=1.0)


LAYER_TENSORS = ("in_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo",
                 "post_norm", "wg", "wu", "wd")


def layer_shapes(s: ModelShape) -> Dict[str, tuple]:
    qd, kd = s.n_q_heads * s.head_dim, s.n_kv_heads * s.head_dim
    return {
        "in_norm": (s.hidden,), "wq": (qd, s.hidden), "wk": (kd, s.hidden),
        "wv": (kd, s.hidden), "q_norm": (s.head_dim,), "k_norm": (s.head_dim,),
        "wo": (s.hidden, qd), "post_norm": (s.hidden,), "wg": (s.ffn, s.hidden),
        "wu": (s.ffn, s.hidden), "wd": (s.hidden, s.ffn),
    }


@dataclass
class Weights:
    """bf16 bit patterns of every tensor (PyTorch (out, in) row-major)."""
    shape: ModelShape
    layers: List[Dict[str, np.ndarray]] = field(default_factory=list)
    codebooks: List[np.ndarray] = field(default_factory=list)
    text_table: Optional[np.ndarray] = None
    audio_table: Optional[np.ndarray] = None
    final_norm: Optional[np.ndarray] = None
    heads: List[np.ndarray] = field(default_factory=list)


def model_weights(shape: ModelShape, seed: int, unit_gains: bool = False,
                  std: float = 0.02, tables: Optional[List[np.ndarray]] = None) -> Weights:
    """All weights of one backbone; ``tables`` reuses codebook tables of another model."""
    w = Weights(shape=shape)
    shp = layer_shapes(shape)
    for l in range(shape.n_layers):
        d = {}
        for name in LAYER_TENSORS:
            r = rng_for(seed, f"layer{l}.{name}")
            if name.endswith("norm"):
                d[name] = gain_bf16(r, shp[name][0], unit_gains)
            else:
                d[name] = normal_bf16(r, shp[name], std)
        w.layers.append(d)
    if tables is not None:
        w.codebooks = list(tables)
    else:
        for k, rows in enumerate(shape.codebook_rows):
            w.codebooks.append(normal_bf16(rng_for(seed, f"codebook{k}"), (rows, shape.hidden), std))
    if shape.text_vocab:
        w.text_table = normal_bf16(rng_for(seed, "text_table"), (shape.text_vocab, shape.hidden), std)
    if shape.audio_codebooks:
        w.audio_table = normal_bf16(rng_for(seed, "audio_table"),
                                    (shape.audio_codebooks * shape.audio_vocab, shape.hidden), std)
    w.final_norm = gain_bf16(rng_for(seed, "final_norm"), shape.hidden, unit_gains)
    for j in range(shape.n_heads_out):
        rows = shape.head_rows * (shape.n_heads_out if shape.audio_codebooks else 1)
        if shape.audio_codebooks:
            # OmniVoice: one (8200, hidden) audio_heads matrix
            if j == 0:
                w.heads.append(normal_bf16(rng_for(seed, "audio_heads"), (rows, shape.hidden), std))
            continue
        w.heads.append(normal_bf16(rng_for(seed, f"head{j}"), (shape.head_rows, shape.hidden), std))
    return w


def uniform_ids(rng: np.random.Generator, rows_per_codebook, n: int) -> np.ndarray:
    """ids[n, K]: column k uniform in [0, rows_per_codebook[k])."""
    cols = [rng.integers(0, r, size=n, dtype=np.int64) for r in rows_per_codebook]
    return np.stack(cols, axis=1).astype(np.int32)


def talker_prefill_ids(seed: int, n_pos: int, rows=TALKER.codebook_rows) -> np.ndarray:
    return uniform_ids(rng_for(seed, "prefill_ids"), rows, n_pos)


def ragged_lengths(seed: int, n: int, lo: int, hi: int, name: str = "lengths") -> np.ndarray:
    """Integers uniform in [lo, hi] inclusive."""
    return rng_for(seed, name).integers(lo, hi + 1, size=n, dtype=np.int64).astype(np.int32)


def block_permutation(seed: int, n_blocks: int) -> np.ndarray:
    return rng_for(seed, "block_perm").permutation(n_blocks).astype(np.int32)


def kv_values(seed: int, name: str, n_tok: int, n_kv_heads: int = 8, head_dim: int = 128) -> np.ndarray:
    """bf16(N(0,1)) K or V rows [n_tok, n_kv_heads, head_dim] (the scale of normed keys)."""
    return normal_bf16(rng_for(seed, name), (n_tok, n_kv_heads, head_dim), 1.0)


def maskgit_inputs(seed: int, step: int, B: int = 8, S: int = 1024, n_text: int = 256,
                   text_vocab: int = 151676, n_cb: int = 8, codebook_size: int = 1024,
                   mask_id: int = 1024):
    """One MaskGIT pass input in the pages' layout.

    ids[B, 8, S] int32 with the text id broadcast on every codebook row at
    text positions s < n_text, audio codes at s >= n_text; audio_mask[B, S]
    (1 at audio positions). Per row a fraction p ~ U[0.1, 1.0] of the
    (codebook, frame) audio cells is set to ``mask_id``.
    """
    r = rng_for(seed, f"maskgit_step{step}")
    T = S - n_text
    ids = np.empty((B, n_cb, S), np.int32)
    text = r.integers(0, text_vocab, size=(B, n_text), dtype=np.int64).astype(np.int32)
    ids[:, :, :n_text] = text[:, None, :]
    codes = r.integers(0, codebook_size, size=(B, n_cb, T), dtype=np.int64).astype(np.int32)
    for b in range(B):
        p = r.uniform(0.1, 1.0)
        n_mask = int(round(p * n_cb * T))
        cells = r.permutation(n_cb * T)[:n_mask]
        flat = codes[b].reshape(-1)
        flat[cells] = mask_id
    ids[:, :, n_text:] = codes
    mask = np.zeros((B, S), np.uint8)
    mask[:, n_text:] = 1
    return ids, mask
