"""Oracle building blocks: one Qwen3-0.6B-shaped decoder stack in float64.

Test infrastructure only (see the package docstring). Each function names
the page and section it follows.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np

__all__ = [
    "bf16_to_f64", "rms_norm", "rope_inv_freq", "rope_half_rotate",
    "mrope_interleaved", "attention_gqa", "silu", "swiglu_mlp",
    "codebook_embed_sum", "omnivoice_embed", "Backbone", "KVCache",
    "argmax_first", "causal_allowed", "keylen_allowed", "round_bf16",
]


def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (the top half of a float32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rms_norm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * gamma.

    omnivoice-cpp ARCHITECTURE.md, GGUF layout (layer_norm_rms_eps 1e-6;
    input_layernorm / post_attention_layernorm / llm.norm weights). Only eps
    is printed; the plain RMSNorm with eps inside the root and a plain gain
    is the reading taken.
    """
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * gamma


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """inv_freq_i = theta^(-2i/head_dim), i < head_dim/2 (rope_freq_base 1e6)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def rope_half_rotate(x: np.ndarray, pos: Sequence[int], theta: float) -> np.ndarray:
    """Half-rotate RoPE on x[T, H, d] at absolute positions pos[T].

    Qwen3-TTS ncnn port, mRoPE conclusion: the model uses 1-D half-rotate
    RoPE with head_dim 128 and rope_theta 1e6. Pair (i, i + d/2) is rotated
    by the angle pos * inv_freq_i.
    """
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(pos, dtype=np.float64)[:, None] * rope_inv_freq(d, theta)[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def mrope_interleaved(x: np.ndarray, pos_thw: np.ndarray, theta: float,
                      sections=(24, 20, 20)) -> np.ndarray:
    """Multimodal RoPE with interleaved sections (t, h, w) = (24, 20, 20).

    Qwen3-TTS ncnn port, mRoPE conclusion: the config carries
    mrope_section=[24,20,20], interleaved=true. Frequency index i takes its
    position from axis i % 3 while that axis still has section budget (the
    interleaved assignment), otherwise from the temporal axis. Written only
    to pin the page's claim that t == h == w makes it equal to 1-D RoPE.
    pos_thw: [T, 3] integer positions.
    """
    d = x.shape[-1]
    half = d // 2
    assert sum(sections) == half
    axis_of = np.zeros(half, dtype=np.int64)
    used = [0, 0, 0]
    for i in range(half):
        a = i % 3
        if used[a] < sections[a]:
            axis_of[i] = a
            used[a] += 1
        else:
            axis_of[i] = 0
            used[0] += 1
    p = np.asarray(pos_thw, dtype=np.float64)[:, axis_of]          # [T, half]
    ang = p * rope_inv_freq(d, theta)[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def causal_allowed(q_pos: Sequence[int], n_keys: int) -> np.ndarray:
    """allowed[i, j] = key position j <= query position q_pos[i] (keys are 0..n_keys-1)."""
    qp = np.asarray(q_pos, dtype=np.int64)[:, None]
    return np.arange(n_keys, dtype=np.int64)[None, :] <= qp


def keylen_allowed(n_q: int, n_keys: int, key_len: int) -> np.ndarray:
    """Bidirectional pass: every query sees keys j < key_len (padding excluded)."""
    return np.broadcast_to(np.arange(n_keys)[None, :] < key_len, (n_q, n_keys))


def attention_gqa(q: np.ndarray, k: np.ndarray, v: np.ndarray, allowed: np.ndarray) -> np.ndarray:
    """Scaled dot-product attention with grouped KV heads.

    q[Tq, Hq, d], k/v[Tk, Hkv, d], allowed[Tq, Tk]. Query head h reads KV head
    floor(h / (Hq/Hkv)) (GQA 2:1 in omnivoice-cpp ARCHITECTURE.md, GGUF layout
    head_count 16 / head_count_kv 8; Qwen3-TTS ncnn port, single-token SDPA:
    GQA attention done on the host). Scale 1/sqrt(d), softmax over allowed keys.
    """
    Tq, Hq, d = q.shape
    Hkv = k.shape[1]
    group = Hq // Hkv
    out = np.empty((Tq, Hq, d), dtype=np.float64)
    for h in range(Hq):
        kh = h // group
        s = (q[:, h, :] @ k[:, kh, :].T) / np.sqrt(d)
        s = np.where(allowed, s, -np.inf)
        m = np.max(s, axis=1, keepdims=True)
        p = np.exp(s - m)
        p = p / np.sum(p, axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, kh, :]
    return out


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def swiglu_mlp(y: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray) -> np.ndarray:
    """down(silu(gate(y)) * up(y)), no biases (omnivoice-cpp ARCHITECTURE.md,
    Qwen3 specifics: SwiGLU MLP, no bias on MLP)."""
    return (silu(y @ wg.T) * (y @ wu.T)) @ wd.T


def codebook_embed_sum(ids: np.ndarray, tables: List[np.ndarray]) -> np.ndarray:
    """Sum of codebook embeddings: e[t] = sum_k E_k[ids[t, k]].

    Qwen3-TTS ncnn port, model structure (Code Predictor): after a frame the
    16 token embeddings are summed to form the Talker's next codec input. An
    id of -1 means "no token from this codebook" (the Code Predictor feeds a
    single codebook per position).
    """
    ids = np.asarray(ids)
    T, K = ids.shape
    out = np.zeros((T, tables[0].shape[1]), dtype=np.float64)
    for t in range(T):
        for k in range(K):
            if ids[t, k] >= 0:
                out[t] += tables[k][ids[t, k]]
    return out


def omnivoice_embed(ids: np.ndarray, audio_mask: np.ndarray, text_table: np.ndarray,
                    audio_table: np.ndarray, audio_vocab: int = 1025) -> np.ndarray:
    """Hybrid text / audio input embedding of the OmniVoice LM.

    omnivoice-cpp ARCHITECTURE.md, Component architecture: text_emb is the
    text-table row of codebook row 0; audio_emb sums the audio-table rows
    ids * audio_mask + 1025 k over the 8 codebooks; where(audio_mask, audio,
    text). ids[B, K, S], audio_mask[B, S] -> [B, S, hidden]. The sum is
    unweighted, as the printed ``.sum(dim=1)`` states.
    """
    ids = np.asarray(ids, dtype=np.int64)
    m = np.asarray(audio_mask).astype(bool)
    B, K, S = ids.shape
    text_emb = text_table[ids[:, 0, :]]                                  # [B, S, H]
    offsets = np.arange(K, dtype=np.int64) * audio_vocab
    shifted = ids * m[:, None, :].astype(np.int64) + offsets[None, :, None]
    audio_emb = audio_table[shifted].sum(axis=1)                         # [B, S, H]
    return np.where(m[:, :, None], audio_emb, text_emb)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Values as stored in bf16: rounded to float32, then to the nearest bf16
    (ties to even on the 16 dropped bits), returned as float64."""
    u = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def argmax_first(x: np.ndarray) -> np.ndarray:
    """Greedy pick along the last axis, lowest index on ties, taken on the
    float32 logits (the precision in which the GPU decides)."""
    return np.argmax(np.asarray(x, dtype=np.float32), axis=-1).astype(np.int32)


@dataclass
class KVCache:
    """Per-layer keys (after q/k-norm and RoPE) and values, contiguous in position."""
    k: List[np.ndarray]
    v: List[np.ndarray]

    @staticmethod
    def empty(n_layers: int, n_kv: int, d: int) -> "KVCache":
        return KVCache([np.zeros((0, n_kv, d)) for _ in range(n_layers)],
                       [np.zeros((0, n_kv, d)) for _ in range(n_layers)])

    def __len__(self) -> int:
        return self.k[0].shape[0]

    def copy(self) -> "KVCache":
        return KVCache([a.copy() for a in self.k], [a.copy() for a in self.v])


class Backbone:
    """A stack of pre-norm Qwen3 decoder layers with q/k norm.

    Layer (omnivoice-cpp ARCHITECTURE.md, GGUF layout tensor list and Qwen3
    specifics): h += o_proj(attn(rope(q_norm(q)), rope(k_norm(k)), v)) with
    q, k, v projected from input_layernorm(h); h += mlp(post_attention_layernorm(h)).
    Weights are float64 copies of the bf16 tensors, PyTorch (out, in) layout.
    """

    def __init__(self, w, shape, kv_storage: Optional[str] = None):
        """kv_storage: None keeps the cache in float64 (the plain definition);
        "bf16" stores every appended key and value rounded to bf16, the cache
        format the GPU path is specified to use, so that its effect on the
        logits and the greedy picks can be measured apart from everything else."""
        self.s = shape
        self.kv_storage = kv_storage
        f = bf16_to_f64
        self.layers = [{k: f(v) for k, v in lw.items()} for lw in w.layers]
        self.codebooks = [f(t) for t in w.codebooks]
        self.text_table = f(w.text_table) if w.text_table is not None else None
        self.audio_table = f(w.audio_table) if w.audio_table is not None else None
        self.final_norm_w = f(w.final_norm)
        self.heads = [f(h) for h in w.heads]

    def new_cache(self) -> KVCache:
        return KVCache.empty(self.s.n_layers, self.s.n_kv_heads, self.s.head_dim)

    def layer(self, l: int, h: np.ndarray, pos: Sequence[int], cache: Optional[KVCache],
              allowed: np.ndarray) -> np.ndarray:
        """One decoder layer on one sequence h[T, hidden]; returns the new residual.

        With a cache, the new keys/values are appended (KV-cache append of the
        ncnn port's host attention) and attention runs over the whole cache.
        """
        return self.layer_multi(l, [h], [pos], [cache], [allowed])[0]

    def layer_multi(self, l: int, hs: List[np.ndarray], poss: List[Sequence[int]],
                    caches: List[Optional[KVCache]], alloweds: List[np.ndarray]) -> List[np.ndarray]:
        """The same layer applied to several independent sequences.

        The projections are row-wise, so they run as one matrix product over
        the rows of all sequences; norms, RoPE, the cache append and attention
        run per sequence.
        """
        s, lw = self.s, self.layers[l]
        sizes = [h.shape[0] for h in hs]
        cut = np.cumsum([0] + sizes)
        H = np.concatenate(hs, axis=0)
        N = H.shape[0]
        y = rms_norm(H, lw["in_norm"], s.rms_eps)
        q = (y @ lw["wq"].T).reshape(N, s.n_q_heads, s.head_dim)
        k = (y @ lw["wk"].T).reshape(N, s.n_kv_heads, s.head_dim)
        v = (y @ lw["wv"].T).reshape(N, s.n_kv_heads, s.head_dim)
        q = rms_norm(q, lw["q_norm"], s.rms_eps)       # per-head RMSNorm before RoPE
        k = rms_norm(k, lw["k_norm"], s.rms_eps)
        o = np.empty((N, s.n_q_heads * s.head_dim))
        for i, (pos, cache, allowed) in enumerate(zip(poss, caches, alloweds)):
            a, b = cut[i], cut[i + 1]
            qi = rope_half_rotate(q[a:b], pos, s.rope_theta)
            ki = rope_half_rotate(k[a:b], pos, s.rope_theta)
            vi = v[a:b]
            if self.kv_storage == "bf16":
                ki, vi = round_bf16(ki), round_bf16(vi)
            if cache is not None:
                cache.k[l] = np.concatenate([cache.k[l], ki], axis=0)
                cache.v[l] = np.concatenate([cache.v[l], vi], axis=0)
                K, V = cache.k[l], cache.v[l]
            else:
                K, V = ki, vi
            o[a:b] = attention_gqa(qi, K, V, allowed).reshape(b - a, -1)
        H = H + o @ lw["wo"].T
        y2 = rms_norm(H, lw["post_norm"], s.rms_eps)
        H = H + swiglu_mlp(y2, lw["wg"], lw["wu"], lw["wd"])
        return [H[cut[i]:cut[i + 1]] for i in range(len(hs))]

    def forward_cached_multi(self, xs: List[np.ndarray], caches: List[KVCache]) -> List[np.ndarray]:
        """Causal forward of several independent sequences, each extending its own cache."""
        poss, alloweds = [], []
        for x, c in zip(xs, caches):
            L0 = len(c)
            p = np.arange(L0, L0 + x.shape[0])
            poss.append(p)
            alloweds.append(causal_allowed(p, L0 + x.shape[0]))
        hs = [np.asarray(x, dtype=np.float64) for x in xs]
        for l in range(self.s.n_layers):
            hs = self.layer_multi(l, hs, poss, caches, alloweds)
        return hs

    def forward_cached(self, x: np.ndarray, pos: Sequence[int], cache: KVCache) -> np.ndarray:
        """Causal forward of T new tokens appended after the cache (prefill or decode).

        Positions are absolute token indices; query at position p sees every
        cached or new key at position <= p. Returns the residual after the
        last layer (before the final norm).
        """
        pos = np.asarray(pos, dtype=np.int64)
        L0 = len(cache)
        assert np.array_equal(pos, np.arange(L0, L0 + x.shape[0])), "tokens must extend the cache"
        allowed = causal_allowed(pos, L0 + x.shape[0])
        h = np.asarray(x, dtype=np.float64)
        for l in range(self.s.n_layers):
            h = self.layer(l, h, pos, cache, allowed)
        return h

    def forward_bidirectional(self, x: np.ndarray, key_len: Optional[int] = None) -> np.ndarray:
        """Full non-causal pass over S positions 0..S-1, no cache (MaskGIT step).

        omnivoice-cpp ARCHITECTURE.md, MaskGIT decoder: each step is a full
        prefill with bidirectional attention; keys >= key_len (padding) are
        excluded.
        """
        S = x.shape[0]
        kl = S if key_len is None else int(key_len)
        allowed = keylen_allowed(S, S, kl)
        h = np.asarray(x, dtype=np.float64)
        pos = np.arange(S)
        for l in range(self.s.n_layers):
            h = self.layer(l, h, pos, None, allowed)
        return h

    def final_norm(self, h: np.ndarray) -> np.ndarray:
        return rms_norm(h, self.final_norm_w, self.s.rms_eps)

    def head_logits(self, h: np.ndarray, j: int = 0) -> np.ndarray:
        """logits = final_norm(h) @ W_j^T (no bias)."""
        return self.final_norm(h) @ self.heads[j].T

    def audio_logits(self, h: np.ndarray) -> np.ndarray:
        """OmniVoice audio heads: x @ audio_heads^T, viewed per codebook.

        omnivoice-cpp ARCHITECTURE.md, Component architecture: logits_flat
        (B, S, 8200) -> (B, 8, S, 1025). Reading: the 8200 features are
        codebook-major (feature k*1025 + v), so logits[b, k, s, v] =
        x[b, s] . W[k*1025 + v]. h[B, S, hidden] -> [B, 8, S, 1025].
        """
        B, S, _ = h.shape
        flat = self.final_norm(h) @ self.heads[0].T                  # [B, S, 8200]
        K, V = self.s.n_heads_out, self.s.head_rows
        return flat.reshape(B, S, K, V).transpose(0, 2, 1, 3)
