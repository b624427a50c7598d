"""Causal prefill attention on tcgen05 and on the decode kernel (GPU), against the fp64 oracle.

A causal prefill of 64 or more positions per sequence runs its attention on
the tcgen05 flash kernel over the paged cache: query s of sequence b sits at
position start_b + s and sees every key up to its own position, the keys of
earlier chunks included. Cases: three ragged sequences prefilled in two
chunks (the second chunk attends to cached keys of the first, its positions
crossing cache blocks), and the 28-layer Talker's 128-position prompt. A
prefill of at most 8 positions per sequence runs on the decode attention
kernel with one query per token (ragged chunks of up to 8, padding tokens
included). Chunks of 257–512 tokens run their products on the split-K GEMM over three or four
token blocks when one launch fits a wave. The engine's profile must show the expected kernel, and an engine
that keeps every prefill on the mma.sync kernel must agree with it. Contexts
of at most 32 keys (the Code Predictor's) run decode attention and the short
prefill one warp per (query, KV head) in 16-key rounds.
"""
import os

import numpy as np
import pytest

import oracle as O
import synth
from tests.gpu_util import HIDDEN_TOL, Engine, dev_bf16_bits, dev_i32, f32_zeros, rel_err_rows

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SHAPE = synth.ModelShape(n_layers=2)


def _chunked_prefill(w, X, lens1, lens2, S1, S2):
    """Two prefill chunks per sequence; returns the hidden rows of both chunks and the kernel kinds run."""
    B = len(lens1)
    with Engine(w, max_slots=B, max_ctx=320, max_batch=B, max_tokens=B * max(S1, S2)) as e:
        m = e.m
        m.tts_bb_profile(e.h, True)
        outs = []
        for lens, S, off in ((lens1, S1, [0] * B), (lens2, S2, lens1)):
            emb = np.zeros((B, S, 1024), np.uint16)
            for b in range(B):
                emb[b, :lens[b]] = X[b, off[b]:off[b] + lens[b]]
            hid = f32_zeros(B * S, 1024)
            m.tts_bb_prefill(e.h, B, S, list(range(B)), lens, embeds=dev_bf16_bits(emb), hidden_out=hid)
            outs.append(hid.cpu().numpy().reshape(B, S, 1024))
        kinds = {k["kind"] for k in m.tts_bb_profile_report(e.h)["kernels"]}
        m.tts_bb_profile(e.h, False)
    return outs, kinds


def test_chunked_ragged_prefill_on_tcgen05():
    w = synth.model_weights(SHAPE, 91)
    lens1, lens2 = [100, 64, 130], [90, 70, 64]
    S1, S2 = 130, 90
    X = synth.normal_bf16(synth.rng_for(91, "prefill_tc"), (3, 220, 1024), 1.0)
    (h1, h2), kinds = _chunked_prefill(w, X, lens1, lens2, S1, S2)
    assert "attn_causal_tcgen05" in kinds, kinds
    # 390 and 270 tokens: the split-K GEMM over three or four 128-token blocks where one launch fits
    # a wave (QKV with the fused q/k norm + RoPE + append), the dense GEMM for gate/up at 390
    assert {"gemm_tcgen05_decode", "gemm_tcgen05"} <= kinds and "qk_norm_rope_append" not in kinds, kinds
    m0 = O.Backbone(w, SHAPE)
    for b in range(3):
        cache = m0.new_cache()
        n1, n2 = lens1[b], lens2[b]
        o1 = m0.forward_cached(O.bf16_to_f64(X[b, :n1]), np.arange(n1), cache)
        o2 = m0.forward_cached(O.bf16_to_f64(X[b, n1:n1 + n2]), np.arange(n1, n1 + n2), cache)
        assert rel_err_rows(h1[b, :n1], o1) <= HIDDEN_TOL
        assert rel_err_rows(h2[b, :n2], o2) <= HIDDEN_TOL
    # the same calls with the prefill attention on the mma.sync kernel
    os.environ["TTS_BB_PREFILL_ATTN"] = "mma"
    try:
        (g1, g2), kinds_mma = _chunked_prefill(w, X, lens1, lens2, S1, S2)
    finally:
        del os.environ["TTS_BB_PREFILL_ATTN"]
    assert "attn_causal_tcgen05" not in kinds_mma and "attn_prefill" in kinds_mma
    for b in range(3):
        assert rel_err_rows(h1[b, :lens1[b]], g1[b, :lens1[b]]) <= HIDDEN_TOL
        assert rel_err_rows(h2[b, :lens2[b]], g2[b, :lens2[b]]) <= HIDDEN_TOL


def test_talker_prompt_prefill_on_tcgen05():
    """The 28-layer Talker's 128-position prompt (the bench's prefill) on the tcgen05 kernel."""
    w = synth.model_weights(synth.TALKER, 1)
    ids = synth.talker_prefill_ids(1, 128)
    m0 = O.Backbone(w, synth.TALKER)
    hp, lg0, a0 = O.talker_prefill(m0, ids, m0.new_cache())
    with Engine(w, max_slots=1, max_ctx=256, max_batch=1, max_tokens=128) as e:
        m = e.m
        m.tts_bb_profile(e.h, True)
        hid = f32_zeros(128, 1024)
        m.tts_bb_prefill(e.h, 1, 128, [0], [128], dev_i32(ids.reshape(1, 128, 16)), hidden_out=hid)
        kinds = {k["kind"] for k in m.tts_bb_profile_report(e.h)["kernels"]}
        m.tts_bb_profile(e.h, False)
    assert "attn_causal_tcgen05" in kinds, kinds
    assert rel_err_rows(hid.cpu().numpy(), hp) <= HIDDEN_TOL


def test_short_ragged_prefill_on_the_decode_kernel():
    w = synth.model_weights(SHAPE, 93)
    lens1, lens2 = [5, 2, 8], [3, 8, 1]
    X = synth.normal_bf16(synth.rng_for(93, "prefill_short"), (3, 16, 1024), 1.0)
    (h1, h2), kinds = _chunked_prefill(w, X, lens1, lens2, 8, 8)
    assert "attn_decode" in kinds and "attn_prefill" not in kinds, kinds
    m0 = O.Backbone(w, SHAPE)
    for b in range(3):
        cache = m0.new_cache()
        n1, n2 = lens1[b], lens2[b]
        o1 = m0.forward_cached(O.bf16_to_f64(X[b, :n1]), np.arange(n1), cache)
        o2 = m0.forward_cached(O.bf16_to_f64(X[b, n1:n1 + n2]), np.arange(n1, n1 + n2), cache)
        assert rel_err_rows(h1[b, :n1], o1) <= HIDDEN_TOL
        assert rel_err_rows(h2[b, :n2], o2) <= HIDDEN_TOL
    os.environ["TTS_BB_PREFILL_ATTN"] = "mma"
    try:
        (g1, g2), kinds_mma = _chunked_prefill(w, X, lens1, lens2, 8, 8)
    finally:
        del os.environ["TTS_BB_PREFILL_ATTN"]
    assert "attn_prefill" in kinds_mma and "attn_decode" not in kinds_mma
    for b in range(3):
        assert rel_err_rows(h1[b, :lens1[b]], g1[b, :lens1[b]]) <= HIDDEN_TOL
        assert rel_err_rows(h2[b, :lens2[b]], g2[b, :lens2[b]]) <= HIDDEN_TOL


def test_short_context_attention_one_warp_per_head():
    """12 sequences, ragged 1..8-token prefills, then decode steps up to 32 keys (max_ctx 32)."""
    w = synth.model_weights(SHAPE, 95)
    B, S, CTX = 12, 8, 32
    r = synth.rng_for(95, "short_ctx")
    lens = [int(x) for x in r.integers(1, S + 1, B)]
    n_dec = CTX - max(lens)
    X = synth.normal_bf16(r, (B, S, 1024), 1.0)
    D = synth.normal_bf16(r, (n_dec, B, 1024), 1.0)
    emb = np.zeros((B, S, 1024), np.uint16)
    for b in range(B):
        emb[b, :lens[b]] = X[b, :lens[b]]
    with Engine(w, max_slots=B, max_ctx=CTX, max_batch=B, max_tokens=B * S) as e:
        m = e.m
        m.tts_bb_profile(e.h, True)
        hid = f32_zeros(B * S, 1024)
        m.tts_bb_prefill(e.h, B, S, list(range(B)), lens, embeds=dev_bf16_bits(emb), hidden_out=hid)
        hp = hid.cpu().numpy().reshape(B, S, 1024)
        kv, hd = list(lens), []
        for t in range(n_dec):
            ho = f32_zeros(B, 1024)
            m.tts_bb_decode_step(e.h, B, list(range(B)), kv, None, embeds=dev_bf16_bits(D[t]), hidden_out=ho)
            hd.append(ho.cpu().numpy())
            kv = [x + 1 for x in kv]
        kinds = {k["kind"] for k in m.tts_bb_profile_report(e.h)["kernels"]}
        m.tts_bb_profile(e.h, False)
    assert "attn_decode_short" in kinds and "attn_decode" not in kinds, kinds
    m0 = O.Backbone(w, SHAPE)
    for b in range(B):
        cache = m0.new_cache()
        n = lens[b]
        o1 = m0.forward_cached(O.bf16_to_f64(X[b, :n]), np.arange(n), cache)
        assert rel_err_rows(hp[b, :n], o1) <= HIDDEN_TOL
        od = np.stack([m0.forward_cached(O.bf16_to_f64(D[t, b:b + 1]), [n + t], cache)[0] for t in range(n_dec)])
        assert rel_err_rows(np.stack([x[b] for x in hd]), od) <= HIDDEN_TOL
