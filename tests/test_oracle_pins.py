"""Pins of the fp64 oracle against what the pages and the mathematics fix.

CPU only. Each check is written so that a plausible mistake in the oracle (a
dropped term, a wrong sign, a wrong pairing or head index, a transposed
operand) fails it; ``test_oracle_mutations.py`` plants such mistakes and
shows that these checks catch them.
"""
import math
import os

import numpy as np
import pytest

import oracle as O
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")
TINY = synth.ModelShape(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16,
                        ffn=96, codebook_rows=(48, 32, 32), n_heads_out=2, head_rows=40)


def _golden_lines(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


def _nums(s):
    return np.array([float(t) for t in s.split()], dtype=np.float64)


# ---------------------------------------------------------------- RMSNorm
def check_rmsnorm(fn=O.rms_norm):
    for ln in _golden_lines("rmsnorm_toy.txt"):
        _, rest = ln.split(" ", 1)
        x, g, eps, want = [p.strip() for p in rest.split("|")]
        got = fn(_nums(x), _nums(g), float(eps))
        if not np.allclose(got, _nums(want), rtol=1e-12, atol=1e-15):
            return False
    # constant vector c*1: every entry equals c / sqrt(c^2 + eps) * gamma
    rng = np.random.default_rng(1)
    g = rng.normal(1, 0.1, 1024)
    for c in (-2.5, 1e-4, 3.0):
        got = fn(np.full(1024, c), g, 1e-6)
        if not np.allclose(got, c / math.sqrt(c * c + 1e-6) * g, rtol=1e-13):
            return False
    return True


def test_rmsnorm_pins():
    assert check_rmsnorm()


def test_rmsnorm_scale_invariance_without_eps():
    x = np.random.default_rng(2).normal(size=(5, 64))
    g = np.random.default_rng(3).normal(size=64)
    assert np.allclose(O.rms_norm(7.3 * x, g, 0.0), O.rms_norm(x, g, 0.0), rtol=1e-13)


# ---------------------------------------------------------------- RoPE
def check_rope(fn=O.rope_half_rotate):
    for ln in _golden_lines("rope_toy.txt"):
        p, x, want = [s.strip() for s in ln.split("|")]
        got = fn(_nums(x)[None, None, :], [int(p)], 1e6)[0, 0]
        if not np.allclose(got, _nums(want), rtol=0, atol=1e-15):
            return False
    rng = np.random.default_rng(4)
    x = rng.normal(size=(6, 3, 128))
    pos = np.array([0, 1, 5, 77, 1000, 40959])
    y = fn(x, pos, 1e6)
    if not np.allclose(y[0], x[0], atol=0):                       # identity at position 0
        return False
    if not np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13):
        return False
    # independent formulation: complex multiply of x_i + j x_{i+64} by exp(j pos theta^(-i/64))
    z = x[..., :64] + 1j * x[..., 64:]
    w = np.exp(1j * pos[:, None, None] * (1e6 ** (-np.arange(64) / 64.0))[None, None, :])
    zr = z * w
    if not np.allclose(np.concatenate([zr.real, zr.imag], -1), y, rtol=1e-12, atol=1e-12):
        return False
    # <R(m) q, R(n) k> depends only on m - n
    q, k = rng.normal(size=(1, 1, 128)), rng.normal(size=(1, 1, 128))
    d1 = np.sum(fn(q, [17], 1e6) * fn(k, [5], 1e6))
    d2 = np.sum(fn(q, [112], 1e6) * fn(k, [100], 1e6))
    return bool(np.isclose(d1, d2, rtol=1e-11))


def test_rope_pins():
    assert check_rope()


def test_mrope_collapses_to_1d_when_t_h_w_equal():
    """Qwen3-TTS ncnn port, mRoPE conclusion: t == h == w makes mRoPE 1-D RoPE."""
    x = np.random.default_rng(5).normal(size=(7, 2, 128))
    pos = np.array([0, 3, 9, 64, 100, 511, 4000])
    same = np.stack([pos, pos, pos], 1)
    assert np.allclose(O.mrope_interleaved(x, same, 1e6), O.rope_half_rotate(x, pos, 1e6), atol=0)
    diff = np.stack([pos, pos + 1, pos], 1)
    assert not np.allclose(O.mrope_interleaved(x, diff, 1e6), O.rope_half_rotate(x, pos, 1e6))


# ---------------------------------------------------------------- attention
def brute_attention(q, k, v, allowed, group):
    """Scalar loops, math.exp: an independent softmax-attention."""
    Tq, Hq, d = q.shape
    out = np.zeros_like(q)
    for h in range(Hq):
        kh = h // group
        for i in range(Tq):
            sc = []
            for j in range(k.shape[0]):
                if allowed[i, j]:
                    sc.append((j, sum(q[i, h, t] * k[j, kh, t] for t in range(d)) / math.sqrt(d)))
            mx = max(s for _, s in sc)
            den = sum(math.exp(s - mx) for _, s in sc)
            for j, s in sc:
                out[i, h] += math.exp(s - mx) / den * v[j, kh]
    return out


def check_attention(fn=O.attention_gqa):
    rng = np.random.default_rng(6)
    for (Tq, Tk, Hq, Hkv, d) in [(3, 5, 4, 2, 6), (1, 9, 2, 1, 4), (4, 4, 4, 4, 3)]:
        q, k, v = (rng.normal(size=(Tq, Hq, d)), rng.normal(size=(Tk, Hkv, d)),
                   rng.normal(size=(Tk, Hkv, d)))
        allowed = O.causal_allowed(np.arange(Tk - Tq, Tk), Tk)
        if not np.allclose(fn(q, k, v, allowed), brute_attention(q, k, v, allowed, Hq // Hkv),
                           rtol=1e-12, atol=1e-12):
            return False
    # all-equal keys: output is the mean of the values
    q = rng.normal(size=(2, 2, 8))
    k = np.repeat(rng.normal(size=(1, 1, 8)), 7, axis=0)
    v = rng.normal(size=(7, 1, 8))
    o = fn(q, k, v, np.ones((2, 7), bool))
    if not np.allclose(o, v.mean(0)[None, :, :].repeat(2, 0).repeat(2, 1), rtol=1e-12):
        return False
    # a single key: output is v_0
    o = fn(q, k[:1], v[:1], np.ones((2, 1), bool))
    return bool(np.allclose(o, np.broadcast_to(v[0], o.shape), rtol=0, atol=0))


def test_attention_pins():
    assert check_attention()


def test_gqa_equals_mha_with_duplicated_kv():
    rng = np.random.default_rng(7)
    q, k, v = rng.normal(size=(5, 16, 128)), rng.normal(size=(9, 8, 128)), rng.normal(size=(9, 8, 128))
    allowed = O.causal_allowed(np.arange(4, 9), 9)
    mha = O.attention_gqa(q, np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1), allowed)
    assert np.allclose(O.attention_gqa(q, k, v, allowed), mha, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- MLP
def check_swiglu(fn=O.swiglu_mlp):
    d = {ln.split()[0]: _nums(ln.split(" ", 1)[1]) for ln in _golden_lines("swiglu_toy.txt")}
    got = fn(d["y"][None], d["gate"].reshape(3, 2), d["up"].reshape(3, 2), d["down"].reshape(2, 3))[0]
    if not np.allclose(got, d["out"], rtol=1e-14, atol=1e-15):
        return False
    rng = np.random.default_rng(8)
    wg, wu, wd = rng.normal(size=(96, 64)), rng.normal(size=(96, 64)), rng.normal(size=(64, 96))
    return bool(np.all(fn(np.zeros((3, 64)), wg, wu, wd) == 0))      # silu(0) = 0


def test_swiglu_pins():
    assert check_swiglu()


# ---------------------------------------------------------------- embeddings
def check_codebook_sum(fn=O.codebook_embed_sum):
    # integer-valued rows: table k row r = 1000 k + r in every column, so the sum is exact
    tables = [np.tile((1000.0 * k + np.arange(rows))[:, None], (1, 4)) for k, rows in enumerate((30, 20, 20))]
    ids = np.array([[3, 7, 19], [29, -1, 0], [-1, -1, 5], [0, 0, 0]], np.int32)
    want = np.array([3 + 1007 + 2019, 29 + 2000, 2005, 0 + 1000 + 2000], np.float64)
    return bool(np.array_equal(fn(ids, tables), np.tile(want[:, None], (1, 4))))


def test_codebook_sum_pins():
    assert check_codebook_sum()


def check_omnivoice_embed(fn=O.omnivoice_embed):
    """Text rows at text positions; sum_k audio[id_k + 1025 k] at audio positions."""
    V, K = 1025, 8
    text = np.stack([1e6 + np.arange(1100), -np.ones(1100)], 1)   # >= 1025 rows: row-0 audio codes index it too
    audio = np.stack([np.arange(K * V, dtype=np.float64), np.ones(K * V)], 1)
    ids = np.zeros((2, K, 5), np.int32)
    ids[:, :, :2] = np.array([[11, 42], [7, 0]])[:, None, :]          # text broadcast on every row
    rng = np.random.default_rng(9)
    ids[:, :, 2:] = rng.integers(0, V, size=(2, K, 3))
    ids[0, 3, 4] = 1024                                                # a mask id is a regular row
    mask = np.zeros((2, 5), np.uint8)
    mask[:, 2:] = 1
    out = fn(ids, mask, text, audio, V)
    for b in range(2):
        for s in range(5):
            if s < 2:
                want = [1e6 + ids[b, 0, s], -1]
            else:
                want = [sum(int(ids[b, k, s]) + V * k for k in range(K)), K]
            if not np.array_equal(out[b, s], np.array(want, np.float64)):
                return False
    return True


def test_omnivoice_embed_pins():
    assert check_omnivoice_embed()


def test_omnivoice_audio_table_shape_matches_pages():
    """8200 = 8 codebooks x 1025 entries (1024 codes + mask id 1024)."""
    assert synth.OMNIVOICE.audio_codebooks * synth.OMNIVOICE.audio_vocab == 8200
    assert synth.OMNIVOICE.n_heads_out * synth.OMNIVOICE.head_rows == 8200


# ---------------------------------------------------------------- heads
def test_argmax_ties_pick_lowest_index():
    x = np.array([[0.5, 2.0, 2.0, -1.0], [3.0, 3.0, 3.0, 3.0]])
    assert O.argmax_first(x).tolist() == [1, 0]


def test_audio_logits_layout():
    w = synth.model_weights(synth.ModelShape(n_layers=0, hidden=16, text_vocab=10, audio_codebooks=8,
                                             audio_vocab=1025, n_heads_out=8, head_rows=1025), 3)
    m = O.Backbone(w, w.shape)
    h = np.random.default_rng(10).normal(size=(2, 3, 16))
    lg = m.audio_logits(h)
    assert lg.shape == (2, 8, 3, 1025)
    y = m.final_norm(h)
    W = O.bf16_to_f64(w.heads[0])
    for (b, k, s, v) in [(0, 0, 0, 0), (1, 7, 2, 1024), (0, 3, 1, 500)]:
        assert np.isclose(lg[b, k, s, v], y[b, s] @ W[k * 1025 + v], rtol=1e-13)


# ---------------------------------------------------------------- whole stack invariants
@pytest.fixture(scope="module")
def tiny():
    w = synth.model_weights(TINY, 11)
    return O.Backbone(w, TINY)


def test_decode_equals_prefill_row(tiny):
    """Cached / recompute equivalence (rightkit-qts, Synthetic tests): decode step t
    equals row t of a full causal prefill."""
    X = np.random.default_rng(12).normal(size=(12, 64))
    full = tiny.forward_cached(X, np.arange(12), tiny.new_cache())
    cache = tiny.new_cache()
    part = tiny.forward_cached(X[:5], np.arange(5), cache)
    assert np.allclose(part, full[:5], rtol=1e-12, atol=1e-12)
    for t in range(5, 12):
        row = tiny.forward_cached(X[t:t + 1], [t], cache)[0]
        assert np.allclose(row, full[t], rtol=1e-11, atol=1e-12)


def test_bidirectional_ignores_padding(tiny):
    """Keys beyond key_len are excluded: valid rows do not see what sits in the padding."""
    rng = np.random.default_rng(13)
    X = rng.normal(size=(10, 64))
    a = tiny.forward_bidirectional(X, key_len=7)
    X2 = X.copy()
    X2[7:] = rng.normal(size=(3, 64))
    b = tiny.forward_bidirectional(X2, key_len=7)
    assert np.allclose(a[:7], b[:7], rtol=1e-13, atol=1e-13)
    # and the pass is not causal: changing the last valid token moves the first row
    X3 = X.copy()
    X3[6] += 1.0
    c = tiny.forward_bidirectional(X3, key_len=7)
    assert not np.allclose(a[0], c[0])


def test_code_predictor_teacher_forcing_replays(tiny):
    rng = np.random.default_rng(14)
    w = synth.model_weights(synth.ModelShape(
        n_layers=1, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16, ffn=96,
        codebook_rows=(40,) * 16, n_heads_out=15, head_rows=40), 15)
    m = O.Backbone(w, w.shape)
    th = rng.normal(size=64)
    codes, logits, _ = O.code_predictor_frame(m, th, 3)
    codes2, logits2, _ = O.code_predictor_frame(m, th, 3, forced=codes)
    assert np.array_equal(codes, codes2) and np.allclose(logits, logits2, atol=0)
    assert np.array_equal(codes, O.argmax_first(logits))
    # the first call is a two-token causal prefill: re-running it as prefill + decode agrees
    cache = m.new_cache()
    x0 = th[None]
    x1 = O.codebook_embed_sum(O.cp_position_ids(16, 0, 3)[None], m.codebooks)
    h0 = m.forward_cached(x0, [0], cache)
    h1 = m.forward_cached(x1, [1], cache)
    assert np.allclose(m.head_logits(h1, 0)[0], logits[0], rtol=1e-11, atol=1e-12)
    del h0


def test_talker_prefill_then_decode_matches_longer_prefill(tiny):
    rng = np.random.default_rng(16)
    ids = synth.uniform_ids(rng, TINY.codebook_rows, 9)
    h_all, _, _ = O.talker_prefill(tiny, ids, tiny.new_cache())
    cache = tiny.new_cache()
    O.talker_prefill(tiny, ids[:6], cache)
    hid, _, _, _ = O.talker_decode_steps(tiny, cache, int(ids[6, 0]), ids[6:, 1:],
                                         forced_id0=ids[6:, 0])
    assert np.allclose(hid, h_all[6:], rtol=1e-11, atol=1e-12)


def test_batched_code_predictor_frames_match_single_frames():
    w = synth.model_weights(synth.ModelShape(
        n_layers=1, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16, ffn=96,
        codebook_rows=(40,) * 16, n_heads_out=15, head_rows=40), 17)
    m = O.Backbone(w, w.shape)
    rng = np.random.default_rng(17)
    th = rng.normal(size=(3, 64))
    c0 = np.array([1, 39, 7])
    codes, logits = O.code_predictor_frames(m, th, c0)
    for f in range(3):
        c1, l1, _ = O.code_predictor_frame(m, th[f], int(c0[f]))
        assert np.array_equal(codes[f], c1)
        assert np.allclose(logits[f], l1, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- Talker -> Code Predictor frame loop
def _frame_models(seed):
    t_shape = synth.ModelShape(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16, ffn=96,
                               codebook_rows=(48,) + (32,) * 15, n_heads_out=1, head_rows=48)
    c_shape = synth.ModelShape(n_layers=1, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16, ffn=96,
                               codebook_rows=(48,) + (32,) * 15, n_heads_out=15, head_rows=32)
    wt = synth.model_weights(t_shape, seed)
    wc = synth.model_weights(c_shape, seed + 1)
    wc.codebooks = wt.codebooks  # the Code Predictor's embeddings are the Talker's tables
    return O.Backbone(wt, t_shape), O.Backbone(wc, c_shape)


def test_frame_loop_composes_the_independent_drivers():
    """The frame loop feeds the Talker exactly [code0, codes 1..15] of the previous
    frame at the next position (checked against the Talker decode driver), and hands
    the Code Predictor the final-normed hidden with fresh state each frame (checked
    against the single-frame Code Predictor driver); teacher forcing with its own
    codes replays it; the cache grows by one position per frame."""
    talker, cp = _frame_models(21)
    rng = np.random.default_rng(21)
    ids = synth.uniform_ids(rng, (48,) + (32,) * 15, 5)
    cache = talker.new_cache()
    O.talker_prefill(talker, ids[:4], cache)
    codes, t_lg, c_lg, handed = O.talker_cp_frames(talker, cp, cache, ids[4], 3)
    assert len(cache) == 4 + 3
    # Talker side: the decode driver fed with the same id rows
    cache2 = talker.new_cache()
    O.talker_prefill(talker, ids[:4], cache2)
    rows = np.stack([ids[4], codes[0], codes[1]])
    hid, lg2, _, fed = O.talker_decode_steps(talker, cache2, int(rows[0, 0]), rows[:, 1:], forced_id0=rows[:, 0])
    assert np.array_equal(fed, rows)
    assert np.allclose(lg2, t_lg, rtol=1e-11, atol=1e-12)
    assert np.array_equal(codes[:, 0], O.argmax_first(t_lg))
    # Code Predictor side: fresh frame from the normed hidden and code 0
    for f in range(3):
        assert np.allclose(handed[f], talker.final_norm(hid[f:f + 1])[0], rtol=1e-12, atol=1e-12)
        c1, l1, _ = O.code_predictor_frame(cp, talker.final_norm(hid[f:f + 1])[0], int(codes[f, 0]))
        assert np.array_equal(codes[f, 1:], c1)
        assert np.allclose(c_lg[f], l1, rtol=1e-11, atol=1e-12)
        # the un-normed hidden (a plausible slip) gives another frame
        _, l_raw, _ = O.code_predictor_frame(cp, hid[f], int(codes[f, 0]))
        assert not np.allclose(l_raw, l1, rtol=1e-6, atol=1e-6)
    # teacher forcing with its own codes replays the free run
    cache3 = talker.new_cache()
    O.talker_prefill(talker, ids[:4], cache3)
    codes3, t3, c3, _ = O.talker_cp_frames(talker, cp, cache3, ids[4], 3, forced=codes)
    assert np.array_equal(codes3, codes) and np.allclose(t3, t_lg, atol=0) and np.allclose(c3, c_lg, atol=0)
