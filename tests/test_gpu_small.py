"""GPU parity on small shapes: every kernel of the path through the C ABI,
compared element by element with the fp64 oracle on the same seeded inputs.

Shapes keep the real widths (hidden 1024, 16/8 heads of 128, SwiGLU 3072) with
few layers, so the oracle finishes in seconds while the kernels still span
several tiles and ragged tails.
"""
import numpy as np
import pytest

import oracle as O
import synth
from tests.gpu_util import (HIDDEN_TOL, LOGIT_TOL, Engine, bf16_tensor_bits, check_logits_and_argmax,
                            dev_bf16_bits, dev_i32, dev_u8, f32_zeros, i32_full, rel_err_rows)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _i32(x):
    return np.asarray(x, dtype=np.int32)


def small_talker(n_layers=2):
    return synth.ModelShape(n_layers=n_layers, codebook_rows=(3072,) + (2048,) * 15, n_heads_out=1, head_rows=3072)


# ---------------------------------------------------------------- a1: gather-sum, bit-exact
def integer_tables(shape, seed):
    """Tables whose rows hold small integers: every sum of 16 rows is exact in fp32."""
    r = synth.rng_for(seed, "int_tables")
    tabs = []
    for rows in shape.codebook_rows:
        vals = r.integers(-8, 9, size=(rows, shape.hidden)).astype(np.float32)
        tabs.append(synth.bf16_bits(vals))
    return tabs


def test_gather_sum_bit_exact():
    shape = synth.ModelShape(n_layers=0, codebook_rows=(3072,) + (2048,) * 15, n_heads_out=1, head_rows=3072)
    w = synth.model_weights(shape, 21, tables=integer_tables(shape, 21))
    r = synth.rng_for(21, "ids")
    B = 7
    ids = synth.uniform_ids(r, shape.codebook_rows, B)
    ids[1, 3] = -1
    ids[2, :] = -1
    ids[2, 15] = 2047
    ids[3, 0] = 3071
    emb = synth.bf16_bits(r.integers(-4, 5, size=(B, 1024)).astype(np.float32))
    want = O.codebook_embed_sum(ids, [O.bf16_to_f64(t) for t in w.codebooks])
    want_e = want + O.bf16_to_f64(emb)
    with Engine(w, max_slots=8, max_ctx=64, max_batch=8) as e:
        hid = f32_zeros(B, 1024)
        m = e.m
        m.tts_bb_decode_step(e.h, B, np.arange(B), np.zeros(B), dev_i32(ids), hidden_out=hid)
        assert np.array_equal(hid.cpu().numpy().astype(np.float64), want)
        hid2 = f32_zeros(B, 1024)
        m.tts_bb_decode_step(e.h, B, np.arange(B), np.ones(B), dev_i32(ids), embeds=dev_bf16_bits(emb), hidden_out=hid2)
        assert np.array_equal(hid2.cpu().numpy().astype(np.float64), want_e)
        # an out-of-table id is skipped and reported
        bad = ids.copy()
        bad[4, 5] = 2048
        hid3 = f32_zeros(B, 1024)
        st = m.tts_bb_decode_step(e.h, B, np.arange(B), np.full(B, 2), dev_i32(bad), hidden_out=hid3, check=False)
        assert st == m.E_BAD_ID
        skip = bad.copy()
        skip[4, 5] = -1
        assert np.array_equal(hid3.cpu().numpy().astype(np.float64),
                              O.codebook_embed_sum(skip, [O.bf16_to_f64(t) for t in w.codebooks]))


# ---------------------------------------------------------------- head + argmax
def test_head_argmax_ties_lowest_index():
    """Rows of the head that are exact copies tie exactly; the lowest index wins."""
    shape = synth.ModelShape(n_layers=0, codebook_rows=(64,), n_heads_out=1, head_rows=3072)
    w = synth.model_weights(shape, 22, unit_gains=True)
    head = w.heads[0].copy()
    head[2000] = head[17]
    head[2999] = head[17]
    w.heads[0] = head
    tab = w.codebooks[0].copy()
    tab[0] = head[17]          # the input points along head row 17: it is the maximum, tied with 2000 and 2999
    tab[1] = head[100]
    w.codebooks = [tab]
    m0 = O.Backbone(w, shape)
    ids = np.array([[0], [1], [5]], np.int32)
    B = len(ids)
    with Engine(w, max_slots=4, max_ctx=64, max_batch=4) as e:
        logits = f32_zeros(B, 3072)
        am = i32_full(B)
        e.m.tts_bb_decode_step(e.h, B, np.arange(B), np.zeros(B), dev_i32(ids), 0, logits, am)
        g = logits.cpu().numpy()
        gam = am.cpu().numpy()
        o = m0.head_logits(O.codebook_embed_sum(ids, m0.codebooks), 0)
        check_logits_and_argmax(g, o, gam, O.argmax_first(o), min_agree=1.0)
        assert g[0, 17] == g[0, 2000] == g[0, 2999]
        assert gam[0] == 17 and gam[1] == 100


# ---------------------------------------------------------------- KV cache: bit-exact paging
def test_kv_write_read_roundtrip_across_shuffled_blocks():
    shape = small_talker(2)
    w = synth.model_weights(shape, 23)
    with Engine(w, max_slots=3, max_ctx=300, max_batch=3) as e:
        m = e.m
        lens = [130, 64, 257]
        data = {}
        # interleave writes so the physical blocks of each slot are scattered
        for chunk in range(5):
            for s in range(3):
                a, b = chunk * 64, min(lens[s], (chunk + 1) * 64)
                if a >= b:
                    continue
                for layer in (0, 1):
                    k = synth.kv_values(23, f"k{s}.{layer}.{chunk}", b - a)
                    v = synth.kv_values(23, f"v{s}.{layer}.{chunk}", b - a)
                    m.tts_bb_debug_kv_write(e.h, layer, s, a, b - a, dev_bf16_bits(k), dev_bf16_bits(v))
                    data[(s, layer, chunk)] = (k, v)
        for s in range(3):
            assert m.tts_bb_slot_len(e.h, s) == lens[s]
            for layer in (0, 1):
                kk = torch.zeros(lens[s], 8, 128, dtype=torch.bfloat16, device="cuda")
                vv = torch.zeros_like(kk)
                m.tts_bb_debug_kv_read(e.h, layer, s, 0, lens[s], kk, vv)
                want_k = np.concatenate([data[(s, layer, c)][0] for c in range(5) if (s, layer, c) in data])
                want_v = np.concatenate([data[(s, layer, c)][1] for c in range(5) if (s, layer, c) in data])
                assert np.array_equal(bf16_tensor_bits(kk), want_k)
                assert np.array_equal(bf16_tensor_bits(vv), want_v)
        # truncate + release hand blocks back; a read past the end is rejected
        m.tts_bb_truncate(e.h, 2, 100)
        assert m.tts_bb_slot_len(e.h, 2) == 100
        assert m.tts_bb_debug_kv_read(e.h, 0, 2, 90, 20, kk, vv, check=False) == m.E_INVALID
        m.tts_bb_release(e.h, 0)
        assert m.tts_bb_slot_len(e.h, 0) == 0


# ---------------------------------------------------------------- one layer: prefill 64 + 16 decodes
def test_one_layer_prefill_then_decode():
    shape = synth.ONE_LAYER
    w = synth.model_weights(shape, 0)
    X = synth.normal_bf16(synth.rng_for(0, "X"), (80, 1024), 1.0)
    m0 = O.Backbone(w, shape)
    hp, hd = O.one_layer_run(m0, O.bf16_to_f64(X), 64)
    cache = m0.new_cache()
    m0.forward_cached(O.bf16_to_f64(X), np.arange(80), cache)
    with Engine(w, max_slots=1, max_ctx=80, max_batch=1, max_tokens=64) as e:
        m = e.m
        Xd = dev_bf16_bits(X)
        hid = f32_zeros(64, 1024)
        m.tts_bb_prefill(e.h, 1, 64, [0], [64], None, embeds=Xd[:64], hidden_out=hid)
        assert rel_err_rows(hid.cpu().numpy(), hp) <= HIDDEN_TOL
        got = []
        for t in range(64, 80):
            h1 = f32_zeros(1, 1024)
            m.tts_bb_decode_step(e.h, 1, [0], [t], None, embeds=Xd[t:t + 1], hidden_out=h1)
            got.append(h1.cpu().numpy()[0])
        err = rel_err_rows(np.array(got), hd)
        assert err <= HIDDEN_TOL, err
        # the cache holds k (after q/k norm + RoPE) and v of all 80 positions
        kk = torch.zeros(80, 8, 128, dtype=torch.bfloat16, device="cuda")
        vv = torch.zeros_like(kk)
        m.tts_bb_debug_kv_read(e.h, 0, 0, 0, 80, kk, vv)
        kg = kk.float().cpu().numpy()
        vg = vv.float().cpu().numpy()
        assert rel_err_rows(kg.reshape(80, -1), cache.k[0].reshape(80, -1)) <= HIDDEN_TOL
        assert rel_err_rows(vg.reshape(80, -1), cache.v[0].reshape(80, -1)) <= HIDDEN_TOL


# ---------------------------------------------------------------- Talker-shaped, teacher forced
def test_talker_two_layers_teacher_forced():
    shape = small_talker(2)
    w = synth.model_weights(shape, 24)
    m0 = O.Backbone(w, shape)
    P, N = 16, 24
    ids = synth.talker_prefill_ids(24, P)
    rest = synth.uniform_ids(synth.rng_for(24, "rest"), shape.codebook_rows[1:], N)
    cache = m0.new_cache()
    hp, lg0, a0 = O.talker_prefill(m0, ids, cache)
    hid_o, lg_o, am_o, fed = O.talker_decode_steps(m0, cache, a0, rest)
    with Engine(w, max_slots=2, max_ctx=64, max_batch=2, max_tokens=64) as e:
        m = e.m
        logits = f32_zeros(1, 3072)
        am = i32_full(1)
        hid = f32_zeros(P, 1024)
        m.tts_bb_prefill(e.h, 1, P, [1], [P], dev_i32(ids.reshape(1, P, 16)), 0, logits, am, hidden_out=hid)
        assert rel_err_rows(hid.cpu().numpy(), hp) <= HIDDEN_TOL
        check_logits_and_argmax(logits.cpu().numpy(), lg0[None], am.cpu().numpy(), [a0], min_agree=1.0)
        gl, ga, gh = [], [], []
        for t in range(N):
            h1 = f32_zeros(1, 1024)
            m.tts_bb_decode_step(e.h, 1, [1], [P + t], dev_i32(fed[t:t + 1]), 0, logits, am, hidden_out=h1)
            gl.append(logits.cpu().numpy()[0]); ga.append(int(am.cpu().numpy()[0])); gh.append(h1.cpu().numpy()[0])
        assert rel_err_rows(np.array(gh), hid_o) <= HIDDEN_TOL
        check_logits_and_argmax(np.array(gl), lg_o, np.array(ga), am_o)


def test_decode_path_selection():
    """Decode batches of one or two run as a single persistent launch; larger
    batches take the multi-kernel path (guards against a silent fallback)."""
    shape = small_talker(2)
    w = synth.model_weights(shape, 25)
    ids = synth.talker_prefill_ids(25, 8)
    with Engine(w, max_slots=4, max_ctx=64, max_batch=4, max_tokens=64) as e:
        m = e.m
        m.tts_bb_prefill(e.h, 3, 8, [0, 1, 2], [8, 8, 8], dev_i32(np.stack([ids] * 3)))
        lens = [8, 8, 8]
        for B, want in ((1, True), (2, True), (3, False)):
            m.tts_bb_profile(e.h, True)
            m.tts_bb_decode_step(e.h, B, list(range(B)), lens[:B], dev_i32(ids[:B].copy()))
            lens[:B] = [x + 1 for x in lens[:B]]
            kinds = {k["kind"]: k["launches"] for k in m.tts_bb_profile_report(e.h)["kernels"]}
            m.tts_bb_profile(e.h, False)
            if want:
                assert kinds == {"decode_step_persistent": 1}, (B, kinds)
            else:
                assert "decode_step_persistent" not in kinds and kinds, (B, kinds)


# ---------------------------------------------------------------- ragged batches, chunked prefill, paging
def test_ragged_prefill_chunks_and_batched_decode():
    shape = small_talker(2)
    w = synth.model_weights(shape, 25)
    m0 = O.Backbone(w, shape)
    r = synth.rng_for(25, "ragged")
    B, S = 4, 70
    lens1 = [70, 1, 33, 64]
    lens2 = [5, 66, 1, 17]                       # second prefill chunk extends each cache
    ids1 = synth.uniform_ids(r, shape.codebook_rows, B * S).reshape(B, S, 16)
    ids2 = synth.uniform_ids(r, shape.codebook_rows, B * S).reshape(B, S, 16)
    slots = [3, 0, 2, 1]
    caches = [m0.new_cache() for _ in range(B)]
    hs1 = m0.forward_cached_multi([O.codebook_embed_sum(ids1[b, :lens1[b]], m0.codebooks) for b in range(B)], caches)
    hs2 = m0.forward_cached_multi([O.codebook_embed_sum(ids2[b, :lens2[b]], m0.codebooks) for b in range(B)], caches)
    n_dec = 3
    dec_ids = synth.uniform_ids(r, shape.codebook_rows, n_dec * B).reshape(n_dec, B, 16)
    dec_h, dec_l = [], []
    for t in range(n_dec):
        hs = m0.forward_cached_multi([O.codebook_embed_sum(dec_ids[t, b:b + 1], m0.codebooks) for b in range(B)], caches)
        dec_h.append(np.concatenate(hs))
        dec_l.append(m0.head_logits(np.concatenate(hs), 0))
    with Engine(w, max_slots=4, max_ctx=160, max_batch=4, max_tokens=B * S) as e:
        m = e.m
        for ids, lens, hs in ((ids1, lens1, hs1), (ids2, lens2, hs2)):
            logits = f32_zeros(B, 3072)
            am = i32_full(B)
            hid = f32_zeros(B, S, 1024)
            m.tts_bb_prefill(e.h, B, S, slots, lens, dev_i32(ids), 0, logits, am, hidden_out=hid)
            g = hid.cpu().numpy()
            for b in range(B):
                assert rel_err_rows(g[b, :lens[b]], hs[b]) <= HIDDEN_TOL
            ol = np.array([m0.head_logits(hs[b][-1:], 0)[0] for b in range(B)])
            check_logits_and_argmax(logits.cpu().numpy(), ol, am.cpu().numpy(), O.argmax_first(ol), min_agree=0.75)
        kv = [lens1[b] + lens2[b] for b in range(B)]
        for t in range(n_dec):
            logits = f32_zeros(B, 3072)
            am = i32_full(B)
            hid = f32_zeros(B, 1024)
            m.tts_bb_decode_step(e.h, B, slots, kv, dev_i32(dec_ids[t]), 0, logits, am, hidden_out=hid)
            assert rel_err_rows(hid.cpu().numpy(), dec_h[t]) <= HIDDEN_TOL
            check_logits_and_argmax(logits.cpu().numpy(), dec_l[t], am.cpu().numpy(), O.argmax_first(dec_l[t]),
                                    min_agree=0.75)
            kv = [x + 1 for x in kv]
        # a wrong kv_lens is rejected before anything runs
        assert m.tts_bb_decode_step(e.h, B, slots, [x + 1 for x in kv], dev_i32(dec_ids[0]), check=False) == m.E_INVALID


# ---------------------------------------------------------------- Code-Predictor-shaped frame
def test_code_predictor_frame_small_batch():
    shape = synth.ModelShape(n_layers=2, codebook_rows=(3072,) + (2048,) * 15, n_heads_out=15, head_rows=2048)
    w = synth.model_weights(shape, 26)
    m0 = O.Backbone(w, shape)
    F = 3
    r = synth.rng_for(26, "cp")
    th = synth.normal_bf16(r, (F, 1024), 1.0)
    code0 = r.integers(0, 3072, size=F)
    ref = [O.code_predictor_frame(m0, O.bf16_to_f64(th[f]), int(code0[f])) for f in range(F)]
    with Engine(w, max_slots=F, max_ctx=17, max_batch=F, max_tokens=2 * F) as e:
        m = e.m
        emb = np.zeros((F, 2, 1024), np.uint16)
        emb[:, 0] = th
        ids = -np.ones((F, 2, 16), np.int32)
        ids[:, 1, 0] = code0
        codes = i32_full(F * 16)
        logits = f32_zeros(F, 2048)
        codes2d = codes.view(F, 16)
        m.tts_bb_prefill(e.h, F, 2, list(range(F)), [2] * F, dev_i32(ids), 0, logits, codes2d[:, 1],
                         embeds=dev_bf16_bits(emb), argmax_stride=16)
        gl = [logits.cpu().numpy().copy()]
        for j in range(1, 15):
            step_ids = -np.ones((F, 16), np.int32)
            # teacher forcing: feed the oracle's code j
            step_ids[:, j] = [ref[f][0][j - 1] for f in range(F)]
            m.tts_bb_decode_step(e.h, F, list(range(F)), [j + 1] * F, dev_i32(step_ids), j, logits,
                                 codes2d[:, j + 1] if j < 15 else None, argmax_stride=16)
            gl.append(logits.cpu().numpy().copy())
        gl = np.array(gl)                                  # [15, F, 2048]
        got_codes = codes2d.cpu().numpy()[:, 1:16]
        for f in range(F):
            check_logits_and_argmax(gl[:, f], ref[f][1], got_codes[f], ref[f][0], min_agree=0.9)


@pytest.mark.parametrize("F", [100, 150])
def test_code_predictor_frames_over_128_tokens(F):
    """Batches above 128 tokens run the decode GEMMs as two token blocks: F = 100 gives a 200-token
    prefill (blocks of 128 + 72), F = 150 a 150-token decode (128 + 22). The GPU chains its own
    codes through the argmax outputs; the oracle replays them."""
    shape = synth.ModelShape(n_layers=2, codebook_rows=(3072,) + (2048,) * 15, n_heads_out=15, head_rows=2048)
    w = synth.model_weights(shape, 27)
    r = synth.rng_for(27, "cp_blocks")
    th = synth.normal_bf16(r, (F, 1024), 1.0)
    code0 = r.integers(0, 3072, size=F).astype(np.int32)
    with Engine(w, max_slots=F, max_ctx=17, max_batch=F, max_tokens=2 * F) as e:
        m = e.m
        emb = np.zeros((F, 2, 1024), np.uint16)
        emb[:, 0] = th
        ids = -np.ones((F, 2, 16), np.int32)
        ids[:, 1, 0] = code0
        steps = i32_full(16 * F * 16, -1).view(16, F, 16)  # call j reads steps[j]; column j carries code j
        logits = f32_zeros(F, 2048)
        m.tts_bb_prefill(e.h, F, 2, list(range(F)), [2] * F, dev_i32(ids), 0, logits, steps[1, :, 1],
                         embeds=dev_bf16_bits(emb), argmax_stride=16)
        gl = [logits.cpu().numpy().copy()]
        for j in range(1, 15):
            m.tts_bb_decode_step(e.h, F, list(range(F)), [j + 1] * F, steps[j], j, logits, steps[j + 1, :, j + 1],
                                 argmax_stride=16)
            gl.append(logits.cpu().numpy().copy())
        s = steps.cpu().numpy()
    got_codes = np.stack([s[j + 1, :, j + 1] for j in range(15)], axis=1)  # [F, 15]: codes 1..15
    gl = np.array(gl)                                                       # [15, F, 2048]
    m0 = O.Backbone(w, shape)
    o_codes, o_logits = O.code_predictor_frames(m0, O.bf16_to_f64(th), code0, forced=got_codes)
    assert np.all((got_codes >= 0) & (got_codes < 2048))
    # every row: logits within tolerance, flips only at oracle near-ties; raw agreement over all rows
    check_logits_and_argmax(gl.transpose(1, 0, 2).reshape(-1, 2048), o_logits.reshape(-1, 2048),
                            got_codes.reshape(-1), o_codes.reshape(-1))


# ---------------------------------------------------------------- MaskGIT bidirectional pass
@pytest.mark.parametrize("attn", ["tcgen05", "mma"])
@pytest.mark.parametrize("key_lens", [(200, 150), (70, 129)])
def test_maskgit_pass_small_with_padding(attn, key_lens, monkeypatch):
    """Bidirectional pass with padded sequences on both attention kernels: the
    tcgen05 one (128-key tiles: a tile with one valid key at 129, one shorter
    than a cache block at 70) and the mma.sync flash kernel."""
    if attn == "mma":
        monkeypatch.setenv("TTS_BB_BIDIR_ATTN", "mma")
    shape = synth.ModelShape(n_layers=2, text_vocab=4096, audio_codebooks=8, audio_vocab=1025, n_heads_out=8,
                             head_rows=1025)
    w = synth.model_weights(shape, 27)
    m0 = O.Backbone(w, shape)
    B, S, n_text = 2, 200, 56
    ids, mask = synth.maskgit_inputs(27, 0, B=B, S=S, n_text=n_text, text_vocab=4096)
    key_lens = np.array(key_lens, np.int32)
    lo, ho = O.maskgit_pass(m0, ids, mask, n_text, key_lens=key_lens)
    with Engine(w, max_slots=0, max_ctx=0, max_batch=B, max_tokens=B * S) as e:
        m = e.m
        logits = f32_zeros(B, 8, S - n_text, 1025)
        hid = f32_zeros(B, S, 1024)
        m.tts_bb_profile(e.h, True)
        m.tts_bb_maskgit_pass(e.h, B, S, dev_i32(ids), dev_u8(mask), key_lens, n_text, logits, hidden_out=hid)
        kinds = {k["kind"] for k in m.tts_bb_profile_report(e.h)["kernels"]}
        m.tts_bb_profile(e.h, False)
        assert ("attn_bidir_tcgen05" in kinds) == (attn == "tcgen05"), kinds
        assert ("attn_prefill" in kinds) == (attn == "mma"), kinds
        g = hid.cpu().numpy()
        gl = logits.cpu().numpy()
        for b in range(B):
            kl = int(key_lens[b])
            assert rel_err_rows(g[b, :kl], ho[b, :kl]) <= HIDDEN_TOL, b
            if kl > n_text:
                err = np.max(np.abs(gl[b][:, :kl - n_text] - lo[b][:, :kl - n_text]))
                assert err <= LOGIT_TOL, (b, err)


@pytest.mark.parametrize("B", [1, 3])
def test_decode_step_host_buffers_match_device_buffers(B):
    """tts_bb_decode_step_host (host ids in, host argmax / logits out, one synchronisation) returns
    bit for bit what tts_bb_decode_step returns on device buffers (B = 1 persistent path, B = 3 graph
    path), over a few greedy steps."""
    import codec_token_tts_gb300 as tbm
    shape = small_talker(2)
    w = synth.model_weights(shape, 81)
    ids = synth.talker_prefill_ids(81, 8)
    rows = synth.uniform_ids(synth.rng_for(81, "rows"), shape.codebook_rows, 4)
    runs = []
    for host in (False, True):
        with Engine(w, max_slots=B, max_ctx=32, max_batch=B, max_tokens=8 * B) as e:
            m = e.m
            m.tts_bb_prefill(e.h, B, 8, list(range(B)), [8] * B, dev_i32(np.stack([ids] * B)))
            got = []
            for t in range(4):
                step = np.ascontiguousarray(np.stack([rows[t]] * B).astype(np.int32))
                sl, kl = np.arange(B, dtype=np.int32), np.full(B, 8 + t, np.int32)
                if host:
                    am = np.zeros(B, np.int32)
                    lg = np.zeros((B, 3072), np.float32)
                    st = tbm.lib.tts_bb_decode_step_host(e.h, B, sl.ctypes.data, kl.ctypes.data, step.ctypes.data, 0,
                                                         am.ctypes.data, lg.ctypes.data)
                    assert st == tbm.OK
                else:
                    amd = i32_full(B)
                    lgd = f32_zeros(B, 3072)
                    m.tts_bb_decode_step(e.h, B, list(range(B)), list(kl), dev_i32(step), 0, lgd, amd)
                    am, lg = amd.cpu().numpy(), lgd.cpu().numpy()
                got.append((am.copy(), lg.copy()))
            runs.append(got)
    for (a0, l0), (a1, l1) in zip(*runs):
        assert np.array_equal(a0, a1) and np.array_equal(l0, l1)
