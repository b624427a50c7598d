"""The decode-attention entry point that allocates nothing.

Callers that may not call cudaMalloc (a plug-in whose host framework owns all
device memory, a real-time audio thread that must not block in the
allocator) use tts_bb_gqa_decode_attention_static: their own q, KV pool, page
table and output, with the split partials in the library's fixed device
array. These tests call it through the C ABI, twice in a row each time, and
check it

  * against the attention that tts_bb_decode_step computes with the engine's
    own scratch (the existing entry point), and against the fp64 oracle on
    the K/V read back from the engine's cache;
  * on a caller-built pool against the oracle with one split (every query
    within the first 64-token block: the split kernel writes the output) and
    with 64 sequences of up to 512 positions (8 splits, the whole array);
  * with positions outside 0..max_position, which are clamped on the device,
    so the call stays inside the caller's page-table rows.

The engine's attention output is made observable with a one-layer model whose
MLP weights are zero and whose o_proj selects half of the 2048 attention
outputs (identity on 1024 of them), so hidden_out - input = that half.
"""
import numpy as np
import pytest

import oracle as O
import synth
from tests.gpu_util import HIDDEN_TOL, Engine, dev_bf16_bits, rel_err_rows, tb

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ONE = 0x3F80  # bf16 1.0


def selector_weights(half):
    w = synth.model_weights(synth.ONE_LAYER, 31)
    lw = w.layers[0]
    for k in ("wg", "wu", "wd"):
        lw[k] = np.zeros_like(lw[k])
    wo = np.zeros_like(lw["wo"])
    wo[np.arange(1024), np.arange(1024) + 1024 * half] = ONE
    lw["wo"] = wo
    return w


def oracle_attention(q_bits, K, V, positions):
    """q_bits [B][16][128] bf16 bits; K/V lists of [n_b][8][128] float64 -> [B][2048]."""
    q = O.bf16_to_f64(q_bits).reshape(len(K), 16, 128)
    out = np.zeros((len(K), 2048))
    for b, p in enumerate(positions):
        allowed = np.ones((1, p + 1), dtype=bool)
        out[b] = O.attention_gqa(q[b][None], K[b][:p + 1], V[b][:p + 1], allowed).reshape(-1)
    return out


def call_static(q_d, pool, table, bps, pos_list, max_position, B, n_calls=2):
    m = tb()
    st = torch.cuda.current_stream().cuda_stream
    pos = torch.tensor(pos_list, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(n_calls):                                    # calls in a row share the scratch
        out = torch.full((B, 16, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert m.tts_bb_gqa_decode_attention_static(q_d, pool, table, bps, pos, B, max_position, out, st) == m.OK
        torch.cuda.synchronize()
        outs.append(out.float().cpu().numpy().reshape(B, 2048))
    return outs


def test_static_decode_attention_matches_engine_and_oracle():
    B = 5
    lens = [1, 63, 64, 130, 200]
    r = synth.rng_for(31, "no_alloc_inputs")
    S = max(lens)
    X = synth.normal_bf16(r, (B, S + 1, 1024), 1.0)           # prefill rows + one decode row per sequence
    slots = [4, 0, 3, 1, 2]
    halves = []
    K, V = [], []
    for half in (0, 1):
        w = selector_weights(half)
        with Engine(w, max_slots=5, max_ctx=256, max_batch=B, max_tokens=B * S) as e:
            m = e.m
            emb = np.zeros((B, S, 1024), np.uint16)
            for b in range(B):
                emb[b, :lens[b]] = X[b, :lens[b]]
            m.tts_bb_prefill(e.h, B, S, slots, lens, None, embeds=dev_bf16_bits(emb))
            dec = np.stack([X[b, lens[b]] for b in range(B)])
            hid = torch.zeros(B, 1024, dtype=torch.float32, device="cuda")
            m.tts_bb_decode_step(e.h, B, slots, lens, None, embeds=dev_bf16_bits(dec), hidden_out=hid)
            halves.append(hid.cpu().numpy().astype(np.float64) - O.bf16_to_f64(dec))
            if half == 0:
                # the engine's cache after the step, gathered into the caller's own paged pool
                bps = (S + 1 + 63) // 64
                perm = synth.block_permutation(31, B * bps)
                pool = torch.zeros(B * bps, 2, 8, 64, 128, dtype=torch.bfloat16, device="cuda")
                table = torch.from_numpy(perm.reshape(B, bps).astype(np.int32)).cuda()
                for b in range(B):
                    n = lens[b] + 1
                    kk = torch.zeros(n, 8, 128, dtype=torch.bfloat16, device="cuda")
                    vv = torch.zeros_like(kk)
                    m.tts_bb_debug_kv_read(e.h, 0, slots[b], 0, n, kk, vv)
                    K.append(kk.double().cpu().numpy())
                    V.append(vv.double().cpu().numpy())
                    for j in range((n + 63) // 64):
                        a, z = j * 64, min(n, (j + 1) * 64)
                        pool[table[b, j], 0, :, : z - a] = kk[a:z].transpose(0, 1)
                        pool[table[b, j], 1, :, : z - a] = vv[a:z].transpose(0, 1)
                lw = w.layers[0]
    engine_attn = np.concatenate(halves, axis=1)               # [B, 2048] from the engine's scratch path

    # queries of the decode tokens (q_norm then RoPE at position lens[b]), rounded to bf16
    sh = synth.ONE_LAYER
    f = O.bf16_to_f64
    q = np.zeros((B, 16, 128))
    for b in range(B):
        y = O.rms_norm(f(X[b, lens[b]])[None], f(lw["in_norm"]), sh.rms_eps)
        qb = (y @ f(lw["wq"]).T).reshape(1, 16, 128)
        q[b] = O.rope_half_rotate(O.rms_norm(qb, f(lw["q_norm"]), sh.rms_eps), [lens[b]], sh.rope_theta)[0]
    q_bits = synth.bf16_bits(q.astype(np.float32))
    q_d = dev_bf16_bits(q_bits)
    want = oracle_attention(q_bits, K, V, lens)
    outs = call_static(q_d, pool, table, bps, lens, max(lens), B)
    for o in outs:
        assert np.all(np.isfinite(o))
        assert rel_err_rows(o, want) <= HIDDEN_TOL, rel_err_rows(o, want)
        assert rel_err_rows(o, engine_attn) <= HIDDEN_TOL, rel_err_rows(o, engine_attn)
    assert np.array_equal(outs[0], outs[1])

    m = tb()
    st = torch.cuda.current_stream().cuda_stream
    pos = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = torch.zeros((B, 16, 128), dtype=torch.bfloat16, device="cuda")
    # sizes beyond the fixed scratch are refused without launching anything
    assert m.tts_bb_gqa_decode_attention_static(q_d, pool, table, bps, pos, 65, max(lens), out, st) == m.E_INVALID
    assert m.tts_bb_gqa_decode_attention_static(q_d, pool, table, bps, pos, B, bps * 64, out, st) == m.E_INVALID
    assert m.tts_bb_gqa_decode_attention_static(q_d, pool, table, bps, pos, B, 2**31 - 1, out, st) == m.E_INVALID


def caller_pool(seed, positions, bps):
    """A caller-built paged pool holding seeded bf16 K/V for each sequence's
    positions 0..positions[b], its blocks scattered by a seeded permutation."""
    B = len(positions)
    perm = synth.block_permutation(seed, B * bps)
    table = perm.reshape(B, bps).astype(np.int32)
    pool = np.zeros((B * bps, 2, 8, 64, 128), np.uint16)
    K, V = [], []
    for b, p in enumerate(positions):
        n = p + 1
        k = synth.kv_values(seed, f"k{b}", n)
        v = synth.kv_values(seed, f"v{b}", n)
        K.append(O.bf16_to_f64(k))
        V.append(O.bf16_to_f64(v))
        for j in range((n + 63) // 64):
            a, z = j * 64, min(n, (j + 1) * 64)
            pool[table[b, j], 0, :, : z - a] = k[a:z].transpose(1, 0, 2)
            pool[table[b, j], 1, :, : z - a] = v[a:z].transpose(1, 0, 2)
    q = synth.normal_bf16(synth.rng_for(seed, "q"), (B, 16, 128), 1.0)
    return dev_bf16_bits(pool), torch.from_numpy(table).cuda(), q, K, V


@pytest.mark.parametrize("case", ["one_split", "whole_array"])
def test_static_decode_attention_split_extremes(case):
    if case == "one_split":                 # every query inside the first block: no combine
        positions = [0, 5, 33, 63]
    else:                                   # 64 sequences up to 512 positions: 8 splits of one block
        positions = [int(x) for x in synth.ragged_lengths(57, 64, 1, 511)]
        positions[17] = 511
    B = len(positions)
    bps = (max(positions) + 1 + 63) // 64
    pool, table, q_bits, K, V = caller_pool(57 if case == "whole_array" else 58, positions, bps)
    outs = call_static(dev_bf16_bits(q_bits), pool, table, bps, positions, max(positions), B)
    want = oracle_attention(q_bits, K, V, positions)
    for o in outs:
        assert np.all(np.isfinite(o))
        assert rel_err_rows(o, want) <= HIDDEN_TOL, rel_err_rows(o, want)
    assert np.array_equal(outs[0], outs[1])


def test_static_decode_attention_clamps_out_of_range_positions():
    """A position above max_position (or below 0) is clamped on the device: the
    call reads only the caller's page-table rows and the other sequences are
    unaffected."""
    positions = [70, 100, 20]
    B = 3
    bps = 2
    pool, table, q_bits, K, V = caller_pool(59, positions, bps)
    q_d = dev_bf16_bits(q_bits)
    good = call_static(q_d, pool, table, bps, positions, 100, B, n_calls=1)[0]
    bad = call_static(q_d, pool, table, bps, [70, 100000, -5], 100, B, n_calls=1)[0]
    assert np.all(np.isfinite(bad))
    assert np.array_equal(bad[0], good[0])
    clamped = oracle_attention(q_bits, K, V, [70, 100, 0])
    assert rel_err_rows(bad, clamped) <= HIDDEN_TOL
