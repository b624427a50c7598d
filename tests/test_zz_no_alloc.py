"""The decode-attention entry point that allocates nothing.

Callers that may not call cudaMalloc (a plug-in whose host framework owns all
device memory, work recorded during CUDA stream capture, a real-time audio
thread) use tts_bb_gqa_decode_attention_static: their own q, KV pool, page
table and output, with the split partials in the library's fixed device
array. This test checks it through the C ABI against the attention that
tts_bb_decode_step computes with the engine's own scratch, on two calls in a
row, within the hidden-state tolerance of the other GPU tests.

The engine's attention output is made observable with a one-layer model whose
MLP weights are zero and whose o_proj selects half of the 2048 attention
outputs (identity on 1024 of them), so hidden_out - input = that half.
"""
import numpy as np
import pytest

import oracle as O
import synth
from tests.gpu_util import HIDDEN_TOL, Engine, dev_bf16_bits, rel_err_rows

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


def test_static_decode_attention_matches_engine():
    B = 5
    lens = [1, 63, 64, 130, 200]
    r = synth.rng_for(31, "no_alloc_inputs")
    S = max(lens)
    X = synth.normal_bf16(r, (B, S + 1, 1024), 1.0)           # prefill rows + one decode row per sequence
    slots = [4, 0, 3, 1, 2]
    halves = []
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
    q_d = dev_bf16_bits(synth.bf16_bits(q.astype(np.float32)))
    pos = torch.tensor(lens, dtype=torch.int32, device="cuda")
    import codec_token_tts_gb300 as m
    st = torch.cuda.current_stream().cuda_stream
    outs = []
    for _ in range(2):                                          # two calls in a row share the scratch
        out = torch.full((B, 16, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert m.tts_bb_gqa_decode_attention_static(q_d, pool, table, bps, pos, B, max(lens), out, st) == m.OK
        torch.cuda.synchronize()
        outs.append(out.float().cpu().numpy().reshape(B, 2048))
    for o in outs:
        assert np.all(np.isfinite(o))
        err = rel_err_rows(o, engine_attn)
        assert err <= HIDDEN_TOL, err
    assert np.array_equal(outs[0], outs[1])

    # sizes beyond the fixed scratch are refused without launching anything
    assert m.tts_bb_gqa_decode_attention_static(q_d, pool, table, bps, pos, 65, max(lens), out, st) == m.E_INVALID
    assert m.tts_bb_gqa_decode_attention_static(q_d, pool, table, bps, pos, B, bps * 64, out, st) == m.E_INVALID
