"""KV-cache append indexing, bit-exact (GPU).

The paged cache's values do not depend on where their blocks sit, so two
engines that run the same calls but place the sequences in different slots
and in differently scrambled block pools must hold bit-identical K/V when
read back through their page tables. Both append paths are exercised: the
batched decode step (q/k norm + RoPE + append kernel, three sequences per
call) and the persistent batch-1 step (append inside its attention unit),
with prefill and decode positions crossing 64-token block boundaries. Each
row appended by a decode step is read back right after the step and must be
unchanged at the end (no later append lands on it).
"""
import numpy as np
import pytest

import synth
from tests.gpu_util import Engine, bf16_tensor_bits, dev_bf16_bits

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SHAPE = synth.ModelShape(n_layers=2)
LENS = [70, 5, 127]          # prefill lengths of the three sequences
N_MULTI, N_SINGLE = 66, 4    # batched decode steps, then batch-1 steps per sequence


def _read(m, h, layer, slot, start, n):
    k = torch.zeros(n, 8, 128, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    m.tts_bb_debug_kv_read(h, layer, slot, start, n, k, v)
    return bf16_tensor_bits(k), bf16_tensor_bits(v)


def _run(w, slots, scramble):
    """The same calls in an engine whose sequences live in `slots`; `scramble` first fills and
    frees other slots so the blocks handed out later come from a shuffled free list."""
    r = synth.rng_for(81, "kv_append_inputs")
    S = max(LENS)
    X = synth.normal_bf16(r, (3, S, 1024), 1.0)
    D = synth.normal_bf16(r, (N_MULTI + 3 * N_SINGLE, 3, 1024), 1.0)
    appended = {}
    with Engine(w, max_slots=8, max_ctx=256, max_batch=4, max_tokens=512, kv_blocks=48) as e:
        m = e.m
        if scramble:
            junk = synth.normal_bf16(synth.rng_for(82, "junk"), (4, 100, 1024), 1.0)
            js = [s for s in range(8) if s not in slots][:4]
            m.tts_bb_prefill(e.h, 4, 100, js, [100, 37, 65, 3], embeds=dev_bf16_bits(junk))
            for s in (js[2], js[0], js[3]):
                m.tts_bb_release(e.h, s)
        emb = np.zeros((3, S, 1024), np.uint16)
        for b in range(3):
            emb[b, :LENS[b]] = X[b, :LENS[b]]
        m.tts_bb_prefill(e.h, 3, S, slots, LENS, embeds=dev_bf16_bits(emb))
        kv = list(LENS)
        for t in range(N_MULTI):                                  # batched decode steps
            m.tts_bb_decode_step(e.h, 3, slots, kv, None, embeds=dev_bf16_bits(D[t]))
            for b in range(3):
                for layer in range(SHAPE.n_layers):
                    appended[(b, layer, kv[b])] = _read(m, e.h, layer, slots[b], kv[b], 1)
            kv = [x + 1 for x in kv]
        for b in (2, 0, 1):                                       # batch-1 steps, interleaved
            for t in range(N_SINGLE):
                row = D[N_MULTI + b * N_SINGLE + t, b:b + 1]
                m.tts_bb_decode_step(e.h, 1, [slots[b]], [kv[b]], None, embeds=dev_bf16_bits(row))
                for layer in range(SHAPE.n_layers):
                    appended[(b, layer, kv[b])] = _read(m, e.h, layer, slots[b], kv[b], 1)
                kv[b] += 1
        assert [m.tts_bb_slot_len(e.h, s) for s in slots] == kv
        final = {(b, layer): _read(m, e.h, layer, slots[b], 0, kv[b]) for b in range(3) for layer in range(SHAPE.n_layers)}
    return final, appended, kv


def test_kv_append_bit_exact_across_block_layouts():
    w = synth.model_weights(SHAPE, 81)
    fa, aa, kva = _run(w, [0, 1, 2], scramble=False)
    fb, ab, kvb = _run(w, [6, 3, 5], scramble=True)
    assert kva == kvb
    for key in fa:
        assert np.array_equal(fa[key][0], fb[key][0]) and np.array_equal(fa[key][1], fb[key][1]), key
    # every appended row is what the step wrote, unchanged by the later appends
    for (b, layer, p), (k1, v1) in aa.items():
        k, v = fa[(b, layer)]
        assert np.array_equal(k[p], k1[0]) and np.array_equal(v[p], v1[0]), (b, layer, p)
    for (b, layer, p), (k1, v1) in ab.items():
        k, v = fb[(b, layer)]
        assert np.array_equal(k[p], k1[0]) and np.array_equal(v[p], v1[0]), (b, layer, p)
    # appended rows hold data (not the pool's zero fill)
    for (b, layer, p), (k1, _) in aa.items():
        assert np.any(k1 != 0), (b, layer, p)
