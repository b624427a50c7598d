"""Failure detection and recovery, made on the host (nothing faults, traps or
hangs the GPU): invalid handles and arguments, unsupported configurations,
injected allocation failure, KV block-pool exhaustion, a device wait forced to
run out (an exchange word withheld) followed by recovery, and bitwise
run-to-run determinism.
"""
import ctypes as C
import os

import numpy as np
import pytest

import synth
from tests.gpu_util import Engine, config_for, dev_i32, f32_zeros, i32_full, tb, weights_for


def small_talker(n_layers=2):
    return synth.ModelShape(n_layers=n_layers, codebook_rows=(3072,) + (2048,) * 15, n_heads_out=1, head_rows=3072)


# ---------------------------------------------------------------- host only (no GPU)
def test_null_handle_is_rejected_everywhere():
    m = tb()
    L = m.lib
    buf = (C.c_int32 * 64)()
    assert L.tts_bb_prefill(None, 1, 1, buf, buf, buf, -1, None, None, None) == m.E_INVALID
    assert L.tts_bb_decode_step(None, 1, buf, buf, buf, -1, None, None, None) == m.E_INVALID
    assert L.tts_bb_maskgit_pass(None, 1, 1, buf, None, buf, -1, None, None) == m.E_INVALID
    assert L.tts_bb_release(None, 0) == m.E_INVALID
    assert L.tts_bb_truncate(None, 0, 0) == m.E_INVALID
    assert L.tts_bb_sync(None) == m.E_INVALID
    assert L.tts_bb_profile(None, 1) == m.E_INVALID
    assert L.tts_bb_debug_fault(None, m.DEBUG_STALL_NEXT_STEP, 0) == m.E_INVALID
    assert L.tts_bb_debug_kv_read(None, 0, 0, 0, 1, None, None) == m.E_INVALID
    assert L.tts_bb_maskgit_update(None, 1, 1, buf, 1, 0, 0, buf, 1, 0, 0, 1, 2.0, 5.0) == m.E_INVALID
    assert L.tts_bb_launch_count(None) == 0
    L.tts_bb_free(None)  # no-op


def _create_status(m, cfg, w):
    out = C.c_void_p()
    st = m.lib.tts_bb_create(C.byref(cfg), C.byref(w.struct), None, C.byref(out))
    if out.value:
        m.lib.tts_bb_free(out.value)
    return st, out.value


def test_create_rejects_bad_and_unsupported_configs_before_touching_the_device():
    m = tb()
    shape = small_talker(1)
    w = synth.model_weights(shape, 30)
    wref = weights_for(w)
    bad = [("max_batch", 0), ("max_batch", 100000), ("n_codebooks", 99), ("rms_eps", 0.0), ("rope_theta", 0.5),
           ("kv_blocks", -1), ("n_layers", -1)]
    for field, val in bad:
        c = config_for(shape)
        setattr(c, field, val)
        st, h = _create_status(m, c, wref)
        assert st == m.E_INVALID and not h, (field, val, st)
    c = config_for(shape)
    c.ffn = 4096  # the kernels are built for SwiGLU widths up to 3072
    st, h = _create_status(m, c, wref)
    assert st == m.E_UNSUPPORTED and not h
    for field in ("max_ctx", "max_tokens", "max_slots"):  # host tables scale with these: capped at 2^20
        c = config_for(shape)
        setattr(c, field, (1 << 20) + 1)
        st, h = _create_status(m, c, wref)
        assert st == m.E_UNSUPPORTED and not h, field
    c = config_for(shape)
    st, h = _create_status(m, c, m.Weights(1, [dict(w.layers[0], wk=None)], w.codebooks, w.final_norm, w.heads))
    assert st == m.E_INVALID and not h


def test_debug_hook_rejects_unknown_and_out_of_range():
    m = tb()
    # a handle is needed for the range checks; without a GPU only the null-handle path runs
    assert m.lib.tts_bb_debug_fault(None, 12345, 0) == m.E_INVALID


# ---------------------------------------------------------------- on the GPU
@pytest.mark.gpu
def test_allocation_failure_injection_fails_creation_cleanly():
    pytest.importorskip("torch")
    m = tb()
    shape = small_talker(2)
    w = synth.model_weights(shape, 31)
    wref = weights_for(w)
    cfg = config_for(shape, max_slots=2, max_ctx=64, max_batch=2, max_tokens=64)
    try:
        for n in (1, 2, 5, 9, 20):
            os.environ["TTS_BB_FAIL_ALLOC_AT"] = str(n)
            st, h = _create_status(m, cfg, wref)
            assert st == m.E_OOM and not h, (n, st)
    finally:
        os.environ.pop("TTS_BB_FAIL_ALLOC_AT", None)
    st, h = _create_status(m, cfg, wref)
    assert st == m.OK


@pytest.mark.gpu
def test_kv_block_pool_exhaustion_then_release():
    pytest.importorskip("torch")
    shape = small_talker(1)
    w = synth.model_weights(shape, 32)
    ids = synth.talker_prefill_ids(32, 100)
    with Engine(w, max_slots=2, max_ctx=256, max_batch=2, max_tokens=128, kv_blocks=2) as e:
        m = e.m
        m.tts_bb_prefill(e.h, 1, 100, [0], [100], dev_i32(ids[None]))  # 2 blocks of 64
        st = m.tts_bb_prefill(e.h, 1, 10, [1], [10], dev_i32(ids[None, :10]), check=False)
        assert st == m.E_OOM
        assert "pool exhausted" in m.lib.tts_bb_last_error(e.h).decode()
        assert m.tts_bb_slot_len(e.h, 1) == 0  # nothing half-done
        m.tts_bb_release(e.h, 0)
        m.tts_bb_prefill(e.h, 1, 10, [1], [10], dev_i32(ids[None, :10]))
        assert m.tts_bb_slot_len(e.h, 1) == 10


def _decode_run(w, ids_prefill, rows, B, fault_at=None):
    """Prefill B slots, then decode len(rows) steps; returns logits per step.
    fault_at: step index at which one persistent step is forced to time out,
    then the position is truncated and the step redone."""
    with Engine(w, max_slots=B, max_ctx=96, max_batch=B, max_tokens=B * 32) as e:
        m = e.m
        P = ids_prefill.shape[0]
        m.tts_bb_prefill(e.h, B, P, list(range(B)), [P] * B, dev_i32(np.stack([ids_prefill] * B)))
        out = []
        logits = f32_zeros(B, 3072)
        am = i32_full(B)
        for t, row in enumerate(rows):
            step_ids = dev_i32(np.stack([row] * B))
            if fault_at == t:
                assert m.tts_bb_debug_fault(e.h, m.DEBUG_WAIT_LIMIT_NS, 20_000_000) == m.OK
                assert m.tts_bb_debug_fault(e.h, m.DEBUG_STALL_NEXT_STEP) == m.OK
                st = m.tts_bb_decode_step(e.h, B, list(range(B)), [P + t] * B, step_ids, 0, logits, am, check=False)
                assert st == m.E_DEVICE_TIMEOUT, st
                for b in range(B):  # drop the position the failed step wrote, then redo the step
                    m.tts_bb_truncate(e.h, b, P + t)
                assert m.tts_bb_debug_fault(e.h, m.DEBUG_WAIT_LIMIT_NS, 2_000_000_000) == m.OK
            m.tts_bb_decode_step(e.h, B, list(range(B)), [P + t] * B, step_ids, 0, logits, am)
            out.append(logits.cpu().numpy().copy())
        return np.array(out)


@pytest.mark.gpu
@pytest.mark.parametrize("B", [1, 2])
def test_device_wait_times_out_then_handle_recovers(B):
    """The persistent decode step's waits are bounded: with one CTA's exchange
    words withheld every wait runs out, the call returns E_DEVICE_TIMEOUT, and
    after truncating the failed position the next steps equal a clean run bit
    for bit."""
    pytest.importorskip("torch")
    shape = small_talker(2)
    w = synth.model_weights(shape, 33)
    ids = synth.talker_prefill_ids(33, 16)
    rows = synth.uniform_ids(synth.rng_for(33, "rows"), shape.codebook_rows, 4)
    clean = _decode_run(w, ids, rows, B)
    faulted = _decode_run(w, ids, rows, B, fault_at=1)
    assert np.array_equal(clean, faulted)


@pytest.mark.gpu
@pytest.mark.parametrize("B", [1, 5])
def test_run_to_run_bitwise_determinism(B):
    """Two identical runs give bitwise-equal logits: fixed-order reductions
    everywhere (exchanges, split-K cluster sums, attention combine), no float
    atomics. B=1 takes the persistent step, B=5 the graph-replayed
    multi-kernel step."""
    pytest.importorskip("torch")
    shape = small_talker(2)
    w = synth.model_weights(shape, 34)
    ids = synth.talker_prefill_ids(34, 16)
    rows = synth.uniform_ids(synth.rng_for(34, "rows"), shape.codebook_rows, 4)
    a = _decode_run(w, ids, rows, B)
    b = _decode_run(w, ids, rows, B)
    assert np.array_equal(a, b)
    assert np.all(np.isfinite(a))
