"""Python binding of the GB300 codec-token TTS backbone engine (libtts_bb.so).

Argument marshalling only: every step of the backbone runs in the CUDA kernels
behind the C ABI declared in include/tts_bb.h. Function names match the C
entry points. Device arrays are passed as integer addresses (for a torch
tensor, ``t.data_ptr()``); host arrays as numpy arrays.

Importing this module loads the compiled library and raises if it is missing:
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, List, Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtts_bb.so")

MAX_CODEBOOKS = 16
MAX_HEADS = 16
KV_BLOCK = 64
LAYER_ROLES = ("in_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "post_norm", "wg", "wu", "wd")

OK, E_INVALID, E_UNSUPPORTED, E_CUDA, E_OOM, E_DEVICE_TIMEOUT, E_BAD_ID, E_NOT_IMPLEMENTED = 0, -1, -2, -3, -4, -5, -6, -7
STATUS_NAMES = {0: "OK", -1: "E_INVALID", -2: "E_UNSUPPORTED", -3: "E_CUDA", -4: "E_OOM",
                -5: "E_DEVICE_TIMEOUT", -6: "E_BAD_ID", -7: "E_NOT_IMPLEMENTED"}


class tts_bb_config(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("hidden", C.c_int), ("n_q_heads", C.c_int), ("n_kv_heads", C.c_int),
                ("head_dim", C.c_int), ("ffn", C.c_int), ("rms_eps", C.c_float), ("rope_theta", C.c_float),
                ("n_codebooks", C.c_int), ("codebook_rows", C.c_int * MAX_CODEBOOKS), ("text_vocab", C.c_int),
                ("audio_codebooks", C.c_int), ("audio_vocab", C.c_int), ("n_heads", C.c_int),
                ("head_rows", C.c_int), ("max_slots", C.c_int), ("max_ctx", C.c_int), ("kv_blocks", C.c_int),
                ("max_batch", C.c_int), ("max_tokens", C.c_int), ("sync_errors", C.c_int)]


class tts_bb_weights(C.Structure):
    _fields_ = [("codebook", C.c_void_p * MAX_CODEBOOKS), ("text_table", C.c_void_p), ("audio_table", C.c_void_p),
                ("layer", C.POINTER(C.c_void_p)), ("final_norm", C.c_void_p), ("head", C.c_void_p * MAX_HEADS)]


class tts_bb_opts(C.Structure):
    _fields_ = [("embeds", C.c_void_p), ("hidden_out", C.c_void_p), ("argmax_stride", C.c_int)]


class TtsBbError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class tts_bb_dac_block(C.Structure):
    _fields_ = [("alpha", C.c_void_p), ("up_w", C.c_void_p), ("up_b", C.c_void_p),
                ("res_alpha1", C.c_void_p * 3), ("res_w1", C.c_void_p * 3), ("res_b1", C.c_void_p * 3),
                ("res_alpha2", C.c_void_p * 3), ("res_w2", C.c_void_p * 3), ("res_b2", C.c_void_p * 3)]


class tts_bb_dac_weights(C.Structure):
    _fields_ = [("fc2_w", C.c_void_p), ("fc2_b", C.c_void_p), ("conv1_w", C.c_void_p), ("conv1_b", C.c_void_p),
                ("block", tts_bb_dac_block * 5), ("final_alpha", C.c_void_p), ("conv2_w", C.c_void_p),
                ("conv2_b", C.c_void_p)]


def _load() -> C.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with codec_token_tts_gb300.build.build() "
                          "(there is no CPU fallback)")
    lib = C.CDLL(LIB_PATH)
    P, I, V = C.c_void_p, C.c_int, None
    sig = {
        "tts_bb_default_config": (V, [C.POINTER(tts_bb_config)]),
        "tts_bb_create": (I, [C.POINTER(tts_bb_config), C.POINTER(tts_bb_weights), P, C.POINTER(P)]),
        "tts_bb_free": (V, [P]),
        "tts_bb_prefill": (I, [P, I, I, P, P, P, I, P, P, C.POINTER(tts_bb_opts)]),
        "tts_bb_decode_step": (I, [P, I, P, P, P, I, P, P, C.POINTER(tts_bb_opts)]),
        "tts_bb_maskgit_pass": (I, [P, I, I, P, P, P, I, P, C.POINTER(tts_bb_opts)]),
        "tts_bb_release": (I, [P, I]),
        "tts_bb_truncate": (I, [P, I, I]),
        "tts_bb_slot_len": (I, [P, I]),
        "tts_bb_sync": (I, [P]),
        "tts_bb_last_error": (C.c_char_p, [P]),
        "tts_bb_version": (C.c_char_p, []),
        "tts_bb_debug_kv_read": (I, [P, I, I, I, I, P, P]),
        "tts_bb_debug_kv_write": (I, [P, I, I, I, I, P, P]),
        "tts_bb_launch_count": (C.c_uint64, [P]),
        "tts_bb_profile": (I, [P, I]),
        "tts_bb_profile_report": (C.c_char_p, [P]),
        "tts_bb_gqa_decode_attention_static": (I, [P, P, P, I, P, I, I, P, P]),
        "tts_bb_debug_fault": (I, [P, I, C.c_int64]),
        "tts_bb_maskgit_update": (I, [P, I, I, P, I, I, I, P, I, I, I, I, C.c_float, C.c_float]),
        "tts_bb_maskgit_schedule": (I, [I, I, C.c_double, P]),
        "tts_bb_frame_step": (I, [P, P, I, P, P, P, P]),
        "tts_bb_decode_step_host": (I, [P, I, P, P, P, I, P, P]),
        "tts_bb_rvq_create": (I, [I, I, I, I, C.POINTER(P), C.POINTER(P), C.POINTER(P), P, C.POINTER(P)]),
        "tts_bb_rvq_decode": (I, [P, I, I, P, P]),
        "tts_bb_rvq_sync": (I, [P]),
        "tts_bb_rvq_free": (V, [P]),
        "tts_bb_quantizer_create": (I, [I, I, I, I, C.POINTER(P), P, P, P, C.POINTER(P)]),
        "tts_bb_quantizer_decode": (I, [P, I, I, P, P]),
        "tts_bb_quantizer_sync": (I, [P]),
        "tts_bb_quantizer_free": (V, [P]),
        "tts_bb_dac_create": (I, [C.POINTER(tts_bb_dac_weights), P, C.POINTER(P)]),
        "tts_bb_dac_decode": (I, [P, I, I, P, P]),
        "tts_bb_dac_sync": (I, [P]),
        "tts_bb_dac_free": (V, [P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()
EXPORTED = ("tts_bb_default_config", "tts_bb_create", "tts_bb_free", "tts_bb_prefill", "tts_bb_decode_step",
            "tts_bb_maskgit_pass", "tts_bb_release", "tts_bb_truncate", "tts_bb_slot_len", "tts_bb_sync",
            "tts_bb_last_error", "tts_bb_version", "tts_bb_debug_kv_read", "tts_bb_debug_kv_write",
            "tts_bb_launch_count", "tts_bb_profile", "tts_bb_profile_report",
            "tts_bb_gqa_decode_attention_static", "tts_bb_debug_fault", "tts_bb_maskgit_update",
            "tts_bb_maskgit_schedule", "tts_bb_frame_step", "tts_bb_rvq_create", "tts_bb_rvq_decode",
            "tts_bb_rvq_sync", "tts_bb_rvq_free", "tts_bb_dac_create", "tts_bb_dac_decode", "tts_bb_dac_sync", "tts_bb_dac_free",
            "tts_bb_decode_step_host", "tts_bb_quantizer_create", "tts_bb_quantizer_decode",
            "tts_bb_quantizer_sync", "tts_bb_quantizer_free")


def _ptr(x) -> Optional[int]:
    """Address of a numpy array, a torch tensor, or an int; None stays None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        assert x.flags["C_CONTIGUOUS"], "arrays passed to the engine must be C-contiguous"
        return x.ctypes.data
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _host_i32(x) -> Optional[np.ndarray]:
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _opts(embeds=None, hidden_out=None, argmax_stride=0):
    if embeds is None and hidden_out is None and not argmax_stride:
        return None
    return C.byref(tts_bb_opts(_ptr(embeds), _ptr(hidden_out), int(argmax_stride)))


def _check(h, status: int):
    if status != OK:
        raise TtsBbError(status, tts_bb_last_error(h))
    return status


# ---------------------------------------------------------------- C entry points
def tts_bb_default_config() -> tts_bb_config:
    c = tts_bb_config()
    lib.tts_bb_default_config(C.byref(c))
    return c


def tts_bb_version() -> str:
    return lib.tts_bb_version().decode()


def tts_bb_last_error(h) -> str:
    return lib.tts_bb_last_error(h).decode()


class Weights:
    """Keeps the pointer arrays (and the arrays they point to) alive until create returns."""

    def __init__(self, n_layers: int, layers: Sequence[Dict[str, object]], codebooks: Sequence[object] = (),
                 final_norm=None, heads: Sequence[object] = (), text_table=None, audio_table=None):
        self.keep = [layers, codebooks, final_norm, heads, text_table, audio_table]
        self.layer_ptrs = (C.c_void_p * (n_layers * len(LAYER_ROLES)))()
        for l in range(n_layers):
            for r, name in enumerate(LAYER_ROLES):
                self.layer_ptrs[l * len(LAYER_ROLES) + r] = _ptr(layers[l][name])
        s = tts_bb_weights()
        for k, t in enumerate(codebooks):
            s.codebook[k] = _ptr(t)
        s.text_table = _ptr(text_table)
        s.audio_table = _ptr(audio_table)
        s.layer = C.cast(self.layer_ptrs, C.POINTER(C.c_void_p))
        s.final_norm = _ptr(final_norm)
        for j, t in enumerate(heads):
            s.head[j] = _ptr(t)
        self.struct = s


def tts_bb_create(cfg: tts_bb_config, weights: Weights, stream: int = 0) -> int:
    out = C.c_void_p()
    st = lib.tts_bb_create(C.byref(cfg), C.byref(weights.struct), C.c_void_p(stream or None), C.byref(out))
    if st != OK:
        raise TtsBbError(st, "tts_bb_create failed")
    return out.value


def tts_bb_free(h) -> None:
    lib.tts_bb_free(h)


def tts_bb_prefill(h, B: int, S: int, slots, lens, ids=None, head_idx: int = -1, logits_out=None, argmax_out=None,
                   embeds=None, hidden_out=None, argmax_stride: int = 0, check: bool = True) -> int:
    sl, ln = _host_i32(slots), _host_i32(lens)
    st = lib.tts_bb_prefill(h, B, S, _ptr(sl), _ptr(ln), _ptr(ids), head_idx, _ptr(logits_out), _ptr(argmax_out),
                            _opts(embeds, hidden_out, argmax_stride))
    return _check(h, st) if check else st


def tts_bb_decode_step(h, B: int, slots, kv_lens, ids=None, head_idx: int = -1, logits_out=None, argmax_out=None,
                       embeds=None, hidden_out=None, argmax_stride: int = 0, check: bool = True) -> int:
    sl, kl = _host_i32(slots), _host_i32(kv_lens)
    st = lib.tts_bb_decode_step(h, B, _ptr(sl), _ptr(kl), _ptr(ids), head_idx, _ptr(logits_out), _ptr(argmax_out),
                                _opts(embeds, hidden_out, argmax_stride))
    return _check(h, st) if check else st


def tts_bb_maskgit_pass(h, B: int, S: int, ids, audio_mask, key_lens=None, audio_start: int = 0, logits_out=None,
                        hidden_out=None, check: bool = True) -> int:
    kl = _host_i32(key_lens)
    st = lib.tts_bb_maskgit_pass(h, B, S, _ptr(ids), _ptr(audio_mask), _ptr(kl), audio_start, _ptr(logits_out),
                                 _opts(None, hidden_out, 0))
    return _check(h, st) if check else st


def tts_bb_maskgit_update(h, n_items: int, T: int, logits, S_logits: int, cond_pos0: int, uncond_pos0: int, ids,
                          S_ids: int, cond_ids_pos0: int, uncond_ids_pos0: int, n_unmask: int,
                          cfg_scale: float = 2.0, layer_penalty: float = 5.0, check: bool = True) -> int:
    st = lib.tts_bb_maskgit_update(h, n_items, T, _ptr(logits), S_logits, cond_pos0, uncond_pos0, _ptr(ids), S_ids,
                                   cond_ids_pos0, uncond_ids_pos0, n_unmask, cfg_scale, layer_penalty)
    return _check(h, st) if check else st


def tts_bb_frame_step(talker, cp, B: int, slots, kv_lens, codes, talker_logits=None, check: bool = True) -> int:
    sl, kl = _host_i32(slots), _host_i32(kv_lens)
    st = lib.tts_bb_frame_step(talker, cp, B, _ptr(sl), _ptr(kl), _ptr(codes), _ptr(talker_logits))
    if check and st != OK:
        raise TtsBbError(st, (lib.tts_bb_last_error(talker) or b"").decode() + " / " +
                         (lib.tts_bb_last_error(cp) or b"").decode())
    return st


def tts_bb_rvq_create(embed, proj_w, proj_b, stream=None):
    """embed, proj_w, proj_b: lists (one per codebook) of device bf16 tensors [n][d], [out][d], [out]."""
    K = len(embed)
    n, d = int(embed[0].shape[0]), int(embed[0].shape[1])
    out_dim = int(proj_w[0].shape[0])
    arr = lambda xs: (C.c_void_p * K)(*[_ptr(x) for x in xs])
    h = C.c_void_p()
    st = lib.tts_bb_rvq_create(K, n, d, out_dim, arr(embed), arr(proj_w), arr(proj_b), stream, C.byref(h))
    if st != OK:
        raise TtsBbError(st, "tts_bb_rvq_create")
    return h.value


def tts_bb_rvq_decode(r, B: int, T: int, codes, out, check: bool = True) -> int:
    st = lib.tts_bb_rvq_decode(r, B, T, _ptr(codes), _ptr(out))
    if check and st != OK:
        raise TtsBbError(st, "tts_bb_rvq_decode")
    return st


def tts_bb_rvq_sync(r) -> int:
    return lib.tts_bb_rvq_sync(r)


def tts_bb_rvq_free(r) -> None:
    lib.tts_bb_rvq_free(r)


def tts_bb_quantizer_create(codebooks, proj_semantic, proj_acoustic, stream=None):
    """codebooks: list (one per codebook) of device bf16 tensors [n][d]; projections device bf16 [out][d]."""
    K = len(codebooks)
    n, d = int(codebooks[0].shape[0]), int(codebooks[0].shape[1])
    out_dim = int(proj_semantic.shape[0])
    books = (C.c_void_p * K)(*[_ptr(x) for x in codebooks])
    h = C.c_void_p()
    st = lib.tts_bb_quantizer_create(K, n, d, out_dim, books, _ptr(proj_semantic), _ptr(proj_acoustic), stream,
                                     C.byref(h))
    if st != OK:
        raise TtsBbError(st, "tts_bb_quantizer_create")
    return h.value


def tts_bb_quantizer_decode(q, B: int, T: int, codes, out, check: bool = True) -> int:
    st = lib.tts_bb_quantizer_decode(q, B, T, _ptr(codes), _ptr(out))
    if check and st != OK:
        raise TtsBbError(st, "tts_bb_quantizer_decode")
    return st


def tts_bb_quantizer_sync(q) -> int:
    return lib.tts_bb_quantizer_sync(q)


def tts_bb_quantizer_free(q) -> None:
    lib.tts_bb_quantizer_free(q)


def tts_bb_dac_create(w: dict, stream=None):
    """w: device fp32 tensors keyed like the oracle's dict (fc2_w, fc2_b, conv1_w, conv1_b,
    blocks[i]{alpha, up_w, up_b, res[j]{alpha1, w1, b1, alpha2, w2, b2}}, final_alpha, conv2_w, conv2_b)."""
    s = tts_bb_dac_weights()
    for k in ("fc2_w", "fc2_b", "conv1_w", "conv1_b", "final_alpha", "conv2_w", "conv2_b"):
        setattr(s, k, _ptr(w[k]))
    for i, blk in enumerate(w["blocks"]):
        bs = s.block[i]
        bs.alpha, bs.up_w, bs.up_b = _ptr(blk["alpha"]), _ptr(blk["up_w"]), _ptr(blk["up_b"])
        for j, ru in enumerate(blk["res"]):
            bs.res_alpha1[j], bs.res_w1[j], bs.res_b1[j] = _ptr(ru["alpha1"]), _ptr(ru["w1"]), _ptr(ru["b1"])
            bs.res_alpha2[j], bs.res_w2[j], bs.res_b2[j] = _ptr(ru["alpha2"]), _ptr(ru["w2"]), _ptr(ru["b2"])
    h = C.c_void_p()
    st = lib.tts_bb_dac_create(C.byref(s), stream, C.byref(h))
    if st != OK:
        raise TtsBbError(st, "tts_bb_dac_create")
    return h.value


def tts_bb_dac_decode(d, B: int, T: int, features, audio, check: bool = True) -> int:
    st = lib.tts_bb_dac_decode(d, B, T, _ptr(features), _ptr(audio))
    if check and st != OK:
        raise TtsBbError(st, "tts_bb_dac_decode")
    return st


def tts_bb_dac_sync(d) -> int:
    return lib.tts_bb_dac_sync(d)


def tts_bb_dac_free(d) -> None:
    lib.tts_bb_dac_free(d)


def tts_bb_maskgit_schedule(num_step: int, n_total: int, t_shift: float = 0.1) -> np.ndarray:
    out = np.zeros(num_step, np.int32)
    st = lib.tts_bb_maskgit_schedule(num_step, n_total, t_shift, _ptr(out))
    if st != OK:
        raise TtsBbError(st, "tts_bb_maskgit_schedule: bad arguments")
    return out


def tts_bb_release(h, slot: int, check: bool = True) -> int:
    st = lib.tts_bb_release(h, slot)
    return _check(h, st) if check else st


def tts_bb_truncate(h, slot: int, length: int, check: bool = True) -> int:
    st = lib.tts_bb_truncate(h, slot, length)
    return _check(h, st) if check else st


def tts_bb_slot_len(h, slot: int) -> int:
    return lib.tts_bb_slot_len(h, slot)


def tts_bb_sync(h, check: bool = True) -> int:
    st = lib.tts_bb_sync(h)
    return _check(h, st) if check else st


def tts_bb_debug_kv_read(h, layer: int, slot: int, pos0: int, n: int, k_out, v_out, check: bool = True) -> int:
    st = lib.tts_bb_debug_kv_read(h, layer, slot, pos0, n, _ptr(k_out), _ptr(v_out))
    return _check(h, st) if check else st


def tts_bb_debug_kv_write(h, layer: int, slot: int, pos0: int, n: int, k, v, check: bool = True) -> int:
    st = lib.tts_bb_debug_kv_write(h, layer, slot, pos0, n, _ptr(k), _ptr(v))
    return _check(h, st) if check else st


def tts_bb_launch_count(h) -> int:
    return int(lib.tts_bb_launch_count(h))


def tts_bb_profile(h, on: bool) -> int:
    return _check(h, lib.tts_bb_profile(h, 1 if on else 0))


def tts_bb_profile_report(h) -> dict:
    import json
    return json.loads(lib.tts_bb_profile_report(h).decode())


DEBUG_WAIT_LIMIT_NS, DEBUG_STALL_NEXT_STEP = 1, 2


def tts_bb_debug_fault(h, what: int, arg: int = 0) -> int:
    """Failure-handling test hook (see include/tts_bb.h); returns the status."""
    return lib.tts_bb_debug_fault(h, what, int(arg))


def tts_bb_gqa_decode_attention_static(q, kv_pool, page_table, blocks_per_seq: int, positions, B: int,
                                       max_position: int, out, stream: int = 0) -> int:
    """Decode attention on caller buffers with the library's fixed scratch (allocates nothing)."""
    return lib.tts_bb_gqa_decode_attention_static(_ptr(q), _ptr(kv_pool), _ptr(page_table), blocks_per_seq,
                                                  _ptr(positions), B, max_position, _ptr(out),
                                                  C.c_void_p(stream or None))
