#!/usr/bin/env python3
"""Benchmark of the codec-token TTS backbone step on GB300 (one JSON line).

Workload (default, ``talker_b1``): the 28-layer Qwen3-0.6B-shaped Talker at
batch 1 — a 128-position prefill of 16 summed codebook embeddings, then decode
steps with query length 1, a 3072-way codec head and the greedy argmax fed
back on the device as the next codebook-0 id. One timed step = one decode step
= one codec token. Positions cycle through 128..383 (256 decode steps per
utterance, the slot is rewound to 128 between utterances), so the KV lengths
seen are exactly those of a 128 + 256 generation.

``--workload serving_b64``: 64 concurrent streams with ragged cached lengths
uniform in [200, 2000], paged KV, one decode step per stream per call; one
timed step = one call = 64 codec tokens.

Inputs are synthetic (seeded bf16 N(0, 0.02) weights and uniform ids) and
resident in HBM before the timed region. The 880 MB of weights streamed per
step exceed the 129 MB L2, so no flush is needed between steps.

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload (the oracle is the reference for this method; it is a deliberately
slow, obviously correct program).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "codec tokens/s per GB300 (decode, batch 1 & 64); % of HBM roofline"
UNIT = "codec tokens/s"
P_PREFILL = 128
N_DECODE = 256
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------- distributed (replicas only)
def dist_setup(backend):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=ws)
    return ws, rank, local


def dist_barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(ws, x: float) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
def this_rank_gpu() -> str:
    """The physical GPU of this rank (cuda:LOCAL_RANK) as nvidia-smi names it."""
    local = int(os.environ.get("LOCAL_RANK", "0"))
    vis = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    return vis[local] if local < len(vis) else str(local)


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.idx = gpu  # nvidia-smi -i: index or UUID
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def wait_first(self, limit_s: float = 3.0):
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < limit_s:
            time.sleep(0.01)
        self.skip = len(self.lines)  # samples taken before the timed region are not counted

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines[getattr(self, "skip", 0):] or self.lines[-1:]  # at least the latest sample
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- workloads
class TalkerB1:
    """Talker batch 1: 128-position prefill, then decode steps at positions 128..383."""
    name = "talker_b1"
    seed = 1
    B = 1

    def __init__(self):
        self.shape = synth.TALKER
        self.w = synth.model_weights(self.shape, self.seed)
        self.prefill_ids = synth.talker_prefill_ids(self.seed, P_PREFILL)
        self.rest = synth.uniform_ids(synth.rng_for(self.seed, "decode_rest"), self.shape.codebook_rows[1:], N_DECODE)

    def config(self):
        return {"workload": "talker_b1: Qwen3-0.6B-shaped Talker, 28 layers, batch 1, 128-position prefill then "
                            "decode at positions 128..383, 3072-way head, greedy id0 fed back",
                "global_batch": 1, "seq_len": P_PREFILL + N_DECODE, "layers": 28,
                "l2": "no flush: 880 MB of weights per step > 129 MB L2"}

    def algorithmic_bytes_per_step(self, pos):
        """Weights + 16 embedding rows + final norm + head, KV read (pos + 1 tokens) and write, logits."""
        w = 28 * 31_461_888 + 16 * 2048 + 2048 + 3072 * 1024 * 2
        return w + 114_688 * (pos + 1) + 114_688 + 3072 * 4


class ServingB64:
    """64 streams, ragged cached lengths U[200, 2000], one decode step per stream per call."""
    name = "serving_b64"
    seed = 2
    B = 64

    def __init__(self):
        self.shape = synth.TALKER
        self.w = synth.model_weights(self.shape, self.seed)
        self.L0 = synth.ragged_lengths(self.seed, self.B, 200, 2000)

    def config(self):
        return {"workload": "serving_b64: 28-layer Talker, 64 streams, ragged KV lengths U[200,2000], paged KV "
                            "(64-token blocks), one decode step per stream per call, 3072-way head",
                "global_batch": 64, "seq_len": int(self.L0.max()), "layers": 28,
                "l2": "no flush: 880 MB weights + ~10 GB KV per step > 129 MB L2"}


def make_engine(wl, m, stream, max_ctx, max_batch, max_tokens, max_slots):
    from tests.gpu_util import config_for, weights_for
    cfg = config_for(wl.shape, max_slots=max_slots, max_ctx=max_ctx, max_batch=max_batch, max_tokens=max_tokens,
                     sync_errors=0)
    wref = weights_for(wl.w)
    return m.tts_bb_create(cfg, wref, stream)


# ---------------------------------------------------------------- our arm: talker_b1
def run_talker_b1(args, ws, rank):
    import torch
    import codec_token_tts_gb300 as m
    from tests.gpu_util import dev_i32

    wl = TalkerB1()
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    h = make_engine(wl, m, stream.cuda_stream, P_PREFILL + N_DECODE, 1, P_PREFILL, 1)
    n_all = max(args.steps, args.warmup) + 1
    # ids for every decode step: column 0 is overwritten by the previous step's argmax
    rest = np.tile(wl.rest, ((n_all + N_DECODE - 1) // N_DECODE, 1))[:n_all]
    ids = np.concatenate([np.zeros((n_all, 1), np.int32), rest], axis=1)
    ids_d = dev_i32(ids)
    logits = torch.zeros(1, 3072, dtype=torch.float32, device="cuda")
    pre_ids = dev_i32(wl.prefill_ids.reshape(1, P_PREFILL, 16))
    first = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.tts_bb_prefill(h, 1, P_PREFILL, [0], [P_PREFILL], pre_ids, 0, logits, first)
    slot, kv = np.zeros(1, np.int32), np.zeros(1, np.int32)

    def steps(n):
        """n decode steps, rewinding to position 128 every 256 steps."""
        for t in range(n):
            pos = P_PREFILL + (t % N_DECODE)
            if pos == P_PREFILL:
                m.tts_bb_truncate(h, 0, P_PREFILL)
                ids_d[t, 0:1].copy_(first)
            kv[0] = pos
            m.lib.tts_bb_decode_step(h, 1, slot.ctypes.data, kv.ctypes.data, ids_d[t].data_ptr(), 0,
                                     logits.data_ptr(), ids_d[t + 1].data_ptr(), None)

    steps(args.warmup)
    m.tts_bb_sync(h)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(this_rank_gpu())
    n0 = m.tts_bb_launch_count(h)
    clocks.start()
    clocks.wait_first()  # the sampler is live before the timed region starts
    dist_barrier(ws)
    torch.cuda.synchronize()
    ev0.record(stream)
    steps(args.steps)
    ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    dist_barrier(ws)
    ms = ev0.elapsed_time(ev1)
    launches = m.tts_bb_launch_count(h) - n0
    m.tts_bb_sync(h)
    ms_max = dist_max(ws, ms)

    # profiled pass: per-kernel event times for the roofline of the dominant kernel
    m.tts_bb_profile(h, True)
    steps(min(args.steps, 2 * N_DECODE))
    rep = m.tts_bb_profile_report(h)
    m.tts_bb_profile(h, False)

    # end to end through the C ABI with host buffers: per step, the ids go from pinned host memory
    # to the device, the step runs, and its argmax (the token fed back) comes back to the host
    host_ids_t = torch.from_numpy(ids.copy()).pin_memory()
    host_am_t = torch.zeros(1, dtype=torch.int32).pin_memory()
    host_ids, host_am = host_ids_t.numpy(), host_am_t.numpy()
    m.tts_bb_truncate(h, 0, P_PREFILL)
    first_host = int(first.cpu().item())
    n_e2e = min(args.steps, 4 * N_DECODE)
    row_bytes = host_ids.strides[0]
    torch.cuda.synchronize()
    dist_barrier(ws)
    t0 = time.perf_counter()
    nxt = first_host
    for t in range(n_e2e):
        pos = P_PREFILL + (t % N_DECODE)
        if pos == P_PREFILL:
            m.tts_bb_truncate(h, 0, P_PREFILL)
            nxt = first_host
        host_ids[t, 0] = nxt
        kv[0] = pos
        m.lib.tts_bb_decode_step_host(h, 1, slot.ctypes.data, kv.ctypes.data, host_ids.ctypes.data + t * row_bytes, 0,
                                      host_am.ctypes.data, None)
        nxt = int(host_am[0])
    e2e_s = dist_max(ws, time.perf_counter() - t0)  # every step ended with a synchronisation
    dist_barrier(ws)
    m.tts_bb_sync(h)
    m.tts_bb_free(h)

    tokens = args.steps * ws
    value = tokens / (ms_max / 1e3)
    pos_bytes = np.mean([wl.algorithmic_bytes_per_step(P_PREFILL + (t % N_DECODE)) for t in range(args.steps)])
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "config": dict(wl.config(), parallelism="replicas" if ws > 1 else "single"),
        "hbm_step_roofline": {"algorithmic_bytes_per_step": pos_bytes,
                              "achieved_gbs": pos_bytes / (ms_max / args.steps) / 1e6,
                              "frac_of_measured": pos_bytes / (ms_max / args.steps) / 1e6 / peaks()[0]["hbm_gbs"],
                              "frac_of_8tbs": pos_bytes / (ms_max / args.steps) / 1e6 / 8000.0,
                              "target_frac": 0.70},
        "clocks": clk, "gpu_launches": int(launches),
        "e2e": {"value": n_e2e * ws / e2e_s, "unit": UNIT, "h2d_bytes_per_step": 16 * 4, "d2h_bytes_per_step": 4 + 4,
                "path": "tts_bb_decode_step_host: ids H2D, step, argmax + error word D2H, one sync per step"},
        "kernel_profile": rep,
    }
    return res, wl


def fill_kv_random(m, h, L0, slots, n_layers, seed):
    """Synthetic cached K/V (bf16 N(0,1), the scale of normed keys) for every stream, written
    through the page table; generated on the device (their values do not affect timing)."""
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    for layer in range(n_layers):
        for b in range(len(L0)):
            n = int(L0[b])
            k = torch.randn(n, 8, 128, generator=g, device="cuda").to(torch.bfloat16)
            v = torch.randn(n, 8, 128, generator=g, device="cuda").to(torch.bfloat16)
            m.tts_bb_debug_kv_write(h, layer, int(slots[b]), 0, n, k, v)
    m.tts_bb_sync(h)


def run_serving_b64(steps, warmup):
    """64 streams, ragged cached lengths U[200, 2000], one decode step per stream per call."""
    import torch
    import codec_token_tts_gb300 as m
    from tests.gpu_util import dev_i32
    wl = ServingB64()
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    h = make_engine(wl, m, stream.cuda_stream, 2000 + steps + warmup + 1, wl.B, wl.B, wl.B)
    slots = synth.block_permutation(wl.seed, wl.B)
    fill_kv_random(m, h, wl.L0, slots, 28, wl.seed)
    ids = synth.uniform_ids(synth.rng_for(wl.seed, "serve_ids"), wl.shape.codebook_rows, (steps + warmup + 1) * wl.B)
    ids_d = dev_i32(ids.reshape(steps + warmup + 1, wl.B, 16))
    logits = torch.zeros(wl.B, 3072, dtype=torch.float32, device="cuda")
    sl = np.ascontiguousarray(slots, np.int32)
    kv = np.ascontiguousarray(wl.L0, np.int32).copy()

    def run(n, t0):
        for t in range(t0, t0 + n):
            # greedy ids written into the next step's codebook-0 column (stride 16)
            m.lib.tts_bb_decode_step(h, wl.B, sl.ctypes.data, kv.ctypes.data, ids_d[t].data_ptr(), 0,
                                     logits.data_ptr(), ids_d[t + 1, :, 0].data_ptr(),
                                     m._opts(None, None, 16))
            kv[:] += 1

    run(warmup, 0)
    m.tts_bb_sync(h)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    run(steps, warmup)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    st = m.tts_bb_sync(h, check=False)
    # profiled steps for the roofline of the dominant kernel
    m.tts_bb_profile(h, True)
    kv0 = kv.copy()
    for b in range(wl.B):
        m.tts_bb_truncate(h, int(slots[b]), int(wl.L0[b]) + warmup)
    kv[:] = wl.L0 + warmup
    run(min(steps, 8), warmup)
    rep = m.tts_bb_profile_report(h)
    m.tts_bb_profile(h, False)
    m.tts_bb_free(h)
    kv_bytes = 114_688 * float(np.sum(wl.L0 + warmup + steps / 2 + 1))
    step_bytes = 28 * 31_461_888 + 64 * 16 * 2048 + 3072 * 1024 * 2 + kv_bytes + 64 * 114_688
    return {"workload": wl.config()["workload"], "value": wl.B / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
            "steps": steps, "status": st, "algorithmic_bytes_per_step": step_bytes,
            "hbm_frac_of_measured": step_bytes / (ms / 1e3) / 1e9 / peaks()[0]["hbm_gbs"],
            "roofline": roofline_from_profile(rep), "kernel_profile": rep}


def run_maskgit(steps, warmup):
    """OmniVoice MaskGIT pass: B=8 x S=1024 (256 text + 768 audio), 28 bidirectional layers, audio heads."""
    import torch
    import codec_token_tts_gb300 as m
    from tests.gpu_util import config_for, dev_i32, dev_u8, weights_for
    seed = 4
    w = synth.model_weights(synth.OMNIVOICE, seed)
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    cfg = config_for(synth.OMNIVOICE, max_slots=0, max_ctx=0, max_batch=8, max_tokens=8192, sync_errors=0)
    h = m.tts_bb_create(cfg, weights_for(w), stream.cuda_stream)
    passes = [synth.maskgit_inputs(seed, s) for s in range(4)]
    ids_d = [dev_i32(p[0]) for p in passes]
    mask_d = [dev_u8(p[1]) for p in passes]
    logits = torch.zeros(8, 8, 768, 1025, dtype=torch.float32, device="cuda")

    def run(n):
        for i in range(n):
            m.tts_bb_maskgit_pass(h, 8, 1024, ids_d[i % 4], mask_d[i % 4], None, 256, logits, check=False)

    run(warmup)
    m.tts_bb_sync(h)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    run(steps)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    st = m.tts_bb_sync(h, check=False)
    m.tts_bb_profile(h, True)
    run(2)
    rep = m.tts_bb_profile_report(h)
    m.tts_bb_profile(h, False)
    refine = run_maskgit_refinement(m, h, seed, stream)
    m.tts_bb_free(h)
    refine["rvq_decode"] = run_rvq_decode(m, stream)
    refine["quantizer_decode"] = run_quantizer_decode(m, stream)
    refine["dac_decode"] = run_dac_decode(m, stream)
    flops = 2 * 8192 * 15_728_640 * 28 + 4 * 8 * 16 * 1024 ** 2 * 128 * 28 + 2 * 8 * 768 * 8200 * 1024
    pk = peaks()[0]
    return {"workload": "maskgit: OmniVoice LM pass, 28 layers, B=8 x S=1024 (256 text + 768 audio), bidirectional, "
                        "8 x 1025 audio heads over the 768 audio positions",
            "value": 1e3 / ms, "unit": "passes/s", "ms_per_pass": ms, "steps": steps, "status": st,
            "tflops": flops / (ms / 1e3) / 1e12, "flop_per_pass": flops,
            "tensor_frac_of_measured_sustained": flops / (ms / 1e3) / 1e12 / pk["bf16_tflops_sustained"],
            "roofline": roofline_from_profile(rep), "refinement": refine, "kernel_profile": rep}


def run_rvq_decode(m, stream, B=4, T=768, reps=20):
    """RVQ codec decode of a refinement's output: 4 items x 768 frames x 8 codebooks of 1024 x 64
    (seeded bf16 tables) -> [4][768][1024] fp32 features."""
    import torch
    from tests.gpu_util import dev_bf16_bits, dev_i32
    K, N, D, OUT = 8, 1024, 64, 1024
    r = synth.rng_for(5, "rvq_tables")
    e = [dev_bf16_bits(synth.normal_bf16(r, (N, D), 1.0)) for _ in range(K)]
    w = [dev_bf16_bits(synth.normal_bf16(r, (OUT, D), 0.05)) for _ in range(K)]
    b = [dev_bf16_bits(synth.normal_bf16(r, (OUT,), 0.1)) for _ in range(K)]
    rv = m.tts_bb_rvq_create(e, w, b, stream.cuda_stream)
    codes = dev_i32(synth.rng_for(5, "rvq_codes").integers(0, N, (B, K, T)))
    out = torch.zeros(B, T, OUT, dtype=torch.float32, device="cuda")
    for _ in range(3):
        m.tts_bb_rvq_decode(rv, B, T, codes, out)
    st = m.tts_bb_rvq_sync(rv)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(reps):
        m.tts_bb_rvq_decode(rv, B, T, codes, out)
    ev1.record(stream)
    torch.cuda.synchronize()
    m.tts_bb_rvq_free(rv)
    us = ev0.elapsed_time(ev1) / reps * 1e3
    # codes read, gathered 64-d rows, packed weights read once, output written
    nbytes = B * K * T * 4 + B * T * K * D * 2 + OUT * K * D * 2 + B * T * OUT * 4
    return {"workload": f"RVQ decode: {B} x {T} frames x {K} codebooks (1024 x 64) -> {OUT}-d fp32",
            "us_per_decode": us, "frames_per_s": B * T / (us / 1e6), "status": st,
            "algorithmic_bytes": nbytes, "hbm_frac_of_measured": nbytes / (us / 1e6) / 1e9 / peaks()[0]["hbm_gbs"]}


def run_quantizer_decode(m, stream, B=4, T=768, reps=20):
    """Qwen3-TTS quantizer lookup: 4 x 768 frames x 16 codebooks (2048 x 256, seeded bf16 tables; the
    pages do not print the codebook width), semantic + acoustic projections -> [4][512][768] fp32."""
    import torch
    from tests.gpu_util import dev_bf16_bits, dev_i32
    K, N, D, OUT = 16, 2048, 256, 512
    r = synth.rng_for(7, "quant_tables")
    books = [dev_bf16_bits(synth.normal_bf16(r, (N, D), 1.0)) for _ in range(K)]
    ps = dev_bf16_bits(synth.normal_bf16(r, (OUT, D), 0.02))
    pa = dev_bf16_bits(synth.normal_bf16(r, (OUT, D), 0.02))
    q = m.tts_bb_quantizer_create(books, ps, pa, stream.cuda_stream)
    codes = dev_i32(synth.rng_for(7, "quant_codes").integers(0, N, (B, K, T)))
    out = torch.zeros(B, OUT, T, dtype=torch.float32, device="cuda")
    for _ in range(3):
        m.tts_bb_quantizer_decode(q, B, T, codes, out)
    st = m.tts_bb_quantizer_sync(q)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(reps):
        m.tts_bb_quantizer_decode(q, B, T, codes, out)
    ev1.record(stream)
    torch.cuda.synchronize()
    m.tts_bb_quantizer_free(q)
    us = ev0.elapsed_time(ev1) / reps * 1e3
    kp = (3 * D + 255) // 256 * 256
    # codes read, 16 gathered rows per frame, packed rows written and read back, packed weights, output
    nbytes = B * K * T * 4 + B * T * K * D * 2 + 2 * B * T * kp * 2 + OUT * kp * 2 + B * T * OUT * 4
    return {"workload": f"Qwen3-TTS quantizer lookup: {B} x {T} frames x {K} codebooks ({N} x {D}) -> {OUT} channels fp32",
            "us_per_decode": us, "frames_per_s": B * T / (us / 1e6), "status": st,
            "algorithmic_bytes": nbytes, "hbm_frac_of_measured": nbytes / (us / 1e6) / 1e9 / peaks()[0]["hbm_gbs"]}


def dac_flops_per_frame():
    """FMA work of the DAC decoder per 25 Hz frame (2 flops per multiply-add)."""
    ch, ratios = (1024, 512, 256, 128, 64, 32), (8, 5, 4, 2, 3)
    f = 2 * 1024 * 256 + 2 * 256 * 1024 * 7
    s = 1
    for i, r in enumerate(ratios):
        s *= r
        ic, oc = ch[i], ch[i + 1]
        f += s * (2 * ic * oc * 2 + 3 * (2 * oc * oc * 7 + 2 * oc * oc))
    return f + 960 * 2 * 32 * 7


def run_dac_decode(m, stream, B=4, T=768, reps=3):
    """DAC decode of RVQ features: 4 items x 768 frames (30.7 s of 24 kHz audio each), seeded fp32
    weights scaled by fan-in."""
    import math
    import torch
    rng = np.random.default_rng(7)

    def f(*shape, std):
        return torch.from_numpy(rng.normal(0, std, shape).astype(np.float32)).cuda()

    def u(n):
        return torch.from_numpy(rng.uniform(0.5, 1.5, n).astype(np.float32)).cuda()

    ch, ratios = (1024, 512, 256, 128, 64, 32), (8, 5, 4, 2, 3)
    w = {"fc2_w": f(256, 1024, std=1 / 32), "fc2_b": f(256, std=0.05), "conv1_w": f(1024, 256, 7, std=1 / math.sqrt(1792)),
         "conv1_b": f(1024, std=0.05), "final_alpha": u(32), "conv2_w": f(1, 32, 7, std=1 / math.sqrt(224)),
         "conv2_b": f(1, std=0.05), "blocks": []}
    for i, r in enumerate(ratios):
        ic, oc = ch[i], ch[i + 1]
        w["blocks"].append({"alpha": u(ic), "up_w": f(ic, oc, 2 * r, std=1 / math.sqrt(2 * ic)), "up_b": f(oc, std=0.05),
                            "res": [{"alpha1": u(oc), "w1": f(oc, oc, 7, std=0.5 / math.sqrt(7 * oc)), "b1": f(oc, std=0.05),
                                     "alpha2": u(oc), "w2": f(oc, oc, 1, std=0.5 / math.sqrt(oc)), "b2": f(oc, std=0.05)}
                                    for _ in range(3)]})
    d = m.tts_bb_dac_create(w, stream.cuda_stream)
    feat = torch.from_numpy(rng.normal(0, 1, (B, T, 1024)).astype(np.float32)).cuda()
    audio = torch.zeros(B, 960 * T, dtype=torch.float32, device="cuda")
    m.tts_bb_dac_decode(d, B, T, feat, audio)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(reps):
        m.tts_bb_dac_decode(d, B, T, feat, audio)
    ev1.record(stream)
    torch.cuda.synchronize()
    finite = bool(torch.isfinite(audio).all().item())
    m.tts_bb_dac_free(d)
    ms = ev0.elapsed_time(ev1) / reps
    flops = dac_flops_per_frame() * B * T
    tf = flops / (ms / 1e3) / 1e12
    # every convolution but conv2 (32 -> 1, on the CUDA cores) runs on the tensor cores as three bf16
    # products per fp32 multiply-add (high x high, high x low, low x high)
    conv2 = 960 * 2 * 32 * 7 * B * T
    tensor_flops = 3 * (flops - conv2)
    pk, src = peaks()
    peak = pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    ach = tensor_flops / (ms / 1e3) / 1e12
    return {"workload": f"DAC decode: {B} items x {T} frames -> {B} x {960 * T} samples (24 kHz), fp32 weights and "
                        "activations (tensor cores: bf16 high + low parts, fp32 accumulation)",
            "ms_per_decode": ms, "audio_s_per_s": B * T / 25.0 / (ms / 1e3), "finite": finite,
            "fp32_equivalent_tflops": tf,
            "roofline": {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                         "peak_source": f"{src} bf16_tflops_sustained", "flop_per_decode": flops,
                         "tensor_flop_per_decode": tensor_flops}}


def run_dac(steps, warmup):
    """The DAC decode alone (4 items x 768 frames); steps decodes timed after warmup."""
    import torch
    import codec_token_tts_gb300 as m
    torch.cuda.set_stream(torch.cuda.Stream())
    return run_dac_decode(m, torch.cuda.current_stream(), reps=max(1, steps))


def run_prefill(steps, warmup, B=16, S=2048):
    """Batched causal prefill on the 28-layer Talker-shaped model: B sequences of S positions from
    position 0 (bf16 N(0, 1) input rows); one step = one prefill call over all B x S tokens."""
    import torch
    import codec_token_tts_gb300 as m
    from tests.gpu_util import dev_bf16_bits
    wl = TalkerB1()
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    h = make_engine(wl, m, stream.cuda_stream, S, B, B * S, B)
    x = dev_bf16_bits(synth.normal_bf16(synth.rng_for(11, "prefill_rows"), (B, S, 1024), 1.0))
    slots = list(range(B))

    def one():
        m.tts_bb_prefill(h, B, S, slots, [S] * B, embeds=x)
        for sl in slots:
            m.tts_bb_release(h, sl)

    for _ in range(warmup):
        one()
    m.tts_bb_sync(h)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(steps):
        one()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    m.tts_bb_profile(h, True)
    one()
    rep = m.tts_bb_profile_report(h)
    m.tts_bb_profile(h, False)
    st = m.tts_bb_sync(h)
    m.tts_bb_free(h)
    ks = {k["kind"]: k for k in rep["kernels"]}
    tot = sum(k["ms"] for k in rep["kernels"])
    pk, _ = peaks()
    att = ks.get("attn_causal_tcgen05") or ks.get("attn_prefill")
    out = {"metric": "prefill tokens/s (28 layers, causal)", "workload": f"prefill: {B} sequences x {S} positions, "
           "28-layer Talker-shaped model, bf16 N(0,1) input rows", "value": B * S / (ms / 1e3), "unit": "tokens/s",
           "ms_per_prefill": ms, "status": st,
           "kernel_share": {k: round(v["ms"] / tot, 4) for k, v in ks.items()}}
    if att:
        tf = att["flops"] / (att["ms"] / 1e3) / 1e12
        out["attention"] = {"kind": att["kind"], "ms": att["ms"], "tflops": tf,
                            "frac_of_measured_sustained": tf / pk["bf16_tflops_sustained"]}
    return out


def run_maskgit_refinement(m, h, seed, stream, n_step=32):
    """32 greedy refinement steps (pass + device update) of 4 items with CFG: rows 0-3 hold the
    conditional prompts (256 text + 768 masked target frames), rows 4-7 the unconditional ones
    (the 768 target frames alone, left-aligned, key_lens 768). Logits over all 1024 positions;
    the update reads positions 256.. of the conditional rows and 0.. of the unconditional ones."""
    import torch
    from tests.gpu_util import dev_i32, dev_u8
    n_items, S, n_text, V = 4, 1024, 256, 1025
    T = S - n_text
    ids0, mask0 = synth.maskgit_inputs(seed, 99)
    ids0, mask0 = ids0.copy(), mask0.copy()
    for i in range(n_items):
        ids0[i, :, n_text:] = 1024
        ids0[n_items + i, :, :T] = 1024
        ids0[n_items + i, :, T:] = 0
        mask0[n_items + i, :T] = 1
        mask0[n_items + i, T:] = 0
    key_lens = [S] * n_items + [T] * n_items
    counts = [int(c) for c in m.tts_bb_maskgit_schedule(n_step, 8 * T, 0.1)]
    init = dev_i32(ids0)
    ids_d = init.clone()
    mask_d = dev_u8(mask0)
    logits = torch.zeros(2 * n_items, 8, S, V, dtype=torch.float32, device="cuda")

    def refine():
        ids_d.copy_(init)
        for n in counts:
            m.tts_bb_maskgit_pass(h, 2 * n_items, S, ids_d, mask_d, key_lens, 0, logits, check=False)
            m.tts_bb_maskgit_update(h, n_items, T, logits, S, n_text, 0, ids_d, S, n_text, 0, n, check=False)

    refine()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    refine()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    done = not bool((ids_d[:n_items, :, n_text:] == 1024).any().item())
    m.tts_bb_profile(h, True)
    refine()
    rep = m.tts_bb_profile_report(h)
    m.tts_bb_profile(h, False)
    upd = [k for k in rep["kernels"] if k["kind"] == "maskgit_update"]
    out = {"workload": f"{n_step}-step greedy MaskGIT refinement, 4 items x (cond + uncond) = 8 rows x 1024, "
                       f"768 x 8 target cells per item, schedule shift 0.1",
           "ms_per_refinement": ms, "ms_per_step": ms / n_step, "all_cells_unmasked": done}
    if upd:
        u = upd[0]
        per = u["ms"] / n_step * 1e3
        gbs = u["bytes"] / (u["ms"] / 1e3) / 1e9
        out["update_us_per_step"] = per
        out["update_roofline"] = {"kernel": "maskgit_update", "bound": "hbm", "achieved": gbs,
                                  "peak": peaks()[0]["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks()[0]["hbm_gbs"],
                                  "bytes_per_step": u["bytes"] / n_step}
    return out


def run_code_predictor(steps, warmup):
    """Code Predictor, 256 frames at once: a 2-token prefill (Talker hidden state + code 0, head 0)
    then 14 decode calls with heads 1..14; one step = the 15 codes of every frame."""
    import torch
    import codec_token_tts_gb300 as m
    from tests.gpu_util import config_for, dev_bf16_bits, dev_i32, weights_for
    seed, F = 3, 256
    w = synth.model_weights(synth.CODE_PREDICTOR, seed)
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    cfg = config_for(synth.CODE_PREDICTOR, max_slots=F, max_ctx=17, max_batch=F, max_tokens=2 * F, sync_errors=0)
    h = m.tts_bb_create(cfg, weights_for(w), stream.cuda_stream)
    r = synth.rng_for(seed, "cp_inputs")
    th = synth.normal_bf16(r, (F, 1024), 1.0)
    code0 = r.integers(0, 3072, size=F).astype(np.int32)
    emb = np.zeros((F, 2, 1024), np.uint16)
    emb[:, 0] = th
    ids = -np.ones((F, 2, 16), np.int32)
    ids[:, 1, 0] = code0
    emb_d, ids_d = dev_bf16_bits(emb), dev_i32(ids)
    codes = torch.full((F, 16), -1, dtype=torch.int32, device="cuda")
    # step ids: column j carries code j (written by the previous call's argmax), -1 elsewhere
    steps_ids = torch.full((15, F, 16), -1, dtype=torch.int32, device="cuda")
    logits = torch.zeros(F, 2048, dtype=torch.float32, device="cuda")
    slots = np.arange(F, dtype=np.int32)

    def frame_batch():
        m.tts_bb_prefill(h, F, 2, slots, [2] * F, ids_d, 0, None, steps_ids[1, :, 1], embeds=emb_d,
                         argmax_stride=16, check=False)
        for j in range(1, 15):
            nxt = steps_ids[j + 1, :, j + 1] if j + 1 < 15 else codes[:, 15]
            m.tts_bb_decode_step(h, F, slots, [j + 1] * F, steps_ids[j], j, None, nxt, argmax_stride=16, check=False)
        for s in slots:
            m.lib.tts_bb_release(h, int(s))

    for _ in range(warmup):
        frame_batch()
    m.tts_bb_sync(h)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(steps):
        frame_batch()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    st = m.tts_bb_sync(h, check=False)
    m.tts_bb_profile(h, True)
    frame_batch()
    rep = m.tts_bb_profile_report(h)
    m.tts_bb_profile(h, False)
    m.tts_bb_free(h)
    # per call: 5 layers + final norm + one 2048 x 1024 head; KV read 20,480 B per cached token per frame
    per_call = 5 * 31_461_888 + 2048 + 2048 * 1024 * 2
    kv = sum(20_480 * F * (j + 1) for j in range(1, 15))
    step_bytes = 15 * per_call + kv + F * 2 * 2048 * 2
    return {"workload": "code_predictor: 5-layer Code Predictor, 256 frames at once, 2-token prefill + 14 decode "
                        "calls (heads 0..14), greedy codes fed back",
            "value": F * 15 / (ms / 1e3), "unit": "codebook tokens/s", "ms_per_step": ms, "steps": steps,
            "status": st, "algorithmic_bytes_per_step": step_bytes,
            "hbm_frac_of_measured": step_bytes / (ms / 1e3) / 1e9 / peaks()[0]["hbm_gbs"],
            "roofline": roofline_from_profile(rep), "kernel_profile": rep}


def run_frame_loop(n_frames, warmup, B=1):
    """Talker -> Code Predictor frame loop (tts_bb_frame_step), B streams: a 128-position Talker
    prefill, then frames at positions 128.. (rewinding every 256 frames); one frame = the Talker
    step (code 0) + the Code Predictor's 2-token prefill and 14 decode calls (codes 1..15)."""
    import torch
    import codec_token_tts_gb300 as m
    from tests.gpu_util import config_for, dev_i32, weights_for
    wt = synth.model_weights(synth.TALKER, 1)
    wc = synth.model_weights(synth.CODE_PREDICTOR, 3)
    wc.codebooks = wt.codebooks  # the Code Predictor embeds with the Talker's tables
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    ht = m.tts_bb_create(config_for(synth.TALKER, max_slots=B, max_ctx=P_PREFILL + N_DECODE, max_batch=B,
                                    max_tokens=B * P_PREFILL, sync_errors=0), weights_for(wt), stream.cuda_stream)
    hc = m.tts_bb_create(config_for(synth.CODE_PREDICTOR, max_slots=B, max_ctx=17, max_batch=B, max_tokens=2 * B,
                                    sync_errors=0), weights_for(wc), stream.cuda_stream)
    pre = np.stack([synth.talker_prefill_ids(1 + b, P_PREFILL + 1) for b in range(B)])
    m.tts_bb_prefill(ht, B, P_PREFILL, list(range(B)), [P_PREFILL] * B, dev_i32(pre[:, :P_PREFILL]), -1, None, None)
    first = dev_i32(pre[:, P_PREFILL])
    codes = first.clone()
    slots = np.arange(B, dtype=np.int32)
    kv = np.zeros(B, np.int32)

    def frames(n):
        for t in range(n):
            pos = P_PREFILL + (t % N_DECODE)
            if pos == P_PREFILL:
                for b in range(B):
                    m.tts_bb_truncate(ht, b, P_PREFILL)
                codes.copy_(first)
            kv[:] = pos
            m.lib.tts_bb_frame_step(ht, hc, B, slots.ctypes.data, kv.ctypes.data, codes.data_ptr(), None)

    frames(warmup)
    m.tts_bb_sync(ht)
    m.tts_bb_sync(hc)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    frames(n_frames)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / n_frames
    st = max(abs(m.tts_bb_sync(ht, check=False)), abs(m.tts_bb_sync(hc, check=False)))
    m.tts_bb_free(hc)
    m.tts_bb_free(ht)
    # per frame: Talker weights + head + 16 embedding rows + KV read; 15 Code Predictor calls of
    # 5 layers + one 2048-row head + their KV; position ~ the mean of 128..383
    talker = 28 * 31_461_888 + 3072 * 1024 * 2 + 16 * 2048 + 2048 + 114_688 * (P_PREFILL + N_DECODE // 2)
    cp = 15 * (5 * 31_461_888 + 2048 * 1024 * 2 + 2048 + 2048) + sum(20_480 * (j + 2) for j in range(15))
    frame_bytes = talker + cp
    return {"workload": f"frame_loop: Talker (28 layers) -> Code Predictor (5 layers, 15 codes) per frame, batch {B}, "
                        f"positions 128..383, greedy codes fed back",
            "value": B * 16 / (ms / 1e3), "unit": "codec tokens/s", "frames_per_s": B / (ms / 1e3),
            "ms_per_frame": ms, "frames": n_frames, "status": st, "algorithmic_bytes_per_frame": frame_bytes,
            "hbm_frac_of_measured": frame_bytes / (ms / 1e3) / 1e9 / peaks()[0]["hbm_gbs"]}


def roofline_from_profile(rep, traffic=None):
    pk, src = peaks()
    ks = rep.get("kernels", [])
    if not ks:
        return None
    top = max(ks, key=lambda k: k["ms"])
    total = sum(k["ms"] for k in ks)
    if top["flops"] and (not top["bytes"] or top["flops"] / max(top["bytes"], 1) > 300):
        ach = top["flops"] / (top["ms"] / 1e3) / 1e12
        peak = pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
        return {"kernel": top["kind"], "bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "traffic": traffic, "peak_source": f"{src} bf16_tflops_sustained",
                "share": top["ms"] / total, "launches": top["launches"]}
    ach = top["bytes"] / (top["ms"] / 1e3) / 1e9
    peak = pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    return {"kernel": top["kind"], "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
            "frac": ach / peak, "frac_of_8tbs": ach / 8000.0, "traffic": traffic, "peak_source": f"{src} hbm_gbs",
            "bytes_per_launch": top["bytes"] / top["launches"], "share": top["ms"] / total,
            "launches": top["launches"]}


# DRAM bytes (read + write) per launch of a kernel, from an ncu capture of this bench's own
# command (dram__bytes_read.sum + dram__bytes_write.sum of a launch after the warm-up steps).
# Valid only while the kernel's sources are the ones that were captured: the sha256 of the listed
# files must match, else the bench reports null.
MEASURED_TRAFFIC = {
    "decode_step_persistent": {"files": ("k_decode_ll.cu", "mega.cuh", "common.cuh"),
                               "sha256": "8b5a376aaaf62ac89fbb081117af10549ecb7b4b6fcc61fbfe8978535806c71e",
                               "bytes_per_launch": 926.255616e6},
}


def measured_traffic(rep):
    """DRAM bytes per launch of the dominant kernel from a capture of its current sources, or None."""
    import hashlib
    ks = rep.get("kernels", [])
    if not ks:
        return None
    rec = MEASURED_TRAFFIC.get(max(ks, key=lambda k: k["ms"])["kind"])
    if rec is None:
        return None
    h = hashlib.sha256()
    for f in rec["files"]:
        with open(os.path.join(ROOT, "codec_token_tts_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return rec["bytes_per_launch"] if h.hexdigest() == rec["sha256"] else None


# ---------------------------------------------------------------- oracle timing (CPU baseline / reference arm)
def oracle_talker_tokens_per_s(budget_s: float, max_steps: int):
    """Time the fp64 oracle on decode steps of the talker_b1 workload (positions 128..)."""
    import oracle as O
    wl = TalkerB1()
    t_setup = time.perf_counter()
    mo = O.Backbone(wl.w, wl.shape)
    cache = mo.new_cache()
    _, _, a0 = O.talker_prefill(mo, wl.prefill_ids, cache)
    setup_s = time.perf_counter() - t_setup
    n = 0
    t0 = time.perf_counter()
    id0 = a0
    max_steps = min(max_steps, len(wl.rest))  # the workload's decode positions (128..383)
    while n < max_steps and (time.perf_counter() - t0) < budget_s:
        _, _, am, _ = O.talker_decode_steps(mo, cache, id0, wl.rest[n:n + 1])
        id0 = int(am[0])
        n += 1
    el = time.perf_counter() - t0
    return n / el, n, el, setup_s


def cpu_info():
    return {"cores": os.cpu_count(), "blas_threads": os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get(
        "OMP_NUM_THREADS") or "default (all cores)"}


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    budget = float(os.environ.get("TTS_BB_REF_BUDGET_S", "120"))
    _ = oracle_talker_tokens_per_s(5.0, max(1, args.warmup)) if args.warmup else None
    v, n, el, setup_s = oracle_talker_tokens_per_s(budget, args.steps)
    ci = cpu_info()
    wl_cfg = {"workload": "talker_b1: Qwen3-0.6B-shaped Talker, 28 layers, batch 1, 128-position prefill then "
                          "decode at positions 128..383, 3072-way head, greedy id0 fed back",
              "global_batch": 1, "seq_len": P_PREFILL + N_DECODE, "layers": 28}
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws, "steps": n,
            "steps_requested": args.steps, "warmup": args.warmup, "ms_per_step": el / n * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": wl_cfg,
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": ci["cores"], "kind": "oracle",
                             "sample": f"{n} decode steps from position 128 after the oracle's 128-position prefill "
                                       f"({setup_s:.1f} s untimed setup), {ci['blas_threads']} BLAS threads"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2048)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="talker_b1", choices=["talker_b1"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=20.0)
    ap.add_argument("--no-secondary", action="store_true", help="skip the batch-64 serving, MaskGIT and Code Predictor lines")
    ap.add_argument("--prefill-batch", type=int, default=16, help="sequences of the --only prefill workload")
    ap.add_argument("--only", choices=["serving_b64", "maskgit", "code_predictor", "frame_loop", "dac", "prefill"],
                    help="run one secondary workload alone (--steps / --warmup apply) and print its line; a profiling aid")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.only:
        import torch
        from tests.gpu_util import build_lib
        torch.cuda.set_device(0)
        build_lib()
        fn = {"serving_b64": run_serving_b64, "maskgit": run_maskgit, "code_predictor": run_code_predictor,
              "frame_loop": run_frame_loop, "dac": run_dac, "prefill": run_prefill}[args.only]
        r = fn(args.steps, args.warmup, B=args.prefill_batch) if args.only == "prefill" else fn(args.steps, args.warmup)
        print(json.dumps({k: v for k, v in r.items() if k != "kernel_profile"}), flush=True)
        return

    if args.impl == "reference":
        ws, rank, _ = dist_setup("gloo")
        res = run_reference(args, ws, rank)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return

    import torch
    ws, rank, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    from tests.gpu_util import build_lib
    build_lib()
    res, wl = run_talker_b1(args, ws, rank)
    res["roofline"] = roofline_from_profile(res["kernel_profile"], measured_traffic(res["kernel_profile"]))
    if not args.no_secondary:
        sv = run_serving_b64(64, 4)
        # the batch-64 half of the metric at the top level of the line (the "also" block holds the details)
        res["batch64"] = {"value": sv["value"], "unit": sv["unit"], "ms_per_step": sv["ms_per_step"],
                          "workload": sv["workload"], "roofline": sv.get("roofline")}
        res["also"] = {"serving_b64": {k: v for k, v in sv.items() if k != "kernel_profile"},
                       "maskgit": run_maskgit(8, 3), "code_predictor": run_code_predictor(16, 3),
                       "frame_loop": run_frame_loop(64, 4)}
    if rank == 0 and not args.no_cpu_baseline:
        v, n, el, setup_s = oracle_talker_tokens_per_s(args.cpu_budget_s, 10_000)
        ci = cpu_info()
        res["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": ci["cores"], "kind": "oracle",
                               "sample": f"{n} Talker decode steps from position 128 in {el:.1f} s after an untimed "
                                         f"128-position prefill ({setup_s:.1f} s), {ci['blas_threads']} BLAS threads"}
    if rank == 0:
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
