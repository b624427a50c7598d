"""GPU parity of the DAC decoder (tts_bb_dac_decode) with the fp64 oracle.

The decoder keeps weights and activations in fp32; the oracle computes in
fp64 from the same fp32 weights. Two paths: the tensor-core convolutions
(default: conv1 and every block convolution as implicit GEMMs on tcgen05 with
each fp32 operand split into bf16 high + low parts, so each product is exact
to ~2^-17 and sums accumulate in fp32) and the CUDA-core fp32 kernels
(TTS_BB_DAC=fp32 at create). Tolerance for both: max |gpu - oracle| /
max |oracle| at most 1e-4 over the whole waveform — rounding of ~2^-17 (split
operands) or 2^-24 (fp32) per product in sums of up to 1024 x 7 products
through 38 layers grows like sqrt(terms x layers) in the typical case, ~1e-5
relative here, with an order of magnitude of margin. Seeded weights are
scaled by their fan-in so activations stay O(1).
"""
import math
import os

import numpy as np
import pytest

import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def dac_weights(seed):
    r = np.random.default_rng(seed)
    f = lambda *shape, std: r.normal(0, std, shape).astype(np.float32)
    C = O.DAC_CHANNELS
    w = {"fc2_w": f(256, 1024, std=1 / 32), "fc2_b": f(256, std=0.05),
         "conv1_w": f(1024, 256, 7, std=1 / math.sqrt(256 * 7)), "conv1_b": f(1024, std=0.05), "blocks": [],
         "final_alpha": r.uniform(0.5, 1.5, 32).astype(np.float32), "conv2_w": f(1, 32, 7, std=1 / math.sqrt(32 * 7)),
         "conv2_b": f(1, std=0.05)}
    for i, ratio in enumerate(O.DAC_RATIOS):
        ic, oc = C[i], C[i + 1]
        res = [{"alpha1": r.uniform(0.5, 1.5, oc).astype(np.float32), "w1": f(oc, oc, 7, std=0.5 / math.sqrt(oc * 7)),
                "b1": f(oc, std=0.05), "alpha2": r.uniform(0.5, 1.5, oc).astype(np.float32),
                "w2": f(oc, oc, 1, std=0.5 / math.sqrt(oc)), "b2": f(oc, std=0.05)} for _ in range(3)]
        w["blocks"].append({"alpha": r.uniform(0.5, 1.5, ic).astype(np.float32),
                            "up_w": f(ic, oc, 2 * ratio, std=1 / math.sqrt(2 * ic)), "up_b": f(oc, std=0.05), "res": res})
    return w


def to_device(w):
    if isinstance(w, dict):
        return {k: to_device(v) for k, v in w.items()}
    if isinstance(w, list):
        return [to_device(v) for v in w]
    return torch.from_numpy(np.ascontiguousarray(w)).cuda()


@pytest.mark.parametrize("path", ["tensor", "fp32"])
@pytest.mark.parametrize("B,T", [(1, 1), (2, 5), (1, 7), (3, 130), (1, 768)])
def test_dac_matches_oracle(B, T, path):
    """(1, 768) is one item of the bench's decode: 30.7 s of audio, every sample compared;
    (3, 130) spans several row tiles with a ragged tail in every block, over three items."""
    import codec_token_tts_gb300 as m
    w = dac_weights(71)
    feat = np.random.default_rng(72).normal(0, 1, (B, T, 1024)).astype(np.float32)
    wd = to_device(w)
    if path == "fp32":
        os.environ["TTS_BB_DAC"] = "fp32"
    try:
        d = m.tts_bb_dac_create(wd, torch.cuda.current_stream().cuda_stream)
    finally:
        os.environ.pop("TTS_BB_DAC", None)
    try:
        audio = torch.full((B, 960 * T), float("nan"), dtype=torch.float32, device="cuda")
        m.tts_bb_dac_decode(d, B, T, torch.from_numpy(feat).cuda(), audio)
        assert m.tts_bb_dac_sync(d) == m.OK
        got = audio.cpu().numpy().astype(np.float64)
    finally:
        m.tts_bb_dac_free(d)
    ref = O.dac_decode(feat.astype(np.float64), w)[:, 0]
    assert ref.shape == (B, 960 * T)
    assert np.all(np.isfinite(got))
    err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert err <= 1e-4, err


def test_dac_rejects_bad_arguments():
    import codec_token_tts_gb300 as m
    d = m.tts_bb_dac_create(to_device(dac_weights(73)), torch.cuda.current_stream().cuda_stream)
    try:
        x = torch.zeros(1, 1, 1024, device="cuda")
        a = torch.zeros(1, 960, device="cuda")
        assert m.tts_bb_dac_decode(d, 0, 1, x, a, check=False) == m.E_INVALID
        assert m.tts_bb_dac_decode(d, 1, 0, x, a, check=False) == m.E_INVALID
        assert m.tts_bb_dac_decode(d, 1, 1, None, a, check=False) == m.E_INVALID
        # rejected on the host before anything is allocated or launched
        assert m.tts_bb_dac_decode(d, 65536, 1, x, a, check=False) == m.E_INVALID
        assert m.tts_bb_dac_decode(d, 1, 2_300_000, x, a, check=False) == m.E_INVALID
    finally:
        m.tts_bb_dac_free(d)
