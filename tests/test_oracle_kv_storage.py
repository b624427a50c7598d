"""The oracle's bf16 KV-storage option (CPU only).

The GPU path stores keys and values in bf16, the format its specification
fixes; the oracle keeps its cache in float64 unless asked to store it the
same way. Pins: bf16 rounding by hand-worked cases (ties to even at the 8th
significant bit) and against the input generator's own rounding; with bf16
storage every cached value is a bf16 number and nothing else changes; on a
small Talker-shaped model the storage moves the logits by far less than the
logits tolerance and can flip a greedy pick only where the float64 oracle's
top two logits lie within that tolerance.
"""
import numpy as np

import oracle as O
import synth
from tests.gpu_util import LOGIT_TOL


def test_round_bf16_hand_cases():
    u = 2.0 ** -7                    # bf16 spacing just above 1.0
    cases = [(1.0, 1.0), (1.0 + u / 2, 1.0),            # tie -> even (1.0)
             (1.0 + 1.5 * u, 1.0 + 2 * u),              # tie -> even (1 + 2u)
             (1.0 + 0.51 * u, 1.0 + u), (-3.0 - 0.49 * u * 2, -3.0),
             (0.0, 0.0), (2.0 ** -130, 2.0 ** -130)]    # a float32 subnormal that bf16 holds exactly
    for x, want in cases:
        assert O.round_bf16(np.array([x]))[0] == want, x


def test_round_bf16_matches_the_input_generator():
    x = np.random.default_rng(5).normal(0, 3, 4096).astype(np.float32)
    x[:16] = np.float32(1.0) + np.float32(2.0 ** -8) * np.arange(16, dtype=np.float32)  # ties and near-ties
    assert np.array_equal(O.round_bf16(x), O.bf16_to_f64(synth.bf16_bits(x)))


SHAPE = synth.ModelShape(n_layers=4, codebook_rows=(3072,) + (2048,) * 15, n_heads_out=1, head_rows=3072)


def test_bf16_kv_storage_moves_logits_within_tolerance_and_flips_only_near_ties():
    w = synth.model_weights(SHAPE, 61)
    ids = synth.talker_prefill_ids(61, 24)
    rest = synth.uniform_ids(synth.rng_for(61, "rest"), SHAPE.codebook_rows[1:], 48)
    out = {}
    fed0 = None
    for mode in (None, "bf16"):
        m = O.Backbone(w, SHAPE, kv_storage=mode)
        cache = m.new_cache()
        _, _, a0 = O.talker_prefill(m, ids, cache)
        _, lg, am, fed = O.talker_decode_steps(m, cache, int(np.asarray(a0).reshape(-1)[0]), rest, forced_id0=fed0)
        if fed0 is None:
            fed0 = fed[:, 0]
        if mode == "bf16":                       # every cached value is a bf16 number
            for l in range(SHAPE.n_layers):
                assert np.array_equal(cache.k[l], O.round_bf16(cache.k[l]))
                assert np.array_equal(cache.v[l], O.round_bf16(cache.v[l]))
        out[mode] = (lg, am)
    (l64, a64), (lb, ab) = out[None], out["bf16"]
    diff = np.abs(lb - l64)
    assert 0.0 < diff.max() <= LOGIT_TOL / 3
    top2 = np.sort(l64, axis=1)[:, -2:]
    gap = top2[:, 1] - top2[:, 0]
    assert np.all(gap[a64 != ab] <= LOGIT_TOL)  # any flip sits at a near-tie
