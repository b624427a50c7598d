"""GPU parity of the Talker -> Code Predictor frame loop (tts_bb_frame_step).

The oracle replays the GPU's codes (teacher forcing), so both see the same
inputs every frame. Talker logits are compared within the logits tolerance
and code 0 under the argmax rule of the other tests. The Code Predictor's
logits stay on the device, so its 15 codes are checked against the oracle's
logits: where the oracle's best id leads by more than the logits tolerance
the codes must agree, elsewhere the GPU's code must be within the tolerance
of the oracle's maximum.
"""
import numpy as np
import pytest

import oracle as O
import synth
from tests.gpu_util import ARGMAX_AGREE, LOGIT_TOL, Engine, check_logits_and_argmax, dev_i32, f32_zeros

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _models(seed, cp_layers=2):
    ts = synth.ModelShape(n_layers=2, codebook_rows=(3072,) + (2048,) * 15, n_heads_out=1, head_rows=3072)
    cs = synth.ModelShape(n_layers=cp_layers, codebook_rows=(3072,) + (2048,) * 15, n_heads_out=15, head_rows=2048)
    wt = synth.model_weights(ts, seed)
    wc = synth.model_weights(cs, seed + 1)
    wc.codebooks = wt.codebooks  # talker-wide embeddings
    return wt, wc


def _check_cp_codes(g_codes, o_logits):
    """g_codes[15]; o_logits[15, 2048]."""
    for j in range(15):
        lg = o_logits[j]
        best = int(np.argmax(lg))
        top2 = np.sort(lg)[-2:]
        if top2[1] - top2[0] > LOGIT_TOL:
            assert g_codes[j] == best, (j, g_codes[j], best)
        else:
            assert lg[best] - lg[g_codes[j]] <= LOGIT_TOL, (j, g_codes[j], best)


@pytest.mark.parametrize("B", [1, 3])
def test_frame_loop_matches_oracle(B):
    wt, wc = _models(51)
    P, n_frames = 16, 3
    r = synth.rng_for(51, "frames")
    prompt = [synth.uniform_ids(r, (3072,) + (2048,) * 15, P + 1) for _ in range(B)]
    with Engine(wt, max_slots=B, max_ctx=64, max_batch=B, max_tokens=B * P) as et, \
            Engine(wc, max_slots=B, max_ctx=17, max_batch=B, max_tokens=2 * B) as ec:
        m = et.m
        m.tts_bb_prefill(et.h, B, P, list(range(B)), [P] * B, dev_i32(np.stack([p[:P] for p in prompt])))
        codes = dev_i32(np.stack([p[P] for p in prompt]))
        logits = f32_zeros(B, 3072)
        got_codes, got_logits = [], []
        for f in range(n_frames):
            m.tts_bb_frame_step(et.h, ec.h, B, list(range(B)), [P + f] * B, codes, logits)
            got_codes.append(codes.cpu().numpy().copy())
            got_logits.append(logits.cpu().numpy().copy())
        assert [m.tts_bb_slot_len(et.h, b) for b in range(B)] == [P + n_frames] * B
        assert [m.tts_bb_slot_len(ec.h, b) for b in range(B)] == [0] * B
    got_codes = np.array(got_codes)    # [frames, B, 16]
    got_logits = np.array(got_logits)  # [frames, B, 3072]
    talker, cp = O.Backbone(wt, wt.shape), O.Backbone(wc, wc.shape)
    for b in range(B):
        cache = talker.new_cache()
        O.talker_prefill(talker, prompt[b][:P], cache)
        o_codes, t_lg, c_lg, _ = O.talker_cp_frames(talker, cp, cache, prompt[b][P], n_frames,
                                                    forced=got_codes[:, b])
        check_logits_and_argmax(got_logits[:, b], t_lg, got_codes[:, b, 0], o_codes[:, 0], min_agree=ARGMAX_AGREE)
        for f in range(n_frames):
            _check_cp_codes(got_codes[f, b, 1:], c_lg[f])
        assert np.all(got_codes[:, b, 0] < 3072) and np.all(got_codes[:, b, 1:] < 2048)


def test_frame_step_rejects_mismatched_handles():
    wt, wc = _models(52)
    with Engine(wt, max_slots=2, max_ctx=64, max_batch=2, max_tokens=32) as et, \
            Engine(wc, max_slots=1, max_ctx=17, max_batch=1, max_tokens=2) as ec:
        m = et.m
        codes = dev_i32(np.zeros((2, 16), np.int32))
        # two streams in the Code Predictor handle's slots do not fit
        assert m.tts_bb_frame_step(et.h, ec.h, 2, [0, 1], [0, 0], codes, check=False) == m.E_INVALID
        # a Talker used as the Code Predictor lacks the 15 heads
        assert m.tts_bb_frame_step(et.h, et.h, 1, [0], [0], codes, check=False) == m.E_INVALID


def test_frame_loop_full_size():
    """The bench's frame loop: 28-layer Talker (3072-row E_0 and head) and 5-layer Code Predictor,
    batch 1, a 128-position prefill then 2 frames, against the teacher-forced oracle."""
    wt = synth.model_weights(synth.TALKER, 1)
    wc = synth.model_weights(synth.CODE_PREDICTOR, 3)
    wc.codebooks = wt.codebooks
    P, n_frames = 128, 2
    pre = synth.talker_prefill_ids(1, P + 1)
    with Engine(wt, max_slots=1, max_ctx=P + 8, max_batch=1, max_tokens=P) as et, \
            Engine(wc, max_slots=1, max_ctx=17, max_batch=1, max_tokens=2) as ec:
        m = et.m
        m.tts_bb_prefill(et.h, 1, P, [0], [P], dev_i32(pre[None, :P]))
        codes = dev_i32(pre[None, P])
        logits = f32_zeros(1, 3072)
        got_codes, got_logits = [], []
        for f in range(n_frames):
            m.tts_bb_frame_step(et.h, ec.h, 1, [0], [P + f], codes, logits)
            got_codes.append(codes.cpu().numpy()[0].copy())
            got_logits.append(logits.cpu().numpy()[0].copy())
    got_codes, got_logits = np.array(got_codes), np.array(got_logits)
    talker, cp = O.Backbone(wt, wt.shape), O.Backbone(wc, wc.shape)
    cache = talker.new_cache()
    O.talker_prefill(talker, pre[:P], cache)
    o_codes, t_lg, c_lg, _ = O.talker_cp_frames(talker, cp, cache, pre[P], n_frames, forced=got_codes)
    check_logits_and_argmax(got_logits, t_lg, got_codes[:, 0], o_codes[:, 0], min_agree=ARGMAX_AGREE)
    for f in range(n_frames):
        _check_cp_codes(got_codes[f, 1:], c_lg[f])
