"""GPU parity of the MaskGIT greedy update (tts_bb_maskgit_update) with the oracle.

Both sides read the same float32 logits. The predictions are integers decided
from z = c + s (c - u) formed in float32 with one rounding per operation on
both sides, so they must match exactly. The scores go through a log-sum-exp
(float32 on the GPU, float64 in the oracle), so the cells taken are compared
where the decision is unique: if the oracle's n-th and (n+1)-th best scores
are more than SCORE_TOL apart the taken sets must be equal; otherwise every
taken cell must be within SCORE_TOL of the boundary or above it, every cell
left masked within SCORE_TOL of it or below, and the count must be exact.
Windows, the unconditional mirror and the cells outside the windows are
checked bit for bit.
"""
import numpy as np
import pytest

import oracle as O
import synth
from tests.gpu_util import Engine, dev_u8, f32_zeros

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

MASK, V, K = 1024, 1025, 8
SCORE_TOL = 1e-4  # float32 log-sum-exp of ~1000 terms against float64
SHAPE = synth.ModelShape(n_layers=2, text_vocab=4096, audio_codebooks=8, audio_vocab=1025, n_heads_out=8,
                         head_rows=1025)


def _check_taken(taken_gpu, score, n_unmask):
    """taken_gpu [K, T] bool; score [K, T] oracle scores (-inf = not masked)."""
    flat = score.reshape(-1)
    tk = taken_gpu.reshape(-1)
    fin = np.isfinite(flat)
    n = min(n_unmask, int(fin.sum()))
    assert tk.sum() == n, (tk.sum(), n)
    assert not tk[~fin].any()
    if n == 0:
        return
    order = sorted(np.nonzero(fin)[0].tolist(), key=lambda i: (-flat[i], i))
    want = np.zeros_like(tk)
    want[order[:n]] = True
    bound = flat[order[n - 1]]
    nxt = flat[order[n]] if n < len(order) else -np.inf
    if bound - nxt > SCORE_TOL:
        assert np.array_equal(tk, want)
    else:
        assert np.all(flat[tk] >= bound - SCORE_TOL)
        assert np.all(flat[fin & ~tk] <= bound + SCORE_TOL)


def _run_case(e, logits, ids, n_items, T, S_log, cpos, upos, S_ids, cidp, uidp, n_unmask, cfg=2.0, pen=5.0):
    m = e.m
    lg = torch.from_numpy(logits).cuda()
    idd = torch.from_numpy(ids.astype(np.int32)).cuda()
    m.tts_bb_maskgit_update(e.h, n_items, T, lg, S_log, cpos, upos, idd, S_ids, cidp, uidp, n_unmask, cfg, pen)
    got = idd.cpu().numpy()
    cond = logits[:n_items, :, cpos:cpos + T]
    unc = logits[n_items:, :, upos:upos + T]
    tok = ids[:n_items, :, cidp:cidp + T]
    new, taken, pred, score = O.maskgit_update(cond, unc, tok, n_unmask, MASK, cfg, pen)
    for i in range(n_items):
        g_tok = got[i, :, cidp:cidp + T]
        was = tok[i] == MASK
        g_taken = was & (g_tok != MASK)
        # predictions of the taken cells are exact; untaken cells keep their ids
        assert np.array_equal(g_tok[g_taken], pred[i][g_taken])
        assert np.array_equal(g_tok[~g_taken], tok[i][~g_taken])
        _check_taken(g_taken, score[i], n_unmask)
        # the unconditional row mirrors the conditional one inside its window
        assert np.array_equal(got[n_items + i, :, uidp:uidp + T], np.where(g_taken, g_tok, ids[n_items + i, :, uidp:uidp + T]))
    # nothing outside the windows moves
    outside = np.ones(ids.shape, bool)
    outside[:n_items, :, cidp:cidp + T] = False
    outside[n_items:, :, uidp:uidp + T] = False
    assert np.array_equal(got[outside], ids[outside])
    return got


@pytest.fixture(scope="module")
def eng():
    w = synth.model_weights(SHAPE, 41)
    with Engine(w, max_slots=0, max_ctx=0, max_batch=4, max_tokens=4 * 200) as e:
        yield e


def _inputs(seed, n_items, T, S_log, S_ids, frac_unmasked=0.3, cpos=0, upos=0, cidp=0, uidp=0):
    r = synth.rng_for(seed, "mg_update")
    logits = r.normal(0, 2.0, (2 * n_items, K, S_log, V)).astype(np.float32)
    ids = r.integers(0, 1024, (2 * n_items, K, S_ids)).astype(np.int64)
    for i in range(n_items):
        m = r.random((K, T)) >= frac_unmasked
        win = ids[i, :, cidp:cidp + T]
        win[m] = MASK
        ids[n_items + i, :, uidp:uidp + T] = win  # the unconditional row holds the same target tokens
    return logits, ids


@pytest.mark.parametrize("n_unmask", [0, 1, 37, 500, 10_000])
def test_update_matches_oracle(eng, n_unmask):
    n_items, T, S_log, S_ids = 3, 200, 260, 300
    logits, ids = _inputs(7, n_items, T, S_log, S_ids, cpos=60, upos=0, cidp=100, uidp=10)
    _run_case(eng, logits, ids, n_items, T, S_log, 60, 0, S_ids, 100, 10, n_unmask)


def test_update_full_size(eng):
    """The shape the bench's refinement runs: 4 items x 8 codebooks x 768 target frames, logits over
    all 1024 positions (conditional window at 256, unconditional at 0), the largest step of the
    32-step schedule, 30 % of the cells already unmasked."""
    n_items, T, S = 4, 768, 1024
    n = int(O.maskgit_schedule(32, K * T, 0.1).max())
    logits, ids = _inputs(11, n_items, T, S, S, cpos=256, upos=0, cidp=256, uidp=0)
    _run_case(eng, logits, ids, n_items, T, S, 256, 0, S, 256, 0, n)


def test_update_ties_take_lowest_index(eng):
    """Equal logits everywhere: every masked cell of a codebook ties, so the
    lowest positions of codebook 0 go first (scores fall by 5 per codebook)."""
    n_items, T = 2, 50
    logits = np.full((2 * n_items, K, T, V), 0.5, np.float32)
    ids = np.full((2 * n_items, K, T), MASK, np.int64)
    ids[0, 0, 3] = 5
    got = _run_case(eng, logits, ids, n_items, T, T, 0, 0, T, 0, 0, 60)
    flat = got[0].reshape(-1)
    assert np.all(flat[:61][np.arange(61) != 3] == 0) and flat[3] == 5 and np.all(flat[61:] == MASK)


def test_update_all_unmasked_and_full_window(eng):
    n_items, T = 1, 64
    logits, ids = _inputs(8, n_items, T, T, T, frac_unmasked=1.0)
    _run_case(eng, logits, ids, n_items, T, T, 0, 0, T, 0, 0, 100)        # nothing masked: no change
    logits, ids = _inputs(9, n_items, T, T, T, frac_unmasked=0.0)
    _run_case(eng, logits, ids, n_items, T, T, 0, 0, T, 0, 0, K * T)      # every cell taken


def test_update_rejects_bad_windows(eng):
    m = eng.m
    lg = f32_zeros(2, K, 10, V)
    ids = torch.zeros(2, K, 10, dtype=torch.int32, device="cuda")
    for args in ((1, 10, lg, 10, 1, 0, ids, 10, 0, 0, 5), (1, 10, lg, 10, 0, 0, ids, 10, 0, 1, 5),
                 (0, 10, lg, 10, 0, 0, ids, 10, 0, 0, 5), (1, 10, lg, 10, 0, 0, ids, 10, 0, 0, -1),
                 # window starts whose end would wrap around a 32-bit int
                 (1, 10, lg, 10, 2**31 - 5, 0, ids, 10, 0, 0, 5), (1, 10, lg, 10, 0, 0, ids, 10, 0, 2**31 - 5, 5)):
        assert m.tts_bb_maskgit_update(eng.h, *args, check=False) == m.E_INVALID


def test_refinement_loop_on_pass_logits(eng):
    """Real pass logits: 2 items (cond rows 0-1, uncond rows 2-3 left-aligned,
    key_lens = T). Each step's update of the pass's own fp32 logits matches
    the oracle's update of the same logits, and the schedule drains every cell."""
    m = eng.m
    n_items, S, n_text = 2, 200, 72
    T = S - n_text
    ids, mask = synth.maskgit_inputs(41, 0, B=2 * n_items, S=S, n_text=n_text, text_vocab=4096)
    ids = ids.astype(np.int64)
    mask = mask.copy()
    for i in range(n_items):  # target window all masked; uncond rows: the T target tokens at [0, T)
        ids[i, :, n_text:] = MASK
        ids[n_items + i, :, :T] = MASK
        ids[n_items + i, :, T:] = 0
        mask[n_items + i, :T] = 1
        mask[n_items + i, T:] = 0
    key_lens = np.array([S] * n_items + [T] * n_items, np.int32)
    counts = m.tts_bb_maskgit_schedule(6, K * T, 0.1)
    assert np.array_equal(counts, O.maskgit_schedule(6, K * T, 0.1))
    idd = torch.from_numpy(ids.astype(np.int32)).cuda()
    logits = f32_zeros(2 * n_items, K, S, V)
    md = dev_u8(mask)
    for step, n in enumerate(counts):
        before = idd.cpu().numpy().astype(np.int64)
        m.tts_bb_maskgit_pass(eng.h, 2 * n_items, S, idd, md, key_lens, 0, logits)
        lg = logits.cpu().numpy()
        assert np.all(np.isfinite(lg))
        m.tts_bb_maskgit_update(eng.h, n_items, T, logits, S, n_text, 0, idd, S, n_text, 0, int(n))
        got = idd.cpu().numpy()
        new, taken, pred, score = O.maskgit_update(lg[:n_items, :, n_text:], lg[n_items:, :, :T],
                                                   before[:n_items, :, n_text:], int(n), MASK)
        for i in range(n_items):
            g_tok = got[i, :, n_text:]
            g_taken = (before[i, :, n_text:] == MASK) & (g_tok != MASK)
            assert np.array_equal(g_tok[g_taken], pred[i][g_taken])
            _check_taken(g_taken, score[i], int(n))
            assert np.array_equal(got[n_items + i, :, :T], g_tok)
    assert not np.any(idd.cpu().numpy()[:n_items, :, n_text:] == MASK)  # the schedule unmasked every cell
