"""GPU parity of the RVQ codec decode (tts_bb_rvq_decode) with the oracle.

Tables with small integer values make every product and sum exact in fp32,
so that case is compared bit for bit; seeded normal bf16 tables are compared
within fp32 accumulation error over K * dim = 512 terms. Both the GEMV path
(<= 8 frames) and the tcgen05 path (ragged last tile) are covered, and a code
outside the table is skipped and reported.
"""
import numpy as np
import pytest

import oracle as O
import synth
from tests.gpu_util import dev_bf16_bits, dev_i32, f32_zeros

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

K, N, D, OUT = 8, 1024, 64, 1024


def _tables(seed, integer):
    r = synth.rng_for(seed, "rvq")
    if integer:
        e = [synth.bf16_bits(r.integers(-8, 9, (N, D)).astype(np.float32)) for _ in range(K)]
        w = [synth.bf16_bits(r.integers(-8, 9, (OUT, D)).astype(np.float32)) for _ in range(K)]
        b = [synth.bf16_bits(r.integers(-50, 51, OUT).astype(np.float32)) for _ in range(K)]
    else:
        e = [synth.normal_bf16(r, (N, D), 1.0) for _ in range(K)]
        w = [synth.normal_bf16(r, (OUT, D), 0.05) for _ in range(K)]
        b = [synth.normal_bf16(r, (OUT,), 0.1) for _ in range(K)]
    return e, w, b


def _run(m, e, w, b, codes):
    ed, wd, bd = [dev_bf16_bits(x) for x in e], [dev_bf16_bits(x) for x in w], [dev_bf16_bits(x) for x in b]
    r = m.tts_bb_rvq_create(ed, wd, bd, torch.cuda.current_stream().cuda_stream)
    try:
        B, _, T = codes.shape
        out = f32_zeros(B, T, OUT)
        m.tts_bb_rvq_decode(r, B, T, dev_i32(codes), out)
        st = m.tts_bb_rvq_sync(r)
        return out.cpu().numpy().astype(np.float64), st
    finally:
        m.tts_bb_rvq_free(r)


@pytest.mark.parametrize("B,T", [(1, 5), (3, 257), (4, 768)])
def test_rvq_exact_on_integer_tables(B, T):
    """(4, 768) is the shape the bench times (a refinement's 4 items x 768 frames)."""
    import codec_token_tts_gb300 as m
    e, w, b = _tables(61, True)
    codes = synth.rng_for(61, f"codes{B}").integers(0, N, (B, K, T))
    got, st = _run(m, e, w, b, codes)
    assert st == m.OK
    ref = O.rvq_decode(codes, [O.bf16_to_f64(x) for x in e], [O.bf16_to_f64(x) for x in w],
                       [O.bf16_to_f64(x) for x in b])
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("B,T", [(2, 3), (4, 300)])
def test_rvq_matches_oracle_on_normal_tables(B, T):
    import codec_token_tts_gb300 as m
    e, w, b = _tables(62, False)
    codes = synth.rng_for(62, f"codes{B}").integers(0, N, (B, K, T))
    got, st = _run(m, e, w, b, codes)
    assert st == m.OK
    ref = O.rvq_decode(codes, [O.bf16_to_f64(x) for x in e], [O.bf16_to_f64(x) for x in w],
                       [O.bf16_to_f64(x) for x in b])
    err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert err < 1e-5, err


def test_rvq_bad_code_is_skipped_and_reported():
    import codec_token_tts_gb300 as m
    e, w, b = _tables(63, True)
    codes = synth.rng_for(63, "codes").integers(0, N, (1, K, 12))
    codes[0, 3, 7] = N  # out of the table
    got, st = _run(m, e, w, b, codes)
    assert st == m.E_BAD_ID
    ok = codes.copy()
    ok[0, 3, 7] = 0
    ef = [O.bf16_to_f64(x) for x in e]
    ref = O.rvq_decode(ok, ef, [O.bf16_to_f64(x) for x in w], [O.bf16_to_f64(x) for x in b])
    # frame 7 of codebook 3 contributes its bias alone
    wf = O.bf16_to_f64(w[3])
    ref[0, 7] -= ef[3][0] @ wf.T
    assert np.array_equal(got, ref)
