"""Qwen3-TTS quantizer lookup on the GPU against the fp64 oracle.

"Qwen3-TTS ncnn port", Codec Decoder split: 16 codebooks of 2048 entries,
codebook 0 (semantic) and codebooks 1..15 (acoustic) through their own
projections, summed into the [B, 512, T] hidden of the codec body. The page
gives no codebook width; these tests use 256 (and 64 for the small case).

* Integer-valued tables and projections make every sum and product exact in
  bf16 / fp32, so the output must equal the oracle bit for bit: any wrong
  code, codebook, projection or output index shows. Both GEMM routes are
  covered: a few frames (matrix-vector kernel) and many frames (tcgen05).
* Normal tables at the full 4 x 768-frame size: within 1e-4 of each output
  row's largest magnitude, the accuracy bound the page reports for its own
  NumPy quantizer against PyTorch.
* Codes outside the table contribute nothing and are reported as BAD_ID.
"""
import numpy as np
import pytest

import oracle as O
import synth
from tests.gpu_util import dev_bf16_bits, dev_i32, tb

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

K, N_ROWS, OUT = 16, 2048, 512


def _int_bits(rng, shape, lo, hi):
    return synth.bf16_bits(rng.integers(lo, hi + 1, shape).astype(np.float32))


def _run(books_bits, ps_bits, pa_bits, codes):
    m = tb()
    B, _, T = codes.shape
    st = torch.cuda.current_stream().cuda_stream
    q = m.tts_bb_quantizer_create([dev_bf16_bits(b) for b in books_bits], dev_bf16_bits(ps_bits),
                                  dev_bf16_bits(pa_bits), st)
    try:
        out = torch.full((B, ps_bits.shape[0], T), float("nan"), dtype=torch.float32, device="cuda")
        m.tts_bb_quantizer_decode(q, B, T, dev_i32(codes), out)
        status = m.tts_bb_quantizer_sync(q)
        return out.cpu().numpy().astype(np.float64), status
    finally:
        m.tts_bb_quantizer_free(q)


def _oracle(books_bits, ps_bits, pa_bits, codes):
    f = O.bf16_to_f64
    return O.split_quantizer_decode(codes, [f(b) for b in books_bits], f(ps_bits), f(pa_bits))


@pytest.mark.parametrize("B,T,d", [(1, 5, 64), (2, 37, 256), (3, 200, 128)])
def test_quantizer_bit_exact_on_integer_tables(B, T, d):
    rng = synth.rng_for(71, f"quant_int_{B}_{T}_{d}")
    books = [_int_bits(rng, (N_ROWS, d), -3, 3) for _ in range(K)]
    ps = _int_bits(rng, (OUT, d), -4, 4)
    pa = _int_bits(rng, (OUT, d), -4, 4)
    codes = rng.integers(0, N_ROWS, (B, K, T)).astype(np.int32)
    got, status = _run(books, ps, pa, codes)
    assert status == tb().OK
    assert np.array_equal(got, _oracle(books, ps, pa, codes))


def test_quantizer_full_size_normal_tables():
    B, T, d = 4, 768, 256
    r = synth.rng_for(72, "quant_full")
    books = [synth.normal_bf16(r, (N_ROWS, d), 1.0) for _ in range(K)]
    ps = synth.normal_bf16(r, (OUT, d), 0.02)
    pa = synth.normal_bf16(r, (OUT, d), 0.02)
    codes = r.integers(0, N_ROWS, (B, K, T)).astype(np.int32)
    got, status = _run(books, ps, pa, codes)
    assert status == tb().OK
    want = _oracle(books, ps, pa, codes)
    err = np.max(np.abs(got - want), axis=2) / np.max(np.abs(want), axis=2)   # per (b, channel) row
    assert float(err.max()) <= 1e-4, float(err.max())


def test_quantizer_bad_codes_are_reported_and_skipped():
    B, T, d = 1, 12, 64
    rng = synth.rng_for(73, "quant_bad")
    books = [_int_bits(rng, (N_ROWS, d), -3, 3) for _ in range(K)]
    ps = _int_bits(rng, (OUT, d), -4, 4)
    pa = _int_bits(rng, (OUT, d), -4, 4)
    codes = rng.integers(0, N_ROWS, (B, K, T)).astype(np.int32)
    bad = codes.copy()
    bad[0, 0, 3] = N_ROWS          # semantic code past the table
    bad[0, 9, 7] = -1              # acoustic code below it
    got, status = _run(books, ps, pa, bad)
    assert status == tb().E_BAD_ID
    # the two bad lookups contribute zero rows: the oracle with those rows removed
    want = _oracle(books, ps, pa, codes)
    f = O.bf16_to_f64
    want[0, :, 3] -= f(ps) @ f(books[0][codes[0, 0, 3]])
    want[0, :, 7] -= f(pa) @ f(books[9][codes[0, 9, 7]])
    assert np.array_equal(got, want)
