"""Pins of oracle pieces against PyTorch's own float64 CPU operators (CPU only).

The pages define the layers by PyTorch's modules (omnivoice-cpp ARCHITECTURE.md,
Qwen3 specifics: RMSNorm, SwiGLU, SDPA with grouped KV heads; Qwen3-TTS ncnn
port, single-token SDPA), so the library's operators are an independent check
of the oracle's numpy code: RMSNorm with eps inside the root, scaled
dot-product attention with grouped query heads (query head h reads KV head
h // 2) under causal, key-length and single-query masks, and SiLU.
"""
import numpy as np
import pytest

import oracle as O

torch = pytest.importorskip("torch")
F = torch.nn.functional


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a))


def test_rms_norm_matches_torch():
    rng = np.random.default_rng(11)
    x = rng.normal(0, 3.0, (7, 1024))
    g = rng.normal(1.0, 0.1, 1024)
    for eps in (1e-6, 0.5):
        want = F.rms_norm(_t(x), (1024,), weight=_t(g), eps=eps).numpy()
        assert np.allclose(O.rms_norm(x, g, eps), want, rtol=1e-13, atol=1e-13)


def _sdpa(q, k, v, allowed):
    """q[Tq, Hq, d], k/v[Tk, Hkv, d] -> [Tq, Hq, d] through torch's SDPA with enable_gqa."""
    out = F.scaled_dot_product_attention(_t(q).permute(1, 0, 2)[None], _t(k).permute(1, 0, 2)[None],
                                         _t(v).permute(1, 0, 2)[None], attn_mask=_t(allowed), enable_gqa=True)
    return out[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("case", ["prefill_chunk", "decode", "bidirectional_padded"])
def test_attention_gqa_matches_torch_sdpa(case):
    rng = np.random.default_rng(12)
    Hq, Hkv, d = 16, 8, 128
    if case == "prefill_chunk":      # 9 new queries at positions 14..22 over a 23-key cache
        Tq, Tk = 9, 23
        allowed = O.causal_allowed(list(range(14, 23)), Tk)
    elif case == "decode":           # one query at the last position
        Tq, Tk = 1, 40
        allowed = O.causal_allowed([39], Tk)
    else:                            # MaskGIT pass: every query sees the first 21 of 30 keys
        Tq, Tk = 30, 30
        allowed = np.ascontiguousarray(O.keylen_allowed(Tq, Tk, 21))
    q = rng.normal(size=(Tq, Hq, d))
    k = rng.normal(size=(Tk, Hkv, d))
    v = rng.normal(size=(Tk, Hkv, d))
    got = O.attention_gqa(q, k, v, allowed)
    want = _sdpa(q, k, v, allowed)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_attention_gqa_head_map_is_floor_half():
    """Swapping the two query heads of one KV head changes nothing else; reading KV head
    h % 8 instead of h // 2 would (checked against torch's grouped SDPA)."""
    rng = np.random.default_rng(13)
    q = rng.normal(size=(5, 16, 128))
    k = rng.normal(size=(7, 8, 128))
    v = rng.normal(size=(7, 8, 128))
    allowed = O.causal_allowed(list(range(2, 7)), 7)
    want = _sdpa(q, k, v, allowed)
    modulo = np.empty_like(want)
    for h in range(16):  # the plausible wrong map, through the oracle's own single-head path
        modulo[:, h:h + 1] = O.attention_gqa(q[:, h:h + 1], k[:, h % 8:h % 8 + 1], v[:, h % 8:h % 8 + 1], allowed)
    assert np.allclose(O.attention_gqa(q, k, v, allowed), want, rtol=1e-12, atol=1e-12)
    assert not np.allclose(modulo, want, rtol=1e-6, atol=1e-6)


def test_silu_matches_torch():
    x = np.linspace(-30, 30, 601)
    assert np.allclose(O.silu(x), F.silu(_t(x)).numpy(), rtol=1e-14, atol=1e-300)
