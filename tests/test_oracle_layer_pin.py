"""Pin of the oracle's decoder-layer composition (CPU only).

omnivoice-cpp ARCHITECTURE.md, Component architecture and its Qwen3
specifics, fix the order of one layer: input_layernorm; q, k, v projections;
per-head q_norm / k_norm (RMSNorm over 128) before RoPE; attention over the
cache; o_proj added to the residual; post_attention_layernorm of the updated
residual; the SwiGLU MLP added to the residual. The pieces are pinned one by
one elsewhere; here the whole layer is rebuilt from PyTorch's float64 CPU
operators in that printed order (RoPE as a complex rotation of the pairs
(i, i + d/2), attention through torch's grouped-query SDPA) and compared with
``Backbone.layer`` on a causal prefill followed by cached decode steps.

Three plausible slips in the composition are planted on the CPU and must fail
the pin: q/k norm applied after RoPE, the MLP fed from input_layernorm's
output, and the attention residual added before o_proj.
"""
import numpy as np
import pytest

import oracle as O
import synth

torch = pytest.importorskip("torch")
F = torch.nn.functional

# q heads x head_dim equals hidden so that the "residual before o_proj" slip is
# expressible; gains are synthetic non-unit values so gain placement matters.
SHAPE = synth.ModelShape(n_layers=1, hidden=32, n_q_heads=4, n_kv_heads=2, head_dim=8, ffn=48,
                         codebook_rows=(), n_heads_out=0, head_rows=0)


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))


def _rope_complex(x, pos, theta):
    """x[T, H, d] rotated as complex numbers z_i = x_i + j x_{i+d/2} times exp(j pos theta^(-2i/d))."""
    d = x.shape[-1]
    half = d // 2
    inv = torch.pow(torch.tensor(float(theta), dtype=torch.float64),
                    -2.0 * torch.arange(half, dtype=torch.float64) / d)
    ang = torch.as_tensor(np.asarray(pos, dtype=np.float64))[:, None] * inv[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]
    z = torch.complex(x[..., :half], x[..., half:]) * rot
    return torch.cat([z.real, z.imag], dim=-1)


def torch_layer(lw, s, H, pos, cache_k, cache_v, allowed):
    """One layer in the printed order from torch float64 operators; returns (H', k, v)."""
    T = H.shape[0]
    eps = s.rms_eps
    y = F.rms_norm(H, (s.hidden,), weight=lw["in_norm"], eps=eps)
    q = F.linear(y, lw["wq"]).view(T, s.n_q_heads, s.head_dim)
    k = F.linear(y, lw["wk"]).view(T, s.n_kv_heads, s.head_dim)
    v = F.linear(y, lw["wv"]).view(T, s.n_kv_heads, s.head_dim)
    q = _rope_complex(F.rms_norm(q, (s.head_dim,), weight=lw["q_norm"], eps=eps), pos, s.rope_theta)
    k = _rope_complex(F.rms_norm(k, (s.head_dim,), weight=lw["k_norm"], eps=eps), pos, s.rope_theta)
    K = torch.cat([cache_k, k], 0)
    V = torch.cat([cache_v, v], 0)
    mask = torch.from_numpy(np.ascontiguousarray(allowed, dtype=bool))
    o = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], K.permute(1, 0, 2)[None],
                                       V.permute(1, 0, 2)[None], attn_mask=mask, enable_gqa=True)
    o = o[0].permute(1, 0, 2).reshape(T, -1)
    H = H + F.linear(o, lw["wo"])
    y2 = F.rms_norm(H, (s.hidden,), weight=lw["post_norm"], eps=eps)
    H = H + F.linear(F.silu(F.linear(y2, lw["wg"])) * F.linear(y2, lw["wu"]), lw["wd"])
    return H, K, V


def check_layer(layer_fn):
    """layer_fn(model, h, pos, cache, allowed) -> new residual (appends to cache).

    A 5-token causal prefill, then three single-token decode steps over the
    cache, each compared with the torch composition."""
    w = synth.model_weights(SHAPE, 41)
    m = O.Backbone(w, SHAPE)
    lw = {k: _t(v) for k, v in m.layers[0].items()}
    rng = np.random.default_rng(42)
    X = rng.normal(0.0, 1.0, (8, SHAPE.hidden))
    cache = m.new_cache()
    tk = torch.zeros((0, SHAPE.n_kv_heads, SHAPE.head_dim), dtype=torch.float64)
    tv = tk.clone()
    steps = [list(range(0, 5)), [5], [6], [7]]
    for pos in steps:
        allowed = O.causal_allowed(pos, pos[-1] + 1)
        got = layer_fn(m, X[pos], pos, cache, allowed)
        want, tk, tv = torch_layer(lw, SHAPE, _t(X[pos]), pos, tk, tv, allowed)
        if not np.allclose(got, want.numpy(), rtol=1e-11, atol=1e-12):
            return False
        if not (np.allclose(cache.k[0], tk.numpy(), rtol=1e-11, atol=1e-12)
                and np.allclose(cache.v[0], tv.numpy(), rtol=1e-11, atol=1e-12)):
            return False
    return True


def _oracle_layer(m, h, pos, cache, allowed):
    return m.layer(0, h, pos, cache, allowed)


def test_layer_composition_matches_torch_in_printed_order():
    assert check_layer(_oracle_layer)


# ---------------------------------------------------------------- planted slips
def _slipped_layer(m, h, pos, cache, allowed, slip):
    """The layer with one composition slip (test-only copy; the oracle is untouched)."""
    s, lw = m.s, m.layers[0]
    T = h.shape[0]
    y = O.rms_norm(h, lw["in_norm"], s.rms_eps)
    q = (y @ lw["wq"].T).reshape(T, s.n_q_heads, s.head_dim)
    k = (y @ lw["wk"].T).reshape(T, s.n_kv_heads, s.head_dim)
    v = (y @ lw["wv"].T).reshape(T, s.n_kv_heads, s.head_dim)
    if slip == "qk_norm_after_rope":
        q = O.rms_norm(O.rope_half_rotate(q, pos, s.rope_theta), lw["q_norm"], s.rms_eps)
        k = O.rms_norm(O.rope_half_rotate(k, pos, s.rope_theta), lw["k_norm"], s.rms_eps)
    else:
        q = O.rope_half_rotate(O.rms_norm(q, lw["q_norm"], s.rms_eps), pos, s.rope_theta)
        k = O.rope_half_rotate(O.rms_norm(k, lw["k_norm"], s.rms_eps), pos, s.rope_theta)
    cache.k[0] = np.concatenate([cache.k[0], k], 0)
    cache.v[0] = np.concatenate([cache.v[0], v], 0)
    o = O.attention_gqa(q, cache.k[0], cache.v[0], allowed).reshape(T, -1)
    if slip == "residual_before_o_proj":
        H = (h + o) @ lw["wo"].T
    else:
        H = h + o @ lw["wo"].T
    y2 = y if slip == "mlp_from_input_norm" else O.rms_norm(H, lw["post_norm"], s.rms_eps)
    return H + O.swiglu_mlp(y2, lw["wg"], lw["wu"], lw["wd"])


def test_slipped_copy_without_slip_passes():
    """The test-only copy is faithful when no slip is planted, so each failure below is the slip's."""
    assert check_layer(lambda m, h, p, c, a: _slipped_layer(m, h, p, c, a, None))


@pytest.mark.parametrize("slip", ["qk_norm_after_rope", "mlp_from_input_norm", "residual_before_o_proj"])
def test_pin_catches_composition_slip(slip):
    assert not check_layer(lambda m, h, p, c, a: _slipped_layer(m, h, p, c, a, slip))
