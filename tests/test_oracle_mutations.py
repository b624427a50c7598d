"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch them.

Each mutant is a one-line slip someone could make writing the oracle: eps
outside the root, (1 + gamma) gains, interleaved RoPE pairs, a flipped sine,
the wrong frequency exponent, a wrong GQA head map, a missing 1/sqrt(d),
SiLU on the wrong branch, a missing codebook offset.
"""
import numpy as np
import pytest

import oracle as O
from tests.test_oracle_pins import (check_attention, check_codebook_sum, check_omnivoice_embed,
                                    check_rmsnorm, check_rope, check_swiglu)


def rms_eps_outside(x, g, eps):
    return x / (np.sqrt(np.mean(x * x, -1, keepdims=True)) + eps) * g


def rms_one_plus_gamma(x, g, eps):
    return x / np.sqrt(np.mean(x * x, -1, keepdims=True) + eps) * (1 + g)


def rope_interleaved(x, pos, theta):
    d = x.shape[-1]
    ang = np.asarray(pos, float)[:, None] * O.rope_inv_freq(d, theta)[None]
    c, s = np.cos(ang)[:, None], np.sin(ang)[:, None]
    a, b = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2], y[..., 1::2] = a * c - b * s, b * c + a * s
    return y


def rope_sign_flip(x, pos, theta):
    return O.rope_half_rotate(x, -np.asarray(pos), theta)


def rope_wrong_exponent(x, pos, theta):
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(pos, float)[:, None] * (theta ** (-np.arange(half) / d))[None]
    c, s = np.cos(ang)[:, None], np.sin(ang)[:, None]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], -1)


def attn_modulo_heads(q, k, v, allowed):
    Hq, Hkv = q.shape[1], k.shape[1]
    out = np.empty_like(q)
    for h in range(Hq):
        one = O.attention_gqa(q[:, h:h + 1], k[:, (h % Hkv):(h % Hkv) + 1], v[:, (h % Hkv):(h % Hkv) + 1], allowed)
        out[:, h] = one[:, 0]
    return out


def attn_no_scale(q, k, v, allowed):
    return O.attention_gqa(q * np.sqrt(q.shape[-1]), k, v, allowed)


def swiglu_wrong_branch(y, wg, wu, wd):
    return ((y @ wg.T) * O.silu(y @ wu.T)) @ wd.T


def cb_sum_ignores_skip(ids, tables):
    ids = np.where(np.asarray(ids) < 0, 0, ids)
    return O.codebook_embed_sum(ids, tables)


def ov_no_offsets(ids, mask, text, audio, V=1025):
    return O.omnivoice_embed(ids, mask, text, audio, 0)


@pytest.mark.parametrize("check,mutant", [
    (check_rmsnorm, rms_eps_outside), (check_rmsnorm, rms_one_plus_gamma),
    (check_rope, rope_interleaved), (check_rope, rope_sign_flip), (check_rope, rope_wrong_exponent),
    (check_attention, attn_modulo_heads), (check_attention, attn_no_scale),
    (check_swiglu, swiglu_wrong_branch), (check_codebook_sum, cb_sum_ignores_skip),
    (check_omnivoice_embed, ov_no_offsets),
])
def test_pin_catches_mutant(check, mutant):
    try:
        ok = check(mutant)
    except (IndexError, ValueError):
        ok = False
    assert not ok
