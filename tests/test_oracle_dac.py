"""Pins of the DAC-decoder oracle (CPU only).

Checks from the page's formulas and from mathematics, not from the oracle
itself ("omnivoice-cpp docs/ARCHITECTURE.md", DAC decoder block channels,
Snake activation, ConvTranspose1d): the printed output lengths (s T per
block, 960 T overall); ConvTranspose1d is the adjoint of the strided
correlation, written here as explicit loops; Conv1d against explicit loops
and a shifting delta kernel; closed forms of the snake; residual units with
zero weights are identities. Planted mistakes are caught.
"""
import math

import numpy as np
import pytest

import oracle as O


def _loops_conv1d(x, w, b, dil, pad):
    IC, T = x.shape
    OC, _, K = w.shape
    T_out = T + 2 * pad - dil * (K - 1)
    y = np.zeros((OC, T_out))
    for o in range(OC):
        for t in range(T_out):
            s = b[o]
            for i in range(IC):
                for k in range(K):
                    ti = t + k * dil - pad
                    if 0 <= ti < T:
                        s += w[o, i, k] * x[i, ti]
            y[o, t] = s
    return y


def _strided_correlation(y, w, stride, pad, T_in):
    """Adjoint of ConvTranspose1d: z[i, t] = sum_o sum_k w[i, o, k] y[o, t s + k - p]."""
    IC, OC, K = w.shape
    z = np.zeros((IC, T_in))
    for i in range(IC):
        for t in range(T_in):
            s = 0.0
            for o in range(OC):
                for k in range(K):
                    to = t * stride + k - pad
                    if 0 <= to < y.shape[1]:
                        s += w[i, o, k] * y[o, to]
            z[i, t] = s
    return z


def check_conv_transpose(fn=O.conv_transpose1d):
    rng = np.random.default_rng(3)
    for r in O.DAC_RATIOS:
        IC, OC, T = 3, 2, 5
        x = rng.normal(size=(IC, T))
        w = rng.normal(size=(IC, OC, 2 * r))
        y = fn(x, w, np.zeros(OC), r, math.ceil(r / 2), r % 2)
        if y.shape != (OC, r * T):  # the page: T_out = stride * T_in exactly for all five blocks
            return False
        g = rng.normal(size=y.shape)
        lhs = float(np.sum(y * g))
        rhs = float(np.sum(x * _strided_correlation(g, w, r, math.ceil(r / 2), T)))
        if abs(lhs - rhs) > 1e-9 * max(1.0, abs(lhs)):
            return False
        bias = rng.normal(size=OC)
        if not np.allclose(fn(x, w, bias, r, math.ceil(r / 2), r % 2) - y, bias[:, None], atol=1e-12):
            return False
    return True


def check_conv1d(fn=O.conv1d):
    rng = np.random.default_rng(4)
    for dil, pad, K in ((1, 3, 7), (3, 9, 7), (9, 27, 7), (1, 0, 1)):
        x = rng.normal(size=(3, 30))
        w = rng.normal(size=(2, 3, K))
        b = rng.normal(size=2)
        got, want = fn(x, w, b, dil, pad), _loops_conv1d(x, w, b, dil, pad)
        if got.shape != want.shape or not np.allclose(got, want, rtol=1e-12, atol=1e-12):
            return False
    # a delta kernel at tap k0 shifts by k0 dil - pad
    x = rng.normal(size=(2, 20))
    w = np.zeros((2, 2, 7))
    w[0, 0, 5] = w[1, 1, 5] = 1.0
    y = fn(x, w, np.zeros(2), 3, 9)
    shift = 5 * 3 - 9
    if y.shape != (2, 20) or not np.allclose(y[:, :20 - shift], x[:, shift:], atol=0) or not np.allclose(y[:, 20 - shift:], 0.0):
        return False
    return True


def check_snake(fn=O.snake):
    a = np.array([0.5, 1.0, 2.0])
    x = np.zeros((3, 4))
    if not np.array_equal(fn(x, a), x):
        return False
    x = (np.pi / (2 * a))[:, None] * np.ones((3, 2))  # sin(a x)^2 = 1
    if not np.allclose(fn(x, a), x + (1.0 / (a + 1e-9))[:, None], rtol=1e-15, atol=1e-15):
        return False
    x = (np.pi / a)[:, None] * np.ones((3, 2))        # sin(a x)^2 = 0
    return np.allclose(fn(x, a), x, rtol=0, atol=1e-12)


def _zero_res_weights(T=3, seed=5):
    rng = np.random.default_rng(seed)
    C = O.DAC_CHANNELS
    w = {"fc2_w": rng.normal(0, 0.03, (256, 1024)), "fc2_b": rng.normal(0, 0.1, 256),
         "conv1_w": rng.normal(0, 0.02, (1024, 256, 7)), "conv1_b": rng.normal(0, 0.1, 1024), "blocks": [],
         "final_alpha": rng.uniform(0.5, 1.5, 32), "conv2_w": rng.normal(0, 0.1, (1, 32, 7)),
         "conv2_b": np.array([0.05])}
    for i, r in enumerate(O.DAC_RATIOS):
        ic, oc = C[i], C[i + 1]
        res = [{"alpha1": np.ones(oc), "w1": np.zeros((oc, oc, 7)), "b1": np.zeros(oc), "alpha2": np.ones(oc),
                "w2": np.zeros((oc, oc, 1)), "b2": np.zeros(oc)} for _ in range(3)]
        w["blocks"].append({"alpha": rng.uniform(0.5, 1.5, ic), "up_w": rng.normal(0, 1 / math.sqrt(ic * r), (ic, oc, 2 * r)),
                            "up_b": rng.normal(0, 0.1, oc), "res": res})
    return w, rng.normal(size=(1, T, 1024))


def test_dac_pins():
    assert check_conv_transpose()
    assert check_conv1d()
    assert check_snake()


def test_convolutions_match_pytorch_cpu_ops():
    """The page's layers are PyTorch's Conv1d and ConvTranspose1d: the library's own
    float64 CPU ops give the same result for the five upsampling blocks (k 2r, stride r,
    padding ceil(r/2), output padding r mod 2) and the dilated k = 7 convolutions."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    rng = np.random.default_rng(6)
    for r in O.DAC_RATIOS:
        x, w, b = rng.normal(size=(4, 9)), rng.normal(size=(4, 3, 2 * r)), rng.normal(size=3)
        want = F.conv_transpose1d(torch.from_numpy(x)[None], torch.from_numpy(w), torch.from_numpy(b), stride=r,
                                  padding=math.ceil(r / 2), output_padding=r % 2)[0].numpy()
        got = O.conv_transpose1d(x, w, b, r, math.ceil(r / 2), r % 2)
        assert got.shape == want.shape == (3, 9 * r)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    for dil in O.DAC_DILATIONS:
        x, w, b = rng.normal(size=(4, 40)), rng.normal(size=(3, 4, 7)), rng.normal(size=3)
        want = F.conv1d(torch.from_numpy(x)[None], torch.from_numpy(w), torch.from_numpy(b), padding=3 * dil,
                        dilation=dil)[0].numpy()
        got = O.conv1d(x, w, b, dil, 3 * dil)
        assert got.shape == want.shape == (3, 40)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_dac_chain_with_identity_residual_units():
    """Zero residual weights make every residual unit the identity: the decode is
    fc2, conv1, then per block ConvTranspose(snake(x)), then snake + conv2; 960 T samples."""
    w, feat = _zero_res_weights()
    got = O.dac_decode(feat, w)
    assert got.shape == (1, 1, 960 * 3)
    x = np.asarray(w["fc2_w"]) @ feat[0].T + np.asarray(w["fc2_b"])[:, None]
    x = _loops_conv1d(x, np.asarray(w["conv1_w"]), np.asarray(w["conv1_b"]), 1, 3)
    for i, r in enumerate(O.DAC_RATIOS):
        blk = w["blocks"][i]
        a = np.asarray(blk["alpha"])[:, None]
        xs = x + (1.0 / (a + 1e-9)) * np.sin(a * x) ** 2
        x = O.conv_transpose1d(xs, blk["up_w"], blk["up_b"], r, math.ceil(r / 2), r % 2)
    a = np.asarray(w["final_alpha"])[:, None]
    xs = x + (1.0 / (a + 1e-9)) * np.sin(a * x) ** 2
    want = O.conv1d(xs, w["conv2_w"], w["conv2_b"], 1, 3)
    assert np.allclose(got[0], want, rtol=1e-12, atol=1e-12)
    assert O.dac_shapes(3) == [3, 24, 120, 480, 960, 2880]


# ---------------------------------------------------------------- planted mistakes
def _convT_floor_pad(x, w, b, s, p, op):
    return O.conv_transpose1d(x, w, b, s, s // 2, op)


def _convT_no_outpad(x, w, b, s, p, op):
    return O.conv_transpose1d(x, w, b, s, p, 0)


def _convT_flipped(x, w, b, s, p, op):
    return O.conv_transpose1d(x, np.asarray(w)[:, :, ::-1], b, s, p, op)


def _conv_no_dilation(x, w, b, dil=1, pad=0):
    return O.conv1d(x, w, b, 1, pad)


def _conv_flipped(x, w, b, dil=1, pad=0):
    return O.conv1d(x, np.asarray(w)[:, :, ::-1], b, dil, pad)


def _snake_no_alpha_inside(x, alpha):
    a = np.asarray(alpha)[:, None]
    return x + (1.0 / (a + 1e-9)) * np.sin(x) ** 2


def _snake_wrong_scale(x, alpha):
    a = np.asarray(alpha)[:, None]
    return x + a * np.sin(a * x) ** 2


@pytest.mark.parametrize("mutant,check", [(_convT_floor_pad, check_conv_transpose), (_convT_no_outpad, check_conv_transpose),
                                          (_convT_flipped, check_conv_transpose), (_conv_no_dilation, check_conv1d),
                                          (_conv_flipped, check_conv1d), (_snake_no_alpha_inside, check_snake),
                                          (_snake_wrong_scale, check_snake)])
def test_dac_mutants_are_caught(mutant, check):
    assert not check(mutant)
