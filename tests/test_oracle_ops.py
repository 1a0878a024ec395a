"""Pins of the oracle's unfused operators against facts that do not come from the
oracle: closed forms, the spec fixed facts (RMSNorm of a constant vector,
RoPE identity at position 0, BN folding == Conv -> BN), hand-derived worked
examples (tests/golden/), an independent complex-number form of the rotation,
brute-force loops, and torch's own fp64 operators as library routines."""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import ops
from conftest import GOLDEN


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ RMSNorm

@pytest.mark.parametrize("c", [3.0, -0.75, 1e-3, 250.0])
def test_rmsnorm_of_constant_vector(c):
    h = 64
    w = np.linspace(0.5, 1.5, h)
    eps = 1e-6
    y = ops.rmsnorm(np.full((1, h), c), eps, w[None, :])
    assert np.allclose(y[0], c / math.sqrt(c * c + eps) * w, rtol=1e-14, atol=0)
    y0 = ops.rmsnorm(np.full((1, h), c), 0.0, w[None, :])
    assert np.array_equal(y0[0], math.copysign(1.0, c) * w)       # exactly sign * w


def test_rmsnorm_single_element_and_scale_invariance():
    assert ops.rmsnorm(np.array([[-2.5]]), 0.0, np.array([[0.7]]))[0, 0] == -0.7
    rng = np.random.default_rng(3)
    x = rng.normal(size=(4, 96))
    for k in (1e-3, 7.0, -2.0):
        assert np.allclose(ops.rmsnorm(k * x, 0.0), math.copysign(1, k) * ops.rmsnorm(x, 0.0), rtol=1e-13, atol=1e-14)


def test_rmsnorm_matches_torch_rms_norm_fp64():
    rng = np.random.default_rng(4)
    x = rng.normal(size=(8, 200))
    w = rng.normal(1, 0.1, 200)
    want = F.rms_norm(torch.from_numpy(x), (200,), torch.from_numpy(w), eps=1e-6).numpy()
    assert np.allclose(ops.rmsnorm(x, 1e-6, w[None, :]), want, rtol=1e-13, atol=1e-14)


def test_ada_modulate_and_gated_residual_closed_forms():
    n = np.array([[1.0, -2.0, 0.5]])
    assert np.array_equal(ops.ada_modulate(n, np.zeros(3), np.zeros(3)), n)
    assert np.array_equal(ops.ada_modulate(n, np.array([1.0, -1.0, 0.0]), np.array([0.0, 3.0, -0.5])),
                          np.array([[2.0, 3.0, 0.0]]))
    x = np.array([[1.0, 2.0]])
    r = np.array([[0.5, -1.0]])
    assert np.array_equal(ops.gated_residual_add(x, r, np.ones(2)), ops.residual_add(x, r))
    assert np.array_equal(ops.gated_residual_add(x, r, np.array([0.0, -2.0])), np.array([[0.5, -5.0]]))


def test_per_head_equals_full_width_for_one_head():
    rng = np.random.default_rng(5)
    u = rng.normal(size=(3, 1, 16))
    w = rng.normal(1, 0.1, 16)
    assert np.allclose(ops.qk_rmsnorm_per_head(u, w, 1e-6), ops.qk_rmsnorm_full_width(u, w, 1e-6),
                       rtol=1e-14, atol=1e-15)


def test_full_width_norm_uses_one_scale_per_token():
    rng = np.random.default_rng(6)
    u = rng.normal(size=(2, 4, 8))
    w = np.ones(32)
    out = ops.qk_rmsnorm_full_width(u, w, 0.0)
    flat = u.reshape(2, 32)
    inv = 1 / np.sqrt((flat ** 2).mean(axis=1))
    assert np.allclose(out.reshape(2, 32), flat * inv[:, None], rtol=1e-14)


# --------------------------------------------------------------------- RoPE

@pytest.mark.parametrize("c", [3.0, -0.25, 1e-3])
def test_layernorm_of_constant_vector_is_the_bias(c):
    """A constant vector has no deviation from its mean: the output is b
    exactly, whatever the weight and eps."""
    w = np.array([0.5, -2.0, 3.0, 1.5, 0.75])
    b = np.array([0.1, -0.2, 0.3, 0.0, 5.0])
    assert np.array_equal(ops.layernorm(np.full((2, 5), c), 1e-5, w, b), np.tile(b, (2, 1)))


def test_layernorm_worked_example():
    """x = (1, 2, 3, 4), eps = 0: mean 2.5, variance 1.25, so
    y = (x - 2.5) / sqrt(1.25) = (-3, -1, 1, 3) / sqrt(5)."""
    y = ops.layernorm(np.array([1.0, 2.0, 3.0, 4.0]), 0.0)
    assert np.allclose(y, np.array([-3.0, -1.0, 1.0, 3.0]) / np.sqrt(5.0), rtol=0, atol=1e-15)


def test_layernorm_shift_and_scale_invariance_and_moments():
    """LN(a x + c) = LN(x) for a > 0 at eps = 0; with w = 1, b = 0 the output
    has mean 0 and variance var / (var + eps)."""
    x = np.random.default_rng(5).normal(size=(7, 64)) * 3 + 1
    base = ops.layernorm(x, 0.0)
    assert np.allclose(ops.layernorm(2.5 * x - 7.0, 0.0), base, rtol=0, atol=1e-12)
    eps = 0.3
    y = ops.layernorm(x, eps)
    var = x.var(axis=-1)
    assert np.allclose(y.mean(axis=-1), 0, atol=1e-13)
    assert np.allclose(y.var(axis=-1), var / (var + eps), rtol=1e-12)


def test_layernorm_matches_torch_layer_norm_fp64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(6)
    x, w, b = rng.normal(size=(5, 128)), rng.normal(size=128), rng.normal(size=128)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (128,), torch.from_numpy(w), torch.from_numpy(b),
                                         eps=1e-5).numpy()
    assert np.allclose(ops.layernorm(x, 1e-5, w, b), ref, rtol=1e-12, atol=1e-12)


def test_qk_layernorm_is_per_head():
    """Each head is normalised on its own: scaling one head leaves the others."""
    rng = np.random.default_rng(8)
    u = rng.normal(size=(2, 3, 16))
    w, b = rng.normal(size=16), rng.normal(size=16)
    y = ops.qk_layernorm_per_head(u, w, b, 1e-6)
    u2 = u.copy()
    u2[:, 1] *= 10
    y2 = ops.qk_layernorm_per_head(u2, w, b, 1e-6)
    assert np.allclose(y[:, [0, 2]], y2[:, [0, 2]], rtol=0, atol=0)
    assert np.allclose(y[:, 1], y2[:, 1], atol=1e-6)      # only eps separates them


def test_gelu_erf_and_silu_match_torch_fp64():
    torch = pytest.importorskip("torch")
    a = np.linspace(-12, 12, 2001)
    t = torch.from_numpy(a)
    assert np.allclose(ops.gelu_erf(a), torch.nn.functional.gelu(t, approximate="none").numpy(), rtol=1e-14, atol=1e-15)
    assert np.allclose(ops.silu(a), torch.nn.functional.silu(t).numpy(), rtol=1e-14, atol=1e-15)


def test_gelu_erf_and_silu_closed_forms():
    """f(a) - f(-a) = a for both (a (Phi(a) + Phi(-a)) = a, a (s(a) + s(-a)) = a);
    f(0) = 0; f(a) -> a for large a and -> 0 for large -a; erf(1) and the
    Gaussian CDF at 1 give GELU(1) = 0.841344746068543."""
    a = np.linspace(-9, 9, 361)
    for f in (ops.gelu_erf, ops.silu):
        assert np.allclose(f(a) - f(-a), a, rtol=0, atol=1e-12)
        assert f(0.0) == 0.0
        assert abs(f(40.0) - 40.0) < 1e-12 and abs(f(-40.0)) < 1e-12
    assert abs(ops.gelu_erf(1.0) - 0.841344746068543) < 1e-15
    assert abs(ops.activation(1.0, ops.ACT_GELU_ERF) - 0.841344746068543) < 1e-15
    assert ops.activation(2.0, ops.ACT_SILU) == ops.silu(2.0)
    assert abs(ops.activation(1.0, ops.ACT_GELU_TANH) - 0.841344746068543) > 1e-4   # the tanh form differs
    assert abs(ops.silu(1.0) - 1.0 / (1.0 + np.exp(-1.0))) == 0.0
    assert np.all(np.isfinite(ops.silu(np.array([-1e4, 1e4]))))


def test_gated_activation_is_gate_act_times_up():
    """up = 1 gives act(gate); gate large gives up * gate; up = 0 gives 0;
    GELU tanh and erf agree to the tanh form's 1e-3 approximation error."""
    rng = np.random.default_rng(3)
    g, u = rng.normal(size=64) * 3, rng.normal(size=64)
    for act in (ops.ACT_GELU_TANH, ops.ACT_GELU_ERF, ops.ACT_SILU):
        assert np.array_equal(ops.gated_activation(g, np.ones(64), act), ops.activation(g, act))
        assert not ops.gated_activation(g, np.zeros(64), act).any()
        assert np.allclose(ops.gated_activation(np.full(3, 50.0), u[:3], act), 50.0 * u[:3], rtol=1e-12)
    assert np.allclose(ops.gelu_tanh(g), ops.gelu_erf(g), rtol=0, atol=1e-3)


def test_fold_norm_weight_equals_scaling_the_input_fp64():
    """Linear(y * (1 + g)) with W equals Linear(y) with the folded W', and the
    plain (non-Gemma) fold equals Linear(y * g)."""
    rng = np.random.default_rng(12)
    y, w, g = rng.normal(size=(5, 24)), rng.normal(size=(7, 24)), rng.normal(size=24) * 0.1
    assert np.allclose(ops.linear(y * (1 + g), w), ops.linear(y, ops.fold_norm_weight(w, g)), rtol=1e-12, atol=1e-12)
    assert np.allclose(ops.linear(y * g, w), ops.linear(y, ops.fold_norm_weight(w, g, gemma_style=False)),
                       rtol=1e-12, atol=1e-12)


def test_fold_norm_weight_worked_example():
    """W = 1.5, gamma = 0.25: 1.5 * 1.25 = 1.875 exactly (binary32 too); a zero
    Gemma weight leaves W unchanged."""
    w = np.array([[1.5, -3.0]], np.float32)
    out = ops.fold_norm_weight(w, np.array([0.25, 0.0], np.float32), dtype=np.float32)
    assert out.dtype == np.float32 and out.tolist() == [[1.875, -3.0]]


def test_linear_dequant_brute_force_and_scales():
    """A 2 x 3 by 4 x 3 product written out term by term; doubling the
    activation scale doubles the bias-free output; zero codes give the bias."""
    xq = np.array([[1.0, -2.0, 0.5], [3.0, 0.0, -1.0]])
    wq = np.array([[1.0, 1.0, 1.0], [0.5, -1.0, 2.0], [0.0, 4.0, -0.25], [1.5, 2.0, 3.0]])
    sw = np.array([0.5, 2.0, 1.0, 0.25])
    b = np.array([0.1, -0.2, 0.3, 0.0])
    y = ops.linear_dequant(xq, 0.5, wq, sw, b)
    for i in range(2):
        for j in range(4):
            want = b[j] + sum(xq[i, k] * 0.5 * wq[j, k] * sw[j] for k in range(3))
            assert abs(y[i, j] - want) < 1e-15
    assert np.allclose(ops.linear_dequant(xq, 1.0, wq, sw), 2 * ops.linear_dequant(xq, 0.5, wq, sw), rtol=0)
    assert np.array_equal(ops.linear_dequant(np.zeros((2, 3)), 0.5, wq, sw, b), np.tile(b, (2, 1)))


def test_rope_worked_example():
    g = load("rope_worked.json")
    u = np.array(g["u"]).reshape(1, 1, 4)
    out = ops.rope_rotate_half(u, np.array([g["pos"]]), g["theta"])
    assert np.allclose(out.ravel(), g["expected"], rtol=0, atol=1e-14)


def test_rope_position_zero_is_identity():
    rng = np.random.default_rng(7)
    u = rng.normal(size=(5, 3, 128))
    assert np.array_equal(ops.rope_rotate_half(u, np.zeros(5), 1e6), u)
    assert np.array_equal(ops.rope_3d_sections(u, np.zeros((5, 3)), (44, 42, 42), 1e4), u)


def test_rope_preserves_pair_norms_and_composes():
    rng = np.random.default_rng(8)
    u = rng.normal(size=(6, 2, 64))
    p1 = rng.integers(0, 5000, 6)
    p2 = rng.integers(0, 5000, 6)
    o = ops.rope_rotate_half(u, p1, 1e4)
    half = 32
    n_in = u[..., :half] ** 2 + u[..., half:] ** 2
    n_out = o[..., :half] ** 2 + o[..., half:] ** 2
    assert np.allclose(n_in, n_out, rtol=1e-12)
    twice = ops.rope_rotate_half(o, p2, 1e4)
    assert np.allclose(twice, ops.rope_rotate_half(u, p1 + p2, 1e4), rtol=0, atol=1e-9)


def test_rope_matches_complex_multiplication():
    rng = np.random.default_rng(9)
    d = 128
    u = rng.normal(size=(10, 4, d))
    pos = rng.integers(0, 4096, 10)
    theta = 1e6
    # independent formulation: z_j = u_j + i u_{j+d/2} rotated by exp(i pos theta^(-2j/d))
    z = u[..., :d // 2] + 1j * u[..., d // 2:]
    ang = pos[:, None].astype(np.float64) * theta ** (-np.arange(d // 2) * 2.0 / d)[None, :]
    zr = z * np.exp(1j * ang)[:, None, :]
    want = np.concatenate([zr.real, zr.imag], axis=-1)
    assert np.allclose(ops.rope_rotate_half(u, pos, theta), want, rtol=0, atol=1e-12)


def test_rope_quarter_turn_sign_convention():
    # D = 4: omega_1 = theta^(-1/2); theta = (2/pi)^2 makes the angle at pos 1 exactly pi/2
    theta = (2.0 / math.pi) ** 2
    u = np.array([0.3, 1.0, -0.2, 2.0]).reshape(1, 1, 4)
    o = ops.rope_rotate_half(u, np.array([1]), theta).ravel()
    assert abs(o[1] - (-2.0)) < 1e-15 and abs(o[3] - 1.0) < 1e-15   # o1 = -u3, o3 = +u1


def test_rope_3d_single_section_equals_1d():
    rng = np.random.default_rng(10)
    u = rng.normal(size=(7, 2, 32))
    pos3 = rng.integers(0, 50, (7, 3))
    assert np.array_equal(ops.rope_3d_sections(u, pos3, (32, 0, 0), 1e4),
                          ops.rope_rotate_half(u, pos3[:, 0], 1e4))
    assert np.array_equal(ops.rope_3d_sections(u, pos3, (0, 0, 32), 1e4),
                          ops.rope_rotate_half(u, pos3[:, 2], 1e4))


def test_rope_3d_chunks_are_independent_rotations():
    rng = np.random.default_rng(11)
    u = rng.normal(size=(4, 3, 128))
    pos3 = rng.integers(0, 60, (4, 3))
    out = ops.rope_3d_sections(u, pos3, (44, 42, 42), 1e4)
    for c, (s, w) in enumerate([(0, 44), (44, 42), (86, 42)]):
        want = ops.rope_rotate_half(u[..., s:s + w], pos3[:, c], 1e4)
        assert np.array_equal(out[..., s:s + w], want)
        h = w // 2    # partner at +w/2 within the chunk: pair norms preserved
        assert np.allclose(u[..., s:s + h] ** 2 + u[..., s + h:s + w] ** 2,
                           out[..., s:s + h] ** 2 + out[..., s + h:s + w] ** 2, rtol=1e-12)
    # the two readings of the 3D layout disagree away from the origin
    alt = ops.rope_3d_global_pairs(u, pos3, (44, 42, 42), 1e4)
    assert not np.allclose(out, alt)


# ------------------------------------------------------------ split layout

def test_split_packed_qkv_layout():
    t, hq, hkv, d = 2, 3, 1, 4
    row = np.arange((hq + 2 * hkv) * d)
    qkv = np.stack([row, row + 1000])
    q, k, v = ops.split_packed_qkv(qkv, hq, hkv, d)
    assert q.shape == (2, 3, 4) and k.shape == (2, 1, 4) and v.shape == (2, 1, 4)
    assert q[1, 2, 3] == 1000 + 2 * 4 + 3
    assert k[0, 0, 0] == 12 and v[0, 0, 0] == 16


# --------------------------------------------------------- Linear and GELU

def test_linear_against_brute_force():
    rng = np.random.default_rng(12)
    x = rng.normal(size=(3, 5))
    w = rng.normal(size=(4, 5))
    b = rng.normal(size=4)
    y = ops.linear(x, w, b)
    for i in range(3):
        for j in range(4):
            s = b[j]
            for kk in range(5):
                s += x[i, kk] * w[j, kk]
            assert abs(y[i, j] - s) < 1e-13
    assert np.allclose(y, F.linear(torch.from_numpy(x), torch.from_numpy(w), torch.from_numpy(b)).numpy(),
                       rtol=1e-14, atol=1e-14)


def test_gelu_constants_are_the_printed_ones():
    g = load("gelu_constants.json")
    assert ops.GELU_C0 == g["c0"] and ops.GELU_C1 == g["c1"]
    assert abs(g["c0"] - math.sqrt(2 / math.pi)) < 1e-10


def test_gelu_closed_form_properties():
    x = np.linspace(-8, 8, 4001)
    g = ops.gelu_tanh(x)
    assert ops.gelu_tanh(np.array([0.0]))[0] == 0.0
    assert np.allclose(g - ops.gelu_tanh(-x), x, rtol=0, atol=1e-13)        # gelu(x) - gelu(-x) = x
    assert np.allclose(ops.gelu_tanh(np.array([30.0, -30.0])), [30.0, 0.0], atol=1e-12)
    # tanh form stays within 5e-4 of the exact (erf) GELU; a wrong constant breaks this
    exact = np.array([0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in x])
    assert np.max(np.abs(g - exact)) < 5e-4
    lib = F.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    assert np.allclose(g, lib, rtol=1e-9, atol=1e-12)


# --------------------------------------------------------------- BatchNorm

def test_batchnorm_matches_torch():
    rng = np.random.default_rng(13)
    y = rng.normal(size=(5, 6))
    gamma, beta, mean = rng.uniform(0.5, 1.5, 6), rng.normal(0, .1, 6), rng.normal(0, .1, 6)
    var = rng.uniform(0.01, 1, 6)
    want = F.batch_norm(torch.from_numpy(y), torch.from_numpy(mean), torch.from_numpy(var),
                        torch.from_numpy(gamma), torch.from_numpy(beta), training=False, eps=1e-2).numpy()
    assert np.allclose(ops.batchnorm_inference(y, gamma, beta, mean, var, 1e-2), want, rtol=1e-13, atol=1e-14)


def test_conv_direct_matches_torch_and_1x1_is_matmul():
    rng = np.random.default_rng(14)
    inp = rng.normal(size=(2, 3, 7, 6))
    w = rng.normal(size=(4, 3, 3, 3))
    b = rng.normal(size=4)
    for stride, pad in [(1, 0), (2, 1), (1, 2)]:
        want = F.conv2d(torch.from_numpy(inp), torch.from_numpy(w), torch.from_numpy(b), stride=stride,
                        padding=pad).numpy()
        assert np.allclose(ops.conv2d_direct(inp, w, b, stride, pad), want, rtol=1e-13, atol=1e-13)
    w1 = rng.normal(size=(5, 3, 1, 1))
    out = ops.conv2d_direct(inp, w1, None)
    mm = np.einsum("oc,nchw->nohw", w1[:, :, 0, 0], inp)
    assert np.allclose(out, mm, rtol=1e-13, atol=1e-13)


def test_bn_fold_equals_conv_then_bn_fp64():
    """North-star fact: folded Conv == Conv -> BN (and the same for Linear)."""
    rng = np.random.default_rng(15)
    inp = rng.normal(size=(1, 3, 6, 5))
    w = rng.normal(size=(4, 3, 3, 3))
    b = rng.normal(size=4)
    gamma, beta = rng.uniform(0.5, 1.5, 4), rng.normal(0, .1, 4)
    mean, var = rng.normal(0, .1, 4), rng.uniform(0.01, 1, 4)
    for eps, bias in [(1e-2, b), (1e-5, None)]:
        ref = ops.batchnorm_inference(ops.conv2d_direct(inp, w, bias, 1, 1), gamma, beta, mean, var, eps,
                                      channel_axis=1)
        wf, bf = ops.bn_fold(w, bias, gamma, beta, mean, var, eps, dtype=np.float64)
        assert np.allclose(ops.conv2d_direct(inp, wf, bf, 1, 1), ref, rtol=1e-12, atol=1e-12)
    x = rng.normal(size=(7, 3 * 9))
    wl = w.reshape(4, -1)
    ref = ops.batchnorm_inference(ops.linear(x, wl, b), gamma, beta, mean, var, 1e-2)
    wf, bf = ops.bn_fold(wl, b, gamma, beta, mean, var, 1e-2, dtype=np.float64)
    assert np.allclose(ops.linear(x, wf, bf), ref, rtol=1e-12, atol=1e-12)


def test_bn_fold_worked_examples_fp32():
    g = load("bn_fold_worked.json")
    from oracle.formats import bf16_encode
    for case in g["cases"]:
        w = np.array(case["w"], np.float32)
        b = None if case["b"] is None else np.array(case["b"], np.float32)
        args = [np.array(case[k], np.float32) for k in ("gamma", "beta", "mean", "var")]
        wf, bf = ops.bn_fold(w, b, *args, np.float32(case["eps"]), dtype=np.float32)
        assert np.array_equal(bf16_encode(wf.astype(np.float64)), bf16_encode(np.array(case["w_out"])))
        assert np.array_equal(bf16_encode(bf.astype(np.float64)), bf16_encode(np.array(case["b_out"])))
        if "w_out_eps0" in case:
            wf0, bf0 = ops.bn_fold(w, b, *args, np.float32(0), dtype=np.float32)
            assert np.array_equal(wf0, np.array(case["w_out_eps0"], np.float32))
            assert np.array_equal(bf0, np.array(case["b_out_eps0"], np.float32))


def test_bn_fold_fp32_is_one_ieee_op_per_step():
    """The binary32 fold equals the same formula with every step computed in
    float64 and rounded once to binary32: for +, -, *, / and sqrt that double
    evaluation is correctly rounded because 53 >= 2*24 + 2 (Figueroa, "When is
    double rounding innocuous?", 1995).  A fused multiply-add, a reordered
    expression or a reciprocal-multiply in place of the division breaks it."""
    rng = np.random.default_rng(16)
    n = 4096
    w = rng.normal(0, 0.02, (n, 8)).astype(np.float32)
    b = rng.normal(0, 0.1, n).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, n).astype(np.float32)
    beta, mean = rng.normal(0, .1, n).astype(np.float32), rng.normal(0, .1, n).astype(np.float32)
    var = rng.uniform(0.01, 1, n).astype(np.float32)
    eps = np.float32(1e-2)
    wf, bf = ops.bn_fold(w, b, gamma, beta, mean, var, eps, dtype=np.float32)

    def r32(v):
        return np.asarray(v, np.float64).astype(np.float32).astype(np.float64)
    d = lambda a: np.asarray(a, np.float64)      # noqa: E731
    s = r32(d(gamma) / r32(np.sqrt(r32(d(var) + d(eps)))))
    assert np.array_equal(wf, r32(d(w) * s[:, None]).astype(np.float32))
    assert np.array_equal(bf, r32(r32(r32(d(b) - d(mean)) * s) + d(beta)).astype(np.float32))


# ------------------------------------------------------- static E4M3 quantiser

def test_quantiser_rounds_y_over_s_to_binary32_before_the_e4m3_decision():
    """The quantiser's input is the FP32 value a fused kernel holds (OpenPPL
    §6.2, HowTo §4.1: FP32 in registers, one conversion at the write).  Values
    placed within half a binary32 ulp (2**-24 at 1.0) of an E4M3 midpoint tell
    that reading from rounding the float64 y / s directly: 1.0625 + 2**-30 is a
    binary32 tie between 1.0 (code 0x38, even fraction) and 1.125 (0x39), so it
    goes to 0x38, while the float64 value lies above the midpoint (0x39);
    1.1875 - 2**-30 ties between 1.125 (0x39) and 1.25 (0x3A, even) and goes to
    0x3A, while the float64 value lies below (0x39).  With the descale 0.5
    (binary32-exact) the same values, halved, give the same codes; negated,
    the codes gain the sign bit."""
    y = np.array([1.0625 + 2.0 ** -30, 1.1875 - 2.0 ** -30])
    assert ops.quant_e4m3_static(y, 1.0).tolist() == [0x38, 0x3A]
    assert ops.quant_e4m3_static(y / 2, 0.5).tolist() == [0x38, 0x3A]
    assert ops.quant_e4m3_static(-y, 1.0).tolist() == [0xB8, 0xBA]
    # away from a midpoint the two readings agree: 1.0625 + 2**-20 is above the tie in binary32 too
    assert ops.quant_e4m3_static(np.array([1.0625 + 2.0 ** -20]), 1.0).tolist() == [0x39]


def test_quantiser_uses_the_binary32_descale():
    """s crosses the C boundary as a binary32: 0.05 is 0.0500000007..., so
    y = 0.05 * 448 in float64 lands just under 448 after the division and is
    still the largest code; y / s for a y past 448 s saturates (0x7E / 0xFE)."""
    s32 = float(np.float32(0.05))
    assert s32 != 0.05
    assert ops.quant_e4m3_static(np.array([448 * 0.05, 1e3, -1e3]), 0.05).tolist() == [0x7E, 0x7E, 0xFE]
    assert ops.quant_e4m3_static(np.array([448 * s32 * (1 + 2.0 ** -20)]), 0.05).tolist() == [0x7E]
