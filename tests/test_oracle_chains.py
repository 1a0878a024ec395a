"""Pins of the oracle's operator chains (bits in, bits out): the hand-derived
worked examples in tests/golden/, mode equivalences that must hold exactly, and
structural facts of the QKV post-processing (V passes through bit for bit,
positions 0 leave only the norm, cache slots permute rows)."""
import json
import os

import numpy as np
import torch

from conftest import GOLDEN
from oracle import chains, ops
from oracle.formats import bf16_decode, bf16_encode, e4m3_decode


def bits(v):
    """Exact bf16 bits of values that are representable (torch as a library encoder)."""
    t = torch.tensor(np.asarray(v, np.float32)).to(torch.bfloat16)
    assert np.array_equal(t.float().numpy(), np.asarray(v, np.float32)), "fixture value not bf16-exact"
    return t.view(torch.int16).numpy().view(np.uint16)


def test_add_rmsnorm_fp8_worked_examples():
    with open(os.path.join(GOLDEN, "rmsnorm_fp8_worked.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        kw = {}
        if "weight" in c:
            kw["weight"] = bits(c["weight"])
        if "gate" in c:
            kw.update(gate=bits(c["gate"]), ada_scale=bits(c["scale"]), ada_shift=bits(c["shift"]))
        res_out, q = chains.add_rmsnorm_fp8(bits(c["x"]), bits(c["res"]), c["eps"], c["s_q"], c["mode"], **kw)
        assert res_out.tolist() == c["res_out_bits"], c["name"]
        assert q.tolist() == c["q_codes"], c["name"]


def _rand_bits(rng, shape, mean=0.0, std=1.0):
    return bits(torch.tensor(rng.normal(mean, std, shape), dtype=torch.float32).to(torch.bfloat16).float().numpy())


def test_add_rmsnorm_mode_equivalences():
    rng = np.random.default_rng(20)
    x, res = _rand_bits(rng, (6, 64)), _rand_bits(rng, (6, 64))
    ones = bits(np.ones(64))
    zeros = bits(np.zeros(64))
    w_out = chains.add_rmsnorm_fp8(x, res, 1e-6, 0.05, chains.NORM_WEIGHT, weight=ones)
    nw_out = chains.add_rmsnorm_fp8(x, res, 1e-6, 0.05, chains.NORM_NOWEIGHT)
    ada0 = chains.add_rmsnorm_fp8(x, res, 1e-6, 0.05, chains.NORM_ADA, gate=ones, ada_scale=zeros,
                                  ada_shift=zeros)
    for a, b in [(w_out, nw_out), (w_out, ada0)]:
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # res_out is the bf16 of x + res, whatever the mode
    assert np.array_equal(w_out[0], bf16_encode(bf16_decode(x) + bf16_decode(res)))


def test_norm_reads_the_rounded_residual():
    """The norm consumes the bf16 residual it just wrote: feeding that residual
    back with x = 0 and gate = 1 (so r is exactly r_hat) reproduces every code."""
    rng = np.random.default_rng(28)
    x, res = _rand_bits(rng, (32, 512)), _rand_bits(rng, (32, 512))
    gate, scale, shift = _rand_bits(rng, 512, 0, .2), _rand_bits(rng, 512, 0, .2), _rand_bits(rng, 512, 0, .2)
    res_out, q = chains.add_rmsnorm_fp8(x, res, 1e-6, 0.05, chains.NORM_ADA, gate=gate, ada_scale=scale,
                                        ada_shift=shift)
    zero = bits(np.zeros((32, 512)))
    ones = bits(np.ones(512))
    res2, q2 = chains.add_rmsnorm_fp8(zero, res_out, 1e-6, 0.05, chains.NORM_ADA, gate=ones, ada_scale=scale,
                                      ada_shift=shift)
    assert np.array_equal(res2, res_out) and np.array_equal(q2, q)


def test_add_rmsnorm_codes_dequantise_close_to_y():
    """code * s is within half an E4M3 step of y (relative 2^-4) wherever y/s is normal."""
    rng = np.random.default_rng(21)
    x, res = _rand_bits(rng, (4, 256)), _rand_bits(rng, (4, 256))
    w = _rand_bits(rng, 256, 1.0, 0.1)
    _, q = chains.add_rmsnorm_fp8(x, res, 1e-6, 0.05, chains.NORM_WEIGHT, weight=w)
    r_hat = bf16_decode(bf16_encode(bf16_decode(x) + bf16_decode(res)))
    y = r_hat / np.sqrt((r_hat ** 2).mean(axis=1, keepdims=True) + 1e-6) * bf16_decode(w)
    deq = e4m3_decode(q) * np.float64(np.float32(0.05))
    normal = np.abs(y / 0.05) >= 2 ** -6
    assert np.all(np.abs(deq - y)[normal] <= np.abs(y)[normal] * 2 ** -4 + 1e-12)


def test_unfused_bf16_y_variant_differs_only_slightly():
    rng = np.random.default_rng(22)
    x, res = _rand_bits(rng, (64, 256)), _rand_bits(rng, (64, 256))
    w = _rand_bits(rng, 256, 1.0, 0.1)
    _, q = chains.add_rmsnorm_fp8(x, res, 1e-6, 0.05, 0, weight=w)
    _, q2 = chains.add_rmsnorm_fp8(x, res, 1e-6, 0.05, 0, weight=w, round_y_bf16=True)
    frac = np.mean(q != q2)
    assert 0 < frac < 0.2


def _qkv(rng, t, hq, hkv, d):
    return _rand_bits(rng, (t, (hq + 2 * hkv) * d))


def test_qkv_position_zero_leaves_only_the_norm_and_v_is_copied():
    rng = np.random.default_rng(23)
    t, hq, hkv, d = 5, 4, 2, 16
    qkv = _qkv(rng, t, hq, hkv, d)
    qw, kw = _rand_bits(rng, d, 1, .1), _rand_bits(rng, d, 1, .1)
    q, kc, vc = chains.qkv_split_norm_rope(qkv, hq, hkv, d, 0, qw, kw, 1e-6, 0, np.zeros(t, np.int32), 1e6)
    qv, kv, vv = ops.split_packed_qkv(bf16_decode(qkv), hq, hkv, d)
    assert np.array_equal(q, bf16_encode(ops.qk_rmsnorm_per_head(qv, bf16_decode(qw), 1e-6)))
    assert np.array_equal(kc, bf16_encode(ops.qk_rmsnorm_per_head(kv, bf16_decode(kw), 1e-6)))
    _, _, vbits = ops.split_packed_qkv(qkv, hq, hkv, d)
    assert np.array_equal(vc, vbits)


def test_qkv_rotation_reaches_q_and_k_but_not_v():
    """Away from position 0 the Q and K outputs are rotations of the norm-only
    outputs: every rotate_half pair keeps its norm (to bf16 rounding) while the
    values change; V stays the input bits."""
    rng = np.random.default_rng(27)
    t, hq, hkv, d = 8, 2, 2, 32
    qkv = _qkv(rng, t, hq, hkv, d)
    qw, kw = _rand_bits(rng, d, 1, .1), _rand_bits(rng, d, 1, .1)
    pos = np.arange(1, t + 1, dtype=np.int32) * 37
    zero = chains.qkv_split_norm_rope(qkv, hq, hkv, d, 0, qw, kw, 1e-6, 0, np.zeros(t, np.int32), 1e4)
    rot = chains.qkv_split_norm_rope(qkv, hq, hkv, d, 0, qw, kw, 1e-6, 0, pos, 1e4)
    for a, b in zip(zero[:2], rot[:2]):
        av, bv = bf16_decode(a), bf16_decode(b)
        assert np.mean(a != b) > 0.5
        na = av[..., :d // 2] ** 2 + av[..., d // 2:] ** 2
        nb = bv[..., :d // 2] ** 2 + bv[..., d // 2:] ** 2
        assert np.allclose(na, nb, rtol=2e-2, atol=1e-3)
    assert np.array_equal(zero[2], rot[2])


def test_qkv_layernorm_constant_heads_give_their_own_bias():
    """LayerNorm mode: a head whose values are all equal normalises to its
    bias exactly, and position 0 does not rotate, so Q carries q_b and K
    carries k_b bit for bit (each head its own constant); V is copied."""
    rng = np.random.default_rng(31)
    t, hq, hkv, d = 3, 2, 2, 16
    consts = rng.normal(size=(t, hq + 2 * hkv, 1))
    qkv = bf16_encode(np.broadcast_to(consts, (t, hq + 2 * hkv, d)).reshape(t, -1))
    qw, kw = _rand_bits(rng, d, 1, .1), _rand_bits(rng, d, 1, .1)
    qb, kb = _rand_bits(rng, d, 0, .5), _rand_bits(rng, d, 0, .5)
    q, kc, vc = chains.qkv_split_norm_rope(qkv, hq, hkv, d, chains.QKNORM_LAYERNORM, qw, kw, 1e-5, 0,
                                           np.zeros(t, np.int32), 1e4, q_b=qb, k_b=kb)
    assert np.array_equal(q, np.broadcast_to(qb, q.shape))
    assert np.array_equal(kc, np.broadcast_to(kb, kc.shape))
    assert np.array_equal(vc, qkv.reshape(t, hq + 2 * hkv, d)[:, hq + hkv:])
    q0, k0, _ = chains.qkv_split_norm_rope(qkv, hq, hkv, d, chains.QKNORM_LAYERNORM, qw, kw, 1e-5, 0,
                                           np.zeros(t, np.int32), 1e4)
    assert not q0.any() and not k0.any()             # no bias: exactly zero


def test_gated_act_splits_gate_then_up_and_rounds_once():
    """The first half of each row is the gate, the second the up projection:
    with up = 1 the output is bf16(act(gate)) and with gate = 1 it is
    bf16(act(1) * up); rows are independent."""
    rng = np.random.default_rng(41)
    d = 8
    gate = _rand_bits(rng, (3, d))
    up = _rand_bits(rng, (3, d))
    ones = bf16_encode(np.ones((3, d)))
    for act in (ops.ACT_GELU_TANH, ops.ACT_GELU_ERF, ops.ACT_SILU):
        y = chains.gated_act(np.concatenate([gate, ones], axis=1), d, act)
        assert np.array_equal(y, bf16_encode(ops.activation(bf16_decode(gate), act)))
        y = chains.gated_act(np.concatenate([ones, up], axis=1), d, act)
        assert np.array_equal(y, bf16_encode(ops.activation(1.0, act) * bf16_decode(up)))
    both = chains.gated_act(np.concatenate([gate, up], axis=1), d, ops.ACT_SILU)
    assert np.array_equal(both[1:2], chains.gated_act(np.concatenate([gate, up], axis=1)[1:2], d, ops.ACT_SILU))


def test_linear_fp8_act_decodes_codes_and_applies_scales():
    """Codes decode through the E4M3 table: 0x38 = 1.0, 0x40 = 2.0, 0xB8 = -1.0,
    0x00 = 0; a hand-summed 1 x 2 by 2 x 2 case, then the activation."""
    xq = np.array([[0x38, 0x40]], np.uint8)                   # (1, 2)
    wq = np.array([[0x38, 0xB8], [0x40, 0x00]], np.uint8)     # rows (1, -1), (2, 0)
    y = chains.linear_fp8_act(xq, 0.5, wq, np.array([1.0, 0.25], np.float32))
    # row 0: 0.5 * (1*1 + 2*(-1)) * 1.0 = -0.5; row 1: 0.5 * (1*2 + 0) * 0.25 = 0.25
    assert bf16_decode(y).tolist() == [[-0.5, 0.25]]
    b = bf16_encode(np.array([1.0, -1.0]))
    y = chains.linear_fp8_act(xq, 0.5, wq, np.array([1.0, 0.25], np.float32), b, act=ops.ACT_SILU)
    assert np.array_equal(y, bf16_encode(ops.silu(np.array([[0.5, -0.75]]))))


def test_fold_norm_weight_bf16_rounds_once_in_binary32():
    rng = np.random.default_rng(44)
    w, g = _rand_bits(rng, (3, 16), 0, .05), _rand_bits(rng, 16, 0, .2)
    out = chains.fold_norm_weight_bf16(w, g)
    wf = bf16_decode(w).astype(np.float32)
    gf = bf16_decode(g).astype(np.float32)
    via_torch = (torch.from_numpy(wf) * (1.0 + torch.from_numpy(gf))).numpy()   # binary32 add, then multiply
    assert np.array_equal(out, bf16_encode(via_torch.astype(np.float64)))


def test_qkv_slots_permute_cache_rows():
    rng = np.random.default_rng(24)
    t, hq, hkv, d = 6, 2, 1, 8
    qkv = _qkv(rng, t, hq, hkv, d)
    qw, kw = _rand_bits(rng, d, 1, .1), _rand_bits(rng, d, 1, .1)
    pos = np.arange(t, dtype=np.int32)
    q0, k0, v0 = chains.qkv_split_norm_rope(qkv, hq, hkv, d, 0, qw, kw, 1e-6, 0, pos, 1e4)
    slots = np.array([9, 3, 0, 7, 1, 5])
    q1, k1, v1 = chains.qkv_split_norm_rope(qkv, hq, hkv, d, 0, qw, kw, 1e-6, 0, pos, 1e4, slots=slots,
                                            cache_rows=10)
    assert np.array_equal(q0, q1)
    assert np.array_equal(k1[slots], k0) and np.array_equal(v1[slots], v0)
    untouched = np.setdiff1d(np.arange(10), slots)
    assert not k1[untouched].any() and not v1[untouched].any()


def test_qkv_full_width_3d_single_section_matches_1d():
    rng = np.random.default_rng(25)
    t, h, d = 4, 3, 16
    qkv = _qkv(rng, t, h, h, d)
    qw, kw = _rand_bits(rng, h * d, 1, .1), _rand_bits(rng, h * d, 1, .1)
    pos3 = rng.integers(0, 40, (t, 3)).astype(np.int32)
    a = chains.qkv_split_norm_rope(qkv, h, h, d, 1, qw, kw, 1e-6, 1, pos3, 1e4, sections=(16, 0, 0))
    b = chains.qkv_split_norm_rope(qkv, h, h, d, 1, qw, kw, 1e-6, 0, pos3[:, 0], 1e4)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_linear_bias_gelu_brute_force_tiny():
    rng = np.random.default_rng(26)
    m, n, k = 3, 4, 8
    x, w, b = _rand_bits(rng, (m, k)), _rand_bits(rng, (n, k), 0, .3), _rand_bits(rng, n, 0, .1)
    y = chains.linear_bias_gelu(x, w, b)
    xv, wv, bv = bf16_decode(x), bf16_decode(w), bf16_decode(b)
    for i in range(m):
        for j in range(n):
            a = bv[j] + sum(xv[i, kk] * wv[j, kk] for kk in range(k))
            g = 0.5 * a * (1 + np.tanh(0.7978845608 * (a + 0.044715 * a ** 3)))
            assert y[i, j] == bf16_encode(g)
    # no activation: plain Linear rounded to bf16, compared with torch fp64
    y0 = chains.linear_bias_gelu(x, w, b, act_gelu=False)
    lib = torch.nn.functional.linear(torch.from_numpy(xv), torch.from_numpy(wv), torch.from_numpy(bv)).numpy()
    assert np.array_equal(y0, bf16_encode(lib))
    # the other epilogue activations, against torch's fp64 ones on the same Linear
    t = torch.from_numpy(lib)
    for act, ref in ((ops.ACT_GELU_ERF, torch.nn.functional.gelu(t, approximate="none")),
                     (ops.ACT_SILU, torch.nn.functional.silu(t))):
        assert np.array_equal(chains.linear_bias_gelu(x, w, b, act=act), bf16_encode(ref.numpy()))


def test_bn_fold_bf16_chain_worked_example():
    with open(os.path.join(GOLDEN, "bn_fold_worked.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        b = None if c["b"] is None else bits(c["b"])
        wb, bb = chains.bn_fold_bf16(bits(c["w"]), b, *[np.array(c[k], np.float32) for k in
                                                          ("gamma", "beta", "mean", "var")], c["eps"])
        assert np.array_equal(wb, bits(c["w_out"]))
        assert np.array_equal(bb, bits(c["b_out"]))
