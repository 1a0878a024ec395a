"""The Python binding's operand checks, on the host: a raw pointer carries no
size, so every wrapper checks each operand's extent against the call's
before it reaches the C ABI.  The tensors here live in host memory, so a
check that let one through would stop at "must be on a CUDA device" instead
of naming the mismatched operand; no kernel is launched."""
import pytest
import torch


@pytest.fixture(scope="module")
def gbf():
    import fusion_add_rmsnorm_gb300 as g
    return g


bf = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)     # noqa: E731
u8 = lambda *s: torch.zeros(*s, dtype=torch.uint8)        # noqa: E731
i32 = lambda *s: torch.zeros(*s, dtype=torch.int32)       # noqa: E731
f32 = lambda *s: torch.zeros(*s, dtype=torch.float32)     # noqa: E731


def raises(match, fn, *a, **k):
    with pytest.raises(ValueError, match=match):
        fn(*a, **k)


def test_add_rmsnorm_operand_extents(gbf):
    x, r, o, q = bf(4, 64), bf(4, 64), bf(4, 64), u8(4, 64)
    f = gbf.add_rmsnorm_fp8
    raises("res_in", f, x, bf(4, 56), o, q, 1)
    raises("res_out", f, x, r, bf(3, 64), q, 1)
    raises("q_out", f, x, r, o, u8(4, 63), 1)
    raises("weight", f, x, r, o, q, 0, weight=bf(32))
    raises("gate", f, x, r, o, q, 1, gate=bf(65))
    raises("ada_scale", f, x, r, o, q, 2, ada_scale=bf(8), ada_shift=bf(64))
    raises("ada_shift", f, x, r, o, q, 2, ada_scale=bf(64), ada_shift=bf(128))
    raises("CUDA device", f, x, r, o, q, 0, weight=bf(64))      # every extent right: the device check speaks


def test_qkv_operand_extents(gbf):
    t, hq, hkv, d = 6, 4, 2, 64
    qkv, qo, kc, vc, pos = bf(t, (hq + 2 * hkv) * d), bf(t, hq, d), bf(t, hkv, d), bf(t, hkv, d), i32(t)
    w = bf(d)
    f = gbf.qkv_split_norm_rope
    raises("qkv", f, bf(t, 7 * d), hq, hkv, d, 0, w, w, 1e-6, 0, pos, 1e4, qo, kc, vc)
    raises("q_w", f, qkv, hq, hkv, d, 0, bf(2 * d), w, 1e-6, 0, pos, 1e4, qo, kc, vc)
    raises("k_w", f, qkv, hq, hkv, d, 1, bf(hq * d), w, 1e-6, 0, pos, 1e4, qo, kc, vc)
    raises("pos", f, qkv, hq, hkv, d, 0, w, w, 1e-6, 0, i32(t - 1), 1e4, qo, kc, vc)
    raises("pos", f, qkv, hq, hkv, d, 0, w, w, 1e-6, 1, pos, 1e4, qo, kc, vc, sections=(22, 22, 20))
    raises("sections", f, qkv, hq, hkv, d, 0, w, w, 1e-6, 1, i32(t, 3), 1e4, qo, kc, vc, sections=(32, 32))
    raises("q_out", f, qkv, hq, hkv, d, 0, w, w, 1e-6, 0, pos, 1e4, bf(t, hq - 1, d), kc, vc)
    raises("slots", f, qkv, hq, hkv, d, 0, w, w, 1e-6, 0, pos, 1e4, qo, kc, vc, slots=i32(t + 1))
    raises("k_cache", f, qkv, hq, hkv, d, 0, w, w, 1e-6, 0, pos, 1e4, qo, kc, vc, cache_rows=t + 1)
    raises("v_cache", f, qkv, hq, hkv, d, 0, w, w, 1e-6, 0, pos, 1e4, qo, kc, bf(t - 1, hkv, d))
    raises("CUDA device", f, qkv, hq, hkv, d, 0, w, w, 1e-6, 0, pos, 1e4, qo, kc, vc)
    g = gbf.qkv_split_layernorm_rope
    raises("q_b", g, qkv, hq, hkv, d, w, bf(d + 8), w, None, 1e-5, pos, 1e4, qo, kc, vc)
    raises("k_w", g, qkv, hq, hkv, d, w, None, bf(8), None, 1e-5, pos, 1e4, qo, kc, vc)
    raises("CUDA device", g, qkv, hq, hkv, d, w, w, w, w, 1e-5, pos, 1e4, qo, kc, vc)


def test_linear_operand_extents(gbf):
    m, n, k = 8, 32, 64
    x, w, b, y = bf(m, k), bf(n, k), bf(n), bf(m, n)
    f = gbf.linear_bias_gelu
    raises("w", f, x, bf(n, k + 64), b, y)
    raises("w", f, x, bf(n * k), b, y)
    raises("bias", f, x, w, bf(n - 16), y)
    raises("y", f, x, w, b, bf(m, n + 16))
    raises("CUDA device", f, x, w, b, y)
    g = gbf.linear_fp8_act
    xq, wq, ws = u8(m, 128), u8(n, 128), f32(n)
    raises("wq", g, xq, 0.05, u8(n, 256), ws, b, y)
    raises("w_scale", g, xq, 0.05, wq, f32(n + 1), b, y)
    raises("y", g, xq, 0.05, wq, ws, b, bf(m - 1, n))
    raises("CUDA device", g, xq, 0.05, wq, ws, b, y)


def test_fold_and_activation_operand_extents(gbf):
    w = bf(16, 64)
    raises("gamma", gbf.fold_norm_weight, w, bf(16), bf(16, 64))
    raises("w_out", gbf.fold_norm_weight, w, bf(64), bf(16, 32))
    v = f32(16)
    raises("gamma", gbf.bn_fold, w, bf(16), f32(15), v, v, v, 1e-2, bf(16, 64), bf(16))
    raises("var", gbf.bn_fold, w, None, v, v, v, f32(64), 1e-2, bf(16, 64), bf(16))
    raises("b_out", gbf.bn_fold, w, None, v, v, v, v, 1e-2, bf(16, 64), bf(8))
    raises("w_out", gbf.bn_fold, w, None, v, v, v, v, 1e-2, bf(16, 65), bf(16))
    raises("CUDA device", gbf.bn_fold, w, None, v, v, v, v, 1e-2, bf(16, 64), bf(16))
    raises("x", gbf.gated_act, bf(4, 64), bf(4, 16))
    raises("x", gbf.gated_act, bf(8, 32), bf(4, 32))
    raises("CUDA device", gbf.gated_act, bf(4, 64), bf(4, 32))
    raises("copy of", gbf.copy, u8(64), u8(32))
    raises("copy of", gbf.copy, u8(64), u8(64), 128)


def test_non_tensor_operand_is_a_type_error(gbf):
    with pytest.raises(TypeError, match="res_in"):
        gbf.add_rmsnorm_fp8(bf(2, 8), [0.0] * 16, bf(2, 8), u8(2, 8), 1)
