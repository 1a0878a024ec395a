"""GPU parity of gbf_linear_fp8_act (E4M3 x E4M3 on tcgen05 with descales,
bias and activation) and of gbf_fold_norm_weight (bit-exact) against the
oracle."""
import numpy as np
import pytest
import torch

import workloads
from oracle import chains, ops
from parity import assert_bf16_close, from_bits, to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gbf():
    import fusion_add_rmsnorm_gb300 as g
    return g


def e4m3_codes(v):
    """Input codes: torch's CPU E4M3 conversion (nearest even) after clamping
    to the finite range; the oracle decodes whatever codes it is given."""
    t = torch.from_numpy(np.ascontiguousarray(v, np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def codes(c):
    """E4M3 codes of the case's activations and weights."""
    xq = e4m3_codes(np.asarray(c["x"], np.float32) / np.float32(c["x_scale"]))
    wq = e4m3_codes(np.asarray(c["w"], np.float32) / c["w_scale"][:, None])
    return xq, wq


def run_gpu(gbf, c, xq, wq, act, with_bias=True):
    y = torch.empty(c["m"], c["n"], dtype=torch.bfloat16, device="cuda")
    gbf.linear_fp8_act(torch.from_numpy(xq).cuda(), float(np.float32(c["x_scale"])), torch.from_numpy(wq).cuda(),
                       torch.from_numpy(c["w_scale"]).cuda(), from_bits(c["bias"]) if with_bias else None, y, act=act)
    torch.cuda.synchronize()
    return to_bits(y)


@pytest.mark.parametrize("m,n,k", [(128, 256, 128), (256, 512, 512), (200, 272, 384), (1, 16, 128),
                                   (129, 256, 1024), (300, 784, 256), (1152, 4352, 256), (256, 16, 128),
                                   (384, 48, 128), (64, 4096, 512)])
@pytest.mark.parametrize("act", [ops.ACT_GELU_TANH, 0, ops.ACT_GELU_ERF, ops.ACT_SILU])
def test_shapes_and_activations(gbf, m, n, k, act):
    c = workloads.fp8_linear_case(m, n, k, seed=m + n + k)
    xq, wq = codes(c)
    y = run_gpu(gbf, c, xq, wq, act)
    ref = chains.linear_fp8_act(xq, np.float32(c["x_scale"]), wq, c["w_scale"], c["bias"],
                                act=None if act == 0 else act)
    assert_bf16_close(y, ref, f"fp8 linear [{m},{n},{k}] act {act}")


def test_no_bias(gbf):
    c = workloads.fp8_linear_case(256, 256, 256, seed=5)
    xq, wq = codes(c)
    y = run_gpu(gbf, c, xq, wq, ops.ACT_GELU_TANH, with_bias=False)
    assert_bf16_close(y, chains.linear_fp8_act(xq, np.float32(c["x_scale"]), wq, c["w_scale"], None,
                                               act=ops.ACT_GELU_TANH), "no bias")


def test_config_sampled_rows(gbf):
    """8192 x 16384 x 4096 in the bench's launch configuration; the oracle
    checks every column of 48 sampled rows."""
    c = workloads.fp8_linear_case(8192, 16384, 4096, seed=0)
    xq, wq = codes(c)
    y = run_gpu(gbf, c, xq, wq, ops.ACT_GELU_TANH)
    rows = np.unique(np.concatenate([[0, 8191], np.random.default_rng(4).choice(8192, 46, replace=False)]))
    ref = chains.linear_fp8_act(xq[rows], np.float32(c["x_scale"]), wq, c["w_scale"], c["bias"],
                                act=ops.ACT_GELU_TANH)
    assert_bf16_close(y[rows], ref, "fp8 linear config rows")


@pytest.mark.parametrize("out_ch,inner", [(1, 8), (7, 64), (33, 1000), (16, 4096), (5, 27)])
@pytest.mark.parametrize("gemma", [True, False])
def test_fold_norm_weight_bit_exact(gbf, out_ch, inner, gemma):
    c = workloads.norm_fold_case(out_ch, inner, seed=out_ch + inner)
    w = from_bits(c["w"])
    out = torch.empty_like(w)
    gbf.fold_norm_weight(w, from_bits(c["gamma"]), out, gemma_style=gemma)
    torch.cuda.synchronize()
    assert np.array_equal(to_bits(out), chains.fold_norm_weight_bf16(c["w"], c["gamma"], gemma))


def test_fold_norm_weight_in_place(gbf):
    c = workloads.norm_fold_case(64, 512, seed=3)
    w = from_bits(c["w"])
    gbf.fold_norm_weight(w, from_bits(c["gamma"]), w)
    torch.cuda.synchronize()
    assert np.array_equal(to_bits(w), chains.fold_norm_weight_bf16(c["w"], c["gamma"]))
