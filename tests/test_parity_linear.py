"""GPU parity of gbf_linear_bias_gelu (tcgen05 GEMM + bias + GELU epilogue)
against the oracle's unfused Linear -> BiasAdd -> GELU(tanh) in float64."""
import numpy as np
import pytest
import torch

import workloads
from oracle import chains, ops
from oracle.formats import bf16_decode, bf16_encode
from parity import assert_bf16_close, from_bits, to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gbf():
    import fusion_add_rmsnorm_gb300 as g
    return g


def run(gbf, x_bits, w_bits, b_bits, act=1):
    x, w = from_bits(x_bits), from_bits(w_bits)
    b = None if b_bits is None else from_bits(b_bits)
    y = torch.full((x.shape[0], w.shape[0]), float("nan"), dtype=torch.bfloat16, device="cuda")
    gbf.linear_bias_gelu(x, w, b, y, act)
    torch.cuda.synchronize()
    s, msg = gbf.device_status()
    assert s == gbf.OK, msg
    return to_bits(y)


@pytest.mark.parametrize("m,n,k", [(128, 256, 64), (256, 512, 256), (200, 256, 128), (130, 272, 192), (1, 16, 64),
                                   (384, 768, 1024), (1000, 2064, 512), (1152, 4352, 256),
                                   (256, 16, 64), (384, 48, 128), (257, 80, 64),
                                   (32, 4096, 512), (100, 2320, 256)])
def test_shapes(gbf, m, n, k):
    c = workloads.linear_gelu_case(m, n, k, seed=m + n + k)
    y = run(gbf, c["x"], c["w"], c["bias"])
    assert_bf16_close(y, chains.linear_bias_gelu(c["x"], c["w"], c["bias"]), f"[{m},{n},{k}]")


def test_no_bias_and_no_activation(gbf):
    c = workloads.linear_gelu_case(256, 512, 320, seed=7, with_bias=False)
    assert_bf16_close(run(gbf, c["x"], c["w"], None), chains.linear_bias_gelu(c["x"], c["w"], None), "no bias")
    c = workloads.linear_gelu_case(256, 512, 320, seed=8)
    assert_bf16_close(run(gbf, c["x"], c["w"], c["bias"], act=0),
                      chains.linear_bias_gelu(c["x"], c["w"], c["bias"], act_gelu=False), "no activation")


def test_linear_config_sampled_rows(gbf):
    """X [8192, 4096] . W [16384, 4096]^T + b, GELU: the oracle checks every
    column of 64 sampled rows (first, last, random)."""
    c = workloads.config_linear_gelu()
    y = run(gbf, c["x"], c["w"], c["bias"])
    rows = np.unique(np.concatenate([[0, 127, 128, 8191], np.random.default_rng(0).choice(8192, 60, replace=False)]))
    ref = chains.linear_bias_gelu(c["x"][rows], c["w"], c["bias"])
    assert_bf16_close(y[rows], ref, "8192x16384x4096 sampled rows")


def test_folded_weights_match_linear_then_bn(gbf):
    """GEMM(W', b') with the BN folded by gbf_bn_fold matches the oracle's
    Linear -> BatchNorm -> GELU on the unfolded weights (M = 256)."""
    c = workloads.linear_gelu_case(256, 1024, 512, seed=3)
    w = from_bits(c["w"])
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()      # noqa: E731
    wf = torch.empty_like(w)
    bf = torch.empty(1024, dtype=torch.bfloat16, device="cuda")
    gbf.bn_fold(w, from_bits(c["bias"]), f32(c["gamma"]), f32(c["beta"]), f32(c["mean"]), f32(c["var"]), c["eps"],
                wf, bf)
    y = run(gbf, c["x"], to_bits(wf), to_bits(bf))
    lin = ops.linear(bf16_decode(c["x"]), bf16_decode(c["w"]), bf16_decode(c["bias"]))
    ref = bf16_encode(ops.gelu_tanh(ops.batchnorm_inference(lin, c["gamma"], c["beta"], c["mean"], c["var"],
                                                            c["eps"])))
    assert_bf16_close(y, ref, "fold + GEMM vs Linear -> BN -> GELU")
