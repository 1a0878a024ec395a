"""The cross-layer loop end to end on the GPU: the `_noweight` add + RMSNorm
writes E4M3 codes, the norm's weight (1 + gamma) is pre-folded into the next
Linear's columns, and the E4M3 Linear + GELU consumes the codes directly
(FlashRT §2.1: `_noweight`, the weight taken into the next GEMM; §3: the last
operator of layer N writes FP8 for layer N + 1).  Three entry points in
sequence, gbf_add_rmsnorm_fp8 (NOWEIGHT) -> gbf_fold_norm_weight ->
gbf_linear_fp8_act, against the oracle's composition of the same operators.

The folded weight is quantised to E4M3 per output row between the fold and
the GEMM; no entry point of the library does that (a weight is quantised once,
at load time), so each side uses its own encoder: torch's E4M3 conversion of
the binary32 quotient on the GPU side, the oracle's encoder of the float64
quotient rounded to binary32 on the oracle side.  The two quotients are
identical (a correctly rounded binary32 division equals the float64 quotient
rounded once), and the fold is bit-exact, so both sides feed the GEMM the
same weight codes."""
import numpy as np
import pytest
import torch

import workloads
from oracle import chains, formats, ops
from parity import assert_bf16_close, assert_fp8_codes, from_bits, to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gbf():
    import fusion_add_rmsnorm_gb300 as g
    return g


def gpu_loop(gbf, c):
    x, res = from_bits(c["x"]), from_bits(c["res"])
    res_out = torch.empty_like(res)
    q = torch.empty(res.shape, dtype=torch.uint8, device="cuda")
    gbf.add_rmsnorm_fp8(x, res, res_out, q, gbf.NORM_NOWEIGHT, eps=c["eps"], fp8_scale=c["x_scale"])
    w = from_bits(c["w"])
    w_fold = torch.empty_like(w)
    gbf.fold_norm_weight(w, from_bits(c["gamma"]), w_fold, gemma_style=True)
    ws = torch.from_numpy(c["w_scale"]).cuda()
    wq = (w_fold.float() / ws[:, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    y = torch.empty(c["rows"], c["n_out"], dtype=torch.bfloat16, device="cuda")
    gbf.linear_fp8_act(q, float(np.float32(c["x_scale"])), wq, ws, from_bits(c["bias"]), y, act=gbf.ACT_GELU_TANH)
    torch.cuda.synchronize()
    return to_bits(res_out), to_bits(q), to_bits(w_fold), to_bits(y)


def weight_codes(w_bits, w_scale):
    return formats.e4m3_encode_sat((formats.bf16_decode(w_bits) / w_scale[:, None].astype(np.float64))
                                   .astype(np.float32))


def oracle_loop(c):
    res_out, q = chains.add_rmsnorm_fp8(c["x"], c["res"], c["eps"], c["x_scale"], chains.NORM_NOWEIGHT)
    w_fold = chains.fold_norm_weight_bf16(c["w"], c["gamma"], gemma_style=True)
    y = chains.linear_fp8_act(q, np.float32(c["x_scale"]), weight_codes(w_fold, c["w_scale"]), c["w_scale"],
                              c["bias"], act=ops.ACT_GELU_TANH)
    return res_out, q, w_fold, y


@pytest.mark.parametrize("rows,hidden,n_out", [(10, 1024, 2048), (256, 4096, 1024), (333, 2048, 784)])
def test_noweight_codes_into_the_folded_fp8_linear(gbf, rows, hidden, n_out):
    c = workloads.cross_layer_case(rows, hidden, n_out, seed=rows + hidden)
    g_res, g_q, g_w, g_y = gpu_loop(gbf, c)
    o_res, o_q, o_w, o_y = oracle_loop(c)
    assert_bf16_close(g_res, o_res, "residual")
    assert_fp8_codes(g_q, o_q, "activation codes")
    assert np.array_equal(g_w, o_w), "folded weight not bit-exact"
    assert_bf16_close(g_y, o_y, "Linear + GELU output")


def test_loop_loses_no_accuracy_against_the_weighted_chain(gbf):
    """FlashRT's acceptance rule for a fusion: against the exact float64
    result of the layer (RMSNorm with weight 1 + gamma, then Linear + bias +
    GELU on the unquantised W), the fused loop's output is as close as the
    unfused chain it replaces: a weighted RMSNorm whose y is stored in bf16,
    quantised to E4M3, then the E4M3 Linear on the unfolded W.  The two put
    the same two quantisations in different places, so their cosines differ
    by sampling noise (about 1e-5 at this size, either sign); the fused loop
    may not fall below the chain by more than 1e-4."""
    c = workloads.cross_layer_case(64, 4096, 2048, seed=7)
    _, _, _, g_y = gpu_loop(gbf, c)
    r_hat = formats.bf16_decode(chains.add_rmsnorm_fp8(c["x"], c["res"], c["eps"], c["x_scale"], 1)[0])
    scale = 1.0 + formats.bf16_decode(c["gamma"])
    exact = ops.activation(ops.linear(ops.rmsnorm(r_hat, c["eps"]) * scale[None, :], formats.bf16_decode(c["w"]),
                                      formats.bf16_decode(c["bias"])), ops.ACT_GELU_TANH).ravel()
    _, q_chain = chains.add_rmsnorm_fp8(c["x"], c["res"], c["eps"], c["x_scale"], chains.NORM_WEIGHT,
                                        weight=formats.bf16_encode(scale), round_y_bf16=True)
    y_chain = chains.linear_fp8_act(q_chain, np.float32(c["x_scale"]), weight_codes(c["w"], c["w_scale"]),
                                    c["w_scale"], c["bias"], act=ops.ACT_GELU_TANH)

    def cos(bits):
        v = formats.bf16_decode(bits).ravel()
        return float(v @ exact / np.linalg.norm(v) / np.linalg.norm(exact))
    assert cos(g_y) >= cos(y_chain) - 1e-4, (cos(g_y), cos(y_chain))
    assert cos(g_y) > 0.999
