"""GPU parity of gbf_bn_fold: bit-exact against the oracle's binary32 fold."""
import numpy as np
import pytest
import torch

import workloads
from oracle import chains
from parity import from_bits, to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gbf():
    import fusion_add_rmsnorm_gb300 as g
    return g


def run(gbf, w_bits, b_bits, gamma, beta, mean, var, eps, inplace=False):
    w = from_bits(w_bits)
    out_ch = w.shape[0]
    b = None if b_bits is None else from_bits(b_bits)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()      # noqa: E731
    w_out = w if inplace else torch.empty_like(w)
    b_out = torch.empty(out_ch, dtype=torch.bfloat16, device="cuda")
    gbf.bn_fold(w, b, dev(gamma), dev(beta), dev(mean), dev(var), eps, w_out, b_out)
    torch.cuda.synchronize()
    return to_bits(w_out), to_bits(b_out)


def check(gbf, c, inplace=False):
    got = run(gbf, c["w"], c["bias"], c["gamma"], c["beta"], c["mean"], c["var"], c["eps"], inplace)
    ref = chains.bn_fold_bf16(c["w"], c["bias"], c["gamma"], c["beta"], c["mean"], c["var"], c["eps"])
    assert np.array_equal(got[0].reshape(ref[0].shape), ref[0]), f"W' mismatches: {np.sum(got[0] != ref[0])}"
    assert np.array_equal(got[1], ref[1]), "b' mismatch"


def test_linear_config_full_size(gbf):
    """W [16384, 4096] with the BN of its output channels, eps 1e-2: bit-exact."""
    c = workloads.linear_gelu_case(1, 16384, 4096, seed=0)
    check(gbf, c)


@pytest.mark.parametrize("out_ch,inner,bias", [(1, 8, True), (64, 27, True), (33, 147, False), (7, 4096, False),
                                               (100, 24, True), (3, 1, True)])
def test_shapes_conv_and_linear(gbf, out_ch, inner, bias):
    c = workloads.linear_gelu_case(1, out_ch, inner, seed=out_ch + inner, with_bias=bias)
    check(gbf, c)


def test_in_place(gbf):
    c = workloads.linear_gelu_case(1, 512, 1024, seed=2)
    check(gbf, c, inplace=True)


def test_worked_example_and_eps_sensitivity(gbf):
    import json, os
    from conftest import GOLDEN
    g = json.load(open(os.path.join(GOLDEN, "bn_fold_worked.json")))
    for case in g["cases"]:
        bits = lambda v: to_bits(torch.tensor(np.asarray(v, np.float32)).to(torch.bfloat16))   # noqa: E731
        got = run(gbf, bits(case["w"]), None if case["b"] is None else bits(case["b"]),
                  *[np.array(case[k], np.float32) for k in ("gamma", "beta", "mean", "var")], case["eps"])
        assert np.array_equal(got[0], bits(case["w_out"]))
        assert np.array_equal(got[1], bits(case["b_out"]))
