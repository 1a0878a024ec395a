"""GPU parity of gbf_gated_act (act(gate) * up over [gate | up] rows) and of
the GEMM epilogue's erf GELU and SiLU against the oracle."""
import numpy as np
import pytest
import torch

import workloads
from oracle import chains, ops
from parity import assert_bf16_close, from_bits, to_bits

pytestmark = pytest.mark.gpu

ACTS = {"silu": ops.ACT_SILU, "gelu_tanh": ops.ACT_GELU_TANH, "gelu_erf": ops.ACT_GELU_ERF}


@pytest.fixture(scope="module")
def gbf():
    import fusion_add_rmsnorm_gb300 as g
    return g


def run_gpu(gbf, c, act):
    x = from_bits(c["x"])
    y = torch.empty(c["rows"], c["d"], dtype=torch.bfloat16, device="cuda")
    gbf.gated_act(x, y, act)
    torch.cuda.synchronize()
    return to_bits(y)


@pytest.mark.parametrize("name", list(ACTS))
@pytest.mark.parametrize("rows,d", [(1, 8), (3, 64), (37, 1032), (5, 4096), (300, 11008), (2, 2056),
                                    (8, 11008), (32, 11008), (151, 1032)])
def test_shapes(gbf, name, rows, d):
    c = workloads.gated_act_case(rows, d, seed=rows + d)
    y = run_gpu(gbf, c, ACTS[name])
    assert_bf16_close(y, chains.gated_act(c["x"], d, ACTS[name]), f"{name} [{rows},{d}]")


@pytest.mark.parametrize("name", list(ACTS))
def test_swiglu_ffn_config_sampled_rows(gbf, name):
    """[4096, 2*11008] in the bench's launch configuration; the oracle checks
    the first, last and 62 random rows."""
    c = workloads.config_swiglu_ffn()
    y = run_gpu(gbf, c, ACTS[name])
    rows = np.unique(np.concatenate([[0, 4095], np.random.default_rng(2).choice(4096, 62, replace=False)]))
    assert_bf16_close(y[rows], chains.gated_act(c["x"][rows], 11008, ACTS[name]), f"{name} sampled")


def test_extreme_gates(gbf):
    """Gates far into both tails: SiLU and GELU go to the gate itself or to
    zero (signed), with no NaN; up = 1 isolates the activation."""
    d = 16
    g = np.array([-1e4, -100, -30, -10, -1, -1e-3, 0, 1e-3, 1, 10, 30, 100, 1e4, 3e38, -3e38, 2], np.float32)
    gb = torch.from_numpy(g).to(torch.bfloat16)
    x = torch.cat([gb, torch.ones(d, dtype=torch.bfloat16)]).reshape(1, 2 * d)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    for name, act in ACTS.items():
        y = run_gpu(gbf, {"x": xb, "rows": 1, "d": d}, act)
        ref = chains.gated_act(xb, d, act)
        yf = from_bits(y).float().cpu().numpy()
        assert np.all(np.isfinite(yf)), name
        assert_bf16_close(y, ref, f"{name} tails")


@pytest.mark.parametrize("name", ["gelu_erf", "silu"])
def test_gemm_epilogue_activations(gbf, name):
    """The Linear epilogue with the erf GELU and SiLU, full comparison."""
    c = workloads.linear_gelu_case(256, 512, 320, seed=9)
    x, w, b = from_bits(c["x"]), from_bits(c["w"]), from_bits(c["bias"])
    y = torch.empty(256, 512, dtype=torch.bfloat16, device="cuda")
    gbf.linear_bias_gelu(x, w, b, y, act=ACTS[name])
    torch.cuda.synchronize()
    ref = chains.linear_bias_gelu(c["x"], c["w"], c["bias"], act=ACTS[name])
    assert_bf16_close(to_bits(y), ref, f"linear + {name}")
