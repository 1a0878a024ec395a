"""GPU parity of gbf_add_rmsnorm_fp8 against the oracle's unfused chain
(residual add -> bf16 residual -> RMSNorm / _noweight / AdaRMSNorm -> E4M3)."""
import numpy as np
import pytest
import torch

import workloads
from oracle import chains
from parity import assert_bf16_close, assert_fp8_codes, from_bits, to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gbf():
    import fusion_add_rmsnorm_gb300 as g
    return g


def run_gpu(gbf, c, inplace=False):
    x, res = from_bits(c["x"]), from_bits(c["res"])
    out = res if inplace else torch.empty_like(res)
    q = torch.empty(res.shape, dtype=torch.uint8, device="cuda")
    dev = lambda k: None if c[k] is None else from_bits(c[k])       # noqa: E731
    gbf.add_rmsnorm_fp8(x, res, out, q, c["mode"], weight=dev("weight"), gate=dev("gate"),
                        ada_scale=dev("scale"), ada_shift=dev("shift"), eps=c["eps"], fp8_scale=c["s_q"])
    torch.cuda.synchronize()
    return to_bits(out), to_bits(q)


def run_oracle(c, rows=None):
    sl = slice(None) if rows is None else rows
    return chains.add_rmsnorm_fp8(c["x"][sl], c["res"][sl], c["eps"], c["s_q"], c["mode"], weight=c["weight"],
                                  gate=c["gate"], ada_scale=c["scale"], ada_shift=c["shift"])


def check(gbf, c, rows=None, inplace=False, what=""):
    res_out, q = run_gpu(gbf, c, inplace)
    ref_res, ref_q = run_oracle(c, rows)
    if rows is not None:
        res_out, q = res_out[rows], q[rows]
    assert_bf16_close(res_out, ref_res, what + " res_out")
    assert_fp8_codes(q, ref_q, what + " q")


def test_tiny_config_residual_rmsnorm_fp8(gbf):
    """x, res bf16 [16, 256], weight 1 + N(0, 0.1), eps 1e-6, scale 0.05."""
    check(gbf, workloads.config_tiny_add_rmsnorm(), what="[16,256]")


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("rows,hidden", [(1, 8), (3, 64), (37, 256), (4, 512), (6, 768), (10, 1024), (5, 1032),
                                         (7, 4096), (3, 8192), (3, 8200), (2, 16384), (2, 24576), (2, 32768),
                                         (5, 520), (7, 1000)])
def test_modes_and_shapes(gbf, mode, gated, rows, hidden):
    c = workloads.add_rmsnorm_case(rows, hidden, mode, seed=rows * 7 + hidden, gated=gated)
    check(gbf, c, what=f"mode {mode} gated {gated} [{rows},{hidden}]")


def test_in_place_residual(gbf):
    c = workloads.add_rmsnorm_case(33, 2048, 0, seed=5)
    check(gbf, c, inplace=True, what="in place")


def test_codes_match_worked_example(gbf):
    """The hand-derived example of tests/golden/rmsnorm_fp8_worked.json (ada, gated)."""
    import json, os
    from conftest import GOLDEN
    g = json.load(open(os.path.join(GOLDEN, "rmsnorm_fp8_worked.json")))["cases"][1]
    # the kernel needs hidden % 8 == 0: repeat the 4-wide example twice
    tile = lambda v: torch.tensor(np.tile(np.asarray(v, np.float32), 2)).to(torch.bfloat16)   # noqa: E731
    c = {"x": to_bits(tile(g["x"][0])[None]), "res": to_bits(tile(g["res"][0])[None]), "mode": 2,
         "eps": 0.0, "s_q": g["s_q"], "weight": None, "gate": to_bits(tile(g["gate"])),
         "scale": to_bits(tile(g["scale"])), "shift": to_bits(tile(g["shift"]))}
    res_out, q = run_gpu(gbf, c)
    assert res_out.tolist()[0] == g["res_out_bits"][0] * 2
    assert q.tolist()[0] == g["q_codes"][0] * 2


def test_pi05_decoder_chain_180_calls(gbf):
    """18 layers x 10 steps of the gated AdaRMSNorm + FP8 call on [10, 1024], the
    residual chaining from call to call on both sides."""
    w = workloads.pi05_decoder_chain()
    res_gpu = from_bits(w["res0"])
    res_ref = w["res0"]
    xs_gpu = [from_bits(x) for x in w["xs"]]
    q = torch.empty(res_gpu.shape, dtype=torch.uint8, device="cuda")
    for call, (gate, shift, scale) in enumerate(w["mods"]):
        layer = call % w["layers"]
        nxt = torch.empty_like(res_gpu)
        gbf.add_rmsnorm_fp8(xs_gpu[layer], res_gpu, nxt, q, 2, gate=from_bits(gate), ada_scale=from_bits(scale),
                            ada_shift=from_bits(shift), eps=w["eps"], fp8_scale=w["s_q"])
        res_ref, q_ref = chains.add_rmsnorm_fp8(w["xs"][layer], res_ref, w["eps"], w["s_q"], 2, gate=gate,
                                                ada_scale=scale, ada_shift=shift)
        torch.cuda.synchronize()
        assert_fp8_codes(to_bits(q), q_ref, f"call {call} q")
        res_gpu = nxt
    assert_bf16_close(to_bits(res_gpu), res_ref, "final residual")


@pytest.mark.parametrize("mode,gated", [(0, False), (1, False), (2, True), (2, False), (0, True)])
def test_large_sweep_shape_sampled_rows(gbf, mode, gated):
    """65536 x 4096 in the bench's launch configuration (two vectors per
    thread; Ada reloads its factors every row); the oracle checks 64 rows."""
    c = workloads.add_rmsnorm_case(65536, 4096, mode, seed=11, gated=gated)
    rows = np.sort(np.random.default_rng(0).choice(65536, 64, replace=False))
    check(gbf, c, rows=rows, what=f"65536x4096 mode {mode} gated {gated}")


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("rows,hidden", [(20011, 1024), (10007, 1032), (5000, 2056), (2003, 8192), (16411, 8192),
                                         (4099, 8200), (1001, 16384)])
def test_large_launch_plans_sampled_rows(gbf, mode, rows, hidden):
    """Launches large enough for the multi-vector plans: two vectors per thread
    with several rows per CTA and a ragged last CTA (1024), a vector count
    that leaves lanes idle (1032), four vectors per thread with the next row
    prefetched and the factors in shared memory (8192; 16411 rows give every
    CTA many trips of the double-buffered reduction), and eight (16384); 2056
    and 8200 leave most of the last vector slot of every thread idle; the
    oracle checks the first, last and 62 random rows."""
    c = workloads.add_rmsnorm_case(rows, hidden, mode, seed=rows + hidden + mode, gated=mode == 2)
    pick = np.unique(np.concatenate([[0, rows - 1], np.random.default_rng(mode).choice(rows, 62, replace=False)]))
    check(gbf, c, rows=pick, what=f"[{rows},{hidden}] mode {mode}")


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_fused_codes_at_least_as_close_as_the_unfused_chain(gbf, mode):
    """FlashRT's acceptance check: the fused path's cosine to the exact result
    is no worse than the unfused chain's.  The unfused chain stores y in bf16
    before the quantiser (one more rounding); the fused kernel quantises the
    float32 y.  Both sets of codes, dequantised, against the exact float64 y."""
    from oracle import formats, ops
    c = workloads.add_rmsnorm_case(64, 4096, mode, seed=500 + mode, gated=(mode == 2))
    res_out, q = run_gpu(gbf, c)
    _, q_unfused = chains.add_rmsnorm_fp8(c["x"], c["res"], c["eps"], c["s_q"], mode, weight=c["weight"],
                                          gate=c["gate"], ada_scale=c["scale"], ada_shift=c["shift"],
                                          round_y_bf16=True)
    r_hat = formats.bf16_decode(res_out)
    n = ops.rmsnorm(r_hat, c["eps"])
    if mode == 0:
        y = n * formats.bf16_decode(c["weight"])[None, :]
    elif mode == 1:
        y = n
    else:
        y = ops.ada_modulate(n, formats.bf16_decode(c["scale"])[None, :], formats.bf16_decode(c["shift"])[None, :])
    y = np.clip(y / c["s_q"], -448.0, 448.0).ravel()

    def cos(codes):
        d = formats.e4m3_decode(codes).astype(np.float64).ravel()
        return float(d @ y / np.linalg.norm(d) / np.linalg.norm(y))
    assert cos(q) >= cos(q_unfused) - 1e-9, (cos(q), cos(q_unfused))


# ------------------------------------------------------------ E4M3 range edges
# The quantiser saturates to +-448 instead of producing NaN (OpenPPL §6.4: a
# fused clamp has to see the quantisation scale; FlashRT §2.1 / §3: the fused
# kernel writes FP8 codes for the next layer).  These cases drive the kernel to
# both ends of the E4M3 range in every mode, with and without the gate, in the
# one-vector launch plan ([16, 256]), the two-vector plan of the bench
# ([65536, 4096]) and the four-vector plan ([2003, 8192]).

E4M3_NAN_CODES = (0x7F, 0xFF)


def check_edge(gbf, c, rows=None, what=""):
    res_out, q = run_gpu(gbf, c)
    ref_res, ref_q = run_oracle(c, rows)
    if rows is not None:
        res_out, q = res_out[rows], q[rows]
    assert_bf16_close(res_out, ref_res, what + " res_out")
    assert_fp8_codes(q, ref_q, what + " q")
    assert not np.isin(q, E4M3_NAN_CODES).any(), f"{what}: NaN code written"
    kind = c["kind"]
    if kind == "saturate":
        sat = np.isin(q, (0x7E, 0xFE))
        assert sat.mean() > 0.2, f"{what}: only {sat.mean():.3f} of codes saturated"
        assert (q == 0x7E).any() and (q == 0xFE).any(), f"{what}: saturation not reached on both signs"
    elif kind == "subnormal":
        mag = q & 0x7F
        assert (mag < 0x08).mean() > 0.5, f"{what}: only {(mag < 0x08).mean():.3f} of codes subnormal or zero"
        assert ((mag > 0) & (mag < 0x08)).any() and (mag == 0).any(), what
    elif kind == "outlier" and q.shape[-1] >= 1024:
        # the outlier's normalised value is about sqrt(hidden) >= 32, past 448 * 0.05 (a gate near zero can
        # take a row's outlier back into range)
        rowsat = np.isin(q, (0x7E, 0xFE)).any(axis=1).mean()
        assert rowsat > 0.9, f"{what}: only {rowsat:.3f} of the outlier rows saturated"
    return q


@pytest.mark.parametrize("kind", workloads.EDGE_KINDS)
@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("gated", [False, True])
def test_e4m3_range_edges_one_vector_plan(gbf, kind, mode, gated):
    c = workloads.add_rmsnorm_edge_case(16, 256, mode, kind, seed=40 + mode, gated=gated)
    q = check_edge(gbf, c, what=f"[16,256] {kind} mode {mode} gated {gated}")
    if kind == "zero_rows" and mode != 2:
        # a zero residual row normalises to zero: every code is +0 or -0 (row 1 sums to zero without a gate)
        assert np.isin(q[::3], (0x00, 0x80)).all()
        assert gated or np.isin(q[1], (0x00, 0x80)).all()


@pytest.mark.parametrize("kind", workloads.EDGE_KINDS)
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_e4m3_range_edges_bench_plan(gbf, kind, mode):
    """65536 x 4096 in the bench's launch configuration; the oracle checks the
    first rows (rows 0 and 1 are the zero rows of that kind), the last row and
    60 random rows."""
    c = workloads.add_rmsnorm_edge_case(65536, 4096, mode, kind, seed=60 + mode, gated=mode == 2)
    rng = np.random.default_rng(workloads.EDGE_KINDS.index(kind))
    pick = np.unique(np.concatenate([[0, 1, 2, 3, 65535], rng.choice(65536, 60, replace=False)]))
    check_edge(gbf, c, rows=pick, what=f"65536x4096 {kind} mode {mode}")


@pytest.mark.parametrize("kind", ["saturate", "outlier"])
@pytest.mark.parametrize("mode", [0, 2])
def test_e4m3_range_edges_four_vector_plan(gbf, kind, mode):
    c = workloads.add_rmsnorm_edge_case(2003, 8192, mode, kind, seed=80 + mode, gated=mode == 2)
    pick = np.unique(np.concatenate([[0, 1, 2002], np.random.default_rng(mode).choice(2003, 40, replace=False)]))
    check_edge(gbf, c, rows=pick, what=f"[2003,8192] {kind} mode {mode}")


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_zero_rows_with_zero_eps_are_nan_on_both_sides(gbf, mode):
    """The degenerate case of the norm: eps = 0 on a residual row that is all
    zeros is 0 / 0.  IEEE arithmetic makes it NaN on both sides, and the
    saturating E4M3 conversion keeps NaN (saturation applies to finite values
    only), so every code of those rows is a NaN code (0x7F or 0xFF) on the GPU
    and in the oracle; every other row matches element by element."""
    c = workloads.add_rmsnorm_edge_case(48, 512, mode, "zero_rows", seed=90 + mode)
    c["eps"] = 0.0
    res_out, q = run_gpu(gbf, c)
    with np.errstate(divide="ignore", invalid="ignore"):
        ref_res, ref_q = run_oracle(c)
    assert_bf16_close(res_out, ref_res, "eps 0 res_out")
    zero = np.zeros(48, bool)
    zero[::3] = True
    if mode != 2:
        zero[1] = True         # x = -res: the residual sums to zero (no gate in these modes)
    nan_codes = (0x7F, 0xFF)
    assert np.isin(q[zero], nan_codes).all() and np.isin(ref_q[zero], nan_codes).all()
    assert_fp8_codes(q[~zero], ref_q[~zero], f"eps 0 mode {mode} nonzero rows")
    assert not np.isin(q[~zero], nan_codes).any()
