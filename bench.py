"""Benchmark of the fused hot path on GB300: one JSON line on stdout.

A step is one pass of every fused operator at its workload size, each on its
own seeded synthetic inputs already resident in HBM:

  add_rmsnorm_fp8      residual + RMSNorm + FP8, x/res bf16 [16, 256], 100 calls as one CUDA graph
  pi05_ada_chain       gated residual + AdaRMSNorm + FP8, 180 calls on [10, 1024]
                       (18 layers x 10 steps), the residual chained call to call
  sweep_weighted       residual + RMSNorm + FP8 at [65536, 4096]
  sweep_noweight       the _noweight variant at [65536, 4096]
  sweep_ada            gated AdaRMSNorm + FP8 at [65536, 4096]
  qwen3_qkv            packed QKV [4096, 48*128], per-head norm, 1D RoPE; four calls on
                       four buffer sets (100 MB each, under the L2 size) back to back
  chameleon_qkv_ln     packed QKV [4096, 96*128], per-head LayerNorm (weight + bias), 1D RoPE
  swiglu_ffn           silu(gate) * up over [gate | up] bf16 [4096, 2*11008]
  wan_qkv3d            packed QKV [32760, 3*5120], full-width norm, 3D RoPE
  linear_bias_gelu     X [8192, 4096] . W[16384, 4096]^T + b, GELU(tanh)
  linear_fp8_gelu      E4M3 X [8192, 4096] . E4M3 W [16384, 4096]^T with descales + b, GELU(tanh)
  bn_fold              W [16384, 4096], BN of its 16384 output channels
  fold_norm_weight     W [16384, 4096] * (1 + gamma[4096]) (the _noweight norm's weight pre-folded)

Timing: every operator is bracketed by CUDA events on the stream it is
launched on; L2 (129 MB) is flushed before each operator, outside the event
pair, by writing a 512 MB buffer and then reading it back, so the operator
starts with a cold L2 that holds no dirty lines of the flush to write back.  K steps are timed after W warm-up steps,
with a barrier and a device synchronisation on both sides; the slowest rank
counts.  `value` is the aggregate HBM throughput of the memory-bound fused
kernels: their algorithmic bytes summed over the step divided by their summed
device time; the GEMM is timed in the same step and reported in TFLOP/s.
After the step, outside its aggregate, `latency_bound.qwen3_qkv_decode_paged`
times decode-shaped QKV post-processing into a paged KV cache (32 sequences'
new tokens, K/V rows by slot mapping into 16-row blocks of a 16,384-row
cache), `latency_bound.swiglu_decode` SwiGLU on [32, 2 x 11008] and
`latency_bound.linear_decode` the Linear + bias + GELU on 32 rows (W-read
bound; cuBLASLt's fused epilogue beside it): CUDA graphs of back-to-back
calls, microseconds per call.

`--impl reference` times the CPU oracle (the unfused operator chains, float64
numpy) on a bounded sample of the same workload instead.
"""
import argparse
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "fused-kernel HBM GB/s (% of GB300 peak) and tokens/s per fused op"
UNIT = "GB/s"
L2_FLUSH_BYTES = 512 << 20
L2_BYTES = 129 * 10**6           # GB300 L2 capacity
BF16_DENSE_NOMINAL_TFLOPS = 2250.0

# ----------------------------------------------------------------- bytes model
# The graph-autofusion article's benefit model (阶段二收益估算): before fusion
# every operator of the chain reads its inputs from HBM and writes its output
# back; after fusion the one kernel reads the chain's inputs once and writes
# its outputs once.  Byte counts per call; N = rows * hidden elements, bf16 = 2
# bytes, an E4M3 code = 1 byte.


def bytes_add_rmsnorm(rows, hidden, mode, gated):
    """Fused: read x, res (4N), write res_out (2N) and the codes (N), read the
    [hidden] vectors the mode uses once: 7N + 2H (weight), + 4H (ada scale and
    shift), + 2H (gate)."""
    n = rows * hidden
    vec = (2 if mode == 0 else 0) + (4 if mode == 2 else 0) + (2 if gated else 0)
    return 7 * n + vec * hidden


def bytes_unfused_add_rmsnorm(rows, hidden, mode, gated):
    """The chain of separate operators, each reading and writing HBM:
    gate multiply (x, gate -> g: 4N + 2H), residual add (6N), RMSNorm (r -> n:
    4N, + 2H for the weight), AdaRMSNorm's * (1 + scale) (4N + 2H) and + shift
    (4N + 2H), quantise (y -> codes: 3N).  Weighted, ungated: 13N + 2H; the
    Pi0.5 gated AdaRMSNorm call: 25N + 6H."""
    n = rows * hidden
    total = (4 * n + 2 * hidden if gated else 0) + 6 * n + 4 * n + 3 * n
    if mode == 0:
        total += 2 * hidden
    elif mode == 2:
        total += 2 * (4 * n + 2 * hidden)
    return total


def bytes_qkv(tokens, hq, hkv, d):
    """Fused QKV post-processing: read the packed row once, write Q, K and V
    once: 2 * T * (Hq + 2 Hkv) * D bf16 values.  The norm weights and the
    positions (under 0.02 % at the configs) are left out, as in the survey's
    table."""
    return 2 * tokens * (hq + 2 * hkv) * d * 2


def bytes_unfused_qkv(tokens, hq, hkv, d, norm):
    """Per-head norm (and the LayerNorm variant): the split is a view; Q norm
    and Q RoPE read and write Q (4q), K norm, K RoPE and the K-cache copy read
    and write K (6kv), the V-cache copy reads and writes V (2kv).  Full-width
    norm (Wan): the split reads and writes all three (2 (q + 2kv)), the two
    norms and the two RoPEs each read and write Q and K (4 (q + kv))."""
    q, kv = tokens * hq * d * 2, tokens * hkv * d * 2
    if norm in (0, 2):
        return 4 * q + 6 * kv + 2 * kv
    return 2 * (q + 2 * kv) + 2 * (q + kv) + 2 * (q + kv)


def bytes_linear(m, n, k, bias=True):
    """Fused Linear + bias + GELU: read X and W, read the bias, write Y once (bf16)."""
    return 2 * (m * k + n * k + (n if bias else 0) + m * n)


def bytes_unfused_linear(m, n, k):
    """GEMM (X, W -> Y), bias add (Y, b -> Y: 4MN + 2N), GELU (Y -> Y: 4MN)."""
    return 2 * (m * k + n * k + m * n) + (4 * m * n + 2 * n) + 4 * m * n


def bytes_bn_fold(out_ch, inner):
    """W read and written (bf16), b read and written, gamma, beta, mean, var read (float32)."""
    return 2 * out_ch * inner * 2 + 2 * out_ch * 2 + 4 * out_ch * 4


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------- GPU ops

class Op:
    name = ""
    bound = "hbm"
    launches = 1

    def algorithmic_bytes(self):
        return 0

    def flops(self):
        return 0

    def units(self):          # tokens (rows) per call
        return 0


class AddRmsNormOp(Op):
    """One call, or (calls > 1, for a launch-bound shape) `calls` identical
    calls captured through the C ABI into one CUDA graph and replayed."""

    def __init__(self, gbf, name, rows, hidden, mode, gated, seed, calls=1):
        import torch
        import workloads
        from workloads import as_torch as from_bits
        self.gbf, self.name, self.rows, self.hidden, self.mode, self.gated = gbf, name, rows, hidden, mode, gated
        c = workloads.add_rmsnorm_case(rows, hidden, mode, seed=seed, gated=gated)
        self.host = c
        dev = lambda k: None if c[k] is None else from_bits(c[k])   # noqa: E731
        self.x, self.res = from_bits(c["x"]), from_bits(c["res"])
        self.w, self.gate, self.scale, self.shift = dev("weight"), dev("gate"), dev("scale"), dev("shift")
        self.out = torch.empty_like(self.res)
        self.q = torch.empty(self.res.shape, dtype=torch.uint8, device="cuda")
        self.eps, self.s_q = c["eps"], c["s_q"]
        self.launches = calls
        self.graph = None
        if calls > 1:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                self.call()
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph):
                for _ in range(calls):
                    self.call()
            torch.cuda.synchronize()

    def call(self):
        self.gbf.add_rmsnorm_fp8(self.x, self.res, self.out, self.q, self.mode, weight=self.w, gate=self.gate,
                                 ada_scale=self.scale, ada_shift=self.shift, eps=self.eps, fp8_scale=self.s_q)

    def run(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            self.call()

    def algorithmic_bytes(self):
        return self.launches * bytes_add_rmsnorm(self.rows, self.hidden, self.mode, self.gated)

    def unfused_bytes(self):
        return self.launches * bytes_unfused_add_rmsnorm(self.rows, self.hidden, self.mode, self.gated)

    def units(self):
        return self.launches * self.rows

    def e2e_buffers(self):
        ins = [t for t in (self.x, self.res, self.w, self.gate, self.scale, self.shift) if t is not None]
        return ins, [self.out, self.q]


class AdaChainOp(Op):
    """180 sequential calls (18 layers x 10 steps) on [10, 1024], captured once
    through the C ABI into a CUDA graph (with the calls' programmatic-dependent
    launch edges) and replayed as one submission per step."""

    def __init__(self, gbf, seed=0, graph=True):
        import torch
        import workloads
        from workloads import as_torch as from_bits
        self.gbf, self.name = gbf, "pi05_ada_chain"
        w = workloads.pi05_decoder_chain(seed)
        self.w = w
        self.launches = len(w["mods"])
        self.res0 = from_bits(w["res0"])
        self.xs = [from_bits(x) for x in w["xs"]]
        self.mods = [tuple(from_bits(m) for m in mod) for mod in w["mods"]]
        self.bufs = [torch.empty_like(self.res0), torch.empty_like(self.res0)]
        self.q = torch.empty(self.res0.shape, dtype=torch.uint8, device="cuda")
        self.graph = None
        if graph:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                self.run_eager()
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph):
                self.run_eager()
            torch.cuda.synchronize()

    def run(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            self.run_eager()

    def run_eager(self):
        res = self.res0
        L = self.w["layers"]
        for call, (gate, shift, scale) in enumerate(self.mods):
            out = self.bufs[call & 1]
            self.gbf.add_rmsnorm_fp8(self.xs[call % L], res, out, self.q, 2, gate=gate, ada_scale=scale,
                                     ada_shift=shift, eps=self.w["eps"], fp8_scale=self.w["s_q"])
            res = out

    def algorithmic_bytes(self):
        return self.launches * bytes_add_rmsnorm(10, 1024, 2, True)

    def unfused_bytes(self):
        return self.launches * bytes_unfused_add_rmsnorm(10, 1024, 2, True)

    def units(self):
        return self.launches * 10

    def e2e_buffers(self):
        ins = [self.res0] + self.xs + [t for m in self.mods for t in m]
        return ins, [self.bufs[(self.launches - 1) & 1], self.q]


class QkvOp(Op):
    """One call per buffer set, back to back.  A workload smaller than L2 runs
    on `sets` distinct copies of its inputs and outputs, so no call finds
    another call's data in L2 (together they are several times the L2 size)
    while the fixed cost of an event-bracketed launch is shared by the calls."""

    def __init__(self, gbf, name, case, sets=1):
        import torch
        from workloads import as_torch as from_bits
        self.gbf, self.name, self.c = gbf, name, case
        c = case
        t, hq, hkv, d = c["tokens"], c["n_q"], c["n_kv"], c["d"]
        qkv = from_bits(c["qkv"])
        self.qw, self.kw = from_bits(c["q_w"]), from_bits(c["k_w"])
        self.ln = c["norm"] == 2            # per-head LayerNorm entry point
        self.qb = None if c.get("q_b") is None else from_bits(c["q_b"])
        self.kb = None if c.get("k_b") is None else from_bits(c["k_b"])
        self.pos = torch.from_numpy(np.ascontiguousarray(c["pos"])).cuda()
        self.sets = []
        for i in range(sets):
            self.sets.append((qkv if i == 0 else qkv.clone(),
                              torch.empty(t, hq, d, dtype=torch.bfloat16, device="cuda"),
                              torch.empty(t, hkv, d, dtype=torch.bfloat16, device="cuda"),
                              torch.empty(t, hkv, d, dtype=torch.bfloat16, device="cuda")))
        self.launches = sets
        self.qkv, self.qo, self.kc, self.vc = self.sets[0]
        c["qkv"] = None      # drop the host copy

    def run(self):
        c = self.c
        for qkv, qo, kc, vc in self.sets:
            if self.ln:
                self.gbf.qkv_split_layernorm_rope(qkv, c["n_q"], c["n_kv"], c["d"], self.qw, self.qb, self.kw,
                                                  self.kb, c["eps"], self.pos, c["theta"], qo, kc, vc)
            else:
                self.gbf.qkv_split_norm_rope(qkv, c["n_q"], c["n_kv"], c["d"], c["norm"], self.qw, self.kw,
                                             c["eps"], c["rope"], self.pos, c["theta"], qo, kc, vc,
                                             sections=c["sections"])

    def algorithmic_bytes(self):
        c = self.c
        return self.launches * bytes_qkv(c["tokens"], c["n_q"], c["n_kv"], c["d"])

    def unfused_bytes(self):
        c = self.c
        return self.launches * bytes_unfused_qkv(c["tokens"], c["n_q"], c["n_kv"], c["d"], c["norm"])

    def units(self):
        return self.launches * self.c["tokens"]

    def e2e_buffers(self):
        params = [t for t in (self.qw, self.kw, self.qb, self.kb, self.pos) if t is not None]
        return [st[0] for st in self.sets] + params, [t for st in self.sets for t in st[1:]]


class GatedActOp(Op):
    """SwiGLU: y = silu(gate) * up over [gate | up] rows."""

    def __init__(self, gbf, name, case, act):
        import torch
        from workloads import as_torch as from_bits
        self.gbf, self.name, self.act = gbf, name, act
        self.rows, self.d = case["rows"], case["d"]
        self.x = from_bits(case["x"])
        self.y = torch.empty(self.rows, self.d, dtype=torch.bfloat16, device="cuda")

    def run(self):
        self.gbf.gated_act(self.x, self.y, self.act)

    def algorithmic_bytes(self):
        return self.rows * self.d * 6                  # read gate + up, write y (bf16)

    def unfused_bytes(self):
        return self.rows * self.d * 10                 # act: read g, write a; mul: read a, u, write y

    def units(self):
        return self.rows

    def e2e_buffers(self):
        return [self.x], [self.y]


class GemmOp(Op):
    bound = "tensor"

    def __init__(self, gbf, case):
        import torch
        from workloads import as_torch as from_bits
        self.gbf, self.name, self.c = gbf, "linear_bias_gelu", case
        self.x, self.w, self.b = from_bits(case["x"]), from_bits(case["w"]), from_bits(case["bias"])
        self.y = torch.empty(case["m"], case["n"], dtype=torch.bfloat16, device="cuda")

    def run(self):
        self.gbf.linear_bias_gelu(self.x, self.w, self.b, self.y, self.gbf.ACT_GELU_TANH)

    def flops(self):
        c = self.c
        return 2 * c["m"] * c["n"] * c["k"]

    def algorithmic_bytes(self):
        c = self.c
        return bytes_linear(c["m"], c["n"], c["k"])

    def unfused_bytes(self):
        c = self.c
        return bytes_unfused_linear(c["m"], c["n"], c["k"])

    def units(self):
        return self.c["m"]

    def e2e_buffers(self):
        return [self.x, self.w, self.b], [self.y]


class GemmFp8Op(Op):
    """Quantised Linear + GELU(tanh): E4M3 activation codes [M, K] (descale
    0.05) and weight codes [N, K] (per-row descales), bias, bf16 out.  The codes
    are made on the device from the case's seeded values by torch's E4M3
    conversion (input preparation, outside the timed region)."""
    bound = "tensor"
    peak_ratio = 2.0          # dense E4M3 vs bf16 on this part (nominal 4.5 / 2.25 PFLOP/s)

    def __init__(self, gbf, case):
        import torch
        from workloads import as_torch as from_bits
        self.gbf, self.name, self.c = gbf, "linear_fp8_gelu", case
        x = torch.from_numpy(case["x"]).cuda()
        w = torch.from_numpy(case["w"]).cuda()
        self.ws = torch.from_numpy(case["w_scale"]).cuda()
        self.xs = float(np.float32(case["x_scale"]))
        self.xq = (x / self.xs).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        self.wq = (w / self.ws[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        del x, w
        self.b = from_bits(case["bias"])
        self.y = torch.empty(case["m"], case["n"], dtype=torch.bfloat16, device="cuda")

    def run(self):
        self.gbf.linear_fp8_act(self.xq, self.xs, self.wq, self.ws, self.b, self.y, self.gbf.ACT_GELU_TANH)

    def flops(self):
        c = self.c
        return 2 * c["m"] * c["n"] * c["k"]

    def algorithmic_bytes(self):
        c = self.c
        return c["m"] * c["k"] + c["n"] * c["k"] + 4 * c["n"] + 2 * c["n"] + 2 * c["m"] * c["n"]

    def unfused_bytes(self):
        y = self.c["m"] * self.c["n"] * 2
        return self.algorithmic_bytes() + 2 * y + 2 * y          # + a separate dequant/bias and GELU pass

    def units(self):
        return self.c["m"]

    def e2e_buffers(self):
        return [self.xq, self.wq, self.ws, self.b], [self.y]


class NormFoldOp(Op):
    """Pre-fold of a Gemma-style norm weight (1 + gamma) into W [N, K]."""

    def __init__(self, gbf, case):
        import torch
        from workloads import as_torch as from_bits
        self.gbf, self.name, self.c = gbf, "fold_norm_weight", case
        self.w, self.g = from_bits(case["w"]), from_bits(case["gamma"])
        self.wo = torch.empty_like(self.w)

    def run(self):
        self.gbf.fold_norm_weight(self.w, self.g, self.wo)

    def algorithmic_bytes(self):
        return 2 * self.c["out_ch"] * self.c["inner"] * 2 + 2 * self.c["inner"]

    def unfused_bytes(self):
        return self.algorithmic_bytes()

    def units(self):
        return self.c["out_ch"]

    def e2e_buffers(self):
        return [self.w, self.g], [self.wo]


class FoldOp(Op):
    def __init__(self, gbf, case):
        import torch
        from workloads import as_torch as from_bits
        self.gbf, self.name, self.c = gbf, "bn_fold", case
        f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()   # noqa: E731
        self.w, self.b = from_bits(case["w"]), from_bits(case["bias"])
        self.g, self.be, self.mu, self.var = (f32(case[k]) for k in ("gamma", "beta", "mean", "var"))
        self.wo = torch.empty_like(self.w)
        self.bo = torch.empty_like(self.b)

    def run(self):
        self.gbf.bn_fold(self.w, self.b, self.g, self.be, self.mu, self.var, self.c["eps"], self.wo, self.bo)

    def algorithmic_bytes(self):
        return bytes_bn_fold(self.c["n"], self.c["k"])

    def unfused_bytes(self):
        return self.algorithmic_bytes()

    def units(self):
        return self.c["n"]          # output channels

    def e2e_buffers(self):
        return [self.w, self.b, self.g, self.be, self.mu, self.var], [self.wo, self.bo]


OP_NAMES = ("add_rmsnorm_fp8", "pi05_ada_chain", "sweep_weighted", "sweep_noweight", "sweep_ada", "qwen3_qkv",
            "chameleon_qkv_ln", "swiglu_ffn", "wan_qkv3d", "linear_bias_gelu", "linear_fp8_gelu", "bn_fold",
            "fold_norm_weight")


def build_ops(gbf, with_gemm, only=None, small=False):
    """The step's operators.  `small` shrinks the large ones to profiling size
    (inputs still larger than L2) for ncu captures; `only` keeps a subset."""
    import workloads
    want = set(only or OP_NAMES)
    rows = 8192 if small else 65536
    ops = []
    if "add_rmsnorm_fp8" in want:
        ops.append(AddRmsNormOp(gbf, "add_rmsnorm_fp8", 16, 256, 0, False, 0, calls=100))
    if "pi05_ada_chain" in want:
        ops.append(AdaChainOp(gbf))
    for name, mode, gated, seed in (("sweep_weighted", 0, False, 11), ("sweep_noweight", 1, False, 12),
                                    ("sweep_ada", 2, True, 13)):
        if name in want:
            ops.append(AddRmsNormOp(gbf, name, rows, 4096, mode, gated, seed))
    if "qwen3_qkv" in want:       # 100 MB per call, under the L2 size: four buffer sets
        ops.append(QkvOp(gbf, "qwen3_qkv", workloads.config_qwen3_qkv(), sets=1 if small else 4))
    if "chameleon_qkv_ln" in want:
        ops.append(QkvOp(gbf, "chameleon_qkv_ln", workloads.config_chameleon_qkv(tokens=2048 if small else 4096)))
    if "swiglu_ffn" in want:
        ops.append(GatedActOp(gbf, "swiglu_ffn", workloads.config_swiglu_ffn(rows=1024 if small else 4096),
                              gbf.ACT_SILU))
    if "wan_qkv3d" in want:
        ops.append(QkvOp(gbf, "wan_qkv3d", workloads.config_wan_qkv(tokens=4096 if small else None)))
    if want & {"linear_bias_gelu", "bn_fold"}:
        lin = workloads.linear_gelu_case(2048, 16384, 4096) if small else workloads.config_linear_gelu()
        if with_gemm and "linear_bias_gelu" in want:
            ops.append(GemmOp(gbf, lin))
        if "bn_fold" in want:
            ops.append(FoldOp(gbf, lin))
    if with_gemm and "linear_fp8_gelu" in want:
        ops.append(GemmFp8Op(gbf, workloads.fp8_linear_case(2048 if small else 8192, 16384, 4096)))
    if "fold_norm_weight" in want:
        ops.append(NormFoldOp(gbf, workloads.norm_fold_case(16384, 4096)))
    return ops


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """SM and memory clocks, power and throttle reasons sampled every 10 ms while the timed
    region runs, read from NVML (libnvidia-ml, through ctypes); falls back to
    nvidia-smi at 50 ms when NVML cannot be loaded."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index):
        self.cuda_index = cuda_index
        self.samples, self.first, self.stop_flag = [], 0, False
        self.mem_mhz = []
        self.nvml, self.dev, self.max_mhz, self.thread, self.proc = None, None, None, None, None

    def _open_nvml(self):
        import ctypes
        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return False
        props = torch.cuda.get_device_properties(self.cuda_index)
        bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0".encode()
        dev = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(dev)) != 0:
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.cuda_index), ctypes.byref(dev)) != 0:
                return False
        mx = ctypes.c_uint()
        lib.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx))
        self.nvml, self.dev, self.max_mhz = lib, dev, float(mx.value)
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        return True

    def _poll(self):
        import ctypes
        clk, mclk, rea, pw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        while not self.stop_flag:
            self.nvml.nvmlDeviceGetClockInfo(self.dev, 1, ctypes.byref(clk))      # NVML_CLOCK_SM
            self.nvml.nvmlDeviceGetClockInfo(self.dev, 2, ctypes.byref(mclk))     # NVML_CLOCK_MEM
            self.reasons_fn(self.dev, ctypes.byref(rea))
            self.nvml.nvmlDeviceGetPowerUsage(self.dev, ctypes.byref(pw))
            self.samples.append((float(clk.value), int(rea.value), pw.value / 1000.0))
            self.mem_mhz.append(float(mclk.value))
            time.sleep(0.01)

    def start(self):
        try:
            ok = self._open_nvml()
        except (OSError, AttributeError):
            ok = False
        if ok:
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.cuda_index),
                                          "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active,power.draw",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read_smi, daemon=True).start()
        except OSError:
            self.proc = None

    def _read_smi(self):
        for line in self.proc.stdout:
            f = [x.strip() for x in line.split(",")]
            try:
                self.max_mhz = float(f[1])
                self.samples.append((float(f[0]), int(f[2], 16), float(f[3])))
            except (ValueError, IndexError):
                continue

    def mark(self):
        """Start of the timed region: keep samples from here on (and the one before)."""
        t0 = time.time()
        while (self.thread or self.proc) and not self.samples and time.time() - t0 < 5:
            time.sleep(0.01)
        self.first = max(0, len(self.samples) - 1)

    def stop(self):
        self.stop_flag = True
        if self.thread is not None:
            self.thread.join(timeout=1)
        if self.proc is not None:
            self.proc.terminate()
        got = self.samples[self.first:]
        if not got:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no clock samples"], "samples": 0}
        reasons = set()
        for _, r, _ in got:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        out = {"sm_mhz": statistics.median(c for c, _, _ in got), "sm_max_mhz": self.max_mhz,
               "reasons": sorted(reasons), "samples": len(got),
               "power_w_max": round(max(p for _, _, p in got), 1),
               "source": "nvml" if self.thread is not None else "nvidia-smi"}
        mem = self.mem_mhz[self.first:]
        if mem:
            out["mem_mhz"] = statistics.median(mem)
        return out


# ------------------------------------------------------------- traffic record

def kernel_traffic(op_name):
    """DRAM bytes per launch of `op_name`'s kernel from the committed ncu record
    (profiles/traffic.json), or None when the kernel's source has changed since
    the counters were taken (or none were taken)."""
    rec = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(rec):
        return None
    with open(rec) as f:
        ent = json.load(f).get("per_op", {}).get(op_name)
    if not ent:
        return None
    if kernel_source_hash(ent["source"]) != ent["source_sha256_16"]:
        return None
    return ent["dram_bytes_per_launch"]


def strip_comments(text):
    """C/C++/CUDA source without its comments and with runs of whitespace
    collapsed (string and character literals are kept as written)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
        elif text.startswith("/*", i):
            i = text.find("*/", i + 2)
            i = n if i < 0 else i + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(source):
    """First 16 hex digits of the SHA-256 of a kernel source followed by the
    headers every kernel includes, comments and layout stripped (a change to
    the code of either invalidates its record; a comment edit does not)."""
    csrc = os.path.join(ROOT, "fusion_add_rmsnorm_gb300", "csrc")
    h = hashlib.sha256()
    for name in (source, "common.cuh", "tma.cuh", "kernels.h"):
        path = os.path.join(csrc, name)
        if not os.path.exists(path):
            return None
        h.update(strip_comments(open(path, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


KERNEL_FILE = {"add_rmsnorm_fp8": "add_rmsnorm_fp8.cu", "pi05_ada_chain": "add_rmsnorm_fp8.cu",
               "sweep_weighted": "add_rmsnorm_fp8.cu", "sweep_noweight": "add_rmsnorm_fp8.cu",
               "sweep_ada": "add_rmsnorm_fp8.cu", "qwen3_qkv": "qkv_norm_rope.cu", "wan_qkv3d": "qkv_norm_rope.cu",
               "chameleon_qkv_ln": "qkv_norm_rope.cu", "swiglu_ffn": "gated_act.cu",
               "linear_bias_gelu": "gemm_tcgen05.cu", "bn_fold": "bn_fold.cu", "linear_fp8_gelu": "gemm_tcgen05.cu",
               "fold_norm_weight": "bn_fold.cu"}


# -------------------------------------------------------------- CPU baseline

def cpu_baseline_sample(scale=1, gemm=True):
    """Time the oracle's unfused chains on a bounded sample of every operator
    of the step, single-threaded, and scale to GB/s of algorithmic bytes.
    Returns a dict; runs in a fresh subprocess (see run_cpu_baseline)."""
    import workloads
    from oracle import chains
    t_start = time.time()
    res = {}
    t_total = 0.0
    byts_total = 0

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    # add + RMSNorm + FP8 at [16, 256], the 180-call chain (10 calls sampled), the sweep (64 rows per mode)
    c = workloads.config_tiny_add_rmsnorm()
    dt = timed(lambda: chains.add_rmsnorm_fp8(c["x"], c["res"], c["eps"], c["s_q"], 0, weight=c["weight"]))
    res["add_rmsnorm_fp8"] = (bytes_add_rmsnorm(16, 256, 0, False), dt)
    w = workloads.pi05_decoder_chain()
    r = w["res0"]

    n_calls = min(10 * scale, 180)

    def chain10():
        nonlocal r
        for call in range(n_calls):
            g, sh, sc = w["mods"][call]
            r, _ = chains.add_rmsnorm_fp8(w["xs"][call % 18], r, w["eps"], w["s_q"], 2, gate=g, ada_scale=sc,
                                          ada_shift=sh)
    res["pi05_ada_chain"] = (n_calls * bytes_add_rmsnorm(10, 1024, 2, True), timed(chain10))
    for name, mode, gated in (("sweep_weighted", 0, False), ("sweep_noweight", 1, False), ("sweep_ada", 2, True)):
        rows = 64 * scale
        c = workloads.add_rmsnorm_case(rows, 4096, mode, seed=3, gated=gated)
        dt = timed(lambda: chains.add_rmsnorm_fp8(c["x"], c["res"], c["eps"], c["s_q"], mode, weight=c["weight"],
                                                  gate=c["gate"], ada_scale=c["scale"], ada_shift=c["shift"]))
        res[name] = (bytes_add_rmsnorm(rows, 4096, mode, gated), dt)
    tq = 256 * scale
    c = workloads.config_qwen3_qkv(tokens=tq)
    dt = timed(lambda: chains.qkv_split_norm_rope(c["qkv"], 32, 8, 128, 0, c["q_w"], c["k_w"], c["eps"], 0, c["pos"],
                                                  c["theta"]))
    res["qwen3_qkv"] = (bytes_qkv(tq, 32, 8, 128), dt)
    tc = 128 * scale
    c = workloads.config_chameleon_qkv(tokens=tc)
    dt = timed(lambda: chains.qkv_split_norm_rope(c["qkv"], 32, 32, 128, chains.QKNORM_LAYERNORM, c["q_w"], c["k_w"],
                                                  c["eps"], 0, c["pos"], c["theta"], q_b=c["q_b"], k_b=c["k_b"]))
    res["chameleon_qkv_ln"] = (bytes_qkv(tc, 32, 32, 128), dt)
    ts = 16 * scale
    c = workloads.config_swiglu_ffn(rows=ts)
    dt = timed(lambda: chains.gated_act(c["x"], 11008, 3))
    res["swiglu_ffn"] = (ts * 11008 * 6, dt)
    tw = 64 * scale
    c = workloads.config_wan_qkv(tokens=tw)
    dt = timed(lambda: chains.qkv_split_norm_rope(c["qkv"], 40, 40, 128, 1, c["q_w"], c["k_w"], c["eps"], 1,
                                                  c["pos"], c["theta"], sections=c["sections"]))
    res["wan_qkv3d"] = (bytes_qkv(tw, 40, 40, 128), dt)
    if gemm:                       # GFLOP/s only; not part of the GB/s value
        mg = 16 * scale
        c = workloads.linear_gelu_case(mg, 16384, 4096, seed=0)
        dt = timed(lambda: chains.linear_bias_gelu(c["x"], c["w"], c["bias"]))
        res["linear_bias_gelu"] = (2 * mg * 16384 * 4096, dt)         # flops
        mf = 16 * scale
        c = workloads.fp8_linear_case(mf, 16384, 4096, seed=0)
        import torch

        def e4m3(v):   # input codes (outside the timed call): clamp, then torch's nearest-even conversion
            return torch.from_numpy(np.ascontiguousarray(v, np.float32)).clamp(-448, 448).to(
                torch.float8_e4m3fn).view(torch.uint8).numpy()
        xq = e4m3(c["x"] / np.float32(c["x_scale"]))
        wq = e4m3(c["w"] / c["w_scale"][:, None])
        dt = timed(lambda: chains.linear_fp8_act(xq, np.float32(c["x_scale"]), wq, c["w_scale"], c["bias"], act=1))
        res["linear_fp8_gelu"] = (2 * mf * 16384 * 4096, dt)       # flops
    cf = 1024 * scale
    c = workloads.norm_fold_case(cf, 4096)
    dt = timed(lambda: chains.fold_norm_weight_bf16(c["w"], c["gamma"]))
    res["fold_norm_weight"] = (2 * cf * 4096 * 2 + 2 * 4096, dt)
    ch = 1024 * scale
    c = workloads.linear_gelu_case(1, ch, 4096, seed=0)
    dt = timed(lambda: chains.bn_fold_bf16(c["w"], c["bias"], c["gamma"], c["beta"], c["mean"], c["var"], c["eps"]))
    res["bn_fold"] = (bytes_bn_fold(ch, 4096), dt)
    for k, (b, dt) in res.items():
        if k not in ("linear_bias_gelu", "linear_fp8_gelu"):
            t_total += dt
            byts_total += b
    return {"gbs": byts_total / t_total / 1e9, "seconds": t_total, "bytes": byts_total, "t_start": t_start,
            "per_op": {k: ({"gflops": b / dt / 1e9} if k in ("linear_bias_gelu", "linear_fp8_gelu") else {"gbs": b / dt / 1e9})
                       for k, (b, dt) in res.items()}}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_cpu_baseline(scale=32, all_cores=True):
    """The oracle's bounded sample in one single-threaded child process; then,
    with all_cores, one such child per host core running a quarter of that
    sample's memory-bound operators at the same time (every child starts its
    timed work at one shared wall-clock instant, after its imports), reported
    as the aggregate over the cores."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--_cpu-baseline-child"]
    r = subprocess.run(cmd + [str(scale)], env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "error": r.stderr[-300:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    out = {"value": round(d["gbs"], 4), "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": (f"float64 numpy oracle, one thread per process: [16,256] add+RMSNorm+FP8; {min(10 * scale, 180)} of "
                      f"the 180 chained [10,1024] AdaRMSNorm calls; {64 * scale} rows of each [65536,4096] sweep; "
                      f"{256 * scale} Qwen3 tokens; {128 * scale} Chameleon tokens; {16 * scale} SwiGLU rows; "
                      f"{64 * scale} Wan tokens; "
                      f"BN fold and norm-weight fold of {1024 * scale} channels each; "
                      "GB/s = algorithmic bytes / oracle time over the memory-bound operators (a "
                      f"{16 * scale}-row sample of each GEMM is in per_op as GFLOP/s)"),
           "seconds": round(d["seconds"], 3), "per_op": d["per_op"]}
    cores = host_cores()
    if not all_cores or cores < 2:
        return out
    part = max(1, scale // 4)
    start = time.time() + 8.0
    procs = [subprocess.Popen(cmd + [str(part), "--_cpu-baseline-start", f"{start:.3f}", "--_cpu-baseline-nogemm"],
                              env=env,
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for _ in range(cores)]
    results = []
    for pr in procs:
        so, se = pr.communicate(timeout=900)
        if pr.returncode == 0:
            results.append(json.loads(so.strip().splitlines()[-1]))
    if len(results) == cores:
        agg = sum(x["bytes"] for x in results) / max(x["seconds"] for x in results) / 1e9
        out["start_spread_s"] = round(max(x["t_start"] for x in results) - min(x["t_start"] for x in results), 3)
        out["one_core"] = {"value": out["value"], "seconds": out["seconds"]}
        out["value"] = round(agg, 4)
        out["cores"] = cores
        out["sample"] += (f"; all cores: {cores} such processes at once, each on a quarter of the memory-bound sample, "
                          "value = their summed bytes / the slowest one's oracle time")
    return out


# ------------------------------------------------------------------ main arm

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, v):
    if pg is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(pg, v):
    if pg is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.SUM)
    return float(t.item())


def copy_probe_gbs(gbf, nbytes=1 << 30, reps=10):
    """Best of `reps` event-timed gbf_copy calls of 1 GiB (read + write bytes
    per second): this library's own copy-kernel bandwidth, reported beside the
    measured peak the fractions use."""
    import torch
    src = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    src.fill_(1)
    dst = torch.empty_like(src)
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        gbf.copy(src, dst)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    del src, dst
    return round(2 * nbytes / (best / 1e3) / 1e9, 1)


def main_gpu(args):
    import torch
    world, rank, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    import fusion_add_rmsnorm_gb300 as gbf
    peaks = load_peaks()
    with_gemm = not args.no_gemm
    ops = build_ops(gbf, with_gemm, args.only.split(",") if args.only else None, args.small)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush_words = flush.view(torch.int64)

    def flush_l2():
        flush.fill_(1)               # evicts everything the last operator left in L2 ...
        flush_words.sum()            # ... and the read-back leaves only clean lines behind
    stream = torch.cuda.current_stream()

    def one_step(record):
        times = {}
        for op in ops:
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            op.run()
            e1.record(stream)
            record.append((op, e0, e1))
        return times

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        one_step([])
    torch.cuda.synchronize()
    status, msg = gbf.device_status()
    if status != gbf.OK:
        raise RuntimeError(f"device status after warm-up: {msg}")

    # The K-step timed region runs `repeats` times back to back (each bracketed
    # by a barrier and a device synchronisation); per operator the mean over a
    # region's K steps is taken, and the median over the regions is reported
    # with the spread (FlashRT §5: re-measure before accepting a number).
    regions = []
    walls = []
    gc.collect()
    gc.disable()                  # no collector pause inside an event pair
    for rep in range(args.repeats):
        barrier(pg)
        torch.cuda.synchronize()
        if rep == 0:
            clocks.mark()
        t_wall0 = time.perf_counter()
        recs = []
        for _ in range(args.steps):
            one_step(recs)
        torch.cuda.synchronize()
        walls.append(time.perf_counter() - t_wall0)
        barrier(pg)
        per_region = {}
        for op, e0, e1 in recs:
            per_region.setdefault(op.name, []).append(e0.elapsed_time(e1))
        regions.append(per_region)
    gc.enable()
    clk = clocks.stop()

    per_op = {op.name: {"op": op} for op in ops}
    region_mem = []                      # (bytes, ms) of the memory-bound rows, per region
    for per_region in regions:
        b = m = 0.0
        for name, ts in per_region.items():
            op = per_op[name]["op"]
            per_op[name].setdefault("region_ms", []).append(sum(ts) / len(ts))
            per_op[name].setdefault("all_ms", []).extend(ts)
            if op.bound != "tensor":
                b += op.algorithmic_bytes()
                m += sum(ts) / len(ts)
        region_mem.append((b, m))

    mem_bytes = mem_ms = 0.0
    step_ms = 0.0
    out_ops = {}
    for name, d in per_op.items():
        op = d["op"]
        ms = statistics.median(d["region_ms"])   # median over the regions of each region's mean
        step_ms += ms
        entry = {"ms": round(ms, 5), "ms_median": round(statistics.median(d["all_ms"]), 5),
                 "ms_regions": [round(x, 5) for x in d["region_ms"]],
                 "spread": round((max(d["region_ms"]) - min(d["region_ms"])) / ms, 4), "launches": op.launches,
                 "tokens_per_s": round(op.units() / (ms / 1e3), 1)}
        if op.bound == "tensor":
            tf = op.flops() / (ms / 1e3) / 1e12
            ratio = getattr(op, "peak_ratio", 1.0)
            peak = peaks["bf16_tflops"] * ratio
            entry.update({"tflops": round(tf, 1), "frac_of_peak": round(tf / peak, 4), "peak_tflops": round(peak, 1),
                          "frac_of_nominal": round(tf / (BF16_DENSE_NOMINAL_TFLOPS * ratio), 4),
                          "bytes": op.algorithmic_bytes(), "unfused_bytes": op.unfused_bytes()})
        else:
            gbs = op.algorithmic_bytes() / (ms / 1e3) / 1e9
            entry.update({"gbs": round(gbs, 1), "frac_of_peak": round(gbs / peaks["hbm_gbs"], 4),
                          "bytes": op.algorithmic_bytes(), "unfused_bytes": op.unfused_bytes()})
            mem_bytes += op.algorithmic_bytes()
            mem_ms += ms
        out_ops[name] = entry

    # value: the median region's aggregate; timing is the slowest rank, bytes sum over ranks
    region_vals = []
    for b, m in region_mem:
        m_max = max_over_ranks(pg, m)
        region_vals.append(sum_over_ranks(pg, b) / (m_max / 1e3) / 1e9 if m_max > 0 else 0.0)
    value = statistics.median(region_vals)
    step_ms_max = max_over_ranks(pg, step_ms)

    # roofline: the memory-bound kernel with the largest share of the step among
    # those whose launch moves more than L2 holds (HBM-bound by construction);
    # the launch-bound chain of small calls is reported by its per-call latency
    big = [(n, d) for n, d in out_ops.items()
           if "gbs" in d and per_op[n]["op"].algorithmic_bytes() // per_op[n]["op"].launches > L2_BYTES]
    mem_ops = big or [(n, d) for n, d in out_ops.items() if "gbs" in d] or \
        [(n, dict(d, gbs=0.0)) for n, d in out_ops.items()]
    dom_name, dom = max(mem_ops, key=lambda kv: kv[1]["ms"])
    dom_op = per_op[dom_name]["op"]
    roofline = {"kernel": dom_name, "bound": "hbm", "achieved": dom["gbs"], "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(dom["gbs"] / peaks["hbm_gbs"], 4),
                "peak_source": f"{peaks['source']} (burst copy)",
                "traffic": kernel_traffic(dom_name),
                "algorithmic_bytes_per_launch": dom_op.algorithmic_bytes() // dom_op.launches}
    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(step_ms_max, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, fp32 math, bf16/e4m3 out",
            "data": "synthetic (seeded numpy PCG64, the workloads' shapes and distributions)",
            "config": {"workload": "fused hot path: " + ", ".join(per_op), "parallelism": f"replicas x{world}",
                       "l2": "flushed (512 MB write, then read back) before every operator, outside its event pair",
                       "value_scope": "memory-bound fused kernels; GEMM timed in the same step, see ops",
                       "repeats": f"the {args.steps}-step timed region ran {args.repeats} times; per operator the "
                                  "median of the regions' means, spread = (max - min) / median"},
            "repeats": args.repeats, "value_regions": [round(v, 1) for v in region_vals],
            "roofline": roofline, "ops": out_ops, "clocks": clk,
            "peaks": {"hbm_gbs_measured_copy": peaks["hbm_gbs"], "bf16_tflops_measured": peaks["bf16_tflops"],
                      "bf16_tflops_measured_sustained": peaks["bf16_tflops_sustained"],
                      "source": peaks["source"], "hbm_gbs_nominal": 7900.0,
                      "bf16_tflops_dense_nominal": BF16_DENSE_NOMINAL_TFLOPS,
                      "nominal_source": "GB300 nominal figures (HBM3e 7.9 TB/s; dense bf16 2.25 PFLOP/s)",
                      "gbf_copy_gbs": copy_probe_gbs(gbf)},
            "latency_bound": {n: {"us_per_launch": round(d["ms"] * 1e3 / d["launches"], 3), "launches": d["launches"]}
                              for n, d in out_ops.items()
                              if "gbs" in d and per_op[n]["op"].algorithmic_bytes() // per_op[n]["op"].launches < (1 << 20)},
            "gpu_launches": args.repeats * args.steps * sum(op.launches for op in ops),
            "wall_s_timed_region": round(sum(walls), 3)}
    if with_gemm and "linear_bias_gelu" in out_ops:
        g = out_ops["linear_bias_gelu"]
        line["roofline_gemm"] = {"kernel": "linear_bias_gelu", "bound": "tensor", "achieved": g["tflops"],
                                 "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                 "frac": round(g["tflops"] / peaks["bf16_tflops"], 4),
                                 "frac_of_nominal": g["frac_of_nominal"],
                                 "peak_source": f"{peaks['source']} (burst cuBLAS bf16)",
                                 "traffic": kernel_traffic("linear_bias_gelu")}
        if args.gemm_sustained_s > 0:
            line["roofline_gemm"]["sustained"] = gemm_sustained(per_op["linear_bias_gelu"]["op"], local, peaks,
                                                                args.gemm_sustained_s)
        line["roofline_gemm"]["library_same_box"] = gemm_library_reference(per_op["linear_bias_gelu"]["op"], flush_l2)

    # decode-shaped QKV into a paged KV cache: launch-bound, timed on its own
    # (outside the step, so the step's aggregate keeps its composition)
    if not args.no_latency_extras:
        if "qwen3_qkv" in per_op:
            line["latency_bound"]["qwen3_qkv_decode_paged"] = measure_decode_paged(gbf, flush_l2)
        if "swiglu_ffn" in per_op:
            line["latency_bound"]["swiglu_decode"] = measure_swiglu_decode(gbf, flush_l2)
        if "linear_bias_gelu" in per_op:
            line["latency_bound"]["linear_decode"] = measure_linear_decode(gbf, flush_l2)

    # end to end through the C ABI with host buffers: H2D inputs, op, D2H outputs
    if not args.no_e2e:
        e2e = measure_e2e(ops, args, stream, copy_streams=args.e2e_copy_streams)
        e2e_ms = max_over_ranks(pg, e2e["mem_ms"])
        line["e2e"] = {"value": round(sum_over_ranks(pg, e2e["mem_bytes"]) / (e2e_ms / 1e3) / 1e9, 1),
                       "unit": UNIT, "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                       "copy_streams_per_direction": e2e["copy_streams"]}
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        line["cpu_baseline"] = run_cpu_baseline()
    if rank == 0:
        print(json.dumps(line))
    if pg is not None:
        pg.destroy_process_group()


def graph_latency_us(gbf, call, flush_l2, calls=100, reps=20):
    """`calls` back-to-back calls of `call` captured through the C ABI into one
    CUDA graph, replayed `reps` times after an L2 flush; median microseconds
    per call."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(calls):
            call()
    torch.cuda.synchronize()
    ts = []
    for it in range(reps + 3):
        flush_l2()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        if it >= 3:
            ts.append(e0.elapsed_time(e1))
    status, msg = gbf.device_status()
    if status != gbf.OK:
        raise RuntimeError(f"device status after a latency graph: {msg}")
    return statistics.median(ts) * 1e3 / calls


def measure_decode_paged(gbf, flush_l2, calls=100):
    """Decode-shaped QKV post-processing into a paged KV cache
    (workloads.qkv_decode_paged_case: 32 sequences' new tokens, Qwen3's 32 +
    2 x 8 heads x 128, per-head RMSNorm and 1D RoPE, K/V rows by slot mapping
    into a 16,384-row cache of 16-row blocks), per-call microseconds."""
    import torch
    import workloads
    from workloads import as_torch as from_bits
    c = workloads.qkv_decode_paged_case()
    t, hq, hkv, d = c["tokens"], c["n_q"], c["n_kv"], c["d"]
    qkv, qw, kw = from_bits(c["qkv"]), from_bits(c["q_w"]), from_bits(c["k_w"])
    pos = torch.from_numpy(c["pos"]).cuda()
    slots = torch.from_numpy(c["slots"]).cuda()
    q = torch.empty(t, hq, d, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(c["cache_rows"], hkv, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)

    def call():
        gbf.qkv_split_norm_rope(qkv, hq, hkv, d, gbf.QKNORM_PER_HEAD, qw, kw, c["eps"], gbf.ROPE_1D, pos,
                                c["theta"], q, kc, vc, slots=slots, cache_rows=c["cache_rows"])
    us = graph_latency_us(gbf, call, flush_l2, calls)
    return {"us_per_launch": round(us, 3), "launches": calls, "tokens": t,
            "cache_rows": c["cache_rows"], "block_rows": 16, "bytes_per_launch": bytes_qkv(t, hq, hkv, d),
            "note": "timed on its own after the step (not part of the step's aggregate)"}


def measure_swiglu_decode(gbf, flush_l2, rows=32, d=11008, calls=100):
    """SwiGLU silu(gate) * up on a decode batch: [rows, 2 x 11008] bf16
    (workloads.config_swiglu_ffn's row width and draws), per-call
    microseconds."""
    import workloads
    from workloads import as_torch as from_bits
    c = workloads.config_swiglu_ffn(rows=rows)
    x = from_bits(c["x"])
    y = x.new_empty(rows, d)

    def call():
        gbf.gated_act(x, y, gbf.ACT_SILU)
    us = graph_latency_us(gbf, call, flush_l2, calls)
    return {"us_per_launch": round(us, 3), "launches": calls, "rows": rows, "bytes_per_launch": rows * d * 6,
            "note": "timed on its own after the step (not part of the step's aggregate)"}


def measure_linear_decode(gbf, flush_l2, m=32, calls=50):
    """The config's Linear + bias + GELU (N 16384, K 4096) on a decode batch of
    m rows, where reading W bounds the call: `calls` calls in one CUDA graph,
    per-call microseconds, with cuBLASLt's fused bias + GELU on the same
    operands timed the same way (a comparison only)."""
    import torch
    import workloads
    from workloads import as_torch as from_bits
    c = workloads.linear_gelu_case(m, 16384, 4096, seed=0)
    x, w, b = from_bits(c["x"]), from_bits(c["w"]), from_bits(c["bias"])
    y = torch.empty(m, 16384, dtype=torch.bfloat16, device="cuda")

    def ours():
        gbf.linear_bias_gelu(x, w, b, y, act=gbf.ACT_GELU_TANH)

    def lt():
        torch._addmm_activation(b, x, w.t(), use_gelu=True)
    us = graph_latency_us(gbf, ours, flush_l2, calls)
    us_lt = graph_latency_us(gbf, lt, flush_l2, calls)
    w_bytes = 16384 * 4096 * 2
    return {"us_per_launch": round(us, 2), "launches": calls, "rows": m, "w_bytes": w_bytes,
            "gbs_of_w": round(w_bytes / us / 1e3, 1), "cublaslt_bias_gelu_us": round(us_lt, 2),
            "note": "timed on its own after the step (not part of the step's aggregate)"}


def gemm_sustained(op, cuda_index, peaks, seconds):
    """The GEMM launched back to back for about `seconds` on its operands (no
    L2 flush between launches: X and W stay partly resident, as they would in
    a model's repeated layer), timed with events around the whole run, with
    the SM clock and power sampled during it.  Reported against the measured
    sustained bf16 peak (a seconds-long cuBLAS loop under the power cap) and as
    time x median SM MHz, which takes the clock out of the comparison."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    op.run()
    e1.record()
    torch.cuda.synchronize()
    n = max(10, int(seconds * 1e3 / max(e0.elapsed_time(e1), 1e-3)))
    clocks = ClockSampler(cuda_index)
    clocks.start()
    clocks.mark()
    e0.record()
    for _ in range(n):
        op.run()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / n
    tf = op.flops() / (ms / 1e3) / 1e12
    sus = peaks.get("bf16_tflops_sustained")
    out = {"launches": n, "seconds": round(e0.elapsed_time(e1) / 1e3, 2), "ms_per_launch": round(ms, 5),
           "tflops": round(tf, 1), "peak": sus, "frac": round(tf / sus, 4) if sus else None,
           "frac_of_nominal": round(tf / BF16_DENSE_NOMINAL_TFLOPS, 4), "clocks": clk}
    if clk.get("sm_mhz"):
        out["ms_x_mhz"] = round(ms * clk["sm_mhz"], 1)
    return out


def gemm_library_reference(op, flush_l2, reps=20):
    """The same Linear + bias + GELU(tanh) through the vendor library on the
    same operands, timed exactly as the step times this library's GEMM (L2
    flushed before each launch, CUDA events, median of `reps`): cuBLASLt with
    its fused bias + GELU epilogue (torch._addmm_activation) and the plain
    cuBLAS GEMM without the epilogue (torch.matmul).  A comparison figure
    only: nothing on the library's own path calls either."""
    import torch
    x, w, b = op.x, op.w, op.b
    wt = w.t()

    def timed(fn):
        ts = []
        for it in range(reps + 3):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            if it >= 3:
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    out = {}
    try:
        out["cublaslt_bias_gelu_ms"] = round(timed(lambda: torch._addmm_activation(b, x, wt, use_gelu=True)), 5)
    except (RuntimeError, AttributeError) as e:
        out["cublaslt_bias_gelu_error"] = str(e)[:200]
    out["cublas_matmul_ms"] = round(timed(lambda: torch.matmul(x, wt)), 5)
    out["ours_ms"] = round(timed(op.run), 5)
    flops = op.flops()
    for k in list(out):
        if k.endswith("_ms"):
            out[k[:-3] + "_tflops"] = round(flops / (out[k] / 1e3) / 1e12, 1)
    return out


def measure_e2e(ops, args, stream, copy_streams=1):
    """The memory-bound operators fed from and drained to pinned host memory,
    timed with events from the first input copy to the last output copy of a
    step.  Within a step the operators are pipelined: the inputs of operator
    i+1 copy in while operator i runs and the outputs of operator i-1 copy
    out (every operator owns its device buffers).  With `copy_streams` > 1
    each tensor from 8 MB up is cut into that many pieces on as many streams
    per direction; on this part that was slower in this pipeline (141-174
    GB/s with four against 188-222 with one, the same box, alternating runs),
    although a bare bidirectional copy gains from more streams.  Steps are
    separated by a synchronisation."""
    import torch
    mem_ops = [op for op in ops if op.bound != "tensor"]
    host = {}
    for op in mem_ops:
        ins, outs = op.e2e_buffers()
        host[op.name] = ([t.cpu().pin_memory() for t in ins], ins, [torch.empty_like(t, device="cpu").pin_memory()
                                                                    for t in outs], outs)
    s_in = [torch.cuda.Stream() for _ in range(copy_streams)]
    s_out = [torch.cuda.Stream() for _ in range(copy_streams)]
    compute = torch.cuda.current_stream()
    h2d = sum(sum(t.numel() * t.element_size() for t in host[op.name][1]) for op in mem_ops)
    d2h = sum(sum(t.numel() * t.element_size() for t in host[op.name][3]) for op in mem_ops)
    mem_bytes = sum(op.algorithmic_bytes() for op in mem_ops)

    big = 8 << 20                 # tensors from 8 MB up are cut into pieces; smaller ones go whole

    def plan(pairs, streams):
        """(stream, src, dst) copies: large tensors split over every stream,
        small ones whole, dealt round-robin (thousands of tiny copies would
        leave the host behind the link)."""
        out, rr = [], 0
        for src, dst in pairs:
            if src.numel() * src.element_size() >= big:
                for st, a, b in zip(streams, torch.chunk(src.reshape(-1), len(streams)),
                                    torch.chunk(dst.reshape(-1), len(streams))):
                    out.append((st, a, b))
            else:
                out.append((streams[rr % len(streams)], src, dst))
                rr += 1
        return out

    plans_in = {op.name: plan(zip(host[op.name][0], host[op.name][1]), s_in) for op in mem_ops}
    plans_out = {op.name: plan(zip(host[op.name][3], host[op.name][2]), s_out) for op in mem_ops}
    steps = max(1, min(args.steps, 3))
    times = []
    for s in range(steps + 1):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(compute)
        for st in s_in + s_out:
            st.wait_event(e0)
        for op in mem_ops:
            hin, din, hout, dout = host[op.name]
            for st, hp, dp in plans_in[op.name]:
                with torch.cuda.stream(st):
                    dp.copy_(hp, non_blocking=True)
            for st in s_in:
                ready = torch.cuda.Event()
                ready.record(st)
                compute.wait_event(ready)
            op.run()
            done = torch.cuda.Event()
            done.record(compute)
            for st in s_out:
                st.wait_event(done)
            for st, dp, hp in plans_out[op.name]:
                with torch.cuda.stream(st):
                    hp.copy_(dp, non_blocking=True)
        for st in s_out:
            fin = torch.cuda.Event()
            fin.record(st)
            compute.wait_event(fin)
        e1.record(compute)
        torch.cuda.synchronize()
        if s > 0:                 # the first pass warms up
            times.append(e0.elapsed_time(e1))
    return {"mem_ms": sum(times) / len(times), "mem_bytes": mem_bytes, "h2d": h2d, "d2h": d2h,
            "copy_streams": copy_streams}


def main_reference(args):
    """The CPU oracle as it stands, timed on this machine's host cores on a bounded
    sample of the same workload, K steps after W warm-up steps."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    times = []
    vals = []
    res = None
    for i in range(args.warmup + args.steps):
        res = run_cpu_baseline(scale=2, all_cores=False)
        if i >= args.warmup:
            times.append(res["seconds"])
            vals.append(res["value"])
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * sum(times) / len(times), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy PCG64)",
            "config": {"workload": "fused hot path (bounded sample per step), CPU oracle of the unfused chains",
                       "parallelism": "1 host thread"},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": res.get("sample")},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "per_op": res["per_op"]}
    print(json.dumps(line))


def main_sweep(args):
    """`--sweep`: the add+RMSNorm+FP8 kernel over rows x hidden x mode, one JSON
    line per point (HBM GB/s and fraction of the measured copy bandwidth).
    Inputs come from torch's seeded generator on the device, drawn as the
    workloads draw them (x, res ~ N(0,1); weight 1+N(0,0.1); gate, shift,
    scale ~ N(0,0.2)); throughput does not depend on the values.  A point whose
    call moves less than 4 x L2 runs `sets` calls on distinct buffer sets back
    to back inside one event pair (together at least 4 x L2, at most 8 sets),
    as the QKV row of the step does: no call finds another's data in L2, and
    the per-call time is not rounded to the 1.024 us event step."""
    import torch
    import fusion_add_rmsnorm_gb300 as gbf
    peaks = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush_words = flush.view(torch.int64)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    shapes = [(r, h) for r in (4096, 16384, 65536) for h in (1024, 4096, 8192)]
    if args.sweep_shapes:
        shapes = [tuple(int(v) for v in sh.split("x")) for sh in args.sweep_shapes.split(",")]
    for rows, hidden in shapes:
        nbytes_call = bytes_add_rmsnorm(rows, hidden, 0, False)
        nsets = max(1, min(8, -(-4 * L2_BYTES // nbytes_call)))
        bf = dict(dtype=torch.bfloat16, device="cuda")
        sets = []
        for _ in range(nsets):
            x = torch.randn(rows, hidden, generator=gen, **bf)
            res = torch.randn(rows, hidden, generator=gen, **bf)
            sets.append((x, res, torch.empty_like(res), torch.empty(rows, hidden, dtype=torch.uint8, device="cuda")))
        vec = lambda m, sd: (m + sd * torch.randn(hidden, generator=gen, device="cuda")).to(torch.bfloat16)  # noqa
        w, gate, scale, shift = vec(1.0, 0.1), vec(0.0, 0.2), vec(0.0, 0.2), vec(0.0, 0.2)
        for name, mode, gated in (("weighted", 0, False), ("noweight", 1, False), ("ada", 2, True)):
            def call():
                for x, res, out, q in sets:
                    gbf.add_rmsnorm_fp8(x, res, out, q, mode, weight=w if mode == 0 else None,
                                        gate=gate if gated else None, ada_scale=scale if mode == 2 else None,
                                        ada_shift=shift if mode == 2 else None, eps=1e-6, fp8_scale=0.05)
            ts = []
            for it in range(args.warmup + args.steps):
                flush.fill_(1)
                flush_words.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                call()
                e1.record()
                torch.cuda.synchronize()
                if it >= args.warmup:
                    ts.append(e0.elapsed_time(e1) / nsets)
            ms = sorted(ts)[len(ts) // 2]
            nbytes = bytes_add_rmsnorm(rows, hidden, mode, gated)
            gbs = nbytes / (ms / 1e3) / 1e9
            print(json.dumps({"sweep": "add_rmsnorm_fp8", "mode": name, "rows": rows, "hidden": hidden,
                              "us_median": round(ms * 1e3, 2), "bytes": nbytes, "gbs": round(gbs, 1),
                              "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 4),
                              "l2_flushed": True, "timed_calls": args.steps, "calls_per_event": nsets}),
                  flush=True)
        del sets


def main_copy_curve(args):
    """`--copy-curve`: the bandwidth a plain copy reaches at the sizes of the
    step's shorter calls, timed exactly as the step times them (L2 flushed,
    then `sets` calls on distinct buffers inside one event pair): this
    library's copy kernel and torch's, one JSON line per point.  It shows what
    any kernel moving that many bytes in one launch can reach, ramp-up and
    tail included."""
    import torch
    import fusion_add_rmsnorm_gb300 as gbf
    peaks = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush_words = flush.view(torch.int64)
    for mb in (12.5, 25, 50, 100, 200, 400):
        n = int(mb * 1e6) // 16 * 16
        for nsets in (1, 4):
            srcs = [torch.ones(n, dtype=torch.uint8, device="cuda") for _ in range(nsets)]
            dsts = [torch.empty_like(t) for t in srcs]
            for impl in ("gbf_copy", "torch"):
                ts = []
                for it in range(args.warmup + args.steps):
                    flush.fill_(1)
                    flush_words.sum()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    for src, dst in zip(srcs, dsts):
                        if impl == "torch":
                            dst.copy_(src)
                        else:
                            gbf.copy(src, dst)
                    e1.record()
                    torch.cuda.synchronize()
                    if it >= args.warmup:
                        ts.append(e0.elapsed_time(e1) / nsets)
                ms = sorted(ts)[len(ts) // 2]
                gbs = 2 * n / (ms / 1e3) / 1e9
                print(json.dumps({"copy_curve": impl, "bytes_moved": 2 * n, "sets": nsets,
                                  "us_median": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                                  "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 4)}), flush=True)
            del srcs, dsts


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--repeats", type=int, default=3, help="times the K-step timed region runs (median reported)")
    ap.add_argument("--gemm-sustained-s", type=float, default=3.0,
                    help="seconds of back-to-back GEMM launches for the sustained figure (0: skip)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-gemm", action="store_true", help="leave the GEMM row out of the step")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end pass")
    ap.add_argument("--no-latency-extras", action="store_true",
                    help="skip the decode-shape latency measurements taken after the step")
    ap.add_argument("--e2e-copy-streams", type=int, default=1, help="copy streams per direction in the e2e pass")
    ap.add_argument("--only", default="", help="comma-separated subset of: " + ", ".join(OP_NAMES))
    ap.add_argument("--small", action="store_true", help="profiling-size cases (still larger than L2)")
    ap.add_argument("--sweep", action="store_true",
                    help="add+RMSNorm+FP8 over rows {4096, 16384, 65536} x hidden {1024, 4096, 8192} x 3 modes")
    ap.add_argument("--copy-curve", action="store_true",
                    help="plain-copy bandwidth at 25 MB..800 MB moved, timed as the step times its calls")
    ap.add_argument("--sweep-shapes", default="",
                    help="with --sweep: comma-separated ROWSxHIDDEN points instead of the grid (e.g. 8192x8192)")
    ap.add_argument("--_cpu-baseline-child", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--_cpu-baseline-start", type=float, default=0.0, help=argparse.SUPPRESS)
    ap.add_argument("--_cpu-baseline-nogemm", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.sweep:
        main_sweep(args)
        return
    if args.copy_curve:
        main_copy_curve(args)
        return
    if args._cpu_baseline_child:
        if args._cpu_baseline_start:
            import workloads  # noqa: F401  (imports done before the shared start)
            from oracle import chains  # noqa: F401
            time.sleep(max(0.0, args._cpu_baseline_start - time.time()))
        print(json.dumps(cpu_baseline_sample(args._cpu_baseline_child, gemm=not args._cpu_baseline_nogemm)))
        return
    if args.impl == "reference":
        main_reference(args)
        return
    main_gpu(args)


if __name__ == "__main__":
    main()
