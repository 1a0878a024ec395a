"""Host logic of bench.py that needs no GPU: the kernel source hash behind the
DRAM-traffic record changes with the code and not with comments or layout."""
import importlib.util
import os

import numpy as np

from conftest import ROOT


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_strip_comments_keeps_code_and_literals():
    b = _bench()
    src = 'int a; // one\n/* two\n three */ const char* s = "x // y /* z */"; char c = \'"\';\n  float f;'
    assert b.strip_comments(src) == 'int a; const char* s = "x // y /* z */"; char c = \'"\'; float f;'


def test_comment_and_layout_edits_do_not_change_the_stripped_source():
    b = _bench()
    code = "__global__ void k(int* p) {\n  p[0] = 1;  // set\n}\n"
    edited = "/* a new header comment */\n__global__ void k(int* p) {\n\n    p[0] = 1;\n}\n"
    changed = "__global__ void k(int* p) {\n  p[0] = 2;\n}\n"
    assert b.strip_comments(code) == b.strip_comments(edited)
    assert b.strip_comments(code) != b.strip_comments(changed)


def test_every_kernel_file_hashes():
    b = _bench()
    for op, src in b.KERNEL_FILE.items():
        h = b.kernel_source_hash(src)
        assert h is not None and len(h) == 16 and int(h, 16) >= 0, op


# The fused and unfused byte counts of the graph-autofusion article's benefit
# model (阶段二收益估算: before fusion every operator reads its inputs and writes
# its output; after, one kernel reads the chain's inputs and writes its outputs
# once), worked out by hand per operator at each configuration:
#   [16, 256] add + RMSNorm + FP8, N = 4096: fused 7N + 2H = 28672 + 512; unfused
#     add 6N + norm 4N + 2H + quant 3N = 24576 + 16896 + 12288;
#   Pi0.5 gated AdaRMSNorm [10, 1024], N = 10240, H = 1024: fused 7N + 6H
#     = 71680 + 6144; unfused mul 43008 + add 61440 + norm 40960 + (1 + scale)
#     43008 + shift 43008 + quant 30720;
#   Qwen3 QKV [4096, 48 x 128]: fused 2 x 4096 x 6144 x 2; unfused Q 4 x 33554432
#     + K 6 x 8388608 + V 2 x 8388608;
#   Wan QKV [32760, 3 x 5120]: Q-sized pass 32760 x 5120 x 2 = 335462400 bytes;
#     fused 6 passes; unfused split 6 + two norms 4 + two ropes 4 = 14 passes;
#   Linear 8192 x 16384 x 4096: fused X 67108864 + W 134217728 + b 32768 + Y
#     268435456; unfused GEMM (no bias) + bias add (4 Y + b) + GELU (4 Y);
#   BN fold [16384, 4096]: W read + written 268435456, b read + written 65536,
#     four float32 parameter vectors 262144.
BENEFIT_MODEL = {
    "add_rmsnorm_fp8": (29184, 53760),
    "pi05_ada_call": (77824, 262144),
    "qwen3_qkv": (100663296, 201326592),
    "wan_qkv3d": (2012774400, 4696473600),
    "linear_bias_gelu": (469794816, 1543536640),
    "bn_fold": (268763136, None),
}


def test_byte_model_matches_the_benefit_model_worked_by_hand():
    b = _bench()
    got = {
        "add_rmsnorm_fp8": (b.bytes_add_rmsnorm(16, 256, 0, False), b.bytes_unfused_add_rmsnorm(16, 256, 0, False)),
        "pi05_ada_call": (b.bytes_add_rmsnorm(10, 1024, 2, True), b.bytes_unfused_add_rmsnorm(10, 1024, 2, True)),
        "qwen3_qkv": (b.bytes_qkv(4096, 32, 8, 128), b.bytes_unfused_qkv(4096, 32, 8, 128, 0)),
        "wan_qkv3d": (b.bytes_qkv(32760, 40, 40, 128), b.bytes_unfused_qkv(32760, 40, 40, 128, 1)),
        "linear_bias_gelu": (b.bytes_linear(8192, 16384, 4096), b.bytes_unfused_linear(8192, 16384, 4096)),
        "bn_fold": (b.bytes_bn_fold(16384, 4096), None),
    }
    assert got == BENEFIT_MODEL


def test_byte_model_fused_never_exceeds_unfused():
    b = _bench()
    for rows, hidden in ((1, 8), (16, 256), (65536, 4096)):
        for mode in (0, 1, 2):
            for gated in (False, True):
                fused = b.bytes_add_rmsnorm(rows, hidden, mode, gated)
                assert fused < b.bytes_unfused_add_rmsnorm(rows, hidden, mode, gated), (rows, hidden, mode, gated)
    for norm in (0, 1, 2):
        assert b.bytes_qkv(64, 8, 2, 128) < b.bytes_unfused_qkv(64, 8, 2, 128, norm)


def test_decode_paged_case_is_a_slot_mapping_into_distinct_blocks():
    """The decode workload the bench times on the paged cache: one token per
    sequence, each in its own 16-row block, at the row of its position."""
    import workloads
    c = workloads.qkv_decode_paged_case()
    pos, slots = c["pos"].astype(np.int64), c["slots"].astype(np.int64)
    assert c["qkv"].shape == (32, (32 + 2 * 8) * 128) and c["cache_rows"] == 16384
    assert pos.min() >= 0 and pos.max() < 4096
    assert slots.min() >= 0 and slots.max() < c["cache_rows"]
    assert np.array_equal(slots % 16, pos % 16)
    assert len(np.unique(slots // 16)) == len(slots)


def test_latency_extras_flag_parses():
    """`--no-latency-extras` (the launch-list capture's flag) is a bench option."""
    import subprocess
    import sys
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"], capture_output=True, text=True)
    assert out.returncode == 0 and "--no-latency-extras" in out.stdout
