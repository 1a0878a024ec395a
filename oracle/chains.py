"""The operator chains that each fused kernel replaces, run one operator at a time.

Test infrastructure only: nothing in the product path imports this package.

Inputs and outputs are raw storage bits (uint16 for bfloat16, uint8 for E4M3,
int32 for positions), exactly the bytes a caller hands to the fused kernel.
Every tensor the fused kernel writes is materialised in its storage format;
every intermediate the fusion removes stays float64 (FlashRT §2.1: the fused
data "only pass through registers / shared memory").  Page names are those of
oracle/ops.py.
"""
import numpy as np

from . import ops
from .formats import bf16_decode, bf16_encode, bf16_round, e4m3_decode

NORM_WEIGHT, NORM_NOWEIGHT, NORM_ADA = 0, 1, 2
QKNORM_PER_HEAD, QKNORM_FULL_WIDTH, QKNORM_LAYERNORM = 0, 1, 2
ROPE_1D, ROPE_3D = 0, 1


def add_rmsnorm_fp8(x, res, eps, s_q, mode, weight=None, gate=None,
                    ada_scale=None, ada_shift=None, round_y_bf16=False):
    """Residual add (optionally gated) -> RMSNorm / _noweight / AdaRMSNorm ->
    static E4M3 quantisation: the "three in one" of FlashRT §2.1 and the
    six-op gate_res_adarms_fp8_static of FlashRT §3.

    x, res: bf16 bits [rows, H]; weight / gate / ada_scale / ada_shift: bf16
    bits [H].  Returns (res_out bf16 bits [rows, H], q E4M3 codes [rows, H]).

    1. r = x + res, or r = res + gate * x with a gate (float64);
    2. res_out = bf16(r): the new residual stream, which the next layer and the
       norm both read (an unfused chain materialises it, so the norm sees the
       rounded value r_hat);
    3. n = r_hat / sqrt(mean(r_hat^2) + eps) over H;
    4. y = n * w (weighted), y = n (_noweight), y = n * (1 + scale) + shift (ada);
       y stays float64 (it never reaches memory in the fused kernel);
    5. q = E4M3(y / s_q), saturating.
    `round_y_bf16` models an unfused chain that stores y in bf16 before the
    quantiser; it is a comparison switch, not the parity reference."""
    xv = bf16_decode(x)
    rv = bf16_decode(res)
    if gate is None:
        r = ops.residual_add(xv, rv)
    else:
        r = ops.gated_residual_add(xv, rv, bf16_decode(gate)[None, :])
    res_out = bf16_encode(r)
    r_hat = bf16_decode(res_out)
    if mode == NORM_WEIGHT:
        y = ops.rmsnorm(r_hat, eps, bf16_decode(weight)[None, :])
    elif mode == NORM_NOWEIGHT:
        y = ops.rmsnorm(r_hat, eps)
    elif mode == NORM_ADA:
        n = ops.rmsnorm(r_hat, eps)
        y = ops.ada_modulate(n, bf16_decode(ada_scale)[None, :], bf16_decode(ada_shift)[None, :])
    else:
        raise ValueError(f"unknown norm mode {mode}")
    if round_y_bf16:
        y = bf16_round(y)
    q = ops.quant_e4m3_static(y, s_q)
    return res_out, q


def qkv_split_norm_rope(qkv, n_q_heads, n_kv_heads, head_dim, norm, q_w, k_w, eps,
                        rope, pos, theta, sections=None, slots=None, cache_rows=None,
                        rope3d=None, q_b=None, k_b=None):
    """Packed-QKV post-processing: split -> Q/K RMSNorm -> RoPE -> write Q and
    the K/V cache; V passes through (FlashRT §2.2: Qwen3 q_norm/k_norm + RoPE +
    KV-cache write; Wan packed-QKV split + two RMSNorms + 3D RoPE; the shared
    contract "Q/K norm -> RoPE, V direct").

    qkv: bf16 bits [T, (Hq + 2 Hkv) * D]; q_w, k_w: bf16 bits [D] (per head) or
    [H * D] (full width); pos: int32 [T] (1D) or [T, 3] (3D).  norm
    QKNORM_LAYERNORM is a per-head LayerNorm instead of the RMSNorm
    (FlashRT §2.2, Chameleon prefill: LayerNorm(Q) + LayerNorm(K) + rotate_half
    RoPE), with optional bf16 biases q_b, k_b [D] (None: 0).  The K and V rows
    of token t go to cache row slots[t] (row t when slots is None) of caches
    holding cache_rows rows (T when None).  Returns bf16 bits
    (q [T, Hq, D], k_cache [cache_rows, Hkv, D], v_cache [cache_rows, Hkv, D]);
    cache rows no token maps to are left zero.

    The normalised Q and K stay float64 between the norm and the rotation
    (the fused kernel keeps them in registers); only the rotated result is
    rounded to bf16.  V is copied bit for bit."""
    t = qkv.shape[0]
    packed = bf16_decode(qkv).reshape(t, -1)
    q, k, _ = ops.split_packed_qkv(packed, n_q_heads, n_kv_heads, head_dim)
    _, _, v_bits = ops.split_packed_qkv(np.asarray(qkv).reshape(t, -1), n_q_heads, n_kv_heads, head_dim)
    qw = bf16_decode(q_w)
    kw = bf16_decode(k_w)
    if norm == QKNORM_PER_HEAD:
        qn = ops.qk_rmsnorm_per_head(q, qw, eps)
        kn = ops.qk_rmsnorm_per_head(k, kw, eps)
    elif norm == QKNORM_FULL_WIDTH:
        qn = ops.qk_rmsnorm_full_width(q, qw, eps)
        kn = ops.qk_rmsnorm_full_width(k, kw, eps)
    elif norm == QKNORM_LAYERNORM:
        qn = ops.qk_layernorm_per_head(q, qw, None if q_b is None else bf16_decode(q_b), eps)
        kn = ops.qk_layernorm_per_head(k, kw, None if k_b is None else bf16_decode(k_b), eps)
    else:
        raise ValueError(f"unknown qk-norm mode {norm}")
    if rope == ROPE_1D:
        qr = ops.rope_rotate_half(qn, pos, theta)
        kr = ops.rope_rotate_half(kn, pos, theta)
    elif rope == ROPE_3D:
        fn = rope3d or ops.rope_3d_sections
        qr = fn(qn, pos, sections, theta)
        kr = fn(kn, pos, sections, theta)
    else:
        raise ValueError(f"unknown rope mode {rope}")
    q_out = bf16_encode(qr)
    rows = t if cache_rows is None else cache_rows
    k_cache = np.zeros((rows, n_kv_heads, head_dim), np.uint16)
    v_cache = np.zeros((rows, n_kv_heads, head_dim), np.uint16)
    dest = np.arange(t) if slots is None else np.asarray(slots, np.int64)
    k_cache[dest] = bf16_encode(kr)
    v_cache[dest] = v_bits
    return q_out, k_cache, v_cache


def linear_bias_gelu(x, w, bias=None, act_gelu=True, act=None):
    """Linear -> BiasAdd -> GELU(tanh) (OpenPPL §4.3 epilogue; Autofuse
    "MatMul -> BiasAdd -> ReLU" pattern with GELU; RFC §3.5 npu_linear).

    x: bf16 bits [M, K]; w: bf16 bits [N, K]; bias: bf16 bits [N] or None.
    The product is an exact-up-to-order float64 dot over K; the output is
    rounded once to bf16.  `act` (ops.ACT_*) selects another activation
    (GELU erf, SiLU; RFC §3.6) in place of act_gelu's GELU(tanh)."""
    a = ops.linear(bf16_decode(x), bf16_decode(w), None if bias is None else bf16_decode(bias))
    if act is not None:
        a = ops.activation(a, act)
    elif act_gelu:
        a = ops.gelu_tanh(a)
    return bf16_encode(a)


def linear_fp8_act(xq, x_scale, wq, w_scale, bias=None, act=None):
    """Quantised MatMul + activation (RFC §2.1 / §3.4: npu_quant_matmul_gelu,
    A8W8 with a tanh or erf GELU): E4M3 activation codes [M, K] with one
    descale (the codes fused_add_rmsnorm_fp8 writes, code * x_scale), E4M3
    weight codes [N, K] with one descale per output channel, optional bf16
    bias [N], then the activation (ops.ACT_*, None for none).  Exact float64
    dot of the decoded values; output rounded once to bf16."""
    a = ops.linear_dequant(e4m3_decode(xq), x_scale, e4m3_decode(wq), w_scale,
                           None if bias is None else bf16_decode(bias))
    if act is not None:
        a = ops.activation(a, act)
    return bf16_encode(a)


def fold_norm_weight_bf16(w, gamma, gemma_style=True):
    """Pre-fold of a norm weight into the next Linear's columns in binary32:
    g = 1 + gamma (or gamma), W' = W * g, each one IEEE binary32 operation,
    then one bf16 rounding (FlashRT §3, the `_noweight` kernel's weight).
    w: bf16 bits [N, K]; gamma: bf16 bits [K]; returns bf16 bits [N, K]."""
    wf = bf16_decode(w).astype(np.float32)
    gf = bf16_decode(gamma).astype(np.float32)
    return bf16_encode(ops.fold_norm_weight(wf, gf, gemma_style, dtype=np.float32).astype(np.float64))


def gated_act(x, d, act):
    """Gated activation of a [rows, 2d] projection holding [gate | up]:
    y = act(gate) * up, rounded once to bf16 (RFC §2.4 / §3.6: npu_swiglu
    for SiLU, npu_gelu_mul for a GELU; two elementwise ops, one HBM pass).

    x: bf16 bits [rows, 2d]; returns bf16 bits [rows, d]."""
    v = bf16_decode(x).reshape(-1, 2 * d)
    return bf16_encode(ops.gated_activation(v[:, :d], v[:, d:], act))


def bn_fold_bf16(w, b, gamma, beta, mean, var, eps):
    """BatchNorm folding of bf16 weights in binary32 (OpenPPL §3.1, §6.2).

    w: bf16 bits [out_ch, inner] (a conv weight [Cout, Cin, kh, kw] flattened
    per output channel); b: bf16 bits [out_ch] or None; gamma, beta, mean, var:
    float32 [out_ch].  The weights are widened to binary32, folded with one
    IEEE binary32 operation per step (ops.bn_fold, float32), and the results
    rounded once to bf16.  Returns (w' bits, b' bits)."""
    wf = bf16_decode(w).astype(np.float32)
    bf = None if b is None else bf16_decode(b).astype(np.float32)
    w_new, b_new = ops.bn_fold(wf, bf, gamma, beta, mean, var, np.float32(eps), dtype=np.float32)
    return bf16_encode(w_new.astype(np.float64)), bf16_encode(b_new.astype(np.float64))
