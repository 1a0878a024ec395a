"""Unfused operators, one function per operator, in float64 unless stated.

Test infrastructure only: nothing in the product path imports this package.

Each function is the plain definition of one operator of the chains that the
fused kernels replace.  Nothing is blocked, fused or reordered; a reader can
check each line against the formula it cites.  Page citations use the page
title and section:

* OpenPPL  -- "OpenPPL算子融合深度解析：从图优化到推理性能提升" (codechina.net)
* HowTo    -- the operator-fusion how-to on discosf.com (its HTML title reads
              "企业官网建设流程全解析"; the body is "算子融合推理优化")
* Autofuse -- the CANN graph-autofusion article (aitangshan.cn)
* RFC      -- "RFC：自动融合: 扩展统一 Pattern Matcher 覆盖量化融合与 GMM/MM+激活"
              (MindIE-SD issue #298)
* FlashRT  -- "FlashRT 跨层融合深度解析：从 RMSNorm+QKV 到被证伪的死胡同优化模式"
"""
import numpy as np

from .formats import e4m3_encode_sat

# ------------------------------------------------------------ residual add


def residual_add(x, res):
    """r = x + res.  The residual Add that OpenPPL §3.3 turns into an epilogue."""
    return np.asarray(x, np.float64) + np.asarray(res, np.float64)


def gated_residual_add(x, res, gate):
    """r = res + gate * x, gate broadcast over tokens.  The gated residual of
    FlashRT §3 (gate_res_adarms_fp8_static: gate multiply + residual)."""
    return np.asarray(res, np.float64) + np.asarray(gate, np.float64) * np.asarray(x, np.float64)


# ----------------------------------------------------------------- RMSNorm


def rms_inverse(r, eps, axis=-1):
    """inv = 1 / sqrt(mean(r**2) + eps) over `axis` (kept as a size-1 axis)."""
    r = np.asarray(r, np.float64)
    ms = np.mean(r * r, axis=axis, keepdims=True)
    return 1.0 / np.sqrt(ms + eps)


def rmsnorm(r, eps, weight=None, axis=-1):
    """n = r * inv; y = n * w when a weight is given (the weighted kernel of
    FlashRT §2.1), y = n for the `_noweight` kernel of FlashRT §2.1/§3, whose
    weight was pre-multiplied into the next GEMM."""
    n = np.asarray(r, np.float64) * rms_inverse(r, eps, axis)
    if weight is None:
        return n
    return n * np.asarray(weight, np.float64)


def ada_modulate(n, scale, shift):
    """AdaRMSNorm modulation y = n * (1 + scale) + shift (FlashRT §3,
    gate_res_adarms_fp8_static); scale and shift broadcast over tokens."""
    return np.asarray(n, np.float64) * (1.0 + np.asarray(scale, np.float64)) + np.asarray(shift, np.float64)


# ------------------------------------------------------ static FP8 quantise


def quant_e4m3_static(y, s_q):
    """Static-scale FP8 quantisation (FlashRT §3, "_static": the activation
    scale is a constant fixed at calibration time).

    The scale is a descale: code = e4m3(y / s_q), dequantised value = code * s_q.
    s_q crosses the C boundary as a binary32, so its binary32 value is used.
    y / s_q is formed in float64 and rounded once to binary32; the E4M3 encoder
    then saturates to +-448 and rounds that binary32 value to nearest even.
    The binary32 step follows the pages' precision rule for fused kernels: the
    intermediate is held in an FP32 register and converted to the storage type
    once, at the write (OpenPPL §6.2: FP32 accumulators, converted only on the
    write-back; HowTo §4.1: keep the FP32 accumulator and convert once before
    writing).  The two readings differ only within half a binary32 ulp of an
    E4M3 midpoint."""
    s = np.float64(np.float32(s_q))
    v = (np.asarray(y, np.float64) / s).astype(np.float32)
    return e4m3_encode_sat(v)


# -------------------------------------------------------------------- RoPE


def rope_frequencies(d, theta):
    """omega_j = theta ** (-2 j / d) for j < d/2: the standard rotary table
    over a rotated width d."""
    j = np.arange(d // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * j / d)


def rope_rotate_half(u, pos, theta):
    """rotate_half RoPE over the last axis (width d, half = d/2).

    u: [..., T, H, d] or [T, H, d]; pos: [T] (one position per token).
    For j < half, with a = pos * omega_j:
        o[j]        = u[j] cos a - u[j + half] sin a
        o[j + half] = u[j + half] cos a + u[j] sin a
    (the Q/K post-processing RoPE of FlashRT §2.2, the RoPE of RFC §2.4)."""
    u = np.asarray(u, np.float64)
    d = u.shape[-1]
    half = d // 2
    omega = rope_frequencies(d, theta)                        # [half]
    a = np.asarray(pos, np.float64)[:, None] * omega[None, :]  # [T, half]
    c = np.cos(a)[:, None, :]
    s = np.sin(a)[:, None, :]
    lo, hi = u[..., :half], u[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def rope_3d_sections(u, pos3, sections, theta):
    """3D RoPE for video tokens (FlashRT §2.2, Wan: packed QKV split + two
    RMSNorms + 3D RoPE).

    Reading taken: the head dimension is cut into contiguous chunks of widths
    sections = (d_t, d_h, d_w); chunk c rotates with the token's c-th grid
    coordinate pos3[:, c], doing rotate_half inside the chunk (partner at
    +d_c/2) with its own table omega_j = theta ** (-2 j / d_c)."""
    u = np.asarray(u, np.float64)
    out = np.empty_like(u)
    start = 0
    for c, width in enumerate(sections):
        if width:
            out[..., start:start + width] = rope_rotate_half(
                u[..., start:start + width], np.asarray(pos3)[:, c], theta)
        start += width
    assert start == u.shape[-1], "sections must cover the head dimension"
    return out


def rope_3d_global_pairs(u, pos3, sections, theta):
    """Alternative reading of the 3D layout, kept only for comparison: one
    rotate_half over the full head (pairs j, j + d/2) whose d/2 frequency slots
    are cut into sections (d_t/2, d_h/2, d_w/2) taking positions t, h, w."""
    u = np.asarray(u, np.float64)
    d = u.shape[-1]
    half = d // 2
    pos3 = np.asarray(pos3, np.float64)
    a = np.empty((u.shape[-3], half))
    j0 = 0
    for c, width in enumerate(sections):
        n = width // 2
        j = np.arange(n, dtype=np.float64)
        a[:, j0:j0 + n] = pos3[:, c:c + 1] * np.power(np.float64(theta), -2.0 * j / width)[None, :]
        j0 += n
    c = np.cos(a)[:, None, :]
    s = np.sin(a)[:, None, :]
    lo, hi = u[..., :half], u[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


# ------------------------------------------------------- packed QKV layout


def split_packed_qkv(qkv, n_q_heads, n_kv_heads, head_dim):
    """Split one packed projection row [Q | K | V] into per-head views.

    The packed row is the output of the merged [3h, h] QKV GEMM of OpenPPL
    §3.2: all Q heads, then all K heads, then all V heads, heads contiguous."""
    t = qkv.shape[0]
    nq = n_q_heads * head_dim
    nk = n_kv_heads * head_dim
    q = qkv[:, :nq].reshape(t, n_q_heads, head_dim)
    k = qkv[:, nq:nq + nk].reshape(t, n_kv_heads, head_dim)
    v = qkv[:, nq + nk:nq + 2 * nk].reshape(t, n_kv_heads, head_dim)
    return q, k, v


def qk_rmsnorm_per_head(u, weight, eps):
    """RMSNorm of every head over its head_dim, weight indexed by d
    (the q_norm / k_norm of FlashRT §2.2, Qwen3 path)."""
    return rmsnorm(u, eps, np.asarray(weight, np.float64)[None, None, :], axis=-1)


def qk_rmsnorm_full_width(u, weight, eps):
    """RMSNorm over all heads x head_dim of a token, weight indexed by
    h * head_dim + d (FlashRT §2.2, Wan path)."""
    t, h, d = u.shape
    flat = np.asarray(u, np.float64).reshape(t, h * d)
    return rmsnorm(flat, eps, np.asarray(weight, np.float64)[None, :], axis=-1).reshape(t, h, d)


def layernorm(u, eps, weight=None, bias=None, axis=-1):
    """LayerNorm over `axis`: mu = mean(u), var = mean((u - mu)**2),
    y = (u - mu) / sqrt(var + eps) * w + b (a missing weight is 1, a missing
    bias 0).  Two passes over the values: the mean first, then the centred
    squares."""
    u = np.asarray(u, np.float64)
    mu = np.mean(u, axis=axis, keepdims=True)
    c = u - mu
    var = np.mean(c * c, axis=axis, keepdims=True)
    y = c / np.sqrt(var + eps)
    if weight is not None:
        y = y * np.asarray(weight, np.float64)
    if bias is not None:
        y = y + np.asarray(bias, np.float64)
    return y


def qk_layernorm_per_head(u, weight, bias, eps):
    """LayerNorm of every head over its head_dim, weight and bias indexed by d
    (the LayerNorm(Q) + LayerNorm(K) of FlashRT §2.2, Chameleon prefill path)."""
    return layernorm(u, eps, np.asarray(weight, np.float64)[None, None, :],
                     None if bias is None else np.asarray(bias, np.float64)[None, None, :], axis=-1)


# ------------------------------------------------------- Linear and GELU


def linear(x, w, b=None):
    """nn.Linear: y = x @ W^T + b with W stored [out, in] (RFC §3.5, npu_linear)."""
    y = np.asarray(x, np.float64) @ np.asarray(w, np.float64).T
    if b is not None:
        y = y + np.asarray(b, np.float64)[None, :]
    return y


GELU_C0 = 0.7978845608      # the two constants exactly as printed in the
GELU_C1 = 0.044715          # ConvEpilogue sketch of OpenPPL §4.3


def gelu_tanh(a):
    """GELU, tanh form: 0.5 a (1 + tanh(0.7978845608 (a + 0.044715 a^3)))
    (OpenPPL §4.3, activation_type 2 of the epilogue)."""
    a = np.asarray(a, np.float64)
    return 0.5 * a * (1.0 + np.tanh(GELU_C0 * (a + GELU_C1 * a * a * a)))


def gelu_erf(a):
    """GELU, exact (erf) form: 0.5 a (1 + erf(a / sqrt(2))) -- the non-tanh
    F.gelu that RFC §2.4 / §3.6 maps to npu_gelu.  erf is scipy's."""
    from scipy.special import erf
    a = np.asarray(a, np.float64)
    return 0.5 * a * (1.0 + erf(a / np.sqrt(2.0)))


def silu(a):
    """SiLU a * sigmoid(a) = a / (1 + exp(-a)) (the gate of npu_swiglu, RFC
    §2.4 / §3.6)."""
    a = np.asarray(a, np.float64)
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


ACT_GELU_TANH, ACT_GELU_ERF, ACT_SILU = 1, 2, 3


def activation(a, act):
    """The activation selected by `act` (ACT_GELU_TANH / ACT_GELU_ERF / ACT_SILU)."""
    if act == ACT_GELU_TANH:
        return gelu_tanh(a)
    if act == ACT_GELU_ERF:
        return gelu_erf(a)
    if act == ACT_SILU:
        return silu(a)
    raise ValueError(f"unknown activation {act}")


def gated_activation(gate, up, act):
    """act(gate) * up: SwiGLU with SiLU (npu_swiglu, vLLM's SiluAndMul),
    GELU x Mul with a GELU (npu_gelu_mul: up_out * gelu(gate_out)); RFC §2.4,
    §3.6."""
    return activation(gate, act) * np.asarray(up, np.float64)


def fold_norm_weight(w, gamma, gemma_style=True, dtype=np.float64):
    """Fold a norm's per-column weight into the next Linear (FlashRT §3: the
    `_noweight` RMSNorm leaves its weight, Gemma-style 1 + gamma, to the next
    GEMM): W'[n, k] = W[n, k] * (1 + gamma[k]) (or * gamma[k]), since
    Linear(y * g) = y @ (W * g)^T.  In `dtype` one operation per step: g, then
    the product."""
    w = np.asarray(w, dtype)
    gamma = np.asarray(gamma, dtype)
    g = (dtype(1.0) + gamma) if gemma_style else gamma
    return w * g[None, :]


def linear_dequant(xq, x_scale, wq, w_scale, b=None):
    """Quantised Linear (RFC §2.1 / §3.4, npu_quant_matmul with x1Scale and
    x2Scale): y = (xq * x_scale) @ (wq * w_scale[:, None])^T + b, with the
    integer-valued or FP8 operands given as their real values, one per-tensor
    activation scale and one scale per weight row (output channel)."""
    x = np.asarray(xq, np.float64) * np.float64(x_scale)
    w = np.asarray(wq, np.float64) * np.asarray(w_scale, np.float64)[:, None]
    return linear(x, w, b)


# -------------------------------------------------------------- BatchNorm


def batchnorm_inference(y, gamma, beta, mean, var, eps, channel_axis=-1):
    """Inference BatchNorm y' = gamma (y - mean) / sqrt(var + eps) + beta
    (OpenPPL §3.1; HowTo §2.1), per channel along `channel_axis`."""
    y = np.asarray(y, np.float64)
    shape = [1] * y.ndim
    shape[channel_axis] = -1

    def ch(p):
        return np.asarray(p, np.float64).reshape(shape)
    return ch(gamma) * (y - ch(mean)) / np.sqrt(ch(var) + eps) + ch(beta)


def bn_fold(w, b, gamma, beta, mean, var, eps, dtype=np.float32):
    """Fold an inference BatchNorm into the producing Conv/Linear weights.

    OpenPPL §3.1 and HowTo §2.1: scale = gamma / sqrt(var + eps), computed
    first; W' = W * scale per output channel (axis 0 of W); then
    b' = (b - mean) * scale + beta from the OLD bias (HowTo §2.1 warns against
    deriving the bias from the already-updated weight).  A missing bias is a
    zero bias (OpenPPL §3.1).  eps is taken from the model, never dropped
    (HowTo §2.1, §4.1).

    dtype float32 evaluates every operation as one IEEE binary32 operation,
    round to nearest, in this order ("fold in FP32", OpenPPL §6.2); numpy
    never contracts a*b+c into a fused multiply-add."""
    w = np.asarray(w, dtype)
    out_ch = w.shape[0]
    b = np.zeros(out_ch, dtype) if b is None else np.asarray(b, dtype)
    gamma = np.asarray(gamma, dtype)
    beta = np.asarray(beta, dtype)
    mean = np.asarray(mean, dtype)
    var = np.asarray(var, dtype)
    eps = dtype(eps)
    scale = gamma / np.sqrt(var + eps)
    w_new = w * scale.reshape((-1,) + (1,) * (w.ndim - 1))
    b_new = (b - mean) * scale + beta
    return w_new, b_new


# -------------------------------------------------- direct convolution


def conv2d_direct(inp, weight, bias, stride=1, pad=0):
    """Direct NCHW convolution, one output element at a time: for each output
    (n, co, ho, wo), sum over (ci, kh, kw) of in[n, ci, ho*stride-pad+kh,
    wo*stride-pad+kw] * W[co, ci, kh, kw], skipping taps outside the input,
    plus bias[co].  The loop order of the naive fused conv kernel in HowTo
    §3.3, without its ReLU.  Pure-Python loops: tiny shapes only."""
    inp = np.asarray(inp, np.float64)
    weight = np.asarray(weight, np.float64)
    n_img, c_in, h, w = inp.shape
    c_out, _, kh_n, kw_n = weight.shape
    h_out = (h + 2 * pad - kh_n) // stride + 1
    w_out = (w + 2 * pad - kw_n) // stride + 1
    out = np.zeros((n_img, c_out, h_out, w_out))
    for n in range(n_img):
        for co in range(c_out):
            for ho in range(h_out):
                for wo in range(w_out):
                    acc = 0.0 if bias is None else float(bias[co])
                    for ci in range(c_in):
                        for kh in range(kh_n):
                            for kw in range(kw_n):
                                hi = ho * stride - pad + kh
                                wi = wo * stride - pad + kw
                                if 0 <= hi < h and 0 <= wi < w:
                                    acc += inp[n, ci, hi, wi] * weight[co, ci, kh, kw]
                    out[n, co, ho, wo] = acc
    return out
