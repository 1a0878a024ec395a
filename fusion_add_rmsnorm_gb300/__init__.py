"""Python binding of libgbfuse.so: fused operator chains for GB300 (sm_103a).

Argument marshalling only.  Every function takes torch tensors that live on
the current CUDA device, derives the extents from them, passes their data
pointers and sizes to the C-ABI entry point of the same name (see
include/gbfuse.h) on the current torch stream, and raises GbfError on a
non-zero status.  A raw pointer carries no size, so before the call each
wrapper checks what the C library cannot: every operand holds exactly the
elements the call will read or write (ValueError otherwise), is a contiguous
torch tensor of the element type the call reads, on the current device.
There is no CPU path: importing this package fails when the compiled library
is missing, and every call fails without a CUDA device.

Build the library with `python -c "import __graft_entry__ as g; g.build()"`
(or `python fusion_add_rmsnorm_gb300/build.py`).
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgbfuse.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run fusion_add_rmsnorm_gb300/build.py "
                      "(this package has no CPU fallback)")

_lib = ctypes.CDLL(LIB_PATH)

OK, EINVAL, EALIGN, EUNSUPPORTED, ELAUNCH, ETIMEOUT, EDEVICE = 0, -1, -2, -3, -4, -5, -6
NORM_WEIGHT, NORM_NOWEIGHT, NORM_ADA = 0, 1, 2
QKNORM_PER_HEAD, QKNORM_FULL_WIDTH = 0, 1
ROPE_1D, ROPE_3D = 0, 1
ACT_NONE, ACT_GELU_TANH, ACT_GELU_ERF, ACT_SILU = 0, 1, 2, 3

_p, _i64, _i32, _f = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float

_SIGNATURES = {
    "gbf_add_rmsnorm_fp8": [_p, _p, _p, _p, _i32, _p, _p, _p, _p, _i64, _i64, _f, _f, _p],
    "gbf_qkv_split_norm_rope": [_p, _i64, _i32, _i32, _i32, _i32, _p, _p, _f, _i32, _p, _p, _f, _p, _p, _p,
                                _p, _i64, _p],
    "gbf_qkv_split_layernorm_rope": [_p, _i64, _i32, _i32, _i32, _p, _p, _p, _p, _f, _p, _f, _p, _p, _p, _p, _i64,
                                     _p],
    "gbf_linear_bias_gelu": [_p, _p, _p, _p, _i64, _i64, _i64, _i32, _p],
    "gbf_gated_act": [_p, _p, _i64, _i64, _i32, _p],
    "gbf_linear_fp8_act": [_p, _f, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _p],
    "gbf_fold_norm_weight": [_p, _p, _i32, _i64, _i64, _p, _p],
    "gbf_bn_fold": [_p, _p, _p, _p, _p, _p, _f, _i64, _i64, _p, _p, _p],
    "gbf_copy": [_p, _p, _i64, _p],
    "gbf_device_status": [_p],
    "gbf_selftest_bounded_wait": [_p],
    "gbf_last_error": [],
    "gbf_version": [],
}
for _name, _args in _SIGNATURES.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = ctypes.c_char_p if _name == "gbf_last_error" else ctypes.c_int

EXPORTED = tuple(_SIGNATURES)


class GbfError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"status {status}: {message}")
        self.status = status


def _check(status):
    if status != OK:
        raise GbfError(status, _lib.gbf_last_error().decode())
    return status


_BF16, _U8, _I32, _F32 = torch.bfloat16, torch.uint8, torch.int32, torch.float32


def _numel(t, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    return t.numel()


def _extent(t, n, name, at_least=False):
    """An operand (None: an absent optional one) must hold n elements (at
    least n with at_least)."""
    if t is None:
        return
    k = _numel(t, name)
    if k < n if at_least else k != n:
        raise ValueError(f"{name}: holds {k} elements, the call needs {'at least ' if at_least else ''}{n}")


def _ptr(t, dtype=None, name="tensor"):
    """Device pointer of a tensor argument after the checks the C ABI cannot
    make from a raw pointer: a torch tensor on the current CUDA device, dense,
    of the element type the call reads (dtype None: any).  None passes through
    (an optional argument)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be on a CUDA device")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name}: is on cuda:{t.device.index}, the current device is cuda:{torch.cuda.current_device()}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def version():
    return _lib.gbf_version()


def raw():
    """The ctypes handle of libgbfuse.so, for callers that pass raw pointers."""
    return _lib


def add_rmsnorm_fp8(x, res_in, res_out, q_out, mode, weight=None, gate=None, ada_scale=None, ada_shift=None,
                    eps=1e-6, fp8_scale=0.05, stream=None):
    """gbf_add_rmsnorm_fp8 on [..., hidden] bf16 tensors (rows = every leading
    index); q_out is uint8 E4M3 codes of the same shape."""
    _numel(x, "x")
    hidden = x.shape[-1] if x.dim() else 0
    rows = x.numel() // hidden if hidden else 0
    for t, name in ((res_in, "res_in"), (res_out, "res_out"), (q_out, "q_out")):
        _extent(t, x.numel(), name)
    for t, name in ((weight, "weight"), (gate, "gate"), (ada_scale, "ada_scale"), (ada_shift, "ada_shift")):
        _extent(t, hidden, name)
    return _check(_lib.gbf_add_rmsnorm_fp8(_ptr(x, _BF16, "x"), _ptr(res_in, _BF16, "res_in"),
                                           _ptr(res_out, _BF16, "res_out"), _ptr(gate, _BF16, "gate"), mode,
                                           _ptr(weight, _BF16, "weight"), _ptr(ada_scale, _BF16, "ada_scale"),
                                           _ptr(ada_shift, _BF16, "ada_shift"), _ptr(q_out, _U8, "q_out"), rows,
                                           hidden, eps, fp8_scale, _stream(stream)))


def _qkv_extents(qkv, n_q_heads, n_kv_heads, head_dim, pos, pos_per_token, q_out, k_cache, v_cache, slots,
                 cache_rows):
    """Tokens and cache rows of a QKV call, after checking every operand's extent."""
    _numel(qkv, "qkv")
    width = (n_q_heads + 2 * n_kv_heads) * head_dim
    if qkv.dim() != 2 or qkv.shape[1] != width:
        raise ValueError(f"qkv: expected [tokens, {width}], got {list(qkv.shape)}")
    tokens = qkv.shape[0]
    _numel(k_cache, "k_cache")
    rows = k_cache.numel() // max(n_kv_heads * head_dim, 1) if cache_rows is None else cache_rows
    _extent(pos, tokens * pos_per_token, "pos")
    _extent(slots, tokens, "slots")
    _extent(q_out, tokens * n_q_heads * head_dim, "q_out")
    _extent(k_cache, rows * n_kv_heads * head_dim, "k_cache", at_least=True)
    _extent(v_cache, rows * n_kv_heads * head_dim, "v_cache", at_least=True)
    return tokens, rows


def qkv_split_norm_rope(qkv, n_q_heads, n_kv_heads, head_dim, norm, q_w, k_w, eps, rope, pos, theta, q_out,
                        k_cache, v_cache, sections=None, slots=None, cache_rows=None, stream=None):
    """gbf_qkv_split_norm_rope; `sections` is a host sequence of three ints."""
    tokens, rows = _qkv_extents(qkv, n_q_heads, n_kv_heads, head_dim, pos, 3 if rope == ROPE_3D else 1, q_out,
                                k_cache, v_cache, slots, cache_rows)
    wq, wk = (head_dim, head_dim) if norm == QKNORM_PER_HEAD else (n_q_heads * head_dim, n_kv_heads * head_dim)
    _extent(q_w, wq, "q_w")
    _extent(k_w, wk, "k_w")
    if sections is not None and len(sections) != 3:
        raise ValueError(f"sections: expected three ints, got {len(sections)}")
    sec = None if sections is None else (ctypes.c_int32 * 3)(*sections)
    return _check(_lib.gbf_qkv_split_norm_rope(_ptr(qkv, _BF16, "qkv"), tokens, n_q_heads, n_kv_heads, head_dim,
                                               norm, _ptr(q_w, _BF16, "q_w"), _ptr(k_w, _BF16, "k_w"), eps, rope,
                                               _ptr(pos, _I32, "pos"),
                                               ctypes.cast(sec, ctypes.c_void_p) if sec is not None else None,
                                               theta, _ptr(q_out, _BF16, "q_out"), _ptr(k_cache, _BF16, "k_cache"),
                                               _ptr(v_cache, _BF16, "v_cache"), _ptr(slots, _I32, "slots"),
                                               rows, _stream(stream)))


def qkv_split_layernorm_rope(qkv, n_q_heads, n_kv_heads, head_dim, q_w, q_b, k_w, k_b, eps, pos, theta, q_out,
                             k_cache, v_cache, slots=None, cache_rows=None, stream=None):
    """gbf_qkv_split_layernorm_rope: per-head LayerNorm (biases may be None) + 1D RoPE."""
    tokens, rows = _qkv_extents(qkv, n_q_heads, n_kv_heads, head_dim, pos, 1, q_out, k_cache, v_cache, slots,
                                cache_rows)
    for t, name in ((q_w, "q_w"), (q_b, "q_b"), (k_w, "k_w"), (k_b, "k_b")):
        _extent(t, head_dim, name)
    return _check(_lib.gbf_qkv_split_layernorm_rope(_ptr(qkv, _BF16, "qkv"), tokens, n_q_heads, n_kv_heads,
                                                    head_dim, _ptr(q_w, _BF16, "q_w"), _ptr(q_b, _BF16, "q_b"),
                                                    _ptr(k_w, _BF16, "k_w"), _ptr(k_b, _BF16, "k_b"), eps,
                                                    _ptr(pos, _I32, "pos"), theta, _ptr(q_out, _BF16, "q_out"),
                                                    _ptr(k_cache, _BF16, "k_cache"), _ptr(v_cache, _BF16, "v_cache"),
                                                    _ptr(slots, _I32, "slots"), rows, _stream(stream)))


def _linear_extents(x, w, bias, y, xname, wname):
    """(M, N, K) of a Linear call after checking x [..., K], w [N, K], bias [N], y [M, N]."""
    _numel(x, xname)
    _numel(w, wname)
    k = x.shape[-1] if x.dim() else 0
    m = x.numel() // k if k else 0
    if w.dim() != 2 or w.shape[1] != k:
        raise ValueError(f"{wname}: expected [N, {k}], got {list(w.shape)}")
    n = w.shape[0]
    _extent(bias, n, "bias")
    _extent(y, m * n, "y")
    return m, n, k


def linear_bias_gelu(x, w, bias, y, act=ACT_GELU_TANH, stream=None):
    """gbf_linear_bias_gelu: y[..., N] = act(x[..., K] @ w[N, K]^T + bias[N])."""
    m, n, k = _linear_extents(x, w, bias, y, "x", "w")
    return _check(_lib.gbf_linear_bias_gelu(_ptr(x, _BF16, "x"), _ptr(w, _BF16, "w"), _ptr(bias, _BF16, "bias"),
                                            _ptr(y, _BF16, "y"), m, n, k, act, _stream(stream)))


def linear_fp8_act(xq, x_scale, wq, w_scale, bias, y, act=ACT_GELU_TANH, stream=None):
    """gbf_linear_fp8_act: y[M, N] = act((xq * x_scale) @ (wq * w_scale[:, None])^T + bias); xq, wq uint8 codes."""
    m, n, k = _linear_extents(xq, wq, bias, y, "xq", "wq")
    _extent(w_scale, n, "w_scale")
    return _check(_lib.gbf_linear_fp8_act(_ptr(xq, _U8, "xq"), x_scale, _ptr(wq, _U8, "wq"),
                                          _ptr(w_scale, _F32, "w_scale"), _ptr(bias, _BF16, "bias"),
                                          _ptr(y, _BF16, "y"), m, n, k, act, _stream(stream)))


def fold_norm_weight(w, gamma, w_out, gemma_style=True, stream=None):
    """gbf_fold_norm_weight: w_out = w * (1 + gamma) (or w * gamma), per column."""
    _numel(w, "w")
    out_ch = w.shape[0] if w.dim() else 0
    inner = w.numel() // max(out_ch, 1)
    _extent(gamma, inner, "gamma")
    _extent(w_out, w.numel(), "w_out")
    return _check(_lib.gbf_fold_norm_weight(_ptr(w, _BF16, "w"), _ptr(gamma, _BF16, "gamma"),
                                            1 if gemma_style else 0, out_ch, inner, _ptr(w_out, _BF16, "w_out"),
                                            _stream(stream)))


def gated_act(x, y, act=ACT_SILU, stream=None):
    """gbf_gated_act: y[rows, d] = act(x[:, :d]) * x[:, d:] for x [rows, 2d]."""
    _numel(y, "y")
    d = y.shape[-1] if y.dim() else 0
    rows = y.numel() // d if d else 0
    _extent(x, 2 * rows * d, "x")
    if _numel(x, "x") and x.shape[-1] != 2 * d:
        raise ValueError(f"x: rows of {x.shape[-1]} values, expected 2 * {d}")
    return _check(_lib.gbf_gated_act(_ptr(x, _BF16, "x"), _ptr(y, _BF16, "y"), rows, d, act, _stream(stream)))


def bn_fold(w, b, gamma, beta, mean, var, eps, w_out, b_out, stream=None):
    """gbf_bn_fold on a weight [out_ch, ...] (flattened per output channel)."""
    _numel(w, "w")
    out_ch = w.shape[0] if w.dim() else 0
    inner = w.numel() // max(out_ch, 1)
    for t, name in ((b, "b"), (gamma, "gamma"), (beta, "beta"), (mean, "mean"), (var, "var"), (b_out, "b_out")):
        _extent(t, out_ch, name)
    _extent(w_out, w.numel(), "w_out")
    return _check(_lib.gbf_bn_fold(_ptr(w, _BF16, "w"), _ptr(b, _BF16, "b"), _ptr(gamma, _F32, "gamma"),
                                   _ptr(beta, _F32, "beta"), _ptr(mean, _F32, "mean"), _ptr(var, _F32, "var"), eps,
                                   out_ch, inner, _ptr(w_out, _BF16, "w_out"), _ptr(b_out, _BF16, "b_out"),
                                   _stream(stream)))


def copy(src, dst, nbytes=None, stream=None):
    """gbf_copy of nbytes (default: all of src) bytes."""
    src_bytes = _numel(src, "src") * src.element_size()
    dst_bytes = _numel(dst, "dst") * dst.element_size()
    n = src_bytes if nbytes is None else nbytes
    if n > src_bytes or n > dst_bytes:
        raise ValueError(f"copy of {n} bytes: src holds {src_bytes}, dst {dst_bytes}")
    return _check(_lib.gbf_copy(_ptr(src, None, "src"), _ptr(dst, None, "dst"), n, _stream(stream)))


def selftest_bounded_wait(stream=None):
    """gbf_selftest_bounded_wait: enqueue the bounded-wait self-test kernel."""
    return _check(_lib.gbf_selftest_bounded_wait(_stream(stream)))


def device_status(stream=None):
    """Synchronise the stream and return (status, message) of the device error word, clearing it."""
    s = _lib.gbf_device_status(_stream(stream))
    return s, (_lib.gbf_last_error().decode() if s else "")
