"""Seeded synthetic inputs for the fused operators.

This module only draws random numbers and stores them: it holds none of the
operators' arithmetic.  It is the one module that both the CUDA path's tests
and bench and the CPU oracle use, so that both see the same input bytes.

Draws use numpy's PCG64 generator seeded per workload; float32 samples are
rounded to bfloat16 by torch's conversion (round to nearest even) and handed
out as raw uint16 bit patterns (numpy) so that either side can decode them.

Shapes and distributions are those of the workloads the pages describe
(FlashRT §2-§3: Pi0.5 decoder, Qwen3 and Wan QKV post-processing; OpenPPL
§3.1/§4.3: Linear + bias + GELU, Conv/Linear + BN); they stand in for the
models' activations, which are not available.
"""
import numpy as np
import torch


def _bf16_bits(a):
    """float32 numpy array -> uint16 numpy array of bfloat16 bits (RNE)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


class Draw:
    """Sequential draws from one seeded stream, in the order requested."""

    def __init__(self, seed=0):
        self.rng = np.random.Generator(np.random.PCG64(seed))

    def normal(self, shape, mean=0.0, std=1.0):
        a = self.rng.standard_normal(size=shape, dtype=np.float32)
        if std != 1.0:
            a *= np.float32(std)
        if mean != 0.0:
            a += np.float32(mean)
        return a

    def uniform(self, shape, lo, hi):
        return (self.rng.random(size=shape, dtype=np.float32) * np.float32(hi - lo) + np.float32(lo))

    def bf16_normal(self, shape, mean=0.0, std=1.0):
        return _bf16_bits(self.normal(shape, mean, std))


# ---------------------------------------------------------------- workloads

def add_rmsnorm_case(rows, hidden, mode, seed=0, gated=False):
    """x, res ~ N(0,1) [rows, hidden]; then, by mode: weight = 1 + N(0, 0.1)
    (weighted), or gate/shift/scale ~ N(0, 0.2) [hidden] (ada).  A gate is
    drawn first when `gated`.  Modes: 0 weighted, 1 noweight, 2 ada."""
    d = Draw(seed)
    c = {"x": d.bf16_normal((rows, hidden)), "res": d.bf16_normal((rows, hidden)),
         "rows": rows, "hidden": hidden, "mode": mode, "eps": 1e-6, "s_q": 0.05,
         "weight": None, "gate": None, "scale": None, "shift": None}
    if gated or mode == 2:
        c["gate"] = d.bf16_normal((hidden,), std=0.2)
    if mode == 0:
        c["weight"] = d.bf16_normal((hidden,), mean=1.0, std=0.1)
    elif mode == 2:
        c["shift"] = d.bf16_normal((hidden,), std=0.2)
        c["scale"] = d.bf16_normal((hidden,), std=0.2)
    return c


EDGE_KINDS = ("saturate", "subnormal", "zero_rows", "outlier")


def add_rmsnorm_edge_case(rows, hidden, mode, kind, seed=0, gated=False):
    """add_rmsnorm_case with inputs that reach the ends of the E4M3 range.

    kind "saturate":  the descale is 0.002 instead of 0.05, so every |y| above
                      0.896 lies past the largest finite code (448 * 0.002);
    kind "subnormal": the descale is 200, so |y / s| of a unit-RMS row mostly
                      falls below 2**-6, among the E4M3 subnormals and zeros;
    kind "zero_rows": every third row of x and res is all zeros, and in row 1
                      (when there is one) x is res with every sign bit flipped,
                      so the residual sum is exactly zero there too;
    kind "outlier":   one column of every row of x holds a value of magnitude
                      10**U(3, 6) with a random sign; the norm's scale is then
                      set by that one value and the other columns land near
                      the bottom of the E4M3 range, while the outlier saturates.
    The other draws are those of add_rmsnorm_case with the same seed; the
    extra draws (outlier columns, magnitudes, signs) come after them."""
    if kind not in EDGE_KINDS:
        raise ValueError(kind)
    c = add_rmsnorm_case(rows, hidden, mode, seed=seed, gated=gated)
    c["kind"] = kind
    if kind == "saturate":
        c["s_q"] = 0.002
    elif kind == "subnormal":
        c["s_q"] = 200.0
    elif kind == "zero_rows":
        c["x"][::3] = 0
        c["res"][::3] = 0
        if rows > 1:
            c["x"][1] = c["res"][1] ^ np.uint16(0x8000)
    else:
        d = Draw(seed + 7919)
        col = d.rng.integers(0, hidden, size=rows)
        mag = np.power(np.float32(10.0), d.uniform((rows,), 3.0, 6.0))
        sign = np.where(d.rng.random(rows) < 0.5, np.float32(-1.0), np.float32(1.0))
        c["x"][np.arange(rows), col] = _bf16_bits(mag * sign)
    return c


def config_tiny_add_rmsnorm(seed=0):
    """Residual + RMSNorm + FP8: x, res bf16 [16, 256] ~ N(0,1), weight
    1 + N(0, 0.1) [256], eps 1e-6, static scale 0.05."""
    return add_rmsnorm_case(16, 256, 0, seed)


def pi05_decoder_chain(seed=0, layers=18, steps=10, tokens=10, hidden=1024):
    """Pi0.5-decoder-shaped gated residual + AdaRMSNorm + FP8 chain: 18 layers
    x 10 flow-matching steps = 180 calls on [10, 1024].  Draw order: the
    initial residual, then 18 per-layer x tensors, then for each call
    (step-major over layers: call = step * layers + layer) gate, shift, scale
    ~ N(0, 0.2) [1024].  The residual chains from call to call."""
    d = Draw(seed)
    res0 = d.bf16_normal((tokens, hidden))
    xs = [d.bf16_normal((tokens, hidden)) for _ in range(layers)]
    mods = []
    for _ in range(layers * steps):
        gate = d.bf16_normal((hidden,), std=0.2)
        shift = d.bf16_normal((hidden,), std=0.2)
        scale = d.bf16_normal((hidden,), std=0.2)
        mods.append((gate, shift, scale))
    return {"res0": res0, "xs": xs, "mods": mods, "layers": layers, "steps": steps,
            "tokens": tokens, "hidden": hidden, "eps": 1e-6, "s_q": 0.05}


def qkv_case(tokens, n_q_heads, n_kv_heads, head_dim, norm, rope, seed=0,
             theta=1e6, grid=None, sections=None, slots=None, cache_rows=None):
    """Packed QKV bf16 [tokens, (Hq + 2 Hkv) * D] ~ N(0,1); then q_w and k_w =
    1 + N(0, 0.1), [D] per head or [H * D] full width.  1D positions are
    0..tokens-1; 3D positions are the (t, h, w) coordinates of token
    n = (t * GH + h) * GW + w on the grid (GT, GH, GW)."""
    d = Draw(seed)
    width = (n_q_heads + 2 * n_kv_heads) * head_dim
    qkv = d.bf16_normal((tokens, width))
    wlen_q = head_dim if norm == 0 else n_q_heads * head_dim
    wlen_k = head_dim if norm == 0 else n_kv_heads * head_dim
    q_w = d.bf16_normal((wlen_q,), mean=1.0, std=0.1)
    k_w = d.bf16_normal((wlen_k,), mean=1.0, std=0.1)
    if rope == 0:
        pos = np.arange(tokens, dtype=np.int32)
    else:
        gt, gh, gw = grid
        n = np.arange(tokens, dtype=np.int64)
        pos = np.stack([n // (gh * gw), (n // gw) % gh, n % gw], axis=1).astype(np.int32)
    return {"qkv": qkv, "tokens": tokens, "n_q": n_q_heads, "n_kv": n_kv_heads, "d": head_dim,
            "norm": norm, "rope": rope, "q_w": q_w, "k_w": k_w, "eps": 1e-6, "theta": theta,
            "pos": pos, "sections": sections, "slots": slots, "cache_rows": cache_rows}


def config_qwen3_qkv(seed=0, tokens=4096):
    """Qwen3-style QKV post-processing: packed [4096, (32+8+8)*128], per-head
    RMSNorm on Q and K, rotate_half RoPE theta 1e6 at positions 0..4095."""
    return qkv_case(tokens, 32, 8, 128, 0, 0, seed, theta=1e6)


def qkv_decode_paged_case(tokens=32, n_q_heads=32, n_kv_heads=8, head_dim=128, cache_rows=16384, block=16,
                          max_pos=4096, seed=0):
    """Decode-shaped QKV post-processing into a paged KV cache: one new token
    per sequence, `tokens` sequences with Qwen3's heads; packed QKV and
    weights as qkv_case (per-head RMSNorm, 1D RoPE theta 1e6); each
    sequence's position drawn uniformly in [0, max_pos); the cache is
    cache_rows // block blocks of `block` rows, each sequence owning a
    distinct block drawn without replacement, and its token's slot is that
    block's row (position mod block), the slot mapping of a paged cache."""
    c = qkv_case(tokens, n_q_heads, n_kv_heads, head_dim, 0, 0, seed, theta=1e6)
    rng = np.random.Generator(np.random.PCG64(seed + 2000))
    pos = rng.integers(0, max_pos, size=tokens).astype(np.int32)
    blocks = rng.choice(cache_rows // block, size=tokens, replace=False).astype(np.int64)
    c["pos"] = pos
    c["slots"] = (blocks * block + pos % block).astype(np.int32)
    c["cache_rows"] = cache_rows
    return c


def layernorm_qkv_case(tokens, n_q_heads, n_kv_heads, head_dim, seed=0, theta=1e4, biases=True):
    """Packed QKV bf16 [tokens, (Hq + 2 Hkv) * D] ~ N(0,1); then q_w, k_w =
    1 + N(0, 0.1) and (when `biases`) q_b, k_b ~ N(0, 0.1), all [D]; eps 1e-5;
    positions 0..tokens-1."""
    c = qkv_case(tokens, n_q_heads, n_kv_heads, head_dim, 0, 0, seed, theta=theta)
    d = Draw(seed + 1000)
    c["norm"] = 2
    c["eps"] = 1e-5
    c["q_b"] = d.bf16_normal((head_dim,), std=0.1) if biases else None
    c["k_b"] = d.bf16_normal((head_dim,), std=0.1) if biases else None
    return c


def config_chameleon_qkv(seed=0, tokens=4096):
    """Chameleon-style prefill QKV post-processing (7B shapes): packed
    [4096, (32+32+32)*128], per-head LayerNorm on Q and K with weight and
    bias, rotate_half RoPE theta 1e4 at positions 0..4095."""
    return layernorm_qkv_case(tokens, 32, 32, 128, seed, theta=1e4)


WAN_GRID = (21, 30, 52)


def config_wan_qkv(seed=0, tokens=None):
    """Wan-style video QKV: packed [32760, 3*5120] on the 21x30x52 grid, 40
    heads x 128, full-width 5120 RMSNorm on Q and K, 3D RoPE with sections
    44/42/42 over (t, h, w), theta 1e4.  `tokens` takes a prefix of the grid."""
    t = WAN_GRID[0] * WAN_GRID[1] * WAN_GRID[2] if tokens is None else tokens
    return qkv_case(t, 40, 40, 128, 1, 1, seed, theta=1e4, grid=WAN_GRID, sections=(44, 42, 42))


def gated_act_case(rows, d, seed=0, std=2.0):
    """Gated-activation input bf16 [rows, 2d] = [gate | up], both ~ N(0, std):
    gate values reach the saturated ends of SiLU and GELU."""
    return {"x": Draw(seed).bf16_normal((rows, 2 * d), std=std), "rows": rows, "d": d}


def config_swiglu_ffn(seed=0, rows=4096):
    """SwiGLU on a LLaMA-7B-shaped FFN (intermediate width 11008): [gate | up]
    bf16 [4096, 2*11008] -> silu(gate) * up bf16 [4096, 11008]."""
    return gated_act_case(rows, 11008, seed)


def linear_gelu_case(m, n, k, seed=0, with_bias=True):
    """X ~ N(0,1) [M, K], W ~ N(0, 0.02) [N, K], bias ~ N(0, 0.1) [N]; then the
    BatchNorm of the Linear's output channels: gamma ~ U(0.5, 1.5),
    beta ~ N(0, 0.1), mean ~ N(0, 0.1), var ~ U(0.01, 1), float32 [N]; eps 1e-2."""
    d = Draw(seed)
    c = {"x": d.bf16_normal((m, k)), "w": d.bf16_normal((n, k), std=0.02),
         "bias": d.bf16_normal((n,), std=0.1) if with_bias else None, "m": m, "n": n, "k": k}
    c["gamma"] = d.uniform((n,), 0.5, 1.5)
    c["beta"] = d.normal((n,), std=0.1)
    c["mean"] = d.normal((n,), std=0.1)
    c["var"] = d.uniform((n,), 0.01, 1.0)
    c["eps"] = 1e-2
    return c


def config_linear_gelu(seed=0):
    """Linear + bias + GELU(tanh): X [8192, 4096], W [16384, 4096], bias [16384],
    plus the BN-fold parameters of W's 16384 output channels."""
    return linear_gelu_case(8192, 16384, 4096, seed)


def as_torch(bits, device="cuda"):
    """numpy storage bits (uint16 bf16 / uint8 / int32 / float32) -> torch tensor on `device`."""
    a = np.ascontiguousarray(bits)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def fp8_linear_case(m, n, k, seed=0):
    """Quantised Linear operands as real values before quantisation: X ~ N(0, 1)
    [M, K] (the activations fused_add_rmsnorm_fp8 quantises, descale 0.05),
    W ~ N(0, 0.02) [N, K], bias ~ N(0, 0.1) [N] (bf16 bits), and one weight
    descale per row ~ U(0.9, 1.1) * 0.1 / 448 (about five standard deviations
    of W at the top code).  The caller encodes the E4M3 codes (the oracle in
    tests, a library conversion on the GPU in the bench)."""
    d = Draw(seed)
    return {"x": d.normal((m, k)), "w": d.normal((n, k), std=0.02), "bias": d.bf16_normal((n,), std=0.1),
            "x_scale": 0.05, "w_scale": (d.uniform((n,), 0.9, 1.1) * (0.1 / 448.0)).astype(np.float32),
            "m": m, "n": n, "k": k}


def norm_fold_case(out_ch, inner, seed=0):
    """W bf16 [out_ch, inner] ~ N(0, 0.02); a norm weight gamma bf16 [inner] ~
    N(0, 0.1) (Gemma-style: the scale is 1 + gamma)."""
    d = Draw(seed)
    return {"w": d.bf16_normal((out_ch, inner), std=0.02), "gamma": d.bf16_normal((inner,), std=0.1),
            "out_ch": out_ch, "inner": inner}


def cross_layer_case(rows, hidden, n_out, seed=0):
    """The loop between two layers: x, res ~ N(0,1) [rows, hidden] into the
    _noweight norm, a Gemma-style norm weight gamma ~ N(0, 0.1) [hidden] (the
    scale is 1 + gamma), the next Linear's W ~ N(0, 0.02) [n_out, hidden] and
    bias ~ N(0, 0.1) [n_out] (bf16 bits), one weight descale per output row ~
    U(0.9, 1.1) * 0.1 / 448 (float32), activation descale 0.05, eps 1e-6."""
    d = Draw(seed)
    return {"x": d.bf16_normal((rows, hidden)), "res": d.bf16_normal((rows, hidden)),
            "gamma": d.bf16_normal((hidden,), std=0.1), "w": d.bf16_normal((n_out, hidden), std=0.02),
            "bias": d.bf16_normal((n_out,), std=0.1),
            "w_scale": (d.uniform((n_out,), 0.9, 1.1) * (0.1 / 448.0)).astype(np.float32),
            "x_scale": 0.05, "eps": 1e-6, "rows": rows, "hidden": hidden, "n_out": n_out}
