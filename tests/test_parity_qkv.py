"""GPU parity of gbf_qkv_split_norm_rope against the oracle's unfused chain
(split -> Q/K RMSNorm -> RoPE -> Q and K/V-cache writes; V bit for bit)."""
import numpy as np
import pytest
import torch

import workloads
from oracle import chains
from parity import assert_bf16_close, from_bits, to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gbf():
    import fusion_add_rmsnorm_gb300 as g
    return g


def run_gpu(gbf, c, slots=None, cache_rows=None):
    t, hq, hkv, d = c["tokens"], c["n_q"], c["n_kv"], c["d"]
    rows = t if cache_rows is None else cache_rows
    q = torch.empty(t, hq, d, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(rows, hkv, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros(rows, hkv, d, dtype=torch.bfloat16, device="cuda")
    pos = torch.from_numpy(np.ascontiguousarray(c["pos"])).cuda()
    sl = None if slots is None else torch.from_numpy(np.asarray(slots, np.int32)).cuda()
    gbf.qkv_split_norm_rope(from_bits(c["qkv"]), hq, hkv, d, c["norm"], from_bits(c["q_w"]), from_bits(c["k_w"]),
                            c["eps"], c["rope"], pos, c["theta"], q, kc, vc, sections=c["sections"], slots=sl,
                            cache_rows=rows)
    torch.cuda.synchronize()
    return to_bits(q), to_bits(kc), to_bits(vc)


def run_oracle(c, tok=None, slots=None, cache_rows=None):
    sel = slice(None) if tok is None else tok
    return chains.qkv_split_norm_rope(c["qkv"][sel], c["n_q"], c["n_kv"], c["d"], c["norm"], c["q_w"], c["k_w"],
                                      c["eps"], c["rope"], c["pos"][sel], c["theta"], sections=c["sections"],
                                      slots=slots, cache_rows=cache_rows)


def check(gbf, c, what, tok=None):
    q, kc, vc = run_gpu(gbf, c)
    rq, rk, rv = run_oracle(c, tok)
    if tok is not None:
        q, kc, vc = q[tok], kc[tok], vc[tok]
    assert_bf16_close(q, rq, what + " Q")
    assert_bf16_close(kc, rk, what + " K")
    assert np.array_equal(vc, rv), what + " V must be copied bit for bit"


def test_qwen3_config_full(gbf):
    """Packed [4096, 48*128], per-head norm, 1D RoPE theta 1e6 at positions 0..4095."""
    check(gbf, workloads.config_qwen3_qkv(), "qwen3")


def test_wan_config_sampled_tokens(gbf):
    """Packed [32760, 3*5120] on the 21x30x52 grid, full-width norm, 3D RoPE
    44/42/42, theta 1e4, in the bench's launch configuration; the oracle checks
    a sample of 192 tokens (first, last, and random)."""
    c = workloads.config_wan_qkv()
    rng = np.random.default_rng(1)
    tok = np.unique(np.concatenate([[0, 1, 51, 1559, c["tokens"] - 1],
                                    rng.choice(c["tokens"], 187, replace=False)]))
    check(gbf, c, "wan", tok)


@pytest.mark.parametrize("norm", [0, 1])
@pytest.mark.parametrize("rope", [0, 1])
@pytest.mark.parametrize("tokens,hq,hkv,d", [(1, 1, 1, 64), (13, 4, 2, 128), (9, 3, 3, 256), (17, 8, 1, 128),
                                             (5, 2, 2, 16)])
def test_all_combinations(gbf, norm, rope, tokens, hq, hkv, d):
    sections = None
    grid = None
    if rope == 1:
        h = d // 2 // 3 * 2
        sections = (d - 2 * h, h, h)
        grid = (3, 4, 5)
    c = workloads.qkv_case(tokens, hq, hkv, d, norm, rope, seed=tokens + d + 10 * norm + 100 * rope,
                           theta=1e4, grid=grid, sections=sections)
    check(gbf, c, f"norm {norm} rope {rope} [{tokens},{hq},{hkv},{d}]")


@pytest.mark.parametrize("norm", [0, 1])
@pytest.mark.parametrize("rope", [0, 1])
def test_many_heads_two_pass_path(gbf, norm, rope):
    """80 Q/K heads of width 256 (48 KB rows): several heads per thread in every
    kernel, and the smallest ring the streamed kernels pick for such rows."""
    sections = (86, 86, 84) if rope else None
    c = workloads.qkv_case(7, 64, 16, 256, norm, rope, seed=31 + norm + 2 * rope, theta=1e4,
                           grid=(2, 2, 2) if rope else None, sections=sections)
    check(gbf, c, f"two-pass norm {norm} rope {rope}")


def test_per_head_1d_wide_rows(gbf):
    """Per-head 1D rows of 160 heads x 256 (80 KB): 20 heads per lane group and
    a batch of loads cut short at the end; an odd token count leaves a partial
    last CTA."""
    c = workloads.qkv_case(9, 96, 32, 256, 0, 0, seed=53, theta=1e6)
    check(gbf, c, "per-head 1D, wide rows")


@pytest.mark.parametrize("tokens", [1, 2, 3, 1000])
def test_per_head_1d_token_counts(gbf, tokens):
    """Token counts that fill one, part of one, and many CTAs of four tokens."""
    c = workloads.qkv_case(tokens, 8, 2, 128, 0, 0, seed=60 + tokens, theta=1e6)
    check(gbf, c, f"per-head 1D, {tokens} tokens")


@pytest.mark.parametrize("rope", [0, 1])
def test_full_width_head_dim_48(gbf, rope):
    """Full-width norm with head_dim 48 (24 rotation slots, not a power of two)."""
    c = workloads.qkv_case(9, 6, 2, 48, 1, rope, seed=41 + rope, theta=1e4, grid=(2, 3, 2) if rope else None,
                           sections=(16, 16, 16) if rope else None)
    check(gbf, c, f"head_dim 48 rope {rope}")


@pytest.mark.parametrize("norm,rope", [(0, 1), (1, 1), (1, 0)])
def test_staged_ring_wraps(gbf, norm, rope):
    """2500 tokens of 8 + 2 x 8 heads x 128 (44/42/42 sections for 3D) on the
    staged kernel: each persistent CTA takes five or six tokens, more than its
    ring holds, so the row buffers are refilled and the ring wraps."""
    c = workloads.qkv_case(2500, 8, 8, 128, norm, rope, seed=70 + norm + 2 * rope, theta=1e4,
                           grid=(10, 10, 25) if rope else None, sections=(44, 42, 42) if rope else None)
    check(gbf, c, f"ring wraps norm {norm} rope {rope}")


@pytest.mark.parametrize("norm,rope", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_zero_tokens_and_outlier_heads(gbf, norm, rope):
    """Padding-like tokens whose Q and K are all zero (the norm of a zero head,
    or of a zero full-width row, is 0 * 1/sqrt(eps) = 0, so their Q and K come
    out zero while V passes through), and heads holding one value of magnitude
    1e4 or 3e4 that sets the head's (or the row's) scale; per-head and staged
    kernels."""
    c = workloads.qkv_case(24, 4, 2, 128, norm, rope, seed=80 + norm + 2 * rope, theta=1e4,
                           grid=(2, 3, 4) if rope else None, sections=(44, 42, 42) if rope else None)
    qkv = c["qkv"].copy()
    d, qk = 128, (4 + 2) * 128
    zero_tokens = [0, 5, 17]
    qkv[zero_tokens, :qk] = 0
    big = lambda v: np.uint16(np.array(v, np.float32).view(np.uint32) >> 16)      # noqa: E731
    qkv[3, 1 * d + 7] = big(1e4)
    qkv[9, 4 * d + 100] = big(-3e4)
    qkv[12, 5 * d + 64] = big(2e4)
    c["qkv"] = qkv
    check(gbf, c, f"zero tokens / outliers norm {norm} rope {rope}")
    q, kc, _ = run_gpu(gbf, c)
    assert np.all(np.isin(q[zero_tokens], (0x0000, 0x8000)))
    assert np.all(np.isin(kc[zero_tokens], (0x0000, 0x8000)))


def test_3d_per_head_with_zero_section(gbf):
    c = workloads.qkv_case(11, 4, 2, 128, 0, 1, seed=3, theta=1e4, grid=(2, 3, 4), sections=(64, 0, 64))
    check(gbf, c, "3D with an empty section")


@pytest.mark.parametrize("norm,rope", [(0, 0), (1, 1)])
def test_slots_scatter_into_a_larger_cache(gbf, norm, rope):
    """Arbitrary cache rows per token (a paged cache's slot mapping), on the
    per-head kernel and on the staged kernel, whose V leaves by bulk store."""
    c = workloads.qkv_case(12, 4, 2, 128, norm, rope, seed=9 + norm, theta=1e6 if rope == 0 else 1e4,
                           grid=(2, 2, 3) if rope else None, sections=(44, 42, 42) if rope else None)
    slots = np.random.default_rng(3).permutation(40)[:12].astype(np.int32)
    q, kc, vc = run_gpu(gbf, c, slots=slots, cache_rows=40)
    rq, rk, rv = run_oracle(c, slots=slots, cache_rows=40)
    assert_bf16_close(q, rq, "Q")
    assert_bf16_close(kc, rk, "K cache")
    assert np.array_equal(vc, rv)
    untouched = np.setdiff1d(np.arange(40), slots)
    assert not kc[untouched].any() and not vc[untouched].any()
    s, _ = gbf.device_status()
    assert s == gbf.OK


def test_decode_paged_cache(gbf):
    """The decode shape the bench times for the paged cache: 32 sequences'
    new tokens at scattered positions, each K/V row written to its block's
    slot of a 16,384-row cache; every other cache row stays untouched."""
    c = workloads.qkv_decode_paged_case()
    q, kc, vc = run_gpu(gbf, c, slots=c["slots"], cache_rows=c["cache_rows"])
    rq, rk, rv = run_oracle(c, slots=c["slots"], cache_rows=c["cache_rows"])
    assert_bf16_close(q, rq, "Q")
    assert_bf16_close(kc[c["slots"]], rk[c["slots"]], "K cache rows")
    assert np.array_equal(vc, rv)
    untouched = np.setdiff1d(np.arange(c["cache_rows"]), c["slots"])
    assert not kc[untouched].any() and not vc[untouched].any()
    s, _ = gbf.device_status()
    assert s == gbf.OK


@pytest.mark.parametrize("norm,rope", [(0, 0), (1, 1)])
def test_out_of_range_slot_is_skipped_and_reported(gbf, norm, rope):
    """A slot outside the cache writes nothing for that token and raises the
    device error word; every other token is still written."""
    grid = (2, 2, 2) if rope else None
    c = workloads.qkv_case(8, 2, 1, 128, norm, rope, seed=4, theta=1e4, grid=grid,
                           sections=(44, 42, 42) if rope else None)
    gbf.device_status()                        # clear
    slots = np.array([0, 1, 2, 99, 4, 5, 6, 7], np.int32)
    q, kc, vc = run_gpu(gbf, c, slots=slots, cache_rows=8)
    s, msg = gbf.device_status()
    assert s == gbf.EDEVICE and "slot" in msg
    good = slots != 99
    rq, rk, rv = run_oracle(c, tok=np.nonzero(good)[0], slots=slots[good], cache_rows=8)
    assert_bf16_close(q, run_oracle(c)[0], "Q is written for every token")
    assert_bf16_close(kc[slots[good]], rk[slots[good]], "K")
    assert not kc[3].any() and not vc[3].any()
    assert gbf.device_status()[0] == gbf.OK      # cleared by the read


# ------------------------------------------------ per-head LayerNorm (Chameleon)

def run_gpu_ln(gbf, c, slots=None, cache_rows=None):
    t, hq, hkv, d = c["tokens"], c["n_q"], c["n_kv"], c["d"]
    rows = t if cache_rows is None else cache_rows
    q = torch.empty(t, hq, d, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(rows, hkv, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros(rows, hkv, d, dtype=torch.bfloat16, device="cuda")
    pos = torch.from_numpy(np.ascontiguousarray(c["pos"])).cuda()
    sl = None if slots is None else torch.from_numpy(np.asarray(slots, np.int32)).cuda()
    opt = lambda k: None if c[k] is None else from_bits(c[k])      # noqa: E731
    gbf.qkv_split_layernorm_rope(from_bits(c["qkv"]), hq, hkv, d, from_bits(c["q_w"]), opt("q_b"),
                                 from_bits(c["k_w"]), opt("k_b"), c["eps"], pos, c["theta"], q, kc, vc, slots=sl,
                                 cache_rows=rows)
    torch.cuda.synchronize()
    return to_bits(q), to_bits(kc), to_bits(vc)


def run_oracle_ln(c, tok=None, slots=None, cache_rows=None):
    sel = slice(None) if tok is None else tok
    return chains.qkv_split_norm_rope(c["qkv"][sel], c["n_q"], c["n_kv"], c["d"], chains.QKNORM_LAYERNORM,
                                      c["q_w"], c["k_w"], c["eps"], 0, c["pos"][sel], c["theta"], slots=slots,
                                      cache_rows=cache_rows, q_b=c["q_b"], k_b=c["k_b"])


def check_ln(gbf, c, what):
    q, kc, vc = run_gpu_ln(gbf, c)
    rq, rk, rv = run_oracle_ln(c)
    assert_bf16_close(q, rq, what + " Q")
    assert_bf16_close(kc, rk, what + " K")
    assert np.array_equal(vc, rv), what + " V must be copied bit for bit"


def test_chameleon_config_full(gbf):
    """Packed [4096, 96*128], per-head LayerNorm with weight and bias on Q and
    K, 1D RoPE theta 1e4 at positions 0..4095."""
    check_ln(gbf, workloads.config_chameleon_qkv(), "chameleon")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("biases", [True, False])
@pytest.mark.parametrize("tokens,hq,hkv", [(1, 1, 1), (13, 4, 2), (9, 3, 3), (37, 8, 1)])
def test_layernorm_shapes(gbf, d, biases, tokens, hq, hkv):
    c = workloads.layernorm_qkv_case(tokens, hq, hkv, d, seed=tokens + d + 7 * hq, biases=biases)
    check_ln(gbf, c, f"LN d {d} biases {biases} [{tokens},{hq},{hkv}]")


@pytest.mark.parametrize("d", [64, 128])
def test_layernorm_many_heads(gbf, d):
    """More heads than one batch per thread holds (64 + 2 x 32 heads): every
    thread of the token takes several batches in turn."""
    c = workloads.layernorm_qkv_case(5, 64, 32, d, seed=91 + d, biases=True)
    check_ln(gbf, c, f"LN many heads d {d}")


def test_layernorm_of_constant_heads_is_the_bias(gbf):
    """Every Q and K head constant: the LayerNorm output is exactly the bias,
    and at position 0 the rotation leaves it alone."""
    c = workloads.layernorm_qkv_case(6, 4, 2, 128, seed=77)
    t, width = c["tokens"], (4 + 4) * 128
    vals = np.random.default_rng(0).normal(size=(t, 8, 1))
    bits = torch.from_numpy(np.broadcast_to(vals, (t, 8, 128)).reshape(t, width).copy()).to(torch.bfloat16)
    c["qkv"] = bits.view(torch.int16).numpy().view(np.uint16)
    c["pos"] = np.zeros(t, np.int32)
    q, kc, _ = run_gpu_ln(gbf, c)
    assert np.array_equal(q, np.broadcast_to(c["q_b"], q.shape))
    assert np.array_equal(kc, np.broadcast_to(c["k_b"], kc.shape))


def test_layernorm_slots_and_out_of_range_slot(gbf):
    c = workloads.layernorm_qkv_case(8, 2, 2, 128, seed=5)
    gbf.device_status()
    slots = np.array([3, 0, 7, 99, 4, 6, 1, 2], np.int32)
    q, kc, vc = run_gpu_ln(gbf, c, slots=slots, cache_rows=10)
    s, msg = gbf.device_status()
    assert s == gbf.EDEVICE and "slot" in msg
    good = slots != 99
    rq, rk, rv = run_oracle_ln(c, tok=np.nonzero(good)[0], slots=slots[good], cache_rows=10)
    assert_bf16_close(q, run_oracle_ln(c)[0], "Q is written for every token")
    assert_bf16_close(kc[slots[good]], rk[slots[good]], "K")
    assert np.array_equal(vc[slots[good]], rv[slots[good]])
    assert not kc[[5, 8, 9]].any() and not vc[[5, 8, 9]].any()
