"""Comparison rules of the GPU parity tests (CUDA path vs the CPU oracle).

bf16 / fp32 outputs: |gpu - ref| <= atol + rtol * |ref| element-wise with
rtol = 1e-2, atol = 2e-2, and the cosine of the two tensors (float64) >= 0.9999.
FP8 E4M3 codes: identical on >= 99.9 % of elements and at most one
representable step apart (monotone code order, +0 and -0 adjacent) elsewhere.
Integer, index and fold outputs: bit-exact (plain equality).
"""
import numpy as np
import torch

from oracle.formats import bf16_decode, e4m3_ordinal

RTOL, ATOL, MIN_COS = 1e-2, 2e-2, 0.9999
MIN_FP8_IDENTICAL = 0.999


def to_bits(t):
    """torch bf16 / uint8 tensor (any device) -> numpy bits."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.uint8:
        return t.numpy()
    raise TypeError(t.dtype)


def from_bits(a, device="cuda"):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def assert_bf16_close(got_bits, ref_bits, what=""):
    g = bf16_decode(got_bits).astype(np.float64).ravel()
    r = bf16_decode(ref_bits).astype(np.float64).ravel()
    assert g.shape == r.shape, what
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - r)
    bad = err > ATOL + RTOL * np.abs(r)
    assert not bad.any(), (f"{what}: {bad.sum()} elements outside tolerance, worst |err| {err.max():.3e} "
                           f"at {int(np.argmax(err))}")
    denom = np.linalg.norm(g) * np.linalg.norm(r)
    if denom > 0:
        cos = float(g @ r / denom)
        assert cos >= MIN_COS, f"{what}: cosine {cos}"
    return float(err.max())


def assert_fp8_codes(got, ref, what=""):
    got = np.asarray(got).ravel()
    ref = np.asarray(ref).ravel()
    assert got.shape == ref.shape, what
    same = np.mean(got == ref)
    steps = np.abs(e4m3_ordinal(got) - e4m3_ordinal(ref))
    assert same >= MIN_FP8_IDENTICAL, f"{what}: only {same:.5f} of codes identical"
    assert steps.max() <= 1, f"{what}: codes up to {steps.max()} steps apart"
    return float(same)
