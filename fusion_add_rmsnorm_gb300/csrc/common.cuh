// Shared device helpers for the fused kernels (sm_103a).
//
// Storage formats: bfloat16 activations and weights, OCP FP8 E4M3 codes,
// float32 arithmetic in registers.  The helpers wrap CUDA intrinsics and PTX
// instructions; the one formula written out, the fast erf, follows a
// published approximation (cited where it is defined), and no math-library
// routine is re-implemented.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define GBF_DEVICE __device__ __forceinline__
#define GBF_HOST_DEVICE __host__ __device__ __forceinline__

namespace gbf {

// Bits of the device-side error word (a library-owned __device__ variable whose
// address every launch receives; read and cleared by gbf_device_status()).
enum : unsigned int {
  DEV_ERR_SLOT_RANGE = 1u << 0,    // a KV-cache slot index was outside [0, cache_rows)
  DEV_ERR_MBAR_TIMEOUT = 1u << 1,  // a bounded mbarrier wait gave up
  DEV_ERR_PAIR_TMEM = 1u << 2,     // the two CTAs of a tensor-core pair got different TMEM bases
};

GBF_DEVICE void raise_error(unsigned int* err, unsigned int bit) {
  if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------- 16-byte I/O

// Streaming 16-byte load that does not allocate in L1.  A plain (coherent)
// load, not the read-only path: under programmatic dependent launch the data
// may have been written by the grid this one waited for.
GBF_DEVICE uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16-byte load that may be served from L1 (small broadcast vectors: weights).
GBF_DEVICE uint4 ld_cached(const void* p) { return *reinterpret_cast<const uint4*>(p); }

GBF_DEVICE void st_16(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// ------------------------------------------------------------- bf16 packing

// 8 bf16 in a uint4 -> 8 floats (exact widening).
GBF_DEVICE void bf16x8_to_f32(uint4 v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// 2 floats -> packed bf16x2 (round to nearest even; lower address = a).
GBF_DEVICE uint32_t f32x2_to_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

GBF_DEVICE uint4 f32x8_to_bf16x8(const float f[8]) {
  uint4 v;
  v.x = f32x2_to_bf16x2(f[0], f[1]);
  v.y = f32x2_to_bf16x2(f[2], f[3]);
  v.z = f32x2_to_bf16x2(f[4], f[5]);
  v.w = f32x2_to_bf16x2(f[6], f[7]);
  return v;
}

GBF_DEVICE float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// a * b + c for bf16 a, b (the halves `lo`/`hi` of packed words) and float32
// c, rounded once to float32.  A bf16 x bf16 product is exact in float32, so
// with c = 0 this is the float32 product of the widened values.
GBF_DEVICE float fma_bf16_lo(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\t"
      "mov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %3;\n\t}"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}
GBF_DEVICE float fma_bf16_hi(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\t"
      "mov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, ah, bh, %3;\n\t}"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}

// --------------------------------------------------------------- E4M3 packing

// 2 floats -> 2 E4M3 codes (round to nearest even, saturate to +-448); the
// code of `a` lands at the lower address.
GBF_DEVICE uint16_t f32x2_to_e4m3x2(float a, float b) {
  return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

GBF_DEVICE uint2 f32x8_to_e4m3x8(const float f[8]) {
  uint2 v;
  v.x = static_cast<uint32_t>(f32x2_to_e4m3x2(f[0], f[1])) | (static_cast<uint32_t>(f32x2_to_e4m3x2(f[2], f[3])) << 16);
  v.y = static_cast<uint32_t>(f32x2_to_e4m3x2(f[4], f[5])) | (static_cast<uint32_t>(f32x2_to_e4m3x2(f[6], f[7])) << 16);
  return v;
}

// ------------------------------------------------------------ reductions

GBF_DEVICE float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over aligned groups of `width` lanes (width a power of two <= 32).
GBF_DEVICE float group_sum(float v, int width) {
  for (int o = width >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over the aligned segment of `width` lanes (a power of two <= 32) that
// holds this lane; only that segment's lanes take part, so segments of one
// warp may follow different control paths.
GBF_DEVICE float segment_sum(float v, int width) {
  const unsigned lane = threadIdx.x & 31u;
  const unsigned seg = width >= 32 ? 0xffffffffu : (((1u << width) - 1u) << (lane & ~static_cast<unsigned>(width - 1)));
  for (int o = width >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(seg, v, o);
  return v;
}

// ------------------------------------------------------------ activations

// GELU, exact form 0.5 a (1 + erf(a / sqrt 2)), with the library erff.
GBF_DEVICE float act_gelu_erf(float a) { return 0.5f * a * (1.0f + erff(a * 0.70710678118654752f)); }

// Fast forms for epilogues, well inside one bf16 rounding:
//  * tanh GELU with the hardware tanh approximation (tanh.approx.f32, relative
//    error below 2^-10.9);
//  * erf GELU with erf(x) = 1 - (a1 t + ... + a5 t^5) e^(-x^2), t = 1/(1 + p x)
//    for x >= 0 (M. Abramowitz, I. Stegun, "Handbook of Mathematical
//    Functions", 1964, formula 7.1.26; absolute error below 1.5e-7), odd in x,
//    with t from the hardware reciprocal approximation (rcp.approx, 1 ulp);
//  * SiLU with the fast exponential and division intrinsics.
GBF_DEVICE float tanh_approx(float a) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(a));
  return t;
}
GBF_DEVICE float rcp_approx(float a) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
  return r;
}
GBF_DEVICE float erf_as7126(float x) {
  const float ax = fabsf(x);
  const float t = rcp_approx(fmaf(0.3275911f, ax, 1.0f));   // argument >= 1: no subnormal or zero
  float poly = fmaf(1.061405429f, t, -1.453152027f);
  poly = fmaf(poly, t, 1.421413741f);
  poly = fmaf(poly, t, -0.284496736f);
  poly = fmaf(poly, t, 0.254829592f);
  poly *= t;
  const float y = 1.0f - poly * __expf(-ax * ax);
  return copysignf(y, x);
}
GBF_DEVICE float fast_act(float a, int act) {
  switch (act) {
    case 1: return 0.5f * a * (1.0f + tanh_approx(0.7978845608f * fmaf(0.044715f * a, a * a, a)));
    case 2: return 0.5f * a * (1.0f + erf_as7126(a * 0.70710678118654752f));
    case 3: return __fdividef(a, 1.0f + __expf(-a));
    default: return a;
  }
}

// fast_act on a pair with packed float32x2 arithmetic; the tanh GELU as
// h + h t with h = a / 2 (one multiply fewer than h (1 + t)).
GBF_DEVICE float2 fast_act2(float2 a, int act) {
  if (act == 1) {
    const float2 a2 = __fmul2_rn(a, a);
    const float2 poly = __ffma2_rn(__fmul2_rn(make_float2(0.044715f, 0.044715f), a), a2, a);
    const float2 inner = __fmul2_rn(make_float2(0.7978845608f, 0.7978845608f), poly);
    const float2 t = make_float2(tanh_approx(inner.x), tanh_approx(inner.y));
    const float2 h = __fmul2_rn(make_float2(0.5f, 0.5f), a);
    return __ffma2_rn(h, t, h);
  }
  return make_float2(fast_act(a.x, act), fast_act(a.y, act));
}

// --------------------------------------------- programmatic dependent launch

// Wait until the grids this launch depends on have completed and their
// memory is visible (a no-op when the launch carried no programmatic edge).
GBF_DEVICE void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next grid in the stream to begin launching.
GBF_DEVICE void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// Launch `kernel` with programmatic stream serialisation: its CTAs may be
// scheduled while the previous kernel in the stream is finishing, and they
// wait for that kernel (completion and memory) in pdl_wait(), which every
// kernel launched this way calls before its first global memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace gbf
