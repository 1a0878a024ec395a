// fused_add_rmsnorm_fp8: (gated) residual add -> RMSNorm / _noweight /
// AdaRMSNorm -> static-scale FP8 E4M3, one read and one write per element.
//
// Method: "FlashRT 跨层融合深度解析", §2.1 (residual + RMSNorm + FP8
// quantisation fused, data passing only through registers, `_noweight` with the
// norm weight folded into the next GEMM) and §3 (gate_res_adarms_fp8_static:
// gate multiply + residual + AdaRMSNorm modulation + FP8 + descale in one
// kernel); the residual Add as an epilogue follows "OpenPPL算子融合深度解析"
// §3.3.
//
// Layout: a row (token) of H bf16 values is split into H/8 16-byte vectors.
// A group of TPR threads (a power of two, 8..1024) owns one row; each thread
// owns NV vectors strided by TPR, so one warp instruction touches TPR*16
// contiguous bytes.  The row is held in registers as the rounded bf16 residual
// (half the registers of float32) between the reduction and the output pass,
// so HBM sees x and res once and res_out and the codes once.
//
// Rounding points: r = x + res (or res + gate*x) in float32 -> res_out =
// bf16_rne(r) -> the norm reads that bf16 value -> y = r_hat * inv * w (or
// * (1 + scale) + shift) in float32, never stored -> code = e4m3_rne_sat(y / s).
#include "common.cuh"
#include "kernels.h"

namespace gbf {
namespace {

constexpr int kMaxBlock = 1024;

template <int MODE, bool GATED, int NV>
__global__ void __launch_bounds__(kMaxBlock)
add_rmsnorm_fp8_kernel(AddRmsNormArgs a) {
  const int tpr = a.tpr;
  const int lane = threadIdx.x & (tpr - 1);
  const int row_in_cta = threadIdx.x / tpr;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * a.rows_per_cta + row_in_cta;
  const bool row_ok = row < a.rows;
  const int nvec = static_cast<int>(a.hidden >> 3);
  const int64_t base = row * a.hidden;

  pdl_wait();

  uint4 xr[NV], rr[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v = lane + k * tpr;
    if (row_ok && v < nvec) {
      xr[k] = ld_stream(static_cast<const __nv_bfloat16*>(a.x) + base + v * 8);
      rr[k] = ld_stream(static_cast<const __nv_bfloat16*>(a.res_in) + base + v * 8);
    }
  }
  pdl_launch_dependents();

  // r = x + res (or res + gate*x) -> res_out = bf16(r); sum of r_hat^2.
  uint4 rh[NV];
  float sumsq = 0.f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v = lane + k * tpr;
    if (row_ok && v < nvec) {
      float xf[8], rf[8], o[8];
      bf16x8_to_f32(xr[k], xf);
      bf16x8_to_f32(rr[k], rf);
      if (GATED) {
        float gf[8];
        bf16x8_to_f32(ld_cached(static_cast<const __nv_bfloat16*>(a.gate) + v * 8), gf);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = fmaf(gf[i], xf[i], rf[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = xf[i] + rf[i];
      }
      rh[k] = f32x8_to_bf16x8(o);
      st_16(static_cast<__nv_bfloat16*>(a.res_out) + base + v * 8, rh[k]);
      float h[8];
      bf16x8_to_f32(rh[k], h);
#pragma unroll
      for (int i = 0; i < 8; ++i) sumsq = fmaf(h[i], h[i], sumsq);
    }
  }

  // Row reduction: shuffles inside the row's lanes, shared memory across warps.
  sumsq = group_sum(sumsq, tpr < 32 ? tpr : 32);
  if (tpr > 32) {
    __shared__ float part[kMaxBlock / 32];
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) part[warp] = sumsq;
    __syncthreads();
    const int wpr = tpr >> 5;               // warps per row
    const int first = (warp / wpr) * wpr;
    float s = 0.f;
    for (int w = 0; w < wpr; ++w) s += part[first + w];
    sumsq = s;
  }
  if (!row_ok) return;

  // inv = 1/sqrt(mean + eps); the descale 1/s is folded into the row factor.
  const float inv = 1.0f / sqrtf(sumsq / static_cast<float>(a.hidden) + a.eps);
  const float rs = 1.0f / a.fp8_scale;
  const float row_factor = inv * rs;

#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v = lane + k * tpr;
    if (v < nvec) {
      float h[8], q[8];
      bf16x8_to_f32(rh[k], h);
      if (MODE == kNormWeight) {
        float wf[8];
        bf16x8_to_f32(ld_cached(static_cast<const __nv_bfloat16*>(a.weight) + v * 8), wf);
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = (h[i] * row_factor) * wf[i];
      } else if (MODE == kNormNoWeight) {
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = h[i] * row_factor;
      } else {
        float sc[8], sh[8];
        bf16x8_to_f32(ld_cached(static_cast<const __nv_bfloat16*>(a.ada_scale) + v * 8), sc);
        bf16x8_to_f32(ld_cached(static_cast<const __nv_bfloat16*>(a.ada_shift) + v * 8), sh);
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = fmaf(h[i] * inv, 1.0f + sc[i], sh[i]) * rs;
      }
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.q_out) + base + v * 8) = f32x8_to_e4m3x8(q);
    }
  }
}

template <int MODE, bool GATED>
cudaError_t launch_mode(const AddRmsNormArgs& a, int nv, dim3 grid, dim3 block, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  switch (nv) {
    case 1: return cudaLaunchKernelEx(&cfg, add_rmsnorm_fp8_kernel<MODE, GATED, 1>, a);
    case 2: return cudaLaunchKernelEx(&cfg, add_rmsnorm_fp8_kernel<MODE, GATED, 2>, a);
    case 4: return cudaLaunchKernelEx(&cfg, add_rmsnorm_fp8_kernel<MODE, GATED, 4>, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

AddRmsNormPlan plan_add_rmsnorm(int64_t rows, int64_t hidden) {
  AddRmsNormPlan p = {};
  const int64_t nvec = hidden / 8;
  int nv = 1;
  while (nv < 4 && nvec > static_cast<int64_t>(nv) * kMaxBlock) nv *= 2;
  int tpr = 8;
  while (static_cast<int64_t>(tpr) * nv < nvec) tpr *= 2;
  p.ok = static_cast<int64_t>(tpr) * nv >= nvec && tpr <= kMaxBlock;
  p.nv = nv;
  p.tpr = tpr;
  // Small rows share a CTA of 256 threads; large rows get a CTA each.
  p.rows_per_cta = tpr >= 256 ? 1 : 256 / tpr;
  p.grid = rows == 0 ? 0 : (rows + p.rows_per_cta - 1) / p.rows_per_cta;
  p.block = tpr * p.rows_per_cta;
  return p;
}

cudaError_t launch_add_rmsnorm_fp8(AddRmsNormArgs a, cudaStream_t stream, bool pdl) {
  const AddRmsNormPlan p = plan_add_rmsnorm(a.rows, a.hidden);
  if (!p.ok) return cudaErrorInvalidValue;
  if (p.grid == 0) return cudaSuccess;
  a.tpr = p.tpr;
  a.rows_per_cta = p.rows_per_cta;
  const dim3 grid(static_cast<unsigned>(p.grid)), block(static_cast<unsigned>(p.block));
  const bool gated = a.gate != nullptr;
  switch (a.mode) {
    case kNormWeight:
      return gated ? launch_mode<kNormWeight, true>(a, p.nv, grid, block, stream, pdl)
                   : launch_mode<kNormWeight, false>(a, p.nv, grid, block, stream, pdl);
    case kNormNoWeight:
      return gated ? launch_mode<kNormNoWeight, true>(a, p.nv, grid, block, stream, pdl)
                   : launch_mode<kNormNoWeight, false>(a, p.nv, grid, block, stream, pdl);
    case kNormAda:
      return gated ? launch_mode<kNormAda, true>(a, p.nv, grid, block, stream, pdl)
                   : launch_mode<kNormAda, false>(a, p.nv, grid, block, stream, pdl);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace gbf
