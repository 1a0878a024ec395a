// bn_fold: fold an inference BatchNorm into the producing Conv/Linear weights.
//
// Method: "OpenPPL算子融合深度解析", §3.1 (scale = gamma / sqrt(var + eps);
// W_new = W * scale per output channel; b_new = (b_conv - mean) * scale + beta;
// a conv without bias gets a zero bias) and §6.2 (fold in FP32, store half);
// the discosf.com operator-fusion how-to, §2.1 (compute the scale first, then
// the weights, then the bias from the old bias) and §4.1 (eps comes from the
// model).  The weight is [out_ch, inner] with inner = Cin*kh*kw for a conv.
//
// Arithmetic: binary32, one IEEE round-to-nearest operation per step in the
// order above (__fadd_rn / __fsqrt_rn / __fdiv_rn / __fmul_rn / __fsub_rn, which
// the compiler never contracts into a fused multiply-add), then one rounding to
// bf16.  The result is therefore bit-identical to any correctly rounded
// binary32 evaluation of the same expression tree.
//
// Layout: one warp per output channel at a time (grid-stride over channels);
// lanes stream the channel's row as 16-byte vectors, four in flight per lane.
// Rows whose length or alignment does not allow 16-byte access take a scalar
// loop.
#include "common.cuh"
#include "kernels.h"

namespace gbf {
namespace {

constexpr int kBnBlock = 256;
constexpr int kBnUnroll = 4;

GBF_DEVICE float fold_scale(const BnFoldArgs& a, int64_t c) {
  return __fdiv_rn(a.gamma[c], __fsqrt_rn(__fadd_rn(a.var[c], a.eps)));
}

template <bool VEC>
__global__ void __launch_bounds__(kBnBlock) bn_fold_kernel(const BnFoldArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kBnBlock + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kBnBlock) >> 5;
  for (int64_t c = warp; c < a.out_ch; c += nwarps) {
    const float s = fold_scale(a, c);
    if (lane == 0) {
      const float b = a.b ? bf16_bits_to_f32(static_cast<const uint16_t*>(a.b)[c]) : 0.0f;
      const float bn = __fadd_rn(__fmul_rn(__fsub_rn(b, a.mean[c]), s), a.beta[c]);
      static_cast<__nv_bfloat16*>(a.b_out)[c] = __float2bfloat16_rn(bn);
    }
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(a.w) + c * a.inner;
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.w_out) + c * a.inner;
    if (VEC) {
      const int nvec = static_cast<int>(a.inner >> 3);
      for (int base = 0; base < nvec; base += 32 * kBnUnroll) {
        uint4 v[kBnUnroll];
#pragma unroll
        for (int k = 0; k < kBnUnroll; ++k) {
          const int i = base + k * 32 + lane;
          if (i < nvec) v[k] = ld_stream(src + i * 8);
        }
#pragma unroll
        for (int k = 0; k < kBnUnroll; ++k) {
          const int i = base + k * 32 + lane;
          if (i < nvec) {
            float f[8];
            bf16x8_to_f32(v[k], f);
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = __fmul_rn(f[e], s);
            st_16(dst + i * 8, f32x8_to_bf16x8(f));
          }
        }
      }
    } else {
      for (int64_t i = lane; i < a.inner; i += 32)
        dst[i] = __float2bfloat16_rn(__fmul_rn(__bfloat162float(src[i]), s));
    }
  }
}

// Norm-weight pre-fold (FlashRT §3, the `_noweight` RMSNorm's Gemma-style
// weight moved into the next GEMM): W'[c, k] = W[c, k] * g[k] with
// g = 1 + gamma (gemma) or gamma, each one binary32 operation, then one bf16
// rounding.  Same layout as the BN fold: a warp per output row.
template <bool VEC>
__global__ void __launch_bounds__(kBnBlock) fold_norm_weight_kernel(const NormFoldArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kBnBlock + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kBnBlock) >> 5;
  const __nv_bfloat16* gam = static_cast<const __nv_bfloat16*>(a.gamma);
  auto g_of = [&](float gv) { return a.gemma ? __fadd_rn(1.0f, gv) : gv; };
  for (int64_t c = warp; c < a.out_ch; c += nwarps) {
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(a.w) + c * a.inner;
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.w_out) + c * a.inner;
    if (VEC) {
      const int nvec = static_cast<int>(a.inner >> 3);
      for (int base = 0; base < nvec; base += 32 * kBnUnroll) {
        // the gamma vectors (L1-resident, shared by every row) are requested
        // with the row's vectors, not after them
        uint4 v[kBnUnroll], gq[kBnUnroll];
#pragma unroll
        for (int k = 0; k < kBnUnroll; ++k) {
          const int i = base + k * 32 + lane;
          if (i < nvec) {
            v[k] = ld_stream(src + i * 8);
            gq[k] = ld_cached(gam + i * 8);
          }
        }
#pragma unroll
        for (int k = 0; k < kBnUnroll; ++k) {
          const int i = base + k * 32 + lane;
          if (i < nvec) {
            float f[8], gv[8];
            bf16x8_to_f32(v[k], f);
            bf16x8_to_f32(gq[k], gv);
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = __fmul_rn(f[e], g_of(gv[e]));
            st_16(dst + i * 8, f32x8_to_bf16x8(f));
          }
        }
      }
    } else {
      for (int64_t i = lane; i < a.inner; i += 32)
        dst[i] = __float2bfloat16_rn(__fmul_rn(__bfloat162float(src[i]), g_of(__bfloat162float(gam[i]))));
    }
  }
}

}  // namespace

cudaError_t launch_fold_norm_weight(const NormFoldArgs& a, cudaStream_t stream) {
  if (a.out_ch == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (a.out_ch + (kBnBlock / 32) - 1) / (kBnBlock / 32);
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 148) * 8;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  const bool vec = (a.inner % 8 == 0) && (reinterpret_cast<uintptr_t>(a.w) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(a.w_out) % 16 == 0) && (reinterpret_cast<uintptr_t>(a.gamma) % 16 == 0);
  return vec ? launch_pdl(fold_norm_weight_kernel<true>, dim3(grid), dim3(kBnBlock), 0, stream, a)
             : launch_pdl(fold_norm_weight_kernel<false>, dim3(grid), dim3(kBnBlock), 0, stream, a);
}

cudaError_t launch_bn_fold(const BnFoldArgs& a, cudaStream_t stream) {
  if (a.out_ch == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (a.out_ch + (kBnBlock / 32) - 1) / (kBnBlock / 32);
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 148) * 8;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  const bool vec = (a.inner % 8 == 0) && (reinterpret_cast<uintptr_t>(a.w) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(a.w_out) % 16 == 0);
  return vec ? launch_pdl(bn_fold_kernel<true>, dim3(grid), dim3(kBnBlock), 0, stream, a)
             : launch_pdl(bn_fold_kernel<false>, dim3(grid), dim3(kBnBlock), 0, stream, a);
}

}  // namespace gbf
