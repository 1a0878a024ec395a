// gated_act: y = act(gate) * up over a [rows, 2d] projection holding
// [gate | up] per row -- SwiGLU with SiLU, GELU x Mul with a GELU.
//
// Method: "RFC：自动融合: 扩展统一 Pattern Matcher 覆盖量化融合与 GMM/MM+激活",
// §2.4 (non-MM fusions: gelu(x) * gate -> npu_gelu_mul, silu gating ->
// npu_swiglu, the erf GELU -> npu_gelu) and §3.6 (the patterns: up_out *
// F.gelu(gate_out); SiluAndMul-style gated FFNs).  Unfused, the activation
// writes act(gate) to HBM and the multiply reads it back; here each row is
// read once and written once.
//
// Design: each row is cut into equal tiles of at most kGaUnroll * kGaBlock
// 16-byte vectors; persistent CTAs walk the (row, tile) pairs (grid-stride),
// each thread issuing its (up to kGaUnroll) gate and up loads before any
// arithmetic; float32 math, one bf16 rounding, 16-byte stores.  A launch
// with fewer (row, tile) pairs than SMs (a decode batch) cuts its rows into
// more, smaller tiles (down to 64 vectors, at most one tile per SM), so the
// work spreads over the SMs and a thread's critical path is about one
// vector.  SiLU uses the fast exponential and division intrinsics and the
// tanh GELU the hardware tanh approximation (both well inside a bf16
// rounding); the erf GELU calls erff.  Launched with programmatic dependent
// launch.
#include <map>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace gbf {
namespace {

constexpr int kGaBlock = 256;
constexpr int kGaUnroll = 4;

// SiLU and tanh GELU by the fast forms; erf GELU with the library erff.
template <int ACT>
GBF_DEVICE float gate_act(float a) {
  return ACT == kActGeluErf ? act_gelu_erf(a) : fast_act(a, ACT);
}

template <int ACT>
__global__ void __launch_bounds__(kGaBlock) gated_act_kernel(const GatedActArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t nv = a.d >> 3;                 // 16-byte vectors per half row
  const int64_t tiles_per_row = a.tiles_per_row;
  const int64_t per_tile = (nv + tiles_per_row - 1) / tiles_per_row;
  const int64_t tiles = a.rows * tiles_per_row;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
  __nv_bfloat16* y = static_cast<__nv_bfloat16*>(a.y);
  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int64_t r = tile / tiles_per_row;
    const int64_t c0 = (tile - r * tiles_per_row) * per_tile;
    const int64_t c1 = c0 + per_tile < nv ? c0 + per_tile : nv;
    const __nv_bfloat16* g = x + r * 2 * a.d;
    const __nv_bfloat16* u = g + a.d;
    __nv_bfloat16* o = y + r * a.d;
    uint4 gv[kGaUnroll], uv[kGaUnroll];
#pragma unroll
    for (int k = 0; k < kGaUnroll; ++k) {
      const int64_t j = c0 + threadIdx.x + k * kGaBlock;
      if (j < c1) {
        gv[k] = ld_stream(g + j * 8);
        uv[k] = ld_stream(u + j * 8);
      }
    }
#pragma unroll
    for (int k = 0; k < kGaUnroll; ++k) {
      const int64_t j = c0 + threadIdx.x + k * kGaBlock;
      if (j >= c1) break;
      float gf[8], uf[8], of[8];
      bf16x8_to_f32(gv[k], gf);
      bf16x8_to_f32(uv[k], uf);
#pragma unroll
      for (int e = 0; e < 8; ++e) of[e] = gate_act<ACT>(gf[e]) * uf[e];
      st_16(o + j * 8, f32x8_to_bf16x8(of));
    }
  }
}

template <int ACT>
cudaError_t launch_act(const GatedActArgs& a, cudaStream_t stream) {
  static std::mutex mu;
  static std::map<int, int> per_sm_cache;   // device -> resident CTAs per SM
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = per_sm_cache.find(dev);
    if (it == per_sm_cache.end()) {
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gated_act_kernel<ACT>, kGaBlock, 0) != cudaSuccess ||
          per_sm < 1)
        per_sm = 1;
      per_sm_cache[dev] = per_sm;
    } else {
      per_sm = it->second;
    }
  }
  const int64_t resident = static_cast<int64_t>(sms) * per_sm;
  const int64_t nv = a.d >> 3;
  GatedActArgs b = a;
  b.tiles_per_row = (nv + kGaUnroll * kGaBlock - 1) / (kGaUnroll * kGaBlock);
  const int64_t fit = sms / a.rows;                       // tiles per row with at most one per SM
  if (fit > b.tiles_per_row) {
    const int64_t most = (nv + 63) / 64;                  // tiles of at least 64 vectors
    b.tiles_per_row = fit < most ? fit : most;
    if (b.tiles_per_row < 1) b.tiles_per_row = 1;
  }
  const int64_t tiles = a.rows * b.tiles_per_row;
  const unsigned grid = static_cast<unsigned>(tiles < resident ? tiles : resident);
  return launch_pdl(gated_act_kernel<ACT>, dim3(grid), dim3(kGaBlock), 0, stream, b);
}

}  // namespace

cudaError_t launch_gated_act(const GatedActArgs& a, cudaStream_t stream) {
  if (a.rows == 0) return cudaSuccess;
  switch (a.act) {
    case kActGeluTanh: return launch_act<kActGeluTanh>(a, stream);
    case kActGeluErf: return launch_act<kActGeluErf>(a, stream);
    case kActSilu: return launch_act<kActSilu>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gbf
