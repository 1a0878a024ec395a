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
// A group of TPR threads (a power of two, 8..512) owns one row; each thread
// owns NV vectors strided by TPR, so one warp instruction touches TPR*16
// contiguous bytes.  CTAs are persistent: a CTA walks rows with a grid-sized
// stride, keeps its columns' weight factors in registers for the whole launch,
// and loads the next row's x and res while it reduces and writes the current
// one.
//
// Rounding points: res_out = bf16(x + res) or bf16(res + gate * x), one
// rounding of the exact value (bf16x2 add / fused multiply-add); the norm reads
// that bf16 value; y = r_hat * inv * w (or * (1 + scale) + shift) stays in
// float32 registers with the descale 1/s folded into the per-column factors;
// code = e4m3_rne_sat(y / s).
#include <map>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace gbf {
namespace {

constexpr int kMaxBlock = 512;
// Threads per CTA of the NV-vector kernel: rows of two vectors per thread use
// at most 256 threads, so three CTAs fit on an SM.
constexpr int max_block(int nv) { return nv == 2 ? 256 : kMaxBlock; }

GBF_DEVICE uint4 bf16x8_add(uint4 a, uint4 b) {
  uint4 r;
  const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
  __nv_bfloat162* pr = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) pr[i] = __hadd2(pa[i], pb[i]);
  return r;
}

// g * x + r per element, one rounding
GBF_DEVICE uint4 bf16x8_fma(uint4 g, uint4 x, uint4 r0) {
  uint4 r;
  const __nv_bfloat162* pg = reinterpret_cast<const __nv_bfloat162*>(&g);
  const __nv_bfloat162* px = reinterpret_cast<const __nv_bfloat162*>(&x);
  const __nv_bfloat162* pr0 = reinterpret_cast<const __nv_bfloat162*>(&r0);
  __nv_bfloat162* pr = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) pr[i] = __hfma2(pg[i], px[i], pr0[i]);
  return r;
}

template <int MODE, bool GATED, int NV>
__global__ void __launch_bounds__(max_block(NV), NV == 2 ? 3 : 1)
add_rmsnorm_fp8_kernel(AddRmsNormArgs a) {
  // Rows of up to 2 vectors per thread keep the next row's inputs in
  // registers (prefetch); wider rows (BIG) issue their loads at the top of
  // each row.  The per-column factors stay in registers (REGF) for 1 vector
  // per thread, and for 2 unless the mode is AdaRMSNorm (two factor vectors
  // plus the gate); otherwise they are reloaded from L1 every row, which keeps
  // three CTAs per SM.
  constexpr bool BIG = NV > 2;
  constexpr bool REGF = NV == 1 || (NV == 2 && MODE != kNormAda);
  const int tpr = a.tpr;
  const int lane = threadIdx.x & (tpr - 1);
  const int row_in_cta = threadIdx.x / tpr;
  const int nvec = static_cast<int>(a.hidden >> 3);
  const int64_t row_stride = static_cast<int64_t>(gridDim.x) * a.rows_per_cta;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
  const __nv_bfloat16* res = static_cast<const __nv_bfloat16*>(a.res_in);
  __nv_bfloat16* res_out = static_cast<__nv_bfloat16*>(a.res_out);
  uint8_t* q_out = static_cast<uint8_t*>(a.q_out);
  const float rs = 1.0f / a.fp8_scale;

  pdl_wait();

  bool vok[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) vok[k] = lane + k * tpr < nvec;

  // Per-column factors (descale folded in):
  //   WEIGHT: fa = w / s;  NOWEIGHT: none;  ADA: fa = (1 + scale) / s, fb = shift / s.
  auto factors = [&](int k, float* fa, float* fb) {
    const int col = (lane + k * tpr) * 8;
    if (MODE == kNormWeight) {
      float w[8];
      bf16x8_to_f32(ld_cached(static_cast<const __nv_bfloat16*>(a.weight) + col), w);
#pragma unroll
      for (int i = 0; i < 8; ++i) fa[i] = w[i] * rs;
    } else if (MODE == kNormAda) {
      float sc[8], sh[8];
      bf16x8_to_f32(ld_cached(static_cast<const __nv_bfloat16*>(a.ada_scale) + col), sc);
      bf16x8_to_f32(ld_cached(static_cast<const __nv_bfloat16*>(a.ada_shift) + col), sh);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        fa[i] = (1.0f + sc[i]) * rs;
        fb[i] = sh[i] * rs;
      }
    }
  };
  constexpr int NF = REGF ? NV : 1;
  float fa[NF][8], fb[NF][8];
  uint4 gate[NF];
  if (REGF) {
#pragma unroll
    for (int k = 0; k < NF; ++k) {
      if (!vok[k]) continue;
      if (GATED) gate[k] = ld_cached(static_cast<const __nv_bfloat16*>(a.gate) + (lane + k * tpr) * 8);
      factors(k, fa[k], fb[k]);
    }
  }

  int64_t row = static_cast<int64_t>(blockIdx.x) * a.rows_per_cta + row_in_cta;
  uint4 xr[NV], rr[NV];
  auto load_row = [&](int64_t r) {
    if (r < a.rows) {
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (vok[k]) {
          const int64_t off = r * a.hidden + (lane + k * tpr) * 8;
          xr[k] = ld_stream(x + off);
          rr[k] = ld_stream(res + off);
        }
    }
  };
  if (!BIG) load_row(row);
  pdl_launch_dependents();

  __shared__ float part[kMaxBlock / 32];
  const int warp = threadIdx.x >> 5;
  const int wpr = tpr >> 5;                        // warps per row (when tpr > 32)
  const int first_warp = tpr > 32 ? (warp / wpr) * wpr : 0;
  // every thread of the CTA runs the same number of trips (the reduction syncs)
  const int64_t rows_cta0 = a.rows - static_cast<int64_t>(blockIdx.x) * a.rows_per_cta;
  const int64_t trips = rows_cta0 <= 0 ? 0 : (rows_cta0 + row_stride - 1) / row_stride;

  for (int64_t trip = 0; trip < trips; ++trip, row += row_stride) {
    const bool row_ok = row < a.rows;
    uint4 cx[NV], cr[NV];
    if (BIG) load_row(row);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      cx[k] = xr[k];
      cr[k] = rr[k];
    }
    if (!BIG) load_row(row + row_stride);          // next row in flight during this one

    uint4 rh[NV];
    float sumsq = 0.f;
    if (row_ok) {
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        if (!vok[k]) continue;
        if (GATED) {
          const uint4 g = REGF ? gate[REGF ? k : 0]
                               : ld_cached(static_cast<const __nv_bfloat16*>(a.gate) + (lane + k * tpr) * 8);
          rh[k] = bf16x8_fma(g, cx[k], cr[k]);
        } else {
          rh[k] = bf16x8_add(cx[k], cr[k]);
        }
        st_16(res_out + row * a.hidden + (lane + k * tpr) * 8, rh[k]);
        float h[8];
        bf16x8_to_f32(rh[k], h);
#pragma unroll
        for (int i = 0; i < 8; ++i) sumsq = fmaf(h[i], h[i], sumsq);
      }
    }
    sumsq = group_sum(sumsq, tpr < 32 ? tpr : 32);
    if (tpr > 32) {
      if ((threadIdx.x & 31) == 0) part[warp] = sumsq;
      __syncthreads();
      float s = 0.f;
      for (int w = 0; w < wpr; ++w) s += part[first_warp + w];
      sumsq = s;
      __syncthreads();                             // part[] is rewritten next trip
    }
    if (!row_ok) continue;
    const float inv = 1.0f / sqrtf(sumsq / static_cast<float>(a.hidden) + a.eps);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (!vok[k]) continue;
      float h[8], q[8];
      bf16x8_to_f32(rh[k], h);
      float fbig_a[8], fbig_b[8];
      const float* fak = REGF ? fa[REGF ? k : 0] : fbig_a;
      const float* fbk = REGF ? fb[REGF ? k : 0] : fbig_b;
      if (!REGF) factors(k, fbig_a, fbig_b);
      if (MODE == kNormWeight) {
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = (h[i] * inv) * fak[i];
      } else if (MODE == kNormNoWeight) {
        const float f = inv * rs;
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = h[i] * f;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = fmaf(h[i] * inv, fak[i], fbk[i]);
      }
      *reinterpret_cast<uint2*>(q_out + row * a.hidden + (lane + k * tpr) * 8) = f32x8_to_e4m3x8(q);
    }
  }
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

// CTAs of `kern` with `block` threads that fit on one SM (cached per kernel
// and block size; the persistent grid is capped at that many per SM).
template <typename K>
int resident_per_sm(K kern, int block) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(reinterpret_cast<const void*>(kern), block);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, block, 0) != cudaSuccess || occ < 1) occ = 1;
  cache[key] = occ;
  return occ;
}

template <int MODE, bool GATED, int NV>
cudaError_t launch_nv(const AddRmsNormArgs& a, int64_t blocks, dim3 block, cudaStream_t s, bool pdl) {
  auto kern = add_rmsnorm_fp8_kernel<MODE, GATED, NV>;
  const int64_t cap = static_cast<int64_t>(sm_count()) * resident_per_sm(kern, static_cast<int>(block.x));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks < cap ? blocks : cap));
  cfg.blockDim = block;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int MODE, bool GATED>
cudaError_t launch_mode(const AddRmsNormArgs& a, int nv, int64_t blocks, dim3 block, cudaStream_t s, bool pdl) {
  switch (nv) {
    case 1: return launch_nv<MODE, GATED, 1>(a, blocks, block, s, pdl);
    case 2: return launch_nv<MODE, GATED, 2>(a, blocks, block, s, pdl);
    case 4: return launch_nv<MODE, GATED, 4>(a, blocks, block, s, pdl);
    case 8: return launch_nv<MODE, GATED, 8>(a, blocks, block, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}


}  // namespace

AddRmsNormPlan plan_add_rmsnorm(int64_t rows, int64_t hidden) {
  AddRmsNormPlan p = {};
  const int64_t nvec = hidden / 8;
  // Vectors per thread: 1 for launch-bound shapes (the most threads per row,
  // the shortest critical path); 2 once there are at least four vectors per
  // thread the GPU holds at once (half the per-row reduction and loop work per
  // element); more when a row would need more than kMaxBlock threads.  Rows
  // keep at least 8 threads.
  const bool large = rows * nvec >= 4LL * sm_count() * 2048;
  const int target = large ? 2 : 1;
  int nv = 1;
  while (nv < 8 && ((nv < target && nvec >= 16 * nv) || nvec > static_cast<int64_t>(nv) * max_block(nv))) nv *= 2;
  int tpr = 8;
  while (static_cast<int64_t>(tpr) * nv < nvec) tpr *= 2;
  p.ok = static_cast<int64_t>(tpr) * nv >= nvec && tpr <= max_block(nv);
  p.nv = nv;
  p.tpr = tpr;
  // Small rows share a CTA of 256 threads; large rows get a CTA each.
  p.rows_per_cta = tpr >= 256 ? 1 : 256 / tpr;
  p.block = tpr * p.rows_per_cta;
  // CTAs needed; the launch caps the persistent grid at the CTAs that fit at once
  p.grid = rows == 0 ? 0 : (rows + p.rows_per_cta - 1) / p.rows_per_cta;
  return p;
}

cudaError_t launch_add_rmsnorm_fp8(AddRmsNormArgs a, cudaStream_t stream, bool pdl) {
  const AddRmsNormPlan p = plan_add_rmsnorm(a.rows, a.hidden);
  if (!p.ok) return cudaErrorInvalidValue;
  if (p.grid == 0) return cudaSuccess;
  a.tpr = p.tpr;
  a.rows_per_cta = p.rows_per_cta;
  const int64_t blocks = p.grid;
  const dim3 block(static_cast<unsigned>(p.block));
  const bool gated = a.gate != nullptr;
  switch (a.mode) {
    case kNormWeight:
      return gated ? launch_mode<kNormWeight, true>(a, p.nv, blocks, block, stream, pdl)
                   : launch_mode<kNormWeight, false>(a, p.nv, blocks, block, stream, pdl);
    case kNormNoWeight:
      return gated ? launch_mode<kNormNoWeight, true>(a, p.nv, blocks, block, stream, pdl)
                   : launch_mode<kNormNoWeight, false>(a, p.nv, blocks, block, stream, pdl);
    case kNormAda:
      return gated ? launch_mode<kNormAda, true>(a, p.nv, blocks, block, stream, pdl)
                   : launch_mode<kNormAda, false>(a, p.nv, blocks, block, stream, pdl);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace gbf
