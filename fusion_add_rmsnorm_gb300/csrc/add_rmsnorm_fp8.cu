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
// stride, keeps its columns' factors (weight, gate, AdaRMSNorm scale and shift)
// in registers or, where registers would cost resident CTAs, in shared memory
// for the whole launch, and (up to four vectors per thread) loads the next
// row's x and res while it reduces and writes the current one.  A row wider
// than one warp reduces through per-warp partial sums in shared memory with
// one barrier per row.
//
// Rounding points: res_out = bf16(x + res) or bf16(res + gate * x), one
// rounding of the exact value (bf16x2 add / fused multiply-add); the norm reads
// that bf16 value; y = r_hat * inv * w (or * (1 + scale) + shift) stays in
// float32 registers with the descale 1/s folded into the per-column factors;
// code = e4m3_rne_sat(y / s).
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "kernels.h"

namespace gbf {
namespace {

// Where a thread keeps the per-column factors (weight, gate, AdaRMSNorm scale
// and shift) of its NV vectors:
//  kFacReg   float32 in registers with the descale folded in (one or two
//            vectors per thread, no AdaRMSNorm at two);
//  kFacPack  packed bf16 in registers, widened at each use (launch-bound
//            plans, at most one row per SM: every factor requested with the
//            row);
//  kFacSmem  packed bf16 in shared memory, copied there once per CTA (wide
//            rows and AdaRMSNorm at two vectors, where registers would cost
//            resident CTAs).
enum { kFacReg = 0, kFacPack = 1, kFacSmem = 2 };

constexpr int kMaxBlock = 512;
constexpr int max_block(int nv) { return nv == 1 || nv == 8 ? kMaxBlock : 256; }
// resident CTAs the register budget is sized for: three of 256 threads at two
// vectors, two at four (each with the next row in flight)
constexpr int min_blocks(int nv, int fac) { return fac == kFacPack ? 1 : nv == 2 ? 3 : nv == 4 ? 2 : 1; }

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

// Factor vectors per column group: the gate (GATED) first, then the weight
// (WEIGHT) or the scale and the shift (ADA).
template <int MODE, bool GATED>
constexpr int factor_count() { return (GATED ? 1 : 0) + (MODE == kNormWeight ? 1 : 0) + (MODE == kNormAda ? 2 : 0); }

// Per-column factors from packed bf16 with the descale folded in:
//   WEIGHT: fa = w / s;  ADA: fa = (1 + scale) / s, fb = shift / s.
template <int MODE>
GBF_DEVICE void unpack_factors(uint4 f0, uint4 f1, float rs, float (&fa)[8], float (&fb)[8]) {
  if (MODE == kNormWeight) {
    float w[8];
    bf16x8_to_f32(f0, w);
#pragma unroll
    for (int i = 0; i < 8; ++i) fa[i] = w[i] * rs;
  } else if (MODE == kNormAda) {
    float sc[8], sh[8];
    bf16x8_to_f32(f0, sc);
    bf16x8_to_f32(f1, sh);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      fa[i] = (1.0f + sc[i]) * rs;
      fb[i] = sh[i] * rs;
    }
  }
}

template <int MODE, bool GATED, int NV, int FAC>
__global__ void __launch_bounds__(max_block(NV), min_blocks(NV, FAC))
add_rmsnorm_fp8_kernel(AddRmsNormArgs a) {
  // Rows of up to four vectors per thread keep the next row's x and res in
  // registers (prefetch); wider rows issue their loads at the top of each row.
  constexpr bool PF = NV <= 4;
  constexpr int NFAC = factor_count<MODE, GATED>();
  constexpr int NREG = FAC == kFacReg ? NV : 1;     // float factor sets held in registers
  constexpr int NPK = FAC == kFacPack ? NV : 1;     // packed factor sets held in registers
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
  // factor sources in the order of factor_count: gate, weight | scale, shift
  const void* fsrc[3] = {GATED ? a.gate : (MODE == kNormWeight ? a.weight : a.ada_scale),
                         GATED ? (MODE == kNormWeight ? a.weight : a.ada_scale) : a.ada_shift, a.ada_shift};
  extern __shared__ uint4 sfac[];                   // kFacSmem: [NFAC][nvec] packed bf16

  pdl_wait();

  bool vok[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) vok[k] = lane + k * tpr < nvec;

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
  if (PF) load_row(row);
  // the factors are requested after the first row, whose loads need nothing
  float fa[NREG][8], fb[NREG][8];
  uint4 gate[NREG];
  uint4 pk[NPK][NFAC > 0 ? NFAC : 1];
  if (FAC == kFacReg) {
#pragma unroll
    for (int k = 0; k < NREG; ++k) {
      if (!vok[k]) continue;
      const int c = lane + k * tpr;
      uint4 f[3] = {};
#pragma unroll
      for (int j = 0; j < NFAC; ++j) f[j] = ld_cached(static_cast<const uint4*>(fsrc[j]) + c);
      if (GATED) gate[k] = f[0];
      unpack_factors<MODE>(f[GATED ? 1 : 0], f[GATED ? 2 : 1], rs, fa[k], fb[k]);
    }
  } else if (FAC == kFacPack) {
#pragma unroll
    for (int k = 0; k < NPK; ++k)
      if (vok[k])
#pragma unroll
        for (int j = 0; j < NFAC; ++j) pk[k][j] = ld_cached(static_cast<const uint4*>(fsrc[j]) + lane + k * tpr);
  }

  if (FAC == kFacSmem && NFAC > 0) {
    // the copy's loads are issued in batches of about eight per thread, so a
    // CTA waits about one round trip per batch, not one per vector
    constexpr int kStageBatch = NFAC >= 3 ? 2 : 8 / (NFAC > 0 ? NFAC : 1);
    for (int i0 = threadIdx.x; i0 < nvec; i0 += kStageBatch * blockDim.x) {
      uint4 f[NFAC > 0 ? NFAC : 1][kStageBatch];
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int i = i0 + u * blockDim.x;
#pragma unroll
        for (int j = 0; j < NFAC; ++j)
          if (i < nvec) f[j][u] = ld_cached(static_cast<const uint4*>(fsrc[j]) + i);
      }
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int i = i0 + u * blockDim.x;
#pragma unroll
        for (int j = 0; j < NFAC; ++j)
          if (i < nvec) sfac[j * nvec + i] = f[j][u];
      }
    }
    __syncthreads();
  }
  pdl_launch_dependents();

  // Packed factors of vector k (gate first): from registers or shared memory.
  auto packed = [&](int k, int j) -> uint4 {
    if (FAC == kFacPack) return pk[FAC == kFacPack ? k : 0][j];
    return sfac[j * nvec + lane + k * tpr];
  };

  // Per-warp partial sums, double-buffered by trip parity: one barrier per
  // row (a warp that reaches trip n + 2 has passed the barrier of trip n + 1,
  // which every warp reaches only after reading trip n's partials).
  __shared__ float part[2][kMaxBlock / 32];
  const int warp = threadIdx.x >> 5;
  const int wpr = tpr >> 5;                        // warps per row (when tpr > 32)
  const int first_warp = tpr > 32 ? (warp / wpr) * wpr : 0;
  // every thread of the CTA runs the same number of trips (the reduction syncs)
  const int64_t rows_cta0 = a.rows - static_cast<int64_t>(blockIdx.x) * a.rows_per_cta;
  const int64_t trips = rows_cta0 <= 0 ? 0 : (rows_cta0 + row_stride - 1) / row_stride;

  for (int64_t trip = 0; trip < trips; ++trip, row += row_stride) {
    const bool row_ok = row < a.rows;
    uint4 cx[NV], cr[NV];
    if (!PF) load_row(row);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      cx[k] = xr[k];
      cr[k] = rr[k];
    }
    if (PF) load_row(row + row_stride);            // next row in flight during this one

    uint4 rh[NV];
    float sumsq = 0.f;
    if (row_ok) {
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        if (!vok[k]) continue;
        if (GATED) {
          const uint4 g = FAC == kFacReg ? gate[FAC == kFacReg ? k : 0] : packed(k, 0);
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
      float* pt = part[trip & 1];
      if ((threadIdx.x & 31) == 0) pt[warp] = sumsq;
      __syncthreads();
      float s = 0.f;
      for (int w = 0; w < wpr; ++w) s += pt[first_warp + w];
      sumsq = s;
    }
    if (!row_ok) continue;
    const float inv = 1.0f / sqrtf(sumsq / static_cast<float>(a.hidden) + a.eps);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (!vok[k]) continue;
      float h[8], q[8];
      bf16x8_to_f32(rh[k], h);
      float ua[8], ub[8];
      const float* fak = fa[0];
      const float* fbk = fb[0];
      if (FAC == kFacReg) {
        fak = fa[FAC == kFacReg ? k : 0];
        fbk = fb[FAC == kFacReg ? k : 0];
      } else if (MODE != kNormNoWeight) {
        unpack_factors<MODE>(packed(k, GATED ? 1 : 0), MODE == kNormAda ? packed(k, GATED ? 2 : 1) : uint4{},
                             rs, ua, ub);
        fak = ua;
        fbk = ub;
      }
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

// CTAs of `kern` with `block` threads and `smem` dynamic shared memory that
// fit on one SM (cached; the persistent grid is capped at that many per SM).
// The default dynamic shared memory limit (48 KB less the static shared
// memory) is below some factor tables, e.g. 48 KB for three [8192] vectors,
// so the kernel's limit is raised once to the device's opt-in maximum: the
// attribute is only an upper bound and never has to shrink.
template <typename K>
int resident_per_sm(K kern, int block, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, size_t>, int> cache;
  static std::map<const void*, bool> raised;
  std::lock_guard<std::mutex> lock(mu);
  const void* fn = reinterpret_cast<const void*>(kern);
  if (smem > 0 && !raised[fn]) {
    int dev = 0, optin = 0;
    cudaFuncAttributes fa = {};
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    // the opt-in maximum covers static and dynamic shared memory together
    if (cudaFuncGetAttributes(&fa, kern) == cudaSuccess && optin > static_cast<int>(fa.sharedSizeBytes) &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - static_cast<int>(fa.sharedSizeBytes)) == cudaSuccess)
      raised[fn] = true;
    cudaGetLastError();
  }
  const auto key = std::make_tuple(fn, block, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, block, smem) != cudaSuccess || occ < 1) {
    cudaGetLastError();
    occ = 1;                                       // the launch itself reports a configuration that cannot run
  }
  cache[key] = occ;
  return occ;
}

template <int MODE, bool GATED, int NV, int FAC>
cudaError_t launch_nv(const AddRmsNormArgs& a, int64_t blocks, dim3 block, cudaStream_t s, bool pdl) {
  auto kern = add_rmsnorm_fp8_kernel<MODE, GATED, NV, FAC>;
  const size_t smem = FAC == kFacSmem ? static_cast<size_t>(factor_count<MODE, GATED>()) * a.hidden * 2 : 0;
  const int per_sm = resident_per_sm(kern, static_cast<int>(block.x), smem);
  const int64_t cap = static_cast<int64_t>(sm_count()) * per_sm;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks < cap ? blocks : cap));
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int MODE, bool GATED>
cudaError_t launch_mode(const AddRmsNormArgs& a, const AddRmsNormPlan& p, cudaStream_t s, bool pdl) {
  const dim3 block(static_cast<unsigned>(p.block));
  switch (p.nv * 4 + p.fac) {
    case 1 * 4 + kFacReg: return launch_nv<MODE, GATED, 1, kFacReg>(a, p.grid, block, s, pdl);
    case 2 * 4 + kFacReg:
      // the planner keeps AdaRMSNorm's factors in shared memory at two vectors
      if constexpr (MODE == kNormAda) return cudaErrorInvalidValue;
      else return launch_nv<MODE, GATED, 2, kFacReg>(a, p.grid, block, s, pdl);
    case 2 * 4 + kFacPack: return launch_nv<MODE, GATED, 2, kFacPack>(a, p.grid, block, s, pdl);
    case 2 * 4 + kFacSmem: return launch_nv<MODE, GATED, 2, kFacSmem>(a, p.grid, block, s, pdl);
    case 4 * 4 + kFacPack: return launch_nv<MODE, GATED, 4, kFacPack>(a, p.grid, block, s, pdl);
    case 4 * 4 + kFacSmem: return launch_nv<MODE, GATED, 4, kFacSmem>(a, p.grid, block, s, pdl);
    case 8 * 4 + kFacSmem: return launch_nv<MODE, GATED, 8, kFacSmem>(a, p.grid, block, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

AddRmsNormPlan plan_add_rmsnorm(int64_t rows, int64_t hidden, int mode) {
  AddRmsNormPlan p = {};
  const int64_t nvec = hidden / 8;
  const bool large = rows * nvec >= 4LL * sm_count() * 2048;
  int nv = 1;
  if (!large && nvec <= 128) {
    // Launch-bound rows of up to 1024 values: at most 64 threads per row (two
    // vectors each above 512 values), the factors requested with the row and
    // kept packed in registers; measured on the 180-call Pi0.5 chain
    // ([10, 1024]), 64 threads x 2 vectors beat 128 x 1 and 32 x 4.
    while (nv < 2 && nvec > 64 * nv) nv *= 2;
    p.fac = nv == 1 ? kFacReg : kFacPack;
  } else {
    // Vectors per thread: 2 for streaming launches and for rows of 2048 values
    // or more in smaller ones (half the per-row reduction and loop work per
    // element, half the warps a row reduces over); more when a row would
    // need more than the block's threads.  Factors: float32 in registers where
    // they fit (one vector, or two without AdaRMSNorm); packed in registers
    // for AdaRMSNorm at two vectors up to 16 rows per SM and for four vectors
    // up to 4 rows per SM (no shared-memory copy and barrier ahead of the
    // first row; the lower occupancy of the larger register set costs less
    // there); else in shared memory.  Measured per call: gated AdaRMSNorm
    // [32, 8192] 2.32 us against 3.22 with shared factors (100-call CUDA
    // graph), [256, 4096] 3.6 against 4.4 with one vector, [2048, 4096] 11.6
    // against 12.6 with shared factors; [1216, 8192] weighted 13.1 with
    // shared factors against 13.9 with packed ones (hence the lower limit at
    // four vectors); [128, 4096] weighted 2.24 against 2.75-2.81 with one
    // vector.
    const int64_t sms = sm_count();
    const int target = large || nvec >= 256 ? 2 : 1;
    while (nv < 8 && ((nv < target && nvec >= 16 * nv) || nvec > static_cast<int64_t>(nv) * max_block(nv)))
      nv *= 2;
    const bool pack = (nv == 2 && rows <= 16 * sms) || (nv == 4 && rows <= 4 * sms);
    p.fac = nv == 1 || (nv == 2 && mode != kNormAda) ? kFacReg : (pack ? kFacPack : kFacSmem);
  }
  int tpr = 8;
  while (static_cast<int64_t>(tpr) * nv < nvec) tpr *= 2;
  p.ok = static_cast<int64_t>(tpr) * nv >= nvec && tpr <= max_block(nv);
  p.nv = nv;
  p.tpr = tpr;
  // Streaming launches: small rows share a CTA of 256 threads, large rows get
  // a CTA each.  Launch-bound ones: a CTA per row (at least one warp), which
  // spreads the few rows over as many SMs.
  p.rows_per_cta = large ? (tpr >= 256 ? 1 : 256 / tpr) : (tpr >= 32 ? 1 : 32 / tpr);
  p.block = tpr * p.rows_per_cta;
  // CTAs needed; the launch caps the persistent grid at the CTAs that fit at once
  p.grid = rows == 0 ? 0 : (rows + p.rows_per_cta - 1) / p.rows_per_cta;
  return p;
}

cudaError_t launch_add_rmsnorm_fp8(AddRmsNormArgs a, cudaStream_t stream, bool pdl) {
  const AddRmsNormPlan p = plan_add_rmsnorm(a.rows, a.hidden, a.mode);
  if (!p.ok) return cudaErrorInvalidValue;
  if (p.grid == 0) return cudaSuccess;
  a.tpr = p.tpr;
  a.rows_per_cta = p.rows_per_cta;
  const bool gated = a.gate != nullptr;
  switch (a.mode) {
    case kNormWeight:
      return gated ? launch_mode<kNormWeight, true>(a, p, stream, pdl)
                   : launch_mode<kNormWeight, false>(a, p, stream, pdl);
    case kNormNoWeight:
      return gated ? launch_mode<kNormNoWeight, true>(a, p, stream, pdl)
                   : launch_mode<kNormNoWeight, false>(a, p, stream, pdl);
    case kNormAda:
      return gated ? launch_mode<kNormAda, true>(a, p, stream, pdl) : launch_mode<kNormAda, false>(a, p, stream, pdl);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace gbf
