// qkv_split_norm_rope: packed QKV split -> Q/K RMSNorm (per head or full width)
// -> rotate_half RoPE (1D, or 3D over (t, h, w) sections) -> Q, K cache, V cache.
//
// Method: "FlashRT 跨层融合深度解析", §2.2: the Qwen3/GROOT post-processing
// (q_norm -> RoPE -> Q staging, k_norm -> RoPE -> KV-cache write), the Wan
// packed-QKV split + two RMSNorms + 3D RoPE read in one streaming pass, and the
// shared "Q/K norm -> RoPE, V passes through" contract; RMSNorm -> RoPE after
// the Q/K projection with an optional cache write is the kv_rms_norm_rope_cache
// target of the MindIE-SD RFC, §2.4 / §3.6.  The packed row layout [Q | K | V]
// is the merged QKV GEMM output of "OpenPPL算子融合深度解析", §3.2.
//
// Rotation slots.  A head of width D has D/2 rotation slots.  Slot p rotates
// the element pair (lo_idx[p], hi_idx[p]) by pos[axis[p]] * omega[p].  1D
// rotate_half: slot j pairs (j, j + D/2) with omega_j = theta^(-2j/D).  3D: the
// head is cut into contiguous chunks of widths sections[c]; slot j of chunk c
// pairs (start_c + j, start_c + j + sections[c]/2) with omega = theta^(-2j /
// sections[c]) and uses the token's c-th grid coordinate.  The host fills the
// table in float64 and hands each frequency over as a (hi, lo) binary32 pair.
//
// Angles: a = pos * omega is formed as a double-binary32 value and reduced
// modulo 2*pi by Cody and Waite's method (W. J. Cody, W. Waite, "Software
// Manual for the Elementary Functions", 1980) with a two-part 2*pi, then
// sincosf() evaluates the reduced argument.  The absolute angle error stays
// near 1e-7 rad at position 4095, where a plain binary32 product would be
// 2.4e-4 rad off.
//
// Two kernels:
//  * qkv_pair_kernel: per-head norm + 1D rotate_half, D/16 threads per head,
//    each thread holding the 16-byte vectors v and v + D/16 of its head, so
//    both members of every rotation pair sit in the same thread's registers
//    (no shuffle for the rotation); the sum of squares is a shuffle reduction
//    over the head's D/16 lanes.  A CTA handles 8 tokens; the D/2 (cos, sin)
//    pairs of each token are computed once into shared memory and reused by
//    all of the token's Q and K heads.
//  * qkv_staged_kernel: every other combination (full-width norm and/or 3D
//    sections).  One CTA per token stages raw * weight of Q and K in shared
//    memory as float32, reduces the sums of squares, rotates the pairs in
//    place, and writes 16-byte vectors.  V is copied from registers in phase 1.
#include "common.cuh"
#include "kernels.h"

namespace gbf {
namespace {

constexpr float kTwoPiHi = 6.28318548202514648438f;      // binary32(2*pi)
constexpr float kTwoPiLo = -1.74845553146951715e-07f;    // 2*pi - kTwoPiHi
constexpr float kInvTwoPi = 0.159154943091895335769f;

// sin and cos of pos * (omega_hi + omega_lo).
GBF_DEVICE float2 rope_cos_sin(int pos, float omega_hi, float omega_lo) {
  const float p = static_cast<float>(pos);               // exact below 2^24
  const float a_hi = p * omega_hi;
  const float a_lo = fmaf(p, omega_hi, -a_hi) + p * omega_lo;  // product error + low part
  const float k = rintf(a_hi * kInvTwoPi);
  float r = fmaf(-k, kTwoPiHi, a_hi);
  r = fmaf(-k, kTwoPiLo, r);
  r += a_lo;
  float s, c;
  sincosf(r, &s, &c);
  return make_float2(c, s);
}

GBF_DEVICE int64_t cache_row(const QkvArgs& a, int64_t t, bool& ok) {
  int64_t slot = a.slots ? static_cast<int64_t>(a.slots[t]) : t;
  ok = slot >= 0 && slot < a.cache_rows;
  return slot;
}

// ----------------------------------------------------------- per-head, 1D

constexpr int kPairBlock = 256;
constexpr int kPairTokens = 8;                    // tokens per CTA

template <int D>
__global__ void __launch_bounds__(kPairBlock)
qkv_pair_kernel(const __grid_constant__ QkvArgs a) {
  constexpr int LPH = D / 16;                     // lanes per head
  constexpr int HALF_VEC = D / 16;                // 16-byte vectors in half a head
  constexpr int SLOTS = D / 2;
  constexpr int GROUPS = kPairBlock / LPH;        // head tasks in flight per CTA
  __shared__ __align__(16) float2 cs[kPairTokens][SLOTS];

  const int heads = a.n_q + 2 * a.n_kv;
  const int64_t width = static_cast<int64_t>(heads) * D;
  const int lane = threadIdx.x % LPH;
  const int group = threadIdx.x / LPH;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kPairTokens;
  const int64_t left = a.tokens - t0;
  const int ntok = left < kPairTokens ? static_cast<int>(left) : kPairTokens;

  // (cos, sin) of every slot of the CTA's tokens; kPairBlock % SLOTS == 0, so
  // each thread keeps one slot and reads its frequency once.
  {
    const int p = threadIdx.x % SLOTS;
    const float om_hi = a.omega_hi[p], om_lo = a.omega_lo[p];
    for (int j = threadIdx.x / SLOTS; j < ntok; j += kPairBlock / SLOTS)
      cs[j][p] = rope_cos_sin(a.pos[t0 + j], om_hi, om_lo);
  }
  float wq_lo[8], wq_hi[8], wk_lo[8], wk_hi[8];
  bf16x8_to_f32(ld_cached(static_cast<const __nv_bfloat16*>(a.q_w) + lane * 8), wq_lo);
  bf16x8_to_f32(ld_cached(static_cast<const __nv_bfloat16*>(a.q_w) + (lane + HALF_VEC) * 8), wq_hi);
  bf16x8_to_f32(ld_cached(static_cast<const __nv_bfloat16*>(a.k_w) + lane * 8), wk_lo);
  bf16x8_to_f32(ld_cached(static_cast<const __nv_bfloat16*>(a.k_w) + (lane + HALF_VEC) * 8), wk_hi);
  __syncthreads();

  // Head tasks (token j, head h), task = j * heads + h.  The loop bound is the
  // same for every thread, so the shuffle reductions see whole warps; two tasks
  // per trip put four 16-byte loads in flight before any arithmetic.
  const int tasks = ntok * heads;
  for (int base = 0; base < tasks; base += 2 * GROUPS) {
    uint4 lo[2], hi[2];
    int task[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      task[u] = base + group + u * GROUPS;
      if (task[u] < tasks) {
        const int j = task[u] / heads, h = task[u] - j * heads;
        const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(a.qkv) + (t0 + j) * width +
                                   static_cast<int64_t>(h) * D;
        lo[u] = ld_stream(src + lane * 8);
        hi[u] = ld_stream(src + (lane + HALF_VEC) * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const bool valid = task[u] < tasks;
      const int j = valid ? task[u] / heads : 0;
      const int h = valid ? task[u] - j * heads : heads;
      const bool is_qk = h < a.n_q + a.n_kv;
      float xl[8], xh[8];
      float ss = 0.f;
      if (is_qk) {
        bf16x8_to_f32(lo[u], xl);
        bf16x8_to_f32(hi[u], xh);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(xl[i], xl[i], fmaf(xh[i], xh[i], ss));
      }
      ss = group_sum(ss, LPH);                    // every lane takes part
      if (!valid) continue;
      const int64_t t = t0 + j;
      bool slot_ok;
      const int64_t crow = cache_row(a, t, slot_ok);
      if (h >= a.n_q && !slot_ok) {
        if (lane == 0) raise_error(a.err, DEV_ERR_SLOT_RANGE);
        continue;
      }
      if (!is_qk) {                               // V: pass through
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.v_cache) +
                             (crow * a.n_kv + (h - a.n_q - a.n_kv)) * D;
        st_16(dst + lane * 8, lo[u]);
        st_16(dst + (lane + HALF_VEC) * 8, hi[u]);
        continue;
      }
      const bool is_q = h < a.n_q;
      const float inv = 1.0f / sqrtf(ss / static_cast<float>(D) + a.eps);
      const float4* csv = reinterpret_cast<const float4*>(&cs[j][lane * 8]);
      float ol[8], oh[8];
#pragma unroll
      for (int i2 = 0; i2 < 4; ++i2) {
        const float4 c2 = csv[i2];                // (cos, sin) of slots 2*i2 and 2*i2+1
        const float cc[2] = {c2.x, c2.z}, sn[2] = {c2.y, c2.w};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = 2 * i2 + e;
          const float ul = xl[i] * (is_q ? wq_lo[i] : wk_lo[i]);
          const float uh = xh[i] * (is_q ? wq_hi[i] : wk_hi[i]);
          ol[i] = (ul * cc[e] - uh * sn[e]) * inv;
          oh[i] = (uh * cc[e] + ul * sn[e]) * inv;
        }
      }
      __nv_bfloat16* dst = is_q ? static_cast<__nv_bfloat16*>(a.q_out) + (t * a.n_q + h) * D
                                : static_cast<__nv_bfloat16*>(a.k_cache) + (crow * a.n_kv + (h - a.n_q)) * D;
      st_16(dst + lane * 8, f32x8_to_bf16x8(ol));
      st_16(dst + (lane + HALF_VEC) * 8, f32x8_to_bf16x8(oh));
    }
  }
}

// ------------------------------------------------------------- staged path

constexpr int kStagedBlock = 256;
constexpr int kStagedUnroll = 4;

__global__ void __launch_bounds__(kStagedBlock)
qkv_staged_kernel(const __grid_constant__ QkvArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int D = a.d;
  const int vph = D >> 3;                          // 16-byte vectors per head
  const int nqk = a.n_q + a.n_kv;
  const int64_t width = static_cast<int64_t>(nqk + a.n_kv) * D;
  const int qk_vec = nqk * vph;
  const int all_vec = (nqk + a.n_kv) * vph;
  float* u = reinterpret_cast<float*>(smem_raw);                  // [nqk * D]
  float2* cs = reinterpret_cast<float2*>(u + nqk * D);            // [n_slots]
  float* head_ss = reinterpret_cast<float*>(cs + a.n_slots);     // [nqk]
  float* red = head_ss + nqk;                                     // [2 * warps]
  unsigned char* lo_idx = reinterpret_cast<unsigned char*>(red + 2 * (kStagedBlock / 32));  // [n_slots]
  unsigned char* hi_idx = lo_idx + a.n_slots;                                               // [n_slots]

  const int64_t t = blockIdx.x;
  const bool full = a.norm == kQkNormFullWidth;
  bool slot_ok;
  const int64_t crow = cache_row(a, t, slot_ok);
  if (!slot_ok && threadIdx.x == 0) raise_error(a.err, DEV_ERR_SLOT_RANGE);

  for (int p = threadIdx.x; p < a.n_slots; p += blockDim.x) {
    const int pos = a.rope == kRope3D ? a.pos[t * 3 + a.axis[p]] : a.pos[t];
    cs[p] = rope_cos_sin(pos, a.omega_hi[p], a.omega_lo[p]);
    lo_idx[p] = a.lo_idx[p];
    hi_idx[p] = a.hi_idx[p];
  }

  // Phase 1: stream the packed row; V goes straight out, Q/K become raw*w in smem.
  const __nv_bfloat16* row = static_cast<const __nv_bfloat16*>(a.qkv) + t * width;
  float ss_q = 0.f, ss_k = 0.f;
  for (int base = 0; base < all_vec; base += kStagedUnroll * kStagedBlock) {
    uint4 val[kStagedUnroll];
#pragma unroll
    for (int k = 0; k < kStagedUnroll; ++k) {
      const int v = base + k * kStagedBlock + threadIdx.x;
      if (v < all_vec) val[k] = ld_stream(row + v * 8);
    }
#pragma unroll
    for (int k = 0; k < kStagedUnroll; ++k) {
      const int v = base + k * kStagedBlock + threadIdx.x;
      float part = 0.f;
      if (v < qk_vec) {
        const int head = v / vph;
        const int d0 = (v - head * vph) * 8;
        const bool is_q = head < a.n_q;
        const int hl = is_q ? head : head - a.n_q;
        const __nv_bfloat16* wv = static_cast<const __nv_bfloat16*>(is_q ? a.q_w : a.k_w) +
                                  (full ? hl * D + d0 : d0);
        float x[8], w[8];
        bf16x8_to_f32(val[k], x);
        bf16x8_to_f32(ld_cached(wv), w);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          part = fmaf(x[i], x[i], part);
          x[i] *= w[i];
        }
        float4* dst = reinterpret_cast<float4*>(u + head * D + d0);
        dst[0] = make_float4(x[0], x[1], x[2], x[3]);
        dst[1] = make_float4(x[4], x[5], x[6], x[7]);
        if (full) {
          if (is_q) ss_q += part; else ss_k += part;
        }
      } else if (v < all_vec && slot_ok) {
        const int vv = v - qk_vec;
        st_16(static_cast<__nv_bfloat16*>(a.v_cache) + crow * a.n_kv * D + vv * 8, val[k]);
      }
      if (!full) {
        // vph consecutive lanes hold one head in this iteration (block % vph == 0)
        const float hs = group_sum(part, vph);
        if (v < qk_vec && (threadIdx.x & (vph - 1)) == 0) head_ss[v / vph] = hs;
      }
    }
  }
  if (full) {
    ss_q = warp_sum(ss_q);
    ss_k = warp_sum(ss_k);
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
      red[2 * warp] = ss_q;
      red[2 * warp + 1] = ss_k;
    }
  }
  __syncthreads();
  float inv_q = 0.f, inv_k = 0.f;
  if (full) {
    float sq = 0.f, sk = 0.f;
    for (int w = 0; w < kStagedBlock / 32; ++w) {
      sq += red[2 * w];
      sk += red[2 * w + 1];
    }
    inv_q = 1.0f / sqrtf(sq / static_cast<float>(a.n_q * D) + a.eps);
    inv_k = 1.0f / sqrtf(sk / static_cast<float>(a.n_kv * D) + a.eps);
  }

  // Phase 2: rotate every (lo, hi) pair in place and apply the norm scale.
  const int pairs = nqk * a.n_slots;
  for (int i = threadIdx.x; i < pairs; i += blockDim.x) {
    const int head = i / a.n_slots;
    const int p = i - head * a.n_slots;
    const float inv = full ? (head < a.n_q ? inv_q : inv_k)
                           : 1.0f / sqrtf(head_ss[head] / static_cast<float>(D) + a.eps);
    float* hu = u + head * D;
    const int il = lo_idx[p], ih = hi_idx[p];
    const float ul = hu[il];
    const float uh = hu[ih];
    const float2 c = cs[p];
    hu[il] = (ul * c.x - uh * c.y) * inv;
    hu[ih] = (uh * c.x + ul * c.y) * inv;
  }
  __syncthreads();

  // Phase 3: 16-byte bf16 stores of Q and K.
  for (int v = threadIdx.x; v < qk_vec; v += blockDim.x) {
    const int head = v / vph;
    const int d0 = (v - head * vph) * 8;
    const float4* src = reinterpret_cast<const float4*>(u + head * D + d0);
    const float4 f0 = src[0], f1 = src[1];
    const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
    __nv_bfloat16* dst;
    if (head < a.n_q) {
      dst = static_cast<__nv_bfloat16*>(a.q_out) + (t * a.n_q + head) * D + d0;
    } else {
      if (!slot_ok) continue;
      dst = static_cast<__nv_bfloat16*>(a.k_cache) + (crow * a.n_kv + head - a.n_q) * D + d0;
    }
    st_16(dst, f32x8_to_bf16x8(f));
  }
}

size_t staged_smem_bytes(const QkvArgs& a) {
  const size_t nqk = static_cast<size_t>(a.n_q + a.n_kv);
  return nqk * a.d * sizeof(float) + a.n_slots * sizeof(float2) + nqk * sizeof(float) +
         2 * (kStagedBlock / 32) * sizeof(float) + 2 * a.n_slots;
}

}  // namespace

cudaError_t launch_qkv_split_norm_rope(const QkvArgs& a, cudaStream_t stream) {
  if (a.tokens == 0) return cudaSuccess;
  if (a.norm == kQkNormPerHead && a.rope == kRope1D && (a.d == 128 || a.d == 64 || a.d == 256)) {
    const dim3 grid(static_cast<unsigned>((a.tokens + kPairTokens - 1) / kPairTokens)), block(kPairBlock);
    switch (a.d) {
      case 64: qkv_pair_kernel<64><<<grid, block, 0, stream>>>(a); break;
      case 128: qkv_pair_kernel<128><<<grid, block, 0, stream>>>(a); break;
      default: qkv_pair_kernel<256><<<grid, block, 0, stream>>>(a); break;
    }
    return cudaGetLastError();
  }
  const size_t smem = staged_smem_bytes(a);
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(qkv_staged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  qkv_staged_kernel<<<static_cast<unsigned>(a.tokens), kStagedBlock, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gbf
