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
// table in float64 and hands each frequency over as a (hi, lo) binary32 pair;
// each CTA copies it to shared memory once (a per-thread index into the
// kernel-parameter arrays would be serialised across the warp).
//
// Angles: a = pos * omega is formed as a double-binary32 value and reduced to
// [-pi, pi] by Cody and Waite's method (W. J. Cody, W. Waite, "Software Manual
// for the Elementary Functions", 1980) with a two-part 2*pi; the reduced angle
// then goes to the __sincosf intrinsic, whose documented absolute error on
// [-pi, pi] is below 2^-21.4.  The angle error stays near 1e-7 rad at
// position 4095, where a plain binary32 product would be 2.4e-4 rad off.
//
// Two kernels, both streaming (outputs leave from registers, no persistent
// state):
//  * qkv_rot1d_kernel (per-head norm, 1D, head_dim 64/128/256): D/16 lanes
//    own a head; lane l holds the 16-byte vectors l and l + D/16, which contain
//    both members of its 8 rotation pairs (j, j + D/2), so the rotation is done
//    in registers and the head's sum of squares is a shuffle reduction over the
//    head's lanes.  Each thread visits every 8th head of its token (V heads are
//    copied), issuing a batch of loads before any arithmetic, and computes the
//    (cos, sin) of its 8 slots once per token.
//  * qkv_staged_kernel (everything else: full-width norm and/or 3D sections):
//    one CTA per token loads the packed row with 16-byte vectors, writes V
//    straight back out, stages the raw bf16 Q and K in shared memory while the
//    sums of squares are reduced, and after one barrier each thread - owning one
//    rotation slot - weights, rotates and scales that slot's pair in every head
//    it visits and stores both outputs directly.
#include <map>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace gbf {
namespace {

constexpr float kTwoPiHi = 6.28318548202514648438f;      // binary32(2*pi)
constexpr float kTwoPiLo = -1.74845553146951715e-07f;    // 2*pi - kTwoPiHi
constexpr float kInvTwoPi = 0.159154943091895335769f;

// (cos, sin) of pos * (omega_hi + omega_lo).
GBF_DEVICE float2 rope_cos_sin(int pos, float omega_hi, float omega_lo) {
  const float p = static_cast<float>(pos);               // exact below 2^24
  const float a_hi = p * omega_hi;
  const float a_lo = fmaf(p, omega_hi, -a_hi) + p * omega_lo;  // product error + low part
  const float k = rintf(a_hi * kInvTwoPi);
  float r = fmaf(-k, kTwoPiHi, a_hi);
  r = fmaf(-k, kTwoPiLo, r);
  r += a_lo;
  float s, c;
  __sincosf(r, &s, &c);
  return make_float2(c, s);
}

// One rotation slot's table entry in shared memory.
struct __align__(16) SlotEntry {
  float om_hi, om_lo;
  int lo, hi_axis;        // hi_axis = hi | axis << 16
};

GBF_DEVICE void stage_slot_table(const QkvArgs& a, SlotEntry* tab) {
  for (int p = threadIdx.x; p < a.n_slots; p += blockDim.x) {
    SlotEntry e;
    e.om_hi = a.omega_hi[p];
    e.om_lo = a.omega_lo[p];
    e.lo = a.lo_idx[p];
    e.hi_axis = a.hi_idx[p] | (a.axis[p] << 16);
    tab[p] = e;
  }
}

GBF_DEVICE int64_t cache_slot(const QkvArgs& a, int64_t t, bool& ok) {
  const int64_t slot = a.slots ? static_cast<int64_t>(a.slots[t]) : t;
  ok = slot >= 0 && slot < a.cache_rows;
  return slot;
}

// --------------------------------------------------------- per-head, 1D

constexpr int kRotGroups = 8;               // head groups per token
constexpr int kRotBlock = 256;
constexpr int kRotBatch = 3;                // heads whose loads are in flight together

template <int LPH>
__global__ void __launch_bounds__(kRotBlock, 4)
qkv_rot1d_kernel(const __grid_constant__ QkvArgs a) {
  constexpr int D = LPH * 16;
  constexpr int SLOTS = D / 2;
  constexpr int TPT = kRotGroups * LPH;     // threads per token
  constexpr int TOK = kRotBlock / TPT;      // tokens per CTA
  __shared__ SlotEntry tab[SLOTS];
  stage_slot_table(a, tab);
  __syncthreads();

  const int lane = threadIdx.x % LPH;
  const int grp = (threadIdx.x / LPH) % kRotGroups;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * TOK + threadIdx.x / TPT;
  if (t >= a.tokens) return;
  const int heads = a.n_q + 2 * a.n_kv;
  const __nv_bfloat16* row = static_cast<const __nv_bfloat16*>(a.qkv) + t * static_cast<int64_t>(heads) * D;
  bool slot_ok;
  const int64_t crow = cache_slot(a, t, slot_ok);
  if (!slot_ok && threadIdx.x % TPT == 0) raise_error(a.err, DEV_ERR_SLOT_RANGE);

  // (cos, sin) of this lane's slots 8*lane .. 8*lane + 7
  const int pos = a.pos[t];
  float cs[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const SlotEntry e = tab[lane * 8 + i];
    const float2 v = rope_cos_sin(pos, e.om_hi, e.om_lo);
    cs[2 * i] = v.x;
    cs[2 * i + 1] = v.y;
  }

  // Heads grp, grp + 8, ... in batches whose loads are all issued first.  The
  // trip count depends only on grp, which all LPH lanes of a head share.
  for (int h0 = grp; h0 < heads; h0 += kRotBatch * kRotGroups) {
    uint4 lo[kRotBatch], hi[kRotBatch];
#pragma unroll
    for (int u = 0; u < kRotBatch; ++u) {
      const int h = h0 + u * kRotGroups;
      if (h < heads) {
        lo[u] = ld_stream(row + h * D + lane * 8);
        hi[u] = ld_stream(row + h * D + (lane + LPH) * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < kRotBatch; ++u) {
      const int h = h0 + u * kRotGroups;
      if (h >= heads) break;
      if (h >= a.n_q + a.n_kv) {               // V: pass through
        if (slot_ok) {
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.v_cache) +
                               (crow * a.n_kv + (h - a.n_q - a.n_kv)) * D;
          st_16(dst + lane * 8, lo[u]);
          st_16(dst + (lane + LPH) * 8, hi[u]);
        }
        continue;
      }
      float xl[8], xh[8];
      bf16x8_to_f32(lo[u], xl);
      bf16x8_to_f32(hi[u], xh);
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(xl[i], xl[i], fmaf(xh[i], xh[i], ss));
      ss = segment_sum(ss, LPH);               // the head's LPH lanes only
      const bool is_q = h < a.n_q;
      if (!is_q && !slot_ok) continue;
      const float inv = 1.0f / sqrtf(ss / static_cast<float>(D) + a.eps);
      const __nv_bfloat16* w = static_cast<const __nv_bfloat16*>(is_q ? a.q_w : a.k_w);
      float wl[8], wh[8], ol[8], oh[8];
      bf16x8_to_f32(ld_cached(w + lane * 8), wl);
      bf16x8_to_f32(ld_cached(w + (lane + LPH) * 8), wh);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float ul = xl[i] * wl[i], uh = xh[i] * wh[i];
        ol[i] = (ul * cs[2 * i] - uh * cs[2 * i + 1]) * inv;
        oh[i] = (uh * cs[2 * i] + ul * cs[2 * i + 1]) * inv;
      }
      __nv_bfloat16* dst = is_q ? static_cast<__nv_bfloat16*>(a.q_out) + (t * a.n_q + h) * D
                                : static_cast<__nv_bfloat16*>(a.k_cache) + (crow * a.n_kv + (h - a.n_q)) * D;
      st_16(dst + lane * 8, f32x8_to_bf16x8(ol));
      st_16(dst + (lane + LPH) * 8, f32x8_to_bf16x8(oh));
    }
  }
}

// ------------------------------------------------------------- staged path

constexpr int kStagedMaxBlock = 256;
constexpr int kStagedUnroll = 4;

template <bool FULL>
__global__ void __launch_bounds__(kStagedMaxBlock, 4)
qkv_staged_kernel(const __grid_constant__ QkvArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int D = a.d;
  const int n_slots = a.n_slots;
  const int nqk = a.n_q + a.n_kv;
  const int vph = D >> 3;
  const int qk_vec = nqk * vph;
  const int all_vec = (nqk + a.n_kv) * vph;
  const int nthreads = blockDim.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
  __nv_bfloat16* raw = reinterpret_cast<__nv_bfloat16*>(smem);                            // [nqk * D]
  SlotEntry* tab = reinterpret_cast<SlotEntry*>(smem + ((nqk * D * 2 + 15) & ~15));      // [n_slots]
  float* inv_head = reinterpret_cast<float*>(tab + n_slots);                              // [nqk]
  float* red = inv_head + nqk;                                                            // [2 * warps]

  stage_slot_table(a, tab);
  const int64_t t = blockIdx.x;
  bool slot_ok;
  const int64_t crow = cache_slot(a, t, slot_ok);
  if (!slot_ok && tid == 0) raise_error(a.err, DEV_ERR_SLOT_RANGE);

  // Phase 1: stream the row; V goes straight out, raw Q/K to shared memory.
  const __nv_bfloat16* row = static_cast<const __nv_bfloat16*>(a.qkv) + t * static_cast<int64_t>(all_vec) * 8;
  float ss_q = 0.f, ss_k = 0.f;
  for (int base = 0; base < all_vec; base += kStagedUnroll * nthreads) {
    uint4 val[kStagedUnroll];
#pragma unroll
    for (int k = 0; k < kStagedUnroll; ++k) {
      const int v = base + k * nthreads + tid;
      if (v < all_vec) val[k] = ld_stream(row + v * 8);
    }
#pragma unroll
    for (int k = 0; k < kStagedUnroll; ++k) {
      const int v = base + k * nthreads + tid;
      float part = 0.f;
      if (v < qk_vec) {
        *reinterpret_cast<uint4*>(raw + v * 8) = val[k];
        float x[8];
        bf16x8_to_f32(val[k], x);
#pragma unroll
        for (int i = 0; i < 8; ++i) part = fmaf(x[i], x[i], part);
        if (FULL) {
          if (v < a.n_q * vph) ss_q += part; else ss_k += part;
        }
      } else if (v < all_vec && slot_ok) {
        st_16(static_cast<__nv_bfloat16*>(a.v_cache) + crow * a.n_kv * D + (v - qk_vec) * 8, val[k]);
      }
      if (!FULL) {
        // vph consecutive lanes hold one head in this trip (the block is a multiple of vph)
        const float hs = group_sum(part, vph);
        if (v < qk_vec && (tid & (vph - 1)) == 0)
          inv_head[v / vph] = 1.0f / sqrtf(hs / static_cast<float>(D) + a.eps);
      }
    }
  }
  if (FULL) {
    ss_q = warp_sum(ss_q);
    ss_k = warp_sum(ss_k);
    if (lane == 0) {
      red[2 * warp] = ss_q;
      red[2 * warp + 1] = ss_k;
    }
  }
  __syncthreads();
  float inv_q = 0.f, inv_k = 0.f;
  if (FULL) {                                   // each warp reduces the warps' partials
    float sq = lane < nwarps ? red[2 * lane] : 0.f;
    float sk = lane < nwarps ? red[2 * lane + 1] : 0.f;
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    inv_q = 1.0f / sqrtf(sq / static_cast<float>(a.n_q * D) + a.eps);
    inv_k = 1.0f / sqrtf(sk / static_cast<float>(a.n_kv * D) + a.eps);
  }

  // Phase 2: this thread's slot in every head it visits.
  const int p = tid % n_slots;
  const int grp = tid / n_slots;
  const int ngrp = nthreads / n_slots;
  const SlotEntry e = tab[p];
  const int lo = e.lo, hi = e.hi_axis & 0xFFFF, axis = e.hi_axis >> 16;
  const int pos = a.rope == kRope3D ? a.pos[t * 3 + axis] : a.pos[t];
  const float2 c = rope_cos_sin(pos, e.om_hi, e.om_lo);
  const uint16_t* qw = static_cast<const uint16_t*>(a.q_w);
  const uint16_t* kw = static_cast<const uint16_t*>(a.k_w);
  __nv_bfloat16* q_out = static_cast<__nv_bfloat16*>(a.q_out) + t * a.n_q * D;
  __nv_bfloat16* k_out = static_cast<__nv_bfloat16*>(a.k_cache) + crow * a.n_kv * D;
  for (int h = grp; h < nqk; h += ngrp) {
    const bool is_q = h < a.n_q;
    const int hl = is_q ? h : h - a.n_q;
    if (!is_q && !slot_ok) continue;
    const uint16_t* w = (is_q ? qw : kw) + (FULL ? hl * D : 0);
    const float xl = __bfloat162float(raw[h * D + lo]);
    const float xh = __bfloat162float(raw[h * D + hi]);
    const float ul = xl * bf16_bits_to_f32(w[lo]);
    const float uh = xh * bf16_bits_to_f32(w[hi]);
    const float inv = FULL ? (is_q ? inv_q : inv_k) : inv_head[h];
    __nv_bfloat16* dst = (is_q ? q_out : k_out) + hl * D;
    dst[lo] = __float2bfloat16_rn((ul * c.x - uh * c.y) * inv);
    dst[hi] = __float2bfloat16_rn((uh * c.x + ul * c.y) * inv);
  }
}

size_t staged_smem_bytes(const QkvArgs& a, int threads) {
  const size_t nqk = static_cast<size_t>(a.n_q + a.n_kv);
  return ((nqk * a.d * 2 + 15) & ~size_t(15)) + a.n_slots * sizeof(SlotEntry) + nqk * sizeof(float) +
         2 * (threads / 32) * sizeof(float);
}

// The dynamic shared memory limit of `fn` is raised once to the device's
// opt-in maximum (the attribute is an upper bound, so it never has to shrink).
template <typename F>
cudaError_t raise_smem_limit(F fn) {
  static std::mutex mu;
  static std::map<const void*, bool> raised;
  std::lock_guard<std::mutex> lock(mu);
  const void* key = reinterpret_cast<const void*>(fn);
  if (raised[key]) return cudaSuccess;
  int dev = 0, optin = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e == cudaSuccess) raised[key] = true;
  return e;
}

}  // namespace

cudaError_t launch_qkv_split_norm_rope(const QkvArgs& a, cudaStream_t stream) {
  if (a.tokens == 0) return cudaSuccess;
  if (a.norm == kQkNormPerHead && a.rope == kRope1D && (a.d == 64 || a.d == 128 || a.d == 256)) {
    const int lph = a.d / 16;
    const int tok_per_cta = kRotBlock / (kRotGroups * lph);
    const unsigned grid = static_cast<unsigned>((a.tokens + tok_per_cta - 1) / tok_per_cta);
    switch (a.d) {
      case 64: qkv_rot1d_kernel<4><<<grid, kRotBlock, 0, stream>>>(a); break;
      case 128: qkv_rot1d_kernel<8><<<grid, kRotBlock, 0, stream>>>(a); break;
      default: qkv_rot1d_kernel<16><<<grid, kRotBlock, 0, stream>>>(a); break;
    }
    return cudaGetLastError();
  }
  // Block: the largest multiple of lcm(D/2, 32) that is <= kStagedMaxBlock.
  int l = a.n_slots;
  while (l % 32) l += a.n_slots;
  const int threads = (kStagedMaxBlock / l) * l;
  if (threads < 32) return cudaErrorInvalidConfiguration;
  const size_t smem = staged_smem_bytes(a, threads);
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  const bool full = a.norm == kQkNormFullWidth;
  cudaError_t e = full ? raise_smem_limit(qkv_staged_kernel<true>) : raise_smem_limit(qkv_staged_kernel<false>);
  if (e != cudaSuccess) return e;
  if (full)
    qkv_staged_kernel<true><<<static_cast<unsigned>(a.tokens), threads, smem, stream>>>(a);
  else
    qkv_staged_kernel<false><<<static_cast<unsigned>(a.tokens), threads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gbf
