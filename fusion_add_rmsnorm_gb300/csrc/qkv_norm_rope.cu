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
// Two kernels:
//  * qkv_rot1d_kernel (per-head RMSNorm or LayerNorm, 1D, head_dim 64/128/
//    256): D/16 lanes own a head; lane l holds the 16-byte vectors l and
//    l + D/16, which contain both members of its 8 rotation pairs (j, j + D/2),
//    so the rotation is done in registers and the head's statistics are a
//    shuffle reduction over the head's lanes.  Each thread visits every G-th
//    head of its token (G head groups, a power of two: a token's G * D/16
//    threads at most 128 in streaming launches, up to 512 with one head per
//    group in launch-bound ones; V heads are copied), issuing a batch of loads
//    before any arithmetic, and the token's (cos, sin) are computed once per
//    token into a shared table.
//  * qkv_staged_kernel (everything else: full-width norm and/or 3D sections,
//    where a rotation pair need not sit in one 16-byte vector): a persistent
//    CTA streams its tokens' packed rows through a ring of shared-memory
//    buffers filled by bulk copies.  Per token, thread 0 sends V out with one
//    bulk shared-to-global copy while phase 1 writes x * w of Q and K to
//    shared memory as float32 and reduces the sums of squares; after one
//    barrier each thread takes its own 16-byte vectors
//    again, reads the 8 rotation partners of their elements, and stores the
//    rotated, normalised vector with one 16-byte store.
#include <map>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tma.cuh"

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

// --------------------------------------------------------- per-head, 1D

// Head groups per token: a template parameter G of the per-head kernels,
// chosen at launch so a thread has at most kRotBatch heads (one batch of
// loads) where the token's 256 threads allow it.
constexpr int kRotBlock = 256;
constexpr int kRotBatch = 3;                // heads whose loads are in flight together

// Loads of one batch of a thread's heads, h0, h0 + G, h0 + 2G, of a token row.
template <int LPH, int G>
GBF_DEVICE void rot1d_load(const __nv_bfloat16* row, int h0, int heads, int lane, uint4 (&lo)[kRotBatch],
                           uint4 (&hi)[kRotBatch]) {
  constexpr int D = LPH * 16;
#pragma unroll
  for (int u = 0; u < kRotBatch; ++u) {
    const int h = h0 + u * G;
    if (h < heads) {
      lo[u] = ld_stream(row + h * D + lane * 8);
      hi[u] = ld_stream(row + h * D + (lane + LPH) * 8);
    }
  }
}

// (cos, sin) table of a CTA's tokens: float4 [tok][i][lane] holds (cos, sin)
// of slots 8 lane + 2i and 8 lane + 2i + 1, so the LPH lanes of a head read
// consecutive float4s.
template <int LPH>
GBF_DEVICE void rot1d_cs_put(float4* cs4, int tc, int p, float2 cs) {
  float* dst = reinterpret_cast<float*>(&cs4[(tc * 4 + ((p & 7) >> 1)) * LPH + (p >> 3)]) + 2 * (p & 1);
  dst[0] = cs.x;
  dst[1] = cs.y;
}

// Norm, rotation and stores of one batch of token t's heads (V heads are
// copied); c2/s2 are the (cos, sin) of this lane's slots 8 lane .. 8 lane + 7
// as pairs (2i, 2i + 1).
template <int LPH, bool LN, int G>
GBF_DEVICE void rot1d_batch(const QkvArgs& a, int64_t t, int h0, int lane, bool slot_ok, int64_t crow,
                            const uint4 (&lo)[kRotBatch], const uint4 (&hi)[kRotBatch], const float2 (&c2)[4],
                            const float2 (&s2)[4]) {
  constexpr int D = LPH * 16;
  const int heads = a.n_q + 2 * a.n_kv;
  // last head of the batch first: V heads come last in the row, and copying
  // them out first frees their registers for the norm work
#pragma unroll
  for (int uu = 0; uu < kRotBatch; ++uu) {
    const int u = kRotBatch - 1 - uu;
    const int h = h0 + u * G;
    if (h >= heads) continue;
    if (h >= a.n_q + a.n_kv) {               // V: pass through
      if (slot_ok) {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.v_cache) +
                             (crow * a.n_kv + (h - a.n_q - a.n_kv)) * D;
        st_16(dst + lane * 8, lo[u]);
        st_16(dst + (lane + LPH) * 8, hi[u]);
      }
      continue;
    }
    const uint32_t xl[4] = {lo[u].x, lo[u].y, lo[u].z, lo[u].w};
    const uint32_t xh[4] = {hi[u].x, hi[u].y, hi[u].z, hi[u].w};
    uint32_t ol[4], oh[4];
    if (!LN) {
      // RMSNorm: o = rotate(x * w) * inv
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        s0 = fma_bf16_lo(xl[i], xl[i], s0);
        s1 = fma_bf16_hi(xl[i], xl[i], s1);
        s0 = fma_bf16_lo(xh[i], xh[i], s0);
        s1 = fma_bf16_hi(xh[i], xh[i], s1);
      }
      const float ss = segment_sum(s0 + s1, LPH);   // the head's LPH lanes only
      const bool is_q = h < a.n_q;
      if (!is_q && !slot_ok) continue;
      const float inv = rsqrtf(ss / static_cast<float>(D) + a.eps);
      const __nv_bfloat16* w = static_cast<const __nv_bfloat16*>(is_q ? a.q_w : a.k_w);
      const uint4 wlv = ld_cached(w + lane * 8), whv = ld_cached(w + (lane + LPH) * 8);
      const uint32_t wl[4] = {wlv.x, wlv.y, wlv.z, wlv.w};
      const uint32_t wh[4] = {whv.x, whv.y, whv.z, whv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // pair (8 lane + 2i + j, the same + D/2) for j = 0, 1 in the two float2 lanes
        const float2 ul = make_float2(fma_bf16_lo(xl[i], wl[i], 0.f), fma_bf16_hi(xl[i], wl[i], 0.f));
        const float2 uh = make_float2(fma_bf16_lo(xh[i], wh[i], 0.f), fma_bf16_hi(xh[i], wh[i], 0.f));
        float2 rl, rh;
        rl.x = fmaf(ul.x, c2[i].x, -(s2[i].x * uh.x)) * inv;
        rl.y = fmaf(ul.y, c2[i].y, -(s2[i].y * uh.y)) * inv;
        rh.x = fmaf(uh.x, c2[i].x, s2[i].x * ul.x) * inv;
        rh.y = fmaf(uh.y, c2[i].y, s2[i].y * ul.y) * inv;
        ol[i] = f32x2_to_bf16x2(rl.x, rl.y);
        oh[i] = f32x2_to_bf16x2(rh.x, rh.y);
      }
    } else {
      // LayerNorm: each lane takes the mean and the centred sum of
      // squares of its own 16 values (two passes over registers), and
      // the head's LPH lanes merge them in one shuffle chain by the
      // pairwise update of Chan, Golub and LeVeque ("Algorithms for
      // computing the sample variance", 1983) for equal counts:
      // mean = (ma + mb) / 2, M2 = M2a + M2b + (mb - ma)^2 n / 2.
      // Then u = (x - mean) * inv * w + b, o = rotate(u).  The sums and
      // the centring use the bf16-input FMA (x * 1 + acc, x * 1 - mean).
      constexpr uint32_t kOnes = 0x3F803F80u;     // bf16x2 (1, 1)
      float m0 = 0.f, m1 = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        m0 = fma_bf16_lo(xl[i], kOnes, m0);
        m1 = fma_bf16_hi(xl[i], kOnes, m1);
        m0 = fma_bf16_lo(xh[i], kOnes, m0);
        m1 = fma_bf16_hi(xh[i], kOnes, m1);
      }
      float mean = (m0 + m1) * (1.0f / 16.0f);
      float v0 = 0.f, v1 = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float c0 = fma_bf16_lo(xl[i], kOnes, -mean), c1 = fma_bf16_hi(xl[i], kOnes, -mean);
        const float c2h = fma_bf16_lo(xh[i], kOnes, -mean), c3 = fma_bf16_hi(xh[i], kOnes, -mean);
        v0 = fmaf(c0, c0, fmaf(c2h, c2h, v0));
        v1 = fmaf(c1, c1, fmaf(c3, c3, v1));
      }
      float m2 = v0 + v1;
      {
        const unsigned seg = LPH >= 32 ? 0xffffffffu
                                       : (((1u << LPH) - 1u) << ((threadIdx.x & 31u) & ~static_cast<unsigned>(LPH - 1)));
        float half_n = 8.0f;                      // n / 2 for the n = 16 values of one lane
#pragma unroll
        for (int o = 1; o < LPH; o <<= 1) {
          const float mo = __shfl_xor_sync(seg, mean, o);
          const float m2o = __shfl_xor_sync(seg, m2, o);
          const float d = mo - mean;
          m2 = (m2 + m2o) + d * d * half_n;     // the same on both lanes of the exchange
          mean = 0.5f * (mean + mo);
          half_n *= 2.0f;
        }
      }
      // centred values are formed again in the output pass (one FMA each)
      // rather than held in registers across it
      const float var = m2 * (1.0f / static_cast<float>(D));
      const bool is_q = h < a.n_q;
      if (!is_q && !slot_ok) continue;
      const float inv = rsqrtf(var + a.eps);
      const __nv_bfloat16* w = static_cast<const __nv_bfloat16*>(is_q ? a.q_w : a.k_w);
      const __nv_bfloat16* bb = static_cast<const __nv_bfloat16*>(is_q ? a.q_b : a.k_b);
      const uint4 wlv = ld_cached(w + lane * 8), whv = ld_cached(w + (lane + LPH) * 8);
      const uint4 blv = bb ? ld_cached(bb + lane * 8) : make_uint4(0, 0, 0, 0);
      const uint4 bhv = bb ? ld_cached(bb + (lane + LPH) * 8) : make_uint4(0, 0, 0, 0);
      const uint32_t wl[4] = {wlv.x, wlv.y, wlv.z, wlv.w}, wh[4] = {whv.x, whv.y, whv.z, whv.w};
      const uint32_t bl[4] = {blv.x, blv.y, blv.z, blv.w}, bh[4] = {bhv.x, bhv.y, bhv.z, bhv.w};
      // (lo, hi) halves of a packed bf16 pair as two floats
      auto pair = [](uint32_t v) { return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u)); };
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 inv2 = make_float2(inv, inv);
        const float2 cl2 = make_float2(fma_bf16_lo(xl[i], kOnes, -mean), fma_bf16_hi(xl[i], kOnes, -mean));
        const float2 ch2 = make_float2(fma_bf16_lo(xh[i], kOnes, -mean), fma_bf16_hi(xh[i], kOnes, -mean));
        const float2 ul = __ffma2_rn(__fmul2_rn(cl2, inv2), pair(wl[i]), pair(bl[i]));
        const float2 uh = __ffma2_rn(__fmul2_rn(ch2, inv2), pair(wh[i]), pair(bh[i]));
        const float2 rl = __ffma2_rn(ul, c2[i], __fmul2_rn(make_float2(-s2[i].x, -s2[i].y), uh));
        const float2 rh = __ffma2_rn(uh, c2[i], __fmul2_rn(s2[i], ul));
        ol[i] = f32x2_to_bf16x2(rl.x, rl.y);
        oh[i] = f32x2_to_bf16x2(rh.x, rh.y);
      }
    }
    const bool is_q = h < a.n_q;
    __nv_bfloat16* dst = is_q ? static_cast<__nv_bfloat16*>(a.q_out) + (t * a.n_q + h) * D
                              : static_cast<__nv_bfloat16*>(a.k_cache) + (crow * a.n_kv + (h - a.n_q)) * D;
    st_16(dst + lane * 8, make_uint4(ol[0], ol[1], ol[2], ol[3]));
    st_16(dst + (lane + LPH) * 8, make_uint4(oh[0], oh[1], oh[2], oh[3]));
  }
}

template <int LPH>
GBF_DEVICE void rot1d_cs_read(const float4* cs_tok, int lane, float2 (&c2)[4], float2 (&s2)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 q = cs_tok[i * LPH + lane];
    c2[i] = make_float2(q.x, q.z);
    s2[i] = make_float2(q.y, q.w);
  }
}

// Threads per CTA of the per-head kernel: the smallest of 128, 256 and 512
// that holds a token's G * LPH threads.  For streaming launches the smaller
// CTA ends sooner (its share of the bandwidth moves fewer tokens), so the
// tail of a launch, where the last CTAs run alone, is shorter; the registers
// per thread are the same either way.
constexpr int rot1d_block(int g, int lph) { return g * lph <= 128 ? 128 : g * lph <= 256 ? kRotBlock : 512; }

// One CTA per TOK tokens; a thread with more than one batch of heads takes
// them in turn.  The first batch is requested before the (cos, sin) table.
template <int LPH, bool LN, int G, int BLOCK>
__global__ void __launch_bounds__(BLOCK, (LN ? 3 : 4) * kRotBlock / BLOCK)
qkv_rot1d_kernel(const __grid_constant__ QkvArgs a) {
  constexpr int D = LPH * 16;
  constexpr int SLOTS = D / 2;
  constexpr int TPT = G * LPH;              // threads per token
  constexpr int TOK = BLOCK / TPT;          // tokens per CTA
  static_assert(TOK >= 1 && TOK * SLOTS <= BLOCK, "a token fits the CTA, at most one (cos, sin) per thread");
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x % LPH;
  const int grp = (threadIdx.x / LPH) % G;
  const int tok = threadIdx.x / TPT;
  const int heads = a.n_q + 2 * a.n_kv;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * TOK + tok;
  const bool live = t < a.tokens;
  const __nv_bfloat16* row = static_cast<const __nv_bfloat16*>(a.qkv) + t * static_cast<int64_t>(heads) * D;
  uint4 lo[kRotBatch], hi[kRotBatch];
  if (live) rot1d_load<LPH, G>(row, grp, heads, lane, lo, hi);
  // the token's cache row (slot mapping) is requested with its data, not
  // after the table
  const int32_t slot_in = live && a.slots ? a.slots[t] : 0;

  __shared__ float4 cs4[TOK * 4 * LPH];
  {
    const int tc = threadIdx.x / SLOTS, p = threadIdx.x % SLOTS;      // slot p of token tc
    const int64_t tcs = static_cast<int64_t>(blockIdx.x) * TOK + tc;
    if (tc < TOK && tcs < a.tokens) rot1d_cs_put<LPH>(cs4, tc, p, rope_cos_sin(a.pos[tcs], a.omega_hi[p], a.omega_lo[p]));
  }
  __syncthreads();
  if (!live) return;
  const int64_t crow = a.slots ? static_cast<int64_t>(slot_in) : t;
  const bool slot_ok = crow >= 0 && crow < a.cache_rows;
  if (!slot_ok && threadIdx.x % TPT == 0) raise_error(a.err, DEV_ERR_SLOT_RANGE);
  float2 c2[4], s2[4];
  rot1d_cs_read<LPH>(cs4 + tok * 4 * LPH, lane, c2, s2);
  // The trip count depends only on grp, which all LPH lanes of a head share.
  for (int h0 = grp; h0 < heads; h0 += kRotBatch * G) {
    if (h0 != grp) rot1d_load<LPH, G>(row, h0, heads, lane, lo, hi);
    rot1d_batch<LPH, LN, G>(a, t, h0, lane, slot_ok, crow, lo, hi, c2, s2);
  }
}

// ------------------------------------------------------------- staged path
//
// A CTA handles the tokens blockIdx.x, blockIdx.x + gridDim.x, ...  Thread 0
// keeps a ring of `nb` shared-memory row buffers filled with bulk copies of the
// packed rows of the CTA's next tokens (completion counted on one mbarrier per
// buffer), so the row of the next token is in flight while the current one is
// computed.  Worker thread tid < active owns the 16-byte vectors
// v = tid + k * active of the row.  active is a multiple of head_dim / 8, so all
// of a thread's vectors sit at the same position P0 = 8 * (tid % (head_dim / 8))
// inside their heads: the thread's rotation partners, (cos, sin) values and
// shared-memory offsets are fixed for the whole token.

constexpr int kStagedBlock = 256;
constexpr int kStagedUnroll = 4;
constexpr uint32_t kBulkChunk = 32768;      // bytes per bulk copy instruction

// Word offset in shared memory of element L of a token's staged Q|K block.  The
// two 16-byte halves of vector L / 8 trade places when bit 2 (and, if swz2 is
// set, bit 4) of the vector index is odd, which spreads a quarter warp's
// 16-byte accesses and the warp's partner reads over the 32 banks.
GBF_DEVICE int staged_word(int L, int swz2) {
  const int v = L >> 3;
  const int s = ((v >> 2) ^ ((v >> 4) & swz2)) & 1;
  return L ^ (s << 2);
}

// Index in the (cos, sin) table of head position P: the pairs of positions
// 8g + 2i and 8g + 2i + 1 share the float4 i * vph + g, so the lanes that own
// consecutive 8-element groups g read consecutive float4s.
GBF_DEVICE int cs_slot(int P, int vph) { return 2 * (((P & 7) >> 1) * vph + (P >> 3)) + (P & 1); }

// Thread 0: copy one packed row into a ring buffer, completion on `bar`.
GBF_DEVICE void load_row(uint8_t* dst, const uint8_t* src, uint32_t bytes, uint64_t* bar) {
  mbar_arrive_expect_tx(bar, bytes);
  for (uint32_t o = 0; o < bytes; o += kBulkChunk) {
    const uint32_t n = bytes - o < kBulkChunk ? bytes - o : kBulkChunk;
    bulk_load(dst + o, src + o, n, bar);
  }
}

struct StagedLayout {
  size_t raw_stride, u_off, tab_off, cs_off, part_off, inv_off, red_off, bar_off, total;
};

GBF_HOST_DEVICE StagedLayout staged_layout(int n_q, int n_kv, int d, int n_slots, int nwarps, int nb) {
  StagedLayout L;
  const size_t nqk = static_cast<size_t>(n_q + n_kv);
  const size_t row = (nqk + n_kv) * d * 2;
  L.raw_stride = (row + 127) & ~size_t(127);
  L.u_off = nb * L.raw_stride;
  L.tab_off = L.u_off + nqk * d * sizeof(float);
  L.cs_off = L.tab_off + n_slots * sizeof(SlotEntry);
  L.part_off = L.cs_off + d * sizeof(float2);
  L.inv_off = L.part_off + d * sizeof(int);
  L.red_off = L.inv_off + nqk * sizeof(float);
  L.bar_off = (L.red_off + 2 * nwarps * sizeof(float) + 7) & ~size_t(7);
  L.total = L.bar_off + nb * sizeof(uint64_t) + sizeof(int);
  return L;
}

// Phase 1 work on one Q|K vector v: x * w to shared memory (float32), the
// sum of squares to ss_q / ss_k (full width) or, per head, the head's inverse
// RMS to inv_head (the head's vph lanes run this together).
template <bool FULL>
GBF_DEVICE void stage_vector(const QkvArgs& a, int v, uint4 xv, uint4 wv, uint32_t u_dst, int own_lo_b,
                             int own_hi_b, int q_vec, int vph, int lg_vph, float* inv_head, float& ss_q,
                             float& ss_k) {
  const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
  const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
  float xw[8], p0 = 0.f, p1 = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    xw[2 * i] = fma_bf16_lo(xs[i], ws[i], 0.f);
    xw[2 * i + 1] = fma_bf16_hi(xs[i], ws[i], 0.f);
    p0 = fma_bf16_lo(xs[i], xs[i], p0);
    p1 = fma_bf16_hi(xs[i], xs[i], p1);
  }
  sts128f(u_dst + own_lo_b, xw[0], xw[1], xw[2], xw[3]);
  sts128f(u_dst + own_hi_b, xw[4], xw[5], xw[6], xw[7]);
  const float part = p0 + p1;
  if (FULL) {
    if (v < q_vec) ss_q += part; else ss_k += part;
  } else {
    const float hs = segment_sum(part, vph);
    if ((threadIdx.x & (vph - 1)) == 0) inv_head[v >> lg_vph] = rsqrtf(hs / static_cast<float>(a.d) + a.eps);
  }
}

// Phase 2 work on one Q|K vector: rotate, normalise, one 16-byte store.
template <bool FULL>
GBF_DEVICE void rotate_vector(int v, float4 o0, float4 o1, const float pv[8], const float2 c2[4],
                              const float2 s2[4], float inv, __nv_bfloat16* q_dst, __nv_bfloat16* k_dst, int q_vec,
                              bool slot_ok) {
  const float2 own[4] = {make_float2(o0.x, o0.y), make_float2(o0.z, o0.w), make_float2(o1.x, o1.y),
                         make_float2(o1.z, o1.w)};
  const float2 inv2 = make_float2(inv, inv);
  uint32_t packed[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p2 = make_float2(pv[2 * i], pv[2 * i + 1]);
    const float2 o = __fmul2_rn(__ffma2_rn(own[i], c2[i], __fmul2_rn(s2[i], p2)), inv2);
    packed[i] = f32x2_to_bf16x2(o.x, o.y);
  }
  const uint4 o16 = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  if (v < q_vec)
    st_16(q_dst + v * 8, o16);
  else if (slot_ok)
    st_16(k_dst + (v - q_vec) * 8, o16);
}

template <bool FULL>
__global__ void __launch_bounds__(kStagedBlock, 3)
qkv_staged_kernel(const __grid_constant__ QkvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_wait();
  pdl_launch_dependents();
  const int D = a.d;
  const int vph = D >> 3;
  const int n_slots = a.n_slots;
  const int nqk = a.n_q + a.n_kv;
  const int q_vec = a.n_q * vph;
  const int qk_vec = nqk * vph;
  const int all_vec = (nqk + a.n_kv) * vph;
  const int active = a.active;
  const int swz2 = a.swz2;
  const int nb = a.nb;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const bool worker = tid < active;
  const StagedLayout L = staged_layout(a.n_q, a.n_kv, D, n_slots, nwarps, nb);
  const uint32_t row_bytes = static_cast<uint32_t>(all_vec) * 16u;
  const uint32_t smem32 = smem_u32(smem);
  const uint32_t u32 = smem32 + static_cast<uint32_t>(L.u_off);          // [qk_vec * 8] x * w
  SlotEntry* tab = reinterpret_cast<SlotEntry*>(smem + L.tab_off);        // [n_slots]
  float2* cs_pos = reinterpret_cast<float2*>(smem + L.cs_off);            // [D] (cos, -+sin), cs_slot order
  int* part_pos = reinterpret_cast<int*>(smem + L.part_off);              // [D] rotation partner
  float* inv_head = reinterpret_cast<float*>(smem + L.inv_off);           // [nqk]
  float* red = reinterpret_cast<float*>(smem + L.red_off);                // [2 * warps]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);         // [nb]
  int* abort_flag = reinterpret_cast<int*>(full + nb);
  const uint8_t* qkv = static_cast<const uint8_t*>(a.qkv);

  for (int p = tid; p < n_slots; p += blockDim.x) {
    SlotEntry e;
    e.om_hi = a.omega_hi[p];
    e.om_lo = a.omega_lo[p];
    e.lo = a.lo_idx[p];
    e.hi_axis = a.hi_idx[p] | (a.axis[p] << 16);
    tab[p] = e;
    part_pos[a.lo_idx[p]] = a.hi_idx[p];
    part_pos[a.hi_idx[p]] = a.lo_idx[p];
  }
  if (tid == 0) {
    for (int b = 0; b < nb; ++b) mbar_init(&full[b], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int b = 0; b < nb; ++b) {
      const int64_t tb = blockIdx.x + static_cast<int64_t>(b) * gridDim.x;
      if (tb < a.tokens) load_row(smem + b * L.raw_stride, qkv + tb * row_bytes, row_bytes, &full[b]);
    }
  }

  const int P0 = worker ? 8 * (tid % vph) : 0;
  const int lg_vph = __ffs(vph) - 1;          // per-head norm: vph is a power of two
  // Byte offsets, from the start of vector v in `u`, of the thread's own
  // halves and of its 8 partners; the same for every v = tid + k * active.
  const int vref = tid + 64 * active;
  const int own_lo_b = 4 * (staged_word(8 * vref, swz2) - 8 * vref);
  const int own_hi_b = 16 - own_lo_b;
  int off_b[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) off_b[e] = 4 * (staged_word(8 * vref + part_pos[P0 + e] - P0, swz2) - 8 * vref);

  const __nv_bfloat16* qw = static_cast<const __nv_bfloat16*>(a.q_w);
  const __nv_bfloat16* kw = static_cast<const __nv_bfloat16*>(a.k_w);
  // weight vector of Q|K vector v
  auto wptr = [&](int v) -> const __nv_bfloat16* {
    return FULL ? (v < q_vec ? qw + v * 8 : kw + (v - q_vec) * 8) : (v < q_vec ? qw : kw) + P0;
  };
  // Thread p < n_slots owns rotation slot p (the launcher guarantees
  // blockDim.x >= n_slots).  Its grid coordinate and every thread's cache row
  // are fetched one token ahead, off the critical path.
  const bool cs_thread = tid < n_slots;
  const SlotEntry my_slot = tab[cs_thread ? tid : 0];
  auto pos_of = [&](int64_t tt) { return a.rope == kRope3D ? a.pos[tt * 3 + (my_slot.hi_axis >> 16)] : a.pos[tt]; };
  auto row_of = [&](int64_t tt) { return a.slots ? static_cast<int64_t>(a.slots[tt]) : tt; };
  int pos_next = cs_thread ? pos_of(blockIdx.x) : 0;
  int64_t crow_next = row_of(blockIdx.x);
  int b = 0;                      // ring buffer of the current token
  uint32_t phase_bits = 0;        // bit j: parity of the next completion of buffer j
  for (int64_t t = blockIdx.x; t < a.tokens; t += gridDim.x) {
    const uint32_t raw32 = smem32 + static_cast<uint32_t>(b * L.raw_stride);
    const int pos = pos_next;
    const int64_t crow = crow_next;
    if (t + gridDim.x < a.tokens) {
      if (cs_thread) pos_next = pos_of(t + gridDim.x);
      crow_next = row_of(t + gridDim.x);
    }
    const bool slot_ok = crow >= 0 && crow < a.cache_rows;
    if (!slot_ok && tid == 0) raise_error(a.err, DEV_ERR_SLOT_RANGE);
    if (cs_thread) {
      const float2 cs = rope_cos_sin(pos, my_slot.om_hi, my_slot.om_lo);
      cs_pos[cs_slot(my_slot.lo, vph)] = make_float2(cs.x, -cs.y);
      cs_pos[cs_slot(my_slot.hi_axis & 0xFFFF, vph)] = cs;
    }

    // Phase 1: x * w of Q/K to `u`; V (contiguous in the row and in its cache
    // row) leaves the ring buffer by one bulk store issued by thread 0.
    const bool ok = mbar_wait_warp(&full[b], (phase_bits >> b) & 1u, abort_flag, a.err);
    if (ok && tid == 0 && slot_ok) {
      uint8_t* v_dst = reinterpret_cast<uint8_t*>(static_cast<__nv_bfloat16*>(a.v_cache) + crow * a.n_kv * D);
      const uint8_t* v_src = smem + b * L.raw_stride + static_cast<size_t>(qk_vec) * 16;
      const uint32_t v_bytes = static_cast<uint32_t>(a.n_kv * D * 2);
      for (uint32_t off = 0; off < v_bytes; off += kBulkChunk)
        bulk_store(v_dst + off, v_src + off, v_bytes - off < kBulkChunk ? v_bytes - off : kBulkChunk);
      bulk_commit();
    }
    float ss_q = 0.f, ss_k = 0.f;
    if (ok && worker) {
      int v = tid;
      for (; v + (kStagedUnroll - 1) * active < qk_vec; v += kStagedUnroll * active) {
        uint4 xv[kStagedUnroll], wv[kStagedUnroll];
#pragma unroll
        for (int k = 0; k < kStagedUnroll; ++k) {
          xv[k] = lds128(raw32 + (v + k * active) * 16);
          wv[k] = ld_cached(wptr(v + k * active));
        }
#pragma unroll
        for (int k = 0; k < kStagedUnroll; ++k) {
          const int vk = v + k * active;
          stage_vector<FULL>(a, vk, xv[k], wv[k], u32 + vk * 32, own_lo_b, own_hi_b, q_vec, vph, lg_vph, inv_head,
                             ss_q, ss_k);
        }
      }
      for (; v < qk_vec; v += active)
        stage_vector<FULL>(a, v, lds128(raw32 + v * 16), ld_cached(wptr(v)), u32 + v * 32, own_lo_b, own_hi_b, q_vec,
                           vph, lg_vph, inv_head, ss_q, ss_k);
    }
    if (FULL) {
      ss_q = warp_sum(ss_q);
      ss_k = warp_sum(ss_k);
      if (lane == 0) {
        red[2 * warp] = ss_q;
        red[2 * warp + 1] = ss_k;
      }
    }
    if (__syncthreads_or(!ok)) {
      // A row never arrived: wait (bounded) for the copies still in flight, then leave.
      if (tid == 0) {
        bulk_wait_all();
        int give_up = 0;
        for (int j = 0, bj = b; j < nb; ++j, bj = bj + 1 == nb ? 0 : bj + 1) {
          if (t + static_cast<int64_t>(j) * gridDim.x >= a.tokens) break;
          mbar_wait(&full[bj], (phase_bits >> bj) & 1u, &give_up, a.err);
        }
      }
      return;
    }
    // The row buffer is consumed: refill it with the token nb turns ahead.
    if (tid == 0) {
      const int64_t tn = t + static_cast<int64_t>(nb) * gridDim.x;
      if (tn < a.tokens) {
        bulk_wait_read_all();       // the V store has read its part of the buffer
        fence_proxy_async_smem();   // the barrier ordered every thread's reads of the buffer before this
        load_row(smem + b * L.raw_stride, qkv + tn * row_bytes, row_bytes, &full[b]);
      }
    }
    phase_bits ^= 1u << b;
    b = b + 1 == nb ? 0 : b + 1;

    // Phase 2: o = (u * cos -+ u_partner * sin) * inv, 16-byte stores from registers.
    float inv_q = 0.f, inv_k = 0.f;
    if (FULL) {                                  // every warp reduces the warps' partials
      float sq = lane < nwarps ? red[2 * lane] : 0.f;
      float sk = lane < nwarps ? red[2 * lane + 1] : 0.f;
      sq = warp_sum(sq);
      sk = warp_sum(sk);
      inv_q = rsqrtf(sq / static_cast<float>(a.n_q * D) + a.eps);
      inv_k = rsqrtf(sk / static_cast<float>(a.n_kv * D) + a.eps);
    }
    if (worker) {
      float2 c2[4], s2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 q = reinterpret_cast<const float4*>(cs_pos)[i * vph + (P0 >> 3)];
        c2[i] = make_float2(q.x, q.z);
        s2[i] = make_float2(q.y, q.w);
      }
      __nv_bfloat16* q_dst = static_cast<__nv_bfloat16*>(a.q_out) + t * a.n_q * D;
      __nv_bfloat16* k_dst = static_cast<__nv_bfloat16*>(a.k_cache) + crow * a.n_kv * D;
      auto inv_of = [&](int v) { return FULL ? (v < q_vec ? inv_q : inv_k) : inv_head[v >> lg_vph]; };
      int v = tid;
      for (; v + active < qk_vec; v += 2 * active) {
        float4 o[2][2];
        float pv[2][8];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t a0 = u32 + (v + k * active) * 32;
          o[k][0] = lds128f(a0 + own_lo_b);
          o[k][1] = lds128f(a0 + own_hi_b);
#pragma unroll
          for (int e = 0; e < 8; ++e) pv[k][e] = lds32f(a0 + off_b[e]);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k)
          rotate_vector<FULL>(v + k * active, o[k][0], o[k][1], pv[k], c2, s2, inv_of(v + k * active), q_dst, k_dst,
                              q_vec, slot_ok);
      }
      if (v < qk_vec) {
        const uint32_t a0 = u32 + v * 32;
        float pv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) pv[e] = lds32f(a0 + off_b[e]);
        rotate_vector<FULL>(v, lds128f(a0 + own_lo_b), lds128f(a0 + own_hi_b), pv, c2, s2, inv_of(v), q_dst, k_dst,
                            q_vec, slot_ok);
      }
    }
    __syncthreads();
  }
  if (tid == 0) bulk_wait_all();     // the last V stores have completed
}

int gcd_int(int x, int y) {
  while (y) {
    const int r = x % y;
    x = y;
    y = r;
  }
  return x;
}

// Worker threads per CTA: a multiple of lcm(vph, 32) (both swizzle bits) or
// else of lcm(vph, 8) (bit 2 only), at most kStagedBlock.
void staged_shape(const QkvArgs& a, int& active, int& swz2) {
  const int vph = a.d / 8;
  const int l32 = vph / gcd_int(vph, 32) * 32;
  if (l32 <= kStagedBlock) {
    active = kStagedBlock / l32 * l32;
    swz2 = 1;
  } else {
    const int l8 = vph / gcd_int(vph, 8) * 8;
    active = kStagedBlock / l8 * l8;
    swz2 = 0;
  }
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

template <bool FULL>
cudaError_t launch_staged(const QkvArgs& a, cudaStream_t stream) {
  QkvArgs b = a;
  staged_shape(a, b.active, b.swz2);
  const int threads = (b.active + 31) & ~31;
  if (threads < b.n_slots) return cudaErrorInvalidValue;   // one rotation slot per thread
  int dev = 0, sms = 0, optin = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  // Ring depth: the one that keeps the most CTAs on an SM (more warps hide
  // more latency than a second buffer does), the deeper one on a tie.
  cudaError_t e = raise_smem_limit(qkv_staged_kernel<FULL>);
  if (e != cudaSuccess) return e;
  size_t smem = 0;
  for (int nb = 2; nb >= 1; --nb) {
    const size_t bytes = staged_layout(b.n_q, b.n_kv, b.d, b.n_slots, threads / 32, nb).total;
    if (bytes > static_cast<size_t>(optin)) continue;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, qkv_staged_kernel<FULL>, threads, bytes);
    if (e != cudaSuccess) return e;
    if (occ > per_sm) {
      per_sm = occ;
      b.nb = nb;
      smem = bytes;
    }
  }
  if (per_sm < 1) return cudaErrorInvalidValue;
  const int64_t resident = static_cast<int64_t>(sms) * per_sm;
  const unsigned grid = static_cast<unsigned>(a.tokens < resident ? a.tokens : resident);
  return launch_pdl(qkv_staged_kernel<FULL>, dim3(grid), dim3(threads), smem, stream, b);
}

template <int LPH, int G>
cudaError_t launch_rot1d_g(const QkvArgs& a, cudaStream_t stream) {
  constexpr int BLOCK = rot1d_block(G, LPH);
  static_assert(G * LPH <= BLOCK, "a token's threads fit one CTA");
  const int tok_per_cta = BLOCK / (G * LPH);
  const unsigned grid = static_cast<unsigned>((a.tokens + tok_per_cta - 1) / tok_per_cta);
  if (a.norm == kQkNormLayerNorm)
    return launch_pdl(qkv_rot1d_kernel<LPH, true, G, BLOCK>, dim3(grid), dim3(BLOCK), 0, stream, a);
  return launch_pdl(qkv_rot1d_kernel<LPH, false, G, BLOCK>, dim3(grid), dim3(BLOCK), 0, stream, a);
}

// G, the head groups of a token (a power of two from 8 up):
//  * streaming launches (more tokens than SMs): the smallest G that leaves a
//    thread at most kRotBatch heads, within the 128 threads a token may use
//    (a thread with more heads takes them in batches).  One token per
//    128-thread CTA measured faster than one per 256-thread CTA with a single
//    batch (Qwen3, 48 heads: 17.1 vs 19.6 us; Chameleon, 96 heads: 32.8 vs
//    34.8 us): the CTAs that run alone at the end of the launch are shorter.
//  * launch-bound ones (at most one token per SM, e.g. decode): a group per
//    head, up to 512 threads per token, so a thread's critical path is one
//    head (Qwen3 decode, 32 tokens into a paged cache: 2.16-2.28 us per call
//    against 2.52-2.59 with 128-thread CTAs).
template <int LPH>
cudaError_t launch_rot1d(const QkvArgs& a, cudaStream_t stream) {
  const int heads = a.n_q + 2 * a.n_kv;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int g = 8;
  if (a.tokens <= sms) {
    constexpr int gwide = 512 / LPH;         // 128, 64, 32 for head_dim 64, 128, 256
    while (g < gwide && g < heads) g *= 2;
  } else {
    constexpr int gmax = 128 / LPH;          // 32, 16, 8
    while (g < gmax && g * kRotBatch < heads) g *= 2;
  }
  if constexpr (512 / LPH >= 128)
    if (g == 128) return launch_rot1d_g<LPH, 128>(a, stream);
  if constexpr (512 / LPH >= 64)
    if (g == 64) return launch_rot1d_g<LPH, 64>(a, stream);
  if (g == 32) return launch_rot1d_g<LPH, 32>(a, stream);
  if (g == 16) return launch_rot1d_g<LPH, 16>(a, stream);
  return launch_rot1d_g<LPH, 8>(a, stream);
}

}  // namespace

bool qkv_uses_rot1d(int norm, int rope, int d) {
  return (norm == kQkNormPerHead || norm == kQkNormLayerNorm) && rope == kRope1D && (d == 64 || d == 128 || d == 256);
}

cudaError_t launch_qkv_split_norm_rope(const QkvArgs& a, cudaStream_t stream) {
  if (a.tokens == 0) return cudaSuccess;
  if (qkv_uses_rot1d(a.norm, a.rope, a.d)) {
    switch (a.d) {
      case 64: return launch_rot1d<4>(a, stream);
      case 128: return launch_rot1d<8>(a, stream);
      default: return launch_rot1d<16>(a, stream);
    }
  }
  return a.norm == kQkNormFullWidth ? launch_staged<true>(a, stream) : launch_staged<false>(a, stream);
}

}  // namespace gbf
