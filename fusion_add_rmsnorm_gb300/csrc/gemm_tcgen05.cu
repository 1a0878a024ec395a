// linear_bias_gelu: Y = GELU_tanh(X W^T + bias) on the 5th-generation tensor
// cores (tcgen05), bf16 operands, float32 accumulation in tensor memory (TMEM),
// bias + GELU applied to the accumulator tile before the single bf16 store.
//
// Method: "OpenPPL算子融合深度解析", §4.3 (the epilogue runs on the GEMM's
// output tile in registers: += bias, then GELU
// 0.5 a (1 + tanh(0.7978845608 (a + 0.044715 a^3))), then one write) and §3.1
// (the activation is applied as an epilogue, never as a separate pass); the
// MatMul -> BiasAdd -> activation pattern of the CANN graph-autofusion article
// (three HBM passes become one); npu_linear of the MindIE-SD RFC, §3.5.
//
// Design (persistent, one CTA per SM; CTA pairs when M spans two tiles):
//   tiles      each CTA owns a BM x BN = 128 x 256 output tile (128 x 128 for a
//              single M tile with fewer 256-wide N tiles than SMs); BK = one
//              128-byte swizzle row of K (64 bf16 or 128 E4M3) per k-block.
//   pairs      a cluster of two CTAs on vertically adjacent M tiles runs as
//              one tcgen05 CTA pair (cta_group::2): the even CTA issues
//              M256 N256 MMAs that read X rows from both CTAs' shared memory
//              and W rows 0..127 of the tile from its own, 128..255 from the
//              other's, writing each CTA's 128 x 256 accumulator into that
//              CTA's TMEM.  Each SM stages 32 KB per k-block instead of 48 KB,
//              which is what bounds a single CTA's MMA rate (shared-memory
//              bandwidth: TMA writes plus operand reads).  A single M tile
//              runs unpaired (cta_group::1, M128 N256).
//   warp 0     TMA producer (each CTA): cp.async.bulk.tensor 2D loads of its
//              X and W k-blocks into a shared-memory ring (128-byte swizzle);
//              in a pair both CTAs' copies complete on the even CTA's
//              barrier, which expects the bytes of both.
//   warp 1     MMA issuer (the even CTA of a pair): one elected thread issues
//              tcgen05.mma from shared-memory descriptors into TMEM and
//              commits each stage back to both CTAs' producers.
//   warp 2     allocates (and at exit frees) 512 TMEM columns: two 128 x 256
//              float32 accumulators, so the epilogue of tile i overlaps the
//              MMAs of tile i + 1.
//   warps 4-11 epilogue (each CTA): tcgen05.ld 32 columns at a time (warp w
//              reads TMEM lanes 32 (w % 4) .. +31, one output row per thread,
//              half of the tile's columns), descales and bias, the activation
//              (fast forms, see common.cuh), round to bf16 into a 32-row x
//              64-column box in shared memory (128-byte swizzle, so the
//              one-row-per-lane writes are conflict-free), written out by
//              one bulk tensor store (cp.async.bulk.tensor) that clips at M
//              and N;
//              then the warp arrives on the even CTA's "accumulator free"
//              barrier.
// Tile order: the N tiles are cut into groups of group_n (chosen at launch,
// 16 or a nearby divisor of the resident cluster count); inside a group the
// tiles run n-fastest, so the CTAs working at one time cover a few 256-row
// units of X against the group's group_n W column blocks.  A group's W
// (group_n x 2 MB at K = 4096) stays in L2 while X streams past it once per
// group, instead of all of X having to stay in L2 for every W column block.
//
// Every mbarrier wait is bounded (about one second of wall time): a wait that
// gives up sets DEV_ERR_MBAR_TIMEOUT in the device error word and raises a
// CTA-wide abort flag; every role then leaves its loop, the MMA issuer drains
// its outstanding tensor-core work, the producers' copies are all waited for
// (bounded), and TMEM is freed before the CTAs exit.  No role returns early:
// both CTAs of a pair always reach the closing cluster barriers.
#include <cuda.h>

#include "kernels.h"
#include "tma.cuh"

namespace gbf {
namespace {

constexpr int BM = 128;                          // output rows per CTA (TMEM lanes)
constexpr int BN = 256;                          // N tile (CTA pairs and most unpaired launches)
constexpr int BN_NARROW = 128;                   // N tile of unpaired launches with few tiles
constexpr int BK_BYTES = 128;                    // one 128-byte swizzle row of K per k-block
constexpr int UMMA_K_BYTES = 32;                 // K of one MMA: 16 bf16 or 32 E4M3 values
// TMEM columns: two float32 accumulators of the N tile (all 512 at BN)
constexpr int tmem_cols(int tn) { return 2 * tn; }
constexpr int kThreads = 384;
constexpr int kEpilogueWarp0 = 4;                // warps 4..11: two per TMEM lane quarter
constexpr int kEpilogueWarps = 8;

// Output staging: each epilogue warp packs 32 rows x 64 columns of bf16 (one
// 128-byte-swizzled TMA box) before a bulk tensor store.
constexpr int kOutCols = 64;
constexpr int kOutBoxBytes = 32 * kOutCols * 2;              // 4 KB
constexpr int kOutBytes = kEpilogueWarps * kOutBoxBytes;      // 32 KB

// Shared-memory ring of one CTA: unpaired, the whole W tile per stage; paired,
// half of it (the other half sits in the other CTA).  AR of the tile's 128 X
// rows are loaded per 128-byte K row: all of them, or, for a decode batch of
// at most 32 or 64 rows, only those (the MMA still reads 128 rows from each
// K row's start, the rest being other bytes of the ring whose products land
// in output rows the clipped stores never write); decode stages then hold
// KH = 2 consecutive K rows, so each W row is read in 256-byte runs and more
// of W is in flight.  32 KB stages take a six-deep ring, 48 KB ones
// (unpaired, 256-wide) three, decode stages as many as 192 KB holds.
template <bool PAIR, int TN, int AR>
struct Ring {
  static constexpr int kKH = AR < BM ? 2 : 1;               // 128-byte K rows per stage
  static constexpr int kBRows = PAIR ? TN / 2 : TN;
  static constexpr int kAStageBytes = AR * BK_BYTES * kKH;
  static constexpr int kBStageBytes = kBRows * BK_BYTES * kKH;
  static constexpr int kStageBytes = kAStageBytes + kBStageBytes;
  static constexpr int kStages = AR < BM ? 196608 / kStageBytes : (kStageBytes <= 32768 ? 6 : 3);
};

template <int S>
struct __align__(8) SharedCtl {
  uint64_t full[S];
  uint64_t empty[S];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t peer_issued[S];   // pair, even CTA: k-blocks the odd CTA issued per stage
  int abort;
};

template <bool PAIR, int TN, int AR>
constexpr size_t smem_bytes() {
  using R = Ring<PAIR, TN, AR>;
  return 1024 /* alignment slack */ + R::kStages * R::kStageBytes + kOutBytes + sizeof(SharedCtl<R::kStages>);
}

// ------------------------------------------------------------ PTX wrappers

GBF_DEVICE void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// A load into this CTA's shared memory completing on an mbarrier that may sit
// in either CTA of the pair (`bar` is a shared::cluster address).
GBF_DEVICE void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Bulk tensor store of the box at shared address `src` to coordinates
// (c0, c1) of `map`; elements outside the tensor are not written.
GBF_DEVICE void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(src)), "r"(c0), "r"(c1)
               : "memory");
}

GBF_DEVICE uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the object at this CTA's shared address `a`, in
// CTA `rank` of the cluster.
GBF_DEVICE uint32_t map_cluster(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

GBF_DEVICE uint32_t ld_cluster_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

GBF_DEVICE void st_cluster_u32(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Arrive on an mbarrier of any CTA of the cluster (shared::cluster address).
GBF_DEVICE void mbar_arrive_cluster(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Count `bytes` of the current phase's expected transactions as done.
GBF_DEVICE void mbar_complete_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Every thread of every CTA of the cluster: release this CTA's prior memory
// operations and wait for all of the cluster's threads.
GBF_DEVICE void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

GBF_DEVICE void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
GBF_DEVICE void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Every tcgen05 instruction of one kernel names the same CTA group: 1 when
// unpaired, 2 in a pair.
template <bool PAIR>
GBF_DEVICE void tmem_alloc(uint32_t* dst, uint32_t cols) {
  if (PAIR) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  } else {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
}

template <bool PAIR>
GBF_DEVICE void tmem_dealloc(uint32_t base, uint32_t cols) {
  if (PAIR)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}

// Arrive on `bar` once the tensor-core work issued so far has completed:
// unpaired, in this CTA; paired, at the same offset in both CTAs.
template <bool PAIR>
GBF_DEVICE void tc_commit(uint64_t* bar) {
  if (PAIR)
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(smem_u32(bar)), "h"(static_cast<uint16_t>(0x3))
        : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// tc_commit arriving on this CTA's `bar` only (the issuer's final drain).
template <bool PAIR>
GBF_DEVICE void tc_commit_self(uint64_t* bar) {
  if (PAIR)
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T with a float32 accumulator: kind::f16 for
// bf16 operands, kind::f8f6f4 for E4M3 operands (both operands one type).
template <bool FP8, bool PAIR>
GBF_DEVICE void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  if (FP8 && PAIR)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  else if (FP8)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  else if (PAIR)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 consecutive float32 columns of this warp's 32 TMEM lanes, one lane per thread.
GBF_DEVICE void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row core groups 1024 bytes apart
// (stride byte offset), descriptor version 1, layout "swizzle 128B".
GBF_DEVICE uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);          // start address
  d |= static_cast<uint64_t>(1) << 16;                          // leading byte offset (unused for SW128 K-major)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                  // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                          // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                          // swizzle 128B
  return d;
}

// Instruction descriptors: float32 D (bits 4-5 = 1), A and B type codes at
// bits 7-9 and 10-12 (kind::f16: bf16 = 1; kind::f8f6f4: E4M3 = 0), both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24 (M = 256 for a CTA pair).
__host__ __device__ constexpr uint32_t idesc(bool fp8, int m, int n) {
  return (1u << 4) | ((fp8 ? 0u : 1u) << 7) | ((fp8 ? 0u : 1u) << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

struct GemmParams {
  const __nv_bfloat16* bias;
  const float* w_scale;      // E4M3 weights: descale per output channel
  float x_scale;             // E4M3 activations: the descale
  unsigned int* err;
  int m, n, k;
  int m_tiles, n_tiles;
  int group_n;               // N tiles per group of the tile order
  int act;
};

// Output tile origin (m0, n0) of linear work index `tile` (see the tile order
// above).  With CTA pairs a work item is two vertically adjacent M tiles
// sharing one W column block: m_units = ceil(m_tiles / cl), and CTA rank
// `rank` of the pair takes M tile unit * cl + rank.
GBF_DEVICE void tile_origin(const GemmParams& p, int m_units, int cl, int rank, int tile, int tn, int& m0, int& n0) {
  const int per_group = p.group_n * m_units;
  const int g = tile / per_group;
  const int idx = tile - g * per_group;
  const int n_base = g * p.group_n;
  const int gs = p.n_tiles - n_base < p.group_n ? p.n_tiles - n_base : p.group_n;
  m0 = ((idx / gs) * cl + rank) * BM;
  n0 = (n_base + idx % gs) * tn;
}

template <bool FP8, bool PAIR, int TN, int AR>
__global__ void __launch_bounds__(kThreads, 1)
linear_bias_gelu_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                        const __grid_constant__ CUtensorMap map_y, const GemmParams p) {
  using R = Ring<PAIR, TN, AR>;
  static_assert(AR == BM || !PAIR, "pairs load every X row");
  static_assert(AR == BM || R::kStages * R::kBStageBytes >= (BM - AR) * BK_BYTES,
                "the MMA's reads past the last A rows stay inside the ring");
  constexpr int S = R::kStages;
  constexpr int CL = PAIR ? 2 : 1;
  constexpr int BK = FP8 ? BK_BYTES : BK_BYTES / 2;         // K elements per k-block
  constexpr uint32_t kIdesc = idesc(FP8, CL * BM, TN);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the same offsets in both CTAs of a pair: the MMAs address the odd CTA's
  // operands by the even CTA's shared addresses
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smem_a = smem;                                   // S x KH x AR rows of 128 bytes
  uint8_t* smem_b = smem + S * R::kAStageBytes;             // S x KH x kBRows rows of 128 bytes
  uint8_t* smem_out = smem + S * R::kStageBytes;            // 8 x 4 KB output boxes (1 KB aligned)
  SharedCtl<S>* ctl = reinterpret_cast<SharedCtl<S>*>(smem_out + kOutBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = rank == 0;            // issues the MMAs (always, unpaired)
  const int m_units = (p.m_tiles + CL - 1) / CL;
  const int first = blockIdx.x / CL, stride = gridDim.x / CL;
  constexpr int KH = R::kKH;
  const int k_blocks = (p.k + BK * KH - 1) / (BK * KH);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&ctl->full[s], 1);         // the even CTA's expect-bytes arrive
      mbar_init(&ctl->empty[s], 1);        // the MMA issuer's commit
      ctl->peer_issued[s] = 0;
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ctl->tmem_full[a], 1);
      mbar_init(&ctl->tmem_empty[a], CL * kEpilogueWarps);   // one arrive per epilogue warp of the pair
    }
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    mbar_fence_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_x)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_w)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_y)) : "memory");
  }
  if (warp == 2) tmem_alloc<PAIR>(&ctl->tmem_base, tmem_cols(TN));
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();                // both CTAs' barriers and TMEM exist before either is used
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  // The pair's MMAs address both CTAs' accumulators by one TMEM address; the
  // whole of TMEM is allocated, so both bases are column 0 -- checked, and on
  // a mismatch (both CTAs see it) the pair does no work and reports it.
  bool usable = true;
  if (PAIR) {
    usable = ld_cluster_u32(map_cluster(smem_u32(&ctl->tmem_base), static_cast<uint32_t>(rank ^ 1))) == tmem_base;
    if (!usable && threadIdx.x == 0) raise_error(p.err, DEV_ERR_PAIR_TMEM);
  }
  const int num_tiles = usable ? m_units * p.n_tiles : 0;

  uint32_t issued[S];                      // producer: k-blocks issued per stage (for the final drain)
#pragma unroll
  for (int s = 0; s < S; ++s) issued[s] = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = first; tile < num_tiles && ok; tile += stride) {
        int m0, n0;
        tile_origin(p, m_units, CL, rank, tile, TN, m0, n0);
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!mbar_wait<PAIR, false>(&ctl->empty[stage], phase ^ 1u, &ctl->abort, p.err)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&ctl->full[stage], CL * R::kStageBytes);
#pragma unroll
          for (int h = 0; h < KH; ++h) {        // KH consecutive 128-byte K rows (beyond K: zero fill)
            const int kc = (kb * KH + h) * BK;
            uint8_t* da = smem_a + stage * R::kAStageBytes + h * AR * BK_BYTES;
            uint8_t* db = smem_b + stage * R::kBStageBytes + h * R::kBRows * BK_BYTES;
            if (PAIR) {
              const uint32_t bar = map_cluster(smem_u32(&ctl->full[stage]), 0);
              tma_load_2d_pair(da, &map_x, bar, kc, m0);
              tma_load_2d_pair(db, &map_w, bar, kc, n0 + rank * R::kBRows);
            } else {
              tma_load_2d(da, &map_x, &ctl->full[stage], kc, m0);
              tma_load_2d(db, &map_w, &ctl->full[stage], kc, n0);
            }
          }
          ++issued[stage];
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (PAIR && !leader)                 // the even CTA drains the odd one's copies (they land on its barriers)
        for (int s = 0; s < S; ++s) st_cluster_u32(map_cluster(smem_u32(&ctl->peer_issued[s]), 0), issued[s]);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int local = 0;
      for (int tile = first; tile < num_tiles && ok; tile += stride, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1u;
        if (!mbar_wait<PAIR, false>(&ctl->tmem_empty[acc], acc_phase ^ 1u, &ctl->abort, p.err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * TN;
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!mbar_wait<false, false>(&ctl->full[stage], phase, &ctl->abort, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem_a + stage * R::kAStageBytes);
          const uint32_t b_addr = smem_u32(smem_b + stage * R::kBStageBytes);
#pragma unroll
          for (int h = 0; h < KH; ++h)
#pragma unroll
            for (int kk = 0; kk < BK_BYTES / UMMA_K_BYTES; ++kk) {
              // advance one MMA's K (32 bytes) inside the swizzled row
              const uint64_t a_desc = smem_desc_sw128(a_addr + h * AR * BK_BYTES + kk * UMMA_K_BYTES);
              const uint64_t b_desc = smem_desc_sw128(b_addr + h * R::kBRows * BK_BYTES + kk * UMMA_K_BYTES);
              tc_mma<FP8, PAIR>(d_tmem, a_desc, b_desc, kIdesc, (kb | h | kk) != 0);
            }
          tc_commit<PAIR>(&ctl->empty[stage]);   // frees the stage (in both CTAs) once these MMAs have read it
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) tc_commit<PAIR>(&ctl->tmem_full[acc]);
      }
      // Drain: all tensor-core work this thread issued has completed.
      tc_commit_self<PAIR>(&ctl->drain);
      int drain_abort = 0;
      mbar_wait(&ctl->drain, 0, &drain_abort, p.err);
    }
  } else if (warp >= kEpilogueWarp0) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;                       // TMEM lanes 32*quarter .. +31 (warp % 4)
    const int half = (warp - kEpilogueWarp0) >> 2;      // columns 128*half .. +127 of the tile
    uint8_t* my_out = smem_out + (warp - kEpilogueWarp0) * kOutBoxBytes;
    const uint32_t out32 = smem_u32(my_out);
    int local = 0;
    for (int tile = first; tile < num_tiles; tile += stride, ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1u;
      bool ok = true;
      if (lane == 0) ok = mbar_wait<PAIR>(&ctl->tmem_full[acc], acc_phase, &ctl->abort, p.err);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      int m0, n0;
      tile_origin(p, m_units, CL, rank, tile, TN, m0, n0);
      const int row0 = m0 + quarter * 32;                 // this warp's 32 rows; lane = row within them
      const uint32_t taddr = tmem_base + acc * TN + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
      for (int box = 0; box < TN / 2 / kOutCols; ++box) {
        const int cbase = half * (TN / 2) + box * kOutCols;   // tile column of the box
        const int col0 = n0 + cbase;
        // the previous box's store has finished reading the staging buffer
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll 1
        for (int sub = 0; sub < kOutCols / 32; ++sub) {
          // the 32 columns' bias and weight descales are requested before the
          // TMEM load, so their latency overlaps it (the same for every lane)
          uint4 braw[4];
          float4 sraw[4][2];
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int col = col0 + sub * 32 + g * 8;
            const bool in = col < p.n;                      // N % 16 == 0: whole 8-column groups
            braw[g] = (p.bias && in) ? ld_cached(p.bias + col) : make_uint4(0, 0, 0, 0);
            if (FP8) {
              sraw[g][0] = in ? *reinterpret_cast<const float4*>(p.w_scale + col) : make_float4(0.f, 0.f, 0.f, 0.f);
              sraw[g][1] = in ? *reinterpret_cast<const float4*>(p.w_scale + col + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
          uint32_t r[32];
          tmem_ld_32cols(taddr + cbase + sub * 32, r);      // this lane's row, 32 columns
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            float v[8];
            float bz[8];
            bf16x8_to_f32(braw[g], bz);
            float sc[8];
            if (FP8) {                                      // descales: activation x weight row
              const float4 s0 = sraw[g][0], s1 = sraw[g][1];
              const float ws[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
              for (int e = 0; e < 8; ++e) sc[e] = p.x_scale * ws[e];
            }
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const float2 acc = make_float2(__uint_as_float(r[g * 8 + e]), __uint_as_float(r[g * 8 + e + 1]));
              const float2 bb = make_float2(bz[e], bz[e + 1]);
              const float2 a = FP8 ? __ffma2_rn(acc, make_float2(sc[e], sc[e + 1]), bb) : __fadd2_rn(acc, bb);
              const float2 o = fast_act2(a, p.act);
              v[e] = o.x;
              v[e + 1] = o.y;
            }
            // 16-byte piece j of row `lane` sits at piece j ^ (row % 8) (the TMA 128-byte swizzle)
            const int j = sub * 4 + g;
            const uint4 pk = f32x8_to_bf16x8(v);
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(out32 + lane * 128 + ((j ^ (lane & 7)) << 4)),
                         "r"(pk.x), "r"(pk.y), "r"(pk.z), "r"(pk.w)
                         : "memory");
          }
        }
        fence_proxy_async_smem();                         // the pieces are visible to the bulk store
        __syncwarp();
        if (lane == 0 && col0 < p.n && row0 < p.m) {
          tma_store_2d(&map_y, my_out, col0, row0);
          bulk_commit();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR)
          mbar_arrive_cluster(map_cluster(smem_u32(&ctl->tmem_empty[acc]), 0));
        else
          mbar_arrive(&ctl->tmem_empty[acc]);
      }
    }
    if (lane == 0) bulk_wait_all();                       // every output store of this warp has completed
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();                // the odd CTA's issue counts are in place
  if (warp == 0 && lane == 0) {
    // Every copy issued to this CTA (or, in a pair, to either CTA) has landed
    // before the CTAs may exit: wait for the last phase of each stage
    // (bounded; immediate on the normal path, where the MMAs consumed them all).
    int drain_abort = 0;                   // own flag: the CTA one may already be set
    if (!PAIR) {
      for (int s = 0; s < S; ++s)
        if (issued[s]) mbar_wait(&ctl->full[s], (issued[s] - 1) & 1u, &drain_abort, nullptr);
    } else if (leader) {
      for (int s = 0; s < S; ++s) {
        const uint32_t mine = issued[s], theirs = ctl->peer_issued[s];
        // After an abort the two producers may stand one k-block apart on a
        // stage (each waits for the MMAs of the one before); complete the
        // phase that only one of them filled.
        if (theirs > mine)
          mbar_arrive_expect_tx(&ctl->full[s], R::kStageBytes);   // the odd CTA's copies alone
        else if (mine > theirs)
          mbar_complete_tx(&ctl->full[s], R::kStageBytes);        // this CTA's copies alone
        const uint32_t last = mine > theirs ? mine : theirs;
        if (last) mbar_wait(&ctl->full[s], (last - 1) & 1u, &drain_abort, nullptr);
      }
    }
  }
  __syncthreads();
  if (PAIR) cluster_sync();                // no copy, commit or remote arrive is left in flight to either CTA
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc<PAIR>(tmem_base, tmem_cols(TN));
  }
}

// ---------------------------------------------------------- host: tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2D tensor [rows, cols] (cols contiguous) of bf16 or of bytes (E4M3), box
// [box_rows, 128 bytes of cols], 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows, bool fp8) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int esize = fp8 ? 1 : 2;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * esize};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK_BYTES / esize), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
            dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool FP8, bool PAIR, int TN, int AR>
cudaError_t launch_gemm(const CUtensorMap& map_x, const CUtensorMap& map_w, const CUtensorMap& map_y,
                        const GemmParams& p, int sms,
                        cudaStream_t stream, const char** why) {
  auto kern = linear_bias_gelu_kernel<FP8, PAIR, TN, AR>;
  constexpr int CL = PAIR ? 2 : 1;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem_bytes<PAIR, TN, AR>()));
  if (e != cudaSuccess) {
    *why = "could not reserve shared memory";
    return e;
  }
  const int units = ((p.m_tiles + CL - 1) / CL) * p.n_tiles;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes<PAIR, TN, AR>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Persistent: as many clusters as can be resident at once (a GPC with an
  // odd SM count leaves one SM out of the pairs), so no cluster waits for a
  // second wave.
  int slots = sms / CL;
  if (PAIR) {
    cfg.gridDim = dim3(static_cast<unsigned>(slots * CL));
    int resident = 0;
    if (cudaOccupancyMaxActiveClusters(&resident, kern, &cfg) == cudaSuccess && resident > 0 && resident < slots)
      slots = resident;
    cudaGetLastError();
  }
  const int clusters = units < slots ? units : slots;
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * CL));
  // Group width: the divisor of the resident cluster count nearest 16 within
  // 12..24 (19 for 76 pairs), so each round of the persistent clusters covers
  // whole M units of one group (a block of tiles sharing its X rows and W
  // columns); 16 if the count has no such divisor.  On the 8192 x 16384 x
  // 4096 Linear, 19 measured 1.5-2 % faster than 16; 20, 24 and 32 slower.
  GemmParams q = p;
  q.group_n = 16;
  for (int d = 0; d <= 8; ++d) {
    if (16 + d <= 24 && clusters % (16 + d) == 0) { q.group_n = 16 + d; break; }
    if (d > 0 && 16 - d >= 12 && clusters % (16 - d) == 0) { q.group_n = 16 - d; break; }
  }
  return cudaLaunchKernelEx(&cfg, kern, map_x, map_w, map_y, q);
}

}  // namespace

cudaError_t launch_linear_bias_gelu(const GemmArgs& a, cudaStream_t stream, const char** why) {
  const bool fp8 = a.fp8 != 0;
  const int m_tiles = static_cast<int>((a.m + BM - 1) / BM);
  const bool pair = m_tiles >= 2;                        // CTA pairs on adjacent M tiles
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // A single M tile (a decode batch of at most 128 rows) with fewer 256-wide
  // N tiles than SMs takes 128-wide N tiles: twice the CTAs stream W, which
  // is nearly all such a launch reads.
  const bool narrow = !pair && (a.n + BN - 1) / BN < sms;
  const int tn = narrow ? BN_NARROW : BN;
  // X rows loaded per stage: 32 or 64 for a narrow launch of that few rows
  const int ar = narrow && a.m <= 32 ? 32 : narrow && a.m <= 64 ? 64 : BM;
  CUtensorMap map_x, map_w, map_y;
  if (!make_map(&map_x, a.x, a.m, a.k, ar, fp8) || !make_map(&map_w, a.w, a.n, a.k, pair ? BN / 2 : tn, fp8) ||
      !make_map(&map_y, a.y, a.m, a.n, 32, false)) {
    *why = "cuTensorMapEncodeTiled is unavailable or rejected the operands";
    return cudaErrorInvalidValue;
  }
  GemmParams p;
  p.bias = static_cast<const __nv_bfloat16*>(a.bias);
  p.w_scale = a.w_scale;
  p.x_scale = a.x_scale;
  p.err = a.err;
  p.m = static_cast<int>(a.m);
  p.n = static_cast<int>(a.n);
  p.k = static_cast<int>(a.k);
  p.m_tiles = m_tiles;
  p.n_tiles = static_cast<int>((a.n + tn - 1) / tn);
  p.act = a.act;
  cudaError_t e;
  if (fp8)
    e = pair        ? launch_gemm<true, true, BN, BM>(map_x, map_w, map_y, p, sms, stream, why)
        : ar == 32  ? launch_gemm<true, false, BN_NARROW, 32>(map_x, map_w, map_y, p, sms, stream, why)
        : ar == 64  ? launch_gemm<true, false, BN_NARROW, 64>(map_x, map_w, map_y, p, sms, stream, why)
        : narrow    ? launch_gemm<true, false, BN_NARROW, BM>(map_x, map_w, map_y, p, sms, stream, why)
                    : launch_gemm<true, false, BN, BM>(map_x, map_w, map_y, p, sms, stream, why);
  else
    e = pair        ? launch_gemm<false, true, BN, BM>(map_x, map_w, map_y, p, sms, stream, why)
        : ar == 32  ? launch_gemm<false, false, BN_NARROW, 32>(map_x, map_w, map_y, p, sms, stream, why)
        : ar == 64  ? launch_gemm<false, false, BN_NARROW, 64>(map_x, map_w, map_y, p, sms, stream, why)
        : narrow    ? launch_gemm<false, false, BN_NARROW, BM>(map_x, map_w, map_y, p, sms, stream, why)
                    : launch_gemm<false, false, BN, BM>(map_x, map_w, map_y, p, sms, stream, why);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace gbf
