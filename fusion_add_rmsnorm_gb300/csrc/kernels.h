// Internal interface between the C-ABI layer (abi.cu) and the kernel
// translation units.  Argument structs are passed to kernels by value.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gbf {

enum { kNormWeight = 0, kNormNoWeight = 1, kNormAda = 2 };
enum { kQkNormPerHead = 0, kQkNormFullWidth = 1, kQkNormLayerNorm = 2 };
enum { kRope1D = 0, kRope3D = 1 };
enum { kActNone = 0, kActGeluTanh = 1, kActGeluErf = 2, kActSilu = 3 };

// ------------------------------------------------------- add + RMSNorm + FP8
struct AddRmsNormArgs {
  const void* x;
  const void* res_in;
  void* res_out;
  const void* gate;       // nullable
  const void* weight;     // kNormWeight
  const void* ada_scale;  // kNormAda
  const void* ada_shift;  // kNormAda
  void* q_out;
  int64_t rows;
  int64_t hidden;
  float eps;
  float fp8_scale;
  int mode;
  int tpr;                // threads per row (set by the launcher)
  int rows_per_cta;       // (set by the launcher)
};

struct AddRmsNormPlan {
  bool ok;
  int nv, tpr, rows_per_cta, block;
  int fac;                // where the per-column factors live (registers, packed registers, shared memory)
  int64_t grid;           // CTAs needed; the launch caps it at the CTAs that fit on the GPU at once
};

AddRmsNormPlan plan_add_rmsnorm(int64_t rows, int64_t hidden, int mode);
cudaError_t launch_add_rmsnorm_fp8(AddRmsNormArgs a, cudaStream_t stream, bool pdl);

// --------------------------------------------- packed QKV split + norm + RoPE
constexpr int kMaxRopeSlots = 128;      // head_dim <= 256

struct QkvArgs {
  const void* qkv;
  const void* q_w;
  const void* k_w;
  const void* q_b;        // LayerNorm biases (nullable: 0)
  const void* k_b;
  const int32_t* pos;
  const int32_t* slots;   // nullable
  void* q_out;
  void* k_cache;
  void* v_cache;
  unsigned int* err;
  int64_t tokens;
  int64_t cache_rows;
  int n_q, n_kv, d;
  int norm, rope;
  float eps;
  int sec[3];             // 3D section widths (sum = d)
  int n_slots;            // rotation slots per head = d / 2
  // staged kernel, set by the launcher: worker threads per CTA, bank swizzle
  // bit, depth of the shared-memory row ring
  int active, swz2, nb;
  // per slot: rotation frequency (hi + lo binary32 split of the float64 value),
  // which grid coordinate drives it, and its (lo, hi) element pair in the head
  float omega_hi[kMaxRopeSlots];
  float omega_lo[kMaxRopeSlots];
  unsigned char axis[kMaxRopeSlots];
  unsigned char lo_idx[kMaxRopeSlots];
  unsigned char hi_idx[kMaxRopeSlots];
};

cudaError_t launch_qkv_split_norm_rope(const QkvArgs& a, cudaStream_t stream);

// ---------------------------------------------- gated activation act(g) * u
struct GatedActArgs {
  const void* x;          // bf16 [rows, 2d]: gate | up
  void* y;                // bf16 [rows, d]
  int64_t rows, d;
  int act;
  int64_t tiles_per_row;  // set by the launcher
};

cudaError_t launch_gated_act(const GatedActArgs& a, cudaStream_t stream);
// True when the register-only per-head 1D kernel handles (norm, rope, d).  Every
// other case stages a token's packed row (bf16) and its Q and K (float32) in
// shared memory, which bounds (6 n_q + 8 n_kv) * d by kQkvStagedMaxBytes.
bool qkv_uses_rot1d(int norm, int rope, int d);
constexpr int64_t kQkvStagedMaxBytes = 196608;

// ------------------------------------------------------------ BN folding
struct BnFoldArgs {
  const void* w;
  const void* b;          // nullable
  const float* gamma;
  const float* beta;
  const float* mean;
  const float* var;
  void* w_out;
  void* b_out;
  float eps;
  int64_t out_ch;
  int64_t inner;
};

cudaError_t launch_bn_fold(const BnFoldArgs& a, cudaStream_t stream);

// ------------------------------------------------------------- copy probe
cudaError_t launch_copy(const void* src, void* dst, int64_t bytes, cudaStream_t stream);

// ------------------------------------------------------- failure self-test
cudaError_t launch_bounded_wait_selftest(unsigned int* err, cudaStream_t stream);

// ------------------------------------------------ Linear + bias + GELU GEMM
struct GemmArgs {
  const void* x;          // [M, K] bf16 (or E4M3 codes when fp8), K-major
  const void* w;          // [N, K] bf16 (or E4M3 codes when fp8), K-major
  const void* bias;       // [N] bf16, nullable
  void* y;                // [M, N] bf16
  const float* w_scale;   // fp8: [N] weight descales
  float x_scale;          // fp8: activation descale
  int fp8;
  unsigned int* err;
  int64_t m, n, k;
  int act;
};

// ------------------------------------------------------- weight folding
struct NormFoldArgs {
  const void* w;          // [out_ch, inner] bf16
  const void* gamma;      // [inner] bf16
  void* w_out;            // [out_ch, inner] bf16 (may equal w)
  int64_t out_ch, inner;
  int gemma;              // W * (1 + gamma) when set, else W * gamma
};

cudaError_t launch_fold_norm_weight(const NormFoldArgs& a, cudaStream_t stream);

cudaError_t launch_linear_bias_gelu(const GemmArgs& a, cudaStream_t stream, const char** why);

}  // namespace gbf
