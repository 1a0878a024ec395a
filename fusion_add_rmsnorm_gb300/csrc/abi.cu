// C-ABI boundary of libgbfuse.so: argument validation, status codes, launches.
//
// Nothing here computes a result: every step of every operator runs in the
// kernels.  The host side checks pointers, extents, alignment and overlap,
// builds the by-value kernel argument structs (for RoPE, the table of rotation
// frequencies in float64 split into binary32 hi/lo pairs), and launches on the
// caller's stream.  It never allocates, frees or synchronises device memory
// (gbf_device_status() is the one call that synchronises, by request).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "gbfuse.h"
#include "common.cuh"
#include "kernels.h"

namespace {

thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_msg[0] = '\0';
  return GBF_OK;
}

int launch_status(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(GBF_ELAUNCH, "%s: launch failed: %s", what, cudaGetErrorString(e));
  return ok();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte ranges [a, a + na) and [b, b + nb) intersect.
bool overlap(const void* a, int64_t na, const void* b, int64_t nb) {
  if (!a || !b || na <= 0 || nb <= 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
}

// The library's one piece of device state: an error word per device.
__device__ unsigned int g_device_error;

constexpr int kMaxDevices = 64;
std::mutex g_err_mu;
unsigned int* g_err_ptr[kMaxDevices] = {};

unsigned int* error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned int*>(p);
  }
  return g_err_ptr[dev];
}

}  // namespace

extern "C" {

GBF_API const char* gbf_last_error(void) { return g_msg; }

GBF_API int gbf_version(void) { return 1 * 10000 + 0 * 100 + 0; }

// ------------------------------------------------------- add + RMSNorm + FP8

GBF_API int gbf_add_rmsnorm_fp8(const void* x, const void* res_in, void* res_out, const void* gate, int mode,
                                const void* weight, const void* ada_scale, const void* ada_shift,
                                uint8_t* q_out, int64_t rows, int64_t hidden, float eps, float fp8_scale,
                                void* stream) {
  const char* fn = "gbf_add_rmsnorm_fp8";
  if (rows < 0 || hidden <= 0) return fail(GBF_EINVAL, "%s: rows (%lld) must be >= 0 and hidden (%lld) > 0", fn,
                                           (long long)rows, (long long)hidden);
  if (mode != GBF_NORM_WEIGHT && mode != GBF_NORM_NOWEIGHT && mode != GBF_NORM_ADA)
    return fail(GBF_EINVAL, "%s: unknown norm mode %d", fn, mode);
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return fail(GBF_EINVAL, "%s: eps must be finite and >= 0", fn);
  if (!(fp8_scale > 0.0f) || !std::isfinite(fp8_scale))
    return fail(GBF_EINVAL, "%s: fp8_scale must be finite and > 0", fn);
  if (hidden % 8 != 0) return fail(GBF_EALIGN, "%s: hidden (%lld) must be a multiple of 8", fn, (long long)hidden);
  if (hidden > 32768) return fail(GBF_EUNSUPPORTED, "%s: hidden (%lld) > 32768", fn, (long long)hidden);
  if (rows == 0) return ok();
  if (!x || !res_in || !res_out || !q_out) return fail(GBF_EINVAL, "%s: x, res_in, res_out, q_out are required", fn);
  if (mode == GBF_NORM_WEIGHT && !weight) return fail(GBF_EINVAL, "%s: weight is required in WEIGHT mode", fn);
  if (mode == GBF_NORM_ADA && (!ada_scale || !ada_shift))
    return fail(GBF_EINVAL, "%s: ada_scale and ada_shift are required in ADA mode", fn);
  const void* ptrs[] = {x, res_in, res_out, q_out, gate,
                        mode == GBF_NORM_WEIGHT ? weight : nullptr,
                        mode == GBF_NORM_ADA ? ada_scale : nullptr,
                        mode == GBF_NORM_ADA ? ada_shift : nullptr};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return fail(GBF_EALIGN, "%s: every tensor must be 16-byte aligned", fn);
  const int64_t nb = rows * hidden * 2, nv = hidden * 2;
  const void* ins[] = {x, res_in, gate, ptrs[5], ptrs[6], ptrs[7]};
  const int64_t in_len[] = {nb, nb, nv, nv, nv, nv};
  for (int i = 0; i < 6; ++i) {
    if (i != 1 && overlap(res_out, nb, ins[i], in_len[i]))
      return fail(GBF_EINVAL, "%s: res_out overlaps an input other than res_in", fn);
    if (overlap(q_out, rows * hidden, ins[i], in_len[i])) return fail(GBF_EINVAL, "%s: q_out overlaps an input", fn);
  }
  if (res_out != res_in && overlap(res_out, nb, res_in, nb))
    return fail(GBF_EINVAL, "%s: res_out partially overlaps res_in (only exact aliasing is allowed)", fn);
  if (overlap(res_out, nb, q_out, rows * hidden)) return fail(GBF_EINVAL, "%s: res_out overlaps q_out", fn);

  gbf::AddRmsNormArgs a = {};
  a.x = x;
  a.res_in = res_in;
  a.res_out = res_out;
  a.gate = gate;
  a.weight = weight;
  a.ada_scale = ada_scale;
  a.ada_shift = ada_shift;
  a.q_out = q_out;
  a.rows = rows;
  a.hidden = hidden;
  a.eps = eps;
  a.fp8_scale = fp8_scale;
  a.mode = mode;
  return launch_status(gbf::launch_add_rmsnorm_fp8(a, static_cast<cudaStream_t>(stream), true), fn);
}

// --------------------------------------------- packed QKV split + norm + RoPE

namespace {

// Both QKV entry points: norm is GBF_QKNORM_PER_HEAD / FULL_WIDTH (RMSNorm, no
// biases) or kQkNormLayerNorm (per-head LayerNorm with optional biases).
int qkv_entry(const char* fn, const void* qkv, int64_t tokens, int n_q_heads, int n_kv_heads, int head_dim,
              int norm, const void* q_w, const void* q_b, const void* k_w, const void* k_b, float eps, int rope,
              const int32_t* pos, const int32_t* sections, float theta, void* q_out, void* k_cache, void* v_cache,
              const int32_t* slots, int64_t cache_rows, void* stream) {
  if (tokens < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0)
    return fail(GBF_EINVAL, "%s: tokens >= 0 and positive head counts / head_dim are required", fn);
  if (norm != GBF_QKNORM_PER_HEAD && norm != GBF_QKNORM_FULL_WIDTH && norm != gbf::kQkNormLayerNorm)
    return fail(GBF_EINVAL, "%s: unknown norm %d", fn, norm);
  if (rope != GBF_ROPE_1D && rope != GBF_ROPE_3D) return fail(GBF_EINVAL, "%s: unknown rope %d", fn, rope);
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return fail(GBF_EINVAL, "%s: eps must be finite and >= 0", fn);
  if (!(theta > 0.0f) || !std::isfinite(theta)) return fail(GBF_EINVAL, "%s: theta must be finite and > 0", fn);
  if (head_dim % 16 != 0 || head_dim > 256)
    return fail(GBF_EUNSUPPORTED, "%s: head_dim (%d) must be a multiple of 16 and <= 256", fn, head_dim);
  if (norm == GBF_QKNORM_PER_HEAD && (head_dim & (head_dim - 1)) != 0)
    return fail(GBF_EUNSUPPORTED, "%s: per-head norm needs a power-of-two head_dim (got %d)", fn, head_dim);
  if (norm == gbf::kQkNormLayerNorm && !gbf::qkv_uses_rot1d(norm, rope, head_dim))
    return fail(GBF_EUNSUPPORTED, "%s: LayerNorm needs 1D RoPE and head_dim 64, 128 or 256 (got %d)", fn, head_dim);
  if (n_q_heads > 4096 || n_kv_heads > 4096) return fail(GBF_EUNSUPPORTED, "%s: too many heads", fn);
  if (!gbf::qkv_uses_rot1d(norm, rope, head_dim) &&
      (6LL * n_q_heads + 8LL * n_kv_heads) * head_dim > gbf::kQkvStagedMaxBytes)
    return fail(GBF_EUNSUPPORTED, "%s: (6 n_q_heads + 8 n_kv_heads) * head_dim must be <= %lld for this norm/rope",
                fn, (long long)gbf::kQkvStagedMaxBytes);
  int sec[3] = {head_dim, 0, 0};
  if (rope == GBF_ROPE_3D) {
    if (!sections) return fail(GBF_EINVAL, "%s: 3D RoPE needs sections[3]", fn);
    int sum = 0;
    for (int c = 0; c < 3; ++c) {
      if (sections[c] < 0 || sections[c] % 2 != 0)
        return fail(GBF_EINVAL, "%s: sections must be even and >= 0", fn);
      sec[c] = sections[c];
      sum += sections[c];
    }
    if (sum != head_dim) return fail(GBF_EINVAL, "%s: sections sum to %d, head_dim is %d", fn, sum, head_dim);
  }
  if (!slots && cache_rows < tokens)
    return fail(GBF_EINVAL, "%s: without slots, cache_rows (%lld) must be >= tokens (%lld)", fn,
                (long long)cache_rows, (long long)tokens);
  if (cache_rows < 0) return fail(GBF_EINVAL, "%s: cache_rows must be >= 0", fn);
  if (tokens == 0) return ok();
  if (!qkv || !q_w || !k_w || !pos || !q_out || !k_cache || !v_cache)
    return fail(GBF_EINVAL, "%s: qkv, q_w, k_w, pos, q_out, k_cache, v_cache are required", fn);
  const void* al[] = {qkv, q_w, k_w, q_out, k_cache, v_cache};
  if ((q_b && reinterpret_cast<uintptr_t>(q_b) % 16) || (k_b && reinterpret_cast<uintptr_t>(k_b) % 16))
    return fail(GBF_EALIGN, "%s: biases must be 16-byte aligned", fn);
  for (const void* p : al)
    if (!aligned16(p)) return fail(GBF_EALIGN, "%s: tensors must be 16-byte aligned", fn);
  const int64_t D = head_dim;
  const int64_t in_b = tokens * (n_q_heads + 2LL * n_kv_heads) * D * 2;
  const int64_t wq_b = (norm == GBF_QKNORM_FULL_WIDTH ? n_q_heads * D : D) * 2;
  const int64_t wk_b = (norm == GBF_QKNORM_FULL_WIDTH ? n_kv_heads * D : D) * 2;
  const int64_t pos_b = tokens * (rope == GBF_ROPE_3D ? 3 : 1) * 4;
  const int64_t qo_b = tokens * n_q_heads * D * 2, c_b = cache_rows * n_kv_heads * D * 2;
  void* outs[] = {q_out, k_cache, v_cache};
  const int64_t out_len[] = {qo_b, c_b, c_b};
  const void* ins[] = {qkv, q_w, k_w, pos, slots, q_b, k_b};
  const int64_t in_len[] = {in_b, wq_b, wk_b, pos_b, slots ? tokens * 4 : 0, q_b ? D * 2 : 0, k_b ? D * 2 : 0};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 7; ++j)
      if (overlap(outs[i], out_len[i], ins[j], in_len[j])) return fail(GBF_EINVAL, "%s: an output overlaps an input", fn);
    for (int j = i + 1; j < 3; ++j)
      if (overlap(outs[i], out_len[i], outs[j], out_len[j])) return fail(GBF_EINVAL, "%s: outputs overlap", fn);
  }

  gbf::QkvArgs a = {};
  a.qkv = qkv;
  a.q_w = q_w;
  a.k_w = k_w;
  a.q_b = q_b;
  a.k_b = k_b;
  a.pos = pos;
  a.slots = slots;
  a.q_out = q_out;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.err = error_word();
  a.tokens = tokens;
  a.cache_rows = slots ? cache_rows : (cache_rows > tokens ? cache_rows : tokens);
  a.n_q = n_q_heads;
  a.n_kv = n_kv_heads;
  a.d = head_dim;
  a.norm = norm;
  a.rope = rope;
  a.eps = eps;
  a.n_slots = head_dim / 2;
  // Rotation table: slot p of chunk c pairs (start + j, start + j + w/2) with
  // frequency theta^(-2j / w); 1D is the single chunk w = head_dim.
  int p = 0, start = 0;
  for (int c = 0; c < 3; ++c) {
    a.sec[c] = sec[c];
    const int w = sec[c], half = w / 2;
    for (int j = 0; j < half; ++j, ++p) {
      const double om = std::pow(static_cast<double>(theta), -2.0 * j / w);
      a.omega_hi[p] = static_cast<float>(om);
      a.omega_lo[p] = static_cast<float>(om - static_cast<double>(a.omega_hi[p]));
      a.axis[p] = static_cast<unsigned char>(c);
      a.lo_idx[p] = static_cast<unsigned char>(start + j);
      a.hi_idx[p] = static_cast<unsigned char>(start + j + half);
    }
    start += w;
  }
  return launch_status(gbf::launch_qkv_split_norm_rope(a, static_cast<cudaStream_t>(stream)), fn);
}

}  // namespace

GBF_API int gbf_qkv_split_norm_rope(const void* qkv, int64_t tokens, int n_q_heads, int n_kv_heads, int head_dim,
                                    int norm, const void* q_w, const void* k_w, float eps, int rope,
                                    const int32_t* pos, const int32_t* sections, float theta, void* q_out,
                                    void* k_cache, void* v_cache, const int32_t* slots, int64_t cache_rows,
                                    void* stream) {
  const char* fn = "gbf_qkv_split_norm_rope";
  if (norm != GBF_QKNORM_PER_HEAD && norm != GBF_QKNORM_FULL_WIDTH)
    return fail(GBF_EINVAL, "%s: unknown norm %d", fn, norm);
  return qkv_entry(fn, qkv, tokens, n_q_heads, n_kv_heads, head_dim, norm, q_w, nullptr, k_w, nullptr, eps, rope,
                   pos, sections, theta, q_out, k_cache, v_cache, slots, cache_rows, stream);
}

GBF_API int gbf_qkv_split_layernorm_rope(const void* qkv, int64_t tokens, int n_q_heads, int n_kv_heads,
                                         int head_dim, const void* q_w, const void* q_b, const void* k_w,
                                         const void* k_b, float eps, const int32_t* pos, float theta, void* q_out,
                                         void* k_cache, void* v_cache, const int32_t* slots, int64_t cache_rows,
                                         void* stream) {
  return qkv_entry("gbf_qkv_split_layernorm_rope", qkv, tokens, n_q_heads, n_kv_heads, head_dim,
                   gbf::kQkNormLayerNorm, q_w, q_b, k_w, k_b, eps, GBF_ROPE_1D, pos, nullptr, theta, q_out, k_cache,
                   v_cache, slots, cache_rows, stream);
}

// --------------------------------------------------- gated activation

GBF_API int gbf_gated_act(const void* x, void* y, int64_t rows, int64_t d, int act, void* stream) {
  const char* fn = "gbf_gated_act";
  if (rows < 0 || d <= 0) return fail(GBF_EINVAL, "%s: rows >= 0 and d > 0 are required", fn);
  if (act != GBF_ACT_GELU_TANH && act != GBF_ACT_GELU_ERF && act != GBF_ACT_SILU)
    return fail(GBF_EINVAL, "%s: act must be GELU_TANH, GELU_ERF or SILU (got %d)", fn, act);
  if (d % 8 != 0) return fail(GBF_EALIGN, "%s: d (%lld) must be a multiple of 8", fn, (long long)d);
  if (rows == 0) return ok();
  if (!x || !y) return fail(GBF_EINVAL, "%s: x and y are required", fn);
  if (!aligned16(x) || !aligned16(y)) return fail(GBF_EALIGN, "%s: x and y must be 16-byte aligned", fn);
  if (overlap(x, rows * 2 * d * 2, y, rows * d * 2)) return fail(GBF_EINVAL, "%s: y overlaps x", fn);
  gbf::GatedActArgs a = {};
  a.x = x;
  a.y = y;
  a.rows = rows;
  a.d = d;
  a.act = act;
  return launch_status(gbf::launch_gated_act(a, static_cast<cudaStream_t>(stream)), fn);
}

// ------------------------------------------------ Linear + bias + GELU GEMM

namespace {

// Both Linear entry points: bf16 operands, or E4M3 codes with descales.
int linear_entry(const char* fn, bool fp8, const void* X, float x_scale, const void* W, const float* w_scale,
                 const void* bias, void* Y, int64_t M, int64_t N, int64_t K, int act, void* stream) {
  if (M < 0 || N <= 0 || K <= 0) return fail(GBF_EINVAL, "%s: M >= 0, N > 0, K > 0 required", fn);
  if (act != GBF_ACT_NONE && act != GBF_ACT_GELU_TANH && act != GBF_ACT_GELU_ERF && act != GBF_ACT_SILU)
    return fail(GBF_EINVAL, "%s: unknown activation %d", fn, act);
  if (fp8 && (!(x_scale > 0.0f) || !std::isfinite(x_scale)))
    return fail(GBF_EINVAL, "%s: x_scale must be finite and > 0", fn);
  const int64_t kq = fp8 ? 128 : 64;
  if (K % kq != 0 || N % 16 != 0)
    return fail(GBF_EUNSUPPORTED, "%s: needs K %% %lld == 0 and N %% 16 == 0 (K=%lld, N=%lld)", fn, (long long)kq,
                (long long)K, (long long)N);
  // the kernel indexes rows, columns, tile counts and TMA coordinates with int32
  const int64_t lim = 1LL << 31;
  if (M >= lim || N >= lim || K >= lim) return fail(GBF_EUNSUPPORTED, "%s: M, N and K must be below 2^31", fn);
  if (((M + 127) / 128) * ((N + 255) / 256) >= lim)
    return fail(GBF_EUNSUPPORTED, "%s: more than 2^31 - 1 output tiles of 128 x 256", fn);
  if (M == 0) return ok();
  if (!X || !W || !Y || (fp8 && !w_scale)) return fail(GBF_EINVAL, "%s: X, W, Y (and w_scale) are required", fn);
  if (!aligned16(X) || !aligned16(W) || !aligned16(Y) || (bias && !aligned16(bias)) ||
      (w_scale && !aligned16(w_scale)))
    return fail(GBF_EALIGN, "%s: X, W, Y, bias, w_scale must be 16-byte aligned", fn);
  const int64_t es = fp8 ? 1 : 2;
  const int64_t yb = M * N * 2;
  if (overlap(Y, yb, X, M * K * es) || overlap(Y, yb, W, N * K * es) || overlap(Y, yb, bias, N * 2) ||
      overlap(Y, yb, w_scale, fp8 ? N * 4 : 0))
    return fail(GBF_EINVAL, "%s: Y overlaps an input", fn);
  gbf::GemmArgs a = {};
  a.x = X;
  a.w = W;
  a.bias = bias;
  a.y = Y;
  a.w_scale = w_scale;
  a.x_scale = x_scale;
  a.fp8 = fp8 ? 1 : 0;
  a.err = error_word();
  a.m = M;
  a.n = N;
  a.k = K;
  a.act = act;
  const char* why = nullptr;
  cudaError_t e = gbf::launch_linear_bias_gelu(a, static_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess && why) return fail(GBF_ELAUNCH, "%s: %s (%s)", fn, why, cudaGetErrorString(e));
  return launch_status(e, fn);
}

}  // namespace

GBF_API int gbf_linear_bias_gelu(const void* X, const void* W, const void* bias, void* Y, int64_t M, int64_t N,
                                 int64_t K, int act, void* stream) {
  return linear_entry("gbf_linear_bias_gelu", false, X, 1.0f, W, nullptr, bias, Y, M, N, K, act, stream);
}

GBF_API int gbf_linear_fp8_act(const uint8_t* Xq, float x_scale, const uint8_t* Wq, const float* w_scale,
                               const void* bias, void* Y, int64_t M, int64_t N, int64_t K, int act, void* stream) {
  return linear_entry("gbf_linear_fp8_act", true, Xq, x_scale, Wq, w_scale, bias, Y, M, N, K, act, stream);
}

// ------------------------------------------------ norm weight pre-fold

GBF_API int gbf_fold_norm_weight(const void* W, const void* gamma, int gemma_style, int64_t out_ch, int64_t inner,
                                 void* W_out, void* stream) {
  const char* fn = "gbf_fold_norm_weight";
  if (out_ch < 0 || inner <= 0) return fail(GBF_EINVAL, "%s: out_ch >= 0 and inner > 0 required", fn);
  if (gemma_style != 0 && gemma_style != 1) return fail(GBF_EINVAL, "%s: gemma_style must be 0 or 1", fn);
  if (out_ch == 0) return ok();
  if (!W || !gamma || !W_out) return fail(GBF_EINVAL, "%s: W, gamma and W_out are required", fn);
  const int64_t wb = out_ch * inner * 2;
  if (W_out != W && overlap(W_out, wb, W, wb)) return fail(GBF_EINVAL, "%s: W_out partially overlaps W", fn);
  if (overlap(W_out, wb, gamma, inner * 2)) return fail(GBF_EINVAL, "%s: W_out overlaps gamma", fn);
  gbf::NormFoldArgs a = {};
  a.w = W;
  a.gamma = gamma;
  a.w_out = W_out;
  a.out_ch = out_ch;
  a.inner = inner;
  a.gemma = gemma_style;
  return launch_status(gbf::launch_fold_norm_weight(a, static_cast<cudaStream_t>(stream)), fn);
}

// ------------------------------------------------------------ BN folding

GBF_API int gbf_bn_fold(const void* W, const void* b, const float* gamma, const float* beta, const float* mean,
                        const float* var, float eps, int64_t out_ch, int64_t inner, void* W_out, void* b_out,
                        void* stream) {
  const char* fn = "gbf_bn_fold";
  if (out_ch < 0 || inner <= 0) return fail(GBF_EINVAL, "%s: out_ch >= 0 and inner > 0 required", fn);
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return fail(GBF_EINVAL, "%s: eps must be finite and >= 0", fn);
  if (out_ch == 0) return ok();
  if (!W || !gamma || !beta || !mean || !var || !W_out || !b_out)
    return fail(GBF_EINVAL, "%s: W, gamma, beta, mean, var, W_out, b_out are required", fn);
  const int64_t wb = out_ch * inner * 2, cb = out_ch * 4, bb = out_ch * 2;
  if (W_out != W && overlap(W_out, wb, W, wb)) return fail(GBF_EINVAL, "%s: W_out partially overlaps W", fn);
  const void* ins[] = {b, gamma, beta, mean, var};
  const int64_t il[] = {bb, cb, cb, cb, cb};
  for (int i = 0; i < 5; ++i)
    if (overlap(W_out, wb, ins[i], il[i]) || overlap(b_out, bb, ins[i], il[i]) || overlap(b_out, bb, W, wb))
      return fail(GBF_EINVAL, "%s: an output overlaps an input", fn);
  if (overlap(b_out, bb, W_out, wb)) return fail(GBF_EINVAL, "%s: b_out overlaps W_out", fn);
  gbf::BnFoldArgs a = {};
  a.w = W;
  a.b = b;
  a.gamma = gamma;
  a.beta = beta;
  a.mean = mean;
  a.var = var;
  a.w_out = W_out;
  a.b_out = b_out;
  a.eps = eps;
  a.out_ch = out_ch;
  a.inner = inner;
  return launch_status(gbf::launch_bn_fold(a, static_cast<cudaStream_t>(stream)), fn);
}

// ------------------------------------------------------------- copy probe

GBF_API int gbf_copy(const void* src, void* dst, int64_t bytes, void* stream) {
  const char* fn = "gbf_copy";
  if (bytes < 0) return fail(GBF_EINVAL, "%s: bytes must be >= 0", fn);
  if (bytes == 0) return ok();
  if (!src || !dst) return fail(GBF_EINVAL, "%s: src and dst are required", fn);
  if (!aligned16(src) || !aligned16(dst)) return fail(GBF_EALIGN, "%s: src and dst must be 16-byte aligned", fn);
  if (overlap(src, bytes, dst, bytes)) return fail(GBF_EINVAL, "%s: src and dst overlap", fn);
  return launch_status(gbf::launch_copy(src, dst, bytes, static_cast<cudaStream_t>(stream)), fn);
}

// --------------------------------------------------- failure-path self-test

GBF_API int gbf_selftest_bounded_wait(void* stream) {
  unsigned int* err = error_word();
  if (!err) return fail(GBF_ELAUNCH, "gbf_selftest_bounded_wait: no device error word (no CUDA device?)");
  return launch_status(gbf::launch_bounded_wait_selftest(err, static_cast<cudaStream_t>(stream)),
                       "gbf_selftest_bounded_wait");
}

// ----------------------------------------------------------- device status

GBF_API int gbf_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(GBF_ELAUNCH, "gbf_device_status: %s", cudaGetErrorString(e));
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_device_error, sizeof word);
  if (e != cudaSuccess) return fail(GBF_ELAUNCH, "gbf_device_status: %s", cudaGetErrorString(e));
  if (word) {
    const unsigned int zero = 0;
    cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
  }
  if (word & gbf::DEV_ERR_MBAR_TIMEOUT)
    return fail(GBF_ETIMEOUT, "gbf_device_status: a bounded wait inside a kernel gave up (word 0x%x)", word);
  if (word) return fail(GBF_EDEVICE, "gbf_device_status: device fault word 0x%x (bit 0: cache slot out of range; "
                         "bit 2: a GEMM CTA pair got different TMEM bases)", word);
  return ok();
}

}  // extern "C"
