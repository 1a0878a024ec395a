/*
 * gbfuse -- fused memory-bound operator chains and a GEMM with a fused epilogue
 * for NVIDIA GB300 (sm_103a).  C ABI of libgbfuse.so.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named "device" are CUDA device (HBM) addresses; `stream` is a
 *    cudaStream_t (NULL = the legacy default stream).  Work is enqueued on
 *    `stream` and the call returns without synchronising.
 *  - Ownership: the caller allocates and frees every buffer.  The library
 *    never allocates or frees device memory.  Its only device state is one
 *    32-bit error word per device, read by gbf_device_status().
 *  - Tensors are dense and row-major.  bf16 = bfloat16 (round to nearest even
 *    on every store); e4m3 = OCP FP8 E4M3 "fn" (max 448, no infinities).
 *  - Alignment: every tensor pointer whose rows are accessed as 16-byte
 *    vectors must be 16-byte aligned (GBF_EALIGN otherwise), as stated per call.
 *  - Errors: a non-zero return means nothing was enqueued (argument errors) or
 *    the launch failed (GBF_ELAUNCH).  gbf_last_error() returns a message for
 *    the calling thread's last failure.  No call throws or aborts.
 *  - Data-dependent faults found on the device (a KV-cache slot out of range,
 *    a bounded wait that gave up) skip the offending writes and set a bit in
 *    the device error word instead of faulting; gbf_device_status() returns it.
 *
 * Citations name the web page and section each operation follows:
 *   FlashRT -- "FlashRT 跨层融合深度解析：从 RMSNorm+QKV 到被证伪的死胡同优化模式"
 *   OpenPPL -- "OpenPPL算子融合深度解析：从图优化到推理性能提升"
 *   HowTo   -- the operator-fusion how-to on discosf.com (HTML title
 *              "企业官网建设流程全解析", body on 算子融合推理优化)
 *   RFC     -- "RFC：自动融合: 扩展统一 Pattern Matcher 覆盖量化融合与 GMM/MM+激活"
 */
#ifndef GBFUSE_H
#define GBFUSE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GBF_API __attribute__((visibility("default")))

typedef enum {
  GBF_OK = 0,
  GBF_EINVAL = -1,       /* a null, negative, overlapping or inconsistent argument */
  GBF_EALIGN = -2,       /* a pointer or extent breaks the 16-byte vector rule */
  GBF_EUNSUPPORTED = -3, /* a shape outside what the kernels implement (no fallback) */
  GBF_ELAUNCH = -4,      /* the CUDA launch itself failed */
  GBF_ETIMEOUT = -5,     /* (device status) a bounded wait inside a kernel gave up */
  GBF_EDEVICE = -6       /* (device status) a data-dependent fault was caught on the device */
} gbf_status;

typedef enum { GBF_NORM_WEIGHT = 0, GBF_NORM_NOWEIGHT = 1, GBF_NORM_ADA = 2 } gbf_norm_mode;
typedef enum { GBF_QKNORM_PER_HEAD = 0, GBF_QKNORM_FULL_WIDTH = 1 } gbf_qknorm;
typedef enum { GBF_ROPE_1D = 0, GBF_ROPE_3D = 1 } gbf_rope;
typedef enum { GBF_ACT_NONE = 0, GBF_ACT_GELU_TANH = 1, GBF_ACT_GELU_ERF = 2, GBF_ACT_SILU = 3 } gbf_act;

/*
 * gbf_add_rmsnorm_fp8 -- residual add (optionally gated), RMSNorm / _noweight /
 * AdaRMSNorm, static-scale FP8 quantisation, in one read and one write.
 * FlashRT §2.1 (residual + RMSNorm + FP8 "three in one"; `_noweight`: the norm
 * weight pre-folded into the next GEMM) and §3 (gate_res_adarms_fp8_static:
 * gate multiply + residual + AdaRMSNorm + FP8 + descale); OpenPPL §3.3 (the
 * residual Add as an epilogue).
 *
 * Per row i of `rows` and column j of `hidden`, in float32:
 *   r        = x + res_in                      (gate == NULL)
 *            = res_in + gate[j] * x            (gate != NULL)
 *   res_out  = bf16(r)                         the new residual stream
 *   inv      = 1 / sqrt(mean_j(res_out^2) + eps)   (the norm reads the bf16 residual)
 *   y        = res_out * inv * weight[j]                         GBF_NORM_WEIGHT
 *            = res_out * inv                                     GBF_NORM_NOWEIGHT
 *            = res_out * inv * (1 + ada_scale[j]) + ada_shift[j] GBF_NORM_ADA
 *   q_out    = e4m3(y / fp8_scale), round to nearest even, saturated to +-448
 * y never reaches memory.  fp8_scale is the descale: dequantised = code * fp8_scale.
 *
 * x, res_in, res_out: device bf16 [rows, hidden]; gate, weight, ada_scale,
 * ada_shift: device bf16 [hidden] (broadcast over rows; weight required for
 * WEIGHT, ada_scale and ada_shift for ADA, ignored otherwise); q_out: device
 * uint8 [rows, hidden].  res_out may equal res_in (in-place update of the
 * residual stream); any other overlap of an output with an input is GBF_EINVAL.
 * Requires hidden % 8 == 0, hidden <= 32768 and 16-byte aligned pointers
 * (GBF_EALIGN / GBF_EUNSUPPORTED otherwise); eps >= 0; fp8_scale > 0 and finite.
 * rows == 0 enqueues nothing.  The launch allows programmatic dependent
 * launch, so back-to-back calls on one stream overlap their launch latency.
 */
GBF_API int gbf_add_rmsnorm_fp8(const void* x, const void* res_in, void* res_out, const void* gate,
                                int mode, const void* weight, const void* ada_scale, const void* ada_shift,
                                uint8_t* q_out, int64_t rows, int64_t hidden, float eps, float fp8_scale,
                                void* stream);

/*
 * gbf_qkv_split_norm_rope -- packed QKV split, Q/K RMSNorm, rotate_half RoPE,
 * Q write and K/V cache write in one pass; V passes through bit for bit.
 * FlashRT §2.2 (Qwen3/GROOT q_norm -> RoPE -> Q, k_norm -> RoPE -> KV cache;
 * Wan packed QKV split + two RMSNorms + 3D RoPE; "Q/K norm -> RoPE, V direct");
 * RFC §2.4 / §3.6 (RMSNorm + RoPE with an optional cache write); OpenPPL §3.2
 * (the packed [Q | K | V] output of the merged QKV GEMM).
 *
 * qkv: device bf16 [tokens, (n_q_heads + 2 n_kv_heads) * head_dim], each row
 *   all Q heads, then all K heads, then all V heads, heads contiguous.
 * norm: GBF_QKNORM_PER_HEAD normalises each head over head_dim with q_w/k_w of
 *   [head_dim]; GBF_QKNORM_FULL_WIDTH normalises all Q (all K) values of a
 *   token together with q_w [n_q_heads*head_dim], k_w [n_kv_heads*head_dim]
 *   (device bf16).  inv = 1/sqrt(mean(x^2) + eps); u = x * inv * w in float32.
 * rope: GBF_ROPE_1D rotates pairs (j, j + head_dim/2) by pos[t] * theta^(-2j/head_dim)
 *   with pos device int32 [tokens]:  o[j] = u[j] cos - u[j+h] sin,
 *   o[j+h] = u[j+h] cos + u[j] sin.  GBF_ROPE_3D cuts each head into contiguous
 *   chunks of widths sections[0..2] (host int32[3], even, summing to head_dim),
 *   chunk c rotating inside itself (pairs j, j + sections[c]/2, frequencies
 *   theta^(-2j/sections[c])) by the token's grid coordinate pos[t*3 + c] (pos
 *   device int32 [tokens, 3]).  sections is ignored for 1D and may be NULL.
 * q_out: device bf16 [tokens, n_q_heads, head_dim].
 * k_cache, v_cache: device bf16 [cache_rows, n_kv_heads, head_dim]; token t
 *   writes row slots[t] (slots device int32 [tokens]) or row t when slots is
 *   NULL (then cache_rows >= tokens is required).  A slot outside
 *   [0, cache_rows) skips that token's K/V writes and sets the device error word.
 * Requires head_dim % 16 == 0 and head_dim <= 256; per-head norm needs a
 * power-of-two head_dim; 16-byte aligned tensors; eps >= 0; theta > 0.
 * Unless norm is per head, rope is 1D and head_dim is 64, 128 or 256, a token's
 * row is staged on chip and (6 n_q_heads + 8 n_kv_heads) * head_dim must be
 * <= 196608 (GBF_EUNSUPPORTED otherwise).  The staged kernel's waits for its
 * row copies are bounded: a wait that gives up sets the device error word
 * (gbf_device_status() returns GBF_ETIMEOUT) and the outputs are undefined.
 * Outputs may not overlap each other or the inputs (GBF_EINVAL).
 */
GBF_API int gbf_qkv_split_norm_rope(const void* qkv, int64_t tokens, int n_q_heads, int n_kv_heads,
                                    int head_dim, int norm, const void* q_w, const void* k_w, float eps,
                                    int rope, const int32_t* pos, const int32_t* sections, float theta,
                                    void* q_out, void* k_cache, void* v_cache, const int32_t* slots,
                                    int64_t cache_rows, void* stream);

/*
 * gbf_qkv_split_layernorm_rope -- the same single pass as
 * gbf_qkv_split_norm_rope with a per-head LayerNorm in place of the RMSNorm:
 * FlashRT §2.2 (Chameleon prefill: LayerNorm(Q) + LayerNorm(K) + two
 * rotate_half RoPEs in one kernel, each lane holding both members of its
 * rotation pairs).
 *
 * Per head of width head_dim: mean = Σx / D, var = Σ(x - mean)² / D,
 * u = (x - mean) / sqrt(var + eps) * w + b in float32, then 1D rotate_half
 * RoPE by pos[t] * theta^(-2j/head_dim) exactly as gbf_qkv_split_norm_rope.
 * q_w, k_w: device bf16 [head_dim]; q_b, k_b: device bf16 [head_dim] or NULL
 * (zero bias).  All other arguments, layouts, the V copy, slots and the device
 * error word are those of gbf_qkv_split_norm_rope with norm per head and
 * rope 1D.  Requires head_dim 64, 128 or 256 (GBF_EUNSUPPORTED otherwise);
 * 16-byte aligned tensors including the biases; eps >= 0; theta > 0.
 */
GBF_API int gbf_qkv_split_layernorm_rope(const void* qkv, int64_t tokens, int n_q_heads, int n_kv_heads,
                                         int head_dim, const void* q_w, const void* q_b, const void* k_w,
                                         const void* k_b, float eps, const int32_t* pos, float theta, void* q_out,
                                         void* k_cache, void* v_cache, const int32_t* slots, int64_t cache_rows,
                                         void* stream);

/*
 * gbf_linear_bias_gelu -- Y = act(X W^T + bias) on the tcgen05 tensor cores,
 * float32 accumulation in tensor memory, bias and GELU applied to the
 * accumulator tile before the single bf16 store.  OpenPPL §4.3 (epilogue:
 * += bias, GELU 0.5 a (1 + tanh(0.7978845608 (a + 0.044715 a^3)))); RFC §3.5
 * (npu_linear: Linear + activation); the graph-autofusion article's
 * MatMul -> BiasAdd -> activation pattern (three HBM passes become one).
 *
 * X: device bf16 [M, K]; W: device bf16 [N, K] (nn.Linear [out, in] layout);
 * bias: device bf16 [N] or NULL (zero); Y: device bf16 [M, N].
 * act: GBF_ACT_GELU_TANH, GBF_ACT_NONE, GBF_ACT_GELU_ERF (0.5 a (1 + erf(a /
 * sqrt 2)), the exact GELU of RFC §3.6) or GBF_ACT_SILU (a / (1 + exp(-a))).
 * Requires K % 64 == 0, N % 16 == 0, M >= 1 and 16-byte aligned X, W, Y
 * (GBF_EUNSUPPORTED / GBF_EALIGN otherwise); Y may not overlap X, W or bias.
 * One launch: when M spans more than one 128-row tile, clusters of two CTAs
 * run as tcgen05 CTA pairs on adjacent 128-row tiles.  The kernel's pipeline
 * waits are bounded: a wait that gives up sets the device error word
 * (gbf_device_status() returns GBF_ETIMEOUT); a CTA pair handed two different
 * tensor-memory bases does no work and sets it too (GBF_EDEVICE).
 */
GBF_API int gbf_linear_bias_gelu(const void* X, const void* W, const void* bias, void* Y, int64_t M,
                                 int64_t N, int64_t K, int act, void* stream);

/*
 * gbf_gated_act -- y = act(gate) * up in one pass: RFC §2.4 / §3.6 (silu
 * gating -> npu_swiglu, gelu(x) * gate -> npu_gelu_mul; two elementwise ops
 * whose intermediate act(gate) never reaches HBM).
 *
 * x: device bf16 [rows, 2d], each row the gate projection (columns 0..d-1)
 * then the up projection (columns d..2d-1); y: device bf16 [rows, d].
 * act: GBF_ACT_SILU (SwiGLU), GBF_ACT_GELU_TANH or GBF_ACT_GELU_ERF (GELU x
 * Mul), else GBF_EINVAL.  Float32 arithmetic, one bf16 rounding per output.
 * Requires d % 8 == 0 and 16-byte aligned x, y (GBF_EALIGN); y may not
 * overlap x (GBF_EINVAL).
 */
GBF_API int gbf_gated_act(const void* x, void* y, int64_t rows, int64_t d, int act, void* stream);

/*
 * gbf_linear_fp8_act -- Y = act((Xq * x_scale) (Wq * w_scale)^T + bias): the
 * quantised MatMul + activation of RFC §2.1 / §3.4 (npu_quant_matmul_gelu
 * with its activation and weight scales), on the tcgen05 tensor cores
 * (kind::f8f6f4, E4M3 x E4M3, float32 accumulation in tensor memory); the
 * descales, bias and activation are applied to the accumulator tile before
 * the single bf16 store.  Xq are E4M3 codes such as gbf_add_rmsnorm_fp8
 * writes (code * x_scale is the value).
 *
 * Xq: device uint8 E4M3 codes [M, K]; x_scale: the activations' descale
 * (finite, > 0); Wq: device uint8 E4M3 codes [N, K] (nn.Linear [out, in]
 * layout); w_scale: device float32 [N], the descale of each weight row; bias:
 * device bf16 [N] or NULL; Y: device bf16 [M, N]; act as gbf_linear_bias_gelu.
 * Requires K % 128 == 0, N % 16 == 0 and 16-byte aligned Xq, Wq, w_scale, Y
 * (GBF_EUNSUPPORTED / GBF_EALIGN); Y may not overlap an input.  Waits are
 * bounded as in gbf_linear_bias_gelu.
 */
GBF_API int gbf_linear_fp8_act(const uint8_t* Xq, float x_scale, const uint8_t* Wq, const float* w_scale,
                               const void* bias, void* Y, int64_t M, int64_t N, int64_t K, int act, void* stream);

/*
 * gbf_fold_norm_weight -- move a norm's per-column weight into the next
 * Linear: W_out[c, k] = W[c, k] * (1 + gamma[k]) (gemma_style = 1, the
 * Gemma-style weight that FlashRT §3's `_noweight` RMSNorm leaves to the
 * next GEMM) or W[c, k] * gamma[k] (gemma_style = 0).  Binary32, one IEEE
 * operation per step (the sum, then the product), then one bf16 rounding:
 * bit-reproducible.
 *
 * W: device bf16 [out_ch, inner]; gamma: device bf16 [inner]; W_out: device
 * bf16 [out_ch, inner], may equal W (in place); other overlaps GBF_EINVAL.
 */
GBF_API int gbf_fold_norm_weight(const void* W, const void* gamma, int gemma_style, int64_t out_ch, int64_t inner,
                                 void* W_out, void* stream);

/*
 * gbf_bn_fold -- fold an inference BatchNorm into the weights of the producing
 * Conv or Linear.  OpenPPL §3.1 (scale = gamma / sqrt(var + eps);
 * W' = W * scale per output channel; b' = (b - mean) * scale + beta; missing
 * bias = 0) and §6.2 (fold in FP32, then store half); HowTo §2.1 (scale first,
 * bias from the old b) and §4.1 (eps from the model).
 *
 * W: device bf16 [out_ch, inner] (a conv weight [Cout, Cin, kh, kw] is passed
 * with inner = Cin*kh*kw); b: device bf16 [out_ch] or NULL; gamma, beta, mean,
 * var: device float32 [out_ch]; W_out: device bf16 [out_ch, inner]; b_out:
 * device bf16 [out_ch] (always written).  Every step is one IEEE binary32
 * operation, round to nearest, no fused multiply-add, then one bf16 rounding,
 * so the result is bit-reproducible.  W_out may equal W (in place); other
 * overlaps are GBF_EINVAL.  eps >= 0 (taken from the model; never assumed).
 * Any inner >= 1 works; rows with inner % 8 == 0 and 16-byte aligned W, W_out
 * use 16-byte vectors.
 */
GBF_API int gbf_bn_fold(const void* W, const void* b, const float* gamma, const float* beta,
                        const float* mean, const float* var, float eps, int64_t out_ch, int64_t inner,
                        void* W_out, void* b_out, void* stream);

/*
 * gbf_copy -- device-to-device copy of `bytes` bytes (src, dst device,
 * 16-byte aligned, not overlapping).  The measured HBM bandwidth of this
 * kernel is the roofline the memory-bound kernels are reported against.
 */
GBF_API int gbf_copy(const void* src, void* dst, int64_t bytes, void* stream);

/*
 * gbf_device_status -- synchronise `stream`, then read and clear the current
 * device's error word.  Returns GBF_OK, GBF_ETIMEOUT (a bounded wait gave up)
 * or GBF_EDEVICE (a cache slot was out of range, or the two CTAs of a GEMM
 * tensor-core pair were given different TMEM bases), or GBF_ELAUNCH if the
 * synchronisation itself reported a CUDA error.
 */
GBF_API int gbf_device_status(void* stream);

/*
 * gbf_selftest_bounded_wait -- exercises the device-side failure path: a
 * one-thread kernel waits, through the same bounded mbarrier wait the
 * pipelined kernels use, on a barrier nothing arrives at.  After about one
 * second the wait gives up, sets the timeout bit of the device error word and
 * the kernel returns normally; the next gbf_device_status(stream) returns
 * GBF_ETIMEOUT and the context stays usable.  Enqueues asynchronously.
 */
GBF_API int gbf_selftest_bounded_wait(void* stream);

/* Message for the calling thread's most recent non-OK return ("" if none). */
GBF_API const char* gbf_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
GBF_API int gbf_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GBFUSE_H */
