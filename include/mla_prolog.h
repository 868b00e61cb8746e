/*
 * mla_prolog.h -- C ABI of the GB300 (sm_103a) MLA KV prolog library
 * (libmla_prolog.so).
 *
 * The operation is the "KV prolog" of DeepSeek-V2 Multi-head Latent
 * Attention.  Sources (web pages, cited by title and section):
 *
 *   [MIG] "DeepSeek-V2-Lite-Chat MLA KV Prolog 迁移指南：基于 PyPTO 融合算子与
 *         aclgraph 的 NPU 推理优化实践"
 *   [R1]  "DeepSeek-R1或Kimi-K2模型在NPU实现高性能推理"
 *
 * [MIG] §"背景：为什么要迁移 MLA KV Prolog" lists the seven steps this
 * library fuses:
 *   1. kv_a_proj  C = X * W_kva                        [T, hidden] x [hidden, 576]
 *   2. split      compressed_kv = C[:, 0:512], k_pe_raw = C[:, 512:576]
 *   3. RMSNorm    n = compressed_kv / sqrt(mean(compressed_kv^2) + eps) * gamma
 *   4. kv_b_proj  KV = n * W_kvb                       [T, 512] x [512, H*256]
 *   5. reshape + split: KV -> [T, H, 256]; k_nope = [..., 0:128], value = [..., 128:256]
 *   6. RoPE on k_pe_raw at each token's position
 *   7. assemble the head-major outputs k_nope [b,H,s,128], value [b,H,s,128],
 *      k_pe [b,1,s,64]
 * with T = b*s token rows, row t = bi*s + si ([MIG] §"源码级原理：KV Prolog 的
 * 混合优化实现", steps 1 and 5).  Shapes: [MIG] §"精度验证：Golden 对比测试"
 * (hidden 2048, W_kva [2048, 576], W_kvb [512, 4096], gamma [512], eps 1e-6,
 * outputs [1,16,1,128], [1,16,1,128], [1,1,1,64]).
 *
 * Readings taken where the pages are silent (the library and its tests use
 * the same ones):
 *   - RoPE (step 6): [MIG] says only "x*cos + x_rot*sin".  The library uses
 *     the DeepSeek-V2 convention: de-interleave x'[j] = x[2j], x'[32+j] =
 *     x[2j+1] (j < 32), then out = x'*cos[p] + rotate_half(x')*sin[p] with
 *     rotate_half(x') = [-x'[32:64], x'[0:32]].  The output keeps the
 *     de-interleaved order.  cos/sin are caller tables [max_pos, 64] fp32,
 *     read entry by entry (any rope scaling is the caller's business).
 *   - Accumulation is fp32; steps 1-3 stay in fp32 on chip and n is rounded
 *     once to the I/O dtype as the operand of step 4; outputs are rounded
 *     to nearest even.
 *   - W8A8 ([R1] §"权重转换" names the W8A8 weight modes; the fused "MLA
 *     prolog" switch enable_mla_prolog is in [R1] §"推理执行"): int8 weights
 *     with one fp32 scale per output channel, per-token dynamic symmetric
 *     int8 activations, int32 accumulation, dequantisation acc*s_x*s_w.
 *
 * Conventions for every entry point:
 *   - The caller owns every tensor.  Device pointers must be 16-byte
 *     aligned (else MLA_ERR_MISALIGNED) and the tensors dense row-major in
 *     the layouts given.  Weights use the pre-transposed [in, out] layout of
 *     [MIG] §"源码级原理" step 1.  Optionally a handle keeps a re-laid-out
 *     copy of W_kva / W_kvb for the decode kernel
 *     (mla_kv_prolog_prepare_weights).
 *   - A handle owns only its device workspace (allocated by create, freed
 *     by destroy).  run never allocates and never synchronises: it enqueues
 *     its kernels on `stream` and returns.  Launch failures come back as
 *     MLA_ERR_CUDA (text in mla_last_cuda_error()).
 *   - Faults the device detects (a position outside [0, max_pos), which is
 *     clamped so that no out-of-bounds read happens; a device wait that ran
 *     out of its time budget) are recorded in a status word in the
 *     workspace; mla_kv_prolog_status() reports and clears it.
 *   - A handle is not safe to use from two streams at once (one workspace).
 */
#ifndef MLA_PROLOG_H
#define MLA_PROLOG_H

#include <stdint.h>
#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_PROLOG_ABI_VERSION 1

typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,     /* null handle/pointer, b or s < 0, bad config value      */
  MLA_ERR_UNSUPPORTED = 2,     /* dimensions outside what the kernels implement          */
  MLA_ERR_TOO_MANY_TOKENS = 3, /* b*s > config.max_tokens                                 */
  MLA_ERR_MISALIGNED = 4,      /* a device pointer not 16-byte aligned                    */
  MLA_ERR_CUDA = 5,            /* a CUDA runtime call failed; see mla_last_cuda_error()   */
  MLA_ERR_DEVICE_TIMEOUT = 6,  /* a device-side wait ran past config.spin_budget_ns       */
  MLA_ERR_BAD_POSITION = 7,    /* a position outside [0, max_pos) was seen (and clamped)  */
  MLA_ERR_NO_MEMORY = 8,       /* workspace allocation failed in create                   */
  MLA_ERR_WRONG_MODE = 9,      /* run of one quant mode on a handle made for the other    */
  MLA_ERR_BAD_SLOT = 10        /* a paged-cache slot past the cache was seen (row dropped)*/
} mla_status;

typedef enum mla_dtype { MLA_F16 = 0, MLA_BF16 = 1 } mla_dtype;
typedef enum mla_quant { MLA_QUANT_NONE = 0, MLA_QUANT_W8A8 = 1 } mla_quant;

/* Kernel-path selection.  AUTO picks by token count T (the T-bucketed
 * selection that replaces the short/long dynamic selection of [MIG]
 * §"源码级原理", last paragraph): the fused split-K decode kernel for small
 * T, the tcgen05 tensor-core prefill kernel for large T.  DECODE / PREFILL
 * force one path (for tests and benchmarks).  On the decode path, launches
 * of at most 16 rows on the packed snapshot (mla_kv_prolog_prepare_weights)
 * with dtype outputs take the cluster kernel where the shape allows it
 * (hidden 2048, the V2-Lite shape, and a device that holds 16-CTA
 * clusters); DECODE_GRID forces the decode path without it (the grid-barrier
 * kernel for every launch).  last_path reports DECODE for both. */
typedef enum mla_path {
  MLA_PATH_AUTO = 0,
  MLA_PATH_DECODE = 1,
  MLA_PATH_PREFILL = 2,
  MLA_PATH_DECODE_GRID = 3
} mla_path;

typedef struct mla_prolog_config {
  int hidden;       /* model width: 2048 (V2-Lite), 7168 (R1); multiple of 64          */
  int kv_lora_rank; /* latent width; must be 512                                        */
  int rope_dim;     /* rope width; must be 64                                           */
  int num_heads;    /* H >= 1 (16 V2-Lite, 128 R1)                                      */
  int nope_dim;     /* must be 128                                                      */
  int v_dim;        /* must be 128                                                      */
  int dtype;        /* mla_dtype of hidden, fp weights, gamma and all outputs           */
  float eps;        /* RMSNorm epsilon (1e-6)                                           */
  int max_tokens;   /* largest b*s any run on this handle will pass (sizes workspace)  */
  int max_pos;      /* rows of the cos/sin tables                                       */
  int quant;        /* mla_quant                                                        */
  int q_lora_rank;  /* W8A8 only: q latent width (1536); multiple of 64, <= 3520        */
  unsigned long long spin_budget_ns; /* device wait limit; 0 selects 1 s               */
} mla_prolog_config;

typedef struct mla_prolog_s* mla_prolog_t;

/* Validate `cfg`, allocate the workspace (split-K partials, normalised
 * latent rows, barrier counters, status word) on the current device and
 * return a handle in *out.  Errors: MLA_ERR_INVALID_ARG (null, non-positive
 * sizes, eps < 0), MLA_ERR_UNSUPPORTED (kv_lora_rank != 512, rope_dim != 64,
 * nope/v != 128, hidden % 64 != 0, W8A8 with dtype != BF16, q_lora_rank
 * % 64 != 0 or q_lora_rank > 3520), MLA_ERR_NO_MEMORY, MLA_ERR_CUDA. */
mla_status mla_kv_prolog_create(const mla_prolog_config* cfg, mla_prolog_t* out);

/* Enqueue one KV prolog (steps 1-7 above) of T = b*s token rows on `stream`.
 *   hidden_states [b*s, hidden]        dtype      (row t = bi*s + si)
 *   positions     [b*s]                int32      rope position of each row
 *   W_kva         [hidden, 576]        dtype      pre-transposed kv_a_proj_with_mqa
 *   gamma_kv      [512]                dtype      kv_a_layernorm weight
 *   W_kvb         [512, H*256]         dtype      pre-transposed kv_b_proj
 *   cos_table, sin_table [max_pos, 64] float32
 *   k_nope        [b, H, s, 128]       dtype      output
 *   value         [b, H, s, 128]       dtype      output
 *   k_pe          [b, 1, s, 64]        dtype      output
 * T = 0 is a no-op returning MLA_OK.  Errors: MLA_ERR_INVALID_ARG,
 * MLA_ERR_TOO_MANY_TOKENS, MLA_ERR_MISALIGNED, MLA_ERR_WRONG_MODE (handle
 * created for W8A8), MLA_ERR_CUDA (also when the device cannot hold all CTAs
 * of the decode kernel at once).  The decode kernel's CTAs wait for one
 * another at grid barriers; it is launched as a plain (not cooperative)
 * launch, so if other work on the device keeps some of its CTAs from
 * starting for longer than spin_budget_ns, the others give up and the call
 * reports MLA_ERR_DEVICE_TIMEOUT through mla_kv_prolog_status.  Device-side
 * faults: see mla_kv_prolog_status. */
mla_status mla_kv_prolog_run(mla_prolog_t h, int b, int s, const void* hidden_states,
                             const int32_t* positions, const void* W_kva, const void* gamma_kv,
                             const void* W_kvb, const float* cos_table, const float* sin_table,
                             void* k_nope, void* value, void* k_pe, cudaStream_t stream);

/* int8 KV cache (the C8 cache of the W8A8C8 mode, [R1] §权重转换): the
 * prolog of mla_kv_prolog_run with step 7 storing int8 codes instead of
 * dtype values.  Per output channel c a static fp32 scale s_c (calibrated
 * by the caller); the code of a value x -- the value the dtype output would
 * hold -- is clamp(rint(x * (1 / s_c)), -127, 127), each step an IEEE fp32
 * operation (rint half to even); x ~= code * s_c.
 *   k_scale [H*128], v_scale [H*128], kpe_scale [64]   float32 (head-major:
 *   channel hh*128 + e of k_nope / value)
 *   k_nope [b, H, s, 128], value [b, H, s, 128], k_pe [b, 1, s, 64]  int8 outputs
 * Other arguments, errors and path selection as for mla_kv_prolog_run. */
mla_status mla_kv_prolog_run_c8(mla_prolog_t h, int b, int s, const void* hidden_states,
                                const int32_t* positions, const void* W_kva, const void* gamma_kv,
                                const void* W_kvb, const float* cos_table, const float* sin_table,
                                const float* k_scale, const float* v_scale, const float* kpe_scale,
                                int8_t* k_nope, int8_t* value, int8_t* k_pe, cudaStream_t stream);

/* Paged KV cache: the prolog of mla_kv_prolog_run with step 7 writing into
 * block-paged caches instead of the dense [b, H, s, d] outputs -- the
 * scatter into the attention's KV cache that follows the prolog.  Token row
 * t = bi*s + si goes to slot slot_mapping[t] = block * page_size + offset:
 *   k_cache   [num_blocks, H, page_size, 128]  dtype   k_nope of the row at [block, :, offset, :]
 *   v_cache   [num_blocks, H, page_size, 128]  dtype   value
 *   kpe_cache [num_blocks, 1, page_size, 64]   dtype   k_pe
 *   slot_mapping [b*s] int32; a negative slot drops the row (padding)
 * Other entries of the caches are left untouched.  A slot at or past
 * num_blocks * page_size drops the row and is reported by
 * mla_kv_prolog_status as MLA_ERR_BAD_SLOT.  Other arguments, errors and
 * path selection as for mla_kv_prolog_run. */
mla_status mla_kv_prolog_run_paged(mla_prolog_t h, int b, int s, const void* hidden_states,
                                   const int32_t* positions, const void* W_kva,
                                   const void* gamma_kv, const void* W_kvb,
                                   const float* cos_table, const float* sin_table,
                                   const int32_t* slot_mapping, int page_size, int num_blocks,
                                   void* k_cache, void* v_cache, void* kpe_cache,
                                   cudaStream_t stream);

/* Latent-cache variant: enqueue steps 1, 2, 3 and 6 of the prolog only --
 * kv_a_proj, split, RMSNorm of compressed_kv and RoPE of k_pe -- for an
 * attention that absorbs kv_b_proj into its query / output projections and
 * caches the normalised latent instead of k_nope / value.  The pages'
 * prolog ([MIG] §背景) ends with kv_b_proj; this entry stops before it.
 *   hidden_states, positions, W_kva, gamma_kv, cos_table, sin_table as for
 *   mla_kv_prolog_run
 *   latent        [b*s, 512]           dtype      output: RMSNorm(compressed_kv) * gamma
 *   k_pe          [b, 1, s, 64]        dtype      output (identical to mla_kv_prolog_run's)
 * Same path selection, packed W_kva snapshot (matched on W_kva alone),
 * errors and device status as mla_kv_prolog_run. */
mla_status mla_kv_prolog_run_latent(mla_prolog_t h, int b, int s, const void* hidden_states,
                                    const int32_t* positions, const void* W_kva,
                                    const void* gamma_kv, const float* cos_table,
                                    const float* sin_table, void* latent, void* k_pe,
                                    cudaStream_t stream);

/* Take a snapshot of W_kva [hidden, 576] and W_kvb [512, H*256] (layouts
 * as for mla_kv_prolog_run) in the decode kernel's own layout: every CTA's
 * kv_a tile and kv_b column slice become one contiguous block, with the
 * 16-byte chunks of each row permuted so that the kernel's shared-memory
 * reads meet no bank conflict.  The kernel then fetches them with a few
 * large bulk copies instead of many narrow strided rows (the tile rows of
 * W_kva are 64 bytes wide).  The layout is a property of this library
 * only: the pages ([MIG] §"源码级原理" step 1) use the plain [in, out]
 * layout, and the arithmetic is unchanged (same products, same order).
 *   Later mla_kv_prolog_run calls on this handle whose W_kva and W_kvb
 *   pointers equal these two take the snapshot on the decode path; other
 *   pointers (and the prefill path) read the weights as passed.  The copy
 *   is made on `stream` (two kernels); call again after changing the
 *   weights in place.  Passing NULL for both forgets the snapshot.
 *   The first call allocates hidden*576*2 + 512*H*256*2 bytes of device
 *   memory owned by the handle (freed by destroy), plus another 512*H*256*2
 *   where the cluster decode kernel applies (its own W_kvb slices, see
 *   mla_path); later calls reuse it.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_MISALIGNED, MLA_ERR_WRONG_MODE
 * (W8A8 handle), MLA_ERR_NO_MEMORY, MLA_ERR_CUDA. */
mla_status mla_kv_prolog_prepare_weights(mla_prolog_t h, const void* W_kva, const void* W_kvb,
                                         cudaStream_t stream);

/* Enqueue the W8A8 full MLA prolog (Q side + KV side) of T = b*s rows on a
 * handle created with quant = MLA_QUANT_W8A8 and dtype = MLA_BF16.
 *   hidden_states [b*s, hidden] bf16; positions [b*s] int32
 *   W_qa  [hidden, q_lora_rank] int8,  sW_qa  [q_lora_rank] f32,  gamma_q [q_lora_rank] bf16
 *   W_qb  [q_lora_rank, H*192]  int8,  sW_qb  [H*192] f32
 *   W_kva [hidden, 576]         int8,  sW_kva [576] f32,          gamma_kv [512] bf16
 *   W_kvb [512, H*256]          int8,  sW_kvb [H*256] f32
 *   cos_table, sin_table [max_pos, 64] f32
 * Outputs (bf16): q_nope [b,H,s,128], q_pe [b,H,s,64], k_nope [b,H,s,128],
 * value [b,H,s,128], k_pe [b,1,s,64].  Steps: quantise each hidden row
 * (amax, inv = 127/amax, q = clamp(rint(x*inv), +-127), s_x = amax/127, all
 * single fp32 operations); q_a_proj and kv_a_proj as int8 GEMMs with int32
 * accumulators, dequantised acc*s_x*s_w; RMSNorm of the q latent (gamma_q)
 * and of compressed_kv (gamma_kv); requantise both rows the same way;
 * q_b_proj -> [H,192] split into q_nope (0:128) and q_pe (128:192), RoPE on
 * q_pe; kv_b_proj -> k_nope / value; RoPE on k_pe.  Errors as for
 * mla_kv_prolog_run. */
mla_status mla_prolog_w8a8_run(mla_prolog_t h, int b, int s, const void* hidden_states,
                               const int32_t* positions, const int8_t* W_qa, const float* sW_qa,
                               const void* gamma_q, const int8_t* W_qb, const float* sW_qb,
                               const int8_t* W_kva, const float* sW_kva, const void* gamma_kv,
                               const int8_t* W_kvb, const float* sW_kvb,
                               const float* cos_table, const float* sin_table, void* q_nope,
                               void* q_pe, void* k_nope, void* value, void* k_pe,
                               cudaStream_t stream);

/* Synchronise `stream`, read the device status word of the handle, clear
 * it (and, if a wait timed out, reset the device barrier counters and the
 * W8A8 accumulator rows and counters) and
 * return MLA_OK, MLA_ERR_BAD_POSITION, MLA_ERR_DEVICE_TIMEOUT or
 * MLA_ERR_BAD_SLOT (in that order of precedence, for the faults recorded
 * since the last call). */
mla_status mla_kv_prolog_status(mla_prolog_t h, cudaStream_t stream);

/* Free the workspace and the handle.  The caller must make sure no run on
 * the handle is still executing (synchronise its stream first). */
mla_status mla_kv_prolog_destroy(mla_prolog_t h);

/* Force a kernel path (mla_path) for later runs on this handle. */
mla_status mla_kv_prolog_set_path(mla_prolog_t h, int path);

/* Number of kernels the last run on this handle enqueued, and the path
 * (mla_path, never AUTO) it took. */
int mla_kv_prolog_last_launches(mla_prolog_t h);
int mla_kv_prolog_last_path(mla_prolog_t h);
/* How many of the last run's launches were the cluster decode kernel
 * (-1 for a null handle). */
int mla_kv_prolog_last_cluster_launches(mla_prolog_t h);

/* The smallest b*s for which MLA_PATH_AUTO takes the prefill kernel on this
 * handle (its model shape and device); smaller b*s take the decode kernel.
 * It replaces the dynamic short / long selection of [MIG]
 * §"源码级原理：KV Prolog 的混合优化实现" (last paragraph: fused op for short
 * inputs, baseline for long ones) by a token-count bucket.  -1 for a null
 * handle. */
int mla_kv_prolog_auto_threshold(mla_prolog_t h);

/* W8A8 building blocks, callable on their own (the full run uses the same
 * kernels; the tests check them bit-exactly):
 *   mla_w8a8_quant_rows: per-row symmetric int8 quantisation of a bf16
 *     matrix x [rows, cols] -> q [rows, cols] int8, scale [rows] f32 (the
 *     fp32 operation sequence described for mla_prolog_w8a8_run).
 *   mla_w8a8_gemm_s32: acc [M, N] int32 = A [M, K] int8 x W [K, N] int8,
 *     W in [in, out] layout; K % 32 == 0, N % 64 == 0 (else
 *     MLA_ERR_UNSUPPORTED); exact for any K (int32 accumulators).
 *   mla_prolog_w8a8_operands: copy the int8 operands and fp32 scales that
 *     the last W8A8 run fed to q_b_proj (q1 [T, q_lora_rank], s1 [T]) and
 *     kv_b_proj (c1 [T, 512], s2 [T]) into caller device buffers.          */
mla_status mla_w8a8_quant_rows(const void* x_bf16, int rows, int cols, int8_t* q, float* scale,
                               cudaStream_t stream);
mla_status mla_w8a8_gemm_s32(const int8_t* A, const int8_t* W, int M, int K, int N,
                             int32_t* acc, cudaStream_t stream);
/* Accumulator capture of the W8A8 prolog (diagnostics and tests; [R1]
 * §"权重转换" W8A8 mode: the int32 accumulators are exact).  While set, every
 * mla_prolog_w8a8_run on the handle also writes the int32 accumulators of
 * its four int8 GEMMs, as its own kernels formed them, into the caller's
 * device buffers (row t = bi*s + si):
 *   acc_a   [T, q_lora_rank + 576]  q_a_proj (columns 0 .. q_lora_rank-1)
 *                                   then kv_a_proj
 *   acc_qb  [T, H*192]              q_b_proj
 *   acc_kvb [T, H*256]              kv_b_proj
 * Each pointer may be NULL (that GEMM is not captured); all NULL turns the
 * capture off.  The buffers must hold the T of every run while set and stay
 * valid until those runs finish.  MLA_ERR_WRONG_MODE on a handle that is
 * not W8A8; MLA_ERR_MISALIGNED for a pointer not 16-byte aligned. */
mla_status mla_prolog_w8a8_capture(mla_prolog_t h, int32_t* acc_a, int32_t* acc_qb,
                                   int32_t* acc_kvb);
mla_status mla_prolog_w8a8_operands(mla_prolog_t h, int T, int8_t* q1, float* s1, int8_t* c1,
                                    float* s2, cudaStream_t stream);

/* No counterpart in the pages: an extra entry point of this library for
 * callers that cannot allocate device memory -- a serving engine or plugin
 * host that owns all device memory in an arena planned up front, or a
 * latency-critical caller that cannot risk a blocking or failing
 * cudaMalloc mid-run.  It runs the fused decode kernel of
 * mla_kv_prolog_run (T = b*s rows, any T, in chunks of 64 or 128 rows) with the
 * same arguments, but needs no handle: its scratch (split-K partials,
 * latent rows, barrier counters, status word) is one fixed __device__
 * array inside the library, about 4.8 MB, held by every device that loads
 * the library until the process exits.  It calls no cudaMalloc, cudaFree
 * or allocating library routine.
 *   cfg            model dimensions as for create; quant must be NONE
 *                  (else MLA_ERR_WRONG_MODE); max_tokens is ignored
 *   device_status  optional device pointer (may be NULL): receives the
 *                  status word of this call (bit 0 bad position, bit 1
 *                  device wait timed out), copied on `stream`
 * Shapes whose split-K scratch would exceed the array are rejected with
 * MLA_ERR_UNSUPPORTED and a message in mla_last_cuda_error().
 * All calls on a device share the array: each call clears the counters
 * and status word first, and calls that overlap on the same GPU race on
 * it (serialise them on one stream).  The first call in each CUDA context
 * (normally once per device) looks up the array's address with
 * cudaGetSymbolAddress while that device is current; the address is cached
 * per context, so a new context (after cudaDeviceReset, say) looks it up
 * again.  Make the first call before any stream capture begins.
 * b * s above INT_MAX gives MLA_ERR_TOO_MANY_TOKENS. */
mla_status mla_kv_prolog_run_noalloc(const mla_prolog_config* cfg, int b, int s,
                                     const void* hidden_states, const int32_t* positions,
                                     const void* W_kva, const void* gamma_kv, const void* W_kvb,
                                     const float* cos_table, const float* sin_table,
                                     void* k_nope, void* value, void* k_pe,
                                     unsigned int* device_status, cudaStream_t stream);

/* Text of a status code (static storage), the text of the last CUDA error
 * seen by this library on the calling thread, and the ABI version. */
const char* mla_status_string(mla_status s);
const char* mla_last_cuda_error(void);
int mla_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_PROLOG_H */
