// internal.h -- launch interfaces between the C-ABI layer (api.cu) and the
// kernel translation units.  Not installed; not part of the ABI.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

// Record the text that mla_last_cuda_error() returns on this thread.
void set_error_text(const char* what);

// Device status bits (kept in the handle's workspace).
enum : unsigned { kStatusBadPosition = 1u, kStatusTimeout = 2u, kStatusBadSlot = 4u };

// Output placement of token row t (shared by the decode and prefill
// kernels): the dense layout [b, X, s, d] (outer = bi, inner = si, count =
// s) or, with a slot mapping, the paged cache [num_blocks, X, page, d]
// (slot = block * page + offset: outer = block, inner = offset, count =
// page).  Element (head hh, column e) of the row is at
// ((outer * X + hh) * count + inner) * d + e.
struct OutLayout {
  const int32_t* slots;  // [T] physical slot per row; null: dense
  int page;              // rows per cache block
  int nslots;            // num_blocks * page
};

// int8 KV-cache outputs: per-channel fp32 scales of k_nope [H*128], value
// [H*128] and k_pe [64]; k == null: outputs in the I/O dtype.  A code is
// clamp(rint(x * (1 / scale)), -127, 127) of the value x the dtype output
// would hold, in IEEE fp32 operations.  The kernels read the reciprocals
// from `inv` ([H*128] of k_nope, [H*128] of value, [64] of k_pe), which
// c8_reciprocals_launch writes before them.
struct C8Scales {
  const float* k;
  const float* v;
  const float* kpe;
  float* inv;
};
// inv[c] = 1 / scale[c] (IEEE fp32 division) for the three scale vectors.
cudaError_t c8_reciprocals_launch(const C8Scales& c8, int heads, cudaStream_t stream);

// Fixed dimensions of the DeepSeek MLA KV prolog this library implements.
constexpr int kRank = 512;         // kv_lora_rank
constexpr int kRope = 64;          // qk_rope_head_dim
constexpr int kNa = kRank + kRope; // kv_a_proj output width (576)
constexpr int kNope = 128;         // qk_nope_head_dim
constexpr int kV = 128;            // v_head_dim
constexpr int kHeadCols = kNope + kV;  // kv_b_proj columns per head (256)

// ---------------------------------------------------------------- decode path
// Upper bound of token rows per decode launch (larger T is processed in
// chunks of the plan's tt_max); also the row stride of the workspace.
constexpr int kDecodeMaxTokens = 128;
// Bytes per normalised latent row in the workspace: the decode kernel's
// shared-memory pitch (512 values + 16 bytes of padding), so one bulk copy
// moves all rows of a launch.
constexpr int kNrmPitch = 1040;
constexpr size_t kDecodeNrmBytes = (size_t)kDecodeMaxTokens * kNrmPitch;

struct DecodeParams {
  CUtensorMap tmap_wkvb;    // W_kvb [512, H*256], box = (ngbox*8 columns, 32 rows)
  CUtensorMap tmap_x;       // packed path: hidden [ntok, hidden], box = (64 columns, 16*mt rows)
  const void* hidden;       // [T, hidden]
  const int32_t* positions; // [T]
  const void* W_kva;        // [hidden, 576]
  const void* gamma;        // [512]
  const void* W_kvb;        // [512, H*256]
  const float* cos_t;       // [max_pos, 64]
  const float* sin_t;
  void* k_nope;             // [b, H, s, 128]
  void* value;              // [b, H, s, 128]
  void* k_pe;               // [b, 1, s, 64]
  void* latent;             // latent-cache variant: normalised compressed_kv [T, 512]; null: full prolog
  OutLayout out;            // dense or paged placement of k_nope / value / k_pe
  C8Scales c8;              // int8 outputs when c8.k is set
  float* partials;          // workspace [KC][kDecodeMaxTokens][576] fp32
  void* nrm;                // workspace [kDecodeMaxTokens][512] dtype
  unsigned* counters;       // workspace: grid barrier {arrivals, generation}
  unsigned* status;         // workspace: device status word
  int hidden_dim, heads, s, t0, TT, max_pos;
  int ntok;                 // rows of `hidden` (b*s)
  int xrows;                // packed path: rows of one hidden-state box
  float eps;
  unsigned long long budget_ns;
  // filled from the plan by decode_launch
  int KB, KC;               // kv_a split-K: rows per chunk (multiple of 64), chunk count
  int kpre, kchunk, nstA;   // W_kvb rows resident / per streamed chunk; phase-A stages
  int ngbox;                // 8-column groups per W_kvb box (odd; >= groups per CTA)
  int off_wb, off_a, off_red, off_misc;  // smem layout (bytes)
  int single_barrier;       // 1: every CTA reduces every row (one grid barrier)
  int pb_wm, pb_ks;         // phase-B warp grid rows (m side) and k-slices
  int tcb;                  // packed weights, phase B on the tensor cores (plan tc_b)
  int tb_res, tb_buf;       // ... W_kvb K blocks resident from the start / in spare buffers
};

// Rows x split-K chunks up to which every CTA reduces all partial rows itself
// (one grid barrier) instead of one CTA per row plus a second barrier.
constexpr int kSingleBarrierRowsTimesChunks = 16;

struct DecodePlan {
  int grid;        // CTAs (one per SM, all resident at once)
  bool two_per_sm; // built to fit two CTAs per SM (the <= kDecodeSmallTokens plan)
  int tt_max;      // token rows per launch (64 or 128)
  int KB, KC;      // split-K of kv_a
  int kpre, kchunk, nstA, ngbox;
  int ngmax;       // most 8-column W_kvb groups of one CTA
  // Phase B on the tensor cores (packed weights; wide column slices, at most
  // 64 rows per launch): the W_kvb slice is packed as 8 K blocks of 64 rows
  // in the MMA's K-major layout; tb_res blocks stay resident from the start,
  // tb_buf more fit in the buffers behind the latent rows, the rest reuse
  // the slots of consumed blocks.
  bool tc_b;
  int tb_res, tb_buf;
  int off_wb, off_a, off_red, off_misc;
  size_t smem;     // dynamic shared memory bytes
  size_t partial_floats;  // workspace floats needed for partials
};

// Plan for a given model shape on the current device; returns false if the
// shape cannot be handled (shared memory or register budget).
bool decode_plan(int hidden, int heads, int num_sms, DecodePlan* plan);
// Launches of at most this many rows can use a plan that fits two CTAs per
// SM (so that a chained next call is resident, copying its weights, while
// this one runs).
constexpr int kDecodeSmallTokens = 32;
// That plan (false if the shape does not fit it: W_kvb slice not resident).
bool decode_plan_small(int hidden, int heads, int num_sms, DecodePlan* plan);
// Phase-B work split for mt m-tiles (a power of two <= 8) and at most ngmax
// column groups per CTA: register-tile variant, warp-grid rows, k-slices.
// False if no variant holds the tile.
bool decode_phase_b(int mt, int ngmax, int* variant, int* wm, int* ks);

// XOR applied to the 16-byte chunk index within row r of a packed W_kvb
// slice of ng chunks per row: the rows of one 8x8 ldmatrix tile then fall
// in distinct banks (odd ng needs none; ng even swaps within aligned pairs,
// quads or octets, so the index stays below ng).
__host__ __device__ inline int pack_swizzle(int ng, int r) {
  if (ng & 1) return 0;
  if (ng & 2) return (r >> 2) & 1;
  if (ng & 4) return (r >> 1) & 3;
  return r & 7;
}
// Pack W_kva / W_kvb (raw [in, out] layouts) into the decode kernel's
// per-CTA contiguous layouts (same byte counts) on `stream`.
cudaError_t decode_pack_weights(const DecodePlan& plan, int hidden, int heads, const void* W_kva,
                                const void* W_kvb, void* pk_kva, void* pk_kvb, cudaStream_t stream);
// Rows of W_kvb per TMA box of the decode kernel.
constexpr int kWkvbBoxRows = 32;
// Packed weights (decode_pack_weights): W_kva / W_kvb point at the packed
// copies, which the kernel reads with 1-D bulk copies.  pdl: launch with
// programmatic stream serialisation (the kernel may start before the
// previous kernel in the stream ends; it reads only the packed snapshot
// before its dependency wait, so the snapshot must not be the previous
// kernel's output).
// xmap (packed path, may be null): the tensor map of the hidden rows for
// this launch's box height (decode_box_rows), encoded by the caller;
// null: encoded here.
cudaError_t decode_launch(bool bf16, bool packed, const DecodePlan& plan, const DecodeParams& p,
                          bool pdl, cudaStream_t stream, const CUtensorMap* xmap = nullptr);
// Rows of one hidden-row TMA box (packed path) for a launch of TT rows of a
// call with ntok rows: 16 * MT, at most ntok.
int decode_box_rows(int TT, int ntok);
// Tensor map of the hidden rows [ntok, hidden] in boxes of 64 columns x
// rows rows with the 128-byte swizzle (packed decode path).
bool decode_encode_xmap(CUtensorMap* map, bool bf16, const void* hidden, int hidden_dim, int ntok,
                        int rows);

// ---------------------------------------------------------------- cluster decode kernel
// The smallest decode launches (at most kClMaxTokens rows, packed snapshot,
// dense or paged outputs in the I/O dtype) run without a grid-wide barrier:
// each 16-CTA cluster computes the whole kv_a row block itself and reduces it
// in distributed shared memory (decode_cl.cu).
constexpr int kClSize = 16;       // CTAs per cluster
constexpr int kClMaxTokens = 16;  // rows per launch
constexpr int kClHidden = 2048;   // hidden size the kernel is built for (128 K rows per CTA)

struct ClPlan {
  int clusters;  // clusters per launch (all resident at once)
  int ngmax;     // most 8-column W_kvb groups of one CTA
  int off_misc;  // shared-memory offset of the barriers / gamma block
  size_t smem;   // dynamic shared memory bytes
};

struct ClParams {
  CUtensorMap tmap_x;       // hidden [ntok, hidden], box = (64 columns, xrows rows), 128-byte swizzle
  const int32_t* positions; // [T]
  const void* W_kva;        // packed snapshot (decode_pack_weights layout, KB rows per unit)
  const void* W_kvb;        // packed snapshot (decode_cl_pack_wkvb: the slices of this grid)
  const void* gamma;        // [512]
  const float* cos_t;       // [max_pos, 64]
  const float* sin_t;
  void* k_nope;             // [b, H, s, 128]
  void* value;              // [b, H, s, 128]
  void* k_pe;               // [b, 1, s, 64]
  OutLayout out;            // dense or paged placement
  unsigned* status;         // workspace: device status word
  int heads, s, t0, TT, max_pos, xrows, KB;
  int off_misc;
  float eps;
  unsigned long long budget_ns;
};

// Plan for this model shape on the current device: false if the shape is
// not the one the kernel is built for (hidden == kClHidden, packed units of
// a multiple of 128 rows) or the device cannot hold a 16-CTA cluster of it.
bool decode_cl_plan(bool bf16, int hidden, int heads, int KB, ClPlan* plan);
// Launch one cluster decode of p.TT <= kClMaxTokens rows.  pdl as for
// decode_launch (the kernel copies only the packed W_kva snapshot before its
// dependency wait).
cudaError_t decode_cl_launch(bool bf16, const ClPlan& plan, const ClParams& p, bool pdl,
                             cudaStream_t stream);
// W_kvb [512, H*256] -> the cluster kernel's per-CTA column slices (the
// decode kernel's packed slice layout for a grid of clusters * 16 CTAs).
cudaError_t decode_cl_pack_wkvb(const ClPlan& plan, int heads, const void* W_kvb, void* out,
                                cudaStream_t stream);

}  // namespace mla

namespace mla {

// ---------------------------------------------------------------- prefill path
struct PrefillParams {
  const void* hidden;
  const int32_t* positions;
  const void* W_kva;
  const void* gamma;
  const void* W_kvb;
  const float* cos_t;
  const float* sin_t;
  void* k_nope;
  void* value;
  void* k_pe;
  void* latent;    // latent-cache variant: normalised compressed_kv [T, 512] (no kv_b); null: full prolog
  OutLayout out;   // dense or paged placement of k_nope / value / k_pe
  C8Scales c8;     // int8 outputs when c8.k is set
  unsigned* status;
  int hidden_dim, heads, s, T, max_pos;
  float eps;
  unsigned long long budget_ns;
  // filled by prefill_launch
  int main_ctas;   // CTAs that own tiles
  int kpe_split;   // 1: the CTAs past main_ctas run the k_pe pass of every tile
};

// Smallest token count for which AUTO selects the tensor-core prefill
// kernel over the decode kernel, for this model shape and SM count.
int prefill_min_tokens(int hidden, int heads, int num_sms);
// Enqueue the prefill kernel(s); *launches receives the kernel count.
// Returns cudaErrorNotSupported for shapes the kernel does not handle.
cudaError_t prefill_launch(bool bf16, const PrefillParams& p, int num_sms, cudaStream_t stream,
                           int* launches);

// ---------------------------------------------------------------- W8A8 path
struct W8Workspace {
  __half* xh;     // [max_tokens, hidden] fp16 codes of the quantised hidden rows
  float* sx;      // [max_tokens]
  int32_t* acc1;  // [max_tokens, q_rank + 576]; rows [0, kW8PairMinRows) zero between calls
  int8_t* q1;     // [max_tokens, q_rank]
  float* s1;      // [max_tokens]
  int8_t* c1;     // [max_tokens, 512]
  float* s2;      // [max_tokens]
  __half* q1h;    // [max_tokens, q_rank] fp16 codes of q1 (the q_b operand)
  __half* c1h;    // [max_tokens, 512] fp16 codes of c1 (the kv_b operand)
  // fp16 copies of the int8 weights for the prefill-size GEMMs (null when
  // max_tokens < kW8PairMinRows): [W_qa | W_kva] [hidden, lda], W_qb [q_rank,
  // ldqb], W_kvb [512, ldkvb], rows padded to multiples of 256 with zeros
  __half* wa16;
  __half* wqb16;
  __half* wkvb16;
  int lda, ldqb, ldkvb;
  unsigned* readers;  // decode-size chain: CTAs done reading acc1
};

// Decode-size W8A8 chain (T <= kW8SmallRows): tensor maps of the four int8
// weight matrices and the per-handle launch plan.
constexpr int kW8SmallRows = 8;
// Longest q_rank + 576 row the W8A8 normalisation handles (q_rank <= 3520).
constexpr int kW8MaxNormCols = 4096;
struct W8Maps {
  CUtensorMap qa, kva;  // W_qa [hidden, q_rank], W_kva [hidden, 576]: box 256 columns x kchunk rows
  CUtensorMap qb, kvb;  // W_qb [q_rank, H*192], W_kvb [512, H*256]: box 128 columns x 256 rows
  const void* src[4];   // the pointers they describe
  bool valid;
};
struct W8SmallPlan {
  int kchunk, splits;   // kv_a/q_a split-K: rows per chunk (multiple of 32, <= 512), chunk count
  int nblk_a1, nblk_a;  // 256-column blocks of q_a, of q_a + kv_a
  int nblk_b1, nblk_b;  // 128-column blocks of q_b, of q_b + kv_b
  int grid_b;           // CTAs of the q_b / kv_b kernel
  int* units;           // device: [grid_b + 1] offsets, then block ids (workspace)
};

struct W8Params {
  const void* hidden;
  const int32_t* positions;
  const int8_t* W_qa;
  const float* sW_qa;
  const void* gamma_q;
  const int8_t* W_qb;
  const float* sW_qb;
  const int8_t* W_kva;
  const float* sW_kva;
  const void* gamma_kv;
  const int8_t* W_kvb;
  const float* sW_kvb;
  const float* cos_t;
  const float* sin_t;
  void* q_nope;
  void* q_pe;
  void* k_nope;
  void* value;
  void* k_pe;
  unsigned* status;
  // accumulator capture (diagnostics; null: off): the int32 accumulators of
  // q_a | kv_a [T, q_rank + 576], of q_b [T, H*192] and of kv_b [T, H*256]
  int32_t* cap_a;
  int32_t* cap_qb;
  int32_t* cap_kvb;
  int hidden_dim, q_rank, heads, s, T, max_pos;
  float eps;
  unsigned long long budget_ns;
};

// Tensor-core int8 GEMMs of the W8A8 prolog (w8mma.cu): up to two weight
// matrices W_i [K_i, N_i] int8 against fp16 activation codes X_i [T, K_i],
// exact int32 sums.  raw: added into C (q_a | kv_a accumulator rows);
// otherwise dequantised into the head-major outputs (q_b, kv_b).
struct W8MmaParams {
  CUtensorMap tw[2];        // filled by w8mma_launch
  CUtensorMap tx[2];
  int K[2], N[2];           // K multiple of 64, N multiple of 32 (N = 0: no matrix)
  int mt[2], ks[2], kbps[2], nunits[2];  // filled: 128-column tiles, K splits, K blocks per split, units
  int mfast[2];             // filled: unit order, weight tiles fastest (1) or token tiles fastest (0)
  unsigned s_mul, s_shift;  // filled: t / s = (umulhi(t, s_mul) + t) >> s_shift
  int NT, xrows, ntiles, stages;         // filled: tokens per tile, box rows, token tiles, ring depth
  int T;
  int raw;                  // 1: int32 sums added into C
  int32_t* C;               // raw: [T, ldc]
  int ldc;
  int coff[2];              // raw: column of matrix i in C
  const float* sx[2];       // heads: per-token activation scales of X_i
  const float* sw[2];       // heads: per-column weight scales of W_i
  const int32_t* positions;
  const float* cos_t;
  const float* sin_t;
  int max_pos;
  void* q_nope;             // heads, matrix 0 (q_b): [b,H,s,128], q_pe [b,H,s,64]
  void* q_pe;
  void* k_nope;             // heads, matrix 1 (kv_b): [b,H,s,128] each
  void* value;
  int32_t* cap[2];          // heads: accumulator capture [T, N_i] (null: off)
  int heads, s;
  unsigned* status;
  unsigned long long budget_ns;
};
size_t w8mma_smem(int NT, int stages);

// Prefill-size int8 GEMMs of the W8A8 prolog on the 2-SM MMA (w8pair.cu):
// activations X_i fp16 codes [T, K_i], weights widened to fp16 [K_i, ldw_i]
// (ldw_i a multiple of 256, columns N_i .. ldw_i-1 zero).
struct W8PairParams {
  int K[2], N[2], ldw[2];   // N = 0: no matrix
  int ntiles[2], nn[2];     // filled: pair tiles per matrix, 256-column tiles
  int nm;                   // filled: 256-row token tiles
  int mfast[2];             // filled: tile order, token tiles fastest (1) or weight tiles fastest (0)
  unsigned s_mul, s_shift;  // filled: t / s
  int T;
  int raw;                  // 1: int32 sums stored into C
  int32_t* C;
  int ldc;
  int coff[2];
  const float* sx[2];
  const float* sw[2];
  const int32_t* positions;
  const float* cos_t;
  const float* sin_t;
  int max_pos;
  void* q_nope;
  void* q_pe;
  void* k_nope;
  void* value;
  int32_t* cap[2];
  int heads, s;
  unsigned* status;
  unsigned long long budget_ns;
};
cudaError_t w8pair_launch(W8PairParams p, const void* X0, const void* X1, const __half* W0, const __half* W1,
                          int num_sms, cudaStream_t stream);
// One int8 matrix [K, N] widened to fp16 rows of ldn elements at `out`,
// columns [0, wcols) written (zeros past N).
struct W8WidenJob {
  const int8_t* W;
  __half* out;
  int K, N, ldn, wcols;
};
cudaError_t w8_widen_launch(const W8WidenJob* jobs, int n, int num_sms, cudaStream_t stream);
// Token count from which the W8A8 prolog runs its GEMMs on the 2-SM kernel
// (widened weights); below it the int8-converting single-SM kernel.
constexpr int kW8PairMinRows = 512;
cudaError_t w8mma_launch(W8MmaParams p, const int8_t* W0, const int8_t* W1, const void* X0, const void* X1,
                         int num_sms, cudaStream_t stream, bool pdl);

size_t w8_workspace_bytes(int hidden, int q_rank, int heads, int max_tokens, int num_sms);
void w8_workspace_carve(void* base, int hidden, int q_rank, int heads, int max_tokens,
                        int num_sms, W8Workspace* w, W8SmallPlan* plan);
// Zero the q_a/kv_a accumulator rows and upload the q_b/kv_b work lists
// (once, when the handle is created; synchronous).
cudaError_t w8_workspace_init(const W8Workspace& w, const W8SmallPlan& plan, int hidden,
                              int q_rank, int heads, int max_tokens, int num_sms);
// Tensor maps of the decode-size chain for these weight pointers (false if
// the CUDA driver rejects one).
bool w8_encode_maps(const W8Params& p, const W8SmallPlan& plan, W8Maps* maps);
cudaError_t w8a8_launch(const W8Params& p, const W8Workspace& w, const W8SmallPlan& plan,
                        const W8Maps* maps, int num_sms, cudaStream_t stream, int* launches);
cudaError_t w8a8_quant_rows_launch(const void* x_bf16, int rows, int cols, int8_t* q,
                                   float* scale, cudaStream_t stream);
cudaError_t w8a8_gemm_s32_launch(const int8_t* A, const int8_t* W, int M, int K, int N,
                                 int32_t* acc, cudaStream_t stream);
cudaError_t w8a8_copy_operands(const W8Workspace& w, int T, int q_rank, int8_t* q1, float* s1,
                               int8_t* c1, float* s2, cudaStream_t stream);

}  // namespace mla
