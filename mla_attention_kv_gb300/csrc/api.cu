// api.cu -- the C ABI of include/mla_prolog.h: handle lifetime, argument
// validation, workspace, T-bucketed path selection and kernel dispatch.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <new>

#include "../../include/mla_prolog.h"
#include "internal.h"
#include "tma.h"

using namespace mla;

struct mla_prolog_s {
  mla_prolog_config cfg;
  int device;
  int num_sms;
  int path_override;
  int last_launches;
  int last_path;
  int last_cl_launches;
  unsigned long long budget_ns;
  // workspace
  void* ws;
  size_t ws_bytes;
  unsigned* status;    // [1]
  unsigned* counters;  // [2] grid barrier
  float* partials;
  void* nrm;
  float* c8inv;  // reciprocal int8 KV-cache scales [H*256 + 64] (mla_kv_prolog_run_c8)
  DecodePlan dplan;
  bool decode_ok;
  DecodePlan dplan_small;  // <= kDecodeSmallTokens rows per launch, two CTAs per SM
  bool small_ok;
  ClPlan clplan;  // cluster decode kernel (launches of <= kClMaxTokens rows)
  bool cl_ok;
  // packed weight snapshot (mla_kv_prolog_prepare_weights): W_kva tiles, W_kvb
  // slices, then (cl_ok) the W_kvb slices of the cluster kernel's grid, and
  // the caller pointers they were taken from
  void* pk;
  size_t pk_kva_bytes, pk_kvb_bytes, pk_bytes;
  const void* pk_src_kva;
  const void* pk_src_kvb;
  // the snapshot was just written: the next decode launch must not read it
  // before its dependency wait (launched without programmatic serialisation)
  bool pk_fresh;
  // W8A8 workspace, decode-size launch plan and tensor maps (see w8a8.cu)
  W8Workspace w8;
  W8SmallPlan w8plan;
  W8Maps w8maps;
  // W8A8 accumulator capture (mla_prolog_w8a8_capture); null: off
  int32_t* cap_a;
  int32_t* cap_qb;
  int32_t* cap_kvb;
  // tensor maps of recently seen W_kvb pointers (decode kernel)
  static constexpr int kMapCache = 64;
  const void* map_ptr[kMapCache];
  CUtensorMap map[kMapCache];
  int map_next;
  // tensor maps of recently seen hidden-row buffers (packed decode path),
  // keyed by pointer, row count and box height
  static constexpr int kXMapCache = 32;
  const void* xmap_ptr[kXMapCache];
  int xmap_ntok[kXMapCache];
  int xmap_rows[kXMapCache];
  CUtensorMap xmap[kXMapCache];
  int xmap_next;
};

// Tensor map of the hidden rows for a packed decode launch, cached.
static const CUtensorMap* hidden_map(mla_prolog_s* h, const void* hidden, int ntok, int rows) {
  for (int i = 0; i < mla_prolog_s::kXMapCache; ++i)
    if (h->xmap_ptr[i] == hidden && h->xmap_ntok[i] == ntok && h->xmap_rows[i] == rows) return &h->xmap[i];
  const int slot = h->xmap_next;
  if (!decode_encode_xmap(&h->xmap[slot], h->cfg.dtype == MLA_BF16, hidden, h->cfg.hidden, ntok, rows))
    return nullptr;
  h->xmap_ptr[slot] = hidden;
  h->xmap_ntok[slot] = ntok;
  h->xmap_rows[slot] = rows;
  h->xmap_next = (slot + 1) % mla_prolog_s::kXMapCache;
  return &h->xmap[slot];
}

// Tensor map of W_kvb [512, H*256] for the decode kernel, cached per pointer.
static const CUtensorMap* wkvb_map(mla_prolog_s* h, const void* W_kvb) {
  for (int i = 0; i < mla_prolog_s::kMapCache; ++i)
    if (h->map_ptr[i] == W_kvb) return &h->map[i];
  const int slot = h->map_next;
  const uint64_t NB = (uint64_t)h->cfg.num_heads * kHeadCols;
  const CUtensorMapDataType dt = h->cfg.dtype == MLA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (!encode_tmap_2d(&h->map[slot], dt, W_kvb, NB, kRank, NB * 2, (uint32_t)h->dplan.ngbox * 8,
                      kWkvbBoxRows, CU_TENSOR_MAP_SWIZZLE_NONE))
    return nullptr;
  h->map_ptr[slot] = W_kvb;
  h->map_next = (slot + 1) % mla_prolog_s::kMapCache;
  return &h->map[slot];
}

static thread_local char g_last_cuda_error[256] = "no error";

static mla_status cuda_fail(cudaError_t e, const char* what) {
  snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s (%d)", what,
           cudaGetErrorString(e), (int)e);
  return MLA_ERR_CUDA;
}

void mla::set_error_text(const char* what) {
  snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s", what);
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" {

int mla_abi_version(void) { return MLA_PROLOG_ABI_VERSION; }

const char* mla_last_cuda_error(void) { return g_last_cuda_error; }

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported dimensions";
    case MLA_ERR_TOO_MANY_TOKENS: return "b*s exceeds max_tokens";
    case MLA_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
    case MLA_ERR_CUDA: return "CUDA runtime error";
    case MLA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MLA_ERR_BAD_POSITION: return "position outside [0, max_pos)";
    case MLA_ERR_NO_MEMORY: return "workspace allocation failed";
    case MLA_ERR_WRONG_MODE: return "run does not match the handle's quant mode";
    case MLA_ERR_BAD_SLOT: return "a cache slot past num_blocks * page_size was seen (row dropped)";
  }
  return "unknown status";
}

mla_status mla_kv_prolog_create(const mla_prolog_config* cfg, mla_prolog_t* out) {
  if (!cfg || !out) return MLA_ERR_INVALID_ARG;
  *out = nullptr;
  const mla_prolog_config& c = *cfg;
  if (c.hidden <= 0 || c.num_heads <= 0 || c.max_tokens <= 0 || c.max_pos <= 0 ||
      !(c.eps >= 0.0f) || (c.dtype != MLA_F16 && c.dtype != MLA_BF16) ||
      (c.quant != MLA_QUANT_NONE && c.quant != MLA_QUANT_W8A8))
    return MLA_ERR_INVALID_ARG;
  if (c.kv_lora_rank != kRank || c.rope_dim != kRope || c.nope_dim != kNope || c.v_dim != kV ||
      c.hidden % 64 != 0)
    return MLA_ERR_UNSUPPORTED;
  if (c.quant == MLA_QUANT_W8A8 &&
      (c.dtype != MLA_BF16 || c.q_lora_rank <= 0 || c.q_lora_rank % 64 != 0 ||
       c.q_lora_rank + kNa > kW8MaxNormCols))
    return MLA_ERR_UNSUPPORTED;

  mla_prolog_s* h = new (std::nothrow) mla_prolog_s();
  if (!h) return MLA_ERR_NO_MEMORY;
  memset(h, 0, sizeof(*h));
  h->cfg = c;
  h->budget_ns = c.spin_budget_ns ? c.spin_budget_ns : 1000000000ull;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "device query");
  }
  h->decode_ok = decode_plan(c.hidden, c.num_heads, h->num_sms, &h->dplan);
  // (the small plan shares the packed snapshot, so it needs the same W_kvb layout)
  h->small_ok = h->decode_ok && !h->dplan.tc_b &&
                decode_plan_small(c.hidden, c.num_heads, h->num_sms, &h->dplan_small) &&
                h->dplan_small.KB == h->dplan.KB && h->dplan_small.KC == h->dplan.KC;
  if (c.quant == MLA_QUANT_NONE && !h->decode_ok) {
    delete h;
    return MLA_ERR_UNSUPPORTED;
  }
  // (the cluster kernel reads the packed W_kva snapshot, laid out by dplan)
  h->cl_ok = c.quant == MLA_QUANT_NONE &&
             decode_cl_plan(c.dtype == MLA_BF16, c.hidden, c.num_heads, h->dplan.KB, &h->clplan);
  // workspace: [status][counters x2][pad] | partials | nrm | w8a8
  size_t off = 256;
  const size_t part_off = off;
  off += h->decode_ok ? h->dplan.partial_floats * sizeof(float) : 0;
  off = (off + 255) & ~(size_t)255;
  const size_t nrm_off = off;
  off += kDecodeNrmBytes;
  off = (off + 255) & ~(size_t)255;
  const size_t c8_off = off;
  off += ((size_t)c.num_heads * kHeadCols + kRope) * sizeof(float);
  off = (off + 255) & ~(size_t)255;
  size_t w8_off = off;
  if (c.quant == MLA_QUANT_W8A8)
    off += w8_workspace_bytes(c.hidden, c.q_lora_rank, c.num_heads, c.max_tokens, h->num_sms);
  h->ws_bytes = off;
  e = cudaMalloc(&h->ws, h->ws_bytes);
  if (e != cudaSuccess) {
    delete h;
    cuda_fail(e, "cudaMalloc workspace");
    return MLA_ERR_NO_MEMORY;
  }
  e = cudaMemset(h->ws, 0, 256);
  if (e != cudaSuccess) {
    cudaFree(h->ws);
    delete h;
    return cuda_fail(e, "cudaMemset workspace");
  }
  unsigned char* base = static_cast<unsigned char*>(h->ws);
  h->status = reinterpret_cast<unsigned*>(base);
  h->counters = reinterpret_cast<unsigned*>(base + 64);
  h->partials = reinterpret_cast<float*>(base + part_off);
  h->nrm = base + nrm_off;
  h->c8inv = reinterpret_cast<float*>(base + c8_off);
  if (c.quant == MLA_QUANT_W8A8) {
    w8_workspace_carve(base + w8_off, c.hidden, c.q_lora_rank, c.num_heads, c.max_tokens,
                       h->num_sms, &h->w8, &h->w8plan);
    e = w8_workspace_init(h->w8, h->w8plan, c.hidden, c.q_lora_rank, c.num_heads, c.max_tokens,
                          h->num_sms);
    if (e != cudaSuccess) {
      cudaFree(h->ws);
      delete h;
      return cuda_fail(e, "W8A8 workspace init");
    }
  }
  *out = h;
  return MLA_OK;
}

mla_status mla_kv_prolog_destroy(mla_prolog_t h) {
  if (!h) return MLA_ERR_INVALID_ARG;
  if (h->pk) cudaFree(h->pk);
  cudaError_t e = cudaFree(h->ws);
  delete h;
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "cudaFree workspace");
}

mla_status mla_kv_prolog_set_path(mla_prolog_t h, int path) {
  if (!h || path < MLA_PATH_AUTO || path > MLA_PATH_DECODE_GRID) return MLA_ERR_INVALID_ARG;
  h->path_override = path;
  return MLA_OK;
}

int mla_kv_prolog_last_launches(mla_prolog_t h) { return h ? h->last_launches : -1; }

int mla_kv_prolog_auto_threshold(mla_prolog_t h) {
  if (!h) return -1;
  return prefill_min_tokens(h->cfg.hidden, h->cfg.num_heads, h->num_sms);
}

mla_status mla_prolog_w8a8_capture(mla_prolog_t h, int32_t* acc_a, int32_t* acc_qb, int32_t* acc_kvb) {
  if (!h) return MLA_ERR_INVALID_ARG;
  if (h->cfg.quant != MLA_QUANT_W8A8) return MLA_ERR_WRONG_MODE;
  if ((acc_a && !aligned16(acc_a)) || (acc_qb && !aligned16(acc_qb)) || (acc_kvb && !aligned16(acc_kvb)))
    return MLA_ERR_MISALIGNED;
  h->cap_a = acc_a;
  h->cap_qb = acc_qb;
  h->cap_kvb = acc_kvb;
  return MLA_OK;
}
int mla_kv_prolog_last_path(mla_prolog_t h) { return h ? h->last_path : -1; }
int mla_kv_prolog_last_cluster_launches(mla_prolog_t h) { return h ? h->last_cl_launches : -1; }

mla_status mla_kv_prolog_status(mla_prolog_t h, cudaStream_t stream) {
  if (!h) return MLA_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned st = 0;
  e = cudaMemcpy(&st, h->status, sizeof(unsigned), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read status");
  if (st) {
    // clear the status word and, after a timeout, the barrier counters
    e = cudaMemset(h->ws, 0, 256);
    if (e != cudaSuccess) return cuda_fail(e, "clear status");
    if ((st & kStatusTimeout) && h->cfg.quant == MLA_QUANT_W8A8) {
      // a chain that gave up may have left partial sums in the accumulator
      // rows, which every call expects zeroed, and a reader count behind
      e = cudaMemset(h->w8.acc1, 0, (size_t)h->cfg.max_tokens * (h->cfg.q_lora_rank + kNa) * 4);
      if (e == cudaSuccess) e = cudaMemset(h->w8.readers, 0, 256);
      if (e != cudaSuccess) return cuda_fail(e, "reset W8A8 workspace");
    }
  }
  if (st & kStatusBadPosition) return MLA_ERR_BAD_POSITION;
  if (st & kStatusTimeout) return MLA_ERR_DEVICE_TIMEOUT;
  if (st & kStatusBadSlot) return MLA_ERR_BAD_SLOT;
  return MLA_OK;
}

// The KV prolog (latent == null) or its latent-cache variant (latent [T, 512]
// written instead of k_nope / value; W_kvb, k_nope and value unused).
static mla_status run_kv(mla_prolog_t h, int b, int s, const void* hidden_states,
                         const int32_t* positions, const void* W_kva, const void* gamma_kv,
                         const void* W_kvb, const float* cos_table, const float* sin_table,
                         void* k_nope, void* value, void* k_pe, void* latent, const OutLayout& lay,
                         const C8Scales& c8, cudaStream_t stream) {
  if (!h || b < 0 || s < 0) return MLA_ERR_INVALID_ARG;
  if (h->cfg.quant != MLA_QUANT_NONE) return MLA_ERR_WRONG_MODE;
  const long long T = (long long)b * s;
  h->last_launches = 0;
  h->last_cl_launches = 0;
  if (T == 0) return MLA_OK;
  if (T > h->cfg.max_tokens) return MLA_ERR_TOO_MANY_TOKENS;
  const void* ptrs[] = {hidden_states, positions, W_kva, gamma_kv, cos_table, sin_table, k_pe,
                        latent ? latent : W_kvb, latent ? latent : k_nope, latent ? latent : value};
  for (const void* q : ptrs)
    if (!q) return MLA_ERR_INVALID_ARG;
  for (const void* q : ptrs)
    if (!aligned16(q)) return MLA_ERR_MISALIGNED;

  const bool bf16 = h->cfg.dtype == MLA_BF16;
  C8Scales c8q = c8;
  if (c8q.k) {  // reciprocal scales, read by the kernel's store epilogue
    c8q.inv = h->c8inv;
    cudaError_t e = c8_reciprocals_launch(c8q, h->cfg.num_heads, stream);
    if (e != cudaSuccess) return cuda_fail(e, "int8 cache scales");
    h->last_launches = 1;
  }
  int path = h->path_override;
  const bool grid_only = path == MLA_PATH_DECODE_GRID;
  if (grid_only) path = MLA_PATH_DECODE;
  if (path == MLA_PATH_AUTO)
    path = T >= prefill_min_tokens(h->cfg.hidden, h->cfg.num_heads, h->num_sms) ? MLA_PATH_PREFILL : MLA_PATH_DECODE;
  h->last_path = path;

  if (path == MLA_PATH_PREFILL) {
    PrefillParams pp = {};
    pp.hidden = hidden_states; pp.positions = positions; pp.W_kva = W_kva; pp.gamma = gamma_kv;
    pp.W_kvb = W_kvb; pp.cos_t = cos_table; pp.sin_t = sin_table; pp.k_nope = k_nope;
    pp.value = value; pp.k_pe = k_pe; pp.latent = latent; pp.out = lay; pp.c8 = c8q; pp.status = h->status;
    pp.hidden_dim = h->cfg.hidden; pp.heads = h->cfg.num_heads; pp.s = s; pp.T = (int)T;
    pp.max_pos = h->cfg.max_pos; pp.eps = h->cfg.eps; pp.budget_ns = h->budget_ns;
    int launches = 0;
    cudaError_t e = prefill_launch(bf16, pp, h->num_sms, stream, &launches);
    h->last_launches += launches;
    if (e == cudaErrorNotSupported) return MLA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return MLA_OK;
  }

  // the packed snapshot serves runs that pass the weights it was taken from
  // (the latent-cache variant needs only its W_kva part)
  const bool packed = h->pk && W_kva == h->pk_src_kva && (latent || W_kvb == h->pk_src_kvb);
  DecodeParams p = {};
  if (packed) {
    W_kva = h->pk;
    W_kvb = static_cast<const unsigned char*>(h->pk) + h->pk_kva_bytes;
  } else if (!latent) {
    const CUtensorMap* tm = wkvb_map(h, W_kvb);
    if (!tm) {
      snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "cuTensorMapEncodeTiled failed for W_kvb");
      return MLA_ERR_CUDA;
    }
    p.tmap_wkvb = *tm;
  }
  p.hidden = hidden_states; p.positions = positions; p.W_kva = W_kva; p.gamma = gamma_kv;
  p.W_kvb = W_kvb; p.cos_t = cos_table; p.sin_t = sin_table; p.k_nope = k_nope; p.value = value;
  p.k_pe = k_pe; p.latent = latent; p.out = lay; p.c8 = c8q; p.partials = h->partials; p.nrm = h->nrm; p.counters = h->counters;
  p.status = h->status; p.hidden_dim = h->cfg.hidden; p.heads = h->cfg.num_heads; p.s = s;
  p.max_pos = h->cfg.max_pos; p.eps = h->cfg.eps;
  p.budget_ns = h->budget_ns;
  p.ntok = (int)T;
  const int tt = h->dplan.tt_max;
  for (long long t0 = 0; t0 < T; t0 += tt) {
    p.t0 = (int)t0;
    p.TT = (int)((T - t0) < tt ? (T - t0) : tt);
    // small launches on the packed snapshot: the two-CTA-per-SM plan (its
    // CTAs copy the snapshot before the dependency wait; raw weights may come
    // from the previous kernel, so they gain nothing from an early start)
    const DecodePlan& pl = (h->small_ok && packed && p.TT <= h->dplan_small.tt_max) ? h->dplan_small : h->dplan;
    const CUtensorMap* xm = nullptr;
    if (packed) {
      xm = hidden_map(h, hidden_states, p.ntok, decode_box_rows(p.TT, p.ntok));
      if (!xm) {
        snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "cuTensorMapEncodeTiled failed for the hidden rows");
        return MLA_ERR_CUDA;
      }
    }
    cudaError_t e;
    if (packed && h->cl_ok && !grid_only && !latent && !c8q.k && p.TT <= kClMaxTokens) {
      // the cluster kernel (no grid-wide barrier)
      ClParams cp = {};
      cp.tmap_x = *xm;
      cp.W_kvb = static_cast<const unsigned char*>(h->pk) + h->pk_kva_bytes + h->pk_kvb_bytes;
      cp.positions = positions; cp.W_kva = W_kva; cp.gamma = gamma_kv; cp.cos_t = cos_table;
      cp.sin_t = sin_table; cp.k_nope = k_nope; cp.value = value; cp.k_pe = k_pe; cp.out = lay;
      cp.status = h->status; cp.heads = h->cfg.num_heads; cp.s = s; cp.t0 = p.t0; cp.TT = p.TT;
      cp.max_pos = h->cfg.max_pos; cp.xrows = decode_box_rows(p.TT, p.ntok); cp.KB = h->dplan.KB;
      cp.off_misc = h->clplan.off_misc; cp.eps = h->cfg.eps;
      cp.budget_ns = h->budget_ns;
      e = decode_cl_launch(bf16, h->clplan, cp, !h->pk_fresh, stream);
      if (e == cudaSuccess) h->last_cl_launches += 1;
    } else {
      e = decode_launch(bf16, packed, pl, p, !(packed && h->pk_fresh), stream, xm);
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    if (packed) h->pk_fresh = false;
    h->last_launches += 1;
  }
  return MLA_OK;
}

mla_status mla_kv_prolog_run(mla_prolog_t h, int b, int s, const void* hidden_states,
                             const int32_t* positions, const void* W_kva, const void* gamma_kv,
                             const void* W_kvb, const float* cos_table, const float* sin_table,
                             void* k_nope, void* value, void* k_pe, cudaStream_t stream) {
  return run_kv(h, b, s, hidden_states, positions, W_kva, gamma_kv, W_kvb, cos_table, sin_table,
                k_nope, value, k_pe, nullptr, OutLayout{nullptr, 0, 0}, C8Scales{nullptr, nullptr, nullptr, nullptr},
                stream);
}

mla_status mla_kv_prolog_run_c8(mla_prolog_t h, int b, int s, const void* hidden_states,
                                const int32_t* positions, const void* W_kva, const void* gamma_kv,
                                const void* W_kvb, const float* cos_table, const float* sin_table,
                                const float* k_scale, const float* v_scale, const float* kpe_scale,
                                int8_t* k_nope, int8_t* value, int8_t* k_pe, cudaStream_t stream) {
  if (!k_scale || !v_scale || !kpe_scale) return MLA_ERR_INVALID_ARG;
  if (!aligned16(k_scale) || !aligned16(v_scale) || !aligned16(kpe_scale)) return MLA_ERR_MISALIGNED;
  return run_kv(h, b, s, hidden_states, positions, W_kva, gamma_kv, W_kvb, cos_table, sin_table,
                k_nope, value, k_pe, nullptr, OutLayout{nullptr, 0, 0},
                C8Scales{k_scale, v_scale, kpe_scale, nullptr}, stream);
}

mla_status mla_kv_prolog_run_paged(mla_prolog_t h, int b, int s, const void* hidden_states,
                                   const int32_t* positions, const void* W_kva,
                                   const void* gamma_kv, const void* W_kvb,
                                   const float* cos_table, const float* sin_table,
                                   const int32_t* slot_mapping, int page_size, int num_blocks,
                                   void* k_cache, void* v_cache, void* kpe_cache,
                                   cudaStream_t stream) {
  if (!slot_mapping || page_size <= 0 || num_blocks <= 0 ||
      (long long)page_size * num_blocks > 0x7fffffffLL)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(slot_mapping)) return MLA_ERR_MISALIGNED;
  return run_kv(h, b, s, hidden_states, positions, W_kva, gamma_kv, W_kvb, cos_table, sin_table,
                k_cache, v_cache, kpe_cache, nullptr,
                OutLayout{slot_mapping, page_size, page_size * num_blocks}, C8Scales{nullptr, nullptr, nullptr, nullptr},
                stream);
}

mla_status mla_kv_prolog_run_latent(mla_prolog_t h, int b, int s, const void* hidden_states,
                                    const int32_t* positions, const void* W_kva,
                                    const void* gamma_kv, const float* cos_table,
                                    const float* sin_table, void* latent, void* k_pe,
                                    cudaStream_t stream) {
  if (!latent) return MLA_ERR_INVALID_ARG;
  return run_kv(h, b, s, hidden_states, positions, W_kva, gamma_kv, nullptr, cos_table, sin_table,
                nullptr, nullptr, k_pe, latent, OutLayout{nullptr, 0, 0}, C8Scales{nullptr, nullptr, nullptr, nullptr},
                stream);
}

mla_status mla_kv_prolog_prepare_weights(mla_prolog_t h, const void* W_kva, const void* W_kvb,
                                         cudaStream_t stream) {
  if (!h) return MLA_ERR_INVALID_ARG;
  if (h->cfg.quant != MLA_QUANT_NONE) return MLA_ERR_WRONG_MODE;
  if (!W_kva && !W_kvb) {  // forget the snapshot
    h->pk_src_kva = h->pk_src_kvb = nullptr;
    return MLA_OK;
  }
  if (!W_kva || !W_kvb) return MLA_ERR_INVALID_ARG;
  if (!aligned16(W_kva) || !aligned16(W_kvb)) return MLA_ERR_MISALIGNED;
  const size_t kva_bytes = (size_t)h->cfg.hidden * kNa * 2;
  const size_t kvb_bytes = (size_t)kRank * h->cfg.num_heads * kHeadCols * 2;
  if (!h->pk) {
    cudaError_t e = cudaMalloc(&h->pk, kva_bytes + kvb_bytes * (h->cl_ok ? 2 : 1));
    if (e != cudaSuccess) {
      h->pk = nullptr;
      cuda_fail(e, "cudaMalloc packed weights");
      return MLA_ERR_NO_MEMORY;
    }
    h->pk_kva_bytes = kva_bytes;
    h->pk_kvb_bytes = kvb_bytes;
    h->pk_bytes = kva_bytes + kvb_bytes * (h->cl_ok ? 2 : 1);
  }
  h->pk_src_kva = h->pk_src_kvb = nullptr;
  unsigned char* base = static_cast<unsigned char*>(h->pk);
  cudaError_t e = decode_pack_weights(h->dplan, h->cfg.hidden, h->cfg.num_heads, W_kva, W_kvb, base,
                                      base + kva_bytes, stream);
  if (e == cudaSuccess && h->cl_ok)
    e = decode_cl_pack_wkvb(h->clplan, h->cfg.num_heads, W_kvb, base + kva_bytes + kvb_bytes, stream);
  if (e != cudaSuccess) return cuda_fail(e, "pack weights");
  h->pk_src_kva = W_kva;
  h->pk_src_kvb = W_kvb;
  h->pk_fresh = true;
  return MLA_OK;
}

mla_status mla_prolog_w8a8_run(mla_prolog_t h, int b, int s, const void* hidden_states,
                               const int32_t* positions, const int8_t* W_qa, const float* sW_qa,
                               const void* gamma_q, const int8_t* W_qb, const float* sW_qb,
                               const int8_t* W_kva, const float* sW_kva, const void* gamma_kv,
                               const int8_t* W_kvb, const float* sW_kvb,
                               const float* cos_table, const float* sin_table, void* q_nope,
                               void* q_pe, void* k_nope, void* value, void* k_pe,
                               cudaStream_t stream) {
  if (!h || b < 0 || s < 0) return MLA_ERR_INVALID_ARG;
  if (h->cfg.quant != MLA_QUANT_W8A8) return MLA_ERR_WRONG_MODE;
  const long long T = (long long)b * s;
  h->last_launches = 0;
  h->last_cl_launches = 0;
  if (T == 0) return MLA_OK;
  if (T > h->cfg.max_tokens) return MLA_ERR_TOO_MANY_TOKENS;
  const void* ptrs[] = {hidden_states, positions, W_qa, sW_qa, gamma_q, W_qb, sW_qb, W_kva,
                        sW_kva, gamma_kv, W_kvb, sW_kvb, cos_table, sin_table, q_nope, q_pe,
                        k_nope, value, k_pe};
  for (const void* q : ptrs)
    if (!q) return MLA_ERR_INVALID_ARG;
  for (const void* q : ptrs)
    if (!aligned16(q)) return MLA_ERR_MISALIGNED;
  W8Params p = {};
  p.hidden = hidden_states; p.positions = positions; p.W_qa = W_qa; p.sW_qa = sW_qa;
  p.gamma_q = gamma_q; p.W_qb = W_qb; p.sW_qb = sW_qb; p.W_kva = W_kva; p.sW_kva = sW_kva;
  p.gamma_kv = gamma_kv; p.W_kvb = W_kvb; p.sW_kvb = sW_kvb; p.cos_t = cos_table;
  p.sin_t = sin_table; p.q_nope = q_nope; p.q_pe = q_pe; p.k_nope = k_nope; p.value = value;
  p.k_pe = k_pe; p.status = h->status; p.hidden_dim = h->cfg.hidden;
  p.q_rank = h->cfg.q_lora_rank; p.heads = h->cfg.num_heads; p.s = s; p.T = (int)T;
  p.max_pos = h->cfg.max_pos; p.eps = h->cfg.eps; p.budget_ns = h->budget_ns;
  p.cap_a = h->cap_a; p.cap_qb = h->cap_qb; p.cap_kvb = h->cap_kvb;
  // tensor maps of the decode-size chain, re-encoded when a weight pointer changes
  const W8Maps* maps = nullptr;
  if (T <= kW8SmallRows) {
    W8Maps& m = h->w8maps;
    if (!m.valid || m.src[0] != W_qa || m.src[1] != W_kva || m.src[2] != W_qb || m.src[3] != W_kvb)
      w8_encode_maps(p, h->w8plan, &m);
    if (!m.valid) return cuda_fail(cudaErrorInvalidValue, "W8A8 tensor maps");
    maps = &m;
  }
  int launches = 0;
  cudaError_t e = w8a8_launch(p, h->w8, h->w8plan, maps, h->num_sms, stream, &launches);
  h->last_launches = launches;
  h->last_path = MLA_PATH_AUTO;
  if (e != cudaSuccess) return cuda_fail(e, "w8a8 launch");
  return MLA_OK;
}

mla_status mla_w8a8_quant_rows(const void* x_bf16, int rows, int cols, int8_t* q, float* scale,
                               cudaStream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 8 != 0) return rows < 0 ? MLA_ERR_INVALID_ARG : MLA_ERR_UNSUPPORTED;
  if (rows == 0) return MLA_OK;
  if (!x_bf16 || !q || !scale) return MLA_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(q) || !aligned16(scale)) return MLA_ERR_MISALIGNED;
  cudaError_t e = w8a8_quant_rows_launch(x_bf16, rows, cols, q, scale, stream);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "quant launch");
}

mla_status mla_w8a8_gemm_s32(const int8_t* A, const int8_t* W, int M, int K, int N,
                             int32_t* acc, cudaStream_t stream) {
  if (M < 0 || K <= 0 || N <= 0) return MLA_ERR_INVALID_ARG;
  if (K % 32 != 0 || N % 64 != 0) return MLA_ERR_UNSUPPORTED;
  if (M == 0) return MLA_OK;
  if (!A || !W || !acc) return MLA_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W) || !aligned16(acc)) return MLA_ERR_MISALIGNED;
  cudaError_t e = w8a8_gemm_s32_launch(A, W, M, K, N, acc, stream);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "gemm launch");
}

mla_status mla_prolog_w8a8_operands(mla_prolog_t h, int T, int8_t* q1, float* s1, int8_t* c1,
                                    float* s2, cudaStream_t stream) {
  if (!h || T < 0 || !q1 || !s1 || !c1 || !s2) return MLA_ERR_INVALID_ARG;
  if (h->cfg.quant != MLA_QUANT_W8A8) return MLA_ERR_WRONG_MODE;
  if (T > h->cfg.max_tokens) return MLA_ERR_TOO_MANY_TOKENS;
  cudaError_t e = w8a8_copy_operands(h->w8, T, h->cfg.q_lora_rank, q1, s1, c1, s2, stream);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "copy operands");
}

}  // extern "C"
