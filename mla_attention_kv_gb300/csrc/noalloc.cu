// noalloc.cu -- a KV-prolog entry point that allocates no device memory.
//
// Who needs it: callers that cannot call cudaMalloc.  A serving engine or a
// plugin host that owns every byte of device memory in an arena it planned
// up front has no way to hand a handle's workspace allocation to this
// library, and a latency-critical caller cannot risk an allocation that
// blocks or fails with out-of-memory in the middle of a run.  For them,
// mla_kv_prolog_run_noalloc runs the same fused decode kernel as
// mla_kv_prolog_run, but its scratch (split-K partial sums, the normalised
// latent rows, the grid-barrier counters and the status word) lives in one
// file-scope __device__ array that is part of the loaded library.  Every
// device that loads the library holds this array (kScratchBytes, about
// 4.8 MB) until the process exits.
//
// Rules that follow from sharing one array:
//   - All calls on a device share the array and see what the previous call
//     left in it.  The entry point clears the barrier counters and the
//     status word at the start of every call (an async memset on `stream`);
//     the partial sums and latent rows are fully rewritten before they are
//     read, so nothing else needs clearing.
//   - Two calls that overlap on the same GPU (for example on two streams
//     without an ordering between them) race on the array and give wrong
//     results.  Serialise them on one stream.
//   - The first call in each CUDA context (normally: once per device, in
//     its primary context) resolves the array's device address with
//     cudaGetSymbolAddress while that device is current.  Make that first
//     call before any stream capture begins.  The address is cached per
//     context, by the context's unique id: a __device__ symbol is placed
//     anew in every context that loads the module, so after
//     cudaDeviceReset, or in a second context on the same device, the
//     lookup is simply done again.
//   - Every T runs the decode kernel, in chunks of 64 or 128 rows (one
//     launch per chunk); T above INT_MAX is rejected.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <limits.h>

#include <mutex>

#include "../../include/mla_prolog.h"
#include "internal.h"
#include "tma.h"

namespace mla {
namespace {

// Largest scratch the decode kernel needs: at most 16 split-K chunks of
// [kDecodeMaxTokens, 576] fp32 partials, [kDecodeMaxTokens, 512] latent
// rows, and a 256-byte header (status word at 0, barrier counters at 64).
constexpr size_t kHeaderBytes = 256;
constexpr size_t kMaxSplitK = 16;
constexpr size_t kPartialBytes = kMaxSplitK * kDecodeMaxTokens * kNa * sizeof(float);
constexpr size_t kNrmBytes = kDecodeNrmBytes;
constexpr size_t kScratchBytes = kHeaderBytes + kPartialBytes + kNrmBytes;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch (and the SM count) per CUDA context, keyed by
// the context's unique id, which the driver never reuses within a process.
constexpr int kMaxContexts = 64;
struct Slot {
  unsigned long long ctx_id;  // 0: empty
  unsigned char* ptr;
  int sms;
};
std::mutex g_mu;
Slot g_slots[kMaxContexts];
int g_next;

// Unique id of the current context (the runtime's driver entry points, so
// the library does not link libcuda); false when there is none.
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &q1) == cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
        q2 == cudaDriverEntryPointSuccess) {
      get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(a);
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(b);
    }
  });
  if (!get_cur || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_cur(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS && *id != 0;
}

mla_status fail(mla_status s, const char* what) {
  set_error_text(what);
  return s;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status mla_kv_prolog_run_noalloc(const mla_prolog_config* cfg, int b, int s,
                                                const void* hidden_states,
                                                const int32_t* positions, const void* W_kva,
                                                const void* gamma_kv, const void* W_kvb,
                                                const float* cos_table, const float* sin_table,
                                                void* k_nope, void* value, void* k_pe,
                                                unsigned int* device_status,
                                                cudaStream_t stream) {
  if (!cfg || b < 0 || s < 0) return MLA_ERR_INVALID_ARG;
  const mla_prolog_config& c = *cfg;
  if (c.hidden <= 0 || c.num_heads <= 0 || c.max_pos <= 0 || !(c.eps >= 0.0f) ||
      (c.dtype != MLA_F16 && c.dtype != MLA_BF16))
    return MLA_ERR_INVALID_ARG;
  if (c.quant != MLA_QUANT_NONE) return MLA_ERR_WRONG_MODE;
  if (c.kv_lora_rank != kRank || c.rope_dim != kRope || c.nope_dim != kNope || c.v_dim != kV ||
      c.hidden % 64 != 0)
    return MLA_ERR_UNSUPPORTED;
  const long long T = (long long)b * s;
  if (T == 0) return MLA_OK;
  if (T > INT_MAX) return fail(MLA_ERR_TOO_MANY_TOKENS, "b * s exceeds INT_MAX");
  const void* ptrs[] = {hidden_states, positions, W_kva, gamma_kv, W_kvb, cos_table, sin_table,
                        k_nope, value, k_pe};
  for (const void* q : ptrs)
    if (!q) return MLA_ERR_INVALID_ARG;
  for (const void* q : ptrs)
    if (reinterpret_cast<uintptr_t>(q) & 15u) return MLA_ERR_MISALIGNED;

  // set-up, once per CUDA context (normally once per device): resolve the
  // scratch array's device address while the device is current.  If this
  // thread has no current context yet, cudaSetDevice on the current device
  // binds the device's primary context (it allocates nothing).
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "no usable current device");
  unsigned long long ctx = 0;
  if (!current_context_id(&ctx)) {
    e = cudaSetDevice(dev);
    if (e != cudaSuccess || !current_context_id(&ctx)) return fail(MLA_ERR_CUDA, "no current CUDA context");
  }
  unsigned char* base = nullptr;
  int sms = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    for (const Slot& sl : g_slots)
      if (sl.ctx_id == ctx) {
        base = sl.ptr;
        sms = sl.sms;
        break;
      }
    if (!base) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_scratch);
      if (e != cudaSuccess || !p) return fail(MLA_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed");
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "device attribute query failed");
      base = static_cast<unsigned char*>(p);
      g_slots[g_next] = Slot{ctx, base, sms};
      g_next = (g_next + 1) % kMaxContexts;
    }
  }

  DecodePlan plan;
  if (!decode_plan(c.hidden, c.num_heads, sms, &plan)) return MLA_ERR_UNSUPPORTED;
  if (plan.partial_floats * sizeof(float) > kPartialBytes)
    return fail(MLA_ERR_UNSUPPORTED, "shape needs more split-K scratch than the fixed array holds");

  CUtensorMap tm;
  const uint64_t NB = (uint64_t)c.num_heads * kHeadCols;
  if (!encode_tmap_2d(&tm, c.dtype == MLA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                      W_kvb, NB, kRank, NB * 2, (uint32_t)plan.ngbox * 8, kWkvbBoxRows,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
    return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled failed for W_kvb");

  // the array keeps the previous call's contents: clear status + counters
  e = cudaMemsetAsync(base, 0, kHeaderBytes, stream);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "clearing the scratch header failed");

  DecodeParams p = {};
  p.tmap_wkvb = tm;
  p.hidden = hidden_states; p.positions = positions; p.W_kva = W_kva; p.gamma = gamma_kv;
  p.W_kvb = W_kvb; p.cos_t = cos_table; p.sin_t = sin_table; p.k_nope = k_nope; p.value = value;
  p.k_pe = k_pe;
  p.status = reinterpret_cast<unsigned*>(base);
  p.counters = reinterpret_cast<unsigned*>(base + 64);
  p.partials = reinterpret_cast<float*>(base + kHeaderBytes);
  p.nrm = base + kHeaderBytes + kPartialBytes;
  p.hidden_dim = c.hidden; p.heads = c.num_heads; p.s = s; p.max_pos = c.max_pos;
  p.eps = c.eps; p.budget_ns = c.spin_budget_ns ? c.spin_budget_ns : 1000000000ull;
  const bool bf16 = c.dtype == MLA_BF16;
  const int tt = plan.tt_max;
  for (long long t0 = 0; t0 < T; t0 += tt) {
    p.t0 = (int)t0;
    p.TT = (int)((T - t0) < tt ? (T - t0) : tt);
    e = decode_launch(bf16, false, plan, p, true, stream);
    if (e != cudaSuccess) return fail(MLA_ERR_CUDA, cudaGetErrorString(e));
  }
  if (device_status) {
    e = cudaMemcpyAsync(device_status, base, sizeof(unsigned), cudaMemcpyDeviceToDevice, stream);
    if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "copying the status word failed");
  }
  return MLA_OK;
}
