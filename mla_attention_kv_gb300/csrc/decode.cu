// decode.cu -- fused MLA KV prolog for small token counts (decode).
//
// One launch (one CTA per SM, all resident at once) performs all seven prolog steps
// of "DeepSeek-V2-Lite-Chat MLA KV Prolog 迁移指南" §背景 for up to
// kDecodeMaxTokens token rows.  At these sizes the work is bound by the
// weight stream (W_kva + W_kvb: 6.5 MB for V2-Lite, 41.8 MB for R1), so the
// kernel is built to put every weight byte in flight at kernel start, read
// it exactly once with 16-byte coalesced copies, and keep the number of
// dependent global round trips after the last weight byte arrives small:
//
//   start    each CTA issues (a) TMA box copies of its W_kvb column slice
//            into shared memory (rows [0, kpre); when the slice is larger
//            than the shared-memory budget, rows past kpre are prefetched
//            into L2 now and copied in, in chunks, once phase A is done),
//            (b) cp.async copies of its kv_a tile and of the hidden columns
//            that tile needs, (c) gamma and the cos/sin row of the token row
//            it owns.
//            (kDecodeMaxTokens is the upper bound; the plan picks 128 rows
//            per launch when the W_kvb slice fits in shared memory, else 64)
//   phase A  kv_a_proj split-K: tile = (KB rows x 32 columns) of W_kva;
//            tokens are the M side of mma.sync m16n8k16 (fp32 accumulate);
//            the CTA writes fp32 partial sums [KC, T, 576] to the workspace.
//   barrier  grid-wide, bounded wait (RMSNorm needs the whole 576 row).
//   phase R  fixed-order sum of the KC partials (deterministic), split
//            (step 2), RMSNorm in fp32 (step 3) and RoPE of k_pe (step 6).
//            Small T: every CTA reduces every row itself into shared memory
//            (no second barrier); otherwise one CTA per row writes the
//            normalised row (rounded once to the I/O dtype) to the
//            workspace and a second barrier publishes it.
//   phase B  kv_b_proj split-N over the resident W_kvb slice; the epilogue
//            does the reshape/split (step 5) and the head-major stores
//            (step 7) straight from the accumulators.
// Consecutive launches are chained with programmatic dependent launch: the
// next call's CTAs take each SM as this call's CTA there exits and copy
// their packed weights before waiting for this call to finish.
// Output options (DecodeParams): the latent-cache variant stops after phase
// R (the owner CTA of each row writes the normalised row); a slot mapping
// places rows in a paged cache; per-channel scales turn the stores into
// int8 codes.
#include <mutex>
#include <type_traits>
#include <utility>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tma.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSubK = 64;          // K rows per phase-A pipeline stage
constexpr int kNbA = 32;           // kv_a columns per split-K tile
constexpr int kNblkA = kNa / kNbA; // 18 column blocks
constexpr int kPitchWA = 80;       // smem row pitch of a 32-column tile (odd multiple of 16)
constexpr int kPitchX = 144;       // smem row pitch of a 64-column hidden tile
constexpr int kPitchN = kNrmPitch; // smem row pitch of a 512-column latent row (= workspace pitch)
constexpr int kMaxMT = kDecodeMaxTokens / 16;
constexpr int kSmemBudget = 227 * 1024;
constexpr int kSmemBudget2 = 112 * 1024;  // two CTAs per SM (228 KB, 1 KB reserved per CTA)
constexpr int kRedBytes = 16384;   // cross-warp reduction scratch (<= 32 chains x 512 B)
constexpr int kMiscBytes = 2048;   // gamma, cos/sin row, mbarriers, flag
constexpr int kMaxStagesA = 16;    // deepest phase-A cp.async ring
constexpr int kMaxStreamBufs = 6;  // W_kvb chunk buffers (mbarriers at misc + 1544 ..)
constexpr int kTcbMinCols = 128;   // narrowest column slice for phase B on the tensor cores

__device__ __forceinline__ int col_group_begin(int cta, int ngroups, int grid) {
  return (int)(((long long)cta * ngroups) / grid);
}

// Arrive on counter c and wait until all G CTAs arrived (bounded).
__device__ __forceinline__ bool bar_arrive_wait(unsigned* c, unsigned G,
                                                unsigned long long budget_ns, unsigned* status) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(c) : "memory");
    if (ld_acquire_gpu(c) < G) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(c) < G) {
        if (globaltimer_ns() - t0 > budget_ns) {
          atomicOr(status, kStatusTimeout);
          ok = 0;
          break;
        }
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Bounded wait on an mbarrier phase, with one CTA-wide answer: thread 0
// waits with the time budget, then (on success) every thread observes the
// completed phase itself so the async-proxy writes are visible to it.
__device__ __forceinline__ bool mbar_wait_cta(uint32_t bar, uint32_t parity,
                                              unsigned long long budget_ns, int* flag) {
  if (threadIdx.x == 0) *flag = mbar_wait_bounded(bar, parity, budget_ns) ? 1 : 0;
  __syncthreads();
  const bool ok = *reinterpret_cast<volatile int*>(flag) != 0;
  if (ok) {
    while (!mbar_test_wait(bar, parity)) {
    }
  }
  return ok;
}

// Exit counter: every CTA adds one once it has passed its last grid
// barrier; the CTA that brings the count to G knows that every CTA has left
// every barrier, and resets the counters for the next launch.  The add is
// issued early and its result is only looked at when the CTA finishes, so
// the round trip stays off the critical path.
__device__ __forceinline__ unsigned bar_exit_arrive(unsigned* counters) {
  unsigned old = 0;
  if (threadIdx.x == 0)
    asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(counters + 2));
  return old;
}
__device__ __forceinline__ void bar_exit_finish(unsigned* counters, unsigned old, unsigned G) {
  if (threadIdx.x == 0 && old == G - 1) {
    counters[0] = 0;
    counters[1] = 0;
    __threadfence();
    counters[2] = 0;
  }
}

// f(std::integral_constant<int, c>) for c = 0 .. sizeof...(Cs) - 1, in order
template <int... Cs, typename F>
__device__ __forceinline__ void for_each_c(std::integer_sequence<int, Cs...>, F&& f) {
  (f(std::integral_constant<int, Cs>{}), ...);
}

// NC: CTAs per SM the launch is built for.  NC = 2 (the plan for <= 32 rows:
// under half the shared memory and 128 registers) lets the CTAs of the next
// call in the stream become resident beside this call's and copy their packed
// weights while it runs.
// TB: phase B on the tensor cores (packed weights, plan tc_b; a separate
// instance, so that the other instances carry no tensor-memory code).
template <typename T, int IM, int QM, bool PK, int NC, bool TB>
__global__ void __launch_bounds__(kThreads, NC) decode_kernel(const __grid_constant__ DecodeParams p) {
  using E = Elem<T>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // 1024-byte aligned base (the hidden-state boxes use the 128-byte swizzle)
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, cta = blockIdx.x;
  const int TT = p.TT;
  // m-tiles of 16 rows, rounded up to a power of two so that the phase-B
  // warp grid covers them exactly (padding rows are zero)
  int MT = 1;
  while (MT * 16 < TT) MT *= 2;
  const int rows_x = MT * 16;
  const int H = p.heads;
  const int NB = H * kHeadCols;      // kv_b columns
  const int NG = NB / 8;             // 8-column groups
  const int g0 = col_group_begin(cta, NG, G), g1 = col_group_begin(cta + 1, NG, G);
  const int ng = p.latent ? 0 : g1 - g0;  // latent-cache variant: no kv_b columns
  const int col0 = g0 * 8;
  const int pitchB = p.ngbox * 16;   // odd multiple of 16: conflict-free ldmatrix
  const T* __restrict__ hid = static_cast<const T*>(p.hidden) + (size_t)p.t0 * p.hidden_dim;
  const T* __restrict__ Wa = static_cast<const T*>(p.W_kva);
  unsigned char* sWB = smem + p.off_wb;
  unsigned char* sA = smem + p.off_a;
  float* sRed = reinterpret_cast<float*>(smem + p.off_red);
  T* sGam = reinterpret_cast<T*>(smem + p.off_misc);
  float* sCos = reinterpret_cast<float*>(smem + p.off_misc + 1024);
  float* sSin = sCos + kRope;
  const bool owner = cta < TT;           // this CTA ropes / normalises token row `cta`

  // ---- start: mbarriers, resident W_kvb rows (TMA), L2 prefetch of the rest
  const uint32_t bar_res = smem_u32(smem + p.off_misc + 1536);
  const uint32_t bar_s0 = bar_res + 8;  // streamed chunk buffers 0 .. kMaxStreamBufs-1
  int* sFlag = reinterpret_cast<int*>(smem + p.off_misc + 1600);
  const uint32_t bar_a0 = bar_res + 128;  // phase-A stages 0 .. kMaxStagesA-1 (packed weights)
  const uint32_t bar_lat = bar_res + 256; // latent rows from the workspace (two-barrier mode)
  const uint32_t bar_r0 = bar_res + 272;  // streamed W_kvb chunk batches 0 .. 15 (one use each)
  // phase B on the tensor cores: all MMAs done; the TMEM address (bar_s0 + 8 j
  // then marks the MMAs of K block j done, freeing its slot for a refill)
  const uint32_t bar_tb = bar_res + 72;
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(smem + p.off_misc + 1632);
  if (tid == 0) {
    if constexpr (PK) {
      tma_prefetch_desc(&p.tmap_x);
      for (int i = 0; i < kMaxStagesA; ++i) mbar_init(bar_a0 + 8 * i, 1);
    } else if (!p.latent) {
      tma_prefetch_desc(&p.tmap_wkvb);
    }
    mbar_init(bar_res, 1);
    for (int i = 0; i < kMaxStreamBufs; ++i) mbar_init(bar_s0 + 8 * i, 1);
    mbar_init(bar_tb, 1);
    fence_mbar_init();
    sFlag[1] = 0;  // resident W_kvb copies not issued yet (packed path)
    mbar_init(bar_lat, 1);
    for (int i = 0; i < kRank / kWkvbBoxRows; ++i) mbar_init(bar_r0 + 8 * i, 1);
  }
  __syncthreads();
  // The W_kvb slice is only needed after the grid barrier: its TMA copies
  // are issued once this CTA's first kv_a stage has landed, so the kv_a
  // loads (on the critical path) are not queued behind them in DRAM.
  // Packed weights: this CTA's W_kvb slice is one contiguous block of 512
  // rows x ng 16-byte chunks (chunk order swizzled per row), copied with
  // 1-D bulk copies; otherwise TMA boxes of the [512, H*256] matrix.
  const unsigned char* wkvb_blk = static_cast<const unsigned char*>(p.W_kvb) + (size_t)g0 * (kRank * 16);
  const int pitchW = PK ? ng * 16 : pitchB;  // smem row pitch of the W_kvb rows
  auto issue_wkvb = [&]() {
    mbar_arrive_expect_tx(bar_res, (uint32_t)(ng > 0 ? p.kpre * pitchW : 0));
    if (ng > 0) {
      if constexpr (PK) {
        for (int r = 0; r < p.kpre; r += kWkvbBoxRows)
          bulk_g2s(smem_u32(sWB + r * pitchW), wkvb_blk + (size_t)r * pitchW, kWkvbBoxRows * pitchW, bar_res);
        if (p.kpre < kRank)
          prefetch_l2_bulk(wkvb_blk + (size_t)p.kpre * pitchW, (uint32_t)((kRank - p.kpre) * pitchW));
      } else {
        for (int r = 0; r < p.kpre; r += kWkvbBoxRows)
          tma_load_2d(smem_u32(sWB + r * pitchB), &p.tmap_wkvb, col0, r, bar_res);
        for (int r = p.kpre; r < kRank; r += kWkvbBoxRows)
          tma_prefetch_2d(&p.tmap_wkvb, col0, r);
      }
    }
  };
  // packed weights: warp 1 issues the resident rows, one 32-row bulk copy per
  // lane (thread 0 alone spends ~40 ns per copy instruction), and records
  // that it did in *sWkvbOn for the drains
  int* sWkvbOn = sFlag + 1;
  // K-major blocks (phase B on the tensor cores): N x 128 bytes per 64 K rows
  const int tbB = ng * 8 * 128;
  // Phase A's ring holds every stage of the unit (the packed plans for phase
  // B on the tensor cores): all its copies are issued at the start, so the
  // streamed W_kvb blocks can follow them into L2 right away
  const bool tb_early = TB && (p.off_red - p.off_a) / (rows_x * 128 + kSubK * 64) >= p.KB / kSubK;
  auto issue_wkvb_warp = [&]() {  // warp 1
    if constexpr (TB) {
      // the first tb_res K blocks, contiguous: 16 KB per lane (the later
      // blocks are prefetched into L2 once phase A's copies are all out: a
      // bulk prefetch occupies the SM's copy engine)
      const uint32_t bytes = (uint32_t)(ng > 0 ? p.tb_res * tbB : 0);
      if (lane == 0) mbar_arrive_expect_tx(bar_res, bytes);
      __syncwarp();
      for (uint32_t o = lane * 16384u; o < bytes; o += 32u * 16384u)
        bulk_g2s(smem_u32(sWB) + o, wkvb_blk + o, bytes - o < 16384u ? bytes - o : 16384u, bar_res);
      if (tb_early && ng > 0 && lane < 8 - p.tb_res)
        prefetch_l2_bulk(wkvb_blk + (size_t)(p.tb_res + lane) * tbB, (uint32_t)tbB);
      if (lane == 0) *reinterpret_cast<volatile int*>(sWkvbOn) = 1;
      return;
    }
    if (lane == 0) mbar_arrive_expect_tx(bar_res, (uint32_t)(ng > 0 ? p.kpre * pitchW : 0));
    __syncwarp();
    if (ng > 0) {
      for (int r = lane * kWkvbBoxRows; r < p.kpre; r += 32 * kWkvbBoxRows)
        bulk_g2s(smem_u32(sWB + r * pitchW), wkvb_blk + (size_t)r * pitchW, kWkvbBoxRows * pitchW, bar_res);
      // (no L2 prefetch of the streamed rows: a bulk prefetch occupies the
      // SM's copy engine and the chunk copies would queue behind it)
    }
    if (lane == 0) *reinterpret_cast<volatile int*>(sWkvbOn) = 1;
  };
  // The next kernel in the stream may launch now (it waits for this one
  // before it reads anything this one writes).
  grid_dep_launch_dependents();
  // Everything that may come from the previous kernel in the stream -- hidden
  // rows, positions, gamma, the raw weights, the workspace -- is read after
  // prologue_inputs (every thread calls it once); the packed weight snapshot
  // is read-only and may be copied before.
  int pos = 0;
  unsigned st0 = 0;
  auto prologue_inputs = [&]() {
    grid_dep_wait();
    if (owner && tid == 0) pos = p.positions[p.t0 + cta];
    st0 = *reinterpret_cast<volatile unsigned*>(p.status);
    if (tid < kRank / 8) cp_async16(smem_u32(sGam) + tid * 16, static_cast<const T*>(p.gamma) + tid * 8);
  };

  // ================================================================ phase A
  bool wkvb_on = false;  // resident W_kvb copies issued (raw path: thread 0's view)
  if constexpr (!PK) prologue_inputs();
  {
    const int units = p.KC * kNblkA;
    const int subs = p.KB / kSubK;
    const int my_units = (units > cta) ? (units - cta + G - 1) / G : 0;
    const int nsub = my_units * subs;
    // raw weights: cp.async ring, W rows padded to kPitchWA, hidden rows to
    // kPitchX.  Packed weights: TMA box of the hidden rows (64 columns,
    // 128-byte swizzle) + one 1-D bulk copy of the pre-swizzled W tile per
    // stage, completion on a per-stage mbarrier.
    const int xbytes = PK ? rows_x * 128 : rows_x * kPitchX;
    const int stage_bytes = PK ? xbytes + kSubK * 64 : kSubK * kPitchWA + rows_x * kPitchX;
    // as many stages in flight as the phase-A region holds at this row
    // count (all of them for small T), at least the plan's depth
    int nst = (p.off_red - p.off_a) / stage_bytes;
    if (nst > subs + 1) nst = subs + 1;
    if (nst > kMaxStagesA) nst = kMaxStagesA;
    if (nst < p.nstA) nst = p.nstA;
    if (nsub == 0) {
      if constexpr (PK) {
        if (warp == 1) issue_wkvb_warp();
      } else if (tid == 0) {
        issue_wkvb();
      }
      wkvb_on = true;
    }

    auto load_sub = [&](int i) {  // raw weights: every thread
      const int u = cta + (i / subs) * G;
      const int kc = u / kNblkA, nb = u - kc * kNblkA;
      const int k0 = kc * p.KB + (i % subs) * kSubK;
      unsigned char* st = sA + (i % nst) * stage_bytes;
      const uint32_t w_s = smem_u32(st + xbytes), x_s = smem_u32(st);
      if (tid < kSubK * 4) {
        const int r = tid >> 2, ch = tid & 3;
        cp_async16(w_s + r * kPitchWA + ch * 16, Wa + (size_t)(k0 + r) * kNa + nb * kNbA + ch * 8);
      }
      for (int c = tid; c < rows_x * 8; c += kThreads) {
        const int r = c >> 3, ch = c & 7;
        const int rr = r < TT ? r : 0;
        cp_async16(x_s + r * kPitchX + ch * 16, hid + (size_t)rr * p.hidden_dim + k0 + ch * 8,
                   r < TT ? 16 : 0);
      }
    };
    const unsigned char* Wpk = static_cast<const unsigned char*>(p.W_kva);
    // a stage's weight part (the packed snapshot: read-only, so it may be
    // copied before the previous kernel in the stream has finished) and its
    // hidden-row part (after the dependency wait); one mbarrier phase covers both
    auto issue_stage_w = [&](int i, int slot) {
      const int u = cta + (i / subs) * G;
      const int sub = i % subs;
      const uint32_t bar = bar_a0 + 8 * slot;
      const uint32_t dst = smem_u32(sA + slot * stage_bytes);
      mbar_arrive_expect_tx(bar, (uint32_t)(p.xrows * 128 + kSubK * 64));
      bulk_g2s(dst + xbytes, Wpk + ((size_t)u * p.KB + sub * kSubK) * 64, kSubK * 64, bar);
    };
    auto issue_stage_x = [&](int i, int slot) {
      const int u = cta + (i / subs) * G;
      const int kc = u / kNblkA;
      const int sub = i % subs;
      tma_load_2d(smem_u32(sA + slot * stage_bytes), &p.tmap_x, kc * p.KB + sub * kSubK, p.t0,
                  bar_a0 + 8 * slot);
    };
    auto issue_stage = [&](int i, int slot) {  // packed weights: one lane
      issue_stage_w(i, slot);
      issue_stage_x(i, slot);
    };

    const int nb8 = warp & 3, khalf = warp >> 2;
    // acc[m] takes the first k16 step of each stage, acc2 the second for the
    // first two m-tiles, so that small T still has two independent chains
    // Accumulator slots: for M m-tiles (compile time) stage i and k16 step j
    // add into acc[((i % SC) * JC + j) * M + m], JC = 2 while M <= 4 and SC =
    // 8 / (M * JC) -- eight independent mma chains whatever M is (one chain
    // per accumulator would be bound by the mma.sync latency).  The slots of
    // each m-tile are folded in a fixed order when the unit is done.
    float acc[kMaxMT][4];
#pragma unroll
    for (int m = 0; m < kMaxMT; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;

    // one stage (64 k rows) in smem slot `slot`, accumulator chain C, for M
    // m-tiles (compile time, so only real tiles are issued): each warp takes
    // two of the four k16 steps (khalf) of its 8-column group nb8
    auto stage_mma = [&](auto mt_c, auto ch_c, int slot) {
      constexpr int M = decltype(mt_c)::value;
      constexpr int C = decltype(ch_c)::value;
      constexpr int JC = M <= 4 ? 2 : 1;
      const unsigned char* st = sA + slot * stage_bytes;
      const uint32_t x_s = smem_u32(st), w_s = smem_u32(st + xbytes);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int kk = khalf + 2 * j;
        uint32_t b0, b1;
        if constexpr (PK)  // packed W rows: 64 bytes, chunk c stored at c ^ ((row >> 1) & 3)
          ldsm_x2_trans(w_s + (kk * 16 + (lane & 15)) * 64 + ((nb8 ^ ((lane >> 1) & 3)) * 16), b0, b1);
        else
          ldsm_x2_trans(w_s + (kk * 16 + (lane & 15)) * kPitchWA + nb8 * 16, b0, b1);
#pragma unroll
        for (int m = 0; m < M; ++m) {
          uint32_t a[4];
          if constexpr (PK)  // 128-byte swizzle: chunk c of row r at c ^ (r & 7)
            ldsm_x4(x_s + (m * 16 + (lane & 15)) * 128 + (((kk * 2 + (lane >> 4)) ^ (lane & 7)) * 16),
                    a[0], a[1], a[2], a[3]);
          else
            ldsm_x4(x_s + (m * 16 + (lane & 15)) * kPitchX + (kk * 16 + (lane >> 4) * 8) * 2, a[0],
                    a[1], a[2], a[3]);
          mma16816<E::kBf16>(acc[(C * JC + (JC == 2 ? j : 0)) * M + m], a, b0, b1);
        }
      }
    };
    // Four or eight m-tiles (M = 4 or 8, compile time): warp w takes m-tiles
    // w & 3 (and (w & 3) + 4) of its k-half for all four 8-column groups, so
    // every hidden fragment crosses shared memory once (the mapping above
    // reads the hidden tile once per column group, four times; the W tile is
    // the small operand).  Accumulator slots: M = 4: j * 4 + g (k16 step j of
    // the stage, group g); M = 8: g * 2 + mi (m-tile (w & 3) + 4 mi).
    const int mg = warp & 3;
    auto stage_mma_m = [&](auto mt_c, int slot) {
      constexpr int MI = decltype(mt_c)::value / 4;
      const unsigned char* st = sA + slot * stage_bytes;
      const uint32_t x_s = smem_u32(st), w_s = smem_u32(st + xbytes);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int kk = khalf + 2 * j;
        uint32_t b[4][2];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          if constexpr (PK)
            ldsm_x2_trans(w_s + (kk * 16 + (lane & 15)) * 64 + ((g ^ ((lane >> 1) & 3)) * 16), b[g][0], b[g][1]);
          else
            ldsm_x2_trans(w_s + (kk * 16 + (lane & 15)) * kPitchWA + g * 16, b[g][0], b[g][1]);
        }
#pragma unroll
        for (int mi = 0; mi < MI; ++mi) {
          const int m = mg + 4 * mi;
          uint32_t a[4];
          if constexpr (PK)
            ldsm_x4(x_s + (m * 16 + (lane & 15)) * 128 + (((kk * 2 + (lane >> 4)) ^ (lane & 7)) * 16), a[0], a[1],
                    a[2], a[3]);
          else
            ldsm_x4(x_s + (m * 16 + (lane & 15)) * kPitchX + (kk * 16 + (lane >> 4) * 8) * 2, a[0], a[1], a[2],
                    a[3]);
#pragma unroll
          for (int g = 0; g < 4; ++g) mma16816<E::kBf16>(acc[MI == 1 ? j * 4 + g : g * 2 + mi], a, b[g][0], b[g][1]);
        }
      }
    };
    // stages [i0, i1), stage i in smem slot slot0 + i - i0 and chain i % SC
    auto stages_mma = [&](int i0, int i1, int slot0) {
      auto run = [&](auto mt_c) {
        constexpr int M = decltype(mt_c)::value;
        constexpr int SC = 8 / (M * (M <= 4 ? 2 : 1));
#pragma unroll 1
        for (int q = i0 - i0 % SC; q < i1; q += SC) {
          for_each_c(std::make_integer_sequence<int, SC>{}, [&](auto ch_c) {
            const int i = q + decltype(ch_c)::value;
            if (i >= i0 && i < i1) stage_mma(mt_c, ch_c, slot0 + i - i0);
          });
        }
      };
      auto run_m = [&](auto mt_c) {
#pragma unroll 1
        for (int i = i0; i < i1; ++i) stage_mma_m(mt_c, slot0 + i - i0);
      };
      switch (MT) {
        case 1: run(std::integral_constant<int, 1>{}); break;
        case 2: run(std::integral_constant<int, 2>{}); break;
        case 4: run_m(std::integral_constant<int, 4>{}); break;
        default: run_m(std::integral_constant<int, 8>{}); break;
      }
    };
    // fold the chain slots of each m-tile into acc[m] (fixed order); with the
    // m-tile mapping the two k16 steps' slots of each group (M = 4; M = 8
    // has one slot per group and m-tile)
    auto fold = [&]() {
      auto run = [&](auto mt_c) {
        constexpr int M = decltype(mt_c)::value;
#pragma unroll
        for (int sl = 1; sl < 8 / M; ++sl)
#pragma unroll
          for (int m = 0; m < M; ++m) {
            acc[m][0] += acc[sl * M + m][0]; acc[m][1] += acc[sl * M + m][1];
            acc[m][2] += acc[sl * M + m][2]; acc[m][3] += acc[sl * M + m][3];
          }
      };
      switch (MT) {
        case 1: run(std::integral_constant<int, 1>{}); break;
        case 2: run(std::integral_constant<int, 2>{}); break;
        case 4:
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            acc[g][0] += acc[4 + g][0]; acc[g][1] += acc[4 + g][1];
            acc[g][2] += acc[4 + g][2]; acc[g][3] += acc[4 + g][3];
          }
          break;
        default: break;
      }
    };
    auto unit_done = [&](int i) {
      // unit done: fold the chains and the two k-halves, write the fp32 partial tile
      fold();
      const int u = cta + (i / subs) * G;
      const int kc = u / kNblkA, nb = u - kc * kNblkA;
      if (MT >= 4) {
        // m-tile mapping: slot s holds group s (M = 4, folded) or group s / 2
        // of m-tile mg + 4 (s % 2) (M = 8); the k-half 1 warps hand theirs over
        const int ns = MT == 4 ? 4 : 8;
        if (khalf == 1) {
#pragma unroll
          for (int s = 0; s < 8; ++s)
            if (s < ns)
              *reinterpret_cast<float4*>(sRed + ((mg * 8 + s) * 32 + lane) * 4) =
                  make_float4(acc[s][0], acc[s][1], acc[s][2], acc[s][3]);
        }
        __syncthreads();
        if (khalf == 0) {
          float* P = p.partials + (size_t)kc * kDecodeMaxTokens * kNa;
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            if (s < ns) {
              const int g = MT == 4 ? s : s >> 1, m = mg + 4 * (MT == 4 ? 0 : s & 1);
              const int col = nb * kNbA + g * 8 + 2 * (lane & 3);
              const float4 o = *reinterpret_cast<const float4*>(sRed + ((mg * 8 + s) * 32 + lane) * 4);
              const int r0 = m * 16 + (lane >> 2);
              if (r0 < TT)
                *reinterpret_cast<float2*>(P + (size_t)r0 * kNa + col) = make_float2(acc[s][0] + o.x, acc[s][1] + o.y);
              if (r0 + 8 < TT)
                *reinterpret_cast<float2*>(P + (size_t)(r0 + 8) * kNa + col) =
                    make_float2(acc[s][2] + o.z, acc[s][3] + o.w);
            }
          }
        }
#pragma unroll
        for (int m = 0; m < kMaxMT; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
        return;
      }
      if (khalf == 1) {
#pragma unroll
        for (int m = 0; m < kMaxMT; ++m)
          if (m < MT)
            *reinterpret_cast<float4*>(sRed + ((nb8 * kMaxMT + m) * 32 + lane) * 4) =
                make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
      }
      __syncthreads();
      if (khalf == 0) {
        float* P = p.partials + (size_t)kc * kDecodeMaxTokens * kNa;
        const int col = nb * kNbA + nb8 * 8 + 2 * (lane & 3);
#pragma unroll
        for (int m = 0; m < kMaxMT; ++m) {
          if (m < MT) {
            const float4 o = *reinterpret_cast<const float4*>(sRed + ((nb8 * kMaxMT + m) * 32 + lane) * 4);
            const int r0 = m * 16 + (lane >> 2);
            if (r0 < TT) *reinterpret_cast<float2*>(P + (size_t)r0 * kNa + col) = make_float2(acc[m][0] + o.x, acc[m][1] + o.y);
            if (r0 + 8 < TT) *reinterpret_cast<float2*>(P + (size_t)(r0 + 8) * kNa + col) = make_float2(acc[m][2] + o.z, acc[m][3] + o.w);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < kMaxMT; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
    };
    // cos/sin row of the owned token (position arrived by now or soon)
    auto load_rope_row = [&]() {
      if (owner) {
        if (tid == 0) reinterpret_cast<volatile int*>(sRed)[0] = pos;
        __syncthreads();
        int pp = reinterpret_cast<volatile int*>(sRed)[0];
        if (pp < 0 || pp >= p.max_pos) {
          if (tid == 0) atomicOr(p.status, kStatusBadPosition);
          pp = pp < 0 ? 0 : p.max_pos - 1;
        }
        if (tid < 16) cp_async16(smem_u32(sCos) + tid * 16, p.cos_t + (size_t)pp * kRope + tid * 4);
        else if (tid < 32) cp_async16(smem_u32(sSin) + (tid - 16) * 16, p.sin_t + (size_t)pp * kRope + (tid - 16) * 4);
      }
    };

    if constexpr (PK) {
      // Stages are consumed in groups, one CTA barrier per group: all of
      // them at once when the ring holds them (small T), else groups of
      // nst / 2 in two halves of the ring (one loads while one computes).
      // The CTA owns at most one unit, so unit_done runs once, at the end.
      const int gsz = nsub <= nst ? (nsub > 0 ? nsub : 1) : nst / 2;
      const int ngroups = (nsub + gsz - 1) / gsz;
      auto issue_group = [&](int k) {  // warp 0: lane L issues stage k * gsz + L (gsz <= 16)
        const int i = k * gsz + lane;
        if (lane < gsz && i < nsub) issue_stage(i, (k & 1) * gsz + lane);
      };
      if (warp == 0) {
        for (int k = 0; k < 2 && k < ngroups; ++k) {
          const int i = k * gsz + lane;
          if (lane < gsz && i < nsub) issue_stage_w(i, (k & 1) * gsz + lane);
        }
      }
      // two CTAs per SM: this call may start while the previous one runs, so
      // the resident W_kvb rows (read-only snapshot) go out now as well
      if constexpr (NC == 2) {
        if (warp == 1 && nsub > 0) issue_wkvb_warp();
      }
      prologue_inputs();
      if (warp == 0) {
        for (int k = 0; k < 2 && k < ngroups; ++k) {
          const int i = k * gsz + lane;
          if (lane < gsz && i < nsub) issue_stage_x(i, (k & 1) * gsz + lane);
        }
      }
      // warp 1: the W_kvb slice goes out once the first kv_a stage is in
      if (NC == 1 && warp == 1 && nsub > 0) {
        int ok = 0;
        if (lane == 0) ok = mbar_wait_bounded(bar_a0, 0, p.budget_ns) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) issue_wkvb_warp();
      }
      int issuedG = ngroups < 2 ? ngroups : 2;
      load_rope_row();
      cp_async_commit();
#pragma unroll 1
      for (int k = 0; k < ngroups; ++k) {
        const int i0 = k * gsz, i1 = (i0 + gsz) < nsub ? i0 + gsz : nsub;
        const int slot0 = (k & 1) * gsz;
        const uint32_t par = (k >> 1) & 1;
        if (tid == 0) {
          int ok = 1;
          for (int i = i0; i < i1 && ok; ++i)
            ok = mbar_wait_bounded(bar_a0 + 8 * (slot0 + i - i0), par, p.budget_ns) ? 1 : 0;
          *sFlag = ok;
        }
        __syncthreads();
        if (*reinterpret_cast<volatile int*>(sFlag) == 0) {
          // a copy never completed: wait (bounded) for the rest in flight, then leave;
          // the other CTAs give up at the grid barrier
          if (tid == 0) {
            atomicOr(p.status, kStatusTimeout);
            for (int kk = k; kk < issuedG; ++kk)
              for (int i = kk * gsz; i < (kk + 1) * gsz && i < nsub; ++i)
                mbar_wait_bounded(bar_a0 + 8 * ((kk & 1) * gsz + i - kk * gsz), (kk >> 1) & 1,
                                  drain_budget(p.budget_ns));
            if (*reinterpret_cast<volatile int*>(sWkvbOn)) mbar_wait_bounded(bar_res, 0, drain_budget(p.budget_ns));
          }
          cp_async_wait<0>();
          __syncthreads();
          return;
        }
        for (int i = i0; i < i1; ++i)  // every thread observes the completed phases
          while (!mbar_test_wait(bar_a0 + 8 * (slot0 + i - i0), par)) {
          }
        stages_mma(i0, i1, slot0);
        if (k + 2 < ngroups) {
          __syncthreads();  // every warp is done with these slots
          if (warp == 0) issue_group(k + 2);
          issuedG = k + 3;
        }
      }
      if (nsub > 0) unit_done(nsub - 1);
    } else {
#pragma unroll 1
      for (int s = 0; s < nst - 1; ++s) {
        if (s < nsub) load_sub(s);
        cp_async_commit();
      }
      load_rope_row();
#pragma unroll 1
      for (int i = 0; i < nsub; ++i) {
        cp_async_wait_dyn(nst - 2);
        __syncthreads();
        if (i == 0) {
          if (tid == 0) issue_wkvb();
          wkvb_on = true;
        }
        if (i + nst - 1 < nsub) load_sub(i + nst - 1);
        cp_async_commit();
        stages_mma(i, i + 1, i % nst);
        if ((i % subs) == subs - 1) unit_done(i);
      }
    }
    cp_async_wait<0>();
    __syncthreads();
  }

  // ---- W_kvb rows as a ring of 32-row chunks: chunks [0, nres) were copied
  // into the resident slots at the start; when the slice is larger than that
  // (R1 shapes), chunks nres, nres+1, ... follow into nbuf buffers in the
  // freed phase-A region (behind the latent rows) and then into whichever
  // slot, resident or buffer, the consumer has just finished with, so the
  // stream stays nslots chunks ahead of the MMAs.
  const int nrm_bytes = rows_x * kPitchN;
  unsigned char* sN = sA;
  unsigned char* sWS = sA + nrm_bytes;
  constexpr int CR = kWkvbBoxRows;
  constexpr int nch = kRank / CR;
  const int nres = p.kpre / CR;
  const bool ring = ng > 0 && nres < nch && !TB;
  int nbuf = (p.off_red - p.off_a - nrm_bytes) / (CR * pitchW);
  if (nbuf > kMaxStreamBufs) nbuf = kMaxStreamBufs;
  if (nbuf < 2) nbuf = 2;  // the plan reserves two at the largest row count
  const int nslots = nres + nbuf;
  auto slot_ptr = [&](int sl) -> unsigned char* {
    return sl < nres ? sWB + sl * CR * pitchW : sWS + (sl - nres) * CR * pitchW;
  };
  // Streamed chunks go out in batches -- the buffer chunks at the end of
  // phase A, then the refills after each run of chunks -- and each batch
  // completes on a barrier of its own (bar_r0 + 8 * batch, used once per
  // launch, so its phase is always 0).  Every thread keeps the batch of
  // each chunk (4 bits per chunk) in `bmap`, computed identically.
  int nbatch = 0;       // batches issued
  uint64_t bmap = 0;    // batch of chunk c in bits [4c, 4c + 4)
  auto batch_of = [&](int c) { return (int)((bmap >> (4 * c)) & 15u); };
  auto issue_batch = [&](int c0, int c1) {  // whole warp 0: lane L copies chunk c0 + L
    const uint32_t bar = bar_r0 + 8 * nbatch;
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)((c1 - c0) * CR * pitchW));
    __syncwarp();
    const int c = c0 + lane;
    if (c < c1) {
      const uint32_t dst = smem_u32(slot_ptr(c % nslots));
      if constexpr (PK) {
        bulk_g2s(dst, wkvb_blk + (size_t)c * CR * pitchW, (uint32_t)(CR * pitchW), bar);
      } else {
        tma_load_2d(dst, &p.tmap_wkvb, col0, c * CR, bar);
      }
    }
  };
  auto note_batch = [&](int c0, int c1) {  // every thread
    for (int c = c0; c < c1; ++c) bmap |= (uint64_t)nbatch << (4 * c);
    ++nbatch;
  };
  int issued = ring ? (nslots < nch ? nslots : nch) : nres;  // chunks issued so far
  if (ring) {
    if (warp == 0) issue_batch(nres, issued);
    note_batch(nres, issued);
  }
  // phase B on the tensor cores: K blocks tb_res .. tb_res + tb_buf - 1 go
  // to the buffers behind the 64 KB of latent rows now, one barrier each
  // (bar_r0 + 8 j, j = block - tb_res)
  unsigned char* sTbBuf = sA + 64 * 128 * 8;
  if (TB && ng > 0) {
    if (warp == 0 && lane < p.tb_buf) {
      const uint32_t bar = bar_r0 + 8 * lane;
      mbar_arrive_expect_tx(bar, (uint32_t)tbB);
      bulk_g2s(smem_u32(sTbBuf) + lane * tbB, wkvb_blk + (size_t)(p.tb_res + lane) * tbB, (uint32_t)tbB, bar);
    }
    // the blocks refilled in phase B: into L2 during the barrier and phase R
    // (unless they went there during phase A)
    const int nsl = p.tb_res + p.tb_buf;
    if (!tb_early && warp == 0 && lane >= 16 && lane - 16 < 8 - nsl)
      prefetch_l2_bulk(wkvb_blk + (size_t)(nsl + lane - 16) * tbB, (uint32_t)tbB);
    nbatch = p.tb_buf;
  }
  // on an early exit, wait (bounded) for this CTA's copies still in flight:
  // the resident rows and every issued chunk not yet observed (at most one
  // outstanding phase per slot)
  bool lat_issued = false;  // thread 0: latent-row bulk copy in flight
  auto drain = [&]() {
    cp_async_wait<0>();
    if (tid == 0) {
      mbar_wait_bounded(bar_res, 0, drain_budget(p.budget_ns));
      if (lat_issued) mbar_wait_bounded(bar_lat, 0, drain_budget(p.budget_ns));
      for (int b = 0; b < nbatch; ++b) mbar_wait_bounded(bar_r0 + 8 * b, 0, drain_budget(p.budget_ns));
    }
    __syncthreads();
  };

  if (st0 & kStatusTimeout) {  // poisoned by an earlier timeout: do nothing
    drain();
    return;
  }
  if (!bar_arrive_wait(p.counters + 0, G, p.budget_ns, p.status)) {
    drain();
    return;
  }

  // k_pe outputs j0, j0 + 1, j0 + 32, j0 + 33 of the row at element offset o
  // (dtype values, or their int8 codes)
  auto store_kpe = [&](size_t o, int j0, float a, float b, float c, float d) {
    if (p.c8.k) {
      int8_t* kp = static_cast<int8_t*>(p.k_pe) + o;
      const float* sc = p.c8.inv + 2 * H * kNope;
      const T ra = E::from_f(a), rb = E::from_f(b), rc = E::from_f(c), rd = E::from_f(d);
      *reinterpret_cast<uint16_t*>(kp + j0) =
          (uint16_t)(kv_code(E::to_f(ra), sc[j0]) | (kv_code(E::to_f(rb), sc[j0 + 1]) << 8));
      *reinterpret_cast<uint16_t*>(kp + j0 + 32) =
          (uint16_t)(kv_code(E::to_f(rc), sc[j0 + 32]) | (kv_code(E::to_f(rd), sc[j0 + 33]) << 8));
    } else {
      T* kp = static_cast<T*>(p.k_pe) + o;
      *reinterpret_cast<uint32_t*>(kp + j0) = E::pack(a, b);
      *reinterpret_cast<uint32_t*>(kp + j0 + 32) = E::pack(c, d);
    }
  };

  // ================================================================ phase R
  const float rms_scale = 1.0f / (float)kRank;
  // Phase B on the tensor cores reads the latent rows as its A operand: 8
  // K blocks of 64 rows x 128 bytes (64 columns), 8-row groups 1024 bytes
  // apart, the 16-byte chunk q of row t at chunk q ^ (t & 7).  Byte offset
  // of element (t, c) -- the same in shared memory and in the workspace.
  auto lat_off = [](int t, int c) -> int {
    return (c >> 6) * (64 * 128) + t * 128 + ((((c >> 3) & 7) ^ (t & 7)) << 4) + (c & 7) * 2;
  };
  constexpr bool tcb = TB;
  if (p.single_barrier) {
    // every CTA reduces every row into its own shared memory
    for (int t = 0; t < TT; ++t) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      const bool rope_row = (t == cta);
      const int ncol = rope_row ? kNa / 4 : kRank / 4;
      if (tid < ncol) {
        const float* P = p.partials + (size_t)t * kNa + tid * 4;
        float4 x[16];
#pragma unroll
        for (int kc = 0; kc < 16; ++kc)
          if (kc < p.KC) x[kc] = __ldcg(reinterpret_cast<const float4*>(P + (size_t)kc * kDecodeMaxTokens * kNa));
#pragma unroll
        for (int kc = 0; kc < 16; ++kc)
          if (kc < p.KC) { v.x += x[kc].x; v.y += x[kc].y; v.z += x[kc].z; v.w += x[kc].w; }
      }
      float ss = (tid < kRank / 4) ? (v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w) : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) sRed[64 + warp] = ss;
      __syncthreads();
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) tot += sRed[64 + w];
      __syncthreads();
      if (tid < kRank / 4) {
        const float inv = 1.0f / sqrtf(tot * rms_scale + p.eps);
        const int c = tid * 4;
        uint2 pk = make_uint2(E::pack(v.x * inv * E::to_f(sGam[c]), v.y * inv * E::to_f(sGam[c + 1])),
                              E::pack(v.z * inv * E::to_f(sGam[c + 2]), v.w * inv * E::to_f(sGam[c + 3])));
        *reinterpret_cast<uint2*>(sN + (tcb ? lat_off(t, c) : t * kPitchN + c * 2)) = pk;
      } else if (rope_row && tid < kNa / 4) {
        const int i = tid - kRank / 4, j0 = 2 * i, j1 = 2 * i + 1;
        int ou, in, cnt;
        if (out_place(p.out, p.t0 + t, p.s, p.status, &ou, &in, &cnt))
          store_kpe(((size_t)ou * cnt + in) * kRope, j0, v.x * sCos[j0] - v.y * sSin[j0],
                    v.z * sCos[j1] - v.w * sSin[j1], v.y * sCos[j0 + 32] + v.x * sSin[j0 + 32],
                    v.w * sCos[j1 + 32] + v.z * sSin[j1 + 32]);
      }
    }
    // zero the padding rows of the last m-tile (the tensor-core phase B
    // leaves them: they only reach accumulator rows that are not stored)
    for (int c = tid; !tcb && c < (rows_x - TT) * 64; c += kThreads) {
      const int r = TT + (c >> 6), ch = c & 63;
      *reinterpret_cast<uint4*>(sN + r * kPitchN + ch * 16) = make_uint4(0, 0, 0, 0);
    }
  } else {
    if (owner) {
      const int t = cta;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (tid < kNa / 4) {
        const float* P = p.partials + (size_t)t * kNa + tid * 4;
        float4 x[16];
#pragma unroll
        for (int kc = 0; kc < 16; ++kc)
          if (kc < p.KC) x[kc] = __ldcg(reinterpret_cast<const float4*>(P + (size_t)kc * kDecodeMaxTokens * kNa));
#pragma unroll
        for (int kc = 0; kc < 16; ++kc)
          if (kc < p.KC) { v.x += x[kc].x; v.y += x[kc].y; v.z += x[kc].z; v.w += x[kc].w; }
      }
      float ss = (tid < kRank / 4) ? (v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w) : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) sRed[64 + warp] = ss;
      __syncthreads();
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) tot += sRed[64 + w];
      if (tid < kRank / 4) {
        const float inv = 1.0f / sqrtf(tot * rms_scale + p.eps);
        const int c = tid * 4;
        uint2 pk = make_uint2(E::pack(v.x * inv * E::to_f(sGam[c]), v.y * inv * E::to_f(sGam[c + 1])),
                              E::pack(v.z * inv * E::to_f(sGam[c + 2]), v.w * inv * E::to_f(sGam[c + 3])));
        if (p.latent) {  // latent-cache variant: the row is an output
          *reinterpret_cast<uint2*>(static_cast<T*>(p.latent) + (size_t)(p.t0 + t) * kRank + c) = pk;
        } else {
          if (tcb)
            *reinterpret_cast<uint2*>(static_cast<unsigned char*>(p.nrm) + lat_off(t, c)) = pk;
          else
            *reinterpret_cast<uint2*>(static_cast<T*>(p.nrm) + (size_t)t * (kNrmPitch / 2) + c) = pk;
          // the row is read back by bulk copies (async proxy)
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
      } else if (tid < kNa / 4) {
        const int i = tid - kRank / 4, j0 = 2 * i, j1 = 2 * i + 1;
        int ou, in, cnt;
        if (out_place(p.out, p.t0 + t, p.s, p.status, &ou, &in, &cnt))
          store_kpe(((size_t)ou * cnt + in) * kRope, j0, v.x * sCos[j0] - v.y * sSin[j0],
                    v.z * sCos[j1] - v.w * sSin[j1], v.y * sCos[j0 + 32] + v.x * sSin[j0 + 32],
                    v.w * sCos[j1 + 32] + v.z * sSin[j1 + 32]);
      }
    }
    if (!p.latent && !bar_arrive_wait(p.counters + 1, G, p.budget_ns, p.status)) {
      drain();
      return;
    }
    // latent rows -> shared memory: the workspace rows have the shared-memory
    // layout, so one bulk copy moves all TT of them (all 64 K blocks' rows
    // for the tensor-core phase B); rows past TT are zeroed (mma.sync phase B)
    const uint32_t lat_bytes = tcb ? 64u * 128u * 8u : (uint32_t)(TT * kNrmPitch);
    if (tid == 0 && !p.latent) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      mbar_arrive_expect_tx(bar_lat, lat_bytes);
      bulk_g2s(smem_u32(sN), p.nrm, lat_bytes, bar_lat);
      lat_issued = true;
    }
    for (int c = tid; !tcb && c < (rows_x - TT) * (kPitchN / 16); c += kThreads)
      *reinterpret_cast<uint4*>(sN + TT * kPitchN + c * 16) = make_uint4(0, 0, 0, 0);
  }
  const unsigned exit_old = bar_exit_arrive(p.counters);

  // ================================================================ phase B
  if (ng == 0) {
    drain();  // (the latent rows' bulk copy may still be landing)
    bar_exit_finish(p.counters, exit_old, G);
    return;
  }
  // Work: MT m-tiles x ng 8-column groups x 32 k16 steps.  The warps form a
  // (wm x wn) grid: a warp takes the IM = MT / wm m-tiles {mw, mw + wm, ...}
  // and every wn-th of the ng * ks (group, k-slice) items, so one latent
  // fragment per k16 step serves all of the warp's groups and each W_kvb
  // fragment is read by wm warps only (shared-memory bandwidth, not the
  // tensor pipe, bounds this loop).  ks divides wn, so all items of a warp
  // share one k-slice and the warp only walks its own steps; the slices of
  // an output tile are summed through shared memory.
  const int wm = p.pb_wm, wn = kWarps / wm, ks = p.pb_ks;
  const int mw = warp % wm, wr = warp / wm;
  const int myslice = wr % ks;
  const int nitems = ng * ks;
  float acc[IM * QM][4];
#pragma unroll
  for (int q = 0; q < IM * QM; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
  const uint32_t nrm_u = smem_u32(sN);
  uint32_t aoff[IM], boff[QM];
  bool qv[QM];
#pragma unroll
  for (int i = 0; i < IM; ++i) aoff[i] = (uint32_t)((mw + i * wm) * 16 * kPitchN);
  // packed slices store chunk g of row r at g ^ pack_swizzle(ng, r); the
  // rows a lane addresses are congruent to lane mod 8
  const int xm = PK ? pack_swizzle(ng, lane & 7) : 0;
#pragma unroll
  for (int q = 0; q < QM; ++q) {
    const int j = wr + q * wn;
    qv[q] = j < nitems;
    boff[q] = (uint32_t)((qv[q] ? ((j / ks) ^ xm) : 0) * 16);  // unused items: group 0 (read, not used)
  }

  // K rows are consumed in chunks: the resident rows, then streamed chunks
  cp_async_wait<0>();
  __syncthreads();
  if (!mbar_wait_cta(bar_res, 0, p.budget_ns, sFlag) ||
      (!p.single_barrier && !mbar_wait_cta(bar_lat, 0, p.budget_ns, sFlag))) {
    if (tid == 0) atomicOr(p.status, kStatusTimeout);
    drain();
    bar_exit_finish(p.counters, exit_old, G);
    return;
  }
  // ---- kv_b on the tensor cores (packed weights, wide slices): D [64 token
  // rows, N = 8 ng columns] in 256 TMEM columns, one MMA (M = 64, N, K = 16)
  // per k16 step, A = the latent rows, B = the K-major W_kvb block; thread
  // 0 issues block by block as each is in shared memory.  Blocks [0, R) are
  // resident, [R, R + NBUF) sit in the buffers, block R + NBUF + j is
  // copied into block j's slot once a commit marks block j's MMAs done.
  bool tcb_done = false;
  if constexpr (TB) {
    {
      const int N = ng * 8;
      const int R = p.tb_res, NBUF = p.tb_buf, NSL = R + NBUF;
      const int nref = 8 - NSL > 0 ? 8 - NSL : 0;
      tc::fence_proxy_async_smem();  // latent rows written by this CTA's threads (one-barrier mode)
      if (warp == 2) tc::tmem_alloc(smem_u32(sTmem), 256);
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      const uint32_t tmem = *sTmem;
      auto slot_addr = [&](int a) -> uint32_t {
        int si = a;
        while (si >= NSL) si -= NSL;
        return si < R ? smem_u32(sWB) + si * tbB : smem_u32(sTbBuf) + (si - R) * tbB;
      };
      const uint32_t idesc = tc::idesc_f16(E::kBf16, 64, N, false, false);
      if (tid == 0) {
        int ok = 1, nref_issued = 0;
        auto issue_refill = [&](int j) {  // block NSL + j into block j's slot
          const uint32_t bar = bar_r0 + 8 * (NBUF + j);
          mbar_arrive_expect_tx(bar, (uint32_t)tbB);
          bulk_g2s(slot_addr(NSL + j), wkvb_blk + (size_t)(NSL + j) * tbB, (uint32_t)tbB, bar);
        };
        for (int a = 0; a < 8 && ok; ++a) {
          if (a >= R) {
            if (a >= NSL) {  // a refill: its slot must be free first
              while (nref_issued <= a - NSL && ok) {
                ok = mbar_wait_bounded(bar_s0 + 8 * nref_issued, 0, p.budget_ns) ? 1 : 0;
                if (ok) issue_refill(nref_issued++);
              }
              if (!ok) break;
            }
            ok = mbar_wait_bounded(bar_r0 + 8 * (a - R), 0, p.budget_ns) ? 1 : 0;
            if (!ok) break;
            tc::fence_after_sync();
          }
          const uint32_t wb = slot_addr(a);
          const uint32_t ab = smem_u32(sN) + a * (64 * 128);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_f16(tmem, tc::sdesc_sw128(ab + kk * 32, 16, 1024), tc::sdesc_sw128(wb + kk * 32, 16, 1024),
                        idesc, a > 0 || kk > 0);
          if (a < nref) tc::commit(bar_s0 + 8 * a);
          // refills whose slots are already free go out now
          while (nref_issued < nref && nref_issued <= a && mbar_test_wait(bar_s0 + 8 * nref_issued, 0))
            issue_refill(nref_issued++);
        }
        tc::commit(bar_tb);
        if (!ok) {
          // wait (bounded) for the refills and MMAs in flight before leaving
          atomicOr(p.status, kStatusTimeout);
          for (int j = 0; j < nref_issued; ++j)
            mbar_wait_bounded(bar_r0 + 8 * (NBUF + j), 0, drain_budget(p.budget_ns));
          mbar_wait_bounded(bar_tb, 0, drain_budget(p.budget_ns));
        }
        *sFlag = ok;
      }
      __syncthreads();
      const bool mma_ok = *reinterpret_cast<volatile int*>(sFlag) != 0;
      __syncthreads();
      if (!mma_ok || !mbar_wait_cta(bar_tb, 0, p.budget_ns, sFlag)) {
        if (tid == 0 && mma_ok) {
          atomicOr(p.status, kStatusTimeout);
          mbar_wait_bounded(bar_tb, 0, drain_budget(p.budget_ns));
        }
        drain();
        tc::fence_before_sync();
        __syncthreads();
        if (warp == 2) tc::tmem_dealloc(tmem, 256);
        bar_exit_finish(p.counters, exit_old, G);
        return;
      }
      tc::fence_after_sync();
      // D row r (token row r) is TMEM lane 32 (r / 16) + r % 16 (M = 64);
      // warps q and q + 4 read lane quadrant q, 32 columns at a time, and
      // stage the rows in the I/O dtype in the W area (free now), the
      // layout the store loop below reads
      {
        const int q = warp & 3;
        for (int ch = warp >> 2; ch * 32 < N; ch += 2) {
          uint32_t v[32];
          tc::ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ch * 32), v);
          tc::wait_ld();
          const int r = q * 16 + lane;
          if (lane < 16 && r < TT) {
#pragma unroll
            for (int g = 0; g < 4; ++g)
              if (ch * 32 + g * 8 < N)
                *reinterpret_cast<uint4*>(sWB + r * pitchB + (ch * 4 + g) * 16) = make_uint4(
                    E::pack(__uint_as_float(v[8 * g]), __uint_as_float(v[8 * g + 1])),
                    E::pack(__uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3])),
                    E::pack(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5])),
                    E::pack(__uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7])));
          }
        }
      }
      tc::fence_before_sync();
      __syncthreads();
      if (warp == 2) tc::tmem_dealloc(tmem, 256);
      tcb_done = true;
    }
  }
  // k16 steps of rows [kbase, kbase + krows) whose W_kvb rows start at
  // shared address wbase; a warp walks only the steps of its k-slice
  auto mma_rows = [&](uint32_t wbase, int kbase, int krows) {
    const int steps = krows / 16;
    const int gs0 = kbase / 16;
    const int st0 = ((myslice - gs0 % ks) + ks) % ks;
#pragma unroll 1
    for (int st = st0; st < steps; st += ks) {
      const uint32_t wrow = wbase + (st * 16 + (lane & 15)) * pitchW;
      const uint32_t arow = nrm_u + (lane & 15) * kPitchN + ((kbase + st * 16) + (lane >> 4) * 8) * 2;
      // every fragment of the step is loaded before the first MMA (unused
      // items read a valid address), so the ldmatrix latencies overlap
      uint32_t a[IM][4], b[QM][2];
#pragma unroll
      for (int i = 0; i < IM; ++i) ldsm_x4(arow + aoff[i], a[i][0], a[i][1], a[i][2], a[i][3]);
#pragma unroll
      for (int q = 0; q < QM; ++q) ldsm_x2_trans(wrow + boff[q], b[q][0], b[q][1]);
#pragma unroll
      for (int q = 0; q < QM; ++q) {
        if (qv[q]) {
#pragma unroll
          for (int i = 0; i < IM; ++i) mma16816<E::kBf16>(acc[q * IM + i], a[i], b[q][0], b[q][1]);
        }
      }
    }
  };
  if (tcb_done) {
    // (phase B ran on the tensor cores above)
  } else if (!ring) {
    mma_rows(smem_u32(sWB), 0, p.kpre);
  } else {
    // Chunks are consumed in runs that are contiguous in shared memory (same
    // region, consecutive slots), one MMA sweep and at most one CTA barrier
    // per run; a run ends where the chunks whose slots feed a refill end, so
    // those refills go out as early as possible.
#pragma unroll 1
    for (int c = 0; c < nch;) {
      const int sl = c % nslots;
      const bool refill = c + nslots < nch;
      int e = c + 1;
      while (e < nch && e % nslots == sl + (e - c) && ((e % nslots) < nres) == (sl < nres) &&
             (e + nslots < nch) == refill)
        ++e;
      if (e > nres) {  // some chunks of the run are streamed: wait for their batches
        const int k0 = c > nres ? c : nres;
        const int b0 = batch_of(k0), b1 = batch_of(e - 1);
        if (tid == 0) {
          int ok = 1;
          for (int b = b0; b <= b1 && ok; ++b) ok = mbar_wait_bounded(bar_r0 + 8 * b, 0, p.budget_ns) ? 1 : 0;
          *sFlag = ok;
        }
        __syncthreads();
        if (*reinterpret_cast<volatile int*>(sFlag) == 0) {
          if (tid == 0) atomicOr(p.status, kStatusTimeout);
          drain();
          bar_exit_finish(p.counters, exit_old, G);
          return;
        }
        for (int b = b0; b <= b1; ++b)  // every thread observes the phases
          while (!mbar_test_wait(bar_r0 + 8 * b, 0)) {
          }
      }
      mma_rows(smem_u32(slot_ptr(sl)), c * CR, (e - c) * CR);
      if (refill) {
        __syncthreads();  // every warp is done with these slots
        if (warp == 0) issue_batch(c + nslots, e + nslots);
        note_batch(c + nslots, e + nslots);
        issued = e + nslots;
      }
      c = e;
    }
  }
  bar_exit_finish(p.counters, exit_old, G);

  // ---- epilogue: the [rows_x, ng * 8] output tile goes to shared memory in
  // the I/O dtype (the W_kvb area is free once every warp is past the loop),
  // then out with 16-byte stores: each 8-column group lies inside one head's
  // k_nope or value half, so consecutive threads write consecutive 16 bytes
  // of the head-major outputs (split, step 5; assemble, step 7).
  __syncthreads();
  unsigned char* sO = sWB;
  auto put = [&](int m, int gi, const float* v) {
    const int r = m * 16 + (lane >> 2);
    unsigned char* d = sO + r * pitchB + gi * 16 + (lane & 3) * 4;
    *reinterpret_cast<uint32_t*>(d) = E::pack(v[0], v[1]);
    *reinterpret_cast<uint32_t*>(d + 8 * pitchB) = E::pack(v[2], v[3]);
  };
  if (tcb_done) {
    // (the tile is staged already)
  } else if (ks == 1) {
#pragma unroll
    for (int q = 0; q < QM; ++q)
      if (qv[q]) {
#pragma unroll
        for (int i = 0; i < IM; ++i) put(mw + i * wm, wr + q * wn, acc[q * IM + i]);
      }
  } else {
    // tile (m, gi) is pair gi * MT + m; its ks slices are summed in order
#pragma unroll
    for (int q = 0; q < QM; ++q)
      if (qv[q]) {
#pragma unroll
        for (int i = 0; i < IM; ++i) {
          const int pr = ((wr + q * wn) / ks) * MT + mw + i * wm;
          *reinterpret_cast<float4*>(sRed + ((pr * ks + myslice) * 32 + lane) * 4) =
              make_float4(acc[q * IM + i][0], acc[q * IM + i][1], acc[q * IM + i][2], acc[q * IM + i][3]);
        }
      }
    __syncthreads();
    for (int pr = warp; pr < MT * ng; pr += kWarps) {
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      for (int k = 0; k < ks; ++k) {
        const float4 o = *reinterpret_cast<const float4*>(sRed + ((pr * ks + k) * 32 + lane) * 4);
        v[0] += o.x; v[1] += o.y; v[2] += o.z; v[3] += o.w;
      }
      put(pr % MT, pr / MT, v);
    }
  }
  __syncthreads();
  T* kn = static_cast<T*>(p.k_nope);
  T* vv = static_cast<T*>(p.value);
  for (int idx = tid; idx < TT * ng; idx += kThreads) {
    const int r = idx / ng, gi = idx - r * ng;
    const int j = col0 + gi * 8;
    const int hh = j / kHeadCols, e = j - hh * kHeadCols;
    T* base = (e < kNope) ? kn : vv;
    const int ee = (e < kNope) ? e : e - kNope;
    int ou, in, cnt;
    if (!out_place(p.out, p.t0 + r, p.s, p.status, &ou, &in, &cnt)) continue;
    const size_t o = (((size_t)ou * H + hh) * cnt + in) * kNope + ee;
    if (p.c8.k) {  // int8 KV cache: codes of the 8 dtype values
      const T* x = reinterpret_cast<const T*>(sO + r * pitchB + gi * 16);
      const float* sc = p.c8.inv + (e < kNope ? 0 : H * kNope) + hh * kNope + ee;
      uint32_t w[2] = {0u, 0u};
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i >> 2] |= kv_code(E::to_f(x[i]), sc[i]) << (8 * (i & 3));
      *reinterpret_cast<uint2*>(reinterpret_cast<int8_t*>(e < kNope ? p.k_nope : p.value) + o) =
          make_uint2(w[0], w[1]);
    } else {
      *reinterpret_cast<uint4*>(base + o) = *reinterpret_cast<const uint4*>(sO + r * pitchB + gi * 16);
    }
  }
}

// Phase-B register tiles: IM m-tiles x QM column groups per warp.
constexpr int kVariants[3][2] = {{1, 4}, {1, 8}, {2, 8}};

template <typename T, bool PK>
const void* kernel_for(int variant, bool two_per_sm, bool tcb) {
  if constexpr (PK) {
    if (tcb) return (const void*)decode_kernel<T, 1, 4, true, 1, true>;  // (no mma.sync phase B)
  }
  if (two_per_sm) {
    if (variant == 0) return (const void*)decode_kernel<T, 1, 4, PK, 2, false>;
    if (variant == 1) return (const void*)decode_kernel<T, 1, 8, PK, 2, false>;
    return (const void*)decode_kernel<T, 2, 8, PK, 2, false>;
  }
  if (variant == 0) return (const void*)decode_kernel<T, 1, 4, PK, 1, false>;
  if (variant == 1) return (const void*)decode_kernel<T, 1, 8, PK, 1, false>;
  return (const void*)decode_kernel<T, 2, 8, PK, 1, false>;
}

}  // namespace

// ---------------------------------------------------------------- int8 KV cache
namespace {
__global__ void c8_reciprocals_kernel(const float* __restrict__ k, const float* __restrict__ v,
                                      const float* __restrict__ kpe, float* __restrict__ inv, int nkv) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < nkv) {
    inv[i] = __fdiv_rn(1.0f, k[i]);
    inv[nkv + i] = __fdiv_rn(1.0f, v[i]);
  }
  if (i < kRope) inv[2 * nkv + i] = __fdiv_rn(1.0f, kpe[i]);
}
}  // namespace

cudaError_t c8_reciprocals_launch(const C8Scales& c8, int heads, cudaStream_t stream) {
  const int nkv = heads * kNope;
  const int n = nkv > kRope ? nkv : kRope;
  c8_reciprocals_kernel<<<(n + 255) / 256, 256, 0, stream>>>(c8.k, c8.v, c8.kpe, c8.inv, nkv);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- weight packing
// W_kva [hidden, 576] -> one contiguous tile per phase-A unit u = kc * 18 + nb
// (the unit CTA u computes): KB rows of 32 columns (64 bytes), the four
// 16-byte chunks of row r stored at c ^ ((r >> 1) & 3) so that ldmatrix of
// 16 consecutive rows meets no bank conflict.
__global__ void pack_wkva_kernel(const uint4* __restrict__ W, uint4* __restrict__ out, int hidden,
                                 int KB) {
  const long n = (long)hidden * (kNa / 8);
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const int row = (int)(i / (kNa / 8)), cc = (int)(i % (kNa / 8));
    const int nb = cc >> 2, c = cc & 3;
    const int kc = row / KB, r = row - kc * KB;
    const long u = (long)kc * kNblkA + nb;
    out[(u * KB + r) * 4 + (c ^ ((r >> 1) & 3))] = W[i];
  }
}

// W_kvb [512, NG*8] -> per CTA c one contiguous block of its column groups
// [g0(c), g0(c+1)): 512 rows x ng 16-byte chunks, chunk j of row r stored at
// j ^ pack_swizzle(ng, r).  Block c starts at g0(c) * 512 chunks.
__global__ void pack_wkvb_kernel(const uint4* __restrict__ W, uint4* __restrict__ out, int NG,
                                 int G) {
  const long n = (long)kRank * NG;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const int r = (int)(i / NG), g = (int)(i % NG);
    // owner: the CTA c with g0(c) <= g < g0(c + 1), g0(c) = floor(c * NG / G)
    const int c = (int)(((long)(g + 1) * G + NG - 1) / NG) - 1;
    const int g0 = col_group_begin(c, NG, G), ng = col_group_begin(c + 1, NG, G) - g0;
    const int j = g - g0;
    out[(long)g0 * kRank + (long)r * ng + (j ^ pack_swizzle(ng, r))] = W[i];
  }
}

// W_kvb for phase B on the tensor cores: CTA c's slice (groups [g0, g0 +
// ng), N = 8 ng columns) is 8 blocks of 64 K rows; block a holds N rows,
// one per output column n, of 64 K values (128 bytes), the 16-byte chunk q
// of row n stored at chunk q ^ (n & 7) -- the K-major, 128-byte-swizzle
// operand layout, 8-row groups 1024 bytes apart.  One output chunk (8 K
// values of one column) per thread step; the slice of CTA c starts where
// the row-major packing's does (g0 * 512 chunks).
__global__ void pack_wkvb_kmajor_kernel(const uint16_t* __restrict__ W, uint4* __restrict__ out, int NG,
                                        int G) {
  const int NB = NG * 8;
  const long n = (long)NB * (kRank / 8);
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const int col = (int)(i / (kRank / 8)), q8 = (int)(i % (kRank / 8));
    const int g = col / 8;
    const int c = (int)(((long)(g + 1) * G + NG - 1) / NG) - 1;
    const int g0 = col_group_begin(c, NG, G), ng = col_group_begin(c + 1, NG, G) - g0;
    const int nrow = col - g0 * 8, N = ng * 8;
    const int a = q8 / 8, q = q8 % 8;
    uint32_t v[4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
      v[t] = (uint32_t)W[(size_t)(q8 * 8 + 2 * t) * NB + col] |
             ((uint32_t)W[(size_t)(q8 * 8 + 2 * t + 1) * NB + col] << 16);
    out[(long)g0 * (kRank * 16 / 16) + (long)a * N * 8 + (long)nrow * 8 + (q ^ (nrow & 7))] =
        make_uint4(v[0], v[1], v[2], v[3]);
  }
}

cudaError_t decode_pack_weights(const DecodePlan& plan, int hidden, int heads, const void* W_kva,
                                const void* W_kvb, void* pk_kva, void* pk_kvb, cudaStream_t stream) {
  const int NG = heads * kHeadCols / 8;
  pack_wkva_kernel<<<plan.grid * 4, 256, 0, stream>>>(static_cast<const uint4*>(W_kva),
                                                     static_cast<uint4*>(pk_kva), hidden, plan.KB);
  if (plan.tc_b)
    pack_wkvb_kmajor_kernel<<<plan.grid * 4, 256, 0, stream>>>(static_cast<const uint16_t*>(W_kvb),
                                                              static_cast<uint4*>(pk_kvb), NG, plan.grid);
  else
    pack_wkvb_kernel<<<plan.grid * 4, 256, 0, stream>>>(static_cast<const uint4*>(W_kvb),
                                                       static_cast<uint4*>(pk_kvb), NG, plan.grid);
  return cudaGetLastError();
}

cudaError_t decode_cl_pack_wkvb(const ClPlan& plan, int heads, const void* W_kvb, void* out,
                                cudaStream_t stream) {
  const int ctas = plan.clusters * kClSize;
  pack_wkvb_kernel<<<ctas * 4, 256, 0, stream>>>(static_cast<const uint4*>(W_kvb), static_cast<uint4*>(out),
                                                  heads * kHeadCols / 8, ctas);
  return cudaGetLastError();
}

// Shared-memory plan for `tt` token rows per launch; false if it cannot be
// laid out (or, with `resident_only`, if W_kvb would have to be streamed).
static bool plan_for(int tt, bool resident_only, int hidden, int heads, int num_sms,
                     DecodePlan* plan, int budget = kSmemBudget) {
  const int G = num_sms;
  // split-K of kv_a: the smallest KB (multiple of 64 dividing hidden) with
  // at most one (KB x 32-column) tile per CTA
  int KB = 0;
  for (int kb = 64; kb <= hidden; kb += 64) {
    if (hidden % kb == 0 && (hidden / kb) * kNblkA <= G) {
      KB = kb;
      break;
    }
  }
  if (KB == 0 || hidden / KB > 16) return false;
  const int KC = hidden / KB;
  const int NG = heads * kHeadCols / 8;
  const int ngmax = (NG + G - 1) / G;
  const int ngbox = ngmax | 1;            // odd 16-byte chunks per row: conflict-free ldmatrix
  if (ngbox * 8 > 256) return false;      // TMA box inner extent
  for (int mt = 1; mt <= tt / 16; mt *= 2) {
    int v, wm, ks;
    if (!decode_phase_b(mt, ngmax, &v, &wm, &ks)) return false;
  }
  const int pitchB = ngbox * 16;
  const int subs = KB / kSubK;
  const int stageA = kSubK * kPitchWA + tt * kPitchX;
  const int nstA = subs < 4 ? (subs < 2 ? 2 : subs) : 4;
  const int nrm_bytes = tt * kPitchN;
  // + 1024 to align the dynamic shared memory base, + up to 1023 to align region A
  const int fixed = kRedBytes + kMiscBytes + 256 + 2048;
  // Region A holds the phase-A ring, later the latent rows plus (when the
  // W_kvb slice does not fit) two stream buffers; the rest of the budget
  // keeps W_kvb rows resident from kernel start.
  int regionA = nstA * stageA;
  if (regionA < nrm_bytes) regionA = nrm_bytes;
  int kpre = (budget - fixed - regionA) / pitchB;
  int kchunk = kWkvbBoxRows;
  if (kpre >= kRank) {
    kpre = kRank;
  } else {
    if (resident_only) return false;
    if (regionA < nrm_bytes + 2 * kWkvbBoxRows * pitchB) regionA = nrm_bytes + 2 * kWkvbBoxRows * pitchB;
    kpre = (budget - fixed - regionA) / pitchB / kWkvbBoxRows * kWkvbBoxRows;
    // Slices for phase B on the tensor cores (below): most of the slice
    // streams in after phase A anyway, so the shared memory goes to a
    // phase-A ring that holds every stage of the CTA's unit (packed path:
    // all its copies in flight at once; resident W_kvb rows would share the
    // copy engine with them), keeping one K block of the slice resident.
    const int blk_tb = ngmax * 8 * 128;
    if (tt <= 64 && budget > kSmemBudget2 && ngmax * 8 >= kTcbMinCols) {
      const int keep = blk_tb > 64 * pitchB ? blk_tb : 64 * pitchB;
      int kpre_tb = (keep + pitchB - 1) / pitchB;
      kpre_tb = (kpre_tb + kWkvbBoxRows - 1) / kWkvbBoxRows * kWkvbBoxRows;
      if (kpre_tb < tt) kpre_tb = tt;
      const int off_a_tb = (kpre_tb * pitchB + 1023) / 1024 * 1024;
      const int all_stages = subs * (tt * 128 + kSubK * 64);
      int region_tb = (budget - 1024 - kMiscBytes - kRedBytes - off_a_tb) / 128 * 128;
      if (region_tb > all_stages) region_tb = all_stages;
      if (region_tb > regionA && kpre_tb <= kpre) {
        regionA = region_tb;
        kpre = kpre_tb;
      }
    }
    kchunk = (regionA - nrm_bytes) / (2 * pitchB) / kWkvbBoxRows * kWkvbBoxRows;
    if (kpre < 0 || kchunk < kWkvbBoxRows) return false;
  }
  plan->grid = G;
  plan->tt_max = tt;
  plan->KB = KB;
  plan->KC = KC;
  plan->kpre = kpre;
  plan->kchunk = kchunk;
  plan->nstA = nstA;
  plan->ngbox = ngbox;
  plan->ngmax = ngmax;
  plan->off_wb = 0;
  plan->off_a = (kpre * pitchB + 1023) / 1024 * 1024;
  plan->off_red = plan->off_a + (regionA + 127) / 128 * 128;
  plan->off_misc = plan->off_red + kRedBytes;
  plan->smem = (size_t)plan->off_misc + kMiscBytes + 1024;  // + base alignment slack
  if (plan->smem > (size_t)budget) return false;
  plan->two_per_sm = budget <= kSmemBudget2;
  if (kpre < tt) return false;  // the output tile is staged in the W_kvb area
  // phase B on the tensor cores for wide column slices (one MMA per k16 step
  // costs the same issue time whatever N is, so it pays from N = 128 on):
  // M = 64 token rows, the latent rows as 8 K blocks of 64 rows x 128 bytes
  // (64 KB) at the start of region A, W_kvb K blocks of N x 128 bytes in
  // the W area and in whole buffers behind the latent rows
  plan->tc_b = false;
  plan->tb_res = plan->tb_buf = 0;
  const int blk = ngmax * 8 * 128;
  const int spare = plan->off_red - plan->off_a - 64 * 128 * 8;
  if (tt <= 64 && !plan->two_per_sm && ngmax * 8 >= kTcbMinCols && spare >= 0 &&
      plan->off_a >= blk && plan->off_a >= 64 * pitchB) {
    plan->tc_b = true;
    plan->tb_res = plan->off_a / blk < 8 ? plan->off_a / blk : 8;
    const int nb = spare / blk;
    plan->tb_buf = nb < 8 - plan->tb_res ? nb : 8 - plan->tb_res;
  }
  plan->partial_floats = (size_t)KC * kDecodeMaxTokens * kNa;
  return true;
}

bool decode_phase_b(int mt, int ngmax, int* variant, int* wm_out, int* ks_out) {
  // cost: mma.sync per warp on the critical path, with fewer than three
  // independent chains counted as three (latency), then fewer slices
  // (less reduction), then the smaller register tile
  long best = -1;
  for (int v = 0; v < 3; ++v) {
    const int IM = kVariants[v][0], QM = kVariants[v][1];
    if (mt % IM != 0 || mt / IM > kWarps) continue;
    const int wm = mt / IM, wn = kWarps / wm;
    for (int ks = 1; ks <= 8; ks *= 2) {
      if (wn % ks != 0) continue;
      const int per = (ngmax * ks + wn - 1) / wn;
      if (per > QM) continue;
      if (ks > 1 && mt * ngmax * ks > kRedBytes / 512) continue;
      const int chains = IM * per;
      const long cost = ((long)(32 / ks) * (chains < 3 ? 3 : chains)) * 64 + ks * 4 + v;
      if (best < 0 || cost < best) {
        best = cost;
        *variant = v;
        *wm_out = wm;
        *ks_out = ks;
      }
    }
  }
  return best >= 0;
}

bool decode_plan_small(int hidden, int heads, int num_sms, DecodePlan* plan) {
  // rows per launch for which two CTAs fit on an SM, W_kvb slice resident
  return num_sms >= kDecodeSmallTokens &&
         plan_for(kDecodeSmallTokens, true, hidden, heads, num_sms, plan, kSmemBudget2);
}

bool decode_plan(int hidden, int heads, int num_sms, DecodePlan* plan) {
  if (hidden % 64 != 0 || heads < 1) return false;
  // 128 rows per launch when the whole W_kvb slice still stays resident
  // (V2-Lite), else 64 (R1 streams part of its slice)
  if (num_sms >= kDecodeMaxTokens && plan_for(kDecodeMaxTokens, true, hidden, heads, num_sms, plan))
    return true;
  return num_sms >= 64 && plan_for(64, false, hidden, heads, num_sms, plan);
}

int decode_box_rows(int TT, int ntok) {
  int mt = 1;
  while (mt * 16 < TT) mt *= 2;
  return 16 * mt < ntok ? 16 * mt : ntok;
}

bool decode_encode_xmap(CUtensorMap* map, bool bf16, const void* hidden, int hidden_dim, int ntok,
                        int rows) {
  return encode_tmap_2d(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        hidden, (uint64_t)hidden_dim, (uint64_t)ntok, (uint64_t)hidden_dim * 2, 64,
                        (uint32_t)rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Per kernel instance and device: the dynamic shared-memory limit, raised
// when a plan needs more than any before (the attribute belongs to the
// kernel, so it is never lowered: another handle's plan may need more), and
// per shared-memory size the number of CTAs the device holds at once, which
// must cover the grid (the CTAs wait for one another at the grid barriers).
// Both are cached: the driver calls cost about a microsecond each, and a
// decode call launches one of 24 instances.
static cudaError_t prepare_instance(const void* fn, size_t smem, int grid) {
  struct Limit {
    const void* fn;
    int dev;
    size_t smem;
  };
  struct Fit {
    const void* fn;
    int dev;
    size_t smem;
    int resident;  // CTAs resident at once at this shared-memory size
  };
  static std::mutex mu;
  static Limit lim[128];
  static Fit fit[256];
  static int nl = 0, nf = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  int i = 0;
  while (i < nl && !(lim[i].fn == fn && lim[i].dev == dev)) ++i;
  if (i == nl || lim[i].smem < smem) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (i < nl) lim[i].smem = smem;
    else if (nl < 128) lim[nl++] = Limit{fn, dev, smem};
  }
  int j = 0;
  while (j < nf && !(fit[j].fn == fn && fit[j].dev == dev && fit[j].smem == smem)) ++j;
  int resident;
  if (j < nf) {
    resident = fit[j].resident;
  } else {
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    resident = per_sm * sms;
    if (nf < 256) fit[nf++] = Fit{fn, dev, smem, resident};
  }
  return resident < grid ? cudaErrorCooperativeLaunchTooLarge : cudaSuccess;
}

cudaError_t decode_launch(bool bf16, bool packed, const DecodePlan& plan, const DecodeParams& p0,
                          bool pdl, cudaStream_t stream, const CUtensorMap* xmap) {
  int mt = 1;
  while (mt * 16 < p0.TT) mt *= 2;
  int variant, wm, ks;
  if (!decode_phase_b(mt, plan.ngmax, &variant, &wm, &ks)) return cudaErrorInvalidValue;
  const bool two = plan.two_per_sm;
  const bool tcb = packed && plan.tc_b;
  const void* fn = packed ? (bf16 ? kernel_for<__nv_bfloat16, true>(variant, two, tcb)
                                  : kernel_for<__half, true>(variant, two, tcb))
                          : (bf16 ? kernel_for<__nv_bfloat16, false>(variant, two, false)
                                  : kernel_for<__half, false>(variant, two, false));
  cudaError_t e = prepare_instance(fn, plan.smem, plan.grid);
  if (e != cudaSuccess) return e;
  DecodeParams p = p0;
  p.KB = plan.KB;
  p.KC = plan.KC;
  p.kpre = plan.kpre;
  p.kchunk = plan.kchunk;
  p.nstA = plan.nstA;
  p.ngbox = plan.ngbox;
  p.pb_wm = wm;
  p.pb_ks = ks;
  p.off_wb = plan.off_wb;
  p.off_a = plan.off_a;
  p.off_red = plan.off_red;
  p.off_misc = plan.off_misc;
  p.tcb = tcb ? 1 : 0;
  p.tb_res = plan.tb_res;
  p.tb_buf = plan.tb_buf;
  if (packed) {
    // hidden rows [ntok, hidden]: boxes of 64 columns x xrows rows, 128-byte
    // swizzle; rows past ntok read as zero.  The box is at most the tensor's
    // height; smem rows past it only feed output rows that are not stored.
    p.xrows = decode_box_rows(p.TT, p.ntok);
    if (xmap)
      p.tmap_x = *xmap;
    else if (!decode_encode_xmap(&p.tmap_x, bf16, p.hidden, p.hidden_dim, p.ntok, p.xrows))
      return cudaErrorInvalidValue;
  }
  // one barrier when every CTA can afford to reduce all rows itself
  // (the latent-cache variant has no phase B: the owners write the rows out)
  p.single_barrier = (!p.latent && p.TT * plan.KC <= kSingleBarrierRowsTimesChunks) ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  // Not a cooperative launch: a cooperative grid starts only once the
  // previous grid has left every SM, which cancels the programmatic
  // dependency (measured: 14.1 us per eager V2-Lite call with both
  // attributes, 10.7 us with the dependency alone).  The grid barriers need
  // every CTA resident at once; prepare_instance checked that the device
  // holds the whole grid, and the dependency launches this grid only after
  // every CTA of the previous one has started, so no CTA of this grid waits
  // for a slot held by a later grid.  A CTA that another process's work
  // keeps off the GPU for longer than the spin budget makes the others
  // give up at the barrier with MLA_ERR_DEVICE_TIMEOUT instead of hanging.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  void* args[] = {&p};
  if (pdl) {
    // a runtime that does not take the dependency attribute: launch this
    // call without it
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaErrorInvalidValue && e != cudaErrorNotSupported) return e;
    cudaGetLastError();
  }
  cfg.numAttrs = 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace mla
