// prefill.cu -- tensor-core (tcgen05 / TMEM / TMA) MLA KV prolog for large
// token counts.
//
// One CTA per 128-row token tile (persistent over tiles when there are
// more tiles than SMs).  The two contractions of "DeepSeek-V2-Lite-Chat MLA
// KV Prolog 迁移指南" §背景 (steps 1 and 4) run as tcgen05.mma with fp32
// accumulators in tensor memory; RMSNorm (step 3) sits between them in the
// epilogue warps, and split / RoPE / reshape / head-major assemble (steps
// 2, 5, 6, 7) are the epilogues, so nothing but the inputs and the three
// outputs touches global memory.
//
// Warp roles (192 threads):
//   warp 0   TMA producer: hidden tile [128 x 64] and this CTA's half of
//            every weight tile, 128-byte swizzled, into shared-memory rings:
//            5 stages for the k_pe pass, 3 for the compressed_kv pass, 5 for
//            kv_b (the rings reuse the same 224 KB at different times).
//   warp 1   allocates 512 TMEM columns (both CTAs of the pair); one thread
//            of the even CTA issues every MMA of the pair.
//   warps 2-5 epilogue; warp w owns TMEM lanes 32*(w%4) .. +31, i.e. token
//            rows of the tile, one row per thread.
// CTAs run in pairs (clusters of two neighbouring tiles) on the 2-SM MMA
// (tcgen05.mma.cta_group::2, M = 256): each CTA holds its own 128 token rows
// and half of the N columns of every weight tile, and both CTAs' copies
// complete on the even CTA's barriers.
// Per tile:
//   (a) k_pe pass: C[:, 512:576] = X * W_kva[:, 512:576], drained by the
//       epilogue: RoPE (de-interleave + rotate_half) -> k_pe.  When CTA
//       pairs are left over after every tile has its own CTA, those pairs
//       run pass (a) for all tiles and the tile CTAs skip it.
//   (b) compressed_kv pass: C[:, 0:512] as two N = 256 MMAs per K step,
//       filling all 512 TMEM columns; the epilogue reads each row twice
//       (sum of squares, then normalise * gamma) and writes the normalised
//       tile, rounded once to the I/O dtype, into shared memory in the
//       K-major 128-byte-swizzled layout of the next MMA's A operand.
//   (c) kv_b: one N = 256 MMA tile per head (128 k_nope + 128 value
//       columns), K = 512 from the shared-memory tile, accumulators
//       double-buffered in TMEM so head j+1 runs while the epilogue stores
//       head j as k_nope[b, j, s, :] / value[b, j, s, :] (on the CTA's last
//       tile through a shared-memory staging area, so that each store
//       instruction writes whole 128-byte row segments).
// Output options (PrefillParams): the latent-cache variant stops after (b)
// and writes the normalised rows; a slot mapping places rows in a paged
// cache; per-channel scales turn the stores into int8 codes.
// The fp32 accumulator width is 512 TMEM columns, which is why the 576
// kv_a columns take two passes.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tma.h"

namespace mla {
namespace {

constexpr int kPfThreads = 192;
constexpr int kCl = 2;                      // CTAs per cluster: one 2-SM MMA pair
constexpr int kBM = 128;                    // token rows per CTA tile (256 per pair)
constexpr int kBK = 64;                     // K elements per TMA box / stage
constexpr uint32_t kA2Bytes = 8 * 16384;    // normalised tile: 8 K-chunks x [128 x 64], [0, 128 KB)
constexpr uint32_t kS0Base = 0;             // k_pe stages: [0, 120 KB)
constexpr uint32_t kS0Bytes = 24576;        // k_pe stage: X 16 KB + the 64 k_pe columns of W 8 KB
constexpr int kS0Stages = 5;
constexpr uint32_t kS1Bytes = 49152;        // compressed_kv stage: X 16 KB + this CTA's half of two N = 256 tiles
constexpr int kS1Stages = 3;                // [0, 144 KB): the last stage reaches past the A2 tile
constexpr uint32_t kS2Base = kS1Stages * kS1Bytes;  // kv_b stages after both: [144 KB, 224 KB)
constexpr uint32_t kS2Bytes = 16384;        // kv_b stage: this CTA's half of [64 K x 256 N]
constexpr int kS2Stages = 5;
constexpr uint32_t kBarBase = kS2Base + kS2Stages * kS2Bytes;  // 229376
// kv_b epilogue staging (last tile): [128 KB, 144 KB), 4 KB per epilogue
// warp, past the normalised tile and before the kv_b ring
constexpr uint32_t kStageBase = kA2Bytes;
constexpr uint32_t kStageWarp = 32 * 128;
static_assert(kStageBase + 4 * kStageWarp <= kS2Base, "staging between the A2 tile and the kv_b ring");
constexpr uint32_t kGamBase = kBarBase + 512;                  // gamma [512], I/O dtype
constexpr uint32_t kSmemBytes = kGamBase + 1024 + 1024;        // + alignment slack
static_assert(kS0Base + kS0Stages * kS0Bytes <= kA2Bytes, "k_pe ring inside the A2 area");
static_assert(kS2Base >= kA2Bytes, "kv_b ring clear of the A2 tile");

struct PfShared {
  uint64_t full0[kS0Stages], empty0[kS0Stages];
  uint64_t full1[kS1Stages], empty1[kS1Stages];
  uint64_t full2[kS2Stages], empty2[kS2Stages];
  uint64_t tfull[2], tempty[2];
  uint64_t a2_ready, a2_free, mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(PfShared) <= 512, "barrier block");

struct PfArgs {
  CUtensorMap tm_x;    // hidden [T, hidden], box {64, 128}, SW128
  CUtensorMap tm_wa;   // W_kva [hidden, 576], box {64, 64}, SW128 (the k_pe columns)
  CUtensorMap tm_wa3;  // W_kva as [hidden][9][64], box {64, 64, 2}: one CTA's half of an N = 256 tile
  CUtensorMap tm_wb3;  // W_kvb as [512][H*4][64], box {64, 64, 2}: one CTA's half of a head
  PrefillParams p;
};

// (A wait on a TMA full barrier needs no tcgen05 fence: the mbarrier
// already orders the async-proxy shared-memory writes before the MMAs that
// read them.  tcgen05.fence::after_thread_sync is only issued where TMEM
// written or read by another thread is reused.)
// Bounded mbarrier wait shared by all roles; gives up on the time budget
// or when another role has already given up.  `cluster`: the phase is
// completed by arrivals from the peer CTA (acquire at cluster scope).
__device__ __forceinline__ bool pf_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                        unsigned long long budget, unsigned* status,
                                        bool cluster = false) {
  auto test = [&]() { return cluster ? tc::test_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (test()) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (!test()) {
    if (((++n) & 63) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > budget) {
        *abort = 1;
        atomicOr(status, kStatusTimeout);
        return false;
      }
    }
  }
  return true;
}

template <typename T>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_kernel(const __grid_constant__ PfArgs args) {
  using E = Elem<T>;
  const PrefillParams& p = args.p;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte aligned base (128-byte swizzle atoms)
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  PfShared* sh = reinterpret_cast<PfShared*>(smem + kBarBase);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = p.hidden_dim, H = p.heads, ntok = p.T;
  const int nk = h / kBK;
  const int ntiles = (ntok + kBM - 1) / kBM;
  volatile int* abort = &sh->abort;
  const unsigned long long budget = p.budget_ns;

  auto bar = [&](uint64_t* b) { return smem_u32(b); };
  // the leader's (cluster rank 0) copy of a barrier, as a cluster address
  auto lead = [&](uint64_t* b) { return tc::mapa(smem_u32(b), 0); };

  if (threadIdx.x == 0) {
    // full barriers: one arrival (the leader's expect_tx for both CTAs'
    // bytes); empty / tfull / a2_free / mma_done: one pair-commit arrival;
    // tempty / a2_ready: one arrival per epilogue warp of both CTAs
    for (int i = 0; i < kS0Stages; ++i) {
      mbar_init(bar(&sh->full0[i]), 1);
      mbar_init(bar(&sh->empty0[i]), 1);
    }
    for (int i = 0; i < kS1Stages; ++i) {
      mbar_init(bar(&sh->full1[i]), 1);
      mbar_init(bar(&sh->empty1[i]), 1);
    }
    for (int i = 0; i < kS2Stages; ++i) {
      mbar_init(bar(&sh->full2[i]), 1);
      mbar_init(bar(&sh->empty2[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(&sh->tfull[i]), 1);
      mbar_init(bar(&sh->tempty[i]), 4 * kCl);
    }
    mbar_init(bar(&sh->a2_ready), 4 * kCl);
    mbar_init(bar(&sh->a2_free), 1);
    mbar_init(bar(&sh->mma_done), 1);
    sh->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc2(smem_u32(&sh->tmem_base), 512);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&args.tm_x);
    tma_prefetch_desc(&args.tm_wa);
    tma_prefetch_desc(&args.tm_wa3);
    if (!p.latent) tma_prefetch_desc(&args.tm_wb3);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();  // both CTAs' barriers are initialised before any copy or commit reaches them
  tc::fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  const uint32_t crank = tc::cluster_rank();
  const bool leader = crank == 0;
  // Main CTAs [0, main_ctas) take tiles blockIdx.x + it * main_ctas.  With
  // kpe_split, the CTA pairs past them are k_pe workers: pair w runs only
  // pass (a) for the tile pairs w, w + nwp, ... (its two CTAs on the two
  // tiles of a pair), and the main CTAs skip pass (a).  Every CTA of a
  // cluster runs the same number of tiles (tiles past the end are
  // all-padding: TMA fills zeros and the epilogue stores nothing).
  const bool worker = p.kpe_split && (int)blockIdx.x >= p.main_ctas;
  const bool do_kpe = !p.kpe_split || worker;
  const bool do_main = !worker;
  const int nwp = ((int)gridDim.x - p.main_ctas) / kCl, wp = ((int)blockIdx.x - p.main_ctas) / kCl;
  const int npairs = (ntiles + kCl - 1) / kCl;
  const int iters = worker ? (wp < npairs ? (npairs - wp + nwp - 1) / nwp : 0)
                           : (ntiles + p.main_ctas - 1) / p.main_ctas;
  auto tile_of = [&](int it) {
    return worker ? kCl * (wp + it * nwp) + (int)crank : (int)blockIdx.x + it * p.main_ctas;
  };

  if (warp == 0) {
    // ============================================================ TMA producer
    // Each CTA loads its own token rows (A) and its half of every weight
    // tile (B) into its own shared memory; the bytes of both CTAs complete
    // on the leader's full barrier, whose expect_tx the leader posts.
    if (lane == 0) {
      uint32_t u0 = 0, u1 = 0, u2 = 0;  // uses of the k_pe / compressed_kv / kv_b rings
      int tiles_done = 0;
      bool ok = true;
      for (int it = 0; it < iters && ok; ++it, ++tiles_done) {
        const int m0 = tile_of(it) * kBM;
        // the rings of this tile overlap the previous tile's A2 area
        if (do_main && tiles_done > 0 && !pf_wait(bar(&sh->a2_free), (tiles_done - 1) & 1, abort, budget, p.status)) { ok = false; break; }
        // (a) k_pe pass
        for (int kc = 0; kc < nk && ok && do_kpe; ++kc, ++u0) {
          const int s = u0 % kS0Stages;
          if (!pf_wait(bar(&sh->empty0[s]), ((u0 / kS0Stages) & 1) ^ 1, abort, budget, p.status)) { ok = false; break; }
          const uint32_t st = sbase + kS0Base + s * kS0Bytes;
          const uint32_t fb = lead(&sh->full0[s]);
          if (leader) mbar_arrive_expect_tx(bar(&sh->full0[s]), kCl * kS0Bytes);
          tma_load_2d_pair(st, &args.tm_x, kc * kBK, m0, fb);
          tma_load_2d_pair(st + 16384, &args.tm_wa, kRank, kc * kBK, fb);
        }
        if (!ok) break;
        if (!do_main) continue;
        // (b) compressed_kv pass: its ring overlaps the k_pe ring, so it
        // starts once every k_pe stage of this tile has been released
        for (uint32_t u = (u0 > (uint32_t)kS0Stages ? u0 - kS0Stages : 0); u < u0 && ok; ++u)
          if (!pf_wait(bar(&sh->empty0[u % kS0Stages]), (u / kS0Stages) & 1, abort, budget, p.status)) ok = false;
        for (int kc = 0; kc < nk && ok; ++kc, ++u1) {
          const int s = u1 % kS1Stages;
          if (!pf_wait(bar(&sh->empty1[s]), ((u1 / kS1Stages) & 1) ^ 1, abort, budget, p.status)) { ok = false; break; }
          const uint32_t st = sbase + s * kS1Bytes;
          const uint32_t fb = lead(&sh->full1[s]);
          if (leader) mbar_arrive_expect_tx(bar(&sh->full1[s]), kCl * kS1Bytes);
          tma_load_2d_pair(st, &args.tm_x, kc * kBK, m0, fb);
          // this CTA's 128 columns of each N = 256 tile: groups 2r, 2r+1 and 4+2r, 5+2r
          tma_load_3d_pair(st + 16384, &args.tm_wa3, 0, kc * kBK, (int)crank * 2, fb);
          tma_load_3d_pair(st + 32768, &args.tm_wa3, 0, kc * kBK, 4 + (int)crank * 2, fb);
        }
        // (c) kv_b: per head, 8 K-chunks; this CTA's 128 of the head's 256 columns
        for (int j = 0; j < H && ok && !p.latent; ++j) {
          for (int kc = 0; kc < kRank / kBK; ++kc, ++u2) {
            const int s = u2 % kS2Stages;
            if (!pf_wait(bar(&sh->empty2[s]), ((u2 / kS2Stages) & 1) ^ 1, abort, budget, p.status)) { ok = false; break; }
            const uint32_t st = sbase + kS2Base + s * kS2Bytes;
            const uint32_t fb = lead(&sh->full2[s]);
            if (leader) mbar_arrive_expect_tx(bar(&sh->full2[s]), kCl * kS2Bytes);
            tma_load_3d_pair(st, &args.tm_wb3, 0, kc * kBK, j * 4 + (int)crank * 2, fb);
          }
        }
      }
      // drain: on the leader every issued copy of both CTAs has landed (the
      // leader's full barriers count them) before the pair may exit; bounded,
      // but neither cut short by an abort nor by a tiny spin budget
      if (leader) {
        for (uint32_t u = (u0 > (uint32_t)kS0Stages ? u0 - kS0Stages : 0); u < u0; ++u)
          mbar_wait_bounded(bar(&sh->full0[u % kS0Stages]), (u / kS0Stages) & 1, drain_budget(budget));
        for (uint32_t u = (u1 > (uint32_t)kS1Stages ? u1 - kS1Stages : 0); u < u1; ++u)
          mbar_wait_bounded(bar(&sh->full1[u % kS1Stages]), (u / kS1Stages) & 1, drain_budget(budget));
        for (uint32_t u = (u2 > (uint32_t)kS2Stages ? u2 - kS2Stages : 0); u < u2; ++u)
          mbar_wait_bounded(bar(&sh->full2[u % kS2Stages]), (u / kS2Stages) & 1, drain_budget(budget));
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer (leader only)
    if (lane == 0 && leader) {
      const bool bf = E::kBf16;
      const uint32_t id128 = tc::idesc_f16(bf, 256, 128, false, true);
      const uint32_t id256 = tc::idesc_f16(bf, 256, 256, false, true);
      // base descriptors at shared-memory offset 0 (the same offsets in both
      // CTAs): K-major A (SW128, SBO 1024) and MN-major B (SW128, LBO 8192
      // between 64-column groups)
      const uint64_t dA0 = tc::sdesc_sw128(sbase, 16, 1024);
      const uint64_t dB0 = tc::sdesc_sw128(sbase, 8192, 1024);
      uint32_t u0 = 0, u1 = 0, u2 = 0;
      uint32_t wcount[2] = {0, 0}, dcount[2] = {0, 0};
      int tiles_done = 0;
      bool ok = true;
      // TMEM buffer b is free once both CTAs' epilogues have drained it
      auto drain_buf = [&](int b) -> bool {
        while (dcount[b] < wcount[b]) {
          if (!pf_wait(bar(&sh->tempty[b]), dcount[b] & 1, abort, budget, p.status, true)) return false;
          ++dcount[b];
        }
        return true;
      };
      for (int it = 0; it < iters && ok; ++it, ++tiles_done) {
        // (a) k_pe into TMEM columns [0, 128): N = 128, each CTA holding the same
        // 64 k_pe columns, so columns 64..127 repeat 0..63 and are not read
        if (do_kpe) {
        if (!drain_buf(0)) { ok = false; break; }
        tc::fence_after_sync();
        for (int kc = 0; kc < nk; ++kc, ++u0) {
          const int s = u0 % kS0Stages;
          if (!pf_wait(bar(&sh->full0[s]), (u0 / kS0Stages) & 1, abort, budget, p.status)) { ok = false; break; }
          // descriptors advance by constant adds (address field in 16-byte units)
          const uint64_t ad = dA0 + (uint64_t)((kS0Base + s * kS0Bytes) >> 4);
          const uint64_t bd = dB0 + (uint64_t)((kS0Base + s * kS0Bytes + 16384) >> 4);
          tc::mma2_f16(tmem, ad, bd, id128, kc > 0);
          tc::mma2_f16(tmem, ad + 2, bd + 128, id128, true);
          tc::mma2_f16(tmem, ad + 4, bd + 256, id128, true);
          tc::mma2_f16(tmem, ad + 6, bd + 384, id128, true);
          tc::commit2_both(bar(&sh->empty0[s]));
        }
        if (!ok) break;
        tc::commit2_both(bar(&sh->tfull[0]));
        ++wcount[0];
        }
        if (!do_main) continue;
        // (b) compressed_kv into TMEM columns [0, 512): two N = 256 tiles per K step
        if (!drain_buf(0) || !drain_buf(1)) { ok = false; break; }
        tc::fence_after_sync();
        for (int kc = 0; kc < nk; ++kc, ++u1) {
          const int s = u1 % kS1Stages;
          if (!pf_wait(bar(&sh->full1[s]), (u1 / kS1Stages) & 1, abort, budget, p.status)) { ok = false; break; }
          const uint64_t ad = dA0 + (uint64_t)((s * kS1Bytes) >> 4);
          const uint64_t bd = dB0 + (uint64_t)((s * kS1Bytes + 16384) >> 4);
          const bool acc = kc > 0;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            tc::mma2_f16(tmem, ad + 2 * k, bd + 128 * k, id256, acc || k > 0);
            tc::mma2_f16(tmem + 256, ad + 2 * k, bd + (16384 >> 4) + 128 * k, id256, acc || k > 0);
          }
          tc::commit2_both(bar(&sh->empty1[s]));
        }
        if (!ok) break;
        tc::commit2_both(bar(&sh->tfull[0]));  // the epilogues drain both halves, then signal a2_ready
        // (c) kv_b, one head per N = 256 tile
        if (!pf_wait(bar(&sh->a2_ready), tiles_done & 1, abort, budget, p.status, true)) { ok = false; break; }
        tc::fence_after_sync();
        for (int j = 0; j < H && ok && !p.latent; ++j) {
          const int b = j & 1;
          if (j >= 2 && !drain_buf(b)) { ok = false; break; }
          tc::fence_after_sync();
          for (int kc = 0; kc < kRank / kBK; ++kc, ++u2) {
            const int s = u2 % kS2Stages;
            if (!pf_wait(bar(&sh->full2[s]), (u2 / kS2Stages) & 1, abort, budget, p.status)) { ok = false; break; }
            const uint64_t ad = dA0 + (uint64_t)((kc * 16384) >> 4);
            const uint64_t bd = dB0 + (uint64_t)((kS2Base + s * kS2Bytes) >> 4);
            const uint32_t d = tmem + b * 256;
            tc::mma2_f16(d, ad, bd, id256, kc > 0);
            tc::mma2_f16(d, ad + 2, bd + 128, id256, true);
            tc::mma2_f16(d, ad + 4, bd + 256, id256, true);
            tc::mma2_f16(d, ad + 6, bd + 384, id256, true);
            tc::commit2_both(bar(&sh->empty2[s]));
          }
          if (!ok) break;
          tc::commit2_both(bar(&sh->tfull[b]));
          ++wcount[b];
        }
        if (!ok) break;
        tc::commit2_both(bar(&sh->a2_free));
      }
      // every MMA issued so far has completed (in both CTAs) before TMEM is released
      tc::commit2_both(bar(&sh->mma_done));
      mbar_wait_bounded(bar(&sh->mma_done), 0, drain_budget(budget));
    } else if (lane == 0) {
      // the peer CTA releases its tensor memory only after the pair's last MMA
      mbar_wait_bounded(bar(&sh->mma_done), 0, drain_budget(budget));
    }
  } else {
    // ============================================================ epilogue
    const int q = warp & 3;                // TMEM lane quadrant
    const int r = q * 32 + lane;           // row within the tile
    const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
    // gamma -> shared memory once (read by every row of every tile)
    const T* gam = reinterpret_cast<const T*>(smem + kGamBase);
    {
      const int e = threadIdx.x - 64;  // 0..127
      reinterpret_cast<uint2*>(smem + kGamBase)[e] = reinterpret_cast<const uint2*>(p.gamma)[e];
      asm volatile("bar.sync 1, 128;" ::: "memory");
    }
    uint32_t uf[2] = {0, 0};
    int tiles_done = 0;
    bool ok = true;
    for (int it = 0; it < iters && ok; ++it, ++tiles_done) {
      const int t = tile_of(it) * kBM + r;
      // output place of this row (dense [b, X, s, d] or a paged cache slot)
      int ou = 0, in = 0, cnt = 1;
      const bool live = t < ntok && out_place(p.out, t, p.s, p.status, &ou, &in, &cnt);
      // (a) k_pe: RoPE on the 64 raw columns
      if (do_kpe) {
      if (!pf_wait(bar(&sh->tfull[0]), uf[0] & 1, abort, budget, p.status)) { ok = false; break; }
      ++uf[0];
      tc::fence_after_sync();
      {
        uint32_t x[64];
        tc::ld32(lane_addr + 0, x);
        tc::ld32(lane_addr + 32, x + 32);
        tc::wait_ld();
        if (live) {
          int pos = p.positions[t];
          if (pos < 0 || pos >= p.max_pos) {
            atomicOr(p.status, kStatusBadPosition);
            pos = pos < 0 ? 0 : p.max_pos - 1;
          }
          float cr[kRope], sr[kRope];
          {
            const float4* c4 = reinterpret_cast<const float4*>(p.cos_t + (size_t)pos * kRope);
            const float4* s4 = reinterpret_cast<const float4*>(p.sin_t + (size_t)pos * kRope);
#pragma unroll
            for (int v = 0; v < kRope / 4; ++v) {
              const float4 a = __ldg(c4 + v), b = __ldg(s4 + v);
              cr[4 * v] = a.x; cr[4 * v + 1] = a.y; cr[4 * v + 2] = a.z; cr[4 * v + 3] = a.w;
              sr[4 * v] = b.x; sr[4 * v + 1] = b.y; sr[4 * v + 2] = b.z; sr[4 * v + 3] = b.w;
            }
          }
          uint32_t o[32];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float a0 = __uint_as_float(x[2 * j]), b0 = __uint_as_float(x[2 * j + 1]);
            const float a1 = __uint_as_float(x[2 * j + 2]), b1 = __uint_as_float(x[2 * j + 3]);
            o[j / 2] = E::pack(a0 * cr[j] - b0 * sr[j], a1 * cr[j + 1] - b1 * sr[j + 1]);
            o[16 + j / 2] = E::pack(b0 * cr[j + 32] + a0 * sr[j + 32], b1 * cr[j + 33] + a1 * sr[j + 33]);
          }
          if (p.c8.k) {  // int8 KV cache: o[k] holds outputs 2k, 2k + 1
            uint32_t w[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const T* e0 = reinterpret_cast<const T*>(&o[2 * k]);
              const T* e1 = reinterpret_cast<const T*>(&o[2 * k + 1]);
              const float4 iv = reinterpret_cast<const float4*>(p.c8.inv + 2 * H * kNope)[k];
              w[k] = kv_code(E::to_f(e0[0]), iv.x) | (kv_code(E::to_f(e0[1]), iv.y) << 8) |
                     (kv_code(E::to_f(e1[0]), iv.z) << 16) | (kv_code(E::to_f(e1[1]), iv.w) << 24);
            }
            uint4* dst = reinterpret_cast<uint4*>(static_cast<int8_t*>(p.k_pe) + ((size_t)ou * cnt + in) * kRope);
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.k_pe) + ((size_t)ou * cnt + in) * kRope);
#pragma unroll
            for (int v = 0; v < 8; ++v) dst[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
          }
        }
      }
      // release TMEM buffer 0 to the leader's MMA thread (one arrival per warp)
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::arrive_cluster_relaxed(lead(&sh->tempty[0]));
      }
      if (!do_main) continue;
      // (b) RMSNorm of compressed_kv -> normalised A tile in shared memory
      if (!pf_wait(bar(&sh->tfull[0]), uf[0] & 1, abort, budget, p.status)) { ok = false; break; }
      ++uf[0];
      tc::fence_after_sync();
      {
        float ss = 0.f;
        for (int c = 0; c < kRank / 32; ++c) {
          uint32_t x[32];
          tc::ld32(lane_addr + c * 32, x);
          tc::wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float v = __uint_as_float(x[j]);
            ss += v * v;
          }
        }
        const float inv = 1.0f / sqrtf(ss / (float)kRank + p.eps);
        unsigned char* a2row = smem + r * 128;
        for (int c = 0; c < kRank / 32; ++c) {
          uint32_t x[32];
          tc::ld32(lane_addr + c * 32, x);
          tc::wait_ld();
          uint32_t o[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const int col = c * 32 + j;
            o[j / 2] = E::pack(__uint_as_float(x[j]) * inv * E::to_f(gam[col]),
                               __uint_as_float(x[j + 1]) * inv * E::to_f(gam[col + 1]));
          }
          if (p.latent) {  // latent-cache variant: the normalised row is an output
            if (live) {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.latent) + (size_t)t * kRank + c * 32);
#pragma unroll
              for (int v = 0; v < 4; ++v) dst[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
            }
            continue;
          }
          // K-chunk c/2 (64 columns), 16-byte chunks (c%2)*4 .. +3 of this row
          unsigned char* chunk = a2row + (c >> 1) * 16384;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int lc = (c & 1) * 4 + v;
            *reinterpret_cast<uint4*>(chunk + ((lc ^ (r & 7)) << 4)) =
                make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
          }
        }
      }
      // the leader's kv_b MMAs read this CTA's A2 rows through the async proxy
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::arrive_cluster(lead(&sh->a2_ready));
      if (p.latent) continue;
      // (c) per head: split into k_nope / value, head-major stores.  On the
      // CTA's last tile the rows are staged through [kStageBase, +16 KB),
      // which no copy touches any more once the compressed_kv stages are
      // consumed (on earlier tiles the next tile's stages land there).
      T* kn = static_cast<T*>(p.k_nope);
      T* vv = static_cast<T*>(p.value);
      const bool staged = it == iters - 1 && !p.c8.k;
      for (int j = 0; j < H; ++j) {
        const int b = j & 1;
        if (!pf_wait(bar(&sh->tfull[b]), uf[b] & 1, abort, budget, p.status)) { ok = false; break; }
        ++uf[b];
        tc::fence_after_sync();
        const size_t orow = (((size_t)ou * H + j) * cnt + in) * kNope;
#pragma unroll 1
        for (int c = 0; c < kHeadCols / 32; c += 2) {  // two TMEM loads in flight
          uint32_t x[2][32];
          tc::ld32(lane_addr + b * 256 + c * 32, x[0]);
          tc::ld32(lane_addr + b * 256 + (c + 1) * 32, x[1]);
          tc::wait_ld();
          if (staged) {
            // the warp's 32 rows x 64 columns (128 B each) go through shared
            // memory (16-byte slots swizzled by row), then out as 128-byte
            // row segments, four rows per store instruction
            unsigned char* stg = smem + kStageBase + (warp & 3) * kStageWarp;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const int sl = h2 * 4 + v;
                *reinterpret_cast<uint4*>(stg + lane * 128 + ((sl ^ (lane & 7)) << 4)) = make_uint4(
                    E::pack(__uint_as_float(x[h2][8 * v + 0]), __uint_as_float(x[h2][8 * v + 1])),
                    E::pack(__uint_as_float(x[h2][8 * v + 2]), __uint_as_float(x[h2][8 * v + 3])),
                    E::pack(__uint_as_float(x[h2][8 * v + 4]), __uint_as_float(x[h2][8 * v + 5])),
                    E::pack(__uint_as_float(x[h2][8 * v + 6]), __uint_as_float(x[h2][8 * v + 7])));
              }
            __syncwarp();
            T* half = (c < 4 ? kn : vv) + (c & 3) * 32;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int rr = 4 * k + (lane >> 3), sl = lane & 7;
              const unsigned long long orow_r = __shfl_sync(0xffffffffu, (unsigned long long)orow, rr);
              const int live_r = __shfl_sync(0xffffffffu, live ? 1 : 0, rr);
              const uint4 val = *reinterpret_cast<const uint4*>(stg + rr * 128 + ((sl ^ (rr & 7)) << 4));
              if (live_r) *reinterpret_cast<uint4*>(half + orow_r + sl * 8) = val;
            }
            __syncwarp();  // the slots are rewritten by the next column pair
            continue;
          }
          if (live) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              uint32_t o[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] = E::pack(__uint_as_float(x[h2][2 * i]), __uint_as_float(x[h2][2 * i + 1]));
              const int cc = c + h2;
              if (p.c8.k) {  // int8 KV cache: codes of the 32 dtype values
                const float4* iv4 = reinterpret_cast<const float4*>(p.c8.inv + (cc < 4 ? 0 : H * kNope) +
                                                                    j * kNope + (cc & 3) * 32);
                uint32_t w[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  const T* e0 = reinterpret_cast<const T*>(&o[2 * k]);
                  const T* e1 = reinterpret_cast<const T*>(&o[2 * k + 1]);
                  const float4 iv = iv4[k];
                  w[k] = kv_code(E::to_f(e0[0]), iv.x) | (kv_code(E::to_f(e0[1]), iv.y) << 8) |
                         (kv_code(E::to_f(e1[0]), iv.z) << 16) | (kv_code(E::to_f(e1[1]), iv.w) << 24);
                }
                uint4* d4 = reinterpret_cast<uint4*>(reinterpret_cast<int8_t*>(cc < 4 ? p.k_nope : p.value) + orow +
                                                     (cc & 3) * 32);
                d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
                d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
              } else {
                T* dst = (cc < 4 ? kn : vv) + orow + (cc & 3) * 32;
                uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
                for (int v = 0; v < 4; ++v) d4[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
              }
            }
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::arrive_cluster_relaxed(lead(&sh->tempty[b]));
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  // neither CTA leaves, or releases the pair's tensor memory, while its peer
  // may still copy into it, read it, or arrive on its barriers
  tc::cluster_sync();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc2(tmem, 512);
  }
}

}  // namespace

// AUTO's switch from the decode kernel to the prefill kernel.  Measured on a
// GB300 (CUDA events per call, L2 flushed, T = 128 .. 4096):
//   - the decode kernel costs one launch per tt rows (128 for V2-Lite shapes,
//     64 for R1 shapes), about 14 us + weight bytes / 1.9 TB/s each
//     (V2-Lite 18.5 us, R1 36 us);
//   - the prefill kernel gives each CTA of a pair one 128-row tile over all
//     columns, so until every SM has a tile a call costs one tile pair's
//     FLOPs at about 22 TFLOP/s (V2-Lite 83 us, R1 475 us), whatever T is.
// The switch is the first T past the largest whole number of decode
// launches that still costs less than one prefill call: V2-Lite 513 (4 x
// 18.5 < 83 < 5 x 18.5), R1 833 (13 x 36 < 475 < 14 x 36).
int prefill_min_tokens(int hidden, int heads, int num_sms) {
  DecodePlan plan;
  if (!decode_plan(hidden, heads, num_sms, &plan)) return 1;
  const double flops_per_row = 2.0 * ((double)hidden * kNa + (double)kRank * heads * kHeadCols);
  const double weight_bytes = 2.0 * ((double)hidden * kNa + (double)kRank * heads * kHeadCols);
  const double prefill_us = 2.0 * kBM * flops_per_row / 22.0e6;
  const double decode_us = 14.0 + weight_bytes / 1.9e6;
  int launches = (int)(prefill_us / decode_us);
  if (launches < 1) launches = 1;
  return launches * plan.tt_max + 1;
}

cudaError_t prefill_launch(bool bf16, const PrefillParams& p, int num_sms, cudaStream_t stream,
                           int* launches) {
  *launches = 0;
  if (p.hidden_dim % kBK != 0 || p.T <= 0) return cudaErrorNotSupported;
  PfArgs a;
  a.p = p;
  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t h = (uint64_t)p.hidden_dim, NB = (uint64_t)p.heads * kHeadCols;
  if (!encode_tmap_2d(&a.tm_x, dt, p.hidden, h, (uint64_t)p.T, h * 2, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&a.tm_wa, dt, p.W_kva, kNa, h, kNa * 2, kBK, kBK, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_3d_colblocks(&a.tm_wa3, dt, p.W_kva, kNa, h, kNa * 2, kBK, kBK, 2, 2, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // (the latent-cache variant reads no W_kvb)
  if (p.latent) {
    a.tm_wb3 = a.tm_wa3;
  } else if (!encode_tmap_3d_colblocks(&a.tm_wb3, dt, p.W_kvb, NB, kRank, NB * 2, kBK, kBK, 2, 2,
                                       CU_TENSOR_MAP_SWIZZLE_128B)) {
    return cudaErrorInvalidValue;
  }
  const void* fn = bf16 ? (const void*)prefill_kernel<__nv_bfloat16> : (const void*)prefill_kernel<__half>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kPfThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // CTA pairs that fit on the GPU at once (two per cluster, one CTA per SM)
  static int max_clusters[2] = {0, 0};
  int& mc = max_clusters[bf16 ? 1 : 0];
  if (mc == 0) {
    cfg.gridDim = dim3(num_sms / kCl * kCl);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = num_sms / kCl;
    }
    mc = n;
  }
  const int ntiles = (p.T + kBM - 1) / kBM;
  const int max_grid = mc * kCl;
  int grid = (ntiles + kCl - 1) / kCl * kCl;
  if (grid > max_grid) grid = max_grid;
  // Pairs left over when every tile has its own CTA take the k_pe pass of
  // all tiles (it re-reads the hidden tile, so the main CTAs save one full
  // read of their rows): used when they are at least one per eight tiles,
  // and not for the latent-cache variant, whose tile CTAs (no kv_b pass)
  // would then wait for the workers.
  const int spare = max_grid - grid;
  a.p.main_ctas = grid;
  a.p.kpe_split = 0;
  if (!p.latent && grid >= ntiles && spare >= kCl && spare * 8 >= ntiles) {
    const int workers = (spare < grid ? spare : grid) / kCl * kCl;
    a.p.kpe_split = 1;
    grid += workers;
  }
  cfg.gridDim = dim3(grid);
  void* kargs[] = {&a};
  e = cudaLaunchKernelExC(&cfg, fn, kargs);
  if (e == cudaSuccess) *launches = 1;
  return e;
}

}  // namespace mla
