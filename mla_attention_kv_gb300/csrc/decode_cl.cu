// decode_cl.cu -- MLA KV prolog for the smallest decode launches without a
// grid-wide barrier.
//
// The seven prolog steps of "DeepSeek-V2-Lite-Chat MLA KV Prolog 迁移指南"
// §背景 for up to kClMaxTokens token rows, on the packed weight snapshot.
// RMSNorm (step 3) needs the whole 512-wide compressed_kv row, so the split-K
// kv_a_proj (step 1) has to be summed before anything after it can start.
// The grid-barrier decode kernel (decode.cu) sums it through L2 behind a
// grid-wide barrier; here each cluster of 16 CTAs computes the whole kv_a
// block of the launch's rows itself and sums it in distributed shared
// memory, so the only waits are on mbarriers of the CTA's own shared memory:
//
//   start    CTA r of a cluster copies K rows [128 r, 128 r + 128) of W_kva
//            (all 576 columns, 147 KB) and its column slice of W_kvb, both
//            from the packed snapshot and before the dependency wait; then
//            the same K columns of the hidden rows (TMA), gamma and the
//            positions.
//   phase A  kv_a partial sums [T, 576] over its 128 K rows (mma.sync
//            m16n8k16, fp32 accumulate; the tokens are the N side for T <= 8,
//            the M side above).
//   round 1  reduce-scatter: CTA r owns latent columns [32 r, 32 r + 32) and
//            raw k_pe columns [512 + 4 r, 512 + 4 r + 4); every CTA sends each
//            owner its [T, 36] partial block with one bulk copy into the
//            owner's shared memory, counted on the owner's mbarrier.
//   phase R  the owner sums the 16 blocks in rank order (split, step 2),
//            takes the sums of squares of its 32 latent columns, and (first
//            cluster only) rotates its k_pe columns (RoPE, step 6).
//   round 2  all-gather: each owner sends its summed [T, 32] block and the
//            T partial sums of squares to every CTA of the cluster.
//   phase B  every CTA normalises all T rows (RMSNorm in fp32, step 3,
//            rounded once to the I/O dtype) and multiplies them by its
//            W_kvb column slice (kv_b_proj, step 4); the epilogue writes the
//            head-major k_nope / value columns (steps 5 and 7).
// The kv_b columns are split over all CTAs of all clusters; every cluster
// computes the same kv_a block (W_kva is read from DRAM once and from L2
// once per cluster).
//
// Two cluster barriers, neither on the critical path: one after the
// mbarriers are initialised (peers signal them), waited for while the
// phase-A operands are landing; and one at exit, so that no CTA leaves while
// a copy into or out of its shared memory is in flight.  Every mbarrier wait is
// bounded; a CTA whose inputs time out still sends its blocks (the outputs
// are then undefined and the status word says so), so every CTA reaches the
// exit barrier in bounded time.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tma.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kKr = kClHidden / kClSize;   // 128 kv_a K rows per CTA
constexpr int kOwnL = kRank / kClSize;     // 32 latent columns owned per CTA
constexpr int kOwnR = kRope / kClSize;     // 4 raw k_pe columns owned per CTA
constexpr int kOwn = kOwnL + kOwnR;        // 36
constexpr int kGroupsA = kNa / 8;          // 72 n8 column groups of kv_a
constexpr int kGpw = kGroupsA / 8;         // 9 per warp
constexpr int kMtN = (kNa / 16 + 7) / 8;   // 5: most 16-column m-tiles per warp (tokens as N)
constexpr int kKs = kKr / 16;              // 8 k16 steps of phase A
constexpr int kXBox = 64;                  // hidden columns per TMA box (128 bytes)
constexpr int kXBoxes = kKr / kXBox;       // 2
constexpr int kMaxNg = 8;                  // most W_kvb groups per CTA (register tile)

// Shared memory (bytes from the 1024-aligned base).  The W_kva slice is
// dead once phase A is done; rounds 1-2 and phase B reuse it.
constexpr int kOffWa = 0;                                    // [18][128 rows][64 B] packed tiles
constexpr int kWaBytes = kKr * kNa * 2;                      // 147456
constexpr int kOffX = kOffWa + kWaBytes;                     // [2 boxes][16 rows][128 B] (swizzled)
constexpr int kXBytes = kXBoxes * 16 * 128;
constexpr int kOffR1 = kOffX + kXBytes;                      // round-1 receive: [16 senders][T][36] f32
constexpr int kR1Bytes = kClSize * kClMaxTokens * kOwn * 4;
constexpr int kOffWb = kOffR1 + kR1Bytes;                    // W_kvb slice [512][ng 16-byte chunks]
// inside the W_kva area, after phase A
constexpr int kOffS1 = 0;                                    // round-1 send: [16 owners][T][36] f32
constexpr int kOffR2 = kOffS1 + kR1Bytes;                    // round-2 receive: [16 owners][S2] f32
constexpr int kS2Max = kClMaxTokens * kOwnL + kClMaxTokens;  // floats per owner block
constexpr int kOffS2 = kOffR2 + kClSize * kS2Max * 4;        // round-2 send: [S2] f32
constexpr int kOffRope = kOffS2 + kS2Max * 4;                // summed raw k_pe columns [T][4] f32
constexpr int kOffN = kOffRope + kClMaxTokens * kOwnR * 4;   // normalised rows [16][kNrmPitch]
constexpr int kOffRed = kOffN + 16 * kNrmPitch;              // phase-B k-slice sums [8 warps][kMaxNg][32][4] f32
static_assert(kOffRed + 8 * kMaxNg * 32 * 16 <= kWaBytes, "phase-B scratch exceeds the W_kva area");
static_assert(kOffX % 1024 == 0, "the swizzled hidden boxes need 1024-byte alignment");
// misc block (at plan.off_misc): mbarriers, cos/sin of the k_pe columns, flags, gamma
constexpr int kMiscBytes = 2048;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_addr(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
// (relaxed: the barriers order no data -- the data travels by bulk copies
// counted on mbarriers, and the mbarrier initialisation is released by
// fence.mbarrier_init)
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Bulk copy from this CTA's shared memory into a peer's (dst and bar are
// cluster addresses of the peer); completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_s2peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "r"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Owner of kv_a column c (0 .. 575) and its index in the owner's 36-wide block.
__device__ __forceinline__ int own_rank(int c) { return c < kRank ? c / kOwnL : (c - kRank) / kOwnR; }
__device__ __forceinline__ int own_index(int c) { return c < kRank ? c % kOwnL : kOwnL + (c - kRank) % kOwnR; }

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) decode_cl_kernel(const __grid_constant__ ClParams p) {
  using E = Elem<T>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = (int)cluster_rank();
  const bool first_cluster = blockIdx.x < kClSize;
  const int TT = p.TT;
  const int NG = p.heads * kHeadCols / 8;
  const int G = gridDim.x, cta = blockIdx.x;
  const int g0 = (int)(((long long)cta * NG) / G), ng = (int)(((long long)(cta + 1) * NG) / G) - g0;
  const int S1 = TT * kOwn;                      // floats per round-1 block
  const int S2 = TT * kOwnL + ((TT + 3) & ~3);   // floats per round-2 block (sums of squares at TT * 32)

  unsigned char* misc = smem + p.off_misc;
  const uint32_t bar_wa = smem_u32(misc), bar_x = bar_wa + 8, bar_wb = bar_wa + 16;
  const uint32_t bar_r1 = bar_wa + 24, bar_r2 = bar_wa + 32;
  float* sCS = reinterpret_cast<float*>(misc + 128);            // [16][8]: cos j0, j0+1, j0+32, j0+33, then sin
  volatile int* sFlag = reinterpret_cast<volatile int*>(misc + 704);
  T* sGam = reinterpret_cast<T*>(misc + 1024);                  // [512]
  const uint32_t sWa = smem_u32(smem + kOffWa), sX = smem_u32(smem + kOffX), sWb = smem_u32(smem + kOffWb);
  float* sR1 = reinterpret_cast<float*>(smem + kOffR1);
  float* sS1 = reinterpret_cast<float*>(smem + kOffS1);
  float* sR2 = reinterpret_cast<float*>(smem + kOffR2);
  float* sS2 = reinterpret_cast<float*>(smem + kOffS2);
  float* sRope = reinterpret_cast<float*>(smem + kOffRope);
  unsigned char* sN = smem + kOffN;
  float* sRed = reinterpret_cast<float*>(smem + kOffRed);

  // ---- barriers; the receive barriers expect every peer's block
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(bar_wa + 8 * i, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar_r1, (uint32_t)(kClSize * S1 * 4));
    mbar_arrive_expect_tx(bar_r2, (uint32_t)(kClSize * S2 * 4));
  }
  __syncthreads();
  cluster_arrive();  // peers may signal this CTA's barriers once they have waited for this

  // ---- W_kva rows [128 r, 128 r + 128): in the packed snapshot, 18 tiles of
  // 128 rows x 64 bytes inside the units (kc, nb) of KB rows (read-only, so
  // copied before the dependency wait)
  const unsigned char* Wpk = static_cast<const unsigned char*>(p.W_kva);
  // W_kvb: this CTA's column groups [g0, g0 + ng) are one contiguous block of
  // 512 rows x ng 16-byte chunks, chunk j of row k stored at j ^ pack_swizzle(ng, k)
  const unsigned char* Wbpk = static_cast<const unsigned char*>(p.W_kvb) + (size_t)g0 * (kRank * 16);
  // Lanes 0..17 copy the W_kva tiles, each cluster starting at another tile
  // (the clusters all read the same W_kva lines); the next ng lanes copy the
  // W_kvb slice, queued behind W_kva on the CTA's copy engine (which the
  // bulk copies of the two exchange rounds use later on as well).
  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_wa, (uint32_t)kWaBytes);
      mbar_arrive_expect_tx(bar_wb, (uint32_t)(ng * kRank * 16));
    }
    __syncwarp();
    if (lane < kNa / 32) {
      const int nb = (lane + 5 * (int)(blockIdx.x / kClSize)) % (kNa / 32);
      const int krow = r * kKr, kc = krow / p.KB, rr = krow - kc * p.KB;
      bulk_g2s(sWa + nb * (kKr * 64), Wpk + (((size_t)kc * (kNa / 32) + nb) * p.KB + rr) * 64, kKr * 64, bar_wa);
    } else if (lane - kNa / 32 < ng) {
      const int j = lane - kNa / 32;
      bulk_g2s(sWb + j * (kRank * 16), Wbpk + (size_t)j * (kRank * 16), kRank * 16, bar_wb);
    }
  }
  grid_dep_launch_dependents();
  grid_dep_wait();
  // ---- after the dependency wait: hidden columns of this CTA's K rows,
  // gamma, and the positions' cos/sin values of the k_pe columns
  if (warp == 1 && lane == 0) {
    mbar_arrive_expect_tx(bar_x, (uint32_t)(kXBoxes * p.xrows * 128));
    for (int b = 0; b < kXBoxes; ++b) tma_load_2d(sX + b * 2048, &p.tmap_x, r * kKr + b * kXBox, p.t0, bar_x);
  }
  if (tid >= 64 && tid < 128) cp_async16(smem_u32(sGam) + (tid - 64) * 16, static_cast<const T*>(p.gamma) + (tid - 64) * 8);
  cp_async_commit();
  if (warp == 4 && lane < TT) {
    int pp = p.positions[p.t0 + lane];
    if (pp < 0 || pp >= p.max_pos) {
      atomicOr(p.status, kStatusBadPosition);
      pp = pp < 0 ? 0 : p.max_pos - 1;
    }
    if (first_cluster) {
      const int j0 = 2 * r;
      const float* c = p.cos_t + (size_t)pp * kRope;
      const float* s = p.sin_t + (size_t)pp * kRope;
      const float2 c0 = *reinterpret_cast<const float2*>(c + j0), c1 = *reinterpret_cast<const float2*>(c + j0 + 32);
      const float2 s0 = *reinterpret_cast<const float2*>(s + j0), s1 = *reinterpret_cast<const float2*>(s + j0 + 32);
      float* d = sCS + lane * 8;
      d[0] = c0.x; d[1] = c0.y; d[2] = c1.x; d[3] = c1.y;
      d[4] = s0.x; d[5] = s0.y; d[6] = s1.x; d[7] = s1.y;
    }
  }
  cluster_wait();  // every peer's barriers are initialised (the operands land meanwhile)

  // ================================================================ phase A
  if (tid == 0)
    sFlag[0] = (mbar_wait_bounded(bar_wa, 0, p.budget_ns) && mbar_wait_bounded(bar_x, 0, p.budget_ns)) ? 1 : 0;
  __syncthreads();
  bool good = sFlag[0] != 0;  // every input of this CTA arrived (the same in every thread)
  if (good) {
    while (!mbar_test_wait(bar_wa, 0)) {
    }
    while (!mbar_test_wait(bar_x, 0)) {
    }
  } else if (tid == 0) {
    atomicOr(p.status, kStatusTimeout);
  }
  // The partial block of owner q goes to sS1 + q * S1 as [TT][36].  Hidden
  // rows: 128-byte swizzle, chunk q of row t at q ^ (t & 7).  W_kva tiles:
  // 64-byte rows (32 columns), chunk c of row k at c ^ ((k >> 1) & 3).
  if (good && TT <= 8) {
    // tokens as the N side (n8): the 576 columns in 36 m-tiles of 16, warp w
    // takes tiles w, w + 8, ...; A = W_kva^T (ldmatrix.trans of the tiles),
    // B = the hidden rows (two k16 steps per ldmatrix.x4)
    float acc[kMtN][4];
#pragma unroll
    for (int i = 0; i < kMtN; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kKs; kk += 2) {
      uint32_t b[4];
      {
        const int n = lane & 7, q = (kk & 3) * 2 + (lane >> 3);
        ldsm_x4(sX + (kk >> 2) * 2048 + n * 128 + ((q ^ n) << 4), b[0], b[1], b[2], b[3]);
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int k = (kk + h2) * 16 + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
        for (int i = 0; i < kMtN; ++i) {
          const int mt = warp + 8 * i;
          if (mt < kNa / 16) {
            const int ch = ((mt & 1) << 1) + ((lane >> 3) & 1);
            uint32_t a[4];
            ldsm_x4_trans(sWa + (mt >> 1) * (kKr * 64) + k * 64 + ((ch ^ ((lane >> 1) & 3)) << 4), a[0], a[1],
                          a[2], a[3]);
            mma16816<E::kBf16>(acc[i], a, b[2 * h2], b[2 * h2 + 1]);
          }
        }
      }
    }
    __syncthreads();  // the W_kva area is free from here on
    // this thread holds columns m and m + 8 of tile mt for tokens n, n + 1
    const int n = 2 * (lane & 3);
#pragma unroll
    for (int i = 0; i < kMtN; ++i) {
      const int mt = warp + 8 * i;
      if (mt < kNa / 16) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int c = mt * 16 + (lane >> 2) + 8 * hh;
          float* d = sS1 + own_rank(c) * S1 + own_index(c);
          if (n < TT) d[n * kOwn] = acc[i][2 * hh];
          if (n + 1 < TT) d[(n + 1) * kOwn] = acc[i][2 * hh + 1];
        }
      }
    }
  } else if (good) {
    // tokens as the M side (16 rows): n8 group g = warp + 8 i of the 72
    float acc[kGpw][4];
#pragma unroll
    for (int i = 0; i < kGpw; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    uint32_t a[kKs][4];
#pragma unroll
    for (int kk = 0; kk < kKs; ++kk)
      ldsm_x4(sX + (kk >> 2) * 2048 + (lane & 15) * 128 + ((((kk & 3) * 2 + (lane >> 4)) ^ (lane & 7)) << 4),
              a[kk][0], a[kk][1], a[kk][2], a[kk][3]);
    // per k16 step, the fragments of all nine groups first (nine independent chains)
    uint32_t wb[kGpw];
#pragma unroll
    for (int i = 0; i < kGpw; ++i) {
      const int g = warp + 8 * i, nb = g >> 2, nb8 = g & 3;
      wb[i] = sWa + nb * (kKr * 64) + (lane & 15) * 64 + ((nb8 ^ ((lane >> 1) & 3)) << 4);
    }
#pragma unroll
    for (int kk = 0; kk < kKs; ++kk) {
      uint32_t b[kGpw][2];
#pragma unroll
      for (int i = 0; i < kGpw; ++i) ldsm_x2_trans(wb[i] + kk * 16 * 64, b[i][0], b[i][1]);
#pragma unroll
      for (int i = 0; i < kGpw; ++i) mma16816<E::kBf16>(acc[i], a[kk], b[i][0], b[i][1]);
    }
    __syncthreads();  // the W_kva area is free from here on
    const int t = lane >> 2;
#pragma unroll
    for (int i = 0; i < kGpw; ++i) {
      const int c = 8 * (warp + 8 * i) + 2 * (lane & 3);
      float* d = sS1 + own_rank(c) * S1 + own_index(c);
      if (t < TT) *reinterpret_cast<float2*>(d + t * kOwn) = make_float2(acc[i][0], acc[i][1]);
      if (t + 8 < TT) *reinterpret_cast<float2*>(d + (t + 8) * kOwn) = make_float2(acc[i][2], acc[i][3]);
    }
  } else {
    __syncthreads();  // (the barrier of the computing paths)
  }

  // ================================================================ round 1
  // one bulk copy per owner, issued by lane 0 of every warp (two each: the
  // copy instructions of one warp issue one after another)
  fence_async_smem();  // the bulk copies (async proxy) read what the threads wrote
  __syncthreads();
  if (lane == 0)
    for (int q = warp; q < kClSize; q += kThreads / 32)
      bulk_s2peer(cluster_addr(smem_u32(sR1) + r * S1 * 4, q), smem_u32(sS1) + q * S1 * 4, S1 * 4,
                  cluster_addr(bar_r1, q));

  // ================================================================ phase R
  if (tid == 0) sFlag[1] = mbar_wait_bounded(bar_r1, 0, p.budget_ns) ? 1 : 0;
  cp_async_wait<0>();  // gamma
  __syncthreads();
  const bool got1 = sFlag[1] != 0;
  if (got1) {
    while (!mbar_test_wait(bar_r1, 0)) {
    }
  } else if (tid == 0) {
    atomicOr(p.status, kStatusTimeout);
  }
  good = good && got1;
  // warp w: rows w, w + 8; lane l sums owned latent column l (lanes 0..3 also
  // k_pe column l) over the 16 blocks in rank order, then the row's sum of
  // squares over the 32 latent columns
  for (int t = warp; t < TT; t += 8) {
    float x[kClSize], y[kClSize];  // all loads first, then the sums
#pragma unroll
    for (int q = 0; q < kClSize; ++q) {
      x[q] = sR1[q * S1 + t * kOwn + lane];
      y[q] = lane < kOwnR ? sR1[q * S1 + t * kOwn + kOwnL + lane] : 0.f;
    }
    float v = 0.f, w = 0.f;
#pragma unroll
    for (int q = 0; q < kClSize; ++q) {
      v += x[q];
      w += y[q];
    }
    sS2[t * kOwnL + lane] = v;
    if (lane < kOwnR) sRope[t * kOwnR + lane] = w;
    float ss = v * v;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) sS2[TT * kOwnL + t] = ss;
  }

  // ================================================================ round 2
  fence_async_smem();
  __syncthreads();
  if (lane == 0)
    for (int q = warp; q < kClSize; q += kThreads / 32)
      bulk_s2peer(cluster_addr(smem_u32(sR2) + r * S2 * 4, q), smem_u32(sS2), S2 * 4, cluster_addr(bar_r2, q));
  // k_pe (first cluster): raw columns 512 + 4 r .. 512 + 4 r + 3 of row t are
  // the de-interleaved pairs (2 r, 2 r + 32) and (2 r + 1, 2 r + 33), rotated
  if (first_cluster && good && warp == 1 && lane < TT) {
    const int t = lane, j0 = 2 * r;
    const float* v = sRope + t * kOwnR;
    const float* cs = sCS + t * 8;
    int ou, in, cnt;
    if (out_place(p.out, p.t0 + t, p.s, p.status, &ou, &in, &cnt)) {
      T* kp = static_cast<T*>(p.k_pe) + ((size_t)ou * cnt + in) * kRope;
      *reinterpret_cast<uint32_t*>(kp + j0) = E::pack(v[0] * cs[0] - v[1] * cs[4], v[2] * cs[1] - v[3] * cs[5]);
      *reinterpret_cast<uint32_t*>(kp + j0 + 32) =
          E::pack(v[1] * cs[2] + v[0] * cs[6], v[3] * cs[3] + v[2] * cs[7]);
    }
  }
  if (tid == 0) {
    sFlag[2] = mbar_wait_bounded(bar_r2, 0, p.budget_ns) ? 1 : 0;
    if (!sFlag[2] || !got1) {
      // every CTA sends both rounds whatever happened to it: wait (bounded)
      // for the copies still in flight before this CTA arrives below
      atomicOr(p.status, kStatusTimeout);
      mbar_wait_bounded(bar_r1, 0, drain_budget(p.budget_ns));
      mbar_wait_bounded(bar_r2, 0, drain_budget(p.budget_ns));
    }
  }
  __syncthreads();
  const bool got2 = sFlag[2] != 0;
  if (got2) {
    while (!mbar_test_wait(bar_r2, 0)) {
    }
  }
  good = good && got2;
  // every copy into this CTA has landed (or was waited for): peers may leave
  // once all CTAs have arrived
  cluster_arrive();

  // ================================================================ phase B
  if (good) {
    if (tid < kRank / 4) {
      // thread c4 normalises columns 4 c4 .. 4 c4 + 3 of every row; lane t
      // of each warp takes the 1 / rms of row t (the 16 partial sums of
      // squares in rank order) and shares it by shuffles
      float inv = 0.f;
      if (lane < TT) {
        float z[kClSize];
#pragma unroll
        for (int q = 0; q < kClSize; ++q) z[q] = sR2[q * S2 + TT * kOwnL + lane];
        float ss = 0.f;
#pragma unroll
        for (int q = 0; q < kClSize; ++q) ss += z[q];
        inv = 1.0f / sqrtf(ss * (1.0f / (float)kRank) + p.eps);
      }
      const int c = tid * 4;
      const float ga = E::to_f(sGam[c]), gb = E::to_f(sGam[c + 1]), gc = E::to_f(sGam[c + 2]),
                  gd = E::to_f(sGam[c + 3]);
      const float* src = sR2 + (c / kOwnL) * S2 + (c % kOwnL);
      for (int t = 0; t < TT; ++t) {
        const float it = __shfl_sync(0xffffffffu, inv, t);
        const float4 v = *reinterpret_cast<const float4*>(src + t * kOwnL);
        *reinterpret_cast<uint2*>(sN + t * kNrmPitch + c * 2) =
            make_uint2(E::pack(v.x * it * ga, v.y * it * gb), E::pack(v.z * it * gc, v.w * it * gd));
      }
    } else {
      // rows TT .. 15 of the MMA operand are zero
      constexpr int kChunks = kRank * 2 / 16;
      for (int e = tid - kRank / 4; e < (16 - TT) * kChunks; e += kThreads - kRank / 4)
        *reinterpret_cast<uint4*>(sN + (TT + e / kChunks) * kNrmPitch + (e % kChunks) * 16) = make_uint4(0, 0, 0, 0);
    }
    if (tid == 0) sFlag[3] = mbar_wait_bounded(bar_wb, 0, p.budget_ns) ? 1 : 0;
    __syncthreads();
    if (sFlag[3] == 0) {
      if (tid == 0) atomicOr(p.status, kStatusTimeout);
      good = false;
    } else {
      while (!mbar_test_wait(bar_wb, 0)) {
      }
    }
  }
  if (good && ng > 0) {
    // kv_b: warp w takes k16 steps w, w + 8, w + 16, w + 24 of every group
    float bc[kMaxNg][4];
#pragma unroll
    for (int gi = 0; gi < kMaxNg; ++gi) bc[gi][0] = bc[gi][1] = bc[gi][2] = bc[gi][3] = 0.f;
    const uint32_t nrm_u = smem_u32(sN);
    const int pitchW = ng * 16;
    const int xm = pack_swizzle(ng, lane & 7);  // the rows a lane addresses are congruent to lane mod 8
#pragma unroll
    for (int s = 0; s < kRank / 16 / 8; ++s) {
      const int st = warp + 8 * s;
      uint32_t a[4];
      ldsm_x4(nrm_u + (lane & 15) * kNrmPitch + (st * 16 + (lane >> 4) * 8) * 2, a[0], a[1], a[2], a[3]);
      const uint32_t wrow = sWb + (st * 16 + (lane & 15)) * pitchW;
#pragma unroll
      for (int gi = 0; gi < kMaxNg; ++gi) {
        if (gi < ng) {
          uint32_t b0, b1;
          ldsm_x2_trans(wrow + ((gi ^ xm) << 4), b0, b1);
          mma16816<E::kBf16>(bc[gi], a, b0, b1);
        }
      }
    }
#pragma unroll
    for (int gi = 0; gi < kMaxNg; ++gi)
      if (gi < ng)
        *reinterpret_cast<float4*>(sRed + ((warp * kMaxNg + gi) * 32 + lane) * 4) =
            make_float4(bc[gi][0], bc[gi][1], bc[gi][2], bc[gi][3]);
    __syncthreads();
    // the 8 k-slices of each fragment summed in order, then stored: the pair of
    // columns of one fragment row lies inside one head's k_nope or value half
    // (steps 5 and 7)
    T* kn = static_cast<T*>(p.k_nope);
    T* vv = static_cast<T*>(p.value);
    for (int e = tid; e < ng * 32; e += kThreads) {
      const int gi = e >> 5, l = e & 31;
      float4 o[8];
#pragma unroll
      for (int w = 0; w < 8; ++w) o[w] = *reinterpret_cast<const float4*>(sRed + ((w * kMaxNg + gi) * 32 + l) * 4);
      float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        v[0] += o[w].x; v[1] += o[w].y; v[2] += o[w].z; v[3] += o[w].w;
      }
      const int j = (g0 + gi) * 8 + 2 * (l & 3);
      const int hh = j / kHeadCols, ec = j - hh * kHeadCols;
      T* base = ec < kNope ? kn : vv;
      const int ee = ec < kNope ? ec : ec - kNope;
#pragma unroll
      for (int h8 = 0; h8 < 2; ++h8) {
        const int t = (l >> 2) + 8 * h8;
        int ou, in, cnt;
        if (t < TT && out_place(p.out, p.t0 + t, p.s, p.status, &ou, &in, &cnt))
          *reinterpret_cast<uint32_t*>(base + (((size_t)ou * p.heads + hh) * cnt + in) * kNope + ee) =
              E::pack(v[2 * h8], v[2 * h8 + 1]);
      }
    }
  }
  // ---- exit: this CTA's own copies in flight (after a timeout) are waited
  // for, then every CTA of the cluster has received everything
  if (tid == 0) {
    mbar_wait_bounded(bar_wa, 0, drain_budget(p.budget_ns));
    mbar_wait_bounded(bar_x, 0, drain_budget(p.budget_ns));
    mbar_wait_bounded(bar_wb, 0, drain_budget(p.budget_ns));
  }
  cp_async_wait<0>();
  __syncthreads();
  cluster_wait();
}

template <typename T>
const void* cl_kernel() {
  return reinterpret_cast<const void*>(&decode_cl_kernel<T>);
}

}  // namespace

// The instance's attributes (shared-memory limit, 16-CTA clusters) are set
// once per device; the plan then asks the device how many such clusters it
// holds at once and sizes the launch to that.
static cudaError_t cl_prepare(const void* fn, size_t smem) {
  static std::mutex mu;
  static struct {
    const void* fn;
    int dev;
    size_t smem;
  } done[16];
  static int nd = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < nd; ++i)
    if (done[i].fn == fn && done[i].dev == dev && done[i].smem >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  int i = 0;
  while (i < nd && !(done[i].fn == fn && done[i].dev == dev)) ++i;
  if (i < nd) done[i].smem = smem;
  else if (nd < 16) done[nd++] = {fn, dev, smem};
  return cudaSuccess;
}

bool decode_cl_plan(bool bf16, int hidden, int heads, int KB, ClPlan* plan) {
  if (hidden != kClHidden || KB <= 0 || KB % kKr != 0 || heads < 1) return false;
  const void* fn = bf16 ? cl_kernel<__nv_bfloat16>() : cl_kernel<__half>();
  const int NG = heads * kHeadCols / 8;
  // the W_kvb slice width depends on the cluster count and the cluster count
  // on the shared memory: ask with the widest slice that fits, then check
  constexpr int kBudget = 227 * 1024;
  int ng_fit = (kBudget - 1024 - kMiscBytes - kOffWb) / (kRank * 16);
  if (ng_fit > kMaxNg) ng_fit = kMaxNg;
  if (ng_fit < 1) return false;
  const size_t smem = (size_t)kOffWb + (size_t)kRank * 16 * ng_fit + kMiscBytes + 1024;
  if (cl_prepare(fn, smem) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClSize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(kClSize);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (clusters < 1) return false;
  const int ctas = clusters * kClSize;
  const int ngmax = (NG + ctas - 1) / ctas;
  if (ngmax > ng_fit) return false;
  plan->clusters = clusters;
  plan->ngmax = ngmax;
  plan->off_misc = kOffWb + kRank * 16 * ngmax;
  plan->smem = (size_t)plan->off_misc + kMiscBytes + 1024;  // + base alignment slack
  return true;
}

cudaError_t decode_cl_launch(bool bf16, const ClPlan& plan, const ClParams& p0, bool pdl,
                             cudaStream_t stream) {
  if (p0.TT < 1 || p0.TT > kClMaxTokens || p0.off_misc != plan.off_misc)
    return cudaErrorInvalidValue;
  const void* fn = bf16 ? cl_kernel<__nv_bfloat16>() : cl_kernel<__half>();
  cudaError_t e = cl_prepare(fn, plan.smem);
  if (e != cudaSuccess) return e;
  ClParams p = p0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.clusters * kClSize);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClSize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  void* args[] = {&p};
  if (pdl) {
    cfg.numAttrs = 2;
    e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaErrorInvalidValue && e != cudaErrorNotSupported) return e;
    cudaGetLastError();
  }
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace mla
