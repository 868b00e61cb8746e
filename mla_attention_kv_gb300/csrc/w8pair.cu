// w8pair.cu -- the int8 GEMMs of the W8A8 prolog at prefill sizes, on the
// 2-SM tensor-core MMA (tcgen05.mma.cta_group::2, M = 256 token rows per CTA
// pair, N = 256 weight columns).
//
// "DeepSeek-R1或Kimi-K2模型在NPU实现高性能推理" §权重转换 (W8A8: int8 weights
// with per-output-channel scales, per-token int8 activations, exact int32
// accumulation).  The products run as fp16 x fp16 -> fp32 tensor-core MMAs
// on the fp16 values of the int8 codes (exact: |v| <= 127), and the
// accumulator restarts every kChunkKB K blocks (1024 K rows), so every
// partial sum is an integer of magnitude <= 1024 * 127^2 < 2^24, exact in
// fp32; the chunks are converted to int32 and added in tensor memory.
//
// At these sizes every weight byte feeds thousands of tokens, so the int8
// weights are first widened to fp16 copies in the workspace (one elementwise
// pass per call, at HBM speed), and both operands then reach shared memory
// through TMA with no conversion work in the GEMM: each CTA of a pair loads
// its own 128 token rows (A, K-major) and half of the tile's 256 weight
// columns (B, MN-major); the leader CTA issues the pair's MMAs.  This is the
// operand balance that keeps shared-memory traffic within its bandwidth
// (A 4 KB + B 4 KB per 128-cycle K16 step and CTA, plus the same again
// written by TMA).
//
// Warp roles (320 threads per CTA): warp 0 TMA producer; warp 1 TMEM
// allocation (512 columns, both CTAs) and, in the leader, the MMA issuer;
// warps 2-9 epilogue: one token row per thread, warps 2-5 on the tile's
// columns 0-127 and warps 6-9 on 128-255.  Tensor memory: the fp32
// chunk accumulator in columns [0, 256), the int32 sums in [256, 512).
// Output stages:
//   RAW    int32 sums stored into C [T, ldc] (q_a | kv_a accumulator rows)
//   HEADS  y = (float)acc * s_x[t] * s_w[n] -> q_b: q_nope, RoPE(q_pe);
//          kv_b: k_nope, value (head-major, row-contiguous 16-byte stores)
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tma.h"

namespace mla {
namespace {

constexpr int kPThreads = 320;
constexpr int kPEpiWarps = 8;             // two per TMEM lane quadrant, one per 128-column half
constexpr int kPCl = 2;
constexpr int kPBM = 128;                 // token rows per CTA
constexpr int kPBN = 256;                 // weight columns per pair tile
constexpr int kPBK = 64;
constexpr int kPChunkKB = 16;             // K blocks per exact fp32 chunk (1024 rows)
constexpr uint32_t kPStage = 32768;       // A 16 KB + this CTA's half of B 16 KB
constexpr int kPStages = 6;
constexpr uint32_t kPBarBase = kPStages * kPStage;  // 196608
constexpr uint32_t kPIntCol = 256;
// HEADS output staging: per epilogue warp its 32 token rows x 128 bytes
constexpr uint32_t kPStgBase = kPBarBase + 512;
constexpr uint32_t kPStgWarp = 32 * 128;
constexpr uint32_t kPSmem = kPStgBase + kPEpiWarps * kPStgWarp + 1024;  // + base alignment slack

struct PShared {
  uint64_t full[kPStages], empty[kPStages];
  uint64_t tfull, tempty;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(PShared) <= 512, "barrier block");

struct PArgs {
  CUtensorMap tx[2];   // activations fp16 [T, K_i], box {64, 128}, SW128
  CUtensorMap tw[2];   // fp16 weights as [K_i][N_i / 64][64], box {64, 64, 2}, SW128
  W8PairParams p;
};

__device__ __forceinline__ bool pw_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                        unsigned long long budget, unsigned* status,
                                        bool cluster = false) {
  auto test = [&]() { return cluster ? tc::test_wait_cluster(bar, parity) : mbar_try_wait_hint(bar, parity, 20000); };
  if (test()) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!test()) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > budget) {
      *abort = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
  return true;
}

struct PTile {
  int sel, mt, nt;
};
__device__ __forceinline__ PTile ptile_of(const W8PairParams& p, int u) {
  PTile r;
  r.sel = u < p.ntiles[0] ? 0 : 1;
  const int v = u - (r.sel ? p.ntiles[0] : 0);
  // mfast: token tiles fastest (the pairs running at the same time share a
  // weight panel, which is then read from DRAM once; for activations smaller
  // than the weights), otherwise weight tiles fastest (they share token rows)
  if (p.mfast[r.sel]) {
    const int nm = p.nm;
    r.mt = v % nm;
    r.nt = v / nm;
  } else {
    const int nn = p.nn[r.sel];
    r.nt = v % nn;
    r.mt = v / nn;
  }
  return r;
}

template <int MODE>
__global__ void __launch_bounds__(kPThreads, 1) w8pair_kernel(const __grid_constant__ PArgs args) {
  const W8PairParams& p = args.p;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  PShared* sh = reinterpret_cast<PShared*>(smem + kPBarBase);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &sh->abort;
  const unsigned long long budget = p.budget_ns;
  auto bar = [&](uint64_t* b) { return smem_u32(b); };
  auto lead = [&](uint64_t* b) { return tc::mapa(smem_u32(b), 0); };
  const int npairs = gridDim.x / kPCl, pair = blockIdx.x / kPCl;
  const int nu = p.ntiles[0] + p.ntiles[1];

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(bar(&sh->full[i]), 1);
      mbar_init(bar(&sh->empty[i]), 1);
    }
    mbar_init(bar(&sh->tfull), 1);
    mbar_init(bar(&sh->tempty), kPEpiWarps * kPCl);
    mbar_init(bar(&sh->mma_done), 1);
    sh->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc2(smem_u32(&sh->tmem_base), 512);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&args.tx[0]);
    tma_prefetch_desc(&args.tx[1]);
    tma_prefetch_desc(&args.tw[0]);
    tma_prefetch_desc(&args.tw[1]);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();
  tc::fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  const uint32_t crank = tc::cluster_rank();
  const bool leader = crank == 0;

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      uint32_t s = 0;
      bool ok = true;
      for (int u = pair; u < nu && ok; u += npairs) {
        const PTile w = ptile_of(p, u);
        const int m0 = w.mt * (kPBM * kPCl) + (int)crank * kPBM;
        const int nkb = p.K[w.sel] / kPBK;
        for (int kb = 0; kb < nkb; ++kb, ++s) {
          const int st = s % kPStages;
          if (!pw_wait(bar(&sh->empty[st]), ((s / kPStages) & 1) ^ 1, abort, budget, p.status)) { ok = false; break; }
          const uint32_t dst = sbase + st * kPStage;
          const uint32_t fb = lead(&sh->full[st]);
          if (leader) mbar_arrive_expect_tx(bar(&sh->full[st]), kPCl * kPStage);
          tma_load_2d_pair(dst, &args.tx[w.sel], kb * kPBK, m0, fb);
          // this CTA's 128 of the tile's 256 columns: 64-column groups 2r, 2r+1
          tma_load_3d_pair(dst + 16384, &args.tw[w.sel], 0, kb * kPBK, w.nt * 4 + (int)crank * 2, fb);
        }
      }
      // the leader's full barriers count both CTAs' bytes: every issued copy
      // has landed before the pair may exit
      if (leader)
        for (uint32_t q = (s > (uint32_t)kPStages ? s - kPStages : 0); q < s; ++q)
          mbar_wait_bounded(bar(&sh->full[q % kPStages]), (q / kPStages) & 1, drain_budget(budget));
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer (leader)
    if (lane == 0 && leader) {
      const uint32_t idesc = tc::idesc_f16(false, 256, kPBN, false, true);
      const uint64_t dA0 = tc::sdesc_sw128(sbase, 16, 1024);
      const uint64_t dB0 = tc::sdesc_sw128(sbase + 16384, 8192, 1024);
      uint32_t s = 0, g = 0;
      bool ok = true;
      for (int u = pair; u < nu && ok; u += npairs) {
        const PTile w = ptile_of(p, u);
        const int nkb = p.K[w.sel] / kPBK;
        for (int kb = 0; kb < nkb && ok; ++kb, ++s) {
          const int ck = kb % kPChunkKB;
          if (ck == 0) {  // a new chunk: both CTAs' epilogues have drained the accumulator
            if (!pw_wait(bar(&sh->tempty), (g & 1) ^ 1, abort, budget, p.status, true)) { ok = false; break; }
            tc::fence_after_sync();
          }
          const int st = s % kPStages;
          if (!pw_wait(bar(&sh->full[st]), (s / kPStages) & 1, abort, budget, p.status)) { ok = false; break; }
          const uint64_t ad = dA0 + (uint64_t)((st * kPStage) >> 4);
          const uint64_t bd = dB0 + (uint64_t)((st * kPStage) >> 4);
#pragma unroll
          for (int k = 0; k < kPBK / 16; ++k)
            tc::mma2_f16(tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(128 * k), idesc, ck > 0 || k > 0);
          tc::commit2_both(bar(&sh->empty[st]));
          if (ck == kPChunkKB - 1 || kb == nkb - 1) {
            tc::commit2_both(bar(&sh->tfull));
            ++g;
          }
        }
      }
      tc::commit2_both(bar(&sh->mma_done));
      mbar_wait_bounded(bar(&sh->mma_done), 0, drain_budget(budget));
    } else if (lane == 0) {
      mbar_wait_bounded(bar(&sh->mma_done), 0, drain_budget(budget));
    }
  } else {
    // ============================================================ epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;  // token row within the CTA's 128
    const int c0 = ((warp - 2) >> 2) * (kPBN / 2);  // this warp's 128 columns
    const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t g = 0;
    bool ok = true;
    for (int u = pair; u < nu && ok; u += npairs) {
      const PTile w = ptile_of(p, u);
      const int nkb = p.K[w.sel] / kPBK;
      const int nch = (nkb + kPChunkKB - 1) / kPChunkKB;
      const int t = w.mt * (kPBM * kPCl) + (int)crank * kPBM + r;
      const bool live = t < p.T;
      for (int c = 0; c < nch && ok; ++c, ++g) {
        if (!pw_wait(bar(&sh->tfull), g & 1, abort, budget, p.status)) { ok = false; break; }
        tc::fence_after_sync();
        // chunk sum -> int32 sums in TMEM (the last chunk included, so that the
        // fp32 accumulator is released before the output stage)
#pragma unroll 1
        for (int j = c0; j < c0 + kPBN / 2; j += 32) {
          uint32_t f[32], iv[32];
          tc::ld32(lane_addr + j, f);
          if (c > 0) tc::ld32(lane_addr + kPIntCol + j, iv);
          tc::wait_ld();
          int v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = (c > 0 ? (int)iv[i] : 0) + __float2int_rn(__uint_as_float(f[i]));
          tc::st16(lane_addr + kPIntCol + j, reinterpret_cast<const uint32_t*>(v));
          tc::st16(lane_addr + kPIntCol + j + 16, reinterpret_cast<const uint32_t*>(v + 16));
        }
        tc::wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::arrive_cluster_relaxed(lead(&sh->tempty));
      }
      if (!ok) break;
      // ---- output stage from the int32 sums (the MMAs of the next tile's
      // first chunk run meanwhile)
      const int n0 = w.nt * kPBN;
      if constexpr (MODE == 0) {
#pragma unroll 1
        for (int j = c0; j < c0 + kPBN / 2; j += 32) {
          uint32_t iv[32];
          tc::ld32(lane_addr + kPIntCol + j, iv);
          tc::wait_ld();
          const int col = n0 + j;
          if (live && col < p.N[w.sel]) {
            int32_t* dst = p.C + (size_t)t * p.ldc + p.coff[w.sel] + col;
            const int ncol = p.N[w.sel] - col < 32 ? p.N[w.sel] - col : 32;  // a multiple of 8
#pragma unroll
            for (int k = 0; k < 8; ++k)
              if (4 * k < ncol)
                *reinterpret_cast<int4*>(dst + 4 * k) =
                    make_int4((int)iv[4 * k], (int)iv[4 * k + 1], (int)iv[4 * k + 2], (int)iv[4 * k + 3]);
          }
        }
      } else {
        const int width = w.sel == 0 ? kNope + kRope : kHeadCols;
        const float sx = live ? p.sx[w.sel][t] : 0.f;
        int pos = 0;
        if (live && w.sel == 0) {
          pos = p.positions[t];
          if (pos < 0 || pos >= p.max_pos) pos = pos < 0 ? 0 : p.max_pos - 1;
        }
        const int bi = (int)((__umulhi((unsigned)t, p.s_mul) + (unsigned)t) >> p.s_shift);
        const int si = t - bi * p.s;
        int32_t* cap = p.cap[w.sel];
        unsigned char* stg = smem + kPStgBase + (warp - 2) * kPStgWarp;
        // 32 columns (one head part) straight from registers: q_pe (RoPE
        // pairs), and any pair of 32-column groups that is not 64 columns of
        // one plain part
        auto direct = [&](const uint32_t* iv, int col) {
          if (!live || col >= p.N[w.sel]) return;
          if (cap) {
            int4* cp = reinterpret_cast<int4*>(cap + (size_t)t * p.N[w.sel] + col);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              cp[k] = make_int4((int)iv[4 * k], (int)iv[4 * k + 1], (int)iv[4 * k + 2], (int)iv[4 * k + 3]);
          }
          const float* swp = p.sw[w.sel] + col;
          float y[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 sw = __ldg(reinterpret_cast<const float4*>(swp) + k);
            y[4 * k] = __fmul_rn(__fmul_rn((float)(int)iv[4 * k], sx), sw.x);
            y[4 * k + 1] = __fmul_rn(__fmul_rn((float)(int)iv[4 * k + 1], sx), sw.y);
            y[4 * k + 2] = __fmul_rn(__fmul_rn((float)(int)iv[4 * k + 2], sx), sw.z);
            y[4 * k + 3] = __fmul_rn(__fmul_rn((float)(int)iv[4 * k + 3], sx), sw.w);
          }
          const int hh = col / width, e = col - hh * width;
          const size_t orow = ((size_t)bi * p.heads + hh) * p.s + si;
          if (w.sel == 1 || e < kNope) {
            __nv_bfloat16* dst = w.sel == 0 ? static_cast<__nv_bfloat16*>(p.q_nope) + orow * kNope + e
                                 : (e < kNope ? static_cast<__nv_bfloat16*>(p.k_nope) + orow * kNope + e
                                              : static_cast<__nv_bfloat16*>(p.value) + orow * kV + (e - kNope));
            uint32_t o[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              __nv_bfloat162 h2 = __floats2bfloat162_rn(y[2 * k], y[2 * k + 1]);
              o[k] = *reinterpret_cast<uint32_t*>(&h2);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k)
              reinterpret_cast<uint4*>(dst)[k] = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
          } else {
            // RoPE of q_pe: columns ie0 .. ie0+31 (ie0 = e - 128, 0 or 32) are
            // the pairs (x[2m], x[2m+1]), m = j0 .. j0+15 with j0 = ie0 / 2
            const int j0 = (e - kNope) >> 1;
            const float* cr = p.cos_t + (size_t)pos * kRope;
            const float* sr = p.sin_t + (size_t)pos * kRope;
            uint32_t lo[8], hi[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float4 c0 = __ldg(reinterpret_cast<const float4*>(cr + j0) + k);
              const float4 s0 = __ldg(reinterpret_cast<const float4*>(sr + j0) + k);
              const float4 c1 = __ldg(reinterpret_cast<const float4*>(cr + 32 + j0) + k);
              const float4 s1 = __ldg(reinterpret_cast<const float4*>(sr + 32 + j0) + k);
              const float* x = y + 8 * k;  // pairs m = j0 + 4k .. j0 + 4k + 3
              __nv_bfloat162 a = __floats2bfloat162_rn(x[0] * c0.x - x[1] * s0.x, x[2] * c0.y - x[3] * s0.y);
              __nv_bfloat162 b = __floats2bfloat162_rn(x[4] * c0.z - x[5] * s0.z, x[6] * c0.w - x[7] * s0.w);
              __nv_bfloat162 cc = __floats2bfloat162_rn(x[1] * c1.x + x[0] * s1.x, x[3] * c1.y + x[2] * s1.y);
              __nv_bfloat162 d = __floats2bfloat162_rn(x[5] * c1.z + x[4] * s1.z, x[7] * c1.w + x[6] * s1.w);
              lo[2 * k] = *reinterpret_cast<uint32_t*>(&a);
              lo[2 * k + 1] = *reinterpret_cast<uint32_t*>(&b);
              hi[2 * k] = *reinterpret_cast<uint32_t*>(&cc);
              hi[2 * k + 1] = *reinterpret_cast<uint32_t*>(&d);
            }
            __nv_bfloat16* qp = static_cast<__nv_bfloat16*>(p.q_pe) + orow * kRope;
            reinterpret_cast<uint4*>(qp + j0)[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            reinterpret_cast<uint4*>(qp + j0)[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
            reinterpret_cast<uint4*>(qp + 32 + j0)[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            reinterpret_cast<uint4*>(qp + 32 + j0)[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
          }
        };
        // 64 columns per step.  The tile, the warp's 128-column half and the
        // step all start at multiples of 64 columns, and 64 divides both head
        // parts' boundaries (128 and 192 or 256), so a step lies inside one
        // part.  A plain part (q_nope, k_nope, value) goes through the warp's
        // staging area: each lane writes its row's 128 bytes (16-byte slots
        // swizzled by row), then each store instruction writes four rows as
        // whole 128-byte segments instead of 32 rows' 16-byte pieces.
#pragma unroll 1
        for (int j = c0; j < c0 + kPBN / 2; j += 64) {
          const int col = n0 + j;
          const int hh = col / width, e = col - hh * width;
          if (!((w.sel == 1 || e < kNope) && col + 64 <= p.N[w.sel])) {
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
              uint32_t iv[32];
              tc::ld32(lane_addr + kPIntCol + j + 32 * h, iv);
              tc::wait_ld();
              direct(iv, col + 32 * h);
            }
            continue;
          }
          __nv_bfloat16* rowp = nullptr;
          if (live) {
            const size_t orow = ((size_t)bi * p.heads + hh) * p.s + si;
            rowp = w.sel == 0 ? static_cast<__nv_bfloat16*>(p.q_nope) + orow * kNope + e
                   : (e < kNope ? static_cast<__nv_bfloat16*>(p.k_nope) + orow * kNope + e
                                : static_cast<__nv_bfloat16*>(p.value) + orow * kV + (e - kNope));
          }
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {  // 32 columns: 16-byte slots 4h .. 4h+3
            uint32_t iv[32];
            tc::ld32(lane_addr + kPIntCol + j + 32 * h, iv);
            tc::wait_ld();
            if (cap && live) {
              int4* cp = reinterpret_cast<int4*>(cap + (size_t)t * p.N[w.sel] + col + 32 * h);
#pragma unroll
              for (int k = 0; k < 8; ++k)
                cp[k] = make_int4((int)iv[4 * k], (int)iv[4 * k + 1], (int)iv[4 * k + 2], (int)iv[4 * k + 3]);
            }
            const float* swp = p.sw[w.sel] + col + 32 * h;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int sl = 4 * h + k;
              const float4 sa = __ldg(reinterpret_cast<const float4*>(swp + 8 * k));
              const float4 sb = __ldg(reinterpret_cast<const float4*>(swp + 8 * k + 4));
              const uint32_t* x = iv + 8 * k;
              __nv_bfloat162 o0 = __floats2bfloat162_rn(__fmul_rn(__fmul_rn((float)(int)x[0], sx), sa.x),
                                                        __fmul_rn(__fmul_rn((float)(int)x[1], sx), sa.y));
              __nv_bfloat162 o1 = __floats2bfloat162_rn(__fmul_rn(__fmul_rn((float)(int)x[2], sx), sa.z),
                                                        __fmul_rn(__fmul_rn((float)(int)x[3], sx), sa.w));
              __nv_bfloat162 o2 = __floats2bfloat162_rn(__fmul_rn(__fmul_rn((float)(int)x[4], sx), sb.x),
                                                        __fmul_rn(__fmul_rn((float)(int)x[5], sx), sb.y));
              __nv_bfloat162 o3 = __floats2bfloat162_rn(__fmul_rn(__fmul_rn((float)(int)x[6], sx), sb.z),
                                                        __fmul_rn(__fmul_rn((float)(int)x[7], sx), sb.w));
              *reinterpret_cast<uint4*>(stg + lane * 128 + ((sl ^ (lane & 7)) << 4)) =
                  make_uint4(*reinterpret_cast<uint32_t*>(&o0), *reinterpret_cast<uint32_t*>(&o1),
                             *reinterpret_cast<uint32_t*>(&o2), *reinterpret_cast<uint32_t*>(&o3));
            }
          }
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int rr = 4 * k + (lane >> 3), sl = lane & 7;
            const unsigned long long pr = __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(rowp), rr);
            const uint4 val = *reinterpret_cast<const uint4*>(stg + rr * 128 + ((sl ^ (rr & 7)) << 4));
            if (pr) reinterpret_cast<uint4*>(pr)[sl] = val;
          }
          __syncwarp();  // the slots are rewritten by the next step
        }
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

// int8 [K, N] -> fp16: row k of job j goes to out + k * ldn, columns
// [0, wcols) (columns N .. wcols-1 zero), 16 values per thread (exact:
// |v| <= 127).  Up to four matrices per launch.
struct WidenJobs {
  W8WidenJob j[4];
  long start[5];  // prefix sums of the jobs' 16-column groups
  int n;
};

__global__ void widen_kernel(const __grid_constant__ WidenJobs J) {
  // four 16-column groups per thread and pass, all loads issued first
  const long n = J.start[J.n], stride = (long)gridDim.x * blockDim.x;
  for (long i0 = blockIdx.x * (long)blockDim.x + threadIdx.x; i0 < n; i0 += 4 * stride) {
    uint4 v[4];
    int job[4], row[4], col[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long i = i0 + u * stride;
      job[u] = -1;
      if (i >= n) continue;
      int q = 0;
      while (i >= J.start[q + 1]) ++q;
      const W8WidenJob& jb = J.j[q];
      const long g = i - J.start[q];
      const int gpr = jb.wcols / 16;
      job[u] = q;
      row[u] = (int)(g / gpr);
      col[u] = (int)(g % gpr) * 16;
      if (col[u] + 16 <= jb.N) v[u] = __ldg(reinterpret_cast<const uint4*>(jb.W + (size_t)row[u] * jb.N + col[u]));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (job[u] < 0) continue;
      const W8WidenJob& jb = J.j[job[u]];
      const int k = row[u], c = col[u];
      __align__(16) __half h[16];
      if (c + 16 <= jb.N) {
        const int8_t* b = reinterpret_cast<const int8_t*>(&v[u]);
#pragma unroll
        for (int x = 0; x < 16; ++x) h[x] = __int2half_rn((int)b[x]);
      } else {
#pragma unroll
        for (int x = 0; x < 16; ++x) h[x] = __int2half_rn(c + x < jb.N ? (int)jb.W[(size_t)k * jb.N + c + x] : 0);
      }
      uint4* d = reinterpret_cast<uint4*>(jb.out + (size_t)k * jb.ldn + c);
      d[0] = *reinterpret_cast<const uint4*>(h);
      d[1] = *reinterpret_cast<const uint4*>(h + 8);
    }
  }
}

}  // namespace

cudaError_t w8_widen_launch(const W8WidenJob* jobs, int n, int num_sms, cudaStream_t stream) {
  if (n < 1 || n > 4) return cudaErrorInvalidValue;
  WidenJobs J = {};
  J.n = n;
  J.start[0] = 0;
  for (int i = 0; i < n; ++i) {
    const W8WidenJob& jb = jobs[i];
    if (jb.N % 16 != 0 || jb.wcols % 16 != 0 || jb.wcols < jb.N || jb.ldn % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(jb.out) & 15u) != 0)
      return cudaErrorNotSupported;
    J.j[i] = jb;
    J.start[i + 1] = J.start[i] + (long)jb.K * (jb.wcols / 16);
  }
  widen_kernel<<<num_sms * 8, 256, 0, stream>>>(J);
  return cudaGetLastError();
}

cudaError_t w8pair_launch(W8PairParams p, const void* X0, const void* X1, const __half* W0, const __half* W1,
                          int num_sms, cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  PArgs a;
  const void* Xs[2] = {X0, X1};
  const __half* Ws[2] = {W0, W1};
  const int mtiles = (p.T + kPBM * kPCl - 1) / (kPBM * kPCl);
  for (int i = 0; i < 2; ++i) {
    if (p.N[i] == 0) {
      p.ntiles[i] = 0;
      p.nn[i] = 1;
      a.tx[i] = a.tx[0];
      a.tw[i] = a.tw[0];
      continue;
    }
    if (p.K[i] % kPBK != 0 || p.ldw[i] % kPBN != 0 || p.N[i] % 32 != 0 || p.N[i] > p.ldw[i])
      return cudaErrorNotSupported;
    if (!encode_tmap_2d(&a.tx[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Xs[i], (uint64_t)p.K[i], (uint64_t)p.T,
                        (uint64_t)p.K[i] * 2, kPBK, kPBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_3d_colblocks(&a.tw[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Ws[i], (uint64_t)p.ldw[i],
                                  (uint64_t)p.K[i], (uint64_t)p.ldw[i] * 2, kPBK, kPBK, 2, 2,
                                  CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    p.nn[i] = (p.N[i] + kPBN - 1) / kPBN;
    p.ntiles[i] = mtiles * p.nn[i];
    p.mfast[i] = (size_t)p.T * p.K[i] < (size_t)p.K[i] * p.ldw[i] ? 1 : 0;
  }
  p.nm = mtiles;
  {
    const unsigned d = (unsigned)(p.s > 0 ? p.s : 1);
    unsigned l = 0;
    while ((1ull << l) < d) ++l;
    p.s_shift = l;
    p.s_mul = (unsigned)((((1ull << l) - d) << 32) / d + 1);
  }
  a.p = p;
  const void* fn = p.raw ? (const void*)w8pair_kernel<0> : (const void*)w8pair_kernel<1>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPCl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int max_clusters = 0;
  if (max_clusters == 0) {
    cfg.gridDim = dim3(num_sms / kPCl * kPCl);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = num_sms / kPCl;
    }
    max_clusters = n;
  }
  const int total = p.ntiles[0] + p.ntiles[1];
  int pairs = total < max_clusters ? total : max_clusters;
  cfg.gridDim = dim3(pairs * kPCl);
  void* kargs[] = {&a};
  return cudaLaunchKernelExC(&cfg, fn, kargs);
}

}  // namespace mla
