// w8mma.cu -- the int8 GEMMs of the W8A8 prolog on the 5th-generation
// tensor cores (tcgen05 / TMEM / TMA), for T > kW8SmallRows token rows.
//
// The W8A8 mode of "DeepSeek-R1或Kimi-K2模型在NPU实现高性能推理" §权重转换 keeps
// int8 weights with per-output-channel scales and int8 activations whose
// products are summed exactly in int32.  sm_103a has no int8 kind of
// tcgen05.mma, so the products run as fp16 x fp16 -> fp32 MMAs, exactly:
//   * every int8 code v (|v| <= 127) is an fp16 value, and every product
//     (|p| <= 127 * 127 < 2^14) is exact in fp32;
//   * the accumulator is restarted every kChunkK = 512 K rows, so every
//     partial sum is an integer of magnitude <= 512 * 127 * 127 < 2^23,
//     exactly representable in fp32 whatever order the tensor core adds in;
//   * each chunk's fp32 sum is converted to int32 (exact) and the chunks are
//     added as int32 in tensor memory.
// The result is the int32 accumulator bit for bit.
//
// Orientation: the weight columns are the MMA's M side (128 per tile, one
// TMEM lane each) and the token rows its N side (NT <= 128 per tile), so
// one tile streams a [K x 128] weight panel once for all of its tokens.
// (The int8 -> fp16 conversion costs shared-memory traffic per weight byte,
// so more tokens per tile make it cheaper per FLOP; 160 is the most that
// leaves room for two fp32 accumulators and the int32 sums in TMEM.)
// The weights stay int8 in memory: TMA brings [64 K x 128] int8 boxes into
// shared memory and four converter warps rewrite each box as the fp16
// MN-major, 128-byte-swizzled A operand (magic-number conversion: the
// biased byte becomes the mantissa of 1024 + u, minus 1152).  The
// activations arrive as fp16 codes (written so by the quantisation kernels)
// in K-major swizzled boxes, the B operand.
//
// Warp roles (320 threads, one CTA per SM, persistent over work units):
//   warp 0     TMA producer: int8 weight box + activation box per K block
//   warp 1     TMEM allocation (512 columns); one thread issues the MMAs
//   warps 2-5  converters: int8 box -> fp16 A operand
//   warps 6-9  epilogue: chunk sums into int32, then the output stage
// Tensor memory: fp32 chunk accumulators in columns [0, 160) and [160,
// 320) (chunks alternate, so the MMAs of one chunk run while the epilogue
// drains the previous one), the tile's int32 sum in [320, 480).
//
// Output stages (mode):
//   RAW    the int32 sums are added (red.add, exact) into C [T, ldc] at
//          column offset coff[matrix]: q_a | kv_a into the accumulator rows
//          that the normalisation kernel reads (K may be split across units).
//   HEADS  dequantise y = (float)acc * s_x[t] * s_w[n] and write the
//          head-major outputs: q_b -> q_nope, RoPE(q_pe) (de-interleaved
//          pairs, rotate_half); kv_b -> k_nope, value.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tma.h"

namespace mla {
namespace {

constexpr int kMmThreads = 320;
constexpr int kMmBM = 128;            // weight columns per tile (TMEM lanes)
constexpr int kMmBK = 64;             // K rows per block
constexpr int kChunkKB = 8;           // K blocks per exact fp32 chunk (512 rows)
constexpr int kMaxStages = 12;        // int8 weight + activation box ring
constexpr int kASlots = 3;            // converted fp16 A operand ring
constexpr uint32_t kWBytes = kMmBM * kMmBK;          // int8 weight box: 8 KB
constexpr uint32_t kABytes = kMmBM * kMmBK * 2;      // fp16 A operand: 16 KB
constexpr int kMaxNT = 160;           // tokens per tile (3 x 160 TMEM columns fit in 512)
constexpr uint32_t kSlotCols = 160;   // TMEM column of fp32 chunk accumulator 1 (0 is at column 0)
constexpr uint32_t kIntCol = 320;     // TMEM column of the int32 sums
constexpr int kEpPitch = 36;          // floats per token row of an epilogue warp's transpose tile
constexpr uint32_t kEpBytes = 32 * kEpPitch * 4;  // per epilogue warp
constexpr int kSmemBudget = 227 * 1024;

struct MmShared {
  uint64_t st_full[kMaxStages], st_empty[kMaxStages];
  uint64_t a_full[kASlots], a_empty[kASlots];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

struct MmUnit {
  int sel, mtile, ntile, kb0, kb1;
};

__device__ __forceinline__ MmUnit unit_of(const W8MmaParams& p, int u) {
  MmUnit r;
  r.sel = u < p.nunits[0] ? 0 : 1;
  int v = u - (r.sel ? p.nunits[0] : 0);
  // Order of the units: with mfast, weight tiles fastest (the CTAs running at
  // the same time share token tiles; for activations larger than the
  // weights), otherwise token tiles fastest (they share weight panels).
  const int ks = p.ks[r.sel];
  int split;
  if (p.mfast[r.sel]) {
    r.mtile = v % p.mt[r.sel];
    v /= p.mt[r.sel];
    split = v % ks;
    r.ntile = v / ks;
  } else {
    r.ntile = v % p.ntiles;
    v /= p.ntiles;
    split = v % ks;
    r.mtile = v / ks;
  }
  r.kb0 = split * p.kbps[r.sel];
  const int nkb = p.K[r.sel] / kMmBK;
  r.kb1 = r.kb0 + p.kbps[r.sel] < nkb ? r.kb0 + p.kbps[r.sel] : nkb;
  return r;
}

// Bounded wait shared by all roles (gives up on the time budget, or when
// another role already has).  try_wait lets the hardware suspend the thread
// until the phase completes (or a time slice ends), so the many waiting
// threads do not flood shared memory with polls.
__device__ __forceinline__ bool mm_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                        unsigned long long budget, unsigned* status) {
  if (mbar_try_wait_hint(bar, parity, 20000)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_hint(bar, parity, 20000)) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > budget) {
      *abort = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
  return true;
}

// Four int8 codes -> two fp16x2 words (exact): byte u = v + 128 becomes the
// low mantissa byte of 0x64uu = 1024 + u, and 1024 + u - 1152 = v.
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
  uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

template <int MODE>
__global__ void __launch_bounds__(kMmThreads, 1) w8mma_kernel(const __grid_constant__ W8MmaParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  // layout: A slots [kASlots][16 KB] | stages [S][8 KB weights + NT x 128 B] |
  // epilogue transpose tiles [4][32 x 36 floats] | barriers.  The activation
  // box has xrows <= NT rows; the MMA reads NT rows (rows past xrows only
  // feed token columns that are not stored).
  const uint32_t xbytes = (uint32_t)p.xrows * 128;
  const uint32_t stage_bytes = (kWBytes + (uint32_t)p.NT * 128 + 1023) / 1024 * 1024;
  const int S = p.stages;
  unsigned char* sA = smem;
  unsigned char* sSt = smem + kASlots * kABytes;
  float* sEp = reinterpret_cast<float*>(sSt + (size_t)S * stage_bytes);
  MmShared* sh = reinterpret_cast<MmShared*>(reinterpret_cast<unsigned char*>(sEp) + 4 * kEpBytes);
  const uint32_t a_base = smem_u32(sA), st_base = smem_u32(sSt);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &sh->abort;
  const unsigned long long budget = p.budget_ns;
  const int G = gridDim.x;
  const int nu = p.nunits[0] + p.nunits[1];
  auto bar = [&](uint64_t* b) { return smem_u32(b); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(bar(&sh->st_full[i]), 1);
      mbar_init(bar(&sh->st_empty[i]), 5);  // four converter warps + the MMA commit
    }
    for (int i = 0; i < kASlots; ++i) {
      mbar_init(bar(&sh->a_full[i]), 4);
      mbar_init(bar(&sh->a_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(&sh->acc_full[i]), 1);
      mbar_init(bar(&sh->acc_empty[i]), 4);
    }
    mbar_init(bar(&sh->mma_done), 1);
    sh->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(smem_u32(&sh->tmem_base), 512);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tw[0]);
    tma_prefetch_desc(&p.tw[1]);
    tma_prefetch_desc(&p.tx[0]);
    tma_prefetch_desc(&p.tx[1]);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  // the activations (and, in RAW mode, the accumulator rows) come from the
  // kernels before this one; the kernel after this one may launch now
  grid_dep_launch_dependents();
  grid_dep_wait();

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      uint32_t s = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nu && ok; u += G) {
        const MmUnit w = unit_of(p, u);
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++s) {
          const int st = s % S;
          if (!mm_wait(bar(&sh->st_empty[st]), ((s / S) & 1) ^ 1, abort, budget, p.status)) { ok = false; break; }
          const uint32_t dst = st_base + st * stage_bytes;
          mbar_arrive_expect_tx(bar(&sh->st_full[st]), kWBytes + xbytes);
          tma_load_2d(dst, &p.tw[w.sel], w.mtile * kMmBM, kb * kMmBK, bar(&sh->st_full[st]));
          tma_load_2d(dst + kWBytes, &p.tx[w.sel], kb * kMmBK, w.ntile * p.NT, bar(&sh->st_full[st]));
        }
      }
      // every issued copy has landed before the CTA may exit (bounded, but
      // not cut short by another role's abort)
      for (uint32_t q = (s > (uint32_t)S ? s - S : 0); q < s; ++q)
        mbar_wait_bounded(bar(&sh->st_full[q % S]), (q / S) & 1, drain_budget(budget));
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_f16(false, kMmBM, p.NT, true, false);
      // A: MN-major fp16, two 64-column groups 8 KB apart, 8-row K groups
      // 1 KB apart; B: K-major 128-byte rows (activation box)
      const uint64_t dA0 = tc::sdesc_sw128(a_base, 8192, 1024);
      const uint64_t dB0 = tc::sdesc_sw128(st_base + kWBytes, 16, 1024);
      uint32_t s = 0, a = 0, g = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nu && ok; u += G) {
        const MmUnit w = unit_of(p, u);
        for (int kb = w.kb0; kb < w.kb1 && ok; ++kb, ++s, ++a) {
          const int ck = (kb - w.kb0) % kChunkKB;
          const uint32_t slot = g & 1;
          if (ck == 0) {  // a new chunk: its fp32 accumulator must be drained
            if (!mm_wait(bar(&sh->acc_empty[slot]), ((g >> 1) & 1) ^ 1, abort, budget, p.status)) { ok = false; break; }
            tc::fence_after_sync();
          }
          const int st = s % S, as = a % kASlots;
          if (!mm_wait(bar(&sh->st_full[st]), (s / S) & 1, abort, budget, p.status)) { ok = false; break; }
          if (!mm_wait(bar(&sh->a_full[as]), (a / kASlots) & 1, abort, budget, p.status)) { ok = false; break; }
          tc::fence_after_sync();
          const uint64_t ad = dA0 + (uint64_t)((as * kABytes) >> 4);
          const uint64_t bd = dB0 + (uint64_t)((st * stage_bytes) >> 4);
          const uint32_t d = tmem + slot * kSlotCols;
#pragma unroll
          for (int k = 0; k < kMmBK / 16; ++k)  // A advances 16 K rows (2 KB), B 32 bytes
            tc::mma_f16(d, ad + (uint64_t)(k * 128), bd + (uint64_t)(k * 2), idesc, ck > 0 || k > 0);
          tc::commit(bar(&sh->st_empty[st]));
          tc::commit(bar(&sh->a_empty[as]));
          if (ck == kChunkKB - 1 || kb == w.kb1 - 1) {
            tc::commit(bar(&sh->acc_full[slot]));
            ++g;
          }
        }
      }
      // every MMA issued has completed before tensor memory is released
      tc::commit(bar(&sh->mma_done));
      mbar_wait_bounded(bar(&sh->mma_done), 0, drain_budget(budget));
    }
  } else if (warp < 6) {
    // ============================================================ converters
    const int ct = threadIdx.x - 64;  // 0..127
    uint32_t s = 0, a = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < nu && ok; u += G) {
      const MmUnit w = unit_of(p, u);
      for (int kb = w.kb0; kb < w.kb1; ++kb, ++s, ++a) {
        const int st = s % S, as = a % kASlots;
        if (!mm_wait(bar(&sh->st_full[st]), (s / S) & 1, abort, budget, p.status) ||
            !mm_wait(bar(&sh->a_empty[as]), ((a / kASlots) & 1) ^ 1, abort, budget, p.status)) {
          ok = false;
          break;
        }
        const unsigned char* src = sSt + (size_t)st * stage_bytes;
        unsigned char* dst = sA + (size_t)as * kABytes;
        // all four loads before the first store (the compiler keeps a load
        // of shared memory behind an earlier store that may alias it)
        uint4 vin[4];
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int item = ct + 128 * it;
          vin[it] = *reinterpret_cast<const uint4*>(src + (item >> 3) * 128 + (item & 7) * 16);
        }
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int item = ct + 128 * it;      // 512 items of 16 int8
          const int k = item >> 3, c = item & 7;
          const uint4 v = vin[it];
          uint32_t h[8];
          i8x4_to_f16(v.x, h[0], h[1]);
          i8x4_to_f16(v.y, h[2], h[3]);
          i8x4_to_f16(v.z, h[4], h[5]);
          i8x4_to_f16(v.w, h[6], h[7]);
          // columns 16c .. 16c+15: group c/4, 16-byte chunks 2(c%4), 2(c%4)+1 of row k
          unsigned char* row = dst + (c >> 2) * 8192 + (k >> 3) * 1024 + (k & 7) * 128;
          const int c0 = 2 * (c & 3);
          *reinterpret_cast<uint4*>(row + (((c0) ^ (k & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (k & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
        tc::fence_proxy_async_smem();  // generic-proxy writes -> the MMA (async proxy)
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(&sh->a_full[as]));
          mbar_arrive(bar(&sh->st_empty[st]));
        }
      }
    }
  } else {
    // ============================================================ epilogue
    const int q = warp & 3;                    // TMEM lane quadrant
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t g = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < nu && ok; u += G) {
      const MmUnit w = unit_of(p, u);
      const int nch = (w.kb1 - w.kb0 + kChunkKB - 1) / kChunkKB;
      const int col = w.mtile * kMmBM + q * 32 + lane;  // this thread's weight column
      const bool col_ok = col < p.N[w.sel];
      const int n0 = w.ntile * p.NT;
      for (int c = 0; c < nch && ok; ++c, ++g) {
        const uint32_t slot = g & 1;
        if (!mm_wait(bar(&sh->acc_full[slot]), (g >> 1) & 1, abort, budget, p.status)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t fa = lane_base + slot * kSlotCols, ia = lane_base + kIntCol;
        const bool last = c == nch - 1;
        for (int j = 0; j < p.NT; j += 32) {
          uint32_t f[32], iv[32];
          tc::ld32(fa + j, f);
          if (c > 0) tc::ld32(ia + j, iv);
          tc::wait_ld();
          int v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = (c > 0 ? (int)iv[i] : 0) + __float2int_rn(__uint_as_float(f[i]));
          if (!last) {
            tc::st16(ia + j, reinterpret_cast<const uint32_t*>(v));
            tc::st16(ia + j + 16, reinterpret_cast<const uint32_t*>(v + 16));
            continue;
          }
          // ---- output stage for tokens n0 + j .. n0 + j + 31 of this column
          if constexpr (MODE == 0) {
            if (col_ok) {
              int32_t* cp = p.C + p.coff[w.sel] + col;
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int t = n0 + j + i;
                if (t < p.T) atomicAdd(cp + (size_t)t * p.ldc, v[i]);
              }
            }
          } else {
            // transpose the warp's 32 columns x 32 tokens of int32 sums through
            // shared memory; then lane (r, c) owns columns 8c .. 8c+7 of token
            // r: dequantise y = (float)acc * s_x[t] * s_w[n] and write 16-byte
            // pieces of the head-major outputs
            const int width = w.sel == 0 ? kNope + kRope : kHeadCols;
            int32_t* cap = p.cap[w.sel];
            int* tile = reinterpret_cast<int*>(sEp) + (size_t)q * (32 * kEpPitch);
#pragma unroll
            for (int i = 0; i < 32; ++i) tile[i * kEpPitch + lane] = v[i];
            if (cap && col_ok) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (n0 + j + i < p.T) cap[(size_t)(n0 + j + i) * p.N[w.sel] + col] = v[i];
            }
            __syncwarp();
            const int c = lane & 3;
            const int fb = w.mtile * kMmBM + q * 32 + 8 * c;   // first of this lane's 8 columns
            const int hh = fb / width, e = fb - hh * width;    // 8 columns inside one head part
            const bool fb_ok = fb < p.N[w.sel];
            float4 swa = make_float4(0.f, 0.f, 0.f, 0.f), swb = swa;
            if (fb_ok) {
              swa = *reinterpret_cast<const float4*>(p.sw[w.sel] + fb);
              swb = *reinterpret_cast<const float4*>(p.sw[w.sel] + fb + 4);
            }
#pragma unroll
            for (int it = 0; it < 4; ++it) {
              const int r = it * 8 + (lane >> 2);
              const int t = n0 + j + r;
              if (t >= p.T || !fb_ok) continue;
              const float sx = p.sx[w.sel][t];
              const int4 ia = *reinterpret_cast<const int4*>(tile + r * kEpPitch + 8 * c);
              const int4 ib = *reinterpret_cast<const int4*>(tile + r * kEpPitch + 8 * c + 4);
              float4 ya, yb;
              ya.x = __fmul_rn(__fmul_rn((float)ia.x, sx), swa.x);
              ya.y = __fmul_rn(__fmul_rn((float)ia.y, sx), swa.y);
              ya.z = __fmul_rn(__fmul_rn((float)ia.z, sx), swa.z);
              ya.w = __fmul_rn(__fmul_rn((float)ia.w, sx), swa.w);
              yb.x = __fmul_rn(__fmul_rn((float)ib.x, sx), swb.x);
              yb.y = __fmul_rn(__fmul_rn((float)ib.y, sx), swb.y);
              yb.z = __fmul_rn(__fmul_rn((float)ib.z, sx), swb.z);
              yb.w = __fmul_rn(__fmul_rn((float)ib.w, sx), swb.w);
              const int bi = (int)((__umulhi((unsigned)t, p.s_mul) + (unsigned)t) >> p.s_shift);
              const int si = t - bi * p.s;
              const size_t orow = ((size_t)bi * p.heads + hh) * p.s + si;
              if (w.sel == 1 || e < kNope) {
                __nv_bfloat16* dst = w.sel == 0 ? static_cast<__nv_bfloat16*>(p.q_nope) + orow * kNope + e
                                     : (e < kNope ? static_cast<__nv_bfloat16*>(p.k_nope) + orow * kNope + e
                                                  : static_cast<__nv_bfloat16*>(p.value) + orow * kV + (e - kNope));
                __nv_bfloat162 o0 = __floats2bfloat162_rn(ya.x, ya.y), o1 = __floats2bfloat162_rn(ya.z, ya.w);
                __nv_bfloat162 o2 = __floats2bfloat162_rn(yb.x, yb.y), o3 = __floats2bfloat162_rn(yb.z, yb.w);
                *reinterpret_cast<uint4*>(dst) =
                    make_uint4(*reinterpret_cast<uint32_t*>(&o0), *reinterpret_cast<uint32_t*>(&o1),
                               *reinterpret_cast<uint32_t*>(&o2), *reinterpret_cast<uint32_t*>(&o3));
              } else {
                // RoPE of q_pe: columns ie .. ie+7 are the pairs (x[2m], x[2m+1])
                // for m = j0 .. j0+3, j0 = ie / 2; out[m] = x[2m] cos[m] -
                // x[2m+1] sin[m], out[m+32] = x[2m+1] cos[m+32] + x[2m] sin[m+32]
                const int j0 = (e - kNope) >> 1;
                int pos = p.positions[t];
                if (pos < 0 || pos >= p.max_pos) pos = pos < 0 ? 0 : p.max_pos - 1;
                const float4 c0 = *reinterpret_cast<const float4*>(p.cos_t + (size_t)pos * kRope + j0);
                const float4 s0 = *reinterpret_cast<const float4*>(p.sin_t + (size_t)pos * kRope + j0);
                const float4 c1 = *reinterpret_cast<const float4*>(p.cos_t + (size_t)pos * kRope + 32 + j0);
                const float4 s1 = *reinterpret_cast<const float4*>(p.sin_t + (size_t)pos * kRope + 32 + j0);
                __nv_bfloat162 lo0 = __floats2bfloat162_rn(ya.x * c0.x - ya.y * s0.x, ya.z * c0.y - ya.w * s0.y);
                __nv_bfloat162 lo1 = __floats2bfloat162_rn(yb.x * c0.z - yb.y * s0.z, yb.z * c0.w - yb.w * s0.w);
                __nv_bfloat162 hi0 = __floats2bfloat162_rn(ya.y * c1.x + ya.x * s1.x, ya.w * c1.y + ya.z * s1.y);
                __nv_bfloat162 hi1 = __floats2bfloat162_rn(yb.y * c1.z + yb.x * s1.z, yb.w * c1.w + yb.z * s1.w);
                __nv_bfloat16* qp = static_cast<__nv_bfloat16*>(p.q_pe) + orow * kRope;
                *reinterpret_cast<uint2*>(qp + j0) =
                    make_uint2(*reinterpret_cast<uint32_t*>(&lo0), *reinterpret_cast<uint32_t*>(&lo1));
                *reinterpret_cast<uint2*>(qp + 32 + j0) =
                    make_uint2(*reinterpret_cast<uint32_t*>(&hi0), *reinterpret_cast<uint32_t*>(&hi1));
              }
            }
            __syncwarp();  // the tile is rewritten by the next 32 tokens
          }
        }
        if (!last) tc::wait_st();
        // chunk slot drained: the MMA may write it again
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(&sh->acc_empty[slot]));
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

bool encode_w8(CUtensorMap* m, const int8_t* W, int K, int N) {
  return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, (uint64_t)N, (uint64_t)K, (uint64_t)N, kMmBM,
                        kMmBK, CU_TENSOR_MAP_SWIZZLE_NONE);
}
bool encode_x16(CUtensorMap* m, const void* X, int T, int K, int rows) {
  return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, X, (uint64_t)K, (uint64_t)T, (uint64_t)K * 2, kMmBK,
                        (uint32_t)rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

size_t w8mma_smem(int NT, int stages) {
  const size_t stage = (kWBytes + (size_t)NT * 128 + 1023) / 1024 * 1024;
  return 1024 + kASlots * (size_t)kABytes + (size_t)stages * stage + 4 * (size_t)kEpBytes + sizeof(MmShared) + 64;
}

cudaError_t w8mma_launch(W8MmaParams p, const int8_t* W0, const int8_t* W1, const void* X0, const void* X1,
                         int num_sms, cudaStream_t stream, bool pdl) {
  if (p.T <= 0) return cudaSuccess;
  for (int i = 0; i < 2; ++i)
    if (p.K[i] % kMmBK != 0 || p.N[i] % 32 != 0) return cudaErrorNotSupported;
  // tokens per tile: a multiple of 32 up to kMaxNT
  p.NT = (p.T + 31) / 32 * 32;
  if (p.NT > kMaxNT) p.NT = kMaxNT;
  p.xrows = p.T < p.NT ? p.T : p.NT;
  p.ntiles = (p.T + p.NT - 1) / p.NT;
  const void* Ws[2] = {W0, W1};
  const void* Xs[2] = {X0, X1};
  int total = 0;
  for (int i = 0; i < 2; ++i) {
    if (!encode_w8(&p.tw[i], static_cast<const int8_t*>(Ws[i]), p.K[i], p.N[i]) ||
        !encode_x16(&p.tx[i], Xs[i], p.T, p.K[i], p.xrows))
      return cudaErrorInvalidValue;
    p.mt[i] = (p.N[i] + kMmBM - 1) / kMmBM;
    const int nkb = p.K[i] / kMmBK;
    // RAW mode may split K (the sums are added atomically): aim for about
    // one unit per SM when the tiles alone are fewer; HEADS keeps whole K
    int ks = 1;
    const int tiles = p.mt[i] * p.ntiles;
    if (p.raw && tiles < num_sms) ks = (num_sms + tiles - 1) / tiles;
    if (ks > nkb) ks = nkb;
    p.kbps[i] = (nkb + ks - 1) / ks;
    p.ks[i] = (nkb + p.kbps[i] - 1) / p.kbps[i];
    p.nunits[i] = p.N[i] > 0 ? tiles * p.ks[i] : 0;
    // keep the larger operand streaming once: weight tiles fastest when the
    // activations outweigh the weights (their panels then stay in L2)
    p.mfast[i] = (size_t)p.T * p.K[i] * 2 > (size_t)p.K[i] * p.N[i] ? 1 : 0;
    total += p.nunits[i];
  }
  // t / s without a divide: l = ceil(log2 s), m = floor(2^32 (2^l - s) / s) + 1
  {
    const unsigned d = (unsigned)(p.s > 0 ? p.s : 1);
    unsigned l = 0;
    while ((1ull << l) < d) ++l;
    p.s_shift = l;
    p.s_mul = (unsigned)((((1ull << l) - d) << 32) / d + 1);
  }
  const size_t stage = (kWBytes + (size_t)p.NT * 128 + 1023) / 1024 * 1024;
  int S = (int)((kSmemBudget - 1024 - kASlots * (size_t)kABytes - 4 * (size_t)kEpBytes - sizeof(MmShared) - 64) / stage);
  if (S > kMaxStages) S = kMaxStages;
  if (S < 2) return cudaErrorNotSupported;
  p.stages = S;
  const size_t smem = w8mma_smem(p.NT, S);
  const void* fn = p.raw ? (const void*)w8mma_kernel<0> : (const void*)w8mma_kernel<1>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(total < num_sms ? total : num_sms);
  cfg.blockDim = dim3(kMmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  void* args[] = {&p};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace mla
