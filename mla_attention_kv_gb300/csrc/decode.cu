// decode.cu -- fused MLA KV prolog for small token counts (decode).
//
// One cooperative launch (one CTA per SM) performs all seven prolog steps
// of "DeepSeek-V2-Lite-Chat MLA KV Prolog 迁移指南" §背景 for up to
// kDecodeMaxTokens token rows.  At these sizes the work is bound by the
// weight stream (W_kva + W_kvb, 6.5 MB for V2-Lite, 41.8 MB for R1), so the
// kernel is organised around reading every weight byte exactly once, with
// 16-byte coalesced copies, from as many SMs as possible:
//
//   phase A  kv_a_proj split-K: the [hidden, 576] weight is cut into
//            (KB rows x 64 columns) tiles, one or more per CTA; each CTA
//            multiplies its tile by the matching hidden columns on the
//            tensor cores (mma.sync m16n8k16, tokens as M) and writes fp32
//            partial sums [KC, T, 576] to the workspace.  At kernel start
//            every CTA also issues an L2 prefetch of its W_kvb slice, so
//            the whole weight set is in flight at once.
//   barrier  grid-wide, bounded wait (the RMSNorm needs the full row).
//   phase R  one CTA per token row: fixed-order sum of the KC partials
//            (deterministic), split (step 2), RMSNorm in fp32 (step 3),
//            the normalised row rounded once to the I/O dtype into the
//            workspace, RoPE of k_pe (step 6) stored straight to k_pe.
//   barrier
//   phase B  kv_b_proj split-N: each CTA owns a contiguous range of 8-column
//            groups of W_kvb, streams it through shared memory (3-stage
//            cp.async pipeline) and multiplies by the normalised rows; the
//            epilogue does the reshape/split (step 5) and the head-major
//            stores (step 7) directly from the accumulators.
#include "common.cuh"
#include "internal.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSubK = 64;          // K rows per pipeline stage
constexpr int kStagesA = 6;
constexpr int kStagesB = 3;
constexpr int kPitchA = 144;       // bytes per smem row of a 64-element tile (odd multiple of 16)
constexpr int kPitchN = 1040;      // bytes per smem row of a 512-element latent row
constexpr int kMaxMT = kDecodeMaxTokens / 16;
constexpr int kMaxPairs = 16;      // phase-B (m-tile, column group) pairs per warp

__host__ __device__ constexpr int odd16_pitch(int bytes) {
  int p = (bytes + 15) / 16 * 16;
  if (((p / 16) & 1) == 0) p += 16;
  return p;
}

__device__ __forceinline__ int col_group_begin(int cta, int ngroups, int grid) {
  return (int)(((long long)cta * ngroups) / grid);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(DecodeParams p) {
  using E = Elem<T>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, cta = blockIdx.x;
  const int TT = p.TT;
  const int MT = (TT + 15) >> 4;
  const int H = p.heads;
  const int NB = H * kHeadCols;      // kv_b columns
  const int NG = NB / 8;             // 8-column groups
  const int g0 = col_group_begin(cta, NG, G), g1 = col_group_begin(cta + 1, NG, G);
  const int ng = g1 - g0;
  const int col0 = g0 * 8;
  const T* __restrict__ hid = static_cast<const T*>(p.hidden) + (size_t)p.t0 * p.hidden_dim;
  const T* __restrict__ Wa = static_cast<const T*>(p.W_kva);
  const T* __restrict__ Wb = static_cast<const T*>(p.W_kvb);

  // ---- warm L2 with this CTA's W_kvb slice (rows of ng*16 bytes)
  if (ng > 0) {
    for (int r = tid; r < kRank; r += kThreads)
      prefetch_l2_bulk(Wb + (size_t)r * NB + col0, (uint32_t)ng * 16u);
  }

  // ================================================================ phase A
  {
    const int units = p.KC * (kNa / 64);
    const int subs_per_unit = p.KB / kSubK;
    const int my_units = (units > cta) ? (units - cta + G - 1) / G : 0;
    const int nsub = my_units * subs_per_unit;
    const int stage_bytes = 2 * 64 * kPitchA;
    const int rows_x = MT * 16;

    auto load_sub = [&](int i) {
      const int u = cta + (i / subs_per_unit) * G;
      const int kc = u / (kNa / 64), nc = u % (kNa / 64);
      const int k0 = kc * p.KB + (i % subs_per_unit) * kSubK;
      unsigned char* st = smem + (i % kStagesA) * stage_bytes;
      const uint32_t w_s = smem_u32(st), x_s = smem_u32(st + 64 * kPitchA);
      // W tile: 64 rows x 64 cols = 64 x 8 chunks of 16 B
      for (int c = tid; c < 64 * 8; c += kThreads) {
        const int r = c >> 3, ch = c & 7;
        cp_async16(w_s + r * kPitchA + ch * 16, Wa + (size_t)(k0 + r) * kNa + nc * 64 + ch * 8);
      }
      // hidden columns k0..k0+63 of the token rows (zero rows past TT)
      for (int c = tid; c < rows_x * 8; c += kThreads) {
        const int r = c >> 3, ch = c & 7;
        const int rr = r < TT ? r : 0;
        cp_async16(x_s + r * kPitchA + ch * 16, hid + (size_t)rr * p.hidden_dim + k0 + ch * 8,
                   r < TT ? 16 : 0);
      }
    };

    float acc[kMaxMT][4];
#pragma unroll
    for (int m = 0; m < kMaxMT; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;

#pragma unroll 1
    for (int s = 0; s < kStagesA - 1; ++s) {
      if (s < nsub) load_sub(s);
      cp_async_commit();
    }
#pragma unroll 1
    for (int i = 0; i < nsub; ++i) {
      cp_async_wait<kStagesA - 2>();
      __syncthreads();
      if (i + kStagesA - 1 < nsub) load_sub(i + kStagesA - 1);
      cp_async_commit();
      const unsigned char* st = smem + (i % kStagesA) * stage_bytes;
      const uint32_t w_s = smem_u32(st), x_s = smem_u32(st + 64 * kPitchA);
#pragma unroll
      for (int kk = 0; kk < kSubK / 16; ++kk) {
        uint32_t b0, b1;
        ldsm_x2_trans(w_s + (kk * 16 + (lane & 15)) * kPitchA + warp * 16, b0, b1);
#pragma unroll
        for (int m = 0; m < kMaxMT; ++m) {
          if (m < MT) {
            uint32_t a[4];
            ldsm_x4(x_s + (m * 16 + (lane & 15)) * kPitchA + (kk * 16 + (lane >> 4) * 8) * 2, a[0],
                    a[1], a[2], a[3]);
            mma16816<E::kBf16>(acc[m], a, b0, b1);
          }
        }
      }
      if ((i % subs_per_unit) == subs_per_unit - 1) {
        const int u = cta + (i / subs_per_unit) * G;
        const int kc = u / (kNa / 64), nc = u % (kNa / 64);
        float* P = p.partials + (size_t)kc * kDecodeMaxTokens * kNa;
        const int col = nc * 64 + warp * 8 + 2 * (lane & 3);
#pragma unroll
        for (int m = 0; m < kMaxMT; ++m) {
          const int r0 = m * 16 + (lane >> 2);
          if (m < MT) {
            if (r0 < TT) *reinterpret_cast<float2*>(P + (size_t)r0 * kNa + col) = make_float2(acc[m][0], acc[m][1]);
            if (r0 + 8 < TT) *reinterpret_cast<float2*>(P + (size_t)(r0 + 8) * kNa + col) = make_float2(acc[m][2], acc[m][3]);
          }
          acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
        }
      }
    }
    cp_async_wait<0>();
  }

  if (!grid_barrier(p.counters, G, p.budget_ns, p.status)) return;

  // ================================================================ phase R
  {
    __shared__ float red[kWarps];
    T* nrm = static_cast<T*>(p.nrm);
    const T* gam = static_cast<const T*>(p.gamma);
#pragma unroll 1
    for (int t = cta; t < TT; t += G) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (tid < kNa / 4) {
        const float* P = p.partials + (size_t)t * kNa + tid * 4;
#pragma unroll 4
        for (int kc = 0; kc < p.KC; ++kc) {
          const float4 x = __ldcg(reinterpret_cast<const float4*>(P + (size_t)kc * kDecodeMaxTokens * kNa));
          v.x += x.x; v.y += x.y; v.z += x.z; v.w += x.w;
        }
      }
      // step 3: mean of squares over the 512 latent entries (threads 0..127)
      float ss = (tid < kRank / 4) ? (v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w) : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) red[warp] = ss;
      __syncthreads();
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) tot += red[w];
      __syncthreads();
      if (tid < kRank / 4) {
        const float inv = 1.0f / sqrtf(tot / (float)kRank + p.eps);
        const int c = tid * 4;
        const float n0 = v.x * inv * E::to_f(gam[c + 0]);
        const float n1 = v.y * inv * E::to_f(gam[c + 1]);
        const float n2 = v.z * inv * E::to_f(gam[c + 2]);
        const float n3 = v.w * inv * E::to_f(gam[c + 3]);
        uint2 pk = make_uint2(E::pack(n0, n1), E::pack(n2, n3));
        *reinterpret_cast<uint2*>(nrm + (size_t)t * kRank + c) = pk;
      } else if (tid < kNa / 4) {
        // step 6: RoPE; this thread holds raw k_pe columns 4i..4i+3, i.e.
        // rotation pairs j = 2i and 2i+1 -> outputs j, j+32 (de-interleaved)
        const int i = tid - kRank / 4;
        const int tg = p.t0 + t;
        int pos = p.positions[tg];
        if (pos < 0 || pos >= p.max_pos) {
          atomicOr(p.status, kStatusBadPosition);
          pos = pos < 0 ? 0 : p.max_pos - 1;
        }
        const float* cr = p.cos_t + (size_t)pos * kRope;
        const float* sr = p.sin_t + (size_t)pos * kRope;
        const int j0 = 2 * i, j1 = 2 * i + 1;
        const float o0 = v.x * cr[j0] - v.y * sr[j0];
        const float o1 = v.z * cr[j1] - v.w * sr[j1];
        const float o2 = v.y * cr[j0 + 32] + v.x * sr[j0 + 32];
        const float o3 = v.w * cr[j1 + 32] + v.z * sr[j1 + 32];
        T* kp = static_cast<T*>(p.k_pe) + (size_t)tg * kRope;
        *reinterpret_cast<uint32_t*>(kp + j0) = E::pack(o0, o1);
        *reinterpret_cast<uint32_t*>(kp + j0 + 32) = E::pack(o2, o3);
      }
    }
  }

  if (!grid_barrier(p.counters, G, p.budget_ns, p.status)) return;

  // ================================================================ phase B
  if (ng > 0) {
    const int pitchB = odd16_pitch(ng * 16);
    unsigned char* nrm_s = smem;
    unsigned char* wst = smem + kDecodeMaxTokens * kPitchN;
    float* redbuf = reinterpret_cast<float*>(wst + kStagesB * kSubK * odd16_pitch(((NG + G - 1) / G) * 16));
    const uint32_t nrm_u = smem_u32(nrm_s);
    const T* nrm = static_cast<const T*>(p.nrm);
    const int rows_x = MT * 16;
    // normalised latent rows (zero rows past TT)
    for (int c = tid; c < rows_x * 64; c += kThreads) {
      const int r = c >> 6, ch = c & 63;
      const int rr = r < TT ? r : 0;
      cp_async16(nrm_u + r * kPitchN + ch * 16, nrm + (size_t)rr * kRank + ch * 8, r < TT ? 16 : 0);
    }
    auto load_w = [&](int kb) {
      const uint32_t dst = smem_u32(wst + (kb % kStagesB) * kSubK * pitchB);
      const int nch = ng;  // 16-byte chunks per row
      for (int c = tid; c < kSubK * nch; c += kThreads) {
        const int r = c / nch, ch = c - r * nch;
        cp_async16(dst + r * pitchB + ch * 16, Wb + (size_t)(kb * kSubK + r) * NB + col0 + ch * 8);
      }
    };
    // work split: pairs (m-tile, column group); with few pairs the k16 steps
    // of each stage are also split across warps and reduced at the end
    const int npairs = MT * ng;
    int ksplit = 1;
    while (ksplit < 4 && npairs * ksplit * 2 <= kWarps) ksplit *= 2;
    const int wpg = kWarps / ksplit;   // warps per k-slice
    const int kslice = warp / wpg, pbase = warp % wpg;
    float acc[kMaxPairs][4];
#pragma unroll
    for (int q = 0; q < kMaxPairs; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;

    load_w(0);
    cp_async_commit();
    load_w(1);
    cp_async_commit();
    constexpr int kSteps = kRank / kSubK;
#pragma unroll 1
    for (int kb = 0; kb < kSteps; ++kb) {
      cp_async_wait<1>();
      __syncthreads();
      if (kb + 2 < kSteps) load_w(kb + 2);
      cp_async_commit();
      const uint32_t w_s = smem_u32(wst + (kb % kStagesB) * kSubK * pitchB);
#pragma unroll
      for (int kk = 0; kk < kSubK / 16; ++kk) {
        if ((kk % ksplit) != kslice) continue;
#pragma unroll
        for (int q = 0; q < kMaxPairs; ++q) {
          const int pr = pbase + q * wpg;
          if (pr < npairs) {
            const int m = pr % MT, gi = pr / MT;
            uint32_t b0, b1, a[4];
            ldsm_x2_trans(w_s + (kk * 16 + (lane & 15)) * pitchB + gi * 16, b0, b1);
            ldsm_x4(nrm_u + (m * 16 + (lane & 15)) * kPitchN + (kb * kSubK + kk * 16 + (lane >> 4) * 8) * 2,
                    a[0], a[1], a[2], a[3]);
            mma16816<E::kBf16>(acc[q], a, b0, b1);
          }
        }
      }
    }
    cp_async_wait<0>();
    if (ksplit > 1) {
      // each warp holds at most one pair when ksplit > 1
      if (kslice > 0 && pbase < npairs) {
        float* dst = redbuf + ((kslice * wpg + pbase) * 32 + lane) * 4;
        dst[0] = acc[0][0]; dst[1] = acc[0][1]; dst[2] = acc[0][2]; dst[3] = acc[0][3];
      }
      __syncthreads();
      if (kslice == 0 && pbase < npairs) {
        for (int ks = 1; ks < ksplit; ++ks) {
          const float* src = redbuf + ((ks * wpg + pbase) * 32 + lane) * 4;
          acc[0][0] += src[0]; acc[0][1] += src[1]; acc[0][2] += src[2]; acc[0][3] += src[3];
        }
      }
    }
    if (kslice == 0) {
      T* kn = static_cast<T*>(p.k_nope);
      T* vv = static_cast<T*>(p.value);
#pragma unroll
      for (int q = 0; q < kMaxPairs; ++q) {
        const int pr = pbase + q * wpg;
        if (pr < npairs) {
          const int m = pr % MT, gi = pr / MT;
          const int j = col0 + gi * 8 + 2 * (lane & 3);
          const int hh = j / kHeadCols, e = j % kHeadCols;
          T* base = (e < kNope) ? kn : vv;
          const int ee = (e < kNope) ? e : e - kNope;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int r = m * 16 + (lane >> 2) + half * 8;
            if (r < TT) {
              const int tg = p.t0 + r;
              const int bi = tg / p.s, si = tg - bi * p.s;
              T* dst = base + (((size_t)bi * H + hh) * p.s + si) * kNope + ee;
              *reinterpret_cast<uint32_t*>(dst) = E::pack(acc[q][2 * half], acc[q][2 * half + 1]);
            }
          }
        }
      }
    }
  }
}

}  // namespace

bool decode_plan(int hidden, int heads, int num_sms, DecodePlan* plan) {
  if (hidden % 64 != 0 || heads < 1 || num_sms < 1) return false;
  const int G = num_sms;
  // split-K chunk: the smallest multiple of 64 dividing hidden that gives at
  // most one (chunk x 64-column) unit per CTA; fewer chunks means fewer
  // partial rows to reduce after the barrier
  int KB = hidden;
  for (int kb = 64; kb <= hidden; kb += 64) {
    if (hidden % kb == 0 && (hidden / kb) * (kNa / 64) <= G) {
      KB = kb;
      break;
    }
  }
  const int KC = hidden / KB;
  const int NG = heads * kHeadCols / 8;
  const int ngmax = (NG + G - 1) / G;
  // phase-B pairs per warp must fit the register tile
  if ((kMaxMT * ngmax + kWarps - 1) / kWarps > kMaxPairs) return false;
  const size_t smemA = (size_t)kStagesA * 2 * 64 * kPitchA;
  const size_t smemB = (size_t)kDecodeMaxTokens * kPitchN +
                       (size_t)kStagesB * kSubK * odd16_pitch(ngmax * 16) +
                       (size_t)kWarps * 32 * 4 * sizeof(float);
  const size_t smem = smemA > smemB ? smemA : smemB;
  if (smem > 227 * 1024) return false;
  plan->grid = G;
  plan->KB = KB;
  plan->KC = KC;
  plan->smem = smem;
  plan->partial_floats = (size_t)KC * kDecodeMaxTokens * kNa;
  return true;
}

cudaError_t decode_launch(bool bf16, const DecodePlan& plan, const DecodeParams& p,
                          cudaStream_t stream) {
  const void* fn = bf16 ? (const void*)decode_kernel<__nv_bfloat16> : (const void*)decode_kernel<__half>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  DecodeParams pp = p;
  void* args[] = {&pp};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace mla
