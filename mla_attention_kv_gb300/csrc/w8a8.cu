// w8a8.cu -- W8A8 full MLA prolog (Q side + KV side): int8 weights with one
// fp32 scale per output channel, per-token dynamic int8 activations, exact
// int32 accumulation, bf16 outputs.
//
// The W8A8 weight mode is the one "DeepSeek-R1或Kimi-K2模型在NPU实现高性能推理"
// §权重转换 converts to (w8a8c16 / w8a8c8); the fused MLA prolog it feeds is
// the enable_mla_prolog switch of §推理执行.  The arithmetic, in order:
//   1. quantise each hidden row: amax = max|x|, inv = 127/amax,
//      q = clamp(rint(x*inv), -127, 127), s_x = amax/127 (each one IEEE fp32
//      operation; amax = 0 gives q = 0, s_x = 0)
//   2. q_a_proj and kv_a_proj: int8 x int8 -> int32 GEMMs (exact), then
//      y = (float)acc * s_x * s_w
//   3. RMSNorm of the q latent (gamma_q) and of compressed_kv (gamma_kv);
//      RoPE of k_pe -> output
//   4. requantise both normalised rows as in 1
//   5. q_b_proj -> [H, 192] -> q_nope (0:128), RoPE(q_pe) (128:192)
//   6. kv_b_proj -> [H, 256] -> k_nope, value
//
// Integer GEMMs run on mma.sync m16n8k32 (s8 x s8 -> s32): the tcgen05 int8
// kind is not available on sm_103a.  Weights arrive [in, out] (N
// contiguous); the kernel transposes each B tile in registers with byte
// permutes so the tensor-core operand is K-contiguous.  When there are too
// few output tiles to fill the GPU the K range is split across CTAs and
// the int32 partials are added with atomics, which is exact and
// order-independent.
#include <type_traits>
#include <utility>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "tma.h"

namespace mla {
namespace {

constexpr int kGThreads = 128;  // 4 warps, 2 x 2 over a 64 x 64 tile
constexpr int kGemvMaxRows = 8; // M up to this takes the dp4a weight-streaming path
constexpr int kGBM = 64, kGBN = 64, kGBK = 32;
constexpr int kPitchA8 = 48;    // smem row pitch (bytes) of a [64 x 32] int8 tile: odd multiple of 16
constexpr int kPitchBt = 48;    // smem row pitch of the transposed [64 n x 32 k] tile

// C[M, N] (+)= A[M, K] * W[K, N]; int8 in, int32 out with leading dim ldc.
// Grid: (N / 64, ceil(M / 64), splits); split z covers K chunk [k_begin, k_end).
__global__ void __launch_bounds__(kGThreads) gemm_s8_kernel(const int8_t* __restrict__ A,
                                                            const int8_t* __restrict__ W, int M,
                                                            int K, int N, int32_t* __restrict__ C,
                                                            int ldc, int kchunk, int atomic) {
  __shared__ __align__(16) unsigned char sA[2][kGBM * kPitchA8];
  __shared__ __align__(16) unsigned char sB[2][kGBN * kPitchBt];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n0 = blockIdx.x * kGBN, m0 = blockIdx.y * kGBM;
  const int kb = blockIdx.z * kchunk;
  const int ke = min(K, kb + kchunk);
  if (kb >= ke) return;
  const int nsteps = (ke - kb) / kGBK;
  const int wm = warp >> 1, wn = warp & 1;  // warp tile rows wm*32, cols wn*32

  // A: 64 rows x 32 bytes = 128 x 16 B (one per thread)
  auto load_a = [&](int stage, int k0) {
    const int r = tid >> 1, ch = tid & 1;
    const int gr = m0 + r;
    cp_async16(smem_u32(&sA[stage][r * kPitchA8 + ch * 16]),
               A + (size_t)(gr < M ? gr : 0) * K + k0 + ch * 16, gr < M ? 16 : 0);
  };
  // B: 32 k rows x 64 n = thread loads 4 k rows x 16 n (4 x 16 B), i.e.
  // 8 k-groups x 4 n-groups = 32 threads... use all 128: k-group = tid>>2 (8 groups of 4 rows)
  // is too few; instead each thread loads one 16 B piece (k row, 16 n) and
  // threads of a quad exchange via shuffles.  Simpler: 32 threads x 4 rows.
  uint4 breg[4];
  auto fetch_b = [&](int k0) {
    if (tid < 32) {
      const int kg = tid >> 2, ng = tid & 3;  // k rows 4kg..4kg+3, n 16ng..16ng+15
#pragma unroll
      for (int i = 0; i < 4; ++i)
        breg[i] = __ldg(reinterpret_cast<const uint4*>(W + (size_t)(k0 + 4 * kg + i) * N + n0 + 16 * ng));
    }
  };
  auto store_b = [&](int stage) {
    if (tid < 32) {
      const int kg = tid >> 2, ng = tid & 3;
      const uint32_t* w0 = reinterpret_cast<const uint32_t*>(&breg[0]);
      const uint32_t* w1 = reinterpret_cast<const uint32_t*>(&breg[1]);
      const uint32_t* w2 = reinterpret_cast<const uint32_t*>(&breg[2]);
      const uint32_t* w3 = reinterpret_cast<const uint32_t*>(&breg[3]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // n 4j..4j+3 within the 16
        const uint32_t lo01 = __byte_perm(w0[j], w1[j], 0x5140), lo23 = __byte_perm(w2[j], w3[j], 0x5140);
        const uint32_t hi01 = __byte_perm(w0[j], w1[j], 0x7362), hi23 = __byte_perm(w2[j], w3[j], 0x7362);
        const uint32_t t0 = __byte_perm(lo01, lo23, 0x5410), t1 = __byte_perm(lo01, lo23, 0x7632);
        const uint32_t t2 = __byte_perm(hi01, hi23, 0x5410), t3 = __byte_perm(hi01, hi23, 0x7632);
        const int n = 16 * ng + 4 * j;
        unsigned char* base = &sB[stage][0] + 4 * kg;
        *reinterpret_cast<uint32_t*>(base + (n + 0) * kPitchBt) = t0;
        *reinterpret_cast<uint32_t*>(base + (n + 1) * kPitchBt) = t1;
        *reinterpret_cast<uint32_t*>(base + (n + 2) * kPitchBt) = t2;
        *reinterpret_cast<uint32_t*>(base + (n + 3) * kPitchBt) = t3;
      }
    }
  };

  int acc[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0;

  load_a(0, kb);
  cp_async_commit();
  fetch_b(kb);
  store_b(0);
  for (int s = 0; s < nsteps; ++s) {
    const int cur = s & 1;
    if (s + 1 < nsteps) {
      load_a(cur ^ 1, kb + (s + 1) * kGBK);
      fetch_b(kb + (s + 1) * kGBK);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    uint32_t a[2][4], bfr[4][2];
#pragma unroll
    for (int i = 0; i < 2; ++i)
      ldsm_x4(smem_u32(&sA[cur][(wm * 32 + i * 16 + (lane & 15)) * kPitchA8 + (lane >> 4) * 16]), a[i][0],
              a[i][1], a[i][2], a[i][3]);
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      uint32_t r0, r1, r2, r3;
      // matrices: (n j*8.., k 0-15), (n j*8.., k 16-31), (n (j+1)*8.., k 0-15), (n (j+1)*8.., k 16-31)
      const int nrow = wn * 32 + j * 8 + (lane & 7) + ((lane >> 4) << 3);
      const int kofs = ((lane >> 3) & 1) * 16;
      ldsm_x4(smem_u32(&sB[cur][nrow * kPitchBt + kofs]), r0, r1, r2, r3);
      bfr[j][0] = r0; bfr[j][1] = r1; bfr[j + 1][0] = r2; bfr[j + 1][1] = r3;
    }
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) mma16832_s8(acc[i][j], a[i], bfr[j][0], bfr[j][1]);
    __syncthreads();
    if (s + 1 < nsteps) store_b(cur ^ 1);
  }
  cp_async_wait<0>();
  // epilogue
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = n0 + wn * 32 + j * 8 + 2 * (lane & 3);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int row = m0 + wm * 32 + i * 16 + (lane >> 2) + hf * 8;
        if (row < M) {
          int32_t* c = C + (size_t)row * ldc + col;
          if (atomic) {
            atomicAdd(c, acc[i][j][2 * hf]);
            atomicAdd(c + 1, acc[i][j][2 * hf + 1]);
          } else {
            *reinterpret_cast<int2*>(c) = make_int2(acc[i][j][2 * hf], acc[i][j][2 * hf + 1]);
          }
        }
      }
    }
  }
}

// Block-wide max / sum over 256 threads.
template <bool kMax>
__device__ __forceinline__ float block_reduce(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = kMax ? fmaxf(v, w) : v + w;
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = kMax ? 0.f : 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r = kMax ? fmaxf(r, scratch[w]) : r + scratch[w];
  return r;
}

// Quantise a float32 value with the fixed fp32 operation sequence.
__device__ __forceinline__ int8_t q8(float x, float inv) {
  float r = rintf(__fmul_rn(x, inv));
  r = fminf(fmaxf(r, -127.f), 127.f);
  return (int8_t)(int)r;
}

// Rows of at most this many columns are held in registers by quant_rows_kernel.
constexpr int kQuantRegCols = 256 * 8 * 4;

// One CTA (256 threads) per row of a bf16 matrix [rows, cols] -> codes +
// scale.  The codes are stored as int8, or (Q = __half) as the fp16 values
// of the same integers (the tensor-core GEMM operand; exact for |q| <= 127).
template <typename Q>
__global__ void __launch_bounds__(256) quant_rows_kernel(const __nv_bfloat16* __restrict__ x, int cols,
                                                         Q* __restrict__ q,
                                                         float* __restrict__ scale) {
  __shared__ float scratch[8];
  // the next kernel of the chain may launch now (it waits for this one
  // before reading its codes)
  grid_dep_launch_dependents();
  const int row = blockIdx.x;
  const __nv_bfloat16* xr = x + (size_t)row * cols;
  // 8 values per 16-byte vector, vector k of thread i at column (i + 256 k) * 8
  auto codes = [&](const uint4& v, int c, float inv) {
    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
    if constexpr (std::is_same<Q, int8_t>::value) {
      char4 lo, hi;
      lo.x = q8(__bfloat162float(e[0]), inv); lo.y = q8(__bfloat162float(e[1]), inv);
      lo.z = q8(__bfloat162float(e[2]), inv); lo.w = q8(__bfloat162float(e[3]), inv);
      hi.x = q8(__bfloat162float(e[4]), inv); hi.y = q8(__bfloat162float(e[5]), inv);
      hi.z = q8(__bfloat162float(e[6]), inv); hi.w = q8(__bfloat162float(e[7]), inv);
      *reinterpret_cast<char4*>(q + (size_t)row * cols + c) = lo;
      *reinterpret_cast<char4*>(q + (size_t)row * cols + c + 4) = hi;
    } else {
      __align__(16) __half h[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = __int2half_rn((int)q8(__bfloat162float(e[i]), inv));
      *reinterpret_cast<uint4*>(q + (size_t)row * cols + c) = *reinterpret_cast<const uint4*>(h);
    }
  };
  auto vmax = [](const uint4& v, float m) {
    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(__bfloat162float(e[i])));
    return m;
  };
  float amax = 0.f;
  if (cols <= kQuantRegCols) {
    // the whole row in registers: every load issued at once, read once
    uint4 v[kQuantRegCols / 2048];
#pragma unroll
    for (int k = 0; k < kQuantRegCols / 2048; ++k) {
      const int c = (threadIdx.x + 256 * k) * 8;
      v[k] = c < cols ? *reinterpret_cast<const uint4*>(xr + c) : make_uint4(0, 0, 0, 0);
      amax = vmax(v[k], amax);
    }
    amax = block_reduce<true>(amax, scratch);
    const float inv = amax > 0.f ? __fdiv_rn(127.0f, amax) : 0.f;
#pragma unroll
    for (int k = 0; k < kQuantRegCols / 2048; ++k) {
      const int c = (threadIdx.x + 256 * k) * 8;
      if (c < cols) codes(v[k], c, inv);
    }
  } else {
    for (int c = threadIdx.x * 8; c < cols; c += 256 * 8)
      amax = vmax(*reinterpret_cast<const uint4*>(xr + c), amax);
    amax = block_reduce<true>(amax, scratch);
    const float inv = amax > 0.f ? __fdiv_rn(127.0f, amax) : 0.f;
    for (int c = threadIdx.x * 8; c < cols; c += 256 * 8) codes(*reinterpret_cast<const uint4*>(xr + c), c, inv);
  }
  if (threadIdx.x == 0) scale[row] = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f;
}

// 16-byte vectors of a [q_rank + 576] row per thread of a 256-thread CTA:
// every global load of a row is issued before the first one is used.
constexpr int kNormVec = kW8MaxNormCols / 4 / 256;

// Per-token normalisation inputs that do not depend on the GEMM: the
// weight scales of the q_a / kv_a columns, gamma_q, gamma_kv (as floats).
// q_rank % 64 == 0, so every piece is a whole number of 16-byte vectors.
__device__ __forceinline__ void norm_load_inputs(const W8Params& p, float* colsc, float* gq,
                                                 float* gk) {
  const int rq = p.q_rank, nq4 = rq / 4, na4 = (rq + kNa) / 4;
  const int nq8 = rq / 8, ng8 = (rq + kRank) / 8;
  float4 v[kNormVec];
  uint4 g[kNormVec / 2];
#pragma unroll
  for (int k = 0; k < kNormVec; ++k) {
    const int i = threadIdx.x + 256 * k;
    v[k] = i < nq4 ? reinterpret_cast<const float4*>(p.sW_qa)[i]
                   : (i < na4 ? reinterpret_cast<const float4*>(p.sW_kva)[i - nq4] : make_float4(0.f, 0.f, 0.f, 0.f));
  }
#pragma unroll
  for (int k = 0; k < kNormVec / 2; ++k) {
    const int i = threadIdx.x + 256 * k;
    g[k] = i < nq8 ? reinterpret_cast<const uint4*>(p.gamma_q)[i]
                   : (i < ng8 ? reinterpret_cast<const uint4*>(p.gamma_kv)[i - nq8] : make_uint4(0u, 0u, 0u, 0u));
  }
#pragma unroll
  for (int k = 0; k < kNormVec; ++k) {
    const int i = threadIdx.x + 256 * k;
    if (i < na4) reinterpret_cast<float4*>(colsc)[i] = v[k];
  }
#pragma unroll
  for (int k = 0; k < kNormVec / 2; ++k) {
    const int i = threadIdx.x + 256 * k;
    if (i < ng8) {
      const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&g[k]);
      float* d = i < nq8 ? gq + 8 * i : gk + 8 * (i - nq8);
#pragma unroll
      for (int j = 0; j < 8; ++j) d[j] = __bfloat162float(e[j]);
    }
  }
}

// cos / sin of token t's position into rope[0, 64) / rope[64, 128) (threads
// 0..127); an out-of-range position is clamped and recorded.
__device__ __forceinline__ void rope_load(const W8Params& p, int t, float* rope) {
  if (threadIdx.x < 2 * kRope) {
    int pos = p.positions[t];
    if (pos < 0 || pos >= p.max_pos) {
      if (threadIdx.x == 0) atomicOr(p.status, kStatusBadPosition);
      pos = pos < 0 ? 0 : p.max_pos - 1;
    }
    const int j = threadIdx.x & (kRope - 1);
    rope[threadIdx.x] = (threadIdx.x < kRope ? p.cos_t : p.sin_t)[(size_t)pos * kRope + j];
  }
}

// One token row (all 256 threads of the CTA): dequantise the [q_rank + 576]
// accumulator row a (scale s), RMSNorm of the q latent and of compressed_kv,
// requantise both (codes to q_out / c_out, scales to *s1_out / *s2_out, any
// address space), RoPE of k_pe to kpe_out (skipped when null).
__device__ void norm_row(const int32_t* a, float s, const W8Params& p, float* yrow,
                         const float* colsc, const float* gq, const float* gk, const float* rope,
                         float* scratch, int8_t* q_out, float* s1_out, int8_t* c_out, float* s2_out,
                         __nv_bfloat16* kpe_out, __half* qh_out = nullptr, __half* ch_out = nullptr) {
  const int rq = p.q_rank, na4 = (rq + kNa) / 4;
  int4 av[kNormVec];
#pragma unroll
  for (int k = 0; k < kNormVec; ++k) {
    const int i = threadIdx.x + 256 * k;
    av[k] = i < na4 ? reinterpret_cast<const int4*>(a)[i] : make_int4(0, 0, 0, 0);
  }
#pragma unroll
  for (int k = 0; k < kNormVec; ++k) {
    const int i = threadIdx.x + 256 * k;
    if (i < na4) {
      const float4 c = reinterpret_cast<const float4*>(colsc)[i];
      float4 y;
      y.x = __fmul_rn(__fmul_rn((float)av[k].x, s), c.x);
      y.y = __fmul_rn(__fmul_rn((float)av[k].y, s), c.y);
      y.z = __fmul_rn(__fmul_rn((float)av[k].z, s), c.z);
      y.w = __fmul_rn(__fmul_rn((float)av[k].w, s), c.w);
      reinterpret_cast<float4*>(yrow)[i] = y;
    }
  }
  __syncthreads();
  // q latent
  float ss = 0.f;
  for (int c = threadIdx.x; c < rq; c += 256) ss += yrow[c] * yrow[c];
  ss = block_reduce<false>(ss, scratch);
  const float invq = 1.0f / sqrtf(ss / (float)rq + p.eps);
  float amax = 0.f;
  for (int c = threadIdx.x; c < rq; c += 256) {
    const float v = yrow[c] * invq * gq[c];
    yrow[c] = v;
    amax = fmaxf(amax, fabsf(v));
  }
  amax = block_reduce<true>(amax, scratch);
  {
    const float inv = amax > 0.f ? __fdiv_rn(127.0f, amax) : 0.f;
    for (int c = threadIdx.x; c < rq; c += 256) {
      const int8_t v = q8(yrow[c], inv);
      q_out[c] = v;
      if (qh_out) qh_out[c] = __int2half_rn((int)v);
    }
    if (threadIdx.x == 0) *s1_out = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f;
  }
  // compressed_kv
  float* ck = yrow + rq;
  ss = 0.f;
  for (int c = threadIdx.x; c < kRank; c += 256) ss += ck[c] * ck[c];
  ss = block_reduce<false>(ss, scratch);
  const float invk = 1.0f / sqrtf(ss / (float)kRank + p.eps);
  amax = 0.f;
  float nv[2];
  for (int i = 0; i < 2; ++i) {
    const int c = threadIdx.x + i * 256;
    nv[i] = ck[c] * invk * gk[c];
    amax = fmaxf(amax, fabsf(nv[i]));
  }
  amax = block_reduce<true>(amax, scratch);
  {
    const float inv = amax > 0.f ? __fdiv_rn(127.0f, amax) : 0.f;
    for (int i = 0; i < 2; ++i) {
      const int8_t v = q8(nv[i], inv);
      c_out[threadIdx.x + i * 256] = v;
      if (ch_out) ch_out[threadIdx.x + i * 256] = __int2half_rn((int)v);
    }
    if (threadIdx.x == 0) *s2_out = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f;
  }
  // RoPE of k_pe (raw columns 512..575 of the kv_a output)
  if (kpe_out && threadIdx.x < 32) {
    const float* kp = ck + kRank;
    const int j = threadIdx.x;
    const float a0 = kp[2 * j], b0 = kp[2 * j + 1];
    const float* cr = rope;
    const float* sr = rope + kRope;
    kpe_out[j] = __float2bfloat16_rn(a0 * cr[j] - b0 * sr[j]);
    kpe_out[j + 32] = __float2bfloat16_rn(b0 * cr[j + 32] + a0 * sr[j + 32]);
  }
  __syncthreads();  // yrow is reused by the next row
}

// Per token (prefill sizes): norm_row on one accumulator row per CTA, which
// it leaves zeroed.  Shared memory: the row [q_rank + 576] | its weight
// scales [q_rank + 576] | gamma_q [q_rank] | gamma_kv [512] | cos, sin [2][64].
__host__ __device__ constexpr size_t norm_smem(int q_rank) {
  return (size_t)(2 * (q_rank + kNa) + q_rank + kRank + 2 * kRope) * sizeof(float);
}

__global__ void __launch_bounds__(256) norm_quant_kernel(int32_t* __restrict__ acc1,
                                                         const float* __restrict__ sx,
                                                         W8Params p, W8Workspace w) {
  extern __shared__ float yrow[];
  __shared__ float scratch[8];
  const int t = blockIdx.x;
  const int rq = p.q_rank, na = rq + kNa;
  float* colsc = yrow + na;
  float* gq = colsc + na;
  float* gk = gq + rq;
  float* rope = gk + kRank;
  // launched with the programmatic dependency: the caller's inputs (scales,
  // gammas, positions, cos/sin) are read while the GEMM before runs; its
  // accumulator rows and the row scales only after it
  grid_dep_launch_dependents();
  norm_load_inputs(p, colsc, gq, gk);
  rope_load(p, t, rope);
  grid_dep_wait();
  int32_t* a = acc1 + (size_t)t * na;
  norm_row(a, sx[t], p, yrow, colsc, gq, gk, rope, scratch, w.q1 + (size_t)t * rq, w.s1 + t,
           w.c1 + (size_t)t * kRank, w.s2 + t,
           static_cast<__nv_bfloat16*>(p.k_pe) + (size_t)t * kRope, w.q1h + (size_t)t * rq,
           w.c1h + (size_t)t * kRank);
  // leave the accumulator row zeroed (the decode-size chain adds into it),
  // after copying it out when the accumulators are captured
  if (p.cap_a)
    for (int c = threadIdx.x; c < na; c += 256) p.cap_a[(size_t)t * na + c] = a[c];
  for (int c = threadIdx.x; c < na; c += 256) a[c] = 0;
}

// Prefill sizes: the same per-token steps as norm_quant_kernel with one warp
// per token row (8 rows per CTA, warp-level reductions only), so that the
// per-column inputs (weight scales, gammas) are read once per 8 rows.
// Shared memory: column scales [q_rank + 576] | gamma_q [q_rank] | gamma_kv
// [512] | per warp: its dequantised row [q_rank + 576].
constexpr int kNormRowsPerCta = 8;
__host__ __device__ constexpr size_t norm_warp_smem(int q_rank) {
  return (size_t)((q_rank + kNa) + q_rank + kRank + kNormRowsPerCta * (q_rank + kNa)) * sizeof(float);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__global__ void __launch_bounds__(256) norm_quant_warp_kernel(int32_t* __restrict__ acc1,
                                                              const float* __restrict__ sx,
                                                              W8Params p, W8Workspace w) {
  extern __shared__ float smf[];
  const int rq = p.q_rank, na = rq + kNa;
  float* colsc = smf;
  float* gq = colsc + na;
  float* gk = gq + rq;
  norm_load_inputs(p, colsc, gq, gk);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kNormRowsPerCta + warp;
  if (t >= p.T) return;
  float* y = gk + kRank + (size_t)warp * na;
  int32_t* a = acc1 + (size_t)t * na;
  const float s = sx[t];
  // the row in pieces of 8 int4 per lane, every load of a piece issued
  // before the first is used (one memory round trip per piece)
  const int n4 = na / 4;
  for (int b0 = 0; b0 < n4; b0 += 32 * 8) {
    int4 av[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int idx = b0 + lane + 32 * i;
      av[i] = idx < n4 ? reinterpret_cast<const int4*>(a)[idx] : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int idx = b0 + lane + 32 * i;
      if (idx >= n4) continue;
      if (p.cap_a) reinterpret_cast<int4*>(p.cap_a + (size_t)t * na)[idx] = av[i];
      const float4 cs = reinterpret_cast<const float4*>(colsc)[idx];
      reinterpret_cast<float4*>(y)[idx] =
          make_float4(__fmul_rn(__fmul_rn((float)av[i].x, s), cs.x), __fmul_rn(__fmul_rn((float)av[i].y, s), cs.y),
                      __fmul_rn(__fmul_rn((float)av[i].z, s), cs.z), __fmul_rn(__fmul_rn((float)av[i].w, s), cs.w));
      // leave the row zeroed if a call of fewer rows can add into it (the
      // paths below kW8PairMinRows rows add their q_a / kv_a sums; this
      // one's GEMM stores them, so the rows past that stay as they are)
      if (t < kW8PairMinRows) reinterpret_cast<int4*>(a)[idx] = make_int4(0, 0, 0, 0);
    }
  }
  __syncwarp();
  // q latent: RMSNorm (gamma_q), requantisation
  float ss = 0.f;
  for (int c = lane; c < rq; c += 32) ss += y[c] * y[c];
  ss = warp_sum(ss);
  const float invq = 1.0f / sqrtf(ss / (float)rq + p.eps);
  float amax = 0.f;
  for (int c = lane; c < rq; c += 32) {
    const float v = y[c] * invq * gq[c];
    y[c] = v;
    amax = fmaxf(amax, fabsf(v));
  }
  amax = warp_max(amax);
  {
    const float inv = amax > 0.f ? __fdiv_rn(127.0f, amax) : 0.f;
    for (int c = lane; c < rq; c += 32) {
      const int8_t v = q8(y[c], inv);
      w.q1[(size_t)t * rq + c] = v;
      w.q1h[(size_t)t * rq + c] = __int2half_rn((int)v);
    }
    if (lane == 0) w.s1[t] = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f;
  }
  // compressed_kv: RMSNorm (gamma_kv), requantisation
  const float* ck = y + rq;
  ss = 0.f;
  for (int c = lane; c < kRank; c += 32) ss += ck[c] * ck[c];
  ss = warp_sum(ss);
  const float invk = 1.0f / sqrtf(ss / (float)kRank + p.eps);
  float nv[kRank / 32];
  amax = 0.f;
#pragma unroll
  for (int i = 0; i < kRank / 32; ++i) {
    const int c = lane + 32 * i;
    nv[i] = ck[c] * invk * gk[c];
    amax = fmaxf(amax, fabsf(nv[i]));
  }
  amax = warp_max(amax);
  {
    const float inv = amax > 0.f ? __fdiv_rn(127.0f, amax) : 0.f;
#pragma unroll
    for (int i = 0; i < kRank / 32; ++i) {
      const int c = lane + 32 * i;
      const int8_t v = q8(nv[i], inv);
      w.c1[(size_t)t * kRank + c] = v;
      w.c1h[(size_t)t * kRank + c] = __int2half_rn((int)v);
    }
    if (lane == 0) w.s2[t] = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f;
  }
  // RoPE of k_pe (raw columns 512..575 of the kv_a output): lane j < 32
  {
    int pos = p.positions[t];
    if (pos < 0 || pos >= p.max_pos) {
      if (lane == 0) atomicOr(p.status, kStatusBadPosition);
      pos = pos < 0 ? 0 : p.max_pos - 1;
    }
    const float* kp = ck + kRank;
    const int j = lane;
    const float a0 = kp[2 * j], b0 = kp[2 * j + 1];
    const float* cr = p.cos_t + (size_t)pos * kRope;
    const float* sr = p.sin_t + (size_t)pos * kRope;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.k_pe) + (size_t)t * kRope;
    out[j] = __float2bfloat16_rn(a0 * cr[j] - b0 * sr[j]);
    out[j + 32] = __float2bfloat16_rn(b0 * cr[j + 32] + a0 * sr[j + 32]);
  }
}

// ---------------------------------------------------------------- decode-size chain (T <= 8)
// Two launches instead of about ten, the second launched with programmatic
// stream serialisation so that it is resident, with its weight copies in
// flight, before the first finishes:
//   front  q_a / kv_a split-K GEMV, about one CTA per SM.  TMA copies of the
//          CTA's weight tile are issued at entry; meanwhile the CTA
//          quantises the hidden rows itself (every CTA finds the same amax,
//          so the codes are those of step 1); int32 partials are summed
//          across the CTA's warps and added atomically into the accumulator
//          rows, which the back kernel leaves zeroed after reading them.
//   back   q_b and kv_b, full K per 128-column block, each CTA walking a
//          fixed list of blocks through a ring of TMA boxes (the first ones
//          issued while the front kernel runs).  After the dependency wait
//          every CTA forms the requantised q_b / kv_b operands itself
//          (RMSNorms, step 4); dequantisation, RoPE(q_pe) and the head-major
//          stores happen in the epilogue, so no int32 accumulator of the
//          second stage goes back to memory.
// The two GEMV kernels also serve the plain int8 GEMM entry for M <= 8 (no
// quantisation, int32 results stored), which is how their integer sums are
// checked bit for bit.

struct W8FrontParams {
  CUtensorMap tm[2];               // W_qa, W_kva (or the one matrix of a plain GEMM)
  const void* x;                   // QUANT: bf16 hidden rows [M, K]; else int8 A [M, K]
  int32_t* acc;                    // [M, ldc]
  float* sx;                       // QUANT: [M] per-row scales
  unsigned* status;
  unsigned long long budget_ns;
  int M, K, ldc;
  int n[2];                        // columns of each matrix
  int bw[2];                       // box width (bytes = columns) of each matrix, <= 256
  int nblk1;                       // 256-column blocks of matrix 0
  int kchunk;                      // K rows per CTA: multiple of 32, <= 512
  int nbox;                        // TMA boxes per CTA (1, or 2 when kchunk > 256)
  int atomic;                      // add into acc (split K) instead of storing
};

__host__ __device__ constexpr size_t w8_front_region(int MT, int kc) {
  return 256 * (size_t)kc > 8192 * (size_t)MT ? 256 * (size_t)kc : 8192 * (size_t)MT;
}

// Grid (column blocks of matrix 0 then of matrix 1, K chunks); 256 threads.
// Shared memory: weight boxes [kchunk][bw], reused for the cross-warp
// reduction [8][MT][256] | codes [MT][kchunk] | per-warp amax [8][MT] |
// mbarrier | flag.
template <int MT, bool QUANT>
__global__ void __launch_bounds__(256) w8_front_kernel(const __grid_constant__ W8FrontParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~(uintptr_t)127);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kc = p.kchunk, k4n = kc >> 2;
  const int bx = blockIdx.x, kb = blockIdx.y * kc;
  const int sel = bx < p.nblk1 ? 0 : 1;
  const int col0 = (sel ? bx - p.nblk1 : bx) * 256;
  const int N = p.n[sel], bw = p.bw[sel];
  const int coff = sel ? p.n[0] : 0;
  const size_t region = w8_front_region(MT, kc);
  unsigned char* sW = sm;
  int* red = reinterpret_cast<int*>(sm);
  uint32_t* sX = reinterpret_cast<uint32_t*>(sm + region);
  float* s_amax = reinterpret_cast<float*>(sm + region + (size_t)MT * kc);
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_amax + 8 * MT);
  int* s_flag = reinterpret_cast<int*>(s_bar + 1);
  const uint32_t bar = smem_u32(s_bar);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    // boxes that start past K are not loaded: their rows meet zero codes
    const int brows = kc / p.nbox;
    int nload = 0;
    for (int i = 0; i < p.nbox; ++i) nload += kb + i * brows < p.K ? 1 : 0;
    mbar_arrive_expect_tx(bar, (uint32_t)(bw * brows * nload));
    for (int i = 0; i < nload; ++i)
      tma_load_2d(smem_u32(sW + (size_t)i * brows * bw), &p.tm[sel], col0, kb + i * brows, bar);
  }
  grid_dep_launch_dependents();
  // activation codes of rows [kb, kb + kc), four per word, zero past K
  if constexpr (QUANT) {
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(p.x);
    const int nv = p.K >> 3;  // 16-byte vectors per row
    float am[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) am[m] = 0.f;
    // all loads of two rows in flight at once (one round trip per row pair)
#pragma unroll
    for (int m0 = 0; m0 < MT; m0 += 2) {
      if (m0 < p.M) {
        for (int base = 0; base < nv; base += 256 * 4) {
          uint4 v[2][4];
#pragma unroll
          for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int i = base + tid + 256 * j;
              v[r][j] = make_uint4(0u, 0u, 0u, 0u);
              if (m0 + r < MT && m0 + r < p.M && i < nv)
                v[r][j] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(m0 + r) * p.K) + i);
            }
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            if (m0 + r < MT) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v[r][j]);
#pragma unroll
                for (int q = 0; q < 8; ++q) am[m0 + r] = fmaxf(am[m0 + r], fabsf(__bfloat162float(e[q])));
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) am[m] = fmaxf(am[m], __shfl_xor_sync(0xffffffffu, am[m], o));
      if (lane == 0) s_amax[warp * MT + m] = am[m];
    }
    __syncthreads();
    auto row_amax = [&](int m) {
      float a = s_amax[m];
#pragma unroll
      for (int w = 1; w < 8; ++w) a = fmaxf(a, s_amax[w * MT + m]);
      return a;
    };
    for (int i = tid; i < MT * k4n; i += 256) {
      const int m = i / k4n, k = kb + 4 * (i - m * k4n);
      uint32_t word = 0;
      if (m < p.M && k < p.K) {
        const float amax = row_amax(m);
        const float inv = amax > 0.f ? __fdiv_rn(127.0f, amax) : 0.f;
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(x + (size_t)m * p.K + k));
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          word |= (uint32_t)(uint8_t)q8(__bfloat162float(e[j]), inv) << (8 * j);
      }
      sX[i] = word;
    }
    if (bx == 0 && blockIdx.y == 0 && tid < p.M) {
      const float amax = row_amax(tid);
      p.sx[tid] = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f;
    }
  } else {
    const int8_t* A = static_cast<const int8_t*>(p.x);
    for (int i = tid; i < MT * k4n; i += 256) {
      const int m = i / k4n, k = kb + 4 * (i - m * k4n);
      sX[i] = (m < p.M && k < p.K) ? __ldg(reinterpret_cast<const uint32_t*>(A + (size_t)m * p.K + k)) : 0u;
    }
  }
  __syncthreads();
  // the weight tile (bounded wait; on expiry record it, let the copy land, leave)
  if (tid == 0) *s_flag = mbar_wait_bounded(bar, 0, p.budget_ns) ? 1 : 0;
  __syncthreads();
  if (*reinterpret_cast<volatile int*>(s_flag) == 0) {
    if (tid == 0) {
      if (p.status) atomicOr(p.status, kStatusTimeout);
      mbar_wait_bounded(bar, 0, drain_budget(p.budget_ns));
    }
    return;
  }
  while (!mbar_test_wait(bar, 0)) {
  }
  // a lane owns 8 columns; warp w takes the 4-row groups w, w + 8, ...
  int acc[MT][8];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[m][c] = 0;
  const bool live = lane * 8 < bw && col0 + lane * 8 < N;
  if (live) {
    for (int g = warp; g < k4n; g += 8) {
      const unsigned char* wr = sW + (size_t)(4 * g) * bw + lane * 8;
      const uint2 r0 = *reinterpret_cast<const uint2*>(wr);
      const uint2 r1 = *reinterpret_cast<const uint2*>(wr + bw);
      const uint2 r2 = *reinterpret_cast<const uint2*>(wr + 2 * bw);
      const uint2 r3 = *reinterpret_cast<const uint2*>(wr + 3 * bw);
      uint32_t w[8];
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // columns 4h .. 4h+3
        const uint32_t x0 = h ? r0.y : r0.x, x1 = h ? r1.y : r1.x;
        const uint32_t x2 = h ? r2.y : r2.x, x3 = h ? r3.y : r3.x;
        const uint32_t lo01 = __byte_perm(x0, x1, 0x5140), lo23 = __byte_perm(x2, x3, 0x5140);
        const uint32_t hi01 = __byte_perm(x0, x1, 0x7362), hi23 = __byte_perm(x2, x3, 0x7362);
        w[4 * h + 0] = __byte_perm(lo01, lo23, 0x5410);
        w[4 * h + 1] = __byte_perm(lo01, lo23, 0x7632);
        w[4 * h + 2] = __byte_perm(hi01, hi23, 0x5410);
        w[4 * h + 3] = __byte_perm(hi01, hi23, 0x7632);
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m < p.M) {
          const int a = (int)sX[m * k4n + g];
#pragma unroll
          for (int c = 0; c < 8; ++c) acc[m][c] = __dp4a((int)w[c], a, acc[m][c]);
        }
      }
    }
  }
  // the 8 warps' partials through shared memory (the weight area is free
  // now), then one coalesced add or store per column and row
  __syncthreads();
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    int* rp = red + (warp * MT + m) * 256 + lane * 8;
    *reinterpret_cast<int4*>(rp) = make_int4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
    *reinterpret_cast<int4*>(rp + 4) = make_int4(acc[m][4], acc[m][5], acc[m][6], acc[m][7]);
  }
  __syncthreads();
  for (int i = tid; i < p.M * 256; i += 256) {
    const int m = i >> 8, col = i & 255;
    if (col >= bw || col0 + col >= N) continue;
    int v = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) v += red[(w * MT + m) * 256 + col];
    int32_t* cp = p.acc + (size_t)m * p.ldc + coff + col0 + col;
    if (p.atomic)
      atomicAdd(cp, v);
    else
      *cp = v;
  }
}

__host__ __device__ constexpr size_t w8_front_smem(int MT, int kc) {
  return 128 + w8_front_region(MT, kc) + (size_t)MT * kc + 32 * (size_t)MT + 64;
}

constexpr int kBackStages = 8;      // most TMA boxes in flight per CTA
constexpr int kBackBox = 32768;     // bytes per ring slot (128 columns x 256 rows)

struct W8BackParams {
  CUtensorMap tm[2];               // W_qb, W_kvb (or one matrix): box bw x brows
  const int8_t* act[2];            // raw mode: int8 rows [M, K] of matrix 0
  const float* scol[2];            // [N] column scales (prolog mode)
  W8Params pr;                     // prolog mode: the call's inputs and outputs
  int32_t* acc1;                   // prolog mode: q_a / kv_a accumulator rows [M, q_rank + 576]
  const float* sx;                 // [M] hidden-row scales
  W8Workspace ws;                  // operand copies (q1, s1, c1, s2) written by CTA 0
  unsigned* readers;               // CTAs done reading acc1 (the last one clears it)
  const int* units;                // [grid + 1] offsets, then block ids; null: block b -> CTA b % grid
  int32_t* raw;                    // raw mode: C [M, raw_ld]
  unsigned* status;
  unsigned long long budget_ns;
  int M, raw_ld, raw_mode;
  int K[2], N[2];
  int bw[2];                       // box width in columns (128, or N when N < 128)
  int brows[2];                    // box height in rows (256, or K when K < 256)
  int nbox[2];                     // boxes per block: ceil(K / brows)
  int kpad[2];                     // nbox * brows: activation row length in shared memory
  int nblk1, nblk;                 // blocks of matrix 0, of both
  int nst;                         // ring slots (<= kBackStages)
  int npre;                        // boxes issued before the dependency wait (<= nst)
};

// Persistent over the CTA's blocks; 256 threads.  In prolog mode every CTA
// first forms the q_b / kv_b operands itself (norm_row on the M accumulator
// rows: cheaper than one more kernel boundary); CTA 0 also writes k_pe and
// the operand copies.  Warp w takes rows [32w, 32w + 32) of each box, a lane
// 4 columns (one 4-byte load per row, a warp one 128-byte row).  Shared
// memory: ring [nst][32 KB] | codes [MT][kpad0] then [MT][kpad1] |
// reduction [8][MT][128] int | norm scratch (prolog mode) | mbarriers.
template <int MT>
__global__ void __launch_bounds__(256) w8_back_kernel(const __grid_constant__ W8BackParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~(uintptr_t)127);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  unsigned char* ring = sm;
  const int nst = p.nst;
  int8_t* sAct0 = reinterpret_cast<int8_t*>(sm + (size_t)nst * kBackBox);
  int8_t* sAct1 = sAct0 + MT * p.kpad[0];
  int* red = reinterpret_cast<int*>(sAct1 + MT * p.kpad[1]);
  const bool prolog = !p.raw_mode;
  const int rq = p.pr.q_rank, na = rq + kNa;
  float* yrow = reinterpret_cast<float*>(red + 8 * MT * 128);
  float* colsc = yrow + (prolog ? na : 0);
  float* gq = colsc + (prolog ? na : 0);
  float* gk = gq + (prolog ? rq : 0);
  float* rope = gk + (prolog ? kRank : 0);      // [MT][128]
  float* srow = rope + (prolog ? MT * 2 * kRope : 0);  // [2][MT]
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(srow + (prolog ? 2 * MT : 0));
  __shared__ float scratch[8];
  __shared__ int s_last;
  unsigned ticket = 0;  // thread 0: this CTA's place among acc1's readers (prolog mode)
  // this CTA's blocks
  int u0, nu;
  const int* ulist = nullptr;
  if (p.units) {
    u0 = p.units[cta];
    nu = p.units[cta + 1] - u0;
    ulist = p.units + G + 1 + u0;
  } else {
    u0 = cta;
    nu = cta < p.nblk ? (p.nblk - 1 - cta) / G + 1 : 0;
  }
  if (nu == 0) {
    // no blocks (only when the grid has more CTAs than blocks): still one
    // of the acc1 readers to count
    if (prolog) {
      grid_dep_wait();
      if (tid == 0 && atomicAdd(p.readers, 1u) == (unsigned)G - 1) {
        for (int i = 0; i < p.M * na; ++i) p.acc1[i] = 0;
        *p.readers = 0u;
      }
    }
    return;
  }
  auto block_of = [&](int i) { return ulist ? ulist[i] : u0 + i * G; };
  // producer state (thread 0): next box to issue
  int iss_u = 0, iss_j = 0, issued = 0;
  auto issue_next = [&]() {
    if (iss_u >= nu) return;
    const int b = block_of(iss_u);
    const int sel = b < p.nblk1 ? 0 : 1;
    const int x = (sel ? b - p.nblk1 : b) * 128;
    const int slot = issued % nst;
    const uint32_t bar = smem_u32(s_bar + slot);
    mbar_arrive_expect_tx(bar, (uint32_t)(p.bw[sel] * p.brows[sel]));
    tma_load_2d(smem_u32(ring + slot * kBackBox), &p.tm[sel], x, iss_j * p.brows[sel], bar);
    ++issued;
    if (++iss_j == p.nbox[sel]) {
      iss_j = 0;
      ++iss_u;
    }
  };
  if (tid == 0) {
    for (int i = 0; i < nst; ++i) mbar_init(smem_u32(s_bar + i), 1);
    fence_mbar_init();
    // weights are read-only inputs: their copies may start before the
    // kernel that produces the activations has finished
    // weights are read-only: their copies may start before the previous
    // kernel has finished
    for (int i = 0; i < p.npre; ++i) issue_next();
  }
  if (prolog) {
    // inputs that do not come from the previous kernel, read while it runs
    norm_load_inputs(p.pr, colsc, gq, gk);
    for (int m = 0; m < p.M; ++m) rope_load(p.pr, m, rope + m * 2 * kRope);
    // codes are written up to K; the padding rows of the last box read zeros
    for (int i = tid; i < MT * p.kpad[0]; i += 256) sAct0[i] = 0;
    for (int i = tid; i < MT * p.kpad[1]; i += 256) sAct1[i] = 0;
    __syncthreads();
    grid_dep_wait();
    if (tid == 0)
      for (int i = p.npre; i < nst; ++i) issue_next();
    for (int m = 0; m < p.M; ++m)
      norm_row(p.acc1 + (size_t)m * na, p.sx[m], p.pr, yrow, colsc, gq, gk, rope + m * 2 * kRope,
               scratch, sAct0 + m * p.kpad[0], srow + m, sAct1 + m * p.kpad[1], srow + MT + m,
               cta == 0 ? static_cast<__nv_bfloat16*>(p.pr.k_pe) + (size_t)m * kRope : nullptr);
    // captured accumulators: CTA 0 copies the q_a / kv_a rows before it
    // counts itself as a reader (the last reader clears them)
    if (cta == 0 && p.pr.cap_a) {
      for (int i = tid; i < p.M * na; i += 256) p.pr.cap_a[i] = p.acc1[i];
      __syncthreads();
    }
    // the last CTA to finish reading acc1 clears it for the next call; it
    // learns that it is last from this add, whose result is only looked at
    // once its blocks are done, so the round trip stays off the critical path
    if (tid == 0) ticket = atomicAdd(p.readers, 1u);
    if (cta == 0) {  // operand copies for inspection
      for (int i = tid; i < p.M * rq; i += 256) p.ws.q1[i] = sAct0[(i / rq) * p.kpad[0] + i % rq];
      for (int i = tid; i < p.M * kRank; i += 256) p.ws.c1[i] = sAct1[(i / kRank) * p.kpad[1] + i % kRank];
      if (tid < p.M) {
        p.ws.s1[tid] = srow[tid];
        p.ws.s2[tid] = srow[MT + tid];
      }
    }
  } else {
    if (tid == 0)
      for (int i = p.npre; i < nst; ++i) issue_next();
    // raw mode: int8 rows of matrix 0 (zero past K)
    const int kp = p.kpad[0], K = p.K[0];
    for (int i = tid; i < MT * (kp >> 4); i += 256) {
      const int m = i / (kp >> 4), k = 16 * (i - m * (kp >> 4));
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (m < p.M && k < K) v = *reinterpret_cast<const uint4*>(p.act[0] + (size_t)m * K + k);
      *reinterpret_cast<uint4*>(sAct0 + m * kp + k) = v;
    }
  }
  __syncthreads();
  int consumed = 0;
  for (int ui = 0; ui < nu; ++ui) {
    const int b = block_of(ui);
    const int sel = b < p.nblk1 ? 0 : 1;
    const int bw = p.bw[sel], kp = p.kpad[sel];
    const int8_t* act = sel ? sAct1 : sAct0;
    int acc[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[m][c] = 0;
    // the epilogue's column scales, loaded now (thread t always handles the
    // column pair t % 64 of the block)
    const int cb = (sel ? b - p.nblk1 : b) * 128;
    float sc0 = 0.f, sc1 = 0.f;
    if (!p.raw_mode && cb + 2 * (tid & 63) < p.N[sel] && 2 * (tid & 63) < bw) {
      sc0 = p.scol[sel][cb + 2 * (tid & 63)];
      sc1 = p.scol[sel][cb + 2 * (tid & 63) + 1];
    }
    for (int j = 0; j < p.nbox[sel]; ++j) {
      const int slot = consumed % nst;
      const uint32_t bar = smem_u32(s_bar + slot);
      const uint32_t par = (uint32_t)(consumed / nst) & 1u;
      const bool ok = mbar_wait_bounded(bar, par, p.budget_ns);
      if (!__syncthreads_and(ok ? 1 : 0)) {
        if (tid == 0) {
          if (p.status) atomicOr(p.status, kStatusTimeout);
          for (int q = consumed; q < issued; ++q)
            mbar_wait_bounded(smem_u32(s_bar + q % nst), (uint32_t)(q / nst) & 1u,
                              drain_budget(p.budget_ns));
        }
        return;
      }
      const int r0 = 32 * warp;
      if (lane * 4 < bw && r0 < p.brows[sel]) {
        const unsigned char* wb = ring + slot * kBackBox + (size_t)r0 * bw + lane * 4;
        const int8_t* ab = act + j * p.brows[sel] + r0;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          if (r0 + 4 * g < p.brows[sel]) {
            const uint32_t x0 = *reinterpret_cast<const uint32_t*>(wb + (4 * g) * bw);
            const uint32_t x1 = *reinterpret_cast<const uint32_t*>(wb + (4 * g + 1) * bw);
            const uint32_t x2 = *reinterpret_cast<const uint32_t*>(wb + (4 * g + 2) * bw);
            const uint32_t x3 = *reinterpret_cast<const uint32_t*>(wb + (4 * g + 3) * bw);
            const uint32_t lo01 = __byte_perm(x0, x1, 0x5140), lo23 = __byte_perm(x2, x3, 0x5140);
            const uint32_t hi01 = __byte_perm(x0, x1, 0x7362), hi23 = __byte_perm(x2, x3, 0x7362);
            const uint32_t w0 = __byte_perm(lo01, lo23, 0x5410), w1 = __byte_perm(lo01, lo23, 0x7632);
            const uint32_t w2 = __byte_perm(hi01, hi23, 0x5410), w3 = __byte_perm(hi01, hi23, 0x7632);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              if (m < p.M) {
                const int a = *reinterpret_cast<const int*>(ab + m * kp + 4 * g);
                acc[m][0] = __dp4a((int)w0, a, acc[m][0]);
                acc[m][1] = __dp4a((int)w1, a, acc[m][1]);
                acc[m][2] = __dp4a((int)w2, a, acc[m][2]);
                acc[m][3] = __dp4a((int)w3, a, acc[m][3]);
              }
            }
          }
        }
      }
      ++consumed;
      __syncthreads();  // every warp is done with the slot
      if (tid == 0) issue_next();
    }
    // sum the 8 warps' partials, then the epilogue (two adjacent columns per item)
#pragma unroll
    for (int m = 0; m < MT; ++m)
      *reinterpret_cast<int4*>(red + (warp * MT + m) * 128 + lane * 4) =
          make_int4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
    __syncthreads();
    for (int idx = tid; idx < p.M * 64; idx += 256) {
      const int m = idx >> 6, col = 2 * (idx & 63);
      const int gc = cb + col;
      if (col >= bw || gc >= p.N[sel]) continue;
      int v0 = 0, v1 = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const int2 r = *reinterpret_cast<const int2*>(red + (w * MT + m) * 128 + col);
        v0 += r.x;
        v1 += r.y;
      }
      if (p.raw_mode) {
        *reinterpret_cast<int2*>(p.raw + (size_t)m * p.raw_ld + gc) = make_int2(v0, v1);
        continue;
      }
      int32_t* cap = sel ? p.pr.cap_kvb : p.pr.cap_qb;
      if (cap) *reinterpret_cast<int2*>(cap + (size_t)m * p.N[sel] + gc) = make_int2(v0, v1);
      const float sr = srow[sel * MT + m];
      const float y0 = __fmul_rn(__fmul_rn((float)v0, sr), sc0);
      const float y1 = __fmul_rn(__fmul_rn((float)v1, sr), sc1);
      const int bi = m / p.pr.s, si = m - bi * p.pr.s;
      if (sel == 0) {
        const int h = gc / (kNope + kRope), e = gc - h * (kNope + kRope);
        const size_t orow = ((size_t)bi * p.pr.heads + h) * p.pr.s + si;
        if (e < kNope) {
          *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.pr.q_nope) + orow * kNope + e) =
              __floats2bfloat162_rn(y0, y1);
        } else {
          const int j = (e - kNope) >> 1;
          const float* cr = rope + m * 2 * kRope;
          const float* sn = cr + kRope;
          __nv_bfloat16* qp = static_cast<__nv_bfloat16*>(p.pr.q_pe) + orow * kRope;
          qp[j] = __float2bfloat16_rn(y0 * cr[j] - y1 * sn[j]);
          qp[j + 32] = __float2bfloat16_rn(y1 * cr[j + 32] + y0 * sn[j + 32]);
        }
      } else {
        const int h = gc / kHeadCols, e = gc - h * kHeadCols;
        const size_t orow = ((size_t)bi * p.pr.heads + h) * p.pr.s + si;
        __nv_bfloat16* dst = e < kNope ? static_cast<__nv_bfloat16*>(p.pr.k_nope) + orow * kNope + e
                                       : static_cast<__nv_bfloat16*>(p.pr.value) + orow * kV + (e - kNope);
        *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(y0, y1);
      }
    }
    __syncthreads();  // the reduction area is reused by the next block
  }
  if (prolog) {
    if (tid == 0) s_last = ticket == (unsigned)G - 1 ? 1 : 0;
    __syncthreads();
    if (s_last) {
      for (int i = tid; i < p.M * na; i += 256) p.acc1[i] = 0;
      if (tid == 0) *p.readers = 0u;
    }
  }
}

// nrm_floats: the prolog-mode norm scratch (0 in raw mode).
__host__ __device__ constexpr size_t w8_back_smem(int MT, int nst, int kp0, int kp1, int nrm_floats) {
  return 128 + (size_t)nst * kBackBox + (size_t)MT * (kp0 + kp1) + 8 * (size_t)MT * 512 +
         4 * (size_t)nrm_floats + 8 * kBackStages + 16;
}
__host__ __device__ constexpr int back_norm_floats(int MT, int q_rank) {
  return 2 * (q_rank + kNa) + q_rank + kRank + MT * 2 * kRope + 2 * MT;
}

// Ring slots that fit next to the codes, the reduction area and the scratch.
int back_stages(int MT, int kp0, int kp1, int nrm_floats) {
  int n = kBackStages;
  while (n > 2 && w8_back_smem(MT, n, kp0, kp1, nrm_floats) > 227 * 1024) --n;
  return n;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int g_num_sms = 148;

// Launch with or without programmatic stream serialisation (the kernel may
// start before the previous kernel in the stream has finished; it calls
// grid_dep_wait before touching that kernel's results).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? at : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int MT, bool QUANT>
cudaError_t launch_front(const W8FrontParams& f, int nblk, int splits, cudaStream_t st) {
  const size_t smem = w8_front_smem(MT, f.kchunk);
  cudaError_t e = cudaFuncSetAttribute(w8_front_kernel<MT, QUANT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_k(w8_front_kernel<MT, QUANT>, dim3(nblk, splits), dim3(256), smem, st, false, f);
}

template <bool QUANT>
cudaError_t launch_front_m(const W8FrontParams& f, int nblk, int splits, cudaStream_t st) {
  if (f.M <= 1) return launch_front<1, QUANT>(f, nblk, splits, st);
  if (f.M <= 2) return launch_front<2, QUANT>(f, nblk, splits, st);
  if (f.M <= 4) return launch_front<4, QUANT>(f, nblk, splits, st);
  return launch_front<8, QUANT>(f, nblk, splits, st);
}

template <int MT>
cudaError_t launch_back(const W8BackParams& b, int grid, cudaStream_t st, bool pdl) {
  W8BackParams bb = b;
  const int nf = b.raw_mode ? 0 : back_norm_floats(MT, b.pr.q_rank);
  // prolog mode: two slots, so that the CTAs fit next to the front kernel's
  // and start their copies while it runs (a deeper ring that has to wait
  // for the front kernel to leave measured no faster)
  bb.nst = b.raw_mode ? back_stages(MT, b.kpad[0], b.kpad[1], nf) : 2;
  if (bb.npre > bb.nst) bb.npre = bb.nst;
  const size_t smem = w8_back_smem(MT, bb.nst, b.kpad[0], b.kpad[1], nf);
  cudaError_t e = cudaFuncSetAttribute(w8_back_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  return launch_k(w8_back_kernel<MT>, dim3(grid), dim3(256), smem, st, pdl, bb);
}

cudaError_t launch_back_m(const W8BackParams& b, int grid, cudaStream_t st, bool pdl) {
  if (b.M <= 1) return launch_back<1>(b, grid, st, pdl);
  if (b.M <= 2) return launch_back<2>(b, grid, st, pdl);
  if (b.M <= 4) return launch_back<4>(b, grid, st, pdl);
  return launch_back<8>(b, grid, st, pdl);
}

// Box geometry of one matrix of the back kernel.
void back_geometry(int K, int N, int* bw, int* brows, int* nbox, int* kpad) {
  *bw = N < 128 ? N : 128;
  *brows = K < 256 ? K : 256;
  *nbox = (K + *brows - 1) / *brows;
  *kpad = *nbox * *brows;
}

// K rows per front-kernel CTA: about one CTA per SM over `nblk` column
// blocks, a multiple of 32 rows, at most two 256-row boxes.
int front_kchunk(int K, int nblk, int num_sms) {
  int target = num_sms / nblk;
  if (target < 1) target = 1;
  int kc = (K + target - 1) / target;
  kc = (kc + 31) / 32 * 32;
  if (kc > 512) kc = 512;
  return kc;
}

bool encode_i8(CUtensorMap* m, const void* base, int rows, int cols, int box_cols, int box_rows) {
  return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, (uint64_t)cols, (uint64_t)rows,
                        (uint64_t)cols, (uint32_t)box_cols, (uint32_t)box_rows,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Plain int8 GEMM for M <= 8 through the two GEMV kernels: full K per CTA
// when K is short, else split K with atomics into a cleared C.
cudaError_t gemv_tma(const int8_t* A, const int8_t* W, int M, int K, int N, int32_t* C, int ldc,
                     cudaStream_t st, int* launches) {
  if (K <= 2048) {
    W8BackParams b = {};
    int bw, brows, nbox, kpad;
    back_geometry(K, N, &bw, &brows, &nbox, &kpad);
    if (!encode_i8(&b.tm[0], W, K, N, bw, brows)) return cudaErrorInvalidValue;
    b.tm[1] = b.tm[0];
    b.act[0] = A;
    b.raw = C;
    b.raw_ld = ldc;
    b.raw_mode = 1;
    b.M = M;
    b.K[0] = K;
    b.N[0] = N;
    b.bw[0] = bw;
    b.brows[0] = brows;
    b.nbox[0] = nbox;
    b.kpad[0] = kpad;
    b.nblk1 = b.nblk = (N + 127) / 128;
    b.status = nullptr;
    b.budget_ns = 1000000000ull;
    const int grid = b.nblk < g_num_sms ? b.nblk : g_num_sms;
    ++*launches;
    return launch_back_m(b, grid, st, false);
  }
  W8FrontParams f = {};
  const int nblk = (N + 255) / 256;
  f.kchunk = front_kchunk(K, nblk, g_num_sms);
  const int splits = (K + f.kchunk - 1) / f.kchunk;
  f.bw[0] = f.bw[1] = N < 256 ? N : 256;
  f.nbox = f.kchunk > 256 ? 2 : 1;
  if (!encode_i8(&f.tm[0], W, K, N, f.bw[0], f.kchunk / f.nbox)) return cudaErrorInvalidValue;
  f.tm[1] = f.tm[0];
  f.x = A;
  f.acc = C;
  f.M = M;
  f.K = K;
  f.ldc = ldc;
  f.n[0] = N;
  f.n[1] = 0;
  f.nblk1 = nblk;
  f.atomic = splits > 1 ? 1 : 0;
  f.budget_ns = 1000000000ull;
  if (splits > 1) {
    cudaError_t e = cudaMemset2DAsync(C, (size_t)ldc * 4, 0, (size_t)N * 4, M, st);
    if (e != cudaSuccess) return e;
    ++*launches;
  }
  ++*launches;
  return launch_front_m<false>(f, nblk, splits, st);
}

// Decode-size chain: front (normal launch) -> back (launched with
// programmatic stream serialisation; it forms the q_b / kv_b operands itself).
cudaError_t launch_small_chain(const W8Params& p, const W8Workspace& w, const W8SmallPlan& pl,
                               const W8Maps& mp, cudaStream_t st, int* launches) {
  const int T = p.T, rq = p.q_rank, H = p.heads;
  W8FrontParams f = {};
  f.tm[0] = mp.qa;
  f.tm[1] = mp.kva;
  f.x = p.hidden;
  f.acc = w.acc1;
  f.sx = w.sx;
  f.status = p.status;
  f.budget_ns = p.budget_ns;
  f.M = T;
  f.K = p.hidden_dim;
  f.ldc = rq + kNa;
  f.n[0] = rq;
  f.n[1] = kNa;
  f.bw[0] = rq < 256 ? rq : 256;
  f.bw[1] = 256;
  f.nblk1 = pl.nblk_a1;
  f.kchunk = pl.kchunk;
  f.nbox = pl.kchunk > 256 ? 2 : 1;
  f.atomic = pl.splits > 1 ? 1 : 0;
  cudaError_t e = launch_front_m<true>(f, pl.nblk_a, pl.splits, st);
  ++*launches;
  if (e != cudaSuccess) return e;
  W8BackParams b = {};
  b.tm[0] = mp.qb;
  b.tm[1] = mp.kvb;
  b.scol[0] = p.sW_qb;
  b.scol[1] = p.sW_kvb;
  b.pr = p;
  b.acc1 = w.acc1;
  b.sx = w.sx;
  b.ws = w;
  b.readers = w.readers;
  b.units = pl.units;
  b.npre = 2;
  b.status = p.status;
  b.budget_ns = p.budget_ns;
  b.M = T;
  b.K[0] = rq;
  b.K[1] = kRank;
  b.N[0] = H * (kNope + kRope);
  b.N[1] = H * kHeadCols;
  for (int i = 0; i < 2; ++i) back_geometry(b.K[i], b.N[i], &b.bw[i], &b.brows[i], &b.nbox[i], &b.kpad[i]);
  b.nblk1 = pl.nblk_b1;
  b.nblk = pl.nblk_b;
  e = launch_back_m(b, pl.grid_b, st, true);
  ++*launches;
  return e;
}

// c_zero: C is known to hold zeros (no clearing before split-K adds).
cudaError_t gemm(const int8_t* A, const int8_t* W, int M, int K, int N, int32_t* C, int ldc,
                 cudaStream_t st, int* launches, bool c_zero = false) {
  // decode sizes stream the weights; the 64 x 64 tensor-core tiles would be
  // mostly padding rows
  if (M <= kGemvMaxRows && K % 16 == 0 && N % 16 == 0) return gemv_tma(A, W, M, K, N, C, ldc, st, launches);
  const int tn = N / kGBN, tm = (M + kGBM - 1) / kGBM;
  int splits = 1;
  const int tiles = tn * tm;
  const int target = 2 * g_num_sms;
  if (tiles < target) {
    splits = (target + tiles - 1) / tiles;
    const int maxs = K / (4 * kGBK);  // at least 4 k-steps per split
    if (splits > maxs) splits = maxs > 0 ? maxs : 1;
  }
  int kchunk = (K + splits - 1) / splits;
  kchunk = (kchunk + kGBK - 1) / kGBK * kGBK;
  splits = (K + kchunk - 1) / kchunk;
  if (splits > 1 && !c_zero) {
    // split-K partials are added atomically: clear the N columns of each row
    cudaError_t e = cudaMemset2DAsync(C, (size_t)ldc * 4, 0, (size_t)N * 4, M, st);
    if (e != cudaSuccess) return e;
    ++*launches;
  }
  ++*launches;
  return launch_k(gemm_s8_kernel, dim3(tn, tm, splits), dim3(kGThreads), 0, st, false, A, W, M, K, N, C,
                  ldc, kchunk, splits > 1 ? 1 : 0);
}

}  // namespace

namespace {

int small_nblk_b(int q_rank, int heads) {
  (void)q_rank;
  return (heads * (kNope + kRope) + 127) / 128 + (heads * kHeadCols + 127) / 128;
}

void small_plan(int hidden, int q_rank, int heads, int num_sms, W8SmallPlan* pl) {
  pl->nblk_a1 = (q_rank + 255) / 256;
  pl->nblk_a = pl->nblk_a1 + (kNa + 255) / 256;
  pl->kchunk = front_kchunk(hidden, pl->nblk_a, num_sms);
  pl->splits = (hidden + pl->kchunk - 1) / pl->kchunk;
  pl->nblk_b1 = (heads * (kNope + kRope) + 127) / 128;
  pl->nblk_b = small_nblk_b(q_rank, heads);
  pl->grid_b = pl->nblk_b < num_sms ? pl->nblk_b : num_sms;
}

// Longest-processing-time-first assignment of the q_b / kv_b blocks (cost:
// boxes per block) to the back kernel's CTAs: [grid + 1] offsets, then ids.
std::vector<int> small_units(int q_rank, int heads, const W8SmallPlan& pl) {
  int bw, brows, nbox0, nbox1, kpad;
  back_geometry(q_rank, heads * (kNope + kRope), &bw, &brows, &nbox0, &kpad);
  back_geometry(kRank, heads * kHeadCols, &bw, &brows, &nbox1, &kpad);
  const int G = pl.grid_b;
  std::vector<long> load(G, 0);
  std::vector<std::vector<int>> lists(G);
  // blocks in decreasing cost (ids of the costlier matrix first; stable)
  std::vector<int> order;
  const bool qfirst = nbox0 >= nbox1;
  for (int pass = 0; pass < 2; ++pass) {
    const bool q = (pass == 0) == qfirst;
    const int lo = q ? 0 : pl.nblk_b1, hi = q ? pl.nblk_b1 : pl.nblk_b;
    for (int b = lo; b < hi; ++b) order.push_back(b);
  }
  for (int b : order) {
    int best = 0;
    for (int c = 1; c < G; ++c)
      if (load[c] < load[best]) best = c;
    load[best] += b < pl.nblk_b1 ? nbox0 : nbox1;
    lists[best].push_back(b);
  }
  std::vector<int> t(G + 1 + pl.nblk_b);
  int off = 0;
  for (int c = 0; c < G; ++c) {
    t[c] = off;
    for (int b : lists[c]) t[G + 1 + off++] = b;
  }
  t[G] = off;
  return t;
}

}  // namespace

// Row pitch (elements) of a widened fp16 weight copy: a multiple of 256.
int wide_ld(int n) { return (n + 255) / 256 * 256; }

// Bytes of the widened weight copies (none below kW8PairMinRows tokens).
size_t wide_bytes(int hidden, int q_rank, int heads, int max_tokens) {
  if (max_tokens < kW8PairMinRows) return 0;
  return align256((size_t)hidden * wide_ld(q_rank + kNa) * 2) +
         align256((size_t)q_rank * wide_ld(heads * (kNope + kRope)) * 2) +
         align256((size_t)kRank * wide_ld(heads * kHeadCols) * 2);
}

size_t w8_workspace_bytes(int hidden, int q_rank, int heads, int max_tokens, int num_sms) {
  const size_t T = (size_t)max_tokens;
  return align256(T * hidden * 2) + align256(T * 4) + align256(T * (q_rank + kNa) * 4) +
         align256(T * q_rank) + align256(T * 4) + align256(T * kRank) + align256(T * 4) +
         align256(T * q_rank * 2) + align256(T * kRank * 2) +
         align256((size_t)(num_sms + 1 + small_nblk_b(q_rank, heads)) * 4) + 256 +
         wide_bytes(hidden, q_rank, heads, max_tokens);
}

void w8_workspace_carve(void* base, int hidden, int q_rank, int heads, int max_tokens,
                        int num_sms, W8Workspace* w, W8SmallPlan* plan) {
  const size_t T = (size_t)max_tokens;
  unsigned char* b = static_cast<unsigned char*>(base);
  w->xh = reinterpret_cast<__half*>(b); b += align256(T * hidden * 2);
  w->sx = reinterpret_cast<float*>(b); b += align256(T * 4);
  w->acc1 = reinterpret_cast<int32_t*>(b); b += align256(T * (q_rank + kNa) * 4);
  w->q1 = reinterpret_cast<int8_t*>(b); b += align256(T * q_rank);
  w->s1 = reinterpret_cast<float*>(b); b += align256(T * 4);
  w->c1 = reinterpret_cast<int8_t*>(b); b += align256(T * kRank);
  w->s2 = reinterpret_cast<float*>(b); b += align256(T * 4);
  w->q1h = reinterpret_cast<__half*>(b); b += align256(T * q_rank * 2);
  w->c1h = reinterpret_cast<__half*>(b); b += align256(T * kRank * 2);
  small_plan(hidden, q_rank, heads, num_sms, plan);
  plan->units = reinterpret_cast<int*>(b);
  b += align256((size_t)(num_sms + 1 + small_nblk_b(q_rank, heads)) * 4);
  w->readers = reinterpret_cast<unsigned*>(b);
  b += 256;
  w->lda = wide_ld(q_rank + kNa);
  w->ldqb = wide_ld(heads * (kNope + kRope));
  w->ldkvb = wide_ld(heads * kHeadCols);
  if (max_tokens >= kW8PairMinRows) {
    w->wa16 = reinterpret_cast<__half*>(b); b += align256((size_t)hidden * w->lda * 2);
    w->wqb16 = reinterpret_cast<__half*>(b); b += align256((size_t)q_rank * w->ldqb * 2);
    w->wkvb16 = reinterpret_cast<__half*>(b);
  } else {
    w->wa16 = w->wqb16 = w->wkvb16 = nullptr;
  }
}

cudaError_t w8_workspace_init(const W8Workspace& w, const W8SmallPlan& plan, int hidden,
                              int q_rank, int heads, int max_tokens, int num_sms) {
  (void)hidden;
  (void)num_sms;
  cudaError_t e = cudaMemset(w.acc1, 0, (size_t)max_tokens * (q_rank + kNa) * 4);
  if (e == cudaSuccess) e = cudaMemset(w.readers, 0, 256);
  if (e != cudaSuccess) return e;
  const std::vector<int> t = small_units(q_rank, heads, plan);
  return cudaMemcpy(plan.units, t.data(), t.size() * sizeof(int), cudaMemcpyHostToDevice);
}

bool w8_encode_maps(const W8Params& p, const W8SmallPlan& pl, W8Maps* m) {
  const int rq = p.q_rank, H = p.heads, h = p.hidden_dim;
  int bw, brows, nbox, kpad;
  m->valid = false;
  const int arows = pl.kchunk > 256 ? pl.kchunk / 2 : pl.kchunk;
  if (!encode_i8(&m->qa, p.W_qa, h, rq, rq < 256 ? rq : 256, arows)) return false;
  if (!encode_i8(&m->kva, p.W_kva, h, kNa, 256, arows)) return false;
  back_geometry(rq, H * (kNope + kRope), &bw, &brows, &nbox, &kpad);
  if (!encode_i8(&m->qb, p.W_qb, rq, H * (kNope + kRope), bw, brows)) return false;
  back_geometry(kRank, H * kHeadCols, &bw, &brows, &nbox, &kpad);
  if (!encode_i8(&m->kvb, p.W_kvb, kRank, H * kHeadCols, bw, brows)) return false;
  m->src[0] = p.W_qa;
  m->src[1] = p.W_kva;
  m->src[2] = p.W_qb;
  m->src[3] = p.W_kvb;
  m->valid = true;
  return true;
}

cudaError_t w8a8_quant_rows_launch(const void* x_bf16, int rows, int cols, int8_t* q,
                                   float* scale, cudaStream_t stream) {
  quant_rows_kernel<int8_t><<<rows, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x_bf16), cols, q, scale);
  return cudaGetLastError();
}

cudaError_t w8a8_gemm_s32_launch(const int8_t* A, const int8_t* W, int M, int K, int N,
                                 int32_t* acc, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
  int launches = 0;
  if (N % kGBN != 0 || K % kGBK != 0) return cudaErrorNotSupported;
  return gemm(A, W, M, K, N, acc, N, stream, &launches);
}

cudaError_t w8a8_copy_operands(const W8Workspace& w, int T, int q_rank, int8_t* q1, float* s1,
                               int8_t* c1, float* s2, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyAsync(q1, w.q1, (size_t)T * q_rank, cudaMemcpyDeviceToDevice, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(s1, w.s1, (size_t)T * 4, cudaMemcpyDeviceToDevice, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(c1, w.c1, (size_t)T * kRank, cudaMemcpyDeviceToDevice, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(s2, w.s2, (size_t)T * 4, cudaMemcpyDeviceToDevice, stream);
  return e;
}

cudaError_t w8a8_launch(const W8Params& p, const W8Workspace& w, const W8SmallPlan& plan,
                        const W8Maps* maps, int num_sms, cudaStream_t st, int* launches) {
  g_num_sms = num_sms;
  *launches = 0;
  const int T = p.T, h = p.hidden_dim, rq = p.q_rank, H = p.heads;
  const int na = rq + kNa;
  cudaError_t e;
  if (T <= kW8SmallRows && maps && maps->valid) {
    e = launch_small_chain(p, w, plan, *maps, st, launches);
    if (e != cudaSuccess) {
      // the accumulator rows must be zero when the next chain starts
      cudaGetLastError();
      cudaMemsetAsync(w.acc1, 0, (size_t)T * na * 4, st);
    }
    return e;
  }
  // 1. quantise hidden rows (fp16 codes: the tensor-core GEMM operand)
  quant_rows_kernel<__half><<<T, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(p.hidden), h, w.xh, w.sx);
  ++*launches;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // Accumulator rows [0, kW8PairMinRows) are left zeroed by every call
  // (norm_quant_kernel, norm_quant_warp_kernel or the decode-size chain), so
  // the paths below kW8PairMinRows rows add their q_a / kv_a sums into them;
  // the pair path stores its sums (every column of rows [0, T)).
  const bool pairk = T >= kW8PairMinRows && w.wa16;
  auto chain_pair = [&]() -> cudaError_t {
    // 1b. the int8 weights widened to fp16 copies ([W_qa | W_kva], W_qb, W_kvb)
    W8WidenJob jobs[4] = {
        {p.W_qa, w.wa16, h, rq, w.lda, rq},
        {p.W_kva, w.wa16 + rq, h, kNa, w.lda, w.lda - rq},
        {p.W_qb, w.wqb16, rq, H * (kNope + kRope), w.ldqb, w.ldqb},
        {p.W_kvb, w.wkvb16, kRank, H * kHeadCols, w.ldkvb, w.ldkvb}};
    cudaError_t e2 = w8_widen_launch(jobs, 4, g_num_sms, st);
    ++*launches;
    if (e2 != cudaSuccess) return e2;
    // 2. q_a_proj and kv_a_proj as one [T, q_rank + 576] accumulator (stored)
    W8PairParams g1 = {};
    g1.K[0] = h; g1.N[0] = na; g1.ldw[0] = w.lda;
    g1.T = T; g1.raw = 1; g1.C = w.acc1; g1.ldc = na; g1.coff[0] = 0;
    g1.heads = H; g1.s = p.s; g1.status = p.status; g1.budget_ns = p.budget_ns;
    e2 = w8pair_launch(g1, w.xh, w.xh, w.wa16, w.wa16, g_num_sms, st);
    ++*launches;
    if (e2 != cudaSuccess) return e2;
    // 3-4. RMSNorms, requantisation, RoPE(k_pe): a warp per token row
    const size_t smem = norm_warp_smem(rq);
    e2 = cudaFuncSetAttribute(norm_quant_warp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e2 == cudaSuccess)
      e2 = launch_k(norm_quant_warp_kernel, dim3((T + kNormRowsPerCta - 1) / kNormRowsPerCta), dim3(256), smem, st,
                    false, w.acc1, (const float*)w.sx, p, w);
    ++*launches;
    if (e2 != cudaSuccess) return e2;
    // 5-6. q_b_proj -> q_nope, RoPE(q_pe); kv_b_proj -> k_nope, value (one launch)
    W8PairParams g2 = {};
    g2.K[0] = rq; g2.N[0] = H * (kNope + kRope); g2.ldw[0] = w.ldqb;
    g2.K[1] = kRank; g2.N[1] = H * kHeadCols; g2.ldw[1] = w.ldkvb;
    g2.T = T; g2.raw = 0;
    g2.sx[0] = w.s1; g2.sx[1] = w.s2; g2.sw[0] = p.sW_qb; g2.sw[1] = p.sW_kvb;
    g2.positions = p.positions; g2.cos_t = p.cos_t; g2.sin_t = p.sin_t; g2.max_pos = p.max_pos;
    g2.q_nope = p.q_nope; g2.q_pe = p.q_pe; g2.k_nope = p.k_nope; g2.value = p.value;
    g2.cap[0] = p.cap_qb; g2.cap[1] = p.cap_kvb;
    g2.heads = H; g2.s = p.s; g2.status = p.status; g2.budget_ns = p.budget_ns;
    e2 = w8pair_launch(g2, w.q1h, w.c1h, w.wqb16, w.wkvb16, g_num_sms, st);
    ++*launches;
    return e2;
  };
  auto chain = [&]() -> cudaError_t {
    if (pairk) return chain_pair();
    // 2. q_a_proj and kv_a_proj into one [T, q_rank + 576] accumulator
    W8MmaParams g1 = {};
    g1.K[0] = h; g1.N[0] = rq; g1.K[1] = h; g1.N[1] = kNa;
    g1.T = T; g1.raw = 1; g1.C = w.acc1; g1.ldc = na; g1.coff[0] = 0; g1.coff[1] = rq;
    g1.status = p.status; g1.budget_ns = p.budget_ns;
    // (the three launches after the quantisation carry the programmatic
    // dependency: each starts while the one before finishes and waits for
    // it before reading its results; the weights are read after that wait)
    cudaError_t e2 = w8mma_launch(g1, p.W_qa, p.W_kva, w.xh, w.xh, g_num_sms, st, true);
    ++*launches;
    if (e2 != cudaSuccess) return e2;
    // 3-4. RMSNorms, requantisation, RoPE(k_pe)
    const size_t smem = norm_smem(rq);
    e2 = cudaFuncSetAttribute(norm_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e2 == cudaSuccess) e2 = launch_k(norm_quant_kernel, dim3(T), dim3(256), smem, st, true, w.acc1, (const float*)w.sx, p, w);
    ++*launches;
    if (e2 != cudaSuccess) return e2;
    // 5-6. q_b_proj -> q_nope, RoPE(q_pe); kv_b_proj -> k_nope, value (one launch)
    W8MmaParams g2 = {};
    g2.K[0] = rq; g2.N[0] = H * (kNope + kRope); g2.K[1] = kRank; g2.N[1] = H * kHeadCols;
    g2.T = T; g2.raw = 0;
    g2.sx[0] = w.s1; g2.sx[1] = w.s2; g2.sw[0] = p.sW_qb; g2.sw[1] = p.sW_kvb;
    g2.positions = p.positions; g2.cos_t = p.cos_t; g2.sin_t = p.sin_t; g2.max_pos = p.max_pos;
    g2.q_nope = p.q_nope; g2.q_pe = p.q_pe; g2.k_nope = p.k_nope; g2.value = p.value;
    g2.cap[0] = p.cap_qb; g2.cap[1] = p.cap_kvb;
    g2.heads = H; g2.s = p.s; g2.status = p.status; g2.budget_ns = p.budget_ns;
    e2 = w8mma_launch(g2, p.W_qb, p.W_kvb, w.q1h, w.c1h, g_num_sms, st, true);
    ++*launches;
    return e2;
  };
  e = chain();
  if (e != cudaSuccess) {
    // the accumulator rows must be zero when the next call starts
    cudaGetLastError();
    cudaMemsetAsync(w.acc1, 0, (size_t)T * na * 4, st);
  }
  return e;
}

}  // namespace mla
