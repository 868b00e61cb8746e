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
#include "common.cuh"
#include "internal.h"

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

// Small-M path (decode sizes): C[m, n] (+)= sum_k A[m, k] * W[k, n] for the
// M <= MT rows.  The weight stream is the cost, so a lane owns 8 consecutive
// columns (a warp 256) and walks K 4 rows at a time with 8-byte coalesced
// loads of each row; the 4 x 8 bytes are transposed with byte permutes into
// 8 words of 4 K-consecutive weights and accumulated with dp4a (int8 x int8
// -> int32).  The 4 warps of a CTA take interleaved 4-row groups of the
// CTA's K range and are summed through shared memory; blockIdx.y splits K
// across CTAs, whose partials are added with atomics (exact).
template <int MT>
__global__ void __launch_bounds__(128) gemv_s8_kernel(const int8_t* __restrict__ A,
                                                      const int8_t* __restrict__ W, int M, int K,
                                                      int N, int32_t* __restrict__ C, int ldc,
                                                      int kchunk, int atomic) {
  __shared__ int red[3][MT][8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * 256 + lane * 8;
  const int kb = blockIdx.y * kchunk;
  const int ke = min(K, kb + kchunk);
  const bool live = n0 < N;
  int acc[MT][8];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[m][c] = 0;
  if (live) {
    const int8_t* wp = W + (size_t)(kb + 4 * warp) * N + n0;
#pragma unroll 4
    for (int k = kb + 4 * warp; k < ke; k += 16) {
      const uint2 r0 = __ldg(reinterpret_cast<const uint2*>(wp));
      const uint2 r1 = __ldg(reinterpret_cast<const uint2*>(wp + N));
      const uint2 r2 = __ldg(reinterpret_cast<const uint2*>(wp + 2 * (size_t)N));
      const uint2 r3 = __ldg(reinterpret_cast<const uint2*>(wp + 3 * (size_t)N));
      wp += 16 * (size_t)N;
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
        if (m < M) {
          const int a = __ldg(reinterpret_cast<const int*>(A + (size_t)m * K + k));
#pragma unroll
          for (int c = 0; c < 8; ++c) acc[m][c] = __dp4a((int)w[c], a, acc[m][c]);
        }
      }
    }
  }
  if (warp > 0) {
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int c = 0; c < 8; ++c) red[warp - 1][m][c][lane] = acc[m][c];
  }
  __syncthreads();
  if (warp == 0 && live) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < M) {
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[m][c] += red[0][m][c][lane] + red[1][m][c][lane] + red[2][m][c][lane];
        int32_t* cp = C + (size_t)m * ldc + n0;
        if (atomic) {
#pragma unroll
          for (int j = 0; j < 8; ++j) atomicAdd(cp + j, acc[m][j]);
        } else {
          *reinterpret_cast<int4*>(cp) = make_int4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
          *reinterpret_cast<int4*>(cp + 4) = make_int4(acc[m][4], acc[m][5], acc[m][6], acc[m][7]);
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

// One CTA (256 threads) per row of a bf16 matrix [rows, cols] -> int8 + scale.
__global__ void __launch_bounds__(256) quant_rows_kernel(const __nv_bfloat16* __restrict__ x, int cols,
                                                         int8_t* __restrict__ q,
                                                         float* __restrict__ scale) {
  __shared__ float scratch[8];
  const int row = blockIdx.x;
  const __nv_bfloat16* xr = x + (size_t)row * cols;
  float amax = 0.f;
  for (int c = threadIdx.x * 8; c < cols; c += 256 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + c);
    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(__bfloat162float(e[i])));
  }
  amax = block_reduce<true>(amax, scratch);
  const float inv = amax > 0.f ? __fdiv_rn(127.0f, amax) : 0.f;
  for (int c = threadIdx.x * 8; c < cols; c += 256 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + c);
    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v);
    char4 lo, hi;
    lo.x = q8(__bfloat162float(e[0]), inv); lo.y = q8(__bfloat162float(e[1]), inv);
    lo.z = q8(__bfloat162float(e[2]), inv); lo.w = q8(__bfloat162float(e[3]), inv);
    hi.x = q8(__bfloat162float(e[4]), inv); hi.y = q8(__bfloat162float(e[5]), inv);
    hi.z = q8(__bfloat162float(e[6]), inv); hi.w = q8(__bfloat162float(e[7]), inv);
    *reinterpret_cast<char4*>(q + (size_t)row * cols + c) = lo;
    *reinterpret_cast<char4*>(q + (size_t)row * cols + c + 4) = hi;
  }
  if (threadIdx.x == 0) scale[row] = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f;
}

// Per token: dequantise the [q_rank + 576] accumulator row, RMSNorm of the
// q latent and of compressed_kv, requantise both, RoPE of k_pe.
__global__ void __launch_bounds__(256) norm_quant_kernel(const int32_t* __restrict__ acc1,
                                                         const float* __restrict__ sx,
                                                         W8Params p, W8Workspace w) {
  extern __shared__ float yrow[];  // [q_rank + 576]
  __shared__ float scratch[8];
  const int t = blockIdx.x;
  const int rq = p.q_rank, na = rq + kNa;
  const float s = sx[t];
  const int32_t* a = acc1 + (size_t)t * na;
  for (int c = threadIdx.x; c < na; c += 256) {
    const float sw = c < rq ? p.sW_qa[c] : p.sW_kva[c - rq];
    yrow[c] = __fmul_rn(__fmul_rn((float)a[c], s), sw);
  }
  __syncthreads();
  // q latent
  float ss = 0.f;
  for (int c = threadIdx.x; c < rq; c += 256) ss += yrow[c] * yrow[c];
  ss = block_reduce<false>(ss, scratch);
  const float invq = 1.0f / sqrtf(ss / (float)rq + p.eps);
  float amax = 0.f;
  const __nv_bfloat16* gq = static_cast<const __nv_bfloat16*>(p.gamma_q);
  for (int c = threadIdx.x; c < rq; c += 256) {
    const float v = yrow[c] * invq * __bfloat162float(gq[c]);
    yrow[c] = v;
    amax = fmaxf(amax, fabsf(v));
  }
  amax = block_reduce<true>(amax, scratch);
  {
    const float inv = amax > 0.f ? __fdiv_rn(127.0f, amax) : 0.f;
    for (int c = threadIdx.x; c < rq; c += 256) w.q1[(size_t)t * rq + c] = q8(yrow[c], inv);
    if (threadIdx.x == 0) w.s1[t] = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f;
  }
  // compressed_kv
  float* ck = yrow + rq;
  ss = 0.f;
  for (int c = threadIdx.x; c < kRank; c += 256) ss += ck[c] * ck[c];
  ss = block_reduce<false>(ss, scratch);
  const float invk = 1.0f / sqrtf(ss / (float)kRank + p.eps);
  amax = 0.f;
  const __nv_bfloat16* gk = static_cast<const __nv_bfloat16*>(p.gamma_kv);
  float nv[2];
  for (int i = 0; i < 2; ++i) {
    const int c = threadIdx.x + i * 256;
    nv[i] = ck[c] * invk * __bfloat162float(gk[c]);
    amax = fmaxf(amax, fabsf(nv[i]));
  }
  amax = block_reduce<true>(amax, scratch);
  {
    const float inv = amax > 0.f ? __fdiv_rn(127.0f, amax) : 0.f;
    for (int i = 0; i < 2; ++i) w.c1[(size_t)t * kRank + threadIdx.x + i * 256] = q8(nv[i], inv);
    if (threadIdx.x == 0) w.s2[t] = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f;
  }
  // RoPE of k_pe (raw columns 512..575 of the kv_a output)
  if (threadIdx.x < 32) {
    int pos = p.positions[t];
    if (pos < 0 || pos >= p.max_pos) {
      if (threadIdx.x == 0) atomicOr(p.status, kStatusBadPosition);
      pos = pos < 0 ? 0 : p.max_pos - 1;
    }
    const float* kp = ck + kRank;
    const int j = threadIdx.x;
    const float a0 = kp[2 * j], b0 = kp[2 * j + 1];
    const float* cr = p.cos_t + (size_t)pos * kRope;
    const float* sr = p.sin_t + (size_t)pos * kRope;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.k_pe) + (size_t)t * kRope;
    out[j] = __float2bfloat16_rn(a0 * cr[j] - b0 * sr[j]);
    out[j + 32] = __float2bfloat16_rn(b0 * cr[j + 32] + a0 * sr[j + 32]);
  }
}

// Dequantise q_b / kv_b accumulators and write the head-major outputs.
// mode 0: row = [H, 192] -> q_nope [b,H,s,128], RoPE(q_pe) [b,H,s,64]
// mode 1: row = [H, 256] -> k_nope [b,H,s,128], value [b,H,s,128]
// Grid (T, H); 64 threads, each 2 (mode 1: 4) columns.
__global__ void __launch_bounds__(64) head_epilogue_kernel(const int32_t* __restrict__ acc,
                                                           const float* __restrict__ srow,
                                                           const float* __restrict__ scol,
                                                           W8Params p, int mode) {
  const int t = blockIdx.x, hh = blockIdx.y, H = p.heads;
  const int bi = t / p.s, si = t - bi * p.s;
  const int width = mode == 0 ? kNope + kRope : kHeadCols;
  const size_t ld = (size_t)H * width;
  const int32_t* a = acc + (size_t)t * ld + (size_t)hh * width;
  const float* sc = scol + (size_t)hh * width;
  const float s = srow[t];
  const size_t orow = ((size_t)bi * H + hh) * p.s + si;
  const int j = threadIdx.x;  // 0..63
  auto deq = [&](int c) { return __fmul_rn(__fmul_rn((float)a[c], s), sc[c]); };
  if (mode == 0) {
    __nv_bfloat16* qn = static_cast<__nv_bfloat16*>(p.q_nope) + orow * kNope;
    qn[2 * j] = __float2bfloat16_rn(deq(2 * j));
    qn[2 * j + 1] = __float2bfloat16_rn(deq(2 * j + 1));
    if (j < 32) {
      int pos = p.positions[t];
      pos = pos < 0 ? 0 : (pos >= p.max_pos ? p.max_pos - 1 : pos);
      const float a0 = deq(kNope + 2 * j), b0 = deq(kNope + 2 * j + 1);
      const float* cr = p.cos_t + (size_t)pos * kRope;
      const float* sr = p.sin_t + (size_t)pos * kRope;
      __nv_bfloat16* qp = static_cast<__nv_bfloat16*>(p.q_pe) + orow * kRope;
      qp[j] = __float2bfloat16_rn(a0 * cr[j] - b0 * sr[j]);
      qp[j + 32] = __float2bfloat16_rn(b0 * cr[j + 32] + a0 * sr[j + 32]);
    }
  } else {
    __nv_bfloat16* kn = static_cast<__nv_bfloat16*>(p.k_nope) + orow * kNope;
    __nv_bfloat16* vv = static_cast<__nv_bfloat16*>(p.value) + orow * kV;
    kn[2 * j] = __float2bfloat16_rn(deq(2 * j));
    kn[2 * j + 1] = __float2bfloat16_rn(deq(2 * j + 1));
    vv[2 * j] = __float2bfloat16_rn(deq(kNope + 2 * j));
    vv[2 * j + 1] = __float2bfloat16_rn(deq(kNope + 2 * j + 1));
  }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int g_num_sms = 148;

// Small-M launch: 256-column blocks x K splits of at least 128 rows (32 per
// warp), aiming at about 4 CTAs per SM.
cudaError_t gemv(const int8_t* A, const int8_t* W, int M, int K, int N, int32_t* C, int ldc,
                 cudaStream_t st, int* launches) {
  const int tn = (N + 255) / 256;
  long per = ((long)K * tn + 4L * g_num_sms - 1) / (4L * g_num_sms);
  int kchunk = (int)((per + 63) / 64 * 64);
  if (kchunk < 128) kchunk = 128;
  if (kchunk > K) kchunk = (K + 15) / 16 * 16;
  const int splits = (K + kchunk - 1) / kchunk;
  if (splits > 1) {
    cudaError_t e = cudaMemset2DAsync(C, (size_t)ldc * 4, 0, (size_t)N * 4, M, st);
    if (e != cudaSuccess) return e;
    ++*launches;
  }
  dim3 grid(tn, splits);
  const int atomic = splits > 1 ? 1 : 0;
  if (M <= 1) gemv_s8_kernel<1><<<grid, 128, 0, st>>>(A, W, M, K, N, C, ldc, kchunk, atomic);
  else if (M <= 2) gemv_s8_kernel<2><<<grid, 128, 0, st>>>(A, W, M, K, N, C, ldc, kchunk, atomic);
  else if (M <= 4) gemv_s8_kernel<4><<<grid, 128, 0, st>>>(A, W, M, K, N, C, ldc, kchunk, atomic);
  else gemv_s8_kernel<8><<<grid, 128, 0, st>>>(A, W, M, K, N, C, ldc, kchunk, atomic);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t gemm(const int8_t* A, const int8_t* W, int M, int K, int N, int32_t* C, int ldc,
                 cudaStream_t st, int* launches) {
  // decode sizes stream the weights; the 64 x 64 tensor-core tiles would be
  // mostly padding rows
  if (M <= kGemvMaxRows && K % 16 == 0 && N % 8 == 0) return gemv(A, W, M, K, N, C, ldc, st, launches);
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
  if (splits > 1) {
    // split-K partials are added atomically: clear the N columns of each row
    cudaError_t e = cudaMemset2DAsync(C, (size_t)ldc * 4, 0, (size_t)N * 4, M, st);
    if (e != cudaSuccess) return e;
    ++*launches;
  }
  dim3 grid(tn, tm, splits);
  gemm_s8_kernel<<<grid, kGThreads, 0, st>>>(A, W, M, K, N, C, ldc, kchunk, splits > 1 ? 1 : 0);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace

size_t w8_workspace_bytes(int hidden, int q_rank, int heads, int max_tokens) {
  const size_t T = (size_t)max_tokens;
  const size_t nb = (size_t)heads * (kHeadCols > kNope + kRope ? kHeadCols : kNope + kRope);
  return align256(T * hidden) + align256(T * 4) + align256(T * (q_rank + kNa) * 4) +
         align256(T * q_rank) + align256(T * 4) + align256(T * kRank) + align256(T * 4) +
         align256(T * nb * 4);
}

void w8_workspace_carve(void* base, int hidden, int q_rank, int heads, int max_tokens,
                        W8Workspace* w) {
  const size_t T = (size_t)max_tokens;
  (void)heads;
  unsigned char* b = static_cast<unsigned char*>(base);
  w->xq = reinterpret_cast<int8_t*>(b); b += align256(T * hidden);
  w->sx = reinterpret_cast<float*>(b); b += align256(T * 4);
  w->acc1 = reinterpret_cast<int32_t*>(b); b += align256(T * (q_rank + kNa) * 4);
  w->q1 = reinterpret_cast<int8_t*>(b); b += align256(T * q_rank);
  w->s1 = reinterpret_cast<float*>(b); b += align256(T * 4);
  w->c1 = reinterpret_cast<int8_t*>(b); b += align256(T * kRank);
  w->s2 = reinterpret_cast<float*>(b); b += align256(T * 4);
  w->acc2 = reinterpret_cast<int32_t*>(b);
}

cudaError_t w8a8_quant_rows_launch(const void* x_bf16, int rows, int cols, int8_t* q,
                                   float* scale, cudaStream_t stream) {
  quant_rows_kernel<<<rows, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x_bf16), cols, q, scale);
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

cudaError_t w8a8_launch(const W8Params& p, const W8Workspace& w, int num_sms, cudaStream_t st,
                        int* launches) {
  g_num_sms = num_sms;
  *launches = 0;
  const int T = p.T, h = p.hidden_dim, rq = p.q_rank, H = p.heads;
  const int na = rq + kNa;
  cudaError_t e;
  // 1. quantise hidden rows
  quant_rows_kernel<<<T, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(p.hidden), h, w.xq, w.sx);
  ++*launches;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // 2. q_a_proj and kv_a_proj into one [T, q_rank + 576] accumulator
  if ((e = gemm(w.xq, p.W_qa, T, h, rq, w.acc1, na, st, launches)) != cudaSuccess) return e;
  if ((e = gemm(w.xq, p.W_kva, T, h, kNa, w.acc1 + rq, na, st, launches)) != cudaSuccess) return e;
  // 3-4. RMSNorms, requantisation, RoPE(k_pe)
  const size_t smem = (size_t)na * sizeof(float);
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(norm_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  norm_quant_kernel<<<T, 256, smem, st>>>(w.acc1, w.sx, p, w);
  ++*launches;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // 5. q_b_proj -> q_nope, RoPE(q_pe)
  if ((e = gemm(w.q1, p.W_qb, T, rq, H * (kNope + kRope), w.acc2, H * (kNope + kRope), st, launches)) != cudaSuccess) return e;
  head_epilogue_kernel<<<dim3(T, H), 64, 0, st>>>(w.acc2, w.s1, p.sW_qb, p, 0);
  ++*launches;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // 6. kv_b_proj -> k_nope, value
  if ((e = gemm(w.c1, p.W_kvb, T, kRank, H * kHeadCols, w.acc2, H * kHeadCols, st, launches)) != cudaSuccess) return e;
  head_epilogue_kernel<<<dim3(T, H), 64, 0, st>>>(w.acc2, w.s2, p.sW_kvb, p, 1);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace mla
