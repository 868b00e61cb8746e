// mma_sync_rates.cu -- throughput of the warp-level tensor-core path
// (mma.sync m16n8k16 f16 / bf16 and m16n8k32 s8) and of FFMA on the current
// GPU.  The library's W8A8 integer GEMMs run on mma.sync s8 (sm_103a has no
// tcgen05 int8 kind), so the s8 rate measured here is the compute roof used
// for the W8A8 workloads.  Each warp keeps 8 independent accumulators so the
// numbers are throughput, not latency.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
template <int KIND>
__global__ void k(float* out, int iters) {
  float acc[8][4] = {};
  int iacc[8][4] = {};
  uint32_t a[4] = {threadIdx.x, threadIdx.x * 3u, threadIdx.x * 5u, threadIdx.x * 7u};
  uint32_t b0 = threadIdx.x * 11u, b1 = threadIdx.x * 13u;
  float f[8] = {1.f, 2.f, 3.f, 4.f, 5.f, 6.f, 7.f, 8.f};
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (KIND == 0)
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                     : "+f"(acc[j][0]), "+f"(acc[j][1]), "+f"(acc[j][2]), "+f"(acc[j][3]) : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
      else if (KIND == 1)
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                     : "+f"(acc[j][0]), "+f"(acc[j][1]), "+f"(acc[j][2]), "+f"(acc[j][3]) : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
      else if (KIND == 2)
        asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                     : "+r"(iacc[j][0]), "+r"(iacc[j][1]), "+r"(iacc[j][2]), "+r"(iacc[j][3]) : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
      else {
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[j][q] = fmaf(acc[j][q], f[j], f[q]);
      }
    }
  }
  float s = 0;
  for (int j = 0; j < 8; ++j) for (int q = 0; q < 4; ++q) s += acc[j][q] + (float)iacc[j][q];
  if (s == 12345.f) out[threadIdx.x] = s;
}
int main() {
  int sms; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  float* o; cudaMalloc(&o, 4096);
  cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
  const char* names[] = {"mma.sync f16 m16n8k16", "mma.sync bf16 m16n8k16", "mma.sync s8 m16n8k32", "ffma (x4 per slot)"};
  for (int kind = 0; kind < 4; ++kind) {
    for (int warps : {4, 8, 16}) {
      int iters = 2000;
      dim3 grid(sms * 2), block(32 * warps);
      auto launch = [&]() {
        if (kind == 0) k<0><<<grid, block>>>(o, iters);
        else if (kind == 1) k<1><<<grid, block>>>(o, iters);
        else if (kind == 2) k<2><<<grid, block>>>(o, iters);
        else k<3><<<grid, block>>>(o, iters);
      };
      launch(); cudaDeviceSynchronize();
      cudaEventRecord(e0); launch(); cudaEventRecord(e1); cudaEventSynchronize(e1);
      float ms; cudaEventElapsedTime(&ms, e0, e1);
      double ops_per_inst = kind == 2 ? 2.0 * 16 * 8 * 32 : (kind == 3 ? 2.0 * 4 * 32 : 2.0 * 16 * 8 * 16);
      double total = ops_per_inst * 8 * iters * (double)grid.x * warps;
      printf("%-24s warps/CTA %2d: %8.1f T(FL)OP/s  (%.3f ms)\n", names[kind], warps, total / ms / 1e9, ms);
    }
  }
  printf("err: %s\n", cudaGetErrorString(cudaGetLastError()));
  return 0;
}
