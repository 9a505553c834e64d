// peak.cu -- measured instruction-pipe peaks of this GPU for the benchmark's integer
// rooflines (built as libmcpeak.so, apart from the emulator library).
//
// Every thread runs kChains independent dependency chains of one instruction, written
// in PTX that maps one to one onto a hardware instruction: lop3.b32 (ALU pipe),
// shf.r.wrap.b32 (ALU pipe) and mad.lo.u32 (integer multiply-add, FMA pipe).  The
// grid is a whole number of waves of resident CTAs on every SM; the rate is lane
// operations per second over the CUDA-event time of one launch.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr int kChains = 8;
constexpr int kThreads = 256;

template <int KIND>
__device__ __forceinline__ uint32_t step(uint32_t x, uint32_t y, uint32_t z) {
  uint32_t r;
  if constexpr (KIND == 0) asm volatile("lop3.b32 %0, %1, %2, %3, 0x96;" : "=r"(r) : "r"(x), "r"(y), "r"(z));
  else if constexpr (KIND == 1) asm volatile("shf.r.wrap.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(y), "r"(z));
  else asm volatile("mad.lo.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(y), "r"(z));
  return r;
}

template <int KIND>
__global__ void __launch_bounds__(kThreads) chains_kernel(int iters, uint32_t seed, uint32_t *sink) {
  uint32_t v[kChains];
  const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
#pragma unroll
  for (int c = 0; c < kChains; c++) v[c] = t * 2654435761u + c + seed;
  const uint32_t y = seed | 1u, z = seed >> 3;
  for (int i = 0; i < iters; i++) {
#pragma unroll
    for (int u = 0; u < 4; u++)
#pragma unroll
      for (int c = 0; c < kChains; c++) v[c] = step<KIND>(v[c], y, z);
  }
  uint32_t acc = 0;
#pragma unroll
  for (int c = 0; c < kChains; c++) acc ^= v[c];
  if (acc == 0x9E3779B9u) sink[0] = acc;      // keeps the chains live
}

template <int KIND>
int run(int iters, double *ops_per_s, uint32_t *sink) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chains_kernel<KIND>, kThreads, 0);
  const int grid = sms * (per_sm > 0 ? per_sm : 1) * 4;
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  chains_kernel<KIND><<<grid, kThreads>>>(iters / 8, 1u, sink);      // warm-up
  cudaEventRecord(e0);
  chains_kernel<KIND><<<grid, kThreads>>>(iters, 7u, sink);
  cudaEventRecord(e1);
  cudaEventSynchronize(e1);
  float ms = 0.f;
  cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (cudaGetLastError() != cudaSuccess || ms <= 0.f) return 2;
  *ops_per_s = (double)grid * kThreads * kChains * 4.0 * iters / (ms * 1e-3);
  return 0;
}

}  // namespace

// kind 0: lop3 (ALU pipe), 1: shf (ALU pipe), 2: mad.lo.u32 (FMA pipe).  sink: one
// device uint32.  Returns 0 and the rate in lane operations per second.
extern "C" int mcpeak_int_rate(int kind, int iters, uint32_t *sink, double *ops_per_s) {
  if (!sink || !ops_per_s || iters < 8) return 1;
  switch (kind) {
    case 0: return run<0>(iters, ops_per_s, sink);
    case 1: return run<1>(iters, ops_per_s, sink);
    case 2: return run<2>(iters, ops_per_s, sink);
    default: return 1;
  }
}
