// Micro-benchmark of tcgen05.mma issue/execution throughput for the shapes the
// attention kernel uses. One CTA per SM; thread 0 issues `iters` groups of 8
// MMAs (K = 128) and times them with clock64 after a final commit.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
#include "ptx_sm103a.cuh"
using namespace flux;

template <int MODE>  // 0: SS M128 N128, 1: TS M128 N128 (A in TMEM), 2: SS M128 N256, 3: SS with precomputed descs
__global__ void __launch_bounds__(128, 1) bench(int iters, unsigned long long* out) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t slot;
  uint8_t* base = (uint8_t*)(((uintptr_t)smem + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_addr(base);
  for (int i = threadIdx.x; i < 128 * 1024 / 16; i += blockDim.x) ((uint4*)base)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) { mbar_init(smem_addr(&bar), 1); fence_mbar_init(); }
  if (threadIdx.x < 32) { tmem_alloc(smem_addr(&slot), 512); tmem_relinquish(); }
  fence_proxy_async_smem();
  tc_fence_before_sync(); __syncthreads(); tc_fence_after_sync();
  const uint32_t tmem = slot;
  volatile int abort_flag = 0;
  if (threadIdx.x == 0) {
    const uint32_t N = (MODE == 2) ? 256 : 128;
    const uint32_t idesc = idesc_bf16_f32(128, N, 0, 0);
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a = sb + (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint32_t b = sb + 32768 + (kk >> 2) * 16384 + (kk & 3) * 32;
        if (MODE == 1)
          mma_ts(tmem + 256, tmem + kk * 8, sdesc_sw128(b, 16, 1024), idesc, kk > 0);
        else
          mma_ss(tmem + ((it & 1) ? 256 : 0), sdesc_sw128(a, 16, 1024), sdesc_sw128(b, 16, 1024), idesc, kk > 0);
      }
    }
    mma_commit(smem_addr(&bar));
    mbar_wait(smem_addr(&bar), 0, &abort_flag);
    const long long t1 = clock64();
    out[blockIdx.x] = (unsigned long long)(t1 - t0);
  }
  tc_fence_before_sync(); __syncthreads();
  if (threadIdx.x < 32) { tc_fence_after_sync(); tmem_dealloc(tmem, 512); }
}

template <int MODE>
void run(const char* name, int sms) {
  unsigned long long* d; cudaMalloc(&d, sms * 8);
  auto k = bench<MODE>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 128 * 1024 + 1024);
  const int iters = 2000;
  k<<<sms, 128, 128 * 1024 + 1024>>>(100, d);
  cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
  cudaEventRecord(e0);
  k<<<sms, 128, 128 * 1024 + 1024>>>(iters, d);
  cudaEventRecord(e1); cudaEventSynchronize(e1);
  float ms; cudaEventElapsedTime(&ms, e0, e1);
  unsigned long long h[1024]; cudaMemcpy(h, d, sms * 8, cudaMemcpyDeviceToHost);
  double avg = 0; for (int i = 0; i < sms; ++i) avg += h[i]; avg /= sms;
  const double N = (MODE == 2) ? 256 : 128;
  const double flops = 2.0 * 128 * N * 128 * iters * sms;
  printf("%-28s cycles/MMA(K16) %7.1f  ideal %5.1f  TFLOP/s %8.1f  err=%s\n", name, avg / (iters * 8.0),
         128.0 * N * 16 * 2 / 8192.0, flops / (ms * 1e-3) / 1e12, cudaGetErrorString(cudaGetLastError()));
  cudaFree(d);
}

int main() {
  int sms = 0; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  run<0>("SS M128 N128", sms);
  run<1>("TS M128 N128 (A in TMEM)", sms);
  run<2>("SS M128 N256", sms);
  return 0;
}
