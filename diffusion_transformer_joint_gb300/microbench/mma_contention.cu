// Which concurrent load slows a stream of tcgen05.mma (SS, M128 N128 K16)?
// One CTA of 512 threads per SM: warp 0 lane 0 issues MMAs; warps 4..15 run
// a background load chosen by MODE. Reports cycles per MMA.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
#include "ptx_sm103a.cuh"
using namespace flux;

template <int MODE>  // 0 none, 1 FMA/ALU issue, 2 smem ld/st v4, 3 TMEM ld/st, 4 smem + FMA
__global__ void __launch_bounds__(512, 1) bench(int iters, unsigned long long* out, float* sink) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t slot;
  __shared__ volatile int stop;
  uint8_t* base = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_addr(base);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 192 * 1024 / 16; i += blockDim.x) ((uint4*)base)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) { mbar_init(smem_addr(&bar), 1); fence_mbar_init(); stop = 0; }
  if (warp == 1) { tmem_alloc(smem_addr(&slot), 512); tmem_relinquish(); }
  fence_proxy_async_smem();
  tc_fence_before_sync(); __syncthreads(); tc_fence_after_sync();
  const uint32_t tmem = slot;
  volatile int abort_flag = 0;
  if (warp == 0) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
      const long long t0 = clock64();
      for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t a = sb + (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint32_t b = sb + 32768 + (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tmem + ((it & 1) ? 128 : 0), sdesc_sw128(a, 16, 1024), sdesc_sw128(b, 16, 1024), idesc, kk > 0);
        }
      }
      mma_commit(smem_addr(&bar));
      mbar_wait(smem_addr(&bar), 0, &abort_flag);
      out[blockIdx.x] = (unsigned long long)(clock64() - t0);
      stop = 1;
    }
  } else if (warp >= 4) {
    float acc[8];
    for (int i = 0; i < 8; ++i) acc[i] = tid * 0.001f + i;
    const uint32_t region = sb + 65536 + (tid - 128) * 64;  // 24 KB x ... inside 192 KB
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int n = 0;
    while (!stop) {
      if (MODE == 1 || MODE == 4) {
#pragma unroll
        for (int r = 0; r < 32; ++r)
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(acc[i], 1.0001f, 0.5f);
      }
      if (MODE == 2 || MODE == 4) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          uint4 v = ld_shared_v4(region + ((r * 16) & 63));
          v.x += 1;
          st_shared_v4(region + ((r * 16 + 32) & 63), v);
        }
      }
      if (MODE == 3) {
        uint32_t r[32];
        tmem_ld32(tmem + 256 + lane_off, r);
        tmem_ld_wait();
        r[0] += 1;
        tmem_st32(tmem + 384 + lane_off, r);
        tmem_st_wait();
        acc[0] += __uint_as_float(r[5]);
      }
      ++n;
    }
    float s = 0; for (int i = 0; i < 8; ++i) s += acc[i];
    if (s == 1234.5f) sink[tid] = s + n;
  }
  tc_fence_before_sync(); __syncthreads();
  if (warp == 1) { tc_fence_after_sync(); tmem_dealloc(tmem, 512); }
}

template <int MODE>
void run(const char* name, int sms) {
  unsigned long long* d; cudaMalloc(&d, sms * 8);
  float* sink; cudaMalloc(&sink, 512 * 4);
  auto k = bench<MODE>;
  const int smem = 192 * 1024 + 1024;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  k<<<sms, 512, smem>>>(50, d, sink);
  k<<<sms, 512, smem>>>(2000, d, sink);
  cudaDeviceSynchronize();
  unsigned long long h[1024]; cudaMemcpy(h, d, sms * 8, cudaMemcpyDeviceToHost);
  double avg = 0; for (int i = 0; i < sms; ++i) avg += h[i]; avg /= sms;
  printf("%-34s cycles/MMA %7.1f (ideal 64)  err=%s\n", name, avg / (2000 * 8.0), cudaGetErrorString(cudaGetLastError()));
  cudaFree(d); cudaFree(sink);
}

int main() {
  int sms = 0; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  run<0>("MMA alone (512-thread CTA)", sms);
  run<1>("MMA + 12 warps FMA issue", sms);
  run<2>("MMA + 12 warps smem ld/st v4", sms);
  run<3>("MMA + 12 warps TMEM ld/st", sms);
  run<4>("MMA + 12 warps smem + FMA", sms);
  return 0;
}
