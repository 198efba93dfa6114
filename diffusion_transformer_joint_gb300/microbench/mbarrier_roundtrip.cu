// Round-trip latency of the MMA -> softmax -> MMA hand-off through mbarriers.
// Thread 0 (warp 0) issues one 128x128x16 MMA and commits it to bar_s; a
// 128-thread "softmax" warpgroup waits on bar_s, then each warp's lane 0
// arrives on bar_p (count 4); thread 0 waits on bar_p and repeats. Cycles
// per iteration minus the MMA's 64 cycles is the hand-off round trip.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
#include "ptx_sm103a.cuh"
using namespace flux;

template <int WAIT>  // 0: try_wait loop (as the kernel), 1: test_wait spin
__device__ __forceinline__ void wait_phase(uint32_t bar, uint32_t parity) {
  if (WAIT == 0) {
    volatile int f = 0;
    mbar_wait(bar, parity, &f);
  } else {
    uint32_t done = 0;
    const long long t0 = clock64();
    while (!done && clock64() - t0 < kWaitBudgetCycles) {
      asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                   "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    }
  }
}

template <int WAIT>
__global__ void __launch_bounds__(256, 1) rt(int iters, unsigned long long* out) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_s, bar_p;
  __shared__ uint32_t slot;
  uint8_t* base = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_addr(base);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 64 * 1024 / 16; i += blockDim.x) ((uint4*)base)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) { mbar_init(smem_addr(&bar_s), 1); mbar_init(smem_addr(&bar_p), 4); fence_mbar_init(); }
  if (warp == 1) { tmem_alloc(smem_addr(&slot), 256); tmem_relinquish(); }
  fence_proxy_async_smem();
  tc_fence_before_sync(); __syncthreads(); tc_fence_after_sync();
  const uint32_t tmem = slot;
  const uint32_t bs = smem_addr(&bar_s), bp = smem_addr(&bar_p);
  if (tid == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
    const uint64_t da = sdesc_sw128(sb, 16, 1024), db = sdesc_sw128(sb + 32768, 16, 1024);
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
      mma_ss(tmem, da, db, idesc, 0);
      mma_commit(bs);
      wait_phase<WAIT>(bp, it & 1);
      tc_fence_after_sync();
    }
    out[blockIdx.x] = (unsigned long long)(clock64() - t0);
  } else if (warp >= 4) {
    for (int it = 0; it < iters; ++it) {
      wait_phase<WAIT>(bs, it & 1);
      tc_fence_after_sync();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bp);
    }
  }
  tc_fence_before_sync(); __syncthreads();
  if (warp == 1) { tc_fence_after_sync(); tmem_dealloc(tmem, 256); }
}

template <int WAIT>
void run(const char* name, int sms) {
  unsigned long long* d; cudaMalloc(&d, sms * 8);
  const int smem = 64 * 1024 + 1024;
  cudaFuncSetAttribute(rt<WAIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  rt<WAIT><<<sms, 256, smem>>>(100, d);
  rt<WAIT><<<sms, 256, smem>>>(4000, d);
  cudaDeviceSynchronize();
  unsigned long long h[1024]; cudaMemcpy(h, d, sms * 8, cudaMemcpyDeviceToHost);
  double avg = 0; for (int i = 0; i < sms; ++i) avg += h[i]; avg /= sms;
  printf("%-34s cycles per MMA + hand-off %7.1f  err=%s\n", name, avg / 4000.0,
         cudaGetErrorString(cudaGetLastError()));
  cudaFree(d);
}

int main() {
  int sms = 0; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  run<0>("try_wait loops (as in the kernel)", sms);
  run<1>("test_wait spin loops", sms);
  return 0;
}
