// Throughput of the block-scaled FP4 MMA (tcgen05 kind::mxf4nvf4, M=128
// N=128 K=64, the attention kernel's S-MMA shape and descriptors) with
// operands resident in shared memory and the accumulator in tensor memory:
// one CTA per SM, one thread issuing `iters` x 2 MMAs back to back.  The
// operands and scales are zeros (the rate does not depend on the values).
// Prints one line per run and "ok"; every wait is bounded (a timeout sets the
// printed error flag).
#include <cstdio>
#include <cstdint>
#include <vector>
#include <cuda_runtime.h>
#include "../../quantized_attention_x16_gb300/csrc/sm100.cuh"

using namespace sa;

__device__ __forceinline__ uint64_t desc_qk(uint32_t saddr, uint32_t sbo, uint32_t swz) { return sdesc(saddr, 16, sbo, swz); }
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) { return sdesc(saddr, 0, 128, kSwizzleNone); }
__device__ __forceinline__ void copy_sf(uint32_t tcol, uint32_t saddr, int nblk) {
  for (int i = 0; i < nblk; ++i) tmem_cp_32x128b_warpx4(tcol + 4 * i, desc_sf(saddr + 512 * i));
}

constexpr int kSmem = 18 * 1024 + 1024;

__global__ void __launch_bounds__(128, 1) probe(int iters, unsigned long long* ns_out, unsigned long long* cyc_out,
                                                int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar;
  __shared__ uint32_t slot;
  __shared__ int abort_flag;
  for (int i = threadIdx.x; i < 18 * 1024 / 16; i += blockDim.x) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  fence_proxy_async_smem();
  __syncthreads();
  const int warp = threadIdx.x / 32;
  if (warp == 0) {
    tmem_alloc(&slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = slot;
  if (warp == 0) {
    const bool leader = elect_one();
    const uint32_t sb = smem_u32(smem);
    const uint32_t sA = sb, sB = sb + 8192, sfA = sb + 16384, sfB = sb + 17408;
    const uint32_t idesc = idesc_nvf4(128, 128);
    unsigned long long t0 = 0, c0 = 0;
    if (leader) {
      copy_sf(tbase + 256, sfA, 2);
      copy_sf(tbase + 264, sfB, 2);
      t0 = globaltimer_ns();
      c0 = clock64();
      for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          mma_nvf4(tbase, desc_qk(sA + kk * 32, 512, kSwizzle64B), desc_qk(sB + kk * 32, 512, kSwizzle64B), idesc,
                   tbase + 256 + 4 * kk, tbase + 264 + 4 * kk, (i | kk) ? 1u : 0u);
      }
      tc_commit(&bar);
    }
    __syncwarp();
    const bool ok = mbar_wait_warp(&bar, 0, &abort_flag, 2000000000ull);
    if (leader) {
      const unsigned long long t1 = globaltimer_ns(), c1 = clock64();
      ns_out[blockIdx.x] = t1 - t0;
      cyc_out[blockIdx.x] = c1 - c0;
      if (!ok) atomicExch(err, 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  unsigned long long *ns, *cyc;
  int* err;
  cudaMalloc(&ns, sms * 8);
  cudaMalloc(&cyc, sms * 8);
  cudaMalloc(&err, 4);
  cudaMemset(err, 0, 4);
  cudaFuncSetAttribute(probe, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  for (int iters : {2000, 20000, 40000}) {
    probe<<<sms, 128, kSmem>>>(iters, ns, cyc, err);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) { printf("cuda error %s\n", cudaGetErrorString(e)); return 1; }
    std::vector<unsigned long long> hn(sms), hc(sms);
    int he = 0;
    cudaMemcpy(hn.data(), ns, sms * 8, cudaMemcpyDeviceToHost);
    cudaMemcpy(hc.data(), cyc, sms * 8, cudaMemcpyDeviceToHost);
    cudaMemcpy(&he, err, 4, cudaMemcpyDeviceToHost);
    unsigned long long mx = 0, mc = 0;
    for (int i = 0; i < sms; ++i) { if (hn[i] > mx) mx = hn[i]; if (hc[i] > mc) mc = hc[i]; }
    const double flops = (double)sms * iters * 2 * (2.0 * 128 * 128 * 64);
    printf("iters %6d: %8.1f us  %8.1f TFLOP/s (whole GPU, slowest SM)  %.0f FLOP/clk/SM  clock %.0f MHz  err %d\n",
           iters, mx / 1e3, flops / (mx * 1e-9) / 1e12, (double)iters * 2 * (2.0 * 128 * 128 * 64) / mc,
           (double)mc / mx * 1e3, he);
  }
  printf("ok\n");
  return 0;
}
