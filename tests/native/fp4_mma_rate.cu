// Throughput of the block-scaled FP4 MMA (tcgen05 kind::mxf4nvf4, M=128,
// K=64 per instruction, N = 128 -- the attention kernel's S-MMA shape and
// descriptors -- and N = 256, the widest single-CTA shape) with operands
// resident in shared memory and the accumulator in tensor memory: one CTA per
// SM, one thread issuing `iters` x 2 MMAs back to back, no TMA.  The operands
// and scales are zeros (the rate does not depend on the values).  Prints one
// line per run and "ok"; every wait is bounded (a timeout sets the printed
// error flag).
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

// A: 128 rows x 64 bytes (K = 128, two 64-deep chunks, 64B swizzle); B: N
// rows likewise; scale blocks (512 bytes per 128 rows x 4 groups) after them.
template <int N>
struct Lay {
  static constexpr int kA = 0, kB = 8192, kSfA = kB + N * 64, kSfB = kSfA + 1024, kBytes = kSfB + (N / 128) * 1024;
};
constexpr int kSmem = Lay<256>::kBytes + 1024;

template <int N>
__global__ void __launch_bounds__(128, 1) probe(int iters, unsigned long long* ns_out, unsigned long long* cyc_out,
                                                int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar;
  __shared__ uint32_t slot;
  __shared__ int abort_flag;
  using Y = Lay<N>;
  for (int i = threadIdx.x; i < Y::kBytes / 16; i += blockDim.x) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
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
    const uint32_t sA = sb + Y::kA, sB = sb + Y::kB, sfA = sb + Y::kSfA, sfB = sb + Y::kSfB;
    const uint32_t idesc = idesc_nvf4(128, N);
    // tensor memory: the accumulator in columns [0, N), A scales at 256 (8
    // columns), B scales at 272 (8 columns per 128 rows of B)
    unsigned long long t0 = 0, c0 = 0;
    if (leader) {
      copy_sf(tbase + 256, sfA, 2);
      copy_sf(tbase + 272, sfB, 2 * (N / 128));
      t0 = globaltimer_ns();
      c0 = clock64();
      for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          mma_nvf4(tbase, desc_qk(sA + kk * 32, 512, kSwizzle64B), desc_qk(sB + kk * 32, 512, kSwizzle64B), idesc,
                   tbase + 256 + 4 * kk, tbase + 272 + 4 * kk, (i | kk) ? 1u : 0u);
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
  cudaFuncSetAttribute(probe<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  cudaFuncSetAttribute(probe<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  for (int n : {128, 256})
  for (int iters : {2000, 20000, 40000}) {
    if (n == 128) probe<128><<<sms, 128, kSmem>>>(iters, ns, cyc, err);
    else probe<256><<<sms, 128, kSmem>>>(iters, ns, cyc, err);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) { printf("cuda error %s\n", cudaGetErrorString(e)); return 1; }
    std::vector<unsigned long long> hn(sms), hc(sms);
    int he = 0;
    cudaMemcpy(hn.data(), ns, sms * 8, cudaMemcpyDeviceToHost);
    cudaMemcpy(hc.data(), cyc, sms * 8, cudaMemcpyDeviceToHost);
    cudaMemcpy(&he, err, 4, cudaMemcpyDeviceToHost);
    unsigned long long mx = 0, mc = 0;
    for (int i = 0; i < sms; ++i) { if (hn[i] > mx) mx = hn[i]; if (hc[i] > mc) mc = hc[i]; }
    const double per_mma = 2.0 * 128 * n * 64;
    const double flops = (double)sms * iters * 2 * per_mma;
    printf("M128 N%d K64 iters %6d: %8.1f us  %8.1f TFLOP/s (whole GPU, slowest SM)  %.0f FLOP/clk/SM  clock %.0f MHz  "
           "err %d\n",
           n, iters, mx / 1e3, flops / (mx * 1e-9) / 1e12, (double)iters * 2 * per_mma / mc, (double)mc / mx * 1e3, he);
  }
  printf("ok\n");
  return 0;
}
