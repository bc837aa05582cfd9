// tc_selftest.cu -- test-only harness: one 128 x N x K GEMM through the library's tcgen05
// primitives (gdn_tc.cuh), so that the descriptor, layout and TMEM conventions the prefill
// kernels rely on are checked in isolation against a CPU product.
#include <cuda_runtime.h>

#include "gdn_tc.cuh"

using namespace gdn::tc;

__global__ void tc_gemm_kernel(const float* __restrict__ A, const float* __restrict__ B,
                               float* __restrict__ D, int N, int K, int passes, uint32_t ncols,
                               int* __restrict__ err) {
  extern __shared__ __align__(1024) unsigned char sm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* a_hi = sm;
  unsigned char* a_lo = a_hi + 128 * K * 2;
  unsigned char* b_hi = a_lo + 128 * K * 2;
  unsigned char* b_lo = b_hi + N * K * 2;
  uint64_t* bar = reinterpret_cast<uint64_t*>(b_lo + N * K * 2);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
  for (int idx = tid; idx < 128 * K; idx += blockDim.x) {
    const int r = idx / K, k = idx - r * K;
    __nv_bfloat16 h, l;
    split_bf16(A[idx], h, l);
    *reinterpret_cast<__nv_bfloat16*>(a_hi + kmajor_off(r, k, K)) = h;
    *reinterpret_cast<__nv_bfloat16*>(a_lo + kmajor_off(r, k, K)) = l;
  }
  for (int idx = tid; idx < N * K; idx += blockDim.x) {
    const int r = idx / K, k = idx - r * K;
    __nv_bfloat16 h, l;
    split_bf16(B[idx], h, l);
    *reinterpret_cast<__nv_bfloat16*>(b_hi + kmajor_off(r, k, K)) = h;
    *reinterpret_cast<__nv_bfloat16*>(b_lo + kmajor_off(r, k, K)) = l;
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (warp == 0) tmem_alloc(slot, ncols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tbase = *slot;
  if (tid == 0) {
    const uint32_t id = idesc_bf16(128, N);
    const uint32_t ah = smem_u32(a_hi), al = smem_u32(a_lo), bh = smem_u32(b_hi), bl = smem_u32(b_lo);
    for (int s = 0; s < K / 16; ++s) {
      mma_bf16(tbase, kstep_desc(ah, K, s), kstep_desc(bh, K, s), id, s > 0 ? 1u : 0u);
      if (passes == 3) {
        mma_bf16(tbase, kstep_desc(ah, K, s), kstep_desc(bl, K, s), id, 1u);
        mma_bf16(tbase, kstep_desc(al, K, s), kstep_desc(bh, K, s), id, 1u);
      }
    }
    mma_commit(bar);
  }
  __syncwarp();
  const bool ok = mbar_wait(bar, 0);
  if (!ok && lane == 0) atomicOr(err, 1);
  fence_after_sync();
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 16) {
      float v[16];
      tmem_ld16(taddr(tbase, warp * 32, c0), v);
      for (int i = 0; i < 16; ++i) D[(size_t)(warp * 32 + lane) * N + c0 + i] = v[i];
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, ncols);
}

extern "C" int tc_gemm(const float* A, const float* B, float* D, int N, int K, int passes, int* err) {
  if (N < 16 || N > 256 || N % 16 || K < 16 || K % 16) return -1;
  uint32_t ncols = 32;
  while (ncols < (uint32_t)N) ncols <<= 1;
  const size_t smem = (size_t)2 * (128 + N) * K * 2 + 64;
  if (cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return -2;
  tc_gemm_kernel<<<1, 128, smem>>>(A, B, D, N, K, passes, ncols, err);
  if (cudaGetLastError() != cudaSuccess) return -3;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -4;
}

// A bounded wait that nothing completes: the mbarrier is initialised for one arrival that never
// comes, so the wait must give up after limit_ns and report it instead of hanging.
__global__ void mbar_timeout_kernel(unsigned long long limit_ns, int* __restrict__ status,
                                    unsigned long long* __restrict__ waited_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  const uint64_t t0 = globaltimer_ns();
  const bool ok = mbar_wait(&bar, 0, limit_ns);
  const uint64_t t1 = globaltimer_ns();
  if (threadIdx.x == 0) {
    *status = ok ? 0 : 4;
    *waited_ns = t1 - t0;
  }
}

extern "C" int tc_timeout_probe(unsigned long long limit_ns, int* status,
                                unsigned long long* waited_ns) {
  mbar_timeout_kernel<<<1, 32>>>(limit_ns, status, waited_ns);
  if (cudaGetLastError() != cudaSuccess) return -3;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -4;
}
