// tc_selftest.cu -- test-only harness: one 128 x N x K GEMM through the library's tcgen05
// primitives (gdn_tc.cuh), so that the descriptor, layout and TMEM conventions the prefill
// kernels rely on are checked in isolation against a CPU product.
#include <cuda_runtime.h>

#include "gdn_tc.cuh"

using namespace gdn::tc;

// Two primitives the library does not use, kept here to measure them: a shared -> TMEM operand
// copy and an MMA reading its A operand from TMEM (with the A operand in TMEM the per-MMA cost
// at small N did not drop, so the prefill kernels keep both operands in shared memory).
// D[tmem] (+)= A[tmem] * B[smem]^T -- A (M = 128 rows on TMEM lanes 0-127, 16 bf16 of K packed
// in 8 columns per K-step) was put there by tmem_cp_128x256b.  Issued by one thread.
static __device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Asynchronous shared -> TMEM copy of one 128-row x 32-byte block (one K-step of a 128-row bf16
// operand in the K-major core-matrix layout the descriptor describes) to lanes 0-127, 8 columns
// from taddr.  Ordered with the MMAs the same thread issues afterwards; tracked by mma_commit.
static __device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t s_desc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;\n" ::"r"(taddr), "l"(s_desc) : "memory");
}


// B's K-direction core matrices are b_lbo bytes apart (128: the dense layout).
__global__ void tc_gemm_kernel(const float* __restrict__ A, const float* __restrict__ B,
                               float* __restrict__ D, int N, int K, int passes, uint32_t ncols,
                               uint32_t b_lbo, int* __restrict__ err) {
  extern __shared__ __align__(1024) unsigned char sm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* a_hi = sm;
  unsigned char* a_lo = a_hi + 128 * K * 2;
  unsigned char* b_hi = a_lo + 128 * K * 2;
  const uint32_t b_sbo = (uint32_t)(K / 8) * b_lbo, b_bytes = (uint32_t)(N / 8) * b_sbo;
  unsigned char* b_lo = b_hi + b_bytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(b_lo + b_bytes);
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
    *reinterpret_cast<__nv_bfloat16*>(b_hi + kmajor_off_p(r, k, b_lbo, b_sbo)) = h;
    *reinterpret_cast<__nv_bfloat16*>(b_lo + kmajor_off_p(r, k, b_lbo, b_sbo)) = l;
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
      mma_bf16(tbase, kstep_desc(ah, K, s), kstep_desc_p(bh, b_lbo, b_sbo, s), id, s > 0 ? 1u : 0u);
      if (passes == 3) {
        mma_bf16(tbase, kstep_desc(ah, K, s), kstep_desc_p(bl, b_lbo, b_sbo, s), id, 1u);
        mma_bf16(tbase, kstep_desc(al, K, s), kstep_desc_p(bh, b_lbo, b_sbo, s), id, 1u);
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

extern "C" int tc_gemm_p(const float* A, const float* B, float* D, int N, int K, int passes,
                         int b_lbo, int* err) {
  if (N < 16 || N > 256 || N % 16 || K < 16 || K % 16 || b_lbo < 128 || b_lbo % 16) return -1;
  uint32_t ncols = 32;
  while (ncols < (uint32_t)N) ncols <<= 1;
  const size_t b_bytes = (size_t)(N / 8) * (K / 8) * b_lbo;
  const size_t smem = (size_t)2 * 128 * K * 2 + 2 * b_bytes + 64;
  if (smem > 200 * 1024) return -1;
  if (cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return -2;
  tc_gemm_kernel<<<1, 128, smem>>>(A, B, D, N, K, passes, ncols, (uint32_t)b_lbo, err);
  if (cudaGetLastError() != cudaSuccess) return -3;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -4;
}

// The same GEMM with A moved into TMEM by tcgen05.cp (hi at columns [N, N + K/2), lo after it)
// and the MMAs reading A from TMEM.
__global__ void tc_gemm_ta_kernel(const float* __restrict__ A, const float* __restrict__ B,
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
    const uint32_t ta_hi = tbase + (uint32_t)N, ta_lo = ta_hi + (uint32_t)(K / 2);
    for (int s = 0; s < K / 16; ++s) {
      tmem_cp_128x256b(ta_hi + 8 * s, kstep_desc(ah, K, s));
      tmem_cp_128x256b(ta_lo + 8 * s, kstep_desc(al, K, s));
    }
    for (int s = 0; s < K / 16; ++s) {
      mma_bf16_ta(tbase, ta_hi + 8 * s, kstep_desc(bh, K, s), id, s > 0 ? 1u : 0u);
      if (passes == 3) {
        mma_bf16_ta(tbase, ta_hi + 8 * s, kstep_desc(bl, K, s), id, 1u);
        mma_bf16_ta(tbase, ta_lo + 8 * s, kstep_desc(bh, K, s), id, 1u);
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

extern "C" int tc_gemm_ta(const float* A, const float* B, float* D, int N, int K, int passes, int* err) {
  if (N < 16 || N > 256 || N % 16 || K < 16 || K % 16 || N + K > 512) return -1;
  uint32_t ncols = 32;
  while (ncols < (uint32_t)(N + K)) ncols <<= 1;
  const size_t smem = (size_t)2 * (128 + N) * K * 2 + 64;
  if (smem > 200 * 1024) return -1;
  if (cudaFuncSetAttribute(tc_gemm_ta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return -2;
  tc_gemm_ta_kernel<<<1, 128, smem>>>(A, B, D, N, K, passes, ncols, err);
  if (cudaGetLastError() != cudaSuccess) return -3;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -4;
}

// The same GEMM with A written into TMEM from registers: thread i of the four warps holds row i
// of A, splits it into bf16 hi / lo pairs (element 2c in the low half of column c) and stores
// them with tcgen05.st (hi at columns [N, N + K/2), lo after it), the way the prefill chain
// kernel puts its S^T and U^T operands in place; the MMAs read A from TMEM.
__global__ void tc_gemm_tast_kernel(const float* __restrict__ A, const float* __restrict__ B,
                                    float* __restrict__ D, int N, int K, int passes, uint32_t ncols,
                                    int* __restrict__ err) {
  extern __shared__ __align__(1024) unsigned char sm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* b_hi = sm;
  unsigned char* b_lo = b_hi + N * K * 2;
  uint64_t* bar = reinterpret_cast<uint64_t*>(b_lo + N * K * 2);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
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
  const uint32_t ta_hi = tbase + (uint32_t)N, ta_lo = ta_hi + (uint32_t)(K / 2);
  const float* arow = A + (size_t)(warp * 32 + lane) * K;
  for (int c0 = 0; c0 < K / 2; c0 += 16) {   // 16 columns = 32 elements of the row at a time
    uint32_t hw[16], lw[16];
    for (int p = 0; p < 16; ++p) split2_bf16(arow[2 * (c0 + p)], arow[2 * (c0 + p) + 1], hw[p], lw[p]);
    tmem_st16_nw(taddr(ta_hi, warp * 32, c0), reinterpret_cast<const float*>(hw));
    tmem_st16_nw(taddr(ta_lo, warp * 32, c0), reinterpret_cast<const float*>(lw));
  }
  tmem_wait_st();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (tid == 0) {
    const uint32_t id = idesc_bf16(128, N);
    const uint32_t bh = smem_u32(b_hi), bl = smem_u32(b_lo);
    for (int s = 0; s < K / 16; ++s) {
      mma_bf16_ta(tbase, ta_hi + 8 * s, kstep_desc(bh, K, s), id, s > 0 ? 1u : 0u);
      if (passes == 3) {
        mma_bf16_ta(tbase, ta_hi + 8 * s, kstep_desc(bl, K, s), id, 1u);
        mma_bf16_ta(tbase, ta_lo + 8 * s, kstep_desc(bh, K, s), id, 1u);
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

extern "C" int tc_gemm_tast(const float* A, const float* B, float* D, int N, int K, int passes,
                            int* err) {
  if (N < 16 || N > 256 || N % 16 || K < 32 || K % 32 || N + K > 512) return -1;
  uint32_t ncols = 32;
  while (ncols < (uint32_t)(N + K)) ncols <<= 1;
  const size_t smem = (size_t)2 * N * K * 2 + 64;
  if (smem > 200 * 1024) return -1;
  if (cudaFuncSetAttribute(tc_gemm_tast_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return -2;
  tc_gemm_tast_kernel<<<1, 128, smem>>>(A, B, D, N, K, passes, ncols, err);
  if (cudaGetLastError() != cudaSuccess) return -3;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -4;
}

// Issue cost of back-to-back MMAs: nmma M = 128, K = 16 bf16 MMAs into one accumulator (the K
// steps of a 128 x 128 A tile in turn), A from shared memory or from TMEM, then one commit and
// its wait; the smallest clock64 span over `reps` repetitions after the first.  The operands
// hold arbitrary bits: only the time is of interest.
__global__ void mma_cost_kernel(int N, int tmem_a, int nmma, int reps, long long* out, int* err) {
  extern __shared__ __align__(1024) unsigned char sm[];
  unsigned char* a = sm;             // 128 x 128 bf16
  unsigned char* b = sm + 32768;     // up to 256 x 128 bf16
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 32768 + 65536);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
  for (int i = threadIdx.x; i < (32768 + 65536) / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(sm)[i] = 0x3f803f80u;   // bf16 1.0 pairs
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (threadIdx.x < 32) tmem_alloc(slot, 512);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tb = *slot;
  if (threadIdx.x == 0) {
    const uint32_t id = idesc_bf16(128, N);
    const uint64_t da = kstep_desc(smem_u32(a), 128, 0), db = kstep_desc(smem_u32(b), 128, 0);
    const uint32_t ta = tb + 256;   // A in TMEM: 8 columns per K-step, columns 256 .. 319
    long long best = 1LL << 62;
    for (int r = 0; r < reps; ++r) {
      const long long t0 = clock64();
      for (int i = 0; i < nmma; ++i) {
        const int k = i & 7;
        if (tmem_a) mma_bf16_ta(tb, ta + 8 * k, desc_add(db, 256 * k), id, i > 0);
        else mma_bf16(tb, desc_add(da, 256 * k), desc_add(db, 256 * k), id, i > 0);
      }
      mma_commit(bar);
      if (!mbar_wait(bar, (uint32_t)(r & 1))) {
        atomicOr(err, 1);
        break;
      }
      const long long t1 = clock64();
      if (r > 0 && t1 - t0 < best) best = t1 - t0;
    }
    *out = best;
  }
  fence_before_sync();
  __syncthreads();
  if (threadIdx.x < 32) tmem_dealloc(tb, 512);
}

extern "C" int tc_mma_cost(int N, int tmem_a, int nmma, long long* out, int* err) {
  if (N < 16 || N > 256 || N % 16 || nmma < 1) return -1;
  const size_t smem = 32768 + 65536 + 64;
  if (cudaFuncSetAttribute(mma_cost_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return -2;
  mma_cost_kernel<<<1, 128, smem>>>(N, tmem_a, nmma, 20, out, err);
  if (cudaGetLastError() != cudaSuccess) return -3;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -4;
}

extern "C" int tc_gemm(const float* A, const float* B, float* D, int N, int K, int passes, int* err) {
  return tc_gemm_p(A, B, D, N, K, passes, 128, err);
}

// D = A B^T with the B operand MN-major: Bt (= B^T, [K][N] row-major) is stored the way the
// prefill keeps its token-row tiles (rows = k, 16-byte units of 8 consecutive n, 8-row groups
// (N/8) * 128 bytes apart) and the MMA reads it as B through an MN-major descriptor:
// N-direction core-matrix stride 128 bytes, K-direction (8 k) stride (N/8) * 128 bytes.
__global__ void tc_gemm_mnb_kernel(const float* __restrict__ A, const float* __restrict__ Bt,
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
  for (int idx = tid; idx < K * N; idx += blockDim.x) {
    const int k = idx / N, n = idx - k * N;   // Bt[k][n] = B[n][k]
    __nv_bfloat16 h, l;
    split_bf16(Bt[idx], h, l);
    *reinterpret_cast<__nv_bfloat16*>(b_hi + kmajor_off(k, n, N)) = h;
    *reinterpret_cast<__nv_bfloat16*>(b_lo + kmajor_off(k, n, N)) = l;
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
    const uint32_t id = idesc_bf16_bmn(128, N);
    const uint32_t ah = smem_u32(a_hi), al = smem_u32(a_lo), bh = smem_u32(b_hi), bl = smem_u32(b_lo);
    const uint32_t lbo = (uint32_t)(N / 8) * 128u;   // one K-step (16 k) = two 8-row groups
    for (int s = 0; s < K / 16; ++s) {
      const uint64_t dbh = sdesc(bh + 2u * lbo * (uint32_t)s, lbo, 128u);
      const uint64_t dbl = sdesc(bl + 2u * lbo * (uint32_t)s, lbo, 128u);
      mma_bf16(tbase, kstep_desc(ah, K, s), dbh, id, s > 0 ? 1u : 0u);
      if (passes == 3) {
        mma_bf16(tbase, kstep_desc(ah, K, s), dbl, id, 1u);
        mma_bf16(tbase, kstep_desc(al, K, s), dbh, id, 1u);
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

extern "C" int tc_gemm_mnb(const float* A, const float* Bt, float* D, int N, int K, int passes,
                           int* err) {
  if (N < 16 || N > 256 || N % 16 || K < 16 || K % 16) return -1;
  uint32_t ncols = 32;
  while (ncols < (uint32_t)N) ncols <<= 1;
  const size_t smem = (size_t)2 * (128 + N) * K * 2 + 64;
  if (smem > 200 * 1024) return -1;
  if (cudaFuncSetAttribute(tc_gemm_mnb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return -2;
  tc_gemm_mnb_kernel<<<1, 128, smem>>>(A, Bt, D, N, K, passes, ncols, err);
  if (cudaGetLastError() != cudaSuccess) return -3;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -4;
}

// Per-round exchange of one float per thread among the 4 CTAs of a cluster (per-token partial
// sums shared over distributed shared memory): every thread stores its value into slot
// [round & 1][own rank][thread] of all four CTAs with st.async (completing bytes on that CTA's
// mbarrier for the buffer), then waits for its own CTA's buffer to fill and sums the 4 slots.
// Thread 0 posts the expected byte count of round r + 1 before it sends round r.
__global__ void __cluster_dims__(4, 1, 1) cluster_xchg_kernel(int rounds, float* __restrict__ out,
                                                              int* __restrict__ err) {
  __shared__ float xbuf[2][4][64];
  __shared__ __align__(8) uint64_t xfull[2];
  const int t = threadIdx.x;
  const uint32_t rank = cluster_ctarank();
  if (t == 0) {
    mbar_init(&xfull[0], 1);
    mbar_init(&xfull[1], 1);
    mbar_fence_init();
    mbar_arrive_expect_tx(&xfull[0], 4 * 64 * 4);
  }
  cluster_sync_all();
  bool ok = true;
  for (int c = 0; c < rounds; ++c) {
    const int b = c & 1;
    if (t == 0 && c + 1 < rounds) {
      mbar_arrive_expect_tx(&xfull[(c + 1) & 1], 4 * 64 * 4);
      fence_acq_rel_cluster();
    }
    const float v = (float)(rank * 1000 + t) + 0.25f * (float)c;
#pragma unroll
    for (uint32_t r = 0; r < 4; ++r)
      st_async_f32(mapa_shared(smem_u32(&xbuf[b][rank][t]), r), v, mapa_shared(smem_u32(&xfull[b]), r));
    if (ok) ok = mbar_wait_cluster(&xfull[b], (uint32_t)(c >> 1) & 1u);
    float sum = 0.f;
#pragma unroll
    for (int r = 0; r < 4; ++r) sum += xbuf[b][r][t];
    out[((size_t)blockIdx.x * rounds + c) * 64 + t] = ok ? sum : -1.f;
  }
  if (!ok) atomicOr(err, 4);
  cluster_sync_all();
}

extern "C" int tc_cluster_xchg(int nclusters, int rounds, float* out, int* err) {
  if (nclusters < 1 || rounds < 1) return -1;
  cluster_xchg_kernel<<<4 * nclusters, 64>>>(rounds, out, err);
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
