// gdn_proj.cu -- the dense projections on either side of the GDN step as one bf16 tcgen05 GEMM
// kernel: the input projection of the hidden states into the step's [q | k | v], z, b and a
// inputs, and the output projection of the gated-normed output back to the hidden size (the
// in_proj_qkv / in_proj_z / in_proj_b / in_proj_a and out_proj weights of "pegainfer PR #1003",
// description bullets, and of "helexa/cortex commit 95dc874 (tp_qwen3_5)",
// TpQwen3_5GatedDeltaNet bullet).
//
//   y[m][n] = bf16( sum_k x[m][k] w[n][k] ),   x [M][K] activations, w [N][K] weights.
//
// At decode batch sizes the weights are nearly all of the bytes, so the kernel is laid out for
// streaming them.  The weights are packed once (proj_pack_kernel) into 16 KiB blocks, each the
// exact shared-memory image of one 128-feature x 64-element tile in the MMA's K-major core-matrix
// layout, ordered so that the blocks of one feature tile are contiguous: a pipeline stage reads
// 16 KiB runs of consecutive bytes and DRAM sees long sequential streams instead of 128 scattered
// 128-byte row pieces.  A CTA owns 256 output features -- two weight tiles, each the MMA's M = 128
// operand with its own f32 accumulator in TMEM (lane = output feature, column = activation row)
// -- and 64 activation rows (N = 64), so one activation tile serves twice the weight bytes; it
// walks the contraction through a ring of shared-memory stages filled with cp.async.  When there
// are too few tiles to cover the SMs, the contraction is split over the CTAs of a thread-block
// cluster (grid z, any size up to 8); each CTA parks its partial tiles in its own shared memory
// and every CTA of the cluster adds up one slice of the columns over distributed shared memory,
// in a fixed order.  The epilogue routes each output feature to one of up to four destination
// tensors, which is how the input projection writes the step's four input buffers in one launch.
#include <mutex>

#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {

namespace {

constexpr int PM = 128;         // output features per weight tile (MMA M, TMEM lanes)
constexpr int PT = 2;           // weight tiles per CTA: 256 features share one activation tile
constexpr int PK = 64;          // contraction elements per stage
constexpr int PLAG = 1;         // a stage is refilled PLAG chunks after its MMAs were issued
constexpr int PTHREADS = 256;
constexpr uint32_t PA_BYTES = PM * PK * 2;   // one weight tile, 16 KiB
constexpr int PROWS_WIDE = 256;   // activation rows per CTA of the wide form
constexpr int WIDE_MIN_ROWS = 512;  // row counts from which an unsplit launch takes the wide form
static_assert(PA_BYTES == GDN_PROJ_BLOCK_BYTES, "a packed block is one weight tile's stage");
static_assert(PTHREADS == PT * PM, "the epilogue maps one thread to one output feature");

// Two forms of the kernel, by activation rows per CTA (the MMA's N, TMEM columns per tile):
//   PN = 64: decode batches; the weight bytes dominate; a 5-stage ring; the contraction can be
//     split over a cluster and reduced through distributed shared memory;
//   PN = 256: prefill-sized row counts; one N = 256 MMA costs ~160 cycles against ~109 for an
//     N = 64 one, so four times the rows per instruction run the tensor pipe faster and each
//     stage's bytes serve four times the FLOPs; 3 stages of 64 KiB; no split (there are tiles
//     enough for every SM).  (Six stages of 32 elements ran slower: the stage fill, not its
//     latency, is the limit.)
template <int PN_>
struct ProjCfg {
  static constexpr int PN = PN_;
  static constexpr int KS = 64;   // contraction elements per stage (32 is supported too)
  static constexpr int STAGES = PN_ == 64 ? 5 : 3;
  static constexpr int DIST = STAGES - PLAG;   // chunks in flight
  static constexpr uint32_t A_BYTES = PM * KS * 2;   // one weight tile's part of a stage
  static constexpr uint32_t B_BYTES = PN * KS * 2;   // activation tile
  static constexpr uint32_t STAGE_BYTES = PT * A_BYTES + B_BYTES;
  static constexpr uint32_t BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr uint32_t SMEM = BAR_OFF + STAGES * 8 + 16;
  static constexpr uint32_t RED_BYTES = PT * PM * PN * 4;   // f32 partial tiles (split only)
  static_assert(PN_ != 64 || RED_BYTES <= BAR_OFF, "partial tile must fit in the stage ring");
  static constexpr int X_COPIES = PN * (KS / 8) / PTHREADS;   // 16-byte activation copies
  static constexpr int W_UNITS = A_BYTES / 16 / PTHREADS;     // 16-byte weight copies per tile
  static_assert(X_COPIES * PTHREADS == PN * (KS / 8), "copies must divide evenly over the threads");
  static_assert(SMEM <= 227 * 1024, "one CTA per SM");
  static_assert(PT * PN <= 512, "both accumulators fit TMEM");
};

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(saddr), "l"(g),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// The activation tile of one stage (PN rows x PK) in the K-major no-swizzle core-matrix layout.
// Copy u covers row 8*(u/64) + u%8, elements 8*((u/8)%8) .. +8, which is byte u*16 of the tile:
// consecutive threads fill consecutive 16-byte slots (no shared-memory bank conflicts).  Rows past
// M are zero-filled (source size 0, address kept in range).
template <int PN>
__device__ __forceinline__ void load_x(uint32_t sb, const __nv_bfloat16* __restrict__ X, int M,
                                       int K, int m0, int k0) {
  constexpr int KG = ProjCfg<PN>::KS / 8;   // 16-byte units per row of the stage
#pragma unroll
  for (int i = 0; i < ProjCfg<PN>::X_COPIES; ++i) {
    const int u = (int)threadIdx.x + i * PTHREADS;
    const int m = m0 + ((u / (8 * KG)) << 3 | (u & 7));
    const __nv_bfloat16* src = X + (size_t)min(m, M - 1) * K + k0 + 8 * ((u >> 3) % KG);
    cp_async16(sb + (uint32_t)u * 16u, src, m < M ? 16u : 0u);
  }
}

// Packs w [N][K] into the block layout: block (nt, kc) = features [128 nt, 128 nt + 128) x
// elements [64 kc, 64 kc + 64) at byte (nt * K/64 + kc) * 16384; inside a block element (r, k) at
// byte ((r/8) * 8 + k/8) * 128 + (r%8) * 16 + (k%8) * 2; features past N are zero.  One thread
// writes one 16-byte unit (8 consecutive elements of one row), so the writes are coalesced.
__global__ void proj_pack_kernel(const __nv_bfloat16* __restrict__ W, int N, int K,
                                 uint4* __restrict__ P, long long units) {
  const int kcs = K / PK;
  for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < units;
       u += (long long)gridDim.x * blockDim.x) {
    const long long blk = u >> 10;
    const int v = (int)(u & 1023);
    const int nt = (int)(blk / kcs), kc = (int)(blk % kcs);
    const int n = nt * PM + (((v >> 6) << 3) | (v & 7));
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (n < N) val = *reinterpret_cast<const uint4*>(W + (size_t)n * K + kc * PK + 8 * ((v >> 3) & 7));
    P[u] = val;
  }
}

// One pipeline stage: chunk c of each of this CTA's weight tiles and the matching activation
// tile.  With 64-element stages chunk c is packed block c (a contiguous 16 KiB copy: 256 threads
// x 4 x 16 bytes, every warp reading 512 consecutive bytes); with 32-element stages it is half h
// = c % 2 of block c / 2, gathered into the stage's own 32-element K-major layout (unit u of the
// half: 8-row group u / 32, 16-byte column u / 8 % 4, row u % 8).  A second tile past the end of
// the packed weight is skipped.
template <int PN>
__device__ __forceinline__ void load_chunk(uint32_t sa, const unsigned char* __restrict__ wblk,
                                           size_t tile_stride, int ntiles,
                                           const __nv_bfloat16* __restrict__ X, int M, int K,
                                           int m0, int kbase, int c) {
  using C = ProjCfg<PN>;
#pragma unroll
  for (int t = 0; t < PT; ++t) {
    if (t < ntiles) {
#pragma unroll
      for (int i = 0; i < C::W_UNITS; ++i) {
        const uint32_t u = threadIdx.x + i * PTHREADS;
        size_t src;
        if constexpr (C::KS == PK) {
          src = (size_t)c * PA_BYTES + u * 16u;
        } else {
          const uint32_t half = (uint32_t)c & 1u;
          src = (size_t)(c >> 1) * PA_BYTES +
                (((u >> 5) * 8u + half * 4u + ((u >> 3) & 3u)) * 128u + (u & 7u) * 16u);
        }
        cp_async16(sa + t * C::A_BYTES + u * 16u, wblk + t * tile_stride + src, 16u);
      }
    }
  }
  load_x<PN>(sa + PT * C::A_BYTES, X, M, K, m0, kbase + c * C::KS);
}

// Grid (ceil(N/(PT*PM)), ceil(M/PN), ks), cluster (1, 1, ks): CTA z of a cluster takes contraction
// chunks [z*nk/ks, (z+1)*nk/ks) of the nk (rounded down: a split need not divide nk, the parts
// then differ by one chunk) and adds up columns [z*PN/ks, (z+1)*PN/ks) (rounded down) of the
// cluster's tile (ks = 1: a plain launch, no cluster).  One CTA per SM: the stage ring takes
// most of the shared memory and keeps PDIST chunks in flight.  Every thread copies its share of
// each stage; thread 0 issues the MMAs.  The CTAs of one launch walk their chunks from different
// starting points (a rotation by feature tile), so that they do not all read the same
// activation lines from L2 at the same moment.
template <int PN>
__global__ void __launch_bounds__(PTHREADS, 1)
proj_kernel(const __nv_bfloat16* __restrict__ X, const unsigned char* __restrict__ WP, int M,
            int N, int K, int nk, const ProjRoute route, int32_t* __restrict__ status) {
  using C = ProjCfg<PN>;
  constexpr int PSTAGES = C::STAGES, PDIST = C::DIST;
  constexpr uint32_t PSTAGE_BYTES = C::STAGE_BYTES, PBAR_OFF = C::BAR_OFF;
  extern __shared__ __align__(1024) unsigned char sm[];
  uint64_t* done = reinterpret_cast<uint64_t*>(sm + PBAR_OFF);   // the stage's MMAs completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + PSTAGES);
  const int n0 = blockIdx.x * PT * PM, m0 = blockIdx.y * PN;
  const int ks = (int)gridDim.z, z = (int)blockIdx.z;
  const int c0 = (int)((long long)z * nk / ks);                  // this CTA's first chunk
  const int nkc = (int)((long long)(z + 1) * nk / ks) - c0;      // and its chunk count (>= 1)
  const int kbase = c0 * C::KS;
  const int nt0 = blockIdx.x * PT, ntot = (N + PM - 1) / PM;
  const int ntiles = min(PT, ntot - nt0);   // weight tiles this CTA holds (the last may hold 1)
  const size_t tile_stride = (size_t)(K / PK) * PA_BYTES;
  const unsigned char* wblk = WP + (size_t)nt0 * tile_stride + (size_t)c0 * C::A_BYTES;
  const int rot = (int)(((unsigned long long)blockIdx.x * nkc / gridDim.x + blockIdx.y * 7ull) %
                        (unsigned)nkc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t s0 = tc::smem_u32(sm);
  if (tid == 0) {
    for (int i = 0; i < PSTAGES; ++i) tc::mbar_init(done + i, 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) tc::tmem_alloc(tslot, PT * PN);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = *tslot;
  // the setup above touches only this CTA's resources; the activations and the packed weights
  // are read after the previous kernel of the stream has completed
  pdl_begin();
  // step j of the walk reads chunk (j + rot) mod nkc
  auto chunk = [&](int j) { const int c = j + rot; return c < nkc ? c : c - nkc; };
  // the first PDIST steps in flight, one cp.async group each (empty groups included, so that the
  // group count stays in step with the step index)
#pragma unroll
  for (int j = 0; j < PDIST; ++j) {
    if (j < nkc)
      load_chunk<PN>(s0 + j * PSTAGE_BYTES, wblk, tile_stride, ntiles, X, M, K, m0, kbase, chunk(j));
    cp_async_commit();
  }
  constexpr uint32_t kIdesc = tc::idesc_bf16(PM, PN);
  bool ok = true;
  for (int kc = 0; kc < nkc; ++kc) {
    const int st = kc % PSTAGES;
    cp_async_wait<PDIST - 1>();     // this thread's copies of step kc landed ...
    tc::fence_proxy_async_smem();   // ... and are visible to the tensor core
    __syncthreads();
    if (tid == 0 && ok) {
      tc::fence_after_sync();
      const uint32_t sa = s0 + st * PSTAGE_BYTES;
      const uint64_t db = tc::kstep_desc(sa + PT * C::A_BYTES, C::KS, 0);
#pragma unroll
      for (int t = 0; t < PT; ++t) {
        if (t < ntiles) {
          const uint64_t da = tc::kstep_desc(sa + t * C::A_BYTES, C::KS, 0);
#pragma unroll
          for (int k = 0; k < C::KS / 16; ++k)
            tc::mma_bf16(tb + t * PN, tc::desc_add(da, 256u * k), tc::desc_add(db, 256u * k),
                         kIdesc, (kc > 0 || k > 0) ? 1u : 0u);
        }
      }
      tc::mma_commit(done + st);
    }
    // refill the stage of step kc - PLAG with step kc + PDIST once its MMAs are done: waiting
    // on MMAs issued PLAG iterations ago keeps the tensor pipe's latency off this loop
    const int nxt = kc + PDIST;
    if (nxt < nkc) {
      const int prev = kc - PLAG;
      if (prev >= 0 && ok && !tc::mbar_wait(done + prev % PSTAGES, (prev / PSTAGES) & 1))
        ok = false;
      if (ok)
        load_chunk<PN>(s0 + (nxt % PSTAGES) * PSTAGE_BYTES, wblk, tile_stride, ntiles, X, M, K, m0,
                       kbase, chunk(nxt));
    }
    cp_async_commit();
  }
  // the last chunk's commit covers every MMA issued before it
  if (ok && !tc::mbar_wait(done + (nkc - 1) % PSTAGES, ((nkc - 1) / PSTAGES) & 1)) ok = false;
  cp_async_wait<0>();
  ok = __syncthreads_and(ok) != 0;
  if (!ok && tid == 0 && status) atomicOr(status, GDN_STATUS_TIMEOUT);
  tc::fence_after_sync();
  // the destination of output feature n (thread -> TMEM lane of one tile)
  auto route_of = [&](int n, size_t& ld) {
    __nv_bfloat16* base = route.ptr[0];
    int seg_start = 0, seg_ld = route.ld[0];
#pragma unroll
    for (int q = 1; q < GDN_MAX_PROJ_SEGMENTS; ++q)
      if (q < route.nseg && n >= route.start[q]) {
        base = route.ptr[q];
        seg_start = route.start[q];
        seg_ld = route.ld[q];
      }
    ld = (size_t)seg_ld;
    return base + (n - seg_start);
  };
  if constexpr (PN == PROWS_WIDE) {
    // wide form: warp w reads TMEM lanes 32 (w % 4) .. of tile w / 4, 16 columns (rows) at a
    // time, and writes them straight out: a warp stores 32 consecutive features of a row
    const int lq = (warp & 3) * 32, t = warp >> 2;
    const int n = n0 + t * PM + lq + lane;
    size_t ld;
    __nv_bfloat16* dst = route_of(n, ld);
    if (ok) {
#pragma unroll 1
      for (int c0 = 0; c0 < PN; c0 += 16) {
        float v[16];
        tc::tmem_ld16(tc::taddr(tb, lq, t * PN + c0), v);
        if (n < N) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int m = m0 + c0 + i;
            if (m < M) dst[(size_t)m * ld] = __float2bfloat16_rn(v[i]);
          }
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tb, PT * PN);
  } else {
    // the partial tiles, [tile][column][lane] f32, into this CTA's stage ring (free now): warp w
    // holds TMEM lanes 32*(w%4).. of tile w/4 (columns 64*(w/4) ..)
    float* red = reinterpret_cast<float*>(sm);
    if (ok) {
      const int lq = (warp & 3) * 32, t = warp >> 2;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float v[32];
        tc::tmem_ld16(tc::taddr(tb, lq, t * PN + 32 * h), v);
        tc::tmem_ld16(tc::taddr(tb, lq, t * PN + 32 * h + 16), v + 16);
#pragma unroll
        for (int i = 0; i < 32; ++i) red[(t * PN + 32 * h + i) * PM + lq + lane] = v[i];
      }
    }
    const bool clustered = ks > 1;
    tc::fence_before_sync();
    if (clustered)
      tc::cluster_sync_all();   // every partial tile of the cluster is written and visible
    else
      __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tb, PT * PN);
    // this CTA's column slice: thread -> lane r = tid % 128 of tile tid / 128, every column
    const int r = tid & (PM - 1), tt = tid >> 7;
    const int n = n0 + tt * PM + r;
    const int cw0 = z * PN / ks, cw1 = (z + 1) * PN / ks;
    size_t ld;
    __nv_bfloat16* dst = route_of(n, ld);
    const uint32_t red_s = tc::smem_u32(red);
    for (int c = cw0; c < cw1; ++c) {
      const int m = m0 + c;
      if (m >= M || n >= N) continue;
      const int e = (tt * PN + c) * PM + r;
      float s;
      if (clustered) {
        s = 0.f;
        const uint32_t off = red_s + (uint32_t)e * 4u;
        for (int q = 0; q < ks; ++q) s += ld_cluster_f32(tc::mapa_shared(off, (uint32_t)q));
      } else {
        s = red[e];
      }
      dst[(size_t)m * ld] = __float2bfloat16_rn(s);
    }
    if (clustered) tc::cluster_sync_all();   // no CTA leaves while another reads its memory
  }
}

int g_num_sms = 0;

}  // namespace

// Clusters of c CTAs (one per SM) that can be resident at once, c = 1..8, read once per process:
// a cluster is placed inside one GPC, so the count is not simply SMs / c.  First done by the
// weight packing (before any projection, normally outside any graph capture).
int g_active_clusters[9] = {0};
void proj_init_once() {
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      g_num_sms = sms;
    else
      g_num_sms = 152;
    if (cudaFuncSetAttribute(proj_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ProjCfg<64>::SMEM) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    for (int c = 1; c <= 8; ++c) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(1, 1, (unsigned)c);
      cfg.blockDim = dim3(PTHREADS, 1, 1);
      cfg.dynamicSmemBytes = ProjCfg<64>::SMEM;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 1;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = (unsigned)c;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, proj_kernel<64>, &cfg) == cudaSuccess) g_active_clusters[c] = n;
      else cudaGetLastError();
    }
  });
}

int proj_auto_split(int M, int N, int K) {
  proj_init_once();
  const int* active = g_active_clusters;
  // one CTA per SM: split the contraction (into parts that may differ by one chunk) while every
  // cluster of the grid is resident at once (one wave) and every CTA keeps at least a full ring
  // of chunks
  constexpr int PN = ProjCfg<64>::PN;
  const long long tiles = (long long)((N + PT * PM - 1) / (PT * PM)) * ((M + PN - 1) / PN);
  const int nk = K / PK;
  int ks = 1;
  for (int c = 2; c <= 8; ++c) {
    // without the residency count (the query failed), only splits that divide nk, within the
    // SM count
    const long long fits = active[c] > 0 ? (long long)active[c]
                                         : (nk % c == 0 ? (long long)g_num_sms / c : 0);
    if (tiles <= fits && nk / c >= ProjCfg<64>::STAGES) ks = c;
  }
  return ks;
}

size_t proj_packed_bytes(int N, int K) { return (size_t)((N + PM - 1) / PM) * PM * (size_t)K * 2; }

int launch_proj_pack(const void* w, int N, int K, void* packed, cudaStream_t stream) {
  proj_init_once();
  const long long units = (long long)proj_packed_bytes(N, K) / 16;
  const int threads = 256;
  const long long want = (units + threads - 1) / threads;
  const int blocks = (int)(want < 4096 ? want : 4096);
  proj_pack_kernel<<<blocks, threads, 0, stream>>>(static_cast<const __nv_bfloat16*>(w), N, K,
                                                   static_cast<uint4*>(packed), units);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int launch_proj(const void* x, const void* wp, int M, int N, int K, int ks, const ProjRoute& route,
                int32_t* status, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(proj_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)ProjCfg<64>::SMEM);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(proj_kernel<PROWS_WIDE>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)ProjCfg<PROWS_WIDE>::SMEM);
  });
  if (attr_err != cudaSuccess) return GDN_ERR_CUDA;
  // unsplit launches over many rows take the wide form
  const bool wide = ks == 1 && M >= WIDE_MIN_ROWS;
  const int pn = wide ? PROWS_WIDE : ProjCfg<64>::PN;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((N + PT * PM - 1) / (PT * PM)), (unsigned)((M + pn - 1) / pn),
                     (unsigned)ks);
  cfg.blockDim = dim3(PTHREADS, 1, 1);
  cfg.dynamicSmemBytes = wide ? ProjCfg<PROWS_WIDE>::SMEM : ProjCfg<64>::SMEM;
  cfg.stream = stream;
  // a programmatic dependent launch (the CTAs may be set up while the previous kernel of the
  // stream drains); a cluster only with a split: nothing to exchange without one
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = (unsigned)ks;
  cfg.attrs = attr;
  cfg.numAttrs = ks > 1 ? 2 : 1;
  const int nk = K / (wide ? ProjCfg<PROWS_WIDE>::KS : PK);   // contraction chunks, split over ks
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  const unsigned char* wb = static_cast<const unsigned char*>(wp);
  const cudaError_t e =
      wide ? cudaLaunchKernelEx(&cfg, proj_kernel<PROWS_WIDE>, xb, wb, M, N, K, nk, route, status)
           : cudaLaunchKernelEx(&cfg, proj_kernel<64>, xb, wb, M, N, K, nk, route, status);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn
