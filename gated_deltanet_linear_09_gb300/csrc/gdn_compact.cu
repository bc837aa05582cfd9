// gdn_compact.cu -- device-to-device slot compaction on retire (sm_103a).
//
// "pegainfer issue #1001", Split 3 bullet: slot-indexed per-request recurrent/conv state with
// D2D compaction on retire.  new[dst_i] = old[src_i] with read-before-write semantics.
//
// Every CTA owns one column range (a run of 16-byte units at the same offset inside every slot)
// and moves it for ALL pairs: it loads the range from every source slot into registers, passes
// a CTA barrier, then stores to every destination slot.  Different CTAs touch disjoint bytes, so
// overlapping source and destination sets (gathering live slots into a prefix, cycles) need no
// staging buffer and every byte is read once and written once.
#include "gdn_internal.h"

namespace gdn {

namespace {

constexpr int kCompactThreads = 256;
// 16-byte units held in registers per thread.  8 (a 32 KiB column tile per CTA over all pairs)
// moves the 56-pair compaction of the B=64 workload at the rate of a plain contiguous copy of
// the same bytes; 16 units per thread (fewer CTAs per SM) was ~16 % slower.
constexpr int kUnitsPerThread = 8;
constexpr int kUnitsPerCta = kCompactThreads * kUnitsPerThread;

__global__ void __launch_bounds__(kCompactThreads)
compact_kernel(const __grid_constant__ CompactPairs pairs, int n, uint4* __restrict__ rec,
               size_t rec_units, uint4* __restrict__ conv, size_t conv_units, int cols) {
  uint4* base = blockIdx.y == 0 ? rec : conv;
  const size_t units = blockIdx.y == 0 ? rec_units : conv_units;
  const size_t col0 = (size_t)blockIdx.x * cols;
  pdl_begin();   // the slots are read after the previous kernel of the stream has completed
  if (col0 >= units) return;
  const int ncol = (int)min((size_t)cols, units - col0);
  const int total = n * ncol;
  uint4 buf[kUnitsPerThread];
#pragma unroll
  for (int k = 0; k < kUnitsPerThread; ++k) {
    const int idx = threadIdx.x + k * kCompactThreads;
    if (idx < total) {
      const int p = idx / ncol, c = idx - p * ncol;
      buf[k] = __ldcs(base + (size_t)pairs.src[p] * units + col0 + c);
    }
  }
  __syncthreads();   // every source unit of this column range is read before any is written
#pragma unroll
  for (int k = 0; k < kUnitsPerThread; ++k) {
    const int idx = threadIdx.x + k * kCompactThreads;
    if (idx < total) {
      const int p = idx / ncol, c = idx - p * ncol;
      __stcs(base + (size_t)pairs.dst[p] * units + col0 + c, buf[k]);
    }
  }
}

}  // namespace

int launch_compact(const CompactPairs& pairs, int n, void* rec, size_t rec_slot_bytes, void* conv,
                   size_t conv_slot_bytes, cudaStream_t stream) {
  if (n <= 0) return GDN_OK;
  const size_t ru = rec_slot_bytes / 16, cu = conv_slot_bytes / 16;
  int cols = kUnitsPerCta / n;
  if (cols < 1) cols = 1;
  if (cols >= 32) cols &= ~31;   // whole 512-byte runs per pair when the pair count allows
  const size_t umax = ru > cu ? ru : cu;
  const size_t tiles = (umax + cols - 1) / cols;
  if (tiles > 0x7fffffffULL) return GDN_ERR_TOO_LARGE;
  // a programmatic dependent launch: the CTAs may be placed while the previous kernel of the
  // stream drains, and wait for it in the kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)tiles, 2);
  cfg.blockDim = dim3(kCompactThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, compact_kernel, pairs, n, static_cast<uint4*>(rec), ru,
                                           static_cast<uint4*>(conv), cu, cols);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn
