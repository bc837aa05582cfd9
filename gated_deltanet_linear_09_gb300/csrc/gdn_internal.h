// gdn_internal.h -- declarations shared by the host API and the kernel translation units.
#pragma once

#include "gdn_common.cuh"

// NVTX ranges around the C-ABI calls: a profiler or tracer attached to the process sees each call
// as a named range on the calling thread (with none attached a range costs a few nanoseconds).
// Compiled out when the NVTX headers are not available.
#if defined(__has_include)
#if __has_include(<nvtx3/nvToolsExt.h>)
#include <nvtx3/nvToolsExt.h>
#define GDN_NVTX 1
#endif
#endif

namespace gdn {

struct CallRange {
  explicit CallRange(const char* name) {
#ifdef GDN_NVTX
    nvtxRangePushA(name);
#else
    (void)name;
#endif
  }
  ~CallRange() {
#ifdef GDN_NVTX
    nvtxRangePop();
#endif
  }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};
#define GDN_CALL_RANGE(name) ::gdn::CallRange gdn_call_range_(name)

int launch_decode(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                  const int32_t* slot_idx, int B, const void* qkv, const void* z, const void* a,
                  const void* b, void* out, cudaStream_t stream);

int launch_decode_multi(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                        const int32_t* slot_idx, int B, int TT, const void* qkv, const void* z,
                        const void* a, const void* b, void* out, cudaStream_t stream);

int launch_conv1d_update(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                         const int32_t* slot_idx, int B, const void* in, void* out,
                         cudaStream_t stream);

struct CompactPairs {
  int32_t src[GDN_MAX_COMPACT_PAIRS];
  int32_t dst[GDN_MAX_COMPACT_PAIRS];
};

int launch_compact(const CompactPairs& pairs, int n, void* rec, size_t rec_slot_bytes, void* conv,
                   size_t conv_slot_bytes, cudaStream_t stream);

// Workspace carve-up of the chunkwise prefill.
struct PrefillWs {
  float* qk;      // [T][Hk][2][dk]   l2-normalised q (scaled) and k
  float* vu;      // [T][Hv][dv]      v after conv+SiLU, then U~ = T diag(beta) V, then U
  float* w;       // [T][Hv][dk]      W = T diag(beta e^gamma) K
  float* gb;      // [T][Hv][2]       (g, beta), g replaced by the in-chunk cumulative gamma
  float* sc;      // [NCmax][Hv][dk][dv] state at the start of every chunk
  size_t bytes;
};

PrefillWs prefill_ws_layout(const KDims& d, int num_seqs, int total_tokens, void* base);

int launch_prefill(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                   const int32_t* cu_seqlens, const int32_t* slot_idx, const uint8_t* has_init,
                   int num_seqs, int total_tokens, const void* qkv, const void* z, const void* a,
                   const void* b, void* out, const PrefillWs& ws, cudaStream_t stream);

// Tensor-core (tcgen05) prefill for dk = dv = 128.
bool prefill_tc_supported(const KDims& d);
size_t prefill_tc_ws_bytes(const KDims& d, int num_seqs, int total_tokens);
// The smallest workspace the tensor-core prefill accepts: the records of one chunk.  Smaller
// workspaces than prefill_tc_ws_bytes run the call in windows of whole chunks.
size_t prefill_tc_ws_min_bytes(const KDims& d);
int launch_prefill_tc(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                      const int32_t* cu_seqlens, const int32_t* slot_idx, const uint8_t* has_init,
                      int num_seqs, int total_tokens, const void* qkv, const void* z, const void* a,
                      const void* b, void* out, void* ws, size_t ws_bytes, cudaStream_t stream);

// Dense bf16 projection (tcgen05 GEMM) with a routing epilogue: output feature n of row m goes
// to ptr[s][m * ld[s] + n - start[s]] for the segment s holding n.
struct ProjRoute {
  int nseg;
  int start[GDN_MAX_PROJ_SEGMENTS];
  int ld[GDN_MAX_PROJ_SEGMENTS];
  __nv_bfloat16* ptr[GDN_MAX_PROJ_SEGMENTS];
};

// Contraction split the library picks for an M x N x K projection (1 to 8).
int proj_auto_split(int M, int N, int K);
size_t proj_packed_bytes(int N, int K);
int launch_proj_pack(const void* w, int N, int K, void* packed, cudaStream_t stream);
int launch_proj(const void* x, const void* wp, int M, int N, int K, int ks, const ProjRoute& route,
                int32_t* status, cudaStream_t stream);

}  // namespace gdn
