// gdn_noalloc.cu -- an allocation-free variant of the chunkwise prefill.
//
// Some callers cannot call cudaMalloc at the point where they run a prefill: code that runs
// inside a memory pool or allocator callback, code that must not grow the device footprint
// after start-up (a serving process that reserved all HBM for slots up front), or code that
// only receives raw pointers from a host runtime that owns every allocation.  For them this
// file keeps the prefill's scratch in a fixed, file-scope device array: every GPU that loads
// the library holds GDN_NOALLOC_PREFILL_SCRATCH_BYTES for it until the process exits.
#include <mutex>

#include "gdn_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_prefill_scratch[GDN_NOALLOC_PREFILL_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the array's name
// is only a host-side stand-in, so the address is looked up once per device (with that device
// current) and cached.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return GDN_OK;
}

}  // namespace

extern "C" int gdn_prefill_chunked_noalloc(const gdn_dims* dims, const gdn_weights* w,
                                           const gdn_pool* pool, const int32_t* cu_seqlens,
                                           const int32_t* slot_idx,
                                           const uint8_t* has_initial_state, int32_t num_seqs,
                                           int32_t total_tokens, const void* qkv, const void* z,
                                           const void* a, const void* b, void* out,
                                           cudaStream_t stream) {
  GDN_CALL_RANGE("gdn_prefill_chunked_noalloc");
  if (num_seqs < 0 || total_tokens < 0) return GDN_ERR_INVALID_ARG;
  // The address comes first, so that even an empty call (no sequences) makes the driver create
  // the array on this device: with lazy module loading that happens on first use, and a caller
  // that reserves the rest of the device memory afterwards wants it to have happened already.
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != GDN_OK) return rc;
  const size_t need = gdn_prefill_workspace_bytes(dims, num_seqs, total_tokens);
  if (need == 0) return gdn_prefill_chunked(dims, w, pool, cu_seqlens, slot_idx, has_initial_state,
                                            num_seqs, total_tokens, qkv, z, a, b, out, nullptr, 0,
                                            stream);
  if (need > (size_t)GDN_NOALLOC_PREFILL_SCRATCH_BYTES) return GDN_ERR_TOO_LARGE;
  return gdn_prefill_chunked(dims, w, pool, cu_seqlens, slot_idx, has_initial_state, num_seqs,
                             total_tokens, qkv, z, a, b, out, scratch,
                             (size_t)GDN_NOALLOC_PREFILL_SCRATCH_BYTES, stream);
}
