// gdn_api.cu -- the extern "C" boundary of libgdn.so: host-side argument checks, then one or
// more kernel launches on the caller's stream.  The contract of every call is documented in
// include/gdn.h; this file only enforces it.
#include <math.h>

#include <vector>

#include "gdn_internal.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Geometry checks shared by every call.  Linear-head divisibility fails closed, as the
// tensor-parallel config of "pegainfer PR #1003" does.
int check_dims(const gdn_dims* dims, gdn::KDims* out) {
  if (!dims) return GDN_ERR_INVALID_ARG;
  const gdn_dims& d = *dims;
  if (d.num_k_heads <= 0 || d.num_v_heads <= 0) return GDN_ERR_INVALID_ARG;
  if (d.num_v_heads % d.num_k_heads != 0) return GDN_ERR_HEAD_DIVISIBILITY;
  if ((d.head_k_dim != 64 && d.head_k_dim != 128) || (d.head_v_dim != 64 && d.head_v_dim != 128))
    return GDN_ERR_UNSUPPORTED_SHAPE;
  if (d.conv_kernel != 4) return GDN_ERR_UNSUPPORTED_SHAPE;
  if (!(d.l2_eps >= 0.f) || !(d.norm_eps >= 0.f) || !(d.q_scale >= 0.f) || !isfinite(d.q_scale))
    return GDN_ERR_INVALID_ARG;
  const long long cqkv = 2LL * d.num_k_heads * d.head_k_dim + (long long)d.num_v_heads * d.head_v_dim;
  if (cqkv > (1LL << 30)) return GDN_ERR_TOO_LARGE;
  if (out) {
    out->Hk = d.num_k_heads;
    out->Hv = d.num_v_heads;
    out->dk = d.head_k_dim;
    out->dv = d.head_v_dim;
    out->K = d.conv_kernel;
    out->r = d.num_v_heads / d.num_k_heads;
    out->cqkv = (int)cqkv;
    out->q_scale = d.q_scale > 0.f ? d.q_scale : 1.0f / sqrtf((float)d.head_k_dim);
    out->l2_eps = d.l2_eps;
    out->norm_eps = d.norm_eps;
  }
  return GDN_OK;
}

size_t act_size(gdn_dtype t) { return t == GDN_BF16 ? 2 : 4; }
bool act_ok(gdn_dtype t) { return t == GDN_F32 || t == GDN_BF16; }

int check_weights(const gdn_weights* w) {
  if (!w || !act_ok(w->act)) return GDN_ERR_INVALID_ARG;
  if (!w->A_log || !w->dt_bias || !w->conv_weight || !w->norm_weight) return GDN_ERR_INVALID_ARG;
  if (!aligned16(w->conv_weight) || !aligned16(w->norm_weight)) return GDN_ERR_MISALIGNED;
  return GDN_OK;
}

int check_pool(const gdn_pool* p) {
  if (!p || !p->rec_state || !p->conv_state || p->num_slots <= 0) return GDN_ERR_INVALID_ARG;
  if (!aligned16(p->rec_state) || !aligned16(p->conv_state)) return GDN_ERR_MISALIGNED;
  return GDN_OK;
}

}  // namespace

extern "C" {

size_t gdn_state_slot_bytes(const gdn_dims* dims, gdn_dtype act) {
  gdn::KDims d;
  if (check_dims(dims, &d) != GDN_OK || !act_ok(act)) return 0;
  return sizeof(float) * (size_t)d.Hv * d.dk * d.dv + act_size(act) * (size_t)(d.K - 1) * d.cqkv;
}

int gdn_conv1d_update(const gdn_dims* dims, const gdn_weights* w, const gdn_pool* pool,
                      const int32_t* slot_idx, int32_t B, const void* qkv_in, void* qkv_out,
                      cudaStream_t stream) {
  GDN_CALL_RANGE("gdn_conv1d_update");
  gdn::KDims d;
  int rc;
  if ((rc = check_dims(dims, &d)) != GDN_OK) return rc;
  if (!w || !act_ok(w->act) || !w->conv_weight) return GDN_ERR_INVALID_ARG;
  if ((rc = check_pool(pool)) != GDN_OK) return rc;
  if (B < 0 || B > 65535) return B < 0 ? GDN_ERR_INVALID_ARG : GDN_ERR_TOO_LARGE;
  if (B == 0) return GDN_OK;
  if (!slot_idx || !qkv_in || !qkv_out) return GDN_ERR_INVALID_ARG;
  if (!aligned16(qkv_in) || !aligned16(qkv_out) || !aligned16(slot_idx)) return GDN_ERR_MISALIGNED;
  return gdn::launch_conv1d_update(d, w, pool, slot_idx, B, qkv_in, qkv_out, stream);
}

int gdn_decode_step(const gdn_dims* dims, const gdn_weights* w, const gdn_pool* pool,
                    const int32_t* slot_idx, int32_t B, const void* qkv, const void* z,
                    const void* a, const void* b, void* out, cudaStream_t stream) {
  GDN_CALL_RANGE("gdn_decode_step");
  gdn::KDims d;
  int rc;
  if ((rc = check_dims(dims, &d)) != GDN_OK) return rc;
  if ((rc = check_weights(w)) != GDN_OK) return rc;
  if ((rc = check_pool(pool)) != GDN_OK) return rc;
  if (B < 0 || B > 65535) return B < 0 ? GDN_ERR_INVALID_ARG : GDN_ERR_TOO_LARGE;
  if (B == 0) return GDN_OK;
  if (!slot_idx || !qkv || !z || !a || !b || !out) return GDN_ERR_INVALID_ARG;
  if (!aligned16(qkv) || !aligned16(z) || !aligned16(out) || !aligned16(slot_idx))
    return GDN_ERR_MISALIGNED;
  return gdn::launch_decode(d, w, pool, slot_idx, B, qkv, z, a, b, out, stream);
}

int gdn_decode_multi(const gdn_dims* dims, const gdn_weights* w, const gdn_pool* pool,
                     const int32_t* slot_idx, int32_t B, int32_t T, const void* qkv,
                     const void* z, const void* a, const void* b, void* out, cudaStream_t stream) {
  GDN_CALL_RANGE("gdn_decode_multi");
  gdn::KDims d;
  int rc;
  if ((rc = check_dims(dims, &d)) != GDN_OK) return rc;
  if ((rc = check_weights(w)) != GDN_OK) return rc;
  if ((rc = check_pool(pool)) != GDN_OK) return rc;
  if (T < 1 || T > GDN_MAX_DECODE_TOKENS) return GDN_ERR_INVALID_ARG;
  if (B < 0 || B > 65535) return B < 0 ? GDN_ERR_INVALID_ARG : GDN_ERR_TOO_LARGE;
  if (B == 0) return GDN_OK;
  if (!slot_idx || !qkv || !z || !a || !b || !out) return GDN_ERR_INVALID_ARG;
  if (!aligned16(qkv) || !aligned16(z) || !aligned16(out) || !aligned16(slot_idx))
    return GDN_ERR_MISALIGNED;
  return gdn::launch_decode_multi(d, w, pool, slot_idx, B, T, qkv, z, a, b, out, stream);
}

size_t gdn_prefill_workspace_bytes(const gdn_dims* dims, int32_t num_seqs, int32_t total_tokens) {
  gdn::KDims d;
  if (check_dims(dims, &d) != GDN_OK || num_seqs < 0 || total_tokens < 0) return 0;
  if (gdn::prefill_tc_supported(d)) return gdn::prefill_tc_ws_bytes(d, num_seqs, total_tokens);
  return gdn::prefill_ws_layout(d, num_seqs, total_tokens, nullptr).bytes;
}

int gdn_prefill_chunked(const gdn_dims* dims, const gdn_weights* w, const gdn_pool* pool,
                        const int32_t* cu_seqlens, const int32_t* slot_idx,
                        const uint8_t* has_initial_state, int32_t num_seqs, int32_t total_tokens,
                        const void* qkv, const void* z, const void* a, const void* b, void* out,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  GDN_CALL_RANGE("gdn_prefill_chunked");
  gdn::KDims d;
  int rc;
  if ((rc = check_dims(dims, &d)) != GDN_OK) return rc;
  if ((rc = check_weights(w)) != GDN_OK) return rc;
  if ((rc = check_pool(pool)) != GDN_OK) return rc;
  if (num_seqs < 0 || total_tokens < 0) return GDN_ERR_INVALID_ARG;
  if (num_seqs > 65535) return GDN_ERR_TOO_LARGE;
  if (num_seqs == 0) return total_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
  if (!cu_seqlens || !slot_idx) return GDN_ERR_INVALID_ARG;
  if (total_tokens > 0 && (!qkv || !z || !a || !b || !out)) return GDN_ERR_INVALID_ARG;
  if (total_tokens > 0 && (!aligned16(qkv) || !aligned16(z) || !aligned16(out)))
    return GDN_ERR_MISALIGNED;
  const bool tc = gdn::prefill_tc_supported(d);
  // the tensor-core path takes any workspace of at least one chunk's records (windows of whole
  // chunks); the CUDA-core path needs the full size
  const size_t need = tc ? gdn::prefill_tc_ws_min_bytes(d)
                         : gdn::prefill_ws_layout(d, num_seqs, total_tokens, nullptr).bytes;
  if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE_TOO_SMALL;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GDN_ERR_MISALIGNED;
  if (tc)
    return gdn::launch_prefill_tc(d, w, pool, cu_seqlens, slot_idx, has_initial_state, num_seqs,
                                  total_tokens, qkv, z, a, b, out, workspace, workspace_bytes, stream);
  const gdn::PrefillWs ws = gdn::prefill_ws_layout(d, num_seqs, total_tokens, workspace);
  return gdn::launch_prefill(d, w, pool, cu_seqlens, slot_idx, has_initial_state, num_seqs,
                             total_tokens, qkv, z, a, b, out, ws, stream);
}

int gdn_state_compact(const gdn_dims* dims, gdn_dtype act, const gdn_pool* pool,
                      const int32_t* src_slots, const int32_t* dst_slots, int32_t n,
                      cudaStream_t stream) {
  GDN_CALL_RANGE("gdn_state_compact");
  gdn::KDims d;
  int rc;
  if ((rc = check_dims(dims, &d)) != GDN_OK) return rc;
  if (!act_ok(act)) return GDN_ERR_INVALID_ARG;
  if ((rc = check_pool(pool)) != GDN_OK) return rc;
  if (n < 0) return GDN_ERR_INVALID_ARG;
  if (n > GDN_MAX_COMPACT_PAIRS) return GDN_ERR_TOO_LARGE;
  if (n == 0) return GDN_OK;
  if (!src_slots || !dst_slots) return GDN_ERR_INVALID_ARG;
  std::vector<unsigned char> seen((size_t)pool->num_slots, 0);
  gdn::CompactPairs pairs;
  for (int i = 0; i < n; ++i) {
    const int s = src_slots[i], t = dst_slots[i];
    if (s < 0 || s >= pool->num_slots || t < 0 || t >= pool->num_slots) return GDN_ERR_SLOT_RANGE;
    if (seen[(size_t)t]) return GDN_ERR_OVERLAP;
    seen[(size_t)t] = 1;
    pairs.src[i] = s;
    pairs.dst[i] = t;
  }
  const size_t rec_bytes = sizeof(float) * (size_t)d.Hv * d.dk * d.dv;
  const size_t conv_bytes = act_size(act) * (size_t)(d.K - 1) * d.cqkv;
  return gdn::launch_compact(pairs, n, pool->rec_state, rec_bytes, pool->conv_state, conv_bytes,
                             stream);
}

size_t gdn_proj_packed_bytes(int32_t N, int32_t K) {
  if (N < 1 || K < 1 || K % 64 != 0) return 0;
  return gdn::proj_packed_bytes(N, K);
}

int gdn_proj_pack(const void* w, int32_t N, int32_t K, void* packed, size_t packed_bytes,
                  cudaStream_t stream) {
  GDN_CALL_RANGE("gdn_proj_pack");
  if (!w || !packed || N < 1 || K < 1) return GDN_ERR_INVALID_ARG;
  if (K % 64 != 0) return GDN_ERR_UNSUPPORTED_SHAPE;
  if ((long long)N * K > (1LL << 40)) return GDN_ERR_TOO_LARGE;
  if (!aligned16(w) || !aligned16(packed)) return GDN_ERR_MISALIGNED;
  if (packed_bytes < gdn::proj_packed_bytes(N, K)) return GDN_ERR_WORKSPACE_TOO_SMALL;
  return gdn::launch_proj_pack(w, N, K, packed, stream);
}

int gdn_linear_bf16(const void* x, const void* w, int32_t M, int32_t N, int32_t K,
                    const gdn_proj_route* route, int32_t k_split, int32_t* status,
                    cudaStream_t stream) {
  GDN_CALL_RANGE("gdn_linear_bf16");
  if (M < 0 || N < 1 || K < 1) return GDN_ERR_INVALID_ARG;
  if (K % 64 != 0) return GDN_ERR_UNSUPPORTED_SHAPE;
  if (M > 65535 * 64) return GDN_ERR_TOO_LARGE;
  if (M == 0) return GDN_OK;   // empty batch: nothing read or written (x may be NULL)
  if (!x || !w || !route) return GDN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w)) return GDN_ERR_MISALIGNED;
  const gdn_proj_route& r = *route;
  if (r.nseg < 1 || r.nseg > GDN_MAX_PROJ_SEGMENTS || r.start[0] != 0) return GDN_ERR_INVALID_ARG;
  gdn::ProjRoute pr = {};
  pr.nseg = r.nseg;
  for (int s = 0; s < r.nseg; ++s) {
    const int end = s + 1 < r.nseg ? r.start[s + 1] : N;
    if (r.start[s] >= end || end > N || !r.dst[s] || r.ld[s] < end - r.start[s])
      return GDN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(r.dst[s]) & 1u) != 0) return GDN_ERR_MISALIGNED;
    pr.start[s] = r.start[s];
    pr.ld[s] = r.ld[s];
    pr.ptr[s] = static_cast<__nv_bfloat16*>(r.dst[s]);
  }
  const int nk = K / 64;
  if (k_split < 0 || k_split > 8) return GDN_ERR_INVALID_ARG;
  if (k_split > nk) return GDN_ERR_INVALID_ARG;   // every part takes at least one chunk
  const int ks = k_split != 0 ? k_split : gdn::proj_auto_split(M, N, K);
  return gdn::launch_proj(x, w, M, N, K, ks, pr, status, stream);
}

int gdn_in_proj(const gdn_dims* dims, const void* hidden, const void* w_in, int32_t rows,
                int32_t hidden_size, void* qkv, void* z, void* b, void* a, int32_t* status,
                cudaStream_t stream) {
  GDN_CALL_RANGE("gdn_in_proj");
  gdn::KDims d;
  int rc;
  if ((rc = check_dims(dims, &d)) != GDN_OK) return rc;
  if (!qkv || !z || !b || !a || hidden_size < 1) return GDN_ERR_INVALID_ARG;
  const long long zdim = (long long)d.Hv * d.dv;
  const long long n = d.cqkv + zdim + 2LL * d.Hv;
  if (n > (1LL << 30)) return GDN_ERR_TOO_LARGE;
  gdn_proj_route r = {};
  r.nseg = 4;
  r.start[0] = 0;
  r.start[1] = d.cqkv;
  r.start[2] = (int32_t)(d.cqkv + zdim);
  r.start[3] = (int32_t)(d.cqkv + zdim + d.Hv);
  r.ld[0] = d.cqkv;
  r.ld[1] = (int32_t)zdim;
  r.ld[2] = d.Hv;
  r.ld[3] = d.Hv;
  r.dst[0] = qkv;
  r.dst[1] = z;
  r.dst[2] = b;
  r.dst[3] = a;
  return gdn_linear_bf16(hidden, w_in, rows, (int32_t)n, hidden_size, &r, 0, status, stream);
}

int gdn_out_proj(const gdn_dims* dims, const void* out, const void* w_out, int32_t rows,
                 int32_t hidden_size, void* y, int32_t* status, cudaStream_t stream) {
  GDN_CALL_RANGE("gdn_out_proj");
  gdn::KDims d;
  int rc;
  if ((rc = check_dims(dims, &d)) != GDN_OK) return rc;
  if (!y || hidden_size < 1) return GDN_ERR_INVALID_ARG;
  gdn_proj_route r = {};
  r.nseg = 1;
  r.ld[0] = hidden_size;
  r.dst[0] = y;
  return gdn_linear_bf16(out, w_out, rows, hidden_size, d.Hv * d.dv, &r, 0, status, stream);
}

const char* gdn_status_string(int code) {
  switch (code) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument";
    case GDN_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (head dims must be 64 or 128, conv kernel 4)";
    case GDN_ERR_HEAD_DIVISIBILITY: return "num_v_heads is not a multiple of num_k_heads";
    case GDN_ERR_SLOT_RANGE: return "slot index out of range";
    case GDN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case GDN_ERR_OVERLAP: return "duplicate destination slot";
    case GDN_ERR_MISALIGNED: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case GDN_ERR_CUDA: return "CUDA launch failed";
    case GDN_ERR_TOO_LARGE: return "size beyond a per-call maximum";
    default: return "unknown status";
  }
}

}  // extern "C"
