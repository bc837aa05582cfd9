// gdn_graphs.cu -- bucketed CUDA-graph decode: one captured gdn_decode_step per batch bucket,
// over static device buffers that the caller fills in place.  The pages measure the whole-model
// version of this A/B (CUDA graph against eager decode, "pegainfer issue #1001", Split 3 bullet)
// and size the graph pool's reserve from the state bytes (same page, reserve bullet); here the
// graphs hold only the GDN decode launch, so a step costs one memset node for the padding rows
// and one graph launch instead of the host work of an eager call.
//
// A launch for B rows replays the smallest bucket >= B; its rows [B, bucket) get slot -1, which
// the decode kernel treats as padding (no state touched, zero output).
#include <new>

#include "gdn_internal.h"

struct gdn_decode_graphs {
  gdn_dims dims;
  gdn_weights w;
  gdn_pool pool;
  int32_t nb = 0;
  int32_t buckets[GDN_MAX_GRAPH_BUCKETS] = {};
  cudaGraph_t graph[GDN_MAX_GRAPH_BUCKETS] = {};
  cudaGraphExec_t exec[GDN_MAX_GRAPH_BUCKETS] = {};
  int32_t* slot = nullptr;
  void* qkv = nullptr;
  void* z = nullptr;
  void* a = nullptr;
  void* b = nullptr;
  void* out = nullptr;
};

namespace {

void release(gdn_decode_graphs* g) {
  for (int i = 0; i < GDN_MAX_GRAPH_BUCKETS; ++i) {
    if (g->exec[i]) cudaGraphExecDestroy(g->exec[i]);
    if (g->graph[i]) cudaGraphDestroy(g->graph[i]);
  }
  void* bufs[] = {g->slot, g->qkv, g->z, g->a, g->b, g->out};
  for (void* p : bufs)
    if (p) cudaFree(p);
  delete g;
}

}  // namespace

extern "C" {

int gdn_decode_graphs_create(const gdn_dims* dims, const gdn_weights* w, const gdn_pool* pool,
                             const int32_t* buckets, int32_t n_buckets, gdn_decode_graphs** out) {
  GDN_CALL_RANGE("gdn_decode_graphs_create");
  if (!out) return GDN_ERR_INVALID_ARG;
  *out = nullptr;
  if (!dims || !w || !pool || !buckets) return GDN_ERR_INVALID_ARG;
  if (n_buckets < 1 || n_buckets > GDN_MAX_GRAPH_BUCKETS) return GDN_ERR_INVALID_ARG;
  for (int i = 0; i < n_buckets; ++i) {
    if (buckets[i] < 1 || (i > 0 && buckets[i] <= buckets[i - 1])) return GDN_ERR_INVALID_ARG;
    if (buckets[i] > 65535) return GDN_ERR_TOO_LARGE;
  }
  // the geometry / weights / pool checks of the decode entry point, before anything is allocated
  int rc = gdn_decode_step(dims, w, pool, nullptr, 0, nullptr, nullptr, nullptr, nullptr, nullptr,
                           nullptr);
  if (rc != GDN_OK) return rc;

  gdn_decode_graphs* g = new (std::nothrow) gdn_decode_graphs;
  if (!g) return GDN_ERR_CUDA;
  g->dims = *dims;
  g->w = *w;
  g->pool = *pool;
  g->nb = n_buckets;
  for (int i = 0; i < n_buckets; ++i) g->buckets[i] = buckets[i];
  const size_t maxb = (size_t)buckets[n_buckets - 1];
  const size_t elt = w->act == GDN_BF16 ? 2 : 4;
  const size_t cqkv = 2 * (size_t)dims->num_k_heads * dims->head_k_dim +
                      (size_t)dims->num_v_heads * dims->head_v_dim;
  const size_t zrow = (size_t)dims->num_v_heads * dims->head_v_dim;
  if (cudaMalloc(reinterpret_cast<void**>(&g->slot), maxb * sizeof(int32_t)) != cudaSuccess ||
      cudaMalloc(&g->qkv, maxb * cqkv * elt) != cudaSuccess ||
      cudaMalloc(&g->z, maxb * zrow * elt) != cudaSuccess ||
      cudaMalloc(&g->a, maxb * dims->num_v_heads * elt) != cudaSuccess ||
      cudaMalloc(&g->b, maxb * dims->num_v_heads * elt) != cudaSuccess ||
      cudaMalloc(&g->out, maxb * zrow * elt) != cudaSuccess) {
    release(g);
    return GDN_ERR_CUDA;
  }
  cudaStream_t cs = nullptr;
  bool ok = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) == cudaSuccess;
  // defined contents, every slot padding; one eager launch of a padding row prepares the kernel
  // (attributes are set on first use, outside any capture) without touching a state
  ok = ok && cudaMemsetAsync(g->slot, 0xFF, maxb * sizeof(int32_t), cs) == cudaSuccess &&
       cudaMemsetAsync(g->qkv, 0, maxb * cqkv * elt, cs) == cudaSuccess &&
       cudaMemsetAsync(g->z, 0, maxb * zrow * elt, cs) == cudaSuccess &&
       cudaMemsetAsync(g->a, 0, maxb * dims->num_v_heads * elt, cs) == cudaSuccess &&
       cudaMemsetAsync(g->b, 0, maxb * dims->num_v_heads * elt, cs) == cudaSuccess;
  ok = ok && gdn_decode_step(dims, w, pool, g->slot, 1, g->qkv, g->z, g->a, g->b, g->out, cs) ==
                 GDN_OK;
  ok = ok && cudaStreamSynchronize(cs) == cudaSuccess;
  for (int i = 0; ok && i < n_buckets; ++i) {
    ok = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
    if (!ok) break;
    const int lrc = gdn_decode_step(dims, w, pool, g->slot, buckets[i], g->qkv, g->z, g->a, g->b,
                                    g->out, cs);
    cudaGraph_t graph = nullptr;
    const bool ended = cudaStreamEndCapture(cs, &graph) == cudaSuccess;
    g->graph[i] = graph;
    ok = ended && lrc == GDN_OK && graph &&
         cudaGraphInstantiate(&g->exec[i], graph, 0) == cudaSuccess;
  }
  if (cs) cudaStreamDestroy(cs);
  if (!ok) {
    cudaGetLastError();
    release(g);
    return GDN_ERR_CUDA;
  }
  *out = g;
  return GDN_OK;
}

int gdn_decode_graphs_buffers(const gdn_decode_graphs* g, int32_t** slot_idx, void** qkv,
                              void** z, void** a, void** b, void** out, int32_t* max_batch) {
  if (!g) return GDN_ERR_INVALID_ARG;
  if (slot_idx) *slot_idx = g->slot;
  if (qkv) *qkv = g->qkv;
  if (z) *z = g->z;
  if (a) *a = g->a;
  if (b) *b = g->b;
  if (out) *out = g->out;
  if (max_batch) *max_batch = g->buckets[g->nb - 1];
  return GDN_OK;
}

int gdn_decode_graphs_launch(gdn_decode_graphs* g, int32_t B, cudaStream_t stream) {
  GDN_CALL_RANGE("gdn_decode_graphs_launch");
  if (!g || B < 0) return GDN_ERR_INVALID_ARG;
  if (B > g->buckets[g->nb - 1]) return GDN_ERR_TOO_LARGE;
  if (B == 0) return GDN_OK;
  int i = 0;
  while (g->buckets[i] < B) ++i;
  const int32_t bucket = g->buckets[i];
  if (bucket > B &&
      cudaMemsetAsync(g->slot + B, 0xFF, (size_t)(bucket - B) * sizeof(int32_t), stream) != cudaSuccess)
    return GDN_ERR_CUDA;
  return cudaGraphLaunch(g->exec[i], stream) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

void gdn_decode_graphs_destroy(gdn_decode_graphs* g) {
  if (g) release(g);
}

}  // extern "C"
