/*
 * gdn.h -- C ABI of the GB300 (sm_103a) Gated DeltaNet layer library (libgdn.so).
 *
 * The layer is the linear-attention block of the Qwen3.5 / Qwen3-Next hybrid models:
 * a causal depthwise conv over the fused [q | k | v] projection channels, l2-normalised
 * q and k, per-V-head gates g = -exp(A_log) * softplus(a + dt_bias) and
 * beta = sigmoid(b), the gated delta rule on a per-request dk x dv recurrent state
 *     S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,   o_t = S_t^T q_t,
 * and a z-gated RMSNorm over each V-head's output.
 *
 * Where the operations are stated:
 *   "pegainfer issue #1001", Split 2 bullet -- one batched decode call over all decode rows
 *       through a step-scoped table of per-row state addresses (here: slot_idx);
 *   "pegainfer issue #1001", Split 3 bullet -- slot-indexed recurrent/conv state with a
 *       scheduler-owned slot index, device-to-device compaction on retire;
 *   "pegainfer PR #1003", description bullets -- rank-local head counts fed to the GDR
 *       decode / conv / chunkwise prefill chains, gated RMSNorm at the local value heads with
 *       a head-shared norm weight, linear-head divisibility failing closed, state and
 *       scratch sized from allocation bytes;
 *   "helexa/cortex commit 95dc874 (tp_qwen3_5)", TpQwen3_5GatedDeltaNet bullet -- the fused
 *       [q | k | v] channel regions (first key_dim, second key_dim, value_dim), the
 *       delta-rule loop per V-head, repeat_interleave of K-heads onto V-heads, l2norm,
 *       softplus and the RmsNormGated tail.
 *
 * Conventions shared by every call
 *   Ownership: the caller owns every buffer.  The library allocates and frees no memory,
 *     never synchronises the device and launches only on the given stream -- except the
 *     CUDA-graph decode object: gdn_decode_graphs_create allocates its static buffers and
 *     captures on an internal stream (synchronously), gdn_decode_graphs_destroy frees them.
 *   Launch order: the decode, multi-token decode, projection and compaction kernels (and a
 *     prefill call's kernels after its first) are launched as programmatic dependents of the
 *     previous kernel on the stream: their blocks may be placed on the GPU while that kernel
 *     finishes, but they read and write nothing that kernel could touch before it has completed
 *     and its writes are visible, so stream order holds as for any launch.
 *   Pointers: device pointers unless marked "host"; base addresses 16-byte aligned; all
 *     tensors dense, row-major, in the layouts below.
 *   Layouts (Cqkv = 2*Hk*dk + Hv*dv, r = Hv/Hk):
 *     rec_state  f32  [num_slots][Hv][dk][dv]        dv fastest
 *     conv_state act  [num_slots][K-1][Cqkv]         previous K-1 raw inputs, oldest first
 *     conv_weight act [Cqkv][K]                      tap K-1 multiplies the current token
 *     norm_weight act [dv]                           shared by all V-heads
 *     A_log, dt_bias f32 [Hv]
 *     qkv act [rows][Cqkv] channels [q heads | k heads | v heads], head-major in each region
 *     z act [rows][Hv*dv];  a, b act [rows][Hv];  out act [rows][Hv*dv]
 *     V-head h reads K-head h / r (repeat_interleave).
 *   Supported: dk, dv in {64, 128}; K = 4; act in {GDN_F32, GDN_BF16}; Hv % Hk == 0.
 *   Errors: negative return codes (below); nothing is launched when a call fails its host
 *     checks.  Errors found on the device (a slot index out of range) never trap: the row
 *     is skipped, its output zeroed, and a bit is OR-ed into *pool->status when that
 *     optional device word is given.
 *   Thread safety: no global mutable state beyond what the first call on a device sets up
 *     once (kernel attributes and device properties, under a once-only guard, read-only after);
 *     concurrent calls on different streams are safe when they touch disjoint slots and
 *     buffers.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Return codes. */
#define GDN_OK 0
#define GDN_ERR_INVALID_ARG (-1)         /* null pointer, negative size, bad eps, bad dtype   */
#define GDN_ERR_UNSUPPORTED_SHAPE (-2)   /* dk or dv not in {64,128}, K != 4                 */
#define GDN_ERR_HEAD_DIVISIBILITY (-3)   /* Hv % Hk != 0 (fails closed)                      */
#define GDN_ERR_SLOT_RANGE (-4)          /* a host-visible slot index outside [0, num_slots) */
#define GDN_ERR_WORKSPACE_TOO_SMALL (-5) /* workspace_bytes below the required size          */
#define GDN_ERR_OVERLAP (-6)             /* duplicate destination slot in a compaction       */
#define GDN_ERR_MISALIGNED (-7)          /* a base pointer not 16-byte aligned               */
#define GDN_ERR_CUDA (-8)                /* a CUDA launch failed (see cudaGetLastError)      */
#define GDN_ERR_TOO_LARGE (-9)           /* a size beyond a documented per-call maximum      */

/* Bits the kernels OR into *gdn_pool.status. */
#define GDN_STATUS_SLOT_RANGE 1
#define GDN_STATUS_BAD_SEQLENS 2
#define GDN_STATUS_TIMEOUT 4       /* a bounded device-side wait gave up; outputs are invalid */

/* Rank-local layer geometry ("local_linear_*" head counts of one tensor-parallel rank; one
 * GPU holds them all here).  q_scale = 0 selects 1/sqrt(head_k_dim).  l2norm divides by
 * sqrt(sum x^2 + l2_eps); the gated RMSNorm divides by sqrt(mean o^2 + norm_eps). */
typedef struct {
  int32_t num_k_heads;
  int32_t num_v_heads;
  int32_t head_k_dim;
  int32_t head_v_dim;
  int32_t conv_kernel;
  float q_scale;
  float l2_eps;
  float norm_eps;
} gdn_dims;

/* Layer parameters (device pointers, layouts above). */
typedef struct {
  const float* A_log;
  const float* dt_bias;
  const void* conv_weight;
  const void* norm_weight;
  gdn_dtype act;
} gdn_weights;

/* The per-request state pool.  status: optional device int32 error word (may be NULL). */
typedef struct {
  float* rec_state;
  void* conv_state;
  int32_t num_slots;
  int32_t* status;
} gdn_pool;

/* Bytes of one slot: recurrent state (f32) plus conv state (act dtype).  Capacity math of
 * "pegainfer PR #1003" (allocation bytes).  Returns 0 for unsupported geometry. */
size_t gdn_state_slot_bytes(const gdn_dims* dims, gdn_dtype act);

/* Standalone causal conv1d update (the "conv" chain of "pegainfer PR #1003"):
 *   qkv_out[i][c] = SiLU( sum_{j<K-1} w[c][j] * conv_state[s][j][c] + w[c][K-1] * qkv_in[i][c] )
 * with s = slot_idx[i] (device int32[B]); then the slot's conv state is shifted by one and
 * holds qkv_in[i] as its newest row.  Rows with s < 0 are padding: qkv_out row zeroed, no
 * state touched.  qkv_in / qkv_out: act [B][Cqkv].  Slots must be distinct across rows. */
int gdn_conv1d_update(const gdn_dims* dims, const gdn_weights* w, const gdn_pool* pool,
                      const int32_t* slot_idx, int32_t B, const void* qkv_in, void* qkv_out,
                      cudaStream_t stream);

/* One batched decode step over B rows (the batched GDR decode of "pegainfer issue #1001",
 * Split 2, with the slot-indexed state of Split 3): for row i with slot s = slot_idx[i]
 * (device int32[B], values distinct; s < 0 = padding row: output zeroed, no state read or
 * written), run conv update + SiLU, l2norm of q (times q_scale) and k, the gates, the gated
 * delta rule on every V-head's state rec_state[s][h], o = S_t^T q, and
 *   out = o / sqrt(mean(o^2) + norm_eps) * norm_weight * SiLU(z)  (one rounding to act).
 * qkv act [B][Cqkv]; z act [B][Hv*dv]; a, b act [B][Hv]; out act [B][Hv*dv].  B <= 65535.
 * qkv, z, a, b and out may be device memory or pinned host memory (any address the GPU can
 * reach through unified addressing): the kernel then reads the inputs and writes the output
 * over the CPU-GPU link itself, with no separate copies.  The state pool stays in device
 * memory.
 * One kernel launch; no host reads of device data, so the call can be captured in a CUDA
 * graph.  An out-of-range s sets GDN_STATUS_SLOT_RANGE and skips the row. */
int gdn_decode_step(const gdn_dims* dims, const gdn_weights* w, const gdn_pool* pool,
                    const int32_t* slot_idx, int32_t B, const void* qkv, const void* z,
                    const void* a, const void* b, void* out, cudaStream_t stream);

/* Largest number of tokens per row of one gdn_decode_multi call. */
#define GDN_MAX_DECODE_TOKENS 8

/* Multi-token decode (speculative verify / multi-token append; the decode step of "pegainfer
 * issue #1001", Split 2, run over T consecutive tokens per row): row i appends tokens
 * 0..T-1 in order to slot s = slot_idx[i], with the same result as T successive
 * gdn_decode_step calls, token t of every row in call t -- but each V-head state is read and
 * written once per call instead of once per token.  1 <= T <= GDN_MAX_DECODE_TOKENS.
 *   qkv  [B][T][Cqkv], z and out [B][T][Hv*dv], a and b [B][T][Hv], activation dtype, device,
 *        row-major; qkv, z, out 16-byte aligned.  slot_idx: device int32[B], distinct slots.
 *   On return the slot holds the state after token T-1 and its last K-1 raw inputs.
 * One kernel launch; no host reads of device data (graph-capturable).  An out-of-range s sets
 * GDN_STATUS_SLOT_RANGE and zeroes that row's outputs.  T outside [1, GDN_MAX_DECODE_TOKENS]:
 * GDN_ERR_INVALID_ARG, nothing launched. */
int gdn_decode_multi(const gdn_dims* dims, const gdn_weights* w, const gdn_pool* pool,
                     const int32_t* slot_idx, int32_t B, int32_t T, const void* qkv,
                     const void* z, const void* a, const void* b, void* out, cudaStream_t stream);

/* Bucketed CUDA-graph decode (the pages' CUDA-graph-versus-eager decode, "pegainfer issue
 * #1001", Split 3 bullet): gdn_decode_step captured once per batch bucket over static device
 * buffers owned by the object, so that a decode step is one padding memset and one graph
 * launch.  The object keeps the dims, weights and pool given at creation (their device memory
 * must outlive it).  Not thread-safe; one object per stream of decode steps. */
#define GDN_MAX_GRAPH_BUCKETS 16
typedef struct gdn_decode_graphs gdn_decode_graphs;

/* buckets: host int32[n_buckets], strictly increasing, each in [1, 65535]; 1 <= n_buckets <=
 * GDN_MAX_GRAPH_BUCKETS.  Allocates the static buffers for the largest bucket (slot_idx,
 * qkv, z, a, b, out in the gdn_decode_step layouts), runs one padding-row decode (touching no
 * state) and captures one graph per bucket on an internal stream; synchronous.  On success
 * *out is the new object; on error nothing is left allocated and *out is NULL.  Errors: the
 * host checks of gdn_decode_step, GDN_ERR_INVALID_ARG for bad buckets, GDN_ERR_TOO_LARGE for a
 * bucket above 65535, GDN_ERR_CUDA for a failed allocation or capture. */
int gdn_decode_graphs_create(const gdn_dims* dims, const gdn_weights* w, const gdn_pool* pool,
                             const int32_t* buckets, int32_t n_buckets, gdn_decode_graphs** out);

/* The static device buffers (each may be NULL to skip): the caller writes rows [0, B) of
 * slot_idx and of the inputs, launches, and reads rows [0, B) of out.  *max_batch = the largest
 * bucket. */
int gdn_decode_graphs_buffers(const gdn_decode_graphs* g, int32_t** slot_idx, void** qkv,
                              void** z, void** a, void** b, void** out, int32_t* max_batch);

/* One decode step of B rows on `stream`: sets slot_idx rows [B, bucket) to -1 (padding) for
 * the smallest bucket >= B and launches that bucket's graph.  The writes of the buffers must
 * be ordered before it on `stream`.  B = 0: no-op.  B above the largest bucket:
 * GDN_ERR_TOO_LARGE, nothing launched. */
int gdn_decode_graphs_launch(gdn_decode_graphs* g, int32_t B, cudaStream_t stream);

/* Frees the graphs and buffers (after the work launched from them has completed). */
void gdn_decode_graphs_destroy(gdn_decode_graphs* g);

/* Workspace bytes gdn_prefill_chunked needs for num_seqs sequences of total_tokens tokens
 * (the chunkwise scratch, "GdrChunkwiseScratch35" of "pegainfer PR #1003"). */
size_t gdn_prefill_workspace_bytes(const gdn_dims* dims, int32_t num_seqs, int32_t total_tokens);

/* Chunkwise prefill (the chunked prefill chain of "pegainfer PR #1003"): sequence n covers
 * packed tokens [cu_seqlens[n], cu_seqlens[n+1]) of qkv/z/a/b/out (device int32[num_seqs+1],
 * non-decreasing, cu_seqlens[0] = 0, cu_seqlens[num_seqs] = total_tokens) and runs every
 * token through the same layer as gdn_decode_step, in chunks of 64 tokens (WY / UT form of
 * the gated delta rule).  has_initial_state (device uint8[num_seqs], or NULL = all zero):
 * 0 starts from zero recurrent and conv state, 1 continues from slot slot_idx[n] (device
 * int32[num_seqs]).  On return the slot holds the state after the sequence's last token and
 * its last K-1 raw inputs.  workspace: device, 256-byte aligned, contents undefined on entry
 * and exit.  gdn_prefill_workspace_bytes(...) holds the records of every chunk at once and is
 * always enough.  With at most four V-heads per K-head (any head dims) the call runs on the
 * tensor cores in windows of whole 64-token chunks, each sequence's state carried from window to
 * window through its slot, with the same results for any window size; any workspace of at least
 * gdn_prefill_workspace_bytes(dims, 1, 1) bytes (one chunk's records for every V-head) is
 * accepted.  When the workspace holds two windows and the sequences' V-heads leave SMs free,
 * consecutive windows overlap on the GPU (programmatic dependent launch; a few tens of chunks'
 * records suffice for that).  More V-heads per K-head take CUDA-core kernels that need the full
 * size (GDN_ERR_WORKSPACE_TOO_SMALL otherwise).  Several kernels on `stream` (two per window
 * on the tensor-core path); no host reads of device data. */
int gdn_prefill_chunked(const gdn_dims* dims, const gdn_weights* w, const gdn_pool* pool,
                        const int32_t* cu_seqlens, const int32_t* slot_idx,
                        const uint8_t* has_initial_state, int32_t num_seqs, int32_t total_tokens,
                        const void* qkv, const void* z, const void* a, const void* b, void* out,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Size of the fixed device scratch array behind gdn_prefill_chunked_noalloc (64 MiB). */
#define GDN_NOALLOC_PREFILL_SCRATCH_BYTES (64u << 20)

/* Allocation-free variant of gdn_prefill_chunked (the pages have no counterpart: this serves
 * callers that cannot allocate device memory -- code running inside an allocator or memory
 * pool callback, a server that reserved all HBM for state slots at start-up, or a host
 * runtime that hands out raw pointers only).  Same arguments and results as
 * gdn_prefill_chunked minus the workspace: the scratch is a file-scope static __device__
 * array of GDN_NOALLOC_PREFILL_SCRATCH_BYTES that every GPU loading the library holds until
 * the process exits.  The call itself allocates and frees nothing.
 *   Size limit: returns GDN_ERR_TOO_LARGE, launching nothing, when
 *     gdn_prefill_workspace_bytes(dims, num_seqs, total_tokens) > GDN_NOALLOC_PREFILL_SCRATCH_BYTES.
 *   First call per device: looks up the array's device address (cudaGetSymbolAddress, with that
 *     device current) and caches it; make that first call before any stream capture.  With lazy
 *     module loading (the CUDA default) the driver creates the array at that lookup, so a caller
 *     that reserves the rest of device memory at start-up should first make one empty call
 *     (num_seqs = 0, total_tokens = 0) on each device.  The cached address belongs to the
 *     device's current context: a cudaDeviceReset between calls is not supported.
 *   Sharing: every call uses the same array, which keeps the last call's contents; the prefill
 *     writes every scratch value before it reads it, so nothing needs clearing.  Calls whose
 *     kernels overlap on the GPU (other streams, other host threads) race on the array:
 *     serialise them. */
int gdn_prefill_chunked_noalloc(const gdn_dims* dims, const gdn_weights* w, const gdn_pool* pool,
                                const int32_t* cu_seqlens, const int32_t* slot_idx,
                                const uint8_t* has_initial_state, int32_t num_seqs,
                                int32_t total_tokens, const void* qkv, const void* z,
                                const void* a, const void* b, void* out, cudaStream_t stream);

/* Maximum number of (src, dst) pairs of one gdn_state_compact call. */
#define GDN_MAX_COMPACT_PAIRS 2048

/* Device-to-device slot compaction on retire ("pegainfer issue #1001", Split 3):
 *   new[dst_slots[i]] = old[src_slots[i]]   for the recurrent and the conv state,
 * every source read before any destination is written, so source and destination sets may
 * overlap (e.g. gathering live slots into a prefix).  src_slots / dst_slots: HOST int32[n],
 * values in [0, num_slots), destinations distinct (GDN_ERR_OVERLAP otherwise), n <=
 * GDN_MAX_COMPACT_PAIRS (GDN_ERR_TOO_LARGE).  Slots that are no destination keep their bytes.
 * Bit-exact copy, one kernel launch, no workspace. */
int gdn_state_compact(const gdn_dims* dims, gdn_dtype act, const gdn_pool* pool,
                      const int32_t* src_slots, const int32_t* dst_slots, int32_t n,
                      cudaStream_t stream);

/* ---- Dense projections on either side of the step -----------------------------------------
 * The layer's input projection (the in_proj_qkv, in_proj_z, in_proj_b and in_proj_a weights)
 * and output projection (out_proj) of "pegainfer PR #1003", description bullets, and of
 * "helexa/cortex commit 95dc874 (tp_qwen3_5)", TpQwen3_5GatedDeltaNet bullet, as one bf16
 * tensor-core GEMM whose epilogue writes each output feature straight into the buffer that
 * consumes it.  The weights are packed once, at load time, into the kernel's tile layout. */
#define GDN_MAX_PROJ_SEGMENTS 4
#define GDN_PROJ_BLOCK_BYTES 16384

/* Bytes of a packed weight of N output features by K inputs: ceil(N/128) * 128 * K * 2.
 * Returns 0 unless N >= 1 and K is a positive multiple of 64. */
size_t gdn_proj_packed_bytes(int32_t N, int32_t K);

/* Packs a linear layer's weight w bf16 [N][K] (row n = output feature n, as stored) into the
 * tile layout gdn_linear_bf16 streams.  Block (nt, kc) -- features [128 nt, 128 nt + 128), inputs
 * [64 kc, 64 kc + 64) -- is GDN_PROJ_BLOCK_BYTES long at byte (nt * K/64 + kc) * 16384; inside it
 * element (r, k) sits at byte ((r/8) * 8 + k/8) * 128 + (r%8) * 16 + (k%8) * 2 (the K-major
 * core-matrix order of the MMA operand); features past N are zero.  w, packed: device, 16-byte
 * aligned, not overlapping; packed_bytes >= gdn_proj_packed_bytes(N, K)
 * (GDN_ERR_WORKSPACE_TOO_SMALL otherwise).  One kernel launch. */
int gdn_proj_pack(const void* w, int32_t N, int32_t K, void* packed, size_t packed_bytes,
                  cudaStream_t stream);

/* Where the output features of gdn_linear_bf16 go.  Segment s holds features
 * [start[s], start[s+1]) (the last one ends at N); feature n of row m is written to
 * ((bf16*)dst[s])[m * ld[s] + (n - start[s])].  1 <= nseg <= GDN_MAX_PROJ_SEGMENTS,
 * start[0] = 0, starts strictly increasing and below N, ld[s] >= the segment's width. */
typedef struct {
  int32_t nseg;
  int32_t start[GDN_MAX_PROJ_SEGMENTS];
  int32_t ld[GDN_MAX_PROJ_SEGMENTS];
  void* dst[GDN_MAX_PROJ_SEGMENTS];
} gdn_proj_route;

/* y = x w^T with one rounding to bf16:  y[m][n] = bf16( sum_k x[m][k] * w[n][k] ), summed in
 * f32, with w given packed (gdn_proj_pack).
 *   x bf16 [M][K], w_packed: device, 16-byte aligned.  K a positive multiple of 64
 *     (GDN_ERR_UNSUPPORTED_SHAPE otherwise); N >= 1; 0 <= M <= 4194240 (GDN_ERR_TOO_LARGE
 *     above); M = 0 returns GDN_OK after those checks, launching nothing and reading no
 *     other argument.  Destinations: device bf16, disjoint from x and w_packed.
 *   k_split: 0 lets the library choose; 1 to 8 splits the contraction over that many CTAs of
 *     a thread-block cluster whose f32 partial sums are added in a fixed order; part z takes
 *     the 64-wide chunks [z n / k_split, (z + 1) n / k_split) of the n = K / 64 (k_split <= n;
 *     GDN_ERR_INVALID_ARG otherwise).  For a given k_split the result is bitwise
 *     reproducible.
 *   status: optional device int32 word; GDN_STATUS_TIMEOUT is OR-ed in if a bounded wait
 *     inside the kernel gave up (the outputs are then invalid).
 * One kernel launch; no host reads of device data (graph-capturable). */
int gdn_linear_bf16(const void* x, const void* w_packed, int32_t M, int32_t N, int32_t K,
                    const gdn_proj_route* route, int32_t k_split, int32_t* status,
                    cudaStream_t stream);

/* Input projection of `rows` tokens (rows = B for gdn_decode_step, B*T for gdn_decode_multi,
 * the packed token count for gdn_prefill_chunked):
 *   hidden bf16 [rows][hidden_size];  w_in_packed = gdn_proj_pack of the bf16 weight
 *   [Cqkv + Hv*dv + 2*Hv][hidden_size] that stacks the rows of in_proj_qkv, in_proj_z,
 *   in_proj_b and in_proj_a in that order;
 *   writes qkv bf16 [rows][Cqkv], z bf16 [rows][Hv*dv], b bf16 [rows][Hv], a bf16 [rows][Hv]
 *   -- the input layouts of the step calls with act = GDN_BF16.
 * hidden_size a positive multiple of 64.  Geometry checks as for the step calls.  One launch of
 * gdn_linear_bf16's kernel with the library's k_split. */
int gdn_in_proj(const gdn_dims* dims, const void* hidden, const void* w_in_packed, int32_t rows,
                int32_t hidden_size, void* qkv, void* z, void* b, void* a, int32_t* status,
                cudaStream_t stream);

/* Output projection: y bf16 [rows][hidden_size] = out [rows][Hv*dv] * w_out^T, with out the
 * step's bf16 output and w_out_packed = gdn_proj_pack of out_proj's bf16 weight
 * [hidden_size][Hv*dv].  hidden_size >= 1.  One launch of gdn_linear_bf16's kernel with the
 * library's k_split. */
int gdn_out_proj(const gdn_dims* dims, const void* out, const void* w_out_packed, int32_t rows,
                 int32_t hidden_size, void* y, int32_t* status, cudaStream_t stream);

/* Text for a return code. */
const char* gdn_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
