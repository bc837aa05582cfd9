// gdn_prefill_tc.cu -- chunkwise prefill on the sm_103a tensor cores (tcgen05 + TMEM), for
// head dims 128 and, zero-padded to 128, 64 (a zero channel adds nothing to the norms, the
// products or the state, so only the channel offsets, the state's strides, the output columns
// and the RMSNorm's 1/dv see the real dims).
//
// Same chunk algebra as the CUDA-core path (UT transform of the gated delta rule; Yang et al.,
// "Parallelizing Linear Transformers with the Delta Rule over Sequence Length", NeurIPS 2024,
// section 3; chunked prefill chain and its scratch from "pegainfer PR #1003"), arranged so that
// every tensor-core product has M = 128:
//
//   intra kernel (chunk x K-head, all in parallel, one CTA per SM):
//     conv + SiLU + l2norm + gates of the chunk's 64 tokens,
//     D1 = [K;Q] K^T (once per K-head)   -> A = beta_i e^{g_i-g_j} KK^T (j<i),  P = QK^T o Gamma
//     per V-head: T = (I + A)^{-1}       (16 x 16 blocks: diagonal inverses, then block rows)
//     D2 = [T diag(beta e^gamma) ; T diag(beta)] [K^T | V^T]   -> W (rows 0-63), U~ (rows 64-127)
//     writes [Q~ ; W] and [P ; K~^T] as split-bf16 operand images (Q~ = e^gamma Q,
//     K~ = e^{gamma_L - gamma} K), U~ (f32) and e^{gamma_L}
//   chain kernel (sequence x V-head, one CTA each, serial over the chunks; transposed products
//   with S^T and U^T as TMEM A operands and the records as B operands):
//     D3^T = S^T [Q~ ; W]^T              -> columns 0-63 (Q~ S)^T, 64-127 (W S)^T
//     U^T  = U~^T - (W S)^T
//     S^T <- e^{gamma_L} S^T + U^T K~ ;  D3^T[:, 0:64] += U^T P^T  (O^T = (Q~ S + P U)^T)
//     z-gated RMSNorm of O over dv -> out
//   The call runs in windows of chunks; a window's intra kernel runs beside the previous window's
//   chains (programmatic dependent launch).
//
// Precision: every product runs as three bf16 passes on split operands
// (x = hi + lo, hi = bf16(x), lo = bf16(x - hi): A_hi B_hi + A_hi B_lo + A_lo B_hi) with f32
// accumulation in TMEM, which keeps about 16 significant bits per operand.
#include <algorithm>

#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {

namespace {

constexpr int CH = 64;
constexpr int D = 128;

// Per (chunk, V-head) record of the workspace.  B3 and B4 are stored as the exact shared-memory
// images of the chain kernel's B operands (split bf16, K-major core-matrix layout, hi then lo),
// so the chain kernel brings each in with one bulk copy.  Offsets in bytes.
constexpr uint32_t R_B3 = 0;                     // [Q~ ; W] rows, 128 x 128: hi 32 KiB, lo 32 KiB
constexpr uint32_t R_B4 = R_B3 + 65536;          // [P ; K~^T] rows, 192 x 64: hi 24 KiB, lo 24 KiB
constexpr uint32_t R_UT = R_B4 + 49152;          // f32 U~, [token][column]
constexpr uint32_t R_SC = R_UT + 32768;          // f32 e^{gamma_L}
constexpr uint32_t REC_BYTES = R_SC + 256;       // 147,712 bytes (multiple of 256)
constexpr uint32_t B3_HALF = 32768, B4_HALF = 24576;

// Float index of U~ element (token t, column col) in its record: row-major, so that a warp of
// the chain kernel reading 32 consecutive columns of a token touches 32 consecutive floats.
__host__ __device__ constexpr int ut_index(int t, int col) { return t * D + col; }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(bar)) : "memory");
}

// Bounded wait shared by every thread of the CTA: after one timeout the CTA stops waiting and
// stops issuing work (control flow stays uniform so that every barrier is still reached).
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              int32_t* status) {
  if (*abort) return false;
  if (tc::mbar_wait(bar, parity)) return true;
  *abort = 1;
  set_status(status, GDN_STATUS_TIMEOUT);
  return false;
}

// Packs 8 floats as split bf16 hi / lo 16-byte units.
__device__ __forceinline__ void split8(const float* v, uint4& hi, uint4& lo) {
  tc::split2_bf16(v[0], v[1], hi.x, lo.x);
  tc::split2_bf16(v[2], v[3], hi.y, lo.y);
  tc::split2_bf16(v[4], v[5], hi.z, lo.z);
  tc::split2_bf16(v[6], v[7], hi.w, lo.w);
}

__device__ __forceinline__ void st_unit(unsigned char* tile, uint32_t off, const uint4& v) {
  *reinterpret_cast<uint4*>(tile + off) = v;
}

__device__ __forceinline__ void gst_unit(unsigned char* g, uint32_t off, const uint4& v) {
  *reinterpret_cast<uint4*>(g + off) = v;
}

// Warp-wide: global chunk -> (sequence, first token, length, the sequence's start and length, its
// slot and has_initial_state flag); false if cu_seqlens is invalid.  Each lane loads its
// sequence's slot and flag beside its cu_seqlens entries, so the lookup costs one round trip.
struct ChunkInfo {
  int seq, t0, len, seq_start, seq_len, slot, init;
};
__device__ bool find_chunk(const int32_t* __restrict__ cu, const int32_t* __restrict__ slot_idx,
                           const uint8_t* __restrict__ has_init, int num_seqs, int total, int c,
                           ChunkInfo& ci) {
  const int lane = threadIdx.x & 31;
  const int cu_first = __ldg(cu), cu_last = __ldg(cu + num_seqs);   // issued beside the loop's loads
  bool ok = true;
  int base = 0;
  ci.seq = -1;
  for (int n0 = 0; n0 < num_seqs; n0 += 32) {
    const int n = n0 + lane;
    int lo = 0, hi = 0, nch = 0, sl = -1, hinit = 0;
    if (n < num_seqs) {
      lo = __ldg(cu + n);
      hi = __ldg(cu + n + 1);
      sl = __ldg(slot_idx + n);
      hinit = has_init != nullptr ? (int)__ldg(has_init + n) : 0;
      if (hi < lo) ok = false;
      else nch = (hi - lo + CH - 1) / CH;
    }
    int incl = nch;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const bool mine = (n < num_seqs) && (c >= base + incl - nch) && (c < base + incl);
    const unsigned m = __ballot_sync(0xffffffffu, mine);
    if (m && ci.seq < 0) {
      const int src = __ffs(m) - 1;
      ci.seq = __shfl_sync(0xffffffffu, n, src);
      ci.seq_start = __shfl_sync(0xffffffffu, lo, src);
      const int hi_s = __shfl_sync(0xffffffffu, hi, src);
      const int ex = __shfl_sync(0xffffffffu, base + incl - nch, src);
      ci.slot = __shfl_sync(0xffffffffu, sl, src);
      ci.init = __shfl_sync(0xffffffffu, hinit, src);
      ci.seq_len = hi_s - ci.seq_start;
      ci.t0 = ci.seq_start + (c - ex) * CH;
      ci.len = min(CH, hi_s - ci.t0);
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  ok = ok && cu_first == 0 && cu_last == total;
  return __all_sync(0xffffffffu, ok);
}

__device__ bool seq_chunk_offset(const int32_t* __restrict__ cu, int num_seqs, int total, int seq,
                                 int& off) {
  const int lane = threadIdx.x & 31;
  bool ok = (__ldg(cu) == 0) && (__ldg(cu + num_seqs) == total);
  int acc = 0;
  for (int n0 = 0; n0 < num_seqs; n0 += 32) {
    const int n = n0 + lane;
    if (n < num_seqs) {
      const int lo = __ldg(cu + n), hi = __ldg(cu + n + 1);
      if (hi < lo) ok = false;
      else if (n < seq) acc += (hi - lo + CH - 1) / CH;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  off = acc;
  return __all_sync(0xffffffffu, ok);
}

// ================================================================== intra-chunk kernel
//
// One CTA per (chunk, K-head): the K-head's conv / l2norm of k and q and the product
// D1 = [K;Q] K^T are formed once and serve its r V-heads, which then run one after another
// (the next V-head's conv, A / P and inverse overlap the current V-head's MMAs).  Every input
// row the chunk needs (the k, q and v channels of its tokens plus three rows of history) and
// the conv weights stream into a shared-memory ring with asynchronous copies at the start, so
// the CTA pays one global-memory round trip instead of one per phase.

constexpr int AS = 68;    // row stride of the A / T matrix (16-byte aligned rows)
constexpr int NTI = 1024; // threads of the intra kernel (32 warps), one CTA per SM
constexpr int RMAX = 4;   // V-heads per K-head on the tensor-core path
constexpr int NROW = CH + 3;   // input rows per chunk: three of history, then the 64 tokens

// TMEM columns of the intra kernel (lanes 0-127): D1 = [K;Q] K^T, then per V-head the two
// row-major products of the A operand [T diag(beta e^gamma) ; T diag(beta)] (128 x 64) with
// K^T (W in lanes 0-63) and with V^T (U~ in lanes 64-127).
constexpr uint32_t TI_D1 = 0, TI_W = 128, TI_U = 256, TI_COLS = 512;

// Input ring: one slot per input tensor (k, q, then the V-heads' v), each NROW rows of 128
// channels followed by the 128 channels' conv weights; 4 slots of bf16 or 2 of f32.
template <typename T>
struct InRing {
  static constexpr uint32_t ROW = 128 * sizeof(T);
  static constexpr uint32_t PITCH = ROW + 16;   // one unit of padding: conflict-free column reads
  static constexpr uint32_t W_OFF = NROW * PITCH;
  static constexpr uint32_t SLOT = W_OFF + 128 * 4 * sizeof(T);
  static constexpr int NSLOT = 8 / (int)sizeof(T);
};
constexpr uint32_t IN_BYTES = 4 * InRing<__nv_bfloat16>::SLOT > 2 * InRing<float>::SLOT
                                  ? 4 * InRing<__nv_bfloat16>::SLOT : 2 * InRing<float>::SLOT;

// Shared memory (one CTA per SM):
//   A1  [K;Q] split-bf16 operand, 128 rows x 128 K: hi (K rows | Q rows) then lo     64 KiB
//   VT  V rows of the current V-head, 64 x 128 K, hi then lo                         32 KiB
//   B2  [T diag(beta e^gamma) ; T diag(beta)] rows, 128 x 64 K, hi then lo            32 KiB
//   IN  the input ring                                                             71 KiB
//   AT  f32 [64][AS]: A of the V-head, overwritten by T = (I + A)^{-1}               17 KiB
//   VEC f32 [RMAX][5][64]: per V-head gamma, beta, e^gamma, e^{gamma_L - gamma}, beta e^gamma
//   PART f32 [4][64]: per token, the four warps' partial sums of squares of the l2norm
struct IntraSmem {
  static constexpr uint32_t A1 = 0;
  static constexpr uint32_t K_HI = 0, Q_HI = 16384, K_LO = 32768, Q_LO = 49152;
  static constexpr uint32_t VT = 65536;
  static constexpr uint32_t B2 = VT + 32768;
  static constexpr uint32_t IN = B2 + 32768;
  static constexpr uint32_t AT = IN + IN_BYTES;
  static constexpr uint32_t VEC = AT + 4 * 64 * AS;
  static constexpr uint32_t PART = VEC + 4 * RMAX * 5 * 64;  // f32 [4][64] l2norm partial sums
  static constexpr uint32_t BAR = PART + 4 * 4 * 64;         // 2 mbarriers
  static constexpr uint32_t MISC = BAR + 16;                  // tmem slot, flags
  static constexpr uint32_t BYTES = MISC + 64;
};
static_assert(IntraSmem::BYTES <= 227 * 1024, "intra kernel shared memory");

__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(tc::smem_u32(sdst)), "l"(gsrc),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
// Waits until at most n of this thread's committed copy groups are still in flight (n <= 3).
__device__ __forceinline__ void cp_async_wait_pending(int n) {
  switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;\n" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;\n" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;\n" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 3;\n" ::: "memory"); break;
  }
}

// Issues (one commit group) the copies of the head's nreal (64 or 128) input channels [cb, cb +
// nreal) of the chunk into the 128 channels of a ring slot (the rest zero: a 64-dim head runs as a
// 128-dim one whose extra channels are zero): ring row m holds the raw input at position
// p0 - 3 + m of the sequence (p0 = the chunk's first position); positions before the sequence
// come from the slot's conv state when init, else zero; positions past the sequence are zero.
// Then the channels' conv weights (zero for the extra channels).
template <typename T>
__device__ __forceinline__ void ring_issue(const KDims& d, const T* __restrict__ qkv,
                                           const T* __restrict__ conv_w, const T* __restrict__ cs,
                                           bool init, int cb, int nreal, int seq_start, int seq_len,
                                           int p0, unsigned char* slot) {
  using R = InRing<T>;
  constexpr int UPR = R::ROW / 16;   // 16-byte units per row
  constexpr int CPU = 16 / (int)sizeof(T);   // channels per unit
  for (int q = threadIdx.x; q < NROW * UPR; q += NTI) {
    const int m = q / UPR, uu = q - m * UPR;
    const int p = p0 - 3 + m;
    const T* src = qkv;
    uint32_t bytes = 0;
    if (uu * CPU >= nreal) {
      // an extra channel of a 64-dim head: zero
    } else if (p >= 0 && p < seq_len) {
      src = qkv + (size_t)(seq_start + p) * d.cqkv + cb;
      bytes = 16;
    } else if (p < 0 && init) {
      src = cs + (size_t)(3 + p) * d.cqkv + cb;
      bytes = 16;
    }
    cp_async16(slot + m * R::PITCH + uu * 16, reinterpret_cast<const unsigned char*>(src) + (bytes ? uu * 16 : 0),
               bytes);
  }
  for (int q = threadIdx.x; q < (int)(128 * 4 * sizeof(T) / 16); q += NTI) {
    const bool real = q * 16 < nreal * 4 * (int)sizeof(T);
    cp_async16(slot + R::W_OFF + q * 16,
               reinterpret_cast<const unsigned char*>(conv_w + (size_t)cb * 4) + (real ? q * 16 : 0),
               real ? 16u : 0u);
  }
  cp_async_commit();
}

__device__ __forceinline__ void unpack_unit(const uint4& u, float* f, __nv_bfloat16*) {
  const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q[i]));
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void unpack_unit(const uint4& u, float* f, float*) {
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z);
  f[3] = __uint_as_float(u.w);
}

// Thread layout of the conv: token t = 8 (warp % 8) + lane % 8 and the 8 channels
// [8 cg, 8 cg + 8), cg = 4 (warp / 8) + lane / 8.  A warp holds 8 consecutive tokens x 32
// channels, so its ring reads (padded rows) and its 16-byte stores into K-major tiles (8
// distinct rows per 128-byte line) are free of bank conflicts.
__device__ __forceinline__ int conv_t() { return 8 * ((threadIdx.x >> 5) & 7) + (threadIdx.x & 7); }
__device__ __forceinline__ int conv_cg() { return 4 * (threadIdx.x >> 8) + ((threadIdx.x >> 3) & 3); }

// y[e] = SiLU(sum_j w[c][j] x[t - 3 + j][c]), c = 8 cg + e, from a ring slot (zero past L).
// The four input rows and the weights of one 16-byte unit are read packed and unpacked channel
// by channel (few registers live at once).
template <typename T>
__device__ __forceinline__ void conv_slot(const unsigned char* slot, int L, float* y) {
  using R = InRing<T>;
  constexpr int CPU = 16 / (int)sizeof(T);   // channels per 16-byte unit (8 bf16, 4 f32)
  constexpr int UPT = 8 / CPU;               // units per thread
  const int t = conv_t(), cg = conv_cg();
#pragma unroll
  for (int u = 0; u < UPT; ++u) {
    const int unit = cg * UPT + u;
    uint4 wq[4], xq[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) wq[q] = *reinterpret_cast<const uint4*>(slot + R::W_OFF + unit * 64 + q * 16);
#pragma unroll
    for (int m = 0; m < 4; ++m) xq[m] = *reinterpret_cast<const uint4*>(slot + (t + m) * R::PITCH + unit * 16);
    const T* wv = reinterpret_cast<const T*>(wq);   // [channel][tap]
    const T* xv = reinterpret_cast<const T*>(xq);   // [row][channel]
#pragma unroll
    for (int e = 0; e < CPU; ++e) {
      float acc = Act<T>::load(wv + e * 4 + 3) * Act<T>::load(xv + 3 * CPU + e);
      acc = fmaf(Act<T>::load(wv + e * 4 + 0), Act<T>::load(xv + 0 * CPU + e), acc);
      acc = fmaf(Act<T>::load(wv + e * 4 + 1), Act<T>::load(xv + 1 * CPU + e), acc);
      acc = fmaf(Act<T>::load(wv + e * 4 + 2), Act<T>::load(xv + 2 * CPU + e), acc);
      y[u * CPU + e] = (t < L) ? silu_fast(acc) : 0.f;
    }
  }
}

// l2 normalisation (times scale) of the thread's 8 values: the 16 threads holding token t's 128
// channels sit in four warps; each warp sums over its 32 channels with shuffles, the four
// partial sums meet in shared memory.  Contains a barrier.
__device__ __forceinline__ void l2norm8(float* y, float* part, float eps, float scale) {
  const int t = conv_t(), lane = threadIdx.x & 31;
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) ss = fmaf(y[e], y[e], ss);
  ss += __shfl_xor_sync(0xffffffffu, ss, 8);
  ss += __shfl_xor_sync(0xffffffffu, ss, 16);
  if (lane < 8) part[(threadIdx.x >> 8) * 64 + t] = ss;
  __syncthreads();
  const float inv = scale * rsqrtf((part[t] + part[64 + t]) + (part[128 + t] + part[192 + t]) + eps);
#pragma unroll
  for (int e = 0; e < 8; ++e) y[e] *= inv;
}

// The thread's 8 values of row t, split, into a 128-column K-major tile (shared or global):
// one 16-byte unit each for hi and lo.
__device__ __forceinline__ void put_row8(unsigned char* hi, unsigned char* lo, const float* v) {
  uint4 hh, ll;
  split8(v, hh, ll);
  const uint32_t off = tc::kmajor_off(conv_t(), 8 * conv_cg(), 128);
  *reinterpret_cast<uint4*>(hi + off) = hh;
  *reinterpret_cast<uint4*>(lo + off) = ll;
}

// The gates of one V-head over the chunk (warp-wide, 2 tokens per lane): gamma (cumulative g
// inside the chunk), beta (0 past L) and the derived per-token scales, into vec[5][64]; returns
// gamma_L on every lane.
template <typename T>
__device__ __forceinline__ float chunk_gates(const KDims& d, const float* __restrict__ A_log,
                                             const float* __restrict__ dt_bias,
                                             const T* __restrict__ a, const T* __restrict__ b,
                                             int h, int t0, int L, float* vec) {
  const int lane = threadIdx.x & 31;
  float g2[2], b2[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int i = 2 * lane + q;
    const int ic = min(i, L - 1);
    gates(__ldg(A_log + h), __ldg(dt_bias + h), Act<T>::ldg(a + (size_t)(t0 + ic) * d.Hv + h),
          Act<T>::ldg(b + (size_t)(t0 + ic) * d.Hv + h), g2[q], b2[q]);
    if (i >= L) {
      g2[q] = 0.f;
      b2[q] = 0.f;
    }
  }
  const float pair = g2[0] + g2[1];
  float incl = pair;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const float gm0 = incl - pair + g2[0], gm1 = incl;
  const float gsel = ((L - 1) & 1) ? gm1 : gm0;
  const float gL = __shfl_sync(0xffffffffu, gsel, (L - 1) >> 1);
  float* gam = vec;
  float* bet = vec + 64;
  float* eg = vec + 128;
  float* dec = vec + 192;
  float* bgk = vec + 256;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int i = 2 * lane + q;
    const float gm = q ? gm1 : gm0;
    const float e = expf(gm);
    gam[i] = gm;
    bet[i] = b2[q];
    eg[i] = e;
    dec[i] = i < L ? expf(gL - gm) : 0.f;
    bgk[i] = b2[q] * e;
  }
  return gL;
}

// sum_q row[q] * col[q * cs .. + 3] over 16 terms: four adjacent outputs (row and col 16-byte
// aligned).
__device__ __forceinline__ float4 dot16x4(const float* row, const float* col, int cs) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int q = 0; q < 16; q += 4) {
    const float4 r4 = *reinterpret_cast<const float4*>(row + q);
    const float rq[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 c4 = *reinterpret_cast<const float4*>(col + (q + k) * cs);
      acc.x = fmaf(rq[k], c4.x, acc.x);
      acc.y = fmaf(rq[k], c4.y, acc.y);
      acc.z = fmaf(rq[k], c4.z, acc.z);
      acc.w = fmaf(rq[k], c4.w, acc.w);
    }
  }
  return acc;
}
__device__ __forceinline__ void add4(float4& a, const float4& b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}
__device__ __forceinline__ float4 neg4(const float4& a) { return make_float4(-a.x, -a.y, -a.z, -a.w); }

// Scratch block q (q < 4) of the inverse: the upper blocks (0,1), (0,2), (0,3), (1,2) of M, which
// hold only zeros of A and are never read as T.
__device__ __forceinline__ float* xblk(float* M, int q) {
  return M + (q < 3 ? 16 * (q + 1) : 16 * 2 + 16 * AS);
}

// In place: M holds the strictly lower-triangular 64 x 64 A (f32, row stride AS, zero on and
// above the diagonal) on entry and the lower blocks of T = (I + A)^{-1} on exit (the upper
// blocks are then undefined; readers mask them).  In 16 x 16 blocks (block (i, k) = rows 16i..,
// columns 16k..):
//   1. the diagonal inverses D_b = (I + A_bb)^{-1} by forward substitution (four warps, one
//      column per lane);
//   2. the two 32 x 32 diagonal halves: T_10 = -D_1 (A_10 D_0), T_32 = -D_3 (A_32 D_2);
//   3. the 32 x 32 off-diagonal half, -T2 (A21 T1) with T1, T2 the halves of step 2: first
//      Y = A21 T1, then T_ik = -sum_m T2_im Y_mk.
// Each block of A is read before T overwrites it.  Five barriers; ends with one.  tri_inverse_n
// inverts nm = 1 or 2 independent matrices at once (the second on the next threads).
__device__ __forceinline__ void tri_inverse_n(float* M0, float* M1, int nm) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp < 4 * nm) {
    float* M = (warp >> 2) ? M1 : M0;
    const int b = warp & 3, c = lane & 15;
    float* mb = M + (16 * b) * AS + 16 * b;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      // x_i = [i == c] - sum_{m<i} A_im x_m; A_im = 0 for m >= i and x_m = 0 for m >= i, so
      // the sum may run over whole groups of four
      float p0 = (i == c) ? 1.f : 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
      for (int m = 0; m < i; m += 4) {
        const float4 a4 = *reinterpret_cast<const float4*>(mb + i * AS + m);
        p0 = fmaf(-a4.x, x[m], p0);
        p1 = fmaf(-a4.y, x[m + 1], p1);
        p2 = fmaf(-a4.z, x[m + 2], p2);
        p3 = fmaf(-a4.w, x[m + 3], p3);
      }
      x[i] = (p0 + p1) + (p2 + p3);
    }
    __syncwarp();
    if (lane < 16) {
#pragma unroll
      for (int i = 0; i < 16; ++i) mb[i * AS + c] = x[i];
    }
  }
  __syncthreads();
  // steps 2 and 3: thread e of a matrix's group computes columns [4 cq, 4 cq + 4) of row rr of a
  // block; matrix 1 takes the threads after matrix 0's
  if (tid < 128 * nm) {  // step 2: X = A_{bi,bi-1} D_{bi-1} for bi = 1, 3 (scratch blocks 0, 1)
    float* M = (tid >> 7) ? M1 : M0;
    const int t = tid & 127;
    const int which = t >> 6, rr = (t >> 2) & 15, c4 = 4 * (t & 3);
    const int bi = which ? 3 : 1, bk = bi - 1;
    *reinterpret_cast<float4*>(xblk(M, which) + rr * AS + c4) =
        dot16x4(M + (16 * bi + rr) * AS + 16 * bk, M + (16 * bk) * AS + 16 * bk + c4, AS);
  }
  __syncthreads();
  if (tid < 128 * nm) {  //         T_{bi,bi-1} = -D_bi X
    float* M = (tid >> 7) ? M1 : M0;
    const int t = tid & 127;
    const int which = t >> 6, rr = (t >> 2) & 15, c4 = 4 * (t & 3);
    const int bi = which ? 3 : 1, bk = bi - 1;
    *reinterpret_cast<float4*>(M + (16 * bi + rr) * AS + 16 * bk + c4) =
        neg4(dot16x4(M + (16 * bi + rr) * AS + 16 * bi, xblk(M, which) + c4, AS));
  }
  __syncthreads();
  // step 3: blocks (bi, bk), bi in {2, 3}, bk in {0, 1}:
  //   Y_{bi,bk} = sum_{m=bk}^{1} A_{bi,m} T_{m,bk}  (scratch block (bi - 2) * 2 + bk)
  if (tid < 256 * nm) {
    float* M = (tid >> 8) ? M1 : M0;
    const int t = tid & 255;
    const int blk = t >> 6, rr = (t >> 2) & 15, c4 = 4 * (t & 3);
    const int bi = 2 + (blk >> 1), bk = blk & 1;
    float4 acc = dot16x4(M + (16 * bi + rr) * AS + 16 * bk, M + (16 * bk) * AS + 16 * bk + c4, AS);
    if (bk == 0) add4(acc, dot16x4(M + (16 * bi + rr) * AS + 16, M + 16 * AS + c4, AS));
    *reinterpret_cast<float4*>(xblk(M, blk) + rr * AS + c4) = acc;
  }
  __syncthreads();
  //   T_{bi,bk} = -sum_{m=2}^{bi} T_{bi,m} Y_{m,bk}
  if (tid < 256 * nm) {
    float* M = (tid >> 8) ? M1 : M0;
    const int t = tid & 255;
    const int blk = t >> 6, rr = (t >> 2) & 15, c4 = 4 * (t & 3);
    const int bi = 2 + (blk >> 1), bk = blk & 1;
    float4 acc = dot16x4(M + (16 * bi + rr) * AS + 32, xblk(M, bk) + c4, AS);
    if (bi == 3) add4(acc, dot16x4(M + (16 * bi + rr) * AS + 48, xblk(M, 2 + bk) + c4, AS));
    *reinterpret_cast<float4*>(M + (16 * bi + rr) * AS + 16 * bk + c4) = neg4(acc);
  }
  __syncthreads();
}
__device__ __forceinline__ void tri_inverse(float* M) { tri_inverse_n(M, M, 1); }

// [T diag(cw) ; T diag(cu)] -> the split-bf16 K-major A operand (128 rows x 64 K) of D2.
// Unit u: row & 7 = u & 7, k-group = (u >> 3) & 7, row group = u >> 6 (consecutive 16-byte
// units); entries above the diagonal are zero.
__device__ __forceinline__ void t_to_b2(const float* Tm, const float* cw, const float* cu,
                                        unsigned char* hi, unsigned char* lo) {
  for (int u = threadIdx.x; u < 1024; u += NTI) {
    const int row = ((u >> 6) << 3) + (u & 7), jg = (u >> 3) & 7;
    const int i = row & 63;
    const float* sc = row < 64 ? cw : cu;
    float v[8];
    if ((jg >> 1) <= (i >> 4)) {
      const float4 a = *reinterpret_cast<const float4*>(Tm + i * AS + 8 * jg);
      const float4 b = *reinterpret_cast<const float4*>(Tm + i * AS + 8 * jg + 4);
      const float t8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = (8 * jg + q <= i) ? t8[q] * sc[8 * jg + q] : 0.f;
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = 0.f;
    }
    uint4 hh, ll;
    split8(v, hh, ll);
    st_unit(hi, (uint32_t)u * 16u, hh);
    st_unit(lo, (uint32_t)u * 16u, ll);
  }
}

template <typename T, bool PAD>
__global__ void __launch_bounds__(NTI, 1)
tc_intra_kernel(KDims d, const float* __restrict__ A_log, const float* __restrict__ dt_bias,
                const T* __restrict__ conv_w, const T* __restrict__ conv_state, int num_slots,
                const int32_t* __restrict__ cu, const int32_t* __restrict__ slot_idx,
                const uint8_t* __restrict__ has_init, int num_seqs, int total,
                const T* __restrict__ qkv, const T* __restrict__ a, const T* __restrict__ b,
                float* __restrict__ ws, int cw0, int rec_base, int32_t* __restrict__ status) {
  extern __shared__ __align__(1024) unsigned char sm[];
  using S = IntraSmem;
  using R = InRing<T>;
  unsigned char* a1 = sm + S::A1;
  unsigned char* vt = sm + S::VT;
  unsigned char* b2 = sm + S::B2;
  unsigned char* ring = sm + S::IN;
  float* At = reinterpret_cast<float*>(sm + S::AT);
  float* vecs = reinterpret_cast<float*>(sm + S::VEC);
  float* part = reinterpret_cast<float*>(sm + S::PART);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + S::BAR);   // [0] D1, [1] D2
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S::MISC);
  int* sh = reinterpret_cast<int*>(sm + S::MISC + 16);   // ok, t0, L, seq_len, seq_start, abort, slot, init

  const int c = cw0 + blockIdx.x, kh = blockIdx.y;   // global chunk index; records from cw0
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = d.r, h0 = kh * r;
  if (warp == 0) {
    ChunkInfo ci = {-1, 0, 0, 0, 0, -1, 0};
    const bool ok = find_chunk(cu, slot_idx, has_init, num_seqs, total, c, ci);
    if (lane == 0 && !ok && c == 0 && kh == 0) set_status(status, GDN_STATUS_BAD_SEQLENS);
    if (lane == 0) {
      sh[0] = ok && ci.seq >= 0;
      sh[1] = ci.t0;
      sh[2] = ci.len;
      sh[3] = ci.seq_len;
      sh[4] = ci.seq_start;
      sh[5] = 0;
      sh[6] = ci.slot;
      sh[7] = ci.init;
    }
  }
  __syncthreads();
  if (!sh[0]) {
    tc::pdl_launch_dependents();
    if (blockIdx.x == 0 && blockIdx.y == 0) tc::pdl_wait_primary();   // see the end of the kernel
    return;
  }
  const int t0 = sh[1], L = sh[2], seq_len = sh[3], seq_start = sh[4];
  volatile int* abort = sh + 5;
  const int s = sh[6];
  const bool valid = s >= 0 && s < num_slots;
  const bool init = valid && sh[7] != 0;
  const T* cs = conv_state + (size_t)(valid ? s : 0) * 3 * d.cqkv;
  auto rec_of = [&](int j) {
    return reinterpret_cast<unsigned char*>(ws) + ((size_t)(rec_base + c - cw0) * d.Hv + h0 + j) * REC_BYTES;
  };

  // ---- every input tensor of the chunk into the ring: k, q, v of V-head 0, 1, ... (tensor i in
  // slot i % NSLOT; later tensors as slots free up)
  const int ntens = 2 + r;
  // head dims: 128 unless the instance runs 64-dim heads zero-padded to 128
  const int dk_ = PAD ? d.dk : D, dv_ = PAD ? d.dv : D;
  auto tens_base = [&](int i) {
    return i == 0 ? d.Hk * dk_ + kh * dk_ : (i == 1 ? kh * dk_ : 2 * d.Hk * dk_ + (h0 + i - 2) * dv_);
  };
  auto tens_n = [&](int i) { return i < 2 ? dk_ : dv_; };
  auto slot_of = [&](int i) { return ring + (i % R::NSLOT) * R::SLOT; };
  const int p0 = t0 - seq_start;
  int issued = 0;
  for (; issued < min(ntens, R::NSLOT); ++issued)
    ring_issue<T>(d, qkv, conv_w, cs, init, tens_base(issued), tens_n(issued), seq_start, seq_len,
                  p0, slot_of(issued));
  // waits for tensor i's copies (all threads), then a barrier makes every thread's copies visible
  auto ring_wait = [&](int i) {
    cp_async_wait_pending(issued - 1 - i);
    __syncthreads();
  };
  if (tid == 32) {
    tc::mbar_init(bar, 1);
    tc::mbar_init(bar + 1, 1);
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(tslot, TI_COLS);
  if (warp >= 2 && warp - 2 < r) {
    const int j = warp - 2;
    const float gL = chunk_gates<T>(d, A_log, dt_bias, a, b, h0 + j, t0, L, vecs + j * 320);
    if (lane == 0) *reinterpret_cast<float*>(rec_of(j) + R_SC) = expf(gL);
  }
  const int tt = conv_t();
  float y[8];   // conv outputs of token tt, channels [8 cg, 8 cg + 8)

  // ---- K: conv, l2norm, A1 K rows
  ring_wait(0);   // also publishes the gates
  conv_slot<T>(slot_of(0), L, y);
  l2norm8(y, part, d.l2_eps, 1.0f);
  put_row8(a1 + S::K_HI, a1 + S::K_LO, y);
  // ---- Q: conv, l2norm (times q_scale), A1 Q rows and per V-head the Q~ rows of B3
  ring_wait(1);   // also: K rows complete, slot 0 and the partial sums free
  if (issued < ntens) {
    ring_issue<T>(d, qkv, conv_w, cs, init, tens_base(issued), tens_n(issued), seq_start, seq_len,
                  p0, slot_of(issued));
    ++issued;
  }
  conv_slot<T>(slot_of(1), L, y);
  l2norm8(y, part, d.l2_eps, d.q_scale);
  put_row8(a1 + S::Q_HI, a1 + S::Q_LO, y);
  for (int j = 0; j < r; ++j) {
    const float e = vecs[j * 320 + 128 + tt];
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = y[q] * e;
    unsigned char* rec = rec_of(j);
    put_row8(rec + R_B3, rec + R_B3 + B3_HALF, v);
  }
  // per V-head K~^T = (diag(e^{gamma_L - gamma}) K)^T rows of B4, from the K tile (hi + lo carry
  // about 16 significant bits): unit (feature f, 8 tokens), consecutive threads take consecutive
  // features, so every warp stores whole 128-byte lines
  for (int u = tid; u < 1024; u += NTI) {
    const int f = u & 127, jg = u >> 7;
    float kx[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t off = tc::kmajor_off(8 * jg + q, f, 128);
      kx[q] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(a1 + S::K_HI + off)) +
              __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(a1 + S::K_LO + off));
    }
    const uint32_t off = 8192u + (uint32_t)(f >> 3) * 1024u + (uint32_t)jg * 128u + (uint32_t)(f & 7) * 16u;
    for (int j = 0; j < r; ++j) {
      const float* dec = vecs + j * 320 + 192 + 8 * jg;
      float v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = kx[q] * dec[q];
      uint4 hh, ll;
      split8(v, hh, ll);
      unsigned char* rec = rec_of(j);
      gst_unit(rec + R_B4, off, hh);
      gst_unit(rec + R_B4 + B4_HALF, off, ll);
    }
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = *tslot;
  // ---- D1 = [K;Q] K^T  (columns [0,64)); A1's hi quarters [K|Q] and lo quarters are 128-row tiles
  if (tid == 0) {
    const uint32_t id = tc::idesc_bf16(128, 64);
    const uint64_t dh = tc::kstep_desc(tc::smem_u32(a1 + S::K_HI), 128, 0);
    const uint64_t dl = tc::kstep_desc(tc::smem_u32(a1 + S::K_LO), 128, 0);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint64_t hk = tc::desc_add(dh, 256 * k), lk = tc::desc_add(dl, 256 * k);
      tc::mma_bf16(tb + TI_D1, hk, hk, id, k > 0);
      tc::mma_bf16(tb + TI_D1, hk, lk, id, 1);
      tc::mma_bf16(tb + TI_D1, lk, hk, id, 1);
    }
    tc::mma_commit(bar);
  }
  // ---- V of the first V-head straight into its tile (overlaps MMA1)
  ring_wait(2);   // also: slot 1 free
  if (issued < ntens) {
    ring_issue<T>(d, qkv, conv_w, cs, init, tens_base(issued), tens_n(issued), seq_start, seq_len,
                  p0, slot_of(issued));
    ++issued;
  }
  conv_slot<T>(slot_of(2), L, y);
  put_row8(vt, vt + 16384, y);
  wait_or_abort(bar, 0, abort, status);
  tc::fence_after_sync();

  // A (to At) and P (to the record) of V-head j from D1: warp w reads TMEM lanes 32 (w % 4) and
  // the 8 columns of eighth w / 4.  Lanes 0-63 are K-rows (A), lanes 64-127 Q-rows (P).
  auto a_and_p = [&](int j, float* Aj) {
    const float* gam = vecs + j * 320;
    const float* bet = gam + 64;
    const int rr = (warp & 3) * 32 + lane, j0 = (warp >> 2) * 8;
    float v[8];
    tc::tmem_ld8(tc::taddr(tb + TI_D1, (warp & 3) * 32, j0), v);
    if (rr < 64) {
      const int i = rr;
      const float gi = gam[i], bi = bet[i];   // beta is 0 past L: rows past L vanish
#pragma unroll
      for (int q = 0; q < 8; q += 4) {
        float a4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int jj = j0 + q + u;
          const float m = (jj < i) ? bi : 0.f;
          a4[u] = m * exp_fast(fminf(gi - gam[jj], 0.f)) * v[q + u];
        }
        *reinterpret_cast<float4*>(Aj + i * AS + j0 + q) = make_float4(a4[0], a4[1], a4[2], a4[3]);
      }
    } else {
      const int i = rr - 64;
      const float gi = gam[i], vi = (i < L) ? 1.f : 0.f;
      unsigned char* rec = rec_of(j);
      float p8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int jj = j0 + u;
        p8[u] = ((jj <= i) ? vi : 0.f) * exp_fast(fminf(gi - gam[jj], 0.f)) * v[u];
      }
      uint4 hh, ll;
      split8(p8, hh, ll);
      const uint32_t off = tc::kmajor_off(i, j0, 64);   // P rows 0..63 of B4
      gst_unit(rec + R_B4, off, hh);
      gst_unit(rec + R_B4 + B4_HALF, off, ll);
    }
  };

  // D2 of V-head j into TMEM columns (wc: W rows, lanes 0-63; uc: U~ rows, lanes 64-127):
  // [T diag(bgk) ; T diag(beta)] x K^T and the same x V^T.  K^T and V^T are read MN-major straight
  // out of the token-row tiles (N-direction core stride 128 B, 8-token stride 2 KiB).
  const uint32_t idn = tc::idesc_bf16_bmn(128, 128);
  auto issue_d2 = [&](uint32_t wc, uint32_t uc) {
    if (tid == 0 && !*abort) {
      const uint64_t dah = tc::kstep_desc(tc::smem_u32(b2), 64, 0);
      const uint64_t dal = tc::kstep_desc(tc::smem_u32(b2 + 16384), 64, 0);
      const uint64_t dkh = tc::sdesc(tc::smem_u32(a1 + S::K_HI), 2048, 128);
      const uint64_t dkl = tc::sdesc(tc::smem_u32(a1 + S::K_LO), 2048, 128);
      const uint64_t dvh = tc::sdesc(tc::smem_u32(vt), 2048, 128);
      const uint64_t dvl = tc::sdesc(tc::smem_u32(vt + 16384), 2048, 128);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t ah = tc::desc_add(dah, 256 * k), al = tc::desc_add(dal, 256 * k);
        const uint32_t o = 4096u * k;
        tc::mma_bf16(tb + wc, ah, tc::desc_add(dkh, o), idn, k > 0);
        tc::mma_bf16(tb + wc, ah, tc::desc_add(dkl, o), idn, 1);
        tc::mma_bf16(tb + wc, al, tc::desc_add(dkh, o), idn, 1);
        tc::mma_bf16(tb + uc, ah, tc::desc_add(dvh, o), idn, k > 0);
        tc::mma_bf16(tb + uc, ah, tc::desc_add(dvl, o), idn, 1);
        tc::mma_bf16(tb + uc, al, tc::desc_add(dvh, o), idn, 1);
      }
      tc::mma_commit(bar + 1);
    }
  };
  // W and U~ rows of V-head j straight from TMEM (columns wc / uc) into the record
  auto readout = [&](int j, uint32_t wc, uint32_t uc) {
    unsigned char* rec = rec_of(j);
    const int lg = warp & 3, cq = (warp >> 2) * 16;   // 16 of the 128 columns per warp
    const int i = (lg & 1) * 32 + lane;
    float v[16];
    if (lg < 2) {
      tc::tmem_ld16(tc::taddr(tb + wc, lg * 32, cq), v);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        uint4 hh, ll;
        split8(v + 8 * u, hh, ll);
        const uint32_t off = tc::kmajor_off(64 + i, cq + 8 * u, 128);   // W rows of B3
        gst_unit(rec + R_B3, off, hh);
        gst_unit(rec + R_B3 + B3_HALF, off, ll);
      }
    } else {
      tc::tmem_ld16(tc::taddr(tb + uc, lg * 32, cq), v);
      // U~ record row-major: each thread stores 16 consecutive columns of its token
      float* ut = reinterpret_cast<float*>(rec + R_UT);
#pragma unroll
      for (int q = 0; q < 16; q += 4)
        *reinterpret_cast<float4*>(ut + ut_index(i, cq + q)) = make_float4(v[q], v[q + 1], v[q + 2], v[q + 3]);
    }
  };
  auto sync_operands = [&]() {
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
  };

  if (r == 2) {
    // ---- two V-heads: both A / P and both inverses at once (the second A in the ring slot of
    // V-head 0's input, consumed by its conv), and V-head 0's readout beside V-head 1's MMAs, which
    // go to the TMEM columns of D1 (consumed) and the last 128
    static_assert(R::SLOT >= 4 * 64 * AS, "a ring slot holds an A matrix");
    float* At1 = reinterpret_cast<float*>(slot_of(2));
    a_and_p(0, At);
    a_and_p(1, At1);
    __syncthreads();
    tri_inverse_n(At, At1, 2);
    t_to_b2(At, vecs + 256, vecs + 64, b2, b2 + 16384);
    sync_operands();
    issue_d2(TI_W, TI_U);
    ring_wait(3);
    conv_slot<T>(slot_of(3), L, y);
    wait_or_abort(bar + 1, 0, abort, status);
    tc::fence_after_sync();
    put_row8(vt, vt + 16384, y);
    t_to_b2(At1, vecs + 320 + 256, vecs + 320 + 64, b2, b2 + 16384);
    sync_operands();
    issue_d2(TI_D1, TI_COLS - 128);
    readout(0, TI_W, TI_U);
    wait_or_abort(bar + 1, 1, abort, status);
    tc::fence_after_sync();
    readout(1, TI_D1, TI_COLS - 128);
    tc::fence_before_sync();
    __syncthreads();
  } else {
    // ---- one V-head after another: the next V-head's conv, A / P and inverse overlap the
    // current V-head's MMAs
    a_and_p(0, At);
    __syncthreads();
    tri_inverse(At);
    t_to_b2(At, vecs + 256, vecs + 64, b2, b2 + 16384);
    sync_operands();
    for (int j = 0; j < r; ++j) {
      issue_d2(TI_W, TI_U);
      if (j + 1 < r) {
        ring_wait(j + 3);   // tensor 2 + (j + 1); also: slot of tensor j + 2 free
        if (issued < ntens) {
          ring_issue<T>(d, qkv, conv_w, cs, init, tens_base(issued), tens_n(issued), seq_start, seq_len,
                  p0, slot_of(issued));
          ++issued;
        }
        conv_slot<T>(slot_of(j + 3), L, y);
        a_and_p(j + 1, At);
        __syncthreads();
        tri_inverse(At);
      }
      wait_or_abort(bar + 1, j & 1, abort, status);
      tc::fence_after_sync();
      readout(j, TI_W, TI_U);
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      if (j + 1 < r) {
        // the D2 operands of V-head j + 1 (VT and B2 were read by the MMAs just completed)
        put_row8(vt, vt + 16384, y);
        t_to_b2(At, vecs + (j + 1) * 320 + 256, vecs + (j + 1) * 320 + 64, b2, b2 + 16384);
        sync_operands();
      }
    }
  }
  if (warp == 1) tc::tmem_dealloc(tb, TI_COLS);
  // The window's chain kernel (a programmatic dependent of this one) may be set up from here on;
  // it reads nothing before this kernel has completed.  Launched as a programmatic dependent of
  // the previous window's chain kernel, this kernel may have run beside it; one CTA waits for that
  // kernel before it exits, so this kernel completes only after it, which orders this window's
  // chain kernel after the previous one.  The other CTAs leave their SMs as soon as their work is
  // done.  (Both are no-ops for an ordinary launch.)
  tc::pdl_launch_dependents();
  if (blockIdx.x == 0 && blockIdx.y == 0) tc::pdl_wait_primary();
}

// ================================================================== serial chain kernel
//
// One CTA per (sequence, V-head), serial over the sequence's chunks in the window.  The products
// run in transposed form: the state S^T (dv x dk) and the chunk's U^T (dv x 64 tokens) are the A
// operands, written into TMEM as split bf16 from registers, and the chunk records (shared memory,
// one bulk copy each) are the B operands.  Every product then has M = dv = 128 with both the
// A reads and the accumulator in TMEM, and one CTA carries the whole head:
//   D3^T = S^T [Q~ ; W]^T           N = 128: columns 0-63 (Q~ S)^T, 64-127 (W S)^T
//   U^T  = U~^T - (W S)^T
//   S^T  <- e^{gamma_L} S^T + U^T K~      N = 128 (dk), accumulated onto the scaled f32 S^T
//   D3^T[:, 0:64] += U^T P^T        -> O^T (dv on the TMEM lanes, tokens on the columns)
//   z-gated RMSNorm over dv (across the lanes) -> out
// A head's chain takes a single SM, so a window's chains leave most SMs to the next window's
// intra kernel, which the launcher starts as a programmatic dependent of this kernel.

constexpr int NTC = 576;   // warps 0-7 main, 8-15 output epilogue, 16 loader, 17 MMA issue
// TMEM columns (lanes 0-127 = dv)
constexpr uint32_t TA_S = 0;     // S^T as split bf16 pairs of dk: hi [0, 64), lo [64, 128)
constexpr uint32_t TA_U = 128;   // U^T as split bf16 pairs of tokens: hi [128, 160), lo [160, 192)
constexpr uint32_t TC_D3 = 192;  // D3^T: 128 columns (tokens of [Q~ ; W])
constexpr uint32_t TC_S = 320;   // f32 S^T, 128 columns (dk): holds e^{gamma_L} S^T while the
                                 // chunk's U^T K~ products accumulate onto it
constexpr uint32_t TC_COLS = 512;

struct ChainSmem {
  static constexpr uint32_t B3 = 0;                          // [Q~ ; W] image, 64 KiB
  static constexpr uint32_t B4 = B3 + 65536;                 // [P ; K~^T] image, 48 KiB
  static constexpr uint32_t UT = B4 + 49152;                 // f32 U~ [64 tokens][128 dv], 32 KiB
  static constexpr uint32_t OT = UT + 32768;                 // f32 O [2 halves][32 tokens][128], 32 KiB
  static constexpr uint32_t BAR = OT + 32768;                // 17 mbarriers
  static constexpr uint32_t MISC = BAR + 256;
  static constexpr uint32_t BYTES = MISC + 64;
};
static_assert(ChainSmem::BYTES <= 227 * 1024, "chain kernel shared memory");

// 16 consecutive dk values v of S^T row (TMEM lane) lb: the split-bf16 operand words of the
// next D3^T products.  No wait.
__device__ __forceinline__ void put_sop16(uint32_t lb, int f0, const float* v) {
  uint32_t hw[8], lw[8];
#pragma unroll
  for (int p = 0; p < 8; ++p) tc::split2_bf16(v[2 * p], v[2 * p + 1], hw[p], lw[p]);
  tc::tmem_st8w_nw(lb + TA_S + f0 / 2, hw);
  tc::tmem_st8w_nw(lb + TA_S + 64 + f0 / 2, lw);
}
// The same values scaled by eg (the next chunk's e^{gamma_L}) into the f32 copy that the next
// U^T K~ products accumulate onto.  No wait.
__device__ __forceinline__ void put_sscl16(uint32_t lb, int f0, const float* v, float eg) {
  uint32_t sw[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) sw[i] = __float_as_uint(eg * v[i]);
  tc::tmem_st16w_nw(lb + TC_S + f0, sw);
}

// 8 consecutive activations held as loaded (16 bytes of bf16 or 32 of f32), converted on use.
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void ldg(const __nv_bfloat16* p) { u = __ldg(reinterpret_cast<const uint4*>(p)); }
  __device__ __forceinline__ float get(int m) const {
    const uint32_t w = m < 2 ? u.x : (m < 4 ? u.y : (m < 6 ? u.z : u.w));
    return __uint_as_float((m & 1) ? (w & 0xffff0000u) : (w << 16));
  }
};
template <> struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void ldg(const float* p) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  }
  __device__ __forceinline__ float get(int m) const {
    const float4& v = m < 4 ? a : b;
    const int k = m & 3;
    return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
  }
};

__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

template <typename T, bool PAD>
__global__ void __launch_bounds__(NTC, 1)
tc_chain_kernel(KDims d, const T* __restrict__ norm_w, float* __restrict__ rec_state,
                T* __restrict__ conv_state, int num_slots, const int32_t* __restrict__ cu,
                const int32_t* __restrict__ slot_idx, const uint8_t* __restrict__ has_init,
                int num_seqs, int total, const T* __restrict__ qkv, const T* __restrict__ z,
                T* __restrict__ out, const float* __restrict__ ws, int cw0, int cw1, int rec_base,
                int32_t* __restrict__ status) {
  extern __shared__ __align__(1024) unsigned char sm[];
  using S = ChainSmem;
  // head dims: 128 unless the instance runs 64-dim heads zero-padded to 128
  const int dk_ = PAD ? d.dk : D, dv_ = PAD ? d.dv : D;
  const float* ut_s = reinterpret_cast<const float*>(sm + S::UT);
  float* ot = reinterpret_cast<float*>(sm + S::OT);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S::BAR);
  uint64_t* b3full = bars + 0;   // B3 landed (loader -> MMA)
  uint64_t* b3empty = bars + 2;  // B3 read by the D3 products (MMA -> loader)
  uint64_t* b4full = bars + 4;   // B4 landed
  uint64_t* b4empty = bars + 5;  // B4 read by the chunk's U^T products
  uint64_t* utfull = bars + 6;   // U~ landed
  uint64_t* utempty = bars + 7;  // U~ read by the main warps (8 arrivals)
  uint64_t* sopf = bars + 8;     // S^T operand, dk [0, 32) and [64, 96) written (8 arrivals)
  uint64_t* mma3 = bars + 9;     // D3^T complete
  uint64_t* uopf = bars + 10;    // U^T operand, tokens [0, 16) and [32, 48) written (8 arrivals)
  uint64_t* sready = bars + 11;  // S^T += U^T K~ complete
  uint64_t* dfull = bars + 12;   // O^T complete in D3^T columns 0-63
  uint64_t* dempty = bars + 13;  // O^T read by the output warps (8 arrivals)
  uint64_t* sscl = bars + 14;    // e^{gamma_L} S^T written for the chunk's U^T K~ (8 arrivals)
  uint64_t* sopf2 = bars + 15;   // the rest of the S^T operand (8 arrivals)
  uint64_t* uopf2 = bars + 16;   // the rest of the U^T operand (8 arrivals)
  // The operands are handed to the MMA warp in two halves each, so that the first half's
  // products run while the second half is written.
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S::MISC);
  int* sh = reinterpret_cast<int*>(sm + S::MISC + 16);

  const int n = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    int off = 0;
    const bool ok = seq_chunk_offset(cu, num_seqs, total, n, off);
    if (lane == 0 && !ok && n == 0 && h == 0) set_status(status, GDN_STATUS_BAD_SEQLENS);
    if (lane == 0) {
      sh[0] = ok;
      sh[1] = off;
      sh[2] = 0;
    }
  }
  if (tid == 0) {
    for (int i = 0; i < 17; ++i)
      tc::mbar_init(bars + i, (i == 7 || i == 8 || i == 10 || i >= 13) ? 8 : 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) tc::tmem_alloc(tslot, TC_COLS);
  // The call's own inputs (cu_seqlens, slot_idx, has_initial_state) were complete before the
  // call's first kernel started: read before the wait.
  const int seq_start0 = __ldg(cu + n), len0 = __ldg(cu + n + 1) - seq_start0;
  const int s = __ldg(slot_idx + n);
  const bool has_init_n = has_init != nullptr && __ldg(has_init + n) != 0;
  // Launched as a programmatic dependent of the window's intra kernel: everything above touches
  // only this CTA's own resources and the call's inputs; the records, the slot's state and the
  // rest come after the intra kernel (and with it the previous window's chains) has completed.
  // Only then may the next window's intra kernel start: it writes the workspace half the previous
  // window's chains read.
  tc::pdl_wait_primary();
  tc::pdl_launch_dependents();   // the next window's intra kernel may take the SMs left free
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = *tslot;
  const int choff = sh[1];
  volatile int* abort = sh + 2;
  const int nch_seq = sh[0] ? (len0 + CH - 1) / CH : 0;
  // The call's global chunks [cw0, cw1) form this window: the sequence's chunks [ca, cb) of it
  // run here, as local chunks 0 .. nch - 1, starting from the slot's state when an earlier window
  // (or has_initial_state) left one there.
  const int ca = max(0, cw0 - choff), cb = min(nch_seq, cw1 - choff);
  const int nch = max(0, cb - ca);
  const bool empty_here = nch_seq == 0 && cw0 == 0;   // an empty sequence resets its slot once
  const int seq_start = seq_start0 + ca * CH, len = len0 - ca * CH;   // tokens from the window on
  // invalid cu_seqlens: nothing is read or written
  const bool valid = sh[0] && s >= 0 && s < num_slots && (nch > 0 || empty_here);
  if (sh[0] && s >= num_slots && h == 0 && tid == 0 && (nch > 0 || empty_here))
    set_status(status, GDN_STATUS_SLOT_RANGE);
  const bool init_seq = valid && has_init_n;
  const bool init = valid && (init_seq || ca > 0);
  const bool seq_ends = valid && ((nch > 0 && cb == nch_seq) || empty_here);
  // the slot's state, dk x dv (a 64-dim head's state is the corner of the 128 x 128 one here)
  float* Sg = rec_state + ((size_t)(valid ? s : 0) * d.Hv + h) * dk_ * dv_;
  auto rec_of = [&](int c) {
    return reinterpret_cast<const unsigned char*>(ws) +
           ((size_t)(rec_base + choff + ca + c - cw0) * d.Hv + h) * REC_BYTES;
  };

  if (warp < 8) {
    // ================= main warps: thread (q, hf) is dv row j = 32 q + lane (its TMEM lane) of
    // S^T for dk [64 hf, 64 hf + 64), and of U^T for tokens [32 hf, 32 hf + 32)
    const int q = warp & 3, hf = warp >> 2;
    const int j = 32 * q + lane;
    const uint32_t lb = tb + ((uint32_t)(32 * q) << 16);
    // this thread's 64 state entries are real (dk rows 64 hf .., dv column j) or all padding
    const bool sreal = !PAD || (64 * hf < dk_ && j < dv_);
    {
      const float eg0 = nch > 0 ? *reinterpret_cast<const float*>(rec_of(0) + R_SC) : 1.f;
      float v[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) v[i] = (init && sreal) ? Sg[(size_t)(64 * hf + i) * dv_ + j] : 0.f;
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int f0 = 64 * hf + 16 * p;
        if (nch > 0) {
          put_sop16(lb, f0, v + 16 * p);
        } else if (valid && !init) {   // an empty sequence without a state: the slot is reset
          if (sreal) {
#pragma unroll
            for (int i = 0; i < 16; ++i) Sg[(size_t)(f0 + i) * dv_ + j] = 0.f;
          }
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(sopf);
        mbar_arrive(sopf2);
      }
      if (nch > 0) {
#pragma unroll
        for (int p = 0; p < 4; ++p) put_sscl16(lb, 64 * hf + 16 * p, v + 16 * p, eg0);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(sscl);
    }
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
      const uint32_t par = c & 1;
      const float egn = (c + 1 < nch) ? *reinterpret_cast<const float*>(rec_of(c + 1) + R_SC) : 1.f;
      // U^T = U~^T - (W S)^T -> the U^T operand
      const bool ok1 = wait_or_abort(mma3, par, abort, status) && wait_or_abort(utfull, par, abort, status);
      tc::fence_after_sync();
      // in two halves of 16 tokens (K-steps 2 hf, then 2 hf + 1 of the U^T products)
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {
        if (ok1) {
          uint32_t rv[16];
          tc::tmem_ld16_nw(lb + TC_D3 + 64 + 32 * hf + 16 * hq, rv);
          tc::tmem_wait_ld();
          tc::reg_fence16(rv);
          uint32_t hw[8], lw[8];
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            const int t = 32 * hf + 16 * hq + 2 * p;
            const float u0 = ut_s[t * D + j] - __uint_as_float(rv[2 * p]);
            const float u1 = ut_s[(t + 1) * D + j] - __uint_as_float(rv[2 * p + 1]);
            tc::split2_bf16(u0, u1, hw[p], lw[p]);
          }
          tc::tmem_st8w_nw(lb + TA_U + 16 * hf + 8 * hq, hw);
          tc::tmem_st8w_nw(lb + TA_U + 32 + 16 * hf + 8 * hq, lw);
          tc::tmem_wait_st();
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(hq ? uopf2 : uopf);
      }
      if (lane == 0) mbar_arrive(utempty);
      // S^T of the next chunk = the accumulated e^{gamma_L} S^T + U^T K~: first its operand (the
      // next D3^T products wait for it), then its copy scaled by the next e^{gamma_L} (needed
      // only by the next U^T K~); after the last chunk, the final state to the slot
      const bool ok2 = wait_or_abort(sready, par, abort, status);
      tc::fence_after_sync();
      auto ld_s32 = [&](int f0, uint32_t* rv) {
        tc::tmem_ld16_nw(lb + TC_S + f0, rv);
        tc::tmem_ld16_nw(lb + TC_S + f0 + 16, rv + 16);
        tc::tmem_wait_ld();
        tc::reg_fence16(rv);
        tc::reg_fence16(rv + 16);
      };
      // in two halves of 32 dk (K-steps 4 hf, 4 hf + 1, then 4 hf + 2, 4 hf + 3 of D3^T)
#pragma unroll 1
      for (int hp = 0; hp < 2; ++hp) {
        if (ok2) {
          const int f0 = 64 * hf + 32 * hp;
          uint32_t rv[32];
          ld_s32(f0, rv);
          const float* v = reinterpret_cast<const float*>(rv);
          if (c + 1 < nch) {
            put_sop16(lb, f0, v);
            put_sop16(lb, f0 + 16, v + 16);
            tc::tmem_wait_st();
          } else if (valid && sreal) {
#pragma unroll
            for (int i = 0; i < 32; ++i) Sg[(size_t)(f0 + i) * dv_ + j] = v[i];
          }
        }
        if (c + 1 < nch) {
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(hp ? sopf2 : sopf);
        }
      }
      if (c + 1 < nch) {
        if (ok2) {
#pragma unroll 1
          for (int hp = 0; hp < 2; ++hp) {
            const int f0 = 64 * hf + 32 * hp;
            uint32_t rv[32];
            ld_s32(f0, rv);
            const float* v = reinterpret_cast<const float*>(rv);
            put_sscl16(lb, f0, v, egn);
            put_sscl16(lb, f0 + 16, v + 16, egn);
          }
          tc::tmem_wait_st();
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(sscl);
      }
    }
  } else if (warp < 16) {
    // ================= output warps: warps 8-11 take the tokens [0, 32) of the chunk, 12-15 the
    // tokens [32, 64).  O^T comes out of TMEM one dv row per thread (lane j) and goes through
    // shared memory as O (token rows), so that thread r of the half then owns 8 consecutive
    // columns (8 (r & 15) ..) of the tokens r / 16 + 8 b, b = 0..3: the sum of squares over dv
    // adds up across 16 consecutive lanes, and z and the output move as 16-byte vectors.
    const int q = warp & 3, th = (warp - 8) >> 2;
    const int r = 32 * q + lane;               // thread of the half, 0..127
    const int o8 = r & 15, tr = r >> 4;        // column octet, first token row
    const uint32_t lb = tb + ((uint32_t)(32 * q) << 16);
    float* oth = ot + th * 32 * D;             // this half's 32 token rows
    const size_t ld = (size_t)d.Hv * dv_;
    const bool ocol = !PAD || 8 * o8 < dv_;    // a real output column octet (dv = 64: half)
    const size_t col = (size_t)h * dv_ + (ocol ? 8 * o8 : 0);
    float wv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (ocol) {
      const float4 w0 = Act<T>::ldg4(norm_w + 8 * o8), w1 = Act<T>::ldg4(norm_w + 8 * o8 + 4);
      wv[0] = w0.x; wv[1] = w0.y; wv[2] = w0.z; wv[3] = w0.w;
      wv[4] = w1.x; wv[5] = w1.y; wv[6] = w1.z; wv[7] = w1.w;
    }
    Raw8<T> zr[4];   // z of the tokens 32 th + tr + 8 b, one chunk ahead
    auto load_z = [&](int c) {
      const int last = min(CH, len - c * CH) - 1;
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        const int t = min(32 * th + tr + 8 * bb, last);
        zr[bb].ldg(z + (size_t)(seq_start + c * CH + t) * ld + col);
      }
    };
    if (nch > 0) load_z(0);
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
      const int L = min(CH, len - c * CH);
      const bool ok = wait_or_abort(dfull, c & 1, abort, status);
      tc::fence_after_sync();
      float o[32];
      if (ok) {
        uint32_t* ou = reinterpret_cast<uint32_t*>(o);
        tc::tmem_ld16_nw(lb + TC_D3 + 32 * th, ou);
        tc::tmem_ld16_nw(lb + TC_D3 + 32 * th + 16, ou + 16);
        tc::tmem_wait_ld();
        tc::reg_fence16(ou);
        tc::reg_fence16(ou + 16);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0.f;
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty);   // D3^T may be overwritten from here on
      if (c > 0) named_sync(1 + th, 128);   // the previous chunk's rows have been read
#pragma unroll
      for (int i = 0; i < 32; ++i) oth[i * D + r] = o[i];
      named_sync(1 + th, 128);
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        const int tl = tr + 8 * bb;   // token of the half
        const float4 v0 = *reinterpret_cast<const float4*>(oth + tl * D + 8 * o8);
        const float4 v1 = *reinterpret_cast<const float4*>(oth + tl * D + 8 * o8 + 4);
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < 8; ++m) ss = fmaf(v[m], v[m], ss);
#pragma unroll
        for (int ofs = 1; ofs < 16; ofs <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, ofs);
        const float inv = valid ? rsqrtf(ss * (1.0f / (float)dv_) + d.norm_eps) : 0.f;
        const int t = 32 * th + tl;
        if (t < L && ocol) {
          T* op = out + (size_t)(seq_start + c * CH + t) * ld + col;
          float y[8];
#pragma unroll
          for (int m = 0; m < 8; ++m) y[m] = v[m] * inv * wv[m] * silu_fast(zr[bb].get(m));
          Act<T>::store4(op, make_float4(y[0], y[1], y[2], y[3]));
          Act<T>::store4(op + 4, make_float4(y[4], y[5], y[6], y[7]));
        }
      }
      if (c + 1 < nch) load_z(c + 1);
    }
  } else if (warp == 16) {
    // ================= loader warp: bulk copies of each chunk's B3 (double-buffered), B4 and U~,
    // each issued as soon as the buffer it refills has been read
    if (lane == 0) {
      int n3 = 0, n4 = 0, nu = 0;   // copies issued per buffer
      auto load_b3 = [&](int c) {
        tc::mbar_arrive_expect_tx(b3full, 2 * B3_HALF);
        tc::bulk_g2s(sm + S::B3, rec_of(c) + R_B3, 2 * B3_HALF, b3full);
        ++n3;
      };
      auto load_b4 = [&](int c) {
        tc::mbar_arrive_expect_tx(b4full, 2 * B4_HALF);
        tc::bulk_g2s(sm + S::B4, rec_of(c) + R_B4, 2 * B4_HALF, b4full);
        ++n4;
      };
      auto load_ut = [&](int c) {
        tc::mbar_arrive_expect_tx(utfull, 32768);
        tc::bulk_g2s(sm + S::UT, rec_of(c) + R_UT, 32768, utfull);
        ++nu;
      };
      if (nch > 0) {
        load_b3(0);
        load_b4(0);
        load_ut(0);
      }
      for (int c = 0; c + 1 < nch; ++c) {
        if (!wait_or_abort(b3empty, c & 1, abort, status)) break;
        load_b3(c + 1);
        if (!wait_or_abort(utempty, c & 1, abort, status)) break;
        load_ut(c + 1);
        if (!wait_or_abort(b4empty, c & 1, abort, status)) break;
        load_b4(c + 1);
      }
      // after a timeout: wait (bounded) for the copies still in flight before the CTA exits
      if (*abort) {
        if (n3 > 0) tc::mbar_wait(b3full, (n3 - 1) & 1, 100000000ull);
        if (n4 > 0) tc::mbar_wait(b4full, (n4 - 1) & 1, 100000000ull);
        if (nu > 0) tc::mbar_wait(utfull, (nu - 1) & 1, 100000000ull);
      }
    }
  } else {
    // ================= MMA warp: one thread issues every product of the chunk step
    if (lane == 0) {
      const uint32_t id128 = tc::idesc_bf16(128, 128), id64 = tc::idesc_bf16(128, 64);
      const uint64_t dB3h = tc::kstep_desc(tc::smem_u32(sm + S::B3), 128, 0);
      const uint64_t dB3l = tc::kstep_desc(tc::smem_u32(sm + S::B3 + B3_HALF), 128, 0);
      const uint64_t dKh = tc::kstep_desc(tc::smem_u32(sm + S::B4) + 8192, 64, 0);   // K~^T rows
      const uint64_t dKl = tc::kstep_desc(tc::smem_u32(sm + S::B4 + B4_HALF) + 8192, 64, 0);
      const uint64_t dPh = tc::kstep_desc(tc::smem_u32(sm + S::B4), 64, 0);          // P rows
      const uint64_t dPl = tc::kstep_desc(tc::smem_u32(sm + S::B4 + B4_HALF), 64, 0);
      const uint32_t aSh = tb + TA_S, aSl = tb + TA_S + 64, aUh = tb + TA_U, aUl = tb + TA_U + 32;
      const uint32_t d3 = tb + TC_D3, xs = tb + TC_S;
      for (int c = 0; c < nch; ++c) {
        const uint32_t par = c & 1;
        // D3^T = S^T [Q~ ; W]^T, K = dk: K-steps 0, 1, 4, 5 on the first half of the operand
        auto d3_step = [&](int k) {
          const uint64_t bh = tc::desc_add(dB3h, 256 * k), bl = tc::desc_add(dB3l, 256 * k);
          tc::mma_bf16_tmem_a(d3, aSh + 8 * k, bh, id128, k > 0);
          tc::mma_bf16_tmem_a(d3, aSh + 8 * k, bl, id128, 1);
          tc::mma_bf16_tmem_a(d3, aSl + 8 * k, bh, id128, 1);
        };
        const bool okA = wait_or_abort(sopf, par, abort, status) && wait_or_abort(b3full, par, abort, status) &&
                         (c == 0 || wait_or_abort(dempty, (c - 1) & 1, abort, status));
        if (okA) {
          tc::fence_after_sync();
          d3_step(0);
          d3_step(1);
          d3_step(4);
          d3_step(5);
        }
        if (okA && wait_or_abort(sopf2, par, abort, status)) {
          tc::fence_after_sync();
          d3_step(2);
          d3_step(3);
          d3_step(6);
          d3_step(7);
          tc::mma_commit(mma3);
          tc::mma_commit(b3empty);
        }
        // S^T += U^T K~, K = tokens: K-steps 0, 2 on the first half of the operand
        auto x_step = [&](int k) {
          const uint64_t kh = tc::desc_add(dKh, 256 * k), kl = tc::desc_add(dKl, 256 * k);
          tc::mma_bf16_tmem_a(xs, aUh + 8 * k, kh, id128, 1);
          tc::mma_bf16_tmem_a(xs, aUh + 8 * k, kl, id128, 1);
          tc::mma_bf16_tmem_a(xs, aUl + 8 * k, kh, id128, 1);
        };
        const bool okU = wait_or_abort(uopf, par, abort, status) && wait_or_abort(b4full, par, abort, status) &&
                         wait_or_abort(sscl, par, abort, status);
        if (okU) {
          tc::fence_after_sync();
          x_step(0);
          x_step(2);
        }
        if (okU && wait_or_abort(uopf2, par, abort, status)) {
          tc::fence_after_sync();
          x_step(1);
          x_step(3);
          tc::mma_commit(sready);
#pragma unroll
          for (int k = 0; k < 4; ++k) {   // O^T = (Q~ S)^T + U^T P^T in D3^T columns 0-63
            const uint64_t ph = tc::desc_add(dPh, 256 * k), pl = tc::desc_add(dPl, 256 * k);
            tc::mma_bf16_tmem_a(d3, aUh + 8 * k, ph, id64, 1);
            tc::mma_bf16_tmem_a(d3, aUh + 8 * k, pl, id64, 1);
            tc::mma_bf16_tmem_a(d3, aUl + 8 * k, ph, id64, 1);
          }
          tc::mma_commit(b4empty);
          tc::mma_commit(dfull);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, TC_COLS);
  // conv state <- the sequence's last K-1 raw inputs (older ones kept when continuing); the
  // sequence's Hv CTAs take one slice of the channels each
  if (seq_ends) {
    T* csw = conv_state + (size_t)s * 3 * d.cqkv;
    const int per = (d.cqkv + d.Hv - 1) / d.Hv;
    const int c_end = min(d.cqkv, (h + 1) * per);
    for (int cch = h * per + tid; cch < c_end; cch += NTC) {
      T v3[3];
#pragma unroll
      for (int m = 0; m < 3; ++m) {
        const int rel = len0 - 3 + m;
        if (rel >= 0) v3[m] = qkv[(size_t)(seq_start0 + rel) * d.cqkv + cch];
        else v3[m] = init_seq ? csw[(size_t)(3 + rel) * d.cqkv + cch] : Act<T>::cvt(0.f);
      }
#pragma unroll
      for (int m = 0; m < 3; ++m) csw[(size_t)m * d.cqkv + cch] = v3[m];
    }
  }
}

template <typename T, bool PAD>
int launch_t(const KDims& d, const gdn_weights* w, const gdn_pool* pool, const int32_t* cu,
             const int32_t* slot_idx, const uint8_t* has_init, int num_seqs, int total,
             const void* qkv, const void* z, const void* a, const void* b, void* out, void* ws,
             size_t ws_bytes, cudaStream_t stream) {
  // Chunks are numbered across the sequences; at most total / 64 + num_seqs of them exist.  The
  // call runs in windows of consecutive chunks: each window's intra kernel writes its records,
  // then its chain kernel carries every sequence's state through the window to the slot.
  // Pipelined: windows alternate between two halves of the workspace, and window w + 1's intra
  // kernel is a programmatic dependent launch of window w's chain kernel, so it starts on the SMs
  // the chains leave free.  One of its CTAs waits for that chain kernel to complete before it
  // exits, so the intra kernel completes after it; the others exit when their work is done.
  // Each chain kernel is a programmatic dependent launch of its window's intra kernel (whose CTAs
  // signal when their work is done), so it is set up as SMs free up and waits for that kernel
  // before reading anything: window w + 1's chains read the slots only after window w's chains
  // have completed, and the half window w + 1's records go to was last read by window w - 1's
  // chains, complete before window w's chain kernel could even start.  Serial (a workspace of
  // fewer than two pipelined windows, or more chains than SMs): every window from the start of
  // the workspace, each launch after the previous one.
  // Chunk count bound: sum over sequences of ceil(len / 64) <= (total + 63 num_seqs) / 64.
  const int nc_max = std::max(1, (int)(((long long)total + (long long)(CH - 1) * num_seqs) / CH));
  const size_t per_chunk = (size_t)d.Hv * REC_BYTES;
  const size_t cap = ws_bytes / per_chunk;
  if (cap < 1) return GDN_ERR_WORKSPACE_TOO_SMALL;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GDN_ERR_CUDA;
  // Pipelined windows are as large as the intra CTAs that fit beside the chains (one per SM);
  // the first one, which runs alone, as large as a full wave of intra CTAs.
  const int chains = num_seqs * d.Hv;
  const bool pipe = cap >= 2 && chains < nsm && total > 0 && nc_max > 1;
  const int pwin = std::max(1, (nsm - chains) / d.Hk);
  const int win = pipe ? (int)std::min<size_t>({(size_t)pwin, cap / 2, (size_t)nc_max})
                       : (int)std::min<size_t>((size_t)nc_max, cap);
  const int win0 = pipe ? (int)std::min<size_t>({(size_t)std::max(win, nsm / d.Hk), cap / 2, (size_t)nc_max})
                        : win;
  auto k1 = tc_intra_kernel<T, PAD>;
  auto k2 = tc_chain_kernel<T, PAD>;
  if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)IntraSmem::BYTES) !=
          cudaSuccess ||
      cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ChainSmem::BYTES) !=
          cudaSuccess)
    return GDN_ERR_CUDA;
  float* wsf = static_cast<float*>(ws);
  const T* conv_w = static_cast<const T*>(w->conv_weight);
  const T* conv_s = static_cast<const T*>(pool->conv_state);
  const T* qkv_t = static_cast<const T*>(qkv);
  const T* a_t = static_cast<const T*>(a);
  const T* b_t = static_cast<const T*>(b);
  int cw1 = 0;
  for (int wi = 0, cw0 = 0; cw0 < nc_max; ++wi, cw0 = cw1) {
    cw1 = std::min(nc_max, cw0 + (wi == 0 ? win0 : win));
    const int rec_base = pipe ? (wi & 1) * win0 : 0;
    if (total > 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(cw1 - cw0), (unsigned)d.Hk);
      cfg.blockDim = dim3(NTI);
      cfg.dynamicSmemBytes = IntraSmem::BYTES;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = (pipe && wi > 0) ? 1 : 0;
      if (cudaLaunchKernelEx(&cfg, k1, d, w->A_log, w->dt_bias, conv_w, conv_s, pool->num_slots, cu,
                             slot_idx, has_init, num_seqs, total, qkv_t, a_t, b_t, wsf, cw0, rec_base,
                             pool->status) != cudaSuccess)
        return GDN_ERR_CUDA;
    }
    {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)num_seqs, (unsigned)d.Hv);
      cfg.blockDim = dim3(NTC);
      cfg.dynamicSmemBytes = ChainSmem::BYTES;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = pipe ? 1 : 0;
      if (cudaLaunchKernelEx(&cfg, k2, d, static_cast<const T*>(w->norm_weight), pool->rec_state,
                             static_cast<T*>(pool->conv_state), pool->num_slots, cu, slot_idx,
                             has_init, num_seqs, total, qkv_t, static_cast<const T*>(z),
                             static_cast<T*>(out), static_cast<const float*>(wsf), cw0, cw1, rec_base,
                             pool->status) != cudaSuccess)
        return GDN_ERR_CUDA;
    }
  }
  return GDN_OK;
}

}  // namespace

// Head dims 64 run as 128-dim heads whose extra channels, state rows and columns are zero.
bool prefill_tc_supported(const KDims& d) { return d.dk <= D && d.dv <= D && d.r <= RMAX; }

size_t prefill_tc_ws_bytes(const KDims& d, int num_seqs, int total) {
  return (size_t)(total / CH + num_seqs) * d.Hv * REC_BYTES;
}

size_t prefill_tc_ws_min_bytes(const KDims& d) { return (size_t)d.Hv * REC_BYTES; }

int launch_prefill_tc(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                      const int32_t* cu, const int32_t* slot_idx, const uint8_t* has_init,
                      int num_seqs, int total, const void* qkv, const void* z, const void* a,
                      const void* b, void* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  const bool pad = d.dk != D || d.dv != D;
  if (w->act == GDN_BF16)
    return pad ? launch_t<__nv_bfloat16, true>(d, w, pool, cu, slot_idx, has_init, num_seqs, total,
                                               qkv, z, a, b, out, ws, ws_bytes, stream)
               : launch_t<__nv_bfloat16, false>(d, w, pool, cu, slot_idx, has_init, num_seqs, total,
                                                qkv, z, a, b, out, ws, ws_bytes, stream);
  return pad ? launch_t<float, true>(d, w, pool, cu, slot_idx, has_init, num_seqs, total, qkv, z, a,
                                     b, out, ws, ws_bytes, stream)
             : launch_t<float, false>(d, w, pool, cu, slot_idx, has_init, num_seqs, total, qkv, z, a,
                                      b, out, ws, ws_bytes, stream);
}

}  // namespace gdn
