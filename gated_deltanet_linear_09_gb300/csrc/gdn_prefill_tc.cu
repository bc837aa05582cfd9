// gdn_prefill_tc.cu -- chunkwise prefill on the sm_103a tensor cores (tcgen05 + TMEM), for
// head dims dk = dv = 128.
//
// Same chunk algebra as the CUDA-core path (UT transform of the gated delta rule; Yang et al.,
// "Parallelizing Linear Transformers with the Delta Rule over Sequence Length", NeurIPS 2024,
// section 3; chunked prefill chain and its scratch from "pegainfer PR #1003"), arranged so that
// every tensor-core product has M = 128:
//
//   intra kernel (chunk x V-head, all in parallel, two CTAs per SM):
//     conv + SiLU + l2norm + gates of the chunk's 64 tokens,
//     D1 = [K;Q] K^T                     -> A = beta_i e^{g_i-g_j} KK^T (j<i),  P = QK^T o Gamma
//     T  = (I + A)^{-1}                  (16 x 16 blocks: diagonal inverses, then block rows)
//     D2 = (beta e^gamma K)^T T^T, (beta V)^T T^T   -> W^T, U~^T
//     writes [Q~ ; W] and [P ; K~^T] as split-bf16 operand images (Q~ = e^gamma Q,
//     K~ = e^{gamma_L - gamma} K), U~ (f32) and e^{gamma_L}
//   state kernel (sequence x V-head x 4 dv slices, a cluster of 4 CTAs; serial over the chunks,
//   the 128 x 32 state slice S held in TMEM):
//     D3 = [Q~ ; W] S                    -> rows 0-63 Q~ S, rows 64-127 W S
//     U  = U~ - W S
//     S <- e^{gamma_L} S + K~^T U ;  D3 += [P ; K~^T_(0..63)] U  (rows 0-63: O = Q~ S + P U)
//     z-gated RMSNorm of O -> out, the sum of squares over dv shared within the cluster
//
// Precision: every product runs as three bf16 passes on split operands
// (x = hi + lo, hi = bf16(x), lo = bf16(x - hi): A_hi B_hi + A_hi B_lo + A_lo B_hi) with f32
// accumulation in TMEM, which keeps about 16 significant bits per operand.
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {

namespace {

constexpr int CH = 64;
constexpr int D = 128;

// Per (chunk, V-head) record of the workspace.  B3 and B4 are stored as the exact shared-memory
// images of the state kernel's A operands (split bf16, K-major core-matrix layout, hi then lo), so
// the state kernel brings each in with one bulk copy.  Offsets in bytes.
constexpr uint32_t R_B3 = 0;                     // [Q~ ; W] rows, 128 x 128: hi 32 KiB, lo 32 KiB
constexpr uint32_t R_B4 = R_B3 + 65536;          // [P ; K~^T] rows, 192 x 64: hi 24 KiB, lo 24 KiB
constexpr uint32_t R_UT = R_B4 + 49152;          // f32 [64][128] U~ rows
constexpr uint32_t R_SC = R_UT + 32768;          // f32 e^{gamma_L}
constexpr uint32_t REC_BYTES = R_SC + 256;       // 147,712 bytes (multiple of 256)
constexpr uint32_t B3_HALF = 32768, B4_HALF = 24576;

__device__ __forceinline__ void bar_sync_main() { asm volatile("bar.sync 1, 256;\n" ::: "memory"); }

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
  __nv_bfloat16 h[8], l[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) tc::split_bf16(v[q], h[q], l[q]);
  hi = *reinterpret_cast<const uint4*>(h);
  lo = *reinterpret_cast<const uint4*>(l);
}

__device__ __forceinline__ void st_unit(unsigned char* tile, uint32_t off, const uint4& v) {
  *reinterpret_cast<uint4*>(tile + off) = v;
}

__device__ __forceinline__ void gst_unit(unsigned char* g, uint32_t off, const uint4& v) {
  *reinterpret_cast<uint4*>(g + off) = v;
}

// Rows [0,64) of X (f32 [64][XS], each row scaled by rs[row]) -> rows [row0, row0+64) of a
// 128-column K-major tile image in global memory.  Consecutive threads write consecutive
// 16-byte units (unit u: row & 7 = u & 7, k-group = (u >> 3) & 15, row group = u >> 7).
__device__ __forceinline__ void x_rows_to_gtile128(const float* X, const float* rs,
                                                   unsigned char* ghi, unsigned char* glo, int row0) {
  for (int u = threadIdx.x; u < 1024; u += blockDim.x) {
    const int r = ((u >> 7) << 3) + (u & 7), kg = (u >> 3) & 15;
    const float sc = rs ? rs[r] : 1.f;
    const float4 a = *reinterpret_cast<const float4*>(X + r * 132 + kg * 8);
    const float4 b = *reinterpret_cast<const float4*>(X + r * 132 + kg * 8 + 4);
    const float v[8] = {a.x * sc, a.y * sc, a.z * sc, a.w * sc, b.x * sc, b.y * sc, b.z * sc, b.w * sc};
    uint4 hh, ll;
    split8(v, hh, ll);
    const uint32_t off = (uint32_t)(row0 * 16 * 16) + (uint32_t)u * 16u;   // row0 is a multiple of 8
    gst_unit(ghi, off, hh);
    gst_unit(glo, off, ll);
  }
}

// Columns of X scaled per token by cs[j] -> a [128 features][64 tokens] K-major tile image in
// global memory (unit u: feature & 7 = u & 7, token group = (u >> 3) & 7, feature group = u >> 6).
__device__ __forceinline__ void x_cols_to_gtile64(const float* X, const float* cs,
                                                  unsigned char* ghi, unsigned char* glo) {
  for (int u = threadIdx.x; u < 1024; u += blockDim.x) {
    const int f = ((u >> 6) << 3) + (u & 7), jg = (u >> 3) & 7;
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = X[(jg * 8 + q) * 132 + f] * cs[jg * 8 + q];
    uint4 hh, ll;
    split8(v, hh, ll);
    gst_unit(ghi, (uint32_t)u * 16u, hh);
    gst_unit(glo, (uint32_t)u * 16u, ll);
  }
}

// Warp-wide: global chunk -> (sequence, first token, length); false if cu_seqlens is invalid.
__device__ bool find_chunk(const int32_t* __restrict__ cu, int num_seqs, int total, int c, int& seq,
                           int& t0, int& len, int& seq_start) {
  const int lane = threadIdx.x & 31;
  bool ok = (__ldg(cu) == 0) && (__ldg(cu + num_seqs) == total);
  int base = 0;
  seq = -1;
  for (int n0 = 0; n0 < num_seqs; n0 += 32) {
    const int n = n0 + lane;
    int lo = 0, hi = 0, nch = 0;
    if (n < num_seqs) {
      lo = __ldg(cu + n);
      hi = __ldg(cu + n + 1);
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
    if (m && seq < 0) {
      const int src = __ffs(m) - 1;
      seq = __shfl_sync(0xffffffffu, n, src);
      seq_start = __shfl_sync(0xffffffffu, lo, src);
      const int hi_s = __shfl_sync(0xffffffffu, hi, src);
      const int ex = __shfl_sync(0xffffffffu, base + incl - nch, src);
      t0 = seq_start + (c - ex) * CH;
      len = min(CH, hi_s - t0);
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
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

constexpr int XS = 132;   // row stride (floats) of the f32 staging tile
constexpr int AS = 68;    // row stride of the A matrix (16-byte aligned rows)
constexpr int NTI = 256;  // threads of the intra kernel (8 warps); two CTAs share an SM

// Shared memory, ~100 KB so that two CTAs fit on one SM.  Regions are reused along the kernel:
//   A1  [0, 64K)   : [K;Q] split-bf16 operand of MMA1  (hi K | hi Q | lo K | lo Q, 16 KiB each);
//                    after MMA1: (beta e^g K)^T hi/lo in the Q quarters, (beta V)^T hi/lo in the
//                    K quarters (each [128 x 64] tile is exactly 16 KiB).
//   X   [64K, +33792): f32 staging [64][XS]; after the V tiles: A [64][AS] (17,408 B) followed by
//                    the B2 tile (T rows, hi 8 KiB + lo 8 KiB); after MMA2: the W readout.
struct IntraSmem {
  static constexpr uint32_t A1 = 0;
  static constexpr uint32_t K_HI = 0, Q_HI = 16384, K_LO = 32768, Q_LO = 49152;
  static constexpr uint32_t X = 65536;
  static constexpr uint32_t AM = X;                        // aliases X
  static constexpr uint32_t B2 = X + 4 * 64 * AS;          // aliases X (17,408 B in)
  static constexpr uint32_t VEC = X + 4 * 64 * XS;         // f32 gam, bet, eg, dec, bgk [5][64]
  static constexpr uint32_t BAR = VEC + 4 * 5 * 64;        // mbarrier
  static constexpr uint32_t MISC = BAR + 16;               // tmem slot, flags
  static constexpr uint32_t BYTES = MISC + 64;
};
static_assert(IntraSmem::B2 + 16384 <= IntraSmem::VEC, "A and B2 must fit in the staging tile");

// conv + SiLU of 128 channels [cb, cb+128) over the chunk's tokens into X (rows >= L zero), split
// into a load step (all loads in flight, results in registers) and a compute step, so that the
// next channel group's loads overlap the current group's processing.
// Thread t: channel t & 127, tokens [32 (t >> 7), +32).
struct ConvIn {
  float w[4];
  float hist[3];
  float xs[32];
};

template <typename T>
__device__ __forceinline__ void conv_load(const KDims& d, const T* __restrict__ qkv,
                                          const T* __restrict__ conv_w, const T* __restrict__ cs,
                                          bool init, int cb, int seq_start, int seq_len, int t0,
                                          int L, ConvIn& in) {
  const int tid = threadIdx.x;
  const int f = tid & 127, i0 = (tid >> 7) * 32;
  const int ch = cb + f;
#pragma unroll
  for (int q = 0; q < 4; ++q) in.w[q] = Act<T>::ldg(conv_w + (size_t)ch * 4 + q);
  const int p0 = (t0 - seq_start) + i0;   // position of token i0 inside its sequence
  // Every load reads a valid address (rows clamped into the sequence / the conv state) and is
  // selected afterwards, so all of them can be in flight at once.
#pragma unroll
  for (int m = 0; m < 3; ++m) {
    const int p = p0 - 3 + m;
    const int pr = min(max(p, 0), seq_len - 1);
    const int pc = min(max(p, -3), -1);
    const float xq = Act<T>::ldg(qkv + (size_t)(seq_start + pr) * d.cqkv + ch);
    const float xc = Act<T>::ldg(cs + (size_t)(3 + pc) * d.cqkv + ch);
    in.hist[m] = (p >= seq_len) ? 0.f : (p >= 0 ? xq : (init ? xc : 0.f));
  }
#pragma unroll
  for (int k = 0; k < 32; ++k)
    in.xs[k] = Act<T>::ldg(qkv + (size_t)(t0 + min(i0 + k, L - 1)) * d.cqkv + ch);
}

// The same, into registers (tokens i0..i0+31 of channel f, zero past L).
__device__ __forceinline__ void conv_compute_regs(const ConvIn& in, int L, float* y) {
  const int i0 = (threadIdx.x >> 7) * 32;
  float xm3 = in.hist[0], xm2 = in.hist[1], xm1 = in.hist[2];
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    float acc = in.w[3] * in.xs[k];
    acc = fmaf(in.w[0], xm3, acc);
    acc = fmaf(in.w[1], xm2, acc);
    acc = fmaf(in.w[2], xm1, acc);
    y[k] = (i0 + k < L) ? silu_fast(acc) : 0.f;
    xm3 = xm2;
    xm2 = xm1;
    xm1 = in.xs[k];
  }
}

__device__ __forceinline__ void conv_compute(const ConvIn& in, int L, float* X) {
  const int tid = threadIdx.x;
  const int f = tid & 127, i0 = (tid >> 7) * 32;
  float xm3 = in.hist[0], xm2 = in.hist[1], xm1 = in.hist[2];
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    float acc = in.w[3] * in.xs[k];
    acc = fmaf(in.w[0], xm3, acc);
    acc = fmaf(in.w[1], xm2, acc);
    acc = fmaf(in.w[2], xm1, acc);
    X[(i0 + k) * XS + f] = (i0 + k < L) ? silu_fast(acc) : 0.f;
    xm3 = xm2;
    xm2 = xm1;
    xm1 = in.xs[k];
  }
}

// Per-row l2 normalisation of X (64 rows x 128), times scale.
// Warp w normalises rows w, w + 8, ..., all eight at once (their reductions interleave).
__device__ __forceinline__ void l2norm_rows(float* X, float eps, float scale) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int RPW = CH / (NTI / 32);
  float4 v[RPW];
  float ss[RPW];
#pragma unroll
  for (int m = 0; m < RPW; ++m) {
    v[m] = *reinterpret_cast<const float4*>(X + (warp + m * (NTI / 32)) * XS + 4 * lane);
    ss[m] = v[m].x * v[m].x + v[m].y * v[m].y + v[m].z * v[m].z + v[m].w * v[m].w;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
#pragma unroll
    for (int m = 0; m < RPW; ++m) ss[m] += __shfl_xor_sync(0xffffffffu, ss[m], off);
#pragma unroll
  for (int m = 0; m < RPW; ++m) {
    const float inv = scale * rsqrtf(ss[m] + eps);
    *reinterpret_cast<float4*>(X + (warp + m * (NTI / 32)) * XS + 4 * lane) =
        make_float4(v[m].x * inv, v[m].y * inv, v[m].z * inv, v[m].w * inv);
  }
}

// Rows [0,64) of X -> rows [0,64) of a 128-column K-major shared tile (hi / lo quarter).
// Unit u: row & 7 = u & 7, k-group = (u >> 3) & 15, row group = u >> 7 (conflict-free stores).
__device__ __forceinline__ void x_rows_to_tile(const float* X, unsigned char* hi, unsigned char* lo) {
  for (int u = threadIdx.x; u < 1024; u += NTI) {
    const int r = ((u >> 7) << 3) + (u & 7), kg = (u >> 3) & 15;
    const float4 a = *reinterpret_cast<const float4*>(X + r * XS + kg * 8);
    const float4 b = *reinterpret_cast<const float4*>(X + r * XS + kg * 8 + 4);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint4 hh, ll;
    split8(v, hh, ll);
    st_unit(hi, (uint32_t)u * 16u, hh);
    st_unit(lo, (uint32_t)u * 16u, ll);
  }
}

// (scale_j * K_j)^T tile [128 features][64 tokens] built from the K rows of A1 (hi + lo, about
// 16 significant bits), written into other shared memory (hi / lo).
__device__ __forceinline__ void a1k_cols_to_tile(const unsigned char* khi, const unsigned char* klo,
                                                 const float* scale, unsigned char* hi,
                                                 unsigned char* lo) {
  for (int u = threadIdx.x; u < 1024; u += NTI) {
    const int f = ((u >> 6) << 3) + (u & 7), jg = (u >> 3) & 7;
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = jg * 8 + q;
      const uint32_t off = tc::kmajor_off(j, f, 128);
      const float kv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(khi + off)) +
                       __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(klo + off));
      v[q] = kv * scale[j];
    }
    uint4 hh, ll;
    split8(v, hh, ll);
    st_unit(hi, (uint32_t)u * 16u, hh);
    st_unit(lo, (uint32_t)u * 16u, ll);
  }
}

template <typename T>
__global__ void __launch_bounds__(NTI, 2)
tc_intra_kernel(KDims d, const float* __restrict__ A_log, const float* __restrict__ dt_bias,
                const T* __restrict__ conv_w, const T* __restrict__ conv_state, int num_slots,
                const int32_t* __restrict__ cu, const int32_t* __restrict__ slot_idx,
                const uint8_t* __restrict__ has_init, int num_seqs, int total,
                const T* __restrict__ qkv, const T* __restrict__ a, const T* __restrict__ b,
                float* __restrict__ ws, int32_t* __restrict__ status) {
  extern __shared__ __align__(1024) unsigned char sm[];
  using S = IntraSmem;
  unsigned char* a1 = sm + S::A1;
  float* X = reinterpret_cast<float*>(sm + S::X);
  float* Am = reinterpret_cast<float*>(sm + S::AM);
  unsigned char* b2h = sm + S::B2;
  unsigned char* b2l = b2h + 8192;
  float* gam = reinterpret_cast<float*>(sm + S::VEC);
  float* bet = gam + 64;
  float* eg = bet + 64;
  float* dec = eg + 64;
  float* bgk = dec + 64;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + S::BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S::MISC);
  int* sh = reinterpret_cast<int*>(sm + S::MISC + 16);   // ok, t0, L, seq, seq_start, abort

  const int c = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    int seq, t0 = 0, len = 0, ss = 0;
    const bool ok = find_chunk(cu, num_seqs, total, c, seq, t0, len, ss);
    if (lane == 0 && !ok && c == 0 && h == 0) set_status(status, GDN_STATUS_BAD_SEQLENS);
    if (lane == 0) {
      sh[0] = ok && seq >= 0;
      sh[1] = t0;
      sh[2] = len;
      sh[3] = seq;
      sh[4] = ss;
      sh[5] = 0;
    }
  }
  __syncthreads();
  if (!sh[0]) return;
  const int t0 = sh[1], L = sh[2], seq = sh[3], seq_start = sh[4];
  const int seq_len = __ldg(cu + seq + 1) - seq_start;
  volatile int* abort = sh + 5;
  const int s = __ldg(slot_idx + seq);
  const bool valid = s >= 0 && s < num_slots;
  const bool init = valid && has_init != nullptr && __ldg(has_init + seq) != 0;
  const T* cs = conv_state + (size_t)(valid ? s : 0) * 3 * d.cqkv;
  const int kh = h / d.r;
  unsigned char* rec = reinterpret_cast<unsigned char*>(ws) + ((size_t)c * d.Hv + h) * REC_BYTES;
  float* rec_ut = reinterpret_cast<float*>(rec + R_UT);

  // K inputs in flight while the gates are formed
  ConvIn cin;
  conv_load<T>(d, qkv, conv_w, cs, init, d.Hk * D + kh * D, seq_start, seq_len, t0, L, cin);
  if (tid == 0) {
    tc::mbar_init(bar, 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) tc::tmem_alloc(tslot, 256);

  // ---- gates of the chunk: gamma (cumulative g), beta and the derived per-token scales
  if (warp == 0) {
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
    const float ex = incl - pair;
    gam[2 * lane] = ex + g2[0];
    gam[2 * lane + 1] = ex + g2[0] + g2[1];
    bet[2 * lane] = b2[0];
    bet[2 * lane + 1] = b2[1];
  }
  __syncthreads();
  const float gL = gam[L - 1];
  if (tid < CH) {
    eg[tid] = expf(gam[tid]);
    dec[tid] = tid < L ? expf(gL - gam[tid]) : 0.f;
    bgk[tid] = bet[tid] * expf(gam[tid]);
  }

  // ---- K: conv, l2norm, A1 K rows, K~^T rows of B4
  conv_compute(cin, L, X);
  conv_load<T>(d, qkv, conv_w, cs, init, kh * D, seq_start, seq_len, t0, L, cin);   // Q, in flight
  __syncthreads();
  l2norm_rows(X, d.l2_eps, 1.0f);
  __syncthreads();
  x_rows_to_tile(X, a1 + S::K_HI, a1 + S::K_LO);
  x_cols_to_gtile64(X, dec, rec + R_B4 + 8192, rec + R_B4 + B4_HALF + 8192);   // rows 64..191
  __syncthreads();
  // ---- Q: conv, l2norm (times q_scale), A1 Q rows, Q~ rows of B3
  conv_compute(cin, L, X);
  conv_load<T>(d, qkv, conv_w, cs, init, 2 * d.Hk * D + h * D, seq_start, seq_len, t0, L, cin);  // V
  __syncthreads();
  l2norm_rows(X, d.l2_eps, d.q_scale);
  __syncthreads();
  x_rows_to_tile(X, a1 + S::Q_HI, a1 + S::Q_LO);
  x_rows_to_gtile128(X, eg, rec + R_B3, rec + R_B3 + B3_HALF, 0);
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = *tslot;
  // ---- D1 = [K;Q] K^T  (cols [0,64)); A1's hi quarters [K|Q] and lo quarters form 128-row tiles
  if (tid == 0) {
    const uint32_t id = tc::idesc_bf16(128, 64);
    const uint32_t ah = tc::smem_u32(a1 + S::K_HI), al = tc::smem_u32(a1 + S::K_LO);
    const uint64_t dh = tc::kstep_desc(ah, 128, 0), dl = tc::kstep_desc(al, 128, 0);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint64_t h = tc::desc_add(dh, 256 * k), l = tc::desc_add(dl, 256 * k);
      tc::mma_bf16(tb, h, h, id, k > 0);
      tc::mma_bf16(tb, h, l, id, 1);
      tc::mma_bf16(tb, l, h, id, 1);
    }
    tc::mma_commit(bar);
  }
  // ---- V (overlaps the MMA): conv into registers
  float vy[32];
  conv_compute_regs(cin, L, vy);
  // ---- A1 is free once MMA1 completed: (beta e^g K)^T into its Q quarters, then (beta V)^T
  // into its K quarters, straight from the V registers (thread: feature f, tokens i0..i0+31,
  // i.e. four 8-token units of the K-major [128 features][64 tokens] tile)
  wait_or_abort(bar, 0, abort, status);
  tc::fence_after_sync();
  a1k_cols_to_tile(a1 + S::K_HI, a1 + S::K_LO, bgk, a1 + S::Q_HI, a1 + S::Q_LO);
  __syncthreads();
  {
    const int f = tid & 127, i0 = (tid >> 7) * 32;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      float v8[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v8[q] = vy[8 * g + q] * bet[i0 + 8 * g + q];
      uint4 hh, ll;
      split8(v8, hh, ll);
      const uint32_t off = tc::kmajor_off(f, i0 + 8 * g, 64);
      st_unit(a1 + S::K_HI, off, hh);
      st_unit(a1 + S::K_LO, off, ll);
    }
  }
  // ---- A and P from D1: warp w reads TMEM lanes 32 (w % 4) and the 32 columns of half w / 4
  {
    const int r = (warp & 3) * 32 + lane, j0 = (warp >> 2) * 32;
    float v[32];
    tc::tmem_ld16(tc::taddr(tb, (warp & 3) * 32, j0), v);
    tc::tmem_ld16(tc::taddr(tb, (warp & 3) * 32, j0 + 16), v + 16);
    // branch-free: exponents clamped to <= 0, masked entries multiplied by zero
    if (r < 64) {
      const int i = r;
      const float gi = gam[i], bi = (i < L) ? bet[i] : 0.f;
#pragma unroll
      for (int q = 0; q < 32; q += 4) {
        float a4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + q + u;
          const float m = (j < i) ? bi : 0.f;
          a4[u] = m * exp_fast(fminf(gi - gam[j], 0.f)) * v[q + u];
        }
        *reinterpret_cast<float4*>(Am + i * AS + j0 + q) = make_float4(a4[0], a4[1], a4[2], a4[3]);
      }
    } else {
      const int i = r - 64;
      const float gi = gam[i], vi = (i < L) ? 1.f : 0.f;
#pragma unroll
      for (int q = 0; q < 32; q += 8) {
        float p8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = j0 + q + u;
          p8[u] = ((j <= i) ? vi : 0.f) * exp_fast(fminf(gi - gam[j], 0.f)) * v[q + u];
        }
        uint4 hh, ll;
        split8(p8, hh, ll);
        const uint32_t off = tc::kmajor_off(i, j0 + q, 64);   // P rows 0..63 of B4
        gst_unit(rec + R_B4, off, hh);
        gst_unit(rec + R_B4 + B4_HALF, off, ll);
      }
    }
  }
  __syncthreads();
  // ---- T = (I + A)^{-1}, A strictly lower triangular, in 16 x 16 blocks: the diagonal inverses
  // D_b = (I + A_bb)^{-1} by forward substitution (the four in parallel), then block row by block
  // row  T_ik = -D_i sum_{j=k}^{i-1} A_ij T_jk  (k < i), each a few dense 16 x 16 products over
  // all threads instead of one 64-step dependent chain.  T replaces A in Am (D_b over A_bb, T_ik
  // over A_ik once block row i of A has been used); the partial sums X_ik live in the unused
  // upper block (k, i).  Each final block also goes to the split-bf16 B2 tile (rows i, K = j).
  {
    auto put_b2 = [&](int row, int col, float v) {
      __nv_bfloat16 hi, lo;
      tc::split_bf16(v, hi, lo);
      const uint32_t off = tc::kmajor_off(row, col, 64);
      *reinterpret_cast<__nv_bfloat16*>(b2h + off) = hi;
      *reinterpret_cast<__nv_bfloat16*>(b2l + off) = lo;
    };
    float dcol[16];
    const int db = tid >> 4, dc = tid & 15;   // threads 0-63: column dc of D_db
    if (tid < 64) {
      const float* ab = Am + (16 * db) * AS + 16 * db;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float arow[16];
#pragma unroll
        for (int m = 0; m < 16; m += 4) {
          const float4 a4 = *reinterpret_cast<const float4*>(ab + i * AS + m);
          arow[m] = a4.x;
          arow[m + 1] = a4.y;
          arow[m + 2] = a4.z;
          arow[m + 3] = a4.w;
        }
        float acc = (i == dc) ? 1.f : 0.f;
#pragma unroll
        for (int j = 0; j < i; ++j) acc = fmaf(-arow[j], dcol[j], acc);
        dcol[i] = acc;
      }
    } else {
      // the six upper blocks of B2 are zero
      for (int u = tid - 64; u < 6 * 256; u += NTI - 64) {
        const int blk = u >> 8, el = u & 255;
        const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        put_b2(16 * bi + (el >> 4), 16 * bj + (el & 15), 0.f);
      }
    }
    __syncthreads();
    if (tid < 64) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        Am[(16 * db + i) * AS + 16 * db + dc] = dcol[i];
        put_b2(16 * db + i, 16 * db + dc, dcol[i]);
      }
    }
    __syncthreads();
    const int r = tid >> 4, cc = tid & 15;   // element (r, cc) of every 16 x 16 block
#pragma unroll
    for (int i = 1; i < 4; ++i) {
      const float* arow = Am + (16 * i + r) * AS;
#pragma unroll
      for (int k = 0; k < i; ++k) {   // X_ik -> block (k, i)
        float acc = 0.f;
#pragma unroll
        for (int j = k; j < i; ++j) {
          const float* tcol = Am + (16 * j) * AS + 16 * k + cc;
#pragma unroll
          for (int m = 0; m < 16; m += 4) {
            const float4 a4 = *reinterpret_cast<const float4*>(arow + 16 * j + m);
            acc = fmaf(a4.x, tcol[m * AS], acc);
            acc = fmaf(a4.y, tcol[(m + 1) * AS], acc);
            acc = fmaf(a4.z, tcol[(m + 2) * AS], acc);
            acc = fmaf(a4.w, tcol[(m + 3) * AS], acc);
          }
        }
        Am[(16 * k + r) * AS + 16 * i + cc] = acc;
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < i; ++k) {   // T_ik = -D_i X_ik -> block (i, k)
        const float* xcol = Am + (16 * k) * AS + 16 * i + cc;
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m += 4) {
          const float4 d4 = *reinterpret_cast<const float4*>(arow + 16 * i + m);
          acc = fmaf(d4.x, xcol[m * AS], acc);
          acc = fmaf(d4.y, xcol[(m + 1) * AS], acc);
          acc = fmaf(d4.z, xcol[(m + 2) * AS], acc);
          acc = fmaf(d4.w, xcol[(m + 3) * AS], acc);
        }
        Am[(16 * i + r) * AS + 16 * k + cc] = -acc;
        put_b2(16 * i + r, 16 * k + cc, -acc);
      }
      if (i < 3) __syncthreads();
    }
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // ---- D2a = (beta e^g K)^T T^T = W^T (cols [64,128)),  D2b = (beta V)^T T^T = U~^T ([128,192))
  if (tid == 0 && !*abort) {
    const uint32_t id = tc::idesc_bf16(128, 64);
    const uint32_t bh = tc::smem_u32(b2h), bl = tc::smem_u32(b2l);
    const uint32_t srcs[2][2] = {{tc::smem_u32(a1 + S::Q_HI), tc::smem_u32(a1 + S::Q_LO)},
                                 {tc::smem_u32(a1 + S::K_HI), tc::smem_u32(a1 + S::K_LO)}};
    const uint64_t dbh = tc::kstep_desc(bh, 64, 0), dbl = tc::kstep_desc(bl, 64, 0);
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const uint32_t dt = tb + 64 + 64 * m;
      const uint64_t dah = tc::kstep_desc(srcs[m][0], 64, 0), dal = tc::kstep_desc(srcs[m][1], 64, 0);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t o = 256 * k;
        tc::mma_bf16(dt, tc::desc_add(dah, o), tc::desc_add(dbh, o), id, k > 0);
        tc::mma_bf16(dt, tc::desc_add(dah, o), tc::desc_add(dbl, o), id, 1);
        tc::mma_bf16(dt, tc::desc_add(dal, o), tc::desc_add(dbh, o), id, 1);
      }
    }
    tc::mma_commit(bar);
  }
  wait_or_abort(bar, 1, abort, status);
  tc::fence_after_sync();
  {
    // warps 0-3: W^T lanes -> X staging [token][feature]; warps 4-7: U~^T lanes -> U~ rows
    const int r = (warp & 3) * 32 + lane;
    const int col = warp < 4 ? 64 : 128;
#pragma unroll
    for (int hb = 0; hb < 64; hb += 32) {
      float v[32];
      tc::tmem_ld16(tc::taddr(tb, (warp & 3) * 32, col + hb), v);
      tc::tmem_ld16(tc::taddr(tb, (warp & 3) * 32, col + hb + 16), v + 16);
      if (warp < 4) {
#pragma unroll
        for (int i = 0; i < 32; ++i) X[(hb + i) * XS + r] = v[i];
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) rec_ut[(hb + i) * D + r] = v[i];
      }
    }
  }
  __syncthreads();
  x_rows_to_gtile128(X, nullptr, rec + R_B3, rec + R_B3 + B3_HALF, 64);   // W rows of B3
  if (tid == 0) *reinterpret_cast<float*>(rec + R_SC) = expf(gL);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, 256);
}

// ================================================================== serial state kernel
//
// One cluster of four CTAs per (sequence, V-head); CTA sigma owns the state columns
// [32 sigma, 32 sigma + 32) of S (dk x dv) -- the chunk recurrence never mixes dv columns, so the
// four slices run independently and only the output RMSNorm (over all dv) needs an exchange of
// per-token partial sums of squares between the CTAs of the cluster.

constexpr int NSL = 4;                        // dv slices (CTAs) per head
constexpr int SW = D / NSL;                   // 32 columns per slice
constexpr uint32_t PLBO = 144;                // padded K-direction core-matrix stride (bytes)
constexpr uint32_t SOP_SBO = (D / 8) * PLBO;  // S operand: N = 32 rows, K = 128 (dk)
constexpr uint32_t SOP_HALF = (SW / 8) * SOP_SBO;
constexpr uint32_t UOP_SBO = (CH / 8) * PLBO; // U operand: N = 32 rows, K = 64 (tokens)
constexpr uint32_t UOP_HALF = (SW / 8) * UOP_SBO;
constexpr int NTS = 448;   // warps 0-7 main, 8-9 and 12-13 epilogue, 10 loader (11 idle)
constexpr int MH = SW / 2; // columns per main warp: warp w takes lanes 32 (w % 4) and half w / 4
constexpr int NDB = 4;     // D3 (output) accumulators in flight between the MMAs and the epilogue
constexpr int XH = 2;      // epilogue column halves: partial sums per token and CTA
constexpr int NXB = 4;     // exchange buffers: chunk c's sums are sent one epilogue step before use

// TMEM columns (lanes 0-127).  Each product runs as two N = 64 MMAs per K-step, A_hi [B_hi ; B_lo]
// and A_lo [B_hi ; B_lo] (the B operand holds the hi rows 0-31 and the lo rows 32-63), so every
// accumulator occupies 64 columns whose two 32-column halves add up to the result.
constexpr uint32_t TC_S = 0;          // S slice, halves [0, 32) + [32, 64)
constexpr uint32_t TC_D3 = 64;        // NDB x 64 columns: rows 0-63 O, rows 64-127 W S
constexpr uint32_t TC_COLS = 512;

struct StateSmem {
  static constexpr uint32_t B3 = 0;                        // 2 slots: [Q~ ; W] rows [128 x 128], hi then lo
  static constexpr uint32_t B4 = B3 + 2 * 65536;           // [P ; K~^T] rows [192 x 64], hi then lo
  static constexpr uint32_t SOP = B4 + 2 * 24576;          // S slice as B operand, hi then lo
  static constexpr uint32_t UOP = SOP + 2 * SOP_HALF;      // U slice as B operand, hi then lo
  static constexpr uint32_t XBUF = UOP + 2 * UOP_HALF;     // f32 [NXB][NSL][XH][64] partial sums
  static constexpr uint32_t BAR = XBUF + NXB * NSL * XH * 64 * 4;   // 20 mbarriers
  static constexpr uint32_t MISC = BAR + 160;
  static constexpr uint32_t BYTES = MISC + 64;
};

template <typename T>
__global__ void __cluster_dims__(NSL, 1, 1) __launch_bounds__(NTS, 1)
tc_state_kernel(KDims d, const T* __restrict__ norm_w, float* __restrict__ rec_state,
                T* __restrict__ conv_state, int num_slots, const int32_t* __restrict__ cu,
                const int32_t* __restrict__ slot_idx, const uint8_t* __restrict__ has_init,
                int num_seqs, int total, const T* __restrict__ qkv, const T* __restrict__ z,
                T* __restrict__ out, const float* __restrict__ ws, int32_t* __restrict__ status) {
  extern __shared__ __align__(1024) unsigned char sm[];
  using S = StateSmem;
  unsigned char* b4h = sm + S::B4;
  unsigned char* b4l = b4h + 24576;
  unsigned char* soph = sm + S::SOP;
  unsigned char* sopl = soph + SOP_HALF;
  unsigned char* uoph = sm + S::UOP;
  unsigned char* uopl = uoph + UOP_HALF;
  float* xbuf = reinterpret_cast<float*>(sm + S::XBUF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S::BAR);
  uint64_t* b3full = bars + 0;   // [2] B3 slot landed (loader -> MMA)
  uint64_t* b3empty = bars + 2;  // [2] B3 slot read by MMA3 (MMA -> loader)
  uint64_t* b4full = bars + 4;   // B4 landed
  uint64_t* b4empty = bars + 5;  // B4 read by MMA4
  uint64_t* mma3 = bars + 6;
  uint64_t* sready = bars + 7;   // S += K~^T U of the chunk done (the next chunk may read S)
  uint64_t* dfull = bars + 8;    // [NDB] O of the chunk complete in D3[j] (MMA -> epilogue)
  uint64_t* dempty = bars + 12;  // [NDB] D3[j] read by the epilogue (epilogue -> MMA)
  uint64_t* xfull = bars + 16;   // [NXB] partial sums of the 4 slices arrived
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S::MISC);
  int* sh = reinterpret_cast<int*>(sm + S::MISC + 16);

  const int n = blockIdx.x / NSL, sig = blockIdx.x % NSL, h = blockIdx.y;
  const uint32_t crank = tc::cluster_ctarank();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    int off = 0;
    const bool ok = seq_chunk_offset(cu, num_seqs, total, n, off);
    if (lane == 0 && !ok && n == 0 && h == 0 && sig == 0) set_status(status, GDN_STATUS_BAD_SEQLENS);
    if (lane == 0) {
      sh[0] = ok;
      sh[1] = off;
      sh[2] = 0;
    }
  }
  if (tid == 0) {
    for (int i = 0; i < 20; ++i) tc::mbar_init(bars + i, (i >= 12 && i < 16) ? 128 : 1);
    tc::mbar_fence_init();
    for (int i = 0; i < NXB; ++i) tc::mbar_arrive_expect_tx(xfull + i, NSL * XH * 64 * 4);   // chunks 0-3
  }
  if (warp == 0) tc::tmem_alloc(tslot, TC_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  tc::cluster_sync_all();   // peers' mbarriers initialised before any exchange
  const uint32_t tb = *tslot;
  const int choff = sh[1];
  volatile int* abort = sh + 2;
  const int seq_start = __ldg(cu + n), len = __ldg(cu + n + 1) - seq_start;
  const int nch = sh[0] ? (len + CH - 1) / CH : 0;
  const int s = __ldg(slot_idx + n);
  // invalid cu_seqlens: nothing is read or written (the CTA still takes part in the cluster syncs)
  const bool valid = sh[0] && s >= 0 && s < num_slots;
  if (sh[0] && s >= num_slots && h == 0 && sig == 0 && tid == 0) set_status(status, GDN_STATUS_SLOT_RANGE);
  const bool init = valid && has_init != nullptr && __ldg(has_init + n) != 0;
  float* Sg = rec_state + ((size_t)(valid ? s : 0) * d.Hv + h) * D * D + sig * SW;
  auto rec_of = [&](int c) {
    return reinterpret_cast<const unsigned char*>(ws) + ((size_t)(choff + c) * d.Hv + h) * REC_BYTES;
  };

  if (warp < 8) {
    // ================= main warps: thread e owns TMEM lane e = row e (dk index) of the S slice and
    // its columns [mh, mh + 16) (of both accumulator halves)
    const int e = (warp & 3) * 32 + lane, mh = (warp >> 2) * MH;
    const uint32_t lane_base = tc::taddr(tb, (warp & 3) * 32, 0);
    {
      float v[MH];
#pragma unroll
      for (int q = 0; q < MH; q += 4) {
        const float4 x = init ? *reinterpret_cast<const float4*>(Sg + (size_t)e * D + mh + q)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        v[q] = x.x;
        v[q + 1] = x.y;
        v[q + 2] = x.z;
        v[q + 3] = x.w;
      }
      tc::tmem_st16(lane_base + TC_S + mh, v);
#pragma unroll
      for (int q = 0; q < MH; ++q) v[q] = 0.f;
      tc::tmem_st16(lane_base + TC_S + SW + mh, v);
    }
    const int t = e - 64;             // token row of W S / U for lanes 64..127
    const bool urow = (warp & 3) >= 2;
    float ut[MH];                     // U~ of token t, columns mh.., loaded one chunk ahead
    if (urow && nch > 0) {
      const float* u0 = reinterpret_cast<const float*>(rec_of(0) + R_UT) + t * D + sig * SW + mh;
#pragma unroll
      for (int q = 0; q < MH; q += 4) {
        const float4 x = *reinterpret_cast<const float4*>(u0 + q);
        ut[q] = x.x;
        ut[q + 1] = x.y;
        ut[q + 2] = x.z;
        ut[q + 3] = x.w;
      }
    }
    float egL_next = nch > 0 ? *reinterpret_cast<const float*>(rec_of(0) + R_SC) : 1.f;
    // operand descriptors, built once (K-step k: + 256 bytes for the dense tiles, + 2 PLBO for
    // the padded ones)
    const uint32_t id64 = tc::idesc_bf16(128, 2 * SW);
    const uint64_t dA3h = tc::kstep_desc(tc::smem_u32(sm + S::B3), 128, 0);   // slot 0; slot 1 + 64 KiB
    const uint64_t dA3l = tc::kstep_desc(tc::smem_u32(sm + S::B3 + B3_HALF), 128, 0);
    const uint64_t dKh = tc::kstep_desc(tc::smem_u32(b4h) + 8192, 64, 0);
    const uint64_t dKl = tc::kstep_desc(tc::smem_u32(b4l) + 8192, 64, 0);
    const uint64_t dPh = tc::kstep_desc(tc::smem_u32(b4h), 64, 0);
    const uint64_t dPl = tc::kstep_desc(tc::smem_u32(b4l), 64, 0);
    const uint64_t dS = tc::kstep_desc_p(tc::smem_u32(soph), PLBO, SOP_SBO, 0);
    const uint64_t dU = tc::kstep_desc_p(tc::smem_u32(uoph), PLBO, UOP_SBO, 0);
    for (int c = 0; c < nch; ++c) {
      const uint32_t par = c & 1, b = c & 1;
      const uint32_t jd = c & (NDB - 1);
      const uint32_t d3 = tb + TC_D3 + 64 * jd;   // D3[jd]: rows 0-63 O (Q~ S + P U), rows 64-127 W S
      // S slice -> B operand (split bf16, unscaled: W S and Q~ S use the chunk's initial state),
      // and S <- e^{gamma_L} S in TMEM for the K~^T U accumulation
      const float egL = egL_next;
      if (c + 1 < nch) egL_next = *reinterpret_cast<const float*>(rec_of(c + 1) + R_SC);
      {
        uint32_t rv[2 * MH];
        tc::tmem_ld16_nw(lane_base + TC_S + mh, rv);
        tc::tmem_ld16_nw(lane_base + TC_S + SW + mh, rv + MH);
        tc::tmem_wait_ld();
        tc::reg_fence16(rv);
        tc::reg_fence16(rv + MH);
        float v[MH];
#pragma unroll
        for (int q = 0; q < MH; ++q) {
          v[q] = __uint_as_float(rv[q]) + __uint_as_float(rv[q + MH]);
          __nv_bfloat16 hi, lo;
          tc::split_bf16(v[q], hi, lo);
          const uint32_t off = tc::kmajor_off_p(mh + q, e, PLBO, SOP_SBO);
          *reinterpret_cast<__nv_bfloat16*>(soph + off) = hi;
          *reinterpret_cast<__nv_bfloat16*>(sopl + off) = lo;
          v[q] *= egL;
        }
        tc::tmem_st16_nw(lane_base + TC_S + mh, v);
#pragma unroll
        for (int q = 0; q < MH; ++q) v[q] = 0.f;
        tc::tmem_st16_nw(lane_base + TC_S + SW + mh, v);
        tc::tmem_wait_st();
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      bar_sync_main();
      tc::fence_after_sync();
      if (tid == 0 && wait_or_abort(b3full + b, (c >> 1) & 1, abort, status) &&
          (c < NDB || wait_or_abort(dempty + jd, ((c / NDB) - 1) & 1, abort, status))) {
        tc::fence_after_sync();
        const uint32_t so = 65536u * b;   // B3 slot of the chunk
#pragma unroll
        for (int k = 0; k < 8; ++k) {   // B = [S_hi ; S_lo], 64 rows
          const uint64_t bk = tc::desc_add(dS, 2 * PLBO * k);
          tc::mma_bf16(d3, tc::desc_add(dA3h, so + 256 * k), bk, id64, k > 0);
          tc::mma_bf16(d3, tc::desc_add(dA3l, so + 256 * k), bk, id64, 1);
        }
        tc::mma_commit(mma3);
        tc::mma_commit(b3empty + b);
      }
      wait_or_abort(mma3, par, abort, status);
      tc::fence_after_sync();
      // U = U~ - W S (tokens 0..63 on lanes 64..127) -> B operand
      if (urow) {
        uint32_t rv[2 * MH];
        tc::tmem_ld16_nw(tc::taddr(d3, (warp & 3) * 32, mh), rv);
        tc::tmem_ld16_nw(tc::taddr(d3, (warp & 3) * 32, SW + mh), rv + MH);
        tc::tmem_wait_ld();
        tc::reg_fence16(rv);
        tc::reg_fence16(rv + MH);
#pragma unroll
        for (int q = 0; q < MH; ++q) {
          __nv_bfloat16 hi, lo;
          tc::split_bf16(ut[q] - (__uint_as_float(rv[q]) + __uint_as_float(rv[q + MH])), hi, lo);
          const uint32_t off = tc::kmajor_off_p(mh + q, t, PLBO, UOP_SBO);
          *reinterpret_cast<__nv_bfloat16*>(uoph + off) = hi;
          *reinterpret_cast<__nv_bfloat16*>(uopl + off) = lo;
        }
        if (c + 1 < nch) {
          const float* un = reinterpret_cast<const float*>(rec_of(c + 1) + R_UT) + t * D + sig * SW + mh;
#pragma unroll
          for (int q = 0; q < MH; q += 4) {
            const float4 x = *reinterpret_cast<const float4*>(un + q);
            ut[q] = x.x;
            ut[q + 1] = x.y;
            ut[q + 2] = x.z;
            ut[q + 3] = x.w;
          }
        }
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      bar_sync_main();
      tc::fence_after_sync();
      if (tid == 0 && wait_or_abort(b4full, par, abort, status)) {
        tc::fence_after_sync();
#pragma unroll
        for (int k = 0; k < 4; ++k) {   // S += K~^T U   (B4 rows 64..191; B = [U_hi ; U_lo])
          const uint64_t bk = tc::desc_add(dU, 2 * PLBO * k);
          tc::mma_bf16(tb + TC_S, tc::desc_add(dKh, 256 * k), bk, id64, 1);
          tc::mma_bf16(tb + TC_S, tc::desc_add(dKl, 256 * k), bk, id64, 1);
        }
        tc::mma_commit(sready);   // the next chunk's S conversion overlaps the O products below
        // D3 += [P ; K~^T rows 0..63] U: rows 0..63 become O; rows 64..127 (W S, consumed) are
        // left as scratch
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t bk = tc::desc_add(dU, 2 * PLBO * k);
          tc::mma_bf16(d3, tc::desc_add(dPh, 256 * k), bk, id64, 1);
          tc::mma_bf16(d3, tc::desc_add(dPl, 256 * k), bk, id64, 1);
        }
        tc::mma_commit(b4empty);
        tc::mma_commit(dfull + jd);
      }
      // S is final for this chunk.  The O products may still run: they read only B4 and the U
      // operand (rewritten only after the next chunk's MMA3, which the pipe orders after them)
      // and write D3[jd], which the next chunk does not touch.
      wait_or_abort(sready, par, abort, status);
      tc::fence_after_sync();
    }
    // final state slice back to the slot
    if (valid) {
      float v[2 * MH];
      tc::tmem_ld16(lane_base + TC_S + mh, v);
      tc::tmem_ld16(lane_base + TC_S + SW + mh, v + MH);
#pragma unroll
      for (int q = 0; q < MH; ++q) v[q] += v[q + MH];
#pragma unroll
      for (int q = 0; q < MH; q += 4)
        *reinterpret_cast<float4*>(Sg + (size_t)e * D + mh + q) = make_float4(v[q], v[q + 1], v[q + 2], v[q + 3]);
    }
  } else if (warp == 11) {
    // idle
  } else if (warp == 10) {
    // ================= loader warp: bulk copies of the chunks' operand images, each issued as soon
    // as MMA has finished reading the buffer it refills (B3 double-buffered, B4 single)
    if (lane == 0) {
      int n3a = 0, n3b = 0, n4 = 0;   // copies issued per buffer
      auto load_b3 = [&](int c) {
        const int j = c & 1;
        tc::mbar_arrive_expect_tx(b3full + j, 2 * B3_HALF);
        tc::bulk_g2s(sm + S::B3 + j * 65536, rec_of(c) + R_B3, 2 * B3_HALF, b3full + j);
        if (j) ++n3b;
        else ++n3a;
      };
      auto load_b4 = [&](int c) {
        tc::mbar_arrive_expect_tx(b4full, 2 * B4_HALF);
        tc::bulk_g2s(b4h, rec_of(c) + R_B4, 2 * B4_HALF, b4full);
        ++n4;
      };
      if (nch > 0) load_b3(0);
      if (nch > 0) load_b4(0);
      if (nch > 1) load_b3(1);
      for (int c = 0; c + 1 < nch; ++c) {
        if (!wait_or_abort(b4empty, c & 1, abort, status)) break;
        load_b4(c + 1);
        if (c + 2 < nch) {
          if (!wait_or_abort(b3empty + (c & 1), (c >> 1) & 1, abort, status)) break;
          load_b3(c + 2);
        }
      }
      // after a timeout: wait (bounded) for the copies still in flight before the CTA exits
      if (*abort) {
        if (n3a > 0) tc::mbar_wait(b3full, (n3a - 1) & 1, 100000000ull);
        if (n3b > 0) tc::mbar_wait(b3full + 1, (n3b - 1) & 1, 100000000ull);
        if (n4 > 0) tc::mbar_wait(b4full, (n4 - 1) & 1, 100000000ull);
      }
    }
  } else {
    // ================= epilogue warps 8, 9, 12, 13: thread t owns token t of the chunk (TMEM lane t
    // of D3) and the 16 columns of half xh of the slice
    const int t = (warp & 3) * 32 + lane, xh = (warp >> 2) & 1;
    constexpr int EW = SW / XH;
    const size_t ld = (size_t)d.Hv * D;
    const size_t col0 = (size_t)h * D + sig * SW + xh * EW;
    float wn[EW];
#pragma unroll
    for (int q = 0; q < EW; q += 4) {
      const float4 x = Act<T>::ldg4(norm_w + sig * SW + xh * EW + q);
      wn[q] = x.x;
      wn[q + 1] = x.y;
      wn[q + 2] = x.z;
      wn[q + 3] = x.w;
    }
    // software-pipelined over the chunks: step c reads chunk c's outputs and sends their partial
    // sums of squares to the cluster, then normalises and stores chunk c - 1, whose sums were
    // sent one step earlier (so the exchange latency overlaps a step of work)
    auto load_z = [&](int c, float4* zz) {
      const int i = min(t, min(CH, len - c * CH) - 1);
      const T* zp = z + (size_t)(seq_start + c * CH + i) * ld + col0;
#pragma unroll
      for (int q = 0; q < EW / 4; ++q) zz[q] = Act<T>::ldg4(zp + 4 * q);
    };
    float4 zc[EW / 4], zp[EW / 4];   // z of chunk c (loaded at step c) and of chunk c - 1
    float oc[EW], op[EW];
    const uint32_t xb_local = tc::smem_u32(xbuf);
    const uint32_t xf_local = tc::smem_u32(xfull);
    bool xok = true;
    for (int c = 0; c <= nch; ++c) {
#pragma unroll
      for (int q = 0; q < EW; ++q) op[q] = oc[q];
#pragma unroll
      for (int q = 0; q < EW / 4; ++q) zp[q] = zc[q];
      if (c < nch) {
        const uint32_t jd = c & (NDB - 1), xb = c & (NXB - 1);
        wait_or_abort(dfull + jd, (c / NDB) & 1, abort, status);
        tc::fence_after_sync();
        float o2[2 * EW];
        const uint32_t da = tc::taddr(tb + TC_D3 + 64 * jd, (warp & 3) * 32, xh * EW);
        tc::tmem_ld16(da, o2);
        tc::tmem_ld16(da + SW, o2 + EW);
        tc::fence_before_sync();
        mbar_arrive(dempty + jd);
        float ss = 0.f;
#pragma unroll
        for (int q = 0; q < EW; ++q) {
          oc[q] = o2[q] + o2[q + EW];
          ss = fmaf(oc[q], oc[q], ss);
        }
        const uint32_t slot_off = (((xb * NSL + crank) * XH + xh) * 64 + t) * 4;
#pragma unroll
        for (uint32_t r = 0; r < NSL; ++r)
          tc::st_async_f32(tc::mapa_shared(xb_local + slot_off, r), ss,
                           tc::mapa_shared(xf_local + xb * 8, r));
        load_z(c, zc);
      }
      if (c >= 1) {
        const int cp = c - 1;
        const uint32_t xb = cp & (NXB - 1);
        const int L = min(CH, len - cp * CH);
        if (xok && !tc::mbar_wait_cluster(xfull + xb, (cp / NXB) & 1)) {
          xok = false;
          *abort = 1;
          set_status(status, GDN_STATUS_TIMEOUT);
        }
        // this buffer's next use is chunk cp + NXB: its peers send that only after this CTA has
        // sent chunk cp + 2, so posting the expected bytes now comes first
        if (warp == 8 && lane == 0 && cp + NXB < nch) {
          tc::mbar_arrive_expect_tx(xfull + xb, NSL * XH * 64 * 4);
          tc::fence_acq_rel_cluster();
        }
        float tot = 0.f;
#pragma unroll
        for (int r = 0; r < NSL * XH; ++r) tot += xbuf[(xb * NSL * XH + r) * 64 + t];
        const float inv = valid ? rsqrtf(tot * (1.0f / (float)D) + d.norm_eps) : 0.f;
        if (t < L) {
          T* o_ptr = out + (size_t)(seq_start + cp * CH + t) * ld + col0;
#pragma unroll
          for (int q = 0; q < EW / 4; ++q) {
            const float4 r4 = make_float4(op[4 * q] * inv * wn[4 * q] * silu_fast(zp[q].x),
                                          op[4 * q + 1] * inv * wn[4 * q + 1] * silu_fast(zp[q].y),
                                          op[4 * q + 2] * inv * wn[4 * q + 2] * silu_fast(zp[q].z),
                                          op[4 * q + 3] * inv * wn[4 * q + 3] * silu_fast(zp[q].w));
            Act<T>::store4(o_ptr + 4 * q, r4);
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, TC_COLS);
  // conv state <- the sequence's last K-1 raw inputs (older ones kept when continuing)
  if (valid && h == 0 && sig == 0) {
    T* csw = conv_state + (size_t)s * 3 * d.cqkv;
    for (int cch = tid; cch < d.cqkv; cch += NTS) {
      T v3[3];
#pragma unroll
      for (int m = 0; m < 3; ++m) {
        const int rel = len - 3 + m;
        if (rel >= 0) v3[m] = qkv[(size_t)(seq_start + rel) * d.cqkv + cch];
        else v3[m] = init ? csw[(size_t)(3 + rel) * d.cqkv + cch] : Act<T>::cvt(0.f);
      }
#pragma unroll
      for (int m = 0; m < 3; ++m) csw[(size_t)m * d.cqkv + cch] = v3[m];
    }
  }
  tc::cluster_sync_all();   // no CTA leaves while a peer may still store into its shared memory
}

template <typename T>
int launch_t(const KDims& d, const gdn_weights* w, const gdn_pool* pool, const int32_t* cu,
             const int32_t* slot_idx, const uint8_t* has_init, int num_seqs, int total,
             const void* qkv, const void* z, const void* a, const void* b, void* out, void* ws,
             cudaStream_t stream) {
  const int nc_max = total / CH + num_seqs;
  auto k1 = tc_intra_kernel<T>;
  auto k2 = tc_state_kernel<T>;
  if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)IntraSmem::BYTES) !=
          cudaSuccess ||
      cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)StateSmem::BYTES) !=
          cudaSuccess)
    return GDN_ERR_CUDA;
  float* wsf = static_cast<float*>(ws);
  if (total > 0)
    k1<<<dim3(nc_max, d.Hv), NTI, IntraSmem::BYTES, stream>>>(
        d, w->A_log, w->dt_bias, static_cast<const T*>(w->conv_weight),
        static_cast<const T*>(pool->conv_state), pool->num_slots, cu, slot_idx, has_init, num_seqs,
        total, static_cast<const T*>(qkv), static_cast<const T*>(a), static_cast<const T*>(b), wsf,
        pool->status);
  k2<<<dim3(NSL * num_seqs, d.Hv), NTS, StateSmem::BYTES, stream>>>(
      d, static_cast<const T*>(w->norm_weight), pool->rec_state, static_cast<T*>(pool->conv_state),
      pool->num_slots, cu, slot_idx, has_init, num_seqs, total, static_cast<const T*>(qkv),
      static_cast<const T*>(z), static_cast<T*>(out), wsf, pool->status);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

bool prefill_tc_supported(const KDims& d) { return d.dk == D && d.dv == D; }

size_t prefill_tc_ws_bytes(const KDims& d, int num_seqs, int total) {
  return (size_t)(total / CH + num_seqs) * d.Hv * REC_BYTES;
}

int launch_prefill_tc(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                      const int32_t* cu, const int32_t* slot_idx, const uint8_t* has_init,
                      int num_seqs, int total, const void* qkv, const void* z, const void* a,
                      const void* b, void* out, void* ws, cudaStream_t stream) {
  if (w->act == GDN_BF16)
    return launch_t<__nv_bfloat16>(d, w, pool, cu, slot_idx, has_init, num_seqs, total, qkv, z, a,
                                   b, out, ws, stream);
  return launch_t<float>(d, w, pool, cu, slot_idx, has_init, num_seqs, total, qkv, z, a, b, out,
                         ws, stream);
}

}  // namespace gdn
