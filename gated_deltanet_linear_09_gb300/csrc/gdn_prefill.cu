// gdn_prefill.cu -- chunkwise (WY / UT transform) prefill of the Gated DeltaNet layer (sm_103a).
//
// The chunked prefill chain with its chunkwise scratch ("pegainfer PR #1003", description
// bullets: local head counts into the GDR decode/conv/chunkwise prefill chains; the
// GdrChunkwiseScratch35 scratch sized from the rank-local geometry).  The chunk algebra is the
// UT-transform form of the delta rule (Yang et al., "Parallelizing Linear Transformers with the
// Delta Rule over Sequence Length", NeurIPS 2024, section 3) with the gates of the gated delta
// rule.  Per sequence, per V-head, per chunk of L <= 64 tokens starting from state S0:
//   gamma_i = sum_{j<=i} g_j;   A_ij = beta_i e^{gamma_i - gamma_j} k_i.k_j  (j < i)
//   T = (I + A)^{-1};  W = T diag(beta e^gamma) K;  U~ = T diag(beta) V;  U = U~ - W S0
//   O = diag(e^gamma) Q S0 + ((Q K^T) o Gamma o M_incl) U
//   S_L = e^{gamma_L} S0 + (diag(e^{gamma_L - gamma}) K)^T U
// Every exponent is <= 0, so nothing overflows even when gamma falls to -1e3 inside a chunk.
//
// Four launches on the caller's stream:
//   prologue  (one CTA per token)        conv + SiLU, l2norm of q/k, gates  -> workspace
//   intra     (chunk x V-head)           gamma, A, T, W, U~                  -> workspace
//   state     (sequence x V-head x dv/32) the serial chunk-to-chunk state pass, U, chunk states
//   output    (chunk x V-head)           O, z-gated RMSNorm                  -> out
#include "gdn_internal.h"

namespace gdn {

namespace {

constexpr int CH = 64;          // chunk size
constexpr int NT = 256;         // threads per CTA
constexpr int BV = 32;          // dv columns per CTA of the state pass

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

// Warp-wide: checks cu_seqlens (cu[0] = 0, non-decreasing, cu[n] = total) and, for global chunk
// index c, finds its sequence, first token and length.  Returns false when cu is invalid.
__device__ bool warp_find_chunk(const int32_t* __restrict__ cu, int num_seqs, int total, int c,
                                int& seq, int& t0, int& len, int& ci) {
  const int lane = lane_id();
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
      const int lo_s = __shfl_sync(0xffffffffu, lo, src);
      const int hi_s = __shfl_sync(0xffffffffu, hi, src);
      const int ex = __shfl_sync(0xffffffffu, base + incl - nch, src);
      ci = c - ex;
      t0 = lo_s + ci * CH;
      len = min(CH, hi_s - t0);
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  return __all_sync(0xffffffffu, ok);
}

// Warp-wide: validity of cu and the number of chunks before sequence `seq`.
__device__ bool warp_seq_chunk_offset(const int32_t* __restrict__ cu, int num_seqs, int total,
                                      int seq, int& off) {
  const int lane = lane_id();
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

// ------------------------------------------------------------------ prologue

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(NT)
prologue_kernel(KDims d, const float* __restrict__ A_log, const float* __restrict__ dt_bias,
                const T* __restrict__ conv_w, const T* __restrict__ conv_state, int num_slots,
                const int32_t* __restrict__ cu, const int32_t* __restrict__ slot_idx,
                const uint8_t* __restrict__ has_init, int num_seqs, int total,
                const T* __restrict__ qkv, const T* __restrict__ a, const T* __restrict__ b,
                PrefillWs ws, int32_t* __restrict__ status) {
  extern __shared__ float ybuf[];   // [2*Hk*DK] conv outputs of the q and k regions
  __shared__ int sh_seq, sh_ok;
  const int t = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    int dummy = 0;
    const bool ok = warp_seq_chunk_offset(cu, num_seqs, total, 0, dummy);
    if (lane == 0) {
      sh_ok = ok;
      int lo = 0, hi = num_seqs - 1;   // last n with cu[n] <= t
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
      }
      sh_seq = lo;
      if (!ok && t == 0) set_status(status, GDN_STATUS_BAD_SEQLENS);
    }
  }
  __syncthreads();
  if (!sh_ok) return;
  const int n = sh_seq;
  const int s = __ldg(slot_idx + n);
  const bool valid = s >= 0 && s < num_slots;
  const bool init = valid && has_init != nullptr && __ldg(has_init + n) != 0;
  const int pos = t - __ldg(cu + n);
  const int qk_ch = 2 * d.Hk * DK;
  const T* cs = conv_state + (size_t)(valid ? s : 0) * 3 * d.cqkv;
  for (int c = tid; c < d.cqkv; c += NT) {
    float x[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int rel = pos - 3 + m;
      if (rel >= 0) x[m] = Act<T>::ldg(qkv + (size_t)(t - 3 + m) * d.cqkv + c);
      else x[m] = init ? Act<T>::ldg(cs + (size_t)(3 + rel) * d.cqkv + c) : 0.f;
    }
    const T* wc = conv_w + (size_t)c * 4;
    float acc = Act<T>::ldg(wc + 3) * x[3];
    acc = fmaf(Act<T>::ldg(wc + 0), x[0], acc);
    acc = fmaf(Act<T>::ldg(wc + 1), x[1], acc);
    acc = fmaf(Act<T>::ldg(wc + 2), x[2], acc);
    const float y = siluf_(acc);
    if (c < qk_ch) ybuf[c] = y;
    else ws.vu[(size_t)t * d.Hv * DV + (c - qk_ch)] = y;
  }
  __syncthreads();
  for (int hk = warp; hk < d.Hk; hk += NT / 32) {
    const float* yq = ybuf + hk * DK;
    const float* yk = ybuf + (d.Hk + hk) * DK;
    float sq = 0.f, sk = 0.f;
    for (int i = lane; i < DK; i += 32) {
      sq = fmaf(yq[i], yq[i], sq);
      sk = fmaf(yk[i], yk[i], sk);
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    const float iq = d.q_scale / sqrtf(sq + d.l2_eps), ik = 1.0f / sqrtf(sk + d.l2_eps);
    float* dst = ws.qk + ((size_t)t * d.Hk + hk) * 2 * DK;
    for (int i = lane; i < DK; i += 32) {
      dst[i] = yq[i] * iq;
      dst[DK + i] = yk[i] * ik;
    }
  }
  for (int h = tid; h < d.Hv; h += NT) {
    float g, beta;
    gates(__ldg(A_log + h), __ldg(dt_bias + h), Act<T>::ldg(a + (size_t)t * d.Hv + h),
          Act<T>::ldg(b + (size_t)t * d.Hv + h), g, beta);
    ws.gb[((size_t)t * d.Hv + h) * 2 + 0] = g;
    ws.gb[((size_t)t * d.Hv + h) * 2 + 1] = beta;
  }
}

// ------------------------------------------------------------------ intra-chunk

template <int DK, int DV>
__global__ void __launch_bounds__(NT)
intra_kernel(KDims d, const int32_t* __restrict__ cu, int num_seqs, int total, PrefillWs ws) {
  extern __shared__ float sm[];
  float* Ks = sm;                          // [CH][DK+1]
  float* Vs = Ks + CH * (DK + 1);          // [CH][DV]
  float* Am = Vs + CH * DV;                // [CH][CH+1]
  float* Tm = Am + CH * (CH + 1);          // [CH][CH+1]
  float* gam = Tm + CH * (CH + 1);         // [CH]
  float* bet = gam + CH;                   // [CH]
  float* ck = bet + CH;                    // [CH] beta e^gamma
  __shared__ int sh[4];
  const int c = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    int seq, t0 = 0, len = 0, ci = 0;
    const bool ok = warp_find_chunk(cu, num_seqs, total, c, seq, t0, len, ci);
    if (lane == 0) {
      sh[0] = ok && seq >= 0;
      sh[1] = t0;
      sh[2] = len;
    }
  }
  __syncthreads();
  if (!sh[0]) return;
  const int t0 = sh[1], L = sh[2];
  const int kh = h / d.r;
  for (int idx = tid; idx < CH * DK; idx += NT) {
    const int j = idx / DK, e = idx - j * DK;
    Ks[j * (DK + 1) + e] = j < L ? ws.qk[(((size_t)(t0 + j) * d.Hk + kh) * 2 + 1) * DK + e] : 0.f;
  }
  for (int idx = tid; idx < CH * DV; idx += NT) {
    const int j = idx / DV, e = idx - j * DV;
    Vs[idx] = j < L ? ws.vu[((size_t)(t0 + j) * d.Hv + h) * DV + e] : 0.f;
  }
  if (warp == 0) {
    // inclusive cumulative sum of g over the chunk (two tokens per lane)
    float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
    const int j0 = 2 * lane, j1 = 2 * lane + 1;
    if (j0 < L) { g0 = ws.gb[((size_t)(t0 + j0) * d.Hv + h) * 2]; b0 = ws.gb[((size_t)(t0 + j0) * d.Hv + h) * 2 + 1]; }
    if (j1 < L) { g1 = ws.gb[((size_t)(t0 + j1) * d.Hv + h) * 2]; b1 = ws.gb[((size_t)(t0 + j1) * d.Hv + h) * 2 + 1]; }
    float pair = g0 + g1, incl = pair;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const float ex = incl - pair;
    const float c0 = ex + g0, c1 = ex + g0 + g1;
    gam[j0] = c0; gam[j1] = c1;
    bet[j0] = b0; bet[j1] = b1;
    ck[j0] = b0 * expf(c0); ck[j1] = b1 * expf(c1);
    if (j0 < L) ws.gb[((size_t)(t0 + j0) * d.Hv + h) * 2] = c0;
    if (j1 < L) ws.gb[((size_t)(t0 + j1) * d.Hv + h) * 2] = c1;
  }
  __syncthreads();
  // A (strictly lower): A_ij = beta_i e^{gamma_i - gamma_j} k_i . k_j
  for (int idx = tid; idx < CH * CH; idx += NT) {
    const int i = idx >> 6, j = idx & 63;
    float v = 0.f;
    if (j < i && i < L) {
      const float* ki = Ks + i * (DK + 1);
      const float* kj = Ks + j * (DK + 1);
      float dot = 0.f;
#pragma unroll 8
      for (int e = 0; e < DK; ++e) dot = fmaf(ki[e], kj[e], dot);
      v = bet[i] * expf(gam[i] - gam[j]) * dot;
    }
    Am[i * (CH + 1) + j] = v;
  }
  __syncthreads();
  // T = (I + A)^{-1}, row by row: T_i = e_i - sum_{j<i} A_ij T_j
  for (int i = 0; i < CH; ++i) {
    if (tid < CH) {
      const int col = tid;
      float v = (i == col) ? 1.f : 0.f;
      for (int j = col; j < i; ++j) v = fmaf(-Am[i * (CH + 1) + j], Tm[j * (CH + 1) + col], v);
      Tm[i * (CH + 1) + col] = (col <= i) ? v : 0.f;
    }
    __syncthreads();
  }
  // W = T diag(beta e^gamma) K ;  U~ = T diag(beta) V
  {
    constexpr int RG = NT / DK;            // row groups
    constexpr int RPT = CH / RG;           // rows per thread
    const int e = tid % DK, rg = tid / DK;
    float acc[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m) acc[m] = 0.f;
    for (int j = 0; j < CH; ++j) {
      const float kj = ck[j] * Ks[j * (DK + 1) + e];
#pragma unroll
      for (int m = 0; m < RPT; ++m) acc[m] = fmaf(Tm[(rg + RG * m) * (CH + 1) + j], kj, acc[m]);
    }
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
      const int i = rg + RG * m;
      if (i < L) ws.w[((size_t)(t0 + i) * d.Hv + h) * DK + e] = acc[m];
    }
  }
  {
    constexpr int RG = NT / DV;
    constexpr int RPT = CH / RG;
    const int e = tid % DV, rg = tid / DV;
    float acc[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m) acc[m] = 0.f;
    for (int j = 0; j < CH; ++j) {
      const float vj = bet[j] * Vs[j * DV + e];
#pragma unroll
      for (int m = 0; m < RPT; ++m) acc[m] = fmaf(Tm[(rg + RG * m) * (CH + 1) + j], vj, acc[m]);
    }
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
      const int i = rg + RG * m;
      if (i < L) ws.vu[((size_t)(t0 + i) * d.Hv + h) * DV + e] = acc[m];
    }
  }
}

// ------------------------------------------------------------------ serial state pass

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(NT)
state_kernel(KDims d, float* __restrict__ rec, T* __restrict__ conv_state, int num_slots,
             const int32_t* __restrict__ cu, const int32_t* __restrict__ slot_idx,
             const uint8_t* __restrict__ has_init, int num_seqs, int total,
             const T* __restrict__ qkv, PrefillWs ws, int32_t* __restrict__ status) {
  extern __shared__ float sm[];
  float* Ss = sm;                    // [DK][BV]
  float* Ws = Ss + DK * BV;          // [CH][DK+1]
  float* Ks = Ws + CH * (DK + 1);    // [CH][DK+1]
  float* Us = Ks + CH * (DK + 1);    // [CH][BV]
  float* dec = Us + CH * BV;         // [CH] e^{gamma_L - gamma_j}
  __shared__ int sh[2];
  const int n = blockIdx.x, h = blockIdx.y, col0 = blockIdx.z * BV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    int off = 0;
    const bool ok = warp_seq_chunk_offset(cu, num_seqs, total, n, off);
    if (lane == 0) { sh[0] = ok; sh[1] = off; }
  }
  __syncthreads();
  if (!sh[0]) return;
  const int choff = sh[1];
  const int t0 = __ldg(cu + n), len = __ldg(cu + n + 1) - t0;
  const int s = __ldg(slot_idx + n);
  const bool valid = s >= 0 && s < num_slots;
  if (!valid && s >= num_slots && h == 0 && blockIdx.z == 0 && tid == 0)
    set_status(status, GDN_STATUS_SLOT_RANGE);
  const bool init = valid && has_init != nullptr && __ldg(has_init + n) != 0;
  const int kh = h / d.r;
  float* Sg = rec + ((size_t)(valid ? s : 0) * d.Hv + h) * DK * DV;
  for (int idx = tid; idx < DK * BV; idx += NT) {
    const int f = idx / BV, cc = idx - f * BV;
    Ss[idx] = init ? Sg[(size_t)f * DV + col0 + cc] : 0.f;
  }
  const int nch = (len + CH - 1) / CH;
  const int cc = tid % BV, rg = tid / BV;   // 8 row groups
  for (int ci = 0; ci < nch; ++ci) {
    const int cg = choff + ci, tc = t0 + ci * CH, L = min(CH, len - ci * CH);
    __syncthreads();
    // chunk-start state for the output pass
    float* scg = ws.sc + ((size_t)cg * d.Hv + h) * DK * DV;
    for (int idx = tid; idx < DK * BV; idx += NT) {
      const int f = idx / BV, c2 = idx - f * BV;
      scg[(size_t)f * DV + col0 + c2] = Ss[idx];
    }
    for (int idx = tid; idx < CH * DK; idx += NT) {
      const int j = idx / DK, e = idx - j * DK;
      Ws[j * (DK + 1) + e] = j < L ? ws.w[((size_t)(tc + j) * d.Hv + h) * DK + e] : 0.f;
      Ks[j * (DK + 1) + e] = j < L ? ws.qk[(((size_t)(tc + j) * d.Hk + kh) * 2 + 1) * DK + e] : 0.f;
    }
    for (int idx = tid; idx < CH * BV; idx += NT) {
      const int j = idx / BV, c2 = idx - j * BV;
      Us[idx] = j < L ? ws.vu[((size_t)(tc + j) * d.Hv + h) * DV + col0 + c2] : 0.f;
    }
    const float gl = ws.gb[((size_t)(tc + L - 1) * d.Hv + h) * 2];
    if (tid < CH) dec[tid] = tid < L ? expf(gl - ws.gb[((size_t)(tc + tid) * d.Hv + h) * 2]) : 0.f;
    __syncthreads();
    // U = U~ - W S   (rows rg + 8m)
    {
      float acc[CH / 8];
#pragma unroll
      for (int m = 0; m < CH / 8; ++m) acc[m] = 0.f;
      for (int f = 0; f < DK; ++f) {
        const float sv = Ss[f * BV + cc];
#pragma unroll
        for (int m = 0; m < CH / 8; ++m) acc[m] = fmaf(Ws[(rg + 8 * m) * (DK + 1) + f], sv, acc[m]);
      }
      __syncthreads();
#pragma unroll
      for (int m = 0; m < CH / 8; ++m) {
        const int i = rg + 8 * m;
        const float u = Us[i * BV + cc] - acc[m];
        Us[i * BV + cc] = (i < L) ? u : 0.f;
        if (i < L) ws.vu[((size_t)(tc + i) * d.Hv + h) * DV + col0 + cc] = u;
      }
    }
    __syncthreads();
    // S = e^{gamma_L} S + (diag(e^{gamma_L - gamma}) K)^T U   (rows f = rg + 8m)
    {
      const float eL = expf(gl);
      float acc[DK / 8];
#pragma unroll
      for (int m = 0; m < DK / 8; ++m) acc[m] = eL * Ss[(rg + 8 * m) * BV + cc];
      for (int j = 0; j < L; ++j) {
        const float u = dec[j] * Us[j * BV + cc];
#pragma unroll
        for (int m = 0; m < DK / 8; ++m) acc[m] = fmaf(Ks[j * (DK + 1) + rg + 8 * m], u, acc[m]);
      }
      __syncthreads();
#pragma unroll
      for (int m = 0; m < DK / 8; ++m) Ss[(rg + 8 * m) * BV + cc] = acc[m];
    }
  }
  __syncthreads();
  if (valid) {
    for (int idx = tid; idx < DK * BV; idx += NT) {
      const int f = idx / BV, c2 = idx - f * BV;
      Sg[(size_t)f * DV + col0 + c2] = Ss[idx];
    }
    if (h == 0 && blockIdx.z == 0) {
      // conv state <- the last K-1 raw inputs (older ones from the slot when continuing)
      T* cs = conv_state + (size_t)s * 3 * d.cqkv;
      for (int c = tid; c < d.cqkv; c += NT) {
        T v[3];
#pragma unroll
        for (int m = 0; m < 3; ++m) {
          const int rel = len - 3 + m;
          if (rel >= 0) v[m] = qkv[(size_t)(t0 + rel) * d.cqkv + c];
          else v[m] = init ? cs[(size_t)(3 + rel) * d.cqkv + c] : Act<T>::cvt(0.f);
        }
#pragma unroll
        for (int m = 0; m < 3; ++m) cs[(size_t)m * d.cqkv + c] = v[m];
      }
    }
  }
}

// ------------------------------------------------------------------ output

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(NT)
output_kernel(KDims d, const T* __restrict__ norm_w, int num_slots, const int32_t* __restrict__ cu,
              const int32_t* __restrict__ slot_idx, int num_seqs, int total,
              const T* __restrict__ z, T* __restrict__ out, PrefillWs ws) {
  extern __shared__ float sm[];
  float* Qs = sm;                      // [CH][DK+1]
  float* Ks = Qs + CH * (DK + 1);      // [CH][DK+1]
  float* Us = Ks + CH * (DK + 1);      // [CH][DV]
  float* Sc = Us + CH * DV;            // [DK][DV], reused for O [CH][DV]
  float* Pm = Sc + DK * DV;            // [CH][CH+1]
  float* gam = Pm + CH * (CH + 1);     // [CH]
  __shared__ int sh[5];
  const int c = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    int seq, t0 = 0, len = 0, ci = 0;
    const bool ok = warp_find_chunk(cu, num_seqs, total, c, seq, t0, len, ci);
    if (lane == 0) {
      sh[0] = ok && seq >= 0;
      sh[1] = t0;
      sh[2] = len;
      sh[3] = seq;
    }
  }
  __syncthreads();
  if (!sh[0]) return;
  const int t0 = sh[1], L = sh[2], seq = sh[3];
  const int s = __ldg(slot_idx + seq);
  T* orow = out + (size_t)t0 * d.Hv * DV + (size_t)h * DV;
  if (s < 0 || s >= num_slots) {
    for (int idx = tid; idx < L * DV; idx += NT) {
      const int i = idx / DV, e = idx - i * DV;
      orow[(size_t)i * d.Hv * DV + e] = Act<T>::cvt(0.f);
    }
    return;
  }
  const int kh = h / d.r;
  for (int idx = tid; idx < CH * DK; idx += NT) {
    const int j = idx / DK, e = idx - j * DK;
    const float* src = ws.qk + (((size_t)(t0 + j) * d.Hk + kh) * 2) * DK;
    Qs[j * (DK + 1) + e] = j < L ? src[e] : 0.f;
    Ks[j * (DK + 1) + e] = j < L ? src[DK + e] : 0.f;
  }
  for (int idx = tid; idx < CH * DV; idx += NT) {
    const int j = idx / DV, e = idx - j * DV;
    Us[idx] = j < L ? ws.vu[((size_t)(t0 + j) * d.Hv + h) * DV + e] : 0.f;
  }
  const float* scg = ws.sc + ((size_t)c * d.Hv + h) * DK * DV;
  for (int idx = tid; idx < DK * DV; idx += NT) Sc[idx] = scg[idx];
  if (tid < CH) gam[tid] = tid < L ? ws.gb[((size_t)(t0 + tid) * d.Hv + h) * 2] : 0.f;
  __syncthreads();
  for (int idx = tid; idx < CH * CH; idx += NT) {
    const int i = idx >> 6, j = idx & 63;
    float v = 0.f;
    if (j <= i && i < L) {
      const float* qi = Qs + i * (DK + 1);
      const float* kj = Ks + j * (DK + 1);
      float dot = 0.f;
#pragma unroll 8
      for (int e = 0; e < DK; ++e) dot = fmaf(qi[e], kj[e], dot);
      v = dot * expf(gam[i] - gam[j]);
    }
    Pm[i * (CH + 1) + j] = v;
  }
  __syncthreads();
  constexpr int RG = NT / DV;
  constexpr int RPT = CH / RG;
  const int e = tid % DV, rg = tid / DV;
  float acc[RPT];
#pragma unroll
  for (int m = 0; m < RPT; ++m) acc[m] = 0.f;
  for (int f = 0; f < DK; ++f) {
    const float sv = Sc[f * DV + e];
#pragma unroll
    for (int m = 0; m < RPT; ++m) acc[m] = fmaf(Qs[(rg + RG * m) * (DK + 1) + f], sv, acc[m]);
  }
#pragma unroll
  for (int m = 0; m < RPT; ++m) acc[m] *= expf(gam[rg + RG * m]);
  for (int j = 0; j < CH; ++j) {
    const float u = Us[j * DV + e];
#pragma unroll
    for (int m = 0; m < RPT; ++m) acc[m] = fmaf(Pm[(rg + RG * m) * (CH + 1) + j], u, acc[m]);
  }
  __syncthreads();
  float* Os = Sc;
#pragma unroll
  for (int m = 0; m < RPT; ++m) Os[(rg + RG * m) * DV + e] = acc[m];
  __syncthreads();
  // z-gated RMSNorm per token (one warp per row)
  for (int i = warp; i < L; i += NT / 32) {
    float ss = 0.f;
    for (int e2 = lane; e2 < DV; e2 += 32) ss = fmaf(Os[i * DV + e2], Os[i * DV + e2], ss);
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss / (float)DV + d.norm_eps);
    const T* zr = z + (size_t)(t0 + i) * d.Hv * DV + (size_t)h * DV;
    for (int e2 = lane; e2 < DV; e2 += 32) {
      const float zz = Act<T>::ldg(zr + e2);
      Act<T>::store(orow + (size_t)i * d.Hv * DV + e2,
                    Os[i * DV + e2] * inv * Act<T>::ldg(norm_w + e2) * siluf_(zz));
    }
  }
}

template <typename K>
bool set_smem(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) ==
         cudaSuccess;
}

template <int DK, int DV, typename T>
int launch_prefill_t(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                     const int32_t* cu, const int32_t* slot_idx, const uint8_t* has_init,
                     int num_seqs, int total, const void* qkv, const void* z, const void* a,
                     const void* b, void* out, const PrefillWs& ws, cudaStream_t stream) {
  const int nc_max = total / CH + num_seqs;
  const size_t smem_pro = sizeof(float) * 2 * d.Hk * DK;
  const size_t smem_intra = sizeof(float) * (CH * (DK + 1) + CH * DV + 2 * CH * (CH + 1) + 3 * CH);
  const size_t smem_state = sizeof(float) * (DK * BV + 2 * CH * (DK + 1) + CH * BV + CH);
  const size_t smem_out =
      sizeof(float) * (2 * CH * (DK + 1) + CH * DV + DK * DV + CH * (CH + 1) + CH);
  auto k0 = prologue_kernel<DK, DV, T>;
  auto k1 = intra_kernel<DK, DV>;
  auto k2 = state_kernel<DK, DV, T>;
  auto k3 = output_kernel<DK, DV, T>;
  if (!set_smem(k0, smem_pro) || !set_smem(k1, smem_intra) || !set_smem(k2, smem_state) ||
      !set_smem(k3, smem_out))
    return GDN_ERR_TOO_LARGE;
  const T* qkv_t = static_cast<const T*>(qkv);
  if (total > 0)
  k0<<<total, NT, smem_pro, stream>>>(d, w->A_log, w->dt_bias, static_cast<const T*>(w->conv_weight),
                                      static_cast<const T*>(pool->conv_state), pool->num_slots, cu,
                                      slot_idx, has_init, num_seqs, total, qkv_t,
                                      static_cast<const T*>(a), static_cast<const T*>(b), ws,
                                      pool->status);
  k1<<<dim3(nc_max, d.Hv), NT, smem_intra, stream>>>(d, cu, num_seqs, total, ws);
  k2<<<dim3(num_seqs, d.Hv, DV / BV), NT, smem_state, stream>>>(
      d, pool->rec_state, static_cast<T*>(pool->conv_state), pool->num_slots, cu, slot_idx,
      has_init, num_seqs, total, qkv_t, ws, pool->status);
  k3<<<dim3(nc_max, d.Hv), NT, smem_out, stream>>>(d, static_cast<const T*>(w->norm_weight),
                                                   pool->num_slots, cu, slot_idx, num_seqs, total,
                                                   static_cast<const T*>(z), static_cast<T*>(out),
                                                   ws);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename T>
int launch_prefill_dims(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                        const int32_t* cu, const int32_t* slot_idx, const uint8_t* has_init,
                        int num_seqs, int total, const void* qkv, const void* z, const void* a,
                        const void* b, void* out, const PrefillWs& ws, cudaStream_t stream) {
#define GDN_PREFILL_CASE(DK_, DV_)                                                                \
  if (d.dk == DK_ && d.dv == DV_)                                                                 \
    return launch_prefill_t<DK_, DV_, T>(d, w, pool, cu, slot_idx, has_init, num_seqs, total, qkv, \
                                         z, a, b, out, ws, stream);
  GDN_PREFILL_CASE(128, 128)
  GDN_PREFILL_CASE(64, 64)
  GDN_PREFILL_CASE(128, 64)
  GDN_PREFILL_CASE(64, 128)
#undef GDN_PREFILL_CASE
  return GDN_ERR_UNSUPPORTED_SHAPE;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

PrefillWs prefill_ws_layout(const KDims& d, int num_seqs, int total, void* base) {
  const size_t T = (size_t)total, nc = (size_t)(total / CH + num_seqs);
  const size_t b_qk = align256(sizeof(float) * T * d.Hk * 2 * d.dk);
  const size_t b_vu = align256(sizeof(float) * T * d.Hv * d.dv);
  const size_t b_w = align256(sizeof(float) * T * d.Hv * d.dk);
  const size_t b_gb = align256(sizeof(float) * T * d.Hv * 2);
  const size_t b_sc = align256(sizeof(float) * nc * d.Hv * d.dk * d.dv);
  PrefillWs ws{};
  ws.bytes = b_qk + b_vu + b_w + b_gb + b_sc;
  char* p = static_cast<char*>(base);
  if (p) {
    ws.qk = reinterpret_cast<float*>(p);
    ws.vu = reinterpret_cast<float*>(p + b_qk);
    ws.w = reinterpret_cast<float*>(p + b_qk + b_vu);
    ws.gb = reinterpret_cast<float*>(p + b_qk + b_vu + b_w);
    ws.sc = reinterpret_cast<float*>(p + b_qk + b_vu + b_w + b_gb);
  }
  return ws;
}

int launch_prefill(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                   const int32_t* cu, const int32_t* slot_idx, const uint8_t* has_init,
                   int num_seqs, int total, const void* qkv, const void* z, const void* a,
                   const void* b, void* out, const PrefillWs& ws, cudaStream_t stream) {
  if (w->act == GDN_BF16)
    return launch_prefill_dims<__nv_bfloat16>(d, w, pool, cu, slot_idx, has_init, num_seqs, total,
                                              qkv, z, a, b, out, ws, stream);
  return launch_prefill_dims<float>(d, w, pool, cu, slot_idx, has_init, num_seqs, total, qkv, z, a,
                                    b, out, ws, stream);
}

}  // namespace gdn
