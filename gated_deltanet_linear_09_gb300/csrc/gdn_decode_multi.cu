// gdn_decode_multi.cu -- multi-token decode: T = 1..GDN_MAX_DECODE_TOKENS consecutive tokens per
// row (speculative-verify or multi-token append), each recurrent state read and written once.
//
// Per token it computes what the single-token decode step computes: the causal conv + SiLU of
// the fused [q | k | v] channels ("helexa/cortex commit 95dc874 (tp_qwen3_5)",
// TpQwen3_5GatedDeltaNet bullet), l2norm of q and k, the gates g = -exp(A_log) softplus(a +
// dt_bias) and beta = sigmoid(b), the delta-rule update of the dk x dv state and the z-gated
// RMSNorm of the output ("pegainfer PR #1003", description bullets).  The T tokens of a row are
// taken together in the chunkwise (UT) form of the gated delta rule with C = T (Yang et al.,
// "Parallelizing Linear Transformers with the Delta Rule over Sequence Length", NeurIPS 2024,
// section 3): one pass over the old state S0 gives S0^T k_t and S0^T q_t for all tokens, a
// T x T unit lower-triangular solve per state column gives the deltas, and the state takes one
// rank-T update -- so a call of T tokens reads and writes each state once, the HBM cost that
// bounds decode, and synchronises once per V-head instead of once per token.
//
// As in the single-token kernel, one CTA owns one (row, K-head) unit: the K-head's q and k conv
// channels, the v channels of its r = Hv/Hk V-heads and their states, which keeps the conv-state
// update race-free within one launch.
#include <mutex>

#include "gdn_internal.h"

namespace gdn {

namespace {

constexpr int kMT = 256;            // threads per CTA
constexpr int kMW = kMT / 32;       // warps

// CPT consecutive f32 state values of one lane, streamed (evict-first) in one vector access.
template <int N> struct StVec;
template <> struct StVec<4> {
  static __device__ __forceinline__ void ld(const float* p, float* v) {
    const float4 t = __ldcs(reinterpret_cast<const float4*>(p));
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  }
  static __device__ __forceinline__ void st(float* p, const float* v) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
  }
};
template <> struct StVec<2> {
  static __device__ __forceinline__ void ld(const float* p, float* v) {
    const float2 t = __ldcs(reinterpret_cast<const float2*>(p));
    v[0] = t.x; v[1] = t.y;
  }
  static __device__ __forceinline__ void st(float* p, const float* v) {
    __stcs(reinterpret_cast<float2*>(p), make_float2(v[0], v[1]));
  }
};

// CPT consecutive floats of shared memory in one access (16- or 8-byte aligned).
template <int N> struct SmVec;
template <> struct SmVec<4> {
  static __device__ __forceinline__ void ld(const float* p, float* v) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  }
  static __device__ __forceinline__ void st(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <> struct SmVec<2> {
  static __device__ __forceinline__ void ld(const float* p, float* v) {
    const float2 t = *reinterpret_cast<const float2*>(p);
    v[0] = t.x; v[1] = t.y;
  }
  static __device__ __forceinline__ void st(float* p, const float* v) {
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
  }
};

// NT > 0: the token count is the compile-time NT (tight code for that T); NT = 0: the runtime
// count tt, with the loops unrolled to GDN_MAX_DECODE_TOKENS and guarded.
template <int DK, int DV, typename T, int NT>
__global__ void __launch_bounds__(kMT, 2)
decode_multi_kernel(KDims d, int tt, const float* __restrict__ A_log,
                    const float* __restrict__ dt_bias, const T* __restrict__ conv_w,
                    const T* __restrict__ norm_w, float* __restrict__ rec,
                    T* __restrict__ conv_state, int num_slots, int32_t* __restrict__ status,
                    const int32_t* __restrict__ slot_idx, const T* __restrict__ qkv,
                    const T* __restrict__ z, const T* __restrict__ a, const T* __restrict__ b,
                    T* __restrict__ out) {
  constexpr int NW = kMW;
  constexpr int CPT = DV / 32;   // state columns per lane
  constexpr int RPW = DK / NW;   // state rows per warp
  constexpr int MT = NT > 0 ? NT : GDN_MAX_DECODE_TOKENS;
  const int TT = NT > 0 ? NT : tt;
  extern __shared__ __align__(16) float smem[];
  const int kh = blockIdx.x, row = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = d.r;
  const int nch = 2 * DK + r * DV;       // channels of this unit: q | k | v of its V-heads
  float* xs = smem;                      // [TT][nch] conv + SiLU outputs (q, k then normalised)
  float* red = xs + TT * nch;            // [NW][2 TT][DV] per-warp partial S^T k_t, S^T q_t
  float* tot = red + NW * 2 * TT * DV;   // [2 TT][DV] totals
  float* kk = tot + 2 * TT * DV;         // [TT][TT] k_t . k_s
  float* qk = kk + TT * TT;              // [TT][TT] q_t . k_s
  float* gg = qk + TT * TT;              // [r][TT] g, then the inclusive cumulative gamma_t
  float* bb = gg + r * TT;               // [r][TT] beta_t
  float* am = bb + r * TT;               // [r][TT][TT] A_ts = beta_t e^{gamma_t - gamma_s} k_t.k_s, s < t
  float* pm = am + r * TT * TT;          // [r][TT][TT] P_ts = e^{gamma_t - gamma_s} q_t.k_s, s <= t
  float* eg = pm + r * TT * TT;          // [r][TT] e^{gamma_t}
  float* el = eg + r * TT;               // [r][TT] e^{gamma_{TT-1} - gamma_s}

  const size_t zld = (size_t)d.Hv * DV;
  pdl_begin();   // nothing is read before the previous kernel of the stream has completed
  const int s = slot_idx[row];
  if (s < 0 || s >= num_slots) {
    if (s >= num_slots && tid == 0 && kh == 0) set_status(status, GDN_STATUS_SLOT_RANGE);
    for (int e = tid; e < TT * r * DV; e += kMT) {
      const int t = e / (r * DV), j = e - t * (r * DV);
      out[((size_t)row * TT + t) * zld + (size_t)kh * r * DV + j] = Act<T>::cvt(0.f);
    }
    return;
  }

  // ---- causal conv + SiLU over the row's TT tokens for each owned channel; the conv state
  // ends up holding the last K-1 = 3 raw inputs of [old state, x_0 .. x_{TT-1}].  The gates of
  // every (V-head, token) are formed meanwhile.
  T* cs = conv_state + (size_t)s * 3 * d.cqkv;
  const T* xr = qkv + (size_t)row * TT * d.cqkv;
  for (int c = tid; c < nch; c += kMT) {
    int ch;
    if (c < DK) ch = kh * DK + c;
    else if (c < 2 * DK) ch = d.Hk * DK + kh * DK + (c - DK);
    else ch = 2 * d.Hk * DK + kh * r * DV + (c - 2 * DK);
    float w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = Act<T>::ldg(conv_w + (size_t)ch * 4 + j);
    T h0 = cs[ch], h1 = cs[d.cqkv + ch], h2 = cs[2 * d.cqkv + ch];
    T xin[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t)
      if (t < TT) xin[t] = xr[(size_t)t * d.cqkv + ch];
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      if (t < TT) {
        float acc = w[3] * Act<T>::load(&xin[t]);
        acc = fmaf(w[0], Act<T>::load(&h0), acc);
        acc = fmaf(w[1], Act<T>::load(&h1), acc);
        acc = fmaf(w[2], Act<T>::load(&h2), acc);
        xs[t * nch + c] = siluf_(acc);
        h0 = h1;
        h1 = h2;
        h2 = xin[t];
      }
    }
    cs[ch] = h0;
    cs[d.cqkv + ch] = h1;
    cs[2 * d.cqkv + ch] = h2;
  }
  for (int e = tid; e < r * TT; e += kMT) {
    const int hh = e / TT, t = e - hh * TT, h = kh * r + hh;
    float g, beta;
    gates(__ldg(A_log + h), __ldg(dt_bias + h), Act<T>::ldg(a + ((size_t)row * TT + t) * d.Hv + h),
          Act<T>::ldg(b + ((size_t)row * TT + t) * d.Hv + h), g, beta);
    gg[e] = g;
    bb[e] = beta;
  }
  __syncthreads();

  // ---- l2norm of q (times q_scale) and k of every token, in place (warp t owns token t)
  for (int t = warp; t < TT; t += NW) {
    float* qs = xs + t * nch;
    float* ks = qs + DK;
    float sq = 0.f, sk = 0.f;
    for (int i = lane; i < DK; i += 32) {
      sq = fmaf(qs[i], qs[i], sq);
      sk = fmaf(ks[i], ks[i], sk);
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    const float iq = d.q_scale / sqrtf(sq + d.l2_eps);
    const float ik = 1.0f / sqrtf(sk + d.l2_eps);
    for (int i = lane; i < DK; i += 32) {
      qs[i] *= iq;
      ks[i] *= ik;
    }
  }
  // cumulative gates gamma_t per V-head
  if (tid < r) {
    float acc = 0.f;
    for (int t = 0; t < TT; ++t) {
      acc += gg[tid * TT + t];
      gg[tid * TT + t] = acc;
    }
  }
  __syncthreads();

  // ---- Gram entries k_t.k_s and q_t.k_s of the normalised vectors (one warp per pair)
  for (int p = warp; p < TT * TT; p += NW) {
    const int t = p / TT, u = p - t * TT;
    const float* qt = xs + t * nch;
    const float* kt = qt + DK;
    const float* ku = xs + u * nch + DK;
    float s1 = 0.f, s2 = 0.f;
    for (int i = lane; i < DK; i += 32) {
      s1 = fmaf(kt[i], ku[i], s1);
      s2 = fmaf(qt[i], ku[i], s2);
    }
    s1 = warp_sum(s1);
    s2 = warp_sum(s2);
    if (lane == 0) {
      kk[p] = s1;
      qk[p] = s2;
    }
  }
  __syncthreads();
  // per V-head coefficients of the chunk form (exponents <= 0: gamma is non-increasing)
  for (int e = tid; e < r * TT * TT; e += kMT) {
    const int hh = e / (TT * TT), t = (e / TT) % TT, u = e % TT;
    const float gt = gg[hh * TT + t], gu = gg[hh * TT + u];
    const float dec = u <= t ? expf(gt - gu) : 0.f;
    am[e] = u < t ? bb[hh * TT + t] * dec * kk[t * TT + u] : 0.f;
    pm[e] = dec * qk[t * TT + u];
  }
  for (int e = tid; e < r * TT; e += kMT) {
    const int hh = e / TT;
    eg[e] = expf(gg[e]);
    el[e] = expf(gg[hh * TT + TT - 1] - gg[e]);
  }
  __syncthreads();

  // ---- the r V-heads of this K-head, in the chunk (UT) form with C = TT: one pass over the old
  // state S0 gives S0^T k_t and S0^T q_t for every token; per column the TT x TT unit lower
  // triangular system (I + A) delta = beta (v - e^gamma S0^T k) is solved by substitution;
  //   o_t = e^{gamma_t} S0^T q_t + sum_{s<=t} P_ts delta_s,
  //   S   = e^{gamma_last} S0 + sum_s e^{gamma_last - gamma_s} k_s delta_s^T   (one rank-TT update)
  int it = 0;   // (V-head, token) counter: picks the warp that writes an output row
  for (int hh = 0; hh < r; ++hh) {
    const int h = kh * r + hh;
    float* Sp = rec + (((size_t)s * d.Hv + h) * DK) * DV;
    float st[RPW][CPT];
#pragma unroll
    for (int i = 0; i < RPW; ++i) StVec<CPT>::ld(Sp + (size_t)(warp * RPW + i) * DV + lane * CPT, st[i]);
    // partial products over this warp's rows
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      if (t < TT) {
        const float* qt = xs + t * nch + warp * RPW;
        const float* kt = qt + DK;
        float pk[CPT], pq[CPT];
#pragma unroll
        for (int c = 0; c < CPT; ++c) pk[c] = pq[c] = 0.f;
#pragma unroll
        for (int i4 = 0; i4 < RPW; i4 += 4) {
          const float4 k4 = *reinterpret_cast<const float4*>(kt + i4);
          const float4 q4 = *reinterpret_cast<const float4*>(qt + i4);
          const float kv[4] = {k4.x, k4.y, k4.z, k4.w}, qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
          for (int ii = 0; ii < 4; ++ii)
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
              pk[c] = fmaf(st[i4 + ii][c], kv[ii], pk[c]);
              pq[c] = fmaf(st[i4 + ii][c], qv[ii], pq[c]);
            }
        }
        SmVec<CPT>::st(red + (warp * 2 * TT + t) * DV + lane * CPT, pk);
        SmVec<CPT>::st(red + (warp * 2 * TT + TT + t) * DV + lane * CPT, pq);
      }
    }
    __syncthreads();
    // totals: warp w sums vectors w, w + NW, ... over the NW partials
    for (int v = warp; v < 2 * TT; v += NW) {
      float acc[CPT];
#pragma unroll
      for (int c = 0; c < CPT; ++c) acc[c] = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        float x[CPT];
        SmVec<CPT>::ld(red + (w * 2 * TT + v) * DV + lane * CPT, x);
#pragma unroll
        for (int c = 0; c < CPT; ++c) acc[c] += x[c];
      }
      SmVec<CPT>::st(tot + v * DV + lane * CPT, acc);
    }
    __syncthreads();
    // deltas and outputs of the lane's columns, token by token
    const float* A = am + hh * TT * TT;
    const float* P = pm + hh * TT * TT;
    float dl[MT][CPT];
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      if (t < TT) {
        const float bt = bb[hh * TT + t], et = eg[hh * TT + t];
        float vt[CPT], kst[CPT], qst[CPT], o[CPT];
        SmVec<CPT>::ld(xs + t * nch + 2 * DK + hh * DV + lane * CPT, vt);
        SmVec<CPT>::ld(tot + t * DV + lane * CPT, kst);
        SmVec<CPT>::ld(tot + (TT + t) * DV + lane * CPT, qst);
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          float x = bt * (vt[c] - et * kst[c]);
          float y = et * qst[c];
#pragma unroll
          for (int u = 0; u < MT; ++u)
            if (u < t) {
              x = fmaf(-A[t * TT + u], dl[u][c], x);
              y = fmaf(P[t * TT + u], dl[u][c], y);
            }
          dl[t][c] = x;
          o[c] = fmaf(P[t * TT + t], x, y);
        }
        // z-gated RMSNorm of (V-head hh, token t), written by one warp
        if (warp == it % NW) {
          float ss = 0.f;
#pragma unroll
          for (int c = 0; c < CPT; ++c) ss = fmaf(o[c], o[c], ss);
          ss = warp_sum(ss);
          const float inv = 1.0f / sqrtf(ss / (float)DV + d.norm_eps);
          const size_t base = ((size_t)row * TT + t) * zld + (size_t)h * DV;
#pragma unroll
          for (int c = 0; c < CPT; ++c) {
            const int j = lane * CPT + c;
            const float zz = Act<T>::ldg(z + base + j);
            Act<T>::store(out + base + j, o[c] * inv * Act<T>::ldg(norm_w + j) * siluf_(zz));
          }
        }
        ++it;
      }
    }
    // rank-TT state update and write-back
    const float gl = eg[hh * TT + TT - 1];
#pragma unroll
    for (int i = 0; i < RPW; ++i)
#pragma unroll
      for (int c = 0; c < CPT; ++c) st[i][c] *= gl;
#pragma unroll
    for (int u = 0; u < MT; ++u) {
      if (u < TT) {
        const float eu = el[hh * TT + u];
        const float* ku = xs + u * nch + DK + warp * RPW;
#pragma unroll
        for (int i4 = 0; i4 < RPW; i4 += 4) {
          const float4 k4 = *reinterpret_cast<const float4*>(ku + i4);
          const float kv[4] = {k4.x * eu, k4.y * eu, k4.z * eu, k4.w * eu};
#pragma unroll
          for (int ii = 0; ii < 4; ++ii)
#pragma unroll
            for (int c = 0; c < CPT; ++c) st[i4 + ii][c] = fmaf(kv[ii], dl[u][c], st[i4 + ii][c]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) StVec<CPT>::st(Sp + (size_t)(warp * RPW + i) * DV + lane * CPT, st[i]);
  }
}

template <int DK, int DV, typename T, int NT>
int launch_multi_t(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                   const int32_t* slot_idx, int B, int TT, const void* qkv, const void* z,
                   const void* a, const void* b, void* out, cudaStream_t stream) {
  const int nch = 2 * DK + d.r * DV;
  const size_t smem = sizeof(float) * ((size_t)TT * nch + (size_t)(kMW + 1) * 2 * TT * DV +
                                       2 * TT * TT + (size_t)d.r * (4 * TT + 2 * TT * TT));
  auto kern = decode_multi_kernel<DK, DV, T, NT>;
  // raised once per kernel to the per-block maximum, so that captured launches never change it
  static std::once_flag once;
  static int attr_rc = 0;
  std::call_once(once, [&] {
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) != cudaSuccess)
      attr_rc = GDN_ERR_CUDA;
  });
  if (attr_rc != 0) return attr_rc;
  if (smem > 227 * 1024) return GDN_ERR_TOO_LARGE;
  // a programmatic dependent launch: the CTAs may be placed while the previous kernel of the
  // stream drains, and wait for it in the kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)d.Hk, (unsigned)B);
  cfg.blockDim = dim3(kMT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, kern, d, TT, w->A_log, w->dt_bias, static_cast<const T*>(w->conv_weight),
      static_cast<const T*>(w->norm_weight), pool->rec_state, static_cast<T*>(pool->conv_state),
      pool->num_slots, pool->status, slot_idx, static_cast<const T*>(qkv),
      static_cast<const T*>(z), static_cast<const T*>(a), static_cast<const T*>(b),
      static_cast<T*>(out));
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename T>
int launch_multi_dims(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                      const int32_t* slot_idx, int B, int TT, const void* qkv, const void* z,
                      const void* a, const void* b, void* out, cudaStream_t stream) {
  if (d.dk == 128 && d.dv == 128) {
    // the main head size: one instance per token count
    switch (TT) {
#define GDN_MULTI_CASE(n) \
  case n: return launch_multi_t<128, 128, T, n>(d, w, pool, slot_idx, B, TT, qkv, z, a, b, out, stream);
      GDN_MULTI_CASE(1) GDN_MULTI_CASE(2) GDN_MULTI_CASE(3) GDN_MULTI_CASE(4)
      GDN_MULTI_CASE(5) GDN_MULTI_CASE(6) GDN_MULTI_CASE(7) GDN_MULTI_CASE(8)
#undef GDN_MULTI_CASE
      default: break;
    }
    return launch_multi_t<128, 128, T, 0>(d, w, pool, slot_idx, B, TT, qkv, z, a, b, out, stream);
  }
  if (d.dk == 64 && d.dv == 64)
    return launch_multi_t<64, 64, T, 0>(d, w, pool, slot_idx, B, TT, qkv, z, a, b, out, stream);
  if (d.dk == 128 && d.dv == 64)
    return launch_multi_t<128, 64, T, 0>(d, w, pool, slot_idx, B, TT, qkv, z, a, b, out, stream);
  if (d.dk == 64 && d.dv == 128)
    return launch_multi_t<64, 128, T, 0>(d, w, pool, slot_idx, B, TT, qkv, z, a, b, out, stream);
  return GDN_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace

int launch_decode_multi(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                        const int32_t* slot_idx, int B, int TT, const void* qkv, const void* z,
                        const void* a, const void* b, void* out, cudaStream_t stream) {
  if (w->act == GDN_BF16)
    return launch_multi_dims<__nv_bfloat16>(d, w, pool, slot_idx, B, TT, qkv, z, a, b, out, stream);
  return launch_multi_dims<float>(d, w, pool, slot_idx, B, TT, qkv, z, a, b, out, stream);
}

}  // namespace gdn
