// gdn_decode_multi.cu -- multi-token decode: T = 1..GDN_MAX_DECODE_TOKENS consecutive tokens per
// row (speculative-verify or multi-token append), each recurrent state read and written once.
//
// Per token the arithmetic is exactly the single-token decode step's: the causal conv + SiLU of
// the fused [q | k | v] channels ("helexa/cortex commit 95dc874 (tp_qwen3_5)",
// TpQwen3_5GatedDeltaNet bullet), l2norm of q and k, the gates g = -exp(A_log) softplus(a +
// dt_bias) and beta = sigmoid(b), the delta-rule update of the dk x dv state and the z-gated
// RMSNorm of the output ("pegainfer PR #1003", description bullets).  The T tokens of a row are
// applied in order to the state while it sits in registers, so a step of T tokens costs one
// state read and one state write instead of T of each -- the HBM cost that bounds decode.
// At T <= 8 this token-by-token form does less work than the chunkwise (UT) form with C = T,
// which would add a T x T triangular solve, and reads the state the same single time.
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

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kMT, 2)
decode_multi_kernel(KDims d, int TT, const float* __restrict__ A_log,
                    const float* __restrict__ dt_bias, const T* __restrict__ conv_w,
                    const T* __restrict__ norm_w, float* __restrict__ rec,
                    T* __restrict__ conv_state, int num_slots, int32_t* __restrict__ status,
                    const int32_t* __restrict__ slot_idx, const T* __restrict__ qkv,
                    const T* __restrict__ z, const T* __restrict__ a, const T* __restrict__ b,
                    T* __restrict__ out) {
  constexpr int NW = kMW;
  constexpr int CPT = DV / 32;   // state columns per lane
  constexpr int RPW = DK / NW;   // state rows per warp
  extern __shared__ float smem[];
  const int kh = blockIdx.x, row = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = d.r;
  const int nch = 2 * DK + r * DV;   // channels of this unit: q | k | v of its V-heads
  float* xs = smem;                  // [TT][nch] conv + SiLU outputs
  float* red = xs + TT * nch;        // [2 buffers][kv|sq][NW][DV]
  float* misc = red + 4 * NW * DV;   // [TT][iq, ik, k.q]

  const size_t zld = (size_t)d.Hv * DV;
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
  // ends up holding the last K-1 = 3 raw inputs of [old state, x_0 .. x_{TT-1}]
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
    T xin[GDN_MAX_DECODE_TOKENS];
#pragma unroll
    for (int t = 0; t < GDN_MAX_DECODE_TOKENS; ++t)
      if (t < TT) xin[t] = xr[(size_t)t * d.cqkv + ch];
#pragma unroll
    for (int t = 0; t < GDN_MAX_DECODE_TOKENS; ++t) {
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
  __syncthreads();

  // ---- per token: l2norm scales of q (times q_scale) and k, and k.q of the normalised vectors
  for (int t = warp; t < TT; t += NW) {
    const float* qs = xs + t * nch;
    const float* ks = qs + DK;
    float sq = 0.f, sk = 0.f, sqk = 0.f;
    for (int i = lane; i < DK; i += 32) {
      const float q = qs[i], k = ks[i];
      sq = fmaf(q, q, sq);
      sk = fmaf(k, k, sk);
      sqk = fmaf(q, k, sqk);
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    sqk = warp_sum(sqk);
    if (lane == 0) {
      const float iq = d.q_scale / sqrtf(sq + d.l2_eps);
      const float ik = 1.0f / sqrtf(sk + d.l2_eps);
      misc[3 * t] = iq;
      misc[3 * t + 1] = ik;
      misc[3 * t + 2] = sqk * iq * ik;
    }
  }
  __syncthreads();

  // ---- the r V-heads of this K-head, each state read once, stepped through the TT tokens in
  // registers, written once
  int it = 0;   // (V-head, token) iteration: selects the reduction buffer and the output warp
  for (int hh = 0; hh < r; ++hh) {
    const int h = kh * r + hh;
    float* Sp = rec + (((size_t)s * d.Hv + h) * DK) * DV;
    float st[RPW][CPT];
#pragma unroll
    for (int i = 0; i < RPW; ++i) StVec<CPT>::ld(Sp + (size_t)(warp * RPW + i) * DV + lane * CPT, st[i]);
    const float Al = __ldg(A_log + h), db = __ldg(dt_bias + h);
    for (int t = 0; t < TT; ++t, ++it) {
      const float* qs = xs + t * nch;
      const float* ks = qs + DK;
      const float* vs = ks + DK + hh * DV;
      const float iq = misc[3 * t], ik = misc[3 * t + 1], kq = misc[3 * t + 2];
      float g, beta;
      gates(Al, db, Act<T>::ldg(a + ((size_t)row * TT + t) * d.Hv + h),
            Act<T>::ldg(b + ((size_t)row * TT + t) * d.Hv + h), g, beta);
      const float eg = expf(g);
      float kr[RPW];
      float pk[CPT], pq[CPT];
#pragma unroll
      for (int c = 0; c < CPT; ++c) pk[c] = pq[c] = 0.f;
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        kr[i] = ks[warp * RPW + i] * ik;
        const float qv = qs[warp * RPW + i] * iq;
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          pk[c] = fmaf(st[i][c], kr[i], pk[c]);
          pq[c] = fmaf(st[i][c], qv, pq[c]);
        }
      }
      float* rb = red + (it & 1) * 2 * NW * DV;
#pragma unroll
      for (int c = 0; c < CPT; ++c) {
        rb[warp * DV + lane * CPT + c] = pk[c];
        rb[NW * DV + warp * DV + lane * CPT + c] = pq[c];
      }
      __syncthreads();
      float delta[CPT], o[CPT];
#pragma unroll
      for (int c = 0; c < CPT; ++c) {
        float kv = 0.f, sqv = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          kv += rb[w * DV + lane * CPT + c];
          sqv += rb[NW * DV + w * DV + lane * CPT + c];
        }
        delta[c] = beta * (vs[lane * CPT + c] - eg * kv);
        o[c] = fmaf(eg, sqv, kq * delta[c]);
      }
#pragma unroll
      for (int i = 0; i < RPW; ++i)
#pragma unroll
        for (int c = 0; c < CPT; ++c) st[i][c] = fmaf(eg, st[i][c], kr[i] * delta[c]);
      // z-gated RMSNorm of this (V-head, token) output, by one warp
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
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) StVec<CPT>::st(Sp + (size_t)(warp * RPW + i) * DV + lane * CPT, st[i]);
  }
}

template <int DK, int DV, typename T>
int launch_multi_t(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                   const int32_t* slot_idx, int B, int TT, const void* qkv, const void* z,
                   const void* a, const void* b, void* out, cudaStream_t stream) {
  const int nch = 2 * DK + d.r * DV;
  const size_t smem = sizeof(float) * ((size_t)TT * nch + 4 * kMW * DV + 3 * TT);
  auto kern = decode_multi_kernel<DK, DV, T>;
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
  kern<<<dim3(d.Hk, B), kMT, smem, stream>>>(
      d, TT, w->A_log, w->dt_bias, static_cast<const T*>(w->conv_weight),
      static_cast<const T*>(w->norm_weight), pool->rec_state, static_cast<T*>(pool->conv_state),
      pool->num_slots, pool->status, slot_idx, static_cast<const T*>(qkv),
      static_cast<const T*>(z), static_cast<const T*>(a), static_cast<const T*>(b),
      static_cast<T*>(out));
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename T>
int launch_multi_dims(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                      const int32_t* slot_idx, int B, int TT, const void* qkv, const void* z,
                      const void* a, const void* b, void* out, cudaStream_t stream) {
  if (d.dk == 128 && d.dv == 128)
    return launch_multi_t<128, 128, T>(d, w, pool, slot_idx, B, TT, qkv, z, a, b, out, stream);
  if (d.dk == 64 && d.dv == 64)
    return launch_multi_t<64, 64, T>(d, w, pool, slot_idx, B, TT, qkv, z, a, b, out, stream);
  if (d.dk == 128 && d.dv == 64)
    return launch_multi_t<128, 64, T>(d, w, pool, slot_idx, B, TT, qkv, z, a, b, out, stream);
  if (d.dk == 64 && d.dv == 128)
    return launch_multi_t<64, 128, T>(d, w, pool, slot_idx, B, TT, qkv, z, a, b, out, stream);
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
