// gdn_decode.cu -- batched Gated DeltaNet decode step and standalone conv1d update (sm_103a).
//
// The batched GDR decode over all decode rows ("pegainfer issue #1001", Split 2 bullet) with
// slot-indexed per-request recurrent and conv state ("pegainfer issue #1001", Split 3 bullet),
// rank-local head counts and the gated RMSNorm at the local V-heads ("pegainfer PR #1003",
// description bullets), fused [q | k | v] channel regions and repeat_interleave of K-heads
// ("helexa/cortex commit 95dc874 (tp_qwen3_5)", TpQwen3_5GatedDeltaNet bullet).
//
// One CTA owns one (row, K-head) unit: the conv channels of that K-head's q and k, the v
// channels of its r = Hv/Hk V-heads, and those V-heads' dk x dv f32 states.  Owning all the
// channels a K-head touches makes the conv-state update race-free without a second launch.
// The state of each V-head is read once and written once (the decode's whole HBM cost):
//   kv = S^T k,  sq = S^T q           (one pass over the old S, held in registers)
//   delta = beta (v - e^g kv),  o = e^g sq + (k.q) delta
//   S' = e^g S + k delta^T            (written back from the same registers)
// Each warp owns dv/8 whole columns of every state (all dk rows), so both products reduce
// inside the warp by shuffles and the warps run through the V-heads without a CTA barrier;
// only the RMSNorm's sum over dv meets in shared memory, once, after the last V-head.
// The kernel is a programmatic dependent launch: in a stream of decode steps the next step's
// CTAs are placed while this one drains and wait for its completion before any read.
#include <mutex>

#include "gdn_internal.h"

namespace gdn {

namespace {

template <int N> struct VecF;
template <> struct VecF<4> {
  static __device__ __forceinline__ void ld(const float* p, float* v) {
    const float4 t = __ldcs(reinterpret_cast<const float4*>(p));
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  }
  static __device__ __forceinline__ void st(float* p, const float* v) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
  }
};

constexpr int kDecodeThreads = 256;
constexpr int kDecodeWarps = kDecodeThreads / 32;

__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(
                   static_cast<unsigned>(__cvta_generic_to_shared(sdst))), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async8(void* sdst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(
                   static_cast<unsigned>(__cvta_generic_to_shared(sdst))), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }
// 4 consecutive activation elements (8 or 16 bytes) into shared memory
template <typename T>
__device__ __forceinline__ void cp_async_quad(T* sdst, const T* gsrc) {
  if constexpr (sizeof(T) == 2) cp_async8(sdst, gsrc);
  else cp_async16(sdst, gsrc);
}

// Shared-memory layout of decode_kernel: the f32 work arrays, then the prefetched z values and
// norm weight.
template <int DK, int DV>
__host__ __device__ inline int decode_float_count(int r) {
  return ((2 * DK + 2 * r * DV + r * kDecodeWarps + 3 + 2 * r) + 3) / 4 * 4;
}

// Conv-state values with an L2 evict-last policy: the step's rows read and rewrite their slots'
// conv state (a few MB) while the recurrent states stream through L2 evict-first, so the next
// step finds it in L2.
template <typename T> struct KeepL2;
template <> struct KeepL2<float> {
  static __device__ __forceinline__ float ld(const float* p, uint64_t pol) {
    float v;
    asm volatile("ld.global.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(pol));
    return v;
  }
  static __device__ __forceinline__ void st(float* p, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
  }
};
template <> struct KeepL2<__nv_bfloat16> {
  static __device__ __forceinline__ __nv_bfloat16 ld(const __nv_bfloat16* p, uint64_t pol) {
    unsigned short v;
    asm volatile("ld.global.L2::cache_hint.b16 %0, [%1], %2;" : "=h"(v) : "l"(p), "l"(pol));
    return __ushort_as_bfloat16(v);
  }
  static __device__ __forceinline__ void st(__nv_bfloat16* p, __nv_bfloat16 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.b16 [%0], %1, %2;" ::"l"(p), "h"(__bfloat16_as_ushort(v)),
                 "l"(pol)
                 : "memory");
  }
};
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// One token of the causal conv for channel ch of the row's conv state cs ([K-1][cqkv],
// K = 4): returns SiLU(sum_j w[j] x_{t-3+j}) and shifts the state by one raw input.
template <typename T>
__device__ __forceinline__ float conv_channel(const T* __restrict__ conv_w, T* __restrict__ cs,
                                              int cqkv, int ch, T xraw) {
  const T* wc = conv_w + (size_t)ch * 4;
  const T s0 = cs[ch], s1 = cs[cqkv + ch], s2 = cs[2 * cqkv + ch];
  float acc = Act<T>::ldg(wc + 3) * Act<T>::load(&xraw);
  acc = fmaf(Act<T>::ldg(wc + 0), Act<T>::load(&s0), acc);
  acc = fmaf(Act<T>::ldg(wc + 1), Act<T>::load(&s1), acc);
  acc = fmaf(Act<T>::ldg(wc + 2), Act<T>::load(&s2), acc);
  cs[ch] = s1;
  cs[cqkv + ch] = s2;
  cs[2 * cqkv + ch] = xraw;
  return siluf_(acc);
}

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kDecodeThreads, 2)
decode_kernel(KDims d, const float* __restrict__ A_log, const float* __restrict__ dt_bias,
              const T* __restrict__ conv_w, const T* __restrict__ norm_w, float* __restrict__ rec,
              T* __restrict__ conv_state, int num_slots, int32_t* __restrict__ status,
              const int32_t* __restrict__ slot_idx, const T* __restrict__ qkv,
              const T* __restrict__ z, const T* __restrict__ a, const T* __restrict__ b,
              T* __restrict__ out) {
  constexpr int NW = kDecodeWarps;
  // A warp owns CW whole state columns (all DK rows), so S^T k and S^T q reduce inside the
  // warp and the V-heads need no CTA barrier.  A lane holds a float4 of 4 columns in RPL rows.
  constexpr int CW = DV / NW;       // state columns per warp
  constexpr int LPR = CW / 4;       // lanes per row segment
  constexpr int G = 32 / LPR;       // row groups per warp
  constexpr int RPL = DK / G;       // state rows per lane
  static_assert(CW % 4 == 0 && DK % G == 0, "state tiling");
  extern __shared__ float4 smem4[];
  const int kh = blockIdx.x, row = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane / LPR, col0 = warp * CW + (lane % LPR) * 4;
  const int r = d.r;
  float* qs = reinterpret_cast<float*>(smem4);
  float* ks = qs + DK;
  float* vs = ks + DK;
  float* os = vs + r * DV;           // raw outputs o of the r V-heads
  float* ssq = os + r * DV;          // per-warp partial sums of o^2, [r][NW]
  float* misc = ssq + r * NW;        // iq, ik, k.q, then (e^g, beta) per V-head
  T* zs = reinterpret_cast<T*>(qs + decode_float_count<DK, DV>(r));   // z of the r V-heads
  T* nws = zs + r * DV;                                                // norm weight

  // A programmatic dependent of the previous kernel in the stream: nothing is read before that
  // kernel has completed and its writes are visible.  The next kernel may be placed on the SMs
  // as soon as every CTA of this one runs (it waits the same way).
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int s = slot_idx[row];
  T* out_row = out + (size_t)row * d.Hv * DV;
  if (s < 0 || s >= num_slots) {
    if (s >= num_slots && tid == 0 && kh == 0) set_status(status, GDN_STATUS_SLOT_RANGE);
    for (int e = tid; e < r * DV; e += kDecodeThreads) out_row[kh * r * DV + e] = Act<T>::cvt(0.f);
    return;
  }
  // The z values and the norm weight go to shared memory by asynchronous copies issued before
  // the conv prologue (their latency would otherwise fall at the end of the CTA).
  {
    const T* zrow = z + (size_t)row * d.Hv * DV + (size_t)kh * r * DV;
    for (int e = tid; e < r * (DV / 4); e += kDecodeThreads) cp_async_quad(zs + 4 * e, zrow + 4 * e);
    for (int e = tid; e < DV / 4; e += kDecodeThreads) cp_async_quad(nws + 4 * e, norm_w + 4 * e);
    cp_async_commit();
  }
  // gate inputs of the r V-heads (threads 32 .. 32 + r - 1), in flight during the conv prologue
  const int gh = tid - 32;
  float g_alog = 0.f, g_dt = 0.f, g_a = 0.f, g_b = 0.f;
  if (gh >= 0 && gh < r) {
    const int h = kh * r + gh;
    g_alog = __ldg(A_log + h);
    g_dt = __ldg(dt_bias + h);
    g_a = Act<T>::ldg(a + (size_t)row * d.Hv + h);
    g_b = Act<T>::ldg(b + (size_t)row * d.Hv + h);
  }

  // ---- conv update + SiLU over the channels this unit owns.  The loads of a thread's channels
  // are all issued before any of them is used (one memory round trip for the prologue).
  const T* x_row = qkv + (size_t)row * d.cqkv;
  T* cs = conv_state + (size_t)s * 3 * d.cqkv;
  const int nch = 2 * DK + r * DV;
  const uint64_t keep = l2_evict_last_policy();
  for (int c0 = 0; c0 < nch; c0 += 3 * kDecodeThreads) {
    int chs[3];
    float* dsts[3];
    T xr[3], s0[3], s1[3], s2[3];
    float wv[3][4];
#pragma unroll
    for (int m = 0; m < 3; ++m) {
      const int c = min(c0 + tid + m * kDecodeThreads, nch - 1);   // clamped: always a valid channel
      if (c < DK) {
        chs[m] = kh * DK + c;
        dsts[m] = qs + c;
      } else if (c < 2 * DK) {
        chs[m] = d.Hk * DK + kh * DK + (c - DK);
        dsts[m] = ks + (c - DK);
      } else {
        chs[m] = 2 * d.Hk * DK + kh * r * DV + (c - 2 * DK);
        dsts[m] = vs + (c - 2 * DK);
      }
      xr[m] = x_row[chs[m]];
      s0[m] = KeepL2<T>::ld(cs + chs[m], keep);
      s1[m] = KeepL2<T>::ld(cs + d.cqkv + chs[m], keep);
      s2[m] = KeepL2<T>::ld(cs + 2 * d.cqkv + chs[m], keep);
#pragma unroll
      for (int j = 0; j < 4; ++j) wv[m][j] = Act<T>::ldg(conv_w + (size_t)chs[m] * 4 + j);
    }
#pragma unroll
    for (int m = 0; m < 3; ++m) {
      if (c0 + tid + m * kDecodeThreads < nch) {
        float acc = wv[m][3] * Act<T>::load(&xr[m]);
        acc = fmaf(wv[m][0], Act<T>::load(&s0[m]), acc);
        acc = fmaf(wv[m][1], Act<T>::load(&s1[m]), acc);
        acc = fmaf(wv[m][2], Act<T>::load(&s2[m]), acc);
        KeepL2<T>::st(cs + chs[m], s1[m], keep);
        KeepL2<T>::st(cs + d.cqkv + chs[m], s2[m], keep);
        KeepL2<T>::st(cs + 2 * d.cqkv + chs[m], xr[m], keep);
        *dsts[m] = siluf_(acc);
      }
    }
  }
  if (gh >= 0 && gh < r) {
    float gg, beta;
    gates(g_alog, g_dt, g_a, g_b, gg, beta);
    misc[3 + 2 * gh] = expf(gg);
    misc[4 + 2 * gh] = beta;
  }
  __syncthreads();

  // ---- l2norm of q (times q_scale) and k, and k.q of the normalised vectors
  if (warp == 0) {
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
      misc[0] = iq;
      misc[1] = ik;
      misc[2] = sqk * iq * ik;
    }
  }
  __syncthreads();
  const float iq = misc[0], ik = misc[1], kq = misc[2];
  float kr[RPL], qr[RPL];
#pragma unroll
  for (int i = 0; i < RPL; ++i) {
    kr[i] = ks[g + G * i] * ik;
    qr[i] = qs[g + G * i] * iq;
  }

  // ---- the r V-heads of this K-head; each warp runs through them on its own columns
  for (int hh = 0; hh < r; ++hh) {
    const int h = kh * r + hh;
    float* Sp = rec + (((size_t)s * d.Hv + h) * DK) * DV + col0;
    float st[RPL][4];
#pragma unroll
    for (int i = 0; i < RPL; ++i) VecF<4>::ld(Sp + (size_t)(g + G * i) * DV, st[i]);
    const float eg = misc[3 + 2 * hh], beta = misc[4 + 2 * hh];

    float pk[4], pq[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) pk[c] = pq[c] = 0.f;
#pragma unroll
    for (int i = 0; i < RPL; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        pk[c] = fmaf(st[i][c], kr[i], pk[c]);
        pq[c] = fmaf(st[i][c], qr[i], pq[c]);
      }
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        pk[c] += __shfl_xor_sync(0xffffffffu, pk[c], off);
        pq[c] += __shfl_xor_sync(0xffffffffu, pq[c], off);
      }
    const float4 vv = *reinterpret_cast<const float4*>(vs + hh * DV + col0);
    const float vc[4] = {vv.x, vv.y, vv.z, vv.w};
    float delta[4], o[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      delta[c] = beta * (vc[c] - eg * pk[c]);
      o[c] = fmaf(eg, pq[c], kq * delta[c]);
    }
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
#pragma unroll
      for (int c = 0; c < 4; ++c) st[i][c] = fmaf(eg, st[i][c], kr[i] * delta[c]);
      VecF<4>::st(Sp + (size_t)(g + G * i) * DV, st[i]);
    }
    if (g == 0) {
      *reinterpret_cast<float4*>(os + hh * DV + col0) = make_float4(o[0], o[1], o[2], o[3]);
      float ss = o[0] * o[0] + o[1] * o[1] + o[2] * o[2] + o[3] * o[3];
#pragma unroll
      for (int off = 1; off < LPR; off <<= 1) ss += __shfl_xor_sync((1u << LPR) - 1u, ss, off);
      if (lane == 0) ssq[hh * NW + warp] = ss;
    }
  }
  cp_async_wait_all();
  __syncthreads();

  // ---- z-gated RMSNorm over each V-head's dv outputs, 4 columns per thread
  constexpr int Q4 = DV / 4;
  for (int e = tid; e < r * Q4; e += kDecodeThreads) {
    const int hh = e / Q4, j = (e - hh * Q4) * 4;
    const int h = kh * r + hh;
    const float4 zz = Act<T>::lds4(zs + hh * DV + j);
    const float4 ww = Act<T>::lds4(nws + j);
    float ss = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) ss += ssq[hh * NW + w];
    const float inv = 1.0f / sqrtf(ss / (float)DV + d.norm_eps);
    const float4 ov = *reinterpret_cast<const float4*>(os + hh * DV + j);
    Act<T>::store4(out_row + (size_t)h * DV + j,
                   make_float4(ov.x * inv * ww.x * siluf_(zz.x), ov.y * inv * ww.y * siluf_(zz.y),
                               ov.z * inv * ww.z * siluf_(zz.z), ov.w * inv * ww.w * siluf_(zz.w)));
  }
}

template <typename T>
__global__ void conv1d_update_kernel(int cqkv, const T* __restrict__ conv_w,
                                     T* __restrict__ conv_state, int num_slots,
                                     int32_t* __restrict__ status,
                                     const int32_t* __restrict__ slot_idx,
                                     const T* __restrict__ in, T* __restrict__ out) {
  const int row = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= cqkv) return;
  const int s = slot_idx[row];
  if (s < 0 || s >= num_slots) {
    if (s >= num_slots && c == 0) set_status(status, GDN_STATUS_SLOT_RANGE);
    out[(size_t)row * cqkv + c] = Act<T>::cvt(0.f);
    return;
  }
  T* cs = conv_state + (size_t)s * 3 * cqkv;
  const float y = conv_channel<T>(conv_w, cs, cqkv, c, in[(size_t)row * cqkv + c]);
  Act<T>::store(out + (size_t)row * cqkv + c, y);
}

template <int DK, int DV, typename T>
int launch_decode_t(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                    const int32_t* slot_idx, int B, const void* qkv, const void* z, const void* a,
                    const void* b, void* out, cudaStream_t stream) {
  const size_t smem = sizeof(float) * decode_float_count<DK, DV>(d.r) + sizeof(T) * (d.r + 1) * DV;
  auto kern = decode_kernel<DK, DV, T>;
  // Raised once per kernel (to the per-block maximum), so that launches -- also those recorded
  // into a CUDA graph -- never need to change the attribute.
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
  // programmatic stream serialization: the CTAs may be placed while the previous kernel of the
  // stream drains, and wait for it in the kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)d.Hk, (unsigned)B);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, kern, d, w->A_log, w->dt_bias, static_cast<const T*>(w->conv_weight),
      static_cast<const T*>(w->norm_weight), pool->rec_state, static_cast<T*>(pool->conv_state),
      pool->num_slots, pool->status, slot_idx, static_cast<const T*>(qkv),
      static_cast<const T*>(z), static_cast<const T*>(a), static_cast<const T*>(b),
      static_cast<T*>(out));
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename T>
int launch_decode_dims(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                       const int32_t* slot_idx, int B, const void* qkv, const void* z,
                       const void* a, const void* b, void* out, cudaStream_t stream) {
  if (d.dk == 128 && d.dv == 128)
    return launch_decode_t<128, 128, T>(d, w, pool, slot_idx, B, qkv, z, a, b, out, stream);
  if (d.dk == 64 && d.dv == 64)
    return launch_decode_t<64, 64, T>(d, w, pool, slot_idx, B, qkv, z, a, b, out, stream);
  if (d.dk == 128 && d.dv == 64)
    return launch_decode_t<128, 64, T>(d, w, pool, slot_idx, B, qkv, z, a, b, out, stream);
  if (d.dk == 64 && d.dv == 128)
    return launch_decode_t<64, 128, T>(d, w, pool, slot_idx, B, qkv, z, a, b, out, stream);
  return GDN_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace

int launch_decode(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                  const int32_t* slot_idx, int B, const void* qkv, const void* z, const void* a,
                  const void* b, void* out, cudaStream_t stream) {
  if (w->act == GDN_BF16)
    return launch_decode_dims<__nv_bfloat16>(d, w, pool, slot_idx, B, qkv, z, a, b, out, stream);
  return launch_decode_dims<float>(d, w, pool, slot_idx, B, qkv, z, a, b, out, stream);
}

int launch_conv1d_update(const KDims& d, const gdn_weights* w, const gdn_pool* pool,
                         const int32_t* slot_idx, int B, const void* in, void* out,
                         cudaStream_t stream) {
  dim3 grid((d.cqkv + 255) / 256, B);
  if (w->act == GDN_BF16) {
    conv1d_update_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
        d.cqkv, static_cast<const __nv_bfloat16*>(w->conv_weight),
        static_cast<__nv_bfloat16*>(pool->conv_state), pool->num_slots, pool->status, slot_idx,
        static_cast<const __nv_bfloat16*>(in), static_cast<__nv_bfloat16*>(out));
  } else {
    conv1d_update_kernel<float><<<grid, 256, 0, stream>>>(
        d.cqkv, static_cast<const float*>(w->conv_weight), static_cast<float*>(pool->conv_state),
        pool->num_slots, pool->status, slot_idx, static_cast<const float*>(in),
        static_cast<float*>(out));
  }
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn
