// Rotary position embedding on Q and K (forward and backward), its cos/sin
// table, and the per-document positions of packed sequences.
//
// Operator: "Fast-LLM: 高效大语言模型训练框架", §三 框架结构 (attention with RoPE) and
// "训练配置示例" (rotary type default, theta; heads / head_groups / head_size for
// grouped-query attention; micro_batch_size in tokens with
// maximum_document_length); "LLaMA-Factory Kernels 系统" (fused RoPE).
// Pairing is rotate-half: element i turns with element i + D/2.
//
// HBM-bound design: one thread moves the two 16-byte vectors at i and i + D/2
// of one head row, so each element is read and written exactly once (in place
// is allowed).  Consecutive threads cover consecutive (token, head, vector)
// units, so all heads of a token sit in one or two neighbouring blocks and the
// token's position and cos/sin row (float32, from a table built once in double
// precision) are re-read from L1 / L2, not from HBM.

#include "common.cuh"

namespace gbln {

namespace {

constexpr int kRopeBlock = 256;

// One thread per (token, head, vector) unit, grid-stride over the flat unit
// index; `per_tok` = (Hq + Hk) * (D/2/VEC) units per token.
template <typename T, int VEC, bool BWD>
__global__ void __launch_bounds__(kRopeBlock)
rope_kernel(const T* q, const T* k, T* qo, T* ko, const int32_t* __restrict__ pos,
            const float2* __restrict__ cs, int64_t max_pos, int64_t T_, int Hq, int Hk,
            int D) {
  const int half = D / 2;
  const int nvh = half / VEC;
  const int per_tok = (Hq + Hk) * nvh;
  const int64_t total = T_ * (int64_t)per_tok;
  const int64_t stride = (int64_t)gridDim.x * kRopeBlock;
  for (int64_t u = (int64_t)blockIdx.x * kRopeBlock + threadIdx.x; u < total; u += stride) {
    const int64_t t = u / per_tok;
    const int rem = (int)(u - t * per_tok);
    const int hd = rem / nvh;
    const int i0 = (rem - hd * nvh) * VEC;
    const T* src;
    T* dst;
    if (hd < Hq) {
      const size_t off = ((size_t)t * Hq + hd) * D;
      src = q + off; dst = qo + off;
    } else {
      const size_t off = ((size_t)t * Hk + (hd - Hq)) * D;
      src = k + off; dst = ko + off;
    }
    float a[VEC], b[VEC], o1[VEC], o2[VEC];
    load_n<T, VEC>(src + i0, a);
    load_n<T, VEC>(src + half + i0, b);
    const int p = __ldg(pos + t);
    if (p < 0 || (int64_t)p >= max_pos) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) { o1[e] = __int_as_float(0x7fc00000); o2[e] = o1[e]; }
    } else {
      const float2* c = cs + (size_t)p * half + i0;
      float cv[VEC], sv[VEC];
      if constexpr (VEC % 2 == 0) {
#pragma unroll
        for (int e = 0; e < VEC; e += 2) {
          const float4 f = __ldg(reinterpret_cast<const float4*>(c + e));
          cv[e] = f.x; sv[e] = f.y; cv[e + 1] = f.z; sv[e + 1] = f.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) { const float2 f = __ldg(c + e); cv[e] = f.x; sv[e] = f.y; }
      }
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        if constexpr (!BWD) {
          o1[e] = a[e] * cv[e] - b[e] * sv[e];
          o2[e] = b[e] * cv[e] + a[e] * sv[e];
        } else {
          o1[e] = a[e] * cv[e] + b[e] * sv[e];
          o2[e] = b[e] * cv[e] - a[e] * sv[e];
        }
      }
    }
    store_n<T, VEC>(dst + i0, o1);
    store_n<T, VEC>(dst + half + i0, o2);
  }
}

__global__ void rope_table_kernel(float2* cs, int64_t max_pos, int half, int D, double theta) {
  const int64_t n = max_pos * half;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < n;
       u += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = u / half;
    const int i = (int)(u - p * half);
    const double f = pow(theta, -2.0 * (double)i / (double)D);
    const double ang = (double)p * f;
    double sn, cn;
    sincos(ang, &sn, &cn);
    cs[u] = make_float2((float)cn, (float)sn);
  }
}

// positions[t] = t - cu[d] for cu[d] <= t < cu[d+1]; binary search per token.
__global__ void positions_kernel(const int32_t* __restrict__ cu, int ndoc, int32_t* pos,
                                 int64_t T_) {
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T_;
       t += (int64_t)gridDim.x * blockDim.x) {
    int lo = 0, hi = ndoc - 1;  // largest d in [0, ndoc) with cu[d] <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
    }
    pos[t] = (int32_t)(t - (int64_t)__ldg(cu + lo));
  }
}

template <typename T, bool BWD>
gbln_status rope_typed(const void* q, const void* k, void* qo, void* ko, const int32_t* pos,
                       const float* cs, int64_t max_pos, int64_t rows, int Hq, int Hk, int D,
                       cudaStream_t s) {
  constexpr int VEC = VecOf<T>::N;
  const int half = D / 2;
  const bool vec = (half % VEC == 0) && aligned16(q) && aligned16(qo) && aligned16(cs) &&
                   (Hk == 0 || (aligned16(k) && aligned16(ko)));
  const int sms = sm_count();
  if (sms <= 0) return GBLN_ERR_CUDA;
  const int64_t cap = (int64_t)sms * (2048 / kRopeBlock) * 8;
  if (vec) {
    const int64_t units = rows * (int64_t)(Hq + Hk) * (half / VEC);
    rope_kernel<T, VEC, BWD><<<grid_for(units, kRopeBlock, cap), kRopeBlock, 0, s>>>(
        (const T*)q, (const T*)k, (T*)qo, (T*)ko, pos, (const float2*)cs, max_pos, rows, Hq, Hk, D);
  } else {
    const int64_t units = rows * (int64_t)(Hq + Hk) * half;
    rope_kernel<T, 1, BWD><<<grid_for(units, kRopeBlock, cap), kRopeBlock, 0, s>>>(
        (const T*)q, (const T*)k, (T*)qo, (T*)ko, pos, (const float2*)cs, max_pos, rows, Hq, Hk, D);
  }
  return launch_status();
}

template <bool BWD>
gbln_status rope_entry(const void* q, const void* k, void* qo, void* ko, const int32_t* pos,
                       const float* cs, int64_t max_pos, int64_t T, int32_t Hq, int32_t Hk,
                       int32_t D, gbln_dtype io, gbln_stream_t stream) {
  if (!dtype_ok(io)) return GBLN_ERR_INVALID_ARG;
  if (T < 0 || Hq < 0 || Hk < 0 || Hq + Hk <= 0 || D <= 0 || (D & 1) || max_pos < 0)
    return GBLN_ERR_INVALID_ARG;
  if ((int64_t)(Hq + Hk) * D > (1 << 24)) return GBLN_ERR_INVALID_ARG;
  if (!pos || !cs) return GBLN_ERR_INVALID_ARG;
  if (Hq > 0 && (!q || !qo)) return GBLN_ERR_INVALID_ARG;
  if (Hk > 0 && (!k || !ko)) return GBLN_ERR_INVALID_ARG;
  if (((uintptr_t)cs & 7u) != 0) return GBLN_ERR_INVALID_ARG;  // float2 table
  if (T == 0) return GBLN_OK;
  cudaStream_t s = (cudaStream_t)stream;
  if (io == GBLN_F32) return rope_typed<float, BWD>(q, k, qo, ko, pos, cs, max_pos, T, Hq, Hk, D, s);
  return rope_typed<bf16, BWD>(q, k, qo, ko, pos, cs, max_pos, T, Hq, Hk, D, s);
}

}  // namespace

}  // namespace gbln

using namespace gbln;

extern "C" gbln_status gbln_rope_table(float* cos_sin, int64_t max_pos, int32_t D, double theta,
                                       gbln_stream_t stream) {
  if (!cos_sin || max_pos < 0 || max_pos > (1LL << 31) || D <= 0 || (D & 1))
    return GBLN_ERR_INVALID_ARG;
  if (!(theta > 0.0 && theta <= 1.7976931348623157e308)) return GBLN_ERR_INVALID_ARG;
  if (max_pos == 0) return GBLN_OK;
  const int half = D / 2;
  const int64_t n = max_pos * half;
  rope_table_kernel<<<grid_for(n, 256, 4096), 256, 0, (cudaStream_t)stream>>>(
      (float2*)cos_sin, max_pos, half, D, theta);
  return launch_status();
}

extern "C" gbln_status gbln_rope_fwd(const void* q, const void* k, void* q_out, void* k_out,
                                     const int32_t* positions, const float* cos_sin,
                                     int64_t max_pos, int64_t T, int32_t Hq, int32_t Hk,
                                     int32_t D, gbln_dtype io, gbln_stream_t stream) {
  return rope_entry<false>(q, k, q_out, k_out, positions, cos_sin, max_pos, T, Hq, Hk, D, io,
                           stream);
}

extern "C" gbln_status gbln_rope_bwd(const void* dq, const void* dk, void* dq_in, void* dk_in,
                                     const int32_t* positions, const float* cos_sin,
                                     int64_t max_pos, int64_t T, int32_t Hq, int32_t Hk,
                                     int32_t D, gbln_dtype io, gbln_stream_t stream) {
  return rope_entry<true>(dq, dk, dq_in, dk_in, positions, cos_sin, max_pos, T, Hq, Hk, D, io,
                          stream);
}

extern "C" gbln_status gbln_positions_from_cu_seqlens(const int32_t* cu_seqlens, int32_t ndoc,
                                                      int32_t* positions, int64_t T,
                                                      gbln_stream_t stream) {
  if (!positions || T < 0 || T > (1LL << 31) - 1 || ndoc < 0) return GBLN_ERR_INVALID_ARG;
  if (T == 0) return GBLN_OK;
  if (!cu_seqlens || ndoc < 1) return GBLN_ERR_INVALID_ARG;  // tokens need a document
  positions_kernel<<<grid_for(T, 256, 8192), 256, 0, (cudaStream_t)stream>>>(cu_seqlens, ndoc,
                                                                               positions, T);
  return launch_status();
}
