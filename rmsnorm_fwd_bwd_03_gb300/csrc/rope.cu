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
// of a head row, so each element is read and written exactly once (in place is
// allowed).  A block covers all heads of one token at a time; each thread
// reads the token's position and its slice of the cos/sin row (float32, from a
// table built once in double precision, served from L1 / L2) once and applies
// it to every head it owns.  No integer division in the token loop.

#include "common.cuh"

namespace gbln {

namespace {

// Block of HP * NVH threads, NVH = D/2/VEC vectors per half head row: thread
// (hl, v) owns vector v (elements v*VEC.. and D/2 + v*VEC..) of heads hl,
// hl + HP, ... of every token the block visits; tokens are strided by gridDim.
// The cos/sin vector of a token is loaded once per thread and reused for all
// its heads; up to HPT heads' loads are issued before any of them is used.
template <typename T, int VEC, bool BWD, int HPT>
__global__ void __launch_bounds__(512)
rope_kernel(const T* q, const T* k, T* qo, T* ko, const int32_t* __restrict__ pos,
            const float2* __restrict__ cs, int64_t max_pos, int64_t T_, int Hq, int Hk,
            int D, int HP) {
  const int half = D / 2;
  const int nvh = half / VEC;
  const int v = threadIdx.x % nvh;
  const int hl = threadIdx.x / nvh;
  const int HT = Hq + Hk;
  const int i0 = v * VEC;
  for (int64_t t = blockIdx.x; t < T_; t += gridDim.x) {
    const int p = __ldg(pos + t);
    const bool ok = p >= 0 && (int64_t)p < max_pos;
    float cv[VEC], sv[VEC];
    if (ok) {
      const float2* c = cs + (size_t)p * half + i0;
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
    } else {  // out-of-range position: never read the table, emit NaN
#pragma unroll
      for (int e = 0; e < VEC; ++e) { cv[e] = __int_as_float(0x7fc00000); sv[e] = cv[e]; }
    }
    for (int h0 = hl; h0 < HT; h0 += HP * HPT) {
      float a[HPT][VEC], b[HPT][VEC];
#pragma unroll
      for (int j = 0; j < HPT; ++j) {
        const int h = h0 + j * HP;
        if (h < HT) {
          const T* src = h < Hq ? q + ((size_t)t * Hq + h) * D : k + ((size_t)t * Hk + (h - Hq)) * D;
          load_n<T, VEC>(src + i0, a[j]);
          load_n<T, VEC>(src + half + i0, b[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < HPT; ++j) {
        const int h = h0 + j * HP;
        if (h < HT) {
          T* dst = h < Hq ? qo + ((size_t)t * Hq + h) * D : ko + ((size_t)t * Hk + (h - Hq)) * D;
          float o1[VEC], o2[VEC];
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            if constexpr (!BWD) {
              o1[e] = a[j][e] * cv[e] - b[j][e] * sv[e];
              o2[e] = b[j][e] * cv[e] + a[j][e] * sv[e];
            } else {
              o1[e] = a[j][e] * cv[e] + b[j][e] * sv[e];
              o2[e] = b[j][e] * cv[e] - a[j][e] * sv[e];
            }
          }
          store_n<T, VEC>(dst + i0, o1);
          store_n<T, VEC>(dst + half + i0, o2);
        }
      }
    }
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

template <typename T, int VEC, bool BWD>
void rope_launch(int hpt, unsigned grid, int block, int HP, cudaStream_t s, const void* q,
                 const void* k, void* qo, void* ko, const int32_t* pos, const float* cs,
                 int64_t max_pos, int64_t rows, int Hq, int Hk, int D) {
#define GBLN_ROPE(N)                                                                      \
  rope_kernel<T, VEC, BWD, N><<<grid, block, 0, s>>>((const T*)q, (const T*)k, (T*)qo,     \
                                                     (T*)ko, pos, (const float2*)cs,       \
                                                     max_pos, rows, Hq, Hk, D, HP)
  switch (hpt) {
    case 1: GBLN_ROPE(1); break;
    case 2: GBLN_ROPE(2); break;
    default: GBLN_ROPE(4); break;
  }
#undef GBLN_ROPE
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
  const int nvh = vec ? half / VEC : half;
  if (nvh > 512) return GBLN_ERR_UNSUPPORTED;  // head size above 1024 (bf16 vector path: 8192)
  const int HT = Hq + Hk;
  // Heads per thread: the smallest of 1, 2, 4 that fits the block in 512 threads
  // (4 with a loop over further heads beyond that).
  int hpt = 1;
  while (hpt < 4 && (int64_t)nvh * ((HT + hpt - 1) / hpt) > 512) hpt *= 2;
  int HP = (HT + hpt - 1) / hpt;
  if ((int64_t)nvh * HP > 512) HP = 512 / nvh;
  const int block = nvh * HP;
  const int per_sm = block > 0 ? 2048 / block : 1;
  const unsigned grid = grid_for(rows, 1, (int64_t)sms * (per_sm > 0 ? per_sm : 1));
  if (vec)
    rope_launch<T, VEC, BWD>(hpt, grid, block, HP, s, q, k, qo, ko, pos, cs, max_pos, rows, Hq, Hk, D);
  else
    rope_launch<T, 1, BWD>(hpt, grid, block, HP, s, q, k, qo, ko, pos, cs, max_pos, rows, Hq, Hk, D);
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
  if (T == 0) return GBLN_OK;  // nothing is read or written: pointers are not examined
  if (!pos || !cs) return GBLN_ERR_INVALID_ARG;
  if (Hq > 0 && (!q || !qo)) return GBLN_ERR_INVALID_ARG;
  if (Hk > 0 && (!k || !ko)) return GBLN_ERR_INVALID_ARG;
  if (((uintptr_t)cs & 7u) != 0) return GBLN_ERR_INVALID_ARG;  // float2 table
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
