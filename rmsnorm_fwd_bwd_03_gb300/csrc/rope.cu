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
// allowed).  A block covers all heads of a few consecutive tokens at a time;
// each thread reads a token's position and its slice of the cos/sin row
// (float32, from a table built once in double precision, served from L1 / L2)
// once and applies it to every head it owns.  No integer division in the loop.

#include "common.cuh"

namespace gbln {

namespace {

// Rotate one vector pair: elements i0.. of the first half (a) and of the second
// half (b) of a head row, with the cos/sin entries c[0..VEC).  On the vector
// path the work goes two elements (one 32-bit word of bf16, or two floats) at
// a time so that only the packed inputs and one float4 of cos/sin are live.
template <typename T, int VEC, bool BWD>
__device__ __forceinline__ void rotate_store(const Packed<T, VEC>& a, const Packed<T, VEC>& b,
                                             const float2* c, bool ok, T* d1, T* d2) {
  const float qnan = __int_as_float(0x7fc00000);
  if constexpr (VEC * sizeof(T) == 16) {
    const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a.r);
    const uint32_t* bw = reinterpret_cast<const uint32_t*>(&b.r);
    uint32_t o1[4], o2[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float x1[2], x2[2];
      if constexpr (sizeof(T) == 2) {
        x1[0] = bf16_lo(aw[w]); x1[1] = bf16_hi(aw[w]);
        x2[0] = bf16_lo(bw[w]); x2[1] = bf16_hi(bw[w]);
      } else {
        x1[0] = __uint_as_float(aw[w]); x2[0] = __uint_as_float(bw[w]);
      }
      constexpr int PER = sizeof(T) == 2 ? 2 : 1;  // elements per 32-bit word
      float cv[2], sv[2];
      if constexpr (PER == 2) {
        const float4 f = ok ? __ldg(reinterpret_cast<const float4*>(c + 2 * w))
                            : make_float4(qnan, qnan, qnan, qnan);
        cv[0] = f.x; sv[0] = f.y; cv[1] = f.z; sv[1] = f.w;
      } else {
        const float2 f = ok ? __ldg(c + w) : make_float2(qnan, qnan);
        cv[0] = f.x; sv[0] = f.y;
      }
      float y1[2], y2[2];
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        if constexpr (!BWD) {
          y1[e] = x1[e] * cv[e] - x2[e] * sv[e];
          y2[e] = x2[e] * cv[e] + x1[e] * sv[e];
        } else {
          y1[e] = x1[e] * cv[e] + x2[e] * sv[e];
          y2[e] = x2[e] * cv[e] - x1[e] * sv[e];
        }
      }
      if constexpr (PER == 2) {
        o1[w] = pack_bf16x2(y1[0], y1[1]);
        o2[w] = pack_bf16x2(y2[0], y2[1]);
      } else {
        o1[w] = __float_as_uint(y1[0]);
        o2[w] = __float_as_uint(y2[0]);
      }
    }
    st_vec(d1, make_uint4(o1[0], o1[1], o1[2], o1[3]));
    st_vec(d2, make_uint4(o2[0], o2[1], o2[2], o2[3]));
  } else {
    float x1[VEC], x2[VEC], y1[VEC], y2[VEC];
    a.get(x1);
    b.get(x2);
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      const float2 f = ok ? __ldg(c + e) : make_float2(qnan, qnan);
      if constexpr (!BWD) {
        y1[e] = x1[e] * f.x - x2[e] * f.y;
        y2[e] = x2[e] * f.x + x1[e] * f.y;
      } else {
        y1[e] = x1[e] * f.x + x2[e] * f.y;
        y2[e] = x2[e] * f.x - x1[e] * f.y;
      }
    }
    store_n<T, VEC>(d1, y1);
    store_n<T, VEC>(d2, y2);
  }
}

// Block of HP * NVH threads, NVH = D/2/VEC vectors per half head row: thread
// (hl, v) owns vector v (elements v*VEC.. and D/2 + v*VEC..) of heads hl,
// hl + HP, ... (HPT of them per pass) of UT consecutive tokens per iteration;
// token groups are strided by gridDim.  All UT * HPT head loads are issued
// before the first is used, and they do not wait on the position -> cos/sin
// lookup, which is served from L1 / L2 and reused across the thread's heads.
template <typename T, int VEC, bool BWD, int HPT, int UT>
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
  for (int64_t tb = (int64_t)blockIdx.x * UT; tb < T_; tb += (int64_t)gridDim.x * UT) {
    int p[UT];
#pragma unroll
    for (int u = 0; u < UT; ++u) p[u] = tb + u < T_ ? __ldg(pos + tb + u) : 0;
    for (int h0 = hl; h0 < HT; h0 += HP * HPT) {
      Packed<T, VEC> a[UT][HPT], b[UT][HPT];
#pragma unroll
      for (int u = 0; u < UT; ++u) {
        const int64_t t = tb + u;
#pragma unroll
        for (int j = 0; j < HPT; ++j) {
          const int h = h0 + j * HP;
          if (t < T_ && h < HT) {
            const T* src = h < Hq ? q + ((size_t)t * Hq + h) * D : k + ((size_t)t * Hk + (h - Hq)) * D;
            a[u][j].load(src + i0);
            b[u][j].load(src + half + i0);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < UT; ++u) {
        const int64_t t = tb + u;
        if (t >= T_) break;
        // out-of-range position: the table is not read and the outputs are NaN
        const bool ok = p[u] >= 0 && (int64_t)p[u] < max_pos;
        const float2* c = cs + (ok ? (size_t)p[u] * half : 0) + i0;
#pragma unroll
        for (int j = 0; j < HPT; ++j) {
          const int h = h0 + j * HP;
          if (h < HT) {
            T* dst = h < Hq ? qo + ((size_t)t * Hq + h) * D : ko + ((size_t)t * Hk + (h - Hq)) * D;
            rotate_store<T, VEC, BWD>(a[u][j], b[u][j], c, ok, dst + i0, dst + half + i0);
          }
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
#define GBLN_ROPE(N, U)                                                                   \
  rope_kernel<T, VEC, BWD, N, U><<<grid, block, 0, s>>>((const T*)q, (const T*)k, (T*)qo,  \
                                                        (T*)ko, pos, (const float2*)cs,    \
                                                        max_pos, rows, Hq, Hk, D, HP)
  switch (hpt) {  // heads x tokens per thread and pass
    case 1: GBLN_ROPE(1, 2); break;
    case 2: GBLN_ROPE(2, 1); break;
    default: GBLN_ROPE(4, 1); break;
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
  const int ut = hpt == 1 ? 2 : 1;
  const unsigned grid = grid_for((rows + ut - 1) / ut, 1, (int64_t)sms * (per_sm > 0 ? per_sm : 1));
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
