// SwiGLU, out = silu(gate) * up, forward and backward.
//
// Operator: "Fast-LLM: 高效大语言模型训练框架", §三 "支持的 MLP 变体" (gated MLP with
// SiLU) and "训练配置示例" (gated: true, activation: silu, intermediate_size);
// "LLaMA-Factory Kernels 系统" (fused SwiGLU); "Kernels（自定义内核）" §Liger.
//
// Pure streaming: 2 reads + 1 write (forward), 3 reads + 2 writes (backward)
// per element, 128-bit accesses, UNROLL independent vectors in flight per
// thread, grid sized to the resident capacity of the GPU and strided over the
// flat [T * I] index space (rows are contiguous, so the row structure does not
// matter).  The sigmoid is recomputed in the backward pass; nothing is saved.

#include "common.cuh"

namespace gbln {

namespace {

constexpr int kSwiBlock = 256;

// sigmoid(g) = 1 / (1 + exp(-g)).  float32 I/O uses the accurate expf and an
// IEEE division.  bf16 I/O moves only 2 bytes per element, so the arithmetic
// per element must stay within a few instructions for the kernel to remain
// HBM-bound: the fast exponential and the fast division (relative errors of a
// few float32 ulp, far below bf16 rounding).  For g < ~-88, exp(-g) = inf and
// both forms give 0 (the fast division returns 0 for divisors beyond 2^126).
template <typename T>
__device__ __forceinline__ float sigmoid(float g) {
  if constexpr (sizeof(T) == 4) {
    return 1.0f / (1.0f + expf(-g));
  } else {
    return __fdividef(1.0f, 1.0f + __expf(-g));
  }
}

// silu(g) = g * sigmoid(g), as one division for bf16.
template <typename T>
__device__ __forceinline__ float silu(float g) {
  if constexpr (sizeof(T) == 4) {
    return g / (1.0f + expf(-g));
  } else {
    return __fdividef(g, 1.0f + __expf(-g));
  }
}

// Packed 16-byte loads stay packed in registers until they are used, so that
// UNROLL vectors per tensor can be in flight without spilling.
template <typename T, int UNROLL>
__global__ void __launch_bounds__(kSwiBlock)
swiglu_fwd_vec(const T* gate, const T* up, T* out, int64_t nvec) {
  constexpr int VEC = VecOf<T>::N;
  const int64_t step = (int64_t)gridDim.x * kSwiBlock * UNROLL;
  for (int64_t b = (int64_t)blockIdx.x * kSwiBlock * UNROLL + threadIdx.x; b < nvec; b += step) {
    uint4 g[UNROLL], u[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kSwiBlock;
      if (i < nvec) {
        g[k] = ld_stream(gate + i * VEC);
        u[k] = ld_stream(up + i * VEC);
      }
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kSwiBlock;
      if (i < nvec) {
        float gf[VEC], uf[VEC], o[VEC];
        unpack<VEC>(g[k], gf);
        unpack<VEC>(u[k], uf);
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = silu<T>(gf[e]) * uf[e];
        st_vec(out + i * VEC, pack<T, VEC>(o));
      }
    }
  }
}

template <typename T, int UNROLL>
__global__ void __launch_bounds__(kSwiBlock)
swiglu_bwd_vec(const T* dout, const T* gate, const T* up, T* dgate, T* dup, int64_t nvec) {
  constexpr int VEC = VecOf<T>::N;
  const int64_t step = (int64_t)gridDim.x * kSwiBlock * UNROLL;
  for (int64_t b = (int64_t)blockIdx.x * kSwiBlock * UNROLL + threadIdx.x; b < nvec; b += step) {
    uint4 d[UNROLL], g[UNROLL], u[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kSwiBlock;
      if (i < nvec) {
        d[k] = ld_stream(dout + i * VEC);
        g[k] = ld_stream(gate + i * VEC);
        u[k] = ld_stream(up + i * VEC);
      }
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kSwiBlock;
      if (i < nvec) {
        float df[VEC], gf[VEC], uf[VEC], dg[VEC], du[VEC];
        unpack<VEC>(d[k], df);
        unpack<VEC>(g[k], gf);
        unpack<VEC>(u[k], uf);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const float sg = sigmoid<T>(gf[e]);
          const float ds = df[e] * sg;
          du[e] = ds * gf[e];
          dg[e] = ds * uf[e] * (1.0f + gf[e] * (1.0f - sg));
        }
        st_vec(dgate + i * VEC, pack<T, VEC>(dg));
        st_vec(dup + i * VEC, pack<T, VEC>(du));
      }
    }
  }
}

// Element-wise path for unaligned pointers or element counts that are not a
// multiple of the vector width.
template <typename T>
__global__ void __launch_bounds__(kSwiBlock)
swiglu_fwd_scalar(const T* gate, const T* up, T* out, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * kSwiBlock + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * kSwiBlock)
    out[i] = from_f32<T>(silu<T>(to_f32(gate[i])) * to_f32(up[i]));
}

template <typename T>
__global__ void __launch_bounds__(kSwiBlock)
swiglu_bwd_scalar(const T* dout, const T* gate, const T* up, T* dgate, T* dup, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * kSwiBlock + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * kSwiBlock) {
    const float d = to_f32(dout[i]), g = to_f32(gate[i]), u = to_f32(up[i]);
    const float sg = sigmoid<T>(g);
    const float ds = d * sg;
    dgate[i] = from_f32<T>(ds * u * (1.0f + g * (1.0f - sg)));
    dup[i] = from_f32<T>(ds * g);
  }
}

unsigned swiglu_grid(int64_t nvec, int unroll) {
  const int sms = sm_count();
  const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * (2048 / kSwiBlock);
  return grid_for((nvec + unroll - 1) / unroll, kSwiBlock, cap);
}

template <typename T>
gbln_status fwd_typed(const void* g, const void* u, void* o, int64_t n, cudaStream_t s) {
  constexpr int VEC = VecOf<T>::N;
  constexpr int UNROLL = 4;
  if (sm_count() <= 0) return GBLN_ERR_CUDA;
  const bool vec = (n % VEC == 0) && aligned16(g) && aligned16(u) && aligned16(o);
  if (vec) {
    const int64_t nvec = n / VEC;
    swiglu_fwd_vec<T, UNROLL><<<swiglu_grid(nvec, UNROLL), kSwiBlock, 0, s>>>(
        (const T*)g, (const T*)u, (T*)o, nvec);
  } else {
    swiglu_fwd_scalar<T><<<swiglu_grid(n, 1), kSwiBlock, 0, s>>>((const T*)g, (const T*)u,
                                                                 (T*)o, n);
  }
  return launch_status();
}

template <typename T>
gbln_status bwd_typed(const void* d, const void* g, const void* u, void* dg, void* du, int64_t n,
                      cudaStream_t s) {
  constexpr int VEC = VecOf<T>::N;
  constexpr int UNROLL = 4;
  if (sm_count() <= 0) return GBLN_ERR_CUDA;
  const bool vec = (n % VEC == 0) && aligned16(d) && aligned16(g) && aligned16(u) &&
                   aligned16(dg) && aligned16(du);
  if (vec) {
    const int64_t nvec = n / VEC;
    swiglu_bwd_vec<T, UNROLL><<<swiglu_grid(nvec, UNROLL), kSwiBlock, 0, s>>>(
        (const T*)d, (const T*)g, (const T*)u, (T*)dg, (T*)du, nvec);
  } else {
    swiglu_bwd_scalar<T><<<swiglu_grid(n, 1), kSwiBlock, 0, s>>>(
        (const T*)d, (const T*)g, (const T*)u, (T*)dg, (T*)du, n);
  }
  return launch_status();
}

bool sizes_ok(int64_t T, int64_t I) {
  if (T < 0 || I <= 0) return false;
  return T <= (INT64_MAX / 16) / I;  // T * I * 16 bytes does not overflow
}

}  // namespace

}  // namespace gbln

using namespace gbln;

extern "C" gbln_status gbln_swiglu_fwd(const void* gate, const void* up, void* out, int64_t T,
                                       int64_t I, gbln_dtype io, gbln_stream_t stream) {
  if (!dtype_ok(io) || !sizes_ok(T, I)) return GBLN_ERR_INVALID_ARG;
  if (T == 0) return GBLN_OK;  // nothing is read or written: pointers are not examined
  if (!gate || !up || !out) return GBLN_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t n = T * I;
  if (io == GBLN_F32) return fwd_typed<float>(gate, up, out, n, s);
  return fwd_typed<bf16>(gate, up, out, n, s);
}

extern "C" gbln_status gbln_swiglu_bwd(const void* dout, const void* gate, const void* up,
                                       void* dgate, void* dup, int64_t T, int64_t I,
                                       gbln_dtype io, gbln_stream_t stream) {
  if (!dtype_ok(io) || !sizes_ok(T, I)) return GBLN_ERR_INVALID_ARG;
  if (T == 0) return GBLN_OK;  // nothing is read or written: pointers are not examined
  if (!dout || !gate || !up || !dgate || !dup) return GBLN_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t n = T * I;
  if (io == GBLN_F32) return bwd_typed<float>(dout, gate, up, dgate, dup, n, s);
  return bwd_typed<bf16>(dout, gate, up, dgate, dup, n, s);
}
