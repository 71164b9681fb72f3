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
// IEEE division; bf16 I/O uses the fast exponential and an IEEE reciprocal (its
// error is far below bf16 rounding).  Both give 0 for g < ~-88 (exp -> inf).
template <typename T>
__device__ __forceinline__ float sigmoid(float g) {
  if constexpr (sizeof(T) == 4) {
    return 1.0f / (1.0f + expf(-g));
  } else {
    return __frcp_rn(1.0f + __expf(-g));
  }
}

template <typename T, int VEC, int UNROLL>
__global__ void __launch_bounds__(kSwiBlock)
swiglu_fwd_kernel(const T* gate, const T* up, T* out, int64_t nvec) {
  const int64_t step = (int64_t)gridDim.x * kSwiBlock * UNROLL;
  for (int64_t b = (int64_t)blockIdx.x * kSwiBlock * UNROLL + threadIdx.x; b < nvec; b += step) {
    float g[UNROLL][VEC], u[UNROLL][VEC];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kSwiBlock;
      if (i < nvec) {
        load_n<T, VEC>(gate + i * VEC, g[k]);
        load_n<T, VEC>(up + i * VEC, u[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kSwiBlock;
      if (i < nvec) {
        float o[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = g[k][e] * sigmoid<T>(g[k][e]) * u[k][e];
        store_n<T, VEC>(out + i * VEC, o);
      }
    }
  }
}

template <typename T, int VEC, int UNROLL>
__global__ void __launch_bounds__(kSwiBlock)
swiglu_bwd_kernel(const T* dout, const T* gate, const T* up, T* dgate, T* dup, int64_t nvec) {
  const int64_t step = (int64_t)gridDim.x * kSwiBlock * UNROLL;
  for (int64_t b = (int64_t)blockIdx.x * kSwiBlock * UNROLL + threadIdx.x; b < nvec; b += step) {
    float d[UNROLL][VEC], g[UNROLL][VEC], u[UNROLL][VEC];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kSwiBlock;
      if (i < nvec) {
        load_n<T, VEC>(dout + i * VEC, d[k]);
        load_n<T, VEC>(gate + i * VEC, g[k]);
        load_n<T, VEC>(up + i * VEC, u[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kSwiBlock;
      if (i < nvec) {
        float dg[VEC], du[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const float s = sigmoid<T>(g[k][e]);
          const float ds = d[k][e] * s;
          du[e] = ds * g[k][e];
          dg[e] = ds * u[k][e] * (1.0f + g[k][e] * (1.0f - s));
        }
        store_n<T, VEC>(dgate + i * VEC, dg);
        store_n<T, VEC>(dup + i * VEC, du);
      }
    }
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
    swiglu_fwd_kernel<T, VEC, UNROLL><<<swiglu_grid(nvec, UNROLL), kSwiBlock, 0, s>>>(
        (const T*)g, (const T*)u, (T*)o, nvec);
  } else {
    swiglu_fwd_kernel<T, 1, UNROLL><<<swiglu_grid(n, UNROLL), kSwiBlock, 0, s>>>(
        (const T*)g, (const T*)u, (T*)o, n);
  }
  return launch_status();
}

template <typename T>
gbln_status bwd_typed(const void* d, const void* g, const void* u, void* dg, void* du, int64_t n,
                      cudaStream_t s) {
  constexpr int VEC = VecOf<T>::N;
  constexpr int UNROLL = 2;
  if (sm_count() <= 0) return GBLN_ERR_CUDA;
  const bool vec = (n % VEC == 0) && aligned16(d) && aligned16(g) && aligned16(u) &&
                   aligned16(dg) && aligned16(du);
  if (vec) {
    const int64_t nvec = n / VEC;
    swiglu_bwd_kernel<T, VEC, UNROLL><<<swiglu_grid(nvec, UNROLL), kSwiBlock, 0, s>>>(
        (const T*)d, (const T*)g, (const T*)u, (T*)dg, (T*)du, nvec);
  } else {
    swiglu_bwd_kernel<T, 1, UNROLL><<<swiglu_grid(n, UNROLL), kSwiBlock, 0, s>>>(
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
  if (!gate || !up || !out) return GBLN_ERR_INVALID_ARG;
  if (T == 0) return GBLN_OK;
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t n = T * I;
  if (io == GBLN_F32) return fwd_typed<float>(gate, up, out, n, s);
  return fwd_typed<bf16>(gate, up, out, n, s);
}

extern "C" gbln_status gbln_swiglu_bwd(const void* dout, const void* gate, const void* up,
                                       void* dgate, void* dup, int64_t T, int64_t I,
                                       gbln_dtype io, gbln_stream_t stream) {
  if (!dtype_ok(io) || !sizes_ok(T, I)) return GBLN_ERR_INVALID_ARG;
  if (!dout || !gate || !up || !dgate || !dup) return GBLN_ERR_INVALID_ARG;
  if (T == 0) return GBLN_OK;
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t n = T * I;
  if (io == GBLN_F32) return bwd_typed<float>(dout, gate, up, dgate, dup, n, s);
  return bwd_typed<bf16>(dout, gate, up, dgate, dup, n, s);
}
