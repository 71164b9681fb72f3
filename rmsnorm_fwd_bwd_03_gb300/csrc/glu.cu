// Gated MLP units (SwiGLU and its GeLU / ReLU siblings) and plain activations,
// forward and backward.
//
// Operator: "Fast-LLM: 高效大语言模型训练框架", §三 "支持的 MLP 变体" (dense MLP, gated
// or not, SiLU / GeLU / ReLU) and "训练配置示例" (gated: true, activation: silu,
// intermediate_size); "LLaMA-Factory Kernels 系统" (fused SwiGLU);
// "Kernels（自定义内核）" §Liger.
//
// Pure streaming: 2 reads + 1 write (gated forward), 3 reads + 2 writes (gated
// backward), 1 + 1 and 2 + 1 for the plain activation, 128-bit accesses,
// UNROLL independent vectors in flight per thread, grid sized to the resident
// capacity of the GPU.  Contiguous tensors are walked as one flat index space;
// row-strided ones (gate and up as the two halves of a packed [T, 2I]
// projection output, for instance) by (row group, column block) units.  The
// activation is recomputed in the backward pass; nothing is saved.  The gated
// forward can also deliver its output as MXFP8 (E4M3 codes and one E8M0 scale
// per 32 values of a row) for the down projection.

#include "common.cuh"

namespace gbln {

namespace {

constexpr int kGluBlock = 256;

// bf16 I/O moves only 2 bytes per element, so the arithmetic per element must
// stay within a few instructions for the kernels to remain HBM-bound.  Their
// exponentials and reciprocals therefore go straight to the hardware's base-2
// exponential and reciprocal approximations in flush-to-zero form
// (ex2.approx.ftz, rcp.approx.ftz), with e^a = 2^(a log2 e).  Their relative
// errors are a few float32 ulp, far below bf16 rounding, and none of the
// formulas needs denormals (a denormal exponential or reciprocal is far below
// bf16 resolution wherever it appears); dropping the denormal handling saves
// instructions.  float32 I/O keeps the accurate library functions.
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_ftz(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// e^a for the bf16 paths (a * log2 e rounded once, then ex2).
__device__ __forceinline__ float exp_fast(float a) { return ex2_ftz(a * kLog2e); }

// sigmoid(g) = 1 / (1 + exp(-g)): expf and an IEEE division for float32 I/O.
// For g < ~-88, exp(-g) = inf and both forms give 0 (the reciprocal of inf is 0).
template <typename T>
__device__ __forceinline__ float sigmoid(float g) {
  if constexpr (sizeof(T) == 4) {
    return 1.0f / (1.0f + expf(-g));
  } else {
    return rcp_ftz(1.0f + exp_fast(-g));
  }
}

// GeLU, tanh form: 0.5 x (1 + tanh(z)) with z = sqrt(2/pi) (x + 0.044715 x^3).
// Since 0.5 (1 + tanh(z)) = sigmoid(2 z), it is evaluated as x * sigmoid(2 z),
// which has no cancellation for negative x.
constexpr float kGeluK = 1.5957691216057308f;   // 2 * sqrt(2 / pi)
constexpr float kGeluC = 0.044715f;
constexpr float kInvSqrt2 = 0.7071067811865476f;
constexpr float kInvSqrt2Pi = 0.3989422804014327f;  // 1 / sqrt(2 pi)

// Normal CDF for the bf16 path from the rational approximation of erfc in
// Abramowitz & Stegun, Handbook of Mathematical Functions, formula 7.1.26
// (absolute error of erf below 1.5e-7): for z >= 0, erfc(z) ~ (a1 t + a2 t^2 +
// a3 t^3 + a4 t^4 + a5 t^5) e^{-z^2} with t = 1 / (1 + p z).  With z = |x| /
// sqrt(2): Phi(x) = erfc(z) / 2 for x < 0 (no cancellation) and 1 - erfc(z) / 2
// for x >= 0.  ex receives e^{-z^2} = e^{-x^2/2}, the Gaussian density's
// exponential, which the backward pass needs as well.  About half the
// instructions of erff; float32 I/O keeps erff.
constexpr float kAsP = 0.3275911f;
constexpr float kAsA1 = 0.254829592f, kAsA2 = -0.284496736f, kAsA3 = 1.421413741f,
                kAsA4 = -1.453152027f, kAsA5 = 1.061405429f;

__device__ __forceinline__ float gauss_cdf_as(float x, float& ex) {
  const float z = fabsf(x) * kInvSqrt2;
  const float t = rcp_ftz(fmaf(kAsP, z, 1.0f));
  ex = exp_fast(-z * z);
  const float poly = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, kAsA5, kAsA4), kAsA3), kAsA2), kAsA1);
  const float half_erfc = 0.5f * poly * ex;
  return x >= 0.f ? 1.0f - half_erfc : half_erfc;
}

// Activation value f(x) and, for the backward pass, f(x) and f'(x) together.
template <typename T, int ACT>
__device__ __forceinline__ float act_f(float x) {
  if constexpr (ACT == GBLN_ACT_SILU) {
    if constexpr (sizeof(T) == 4) return x / (1.0f + expf(-x));
    else return x * rcp_ftz(1.0f + exp_fast(-x));
  } else if constexpr (ACT == GBLN_ACT_GELU_TANH) {
    return x * sigmoid<T>(kGeluK * (x + kGeluC * x * x * x));
  } else if constexpr (ACT == GBLN_ACT_GELU_ERF) {
    if constexpr (sizeof(T) == 4) {
      return 0.5f * x * (1.0f + erff(x * kInvSqrt2));
    } else {
      float ex;
      return x * gauss_cdf_as(x, ex);
    }
  } else {
    return x > 0.f ? x : 0.f;
  }
}

template <typename T, int ACT>
__device__ __forceinline__ void act_fd(float x, float& f, float& d) {
  if constexpr (ACT == GBLN_ACT_SILU) {
    const float s = sigmoid<T>(x);
    f = x * s;
    d = s * (1.0f + x * (1.0f - s));
  } else if constexpr (ACT == GBLN_ACT_GELU_TANH) {
    const float s = sigmoid<T>(kGeluK * (x + kGeluC * x * x * x));
    f = x * s;
    d = s + x * s * (1.0f - s) * kGeluK * (1.0f + 3.0f * kGeluC * x * x);
  } else if constexpr (ACT == GBLN_ACT_GELU_ERF) {
    if constexpr (sizeof(T) == 4) {
      const float cdf = 0.5f * (1.0f + erff(x * kInvSqrt2));
      f = x * cdf;
      d = cdf + x * kInvSqrt2Pi * expf(-0.5f * x * x);
    } else {
      float ex;
      const float cdf = gauss_cdf_as(x, ex);
      f = x * cdf;
      d = cdf + x * kInvSqrt2Pi * ex;
    }
  } else {
    f = x > 0.f ? x : 0.f;
    d = x > 0.f ? 1.f : 0.f;
  }
}

// ---------------------------------------------------------------------------
// Contiguous tensors: flat index over n / VEC vectors.  Packed 16-byte loads
// stay packed in registers until used, so UNROLL vectors per tensor can be in
// flight without spilling.
// ---------------------------------------------------------------------------
template <typename T, int ACT, int UNROLL>
__global__ void __launch_bounds__(kGluBlock)
glu_fwd_vec(const T* gate, const T* up, T* out, int64_t nvec) {
  constexpr int VEC = VecOf<T>::N;
  const int64_t step = (int64_t)gridDim.x * kGluBlock * UNROLL;
  for (int64_t b = (int64_t)blockIdx.x * kGluBlock * UNROLL + threadIdx.x; b < nvec; b += step) {
    uint4 g[UNROLL], u[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kGluBlock;
      if (i < nvec) {
        g[k] = ld_stream(gate + i * VEC);
        u[k] = ld_stream(up + i * VEC);
      }
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kGluBlock;
      if (i < nvec) {
        float gf[VEC], uf[VEC], o[VEC];
        unpack<VEC>(g[k], gf);
        unpack<VEC>(u[k], uf);
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = act_f<T, ACT>(gf[e]) * uf[e];
        st_vec(out + i * VEC, pack<T, VEC>(o));
      }
    }
  }
}

template <typename T, int ACT, int UNROLL>
__global__ void __launch_bounds__(kGluBlock)
glu_bwd_vec(const T* dout, const T* gate, const T* up, T* dgate, T* dup, int64_t nvec) {
  constexpr int VEC = VecOf<T>::N;
  const int64_t step = (int64_t)gridDim.x * kGluBlock * UNROLL;
  for (int64_t b = (int64_t)blockIdx.x * kGluBlock * UNROLL + threadIdx.x; b < nvec; b += step) {
    uint4 d[UNROLL], g[UNROLL], u[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kGluBlock;
      if (i < nvec) {
        d[k] = ld_stream(dout + i * VEC);
        g[k] = ld_stream(gate + i * VEC);
        u[k] = ld_stream(up + i * VEC);
      }
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kGluBlock;
      if (i < nvec) {
        float df[VEC], gf[VEC], uf[VEC], dg[VEC], du[VEC];
        unpack<VEC>(d[k], df);
        unpack<VEC>(g[k], gf);
        unpack<VEC>(u[k], uf);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          float f, fp;
          act_fd<T, ACT>(gf[e], f, fp);
          du[e] = df[e] * f;
          dg[e] = df[e] * uf[e] * fp;
        }
        st_vec(dgate + i * VEC, pack<T, VEC>(dg));
        st_vec(dup + i * VEC, pack<T, VEC>(du));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Row-strided tensors.  A unit is (group of UNROLL consecutive rows, block of
// blockDim.x column vectors); thread t takes column vector j * blockDim.x + t
// of each row of the group, so a warp's accesses stay contiguous within a row.
// The host picks the block width so that the column blocks tile the row.
// VEC = 1 is the element-wise path (unaligned pointers or strides).
// ---------------------------------------------------------------------------
template <typename T, int VEC, int ACT, int UNROLL>
__global__ void __launch_bounds__(kGluBlock)
glu_fwd_rows(const T* gate, const T* up, T* out, int64_t T_, int64_t ncol, int64_t ldg,
             int64_t ldu, int64_t ldo) {
  const int cb = blockDim.x;
  const int64_t ncb = (ncol + cb - 1) / cb;
  const int64_t units = (T_ + UNROLL - 1) / UNROLL * ncb;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int64_t rg = u / ncb;
    const int64_t c = (u - rg * ncb) * cb + threadIdx.x;
    if (c >= ncol) continue;
    const int64_t r0 = rg * UNROLL;
    Packed<T, VEC> g[UNROLL], v[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      if (r0 + k < T_) {
        g[k].load(gate + (r0 + k) * ldg + c * VEC);
        v[k].load(up + (r0 + k) * ldu + c * VEC);
      }
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      if (r0 + k < T_) {
        float gf[VEC], uf[VEC], o[VEC];
        g[k].get(gf);
        v[k].get(uf);
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = act_f<T, ACT>(gf[e]) * uf[e];
        store_n<T, VEC>(out + (r0 + k) * ldo + c * VEC, o);
      }
    }
  }
}

template <typename T, int VEC, int ACT, int UNROLL>
__global__ void __launch_bounds__(kGluBlock)
glu_bwd_rows(const T* dout, const T* gate, const T* up, T* dgate, T* dup, int64_t T_,
             int64_t ncol, int64_t ldd, int64_t ldg, int64_t ldu, int64_t lddg, int64_t lddu) {
  const int cb = blockDim.x;
  const int64_t ncb = (ncol + cb - 1) / cb;
  const int64_t units = (T_ + UNROLL - 1) / UNROLL * ncb;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int64_t rg = u / ncb;
    const int64_t c = (u - rg * ncb) * cb + threadIdx.x;
    if (c >= ncol) continue;
    const int64_t r0 = rg * UNROLL;
    Packed<T, VEC> d[UNROLL], g[UNROLL], v[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      if (r0 + k < T_) {
        d[k].load(dout + (r0 + k) * ldd + c * VEC);
        g[k].load(gate + (r0 + k) * ldg + c * VEC);
        v[k].load(up + (r0 + k) * ldu + c * VEC);
      }
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      if (r0 + k < T_) {
        float df[VEC], gf[VEC], uf[VEC], dg[VEC], du[VEC];
        d[k].get(df);
        g[k].get(gf);
        v[k].get(uf);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          float f, fp;
          act_fd<T, ACT>(gf[e], f, fp);
          du[e] = df[e] * f;
          dg[e] = df[e] * uf[e] * fp;
        }
        store_n<T, VEC>(dgate + (r0 + k) * lddg + c * VEC, dg);
        store_n<T, VEC>(dup + (r0 + k) * lddu + c * VEC, du);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Plain activation y = f(x), dx = dy * f'(x) over n contiguous elements.
// ---------------------------------------------------------------------------
template <typename T, int VEC, int ACT, int UNROLL>
__global__ void __launch_bounds__(kGluBlock)
act_fwd_kernel(const T* x, T* y, int64_t nv) {
  const int64_t step = (int64_t)gridDim.x * kGluBlock * UNROLL;
  for (int64_t b = (int64_t)blockIdx.x * kGluBlock * UNROLL + threadIdx.x; b < nv; b += step) {
    Packed<T, VEC> a[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kGluBlock;
      if (i < nv) a[k].load(x + i * VEC);
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kGluBlock;
      if (i < nv) {
        float v[VEC];
        a[k].get(v);
#pragma unroll
        for (int e = 0; e < VEC; ++e) v[e] = act_f<T, ACT>(v[e]);
        store_n<T, VEC>(y + i * VEC, v);
      }
    }
  }
}

template <typename T, int VEC, int ACT, int UNROLL>
__global__ void __launch_bounds__(kGluBlock)
act_bwd_kernel(const T* dy, const T* x, T* dx, int64_t nv) {
  const int64_t step = (int64_t)gridDim.x * kGluBlock * UNROLL;
  for (int64_t b = (int64_t)blockIdx.x * kGluBlock * UNROLL + threadIdx.x; b < nv; b += step) {
    Packed<T, VEC> a[UNROLL], d[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kGluBlock;
      if (i < nv) {
        a[k].load(x + i * VEC);
        d[k].load(dy + i * VEC);
      }
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const int64_t i = b + (int64_t)k * kGluBlock;
      if (i < nv) {
        float v[VEC], dv[VEC];
        a[k].get(v);
        d[k].get(dv);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          float f, fp;
          act_fd<T, ACT>(v[e], f, fp);
          v[e] = dv[e] * fp;
        }
        store_n<T, VEC>(dx + i * VEC, v);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Forward with MXFP8 output (codes [T, I] and one scale byte per 32 values of
// a row), for the down projection's FP8 operand.  Same units as glu_fwd_rows;
// I is a multiple of 32, so an MX block is 32 / VEC consecutive column
// vectors, held by consecutive lanes.  Every lane runs the quantisation (its
// warp shuffles need all 32), inactive lanes with nothing to store.
// ---------------------------------------------------------------------------
template <typename T, int VEC, int ACT, int UNROLL>
__global__ void __launch_bounds__(kGluBlock)
glu_fwd_mx(const T* gate, const T* up, MxOut mx, int64_t T_, int64_t ncol, int64_t ldg,
           int64_t ldu) {
  constexpr int LB = kMxBlock / VEC;
  const int64_t I = ncol * VEC;
  const int cb = blockDim.x;
  const int64_t ncb = (ncol + cb - 1) / cb;
  const int64_t units = (T_ + UNROLL - 1) / UNROLL * ncb;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int64_t rg = u / ncb;
    const int64_t c = (u - rg * ncb) * cb + threadIdx.x;
    const bool colok = c < ncol;
    const int64_t r0 = rg * UNROLL;
    Packed<T, VEC> g[UNROLL], v[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      if (colok && r0 + k < T_) {
        g[k].load(gate + (r0 + k) * ldg + c * VEC);
        v[k].load(up + (r0 + k) * ldu + c * VEC);
      }
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      if (r0 + k >= T_) break;  // uniform across the block
      float o[VEC];
      if (colok) {
        float gf[VEC], uf[VEC];
        g[k].get(gf);
        v[k].get(uf);
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = act_f<T, ACT>(gf[e]) * uf[e];
      }
      mx_store<VEC>(o, colok, c % LB == 0, mx.q + (r0 + k) * I + c * VEC,
                    mx.sc + (r0 + k) * (I / kMxBlock) + c / LB);
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

unsigned resident_grid(int64_t units, int threads = kGluBlock) {
  const int sms = sm_count();
  const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * (2048 / threads);
  return grid_for(units, 1, cap);
}

// Threads per block of the row-strided kernels: the multiple of 32 in
// [128, kGluBlock] whose column blocks cover a row of ncol units with the
// fewest idle lanes, the widest on a tie.  A bf16 row of 3072 values (384
// vectors) gets two blocks of 192 instead of one and a half of 256.
int col_block(int64_t ncol) {
  int best = kGluBlock;
  int64_t best_slots = -1;
  for (int b = kGluBlock; b >= 128; b -= 32) {
    const int64_t slots = (ncol + b - 1) / b * b;
    if (best_slots < 0 || slots < best_slots) {
      best = b;
      best_slots = slots;
    }
  }
  return best;
}

template <typename T, int ACT>
void glu_fwd_launch(const void* g, const void* u, void* o, int64_t rows, int64_t I, int64_t ldg,
                    int64_t ldu, int64_t ldo, cudaStream_t s) {
  constexpr int VEC = VecOf<T>::N;
  const bool contiguous = ldg == I && ldu == I && ldo == I;
  const bool aligned = aligned16(g) && aligned16(u) && aligned16(o);
  if (contiguous && aligned && (rows * I) % VEC == 0) {
    constexpr int U = 4;
    const int64_t nvec = rows * I / VEC;
    glu_fwd_vec<T, ACT, U><<<resident_grid((nvec + U - 1) / U / kGluBlock + 1), kGluBlock, 0, s>>>(
        (const T*)g, (const T*)u, (T*)o, nvec);
  } else if (aligned && I % VEC == 0 && ldg % VEC == 0 && ldu % VEC == 0 && ldo % VEC == 0) {
    constexpr int U = 4;
    const int64_t ncol = I / VEC;
    const int cb = col_block(ncol);
    const int64_t units = (rows + U - 1) / U * ((ncol + cb - 1) / cb);
    glu_fwd_rows<T, VEC, ACT, U><<<resident_grid(units, cb), cb, 0, s>>>(
        (const T*)g, (const T*)u, (T*)o, rows, ncol, ldg, ldu, ldo);
  } else {
    constexpr int U = 4;
    const int cb = col_block(I);
    const int64_t units = (rows + U - 1) / U * ((I + cb - 1) / cb);
    glu_fwd_rows<T, 1, ACT, U><<<resident_grid(units, cb), cb, 0, s>>>(
        (const T*)g, (const T*)u, (T*)o, rows, I, ldg, ldu, ldo);
  }
}

template <typename T, int ACT>
void glu_fwd_mx_launch(const void* g, const void* u, MxOut mx, int64_t rows, int64_t I, int64_t ldg,
                       int64_t ldu, cudaStream_t s) {
  constexpr int VEC = VecOf<T>::N;
  constexpr int U = 4;
  const bool vec = aligned16(g) && aligned16(u) && ldg % VEC == 0 && ldu % VEC == 0 &&
                   reinterpret_cast<uintptr_t>(mx.q) % VEC == 0;  // VEC codes per lane
  if (vec) {
    const int64_t ncol = I / VEC;
    const int cb = col_block(ncol);
    const int64_t units = (rows + U - 1) / U * ((ncol + cb - 1) / cb);
    glu_fwd_mx<T, VEC, ACT, U><<<resident_grid(units, cb), cb, 0, s>>>((const T*)g, (const T*)u, mx,
                                                                          rows, ncol, ldg, ldu);
  } else {
    const int cb = col_block(I);
    const int64_t units = (rows + U - 1) / U * ((I + cb - 1) / cb);
    glu_fwd_mx<T, 1, ACT, U><<<resident_grid(units, cb), cb, 0, s>>>((const T*)g, (const T*)u, mx,
                                                                        rows, I, ldg, ldu);
  }
}

template <typename T, int ACT>
void glu_bwd_launch(const void* d, const void* g, const void* u, void* dg, void* du, int64_t rows,
                    int64_t I, int64_t ldd, int64_t ldg, int64_t ldu, int64_t lddg, int64_t lddu,
                    cudaStream_t s) {
  constexpr int VEC = VecOf<T>::N;
  const bool contiguous = ldd == I && ldg == I && ldu == I && lddg == I && lddu == I;
  const bool aligned = aligned16(d) && aligned16(g) && aligned16(u) && aligned16(dg) && aligned16(du);
  if (contiguous && aligned && (rows * I) % VEC == 0) {
    constexpr int U = 4;
    const int64_t nvec = rows * I / VEC;
    glu_bwd_vec<T, ACT, U><<<resident_grid((nvec + U - 1) / U / kGluBlock + 1), kGluBlock, 0, s>>>(
        (const T*)d, (const T*)g, (const T*)u, (T*)dg, (T*)du, nvec);
  } else if (aligned && I % VEC == 0 && ldd % VEC == 0 && ldg % VEC == 0 && ldu % VEC == 0 &&
             lddg % VEC == 0 && lddu % VEC == 0) {
    constexpr int U = 2;
    const int64_t ncol = I / VEC;
    const int cb = col_block(ncol);
    const int64_t units = (rows + U - 1) / U * ((ncol + cb - 1) / cb);
    glu_bwd_rows<T, VEC, ACT, U><<<resident_grid(units, cb), cb, 0, s>>>(
        (const T*)d, (const T*)g, (const T*)u, (T*)dg, (T*)du, rows, ncol, ldd, ldg, ldu, lddg, lddu);
  } else {
    constexpr int U = 2;
    const int cb = col_block(I);
    const int64_t units = (rows + U - 1) / U * ((I + cb - 1) / cb);
    glu_bwd_rows<T, 1, ACT, U><<<resident_grid(units, cb), cb, 0, s>>>(
        (const T*)d, (const T*)g, (const T*)u, (T*)dg, (T*)du, rows, I, ldd, ldg, ldu, lddg, lddu);
  }
}

template <typename T, int ACT>
void act_fwd_launch(const void* x, void* y, int64_t n, cudaStream_t s) {
  constexpr int VEC = VecOf<T>::N;
  constexpr int U = 4;
  if (aligned16(x) && aligned16(y) && n % VEC == 0) {
    const int64_t nv = n / VEC;
    act_fwd_kernel<T, VEC, ACT, U><<<resident_grid((nv + U - 1) / U / kGluBlock + 1), kGluBlock, 0, s>>>(
        (const T*)x, (T*)y, nv);
  } else {
    act_fwd_kernel<T, 1, ACT, U><<<resident_grid((n + U - 1) / U / kGluBlock + 1), kGluBlock, 0, s>>>(
        (const T*)x, (T*)y, n);
  }
}

template <typename T, int ACT>
void act_bwd_launch(const void* dy, const void* x, void* dx, int64_t n, cudaStream_t s) {
  constexpr int VEC = VecOf<T>::N;
  constexpr int U = 4;
  if (aligned16(x) && aligned16(dy) && aligned16(dx) && n % VEC == 0) {
    const int64_t nv = n / VEC;
    act_bwd_kernel<T, VEC, ACT, U><<<resident_grid((nv + U - 1) / U / kGluBlock + 1), kGluBlock, 0, s>>>(
        (const T*)dy, (const T*)x, (T*)dx, nv);
  } else {
    act_bwd_kernel<T, 1, ACT, U><<<resident_grid((n + U - 1) / U / kGluBlock + 1), kGluBlock, 0, s>>>(
        (const T*)dy, (const T*)x, (T*)dx, n);
  }
}

// Dispatch on (io, act) to a templated launcher F<T, ACT>::run(args...).
#define GBLN_DISPATCH_ACT(T, act, CALL)                       \
  switch (act) {                                              \
    case GBLN_ACT_SILU: CALL(T, GBLN_ACT_SILU); break;        \
    case GBLN_ACT_GELU_TANH: CALL(T, GBLN_ACT_GELU_TANH); break; \
    case GBLN_ACT_GELU_ERF: CALL(T, GBLN_ACT_GELU_ERF); break; \
    default: CALL(T, GBLN_ACT_RELU); break;                   \
  }

bool act_ok(int a) { return a >= GBLN_ACT_SILU && a <= GBLN_ACT_RELU; }

bool sizes_ok(int64_t T, int64_t I) {
  if (T < 0 || I <= 0) return false;
  return T <= (INT64_MAX / 16) / I;  // T * I * 16 bytes does not overflow
}

// Strides: at least the row width, and the last row's end must not overflow.
bool ld_ok(int64_t T, int64_t I, int64_t ld) {
  return ld >= I && (T == 0 || ld <= (INT64_MAX / 16 - I) / (T > 1 ? T - 1 : 1));
}

}  // namespace

}  // namespace gbln

using namespace gbln;

extern "C" gbln_status gbln_glu_fwd(const void* gate, const void* up, void* out, int64_t T,
                                    int64_t I, int64_t ld_gate, int64_t ld_up, int64_t ld_out,
                                    gbln_act act, gbln_dtype io, gbln_stream_t stream) {
  if (!dtype_ok(io) || !act_ok(act) || !sizes_ok(T, I)) return GBLN_ERR_INVALID_ARG;
  if (!ld_ok(T, I, ld_gate) || !ld_ok(T, I, ld_up) || !ld_ok(T, I, ld_out)) return GBLN_ERR_INVALID_ARG;
  if (T == 0) return GBLN_OK;  // nothing is read or written: pointers are not examined
  if (!gate || !up || !out) return GBLN_ERR_INVALID_ARG;
  if (sm_count() <= 0) return GBLN_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
#define GBLN_GLU_FWD(TY, A) glu_fwd_launch<TY, A>(gate, up, out, T, I, ld_gate, ld_up, ld_out, s)
  if (io == GBLN_F32) {
    GBLN_DISPATCH_ACT(float, act, GBLN_GLU_FWD)
  } else {
    GBLN_DISPATCH_ACT(bf16, act, GBLN_GLU_FWD)
  }
#undef GBLN_GLU_FWD
  return launch_status();
}

extern "C" gbln_status gbln_glu_fwd_mxfp8(const void* gate, const void* up, uint8_t* out_e4m3,
                                          uint8_t* out_scale, int64_t T, int64_t I,
                                          int64_t ld_gate, int64_t ld_up, gbln_act act,
                                          gbln_dtype io, gbln_stream_t stream) {
  if (!dtype_ok(io) || !act_ok(act) || !sizes_ok(T, I) || I % kMxBlock != 0) return GBLN_ERR_INVALID_ARG;
  if (!ld_ok(T, I, ld_gate) || !ld_ok(T, I, ld_up)) return GBLN_ERR_INVALID_ARG;
  if (T == 0) return GBLN_OK;  // nothing is read or written: pointers are not examined
  if (!gate || !up || !out_e4m3 || !out_scale) return GBLN_ERR_INVALID_ARG;
  if (sm_count() <= 0) return GBLN_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  const MxOut mx{out_e4m3, out_scale};
#define GBLN_GLU_FWD_MX(TY, A) glu_fwd_mx_launch<TY, A>(gate, up, mx, T, I, ld_gate, ld_up, s)
  if (io == GBLN_F32) {
    GBLN_DISPATCH_ACT(float, act, GBLN_GLU_FWD_MX)
  } else {
    GBLN_DISPATCH_ACT(bf16, act, GBLN_GLU_FWD_MX)
  }
#undef GBLN_GLU_FWD_MX
  return launch_status();
}

extern "C" gbln_status gbln_glu_bwd(const void* dout, const void* gate, const void* up,
                                    void* dgate, void* dup, int64_t T, int64_t I,
                                    int64_t ld_dout, int64_t ld_gate, int64_t ld_up,
                                    int64_t ld_dgate, int64_t ld_dup, gbln_act act,
                                    gbln_dtype io, gbln_stream_t stream) {
  if (!dtype_ok(io) || !act_ok(act) || !sizes_ok(T, I)) return GBLN_ERR_INVALID_ARG;
  if (!ld_ok(T, I, ld_dout) || !ld_ok(T, I, ld_gate) || !ld_ok(T, I, ld_up) ||
      !ld_ok(T, I, ld_dgate) || !ld_ok(T, I, ld_dup))
    return GBLN_ERR_INVALID_ARG;
  if (T == 0) return GBLN_OK;  // nothing is read or written: pointers are not examined
  if (!dout || !gate || !up || !dgate || !dup) return GBLN_ERR_INVALID_ARG;
  if (sm_count() <= 0) return GBLN_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
#define GBLN_GLU_BWD(TY, A) \
  glu_bwd_launch<TY, A>(dout, gate, up, dgate, dup, T, I, ld_dout, ld_gate, ld_up, ld_dgate, ld_dup, s)
  if (io == GBLN_F32) {
    GBLN_DISPATCH_ACT(float, act, GBLN_GLU_BWD)
  } else {
    GBLN_DISPATCH_ACT(bf16, act, GBLN_GLU_BWD)
  }
#undef GBLN_GLU_BWD
  return launch_status();
}

extern "C" gbln_status gbln_swiglu_fwd(const void* gate, const void* up, void* out, int64_t T,
                                       int64_t I, gbln_dtype io, gbln_stream_t stream) {
  return gbln_glu_fwd(gate, up, out, T, I, I, I, I, GBLN_ACT_SILU, io, stream);
}

extern "C" gbln_status gbln_swiglu_bwd(const void* dout, const void* gate, const void* up,
                                       void* dgate, void* dup, int64_t T, int64_t I,
                                       gbln_dtype io, gbln_stream_t stream) {
  return gbln_glu_bwd(dout, gate, up, dgate, dup, T, I, I, I, I, I, I, GBLN_ACT_SILU, io, stream);
}

extern "C" gbln_status gbln_act_fwd(const void* x, void* y, int64_t n, gbln_act act,
                                    gbln_dtype io, gbln_stream_t stream) {
  if (!dtype_ok(io) || !act_ok(act) || !sizes_ok(n, 1)) return GBLN_ERR_INVALID_ARG;
  if (n == 0) return GBLN_OK;
  if (!x || !y) return GBLN_ERR_INVALID_ARG;
  if (sm_count() <= 0) return GBLN_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
#define GBLN_ACT_FWD(TY, A) act_fwd_launch<TY, A>(x, y, n, s)
  if (io == GBLN_F32) {
    GBLN_DISPATCH_ACT(float, act, GBLN_ACT_FWD)
  } else {
    GBLN_DISPATCH_ACT(bf16, act, GBLN_ACT_FWD)
  }
#undef GBLN_ACT_FWD
  return launch_status();
}

extern "C" gbln_status gbln_act_bwd(const void* dy, const void* x, void* dx, int64_t n,
                                    gbln_act act, gbln_dtype io, gbln_stream_t stream) {
  if (!dtype_ok(io) || !act_ok(act) || !sizes_ok(n, 1)) return GBLN_ERR_INVALID_ARG;
  if (n == 0) return GBLN_OK;
  if (!dy || !x || !dx) return GBLN_ERR_INVALID_ARG;
  if (sm_count() <= 0) return GBLN_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
#define GBLN_ACT_BWD(TY, A) act_bwd_launch<TY, A>(dy, x, dx, n, s)
  if (io == GBLN_F32) {
    GBLN_DISPATCH_ACT(float, act, GBLN_ACT_BWD)
  } else {
    GBLN_DISPATCH_ACT(bf16, act, GBLN_ACT_BWD)
  }
#undef GBLN_ACT_BWD
  return launch_status();
}
