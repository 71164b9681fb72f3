// Shared device helpers of libgbln: 128-bit loads / stores and packs of bf16 /
// f32, fp32 row reductions (warp shuffles, named barriers, compensated sums),
// the fixed-order column sum that finishes the weight gradients, the MXFP8
// quantisation epilogue, TMA bulk copies with bounded mbarrier waits, the L2
// prefetch, and the host-side argument checks.  Nothing here is used by the
// CPU oracle, and nothing from it is used here.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "gbln.h"

namespace gbln {

typedef __nv_bfloat16 bf16;

// Elements per 16-byte access.
template <typename T> struct VecOf;
template <> struct VecOf<float> { static constexpr int N = 4; };
template <> struct VecOf<bf16> { static constexpr int N = 8; };

// ---------------------------------------------------------------------------
// Loads and stores of N consecutive elements as float32.
// N * sizeof(T) == 16 uses one 128-bit access (pointer must be 16-B aligned);
// N == 1 is the element-wise path for unaligned rows.
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(bf16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

// Streaming read of data touched once: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
// Read-only data reused across rows (weights, cos/sin table): cached path.
__device__ __forceinline__ uint4 ld_reuse(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_vec(void* p, uint4 v) {
  *reinterpret_cast<uint4*>(p) = v;
}

template <int N> __device__ __forceinline__ void unpack(uint4 a, float (&v)[N]);
template <> __device__ __forceinline__ void unpack<4>(uint4 a, float (&v)[4]) {
  v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
  v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
}
template <> __device__ __forceinline__ void unpack<8>(uint4 a, float (&v)[8]) {
  v[0] = bf16_lo(a.x); v[1] = bf16_hi(a.x); v[2] = bf16_lo(a.y); v[3] = bf16_hi(a.y);
  v[4] = bf16_lo(a.z); v[5] = bf16_hi(a.z); v[6] = bf16_lo(a.w); v[7] = bf16_hi(a.w);
}

template <typename T, int N> __device__ __forceinline__ uint4 pack(const float (&v)[N]);
template <> __device__ __forceinline__ uint4 pack<float, 4>(const float (&v)[4]) {
  return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                    __float_as_uint(v[3]));
}
template <> __device__ __forceinline__ uint4 pack<bf16, 8>(const float (&v)[8]) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

// Generic N-element load/store: one 128-bit access when N fills 16 bytes, else scalars.
template <typename T, int N, bool STREAM = true>
__device__ __forceinline__ void load_n(const T* p, float (&v)[N]) {
  if constexpr (N * sizeof(T) == 16) {
    unpack<N>(STREAM ? ld_stream(p) : ld_reuse(p), v);
  } else {
#pragma unroll
    for (int e = 0; e < N; ++e) v[e] = to_f32(p[e]);
  }
}
template <typename T, int N>
__device__ __forceinline__ void store_n(T* p, const float (&v)[N]) {
  if constexpr (N * sizeof(T) == 16) {
    st_vec(p, pack<T, N>(v));
  } else {
#pragma unroll
    for (int e = 0; e < N; ++e) p[e] = from_f32<T>(v[e]);
  }
}
// N elements of T kept in their storage format between load and use (one
// 16-byte register quad on the vector path, N scalars otherwise), so that many
// loads can be in flight without holding their float32 expansion.
template <typename T, int N, bool VECTOR = (N * sizeof(T) == 16)>
struct Packed;
template <typename T, int N>
struct Packed<T, N, true> {
  uint4 r;
  __device__ __forceinline__ void load(const T* p) { r = ld_stream(p); }
  __device__ __forceinline__ void get(float (&v)[N]) const { unpack<N>(r, v); }
};
template <typename T, int N>
struct Packed<T, N, false> {
  T r[N];
  __device__ __forceinline__ void load(const T* p) {
#pragma unroll
    for (int e = 0; e < N; ++e) r[e] = p[e];
  }
  __device__ __forceinline__ void get(float (&v)[N]) const {
#pragma unroll
    for (int e = 0; e < N; ++e) v[e] = to_f32(r[e]);
  }
};

// Round float32 values to T and back (what a store followed by a load would see).
template <typename T, int N>
__device__ __forceinline__ void round_to(float (&v)[N]) {
  if constexpr (sizeof(T) == 2) {
#pragma unroll
    for (int e = 0; e < N; ++e) v[e] = __bfloat162float(__float2bfloat16_rn(v[e]));
  }
}

// Sum over groups of W consecutive lanes (W a power of two <= 32); every lane
// of the group gets the total.  The butterfly order is fixed: deterministic.
template <int W>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o, W);
  return v;
}

// ---------------------------------------------------------------------------
// Row-wise helpers shared by the normalisation kernels.
// ---------------------------------------------------------------------------

// Load VEC weights (as float) for the 16-byte activation vector at index iv.
template <typename W, int VEC>
__device__ __forceinline__ void load_weight(const W* w, int iv, float (&out)[VEC]) {
  if constexpr (sizeof(W) * VEC == 16) {
    unpack<VEC>(ld_reuse(w + (size_t)iv * VEC), out);
  } else {  // float weights with bf16 activations: two 16-byte loads
    float a[4], b[4];
    unpack<4>(ld_reuse(w + (size_t)iv * VEC), a);
    unpack<4>(ld_reuse(w + (size_t)iv * VEC + 4), b);
#pragma unroll
    for (int e = 0; e < 4; ++e) { out[e] = a[e]; out[e + 4] = b[e]; }
  }
}

// Sum of v over the TPR threads of a row group; identical value in every thread.
// TPR <= 32: shuffles.  TPR > 32 (one row per block): shuffles + shared memory
// red[TPR / 32]; safe to call back to back.
// ---------------------------------------------------------------------------
// MXFP8 output (OCP Microscaling Formats (MX) v1.0): E4M3 elements, and one
// E8M0 scale byte (exponent + 127) per block of 32 consecutive values of a row.
// The shared exponent is floor(log2(amax)) - 8, 8 being the exponent of E4M3's
// largest normal (1.75 * 2^8), clamped to E8M0's [-127, 127]; an all-zero
// block takes -127.  Elements are value / 2^exponent rounded to nearest even
// and saturated to +-448 by the hardware conversion.
// ---------------------------------------------------------------------------
constexpr int kMxBlock = 32;

__device__ __forceinline__ int mx_shared_exp(float amax) {
  const int eb = (int)((__float_as_uint(amax) >> 23) & 0xffu);  // 0 for zero and subnormals
  const int se = eb - 127 - 8;
  return eb == 0 ? -127 : (se < -127 ? -127 : se);
}
// 2^-se, exact (se in [-127, 119] gives a normal float).
__device__ __forceinline__ float mx_inv_scale(int se) {
  return __uint_as_float((uint32_t)(127 - se) << 23);
}
// Two E4M3 codes, a in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Quantise this lane's VEC consecutive values o of an MX block that spans
// 32 / VEC consecutive lanes (aligned to 32 / VEC within the warp).  All 32
// lanes of the warp must call it; lanes with active == false contribute
// nothing and store nothing.  q: this lane's first code; sc: the block's scale
// byte, written by the block's first lane (first == true).
template <int VEC>
__device__ __forceinline__ void mx_store(const float (&o)[VEC], bool active, bool first,
                                         uint8_t* q, uint8_t* sc) {
  constexpr int LB = kMxBlock / VEC;
  float a = 0.f;
  if (active) {
#pragma unroll
    for (int e = 0; e < VEC; ++e) a = fmaxf(a, fabsf(o[e]));
  }
#pragma unroll
  for (int m = 1; m < LB; m <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
  if (!active) return;
  const int se = mx_shared_exp(a);
  const float inv = mx_inv_scale(se);
  if constexpr (VEC == 8) {
    uint2 p;
    p.x = e4m3x2(o[0] * inv, o[1] * inv) | (e4m3x2(o[2] * inv, o[3] * inv) << 16);
    p.y = e4m3x2(o[4] * inv, o[5] * inv) | (e4m3x2(o[6] * inv, o[7] * inv) << 16);
    *reinterpret_cast<uint2*>(q) = p;
  } else if constexpr (VEC == 4) {
    *reinterpret_cast<uint32_t*>(q) =
        e4m3x2(o[0] * inv, o[1] * inv) | (e4m3x2(o[2] * inv, o[3] * inv) << 16);
  } else {
#pragma unroll
    for (int e = 0; e < VEC; ++e) q[e] = (uint8_t)(e4m3x2(o[e] * inv, 0.f) & 0xffu);
  }
  if (first) *sc = (uint8_t)(se + 127);
}

struct MxOut {
  uint8_t* q;   // [rows, H] E4M3 codes
  uint8_t* sc;  // [rows, H / 32] E8M0 scales
};

// Compensated (Kahan) running sum.  The element-wise kernels take rows of any
// width, so one thread may add up tens of thousands of terms; a plain float
// sum then drifts by about sqrt(n) ulp (rstd off by 1.3e-5 at 2^24 columns),
// while the compensated sum keeps the error near one ulp whatever n is.
struct KahanSum {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float v) {
    const float y = v - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
  }
};

// Ask the TMA unit to bring `bytes` at p (16-byte aligned, a multiple of 16)
// into L2 ahead of use: no completion to wait for, nothing is written.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Barrier `id` (1..15) over `threads` threads of the block (a multiple of 32).
__device__ __forceinline__ void bar_sync_named(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

template <int TPR>
__device__ __forceinline__ float row_sum(float v, float* red) {
  if constexpr (TPR <= 32) {
    return group_sum<TPR>(v);
  } else {
    v = group_sum<32>(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();  // red[] may still be read from the previous call
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < TPR / 32; ++i) s += red[i];
    return s;
  }
}

// Fixed-order column sums of a [P, ld] float32 buffer: o[j] = (acc ? o[j] : 0)
// + sum_p partial[p * ld + j] for j < ncol, where o is out0 for j < split and
// out1 - split beyond (dW and dB of one [P, 2H] buffer in one launch).  Block (32, kColSumStripes):
// column j = 32 * blockIdx.x + tx; row stripe ty sums p = ty, ty + stripes, ...
// in order (loads unrolled so several are in flight; the additions stay in
// that order), then the stripes are added in order.  Bitwise reproducible.
constexpr int kColSumStripes = 32;

template <int DUMMY = 0>
__global__ void __launch_bounds__(32 * kColSumStripes)
colsum_kernel(const float* __restrict__ partial, int64_t P, int ncol, int ld, float* out0,
              float* out1, int split, int accumulate) {
  __shared__ float s[kColSumStripes][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int j = blockIdx.x * 32 + tx;
  float a = 0.f;
  if (j < ncol) {
#pragma unroll 8
    for (int64_t q = ty; q < P; q += kColSumStripes) a += __ldg(partial + (size_t)q * ld + j);
  }
  s[ty][tx] = a;
  __syncthreads();
  if (ty == 0 && j < ncol) {
    float t = 0.f;
#pragma unroll
    for (int q = 0; q < kColSumStripes; ++q) t += s[q][tx];
    float* o = j < split ? out0 + j : out1 + (j - split);
    *o = accumulate ? *o + t : t;
  }
}

// ---------------------------------------------------------------------------
// TMA bulk copies (global -> shared) completed on an mbarrier.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
// Make the initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Arrive once and announce `bytes` of transaction to come.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes) : "memory");
}
// Plain arrive (release): the caller's earlier shared-memory reads are done.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// Bounded wait for the phase with the given parity: false after `limit` polls
// (each poll may itself suspend the thread for a short, hardware-defined time).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// 1-D bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned)
// from global to this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// Order this thread's earlier generic-proxy accesses to shared memory before
// later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(const void* p) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(smem_addr(p)));
  return r;
}

// Polls of an mbarrier before a kernel gives up (a bulk copy lands in
// microseconds; this bound is far beyond any legitimate wait).
constexpr uint32_t kWaitPolls = 1u << 22;
// Bits of the per-device error word (see gbln_device_error).
constexpr uint32_t kErrWaitTimeout = 1u;   // a bounded wait on an mbarrier ran out
constexpr uint32_t kErrBadPosition = 2u;   // a RoPE position outside [0, max_pos)

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

int sm_count();  // SM count of the current device (cached per device); <= 0 on failure
// Device address of the current device's error word (cached per device); null on failure.
unsigned int* device_error_word();

inline size_t dtype_size(gbln_dtype t) { return t == GBLN_BF16 ? 2 : 4; }
inline bool dtype_ok(int t) { return t == GBLN_F32 || t == GBLN_BF16; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline gbln_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? GBLN_OK : GBLN_ERR_CUDA;
}

inline unsigned grid_for(int64_t work, int block, int64_t cap) {
  int64_t g = (work + block - 1) / block;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (unsigned)g;
}

}  // namespace gbln
