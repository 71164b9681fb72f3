// LayerNorm with fused residual add: forward, backward (dX + per-block dW / dB
// partials) and the fixed-order dW / dB finalize.
//
// Operator: "Fast-LLM: 高效大语言模型训练框架", §三 技术架构, "Transformer Block 结构"
// (normalization LayerNorm / RMSNorm).  Standard form: subtract the row mean,
// divide by sqrt(biased variance + eps), scale by the weight, add the bias.
//
// Same HBM-bound structure as the RMSNorm kernels: each row is read once with
// 128-bit loads into registers; the mean and then the variance of the centred
// values are reduced in fp32 from registers (two passes over registers, one
// over HBM); the weight and bias gradients are accumulated per thread for
// fixed columns over a contiguous chunk of rows (in registers for rows of up
// to 64 vectors, otherwise in shared-memory slots so that 1024 threads stay
// resident per SM), reduced across the block's row groups in a fixed order and
// written as one [dW | dB] partial row per block; a second launch sums the
// partial rows in a fixed order (bitwise reproducible).

#include <atomic>

#include "common.cuh"

namespace gbln {

namespace {

constexpr int kLnWarpBlock = 256;
constexpr int kLnGenericBlock = 256;

// ---------------------------------------------------------------------------
// Forward, vector path (row group of TPR threads per row; BLOCK / TPR rows per block)
// ---------------------------------------------------------------------------
template <typename T, typename W, int TPR, int VPT, int BLOCK, bool RES, bool BIAS>
__global__ void __launch_bounds__(BLOCK)
ln_fwd_vec(const T* x, const T* r, const W* __restrict__ w, const W* __restrict__ b, T* y, T* hout,
           float* __restrict__ mean_out, float* __restrict__ rstd, int64_t rows, int H,
           float inv_H, float eps) {
  constexpr int VEC = VecOf<T>::N;
  constexpr int RPC = BLOCK / TPR;
  __shared__ float red[BLOCK / 32 > 0 ? BLOCK / 32 : 1];
  const int g = threadIdx.x / TPR, l = threadIdx.x % TPR;
  const int64_t row = (int64_t)blockIdx.x * RPC + g;
  if (row >= rows) return;  // uniform per row group; one row per block when TPR > 32
  const int nvec = H / VEC;
  const size_t base = (size_t)row * H;

  uint4 xa[VPT], ra[VPT];
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int iv = l + v * TPR;
    if (iv < nvec) {
      xa[v] = ld_stream(x + base + (size_t)iv * VEC);
      if constexpr (RES) ra[v] = ld_stream(r + base + (size_t)iv * VEC);
    }
  }
  float h[VPT][VEC];
  float s1 = 0.f;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int iv = l + v * TPR;
    if (iv < nvec) {
      unpack<VEC>(xa[v], h[v]);
      if constexpr (RES) {
        float bb[VEC];
        unpack<VEC>(ra[v], bb);
#pragma unroll
        for (int e = 0; e < VEC; ++e) h[v][e] += bb[e];
        round_to<T, VEC>(h[v]);  // the stored h is what gets normalised
        st_vec(hout + base + (size_t)iv * VEC, pack<T, VEC>(h[v]));
      }
#pragma unroll
      for (int e = 0; e < VEC; ++e) s1 += h[v][e];
    }
  }
  const float mu = row_sum<TPR>(s1, red) * inv_H;
  float s2 = 0.f;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int iv = l + v * TPR;
    if (iv < nvec) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        h[v][e] -= mu;
        s2 = fmaf(h[v][e], h[v][e], s2);
      }
    }
  }
  const float rs = rsqrtf(row_sum<TPR>(s2, red) * inv_H + eps);
  if (l == 0) {
    mean_out[row] = mu;
    rstd[row] = rs;
  }
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int iv = l + v * TPR;
    if (iv < nvec) {
      float wv[VEC], o[VEC];
      load_weight<W, VEC>(w, iv, wv);
#pragma unroll
      for (int e = 0; e < VEC; ++e) o[e] = wv[e] * (h[v][e] * rs);
      if constexpr (BIAS) {
        float bv[VEC];
        load_weight<W, VEC>(b, iv, bv);
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] += bv[e];
      }
      st_vec(y + base + (size_t)iv * VEC, pack<T, VEC>(o));
    }
  }
}

// Forward, element-wise path: one block per row, passes over the row.
template <typename T, typename W, bool RES, bool BIAS>
__global__ void __launch_bounds__(kLnGenericBlock)
ln_fwd_generic(const T* x, const T* r, const W* __restrict__ w, const W* __restrict__ b, T* y,
               T* hout, float* __restrict__ mean_out, float* __restrict__ rstd, int64_t rows,
               int H, float inv_H, float eps) {
  __shared__ float red[kLnGenericBlock / 32];
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const size_t base = (size_t)row * H;
    KahanSum s1;
    for (int j = threadIdx.x; j < H; j += kLnGenericBlock) {
      float a = to_f32(x[base + j]);
      if constexpr (RES) {
        const T hv = from_f32<T>(a + to_f32(r[base + j]));
        hout[base + j] = hv;
        a = to_f32(hv);
      }
      s1.add(a);
    }
    const float mu = row_sum<kLnGenericBlock>(s1.s, red) * inv_H;
    KahanSum s2;
    for (int j = threadIdx.x; j < H; j += kLnGenericBlock) {
      const float c = (RES ? to_f32(hout[base + j]) : to_f32(x[base + j])) - mu;  // own write
      s2.add(c * c);
    }
    const float rs = rsqrtf(row_sum<kLnGenericBlock>(s2.s, red) * inv_H + eps);
    if (threadIdx.x == 0) {
      mean_out[row] = mu;
      rstd[row] = rs;
    }
    for (int j = threadIdx.x; j < H; j += kLnGenericBlock) {
      const float c = (RES ? to_f32(hout[base + j]) : to_f32(x[base + j])) - mu;
      float o = to_f32(w[j]) * (c * rs);
      if constexpr (BIAS) o += to_f32(b[j]);
      y[base + j] = from_f32<T>(o);
    }
  }
}

// ---------------------------------------------------------------------------
// Backward, vector path.  gridDim.x = P blocks; block p owns the contiguous
// rows [p*rows/P, (p+1)*rows/P).  Partial row p holds [dW (H) | dB (H)].
// ---------------------------------------------------------------------------
template <typename T, typename W, int TPR, int VPT, int BLOCK, bool DRES>
__global__ void __launch_bounds__(BLOCK)
ln_bwd_vec(const T* dy, const T* dres, const T* h, const W* __restrict__ w,
           const float* __restrict__ mean, const float* __restrict__ rstd, T* dx,
           float* __restrict__ partial, int64_t rows, int H, float inv_H) {
  constexpr int VEC = VecOf<T>::N;
  constexpr int RPC = BLOCK / TPR;
  __shared__ float red[BLOCK / 32 > 0 ? BLOCK / 32 : 1];
  const int g = threadIdx.x / TPR, l = threadIdx.x % TPR;
  const int nvec = H / VEC;
  const int64_t P = gridDim.x, p = blockIdx.x;
  const int64_t r0 = p * rows / P, r1 = (p + 1) * rows / P;

  float accw[VPT][VEC], accb[VPT][VEC];
#pragma unroll
  for (int v = 0; v < VPT; ++v)
#pragma unroll
    for (int e = 0; e < VEC; ++e) { accw[v][e] = 0.f; accb[v][e] = 0.f; }

  for (int64_t row = r0 + g; row < r1; row += RPC) {
    const size_t base = (size_t)row * H;
    uint4 dya[VPT], ha[VPT], dra[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int iv = l + v * TPR;
      if (iv < nvec) {
        dya[v] = ld_stream(dy + base + (size_t)iv * VEC);
        ha[v] = ld_stream(h + base + (size_t)iv * VEC);
        if constexpr (DRES) dra[v] = ld_stream(dres + base + (size_t)iv * VEC);
      }
    }
    const float mu = mean[row], rs = rstd[row];
    float sg = 0.f, sgn = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int iv = l + v * TPR;
      if (iv < nvec) {
        float d[VEC], n[VEC], wv[VEC];
        unpack<VEC>(dya[v], d);
        unpack<VEC>(ha[v], n);
        load_weight<W, VEC>(w, iv, wv);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          n[e] = (n[e] - mu) * rs;
          const float gg = d[e] * wv[e];
          sg += gg;
          sgn = fmaf(gg, n[e], sgn);
          accw[v][e] = fmaf(d[e], n[e], accw[v][e]);
          accb[v][e] += d[e];
        }
      }
    }
    const float mg = row_sum<TPR>(sg, red) * inv_H;
    const float mgn = row_sum<TPR>(sgn, red) * inv_H;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int iv = l + v * TPR;
      if (iv < nvec) {
        float d[VEC], n[VEC], wv[VEC], o[VEC];
        unpack<VEC>(dya[v], d);
        unpack<VEC>(ha[v], n);
        load_weight<W, VEC>(w, iv, wv);
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = rs * (d[e] * wv[e] - mg - ((n[e] - mu) * rs) * mgn);
        if constexpr (DRES) {
          float d2[VEC];
          unpack<VEC>(dra[v], d2);
#pragma unroll
          for (int e = 0; e < VEC; ++e) o[e] += d2[e];
        }
        st_vec(dx + base + (size_t)iv * VEC, pack<T, VEC>(o));
      }
    }
  }

  float* prow = partial + (size_t)p * 2 * H;
  if constexpr (RPC == 1) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int iv = l + v * TPR;
      if (iv < nvec) {
#pragma unroll
        for (int e = 0; e < VEC; e += 4) {
          *reinterpret_cast<float4*>(prow + (size_t)iv * VEC + e) =
              make_float4(accw[v][e], accw[v][e + 1], accw[v][e + 2], accw[v][e + 3]);
          *reinterpret_cast<float4*>(prow + H + (size_t)iv * VEC + e) =
              make_float4(accb[v][e], accb[v][e + 1], accb[v][e + 2], accb[v][e + 3]);
        }
      }
    }
  } else {
    // Fixed-order reduction over the RPC row groups, dW then dB through one buffer.
    __shared__ float sacc[RPC][TPR * VPT * VEC];
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      if (part) __syncthreads();  // the dW sums have been read
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const int iv = l + v * TPR;
        if (iv < nvec) {
#pragma unroll
          for (int e = 0; e < VEC; ++e) sacc[g][iv * VEC + e] = part ? accb[v][e] : accw[v][e];
        }
      }
      __syncthreads();
      for (int j = threadIdx.x; j < H; j += BLOCK) {
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < RPC; ++q) s += sacc[q][j];
        prow[part * H + j] = s;
      }
    }
  }
}

// Backward, vector path for one row per block (TPR = BLOCK > 32): the dW and
// dB accumulators live in shared memory instead of registers, so the kernel
// fits 64 registers and 1024 threads stay resident per SM.  Four consecutive
// columns of a thread form one 16-byte slot, slot k of thread t at acc[k * TPR
// + t] (consecutive threads hit consecutive 16-byte bank groups), so each
// read-modify-write covers four columns.
template <typename T, typename W, int TPR, int VPT, bool DRES>
__global__ void __launch_bounds__(TPR, 1024 / TPR)
ln_bwd_cta(const T* dy, const T* dres, const T* h, const W* __restrict__ w,
           const float* __restrict__ mean, const float* __restrict__ rstd, T* dx,
           float* __restrict__ partial, int64_t rows, int H, float inv_H) {
  constexpr int VEC = VecOf<T>::N;
  constexpr int Q = VEC / 4;         // 16-byte slots per vector
  constexpr int NSL = VPT * Q;       // slots per thread and gradient
  extern __shared__ float4 acc[];    // [2 * NSL][TPR]: dW slots, then dB slots
  __shared__ float red[TPR / 32];
  const int l = threadIdx.x;
  const int nvec = H / VEC;
  const int64_t P = gridDim.x, p = blockIdx.x;
  const int64_t r0 = p * rows / P, r1 = (p + 1) * rows / P;
#pragma unroll
  for (int k = 0; k < 2 * NSL; ++k) acc[k * TPR + l] = make_float4(0.f, 0.f, 0.f, 0.f);

  for (int64_t row = r0; row < r1; ++row) {  // same trip count in every thread
    // thread 0 asks for the block's next row in L2 while this one is processed
    if (l == 0 && row + 1 < r1) {
      const size_t nb = (size_t)(row + 1) * H;
      const uint32_t rb = (uint32_t)(H * sizeof(T));
      prefetch_l2(dy + nb, rb);
      prefetch_l2(h + nb, rb);
      if constexpr (DRES) prefetch_l2(dres + nb, rb);
    }
    const size_t base = (size_t)row * H;
    uint4 dya[VPT], ha[VPT], dra[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int iv = l + v * TPR;
      if (iv < nvec) {
        dya[v] = ld_stream(dy + base + (size_t)iv * VEC);
        ha[v] = ld_stream(h + base + (size_t)iv * VEC);
        if constexpr (DRES) dra[v] = ld_stream(dres + base + (size_t)iv * VEC);
      }
    }
    const float mu = mean[row], rs = rstd[row];
    float sg = 0.f, sgn = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int iv = l + v * TPR;
      if (iv < nvec) {
        float d[VEC], n[VEC], wv[VEC];
        unpack<VEC>(dya[v], d);
        unpack<VEC>(ha[v], n);
        load_weight<W, VEC>(w, iv, wv);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          n[e] = (n[e] - mu) * rs;
          const float gg = d[e] * wv[e];
          sg += gg;
          sgn = fmaf(gg, n[e], sgn);
        }
#pragma unroll
        for (int q = 0; q < Q; ++q) {
          float4* aw = acc + (v * Q + q) * TPR + l;
          float4* ab = acc + (NSL + v * Q + q) * TPR + l;
          float4 a = *aw, b = *ab;
          a.x = fmaf(d[4 * q], n[4 * q], a.x);
          a.y = fmaf(d[4 * q + 1], n[4 * q + 1], a.y);
          a.z = fmaf(d[4 * q + 2], n[4 * q + 2], a.z);
          a.w = fmaf(d[4 * q + 3], n[4 * q + 3], a.w);
          b.x += d[4 * q]; b.y += d[4 * q + 1]; b.z += d[4 * q + 2]; b.w += d[4 * q + 3];
          *aw = a;
          *ab = b;
        }
      }
    }
    const float mg = row_sum<TPR>(sg, red) * inv_H;
    const float mgn = row_sum<TPR>(sgn, red) * inv_H;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int iv = l + v * TPR;
      if (iv < nvec) {
        float d[VEC], n[VEC], wv[VEC], o[VEC];
        unpack<VEC>(dya[v], d);
        unpack<VEC>(ha[v], n);
        load_weight<W, VEC>(w, iv, wv);
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = rs * (d[e] * wv[e] - mg - ((n[e] - mu) * rs) * mgn);
        if constexpr (DRES) {
          float d2[VEC];
          unpack<VEC>(dra[v], d2);
#pragma unroll
          for (int e = 0; e < VEC; ++e) o[e] += d2[e];
        }
        st_vec(dx + base + (size_t)iv * VEC, pack<T, VEC>(o));
      }
    }
  }
  float* prow = partial + (size_t)p * 2 * H;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int iv = l + v * TPR;
    if (iv < nvec) {
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        *reinterpret_cast<float4*>(prow + iv * VEC + 4 * q) = acc[(v * Q + q) * TPR + l];
        *reinterpret_cast<float4*>(prow + H + iv * VEC + 4 * q) = acc[(NSL + v * Q + q) * TPR + l];
      }
    }
  }
}

// Backward for rows of 65..128 vectors: kLnGroups row groups of 64 threads per
// block, each with its own shared-memory accumulators (layout as ln_bwd_cta) and
// its own named barrier for the row sums, so groups walk their rows (r0 + g,
// r0 + g + kLnGroups, ...) independently.  At 64 registers 1024 threads stay
// resident per SM while the block count, and with it the number of partial
// rows, stays at 4 per SM.  The groups' accumulators are summed in a fixed
// order at the end.
constexpr int kLnGroups = 4;
constexpr int kLnGroupThreads = 64;

template <typename T, typename W, int VPT, bool DRES>
__global__ void __launch_bounds__(kLnGroups * kLnGroupThreads, 1024 / (kLnGroups * kLnGroupThreads))
ln_bwd_grp(const T* dy, const T* dres, const T* h, const W* __restrict__ w,
           const float* __restrict__ mean, const float* __restrict__ rstd, T* dx,
           float* __restrict__ partial, int64_t rows, int H, float inv_H) {
  constexpr int TPR = kLnGroupThreads;
  constexpr int VEC = VecOf<T>::N;
  constexpr int Q = VEC / 4;
  constexpr int NSL = VPT * Q;
  extern __shared__ float4 acc_all[];  // [kLnGroups][2 * NSL][TPR]
  __shared__ float2 red2[kLnGroups][2][TPR / 32];
  const int g = threadIdx.x / TPR, l = threadIdx.x % TPR, lane = threadIdx.x % 32;
  float4* acc = acc_all + (size_t)g * 2 * NSL * TPR;
  const int nvec = H / VEC;
  const int64_t P = gridDim.x, p = blockIdx.x;
  const int64_t r0 = p * rows / P, r1 = (p + 1) * rows / P;
#pragma unroll
  for (int k = 0; k < 2 * NSL; ++k) acc[k * TPR + l] = make_float4(0.f, 0.f, 0.f, 0.f);

  int par = 0;
  for (int64_t row = r0 + g; row < r1; row += kLnGroups) {
    const size_t base = (size_t)row * H;
    uint4 dya[VPT], ha[VPT], dra[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int iv = l + v * TPR;
      if (iv < nvec) {
        dya[v] = ld_stream(dy + base + (size_t)iv * VEC);
        ha[v] = ld_stream(h + base + (size_t)iv * VEC);
        if constexpr (DRES) dra[v] = ld_stream(dres + base + (size_t)iv * VEC);
      }
    }
    const float mu = mean[row], rs = rstd[row];
    float sg = 0.f, sgn = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int iv = l + v * TPR;
      if (iv < nvec) {
        float d[VEC], n[VEC], wv[VEC];
        unpack<VEC>(dya[v], d);
        unpack<VEC>(ha[v], n);
        load_weight<W, VEC>(w, iv, wv);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          n[e] = (n[e] - mu) * rs;
          const float gg = d[e] * wv[e];
          sg += gg;
          sgn = fmaf(gg, n[e], sgn);
        }
#pragma unroll
        for (int q = 0; q < Q; ++q) {
          float4* aw = acc + (v * Q + q) * TPR + l;
          float4* ab = acc + (NSL + v * Q + q) * TPR + l;
          float4 a = *aw, b = *ab;
          a.x = fmaf(d[4 * q], n[4 * q], a.x);
          a.y = fmaf(d[4 * q + 1], n[4 * q + 1], a.y);
          a.z = fmaf(d[4 * q + 2], n[4 * q + 2], a.z);
          a.w = fmaf(d[4 * q + 3], n[4 * q + 3], a.w);
          b.x += d[4 * q]; b.y += d[4 * q + 1]; b.z += d[4 * q + 2]; b.w += d[4 * q + 3];
          *aw = a;
          *ab = b;
        }
      }
    }
    // Row sums over the group's two warps.  red2 is double-buffered by row
    // parity: a thread can only write a buffer again after the group's next
    // barrier, which every thread reaches after reading this one.
    sg = group_sum<32>(sg);
    sgn = group_sum<32>(sgn);
    if (lane == 0) red2[g][par][l / 32] = make_float2(sg, sgn);
    bar_sync_named(1 + g, TPR);
    float2 ssum = red2[g][par][0];
#pragma unroll
    for (int k = 1; k < TPR / 32; ++k) {
      ssum.x += red2[g][par][k].x;
      ssum.y += red2[g][par][k].y;
    }
    par ^= 1;
    const float mg = ssum.x * inv_H, mgn = ssum.y * inv_H;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int iv = l + v * TPR;
      if (iv < nvec) {
        float d[VEC], n[VEC], wv[VEC], o[VEC];
        unpack<VEC>(dya[v], d);
        unpack<VEC>(ha[v], n);
        load_weight<W, VEC>(w, iv, wv);
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = rs * (d[e] * wv[e] - mg - ((n[e] - mu) * rs) * mgn);
        if constexpr (DRES) {
          float d2[VEC];
          unpack<VEC>(dra[v], d2);
#pragma unroll
          for (int e = 0; e < VEC; ++e) o[e] += d2[e];
        }
        st_vec(dx + base + (size_t)iv * VEC, pack<T, VEC>(o));
      }
    }
  }
  __syncthreads();
  // Fixed-order sum over the groups: column j is component j % 4 of slot
  // (v * Q + (j % VEC) / 4) of thread l, where j / VEC = l + v * TPR.
  float* prow = partial + (size_t)p * 2 * H;
  const float* af = reinterpret_cast<const float*>(acc_all);
  for (int j = threadIdx.x; j < H; j += kLnGroups * TPR) {
    const int iv = j / VEC, e = j % VEC;
    const int lt = iv % TPR, v = iv / TPR;
    const size_t sw = ((size_t)(v * Q + e / 4) * TPR + lt) * 4 + e % 4;
    const size_t sb = ((size_t)(NSL + v * Q + e / 4) * TPR + lt) * 4 + e % 4;
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int q = 0; q < kLnGroups; ++q) {
      a += af[(size_t)q * 2 * NSL * TPR * 4 + sw];
      b += af[(size_t)q * 2 * NSL * TPR * 4 + sb];
    }
    prow[j] = a;
    prow[H + j] = b;
  }
}

// Backward, element-wise path: P blocks over contiguous row chunks, one row at
// a time; thread t owns columns t, t + 256, ... of the partial row.
template <typename T, typename W, bool DRES>
__global__ void __launch_bounds__(kLnGenericBlock)
ln_bwd_generic(const T* dy, const T* dres, const T* h, const W* __restrict__ w,
               const float* __restrict__ mean, const float* __restrict__ rstd, T* dx,
               float* __restrict__ partial, int64_t rows, int H, float inv_H) {
  __shared__ float red[kLnGenericBlock / 32];
  const int64_t P = gridDim.x, p = blockIdx.x;
  const int64_t r0 = p * rows / P, r1 = (p + 1) * rows / P;
  float* prow = partial + (size_t)p * 2 * H;
  for (int j = threadIdx.x; j < 2 * H; j += kLnGenericBlock) prow[j] = 0.f;
  for (int64_t row = r0; row < r1; ++row) {
    const size_t base = (size_t)row * H;
    const float mu = mean[row], rs = rstd[row];
    KahanSum sg, sgn;
    for (int j = threadIdx.x; j < H; j += kLnGenericBlock) {
      const float gg = to_f32(dy[base + j]) * to_f32(w[j]);
      sg.add(gg);
      sgn.add(gg * ((to_f32(h[base + j]) - mu) * rs));
    }
    const float mg = row_sum<kLnGenericBlock>(sg.s, red) * inv_H;
    const float mgn = row_sum<kLnGenericBlock>(sgn.s, red) * inv_H;
    for (int j = threadIdx.x; j < H; j += kLnGenericBlock) {
      const float d = to_f32(dy[base + j]);
      const float n = (to_f32(h[base + j]) - mu) * rs;
      float o = rs * (d * to_f32(w[j]) - mg - n * mgn);
      if constexpr (DRES) o += to_f32(dres[base + j]);
      prow[j] = fmaf(d, n, prow[j]);
      prow[H + j] += d;
      dx[base + j] = from_f32<T>(o);
    }
  }
}

// ---------------------------------------------------------------------------
// Geometry (shared by forward, backward and num_partials)
// ---------------------------------------------------------------------------
struct LnGeometry {
  bool vec;
  bool smem_acc;  // backward with shared-memory accumulators (ln_bwd_cta / ln_bwd_grp)
  bool grouped;   // backward: ln_bwd_grp (several 64-thread row groups per block)
  int tpr, vpt, block, rpc, bps;
};

// Forward: up to 4 vectors per thread (~50 registers).  Backward: up to 2, since
// each thread also carries dW and dB accumulators for its columns (~100
// registers at 2 vectors, 150-165 at 4, which would leave too few resident
// blocks for the persistent grid).
LnGeometry ln_geometry(int64_t H, size_t io_size, bool bwd) {
  LnGeometry g{};
  const int max_vpt = bwd ? 2 : 4;
  const int64_t row_bytes = H * (int64_t)io_size;
  const int64_t nvec = row_bytes / 16;
  if (row_bytes % 16 != 0 || nvec > 512LL * max_vpt) {
    g.vec = false; g.tpr = kLnGenericBlock; g.vpt = 0; g.block = kLnGenericBlock; g.rpc = 1; g.bps = 4;
    return g;
  }
  g.vec = true;
  // Backward (2 vectors per thread): rows of up to 64 vectors take a warp per
  // row with register accumulators; rows of up to 128 a 64-thread row group,
  // four groups per block (ln_bwd_grp); wider rows one block per row (ln_bwd_cta);
  // both keep the accumulators in shared memory (at most 64 registers, 1024
  // threads per SM).  Blocks per SM set P, the number of [dW | dB] partial rows.
  const int64_t warp_limit = bwd ? 64 : 32LL * max_vpt;
  if (nvec <= warp_limit) {
    g.tpr = 32;
    g.vpt = nvec <= 32 ? 1 : (nvec <= 64 ? 2 : 4);
    g.block = kLnWarpBlock;
    g.rpc = kLnWarpBlock / 32;
    g.bps = 2;
  } else {
    int tpr = 64;
    while ((int64_t)tpr * max_vpt < nvec) tpr *= 2;  // <= 512
    g.tpr = tpr;
    g.vpt = max_vpt;
    g.block = tpr;
    g.rpc = 1;
    g.smem_acc = bwd;
    g.bps = 1024 / tpr;
    if (bwd && tpr == kLnGroupThreads) {  // 65..128 vectors: grouped blocks
      g.grouped = true;
      g.block = kLnGroups * kLnGroupThreads;
      g.rpc = kLnGroups;
      g.bps = 1024 / g.block;
    }
  }
  return g;
}

int64_t ln_partials_for(int64_t T, const LnGeometry& g, int sms) {
  if (T <= 0) return 0;
  int64_t P = (int64_t)sms * g.bps;
  const int64_t groups = (T + g.rpc - 1) / g.rpc;
  if (P > groups) P = groups;
  return P < 1 ? 1 : P;
}

template <typename T, typename W, int TPR, int VPT, int BLOCK>
void ln_fwd_vec_launch(bool res, bool bias, const void* x, const void* r, const void* w,
                       const void* b, void* y, void* hout, float* mean, float* rstd, int64_t rows,
                       int H, float inv_H, float eps, cudaStream_t s) {
  const unsigned grid = (unsigned)((rows + BLOCK / TPR - 1) / (BLOCK / TPR));
#define GBLN_LN_FWD(R, B)                                                                    \
  ln_fwd_vec<T, W, TPR, VPT, BLOCK, R, B><<<grid, BLOCK, 0, s>>>(                            \
      (const T*)x, (const T*)r, (const W*)w, (const W*)b, (T*)y, (T*)hout, mean, rstd, rows, \
      H, inv_H, eps)
  if (res) { if (bias) GBLN_LN_FWD(true, true); else GBLN_LN_FWD(true, false); }
  else { if (bias) GBLN_LN_FWD(false, true); else GBLN_LN_FWD(false, false); }
#undef GBLN_LN_FWD
}

template <typename T, typename W>
gbln_status ln_fwd_typed(const void* x, const void* r, const void* w, const void* b, void* y,
                         void* hout, float* mean, float* rstd, int64_t rows, int64_t H, float eps,
                         cudaStream_t s) {
  const bool res = r != nullptr, bias = b != nullptr;
  const LnGeometry g = ln_geometry(H, sizeof(T), false);
  const bool vec = g.vec && aligned16(x) && aligned16(w) && aligned16(y) &&
                   (!bias || aligned16(b)) && (!res || (aligned16(r) && aligned16(hout)));
  const float inv_H = 1.0f / (float)H;
  const int hh = (int)H;
  if (!vec) {
    const unsigned grid = (unsigned)(rows < 65535LL * 32 ? rows : 65535LL * 32);
#define GBLN_LN_FWDG(R, B)                                                                   \
  ln_fwd_generic<T, W, R, B><<<grid, kLnGenericBlock, 0, s>>>(                               \
      (const T*)x, (const T*)r, (const W*)w, (const W*)b, (T*)y, (T*)hout, mean, rstd, rows, \
      hh, inv_H, eps)
    if (res) { if (bias) GBLN_LN_FWDG(true, true); else GBLN_LN_FWDG(true, false); }
    else { if (bias) GBLN_LN_FWDG(false, true); else GBLN_LN_FWDG(false, false); }
#undef GBLN_LN_FWDG
    return launch_status();
  }
  if (g.tpr == 32) {
    if (g.vpt == 1) ln_fwd_vec_launch<T, W, 32, 1, kLnWarpBlock>(res, bias, x, r, w, b, y, hout, mean, rstd, rows, hh, inv_H, eps, s);
    else if (g.vpt == 2) ln_fwd_vec_launch<T, W, 32, 2, kLnWarpBlock>(res, bias, x, r, w, b, y, hout, mean, rstd, rows, hh, inv_H, eps, s);
    else ln_fwd_vec_launch<T, W, 32, 4, kLnWarpBlock>(res, bias, x, r, w, b, y, hout, mean, rstd, rows, hh, inv_H, eps, s);
  } else {
    switch (g.tpr) {
      case 64: ln_fwd_vec_launch<T, W, 64, 4, 64>(res, bias, x, r, w, b, y, hout, mean, rstd, rows, hh, inv_H, eps, s); break;
      case 128: ln_fwd_vec_launch<T, W, 128, 4, 128>(res, bias, x, r, w, b, y, hout, mean, rstd, rows, hh, inv_H, eps, s); break;
      case 256: ln_fwd_vec_launch<T, W, 256, 4, 256>(res, bias, x, r, w, b, y, hout, mean, rstd, rows, hh, inv_H, eps, s); break;
      default: ln_fwd_vec_launch<T, W, 512, 4, 512>(res, bias, x, r, w, b, y, hout, mean, rstd, rows, hh, inv_H, eps, s); break;
    }
  }
  return launch_status();
}

template <typename T, typename W, int TPR, int VPT, int BLOCK>
void ln_bwd_vec_launch(bool dres, unsigned P, const void* dy, const void* dr, const void* h,
                       const void* w, const float* mean, const float* rstd, void* dx,
                       float* partial, int64_t rows, int H, float inv_H, cudaStream_t s) {
  if (dres)
    ln_bwd_vec<T, W, TPR, VPT, BLOCK, true><<<P, BLOCK, 0, s>>>(
        (const T*)dy, (const T*)dr, (const T*)h, (const W*)w, mean, rstd, (T*)dx, partial, rows, H, inv_H);
  else
    ln_bwd_vec<T, W, TPR, VPT, BLOCK, false><<<P, BLOCK, 0, s>>>(
        (const T*)dy, nullptr, (const T*)h, (const W*)w, mean, rstd, (T*)dx, partial, rows, H, inv_H);
}

template <typename T, typename W, int TPR, int VPT>
gbln_status ln_bwd_cta_launch(bool dres, unsigned P, const void* dy, const void* dr, const void* h,
                              const void* w, const float* mean, const float* rstd, void* dx,
                              float* partial, int64_t rows, int H, float inv_H, cudaStream_t s) {
  constexpr int VEC = VecOf<T>::N;
  const size_t smem = (size_t)2 * VPT * VEC * TPR * sizeof(float);
  static std::atomic<uint64_t> attr_done{0};  // one bit per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return GBLN_ERR_CUDA; }
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    if (cudaFuncSetAttribute(ln_bwd_cta<T, W, TPR, VPT, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(ln_bwd_cta<T, W, TPR, VPT, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
      cudaGetLastError();
      return GBLN_ERR_CUDA;
    }
    attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  if (dres)
    ln_bwd_cta<T, W, TPR, VPT, true><<<P, TPR, smem, s>>>(
        (const T*)dy, (const T*)dr, (const T*)h, (const W*)w, mean, rstd, (T*)dx, partial, rows, H, inv_H);
  else
    ln_bwd_cta<T, W, TPR, VPT, false><<<P, TPR, smem, s>>>(
        (const T*)dy, nullptr, (const T*)h, (const W*)w, mean, rstd, (T*)dx, partial, rows, H, inv_H);
  return GBLN_OK;
}

template <typename T, typename W>
gbln_status ln_bwd_grp_launch(bool dres, unsigned P, const void* dy, const void* dr, const void* h,
                              const void* w, const float* mean, const float* rstd, void* dx,
                              float* partial, int64_t rows, int H, float inv_H, cudaStream_t s) {
  constexpr int VPT = 2;
  const size_t smem = (size_t)kLnGroups * 2 * VPT * VecOf<T>::N * kLnGroupThreads * sizeof(float);
  static std::atomic<uint64_t> attr_done{0};  // one bit per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return GBLN_ERR_CUDA; }
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    if (cudaFuncSetAttribute(ln_bwd_grp<T, W, VPT, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(ln_bwd_grp<T, W, VPT, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
      cudaGetLastError();
      return GBLN_ERR_CUDA;
    }
    attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  constexpr int B = kLnGroups * kLnGroupThreads;
  if (dres)
    ln_bwd_grp<T, W, VPT, true><<<P, B, smem, s>>>(
        (const T*)dy, (const T*)dr, (const T*)h, (const W*)w, mean, rstd, (T*)dx, partial, rows, H, inv_H);
  else
    ln_bwd_grp<T, W, VPT, false><<<P, B, smem, s>>>(
        (const T*)dy, nullptr, (const T*)h, (const W*)w, mean, rstd, (T*)dx, partial, rows, H, inv_H);
  return GBLN_OK;
}

template <typename T, typename W>
gbln_status ln_bwd_typed(const void* dy, const void* dr, const void* h, const void* w,
                         const float* mean, const float* rstd, void* dx, float* partial, int64_t P,
                         int64_t rows, int64_t H, cudaStream_t s) {
  const bool dres = dr != nullptr;
  const LnGeometry g = ln_geometry(H, sizeof(T), true);
  const bool vec = g.vec && aligned16(dy) && aligned16(h) && aligned16(w) && aligned16(dx) &&
                   aligned16(partial) && (!dres || aligned16(dr));
  const float inv_H = 1.0f / (float)H;
  const int hh = (int)H;
  const unsigned grid = (unsigned)P;
  if (!vec) {
    if (dres)
      ln_bwd_generic<T, W, true><<<grid, kLnGenericBlock, 0, s>>>(
          (const T*)dy, (const T*)dr, (const T*)h, (const W*)w, mean, rstd, (T*)dx, partial, rows, hh, inv_H);
    else
      ln_bwd_generic<T, W, false><<<grid, kLnGenericBlock, 0, s>>>(
          (const T*)dy, nullptr, (const T*)h, (const W*)w, mean, rstd, (T*)dx, partial, rows, hh, inv_H);
    return launch_status();
  }
  if (g.tpr == 32) {
    if (g.vpt == 1) ln_bwd_vec_launch<T, W, 32, 1, kLnWarpBlock>(dres, grid, dy, dr, h, w, mean, rstd, dx, partial, rows, hh, inv_H, s);
    else ln_bwd_vec_launch<T, W, 32, 2, kLnWarpBlock>(dres, grid, dy, dr, h, w, mean, rstd, dx, partial, rows, hh, inv_H, s);
  } else if (g.grouped) {
    const gbln_status st = ln_bwd_grp_launch<T, W>(dres, grid, dy, dr, h, w, mean, rstd, dx, partial, rows, hh, inv_H, s);
    if (st != GBLN_OK) return st;
  } else {
    gbln_status st = GBLN_OK;
    switch (g.tpr) {
      case 128: st = ln_bwd_cta_launch<T, W, 128, 2>(dres, grid, dy, dr, h, w, mean, rstd, dx, partial, rows, hh, inv_H, s); break;
      case 256: st = ln_bwd_cta_launch<T, W, 256, 2>(dres, grid, dy, dr, h, w, mean, rstd, dx, partial, rows, hh, inv_H, s); break;
      default: st = ln_bwd_cta_launch<T, W, 512, 2>(dres, grid, dy, dr, h, w, mean, rstd, dx, partial, rows, hh, inv_H, s); break;
    }
    if (st != GBLN_OK) return st;
  }
  return launch_status();
}

constexpr int64_t kMaxH = 1 << 24;
constexpr int64_t kMaxRows = (1LL << 31) - 1;

bool dtypes_ok(int io, int wt) {
  return (io == GBLN_F32 && wt == GBLN_F32) || (io == GBLN_BF16 && (wt == GBLN_BF16 || wt == GBLN_F32));
}

}  // namespace

}  // namespace gbln

using namespace gbln;

extern "C" gbln_status gbln_layernorm_fwd(const void* x, const void* residual, const void* weight,
                                          const void* bias, void* y, void* residual_out,
                                          float* mean, float* rstd, int64_t T, int64_t H,
                                          float eps, gbln_dtype io, gbln_dtype wt,
                                          gbln_stream_t stream) {
  if (!dtype_ok(io) || !dtype_ok(wt)) return GBLN_ERR_INVALID_ARG;
  if (T < 0 || T > kMaxRows || H <= 0 || H > kMaxH) return GBLN_ERR_INVALID_ARG;
  if (!(eps >= 0.0f && eps <= 3.4028235e38f)) return GBLN_ERR_INVALID_ARG;  // also rejects NaN
  if (!dtypes_ok(io, wt)) return GBLN_ERR_UNSUPPORTED;
  if (T == 0) return GBLN_OK;  // nothing is read or written: pointers are not examined
  if (!x || !weight || !y || !mean || !rstd) return GBLN_ERR_INVALID_ARG;
  if (residual && !residual_out) return GBLN_ERR_INVALID_ARG;
  const void* r = residual;
  void* ho = residual ? residual_out : nullptr;
  cudaStream_t s = (cudaStream_t)stream;
  if (io == GBLN_F32) return ln_fwd_typed<float, float>(x, r, weight, bias, y, ho, mean, rstd, T, H, eps, s);
  if (wt == GBLN_BF16) return ln_fwd_typed<bf16, bf16>(x, r, weight, bias, y, ho, mean, rstd, T, H, eps, s);
  return ln_fwd_typed<bf16, float>(x, r, weight, bias, y, ho, mean, rstd, T, H, eps, s);
}

extern "C" int64_t gbln_layernorm_bwd_num_partials(int64_t T, int64_t H, gbln_dtype io) {
  if (!dtype_ok(io) || T < 0 || T > kMaxRows || H <= 0 || H > kMaxH) return -1;
  if (T == 0) return 0;
  const int sms = sm_count();
  if (sms <= 0) return -1;
  return ln_partials_for(T, ln_geometry(H, dtype_size(io), true), sms);
}

extern "C" gbln_status gbln_layernorm_bwd(const void* dy, const void* dresidual_out,
                                          const void* h, const void* weight, const float* mean,
                                          const float* rstd, void* dx, float* dwdb_partial,
                                          int64_t P_cap, int64_t T, int64_t H, gbln_dtype io,
                                          gbln_dtype wt, gbln_stream_t stream) {
  if (!dtype_ok(io) || !dtype_ok(wt)) return GBLN_ERR_INVALID_ARG;
  if (T < 0 || T > kMaxRows || H <= 0 || H > kMaxH || P_cap < 0) return GBLN_ERR_INVALID_ARG;
  if (!dtypes_ok(io, wt)) return GBLN_ERR_UNSUPPORTED;
  if (T == 0) return GBLN_OK;  // nothing is read or written: pointers are not examined
  if (!dy || !h || !weight || !mean || !rstd || !dx || !dwdb_partial) return GBLN_ERR_INVALID_ARG;
  const int sms = sm_count();
  if (sms <= 0) return GBLN_ERR_CUDA;
  const int64_t P = ln_partials_for(T, ln_geometry(H, dtype_size(io), true), sms);
  if (P_cap < P) return GBLN_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  if (io == GBLN_F32)
    return ln_bwd_typed<float, float>(dy, dresidual_out, h, weight, mean, rstd, dx, dwdb_partial, P, T, H, s);
  if (wt == GBLN_BF16)
    return ln_bwd_typed<bf16, bf16>(dy, dresidual_out, h, weight, mean, rstd, dx, dwdb_partial, P, T, H, s);
  return ln_bwd_typed<bf16, float>(dy, dresidual_out, h, weight, mean, rstd, dx, dwdb_partial, P, T, H, s);
}

extern "C" gbln_status gbln_layernorm_dwdb_finalize(const float* dwdb_partial, int64_t P,
                                                    int64_t H, float* dw, float* db,
                                                    int accumulate, gbln_stream_t stream) {
  if (P < 0 || H <= 0 || H > kMaxH) return GBLN_ERR_INVALID_ARG;
  if (!dw || !db || (P > 0 && !dwdb_partial)) return GBLN_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const int acc = accumulate ? 1 : 0;
  // one launch over the 2H columns [dW | dB] of the partial rows
  colsum_kernel<<<(unsigned)((2 * H + 31) / 32), 32 * kColSumStripes, 0, s>>>(
      dwdb_partial, P, (int)(2 * H), (int)(2 * H), dw, db, (int)H, acc);
  return launch_status();
}
