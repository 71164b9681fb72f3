// RMSNorm with fused residual add: forward, backward (dX + per-block dW
// partials) and the fixed-order dW finalize.
//
// Operator: "Fast-LLM: 高效大语言模型训练框架", §三 技术架构, "Transformer Block 结构"
// (normalization RMSNorm) and "训练配置示例" (rms_norm, epsilon); fused form as in
// "LLaMA-Factory Kernels 系统" (fused RMSNorm) and "Kernels（自定义内核）" §Liger.
//
// HBM-bound design: each row is read once with 128-bit loads into registers,
// reduced in fp32 with warp shuffles (plus shared memory across warps for wide
// rows), and written once.  The weight gradient is accumulated per thread over
// a contiguous chunk of rows (in registers, or for rows of 65..128 vectors in
// shared-memory slots of 64-thread row groups), reduced across the block's row
// groups in a fixed order and written as one partial row per block; a second
// launch sums the partial rows in a fixed order.  No atomics: bitwise
// reproducible for a fixed shape and SM count.  The forward can also deliver y
// as MXFP8 (E4M3 codes and one E8M0 scale per 32 values) for the next GEMM.

#include <atomic>

#include "common.cuh"

namespace gbln {

namespace {

constexpr int kWarpBlock = 256;      // block of the warp-per-row regime
constexpr int kMaxVecPerRow = 2048;  // 512 threads x 4 vectors: register-resident limit
constexpr int kGenericBlock = 256;

// ---------------------------------------------------------------------------
// Forward, vector path.  A row group of TPR threads owns one row; thread l owns
// the 16-byte vectors l, l + TPR, ..., (VPT of them).  BLOCK / TPR rows per block.
// ---------------------------------------------------------------------------
// MX: y is also written as MXFP8 (mx.q, mx.sc); y itself may then be null.
template <typename T, typename W, int TPR, int VPT, int BLOCK, bool RES, bool MX = false>
__global__ void __launch_bounds__(BLOCK)
rms_fwd_vec(const T* x, const T* r, const W* __restrict__ w, T* y, T* hout,
            float* __restrict__ rstd, int64_t rows, int H, float inv_H, float eps, MxOut mx = {}) {
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
  float ss = 0.f;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int iv = l + v * TPR;
    if (iv < nvec) {
      unpack<VEC>(xa[v], h[v]);
      if constexpr (RES) {
        float b[VEC];
        unpack<VEC>(ra[v], b);
#pragma unroll
        for (int e = 0; e < VEC; ++e) h[v][e] += b[e];
        round_to<T, VEC>(h[v]);  // the stored h is what gets normalised
        st_vec(hout + base + (size_t)iv * VEC, pack<T, VEC>(h[v]));
      }
#pragma unroll
      for (int e = 0; e < VEC; ++e) ss = fmaf(h[v][e], h[v][e], ss);
    }
  }
  ss = row_sum<TPR>(ss, red);
  const float rs = rsqrtf(ss * inv_H + eps);
  if (l == 0) rstd[row] = rs;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int iv = l + v * TPR;
    float o[VEC];
    if (iv < nvec) {
      float wv[VEC];
      load_weight<W, VEC>(w, iv, wv);
#pragma unroll
      for (int e = 0; e < VEC; ++e) o[e] = wv[e] * (h[v][e] * rs);
      if (!MX || y) st_vec(y + base + (size_t)iv * VEC, pack<T, VEC>(o));
    }
    if constexpr (MX) {
      // an MX block is 32 / VEC consecutive vectors: lanes l .. l + 32 / VEC - 1
      constexpr int LB = kMxBlock / VEC;
      mx_store<VEC>(o, iv < nvec, iv % LB == 0, mx.q + base + (size_t)iv * VEC,
                    mx.sc + (size_t)row * (H / kMxBlock) + iv / LB);
    }
  }
}

// ---------------------------------------------------------------------------
// Forward, element-wise path (any alignment, any H): one block per row, two
// passes over the row; the second re-reads h (cache hit for all but huge H).
// ---------------------------------------------------------------------------
template <typename T, typename W, bool RES, bool MX = false>
__global__ void __launch_bounds__(kGenericBlock)
rms_fwd_generic(const T* x, const T* r, const W* __restrict__ w, T* y, T* hout,
                float* __restrict__ rstd, int64_t rows, int H, float inv_H, float eps, MxOut mx = {}) {
  __shared__ float red[kGenericBlock / 32];
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const size_t base = (size_t)row * H;
    KahanSum ks;
    for (int j = threadIdx.x; j < H; j += kGenericBlock) {
      float a = to_f32(x[base + j]);
      if constexpr (RES) {
        T hv = from_f32<T>(a + to_f32(r[base + j]));
        hout[base + j] = hv;
        a = to_f32(hv);
      }
      ks.add(a * a);
    }
    const float ss = row_sum<kGenericBlock>(ks.s, red);
    const float rs = rsqrtf(ss * inv_H + eps);
    if (threadIdx.x == 0) rstd[row] = rs;
    // With MX, H is a multiple of 32, so each warp's pass covers one MX block.
    for (int j = threadIdx.x; j < H; j += kGenericBlock) {
      const float a = RES ? to_f32(hout[base + j]) : to_f32(x[base + j]);  // own write
      float o[1] = {to_f32(w[j]) * (a * rs)};
      if (!MX || y) y[base + j] = from_f32<T>(o[0]);
      if constexpr (MX)
        mx_store<1>(o, true, j % kMxBlock == 0, mx.q + base + j, mx.sc + (size_t)row * (H / kMxBlock) + j / kMxBlock);
    }
  }
}

// ---------------------------------------------------------------------------
// Backward, vector path.  gridDim.x = P blocks; block p owns the contiguous
// rows [p*rows/P, (p+1)*rows/P).  Row group g takes rows r0+g, r0+g+RPC, ...
// ---------------------------------------------------------------------------
template <typename T, typename W, int TPR, int VPT, int BLOCK, bool DRES>
__global__ void __launch_bounds__(BLOCK)
rms_bwd_vec(const T* dy, const T* dres, const T* h, const W* __restrict__ w,
            const float* __restrict__ rstd, T* dx, float* __restrict__ partial,
            int64_t rows, int H, float inv_H) {
  constexpr int VEC = VecOf<T>::N;
  constexpr int RPC = BLOCK / TPR;
  __shared__ float red[BLOCK / 32 > 0 ? BLOCK / 32 : 1];
  const int g = threadIdx.x / TPR, l = threadIdx.x % TPR;
  const int nvec = H / VEC;
  const int64_t P = gridDim.x, p = blockIdx.x;
  const int64_t r0 = p * rows / P, r1 = (p + 1) * rows / P;

  float acc[VPT][VEC];
#pragma unroll
  for (int v = 0; v < VPT; ++v)
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[v][e] = 0.f;

  // With one row per block (TPR > 32) every thread runs the same trip count,
  // so the __syncthreads inside row_sum is reached by all.  Only the packed
  // inputs stay in registers across the reduction; n and g are recomputed.
  for (int64_t row = r0 + g; row < r1; row += RPC) {
    // One row per block (wide rows): thread 0 asks for the block's next row in
    // L2 while this one is processed, so its loads wait on L2, not DRAM.  (For
    // several rows per block the same prefetch measured slower.)
    if constexpr (RPC == 1) {
      if (threadIdx.x == 0 && row + 1 < r1) {
        const size_t nb = (size_t)(row + 1) * H;
        const uint32_t rb = (uint32_t)(H * sizeof(T));
        prefetch_l2(dy + nb, rb);
        prefetch_l2(h + nb, rb);
        if constexpr (DRES) prefetch_l2(dres + nb, rb);
      }
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
    const float rs = rstd[row];
    float dot = 0.f;
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
          n[e] *= rs;
          dot = fmaf(d[e] * wv[e], n[e], dot);
          acc[v][e] = fmaf(d[e], n[e], acc[v][e]);
        }
      }
    }
    dot = row_sum<TPR>(dot, red);
    const float c = dot * inv_H;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int iv = l + v * TPR;
      if (iv < nvec) {
        float d[VEC], n[VEC], wv[VEC], o[VEC];
        unpack<VEC>(dya[v], d);
        unpack<VEC>(ha[v], n);
        load_weight<W, VEC>(w, iv, wv);
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = rs * (d[e] * wv[e] - (n[e] * rs) * c);
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

  float* prow = partial + (size_t)p * H;
  if constexpr (RPC == 1) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int iv = l + v * TPR;
      if (iv < nvec) {
#pragma unroll
        for (int e = 0; e < VEC; e += 4)
          *reinterpret_cast<float4*>(prow + (size_t)iv * VEC + e) =
              make_float4(acc[v][e], acc[v][e + 1], acc[v][e + 2], acc[v][e + 3]);
      }
    }
  } else {
    // Fixed-order reduction over the RPC row groups through shared memory.
    __shared__ float sacc[RPC][TPR * VPT * VEC];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int iv = l + v * TPR;
      if (iv < nvec) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) sacc[g][iv * VEC + e] = acc[v][e];
      }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < H; j += BLOCK) {
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < RPC; ++q) s += sacc[q][j];
      prow[j] = s;
    }
  }
}

// ---------------------------------------------------------------------------
// Backward, element-wise path: P blocks, each over its contiguous row chunk,
// one row at a time; thread t owns columns t, t+256, ... of the partial row.
// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// Backward for rows of 65..128 vectors: kRmsGroups row groups of 64 threads (two
// vectors per thread) per block, the dW accumulators of each group in shared
// memory (four consecutive columns of a thread per 16-byte slot, slot k of
// thread t at acc[k * 64 + t]), a named barrier per group for its row sums.
// At 64 registers 1024 threads stay resident per SM (the warp-per-row kernel
// holds four vectors and the accumulators in ~124 registers: 512 threads).
// Groups walk rows r0 + g, r0 + g + kRmsGroups, ...; their accumulators are
// summed in a fixed order at the end.
// ---------------------------------------------------------------------------
constexpr int kRmsGroups = 4;
constexpr int kRmsGroupThreads = 64;

template <typename T, typename W, bool DRES>
__global__ void __launch_bounds__(kRmsGroups * kRmsGroupThreads, 1024 / (kRmsGroups * kRmsGroupThreads))
rms_bwd_grp(const T* dy, const T* dres, const T* h, const W* __restrict__ w,
            const float* __restrict__ rstd, T* dx, float* __restrict__ partial,
            int64_t rows, int H, float inv_H) {
  constexpr int TPR = kRmsGroupThreads, VPT = 2;
  constexpr int VEC = VecOf<T>::N;
  constexpr int Q = VEC / 4;
  constexpr int NSL = VPT * Q;
  extern __shared__ float4 acc_all[];  // [kRmsGroups][NSL][TPR]
  __shared__ float red[kRmsGroups][2][TPR / 32];
  const int g = threadIdx.x / TPR, l = threadIdx.x % TPR, lane = threadIdx.x % 32;
  float4* acc = acc_all + (size_t)g * NSL * TPR;
  const int nvec = H / VEC;
  const int64_t P = gridDim.x, p = blockIdx.x;
  const int64_t r0 = p * rows / P, r1 = (p + 1) * rows / P;
#pragma unroll
  for (int k = 0; k < NSL; ++k) acc[k * TPR + l] = make_float4(0.f, 0.f, 0.f, 0.f);

  int par = 0;
  for (int64_t row = r0 + g; row < r1; row += kRmsGroups) {
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
    const float rs = rstd[row];
    float dot = 0.f;
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
          n[e] *= rs;
          dot = fmaf(d[e] * wv[e], n[e], dot);
        }
#pragma unroll
        for (int q = 0; q < Q; ++q) {
          float4* aw = acc + (v * Q + q) * TPR + l;
          float4 a = *aw;
          a.x = fmaf(d[4 * q], n[4 * q], a.x);
          a.y = fmaf(d[4 * q + 1], n[4 * q + 1], a.y);
          a.z = fmaf(d[4 * q + 2], n[4 * q + 2], a.z);
          a.w = fmaf(d[4 * q + 3], n[4 * q + 3], a.w);
          *aw = a;
        }
      }
    }
    // Row sum over the group's two warps; red is double-buffered by row parity
    // (a buffer is written again only after the group's next barrier, which
    // every thread reaches after reading it).
    dot = group_sum<32>(dot);
    if (lane == 0) red[g][par][l / 32] = dot;
    bar_sync_named(1 + g, TPR);
    float tot = red[g][par][0];
#pragma unroll
    for (int k = 1; k < TPR / 32; ++k) tot += red[g][par][k];
    par ^= 1;
    const float c = tot * inv_H;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int iv = l + v * TPR;
      if (iv < nvec) {
        float d[VEC], n[VEC], wv[VEC], o[VEC];
        unpack<VEC>(dya[v], d);
        unpack<VEC>(ha[v], n);
        load_weight<W, VEC>(w, iv, wv);
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = rs * (d[e] * wv[e] - (n[e] * rs) * c);
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
  // v * Q + (j % VEC) / 4 of thread lt, where j / VEC = lt + v * TPR.
  float* prow = partial + (size_t)p * H;
  const float* af = reinterpret_cast<const float*>(acc_all);
  for (int j = threadIdx.x; j < H; j += kRmsGroups * TPR) {
    const int iv = j / VEC, e = j % VEC;
    const int lt = iv % TPR, v = iv / TPR;
    const size_t sl = ((size_t)(v * Q + e / 4) * TPR + lt) * 4 + e % 4;
    float a = 0.f;
#pragma unroll
    for (int q = 0; q < kRmsGroups; ++q) a += af[(size_t)q * NSL * TPR * 4 + sl];
    prow[j] = a;
  }
}

template <typename T, typename W, bool DRES>
__global__ void __launch_bounds__(kGenericBlock)
rms_bwd_generic(const T* dy, const T* dres, const T* h, const W* __restrict__ w,
                const float* __restrict__ rstd, T* dx, float* __restrict__ partial,
                int64_t rows, int H, float inv_H) {
  __shared__ float red[kGenericBlock / 32];
  const int64_t P = gridDim.x, p = blockIdx.x;
  const int64_t r0 = p * rows / P, r1 = (p + 1) * rows / P;
  float* prow = partial + (size_t)p * H;
  for (int j = threadIdx.x; j < H; j += kGenericBlock) prow[j] = 0.f;
  for (int64_t row = r0; row < r1; ++row) {
    const size_t base = (size_t)row * H;
    const float rs = rstd[row];
    KahanSum kd;
    for (int j = threadIdx.x; j < H; j += kGenericBlock)
      kd.add(to_f32(dy[base + j]) * to_f32(w[j]) * (to_f32(h[base + j]) * rs));
    const float dot = row_sum<kGenericBlock>(kd.s, red);
    const float c = dot * inv_H;
    for (int j = threadIdx.x; j < H; j += kGenericBlock) {
      const float d = to_f32(dy[base + j]);
      const float n = to_f32(h[base + j]) * rs;
      float o = rs * (d * to_f32(w[j]) - n * c);
      if constexpr (DRES) o += to_f32(dres[base + j]);
      prow[j] = fmaf(d, n, prow[j]);
      dx[base + j] = from_f32<T>(o);
    }
  }
}

// ---------------------------------------------------------------------------
// Launch geometry, shared by forward, backward and num_partials.
// ---------------------------------------------------------------------------
struct Geometry {
  bool vec;     // vector path possible (alignment checked separately)
  int tpr;      // threads per row
  int vpt;      // 16-byte vectors per thread
  int block;    // threads per block
  int rpc;      // rows per block (per pass of the row loop)
  int bps;      // backward: blocks per SM
};

Geometry geometry(int64_t H, size_t io_size) {
  Geometry g{};
  const int64_t row_bytes = H * (int64_t)io_size;
  const int64_t nvec = row_bytes / 16;
  if (row_bytes % 16 != 0 || nvec > kMaxVecPerRow) {
    g.vec = false; g.tpr = kGenericBlock; g.vpt = 0; g.block = kGenericBlock; g.rpc = 1; g.bps = 4;
    return g;
  }
  g.vec = true;
  if (nvec <= 128) {
    g.tpr = 32;
    g.vpt = nvec <= 32 ? 1 : (nvec <= 64 ? 2 : 4);
    g.block = kWarpBlock;
    g.rpc = kWarpBlock / 32;
    g.bps = 2;  // ~120 registers per thread: 512 resident threads per SM
  } else {
    int tpr = 64;
    while ((int64_t)tpr * 4 < nvec) tpr *= 2;  // <= 512 by kMaxVecPerRow
    g.tpr = tpr;
    g.vpt = 4;
    g.block = tpr;
    g.rpc = 1;
    g.bps = 512 / tpr > 0 ? 512 / tpr : 1;
  }
  return g;
}

// Backward geometry: rows of 65..128 vectors go to rms_bwd_grp (64-thread row
// groups, four per block, four blocks per SM); everything else as the forward.
Geometry bwd_geometry(int64_t H, size_t io_size) {
  Geometry g = geometry(H, io_size);
  if (g.vec && g.tpr == 32 && g.vpt == 4) {
    g.tpr = kRmsGroupThreads;
    g.vpt = 2;
    g.block = kRmsGroups * kRmsGroupThreads;
    g.rpc = kRmsGroups;
    g.bps = 1024 / g.block;
  }
  return g;
}

int64_t partials_for(int64_t T, const Geometry& g, int sms) {
  if (T <= 0) return 0;
  int64_t P = (int64_t)sms * g.bps;
  const int64_t groups = (T + g.rpc - 1) / g.rpc;
  if (P > groups) P = groups;
  return P < 1 ? 1 : P;
}

template <typename T, typename W, int TPR, int VPT, int BLOCK, bool MX>
void fwd_vec(bool res, const void* x, const void* r, const void* w, void* y, void* hout,
             float* rstd, int64_t rows, int H, float inv_H, float eps, MxOut mx, cudaStream_t s) {
  const unsigned grid = (unsigned)((rows + BLOCK / TPR - 1) / (BLOCK / TPR));
  if (res)
    rms_fwd_vec<T, W, TPR, VPT, BLOCK, true, MX><<<grid, BLOCK, 0, s>>>(
        (const T*)x, (const T*)r, (const W*)w, (T*)y, (T*)hout, rstd, rows, H, inv_H, eps, mx);
  else
    rms_fwd_vec<T, W, TPR, VPT, BLOCK, false, MX><<<grid, BLOCK, 0, s>>>(
        (const T*)x, nullptr, (const W*)w, (T*)y, nullptr, rstd, rows, H, inv_H, eps, mx);
}

template <typename T, typename W, bool MX = false>
gbln_status fwd_typed(const void* x, const void* r, const void* w, void* y, void* hout,
                      float* rstd, int64_t rows, int64_t H, float eps, cudaStream_t s,
                      MxOut mx = {}) {
  const bool res = r != nullptr;
  const Geometry g = geometry(H, sizeof(T));
  constexpr size_t kCodeAlign = 16 / sizeof(T);  // bytes of codes per 16-byte input vector
  const bool vec = g.vec && aligned16(x) && aligned16(w) && aligned16(y) &&
                   (!res || (aligned16(r) && aligned16(hout))) &&
                   (!MX || (reinterpret_cast<uintptr_t>(mx.q) % kCodeAlign) == 0);
  const float inv_H = 1.0f / (float)H;
  const int h = (int)H;
  if (!vec) {
    const unsigned grid = (unsigned)(rows < 65535LL * 32 ? rows : 65535LL * 32);
    if (res)
      rms_fwd_generic<T, W, true, MX><<<grid, kGenericBlock, 0, s>>>(
          (const T*)x, (const T*)r, (const W*)w, (T*)y, (T*)hout, rstd, rows, h, inv_H, eps, mx);
    else
      rms_fwd_generic<T, W, false, MX><<<grid, kGenericBlock, 0, s>>>(
          (const T*)x, nullptr, (const W*)w, (T*)y, nullptr, rstd, rows, h, inv_H, eps, mx);
    return launch_status();
  }
  if (g.tpr == 32) {
    if (g.vpt == 1) fwd_vec<T, W, 32, 1, kWarpBlock, MX>(res, x, r, w, y, hout, rstd, rows, h, inv_H, eps, mx, s);
    else if (g.vpt == 2) fwd_vec<T, W, 32, 2, kWarpBlock, MX>(res, x, r, w, y, hout, rstd, rows, h, inv_H, eps, mx, s);
    else fwd_vec<T, W, 32, 4, kWarpBlock, MX>(res, x, r, w, y, hout, rstd, rows, h, inv_H, eps, mx, s);
  } else {
    switch (g.tpr) {
      case 64: fwd_vec<T, W, 64, 4, 64, MX>(res, x, r, w, y, hout, rstd, rows, h, inv_H, eps, mx, s); break;
      case 128: fwd_vec<T, W, 128, 4, 128, MX>(res, x, r, w, y, hout, rstd, rows, h, inv_H, eps, mx, s); break;
      case 256: fwd_vec<T, W, 256, 4, 256, MX>(res, x, r, w, y, hout, rstd, rows, h, inv_H, eps, mx, s); break;
      default: fwd_vec<T, W, 512, 4, 512, MX>(res, x, r, w, y, hout, rstd, rows, h, inv_H, eps, mx, s); break;
    }
  }
  return launch_status();
}

template <typename T, typename W, int TPR, int VPT, int BLOCK>
void bwd_vec(bool dres, unsigned P, const void* dy, const void* dr, const void* h, const void* w,
             const float* rstd, void* dx, float* partial, int64_t rows, int H, float inv_H,
             cudaStream_t s) {
  if (dres)
    rms_bwd_vec<T, W, TPR, VPT, BLOCK, true><<<P, BLOCK, 0, s>>>(
        (const T*)dy, (const T*)dr, (const T*)h, (const W*)w, rstd, (T*)dx, partial, rows, H, inv_H);
  else
    rms_bwd_vec<T, W, TPR, VPT, BLOCK, false><<<P, BLOCK, 0, s>>>(
        (const T*)dy, nullptr, (const T*)h, (const W*)w, rstd, (T*)dx, partial, rows, H, inv_H);
}

template <typename T, typename W>
gbln_status bwd_grp(bool dres, unsigned P, const void* dy, const void* dr, const void* h,
                    const void* w, const float* rstd, void* dx, float* partial, int64_t rows, int H,
                    float inv_H, cudaStream_t s) {
  const size_t smem = (size_t)kRmsGroups * 2 * VecOf<T>::N * kRmsGroupThreads * sizeof(float);
  static std::atomic<uint64_t> attr_done{0};  // one bit per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return GBLN_ERR_CUDA; }
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    if (cudaFuncSetAttribute(rms_bwd_grp<T, W, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(rms_bwd_grp<T, W, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
      cudaGetLastError();
      return GBLN_ERR_CUDA;
    }
    attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  constexpr int B = kRmsGroups * kRmsGroupThreads;
  if (dres)
    rms_bwd_grp<T, W, true><<<P, B, smem, s>>>(
        (const T*)dy, (const T*)dr, (const T*)h, (const W*)w, rstd, (T*)dx, partial, rows, H, inv_H);
  else
    rms_bwd_grp<T, W, false><<<P, B, smem, s>>>(
        (const T*)dy, nullptr, (const T*)h, (const W*)w, rstd, (T*)dx, partial, rows, H, inv_H);
  return launch_status();
}

template <typename T, typename W>
gbln_status bwd_typed(const void* dy, const void* dr, const void* h, const void* w,
                      const float* rstd, void* dx, float* partial, int64_t P, int64_t rows,
                      int64_t H, cudaStream_t s) {
  const bool dres = dr != nullptr;
  const Geometry g = bwd_geometry(H, sizeof(T));
  const bool vec = g.vec && aligned16(dy) && aligned16(h) && aligned16(w) && aligned16(dx) &&
                   aligned16(partial) && (!dres || aligned16(dr));
  const float inv_H = 1.0f / (float)H;
  const int hh = (int)H;
  const unsigned grid = (unsigned)P;
  if (!vec) {
    if (dres)
      rms_bwd_generic<T, W, true><<<grid, kGenericBlock, 0, s>>>(
          (const T*)dy, (const T*)dr, (const T*)h, (const W*)w, rstd, (T*)dx, partial, rows, hh, inv_H);
    else
      rms_bwd_generic<T, W, false><<<grid, kGenericBlock, 0, s>>>(
          (const T*)dy, nullptr, (const T*)h, (const W*)w, rstd, (T*)dx, partial, rows, hh, inv_H);
    return launch_status();
  }
  if (g.tpr == 32) {
    if (g.vpt == 1) bwd_vec<T, W, 32, 1, kWarpBlock>(dres, grid, dy, dr, h, w, rstd, dx, partial, rows, hh, inv_H, s);
    else bwd_vec<T, W, 32, 2, kWarpBlock>(dres, grid, dy, dr, h, w, rstd, dx, partial, rows, hh, inv_H, s);
  } else if (g.rpc == kRmsGroups) {
    return bwd_grp<T, W>(dres, grid, dy, dr, h, w, rstd, dx, partial, rows, hh, inv_H, s);
  } else {
    switch (g.tpr) {
      case 64: bwd_vec<T, W, 64, 4, 64>(dres, grid, dy, dr, h, w, rstd, dx, partial, rows, hh, inv_H, s); break;
      case 128: bwd_vec<T, W, 128, 4, 128>(dres, grid, dy, dr, h, w, rstd, dx, partial, rows, hh, inv_H, s); break;
      case 256: bwd_vec<T, W, 256, 4, 256>(dres, grid, dy, dr, h, w, rstd, dx, partial, rows, hh, inv_H, s); break;
      default: bwd_vec<T, W, 512, 4, 512>(dres, grid, dy, dr, h, w, rstd, dx, partial, rows, hh, inv_H, s); break;
    }
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

extern "C" gbln_status gbln_rmsnorm_fwd(const void* x, const void* residual, const void* weight,
                                        void* y, void* residual_out, float* rstd, int64_t T,
                                        int64_t H, float eps, gbln_dtype io, gbln_dtype wt,
                                        gbln_stream_t stream) {
  if (!dtype_ok(io) || !dtype_ok(wt)) return GBLN_ERR_INVALID_ARG;
  if (T < 0 || T > kMaxRows || H <= 0 || H > kMaxH) return GBLN_ERR_INVALID_ARG;
  if (!(eps >= 0.0f && eps <= 3.4028235e38f)) return GBLN_ERR_INVALID_ARG;  // also rejects NaN
  if (!dtypes_ok(io, wt)) return GBLN_ERR_UNSUPPORTED;
  if (T == 0) return GBLN_OK;  // nothing is read or written: pointers are not examined
  if (!x || !weight || !y || !rstd) return GBLN_ERR_INVALID_ARG;
  if (residual && !residual_out) return GBLN_ERR_INVALID_ARG;
  const void* r = residual;
  void* ho = residual ? residual_out : nullptr;
  cudaStream_t s = (cudaStream_t)stream;
  if (io == GBLN_F32) return fwd_typed<float, float>(x, r, weight, y, ho, rstd, T, H, eps, s);
  if (wt == GBLN_BF16) return fwd_typed<bf16, bf16>(x, r, weight, y, ho, rstd, T, H, eps, s);
  return fwd_typed<bf16, float>(x, r, weight, y, ho, rstd, T, H, eps, s);
}

extern "C" gbln_status gbln_rmsnorm_fwd_mxfp8(const void* x, const void* residual,
                                              const void* weight, void* y, uint8_t* y_e4m3,
                                              uint8_t* y_scale, void* residual_out, float* rstd,
                                              int64_t T, int64_t H, float eps, gbln_dtype io,
                                              gbln_dtype wt, gbln_stream_t stream) {
  if (!dtype_ok(io) || !dtype_ok(wt)) return GBLN_ERR_INVALID_ARG;
  if (T < 0 || T > kMaxRows || H <= 0 || H > kMaxH || H % kMxBlock != 0) return GBLN_ERR_INVALID_ARG;
  if (!(eps >= 0.0f && eps <= 3.4028235e38f)) return GBLN_ERR_INVALID_ARG;
  if (!dtypes_ok(io, wt)) return GBLN_ERR_UNSUPPORTED;
  if (T == 0) return GBLN_OK;  // nothing is read or written: pointers are not examined
  if (!x || !weight || !y_e4m3 || !y_scale || !rstd) return GBLN_ERR_INVALID_ARG;
  if (residual && !residual_out) return GBLN_ERR_INVALID_ARG;
  const void* r = residual;
  void* ho = residual ? residual_out : nullptr;
  const MxOut mx{y_e4m3, y_scale};
  cudaStream_t s = (cudaStream_t)stream;
  if (io == GBLN_F32) return fwd_typed<float, float, true>(x, r, weight, y, ho, rstd, T, H, eps, s, mx);
  if (wt == GBLN_BF16) return fwd_typed<bf16, bf16, true>(x, r, weight, y, ho, rstd, T, H, eps, s, mx);
  return fwd_typed<bf16, float, true>(x, r, weight, y, ho, rstd, T, H, eps, s, mx);
}

extern "C" int64_t gbln_rmsnorm_bwd_num_partials(int64_t T, int64_t H, gbln_dtype io) {
  if (!dtype_ok(io) || T < 0 || T > kMaxRows || H <= 0 || H > kMaxH) return -1;
  if (T == 0) return 0;
  const int sms = sm_count();
  if (sms <= 0) return -1;
  return partials_for(T, bwd_geometry(H, dtype_size(io)), sms);
}

extern "C" gbln_status gbln_rmsnorm_bwd(const void* dy, const void* dresidual_out, const void* h,
                                        const void* weight, const float* rstd, void* dx,
                                        float* dw_partial, int64_t P_cap, int64_t T, int64_t H,
                                        gbln_dtype io, gbln_dtype wt, gbln_stream_t stream) {
  if (!dtype_ok(io) || !dtype_ok(wt)) return GBLN_ERR_INVALID_ARG;
  if (T < 0 || T > kMaxRows || H <= 0 || H > kMaxH || P_cap < 0) return GBLN_ERR_INVALID_ARG;
  if (!dtypes_ok(io, wt)) return GBLN_ERR_UNSUPPORTED;
  if (T == 0) return GBLN_OK;  // nothing is read or written: pointers are not examined
  if (!dy || !h || !weight || !rstd || !dx || !dw_partial) return GBLN_ERR_INVALID_ARG;
  const int sms = sm_count();
  if (sms <= 0) return GBLN_ERR_CUDA;
  const int64_t P = partials_for(T, bwd_geometry(H, dtype_size(io)), sms);
  if (P_cap < P) return GBLN_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  if (io == GBLN_F32)
    return bwd_typed<float, float>(dy, dresidual_out, h, weight, rstd, dx, dw_partial, P, T, H, s);
  if (wt == GBLN_BF16)
    return bwd_typed<bf16, bf16>(dy, dresidual_out, h, weight, rstd, dx, dw_partial, P, T, H, s);
  return bwd_typed<bf16, float>(dy, dresidual_out, h, weight, rstd, dx, dw_partial, P, T, H, s);
}

extern "C" gbln_status gbln_rmsnorm_dw_finalize(const float* dw_partial, int64_t P, int64_t H,
                                                float* dw, int accumulate,
                                                gbln_stream_t stream) {
  if (P < 0 || H <= 0 || H > kMaxH) return GBLN_ERR_INVALID_ARG;
  if (!dw || (P > 0 && !dw_partial)) return GBLN_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  colsum_kernel<<<(unsigned)((H + 31) / 32), 32 * kColSumStripes, 0, s>>>(
      dw_partial, P, (int)H, (int)H, dw, dw, (int)H, accumulate ? 1 : 0);
  return launch_status();
}

// ---------------------------------------------------------------------------
// Backward without caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// backward pass: code recorded into a CUDA graph under a capture mode that
// forbids cudaMalloc, runtimes whose memory is owned by a pool they may not
// bypass, and latency-critical loops where an allocation could synchronise
// the device.  For them the dW partials live in the fixed array below, which
// is part of the loaded module: every GPU that loads the library holds it
// (16 MiB) until the process exits.
// ---------------------------------------------------------------------------
namespace gbln {
namespace {

constexpr int64_t kScratchFloats = 4LL << 20;  // 16 MiB of float32 dW partials
static __device__ __align__(256) float g_dw_scratch[kScratchFloats];

constexpr int kMaxScratchDevices = 64;
std::atomic<float*> g_scratch_ptr[kMaxScratchDevices];

// Device address of g_dw_scratch on the current device (looked up once per
// device; in host code the symbol itself is only a host-side stand-in).
float* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) {
    cudaGetLastError();
    return nullptr;
  }
  float* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_dw_scratch) != cudaSuccess || addr == nullptr) {
    cudaGetLastError();
    return nullptr;
  }
  p = static_cast<float*>(addr);
  g_scratch_ptr[dev].store(p, std::memory_order_release);
  return p;
}

}  // namespace
}  // namespace gbln

extern "C" gbln_status gbln_rmsnorm_bwd_noalloc(const void* dy, const void* dresidual_out,
                                                const void* h, const void* weight,
                                                const float* rstd, void* dx, float* dw,
                                                int64_t T, int64_t H, gbln_dtype io,
                                                gbln_dtype wt, gbln_stream_t stream) {
  if (!dtype_ok(io) || !dtype_ok(wt)) return GBLN_ERR_INVALID_ARG;
  if (T < 0 || T > kMaxRows || H <= 0 || H > kMaxH) return GBLN_ERR_INVALID_ARG;
  if (!dtypes_ok(io, wt)) return GBLN_ERR_UNSUPPORTED;
  if (H > kScratchFloats) return GBLN_ERR_WORKSPACE;  // one partial row must fit
  if (!dw) return GBLN_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (T == 0) {  // no rows: dW = 0
    colsum_kernel<<<(unsigned)((H + 31) / 32), 32 * kColSumStripes, 0, s>>>(nullptr, 0, (int)H, (int)H, dw, dw, (int)H, 0);
    return launch_status();
  }
  if (!dy || !h || !weight || !rstd || !dx) return GBLN_ERR_INVALID_ARG;
  const int sms = sm_count();
  if (sms <= 0) return GBLN_ERR_CUDA;
  float* scratch = scratch_on_current_device();
  if (!scratch) return GBLN_ERR_CUDA;
  // Same kernels as gbln_rmsnorm_bwd + gbln_rmsnorm_dw_finalize; fewer partial
  // rows when the usual count would not fit the fixed array.
  int64_t P = partials_for(T, bwd_geometry(H, dtype_size(io)), sms);
  if (P * H > kScratchFloats) P = kScratchFloats / H;
  gbln_status st;
  if (io == GBLN_F32)
    st = bwd_typed<float, float>(dy, dresidual_out, h, weight, rstd, dx, scratch, P, T, H, s);
  else if (wt == GBLN_BF16)
    st = bwd_typed<bf16, bf16>(dy, dresidual_out, h, weight, rstd, dx, scratch, P, T, H, s);
  else
    st = bwd_typed<bf16, float>(dy, dresidual_out, h, weight, rstd, dx, scratch, P, T, H, s);
  if (st != GBLN_OK) return st;
  colsum_kernel<<<(unsigned)((H + 31) / 32), 32 * kColSumStripes, 0, s>>>(scratch, P, (int)H, (int)H, dw, dw, (int)H, 0);
  return launch_status();
}
