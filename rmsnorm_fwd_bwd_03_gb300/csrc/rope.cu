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

#include <atomic>

#include "common.cuh"

namespace gbln {

namespace {

// Rotate one vector pair: elements i0.. of the first half (a) and of the second
// half (b) of a head row, with the cos/sin entries c[0..VEC).  On the vector
// path the work goes two elements (one 32-bit word of bf16, or two floats) at
// a time so that only the packed inputs and one float4 of cos/sin are live.
// TABLE_IN_SMEM: c points into shared memory (plain loads) instead of the
// global table (read-only cached loads).
template <typename T, int VEC, bool BWD, bool TABLE_IN_SMEM = false>
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
        const float4* c4 = reinterpret_cast<const float4*>(c + 2 * w);
        const float4 f = ok ? (TABLE_IN_SMEM ? *c4 : __ldg(c4)) : make_float4(qnan, qnan, qnan, qnan);
        cv[0] = f.x; sv[0] = f.y; cv[1] = f.z; sv[1] = f.w;
      } else {
        const float2 f = ok ? (TABLE_IN_SMEM ? c[w] : __ldg(c + w)) : make_float2(qnan, qnan);
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
      const float2 f = ok ? (TABLE_IN_SMEM ? c[e] : __ldg(c + e)) : make_float2(qnan, qnan);
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

// ---------------------------------------------------------------------------
// Staged path: a persistent block walks tiles of TT consecutive tokens.  One
// producer thread reads the tile's positions and fills a stage of a ring of S
// shared-memory stages with TMA bulk copies: the tile's Q rows and K rows (two
// contiguous runs) and each token's cos/sin row from the table, all completing
// on the stage's mbarrier.  S tiles stay in flight per block without holding
// registers, and the threads then work from shared memory only: rotate and
// store straight to global memory with 128-bit stores.  Thread (r, v): vector
// v of the half rows, head lanes r, r + HPL, ...
// Stage layout: [TT Q rows][TT K rows][TT cos/sin rows][TT positions].
// ---------------------------------------------------------------------------
constexpr int kRopeStages = 4;
constexpr int kStagedMaxThreads = 32 + 256;  // producer warp + up to 8 consumer warps
// Bytes of Q, K and cos/sin rows per stage (whole tokens; at least one token).
constexpr size_t kStageTarget = 24 * 1024;

struct StageGeom {
  size_t qrow, krow, csrow, stage;
  int TT;
  __host__ __device__ size_t cs_off() const { return (size_t)TT * (qrow + krow); }
  __host__ __device__ size_t pos_off() const { return cs_off() + (size_t)TT * csrow; }
};

template <typename T>
__host__ __device__ inline StageGeom stage_geom(int Hq, int Hk, int D, int TT) {
  StageGeom g;
  g.qrow = (size_t)Hq * D * sizeof(T);
  g.krow = (size_t)Hk * D * sizeof(T);
  g.csrow = (size_t)(D / 2) * sizeof(float2);
  g.TT = TT;
  g.stage = g.pos_off() + (((size_t)TT * sizeof(int) + 15) / 16) * 16;
  return g;
}

// Warp 0 is the producer (its lane 0 issues); warps 1.. consume.  full[s]
// completes when stage s holds its tile; empty[s] completes when every
// consumer warp has finished reading it.  All waits are bounded.
template <typename T, bool BWD>
__global__ void __launch_bounds__(kStagedMaxThreads)
rope_staged_kernel(const T* __restrict__ q, const T* __restrict__ k, T* qo, T* ko,
                   const int32_t* __restrict__ pos, const float2* __restrict__ cs,
                   int64_t max_pos, int64_t T_, int Hq, int Hk, int D, int TT, int HPL,
                   unsigned int* err) {
  constexpr int VEC = VecOf<T>::N;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t full[kRopeStages], empty[kRopeStages];
  const int half = D / 2, nvh = half / VEC, HT = Hq + Hk;
  const int ncw = (int)(blockDim.x / 32) - 1;  // consumer warps
  const StageGeom g = stage_geom<T>(Hq, Hk, D, TT);
  const int64_t ntiles = (T_ + TT - 1) / TT;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int st = 0; st < kRopeStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], ncw);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == 0) {
    if (lane != 0) return;
    // ---- producer ----
    int64_t j = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++j) {
      const int st = (int)(j % kRopeStages);
      if (j >= kRopeStages &&
          !mbar_wait(&empty[st], (uint32_t)(((j / kRopeStages) - 1) & 1), kWaitPolls)) {
        atomicOr(err, kErrWaitTimeout);
        break;
      }
      fence_proxy_async_smem();
      const int64_t t0 = tile * TT;
      const int ntok = (int)(T_ - t0 < TT ? T_ - t0 : (int64_t)TT);
      unsigned char* base = smem + (size_t)st * g.stage;
      int* spos = reinterpret_cast<int*>(base + g.pos_off());
      uint32_t bytes = (uint32_t)(ntok * (g.qrow + g.krow));
      for (int tok = 0; tok < ntok; ++tok) {
        const int p = __ldg(pos + t0 + tok);
        const bool ok = p >= 0 && (int64_t)p < max_pos;
        spos[tok] = ok ? p : -1;
        if (ok) bytes += (uint32_t)g.csrow;
      }
      mbar_arrive_expect_tx(&full[st], bytes);  // also releases the spos writes
      bulk_load(base, reinterpret_cast<const unsigned char*>(q) + t0 * g.qrow,
                (uint32_t)(ntok * g.qrow), &full[st]);
      if (g.krow)
        bulk_load(base + (size_t)TT * g.qrow, reinterpret_cast<const unsigned char*>(k) + t0 * g.krow,
                  (uint32_t)(ntok * g.krow), &full[st]);
      for (int tok = 0; tok < ntok; ++tok)
        if (spos[tok] >= 0)
          bulk_load(base + g.cs_off() + (size_t)tok * g.csrow, cs + (size_t)spos[tok] * half,
                    (uint32_t)g.csrow, &full[st]);
    }
    // Do not leave while copies into this block's shared memory are in flight.
    for (int64_t jj = (j > kRopeStages ? j - kRopeStages : 0); jj < j; ++jj)
      mbar_wait(&full[jj % kRopeStages], (uint32_t)((jj / kRopeStages) & 1), kWaitPolls);
    return;
  }

  // ---- consumers ----
  const int c = threadIdx.x - 32;
  const int v = c % nvh, r = c / nvh;
  const bool active = r < HPL;
  const int i0 = v * VEC;
  int64_t j = 0;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++j) {
    const int st = (int)(j % kRopeStages);
    if (!mbar_wait(&full[st], (uint32_t)((j / kRopeStages) & 1), kWaitPolls)) {
      atomicOr(err, kErrWaitTimeout);
      break;
    }
    if (active) {
      const int64_t t0 = tile * TT;
      const int ntok = (int)(T_ - t0 < TT ? T_ - t0 : (int64_t)TT);
      const unsigned char* base = smem + (size_t)st * g.stage;
      const unsigned char* sq = base;
      const unsigned char* sk = base + (size_t)TT * g.qrow;
      const float2* scs = reinterpret_cast<const float2*>(base + g.cs_off());
      const int* spos = reinterpret_cast<const int*>(base + g.pos_off());
      for (int tok = 0; tok < ntok; ++tok) {
        const int64_t t = t0 + tok;
        const bool ok = spos[tok] >= 0;
        const float2* cc = scs + (size_t)tok * half + i0;
        for (int h = r; h < HT; h += HPL) {
          const T* src = reinterpret_cast<const T*>(h < Hq ? sq + (size_t)tok * g.qrow
                                                           : sk + (size_t)tok * g.krow) +
                         (size_t)(h < Hq ? h : h - Hq) * D;
          T* dst = h < Hq ? qo + ((size_t)t * Hq + h) * D : ko + ((size_t)t * Hk + (h - Hq)) * D;
          Packed<T, VEC> a, b;
          a.r = ld_shared_v4(src + i0);
          b.r = ld_shared_v4(src + half + i0);
          rotate_store<T, VEC, BWD, true>(a, b, cc, ok, dst + i0, dst + half + i0);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
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

// positions[t] = t - cu[d] for cu[d] <= t < cu[d+1]: binary search per token
// over the document boundaries, staged in shared memory when they fit (one
// coalesced read per block instead of a chain of dependent global loads).
constexpr int kPosSmemDocs = 4096;

__global__ void __launch_bounds__(256)
positions_kernel(const int32_t* __restrict__ cu, int ndoc, int32_t* pos, int64_t T_) {
  __shared__ int32_t scu[kPosSmemDocs];
  const bool staged = ndoc <= kPosSmemDocs;
  if (staged) {
    for (int i = threadIdx.x; i < ndoc; i += blockDim.x) scu[i] = __ldg(cu + i);
    __syncthreads();
  }
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T_;
       t += (int64_t)gridDim.x * blockDim.x) {
    int lo = 0, hi = ndoc - 1;  // largest d in [0, ndoc) with cu[d] <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      const int32_t c = staged ? scu[mid] : __ldg(cu + mid);
      if ((int64_t)c <= t) lo = mid; else hi = mid - 1;
    }
    pos[t] = (int32_t)(t - (int64_t)(staged ? scu[lo] : __ldg(cu + lo)));
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
  // Staged (TMA bulk) path: vector layout and a token small enough that four
  // stages of at least one token fit two blocks per SM.  In place is fine: a
  // tile is completely in shared memory before any of its outputs is stored.
  const size_t tok_bytes = (size_t)HT * D * sizeof(T) + (size_t)half * sizeof(float2);
  if (vec && nvh <= 256 && tok_bytes <= kStageTarget) {
    unsigned int* err = device_error_word();
    if (!err) return GBLN_ERR_CUDA;
    const int TT = (int)(kStageTarget / tok_bytes);
    const StageGeom geo = stage_geom<T>(Hq, Hk, D, TT);
    const size_t smem = (size_t)kRopeStages * geo.stage;
    const int hpl = 256 / nvh < HT ? 256 / nvh : HT;
    const int threads = 32 + ((nvh * hpl + 31) / 32) * 32;
    auto kern = rope_staged_kernel<T, BWD>;
    static std::atomic<uint64_t> attr_done{0};  // one bit per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return GBLN_ERR_CUDA; }
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)(kRopeStages * (kStageTarget + 1024))) != cudaSuccess) {
        cudaGetLastError();
        return GBLN_ERR_CUDA;
      }
      attr_done.fetch_or(bit, std::memory_order_acq_rel);
    }
    const int64_t ntiles = (rows + TT - 1) / TT;
    const unsigned sgrid = grid_for(ntiles, 1, (int64_t)sms * 2);
    kern<<<sgrid, threads, smem, s>>>((const T*)q, (const T*)k, (T*)qo, (T*)ko, pos,
                                      (const float2*)cs, max_pos, rows, Hq, Hk, D, TT, hpl, err);
    return launch_status();
  }
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
  positions_kernel<<<grid_for(T, 256, 1024), 256, 0, (cudaStream_t)stream>>>(cu_seqlens, ndoc,
                                                                               positions, T);
  return launch_status();
}
