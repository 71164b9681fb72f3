// Rotary position embedding on Q and K (forward and backward), its cos/sin
// table, and the per-document positions of packed sequences.
//
// Operator: "Fast-LLM: 高效大语言模型训练框架", §三 框架结构 (attention with RoPE) and
// "训练配置示例" (rotary type default, theta; heads / head_groups / head_size for
// grouped-query attention; micro_batch_size in tokens with
// maximum_document_length); "LLaMA-Factory Kernels 系统" (fused RoPE).
// Default pairing is rotate-half (element i turns with element i + D/2); the
// interleaved pairing (2i with 2i + 1) is the other common rotary type.
// Q and K may sit in strided rows (e.g. inside one packed QKV projection output).
//
// HBM-bound design: each element is read and written exactly once (in place is
// allowed); cos/sin come from a float32 table built once in double precision.
// The main path is one warp per (token, chunk of head rows) with the token's
// cos/sin held in registers across the rows a lane rotates (rope_warp_kernel);
// tokens with many heads per lane take a warp-specialised TMA pipeline
// (rope_staged_kernel); a register path covers layouts neither takes.

#include <atomic>

#include "common.cuh"

namespace gbln {

namespace {

// (cos, sin) of NP consecutive pairs, loaded once per token into registers and
// reused for every head row the thread rotates for that token.  An
// out-of-range position loads nothing: all entries are NaN, so are the outputs.
template <int NP>
struct CsUnit {
  float2 c[NP];
};

// SMEM: c points into shared memory (plain loads), else into the global table
// (read-only cached loads).  c is 16-byte aligned whenever NP is even.
template <int NP, bool SMEM>
__device__ __forceinline__ CsUnit<NP> load_cs(const float2* c, bool ok) {
  CsUnit<NP> u;
  if (!ok) {
    const float qnan = __int_as_float(0x7fc00000);
#pragma unroll
    for (int i = 0; i < NP; ++i) u.c[i] = make_float2(qnan, qnan);
    return u;
  }
  if constexpr (NP % 2 == 0) {
#pragma unroll
    for (int i = 0; i < NP; i += 2) {
      const float4* p4 = reinterpret_cast<const float4*>(c + i);
      const float4 f = SMEM ? *p4 : __ldg(p4);
      u.c[i] = make_float2(f.x, f.y);
      u.c[i + 1] = make_float2(f.z, f.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < NP; ++i) u.c[i] = SMEM ? c[i] : __ldg(c + i);
  }
  return u;
}

// Rotate one vector pair: elements i0.. of the first half (a) and of the second
// half (b) of a head row, with the unit's cos/sin entries cs.  On the vector
// path the work goes two elements (one 32-bit word of bf16, or two floats) at
// a time.
template <typename T, int VEC, bool BWD>
__device__ __forceinline__ void rotate_store(const Packed<T, VEC>& a, const Packed<T, VEC>& b,
                                             const CsUnit<VEC>& cs, T* d1, T* d2) {
  if constexpr (VEC * sizeof(T) == 16) {
    const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a.r);
    const uint32_t* bw = reinterpret_cast<const uint32_t*>(&b.r);
    uint32_t o1[4], o2[4];
    constexpr int PER = sizeof(T) == 2 ? 2 : 1;  // elements per 32-bit word
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float x1[2], x2[2];
      if constexpr (PER == 2) {
        x1[0] = bf16_lo(aw[w]); x1[1] = bf16_hi(aw[w]);
        x2[0] = bf16_lo(bw[w]); x2[1] = bf16_hi(bw[w]);
      } else {
        x1[0] = __uint_as_float(aw[w]); x2[0] = __uint_as_float(bw[w]);
      }
      float y1[2], y2[2];
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        const float2 f = cs.c[PER * w + e];
        if constexpr (!BWD) {
          y1[e] = x1[e] * f.x - x2[e] * f.y;
          y2[e] = x2[e] * f.x + x1[e] * f.y;
        } else {
          y1[e] = x1[e] * f.x + x2[e] * f.y;
          y2[e] = x2[e] * f.x - x1[e] * f.y;
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
      const float2 f = cs.c[e];
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

// Interleaved pairing: one vector of N elements holds N/2 pairs (2m, 2m + 1),
// rotated with the unit's cos/sin entries cs.
template <typename T, int N, bool BWD>
__device__ __forceinline__ void rotate_il_store(const Packed<T, N>& a, const CsUnit<(N >= 2 ? N / 2 : 1)>& cs,
                                                T* d) {
  float x[N], y[N];
  a.get(x);
#pragma unroll
  for (int m = 0; m < N / 2; ++m) {
    const float2 f = cs.c[m];
    const float x0 = x[2 * m], x1 = x[2 * m + 1];
    if constexpr (!BWD) {
      y[2 * m] = x0 * f.x - x1 * f.y;
      y[2 * m + 1] = x1 * f.x + x0 * f.y;
    } else {
      y[2 * m] = x0 * f.x + x1 * f.y;
      y[2 * m + 1] = x1 * f.x - x0 * f.y;
    }
  }
  store_n<T, N>(d, y);
}

// The same rotations reading cos/sin from shared memory as they go, one
// 16-byte piece per pair of elements, for threads that rotate a single head
// row per token (nothing to reuse; fewer live registers than CsUnit).
template <typename T, int VEC, bool BWD>
__device__ __forceinline__ void rotate_store_smem(const Packed<T, VEC>& a, const Packed<T, VEC>& b,
                                                  const float2* c, bool ok, T* d1, T* d2) {
  if constexpr (VEC * sizeof(T) == 16 && sizeof(T) == 2) {
    const float qnan = __int_as_float(0x7fc00000);
    const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a.r);
    const uint32_t* bw = reinterpret_cast<const uint32_t*>(&b.r);
    uint32_t o1[4], o2[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float4 f = ok ? *reinterpret_cast<const float4*>(c + 2 * w) : make_float4(qnan, qnan, qnan, qnan);
      const float x1[2] = {bf16_lo(aw[w]), bf16_hi(aw[w])};
      const float x2[2] = {bf16_lo(bw[w]), bf16_hi(bw[w])};
      const float cv[2] = {f.x, f.z}, sv[2] = {f.y, f.w};
      float y1[2], y2[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if constexpr (!BWD) {
          y1[e] = x1[e] * cv[e] - x2[e] * sv[e];
          y2[e] = x2[e] * cv[e] + x1[e] * sv[e];
        } else {
          y1[e] = x1[e] * cv[e] + x2[e] * sv[e];
          y2[e] = x2[e] * cv[e] - x1[e] * sv[e];
        }
      }
      o1[w] = pack_bf16x2(y1[0], y1[1]);
      o2[w] = pack_bf16x2(y2[0], y2[1]);
    }
    st_vec(d1, make_uint4(o1[0], o1[1], o1[2], o1[3]));
    st_vec(d2, make_uint4(o2[0], o2[1], o2[2], o2[3]));
  } else {
    rotate_store<T, VEC, BWD>(a, b, load_cs<VEC, true>(c, ok), d1, d2);
  }
}

// Everything a RoPE launch needs.  ld* are token strides in elements (a head
// row h of token t starts at base + t * ld + h * D).
template <typename T>
struct RopeArgs {
  const T* q;
  const T* k;
  T* qo;
  T* ko;
  const int32_t* pos;
  const float2* cs;
  int64_t max_pos, rows;
  int Hq, Hk, D;
  int64_t ldq, ldk, ldqo, ldko;
  unsigned int* err;  // device error word: kErrBadPosition for an out-of-range position
  __device__ __forceinline__ const T* src(int64_t t, int h) const {
    return h < Hq ? q + t * ldq + (int64_t)h * D : k + t * ldk + (int64_t)(h - Hq) * D;
  }
  __device__ __forceinline__ T* dst(int64_t t, int h) const {
    return h < Hq ? qo + t * ldqo + (int64_t)h * D : ko + t * ldko + (int64_t)(h - Hq) * D;
  }
};

// Register path.  Block of HP * NU threads, NU = units per head row (a unit is
// the two VEC-element vectors at i and i + D/2 for rotate-half pairing, one
// VEC-element vector of VEC/2 pairs for interleaved pairing): thread (hl, v)
// owns unit v of heads hl, hl + HP, ... (HPT of them per pass) of UT
// consecutive tokens per iteration; token groups are strided by gridDim.  All
// UT * HPT head loads are issued before the first is used; cos/sin come from
// L1 / L2 and are reused across the thread's heads.
template <typename T, int VEC, bool BWD, bool IL, int HPT, int UT>
__global__ void __launch_bounds__(512)
rope_kernel(const RopeArgs<T> A, int HP) {
  const int half = A.D / 2;
  const int nu = IL ? A.D / VEC : half / VEC;
  const int v = threadIdx.x % nu;
  const int hl = threadIdx.x / nu;
  const int HT = A.Hq + A.Hk;
  const int i0 = v * VEC;                 // first element of the unit
  const int c0 = IL ? i0 / 2 : i0;        // first cos/sin entry of the unit
  constexpr int NP = IL ? (VEC >= 2 ? VEC / 2 : 1) : VEC;  // cos/sin pairs of the unit
  for (int64_t tb = (int64_t)blockIdx.x * UT; tb < A.rows; tb += (int64_t)gridDim.x * UT) {
    int p[UT];
#pragma unroll
    for (int u = 0; u < UT; ++u) p[u] = tb + u < A.rows ? __ldg(A.pos + tb + u) : 0;
    for (int h0 = hl; h0 < HT; h0 += HP * HPT) {
      Packed<T, VEC> a[UT][HPT], b[UT][HPT];
#pragma unroll
      for (int u = 0; u < UT; ++u) {
        const int64_t t = tb + u;
#pragma unroll
        for (int j = 0; j < HPT; ++j) {
          const int h = h0 + j * HP;
          if (t < A.rows && h < HT) {
            const T* src = A.src(t, h);
            a[u][j].load(src + i0);
            if constexpr (!IL) b[u][j].load(src + half + i0);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < UT; ++u) {
        const int64_t t = tb + u;
        if (t >= A.rows) break;
        // out-of-range position: the table is not read, the outputs are NaN and
        // the device error word records it
        const bool ok = p[u] >= 0 && (int64_t)p[u] < A.max_pos;
        if (!ok && threadIdx.x == 0 && h0 == hl) atomicOr(A.err, kErrBadPosition);
        const CsUnit<NP> cs = load_cs<NP, false>(A.cs + (ok ? (size_t)p[u] * half : 0) + c0, ok);
#pragma unroll
        for (int j = 0; j < HPT; ++j) {
          const int h = h0 + j * HP;
          if (h < HT) {
            T* dst = A.dst(t, h);
            if constexpr (IL)
              rotate_il_store<T, VEC, BWD>(a[u][j], cs, dst + i0);
            else
              rotate_store<T, VEC, BWD>(a[u][j], b[u][j], cs, dst + i0, dst + half + i0);
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Warp path: one warp per (token, chunk of head rows), nothing staged.  With nu
// units per head row (a unit as in the register path) dividing 32, lane
// (g, v) = (lane / nu, lane % nu) owns unit v of the chunk's head rows g,
// g + G, g + 2G, ... (G = 32 / nu), at most kWarpHeads of them.  The lane reads
// its token's cos/sin entries for unit v once (VEC pairs straight into
// registers) and rotates every head row it owns with them, so the table costs
// 64 bytes per lane and token instead of 64 bytes per 32 bytes of Q/K.  All of
// a lane's row loads are issued before the first is used; for fixed j the warp
// covers G consecutive head rows, so each load instruction touches whole
// 128-byte segments.  No loop and no shared memory: the block scheduler keeps
// enough warps resident to cover DRAM latency.
// ---------------------------------------------------------------------------
constexpr int kWarpHeads = 6;

template <typename T, bool BWD, bool IL>
__global__ void __launch_bounds__(256, 3)
rope_warp_kernel(const RopeArgs<T> A, int nchunk, int ch) {
  constexpr int VEC = VecOf<T>::N;
  constexpr int NP = IL ? VEC / 2 : VEC;  // cos/sin pairs of a unit
  const int half = A.D / 2, HT = A.Hq + A.Hk;
  const int nu = IL ? A.D / VEC : half / VEC;
  const int G = 32 / nu;
  const int lane = threadIdx.x & 31;
  const int v = lane % nu, g = lane / nu;
  const int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t t = item / nchunk;
  if (t >= A.rows) return;  // uniform per warp
  const int c = (int)(item - t * nchunk);
  const int i0 = v * VEC, c0 = IL ? i0 / 2 : i0;
  const int hb = g + G * c * ch;
  const int p = __ldg(A.pos + t);
  Packed<T, VEC> a[kWarpHeads], b[kWarpHeads];
#pragma unroll
  for (int j = 0; j < kWarpHeads; ++j) {
    const int h = hb + G * j;
    if (j < ch && h < HT) {
      const T* src = A.src(t, h);
      a[j].load(src + i0);
      if constexpr (!IL) b[j].load(src + half + i0);
    }
  }
  // out-of-range position: the table is not read, the outputs are NaN and the
  // device error word records it
  const bool ok = p >= 0 && (int64_t)p < A.max_pos;
  if (!ok && lane == 0 && c == 0) atomicOr(A.err, kErrBadPosition);
  const CsUnit<NP> cs = load_cs<NP, false>(A.cs + (ok ? (size_t)p * half : 0) + c0, ok);
#pragma unroll
  for (int j = 0; j < kWarpHeads; ++j) {
    const int h = hb + G * j;
    if (j < ch && h < HT) {
      T* dst = A.dst(t, h);
      if constexpr (IL)
        rotate_il_store<T, VEC, BWD>(a[j], cs, dst + i0);
      else
        rotate_store<T, VEC, BWD>(a[j], b[j], cs, dst + i0, dst + half + i0);
    }
  }
}

// ---------------------------------------------------------------------------
// Staged path: a persistent block walks tiles of TT consecutive tokens.  One
// producer thread reads the tile's positions and fills a stage of a ring of S
// shared-memory stages with TMA bulk copies: the tile's Q rows and K rows and
// each token's cos/sin row from the table, all completing on the stage's
// mbarrier.  S tiles stay in flight per block without holding registers, and
// the threads then work from shared memory only: rotate and store straight to
// global memory with 128-bit stores.
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
// consumer warp has finished reading it.  All waits are bounded.  With
// contiguous Q (K) rows a tile's rows are one bulk copy, otherwise one per
// token.  Consumer thread (r, v): unit v of the head rows, head lanes r,
// r + HPL, ... (a unit as in the register path).
template <typename T, bool BWD, bool IL, bool HOIST>
__global__ void __launch_bounds__(kStagedMaxThreads)
rope_staged_kernel(const RopeArgs<T> A, int TT, int HPL, unsigned int* err) {
  constexpr int VEC = VecOf<T>::N;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t full[kRopeStages], empty[kRopeStages];
  const int D = A.D, Hq = A.Hq, Hk = A.Hk;
  const int half = D / 2, HT = Hq + Hk;
  const int nu = IL ? D / VEC : half / VEC;
  const int ncw = (int)(blockDim.x / 32) - 1;  // consumer warps
  const StageGeom g = stage_geom<T>(Hq, Hk, D, TT);
  const int64_t ntiles = (A.rows + TT - 1) / TT;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const bool qcontig = A.ldq == (int64_t)Hq * D, kcontig = A.ldk == (int64_t)Hk * D;

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
      const int ntok = (int)(A.rows - t0 < TT ? A.rows - t0 : (int64_t)TT);
      unsigned char* base = smem + (size_t)st * g.stage;
      int* spos = reinterpret_cast<int*>(base + g.pos_off());
      uint32_t bytes = (uint32_t)(ntok * (g.qrow + g.krow));
      for (int tok = 0; tok < ntok; ++tok) {
        const int p = __ldg(A.pos + t0 + tok);
        const bool ok = p >= 0 && (int64_t)p < A.max_pos;
        if (!ok) atomicOr(err, kErrBadPosition);
        spos[tok] = ok ? p : -1;
        if (ok) bytes += (uint32_t)g.csrow;
      }
      mbar_arrive_expect_tx(&full[st], bytes);  // also releases the spos writes
      if (g.qrow) {
        if (qcontig)
          bulk_load(base, A.q + t0 * A.ldq, (uint32_t)(ntok * g.qrow), &full[st]);
        else
          for (int tok = 0; tok < ntok; ++tok)
            bulk_load(base + (size_t)tok * g.qrow, A.q + (t0 + tok) * A.ldq, (uint32_t)g.qrow, &full[st]);
      }
      if (g.krow) {
        unsigned char* kb = base + (size_t)TT * g.qrow;
        if (kcontig)
          bulk_load(kb, A.k + t0 * A.ldk, (uint32_t)(ntok * g.krow), &full[st]);
        else
          for (int tok = 0; tok < ntok; ++tok)
            bulk_load(kb + (size_t)tok * g.krow, A.k + (t0 + tok) * A.ldk, (uint32_t)g.krow, &full[st]);
      }
      for (int tok = 0; tok < ntok; ++tok)
        if (spos[tok] >= 0)
          bulk_load(base + g.cs_off() + (size_t)tok * g.csrow, A.cs + (size_t)spos[tok] * half,
                    (uint32_t)g.csrow, &full[st]);
    }
    // Do not leave while copies into this block's shared memory are in flight.
    for (int64_t jj = (j > kRopeStages ? j - kRopeStages : 0); jj < j; ++jj)
      mbar_wait(&full[jj % kRopeStages], (uint32_t)((jj / kRopeStages) & 1), kWaitPolls);
    return;
  }

  // ---- consumers ----
  const int c = threadIdx.x - 32;
  const int v = c % nu, r = c / nu;
  const bool active = r < HPL;
  const int i0 = v * VEC;
  const int c0 = IL ? i0 / 2 : i0;
  constexpr int NP = IL ? (VEC >= 2 ? VEC / 2 : 1) : VEC;  // cos/sin pairs of a unit
  int64_t j = 0;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++j) {
    const int st = (int)(j % kRopeStages);
    if (!mbar_wait(&full[st], (uint32_t)((j / kRopeStages) & 1), kWaitPolls)) {
      atomicOr(err, kErrWaitTimeout);
      break;
    }
    if (active) {
      const int64_t t0 = tile * TT;
      const int ntok = (int)(A.rows - t0 < TT ? A.rows - t0 : (int64_t)TT);
      const unsigned char* base = smem + (size_t)st * g.stage;
      const unsigned char* sq = base;
      const unsigned char* sk = base + (size_t)TT * g.qrow;
      const float2* scs = reinterpret_cast<const float2*>(base + g.cs_off());
      const int* spos = reinterpret_cast<const int*>(base + g.pos_off());
      for (int tok = 0; tok < ntok; ++tok) {
        const int64_t t = t0 + tok;
        const bool ok = spos[tok] >= 0;
        const float2* cc = scs + (size_t)tok * half + c0;
        CsUnit<NP> cs;
        if constexpr (HOIST) cs = load_cs<NP, true>(cc, ok);
        for (int h = r; h < HT; h += HPL) {
          const T* src = reinterpret_cast<const T*>(h < Hq ? sq + (size_t)tok * g.qrow
                                                           : sk + (size_t)tok * g.krow) +
                         (size_t)(h < Hq ? h : h - Hq) * D;
          T* dst = A.dst(t, h);
          Packed<T, VEC> a;
          a.r = ld_shared_v4(src + i0);
          if constexpr (IL) {
            if constexpr (HOIST) rotate_il_store<T, VEC, BWD>(a, cs, dst + i0);
            else rotate_il_store<T, VEC, BWD>(a, load_cs<NP, true>(cc, ok), dst + i0);
          } else {
            Packed<T, VEC> b;
            b.r = ld_shared_v4(src + half + i0);
            if constexpr (HOIST) rotate_store<T, VEC, BWD>(a, b, cs, dst + i0, dst + half + i0);
            else rotate_store_smem<T, VEC, BWD>(a, b, cc, ok, dst + i0, dst + half + i0);
          }
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

template <typename T, int VEC, bool BWD, bool IL>
void rope_launch(int hpt, unsigned grid, int block, int HP, cudaStream_t s, const RopeArgs<T>& A) {
  switch (hpt) {  // heads x tokens per thread and pass
    case 1: rope_kernel<T, VEC, BWD, IL, 1, 2><<<grid, block, 0, s>>>(A, HP); break;
    case 2: rope_kernel<T, VEC, BWD, IL, 2, 1><<<grid, block, 0, s>>>(A, HP); break;
    default: rope_kernel<T, VEC, BWD, IL, 4, 1><<<grid, block, 0, s>>>(A, HP); break;
  }
}

template <typename T, bool BWD, bool IL>
gbln_status rope_typed(const RopeArgs<T>& A, cudaStream_t s) {
  constexpr int VEC = VecOf<T>::N;
  const int D = A.D, half = D / 2, HT = A.Hq + A.Hk;
  const bool ld16 = (A.ldq * (int64_t)sizeof(T)) % 16 == 0 && (A.ldqo * (int64_t)sizeof(T)) % 16 == 0 &&
                    (A.Hk == 0 || ((A.ldk * (int64_t)sizeof(T)) % 16 == 0 &&
                                   (A.ldko * (int64_t)sizeof(T)) % 16 == 0));
  const bool vec = (half % VEC == 0) && ld16 && aligned16(A.q) && aligned16(A.qo) &&
                   aligned16(A.cs) && (A.Hk == 0 || (aligned16(A.k) && aligned16(A.ko)));
  const int sms = sm_count();
  if (sms <= 0) return GBLN_ERR_CUDA;
  if (!A.err) return GBLN_ERR_CUDA;
  // elements per unit: VEC on the vector path; on the element-wise path 1
  // (rotate-half) or one pair (interleaved)
  const int unit = vec ? VEC : (IL ? 2 : 1);
  const int nu = IL ? D / unit : half / unit;
  if (nu > 512) return GBLN_ERR_UNSUPPORTED;  // head size above 1024 (bf16 vector path: 8192)
  // Warp path: vector layout with a unit count that divides a warp, and at most
  // two chunks of head rows per lane and token (up to 40 heads of 128 at bf16).
  // With more (70B widths: 72 heads) the staged pipeline below measured faster.
  const int G = vec && nu <= 32 && 32 % nu == 0 ? 32 / nu : 0;
  const int L = G ? (HT + G - 1) / G : 0;  // head rows per lane and token
  if (G && L <= 2 * kWarpHeads) {
    const int nchunk = (L + kWarpHeads - 1) / kWarpHeads;
    const int ch = (L + nchunk - 1) / nchunk;
    const int64_t blocks = (A.rows * nchunk + 7) / 8;  // 8 warps per block
    if (blocks <= 0x7fffffffLL) {
      rope_warp_kernel<T, BWD, IL><<<(unsigned)blocks, 256, 0, s>>>(A, nchunk, ch);
      return launch_status();
    }
  }
  // Staged (TMA bulk) path: vector layout and a token small enough that four
  // stages of at least one token fit two blocks per SM.  In place is fine: a
  // tile is completely in shared memory before any of its outputs is stored.
  const size_t tok_bytes = (size_t)HT * D * sizeof(T) + (size_t)half * sizeof(float2);
  if (vec && nu <= 256 && tok_bytes <= kStageTarget) {
    unsigned int* err = A.err;
    const int TT = (int)(kStageTarget / tok_bytes);
    const StageGeom geo = stage_geom<T>(A.Hq, A.Hk, D, TT);
    const size_t smem = (size_t)kRopeStages * geo.stage;
    const int hpl = 256 / nu < HT ? 256 / nu : HT;
    const int threads = 32 + ((nu * hpl + 31) / 32) * 32;
    // Threads with several head rows per token keep the token's cos/sin in
    // registers; with one row per token they read it as they go.
    auto kern = HT > hpl ? rope_staged_kernel<T, BWD, IL, true> : rope_staged_kernel<T, BWD, IL, false>;
    static std::atomic<uint64_t> attr_done{0};  // one bit per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return GBLN_ERR_CUDA; }
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
      const int cap = (int)(kRopeStages * (kStageTarget + 1024));
      if (cudaFuncSetAttribute(rope_staged_kernel<T, BWD, IL, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, cap) != cudaSuccess ||
          cudaFuncSetAttribute(rope_staged_kernel<T, BWD, IL, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, cap) != cudaSuccess) {
        cudaGetLastError();
        return GBLN_ERR_CUDA;
      }
      attr_done.fetch_or(bit, std::memory_order_acq_rel);
    }
    const int64_t ntiles = (A.rows + TT - 1) / TT;
    const unsigned sgrid = grid_for(ntiles, 1, (int64_t)sms * 2);
    kern<<<sgrid, threads, smem, s>>>(A, TT, hpl, err);
    return launch_status();
  }
  // Heads per thread: the smallest of 1, 2, 4 that fits the block in 512 threads
  // (4 with a loop over further heads beyond that).
  int hpt = 1;
  while (hpt < 4 && (int64_t)nu * ((HT + hpt - 1) / hpt) > 512) hpt *= 2;
  int HP = (HT + hpt - 1) / hpt;
  if ((int64_t)nu * HP > 512) HP = 512 / nu;
  const int block = nu * HP;
  const int per_sm = block > 0 ? 2048 / block : 1;
  const int ut = hpt == 1 ? 2 : 1;
  const unsigned grid = grid_for((A.rows + ut - 1) / ut, 1, (int64_t)sms * (per_sm > 0 ? per_sm : 1));
  if (vec)
    rope_launch<T, VEC, BWD, IL>(hpt, grid, block, HP, s, A);
  else if (IL)
    rope_launch<T, 2, BWD, IL>(hpt, grid, block, HP, s, A);
  else
    rope_launch<T, 1, BWD, IL>(hpt, grid, block, HP, s, A);
  return launch_status();
}

template <bool BWD>
gbln_status rope_entry(const void* q, const void* k, void* qo, void* ko, const int32_t* pos,
                       const float* cs, int64_t max_pos, int64_t T, int32_t Hq, int32_t Hk,
                       int32_t D, int64_t ldq, int64_t ldk, int64_t ldqo, int64_t ldko,
                       int pairing, gbln_dtype io, gbln_stream_t stream) {
  if (!dtype_ok(io) || (pairing != GBLN_ROPE_HALF && pairing != GBLN_ROPE_INTERLEAVED))
    return GBLN_ERR_INVALID_ARG;
  if (T < 0 || T > (1LL << 40) || Hq < 0 || Hk < 0 || Hq + Hk <= 0 || D <= 0 || (D & 1) ||
      max_pos < 0)
    return GBLN_ERR_INVALID_ARG;
  if ((int64_t)(Hq + Hk) * D > (1 << 24)) return GBLN_ERR_INVALID_ARG;
  const int64_t qw = (int64_t)Hq * D, kw = (int64_t)Hk * D, lim = 1LL << 40;
  if (ldq < qw || ldqo < qw || (Hk > 0 && (ldk < kw || ldko < kw))) return GBLN_ERR_INVALID_ARG;
  if (ldq > lim || ldqo > lim || ldk > lim || ldko > lim) return GBLN_ERR_INVALID_ARG;
  if (T == 0) return GBLN_OK;  // nothing is read or written: pointers are not examined
  if (!pos || !cs) return GBLN_ERR_INVALID_ARG;
  if (Hq > 0 && (!q || !qo)) return GBLN_ERR_INVALID_ARG;
  if (Hk > 0 && (!k || !ko)) return GBLN_ERR_INVALID_ARG;
  if (((uintptr_t)cs & 7u) != 0) return GBLN_ERR_INVALID_ARG;  // float2 table
  cudaStream_t s = (cudaStream_t)stream;
  const bool il = pairing == GBLN_ROPE_INTERLEAVED;
#define GBLN_ROPE_ARGS(TY)                                                                     \
  RopeArgs<TY> A{(const TY*)q, (const TY*)k, (TY*)qo, (TY*)ko, pos, (const float2*)cs, max_pos, \
                 T, Hq, Hk, D, ldq, Hk > 0 ? ldk : 0, ldqo, Hk > 0 ? ldko : 0, device_error_word()}
  if (io == GBLN_F32) {
    GBLN_ROPE_ARGS(float);
    return il ? rope_typed<float, BWD, true>(A, s) : rope_typed<float, BWD, false>(A, s);
  }
  GBLN_ROPE_ARGS(bf16);
  return il ? rope_typed<bf16, BWD, true>(A, s) : rope_typed<bf16, BWD, false>(A, s);
#undef GBLN_ROPE_ARGS
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
  const int64_t qw = (int64_t)Hq * D, kw = (int64_t)Hk * D;
  return rope_entry<false>(q, k, q_out, k_out, positions, cos_sin, max_pos, T, Hq, Hk, D, qw, kw,
                           qw, kw, GBLN_ROPE_HALF, io, stream);
}

extern "C" gbln_status gbln_rope_bwd(const void* dq, const void* dk, void* dq_in, void* dk_in,
                                     const int32_t* positions, const float* cos_sin,
                                     int64_t max_pos, int64_t T, int32_t Hq, int32_t Hk,
                                     int32_t D, gbln_dtype io, gbln_stream_t stream) {
  const int64_t qw = (int64_t)Hq * D, kw = (int64_t)Hk * D;
  return rope_entry<true>(dq, dk, dq_in, dk_in, positions, cos_sin, max_pos, T, Hq, Hk, D, qw, kw,
                          qw, kw, GBLN_ROPE_HALF, io, stream);
}

extern "C" gbln_status gbln_rope_fwd_ex(const void* q, const void* k, void* q_out, void* k_out,
                                        const int32_t* positions, const float* cos_sin,
                                        int64_t max_pos, int64_t T, int32_t Hq, int32_t Hk,
                                        int32_t D, int64_t ld_q, int64_t ld_k, int64_t ld_q_out,
                                        int64_t ld_k_out, gbln_rope_pairing pairing,
                                        gbln_dtype io, gbln_stream_t stream) {
  return rope_entry<false>(q, k, q_out, k_out, positions, cos_sin, max_pos, T, Hq, Hk, D, ld_q,
                           ld_k, ld_q_out, ld_k_out, pairing, io, stream);
}

extern "C" gbln_status gbln_rope_bwd_ex(const void* dq, const void* dk, void* dq_in, void* dk_in,
                                        const int32_t* positions, const float* cos_sin,
                                        int64_t max_pos, int64_t T, int32_t Hq, int32_t Hk,
                                        int32_t D, int64_t ld_dq, int64_t ld_dk, int64_t ld_dq_in,
                                        int64_t ld_dk_in, gbln_rope_pairing pairing,
                                        gbln_dtype io, gbln_stream_t stream) {
  return rope_entry<true>(dq, dk, dq_in, dk_in, positions, cos_sin, max_pos, T, Hq, Hk, D, ld_dq,
                          ld_dk, ld_dq_in, ld_dk_in, pairing, io, stream);
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
