// spec_verify.cu — the verify step of speculative sampling as hand-written sm_103a kernels (a streaming
// pass over every logit row, then a per-request pass; a nucleus pass between them for top-p).
//
// What is computed (host + section of the page that defines it):
//   cf-1.com/news/5155685 §2.2, 2kiu.com/news/5895634 §2.2  accept x ~ q with probability
//       min(1, p(x)/q(x)); on rejection draw from norm(max(0, p - q));
//   cf-1.com/news/5155685 §2.1, gsyq.cn/news/428210 §3.1     cut the output at the first rejection;
//   gsyq.cn/news/428210 §3.2                                  all K accepted: one more token from p;
//   gsyq.cn/news/428210 §3.3                                  temperature / top-k on both sides.
//
// Design.  The work is a stream over every logit of every valid row (HBM bound), plus a small
// per-request tail, in two kernels chained by programmatic dependent launch:
//   * the streaming pass: every (request, row, 16 KB chunk) item is read once and each warp leaves
//     a summary of its share -- (max, sum of exp) for sampling, (max, lowest argmax) for greedy
//     (stats_item_kernel: short-lived blocks of two items each, loaded straight into registers),
//     or a running candidate set for top-k (stats_kernel: a persistent grid whose blocks each own
//     a contiguous range of items, with a cp.async ring);
//   * the per-request pass (finish_kernel; 8-block clusters for small batches): one block per
//     request merges its rows' summaries into normalisers, runs the ratio test and the
//     first-rejection scan, and draws the resampled or bonus token by inverse CDF, re-reading only
//     the rows (or the chunk) the draw needs;
//   * with top-p and no top-k, a nucleus pass between them finds each row's nucleus.
// There is no tensor-core work: nothing here is a contraction.

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <float.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "spec_verify.h"

namespace sv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunkBytes = 16384;      // bytes of logits per work item (16 B per thread x 4)
constexpr int kCluster = 8;              // blocks sharing one request's draw when requests are few
constexpr int kStagesTopK = 2;           // top-k streaming pass: cp.async ring stages (4 blocks per SM)
constexpr int kItemBlocksPerSM = 6;      // sampling / greedy streaming pass: resident blocks per SM
constexpr int kItemsPerBlock = 2;        // items (16 KB each) per block of that pass
constexpr int kMultiTiles = 2;           // multi-draft stage passes: tiles in flight per warp
constexpr int kMultiCluster = 4;         // multi-draft, sampling: blocks per request (a cluster)
constexpr int kTile = 256;               // inverse-CDF tile: 32 lanes x 8 logits
constexpr int kCandCap = 256;            // top-k candidates stored per chunk
constexpr int kSegCap = 1024;            // running top-k candidates of a row segment (per buffer)
constexpr int kSegCompact = 320;         // compact the running set once it grows past this
constexpr int kRowCap = 256;             // candidates >= the row's lower bound, per row
constexpr int kMaxRows = 2 * SPEC_MAX_K + 1;
constexpr int kUnrollA = 4;              // tiles in flight per warp in the CDF passes (scalar rows)
constexpr int kDrawStages = 2;           // cp.async ring of the CDF pass over aligned rows
constexpr int kDrawStageBytes = 16384;   // per stage: the same 8 KB span of the p row and the q row

enum Mode { kSample = 0, kTopK = 1, kGreedy = 2 };

// Per-dtype chunking: every item is 16 KB of logits, 4 x 16-byte vectors per thread.
template <typename T>
struct Cfg {
  static constexpr int CH = kChunkBytes / (int)sizeof(T);  // logits per item
  static constexpr int PER = CH / kThreads;                 // logits per thread
  static constexpr int VW = 16 / (int)sizeof(T);            // logits per 16-byte vector
  static constexpr int LOADS = PER / VW;                    // vectors per thread
};

// Per-chunk top-k metadata word: count | flags.
constexpr uint32_t kMetaOverflow = 1u << 30;
constexpr uint32_t kMetaNaN = 1u << 31;
constexpr uint32_t kMetaCount = (1u << 30) - 1;

struct Params {
  const void* p;
  const void* q;
  const int32_t* draft;
  const int32_t* kpr;
  const float* ua;
  const float* ur;
  int32_t* out_tokens;
  int32_t* out_nacc;
  float* p_draft;
  float* q_draft;
  float* acc_margin;
  float* samp_margin;
  float* resid_mass;
  float* lognorm;
  float* rowcut;                  // per row: the smallest kept logit (top-k threshold / nucleus cut)
  float* sample_prob;             // draft-token sampling (K = 0): q(x) of each row's drawn token, or null
  int test_hooks;                 // spec_verify_set_test_hooks: 0 in normal operation
  int32_t* flags;
  void* pass1_done;               // optional cudaEvent_t recorded after the streaming pass
  int B, K, V, top_k, nchunk, R;  // R = padded rows per request (2K+1, or K+1 in greedy)
  float c2;                       // log2(e) / T of the target rows
  float invT;                     // 1 / T
  float c2q;                      // log2(e) / T_q of the draft rows (T_q = T unless set apart)
  float invTq;                    // 1 / T_q
  float top_p;                    // nucleus mass of every row; >= 1 = off
  float2* partial;                // [B, R, nchunk, warps] (max, sum) or (max, argmax) per warp
  uint2* cmeta;                   // [B, R, nchunk] top-k: (k-th largest key of the chunk, count|flags)
  uint2* cand;                    // [B, R, nchunk, kCandCap] top-k: (key, token)
  float2* rowstat;                // [B, R] top-p, sampling mode: (kept mass, cut) of each row
  const uint32_t* rowmap;         // ragged: [rows] (b << 6 | padded row); null = uniform layout
  const uint32_t* total_rows;     // ragged: number of valid rows
  uint32_t uniform_items;         // uniform layout: B * R * nchunk
};

// ------------------------------------------------------------------------------------------------
// small helpers
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<uint16_t>(uint16_t x) { return __uint_as_float((uint32_t)x << 16); }

template <typename T>
__device__ __forceinline__ float load1(const T* p) { return to_f<T>(__ldg(p)); }

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 2^x on the SFU (ex2.approx.ftz: relative error ~2^-22; results below 2^-126 flush to 0, which
// is far below what a sum of at most 2^21 terms, each relative to the row maximum, can resolve)
__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Programmatic dependent launch: a kernel lets the next kernel of the stream start launching
// (its blocks then wait in pdl_wait until this grid has finished and its writes are visible).
// Both are no-ops when the kernels are launched the ordinary way.
__device__ __forceinline__ void pdl_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Total order on floats as unsigned keys (-0 is folded into +0; NaN handled by callers).
__device__ __forceinline__ uint32_t fkey(float f) {
  uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float keyf(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

// Merge two (max, sum of exp2((z - max) * c2)) pairs.  A pair with sum 0 carries no mass.
__device__ __forceinline__ void lse_merge(float& m, float& s, float mo, float so, float c2) {
  float mn = fmaxf(m, mo);
  float a = (s == 0.0f) ? 0.0f : s * ex2((m - mn) * c2);
  float b = (so == 0.0f) ? 0.0f : so * ex2((mo - mn) * c2);
  m = mn;
  s = a + b;
}

__device__ __forceinline__ void lse_warp(float& m, float& s, float c2) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float mo = __shfl_xor_sync(0xFFFFFFFFu, m, o);
    float so = __shfl_xor_sync(0xFFFFFFFFu, s, o);
    lse_merge(m, s, mo, so, c2);
  }
}

// argmax with the lowest index on ties
__device__ __forceinline__ void amax_merge(float& v, int& i, float vo, int io) {
  if (vo > v || (vo == v && io < i)) {
    v = vo;
    i = io;
  }
}

// max that returns NaN if either input is NaN (so a NaN logit poisons its row's sum)
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}

// Row pointers in the padded layouts p [B, K+1, V] and q [B, K, V].
template <typename T>
__device__ __forceinline__ const T* prow(const Params& P, int b, int j) {
  return static_cast<const T*>(P.p) + ((size_t)b * (P.K + 1) + j) * (size_t)P.V;
}
template <typename T>
__device__ __forceinline__ const T* qrow(const Params& P, int b, int j) {
  return static_cast<const T*>(P.q) + ((size_t)b * P.K + j) * (size_t)P.V;
}
// Padded row index rp: p rows 0..K, q rows K+1..2K.
template <typename T>
__device__ __forceinline__ const T* row_ptr(const Params& P, int b, int rp) {
  return rp <= P.K ? prow<T>(P, b, rp) : qrow<T>(P, b, rp - P.K - 1);
}

__device__ __forceinline__ int clamp_k(const Params& P, int b, int* bad) {
  int k = P.kpr ? __ldg(P.kpr + b) : P.K;
  if (k < 0 || k > P.K) {
    if (bad) *bad = 1;
    k = k < 0 ? 0 : P.K;
  }
  return k;
}

// ------------------------------------------------------------------------------------------------
// chunk loading: 32 logits per thread; slot i of thread t holds chunk-local logit elem(i, t)
// ------------------------------------------------------------------------------------------------
template <typename T, bool VEC>
__device__ __forceinline__ int elem_of(int i, int t) {
  if (VEC) {
    constexpr int VW = Cfg<T>::VW;
    return ((i / VW) * kThreads + t) * VW + (i % VW);
  }
  return i * kThreads + t;
}

// Unpacks the thread's 16-byte vectors of a chunk into floats; vectors at or past n read -inf.
template <typename T>
__device__ __forceinline__ void unpack(const uint4 (&raw)[Cfg<T>::LOADS], int n, float (&v)[Cfg<T>::PER]) {
  constexpr int VW = Cfg<T>::VW;
  const int t = threadIdx.x;
  const bool full = n >= Cfg<T>::CH;
#pragma unroll
  for (int l = 0; l < Cfg<T>::LOADS; ++l) {
    const uint32_t w[4] = {raw[l].x, raw[l].y, raw[l].z, raw[l].w};
    const bool ok = full || (l * kThreads + t) * VW < n;
    if (sizeof(T) == 2) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[l * 8 + 2 * k] = ok ? bf16_lo(w[k]) : -INFINITY;
        v[l * 8 + 2 * k + 1] = ok ? bf16_hi(w[k]) : -INFINITY;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) v[l * 4 + k] = ok ? __uint_as_float(w[k]) : -INFINITY;
    }
  }
}

// Loads logits [0, n) of the chunk at `base` straight from global memory (any alignment).
template <typename T, bool VEC>
__device__ __forceinline__ void load_chunk(const T* __restrict__ base, int n, float (&v)[Cfg<T>::PER]) {
  const int t = threadIdx.x;
  if (VEC) {
    constexpr int VW = Cfg<T>::VW;
    uint4 raw[Cfg<T>::LOADS];
#pragma unroll
    for (int l = 0; l < Cfg<T>::LOADS; ++l) {
      const int e0 = (l * kThreads + t) * VW;
      raw[l] = e0 < n ? ldg_stream(base + e0) : make_uint4(0u, 0u, 0u, 0u);
    }
    unpack<T>(raw, n, v);
  } else {
#pragma unroll
    for (int i = 0; i < Cfg<T>::PER; ++i) {
      const int e = i * kThreads + t;
      v[i] = e < n ? load1<T>(base + e) : -INFINITY;
    }
  }
}

// The thread's 16-byte vectors of the chunk at `base` (16-byte aligned), not yet unpacked;
// vectors at or past n read nothing.
template <typename T>
__device__ __forceinline__ void load_raw(const T* __restrict__ base, int n, uint4 (&raw)[Cfg<T>::LOADS]) {
#pragma unroll
  for (int l = 0; l < Cfg<T>::LOADS; ++l) {
    const int e0 = (l * kThreads + threadIdx.x) * Cfg<T>::VW;
    raw[l] = e0 < n ? ldg_stream(base + e0) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// cp.async ring: each thread copies its own 16-byte vectors of a chunk into a stage and later
// reads exactly those bytes back, so only its own wait_group orders the copy and the read.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(gmem), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ------------------------------------------------------------------------------------------------
// shared memory
// ------------------------------------------------------------------------------------------------
struct Smem {
  float red_m[kWarps];
  float red_s[kWarps];
  int red_i[kWarps];
  uint32_t red_k[kWarps];
  int red_c[kWarps];
  // running top-k of the row segment a block streams
  int seg_n, seg_c0, seg_flags, seg_tight, seg_cur, seg_kept;
  uint32_t seg_theta;
  uint32_t hist[256];
  // finisher
  float rowM[kMaxRows];
  float rowS[kMaxRows];
  float rowT[kMaxRows];  // top-k threshold (-inf when off)
  int rowG[kMaxRows];    // greedy argmax
  int rowFlag[kMaxRows];
  int Kb, jstar, flags, nonfinite;
  int tile, seg_first, found;
  int rowListed[kMaxRows];  // top-k: the row's kept set is complete in its chunk lists
  float tile_base, total;
  float incl[kThreads];
  int y;
  float margin;
  float cl_total, cl_base, cl_R;  // cluster draw: this block's range total; the owner's offset, R
  int cl_owner;
  int nuc_digit;     // nucleus search: the bin of the cut at the current level
  float nuc_above;   // mass of the bins above it
  float nuc_bin;     // mass of the bin itself
  uint32_t nuc_count;  // logits in it
  float nuc_target;  // top_p * the row's kept mass
  int nuc_n;         // logits gathered
  uint32_t nuc_key;  // key of the cut
  uint32_t red_cnt[32];
};

// ------------------------------------------------------------------------------------------------
// per-item work
// ------------------------------------------------------------------------------------------------
// Sampling: each warp summarises its share of the chunk as (max, sum of 2^((z - max) * c2)) and
// writes it to out[warp]; the request's tail merges the warps' and chunks' pairs per row.
template <typename T>
__device__ __forceinline__ void item_sample(float c2, const float (&v)[Cfg<T>::PER], float2* out) {
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < Cfg<T>::PER; ++i) m = fmax_nan(m, v[i]);
  float s = 0.0f;
  if (m != -INFINITY) {
#pragma unroll
    for (int i = 0; i < Cfg<T>::PER; ++i) s += ex2((v[i] - m) * c2);
  }
  lse_warp(m, s, c2);
  if ((threadIdx.x & 31) == 0) out[threadIdx.x >> 5] = make_float2(m, s);
}

// Greedy: each warp writes its (max, lowest token id at the max) to out[warp]; a NaN anywhere in
// the warp's share is marked by the id -1.
template <typename T, bool VEC>
__device__ __forceinline__ void item_greedy(const float (&v)[Cfg<T>::PER], int n, int v0, float2* out) {
  const int t = threadIdx.x;
  float best = -INFINITY;
  int bi = 0x7FFFFFFF;
  bool nan = false;
#pragma unroll
  for (int i = 0; i < Cfg<T>::PER; ++i) {
    const int e = elem_of<T, VEC>(i, t);
    if (e < n) {
      nan |= v[i] != v[i];
      amax_merge(best, bi, v[i], v0 + e);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float vo = __shfl_xor_sync(0xFFFFFFFFu, best, o);
    int io = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
    amax_merge(best, bi, vo, io);
  }
  nan = __any_sync(0xFFFFFFFFu, nan);
  if ((t & 31) == 0) out[t >> 5] = make_float2(best, __int_as_float(nan ? -1 : bi));
}

// Descending bitonic sort of one key per lane across a warp.
__device__ __forceinline__ uint32_t warp_sort_desc(uint32_t x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, x, j);
      bool up = ((lane & k) == 0);      // this pair's block sorts descending when up
      bool lower = ((lane & j) == 0);   // this lane holds the lower index of the pair
      uint32_t hi = max(x, y), lo = min(x, y);
      x = (up == lower) ? hi : lo;
    }
  }
  return x;
}

// ------------------------------------------------------------------------------------------------
// top-k in the streaming pass: a running candidate set per row segment
// ------------------------------------------------------------------------------------------------
// A block streams a contiguous range of items, i.e. whole rows or a row's head or tail (a
// segment).  It keeps the segment's candidates in shared memory together with a lower bound
// theta on the row's k-th largest logit: every logit < theta can be dropped, since k logits of the
// row are already known to be >= theta.  After the first chunk theta is tight, so almost every
// logit of the following chunks is settled by one compare.  At the segment's end the candidates
// >= the segment's k-th largest (ties kept) are written, sorted, at the segment's first chunk slot.

// Lower bound on a chunk's k-th largest from the per-thread maxima (whole block): in each warp with
// data, the c_w-th largest thread maximum, c_w = min(ceil(k / warps with data), threads with data);
// those maxima are distinct logits, so >= sum_w c_w logits are >= min_w.  Returns key 0 if that
// count falls short of k.
template <typename T, bool VEC>
__device__ uint32_t chunk_bound(const float (&v)[Cfg<T>::PER], int n, int k, Smem& sm) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  uint32_t tmax = 0;
#pragma unroll
  for (int i = 0; i < Cfg<T>::PER; ++i) {
    const int e = elem_of<T, VEC>(i, t);
    if (e < n && v[i] == v[i]) tmax = max(tmax, fkey(v[i]));
  }
  const unsigned has = __ballot_sync(0xFFFFFFFFu, tmax != 0u);
  if (lane == 0) sm.red_c[warp] = __popc(has);
  __syncthreads();
  int nw = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) nw += sm.red_c[w] > 0;
  const int kp = (k + nw - 1) / max(nw, 1);
  const uint32_t sorted = warp_sort_desc(tmax);
  const int cw = min(kp, __popc(has));
  const uint32_t thw = cw > 0 ? __shfl_sync(0xFFFFFFFFu, sorted, cw - 1) : 0xFFFFFFFFu;
  __syncthreads();
  if (lane == 0) {
    sm.red_k[warp] = thw;
    sm.red_c[warp] = cw;
  }
  __syncthreads();
  uint32_t theta = 0xFFFFFFFFu;
  int certified = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    if (sm.red_c[w] > 0) theta = min(theta, sm.red_k[w]);
    certified += sm.red_c[w];
  }
  __syncthreads();
  return (kp > 32 || certified < k) ? 0u : theta;
}

// Appends the chunk's logits >= theta (key 0: every logit) to the segment buffer.  Once theta is
// tight almost no logit survives, so each thread first takes its own maximum (a tree of max.NaN;
// logits past the row read -inf) and only a thread whose maximum reaches theta walks its logits
// one by one, reserving its slots with one shared atomic.
template <typename T, bool VEC>
__device__ void seg_filter(const float (&v)[Cfg<T>::PER], int n, int v0, uint32_t theta, uint2* buf, Smem& sm) {
  const int t = threadIdx.x, lane = t & 31;
  const float tf = theta == 0u ? -INFINITY : keyf(theta);
  const bool full = n >= Cfg<T>::CH;  // no logit past the row in this chunk
  float m[Cfg<T>::PER / 2];
#pragma unroll
  for (int i = 0; i < Cfg<T>::PER / 2; ++i) m[i] = fmax_nan(v[2 * i], v[2 * i + 1]);
#pragma unroll
  for (int w = Cfg<T>::PER / 4; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = fmax_nan(m[i], m[i + w]);
  const float mx = m[0];
  if (__any_sync(0xFFFFFFFFu, mx != mx) && lane == 0) atomicOr(&sm.seg_flags, (int)kMetaNaN);
  if (!(mx >= tf)) return;
  // a lane with survivors reserves its own slots (survivors are few once the bound is tight)
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < Cfg<T>::PER; ++i) cnt += (full || elem_of<T, VEC>(i, t) < n) && v[i] >= tf;
  int base = atomicAdd(&sm.seg_n, cnt);
  {
#pragma unroll
    for (int i = 0; i < Cfg<T>::PER; ++i) {
      const int e = elem_of<T, VEC>(i, t);
      if ((full || e < n) && v[i] >= tf) {
        if (base < kSegCap) buf[base] = make_uint2(fkey(v[i]), (uint32_t)(v0 + e));
        ++base;
      }
    }
  }
}

// A cut of the segment buffer src[0..n) (n >= k): a key c with at least k keys >= c, found by
// histograms of the keys over 256 equal bins of a range [lo, hi]: the bin holding the k-th largest
// key (counting from the top) is taken whole when it holds few keys, and is otherwise made the next
// range (logits straddling 0 or spanning several binades put most keys in one bin of the full key
// range; the bin at the next level is 2^8 times narrower).  The returned cut is that bin's lower
// edge, so every key >= c is a candidate and k of them certify c as a lower bound on the row's
// k-th largest.  Whole block.
__device__ uint32_t seg_cut(const uint2* src, int n, int k, Smem& sm) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  constexpr uint32_t kFewKeys = 48;  // a cut bin with at most this many keys is taken whole
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int i = t; i < n; i += kThreads) {
    const uint32_t key = src[i].x;
    lo = min(lo, key);
    hi = max(hi, key);
  }
  lo = __reduce_min_sync(0xFFFFFFFFu, lo);
  hi = __reduce_max_sync(0xFFFFFFFFu, hi);
  if (lane == 0) {
    sm.red_k[warp] = lo;
    sm.red_c[warp] = (int)hi;
  }
  __syncthreads();
  lo = 0xFFFFFFFFu;
  hi = 0u;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    lo = min(lo, sm.red_k[w]);
    hi = max(hi, (uint32_t)sm.red_c[w]);
  }
  int above = 0;  // keys above the current range
  uint32_t cut = lo;
  for (;;) {  // every thread holds the same lo, hi, above
    const uint32_t span = hi - lo;
    const int shift = span < 256u ? 0 : 32 - __clz(span) - 8;  // (hi - lo) >> shift < 256
    sm.hist[t] = 0u;  // 256 threads, 256 bins
    __syncthreads();
    for (int i = t; i < n; i += kThreads) {
      const uint32_t key = src[i].x;
      if (key >= lo && key <= hi) atomicAdd(&sm.hist[(key - lo) >> shift], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255-8l .. 248-8l (descending); the bin where the count of keys in it and
      // above first reaches k
      int c8[8], s = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        c8[q] = (int)sm.hist[255 - 8 * lane - q];
        s += c8[q];
      }
      int incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, above + incl >= k);
      const int hl = __ffs(hit) - 1;  // hit != 0: n >= k keys in all, every one in [lo, hi] or above
      if (lane == hl) {
        int acc = above + incl - s, q = 0;
        while (q < 7 && acc + c8[q] < k) acc += c8[q++];
        const uint32_t bin = (uint32_t)(255 - 8 * lane - q);
        sm.red_k[0] = lo + (bin << shift);
        sm.red_c[0] = acc;                       // keys above the bin
        sm.red_c[1] = c8[q] <= (int)kFewKeys || shift == 0;  // take the bin whole
      }
    }
    __syncthreads();
    const uint32_t blo = sm.red_k[0];
    const int acc = sm.red_c[0], whole = sm.red_c[1];
    __syncthreads();  // red_k / red_c and the bins are reused
    if (whole) {
      cut = blo;
      break;
    }
    above = acc;
    const uint64_t bhi = (uint64_t)blo + ((1ull << shift) - 1ull);  // the bin's keys become the range
    hi = bhi < (uint64_t)hi ? (uint32_t)bhi : hi;
    lo = blo;
  }
  return cut;
}

// Keeps the segment's entries >= a cut with at least k entries at or above it (all of them when
// fewer than k) in the other buffer; theta becomes that cut.  With `sorted` the kept entries are
// placed by key descending (buffer index ascending among equal keys).  Whole block.
__device__ void seg_compact(int k, bool sorted, uint2* bufs, Smem& sm) {
  const int t = threadIdx.x, lane = t & 31;
  const int cur = sm.seg_cur;
  const uint2* src = bufs + (size_t)cur * kSegCap;
  uint2* dst = bufs + (size_t)(cur ^ 1) * kSegCap;
  int n = sm.seg_n;
  if (n > kSegCap) {  // candidates were lost: the row takes the exact path
    if (t == 0) sm.seg_flags |= (int)kMetaOverflow;
    n = kSegCap;
  }
  const uint32_t kth = n >= k ? seg_cut(src, n, k, sm) : 0u;
  if (t == 0) sm.seg_kept = 0;
  __syncthreads();
  for (int i0 = 0; i0 < n; i0 += kThreads) {  // keep the entries >= kth (unordered), a slot range per warp
    const int i = i0 + t;
    const bool keep = i < n && src[i].x >= kth;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, keep);
    int base = 0;
    if (lane == 0 && m) base = atomicAdd(&sm.seg_kept, __popc(m));
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
    if (keep) dst[base + __popc(m & ((1u << lane) - 1u))] = src[i];
  }
  if (sorted) {  // place the kept entries by key descending, then position, back in src
    __syncthreads();
    const int m = sm.seg_kept;
    uint2* out = const_cast<uint2*>(src);
    for (int i = t; i < m; i += kThreads) {
      const uint32_t ki = dst[i].x, vi = dst[i].y;
      int pos = 0;
      for (int j = 0; j < m; ++j) {
        const uint32_t kj = dst[j].x;
        pos += (kj > ki) | ((kj == ki) & (dst[j].y < vi));
      }
      out[pos] = dst[i];
    }
  }
  __syncthreads();
  if (t == 0) {
    sm.seg_n = sm.seg_kept;
    sm.seg_cur = sorted ? cur : cur ^ 1;
    if (n >= k) {
      sm.seg_theta = max(sm.seg_theta, kth);
      sm.seg_tight = 1;
    }
  }
  __syncthreads();
}

// One chunk of a top-k row in the streaming pass.
template <typename T, bool VEC>
__device__ void topk_chunk(const Params& P, const float (&v)[Cfg<T>::PER], int n, int b, int rp, int c,
                           bool seg_start, bool seg_end, uint2* bufs, Smem& sm, int& seg_next, int& seg_m) {
  const int k = P.top_k;
  if (seg_start) {
    seg_next = 0;  // the block's check schedule: identical registers in every thread
    seg_m = 0;
    if (threadIdx.x == 0) {
      sm.seg_n = 0;
      sm.seg_theta = 0;
      sm.seg_c0 = c;
      sm.seg_flags = 0;
      sm.seg_tight = 0;
      sm.seg_cur = 0;
    }
    __syncthreads();
  }
  uint32_t theta = sm.seg_theta;
  if (!sm.seg_tight) theta = max(theta, chunk_bound<T, VEC>(v, n, k, sm));
  const bool tight = sm.seg_tight;
  seg_filter<T, VEC>(v, n, c * Cfg<T>::CH, theta, bufs + (size_t)sm.seg_cur * kSegCap, sm);
  // The block meets (and maybe compacts) only on its check schedule.  A bound refreshed over m
  // chunks lets about k / m survivors through per chunk; the next check comes when twice that
  // rate would fill the buffer's free room (after 1..32 chunks).  Every thread derives the same
  // schedule from values it reads between two barriers, so all of them meet at the same chunks.
  const int dc = c - sm.seg_c0;
  if (seg_end || !tight || dc >= seg_next) {
    __syncthreads();
    if (seg_end || sm.seg_n > kSegCompact || (!tight && sm.seg_n >= k)) {
      seg_compact(k, seg_end, bufs, sm);
      seg_m = dc + 1;
    }
    const int fill = min(sm.seg_n, kSegCap);
    __syncthreads();  // nobody adds to the set before every thread has read its size
    const int gap = ((kSegCap - fill) * max(seg_m, 1)) / (2 * k);
    seg_next = dc + min(32, max(1, gap));
  }
  const size_t row_slot = ((size_t)b * P.R + rp) * P.nchunk;
  if (threadIdx.x == 0 && c != sm.seg_c0) P.cmeta[row_slot + c] = make_uint2(0u, 0u);
  if (seg_end) {  // the segment's list, sorted, at its first chunk's slot
    const int nk = sm.seg_n;
    const uint2* src = bufs + (size_t)sm.seg_cur * kSegCap;
    uint2* out = P.cand + (row_slot + sm.seg_c0) * kCandCap;
    for (int i = threadIdx.x; i < min(nk, kCandCap); i += kThreads) out[i] = src[i];
    if (threadIdx.x == 0) {
      const uint32_t fl = (uint32_t)sm.seg_flags | (nk > kCandCap ? kMetaOverflow : 0u);
      P.cmeta[row_slot + sm.seg_c0] = make_uint2(nk >= k ? sm.seg_theta : 0u, (uint32_t)min(nk, kCandCap) | fl);
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------------------------------------
// finisher pieces
// ------------------------------------------------------------------------------------------------
// Loads the 8 logits [e0, e0+8) of a row (e0 a multiple of 8); logits at or past V read -inf.
template <typename T, bool VEC>
__device__ __forceinline__ void load8(const T* __restrict__ row, int e0, int V, float (&z)[8]) {
  if (VEC) {
    if (sizeof(T) == 2) {
      if (e0 < V) {
        uint4 r = ldg_stream(row + e0);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          z[2 * k] = bf16_lo(w[k]);
          z[2 * k + 1] = bf16_hi(w[k]);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) z[k] = -INFINITY;
      }
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        int e = e0 + 4 * h;
        if (e < V) {
          uint4 r = ldg_stream(row + e);
          z[4 * h] = __uint_as_float(r.x);
          z[4 * h + 1] = __uint_as_float(r.y);
          z[4 * h + 2] = __uint_as_float(r.z);
          z[4 * h + 3] = __uint_as_float(r.w);
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) z[4 * h + k] = -INFINITY;
        }
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) z[k] = (e0 + k < V) ? load1<T>(row + e0 + k) : -INFINITY;
  }
}

// Weights of the inverse-CDF draw for 8 logits: the residual max(0, P - Q) when `resid`, else the
// (unnormalised) target weights exp((z_p - M_p)/T) on the kept set.
struct DrawRows {
  float Lp, Tp;  // target row: log2 normaliser (max * c2 + log2 sum), truncation threshold
  float Lq, Tq;  // draft row
  float Mp2;     // target row max * c2 (scale of the weights of a draw from p alone)
  float c2q;     // the draft row's scale log2(e) / T_q
  bool resid;
};

// Weights of the inverse-CDF draw for 8 logits: the residual max(0, P - Q) with
// P = 2^(z_p * c2 - Lp), Q = 2^(z_q * c2q - Lq) when `resid`, else the target weights
// 2^(z_p * c2 - Mp2) relative to the row max.  Logits below a row's truncation threshold
// (top-k and / or top-p) weigh 0 (MASK).
// Both passes of a draw compute them with these same instructions, so they agree bit for bit.
template <bool MASK>
__device__ __forceinline__ void weights_of(const float (&zp)[8], const float (&zq)[8], const DrawRows& d,
                                           float c2, float (&w)[8]) {
  const float2 cc = make_float2(c2, c2);
  if (d.resid) {
    const float2 nlp = make_float2(-d.Lp, -d.Lp), nlq = make_float2(-d.Lq, -d.Lq);
    const float2 ccq = make_float2(d.c2q, d.c2q);
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
      const float2 a = __ffma2_rn(make_float2(zp[k], zp[k + 1]), cc, nlp);
      const float2 b = __ffma2_rn(make_float2(zq[k], zq[k + 1]), ccq, nlq);
      float pa = ex2(a.x), pb = ex2(a.y), qa = ex2(b.x), qb = ex2(b.y);
      if (MASK) {
        pa = zp[k] >= d.Tp ? pa : 0.0f;
        pb = zp[k + 1] >= d.Tp ? pb : 0.0f;
        qa = zq[k] >= d.Tq ? qa : 0.0f;
        qb = zq[k + 1] >= d.Tq ? qb : 0.0f;
      }
      const float2 r = __fadd2_rn(make_float2(pa, pb), make_float2(-qa, -qb));
      w[k] = fmaxf(r.x, 0.0f);
      w[k + 1] = fmaxf(r.y, 0.0f);
    }
  } else {
    const float2 nm = make_float2(-d.Mp2, -d.Mp2);
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
      const float2 a = __ffma2_rn(make_float2(zp[k], zp[k + 1]), cc, nm);
      w[k] = ex2(a.x);
      w[k + 1] = ex2(a.y);
      if (MASK) {
        w[k] = zp[k] >= d.Tp ? w[k] : 0.0f;
        w[k + 1] = zp[k + 1] >= d.Tp ? w[k + 1] : 0.0f;
      }
    }
  }
}

template <typename T, bool VEC, bool MASK>
__device__ __forceinline__ void weights8(const T* pr, const T* qr, int e0, int V, const DrawRows& d,
                                         float c2, float (&w)[8]) {
  float zp[8], zq[8];
  load8<T, VEC>(pr, e0, V, zp);
  if (d.resid)
    load8<T, VEC>(qr, e0, V, zq);
  else
#pragma unroll
    for (int k = 0; k < 8; ++k) zq[k] = -INFINITY;
  weights_of<MASK>(zp, zq, d, c2, w);
}

// Inverse-CDF draw over the logits [v0, vend) of a row: y = the smallest v with target < C_v,
// C_v cumulative in ascending token id, computed hierarchically (8 logits per lane, 256 per warp
// tile, tiles by segments per thread).  With `full`, the range is the whole row and
// target = u * (its total), which is also the margin scale; otherwise `target` is the mass the
// draw must pass inside the range and `Rm` the margin scale.  Returns the range total; sets
// sm.y, sm.margin and the clamp flag.  `phase` splits the work for a cluster of blocks sharing
// one row: 1 = only the tile sums and the range total (kept in wt / sm for a later phase 2),
// 2 = only the search, over the sums a phase-1 call on the same range left; 0 = both.
template <typename T, bool VEC, bool MASK>
__device__ float draw_range(const Params& P, const T* pr, const T* qr, const DrawRows& d, int v0,
                            int vend, bool full, float u, float target_in, float Rm, float* wt,
                            uint4* ring, Smem& sm, int* clamp, int phase = 0) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int V = vend;
  const int ntile = (vend - v0 + kTile - 1) / kTile;
  // pass A: tile sums
  if (phase != 2) {
  if constexpr (VEC) {
    // Aligned rows stream through a cp.async ring: stage k holds elements [v0 + k*SE, + SE) of the
    // p row and of the q row (the q half is not read for a draw from p alone).  Each thread copies
    // 4 of the stage's 16-byte vectors; after the barrier every warp reads whole tiles.
    constexpr int SE = kDrawStageBytes / 2 / (int)sizeof(T);  // elements per row per stage
    constexpr int TPS = SE / kTile;                            // tiles per stage
    constexpr int VPR = kDrawStageBytes / 2 / 16;              // 16-byte vectors per row per stage
    constexpr int VW = 16 / (int)sizeof(T);
    const int nstage = (vend - v0 + SE - 1) / SE;
    auto issue = [&](int k) {
      if (k < nstage) {
        uint4* dst = ring + (size_t)(k % kDrawStages) * (kDrawStageBytes / 16);
        const int base = v0 + k * SE;
#pragma unroll
        for (int i = t; i < 2 * VPR; i += kThreads) {
          const bool isq = i >= VPR;
          const int e = base + (isq ? i - VPR : i) * VW;
          const bool ok = e < vend && (!isq || d.resid);
          const T* row = isq ? qr : pr;
          cp_async16(dst + i, ok ? row + e : row, ok ? 16 : 0);
        }
      }
      cp_async_commit();
    };
#pragma unroll
    for (int k = 0; k < kDrawStages; ++k) issue(k);
    for (int k = 0; k < nstage; ++k) {
      cp_async_wait<kDrawStages - 1>();
      __syncthreads();  // every thread's copies of stage k are in shared memory
      const uint4* st = ring + (size_t)(k % kDrawStages) * (kDrawStageBytes / 16);
      for (int ti = warp; ti < TPS; ti += kWarps) {
        const int tile = k * TPS + ti;
        if (tile >= ntile) break;
        float zp[8], zq[8];
        const int e0 = v0 + tile * kTile + lane * 8;
        if (sizeof(T) == 2) {
          const uint4 a = st[ti * 32 + lane], b = st[VPR + ti * 32 + lane];
          const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            zp[2 * q4] = bf16_lo(wa[q4]);
            zp[2 * q4 + 1] = bf16_hi(wa[q4]);
            zq[2 * q4] = bf16_lo(wb[q4]);
            zq[2 * q4 + 1] = bf16_hi(wb[q4]);
          }
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 a = st[ti * 64 + lane * 2 + h], b = st[VPR + ti * 64 + lane * 2 + h];
            zp[4 * h] = __uint_as_float(a.x);
            zp[4 * h + 1] = __uint_as_float(a.y);
            zp[4 * h + 2] = __uint_as_float(a.z);
            zp[4 * h + 3] = __uint_as_float(a.w);
            zq[4 * h] = __uint_as_float(b.x);
            zq[4 * h + 1] = __uint_as_float(b.y);
            zq[4 * h + 2] = __uint_as_float(b.z);
            zq[4 * h + 3] = __uint_as_float(b.w);
          }
        }
        if (e0 + 8 > vend) {  // the range's last, partial tile: logits past it carry no mass
#pragma unroll
          for (int q8 = 0; q8 < 8; ++q8)
            if (e0 + q8 >= vend) zp[q8] = zq[q8] = -INFINITY;
        }
        float w[8];
        weights_of<MASK>(zp, zq, d, P.c2, w);
        float sum = 0.0f;
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) sum += w[q8];
        sum = warp_sum(sum);
        if (lane == 0) wt[tile] = sum;
      }
      __syncthreads();  // stage k fully read: its slot may be refilled
      issue(k + kDrawStages);
    }
    cp_async_wait<0>();
  } else {
    for (int i0 = warp; i0 < ntile; i0 += kWarps * kUnrollA) {
      float w[kUnrollA][8];
#pragma unroll
      for (int u4 = 0; u4 < kUnrollA; ++u4) {
        int i = i0 + u4 * kWarps;
        if (i < ntile)
          weights8<T, VEC, MASK>(pr, qr, v0 + i * kTile + lane * 8, V, d, P.c2, w[u4]);
        else
#pragma unroll
          for (int k = 0; k < 8; ++k) w[u4][k] = 0.0f;
      }
#pragma unroll
      for (int u4 = 0; u4 < kUnrollA; ++u4) {
        int i = i0 + u4 * kWarps;
        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) s += w[u4][k];
        s = warp_sum(s);
        if (lane == 0 && i < ntile) wt[i] = s;
      }
    }
  }
  }  // phase != 2
  __syncthreads();  // every tile sum written
  // segments of tiles per thread, then a block inclusive scan of the segment sums
  const int L = (ntile + kThreads - 1) / kThreads;
  const int s0 = t * L, s1 = min(s0 + L, ntile);
  float incl;
  if (phase != 2) {
    float seg = 0.0f;
    for (int i = s0; i < s1; ++i) seg += wt[i];
    float x = seg;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      float y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) sm.red_s[warp] = x;
    if (t == 0) sm.seg_first = kThreads;
    __syncthreads();
    float off = 0.0f;
    for (int w = 0; w < warp; ++w) off += sm.red_s[w];
    incl = x + off;
    sm.incl[t] = incl;
    if (t == kThreads - 1) sm.total = incl;
  } else {
    incl = sm.incl[t];
    if (t == 0) sm.seg_first = kThreads;
  }
  __syncthreads();
  const float total = sm.total;
  if (!(total > 0.0f) || phase == 1) return total;  // caller handles an empty residual
  const float R = full ? total : Rm;
  const float target = full ? u * total : target_in;
  if (target < incl) atomicMin(&sm.seg_first, t);
  if (t == 0) sm.found = 0;
  __syncthreads();
  const int tf = sm.seg_first;
  if (t == (tf == kThreads ? 0 : tf)) {
    int found = -1;
    float run = 0.0f;
    if (tf < kThreads) {
      run = t == 0 ? 0.0f : sm.incl[t - 1];
      for (int i = s0; i < s1; ++i) {
        if (target < run + wt[i]) {
          found = i;
          break;
        }
        run += wt[i];
      }
    }
    if (found >= 0) {
      sm.tile = found;
      sm.tile_base = run;
      sm.found = 1;
    } else {
      // rounding left the target past the sums: the last tile with mass before the limit
      const int lim = tf < kThreads ? s1 : ntile;
      int i = lim - 1;
      while (i >= 0 && !(wt[i] > 0.0f)) --i;
      if (i < 0) {
        i = lim;
        while (i < ntile - 1 && !(wt[i] > 0.0f)) ++i;
      }
      float base = 0.0f;
      for (int j = 0; j < i; ++j) base += wt[j];
      sm.tile = i;
      sm.tile_base = base;
      sm.found = 2;
    }
  }
  __syncthreads();
  // inside the tile: one warp, 8 logits per lane
  if (warp == 0) {
    const int tile = sm.tile;
    const float tbase = sm.tile_base;
    bool clamped = sm.found == 2;
    float w[8];
    weights8<T, VEC, MASK>(pr, qr, v0 + tile * kTile + lane * 8, V, d, P.c2, w);
    float ls = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) ls += w[k];
    float li = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      float y = __shfl_up_sync(0xFFFFFFFFu, li, o);
      if (lane >= o) li += y;
    }
    float le = __shfl_up_sync(0xFFFFFFFFu, li, 1);
    if (lane == 0) le = 0.0f;
    const float tl = target - tbase;
    unsigned hit = clamped ? 0u : __ballot_sync(0xFFFFFFFFu, tl < li);
    int yl, ye = -1;
    float run, margin = 0.0f;
    if (hit) {
      yl = __ffs(hit) - 1;
      if (lane == yl) {
        run = le;
        for (int k = 0; k < 8; ++k) {
          if (tl < run + w[k]) {
            ye = k;
            margin = fminf(tl - run, run + w[k] - tl) / R;
            break;
          }
          run += w[k];
        }
        if (ye < 0) {  // sub-ulp disagreement between levels: last logit with mass in the lane
          for (int k = 7; k >= 0; --k)
            if (w[k] > 0.0f) {
              ye = k;
              break;
            }
          margin = 0.0f;
          clamped = true;
        }
      }
    } else {
      unsigned pos = __ballot_sync(0xFFFFFFFFu, ls > 0.0f);
      yl = pos ? 31 - __clz(pos) : 0;
      if (lane == yl) {
        for (int k = 7; k >= 0; --k)
          if (w[k] > 0.0f) {
            ye = k;
            break;
          }
        if (ye < 0) ye = 0;
      }
      clamped = true;
    }
    if (lane == yl) {
      sm.y = v0 + tile * kTile + yl * 8 + ye;
      sm.margin = clamped ? 0.0f : margin;
      if (clamped) *clamp = 1;
    }
  }
  __syncthreads();
  return total;
}

// Row threshold, max and sum for top-k from the chunks' candidates.  One warp per row.
// Returns false if the row needs the exact full-row path (candidate overflow).
template <typename T>
__device__ bool topk_row_fast(const Params& P, int b, int rp, uint2* buf, float& M, float& S,
                              float& thr, int& flags) {
  const float c2 = rp > P.K ? P.c2q : P.c2;
  const int lane = threadIdx.x & 31;
  const int nch = P.nchunk;
  const uint2* meta = P.cmeta + ((size_t)b * P.R + rp) * nch;
  const uint2* cand = P.cand + ((size_t)b * P.R + rp) * nch * (size_t)kCandCap;
  bool ovf = false, nan = false;
  for (int c = lane; c < nch; c += 32) {
    const uint2 mt = __ldcg(meta + c);
    ovf |= (mt.y & kMetaOverflow) != 0;
    nan |= (mt.y & kMetaNaN) != 0;
  }
  ovf = __any_sync(0xFFFFFFFFu, ovf);
  nan = __any_sync(0xFFFFFFFFu, nan);
  if (nan) flags |= SPEC_FLAG_NONFINITE;
  if (ovf) return false;
  const int k = P.top_k;
  // Only the chunks where a block's row segment starts hold a list (sorted, key descending); the
  // lists are read by the whole warp, 32 entries per load, one list at a time.
  // Lower bound L on the row's k-th largest: pool the m = ceil(k / nch) largest keys of every
  // chunk's list; the pool's k-th largest has >= k distinct logits at or above it.
  const int m = (k + nch - 1) / nch;
  int np = 0;
  for (int c0 = 0; c0 < nch; c0 += 32) {
    const int cnt = c0 + lane < nch ? (int)(__ldcg(&meta[c0 + lane].y) & kMetaCount) : 0;
    for (unsigned has = __ballot_sync(0xFFFFFFFFu, cnt > 0); has; has &= has - 1) {
      const int l = __ffs(has) - 1;
      const int take = min(m, __shfl_sync(0xFFFFFFFFu, cnt, l));
      for (int i = lane; i < take; i += 32)
        if (np + i < kRowCap) buf[np + i] = __ldcg(cand + (size_t)(c0 + l) * kCandCap + i);
      np += take;
    }
  }
  if (np > kRowCap) return false;
  __syncwarp();
  uint32_t Lk = 0;
  if (np >= k) {  // the k-th largest pooled key, by counting (ties share a rank)
    uint32_t cand_k = 0;
    for (int i = lane; i < np; i += 32) {
      const uint32_t ki = buf[i].x;
      int greater = 0;
      for (int j = 0; j < np; ++j) greater += buf[j].x > ki;
      if (greater < k) cand_k = cand_k == 0 ? ki : min(cand_k, ki);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, cand_k, o);
      cand_k = cand_k == 0 ? y : (y == 0 ? cand_k : min(cand_k, y));
    }
    Lk = cand_k;
  }
  __syncwarp();
  // gather every candidate >= L: a prefix of each chunk's sorted list
  int n = 0;
  for (int c0 = 0; c0 < nch; c0 += 32) {
    const int cnt = c0 + lane < nch ? (int)(__ldcg(&meta[c0 + lane].y) & kMetaCount) : 0;
    for (unsigned has = __ballot_sync(0xFFFFFFFFu, cnt > 0); has; has &= has - 1) {
      const int l = __ffs(has) - 1;
      const int cn = __shfl_sync(0xFFFFFFFFu, cnt, l);
      const uint2* lst = cand + (size_t)(c0 + l) * kCandCap;
      for (int i0 = 0; i0 < cn; i0 += 32) {
        const int i = i0 + lane;
        const uint2 e = i < cn ? __ldcg(lst + i) : make_uint2(0u, 0u);
        const bool keep = i < cn && e.x >= Lk;
        const unsigned mk = __ballot_sync(0xFFFFFFFFu, keep);
        const int pos = n + __popc(mk & ((1u << lane) - 1u));
        if (keep && pos < kRowCap) buf[pos] = e;
        n += __popc(mk);
        if (mk != 0xFFFFFFFFu) break;  // sorted: the rest lie below L (or past the list)
      }
    }
  }
  if (n > kRowCap) return false;
  __syncwarp();
  // exact k-th largest among the gathered candidates
  uint32_t kth = 0xFFFFFFFFu, mx = 0;
  for (int i = lane; i < n; i += 32) {
    uint32_t ki = buf[i].x;
    int greater = 0;
    for (int j = 0; j < n; ++j) greater += buf[j].x > ki;
    if (greater < k) kth = min(kth, ki);
    mx = max(mx, ki);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kth = min(kth, __shfl_xor_sync(0xFFFFFFFFu, kth, o));
    mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  }
  if (n == 0) return false;
  M = keyf(mx);
  thr = keyf(kth);
  float s = 0.0f;
  int kept = 0;
  for (int i = lane; i < n; i += 32) {
    if (buf[i].x >= kth) {
      s += ex2((keyf(buf[i].x) - M) * c2);
      ++kept;
    }
  }
  S = warp_sum(s);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kept += __shfl_xor_sync(0xFFFFFFFFu, kept, o);
  if (kept > k) flags |= SPEC_FLAG_TOPK_TIE;
  return true;
}

// Exact top-k statistics of a whole row by radix selection over the row (whole CTA).
template <typename T, bool VEC>
__device__ void topk_row_exact(const Params& P, const T* row, float c2, uint32_t* hist, Smem& sm,
                               float& M, float& S, float& thr, int& flags) {
  const int t = threadIdx.x;
  const int V = P.V, k = P.top_k;
  uint32_t prefix = 0, mask = 0;
  int kk = k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = t; i < 256; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int e = t; e < V; e += kThreads) {
      float z = load1<T>(row + e);
      if (z != z) continue;
      uint32_t key = fkey(z);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (t == 0) {
      int acc = 0, d = 255;
      for (; d > 0; --d) {
        if (acc + (int)hist[d] >= kk) break;
        acc += (int)hist[d];
      }
      sm.red_c[0] = d;
      sm.red_c[1] = kk - acc;
    }
    __syncthreads();
    prefix |= (uint32_t)sm.red_c[0] << shift;
    mask |= 255u << shift;
    kk = sm.red_c[1];
    __syncthreads();
  }
  thr = keyf(prefix);
  // max and sum over the kept set
  float m = -INFINITY;
  for (int e = t; e < V; e += kThreads) {
    float z = load1<T>(row + e);
    if (z >= thr) m = fmaxf(m, z);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((t & 31) == 0) sm.red_m[t >> 5] = m;
  __syncthreads();
  m = -INFINITY;
  for (int w = 0; w < kWarps; ++w) m = fmaxf(m, sm.red_m[w]);
  float s = 0.0f;
  int kept = 0;
  for (int e = t; e < V; e += kThreads) {
    float z = load1<T>(row + e);
    if (z >= thr) {
      s += ex2((z - m) * c2);
      ++kept;
    }
  }
  s = warp_sum(s);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kept += __shfl_xor_sync(0xFFFFFFFFu, kept, o);
  __syncthreads();
  if ((t & 31) == 0) {
    sm.red_s[t >> 5] = s;
    sm.red_c[t >> 5] = kept;
  }
  __syncthreads();
  s = 0.0f;
  kept = 0;
  for (int w = 0; w < kWarps; ++w) {
    s += sm.red_s[w];
    kept += sm.red_c[w];
  }
  M = m;
  S = s;
  if (kept > k) flags |= SPEC_FLAG_TOPK_TIE;
  __syncthreads();
}

// Nucleus (top-p) of one row, after its temperature and its top-k threshold `thr`: the smallest
// set of most likely logits whose mass reaches top_p of the row's kept mass S, with the whole tie
// group at the cut (gsyq.cn §3.3 names top_p among the parameters both sides share).  Every
// logit's weight w = 2^x, x = (z - M) * c2, and its bucket, floor(-2x) capped at 31 (half a
// binade per bucket; bucket 31 is the tail, w < 2^-15.5), are computed the same way everywhere,
// so all steps agree on them.  The tail's mass is S less the other buckets.
//   Common path (nucleus_row): one read of the row lists the head logits (buckets 0..30, a few
//   percent of a long row) in shared memory; their buckets give the one holding the cut; its
//   logits, sorted by key, give the exact cut (nuc_select).
//   Multi-pass path, when the head does not fit, the cut lies in the tail, or its bucket holds
//   more than kNucCap logits: one pass bins every logit by bucket, each thread in its own column
//   of shared memory (no atomics); then the bucket holding the cut is split by 4-bit digits of
//   the key, one pass per digit, until the part holding the cut fits kNucCap (or is one key);
//   a last pass gathers it for nuc_select.
constexpr int kNucBins = 32;
constexpr int kNucCap = 2048;
constexpr size_t kNucBytes = (size_t)kNucBins * kThreads * (sizeof(float) + sizeof(uint16_t));

// The bucket of a logit: floor(-2x), x = (z - M) * c2 <= 0, capped at the tail bucket.
__device__ __forceinline__ int nuc_bucket_of(float z, float M, float c2) {
  return min(kNucBins - 1, __float2int_rd(-2.0f * ((z - M) * c2)));  // z <= M: never negative
}

struct NucSel {     // which logits the current pass looks at
  int bucket;       // level-0 bucket (-1: all kept logits)
  uint32_t mask;    // key bits fixed by the digit levels so far
  uint32_t prefix;  // their value
};


// One pass over the row: per-thread bins (mass, count) of the selected logits, by level-0 bucket
// (shift < 0) or by the key digit at `shift`; or, with `gather`, the selected logits themselves.
template <typename T, bool VEC>
__device__ __forceinline__ void nuc_pass(const Params& P, const T* row, float M, float c2, uint32_t kthr,
                                         const NucSel& sel, int shift, bool gather, unsigned char* nbuf,
                                         Smem& sm) {
  const int t = threadIdx.x, lane = t & 31;
  float* mass = reinterpret_cast<float*>(nbuf);
  uint16_t* cnt = reinterpret_cast<uint16_t*>(nbuf + (size_t)kNucBins * kThreads * sizeof(float));
  uint32_t* gk = reinterpret_cast<uint32_t*>(nbuf);
  float* gw = reinterpret_cast<float*>(nbuf + (size_t)kNucCap * sizeof(uint32_t));
  if (!gather) {
#pragma unroll
    for (int b = 0; b < kNucBins; ++b) {
      mass[b * kThreads + t] = 0.0f;
      cnt[b * kThreads + t] = 0;
    }
  } else if (t == 0) {
    sm.nuc_n = 0;
  }
  const bool level0 = !gather && shift < 0;
  uint32_t tail = 0;  // level 0: logits in the tail bucket, counted in a register
  __syncthreads();
  for (int c = 0; c < P.nchunk; ++c) {
    const int v0 = c * Cfg<T>::CH;
    float v[Cfg<T>::PER];
    load_chunk<T, VEC>(row + v0, min(Cfg<T>::CH, P.V - v0), v);
#pragma unroll
    for (int i = 0; i < Cfg<T>::PER; ++i) {
      const uint32_t k = fkey(v[i]);
      const float x = (v[i] - M) * c2;
      const int bk = nuc_bucket_of(v[i], M, c2);
      const bool in = v[i] > -INFINITY && k >= kthr && (sel.bucket < 0 || bk == sel.bucket) &&
                      (k & sel.mask) == sel.prefix;
      if (!gather) {
        if (in && level0 && bk == kNucBins - 1) {
          ++tail;
        } else if (in) {
          const int bin = level0 ? bk : (int)((k >> shift) & 15u);
          mass[bin * kThreads + t] += ex2(x);
          cnt[bin * kThreads + t] += 1;
        }
      } else {
        const unsigned m = __ballot_sync(0xFFFFFFFFu, in);
        if (m) {
          int base = 0;
          if (lane == __ffs(m) - 1) base = atomicAdd(&sm.nuc_n, __popc(m));
          base = __shfl_sync(0xFFFFFFFFu, base, __ffs(m) - 1);
          const int idx = base + __popc(m & ((1u << lane) - 1u));
          if (in && idx < kNucCap) {
            gk[idx] = k;
            gw[idx] = ex2(x);
          }
        }
      }
    }
  }
  if (level0) cnt[(kNucBins - 1) * kThreads + t] = (uint16_t)tail;
  __syncthreads();
}

// Bins of the last pass summed over threads; warp 0 finds the bin where the mass counted from the
// top (bin 0 first; for digits, the highest digit first) first reaches the target, or, if
// rounding leaves the target unreached, the lowest bin with mass.  Results in sm.nuc_*.
__device__ __forceinline__ void nuc_pick(unsigned char* nbuf, Smem& sm, int nbins, bool digits, float above,
                                         bool level0, float top_p, float S) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const float* mass = reinterpret_cast<const float*>(nbuf);
  const uint16_t* cnt = reinterpret_cast<const uint16_t*>(nbuf + (size_t)kNucBins * kThreads * sizeof(float));
  for (int b = warp; b < nbins; b += kWarps) {
    float s = 0.0f;
    uint32_t n = 0;
    for (int j = lane; j < kThreads; j += 32) {
      s += mass[b * kThreads + j];
      n += cnt[b * kThreads + j];
    }
    s = warp_sum(s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xFFFFFFFFu, n, o);
    if (lane == 0) {
      sm.incl[b] = s;
      sm.red_cnt[b] = n;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // lane l takes the l-th bin in order from the top
    const int b = digits ? nbins - 1 - lane : lane;
    float s = lane < nbins ? sm.incl[b] : 0.0f;
    if (level0) {  // the tail's mass is what the other buckets leave of S
      const float head = warp_sum(lane < kNucBins - 1 ? s : 0.0f);
      if (lane == kNucBins - 1) s = fmaxf(S - head, 0.0f);
      if (lane == 0) sm.nuc_target = top_p * S;
    }
    __syncwarp();
    const float target = sm.nuc_target;
    float incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, lane < nbins && above + incl >= target);
    const unsigned nz = __ballot_sync(0xFFFFFFFFu, s > 0.0f);
    const int L = hit ? __ffs(hit) - 1 : (nz ? 31 - __clz(nz) : 0);
    if (lane == L) {
      sm.nuc_digit = b;
      sm.nuc_above = above + incl - s;
      sm.nuc_bin = s;
      sm.nuc_count = sm.red_cnt[b];
    }
  }
  __syncthreads();
}

// Exact cut among n gathered logits (keys gk, weights gw, n <= kNucCap) that hold the cut, with
// `above` the mass of every kept logit above them: a bitonic sort by key, descending (in warp 0's
// registers when n <= 32, the usual size of a boundary sub-bucket), then a scan from the top to the
// first tie group where the mass reaches the target.  Leaves the nucleus mass in sm.nuc_above and
// the cut key in sm.nuc_key.
__device__ __forceinline__ void nuc_select(uint32_t* gk, float* gw, int n, float above, float target, Smem& sm) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (n <= 32) {  // one logit per lane of warp 0: a bitonic sort by shuffles, no block barrier
    if (warp == 0) {
      uint32_t k = lane < n ? gk[lane] : 0u;  // key 0: below every real key, sorts last
      float w = lane < n ? gw[lane] : 0.0f;
#pragma unroll
      for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
        for (int j = kk >> 1; j > 0; j >>= 1) {
          const uint32_t ok = __shfl_xor_sync(0xFFFFFFFFu, k, j);
          const float ow = __shfl_xor_sync(0xFFFFFFFFu, w, j);
          const bool take_max = ((lane & kk) == 0) == ((lane & j) == 0);  // descending overall
          if (take_max ? ok > k : ok < k) {
            k = ok;
            w = ow;
          }
        }
      }
      float incl = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, lane < n && above + incl >= target);
      // rounding left the target unreached: keep everything gathered
      const int at = hit ? __ffs(hit) - 1 : n - 1;
      const uint32_t kc = __shfl_sync(0xFFFFFFFFu, k, at);
      // the nucleus mass: everything above, and every gathered logit down to the whole tie group
      const float kept = warp_sum(lane < n && k >= kc ? w : 0.0f);
      if (lane == 0) {
        sm.nuc_above = above + kept;
        sm.nuc_key = kc;
      }
    }
    __syncthreads();
    return;
  }
  int N = 32;
  while (N < n) N <<= 1;
  for (int i = n + t; i < N; i += kThreads) {
    gk[i] = 0u;  // below every real key: sorts last
    gw[i] = 0.0f;
  }
  __syncthreads();
  for (int k = 2; k <= N; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = t; i < N; i += kThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool desc = (i & k) == 0;
          const uint32_t a = gk[i], b = gk[ixj];
          if (desc ? (a < b) : (a > b)) {
            gk[i] = b;
            gk[ixj] = a;
            const float wa = gw[i];
            gw[i] = gw[ixj];
            gw[ixj] = wa;
          }
        }
      }
      __syncthreads();
    }
  }
  if (warp == 0) {
    float cum = above;
    int at = -1;
    for (int base = 0; base < n && at < 0; base += 32) {
      const int i = base + lane;
      const float w = i < n ? gw[i] : 0.0f;
      float incl = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, i < n && cum + incl >= target);
      if (hit) {
        const int L = __ffs(hit) - 1;
        at = base + L;
        cum += __shfl_sync(0xFFFFFFFFu, incl, L);
      } else {
        cum += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
    }
    if (lane == 0) {
      if (at < 0) at = n - 1;  // rounding left the target unreached: keep everything gathered
      const uint32_t kc = gk[at];
      for (int i = at + 1; i < n && gk[i] == kc; ++i) cum += gw[i];  // the rest of the tie group
      sm.nuc_above = cum;
      sm.nuc_key = kc;
    }
  }
  __syncthreads();
}

// Shared-memory layout of the nucleus search (kNucBufBytes): the common path keeps the row's head
// logits in per-thread columns (entry i of thread t at i * kThreads + t, in the row's own type)
// followed by per-thread bins that later hold the sort area; the multi-pass path reuses the same
// bytes for its bins and gathers.  The common path's buckets are whole binades of the weight:
// hb = floor(-x) capped at 15 (the tail, w < 2^-15), then 16 sub-buckets of the chosen one.
constexpr int kHeadBins = 16;
constexpr int kHeadSpanFirst = 13;  // binades of the weight listed by the first read of a row
constexpr size_t kNucListBytes = 49152;
constexpr size_t kNucBinBytes = (size_t)kHeadBins * kThreads * sizeof(float);
constexpr size_t kNucBufBytes = kNucListBytes + kNucBinBytes;
static_assert(kNucBufBytes >= kNucBytes, "nucleus buffer");
static_assert(kNucBinBytes >= (size_t)kNucCap * (sizeof(uint32_t) + sizeof(float)), "nucleus sort area");

// Per-thread bins (column t of `bins`, nbins <= 32) summed over the block; warp 0 walks them from
// bin 0 (the heaviest weights) and picks the bin where `above` plus the mass so far first reaches
// the target.  With `tail_from_S`, the last bin's mass is S less the others.  Results in sm.nuc_*.
__device__ __forceinline__ void nuc_walk_bins(const float* bins, int nbins, Smem& sm, float above, float target,
                                              bool tail_from_S, float S) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int b = warp; b < nbins; b += kWarps) {
    float s = 0.0f;
#pragma unroll
    for (int j = lane; j < kThreads; j += 32) s += bins[b * kThreads + j];
    s = warp_sum(s);
    if (lane == 0) sm.incl[b] = s;
  }
  __syncthreads();
  if (warp == 0) {
    float s = lane < nbins ? sm.incl[lane] : 0.0f;
    if (tail_from_S) {
      const float head = warp_sum(lane < nbins - 1 ? s : 0.0f);
      if (lane == nbins - 1) s = fmaxf(S - head, 0.0f);
    }
    float incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, lane < nbins && above + incl >= target);
    const unsigned nz = __ballot_sync(0xFFFFFFFFu, s > 0.0f);
    const int L = hit ? __ffs(hit) - 1 : (nz ? 31 - __clz(nz) : 0);
    if (lane == L) {
      sm.nuc_digit = L;
      sm.nuc_above = above + incl - s;
      sm.nuc_bin = s;
    }
    if (lane == 0) sm.nuc_n = 0;
  }
  __syncthreads();
}

// S is the row's kept mass relative to M (before top-p).  Returns the nucleus mass relative to M
// and the cut as a logit value.  All threads of the block call it; `nbuf` is kNucBufBytes of
// shared memory.
template <typename T, bool VEC>
__device__ __forceinline__ void nucleus_row(const Params& P, const T* row, float M, float c2, float thr, float S,
                                            unsigned char* nbuf, Smem& sm, float& S_kept, float& cut) {
  const int t = threadIdx.x;
  const float target = P.top_p * S;
  // ---- common path: one read of the row lists the head logits in per-thread columns ----
  constexpr int kCap = (int)(kNucListBytes / sizeof(T) / kThreads);
  float* bins = reinterpret_cast<float*>(nbuf + kNucListBytes);
  // Each thread appends to its own column (entry i at byte (i * kThreads + t) * sizeof(T)) through a
  // running offset.  A chunk adds at most PER entries, so a column found full before a chunk is
  // wound back to its last entry and can only run on into the bins behind the list (free until
  // the list has been read), by less than PER rows of the columns; its row takes the multi-pass
  // path.
  constexpr uint32_t kStride = kThreads * sizeof(T);
  static_assert((size_t)Cfg<T>::PER * kStride <= kNucBinBytes, "a chunk's overrun stays in the bins");
  const uint32_t col0 = t * (uint32_t)sizeof(T), col_end = col0 + (uint32_t)kCap * kStride;
  // Every head logit of the current span (binade hb < span) lies above zcut: the bound
  // M - span / c2, widened by a relative 1e-4 against rounding, or the top-k threshold if that is
  // higher.  A listed logit whose bucket turns out to be the tail is ignored below.
  float zcut = 0.0f;
  uint32_t zc2 = 0u;
  uint32_t wp = col0;
  bool crowded = false;
  auto scan = [&](const float (&v)[Cfg<T>::PER]) {
    if (wp >= col_end) {
      crowded = true;
      wp = col_end - kStride;
    }
#pragma unroll
    for (int i = 0; i < Cfg<T>::PER; ++i) {
      if (v[i] > zcut) {
        if (sizeof(T) == 2)
          *reinterpret_cast<uint16_t*>(nbuf + wp) = (uint16_t)(__float_as_uint(v[i]) >> 16);
        else
          *reinterpret_cast<float*>(nbuf + wp) = v[i];
        wp += kStride;
      }
    }
  };
  // bf16 logits are compared in pairs against the largest bf16 value <= zcut (no bf16 value lies
  // between the two, so z > zcut is z > that value)
  auto scan_raw = [&](const uint4 (&raw)[Cfg<T>::LOADS], int nn) {
    if (wp >= col_end) {
      crowded = true;
      wp = col_end - kStride;
    }
#pragma unroll
    for (int l = 0; l < Cfg<T>::LOADS; ++l) {
      if ((l * kThreads + t) * Cfg<T>::VW >= nn) continue;  // past the row (tail chunk)
      const uint32_t w[4] = {raw[l].x, raw[l].y, raw[l].z, raw[l].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t m = __hgt2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w[k]),
                                       *reinterpret_cast<const __nv_bfloat162*>(&zc2));
        if (m & 0xFFFFu) {
          *reinterpret_cast<uint16_t*>(nbuf + wp) = (uint16_t)w[k];
          wp += kStride;
        }
        if (m >> 16) {
          *reinterpret_cast<uint16_t*>(nbuf + wp) = (uint16_t)(w[k] >> 16);
          wp += kStride;
        }
      }
    }
  };
  auto scan_vec = [&](const uint4 (&raw)[Cfg<T>::LOADS], int nn) {
    if (sizeof(T) == 2) {
      scan_raw(raw, nn);
    } else {
      float v[Cfg<T>::PER];
      unpack<T>(raw, nn, v);
      scan(v);
    }
  };
  auto entry = [&](int i) -> float {
    return sizeof(T) == 2 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(nbuf)[i * kThreads + t] << 16)
                          : reinterpret_cast<const float*>(nbuf)[i * kThreads + t];
  };
  // the binade and sub-bucket of a listed logit, from -x exactly as its weight 2^x is formed
  auto hbin = [&](float nx) { return min(kHeadBins - 1, __float2int_rd(nx)); };
  auto sbin = [&](float nx, int hb) { return min(kHeadBins - 1, __float2int_rd((nx - (float)hb) * 16.0f)); };
  // The head is listed first down to 2^-kHeadSpanFirst of the max's weight (on rows like these
  // the cut lies well inside, and a shorter list is searched faster); a cut below that span is
  // looked for again in a second read down to 2^-15 before the multi-pass search.
  for (int span = kHeadSpanFirst;; span = kHeadBins - 1) {
    zcut = fmaxf(M - ((float)span / c2) * 1.0001f, thr == -INFINITY ? -FLT_MAX : nextafterf(thr, -INFINITY));
    if (sizeof(T) == 2) {  // the largest bf16 value <= zcut, in both halves
      const uint32_t zb = __float_as_uint(zcut);
      uint32_t h = zb >> 16;
      if ((zb & 0xFFFFu) != 0u && (zb >> 31)) ++h;  // negative: rounding the magnitude up rounds down
      zc2 = h | (h << 16);
    }
    wp = col0;
    crowded = false;
    if (VEC) {  // two chunks' loads in flight ahead of the one being scanned
      uint4 r0[Cfg<T>::LOADS], r1[Cfg<T>::LOADS];
      load_raw<T>(row, min(Cfg<T>::CH, P.V), r0);
      if (P.nchunk > 1) load_raw<T>(row + Cfg<T>::CH, min(Cfg<T>::CH, P.V - Cfg<T>::CH), r1);
      for (int c = 0; c < P.nchunk; ++c) {
        const int v0 = c * Cfg<T>::CH;
        uint4 cur[Cfg<T>::LOADS];
#pragma unroll
        for (int l = 0; l < Cfg<T>::LOADS; ++l) {
          cur[l] = r0[l];
          r0[l] = r1[l];
        }
        if (c + 2 < P.nchunk) load_raw<T>(row + v0 + 2 * Cfg<T>::CH, min(Cfg<T>::CH, P.V - v0 - 2 * Cfg<T>::CH), r1);
        scan_vec(cur, min(Cfg<T>::CH, P.V - v0));
      }
    } else {
      for (int c = 0; c < P.nchunk; ++c) {
        const int v0 = c * Cfg<T>::CH;
        float v[Cfg<T>::PER];
        load_chunk<T, VEC>(row + v0, min(Cfg<T>::CH, P.V - v0), v);
        scan(v);
      }
    }
    const int cnt = crowded ? kCap + 1 : (int)((wp - col0) / kStride);
    const bool overflow = __syncthreads_or(cnt > kCap);
    bool done = false, deeper = false;
    if (!overflow) {
#pragma unroll
      for (int b = 0; b < kHeadBins; ++b) bins[b * kThreads + t] = 0.0f;
      for (int i = 0; i < cnt; ++i) {
        const float z = entry(i);
        const float x = (z - M) * c2;
        const int hb = hbin(-x);
        if (hb < span) bins[hb * kThreads + t] += ex2(x);
      }
      __syncthreads();
      nuc_walk_bins(bins, span + 1, sm, 0.0f, target, true, S);
      const int bsel = sm.nuc_digit;
      deeper = bsel >= span;  // uniform: read after the walk's barrier
      if (!deeper) {
        const float above1 = sm.nuc_above;
#pragma unroll
        for (int b = 0; b < kHeadBins; ++b) bins[b * kThreads + t] = 0.0f;
        for (int i = 0; i < cnt; ++i) {
          const float z = entry(i);
          const float x = (z - M) * c2;
          if (hbin(-x) == bsel) bins[sbin(-x, bsel) * kThreads + t] += ex2(x);
        }
        __syncthreads();
        nuc_walk_bins(bins, kHeadBins, sm, above1, target, false, 0.0f);
        const int ssel = sm.nuc_digit;
        const float above2 = sm.nuc_above;
        // gather the chosen sub-bucket into the sort area (the bins are consumed)
        uint32_t* sk = reinterpret_cast<uint32_t*>(bins);
        float* sw = bins + kNucCap;
        for (int i = 0; i < cnt; ++i) {
          const float z = entry(i);
          const float x = (z - M) * c2;
          if (hbin(-x) == bsel && sbin(-x, bsel) == ssel) {
            const int idx = atomicAdd(&sm.nuc_n, 1);
            if (idx < kNucCap) {
              sk[idx] = fkey(z);
              sw[idx] = ex2(x);
            }
          }
        }
        __syncthreads();
        const int n = sm.nuc_n;
        if (n <= kNucCap) {
          nuc_select(sk, sw, n, above2, target, sm);
          done = true;
        }
      }
    }
    if (done) {
      S_kept = sm.nuc_above;
      cut = keyf(sm.nuc_key);
      __syncthreads();
      return;
    }
    __syncthreads();
    if (!deeper || span == kHeadBins - 1) break;
  }
  // ---- multi-pass path: a crowded head, a cut in the tail, or a large boundary bucket ----
  const uint32_t kthr = thr == -INFINITY ? 0u : fkey(thr);  // keys below it are outside top-k
  NucSel sel{-1, 0u, 0u};
  nuc_pass<T, VEC>(P, row, M, c2, kthr, sel, -1, false, nbuf, sm);
  nuc_pick(nbuf, sm, kNucBins, false, 0.0f, true, P.top_p, S);
  sel.bucket = sm.nuc_digit;
  float above = sm.nuc_above, binmass = sm.nuc_bin;
  uint32_t count = sm.nuc_count;
  bool exact_key = false;
  for (int shift = 28; count > (uint32_t)kNucCap; shift -= 4) {
    if (shift < 0) {  // every logit left has the same key: that key is the cut
      exact_key = true;
      break;
    }
    __syncthreads();
    nuc_pass<T, VEC>(P, row, M, c2, kthr, sel, shift, false, nbuf, sm);
    nuc_pick(nbuf, sm, 16, true, above, false, P.top_p, 0.0f);
    sel.mask |= 15u << shift;
    sel.prefix |= (uint32_t)sm.nuc_digit << shift;
    above = sm.nuc_above;
    binmass = sm.nuc_bin;
    count = sm.nuc_count;
  }
  if (exact_key) {
    S_kept = above + binmass;
    cut = keyf(sel.prefix);
    __syncthreads();
    return;
  }
  __syncthreads();
  nuc_pass<T, VEC>(P, row, M, c2, kthr, sel, 0, true, nbuf, sm);
  const int n = min((int)count, sm.nuc_n);
  nuc_select(reinterpret_cast<uint32_t*>(nbuf), reinterpret_cast<float*>(nbuf + (size_t)kNucCap * sizeof(uint32_t)),
             n, above, sm.nuc_target, sm);
  S_kept = sm.nuc_above;
  cut = keyf(sm.nuc_key);
  __syncthreads();
}

// Top-k draws over the kept set: p's kept tokens (key >= the row's threshold) are prefixes of row
// js's sorted chunk lists; their weights are those of draw_range (the residual max(0, P - Q), Q
// read at each token, or the target weights for a draw from p alone), and the inverse CDF runs
// over them sorted by token id, so it draws what the full-row pass draws (only the summation
// order differs).  Returns false (nothing drawn) if the kept set exceeds the list buffer
// (kWarps * kRowCap pairs); otherwise sets sm.y, sm.margin and *R_out.  Whole block.
template <typename T>
__device__ bool draw_list(const Params& P, int b, int js, const T* qr, const DrawRows& d, float u, uint2* lst,
                          Smem& sm, int* clamp, float* R_out) {
  constexpr int kCap = kWarps * kRowCap;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int nch = P.nchunk;
  const uint2* meta = P.cmeta + ((size_t)b * P.R + js) * nch;
  const uint2* cand = P.cand + ((size_t)b * P.R + js) * nch * (size_t)kCandCap;
  const uint32_t kt = fkey(d.Tp);
  // The prefix of chunk list c at or above the threshold (the lists are sorted, key descending),
  // read by the whole warp, 32 entries per load; with `out`, copied there.  Warps take the chunks
  // in turn; a block scan of the warps' totals places their copies.
  auto take_list = [&](int c, uint2* out) {
    const int cnt = (int)(__ldcg(&meta[c].y) & kMetaCount);
    const uint2* src = cand + (size_t)c * kCandCap;
    int n = 0;
    for (int i0 = 0; i0 < cnt; i0 += 32) {
      const int i = i0 + lane;
      const uint2 e = i < cnt ? __ldcg(src + i) : make_uint2(0u, 0u);
      const bool keep = i < cnt && e.x >= kt;
      const unsigned mk = __ballot_sync(0xFFFFFFFFu, keep);
      if (out && keep) out[n + __popc(mk & ((1u << lane) - 1u))] = e;
      n += __popc(mk);
      if (mk != 0xFFFFFFFFu) break;
    }
    return n;
  };
  int mine = 0;
  for (int c = warp; c < nch; c += kWarps) mine += take_list(c, nullptr);
  if (lane == 0) sm.red_i[warp] = mine;
  __syncthreads();
  int base = 0, n = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) base += sm.red_i[w];
    n += sm.red_i[w];
  }
  if (n > kCap || n == 0) {
    __syncthreads();
    return false;
  }
  for (int c = warp; c < nch; c += kWarps) base += take_list(c, lst + base);
  __syncthreads();
  // weights, as (token, weight bits)
  for (int i = t; i < n; i += kThreads) {
    const uint2 e = lst[i];
    const float zp = keyf(e.x);
    float w;
    if (d.resid) {
      const float pa = ex2(fmaf(zp, P.c2, -d.Lp));
      const float zq = load1<T>(qr + e.y);
      const float qa = zq >= d.Tq ? ex2(fmaf(zq, d.c2q, -d.Lq)) : 0.0f;
      w = fmaxf(pa - qa, 0.0f);
    } else {
      w = ex2(fmaf(zp, P.c2, -d.Mp2));
    }
    lst[i] = make_uint2(e.y, __float_as_uint(w));
  }
  __syncthreads();
  // order by token id: tokens are distinct, so each entry's place is the number of smaller ones
  // (up to kCap / 2 entries, into the buffer's upper half); a bitonic sort for more
  uint2* srt = lst;
  if (n <= kCap / 2) {
    srt = lst + kCap / 2;
    for (int i = t; i < n; i += kThreads) {
      const uint2 e = lst[i];
      int pos = 0;
      for (int j = 0; j < n; ++j) pos += lst[j].x < e.x;
      srt[pos] = e;
    }
    __syncthreads();
  } else {
    int N = 32;
    while (N < n) N <<= 1;
    for (int i = n + t; i < N; i += kThreads) lst[i] = make_uint2(0xFFFFFFFFu, 0u);  // sorts last
    __syncthreads();
    for (int k = 2; k <= N; k <<= 1) {  // bitonic sort by token id, ascending
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int i = t; i < N; i += kThreads) {
          const int ixj = i ^ j;
          if (ixj > i) {
            const uint2 a = lst[i], c = lst[ixj];
            if (((i & k) == 0) ? (a.x > c.x) : (a.x < c.x)) {
              lst[i] = c;
              lst[ixj] = a;
            }
          }
        }
        __syncthreads();
      }
    }
  }
  // cumulative sums in token order: each thread owns a run of consecutive entries
  constexpr int kPer = kCap / kThreads;
  const int i0 = t * kPer;
  float run = 0.0f;
#pragma unroll
  for (int j = 0; j < kPer; ++j)
    if (i0 + j < n) run += __uint_as_float(srt[i0 + j].y);
  float incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.red_s[warp] = incl;
  if (t == 0) {
    sm.y = -1;
    sm.margin = 0.0f;
  }
  __syncthreads();
  float before = incl - run, R = 0.0f;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) before += sm.red_s[w];
    R += sm.red_s[w];
  }
  const float target = u * R;
  float C = before;
  int last = -1;
  for (int j = 0; j < kPer; ++j) {
    const int i = i0 + j;
    if (i >= n) break;
    const float w = __uint_as_float(srt[i].y);
    const float prev = C;
    C += w;
    if (w > 0.0f) last = i;
    if (w > 0.0f && target >= prev && target < C) {
      sm.y = (int)srt[i].x;
      sm.margin = fminf(u - prev / R, C / R - u);
    }
  }
  // rounding put u * R at or past the total: the last token with weight, flagged
  __syncthreads();
  if (t == 0) sm.found = -1;
  __syncthreads();
  if (last >= 0) atomicMax(&sm.found, last);
  __syncthreads();
  if (t == 0 && sm.y < 0 && sm.found >= 0) {
    sm.y = (int)srt[sm.found].x;
    sm.margin = 0.0f;
    *clamp = 1;
  }
  __syncthreads();
  *R_out = R;
  return true;
}

// A draw over the whole row split across the CL blocks of a cluster: each block sums its share
// of the row's tiles (draw_range phase 1), the shares' totals are read from every block's shared
// memory in rank order (so every block forms the same R, target and owner), and the block whose
// share holds u * R searches its own tile sums (phase 2) and hands the token to rank 0.  Every
// block of the cluster calls it; returns R.
template <typename T, bool VEC, bool MASK, int CL>
__device__ float cluster_draw(const Params& P, const T* pr, const T* qr, const DrawRows& d, float u, float* wt,
                              uint4* ring, Smem& sm, int* clamp) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int ntile = (P.V + kTile - 1) / kTile;
  const int per = (ntile + CL - 1) / CL;
  const int v0 = min(P.V, rank * per * kTile), v1 = min(P.V, v0 + per * kTile);
  const float Rr = v1 > v0 ? draw_range<T, VEC, MASK>(P, pr, qr, d, v0, v1, false, u, 0.0f, 0.0f, wt, ring, sm, clamp, 1)
                           : 0.0f;
  if (threadIdx.x == 0) sm.cl_total = Rr;
  cl.sync();
  if (threadIdx.x == 0) {
    float tot[CL], R = 0.0f;
#pragma unroll
    for (int r = 0; r < CL; ++r) {
      tot[r] = *cl.map_shared_rank(&sm.cl_total, r);
      R += tot[r];
    }
    const float target = u * R;
    int owner = -1, last = -1;
    float cum = 0.0f, base = 0.0f, base_last = 0.0f;
    for (int r = 0; r < CL; ++r) {
      if (tot[r] > 0.0f) {
        if (owner < 0 && target < cum + tot[r]) {
          owner = r;
          base = cum;
        }
        last = r;
        base_last = cum;
      }
      cum += tot[r];
    }
    if (owner < 0) {  // rounding: the last share with mass searches (and clamps)
      owner = last;
      base = base_last;
    }
    sm.cl_owner = owner;
    sm.cl_base = base;
    sm.cl_R = R;
  }
  __syncthreads();
  const float R = sm.cl_R;
  if (R > 0.0f && rank == sm.cl_owner) {
    draw_range<T, VEC, MASK>(P, pr, qr, d, v0, v1, false, u, u * R - sm.cl_base, R, wt, ring, sm, clamp, 2);
    Smem* lead = cl.map_shared_rank(&sm, 0);
    if (threadIdx.x == 0) {
      lead->y = sm.y;
      lead->margin = sm.margin;
    }
    if (*clamp) atomicOr(&lead->flags, SPEC_FLAG_CDF_CLAMP);
    *clamp = 0;
  }
  cl.sync();  // rank 0 holds the token; no block leaves while another may still write to it
  return R;
}

// The per-request tail, run by the CTA that completed the request's last item.
template <typename T, int MODE, bool VEC, bool NUC, int CL = 1>
__device__ void finish_request(const Params& P, int b, Smem& sm, unsigned char* dyn) {
  constexpr bool MASK = MODE == kTopK || NUC;  // draws skip logits below a row threshold
  // With CL > 1 the CL blocks of a cluster all run the request's decision (identically) and share
  // its full-row draw; only rank 0 writes results.
  const bool lead = CL == 1 || cooperative_groups::this_cluster().block_rank() == 0;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int K = P.K;
  // Warp 0 starts the loads of the ratio test right away (draft tokens, uniforms, the logits at
  // the draft tokens; rows j < K always exist in the padded layout), so they overlap the merge of
  // the row summaries instead of following it.
  int x = 0;
  float zpx = -INFINITY, zqx = -INFINITY, uu = 0.0f;
  if (warp == 0 && lane < K) {
    x = __ldg(P.draft + (size_t)b * K + lane);
    if (MODE != kGreedy) {
      uu = __ldg(P.ua + (size_t)b * K + lane);
      if (x >= 0 && x < P.V) {
        zpx = load1<T>(prow<T>(P, b, lane) + x);
        zqx = load1<T>(qrow<T>(P, b, lane) + x);
      }
    }
  }
  int bad_k = 0;
  const int Kb = clamp_k(P, b, &bad_k);  // every thread reads it: no barrier needed
  if (t == 0) {
    sm.Kb = Kb;
    sm.flags = bad_k ? SPEC_FLAG_BAD_K : 0;
    sm.nonfinite = 0;
  }
  const int nrows = MODE == kGreedy ? Kb + 1 : 2 * Kb + 1;
  // ---- row statistics ----
  if (MODE == kSample) {
    // each row's summaries merged by a group of G lanes, so that every row's loads go out in one
    // round (G divides 32: a group never spans two warps)
    const int G = nrows <= 8 ? 32 : (nrows <= 16 ? 16 : (nrows <= 32 ? 8 : 4));
    const int gi = t / G, gl = t % G, per = P.nchunk * kWarps;
    for (int r0 = 0; r0 < nrows; r0 += kThreads / G) {
      const int r = r0 + gi;
      float m = -INFINITY, s = 0.0f, c2 = P.c2;
      if (r < nrows) {
        const int rp = r <= Kb ? r : K + 1 + (r - Kb - 1);
        const float2* part = P.partial + ((size_t)b * P.R + rp) * per;
        c2 = r > Kb ? P.c2q : P.c2;
#pragma unroll 4
        for (int c = gl; c < per; c += G) {
          float2 pc = __ldg(part + c);
          lse_merge(m, s, pc.x, pc.y, c2);
        }
      }
      for (int o = G >> 1; o > 0; o >>= 1) {
        const float mo = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        const float so = __shfl_xor_sync(0xFFFFFFFFu, s, o);
        lse_merge(m, s, mo, so, c2);
      }
      if (r < nrows && gl == 0) {
        sm.rowM[r] = m;
        sm.rowS[r] = s;
        sm.rowT[r] = -INFINITY;
        sm.rowFlag[r] = (!(s > 0.0f) || isinf(m) || isnan(s)) ? SPEC_FLAG_NONFINITE : 0;
      }
    }
  } else if (MODE == kGreedy) {
    for (int r = warp; r < nrows; r += kWarps) {
      const float2* part = P.partial + ((size_t)b * P.R + r) * P.nchunk * kWarps;
      float best = -INFINITY;
      int bi = 0x7FFFFFFF;
      bool nan = false;
      for (int c = lane; c < P.nchunk * kWarps; c += 32) {
        float2 pc = __ldg(part + c);
        int idx = __float_as_int(pc.y);
        if (idx < 0) nan = true;
        amax_merge(best, bi, pc.x, idx);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float vo = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        int io = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        amax_merge(best, bi, vo, io);
      }
      nan = __any_sync(0xFFFFFFFFu, nan);
      if (lane == 0) {
        sm.rowG[r] = bi;
        sm.rowFlag[r] = nan ? SPEC_FLAG_NONFINITE : 0;
      }
    }
  } else {  // kTopK
    uint2* buf = reinterpret_cast<uint2*>(dyn + (VEC ? (size_t)kDrawStages * kDrawStageBytes : 0)) + (size_t)warp * kRowCap;
    for (int r = warp; r < nrows; r += kWarps) {
      const int rp = r <= Kb ? r : K + 1 + (r - Kb - 1);
      float M = NAN, S = NAN, thr = NAN;
      int fl = 0;
      bool ok = topk_row_fast<T>(P, b, rp, buf, M, S, thr, fl);
      if (lane == 0) {
        sm.rowM[r] = M;
        sm.rowS[r] = S;
        sm.rowT[r] = thr;
        if (!ok && !(fl & SPEC_FLAG_NONFINITE)) fl |= 0x40000000;  // needs the exact path
        if (ok && (!(S > 0.0f) || isinf(M) || isnan(S))) fl |= SPEC_FLAG_NONFINITE;
        sm.rowFlag[r] = fl;
        sm.rowListed[r] = ok;
      }
      __syncwarp();
    }
    __syncthreads();
    for (int r = 0; r < nrows; ++r) {
      if (sm.rowFlag[r] & 0x40000000) {
        const int rp = r <= Kb ? r : K + 1 + (r - Kb - 1);
        float M, S, thr;
        int fl = 0;
        topk_row_exact<T, VEC>(P, row_ptr<T>(P, b, rp), rp > K ? P.c2q : P.c2,
                               reinterpret_cast<uint32_t*>(dyn + (VEC ? (size_t)kDrawStages * kDrawStageBytes : 0)),
                               sm, M, S, thr, fl);
        if (t == 0) {
          sm.rowM[r] = M;
          sm.rowS[r] = S;
          sm.rowT[r] = thr;
          sm.rowFlag[r] = fl | ((!(S > 0.0f) || isinf(M) || isnan(S)) ? SPEC_FLAG_NONFINITE : 0);
        }
        __syncthreads();
      }
    }
  }
  __syncthreads();
  if (NUC && MODE == kSample) {  // top-p: the nucleus pass left each row's kept mass and cut
    for (int r = t; r < nrows; r += kThreads) {
      if (sm.rowFlag[r] & SPEC_FLAG_NONFINITE) continue;
      const int rp = r <= Kb ? r : K + 1 + (r - Kb - 1);
      const float2 ns = P.rowstat[(size_t)b * P.R + rp];
      sm.rowS[r] = ns.x;
      sm.rowT[r] = ns.y;
    }
    __syncthreads();
  } else if (NUC) {  // top-p after top-k: cut every valid row's kept set down to its nucleus
    unsigned char* nbuf = dyn + (VEC ? (size_t)kDrawStages * kDrawStageBytes : 0) +
                          (MODE == kTopK ? (size_t)kWarps * kRowCap * sizeof(uint2) : 0);
    for (int r = 0; r < nrows; ++r) {
      if (sm.rowFlag[r] & SPEC_FLAG_NONFINITE) continue;  // uniform: every thread reads the same flag
      const int rp = r <= Kb ? r : K + 1 + (r - Kb - 1);
      float S, cut;
      nucleus_row<T, VEC>(P, row_ptr<T>(P, b, rp), sm.rowM[r], r > Kb ? P.c2q : P.c2, sm.rowT[r], sm.rowS[r],
                          nbuf, sm, S, cut);
      if (t == 0) {
        sm.rowS[r] = S;
        sm.rowT[r] = cut;
      }
      __syncthreads();
    }
  }
  if (t == 0) {
    int f = 0;
    for (int r = 0; r < nrows; ++r) f |= sm.rowFlag[r];
    sm.flags |= f;
    sm.nonfinite = (f & SPEC_FLAG_NONFINITE) != 0;
  }
  __syncthreads();

  // ---- ratio test and first rejection (warp 0; K <= 16) ----
  int32_t* tok = P.out_tokens + (size_t)b * (K + 1);
  if (warp == 0) {
    bool examined_bad = false;
    int jstar;
    float a = NAN, cq = NAN, am = NAN;
    if (MODE == kGreedy) {
      bool acc = true, bad = false;
      if (lane < Kb) {
        bad = x < 0 || x >= P.V;
        acc = x == sm.rowG[lane];
      }
      unsigned rej = __ballot_sync(0xFFFFFFFFu, lane < Kb && !acc);
      jstar = rej ? __ffs(rej) - 1 : Kb;
      unsigned badm = __ballot_sync(0xFFFFFFFFu, bad);
      examined_bad = jstar < Kb && ((badm >> jstar) & 1u);
      if (lane <= K) {
        int v = -1;
        if (lane < jstar) v = x;
        else if (lane == jstar) v = sm.rowG[jstar];
        tok[lane] = v;
      }
      if (lane == 0) {
        sm.jstar = jstar;
        sm.y = sm.rowG[jstar];
        sm.margin = INFINITY;
      }
    } else {
      bool acc = true, bad = false;
      if (lane < Kb) {
        bad = x < 0 || x >= P.V;
        a = 0.0f;
        cq = 0.0f;
        if (!bad) {
          const int rq = Kb + 1 + lane;
          if (zpx >= sm.rowT[lane]) a = ex2((zpx - sm.rowM[lane]) * P.c2) / sm.rowS[lane];
          if (zqx >= sm.rowT[rq]) cq = ex2((zqx - sm.rowM[rq]) * P.c2q) / sm.rowS[rq];
        }
        acc = uu * cq < a;
        am = cq > 0.0f ? fabsf(uu - a / cq) : INFINITY;
      }
      unsigned rej = __ballot_sync(0xFFFFFFFFu, lane < Kb && !acc);
      jstar = rej ? __ffs(rej) - 1 : Kb;
      unsigned badm = __ballot_sync(0xFFFFFFFFu, bad);
      examined_bad = jstar < Kb && ((badm >> jstar) & 1u);
      if (lane < K && lead) {
        const bool ex = lane <= jstar && lane < Kb;
        if (P.p_draft) P.p_draft[(size_t)b * K + lane] = ex ? a : NAN;
        if (P.q_draft) P.q_draft[(size_t)b * K + lane] = ex ? cq : NAN;
        if (P.acc_margin) P.acc_margin[(size_t)b * K + lane] = ex ? am : NAN;
      }
      if (lane <= K && lead) tok[lane] = lane < jstar ? x : -1;
      if (lane == 0) sm.jstar = jstar;
    }
    if (lane == 0 && examined_bad) sm.flags |= SPEC_FLAG_BAD_TOKEN;
  }
  __syncthreads();

  // ---- resample at the first rejection, or the bonus draw ----
  if (MODE != kGreedy && !sm.nonfinite) {
    const int js = sm.jstar;
    const float u = __ldg(P.ur + b);
    DrawRows d;
    const int rq = Kb + 1 + js;
    d.resid = js < Kb;
    d.Mp2 = sm.rowM[js] * P.c2;
    d.Lp = d.Mp2 + log2f(sm.rowS[js]);
    d.Tp = sm.rowT[js];
    d.Lq = d.resid ? sm.rowM[rq] * P.c2q + log2f(sm.rowS[rq]) : 0.0f;
    d.c2q = P.c2q;
    d.Tq = d.resid ? sm.rowT[rq] : 0.0f;
    const T* pr = prow<T>(P, b, js);
    const T* qr = d.resid ? qrow<T>(P, b, js) : pr;
    uint4* ring = reinterpret_cast<uint4*>(dyn);
    float* wt = reinterpret_cast<float*>(dyn + (VEC ? (size_t)kDrawStages * kDrawStageBytes : 0) +
                                         (MODE == kTopK ? (size_t)kWarps * kRowCap * sizeof(uint2) : 0));
    int clamp = 0;
    bool drawn = false;
    float R = 0.0f;
    if (MODE == kSample && !NUC && !d.resid && !lead) {
      drawn = true;  // a bonus draw reads one chunk: rank 0 does it alone
      R = 1.0f;
    } else if (MODE == kSample && !NUC && !d.resid) {
      // Bonus draw: the chunk masses follow from the stored (max, sum) pairs, so only the chunk
      // holding u * S is read again.
      const int nch = P.nchunk;
      const float2* part = P.partial + ((size_t)b * P.R + js) * nch * kWarps;
      for (int c = t; c < nch; c += kThreads) {
        float mass = 0.0f;
        for (int w = 0; w < kWarps; ++w) {
          const float2 pc = __ldg(part + (size_t)c * kWarps + w);
          if (pc.y != 0.0f) mass += pc.y * ex2(pc.x * P.c2 - d.Mp2);
        }
        wt[c] = mass;
      }
      __syncthreads();
      if (t == 0) {
        float S = 0.0f;
        for (int c = 0; c < nch; ++c) S += wt[c];
        const float target = u * S;
        float cum = 0.0f;
        int cs = -1;
        for (int c = 0; c < nch; ++c) {
          if (target < cum + wt[c]) {
            cs = c;
            break;
          }
          cum += wt[c];
        }
        if (cs < 0) {  // rounding put u * S past the sum: the last chunk with mass (clamped below)
          cs = nch - 1;
          while (cs > 0 && !(wt[cs] > 0.0f)) --cs;
          cum = 0.0f;
          for (int c = 0; c < cs; ++c) cum += wt[c];
        }
        sm.tile = cs;
        sm.tile_base = target - cum;
        sm.total = S;
      }
      __syncthreads();
      const int cs = sm.tile;
      const float tin = sm.tile_base, S = sm.total;
      __syncthreads();
      const int v0 = cs * Cfg<T>::CH;
      const float rc = draw_range<T, VEC, MASK>(P, pr, pr, d, v0, min(P.V, v0 + Cfg<T>::CH), false, u, tin, S,
                                                wt, ring, sm, &clamp);
      drawn = rc > 0.0f;
      R = S;
    }
    // after top-k, p's kept set (at most a few hundred tokens) is complete in row js's chunk lists
    // unless that row took the exact path: the draw runs over it instead of over the whole row
    uint2* klist = reinterpret_cast<uint2*>(dyn + (VEC ? (size_t)kDrawStages * kDrawStageBytes : 0));
    const bool listed = MODE == kTopK && sm.rowListed[js];
    if (listed && !drawn) drawn = draw_list<T>(P, b, js, qr, d, u, klist, sm, &clamp, &R);
    if (!drawn) {
      if (CL > 1 && d.resid)
        R = cluster_draw<T, VEC, MASK, CL>(P, pr, qr, d, u, wt, ring, sm, &clamp);
      else
        R = draw_range<T, VEC, MASK>(P, pr, qr, d, 0, P.V, true, u, 0.0f, 0.0f, wt, ring, sm, &clamp);
    }
    float resid_mass = d.resid ? R : 0.0f;
    if (!(R > 0.0f)) {
      // max(0, p - q) vanished through rounding: draw from p instead (R is the same in every
      // block of a cluster, so they all take this branch together)
      const bool was_resid = d.resid;
      d.resid = false;
      if (t == 0) sm.flags |= SPEC_FLAG_RESIDUAL_ZERO;
      if (CL > 1 && was_resid)
        R = cluster_draw<T, VEC, MASK, CL>(P, pr, pr, d, u, wt, ring, sm, &clamp);
      else if (!(listed && draw_list<T>(P, b, js, pr, d, u, klist, sm, &clamp, &R)))
        R = draw_range<T, VEC, MASK>(P, pr, pr, d, 0, P.V, true, u, 0.0f, 0.0f, wt, ring, sm, &clamp);
    }
    if (clamp) atomicOr(&sm.flags, SPEC_FLAG_CDF_CLAMP);
    __syncthreads();
    if (t == 0 && lead) {
      tok[js] = sm.y;
      if (P.resid_mass) P.resid_mass[b] = resid_mass;
      if (P.samp_margin) P.samp_margin[b] = sm.margin;
    }
  } else if (MODE != kGreedy) {  // non-finite rows: no result
    if (t <= K) tok[t] = -1;
    if (t == 0) {
      sm.jstar = 0;
      if (P.resid_mass) P.resid_mass[b] = NAN;
      if (P.samp_margin) P.samp_margin[b] = NAN;
    }
  } else {
    if (sm.nonfinite && t <= K) tok[t] = -1;
    if (t == 0) {
      if (sm.nonfinite) sm.jstar = 0;
      if (P.resid_mass) P.resid_mass[b] = 0.0f;
      if (P.samp_margin) P.samp_margin[b] = INFINITY;
    }
  }
  __syncthreads();
  if (!lead) return;
  if (t == 0) {
    P.out_nacc[b] = sm.jstar;
    if (P.flags) P.flags[b] = sm.flags;
  }
  if (P.lognorm || P.rowcut) {
    const int R = 2 * K + 1;
    for (int r = t; r < R; r += kThreads) {
      float v = NAN, cut = NAN;
      if (MODE != kGreedy) {
        int rr = -1;  // compact row index of padded row r
        if (r <= K) rr = r <= Kb ? r : -1;
        else rr = (r - K - 1) < Kb ? Kb + 1 + (r - K - 1) : -1;
        if (rr >= 0) {
          v = sm.rowM[rr] * (rr > Kb ? P.invTq : P.invT) + logf(sm.rowS[rr]);
          cut = sm.rowT[rr];
        }
      }
      if (P.lognorm) P.lognorm[(size_t)b * R + r] = v;
      if (P.rowcut) P.rowcut[(size_t)b * R + r] = cut;
    }
  }
  if (P.sample_prob && t == 0) {
    // q(x) of the drawn token under the row's distribution: exp(z_x / T - log-normaliser), 1 for
    // the greedy draft's one-hot, NaN for a row without a result.  Thread 0 wrote tok[0].
    const int y = tok[0];
    float pr = NAN;
    if (y >= 0 && y < P.V)
      pr = MODE == kGreedy ? 1.0f
                           : expf(load1<T>(prow<T>(P, b, 0) + y) * P.invT - (sm.rowM[0] * P.invT + logf(sm.rowS[0])));
    P.sample_prob[b] = pr;
  }
  if (MODE == kGreedy && t < K) {
    if (P.p_draft) P.p_draft[(size_t)b * K + t] = NAN;
    if (P.q_draft) P.q_draft[(size_t)b * K + t] = NAN;
    if (P.acc_margin) P.acc_margin[(size_t)b * K + t] = NAN;
  }
}

// ------------------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------------------
// Position in the item space of one CTA's contiguous range: request b, padded row rp, chunk c,
// and the row's first byte.  Advanced one chunk at a time without divisions.
struct Cursor {
  int b, rp, c;
  uint32_t crow;  // compact row index (ragged layout)
  const char* row;
};

template <typename T>
__device__ __forceinline__ const char* row_bytes(const Params& P, int b, int rp) {
  return reinterpret_cast<const char*>(row_ptr<T>(P, b, rp));
}

template <typename T>
__device__ __forceinline__ void cursor_at(const Params& P, uint32_t item, Cursor& k) {
  const uint32_t row = item / (uint32_t)P.nchunk;
  k.c = (int)(item - row * (uint32_t)P.nchunk);
  k.crow = row;
  if (P.rowmap) {
    const uint32_t e = __ldg(P.rowmap + row);
    k.b = (int)(e >> 6);
    k.rp = (int)(e & 63u);
  } else {
    k.b = (int)(row / (uint32_t)P.R);
    k.rp = (int)(row - (uint32_t)k.b * P.R);
  }
  k.row = row_bytes<T>(P, k.b, k.rp);
}

template <typename T>
__device__ __forceinline__ void cursor_next(const Params& P, Cursor& k) {
  if (++k.c < P.nchunk) return;
  k.c = 0;
  ++k.crow;
  if (P.rowmap) {
    const uint32_t e = __ldg(P.rowmap + k.crow);
    k.b = (int)(e >> 6);
    k.rp = (int)(e & 63u);
  } else if (++k.rp == P.R) {
    k.rp = 0;
    ++k.b;
  }
  k.row = row_bytes<T>(P, k.b, k.rp);
}

// Top-k mode's per-thread ring: starts the copy of the cursor's chunk into `stage`, each thread
// its own 16-byte vectors (which it alone reads back).
template <typename T>
__device__ __forceinline__ void issue_at(const Params& P, const Cursor& k, uint4* stage) {
  const int v0 = k.c * Cfg<T>::CH;
  const int n = min(Cfg<T>::CH, P.V - v0);
  const char* base = k.row + (size_t)v0 * sizeof(T);
#pragma unroll
  for (int l = 0; l < Cfg<T>::LOADS; ++l) {
    const int e0 = (l * kThreads + threadIdx.x) * Cfg<T>::VW;
    const bool ok = e0 < n;
    cp_async16(stage + l * kThreads + threadIdx.x, ok ? base + (size_t)e0 * sizeof(T) : base, ok ? 16 : 0);
  }
}

__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Sampling summary of one chunk straight from its packed 16-byte vectors: the max on packed
// values, then 2^((z - max) * c2) in packed f32x2 arithmetic, then a warp max and a rescaled warp
// sum.  Writes (max, sum) for the warp's share to out[warp].
template <typename T>
__device__ __forceinline__ void sample_vec(float c2, uint4 (&raw)[Cfg<T>::LOADS], int n, float2* out) {
  const int t = threadIdx.x;
  if (n < Cfg<T>::CH) {  // tail chunk: vectors at or past n hold no logits
#pragma unroll
    for (int l = 0; l < Cfg<T>::LOADS; ++l)
      if ((l * kThreads + t) * Cfg<T>::VW >= n)
        raw[l] = sizeof(T) == 2 ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                                : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
  }
  float m;
  if (sizeof(T) == 2) {
    uint32_t mx = raw[0].x;
#pragma unroll
    for (int l = 0; l < Cfg<T>::LOADS; ++l) {
      if (l > 0) mx = bmax2_nan(mx, raw[l].x);
      mx = bmax2_nan(mx, raw[l].y);
      mx = bmax2_nan(mx, raw[l].z);
      mx = bmax2_nan(mx, raw[l].w);
    }
    m = fmax_nan(bf16_lo(mx), bf16_hi(mx));
  } else {
    m = -INFINITY;
#pragma unroll
    for (int l = 0; l < Cfg<T>::LOADS; ++l) {
      m = fmax_nan(m, __uint_as_float(raw[l].x));
      m = fmax_nan(m, __uint_as_float(raw[l].y));
      m = fmax_nan(m, __uint_as_float(raw[l].z));
      m = fmax_nan(m, __uint_as_float(raw[l].w));
    }
  }
  float s = 0.0f;
  if (m != -INFINITY) {
    // 2^((z - m) * c2) as 2^(z * c2 - m * c2): one packed FMA per pair of logits
    const float2 negmc = make_float2(-m * c2, -m * c2), cc = make_float2(c2, c2);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int l = 0; l < Cfg<T>::LOADS; ++l) {
      const uint32_t w[4] = {raw[l].x, raw[l].y, raw[l].z, raw[l].w};
      if (sizeof(T) == 2) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 d = __ffma2_rn(make_float2(bf16_lo(w[k]), bf16_hi(w[k])), cc, negmc);
          acc = __fadd2_rn(acc, make_float2(ex2(d.x), ex2(d.y)));
        }
      } else {
#pragma unroll
        for (int k = 0; k < 4; k += 2) {
          const float2 d = __ffma2_rn(make_float2(__uint_as_float(w[k]), __uint_as_float(w[k + 1])), cc, negmc);
          acc = __fadd2_rn(acc, make_float2(ex2(d.x), ex2(d.y)));
        }
      }
    }
    s = acc.x + acc.y;
  }
  // warp: max first (NaN-propagating), then every lane rescales its sum to it and the sums add up
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmax_nan(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
  float sc = s == 0.0f ? 0.0f : s * ex2((m - M) * c2);
  sc = warp_sum(sc);
  if ((t & 31) == 0) out[t >> 5] = make_float2(M, sc);
}

// Greedy summary of one chunk straight from its packed vectors: the warp's max (on packed values,
// NaN-propagating), then only lanes whose own max equals it look for their first element at that
// value; the warp keeps the lowest token id.  A NaN is marked by the id -1.
template <typename T>
__device__ __forceinline__ void greedy_vec(uint4 (&raw)[Cfg<T>::LOADS], int n, int v0, float2* out) {
  const int t = threadIdx.x, lane = t & 31;
  constexpr int VW = Cfg<T>::VW;
  if (n < Cfg<T>::CH) {  // tail chunk: vectors at or past n hold no logits
#pragma unroll
    for (int l = 0; l < Cfg<T>::LOADS; ++l)
      if ((l * kThreads + t) * VW >= n)
        raw[l] = sizeof(T) == 2 ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                                : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
  }
  float m;
  if (sizeof(T) == 2) {
    uint32_t mx = raw[0].x;
#pragma unroll
    for (int l = 0; l < Cfg<T>::LOADS; ++l) {
      if (l > 0) mx = bmax2_nan(mx, raw[l].x);
      mx = bmax2_nan(mx, raw[l].y);
      mx = bmax2_nan(mx, raw[l].z);
      mx = bmax2_nan(mx, raw[l].w);
    }
    m = fmax_nan(bf16_lo(mx), bf16_hi(mx));
  } else {
    m = -INFINITY;
#pragma unroll
    for (int l = 0; l < Cfg<T>::LOADS; ++l) {
      m = fmax_nan(m, __uint_as_float(raw[l].x));
      m = fmax_nan(m, __uint_as_float(raw[l].y));
      m = fmax_nan(m, __uint_as_float(raw[l].z));
      m = fmax_nan(m, __uint_as_float(raw[l].w));
    }
  }
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmax_nan(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
  int idx = 0x7FFFFFFF;
  if (M == M && m == M) {  // this lane holds the max: its first element at that value
#pragma unroll
    for (int l = Cfg<T>::LOADS - 1; l >= 0; --l) {
      const uint32_t w[4] = {raw[l].x, raw[l].y, raw[l].z, raw[l].w};
      const int e0 = (l * kThreads + t) * VW;
#pragma unroll
      for (int k = VW - 1; k >= 0; --k) {
        const float z = sizeof(T) == 2 ? (k & 1 ? bf16_hi(w[k >> 1]) : bf16_lo(w[k >> 1])) : __uint_as_float(w[k]);
        if (z == M) idx = e0 + k;  // scanning downwards leaves the lowest index
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(0xFFFFFFFFu, idx, o));
  if (lane == 0) out[t >> 5] = make_float2(M, __int_as_float(M == M ? v0 + idx : -1));
}

// Pass 1 for top-k (and for rows that are not 16-byte aligned, in every mode): stream every valid
// row once.  Each CTA owns a contiguous range of items (request, row, chunk), so successive items
// walk memory in order, the cursor needs no divisions and a row segment's candidate set carries
// over from chunk to chunk.  No block waits for another and nothing is counted: pass 2 starts
// when this grid is done.
template <typename T, int MODE, bool VEC>
__global__ void __launch_bounds__(kThreads, 4) stats_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ Smem sm;
  pdl_launch_next();  // the next pass may launch now; it waits for this grid before reading
  const uint32_t total = P.rowmap ? __ldg(P.total_rows) * (uint32_t)P.nchunk : P.uniform_items;
  const uint32_t lo = (uint32_t)(((uint64_t)total * blockIdx.x) / gridDim.x);
  const uint32_t hi = (uint32_t)(((uint64_t)total * (blockIdx.x + 1)) / gridDim.x);
  if (lo >= hi) return;
  uint4* stages = reinterpret_cast<uint4*>(dyn);
  constexpr int ST = kStagesTopK;
  uint2* surv = reinterpret_cast<uint2*>(dyn + (VEC ? (size_t)ST * kChunkBytes : 0));
  Cursor cc;
  cursor_at<T>(P, lo, cc);
  bool seg_start = true, seg_end = false;  // row segments of the top-k path
  int seg_next = 0, seg_m = 0;
  auto summarise_f = [&](const Cursor& k, const float (&v)[Cfg<T>::PER]) {
    const int v0 = k.c * Cfg<T>::CH;
    const int n = min(Cfg<T>::CH, P.V - v0);
    const size_t slot = ((size_t)k.b * P.R + k.rp) * P.nchunk + k.c;
    if (MODE == kSample)
      item_sample<T>(k.rp > P.K ? P.c2q : P.c2, v, P.partial + slot * kWarps);
    else if (MODE == kGreedy)
      item_greedy<T, VEC>(v, n, v0, P.partial + slot * kWarps);
    else
      topk_chunk<T, VEC>(P, v, n, k.b, k.rp, k.c, seg_start, seg_end, surv, sm, seg_next, seg_m);
  };
  if (VEC && MODE == kTopK) {
    // A per-thread ring: each thread copies its own vectors of a chunk and refills its slots as
    // soon as it has read them.  (A ring shared by the block refills a stage only once every warp
    // has read it; between the block barriers of the candidate set that cost the fp32 top-k pass
    // 6%.)
    Cursor ic = cc;
#pragma unroll
    for (int s = 0; s < ST; ++s) {
      if (lo + s < hi) {
        issue_at<T>(P, ic, stages + (size_t)s * (kChunkBytes / 16));
        cursor_next<T>(P, ic);
      }
      cp_async_commit();
    }
    int s = 0;
    for (uint32_t it = lo; it < hi; ++it) {
      uint4* st = stages + (size_t)s * (kChunkBytes / 16);
      cp_async_wait<ST - 1>();  // this thread's copies of this item have landed
      uint4 raw[Cfg<T>::LOADS];
#pragma unroll
      for (int l = 0; l < Cfg<T>::LOADS; ++l) raw[l] = st[l * kThreads + threadIdx.x];
      if (it + ST < hi) {  // the stage's bytes are in registers: refill it
        issue_at<T>(P, ic, st);
        cursor_next<T>(P, ic);
      }
      cp_async_commit();
      seg_end = it + 1 == hi || cc.c + 1 == P.nchunk;
      const int n = min(Cfg<T>::CH, P.V - cc.c * Cfg<T>::CH);
      float v[Cfg<T>::PER];
      unpack<T>(raw, n, v);
      summarise_f(cc, v);
      seg_start = seg_end;
      cursor_next<T>(P, cc);
      s = s + 1 == ST ? 0 : s + 1;
    }
    cp_async_wait<0>();
  } else {
    for (uint32_t it = lo; it < hi; ++it) {
      const int v0 = cc.c * Cfg<T>::CH;
      float v[Cfg<T>::PER];
      load_chunk<T, VEC>(reinterpret_cast<const T*>(cc.row) + v0, min(Cfg<T>::CH, P.V - v0), v);
      seg_end = it + 1 == hi || cc.c + 1 == P.nchunk;
      summarise_f(cc, v);
      seg_start = seg_end;
      cursor_next<T>(P, cc);
    }
  }
}

// Pass 1 in sampling and greedy modes (aligned rows): one short-lived block per IPB consecutive
// items.  Each thread loads its 16-byte vectors of the block's items straight into registers (all
// IPB x 16 KB of the block in flight at once), the block summarises them and exits, and the
// hardware keeps every SM filled with new blocks: no ring to manage, no barrier, no wait, and no
// ramp or tail of a persistent grid's static ranges.  Test hook bit 0 makes every block treat
// its items as lost -- summaries NaN, as a failed load would leave them -- so that the flagging
// of the requests they touch can be tested without any fault.
template <typename T, int MODE, int IPB>
__global__ void __launch_bounds__(kThreads, kItemBlocksPerSM) stats_item_kernel(const Params P) {
  pdl_launch_next();  // the next pass may launch now; it waits for this grid before reading
  const uint32_t total = P.rowmap ? __ldg(P.total_rows) * (uint32_t)P.nchunk : P.uniform_items;
  const uint32_t it0 = blockIdx.x * (uint32_t)IPB;
  if (it0 >= total) return;
  const int t = threadIdx.x;
  Cursor cc;
  cursor_at<T>(P, it0, cc);
  if (P.test_hooks & 1) {
    for (int i = 0; i < IPB && it0 + i < total; ++i) {
      const size_t slot = ((size_t)cc.b * P.R + cc.rp) * P.nchunk + cc.c;
      if (t < kWarps) P.partial[slot * kWarps + t] = make_float2(NAN, MODE == kGreedy ? __int_as_float(-1) : NAN);
      if (i + 1 < IPB) cursor_next<T>(P, cc);
    }
    return;
  }
  uint4 raw[IPB][Cfg<T>::LOADS];
  int nn[IPB];
  {
    Cursor k = cc;
#pragma unroll
    for (int i = 0; i < IPB; ++i) {
      nn[i] = 0;
      if (it0 + i < total) {
        const int v0 = k.c * Cfg<T>::CH;
        nn[i] = min(Cfg<T>::CH, P.V - v0);
        const char* base = k.row + (size_t)v0 * sizeof(T);
#pragma unroll
        for (int l = 0; l < Cfg<T>::LOADS; ++l) {
          const int e0 = (l * kThreads + t) * Cfg<T>::VW;
          raw[i][l] = e0 < nn[i] ? ldg_stream(base + (size_t)e0 * sizeof(T)) : make_uint4(0u, 0u, 0u, 0u);
        }
        if (i + 1 < IPB) cursor_next<T>(P, k);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < IPB; ++i) {
    if (nn[i] > 0) {
      const size_t slot = ((size_t)cc.b * P.R + cc.rp) * P.nchunk + cc.c;
      if (MODE == kSample)
        sample_vec<T>(cc.rp > P.K ? P.c2q : P.c2, raw[i], nn[i], P.partial + slot * kWarps);
      else
        greedy_vec<T>(raw[i], nn[i], cc.c * Cfg<T>::CH, P.partial + slot * kWarps);
      if (i + 1 < IPB) cursor_next<T>(P, cc);
    }
  }
}

// Top-p in sampling mode, between the two passes: one block per valid row merges the row's
// chunk summaries into its (max, sum), exactly as the per-request pass does, finds the row's
// nucleus and leaves (kept mass, cut) for the per-request pass.  Non-finite rows are left to the
// per-request pass, which flags them.
// Three blocks per SM is what its shared memory allows; saying so lets the compiler keep the list
// pass in 80 registers instead of spilling at 64.
template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads, 3) nucleus_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ Smem sm;
  pdl_wait();
  pdl_launch_next();
  const int t = threadIdx.x, lane = t & 31;
  int b, rp;
  if (P.rowmap) {
    if (blockIdx.x >= __ldg(P.total_rows)) return;
    const uint32_t e = __ldg(P.rowmap + blockIdx.x);
    b = (int)(e >> 6);
    rp = (int)(e & 63u);
  } else {
    b = (int)(blockIdx.x / (unsigned)P.R);
    rp = (int)(blockIdx.x % (unsigned)P.R);
  }
  const float c2 = rp > P.K ? P.c2q : P.c2;
  if (t < 32) {
    const float2* part = P.partial + ((size_t)b * P.R + rp) * P.nchunk * kWarps;
    float m = -INFINITY, s = 0.0f;
#pragma unroll 4
    for (int c = lane; c < P.nchunk * kWarps; c += 32) {
      float2 pc = __ldg(part + c);
      lse_merge(m, s, pc.x, pc.y, c2);
    }
    lse_warp(m, s, c2);
    if (lane == 0) {
      sm.rowM[0] = m;
      sm.rowS[0] = s;
      sm.rowFlag[0] = (!(s > 0.0f) || isinf(m) || isnan(s)) ? 1 : 0;
    }
  }
  __syncthreads();
  if (sm.rowFlag[0]) return;
  float S, cut;
  nucleus_row<T, VEC>(P, row_ptr<T>(P, b, rp), sm.rowM[0], c2, -INFINITY, sm.rowS[0], dyn, sm, S, cut);
  if (t == 0) P.rowstat[(size_t)b * P.R + rp] = make_float2(S, cut);
}

// Pass 2: one block per request merges its rows' summaries, runs the ratio test and the
// first-rejection scan, and draws the resampled or bonus token.
template <typename T, int MODE, bool VEC, bool NUC>
__global__ void __launch_bounds__(kThreads) finish_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ Smem sm;
  pdl_wait();
  pdl_launch_next();
  for (int b = blockIdx.x; b < P.B; b += gridDim.x) {
    finish_request<T, MODE, VEC, NUC>(P, b, sm, dyn);
    __syncthreads();
  }
}

// Pass 2 for batches of fewer requests than SMs (sampling mode): a cluster of kCluster blocks per
// request, which share the full-row residual draw (cluster_draw).
template <typename T, bool VEC>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads) finish_cluster_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ Smem sm;
  pdl_wait();
  pdl_launch_next();
  finish_request<T, kSample, VEC, false, kCluster>(P, (int)(blockIdx.x / kCluster), sm, dyn);
}

// ------------------------------------------------------------------------------------------------
// multi-draft verify (spec_verify_multi)
// ------------------------------------------------------------------------------------------------
// Several draft chains per request (2kiu.com §7 and cf-1.com §2.3 name ensembles of draft models).
// The first position is shared: the chains' first drafts are tested in turn, each against what the
// earlier rejections leave of p -- r_0 = P_0; candidate n is accepted iff u_n q_n(x_n) < r_n(x_n);
// a rejection leaves r_{n+1} = max(0, r_n - q_n) / R_n with R_n = sum_v max(0, r_n(v) - q_n(v)) --
// so that the first emitted token is distributed as P_0.  The first accepted chain is verified on
// with the single-draft rule; with every candidate rejected one token is drawn from r_N.  The
// streaming pass summarises every row the step reads: sub-request b N + n holds chain n of request
// b, and a row table leaves out row 0 of every chain after the first (the shared position is read
// once).  The per-request pass below takes the decisions: in sampling mode a cluster of
// kMultiCluster blocks per request, which share each stage pass and draw; greedy, one block.

// The rows of the first position's stage n (weights max(0, r_n - q_n)): P_0 and Q_0..Q_n.
struct MultiRows {
  const void* row[SPEC_MAX_DRAFTS + 1];  // P_0, then Q_0, Q_1, ...
  float L[SPEC_MAX_DRAFTS + 1];          // their log2 normalisers (max * c2 + log2 sum)
  float Rinv[SPEC_MAX_DRAFTS];           // 1 / R_i, or 0 where R_i vanished (r_{i+1} = r_i then)
  int n;                                 // the stage
  bool sub;                              // weights max(0, r_n - q_n); else r_n itself
};

// The stage's weights for 8 logits [e0, e0 + 8) (logits past V weigh 0): r follows the recursion
// above term by term; every pass computes it with the same instructions.  Over aligned rows the
// 16-byte vectors of every row the stage reads (P_0, then Q_0 .. Q_last) are loaded first
// (multi_load8) and used after (multi_weights_raw), so that all of them are in flight at once.
template <typename T>
struct MultiRaw {
  static constexpr int NV = 8 * (int)sizeof(T) / 16;  // vectors per row
  uint4 v[SPEC_MAX_DRAFTS + 1][NV];
};
template <typename T>
__device__ __forceinline__ void multi_load8(const Params& P, const MultiRows& mr, int e0, MultiRaw<T>& m) {
  constexpr int NV = MultiRaw<T>::NV, VW = 16 / (int)sizeof(T);
  const int last = mr.sub ? mr.n : mr.n - 1;
  const uint4 ninf = sizeof(T) == 2 ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                                    : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
#pragma unroll
  for (int r = 0; r <= SPEC_MAX_DRAFTS; ++r)
#pragma unroll
    for (int h = 0; h < NV; ++h) {
      const int e = e0 + h * VW;
      m.v[r][h] = r <= last + 1 && e < P.V ? ldg_stream(static_cast<const T*>(mr.row[r]) + e) : ninf;
    }
}
template <typename T>
__device__ __forceinline__ void multi_weights_raw(const Params& P, const MultiRows& mr, const MultiRaw<T>& m,
                                                  float (&w)[8]) {
  constexpr int NV = MultiRaw<T>::NV;
  const int last = mr.sub ? mr.n : mr.n - 1;
  auto unpack8 = [&](int r, float (&z)[8]) {
#pragma unroll
    for (int h = 0; h < NV; ++h) {
      const uint32_t q[4] = {m.v[r][h].x, m.v[r][h].y, m.v[r][h].z, m.v[r][h].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (sizeof(T) == 2) {
          z[h * 8 + 2 * k] = bf16_lo(q[k]);
          z[h * 8 + 2 * k + 1] = bf16_hi(q[k]);
        } else {
          z[h * 4 + k] = __uint_as_float(q[k]);
        }
      }
    }
  };
  float z[8];
  unpack8(0, z);
#pragma unroll
  for (int k = 0; k < 8; ++k) w[k] = ex2(fmaf(z[k], P.c2, -mr.L[0]));
#pragma unroll
  for (int i = 0; i < SPEC_MAX_DRAFTS; ++i) {
    if (i <= last) {
      unpack8(1 + i, z);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float d = w[k] - ex2(fmaf(z[k], P.c2q, -mr.L[1 + i]));
        if (i < mr.n)
          w[k] = mr.Rinv[i] > 0.0f ? fmaxf(d, 0.0f) * mr.Rinv[i] : w[k];
        else
          w[k] = fmaxf(d, 0.0f);
      }
    }
  }
}
template <typename T, bool VEC>
__device__ __forceinline__ void multi_weights8(const Params& P, const MultiRows& mr, int e0, float (&w)[8]) {
  if constexpr (VEC) {
    MultiRaw<T> m;
    multi_load8<T>(P, mr, e0, m);
    multi_weights_raw<T>(P, mr, m, w);
  } else {
    const int last = mr.sub ? mr.n : mr.n - 1;
    float z[8];
    load8<T, VEC>(static_cast<const T*>(mr.row[0]), e0, P.V, z);
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = ex2(fmaf(z[k], P.c2, -mr.L[0]));
    for (int i = 0; i <= last; ++i) {
      load8<T, VEC>(static_cast<const T*>(mr.row[1 + i]), e0, P.V, z);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float d = w[k] - ex2(fmaf(z[k], P.c2q, -mr.L[1 + i]));
        if (i < mr.n)
          w[k] = mr.Rinv[i] > 0.0f ? fmaxf(d, 0.0f) * mr.Rinv[i] : w[k];
        else
          w[k] = fmaxf(d, 0.0f);
      }
    }
  }
}

// One block-wide pass over the stage's weights: tile sums (256 logits a warp tile), a block scan of
// per-thread runs of tiles; returns the total.  With `draw`, also the inverse CDF in ascending token
// id at target u * total (the tile, then the lane, then the logit), setting sm.y, sm.margin and, when
// rounding leaves the target past the sums, *clamp with the last logit that has weight.
template <typename T, bool VEC>
__device__ float multi_pass(const Params& P, const MultiRows& mr, bool draw, float u, float* wt, Smem& sm,
                            int* clamp) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int ntile = (P.V + kTile - 1) / kTile;
  auto tile_sum = [&](int i, const float (&w)[8]) {
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) s += w[k];
    s = warp_sum(s);
    if (lane == 0 && i < ntile) wt[i] = s;
  };
  if constexpr (VEC) {
    for (int i0 = warp; i0 < ntile; i0 += kMultiTiles * kWarps) {  // kMultiTiles tiles a warp, all loads first
      MultiRaw<T> m[kMultiTiles];
#pragma unroll
      for (int g = 0; g < kMultiTiles; ++g) multi_load8<T>(P, mr, (i0 + g * kWarps) * kTile + lane * 8, m[g]);
#pragma unroll
      for (int g = 0; g < kMultiTiles; ++g) {
        float w[8];
        multi_weights_raw<T>(P, mr, m[g], w);
        tile_sum(i0 + g * kWarps, w);
      }
    }
  } else {
    for (int i = warp; i < ntile; i += kWarps) {
      float w[8];
      multi_weights8<T, VEC>(P, mr, i * kTile + lane * 8, w);
      tile_sum(i, w);
    }
  }
  __syncthreads();
  const int L = (ntile + kThreads - 1) / kThreads;
  const int s0 = t * L, s1 = min(s0 + L, ntile);
  float seg = 0.0f;
  for (int i = s0; i < s1; ++i) seg += wt[i];
  float incl = seg;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.red_s[warp] = incl;
  if (t == 0) {
    sm.seg_first = kThreads;
    sm.found = 0;
  }
  __syncthreads();
  float off = 0.0f, total = 0.0f;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) off += sm.red_s[w];
    total += sm.red_s[w];
  }
  incl += off;
  if (!draw || !(total > 0.0f)) {
    __syncthreads();
    return total;
  }
  const float target = u * total;
  if (target < incl) atomicMin(&sm.seg_first, t);
  __syncthreads();
  const int tf = sm.seg_first;
  if (t == (tf == kThreads ? 0 : tf)) {
    int found = -1;
    float run = incl - seg;
    if (tf < kThreads)
      for (int i = s0; i < s1; ++i) {
        if (target < run + wt[i]) {
          found = i;
          break;
        }
        run += wt[i];
      }
    if (found < 0) {  // rounding left the target past the sums: the last tile with weight
      int i = ntile - 1;
      while (i > 0 && !(wt[i] > 0.0f)) --i;
      run = 0.0f;
      for (int j = 0; j < i; ++j) run += wt[j];
      found = i;
      sm.found = 2;
    } else {
      sm.found = 1;
    }
    sm.tile = found;
    sm.tile_base = run;
  }
  __syncthreads();
  if (warp == 0) {
    const int tile = sm.tile;
    bool clamped = sm.found == 2;
    float w[8];
    multi_weights8<T, VEC>(P, mr, tile * kTile + lane * 8, w);
    float ls = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) ls += w[k];
    float li = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xFFFFFFFFu, li, o);
      if (lane >= o) li += y;
    }
    const float tl = target - sm.tile_base;
    const unsigned hit = clamped ? 0u : __ballot_sync(0xFFFFFFFFu, tl < li);
    int yl, ye = -1;
    float margin = 0.0f;
    if (hit) {
      yl = __ffs(hit) - 1;
      if (lane == yl) {
        float run = li - ls;
        for (int k = 0; k < 8; ++k) {
          if (tl < run + w[k]) {
            ye = k;
            margin = fminf(tl - run, run + w[k] - tl) / total;
            break;
          }
          run += w[k];
        }
        if (ye < 0) {  // sub-ulp disagreement between the levels: the lane's last logit with weight
          for (int k = 7; k >= 0 && ye < 0; --k)
            if (w[k] > 0.0f) ye = k;
          clamped = true;
        }
      }
    } else {
      const unsigned pos = __ballot_sync(0xFFFFFFFFu, ls > 0.0f);
      yl = pos ? 31 - __clz(pos) : 0;
      if (lane == yl)
        for (int k = 7; k >= 0 && ye < 0; --k)
          if (w[k] > 0.0f) ye = k;
      clamped = true;
    }
    if (lane == yl) {
      sm.y = tile * kTile + yl * 8 + (ye < 0 ? 0 : ye);
      sm.margin = clamped ? 0.0f : margin;
      if (clamped) *clamp = 1;
    }
  }
  __syncthreads();
  return total;
}

// multi_pass shared by the CL blocks of a cluster: each block sums the stage's weights over its
// own contiguous share of the tiles; the shares' totals are read from every block's shared memory
// in rank order, so every block forms the same R; with `draw`, the block whose share holds the
// target searches its tiles and writes the token into rank 0's shared memory.  Every block takes
// both cluster barriers on every path.
template <typename T, bool VEC, int CL>
__device__ float multi_pass_cluster(const Params& P, const MultiRows& mr, bool draw, float u, float* wt, Smem& sm,
                                    int* clamp) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int ntile = (P.V + kTile - 1) / kTile;
  const int per = (ntile + CL - 1) / CL;
  const int i0 = min(ntile, rank * per), nt = min(ntile, i0 + per) - i0;
  auto tile_sum = [&](int i, const float (&w)[8]) {
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) s += w[k];
    s = warp_sum(s);
    if (lane == 0 && i < nt) wt[i] = s;
  };
  if constexpr (VEC) {
    for (int j0 = warp; j0 < nt; j0 += kMultiTiles * kWarps) {
      MultiRaw<T> m[kMultiTiles];
#pragma unroll
      for (int g = 0; g < kMultiTiles; ++g) {
        const int j = j0 + g * kWarps;
        multi_load8<T>(P, mr, (j < nt ? i0 + j : ntile) * kTile + lane * 8, m[g]);
      }
#pragma unroll
      for (int g = 0; g < kMultiTiles; ++g) {
        float w[8];
        multi_weights_raw<T>(P, mr, m[g], w);
        tile_sum(j0 + g * kWarps, w);
      }
    }
  } else {
    for (int j = warp; j < nt; j += kWarps) {
      float w[8];
      multi_weights8<T, VEC>(P, mr, (i0 + j) * kTile + lane * 8, w);
      tile_sum(j, w);
    }
  }
  __syncthreads();
  // this share's runs of tiles per thread, a block scan, and its total
  const int L = (nt + kThreads - 1) / kThreads;
  const int s0 = t * L, s1 = min(s0 + L, nt);
  float seg = 0.0f;
  for (int i = s0; i < s1; ++i) seg += wt[i];
  float incl = seg;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.red_s[warp] = incl;
  __syncthreads();
  float off = 0.0f, mine = 0.0f;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) off += sm.red_s[w];
    mine += sm.red_s[w];
  }
  incl += off;
  if (t == 0) sm.cl_total = mine;
  cl.sync();
  float tot[CL], R = 0.0f;
#pragma unroll
  for (int r = 0; r < CL; ++r) {
    tot[r] = *cl.map_shared_rank(&sm.cl_total, r);
    R += tot[r];
  }
  if (draw && R > 0.0f) {
    const float target = u * R;
    int owner = -1, last = -1;
    float cum = 0.0f, base = 0.0f, base_last = 0.0f;
    for (int r = 0; r < CL; ++r) {
      if (tot[r] > 0.0f) {
        if (owner < 0 && target < cum + tot[r]) {
          owner = r;
          base = cum;
        }
        last = r;
        base_last = cum;
      }
      cum += tot[r];
    }
    if (owner < 0) {  // rounding: the last share with mass searches (and clamps)
      owner = last;
      base = base_last;
    }
    if (rank == owner) {
      const float tl0 = target - base;  // the mass to pass inside this share
      if (t == 0) {
        sm.seg_first = kThreads;
        sm.found = 0;
      }
      __syncthreads();
      if (tl0 < incl) atomicMin(&sm.seg_first, t);
      __syncthreads();
      const int tf = sm.seg_first;
      if (t == (tf == kThreads ? 0 : tf)) {
        int found = -1;
        float run = incl - seg;
        if (tf < kThreads)
          for (int i = s0; i < s1; ++i) {
            if (tl0 < run + wt[i]) {
              found = i;
              break;
            }
            run += wt[i];
          }
        if (found < 0) {  // rounding left the target past the sums: the last tile with weight
          int i = nt - 1;
          while (i > 0 && !(wt[i] > 0.0f)) --i;
          run = 0.0f;
          for (int j = 0; j < i; ++j) run += wt[j];
          found = i;
          sm.found = 2;
        } else {
          sm.found = 1;
        }
        sm.tile = found;
        sm.tile_base = run;
      }
      __syncthreads();
      if (warp == 0) {
        const int tile = i0 + sm.tile;
        bool clamped = sm.found == 2;
        float w[8];
        multi_weights8<T, VEC>(P, mr, tile * kTile + lane * 8, w);
        float ls = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) ls += w[k];
        float li = ls;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xFFFFFFFFu, li, o);
          if (lane >= o) li += y;
        }
        const float tl = tl0 - sm.tile_base;
        const unsigned hit = clamped ? 0u : __ballot_sync(0xFFFFFFFFu, tl < li);
        int yl, ye = -1;
        float margin = 0.0f;
        if (hit) {
          yl = __ffs(hit) - 1;
          if (lane == yl) {
            float run = li - ls;
            for (int k = 0; k < 8; ++k) {
              if (tl < run + w[k]) {
                ye = k;
                margin = fminf(tl - run, run + w[k] - tl) / R;
                break;
              }
              run += w[k];
            }
            if (ye < 0) {
              for (int k = 7; k >= 0 && ye < 0; --k)
                if (w[k] > 0.0f) ye = k;
              clamped = true;
            }
          }
        } else {
          const unsigned pos = __ballot_sync(0xFFFFFFFFu, ls > 0.0f);
          yl = pos ? 31 - __clz(pos) : 0;
          if (lane == yl)
            for (int k = 7; k >= 0 && ye < 0; --k)
              if (w[k] > 0.0f) ye = k;
          clamped = true;
        }
        if (lane == yl) {
          Smem* lead = cl.map_shared_rank(&sm, 0);
          lead->y = tile * kTile + yl * 8 + (ye < 0 ? 0 : ye);
          lead->margin = clamped ? 0.0f : margin;
          if (clamped) *clamp = 1;
        }
      }
      if (*clamp) atomicOr(&cl.map_shared_rank(&sm, 0)->flags, SPEC_FLAG_CDF_CLAMP);
      *clamp = 0;
    }
  }
  cl.sync();  // rank 0 holds the token; no block leaves while another may still read its total
  return R;
}

// The bonus-style draw of a whole row from p alone (its chunk masses from the stored (max, sum)
// pairs pick the chunk; only that chunk is read again).  Whole block; result in sm.y, sm.margin.
template <typename T, bool VEC>
__device__ void draw_from_summaries(const Params& P, const float2* part, const T* pr, float M, float u, float* wt,
                                    uint4* ring, Smem& sm, int* clamp) {
  const int t = threadIdx.x;
  const int nch = P.nchunk;
  const float Mp2 = M * P.c2;
  for (int c = t; c < nch; c += kThreads) {
    float mass = 0.0f;
    for (int w = 0; w < kWarps; ++w) {
      const float2 pc = __ldcg(part + (size_t)c * kWarps + w);
      if (pc.y != 0.0f) mass += pc.y * ex2(pc.x * P.c2 - Mp2);
    }
    wt[c] = mass;
  }
  __syncthreads();
  if (t == 0) {
    float S = 0.0f;
    for (int c = 0; c < nch; ++c) S += wt[c];
    const float target = u * S;
    float cum = 0.0f;
    int cs = -1;
    for (int c = 0; c < nch; ++c) {
      if (target < cum + wt[c]) {
        cs = c;
        break;
      }
      cum += wt[c];
    }
    if (cs < 0) {  // rounding put u * S past the sum: the last chunk with mass (clamped below)
      cs = nch - 1;
      while (cs > 0 && !(wt[cs] > 0.0f)) --cs;
      cum = 0.0f;
      for (int c = 0; c < cs; ++c) cum += wt[c];
    }
    sm.tile = cs;
    sm.tile_base = target - cum;
    sm.total = S;
  }
  __syncthreads();
  const int cs = sm.tile;
  const float tin = sm.tile_base, S = sm.total;
  __syncthreads();
  DrawRows d;
  d.resid = false;
  d.Mp2 = Mp2;
  d.Lp = 0.0f;
  d.Tp = -INFINITY;
  d.Lq = 0.0f;
  d.c2q = P.c2q;
  d.Tq = 0.0f;
  const int v0 = cs * Cfg<T>::CH;
  draw_range<T, VEC, false>(P, pr, pr, d, v0, min(P.V, v0 + Cfg<T>::CH), false, u, tin, S, wt, ring, sm, clamp);
}

// The per-request pass of spec_verify_multi (MODE kSample or kGreedy; P.B counts sub-requests,
// P.K is the drafts per chain).  Dynamic shared memory: the CDF ring, the tile / chunk sums, then
// the rows' (max, sum) or argmax.
template <typename T, int MODE, bool VEC, int CL>
__global__ void __launch_bounds__(kThreads, sizeof(T) == 2 ? 3 : 2) finish_multi_kernel(const Params P, int N, int32_t* out_chain) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ Smem sm;
  pdl_wait();
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  // with CL > 1 the CL blocks of a cluster all take the request's decisions (identically) and
  // share its stage passes and draws; only rank 0 writes results
  const bool lead = CL == 1 || cooperative_groups::this_cluster().block_rank() == 0;
  const int b = (int)(blockIdx.x / CL), K = P.K, R = P.R, V = P.V;
  uint4* ring = reinterpret_cast<uint4*>(dyn);
  const int ntile = (V + kTile - 1) / kTile;
  float* wt = reinterpret_cast<float*>(dyn + (VEC ? (size_t)kDrawStages * kDrawStageBytes : 0));
  float* rM = wt + (ntile > P.nchunk ? ntile : P.nchunk);
  float* rS = rM + N * R;  // greedy: the argmax, as int bits
  const int s0 = b * N;    // chain n of request b is sub-request s0 + n
  auto part = [&](int n, int rp) { return P.partial + ((size_t)(s0 + n) * R + rp) * P.nchunk * kWarps; };
  auto prow_n = [&](int n, int j) { return static_cast<const T*>(P.p) + ((size_t)(s0 + n) * (K + 1) + j) * (size_t)V; };
  auto qrow_n = [&](int n, int j) { return static_cast<const T*>(P.q) + ((size_t)(s0 + n) * K + j) * (size_t)V; };
  // ---- every row the step read: (max, sum) or (max, lowest argmax); a non-finite row anywhere in
  // the request leaves it without a result ----
  if (t == 0) {
    sm.flags = 0;
    sm.nonfinite = 0;
  }
  __syncthreads();
  for (int r = warp; r < N * R; r += kWarps) {
    const int n = r / R, rp = r - n * R;
    if (n > 0 && rp == 0) continue;  // the shared position is chain 0's row
    const float2* pc0 = part(n, rp);
    if (MODE == kSample) {
      const float c2 = rp > K ? P.c2q : P.c2;
      float m = -INFINITY, s = 0.0f;
      for (int c = lane; c < P.nchunk * kWarps; c += 32) {
        const float2 pc = __ldcg(pc0 + c);
        lse_merge(m, s, pc.x, pc.y, c2);
      }
      lse_warp(m, s, c2);
      if (lane == 0) {
        rM[r] = m;
        rS[r] = s;
        if (!(s > 0.0f) || isinf(m) || isnan(s)) sm.nonfinite = 1;
      }
    } else {
      float best = -INFINITY;
      int bi = 0x7FFFFFFF;
      bool nan = false;
      for (int c = lane; c < P.nchunk * kWarps; c += 32) {
        const float2 pc = __ldcg(pc0 + c);
        const int idx = __float_as_int(pc.y);
        if (idx < 0) nan = true;
        amax_merge(best, bi, pc.x, idx);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float vo = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        const int io = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        amax_merge(best, bi, vo, io);
      }
      nan = __any_sync(0xFFFFFFFFu, nan);
      if (lane == 0) {
        rS[r] = __int_as_float(bi);
        if (nan) sm.nonfinite = 1;
      }
    }
  }
  __syncthreads();
  int32_t* tok = P.out_tokens + (size_t)b * (K + 1);
  auto finish = [&](int nacc, int chain) {
    if (t == 0 && lead) {
      P.out_nacc[b] = nacc;
      if (out_chain) out_chain[b] = chain;
      if (P.flags) P.flags[b] = sm.flags;
    }
  };
  if (sm.nonfinite) {
    if (t <= K && lead) tok[t] = -1;
    if (t == 0) sm.flags |= SPEC_FLAG_NONFINITE;
    __syncthreads();
    finish(0, -1);
    return;
  }
  auto draft = [&](int n, int j) { return __ldg(P.draft + (size_t)(s0 + n) * K + j); };
  if (MODE == kGreedy) {
    if (warp == 0) {
      const int g0 = __float_as_int(rS[0]);
      int chain = -1;
      bool bad = false;
      for (int n = 0; n < N && K > 0 && chain < 0; ++n) {
        const int x = draft(n, 0);
        bad |= x < 0 || x >= V;
        if (x == g0) chain = n;
      }
      int nacc = 0;
      if (chain >= 0) {  // the chain's positions 1..K-1, one per lane, then its argmax at K
        nacc = 1;
        const int j = lane + 1;
        bool acc = true;
        int x = 0;
        if (j < K) {
          x = draft(chain, j);
          acc = x == __float_as_int(rS[chain * R + j]);
        }
        const unsigned rej = __ballot_sync(0xFFFFFFFFu, j < K && !acc);
        const int js = rej ? __ffs(rej) : K;  // the first position (1..K) that emits the argmax
        nacc = js;
        if (rej && lane == js - 1) bad |= x < 0 || x >= V;
        bad = __any_sync(0xFFFFFFFFu, bad);
        if (lane <= K) {
          int v = -1;
          if (lane == 0) v = g0;
          else if (lane < js) v = draft(chain, lane);
          else if (lane == js) v = __float_as_int(rS[chain * R + js]);
          tok[lane] = v;
        }
      } else {
        if (lane <= K) tok[lane] = lane == 0 ? g0 : -1;
      }
      if (lane == 0 && bad) sm.flags |= SPEC_FLAG_BAD_TOKEN;
      if (lane == 0) sm.jstar = nacc, sm.y = chain;
    }
    __syncthreads();
    finish(sm.jstar, sm.y);
    return;
  }
  // ---- sampling: the first position's candidates in turn ----
  const float u = __ldg(P.ur + b);
  auto Lp = [&](int n, int j) { return rM[n * R + j] * P.c2 + log2f(rS[n * R + j]); };
  auto Lq = [&](int n, int j) { return rM[n * R + K + 1 + j] * P.c2q + log2f(rS[n * R + K + 1 + j]); };
  int clamp = 0;
  if (K == 0) {  // no drafts: the one token is drawn from P_0 (one chunk: rank 0 alone)
    if (lead) draw_from_summaries<T, VEC>(P, part(0, 0), prow_n(0, 0), rM[0], u, wt, ring, sm, &clamp);
    if (t == 0 && lead) tok[0] = sm.y;
    if (clamp) atomicOr(&sm.flags, SPEC_FLAG_CDF_CLAMP);  // set by the lane that drew
    __syncthreads();
    finish(0, -1);
    return;
  }
  MultiRows mr;
  mr.row[0] = prow_n(0, 0);
  mr.L[0] = Lp(0, 0);
  for (int n = 0; n < N; ++n) {
    mr.row[1 + n] = qrow_n(n, 0);
    mr.L[1 + n] = Lq(n, 0);
    mr.Rinv[n] = 0.0f;
  }
  int chain = -1;
  for (int n = 0; n < N; ++n) {
    if (t == 0) {  // candidate n against r_n
      const int x = draft(n, 0);
      float a = 0.0f, c = 0.0f;
      if (x >= 0 && x < V) {
        a = ex2(fmaf(load1<T>(static_cast<const T*>(mr.row[0]) + x), P.c2, -mr.L[0]));
        for (int i = 0; i < n; ++i) {
          const float d = a - ex2(fmaf(load1<T>(static_cast<const T*>(mr.row[1 + i]) + x), P.c2q, -mr.L[1 + i]));
          a = mr.Rinv[i] > 0.0f ? fmaxf(d, 0.0f) * mr.Rinv[i] : a;
        }
        c = ex2(fmaf(load1<T>(static_cast<const T*>(mr.row[1 + n]) + x), P.c2q, -mr.L[1 + n]));
      } else {
        sm.flags |= SPEC_FLAG_BAD_TOKEN;
      }
      sm.found = __ldg(P.ua + (size_t)(s0 + n) * K) * c < a;
    }
    __syncthreads();
    const bool accepted = sm.found;
    __syncthreads();
    if (accepted) {
      chain = n;
      break;
    }
    // rejected: R_n, the mass of max(0, r_n - q_n); for the last candidate the draw from it
    mr.n = n;
    mr.sub = true;
    const bool last = n == N - 1;
    const float Rn = CL > 1 ? multi_pass_cluster<T, VEC, CL>(P, mr, last, u, wt, sm, &clamp)
                            : multi_pass<T, VEC>(P, mr, last, u, wt, sm, &clamp);
    mr.Rinv[n] = Rn > 0.0f ? 1.0f / Rn : 0.0f;
    if (!(Rn > 0.0f)) {
      if (t == 0) sm.flags |= SPEC_FLAG_RESIDUAL_ZERO;
      __syncthreads();
      if (last) {  // nothing of r_n survives q_n (rounding): the draw from r_n itself
        mr.sub = false;
        if (CL > 1)
          multi_pass_cluster<T, VEC, CL>(P, mr, true, u, wt, sm, &clamp);
        else
          multi_pass<T, VEC>(P, mr, true, u, wt, sm, &clamp);
      }
    }
  }
  if (chain < 0) {
    if (t <= K && lead) tok[t] = t == 0 ? sm.y : -1;
    if (clamp) atomicOr(&sm.flags, SPEC_FLAG_CDF_CLAMP);  // set by the lane that drew
    __syncthreads();
    finish(0, -1);
    return;
  }
  // ---- the accepted chain from its second position: the single-draft rule on its own rows ----
  if (warp == 0) {
    const int j = lane + 1;  // position j, 1..K-1
    bool acc = true, bad = false;
    int x = 0;
    if (j < K) {
      x = draft(chain, j);
      bad = x < 0 || x >= V;
      float a = 0.0f, cq = 0.0f;
      if (!bad) {
        a = ex2(fmaf(load1<T>(prow_n(chain, j) + x), P.c2, -Lp(chain, j)));
        cq = ex2(fmaf(load1<T>(qrow_n(chain, j) + x), P.c2q, -Lq(chain, j)));
      }
      acc = __ldg(P.ua + (size_t)(s0 + chain) * K + j) * cq < a;
    }
    const unsigned rej = __ballot_sync(0xFFFFFFFFu, j < K && !acc);
    const int js = rej ? __ffs(rej) : K;  // the position that draws (a rejection, or K: the bonus)
    if (rej && lane == js - 1 && bad) sm.flags |= SPEC_FLAG_BAD_TOKEN;
    if (lane <= K && lead) tok[lane] = lane == 0 ? draft(chain, 0) : (lane < js ? draft(chain, lane) : -1);
    if (lane == 0) sm.jstar = js;
  }
  __syncthreads();
  const int js = sm.jstar;
  if (js < K) {  // the residual max(0, P - Q) at the rejected position
    DrawRows d;
    d.resid = true;
    d.Mp2 = rM[chain * R + js] * P.c2;
    d.Lp = Lp(chain, js);
    d.Tp = -INFINITY;
    d.Lq = Lq(chain, js);
    d.c2q = P.c2q;
    d.Tq = -INFINITY;
    const float Rr =
        CL > 1 ? cluster_draw<T, VEC, false, CL>(P, prow_n(chain, js), qrow_n(chain, js), d, u, wt, ring, sm, &clamp)
               : draw_range<T, VEC, false>(P, prow_n(chain, js), qrow_n(chain, js), d, 0, V, true, u, 0.0f, 0.0f, wt,
                                           ring, sm, &clamp);
    if (!(Rr > 0.0f)) {  // max(0, p - q) vanished through rounding: draw from p (R is the same in every block)
      if (t == 0) sm.flags |= SPEC_FLAG_RESIDUAL_ZERO;
      d.resid = false;
      if (CL > 1)
        cluster_draw<T, VEC, false, CL>(P, prow_n(chain, js), prow_n(chain, js), d, u, wt, ring, sm, &clamp);
      else
        draw_range<T, VEC, false>(P, prow_n(chain, js), prow_n(chain, js), d, 0, V, true, u, 0.0f, 0.0f, wt, ring, sm,
                                  &clamp);
    }
  } else if (lead) {  // every draft of the chain accepted: the extra token from its row K (one chunk)
    draw_from_summaries<T, VEC>(P, part(chain, K), prow_n(chain, K), rM[chain * R + K], u, wt, ring, sm, &clamp);
  }
  if (t == 0 && lead) tok[js] = sm.y;
  if (clamp) atomicOr(&sm.flags, SPEC_FLAG_CDF_CLAMP);  // set by the lane that drew
  __syncthreads();
  finish(js, chain);
}

// The row table of spec_verify_multi: request b's chains in order, every row of chain 0 and the
// rows after the first of the other chains (entries (sub-request << 6) | padded row).
__global__ void __launch_bounds__(256) build_rowmap_multi(int B, int N, int R, uint32_t* rowmap, uint32_t* total_rows) {
  const uint32_t per_req = (uint32_t)(N * R - (N - 1));
  for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < B * N; s += gridDim.x * blockDim.x) {
    const int b = s / N, n = s - b * N;
    uint32_t off = (uint32_t)b * per_req + (n == 0 ? 0u : (uint32_t)R + (uint32_t)(n - 1) * (uint32_t)(R - 1));
    for (int rp = n == 0 ? 0 : 1; rp < R; ++rp) rowmap[off++] = ((uint32_t)s << 6) | (uint32_t)rp;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *total_rows = (uint32_t)B * per_req;
}

// Ragged batches: a table of valid rows in request-major order, so no item is spent on padding.
__global__ void __launch_bounds__(1024) build_rowmap(const int32_t* __restrict__ kpr, int B, int K,
                                                     int greedy, uint32_t* rowmap,
                                                     uint32_t* total_rows) {
  __shared__ uint32_t warp_tot[32];
  __shared__ uint32_t carry;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (t == 0) carry = 0;
  __syncthreads();
  for (int b0 = 0; b0 < B; b0 += 1024) {
    const int b = b0 + t;
    uint32_t rows = 0;
    int kb = 0;
    if (b < B) {
      kb = kpr[b];
      kb = kb < 0 ? 0 : (kb > K ? K : kb);
      rows = greedy ? kb + 1 : 2 * kb + 1;
    }
    uint32_t x = rows;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    uint32_t off = carry;
    for (int w = 0; w < warp; ++w) off += warp_tot[w];
    off += x - rows;
    for (uint32_t r = 0; r < rows; ++r) {
      // compact row r of request b -> padded row: p rows 0..kb, then q rows K+1..K+kb
      const uint32_t rp = r <= (uint32_t)kb ? r : (uint32_t)K + 1 + (r - kb - 1);
      rowmap[off + r] = ((uint32_t)b << 6) | rp;
    }
    __syncthreads();
    if (t == 1023) carry = off + rows;
    __syncthreads();
  }
  if (t == 0) *total_rows = carry;
}

// ------------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------------
struct Layout {
  size_t partial, cmeta, cand, rowstat, rowmap, total_rows, bytes;
  int R, nchunk;
  uint64_t rows_padded;
};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace: per-chunk summaries (one pair per warp), top-k candidates, the ragged row table.
// Nothing in it outlives a call, so it needs no initialisation.
static bool make_layout(int B, int K, int V, int es, int mode, bool ragged, Layout* L) {
  const int ch = kChunkBytes / es;
  L->R = mode == kGreedy ? K + 1 : 2 * K + 1;
  L->nchunk = (V + ch - 1) / ch;
  L->rows_padded = (uint64_t)B * L->R;
  const uint64_t items = L->rows_padded * (uint64_t)L->nchunk;
  if (items >= (1ull << 31) || (uint64_t)B >= (1ull << 25)) return false;
  size_t o = 0;
  L->partial = o;
  o = align256(o + (size_t)items * kWarps * sizeof(float2));
  L->cmeta = o;
  L->cand = o;
  if (mode == kTopK) {
    o = align256(o + (size_t)items * sizeof(uint2));
    L->cand = o;
    o = align256(o + (size_t)items * kCandCap * sizeof(uint2));
  }
  L->rowstat = o;
  if (mode != kGreedy) o = align256(o + (size_t)L->rows_padded * sizeof(float2));
  L->rowmap = o;
  L->total_rows = o;
  if (ragged) {
    o = align256(o + (size_t)L->rows_padded * sizeof(uint32_t));
    L->total_rows = o;
    o = align256(o + sizeof(uint32_t));
  }
  L->bytes = o > 0 ? o : 256;
  return true;
}

static int mode_of(float temperature, int top_k, int V) {
  if (temperature == 0.0f) return kGreedy;
  return (top_k > 0 && top_k < V) ? kTopK : kSample;
}

// dynamic shared memory of the two passes
static size_t stats_smem(int mode, bool vec) {
  return mode == kTopK ? (vec ? (size_t)kStagesTopK * kChunkBytes : 0) + (size_t)2 * kSegCap * sizeof(uint2) : 0;
}
static size_t finish_smem(int mode, int V, int es, bool vec, bool nuc) {
  const int ntile = (V + kTile - 1) / kTile;
  const int nch = (V + kChunkBytes / es - 1) / (kChunkBytes / es);
  size_t bytes = (size_t)(ntile > nch ? ntile : nch) * sizeof(float);  // tile / chunk sums
  if (nuc && mode == kTopK && bytes < kNucBufBytes) bytes = kNucBufBytes;  // the nucleus search
  if (mode == kGreedy) return 16;
  if (mode == kTopK) bytes += (size_t)kWarps * kRowCap * sizeof(uint2);
  if (vec) bytes += (size_t)kDrawStages * kDrawStageBytes;  // cp.async ring of the CDF pass
  return bytes;
}

template <typename K>
static cudaError_t prepare(K kern, size_t dsm) {
  if (dsm > 32 * 1024) return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dsm);
  return cudaSuccess;
}

// Launches a pass after the previous kernel of the stream; with `pdl` it may start launching while
// that kernel drains (programmatic stream serialization; the kernel waits in pdl_wait).
template <typename... A>
static cudaError_t launch_after(void (*kern)(A...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                                A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

static cudaError_t sm_count(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  return e;
}

// The streaming pass over `items` (an upper bound when the layout is ragged): short-lived blocks
// in sampling and greedy modes over aligned rows, else the persistent grid, one resident wave of
// it with static contiguous ranges.
template <typename T, int MODE, bool VEC>
static cudaError_t launch_stream(const Params& P, uint64_t items, cudaStream_t st) {
  if constexpr (VEC && MODE != kTopK) {
    const uint64_t g = (items + kItemsPerBlock - 1) / kItemsPerBlock;
    stats_item_kernel<T, MODE, kItemsPerBlock><<<(unsigned)(g > 0 ? g : 1), kThreads, 0, st>>>(P);
    return cudaGetLastError();
  } else {
    auto k1 = stats_kernel<T, MODE, VEC>;
    const size_t d1 = stats_smem(MODE, VEC);
    int sms = 0, occ = 0;
    cudaError_t e = prepare(k1, d1);
    if (e == cudaSuccess) e = sm_count(&sms);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k1, kThreads, d1);
    if (e != cudaSuccess) return e;
    uint64_t grid = (uint64_t)sms * (uint64_t)(occ > 0 ? occ : 1);
    if (items < grid) grid = items > 0 ? items : 1;
    k1<<<(unsigned)grid, kThreads, d1, st>>>(P);
    return cudaGetLastError();
  }
}

// The same with the blocks in clusters of `cl` along x.
template <typename... A>
static cudaError_t launch_cluster_after(void (*kern)(A...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                        bool pdl, unsigned cl, A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = cl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename T, int MODE, bool VEC>
static cudaError_t launch_t(const Params& P, uint32_t items, cudaStream_t st) {
  const int es = (int)sizeof(T);
  const bool nuc = MODE != kGreedy && P.top_p < 1.0f;
  auto k2 = nuc ? finish_kernel<T, MODE, VEC, MODE != kGreedy> : finish_kernel<T, MODE, VEC, false>;
  const size_t d2 = finish_smem(MODE, P.V, es, VEC, nuc);
  int sms = 0;
  cudaError_t e = prepare(k2, d2);
  if (e == cudaSuccess) e = sm_count(&sms);
  if (e == cudaSuccess) e = launch_stream<T, MODE, VEC>(P, items, st);
  if (e == cudaSuccess && P.pass1_done) e = cudaEventRecord(static_cast<cudaEvent_t>(P.pass1_done), st);
  if (e != cudaSuccess) return e;
  // the kernel after the streaming pass overlaps its launch with the pass's tail, unless an event
  // is recorded between them
  const bool pdl = P.pass1_done == nullptr;
  if (nuc && MODE == kSample) {
    auto kn = nucleus_kernel<T, VEC>;
    e = prepare(kn, kNucBufBytes);
    if (e == cudaSuccess)
      e = launch_after(kn, dim3((unsigned)((uint64_t)P.B * P.R)), dim3(kThreads), kNucBufBytes, st, pdl, P);
    if (e != cudaSuccess) return e;
  }
  const bool pdl2 = pdl || (nuc && MODE == kSample);
  if (MODE == kSample && !nuc && P.B <= sms && P.V >= 16384) {
    // few requests: a cluster per request spreads each full-row draw over kCluster SMs
    auto kc = finish_cluster_kernel<T, VEC>;
    e = prepare(kc, d2);
    if (e == cudaSuccess) e = launch_after(kc, dim3((unsigned)P.B * kCluster), dim3(kThreads), d2, st, pdl2, P);
    return e;
  }
  return launch_after(k2, dim3((unsigned)P.B), dim3(kThreads), d2, st, pdl2, P);
}

template <typename T>
static cudaError_t launch_mode(int mode, bool vec, const Params& P, uint32_t items, cudaStream_t st) {
  switch (mode) {
    case kSample:
      return vec ? launch_t<T, kSample, true>(P, items, st) : launch_t<T, kSample, false>(P, items, st);
    case kTopK:
      return vec ? launch_t<T, kTopK, true>(P, items, st) : launch_t<T, kTopK, false>(P, items, st);
    default:
      return vec ? launch_t<T, kGreedy, true>(P, items, st) : launch_t<T, kGreedy, false>(P, items, st);
  }
}

// spec_verify_multi: the row table, the streaming pass over the table, the per-request pass.
template <typename T, int MODE, bool VEC>
static cudaError_t launch_multi(const Params& P, int Breq, int N, int32_t* out_chain, cudaStream_t st) {
  auto k2 = finish_multi_kernel<T, MODE, VEC, 1>;
  auto kc = finish_multi_kernel<T, MODE, VEC, kMultiCluster>;
  const int ntile = (P.V + kTile - 1) / kTile;
  const size_t d2 = (VEC ? (size_t)kDrawStages * kDrawStageBytes : 0) +
                    (size_t)(ntile > P.nchunk ? ntile : P.nchunk) * sizeof(float) + (size_t)2 * N * P.R * sizeof(float);
  cudaError_t e = prepare(k2, d2);
  if (e == cudaSuccess && MODE == kSample) e = prepare(kc, d2);
  if (e != cudaSuccess) return e;
  const uint32_t rows = (uint32_t)Breq * (uint32_t)(N * P.R - (N - 1));
  const uint64_t items = (uint64_t)rows * (uint64_t)P.nchunk;
  const unsigned rb = (unsigned)(((uint64_t)Breq * N + 255) / 256);
  build_rowmap_multi<<<rb < 1024u ? (rb > 0 ? rb : 1u) : 1024u, 256, 0, st>>>(
      Breq, N, P.R, const_cast<uint32_t*>(P.rowmap), const_cast<uint32_t*>(P.total_rows));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_stream<T, MODE, VEC>(P, items, st);
  if (e != cudaSuccess) return e;
  if (MODE == kSample)  // a cluster per request shares its stage passes and draws
    return launch_cluster_after(kc, dim3((unsigned)Breq * kMultiCluster), dim3(kThreads), d2, st, true,
                                (unsigned)kMultiCluster, P, N, out_chain);
  return launch_after(k2, dim3((unsigned)Breq), dim3(kThreads), d2, st, true, P, N, out_chain);
}

}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_verify_workspace_bytes(int32_t B, int32_t K_max, int32_t V, spec_dtype_t dtype,
                                   int32_t top_k) {
  if (B < 0 || K_max < 0 || V <= 0 || K_max > SPEC_MAX_K || V > SPEC_MAX_V) return 0;
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return 0;
  if (top_k < 0) return 0;
  // the largest layout over the three modes, so one workspace serves any temperature
  Layout a, b;
  const int heavy = (top_k > 0 && top_k < V) ? kTopK : kSample;
  const int es = dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  if (!make_layout(B, K_max, V, es, heavy, true, &a) || !make_layout(B, K_max, V, es, kGreedy, true, &b)) return 0;
  return a.bytes > b.bytes ? a.bytes : b.bytes;
}

}  // extern "C"

namespace sv {
std::atomic<int32_t> g_test_hooks{0};  // spec_verify_set_test_hooks
}  // namespace sv

// The host-side checks of a verify call, in order, and the workspace layout of the call's own mode
// (sampling, top-k or greedy) and row layout.  SPEC_OK with *empty set for B == 0 (nothing to do).
static spec_status_t check_call(const void* p_logits, const void* q_logits, const int32_t* draft_tokens,
                                const int32_t* k_per_row, const float* u_accept, const float* u_resample,
                                const spec_sampling_t* sampling, const int32_t* out_tokens,
                                const int32_t* out_num_accepted, int32_t B, int32_t K_max, int32_t V,
                                spec_dtype_t dtype, int* mode_out, Layout* L, bool* empty) {
  *empty = false;
  if (B < 0 || K_max < 0 || V <= 0 || !sampling) return SPEC_ERR_INVALID_ARG;
  const float temperature = sampling->temperature, tq = sampling->draft_temperature;
  const int32_t top_k = sampling->top_k;
  const float top_p = sampling->top_p;
  if (!(temperature >= 0.0f) || isinf(temperature) || top_k < 0) return SPEC_ERR_INVALID_ARG;
  if (temperature > 0.0f && (!(tq > 0.0f) || isinf(tq))) return SPEC_ERR_INVALID_ARG;
  if (!(top_p > 0.0f)) return SPEC_ERR_INVALID_ARG;
  if (K_max > SPEC_MAX_K || V > SPEC_MAX_V) return SPEC_ERR_UNSUPPORTED;
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED;
  const int mode = mode_of(temperature, top_k, V);
  if (mode == kTopK && top_k > SPEC_MAX_TOPK) return SPEC_ERR_UNSUPPORTED;
  *mode_out = mode;
  if (B == 0) {  // nothing to read or write (empty arrays may have null pointers)
    *empty = true;
    return SPEC_OK;
  }
  if (!p_logits || !out_tokens || !out_num_accepted) return SPEC_ERR_INVALID_ARG;
  if (K_max > 0 && !draft_tokens) return SPEC_ERR_INVALID_ARG;
  if (mode != kGreedy && (!u_resample || (K_max > 0 && (!q_logits || !u_accept))))
    return SPEC_ERR_INVALID_ARG;
  if (!make_layout(B, K_max, V, dtype == SPEC_DTYPE_BF16 ? 2 : 4, mode, k_per_row != nullptr, L))
    return SPEC_ERR_UNSUPPORTED;
  return SPEC_OK;
}

// spec_verify_ex with, for the sampler, q(x) of each request's drawn token written to sample_prob.
static spec_status_t verify_impl(const void* p_logits, const void* q_logits, const int32_t* draft_tokens,
                                 const int32_t* k_per_row, const float* u_accept, const float* u_resample,
                                 const spec_sampling_t* sampling, int32_t* out_tokens, int32_t* out_num_accepted,
                                 const spec_verify_stats_t* out_stats, int32_t B, int32_t K_max, int32_t V,
                                 spec_dtype_t dtype, void* workspace, size_t workspace_bytes, void* stream,
                                 float* sample_prob) {
  int mode = kSample;
  Layout L;
  bool empty = false;
  const spec_status_t chk = check_call(p_logits, q_logits, draft_tokens, k_per_row, u_accept, u_resample, sampling,
                                       out_tokens, out_num_accepted, B, K_max, V, dtype, &mode, &L, &empty);
  if (chk != SPEC_OK || empty) return chk;
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < L.bytes) return SPEC_ERR_WORKSPACE;
  const float temperature = sampling->temperature, tq = sampling->draft_temperature;
  const int32_t top_k = sampling->top_k;
  const float top_p = sampling->top_p;
  const bool ragged = k_per_row != nullptr;

  const size_t es = dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  const bool vec = ((uintptr_t)p_logits % 16 == 0) && (!q_logits || (uintptr_t)q_logits % 16 == 0) &&
                   ((size_t)V * es % 16 == 0);
  char* ws = static_cast<char*>(workspace);
  Params P;
  P.p = p_logits;
  P.q = mode == kGreedy ? nullptr : q_logits;
  P.draft = draft_tokens;
  P.kpr = k_per_row;
  P.ua = u_accept;
  P.ur = u_resample;
  P.out_tokens = out_tokens;
  P.out_nacc = out_num_accepted;
  spec_verify_stats_t st = {};
  if (out_stats) st = *out_stats;
  P.p_draft = st.p_draft;
  P.q_draft = st.q_draft;
  P.acc_margin = st.accept_margin;
  P.samp_margin = st.sample_margin;
  P.resid_mass = st.residual_mass;
  P.lognorm = st.row_lognorm;
  P.rowcut = st.row_cut;
  P.sample_prob = sample_prob;
  P.test_hooks = sv::g_test_hooks.load(std::memory_order_relaxed);
  P.flags = st.flags;
  P.pass1_done = st.pass1_done;
  P.B = B;
  P.K = K_max;
  P.V = V;
  P.top_k = top_k;
  P.nchunk = L.nchunk;
  P.R = L.R;
  const double T = temperature, Tq = tq;
  P.c2 = mode == kGreedy ? 0.0f : (float)(1.4426950408889634 / T);
  P.invT = mode == kGreedy ? 0.0f : (float)(1.0 / T);
  P.c2q = mode == kGreedy ? 0.0f : (float)(1.4426950408889634 / Tq);
  P.invTq = mode == kGreedy ? 0.0f : (float)(1.0 / Tq);
  P.top_p = top_p >= 1.0f ? 1.0f : top_p;
  P.partial = reinterpret_cast<float2*>(ws + L.partial);
  P.cmeta = reinterpret_cast<uint2*>(ws + L.cmeta);
  P.cand = reinterpret_cast<uint2*>(ws + L.cand);
  P.rowstat = reinterpret_cast<float2*>(ws + L.rowstat);
  P.rowmap = ragged ? reinterpret_cast<const uint32_t*>(ws + L.rowmap) : nullptr;
  P.total_rows = ragged ? reinterpret_cast<const uint32_t*>(ws + L.total_rows) : nullptr;
  P.uniform_items = (uint32_t)(L.rows_padded * (uint64_t)L.nchunk);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (ragged) {
    build_rowmap<<<1, 1024, 0, s>>>(k_per_row, B, K_max, mode == kGreedy,
                                    reinterpret_cast<uint32_t*>(ws + L.rowmap),
                                    reinterpret_cast<uint32_t*>(ws + L.total_rows));
    if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  }
  const uint32_t items = P.uniform_items;  // an upper bound on the grid's useful size
  cudaError_t e = dtype == SPEC_DTYPE_BF16 ? launch_mode<uint16_t>(mode, vec, P, items, s)
                                           : launch_mode<float>(mode, vec, P, items, s);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

extern "C" {

spec_status_t spec_verify_ex(const void* p_logits, const void* q_logits, const int32_t* draft_tokens,
                             const int32_t* k_per_row, const float* u_accept, const float* u_resample,
                             const spec_sampling_t* sampling, int32_t* out_tokens,
                             int32_t* out_num_accepted, const spec_verify_stats_t* out_stats, int32_t B,
                             int32_t K_max, int32_t V, spec_dtype_t dtype, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return verify_impl(p_logits, q_logits, draft_tokens, k_per_row, u_accept, u_resample, sampling, out_tokens,
                     out_num_accepted, out_stats, B, K_max, V, dtype, workspace, workspace_bytes, stream, nullptr);
}

spec_status_t spec_verify(const void* p_logits, const void* q_logits, const int32_t* draft_tokens,
                          const int32_t* k_per_row, const float* u_accept, const float* u_resample,
                          float temperature, int32_t top_k, int32_t* out_tokens,
                          int32_t* out_num_accepted, const spec_verify_stats_t* out_stats, int32_t B,
                          int32_t K_max, int32_t V, spec_dtype_t dtype, void* workspace,
                          size_t workspace_bytes, void* stream) {
  const spec_sampling_t sp = {temperature, temperature, top_k, 1.0f};
  return spec_verify_ex(p_logits, q_logits, draft_tokens, k_per_row, u_accept, u_resample, &sp, out_tokens,
                        out_num_accepted, out_stats, B, K_max, V, dtype, workspace, workspace_bytes, stream);
}

size_t spec_verify_host_staging_bytes(int32_t B, int32_t K_max, int32_t V, spec_dtype_t dtype,
                                      int32_t top_k, int32_t has_k_per_row) {
  const size_t ws = spec_verify_workspace_bytes(B, K_max, V, dtype, top_k);
  if (ws == 0) return 0;
  const size_t es = dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  size_t o = 0;
  o = align256(o + (size_t)B * (K_max + 1) * V * es);  // p
  o = align256(o + (size_t)B * K_max * V * es);        // q
  o = align256(o + (size_t)B * K_max * 4);             // draft
  o = align256(o + (size_t)(has_k_per_row ? B : 0) * 4);
  o = align256(o + (size_t)B * K_max * 4);  // ua
  o = align256(o + (size_t)B * 4);          // ur
  o = align256(o + (size_t)B * (K_max + 1) * 4);  // tokens
  o = align256(o + (size_t)B * 4);                // n_acc
  return o + ws;
}

spec_status_t spec_verify_host_ex(const void* p_logits, const void* q_logits,
                                  const int32_t* draft_tokens, const int32_t* k_per_row,
                                  const float* u_accept, const float* u_resample,
                                  const spec_sampling_t* sampling, int32_t* out_tokens,
                                  int32_t* out_num_accepted, int32_t B, int32_t K_max, int32_t V,
                                  spec_dtype_t dtype, void* staging, size_t staging_bytes, void* stream) {
  if (!sampling) return SPEC_ERR_INVALID_ARG;
  const float temperature = sampling->temperature;
  const int32_t top_k = sampling->top_k;
  if (B < 0 || K_max < 0 || V <= 0 || K_max > SPEC_MAX_K || V > SPEC_MAX_V) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED;
  const size_t need = spec_verify_host_staging_bytes(B, K_max, V, dtype, top_k, k_per_row != nullptr);
  if (need == 0) return SPEC_ERR_INVALID_ARG;
  if (!staging || ((uintptr_t)staging & 255u) || staging_bytes < need) return SPEC_ERR_WORKSPACE;
  if (!p_logits || !out_tokens || !out_num_accepted) return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  const bool greedy = temperature == 0.0f;
  const size_t es = dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  char* d = static_cast<char*>(staging);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    char* p = d + o;
    o = align256(o + bytes);
    return p;
  };
  const size_t np = (size_t)B * (K_max + 1) * V * es, nq = (size_t)B * K_max * V * es;
  char* dp = take(np);
  char* dq = take(nq);
  char* dx = take((size_t)B * K_max * 4);
  char* dk = take((size_t)(k_per_row ? B : 0) * 4);
  char* dua = take((size_t)B * K_max * 4);
  char* dur = take((size_t)B * 4);
  char* dtok = take((size_t)B * (K_max + 1) * 4);
  char* dn = take((size_t)B * 4);
  char* dws = d + o;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(dp, p_logits, np, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && !greedy && q_logits && nq) e = cudaMemcpyAsync(dq, q_logits, nq, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && draft_tokens && K_max) e = cudaMemcpyAsync(dx, draft_tokens, (size_t)B * K_max * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && k_per_row) e = cudaMemcpyAsync(dk, k_per_row, (size_t)B * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && !greedy && u_accept && K_max) e = cudaMemcpyAsync(dua, u_accept, (size_t)B * K_max * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && !greedy && u_resample) e = cudaMemcpyAsync(dur, u_resample, (size_t)B * 4, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  spec_status_t r = spec_verify_ex(dp, greedy ? nullptr : (q_logits ? dq : nullptr),
                                   draft_tokens ? (const int32_t*)dx : nullptr, k_per_row ? (const int32_t*)dk : nullptr,
                                   greedy ? nullptr : (u_accept ? (const float*)dua : nullptr),
                                   greedy ? nullptr : (u_resample ? (const float*)dur : nullptr), sampling,
                                   (int32_t*)dtok, (int32_t*)dn, nullptr, B, K_max, V, dtype, dws,
                                   staging_bytes - (size_t)(dws - d), stream);
  if (r != SPEC_OK) return r;
  e = cudaMemcpyAsync(out_tokens, dtok, (size_t)B * (K_max + 1) * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(out_num_accepted, dn, (size_t)B * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status_t spec_verify_host(const void* p_logits, const void* q_logits,
                               const int32_t* draft_tokens, const int32_t* k_per_row,
                               const float* u_accept, const float* u_resample, float temperature,
                               int32_t top_k, int32_t* out_tokens, int32_t* out_num_accepted,
                               int32_t B, int32_t K_max, int32_t V, spec_dtype_t dtype,
                               void* staging, size_t staging_bytes, void* stream) {
  const spec_sampling_t sp = {temperature, temperature, top_k, 1.0f};
  return spec_verify_host_ex(p_logits, q_logits, draft_tokens, k_per_row, u_accept, u_resample, &sp,
                             out_tokens, out_num_accepted, B, K_max, V, dtype, staging, staging_bytes, stream);
}

size_t spec_sample_workspace_bytes(int32_t rows, int32_t V, spec_dtype_t dtype, int32_t top_k) {
  const size_t ws = spec_verify_workspace_bytes(rows, 0, V, dtype, top_k);
  if (ws == 0) return 0;
  return ws + align256((size_t)rows * sizeof(int32_t));  // + the accepted counts
}

spec_status_t spec_sample(const void* logits, const float* u, const spec_sampling_t* sampling, int32_t* out_tokens,
                          float* out_prob, int32_t rows, int32_t V, spec_dtype_t dtype, void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (rows < 0 || V <= 0 || !sampling) return SPEC_ERR_INVALID_ARG;
  if (V > SPEC_MAX_V) return SPEC_ERR_UNSUPPORTED;
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED;
  spec_sampling_t sp = *sampling;
  sp.draft_temperature = sp.temperature > 0.0f ? sp.temperature : 1.0f;  // there are no q rows
  const size_t base = spec_verify_workspace_bytes(rows, 0, V, dtype, sp.top_k > 0 ? sp.top_k : 0);
  if (base == 0) return SPEC_ERR_INVALID_ARG;
  const size_t need = spec_sample_workspace_bytes(rows, V, dtype, sp.top_k > 0 ? sp.top_k : 0);
  char* ws = static_cast<char*>(workspace);
  if (rows > 0 && (!ws || ((uintptr_t)ws & 255u) || workspace_bytes < need)) return SPEC_ERR_WORKSPACE;
  int32_t* nacc = rows > 0 ? reinterpret_cast<int32_t*>(ws + base) : nullptr;
  // a request with no drafts: its one token is the draw from p at position 0 (the bonus draw); the
  // per-request pass also writes q(x) of the drawn token
  return verify_impl(logits, nullptr, nullptr, nullptr, nullptr, u, &sp, out_tokens, nacc, nullptr, rows, 0, V,
                     dtype, ws, base, stream, rows > 0 ? out_prob : nullptr);
}

size_t spec_verify_multi_workspace_bytes(int32_t B, int32_t N, int32_t K_max, int32_t V, spec_dtype_t dtype) {
  if (B < 0 || N < 1 || N > SPEC_MAX_DRAFTS || K_max < 0 || K_max > SPEC_MAX_K || V <= 0 || V > SPEC_MAX_V) return 0;
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return 0;
  if ((int64_t)B * N >= (1ll << 25)) return 0;
  const int es = dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  Layout a, g;
  if (!make_layout(B * N, K_max, V, es, kSample, true, &a) || !make_layout(B * N, K_max, V, es, kGreedy, true, &g))
    return 0;
  return a.bytes > g.bytes ? a.bytes : g.bytes;
}

spec_status_t spec_verify_multi(const void* p_logits, const void* q_logits, const int32_t* draft_tokens,
                                const float* u_accept, const float* u_resample, const spec_sampling_t* sampling,
                                int32_t* out_tokens, int32_t* out_num_accepted, int32_t* out_chain,
                                int32_t* out_flags, int32_t B, int32_t N, int32_t K_max, int32_t V,
                                spec_dtype_t dtype, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || N < 1 || K_max < 0 || V <= 0 || !sampling) return SPEC_ERR_INVALID_ARG;
  const float T = sampling->temperature, Tq = sampling->draft_temperature;
  if (!(T >= 0.0f) || isinf(T) || sampling->top_k < 0) return SPEC_ERR_INVALID_ARG;
  if (T > 0.0f && (!(Tq > 0.0f) || isinf(Tq))) return SPEC_ERR_INVALID_ARG;
  if (!(sampling->top_p > 0.0f)) return SPEC_ERR_INVALID_ARG;
  if (N > SPEC_MAX_DRAFTS || K_max > SPEC_MAX_K || V > SPEC_MAX_V) return SPEC_ERR_UNSUPPORTED;
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED;
  if ((sampling->top_k > 0 && sampling->top_k < V) || sampling->top_p < 1.0f) return SPEC_ERR_UNSUPPORTED;
  if ((int64_t)B * N >= (1ll << 25)) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  const bool greedy = T == 0.0f;
  if (!p_logits || !out_tokens || !out_num_accepted) return SPEC_ERR_INVALID_ARG;
  if (K_max > 0 && !draft_tokens) return SPEC_ERR_INVALID_ARG;
  if (!greedy && (!u_resample || (K_max > 0 && (!q_logits || !u_accept)))) return SPEC_ERR_INVALID_ARG;
  const int mode = greedy ? kGreedy : kSample;
  const size_t es = dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  Layout L;
  if (!make_layout(B * N, K_max, V, (int)es, mode, true, &L)) return SPEC_ERR_UNSUPPORTED;
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < L.bytes) return SPEC_ERR_WORKSPACE;
  const bool vec = ((uintptr_t)p_logits % 16 == 0) && (!q_logits || (uintptr_t)q_logits % 16 == 0) &&
                   ((size_t)V * es % 16 == 0);
  char* ws = static_cast<char*>(workspace);
  Params P = {};
  P.p = p_logits;
  P.q = greedy ? nullptr : q_logits;
  P.draft = draft_tokens;
  P.kpr = nullptr;
  P.ua = u_accept;
  P.ur = u_resample;
  P.out_tokens = out_tokens;
  P.out_nacc = out_num_accepted;
  P.flags = out_flags;
  P.test_hooks = sv::g_test_hooks.load(std::memory_order_relaxed);
  P.B = B * N;
  P.K = K_max;
  P.V = V;
  P.top_k = 0;
  P.nchunk = L.nchunk;
  P.R = L.R;
  P.c2 = greedy ? 0.0f : (float)(1.4426950408889634 / (double)T);
  P.invT = greedy ? 0.0f : (float)(1.0 / (double)T);
  P.c2q = greedy ? 0.0f : (float)(1.4426950408889634 / (double)Tq);
  P.invTq = greedy ? 0.0f : (float)(1.0 / (double)Tq);
  P.top_p = 1.0f;
  P.partial = reinterpret_cast<float2*>(ws + L.partial);
  P.cmeta = reinterpret_cast<uint2*>(ws + L.cmeta);
  P.cand = reinterpret_cast<uint2*>(ws + L.cand);
  P.rowstat = reinterpret_cast<float2*>(ws + L.rowstat);
  P.rowmap = reinterpret_cast<const uint32_t*>(ws + L.rowmap);
  P.total_rows = reinterpret_cast<const uint32_t*>(ws + L.total_rows);
  P.uniform_items = (uint32_t)(L.rows_padded * (uint64_t)L.nchunk);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (dtype == SPEC_DTYPE_BF16)
    e = greedy ? (vec ? launch_multi<uint16_t, kGreedy, true>(P, B, N, out_chain, s)
                      : launch_multi<uint16_t, kGreedy, false>(P, B, N, out_chain, s))
               : (vec ? launch_multi<uint16_t, kSample, true>(P, B, N, out_chain, s)
                      : launch_multi<uint16_t, kSample, false>(P, B, N, out_chain, s));
  else
    e = greedy ? (vec ? launch_multi<float, kGreedy, true>(P, B, N, out_chain, s)
                      : launch_multi<float, kGreedy, false>(P, B, N, out_chain, s))
               : (vec ? launch_multi<float, kSample, true>(P, B, N, out_chain, s)
                      : launch_multi<float, kSample, false>(P, B, N, out_chain, s));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

void spec_verify_set_test_hooks(int32_t hooks) { sv::g_test_hooks.store(hooks, std::memory_order_relaxed); }

const char* spec_verify_status_string(spec_status_t status) {
  switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_UNSUPPORTED: return "unsupported size, dtype or option";
    case SPEC_ERR_CUDA: return "CUDA runtime error";
    case SPEC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SPEC_ERR_TIMEOUT: return "timeout";
  }
  return "unknown status";
}

}  // extern "C"

// ------------------------------------------------------------------------------------------------
// spec_verify_static: the same step with its scratch in a fixed device array
// ------------------------------------------------------------------------------------------------
// Some callers have no way to hand this library device memory: a custom operator inside a host
// framework whose memory pool owns every allocation, or a loop that must never block (cudaMalloc
// and cudaFree can synchronise the device).  For them, the scratch lives in one file-scope device
// array that every GPU loading this library holds until the process exits.  Its address is a
// device address that host code can only learn through cudaGetSymbolAddress, once per device.

namespace sv {
constexpr size_t kStaticScratchBytes = (size_t)SPEC_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];  // per device: the array's device address
}  // namespace sv

static __device__ __align__(256) unsigned char g_static_scratch[sv::kStaticScratchBytes];

extern "C" spec_status_t spec_verify_static(const void* p_logits, const void* q_logits,
                                            const int32_t* draft_tokens, const int32_t* k_per_row,
                                            const float* u_accept, const float* u_resample,
                                            float temperature, int32_t top_k, int32_t* out_tokens,
                                            int32_t* out_num_accepted,
                                            const spec_verify_stats_t* out_stats, int32_t B,
                                            int32_t K_max, int32_t V, spec_dtype_t dtype,
                                            void* stream) {
  // the same host-side checks as spec_verify, in the same order, then the workspace of this call's
  // own mode and row layout against the fixed array
  const spec_sampling_t sp = {temperature, temperature, top_k, 1.0f};
  int mode = 0;
  sv::Layout L;
  bool empty = false;
  const spec_status_t chk = check_call(p_logits, q_logits, draft_tokens, k_per_row, u_accept, u_resample, &sp,
                                       out_tokens, out_num_accepted, B, K_max, V, dtype, &mode, &L, &empty);
  if (chk != SPEC_OK || empty) return chk;
  if (L.bytes > sv::kStaticScratchBytes) return SPEC_ERR_WORKSPACE;  // beyond the fixed array
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= sv::kMaxDevices) return SPEC_ERR_CUDA;
  void* scratch = sv::g_scratch_addr[dev].load(std::memory_order_acquire);
  if (scratch == nullptr) {  // first call on this device (the current one): look the address up
    if (cudaGetSymbolAddress(&scratch, g_static_scratch) != cudaSuccess || scratch == nullptr)
      return SPEC_ERR_CUDA;
    sv::g_scratch_addr[dev].store(scratch, std::memory_order_release);
  }
  return spec_verify(p_logits, q_logits, draft_tokens, k_per_row, u_accept, u_resample, temperature,
                     top_k, out_tokens, out_num_accepted, out_stats, B, K_max, V, dtype, scratch,
                     sv::kStaticScratchBytes, stream);
}
