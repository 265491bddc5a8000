// Acceptance: greedy longest matching path, or tree rejection sampling.
//
// Greedy: "최적화 2편" (beengineer500), section 1.3 — drafts matching the
// target's own prediction are kept, the first mismatch takes the target's
// prediction and everything after it is dropped; an all-match yields one extra
// token. On the tree the matching child is unique (siblings carry distinct
// tokens), so the walk is the longest matching path.
//
// Rejection sampling: "Medusa 심층 아키텍처" (techknowgenie), section "수학적
// 무손실 보장", equations alpha(x) = min(1, p(x)/q(x)) and
// p'(x) = max(0, p(x) - q(x)) / sum_y max(0, p(y) - q(y)); "Speculative Decoding
// 원리와 가속 아키텍처" (blog.huny.dev), section 2.1. Applied at each depth of the
// walk, siblings tried in rank order, the residual carried across siblings;
// draws use inverse CDF (smallest y with cdf(y) > u * total).
//
// Two launches per call. Greedy: every tree node's target-row argmax in
// parallel (one CTA per row), then a one-thread-per-sequence walk. Rejection
// sampling: the max and softmax normaliser of every head's logit row in
// parallel, then one CTA per sequence walks; at each visited node one sweep
// gives the target row's max and normaliser, an acceptance test is O(1), and
// only a rejection (the residual's normaliser) and the final draw (inverse CDF)
// sweep the row again. Bulk sums use the hardware base-2 exponential; the
// acceptance ratios use the accurate one.
// Sums use compensated float32 pairs: float64 is slow on this part and plain
// float32 prefix sums over 32k entries drift by ~1e-6 of the total, the width
// of the inverse-CDF tie band.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace medusa {
namespace {

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// ---------------------------------------------------------------- compensated sums
struct FF {
  float hi, lo;
};
__device__ __forceinline__ FF two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  return {s, (a - (s - bb)) + (b - bb)};
}
__device__ __forceinline__ FF ff_norm(float hi, float lo) {
  const float s = hi + lo;
  return {s, lo - (s - hi)};
}
__device__ __forceinline__ FF ff_add(FF x, float y) {
  FF s = two_sum(x.hi, y);
  return ff_norm(s.hi, s.lo + x.lo);
}
__device__ __forceinline__ FF ff_add(FF x, FF y) {
  FF s = two_sum(x.hi, y.hi);
  return ff_norm(s.hi, s.lo + x.lo + y.lo);
}
__device__ __forceinline__ FF ff_shfl_xor(FF v, int o) {
  return {__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ FF ff_shfl_up(FF v, int o) {
  return {__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ float ff_diff(FF a, FF b) { return (a.hi - b.hi) + (a.lo - b.lo); }

template <int NW>
struct Scratch {
  float hi[NW], lo[NW], f[NW];
  int i[NW];
  FF tot;
  float bf;
  int bi;
};

template <int NW>
__device__ FF block_sum_ff(FF v, Scratch<NW>& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = ff_add(v, ff_shfl_xor(v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    s.hi[threadIdx.x >> 5] = v.hi;
    s.lo[threadIdx.x >> 5] = v.lo;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    FF w = threadIdx.x < NW ? FF{s.hi[threadIdx.x], s.lo[threadIdx.x]} : FF{0.f, 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w = ff_add(w, ff_shfl_xor(w, o));
    if (threadIdx.x == 0) s.tot = w;
  }
  __syncthreads();
  return s.tot;
}

template <int NW>
__device__ float block_max(float v, Scratch<NW>& s) {
  v = warp_max(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s.f[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float w = threadIdx.x < NW ? s.f[threadIdx.x] : -INFINITY;
    w = warp_max(w);
    if (threadIdx.x == 0) s.bf = w;
  }
  __syncthreads();
  return s.bf;
}

template <int NW>
__device__ int block_min_i(int v, Scratch<NW>& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s.i[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    int w = threadIdx.x < NW ? s.i[threadIdx.x] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w = min(w, __shfl_xor_sync(0xffffffffu, w, o));
    if (threadIdx.x == 0) s.bi = w;
  }
  __syncthreads();
  return s.bi;
}

// Exclusive scan (thread order) of one FF per thread; also returns the total.
template <int NW>
__device__ FF block_exscan_ff(FF v, Scratch<NW>& s, FF* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  FF incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    FF t = ff_shfl_up(incl, o);
    if (lane >= o) incl = ff_add(incl, t);
  }
  __syncthreads();
  if (lane == 31) {
    s.hi[warp] = incl.hi;
    s.lo[warp] = incl.lo;
  }
  __syncthreads();
  if (warp == 0) {
    FF w = lane < NW ? FF{s.hi[lane], s.lo[lane]} : FF{0.f, 0.f};
    FF wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      FF t = ff_shfl_up(wi, o);
      if (lane >= o) wi = ff_add(wi, t);
    }
    __syncwarp();
    if (lane < NW) {
      FF ex = ff_add(wi, FF{-w.hi, -w.lo});
      s.hi[lane] = ex.hi;
      s.lo[lane] = ex.lo;
    }
    if (lane == 31) s.tot = wi;
  }
  __syncthreads();
  *total = s.tot;
  FF base{s.hi[warp], s.lo[warp]};
  return ff_add(base, ff_add(incl, FF{-v.hi, -v.lo}));
}

// ---------------------------------------------------------------- vector row access
// 8 consecutive entries of a row as floats (one 16-byte load for bf16, two for f32).
template <typename T>
__device__ __forceinline__ void load8(const T* row, int v, float* x);
template <>
__device__ __forceinline__ void load8<uint16_t>(const uint16_t* row, int v, float* x) {
  const uint4 u = *reinterpret_cast<const uint4*>(row + v);
  x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
  x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}
template <>
__device__ __forceinline__ void load8<float>(const float* row, int v, float* x) {
  const float4 a = *reinterpret_cast<const float4*>(row + v);
  const float4 b = *reinterpret_cast<const float4*>(row + v + 4);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// ---------------------------------------------------------------- row pass (parallel)
constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / 32;

// Greedy: amax[b][n] = argmax_v target[b][n][v] (lowest index on ties). grid (N, B).
// VEC: rows are read 8 entries at a time (V % 8 == 0), all of a thread's loads in flight.
template <typename T, bool VEC>
__global__ void __launch_bounds__(kRowThreads)
row_argmax_kernel(const T* __restrict__ tl, int N, int V, int32_t* __restrict__ amax) {
  const int n = blockIdx.x, b = blockIdx.y;
  const T* row = tl + ((size_t)b * N + n) * V;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  if (VEC) {
    constexpr int kU = 8;   // vectors per thread per round
    for (int base = 0; base < V; base += kU * 8 * kRowThreads) {
      float x[kU][8];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int v = base + 8 * (threadIdx.x + u * kRowThreads);
        if (v < V) load8<T>(row, v, x[u]);
        else
#pragma unroll
          for (int e = 0; e < 8; ++e) x[u][e] = -INFINITY;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int v = base + 8 * (threadIdx.x + u * kRowThreads) + e;
          if (better(x[u][e], v, bv, bi)) {
            bv = x[u][e];
            bi = v;
          }
        }
    }
  } else {
#pragma unroll 4
    for (int v = threadIdx.x; v < V; v += kRowThreads) {
      const float x = Elt<T>::load(row, v);
      if (better(x, v, bv, bi)) {
        bv = x;
        bi = v;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
  __shared__ float sv[kRowWarps];
  __shared__ int si[kRowWarps];
  if ((threadIdx.x & 31) == 0) {
    sv[threadIdx.x >> 5] = bv;
    si[threadIdx.x >> 5] = bi;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    bv = threadIdx.x < kRowWarps ? sv[threadIdx.x] : -INFINITY;
    bi = threadIdx.x < kRowWarps ? si[threadIdx.x] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (threadIdx.x == 0) amax[(size_t)b * N + n] = bi;
  }
}

// exp(y * c) for the bulk sums, c = log2(e) / T folded in by the caller: one
// multiply and the hardware base-2 exponential. Relative error stays near
// 2e-7 where the probability mass is (|y * c| of a few units).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Sum of 8 values as a short tree (independent adds), then into the compensated pair.
__device__ __forceinline__ FF ff_add8(FF acc, const float* e) {
  const float a = (e[0] + e[1]) + (e[2] + e[3]);
  const float b = (e[4] + e[5]) + (e[6] + e[7]);
  return ff_add(ff_add(acc, a), b);
}

// Rejection sampling, head rows: m = max and Z = sum exp((v - m) / T) of every
// head's logit row. grid (K, B); stats[b][k] = (m, Z). Two sweeps (the second
// hits L2); rows with V % 8 == 0 are read 8 entries at a time.
template <bool VEC>
__global__ void __launch_bounds__(kRowThreads)
head_stats_kernel(const float* __restrict__ hl, int K, int V, float c, float2* __restrict__ stats) {
  __shared__ Scratch<kRowWarps> s;
  const int k = blockIdx.x, b = blockIdx.y;
  const float* row = hl + ((size_t)b * K + k) * V;
  float mx = -INFINITY;
  if (VEC) {
#pragma unroll 2
    for (int v = 8 * threadIdx.x; v < V; v += 8 * kRowThreads) {
      float x[8];
      load8<float>(row, v, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) mx = fmaxf(mx, x[e]);
    }
  } else {
    for (int v = threadIdx.x; v < V; v += kRowThreads) mx = fmaxf(mx, row[v]);
  }
  const float m = block_max(mx, s);
  FF loc{0.f, 0.f};
  if (VEC) {
#pragma unroll 2
    for (int v = 8 * threadIdx.x; v < V; v += 8 * kRowThreads) {
      float x[8];
      load8<float>(row, v, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = fast_exp2((x[e] - m) * c);
      loc = ff_add8(loc, x);
    }
  } else {
    for (int v = threadIdx.x; v < V; v += kRowThreads) loc = ff_add(loc, fast_exp2((row[v] - m) * c));
  }
  const FF z = block_sum_ff(loc, s);
  if (threadIdx.x == 0) stats[(size_t)b * K + k] = make_float2(m, z.hi + z.lo);
}

// ---------------------------------------------------------------- walks
struct WalkOut {
  int32_t* acc;
  int32_t* path;
  int32_t* out_tokens;
  int32_t* n_out;
  uint32_t* flags;
};

// Greedy walk from the per-row argmax. One thread per sequence.
__global__ void greedy_walk_kernel(TreeShape ts, int B, const int32_t* __restrict__ tokens,
                                   const int32_t* __restrict__ first_child, const int32_t* __restrict__ amax,
                                   WalkOut w) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int N = ts.N, K = ts.K;
  const int32_t* tok = tokens + (size_t)b * N;
  const int32_t* am = amax + (size_t)b * N;
  int32_t* path = w.path + (size_t)b * (K + 1);
  int32_t* out = w.out_tokens + (size_t)b * (K + 1);
  int cur = 0, acc = 0;
  path[0] = 0;
  for (int dep = 1; dep <= K; ++dep) {
    const int a = am[cur];
    const int fc = first_child[cur];
    int nx = -1;
    for (int j = 0; j < ts.s[dep] && fc >= 0 && fc + j < N; ++j)
      if (tok[fc + j] == a) nx = fc + j;
    if (nx < 0) break;
    out[acc] = a;
    cur = nx;
    ++acc;
    path[acc] = cur;
  }
  out[acc] = am[cur];
  for (int r = acc + 1; r <= K; ++r) {
    path[r] = -1;
    out[r] = -1;
  }
  w.acc[b] = acc;
  w.n_out[b] = acc + 1;
}

constexpr int kVThreads = 1024;
constexpr int kVWarps = kVThreads / 32;
// Padded row stride of the inverse-CDF transpose: entry v sits at
// buf[(v % C) * kPad + v / C] so that both the scattered writes and the
// contiguous per-thread reads are free of bank conflicts.
constexpr int kPad = kVThreads + 1;

// State of the walk at one depth: p_0 = softmax(target[cur] / T), q = softmax(head / T),
// and p_j = max(0, p_{j-1} - q) / Z_j after j rejections (p_j = p_{j-1} when Z_j < 1e-30).
struct WalkState {
  float mt, inv_zt, mq, inv_zq;
  int levels;
  float inv_zr[kMaxS + 1];
  int kept[kMaxS + 1];
};

__device__ __forceinline__ float apply_levels(const WalkState& ws, float p, float q) {
  for (int j = 1; j <= ws.levels; ++j)
    if (ws.kept[j]) p = fmaxf(0.f, p - q) * ws.inv_zr[j];
  return p;
}

// One entry with the accurate exponential (acceptance tests).
template <typename T>
__device__ __forceinline__ float p_exact(const WalkState& ws, const T* trow, const float* hrow, float Tmp, int v,
                                         float* qv) {
  const float q = hrow ? expf((hrow[v] - ws.mq) / Tmp) * ws.inv_zq : 0.f;
  *qv = q;
  return apply_levels(ws, expf((Elt<T>::load(trow, v) - ws.mt) / Tmp) * ws.inv_zt, q);
}

// One entry / 8 consecutive entries with the fast exponential (row sweeps); c = log2(e) / T.
template <typename T>
__device__ __forceinline__ float p_fast(const WalkState& ws, const T* trow, const float* hrow, float c, int v,
                                        float* qv) {
  const float q = hrow ? fast_exp2((hrow[v] - ws.mq) * c) * ws.inv_zq : 0.f;
  *qv = q;
  return apply_levels(ws, fast_exp2((Elt<T>::load(trow, v) - ws.mt) * c) * ws.inv_zt, q);
}

template <typename T>
__device__ __forceinline__ void p_fast8(const WalkState& ws, const T* trow, const float* hrow, float c, int v0,
                                        float* p, float* q) {
  float t8[8], h8[8];
  load8<T>(trow, v0, t8);
  if (hrow) load8<float>(hrow, v0, h8);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    q[e] = hrow ? fast_exp2((h8[e] - ws.mq) * c) * ws.inv_zq : 0.f;
    p[e] = apply_levels(ws, fast_exp2((t8[e] - ws.mt) * c) * ws.inv_zt, q[e]);
  }
}

// Row max and softmax normaliser of a target row in one sweep: per-thread
// (max, sum exp) pairs merged across the block by rescaling to the larger max.
template <typename T, int C, bool VEC>
__device__ float2 target_stats(const T* trow, int V, float c, Scratch<kVWarps>& s, float* pm, float* ps) {
  float mx = -INFINITY;
  FF sum{0.f, 0.f};
  if (VEC) {
#pragma unroll 1
    for (int i = 0; i < C / 8; ++i) {
      const int v0 = 8 * (threadIdx.x + i * kVThreads);
      if (v0 >= V) break;
      float x[8];
      load8<T>(trow, v0, x);
      float m8 = x[0];
#pragma unroll
      for (int e = 1; e < 8; ++e) m8 = fmaxf(m8, x[e]);
      if (m8 > mx) {   // rescale the running sum to the new maximum
        const float r = mx == -INFINITY ? 0.f : fast_exp2((mx - m8) * c);
        sum = FF{sum.hi * r, sum.lo * r};
        mx = m8;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = fast_exp2((x[e] - mx) * c);
      sum = ff_add8(sum, x);
    }
  } else {
#pragma unroll 1
    for (int i = 0; i < C; ++i) {
      const int v = threadIdx.x + i * kVThreads;
      if (v >= V) break;
      const float x = Elt<T>::load(trow, v);
      if (x > mx) {
        const float r = mx == -INFINITY ? 0.f : fast_exp2((mx - x) * c);
        sum = FF{sum.hi * r, sum.lo * r};
        mx = x;
      }
      sum = ff_add(sum, fast_exp2((x - mx) * c));
    }
  }
  const float m = block_max(mx, s);
  const float r = mx == -INFINITY ? 0.f : fast_exp2((mx - m) * c);
  const FF z = block_sum_ff(FF{sum.hi * r, sum.lo * r}, s);
  (void)pm;
  (void)ps;
  return make_float2(m, z.hi + z.lo);
}

// Inverse CDF of the current p over the row; sets *near for the 1e-6 tie band.
template <typename T, int C, bool VEC>
__device__ __forceinline__ int walk_inverse_cdf(const WalkState& ws, const T* trow, const float* hrow, float c,
                                                int V, float u, float* buf, Scratch<kVWarps>& s, bool* near) {
  __syncthreads();
  if (VEC) {   // entries v = 8 * (t + i * kVThreads) + e
#pragma unroll 1
    for (int i = 0; i < C / 8; ++i) {
      const int v0 = 8 * (threadIdx.x + i * kVThreads);
      float p[8], q[8];
      if (v0 < V) p_fast8<T>(ws, trow, hrow, c, v0, p, q);
      else
#pragma unroll
        for (int e = 0; e < 8; ++e) p[e] = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) buf[((v0 + e) % C) * kPad + (v0 + e) / C] = p[e];
    }
  } else {
#pragma unroll 1
    for (int i = 0; i < C; ++i) {
      const int v = threadIdx.x + i * kVThreads;
      float q;
      const float p = v < V ? p_fast<T>(ws, trow, hrow, c, v, &q) : 0.f;
      buf[(v % C) * kPad + v / C] = p;
    }
  }
  __syncthreads();
  const int v0 = threadIdx.x * C;   // this thread now holds entries [v0, v0 + C)
  FF loc{0.f, 0.f};
#pragma unroll
  for (int i = 0; i < C; ++i) loc = ff_add(loc, buf[i * kPad + threadIdx.x]);
  FF total;
  FF cum = block_exscan_ff(loc, s, &total);
  const float th = u * total.hi;
  const FF thr = ff_norm(th, fmaf(u, total.hi, -th) + u * total.lo);   // u * total as an exact pair
  const float band = 1e-6f * (total.hi + total.lo);
  int cand = 0x7fffffff;
  float d_at = 0.f, d_prev = 0.f;
#pragma unroll
  for (int i = 0; i < C; ++i) {
    const FF cp = cum;
    cum = ff_add(cum, buf[i * kPad + threadIdx.x]);
    if (cand == 0x7fffffff && v0 + i < V && ff_diff(cum, thr) > 0.f) {
      cand = v0 + i;
      d_at = ff_diff(cum, thr);
      d_prev = ff_diff(thr, cp);
    }
  }
  const int y = block_min_i(cand, s);
  __shared__ int near_flag;
  if (threadIdx.x == 0) near_flag = 0;
  __syncthreads();
  if (cand == y && y != 0x7fffffff) near_flag = (d_at < band || (y > 0 && d_prev < band)) ? 1 : 0;
  __syncthreads();
  *near = near_flag != 0;
  if (y == 0x7fffffff) {   // only reachable if rounding left u*total at or above the last cumulative sum
    *near = true;
    return V - 1;
  }
  return y;
}

// One CTA per sequence.
template <typename T, int C, bool VEC>
__global__ void __launch_bounds__(kVThreads, 1)
rs_walk_kernel(TreeShape ts, int V, float Tmp, const int32_t* __restrict__ tokens,
               const int32_t* __restrict__ first_child, const T* __restrict__ tl, const float* __restrict__ hl,
               const float2* __restrict__ hstats, const float* __restrict__ u_acc, const float* __restrict__ u_res,
               WalkOut w) {
  extern __shared__ float buf[];   // inverse-CDF transpose, [C][kPad]
  __shared__ Scratch<kVWarps> s;
  __shared__ WalkState ws;
  __shared__ int path[kMaxK + 1], out[kMaxK + 1];
  const int b = blockIdx.x, N = ts.N, K = ts.K;
  const float c = 1.4426950408889634f / Tmp;
  const int32_t* tok = tokens + (size_t)b * N;
  uint32_t fl = 0;
  int cur = 0, acc = 0;
  bool done = false;
  if (threadIdx.x == 0) path[0] = 0;
  for (int dep = 1; dep <= K + 1 && !done; ++dep) {
    const T* trow = tl + ((size_t)b * N + cur) * V;
    const float2 tst = target_stats<T, C, VEC>(trow, V, c, s, nullptr, nullptr);
    if (dep == K + 1) {
      // accepted leaf: the bonus is drawn from softmax(target[leaf] / T)
      __syncthreads();
      if (threadIdx.x == 0) {
        ws.mt = tst.x;
        ws.inv_zt = 1.f / tst.y;
        ws.levels = 0;
      }
      __syncthreads();
      bool near = false;
      const int y = walk_inverse_cdf<T, C, VEC>(ws, trow, nullptr, c, V, u_res[(size_t)b * (K + 1) + K], buf, s,
                                                &near);
      if (near) fl |= MEDUSA_FLAG_CDF_NEAR_TIE;
      if (threadIdx.x == 0) out[acc] = y;
      break;
    }
    const float* hrow = hl + ((size_t)b * K + (dep - 1)) * V;
    __syncthreads();
    if (threadIdx.x == 0) {
      const float2 q = hstats[(size_t)b * K + dep - 1];
      ws.mt = tst.x;
      ws.inv_zt = 1.f / tst.y;
      ws.mq = q.x;
      ws.inv_zq = 1.f / q.y;
      ws.levels = 0;
    }
    __syncthreads();
    const int fc = first_child[cur];
    int accepted = -1;
    for (int j = 0; j < ts.s[dep] && fc >= 0 && fc + j < N; ++j) {
      const int child = fc + j;
      const int x = min(max(tok[child], 0), V - 1);
      float qx;
      const float px = p_exact<T>(ws, trow, hrow, Tmp, x, &qx);
      const float r = fminf(1.f, px / qx);
      const float u = u_acc[((size_t)b * K + (dep - 1)) * ts.s_max + j];
      if (fabsf(u - r) < 1e-6f) fl |= MEDUSA_FLAG_RS_NEAR_TIE;
      if (u < r) {
        accepted = child;
        break;
      }
      // residual: Z_{j+1} = sum_v max(0, p_j(v) - q(v)) over the row
      FF loc{0.f, 0.f};
      if (VEC) {
#pragma unroll 1
        for (int i = 0; i < C / 8; ++i) {
          const int v0 = 8 * (threadIdx.x + i * kVThreads);
          if (v0 >= V) break;
          float p[8], q[8];
          p_fast8<T>(ws, trow, hrow, c, v0, p, q);
#pragma unroll
          for (int e = 0; e < 8; ++e) p[e] = fmaxf(0.f, p[e] - q[e]);
          loc = ff_add8(loc, p);
        }
      } else {
#pragma unroll 1
        for (int i = 0; i < C; ++i) {
          const int v = threadIdx.x + i * kVThreads;
          if (v >= V) break;
          float q;
          const float p = p_fast<T>(ws, trow, hrow, c, v, &q);
          loc = ff_add(loc, fmaxf(0.f, p - q));
        }
      }
      const FF tot = block_sum_ff(loc, s);
      const float ft = tot.hi + tot.lo;
      if (threadIdx.x == 0) {
        const int l = ws.levels + 1;
        ws.kept[l] = ft >= 1e-30f;
        ws.inv_zr[l] = ft >= 1e-30f ? 1.f / ft : 1.f;
        ws.levels = l;
      }
      __syncthreads();
    }
    if (accepted < 0) {
      bool near = false;
      const int y = walk_inverse_cdf<T, C, VEC>(ws, trow, hrow, c, V, u_res[(size_t)b * (K + 1) + (dep - 1)], buf, s,
                                                &near);
      if (near) fl |= MEDUSA_FLAG_CDF_NEAR_TIE;
      if (threadIdx.x == 0) out[acc] = y;
      done = true;
      break;
    }
    cur = accepted;
    if (threadIdx.x == 0) {
      out[acc] = tok[cur];
      path[acc + 1] = cur;
    }
    ++acc;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    w.acc[b] = acc;
    w.n_out[b] = acc + 1;
    for (int r = 0; r <= K; ++r) {
      w.path[(size_t)b * (K + 1) + r] = r <= acc ? path[r] : -1;
      w.out_tokens[(size_t)b * (K + 1) + r] = r <= acc ? out[r] : -1;
    }
    w.flags[b] |= fl;
  }
}

template <typename T, int C, bool VEC>
cudaError_t launch_rs_walk_v(const medusa_cfg& c, const TreeShape& ts, const int32_t* tokens,
                             const int32_t* first_child, const void* tl, const float* hl, const float2* stats,
                             const float* ua, const float* ur, const WalkOut& w, cudaStream_t st) {
  const size_t smem = (size_t)C * kPad * sizeof(float);
  cudaError_t e =
      cudaFuncSetAttribute(rs_walk_kernel<T, C, VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  rs_walk_kernel<T, C, VEC><<<c.B, kVThreads, smem, st>>>(ts, c.V, c.temperature, tokens, first_child,
                                                          static_cast<const T*>(tl), hl, stats, ua, ur, w);
  note_launches(1);
  return cudaGetLastError();
}

// Vector loads need V % 8 == 0 (aligned rows) and at least 8 entries per thread.
template <typename T, int C>
cudaError_t launch_rs_walk(const medusa_cfg& c, const TreeShape& ts, const int32_t* tokens, const int32_t* first_child,
                           const void* tl, const float* hl, const float2* stats, const float* ua, const float* ur,
                           const WalkOut& w, cudaStream_t st) {
  if (C >= 8 && c.V % 8 == 0)
    return launch_rs_walk_v<T, C, (C >= 8)>(c, ts, tokens, first_child, tl, hl, stats, ua, ur, w, st);
  return launch_rs_walk_v<T, C, false>(c, ts, tokens, first_child, tl, hl, stats, ua, ur, w, st);
}

template <typename T>
cudaError_t run_rs(const medusa_cfg& c, const TreeShape& ts, const int32_t* tokens, const int32_t* first_child,
                   const void* tl, const float* hl, const float* ua, const float* ur, const WalkOut& w, float2* stats,
                   cudaStream_t st) {
  const float cs = 1.4426950408889634f / c.temperature;
  if (c.V % 8 == 0)
    head_stats_kernel<true><<<dim3(ts.K, c.B), kRowThreads, 0, st>>>(hl, ts.K, c.V, cs, stats);
  else
    head_stats_kernel<false><<<dim3(ts.K, c.B), kRowThreads, 0, st>>>(hl, ts.K, c.V, cs, stats);
  note_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int need = (c.V + kVThreads - 1) / kVThreads;
  if (need <= 1) return launch_rs_walk<T, 1>(c, ts, tokens, first_child, tl, hl, stats, ua, ur, w, st);
  if (need <= 2) return launch_rs_walk<T, 2>(c, ts, tokens, first_child, tl, hl, stats, ua, ur, w, st);
  if (need <= 4) return launch_rs_walk<T, 4>(c, ts, tokens, first_child, tl, hl, stats, ua, ur, w, st);
  if (need <= 8) return launch_rs_walk<T, 8>(c, ts, tokens, first_child, tl, hl, stats, ua, ur, w, st);
  if (need <= 16) return launch_rs_walk<T, 16>(c, ts, tokens, first_child, tl, hl, stats, ua, ur, w, st);
  return launch_rs_walk<T, 32>(c, ts, tokens, first_child, tl, hl, stats, ua, ur, w, st);
}

template <typename T>
cudaError_t run_greedy(const medusa_cfg& c, const TreeShape& ts, const int32_t* tokens, const int32_t* first_child,
                       const void* tl, const WalkOut& w, int32_t* amax, cudaStream_t st) {
  if (c.V % 8 == 0)
    row_argmax_kernel<T, true><<<dim3(ts.N, c.B), kRowThreads, 0, st>>>(static_cast<const T*>(tl), ts.N, c.V, amax);
  else
    row_argmax_kernel<T, false><<<dim3(ts.N, c.B), kRowThreads, 0, st>>>(static_cast<const T*>(tl), ts.N, c.V, amax);
  note_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  greedy_walk_kernel<<<(c.B + 127) / 128, 128, 0, st>>>(ts, c.B, tokens, first_child, amax, w);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

size_t verify_workspace(const medusa_cfg& c) {
  const TreeShape ts = tree_shape(c);
  const size_t greedy = (size_t)c.B * ts.N * sizeof(int32_t);
  const size_t rs = (size_t)c.B * ts.K * sizeof(float2);
  return align_up(greedy > rs ? greedy : rs, 256);
}

cudaError_t launch_verify(const medusa_cfg& c, const int32_t* tokens, const int32_t* parent, const int32_t* first_child,
                          const void* tl, const float* hl, const float* u_acc, const float* u_res, int32_t* acc,
                          int32_t* path, int32_t* out_tokens, int32_t* n_out, uint32_t* flags, void* ws,
                          cudaStream_t st) {
  (void)parent;
  const TreeShape ts = tree_shape(c);
  WalkOut w{acc, path, out_tokens, n_out, flags};
  if (c.mode == MEDUSA_GREEDY) {
    int32_t* amax = static_cast<int32_t*>(ws);
    return c.dtype == MEDUSA_F32 ? run_greedy<float>(c, ts, tokens, first_child, tl, w, amax, st)
                                 : run_greedy<uint16_t>(c, ts, tokens, first_child, tl, w, amax, st);
  }
  float2* stats = static_cast<float2*>(ws);
  return c.dtype == MEDUSA_F32 ? run_rs<float>(c, ts, tokens, first_child, tl, hl, u_acc, u_res, w, stats, st)
                               : run_rs<uint16_t>(c, ts, tokens, first_child, tl, hl, u_acc, u_res, w, stats, st);
}

}  // namespace medusa
