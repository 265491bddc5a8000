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
// One CTA per sequence walks at most K+1 rows serially. The current
// distribution p lives in registers (C entries per thread, interleaved so row
// loads coalesce), q sits in shared memory, and the inverse CDF transposes p
// into contiguous slices for an index-ordered prefix sum. Sums and prefix sums
// use compensated float32.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace medusa {
namespace {

constexpr int kVThreads = 1024;
constexpr int kVWarps = kVThreads / 32;

struct BlockScratch {
  float f[kVWarps];
  int i[kVWarps];
  float bf;
  int bi;
};

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__device__ float block_max(float v, BlockScratch& s) {
  v = warp_max(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s.f[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float w = threadIdx.x < kVWarps ? s.f[threadIdx.x] : -INFINITY;
    w = warp_max(w);
    if (threadIdx.x == 0) s.bf = w;
  }
  __syncthreads();
  return s.bf;
}


__device__ int block_min_i(int v, BlockScratch& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s.i[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    int w = threadIdx.x < kVWarps ? s.i[threadIdx.x] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w = min(w, __shfl_xor_sync(0xffffffffu, w, o));
    if (threadIdx.x == 0) s.bi = w;
  }
  __syncthreads();
  return s.bi;
}


// Block argmax of a logit row (ties to the lowest index).
template <typename T>
__device__ int block_argmax(const T* row, int V, BlockScratch& s) {
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int v = threadIdx.x; v < V; v += kVThreads) {
    float x = Elt<T>::load(row, v);
    if (better(x, v, bv, bi)) {
      bv = x;
      bi = v;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    s.f[threadIdx.x >> 5] = bv;
    s.i[threadIdx.x >> 5] = bi;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    bv = threadIdx.x < kVWarps ? s.f[threadIdx.x] : -INFINITY;
    bi = threadIdx.x < kVWarps ? s.i[threadIdx.x] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (threadIdx.x == 0) s.bi = bi;
  }
  __syncthreads();
  return s.bi;
}

struct WalkOut {
  int32_t* acc;
  int32_t* path;
  int32_t* out_tokens;
  int32_t* n_out;
  uint32_t* flags;
};

__device__ void write_walk(const WalkOut& w, int b, int K, int acc, const int* path, const int* out, uint32_t fl) {
  if (threadIdx.x != 0) return;
  w.acc[b] = acc;
  w.n_out[b] = acc + 1;
  for (int r = 0; r <= K; ++r) {
    w.path[(size_t)b * (K + 1) + r] = r <= acc ? path[r] : -1;
    w.out_tokens[(size_t)b * (K + 1) + r] = r <= acc ? out[r] : -1;
  }
  w.flags[b] |= fl;
}

template <typename T>
__global__ void __launch_bounds__(kVThreads)
verify_greedy_kernel(TreeShape ts, int V, const int32_t* __restrict__ tokens, const int32_t* __restrict__ first_child,
                     const T* __restrict__ tl, WalkOut w) {
  __shared__ BlockScratch s;
  __shared__ int path[kMaxK + 1], out[kMaxK + 1];
  __shared__ int next;
  const int b = blockIdx.x, N = ts.N, K = ts.K;
  const int32_t* tok = tokens + (size_t)b * N;
  int cur = 0, acc = 0;
  if (threadIdx.x == 0) path[0] = 0;
  for (int dep = 1; dep <= K + 1; ++dep) {
    const int a = block_argmax(tl + ((size_t)b * N + cur) * V, V, s);
    if (dep == K + 1) {
      if (threadIdx.x == 0) out[acc] = a;
      break;
    }
    if (threadIdx.x == 0) {
      int nx = -1;
      const int fc = first_child[cur];
      for (int j = 0; j < ts.s[dep] && fc >= 0 && fc + j < N; ++j)
        if (tok[fc + j] == a) nx = fc + j;
      next = nx;
      if (nx < 0) out[acc] = a;
      else {
        out[acc] = a;
        path[acc + 1] = nx;
      }
    }
    __syncthreads();
    const int nx = next;
    if (nx < 0) break;
    cur = nx;
    ++acc;
  }
  __syncthreads();
  write_walk(w, b, K, acc, path, out, 0u);
}

// ---------------------------------------------------------------- rejection sampling
// Sums use compensated float32 pairs (hi + lo, Knuth's TwoSum): float64 is slow
// on this GPU and plain float32 prefix sums over 32k entries drift by ~1e-6 of
// the total, the size of the inverse-CDF tie band.
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
// a - b as a float (for comparisons and tie bands)
__device__ __forceinline__ float ff_diff(FF a, FF b) { return (a.hi - b.hi) + (a.lo - b.lo); }

struct FFScratch {
  float hi[kVWarps], lo[kVWarps];
  FF tot;
};

__device__ FF block_sum_ff(FF v, FFScratch& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = ff_add(v, ff_shfl_xor(v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    s.hi[threadIdx.x >> 5] = v.hi;
    s.lo[threadIdx.x >> 5] = v.lo;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    FF w = threadIdx.x < kVWarps ? FF{s.hi[threadIdx.x], s.lo[threadIdx.x]} : FF{0.f, 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w = ff_add(w, ff_shfl_xor(w, o));
    if (threadIdx.x == 0) s.tot = w;
  }
  __syncthreads();
  return s.tot;
}

// Exclusive scan (thread order) of one FF per thread; also returns the total.
__device__ FF block_exscan_ff(FF v, FFScratch& s, FF* total) {
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
    FF w = lane < kVWarps ? FF{s.hi[lane], s.lo[lane]} : FF{0.f, 0.f};
    FF wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      FF t = ff_shfl_up(wi, o);
      if (lane >= o) wi = ff_add(wi, t);
    }
    __syncwarp();
    if (lane < kVWarps) {
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

// Thread t owns vocabulary entries v = t + i * kVThreads (i < C): every row load
// is coalesced and q sits in shared memory in natural order (conflict-free).
// Only the inverse CDF needs index-ordered prefix sums: p is then transposed
// through shared memory so that thread t holds [t*C, t*C + C); the one-word pad
// of kPad keeps that transpose free of bank conflicts.
constexpr int kPad = kVThreads + 1;

// p = softmax(row / T), normalised, in this thread's registers.
template <typename R, int C>
__device__ __forceinline__ void softmax_slice(const R* row, int V, float T, float* p, BlockScratch& s, FFScratch& f) {
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < C; ++i) {
    const int v = threadIdx.x + i * kVThreads;
    p[i] = v < V ? Elt<R>::load(row, v) : -INFINITY;
    mx = fmaxf(mx, p[i]);
  }
  const float m = block_max(mx, s);
  FF loc{0.f, 0.f};
#pragma unroll
  for (int i = 0; i < C; ++i) {
    const int v = threadIdx.x + i * kVThreads;
    p[i] = v < V ? expf((p[i] - m) / T) : 0.f;
    loc = ff_add(loc, p[i]);
  }
  const FF z = block_sum_ff(loc, f);
  const float zf = z.hi + z.lo;
#pragma unroll
  for (int i = 0; i < C; ++i) p[i] = p[i] / zf;
}

// q = softmax(head row / T) into qs[v] (shared memory, natural order).
template <int C>
__device__ __forceinline__ void q_to_smem(const float* hz, int V, float T, float* qs, BlockScratch& s, FFScratch& f) {
  float mx = -INFINITY;
#pragma unroll 8
  for (int i = 0; i < C; ++i) {
    const int v = threadIdx.x + i * kVThreads;
    if (v < V) mx = fmaxf(mx, hz[v]);
  }
  const float m = block_max(mx, s);
  FF loc{0.f, 0.f};
#pragma unroll 8
  for (int i = 0; i < C; ++i) {
    const int v = threadIdx.x + i * kVThreads;
    if (v < V) {
      const float e = expf((hz[v] - m) / T);
      qs[v] = e;
      loc = ff_add(loc, e);
    }
  }
  const FF z = block_sum_ff(loc, f);
  const float zf = z.hi + z.lo;
#pragma unroll 8
  for (int i = 0; i < C; ++i) {
    const int v = threadIdx.x + i * kVThreads;
    if (v < V) qs[v] /= zf;
  }
  __syncthreads();
}

// Smallest y with cdf(y) > u * total; *near when u*total lies within 1e-6 * total
// of cdf(y) or cdf(y-1). Clobbers p (it is transposed into contiguous slices).
template <int C>
__device__ __forceinline__ int inverse_cdf(float* p, int V, float u, float* buf, BlockScratch& s, FFScratch& f, bool* near) {
  __syncthreads();
#pragma unroll
  for (int i = 0; i < C; ++i) {
    const int v = threadIdx.x + i * kVThreads;
    buf[(v % C) * kPad + v / C] = p[i];
  }
  __syncthreads();
  const int v0 = threadIdx.x * C;   // now this thread holds entries [v0, v0 + C)
  FF loc{0.f, 0.f};
#pragma unroll
  for (int i = 0; i < C; ++i) {
    p[i] = buf[i * kPad + threadIdx.x];
    loc = ff_add(loc, p[i]);
  }
  FF total;
  FF c = block_exscan_ff(loc, f, &total);
  const float th = u * total.hi;
  const FF thr = ff_norm(th, fmaf(u, total.hi, -th) + u * total.lo);   // u * total as an exact pair
  const float band = 1e-6f * (total.hi + total.lo);
  int cand = 0x7fffffff;
  float d_at = 0.f, d_prev = 0.f;
#pragma unroll
  for (int i = 0; i < C; ++i) {
    const FF cp = c;
    c = ff_add(c, p[i]);
    if (cand == 0x7fffffff && v0 + i < V && ff_diff(c, thr) > 0.f) {
      cand = v0 + i;
      d_at = ff_diff(c, thr);
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

template <typename T, int C>
__global__ void __launch_bounds__(kVThreads, 1)
verify_rs_kernel(TreeShape ts, int V, float Tmp, const int32_t* __restrict__ tokens,
                 const int32_t* __restrict__ first_child, const T* __restrict__ tl, const float* __restrict__ hl,
                 const float* __restrict__ u_acc, const float* __restrict__ u_res, WalkOut w) {
  extern __shared__ float buf[];   // q (natural order), or p transposed for the inverse CDF
  __shared__ BlockScratch s;
  __shared__ FFScratch f;
  __shared__ int path[kMaxK + 1], out[kMaxK + 1];
  __shared__ float px_sh;
  const int b = blockIdx.x, N = ts.N, K = ts.K;
  const int32_t* tok = tokens + (size_t)b * N;
  float p[C];
  uint32_t fl = 0;
  int cur = 0, acc = 0;
  if (threadIdx.x == 0) path[0] = 0;
  softmax_slice<T, C>(tl + (size_t)b * N * V, V, Tmp, p, s, f);
  bool done = false;
  for (int dep = 1; dep <= K && !done; ++dep) {
    q_to_smem<C>(hl + ((size_t)b * K + (dep - 1)) * V, V, Tmp, buf, s, f);
    const int fc = first_child[cur];
    int accepted = -1;
    for (int j = 0; j < ts.s[dep] && fc >= 0 && fc + j < N; ++j) {
      const int child = fc + j;
      const int x = min(max(tok[child], 0), V - 1);
      if ((x % kVThreads) == (int)threadIdx.x) {
#pragma unroll
        for (int i = 0; i < C; ++i)
          if (i == x / kVThreads) px_sh = p[i];
      }
      __syncthreads();
      const float px = px_sh;
      const float qx = buf[x];
      const float r = fminf(1.f, px / qx);
      const float u = u_acc[((size_t)b * K + (dep - 1)) * ts.s_max + j];
      if (fabsf(u - r) < 1e-6f) fl |= MEDUSA_FLAG_RS_NEAR_TIE;
      __syncthreads();
      if (u < r) {
        accepted = child;
        break;
      }
      // residual max(0, p - q) / sum, kept only when the sum is not degenerate
      FF loc{0.f, 0.f};
#pragma unroll
      for (int i = 0; i < C; ++i) {
        const int v = threadIdx.x + i * kVThreads;
        if (v < V) loc = ff_add(loc, fmaxf(0.f, p[i] - buf[v]));
      }
      const FF tot = block_sum_ff(loc, f);
      const float ft = tot.hi + tot.lo;
      if (ft >= 1e-30f) {
#pragma unroll
        for (int i = 0; i < C; ++i) {
          const int v = threadIdx.x + i * kVThreads;
          p[i] = v < V ? fmaxf(0.f, p[i] - buf[v]) / ft : 0.f;
        }
      }
    }
    if (accepted < 0) {
      bool near = false;
      const int y = inverse_cdf<C>(p, V, u_res[(size_t)b * (K + 1) + (dep - 1)], buf, s, f, &near);
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
    softmax_slice<T, C>(tl + ((size_t)b * N + cur) * V, V, Tmp, p, s, f);
  }
  if (!done) {
    bool near = false;
    const int y = inverse_cdf<C>(p, V, u_res[(size_t)b * (K + 1) + K], buf, s, f, &near);
    if (near) fl |= MEDUSA_FLAG_CDF_NEAR_TIE;
    if (threadIdx.x == 0) out[acc] = y;
  }
  __syncthreads();
  write_walk(w, b, K, acc, path, out, fl);
}

template <typename T, int C>
cudaError_t launch_rs(const medusa_cfg& c, const TreeShape& ts, const int32_t* tokens, const int32_t* first_child,
                      const void* tl, const float* hl, const float* ua, const float* ur, const WalkOut& w,
                      cudaStream_t st) {
  const size_t smem = (size_t)C * kPad * sizeof(float);   // >= V floats for q as well
  cudaError_t e = cudaFuncSetAttribute(verify_rs_kernel<T, C>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  verify_rs_kernel<T, C><<<c.B, kVThreads, smem, st>>>(ts, c.V, c.temperature, tokens, first_child,
                                                       static_cast<const T*>(tl), hl, ua, ur, w);
  note_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_rs(const medusa_cfg& c, const TreeShape& ts, const int32_t* tokens, const int32_t* first_child,
                        const void* tl, const float* hl, const float* ua, const float* ur, const WalkOut& w,
                        cudaStream_t st) {
  const int need = (c.V + kVThreads - 1) / kVThreads;
  if (need <= 1) return launch_rs<T, 1>(c, ts, tokens, first_child, tl, hl, ua, ur, w, st);
  if (need <= 2) return launch_rs<T, 2>(c, ts, tokens, first_child, tl, hl, ua, ur, w, st);
  if (need <= 4) return launch_rs<T, 4>(c, ts, tokens, first_child, tl, hl, ua, ur, w, st);
  if (need <= 8) return launch_rs<T, 8>(c, ts, tokens, first_child, tl, hl, ua, ur, w, st);
  if (need <= 16) return launch_rs<T, 16>(c, ts, tokens, first_child, tl, hl, ua, ur, w, st);
  return launch_rs<T, 32>(c, ts, tokens, first_child, tl, hl, ua, ur, w, st);
}

}  // namespace

cudaError_t launch_verify(const medusa_cfg& c, const int32_t* tokens, const int32_t* parent, const int32_t* first_child,
                          const void* tl, const float* hl, const float* u_acc, const float* u_res, int32_t* acc,
                          int32_t* path, int32_t* out_tokens, int32_t* n_out, uint32_t* flags, cudaStream_t st) {
  (void)parent;
  const TreeShape ts = tree_shape(c);
  WalkOut w{acc, path, out_tokens, n_out, flags};
  if (c.mode == MEDUSA_GREEDY) {
    if (c.dtype == MEDUSA_F32)
      verify_greedy_kernel<float><<<c.B, kVThreads, 0, st>>>(ts, c.V, tokens, first_child,
                                                              static_cast<const float*>(tl), w);
    else
      verify_greedy_kernel<uint16_t><<<c.B, kVThreads, 0, st>>>(ts, c.V, tokens, first_child,
                                                                 static_cast<const uint16_t*>(tl), w);
    note_launches(1);
    return cudaGetLastError();
  }
  if (c.dtype == MEDUSA_F32) return dispatch_rs<float>(c, ts, tokens, first_child, tl, hl, u_acc, u_res, w, st);
  return dispatch_rs<uint16_t>(c, ts, tokens, first_child, tl, hl, u_acc, u_res, w, st);
}

}  // namespace medusa
