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
// One CTA per sequence walks at most K+1 rows serially. Each thread owns a
// contiguous slice of the vocabulary (C entries) so prefix sums for the
// inverse CDF keep index order; the current distribution p lives in registers
// and q is recomputed from the head logits when needed. Cumulative sums use
// float64.
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
  double dd[kVWarps];
  float bf;
  int bi;
  double bd;
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

__device__ double block_sum_d(double v, BlockScratch& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s.dd[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    double w = threadIdx.x < kVWarps ? s.dd[threadIdx.x] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
    if (threadIdx.x == 0) s.bd = w;
  }
  __syncthreads();
  return s.bd;
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

// Exclusive prefix sum of one double per thread, in thread order.
__device__ double block_exclusive_scan_d(double v, BlockScratch& s, double* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    double t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();
  if (lane == 31) s.dd[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    double w = lane < kVWarps ? s.dd[lane] : 0.0;
    double wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      double t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < kVWarps) s.dd[lane] = wi - w;   // exclusive warp offsets
    if (lane == 31) s.bd = wi;
  }
  __syncthreads();
  *total = s.bd;
  return s.dd[warp] + incl - v;
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

// softmax(row / T) of a T-typed or float row into this thread's C registers (normalised).
template <typename R, int C>
__device__ void softmax_slice(const R* row, int V, float T, float* p, BlockScratch& s) {
  const int v0 = threadIdx.x * C;
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < C; ++i) {
    p[i] = (v0 + i < V) ? Elt<R>::load(row, v0 + i) : -INFINITY;
    mx = fmaxf(mx, p[i]);
  }
  const float m = block_max(mx, s);
  double loc = 0.0;
#pragma unroll
  for (int i = 0; i < C; ++i) {
    p[i] = (v0 + i < V) ? expf((p[i] - m) / T) : 0.f;
    loc += p[i];
  }
  const float z = (float)block_sum_d(loc, s);
#pragma unroll
  for (int i = 0; i < C; ++i) p[i] = p[i] / z;
}

// q(v) for head row hz: exp((hz[v] - mq) / T) / zq
struct QRow {
  const float* hz;
  float mq, zq, T;
  __device__ float at(int v) const { return expf((hz[v] - mq) / T) / zq; }
};

template <int C>
__device__ QRow q_stats(const float* hz, int V, float T, BlockScratch& s) {
  const int v0 = threadIdx.x * C;
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < C; ++i)
    if (v0 + i < V) mx = fmaxf(mx, hz[v0 + i]);
  QRow q;
  q.hz = hz;
  q.T = T;
  q.mq = block_max(mx, s);
  double loc = 0.0;
#pragma unroll
  for (int i = 0; i < C; ++i)
    if (v0 + i < V) loc += expf((hz[v0 + i] - q.mq) / T);
  q.zq = (float)block_sum_d(loc, s);
  return q;
}

// Inverse CDF over this thread's p slice; returns y and sets *near.
template <int C>
__device__ int inverse_cdf(const float* p, int V, float u, BlockScratch& s, bool* near) {
  const int v0 = threadIdx.x * C;
  double loc = 0.0;
#pragma unroll
  for (int i = 0; i < C; ++i) loc += (double)p[i];
  double total;
  const double excl = block_exclusive_scan_d(loc, s, &total);
  const double thr = (double)u * total;
  int cand = 0x7fffffff;
  double c_at = 0.0, c_prev = 0.0;
  double c = excl;
#pragma unroll
  for (int i = 0; i < C; ++i) {
    double cp = c;
    c += (double)p[i];
    if (cand == 0x7fffffff && v0 + i < V && c > thr) {
      cand = v0 + i;
      c_at = c;
      c_prev = cp;
    }
  }
  const int y = block_min_i(cand, s);
  __shared__ int near_flag;
  if (threadIdx.x == 0) near_flag = 0;
  __syncthreads();
  if (cand == y && y != 0x7fffffff) {
    bool nr = fabs(thr - c_at) < 1e-6 * total || (y > 0 && fabs(thr - c_prev) < 1e-6 * total);
    near_flag = nr ? 1 : 0;
  }
  __syncthreads();
  *near = near_flag != 0;
  if (y == 0x7fffffff) {   // only reachable if rounding left thr above the last cumulative sum
    *near = true;
    return V - 1;
  }
  return y;
}

template <typename T, int C>
__global__ void __launch_bounds__(kVThreads)
verify_rs_kernel(TreeShape ts, int V, float Tmp, const int32_t* __restrict__ tokens,
                 const int32_t* __restrict__ first_child, const T* __restrict__ tl, const float* __restrict__ hl,
                 const float* __restrict__ u_acc, const float* __restrict__ u_res, WalkOut w) {
  __shared__ BlockScratch s;
  __shared__ int path[kMaxK + 1], out[kMaxK + 1];
  __shared__ float px_sh;
  const int b = blockIdx.x, N = ts.N, K = ts.K;
  const int32_t* tok = tokens + (size_t)b * N;
  const int v0 = threadIdx.x * C;
  float p[C];
  uint32_t fl = 0;
  int cur = 0, acc = 0;
  if (threadIdx.x == 0) path[0] = 0;
  softmax_slice<T, C>(tl + (size_t)b * N * V, V, Tmp, p, s);
  bool done = false;
  for (int dep = 1; dep <= K && !done; ++dep) {
    const QRow q = q_stats<C>(hl + ((size_t)b * K + (dep - 1)) * V, V, Tmp, s);
    const int fc = first_child[cur];
    int accepted = -1;
    for (int j = 0; j < ts.s[dep] && fc >= 0 && fc + j < N; ++j) {
      const int child = fc + j;
      const int x = min(max(tok[child], 0), V - 1);
      __syncthreads();
      if (x >= v0 && x < v0 + C) {
#pragma unroll
        for (int i = 0; i < C; ++i)
          if (v0 + i == x) px_sh = p[i];
      }
      __syncthreads();
      const float px = px_sh;
      const float qx = q.at(x);
      const float r = fminf(1.f, px / qx);
      const float u = u_acc[((size_t)b * K + (dep - 1)) * ts.s_max + j];
      if (fabsf(u - r) < 1e-6f) fl |= MEDUSA_FLAG_RS_NEAR_TIE;
      if (u < r) {
        accepted = child;
        break;
      }
      // residual: max(0, p - q) / sum, kept only when the sum is not degenerate
      double loc = 0.0;
#pragma unroll
      for (int i = 0; i < C; ++i)
        if (v0 + i < V) loc += (double)fmaxf(0.f, p[i] - q.at(v0 + i));
      const double tot = block_sum_d(loc, s);
      if (tot >= 1e-30) {
        const float ft = (float)tot;
#pragma unroll
        for (int i = 0; i < C; ++i) p[i] = (v0 + i < V) ? fmaxf(0.f, p[i] - q.at(v0 + i)) / ft : 0.f;
      }
    }
    if (accepted < 0) {
      bool near = false;
      const int y = inverse_cdf<C>(p, V, u_res[(size_t)b * (K + 1) + (dep - 1)], s, &near);
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
    softmax_slice<T, C>(tl + ((size_t)b * N + cur) * V, V, Tmp, p, s);
  }
  if (!done) {
    bool near = false;
    const int y = inverse_cdf<C>(p, V, u_res[(size_t)b * (K + 1) + K], s, &near);
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
  verify_rs_kernel<T, C><<<c.B, kVThreads, 0, st>>>(ts, c.V, c.temperature, tokens, first_child,
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
