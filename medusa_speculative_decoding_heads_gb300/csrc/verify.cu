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
// Greedy: one launch, one CTA per sequence, which argmaxes the target row of
// the current node, moves to the child carrying that token and repeats, so
// only the acc + 1 rows the walk visits are read. Rejection sampling (two
// launches): the max and softmax normaliser of every head's logit row in
// parallel, then one cluster of CTAs per sequence walks, each CTA owning a slice
// of the vocabulary; at each visited node one sweep gives the target row's max
// and normaliser, an acceptance test is O(1), and only a rejection (the
// residual's normaliser) and the final draw (inverse CDF) sweep the row again.
// The slices' partial results meet through distributed shared memory. Bulk sums use the hardware base-2 exponential; the
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
constexpr int kMaxHsSlices = 8;    // CTAs per head row in the rejection-sampling stats pass

// CTAs per row for a pass over `rows` rows of V entries: enough for about two
// CTAs per SM, at most `cap`, each slice a multiple of 8 entries.
int row_slices(long rows, int V, int cap) {
  long p = (2 * 152 + rows - 1) / rows;
  p = p < 1 ? 1 : (p > cap ? cap : p);
  const long by_len = (V + 8 * kRowThreads - 1) / (8 * kRowThreads);   // at least 8 entries per thread
  return (int)(p < by_len ? p : (by_len < 1 ? 1 : by_len));
}
int slice_len(int V, int P) { return ((V + P - 1) / P + 7) / 8 * 8; }

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

// ---------------------------------------------------------------- walks
struct WalkOut {
  int32_t* acc;
  int32_t* path;
  int32_t* out_tokens;
  int32_t* n_out;
  uint32_t* flags;
};

// Greedy walk, one CTA per sequence. At each visited node all threads take the
// argmax of its target row (largest value, lowest token id among equal values:
// 16-byte loads, eight in flight per thread, then warp and block reductions);
// thread 0 looks for the child carrying that token among the node's children
// (held in shared memory with the sequence's tokens) and the CTA descends or
// stops. Rows the walk does not reach are never read.
// The links a walk follows: the root has no parent, every other node's parent
// comes before it, and a first child (if any) comes after its node. The walks
// only follow links that stay inside the tree, whatever these arrays hold.
__device__ __forceinline__ bool tree_links_ok(int i, int N, int par, int fc) {
  return (i == 0 ? par == -1 : (par >= 0 && par < i)) && (fc == -1 || (fc > i && fc < N));
}

constexpr int kGwThreads = 512;
constexpr int kGwWarps = kGwThreads / 32;

template <typename T, bool VEC>
__global__ void __launch_bounds__(kGwThreads)
greedy_walk_kernel(TreeShape ts, int V, const int32_t* __restrict__ tokens, const int32_t* __restrict__ parent,
                   const int32_t* __restrict__ first_child, const T* __restrict__ tl, WalkOut w) {
  __shared__ int s_tok[kMaxN], s_par[kMaxN], s_fc[kMaxN];
  __shared__ float sv[kGwWarps];
  __shared__ int si[kGwWarps];
  __shared__ int s_next;
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, N = ts.N, K = ts.K;
  for (int i = threadIdx.x; i < N; i += kGwThreads) {
    s_tok[i] = tokens[(size_t)b * N + i];
    s_par[i] = parent[i];
    s_fc[i] = first_child[i];
    MEDUSA_CHECK(tree_links_ok(i, N, s_par[i], s_fc[i]), MEDUSA_CHECK_TREE);
  }
  int32_t* path = w.path + (size_t)b * (K + 1);
  int32_t* out = w.out_tokens + (size_t)b * (K + 1);
  int cur = 0, acc = 0;
  if (threadIdx.x == 0) path[0] = 0;
  while (true) {
    const T* row = tl + ((size_t)b * N + cur) * V;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    if (VEC) {
      constexpr int kU = 8;   // 16-byte vectors per thread per round
      for (int base = 0; base < V; base += kU * 8 * kGwThreads) {
        float x[kU][8];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int v = base + 8 * (threadIdx.x + u * kGwThreads);
          if (v < V) load8<T>(row, v, x[u]);
          else
#pragma unroll
            for (int e = 0; e < 8; ++e) x[u][e] = -INFINITY;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int v = base + 8 * (threadIdx.x + u * kGwThreads) + e;
            if (v < V && better(x[u][e], v, bv, bi)) {
              bv = x[u][e];
              bi = v;
            }
          }
      }
    } else {
#pragma unroll 4
      for (int v = threadIdx.x; v < V; v += kGwThreads) {
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
    if ((threadIdx.x & 31) == 0) {
      sv[threadIdx.x >> 5] = bv;
      si[threadIdx.x >> 5] = bi;
    }
    __syncthreads();   // also publishes the tree arrays on the first pass
    if (threadIdx.x < 32) {
      bv = threadIdx.x < kGwWarps ? sv[threadIdx.x] : -INFINITY;
      bi = threadIdx.x < kGwWarps ? si[threadIdx.x] : 0x7fffffff;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (threadIdx.x == 0) {
        // bi is the target's token after `cur`: the next draft if a child carries it, else the bonus
        int nx = -1;
        const int fc = acc < K ? s_fc[cur] : -1;
        for (int j = 0; fc >= 0 && fc + j < N && s_par[fc + j] == cur; ++j)
          if (s_tok[fc + j] == bi) nx = fc + j;
        out[acc] = bi;
        if (nx >= 0) path[acc + 1] = nx;
        s_next = nx;
      }
    }
    __syncthreads();
    const int nx = s_next;
    if (nx < 0) break;
    cur = nx;
    ++acc;
  }
  if (threadIdx.x == 0) {
    for (int r = acc + 1; r <= K; ++r) {
      path[r] = -1;
      out[r] = -1;
    }
    w.acc[b] = acc;
    w.n_out[b] = acc + 1;
  }
}

constexpr int kVThreads = 256;
constexpr int kVWarps = kVThreads / 32;
// Padded row stride of the inverse-CDF transpose: entry v sits at
// buf[(v % C) * kPad + v / C] so that both the scattered writes and the
// contiguous per-thread reads are free of bank conflicts.
constexpr int kPad = kVThreads + 1;
constexpr int kMaxCluster = 8;   // CTAs per sequence (portable cluster size)

// ---------------------------------------------------------------- cluster exchange
// The CTAs of one cluster share one sequence's walk: CTA r owns the vocabulary
// slice [r * S, (r + 1) * S). Block-level partials are traded through
// distributed shared memory: thread r stores this CTA's value into slot[rank]
// of CTA r and arrives (release, cluster scope) on CTA r's mbarrier; every CTA
// waits (acquire, bounded) for all arrivals and reads the slots in rank order,
// so all CTAs combine the same numbers in the same order and take identical
// decisions. Two barriers alternate, so a CTA can run at most one exchange ahead.
struct Xchg {
  uint64_t bar[2];
  float2 f[2][kMaxCluster];
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ void tc_free_mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ uint32_t cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_ctas() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t remote(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// All threads call with the same block-uniform value; returns every CTA's value in vals[rank].
__device__ __forceinline__ void xchg(Xchg& x, int& xn, float2 mine, float2 (&vals)[kMaxCluster], uint32_t ncta,
                                     uint32_t rank, uint32_t* fl) {
  const int par = xn & 1;
  __syncthreads();
  if (threadIdx.x < ncta) {
    const uint32_t slot = remote(&x.f[par][rank], threadIdx.x);
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(slot), "f"(mine.x), "f"(mine.y) : "memory");
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote(&x.bar[par], threadIdx.x))
                 : "memory");
  }
  const uint32_t parity = (xn >> 1) & 1;
  const uint32_t baddr = smem_u32(&x.bar[par]);
  uint32_t ok = 0;
  const long long t0 = clock64();
  while (true) {
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(baddr), "r"(parity)
        : "memory");
    if (ok) break;
    if (clock64() - t0 > 4000000000LL) {   // a peer never arrived: record it and carry on
      *fl |= MEDUSA_FLAG_TIMEOUT;
      break;
    }
  }
#pragma unroll
  for (uint32_t r = 0; r < kMaxCluster; ++r) vals[r] = r < ncta ? x.f[par][r] : make_float2(0.f, 0.f);
  ++xn;
}

// State of the walk at one depth: p_0 = softmax(target[cur] / T), q = softmax(head / T),
// and p_j = max(0, p_{j-1} - q) / Z_j after j rejections (p_j = p_{j-1} when Z_j < 1e-30).
struct WalkState {
  float mt, inv_zt, mq, inv_zq;
  int levels;
  float inv_zr[kMaxS + 1];
  int kept[kMaxS + 1];
};

// Unrolled over every possible level so that a register copy of the state is
// indexed statically (a runtime-bounded loop would put it in local memory).
__device__ __forceinline__ float apply_levels(const WalkState& ws, float p, float q) {
#pragma unroll
  for (int j = 1; j <= kMaxS; ++j)
    if (j <= ws.levels && ws.kept[j]) p = fmaxf(0.f, p - q) * ws.inv_zr[j];
  return p;
}

// Entry v of this CTA's slice for thread t, step i: VEC takes 8 consecutive
// entries per step (v0 = lo + 8 (t + i * kVThreads)), otherwise one (lo + t + i * kVThreads).

// (max, sum of 2^((v - max) c)) pairs merged by rescaling to the larger max.
struct MS {
  float m;
  FF s;
};
__device__ __forceinline__ MS ms_merge(MS a, MS b, float c) {
  const float M = fmaxf(a.m, b.m);
  if (M == -INFINITY) return a;
  const float ra = a.m == -INFINITY ? 0.f : fast_exp2((a.m - M) * c);
  const float rb = b.m == -INFINITY ? 0.f : fast_exp2((b.m - M) * c);
  return MS{M, ff_add(FF{a.s.hi * ra, a.s.lo * ra}, FF{b.s.hi * rb, b.s.lo * rb})};
}
// One block-wide merge (a single round of shared memory) of every thread's pair.
template <int NW>
__device__ MS block_ms(MS v, float c, Scratch<NW>& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const MS w{__shfl_xor_sync(0xffffffffu, v.m, o), ff_shfl_xor(v.s, o)};
    v = ms_merge(v, w, c);
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    s.f[threadIdx.x >> 5] = v.m;
    s.hi[threadIdx.x >> 5] = v.s.hi;
    s.lo[threadIdx.x >> 5] = v.s.lo;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    MS w = threadIdx.x < NW ? MS{s.f[threadIdx.x], FF{s.hi[threadIdx.x], s.lo[threadIdx.x]}}
                            : MS{-INFINITY, FF{0.f, 0.f}};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const MS u{__shfl_xor_sync(0xffffffffu, w.m, o), ff_shfl_xor(w.s, o)};
      w = ms_merge(w, u, c);
    }
    if (threadIdx.x == 0) {
      s.bf = w.m;
      s.tot = w.s;
    }
  }
  __syncthreads();
  return MS{s.bf, s.tot};
}

// Rejection sampling, head rows: (m, Z) of slice p of head row (b, k), with
// m = max and Z = sum exp((v - m) / T) over the slice; part[(b * K + k) * P + p],
// grid (P, K, B). Each thread reads 16 entries per round (all loads in flight)
// and folds them into its running pair; the walk merges the P slices of a row
// by rescaling to the larger max. VEC: slices start at multiples of 8 (V % 8 == 0).
template <bool VEC>
__global__ void __launch_bounds__(kRowThreads)
head_stats_kernel(const float* __restrict__ hl, int K, int V, int chunk, float c, float2* __restrict__ part) {
  pdl_wait();
  pdl_trigger();
  __shared__ Scratch<kRowWarps> s;
  const int p = blockIdx.x, k = blockIdx.y, b = blockIdx.z, P = gridDim.x;
  const float* row = hl + ((size_t)b * K + k) * V;
  const int v0 = min(V, p * chunk), v1 = min(V, v0 + chunk);
  constexpr int kPer = 16;
  MS run{-INFINITY, FF{0.f, 0.f}};
  for (int base = v0; base < v1; base += kPer * kRowThreads) {
    float x[kPer];
    if (VEC) {
#pragma unroll
      for (int i = 0; i < kPer / 8; ++i) {
        const int v = base + 8 * (threadIdx.x + i * kRowThreads);
        if (v < v1) load8<float>(row, v, x + 8 * i);
        else
#pragma unroll
          for (int e = 0; e < 8; ++e) x[8 * i + e] = -INFINITY;
      }
    } else {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int v = base + threadIdx.x + i * kRowThreads;
        x[i] = v < v1 ? row[v] : -INFINITY;
      }
    }
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPer; ++i) m = fmaxf(m, x[i]);
    if (m == -INFINITY) continue;
    FF sum{0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kPer; i += 8) {
      float e8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) e8[e] = fast_exp2((x[i + e] - m) * c);
      sum = ff_add8(sum, e8);
    }
    run = ms_merge(run, MS{m, sum}, c);
  }
  const MS blk = block_ms(run, c, s);
  if (threadIdx.x == 0) part[((size_t)b * K + k) * P + p] = make_float2(blk.m, blk.s.hi + blk.s.lo);
}

// Merges the P slice pairs of one head row into (m, Z) of the whole row.
// Unused slots hold (-inf, 0).
__device__ __forceinline__ float2 merge_head_stats(const float2 (&hp)[kMaxHsSlices], float c) {
  float M = -INFINITY;
#pragma unroll
  for (int p = 0; p < kMaxHsSlices; ++p) M = fmaxf(M, hp[p].x);
  FF Z{0.f, 0.f};
#pragma unroll
  for (int p = 0; p < kMaxHsSlices; ++p)
    if (hp[p].x != -INFINITY) Z = ff_add(Z, hp[p].y * fast_exp2((hp[p].x - M) * c));
  return make_float2(M, Z.hi + Z.lo);
}

// This thread's C entries of a row slice [lo, hi), as floats, all loads in
// flight at once; entries past hi read as `pad`. VEC: entry 8 i + e is
// v = lo + 8 (t + i kVThreads) + e (V % 8 == 0, so a group of 8 is in or out
// as a whole); otherwise entry i is v = lo + t + i kVThreads.
template <typename T, int C, bool VEC>
__device__ __forceinline__ void load_slice(const T* row, int lo, int hi, float (&x)[C], float pad) {
  if (VEC) {
#pragma unroll
    for (int i = 0; i < C / 8; ++i) {
      const int v0 = lo + 8 * (threadIdx.x + i * kVThreads);
      if (v0 < hi) load8<T>(row, v0, x + 8 * i);
      else
#pragma unroll
        for (int e = 0; e < 8; ++e) x[8 * i + e] = pad;
    }
  } else {
#pragma unroll
    for (int i = 0; i < C; ++i) {
      const int v = lo + threadIdx.x + i * kVThreads;
      x[i] = v < hi ? Elt<T>::load(row, v) : pad;
    }
  }
}

// Row max and softmax normaliser of a target row from this thread's entries
// xv (padded with -inf), merged across the block and then across the cluster
// by rescaling to the larger max.
template <int C>
__device__ float2 target_stats(const float (&xv)[C], float c, Scratch<kVWarps>& s, Xchg& x, int& xn, uint32_t ncta,
                               uint32_t rank, uint32_t* fl) {
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < C; ++i) mx = fmaxf(mx, xv[i]);
  FF sum{0.f, 0.f};
  if (mx != -INFINITY) {
#pragma unroll
    for (int i = 0; i < C; i += 8) {
      float e8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) e8[e] = (i + e < C) ? fast_exp2((xv[i + e] - mx) * c) : 0.f;
      sum = ff_add8(sum, e8);
    }
  }
  const MS blk = block_ms(MS{mx, sum}, c, s);
  float2 vals[kMaxCluster];
  xchg(x, xn, make_float2(blk.m, blk.s.hi + blk.s.lo), vals, ncta, rank, fl);
  float M = -INFINITY;
#pragma unroll
  for (uint32_t k = 0; k < kMaxCluster; ++k)
    if (k < ncta) M = fmaxf(M, vals[k].x);
  FF Z{0.f, 0.f};
#pragma unroll
  for (uint32_t k = 0; k < kMaxCluster; ++k)
    if (k < ncta && vals[k].x != -INFINITY) Z = ff_add(Z, vals[k].y * fast_exp2((vals[k].x - M) * c));
  return make_float2(M, Z.hi + Z.lo);
}

// p_0 = softmax(target / T) and q = softmax(head / T) at this thread's entries
// (c = log2(e) / T; padded entries give 0); without a head row q = 0.
template <int C>
__device__ __forceinline__ void start_levels(const float (&tv)[C], const float (&hv)[C], bool has_h,
                                             const WalkState& ws, float c, float (&pc)[C], float (&qc)[C]) {
#pragma unroll
  for (int i = 0; i < C; ++i) {
    pc[i] = fast_exp2((tv[i] - ws.mt) * c) * ws.inv_zt;
    qc[i] = has_h ? fast_exp2((hv[i] - ws.mq) * c) * ws.inv_zq : 0.f;
  }
}

// p_j -> p_{j+1} = max(0, p_j - q) / Z_{j+1} (skipped when Z_{j+1} < 1e-30), at
// this thread's entries.
template <int C>
__device__ __forceinline__ void next_level(float (&pc)[C], const float (&qc)[C], float ft) {
  if (!(ft >= 1e-30f)) return;
  const float a = 1.f / ft;
#pragma unroll
  for (int i = 0; i < C; ++i) pc[i] = fmaxf(0.f, pc[i] - qc[i]) * a;
}

// Sum over the row of max(0, p_j - q) (the next residual's normaliser), from
// this thread's p_j and q (zero past the slice).
template <int C>
__device__ float residual_sum(const float (&pc)[C], const float (&qc)[C], Scratch<kVWarps>& s, Xchg& x, int& xn,
                              uint32_t ncta, uint32_t rank, uint32_t* fl) {
  FF loc{0.f, 0.f};
#pragma unroll
  for (int i = 0; i < C; i += 8) {
    float d8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) d8[e] = (i + e < C) ? fmaxf(0.f, pc[i + e] - qc[i + e]) : 0.f;
    loc = ff_add8(loc, d8);
  }
  const FF tot = block_sum_ff(loc, s);
  float2 vals[kMaxCluster];
  xchg(x, xn, make_float2(tot.hi, tot.lo), vals, ncta, rank, fl);
  FF all{0.f, 0.f};
#pragma unroll
  for (uint32_t k = 0; k < kMaxCluster; ++k)
    if (k < ncta) all = ff_add(all, FF{vals[k].x, vals[k].y});
  return all.hi + all.lo;
}

// Inverse CDF of the current p over the row (smallest y with cdf(y) > u * total),
// from this thread's p (zero past the slice); sets *near for the 1e-6 tie band.
template <int C, bool VEC>
__device__ int walk_inverse_cdf(const float (&pc)[C], int lo, int hi, int V, float u, float* buf,
                                Scratch<kVWarps>& s, Xchg& x, int& xn, uint32_t ncta, uint32_t rank, uint32_t* fl,
                                bool* near) {
  __syncthreads();
  // this thread's entries, local index l = v - lo, into the transpose
#pragma unroll
  for (int i = 0; i < C; ++i) {
    const int l = VEC ? 8 * (threadIdx.x + (i / 8) * kVThreads) + (i % 8) : threadIdx.x + i * kVThreads;
    buf[(l % C) * kPad + l / C] = pc[i];
  }
  __syncthreads();
  const int l0 = threadIdx.x * C;   // this thread now holds local entries [l0, l0 + C)
  FF loc{0.f, 0.f};
#pragma unroll
  for (int i = 0; i < C; ++i) loc = ff_add(loc, buf[i * kPad + threadIdx.x]);
  FF cta_total;
  FF cum = block_exscan_ff(loc, s, &cta_total);
  // offsets of the slices before this one, and the row total
  float2 vals[kMaxCluster];
  xchg(x, xn, make_float2(cta_total.hi, cta_total.lo), vals, ncta, rank, fl);
  FF total{0.f, 0.f}, before{0.f, 0.f};
#pragma unroll
  for (uint32_t k = 0; k < kMaxCluster; ++k)
    if (k < ncta) {
      if (k == rank) before = total;
      total = ff_add(total, FF{vals[k].x, vals[k].y});
    }
  cum = ff_add(before, cum);
  const float th = u * total.hi;
  const FF thr = ff_norm(th, fmaf(u, total.hi, -th) + u * total.lo);   // u * total as an exact pair
  const float band = 1e-6f * (total.hi + total.lo);
  int cand = 0x7fffffff;
  float d_at = 0.f, d_prev = 0.f;
#pragma unroll
  for (int i = 0; i < C; ++i) {
    const FF cp = cum;
    cum = ff_add(cum, buf[i * kPad + threadIdx.x]);
    if (cand == 0x7fffffff && lo + l0 + i < hi && ff_diff(cum, thr) > 0.f) {
      cand = lo + l0 + i;
      d_at = ff_diff(cum, thr);
      d_prev = ff_diff(thr, cp);
    }
  }
  const int y_cta = block_min_i(cand, s);
  __shared__ int near_flag;
  if (threadIdx.x == 0) near_flag = 0;
  __syncthreads();
  if (cand == y_cta && y_cta != 0x7fffffff) near_flag = (d_at < band || (y_cta > 0 && d_prev < band)) ? 1 : 0;
  __syncthreads();
  // the first slice holding a crossing wins
  xchg(x, xn, make_float2(__int_as_float(y_cta), __int_as_float(near_flag)), vals, ncta, rank, fl);
  int y = 0x7fffffff, nf = 0;
#pragma unroll
  for (uint32_t k = 0; k < kMaxCluster; ++k)
    if (k < ncta) {
      const int yk = __float_as_int(vals[k].x);
      if (yk < y) {
        y = yk;
        nf = __float_as_int(vals[k].y);
      }
    }
  *near = nf != 0;
  if (y == 0x7fffffff) {   // only reachable if rounding left u*total at or above the last cumulative sum
    *near = true;
    return V - 1;
  }
  return y;
}

// One cluster of CTAs per sequence; CTA `rank` owns the vocabulary slice
// [rank * S, rank * S + S) with S = slice (a multiple of 8).
template <typename T, int C, bool VEC>
__global__ void __launch_bounds__(kVThreads, 1)
rs_walk_kernel(TreeShape ts, int V, int slice, float Tmp, const int32_t* __restrict__ tokens,
               const int32_t* __restrict__ parent, const int32_t* __restrict__ first_child,
               const T* __restrict__ tl, const float* __restrict__ hl,
               const float2* __restrict__ hstats, int hsP, const float* __restrict__ u_acc,
               const float* __restrict__ u_res, WalkOut w) {
  pdl_trigger();
  extern __shared__ float buf[];   // inverse-CDF transpose, [C][kPad]
  __shared__ Scratch<kVWarps> s;
  __shared__ WalkState ws;
  __shared__ Xchg x;
  __shared__ int path[kMaxK + 1], out[kMaxK + 1];
  const uint32_t ncta = cluster_ctas(), rank = cta_rank();
  const int b = blockIdx.x / ncta, N = ts.N, K = ts.K;
  const int lo = min(V, (int)rank * slice), hi = min(V, lo + slice);
  const float c = 1.4426950408889634f / Tmp;
  // the exchange barriers and the cluster barrier touch no global memory, so they are set
  // up before the wait on the previous kernel and overlap its tail
  if (threadIdx.x == 0) {
    tc_free_mbar_init(&x.bar[0], ncta);
    tc_free_mbar_init(&x.bar[1], ncta);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    path[0] = 0;
  }
  cluster_sync();   // every CTA's barriers exist before any peer arrives on them
  pdl_wait();
  // this sequence's tree tokens and the tree's first-child table, staged once
  __shared__ int s_tok[kMaxN], s_fc[kMaxN], s_par[kMaxN];
  for (int i = threadIdx.x; i < N; i += kVThreads) {
    s_tok[i] = tokens[(size_t)b * N + i];
    s_fc[i] = first_child[i];
    s_par[i] = parent[i];
    MEDUSA_CHECK(tree_links_ok(i, N, s_par[i], s_fc[i]), MEDUSA_CHECK_TREE);
  }
  uint32_t fl = 0;
  int xn = 0;
  // the candidates of the current depth: token, its target and head logits, and
  // the acceptance uniform, fetched before the row sweep so that their load
  // latency overlaps it
  __shared__ float cand_t[kMaxS], cand_h[kMaxS], cand_u[kMaxS];
  __shared__ int cand_n;
  __shared__ float2 cand_q;
  int cur = 0, acc = 0;
  for (int dep = 1; dep <= K + 1; ++dep) {
    const T* trow = tl + ((size_t)b * N + cur) * V;
    __syncthreads();   // the previous depth's candidates have been read (and the staging is done)
    // candidate j's logits and uniform: loads issued now, stored after the row sweep
    const bool fetch = dep <= K && threadIdx.x < ts.s[dep];
    float ct = 0.f, ch = 0.f, cu = 0.f;
    float2 hq[kMaxHsSlices];   // the slices of this depth's head-row (m, Z), merged after the sweep
    if (fetch) {
      const int fc = s_fc[cur];
      const int j = threadIdx.x;
      const bool child = fc >= 0 && fc + j < N && s_par[fc + j] == cur;
      MEDUSA_CHECK(!child || (s_tok[fc + j] >= 0 && s_tok[fc + j] < V), MEDUSA_CHECK_TOKEN);
      const int xt = child ? min(max(s_tok[fc + j], 0), V - 1) : 0;
      ct = Elt<T>::load(trow, xt);
      ch = hl[((size_t)b * K + (dep - 1)) * V + xt];
      cu = u_acc[((size_t)b * K + (dep - 1)) * ts.s_max + j];
      if (j == 0)
#pragma unroll
        for (int p = 0; p < kMaxHsSlices; ++p)
          hq[p] = p < hsP ? hstats[((size_t)b * K + dep - 1) * hsP + p] : make_float2(-INFINITY, 0.f);
    }
    if (dep <= K) {
      // warm L2 with this CTA's slice of every child's target row (the next depth reads one of them)
      const int fc = s_fc[cur];
      const int lines = ((hi - lo) * (int)sizeof(T) + 127) / 128;   // every prefetched line starts inside the slice
      for (int t = threadIdx.x; t < ts.s[dep] * lines; t += kVThreads) {
        const int j = t / lines, l = t % lines;
        if (fc >= 0 && fc + j < N && s_par[fc + j] == cur) {
          const char* pr = reinterpret_cast<const char*>(tl + ((size_t)b * N + fc + j) * V + lo) + 128 * l;
          asm volatile("prefetch.global.L2 [%0];" ::"l"(pr));
        }
      }
    }
    // this thread's entries of the node's target row and of the depth's head row
    float tv[C], hv[C];
    load_slice<T, C, VEC>(trow, lo, hi, tv, -INFINITY);
    if (dep <= K) load_slice<float, C, VEC>(hl + ((size_t)b * K + (dep - 1)) * V, lo, hi, hv, -INFINITY);
    else
#pragma unroll
      for (int i = 0; i < C; ++i) hv[i] = -INFINITY;
    const float2 tst = target_stats<C>(tv, c, s, x, xn, ncta, rank, &fl);
    float pc[C], qc[C];   // p_j and q at this thread's entries
    if (fetch) {
      const int fc = s_fc[cur];
      const int j = threadIdx.x;
      cand_t[j] = ct;
      cand_h[j] = ch;
      cand_u[j] = cu;
      if (j == 0) {
        int nc = 0;
        while (nc < ts.s[dep] && fc >= 0 && fc + nc < N && s_par[fc + nc] == cur) ++nc;   // cur's children
        cand_n = nc;
        cand_q = merge_head_stats(hq, c);
      }
    }
    if (dep == K + 1) {
      // accepted leaf: the bonus is drawn from softmax(target[leaf] / T)
      __syncthreads();
      if (threadIdx.x == 0) {
        ws.mt = tst.x;
        ws.inv_zt = 1.f / tst.y;
        ws.levels = 0;
      }
      __syncthreads();
      start_levels<C>(tv, hv, false, ws, c, pc, qc);
      bool near = false;
      const int y = walk_inverse_cdf<C, VEC>(pc, lo, hi, V, u_res[(size_t)b * (K + 1) + K], buf, s, x, xn, ncta, rank,
                                             &fl, &near);
      if (near) fl |= MEDUSA_FLAG_CDF_NEAR_TIE;
      if (threadIdx.x == 0) out[acc] = y;
      break;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      const float2 q = cand_q;
      ws.mt = tst.x;
      ws.inv_zt = 1.f / tst.y;
      ws.mq = q.x;
      ws.inv_zq = 1.f / q.y;
      ws.levels = 0;
    }
    __syncthreads();
    start_levels<C>(tv, hv, true, ws, c, pc, qc);
    const int fc = s_fc[cur];
    const int nc = cand_n;
    int accepted = -1;
    for (int j = 0; j < nc; ++j) {
      const int child = fc + j;
      const float qx = expf((cand_h[j] - ws.mq) / Tmp) * ws.inv_zq;
      const float px = apply_levels(ws, expf((cand_t[j] - ws.mt) / Tmp) * ws.inv_zt, qx);
      const float r = fminf(1.f, px / qx);
      const float u = cand_u[j];
      if (fabsf(u - r) < 1e-6f) fl |= MEDUSA_FLAG_RS_NEAR_TIE;
      if (u < r) {
        accepted = child;
        break;
      }
      // residual: Z_{j+1} = sum_v max(0, p_j(v) - q(v)) over the row
      const float ft = residual_sum<C>(pc, qc, s, x, xn, ncta, rank, &fl);
      next_level<C>(pc, qc, ft);
      __syncthreads();
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
      const int y = walk_inverse_cdf<C, VEC>(pc, lo, hi, V, u_res[(size_t)b * (K + 1) + (dep - 1)], buf, s, x, xn,
                                             ncta, rank, &fl, &near);
      if (near) fl |= MEDUSA_FLAG_CDF_NEAR_TIE;
      if (threadIdx.x == 0) out[acc] = y;
      break;
    }
    cur = accepted;
    if (threadIdx.x == 0) {
      out[acc] = s_tok[cur];
      path[acc + 1] = cur;
    }
    ++acc;
  }
  __syncthreads();
  if (rank == 0 && threadIdx.x == 0) {
    w.acc[b] = acc;
    w.n_out[b] = acc + 1;
    for (int r = 0; r <= K; ++r) {
      w.path[(size_t)b * (K + 1) + r] = r <= acc ? path[r] : -1;
      w.out_tokens[(size_t)b * (K + 1) + r] = r <= acc ? out[r] : -1;
    }
  }
  // flags from every CTA (near ties are seen by the slice that owns them)
  __shared__ uint32_t fl_all;
  if (threadIdx.x == 0) fl_all = 0;
  __syncthreads();
  if (fl) atomicOr(&fl_all, fl);
  __syncthreads();
  if (threadIdx.x == 0 && fl_all) atomicOr(&w.flags[b], fl_all);
  cluster_sync();   // no CTA leaves while a peer may still write into its shared memory
}

template <typename T, int C, bool VEC>
cudaError_t launch_rs_walk_v(const medusa_cfg& c, const TreeShape& ts, int ncta, int slice, const int32_t* tokens,
                             const int32_t* parent, const int32_t* first_child, const void* tl, const float* hl, const float2* stats, int hsP,
                             const float* ua, const float* ur, const WalkOut& w, cudaStream_t st) {
  const size_t smem = (size_t)C * kPad * sizeof(float);
  auto kern = rs_walk_kernel<T, C, VEC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c.B * ncta);
  cfg.blockDim = dim3(kVThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ncta;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // as launch_pdl
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, ts, c.V, slice, c.temperature, tokens, parent, first_child,
                         static_cast<const T*>(tl), hl, stats, hsP, ua, ur, w);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Vector loads need V % 8 == 0 (aligned rows and slices) and at least 8 entries per thread.
template <typename T, int C>
cudaError_t launch_rs_walk(const medusa_cfg& c, const TreeShape& ts, int ncta, int slice, const int32_t* tokens,
                           const int32_t* parent, const int32_t* first_child, const void* tl, const float* hl, const float2* stats, int hsP,
                           const float* ua, const float* ur, const WalkOut& w, cudaStream_t st) {
  if (C >= 8 && c.V % 8 == 0)
    return launch_rs_walk_v<T, C, (C >= 8)>(c, ts, ncta, slice, tokens, parent, first_child, tl, hl, stats, hsP, ua, ur, w, st);
  return launch_rs_walk_v<T, C, false>(c, ts, ncta, slice, tokens, parent, first_child, tl, hl, stats, hsP, ua, ur, w, st);
}

// CTAs per sequence: the largest power of two (at most 8) that keeps the whole
// grid within one CTA per SM (eight per sequence at B = 32 measured no faster
// than four: the walk's time is its chain of cluster exchanges, not the slices),
// and at least enough that a CTA's slice fits the 32 entries per thread the walk
// holds in registers (V <= 32768 needs at most 4; more CTAs than one wave is only
// slower).
int rs_cluster_ctas(int B, int V) {
  int n = 1;
  while (n < kMaxCluster && (long)B * n <= 152) n *= 2;
  while (n < kMaxCluster && (long)n * 32 * kVThreads < V) n *= 2;
  return n;
}

template <typename T>
cudaError_t run_rs(const medusa_cfg& c, const TreeShape& ts, const int32_t* tokens, const int32_t* parent,
                   const int32_t* first_child,
                   const void* tl, const float* hl, const float* ua, const float* ur, const WalkOut& w, float2* stats,
                   cudaStream_t st) {
  const float cs = 1.4426950408889634f / c.temperature;
  const int hsP = row_slices((long)c.B * ts.K, c.V, kMaxHsSlices);
  const int hs_chunk = slice_len(c.V, hsP);
  if (c.V % 8 == 0)
    launch_pdl(head_stats_kernel<true>, dim3(hsP, ts.K, c.B), kRowThreads, 0, st, hl, ts.K, c.V, hs_chunk, cs, stats);
  else
    launch_pdl(head_stats_kernel<false>, dim3(hsP, ts.K, c.B), kRowThreads, 0, st, hl, ts.K, c.V, hs_chunk, cs, stats);
  note_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int ncta = rs_cluster_ctas(c.B, c.V);
  const int slice = (((c.V + ncta - 1) / ncta) + 7) / 8 * 8;
  const int need = (slice + kVThreads - 1) / kVThreads;
  if (need > 32) return cudaErrorInvalidValue;   // unreachable for V <= 32768 (checked by the entry point)
#define MEDUSA_RS(CC) return launch_rs_walk<T, CC>(c, ts, ncta, slice, tokens, parent, first_child, tl, hl, stats, hsP, ua, ur, w, st)
  if (need <= 1) MEDUSA_RS(1);
  if (need <= 2) MEDUSA_RS(2);
  if (need <= 4) MEDUSA_RS(4);
  if (need <= 8) MEDUSA_RS(8);
  if (need <= 16) MEDUSA_RS(16);
  MEDUSA_RS(32);
#undef MEDUSA_RS
}

template <typename T>
cudaError_t run_greedy(const medusa_cfg& c, const TreeShape& ts, const int32_t* tokens, const int32_t* parent,
                       const int32_t* first_child, const void* tl, const WalkOut& w, cudaStream_t st) {
  const T* rows = static_cast<const T*>(tl);
  if (c.V % 8 == 0)
    launch_pdl(greedy_walk_kernel<T, true>, c.B, kGwThreads, 0, st, ts, c.V, tokens, parent, first_child, rows, w);
  else
    launch_pdl(greedy_walk_kernel<T, false>, c.B, kGwThreads, 0, st, ts, c.V, tokens, parent, first_child, rows, w);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

MEDUSA_CHECK_TAKE(verify_take_checks)

size_t verify_workspace(const medusa_cfg& c) {
  const TreeShape ts = tree_shape(c);
  return align_up((size_t)c.B * ts.K * kMaxHsSlices * sizeof(float2), 256);   // head-row statistics (rejection)
}

cudaError_t launch_verify(const medusa_cfg& c, const int32_t* tokens, const int32_t* parent, const int32_t* first_child,
                          const void* tl, const float* hl, const float* u_acc, const float* u_res, int32_t* acc,
                          int32_t* path, int32_t* out_tokens, int32_t* n_out, uint32_t* flags, void* ws,
                          cudaStream_t st) {
  const TreeShape ts = tree_shape(c);
  WalkOut w{acc, path, out_tokens, n_out, flags};
  if (c.mode == MEDUSA_GREEDY)
    return c.dtype == MEDUSA_F32 ? run_greedy<float>(c, ts, tokens, parent, first_child, tl, w, st)
                                 : run_greedy<uint16_t>(c, ts, tokens, parent, first_child, tl, w, st);
  float2* stats = static_cast<float2*>(ws);
  return c.dtype == MEDUSA_F32 ? run_rs<float>(c, ts, tokens, parent, first_child, tl, hl, u_acc, u_res, w, stats, st)
                               : run_rs<uint16_t>(c, ts, tokens, parent, first_child, tl, hl, u_acc, u_res, w, stats, st);
}

}  // namespace medusa
