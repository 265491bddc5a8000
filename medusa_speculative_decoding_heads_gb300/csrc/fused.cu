// The whole verify step in one persistent launch: heads, tree, tree attention,
// greedy acceptance and KV compaction (small batches, bf16, head dim 128).
//
// One cooperative grid of one CTA per SM runs six phases separated by a grid
// barrier (a count and a generation word in the workspace; every wait is
// bounded and an expired one is recorded, not trapped):
//   0  residual block r_k = h + SiLU(W_k h + b_k) ("Medusa 심층 아키텍처",
//      section "잔차 블록(Residual Block)을 포함한 Medusa 헤드 구조"): one warp per
//      output row, 16-byte weight loads, h staged in shared memory as f32;
//   1  vocab projection z_k = U_k r_k (same section): one warp per vocabulary
//      row, head by head with r_k staged; each warp keeps, per sequence, its
//      eight best (value desc, index asc) in registers;
//   2  top-s per (sequence, head) merged from the warps' lists ("트리 어텐션":
//      each head keeps its top-s) and the tree: layout, ancestor mask, tokens
//      (Cartesian product, or a pruned tree's node list), position ids;
//   3  tree attention ("트리 어텐션", TreeMask equation) with the mma.sync unit of
//      attention_mma_unit.cuh over (row block, sequence x KV head, KV split);
//   4  the split partials merged by running max / exp-sum ("최적화 2편" §3.3)
//      into O, and the greedy walk ("최적화 2편" §1.3) on one CTA per sequence,
//      reading only the target rows it visits;
//   5  compaction of the accepted path's K/V rows ("Speculative Decoding 원리와
//      가속 아키텍처" §5 Case 2), L_b += acc_b + 1.
// The weight GEMVs run on CUDA cores (at B <= 4 every weight byte meets at most
// four FMAs per element), attention on the legacy tensor-core path.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attention_mma_unit.cuh"
#include "common.cuh"

namespace medusa {

__device__ uint32_t g_fused_error = 0;

namespace {

#ifndef MEDUSA_FUSED_THREADS
#define MEDUSA_FUSED_THREADS 384
#endif
#ifndef MEDUSA_FUSED_UNROLL
#define MEDUSA_FUSED_UNROLL 16
#endif
constexpr int kFT = MEDUSA_FUSED_THREADS;   // threads per CTA
constexpr int kFW = kFT / 32;     // warps per CTA
constexpr int kFusedMaxB = 4;
constexpr int kList = kMaxS;      // entries of a warp's candidate list
constexpr int kGemvUnroll = MEDUSA_FUSED_UNROLL;   // 16-byte weight loads in flight per lane
constexpr uint32_t kFusedBarrierCode = 0x40000000u;

struct FusedArgs {
  int B, d, V, K, Hq, Hkv, L_cap, shared_vocab, nsplit, chunk, row_blocks, compact;
  TreeShape ts;
  int16_t tree_parent[kMaxN];
  uint8_t tree_rank[kMaxN];
  float scale_log2;
  const uint16_t* h;
  const uint16_t* W;
  const uint16_t* bias;
  const uint16_t* U;
  const int32_t* root;
  int32_t* L;
  const uint16_t* Q;
  uint16_t* Kc;
  uint16_t* Vc;
  const uint16_t* tl;
  float* logits;
  int32_t* topk;
  int32_t* parent;
  int32_t* depth;
  int32_t* first_child;
  uint8_t* mask;
  uint64_t* bits;
  int32_t* tokens;
  int32_t* pos;
  uint32_t* flags;
  uint16_t* O;
  int32_t* acc;
  int32_t* path;
  int32_t* out_tokens;
  int32_t* n_out;
  int32_t* kv_map;
  float* r;        // [K][B][d]
  float* cand_v;   // [K][B][warps][kList]
  int* cand_i;
  float* o_part;   // [B][nsplit][N][Hq][128]
  float* ml_part;  // [B][nsplit][N][Hq][2]
  uint32_t* sync;  // [0] arrivals, [1] generation (arrivals zeroed before the launch)
};

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Grid-wide barrier of this cooperative launch. Returns false (CTA-uniform) when
// the wait expired; the expiry is recorded in g_fused_error.
__device__ bool grid_barrier(uint32_t* sync) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const uint32_t gen0 = ld_acquire(sync + 1);
    __threadfence();
    if (atomicAdd(sync, 1u) == gridDim.x - 1) {
      atomicExch(sync, 0u);   // ready for the next barrier before anyone is released
      __threadfence();
      atomicAdd(sync + 1, 1u);
    } else {
      const long long t0 = clock64();
      while (ld_acquire(sync + 1) == gen0) {
        if (clock64() - t0 > 4000000000LL) {
          atomicOr(&g_fused_error, kFusedBarrierCode);
          ok = 0;
          break;
        }
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Dot products of one bf16 weight row (d entries) with the BB vectors xs[b][d]
// (f32, shared memory); lane l takes the 16-byte chunks l, l + 32, ...; the sums
// are left in every lane.
template <int BB>
__device__ __forceinline__ void row_dot(const uint16_t* __restrict__ wrow, const float* __restrict__ xs, int d,
                                        float (&acc)[BB]) {
  const int lane = threadIdx.x & 31;
  const int nch = d >> 3;
#pragma unroll
  for (int b = 0; b < BB; ++b) acc[b] = 0.f;
  for (int c0 = lane; c0 < nch; c0 += 32 * kGemvUnroll) {
    uint4 w[kGemvUnroll];
#pragma unroll
    for (int u = 0; u < kGemvUnroll; ++u) {
      const int c = c0 + 32 * u;
      w[u] = c < nch ? ld_stream(wrow + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kGemvUnroll; ++u) {
      const int c = c0 + 32 * u;
      if (c < nch) {
        const float wf[8] = {bf16_lo(w[u].x), bf16_hi(w[u].x), bf16_lo(w[u].y), bf16_hi(w[u].y),
                             bf16_lo(w[u].z), bf16_hi(w[u].z), bf16_lo(w[u].w), bf16_hi(w[u].w)};
#pragma unroll
        for (int b = 0; b < BB; ++b) {
          const float4 x0 = *reinterpret_cast<const float4*>(xs + (size_t)b * d + 8 * c);
          const float4 x1 = *reinterpret_cast<const float4*>(xs + (size_t)b * d + 8 * c + 4);
          acc[b] += wf[0] * x0.x + wf[1] * x0.y + wf[2] * x0.z + wf[3] * x0.w + wf[4] * x1.x + wf[5] * x1.y +
                    wf[6] * x1.z + wf[7] * x1.w;
        }
      }
    }
  }
#pragma unroll
  for (int b = 0; b < BB; ++b)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], o);
}

// A sorted (value desc, index asc) list of kList candidates.
__device__ __forceinline__ void list_insert(float (&lv)[kList], int (&li)[kList], float x, int v) {
  if (!better(x, v, lv[kList - 1], li[kList - 1])) return;
  float cv = x;
  int ci = v;
#pragma unroll
  for (int k = 0; k < kList; ++k)
    if (better(cv, ci, lv[k], li[k])) {
      const float tv = lv[k];
      const int ti = li[k];
      lv[k] = cv;
      li[k] = ci;
      cv = tv;
      ci = ti;
    }
}

// Pops the best `s` of the warp's lanes' lists in order into (ov, oi) (every lane).
__device__ __forceinline__ void warp_pop(float (&lv)[kList], int (&li)[kList], int s, float* ov, int* oi) {
  const int lane = threadIdx.x & 31;
  for (int r = 0; r < s; ++r) {
    float v = lv[0];
    int i = li[0], who = lane;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
      const int w2 = __shfl_xor_sync(0xffffffffu, who, o);
      if (better(v2, i2, v, i)) {
        v = v2;
        i = i2;
        who = w2;
      }
    }
    ov[r] = v;
    oi[r] = i;
    if (lane == who) {
#pragma unroll
      for (int k = 0; k < kList - 1; ++k) {
        lv[k] = lv[k + 1];
        li[k] = li[k + 1];
      }
      lv[kList - 1] = -INFINITY;
      li[kList - 1] = 0x7fffffff;
    }
  }
}

// Depth, parent and rank of node n (Cartesian tree from the level counts, or the
// pruned tree's node list), and its first child (-1 for none).
__device__ void node_links(const FusedArgs& a, int n, int& dep, int& par, int& rank, int& fc) {
  const TreeShape& ts = a.ts;
  const int N = ts.N;
  dep = 0;
  par = -1;
  rank = 0;
  fc = -1;
  if (ts.pruned) {
    par = a.tree_parent[n];
    for (int j = par; j >= 0; j = a.tree_parent[j]) ++dep;
    rank = n > 0 ? a.tree_rank[n] : 0;
    for (int c = n + 1; c < N && fc < 0; ++c)
      if (a.tree_parent[c] == n) fc = c;
  } else {
    while (dep < ts.K && n >= ts.off[dep + 1]) ++dep;
    const int t = n - ts.off[dep];
    par = dep > 0 ? ts.off[dep - 1] + t / ts.s[dep] : -1;
    rank = dep > 0 ? t % ts.s[dep] : 0;
    fc = dep < ts.K ? ts.off[dep + 1] + t * ts.s[dep + 1] : -1;
  }
}

template <int BB>
__global__ void __launch_bounds__(kFT, 1) medusa_step_fused_kernel(const __grid_constant__ FusedArgs a) {
  extern __shared__ __align__(128) uint8_t fsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kFW + warp, TW = gridDim.x * kFW;
  const int B = BB, d = a.d, V = a.V, K = a.K, N = a.ts.N;
  float* xs = reinterpret_cast<float*>(fsm);   // phases 0 and 1: the vectors, [B][d] f32

  // ---------------------------------------------------------------- 0 residual block
  for (int e = threadIdx.x; e < B * d; e += kFT) xs[e] = bf16_to_f32(a.h[e]);
  __syncthreads();
  for (int row = gw; row < K * d; row += TW) {
    const int k = row / d, j = row - k * d;
    float s[BB];
    row_dot<BB>(a.W + (size_t)row * d, xs, d, s);
    if (lane < B) {
      float x = s[0];
#pragma unroll
      for (int b = 1; b < BB; ++b)
        if (lane == b) x = s[b];
      if (a.bias) x += bf16_to_f32(a.bias[(size_t)k * d + j]);
      a.r[((size_t)k * B + lane) * d + j] = xs[(size_t)lane * d + j] + x / (1.f + expf(-x));
    }
  }
  if (!grid_barrier(a.sync)) return;

  // ---------------------------------------------------------------- 1 vocab projection + lists
  for (int k = 0; k < K; ++k) {
    __syncthreads();   // the previous head's rows are done with xs
    for (int e = threadIdx.x; e < B * d; e += kFT) xs[e] = __ldcg(a.r + (size_t)k * B * d + e);
    __syncthreads();
    float lv[kList];
    int li[kList];
#pragma unroll
    for (int i = 0; i < kList; ++i) {
      lv[i] = -INFINITY;
      li[i] = 0x7fffffff;
    }
    const uint16_t* Uk = a.U + (a.shared_vocab ? (size_t)0 : (size_t)k * V * d);
    for (int v = gw; v < V; v += TW) {
      float s[BB];
      row_dot<BB>(Uk + (size_t)v * d, xs, d, s);
      if (lane < B) {
        float x = s[0];
#pragma unroll
        for (int b = 1; b < BB; ++b)
          if (lane == b) x = s[b];
        if (a.logits) a.logits[((size_t)lane * K + k) * V + v] = x;
        list_insert(lv, li, x, v);   // lane b keeps sequence b's list
      }
    }
    if (lane < B) {
      const size_t o = (((size_t)k * B + lane) * TW + gw) * kList;
#pragma unroll
      for (int i = 0; i < kList; ++i) {
        a.cand_v[o + i] = lv[i];
        a.cand_i[o + i] = li[i];
      }
    }
  }
  if (!grid_barrier(a.sync)) return;

  // ---------------------------------------------------------------- 2 top-s and the tree
  {
    __shared__ float wv[kFW][kList];
    __shared__ int wi[kFW][kList];
    __shared__ int best[kList];
    for (int item = blockIdx.x; item <= K * B; item += gridDim.x) {
      if (item == K * B) {
        // the tree layout (shared by all sequences), then per sequence the root token,
        // position ids and the capacity flag
        __shared__ uint64_t sb[kMaxN][2];
        for (int n = threadIdx.x; n < N; n += kFT) {
          int dep, par, rank, fc;
          node_links(a, n, dep, par, rank, fc);
          a.parent[n] = par;
          a.depth[n] = dep;
          a.first_child[n] = fc;
          uint64_t w0 = 0, w1 = 0;
          for (int j = n; j >= 0;) {
            if (j < 64) w0 |= 1ull << j;
            else w1 |= 1ull << (j - 64);
            int dj, pj, rj, fj;
            node_links(a, j, dj, pj, rj, fj);
            j = pj;
          }
          sb[n][0] = w0;
          sb[n][1] = w1;
          a.bits[2 * n] = w0;
          a.bits[2 * n + 1] = w1;
          for (int b = 0; b < B; ++b) {
            const int Lb = a.L[b];
            a.pos[(size_t)b * N + n] = Lb + dep;
            if (n == 0) {
              a.tokens[(size_t)b * N] = a.root[b];
              if (a.flags) a.flags[b] = (Lb < 0 || Lb + N > a.L_cap) ? MEDUSA_FLAG_CAPACITY : 0u;
            }
          }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < N * N; e += kFT) {
          const int i = e / N, j = e - i * N;
          a.mask[e] = uint8_t((sb[i][j >> 6] >> (j & 63)) & 1ull);
        }
        __syncthreads();
        continue;
      }
      const int k = item / B, b = item - k * B;
      const int s = a.ts.s[k + 1];
      float lv[kList];
      int li[kList];
#pragma unroll
      for (int i = 0; i < kList; ++i) {
        lv[i] = -INFINITY;
        li[i] = 0x7fffffff;
      }
      const size_t base = ((size_t)k * B + b) * TW * kList;
      for (int w = threadIdx.x; w < TW; w += kFT)
        for (int i = 0; i < s; ++i) list_insert(lv, li, __ldcg(a.cand_v + base + (size_t)w * kList + i),
                                                __ldcg(a.cand_i + base + (size_t)w * kList + i));
      float ov[kList];
      int oi[kList];
      warp_pop(lv, li, s, ov, oi);
      if (lane == 0)
        for (int r = 0; r < s; ++r) {
          wv[warp][r] = ov[r];
          wi[warp][r] = oi[r];
        }
      __syncthreads();
      if (warp == 0) {
#pragma unroll
        for (int i = 0; i < kList; ++i) {
          const bool have = lane < kFW && i < s;
          lv[i] = have ? wv[lane][i] : -INFINITY;
          li[i] = have ? wi[lane][i] : 0x7fffffff;
        }
        warp_pop(lv, li, s, ov, oi);
        if (lane == 0)
          for (int r = 0; r < s; ++r) best[r] = oi[r];
        if (lane < a.ts.s_max) a.topk[((size_t)b * K + k) * a.ts.s_max + lane] = lane < s ? oi[lane] : -1;
      }
      __syncthreads();
      for (int n = threadIdx.x; n < N; n += kFT) {   // head k's candidates are the tokens of depth k + 1
        int dep, par, rank, fc;
        node_links(a, n, dep, par, rank, fc);
        if (dep == k + 1) a.tokens[(size_t)b * N + n] = best[rank];
      }
      __syncthreads();
    }
  }
  if (!grid_barrier(a.sync)) return;

  // ---------------------------------------------------------------- 3 tree attention
  {
    const int units = a.row_blocks * B * a.Hkv * a.nsplit;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const int rbx = u % a.row_blocks, rest = u / a.row_blocks;
      const int y = rest % (B * a.Hkv), split = rest / (B * a.Hkv);
      mma_attn::tree_attn_mma_unit<128>(a.Q, a.Kc, a.Vc, a.L, a.bits, N, a.Hq, a.Hkv, a.L_cap, a.chunk, a.scale_log2,
                                        a.o_part, a.ml_part, rbx, y, split, a.nsplit, fsm);
    }
  }
  if (!grid_barrier(a.sync)) return;

  // ---------------------------------------------------------------- 4 merge into O; greedy walk
  {
    const size_t rows = (size_t)B * N * a.Hq;
    const int ns = a.nsplit;
    for (size_t e = (size_t)blockIdx.x * kFT + threadIdx.x; e < rows * 32; e += (size_t)gridDim.x * kFT) {
      const size_t row = e >> 5;
      const int q4 = (int)(e & 31) * 4;   // four head dims
      const int b = (int)(row / ((size_t)N * a.Hq));
      const size_t nh = row - (size_t)b * N * a.Hq;   // node * Hq + head
      float M = -INFINITY;
      for (int sp = 0; sp < ns; ++sp) M = fmaxf(M, __ldcg(a.ml_part + 2 * ((((size_t)b * ns + sp) * N * a.Hq) + nh)));
      float l = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
      if (M != -INFINITY)
        for (int sp = 0; sp < ns; ++sp) {
          const size_t pr = ((size_t)b * ns + sp) * N * a.Hq + nh;
          const float m = __ldcg(a.ml_part + 2 * pr);
          if (m == -INFINITY) continue;
          const float f = exp2f(m - M);
          l += f * __ldcg(a.ml_part + 2 * pr + 1);
          const float4 v = __ldcg(reinterpret_cast<const float4*>(a.o_part + pr * 128 + q4));
          o[0] += f * v.x;
          o[1] += f * v.y;
          o[2] += f * v.z;
          o[3] += f * v.w;
        }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint16_t* op = a.O + row * 128 + q4;
      *reinterpret_cast<uint2*>(op) =
          make_uint2((uint32_t)f32_to_bf16(o[0] * inv) | ((uint32_t)f32_to_bf16(o[1] * inv) << 16),
                     (uint32_t)f32_to_bf16(o[2] * inv) | ((uint32_t)f32_to_bf16(o[3] * inv) << 16));
    }
    if (blockIdx.x < B) {
      // greedy walk of sequence b: argmax of the current node's target row (lowest token id
      // among equal values), then the child carrying that token, if any
      const int b = blockIdx.x, KK = a.ts.K;
      __shared__ float sv[kFW];
      __shared__ int si[kFW];
      __shared__ int s_next;
      int32_t* path = a.path + (size_t)b * (KK + 1);
      int32_t* out = a.out_tokens + (size_t)b * (KK + 1);
      int cur = 0, acc = 0;
      if (threadIdx.x == 0) path[0] = 0;
      while (true) {
        const uint16_t* row = a.tl + ((size_t)b * N + cur) * V;
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        if ((V & 7) == 0) {
          for (int v0 = 8 * threadIdx.x; v0 < V; v0 += 8 * kFT) {
            const uint4 u = *reinterpret_cast<const uint4*>(row + v0);
            const float x[8] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y),
                                bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w)};
#pragma unroll
            for (int e2 = 0; e2 < 8; ++e2)
              if (better(x[e2], v0 + e2, bv, bi)) {
                bv = x[e2];
                bi = v0 + e2;
              }
          }
        } else {
          for (int v = threadIdx.x; v < V; v += kFT) {
            const float x = bf16_to_f32(row[v]);
            if (better(x, v, bv, bi)) {
              bv = x;
              bi = v;
            }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
          const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
          if (better(v2, i2, bv, bi)) {
            bv = v2;
            bi = i2;
          }
        }
        if (lane == 0) {
          sv[warp] = bv;
          si[warp] = bi;
        }
        __syncthreads();
        if (threadIdx.x < 32) {
          bv = lane < kFW ? sv[lane] : -INFINITY;
          bi = lane < kFW ? si[lane] : 0x7fffffff;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
            const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(v2, i2, bv, bi)) {
              bv = v2;
              bi = i2;
            }
          }
          if (lane == 0) {
            int nx = -1;
            const int fc = acc < KK ? __ldcg(a.first_child + cur) : -1;
            for (int j = 0; fc >= 0 && fc + j < N && __ldcg(a.parent + fc + j) == cur; ++j)
              if (__ldcg(a.tokens + (size_t)b * N + fc + j) == bi) nx = fc + j;
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
        for (int rr = acc + 1; rr <= KK; ++rr) {
          path[rr] = -1;
          out[rr] = -1;
        }
        a.acc[b] = acc;
        a.n_out[b] = acc + 1;
      }
    }
  }
  if (!grid_barrier(a.sync)) return;

  // ---------------------------------------------------------------- 5 compaction
  if (a.compact && blockIdx.x < B) {
    const int b = blockIdx.x, KK = a.ts.K;
    const int Lb = a.L[b];
    const int acc = __ldcg(a.acc + b);
    const bool ok = Lb >= 0 && Lb + N <= a.L_cap && acc >= 0 && acc <= KK;
    const int32_t* pb = a.path + (size_t)b * (KK + 1);
    constexpr int kRowVec = 128 * 2 / 16;   // 16-byte vectors per row
    if (ok) {
      int src[kMaxK + 1];
#pragma unroll
      for (int r = 0; r <= kMaxK; ++r) {
        const int sn = r <= acc ? __ldcg(pb + r) : r;
        src[r] = sn < 0 ? 0 : (sn >= N ? N - 1 : sn);
      }
      const int items = a.Hkv * 2 * kRowVec;
      for (int i = threadIdx.x; i < items; i += kFT) {
        const int col = i % kRowVec, hk = i / kRowVec;
        uint4* base = reinterpret_cast<uint4*>((hk & 1) ? a.Vc : a.Kc) +
                      ((size_t)b * a.Hkv + (hk >> 1)) * a.L_cap * kRowVec + col;
        uint4 v[kMaxK + 1];
#pragma unroll
        for (int r = 0; r <= kMaxK; ++r)
          if (r <= acc) v[r] = base[(size_t)(Lb + src[r]) * kRowVec];
#pragma unroll
        for (int r = 0; r <= kMaxK; ++r)
          if (r <= acc && src[r] != r) base[(size_t)(Lb + r) * kRowVec] = v[r];
      }
    }
    __syncthreads();   // every thread has read L[b]
    if (threadIdx.x <= KK) a.kv_map[(size_t)b * (KK + 1) + threadIdx.x] = (ok && threadIdx.x <= acc) ? __ldcg(pb + threadIdx.x) : -1;
    if (threadIdx.x == 0 && ok) a.L[b] = Lb + acc + 1;
  }
}

// Workspace layout of the fused step.
struct FusedPlan {
  int row_blocks, nsplit, chunk, warps_total;
  size_t r, cand_v, cand_i, o_part, ml_part, sync, total, smem;
};

int fused_grid() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
  }
  return n;
}

FusedPlan plan_fused(const medusa_cfg& c) {
  FusedPlan p{};
  const TreeShape ts = tree_shape(c);
  const int grid = fused_grid();
  const int NG = ts.N * (c.Hq / c.Hkv);
  p.row_blocks = ((NG + 15) / 16 + kFW - 1) / kFW;
  const int Lmax = c.L_cap - ts.N;
  const long units = (long)p.row_blocks * c.B * c.Hkv;
  int want = (int)(grid / units);
  const int by_len = (Lmax + 255) / 256;
  p.nsplit = want < by_len ? want : by_len;
  if (p.nsplit > 32) p.nsplit = 32;
  if (p.nsplit < 1) p.nsplit = 1;
  p.chunk = Lmax > 0 ? ((Lmax + p.nsplit - 1) / p.nsplit + mma_attn::kKeys - 1) / mma_attn::kKeys * mma_attn::kKeys
                     : mma_attn::kKeys;
  p.warps_total = grid * kFW;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  p.r = take((size_t)c.K * c.B * c.d * 4);
  p.cand_v = take((size_t)c.K * c.B * p.warps_total * kList * 4);
  p.cand_i = take((size_t)c.K * c.B * p.warps_total * kList * 4);
  const size_t rows = (size_t)c.B * p.nsplit * ts.N * c.Hq;
  p.o_part = take(rows * 128 * 4);
  p.ml_part = take(rows * 2 * 4);
  p.sync = take(2 * sizeof(uint32_t));
  p.total = off;
  const size_t vec = (size_t)c.B * c.d * 4;
  const size_t att = 2 * (size_t)mma_attn::kStages * mma_attn::kKeys * 128 * 2;
  p.smem = vec > att ? vec : att;
  return p;
}

}  // namespace

bool fused_supported(const medusa_cfg& c) {
  return c.dtype == MEDUSA_BF16 && c.D == 128 && c.mode == MEDUSA_GREEDY && c.B >= 1 && c.B <= kFusedMaxB &&
         c.d % 8 == 0 && (size_t)c.B * c.d * 4 <= 200 * 1024;
}

size_t fused_workspace(const medusa_cfg& c) { return fused_supported(c) ? plan_fused(c).total : 0; }

cudaError_t fused_take_error(uint32_t* out, cudaStream_t st) {
  static const uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_fused_error, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbolAsync(g_fused_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, st);
}

cudaError_t launch_fused_step(const medusa_cfg& c, const medusa_step_args& s, cudaStream_t st) {
  const FusedPlan p = plan_fused(c);
  const TreeShape ts = tree_shape(c);
  char* ws = static_cast<char*>(s.workspace);
  FusedArgs a{};
  a.B = c.B;
  a.d = c.d;
  a.V = c.V;
  a.K = c.K;
  a.Hq = c.Hq;
  a.Hkv = c.Hkv;
  a.L_cap = c.L_cap;
  a.shared_vocab = c.shared_vocab;
  a.nsplit = p.nsplit;
  a.chunk = p.chunk;
  a.row_blocks = p.row_blocks;
  a.compact = s.kv_compact;
  a.ts = ts;
  if (ts.pruned)
    for (int n = 0; n < ts.N; ++n) {
      a.tree_parent[n] = c.tree_parent[n];
      a.tree_rank[n] = c.tree_rank[n];
    }
  a.scale_log2 = (float)(1.4426950408889634 / sqrt(128.0));
  a.h = static_cast<const uint16_t*>(s.h);
  a.W = static_cast<const uint16_t*>(s.W);
  a.bias = static_cast<const uint16_t*>(s.bias);
  a.U = static_cast<const uint16_t*>(s.U);
  a.root = s.root_token;
  a.L = s.L;
  a.Q = static_cast<const uint16_t*>(s.Q);
  a.Kc = static_cast<uint16_t*>(s.Kc);
  a.Vc = static_cast<uint16_t*>(s.Vc);
  a.tl = static_cast<const uint16_t*>(s.target_logits);
  a.logits = s.logits;
  a.topk = s.topk;
  a.parent = s.parent;
  a.depth = s.depth;
  a.first_child = s.first_child;
  a.mask = s.mask;
  a.bits = s.anc_bits;
  a.tokens = s.tokens;
  a.pos = s.pos;
  a.flags = s.flags;
  a.O = static_cast<uint16_t*>(s.O);
  a.acc = s.acc;
  a.path = s.path;
  a.out_tokens = s.out_tokens;
  a.n_out = s.n_out;
  a.kv_map = s.kv_map;
  a.r = reinterpret_cast<float*>(ws + p.r);
  a.cand_v = reinterpret_cast<float*>(ws + p.cand_v);
  a.cand_i = reinterpret_cast<int*>(ws + p.cand_i);
  a.o_part = reinterpret_cast<float*>(ws + p.o_part);
  a.ml_part = reinterpret_cast<float*>(ws + p.ml_part);
  a.sync = reinterpret_cast<uint32_t*>(ws + p.sync);
  cudaError_t e = cudaMemsetAsync(a.sync, 0, 2 * sizeof(uint32_t), st);   // the barrier's arrival count
  if (e != cudaSuccess) return e;
  void (*kern)(const FusedArgs) = nullptr;
  switch (c.B) {
    case 1: kern = medusa_step_fused_kernel<1>; break;
    case 2: kern = medusa_step_fused_kernel<2>; break;
    case 3: kern = medusa_step_fused_kernel<3>; break;
    default: kern = medusa_step_fused_kernel<4>; break;
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFT, p.smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(fused_grid());
  cfg.blockDim = dim3(kFT);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident at once: the grid barrier needs it
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace medusa
