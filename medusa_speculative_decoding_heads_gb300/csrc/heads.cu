// Medusa heads: residual block, vocab projection and per-head top-s.
//
// "Medusa 심층 아키텍처" (techknowgenie), section "잔차 블록(Residual Block)을
// 포함한 Medusa 헤드 구조", equations h_t^(k) = SiLU(h_t W_res^(k)) + h_t and
// p_k = softmax(h_t^(k) W_head^(k)); the section "소스코드 레벨 구조 분석"
// (MedusaHead: Linear(d,d), SiLU, + residual, Linear(d,V); generate_candidates:
// torch.topk(...).indices per head).
//
// Both projections are "many weight rows times a handful of vectors": the
// weights stream from HBM once per call and each weight tile meets all B input
// vectors while it is on chip.
//
// The bf16 projections run on the tcgen05 path (heads_tc.cu); this file keeps
// the per-head top-s selection, the float32 path and the dispatch.
//
// f32 path (CUDA cores): plain FMA GEMV, used for float32 weights.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace medusa {
namespace {

// ---------------------------------------------------------------- float32 path
// out[b][g][row] = sum_i A[g][row][i] * X[b][g or 0][i]  (+ optional residual epilogue)
constexpr int kF32Rows = 4;       // rows per warp
constexpr int kF32B = 8;          // batch handled per pass
constexpr int kF32DChunk = 1024;

template <bool RESIDUAL>
__global__ void __launch_bounds__(256)
heads_f32_kernel(const float* __restrict__ A, size_t a_group_stride, int rows, int d, const float* __restrict__ X,
                 size_t x_b_stride, size_t x_group_stride, int B, int G, float* __restrict__ out,
                 const float* __restrict__ h, const float* __restrict__ bias) {
  pdl_wait();
  pdl_trigger();
  __shared__ float xs[kF32B][kF32DChunk];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.y;
  const int row0 = (blockIdx.x * 8 + warp) * kF32Rows;
  const float* Xg = X + (size_t)g * x_group_stride;
  for (int b0 = 0; b0 < B; b0 += kF32B) {
    const int nb = min(kF32B, B - b0);
    float acc[kF32Rows][kF32B];
#pragma unroll
    for (int r = 0; r < kF32Rows; ++r)
#pragma unroll
      for (int b = 0; b < kF32B; ++b) acc[r][b] = 0.f;
    for (int k0 = 0; k0 < d; k0 += kF32DChunk) {
      const int kn = min(kF32DChunk, d - k0);
      __syncthreads();
      for (int i = threadIdx.x; i < kF32B * kF32DChunk; i += blockDim.x) {
        int b = i / kF32DChunk, k = i % kF32DChunk;
        xs[b][k] = (b < nb && k < kn) ? Xg[(size_t)(b0 + b) * x_b_stride + k0 + k] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < kF32Rows; ++r) {
        int row = row0 + r;
        if (row >= rows) continue;
        const float* ar = A + (size_t)g * a_group_stride + (size_t)row * d + k0;
        for (int k = lane; k < kn; k += 32) {
          float a = ar[k];
#pragma unroll
          for (int b = 0; b < kF32B; ++b) acc[r][b] = fmaf(a, xs[b][k], acc[r][b]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kF32Rows; ++r)
#pragma unroll
      for (int b = 0; b < kF32B; ++b) acc[r][b] = warp_sum(acc[r][b]);
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < kF32Rows; ++r) {
        int row = row0 + r;
        if (row >= rows) continue;
        for (int b = 0; b < nb; ++b) {
          float v = acc[r][b];
          size_t oi = ((size_t)(b0 + b) * G + g) * rows + row;
          if (RESIDUAL) {
            float pre = v + (bias ? bias[(size_t)g * rows + row] : 0.f);
            v = h[(size_t)(b0 + b) * rows + row] + pre / (1.f + expf(-pre));
          }
          out[oi] = v;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- top-s per (b, k)
// Order: value descending, index ascending. Two kernels: many CTAs each reduce a
// slice of a row to its top-s candidates, then one warp per row merges them.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

constexpr int kTopThreads = 256;

// Warp-wide best of (v, i) pairs; returns the winner's pair and lane in all lanes.
__device__ __forceinline__ void warp_best(float& v, int& i, int& who) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    const int ow = __shfl_xor_sync(0xffffffffu, who, o);
    if (better(ov, oi, v, i)) {
      v = ov;
      i = oi;
      who = ow;
    }
  }
}

// Pops the s best of the lanes' sorted lists (lv/li, kMaxS deep) in order.
__device__ __forceinline__ void warp_top_s(float* lv, int* li, int s, float* ov, int* oi) {
  const int lane = threadIdx.x & 31;
  for (int r = 0; r < s; ++r) {
    float v = lv[0];
    int i = li[0];
    int who = lane;
    warp_best(v, i, who);
    ov[r] = v;
    oi[r] = i;
    if (lane == who) {
#pragma unroll
      for (int k = 0; k < kMaxS - 1; ++k) {
        lv[k] = lv[k + 1];
        li[k] = li[k + 1];
      }
      lv[kMaxS - 1] = -INFINITY;
      li[kMaxS - 1] = 0x7fffffff;
    }
  }
}

__device__ __forceinline__ void list_insert(float* lv, int* li, float x, int v) {
  if (!better(x, v, lv[kMaxS - 1], li[kMaxS - 1])) return;
  float cv = x;
  int ci = v;
#pragma unroll
  for (int k = 0; k < kMaxS; ++k) {
    if (better(cv, ci, lv[k], li[k])) {
      const float tv = lv[k];
      const int ti = li[k];
      lv[k] = cv;
      li[k] = ci;
      cv = tv;
      ci = ti;
    }
  }
}

// The s best of a lane's (value, index) list, kept sorted; S = the list length.
template <int S>
__device__ __forceinline__ void list_insert_s(float* lv, int* li, float x, int v) {
  if (!better(x, v, lv[S - 1], li[S - 1])) return;
  float cv = x;
  int ci = v;
#pragma unroll
  for (int k = 0; k < S; ++k) {
    if (better(cv, ci, lv[k], li[k])) {
      const float tv = lv[k];
      const int ti = li[k];
      lv[k] = cv;
      li[k] = ci;
      cv = tv;
      ci = ti;
    }
  }
}

// Pops the S best of the lanes' sorted lists in order.
template <int S>
__device__ __forceinline__ void warp_top_s_t(float* lv, int* li, float* ov, int* oi) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < S; ++r) {
    float v = lv[0];
    int i = li[0];
    int who = lane;
    warp_best(v, i, who);
    ov[r] = v;
    oi[r] = i;
    if (lane == who) {
#pragma unroll
      for (int k = 0; k < S - 1; ++k) {
        lv[k] = lv[k + 1];
        li[k] = li[k + 1];
      }
      lv[S - 1] = -INFINITY;
      li[S - 1] = 0x7fffffff;
    }
  }
}

// One CTA: the S best of row[v0, v1). With VEC4 (rows and slices aligned to 4
// floats) every thread issues two 16-byte loads per step before inserting.
template <int S, bool VEC4>
__device__ __forceinline__ void topk_slice(const float* __restrict__ row, int v0, int v1, float* __restrict__ out_v,
                                           int* __restrict__ out_i) {
  float lv[S];
  int li[S];
#pragma unroll
  for (int i = 0; i < S; ++i) {
    lv[i] = -INFINITY;
    li[i] = 0x7fffffff;
  }
  if (VEC4) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int g0 = v0 >> 2, g1 = v1 >> 2;
    for (int g = g0 + threadIdx.x; g < g1; g += 2 * kTopThreads) {
      const float4 a = r4[g];
      const bool two = g + kTopThreads < g1;
      const float4 c = two ? r4[g + kTopThreads] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      list_insert_s<S>(lv, li, a.x, 4 * g);
      list_insert_s<S>(lv, li, a.y, 4 * g + 1);
      list_insert_s<S>(lv, li, a.z, 4 * g + 2);
      list_insert_s<S>(lv, li, a.w, 4 * g + 3);
      if (two) {
        const int gc = g + kTopThreads;
        list_insert_s<S>(lv, li, c.x, 4 * gc);
        list_insert_s<S>(lv, li, c.y, 4 * gc + 1);
        list_insert_s<S>(lv, li, c.z, 4 * gc + 2);
        list_insert_s<S>(lv, li, c.w, 4 * gc + 3);
      }
    }
  } else {
    for (int v = v0 + threadIdx.x; v < v1; v += kTopThreads) list_insert_s<S>(lv, li, row[v], v);
  }
  __shared__ float wv[kTopThreads / 32][kMaxS];
  __shared__ int wi[kTopThreads / 32][kMaxS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float tv[S];
  int ti[S];
  warp_top_s_t<S>(lv, li, tv, ti);
  if (lane == 0)
#pragma unroll
    for (int r = 0; r < S; ++r) {
      wv[warp][r] = tv[r];
      wi[warp][r] = ti[r];
    }
  __syncthreads();
  if (warp == 0) {
    // lane w < 8 holds warp w's sorted list
#pragma unroll
    for (int i = 0; i < S; ++i) {
      const bool have = lane < kTopThreads / 32;
      lv[i] = have ? wv[lane][i] : -INFINITY;
      li[i] = have ? wi[lane][i] : 0x7fffffff;
    }
    warp_top_s_t<S>(lv, li, tv, ti);
    if (lane == 0)
#pragma unroll
      for (int r = 0; r < S; ++r) {
        out_v[r] = tv[r];
        out_i[r] = ti[r];
      }
  }
}

// grid (P, K, B): slice p of row (b, k) -> s candidates at cand[((b*K + k)*P + p)*s_max + r].
template <bool VEC4>
__global__ void __launch_bounds__(kTopThreads)
topk_partial_kernel(const float* __restrict__ z, int V, TreeShape ts, int chunk, float* __restrict__ cv,
                    int* __restrict__ ci) {
  pdl_wait();
  pdl_trigger();
  const int p = blockIdx.x, k = blockIdx.y, b = blockIdx.z, P = gridDim.x;
  const int K = ts.K, s = ts.s[k + 1], s_max = ts.s_max;
  const float* row = z + ((size_t)b * K + k) * V;
  const int v0 = min(V, p * chunk), v1 = min(V, v0 + chunk);
  const size_t o = (((size_t)b * K + k) * P + p) * s_max;
  switch (s) {
    case 1: topk_slice<1, VEC4>(row, v0, v1, cv + o, ci + o); break;
    case 2: topk_slice<2, VEC4>(row, v0, v1, cv + o, ci + o); break;
    case 3: topk_slice<3, VEC4>(row, v0, v1, cv + o, ci + o); break;
    case 4: topk_slice<4, VEC4>(row, v0, v1, cv + o, ci + o); break;
    case 5: topk_slice<5, VEC4>(row, v0, v1, cv + o, ci + o); break;
    case 6: topk_slice<6, VEC4>(row, v0, v1, cv + o, ci + o); break;
    case 7: topk_slice<7, VEC4>(row, v0, v1, cv + o, ci + o); break;
    default: topk_slice<8, VEC4>(row, v0, v1, cv + o, ci + o); break;
  }
}

// grid (K, B), one warp: merge P slices' candidates into topk[b][k][:].
__global__ void topk_merge_kernel(const float* __restrict__ cv, const int* __restrict__ ci, int P, TreeShape ts,
                                  int32_t* __restrict__ topk) {
  pdl_wait();
  pdl_trigger();
  const int k = blockIdx.x, b = blockIdx.y, lane = threadIdx.x;
  const int K = ts.K, s = ts.s[k + 1], s_max = ts.s_max;
  float lv[kMaxS];
  int li[kMaxS];
#pragma unroll
  for (int i = 0; i < kMaxS; ++i) {
    lv[i] = -INFINITY;
    li[i] = 0x7fffffff;
  }
  const size_t base = ((size_t)b * K + k) * P * s_max;
  for (int p = lane; p < P; p += 32)
    for (int r = 0; r < s; ++r) list_insert(lv, li, cv[base + (size_t)p * s_max + r], ci[base + (size_t)p * s_max + r]);
  float tv[kMaxS];
  int ti[kMaxS];
  warp_top_s(lv, li, s, tv, ti);
  if (lane == 0)
    for (int r = 0; r < s_max; ++r) topk[((size_t)b * K + k) * s_max + r] = r < s ? ti[r] : -1;
}

int topk_slices(const medusa_cfg& c) {
  int P = (4 * 152 + c.K * c.B - 1) / (c.K * c.B);
  P = P < 1 ? 1 : (P > 64 ? 64 : P);
  const int max_by_len = (c.V + 255) / 256;
  return P < max_by_len ? P : (max_by_len < 1 ? 1 : max_by_len);
}

struct HeadsPlan {
  size_t r, zbuf, cand, tc, total;   // byte offsets / sizes
};

// Workspace of one heads pass: r (float32 path), the logits when the caller
// keeps none, the top-s candidates and the tcgen05 path's own buffers.
HeadsPlan plan_heads(const medusa_cfg& c) {
  HeadsPlan p{};
  const size_t B = c.B, d = c.d, V = c.V, K = c.K;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  p.r = take(c.dtype == MEDUSA_BF16 ? 0 : B * K * d * 4);
  p.zbuf = take(B * K * V * 4);
  p.cand = take((size_t)B * K * topk_slices(c) * kMaxS * 8);
  p.tc = take(c.dtype == MEDUSA_BF16 ? plan_heads_tc(c).total : 0);
  p.total = off;
  return p;
}

}  // namespace

// Enough for every batch slice that medusa_heads runs (bf16: slices of at most kHeadsBatch sequences).
size_t heads_workspace(const medusa_cfg& c) {
  if (c.dtype != MEDUSA_BF16 || c.B <= kHeadsBatch) return plan_heads(c).total;
  medusa_cfg full = c, tail = c;
  full.B = kHeadsBatch;
  tail.B = c.B % kHeadsBatch == 0 ? kHeadsBatch : c.B % kHeadsBatch;
  const size_t a = plan_heads(full).total, t = plan_heads(tail).total;
  return a > t ? a : t;
}

cudaError_t launch_heads(const medusa_cfg& c, const void* h, const void* W, const void* bias, const void* U,
                         float* logits, int32_t* topk, void* ws, cudaStream_t st) {
  const HeadsPlan p = plan_heads(c);
  char* base = static_cast<char*>(ws);
  const int B = c.B, d = c.d, V = c.V, K = c.K;
  float* z = logits ? logits : reinterpret_cast<float*>(base + p.zbuf);
  const size_t u_stride = c.shared_vocab ? 0 : (size_t)V * d;   // elements between heads' vocab projections

  if (c.dtype == MEDUSA_BF16) {
    if (!heads_tc_supported(c)) return cudaErrorNotSupported;   // medusa_heads slices larger batches
    cudaError_t e = launch_heads_tc(c, h, W, bias, U, z, base + p.tc, st);
    if (e != cudaSuccess) return e;
  } else {
    float* r = reinterpret_cast<float*>(base + p.r);
    dim3 g1((d + 32 - 1) / 32, K);
    launch_pdl(heads_f32_kernel<true>, g1, 256, 0, st, static_cast<const float*>(W), (size_t)d * d, d, d,
                                               static_cast<const float*>(h),
                                               (size_t)d, 0, B, K, r, static_cast<const float*>(h),
                                               static_cast<const float*>(bias));
    note_launches(1);
    dim3 g2((V + 32 - 1) / 32, K);
    launch_pdl(heads_f32_kernel<false>, g2, 256, 0, st, static_cast<const float*>(U), u_stride, V, d, r, (size_t)K * d,
                                                (size_t)d, B,
                                                K, z, nullptr, nullptr);
    note_launches(1);
  }
  const TreeShape ts = tree_shape(c);
  const int P = topk_slices(c);
  const bool vec4 = V % 4 == 0 && (reinterpret_cast<uintptr_t>(z) & 15u) == 0;
  const int chunk = vec4 ? ((V + P - 1) / P + 3) / 4 * 4 : (V + P - 1) / P;
  float* cv = reinterpret_cast<float*>(base + p.cand);
  int* ci = reinterpret_cast<int*>(cv + (size_t)B * K * P * kMaxS);
  if (vec4)
    launch_pdl(topk_partial_kernel<true>, dim3(P, K, B), kTopThreads, 0, st, z, V, ts, chunk, cv, ci);
  else
    launch_pdl(topk_partial_kernel<false>, dim3(P, K, B), kTopThreads, 0, st, z, V, ts, chunk, cv, ci);
  note_launches(1);
  launch_pdl(topk_merge_kernel, dim3(K, B), 32, 0, st, cv, ci, P, ts, topk);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace medusa
