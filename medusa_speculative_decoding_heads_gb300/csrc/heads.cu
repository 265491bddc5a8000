// Medusa heads: residual block, vocab projection and per-head top-s.
//
// "Medusa 심층 아키텍처" (techknowgenie), section "잔차 블록(Residual Block)을
// 포함한 Medusa 헤드 구조", equations h_t^(k) = SiLU(h_t W_res^(k)) + h_t and
// p_k = softmax(h_t^(k) W_head^(k)); the section "소스코드 레벨 구조 분석"
// (MedusaHead: Linear(d,d), SiLU, + residual, Linear(d,V); generate_candidates:
// torch.topk(...).indices per head).
//
// Both projections are "many weight rows times a handful of vectors": the
// weights stream from HBM exactly once and each weight row meets all B input
// vectors while it is in registers.
//
// The tcgen05 path (heads_tc.cu) serves bf16 with B <= 32 and d % 64 == 0; this
// file keeps the per-head top-s selection and the paths for other shapes.
//
// bf16 path (tensor cores, mma.sync m16n8k16, swap-AB): the weight rows are the
// 16-row A operand, the batch is the 8-wide B operand. Products of two bf16
// values are exact in the f32 accumulator, so the d x d layer on the bf16
// hidden state is exact up to f32 accumulation. The vocab projection consumes
// the f32 residual r, split as r = hi + lo with hi, lo bf16 (two MMAs), which
// keeps 16 significant bits of r — enough that the logits agree with a float64
// evaluation to ~1e-6 relative and the top-s order is the exact order except at
// near ties.
//
// Each lane loads 16-byte vectors of a weight row directly into registers and
// the k index inside a 64-wide chunk is permuted identically for the weights
// and the vectors, so no shuffle or shared-memory transpose is needed.
//
// f32 path (CUDA cores): plain FMA GEMV, used for float32 weights.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace medusa {
namespace {

constexpr int kWarps = 8;
constexpr int kRT = 2;                      // 16-row tiles per warp
constexpr int kRowsPerCta = kWarps * kRT * 16;
constexpr int kChunk = 64;                  // k elements per pipeline step
constexpr int kXStages = 4;

__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ uint32_t pick(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Packed vector operand ("Xp"): for group g, chunk c, n-tile t, part p (hi/lo),
// half hh and lane l = 4*gid + cq, 8 bf16 = X[8t+gid][64c + 32hh + 8cq + 0..7].
// One (g, c, t, p) block is 1 KB: [hh][lane][8].
__host__ __device__ __forceinline__ size_t xp_index(int c, int t, int p, int hh, int lane, int NT, int P) {
  return ((((size_t)c * NT + t) * P + p) * 2 + hh) * 256 + (size_t)lane * 8;
}

// out[ks][b][g][row] (+)= sum over this split's chunks of A[g][row][:] . X[b][g][:]
template <int NT, int P>
__global__ void __launch_bounds__(kWarps * 32, 1)
heads_mma_kernel(const uint16_t* __restrict__ A, size_t a_group_stride, int rows, int d,
                 const uint16_t* __restrict__ Xp, size_t xp_group_stride, int chunks_per_split,
                 float* __restrict__ out, size_t out_split_stride, int B, int G) {
  pdl_wait();
  pdl_trigger();
  __shared__ __align__(16) uint16_t xs[kXStages][NT * P * 2 * 256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, cq = lane & 3;
  const int g = blockIdx.y, ks = blockIdx.z;
  const int nchunks = d / kChunk;
  const int c0 = ks * chunks_per_split;
  const int c1 = min(nchunks, c0 + chunks_per_split);
  const int row_base = blockIdx.x * kRowsPerCta + warp * kRT * 16;

  const uint16_t* Ag = A + (size_t)g * a_group_stride;
  const uint16_t* Xg = Xp + (size_t)g * xp_group_stride;

  // Row pointers of this lane (rows gid and gid+8 of each tile), clamped for ragged tails.
  const uint16_t* arow[kRT][2];
#pragma unroll
  for (int rt = 0; rt < kRT; ++rt)
#pragma unroll
    for (int r2 = 0; r2 < 2; ++r2) {
      int row = min(row_base + rt * 16 + gid + 8 * r2, rows - 1);
      arow[rt][r2] = Ag + (size_t)row * d + 8 * cq;
    }

  float acc[kRT][NT][4];
#pragma unroll
  for (int rt = 0; rt < kRT; ++rt)
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[rt][t][i] = 0.f;

  constexpr int kXVec = NT * P * 2 * 256 / 8;   // 16-byte vectors per stage
  auto load_x = [&](int stage, int c) {
    const uint16_t* src = Xg + xp_index(c, 0, 0, 0, 0, NT, P);
    for (int v = threadIdx.x; v < kXVec; v += kWarps * 32) cp_async16(&xs[stage][v * 8], src + (size_t)v * 8);
  };

  // Prologue: X stages and the first A chunk.
#pragma unroll
  for (int s = 0; s < kXStages - 1; ++s) {
    if (c0 + s < c1) load_x(s, c0 + s);
    cp_async_commit();
  }
  uint4 a_cur[kRT][2][2], a_nxt[kRT][2][2];
  if (c0 < c1) {
#pragma unroll
    for (int rt = 0; rt < kRT; ++rt)
#pragma unroll
      for (int r2 = 0; r2 < 2; ++r2)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) a_cur[rt][r2][hh] = ldg_stream(arow[rt][r2] + (size_t)c0 * kChunk + 32 * hh);
  }

  for (int c = c0; c < c1; ++c) {
    const int it = c - c0;
    if (c + 1 < c1) {
#pragma unroll
      for (int rt = 0; rt < kRT; ++rt)
#pragma unroll
        for (int r2 = 0; r2 < 2; ++r2)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            a_nxt[rt][r2][hh] = ldg_stream(arow[rt][r2] + (size_t)(c + 1) * kChunk + 32 * hh);
    }
    {
      int cn = c + kXStages - 1;
      if (cn < c1) load_x((it + kXStages - 1) % kXStages, cn);
      cp_async_commit();
    }
    cp_async_wait<kXStages - 1>();
    __syncthreads();
    const uint16_t* xst = xs[it % kXStages];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      uint4 xw[NT][P];
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int p = 0; p < P; ++p)
          xw[t][p] = *reinterpret_cast<const uint4*>(xst + xp_index(0, t, p, hh, lane, NT, P));
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
#pragma unroll
        for (int rt = 0; rt < kRT; ++rt) {
          uint32_t a0 = pick(a_cur[rt][0][hh], 2 * jj), a2 = pick(a_cur[rt][0][hh], 2 * jj + 1);
          uint32_t a1 = pick(a_cur[rt][1][hh], 2 * jj), a3 = pick(a_cur[rt][1][hh], 2 * jj + 1);
#pragma unroll
          for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int p = 0; p < P; ++p)
              mma_bf16(acc[rt][t], a0, a1, a2, a3, pick(xw[t][p], 2 * jj), pick(xw[t][p], 2 * jj + 1));
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int rt = 0; rt < kRT; ++rt)
#pragma unroll
      for (int r2 = 0; r2 < 2; ++r2)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) a_cur[rt][r2][hh] = a_nxt[rt][r2][hh];
  }
  cp_async_wait<0>();

  float* o = out + (size_t)ks * out_split_stride;
  const size_t bstride = (size_t)G * rows;
#pragma unroll
  for (int rt = 0; rt < kRT; ++rt)
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        int row = row_base + rt * 16 + gid + ((i & 2) ? 8 : 0);
        int b = 8 * t + 2 * cq + (i & 1);
        if (row < rows && b < B) o[(size_t)b * bstride + (size_t)g * rows + row] = acc[rt][t][i];
      }
}

// Pack the bf16 hidden state into the vector-operand layout (hi part only).
template <int NT>
__global__ void pack_h_kernel(const uint16_t* __restrict__ h, uint16_t* __restrict__ Xp, int B, int d) {
  pdl_wait();
  pdl_trigger();
  const int nchunks = d / kChunk;
  const size_t total = (size_t)nchunks * NT * 2 * 32;   // (c, t, hh, lane) vectors of 8
  for (size_t v = blockIdx.x * (size_t)blockDim.x + threadIdx.x; v < total; v += (size_t)gridDim.x * blockDim.x) {
    int lane = v % 32;
    int hh = (v / 32) % 2;
    int t = (v / 64) % NT;
    int c = v / (64 * NT);
    int n = 8 * t + (lane >> 2);
    int k0 = c * kChunk + 32 * hh + 8 * (lane & 3);
    uint4 val = make_uint4(0, 0, 0, 0);
    if (n < B) val = *reinterpret_cast<const uint4*>(h + (size_t)n * d + k0);
    *reinterpret_cast<uint4*>(Xp + xp_index(c, t, 0, hh, lane, NT, 1)) = val;
  }
}

// r = h + SiLU(sum_splits pre + bias), then pack hi/lo of r for the vocab projection.
// One thread per (b, k, 8 consecutive features).
template <int NT>
__global__ void residual_pack_kernel(const float* __restrict__ part, int ksplit, const uint16_t* __restrict__ h,
                                     const uint16_t* __restrict__ bias, uint16_t* __restrict__ Xp2, int B, int K,
                                     int d) {
  pdl_wait();
  pdl_trigger();
  const int nchunks = d / kChunk;
  const size_t total = (size_t)K * nchunks * NT * 2 * 32;   // (k, c, t, hh, lane)
  const size_t split_stride = (size_t)B * K * d;
  for (size_t v = blockIdx.x * (size_t)blockDim.x + threadIdx.x; v < total; v += (size_t)gridDim.x * blockDim.x) {
    int lane = v % 32;
    int hh = (v / 32) % 2;
    int t = (v / 64) % NT;
    int c = (v / (64 * NT)) % nchunks;
    int k = v / ((size_t)64 * NT * nchunks);
    int n = 8 * t + (lane >> 2);
    int o0 = c * kChunk + 32 * hh + 8 * (lane & 3);
    uint16_t hi[8], lo[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      hi[e] = 0;
      lo[e] = 0;
    }
    if (n < B) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        int o = o0 + e;
        float pre = 0.f;
        for (int s = 0; s < ksplit; ++s) pre += part[s * split_stride + ((size_t)n * K + k) * d + o];
        if (bias) pre += bf16_to_f32(bias[(size_t)k * d + o]);
        float r = bf16_to_f32(h[(size_t)n * d + o]) + pre / (1.f + expf(-pre));
        hi[e] = f32_to_bf16(r);
        lo[e] = f32_to_bf16(r - bf16_to_f32(hi[e]));
      }
    }
    uint4 vh, vl;
    vh.x = hi[0] | (uint32_t(hi[1]) << 16); vh.y = hi[2] | (uint32_t(hi[3]) << 16);
    vh.z = hi[4] | (uint32_t(hi[5]) << 16); vh.w = hi[6] | (uint32_t(hi[7]) << 16);
    vl.x = lo[0] | (uint32_t(lo[1]) << 16); vl.y = lo[2] | (uint32_t(lo[3]) << 16);
    vl.z = lo[4] | (uint32_t(lo[5]) << 16); vl.w = lo[6] | (uint32_t(lo[7]) << 16);
    uint16_t* base = Xp2 + (size_t)k * nchunks * NT * 2 * 512;
    *reinterpret_cast<uint4*>(base + xp_index(c, t, 0, hh, lane, NT, 2)) = vh;
    *reinterpret_cast<uint4*>(base + xp_index(c, t, 1, hh, lane, NT, 2)) = vl;
  }
}

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
  int NT;          // 8-wide batch tiles (bf16 path)
  int ksplit1;     // split of d for the d x d layer
  size_t xp1, xp2, part1, zbuf, cand, tc, total;   // byte offsets / sizes
};

HeadsPlan plan_heads(const medusa_cfg& c) {
  HeadsPlan p{};
  const size_t B = c.B, d = c.d, V = c.V, K = c.K;
  p.NT = c.B <= 8 ? 1 : c.B <= 16 ? 2 : 4;
  const int nchunks = c.d / kChunk;
  const int blocks1 = ((c.d + kRowsPerCta - 1) / kRowsPerCta) * c.K;
  int ks = (2 * 152 + blocks1 - 1) / blocks1;
  ks = ks < 1 ? 1 : ks;
  ks = ks > nchunks ? nchunks : ks;
  p.ksplit1 = (c.dtype == MEDUSA_BF16) ? ks : 1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  if (heads_tc_supported(c)) {
    p.xp1 = p.xp2 = p.part1 = take(0);
  } else if (c.dtype == MEDUSA_BF16) {
    p.xp1 = take((size_t)nchunks * p.NT * 1024);
    p.xp2 = take(K * nchunks * p.NT * 2048);
    p.part1 = take((size_t)p.ksplit1 * B * K * d * 4);
  } else {
    p.xp1 = take(0);
    p.xp2 = take(B * K * d * 4);           // r (float32)
    p.part1 = take(0);
  }
  p.zbuf = take(B * K * V * 4);
  p.cand = take((size_t)B * K * topk_slices(c) * kMaxS * 8);
  if (heads_tc_supported(c)) p.tc = take(plan_heads_tc(c).total);
  p.total = off;
  return p;
}

}  // namespace

size_t heads_workspace(const medusa_cfg& c) { return plan_heads(c).total; }

cudaError_t launch_heads(const medusa_cfg& c, const void* h, const void* W, const void* bias, const void* U,
                         float* logits, int32_t* topk, void* ws, cudaStream_t st) {
  const HeadsPlan p = plan_heads(c);
  char* base = static_cast<char*>(ws);
  const int B = c.B, d = c.d, V = c.V, K = c.K;
  float* z = logits ? logits : reinterpret_cast<float*>(base + p.zbuf);
  const size_t u_stride = c.shared_vocab ? 0 : (size_t)V * d;   // elements between heads' vocab projections

  if (heads_tc_supported(c)) {
    cudaError_t e = launch_heads_tc(c, h, W, bias, U, z, base + p.tc, st);
    if (e != cudaSuccess) return e;
  } else if (c.dtype == MEDUSA_BF16) {
    uint16_t* xp1 = reinterpret_cast<uint16_t*>(base + p.xp1);
    uint16_t* xp2 = reinterpret_cast<uint16_t*>(base + p.xp2);
    float* part1 = reinterpret_cast<float*>(base + p.part1);
    const int nchunks = d / kChunk;
    const int cps1 = (nchunks + p.ksplit1 - 1) / p.ksplit1;
    dim3 g1((d + kRowsPerCta - 1) / kRowsPerCta, K, p.ksplit1);
    dim3 g2((V + kRowsPerCta - 1) / kRowsPerCta, K, 1);
    const size_t xp2_group = (size_t)nchunks * p.NT * 2 * 512;
#define MEDUSA_HEADS_BF16(NT_)                                                                                   \
  do {                                                                                                           \
    launch_pdl(pack_h_kernel<NT_>, 64, 256, 0, st, static_cast<const uint16_t*>(h), xp1, B, d);                           \
    launch_pdl(heads_mma_kernel<NT_, 1>, g1, kWarps * 32, 0, st, static_cast<const uint16_t*>(W), (size_t)d * d, d, d,   \
                                                        xp1, 0, cps1, part1, (size_t)B * K * d, B, K);          \
    launch_pdl(residual_pack_kernel<NT_>, 256, 256, 0, st, part1, p.ksplit1, static_cast<const uint16_t*>(h),           \
                                                   static_cast<const uint16_t*>(bias), xp2, B, K, d);           \
    launch_pdl(heads_mma_kernel<NT_, 2>, g2, kWarps * 32, 0, st, static_cast<const uint16_t*>(U), u_stride, V, d,      \
                                                        xp2, xp2_group, nchunks, z, 0, B, K);                   \
    note_launches(4);                                                                                            \
  } while (0)
    if (p.NT == 1) MEDUSA_HEADS_BF16(1);
    else if (p.NT == 2) MEDUSA_HEADS_BF16(2);
    else MEDUSA_HEADS_BF16(4);
#undef MEDUSA_HEADS_BF16
  } else {
    float* r = reinterpret_cast<float*>(base + p.xp2);
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
