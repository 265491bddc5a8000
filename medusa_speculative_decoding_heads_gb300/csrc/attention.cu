// Tree attention: every tree node attends to the committed KV cache plus its
// own ancestors, all nodes in one pass.
//
// "Medusa 심층 아키텍처" (techknowgenie), section "트리 어텐션": the TreeMask
// equation and the statement that all tree tokens are evaluated in one pass
// without branches seeing each other. Block-wise partial softmax results are
// merged with the running maximum and exp-sum ("최적화 2편" (beengineer500),
// section 3.3: the online-softmax property that makes block-wise partials
// exact), which lets the committed prefix be split across CTAs.
//
// bf16 with D = 128 takes the tcgen05 kernel (attention_tc.cu, which also reads
// a paged cache through a block table), bf16 with D = 64 the mma.sync kernel
// (attention_mma.cu). This file holds the float32 kernel (CUDA cores, float32
// softmax and accumulation), the split plan and the merge: grid (query-row
// groups, KV head x sequence, KV split). The committed prefix is unmasked; the
// last split also visits the N tree rows, where the ancestor bitmask is applied
// in registers.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace medusa {
namespace {

constexpr int kAttnWarps = 8;
constexpr int kRowsPerWarp = 2;
constexpr int kRowsPerCta = kAttnWarps * kRowsPerWarp;
constexpr int kKeyTile = 32;

struct AttnPlan {
  int G, NG, row_groups, nsplit, chunk;
  size_t o_part, ml_part, x_part, total;
};

// Kernel choice: float32 -> CUDA cores; bf16 with D = 128 -> tcgen05; bf16 with D = 64 -> mma.sync.
enum AttnPath { kPathF32 = 0, kPathMma = 1, kPathTc = 2 };

int attention_path(const medusa_cfg& c) {
  if (c.dtype == MEDUSA_F32) return kPathF32;
  return c.D == 128 ? kPathTc : kPathMma;
}

AttnPlan plan_attention(const medusa_cfg& c) {
  AttnPlan p{};
  const TreeShape ts = tree_shape(c);
  p.G = c.Hq / c.Hkv;
  p.NG = ts.N * p.G;
  const int path = attention_path(c);
  int tile = kKeyTile;
  if (path == kPathTc) {
    p.row_groups = attention_tc_ctas_x(p.NG);
    tile = 128;
  } else if (path == kPathMma) {
    attention_mma_warps(p.NG, &p.row_groups);
    tile = 64;
  } else {
    p.row_groups = (p.NG + kRowsPerCta - 1) / kRowsPerCta;
  }
  const int Lmax = c.L_cap - ts.N;   // longest committed prefix that fits
  // Split the KV range only while the whole grid still fits one wave (one CTA
  // per SM): every CTA pays a pipeline fill and an epilogue, and splits add a
  // merge pass, so beyond one wave more splits cost more than they balance.
  const long ctas = (long)p.row_groups * c.Hkv * c.B;
  int want = (int)(152 / ctas);
  int by_len = (Lmax + 255) / 256;
  p.nsplit = want < by_len ? want : by_len;
  if (p.nsplit > 32) p.nsplit = 32;   // the merge gives one lane per split
  if (p.nsplit < 1) p.nsplit = 1;
  p.chunk = Lmax > 0 ? ((Lmax + p.nsplit - 1) / p.nsplit + tile - 1) / tile * tile : tile;
  const size_t rows = (size_t)c.B * p.nsplit * ts.N * c.Hq;
  size_t off = 0;
  p.o_part = off;
  off = align_up(off + rows * c.D * 4, 256);
  p.ml_part = off;
  off = align_up(off + rows * 2 * 4, 256);
  p.x_part = off;   // leftover rows' partials (tcgen05 path with a short remainder of query rows)
  off = align_up(off + (path == kPathTc ? attention_tc_xpart_bytes(c, p.nsplit) : 0), 256);
  p.total = off;
  return p;
}

// Partial results for query row (b, split, node i, q head h): unnormalised O,
// running max m (log2 domain) and exp-sum l.
template <typename T, int D>
__global__ void __launch_bounds__(kAttnWarps * 32)
tree_attn_partial_kernel(const T* __restrict__ Q, const T* __restrict__ Kc, const T* __restrict__ Vc,
                         const int32_t* __restrict__ L, const uint64_t* __restrict__ bits, int N, int Hq, int Hkv,
                         int L_cap, int chunk, float scale_log2, float* __restrict__ o_part,
                         float* __restrict__ ml_part) {
  pdl_wait();
  pdl_trigger();
  constexpr int DPL = D / 32;   // head-dim values per lane
  __shared__ float qs[kRowsPerCta][D];
  __shared__ float ks[kKeyTile][D + 1];
  __shared__ float vs[kKeyTile][D];
  const int G = Hq / Hkv;
  const int NG = N * G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.y % Hkv, b = blockIdx.y / Hkv;
  const int split = blockIdx.z, nsplit = gridDim.z;
  const int Lb = L[b];
  const bool valid = Lb >= 0 && Lb + N <= L_cap;

  // Query rows of this CTA: qi = node * G + g  ->  head kvh * G + g
  for (int e = threadIdx.x; e < kRowsPerCta * D; e += blockDim.x) {
    int r = e / D, dd = e % D;
    int qi = blockIdx.x * kRowsPerCta + r;
    float v = 0.f;
    if (qi < NG) {
      int node = qi / G, h = kvh * G + qi % G;
      v = Elt<T>::load(Q, (((size_t)b * N + node) * Hq + h) * D + dd) * scale_log2;
    }
    qs[r][dd] = v;
  }

  float m[kRowsPerWarp], l[kRowsPerWarp], o[kRowsPerWarp][DPL];
  uint64_t rb0[kRowsPerWarp], rb1[kRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) o[r][j] = 0.f;
    int qi = blockIdx.x * kRowsPerCta + warp * kRowsPerWarp + r;
    int node = qi < NG ? qi / G : 0;
    rb0[r] = bits[2 * node];
    rb1[r] = bits[2 * node + 1];
  }

  const size_t head_base = ((size_t)b * Hkv + kvh) * L_cap;
  const int k_begin = split * chunk;
  const int k_end = valid ? min(Lb, k_begin + chunk) : 0;
  const int tree_tiles = (valid && split == nsplit - 1) ? (N + kKeyTile - 1) / kKeyTile : 0;
  const int prefix_tiles = k_end > k_begin ? (k_end - k_begin + kKeyTile - 1) / kKeyTile : 0;

  for (int tile = 0; tile < prefix_tiles + tree_tiles; ++tile) {
    const bool is_tree = tile >= prefix_tiles;
    const int key0 = is_tree ? (tile - prefix_tiles) * kKeyTile : k_begin + tile * kKeyTile;   // tree: node index
    const int nkeys = is_tree ? min(kKeyTile, N - key0) : min(kKeyTile, k_end - key0);
    __syncthreads();
    for (int e = threadIdx.x; e < kKeyTile * D; e += blockDim.x) {
      int j = e / D, dd = e % D;
      float kv = 0.f, vv = 0.f;
      if (j < nkeys) {
        size_t row = head_base + (is_tree ? (size_t)Lb + key0 + j : (size_t)key0 + j);
        kv = Elt<T>::load(Kc, row * D + dd);
        vv = Elt<T>::load(Vc, row * D + dd);
      }
      ks[j][dd] = kv;
      vs[j][dd] = vv;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int rloc = warp * kRowsPerWarp + r;
      float s = 0.f;
#pragma unroll 8
      for (int dd = 0; dd < D; ++dd) s = fmaf(qs[rloc][dd], ks[lane][dd], s);
      bool vis = lane < nkeys;
      if (is_tree && vis) {
        int j = key0 + lane;
        uint64_t w = j < 64 ? rb0[r] : rb1[r];
        vis = (w >> (j & 63)) & 1ull;
      }
      s = vis ? s : -INFINITY;
      float mt = warp_max(s);
      if (mt == -INFINITY) continue;
      float mn = fmaxf(m[r], mt);
      float corr = exp2f(m[r] - mn);
      float pj = vis ? exp2f(s - mn) : 0.f;
      l[r] = l[r] * corr + warp_sum(pj);
#pragma unroll
      for (int j = 0; j < DPL; ++j) o[r][j] *= corr;
      for (int j = 0; j < kKeyTile; ++j) {
        float pb = __shfl_sync(0xffffffffu, pj, j);
#pragma unroll
        for (int jj = 0; jj < DPL; ++jj) o[r][jj] = fmaf(pb, vs[j][lane + 32 * jj], o[r][jj]);
      }
      m[r] = mn;
    }
  }

#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    int qi = blockIdx.x * kRowsPerCta + warp * kRowsPerWarp + r;
    if (qi >= NG) continue;
    int node = qi / G, h = kvh * G + qi % G;
    size_t row = (((size_t)b * nsplit + split) * N + node) * Hq + h;
#pragma unroll
    for (int j = 0; j < DPL; ++j) o_part[row * D + lane + 32 * j] = o[r][j];
    if (lane == 0) {
      ml_part[2 * row] = m[r];
      ml_part[2 * row + 1] = l[r];
    }
  }
}

// O[b][i][h] = sum_s O_s 2^(m_s - M) / sum_s l_s 2^(m_s - M); one warp per output
// row, lane s holds split s's (m, l) (nsplit <= 32).
template <typename T, int D>
__global__ void tree_attn_merge_kernel(const float* __restrict__ o_part, const float* __restrict__ ml_part, int B,
                                       int N, int Hq, int nsplit, const int32_t* __restrict__ L, int L_cap,
                                       T* __restrict__ O) {
  pdl_wait();
  pdl_trigger();
  const size_t rows = (size_t)B * N * Hq;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if ((size_t)warp >= rows) return;
  const int h = warp % Hq;
  const int node = (warp / Hq) % N;
  const int b = warp / (Hq * N);
  const int Lb = L[b];
  const bool valid = Lb >= 0 && Lb + N <= L_cap;
  const size_t split_stride = (size_t)N * Hq;
  const size_t row0 = ((size_t)b * nsplit * N + node) * Hq + h;   // split 0's partial row
  float ms = -INFINITY, ls = 0.f;
  if (lane < nsplit) {
    ms = ml_part[2 * (row0 + lane * split_stride)];
    ls = ml_part[2 * (row0 + lane * split_stride) + 1];
  }
  const float M = warp_max(ms);
  const float w = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
  const float lsum = warp_sum(ls * w);
  float acc[D / 32];
#pragma unroll
  for (int j = 0; j < D / 32; ++j) acc[j] = 0.f;
#pragma unroll 4
  for (int s = 0; s < nsplit; ++s) {
    const float ws = __shfl_sync(0xffffffffu, w, s);
    if (ws == 0.f) continue;   // an empty split need not have written its partial O
    const float* op = o_part + (row0 + s * split_stride) * D;
#pragma unroll
    for (int j = 0; j < D / 32; ++j) acc[j] += op[lane + 32 * j] * ws;
  }
  const size_t out = (((size_t)b * N + node) * Hq + h) * D;
#pragma unroll
  for (int j = 0; j < D / 32; ++j) Elt<T>::store(O, out + lane + 32 * j, (valid && lsum > 0.f) ? acc[j] / lsum : 0.f);
}

template <typename T, int D>
cudaError_t run(const medusa_cfg& c, const AttnPlan& p, const void* Q, const void* Kc, const void* Vc,
                const int32_t* L, const uint64_t* bits, void* O, char* ws, cudaStream_t st, const PagedKV* paged) {
  const TreeShape ts = tree_shape(c);
  float* o_part = reinterpret_cast<float*>(ws + p.o_part);
  float* ml_part = reinterpret_cast<float*>(ws + p.ml_part);
  cudaError_t e;
  const int path = attention_path(c);
  float* x_part = reinterpret_cast<float*>(ws + p.x_part);
  if (path == kPathTc) {
    e = launch_attention_tc(c, p.nsplit, p.chunk, Q, Kc, Vc, L, bits, o_part, ml_part, x_part, O, st, paged);
    if (e == cudaSuccess && p.nsplit == 1) e = launch_attention_tc_xmerge(c, 1, x_part, L, O, st);
    if (e != cudaSuccess || p.nsplit == 1) return e;   // a single split writes O itself (leftover rows merged)
  } else if (path == kPathMma) {
    e = launch_attention_mma(c, p.nsplit, p.chunk, Q, Kc, Vc, L, bits, o_part, ml_part, st);
  } else {
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)D));
    dim3 grid(p.row_groups, c.Hkv * c.B, p.nsplit);
    launch_pdl(tree_attn_partial_kernel<T, D>, grid, kAttnWarps * 32, 0, st, 
        static_cast<const T*>(Q), static_cast<const T*>(Kc), static_cast<const T*>(Vc), L, bits, ts.N, c.Hq, c.Hkv,
        c.L_cap, p.chunk, scale_log2, o_part, ml_part);
    note_launches(1);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  const size_t rows = (size_t)c.B * ts.N * c.Hq;
  launch_pdl(tree_attn_merge_kernel<T, D>, (unsigned)((rows * 32 + 255) / 256), 256, 0, st, 
      o_part, ml_part, c.B, ts.N, c.Hq, p.nsplit, L, c.L_cap, static_cast<T*>(O));
  note_launches(1);
  e = cudaGetLastError();
  if (e == cudaSuccess && path == kPathTc) e = launch_attention_tc_xmerge(c, p.nsplit, x_part, L, O, st);
  return e;
}

}  // namespace

size_t attention_workspace(const medusa_cfg& c) { return plan_attention(c).total; }

cudaError_t launch_attention(const medusa_cfg& c, const void* Q, const void* Kc, const void* Vc, const int32_t* L,
                             const uint64_t* bits, void* O, void* ws, cudaStream_t st, const PagedKV* paged) {
  const AttnPlan p = plan_attention(c);
  char* w = static_cast<char*>(ws);
  if (paged && attention_path(c) != kPathTc) return cudaErrorNotSupported;   // paged: the tcgen05 kernel only
  if (c.dtype == MEDUSA_F32) {
    return c.D == 64 ? run<float, 64>(c, p, Q, Kc, Vc, L, bits, O, w, st, paged)
                     : run<float, 128>(c, p, Q, Kc, Vc, L, bits, O, w, st, paged);
  }
  return c.D == 64 ? run<uint16_t, 64>(c, p, Q, Kc, Vc, L, bits, O, w, st, paged)
                   : run<uint16_t, 128>(c, p, Q, Kc, Vc, L, bits, O, w, st, paged);
}

}  // namespace medusa
