// KV compaction of the accepted path, in place; and its paged-cache form, which
// commits the accepted path's staged tree rows into the pages of every layer.
//
// "Speculative Decoding 원리와 가속 아키텍처" (blog.huny.dev), section 5 Case 2
// (rejected drafts are rolled back) and section 6 (the tree verification needs
// an extra KV buffer); "최적화 2편" (beengineer500), section 1.3 (everything
// after the first mismatch is dropped).
//
// For r = 0..acc_b: row L_b + r <- row L_b + path_r in every KV head, then
// L_b += acc_b + 1. path is strictly increasing with path_r >= r (node ids at
// depth r are at least r), so a destination r is never the source of a later
// slot. Each thread owns one 16-byte column slice of a (head, K or V) row set
// and loads every source slice before storing any, so the in-place update
// needs no barrier.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace medusa {
namespace {

__device__ __forceinline__ bool valid_walk(int Lb, int N, int L_cap, int a, int K) {
  return Lb >= 0 && Lb + N <= L_cap && a >= 0 && a <= K;
}

// Path slot r holds a node of the tree, the root at r = 0 and a deeper node
// than slot r - 1 after it (so node ids grow strictly and slot r's node is at
// least r, which the in-place move relies on).
__device__ __forceinline__ bool path_node_ok(const int32_t* pb, int r, int N) {
  const int s = pb[r];
  return s >= 0 && s < N && (r == 0 ? s == 0 : s > pb[r - 1]);
}

__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

constexpr int kCompactThreads = 256;
constexpr int kCompactCluster = 8;   // CTAs per sequence (portable cluster size)

// One cluster of ncta CTAs per sequence, grid (ncta, B): CTA r moves the K and
// V rows of KV heads [r Hkv / ncta, (r + 1) Hkv / ncta), one 16-byte column
// slice per thread and step. After a cluster barrier (so that every CTA has
// read L[b]), CTA 0 writes the KV map and advances L[b].
__global__ void __launch_bounds__(kCompactThreads)
kv_compact_kernel(uint4* __restrict__ Kc, uint4* __restrict__ Vc, int Hkv, int row_vec, int L_cap, int N, int K,
                  int32_t* __restrict__ L, const int32_t* __restrict__ acc, const int32_t* __restrict__ path,
                  int32_t* __restrict__ kv_map) {
  pdl_wait();
  pdl_trigger();
  const int rank = blockIdx.x, ncta = gridDim.x, b = blockIdx.y;
  const int Lb = L[b];
  const int a = acc[b];
  const bool ok = valid_walk(Lb, N, L_cap, a, K);
  const int32_t* pb = path + (size_t)b * (K + 1);
  MEDUSA_CHECK(!(Lb >= 0 && Lb + N <= L_cap) || (a >= 0 && a <= K), MEDUSA_CHECK_PATH);
  if (ok) {
    int src[kMaxK + 1];
#pragma unroll
    for (int r = 0; r <= kMaxK; ++r) {
      const int s = r <= a ? pb[r] : r;
      MEDUSA_CHECK(r > a || path_node_ok(pb, r, N), MEDUSA_CHECK_PATH);
      src[r] = s < 0 ? 0 : (s >= N ? N - 1 : s);
    }
    const int h0 = rank * Hkv / ncta, h1 = (rank + 1) * Hkv / ncta;
    const int items = (h1 - h0) * 2 * row_vec;   // (head, K or V, column)
    for (int i = threadIdx.x; i < items; i += kCompactThreads) {
      const int col = i % row_vec, hk = i / row_vec;
      uint4* base = ((hk & 1) ? Vc : Kc) + ((size_t)b * Hkv + h0 + (hk >> 1)) * L_cap * row_vec + col;
      uint4 v[kMaxK + 1];
#pragma unroll
      for (int r = 0; r <= kMaxK; ++r)
        if (r <= a) v[r] = base[(size_t)(Lb + src[r]) * row_vec];
#pragma unroll
      for (int r = 0; r <= kMaxK; ++r)
        if (r <= a && src[r] != r) base[(size_t)(Lb + r) * row_vec] = v[r];
    }
  }
  cluster_barrier();
  if (rank == 0) {
    for (int r = threadIdx.x; r <= K; r += kCompactThreads)
      kv_map[(size_t)b * (K + 1) + r] = (ok && r <= a) ? pb[r] : -1;
    if (threadIdx.x == 0 && ok) L[b] = Lb + a + 1;
  }
}

// Paged cache, every layer: logical row L_b + r (r = 0..acc_b) of sequence b
// receives the staged tree row path[b][r]; grid (ncta, B) in clusters of ncta
// CTAs per sequence, CTA `rank` taking (layer, KV head) pairs rank, rank + ncta,
// ... with one 16-byte column slice per thread and step. Sources (staging) and
// destinations (pages) never overlap, so no ordering is needed beyond the
// cluster barrier before CTA 0 writes the KV map and advances L_b.
__global__ void __launch_bounds__(kCompactThreads)
kv_commit_paged_kernel(uint4* __restrict__ Kp, uint4* __restrict__ Vp, const uint4* __restrict__ Kt,
                       const uint4* __restrict__ Vt, const int32_t* __restrict__ block_table, int max_pages,
                       int num_pages, int page_rows, int n_layers, size_t pool_layer_vec, size_t tree_layer_vec,
                       int Hkv, int row_vec,
                       int N, int K, int32_t* __restrict__ L, const int32_t* __restrict__ acc,
                       const int32_t* __restrict__ path, int32_t* __restrict__ kv_map) {
  pdl_wait();
  pdl_trigger();
  const int rank = blockIdx.x, ncta = gridDim.x, b = blockIdx.y;
  const int Lb = L[b];
  const int a = acc[b];
  const bool ok = Lb >= 0 && Lb + N <= max_pages * page_rows && a >= 0 && a <= K;
  const int32_t* pb = path + (size_t)b * (K + 1);
  MEDUSA_CHECK(!(Lb >= 0 && Lb + N <= max_pages * page_rows) || (a >= 0 && a <= K), MEDUSA_CHECK_PATH);
  if (ok) {
    int src[kMaxK + 1];
    size_t dst[kMaxK + 1];   // pool row of logical row Lb + r, before the head offset
    bool live[kMaxK + 1];    // r <= acc and the row's page lies inside the pool
#pragma unroll
    for (int r = 0; r <= kMaxK; ++r) {
      const int sr = r <= a ? pb[r] : 0;
      MEDUSA_CHECK(r > a || path_node_ok(pb, r, N), MEDUSA_CHECK_PATH);
      src[r] = sr < 0 ? 0 : (sr >= N ? N - 1 : sr);
      const int row = Lb + (r <= a ? r : 0);
      const int page = block_table[(size_t)b * max_pages + row / page_rows];
      const bool in_pool = page >= 0 && page < num_pages;
      MEDUSA_CHECK(r > a || in_pool, MEDUSA_CHECK_PAGE);
      live[r] = r <= a && in_pool;   // a page id outside the pool: that row is not written
      dst[r] = (size_t)(in_pool ? page : 0) * Hkv * page_rows + row % page_rows;
    }
    const int pairs = n_layers * Hkv * 2;              // (layer, head, K or V)
    for (int i = rank * kCompactThreads + threadIdx.x; i < pairs * row_vec; i += ncta * kCompactThreads) {
      const int col = i % row_vec, pr = i / row_vec;
      const int kv = pr & 1, h = (pr >> 1) % Hkv, layer = (pr >> 1) / Hkv;
      const uint4* sbase = (kv ? Vt : Kt) + layer * tree_layer_vec + ((size_t)b * Hkv + h) * N * row_vec + col;
      uint4* dbase = (kv ? Vp : Kp) + layer * pool_layer_vec + (size_t)h * page_rows * row_vec + col;
#pragma unroll
      for (int r = 0; r <= kMaxK; ++r)
        if (live[r]) dbase[dst[r] * row_vec] = sbase[(size_t)src[r] * row_vec];
    }
  }
  cluster_barrier();
  if (rank == 0) {
    for (int r = threadIdx.x; r <= K; r += kCompactThreads)
      kv_map[(size_t)b * (K + 1) + r] = (ok && r <= a) ? pb[r] : -1;
    if (threadIdx.x == 0 && ok) L[b] = Lb + a + 1;
  }
}

}  // namespace

MEDUSA_CHECK_TAKE(compact_take_checks)

cudaError_t launch_kv_compact(const medusa_cfg& c, void* Kc, void* Vc, int32_t* L, const int32_t* acc,
                              const int32_t* path, int32_t* kv_map, cudaStream_t st) {
  const TreeShape ts = tree_shape(c);
  const int elt = c.dtype == MEDUSA_F32 ? 4 : 2;
  const int row_vec = c.D * elt / 16;
  const int ncta = c.Hkv < kCompactCluster ? c.Hkv : kCompactCluster;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ncta, c.B);
  cfg.blockDim = dim3(kCompactThreads);
  cfg.dynamicSmemBytes = 0;
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, kv_compact_kernel, static_cast<uint4*>(Kc), static_cast<uint4*>(Vc), c.Hkv,
                                     row_vec, c.L_cap, ts.N, c.K, L, acc, path, kv_map);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_kv_commit_paged(const medusa_cfg& c, void* Kp, void* Vp, const PagedKV& pg, int n_layers,
                                   size_t pool_layer_elems, size_t tree_layer_elems, int32_t* L, const int32_t* acc,
                                   const int32_t* path, int32_t* kv_map, cudaStream_t st) {
  const TreeShape ts = tree_shape(c);
  const int elt = c.dtype == MEDUSA_F32 ? 4 : 2;
  const int row_vec = c.D * elt / 16;
  const int per16 = 16 / elt;   // elements per 16-byte vector
  const int work = n_layers * c.Hkv * 2;
  const int ncta = work < kCompactCluster ? work : kCompactCluster;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ncta, c.B);
  cfg.blockDim = dim3(kCompactThreads);
  cfg.dynamicSmemBytes = 0;
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, kv_commit_paged_kernel, static_cast<uint4*>(Kp), static_cast<uint4*>(Vp),
                                     static_cast<const uint4*>(pg.Kt), static_cast<const uint4*>(pg.Vt), pg.block_table,
                                     c.L_cap / pg.page_rows, pg.num_pages, pg.page_rows, n_layers, pool_layer_elems / per16,
                                     tree_layer_elems / per16, c.Hkv, row_vec, ts.N, c.K, L, acc, path, kv_map);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace medusa
