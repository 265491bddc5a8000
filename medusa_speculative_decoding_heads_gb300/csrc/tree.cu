// Candidate tree (Cartesian, or pruned from a node list): layout, ancestor mask,
// tokens and position ids.
//
// "Medusa 심층 아키텍처" (techknowgenie), section "트리 어텐션": each head keeps its
// top-s candidates and the candidates of consecutive heads are combined into a
// tree (the page's example: top-2 x top-3 x top-2); the TreeMask equation makes
// node i see node j iff j is an ancestor of i or j = i.
//
// Node order: breadth first, lexicographic in the sibling-rank path. With
// cnt_d = prod_{j<=d} s_j and off_d = sum_{e<d} cnt_e, the node at depth d and
// level index t has parent off_{d-1} + t / s_d, rank t % s_d and first child
// off_{d+1} + t * s_{d+1}; its token is head d's candidate of that rank.
//
// A pruned tree (a subset of those nodes, given by each node's parent and
// rank in the same order; "Medusa 심층 아키텍처", sections "벤치마크 실측 지표"
// and "트리 크기(Tree Size)와 검증 오버헤드의 균형": trees of 32-64 nodes) takes
// its links from that list: depth from the parent chain, first child = the
// first later node whose parent it is.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace medusa {
namespace {

__device__ __forceinline__ int node_depth(const TreeShape& ts, int n) {
  int d = 0;
  while (d < ts.K && n >= ts.off[d + 1]) ++d;
  return d;
}

__device__ __forceinline__ int node_parent(const TreeShape& ts, int n) {
  if (n == 0) return -1;
  int d = node_depth(ts, n);
  int t = n - ts.off[d];
  return ts.off[d - 1] + t / ts.s[d];
}

// The pruned tree's node list (node n: parent and rank in its head's top-s list).
struct TreeNodes {
  int16_t parent[kMaxN];
  uint8_t rank[kMaxN];
};

__global__ void __launch_bounds__(kMaxN)
tree_build_kernel(TreeShape ts, TreeNodes tn, int B, int L_cap, int V, const int32_t* __restrict__ root,
                  const int32_t* __restrict__ topk,
                  const int32_t* __restrict__ L, int32_t* __restrict__ parent, int32_t* __restrict__ depth,
                  int32_t* __restrict__ first_child, uint8_t* __restrict__ mask, uint64_t* __restrict__ bits,
                  int32_t* __restrict__ tokens, int32_t* __restrict__ pos, uint32_t* __restrict__ flags) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint64_t sb[kMaxN][2];
  const int b = blockIdx.x;
  const int n = threadIdx.x;
  const int N = ts.N;
  const int Lb = L[b];
  if (n == 0 && flags) flags[b] = (Lb < 0 || Lb + N > L_cap) ? MEDUSA_FLAG_CAPACITY : 0u;
  // depth, parent, rank and first child of node n
  int d = 0, par = -1, rank = 0, fc = -1;
  if (n < N) {
    if (ts.pruned) {
      par = tn.parent[n];
      for (int j = par; j >= 0; j = tn.parent[j]) ++d;
      rank = n > 0 ? tn.rank[n] : 0;
      for (int c = n + 1; c < N && fc < 0; ++c)
        if (tn.parent[c] == n) fc = c;
    } else {
      d = node_depth(ts, n);
      const int t = n - ts.off[d];
      par = d > 0 ? ts.off[d - 1] + t / ts.s[d] : -1;
      rank = d > 0 ? t % ts.s[d] : 0;
      fc = d < ts.K ? ts.off[d + 1] + t * ts.s[d + 1] : -1;
    }
  }
  if (n < N) {
    const int tok = d == 0 ? root[b] : topk[((size_t)b * ts.K + (d - 1)) * ts.s_max + rank];
    MEDUSA_CHECK(tok >= 0 && tok < V, MEDUSA_CHECK_TOKEN);
    tokens[(size_t)b * N + n] = tok;
    pos[(size_t)b * N + n] = Lb + d;
  }
  if (b != 0) return;   // the tree arrays are the same for every sequence: block 0 writes them
  if (n < N) {
    parent[n] = par;
    depth[n] = d;
    first_child[n] = fc;
    uint64_t w0 = 0, w1 = 0;
    for (int j = n; j >= 0; j = ts.pruned ? (int)tn.parent[j] : node_parent(ts, j)) {
      if (j < 64) w0 |= 1ull << j;
      else w1 |= 1ull << (j - 64);
    }
    sb[n][0] = w0;
    sb[n][1] = w1;
    bits[2 * n] = w0;
    bits[2 * n + 1] = w1;
  }
  __syncthreads();
  // mask row-major N x N, written with consecutive threads on consecutive bytes
  for (int e = n; e < N * N; e += kMaxN) {
    const int i = e / N, j = e - i * N;
    mask[e] = uint8_t((sb[i][j >> 6] >> (j & 63)) & 1ull);
  }
}

}  // namespace

MEDUSA_CHECK_TAKE(tree_take_checks)

cudaError_t launch_tree_build(const medusa_cfg& c, const int32_t* root, const int32_t* topk, const int32_t* L,
                              int32_t* parent, int32_t* depth, int32_t* first_child, uint8_t* mask, uint64_t* bits,
                              int32_t* tokens, int32_t* pos, uint32_t* flags, cudaStream_t st) {
  const TreeShape ts = tree_shape(c);
  TreeNodes tn{};
  if (ts.pruned)
    for (int n = 0; n < ts.N; ++n) {
      tn.parent[n] = c.tree_parent[n];
      tn.rank[n] = c.tree_rank[n];
    }
  launch_pdl(tree_build_kernel, c.B, kMaxN, 0, st, ts, tn, c.B, c.L_cap, c.V, root, topk, L, parent, depth, first_child, mask,
             bits, tokens, pos, flags);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace medusa
