// KV compaction of the accepted path, in place.
//
// "Speculative Decoding 원리와 가속 아키텍처" (blog.huny.dev), section 5 Case 2
// (rejected drafts are rolled back) and section 6 (the tree verification needs
// an extra KV buffer); "최적화 2편" (beengineer500), section 1.3 (everything
// after the first mismatch is dropped).
//
// For r = 0..acc_b: row L_b + r <- row L_b + path_r in every KV head, then
// L_b += acc_b + 1. path is strictly increasing with path_r >= r (node ids at
// depth r are at least r), so a destination r is never the source of a later
// slot. Each lane owns one fixed 16-byte column slice of a row and loads every
// source slice before storing any, so the in-place update needs no barrier.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace medusa {
namespace {

__device__ __forceinline__ bool valid_walk(int Lb, int N, int L_cap, int a, int K) {
  return Lb >= 0 && Lb + N <= L_cap && a >= 0 && a <= K;
}

// grid (Hkv, B), block 64: warp 0 moves K rows, warp 1 moves V rows.
__global__ void __launch_bounds__(64)
kv_compact_kernel(uint4* __restrict__ Kc, uint4* __restrict__ Vc, int row_vec, int L_cap, int N, int K,
                  const int32_t* __restrict__ L, const int32_t* __restrict__ acc, const int32_t* __restrict__ path) {
  pdl_wait();
  pdl_trigger();
  const int h = blockIdx.x, b = blockIdx.y, Hkv = gridDim.x;
  const int Lb = L[b];
  const int a = acc[b];
  if (!valid_walk(Lb, N, L_cap, a, K)) return;
  uint4* base = (threadIdx.x < 32 ? Kc : Vc) + ((size_t)b * Hkv + h) * L_cap * row_vec;
  const int32_t* pb = path + (size_t)b * (K + 1);
  for (int col = threadIdx.x & 31; col < row_vec; col += 32) {
    uint4 v[kMaxK + 1];
#pragma unroll
    for (int r = 0; r <= kMaxK; ++r) {
      if (r > a) break;
      int src = pb[r];
      src = src < 0 ? 0 : (src >= N ? N - 1 : src);
      v[r] = base[(size_t)(Lb + src) * row_vec + col];
    }
#pragma unroll
    for (int r = 0; r <= kMaxK; ++r) {
      if (r > a) break;
      if (pb[r] != r) base[(size_t)(Lb + r) * row_vec + col] = v[r];
    }
  }
}

__global__ void kv_finish_kernel(int B, int N, int K, int L_cap, int32_t* __restrict__ L, const int32_t* __restrict__ acc,
                                 const int32_t* __restrict__ path, int32_t* __restrict__ kv_map) {
  pdl_wait();
  pdl_trigger();
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += gridDim.x * blockDim.x) {
    const int Lb = L[b];
    const int a = acc[b];
    const bool ok = valid_walk(Lb, N, L_cap, a, K);
    for (int r = 0; r <= K; ++r) kv_map[(size_t)b * (K + 1) + r] = (ok && r <= a) ? path[(size_t)b * (K + 1) + r] : -1;
    if (ok) L[b] = Lb + a + 1;
  }
}

}  // namespace

cudaError_t launch_kv_compact(const medusa_cfg& c, void* Kc, void* Vc, int32_t* L, const int32_t* acc,
                              const int32_t* path, int32_t* kv_map, cudaStream_t st) {
  const TreeShape ts = tree_shape(c);
  const int elt = c.dtype == MEDUSA_F32 ? 4 : 2;
  const int row_vec = c.D * elt / 16;
  launch_pdl(kv_compact_kernel, dim3(c.Hkv, c.B), 64, 0, st, static_cast<uint4*>(Kc), static_cast<uint4*>(Vc), row_vec,
                                                      c.L_cap, ts.N, c.K, L, acc, path);
  note_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  launch_pdl(kv_finish_kernel, (c.B + 127) / 128, 128, 0, st, c.B, ts.N, c.K, c.L_cap, L, acc, path, kv_map);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace medusa
