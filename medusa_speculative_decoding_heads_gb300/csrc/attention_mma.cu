// Stand-alone launch of the mma.sync tree attention (bf16 with D = 64; the unit
// itself is in attention_mma_unit.cuh, shared with the persistent step kernel).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attention_mma_unit.cuh"
#include "common.cuh"

namespace medusa {
namespace {

using mma_attn::kKeys;
using mma_attn::kMaxWarps;
using mma_attn::kStages;

template <int D>
__global__ void __launch_bounds__(kMaxWarps * 32)
tree_attn_mma_kernel(const uint16_t* __restrict__ Q, const uint16_t* __restrict__ Kc, const uint16_t* __restrict__ Vc,
                     const int32_t* __restrict__ L, const uint64_t* __restrict__ bits, int N, int Hq, int Hkv,
                     int L_cap, int chunk, float scale_log2, float* __restrict__ o_part, float* __restrict__ ml_part) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smem[];
  mma_attn::tree_attn_mma_unit<D>(Q, Kc, Vc, L, bits, N, Hq, Hkv, L_cap, chunk, scale_log2, o_part, ml_part,
                                  blockIdx.x, blockIdx.y, blockIdx.z, gridDim.z, smem);
}

}  // namespace

// Shared-memory bytes and CTA shape of the tensor-core path.
int attention_mma_warps(int NG, int* row_blocks) {
  const int mtiles = (NG + 15) / 16;
  int rb = (mtiles + kMaxWarps - 1) / kMaxWarps;
  *row_blocks = rb;
  return (mtiles + rb - 1) / rb;
}

cudaError_t launch_attention_mma(const medusa_cfg& c, int nsplit, int chunk, const void* Q, const void* Kc,
                                 const void* Vc, const int32_t* L, const uint64_t* bits, float* o_part, float* ml_part,
                                 cudaStream_t st) {
  const TreeShape ts = tree_shape(c);
  const int G = c.Hq / c.Hkv;
  int rb = 1;
  const int warps = attention_mma_warps(ts.N * G, &rb);
  const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)c.D));
  dim3 grid(rb, c.Hkv * c.B, nsplit);
  cudaError_t e;
  if (c.D == 128) {
    const size_t smem = 2 * kStages * kKeys * 128 * 2;
    e = cudaFuncSetAttribute(tree_attn_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    launch_pdl(tree_attn_mma_kernel<128>, grid, warps * 32, smem, st, 
        static_cast<const uint16_t*>(Q), static_cast<const uint16_t*>(Kc), static_cast<const uint16_t*>(Vc), L, bits,
        ts.N, c.Hq, c.Hkv, c.L_cap, chunk, scale_log2, o_part, ml_part);
  } else {
    const size_t smem = 2 * kStages * kKeys * 64 * 2;
    e = cudaFuncSetAttribute(tree_attn_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    launch_pdl(tree_attn_mma_kernel<64>, grid, warps * 32, smem, st, 
        static_cast<const uint16_t*>(Q), static_cast<const uint16_t*>(Kc), static_cast<const uint16_t*>(Vc), L, bits,
        ts.N, c.Hq, c.Hkv, c.L_cap, chunk, scale_log2, o_part, ml_part);
  }
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace medusa
