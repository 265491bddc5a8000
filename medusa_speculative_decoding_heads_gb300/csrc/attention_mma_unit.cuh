// Tree attention on legacy tensor cores (mma.sync m16n8k16, bf16 inputs, float32
// softmax and accumulation) as a device-side work unit, shared by the stand-alone
// kernel of attention_mma.cu and the persistent step kernel of fused.cu.
//
// "Medusa 심층 아키텍처" (techknowgenie), section "트리 어텐션": every tree node
// attends to the committed cache plus its ancestors (TreeMask equation), all
// nodes in one pass; block-wise partial softmax results merge exactly through
// the running maximum and exp-sum ("최적화 2편" (beengineer500), section 3.3).
//
// All N x G query rows that share one KV head (G = Hq / Hkv) go through the same
// K/V tiles, so each tile is fetched once per unit and reused by every tree node
// and every query head of the group. Each warp owns 16 query rows:
//   S = Q K^T  (Q fragments in registers, K tile via ldmatrix)
//   online softmax on the S fragments (exp2, row max / sum over the lane quad)
//   O += P V   (P re-packed from the S accumulators, V tile via ldmatrix.trans)
// K/V tiles of 64 keys are staged in shared memory by cp.async in a 3-deep ring
// with a 16-byte-chunk XOR swizzle (conflict-free ldmatrix). The committed
// prefix is unmasked; the tree keys (rows L_b .. L_b+N-1) come last and use the
// ancestor bitmask of each row's node.
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace medusa {
namespace mma_attn {

constexpr int kKeys = 64;      // keys per tile
constexpr int kStages = 3;
constexpr int kMaxWarps = 12;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  return uint32_t(f32_to_bf16(lo)) | (uint32_t(f32_to_bf16(hi)) << 16);
}

// Byte offset of 16-byte chunk c of tile row r (row = D bf16).
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return uint32_t(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

// One work unit of the tensor-core tree attention: row block `rbx` of the N x G query
// rows of (sequence, KV head) y = b * Hkv + kvh against KV range `split` of `nsplit`,
// with every warp of the CTA taking 16 query rows (rows past N x G are computed on
// zeros and not written). `smem` holds 2 * kStages * 64 * D * 2 bytes; the unit begins
// and ends with the CTA synchronised and no copy in flight.
template <int D>
__device__ __forceinline__ void tree_attn_mma_unit(const uint16_t* __restrict__ Q, const uint16_t* __restrict__ Kc,
                                                   const uint16_t* __restrict__ Vc, const int32_t* __restrict__ L,
                                                   const uint64_t* __restrict__ bits, int N, int Hq, int Hkv, int L_cap,
                                                   int chunk, float scale_log2, float* __restrict__ o_part,
                                                   float* __restrict__ ml_part, int rbx, int y, int split, int nsplit,
                                                   uint8_t* smem) {
  constexpr int KS = D / 16;        // k-steps of Q K^T
  constexpr int NT = D / 8;         // n-tiles of P V
  constexpr int CH = D / 8;         // 16-byte chunks per row
  constexpr int TILE_BYTES = kKeys * D * 2;
  uint8_t* ks_base = smem;                               // [stage][K tile]
  uint8_t* vs_base = smem + kStages * TILE_BYTES;        // [stage][V tile]

  const int warps = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = Hq / Hkv, NG = N * G;
  const int kvh = y % Hkv, b = y / Hkv;
  const int Lb = L[b];
  const bool valid = Lb >= 0 && Lb + N <= L_cap;

  const int row0 = (rbx * warps + warp) * 16;            // first query row of this warp
  int qrow[2], qnode[2];
  uint64_t mb0[2], mb1[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    qrow[i] = row0 + g + 8 * i;
    qnode[i] = qrow[i] < NG ? qrow[i] / G : 0;
    mb0[i] = bits[2 * qnode[i]];
    mb1[i] = bits[2 * qnode[i] + 1];
  }

  // Q fragments (A operand) straight from global memory.
  uint32_t qa[KS][4];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool ok = qrow[i] < NG;
    const uint16_t* qp = Q + (((size_t)b * N + qnode[i]) * Hq + (kvh * G + (ok ? qrow[i] % G : 0))) * D;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint32_t lo = ok ? *reinterpret_cast<const uint32_t*>(qp + 16 * kk + 2 * t) : 0u;
      uint32_t hi = ok ? *reinterpret_cast<const uint32_t*>(qp + 16 * kk + 8 + 2 * t) : 0u;
      qa[kk][i] = lo;       // a0 (row g) / a1 (row g+8)
      qa[kk][2 + i] = hi;   // a2 / a3
    }
  }

  const size_t head_base = ((size_t)b * Hkv + kvh) * L_cap;
  const int k_begin = split * chunk;
  const int k_end = valid ? min(Lb, k_begin + chunk) : 0;
  const int ptiles = k_end > k_begin ? (k_end - k_begin + kKeys - 1) / kKeys : 0;
  const int ttiles = (valid && split == nsplit - 1) ? (N + kKeys - 1) / kKeys : 0;
  const int ntiles = ptiles + ttiles;

  // Tile j: first cache row and number of valid keys.
  auto tile_src = [&](int j, int& first, int& nkeys, bool& tree) {
    tree = j >= ptiles;
    if (!tree) {
      first = k_begin + j * kKeys;
      nkeys = min(kKeys, k_end - first);
    } else {
      const int j0 = (j - ptiles) * kKeys;
      first = Lb + j0;
      nkeys = min(kKeys, N - j0);
    }
  };
  auto load_tile = [&](int j, int stage) {
    int first, nkeys;
    bool tree;
    tile_src(j, first, nkeys, tree);
    const uint32_t kd = smem_u32(ks_base + stage * TILE_BYTES);
    const uint32_t vd = smem_u32(vs_base + stage * TILE_BYTES);
    for (int e = threadIdx.x; e < kKeys * CH; e += blockDim.x) {
      const int r = e / CH, c = e % CH;
      const bool ok = r < nkeys;
      const size_t row = head_base + (size_t)(ok ? first + r : first);
      cp_async16_zfill(kd + swz<D>(r, c), Kc + row * D + c * 8, ok);
      cp_async16_zfill(vd + swz<D>(r, c), Vc + row * D + c * 8, ok);
    }
  };

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < ntiles) load_tile(s, s);
    cp_commit();
  }

  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int i = 0; i < 4; ++i) o[n][i] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};

  for (int j = 0; j < ntiles; ++j) {
    if (j + kStages - 1 < ntiles) load_tile(j + kStages - 1, (j + kStages - 1) % kStages);
    cp_commit();
    cp_wait<kStages - 1>();
    __syncthreads();
    const int stage = j % kStages;
    const uint32_t kt = smem_u32(ks_base + stage * TILE_BYTES);
    const uint32_t vt = smem_u32(vs_base + stage * TILE_BYTES);
    int first, nkeys;
    bool tree;
    tile_src(j, first, nkeys, tree);
    const int key_off = tree ? first - Lb : 0;   // tree node index of key 0 of the tile

    // S = Q K^T for 64 keys: 8 n-tiles of 8 keys.
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) s[n][i] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
      for (int p = 0; p < 4; ++p) {     // key pairs of n-tiles (16 keys)
        const int key = 16 * p + ((lane >> 4) << 3) + (lane & 7);
        const int chk = 2 * kk + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kt + swz<D>(key, chk), b0, b1, b2, b3);
        mma16816(s[2 * p], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
        mma16816(s[2 * p + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
      }
    }

    // Mask, scale, online softmax.
    float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = i >> 1;
        const int key = 8 * n + 2 * t + (i & 1);
        bool vis = key < nkeys;
        if (tree && vis) {
          const int jn = key_off + key;
          const uint64_t w = jn < 64 ? mb0[r] : mb1[r];
          vis = (w >> (jn & 63)) & 1ull;
        }
        const float v = vis ? s[n][i] * scale_log2 : -INFINITY;
        s[n][i] = v;
        mt[r] = fmaxf(mt[r], v);
      }
    float corr[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mt[r] = fmaxf(mt[r], __shfl_xor_sync(0xffffffffu, mt[r], 1));
      mt[r] = fmaxf(mt[r], __shfl_xor_sync(0xffffffffu, mt[r], 2));
      const float mn = fmaxf(m_run[r], mt[r]);
      const float muse = mn == -INFINITY ? 0.f : mn;
      corr[r] = exp2f(m_run[r] - muse);
      m_run[r] = mn;
      mt[r] = muse;
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float p = exp2f(s[n][i] - mt[i >> 1]);
        s[n][i] = p;
        rs[i >> 1] += p;
      }
#pragma unroll
    for (int r = 0; r < 2; ++r) l_run[r] = l_run[r] * corr[r] + rs[r];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      o[n][0] *= corr[0];
      o[n][1] *= corr[0];
      o[n][2] *= corr[1];
      o[n][3] *= corr[1];
    }

    // O += P V: 4 k-steps of 16 keys.
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint32_t a0 = pack_bf16(s[2 * ks][0], s[2 * ks][1]);
      const uint32_t a1 = pack_bf16(s[2 * ks][2], s[2 * ks][3]);
      const uint32_t a2 = pack_bf16(s[2 * ks + 1][0], s[2 * ks + 1][1]);
      const uint32_t a3 = pack_bf16(s[2 * ks + 1][2], s[2 * ks + 1][3]);
#pragma unroll
      for (int q = 0; q < NT / 2; ++q) {
        const int key = 16 * ks + (((lane >> 3) & 1) << 3) + (lane & 7);
        const int chk = 2 * q + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vt + swz<D>(key, chk), b0, b1, b2, b3);
        mma16816(o[2 * q], a0, a1, a2, a3, b0, b1);
        mma16816(o[2 * q + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_wait<0>();
  __syncthreads();

  // Partials: unnormalised O, running max and exp-sum per query row.
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (qrow[r] >= NG) continue;
    const int h = kvh * G + qrow[r] % G;
    const size_t row = (((size_t)b * nsplit + split) * N + qnode[r]) * Hq + h;
    float* op = o_part + row * D;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      float2 v = make_float2(o[n][2 * r], o[n][2 * r + 1]);
      *reinterpret_cast<float2*>(op + 8 * n + 2 * t) = v;
    }
    if (t == 0) {
      ml_part[2 * row] = m_run[r];
      ml_part[2 * row + 1] = l_run[r];
    }
  }
}

}  // namespace mma_attn
}  // namespace medusa
