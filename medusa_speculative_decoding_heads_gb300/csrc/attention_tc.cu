// Tree attention on 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA).
//
// "Medusa 심층 아키텍처" (techknowgenie), section "트리 어텐션": every tree node
// attends to the committed KV cache and to its own ancestors (TreeMask
// equation), all nodes in one pass. Block-wise partials merge exactly through
// the running maximum and exp-sum ("최적화 2편" (beengineer500), section 3.3).
//
// One CTA = 128 query rows (tree nodes x query heads of one KV head) against one
// KV range of one sequence; 10 warps:
//   warp 8  TMA producer: K and V tiles of 128 keys (two 64-column boxes each,
//           128-byte swizzle) into a 3-stage ring; allocates / frees TMEM.
//   warp 9  MMA issuer (one thread): S_j = Q K_j^T into TMEM (double buffer,
//           Q itself held in TMEM), then O += P_j V_j with P_j read from TMEM
//           and V as an MN-major shared-memory operand; O stays in TMEM.
//           Shared memory holds only the K/V ring, so three 64 KB stages fit.
//   warps 0-7  softmax: query row i = TMEM lane i is shared by warps w and w+4
//           (64 columns each; the row maximum is combined through shared
//           memory); each thread reads its half of S_j,
//           applies the prefix range or the ancestor bitmask, keeps the running
//           max / exp-sum (the max moves, and O is rescaled, only on a jump of
//           more than 2^8), writes P_j (bf16 pairs) over its S slot in TMEM;
//           tile j+1's softmax never waits for PV_j unless O must be rescaled.
// Every mbarrier wait is bounded (a few seconds of clock cycles); on expiry the
// thread records a code in a device error word and leaves its loop.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "tc_common.cuh"

namespace medusa {

__device__ uint32_t g_attention_tc_error = 0;

namespace {

constexpr int kKeys = 128;
constexpr int kRows = 128;
constexpr int kD = 128;
constexpr int kHalf = kRows * 128;          // bytes of one 64-column swizzled half tile (16 KB)
constexpr int kTile = 2 * kHalf;            // 32 KB: a 128 x 128 bf16 tile
constexpr int kStages = 3;                  // K/V ring depth
constexpr int kSmemBytes = 2 * kStages * kTile + 1024;
constexpr uint32_t kTmemCols = 512;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The running maximum is only moved (and O rescaled) when a tile's maximum
// exceeds it by more than this many binary orders of magnitude; in between, P
// entries stay below 2^kLazy, far inside bf16/f32 range.
constexpr float kLazy = 8.f;

constexpr int kSoftmaxWarps = 8;             // two threads per query row, 64 columns each
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;
constexpr int kThreads = (kSoftmaxWarps + 2) * 32;

// TMEM columns: S double buffer (P_j overwrites the first 64 columns of its S
// slot once both halves of the row have read S_j), O, and Q (bf16 pairs).
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColQ = 384;

__global__ void __launch_bounds__(kThreads, 1)
tree_attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const uint16_t* __restrict__ Q, const int32_t* __restrict__ L, const uint64_t* __restrict__ bits,
                    int N, int Hq, int Hkv, int L_cap, int chunk, float scale_log2, float* __restrict__ o_part,
                    float* __restrict__ ml_part, uint16_t* __restrict__ O) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Ks = sm;                        // [kStages]
  uint8_t* Vs = sm + kStages * kTile;      // [kStages]
  __shared__ __align__(8) uint64_t kv_full[kStages], kv_empty[kStages], s_full[2], p_full[2], p_free[2];
  __shared__ __align__(8) uint64_t x_bar[2], sum_bar;   // row-max / row-sum exchange between column halves
  __shared__ uint32_t tmem_slot;
  __shared__ float xmax[2][2][kRows];   // [tile parity][column half][row]: partial row maxima
  __shared__ float xsum[2][kRows];
  uint32_t* err = &g_attention_tc_error;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = Hq / Hkv, NG = N * G;
  const int mt = blockIdx.x, kvh = blockIdx.y % Hkv, b = blockIdx.y / Hkv;
  const int split = blockIdx.z, nsplit = gridDim.z;
  const int Lb = L[b];
  const bool valid = Lb >= 0 && Lb + N <= L_cap;
  const int k_begin = split * chunk;
  const int k_end = valid ? min(Lb, k_begin + chunk) : 0;
  const int ptiles = k_end > k_begin ? (k_end - k_begin + kKeys - 1) / kKeys : 0;
  const int ntiles = ptiles + ((valid && split == nsplit - 1) ? 1 : 0);   // N <= 128: one tree tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&kv_full[s], 1);
      tc::mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&s_full[s], 1);
      tc::mbar_init(&p_full[s], kSoftmaxThreads);
      tc::mbar_init(&p_free[s], 1);
      tc::mbar_init(&x_bar[s], kSoftmaxThreads);
    }
    tc::mbar_init(&sum_bar, kSoftmaxThreads);
    tc::mbar_fence_init();
  }
  if (warp == kProducerWarp) tc::tmem_alloc(&tmem_slot, kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t tS[2] = {tmem + kColS0, tmem + kColS1};
  const uint32_t tO = tmem + kColO, tQ = tmem + kColQ;

  // Softmax thread (row, hf): row = TMEM lane = 32 * (warp % 4) + lane; hf = column half.
  const bool smx = warp < kSoftmaxWarps;
  const int row = 32 * (warp & 3) + lane;
  const int hf = (warp >> 2) & 1;
  const int qi = mt * kRows + row;
  const bool row_ok = smx && qi < NG;
  const int node = row_ok ? qi / G : 0;
  const int qh = kvh * G + (row_ok ? qi % G : 0);
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;

  if (smx) {
    // Q row half (64 head dims) into TMEM as bf16 pairs: the S MMA reads A from TMEM.
    const uint4* qp = reinterpret_cast<const uint4*>(Q + (((size_t)b * N + node) * Hq + qh) * kD + hf * 64);
    uint32_t qv[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = row_ok ? qp[c] : make_uint4(0, 0, 0, 0);
      qv[4 * c] = v.x;
      qv[4 * c + 1] = v.y;
      qv[4 * c + 2] = v.z;
      qv[4 * c + 3] = v.w;
    }
    tc::tmem_st32(tQ + lane_base + hf * 32, qv);
    tc::tmem_wait_st();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();

  if (warp == kProducerWarp) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      const int head_row = (b * Hkv + kvh) * L_cap;
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int s = j % kStages;
        if (j >= kStages && !tc::mbar_wait(&kv_empty[s], ((j / kStages) - 1) & 1, err, 1)) break;
        const int row0 = j < ptiles ? head_row + k_begin + j * kKeys : head_row + Lb;
        tc::mbar_arrive_expect(&kv_full[s], 2 * kTile);
        tc::tma_load_2d(Ks + s * kTile, &tmK, 0, row0, &kv_full[s]);
        tc::tma_load_2d(Ks + s * kTile + kHalf, &tmK, 64, row0, &kv_full[s]);
        tc::tma_load_2d(Vs + s * kTile, &tmV, 0, row0, &kv_full[s]);
        tc::tma_load_2d(Vs + s * kTile + kHalf, &tmV, 64, row0, &kv_full[s]);
        issued = j + 1;
      }
      // Drain: never leave the CTA with tile loads still landing in shared memory.
      for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
        tc::mbar_wait(&kv_full[j % kStages], (j / kStages) & 1, err, 128);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t idS = tc::idesc_bf16_f32(kRows, kKeys, 0, 0);
      constexpr uint32_t idPV = tc::idesc_bf16_f32(kRows, kD, 0, 1);
      for (int j = 0; j <= ntiles; ++j) {
        if (j < ntiles) {
          const int ks = j % kStages, s = j & 1;
          if (!tc::mbar_wait(&kv_full[ks], (j / kStages) & 1, err, 2)) break;
          // S slot j&1 still holds P_{j-2} until PV_{j-2} has completed
          if (j >= 2 && !tc::mbar_wait(&p_free[s], ((j - 2) >> 1) & 1, err, 4)) break;
          tc::fence_after();
          const uint32_t ka = tc::saddr(Ks + ks * kTile);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
            tc::mma_bf16_tmem_a(tS[s], tQ + kk * 8, tc::sw128_desc(ka + off, 16, 1024), idS, kk > 0);
          }
          tc::commit(&s_full[s]);
        }
        if (j >= 1) {
          const int jp = j - 1, ks = jp % kStages, s = jp & 1;
          if (!tc::mbar_wait(&p_full[s], (jp >> 1) & 1, err, 8)) break;
          tc::fence_after();
          const uint32_t va = tc::saddr(Vs + ks * kTile);
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk) {
            const uint64_t bd = tc::sw128_desc(va + kk * 2048, kHalf, 1024);
            tc::mma_bf16_tmem_a(tO, tS[s] + kk * 8, bd, idPV, (jp > 0 || kk > 0) ? 1 : 0);
          }
          tc::commit(&kv_empty[ks]);
          tc::commit(&p_free[s]);
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    const uint32_t col0 = hf * 64;                // this thread's S / O columns
    const uint64_t nbits = hf ? bits[2 * node + 1] : bits[2 * node];   // tree keys of this column half
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j & 1;
      ok = tc::mbar_wait(&s_full[s], (j >> 1) & 1, err, 16);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::fence_after();
      uint32_t sv[64];
      tc::tmem_ld32(tS[s] + lane_base + col0, sv);
      tc::tmem_ld32(tS[s] + lane_base + col0 + 32, sv + 32);
      tc::tmem_wait_ld();

      const bool tree = j >= ptiles;
      const int nkeys = tree ? N : min(kKeys, k_end - (k_begin + j * kKeys));
      if (tree || nkeys < kKeys) {
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          const int key = col0 + k;
          bool vis = key < nkeys;
          if (tree) vis = vis && ((nbits >> k) & 1ull);
          if (!vis) sv[k] = __float_as_uint(-INFINITY);
        }
      }
      float m8[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) m8[a] = __uint_as_float(sv[a]);
#pragma unroll
      for (int k = 8; k < 64; ++k) m8[k & 7] = fmaxf(m8[k & 7], __uint_as_float(sv[k]));
      float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      xmax[s][hf][row] = mx;
      // Arriving here also tells the partner thread that this half of S_j has been read.
      tc::fence_before();
      tc::mbar_arrive(&x_bar[s]);
      ok = tc::mbar_wait(&x_bar[s], (j >> 1) & 1, err, 256);
      tc::fence_after();
      mx = fmaxf(mx, xmax[s][hf ^ 1][row]);

      const float m_tile = mx * scale_log2;
      float corr = 1.f;
      if (m_tile > m_run + kLazy) {       // also taken on the first visible tile (m_run = -inf)
        corr = tc::ex2(m_run - m_tile);
        m_run = m_tile;
      }
      const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
      float l4[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
      if (row_ok) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float p0 = tc::ex2(fmaf(__uint_as_float(sv[2 * k]), scale_log2, neg_m));
          const float p1 = tc::ex2(fmaf(__uint_as_float(sv[2 * k + 1]), scale_log2, neg_m));
          l4[k & 3] += p0 + p1;
          pk[k] = pack_bf16x2(p0, p1);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) pk[k] = 0u;
      }
      l_run = l_run * corr + ((l4[0] + l4[1]) + (l4[2] + l4[3]));

      if (j >= 1 && __any_sync(0xffffffffu, corr != 1.f)) {
        // O is rescaled only after every earlier PV product has landed (PV_{j-1} is the last one).
        ok = tc::mbar_wait(&p_free[(j - 1) & 1], ((j - 1) >> 1) & 1, err, 64);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc::fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t ov[32];
          tc::tmem_ld32(tO + lane_base + col0 + c * 32, ov);
          tc::tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 32; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * corr);
          tc::tmem_st32(tO + lane_base + col0 + c * 32, ov);
        }
      }
      // P_j (this half: keys 64*hf .. +63) over the first 64 columns of the S slot.
      tc::tmem_st32(tS[s] + lane_base + hf * 32, pk);
      tc::tmem_wait_st();
      tc::fence_before();
      tc::mbar_arrive(&p_full[s]);
    }
    if (ok && ntiles > 0) ok = tc::mbar_wait(&p_free[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, err, 64);
    const bool have = __all_sync(0xffffffffu, ok) && ntiles > 0;
    tc::fence_after();
    xsum[hf][row] = l_run;
    tc::mbar_arrive(&sum_bar);
    tc::mbar_wait(&sum_bar, 0, err, 512);
    const float l_tot = l_run + xsum[hf ^ 1][row];
    if (nsplit == 1) {
      // Single KV split: normalise and write O (bf16) directly, no merge pass.
      const float inv = (have && l_tot > 0.f) ? 1.f / l_tot : 0.f;
      uint16_t* op = O + (((size_t)b * N + node) * Hq + qh) * kD + col0;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t ov[32];
        if (have) {
          tc::tmem_ld32(tO + lane_base + col0 + c * 32, ov);
          tc::tmem_wait_ld();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) ov[x] = 0u;
        }
        if (row_ok) {
#pragma unroll
          for (int x = 0; x < 32; x += 8)
            *reinterpret_cast<uint4*>(op + c * 32 + x) =
                make_uint4(pack_bf16x2(__uint_as_float(ov[x]) * inv, __uint_as_float(ov[x + 1]) * inv),
                           pack_bf16x2(__uint_as_float(ov[x + 2]) * inv, __uint_as_float(ov[x + 3]) * inv),
                           pack_bf16x2(__uint_as_float(ov[x + 4]) * inv, __uint_as_float(ov[x + 5]) * inv),
                           pack_bf16x2(__uint_as_float(ov[x + 6]) * inv, __uint_as_float(ov[x + 7]) * inv));
        }
      }
    } else {
      const size_t orow = (((size_t)b * nsplit + split) * N + node) * Hq + qh;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t ov[32];
        if (have) {
          tc::tmem_ld32(tO + lane_base + col0 + c * 32, ov);
          tc::tmem_wait_ld();
        }
        if (row_ok) {
          float* op = o_part + orow * kD + col0 + c * 32;
#pragma unroll
          for (int x = 0; x < 32; x += 4)
            *reinterpret_cast<float4*>(op + x) =
                have ? make_float4(__uint_as_float(ov[x]), __uint_as_float(ov[x + 1]), __uint_as_float(ov[x + 2]),
                                   __uint_as_float(ov[x + 3]))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      if (row_ok && hf == 0) {
        ml_part[2 * orow] = have ? m_run : -INFINITY;
        ml_part[2 * orow + 1] = have ? l_tot : 0.f;
      }
    }
  }

  tc::fence_before();
  __syncthreads();
  if (warp == kProducerWarp) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

}  // namespace

bool encode_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t pitch_bytes,
                         uint32_t box_cols, uint32_t box_rows) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int attention_tc_mtiles(int NG) { return (NG + kRows - 1) / kRows; }

cudaError_t launch_attention_tc(const medusa_cfg& c, int nsplit, int chunk, const void* Q, const void* Kc,
                                const void* Vc, const int32_t* L, const uint64_t* bits, float* o_part, float* ml_part,
                                void* O, cudaStream_t st) {
  const TreeShape ts = tree_shape(c);
  const uint64_t rows = (uint64_t)c.B * c.Hkv * c.L_cap;
  CUtensorMap tmK, tmV;
  if (!encode_tmap_2d_bf16(&tmK, Kc, rows, kD, kD * 2, 64, kKeys) ||
      !encode_tmap_2d_bf16(&tmV, Vc, rows, kD, kD * 2, 64, kKeys))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tree_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)kD));
  dim3 grid(attention_tc_mtiles(ts.N * (c.Hq / c.Hkv)), c.Hkv * c.B, nsplit);
  tree_attn_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(tmK, tmV, static_cast<const uint16_t*>(Q), L, bits, ts.N, c.Hq,
                                                     c.Hkv, c.L_cap, chunk, scale_log2, o_part, ml_part,
                                                     static_cast<uint16_t*>(O));
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace medusa
