// Tree attention on 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA).
//
// "Medusa 심층 아키텍처" (techknowgenie), section "트리 어텐션": every tree node
// attends to the committed KV cache and to its own ancestors (TreeMask
// equation), all nodes in one pass. Block-wise partials merge exactly through
// the running maximum and exp-sum ("최적화 2편" (beengineer500), section 3.3).
//
// One CTA = one 128-row Q tile (tree nodes x query heads of one KV head) against
// one KV range of one sequence, in tiles of 128 keys. 20 warps (24 with leftover rows):
//   warp 16 TMA producer of K tiles (two 64-column boxes, 128-byte swizzle) into a
//           3-stage K ring; a K stage is free again as soon as S_j (and S'_j) has
//           read it. Allocates TMEM.
//   warp 19 (23 with leftover rows) TMA producer of V tiles into a 3-stage V ring;
//           a V stage is free again once PV_j (and PV'_j) has read it. With K and V
//           in rings of their own, no stage stays held across the softmax, so
//           more of the shared memory holds loads in flight.
//   warp 17 S issuer: S_j = Q K_j^T (Q held in TMEM, K from shared memory) into
//           one of two S tiles in TMEM, so that S_{j+1} is computed while the
//           softmax works on S_j.
//   warp 18 PV issuer: O += P_j V_j with P_j read from TMEM and V as an MN-major
//           shared-memory operand.
//   warps 0-15 softmax: thread = query row = TMEM lane; warpgroup q takes keys
//           [32q, 32q + 32) of every tile. The four warpgroups trade their
//           tile maxima (rounded up to bf16, so that all take exactly the same
//           running max) once per tile; the running max moves (and O is
//           rescaled) only on a jump of more than 2^8.
//   warps 19-22 leftover rows: when the query rows of a KV head end in a short
//           remainder of at most 8 rows (4 rows for 65 nodes x 4 heads), the
//           full tiles' CTAs carry them instead of a CTA of their own: CTA mt of
//           the MT Q tiles takes the key tiles j = mt (mod MT), so that the CTAs
//           sharing each K/V tile through L2 keep the same pace, with transposed
//           narrow products on those K/V tiles: S'^T = K Q'^T (M = 128 keys,
//           N = 16 rows) right behind S_j, and O'^T += V^T P'^T (M = 128 head
//           dims) right behind PV_j, whose completion then frees the stage. Q'
//           and P' sit in shared memory. Thread = key (S') or head dim (O'); a
//           row's maximum over a warp's 32 keys is one redux.sync, and the four
//           warps' maxima meet in shared memory. The per-row loops run to the
//           leftover row count rounded up to 2, 4 or 8 (the kernel's template
//           argument): these warps share the SM sub-partitions' issue slots with
//           the softmax warps. Each CTA writes its partial (O', m, l);
//           tree_attn_xmerge_kernel merges them.
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

constexpr int kKeys = 128;                  // keys per tile
constexpr int kRows = 128;                  // query rows per Q tile (MMA M)
constexpr int kD = 128;
constexpr int kHalf = 128 * 128;            // 128 rows x 64 bf16: one 128-byte-swizzled half of a tile (16 KB)
constexpr int kOperand = 2 * kHalf;         // a 128 x 128 bf16 tile, K or V (32 KB)
#ifndef MEDUSA_ATTN_KSTAGES
#define MEDUSA_ATTN_KSTAGES 3
#endif
#ifndef MEDUSA_ATTN_VSTAGES
#define MEDUSA_ATTN_VSTAGES 3
#endif
constexpr int kStagesK = MEDUSA_ATTN_KSTAGES;   // stages of the K ring
constexpr int kStagesV = MEDUSA_ATTN_VSTAGES;   // stages of the V ring
constexpr int kGroups = 4;                  // softmax warpgroups, 32 keys each
constexpr int kXchg = kGroups * kRows * 4;   // exp-sums [group][row] for the epilogue (2 KB)
constexpr int kXRows = 16;                   // N of the narrow products (the smallest N with M = 128)
constexpr int kXMax = 8;                     // leftover query rows one CTA carries (rows kXMax.. of Q', P' stay 0)
constexpr int kXHalf = kXRows * 128;         // 16 rows x 64 bf16, one 128-byte-swizzled half (2 KB)
// shared memory: K/V ring | exp-sums | and with leftover rows: Q' [16 rows][128 dims] | P' two slots
// [16 rows][128 keys] | their reductions (maxima [2][4 warps][16], sums [4 warps][16])
constexpr int kOffV = kStagesK * kOperand;   // the V ring follows the K ring
constexpr int kOffXl = (kStagesK + kStagesV) * kOperand;
constexpr int kOffQx = kOffXl + kXchg;   // 1024-byte aligned, as the swizzled operands need
constexpr int kOffPx = kOffQx + 2 * kXHalf;
constexpr int kOffRed = kOffPx + 4 * kXHalf;
__host__ __device__ constexpr int smem_of(bool fold) { return (fold ? kOffRed + 1024 : kOffQx) + 1024; }   // + alignment slack
static_assert(kOffQx % 1024 == 0 && kOffPx % 1024 == 0, "swizzled operands start on 1024-byte boundaries");
constexpr uint32_t kTmemCols = 512;
constexpr int kSoftmaxWarps = 4 * kGroups;
constexpr int kProducerWarp = 16;
constexpr int kMmaSWarp = 17;   // issues S = Q K^T (and S'^T = K Q'^T)
constexpr int kMmaPWarp = 18;   // issues O += P V (and O'^T += V^T P'^T)
constexpr int kXWarp0 = 19;     // warps 19-22: softmax of the leftover rows
__host__ __device__ constexpr int vproducer_warp(bool fold) { return fold ? 23 : 19; }
// 20 warps; 24 for configurations whose query rows per KV head end in a short remainder
__host__ __device__ constexpr int threads_of(bool fold) { return (vproducer_warp(fold) + 1) * 32; }
constexpr int kSortMax = 256;   // batches up to this size are taken longest sequence first

// TMEM columns: two S tiles (128 f32 columns each; warpgroup q writes P of its
// keys [32q, 32q + 32) as bf16 pairs over columns [32q, 32q + 16)), the O
// accumulator (128 f32 columns), Q as bf16 pairs (64 columns), the per-tile
// maxima of the four warpgroups (columns 4 * (tile parity) + group) and the
// leftover rows' two S'^T tiles and O'^T accumulator (16 columns each).
__host__ __device__ constexpr uint32_t col_S(int slot) { return 128u * slot; }
constexpr uint32_t kColO = 256;
constexpr uint32_t kColQ = 384;
constexpr uint32_t kColX = 448;
constexpr uint32_t kColS2 = 464;   // two S'^T tiles of 16 columns (lane = key, column = leftover row)
constexpr uint32_t kColO2 = 496;   // O'^T (lane = head dim, column = leftover row)

// Query rows past the last full 128-row tile that the last tile's CTA carries:
// a remainder of 1..8 rows after at least one full tile, else none.
__host__ __device__ inline int extra_rows(int NG) {
  const int r = NG % kRows;
  return (NG > kRows && r > 0 && r <= kXMax) ? r : 0;
}

// The running maximum is only moved (and O rescaled) when a tile's maximum
// exceeds it by more than this many binary orders of magnitude; in between, P
// entries stay below 2^kLazy, far inside bf16/f32 range.
constexpr float kLazy = 8.f;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// x rounded up to a bf16 value (its upper 16 bits); -inf stays -inf.
__device__ __forceinline__ uint16_t bf16_ceil(float x) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t r = (x > 0.f) ? ((u + 0xFFFFu) & 0xFFFF0000u) : (u & 0xFFFF0000u);
  return (uint16_t)(r >> 16);
}
__device__ __forceinline__ float bf16_value(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Masks 32 scores of tile keys [k0, k0 + 32): a key is visible when it is inside
// the tile's range and (tree tiles) its bit is set; `word` holds the node's mask
// bits of the 64 keys starting at k0 & ~63.
__device__ __forceinline__ void mask32(uint32_t* v, int k0, int nkeys, bool tree, uint64_t word) {
  if (tree || k0 + 32 > nkeys) {
    const int sh = k0 & 63;
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (!(k0 + k < nkeys && (!tree || ((word >> (sh + k)) & 1ull)))) v[k] = __float_as_uint(-INFINITY);
  }
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float max32(const uint32_t* v) {
  float m4[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t* c = v + 8 * j;
    float m = fmax3(__uint_as_float(c[0]), __uint_as_float(c[1]), __uint_as_float(c[2]));
    m = fmax3(m, __uint_as_float(c[3]), __uint_as_float(c[4]));
    m = fmax3(m, __uint_as_float(c[5]), __uint_as_float(c[6]));
    m4[j] = fmaxf(m, __uint_as_float(c[7]));
  }
  return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
}

// p = 2^(s * scale_log2 - m) for 32 scores, packed as 16 bf16 pairs; returns their sum.
__device__ __forceinline__ float exp32(const uint32_t* v, float scale_log2, float neg_m, uint32_t* pk) {
  const float2 sc = make_float2(scale_log2, scale_log2), nm = make_float2(neg_m, neg_m);
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float2 x = __ffma2_rn(make_float2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1])), sc, nm);
    float2 p;
    p.x = tc::ex2(x.x);
    p.y = tc::ex2(x.y);
    if (k & 1)
      acc1 = __fadd2_rn(acc1, p);
    else
      acc0 = __fadd2_rn(acc0, p);
    pk[k] = pack_bf16x2(p.x, p.y);
  }
  const float2 a = __fadd2_rn(acc0, acc1);
  return a.x + a.y;
}

// kXR: 0 without leftover rows, else the number of leftover rows rounded up to 2, 4 or 8
// (the leftover softmax's per-row loops run to kXR).
template <int kXR>
__global__ void __launch_bounds__(threads_of(kXR > 0), 1)
tree_attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmKt, const __grid_constant__ CUtensorMap tmVt,
                    const uint16_t* __restrict__ Q, const int32_t* __restrict__ L, const uint64_t* __restrict__ bits,
                    int N, int Hq, int Hkv, int L_cap, int chunk, float scale_log2, float* __restrict__ o_part,
                    float* __restrict__ ml_part, uint16_t* __restrict__ O, const int32_t* __restrict__ block_table,
                    int page_rows, int num_pages, float* __restrict__ x_part) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = sm;                                                    // K ring [stage], then V ring [stage]
  float* xl = reinterpret_cast<float*>(sm + kOffXl);   // [group][row] exp-sums
  __shared__ __align__(8) uint64_t k_full[kStagesK], k_empty[kStagesK], v_full[kStagesV], v_empty[kStagesV];
  __shared__ __align__(8) uint64_t s_full[2], p_full[2], p_free[2], xbar;
  __shared__ __align__(8) uint64_t s2_full[2], p2_full[2], p2_free[2], xbar2;   // leftover rows
  __shared__ uint32_t tmem_slot;
  __shared__ int seq;
  uint32_t* err = &g_attention_tc_error;

  // Barriers and TMEM are set up before the wait on the previous kernel (neither touches
  // global memory), so that this overlaps its tail.
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesK; ++i) {
      tc::mbar_init(&k_full[i], 1);
      tc::mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < kStagesV; ++i) {
      tc::mbar_init(&v_full[i], 1);
      tc::mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&s_full[i], 1);
      tc::mbar_init(&p_full[i], kSoftmaxWarps * 32);
      tc::mbar_init(&p_free[i], 1);
    }
    tc::mbar_init(&xbar, kSoftmaxWarps * 32);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&s2_full[i], 1);
      tc::mbar_init(&p2_full[i], 128);
      tc::mbar_init(&p2_free[i], 1);
    }
    tc::mbar_init(&xbar2, 128);
    tc::mbar_fence_init();
  }
  if ((threadIdx.x >> 5) == kProducerWarp) tc::tmem_alloc(&tmem_slot, kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  pdl_wait();   // the previous kernel's writes (L, the cache) are visible from here on

  // Launch order: x = Q tile (fastest, so the tiles of one KV head share its K/V
  // through L2), y = (sequence rank, KV head), z = KV split. Sequences are taken
  // longest first, so that the block scheduler's tail holds the smallest units.
  const int mt = blockIdx.x, split = blockIdx.z, nsplit = gridDim.z;
  const int kvh = blockIdx.y % Hkv, rank = blockIdx.y / Hkv, B = gridDim.y / Hkv;
  int b = rank;
  if (B <= kSortMax) {
    for (int t = threadIdx.x; t < B; t += blockDim.x) {
      const int lt = L[t];
      int r = 0;
      for (int u = 0; u < B; ++u) {
        const int lu = L[u];
        r += (lu > lt || (lu == lt && u < t)) ? 1 : 0;
      }
      if (r == rank) seq = t;
    }
    __syncthreads();
    b = seq;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = Hq / Hkv, NG = N * G;
  // Leftover rows: every Q-tile CTA of the KV head carries them on its share of the key tiles
  // (tiles j with j % MT == mt), so that the CTAs that share each K/V tile through L2 keep the
  // same pace; their partial results merge in tree_attn_xmerge_kernel.
  const int MT = (int)gridDim.x;
  constexpr bool kFold = kXR > 0;
  const int R = kFold ? extra_rows(NG) : 0;
  const bool xtra = R > 0;
  const bool xs = xtra && warp >= kXWarp0 && warp < kXWarp0 + 4;   // a leftover-row softmax thread
  const int xt = 32 * (warp & 3) + lane;     // its TMEM lane: key of S'^T, head dim of O'^T
  const int xq0 = kRows * MT;                // query row index of leftover row 0
  // this CTA's leftover partial (o[D], m, l) of row r: x_part + (xbase + r) * (kD + 2)
  const size_t xbase = ((((size_t)b * Hkv + kvh) * nsplit + split) * MT + mt) * kXMax;
  const int Lb = L[b];
  const bool valid = Lb >= 0 && Lb + N <= L_cap;
  const int k_begin = split * chunk;
  const int k_end = valid ? min(Lb, k_begin + chunk) : 0;
  const int ptiles = k_end > k_begin ? (k_end - k_begin + kKeys - 1) / kKeys : 0;
  const int ntiles = ptiles + ((valid && split == nsplit - 1) ? 1 : 0);   // N <= 128: one tree tile

  // Softmax thread: warpgroup q (keys [32q, 32q + 32) of every tile), row = TMEM lane.
  const bool smx = warp < kSoftmaxWarps;
  const int q = (warp >> 2) & 3;
  const int row = 32 * (warp & 3) + lane;
  const int qi = mt * kRows + row;
  const bool row_ok = smx && qi < NG;
  const int node = row_ok ? qi / G : 0;
  const int qh = kvh * G + (row_ok ? qi % G : 0);
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;

  if (ntiles == 0) {
    // Nothing to attend to in this range: an empty partial (or zeros for an
    // invalid sequence), without touching TMEM or the barriers.
    if (row_ok) {
      if (nsplit == 1) {
        uint4* op = reinterpret_cast<uint4*>(O + (((size_t)b * N + node) * Hq + qh) * kD + 32 * q);
#pragma unroll
        for (int x = 0; x < 4; ++x) op[x] = make_uint4(0, 0, 0, 0);
      } else if (q == 0) {
        const size_t orow = (((size_t)b * nsplit + split) * N + node) * Hq + qh;
        ml_part[2 * orow] = -INFINITY;
        ml_part[2 * orow + 1] = 0.f;
      }
    }
    if (xs && xt == 0)
      for (int r = 0; r < R; ++r) {   // an empty leftover partial
        x_part[(xbase + r) * (kD + 2) + kD] = -INFINITY;
        x_part[(xbase + r) * (kD + 2) + kD + 1] = 0.f;
        if (nsplit > 1 && mt == 0) {   // the split merge leaves these rows empty; the leftover merge fills them
          const int xqi = xq0 + r;
          const size_t orow = (((size_t)b * nsplit + split) * N + xqi / G) * Hq + kvh * G + xqi % G;
          ml_part[2 * orow] = -INFINITY;
          ml_part[2 * orow + 1] = 0.f;
        }
      }
    if (warp == kProducerWarp) tc::tmem_dealloc(tmem_slot, kTmemCols);
    return;
  }

  const uint32_t tmem = tmem_slot;
  const uint32_t tQ = tmem + kColQ;

  if (smx) {
    // Q row into TMEM as bf16 pairs (the S product's A operand): warpgroup q
    // stages head dims [32q, 32q + 32), 16 columns.
    const uint4* qp = reinterpret_cast<const uint4*>(Q + (((size_t)b * N + node) * Hq + qh) * kD + 32 * q);
    uint32_t qv[16];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 v = row_ok ? qp[c] : make_uint4(0, 0, 0, 0);
      qv[4 * c] = v.x;
      qv[4 * c + 1] = v.y;
      qv[4 * c + 2] = v.z;
      qv[4 * c + 3] = v.w;
    }
    tc::tmem_st16(tQ + lane_base + 16 * q, qv);
    tc::tmem_wait_st();
  }
  if (xs) {
    // Q' (the B operand of S'^T = K Q'^T) into shared memory: [16 rows][128 dims], K-major,
    // two 64-dim halves, 128-byte swizzle; rows past R and both P' slots are zeroed.
    for (int c = xt; c < kXRows * 16; c += 128) {
      const int r = c >> 4, ch = c & 15;   // row, 16-byte chunk (8 dims) along D
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < R) {
        const int xqi = xq0 + r;
        v = *reinterpret_cast<const uint4*>(Q + (((size_t)b * N + xqi / G) * Hq + kvh * G + xqi % G) * kD + 8 * ch);
      }
      *reinterpret_cast<uint4*>(sm + kOffQx + (ch >> 3) * kXHalf + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) = v;
    }
    for (int c = xt; c < 4 * kXHalf / 16; c += 128)
      reinterpret_cast<uint4*>(sm + kOffPx)[c] = make_uint4(0, 0, 0, 0);
    tc::fence_proxy_async();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();

  if (warp == kProducerWarp || warp == vproducer_warp(kFold)) {
    // ------------------------------------------------------------ TMA producers
    // Warp 16 loads the K tiles, the V producer warp the V tiles, each into its own
    // ring, waiting only for its own ring's stages. Paged cache: prefix tile j
    // (keys k_begin + 128 j ..) lies inside one page (page_rows is a multiple of
    // 128), pool row (page * Hkv + kvh) * page_rows + key % page_rows; every 32
    // tiles each lane fetches one block-table entry and lane 0 takes them by
    // shuffle. The tree tile comes from the staging buffer, row (b * Hkv + kvh) * N.
    // Contiguous cache: row (b * Hkv + kvh) * L_cap + key.
    const bool isv = warp != kProducerWarp;
    uint64_t* full = isv ? v_full : k_full;
    uint64_t* empty = isv ? v_empty : k_empty;
    uint8_t* base = ring + (isv ? kOffV : 0);
    const CUtensorMap* mp = isv ? &tmV : &tmK;     // prefix rows
    const CUtensorMap* mt_ = isv ? &tmVt : &tmKt;  // tree rows (the same map unless paged)
    const int nst = isv ? kStagesV : kStagesK;
    const int max_pages = page_rows > 0 ? L_cap / page_rows : 0;
    const int head_row = (b * Hkv + kvh) * L_cap;
    int page_reg = 0, issued = 0;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % nst;
      bool ok = true;
      if (j >= nst) ok = tc::mbar_wait<true>(&empty[st], ((j / nst) - 1) & 1, err, 1);
      if (!__all_sync(0xffffffffu, ok)) break;
      const bool tree = j >= ptiles;
      int row0;
      if (page_rows > 0) {
        if (!tree && (j & 31) == 0) {
          const int jj = j + lane;
          page_reg = jj < ptiles ? block_table[(size_t)b * max_pages + (k_begin + jj * kKeys) / page_rows] : 0;
        }
        const int page = __shfl_sync(0xffffffffu, page_reg, j & 31);
        // a page id outside the pool addresses rows past the tensor map, which TMA fills with zeros
        MEDUSA_CHECK(isv || tree || lane != 0 || (page >= 0 && page < num_pages), MEDUSA_CHECK_PAGE);
        const int key0 = k_begin + j * kKeys;
        row0 = tree ? (b * Hkv + kvh) * N : (page * Hkv + kvh) * page_rows + key0 % page_rows;
      } else {
        row0 = tree ? head_row + Lb : head_row + k_begin + j * kKeys;
      }
      if (lane == 0) {
        const CUtensorMap* m = tree ? mt_ : mp;
        uint8_t* dst = base + st * kOperand;
        tc::mbar_arrive_expect(&full[st], kOperand);
        tc::tma_load_2d(dst, m, 0, row0, &full[st]);
        tc::tma_load_2d(dst + kHalf, m, 64, row0, &full[st]);
      }
      __syncwarp();
      issued = j + 1;
    }
    if (lane == 0)   // drain: never leave the CTA with tile loads still landing in shared memory
      for (int j = issued > nst ? issued - nst : 0; j < issued; ++j)
        tc::mbar_wait(&full[j % nst], (j / nst) & 1, err, 128);
  } else if (warp == kMmaSWarp) {
    // ------------------------------------------------------------------ S issuer
    // The whole warp walks the schedule (uniform waits); one elected lane issues.
    constexpr uint32_t idS = tc::idesc_bf16_f32(kRows, kKeys, 0, 0);
    constexpr uint32_t idS2 = tc::idesc_bf16_f32(kKeys, kXRows, 0, 0);
    const uint64_t dK = tc::sw128_desc(tc::saddr(ring), 16, 1024);
    const uint64_t dQx = tc::sw128_desc(tc::saddr(sm + kOffQx), 16, 1024);
    for (int j = 0; j < ntiles; ++j) {
      const int slot = j & 1, st = j % kStagesK;
      bool ok = tc::mbar_wait<true>(&k_full[st], (j / kStagesK) & 1, err, 2);
      // S tile `slot` still holds P_{j-2} until PV_{j-2} completes
      if (ok && j >= 2) ok = tc::mbar_wait<true>(&p_free[slot], ((j >> 1) - 1) & 1, err, 4);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc::fence_after();
      if (tc::elect_one()) {
        const uint64_t b0 = dK + (uint64_t)((st * kOperand) >> 4);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
          tc::mma_bf16_tmem_a(tmem + col_S(slot), tQ + kk * 8, b0 + off, idS, kk > 0);
        }
        tc::commit(&s_full[slot]);
      }
      __syncwarp();
      if (xtra && j % MT == mt) {
        // S'^T = K_j Q'^T for this CTA's narrow tile jx, once PV'_{jx-2} completed: its softmax
        // had read S' slot jx & 1, and P' slot jx & 1 is free for the softmax of tile jx
        const int jx = j / MT, sx = jx & 1;
        if (jx >= 2 && !__all_sync(0xffffffffu, tc::mbar_wait<true>(&p2_free[sx], ((jx >> 1) - 1) & 1, err, 1024)))
          break;
        tc::fence_after();
        if (tc::elect_one()) {
          const uint64_t a0 = dK + (uint64_t)((st * kOperand) >> 4);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
            const uint32_t offx = ((kk >> 2) * kXHalf + (kk & 3) * 32) >> 4;
            tc::mma_bf16(tmem + kColS2 + 16 * sx, a0 + off, dQx + offx, idS2, kk > 0);
          }
          tc::commit(&s2_full[sx]);
        }
        __syncwarp();
      }
      // the K stage is free once this tile's S (and S') products have read it
      if (tc::elect_one()) tc::commit(&k_empty[st]);
      __syncwarp();
    }
  } else if (warp == kMmaPWarp) {
    // ------------------------------------------------------------------ PV issuer
    // The completion of PV_j (and of PV'_j on a tile with leftover rows) frees V stage j.
    constexpr uint32_t idPV = tc::idesc_bf16_f32(kRows, kD, 0, 1);
    constexpr uint32_t idPV2 = tc::idesc_bf16_f32(kD, kXRows, 1, 0);   // A = V^T (MN-major), B = P' (K-major)
    const uint64_t dV = tc::sw128_desc(tc::saddr(ring + kOffV), kHalf, 1024);   // MN-major: LBO = 64-column half
    const uint64_t dPx = tc::sw128_desc(tc::saddr(sm + kOffPx), 16, 1024);
    // O'^T += V_t^T P'^T for narrow tile jx (key tile t) once its leftover softmax has arrived;
    // its completion also frees the stage
    auto issue_pv2 = [&](int t, int jx) {
      if (!__all_sync(0xffffffffu, tc::mbar_wait<true>(&p2_full[jx & 1], (jx >> 1) & 1, err, 2048))) return false;
      tc::fence_after();
      if (tc::elect_one()) {
        const uint64_t a0 = dV + (uint64_t)(((t % kStagesV) * kOperand) >> 4);
        const uint64_t p0 = dPx + (uint64_t)(((jx & 1) * 2 * kXHalf) >> 4);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint32_t offx = ((kk >> 2) * kXHalf + (kk & 3) * 32) >> 4;
          tc::mma_bf16(tmem + kColO2, a0 + (uint64_t)((kk * 2048) >> 4), p0 + offx, idPV2, (jx > 0 || kk > 0) ? 1 : 0);
        }
        tc::commit(&p2_free[jx & 1]);
        tc::commit(&v_empty[t % kStagesV]);
      }
      __syncwarp();
      return true;
    };
    for (int j = 0; j < ntiles; ++j) {
      const int slot = j & 1, st = j % kStagesV;
      bool ok = tc::mbar_wait<true>(&v_full[st], (j / kStagesV) & 1, err, 1u << 17);
      if (ok) ok = tc::mbar_wait<true>(&p_full[slot], (j >> 1) & 1, err, 8);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc::fence_after();
      if (tc::elect_one()) {
        const uint64_t b0 = dV + (uint64_t)((st * kOperand) >> 4);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)   // keys [16kk, 16kk + 16): group kk / 2, P columns 32(kk/2) + 8(kk%2)
          tc::mma_bf16_tmem_a(tmem + kColO, tmem + col_S(slot) + 32 * (kk >> 1) + 8 * (kk & 1),
                              b0 + (uint64_t)((kk * 2048) >> 4), idPV, (j > 0 || kk > 0) ? 1 : 0);
        tc::commit(&p_free[slot]);
        if (!(xtra && j % MT == mt)) tc::commit(&v_empty[st]);
      }
      __syncwarp();
      if (xtra && j % MT == mt && !issue_pv2(j, j / MT)) break;
    }
  } else if (smx) {
    // ------------------------------------------------------------------ softmax
    const uint32_t c_q = 32u * q;   // this warpgroup's 32 columns of S (and of O)
    const uint32_t tO = tmem + kColO + lane_base + c_q;
    const uint64_t word = bits[2 * node + (q >> 1)];   // mask bits of tree keys [64(q/2), 64(q/2) + 64)
    float m_run = -INFINITY, l_run = 0.f;              // l_run: this warpgroup's share of the exp-sum
    bool ok = true;
    int j = 0;
    for (; j < ntiles; ++j) {
      const int slot = j & 1;
      ok = tc::mbar_wait(&s_full[slot], (j >> 1) & 1, err, 16);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::fence_after();
      const uint32_t tS = tmem + col_S(slot) + lane_base + c_q;
      const bool tree = j >= ptiles;
      const int nkeys = tree ? N : min(kKeys, k_end - (k_begin + j * kKeys));
      uint32_t v[32], pk[16];
      tc::tmem_ld32(tS, v);
      tc::tmem_wait_ld();
      mask32(v, (int)c_q, nkeys, tree, word);
      // Trade tile maxima (log2 units, rounded up to bf16) with the other
      // warpgroups through TMEM. While the exchange completes, P is computed with
      // the current running max; it is recomputed only for rows whose max then
      // has to move.
      const uint16_t mine = bf16_ceil(max32(v) * scale_log2);
      const uint32_t tX = tmem + kColX + lane_base + 4 * (j & 1);
      tc::tmem_st1(tX + q, (uint32_t)mine << 16);
      tc::tmem_wait_st();
      tc::fence_before();
      tc::mbar_arrive(&xbar);
      float l_tile = 0.f;
      const bool spec = m_run != -INFINITY && bf16_value(mine) <= m_run + kLazy;
      if (__all_sync(0xffffffffu, spec)) {
        if (row_ok) l_tile = exp32(v, scale_log2, -m_run, pk);
        else {
#pragma unroll
          for (int k = 0; k < 16; ++k) pk[k] = 0u;
        }
        tc::tmem_st16(tS, pk);   // P of keys [32q, 32q + 32) over this group's first 16 columns
      }
      ok = tc::mbar_wait(&xbar, j & 1, err, 32);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::fence_after();
      uint32_t xm[4];
      tc::tmem_ld4(tX, xm);
      tc::tmem_wait_ld();
      const float m_tile = fmaxf(fmaxf(__uint_as_float(xm[0]), __uint_as_float(xm[1])),
                                 fmaxf(__uint_as_float(xm[2]), __uint_as_float(xm[3])));
      float corr = 1.f;
      const bool move = m_tile > m_run + kLazy;   // also on the first visible tile (m_run = -inf)
      if (__any_sync(0xffffffffu, move || !__all_sync(0xffffffffu, spec))) {
        if (move) {
          corr = tc::ex2(m_run - m_tile);
          m_run = m_tile;
        }
        const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
        if (row_ok) l_tile = exp32(v, scale_log2, neg_m, pk);
        else {
#pragma unroll
          for (int k = 0; k < 16; ++k) pk[k] = 0u;
        }
        tc::tmem_st16(tS, pk);
      }
      l_run = l_run * corr + l_tile;
      if (j >= 1 && __any_sync(0xffffffffu, corr != 1.f)) {
        // rescale this group's 32 columns of O once PV_{j-1} has landed
        ok = tc::mbar_wait(&p_free[(j - 1) & 1], ((j - 1) >> 1) & 1, err, 64);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc::fence_after();
        uint32_t ov[32];
        tc::tmem_ld32(tO, ov);
        tc::tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * corr);
        tc::tmem_st32(tO, ov);
      }
      tc::tmem_wait_st();
      tc::fence_before();
      tc::mbar_arrive(&p_full[slot]);
    }
    // The last PV: completion (ntiles-1) / 2 of its slot's p_free.
    if (ok) ok = tc::mbar_wait(&p_free[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, err, 256);
    const bool have = __all_sync(0xffffffffu, ok);
    tc::fence_after();
    // Sum the four groups' exp-sums.
    xl[q * kRows + row] = l_run;
    tc::mbar_arrive(&xbar);
    tc::mbar_wait(&xbar, ntiles & 1, err, 512);
    const float l_tot = (xl[row] + xl[kRows + row]) + (xl[2 * kRows + row] + xl[3 * kRows + row]);
    uint32_t ov[32];
    if (have) {   // warp-uniform: the TMEM load is a collective of the warp
      tc::tmem_ld32(tO, ov);
      tc::tmem_wait_ld();
    } else {
#pragma unroll
      for (int x = 0; x < 32; ++x) ov[x] = 0u;
    }
    if (row_ok) {
      if (nsplit == 1) {
        const float inv = (have && l_tot > 0.f) ? 1.f / l_tot : 0.f;
        uint16_t* op = O + (((size_t)b * N + node) * Hq + qh) * kD + c_q;
#pragma unroll
        for (int x = 0; x < 32; x += 8)
          *reinterpret_cast<uint4*>(op + x) =
              make_uint4(pack_bf16x2(__uint_as_float(ov[x]) * inv, __uint_as_float(ov[x + 1]) * inv),
                         pack_bf16x2(__uint_as_float(ov[x + 2]) * inv, __uint_as_float(ov[x + 3]) * inv),
                         pack_bf16x2(__uint_as_float(ov[x + 4]) * inv, __uint_as_float(ov[x + 5]) * inv),
                         pack_bf16x2(__uint_as_float(ov[x + 6]) * inv, __uint_as_float(ov[x + 7]) * inv));
      } else {
        const size_t orow = (((size_t)b * nsplit + split) * N + node) * Hq + qh;
        float* op = o_part + orow * kD + c_q;
#pragma unroll
        for (int x = 0; x < 32; x += 4)
          *reinterpret_cast<float4*>(op + x) = make_float4(__uint_as_float(ov[x]), __uint_as_float(ov[x + 1]),
                                                           __uint_as_float(ov[x + 2]), __uint_as_float(ov[x + 3]));
        if (q == 0) {
          ml_part[2 * orow] = have ? m_run : -INFINITY;
          ml_part[2 * orow + 1] = have ? l_tot : 0.f;
        }
      }
    }
  } else if (xs) {
    // ------------------------------------------------------- leftover-row softmax
    // Thread xt holds key xt of S'^T (one score per leftover row) and head dim xt of
    // O'^T. This CTA's narrow tiles are the key tiles j = jx * MT + mt. Row maxima: one
    // redux.sync per row and warp, then the four warps' values through shared memory
    // (double-buffered by the narrow tile's parity, one mbarrier phase per narrow tile).
    const uint32_t xl_base = (uint32_t)(32 * (warp & 3)) << 16;
    float* red = reinterpret_cast<float*>(sm + kOffRed);   // maxima [parity][row][warp], then sums [warp][row]
    const int nx = ntiles > mt ? (ntiles - 1 - mt) / MT + 1 : 0;
    float m_run[kXMax], l_t[kXMax], corr[kXMax];
#pragma unroll
    for (int r = 0; r < kXMax; ++r) {
      m_run[r] = -INFINITY;
      l_t[r] = 0.f;
    }
    bool ok = true;
    for (int jx = 0; jx < nx; ++jx) {
      const int j = jx * MT + mt, slot = jx & 1;
      ok = tc::mbar_wait(&s2_full[slot], (jx >> 1) & 1, err, 4096);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::fence_after();
      uint32_t v[kXMax];
      tc::tmem_ld8(tmem + kColS2 + 16 * slot + xl_base, v);
      tc::tmem_wait_ld();
      const bool tree = j >= ptiles;
      const int nkeys = tree ? N : min(kKeys, k_end - (k_begin + j * kKeys));
      float x[kXR > 0 ? kXR : 1];
#pragma unroll
      for (int r = 0; r < kXR; ++r) {
        bool vis = r < R && xt < nkeys;
        if (vis && tree) vis = (bits[2 * ((xq0 + r) / G) + (xt >> 6)] >> (xt & 63)) & 1ull;
        x[r] = vis ? __uint_as_float(v[r]) * scale_log2 : -INFINITY;
      }
      float* rm = red + 64 * slot;   // tile maxima [row][warp]
#pragma unroll
      for (int r = 0; r < kXR; ++r) {
        if (r < R) {
          float m;
          asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(x[r]));
          if (lane == 0) rm[4 * r + (warp & 3)] = m;
        }
      }
      tc::mbar_arrive(&xbar2);
      ok = tc::mbar_wait(&xbar2, jx & 1, err, 8192);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      bool any = false;
#pragma unroll
      for (int r = 0; r < kXR; ++r) {
        corr[r] = 1.f;
        if (r < R) {
          const float4 mw = *reinterpret_cast<const float4*>(rm + 4 * r);
          const float m_tile = fmaxf(fmaxf(mw.x, mw.y), fmaxf(mw.z, mw.w));
          if (m_tile > m_run[r] + kLazy) {   // also on the first tile (m_run = -inf): corr = 0
            corr[r] = tc::ex2(m_run[r] - m_tile);
            m_run[r] = m_tile;
            any = true;
          }
        }
      }
      // P' row r, key xt -> the B operand of O'^T += V^T P'^T ([row][key], K-major, 128-byte
      // swizzle, two 64-key halves). Its slot last fed PV'_{jx-2}, complete before S'_jx.
      uint8_t* pr = sm + kOffPx + slot * 2 * kXHalf + (xt >> 6) * kXHalf;
      const int cc = xt & 63;
#pragma unroll
      for (int r = 0; r < kXR; ++r) {
        if (r < R) {
          const float pv = x[r] == -INFINITY ? 0.f : tc::ex2(x[r] - m_run[r]);
          l_t[r] = l_t[r] * corr[r] + pv;
          uint16_t hv;
          asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(hv) : "f"(pv));
          *reinterpret_cast<uint16_t*>(pr + r * 128 + ((((cc >> 3) ^ (r & 7)) << 4) | ((cc & 7) << 1))) = hv;
        }
      }
      if (jx >= 1 && any) {
        // rescale O'^T once PV'_{jx-1} has landed (thread = head dim, column = row)
        ok = tc::mbar_wait(&p2_free[(jx - 1) & 1], ((jx - 1) >> 1) & 1, err, 16384);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc::fence_after();
        uint32_t ov[kXMax];
        tc::tmem_ld8(tmem + kColO2 + xl_base, ov);
        tc::tmem_wait_ld();
#pragma unroll
        for (int r = 0; r < kXR; ++r) ov[r] = __float_as_uint(__uint_as_float(ov[r]) * corr[r]);
        tc::tmem_st8(tmem + kColO2 + xl_base, ov);
      }
      tc::fence_proxy_async();   // the P' stores, visible to the tensor core
      tc::tmem_wait_st();
      tc::fence_before();
      tc::mbar_arrive(&p2_full[slot]);
    }
    if (ok && nx > 0) ok = tc::mbar_wait(&p2_free[(nx - 1) & 1], ((nx - 1) >> 1) & 1, err, 32768);
    const bool have = __all_sync(0xffffffffu, ok) && nx > 0;
    tc::fence_after();
    // row sums over the 128 key lanes
    float* rs = red + 128;
#pragma unroll
    for (int r = 0; r < kXMax; ++r) {
      if (r < R) {
        float t = l_t[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) rs[16 * (warp & 3) + r] = t;
      }
    }
    tc::mbar_arrive(&xbar2);
    const bool summed = tc::mbar_wait(&xbar2, nx & 1, err, 65536);
    uint32_t ov[kXMax];
    if (have) {   // warp-uniform: the TMEM load is a collective of the warp
      tc::tmem_ld8(tmem + kColO2 + xl_base, ov);
      tc::tmem_wait_ld();
    } else {
#pragma unroll
      for (int r = 0; r < kXMax; ++r) ov[r] = 0u;
    }
    // this CTA's partial of every leftover row: unnormalised O', running max (log2) and exp-sum
#pragma unroll
    for (int r = 0; r < kXMax; ++r) {
      if (r < R) {
        float* xp = x_part + (xbase + r) * (kD + 2);
        xp[xt] = __uint_as_float(ov[r]);
        if (xt == 0) {
          const bool live = have && summed;
          xp[kD] = live ? m_run[r] : -INFINITY;
          xp[kD + 1] = live ? (rs[r] + rs[16 + r]) + (rs[32 + r] + rs[48 + r]) : 0.f;
          if (nsplit > 1 && mt == 0) {   // the split merge leaves these rows empty; the leftover merge fills them
            const int xqi = xq0 + r;
            const size_t orow = (((size_t)b * nsplit + split) * N + xqi / G) * Hq + kvh * G + xqi % G;
            ml_part[2 * orow] = -INFINITY;
            ml_part[2 * orow + 1] = 0.f;
          }
        }
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

// A wait on an mbarrier that no thread or copy ever completes, bounded like every
// wait of the kernels above: it exercises the expiry path (record a code, return)
// without faulting or hanging the GPU.
__global__ void wait_selftest_kernel(long long cycles) {
  __shared__ __align__(8) uint64_t never;
  if (threadIdx.x == 0) {
    tc::mbar_init(&never, 1);
    tc::mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) tc::mbar_wait<true>(&never, 0, &g_attention_tc_error, kWaitSelfTestCode, cycles);
}

// Leftover rows: O = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c over the partials of the
// MT Q-tile CTAs and the KV splits of its (sequence, KV head) (the running max / exp-sum
// merge of "최적화 2편" section 3.3). One warp per leftover row; lane = 4 head dims.
__global__ void __launch_bounds__(256)
tree_attn_xmerge_kernel(const float* __restrict__ x_part, int B, int Hkv, int nsplit, int MT, int R, int N, int G,
                        const int32_t* __restrict__ L, int L_cap, uint16_t* __restrict__ O) {
  pdl_wait();
  pdl_trigger();
  const int row = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  if (row >= B * Hkv * R) return;
  const int r = row % R, kvh = (row / R) % Hkv, b = row / (R * Hkv);
  const int Lb = L[b];
  const bool valid = Lb >= 0 && Lb + N <= L_cap;
  const int parts = nsplit * MT;
  const float* p0 = x_part + ((size_t)(b * Hkv + kvh) * parts * kXMax + r) * (kD + 2);   // partial c at + c * kXMax
  float M = -INFINITY;
  for (int c = 0; c < parts; ++c) M = fmaxf(M, p0[(size_t)c * kXMax * (kD + 2) + kD]);
  float l = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
  for (int c = 0; c < parts; ++c) {
    const float* pc = p0 + (size_t)c * kXMax * (kD + 2);
    const float m = pc[kD];
    if (m == -INFINITY) continue;   // an empty partial need not have written its O
    const float w = exp2f(m - M);
    l += w * pc[kD + 1];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] += w * pc[lane + 32 * e];
  }
  const int qi = kRows * MT + r, Hq = Hkv * G;
  uint16_t* out = O + (((size_t)b * N + qi / G) * Hq + kvh * G + qi % G) * kD;
  const float inv = (valid && l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    uint16_t hv;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(hv) : "f"(o[e] * inv));
    out[lane + 32 * e] = hv;
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

MEDUSA_CHECK_TAKE(attention_tc_take_checks)

// Q-tile CTAs per (sequence, KV head): a short remainder of rows rides with the full tiles' CTAs.
cudaError_t attention_tc_take_error(uint32_t* out, cudaStream_t st) {
  static const uint32_t zero = 0;
  cudaError_t e =
      cudaMemcpyFromSymbolAsync(out, g_attention_tc_error, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbolAsync(g_attention_tc_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, st);
}

cudaError_t launch_wait_selftest(long long cycles, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(cycles);
  note_launches(1);
  return cudaGetLastError();
}

int attention_tc_mtiles(int NG) { return NG / kRows + ((NG % kRows != 0 && extra_rows(NG) == 0) ? 1 : 0); }
int attention_tc_ctas_x(int NG) { return attention_tc_mtiles(NG); }

// Workspace for the leftover rows' partials: (sequence, KV head, split, Q-tile CTA, row) x (D + 2) floats.
size_t attention_tc_xpart_bytes(const medusa_cfg& c, int nsplit) {
  const int NG = tree_shape(c).N * (c.Hq / c.Hkv);
  if (c.dtype != MEDUSA_BF16 || c.D != kD || extra_rows(NG) == 0) return 0;
  return (size_t)c.B * c.Hkv * nsplit * attention_tc_mtiles(NG) * kXMax * (kD + 2) * sizeof(float);
}

cudaError_t launch_attention_tc_xmerge(const medusa_cfg& c, int nsplit, const float* x_part, const int32_t* L, void* O,
                                       cudaStream_t st) {
  const TreeShape ts = tree_shape(c);
  const int G = c.Hq / c.Hkv, NG = ts.N * G, R = extra_rows(NG);
  if (R == 0) return cudaSuccess;
  const int rows = c.B * c.Hkv * R;
  launch_pdl(tree_attn_xmerge_kernel, (rows * 32 + 255) / 256, 256, 0, st, x_part, c.B, c.Hkv, nsplit,
             attention_tc_mtiles(NG), R, ts.N, G, L, c.L_cap, static_cast<uint16_t*>(O));
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_attention_tc(const medusa_cfg& c, int nsplit, int chunk, const void* Q, const void* Kc,
                                const void* Vc, const int32_t* L, const uint64_t* bits, float* o_part, float* ml_part,
                                float* x_part, void* O, cudaStream_t st, const PagedKV* paged) {
  const TreeShape ts = tree_shape(c);
  CUtensorMap tmK, tmV, tmKt, tmVt;
  if (paged) {   // pool [pages][Hkv][page_rows][D]; staged tree rows [B][Hkv][N][D]
    const uint64_t prow = (uint64_t)paged->num_pages * c.Hkv * paged->page_rows, trow = (uint64_t)c.B * c.Hkv * ts.N;
    if (!encode_tmap_2d_bf16(&tmK, Kc, prow, kD, kD * 2, 64, kKeys) ||
        !encode_tmap_2d_bf16(&tmV, Vc, prow, kD, kD * 2, 64, kKeys) ||
        !encode_tmap_2d_bf16(&tmKt, paged->Kt, trow, kD, kD * 2, 64, kKeys) ||
        !encode_tmap_2d_bf16(&tmVt, paged->Vt, trow, kD, kD * 2, 64, kKeys))
      return cudaErrorInvalidValue;
  } else {
    const uint64_t rows = (uint64_t)c.B * c.Hkv * c.L_cap;
    if (!encode_tmap_2d_bf16(&tmK, Kc, rows, kD, kD * 2, 64, kKeys) ||
        !encode_tmap_2d_bf16(&tmV, Vc, rows, kD, kD * 2, 64, kKeys))   // boxes of 128 keys x 64 head dims
      return cudaErrorInvalidValue;
    tmKt = tmK;
    tmVt = tmV;
  }
  const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)kD));
  const int NG = ts.N * (c.Hq / c.Hkv);
  const bool fold = extra_rows(NG) > 0;
  const int R = extra_rows(NG);
  auto kernel = !fold ? tree_attn_tc_kernel<0>
                      : R <= 2 ? tree_attn_tc_kernel<2> : R <= 4 ? tree_attn_tc_kernel<4> : tree_attn_tc_kernel<8>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_of(fold));
  if (e != cudaSuccess) return e;
  dim3 grid(attention_tc_mtiles(NG), c.Hkv * c.B, nsplit);
  launch_pdl(kernel, grid, threads_of(fold), smem_of(fold), st, tmK, tmV, tmKt, tmVt, static_cast<const uint16_t*>(Q),
             L, bits, ts.N, c.Hq, c.Hkv, c.L_cap, chunk, scale_log2, o_part, ml_part, static_cast<uint16_t*>(O),
             paged ? paged->block_table : static_cast<const int32_t*>(nullptr), paged ? paged->page_rows : 0,
             paged ? paged->num_pages : 0, x_part);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace medusa
