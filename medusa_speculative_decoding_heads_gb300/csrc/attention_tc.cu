// Tree attention on 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA).
//
// "Medusa 심층 아키텍처" (techknowgenie), section "트리 어텐션": every tree node
// attends to the committed KV cache and to its own ancestors (TreeMask
// equation), all nodes in one pass. Block-wise partials merge exactly through
// the running maximum and exp-sum ("최적화 2편" (beengineer500), section 3.3).
//
// One CTA runs two streams against one KV range of one sequence, in tiles of
// 128 keys. Paired CTAs hold two 128-row Q tiles (tree nodes x query heads) of
// the same KV head, and both streams consume every K/V tile. A CTA with a
// single Q tile splits the key tiles between its streams (even / odd) and
// merges the two partial results at the end. 11 warps:
//   warp 8  TMA producer: K and V tiles (two 64-column boxes each, 128-byte
//           swizzle) into a 2-stage (paired) or 3-stage ring; allocates TMEM.
//   warp 9  S issuer: S = Q K^T (Q and K from shared memory) into the
//           stream's S tile in TMEM.
//   warp 10 PV issuer: O += P V with P read from TMEM and V as an MN-major
//           shared-memory operand. Two issuing warps keep the tensor pipe fed
//           while either one waits on a barrier.
//   warps 0-3 / 4-7  one softmax warpgroup per stream: thread = query row =
//           TMEM lane, a whole 128-key row per thread, so no exchange between
//           warps; the running max moves (and O is rescaled) only on a jump of
//           more than 2^8.
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
constexpr int kOperand = 2 * kHalf;         // a 128 x 128 bf16 tile: Q, K or V (32 KB)
constexpr int kStage = 2 * kOperand;        // K + V of one key tile
constexpr int kSmemBytes = 7 * kOperand + 1024;   // two Q tiles + 2 stages, or one Q tile + 3 stages
constexpr uint32_t kTmemCols = 512;
constexpr int kGroupThreads = 128;
constexpr int kProducerWarp = 8;
constexpr int kMmaSWarp = 9;    // issues S = Q K^T
constexpr int kMmaPWarp = 10;   // issues O += P V
constexpr int kThreads = 352;
constexpr int kSortMax = 256;   // batches up to this size are taken longest sequence first

// TMEM columns: per stream s an S tile (128 f32 columns; P is written over it as
// bf16 pairs, keys 0..63 in columns 0..31 and keys 64..127 in columns 64..95)
// and an O accumulator (128 f32 columns).
__host__ __device__ constexpr uint32_t col_S(int s) { return 128u * s; }
__host__ __device__ constexpr uint32_t col_O(int s) { return 256u + 128u * s; }

// The running maximum is only moved (and O rescaled) when a tile's maximum
// exceeds it by more than this many binary orders of magnitude; in between, P
// entries stay below 2^kLazy, far inside bf16/f32 range.
constexpr float kLazy = 8.f;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Masks 64 scores of keys [k0, k0 + 64) of a tile: a key is visible when it is
// inside the tile's range and (tree tiles) its bit is set in the node's mask word.
__device__ __forceinline__ void mask64(uint32_t* v, int k0, int nkeys, bool tree, uint64_t word) {
  if (tree || k0 + 64 > nkeys) {
#pragma unroll
    for (int k = 0; k < 64; ++k)
      if (!(k0 + k < nkeys && (!tree || ((word >> k) & 1ull)))) v[k] = __float_as_uint(-INFINITY);
  }
}
__device__ __forceinline__ float max64(const uint32_t* v) {
  float m8[8];
#pragma unroll
  for (int a = 0; a < 8; ++a) m8[a] = __uint_as_float(v[a]);
#pragma unroll
  for (int k = 8; k < 64; ++k) m8[k & 7] = fmaxf(m8[k & 7], __uint_as_float(v[k]));
  return fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
}
// p = 2^(s * scale_log2 - m) for 64 scores, packed as 32 bf16 pairs; returns their sum.
__device__ __forceinline__ float exp64(const uint32_t* v, float scale_log2, float neg_m, uint32_t* pk) {
  float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    const float p0 = tc::ex2(fmaf(__uint_as_float(v[2 * k]), scale_log2, neg_m));
    const float p1 = tc::ex2(fmaf(__uint_as_float(v[2 * k + 1]), scale_log2, neg_m));
    l4[k & 3] += p0 + p1;
    pk[k] = pack_bf16x2(p0, p1);
  }
  return (l4[0] + l4[1]) + (l4[2] + l4[3]);
}

struct Bars {
  uint64_t kv_full[3], kv_empty[3], s_full[2], p_full[2], p_free[2], ml_bar;
  uint32_t tmem_slot;
};

// One CTA's work; PAIRED selects the mode (two Q tiles sharing every K/V tile, or
// one Q tile whose key tiles alternate between the streams).
template <bool PAIRED>
__device__ __forceinline__ void attn_cta(const CUtensorMap* tmK, const CUtensorMap* tmV, const uint16_t* __restrict__ Q,
                                         const int32_t* __restrict__ L, const uint64_t* __restrict__ bits, int N,
                                         int Hq, int Hkv, int L_cap, int chunk, float scale_log2,
                                         float* __restrict__ o_part, float* __restrict__ ml_part,
                                         uint16_t* __restrict__ O, uint8_t* sm, Bars& bar, int b, int kvh, int xt,
                                         int split, int nsplit) {
  uint64_t* kv_full = bar.kv_full;
  uint64_t* kv_empty = bar.kv_empty;
  uint64_t* s_full = bar.s_full;
  uint64_t* p_full = bar.p_full;
  uint64_t* p_free = bar.p_free;
  uint64_t& ml_bar = bar.ml_bar;
  uint32_t& tmem_slot = bar.tmem_slot;
  uint32_t* err = &g_attention_tc_error;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = Hq / Hkv, NG = N * G;
  // Two streams per CTA. Paired: Q tiles 2x and 2x+1 of one KV head, both against
  // every key tile. Split: one Q tile, stream s taking key tiles j with j % 2 == s.
  constexpr bool paired = PAIRED;
  constexpr int nst = paired ? 2 : 3;                     // K/V ring stages
  uint8_t* ring = sm + (paired ? 2 : 1) * kOperand;       // Q tile(s) first
  const int Lb = L[b];
  const bool valid = Lb >= 0 && Lb + N <= L_cap;
  const int k_begin = split * chunk;
  const int k_end = valid ? min(Lb, k_begin + chunk) : 0;
  const int ptiles = k_end > k_begin ? (k_end - k_begin + kKeys - 1) / kKeys : 0;
  const int ntiles = ptiles + ((valid && split == nsplit - 1) ? 1 : 0);   // N <= 128: one tree tile
  const int nitems = paired ? 2 * ntiles : ntiles;                         // (stream, key tile) pairs

  // Softmax thread: stream s = warpgroup, row = TMEM lane.
  const bool smx = warp < kProducerWarp;
  const int s = (warp >> 2) & 1;
  const int row = 32 * (warp & 3) + lane;
  const int mt = 2 * xt + (paired ? s : 0);
  const int qi = mt * kRows + row;
  const bool row_ok = smx && qi < NG;
  const int node = row_ok ? qi / G : 0;
  const int qh = kvh * G + (row_ok ? qi % G : 0);
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;

  if (ntiles == 0) {
    // Nothing to attend to in this range: an empty partial (or zeros for an
    // invalid sequence), without touching TMEM or the barriers.
    if (row_ok && (paired || s == 0)) {
      if (nsplit == 1) {
        uint4* op = reinterpret_cast<uint4*>(O + (((size_t)b * N + node) * Hq + qh) * kD);
#pragma unroll
        for (int x = 0; x < kD / 8; ++x) op[x] = make_uint4(0, 0, 0, 0);
      } else {
        const size_t orow = (((size_t)b * nsplit + split) * N + node) * Hq + qh;
        ml_part[2 * orow] = -INFINITY;
        ml_part[2 * orow + 1] = 0.f;
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < 3; ++s) {
      tc::mbar_init(&kv_full[s], 1);
      tc::mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&s_full[s], 1);
      tc::mbar_init(&p_full[s], kGroupThreads);
      tc::mbar_init(&p_free[s], 1);
    }
    tc::mbar_init(&ml_bar, 2 * kGroupThreads);
    tc::mbar_fence_init();
  }
  if (warp == kProducerWarp) tc::tmem_alloc(&tmem_slot, kTmemCols);

  if (smx) {
    // Q rows into shared memory, K-major with the 128-byte swizzle (16-byte chunk
    // c of row r at chunk c ^ (r & 7)). Paired: each stream its own tile; split:
    // stream s stages head dims [64s, 64s + 64) of the one tile.
    const uint4* qp = reinterpret_cast<const uint4*>(Q + (((size_t)b * N + node) * Hq + qh) * kD);
    uint8_t* qs = sm + (paired ? s : 0) * kOperand + row * 128;
    for (int h = paired ? 0 : s; h < (paired ? 2 : s + 1); ++h)
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = row_ok ? qp[h * 8 + c] : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(qs + h * kHalf + ((c ^ (row & 7)) << 4)) = v;
      }
    tc::fence_proxy_async();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      const int head_row = (b * Hkv + kvh) * L_cap;
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int st = j % nst;
        if (j >= nst && !tc::mbar_wait<true>(&kv_empty[st], ((j / nst) - 1) & 1, err, 1)) break;
        const int row0 = j < ptiles ? head_row + k_begin + j * kKeys : head_row + Lb;
        uint8_t* dst = ring + st * kStage;
        tc::mbar_arrive_expect(&kv_full[st], kStage);
        tc::tma_load_2d(dst, tmK, 0, row0, &kv_full[st]);
        tc::tma_load_2d(dst + kHalf, tmK, 64, row0, &kv_full[st]);
        tc::tma_load_2d(dst + kOperand, tmV, 0, row0, &kv_full[st]);
        tc::tma_load_2d(dst + kOperand + kHalf, tmV, 64, row0, &kv_full[st]);
        issued = j + 1;
      }
      // Drain: never leave the CTA with tile loads still landing in shared memory.
      for (int j = issued > nst ? issued - nst : 0; j < issued; ++j)
        tc::mbar_wait(&kv_full[j % nst], (j / nst) & 1, err, 128);
    }
  } else if (warp == kMmaSWarp) {
    // ------------------------------------------------------------------ S issuer
    // The whole warp walks the schedule (uniform waits); one elected lane issues.
    // Item w = (stream w % 2, key tile w / 2 paired or w split).
    constexpr uint32_t idS = tc::idesc_bf16_f32(kRows, kKeys, 0, 0);
    const uint64_t dQ = tc::sw128_desc(tc::saddr(sm), 16, 1024);
    const uint64_t dK = tc::sw128_desc(tc::saddr(ring), 16, 1024);
    for (int w = 0; w < nitems; ++w) {
      const int ss = w & 1, j = paired ? (w >> 1) : w, st = j % nst;
      bool ok = true;
      if (!paired || ss == 0) ok = tc::mbar_wait<true>(&kv_full[st], (j / nst) & 1, err, 2);
      // the S tile of stream ss still holds P of its previous item until that PV completes
      if (ok && w >= 2) ok = tc::mbar_wait<true>(&p_free[ss], ((w >> 1) - 1) & 1, err, 4);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc::fence_after();
      if (tc::elect_one()) {
        const uint64_t a0 = dQ + (uint64_t)((paired ? ss * kOperand : 0) >> 4);
        const uint64_t b0 = dK + (uint64_t)((st * kStage) >> 4);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
          tc::mma_bf16(tmem + col_S(ss), a0 + off, b0 + off, idS, kk > 0);
        }
        tc::commit(&s_full[ss]);
      }
      __syncwarp();
    }
  } else if (warp == kMmaPWarp) {
    // ------------------------------------------------------------------ PV issuer
    // S(w) completed before P(w) was released, so the completion of PV(w) also
    // covers every read of the stage's K tile.
    constexpr uint32_t idPV = tc::idesc_bf16_f32(kRows, kD, 0, 1);
    const uint64_t dV = tc::sw128_desc(tc::saddr(ring + kOperand), kHalf, 1024);   // MN-major: LBO = 64-column half
    for (int w = 0; w < nitems; ++w) {
      const int ss = w & 1, j = paired ? (w >> 1) : w, st = j % nst;
      const bool ok = tc::mbar_wait<true>(&p_full[ss], (w >> 1) & 1, err, 8);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc::fence_after();
      if (tc::elect_one()) {
        const uint64_t b0 = dV + (uint64_t)((st * kStage) >> 4);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          tc::mma_bf16_tmem_a(tmem + col_O(ss), tmem + col_S(ss) + kk * 8 + (kk >= 4 ? 32 : 0),
                              b0 + (uint64_t)((kk * 2048) >> 4), idPV, (w >= 2 || kk > 0) ? 1 : 0);
        tc::commit(&p_free[ss]);
        if (!paired || ss == 1) tc::commit(&kv_empty[st]);
      }
      __syncwarp();
    }
  } else if (smx) {
    // ------------------------------------------------------------------ softmax warpgroups
    const uint32_t tS = tmem + col_S(s) + lane_base, tO = tmem + col_O(s) + lane_base;
    const uint64_t nb0 = bits[2 * node], nb1 = bits[2 * node + 1];
    float m_run = -INFINITY, l_run = 0.f;
    int n = 0;   // items of this stream processed
    bool ok = true;
    for (int w = s; w < nitems; w += 2, ++n) {
      ok = tc::mbar_wait(&s_full[s], n & 1, err, 16);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc::fence_after();
      const int j = paired ? (w >> 1) : w;
      const bool tree = j >= ptiles;
      const int nkeys = tree ? N : min(kKeys, k_end - (k_begin + j * kKeys));
      uint32_t v[64], pk[32];
      // pass 1: row maximum over the 128 scores (two halves of 64)
      tc::tmem_ld32(tS, v);
      tc::tmem_ld32(tS + 32, v + 32);
      tc::tmem_wait_ld();
      mask64(v, 0, nkeys, tree, nb0);
      float mx = max64(v);
      tc::tmem_ld32(tS + 64, v);
      tc::tmem_ld32(tS + 96, v + 32);
      tc::tmem_wait_ld();
      mask64(v, 64, nkeys, tree, nb1);
      mx = fmaxf(mx, max64(v));

      const float m_tile = mx * scale_log2;
      float corr = 1.f;
      if (m_tile > m_run + kLazy) {   // also taken on the first visible tile (m_run = -inf)
        corr = tc::ex2(m_run - m_tile);
        m_run = m_tile;
      }
      const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
      float l_tile = 0.f;
      // pass 2: keys 64..127 are still in registers; their P goes to columns
      // 64..95 (already read), then keys 0..63 are reloaded and their P goes to 0..31.
      if (row_ok) {
        l_tile = exp64(v, scale_log2, neg_m, pk);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) pk[k] = 0u;
      }
      tc::tmem_st32(tS + 64, pk);
      tc::tmem_ld32(tS, v);
      tc::tmem_ld32(tS + 32, v + 32);
      tc::tmem_wait_ld();
      mask64(v, 0, nkeys, tree, nb0);
      if (row_ok) {
        l_tile += exp64(v, scale_log2, neg_m, pk);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) pk[k] = 0u;
      }
      l_run = l_run * corr + l_tile;
      // S(w) was issued after PV of this stream's previous item completed, so O is
      // quiescent here and can be rescaled before P(w) is released.
      if (n >= 1 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t ov[32];
          tc::tmem_ld32(tO + c * 32, ov);
          tc::tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 32; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * corr);
          tc::tmem_st32(tO + c * 32, ov);
        }
      }
      // P of keys 0..63 over columns 0..31 of this row's S tile (only this thread reads the row).
      tc::tmem_st32(tS, pk);
      tc::tmem_wait_st();
      tc::fence_before();
      tc::mbar_arrive(&p_full[s]);
    }
    // The last PV of this stream: its (n-1)-th completion of p_free.
    if (ok && n > 0) ok = tc::mbar_wait(&p_free[s], (n - 1) & 1, err, 256);
    const bool have = __all_sync(0xffffffffu, ok) && n > 0;
    tc::fence_after();

    if (paired) {
      // Each stream owns its rows: normalise (or write the split's partial) directly.
      const float inv = (have && l_run > 0.f) ? 1.f / l_run : 0.f;
      const size_t orow = nsplit == 1 ? (((size_t)b * N + node) * Hq + qh)
                                      : ((((size_t)b * nsplit + split) * N + node) * Hq + qh);
#pragma unroll 1
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t ov[32];
        if (have) {   // warp-uniform: the TMEM load is a collective of the warp
          tc::tmem_ld32(tO + c * 32, ov);
          tc::tmem_wait_ld();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) ov[x] = 0u;
        }
        if (!row_ok) continue;
        if (nsplit == 1) {
          uint16_t* op = O + orow * kD + c * 32;
#pragma unroll
          for (int x = 0; x < 32; x += 8)
            *reinterpret_cast<uint4*>(op + x) =
                make_uint4(pack_bf16x2(__uint_as_float(ov[x]) * inv, __uint_as_float(ov[x + 1]) * inv),
                           pack_bf16x2(__uint_as_float(ov[x + 2]) * inv, __uint_as_float(ov[x + 3]) * inv),
                           pack_bf16x2(__uint_as_float(ov[x + 4]) * inv, __uint_as_float(ov[x + 5]) * inv),
                           pack_bf16x2(__uint_as_float(ov[x + 6]) * inv, __uint_as_float(ov[x + 7]) * inv));
        } else {
          float* op = o_part + orow * kD + c * 32;
#pragma unroll
          for (int x = 0; x < 32; x += 4)
            *reinterpret_cast<float4*>(op + x) = make_float4(__uint_as_float(ov[x]), __uint_as_float(ov[x + 1]),
                                                             __uint_as_float(ov[x + 2]), __uint_as_float(ov[x + 3]));
        }
      }
      if (row_ok && nsplit > 1) {
        ml_part[2 * orow] = have ? m_run : -INFINITY;
        ml_part[2 * orow + 1] = have ? l_run : 0.f;
      }
    } else {
      // Split: merge the two streams' partials of the same rows. The exchange
      // lives in the Q tile's shared memory, idle once every MMA has completed.
      // First phase of ml_bar: both streams are past their last PV, so every MMA
      // (each S was issued before the last PV) has stopped reading the Q tile.
      tc::mbar_arrive(&ml_bar);
      tc::mbar_wait(&ml_bar, 0, err, 512);
      float* xm = reinterpret_cast<float*>(sm);
      float* xl = xm + 2 * kRows;
      xm[s * kRows + row] = have ? m_run : -INFINITY;
      xl[s * kRows + row] = have ? l_run : 0.f;
      tc::mbar_arrive(&ml_bar);
      tc::mbar_wait(&ml_bar, 1, err, 512);
      const float m0 = xm[row], m1 = xm[kRows + row];
      const float M = fmaxf(m0, m1);
      const float w0 = m0 == -INFINITY ? 0.f : tc::ex2(m0 - M);
      const float w1 = m1 == -INFINITY ? 0.f : tc::ex2(m1 - M);
      const float l_tot = xl[row] * w0 + xl[kRows + row] * w1;
      // thread of stream s finalises head dims [64s, 64s + 64)
      const uint32_t c0 = s * 64;
      float acc[64];
#pragma unroll
      for (int x = 0; x < 64; ++x) acc[x] = 0.f;
#pragma unroll
      for (int src = 0; src < 2; ++src) {
        const float wsrc = src == 0 ? w0 : w1;
        if (__any_sync(0xffffffffu, wsrc != 0.f)) {   // a stream with no items has an unwritten O
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t ov[32];
            tc::tmem_ld32(tmem + col_O(src) + lane_base + c0 + c * 32, ov);
            tc::tmem_wait_ld();
            if (wsrc != 0.f) {
#pragma unroll
              for (int x = 0; x < 32; ++x) acc[c * 32 + x] += __uint_as_float(ov[x]) * wsrc;
            }
          }
        }
      }
      if (nsplit == 1) {
        const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
        if (row_ok) {
          uint16_t* op = O + (((size_t)b * N + node) * Hq + qh) * kD + c0;
#pragma unroll
          for (int x = 0; x < 64; x += 8)
            *reinterpret_cast<uint4*>(op + x) = make_uint4(
                pack_bf16x2(acc[x] * inv, acc[x + 1] * inv), pack_bf16x2(acc[x + 2] * inv, acc[x + 3] * inv),
                pack_bf16x2(acc[x + 4] * inv, acc[x + 5] * inv), pack_bf16x2(acc[x + 6] * inv, acc[x + 7] * inv));
        }
      } else if (row_ok) {
        const size_t orow = (((size_t)b * nsplit + split) * N + node) * Hq + qh;
        float* op = o_part + orow * kD + c0;
#pragma unroll
        for (int x = 0; x < 64; x += 4)
          *reinterpret_cast<float4*>(op + x) = make_float4(acc[x], acc[x + 1], acc[x + 2], acc[x + 3]);
        if (s == 0) {
          ml_part[2 * orow] = M;
          ml_part[2 * orow + 1] = l_tot;
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

__global__ void __launch_bounds__(kThreads, 1)
tree_attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const uint16_t* __restrict__ Q, const int32_t* __restrict__ L, const uint64_t* __restrict__ bits,
                    int N, int Hq, int Hkv, int L_cap, int chunk, int mtiles, float scale_log2,
                    float* __restrict__ o_part, float* __restrict__ ml_part, uint16_t* __restrict__ O) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) Bars bar;
  __shared__ int seq;
  // Launch order: x = KV split (fastest), y = (sequence rank, KV head), z = Q tile
  // pair. Paired CTAs (the larger units) come first, and sequences are taken
  // longest first, so that the block scheduler's tail holds the smallest units.
  const int xt = blockIdx.z, split = blockIdx.x, nsplit = gridDim.x;
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
  if (2 * xt + 1 < mtiles)
    attn_cta<true>(&tmK, &tmV, Q, L, bits, N, Hq, Hkv, L_cap, chunk, scale_log2, o_part, ml_part, O, sm, bar, b, kvh,
                   xt, split, nsplit);
  else
    attn_cta<false>(&tmK, &tmV, Q, L, bits, N, Hq, Hkv, L_cap, chunk, scale_log2, o_part, ml_part, O, sm, bar, b, kvh,
                    xt, split, nsplit);
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
int attention_tc_ctas_x(int NG) { return (attention_tc_mtiles(NG) + 1) / 2; }

cudaError_t launch_attention_tc(const medusa_cfg& c, int nsplit, int chunk, const void* Q, const void* Kc,
                                const void* Vc, const int32_t* L, const uint64_t* bits, float* o_part, float* ml_part,
                                void* O, cudaStream_t st) {
  const TreeShape ts = tree_shape(c);
  const uint64_t rows = (uint64_t)c.B * c.Hkv * c.L_cap;
  CUtensorMap tmK, tmV;
  if (!encode_tmap_2d_bf16(&tmK, Kc, rows, kD, kD * 2, 64, kKeys) ||
      !encode_tmap_2d_bf16(&tmV, Vc, rows, kD, kD * 2, 64, kKeys))   // boxes of 128 keys x 64 head dims
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tree_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)kD));
  const int NG = ts.N * (c.Hq / c.Hkv);
  dim3 grid(nsplit, c.Hkv * c.B, attention_tc_ctas_x(NG));
  tree_attn_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(tmK, tmV, static_cast<const uint16_t*>(Q), L, bits, ts.N, c.Hq,
                                                     c.Hkv, c.L_cap, chunk, attention_tc_mtiles(NG), scale_log2,
                                                     o_part, ml_part, static_cast<uint16_t*>(O));
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace medusa
