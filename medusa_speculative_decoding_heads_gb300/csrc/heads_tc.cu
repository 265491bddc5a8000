// Medusa heads on tcgen05 tensor cores with TMA-fed weight streaming.
//
// "Medusa 심층 아키텍처" (techknowgenie), section "잔차 블록(Residual Block)을 포함한
// Medusa 헤드 구조", equations
// h_t^(k) = SiLU(h_t W_res^(k)) + h_t and p_k = softmax(h_t^(k) W_head^(k)).
//
// Both projections are weight-streaming GEMVs: every weight byte is read once
// and meets all B vectors of the batch. Swap-AB: 128 weight rows are the MMA's
// M dimension (A operand, K-major, straight from the row-major weights), the
// batch vectors are the N dimension (B operand). The vocab projection consumes
// the f32 residual as bf16 hi and lo vectors, i.e. N = 2 * NB columns; the two
// columns of a sequence are added in the epilogue. When every head shares one
// frozen vocab projection (the same section's note on W_head^(k)), all heads'
// hi/lo vectors form one B operand and the projection is streamed once.
//
// Persistent CTAs (one per SM) walk a static list of work units (head, 128-row
// tile, k range). The vocab projection takes whole tiles round robin. The
// d x d residual layer has too few tiles for that to balance (e.g. 128 tiles
// of 64 chunks on 152 SMs), so it splits the flat (tile, chunk) sequence into
// equal contiguous ranges, one per CTA (a stream-K split): a range that
// crosses tiles yields one unit per tile, each writing its partial sums to the
// slot numbered by its position among the CTAs that share the tile. 6 warps:
//   warp 4  TMA producer: 64-wide k chunks of the weight tile and of the vector
//           tile into a deep shared-memory ring (128-byte swizzle).
//   warp 5  MMA issuer: four K=16 MMAs per chunk into one of two TMEM
//           accumulators; commits free ring slots and completed units.
//   warps 0-3  epilogue: thread i = weight row i = TMEM lane i; adds the hi/lo
//           columns and writes f32 outputs (coalesced across the warp).
// All mbarrier waits are bounded (see tc_common.cuh).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "tc_common.cuh"

namespace medusa {

__device__ uint32_t g_heads_tc_error = 0;

namespace {

constexpr int kRowsTile = 128;
constexpr int kChunkK = 64;
constexpr int kATile = kRowsTile * 128;     // 16 KB: 128 rows x 64 bf16
constexpr int kSmemBudget = 200 * 1024;
// Columns per TMEM accumulator (two accumulators; the allocation is a power of two).
__host__ __device__ constexpr uint32_t acc_cols(int ncol) { return ncol <= 64 ? 64u : (ncol <= 128 ? 128u : 256u); }

template <int NCOL>
struct HeadsGeom {
  static constexpr int kXTile = NCOL * 128;
  static constexpr int kStage = kATile + kXTile;
  static constexpr int kStages = (kSmemBudget / kStage) > 12 ? 12 : (kSmemBudget / kStage);
  static constexpr int kSmem = kStages * kStage + 1024;
};

// First CTA of a stream-K split whose chunk range reaches flat chunk x, for T
// chunks over P CTAs (CTA c owns [c T / P, (c + 1) T / P)): the largest c with
// floor(c T / P) <= x.
__host__ __device__ __forceinline__ int stream_first_cta(long long x, long long T, long long P) {
  return (int)(((x + 1) * P + T - 1) / T - 1);
}

// The i-th work unit of this CTA: head g, tile t, chunks [c0, c1), output slot.
// Round robin: unit u = blockIdx.x + i * gridDim.x of G * tiles * ksplit, slot = k-split.
// Stream: the i-th tile that this CTA's chunk range touches.
template <bool kStream>
__device__ __forceinline__ bool unit_of(int i, int G, int tiles, int nchunks, int nk, int ksplit, int& g, int& t,
                                        int& c0, int& c1, int& slot) {
  if (!kStream) {
    const int u = blockIdx.x + i * gridDim.x;
    if (u >= G * tiles * ksplit) return false;
    slot = u % ksplit;
    t = (u / ksplit) % tiles;
    g = u / (ksplit * tiles);
    c0 = slot * nk;
    c1 = min(nchunks, c0 + nk);
    return true;
  }
  const long long T = (long long)G * tiles * nchunks, P = gridDim.x;
  const long long f0 = blockIdx.x * T / P, f1 = (blockIdx.x + 1) * T / P;
  const long long tf = f0 / nchunks + i, s0 = tf * nchunks;
  if (s0 >= f1) return false;
  c0 = (int)((f0 > s0 ? f0 : s0) - s0);
  c1 = (int)((f1 < s0 + nchunks ? f1 : s0 + nchunks) - s0);
  g = (int)(tf / tiles);
  t = (int)(tf % tiles);
  slot = (int)blockIdx.x - stream_first_cta(s0, T, P);
  return true;
}

// out[slot][b][g][r] = sum_k A[g*rows + r][k] * X[g*x_rows + col(b)][k] over the
// unit's k range; col(b) = b (+ NB for the lo part when HILO). The residual
// layer (!HILO) uses the stream-K schedule, the vocab projection round robin.
//
// The X block of a unit holds nxh head blocks of HB columns each (one, except
// when all heads share one vocab projection: then one MMA of N = nxh * HB
// columns, rounded up with zero rows, serves every head from a single stream
// of the weights). Within a head block, column j < HB / 2 is sequence j's hi
// part and j + HB / 2 its lo part (HILO), or column j is sequence j (!HILO).
// Output element (slot, b, head, r) goes to
// out + slot * out_split_stride + b * bstride + (g + head) * hstride + r.
// a_head_rows is the row offset of head g in A (0 when the heads share A).
template <int NCOL, bool HILO, int HB>
__global__ void __launch_bounds__(192, 1)
heads_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmX, int rows, int G,
                int a_head_rows, int x_rows, int nchunks, int nk, int ksplit, int B, int nxh, float* __restrict__ out,
                size_t out_split_stride, size_t bstride, size_t hstride) {
  constexpr uint32_t kAccCols = acc_cols(NCOL);
  static_assert(NCOL < 64 ? HB == NCOL : 64 % HB == 0, "head blocks must tile the 64-column passes");
  pdl_trigger();
  using Geo = HeadsGeom<NCOL>;
  constexpr int S = Geo::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* As = sm;                       // [S][16 KB]
  uint8_t* Xs = sm + S * kATile;          // [S][NCOL * 128]
  __shared__ __align__(8) uint64_t full[S], empty[S], acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_slot;
  uint32_t* err = &g_heads_tc_error;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool kStream = !HILO;
  const int tiles = (rows + kRowsTile - 1) / kRowsTile;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&acc_full[a], 1);
      tc::mbar_init(&acc_empty[a], 128);
    }
    tc::mbar_fence_init();
  }
  if (warp == 4) tc::tmem_alloc(&tmem_slot, 2 * kAccCols);   // 128, 256 or 512 columns
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_slot;
  if (warp == 4 && lane == 0) {
    // Warm L2 with the weight boxes of this CTA's first S chunks while the
    // previous kernel finishes (a prefetch is only a hint, so it cannot observe
    // stale data; the real loads come after the wait below).
    int n = 0, g, t, c0, c1, slot;
    for (int i = 0; n < S && unit_of<kStream>(i, G, tiles, nchunks, nk, ksplit, g, t, c0, c1, slot); ++i)
      for (int c = c0; c < c1 && n < S; ++c, ++n)
        tc::tma_prefetch_2d(&tmA, c * kChunkK, g * a_head_rows + t * kRowsTile);
  }
  pdl_wait();   // the setup above overlaps the previous kernel's tail; no global access before this

  if (warp == 4) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      int it = 0, g, t, c0, c1, slot;
      bool ok = true;
      for (int i = 0; ok && unit_of<kStream>(i, G, tiles, nchunks, nk, ksplit, g, t, c0, c1, slot); ++i) {
        for (int c = c0; c < c1; ++c, ++it) {
          const int s = it % S;
          if (it >= S && !tc::mbar_wait(&empty[s], ((it / S) - 1) & 1, err, 1)) {
            ok = false;
            break;
          }
          tc::mbar_arrive_expect(&full[s], kATile + Geo::kXTile);
          tc::tma_load_2d(As + s * kATile, &tmA, c * kChunkK, g * a_head_rows + t * kRowsTile, &full[s]);
          tc::tma_load_2d(Xs + s * Geo::kXTile, &tmX, c * kChunkK, g * x_rows, &full[s]);
        }
      }
      // Drain the loads still in flight before the CTA can exit.
      for (int j = it > S ? it - S : 0; j < it; ++j) tc::mbar_wait(&full[j % S], (j / S) & 1, err, 2);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kRowsTile, NCOL, 0, 0);
      int it = 0, ui = 0, g, t, c0, c1, slot;
      bool ok = true;
      for (; ok && unit_of<kStream>(ui, G, tiles, nchunks, nk, ksplit, g, t, c0, c1, slot); ++ui) {
        const int a = ui & 1;
        if (ui >= 2 && !tc::mbar_wait(&acc_empty[a], ((ui >> 1) - 1) & 1, err, 4)) break;
        tc::fence_after();
        const uint32_t dacc = tmem + a * kAccCols;
        for (int c = c0; c < c1; ++c, ++it) {
          const int s = it % S;
          if (!tc::mbar_wait(&full[s], (it / S) & 1, err, 8)) {
            ok = false;
            break;
          }
          tc::fence_after();
          const uint32_t aa = tc::saddr(As + s * kATile), xa = tc::saddr(Xs + s * Geo::kXTile);
#pragma unroll
          for (int kk = 0; kk < kChunkK / 16; ++kk)
            tc::mma_bf16(dacc, tc::sw128_desc(aa + kk * 32, 16, 1024), tc::sw128_desc(xa + kk * 32, 16, 1024), idesc,
                         (c > c0 || kk > 0) ? 1 : 0);
          tc::commit(&empty[s]);
        }
        tc::commit(&acc_full[a]);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const int i = threadIdx.x;
    int g, t, c0, c1, slot;
    for (int ui = 0; unit_of<kStream>(ui, G, tiles, nchunks, nk, ksplit, g, t, c0, c1, slot); ++ui) {
      const int a = ui & 1;
      const bool ok = tc::mbar_wait(&acc_full[a], (ui >> 1) & 1, err, 16);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc::fence_after();
      const int r = t * kRowsTile + i;
      float* ob = out + (size_t)slot * out_split_stride + (size_t)g * hstride + r;
      constexpr int kWin = NCOL < 64 ? NCOL : 64;       // columns per pass (two 32-column loads)
      constexpr int kWins = (NCOL + 63) / 64;
      constexpr int kHalf = HILO ? HB / 2 : HB;         // sequences per head block
      constexpr int kPerWin = NCOL < 64 ? 1 : 64 / HB;  // head blocks per pass
#pragma unroll 1
      for (int w = 0; w < kWins; ++w) {
        uint32_t v[64];
        tc::tmem_ld32(tmem + a * kAccCols + lane_base + 64 * w, v);
        if (kWin > 32) tc::tmem_ld32(tmem + a * kAccCols + lane_base + 64 * w + 32, v + 32);
        tc::tmem_wait_ld();
        if (w == kWins - 1) {   // the accumulator is free once its last columns are in registers
          tc::fence_before();
          tc::mbar_arrive(&acc_empty[a]);
        }
        if (r < rows) {
#pragma unroll
          for (int j = 0; j < kWin; ++j) {
            const int cc = j % HB, head = w * kPerWin + j / HB;
            if (cc < kHalf && cc < B && head < nxh) {
              float x = __uint_as_float(v[j]);
              if (HILO) x += __uint_as_float(v[j + kHalf]);
              ob[(size_t)cc * bstride + (size_t)head * hstride] = x;
            }
          }
        }
      }
    }
  }

  tc::fence_before();
  __syncthreads();
  if (warp == 4) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, 2 * kAccCols);
  }
}

// r = h + SiLU(sum_slots pre + bias); X2[k][n][o] = bf16(r), X2[k][NB+n][o] = bf16(r - bf16(r)).
// Output o of head k lies in tile k * tiles + o / 128 of the residual layer's
// stream-K split (nchunks chunks per tile over P CTAs); its partial sums sit
// in the slots of the CTAs whose ranges touch that tile, added in slot order.
__global__ void residual_pack_tc_kernel(const float* __restrict__ part, int tiles, int nchunks, int P,
                                        const uint16_t* __restrict__ h, const uint16_t* __restrict__ bias,
                                        uint16_t* __restrict__ X2, int B, int NB, int K, int d) {
  pdl_wait();
  pdl_trigger();
  // four consecutive outputs o per thread: 16-byte partial loads, 8-byte stores
  const int d4 = d >> 2;
  const size_t total = (size_t)K * NB * d4;
  const size_t split_stride = (size_t)B * K * d;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int o = (int)(e % d4) * 4;
    const int n = (int)((e / d4) % NB);
    const int k = (int)(e / ((size_t)d4 * NB));
    uint32_t hi2[2] = {0u, 0u}, lo2[2] = {0u, 0u};
    if (n < B) {
      float pre[4] = {0.f, 0.f, 0.f, 0.f};
      const float* pp = part + ((size_t)n * K + k) * d + o;
      // 32-bit form of stream_first_cta (the host checks that (T + 1) * P fits)
      const uint32_t T = (uint32_t)(K * tiles * nchunks), tf = (uint32_t)(k * tiles + o / kRowsTile);
      const uint32_t x0 = tf * nchunks, x1 = x0 + nchunks - 1;
      const int nslots = (int)(((x1 + 1) * (uint32_t)P + T - 1) / T - ((x0 + 1) * (uint32_t)P + T - 1) / T) + 1;
      for (int s = 0; s < nslots; ++s) {
        const float4 v = *reinterpret_cast<const float4*>(pp + s * split_stride);
        pre[0] += v.x;
        pre[1] += v.y;
        pre[2] += v.z;
        pre[3] += v.w;
      }
      const uint2 hv = *reinterpret_cast<const uint2*>(h + (size_t)n * d + o);
      uint2 bv = make_uint2(0u, 0u);
      if (bias) bv = *reinterpret_cast<const uint2*>(bias + (size_t)k * d + o);
      const uint32_t hw[2] = {hv.x, hv.y}, bw[2] = {bv.x, bv.y};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint16_t hq = (uint16_t)(hw[q >> 1] >> (16 * (q & 1)));
        const uint16_t bq = (uint16_t)(bw[q >> 1] >> (16 * (q & 1)));
        float x = pre[q];
        if (bias) x += bf16_to_f32(bq);
        const float r = bf16_to_f32(hq) + x / (1.f + expf(-x));
        const uint16_t rh = f32_to_bf16(r);
        const uint16_t rl = f32_to_bf16(r - bf16_to_f32(rh));
        hi2[q >> 1] |= (uint32_t)rh << (16 * (q & 1));
        lo2[q >> 1] |= (uint32_t)rl << (16 * (q & 1));
      }
    }
    uint16_t* xk = X2 + (size_t)k * 2 * NB * d;
    *reinterpret_cast<uint2*>(xk + (size_t)n * d + o) = make_uint2(hi2[0], hi2[1]);
    *reinterpret_cast<uint2*>(xk + (size_t)(NB + n) * d + o) = make_uint2(lo2[0], lo2[1]);
  }
}

template <int NCOL, bool HILO, int HB>
cudaError_t run_gemv(const CUtensorMap& tmA, const CUtensorMap& tmX, int rows, int G, int a_head_rows, int x_rows,
                     int nchunks, int ks, int B, int nxh, float* out, size_t out_split_stride, size_t bstride,
                     size_t hstride, int num_sms, cudaStream_t st) {
  using Geo = HeadsGeom<NCOL>;
  const int nk = (nchunks + ks - 1) / ks;   // round robin: ks divides the chunks so that no split is empty
  const int tiles = (rows + kRowsTile - 1) / kRowsTile;
  // stream-K (!HILO): one CTA per SM, or one per chunk when there are fewer chunks
  const long long nunits = HILO ? (long long)G * tiles * ks : (long long)G * tiles * nchunks;
  cudaError_t e = cudaFuncSetAttribute(heads_tc_kernel<NCOL, HILO, HB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Geo::kSmem);
  if (e != cudaSuccess) return e;
  const int grid = nunits < num_sms ? (int)nunits : num_sms;
  launch_pdl(heads_tc_kernel<NCOL, HILO, HB>, grid, 192, Geo::kSmem, st, tmA, tmX, rows, G, a_head_rows, x_rows,
             nchunks, nk, ks, B, nxh, out, out_split_stride, bstride, hstride);
  note_launches(1);
  return cudaGetLastError();
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
  }
  return n;
}

}  // namespace

// CTAs of the residual layer's stream-K split.
static int stream_ctas(const medusa_cfg& c) {
  const long long T = (long long)c.K * ((c.d + kRowsTile - 1) / kRowsTile) * (c.d / kChunkK);
  return (int)(T < sm_count() ? T : sm_count());
}

// MMA width of the shared-projection GEMV: all K head blocks of NCOL2 columns
// in one B operand, rounded up to 64, 128 or 256 (0: too wide for one MMA).
static int shared_block(int K, int ncol2) {
  const int n = K * ncol2;
  return n <= 64 ? 64 : (n <= 128 ? 128 : (n <= 256 ? 256 : 0));
}

// Workspace layout of the tensor-core heads path.
HeadsTcPlan plan_heads_tc(const medusa_cfg& c) {
  HeadsTcPlan p{};
  p.NB = c.B <= 8 ? 8 : (c.B + 7) / 8 * 8;               // batch columns per part (hi or lo)
  if (c.shared_vocab) p.NB = c.B <= 8 ? 8 : (c.B <= 16 ? 16 : 32);   // head blocks of 16, 32 or 64 columns
  p.NCOL1 = c.B <= 16 ? 16 : 32;                          // d x d layer: h only
  p.NCOL2 = 2 * p.NB;                                     // vocab projection: hi and lo
  // partial-sum slots of the residual layer: at most the CTAs whose equal
  // chunk ranges (>= floor(T / P) chunks each) can touch one tile
  const long long nchunks = c.d / kChunkK;
  const long long T = (long long)c.K * ((c.d + kRowsTile - 1) / kRowsTile) * nchunks;
  const long long P = stream_ctas(c), per = T / P;
  long long slots = (nchunks + per - 1) / per + 1;
  p.slots1 = (int)(slots < P ? slots : P);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  // hi/lo vectors [K][NCOL2][d]; with a shared projection, padded to the MMA's N
  // rows (the rows past K * NCOL2 only feed output columns that are never read)
  const int xrows = c.shared_vocab && shared_block(c.K, p.NCOL2) ? shared_block(c.K, p.NCOL2) : c.K * p.NCOL2;
  p.x2 = take((size_t)xrows * c.d * 2);
  p.part1 = take((size_t)p.slots1 * c.B * c.K * c.d * 4);
  p.total = off;
  return p;
}

cudaError_t heads_tc_take_error(uint32_t* out, cudaStream_t st) {
  static const uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_heads_tc_error, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbolAsync(g_heads_tc_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, st);
}

bool heads_tc_supported(const medusa_cfg& c) { return c.dtype == MEDUSA_BF16 && c.B <= 32 && c.d % 64 == 0; }

cudaError_t launch_heads_tc(const medusa_cfg& c, const void* h, const void* W, const void* bias, const void* U,
                            float* z, char* ws, cudaStream_t st) {
  const HeadsTcPlan p = plan_heads_tc(c);
  uint16_t* x2 = reinterpret_cast<uint16_t*>(ws + p.x2);
  float* part1 = reinterpret_cast<float*>(ws + p.part1);
  const int B = c.B, d = c.d, V = c.V, K = c.K;
  const int nchunks = d / kChunkK;
  CUtensorMap tmW, tmX1, tmU, tmX2;
  if (!encode_tmap_2d_bf16(&tmW, W, (uint64_t)K * d, d, (uint64_t)d * 2, kChunkK, kRowsTile) ||
      // the residual layer reads h itself: rows B..NCOL1-1 of each box lie past
      // the tensor and arrive as zeros
      !encode_tmap_2d_bf16(&tmX1, h, (uint64_t)B, d, (uint64_t)d * 2, kChunkK, p.NCOL1) ||
      !encode_tmap_2d_bf16(&tmU, U, (uint64_t)(c.shared_vocab ? 1 : K) * V, d, (uint64_t)d * 2, kChunkK, kRowsTile) ||
      !encode_tmap_2d_bf16(&tmX2, x2, (uint64_t)K * p.NCOL2, d, (uint64_t)d * 2, kChunkK, p.NCOL2))
    return cudaErrorInvalidValue;
  const int sms = sm_count();

  const int P1 = stream_ctas(c);
  if (((long long)K * ((d + kRowsTile - 1) / kRowsTile) * nchunks + 1) * P1 >= (1LL << 32)) return cudaErrorInvalidValue;
  cudaError_t e = p.NCOL1 == 16
                      ? run_gemv<16, false, 16>(tmW, tmX1, d, K, d, 0, nchunks, 1, B, 1, part1, (size_t)B * K * d,
                                                (size_t)K * d, (size_t)d, P1, st)
                      : run_gemv<32, false, 32>(tmW, tmX1, d, K, d, 0, nchunks, 1, B, 1, part1, (size_t)B * K * d,
                                                (size_t)K * d, (size_t)d, P1, st);
  if (e != cudaSuccess) return e;
  const bool shared = c.shared_vocab && shared_block(K, p.NCOL2);
  const int rp_blocks = (int)(((size_t)K * p.NB * (d / 4) + 255) / 256);
  launch_pdl(residual_pack_tc_kernel, rp_blocks < 1024 ? rp_blocks : 1024, 256, 0, st, part1,
             (d + kRowsTile - 1) / kRowsTile, nchunks, P1, static_cast<const uint16_t*>(h),
             static_cast<const uint16_t*>(bias), x2, B, p.NB, K, d);
  note_launches(1);
  const size_t bs = (size_t)K * V;   // z [B][K][V]
  if (shared) {
    // one stream of U for all heads: X = every head's hi/lo vectors, N = K * NCOL2 rounded up
    const int nt = shared_block(K, p.NCOL2);
    CUtensorMap tmXs;
    if (!encode_tmap_2d_bf16(&tmXs, x2, (uint64_t)nt, d, (uint64_t)d * 2, kChunkK, nt))
      return cudaErrorInvalidValue;
#define MEDUSA_SHARED(NT, HB) \
  if (nt == NT && p.NCOL2 == HB) return run_gemv<NT, true, HB>(tmU, tmXs, V, 1, 0, 0, nchunks, 1, B, K, z, 0, bs, V, sms, st)
    MEDUSA_SHARED(64, 16);
    MEDUSA_SHARED(128, 16);
    MEDUSA_SHARED(64, 32);
    MEDUSA_SHARED(128, 32);
    MEDUSA_SHARED(256, 32);
    MEDUSA_SHARED(64, 64);
    MEDUSA_SHARED(128, 64);
    MEDUSA_SHARED(256, 64);
#undef MEDUSA_SHARED
    return cudaErrorInvalidValue;
  }
  // one vocab projection per head (or a shared one too wide for one block: head g reads rows g * a_rows of U)
  const int a_rows = c.shared_vocab ? 0 : V;
  switch (p.NCOL2) {
    case 16: return run_gemv<16, true, 16>(tmU, tmX2, V, K, a_rows, p.NCOL2, nchunks, 1, B, 1, z, 0, bs, V, sms, st);
    case 32: return run_gemv<32, true, 32>(tmU, tmX2, V, K, a_rows, p.NCOL2, nchunks, 1, B, 1, z, 0, bs, V, sms, st);
    case 48: return run_gemv<48, true, 48>(tmU, tmX2, V, K, a_rows, p.NCOL2, nchunks, 1, B, 1, z, 0, bs, V, sms, st);
    default: return run_gemv<64, true, 64>(tmU, tmX2, V, K, a_rows, p.NCOL2, nchunks, 1, B, 1, z, 0, bs, V, sms, st);
  }
}

}  // namespace medusa
