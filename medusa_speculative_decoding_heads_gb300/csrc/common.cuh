// Shared device/host helpers of libmedusa (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/medusa.h"

namespace medusa {

// Programmatic dependent launch. Every kernel of the library is launched with
// programmatic stream serialization, so it may start while the previous kernel
// on the stream is still finishing; pdl_wait() blocks until that kernel has
// completed and its memory is visible, and must precede every access to global
// memory that another kernel wrote or will read. pdl_trigger() lets the next
// kernel launch as soon as every CTA of this one has started.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

constexpr int kMaxK = 8;
constexpr int kMaxS = 8;
constexpr int kMaxN = 128;
constexpr int kHeadsBatch = 32;   // sequences per bf16 heads pass (larger batches run in slices)

// Tree shape derived from the configuration: level counts and offsets.
struct TreeShape {
  int K;
  int N;
  int s_max;
  int s[kMaxK + 1];     // s[1..K]
  int cnt[kMaxK + 1];   // cnt[d] = prod_{j<=d} s_j, cnt[0] = 1
  int off[kMaxK + 2];   // off[d] = sum_{e<d} cnt[e]; off[K+1] = N (Cartesian tree)
  int pruned;           // 1: N comes from a pruned tree's node list (cnt/off unused)
};

inline TreeShape tree_shape(const medusa_cfg& c) {
  TreeShape t{};
  t.K = c.K;
  t.cnt[0] = 1;
  t.off[0] = 0;
  t.s_max = 0;
  for (int d = 1; d <= c.K; ++d) {
    t.s[d] = c.branching[d - 1];
    t.cnt[d] = t.cnt[d - 1] * t.s[d];
    t.s_max = t.s[d] > t.s_max ? t.s[d] : t.s_max;
  }
  for (int d = 1; d <= c.K + 1; ++d) t.off[d] = t.off[d - 1] + t.cnt[d - 1];
  t.N = t.off[c.K + 1];
  if (c.tree_nodes > 0) {   // a pruned tree: its own node count
    t.N = c.tree_nodes;
    t.pruned = 1;
  }
  return t;
}

// bf16 <-> f32 as bit patterns (bf16 is the top half of an IEEE f32).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t v) { return __uint_as_float(uint32_t(v) << 16); }

// Round-to-nearest-even f32 -> bf16 bit pattern (inputs here are finite).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  uint32_t r = 0x7fffu + ((u >> 16) & 1u);
  return uint16_t((u + r) >> 16);
}

template <typename T> struct Elt;
template <> struct Elt<float> {
  __device__ __forceinline__ static float load(const float* p, size_t i) { return p[i]; }
  __device__ __forceinline__ static void store(float* p, size_t i, float v) { p[i] = v; }
};
template <> struct Elt<uint16_t> {
  __device__ __forceinline__ static float load(const uint16_t* p, size_t i) { return bf16_to_f32(p[i]); }
  __device__ __forceinline__ static void store(uint16_t* p, size_t i, float v) { p[i] = f32_to_bf16(v); }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Launchers (each returns a cudaError_t from the launch).
cudaError_t launch_heads(const medusa_cfg& c, const void* h, const void* W, const void* bias,
                         const void* U, float* logits, int32_t* topk, void* ws, cudaStream_t st);
size_t heads_workspace(const medusa_cfg& c);

// Tensor-core (tcgen05) heads path.
struct HeadsTcPlan {
  int NB, NCOL1, NCOL2, slots1;   // slots1: partial-sum slots of the residual layer
  size_t x2, part1, total;
};
HeadsTcPlan plan_heads_tc(const medusa_cfg& c);
bool heads_tc_supported(const medusa_cfg& c);
cudaError_t launch_heads_tc(const medusa_cfg& c, const void* h, const void* W, const void* bias, const void* U,
                            float* z, char* ws, cudaStream_t st);

cudaError_t launch_tree_build(const medusa_cfg& c, const int32_t* root, const int32_t* topk,
                              const int32_t* L, int32_t* parent, int32_t* depth, int32_t* first_child,
                              uint8_t* mask, uint64_t* bits, int32_t* tokens, int32_t* pos,
                              uint32_t* flags, cudaStream_t st);

// A paged KV cache: pool [num_pages][Hkv][page_rows][D] (Kc/Vc point at it),
// block_table [B][L_cap / page_rows], the tree's rows staged in Kt/Vt [B][Hkv][N][D].
struct PagedKV {
  int num_pages, page_rows;
  const int32_t* block_table;
  const void* Kt;
  const void* Vt;
};

cudaError_t launch_attention(const medusa_cfg& c, const void* Q, const void* Kc, const void* Vc,
                             const int32_t* L, const uint64_t* bits, void* O, void* ws, cudaStream_t st,
                             const PagedKV* paged = nullptr);
cudaError_t launch_kv_commit_paged(const medusa_cfg& c, void* Kp, void* Vp, const PagedKV& pg, int n_layers,
                                   size_t pool_layer_elems, size_t tree_layer_elems, int32_t* L, const int32_t* acc,
                                   const int32_t* path, int32_t* kv_map, cudaStream_t st);
size_t attention_workspace(const medusa_cfg& c);
// Read-and-clear of the device words in which the tcgen05 kernels record expired waits
// (stream-ordered; the caller synchronises before reading *out).
cudaError_t heads_tc_take_error(uint32_t* out, cudaStream_t st);
cudaError_t attention_tc_take_error(uint32_t* out, cudaStream_t st);
// One bounded mbarrier wait that nothing completes: records kWaitSelfTestCode in the
// attention kernels' error word after about `cycles` SM clocks.
constexpr uint32_t kWaitSelfTestCode = 0x80000000u;
cudaError_t launch_wait_selftest(long long cycles, cudaStream_t st);
int attention_mma_warps(int NG, int* row_blocks);
int attention_tc_mtiles(int NG);
int attention_tc_ctas_x(int NG);
cudaError_t launch_attention_tc(const medusa_cfg& c, int nsplit, int chunk, const void* Q, const void* Kc,
                                const void* Vc, const int32_t* L, const uint64_t* bits, float* o_part, float* ml_part,
                                float* x_part, void* O, cudaStream_t st, const PagedKV* paged);
size_t attention_tc_xpart_bytes(const medusa_cfg& c, int nsplit);
cudaError_t launch_attention_tc_xmerge(const medusa_cfg& c, int nsplit, const float* x_part, const int32_t* L, void* O,
                                       cudaStream_t st);
cudaError_t launch_attention_mma(const medusa_cfg& c, int nsplit, int chunk, const void* Q, const void* Kc,
                                 const void* Vc, const int32_t* L, const uint64_t* bits, float* o_part, float* ml_part,
                                 cudaStream_t st);

cudaError_t launch_verify(const medusa_cfg& c, const int32_t* tokens, const int32_t* parent,
                          const int32_t* first_child, const void* tl, const float* hl,
                          const float* u_acc, const float* u_res, int32_t* acc, int32_t* path,
                          int32_t* out_tokens, int32_t* n_out, uint32_t* flags, void* ws, cudaStream_t st);
size_t verify_workspace(const medusa_cfg& c);

cudaError_t launch_kv_compact(const medusa_cfg& c, void* Kc, void* Vc, int32_t* L, const int32_t* acc,
                              const int32_t* path, int32_t* kv_map, cudaStream_t st);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The whole step as one persistent cooperative launch (fused.cu): small batches,
// bf16, D = 128, greedy acceptance.
bool fused_supported(const medusa_cfg& c);
size_t fused_workspace(const medusa_cfg& c);
cudaError_t launch_fused_step(const medusa_cfg& c, const medusa_step_args& s, cudaStream_t st);
cudaError_t fused_take_error(uint32_t* out, cudaStream_t st);

// Checked build (-DMEDUSA_CHECKED). Where a kernel meets an index it read from
// device memory (a token id, a tree link, a path node, a page id) outside the
// range it may address, it already clamps the index or skips the access; the
// checked build also ORs a MEDUSA_CHECK_* code into a device word of the
// translation unit, which medusa_poll_checks reads and clears. Nothing traps.
// In the normal build MEDUSA_CHECK compiles to nothing.
#ifdef MEDUSA_CHECKED
namespace {
__device__ uint32_t g_check_word = 0;
}
#define MEDUSA_CHECK(cond, code)                                  \
  do {                                                            \
    if (!(cond)) atomicOr(&::medusa::g_check_word, (uint32_t)(code)); \
  } while (0)
// Defines `cudaError_t fn(uint32_t* out, cudaStream_t st)`: stream-ordered read-and-clear of
// this translation unit's check word (the caller synchronises before reading *out).
#define MEDUSA_CHECK_TAKE(fn)                                                                                \
  cudaError_t fn(uint32_t* out, cudaStream_t st) {                                                          \
    static const uint32_t zero = 0;                                                                         \
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_check_word, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, st); \
    if (e != cudaSuccess) return e;                                                                         \
    return cudaMemcpyToSymbolAsync(g_check_word, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, st);  \
  }
#else
#define MEDUSA_CHECK(cond, code) \
  do {                           \
  } while (0)
#define MEDUSA_CHECK_TAKE(fn)                              \
  cudaError_t fn(uint32_t* out, cudaStream_t) {            \
    *out = 0;                                              \
    return cudaSuccess;                                    \
  }
#endif
cudaError_t tree_take_checks(uint32_t* out, cudaStream_t st);
cudaError_t verify_take_checks(uint32_t* out, cudaStream_t st);
cudaError_t compact_take_checks(uint32_t* out, cudaStream_t st);
cudaError_t attention_tc_take_checks(uint32_t* out, cudaStream_t st);

// Configuration checks shared by every entry point (MEDUSA_OK or an error status).
int check_cfg_public(const medusa_cfg* c);

// Host-side count of kernels this library has enqueued (diagnostics).
void note_launches(int n);

}  // namespace medusa
