// C ABI entry points of libmedusa: argument checks, then kernel launches.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "common.cuh"

namespace medusa {

static std::atomic<unsigned long long> g_launches{0};
void note_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks shared by every call: sizes, enums and the built limits.
int check_cfg(const medusa_cfg* c) {
  if (!c) return MEDUSA_ERR_INVALID_ARG;
  if (c->B < 1 || c->d < 1 || c->V < 1 || c->K < 1 || c->Hq < 1 || c->Hkv < 1 || c->D < 1 || c->L_cap < 1)
    return MEDUSA_ERR_INVALID_ARG;
  if (c->dtype != MEDUSA_F32 && c->dtype != MEDUSA_BF16) return MEDUSA_ERR_INVALID_ARG;
  if (c->mode != MEDUSA_GREEDY && c->mode != MEDUSA_REJECTION) return MEDUSA_ERR_INVALID_ARG;
  if (c->K > kMaxK) return MEDUSA_ERR_UNSUPPORTED;
  for (int k = 0; k < c->K; ++k) {
    if (c->branching[k] < 1) return MEDUSA_ERR_INVALID_ARG;
    if (c->branching[k] > kMaxS || c->branching[k] > c->V) return MEDUSA_ERR_UNSUPPORTED;
  }
  long n = 1, cnt = 1;
  if (c->tree_nodes == 0) {
    for (int k = 0; k < c->K; ++k) {
      cnt *= c->branching[k];
      n += cnt;
      if (n > kMaxN) return MEDUSA_ERR_UNSUPPORTED;
    }
  } else {
    // a pruned tree: breadth first, (parent, rank) increasing within a depth, ranks inside the top-s lists
    if (c->tree_nodes < 1 || c->tree_nodes > kMaxN) return MEDUSA_ERR_UNSUPPORTED;
    n = c->tree_nodes;
    if (c->tree_parent[0] != -1) return MEDUSA_ERR_INVALID_ARG;
    int depth[kMaxN];
    depth[0] = 0;
    for (int i = 1; i < n; ++i) {
      const int p = c->tree_parent[i];
      if (p < 0 || p >= i) return MEDUSA_ERR_INVALID_ARG;
      depth[i] = depth[p] + 1;
      if (depth[i] > c->K || c->tree_rank[i] >= c->branching[depth[i] - 1]) return MEDUSA_ERR_INVALID_ARG;
      if (i > 1) {
        const int q = c->tree_parent[i - 1];
        if (depth[i] < depth[i - 1] || depth[i] > depth[i - 1] + 1) return MEDUSA_ERR_INVALID_ARG;
        if (depth[i] == depth[i - 1] && !(p > q || (p == q && c->tree_rank[i] > c->tree_rank[i - 1])))
          return MEDUSA_ERR_INVALID_ARG;
      }
    }
  }
  if (c->Hq % c->Hkv != 0) return MEDUSA_ERR_UNSUPPORTED;
  if (c->D != 64 && c->D != 128) return MEDUSA_ERR_UNSUPPORTED;
  if (c->L_cap < n) return MEDUSA_ERR_CAPACITY;
  if (c->mode == MEDUSA_REJECTION && !(c->temperature > 0.f)) return MEDUSA_ERR_INVALID_ARG;
  if (c->shared_vocab != 0 && c->shared_vocab != 1) return MEDUSA_ERR_INVALID_ARG;
  return MEDUSA_OK;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? MEDUSA_OK : MEDUSA_ERR_CUDA; }

}  // namespace

int check_cfg_public(const medusa_cfg* c) { return check_cfg(c); }

}  // namespace medusa

using namespace medusa;

extern "C" {

int medusa_node_count(const medusa_cfg* cfg, int32_t* N) {
  int s = check_cfg(cfg);
  if (s != MEDUSA_OK && s != MEDUSA_ERR_CAPACITY) return s;
  if (!N) return MEDUSA_ERR_INVALID_ARG;
  *N = tree_shape(*cfg).N;
  return MEDUSA_OK;
}

int medusa_workspace_size(const medusa_cfg* cfg, size_t* bytes) {
  int s = check_cfg(cfg);
  if (s != MEDUSA_OK) return s;
  if (!bytes) return MEDUSA_ERR_INVALID_ARG;
  *bytes = align_up(heads_workspace(*cfg), 256) + align_up(attention_workspace(*cfg), 256) + verify_workspace(*cfg);
  const size_t fused = fused_workspace(*cfg);   // the persistent step's own layout of the same buffer
  if (fused > *bytes) *bytes = fused;
  return MEDUSA_OK;
}

int medusa_heads(const medusa_cfg* cfg, const void* h, const void* W, const void* bias, const void* U, float* logits,
                 int32_t* topk, void* workspace, medusa_stream_t stream) {
  int s = check_cfg(cfg);
  if (s != MEDUSA_OK) return s;
  if (!h || !W || !U || !topk || !workspace) return MEDUSA_ERR_INVALID_ARG;
  if (!logits && cfg->mode == MEDUSA_REJECTION) return MEDUSA_ERR_INVALID_ARG;
  if (cfg->dtype == MEDUSA_BF16) {
    if (cfg->d % 64 != 0) return MEDUSA_ERR_UNSUPPORTED;
    if (!aligned16(h) || !aligned16(W) || !aligned16(U) || (bias && !aligned16(bias))) return MEDUSA_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MEDUSA_ERR_INVALID_ARG;
  // bf16 batches run as consecutive slices of at most kHeadsBatch sequences (the
  // GEMVs' widest batch operand), each streaming the weights once.
  const int slice = cfg->dtype == MEDUSA_BF16 ? kHeadsBatch : cfg->B;
  const size_t h_row = (size_t)cfg->d * (cfg->dtype == MEDUSA_BF16 ? 2 : 4);
  const TreeShape ts = tree_shape(*cfg);
  for (int b0 = 0; b0 < cfg->B; b0 += slice) {
    medusa_cfg c = *cfg;
    c.B = cfg->B - b0 < slice ? cfg->B - b0 : slice;
    cudaError_t e = launch_heads(c, static_cast<const char*>(h) + b0 * h_row, W, bias, U,
                                 logits ? logits + (size_t)b0 * cfg->K * cfg->V : nullptr,
                                 topk + (size_t)b0 * cfg->K * ts.s_max, workspace, (cudaStream_t)stream);
    if (e != cudaSuccess) return from_cuda(e);
  }
  return MEDUSA_OK;
}

int medusa_tree_build(const medusa_cfg* cfg, const int32_t* root_token, const int32_t* topk, const int32_t* L,
                      int32_t* parent, int32_t* depth, int32_t* first_child, uint8_t* mask, uint64_t* anc_bits,
                      int32_t* tokens, int32_t* pos, uint32_t* flags, medusa_stream_t stream) {
  int s = check_cfg(cfg);
  if (s != MEDUSA_OK) return s;
  if (!root_token || !topk || !L || !parent || !depth || !first_child || !mask || !anc_bits || !tokens || !pos)
    return MEDUSA_ERR_INVALID_ARG;
  return from_cuda(launch_tree_build(*cfg, root_token, topk, L, parent, depth, first_child, mask, anc_bits, tokens,
                                     pos, flags, (cudaStream_t)stream));
}

int medusa_tree_attention(const medusa_cfg* cfg, const void* Q, const void* Kc, const void* Vc, const int32_t* L,
                          const uint64_t* anc_bits, void* O, void* workspace, medusa_stream_t stream) {
  int s = check_cfg(cfg);
  if (s != MEDUSA_OK) return s;
  if (!Q || !Kc || !Vc || !L || !anc_bits || !O || !workspace) return MEDUSA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(Kc) || !aligned16(Vc) || !aligned16(O)) return MEDUSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MEDUSA_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace) + align_up(heads_workspace(*cfg), 256);
  return from_cuda(launch_attention(*cfg, Q, Kc, Vc, L, anc_bits, O, ws, (cudaStream_t)stream));
}

int medusa_verify(const medusa_cfg* cfg, const int32_t* tokens, const int32_t* parent, const int32_t* first_child,
                  const void* target_logits, const float* head_logits, const float* u_acc, const float* u_res,
                  int32_t* acc, int32_t* path, int32_t* out_tokens, int32_t* n_out, uint32_t* flags,
                  void* workspace, medusa_stream_t stream) {
  int s = check_cfg(cfg);
  if (s != MEDUSA_OK) return s;
  if (!tokens || !parent || !first_child || !target_logits || !acc || !path || !out_tokens || !n_out || !flags ||
      !workspace)
    return MEDUSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MEDUSA_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace) + align_up(heads_workspace(*cfg), 256) +
             align_up(attention_workspace(*cfg), 256);
  if (cfg->mode == MEDUSA_REJECTION) {
    if (!head_logits || !u_acc || !u_res) return MEDUSA_ERR_INVALID_ARG;
    if (cfg->V > 32768) return MEDUSA_ERR_UNSUPPORTED;
  }
  return from_cuda(launch_verify(*cfg, tokens, parent, first_child, target_logits, head_logits, u_acc, u_res, acc,
                                 path, out_tokens, n_out, flags, ws, (cudaStream_t)stream));
}

int medusa_kv_compact(const medusa_cfg* cfg, void* Kc, void* Vc, int32_t* L, const int32_t* acc, const int32_t* path,
                      int32_t* kv_map, medusa_stream_t stream) {
  int s = check_cfg(cfg);
  if (s != MEDUSA_OK) return s;
  if (!Kc || !Vc || !L || !acc || !path || !kv_map) return MEDUSA_ERR_INVALID_ARG;
  if (!aligned16(Kc) || !aligned16(Vc)) return MEDUSA_ERR_INVALID_ARG;
  return from_cuda(launch_kv_compact(*cfg, Kc, Vc, L, acc, path, kv_map, (cudaStream_t)stream));
}

int medusa_tree_attention_paged(const medusa_cfg* cfg, const void* Q, const void* Kp, const void* Vp, int32_t num_pages,
                                int32_t page_rows, const int32_t* block_table, const void* Kt, const void* Vt,
                                const int32_t* L, const uint64_t* anc_bits, void* O, void* workspace,
                                medusa_stream_t stream) {
  int s = check_cfg(cfg);
  if (s != MEDUSA_OK) return s;
  if (!Q || !Kp || !Vp || !block_table || !Kt || !Vt || !L || !anc_bits || !O || !workspace || num_pages < 1)
    return MEDUSA_ERR_INVALID_ARG;
  if (page_rows < 128 || page_rows % 128 != 0 || cfg->L_cap % page_rows != 0) return MEDUSA_ERR_UNSUPPORTED;
  if (cfg->dtype != MEDUSA_BF16 || cfg->D != 128) return MEDUSA_ERR_UNSUPPORTED;
  if (!aligned16(Q) || !aligned16(Kp) || !aligned16(Vp) || !aligned16(Kt) || !aligned16(Vt) || !aligned16(O))
    return MEDUSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MEDUSA_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace) + align_up(heads_workspace(*cfg), 256);
  const PagedKV pg{num_pages, page_rows, block_table, Kt, Vt};
  return from_cuda(launch_attention(*cfg, Q, Kp, Vp, L, anc_bits, O, ws, (cudaStream_t)stream, &pg));
}

int medusa_kv_commit_paged(const medusa_cfg* cfg, void* Kp, void* Vp, int32_t page_rows, const int32_t* block_table,
                           const void* Kt, const void* Vt, int32_t n_layers, size_t pool_layer_elems,
                           size_t tree_layer_elems, int32_t* L, const int32_t* acc, const int32_t* path,
                           int32_t* kv_map, medusa_stream_t stream) {
  int s = check_cfg(cfg);
  if (s != MEDUSA_OK) return s;
  if (!Kp || !Vp || !block_table || !Kt || !Vt || !L || !acc || !path || !kv_map || n_layers < 1)
    return MEDUSA_ERR_INVALID_ARG;
  if (page_rows < 128 || page_rows % 128 != 0 || cfg->L_cap % page_rows != 0) return MEDUSA_ERR_UNSUPPORTED;
  const size_t per16 = cfg->dtype == MEDUSA_F32 ? 4 : 8;
  if (!aligned16(Kp) || !aligned16(Vp) || !aligned16(Kt) || !aligned16(Vt) || pool_layer_elems % per16 != 0 ||
      tree_layer_elems % per16 != 0 || (n_layers > 1 && (pool_layer_elems == 0 || tree_layer_elems == 0)))
    return MEDUSA_ERR_INVALID_ARG;
  // pages in one layer's pool; a page id at or beyond it is never written (unknown when the
  // caller passes no layer size for a single layer)
  const size_t page_elems = (size_t)cfg->Hkv * page_rows * cfg->D;
  const size_t pages = pool_layer_elems ? pool_layer_elems / page_elems : (size_t)INT32_MAX;
  const PagedKV pg{(int)(pages < (size_t)INT32_MAX ? pages : (size_t)INT32_MAX), page_rows, block_table, Kt, Vt};
  return from_cuda(launch_kv_commit_paged(*cfg, Kp, Vp, pg, n_layers, pool_layer_elems, tree_layer_elems, L, acc, path,
                                          kv_map, (cudaStream_t)stream));
}

}  // extern "C"

struct medusa_step_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  unsigned long long kernels = 0;   // kernel launches one replay stands for
};

extern "C" {

int medusa_step_graph_create(const medusa_cfg* cfg, const medusa_step_args* a, medusa_step_graph** out) {
  if (!cfg || !a || !out) return MEDUSA_ERR_INVALID_ARG;
  *out = nullptr;
  int status = check_cfg(cfg);
  if (status != MEDUSA_OK) return status;
  cudaStream_t st = nullptr;
  if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return MEDUSA_ERR_CUDA;
  if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaStreamDestroy(st);
    return MEDUSA_ERR_CUDA;
  }
  const unsigned long long before = g_launches.load(std::memory_order_relaxed);
  const medusa_stream_t ms = (medusa_stream_t)st;
  status = medusa_heads(cfg, a->h, a->W, a->bias, a->U, a->logits, a->topk, a->workspace, ms);
  if (status == MEDUSA_OK)
    status = medusa_tree_build(cfg, a->root_token, a->topk, a->L, a->parent, a->depth, a->first_child, a->mask,
                               a->anc_bits, a->tokens, a->pos, a->flags, ms);
  if (status == MEDUSA_OK)
    status = medusa_tree_attention(cfg, a->Q, a->Kc, a->Vc, a->L, a->anc_bits, a->O, a->workspace, ms);
  if (status == MEDUSA_OK)
    status = medusa_verify(cfg, a->tokens, a->parent, a->first_child, a->target_logits, a->logits, a->u_acc, a->u_res,
                           a->acc, a->path, a->out_tokens, a->n_out, a->flags, a->workspace, ms);
  if (status == MEDUSA_OK && a->kv_compact)
    status = medusa_kv_compact(cfg, a->Kc, a->Vc, a->L, a->acc, a->path, a->kv_map, ms);
  const unsigned long long kernels = g_launches.load(std::memory_order_relaxed) - before;
  g_launches.fetch_sub(kernels, std::memory_order_relaxed);   // captured, not launched
  cudaGraph_t graph = nullptr;
  const cudaError_t ended = cudaStreamEndCapture(st, &graph);   // ends the capture on every path
  cudaStreamDestroy(st);
  if (status == MEDUSA_OK && (ended != cudaSuccess || !graph)) status = MEDUSA_ERR_CUDA;
  cudaGraphExec_t exec = nullptr;
  if (status == MEDUSA_OK && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) status = MEDUSA_ERR_CUDA;
  if (status != MEDUSA_OK) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();   // a failed call inside the capture leaves no sticky error behind
    return status;
  }
  medusa_step_graph* g = new medusa_step_graph;
  g->graph = graph;
  g->exec = exec;
  g->kernels = kernels;
  *out = g;
  return MEDUSA_OK;
}

int medusa_step_graph_launch(medusa_step_graph* g, medusa_stream_t stream) {
  if (!g) return MEDUSA_ERR_INVALID_ARG;
  if (cudaGraphLaunch(g->exec, (cudaStream_t)stream) != cudaSuccess) return MEDUSA_ERR_CUDA;
  g_launches.fetch_add(g->kernels, std::memory_order_relaxed);
  return MEDUSA_OK;
}

int medusa_step_graph_destroy(medusa_step_graph* g) {
  if (!g) return MEDUSA_ERR_INVALID_ARG;
  const bool ok = cudaGraphExecDestroy(g->exec) == cudaSuccess && cudaGraphDestroy(g->graph) == cudaSuccess;
  delete g;
  return ok ? MEDUSA_OK : MEDUSA_ERR_CUDA;
}

int medusa_poll_errors(medusa_stream_t stream, uint32_t* heads_codes, uint32_t* attention_codes) {
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t h = 0, a = 0, f = 0;
  cudaError_t e = heads_tc_take_error(&h, st);
  if (e == cudaSuccess) e = attention_tc_take_error(&a, st);
  if (e == cudaSuccess) e = fused_take_error(&f, st);
  a |= f;
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return MEDUSA_ERR_CUDA;
  if (heads_codes) *heads_codes = h;
  if (attention_codes) *attention_codes = a;
  return (h | a) ? MEDUSA_ERR_TIMEOUT : MEDUSA_OK;
}

int medusa_step_fused(const medusa_cfg* cfg, const medusa_step_args* a, medusa_stream_t stream) {
  if (!cfg || !a) return MEDUSA_ERR_INVALID_ARG;
  int s = check_cfg(cfg);
  if (s != MEDUSA_OK) return s;
  if (!fused_supported(*cfg)) return MEDUSA_ERR_UNSUPPORTED;
  if (!a->h || !a->W || !a->U || !a->topk || !a->root_token || !a->L || !a->parent || !a->depth ||
      !a->first_child || !a->mask || !a->anc_bits || !a->tokens || !a->pos || !a->Q || !a->Kc || !a->Vc || !a->O ||
      !a->target_logits || !a->acc || !a->path || !a->out_tokens || !a->n_out || (a->kv_compact && !a->kv_map) ||
      !a->workspace)
    return MEDUSA_ERR_INVALID_ARG;
  if (!aligned16(a->h) || !aligned16(a->W) || !aligned16(a->U) || (a->bias && !aligned16(a->bias)) ||
      !aligned16(a->Q) || !aligned16(a->Kc) || !aligned16(a->Vc) || !aligned16(a->O) || !aligned16(a->target_logits))
    return MEDUSA_ERR_INVALID_ARG;
  return from_cuda(launch_fused_step(*cfg, *a, (cudaStream_t)stream));
}

int medusa_checked_build(void) {
#ifdef MEDUSA_CHECKED
  return 1;
#else
  return 0;
#endif
}

int medusa_poll_checks(medusa_stream_t stream, uint32_t* codes) {
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t w[4] = {0, 0, 0, 0};
  cudaError_t e = tree_take_checks(&w[0], st);
  if (e == cudaSuccess) e = verify_take_checks(&w[1], st);
  if (e == cudaSuccess) e = compact_take_checks(&w[2], st);
  if (e == cudaSuccess) e = attention_tc_take_checks(&w[3], st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return MEDUSA_ERR_CUDA;
  const uint32_t all = w[0] | w[1] | w[2] | w[3];
  if (codes) *codes = all;
  return all ? MEDUSA_ERR_BOUNDS : MEDUSA_OK;
}

int medusa_selftest_wait_timeout(uint32_t budget_us, medusa_stream_t stream) {
  if (budget_us < 1 || budget_us > 1000000) return MEDUSA_ERR_INVALID_ARG;
  return from_cuda(launch_wait_selftest((long long)budget_us * 2100, (cudaStream_t)stream));   // <= 2.1 GHz SM clock
}

uint64_t medusa_launch_count(void) { return (uint64_t)g_launches.load(std::memory_order_relaxed); }

const char* medusa_status_string(int status) {
  switch (status) {
    case MEDUSA_OK: return "ok";
    case MEDUSA_ERR_INVALID_ARG: return "invalid argument";
    case MEDUSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MEDUSA_ERR_CAPACITY: return "KV cache capacity exceeded";
    case MEDUSA_ERR_CUDA: return "CUDA launch error";
    case MEDUSA_ERR_TIMEOUT: return "device wait timed out";
    case MEDUSA_ERR_BOUNDS: return "out-of-range index met on the device (checked build)";
    default: return "unknown status";
  }
}

}  // extern "C"
