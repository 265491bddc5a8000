/*
 * medusa.h — C ABI of libmedusa: one Medusa speculative-decoding verify step on
 * one GB300 GPU (sm_103a).
 *
 * The step, as the source pages describe it:
 *   1. K Medusa heads on the backbone's last hidden state h: a residual block
 *      r_k = h + SiLU(W_k h + b_k) and a vocab projection z_k = U_k r_k, then a
 *      top-s_k list per head  ["Medusa 심층 아키텍처" (techknowgenie), section
 *      "잔차 블록(Residual Block)을 포함한 Medusa 헤드 구조", equations h_t^(k) and
 *      p_k; section "소스코드 레벨 구조 분석", MedusaHead and generate_candidates].
 *   2. The Cartesian candidate tree, its ancestor mask and position ids
 *      [same page, section "트리 어텐션", tree-topology example and the TreeMask
 *      equation].
 *   3. Tree attention: every node attends to the committed KV cache plus its own
 *      ancestors, all nodes in one pass [same page, section "트리 어텐션"].
 *   4. Acceptance — greedy longest matching path with a bonus token ["최적화 2편"
 *      (beengineer500), section 1.3] or rejection sampling with r = min(1, p/q)
 *      and residual max(0, p - q)/sum ["Medusa 심층 아키텍처", section "수학적
 *      무손실 보장", equations alpha(x) and p'(x); "Speculative Decoding 원리와
 *      가속 아키텍처" (blog.huny.dev), section 2.1] — then compaction of the
 *      accepted path's KV rows [blog.huny.dev, section 5 Case 2 and section 6].
 *
 * Conventions (every entry point):
 *   - Pointers are DEVICE pointers unless a parameter says otherwise; the caller
 *     owns every buffer. The library never allocates or frees device memory;
 *     scratch comes from a caller-provided workspace of medusa_workspace_size()
 *     bytes (256-byte aligned).
 *   - Calls only enqueue work on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronize (except medusa_poll_errors, which
 *     reads back the device's expired-wait words).
 *   - Return MEDUSA_OK (0) or a negative MEDUSA_ERR_*; on error nothing is
 *     enqueued. Device-side data errors never trap: they set bits in a
 *     per-sequence `flags` word and the affected sequence is skipped.
 *   - Layouts are dense row-major with the shapes given; "elt" is float when
 *     cfg->dtype == MEDUSA_F32 and bf16 (uint16 bit pattern) when MEDUSA_BF16.
 *   - N = 1 + sum_{k=1..K} prod_{j<=k} s_j is the node count of the Cartesian
 *     tree, or cfg->tree_nodes for a pruned tree (N <= 128); s_max = max_k s_k
 *     (<= 8), K <= 8.
 *   - Tree node order: breadth first; within a depth, lexicographic in the
 *     path of sibling ranks (first rank most significant). Node 0 is the root,
 *     which is the already committed next token of each sequence.
 */
#ifndef MEDUSA_H_
#define MEDUSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MEDUSA_API __attribute__((visibility("default")))
#else
#define MEDUSA_API
#endif

typedef struct CUstream_st* medusa_stream_t; /* same type as cudaStream_t */

enum { MEDUSA_F32 = 0, MEDUSA_BF16 = 1 };
enum { MEDUSA_GREEDY = 0, MEDUSA_REJECTION = 1 };

enum {
  MEDUSA_OK = 0,
  MEDUSA_ERR_INVALID_ARG = -1, /* null pointer, non-positive size, bad enum   */
  MEDUSA_ERR_UNSUPPORTED = -2, /* valid but outside the built limits          */
  MEDUSA_ERR_CAPACITY = -3,    /* host-visible capacity violation              */
  MEDUSA_ERR_CUDA = -4,        /* a CUDA launch or attribute call failed       */
  MEDUSA_ERR_TIMEOUT = -5,     /* a bounded device-side wait expired (medusa_poll_errors) */
  MEDUSA_ERR_BOUNDS = -6       /* checked build: a kernel met an out-of-range index (medusa_poll_checks) */
};

/* Per-sequence flag bits (uint32). */
#define MEDUSA_FLAG_RS_NEAR_TIE 1u  /* some acceptance test had |u - r| < 1e-6            */
#define MEDUSA_FLAG_CDF_NEAR_TIE 2u /* an inverse-CDF draw fell within 1e-6*total of a step */
#define MEDUSA_FLAG_CAPACITY 4u     /* L_b < 0 or L_b + N > L_cap: sequence skipped      */
#define MEDUSA_FLAG_TIMEOUT 8u      /* a bounded device-side wait gave up: outputs of this */
                                    /* sequence are not valid                              */

typedef struct {
  int32_t B;            /* sequences in the step                                 */
  int32_t d;            /* hidden size                                           */
  int32_t V;            /* vocabulary size                                       */
  int32_t K;            /* Medusa heads = tree depth (1..8)                      */
  int32_t branching[8]; /* s_1..s_K: candidates kept per head (1..8)             */
  int32_t Hq;           /* query heads                                           */
  int32_t Hkv;          /* KV heads (Hq % Hkv == 0)                              */
  int32_t D;            /* head dim (64 or 128)                                  */
  int32_t L_cap;        /* KV cache rows per (sequence, KV head)                 */
  int32_t dtype;        /* MEDUSA_F32 or MEDUSA_BF16                             */
  int32_t mode;         /* MEDUSA_GREEDY or MEDUSA_REJECTION                     */
  float temperature;    /* T > 0 for MEDUSA_REJECTION (logits are divided by T)  */
  int32_t shared_vocab; /* 0: one vocab projection U_k per head; 1: all heads    */
                        /* share one frozen projection U (the base model's LM    */
                        /* head), "Medusa 심층 아키텍처", section "잔차 블록을     */
                        /* 포함한 Medusa 헤드 구조", the note under the p_k      */
                        /* equation: W_head^(k) may be the frozen W_lm_head.     */
  int32_t tree_nodes;   /* 0: the full Cartesian tree of branching[]. 1..128: a   */
                        /* pruned tree of that many nodes (node 0 = root), given  */
                        /* by tree_parent/tree_rank in breadth-first order,       */
                        /* lexicographic in the rank path within a depth (so a    */
                        /* node's children are contiguous and in rank order).     */
                        /* "Medusa 심층 아키텍처", sections "벤치마크 실측 지표"  */
                        /* (4 heads, 64 tree branches) and "트리 크기(Tree Size)와 */
                        /* 검증 오버헤드의 균형" (32-64 nodes usually best).        */
  int16_t tree_parent[128]; /* pruned tree: parent node (-1 at the root)          */
  uint8_t tree_rank[128];   /* pruned tree: the node's rank in its head's top-s   */
                            /* list (< branching[depth - 1]); its token is        */
                            /* topk[b][depth - 1][rank]                           */
} medusa_cfg;

/* Node count N of the configured tree. Host only; `N` is a host pointer. */
MEDUSA_API int medusa_node_count(const medusa_cfg* cfg, int32_t* N);

/* Workspace bytes needed by medusa_heads, medusa_tree_attention and
 * medusa_verify for this configuration (one workspace serves all three: they
 * use disjoint parts). Host only; `bytes` is a host pointer. */
MEDUSA_API int medusa_workspace_size(const medusa_cfg* cfg, size_t* bytes);

/* Step 1 — Medusa heads and per-head top-s.
 *   h      [B][d] elt          backbone last hidden state
 *   W      [K][d][d] elt       W[k][o][i]: residual-layer weight, input i -> output o
 *   bias   [K][d] elt          b_k, may be NULL (zero bias)
 *   U      [K][V][d] elt       U[k][v][i]: vocab projection of head k; with
 *                              cfg->shared_vocab, [V][d]: one projection for every
 *                              head (its weights are streamed once for all heads)
 *   logits [B][K][V] float     z_k per sequence; may be NULL in MEDUSA_GREEDY mode
 *                              (then kept in the workspace). Needed as
 *                              `head_logits` by medusa_verify in MEDUSA_REJECTION.
 *   topk   [B][K][s_max] int32 indices of the s_k largest z_k entries, descending,
 *                              ties to the lower index; -1 beyond s_k.
 * r_k is kept in float32; accumulation is float32. bf16 needs d % 64 == 0
 * (MEDUSA_ERR_UNSUPPORTED otherwise) and 16-byte aligned h, W, bias and U
 * (MEDUSA_ERR_INVALID_ARG otherwise); a bf16 batch above 32 sequences runs as
 * consecutive slices of at most 32, each streaming W and U once. */
MEDUSA_API int medusa_heads(const medusa_cfg* cfg, const void* h, const void* W, const void* bias,
                 const void* U, float* logits, int32_t* topk, void* workspace,
                 medusa_stream_t stream);

/* Step 2 — Cartesian candidate tree.
 *   root_token [B] int32, topk [B][K][s_max] int32, L [B] int32 (committed lengths).
 * Outputs (the first five are identical for every sequence):
 *   parent [N] int32 (-1 at the root), depth [N] int32, first_child [N] int32
 *   (-1 at a leaf; children of a node are contiguous, in rank order),
 *   mask [N][N] uint8 (1 iff column is an ancestor of the row or the row itself),
 *   anc_bits [N][2] uint64 (bit j of word j/64 = mask[i][j]),
 *   tokens [B][N] int32 (root_token, then topk[b][depth-1][rank]),
 *   pos [B][N] int32 (L_b + depth),
 *   flags [B] uint32 (may be NULL): OVERWRITTEN with MEDUSA_FLAG_CAPACITY or 0. */
MEDUSA_API int medusa_tree_build(const medusa_cfg* cfg, const int32_t* root_token, const int32_t* topk,
                      const int32_t* L, int32_t* parent, int32_t* depth, int32_t* first_child,
                      uint8_t* mask, uint64_t* anc_bits, int32_t* tokens, int32_t* pos,
                      uint32_t* flags, medusa_stream_t stream);

/* Step 3 — tree attention.
 *   Q  [B][N][Hq][D] elt          queries of the tree nodes
 *   Kc [B][Hkv][L_cap][D] elt     keys: committed rows [0, L_b), tree rows L_b + j
 *   Vc [B][Hkv][L_cap][D] elt     values, same layout
 *   L  [B] int32, anc_bits [N][2] uint64 (from medusa_tree_build)
 *   O  [B][N][Hq][D] elt          softmax(q.k / sqrt(D)) v over the committed rows
 *                                 and the node's ancestors-or-self; KV head of
 *                                 query head h is h / (Hq / Hkv).
 * Softmax and accumulation in float32. A sequence with L_b < 0 or
 * L_b + N > L_cap gets O = 0. */
MEDUSA_API int medusa_tree_attention(const medusa_cfg* cfg, const void* Q, const void* Kc, const void* Vc,
                          const int32_t* L, const uint64_t* anc_bits, void* O, void* workspace,
                          medusa_stream_t stream);

/* Step 4 — acceptance walk (cfg->mode).
 *   tokens [B][N], parent [N], first_child [N] int32 (from medusa_tree_build)
 *   target_logits [B][N][V] elt   target model logits at every tree node
 *   head_logits [B][K][V] float   z from medusa_heads (MEDUSA_REJECTION only, else NULL)
 *   u_acc [B][K][s_max] float     acceptance uniforms (REJECTION only, else NULL)
 *   u_res [B][K+1] float          resampling uniforms (REJECTION only, else NULL)
 *   workspace                     as for medusa_heads (256-byte aligned)
 * Outputs: acc [B] accepted drafts; path [B][K+1] node ids (path[0] = 0, -1 pad);
 *   out_tokens [B][K+1] the accepted tokens then the bonus/correction token
 *   (-1 pad); n_out [B] = acc + 1; flags [B] uint32: this call ORs in its
 *   MEDUSA_FLAG_* bits (clear or initialise it first, e.g. with medusa_tree_build);
 *   MEDUSA_FLAG_TIMEOUT marks a sequence whose walk gave up on a bounded wait.
 * GREEDY walks each sequence on one CTA that reads only the target rows of
 * the nodes it visits (acc + 1 rows), taking each row's argmax as it goes.
 * REJECTION reduces every head row (max and softmax normaliser) in parallel
 * first; each sequence's walk then runs on a cluster of up to 8 CTAs that split
 * the vocabulary and trade their partial sums through distributed shared
 * memory: per depth one load of the visited target row and the depth's head
 * row (kept in registers), then one exchange per statistic, per rejection and
 * for the final draw.
 * GREEDY: the child whose token equals argmax(target_logits[node]) (ties to
 * the lowest id) is accepted until none matches; the bonus is that argmax at
 * the last accepted node.
 * REJECTION: at the current node, p = softmax(target/T), q = softmax(z_depth/T);
 * children in rank order are accepted when u < min(1, p(x)/q(x)), each
 * rejection replacing p by max(0, p - q)/sum; when all are rejected the bonus
 * is the smallest y with cdf_p(y) > u_res * sum(p); after an accepted leaf it is
 * drawn from softmax(target[leaf]/T). Requires V <= 32768. */
MEDUSA_API int medusa_verify(const medusa_cfg* cfg, const int32_t* tokens, const int32_t* parent,
                  const int32_t* first_child, const void* target_logits, const float* head_logits,
                  const float* u_acc, const float* u_res, int32_t* acc, int32_t* path,
                  int32_t* out_tokens, int32_t* n_out, uint32_t* flags, void* workspace,
                             medusa_stream_t stream);

/* Step 5 — KV compaction of the accepted path, in place.
 *   Kc, Vc [B][Hkv][L_cap][D] elt: for r = 0..acc_b, row L_b + r <- row L_b + path[b][r]
 *   in every KV head (sources are read before they can be overwritten).
 *   L [B] int32 in/out: L_b += acc_b + 1.
 *   kv_map [B][K+1] int32: source node per destination slot, -1 pad.
 * Sequences with L_b < 0 or L_b + N > L_cap are left unchanged (kv_map = -1). */
MEDUSA_API int medusa_kv_compact(const medusa_cfg* cfg, void* Kc, void* Vc, int32_t* L, const int32_t* acc,
                      const int32_t* path, int32_t* kv_map, medusa_stream_t stream);

/* The whole step as one launch. medusa_step_graph_create captures the five
 * calls above, in order, on a private stream into a CUDA graph (the kernels keep
 * their programmatic-dependent-launch edges) and instantiates it;
 * medusa_step_graph_launch then enqueues the step on `stream` with a single
 * launch. The graph holds the pointers in `args`: every later launch reads the
 * inputs from, and writes the outputs to, the same buffers, so a caller writes
 * each step's inputs there (any lengths L within cfg->L_cap; the plan depends on
 * the configuration only). Each call's checks run during creation: the first
 * failing one's status is returned and nothing is kept. Creation and destruction
 * use host memory and the driver's graph objects; they synchronise nothing but
 * the private stream. Fields as in the calls above; head_logits for
 * medusa_verify is `logits`; kv_compact = 0 leaves out step 5. */
typedef struct {
  const void* h; const void* W; const void* bias; const void* U; float* logits; int32_t* topk;
  const int32_t* root_token; int32_t* L; int32_t* parent; int32_t* depth; int32_t* first_child;
  uint8_t* mask; uint64_t* anc_bits; int32_t* tokens; int32_t* pos; uint32_t* flags;
  const void* Q; void* Kc; void* Vc; void* O;
  const void* target_logits; const float* u_acc; const float* u_res;
  int32_t* acc; int32_t* path; int32_t* out_tokens; int32_t* n_out; int32_t* kv_map;
  void* workspace;
  int32_t kv_compact;
} medusa_step_args;
typedef struct medusa_step_graph medusa_step_graph;   /* opaque */
MEDUSA_API int medusa_step_graph_create(const medusa_cfg* cfg, const medusa_step_args* args,
                                        medusa_step_graph** graph);
MEDUSA_API int medusa_step_graph_launch(medusa_step_graph* graph, medusa_stream_t stream);
MEDUSA_API int medusa_step_graph_destroy(medusa_step_graph* graph);

/* The whole step as one persistent kernel. Runs the five calls above (heads,
 * tree, tree attention, greedy acceptance and, unless args->kv_compact is 0, KV
 * compaction) as phases of a single cooperative launch with one CTA per SM; the
 * phases meet at a grid-wide barrier whose every wait is bounded (an expired
 * wait is recorded for medusa_poll_errors, as MEDUSA_FUSED_WAIT_CODE in its
 * attention word; that call's outputs are then invalid). Buffers, layouts and
 * results are those of the five calls ("Medusa 심층 아키텍처", section "트리
 * 어텐션": all candidates verified in one forward pass); `logits` may be NULL.
 * Supported: bf16, D = 128, MEDUSA_GREEDY, B <= 4 and B * d * 4 <= 200 KB
 * (MEDUSA_ERR_UNSUPPORTED otherwise, nothing enqueued); h, W, bias, U, Q, Kc,
 * Vc, O and target_logits 16-byte aligned (MEDUSA_ERR_INVALID_ARG otherwise).
 * The weight GEMVs run on CUDA cores and attention on mma.sync tensor cores.
 * The workspace of medusa_workspace_size covers it. Enqueues a 8-byte memset of
 * the workspace (the barrier's count) and the kernel. No counterpart on the
 * pages as an interface. */
#define MEDUSA_FUSED_WAIT_CODE 0x40000000u
MEDUSA_API int medusa_step_fused(const medusa_cfg* cfg, const medusa_step_args* args, medusa_stream_t stream);

/* Tree attention over a paged KV cache. A page pool is read as a storage
 * layout of the same logical cache that medusa_tree_attention takes.
 *   Kp, Vp [num_pages][Hkv][page_rows][D] bf16  page pool of the committed rows
 *   block_table [B][L_cap / page_rows] int32   logical rows [i P, (i+1) P) of
 *                                               sequence b live in page
 *                                               block_table[b][i] (P = page_rows)
 *   Kt, Vt [B][Hkv][N][D] bf16                  the tree nodes' keys and values,
 *                                               staged outside the cache
 *   Q, L, anc_bits, O, workspace                as for medusa_tree_attention
 * Every node attends to the logical rows [0, L_b) and to its ancestors-or-self
 * among the staged rows. page_rows must be a positive multiple of 128 dividing
 * cfg->L_cap; bf16 with D = 128 only (MEDUSA_ERR_UNSUPPORTED otherwise). */
MEDUSA_API int medusa_tree_attention_paged(const medusa_cfg* cfg, const void* Q, const void* Kp, const void* Vp,
                                int32_t num_pages, int32_t page_rows, const int32_t* block_table,
                                const void* Kt, const void* Vt, const int32_t* L, const uint64_t* anc_bits,
                                void* O, void* workspace, medusa_stream_t stream);

/* Commit the accepted path into a paged cache, in every layer.
 * For layer l < n_layers the pools are Kp + l * pool_layer_elems (elements of
 * the cfg's type; same for Vp) and the staged rows Kt + l * tree_layer_elems:
 * for r = 0..acc_b, logical row L_b + r of sequence b receives the staged row
 * path[b][r] in every KV head; then L_b += acc_b + 1 (in/out) and kv_map as for
 * medusa_kv_compact. Sequences with L_b < 0 or L_b + N > L_cap are left as they
 * are (kv_map = -1). Layouts and page_rows as for medusa_tree_attention_paged
 * (any dtype and D). A row whose block-table page id lies outside
 * [0, pool_layer_elems / (Hkv * page_rows * D)) is not written (when
 * pool_layer_elems is 0, with one layer, page ids are not range-checked). */
MEDUSA_API int medusa_kv_commit_paged(const medusa_cfg* cfg, void* Kp, void* Vp, int32_t page_rows,
                           const int32_t* block_table, const void* Kt, const void* Vt, int32_t n_layers,
                           size_t pool_layer_elems, size_t tree_layer_elems, int32_t* L, const int32_t* acc,
                           const int32_t* path, int32_t* kv_map, medusa_stream_t stream);

/* Tree attention for callers that cannot allocate device memory.
 * No counterpart on the source pages: this is a deployment variant of
 * medusa_tree_attention for callers that cannot call cudaMalloc (for example a
 * serving engine that reserved nearly all device memory for its KV cache at
 * start-up and forbids later allocations, or a plug-in inside a framework whose
 * allocator owns every device byte). Arguments, layouts and results are those
 * of medusa_tree_attention; there is no workspace argument. The split-KV
 * partial results live instead in one static device array of
 * MEDUSA_NOALLOC_SCRATCH_BYTES that the library holds on every GPU that loads
 * it, until the process exits.
 *   - Returns MEDUSA_ERR_UNSUPPORTED, enqueueing nothing, when the
 *     configuration needs more scratch than that. The scratch it needs is the
 *     tree-attention share of medusa_workspace_size: B * S * N * Hq * D * 4
 *     bytes of partial outputs and B * S * N * Hq * 2 * 4 bytes of running
 *     maxima and sums for the S KV splits the library picks (1 <= S <= 32,
 *     more only while the grid fits one wave), plus, on the bf16 D = 128
 *     path when a KV head's N * Hq / Hkv query rows leave 1..8 rows past its
 *     full 128-row tiles, B * Hkv * S * (full tiles) * 8 * (D + 2) * 4 bytes
 *     for those rows; each part is rounded up to 256 bytes. A refusal is
 *     immediate, so one call at set-up tells a caller whether a shape fits.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.
 *   - Every call uses the same array: calls whose kernels may overlap on the
 *     GPU (other streams, concurrent graph replays) race and must not be
 *     issued. Each call writes all the scratch it reads. */
#define MEDUSA_NOALLOC_SCRATCH_BYTES (64u << 20)
MEDUSA_API int medusa_tree_attention_noalloc(const medusa_cfg* cfg, const void* Q, const void* Kc, const void* Vc,
                                             const int32_t* L, const uint64_t* anc_bits, void* O,
                                             medusa_stream_t stream);

/* Failure detection. Every spin-wait of the tcgen05 kernels (the heads GEMVs and
 * tree attention: pipeline mbarriers, the softmax exchanges) is bounded by a
 * clock budget of about two seconds. On expiry the waiting thread ORs a code
 * naming the wait into a device word of its kernel family, leaves its loop, and
 * the kernel returns; the GPU context stays usable, but that call's outputs are
 * invalid. The acceptance walks report the same per sequence in `flags`
 * (MEDUSA_FLAG_TIMEOUT).
 * medusa_poll_errors reads and clears both words, in stream order, and then
 * synchronises `stream`. Returns MEDUSA_OK when no wait expired since the last
 * poll, MEDUSA_ERR_TIMEOUT when one did (the codes, if the pointers are not
 * NULL, receive the words' values: host pointers), MEDUSA_ERR_CUDA on a CUDA
 * error. Not capturable in a CUDA graph (it synchronises). */
MEDUSA_API int medusa_poll_errors(medusa_stream_t stream, uint32_t* heads_codes, uint32_t* attention_codes);

/* Self-test of that path: enqueues one kernel whose single thread waits on an
 * mbarrier that nothing completes, bounded by about `budget_us` microseconds
 * (1 .. 1000000; MEDUSA_ERR_INVALID_ARG otherwise). It faults nothing and hangs
 * nothing: after the budget it records MEDUSA_WAIT_SELFTEST_CODE in the
 * attention word and returns, so the next medusa_poll_errors returns
 * MEDUSA_ERR_TIMEOUT with that bit set in *attention_codes. */
#define MEDUSA_WAIT_SELFTEST_CODE 0x80000000u
MEDUSA_API int medusa_selftest_wait_timeout(uint32_t budget_us, medusa_stream_t stream);

/* Checked build. The library built with -DMEDUSA_CHECKED (libmedusa_checked.so)
 * runs the same kernels with range checks on every index they read from device
 * memory: root and top-s token ids (medusa_tree_build: [0, V)), the tree links
 * and child tokens a walk follows (medusa_verify), acc and the path's node ids
 * (medusa_kv_compact and medusa_kv_commit_paged: acc in [0, K], node ids in
 * [0, N), each deeper than the one before), and block-table page ids
 * (the paged calls: [0, pages)). Every build already clamps such an index or
 * skips the access it would make; the checked build also ORs the matching
 * MEDUSA_CHECK_* bit into a device word. Nothing traps.
 * medusa_checked_build returns 1 in the checked build, 0 otherwise.
 * medusa_poll_checks reads and clears those words in stream order, then
 * synchronises `stream`: MEDUSA_OK when no check failed since the last poll (and
 * always in the normal build, with *codes = 0), MEDUSA_ERR_BOUNDS when one did
 * (*codes, a host pointer that may be NULL, receives the OR of the bits),
 * MEDUSA_ERR_CUDA on a CUDA error. Not capturable in a CUDA graph. No
 * counterpart on the pages: a debug aid. */
#define MEDUSA_CHECK_TOKEN 0x1u  /* a token id outside [0, V)                                */
#define MEDUSA_CHECK_TREE 0x2u   /* a parent / first-child link outside the tree or inconsistent */
#define MEDUSA_CHECK_PATH 0x4u   /* acc outside [0, K] or a path node outside [0, N) / not deeper */
#define MEDUSA_CHECK_PAGE 0x8u   /* a block-table page id outside the pool                   */
MEDUSA_API int medusa_checked_build(void);
MEDUSA_API int medusa_poll_checks(medusa_stream_t stream, uint32_t* codes);

/* Number of kernels this library has enqueued in this process so far (host-side
 * counter, for diagnostics; no counterpart on the pages). */
MEDUSA_API uint64_t medusa_launch_count(void);

/* Human-readable text of a status code (static storage). */
MEDUSA_API const char* medusa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MEDUSA_H_ */
