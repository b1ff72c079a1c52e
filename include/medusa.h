/*
 * medusa.h -- C ABI of libmedusa: the data-parallel hot path of one Medusa
 * tree-speculative decoding step on a single GB300 (sm_103a).
 *
 * Sources (cited by page title and section):
 *   [MED]  "Medusa: Simple LLM Inference Acceleration Framework with Multiple
 *          Decoding Heads" (paper digest): Method items 1-5; the box
 *          "Algorithm: Medusa decoding step"; "Paper vs code"; "Pitfalls".
 *   [MEDZ] "085 | Medusa" explainer: section 二.2 (tree attention) and 二.3
 *          (strict and typical acceptance).
 *
 * One verify step is six calls, enqueued in this order on one stream:
 *   medusa_tree_attn        tree-masked attention + KV append   (box step 3)
 *   medusa_lm_head_verify   LM head over every tree row          (box step 3)
 *   medusa_accept           greedy / typical acceptance          (box 4-5)
 *   medusa_kv_compact       accepted path's KV into place        (box 6)
 *   medusa_heads_topk       K Medusa heads + top-s               (box 1)
 *     (or: medusa_heads_hidden over every tree row, which can run beside the
 *      acceptance, then medusa_heads_logits_topk on the accepted row; or
 *      medusa_lm_head_verify_heads_hidden in place of the LM head call, one
 *      pass computing both, then medusa_heads_logits_topk)
 *   medusa_build_candidates next step's candidate tokens         (box 2)
 *     (medusa_heads_topk_candidates: the last two in one call)
 * In a decode loop, medusa_append_tokens (box step 6) appends each step's
 * tokens to the output.
 *
 * Conventions
 *   - Every step call returns MEDUSA_OK (0) or a negative status; on error
 *     nothing was enqueued and medusa_last_error() (per thread) says why.
 *   - The library never allocates, frees or synchronises.  All pointers are
 *     owned by the caller; tensors are dense, row-major, with the shapes given
 *     below.  "device" pointers must be CUDA device (or managed) memory of the
 *     current device; "host" pointers are read during the call only.
 *   - Work is enqueued on `stream` (a cudaStream_t; 0 = legacy default).
 *   - Scratch ("workspace") is caller-provided device memory of at least the
 *     size returned by the matching *_workspace_size query, 256-byte aligned.
 *     Its contents are not preserved.  Calls whose kernels hand out work or
 *     elect a last CTA through counters kept in it (medusa_accept,
 *     medusa_heads_topk, medusa_heads_logits_topk) need it zero-filled before
 *     the first call and leave it ready for the next call of the same entry
 *     point; the others need no initialisation.
 *   - Device-side data errors (a token or node index out of range, a prefix
 *     that overflows its sequence's capacity) cannot be seen by the host
 *     without a synchronisation.  Calls that read such data take `err`, a
 *     nullable device int32: a kernel that meets bad data ORs a
 *     MEDUSA_DEVERR_* bit into *err and skips the offending access.  Nothing
 *     traps.
 *   - Element types: MEDUSA_F32 (IEEE binary32) or MEDUSA_BF16 (bfloat16).
 *     Logits are always float32; accumulation is always float32.
 *
 * Tree layout (medusa_tree_t)
 *   T = 1 + N rows: row 0 is the root (the token chosen by the previous step),
 *   rows 1..N the candidate nodes in breadth-first order (depth, then
 *   lexicographic rank path), so every parent precedes its children.  A node
 *   at depth k with rank r holds the r-th best token of Medusa head k
 *   ([MED] Method 2).  anc_mask row i, bit j (word j/32, bit j%32) is set iff
 *   node j is an ancestor of i or i itself ([MED] Method 3).
 */
#ifndef MEDUSA_H
#define MEDUSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MEDUSA_MAX_T 512  /* tree rows, root included */
#define MEDUSA_MAX_K 8    /* tree depth / Medusa heads */
#define MEDUSA_MAX_S 16   /* top-s per head */
#define MEDUSA_MAX_B 16   /* sequences per call */

typedef enum { MEDUSA_F32 = 0, MEDUSA_BF16 = 1 } medusa_dtype;

enum {
  MEDUSA_OK = 0,
  MEDUSA_ERR_INVALID = -1,     /* null pointer, bad shape or tree */
  MEDUSA_ERR_UNSUPPORTED = -2, /* dtype or size outside the supported set */
  MEDUSA_ERR_CAPACITY = -3,    /* a known size exceeds a buffer's capacity */
  MEDUSA_ERR_WORKSPACE = -4,   /* workspace smaller than the query returned */
  MEDUSA_ERR_CUDA = -5         /* a CUDA runtime call or launch failed */
};

/* bits ORed into the device error word */
enum {
  MEDUSA_DEVERR_TOKEN = 1,    /* token outside [0, V) */
  MEDUSA_DEVERR_NODE = 2,     /* node index outside [0, T) */
  MEDUSA_DEVERR_CAPACITY = 4, /* prefix_len + T exceeds seq_cap */
  MEDUSA_DEVERR_LENGTH = 8,   /* accept_len outside [0, K] */
  MEDUSA_DEVERR_TIMEOUT = 16  /* a bounded on-chip wait gave up (internal fault) */
};

typedef struct medusa_tree {
  const int32_t* parent;    /* device [T]; parent[0] = -1, parent[i] < i */
  const int32_t* depth;     /* device [T]; depth[0] = 0 */
  const int32_t* rank;      /* device [T]; 1-based rank, rank[0] = 0 */
  const uint32_t* anc_mask; /* device [T][W] ancestor-or-self bitmask */
  int32_t T;                /* rows, 1 <= T <= MEDUSA_MAX_T */
  int32_t W;                /* words per mask row = ceil(T / 32) */
  int32_t K;                /* tree depth (deepest node), <= MEDUSA_MAX_K */
  int32_t s[MEDUSA_MAX_K];  /* largest rank used at depth k+1 (host values) */
} medusa_tree_t;

/* Thread-local description of the last error returned on this thread. */
const char* medusa_last_error(void);
/* Library version string. */
const char* medusa_version(void);

/* ======================= host tree helpers (no CUDA) ===================== */

/* Compile a set of rank paths into the breadth-first layout above
 * ([MED] Method 2 and 3).  paths: host [n_paths][max_depth], 1-based ranks,
 * row i uses its first path_len[i] entries; any order.  Every proper prefix
 * of a path must itself be in the set.  Outputs (host, caller-sized):
 * parent/depth/rank [n_paths+1], anc_mask [(n_paths+1) * W] with
 * W = ceil((n_paths+1)/32), s [max_depth], node_paths [n_paths+1][max_depth]
 * (nullable; zero padded).  *T_out = n_paths + 1, *K_out = deepest level.
 * Returns MEDUSA_ERR_INVALID on a duplicate, a missing prefix or a rank < 1,
 * MEDUSA_ERR_UNSUPPORTED if T > MEDUSA_MAX_T or depth > MEDUSA_MAX_K or a
 * rank > MEDUSA_MAX_S. */
int medusa_tree_compile(const int32_t* paths, const int32_t* path_len,
                        int n_paths, int max_depth, int32_t* parent,
                        int32_t* depth, int32_t* rank, uint32_t* anc_mask,
                        int32_t* s, int32_t* node_paths, int* T_out,
                        int* K_out);

/* Cartesian candidate tree ([MED] Method 2, fig. 2): all paths with
 * i_k <= s[k], breadth-first, cut after max_nodes non-root nodes.
 * paths: host [max_nodes][K]; returns the node count or a negative status. */
int medusa_tree_cartesian(const int32_t* s, int K, int max_nodes,
                          int32_t* paths, int32_t* path_len);

/* Greedy sparse tree ([MED] Method 4): node accuracy is the product of the
 * per-head top-i accuracies acc[k][i-1] along its path; starting from the
 * root, add the connected node of highest accuracy (ties within 1e-9 in log
 * space go to the lexicographically smallest path) until `budget` nodes.
 * acc: host [K][R]; paths: host [budget][K].  Returns the node count. */
int medusa_tree_greedy(const double* acc, int K, int R, int budget,
                       int32_t* paths, int32_t* path_len);

/* =============================== step calls ============================== */

/* Scratch bytes medusa_tree_attn needs for these sizes. */
size_t medusa_tree_attn_workspace_size(int B, int H, int Dh, int T,
                                       int max_prefix);

/* Tree-masked attention with tree position ids ([MED] Method 3, Pitfalls;
 * [MEDZ] 二.2).
 *   q, k_new, v_new: device [B][T][H][Dh], pre-rotation projections of the
 *                    tree rows.
 *   k_cache, v_cache: device [tokens][H][Dh]; sequence b owns rows
 *                    [seq_start[b], seq_start[b] + seq_cap[b]); its first
 *                    prefix_len[b] rows hold already-rotated keys.
 *   seq_start [B] int64, prefix_len [B] int32, seq_cap [B] int64: device.
 *   max_prefix: host upper bound on every prefix_len[b] (sizes the grid).
 * For row i of sequence b at depth d_i, with L = prefix_len[b]:
 *   pos = L + d_i;  q', k' = RoPE(q, pos), RoPE(k_new, pos) (rotate-half
 *   pairs (j, j + Dh/2), inv_freq_j = rope_theta^(-2j/Dh), angle formed in
 *   float32);  k', v_new are written to slot seq_start[b] + L + i;
 *   out[b][i] = softmax(scale * q' . K_S^T) V_S over S = the L prefix slots
 *   plus the slots of every ancestor-or-self of i.
 * out: device [B][T][H][Dh] (dtype).  Dh must be 64 or 128.
 * A sequence with L + T > seq_cap[b] sets MEDUSA_DEVERR_CAPACITY and is
 * skipped; L > max_prefix does the same. */
int medusa_tree_attn(const void* q, const void* k_new, const void* v_new,
                     void* k_cache, void* v_cache, const int64_t* seq_start,
                     const int32_t* prefix_len, const int64_t* seq_cap,
                     const medusa_tree_t* tree, int B, int H, int Dh,
                     int max_prefix, float rope_theta, float scale,
                     medusa_dtype dtype, void* out, void* workspace,
                     size_t workspace_bytes, int32_t* err, void* stream);

/* medusa_tree_attn with the number of CTAs that split the keys of one
 * (sequence, head, block of up to 80 query rows), bf16 only: key_splits = 8
 * (what medusa_tree_attn uses) spreads the work over many short CTAs;
 * key_splits = 1 runs one long CTA per unit (32 CTAs for one sequence of 32
 * heads), for a caller that runs the attention on SMs that a concurrent
 * kernel leaves idle; 2 and 4 lie between.  Same results up to the
 * order of the fp32 softmax sums.  Other values: MEDUSA_ERR_UNSUPPORTED. */
int medusa_tree_attn_splits(const void* q, const void* k_new,
                            const void* v_new, void* k_cache, void* v_cache,
                            const int64_t* seq_start,
                            const int32_t* prefix_len, const int64_t* seq_cap,
                            const medusa_tree_t* tree, int B, int H, int Dh,
                            int max_prefix, float rope_theta, float scale,
                            medusa_dtype dtype, void* out, void* workspace,
                            size_t workspace_bytes, int key_splits,
                            int32_t* err, void* stream);

/* medusa_tree_attn on the tensor cores (tcgen05 MMAs with the accumulators
 * in tensor memory, TMA tile loads), bf16 with Dh = 128 only.  A cluster of
 * key_splits CTAs (1, 2, 4 or 8) per (sequence, head, block of up to 128
 * query rows) takes contiguous runs of the key tiles of 128; S = Q K^T and
 * P V run on the tensor cores, the masked online softmax on two threads per
 * query row.  With key_splits > 1 each CTA keeps its partial (max, sum, O) in
 * its shared memory and, after a cluster barrier, finalises one slice of the
 * output columns from every CTA's partial through distributed shared memory.
 * The CTA whose tiles hold the tree's keys first appends them (rotated) and
 * the values to the cache (every row block of a sequence writes the same
 * bytes) and reads them back with the prefix.  cache_rows: rows of k_cache /
 * v_cache (the tiles' loads stop there).  Same arguments otherwise (no
 * workspace), same results up to the order of the fp32 sums; a bounded
 * on-chip wait that gives up sets MEDUSA_DEVERR_TIMEOUT.  Other dtypes, head
 * sizes or key_splits: MEDUSA_ERR_UNSUPPORTED. */
int medusa_tree_attn_tc(const void* q, const void* k_new, const void* v_new,
                        void* k_cache, void* v_cache, int64_t cache_rows,
                        const int64_t* seq_start, const int32_t* prefix_len,
                        const int64_t* seq_cap, const medusa_tree_t* tree,
                        int B, int H, int Dh, int max_prefix,
                        float rope_theta, float scale, medusa_dtype dtype,
                        void* out, int key_splits, int32_t* err,
                        void* stream);

/* Copy `bytes` from page-locked, device-mapped host memory (src_host, e.g.
 * cudaHostAlloc) into device memory (dst) with a kernel of 16-byte loads,
 * enqueued on `stream`: the step's inputs staged from host buffers.  Both
 * pointers and `bytes` must be multiples of 16; the runtime is asked for the
 * host buffer's device address first, and memory that is not mapped returns
 * MEDUSA_ERR_INVALID without launching anything.  No counterpart in the
 * pages: the end-to-end step's host-to-device leg. */
int medusa_copy_from_host(void* dst, const void* src_host, size_t bytes,
                          void* stream);

/* Read-out of a device error word (the `err` argument of the step calls).
 * Enqueues on `stream` one single-thread kernel that writes *err into *out
 * and then, if clear != 0, sets *err back to 0, so that the next step starts
 * from a clean word.  err: device memory.  out: device memory or page-locked
 * host memory mapped into the device's address space (e.g. cudaHostAlloc, or
 * a pinned torch tensor); *out holds the word once the stream has reached
 * this point, and the call itself does not synchronise.  The bits are the
 * MEDUSA_DEVERR_* values above.  Returns MEDUSA_ERR_INVALID for a NULL or
 * misaligned pointer, or memory the device cannot address.  No counterpart
 * in the pages: the error convention of this library. */
int medusa_check_errors(int32_t* err, int32_t* out, int clear, void* stream);

/* Scratch bytes medusa_lm_head_verify needs (currently 0). */
size_t medusa_lm_head_workspace_size(int rows, int d, int V);

/* Layout of the vocabulary matrix handed to medusa_lm_head_verify.
 *   MEDUSA_W_ROWS   [V][d] row-major (nn.Linear layout).
 *   MEDUSA_W_TILES  bf16 only: the matrix cut into tiles of 128 vocabulary
 *                   rows x 64 columns, each tile 16 KB contiguous (row-major
 *                   inside), tiles ordered by vocabulary block, then column
 *                   block.  Element (v, j) sits at element offset
 *                     ((v / 128) * (d / 64) + j / 64) * 8192
 *                       + (v % 128) * 64 + j % 64,
 *                   rows v >= V of the last block are zero.  Every load the
 *                   tensor-core kernel issues is then one contiguous 16 KB
 *                   run of HBM instead of 128 runs of 128 bytes; the decode
 *                   step is memory-bound ([MED] "Problem"), so this is the
 *                   layout to keep resident.  Written by medusa_lm_head_tile. */
typedef enum { MEDUSA_W_ROWS = 0, MEDUSA_W_TILES = 1 } medusa_w_layout;

/* Bytes of the MEDUSA_W_TILES copy of a bf16 [V][d] matrix:
 * ceil(V / 128) * 128 * d * 2 (d a multiple of 64), 0 for invalid sizes. */
size_t medusa_lm_head_tiled_bytes(int d, int V);

/* Rewrite a row-major bf16 w_lm [V][d] (device) into the MEDUSA_W_TILES
 * layout at w_tiled (device, medusa_lm_head_tiled_bytes(d, V) bytes, 16-byte
 * aligned, must not overlap w_lm).  Any row-major [R][d] matrix can be tiled
 * the same way (the heads' W1 as [K*d][d] for medusa_heads_hidden).  A
 * one-off preparation step with no counterpart in the paper; the copy is
 * exact.  Returns MEDUSA_ERR_UNSUPPORTED when d is not a multiple of 64. */
int medusa_lm_head_tile(const void* w_lm, void* w_tiled, int d, int V,
                        void* stream);

/* Verification LM head over every tree row ([MED] Method 3, box step 3):
 *   logits[r][v] = sum_j hidden[r][j] * w_lm[v][j]
 * hidden: device [rows][d]; w_lm: device, [V][d] in the layout w_layout
 * names; logits: device [rows][V] float32.  bf16: d must be a multiple of 64
 * and both inputs 16-byte aligned; both layouts give bit-identical logits.
 * f32 accepts MEDUSA_W_ROWS only.  The tensor-core kernel's bounded on-chip
 * waits report MEDUSA_DEVERR_TIMEOUT through err (nullable) if they ever
 * give up.  Rows beyond 256 are processed in balanced chunks of at most 256
 * that multiply the same weight k-block (the weights are read once); 257 to
 * 264 rows as one 256-row chunk plus the rest by mma.sync beside it; 129 to
 * 256 rows run on clusters of two CTAs (one tcgen05 MMA of M = 256 over a
 * vocabulary tile of each, each CTA loading half of the hidden rows). */
int medusa_lm_head_verify(const void* hidden, const void* w_lm, float* logits,
                          int rows, int d, int V, medusa_dtype dtype,
                          medusa_w_layout w_layout, void* workspace,
                          size_t workspace_bytes, int32_t* err, void* stream);

/* CTAs (one per SM; both CTAs of each pair counted) that
 * medusa_lm_head_verify launches for bf16 `rows` x V on the current device,
 * 0 for invalid sizes.  A caller that runs other work
 * beside the LM head (the tree attention of the same step) sizes it to the
 * SMs left free.  No counterpart in the pages. */
int medusa_lm_head_ctas(int rows, int V);

/* The LM head with the acceptance's row statistics fused into its epilogue
 * (the logits round trip skipped).  For every tree row r and vocabulary group
 * g (a run of 128 or 256 vocabulary rows; medusa_lm_head_stat_groups(rows, V)
 * groups on the current device) one 16-byte record
 *   { max_v z[r][v], its index (lowest among equal maxima),
 *     sum_v e^(y_v - m), sum_v e^(y_v - m)(y_v - m) }   over v in g,
 * y = z / temperature, m = max y (the sums are 0 in greedy mode), stored as
 * float4 at stats[g * rows + r] (the index's bits in the second float).
 * medusa_accept_stats merges them.  logits (device [rows][V] float32) is
 * optional in greedy mode (NULL: not written) and required in typical mode
 * (p^(token) is read from it).  mode 0 greedy, 1 typical.  bf16 only; the
 * other arguments as medusa_lm_head_verify.  Returns MEDUSA_ERR_CAPACITY if
 * stats_bytes < groups * rows * 16. */
int medusa_lm_head_stat_groups(int rows, int V);
int medusa_lm_head_verify_stats(const void* hidden, const void* w_lm,
                                float* logits, int rows, int d, int V,
                                medusa_dtype dtype, medusa_w_layout w_layout,
                                int mode, float temperature, void* stats,
                                size_t stats_bytes, int32_t* err,
                                void* stream);

/* medusa_accept from the statistics of medusa_lm_head_verify_stats (groups =
 * medusa_lm_head_stat_groups(B*T, V), stats covering B*T rows): the same
 * rules, ties and outputs as medusa_accept, one kernel, no workspace;
 * logits (device [B][T][V]) is read only in typical mode. */
int medusa_accept_stats(const void* stats, int groups, const float* logits,
                        const int32_t* tokens, const medusa_tree_t* tree,
                        int B, int V, int mode, float temperature, float eps,
                        float delta, int32_t* accept_len,
                        int32_t* accepted_nodes, int32_t* next_root,
                        int32_t* best_node, float* best_logp, int32_t* err,
                        void* stream);

/* Scratch bytes medusa_accept needs. */
size_t medusa_accept_workspace_size(int B, int T);

/* Acceptance ([MED] Method 5, box steps 4-5; [MEDZ] 二.3).
 *   logits: device [B][T][V] float32 (the LM head at every tree row);
 *   tokens: device [B][T] int32, the candidate tokens that were verified.
 * Node c (c >= 1, parent p) passes when
 *   mode 0 (greedy):  argmax_v logits[p][v] == tokens[c]  (lowest index wins
 *                     among equal maxima);
 *   mode 1 (typical): p^(tokens[c]) > min(eps, delta * exp(-H(p^))), with
 *                     p^ = softmax(logits[p] / temperature) and H its entropy.
 * The root always passes; a node is accepted when it and all its ancestors
 * pass.  The best node is the accepted node of greatest depth; ties go to the
 * larger summed log p^ (typical), then to the lower node index.
 * Outputs (device): accept_len [B] = depth of the best node;
 * accepted_nodes [B][K+1] (root .. best, -1 padded; K = tree->K);
 * next_root [B] = argmax of the best node's row; best_node [B];
 * best_logp [B] float32 (summed log p^ of the accepted non-root nodes;
 * 0 for greedy; nullable).
 * One kernel: a CTA per tree row, and the last row of each sequence to finish
 * (a counter in the workspace) makes that sequence's decisions.  The
 * workspace must therefore be zero-filled (cudaMemset) before its first call;
 * every call leaves its counters zero again. */
int medusa_accept(const float* logits, const int32_t* tokens,
                  const medusa_tree_t* tree, int B, int V, int mode,
                  float temperature, float eps, float delta,
                  int32_t* accept_len, int32_t* accepted_nodes,
                  int32_t* next_root, int32_t* best_node, float* best_logp,
                  void* workspace, size_t workspace_bytes, int32_t* err,
                  void* stream);

/* Allocation-free variant of medusa_accept.  The paper has no counterpart:
 * this entry point exists for callers that cannot allocate device memory,
 * such as a plugin or a plain C host program that is handed only input and
 * output pointers by the framework that owns the GPU's memory, or a decode
 * loop that must not call cudaMalloc because it can synchronise the device
 * and take unbounded time.
 * Arguments, outputs and errors are those of medusa_accept, without the
 * workspace.  Its scratch is one file-scope __device__ array, zero when the
 * library loads, of 256 bytes of counters and MEDUSA_ACCEPT_NOALLOC_MAX_ROWS
 * row records of 64 bytes (512 KiB), which every GPU that loads the library
 * holds until the process exits.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it for the
 *     device's current context; make that first call before any stream
 *     capture.  After cudaDeviceReset the next call finds a new context and
 *     looks the address up again (the array, reloaded with the module, is
 *     zero again): make that call outside capture too.
 *   - B * tree->T above MEDUSA_ACCEPT_NOALLOC_MAX_ROWS returns
 *     MEDUSA_ERR_CAPACITY.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Every call shares the one array, which keeps the last call's row
 *     records and leaves its counters zero.  Calls that overlap on the GPU
 *     (other streams or threads without ordering between them) race on it:
 *     the caller serialises them. */
#define MEDUSA_ACCEPT_NOALLOC_MAX_ROWS (MEDUSA_MAX_B * MEDUSA_MAX_T)
int medusa_accept_noalloc(const float* logits, const int32_t* tokens,
                          const medusa_tree_t* tree, int B, int V, int mode,
                          float temperature, float eps, float delta,
                          int32_t* accept_len, int32_t* accepted_nodes,
                          int32_t* next_root, int32_t* best_node,
                          float* best_logp, int32_t* err, void* stream);

/* KV compaction to the accepted path ([MED] box step 6, Pitfalls: the
 * accepted KV must be gathered into contiguous slots, not sliced).
 * For each sequence b with L = prefix_len[b], A = accept_len[b]:
 *   slot L + j <- slot L + accepted_nodes[b][j] for j = 0..A (K and V; every
 *   source is read before any destination is written);
 *   prefix_len[b] = L + A + 1;  src_slots[b][j] = L + accepted_nodes[b][j]
 *   for j <= A, -1 after (nullable).
 * accepted_nodes, accept_len, prefix_len (in-out), src_slots: device.
 * Kmax: the row stride of accepted_nodes minus one (= tree->K).  T: the
 * tree's rows (= tree->T), which medusa_tree_attn appended at slots
 * L .. L + T - 1.  A sequence whose accept_len is outside [0, Kmax] sets
 * MEDUSA_DEVERR_LENGTH, one whose accepted_nodes[b][j] is outside [j, T)
 * sets MEDUSA_DEVERR_NODE; either is left untouched (prefix_len included). */
int medusa_kv_compact(void* k_cache, void* v_cache, const int64_t* seq_start,
                      int32_t* prefix_len, const int32_t* accepted_nodes,
                      const int32_t* accept_len, int B, int H, int Dh,
                      int Kmax, int T, medusa_dtype dtype, int32_t* src_slots,
                      int32_t* err, void* stream);

/* Scratch bytes medusa_heads_topk needs. */
size_t medusa_heads_topk_workspace_size(int B, int K, int d, int V,
                                        int s_max);

/* Medusa heads and top-s ([MED] Method 1 and 2; "Paper vs code": optional
 * ResBlock bias).  For each sequence b and each head k with s[k] > 0:
 *   h = hidden[b][last_node[b]];
 *   u = dtype( SiLU(W1_k h + b1_k) + h )        (rounded to the weight type)
 *   head_logits[b][k] = W2_k u                  (float32)
 *   topk[b][k][0 .. s[k]-1] = indices of the s[k] largest logits (value
 *   descending, index ascending); topk[b][k][s[k] ..] = -1.
 * hidden: device [B][T][d]; last_node: device [B] (row index < T, usually
 * medusa_accept's best_node); w1: device [K][d][d] (out x in); b1: device
 * [K][d] or NULL; w2: device [K][V][d]; s: host [K], 0 <= s[k] <= s_max <=
 * MEDUSA_MAX_S; head_logits: device [B][K][V] (rows of skipped heads are not
 * written); topk: device [B][K][s_max].
 * Both projections hand their rows out at run time from counters in the
 * workspace, so that CTAs whose SMs are still busy with concurrent work take
 * fewer rows.  Unlike other scratch, this workspace must be zero-filled
 * (cudaMemset) before its first call; every call leaves the counters ready
 * for the next one (zero it again only after a call that failed to launch). */
int medusa_heads_topk(const void* hidden, const int32_t* last_node, int T,
                      const void* w1, const void* b1, const void* w2,
                      const int32_t* s, int K, int B, int d, int V,
                      medusa_dtype dtype, float* head_logits, int32_t* topk,
                      int s_max, void* workspace, size_t workspace_bytes,
                      int32_t* err, void* stream);

/* medusa_heads_topk followed by medusa_build_candidates in one call: the
 * heads' W2 kernel, once the last head's top-s is merged, writes the next
 * step's candidate tokens (tokens[b][0] = next_root[b], tokens[b][n] =
 * topk[b][depth[n]-1][rank[n]-1]), saving the candidate kernel's launch on
 * the step's critical path.  Arguments and workspace (zero-filled once) as
 * medusa_heads_topk; next_root, tree and tokens as medusa_build_candidates
 * (K >= tree->K, tree->s[k] <= s_max). */
int medusa_heads_topk_candidates(const void* hidden, const int32_t* last_node,
                                 int T, const void* w1, const void* b1,
                                 const void* w2, const int32_t* s, int K, int B,
                                 int d, int V, medusa_dtype dtype,
                                 float* head_logits, int32_t* topk, int s_max,
                                 void* workspace, size_t workspace_bytes,
                                 const int32_t* next_root,
                                 const medusa_tree_t* tree, int32_t* tokens,
                                 int32_t* err, void* stream);

/* The heads' first projection for every tree row ([MED] Method 1, computed
 * ahead of the acceptance):
 *   u[r][k] = dtype( SiLU(W1_k hidden[r] + b1_k) + hidden[r] )
 * for every row r < rows and every head k with s[k] > 0 (entries of other
 * heads are not written).  Running it over all rows, not only the accepted
 * node's, costs no extra weight bytes (W1 is read once either way: a GEMM
 * on the tensor cores instead of a GEMV) and no longer depends on the
 * acceptance, so it can overlap it; medusa_heads_logits_topk then reads the
 * accepted node's row.  hidden: device [rows][d]; w1: device [K][d][d]
 * (out x in) in w1_layout (MEDUSA_W_TILES: medusa_lm_head_tile of w1 seen as
 * a [K*d][d] matrix); b1: device [K][d] or NULL; s: host [K]; u: device
 * [rows][K][d] of dtype.  bf16: d a multiple of 128, 16-byte aligned
 * tensors, bounded on-chip waits as medusa_lm_head_verify; f32: rows
 * layout only.  Rows beyond 256 run in chunks of at most 256 (W1 is read
 * once per chunk). */
int medusa_heads_hidden(const void* hidden, int rows, const void* w1,
                        medusa_w_layout w1_layout, const void* b1,
                        const int32_t* s, int K, int d, medusa_dtype dtype,
                        void* u, int32_t* err, void* stream);

/* medusa_lm_head_verify and medusa_heads_hidden in one launch, bf16 only:
 * the logits of every tree row and u (as medusa_heads_hidden) for every row
 * and used head.  Both products take the same hidden rows as the MMA's N
 * side, so one CTA streams its share of the W tiles and of the stacked W1
 * tiles over a single pass of the hidden k-blocks; the launch takes the
 * fewest CTAs (at most one per SM) that keep every CTA at no more than three
 * (at most four) 128-row weight tiles, which leaves the other SMs free for
 * concurrent work such as the tree attention.  Arguments as the two calls
 * (w_lm [V][d] in w_layout, w1 [K][d][d] in w1_layout, b1 nullable, s host
 * [K], logits [rows][V] fp32, u [rows][K][d] bf16).  rows <= 256, d a
 * multiple of 128, 16-byte aligned tensors; MEDUSA_ERR_UNSUPPORTED when no
 * plan fits (the caller then makes the two calls).  With no used head it is
 * medusa_lm_head_verify. */
int medusa_lm_head_verify_heads_hidden(const void* hidden, int rows, int d,
                                       const void* w_lm,
                                       medusa_w_layout w_layout, int V,
                                       float* logits, const void* w1,
                                       medusa_w_layout w1_layout,
                                       const void* b1, const int32_t* s, int K,
                                       void* u, medusa_dtype dtype,
                                       int32_t* err, void* stream);

/* Scratch bytes medusa_heads_logits_topk needs. */
size_t medusa_heads_logits_topk_workspace_size(int B, int K, int V, int s_max);

/* The heads' second projection and top-s ([MED] Method 1 and 2) from
 * medusa_heads_hidden's output: for each sequence b and head k with s[k] > 0,
 *   head_logits[b][k] = W2_k u[b * T + node[b]][k]   (float32)
 *   topk[b][k][..] as medusa_heads_topk.
 * u: device [B*T][K][d]; node: device [B] (usually medusa_accept's
 * best_node; outside [0, T) raises MEDUSA_DEVERR_NODE and reads row 0); w2,
 * s, head_logits, topk as medusa_heads_topk.  The workspace holds per-head
 * arrival counters that must be zero on entry: zero it once (cudaMemset)
 * before the first call; every call leaves it zeroed again (after a call
 * that reported MEDUSA_DEVERR_TIMEOUT, zero it again). */
int medusa_heads_logits_topk(const void* u, int T, const int32_t* node,
                             const void* w2, const int32_t* s, int K, int B,
                             int d, int V, medusa_dtype dtype,
                             float* head_logits, int32_t* topk, int s_max,
                             void* workspace, size_t workspace_bytes,
                             int32_t* err, void* stream);

/* Candidate fill for the next step ([MED] box steps 1-2):
 *   tokens[b][0] = next_root[b];
 *   tokens[b][n] = topk[b][depth[n]-1][rank[n]-1] for n >= 1.
 * next_root: device [B]; topk: device [B][K][s_max] with K >= tree->K;
 * tokens: device [B][T]. */
int medusa_build_candidates(const int32_t* next_root, const int32_t* topk,
                            int s_max, int K, const medusa_tree_t* tree,
                            int B, int32_t* tokens, void* stream);

/* Scratch bytes medusa_accept_rejection needs (2 B rows of V floats: the
 * target and draft rows of each sequence). */
size_t medusa_accept_rejection_workspace_size(int B, int V);

/* Rejection-sampling acceptance over the tree, an alternative to
 * medusa_accept's greedy / typical rules that keeps the target
 * distribution ([MED] Method 5; [SPEC] introduction and "Maths": accept a
 * drafted x with probability min(1, p(x)/q(x)), at a rejection draw from the
 * normalised residual [p - q]_+).  Walked along the tree: from the root, the
 * children of the current node are tried in rank order, child n (depth k,
 * token x = tokens[b][n]) being accepted iff
 *     uniforms[b][cur][j] * q_k(x) < p(x)        (j = its position in that order)
 * with p = softmax(logits[b][cur] / temperature), replaced by the normalised
 * residual after each rejection, and q_k = softmax(draft_logits[b][k-1] /
 * temperature), the distribution of the head that drafted depth k.  The walk
 * moves to the accepted child and repeats; where it stops (no child accepted,
 * or a node without children) the next token is the first x, in vocabulary
 * order, whose running sum of p exceeds uniforms[b][cur][m], m = the number
 * of children of that node.  Lossless when the children of every node are
 * independent draws from q_k.
 * logits: device [B][T][V] float32; draft_logits: device [B][Kd][V] float32
 * (Kd >= tree->K; e.g. medusa_heads_topk's head_logits of the previous
 * step); tokens: device [B][T]; uniforms: device [B][T][u_stride] in [0, 1),
 * u_stride greater than every node's child count (MEDUSA_MAX_S + 1 always
 * suffices).  Outputs (device): accept_len [B], accepted_nodes [B][K+1] (root
 * .. last accepted node, -1 padded), next_token [B] (the token drawn after the
 * accepted path).  B may be up to 65535 here.  A draft token outside [0, V)
 * is never accepted and raises MEDUSA_DEVERR_TOKEN. */
int medusa_accept_rejection(const float* logits, const float* draft_logits,
                            int Kd, const int32_t* tokens,
                            const medusa_tree_t* tree, int B, int V,
                            float temperature, const float* uniforms,
                            int u_stride, int32_t* accept_len,
                            int32_t* accepted_nodes, int32_t* next_token,
                            void* workspace, size_t workspace_bytes,
                            int32_t* err, void* stream);

/* Append a step's output tokens ([MED] box step 6: "append the root plus the
 * accepted tokens", 1 + accept_len of them):
 *   out[b][out_len[b] + j] = tokens[b][accepted_nodes[b][j]], j = 0..accept_len[b]
 *   out_len[b] += accept_len[b] + 1.
 * tokens: device [B][T] (the step's tree tokens); accepted_nodes: device
 * [B][Kmax+1] and accept_len: device [B] (medusa_accept's outputs); out:
 * device [B][out_cap]; out_len: device [B], in/out.  A sequence whose
 * accept_len is outside [0, Kmax] (MEDUSA_DEVERR_LENGTH), whose output would
 * pass out_cap (MEDUSA_DEVERR_CAPACITY) or whose path holds a node outside
 * [0, T) (MEDUSA_DEVERR_NODE) is left with out_len unchanged. */
int medusa_append_tokens(const int32_t* tokens, const int32_t* accepted_nodes,
                         const int32_t* accept_len, int B, int T, int Kmax,
                         int32_t* out, int32_t* out_len, int out_cap,
                         int32_t* err, void* stream);

/* A stand-in for the backbone forward, with no counterpart in the paper:
 *   hidden[r] = emb[tokens[r]], r < rows
 * so that the verify step can run in a closed loop on the device without a
 * transformer (the stand-in model's hidden state of a token is its embedding
 * row; attention inputs are taken from the same rows).  tokens: device
 * [rows]; emb: device [V][d] of dtype; hidden: device [rows][d].  Rows must
 * be multiples of 16 bytes, pointers 16-byte aligned.  A token outside
 * [0, V) gives a zero row and MEDUSA_DEVERR_TOKEN. */
int medusa_standin_embed(const int32_t* tokens, int rows, const void* emb,
                         int V, int d, medusa_dtype dtype, void* hidden,
                         int32_t* err, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MEDUSA_H */
