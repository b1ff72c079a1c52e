/*
 * oracle.h -- CPU oracle for one Medusa tree-speculative verify step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library, its
 * Python binding) may include, link, load or call this code.  Only the tests,
 * the smoke check and the CPU-baseline leg of the benchmark use it.
 *
 * The oracle is plain, single-threaded C99 with double accumulation.  It
 * follows the method as stated on the pages it cites, with no blocking,
 * fusion or reordering beyond the definitions.  It shares no code, header,
 * table or constant with the GPU library.
 *
 * Sources (cited by page title and section):
 *   [MED]  "Medusa: Simple LLM Inference Acceleration Framework with Multiple
 *          Decoding Heads" (paper digest page): Method items 1-5, the box
 *          "Algorithm: Medusa decoding step", "Paper vs code", "Pitfalls".
 *   [MEDZ] "085 | Medusa: 让一个模型提前猜多步，再一次验证候选树" (explainer):
 *          section 二.2 (tree attention), 二.3 (strict vs typical acceptance),
 *          the two-token worked example, "候选树中相同深度不表示相同上下文".
 *   [SPEC] "Speculative decoding -- Draft, verify, and the expected tokens per
 *          step": section "Maths".
 *
 * Element types: ORC_F32 (IEEE binary32) and ORC_BF16 (raw bfloat16 bits,
 * uint16).  Inputs are widened exactly to double; outputs stored in a narrow
 * type are rounded to nearest, ties to even.
 *
 * Every function returns 0 on success and a negative value on a bad argument.
 */
#ifndef MEDUSA_ORACLE_H
#define MEDUSA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1 };

/* ---- element access ---------------------------------------------------- */
double   orc_load(const void* p, int dt, int64_t i);
void     orc_store(void* p, int dt, int64_t i, double x);
uint16_t orc_bf16_round(double x);  /* nearest bf16, ties to even */

/* ---- candidate tree ([MED] Method 2 and 4, algorithm box step 2) -------- */
/* paths: [n_paths][max_depth] 1-based ranks (ragged, path_len[i] used).
 * Output in breadth-first order (depth, then lexicographic path); node 0 is
 * the root (empty path).  T = n_paths + 1.
 *   node_paths [T][max_depth] (zero padded), parent [T], depth [T], rank [T],
 *   anc [T][T] (1 iff column node is an ancestor-or-self of row node),
 *   s [max_depth] (largest rank used at each depth, 0 past the tree's depth).
 * Returns T, or -1 on a malformed set (duplicate, missing prefix, rank < 1). */
int orc_tree_compile(const int32_t* paths, const int32_t* path_len, int n_paths,
                     int max_depth, int32_t* node_paths, int32_t* parent,
                     int32_t* depth, int32_t* rank, uint8_t* anc, int32_t* s,
                     int32_t* K_out);

/* Cartesian tree: every path (i_1..i_k), k <= K, i_j <= s_j, in breadth-first
 * order, cut after max_nodes non-root nodes.  Returns the node count. */
int orc_tree_cartesian(const int32_t* s, int K, int max_nodes,
                       int32_t* paths /*[max_nodes][K]*/, int32_t* path_len);

/* Greedy sparse tree ([MED] Method 4): node accuracy = prod_j acc[j][i_j-1];
 * repeatedly add the connected node of highest accuracy (ties within 1e-9 in
 * log space go to the lexicographically smallest path) until `budget` nodes.
 * acc: [K][R].  Returns the node count; paths in the order they were added. */
int orc_tree_greedy(const double* acc, int K, int R, int budget,
                    int32_t* paths /*[budget][K]*/, int32_t* path_len);

/* Expected acceptance length of a tree: 1 + sum over nodes of prod_j acc. */
double orc_tree_expected_len(const int32_t* paths, const int32_t* path_len,
                             int n_paths, int max_depth, const double* acc,
                             int R);

/* ---- rotary position embedding (rotate-half pairing (i, i+Dh/2)) -------- */
/* x [Dh] rotated in place for position pos; angle = fp32(pos) * fp32(inv_freq)
 * formed in fp32, inv_freq_i = fp32(theta^(-2i/Dh)), cos/sin in double. */
void orc_rope(double* x, int Dh, int64_t pos, double theta);

/* ---- tree attention ([MED] Method 3; [MEDZ] 二.2) ----------------------- */
/* q, k_new, v_new: [B][T][H][Dh] (dt).  k_cache, v_cache: [tokens][H][Dh]
 * (dt); the prefix rows [seq_start[b], seq_start[b]+prefix_len[b]) hold
 * already-rotated keys.  Row i of sequence b is rotated at position
 * prefix_len[b] + depth[i], written into slot seq_start[b]+prefix_len[b]+i,
 * and attends to the prefix plus every node j with anc[i][j] = 1.
 * out: [B][T][H][Dh] (dt); out_d (nullable) receives the unrounded result. */
int orc_tree_attn(int dt, const void* q, const void* k_new, const void* v_new,
                  void* k_cache, void* v_cache, const int64_t* seq_start,
                  const int32_t* prefix_len, const int32_t* depth,
                  const uint8_t* anc, int T, int B, int H, int Dh,
                  double rope_theta, double scale, void* out, double* out_d);

/* Plain attention of one query over n keys (no mask): the reference that
 * tree attention must reduce to along each root-to-node path ([MEDZ]
 * "候选树中相同深度不表示相同上下文"). */
void orc_attn_one(int n, int Dh, const double* q, const double* k,
                  const double* v, double scale, double* out);

/* ---- LM head over all tree rows ([MED] Method 3, algorithm box step 3) -- */
/* hidden [rows][d] (dt), w [V][d] (dt) -> logits [rows][V] in double. */
int orc_lm_head(int dt, const void* hidden, const void* w, int rows, int d,
                int V, double* logits);

/* ---- acceptance ([MED] Method 5, algorithm box steps 4-5) --------------- */
/* logits [B][T][V] fp32, tokens [B][T].  mode 0 greedy, 1 typical.
 * Outputs: accept_len [B], accepted_nodes [B][K+1] (root..best, -1 padded),
 * next_root [B] (argmax of the best node's row), best_node [B],
 * best_logp [B] (sum of log p-hat over the accepted non-root nodes; 0 for
 * greedy).  Diagnostics (nullable): row_gap [B][T] (top1 - top2 logit),
 * node_margin [B][T] (typical: p-hat(tok) - threshold; greedy: 1/0/-1 for
 * match/no match), node_logp [B][T] (running path log-prob). */
int orc_accept(const float* logits, const int32_t* tokens,
               const int32_t* parent, const int32_t* depth, int T, int K,
               int B, int V, int mode, double temperature, double eps,
               double delta, int32_t* accept_len, int32_t* accepted_nodes,
               int32_t* next_root, int32_t* best_node, double* best_logp,
               double* row_gap, double* node_margin, double* node_logp);

/* ---- KV compaction ([MED] algorithm box step 6, Pitfalls) --------------- */
/* For j = 0..A: slot L+j <- slot L+a_j (K and V), prefix_len += A+1,
 * src_slots [B][K+1] = L + a_j (or -1). */
int orc_kv_compact(int dt, void* k_cache, void* v_cache,
                   const int64_t* seq_start, int32_t* prefix_len,
                   const int32_t* accepted_nodes, const int32_t* accept_len,
                   int B, int H, int Dh, int K, int32_t* src_slots);

/* ---- Medusa heads + top-s ([MED] Method 1 and 2) ------------------------ */
/* h = hidden[b][last_node[b]];  u = dt(SiLU(W1_k h + b1_k) + h);
 * z = W2_k u;  topk[b][k][0..s_k-1] = indices of the s_k largest z (value
 * descending, index ascending), -1 after.  Heads with s[k] = 0 are skipped.
 * hidden [B][T][d]; w1 [K][d][d]; b1 [K][d] or NULL; w2 [K][V][d] (all dt).
 * head_logits [B][K][V] double; u_out (nullable) [B][K][d] dt. */
int orc_heads(int dt, const void* hidden, const int32_t* last_node, int T,
              const void* w1, const void* b1, const void* w2, const int32_t* s,
              int K, int B, int d, int V, double* head_logits, int32_t* topk,
              int s_max, void* u_out);

/* Top-s of fp32 values (value descending, index ascending). */
int orc_topk_f32(const float* z, int V, int s, int32_t* out);

/* ---- candidate fill ([MED] algorithm box steps 1-2) --------------------- */
/* tokens[b][0] = next_root[b]; tokens[b][n] = topk[b][depth n - 1][rank n - 1]. */
int orc_build_candidates(const int32_t* next_root, const int32_t* topk,
                         int s_max, int K, const int32_t* depth,
                         const int32_t* rank, int T, int B, int32_t* tokens);

/* ---- rejection-sampling verification ([SPEC] Maths; [MEDZ] example) ----- */
/* Emitted distribution of one draft-then-verify step:
 * min(p,q) + (1-beta) * [p-q]_+ / (1-beta);  returns beta = sum min(p,q). */
double orc_rejection_emit(const double* p, const double* q, int n,
                          double* emitted);

/* ---- rejection-sampling acceptance over the tree ------------------------ */
/* [SPEC] "Maths" and the verify rule of its introduction (accept a drafted x
 * with probability min(1, p(x)/q(x)); at a rejection draw from the residual
 * [p-q]_+ normalised; a fully accepted draft earns one more target token),
 * walked along the candidate tree (reading: a node's children are tried in
 * rank order; after each rejection the target becomes the normalised
 * residual; q stays the drafting head's distribution).  Lossless when the
 * children of a node are independent draws from q.  Per sequence b, from the
 * root: p = softmax(logits[b][node] / tau); child n of depth k is drafted
 * from q_k = softmax(draft[b][k-1] / tau); child j of node n is accepted iff
 * u[b][n][j] * q(x) < p(x); the final token is the first x whose running sum
 * of p exceeds u[b][n][m], m = the number of children of the node where the
 * walk stopped.  Arrays: logits [B][T][V] and draft [B][K][V] float32,
 * tokens [B][T], parent/depth/rank [T], u [B][T][u_stride] (u_stride > the
 * largest child count).  Outputs accept_len [B], accepted_nodes [B][K+1]
 * (-1 padded), next_token [B]; margin [B] (nullable) = the smallest relative
 * gap |u q - p| / max(p, q) of the tests made and of the final draw to a
 * running-sum boundary (a diagnostic of how close float rounding came to
 * changing a decision).  Returns 0, or -1 on bad arguments. */
int orc_rejection_tree(const float* logits, const float* draft,
                       const int32_t* tokens, const int32_t* parent,
                       const int32_t* depth, const int32_t* rank, int T,
                       int K, int B, int V, double temperature,
                       const float* u, int u_stride, int32_t* accept_len,
                       int32_t* accepted_nodes, int32_t* next_token,
                       double* margin);

#ifdef __cplusplus
}
#endif
#endif
