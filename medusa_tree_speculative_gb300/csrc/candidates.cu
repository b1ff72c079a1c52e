// Candidate fill for the next step.
//
// "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
// Heads", decoding-step box (steps 1-2): the root gets the LM head's choice
// t0, and the node for rank path (i_1..i_k) gets the i_k-th best token of
// Medusa head k.  With the tree in breadth-first layout this is a gather:
// tokens[n] = topk[depth[n]-1][rank[n]-1].
#include "common.cuh"
#include "internal.h"

namespace medusa {
namespace {

__global__ void __launch_bounds__(MEDUSA_MAX_T) build_candidates_kernel(
    const int32_t* next_root, const int32_t* topk, int s_max, int K, medusa_tree_t tree,
    int32_t* tokens) {
  const int b = blockIdx.x, n = threadIdx.x;
  if (n >= tree.T) return;
  int32_t tok;
  if (n == 0) {
    tok = next_root[b];
  } else {
    const int k = tree.depth[n] - 1, r = tree.rank[n] - 1;
    tok = (k >= 0 && k < K && r >= 0 && r < s_max) ? topk[((int64_t)b * K + k) * s_max + r] : -1;
  }
  tokens[(int64_t)b * tree.T + n] = tok;
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" int medusa_build_candidates(const int32_t* next_root, const int32_t* topk, int s_max, int K,
                                       const medusa_tree_t* tree, int B, int32_t* tokens, void* stream) {
  const char* fn = "medusa_build_candidates";
  if (int rc = check_tree(tree, fn)) return rc;
  if (!next_root || !topk || !tokens) return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (B < 1 || B > MEDUSA_MAX_B || s_max < 1 || K < tree->K)
    return fail(MEDUSA_ERR_INVALID, "%s: B=%d s_max=%d K=%d (tree depth %d)", fn, B, s_max, K, tree->K);
  for (int k = 0; k < tree->K; ++k)
    if (tree->s[k] > s_max) return fail(MEDUSA_ERR_INVALID, "%s: tree s[%d]=%d > s_max=%d", fn, k, tree->s[k], s_max);
  launch_kernel(build_candidates_kernel, dim3(B), dim3((tree->T + 31) / 32 * 32), 0, as_stream(stream), next_root,
             topk, s_max, K, *tree, tokens);
  return check_launch(fn);
}
