// Rejection-sampling acceptance over the candidate tree.
//
// "Speculative decoding -- Draft, verify, and the expected tokens per step",
// introduction and "Maths": a drafted token x is accepted with probability
// min(1, p(x)/q(x)); at a rejection the replacement is drawn from the
// normalised positive residual [p - q]_+, and a fully accepted draft earns one
// more target token; the emitted tokens then follow the target exactly.
// "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
// Heads", Method 5: rejection sampling keeps the original model's
// distribution.  Walked along the tree (the pages give the rule for a chain):
// from the root, a node's children are tried in rank order against the
// target p at the node; after each rejection p becomes the normalised
// residual; q_k, the distribution of the head that drafted depth k, stays.
// The walk moves to the first accepted child; where it stops, the next token
// is drawn from p (inverse CDF).  Lossless when a node's children are
// independent draws from q_k.  The uniforms are inputs.
//
// One CTA of 1024 threads per sequence; p lives in a workspace row (V floats),
// q is recomputed from the draft logits when needed.  V-wide passes are
// block reductions; the final draw is a block-wide prefix sum in double.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace medusa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

MDEV float block_max(float v, float* red) {
  v = warp_max(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = lane < kWarps ? red[lane] : -INFINITY;
  return warp_max(v);
}

MDEV float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = lane < kWarps ? red[lane] : 0.f;
  return warp_sum(v);
}

// p = softmax(z * inv_tau) over V into prow.
MDEV void softmax_to(const float* z, int V, float inv_tau, float* prow, float* red) {
  float m = -INFINITY;
  for (int v = threadIdx.x; v < V; v += kThreads) m = fmaxf(m, z[v] * inv_tau);
  m = block_max(m, red);
  float S = 0.f;
  for (int v = threadIdx.x; v < V; v += kThreads) S += expf(z[v] * inv_tau - m);
  S = block_sum(S, red);
  const float inv = 1.f / S;
  for (int v = threadIdx.x; v < V; v += kThreads) prow[v] = expf(z[v] * inv_tau - m) * inv;
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads) reject_tree_kernel(
    const float* logits, const float* draft, int Kd, const int32_t* tokens, medusa_tree_t tree, int V,
    float inv_tau, const float* uni, int u_stride, int32_t* accept_len, int32_t* accepted_nodes,
    int32_t* next_token, float* pws, int32_t* err) {
  const int b = blockIdx.x, tid = threadIdx.x;
  const int T = tree.T, K = tree.K;
  float* P = pws + (int64_t)b * V;
  __shared__ float red[kWarps];
  __shared__ int kid_by_rank[MEDUSA_MAX_S + 1];
  __shared__ int kids[MEDUSA_MAX_S + 1];
  __shared__ int s_m, s_acc, s_tok;
  __shared__ float s_lse_q;
  __shared__ double chunk_sum[kThreads];

  int32_t* an = accepted_nodes + (int64_t)b * (K + 1);
  for (int j = tid; j <= K; j += kThreads) an[j] = j == 0 ? 0 : -1;
  softmax_to(logits + (int64_t)b * T * V, V, inv_tau, P, red);
  int cur = 0, len = 0, m = 0;
  for (int guard = 0; guard <= K; ++guard) {
    // children of cur in rank order (ranks of siblings are distinct, 1..MEDUSA_MAX_S)
    if (tid <= MEDUSA_MAX_S) kid_by_rank[tid] = -1;
    __syncthreads();
    for (int n = 1 + tid; n < T; n += kThreads)
      if (tree.parent[n] == cur) {
        const int r = tree.rank[n];
        if (r >= 1 && r <= MEDUSA_MAX_S) kid_by_rank[r] = n;
        else set_err(err, MEDUSA_DEVERR_NODE);
      }
    __syncthreads();
    if (tid == 0) {
      int c = 0;
      for (int r = 1; r <= MEDUSA_MAX_S; ++r)
        if (kid_by_rank[r] >= 0) kids[c++] = kid_by_rank[r];
      s_m = c;
    }
    __syncthreads();
    m = s_m;
    if (m == 0 || m >= u_stride) break;
    const int k = tree.depth[kids[0]];
    if (k < 1 || k > K || k > Kd) break;
    // q_k: log-sum-exp of the drafting head's logits
    const float* dz = draft + ((int64_t)b * Kd + (k - 1)) * V;
    {
      float mx = -INFINITY;
      for (int v = tid; v < V; v += kThreads) mx = fmaxf(mx, dz[v] * inv_tau);
      mx = block_max(mx, red);
      float S = 0.f;
      for (int v = tid; v < V; v += kThreads) S += expf(dz[v] * inv_tau - mx);
      S = block_sum(S, red);
      if (tid == 0) s_lse_q = mx + logf(S);
      __syncthreads();
    }
    const float lse_q = s_lse_q;
    int acc = -1;
    for (int j = 0; j < m; ++j) {
      const int n = kids[j];
      const int x = tokens[(int64_t)b * T + n];
      if (x < 0 || x >= V) {  // an invalid draft is never accepted
        if (tid == 0) set_err(err, MEDUSA_DEVERR_TOKEN);
        continue;
      }
      const float u = uni[((int64_t)b * T + cur) * u_stride + j];
      const float qx = expf(dz[x] * inv_tau - lse_q);
      const float px = P[x];
      if (u * qx < px) {
        acc = n;
        break;
      }
      // rejected: p <- [p - q]_+ normalised
      float S = 0.f;
      for (int v = tid; v < V; v += kThreads) {
        const float r = fmaxf(0.f, P[v] - expf(dz[v] * inv_tau - lse_q));
        P[v] = r;
        S += r;
      }
      S = block_sum(S, red);
      if (S > 0.f) {
        const float inv = 1.f / S;
        for (int v = tid; v < V; v += kThreads) P[v] *= inv;
      }
      __syncthreads();
    }
    if (acc < 0) break;
    ++len;
    if (tid == 0) an[len] = acc;
    cur = acc;
    softmax_to(logits + ((int64_t)b * T + cur) * V, V, inv_tau, P, red);
    m = 0;
  }
  // final draw: the first x with mass whose running sum of p exceeds u
  const float u = uni[((int64_t)b * T + cur) * u_stride + (m < u_stride ? m : u_stride - 1)];
  const int per = (V + kThreads - 1) / kThreads;
  const int v0 = min(V, tid * per), v1 = min(V, v0 + per);
  double loc = 0.0;  // running sums in double: the draw's boundaries stay exact to ~1e-12
  for (int v = v0; v < v1; ++v) loc += (double)P[v];
  chunk_sum[tid] = loc;
  if (tid == 0) s_tok = -1;
  __syncthreads();
  // exclusive prefix over the chunks (Hillis-Steele in shared memory)
  for (int off = 1; off < kThreads; off <<= 1) {
    const double add = tid >= off ? chunk_sum[tid - off] : 0.0;
    __syncthreads();
    chunk_sum[tid] += add;
    __syncthreads();
  }
  double c = chunk_sum[tid] - loc;  // mass before this thread's chunk
  if (v0 < v1 && (double)u < chunk_sum[tid] && (double)u >= c) {
    int tok = -1;
    for (int v = v0; v < v1 && tok < 0; ++v) {
      const float pv = P[v];
      if (pv <= 0.f) continue;
      c += (double)pv;
      if ((double)u < c) tok = v;
    }
    if (tok < 0)  // rounding: the last token with mass in the chunk
      for (int v = v1 - 1; v >= v0 && tok < 0; --v)
        if (P[v] > 0.f) tok = v;
    s_tok = tok;  // the chunks' running-sum intervals are disjoint: one thread at most gets here
  }
  __syncthreads();
  if (tid == 0) {
    int tok = s_tok;
    if (tok < 0)  // u beyond the rounded total: the last token with mass
      for (int v = V - 1; v >= 0 && tok < 0; --v)
        if (P[v] > 0.f) tok = v;
    accept_len[b] = len;
    next_token[b] = tok;
  }
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_accept_rejection_workspace_size(int B, int V) {
  if (B < 1 || V < 1) return 0;
  return align_up((size_t)B * V * sizeof(float), 256);
}

extern "C" int medusa_accept_rejection(const float* logits, const float* draft_logits, int Kd,
                                       const int32_t* tokens, const medusa_tree_t* tree, int B, int V,
                                       float temperature, const float* uniforms, int u_stride,
                                       int32_t* accept_len, int32_t* accepted_nodes, int32_t* next_token,
                                       void* workspace, size_t workspace_bytes, int32_t* err, void* stream) {
  const char* fn = "medusa_accept_rejection";
  if (int rc = check_tree(tree, fn)) return rc;
  if (!logits || !draft_logits || !tokens || !uniforms || !accept_len || !accepted_nodes || !next_token)
    return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (B < 1 || B > 65535 || V < 1 || Kd < tree->K || u_stride < 2)
    return fail(MEDUSA_ERR_INVALID, "%s: B=%d V=%d Kd=%d (tree depth %d) u_stride=%d", fn, B, V, Kd, tree->K,
                u_stride);
  if (!(temperature > 0.f)) return fail(MEDUSA_ERR_INVALID, "%s: temperature must be > 0", fn);
  const size_t need = medusa_accept_rejection_workspace_size(B, V);
  if (!workspace || workspace_bytes < need)
    return fail(MEDUSA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, workspace_bytes, need);
  launch_kernel(reject_tree_kernel, dim3(B), dim3(kThreads), 0, as_stream(stream), logits, draft_logits, Kd,
                tokens, *tree, V, 1.f / temperature, uniforms, u_stride, accept_len, accepted_nodes, next_token,
                static_cast<float*>(workspace), err);
  return check_launch(fn);
}
