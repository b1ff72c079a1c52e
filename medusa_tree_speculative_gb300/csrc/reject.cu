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
// One CTA of 1024 threads per sequence.  At each node the kernel
// exponentiates every logit once: a pass of maxima (the node's logits and
// the drafting head's, no exponentials), then a pass that writes
// e^(z/tau - max) for both to two workspace rows and sums them, so p and q
// are the rows times scalars.  A rejection is one pass that writes the
// residual [p - q]_+ over the target row and sums it; the acceptance tests
// and the final draw (per-warp segment sums in double, a prefix over the
// segments, a scan of one segment) read the rows.  Every pass keeps 16 loads
// in flight per thread: one CTA per sequence is latency-bound otherwise.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace medusa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

MDEV float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = lane < kWarps ? red[lane] : 0.f;
  return warp_sum(v);
}

// Two block-wide reductions at once (max or sum); every thread gets both.
template <bool MAX>
MDEV void block_pair(float& a, float& b, float2* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float xa = __shfl_xor_sync(0xffffffffu, a, o), xb = __shfl_xor_sync(0xffffffffu, b, o);
    a = MAX ? fmaxf(a, xa) : a + xa;
    b = MAX ? fmaxf(b, xb) : b + xb;
  }
  __syncthreads();
  if (lane == 0) red[warp] = make_float2(a, b);
  __syncthreads();
  const float init = MAX ? -INFINITY : 0.f;
  const float2 r = lane < kWarps ? red[lane] : make_float2(init, init);
  a = r.x;
  b = r.y;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float xa = __shfl_xor_sync(0xffffffffu, a, o), xb = __shfl_xor_sync(0xffffffffu, b, o);
    a = MAX ? fmaxf(a, xa) : a + xa;
    b = MAX ? fmaxf(b, xb) : b + xb;
  }
}

constexpr int kU = 16;  // loads in flight per thread in every V-wide pass

// Rows are read in rounds of kU coalesced loads per thread: element
// v = base + u * kThreads + threadIdx.x of round `base`.
#define MEDUSA_ROUNDS(V) for (int base = 0; base < (V); base += kU * kThreads)
#define MEDUSA_IDX(u) (base + (u) * kThreads + (int)threadIdx.x)

// The node's target row Pw and the drafting head's row Qw (workspace):
// p(v) = Pw[v] * sp, q(v) = Qw[v] * sq.  Rows are written with e^(y - max)
// of y = logit / tau once per node.
MDEV void exp_rows(const float* z, const float* dz, int V, float inv_tau, float* Pw, float* Qw, float& sp,
                   float& sq, float2* red) {
  float mp = -INFINITY, mq = -INFINITY;
  MEDUSA_ROUNDS(V) {
    float a[kU], c[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = MEDUSA_IDX(u);
      a[u] = v < V ? z[v] : -INFINITY;
      c[u] = (dz && v < V) ? dz[v] : -INFINITY;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      mp = fmaxf(mp, a[u] * inv_tau);
      mq = fmaxf(mq, c[u] * inv_tau);
    }
  }
  block_pair<true>(mp, mq, red);
  float Sp = 0.f, Sq = 0.f;
  MEDUSA_ROUNDS(V) {
    float a[kU], c[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = MEDUSA_IDX(u);
      a[u] = v < V ? z[v] : 0.f;
      c[u] = (dz && v < V) ? dz[v] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = MEDUSA_IDX(u);
      if (v < V) {
        const float ep = expf(a[u] * inv_tau - mp);
        Pw[v] = ep;
        Sp += ep;
        if (dz) {
          const float eq = expf(c[u] * inv_tau - mq);
          Qw[v] = eq;
          Sq += eq;
        }
      }
    }
  }
  block_pair<false>(Sp, Sq, red);  // its barriers also publish the rows
  sp = 1.f / Sp;
  sq = dz ? 1.f / Sq : 0.f;
}

// p <- [p - q]_+ (unnormalised, over Pw); returns its sum.
MDEV float residual(float* Pw, const float* Qw, float sp, float sq, int V, float* red) {
  float S = 0.f;
  MEDUSA_ROUNDS(V) {
    float a[kU], c[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = MEDUSA_IDX(u);
      a[u] = v < V ? Pw[v] : 0.f;
      c[u] = v < V ? Qw[v] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = MEDUSA_IDX(u);
      if (v < V) {
        const float r = fmaxf(0.f, a[u] * sp - c[u] * sq);
        Pw[v] = r;
        S += r;
      }
    }
  }
  return block_sum(S, red);  // its barriers also publish the residual row
}

MDEV double warp_sum_d(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Inverse CDF: the first v with p(v) = Pw[v] * sp > 0 whose running sum of p,
// in index order and in double, exceeds u; the last v with mass when u is
// beyond the total.  Warp w takes the w-th contiguous segment of V: segment
// sums, an exclusive prefix over the segments, then the one warp whose
// interval holds u scans its segment 32 elements at a time.  Result valid
// in every thread.
MDEV int draw(const float* Pw, float sp, int V, double u, double* wsum, int* s_tok) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = (V + kWarps - 1) / kWarps;
  const int s0 = min(V, warp * seg), s1 = min(V, s0 + seg);
  double acc = 0.0;
  for (int base = s0; base < s1; base += 32 * kU) {
    float a[kU];
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int v = base + q * 32 + lane;
      a[q] = v < s1 ? Pw[v] : 0.f;
    }
#pragma unroll
    for (int q = 0; q < kU; ++q) acc += (double)(a[q] * sp);
  }
  acc = warp_sum_d(acc);
  if (lane == 0) wsum[warp] = acc;
  if (threadIdx.x == 0) *s_tok = -1;
  __syncthreads();
  double before = 0.0;  // the same sums in the same order in every warp: the intervals are disjoint
  for (int w = 0; w < warp; ++w) before += wsum[w];
  if (s0 < s1 && u >= before && u < before + wsum[warp]) {
    double run = before;
    int tok = -1;
    for (int base = s0; base < s1 && tok < 0; base += 32) {
      const int v = base + lane;
      const float pv = v < s1 ? Pw[v] * sp : 0.f;
      double c = (double)pv;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, c, o);
        if (lane >= o) c += y;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, pv > 0.f && u < run + c);
      if (hit) tok = base + __ffs(hit) - 1;
      run += __shfl_sync(0xffffffffu, c, 31);
    }
    for (int base = s1 - 32; tok < 0 && base > s0 - 32; base -= 32) {  // rounding: the segment's last with mass
      const int v = base + lane;
      const unsigned hit = __ballot_sync(0xffffffffu, v >= s0 && v < s1 && Pw[v] * sp > 0.f);
      if (hit) tok = base + 31 - __clz(hit);
    }
    if (lane == 0) *s_tok = tok;
  }
  __syncthreads();
  int tok = *s_tok;
  if (tok < 0) {  // u beyond the rounded total: the last token with mass
    __syncthreads();
    if (threadIdx.x == 0)
      for (int v = V - 1; v >= 0 && *s_tok < 0; --v)
        if (Pw[v] * sp > 0.f) *s_tok = v;
    __syncthreads();
    tok = *s_tok;
  }
  return tok;
}

__global__ void __launch_bounds__(kThreads) reject_tree_kernel(
    const float* logits, const float* draft, int Kd, const int32_t* tokens, medusa_tree_t tree, int V,
    float inv_tau, const float* uni, int u_stride, int32_t* accept_len, int32_t* accepted_nodes,
    int32_t* next_token, float* pws, int32_t* err) {
  const int b = blockIdx.x, tid = threadIdx.x;
  const int T = tree.T, K = tree.K;
  float* Pw = pws + (int64_t)b * 2 * V;  // target row
  float* Qw = Pw + V;                    // drafting head's row
  __shared__ float red[kWarps];
  __shared__ float2 red2[kWarps];
  __shared__ int kid_by_rank[MEDUSA_MAX_S + 1];
  __shared__ int kids[MEDUSA_MAX_S + 1];
  __shared__ int s_m, s_tok;
  __shared__ double wsum[kWarps];

  int32_t* an = accepted_nodes + (int64_t)b * (K + 1);
  for (int j = tid; j <= K; j += kThreads) an[j] = j == 0 ? 0 : -1;
  float sp = 0.f, sq = 0.f;
  int cur = 0, len = 0, m = 0;
  for (int guard = 0;; ++guard) {
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
    const int k = m > 0 ? tree.depth[kids[0]] : 0;
    const bool walk = guard <= K && m > 0 && m < u_stride && k >= 1 && k <= K && k <= Kd;
    const float* dz = walk ? draft + ((int64_t)b * Kd + (k - 1)) * V : nullptr;
    // p at this node (and q of the children's head when the walk goes on)
    exp_rows(logits + ((int64_t)b * T + cur) * V, dz, V, inv_tau, Pw, Qw, sp, sq, red2);
    if (!walk) break;
    int acc = -1;
    for (int j = 0; j < m; ++j) {
      const int n = kids[j];
      const int x = tokens[(int64_t)b * T + n];
      if (x < 0 || x >= V) {  // an invalid draft is never accepted
        if (tid == 0) set_err(err, MEDUSA_DEVERR_TOKEN);
        continue;
      }
      const float u = uni[((int64_t)b * T + cur) * u_stride + j];
      const float qx = Qw[x] * sq;
      const float px = Pw[x] * sp;
      if (u * qx < px) {
        acc = n;
        break;
      }
      // rejected: p <- [p - q]_+ / sum, the residual and its sum in one pass
      const float S = residual(Pw, Qw, sp, sq, V, red);
      sp = S > 0.f ? 1.f / S : 0.f;
    }
    if (acc < 0) break;
    ++len;
    if (tid == 0) an[len] = acc;
    cur = acc;
    m = 0;
  }
  // final draw from p at the node where the walk stopped
  const float u = uni[((int64_t)b * T + cur) * u_stride + (m < u_stride ? m : u_stride - 1)];
  const int tok = draw(Pw, sp, V, (double)u, wsum, &s_tok);
  if (tid == 0) {
    accept_len[b] = len;
    next_token[b] = tok;
  }
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_accept_rejection_workspace_size(int B, int V) {
  if (B < 1 || V < 1) return 0;
  return align_up((size_t)B * 2 * V * sizeof(float), 256);  // target and draft rows per sequence
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
