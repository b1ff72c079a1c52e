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
// Two kernels.  The first computes, for every tree row's target logits and
// every drafting head's logits at once (two 512-thread CTAs per row), the
// softmax statistics (max, sum e^(y - max)) of y = logit / tau, so that the
// walk tests a drafted token in O(1): p(x) = e^(y_x - m) / S.  The walk runs
// on a thread-block cluster of 8 CTAs (1024 threads each) per sequence, each
// CTA owning one eighth of the vocabulary and keeping its slices of the
// current p and of the node's q in shared memory; sums are combined through
// distributed shared memory.  A rejection is one pass over the slices that
// writes the residual [p - q]_+ (at a node's first rejection p and q come
// from the logits and the statistics) and returns, through the same cluster
// reduction as its sum, the residual at the next child's token, so the CTAs
// never read one another's slices; the final draw writes p out first unless
// a rejection there did, then takes per-warp segment sums in double, a
// prefix over the CTAs and the segments, and a scan of one segment.  Every
// pass keeps 16 loads in flight per thread.
#include <math.h>

#include "cluster.cuh"
#include "common.cuh"
#include "internal.h"

namespace medusa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kCluster = 8;  // CTAs per sequence, each owning a slice of the vocabulary
constexpr int kU = 16;       // loads in flight per thread in every V-wide pass

template <bool MAX>
MDEV float op2(float x, float y) { return MAX ? fmaxf(x, y) : x + y; }

// Two block-wide reductions at once (max or sum); every thread gets both.
template <bool MAX>
MDEV void block_pair(float& a, float& b, float2* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = op2<MAX>(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = op2<MAX>(b, __shfl_xor_sync(0xffffffffu, b, o));
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
    a = op2<MAX>(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = op2<MAX>(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
}

MDEV double warp_sum_d(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ---- thread-block cluster: barrier and distributed shared memory

// Reductions over the cluster's CTAs: a block reduction, each CTA's result
// in its exchange slot (two slots used in turn: a CTA reuses a slot only
// after the next cluster barrier, which every reader of it has reached),
// one cluster barrier, then every thread combines the CTAs' values in rank
// order, so every CTA gets the same bits.  The barrier's release / acquire
// also publishes the workspace rows each CTA wrote before it.
struct ClusterRed {
  float2* red;   // [kWarps] block scratch
  float2* xf;    // [2] exchange slots, floats
  double* xd;    // [2] exchange slots, doubles
  int ph;
  template <bool MAX>
  MDEV void pair(float& a, float& b) {
    block_pair<MAX>(a, b, red);
    const int slot = ph++ & 1;
    if (threadIdx.x == 0) xf[slot] = make_float2(a, b);
    cluster_sync();
    float ra = MAX ? -INFINITY : 0.f, rb = ra;
#pragma unroll
    for (int r = 0; r < kCluster; ++r) {
      const float2 v = ld_cluster_f2(cluster_map(smem_u32(&xf[slot]), (uint32_t)r));
      ra = op2<MAX>(ra, v.x);
      rb = op2<MAX>(rb, v.y);
    }
    a = ra;
    b = rb;
  }
  MDEV float sum(float a) {
    float b = 0.f;
    pair<false>(a, b);
    return a;
  }
  // every CTA's double (one per CTA, written by thread 0) in rank order
  MDEV void gather_d(double mine, double* out) {
    const int slot = ph++ & 1;
    if (threadIdx.x == 0) xd[slot] = mine;
    cluster_sync();
#pragma unroll
    for (int r = 0; r < kCluster; ++r) out[r] = ld_cluster_f64(cluster_map(smem_u32(&xd[slot]), (uint32_t)r));
  }
};

// A CTA's passes cover its slice [lo, hi) of the vocabulary in rounds of kU
// coalesced loads per thread: element lo + base + u * kThreads + threadIdx.x.
#define MEDUSA_ROUNDS(lo, hi) for (int base = (lo); base < (hi); base += kU * kThreads)
#define MEDUSA_IDX(u) (base + (u) * kThreads + (int)threadIdx.x)

// ---- row statistics, all rows at once (a separate kernel before the walk)
// (max, sum e^(y - max)) of y = logit / tau for every tree row's target
// logits and every drafting head's logits, two 512-thread CTAs per row (one
// per half of the vocabulary), so that the walk tests a drafted token in
// O(1): p(x) = e^(y_x - m) / S.
constexpr int kStatThreads = 512;

struct Soft2 {
  float m, S;
};
MDEV Soft2 soft2_merge(Soft2 a, Soft2 b) {
  if (a.m == -INFINITY) return b;
  if (b.m == -INFINITY) return a;
  const float M = fmaxf(a.m, b.m);
  return Soft2{M, a.S * expf(a.m - M) + b.S * expf(b.m - M)};
}

__global__ void __launch_bounds__(kStatThreads) reject_stats_kernel(const float* logits, const float* draft, int T,
                                                                    int Kd, int V, float inv_tau, float2* stats) {
  const int row = blockIdx.x >> 1, half = blockIdx.x & 1, b = blockIdx.y;
  const float* z = row < T ? logits + ((int64_t)b * T + row) * V : draft + ((int64_t)b * Kd + (row - T)) * V;
  const int lo = (int)((int64_t)V * half / 2), hi = (int)((int64_t)V * (half + 1) / 2);
  Soft2 t{-INFINITY, 0.f};
  for (int v0 = lo + (int)threadIdx.x; v0 < hi; v0 += kU * kStatThreads) {
    float y[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = v0 + u * kStatThreads;
      y[u] = v < hi ? __ldg(z + v) * inv_tau : -INFINITY;
    }
    float m = t.m;
#pragma unroll
    for (int u = 0; u < kU; ++u) m = fmaxf(m, y[u]);
    float S = t.m == -INFINITY ? 0.f : t.S * expf(t.m - m);
#pragma unroll
    for (int u = 0; u < kU; ++u) S += y[u] == -INFINITY ? 0.f : expf(y[u] - m);
    t = Soft2{m, S};
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    t = soft2_merge(t, Soft2{__shfl_xor_sync(0xffffffffu, t.m, o), __shfl_xor_sync(0xffffffffu, t.S, o)});
  __shared__ float2 part[kStatThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) part[warp] = make_float2(t.m, t.S);
  __syncthreads();
  if (warp == 0) {
    t = lane < kStatThreads / 32 ? Soft2{part[lane].x, part[lane].y} : Soft2{-INFINITY, 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      t = soft2_merge(t, Soft2{__shfl_xor_sync(0xffffffffu, t.m, o), __shfl_xor_sync(0xffffffffu, t.S, o)});
    if (lane == 0) stats[((int64_t)b * (T + Kd) + row) * 2 + half] = make_float2(t.m, t.S);
  }
}

// A row's (max, sum) from its two halves (the same bits in every CTA).
MDEV Soft2 row_soft(const float2* stats, int64_t idx) {
  const float2 a = __ldcg(stats + 2 * idx), c = __ldcg(stats + 2 * idx + 1);
  return soft2_merge(Soft2{a.x, a.y}, Soft2{c.x, c.y});
}

// This CTA's slice of p, unnormalised (sP[v - lo] = e^(y_v - m)); returns
// the cluster-wide sum, so that p = sP / sum.
MDEV float materialize(const float* z, float inv_tau, float m, float* sP, int lo, int hi, ClusterRed& R) {
  float S = 0.f;
  MEDUSA_ROUNDS(lo, hi) {
    float a[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = MEDUSA_IDX(u);
      a[u] = v < hi ? z[v] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = MEDUSA_IDX(u);
      if (v < hi) {
        const float e = expf(a[u] * inv_tau - m);
        sP[v - lo] = e;
        S += e;
      }
    }
  }
  return R.sum(S);  // its cluster barrier also publishes the slice
}

// p <- [p - q]_+ over this CTA's slice sP (unnormalised).  At a node's first
// rejection (!MAT) p and q come from the logits and the row statistics
// (p(v) = e^(y_v - P.m) / P.S, q likewise from the drafting head's logits)
// and q is kept in sQ for the node's later rejections; afterwards p(v) =
// sP[v - lo] * sp.  Returns the cluster-wide sum and the new (unnormalised)
// value at token xn (-1: none), which only the CTA owning xn contributes, so
// that every CTA tests the next child on the same bits without reading
// another CTA's slice.
template <bool MAT>
MDEV float2 residual(const float* z, const float* dz, float inv_tau, Soft2 P, Soft2 Q, float* sP, float* sQ,
                     float sp, int xn, int lo, int hi, ClusterRed& R) {
  const float ip = 1.f / P.S, iq = 1.f / Q.S;
  float S = 0.f, rx = 0.f;
  MEDUSA_ROUNDS(lo, hi) {
    float a[kU], c[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = MEDUSA_IDX(u);
      a[u] = v < hi ? (MAT ? sP[v - lo] : z[v]) : 0.f;
      c[u] = v < hi ? (MAT ? sQ[v - lo] : dz[v]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = MEDUSA_IDX(u);
      if (v < hi) {
        const float pv = MAT ? a[u] * sp : expf(a[u] * inv_tau - P.m) * ip;
        const float qv = MAT ? c[u] : expf(c[u] * inv_tau - Q.m) * iq;
        if (!MAT) sQ[v - lo] = qv;
        const float r = fmaxf(0.f, pv - qv);
        sP[v - lo] = r;
        S += r;
        if (v == xn) rx = r;
      }
    }
  }
  R.pair<false>(S, rx);  // rx is nonzero in one thread of one CTA at most
  return make_float2(S, rx);
}

// The last v in [lo, hi) with p(v) > 0 (-1 if none), in every thread; sP is
// this CTA's slice (sP[v - lo]).
MDEV int last_with_mass(const float* sP, float sp, int lo, int hi, float2* red) {
  float best = -1.f, dummy = -1.f;  // indices below 2^24 are exact in float
  for (int v = lo + (int)threadIdx.x; v < hi; v += kThreads)
    if (sP[v - lo] * sp > 0.f) best = (float)v;
  block_pair<true>(best, dummy, red);
  return (int)best;
}

// Inverse CDF over the cluster: the first v with p(v) = sP[v - lo] * sp > 0
// whose running sum of p, in index order and in double, exceeds u; the last
// v with mass when u is beyond the total.  Each warp of each CTA sums a
// contiguous segment of the CTA's slice; the CTAs' totals are exchanged and
// summed in rank order (the same bits in every CTA, so the CTAs' intervals
// are disjoint); the CTA whose interval holds u finds the warp whose
// segment holds it, and that warp scans its segment 32 elements at a time.
// Returns the token in the CTA that found it (rank 0 for the beyond-total
// case), -2 in the others.
MDEV int draw(const float* sP, float sp, int lo, int hi, double u, double* wsum, int* s_tok, ClusterRed& R,
              int crank) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = (hi - lo + kWarps - 1) / kWarps;
  const int s0 = min(hi, lo + warp * seg), s1 = min(hi, s0 + seg);
  double acc = 0.0;
  for (int base = s0; base < s1; base += 32 * kU) {
    float a[kU];
#pragma unroll
    for (int q = 0; q < kU; ++q) {
      const int v = base + q * 32 + lane;
      a[q] = v < s1 ? sP[v - lo] : 0.f;
    }
#pragma unroll
    for (int q = 0; q < kU; ++q) acc += (double)(a[q] * sp);
  }
  acc = warp_sum_d(acc);
  if (lane == 0) wsum[warp] = acc;
  if (threadIdx.x == 0) *s_tok = -2;
  __syncthreads();
  double mine = 0.0, off = 0.0;  // this CTA's total, and the mass before this warp's segment
  for (int w = 0; w < kWarps; ++w) {
    if (w == warp) off = mine;
    mine += wsum[w];
  }
  double tot[kCluster];
  R.gather_d(mine, tot);
  double before = 0.0, total = 0.0;
  for (int r = 0; r < kCluster; ++r) {
    if (r == crank) before = total;
    total += tot[r];
  }
  if (u >= total) {  // beyond the rounded total: the last token with mass, cluster-wide
    float last = (float)last_with_mass(sP, sp, lo, hi, R.red), dummy = -1.f;
    R.pair<true>(last, dummy);
    return crank == 0 ? (int)last : -2;
  }
  const bool mine_u = u >= before && u < before + tot[crank];  // exactly one CTA
  if (mine_u) {
    const double ul = u - before;
    if (s0 < s1 && ul >= off && ul < off + wsum[warp]) {
      double run = off;
      int tok = -1;
      for (int base = s0; base < s1 && tok < 0; base += 32) {
        const int v = base + lane;
        const float pv = v < s1 ? sP[v - lo] * sp : 0.f;
        double c = (double)pv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const double y = __shfl_up_sync(0xffffffffu, c, o);
          if (lane >= o) c += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, pv > 0.f && ul < run + c);
        if (hit) tok = base + __ffs(hit) - 1;
        run += __shfl_sync(0xffffffffu, c, 31);
      }
      for (int base = s1 - 32; tok < 0 && base > s0 - 32; base -= 32) {  // rounding: the segment's last with mass
        const int v = base + lane;
        const unsigned hit = __ballot_sync(0xffffffffu, v >= s0 && v < s1 && sP[v - lo] * sp > 0.f);
        if (hit) tok = base + 31 - __clz(hit);
      }
      if (lane == 0) *s_tok = tok;
    }
  }
  __syncthreads();
  int tok = *s_tok;
  if (mine_u && tok < 0) tok = last_with_mass(sP, sp, lo, hi, R.red);  // rounding between the warps' intervals
  return mine_u ? tok : -2;
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads) reject_tree_kernel(
    const float* logits, const float* draft, int Kd, const int32_t* tokens, medusa_tree_t tree, int V,
    float inv_tau, const float* uni, int u_stride, int32_t* accept_len, int32_t* accepted_nodes,
    int32_t* next_token, const float2* stats, int32_t* err) {
  const int crank = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;  // gridDim.x == kCluster
  const int T = tree.T, K = tree.K;
  const int lo = (int)((int64_t)crank * V / kCluster), hi = (int)((int64_t)(crank + 1) * V / kCluster);
  // this CTA's slices of the current p (once a pass has written it) and of
  // the node's q (from its first rejection on)
  extern __shared__ float s_slices[];
  float* sP = s_slices;
  float* sQ = s_slices + (V + kCluster - 1) / kCluster;
  __shared__ float2 red[kWarps];
  __shared__ float2 xf[2];
  __shared__ double xd[2];
  __shared__ int kid_by_rank[MEDUSA_MAX_S + 1];
  __shared__ int kids[MEDUSA_MAX_S + 1];
  __shared__ int s_m, s_tok;
  __shared__ double wsum[kWarps];
  ClusterRed R{red, xf, xd, 0};

  int32_t* an = accepted_nodes + (int64_t)b * (K + 1);
  if (crank == 0)
    for (int j = tid; j <= K; j += kThreads) an[j] = j == 0 ? 0 : -1;
  float sp = 0.f;     // p(v) = sP[v - lo] * sp once `mat`
  bool mat = false;   // sP holds the current node's p (after a rejection there)
  float pnext = 0.f;  // once `mat`: the unnormalised p at the next child's token
  Soft2 P{-INFINITY, 0.f};
  const float* zc = logits;
  int cur = 0, len = 0, m = 0;
  // every decision below depends only on values that are the same in every
  // CTA of the cluster (tree, tokens, uniforms, cluster-reduced scalars and
  // workspace entries read from L2), so all CTAs take the same path through
  // the same cluster barriers
  for (int guard = 0;; ++guard) {
    // children of cur in rank order (ranks of siblings are distinct, 1..MEDUSA_MAX_S)
    if (tid <= MEDUSA_MAX_S) kid_by_rank[tid] = -1;
    __syncthreads();
    for (int n = 1 + tid; n < T; n += kThreads)
      if (tree.parent[n] == cur) {
        const int r = tree.rank[n];
        if (r >= 1 && r <= MEDUSA_MAX_S) kid_by_rank[r] = n;
        else if (crank == 0) set_err(err, MEDUSA_DEVERR_NODE);
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
    // p at this node and q of the children's head, from the row statistics
    zc = logits + ((int64_t)b * T + cur) * V;
    P = row_soft(stats, (int64_t)b * (T + Kd) + cur);
    mat = false;
    if (!walk) break;
    const float* dz = draft + ((int64_t)b * Kd + (k - 1)) * V;
    const Soft2 Q = row_soft(stats, (int64_t)b * (T + Kd) + T + (k - 1));
    int acc = -1;
    for (int j = 0; j < m; ++j) {
      const int n = kids[j];
      const int x = tokens[(int64_t)b * T + n];
      if (x < 0 || x >= V) {  // an invalid draft is never accepted
        if (tid == 0 && crank == 0) set_err(err, MEDUSA_DEVERR_TOKEN);
        continue;
      }
      int xn = -1;  // the token of the next child with a valid draft
      for (int jj = j + 1; jj < m && xn < 0; ++jj) {
        const int t = tokens[(int64_t)b * T + kids[jj]];
        if (t >= 0 && t < V) xn = t;
      }
      const float u = uni[((int64_t)b * T + cur) * u_stride + j];
      const float qx = expf(__ldg(dz + x) * inv_tau - Q.m) / Q.S;
      const float px = mat ? pnext * sp : expf(__ldg(zc + x) * inv_tau - P.m) / P.S;
      if (u * qx < px) {
        acc = n;
        break;
      }
      // rejected: p <- [p - q]_+ / sum, the residual and its sum in one pass
      const float2 r = mat ? residual<true>(zc, dz, inv_tau, P, Q, sP, sQ, sp, xn, lo, hi, R)
                           : residual<false>(zc, dz, inv_tau, P, Q, sP, sQ, sp, xn, lo, hi, R);
      sp = r.x > 0.f ? 1.f / r.x : 0.f;
      pnext = r.y;
      mat = true;
    }
    if (acc < 0) break;
    ++len;
    if (tid == 0 && crank == 0) an[len] = acc;
    cur = acc;
    m = 0;
  }
  // final draw from p at the node where the walk stopped (written out first
  // unless a rejection there already did)
  if (!mat) {
    const float S = materialize(zc, inv_tau, P.m, sP, lo, hi, R);
    sp = S > 0.f ? 1.f / S : 0.f;
  }
  const float u = uni[((int64_t)b * T + cur) * u_stride + (m < u_stride ? m : u_stride - 1)];
  const int tok = draw(sP, sp, lo, hi, (double)u, wsum, &s_tok, R, crank);
  if (tid == 0) {
    if (tok != -2) next_token[b] = tok;
    if (crank == 0) accept_len[b] = len;
  }
  cluster_sync();  // no CTA leaves while another may still read its exchange slots
}

}  // namespace
}  // namespace medusa

using namespace medusa;

// Workspace: a row of V floats per sequence for the current p (and a spare
// row), then the row statistics [B][T + Kd][2] (float2) at the library's
// maximum T and K.
static size_t rows_bytes(int B, int V) { return align_up((size_t)B * 2 * V * sizeof(float), 256); }

extern "C" size_t medusa_accept_rejection_workspace_size(int B, int V) {
  if (B < 1 || V < 1) return 0;
  return rows_bytes(B, V) + align_up((size_t)B * (MEDUSA_MAX_T + MEDUSA_MAX_K) * 2 * sizeof(float2), 256);
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
  if (Kd > MEDUSA_MAX_K) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: Kd=%d above the maximum", fn, Kd);
  float2* stats = reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + rows_bytes(B, V));
  launch_kernel(reject_stats_kernel, dim3((tree->T + Kd) * 2, B), dim3(kStatThreads), 0, as_stream(stream), logits,
                draft_logits, tree->T, Kd, V, 1.f / temperature, stats);
  const size_t smem = 2 * (size_t)((V + kCluster - 1) / kCluster) * sizeof(float);  // p and q slices
  if (smem > 200 * 1024) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: V=%d above the shared-memory slices", fn, V);
  cudaFuncSetAttribute(reject_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_kernel(reject_tree_kernel, dim3(kCluster, B), dim3(kThreads), smem, as_stream(stream), logits, draft_logits, Kd,
                tokens, *tree, V, 1.f / temperature, uniforms, u_stride, accept_len, accepted_nodes, next_token,
                stats, err);
  return check_launch(fn);
}
