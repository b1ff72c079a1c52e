// Acceptance of the longest verified root path.
//
// "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
// Heads", Method 5 (section 2.3.1) and the decoding-step box (steps 4-5):
// greedy acceptance keeps a candidate while it equals the backbone's argmax at
// its parent; typical acceptance always takes the first token and keeps each
// later one while p(x) > min(eps, delta * exp(-H(p))); the step keeps the
// longest accepted prefix, ties broken by summed log-probability ("Paper vs
// code", typical acceptance).  Explainer "085 | Medusa", section 二.3: a
// rejected token ends the accepted prefix.
//
// One kernel, two 512-thread CTAs per tree row, one per half of the
// vocabulary (eight 16-byte loads in flight per thread, so a 32K-wide row
// arrives in one round of loads): argmax of the half and, for typical
// acceptance, its running softmax (max, sum, entropy term) at the given
// temperature.  The last CTA of a sequence to finish (a counter in the
// workspace) merges each row's halves into its argmax, log-sum-exp and
// entropy and makes the sequence's decisions, one thread per node: per-node
// acceptance, the accepted-prefix chain level by level, and the best node
// (select_body).  The nodes' depth, parent and token are loaded before the
// row pass, so the decisions start without waiting on global memory.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "stats.cuh"

namespace medusa {
namespace {

struct RowStat {
  int argmax;
  float lse;      // log sum_v exp(z_v), z = logits / temperature
  float entropy;  // H(p^)
  float pad;
};

// Running (max, sum e^(z-max), sum e^(z-max)(z-max)) of a softmax, mergeable.
struct Soft {
  float m, S, A;
};

__device__ __forceinline__ Soft soft_merge(Soft x, Soft y) {
  if (x.m == -INFINITY) return y;
  if (y.m == -INFINITY) return x;
  const float M = fmaxf(x.m, y.m);
  const float ex = expf(x.m - M), ey = expf(y.m - M);
  Soft r;
  r.m = M;
  r.S = x.S * ex + y.S * ey;
  r.A = ex * (x.A + (x.m - M) * x.S) + ey * (y.A + (y.m - M) * y.S);
  return r;
}

// One half row's record: its argmax (index, value) and running softmax.
struct HalfStat {
  int idx;
  float val;
  float m, S, A;
  float pad[3];
};

constexpr int kRowSplit = 2;     // CTAs per row
constexpr int kRowThreads = 512;  // >= MEDUSA_MAX_T: the last CTA gives every node a thread
constexpr int kRowLoads = 8;     // 16-byte loads in flight per thread: 64 KB per CTA, half a 32K-wide row at once
static_assert(kRowThreads >= MEDUSA_MAX_T, "one thread per node in the decisions");

// Barrier 1 over the first n threads of the block (n a multiple of 32).
MDEV void sel_sync(int n) { asm volatile("bar.sync 1, %0;\n" ::"r"(n) : "memory"); }

// A node's tree row and token, loaded before they are needed.
struct NodeIn {
  int depth, parent, token;
};
MDEV NodeIn load_node(const medusa_tree_t& tree, const int32_t* tokens, int b, int c) {
  NodeIn n{0, -1, 0};
  if (c < tree.T) {
    n.depth = __ldg(tree.depth + c);
    n.parent = __ldg(tree.parent + c);
    n.token = __ldg(tokens + (int64_t)b * tree.T + c);
  }
  return n;
}

MDEV void select_body(int b, const float* logits, NodeIn node, const medusa_tree_t& tree, int V,
                      int mode, float inv_temp, float eps, float delta, const RowStat* st, int32_t* accept_len,
                      int32_t* accepted_nodes, int32_t* next_root, int32_t* best_node, float* best_logp,
                      int32_t* err, int nthreads);

// The arguments of the row pass and of the decisions that follow it.
struct AcceptArgs {
  const float* logits;
  const int32_t* tokens;
  medusa_tree_t tree;
  int V, mode;
  float inv_temp, eps, delta;
  HalfStat* stats;  // [B][T][kRowSplit] half-row records
  int* counters;   // [B] rows finished per sequence; zero on entry, left zero
  int32_t *accept_len, *accepted_nodes, *next_root, *best_node;
  float* best_logp;
  int32_t* err;
};

template <bool TYPICAL>
__global__ void __launch_bounds__(kRowThreads) accept_rowstat_kernel(const __grid_constant__ AcceptArgs a) {
  const int T = a.tree.T, V = a.V;
  const float inv_temp = a.inv_temp;
  const int p = blockIdx.x / kRowSplit, half = blockIdx.x % kRowSplit, b = blockIdx.y;
  // the node this thread would decide for, were this CTA the sequence's last
  const NodeIn node = load_node(a.tree, a.tokens, b, threadIdx.x);
  const float* z = a.logits + ((int64_t)b * T + p) * V;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  Soft sf{-INFINITY, 0.f, 0.f};
  auto consume = [&](float x, int v) {
    if (ranks_before(x, v, bv, bi)) { bv = x; bi = v; }
    if (TYPICAL) {
      const float y = x * inv_temp;
      if (y > sf.m) {
        const float e = expf(sf.m - y);  // 0 when the old max is -inf
        sf.A = sf.m == -INFINITY ? 0.f : e * (sf.A + (sf.m - y) * sf.S);
        sf.S = sf.S * e + 1.f;
        sf.m = y;
      } else {
        const float e = expf(y - sf.m);
        sf.S += e;
        sf.A += e * (y - sf.m);
      }
    }
  };
  if ((V & 3) == 0) {
    const float4* z4 = reinterpret_cast<const float4*>(z);
    const int n4 = V >> 2, lo = (int)((int64_t)n4 * half / kRowSplit), hi = (int)((int64_t)n4 * (half + 1) / kRowSplit);
    for (int i = lo + threadIdx.x; i < hi && !TYPICAL; i += kRowLoads * kRowThreads) {  // greedy: argmax only
      float4 r[kRowLoads];
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) {
        const int ii = i + u * kRowThreads;
        if (ii < hi) r[u] = __ldg(z4 + ii);
      }
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) {
        const int ii = i + u * kRowThreads;
        if (ii < hi) {
          consume(r[u].x, 4 * ii);
          consume(r[u].y, 4 * ii + 1);
          consume(r[u].z, 4 * ii + 2);
          consume(r[u].w, 4 * ii + 3);
        }
      }
    }
    for (int i = lo + threadIdx.x; i < hi && TYPICAL; i += kRowLoads * kRowThreads) {
      float4 r[kRowLoads];
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) {
        const int ii = i + u * kRowThreads;
        r[u] = ii < hi ? __ldg(z4 + ii) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
      // the round's values are all in registers: argmax, then (typical) the
      // round's max and its sums as independent exponentials, merged into the
      // running softmax once per round instead of once per value
      float rm = -INFINITY;
#pragma unroll
      for (int u = 0; u < kRowLoads; ++u) {
        const int ii = i + u * kRowThreads;
        const float e[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (ii < hi && ranks_before(e[q], 4 * ii + q, bv, bi)) { bv = e[q]; bi = 4 * ii + q; }
          rm = fmaxf(rm, e[q]);  // padding values are -inf
        }
      }
      if (rm > -INFINITY) {
        const float my = rm * inv_temp;  // the round's max of y = z / temperature
        float rS = 0.f, rA = 0.f;
#pragma unroll
        for (int u = 0; u < kRowLoads; ++u) {
          const float e[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float d = e[q] * inv_temp - my;  // -inf for a padding value: exp 0, and 0 * -inf skipped
            const float x = expf(d);
            rS += x;
            rA += x > 0.f ? x * d : 0.f;
          }
        }
        sf = soft_merge(sf, Soft{my, rS, rA});
      }
    }
  } else {
    const int lo = (int)((int64_t)V * half / kRowSplit), hi = (int)((int64_t)V * (half + 1) / kRowSplit);
    for (int v = lo + threadIdx.x; v < hi; v += kRowThreads) consume(z[v], v);
  }
  constexpr int NW = kRowThreads / 32;
  __shared__ float sv[NW], sS[NW], sA[NW], sm[NW];
  __shared__ int si[NW];
  warp_argmax(bv, bi);
  if (TYPICAL) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Soft y{__shfl_xor_sync(0xffffffffu, sf.m, o), __shfl_xor_sync(0xffffffffu, sf.S, o),
             __shfl_xor_sync(0xffffffffu, sf.A, o)};
      sf = soft_merge(sf, y);
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { sv[warp] = bv; si[warp] = bi; sm[warp] = sf.m; sS[warp] = sf.S; sA[warp] = sf.A; }
  __syncthreads();
  if (warp == 0) {
    bv = lane < NW ? sv[lane] : -INFINITY;
    bi = lane < NW ? si[lane] : 0x7fffffff;
    warp_argmax(bv, bi);
    if (TYPICAL) {
      sf = lane < NW ? Soft{sm[lane], sS[lane], sA[lane]} : Soft{-INFINITY, 0.f, 0.f};
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        Soft y{__shfl_xor_sync(0xffffffffu, sf.m, o), __shfl_xor_sync(0xffffffffu, sf.S, o),
               __shfl_xor_sync(0xffffffffu, sf.A, o)};
        sf = soft_merge(sf, y);
      }
    }
    if (lane == 0) {
      float4* rec = reinterpret_cast<float4*>(a.stats + ((int64_t)b * T + p) * kRowSplit + half);
      rec[0] = make_float4(__int_as_float(bi), bv, sf.m, sf.S);
      rec[1] = make_float4(sf.A, 0.f, 0.f, 0.f);
    }
  }
  // the last CTA of the sequence to finish makes its decisions
  __shared__ bool s_last;
  __shared__ RowStat rs[MEDUSA_MAX_T];
  __syncthreads();
  if (threadIdx.x == 0) s_last = arrive_acq_rel(a.counters + b) == kRowSplit * T - 1;
  __syncthreads();
  if (!s_last) return;
  // one thread per node: the other warps leave, so the decisions' barriers
  // wait for ceil(T / 32) warps only
  const int nthr = (T + 31) & ~31;
  if ((int)threadIdx.x >= nthr) return;
  const int c = threadIdx.x;
  if (c < T) {
    // the row's halves: argmax (value, then lower index), softmax merged
    const float4* rec = reinterpret_cast<const float4*>(a.stats + ((int64_t)b * T + c) * kRowSplit);
    int ri = 0x7fffffff;
    float rv = -INFINITY;
    Soft rsf{-INFINITY, 0.f, 0.f};
#pragma unroll
    for (int h = 0; h < kRowSplit; ++h) {
      const float4 x0 = __ldcg(rec + 2 * h), x1 = __ldcg(rec + 2 * h + 1);
      const int xi = __float_as_int(x0.x);
      if (ranks_before(x0.y, xi, rv, ri)) { rv = x0.y; ri = xi; }
      if (TYPICAL) rsf = soft_merge(rsf, Soft{x0.z, x0.w, x1.x});
    }
    // H = log S - A / S  (p^_v = e^(z_v - m) / S)
    rs[c] = RowStat{ri, TYPICAL ? rsf.m + logf(rsf.S) : 0.f, TYPICAL ? logf(rsf.S) - rsf.A / rsf.S : 0.f, 0.f};
  }
  sel_sync(nthr);
  select_body(b, a.logits, node, a.tree, V, a.mode, inv_temp, a.eps, a.delta, rs, a.accept_len,
              a.accepted_nodes, a.next_root, a.best_node, a.best_logp, a.err, nthr);
  if (threadIdx.x == 0) a.counters[b] = 0;  // every row of the sequence has arrived
}

// Sequence b's decisions from its rows' statistics `st` ([T], global or
// shared memory) and each thread's node (loaded by the caller); one thread
// per node: threads 0 .. nthreads-1 of the block
// take part (nthreads >= T, a multiple of 32; the block's other warps may
// have exited), synchronised on barrier 1.
MDEV void select_body(int b, const float* logits, NodeIn node, const medusa_tree_t& tree, int V,
                      int mode, float inv_temp, float eps, float delta, const RowStat* st, int32_t* accept_len,
                      int32_t* accepted_nodes, int32_t* next_root, int32_t* best_node, float* best_logp,
                      int32_t* err, int nthreads) {
  const int c = threadIdx.x;
  const int T = tree.T;
  __shared__ uint8_t ok[MEDUSA_MAX_T];
  __shared__ float lp[MEDUSA_MAX_T];
  __shared__ int dep[MEDUSA_MAX_T];
  __shared__ int par[MEDUSA_MAX_T];
  __shared__ int amax[MEDUSA_MAX_T];  // each row's argmax (the next root if the row is the best node)
  // key of the best node: depth (high bits) then -node index; typical also
  // compares the summed log-probability, so it is resolved in a second pass
  __shared__ int red_key[32];
  __shared__ float red_lp[32];
  int depth_c = 0, parent_c = -1;
  bool pass = false;
  float lpc = 0.f;
  if (c < T) {
    depth_c = node.depth;
    parent_c = node.parent;
    amax[c] = st[c].argmax;
    if (c == 0) {
      pass = true;
      depth_c = 0;
    } else if (parent_c < 0 || parent_c >= c || depth_c < 1 || depth_c > tree.K) {
      // malformed tree row: never accepted, never followed
      set_err(err, MEDUSA_DEVERR_NODE);
      parent_c = 0;
      depth_c = 0;
    } else {
      const int tok = node.token;
      const RowStat rp = st[parent_c];
      if (mode == 0) {
        pass = tok == rp.argmax;
      } else if (tok < 0 || tok >= V) {
        set_err(err, MEDUSA_DEVERR_TOKEN);
      } else {
        const float zt = logits[((int64_t)b * T + parent_c) * V + tok] * inv_temp;
        lpc = zt - rp.lse;
        const float thr = fminf(eps, delta * expf(-rp.entropy));
        pass = expf(lpc) > thr;
      }
    }
    dep[c] = depth_c;
    par[c] = parent_c;
    ok[c] = c == 0 ? 1 : 0;
    lp[c] = 0.f;
  }
  sel_sync(nthreads);
  // the accepted-prefix chain, one depth level at a time
  for (int k = 1; k <= tree.K; ++k) {
    if (c < T && depth_c == k) {
      ok[c] = (pass && ok[parent_c]) ? 1 : 0;
      lp[c] = lp[parent_c] + lpc;
    }
    sel_sync(nthreads);
  }
  // best node: max depth; typical: then max log-prob; then min index
  const int warp = c >> 5, lane = c & 31, nw = (nthreads + 31) >> 5;
  int key = (c < T && ok[c]) ? (depth_c << 16) | (0xffff - c) : -1;
  float mylp = (c < T && ok[c]) ? lp[c] : -INFINITY;
  // pass 1: deepest accepted depth
  int kmax = key;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  if (lane == 0) red_key[warp] = kmax;
  sel_sync(nthreads);
  if (c == 0) {
    int m = -1;
    for (int w = 0; w < nw; ++w) m = max(m, red_key[w]);
    red_key[0] = m;
  }
  sel_sync(nthreads);
  const int best_depth = red_key[0] >> 16;
  sel_sync(nthreads);
  // pass 2 among nodes at that depth: (log-prob for typical, then low index)
  float cand_lp = (key >= 0 && depth_c == best_depth) ? (mode == 1 ? mylp : 0.f) : -INFINITY;
  int cand_i = (key >= 0 && depth_c == best_depth) ? c : 0x7fffffff;
  warp_argmax(cand_lp, cand_i);
  if (lane == 0) { red_lp[warp] = cand_lp; red_key[warp] = cand_i; }
  sel_sync(nthreads);
  if (c == 0) {
    float bl = -INFINITY;
    int bi = 0x7fffffff;
    for (int w = 0; w < nw; ++w)
      if (ranks_before(red_lp[w], red_key[w], bl, bi)) { bl = red_lp[w]; bi = red_key[w]; }
    if (bi < 0 || bi >= T) bi = 0;  // the root is always accepted
    const int K = tree.K;
    int32_t* an = accepted_nodes + (int64_t)b * (K + 1);
    for (int j = 0; j <= K; ++j) an[j] = -1;
    // walk parents from the best node: one step per level, depth dep[bi] <= K
    int n = bi;
    for (int j = dep[bi]; j >= 0 && n >= 0 && n < T; --j) {
      an[j] = n;
      n = j > 0 ? par[n] : -1;
    }
    accept_len[b] = dep[bi];
    next_root[b] = amax[bi];
    best_node[b] = bi;
    if (best_logp) best_logp[b] = mode == 1 ? lp[bi] : 0.f;
  }
}

// Acceptance from the LM head's fused statistics (medusa_lm_head_verify_stats):
// the rows' per-group records are merged (a fixed share of the groups per
// thread, then the shares in order), then the same decisions as above.
constexpr int kStatThreads = 1024;

__global__ void __launch_bounds__(kStatThreads) accept_stats_kernel(
    const float4* part, int groups, int rows_total, const float* logits, const int32_t* tokens,
    medusa_tree_t tree, int V, int mode, float inv_temp, float eps, float delta, int32_t* accept_len,
    int32_t* accepted_nodes, int32_t* next_root, int32_t* best_node, float* best_logp, int32_t* err) {
  const int b = blockIdx.x, tid = threadIdx.x, T = tree.T;
  const NodeIn node = load_node(tree, tokens, b, tid);
  __shared__ RowStat rs[MEDUSA_MAX_T];
  __shared__ float4 share[kStatThreads];
  const int P = max(1, kStatThreads / T);  // threads per row
  const int r = tid / P, sh = tid % P;
  StatRec m = stat_empty();
  if (r < T)
    for (int g = sh; g < groups; g += P) {
      const float4 x = __ldg(part + (int64_t)g * rows_total + (int64_t)b * T + r);
      m = mode == 1 ? stat_merge<true>(m, stat_load(x), inv_temp) : stat_merge<false>(m, stat_load(x), inv_temp);
    }
  share[tid] = stat_store(m);
  __syncthreads();
  if (r < T && sh == 0) {
    StatRec a = stat_empty();
    for (int q = 0; q < P; ++q)
      a = mode == 1 ? stat_merge<true>(a, stat_load(share[tid + q]), inv_temp)
                    : stat_merge<false>(a, stat_load(share[tid + q]), inv_temp);
    RowStat o;
    o.argmax = a.i;
    // H = log S - A / S  (p^_v = e^(y_v - m) / S, m = max y)
    o.lse = mode == 1 ? a.v * inv_temp + logf(a.S) : 0.f;
    o.entropy = mode == 1 ? logf(a.S) - a.A / a.S : 0.f;
    o.pad = 0.f;
    rs[r] = o;
  }
  __syncthreads();
  select_body(b, logits, node, tree, V, mode, inv_temp, eps, delta, rs, accept_len, accepted_nodes, next_root,
              best_node, best_logp, err, blockDim.x);
}

// Workspace: per-sequence counters (256 bytes, at a fixed place so that
// calls of any size find them zero), then two half-row records of 32 bytes
// per (sequence, tree row).
constexpr size_t kCounterBytes = 256;
static_assert(MEDUSA_MAX_B * sizeof(int) <= kCounterBytes, "counters");

// Scratch of medusa_accept_noalloc: the counters and the half-row records
// of every (sequence, tree row) at the library's maximum sizes, 256 bytes +
// 16 x 512 x 64 bytes = 512 KiB per device, zero when the library loads.
constexpr int kNoAllocRows = MEDUSA_ACCEPT_NOALLOC_MAX_ROWS;
constexpr size_t kNoAllocBytes = kCounterBytes + sizeof(HalfStat) * kRowSplit * (size_t)kNoAllocRows;
static __device__ __align__(256) uint8_t g_accept_scratch[kNoAllocBytes];

// The scratch's device address, cached per device together with the unique
// id of the context it was looked up in.  A context created after
// cudaDeviceReset loads the module again, and the array may move; its id
// differs (context ids are never reused in a process), so the address is
// looked up again.
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};
unsigned long long g_noalloc_ctx[kMaxDevices] = {};

// cuCtxGetCurrent and cuCtxGetId through the runtime's driver entry points
// (the library does not link libcuda).
using CtxGetCurrentFn = int (*)(void**);
using CtxGetIdFn = int (*)(void*, unsigned long long*);

int current_context_id(const char* fn, unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return fail(MEDUSA_ERR_CUDA, "%s: cuCtxGetCurrent / cuCtxGetId unavailable", fn);
  void* ctx = nullptr;
  *id = 0;
  if (get_current(&ctx) != 0) return fail(MEDUSA_ERR_CUDA, "%s: cuCtxGetCurrent failed", fn);
  if (ctx && get_id(ctx, id) != 0) return fail(MEDUSA_ERR_CUDA, "%s: cuCtxGetId failed", fn);
  return MEDUSA_OK;
}

// Device address of g_accept_scratch in the current device's context.  The
// host-side symbol is only a stand-in, so the address is looked up with that
// device current (cudaGetSymbolAddress) and cached for the context.
int noalloc_scratch(const char* fn, void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "%s: cudaGetDevice: %s", fn, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(MEDUSA_ERR_UNSUPPORTED, "%s: device ordinal %d outside 0..%d", fn, dev, kMaxDevices - 1);
  unsigned long long id = 0;
  if (int rc = current_context_id(fn, &id)) return rc;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev] || id == 0 || g_noalloc_ctx[dev] != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_accept_scratch);
    if (e != cudaSuccess || !p)
      return fail(MEDUSA_ERR_CUDA, "%s: cudaGetSymbolAddress: %s", fn, cudaGetErrorString(e));
    if (id == 0) {  // no context was current: the lookup made the primary context current
      if (int rc = current_context_id(fn, &id)) return rc;
      if (id == 0) return fail(MEDUSA_ERR_CUDA, "%s: no current context after the symbol lookup", fn);
    }
    g_noalloc_addr[dev] = p;
    g_noalloc_ctx[dev] = id;
  }
  *out = g_noalloc_addr[dev];
  return MEDUSA_OK;
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_accept_workspace_size(int B, int T) {
  if (B < 1 || T < 1) return 0;
  return kCounterBytes + align_up((size_t)B * T * kRowSplit * sizeof(HalfStat), 256);
}

extern "C" int medusa_accept(const float* logits, const int32_t* tokens, const medusa_tree_t* tree,
                             int B, int V, int mode, float temperature, float eps, float delta,
                             int32_t* accept_len, int32_t* accepted_nodes, int32_t* next_root,
                             int32_t* best_node, float* best_logp, void* workspace,
                             size_t workspace_bytes, int32_t* err, void* stream) {
  const char* fn = "medusa_accept";
  if (int rc = check_tree(tree, fn)) return rc;
  if (!logits || !tokens || !accept_len || !accepted_nodes || !next_root || !best_node)
    return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (B < 1 || B > MEDUSA_MAX_B || V < 1) return fail(MEDUSA_ERR_INVALID, "%s: B=%d V=%d", fn, B, V);
  if (mode != 0 && mode != 1) return fail(MEDUSA_ERR_INVALID, "%s: mode %d", fn, mode);
  if (mode == 1 && !(temperature > 0.f)) return fail(MEDUSA_ERR_INVALID, "%s: temperature must be > 0", fn);
  const size_t need = medusa_accept_workspace_size(B, tree->T);
  if (!workspace || workspace_bytes < need)
    return fail(MEDUSA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) % 16)
    return fail(MEDUSA_ERR_INVALID, "%s: workspace not 16-byte aligned", fn);
  cudaStream_t s = as_stream(stream);
  AcceptArgs a{};
  a.logits = logits; a.tokens = tokens; a.tree = *tree; a.V = V; a.mode = mode;
  a.inv_temp = mode == 1 ? 1.f / temperature : 1.f;
  a.eps = eps; a.delta = delta;
  a.counters = static_cast<int*>(workspace);
  a.stats = reinterpret_cast<HalfStat*>(static_cast<uint8_t*>(workspace) + kCounterBytes);
  a.accept_len = accept_len; a.accepted_nodes = accepted_nodes; a.next_root = next_root;
  a.best_node = best_node; a.best_logp = best_logp; a.err = err;
  dim3 g(tree->T * kRowSplit, B);
  if (mode == 1)
    launch_kernel(accept_rowstat_kernel<true>, g, dim3(kRowThreads), 0, s, a);
  else
    launch_kernel(accept_rowstat_kernel<false>, g, dim3(kRowThreads), 0, s, a);
  return check_launch(fn);
}

// Allocation-free acceptance for callers that cannot allocate device memory:
// the same kernels as medusa_accept, with the file-scope scratch above in
// place of a caller workspace.  It allocates nothing; the first call on a
// device looks up the scratch address.
extern "C" int medusa_accept_noalloc(const float* logits, const int32_t* tokens, const medusa_tree_t* tree,
                                     int B, int V, int mode, float temperature, float eps, float delta,
                                     int32_t* accept_len, int32_t* accepted_nodes, int32_t* next_root,
                                     int32_t* best_node, float* best_logp, int32_t* err, void* stream) {
  const char* fn = "medusa_accept_noalloc";
  if (int rc = check_tree(tree, fn)) return rc;
  if (B < 1) return fail(MEDUSA_ERR_INVALID, "%s: B=%d", fn, B);
  if ((long)B * tree->T > kNoAllocRows)
    return fail(MEDUSA_ERR_CAPACITY, "%s: B*T = %ld tree rows exceed the static scratch of %d rows", fn,
                (long)B * tree->T, kNoAllocRows);
  void* scratch = nullptr;
  if (int rc = noalloc_scratch(fn, &scratch)) return rc;
  return medusa_accept(logits, tokens, tree, B, V, mode, temperature, eps, delta, accept_len, accepted_nodes,
                       next_root, best_node, best_logp, scratch, kNoAllocBytes, err, stream);
}

extern "C" int medusa_accept_stats(const void* stats, int groups, const float* logits, const int32_t* tokens,
                                   const medusa_tree_t* tree, int B, int V, int mode, float temperature, float eps,
                                   float delta, int32_t* accept_len, int32_t* accepted_nodes, int32_t* next_root,
                                   int32_t* best_node, float* best_logp, int32_t* err, void* stream) {
  const char* fn = "medusa_accept_stats";
  if (int rc = check_tree(tree, fn)) return rc;
  if (!stats || !tokens || !accept_len || !accepted_nodes || !next_root || !best_node)
    return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (B < 1 || B > MEDUSA_MAX_B || V < 1 || groups < 1)
    return fail(MEDUSA_ERR_INVALID, "%s: B=%d V=%d groups=%d", fn, B, V, groups);
  if (mode != 0 && mode != 1) return fail(MEDUSA_ERR_INVALID, "%s: mode %d", fn, mode);
  if (mode == 1 && !(temperature > 0.f)) return fail(MEDUSA_ERR_INVALID, "%s: temperature must be > 0", fn);
  if (mode == 1 && !logits) return fail(MEDUSA_ERR_INVALID, "%s: typical acceptance needs the logits", fn);
  if (reinterpret_cast<uintptr_t>(stats) % 16) return fail(MEDUSA_ERR_INVALID, "%s: stats not 16-byte aligned", fn);
  const float inv_temp = mode == 1 ? 1.f / temperature : 1.f;
  launch_kernel(accept_stats_kernel, dim3(B), dim3(kStatThreads), 0, as_stream(stream),
                static_cast<const float4*>(stats), groups, B * tree->T, logits, tokens, *tree, V, mode, inv_temp, eps,
                delta, accept_len, accepted_nodes, next_root, best_node, best_logp, err);
  return check_launch(fn);
}
