// Medusa heads and top-s selection.
//
// "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
// Heads", Method 1 (section 2.1.1): head k maps the last hidden state h to
// p^(k) = softmax(W2^(k) (SiLU(W1^(k) h) + h)), W1 in R^{d x d},
// W2 in R^{d x V}; "Paper vs code": the code's residual block has a bias
// (optional here).  Method 2: the top-s_k tokens of head k form level k of
// the candidate tree (softmax is monotone, so top-s of the logits is used).
//
// At batch size 1 both projections are matrix-vector products over weights
// read once per step (about 80% of a 7B-shaped step's bytes), so they are
// HBM-bound GEMVs: one warp per output row, 16-byte streaming loads with
// eight loads in flight per lane, the input vector re-read from L1.
//   gemv<W1>  u[b][k] = dtype(SiLU(W1_k h_b + b1_k) + h_b)   (scratch)
//   gemv<W2>  head_logits[b][k] = W2_k u[b][k]              (fp32)
//   topk      per (head, sequence) in chunks of ~1024 logits, one CTA each:
//             per-lane sorted lists merged warp by warp (value descending,
//             index ascending); the last chunk to finish merges the chunks
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace medusa {
namespace {

struct GemvArgs {
  const void* w;        // [K][rows][d]
  int rows, d;
  int nused;
  int heads[MEDUSA_MAX_K];  // ids of the heads with s_k > 0
  const void* hidden;   // [B][T][d]
  const int32_t* last_node;
  int T, B, K;
  const void* b1;       // [K][d] or null
  void* u;              // [B][K][d] element type
  float* logits;        // [B][K][V]
  int* counters;        // top-s arrival counters, zeroed by the W1 pass
  int ncounters;
  int32_t* err;
};

template <typename TE> struct Vec;
template <> struct Vec<uint16_t> {
  static constexpr int N = 8;
  static MDEV void unpack(const uint4& v, float* f) { unpack8_bf16(v, f); }
};
template <> struct Vec<float> {
  static constexpr int N = 4;
  static MDEV void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
};

constexpr int UNROLL = 8;

template <typename TE, int NB, bool W1>
__global__ void __launch_bounds__(256) heads_gemv_kernel(GemvArgs a) {
  constexpr int EPV = Vec<TE>::N;
  const int lane = threadIdx.x & 31;
  const int64_t warp_g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int nvec = a.d / EPV;
  const int64_t total = (int64_t)a.nused * a.rows;
  const TE* W = static_cast<const TE*>(a.w);
  __shared__ int head_id[MEDUSA_MAX_K];
  if (threadIdx.x < MEDUSA_MAX_K) head_id[threadIdx.x] = a.heads[threadIdx.x];
  __syncthreads();
  if (W1 && blockIdx.x == 0)
    for (int i = threadIdx.x; i < a.ncounters; i += blockDim.x) a.counters[i] = 0;

  // input vectors of this call, one per sequence (W1: hidden[b][last_node]);
  // an out-of-range node reads row 0 and raises the error bit
  const TE* xin[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if (W1) {
      int n = b < a.B ? a.last_node[b] : 0;
      if (n < 0 || n >= a.T) {
        if (lane == 0 && warp_g == 0) set_err(a.err, MEDUSA_DEVERR_NODE);
        n = 0;
      }
      xin[b] = static_cast<const TE*>(a.hidden) + ((int64_t)(b < a.B ? b : 0) * a.T + n) * a.d;
    } else {
      xin[b] = nullptr;
    }
  }

  for (int64_t g = warp_g; g < total; g += nwarps) {
    const int slot = (int)(g / a.rows);
    const int j = (int)(g % a.rows);
    const int k = head_id[slot];
    const TE* wrow = W + ((int64_t)k * a.rows + j) * a.d;
    const TE* x[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b)
      x[b] = W1 ? xin[b] : static_cast<const TE*>(a.u) + ((int64_t)(b < a.B ? b : 0) * a.K + k) * a.d;
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
    for (int c0 = lane; c0 < nvec; c0 += 32 * UNROLL) {
      uint4 wv[UNROLL];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int c = c0 + u * 32;
        if (c < nvec) wv[u] = ldg_stream(wrow + (int64_t)c * EPV);
      }
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int c = c0 + u * 32;
        if (c < nvec) {
          float wf[EPV];
          Vec<TE>::unpack(wv[u], wf);
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            if (b < a.B) {
              float xf[EPV];
              Vec<TE>::unpack(ldg_v4(x[b] + (int64_t)c * EPV), xf);
#pragma unroll
              for (int e = 0; e < EPV; ++e) acc[b] = fmaf(wf[e], xf[e], acc[b]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = warp_sum(acc[b]);
    if (lane < NB && lane < a.B) {
      float y = 0.f;
#pragma unroll
      for (int b = 0; b < NB; ++b)
        if (b == lane) y = acc[b];
      const int b = lane;
      if (W1) {
        if (a.b1) y += to_f32(static_cast<const TE*>(a.b1)[(int64_t)k * a.d + j]);
        const float silu = y / (1.f + expf(-y));
        const float u = silu + to_f32(xin[b][j]);
        static_cast<TE*>(a.u)[((int64_t)b * a.K + k) * a.d + j] = from_f32<TE>(u);
      } else {
        a.logits[((int64_t)b * a.K + k) * a.rows + j] = y;
      }
    }
  }
}

// ---------------------------------------------------------------- top-s --

template <int S>
struct TopList {
  float v[S];
  int i[S];
  MDEV void init() {
#pragma unroll
    for (int t = 0; t < S; ++t) { v[t] = -INFINITY; i[t] = 0x7fffffff; }
  }
  MDEV void insert(float x, int xi) {
    if (!ranks_before(x, xi, v[S - 1], i[S - 1])) return;
    v[S - 1] = x;
    i[S - 1] = xi;
#pragma unroll
    for (int t = S - 1; t > 0; --t) {
      if (ranks_before(v[t], i[t], v[t - 1], i[t - 1])) {
        const float tv = v[t]; v[t] = v[t - 1]; v[t - 1] = tv;
        const int ti = i[t]; i[t] = i[t - 1]; i[t - 1] = ti;
      }
    }
  }
  MDEV void pop() {
#pragma unroll
    for (int t = 0; t + 1 < S; ++t) { v[t] = v[t + 1]; i[t] = i[t + 1]; }
    v[S - 1] = -INFINITY;
    i[S - 1] = 0x7fffffff;
  }
  // Warp-wide: the S best of all lanes' lists, in order, to out_v/out_i
  // (valid on every lane).  Consumes the lists.
  MDEV void warp_select(float* out_v, int* out_i) {
#pragma unroll
    for (int r = 0; r < S; ++r) {
      float bv = v[0];
      int bi = i[0];
      warp_argmax(bv, bi);
      if (i[0] == bi && v[0] == bv) pop();
      out_v[r] = bv;
      out_i[r] = bi;
    }
  }
};

struct HeadTable {
  int32_t h[MEDUSA_MAX_K];  // ids of the used heads
  int32_t s[MEDUSA_MAX_K];  // their s_k
};

struct TopkArgs {
  const float* logits;  // [B][K][V]
  int K, V, s_max, nchunk;
  HeadTable tab;
  float* cand_v;  // [nused][B][nchunk][S] candidate values (scratch)
  int* cand_i;    // same layout, indices
  int* counters;  // [nused][B] arrivals, zero on entry
  int32_t* topk;  // [B][K][s_max]
};

// Block-wide: the S best of all threads' lists, valid in warp 0.  Consumes
// the lists; `wv`/`wi` are [32][S] shared staging.
template <int S>
MDEV void block_select(TopList<S>& L, float (*wv)[S], int (*wi)[S], float* ov, int* oi) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  L.warp_select(ov, oi);
  if (lane == 0) {
#pragma unroll
    for (int t = 0; t < S; ++t) { wv[warp][t] = ov[t]; wi[warp][t] = oi[t]; }
  }
  __syncthreads();
  if (warp == 0) {
    TopList<S> M;
#pragma unroll
    for (int t = 0; t < S; ++t) {
      M.v[t] = lane < nw ? wv[lane][t] : -INFINITY;
      M.i[t] = lane < nw ? wi[lane][t] : 0x7fffffff;
    }
    M.warp_select(ov, oi);
  }
}

// Grid (nchunk, nused, B).  Each CTA selects the top S of one contiguous
// chunk of a head's logits; the last CTA of the head to finish merges the
// nchunk candidate lists and writes the head's top s.
template <int S>
__global__ void __launch_bounds__(256) topk_kernel(const __grid_constant__ TopkArgs a) {
  const int chunk = blockIdx.x, slot = blockIdx.y, b = blockIdx.z;
  const int k = a.tab.h[slot], s = a.tab.s[slot];
  const int nused = gridDim.y;
  const float* z = a.logits + ((int64_t)b * a.K + k) * a.V;
  const int per = (a.V + a.nchunk - 1) / a.nchunk;
  const int v0 = chunk * per, v1 = min(a.V, v0 + per);
  __shared__ float wv[32][S];
  __shared__ int wi[32][S];
  __shared__ bool last;
  TopList<S> L;
  L.init();
  for (int base = v0 + threadIdx.x; base < v1; base += 4 * blockDim.x) {
    float x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = base + u * blockDim.x;
      x[u] = v < v1 ? z[v] : -INFINITY;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = base + u * blockDim.x;
      if (v < v1) L.insert(x[u], v);
    }
  }
  float ov[S];
  int oi[S];
  block_select<S>(L, wv, wi, ov, oi);
  const int64_t cbase = (((int64_t)slot * gridDim.z + b) * a.nchunk + chunk) * S;
  if (threadIdx.x < 32 && threadIdx.x == 0) {
#pragma unroll
    for (int t = 0; t < S; ++t) { a.cand_v[cbase + t] = ov[t]; a.cand_i[cbase + t] = oi[t]; }
  }
  // the last chunk of this (head, sequence) to arrive merges all chunks
  if (threadIdx.x == 0) {
    __threadfence();
    const int prev = atomicAdd(a.counters + slot * gridDim.z + b, 1);
    last = prev == a.nchunk - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int64_t hbase = ((int64_t)slot * gridDim.z + b) * a.nchunk * S;
  L.init();
  for (int e = threadIdx.x; e < a.nchunk * S; e += blockDim.x)
    L.insert(__ldcg(a.cand_v + hbase + e), __ldcg(a.cand_i + hbase + e));
  __syncthreads();
  block_select<S>(L, wv, wi, ov, oi);
  if (threadIdx.x < 32) {
    int32_t* out = a.topk + ((int64_t)b * a.K + k) * a.s_max;
    for (int t = threadIdx.x; t < a.s_max; t += 32) {
      int idx = -1;
#pragma unroll
      for (int q = 0; q < S; ++q)
        if (q == t) idx = oi[q];
      out[t] = (t < s && idx >= 0 && idx < a.V) ? idx : -1;
    }
  }
  if (threadIdx.x == 0) a.counters[slot * gridDim.z + b] = 0;  // ready for the next call
  (void)nused;
}

int topk_chunks(int V) { return std::max(1, std::min(64, (V + 1023) / 1024)); }

template <typename TE, int NB>
void launch_gemv(const GemvArgs& a, bool w1, cudaStream_t s) {
  const int blocks = std::max(1, std::min(sm_count() * 4, (int)((int64_t(a.nused) * a.rows + 7) / 8)));
  if (w1)
    launch_kernel(heads_gemv_kernel<TE, NB, true>, dim3(blocks), dim3(256), 0, s, a);
  else
    launch_kernel(heads_gemv_kernel<TE, NB, false>, dim3(blocks), dim3(256), 0, s, a);
}

template <typename TE>
void launch_gemv_b(const GemvArgs& a, bool w1, cudaStream_t s) {
  if (a.B == 1) launch_gemv<TE, 1>(a, w1, s);
  else if (a.B <= 4) launch_gemv<TE, 4>(a, w1, s);
  else launch_gemv<TE, MEDUSA_MAX_B>(a, w1, s);
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_heads_topk_workspace_size(int B, int K, int d, int V, int s_max) {
  (void)V; (void)s_max;
  if (B < 1 || K < 1 || d < 1) return 0;
  // u [B][K][d] (fp32 size covers both element types), top-s candidates and counters
  const size_t u = align_up((size_t)B * K * d * sizeof(float), 256);
  const size_t cand = align_up((size_t)K * B * topk_chunks(V) * MEDUSA_MAX_S * 4, 256);
  return u + 2 * cand + align_up((size_t)K * B * sizeof(int), 256);
}

extern "C" int medusa_heads_topk(const void* hidden, const int32_t* last_node, int T, const void* w1,
                                 const void* b1, const void* w2, const int32_t* s, int K, int B, int d,
                                 int V, medusa_dtype dtype, float* head_logits, int32_t* topk, int s_max,
                                 void* workspace, size_t workspace_bytes, int32_t* err, void* stream) {
  const char* fn = "medusa_heads_topk";
  if (!hidden || !last_node || !w1 || !w2 || !s || !head_logits || !topk)
    return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (T < 1 || K < 1 || B < 1 || d < 1 || V < 1 || s_max < 1)
    return fail(MEDUSA_ERR_INVALID, "%s: T=%d K=%d B=%d d=%d V=%d s_max=%d", fn, T, K, B, d, V, s_max);
  if (K > MEDUSA_MAX_K || B > MEDUSA_MAX_B || s_max > MEDUSA_MAX_S)
    return fail(MEDUSA_ERR_UNSUPPORTED, "%s: K=%d B=%d s_max=%d above the maximum", fn, K, B, s_max);
  if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: dtype", fn);
  const int epv = dtype == MEDUSA_BF16 ? 8 : 4;
  if (d % epv) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: d=%d not a multiple of %d", fn, d, epv);
  if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(w1) |
       reinterpret_cast<uintptr_t>(w2)) % 16)
    return fail(MEDUSA_ERR_INVALID, "%s: hidden / w1 / w2 not 16-byte aligned", fn);
  const size_t need = medusa_heads_topk_workspace_size(B, K, d, V, s_max);
  if (!workspace || workspace_bytes < need)
    return fail(MEDUSA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, workspace_bytes, need);
  GemvArgs a{};
  a.nused = 0;
  int smax_used = 0;
  for (int k = 0; k < K; ++k) {
    if (s[k] < 0 || s[k] > s_max || s[k] > V)
      return fail(MEDUSA_ERR_INVALID, "%s: s[%d]=%d outside [0, min(s_max, V)]", fn, k, s[k]);
    if (s[k] > 0) { a.heads[a.nused++] = k; smax_used = std::max(smax_used, (int)s[k]); }
  }
  if (a.nused == 0) return MEDUSA_OK;
  cudaStream_t st = as_stream(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t u_bytes = align_up((size_t)B * K * d * sizeof(float), 256);
  const int nchunk = topk_chunks(V);
  const size_t cand_bytes = align_up((size_t)K * B * nchunk * MEDUSA_MAX_S * 4, 256);
  a.counters = reinterpret_cast<int*>(ws + u_bytes + 2 * cand_bytes);
  a.ncounters = K * B;
  a.hidden = hidden; a.last_node = last_node; a.T = T; a.B = B; a.K = K; a.d = d;
  a.b1 = b1; a.u = ws; a.logits = head_logits; a.err = err;

  // W1 + SiLU + residual
  a.w = w1; a.rows = d;
  if (dtype == MEDUSA_BF16) launch_gemv_b<uint16_t>(a, true, st); else launch_gemv_b<float>(a, true, st);
  if (int rc = check_launch(fn)) return rc;
  // W2
  a.w = w2; a.rows = V;
  if (dtype == MEDUSA_BF16) launch_gemv_b<uint16_t>(a, false, st); else launch_gemv_b<float>(a, false, st);
  if (int rc = check_launch(fn)) return rc;
  // top-s over each used head's logits (the head table travels by value)
  TopkArgs ta{};
  for (int i = 0; i < a.nused; ++i) { ta.tab.h[i] = a.heads[i]; ta.tab.s[i] = s[a.heads[i]]; }
  ta.logits = head_logits; ta.K = K; ta.V = V; ta.s_max = s_max; ta.nchunk = nchunk;
  ta.cand_v = reinterpret_cast<float*>(ws + u_bytes);
  ta.cand_i = reinterpret_cast<int*>(ws + u_bytes + cand_bytes);
  ta.counters = a.counters;
  ta.topk = topk;
  dim3 g(nchunk, a.nused, B);
  if (smax_used <= 2) launch_kernel(topk_kernel<2>, g, dim3(256), 0, st, ta);
  else if (smax_used <= 4) launch_kernel(topk_kernel<4>, g, dim3(256), 0, st, ta);
  else if (smax_used <= 8) launch_kernel(topk_kernel<8>, g, dim3(256), 0, st, ta);
  else launch_kernel(topk_kernel<16>, g, dim3(256), 0, st, ta);
  return check_launch(fn);
}
