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
// HBM-bound GEMVs: 16-byte streaming loads, eight in flight per lane, the
// input vector re-read from L1.  Two kernels:
//   w1        u[b][k] = dtype(SiLU(W1_k h_b + b1_k) + h_b) into scratch.  A CTA
//             takes four rows at a time, two warps per row (one half each);
//             the halves meet in shared memory for the epilogue.
//   w2_topk   head_logits[b][k] = W2_k u[b][k] (fp32), fused with top-s: a
//             fixed set of CTAs serves each head; after its warps have
//             streamed their rows a CTA merges the running top-S lists its
//             warps kept while streaming (one per warp and sequence, in shared
//             memory), and the last CTA of a head to finish merges every
//             CTA's list into topk (value descending, index ascending).
// With several sequences (bf16) the dot products run on the tensor cores
// instead (mma.sync m16n8k16: the sequences as M, eight weight rows as N): a
// CTA takes eight rows at a time and splits the hidden dimension over its
// warps, so each 16-byte weight load feeds every sequence without being
// widened to fp32, and the sequences' vectors are read once per eight rows
// instead of once per row.
// Rows are handed out at run time, not split up front: W1's row quads and
// each head's W2 rows come from atomic counters, the next one requested
// before the current one is streamed.  CTAs whose SMs are busy with other
// work when the call starts, or that get less bandwidth, then take fewer
// rows, and the call ends within about one row's time of the last free one
// instead of waiting for the slowest fixed share.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace medusa {
namespace {

constexpr int kWarps = 8;  // 256-thread CTAs
constexpr int UNROLL = 8;  // 16-byte loads in flight per lane (CUDA-core GEMVs)
// mma_rows8: 16-byte weight loads in flight per lane (each with the
// sequences' 16 bytes).  Four keep the tensor-core kernels at 64 registers,
// four CTAs per SM: 32 warps per SM hide each other's unit barriers, where
// eight loads per lane at two CTAs per SM streamed about 13% slower.
constexpr int kMmaLoads = 4;
constexpr int kMaxS = MEDUSA_MAX_S;
constexpr int kMaxGroups = 128;  // W2 row groups per CTA above which a group grows (w2_row_group)

struct HeadsArgs {
  const void* w1;      // [K][d][d]
  const void* w2;      // [K][V][d]
  const void* b1;      // [K][d] or null
  const void* hidden;  // [B][T][d]
  const int32_t* last_node;
  int T, B, K, d, V, s_max;
  int nused;
  int32_t heads[MEDUSA_MAX_K];  // ids of the heads with s_k > 0
  int32_t s[MEDUSA_MAX_K];      // their s_k
  void* u;                      // [B][K][d] element type (scratch), or [B*T][K][d] when u_node is set
  const int32_t* u_node;        // u rows per sequence: row b * T + u_node[b] of u (null: row b)
  float* logits;                // [B][K][V]
  int32_t* topk;                // [B][K][s_max]
  float* cand_v;                // [nused][B][cpc][kMaxS] per-CTA candidates (scratch)
  int* cand_i;
  int* counters;                // [nused] CTA arrivals per head, zeroed by w1
  int* rowctr;                  // [nused] W2 row groups handed out per head, zeroed by w1
  int* tickets;                 // W2 CTAs started: a CTA serves head (ticket % nused)
  int* exited;                  // W2 CTAs finished
  int* w1ctr;                   // W1 row quads handed out; zeroed by w2 for the next call
  int cpc;                      // w2 CTAs per used head
  int rgroup;                   // W2 rows per warp in a group of kWarps * rgroup rows
  // optional candidate fill (medusa_heads_topk_candidates): the last head to
  // finish writes tokens[b][n] as medusa_build_candidates does
  int32_t* tokens;              // [B][cT], or null
  const int32_t* next_root;     // [B]
  const int32_t* c_depth;       // tree depth / rank, device [cT]
  const int32_t* c_rank;
  int cT;
  int* heads_done;              // heads merged so far; zero on entry, left zero
  int fill_levels;              // every tree level's head is in use: each head fills its own level
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

// acc[b] += w . x[b] over this lane's share of `nvec` 16-byte vectors.
template <typename TE, int NB>
MDEV void dot_rows(const TE* w, const TE* const* x, int nvec, int B, int lane, float* acc) {
  constexpr int EPV = Vec<TE>::N;
  for (int c0 = lane; c0 < nvec; c0 += 32 * UNROLL) {
    uint4 wv[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int c = c0 + u * 32;
      if (c < nvec) wv[u] = ldg_stream(w + (int64_t)c * EPV);
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int c = c0 + u * 32;
      if (c < nvec) {
        float wf[EPV];
        Vec<TE>::unpack(wv[u], wf);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (b < B) {
            float xf[EPV];
            Vec<TE>::unpack(ldg_v4(x[b] + (int64_t)c * EPV), xf);
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc[b] = fmaf(wf[e], xf[e], acc[b]);
          }
        }
      }
    }
  }
}

// C (16 sequences x 8 weight rows, the m16n8k16 accumulator fragment) +=
// X . W^T over the 32-column chunks [c0, c1) of the hidden dimension.  Lane
// (g, t) = (lane / 4, lane % 4) streams 16 bytes of weight row g (columns
// 32 ch + 8 t .. + 8) per chunk and the same columns of sequences g and g + 8
// (xlo, xhi: null past B); its eight columns feed two MMAs.  In each MMA
// lane t holds the k slots {2t, 2t+1, 2t+8, 2t+9} of both operands, which
// here are columns {8t, 8t+1, 8t+2, 8t+3} (first MMA) and {8t+4 .. 8t+7}
// (second): one permutation of k shared by the two operands, so every dot
// product is unchanged.  wrow, xlo, xhi already include the lane's 8 t.
template <bool HI>
MDEV void mma_rows8(const uint16_t* wrow, const uint16_t* xlo, const uint16_t* xhi, int c0, int c1, float* c) {
  for (int cb = c0; cb < c1; cb += kMmaLoads) {
    uint4 wv[kMmaLoads], xl[kMmaLoads], xh[kMmaLoads];
#pragma unroll
    for (int u = 0; u < kMmaLoads; ++u) {
      const int ch = cb + u;
      if (ch < c1) {
        wv[u] = ldg_stream(wrow + ch * 32);
        xl[u] = xlo ? ldg_v4(xlo + ch * 32) : make_uint4(0, 0, 0, 0);
        if (HI) xh[u] = xhi ? ldg_v4(xhi + ch * 32) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < kMmaLoads; ++u) {
      if (cb + u < c1) {
        const uint32_t a0[4] = {xl[u].x, HI ? xh[u].x : 0u, xl[u].y, HI ? xh[u].y : 0u};
        mma_bf16_16816(c, a0, wv[u].x, wv[u].y);
        const uint32_t a1[4] = {xl[u].z, HI ? xh[u].z : 0u, xl[u].w, HI ? xh[u].w : 0u};
        mma_bf16_16816(c, a1, wv[u].z, wv[u].w);
      }
    }
  }
}

// Element (sequence s, row r) of the warps' summed fragments, or, for the
// thread that calls it, which (lane, register) holds it.
MDEV float frag_sum(const float4 (*part)[32], int s, int r) {
  const int src = 4 * (s & 7) + (r >> 1), reg = ((s >> 3) << 1) + (r & 1);
  float y = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const float4 v = part[w][src];
    y += reg == 0 ? v.x : reg == 1 ? v.y : reg == 2 ? v.z : v.w;
  }
  return y;
}

// ---------------------------------------------------------------- W1 pass --
template <typename TE, int NB>
__global__ void __launch_bounds__(kWarps * 32) heads_w1_kernel(const __grid_constant__ HeadsArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ float part[kWarps][NB];
  __shared__ int s_q;
  if (blockIdx.x == 0 && threadIdx.x < a.nused) {  // for w2_topk
    a.counters[threadIdx.x] = 0;
    a.rowctr[threadIdx.x] = 0;
    if (threadIdx.x == 0) *a.tickets = 0;  // W2's tickets: W2 leaves them counted when W1 runs first
    if (threadIdx.x == 0 && a.heads_done) *a.heads_done = 0;
  }

  // h_b = hidden[b][last_node[b]]; an out-of-range node reads row 0 and raises the error bit
  const TE* x[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    int n = b < a.B ? a.last_node[b] : 0;
    if (n < 0 || n >= a.T) {
      if (threadIdx.x == 0 && blockIdx.x == 0) set_err(a.err, MEDUSA_DEVERR_NODE);
      n = 0;
    }
    x[b] = static_cast<const TE*>(a.hidden) + ((int64_t)(b < a.B ? b : 0) * a.T + n) * a.d;
  }
  const TE* W = static_cast<const TE*>(a.w1);
  const int half = a.d / 2;
  const int hvec = half / Vec<TE>::N;
  const int64_t total = (int64_t)a.nused * a.d;
  const int64_t nquads = (total + kWarps / 2 - 1) / (kWarps / 2);
  const int hf = warp & 1;
  if (threadIdx.x == 0) s_q = atomicAdd(a.w1ctr, 1);
  __syncthreads();
  for (int64_t q = s_q; q < nquads;) {
    int qn = 0;
    if (threadIdx.x == 0) qn = atomicAdd(a.w1ctr, 1);  // the next quad; waited for after this one's loads
    const int64_t g = q * (kWarps / 2) + (warp >> 1);  // row of the stacked used heads
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
    int k = 0, j = 0;
    if (g < total) {
      const int slot = (int)(g / a.d);
      j = (int)(g % a.d);
      k = a.heads[slot];
      const TE* xs[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) xs[b] = x[b] + hf * half;
      dot_rows<TE, NB>(W + ((int64_t)k * a.d + j) * a.d + hf * half, xs, hvec, a.B, lane, acc);
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = warp_sum(acc[b]);
    if (lane == 0) {
#pragma unroll
      for (int b = 0; b < NB; ++b) part[warp][b] = acc[b];
    }
    __syncthreads();
    if (hf == 0 && g < total && lane < a.B && lane < NB) {
      const int b = lane;
      float y = part[warp][b] + part[warp + 1][b];
      if (a.b1) y += to_f32(static_cast<const TE*>(a.b1)[(int64_t)k * a.d + j]);
      const float silu = y / (1.f + expf(-y));
      static_cast<TE*>(a.u)[((int64_t)b * a.K + k) * a.d + j] = from_f32<TE>(silu + to_f32(x[b][j]));
    }
    if (threadIdx.x == 0) s_q = qn;  // every thread read the current quad before the barrier above
    __syncthreads();
    q = s_q;
  }
}

// W1 on the tensor cores (bf16, several sequences): eight stacked W1 rows per
// CTA at a time, handed out from the same counter as the row quads above,
// the hidden dimension split over the eight warps; the warps' fragments meet
// in shared memory and one thread per (sequence, row) applies the epilogue.
template <bool HI>
__global__ void __launch_bounds__(kWarps * 32, 4) heads_w1_mma_kernel(const __grid_constant__ HeadsArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  __shared__ float4 part[2][kWarps][32];
  __shared__ int s_q[2];
  if (blockIdx.x == 0 && threadIdx.x < a.nused) {  // for w2_topk (as in heads_w1_kernel)
    a.counters[threadIdx.x] = 0;
    a.rowctr[threadIdx.x] = 0;
    if (threadIdx.x == 0) *a.tickets = 0;
    if (threadIdx.x == 0 && a.heads_done) *a.heads_done = 0;
  }
  // h_b = hidden[b][last_node[b]]; an out-of-range node reads row 0 and raises the error bit
  auto seq_row = [&](int b) -> const uint16_t* {
    int n = a.last_node[b];
    if (n < 0 || n >= a.T) {
      if (blockIdx.x == 0) set_err(a.err, MEDUSA_DEVERR_NODE);
      n = 0;
    }
    return static_cast<const uint16_t*>(a.hidden) + ((int64_t)b * a.T + n) * a.d;
  };
  const uint16_t* xlo = g < a.B ? seq_row(g) + 8 * t : nullptr;
  const uint16_t* xhi = HI && g + 8 < a.B ? seq_row(g + 8) + 8 * t : nullptr;
  // the epilogue thread's sequence (s, row r of the eight)
  const int es = threadIdx.x >> 3, er = threadIdx.x & 7;
  const uint16_t* xe = es < a.B ? seq_row(es) : nullptr;
  const uint16_t* W = static_cast<const uint16_t*>(a.w1);
  const int nch = a.d / 32;
  const int c0 = warp * nch / kWarps, c1 = (warp + 1) * nch / kWarps;
  const int64_t units = (int64_t)a.nused * a.d / 8;
  if (threadIdx.x == 0) s_q[0] = atomicAdd(a.w1ctr, 1);
  __syncthreads();
  int64_t q = s_q[0];
  for (int it = 0; q < units; ++it) {
    int qn = 0;
    if (threadIdx.x == 0) qn = atomicAdd(a.w1ctr, 1);  // the next unit; waited for after this one's loads
    const int64_t r0 = q * 8;  // first stacked row; eight rows never straddle two heads (d % 8 == 0)
    const int slot = (int)(r0 / a.d), j0 = (int)(r0 % a.d), k = a.heads[slot];
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    mma_rows8<HI>(W + ((int64_t)k * a.d + j0 + g) * a.d + 8 * t, xlo, xhi, c0, c1, c);
    part[it & 1][warp][lane] = make_float4(c[0], c[1], c[2], c[3]);
    if (threadIdx.x == 0) s_q[(it + 1) & 1] = qn;
    __syncthreads();
    if (xe) {
      const int j = j0 + er;
      float y = frag_sum(part[it & 1], es, er);
      if (a.b1) y += bf16_bits_to_f32(static_cast<const uint16_t*>(a.b1)[(int64_t)k * a.d + j]);
      const float silu = y / (1.f + expf(-y));
      static_cast<uint16_t*>(a.u)[((int64_t)es * a.K + k) * a.d + j] = f32_to_bf16_bits(silu + bf16_bits_to_f32(xe[j]));
    }
    q = s_q[(it + 1) & 1];
  }
}

// ---------------------------------------------------------- top-s helpers --

// A register list of the S best (value, index) pairs, sorted.
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
  // Warp-wide: the S best of all lanes' lists, in order, on every lane.
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

// Insert (x, xi) into a sorted list of S (value, index) pairs in shared
// memory, kept by one thread.
template <int S>
MDEV void list_insert(float* v, int* i, float x, int xi) {
  if (!ranks_before(x, xi, v[S - 1], i[S - 1])) return;
  int t = S - 1;
  while (t > 0 && ranks_before(x, xi, v[t - 1], i[t - 1])) {
    v[t] = v[t - 1];
    i[t] = i[t - 1];
    --t;
  }
  v[t] = x;
  i[t] = xi;
}

// Block-wide: the S best of all threads' lists, valid in warp 0.
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

// ------------------------------------------------------- W2 pass + top-s --
// MMA (bf16, several sequences): the rows stream through mma_rows8 in units
// of eight per CTA (the hidden dimension split over the warps); after each
// unit warp w sums row w's fragments and lane s inserts sequence s's value
// into warp w's running top S of that sequence.
template <typename TE, int NB, int S, bool MMA>
MDEV void w2_topk_body(const HeadsArgs& a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ float wv[32][S];
  __shared__ int wi[32][S];
  __shared__ bool last;
  __shared__ float lv[kWarps][NB][S];  // per-warp running top S, per sequence
  __shared__ int li[kWarps][NB][S];
  __shared__ int s_g[2];
  __shared__ int s_ticket;
  // the head this CTA serves goes by the order in which CTAs start, not by
  // blockIdx, so CTAs held back by other work spread over every head
  if (threadIdx.x == 0) s_ticket = atomicAdd(a.tickets, 1);
  // the candidate fill's first node per thread, in case this CTA does it
  int fill_depth = 0, fill_rank = 0;
  if (a.tokens && (int)threadIdx.x < a.B * a.cT) {
    fill_depth = __ldg(a.c_depth + threadIdx.x % a.cT);
    fill_rank = __ldg(a.c_rank + threadIdx.x % a.cT);
  }
  __syncthreads();
  const int slot = s_ticket % a.nused, part = s_ticket / a.nused;
  const int k = a.heads[slot];

  auto seq_x = [&](int b) -> const TE* {
    const int bb = b < a.B ? b : 0;
    int64_t row = bb;
    if (a.u_node) {  // an out-of-range node reads row 0 of the sequence and raises the error bit
      int n = a.u_node[bb];
      if (n < 0 || n >= a.T) {
        if (blockIdx.x == 0) set_err(a.err, MEDUSA_DEVERR_NODE);
        n = 0;
      }
      row = (int64_t)bb * a.T + n;
    }
    return static_cast<const TE*>(a.u) + (row * a.K + k) * a.d;
  };
  const TE* W = static_cast<const TE*>(a.w2) + (int64_t)k * a.V * a.d;
  const int nvec = a.d / Vec<TE>::N;
  // this head's rows in groups of GR = kWarps * RW (RW consecutive rows per
  // warp) from its counter, every group streamed exactly once
  const int RW = a.rgroup, GR = kWarps * RW;
  const int ngroups = (a.V + GR - 1) / GR;
  int* ctr = a.rowctr + slot;
  if (threadIdx.x == 0) s_g[0] = atomicAdd(ctr, 1);
  if (blockIdx.x == 0 && threadIdx.x == 32 && a.w1ctr) *a.w1ctr = 0;  // this call's w1 is done
  // each warp keeps the running top S of the rows it streams, one list per
  // sequence in shared memory (lane b keeps sequence b's)
#pragma unroll 1
  for (int e = lane; e < NB * S; e += 32) {
    lv[warp][e / S][e % S] = -INFINITY;
    li[warp][e / S][e % S] = 0x7fffffff;
  }
  __syncthreads();
  if constexpr (MMA) {
    static_assert(sizeof(TE) == 2 && (NB == 8 || NB == 16), "tensor-core rows: bf16, 8 or 16 sequences");
    constexpr bool HI = NB == 16;
    __shared__ float4 part[2][kWarps][32];
    const int gl = lane >> 2, t = lane & 3;
    const TE* xlo = gl < a.B ? seq_x(gl) + 8 * t : nullptr;
    const TE* xhi = HI && gl + 8 < a.B ? seq_x(gl + 8) + 8 * t : nullptr;
    const int nch = a.d / 32;
    const int c0 = warp * nch / kWarps, c1 = (warp + 1) * nch / kWarps;
    const int units = (a.V + 7) / 8;
    int g = s_g[0];
    for (int it = 0; g < units; ++it) {
      int gn = units;
      if (threadIdx.x == 0) gn = atomicAdd(ctr, 1);  // the next unit; waited for after this one's loads
      const int row0 = g * 8;
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      mma_rows8<HI>(W + (int64_t)min(row0 + gl, a.V - 1) * a.d + 8 * t, xlo, xhi, c0, c1, c);
      part[it & 1][warp][lane] = make_float4(c[0], c[1], c[2], c[3]);
      if (threadIdx.x == 0) s_g[(it + 1) & 1] = gn;
      __syncthreads();
      {  // warp w takes row w of the eight, lane s sequence s (into warp w's list of s):
         // every warp does an equal share, so none lags into the next unit's loads
        const int row = row0 + warp;
        if (lane < a.B && lane < NB && row < a.V) {
          const float y = frag_sum(part[it & 1], lane, warp);
          a.logits[((int64_t)lane * a.K + k) * a.V + row] = y;
          list_insert<S>(lv[warp][lane], li[warp][lane], y, row);
        }
      }
      g = s_g[(it + 1) & 1];
    }
  } else {
    const TE* x[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) x[b] = seq_x(b);
    int g = s_g[0];
    for (int it = 0; g < ngroups; ++it) {
      int gn = ngroups;
      if (threadIdx.x == 0) gn = atomicAdd(ctr, 1);  // the next group; waited for after this one's loads
      const int jb = g * GR + warp * RW;
      const int je = min(a.V, jb + RW);
      for (int j = jb; j < je; ++j) {
        float acc[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[b] = 0.f;
        dot_rows<TE, NB>(W + (int64_t)j * a.d, x, nvec, a.B, lane, acc);
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[b] = warp_sum(acc[b]);
        if (lane < a.B && lane < NB) {
          float y = 0.f;
#pragma unroll
          for (int b = 0; b < NB; ++b)
            if (b == lane) y = acc[b];
          a.logits[((int64_t)lane * a.K + k) * a.V + j] = y;
          list_insert<S>(lv[warp][lane], li[warp][lane], y, j);
        }
      }
      if (threadIdx.x == 0) s_g[(it + 1) & 1] = gn;  // the other slot: read by all before the last barrier
      __syncthreads();
      g = s_g[(it + 1) & 1];
    }
  }
  __syncthreads();  // every warp's lists are complete

  // this CTA's top S per sequence: one warp per sequence merges the warps' lists
  for (int b = warp; b < a.B; b += kWarps) {
    TopList<S> L;
    L.init();
    for (int e = lane; e < kWarps * S; e += 32) L.insert(lv[e / S][b][e % S], li[e / S][b][e % S]);
    float ov[S];
    int oi[S];
    L.warp_select(ov, oi);
    if (lane == 0) {
      const int64_t base = (((int64_t)slot * a.B + b) * a.cpc + part) * kMaxS;
#pragma unroll
      for (int t = 0; t < S; ++t) { a.cand_v[base + t] = ov[t]; a.cand_i[base + t] = oi[t]; }
    }
  }
  // the last CTA of this head to arrive merges all its CTAs' candidates
  __syncthreads();
  if (threadIdx.x == 0) last = arrive_acq_rel(a.counters + slot) == a.cpc - 1;
  __syncthreads();
  if (last) {
    const int s_k = a.s[slot];
    for (int b = 0; b < a.B; ++b) {
      const int64_t base = ((int64_t)slot * a.B + b) * a.cpc * kMaxS;
      TopList<S> L;
      L.init();
      // the CTAs' lists from L2: eight loads in flight per thread, then the inserts
      for (int e0 = threadIdx.x; e0 < a.cpc * S; e0 += 8 * blockDim.x) {
        float cv[8];
        int ci[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int e = e0 + u * blockDim.x;
          cv[u] = -INFINITY;
          ci[u] = 0x7fffffff;
          if (e < a.cpc * S) {
            const int64_t at = base + (int64_t)(e / S) * kMaxS + e % S;
            cv[u] = __ldcg(a.cand_v + at);
            ci[u] = __ldcg(a.cand_i + at);
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) L.insert(cv[u], ci[u]);
      }
      float ov[S];
      int oi[S];
      block_select<S>(L, wv, wi, ov, oi);
      if (warp == 0) {
        int32_t* out = a.topk + ((int64_t)b * a.K + k) * a.s_max;
        for (int t = lane; t < a.s_max; t += 32) {
          int idx = -1;
#pragma unroll
          for (int q = 0; q < S; ++q)
            if (q == t) idx = oi[q];
          out[t] = (t < s_k && idx >= 0 && idx < a.V) ? idx : -1;
        }
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) {  // ready for the next call (every CTA of the head has stopped taking rows)
      a.counters[slot] = 0;
      a.rowctr[slot] = 0;
    }
    if (a.tokens && a.fill_levels) {
      // a node at depth k + 1 takes head k's token of its rank, so each head
      // fills its own tree level as soon as its top-s is merged (slot 0 also
      // the roots), without waiting for the other heads
      __syncthreads();  // this head's topk is written (by warp 0 of this CTA)
      for (int e = threadIdx.x; e < a.B * a.cT; e += blockDim.x) {
        const int b = e / a.cT, n = e % a.cT;
        if (n == 0) {
          if (slot == 0) a.tokens[(int64_t)b * a.cT] = a.next_root[b];
          continue;
        }
        // the first round's node was loaded when the CTA started
        const int dep = e == (int)threadIdx.x ? fill_depth : a.c_depth[n];
        if (dep - 1 != k) continue;
        const int r = (e == (int)threadIdx.x ? fill_rank : a.c_rank[n]) - 1;
        a.tokens[(int64_t)b * a.cT + n] =
            (r >= 0 && r < a.s_max) ? __ldcg(a.topk + ((int64_t)b * a.K + k) * a.s_max + r) : -1;
      }
    } else if (a.tokens) {
      // the last head to be merged fills the next step's candidates
      __syncthreads();  // this head's topk is written
      if (threadIdx.x == 0) last = arrive_acq_rel(a.heads_done) == a.nused - 1;
      __syncthreads();
      if (last) {
        for (int e = threadIdx.x; e < a.B * a.cT; e += blockDim.x) {
          const int b = e / a.cT, n = e % a.cT;
          int32_t tok;
          if (n == 0) {
            tok = a.next_root[b];
          } else {
            // the first round's node was loaded when the CTA started
            const int kk = (e == (int)threadIdx.x ? fill_depth : a.c_depth[n]) - 1;
            const int r = (e == (int)threadIdx.x ? fill_rank : a.c_rank[n]) - 1;
            tok = (kk >= 0 && kk < a.K && r >= 0 && r < a.s_max)
                      ? __ldcg(a.topk + ((int64_t)b * a.K + kk) * a.s_max + r)
                      : -1;
          }
          a.tokens[(int64_t)b * a.cT + n] = tok;
        }
        if (threadIdx.x == 0) *a.heads_done = 0;
      }
    }
  }
  // W2 on its own: the last CTA to leave (every CTA has drawn its ticket)
  // resets the tickets (after W1, W1 resets them at the next call's start)
  if (a.exited && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.exited, 1) == (int)gridDim.x - 1) *a.tickets = *a.exited = 0;
  }
}

// The CUDA-core W2 kernel, and the tensor-core one bounded to 64 registers
// (four CTAs per SM); separate kernels so that each keeps its own register
// budget.
template <typename TE, int NB, int S>
__global__ void __launch_bounds__(kWarps * 32) heads_w2_topk_kernel(const __grid_constant__ HeadsArgs a) {
  w2_topk_body<TE, NB, S, false>(a);
}
template <int NB, int S>
__global__ void __launch_bounds__(kWarps * 32, 4) heads_w2_mma_kernel(const __grid_constant__ HeadsArgs a) {
  w2_topk_body<uint16_t, NB, S, true>(a);
}

// W2 CTAs per used head: about four per SM in total, at least 8 rows each.
int w2_ctas_per_head(int nused, int V) {
  const int target = std::max(1, 4 * sm_count() / std::max(1, nused));
  return std::max(1, std::min(target, (V + 7) / 8));
}

template <typename TE, int NB>
int launch_heads(const HeadsArgs& a, int smax_used, cudaStream_t s) {
  const int64_t quads = ((int64_t)a.nused * a.d + kWarps / 2 - 1) / (kWarps / 2);
  const int g1 = (int)std::max<int64_t>(1, std::min<int64_t>(4 * sm_count(), quads));
  launch_kernel(heads_w1_kernel<TE, NB>, dim3(g1), dim3(kWarps * 32), 0, s, a);
  const dim3 g2(a.nused * a.cpc);
  if (smax_used <= 8)
    launch_kernel(heads_w2_topk_kernel<TE, NB, 8>, g2, dim3(kWarps * 32), 0, s, a);
  else
    launch_kernel(heads_w2_topk_kernel<TE, NB, 16>, g2, dim3(kWarps * 32), 0, s, a);
  return check_launch("medusa_heads_topk");
}

// W2 pass + top-s alone (u computed elsewhere, counters zero on entry).
template <typename TE, int NB>
int launch_w2(const HeadsArgs& a, int smax_used, cudaStream_t s, const char* fn) {
  const dim3 g2(a.nused * a.cpc);
  if (smax_used <= 8)
    launch_kernel(heads_w2_topk_kernel<TE, NB, 8>, g2, dim3(kWarps * 32), 0, s, a);
  else
    launch_kernel(heads_w2_topk_kernel<TE, NB, 16>, g2, dim3(kWarps * 32), 0, s, a);
  return check_launch(fn);
}

// Tensor-core rows (bf16): several sequences and a hidden dimension of at
// least one 32-column chunk per warp.
bool use_mma(const HeadsArgs& a, bool bf16) { return bf16 && a.B >= 2 && a.d % 32 == 0 && a.d / 32 >= kWarps; }

template <int NB>
void launch_w2_mma(const HeadsArgs& a, int smax_used, cudaStream_t s) {
  const dim3 g2(a.nused * a.cpc);
  if (smax_used <= 8)
    launch_kernel(heads_w2_mma_kernel<NB, 8>, g2, dim3(kWarps * 32), 0, s, a);
  else
    launch_kernel(heads_w2_mma_kernel<NB, 16>, g2, dim3(kWarps * 32), 0, s, a);
}

int launch_heads_mma(const HeadsArgs& a, int smax_used, cudaStream_t s) {
  const int64_t units = (int64_t)a.nused * a.d / 8;
  const int g1 = (int)std::max<int64_t>(1, std::min<int64_t>(4 * sm_count(), units));
  if (a.B <= 8) {
    launch_kernel(heads_w1_mma_kernel<false>, dim3(g1), dim3(kWarps * 32), 0, s, a);
    launch_w2_mma<8>(a, smax_used, s);
  } else {
    launch_kernel(heads_w1_mma_kernel<true>, dim3(g1), dim3(kWarps * 32), 0, s, a);
    launch_w2_mma<16>(a, smax_used, s);
  }
  return check_launch("medusa_heads_topk");
}

template <typename TE>
int launch_w2_b(const HeadsArgs& a, int smax_used, cudaStream_t s, const char* fn) {
  if (use_mma(a, sizeof(TE) == 2)) {
    if (a.B <= 8)
      launch_w2_mma<8>(a, smax_used, s);
    else
      launch_w2_mma<16>(a, smax_used, s);
    return check_launch(fn);
  }
  if (a.B == 1) return launch_w2<TE, 1>(a, smax_used, s, fn);
  if (a.B <= 4) return launch_w2<TE, 4>(a, smax_used, s, fn);
  return launch_w2<TE, MEDUSA_MAX_B>(a, smax_used, s, fn);
}

template <typename TE>
int launch_heads_b(const HeadsArgs& a, int smax_used, cudaStream_t s) {
  if (use_mma(a, sizeof(TE) == 2)) return launch_heads_mma(a, smax_used, s);
  if (a.B == 1) return launch_heads<TE, 1>(a, smax_used, s);
  if (a.B <= 4) return launch_heads<TE, 4>(a, smax_used, s);
  return launch_heads<TE, MEDUSA_MAX_B>(a, smax_used, s);
}

// W2 rows per warp in a group: one, unless the head's CTAs would take more
// than kMaxGroups / 2 groups each (fewer counter requests for huge V).
int w2_row_group(int cpc, int V) {
  const int64_t cap = (int64_t)cpc * kWarps * (kMaxGroups / 2);
  return (int)std::max<int64_t>(1, (V + cap - 1) / cap);
}

// Scratch: u [B][K][d] | candidate values | candidate indices | counters
// (CTA arrivals [MEDUSA_MAX_K], W2 row groups [MEDUSA_MAX_K], W1 quads [1],
// heads merged [1], W2 tickets [1], W2 CTAs finished [1]).
struct Layout {
  size_t u, cand, counters, total;
};
Layout heads_layout(int B, int K, int nused, int d, int V) {
  Layout l;
  l.u = align_up((size_t)B * K * d * sizeof(float), 256);  // fp32 size covers both element types
  l.cand = align_up((size_t)nused * B * w2_ctas_per_head(nused, V) * kMaxS * 4, 256);
  l.counters = align_up((size_t)(2 * MEDUSA_MAX_K + 4) * sizeof(int), 256);
  l.total = l.u + 2 * l.cand + l.counters;
  return l;
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_heads_topk_workspace_size(int B, int K, int d, int V, int s_max) {
  (void)s_max;
  if (B < 1 || K < 1 || d < 1 || V < 1) return 0;
  size_t best = 0;  // large enough whichever heads are in use
  for (int n = 1; n <= K; ++n) best = std::max(best, heads_layout(B, K, n, d, V).total);
  return best;
}

namespace {
struct CandFill {
  const int32_t* next_root;
  const medusa_tree_t* tree;
  int32_t* tokens;
};

int heads_topk_impl(const void* hidden, const int32_t* last_node, int T, const void* w1, const void* b1,
                    const void* w2, const int32_t* s, int K, int B, int d, int V, medusa_dtype dtype,
                    float* head_logits, int32_t* topk, int s_max, void* workspace, size_t workspace_bytes,
                    const CandFill* cf, int32_t* err, void* stream, const char* fn) {
  if (!hidden || !last_node || !w1 || !w2 || !s || !head_logits || !topk)
    return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (T < 1 || K < 1 || B < 1 || d < 1 || V < 1 || s_max < 1)
    return fail(MEDUSA_ERR_INVALID, "%s: T=%d K=%d B=%d d=%d V=%d s_max=%d", fn, T, K, B, d, V, s_max);
  if (K > MEDUSA_MAX_K || B > MEDUSA_MAX_B || s_max > MEDUSA_MAX_S)
    return fail(MEDUSA_ERR_UNSUPPORTED, "%s: K=%d B=%d s_max=%d above the maximum", fn, K, B, s_max);
  if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: dtype", fn);
  const int epv = dtype == MEDUSA_BF16 ? 8 : 4;
  if (d % (2 * epv)) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: d=%d not a multiple of %d", fn, d, 2 * epv);
  if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(w1) |
       reinterpret_cast<uintptr_t>(w2)) % 16)
    return fail(MEDUSA_ERR_INVALID, "%s: hidden / w1 / w2 not 16-byte aligned", fn);
  const size_t need = medusa_heads_topk_workspace_size(B, K, d, V, s_max);
  if (!workspace || workspace_bytes < need)
    return fail(MEDUSA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(MEDUSA_ERR_INVALID, "%s: workspace not 256-byte aligned", fn);
  HeadsArgs a{};
  int smax_used = 0;
  for (int k = 0; k < K; ++k) {
    if (s[k] < 0 || s[k] > s_max || s[k] > V)
      return fail(MEDUSA_ERR_INVALID, "%s: s[%d]=%d outside [0, min(s_max, V)]", fn, k, s[k]);
    if (s[k] > 0) {
      a.heads[a.nused] = k;
      a.s[a.nused] = s[k];
      ++a.nused;
      smax_used = std::max(smax_used, (int)s[k]);
    }
  }
  if (a.nused == 0) return MEDUSA_OK;
  const Layout l = heads_layout(B, K, a.nused, d, V);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.w1 = w1; a.w2 = w2; a.b1 = b1; a.hidden = hidden; a.last_node = last_node;
  a.T = T; a.B = B; a.K = K; a.d = d; a.V = V; a.s_max = s_max;
  a.u = ws;
  a.cand_v = reinterpret_cast<float*>(ws + l.u);
  a.cand_i = reinterpret_cast<int*>(ws + l.u + l.cand);
  a.counters = reinterpret_cast<int*>(ws + l.u + 2 * l.cand);
  a.rowctr = a.counters + MEDUSA_MAX_K;
  a.w1ctr = a.counters + 2 * MEDUSA_MAX_K;
  a.tickets = a.counters + 2 * MEDUSA_MAX_K + 2;
  a.exited = nullptr;  // W1 resets the tickets at the start of each call
  a.cpc = w2_ctas_per_head(a.nused, V);
  a.rgroup = w2_row_group(a.cpc, V);
  a.logits = head_logits; a.topk = topk; a.err = err;
  if (cf) {
    a.tokens = cf->tokens; a.next_root = cf->next_root;
    a.c_depth = cf->tree->depth; a.c_rank = cf->tree->rank; a.cT = cf->tree->T;
    a.heads_done = a.counters + 2 * MEDUSA_MAX_K + 1;
    a.fill_levels = 1;
    for (int k = 0; k < cf->tree->K; ++k) a.fill_levels &= s[k] > 0;
  }
  cudaStream_t st = as_stream(stream);
  return dtype == MEDUSA_BF16 ? launch_heads_b<uint16_t>(a, smax_used, st)
                              : launch_heads_b<float>(a, smax_used, st);
}
}  // namespace

extern "C" int medusa_heads_topk(const void* hidden, const int32_t* last_node, int T, const void* w1,
                                 const void* b1, const void* w2, const int32_t* s, int K, int B, int d,
                                 int V, medusa_dtype dtype, float* head_logits, int32_t* topk, int s_max,
                                 void* workspace, size_t workspace_bytes, int32_t* err, void* stream) {
  return heads_topk_impl(hidden, last_node, T, w1, b1, w2, s, K, B, d, V, dtype, head_logits, topk, s_max, workspace,
                         workspace_bytes, nullptr, err, stream, "medusa_heads_topk");
}

extern "C" int medusa_heads_topk_candidates(const void* hidden, const int32_t* last_node, int T, const void* w1,
                                            const void* b1, const void* w2, const int32_t* s, int K, int B, int d,
                                            int V, medusa_dtype dtype, float* head_logits, int32_t* topk,
                                            int s_max, void* workspace, size_t workspace_bytes,
                                            const int32_t* next_root, const medusa_tree_t* tree, int32_t* tokens,
                                            int32_t* err, void* stream) {
  const char* fn = "medusa_heads_topk_candidates";
  if (int rc = check_tree(tree, fn)) return rc;
  if (!next_root || !tokens) return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (K < tree->K || s_max < 1)
    return fail(MEDUSA_ERR_INVALID, "%s: K=%d below the tree depth %d", fn, K, tree->K);
  for (int k = 0; k < tree->K; ++k)
    if (tree->s[k] > s_max) return fail(MEDUSA_ERR_INVALID, "%s: tree s[%d]=%d > s_max=%d", fn, k, tree->s[k], s_max);
  bool any = false;
  for (int k = 0; k < K && s; ++k) any = any || s[k] > 0;
  if (!any)  // no head runs: the fill alone
    return medusa_build_candidates(next_root, topk, s_max, K, tree, B, tokens, stream);
  const CandFill cf{next_root, tree, tokens};
  return heads_topk_impl(hidden, last_node, T, w1, b1, w2, s, K, B, d, V, dtype, head_logits, topk, s_max, workspace,
                         workspace_bytes, &cf, err, stream, fn);
}

extern "C" size_t medusa_heads_logits_topk_workspace_size(int B, int K, int V, int s_max) {
  (void)s_max;
  if (B < 1 || K < 1 || V < 1) return 0;
  size_t best = 0;  // large enough whichever heads are in use
  for (int n = 1; n <= K; ++n) {
    const Layout l = heads_layout(B, K, n, 1, V);
    best = std::max(best, 2 * l.cand + l.counters);
  }
  return best;
}

extern "C" int medusa_heads_logits_topk(const void* u, int T, const int32_t* node, const void* w2,
                                        const int32_t* s, int K, int B, int d, int V, medusa_dtype dtype,
                                        float* head_logits, int32_t* topk, int s_max, void* workspace,
                                        size_t workspace_bytes, int32_t* err, void* stream) {
  const char* fn = "medusa_heads_logits_topk";
  if (!u || !node || !w2 || !s || !head_logits || !topk) return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (T < 1 || K < 1 || B < 1 || d < 1 || V < 1 || s_max < 1)
    return fail(MEDUSA_ERR_INVALID, "%s: T=%d K=%d B=%d d=%d V=%d s_max=%d", fn, T, K, B, d, V, s_max);
  if (K > MEDUSA_MAX_K || B > MEDUSA_MAX_B || s_max > MEDUSA_MAX_S)
    return fail(MEDUSA_ERR_UNSUPPORTED, "%s: K=%d B=%d s_max=%d above the maximum", fn, K, B, s_max);
  if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: dtype", fn);
  const int epv = dtype == MEDUSA_BF16 ? 8 : 4;
  if (d % epv) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: d=%d not a multiple of %d", fn, d, epv);
  if ((reinterpret_cast<uintptr_t>(u) | reinterpret_cast<uintptr_t>(w2)) % 16)
    return fail(MEDUSA_ERR_INVALID, "%s: u / w2 not 16-byte aligned", fn);
  const size_t need = medusa_heads_logits_topk_workspace_size(B, K, V, s_max);
  if (!workspace || workspace_bytes < need)
    return fail(MEDUSA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(MEDUSA_ERR_INVALID, "%s: workspace not 256-byte aligned", fn);
  HeadsArgs a{};
  int smax_used = 0;
  for (int k = 0; k < K; ++k) {
    if (s[k] < 0 || s[k] > s_max || s[k] > V)
      return fail(MEDUSA_ERR_INVALID, "%s: s[%d]=%d outside [0, min(s_max, V)]", fn, k, s[k]);
    if (s[k] > 0) {
      a.heads[a.nused] = k;
      a.s[a.nused] = s[k];
      ++a.nused;
      smax_used = std::max(smax_used, (int)s[k]);
    }
  }
  if (a.nused == 0) return MEDUSA_OK;
  const Layout l = heads_layout(B, K, a.nused, 1, V);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.w2 = w2; a.u = const_cast<void*>(u); a.u_node = node;
  a.T = T; a.B = B; a.K = K; a.d = d; a.V = V; a.s_max = s_max;
  a.cand_v = reinterpret_cast<float*>(ws);
  a.cand_i = reinterpret_cast<int*>(ws + l.cand);
  a.counters = reinterpret_cast<int*>(ws + 2 * l.cand);
  a.rowctr = a.counters + MEDUSA_MAX_K;
  a.tickets = a.counters + 2 * MEDUSA_MAX_K + 2;
  a.exited = a.counters + 2 * MEDUSA_MAX_K + 3;
  a.cpc = w2_ctas_per_head(a.nused, V);
  a.rgroup = w2_row_group(a.cpc, V);
  a.logits = head_logits; a.topk = topk; a.err = err;
  cudaStream_t st = as_stream(stream);
  return dtype == MEDUSA_BF16 ? launch_w2_b<uint16_t>(a, smax_used, st, fn)
                              : launch_w2_b<float>(a, smax_used, st, fn);
}
