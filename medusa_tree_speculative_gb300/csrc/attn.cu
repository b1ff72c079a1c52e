// Tree-masked attention with tree position ids.
//
// "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
// Heads", Method 3 (section 2.1.2, fig. 2) and Pitfalls: all tree nodes are
// appended after the KV cache; each node attends to the cached prefix and to
// its own ancestors (and itself) only; its position id is prefix length +
// depth.  Explainer "085 | Medusa", section 二.2: siblings must stay invisible.
//
// bf16: one kernel.  A thread-block cluster of CL CTAs (CL = 1, 2, 4 or 8)
// serves one (sequence, head, block of query rows).  Each CTA takes a balanced share of the L
// cached prefix keys and a balanced share of the tree keys (flash-decoding
// split; tree keys cost more, so every CTA gets a few).  Each CTA
//   * issues the cp.async copies of its first prefix tile and the loads of
//     its query rows before building the cos/sin tables at pos = L + depth,
//   * rotates its query rows and folds in scale * log2(e),
//   * streams its keys through three shared tile stages (two tiles in flight
//     while one is used; the query rows are staged in the third): prefix keys by
//     cp.async from the cache; tree keys rotated from k_new on the fly and,
//     by the CTAs of the last row block, appended to the cache at slot L + i,
//   * applies the ancestor bitmask to tree keys, runs QK^T and PV on tensor
//     cores (bf16 in, fp32 accumulate) over the 16-key blocks that hold keys,
//     with the online softmax in registers,
//   * after a cluster barrier that every CTA reaches when it has left its key
//     loop, pushes its partial (max, sum, unnormalised O) for each query row
//     into the tile buffers of the CTA that owns the row (rows are dealt
//     round robin).
// After a second cluster barrier each CTA merges its own rows from local
// shared memory and writes the output.  With CL = 1 (few, long CTAs, for a
// caller that runs the attention on the SMs another kernel leaves idle) the
// CTA walks every key and writes its rows directly.  No scratch memory, no
// inter-kernel combine pass.
//
// f32: rope_append (RoPE + KV append, q' staged in scratch) and a plain
// CUDA-core kernel, one CTA per (row, head, sequence).
#include <math.h>

#include <algorithm>
#include <cmath>

#include "cluster.cuh"
#include "common.cuh"
#include "internal.h"

namespace medusa {
namespace {

constexpr int KT = 64;        // keys per shared-memory tile
constexpr int MAX_WARPS = 5;  // 16 query rows per warp; two CTAs per SM
constexpr int kMaxSplits = 8; // most CTAs per cluster (key splits)
constexpr float LOG2E = 1.4426950408889634f;

struct AttnArgs {
  const void* q;
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  const int64_t* seq_start;
  const int32_t* prefix_len;
  const int64_t* seq_cap;
  const int32_t* depth;
  const uint32_t* anc;
  int T, W, K, B, H, Dh, max_prefix;
  float inv_freq[64];  // float(theta^(-2j/Dh)), j < Dh/2, formed on the host in double
  float qscale;        // scale (f32 path) or scale * log2(e) (bf16 path)
  void* out;
  void* qrot;  // f32 path: [B][T][H][Dh]
  int warps, rowblocks;
  int32_t* err;
};

// Query rows are split into row blocks of at most 16 * MAX_WARPS rows, balanced.
void row_split(int T, int& rowblocks, int& warps) {
  rowblocks = (T + 16 * MAX_WARPS - 1) / (16 * MAX_WARPS);
  const int rows = (T + rowblocks - 1) / rowblocks;
  warps = (rows + 15) / 16;
}

// Query rows are dealt to the cluster's CTAs round robin for the merge.
__host__ __device__ constexpr int rows_per_owner(int nrows, int CL) { return (nrows + CL - 1) / CL; }

// Key/value tile stages: three, so that two tiles are in flight while one is
// used (beside a kernel that keeps HBM busy, a tile's loads take several
// microseconds).  The tile buffers also hold the query rows (the last stage,
// first filled after the query fragments have moved to registers) and, once
// every CTA of the cluster has left its key loop, the partials pushed by the
// cluster's CTAs (fp32 O and (max, sum), from the first stage on).
constexpr int kStages = 3;

// Bytes of the pushed partials a CTA receives.
__host__ __device__ constexpr int recv_bytes(int Dh, int warps, int CL) {
  return CL == 1 ? 0 : CL * rows_per_owner(warps * 16, CL) * (Dh + 2) * 4;
}
static_assert(recv_bytes(128, MAX_WARPS, 8) <= kStages * 2 * KT * 128 * 2, "partials fit the tile buffers");
static_assert(recv_bytes(64, MAX_WARPS, 8) <= kStages * 2 * KT * 64 * 2, "partials fit the tile buffers");
static_assert(2 * KT >= MAX_WARPS * 16, "query rows must fit one K+V stage");

size_t smem_bytes(int Dh, int K) {
  return (size_t)kStages * 2 * KT * Dh * 2     // K and V tiles per stage, bf16
         + (size_t)2 * (K + 1) * (Dh / 2) * 4;  // cos / sin per tree depth
}

// Sequence b is usable iff 0 <= L <= max_prefix and L + T fits its capacity.
__device__ bool seq_ok(const AttnArgs& a, int b, int& L, int64_t& st) {
  L = a.prefix_len[b];
  st = a.seq_start[b];
  return L >= 0 && L <= a.max_prefix && (int64_t)L + a.T <= a.seq_cap[b];
}

// Key j of a sequence is visible to query row r iff j is in the prefix or j
// is the slot of an ancestor-or-self of r.
__device__ __forceinline__ bool key_visible(const AttnArgs& a, int L, int r, int j) {
  if (j < L) return true;
  const int node = j - L;
  if (node >= a.T || r >= a.T) return false;
  return (__ldg(a.anc + (int64_t)r * a.W + (node >> 5)) >> (node & 31)) & 1u;
}

// Rotate eight (x1, x2) pairs of bf16: x1' = x1 c - x2 s, x2' = x2 c + x1 s,
// each times `mul`, rounded back to bf16.
__device__ __forceinline__ void rope8(const uint4& lo, const uint4& hi, const float* c, const float* s,
                                      float mul, uint4& olo, uint4& ohi) {
  float a[8], b[8];
  unpack8_bf16(lo, a);
  unpack8_bf16(hi, b);
  float r1[8], r2[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    r1[i] = (a[i] * c[i] - b[i] * s[i]) * mul;
    r2[i] = (b[i] * c[i] + a[i] * s[i]) * mul;
  }
  olo = make_uint4(pack2_bf16(r1[0], r1[1]), pack2_bf16(r1[2], r1[3]), pack2_bf16(r1[4], r1[5]),
                   pack2_bf16(r1[6], r1[7]));
  ohi = make_uint4(pack2_bf16(r2[0], r2[1]), pack2_bf16(r2[2], r2[3]), pack2_bf16(r2[4], r2[5]),
                   pack2_bf16(r2[6], r2[7]));
}


// ---------------------------------------------------------------------------
// bf16: clustered split-K tree attention
// ---------------------------------------------------------------------------
template <int DH, int CL>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(MAX_WARPS * 32, 2)
    attn_tree_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int CH = DH / 8;    // 16-byte chunks per row
  constexpr int HALF = DH / 2;
  constexpr int HCH = CH / 2;   // chunks per rotary half
  constexpr int QI = HCH / 2;   // query items per thread: rows * HCH / (rows * 2)
  constexpr int S = kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* kvbuf = reinterpret_cast<uint16_t*>(smem);  // [S][K, V][KT][DH]
  // [rows][DH] until the q fragments are loaded: the last stage
  uint16_t* qbuf = kvbuf + (S - 1) * 2 * KT * DH;
  const int nrows = a.warps * 16;
  const int RPO = rows_per_owner(nrows, CL);
  // after every CTA of the cluster has left its key loop: the pushed partials
  float* recv_o = reinterpret_cast<float*>(smem);  // [CL][RPO][DH]
  float* recv_ml = recv_o + CL * RPO * DH;         // [CL][RPO][2]
  float* cs = reinterpret_cast<float*>(kvbuf + S * 2 * KT * DH);  // [K+1][HALF]
  float* sn = cs + (a.K + 1) * HALF;

  const uint32_t crank = CL > 1 ? cluster_rank() : 0u;
  const int h = blockIdx.y, b = blockIdx.z / a.rowblocks, rb = blockIdx.z % a.rowblocks;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int row0 = rb * nrows;
  const int HD = a.H * DH;

  int L;
  int64_t st;
  const bool ok = seq_ok(a, b, L, st);
  if (!ok && crank == 0 && h == 0 && rb == 0 && tid == 0) set_err(a.err, MEDUSA_DEVERR_CAPACITY);
  // this CTA's keys: a balanced share of the prefix, then a balanced share of
  // the tree keys that rows of this block can see (all T in the last block,
  // whose CTAs also append them); every CTA reaches both cluster barriers
  const int last_row = min(a.T, row0 + nrows) - 1;
  const int Lk = ok ? L : 0, ntree = ok ? last_row + 1 : 0;
  const int p0 = (int)((int64_t)crank * Lk / CL), p1 = (int)((int64_t)(crank + 1) * Lk / CL);
  const int t0 = (int)crank * ntree / CL, t1 = ((int)crank + 1) * ntree / CL;
  const int np = p1 - p0, nv = np + (t1 - t0);
  const int ntiles = (nv + KT - 1) / KT;
  // ancestor bits of 64 consecutive tree nodes n0 .. n0 + 63 for one query
  // row (a tile's window of this CTA's tree keys)
  const int ra = row0 + (tid >> 5) * 16 + ((tid & 31) >> 2);
  const int rbw = ra + 8;
  auto vis_bits = [&](int r, int n0) -> uint64_t {
    if (!ok || r >= a.T || n0 >= t1) return 0;
    const uint32_t* row = a.anc + (int64_t)r * a.W;
    const int w0 = n0 >> 5, sh = n0 & 31;
    const uint64_t lo = __ldg(row + w0);
    const uint64_t mid = w0 + 1 < a.W ? __ldg(row + w0 + 1) : 0;
    const uint64_t hi = w0 + 2 < a.W ? __ldg(row + w0 + 2) : 0;
    return ((lo | (mid << 32)) >> sh) | (sh ? hi << (64 - sh) : 0);
  };
  // the window of this CTA's first tree keys, loaded before the long-latency work below
  uint64_t vis_a = vis_bits(ra, t0), vis_b = vis_bits(rbw, t0);
  int vis_win = 0;

  const uint16_t* kcache = static_cast<const uint16_t*>(a.k_cache);
  const uint16_t* vcache = static_cast<const uint16_t*>(a.v_cache);
  uint16_t* kcache_w = static_cast<uint16_t*>(a.k_cache);
  uint16_t* vcache_w = static_cast<uint16_t*>(a.v_cache);
  const uint16_t* knew = static_cast<const uint16_t*>(a.k_new);
  const uint16_t* vnew = static_cast<const uint16_t*>(a.v_new);

  // ---- tile loader over this CTA's key list: v < np prefix key p0 + v (by
  // cp.async), np <= v < nv tree node t0 + v - np (rotated here), other rows
  // of the 16-key blocks in use are zero.  Pass 0 issues the prefix copies
  // only; pass 1 the rest; pass 2 everything.
  auto load_tile = [&](int v0, int buf, int pass) {
    const int rows = min(KT, (nv - v0 + 15) / 16 * 16);
    for (int e = tid; e < rows * HCH; e += nthr) {
      const int rr = e / HCH, c = e % HCH;
      const int v = v0 + rr;
      uint16_t* kd = kvbuf + (buf * 2 * KT + rr) * DH;
      uint16_t* vd = kd + KT * DH;
      const int s1 = (c ^ (rr & 7)) * 8, s2 = ((c + HCH) ^ (rr & 7)) * 8;
      if (v < np) {
        if (pass == 1) continue;
        const int64_t off = (st + p0 + v) * HD + (int64_t)h * DH;
        cp_async16(smem_u32(kd + s1), kcache + off + c * 8, 16);
        cp_async16(smem_u32(kd + s2), kcache + off + (c + HCH) * 8, 16);
        cp_async16(smem_u32(vd + s1), vcache + off + c * 8, 16);
        cp_async16(smem_u32(vd + s2), vcache + off + (c + HCH) * 8, 16);
      } else if (pass == 0) {
        continue;
      } else if (v < nv) {
        const int n = t0 + v - np;  // tree node
        const int64_t src = (((int64_t)b * a.T + n) * a.H + h) * DH;
        const int d = min(max(__ldg(a.depth + n), 0), a.K);
        uint4 klo, khi;
        rope8(ldg_v4(knew + src + c * 8), ldg_v4(knew + src + (c + HCH) * 8), cs + d * HALF + c * 8,
              sn + d * HALF + c * 8, 1.f, klo, khi);
        const uint4 vlo = ldg_v4(vnew + src + c * 8), vhi = ldg_v4(vnew + src + (c + HCH) * 8);
        *reinterpret_cast<uint4*>(kd + s1) = klo;
        *reinterpret_cast<uint4*>(kd + s2) = khi;
        *reinterpret_cast<uint4*>(vd + s1) = vlo;
        *reinterpret_cast<uint4*>(vd + s2) = vhi;
        if (rb == a.rowblocks - 1) {  // the last row block holds every tree key: append K', V at L + n
          const int64_t dst = (st + L + n) * HD + (int64_t)h * DH;
          *reinterpret_cast<uint4*>(kcache_w + dst + c * 8) = klo;
          *reinterpret_cast<uint4*>(kcache_w + dst + (c + HCH) * 8) = khi;
          *reinterpret_cast<uint4*>(vcache_w + dst + c * 8) = vlo;
          *reinterpret_cast<uint4*>(vcache_w + dst + (c + HCH) * 8) = vhi;
        }
      } else {
        const uint4 z = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(kd + s1) = z;
        *reinterpret_cast<uint4*>(kd + s2) = z;
        *reinterpret_cast<uint4*>(vd + s1) = z;
        *reinterpret_cast<uint4*>(vd + s2) = z;
      }
    }
  };

  // ---- first the long-latency work: the prefix copies of the first S - 1
  // tiles (one commit group each), the query loads
#pragma unroll
  for (int j = 0; j < S - 1; ++j) {
    if (j < ntiles) load_tile(j * KT, j, 0);
    cp_async_commit();
  }
  const uint16_t* q = static_cast<const uint16_t*>(a.q);
  uint4 qlo[QI], qhi[QI];
  int qd[QI];
#pragma unroll
  for (int i = 0; i < QI; ++i) {
    const int e = tid + i * nthr;  // < nrows * HCH
    const int r = row0 + e / HCH, c = e % HCH;
    qlo[i] = qhi[i] = make_uint4(0, 0, 0, 0);
    qd[i] = 0;
    if (ok && r < a.T) {
      const int64_t src = (((int64_t)b * a.T + r) * a.H + h) * DH;
      qlo[i] = ldg_v4(q + src + c * 8);
      qhi[i] = ldg_v4(q + src + (c + HCH) * 8);
      qd[i] = min(max(__ldg(a.depth + r), 0), a.K);
    }
  }
  // ---- cos/sin at positions L + d for every tree depth d
  if (ok) {
    for (int e = tid; e < (a.K + 1) * HALF; e += nthr) {
      const int d = e / HALF, j = e % HALF;
      const float ang = __fmul_rn((float)(L + d), a.inv_freq[j]);
      float s, c;
      sincosf(ang, &s, &c);
      cs[e] = c;
      sn[e] = s;
    }
  }
  __syncthreads();
  // ---- query rows: rotate at L + depth, scale, round to bf16
#pragma unroll
  for (int i = 0; i < QI; ++i) {
    const int e = tid + i * nthr;
    const int rr = e / HCH, c = e % HCH;
    uint4 lo = qlo[i], hi = qhi[i];
    if (ok && row0 + rr < a.T)
      rope8(qlo[i], qhi[i], cs + qd[i] * HALF + c * 8, sn + qd[i] * HALF + c * 8, a.qscale, lo, hi);
    *reinterpret_cast<uint4*>(qbuf + rr * DH + ((c ^ (rr & 7)) * 8)) = lo;
    *reinterpret_cast<uint4*>(qbuf + rr * DH + (((c + HCH) ^ (rr & 7)) * 8)) = hi;
  }
  // tree keys and zero rows of those tiles (they need the tables)
#pragma unroll
  for (int j = 0; j < S - 1; ++j)
    if (j < ntiles) load_tile(j * KT, j, 1);
  __syncthreads();
  uint32_t qf[DH / 16][4];
  {
    const int rr = warp * 16 + (lane & 15);
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk) {
      const int c = kk * 2 + (lane >> 4);
      ldmatrix_x4(qf[kk], smem_u32(qbuf + rr * DH + ((c ^ (rr & 7)) * 8)));
    }
  }
  // the query buffer becomes the last tile stage
  __syncthreads();

  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  float o[DH / 8][4];
#pragma unroll
  for (int n = 0; n < DH / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

  for (int t = 0; t < ntiles; ++t) {
    const int v0 = t * KT;
    const int buf = t % S;
    // tile t + S - 1 into the stage tile t - 1 used (freed by the barrier that
    // ended the previous iteration); one commit group per tile, empty past the
    // end, so that S - 1 pending groups mean tile t has landed
    const int nxt = t + S - 1;
    if (nxt < ntiles) load_tile(nxt * KT, nxt % S, 2);
    cp_async_commit();
    cp_async_wait<S - 1>();
    __syncthreads();
    const uint16_t* kb = kvbuf + buf * 2 * KT * DH;
    const uint16_t* vb = kb + KT * DH;
    const int nb = min(KT / 16, (nv - v0 + 15) / 16);  // 16-key blocks holding keys

    // S = q' K^T  (16 rows x 64 keys per warp)
    float s[KT / 8][4];
#pragma unroll
    for (int n = 0; n < KT / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk) {
#pragma unroll
      for (int np16 = 0; np16 < KT / 16; ++np16) {
        if (np16 < nb) {
          const int rr = np16 * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int c = kk * 2 + ((lane >> 3) & 1);
          uint32_t r[4];
          ldmatrix_x4(r, smem_u32(kb + rr * DH + ((c ^ (rr & 7)) * 8)));
          mma_bf16_16816(s[2 * np16], qf[kk], r[0], r[1]);
          mma_bf16_16816(s[2 * np16 + 1], qf[kk], r[2], r[3]);
        }
      }
    }
    // mask: past this CTA's keys; ancestor bits on tree keys (bit v - np -
    // vis_win of the window that starts at this tile's first tree key)
    if (v0 + KT > np) {
      const int win = max(v0, np) - np;
      if (win != vis_win) {
        vis_a = vis_bits(ra, t0 + win);
        vis_b = vis_bits(rbw, t0 + win);
        vis_win = win;
      }
#pragma unroll
      for (int n = 0; n < KT / 8; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int v = v0 + n * 8 + (lane & 3) * 2 + (e & 1);
          const uint64_t vis = e < 2 ? vis_a : vis_b;
          if (v >= nv || (v >= np && !((vis >> (v - np - win)) & 1ull))) s[n][e] = -INFINITY;
        }
      }
    }
    // online softmax (log2 domain: q' carries log2(e))
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int n = 0; n < KT / 8; ++n) {
      mx_a = fmaxf(mx_a, fmaxf(s[n][0], s[n][1]));
      mx_b = fmaxf(mx_b, fmaxf(s[n][2], s[n][3]));
    }
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float base_a = mn_a == -INFINITY ? 0.f : mn_a;
    const float base_b = mn_b == -INFINITY ? 0.f : mn_b;
    const float al_a = exp2f(m_a - base_a), al_b = exp2f(m_b - base_b);
    m_a = mn_a;
    m_b = mn_b;
    l_a *= al_a;
    l_b *= al_b;
#pragma unroll
    for (int n = 0; n < DH / 8; ++n) {
      o[n][0] *= al_a; o[n][1] *= al_a;
      o[n][2] *= al_b; o[n][3] *= al_b;
    }
    uint32_t pf[KT / 16][4];
#pragma unroll
    for (int n = 0; n < KT / 8; ++n) {
      const float p0 = exp2f(s[n][0] - base_a), p1 = exp2f(s[n][1] - base_a);
      const float p2 = exp2f(s[n][2] - base_b), p3 = exp2f(s[n][3] - base_b);
      l_a += p0 + p1;
      l_b += p2 + p3;
      pf[n >> 1][(n & 1) * 2 + 0] = pack2_bf16(p0, p1);
      pf[n >> 1][(n & 1) * 2 + 1] = pack2_bf16(p2, p3);
    }
    // O += P V
#pragma unroll
    for (int j = 0; j < KT / 16; ++j) {
      if (j < nb) {
#pragma unroll
        for (int dp = 0; dp < DH / 16; ++dp) {
          const int rr = j * 16 + (lane & 15);
          const int c = dp * 2 + (lane >> 4);
          uint32_t r[4];
          ldmatrix_x4_trans(r, smem_u32(vb + rr * DH + ((c ^ (rr & 7)) * 8)));
          mma_bf16_16816(o[2 * dp], pf[j], r[0], r[1]);
          mma_bf16_16816(o[2 * dp + 1], pf[j], r[2], r[3]);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);

  const int la = warp * 16 + (lane >> 2), lb = la + 8;
  if constexpr (CL == 1) {
    // ---- every key was this CTA's: normalise and write the rows
    if (!ok) return;
    uint16_t* out = static_cast<uint16_t*>(a.out);
    const float ia = l_a > 0.f ? 1.f / l_a : 0.f, ib = l_b > 0.f ? 1.f / l_b : 0.f;
    const bool wa = row0 + la < a.T, wb = row0 + lb < a.T;
    uint16_t* oa = out + (((int64_t)b * a.T + row0 + la) * a.H + h) * DH;
    uint16_t* ob = out + (((int64_t)b * a.T + row0 + lb) * a.H + h) * DH;
#pragma unroll
    for (int n = 0; n < DH / 8; ++n) {
      const int col = n * 8 + (lane & 3) * 2;
      if (wa) *reinterpret_cast<uint32_t*>(oa + col) = pack2_bf16(o[n][0] * ia, o[n][1] * ia);
      if (wb) *reinterpret_cast<uint32_t*>(ob + col) = pack2_bf16(o[n][2] * ib, o[n][3] * ib);
    }
    return;
  }

  // ---- push this CTA's partial of each local row to the row's owner
  // (rank rr % CL, slot rr / CL), into the owner's tile buffers: every CTA
  // has left its key loop (and its copies have landed) at this barrier
  cluster_sync();
  const uint32_t o_base = smem_u32(recv_o), ml_base = smem_u32(recv_ml);
  if (row0 + la < a.T) {
    const uint32_t ra_o = cluster_map(o_base + (((int)crank * RPO + la / CL) * DH) * 4, (uint32_t)(la % CL));
    const uint32_t rb_o = cluster_map(o_base + (((int)crank * RPO + lb / CL) * DH) * 4, (uint32_t)(lb % CL));
    const bool push_b = row0 + lb < a.T;
#pragma unroll
    for (int n = 0; n < DH / 8; ++n) {
      const int col = n * 8 + (lane & 3) * 2;
      st_cluster_f32x2(ra_o + col * 4, o[n][0], o[n][1]);
      if (push_b) st_cluster_f32x2(rb_o + col * 4, o[n][2], o[n][3]);
    }
    if ((lane & 3) == 0) {
      st_cluster_f32x2(cluster_map(ml_base + (((int)crank * RPO + la / CL) * 2) * 4, (uint32_t)(la % CL)), m_a, l_a);
      if (push_b)
        st_cluster_f32x2(cluster_map(ml_base + (((int)crank * RPO + lb / CL) * 2) * 4, (uint32_t)(lb % CL)), m_b,
                         l_b);
    }
  }
  cluster_sync();  // every partial has landed; nothing remote is touched after this

  // ---- merge this CTA's rows (local rows crank, crank + CL, ...) from local shared memory
  __shared__ float wgt[(MAX_WARPS * 16 + CL - 1) / CL][CL];  // per (row, source rank): weight / denominator
  const int my_rows = ok ? (nrows - (int)crank + CL - 1) / CL : 0;
  for (int i = tid; i < my_rows; i += nthr) {
    float m[CL], l[CL], M = -INFINITY;
#pragma unroll
    for (int c = 0; c < CL; ++c) {
      m[c] = recv_ml[(c * RPO + i) * 2];
      l[c] = recv_ml[(c * RPO + i) * 2 + 1];
      M = fmaxf(M, m[c]);
    }
    float den = 0.f, w[CL];
#pragma unroll
    for (int c = 0; c < CL; ++c) {
      w[c] = m[c] == -INFINITY ? 0.f : exp2f(m[c] - M);
      den += w[c] * l[c];
    }
#pragma unroll
    for (int c = 0; c < CL; ++c) wgt[i][c] = den > 0.f ? w[c] / den : 0.f;
  }
  __syncthreads();
  uint16_t* out = static_cast<uint16_t*>(a.out);
  for (int e = tid; e < my_rows * (DH / 2); e += nthr) {
    const int i = e / (DH / 2), d = (e % (DH / 2)) * 2;
    const int r = row0 + (int)crank + i * CL;
    if (r >= a.T) continue;
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < CL; ++c) {
      const float wc = wgt[i][c];
      if (wc != 0.f) {
        const float2 v = *reinterpret_cast<const float2*>(recv_o + (c * RPO + i) * DH + d);
        acc.x += wc * v.x;
        acc.y += wc * v.y;
      }
    }
    *reinterpret_cast<uint32_t*>(out + (((int64_t)b * a.T + r) * a.H + h) * DH + d) = pack2_bf16(acc.x, acc.y);
  }
}

// ---------------------------------------------------------------------------
// f32: RoPE + KV append, then one CTA per (row, head, sequence)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) rope_append_f32_kernel(const __grid_constant__ AttnArgs a) {
  const int i = blockIdx.x, b = blockIdx.y;
  int L;
  int64_t st;
  if (!seq_ok(a, b, L, st)) {
    if (i == 0 && threadIdx.x == 0) set_err(a.err, MEDUSA_DEVERR_CAPACITY);
    return;
  }
  const int half = a.Dh / 2;
  __shared__ float cs[64], sn[64];
  const int64_t pos = (int64_t)L + a.depth[i];
  for (int j = threadIdx.x; j < half; j += blockDim.x) {
    const float ang = __fmul_rn((float)pos, a.inv_freq[j]);
    float s, c;
    sincosf(ang, &s, &c);
    cs[j] = c;
    sn[j] = s;
  }
  __syncthreads();
  const float* __restrict__ q = static_cast<const float*>(a.q);
  const float* __restrict__ kn = static_cast<const float*>(a.k_new);
  const float* __restrict__ vn = static_cast<const float*>(a.v_new);
  float* kc = static_cast<float*>(a.k_cache);
  float* vc = static_cast<float*>(a.v_cache);
  float* qr = static_cast<float*>(a.qrot);
  const int64_t row = ((int64_t)b * a.T + i) * a.H * a.Dh;
  const int64_t slot = (st + L + i) * (int64_t)a.H * a.Dh;
  for (int e = threadIdx.x; e < a.H * half; e += blockDim.x) {
    const int h = e / half, j = e % half;
    const int64_t o1 = (int64_t)h * a.Dh + j, o2 = o1 + half;
    const float c = cs[j], s = sn[j];
    const float q1 = q[row + o1], q2 = q[row + o2];
    const float k1 = kn[row + o1], k2 = kn[row + o2];
    qr[row + o1] = (q1 * c - q2 * s) * a.qscale;
    qr[row + o2] = (q2 * c + q1 * s) * a.qscale;
    kc[slot + o1] = k1 * c - k2 * s;
    kc[slot + o2] = k2 * c + k1 * s;
    vc[slot + o1] = vn[row + o1];
    vc[slot + o2] = vn[row + o2];
  }
}

// Warps stride over the visible keys with an online softmax; lanes split the
// head dimension.
__global__ void __launch_bounds__(128) attn_f32_kernel(AttnArgs a) {
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  int L;
  int64_t st;
  if (!seq_ok(a, b, L, st)) return;
  constexpr int NW = 4, PER = 4;  // Dh <= 32 * PER
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Dh = a.Dh, HD = a.H * a.Dh;
  const float* qr = static_cast<const float*>(a.qrot) + (((int64_t)b * a.T + i) * a.H + h) * Dh;
  const float* kc = static_cast<const float*>(a.k_cache);
  const float* vc = static_cast<const float*>(a.v_cache);
  float qv[PER], ov[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int d = lane + 32 * e;
    qv[e] = d < Dh ? qr[d] : 0.f;
    ov[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int j = warp; j < L + a.T; j += NW) {
    if (!key_visible(a, L, i, j)) continue;
    const int64_t off = (st + j) * HD + (int64_t)h * Dh;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int d = lane + 32 * e;
      if (d < Dh) dot += qv[e] * kc[off + d];
    }
    const float sc = warp_sum(dot);  // q' already carries the scale
    const float mn = fmaxf(m, sc);
    const float al = expf(m - mn), p = expf(sc - mn);
    m = mn;
    l = l * al + p;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int d = lane + 32 * e;
      ov[e] = ov[e] * al + (d < Dh ? p * vc[off + d] : 0.f);
    }
  }
  __shared__ float sm[NW], sl[NW], so[NW][32 * PER];
  if (lane == 0) { sm[warp] = m; sl[warp] = l; }
#pragma unroll
  for (int e = 0; e < PER; ++e) so[warp][lane + 32 * e] = ov[e];
  __syncthreads();
  if (warp == 0) {
    float M = -INFINITY;
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sm[w]);
    float den = 0.f;
    for (int w = 0; w < NW; ++w) den += sm[w] == -INFINITY ? 0.f : expf(sm[w] - M) * sl[w];
    float* out = static_cast<float*>(a.out) + (((int64_t)b * a.T + i) * a.H + h) * Dh;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int d = lane + 32 * e;
      if (d >= Dh) continue;
      float num = 0.f;
      for (int w = 0; w < NW; ++w) num += sm[w] == -INFINITY ? 0.f : expf(sm[w] - M) * so[w][d];
      out[d] = den > 0.f ? num / den : 0.f;
    }
  }
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_tree_attn_workspace_size(int B, int H, int Dh, int T, int max_prefix) {
  if (B < 1 || H < 1 || Dh < 1 || T < 1 || max_prefix < 0) return 0;
  // the f32 path stages q' in scratch; the bf16 path needs none
  return align_up((size_t)B * T * H * Dh * sizeof(float), 256);
}

namespace medusa {
namespace {

template <int DH, int CL>
void launch_attn_bf16(const AttnArgs& a, int B, int H, cudaStream_t s) {
  dim3 grid(CL, H, B * a.rowblocks);
  const size_t sm = smem_bytes(DH, a.K);
  cudaFuncSetAttribute(attn_tree_kernel<DH, CL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  launch_kernel(attn_tree_kernel<DH, CL>, grid, dim3(a.warps * 32), sm, s, a);
}

template <int DH>
void launch_attn_bf16(const AttnArgs& a, int B, int H, int splits, cudaStream_t s) {
  switch (splits) {
    case 1: launch_attn_bf16<DH, 1>(a, B, H, s); break;
    case 2: launch_attn_bf16<DH, 2>(a, B, H, s); break;
    case 4: launch_attn_bf16<DH, 4>(a, B, H, s); break;
    default: launch_attn_bf16<DH, kMaxSplits>(a, B, H, s); break;
  }
}

}  // namespace
}  // namespace medusa

extern "C" int medusa_tree_attn(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                void* v_cache, const int64_t* seq_start, const int32_t* prefix_len,
                                const int64_t* seq_cap, const medusa_tree_t* tree, int B, int H,
                                int Dh, int max_prefix, float rope_theta, float scale,
                                medusa_dtype dtype, void* out, void* workspace,
                                size_t workspace_bytes, int32_t* err, void* stream) {
  return medusa_tree_attn_splits(q, k_new, v_new, k_cache, v_cache, seq_start, prefix_len, seq_cap, tree, B, H,
                                 Dh, max_prefix, rope_theta, scale, dtype, out, workspace, workspace_bytes,
                                 kMaxSplits, err, stream);
}

extern "C" int medusa_tree_attn_splits(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                       void* v_cache, const int64_t* seq_start, const int32_t* prefix_len,
                                       const int64_t* seq_cap, const medusa_tree_t* tree, int B, int H,
                                       int Dh, int max_prefix, float rope_theta, float scale,
                                       medusa_dtype dtype, void* out, void* workspace,
                                       size_t workspace_bytes, int key_splits, int32_t* err, void* stream) {
  const char* fn = "medusa_tree_attn";
  if (int rc = check_tree(tree, fn)) return rc;
  if (key_splits != 1 && key_splits != 2 && key_splits != 4 && key_splits != kMaxSplits)
    return fail(MEDUSA_ERR_UNSUPPORTED, "%s: key_splits=%d not in {1,2,4,8}", fn, key_splits);
  if (key_splits != kMaxSplits && dtype != MEDUSA_BF16)
    return fail(MEDUSA_ERR_UNSUPPORTED, "%s: key_splits=%d needs bf16", fn, key_splits);
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !seq_start || !prefix_len || !seq_cap || !out)
    return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (B < 1 || B > MEDUSA_MAX_B || H < 1 || max_prefix < 0)
    return fail(MEDUSA_ERR_INVALID, "%s: bad B=%d H=%d max_prefix=%d", fn, B, H, max_prefix);
  if (Dh != 64 && Dh != 128) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: Dh=%d not in {64,128}", fn, Dh);
  if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: dtype", fn);
  if (!(rope_theta > 0.f) || !(scale > 0.f)) return fail(MEDUSA_ERR_INVALID, "%s: rope_theta/scale", fn);
  const bool bf16 = dtype == MEDUSA_BF16;
  if (bf16 && ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_new) |
                reinterpret_cast<uintptr_t>(v_new) | reinterpret_cast<uintptr_t>(k_cache) |
                reinterpret_cast<uintptr_t>(v_cache)) % 16))
    return fail(MEDUSA_ERR_INVALID, "%s: tensors not 16-byte aligned", fn);
  const size_t need = bf16 ? 0 : medusa_tree_attn_workspace_size(B, H, Dh, tree->T, max_prefix);
  if (need && (!workspace || workspace_bytes < need))
    return fail(MEDUSA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, workspace_bytes, need);
  if (need && reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(MEDUSA_ERR_INVALID, "%s: workspace not 256-byte aligned", fn);

  AttnArgs a{};
  a.q = q; a.k_new = k_new; a.v_new = v_new; a.k_cache = k_cache; a.v_cache = v_cache;
  a.seq_start = seq_start; a.prefix_len = prefix_len; a.seq_cap = seq_cap;
  a.depth = tree->depth; a.anc = tree->anc_mask; a.T = tree->T; a.W = tree->W; a.K = tree->K;
  a.B = B; a.H = H; a.Dh = Dh; a.max_prefix = max_prefix;
  for (int j = 0; j < Dh / 2; ++j)
    a.inv_freq[j] = (float)(1.0 / std::pow((double)rope_theta, (2.0 * j) / (double)Dh));
  a.qscale = bf16 ? scale * LOG2E : scale;
  a.out = out;
  a.qrot = workspace;
  a.err = err;
  row_split(tree->T, a.rowblocks, a.warps);
  cudaStream_t s = as_stream(stream);

  if (bf16) {
    if (Dh == 128)
      launch_attn_bf16<128>(a, B, H, key_splits, s);
    else
      launch_attn_bf16<64>(a, B, H, key_splits, s);
    return check_launch(fn);
  }
  dim3 g1(tree->T, B);
  launch_kernel(rope_append_f32_kernel, g1, dim3(256), 0, s, a);
  if (int rc = check_launch(fn)) return rc;
  dim3 g2(tree->T, H, B);
  launch_kernel(attn_f32_kernel, g2, dim3(128), 0, s, a);
  return check_launch(fn);
}
