// Tree-masked attention with tree position ids.
//
// "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
// Heads", Method 3 (section 2.1.2, fig. 2) and Pitfalls: all tree nodes are
// appended after the KV cache; each node attends to the cached prefix and to
// its own ancestors (and itself) only; its position id is prefix length +
// depth.  Explainer "085 | Medusa", section 二.2: siblings must stay invisible.
//
// Three kernels per call:
//   1. rope_append   rotate q and k_new at pos = L + depth, write k', v_new
//                    into cache slots L + i, stage q' (pre-scaled) in scratch.
//   2. attn_partial  flash-decoding split over the L + T keys of each
//                    sequence: one CTA per (key split, head, row block); the
//                    ancestor bitmask is applied to the tree keys; QK^T and PV
//                    run on tensor cores (bf16 in, fp32 accumulate), the
//                    online softmax in registers (log2 domain).
//   3. attn_combine  merge the splits' (max, sum, unnormalised O).
// The f32 element type runs a plain CUDA-core kernel in place of 2-3.
#include <math.h>

#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace medusa {
namespace {

constexpr int KT = 64;         // keys per shared-memory tile
constexpr int MAX_WARPS = 8;   // 16 query rows per warp
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
  int T, W, B, H, Dh, max_prefix;
  float inv_freq[64];  // float(theta^(-2j/Dh)), j < Dh/2, formed on the host in double
  float qscale;  // folded into q': scale (f32 path) or scale*log2(e) (bf16)
  void* out;
  void* qrot;      // [B][T][H][Dh] element type
  float* part_o;   // [B][H][n_splits][T][Dh]
  float* part_ml;  // [B][H][n_splits][T][2]
  int n_splits, chunk, warps, rowblocks;
  int32_t* err;
};

struct Plan {
  int warps, rowblocks, n_splits, chunk;
  size_t q_bytes, o_bytes, ml_bytes, total;
};

Plan make_plan(int B, int H, int Dh, int T, int max_prefix, size_t esz, bool mma_path) {
  Plan p{};
  p.warps = std::min(MAX_WARPS, (T + 15) / 16);
  p.rowblocks = (T + 16 * p.warps - 1) / (16 * p.warps);
  const long keys = (long)max_prefix + T;
  if (mma_path) {
    const long per_split = (long)B * H * p.rowblocks;
    const long target = 2L * sm_count();
    long ns = (target + per_split - 1) / per_split;
    ns = std::max(1L, std::min(ns, (keys + KT - 1) / KT));
    long chunk = (keys + ns - 1) / ns;
    chunk = (chunk + KT - 1) / KT * KT;
    p.chunk = (int)chunk;
    p.n_splits = (int)((keys + chunk - 1) / chunk);
  } else {
    p.chunk = (int)keys;
    p.n_splits = 1;
  }
  p.q_bytes = align_up((size_t)B * T * H * Dh * esz, 256);
  if (mma_path) {
    p.o_bytes = align_up((size_t)B * H * p.n_splits * T * Dh * sizeof(float), 256);
    p.ml_bytes = align_up((size_t)B * H * p.n_splits * T * 2 * sizeof(float), 256);
  }
  p.total = p.q_bytes + p.o_bytes + p.ml_bytes;
  return p;
}

// Sequence b is usable iff 0 <= L <= max_prefix and L + T fits its capacity.
__device__ bool seq_ok(const AttnArgs& a, int b, int& L, int64_t& st) {
  L = a.prefix_len[b];
  st = a.seq_start[b];
  return L >= 0 && L <= a.max_prefix && (int64_t)L + a.T <= a.seq_cap[b];
}

// ---------------------------------------------------------------------------
// 1. RoPE + KV append
// ---------------------------------------------------------------------------
template <typename TE>
__global__ void __launch_bounds__(256) rope_append_kernel(AttnArgs a) {
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
    // angle formed in float: float(pos) * inv_freq_j
    const float ang = __fmul_rn((float)pos, a.inv_freq[j]);
    float s, c;
    sincosf(ang, &s, &c);
    cs[j] = c;
    sn[j] = s;
  }
  __syncthreads();
  const TE* q = static_cast<const TE*>(a.q);
  const TE* kn = static_cast<const TE*>(a.k_new);
  const TE* vn = static_cast<const TE*>(a.v_new);
  TE* kc = static_cast<TE*>(a.k_cache);
  TE* vc = static_cast<TE*>(a.v_cache);
  TE* qr = static_cast<TE*>(a.qrot);
  const int64_t row = ((int64_t)b * a.T + i) * a.H * a.Dh;
  const int64_t slot = (st + L + i) * (int64_t)a.H * a.Dh;
  for (int e = threadIdx.x; e < a.H * half; e += blockDim.x) {
    const int h = e / half, j = e % half;
    const int64_t o1 = (int64_t)h * a.Dh + j, o2 = o1 + half;
    const float c = cs[j], s = sn[j];
    const float q1 = to_f32(q[row + o1]), q2 = to_f32(q[row + o2]);
    const float k1 = to_f32(kn[row + o1]), k2 = to_f32(kn[row + o2]);
    qr[row + o1] = from_f32<TE>((q1 * c - q2 * s) * a.qscale);
    qr[row + o2] = from_f32<TE>((q2 * c + q1 * s) * a.qscale);
    kc[slot + o1] = from_f32<TE>(k1 * c - k2 * s);
    kc[slot + o2] = from_f32<TE>(k2 * c + k1 * s);
    vc[slot + o1] = vn[row + o1];
    vc[slot + o2] = vn[row + o2];
  }
}

// Key j of a sequence is visible to query row r iff j is in the prefix or j
// is the slot of an ancestor-or-self of r.
__device__ __forceinline__ bool key_visible(const AttnArgs& a, int L, int r, int j) {
  if (j < L) return true;
  const int node = j - L;
  if (node >= a.T || r >= a.T) return false;
  return (__ldg(a.anc + (int64_t)r * a.W + (node >> 5)) >> (node & 31)) & 1u;
}

// ---------------------------------------------------------------------------
// 2. split-K partial attention on tensor cores (bf16)
// ---------------------------------------------------------------------------
template <int DH>
__global__ void __launch_bounds__(MAX_WARPS * 32) attn_partial_kernel(AttnArgs a) {
  constexpr int CH = DH / 8;  // 16-byte chunks per row
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* kbuf = reinterpret_cast<uint16_t*>(smem);  // [2][KT][DH]
  uint16_t* vbuf = kbuf + 2 * KT * DH;                // [2][KT][DH]

  const int split = blockIdx.x, h = blockIdx.y;
  const int b = blockIdx.z / a.rowblocks, rb = blockIdx.z % a.rowblocks;
  int L;
  int64_t st;
  if (!seq_ok(a, b, L, st)) return;
  const int n_keys = L + a.T;
  const int k_begin = split * a.chunk;
  const int k_end = min(n_keys, k_begin + a.chunk);
  if (k_begin >= k_end) return;  // combine skips splits past n_keys

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nthr = blockDim.x;
  const int row0 = rb * a.warps * 16;
  const int nrows = a.warps * 16;
  const int HD = a.H * DH;

  // ---- stage q' rows (already rotated and scaled) through shared memory
  const uint16_t* qrot = static_cast<const uint16_t*>(a.qrot);
  for (int e = threadIdx.x; e < nrows * CH; e += nthr) {
    const int rr = e / CH, c = e % CH;
    const int r = row0 + rr;
    const uint16_t* src = qrot + ((int64_t)b * a.T + min(r, a.T - 1)) * HD + (int64_t)h * DH + c * 8;
    cp_async16(smem_u32(kbuf + rr * DH + ((c ^ (rr & 7)) * 8)), src, r < a.T ? 16 : 0);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  uint32_t qf[DH / 16][4];
  {
    const int rr = warp * 16 + (lane & 15);
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk) {
      const int c = kk * 2 + (lane >> 4);
      ldmatrix_x4(qf[kk], smem_u32(kbuf + rr * DH + ((c ^ (rr & 7)) * 8)));
    }
  }
  __syncthreads();

  const uint16_t* kcache = static_cast<const uint16_t*>(a.k_cache);
  const uint16_t* vcache = static_cast<const uint16_t*>(a.v_cache);
  auto load_tile = [&](int kt, int buf) {
    for (int e = threadIdx.x; e < KT * CH; e += nthr) {
      const int rr = e / CH, c = e % CH;
      const int j = kt + rr;
      const bool ok = j < k_end;
      const int64_t off = (st + (ok ? j : k_begin)) * HD + (int64_t)h * DH + c * 8;
      const int sw = (c ^ (rr & 7)) * 8;
      cp_async16(smem_u32(kbuf + (buf * KT + rr) * DH + sw), kcache + off, ok ? 16 : 0);
      cp_async16(smem_u32(vbuf + (buf * KT + rr) * DH + sw), vcache + off, ok ? 16 : 0);
    }
  };

  const int ra = row0 + warp * 16 + (lane >> 2);  // this thread's two rows
  const int rbw = ra + 8;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  float o[DH / 8][4];
#pragma unroll
  for (int n = 0; n < DH / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

  const int ntiles = (k_end - k_begin + KT - 1) / KT;
  load_tile(k_begin, 0);
  cp_async_commit();
  for (int t = 0; t < ntiles; ++t) {
    const int kt = k_begin + t * KT;
    const int buf = t & 1;
    if (t + 1 < ntiles) {
      load_tile(kt + KT, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint16_t* kb = kbuf + buf * KT * DH;
    const uint16_t* vb = vbuf + buf * KT * DH;

    // S = q' K^T  (16 rows x 64 keys per warp)
    float s[KT / 8][4];
#pragma unroll
    for (int n = 0; n < KT / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < KT / 16; ++np) {
        const int rr = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int c = kk * 2 + ((lane >> 3) & 1);
        uint32_t r[4];
        ldmatrix_x4(r, smem_u32(kb + rr * DH + ((c ^ (rr & 7)) * 8)));
        mma_bf16_16816(s[2 * np], qf[kk], r[0], r[1]);
        mma_bf16_16816(s[2 * np + 1], qf[kk], r[2], r[3]);
      }
    }
    // mask: the tail past k_end everywhere; ancestor bits on tree keys
    const bool tail = kt + KT > k_end;
    const bool tree = kt + KT > L;
    if (tail || tree) {
#pragma unroll
      for (int n = 0; n < KT / 8; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = kt + n * 8 + (lane & 3) * 2 + (e & 1);
          const int r = e < 2 ? ra : rbw;
          if (j >= k_end || !key_visible(a, L, r, j)) s[n][e] = -INFINITY;
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
    __syncthreads();
  }
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);

  const int64_t base = (((int64_t)b * a.H + h) * a.n_splits + split) * a.T;
#pragma unroll
  for (int n = 0; n < DH / 8; ++n) {
    const int col = n * 8 + (lane & 3) * 2;
    if (ra < a.T)
      *reinterpret_cast<float2*>(a.part_o + (base + ra) * DH + col) = make_float2(o[n][0], o[n][1]);
    if (rbw < a.T)
      *reinterpret_cast<float2*>(a.part_o + (base + rbw) * DH + col) = make_float2(o[n][2], o[n][3]);
  }
  if ((lane & 3) == 0) {
    if (ra < a.T) *reinterpret_cast<float2*>(a.part_ml + (base + ra) * 2) = make_float2(m_a, l_a);
    if (rbw < a.T) *reinterpret_cast<float2*>(a.part_ml + (base + rbw) * 2) = make_float2(m_b, l_b);
  }
}

// ---------------------------------------------------------------------------
// 3. merge the key splits
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) attn_combine_kernel(AttnArgs a) {
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  int L;
  int64_t st;
  if (!seq_ok(a, b, L, st)) return;
  const int used = (L + a.T + a.chunk - 1) / a.chunk;
  const int64_t base = ((int64_t)b * a.H + h) * a.n_splits * a.T;
  float M = -INFINITY;
  for (int sp = 0; sp < used; ++sp) M = fmaxf(M, a.part_ml[(base + (int64_t)sp * a.T + i) * 2]);
  const float Mb = M == -INFINITY ? 0.f : M;
  uint16_t* out = static_cast<uint16_t*>(a.out);
  for (int d = threadIdx.x; d < a.Dh; d += blockDim.x) {
    float num = 0.f, den = 0.f;
    for (int sp = 0; sp < used; ++sp) {
      const int64_t r = base + (int64_t)sp * a.T + i;
      const float w = exp2f(a.part_ml[r * 2] - Mb);
      den += w * a.part_ml[r * 2 + 1];
      num += w * a.part_o[r * a.Dh + d];
    }
    out[(((int64_t)b * a.T + i) * a.H + h) * a.Dh + d] = f32_to_bf16_bits(den > 0.f ? num / den : 0.f);
  }
}

// ---------------------------------------------------------------------------
// f32: one CTA per (row, head, sequence); warps stride over the visible keys
// with an online softmax; lanes split the head dimension.
// ---------------------------------------------------------------------------
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
  // the bf16 plan is the larger of the two; callers may size for either type
  Plan p = make_plan(B, H, Dh, T, max_prefix, 4, true);
  Plan pb = make_plan(B, H, Dh, T, max_prefix, 2, true);
  return std::max(p.q_bytes + pb.o_bytes + pb.ml_bytes, pb.total);
}

extern "C" int medusa_tree_attn(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                void* v_cache, const int64_t* seq_start, const int32_t* prefix_len,
                                const int64_t* seq_cap, const medusa_tree_t* tree, int B, int H,
                                int Dh, int max_prefix, float rope_theta, float scale,
                                medusa_dtype dtype, void* out, void* workspace,
                                size_t workspace_bytes, int32_t* err, void* stream) {
  const char* fn = "medusa_tree_attn";
  if (int rc = check_tree(tree, fn)) return rc;
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !seq_start || !prefix_len || !seq_cap || !out)
    return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (B < 1 || B > MEDUSA_MAX_B || H < 1 || max_prefix < 0)
    return fail(MEDUSA_ERR_INVALID, "%s: bad B=%d H=%d max_prefix=%d", fn, B, H, max_prefix);
  if (Dh != 64 && Dh != 128) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: Dh=%d not in {64,128}", fn, Dh);
  if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: dtype", fn);
  if (!(rope_theta > 0.f) || !(scale > 0.f)) return fail(MEDUSA_ERR_INVALID, "%s: rope_theta/scale", fn);
  const bool bf16 = dtype == MEDUSA_BF16;
  Plan p = make_plan(B, H, Dh, tree->T, max_prefix, bf16 ? 2 : 4, bf16);
  if (!workspace || workspace_bytes < p.total)
    return fail(MEDUSA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, workspace_bytes, p.total);
  if (reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(MEDUSA_ERR_INVALID, "%s: workspace not 256-byte aligned", fn);

  AttnArgs a{};
  a.q = q; a.k_new = k_new; a.v_new = v_new; a.k_cache = k_cache; a.v_cache = v_cache;
  a.seq_start = seq_start; a.prefix_len = prefix_len; a.seq_cap = seq_cap;
  a.depth = tree->depth; a.anc = tree->anc_mask; a.T = tree->T; a.W = tree->W;
  a.B = B; a.H = H; a.Dh = Dh; a.max_prefix = max_prefix;
  for (int j = 0; j < Dh / 2; ++j)
    a.inv_freq[j] = (float)(1.0 / std::pow((double)rope_theta, (2.0 * j) / (double)Dh));
  a.qscale = bf16 ? scale * LOG2E : scale;
  a.out = out;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.qrot = ws;
  a.part_o = reinterpret_cast<float*>(ws + p.q_bytes);
  a.part_ml = reinterpret_cast<float*>(ws + p.q_bytes + p.o_bytes);
  a.n_splits = p.n_splits; a.chunk = p.chunk; a.warps = p.warps; a.rowblocks = p.rowblocks;
  a.err = err;
  cudaStream_t s = as_stream(stream);

  dim3 g1(tree->T, B);
  if (bf16) {
    rope_append_kernel<uint16_t><<<g1, 256, 0, s>>>(a);
    if (int rc = check_launch(fn)) return rc;
    dim3 g2(p.n_splits, H, B * p.rowblocks);
    const size_t sm = 2 * 2 * KT * Dh * sizeof(uint16_t);
    if (Dh == 128) {
      cudaFuncSetAttribute(attn_partial_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
      attn_partial_kernel<128><<<g2, p.warps * 32, sm, s>>>(a);
    } else {
      attn_partial_kernel<64><<<g2, p.warps * 32, sm, s>>>(a);
    }
    if (int rc = check_launch(fn)) return rc;
    dim3 g3(tree->T, H, B);
    attn_combine_kernel<<<g3, 128, 0, s>>>(a);
    return check_launch(fn);
  }
  rope_append_kernel<float><<<g1, 256, 0, s>>>(a);
  if (int rc = check_launch(fn)) return rc;
  dim3 g2(tree->T, H, B);
  attn_f32_kernel<<<g2, 128, 0, s>>>(a);
  return check_launch(fn);
}
