// Tree-masked attention with tree position ids on the tensor cores
// (tcgen05, accumulators in tensor memory).
//
// "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
// Heads", Method 3 (section 2.1.2, fig. 2) and Pitfalls: all tree nodes are
// appended after the KV cache; each node attends to the cached prefix and to
// its own ancestors (and itself) only; its position id is prefix length +
// depth.  Explainer "085 | Medusa", section 二.2: siblings must stay invisible.
//
// bf16, Dh = 128.  One CTA per (sequence, head, block of up to 128 query
// rows) walks every key of the sequence in tiles of 128 keys:
//   * first every thread helps append the tree's keys (rotated at L + depth)
//     and values to the cache at slot L + i, so that the tree keys arrive
//     through the same tensor-map loads as the prefix; the query rows are
//     rotated, scaled by scale * log2(e) and stored in shared memory in the
//     128-byte-swizzled K-major layout the MMA reads;
//   * warp 0 (one thread) loads key tiles with TMA into a ring of three
//     stages and value tiles into a ring of two;
//   * warp 1 allocates tensor memory and one thread issues the MMAs:
//     S_t = Q K_t^T (M = 128 query rows, N = 128 keys, K = 128) into one of
//     two S accumulators, two tiles ahead, and PV_t = P_t V_t (N = 128 value
//     columns, K = 128 keys; P is read from tensor memory, where it replaced
//     S_t; V is read in its cache layout, keys x values, as an MN-major
//     operand) into one of two more accumulators in turn;
//   * warps 2-9 give each query row (its tensor-memory lane) two threads,
//     one per half of the tile's keys and of the output columns: read S_t,
//     mask it (keys past the sequence; tree keys that are not an
//     ancestor-or-self of the row), agree on the row's running max through
//     shared memory, write P_t = 2^(S - max) in bf16 over S_t in tensor
//     memory for the PV MMA, and fold PV_{t-1} into the output registers with
//     the online-softmax rescale while PV_t runs.
// Keeping P in tensor memory leaves the shared memory it would take to a
// third key stage: a key tile's load is issued three tiles before its S MMA
// instead of two, which covers the HBM latency under load (2-4 us).
// Every mbarrier wait is bounded; a wait that gives up sets
// MEDUSA_DEVERR_TIMEOUT, lets the copies in flight land, frees tensor memory
// and returns.
#include <cuda.h>
#include <math.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "cluster.cuh"
#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace medusa {
namespace {

using namespace sm100;

constexpr int DH = 128;        // head dimension (two 64-wide swizzle spans)
constexpr int BN = 128;        // keys per tile (MMA N of S, K of PV)
constexpr int BMR = 128;       // query rows per CTA (MMA M)
constexpr int kThreads = 320;  // warp 0 loads, warp 1 MMAs, warps 2-9 softmax (two per row quarter)
constexpr int kSoftThreads = 256;
constexpr int kMaxWords = (MEDUSA_MAX_T + 31) / 32;
constexpr float kLog2e = 1.4426950408889634f;

// Shared memory (1024-byte aligned regions).
constexpr uint32_t kQOff = 0;                    // Q   [2 k-chunks][128 rows][128 B]
constexpr uint32_t kKOff = 32768;                // K   [3 stages][2 k-chunks][128 keys][128 B]
constexpr uint32_t kVOff = 131072;               // V   [2 stages][2 column halves][128 keys][128 B]
constexpr int kKStages = 3;
constexpr uint32_t kTileBytes = 32768;           // one K or V tile
constexpr uint32_t kBarOff = 196608;             // mbarriers, tensor-memory slot, flags
constexpr uint32_t kAncOff = kBarOff + 192 + 2048;  // ancestor words [128 rows][kMaxWords]
constexpr uint32_t kCsOff = kAncOff + BMR * kMaxWords * 4;  // cos / sin [K+1][64] each
constexpr uint32_t kTmemCols = 512;              // S0, S1 (P_t over S_t), PV0, PV1 (128 columns each)
constexpr int kPartStride = DH + 4;              // merge: floats per partial row (padded)
constexpr uint32_t kPartOff = kKOff;             // merge: this CTA's O partial [128 rows][kPartStride] fp32
constexpr uint32_t kMlOff = kPartOff + BMR * kPartStride * 4;  // merge: (max, sum) [128 rows]
constexpr uint32_t kXOff = kBarOff + 192;        // partial row maxima [2 tiles][2 halves][128 rows] (floats)

struct AttnTcArgs {
  const uint16_t* q;
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint16_t* k_cache;
  uint16_t* v_cache;
  const int64_t* seq_start;
  const int32_t* prefix_len;
  const int64_t* seq_cap;
  const int32_t* depth;
  const uint32_t* anc;
  int T, W, K, B, H, max_prefix, rowblocks;
  float inv_freq[DH / 2];  // float(theta^(-2j/Dh)), formed on the host in double
  float qscale;            // scale * log2(e)
  uint16_t* out;
  int32_t* err;
};

// Shared-memory matrix descriptor of an MN-major operand in 128-byte
// swizzled rows: rows of 64 elements along MN (128 B) stacked along K, 8-row
// atoms of 1024 B; `lbo` = bytes between 64-element groups along MN, `sbo` =
// bytes between 8-row groups along K.
MDEV uint64_t desc_mnmajor_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Generic-proxy writes visible to the async proxy (tensor cores, TMA).
MDEV void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
MDEV void fence_async_global() { asm volatile("fence.proxy.async.global;\n" ::: "memory"); }

MDEV bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 255 && *abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

// Sequence b is usable iff 0 <= L <= max_prefix and L + T fits its capacity.
MDEV bool seq_ok(const AttnTcArgs& a, int b, int& L, int64_t& st) {
  L = a.prefix_len[b];
  st = a.seq_start[b];
  return L >= 0 && L <= a.max_prefix && (int64_t)L + a.T <= a.seq_cap[b];
}

// 16 bytes of row r, 16-byte chunk c (0..7) of a 128-byte-swizzled region.
MDEV uint32_t sw128(uint32_t region, int r, int c) { return region + r * 128 + ((c ^ (r & 7)) << 4); }

// Rotate eight (x1, x2) pairs of bf16: x1' = x1 c - x2 s, x2' = x2 c + x1 s,
// each times `mul`, rounded back to bf16.
MDEV void rope8(const uint4& lo, const uint4& hi, const float* c, const float* s, float mul, uint4& olo,
                uint4& ohi) {
  float x1[8], x2[8];
  unpack8_bf16(lo, x1);
  unpack8_bf16(hi, x2);
  float r1[8], r2[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    r1[i] = (x1[i] * c[i] - x2[i] * s[i]) * mul;
    r2[i] = (x2[i] * c[i] + x1[i] * s[i]) * mul;
  }
  olo = make_uint4(pack2_bf16(r1[0], r1[1]), pack2_bf16(r1[2], r1[3]), pack2_bf16(r1[4], r1[5]),
                   pack2_bf16(r1[6], r1[7]));
  ohi = make_uint4(pack2_bf16(r2[0], r2[1]), pack2_bf16(r2[2], r2[3]), pack2_bf16(r2[4], r2[5]),
                   pack2_bf16(r2[6], r2[7]));
}

// (a, b) += (x, y) as one packed fp32x2 add, round to nearest.
MDEV void add2(float& a, float& b, float x, float y) {
  asm("{\n .reg .b64 A, X;\n mov.b64 A, {%0, %1};\n mov.b64 X, {%2, %3};\n add.rn.f32x2 A, A, X;\n"
      " mov.b64 {%0, %1}, A;\n}\n"
      : "+f"(a), "+f"(b)
      : "f"(x), "f"(y));
}
// (a, b) = (a, b) * s + (x, y) as one packed fp32x2 fused multiply-add.
MDEV void fma2(float& a, float& b, float s, float x, float y) {
  asm("{\n .reg .b64 A, S, X;\n mov.b64 A, {%0, %1};\n mov.b64 S, {%2, %2};\n mov.b64 X, {%3, %4};\n"
      " fma.rn.f32x2 A, A, S, X;\n mov.b64 {%0, %1}, A;\n}\n"
      : "+f"(a), "+f"(b)
      : "f"(s), "f"(x), "f"(y));
}
// 2^x with the hardware approximation (subnormal results flush to 0; 2^-inf = 0).
MDEV float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

MDEV void st_shared_f4(uint32_t addr, float x, float y, float z, float w) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "f"(x), "f"(y), "f"(z), "f"(w) : "memory");
}
MDEV void st_shared_f2(uint32_t addr, float x, float y) {
  asm volatile("st.shared.v2.f32 [%0], {%1, %2};\n" ::"r"(addr), "f"(x), "f"(y) : "memory");
}

MDEV void st_shared_v4(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

template <int CL>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ AttnTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* k_full = bars;       // [3] TMA -> MMA
  uint64_t* k_empty = bars + 3;  // [3] MMA -> TMA
  uint64_t* v_full = bars + 6;   // [2]
  uint64_t* v_empty = bars + 8;  // [2]
  uint64_t* s_full = bars + 10;  // [2] MMA -> softmax: S_t ready
  // [2] softmax -> MMA: P_t written over S_t (256 arrivals).  Two barriers,
  // tile t on t & 1: the softmax may finish P_{t+1} before the MMA thread
  // has waited for P_t (P_{t+1} does not wait for PV_t), and with one
  // barrier the phase the MMA thread waits for would already be two back.
  uint64_t* p_full = bars + 12;
  uint64_t* pv_full = bars + 14; // [2] MMA -> softmax: PV_t ready (accumulator t & 1)
  uint64_t* pv_empty = bars + 16;// [2] softmax -> MMA: PV accumulator read (256 arrivals)
  uint64_t* mma_done = bars + 18;// every MMA issued so far has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 19);
  int* s_abort = reinterpret_cast<int*>(bars + 20);
  uint64_t* xm_full = bars + 21; // [2] softmax halves: the row's partial maxima written (256 arrivals)
  float* xmax = reinterpret_cast<float*>(smem + kXOff);  // [2 tiles][2 halves][128 rows]
  uint32_t* ancs = reinterpret_cast<uint32_t*>(smem + kAncOff);
  float* cs = reinterpret_cast<float*>(smem + kCsOff);
  float* sn = cs + (a.K + 1) * (DH / 2);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, b = blockIdx.z / a.rowblocks, rb = blockIdx.z % a.rowblocks;
  const int row0 = rb * BMR;
  int L;
  int64_t st;
  if (!seq_ok(a, b, L, st)) {  // the whole CTA leaves before any barrier or allocation
    if (h == 0 && rb == 0 && blockIdx.x == 0 && tid == 0) set_err(a.err, MEDUSA_DEVERR_CAPACITY);
    return;
  }
  const int nkeys = L + a.T, ntiles = (nkeys + BN - 1) / BN;
  const int HD = a.H * DH;
  // this CTA's run of key tiles, [t_begin, t_begin + nt): the first CTAs of
  // the unit take the extra tiles, the last one holds the tree's keys
  constexpr int sp = CL;
  const int crank = blockIdx.x;
  const int t_begin = (int)(((int64_t)crank * ntiles + sp - 1) / sp);
  const int nt = (int)(((int64_t)(crank + 1) * ntiles + sp - 1) / sp) - t_begin;
  // tree nodes whose keys fall in this CTA's tiles (this CTA appends them)
  const int n_lo = max(0, t_begin * BN - L), n_hi = min(a.T, (t_begin + nt) * BN - L);
  const int nlive = min(BMR, a.T - row0);  // query rows of this block
  int n_early = 0;  // tiles the loader issued before the prologue (thread 0 only)

  if (tid == 0) {
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kSoftThreads);
      mbar_init(&pv_full[i], 1);
      mbar_init(&pv_empty[i], kSoftThreads);
      mbar_init(&xm_full[i], kSoftThreads);
    }
    mbar_init(mma_done, 1);
    fence_barrier_init();
    *s_abort = 0;
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    // the first tiles that hold prefix keys only need no appended row: they
    // load while the prologue runs (fresh stages, nothing to wait for)
    for (; n_early < 2 && n_early < nt && (t_begin + n_early + 1) * BN <= L; ++n_early) {
      const int y = (int)(st + (int64_t)(t_begin + n_early) * BN);
      mbar_expect_tx(&k_full[n_early], kTileBytes);
      for (int kc = 0; kc < 2; ++kc)
        tma_load_2d(smem + kKOff + n_early * kTileBytes + kc * 16384, &tmK, &k_full[n_early], h * DH + kc * 64, y);
      mbar_expect_tx(&v_full[n_early], kTileBytes);
      for (int kc = 0; kc < 2; ++kc)
        tma_load_2d(smem + kVOff + n_early * kTileBytes + kc * 16384, &tmV, &v_full[n_early], h * DH + kc * 64, y);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  // query rows of this block: their loads go out first and land while the
  // rotation tables are formed
  constexpr int kQPer = (BMR * 8 + kThreads - 1) / kThreads;
  uint4 qlo[kQPer], qhi[kQPer];
  int qd[kQPer];
#pragma unroll
  for (int k = 0; k < kQPer; ++k) {
    const int e = tid + k * kThreads, r = e >> 3, c = e & 7;  // row, 16-byte chunk of the first half
    qlo[k] = make_uint4(0, 0, 0, 0);
    qhi[k] = qlo[k];
    qd[k] = 0;
    if (r < nlive) {
      const int64_t src = (((int64_t)b * a.T + row0 + r) * a.H + h) * DH;
      qd[k] = min(max(__ldg(a.depth + row0 + r), 0), a.K);
      qlo[k] = ldg_v4(a.q + src + c * 8);
      qhi[k] = ldg_v4(a.q + src + 64 + c * 8);
    }
  }
  // cos / sin at positions L + d for every tree depth d
  for (int e = tid; e < (a.K + 1) * (DH / 2); e += kThreads) {
    const int d = e / (DH / 2), j = e % (DH / 2);
    const float ang = __fmul_rn((float)(L + d), a.inv_freq[j]);
    float s, c;
    sincosf(ang, &s, &c);
    cs[e] = c;
    sn[e] = s;
  }
  // ancestor words of this block's rows
  for (int e = tid; e < BMR * a.W; e += kThreads) {
    const int r = e / a.W, w = e % a.W;
    ancs[r * kMaxWords + w] = r < nlive ? __ldg(a.anc + (int64_t)(row0 + r) * a.W + w) : 0u;
  }
  __syncthreads();
  // query rows rotated at L + depth, times scale * log2(e), bf16, swizzled
  // K-major; rows past the tree are zero
#pragma unroll
  for (int k = 0; k < kQPer; ++k) {
    const int e = tid + k * kThreads, r = e >> 3, c = e & 7;
    if (e < BMR * 8) {
      uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
      if (r < nlive) rope8(qlo[k], qhi[k], cs + qd[k] * 64 + c * 8, sn + qd[k] * 64 + c * 8, a.qscale, lo, hi);
      st_shared_v4(sw128(sbase + kQOff, r, c), lo);
      st_shared_v4(sw128(sbase + kQOff + 16384, r, c), hi);
    }
  }
  // the tree's keys (rotated at L + depth) and values into the cache at slot
  // L + i, for the nodes whose keys fall in this CTA's tiles; every row block
  // of the sequence writes the same bytes
  const int items = (n_hi - n_lo) * 8;  // 16-byte chunks of the first half
  for (int e0 = tid; e0 < items; e0 += 2 * kThreads) {
    uint4 kl[2], kh[2], vl[2], vh[2];
    int dd[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = e0 + u * kThreads;
      if (e < items) {
        const int i = n_lo + (e >> 3), c = e & 7;
        const int64_t src = (((int64_t)b * a.T + i) * a.H + h) * DH + c * 8;
        dd[u] = min(max(__ldg(a.depth + i), 0), a.K);
        kl[u] = ldg_v4(a.k_new + src);
        kh[u] = ldg_v4(a.k_new + src + 64);
        vl[u] = ldg_v4(a.v_new + src);
        vh[u] = ldg_v4(a.v_new + src + 64);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = e0 + u * kThreads;
      if (e < items) {
        const int i = n_lo + (e >> 3), c = e & 7;
        const int64_t dst = (st + L + i) * HD + (int64_t)h * DH + c * 8;
        uint4 klo, khi;
        rope8(kl[u], kh[u], cs + dd[u] * 64 + c * 8, sn + dd[u] * 64 + c * 8, 1.f, klo, khi);
        *reinterpret_cast<uint4*>(a.k_cache + dst) = klo;
        *reinterpret_cast<uint4*>(a.k_cache + dst + 64) = khi;
        *reinterpret_cast<uint4*>(a.v_cache + dst) = vl[u];
        *reinterpret_cast<uint4*>(a.v_cache + dst + 64) = vh[u];
      }
    }
  }
  if (items > 0) fence_async_global();  // the appended rows are read back through the tensor maps
  fence_async_smem();  // Q is read by the tensor cores
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  volatile int* abort_flag = s_abort;

  if (warp == 0) {
    // ---------------- TMA: key tiles (three stages) and value tiles (two)
    // The two rings advance on their own: a key tile goes out as soon as its
    // stage is free (S of the tile three back has completed), a value tile
    // as soon as its stage is (PV of the tile two back), never before its
    // key tile; the thread polls both without blocking on either, sleeping
    // briefly between polls.
    if (lane == 0) {
      int tk = n_early, tv = n_early;  // next key / value tile to load
      bool ok = true;
      uint32_t idle = 0;
      while (tk < nt || tv < nt) {
        bool moved = false;
        if (tk < nt) {
          const int ks = tk % kKStages;
          if (mbar_test_wait(&k_empty[ks], ((uint32_t)(tk / kKStages) & 1u) ^ 1u)) {
            const int y = (int)(st + (int64_t)(t_begin + tk) * BN);
            mbar_expect_tx(&k_full[ks], kTileBytes);
            for (int kc = 0; kc < 2; ++kc)
              tma_load_2d(smem + kKOff + ks * kTileBytes + kc * 16384, &tmK, &k_full[ks], h * DH + kc * 64, y);
            ++tk;
            moved = true;
          }
        }
        if (tv < tk) {
          const int vs = tv & 1;
          if (mbar_test_wait(&v_empty[vs], ((uint32_t)(tv >> 1) & 1u) ^ 1u)) {
            const int y = (int)(st + (int64_t)(t_begin + tv) * BN);
            mbar_expect_tx(&v_full[vs], kTileBytes);
            for (int kc = 0; kc < 2; ++kc)
              tma_load_2d(smem + kVOff + vs * kTileBytes + kc * 16384, &tmV, &v_full[vs], h * DH + kc * 64, y);
            ++tv;
            moved = true;
          }
        }
        if (moved) {
          idle = 0;
        } else if (++idle > kSpinLimit || ((idle & 255) == 255 && *abort_flag)) {
          if (idle > kSpinLimit) *abort_flag = 1;
          ok = false;
          break;
        } else {
          __nanosleep(64);  // leave the issue slots to the softmax warps on this sub-partition
        }
      }
      if (!ok) {
        // let the tiles already issued land before the CTA can exit (a key
        // tile is issued at most three tiles ahead of its use, a value tile two)
        for (int j = max(0, tk - kKStages); j < tk; ++j) mbar_wait(&k_full[j % kKStages], (uint32_t)(j / kKStages) & 1u);
        for (int j = max(0, tv - 2); j < tv; ++j) mbar_wait(&v_full[j & 1], (uint32_t)(j >> 1) & 1u);
        set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
      }
    }
    if constexpr (CL > 1) {  // the merge's two cluster barriers
      __syncwarp();
      cluster_sync();
      cluster_sync();
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(BMR, BN);
      const uint32_t idPV = idesc_bf16_f32(BMR, DH) | (1u << 16);  // B (V) MN-major
      bool ok = true;
      // S_t into accumulator t & 1, which P_{t-2} occupied until PV_{t-2}
      // completed
      auto issue_s = [&](int t) {
        const int s = t & 1, ks = t % kKStages;
        const uint32_t kph = (uint32_t)(t / kKStages) & 1u;
        if (!wait_or_abort(&k_full[ks], kph, abort_flag) ||
            (t >= 2 && !wait_or_abort(&pv_full[s], (uint32_t)((t - 2) >> 1) & 1u, abort_flag))) {
          ok = false;
          return;
        }
        tc_fence_after();
        const uint32_t dS = tmem_base + (uint32_t)s * BN;
        for (int kc = 0; kc < 2; ++kc) {
          const uint64_t da = desc_kmajor_sw128(sbase + kQOff + kc * 16384);
          const uint64_t db = desc_kmajor_sw128(sbase + kKOff + ks * kTileBytes + kc * 16384);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // +32 bytes of K per instruction
            umma_bf16(dS, da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2), idS, (kc | kk) != 0);
        }
        umma_commit(&k_empty[ks]);  // the key stage is free once these MMAs have read it
        umma_commit(&s_full[s]);
      };
      if (nt > 0) issue_s(0);
      if (ok && nt > 1) issue_s(1);
      int t = 0;  // local tile index
      for (; t < nt && ok; ++t) {
        const int s = t & 1;
        const uint32_t ph = (uint32_t)(t >> 1) & 1u;
        if (!wait_or_abort(&p_full[s], ph, abort_flag) || !wait_or_abort(&v_full[s], ph, abort_flag) ||
            !wait_or_abort(&pv_empty[s], ph ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dPV = tmem_base + (uint32_t)(2 + s) * BN;  // two accumulators in turn
        const uint32_t aP = tmem_base + (uint32_t)s * BN;         // P_t: keys 2c, 2c+1 in column c
#pragma unroll
        for (int j = 0; j < BN / 16; ++j) {
          const int key0 = j * 16;  // 16 keys per instruction: eight columns of P, two 8-row groups of V
          const uint64_t db = desc_mnmajor_sw128(sbase + kVOff + s * kTileBytes + key0 * 128, 16384, 1024);
          umma_bf16_ts(dPV, aP + (uint32_t)(j * 8), db, idPV, j != 0);
        }
        umma_commit(&v_empty[s]);
        umma_commit(&pv_full[s]);
        if (t + 2 < nt) issue_s(t + 2);
      }
      if (!ok) set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
      // every MMA issued completes before tensor memory or the stages go away
      umma_commit(mma_done);
      if (!mbar_wait(mma_done, 0)) set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
    }
    if constexpr (CL > 1) {  // the merge's two cluster barriers
      __syncwarp();
      cluster_sync();
      cluster_sync();
    }
  } else {
    // ---------------- softmax: two threads per query row (its tensor-memory
    // lane); each owns 64 of a tile's keys and 64 of the output columns
    const int g = warp & 3;          // this warp may read lanes 32g .. 32g+31
    const int hh = (warp - 2) >> 2;  // key half of S_t, column half of PV_t
    const int r = 32 * g + lane;
    const uint32_t trow = tmem_base + ((uint32_t)(32 * g) << 16) + (uint32_t)(hh * 64);
    const uint32_t* myanc = ancs + r * kMaxWords;
    float o[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) o[j] = 0.f;
    float m = -INFINITY, l = 0.f, a_prev = 1.f;
    bool ok = true;
    // PV_j folded into the output: o = o * alpha_j + PV_j
    auto fold = [&](int j, float alpha) {
      uint32_t v[64];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld_32x32b_x16(trow + (uint32_t)((2 + (j & 1)) * BN + q * 16), v + q * 16);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 64; i += 2) fma2(o[i], o[i + 1], alpha, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
      tc_fence_before();
      mbar_arrive(&pv_empty[j & 1]);
    };
    int t = 0;  // local tile index: key tile t_begin + t
    for (; t < nt; ++t) {
      const int s = t & 1;
      const uint32_t ph = (uint32_t)(t >> 1) & 1u;
      const bool got = wait_or_abort(&s_full[s], ph, abort_flag);
      if (__any_sync(0xffffffffu, !got)) { ok = false; break; }
      __syncwarp();
      tc_fence_after();
      const int key0 = (t_begin + t) * BN + hh * 64;
      // this thread's visible keys as 64 bits: prefix keys always, tree node
      // n = j - L when it is an ancestor-or-self of the row, nothing past the keys
      uint32_t vm[2];
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const int j0 = key0 + 32 * w;
        uint32_t bits = 0u;
        if (j0 + 32 <= L) {
          bits = 0xffffffffu;
        } else if (j0 < nkeys) {
          const int n0 = j0 - L;  // tree node of bit 0 (negative: prefix keys first)
          if (n0 >= 0) {
            const int q = n0 >> 5, sh = n0 & 31;
            const uint32_t lo = myanc[q], hi = q + 1 < kMaxWords ? myanc[q + 1] : 0u;
            bits = sh ? (lo >> sh) | (hi << (32 - sh)) : lo;
          } else {
            bits = (0xffffffffu >> (32 + n0)) | (myanc[0] << (-n0));  // -n0 prefix keys, then nodes 0..
          }
          const int past = nkeys - j0;  // keys past the sequence read nothing
          if (past < 32) bits &= (1u << past) - 1u;
        }
        vm[w] = bits;
      }
      uint32_t v[64];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld_32x32b_x16(trow + (uint32_t)(s * BN + q * 16), v + q * 16);
      tmem_ld_wait();
      // hidden keys become -inf (2^-inf = 0 below); most tiles hide nothing
      if (!__all_sync(0xffffffffu, (vm[0] & vm[1]) == 0xffffffffu)) {
#pragma unroll
        for (int i = 0; i < 64; ++i) v[i] = ((vm[i >> 5] >> (i & 31)) & 1u) ? v[i] : 0xff800000u;
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < 64; ++i) mx[i & 3] = fmaxf(mx[i & 3], __uint_as_float(v[i]));
      // the row's tile maximum from both halves
      xmax[((t & 1) * 2 + hh) * BMR + r] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      mbar_arrive(&xm_full[s]);
      const bool xgot = wait_or_abort(&xm_full[s], ph, abort_flag);
      if (__any_sync(0xffffffffu, !xgot)) { ok = false; break; }
      const float mt = fmaxf(xmax[((t & 1) * 2 + hh) * BMR + r], xmax[((t & 1) * 2 + (hh ^ 1)) * BMR + r]);
      const float mn = fmaxf(m, mt);
      const float base = mn == -INFINITY ? 0.f : mn;
      const float alpha = exp2f(m - base);  // 0 while nothing was visible
      // p = 2^(s - max) as bf16 pairs over this thread's half of S_t in
      // tensor memory (columns hh*32 .. hh*32+31 of accumulator t & 1: every
      // thread has read its S_t before the row-max exchange above), and its
      // sum (pairs of lanes in f32x2)
      float sa[2] = {0.f, 0.f}, sb[2] = {0.f, 0.f};
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {  // 32 keys, 16 columns at a time
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float x0 = __uint_as_float(v[32 * hq + 2 * i]), x1 = __uint_as_float(v[32 * hq + 2 * i + 1]);
          add2(x0, x1, -base, -base);
          const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);
          add2(sa[i & 1], sb[i & 1], p0, p1);
          pk[i] = pack2_bf16(p0, p1);
        }
        tmem_st_32x32b_x16(tmem_base + ((uint32_t)(32 * g) << 16) + (uint32_t)(s * BN + hh * 32 + hq * 16), pk);
      }
      tmem_st_wait();
      l = l * alpha + ((sa[0] + sb[0]) + (sa[1] + sb[1]));
      m = mn;
      // the last tile's value rows past the sequence's keys are zeroed (their
      // p is 0, but the rows hold whatever the cache has there)
      if ((t_begin + t) * BN + BN > nkeys && (t_begin + t) * BN + r >= nkeys) {
        if (wait_or_abort(&v_full[s], ph, abort_flag)) {
          const uint32_t vrow = sbase + kVOff + s * kTileBytes + (uint32_t)hh * 16384 + r * 128;
          for (int c = 0; c < 8; ++c) st_shared_v4(vrow + c * 16, make_uint4(0, 0, 0, 0));
        }
      }
      fence_async_smem();  // zeroed V rows are read by the tensor cores
      tc_fence_before();
      mbar_arrive(&p_full[s]);
      // PV_{t-1} folds in while PV_t runs (it normally has completed: it was
      // issued a tile's softmax ago)
      if (t > 0) {
        const bool pgot = wait_or_abort(&pv_full[(t - 1) & 1], (uint32_t)((t - 1) >> 1) & 1u, abort_flag);
        if (__any_sync(0xffffffffu, !pgot)) { ok = false; break; }
        __syncwarp();
        tc_fence_after();
        fold(t - 1, a_prev);
      }
      a_prev = alpha;
    }
    if (ok && nt > 0) {
      const int j = nt - 1;
      const bool pgot = wait_or_abort(&pv_full[j & 1], (uint32_t)(j >> 1) & 1u, abort_flag);
      if (__any_sync(0xffffffffu, !pgot)) {
        ok = false;
      } else {
        __syncwarp();
        tc_fence_after();
        fold(j, a_prev);
      }
    }
    // the row's sum from both halves
    if (ok) {
      const int s = nt & 1;
      xmax[(s * 2 + hh) * BMR + r] = l;
      mbar_arrive(&xm_full[s]);
      const bool lgot = wait_or_abort(&xm_full[s], (uint32_t)(nt >> 1) & 1u, abort_flag);
      if (__any_sync(0xffffffffu, !lgot)) ok = false;
      else l += xmax[(s * 2 + (hh ^ 1)) * BMR + r];
    }
    if (!ok && lane == 0) set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
    const bool live = r < nlive;
    if constexpr (CL == 1) {
      if (live) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint16_t* dst = a.out + (((int64_t)b * a.T + row0 + r) * a.H + h) * DH + hh * 64;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(dst + c * 8) = make_uint4(
              pack2_bf16(o[c * 8] * inv, o[c * 8 + 1] * inv), pack2_bf16(o[c * 8 + 2] * inv, o[c * 8 + 3] * inv),
              pack2_bf16(o[c * 8 + 4] * inv, o[c * 8 + 5] * inv), pack2_bf16(o[c * 8 + 6] * inv, o[c * 8 + 7] * inv));
      }
    } else {
      // the cluster's CTAs hold partials (max m_c, sum l_c, O_c) over disjoint
      // key runs; CTA c finalises output columns c*CW .. c*CW+CW-1:
      //   O = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c,  M = max_c m_c
      // Each partial goes to its own CTA's key/value stages (free: the last
      // PV has completed) and is read from there by the other CTAs.
      if (live) {
        const uint32_t row = sbase + kPartOff + (uint32_t)(r * kPartStride + hh * 64) * 4;
#pragma unroll
        for (int k = 0; k < 16; ++k) st_shared_f4(row + k * 16, o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
        if (hh == 0) st_shared_f2(sbase + kMlOff + r * 8, m, l);
      }
      __syncwarp();
      cluster_sync();  // every partial is in place
      constexpr int CW = DH / CL, tpr = CW / 8;  // columns per CTA; threads per row, 8 columns each
      const int u = tid - 64;
      for (int rr = u / tpr; rr < nlive; rr += kSoftThreads / tpr) {
        const int col = crank * CW + (u % tpr) * 8;
        float pm[CL], pl[CL];
#pragma unroll
        for (int c = 0; c < CL; ++c) {
          const float2 t = ld_cluster_f2(cluster_map(sbase + kMlOff + rr * 8, (uint32_t)c));
          pm[c] = t.x;
          pl[c] = t.y;
        }
        float mmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < CL; ++c) mmax = fmaxf(mmax, pm[c]);
        float lsum = 0.f;
#pragma unroll
        for (int c = 0; c < CL; ++c) {
          pm[c] = pm[c] == -INFINITY ? 0.f : exp2f(pm[c] - mmax);  // the partial's weight
          lsum += pm[c] * pl[c];
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        float acc[8];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {  // four columns at a time: every partial's loads in flight
          float4 x[CL];
#pragma unroll
          for (int c = 0; c < CL; ++c)
            x[c] = ld_cluster_f4(
                cluster_map(sbase + kPartOff + (uint32_t)(rr * kPartStride + col + hf * 4) * 4, (uint32_t)c));
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
          for (int c = 0; c < CL; ++c) {
            s0 += pm[c] * x[c].x; s1 += pm[c] * x[c].y; s2 += pm[c] * x[c].z; s3 += pm[c] * x[c].w;
          }
          acc[hf * 4] = s0; acc[hf * 4 + 1] = s1; acc[hf * 4 + 2] = s2; acc[hf * 4 + 3] = s3;
        }
        uint16_t* dst = a.out + (((int64_t)b * a.T + row0 + rr) * a.H + h) * DH + col;
        *reinterpret_cast<uint4*>(dst) =
            make_uint4(pack2_bf16(acc[0] * inv, acc[1] * inv), pack2_bf16(acc[2] * inv, acc[3] * inv),
                       pack2_bf16(acc[4] * inv, acc[5] * inv), pack2_bf16(acc[6] * inv, acc[7] * inv));
      }
      __syncwarp();
      cluster_sync();  // no CTA leaves while its partial may still be read
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ host --

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

// The cache [rows][H * 128] bf16 as tiles of 128 rows x 64 values, 128-byte
// swizzle; rows past the cache read zeros.
bool make_cache_map(CUtensorMap* m, const void* base, int64_t rows, int H) {
  EncodeTiled enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)H * DH, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)H * DH * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)BN};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int CL>
void launch_tc(dim3 grid, size_t smem, cudaStream_t s, const CUtensorMap& tmK, const CUtensorMap& tmV,
               const AttnTcArgs& a) {
  cudaFuncSetAttribute(attn_tc_kernel<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_kernel(attn_tc_kernel<CL>, grid, dim3(kThreads), smem, s, tmK, tmV, a);
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" int medusa_tree_attn_tc(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                   void* v_cache, int64_t cache_rows, const int64_t* seq_start,
                                   const int32_t* prefix_len, const int64_t* seq_cap, const medusa_tree_t* tree,
                                   int B, int H, int Dh, int max_prefix, float rope_theta, float scale,
                                   medusa_dtype dtype, void* out, int key_splits, int32_t* err, void* stream) {
  const char* fn = "medusa_tree_attn_tc";
  if (key_splits != 1 && key_splits != 2 && key_splits != 4 && key_splits != 8)
    return fail(MEDUSA_ERR_UNSUPPORTED, "%s: key_splits=%d not in {1,2,4,8}", fn, key_splits);
  if (int rc = check_tree(tree, fn)) return rc;
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !seq_start || !prefix_len || !seq_cap || !out)
    return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (B < 1 || B > MEDUSA_MAX_B || H < 1 || max_prefix < 0 || cache_rows < 1)
    return fail(MEDUSA_ERR_INVALID, "%s: bad B=%d H=%d max_prefix=%d cache_rows=%lld", fn, B, H, max_prefix,
                (long long)cache_rows);
  if (dtype != MEDUSA_BF16) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: bf16 only", fn);
  if (Dh != DH) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: Dh=%d (the tensor-core path takes 128)", fn, Dh);
  if (tree->K > MEDUSA_MAX_K) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: tree depth %d", fn, tree->K);
  if (!(rope_theta > 0.f) || !(scale > 0.f)) return fail(MEDUSA_ERR_INVALID, "%s: rope_theta/scale", fn);
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
       reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
       reinterpret_cast<uintptr_t>(out)) % 16)
    return fail(MEDUSA_ERR_INVALID, "%s: tensors not 16-byte aligned", fn);
  AttnTcArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.k_cache = static_cast<uint16_t*>(k_cache);
  a.v_cache = static_cast<uint16_t*>(v_cache);
  a.seq_start = seq_start; a.prefix_len = prefix_len; a.seq_cap = seq_cap;
  a.depth = tree->depth; a.anc = tree->anc_mask; a.T = tree->T; a.W = tree->W; a.K = tree->K;
  a.B = B; a.H = H; a.max_prefix = max_prefix;
  a.rowblocks = (tree->T + BMR - 1) / BMR;
  for (int j = 0; j < DH / 2; ++j) a.inv_freq[j] = (float)(1.0 / std::pow((double)rope_theta, (2.0 * j) / (double)DH));
  a.qscale = scale * kLog2e;
  a.out = static_cast<uint16_t*>(out);
  a.err = err;
  CUtensorMap tmK, tmV;
  if (!make_cache_map(&tmK, k_cache, cache_rows, H) || !make_cache_map(&tmV, v_cache, cache_rows, H))
    return fail(MEDUSA_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed", fn);
  const size_t smem = 1024 + kCsOff + (size_t)2 * (tree->K + 1) * (DH / 2) * 4;
  const dim3 grid(key_splits, H, B * a.rowblocks);
  switch (key_splits) {  // the key_splits CTAs of a (sequence, head, row block) form one cluster
    case 1: launch_tc<1>(grid, smem, as_stream(stream), tmK, tmV, a); break;
    case 2: launch_tc<2>(grid, smem, as_stream(stream), tmK, tmV, a); break;
    case 4: launch_tc<4>(grid, smem, as_stream(stream), tmK, tmV, a); break;
    default: launch_tc<8>(grid, smem, as_stream(stream), tmK, tmV, a); break;
  }
  return check_launch(fn);
}
