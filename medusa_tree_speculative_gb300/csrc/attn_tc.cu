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
//   * warp 0 (one thread) loads key and value tiles with TMA into two rings
//     of two stages;
//   * warp 1 allocates tensor memory and one thread issues the MMAs:
//     S_t = Q K_t^T (M = 128 query rows, N = 128 keys, K = 128) into one of
//     two S accumulators, two tiles ahead, and PV_t = P_t V_t (N = 128 value
//     columns, K = 128 keys; V is read in its cache layout, keys x values,
//     as an MN-major operand) into a third accumulator;
//   * warps 2-5 own one query row per thread (its tensor-memory lane): read
//     S_t, mask it (keys past the sequence; tree keys that are not an
//     ancestor-or-self of the row), update the running max, write
//     P_t = 2^(S - max) in bf16 to shared memory for the PV MMA, and fold
//     PV_t into the row's output registers with the online-softmax rescale.
// Every mbarrier wait is bounded; a wait that gives up sets
// MEDUSA_DEVERR_TIMEOUT, lets the copies in flight land, frees tensor memory
// and returns.
#include <cuda.h>
#include <math.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace medusa {
namespace {

using namespace sm100;

constexpr int DH = 128;        // head dimension (two 64-wide swizzle spans)
constexpr int BN = 128;        // keys per tile (MMA N of S, K of PV)
constexpr int BMR = 128;       // query rows per CTA (MMA M)
constexpr int kThreads = 192;  // warp 0 loads, warp 1 MMAs, warps 2-5 softmax
constexpr int kMaxWords = (MEDUSA_MAX_T + 31) / 32;
constexpr float kLog2e = 1.4426950408889634f;

// Shared memory (1024-byte aligned regions).
constexpr uint32_t kQOff = 0;                    // Q   [2 k-chunks][128 rows][128 B]
constexpr uint32_t kPOff = 32768;                // P   [2 k-chunks][128 rows][128 B]
constexpr uint32_t kKOff = 65536;                // K   [2 stages][2 k-chunks][128 keys][128 B]
constexpr uint32_t kVOff = 131072;               // V   [2 stages][2 column halves][128 keys][128 B]
constexpr uint32_t kTileBytes = 32768;           // one K or V tile
constexpr uint32_t kBarOff = 196608;             // mbarriers, tensor-memory slot, flags
constexpr uint32_t kAncOff = kBarOff + 256;      // ancestor words [128 rows][kMaxWords]
constexpr uint32_t kCsOff = kAncOff + BMR * kMaxWords * 4;  // cos / sin [K+1][64] each
constexpr uint32_t kTmemCols = 512;              // S0, S1, PV (128 columns each)

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

MDEV void st_shared_v4(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ AttnTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* k_full = bars;       // [2] TMA -> MMA
  uint64_t* k_empty = bars + 2;  // [2] MMA -> TMA
  uint64_t* v_full = bars + 4;   // [2]
  uint64_t* v_empty = bars + 6;  // [2]
  uint64_t* s_full = bars + 8;   // [2] MMA -> softmax: S_t ready
  uint64_t* s_empty = bars + 10; // [2] softmax -> MMA: S buffer read (128 arrivals)
  uint64_t* p_full = bars + 12;  // softmax -> MMA: P_t written (128 arrivals)
  uint64_t* pv_full = bars + 13; // MMA -> softmax: PV_t ready
  uint64_t* pv_empty = bars + 14;// softmax -> MMA: PV accumulator read (128 arrivals)
  uint64_t* mma_done = bars + 15;// every MMA issued so far has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  int* s_abort = reinterpret_cast<int*>(bars + 17);
  uint32_t* ancs = reinterpret_cast<uint32_t*>(smem + kAncOff);
  float* cs = reinterpret_cast<float*>(smem + kCsOff);
  float* sn = cs + (a.K + 1) * (DH / 2);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, b = blockIdx.z / a.rowblocks, rb = blockIdx.z % a.rowblocks;
  const int row0 = rb * BMR;
  int L;
  int64_t st;
  if (!seq_ok(a, b, L, st)) {  // the whole CTA leaves before any barrier or allocation
    if (h == 0 && rb == 0 && tid == 0) set_err(a.err, MEDUSA_DEVERR_CAPACITY);
    return;
  }
  const int nkeys = L + a.T, ntiles = (nkeys + BN - 1) / BN;
  const int HD = a.H * DH;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(pv_full, 1);
    mbar_init(pv_empty, 128);
    mbar_init(mma_done, 1);
    fence_barrier_init();
    *s_abort = 0;
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
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
  __syncthreads();
  // the tree's keys (rotated at L + depth) and values into the cache at slot
  // L + i; every row block of the sequence writes the same bytes
  for (int e = tid; e < a.T * 8; e += kThreads) {
    const int i = e >> 3, c = e & 7;  // node, 16-byte chunk of the first half
    const int64_t src = (((int64_t)b * a.T + i) * a.H + h) * DH;
    const int64_t dst = (st + L + i) * HD + (int64_t)h * DH;
    const int d = min(max(__ldg(a.depth + i), 0), a.K);
    uint4 klo, khi;
    rope8(ldg_v4(a.k_new + src + c * 8), ldg_v4(a.k_new + src + 64 + c * 8), cs + d * 64 + c * 8,
          sn + d * 64 + c * 8, 1.f, klo, khi);
    *reinterpret_cast<uint4*>(a.k_cache + dst + c * 8) = klo;
    *reinterpret_cast<uint4*>(a.k_cache + dst + 64 + c * 8) = khi;
    *reinterpret_cast<uint4*>(a.v_cache + dst + c * 8) = ldg_v4(a.v_new + src + c * 8);
    *reinterpret_cast<uint4*>(a.v_cache + dst + 64 + c * 8) = ldg_v4(a.v_new + src + 64 + c * 8);
  }
  fence_async_global();  // the appended rows are read back through the tensor maps
  // query rows: rotated at L + depth, times scale * log2(e), bf16, swizzled K-major
  for (int e = tid; e < BMR * 8; e += kThreads) {
    const int r = e >> 3, c = e & 7;
    const int rr = row0 + r;
    uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
    if (rr < a.T) {
      const int64_t src = (((int64_t)b * a.T + rr) * a.H + h) * DH;
      const int d = min(max(__ldg(a.depth + rr), 0), a.K);
      rope8(ldg_v4(a.q + src + c * 8), ldg_v4(a.q + src + 64 + c * 8), cs + d * 64 + c * 8, sn + d * 64 + c * 8,
            a.qscale, lo, hi);
    }
    st_shared_v4(sw128(sbase + kQOff, r, c), lo);
    st_shared_v4(sw128(sbase + kQOff + 16384, r, c), hi);
  }
  // ancestor words of this block's rows
  for (int e = tid; e < BMR * a.W; e += kThreads) {
    const int r = e / a.W, w = e % a.W;
    const int rr = row0 + r;
    ancs[r * kMaxWords + w] = rr < a.T ? __ldg(a.anc + (int64_t)rr * a.W + w) : 0u;
  }
  fence_async_smem();  // Q is read by the tensor cores
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  volatile int* abort_flag = s_abort;

  if (warp == 0) {
    // ---------------- TMA: key and value tiles, two stages each
    if (lane == 0) {
      int t = 0;
      bool ok = true;
      for (; t < ntiles && ok; ++t) {
        const int s = t & 1;
        const uint32_t ph = (uint32_t)(t >> 1) & 1u;
        const int y = (int)(st + (int64_t)t * BN);
        if (!wait_or_abort(&k_empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
        mbar_expect_tx(&k_full[s], kTileBytes);
        for (int kc = 0; kc < 2; ++kc)
          tma_load_2d(smem + kKOff + s * kTileBytes + kc * 16384, &tmK, &k_full[s], h * DH + kc * 64, y);
        if (!wait_or_abort(&v_empty[s], ph ^ 1u, abort_flag)) {
          ok = false;
          mbar_wait(&k_full[s], ph);  // the key tile issued above lands first
          break;
        }
        mbar_expect_tx(&v_full[s], kTileBytes);
        for (int kc = 0; kc < 2; ++kc)
          tma_load_2d(smem + kVOff + s * kTileBytes + kc * 16384, &tmV, &v_full[s], h * DH + kc * 64, y);
      }
      if (!ok) {
        // let the tiles already issued land before the CTA can exit
        for (int j = max(0, t - 2); j < t; ++j) {
          mbar_wait(&k_full[j & 1], (uint32_t)(j >> 1) & 1u);
          mbar_wait(&v_full[j & 1], (uint32_t)(j >> 1) & 1u);
        }
        set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(BMR, BN);
      const uint32_t idPV = idesc_bf16_f32(BMR, DH) | (1u << 16);  // B (V) MN-major
      bool ok = true;
      auto issue_s = [&](int t) {
        const int s = t & 1;
        const uint32_t ph = (uint32_t)(t >> 1) & 1u;
        if (!wait_or_abort(&k_full[s], ph, abort_flag) || !wait_or_abort(&s_empty[s], ph ^ 1u, abort_flag)) {
          ok = false;
          return;
        }
        tc_fence_after();
        const uint32_t dS = tmem_base + (uint32_t)s * BN;
        for (int kc = 0; kc < 2; ++kc) {
          const uint64_t da = desc_kmajor_sw128(sbase + kQOff + kc * 16384);
          const uint64_t db = desc_kmajor_sw128(sbase + kKOff + s * kTileBytes + kc * 16384);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // +32 bytes of K per instruction
            umma_bf16(dS, da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2), idS, (kc | kk) != 0);
        }
        umma_commit(&k_empty[s]);  // the key stage is free once these MMAs have read it
        umma_commit(&s_full[s]);
      };
      issue_s(0);
      if (ok && ntiles > 1) issue_s(1);
      int t = 0;
      for (; t < ntiles && ok; ++t) {
        const int s = t & 1;
        const uint32_t ph = (uint32_t)(t >> 1) & 1u;
        if (!wait_or_abort(p_full, (uint32_t)t & 1u, abort_flag) || !wait_or_abort(&v_full[s], ph, abort_flag) ||
            !wait_or_abort(pv_empty, ((uint32_t)t & 1u) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dPV = tmem_base + 2 * BN;
        for (int kc = 0; kc < 2; ++kc) {
          const uint64_t da = desc_kmajor_sw128(sbase + kPOff + kc * 16384);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int key0 = kc * 64 + kk * 16;  // 16 keys per instruction: two 8-row groups of V
            const uint64_t db = desc_mnmajor_sw128(sbase + kVOff + s * kTileBytes + key0 * 128, 16384, 1024);
            umma_bf16(dPV, da + (uint64_t)(kk * 2), db, idPV, (kc | kk) != 0);
          }
        }
        umma_commit(&v_empty[s]);
        umma_commit(pv_full);
        if (t + 2 < ntiles) issue_s(t + 2);
      }
      if (!ok) set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
      // every MMA issued completes before tensor memory or the stages go away
      umma_commit(mma_done);
      if (!mbar_wait(mma_done, 0)) set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
    }
  } else {
    // ---------------- softmax: one query row per thread (tensor-memory lane)
    const int g = warp & 3;  // this warp may read lanes 32g .. 32g+31
    const int r = 32 * g + lane;
    const uint32_t trow = tmem_base + ((uint32_t)(32 * g) << 16);
    const uint32_t* myanc = ancs + r * kMaxWords;
    float o[DH];
#pragma unroll
    for (int j = 0; j < DH; ++j) o[j] = 0.f;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int s = t & 1;
      const uint32_t ph = (uint32_t)(t >> 1) & 1u;
      const bool got = wait_or_abort(&s_full[s], ph, abort_flag);
      if (__any_sync(0xffffffffu, !got)) { ok = false; break; }
      __syncwarp();
      tc_fence_after();
      const int key0 = t * BN;
      // this row's visible keys of the tile as 128 bits: prefix keys always,
      // tree node n = j - L when it is an ancestor-or-self, nothing past the keys
      uint32_t vm[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
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
      // pass 1: the tile's maximum over visible keys, 64 columns per load
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
      for (int hc = 0; hc < BN / 64; ++hc) {
        const uint32_t vw[2] = {hc ? vm[2] : vm[0], hc ? vm[3] : vm[1]};
        uint32_t v[64];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld_32x32b_x16(trow + (uint32_t)(s * BN + hc * 64 + q * 16), v + q * 16);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const float x = ((vw[i >> 5] >> (i & 31)) & 1u) ? __uint_as_float(v[i]) : -INFINITY;
          mx[i & 3] = fmaxf(mx[i & 3], x);
        }
      }
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      const float mn = fmaxf(m, mt);
      const float base = mn == -INFINITY ? 0.f : mn;
      const float alpha = exp2f(m - base);  // 0 while nothing was visible
      // pass 2: p = 2^(s - max) into P (bf16, swizzled K-major), and its sum
      float sm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int hc = 0; hc < BN / 64; ++hc) {
        const uint32_t vw[2] = {hc ? vm[2] : vm[0], hc ? vm[3] : vm[1]};
        uint32_t v[64];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld_32x32b_x16(trow + (uint32_t)(s * BN + hc * 64 + q * 16), v + q * 16);
        tmem_ld_wait();
        const uint32_t region = sbase + kPOff + (uint32_t)hc * 16384;  // keys hc*64 .. hc*64+63
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {  // 16-byte chunks of the 128-byte row: 8 keys each
          float p[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int k = ch * 8 + i;
            const float x = __uint_as_float(v[k]) - base;
            p[i] = ((vw[k >> 5] >> (k & 31)) & 1u) ? exp2f(x) : 0.f;
            sm[i & 3] += p[i];
          }
          st_shared_v4(sw128(region, r, ch), make_uint4(pack2_bf16(p[0], p[1]), pack2_bf16(p[2], p[3]),
                                                         pack2_bf16(p[4], p[5]), pack2_bf16(p[6], p[7])));
        }
      }
      const float ls = (sm[0] + sm[1]) + (sm[2] + sm[3]);
      l = l * alpha + ls;
      m = mn;
      // the last tile's value rows past the sequence's keys are zeroed (their
      // p is 0, but the rows hold whatever the cache has there)
      if (key0 + BN > nkeys && key0 + r >= nkeys) {
        const bool vgot = wait_or_abort(&v_full[s], ph, abort_flag);
        if (vgot) {
          const uint4 z = make_uint4(0, 0, 0, 0);
          for (int c = 0; c < 8; ++c) {
            st_shared_v4(sbase + kVOff + s * kTileBytes + r * 128 + c * 16, z);
            st_shared_v4(sbase + kVOff + s * kTileBytes + 16384 + r * 128 + c * 16, z);
          }
        }
      }
      fence_async_smem();  // P (and zeroed V rows) are read by the tensor cores
      tc_fence_before();
      mbar_arrive(&s_empty[s]);
      mbar_arrive(p_full);
      // PV_t folded into the output with the rescale of the running max
      const bool pgot = wait_or_abort(pv_full, (uint32_t)t & 1u, abort_flag);
      if (__any_sync(0xffffffffu, !pgot)) { ok = false; break; }
      __syncwarp();
      tc_fence_after();
#pragma unroll
      for (int hc = 0; hc < DH / 64; ++hc) {
        uint32_t v[64];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld_32x32b_x16(trow + (uint32_t)(2 * BN + hc * 64 + q * 16), v + q * 16);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 64; ++i) o[hc * 64 + i] = o[hc * 64 + i] * alpha + __uint_as_float(v[i]);
      }
      tc_fence_before();
      mbar_arrive(pv_empty);
    }
    if (!ok) {
      if (lane == 0) set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
    } else if (row0 + r < a.T) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint16_t* dst = a.out + (((int64_t)b * a.T + row0 + r) * a.H + h) * DH;
#pragma unroll
      for (int c = 0; c < DH / 8; ++c)
        *reinterpret_cast<uint4*>(dst + c * 8) =
            make_uint4(pack2_bf16(o[c * 8] * inv, o[c * 8 + 1] * inv), pack2_bf16(o[c * 8 + 2] * inv, o[c * 8 + 3] * inv),
                       pack2_bf16(o[c * 8 + 4] * inv, o[c * 8 + 5] * inv), pack2_bf16(o[c * 8 + 6] * inv, o[c * 8 + 7] * inv));
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

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" int medusa_tree_attn_tc(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                   void* v_cache, int64_t cache_rows, const int64_t* seq_start,
                                   const int32_t* prefix_len, const int64_t* seq_cap, const medusa_tree_t* tree,
                                   int B, int H, int Dh, int max_prefix, float rope_theta, float scale,
                                   medusa_dtype dtype, void* out, int32_t* err, void* stream) {
  const char* fn = "medusa_tree_attn_tc";
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
  cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_kernel(attn_tc_kernel, dim3(1, H, B * a.rowblocks), dim3(kThreads), smem, as_stream(stream), tmK, tmV, a);
  return check_launch(fn);
}
