// Verification LM head over every flattened tree row.
//
// "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
// Heads", Method 3 and the decoding-step box (step 3): the backbone runs once
// over all tree nodes, so the LM head produces logits for every node;
// decoding is memory-bound ("Problem"): the vocabulary matrix is read once per
// step and dominates the bytes.
//
// logits[r][v] = sum_j hidden[r][j] * w[v][j]
//
// bf16: tcgen05 tensor-core GEMM with TMEM accumulators, swap-AB: the
// vocabulary is the MMA's M dimension (128-row tiles of W, K-major) and the
// tree rows its N dimension (all rows of a chunk, padded to 16, K-major), so
// one instruction covers every tree row.  When the vocabulary has more tiles
// than there are SMs, a work item is a pair of adjacent tiles that share each
// hidden k-block (halving the L2->SM traffic per weight byte).  Persistent
// CTAs, balanced to the same number of work items each, own contiguous runs
// of the vocabulary: each weight byte is read once and no partial sums are
// exchanged.  Warp roles:
//   warp 0     one thread issues TMA loads of W and hidden k-blocks (64 wide,
//              128-byte swizzle) into a ring of shared stages,
//   warp 1     allocates TMEM; one thread issues the MMAs (4 per stage) and
//              commits stage releases and finished accumulators to mbarriers,
//   warps 2-5  read the accumulator back from TMEM (one TMEM lane per
//              vocabulary row) and store fp32 logits, coalesced along the
//              vocabulary.
// Two accumulators alternate so the epilogue of one tile overlaps the MMAs of
// the next.  W is read in 128 x 64 boxes: from a row-major matrix each box is
// 128 separate 128-byte runs; from the tiled layout (medusa_lm_head_tile) it
// is one contiguous 16 KB run, which keeps HBM pages open and measured about
// 9% faster for the 32000 x 4096 matrix.  Every mbarrier wait is bounded; a timeout sets
// MEDUSA_DEVERR_TIMEOUT and the kernel winds down.
// The same kernel, with a second epilogue, computes the Medusa heads' first
// projection for every tree row (medusa_heads_hidden; Method 1, "heads over
// all rows"): M runs over the stacked W1 rows of the heads in use and each
// accumulator becomes u = bf16(SiLU(acc + b1) + h); the residual values are
// staged in shared memory by the idle epilogue warps during the main loop.
// From 129 to 256 tree rows the logits run on CTA pairs instead
// (lm_head_pair_kernel, tcgen05 cta_group::2): one MMA of M = 256 covers a
// vocabulary tile of each CTA, and each CTA loads half of the hidden rows.
// f32: plain CUDA-core kernels (one warp per output element).
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "cluster.cuh"
#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"
#include "stats.cuh"

namespace medusa {
namespace {

using namespace sm100;

constexpr int BM = 128;        // vocabulary rows per tile (MMA M)
constexpr int BK = 64;         // k per stage: 128 bytes of bf16, one swizzle span
constexpr int UK = 16;         // k per MMA instruction
constexpr int kThreads = 192;  // 6 warps
constexpr int kMaxN = 256;     // tree rows per chunk (MMA N)
constexpr int kMaxTiles = 4;   // weight tiles per work item (sharing each hidden k-block)
constexpr size_t kSmemBudget = 200 * 1024;
constexpr int kMaxXRows = 8;   // rows past 256 formed by the epilogue warps (XROWS plan): one mma.sync N

struct LmArgs {
  float* logits;
  int rows, d, V;
  int npad;     // MMA N of every chunk (multiple of 16, <= kMaxN)
  int cpi;      // row chunks per work item: they share each weight k-block (more than kMaxN rows)
  int ncol;     // accumulator columns per weight tile = cpi * npad (tree rows r0 .. r0 + ncol)
  int nacc;     // accumulators in TMEM: 2 (the epilogue of one item overlaps the next) or 1
  int nchunks;  // work items along the tree rows (each cpi chunks)
  int nt;       // vocabulary tiles per work item (1 or 2): they share each hidden k-block
  int ngroups;  // work items along the vocabulary = ceil(tiles / nt)
  int stages;
  uint32_t tmem_cols;
  int tiled;      // W in the 128 x 64 tile layout (each box one contiguous 16 KB run)
  int ntiles;     // valid 128-row tiles along M
  int oob_block;  // a weight block index past the tensor (its loads read zeros)
  // epilogue: mode 0 stores fp32 logits [rows][V]; mode 1 is the Medusa-head
  // projection u[r][k][j] = bf16(SiLU(acc + b1[k][j]) + hidden[r][j]) for the
  // stacked rows of the used heads (M = nused * d)
  int mode;
  const uint16_t* hidden;
  const uint16_t* b1;
  uint16_t* u;
  int K;                        // heads in u's layout
  int tpr;                      // 128-row tiles per head (d / 128)
  int32_t heads[MEDUSA_MAX_K];  // slot -> head id
  // mode 0, acceptance statistics (fused epilogue): per (vocabulary group,
  // row) a record {max logit, its index (lowest on ties), and for typical
  // acceptance sum e^(y-m), sum e^(y-m)(y-m) with y = logit * inv_temp,
  // m = max y}; stat_mode 0 none, 1 argmax, 2 argmax + softmax sums
  float4* stats;
  int stat_mode;
  float inv_temp;
  int write_logits;
  uint32_t part_off;  // byte offset of the per-warp partial records in shared memory
  // joint launch (LM head and the heads' first projection in one pass over
  // the same hidden k-blocks): CTA c owns vocabulary tiles [c*lm_tiles/G,
  // (c+1)*lm_tiles/G) of W and stacked W1 tiles [c*w1_tiles/G, ...) of the
  // second map, G = gridDim.x; mode 0 epilogue on the former (V rows), mode 1
  // on the latter (Vu = used heads * d rows)
  int lm_tiles, w1_tiles, tiled1, Vu;
  // rows past one 256-row chunk (1 .. kMaxXRows; lm_head_tc_kernel<.., .., true>):
  // their hidden k-block sits at byte xr_off of each stage and the epilogue
  // warps form their logits on the CUDA cores from the same weight stage
  int xr;
  uint32_t xr_off;
  int32_t* err;
};

// ---- acceptance statistics (records and their merge: stats.cuh)

template <bool TYP>
MDEV StatRec rec_shfl(const StatRec& x, int mask) {
  StatRec r;
  r.v = __shfl_xor_sync(0xffffffffu, x.v, mask);
  r.i = __shfl_xor_sync(0xffffffffu, x.i, mask);
  r.S = TYP ? __shfl_xor_sync(0xffffffffu, x.S, mask) : 0.f;
  r.A = TYP ? __shfl_xor_sync(0xffffffffu, x.A, mask) : 0.f;
  return r;
}

// One halving step of the transpose-reduce: lanes with (lane & D) keep the
// upper half of their N records and send the lower half to lane ^ D.
template <bool TYP, int N, int D>
MDEV void tr_step(StatRec (&x)[16], int lane, float inv_temp) {
  const bool hi = lane & D;
#pragma unroll
  for (int j = 0; j < N / 2; ++j) {
    const StatRec keep = hi ? x[j + N / 2] : x[j];
    const StatRec send = hi ? x[j] : x[j + N / 2];
    x[j] = stat_merge<TYP>(keep, rec_shfl<TYP>(send, D), inv_temp);
  }
}

// 32 lanes x 16 columns -> each column reduced over the 32 lanes; lane L (and
// L ^ 1) ends with column 8 b4 + 4 b3 + 2 b2 + b1 of L's bits.  16 shuffles
// per field instead of 80 for column-by-column butterflies.
template <bool TYP>
MDEV StatRec transpose_reduce(StatRec (&x)[16], int lane, float inv_temp) {
  tr_step<TYP, 16, 16>(x, lane, inv_temp);
  tr_step<TYP, 8, 8>(x, lane, inv_temp);
  tr_step<TYP, 4, 4>(x, lane, inv_temp);
  tr_step<TYP, 2, 2>(x, lane, inv_temp);
  return stat_merge<TYP>(x[0], rec_shfl<TYP>(x[0], 1), inv_temp);
}
// ldmatrix: four (two) 8x8 bf16 matrices, lane l giving the address of row
// l % 8 of matrix l / 8.
MDEV void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
MDEV void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];\n" : "=r"(r0), "=r"(r1) : "r"(addr));
}

MDEV uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

MDEV int tr_column(int lane) {
  return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}

// Named barrier 1 over the four epilogue warps, OR-reducing a predicate.
MDEV bool epilogue_any(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)p)
      : "memory");
  return r != 0;
}
MDEV void epilogue_sync() { asm volatile("bar.sync 1, 128;\n" ::: "memory"); }

struct HeadSlots {
  int32_t id[MEDUSA_MAX_K];
};

// Weight block (128 rows) that M-tile `tile` reads.
MDEV int weight_block(const LmArgs& a, int tile) {
  if (tile >= a.ntiles) return a.oob_block;
  if (a.mode == 0) return tile;
  return a.heads[tile / a.tpr] * a.tpr + tile % a.tpr;
}

// Where tile t of a work item comes from and how its epilogue runs.
struct TileSrc {
  int sel;   // 0: the W map, 1: the W1 map (joint launch)
  int blk;   // 128-row weight block in that map (a.oob_block: past the tensor, reads zeros)
  int mode;  // epilogue: 0 logits, 1 head projection u, -1 none (padding tile)
  int v0;    // first output row of the tile (vocabulary row, or stacked W1 row)
  int rs;    // residual slot of a mode-1 tile
};
template <bool JOINT>
MDEV TileSrc tile_src(const LmArgs& a, int item, int t) {
  if (!JOINT) {
    const int tile = (item / a.nchunks) * a.nt + t;
    return TileSrc{0, weight_block(a, tile), a.mode, tile * BM, t};
  }
  const int G = (int)gridDim.x;
  const int l0 = (int)((int64_t)item * a.lm_tiles / G), l1 = (int)((int64_t)(item + 1) * a.lm_tiles / G);
  const int w0 = (int)((int64_t)item * a.w1_tiles / G), w1 = (int)((int64_t)(item + 1) * a.w1_tiles / G);
  if (t < l1 - l0) return TileSrc{0, l0 + t, 0, (l0 + t) * BM, 0};
  const int k = t - (l1 - l0);
  if (k < w1 - w0) {
    const int tile = w0 + k;
    return TileSrc{1, a.heads[tile / a.tpr] * a.tpr + tile % a.tpr, 1, tile * BM, k};
  }
  return TileSrc{0, a.oob_block, -1, 0, 0};
}

MDEV bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 255 && *abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

// STATS: the epilogue also produces the acceptance statistics (a separate
// instantiation, so that the plain path keeps its registers and barriers).
// JOINT: one work item per CTA mixing W and W1 tiles (tile_src).
// XROWS: 257 .. 256 + kMaxXRows rows: one 256-row chunk on the tensor cores
// and the a.xr rows past it on the CUDA cores of the epilogue warps, which
// read each weight stage too (the third map is then the extra rows' hidden).
template <bool STATS, bool JOINT, bool XROWS = false>
__global__ void __launch_bounds__(kThreads, 1)
    lm_head_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                      const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ LmArgs a) {
  static_assert(!(STATS && JOINT), "the joint launch has no statistics epilogue");
  static_assert(!(XROWS && (STATS || JOINT)), "extra rows: plain logits only");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t a_bytes = (uint32_t)a.nt * BM * BK * 2;  // nt W tiles, 16 KB each
  const uint32_t b_bytes = (uint32_t)a.ncol * BK * 2;
  const uint32_t stage_bytes = a_bytes + b_bytes + (XROWS ? 16u * BK * 2 : 0u);  // XROWS: a 16-row box at xr_off
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)a.stages * stage_bytes);
  uint64_t* empty = full + a.stages;
  uint64_t* tfull = empty + a.stages;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  // mode 1: the residual tile hidden[r0 + i][j] of the current item, [nt][ncol][128] bf16
  uint16_t* res = reinterpret_cast<uint16_t*>(smem + (size_t)a.stages * stage_bytes + 1024);
  // acceptance statistics: partial records [nt][4 warps][ncol]
  float4* part = reinterpret_cast<float4*>(smem + a.part_off);
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], XROWS ? 1 + 4 : 1);  // XROWS: the MMAs and the four epilogue warps read it
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4 * 32);
    }
    fence_barrier_init();
    s_abort = 0;
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmH);
    if (JOINT || XROWS) tma_prefetch_desc(&tmW1);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  volatile int* abort_flag = &s_abort;

  const int items = JOINT ? (int)gridDim.x : a.ngroups * a.nchunks;
  const uint32_t acc_cols = (uint32_t)(a.nt * a.ncol);  // one accumulator: nt tiles side by side
  const int i0 = (int)((long)blockIdx.x * items / gridDim.x);
  const int i1 = (int)((long)(blockIdx.x + 1) * items / gridDim.x);
  const int nkb = a.d / BK;

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int item = i0; item < i1 && ok; ++item) {
        const int r0 = (item % a.nchunks) * a.ncol;
        // weight blocks of the item's tiles (rows past V, a missing tile, read zeros)
        int blk[kMaxTiles], sel[kMaxTiles];
        for (int t = 0; t < a.nt; ++t) {
          const TileSrc ts = tile_src<JOINT>(a, item, t);
          blk[t] = ts.blk;
          sel[t] = ts.sel;
        }
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % a.stages;
          const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
          if (!wait_or_abort(&empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
          uint8_t* st = smem + (size_t)s * stage_bytes;
          mbar_expect_tx(&full[s], stage_bytes);
          for (int t = 0; t < a.nt; ++t) {
            const CUtensorMap* m = JOINT && sel[t] ? &tmW1 : &tmW;
            if (JOINT && sel[t] ? a.tiled1 : a.tiled)
              tma_load_2d(st + t * (BM * BK * 2), m, &full[s], 0, (blk[t] * nkb + kb) * BM);
            else
              tma_load_2d(st + t * (BM * BK * 2), m, &full[s], kb * BK, blk[t] * BM);
          }
          if (a.cpi == 1)
            tma_load_2d(st + a_bytes, &tmH, &full[s], kb * BK, r0);
          else
            for (int c = 0; c < a.cpi; ++c)  // the item's row chunks (rows past the last read zeros)
              tma_load_2d(st + a_bytes + c * (a.npad * BK * 2), &tmH, &full[s], kb * BK, r0 + c * a.npad);
          if (XROWS) tma_load_2d(st + a.xr_off, &tmW1, &full[s], kb * BK, a.npad);  // the rows past the chunk
        }
      }
      if (!ok) {
        // let the loads already issued land before the CTA can exit
        for (int j = max(0, it - a.stages); j < it; ++j)
          mbar_wait(&full[j % a.stages], (uint32_t)(j / a.stages) & 1u);
        set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, a.npad);
      int it = 0, local = 0;
      bool ok = true;
      for (int item = i0; item < i1 && ok; ++item, ++local) {
        const int acc = a.nacc == 2 ? local & 1 : 0;
        const uint32_t aph = (uint32_t)(a.nacc == 2 ? local >> 1 : local) & 1u;
        if (!wait_or_abort(&tempty[acc], aph ^ 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)acc * acc_cols;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % a.stages;
          const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
          if (!wait_or_abort(&full[s], ph, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + (size_t)s * stage_bytes);
          if (a.cpi == 1) {
            const uint64_t db = desc_kmajor_sw128(sa + a_bytes);
            for (int t = 0; t < a.nt; ++t) {
              const uint64_t da = desc_kmajor_sw128(sa + t * (BM * BK * 2));
#pragma unroll
              for (int kk = 0; kk < BK / UK; ++kk)  // +32 bytes of K per instruction
                umma_bf16(d_tmem + (uint32_t)(t * a.npad), da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2),
                          idesc, (kb | kk) != 0);
            }
          } else if (a.cpi == 2) {  // two row chunks against the same weight block
            const uint64_t db0 = desc_kmajor_sw128(sa + a_bytes);
            const uint64_t db1 = desc_kmajor_sw128(sa + a_bytes + a.npad * BK * 2);
            for (int t = 0; t < a.nt; ++t) {
              const uint64_t da = desc_kmajor_sw128(sa + t * (BM * BK * 2));
              const uint32_t d0 = d_tmem + (uint32_t)(t * a.ncol);
#pragma unroll
              for (int kk = 0; kk < BK / UK; ++kk)
                umma_bf16(d0, da + (uint64_t)(kk * 2), db0 + (uint64_t)(kk * 2), idesc, (kb | kk) != 0);
#pragma unroll
              for (int kk = 0; kk < BK / UK; ++kk)
                umma_bf16(d0 + (uint32_t)a.npad, da + (uint64_t)(kk * 2), db1 + (uint64_t)(kk * 2), idesc,
                          (kb | kk) != 0);
            }
          } else {
            for (int t = 0; t < a.nt; ++t) {
              const uint64_t da = desc_kmajor_sw128(sa + t * (BM * BK * 2));
              for (int c = 0; c < a.cpi; ++c) {  // every row chunk against the same weight block
                const uint64_t db = desc_kmajor_sw128(sa + a_bytes + c * (a.npad * BK * 2));
#pragma unroll
                for (int kk = 0; kk < BK / UK; ++kk)  // +32 bytes of K per instruction
                  umma_bf16(d_tmem + (uint32_t)(t * a.ncol + c * a.npad), da + (uint64_t)(kk * 2),
                            db + (uint64_t)(kk * 2), idesc, (kb | kk) != 0);
              }
            }
          }
          umma_commit(&empty[s]);  // the stage is free once these MMAs have read it
        }
        if (ok) umma_commit(&tfull[acc]);  // accumulator complete
      }
      if (!ok) {
        if (it > 0) mbar_wait(&empty[(it - 1) % a.stages], (uint32_t)((it - 1) / a.stages) & 1u);
        set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
      }
    }
  } else {
    // ---------------- epilogue: TMEM -> registers -> logits
    const int g = warp & 3;  // this warp may read TMEM lanes 32g .. 32g+31
    // mode 1: the residual values this thread will need, staged in shared
    // memory while the main loop runs (loads issued after the weight stream
    // has saturated HBM would each wait out the loaded latency)
    const int u_rows = JOINT ? a.Vu : a.V;  // stacked W1 rows of the used heads
    auto load_res = [&](int item) {
      const int r0 = (item % a.nchunks) * a.ncol;
      for (int t = 0; t < a.nt; ++t) {
        const TileSrc ts = tile_src<JOINT>(a, item, t);
        if (ts.mode != 1) continue;
        const int v = ts.v0 + 32 * g + lane;
        const int j = v % a.d;
        for (int i0 = 0; i0 < a.ncol; i0 += 16) {  // 16 loads in flight, then 16 stores
          uint16_t hv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int row = r0 + i0 + i;
            hv[i] = (v < u_rows && row < a.rows) ? __ldg(a.hidden + (int64_t)row * a.d + j) : (uint16_t)0;
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) res[(ts.rs * a.ncol + i0 + i) * BM + 32 * g + lane] = hv[i];
        }
      }
    };
    if ((JOINT || a.mode == 1) && i0 < i1) load_res(i0);
    int local = 0, xit = 0;
    for (int item = i0; item < i1; ++item, ++local) {
      const int acc = a.nacc == 2 ? local & 1 : 0;
      const uint32_t aph = (uint32_t)(a.nacc == 2 ? local >> 1 : local) & 1u;
      // XROWS: the rows past the chunk (up to eight, N of an mma.sync
      // m16n8k16) against this warp's 64 weight rows (four 16-row blocks of
      // tile g / 2), k-block by k-block beside the MMAs; each stage is
      // released by the four warps and the MMAs.  Operands come from the
      // stage by ldmatrix, the 128-byte swizzle undone in the row addresses
      // (16-byte chunk c of a row r at chunk c ^ (r & 7)).
      float xc[4][4];
      if constexpr (XROWS) {
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int q = 0; q < 4; ++q) xc[m][q] = 0.f;
        const int xt = g >> 1, xrow0 = (g & 1) * 64;  // this warp's tile and first row in it
        const int lr = lane & 7, lm = lane >> 3;      // row in an 8x8 matrix, which matrix
        bool xok = true;
        for (int kb = 0; kb < nkb; ++kb, ++xit) {
          const int s = xit % a.stages;
          const bool xgot = wait_or_abort(&full[s], (uint32_t)(xit / a.stages) & 1u, abort_flag);
          if (__any_sync(0xffffffffu, !xgot)) { xok = false; break; }
          const uint32_t st = smem_u32(smem + (size_t)s * stage_bytes);
          if (xt < a.nt) {
            const uint32_t wb = st + (uint32_t)xt * (BM * BK * 2), hb = st + a.xr_off;
#pragma unroll
            for (int ks = 0; ks < BK / UK; ++ks) {
              uint32_t b0, b1;  // extra rows lr, k chunk 2 ks + (lm & 1)
              const int bch = 2 * ks + (lm & 1);
              ldsm_x2(hb + lr * 128 + ((bch ^ lr) << 4), b0, b1);
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                const int ar = xrow0 + m * 16 + (lm & 1) * 8 + lr, ach = 2 * ks + (lm >> 1);
                uint32_t af[4];
                ldsm_x4(wb + ar * 128 + ((ach ^ (ar & 7)) << 4), af);
                mma_bf16_16816(xc[m], af, b0, b1);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (!xok) {
          if (lane == 0) set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
          break;
        }
      }
      const bool got = wait_or_abort(&tfull[acc], aph, abort_flag);
      // with statistics the four warps share named barriers, so they take one decision
      if (STATS ? epilogue_any(!got) : __any_sync(0xffffffffu, !got)) {
        if (lane == 0) set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
        break;
      }
      __syncwarp();
      tc_fence_after();
      const int r0 = (item % a.nchunks) * a.ncol;
      for (int t = 0; t < a.nt; ++t) {
        const TileSrc ts = tile_src<JOINT>(a, item, t);
        if (JOINT && ts.mode < 0) continue;  // padding tile: nothing to store
        const int v = ts.v0 + 32 * g + lane;
        const int tmode = JOINT ? ts.mode : a.mode;
        for (int c = 0; c < a.ncol / 16; ++c) {  // column c * 16 + i holds tree row r0 + c * 16 + i
          uint32_t r[16];
          tmem_ld_32x32b_x16(tmem_base + ((uint32_t)(32 * g) << 16) + (uint32_t)acc * acc_cols +
                                 (uint32_t)(t * a.ncol + c * 16),
                             r);
          tmem_ld_wait();
          if (STATS) {  // this warp's 32 vocabulary rows reduced per column
            StatRec x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const bool valid = v < a.V && r0 + c * 16 + i < a.rows;
              x[i].v = valid ? __uint_as_float(r[i]) : -INFINITY;
              x[i].i = v;
              x[i].S = valid ? 1.f : 0.f;
              x[i].A = 0.f;
            }
            const StatRec red = a.stat_mode == 2 ? transpose_reduce<true>(x, lane, a.inv_temp)
                                             : transpose_reduce<false>(x, lane, a.inv_temp);
            if (!(lane & 1))
              part[(t * 4 + g) * a.ncol + c * 16 + tr_column(lane)] =
                  make_float4(red.v, __int_as_float(red.i), red.S, red.A);
          }
          if (v < (tmode == 0 ? a.V : u_rows)) {
            if (tmode == 0) {
              if (a.write_logits) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const int row = r0 + c * 16 + i;
                  if (row < a.rows) a.logits[(int64_t)row * a.V + v] = __uint_as_float(r[i]);
                }
              }
            } else {
              const int slot = v / a.d, j = v % a.d, k = a.heads[slot];
              const float bias = a.b1 ? bf16_bits_to_f32(__ldg(a.b1 + (int64_t)k * a.d + j)) : 0.f;
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int row = r0 + c * 16 + i;
                if (row < a.rows) {
                  const float y = __uint_as_float(r[i]) + bias;
                  const float silu = y / (1.f + expf(-y));
                  const float h = bf16_bits_to_f32(res[(ts.rs * a.ncol + c * 16 + i) * BM + 32 * g + lane]);
                  a.u[((int64_t)row * a.K + k) * a.d + j] = f32_to_bf16_bits(silu + h);
                }
              }
            }
          }
        }
      }
      if constexpr (XROWS) {  // C fragment: (row lane / 4 [+ 8], extra row 2 (lane % 4) [+ 1])
        const int xt = g >> 1;
        if (xt < a.nt) {
          const int v0 = tile_src<JOINT>(a, item, xt).v0 + (g & 1) * 64 + (lane >> 2);
#pragma unroll
          for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int v = v0 + m * 16 + (q >> 1) * 8, j = 2 * (lane & 3) + (q & 1);
              const int row = r0 + a.npad + j;
              if (j < a.xr && row < a.rows && v < a.V) a.logits[(int64_t)row * a.V + v] = xc[m][q];
            }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (STATS) {  // the item's record per row: merge the warps' and tiles' partials in a fixed order
        epilogue_sync();
        const int group = item / a.nchunks;
        for (int e = threadIdx.x - 64; e < a.ncol; e += 128) {
          StatRec m = stat_empty();
          for (int q = 0; q < a.nt * 4; ++q) {
            const StatRec y = stat_load(part[q * a.ncol + e]);
            m = a.stat_mode == 2 ? stat_merge<true>(m, y, a.inv_temp) : stat_merge<false>(m, y, a.inv_temp);
          }
          if (r0 + e < a.rows)
            a.stats[(int64_t)group * a.rows + r0 + e] = make_float4(m.v, __int_as_float(m.i), m.S, m.A);
        }
        epilogue_sync();
      }
      if ((JOINT || a.mode == 1) && item + 1 < i1) {
        __syncwarp();
        load_res(item + 1);  // this warp's own slice of the tile: no other warp reads it
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

// ---- the same GEMM on CTA pairs (tcgen05 cta_group::2), logits only
//
// Each cluster of two CTAs owns runs of work items of 2 * nt vocabulary
// tiles; one MMA of M = 256 covers a tile of each CTA (tile (group * nt + j)
// * 2 + rank) against all of a row chunk, whose hidden k-block is split
// between the two CTAs' stages (the first npad / 2 rows in the even CTA, the
// rest in the odd one).  So each SM pulls half of every hidden k-block where
// the one-CTA kernel pulls all of it: with more tree rows than a weight tile
// has (256 and more), the hidden k-blocks are most of what an SM loads, and
// what one SM can pull into shared memory bounds the call.
//   warp 0     (both CTAs) TMA: its weight tiles and its half of each row
//              chunk into its own stage; completion is counted on the even
//              CTA's `full` barrier, which expects both CTAs' bytes;
//   warp 1     (both CTAs) allocates the pair's tensor memory; in the even
//              CTA one thread issues the MMAs and commits stage releases and
//              finished accumulators to the barriers of both CTAs;
//   warps 2-5  (both CTAs) read their own tensor memory (their 128
//              vocabulary rows) and store the logits; each warp then arrives
//              on the even CTA's `tempty`.
// Every wait is bounded; a CTA that gave up waits 20 us for its copies in
// flight before the closing cluster barrier, after which the tensor memory
// is freed.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    lm_head_pair_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                        const __grid_constant__ LmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t rank = cluster_rank();            // 0: the CTA that issues the MMAs
  const int hrows = a.npad / 2;                    // rows of a chunk this CTA holds
  const uint32_t a_bytes = (uint32_t)a.nt * BM * BK * 2;
  const uint32_t h_bytes = (uint32_t)hrows * BK * 2;  // one chunk's half k-block
  const uint32_t stage_bytes = a_bytes + (uint32_t)a.cpi * h_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)a.stages * stage_bytes);
  uint64_t* empty = full + a.stages;
  uint64_t* tfull = empty + a.stages;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);   // the even CTA's expect_tx; both CTAs' bytes
      mbar_init(&empty[s], 1);  // the pair MMAs that read the stage
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 2 * 4);  // one arrival per epilogue warp of either CTA
    }
    mbar_init(mma_done, 1);
    fence_barrier_init();
    s_abort = 0;
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmH);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, a.tmem_cols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers initialised, the pair's tensor memory allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  volatile int* abort_flag = &s_abort;

  const int items = a.ngroups * a.nchunks;
  const int pairs = (int)gridDim.x / 2, pair = (int)blockIdx.x / 2;
  const int i0 = (int)((long)pair * items / pairs), i1 = (int)((long)(pair + 1) * items / pairs);
  const uint32_t acc_cols = (uint32_t)(a.nt * a.ncol);
  const int nkb = a.d / BK;

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs)
    if (lane == 0) {
      const uint32_t full0 = cluster_map(smem_u32(full), 0);  // the even CTA's `full` barriers
      int it = 0;
      bool ok = true;
      for (int item = i0; item < i1 && ok; ++item) {
        const int r0 = (item % a.nchunks) * a.ncol;
        int blk[2];
        for (int j = 0; j < a.nt; ++j) blk[j] = weight_block(a, ((item / a.nchunks) * a.nt + j) * 2 + (int)rank);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % a.stages;
          const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
          if (!wait_or_abort(&empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
          uint8_t* st = smem + (size_t)s * stage_bytes;
          if (rank == 0) mbar_expect_tx(&full[s], 2 * stage_bytes);
          const uint32_t bar = full0 + (uint32_t)s * 8u;
          for (int j = 0; j < a.nt; ++j) {
            if (a.tiled)
              tma_load_2d_pair(st + j * (BM * BK * 2), &tmW, bar, 0, (blk[j] * nkb + kb) * BM);
            else
              tma_load_2d_pair(st + j * (BM * BK * 2), &tmW, bar, kb * BK, blk[j] * BM);
          }
          for (int c = 0; c < a.cpi; ++c)  // this CTA's half of each row chunk (rows past the last read zeros)
            tma_load_2d_pair(st + a_bytes + c * h_bytes, &tmH, bar, kb * BK, r0 + c * a.npad + (int)rank * hrows);
        }
      }
      if (!ok) set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (even CTA)
    if (rank == 0 && lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(2 * BM, a.npad);
      int it = 0, local = 0;
      bool ok = true;
      for (int item = i0; item < i1 && ok; ++item, ++local) {
        const int acc = a.nacc == 2 ? local & 1 : 0;
        const uint32_t aph = (uint32_t)(a.nacc == 2 ? local >> 1 : local) & 1u;
        bool got = false;  // both CTAs' epilogues have drained the accumulator
        for (uint32_t i = 0; i < kSpinLimit && !got; ++i) {
          got = mbar_try_wait_cluster(&tempty[acc], aph ^ 1u);
          if (!got && (i & 255) == 255 && *abort_flag) break;
        }
        if (!got) { *abort_flag = 1; ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)acc * acc_cols;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % a.stages;
          const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
          if (!wait_or_abort(&full[s], ph, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + (size_t)s * stage_bytes);
          for (int j = 0; j < a.nt; ++j) {
            const uint64_t da = desc_kmajor_sw128(sa + j * (BM * BK * 2));
            for (int c = 0; c < a.cpi; ++c) {
              const uint64_t db = desc_kmajor_sw128(sa + a_bytes + c * h_bytes);
#pragma unroll
              for (int kk = 0; kk < BK / UK; ++kk)  // +32 bytes of K per instruction
                umma_bf16_pair(d_tmem + (uint32_t)(j * a.ncol + c * a.npad), da + (uint64_t)(kk * 2),
                               db + (uint64_t)(kk * 2), idesc, (kb | kk) != 0);
            }
          }
          umma_commit_pair_mc(&empty[s], 0x3);  // both CTAs' stages are free once these MMAs have read them
        }
        if (ok) umma_commit_pair_mc(&tfull[acc], 0x3);  // both halves of the accumulator complete
      }
      if (!ok) set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
      // every MMA issued completes before either CTA's stages or tensor memory go away
      umma_commit_pair(mma_done);
      if (!mbar_wait(mma_done, 0)) set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
    }
  } else {
    // ---------------- epilogue (both CTAs): TMEM -> registers -> logits
    const int g = warp & 3;  // this warp may read TMEM lanes 32g .. 32g+31
    const uint32_t tempty0 = cluster_map(smem_u32(tempty), 0);
    int local = 0;
    for (int item = i0; item < i1; ++item, ++local) {
      const int acc = a.nacc == 2 ? local & 1 : 0;
      const uint32_t aph = (uint32_t)(a.nacc == 2 ? local >> 1 : local) & 1u;
      const bool got = wait_or_abort(&tfull[acc], aph, abort_flag);
      if (__any_sync(0xffffffffu, !got)) {
        if (lane == 0) set_err(a.err, MEDUSA_DEVERR_TIMEOUT);
        break;
      }
      __syncwarp();
      tc_fence_after();
      const int r0 = (item % a.nchunks) * a.ncol;
      for (int j = 0; j < a.nt; ++j) {
        const int v = (((item / a.nchunks) * a.nt + j) * 2 + (int)rank) * BM + 32 * g + lane;
        for (int c = 0; c < a.ncol / 16; ++c) {  // column c * 16 + i holds tree row r0 + c * 16 + i
          uint32_t r[16];
          tmem_ld_32x32b_x16(tmem_base + ((uint32_t)(32 * g) << 16) + (uint32_t)acc * acc_cols +
                                 (uint32_t)(j * a.ncol + c * 16),
                             r);
          tmem_ld_wait();
          if (v < a.V) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int row = r0 + c * 16 + i;
              if (row < a.rows) a.logits[(int64_t)row * a.V + v] = __uint_as_float(r[i]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0 + (uint32_t)acc * 8u);
    }
  }
  __syncwarp();
  if (threadIdx.x == 0 && *abort_flag) {
    // a wait gave up: let the copies this CTA issued land before the pair can exit
    uint64_t t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    do {
      __nanosleep(1000);
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    } while (t - t0 < 20000);
  }
  __syncwarp();
  tc_fence_before();
  cluster_sync();  // no CTA leaves while the pair's MMAs or the other CTA may still use its memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, a.tmem_cols);
  }
}

// Row-major [V][d] -> 128 x 64 tiles (16 bytes per thread, grid-stride);
// rows past V in the last tile are written as zeros.
__global__ void __launch_bounds__(256) lm_head_tile_kernel(const uint16_t* __restrict__ w,
                                                           uint16_t* __restrict__ out, int d, int V,
                                                           int64_t chunks) {
  const int nkb = d / BK;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < chunks;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int c8 = (int)(g & 7);
    const int r = (int)((g >> 3) & (BM - 1));
    const int64_t tk = g >> 10;  // tile index: vocabulary block * nkb + column block
    const int kb = (int)(tk % nkb);
    const int64_t v = (tk / nkb) * BM + r;
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (v < V) x = ldg_stream(w + v * d + kb * BK + c8 * 8);
    reinterpret_cast<uint4*>(out)[g] = x;
  }
}

// f32: one warp per logit; lanes split the hidden dimension.
__global__ void __launch_bounds__(256) lm_head_f32_kernel(const float* hidden, const float* w,
                                                          float* logits, int rows, int d, int V) {
  const int64_t g = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (g >= (int64_t)rows * V) return;
  const int r = (int)(g / V), v = (int)(g % V);
  const float* h = hidden + (int64_t)r * d;
  const float* wr = w + (int64_t)v * d;
  float acc = 0.f;
  for (int j = lane; j < d; j += 32) acc += h[j] * wr[j];
  acc = warp_sum(acc);
  if (lane == 0) logits[(int64_t)r * V + v] = acc;
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
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

// Row-major bf16 matrix [outer][inner] -> tiles of box_outer rows x 64
// columns, 128-byte swizzle, zero fill outside the matrix.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  EncodeTiled enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_lm_head_workspace_size(int rows, int d, int V) {
  (void)rows; (void)d; (void)V;
  return 0;
}

extern "C" size_t medusa_lm_head_tiled_bytes(int d, int V) {
  if (d < 1 || V < 1 || d % BK) return 0;
  return (size_t)((V + BM - 1) / BM) * BM * (size_t)d * 2;
}

extern "C" int medusa_lm_head_tile(const void* w_lm, void* w_tiled, int d, int V, void* stream) {
  const char* fn = "medusa_lm_head_tile";
  if (!w_lm || !w_tiled) return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (d < 1 || V < 1) return fail(MEDUSA_ERR_INVALID, "%s: d=%d V=%d", fn, d, V);
  if (d % BK) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: d=%d not a multiple of %d", fn, d, BK);
  if ((reinterpret_cast<uintptr_t>(w_lm) | reinterpret_cast<uintptr_t>(w_tiled)) % 16)
    return fail(MEDUSA_ERR_INVALID, "%s: w_lm / w_tiled not 16-byte aligned", fn);
  const size_t nbytes = medusa_lm_head_tiled_bytes(d, V);
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(w_lm), b0 = reinterpret_cast<uintptr_t>(w_tiled);
  if (a0 < b0 + nbytes && b0 < a0 + (size_t)V * d * 2)
    return fail(MEDUSA_ERR_INVALID, "%s: w_tiled overlaps w_lm", fn);
  const int64_t chunks = (int64_t)(nbytes / 16);
  const int grid = (int)std::min<int64_t>((chunks + 255) / 256, (int64_t)sm_count() * 8);
  launch_kernel(lm_head_tile_kernel, dim3(grid), dim3(256), 0, as_stream(stream),
                static_cast<const uint16_t*>(w_lm), static_cast<uint16_t*>(w_tiled), d, V, chunks);
  return check_launch(fn);
}

namespace medusa {
namespace {

// Map of a weight matrix with `wrows` rows of d: row-major, or its tile copy
// (then a [blocks * (d / 64) * 128][64] matrix whose 128-row boxes are the tiles).
bool make_weight_map(CUtensorMap* m, const void* w, bool tiled, int64_t wrows, int d) {
  const int64_t wblocks = (wrows + BM - 1) / BM;
  return tiled ? make_map(m, w, (uint64_t)BK, (uint64_t)wblocks * BM * (d / BK), BM)
               : make_map(m, w, (uint64_t)d, (uint64_t)wrows, BM);
}

// Plan and launch the tensor-core GEMM: `a` carries the epilogue fields; the
// weight tensor has `wrows` rows of d (row-major) or is its tile copy.
// Work plan: the tree rows in MMA column chunks of at most kMaxN (padded to
// 16); as many chunks per work item (cpi) as one accumulator of 512 TMEM
// columns holds, so that more than kMaxN rows still read each weight block
// once; and whether a work item is one tile or two adjacent tiles sharing
// each hidden k-block (nt = 2 halves the hidden re-reads per weight byte,
// while one accumulator of both tiles fits in TMEM and there are more tiles
// than SMs).  The shared-memory ring must keep at least three stages (two
// for the smallest plan), counting the residual tile of the heads'
// projection (mode 1) and the partial records of the statistics epilogue;
// where it would not, fewer chunks or tiles share an item.
struct LmPlan {
  int nchunks, npad, cpi, ncol, nt, nacc, ngroups, stages;
  size_t stage_bytes, res_bytes, part_bytes;
};
LmPlan plan_tc(int rows, int ntiles, bool mode1, bool stats) {
  LmPlan p{};
  const int nct = (rows + kMaxN - 1) / kMaxN;
  p.npad = ((rows + nct - 1) / nct + 15) / 16 * 16;
  for (int cpi = std::max(1, std::min(nct, 512 / p.npad)); cpi >= 1; --cpi) {
    for (int nt = 2; nt >= 1; --nt) {
      if (nt == 2 && !(2 * cpi * p.npad <= 512 && ntiles > sm_count())) continue;
      p.cpi = cpi;
      p.nt = nt;
      p.ncol = cpi * p.npad;
      p.stage_bytes = (size_t)nt * BM * BK * 2 + (size_t)p.ncol * BK * 2;
      p.res_bytes = mode1 ? (size_t)nt * p.ncol * BM * 2 : 0;
      p.part_bytes = stats ? (size_t)nt * 4 * p.ncol * 16 : 0;
      const size_t fixed = 1024 + 256 + p.res_bytes + p.part_bytes;
      p.stages = kSmemBudget > fixed ? (int)std::min<size_t>(8, (kSmemBudget - fixed) / p.stage_bytes) : 0;
      if (p.stages >= 3 || (p.stages >= 2 && cpi == 1 && nt == 1)) {
        p.nchunks = (nct + cpi - 1) / cpi;
        p.nacc = 2 * nt * p.ncol <= 512 ? 2 : 1;  // a second accumulator where it fits
        p.ngroups = (ntiles + nt - 1) / nt;
        return p;
      }
    }
  }
  p.stages = 0;  // nothing fits
  return p;
}

// Pair plan (lm_head_pair_kernel): as plan_tc, with each CTA's stage holding
// its nt weight tiles and half of every row chunk's hidden k-block.
LmPlan plan_pair(int rows, int ntiles) {
  LmPlan p{};
  const int nct = (rows + kMaxN - 1) / kMaxN;
  p.npad = ((rows + nct - 1) / nct + 15) / 16 * 16;
  for (int cpi = std::max(1, std::min(nct, 512 / p.npad)); cpi >= 1; --cpi) {
    for (int nt = 2; nt >= 1; --nt) {
      if (nt == 2 && !(2 * cpi * p.npad <= 512 && ntiles > sm_count())) continue;
      p.cpi = cpi;
      p.nt = nt;
      p.ncol = cpi * p.npad;
      p.stage_bytes = (size_t)nt * BM * BK * 2 + (size_t)cpi * (p.npad / 2) * BK * 2;
      p.stages = (int)std::min<size_t>(8, (kSmemBudget - 1024 - 256) / p.stage_bytes);
      if (p.stages >= 3) {
        p.nchunks = (nct + cpi - 1) / cpi;
        p.nacc = 2 * nt * p.ncol <= 512 ? 2 : 1;
        p.ngroups = (ntiles + 2 * nt - 1) / (2 * nt);
        return p;
      }
    }
  }
  p.stages = 0;
  return p;
}

// The pair kernel serves plain logits for one row chunk of more than 128
// rows, where it measured faster (256 rows: 63.5 against 66.0 us at d = 4096,
// 90.1 against 94.5 us at d = 6656).  Below that, and with two chunks, it is
// not: a pair MMA of M = 256 takes longer than an M = 128 one on each SM,
// which gives back what the halved hidden k-blocks save (257 rows: 94.2
// against 92.4 us; one row: 51.2 against 45.8 us).
constexpr int kPairMinRows = 129;

bool use_pair(const LmArgs& a, int rows) {
  return a.mode == 0 && a.stat_mode == 0 && rows >= kPairMinRows && rows <= kMaxN &&
         plan_pair(rows, a.ntiles).stages >= 3;
}

// CTA pairs that can run at once with one CTA per SM (a GPC with an odd
// number of SMs leaves one idle), cached per device; half the SMs if the
// query fails.
int pair_slots() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return std::max(1, sm_count() / 2);
  if (cached[dev] > 0) return cached[dev];
  const int smem = 1024 + (int)kSmemBudget;  // enough to hold one CTA per SM
  int n = 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(2 * std::max(1, sm_count() / 2)));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaFuncSetAttribute(lm_head_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, lm_head_pair_kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();  // clear a failed query
    n = std::max(1, sm_count() / 2);
  }
  cached[dev] = std::min(n, std::max(1, sm_count() / 2));
  return cached[dev];
}

// Clusters of the pair plan, each CTA of a cluster with the same number of
// work items (ceil or floor of items / pairs).
int pair_grid(const LmPlan& p) {
  const int items = p.ngroups * p.nchunks, npairs = pair_slots();
  const int per_pair = (items + npairs - 1) / npairs;
  return 2 * ((items + per_pair - 1) / per_pair);
}

int launch_pair(LmArgs& a, const void* w, bool tiled, int64_t wrows, const void* hidden, int rows, int d,
                cudaStream_t s, const char* fn) {
  a.rows = rows; a.d = d; a.tiled = tiled;
  const LmPlan p = plan_pair(rows, a.ntiles);
  a.nchunks = p.nchunks; a.npad = p.npad; a.cpi = p.cpi; a.ncol = p.ncol;
  a.nt = p.nt; a.nacc = p.nacc; a.ngroups = p.ngroups; a.stages = p.stages;
  uint32_t cols = 32;
  while (cols < (uint32_t)(a.nacc * a.nt * a.ncol)) cols <<= 1;
  a.tmem_cols = cols;
  a.oob_block = (int)((wrows + BM - 1) / BM);
  CUtensorMap tmW, tmH;
  if (!make_weight_map(&tmW, w, tiled, wrows, d) ||
      !make_map(&tmH, hidden, (uint64_t)d, (uint64_t)rows, (uint32_t)(a.npad / 2)))
    return fail(MEDUSA_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed", fn);
  const size_t smem = 1024 + (size_t)a.stages * p.stage_bytes + 256;  // ring | barriers, tensor-memory slot
  cudaFuncSetAttribute(lm_head_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_kernel(lm_head_pair_kernel, dim3(pair_grid(p)), dim3(kThreads), smem, s, tmW, tmH, a);
  return check_launch(fn);
}

// Extra-rows plan (lm_head_tc_kernel<false, false, true>): 257 .. 256 +
// kMaxXRows rows as one 256-row chunk, so that every weight k-block takes
// four MMAs per tile where two chunks of 144 rows took eight (the MMAs
// bounded the two-chunk call: an instruction of M = 128 costs about the same
// at N = 144 as at N = 256), and the rows past it on the CUDA cores of the
// epilogue warps, which read each weight stage beside the MMAs with
// ldmatrix + mma.sync (eight extra rows are one N = 8 fragment).
struct XPlan {
  int nt, stages, grid;
  size_t stage_bytes;
};
XPlan plan_xrows(int ntiles) {
  XPlan p{};
  p.nt = ntiles > sm_count() ? 2 : 1;  // two tiles on one 512-column accumulator share each hidden k-block
  p.stage_bytes = (size_t)p.nt * BM * BK * 2 + (size_t)kMaxN * BK * 2 + 16 * BK * 2;
  p.stages = (int)std::min<size_t>(8, (kSmemBudget - 1024 - 256) / p.stage_bytes);
  const int items = (ntiles + p.nt - 1) / p.nt;
  const int per_cta = (items + sm_count() - 1) / sm_count();
  p.grid = (items + per_cta - 1) / per_cta;
  return p;
}

bool use_xrows(const LmArgs& a, int rows) {
  return a.mode == 0 && a.stat_mode == 0 && rows > kMaxN && rows <= kMaxN + kMaxXRows &&
         plan_xrows(a.ntiles).stages >= 3;
}

int launch_xrows(LmArgs& a, const void* w, bool tiled, int64_t wrows, const void* hidden, int rows, int d,
                 cudaStream_t s, const char* fn) {
  const XPlan p = plan_xrows(a.ntiles);
  a.rows = rows; a.d = d; a.tiled = tiled;
  a.npad = kMaxN; a.cpi = 1; a.ncol = kMaxN; a.nchunks = 1;
  a.nt = p.nt; a.nacc = 1; a.stages = p.stages;
  a.ngroups = (a.ntiles + a.nt - 1) / a.nt;
  a.xr = rows - kMaxN;
  a.xr_off = (uint32_t)((size_t)a.nt * BM * BK * 2 + (size_t)kMaxN * BK * 2);
  a.part_off = (uint32_t)align_up((size_t)a.stages * p.stage_bytes + 1024, 16);
  a.tmem_cols = a.nt == 2 ? 512u : 256u;
  a.oob_block = (int)((wrows + BM - 1) / BM);
  CUtensorMap tmW, tmH, tmX;
  if (!make_weight_map(&tmW, w, tiled, wrows, d) || !make_map(&tmH, hidden, (uint64_t)d, (uint64_t)rows, kMaxN) ||
      !make_map(&tmX, hidden, (uint64_t)d, (uint64_t)rows, 16))
    return fail(MEDUSA_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed", fn);
  const size_t smem = 1024 + a.part_off;
  auto kern = lm_head_tc_kernel<false, false, true>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_kernel(kern, dim3(p.grid), dim3(kThreads), smem, s, tmW, tmH, tmX, a);
  return check_launch(fn);
}

int launch_tc(LmArgs& a, const void* w, bool tiled, int64_t wrows, const void* hidden, int rows, int d,
              cudaStream_t s, const char* fn) {
  if (use_pair(a, rows)) return launch_pair(a, w, tiled, wrows, hidden, rows, d, s, fn);
  if (use_xrows(a, rows)) return launch_xrows(a, w, tiled, wrows, hidden, rows, d, s, fn);
  a.rows = rows; a.d = d; a.tiled = tiled;
  const LmPlan p = plan_tc(rows, a.ntiles, a.mode == 1, a.stat_mode != 0);
  if (p.stages < 2) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: shared memory for %d tree rows", fn, rows);
  a.nchunks = p.nchunks; a.npad = p.npad; a.cpi = p.cpi; a.ncol = p.ncol;
  a.nt = p.nt; a.nacc = p.nacc; a.ngroups = p.ngroups; a.stages = p.stages;
  const size_t stage_bytes = p.stage_bytes, res_bytes = p.res_bytes, part_bytes = p.part_bytes;
  a.part_off = (uint32_t)align_up((size_t)a.stages * stage_bytes + 1024 + res_bytes, 16);
  uint32_t cols = 32;
  while (cols < (uint32_t)(a.nacc * a.nt * a.ncol)) cols <<= 1;
  a.tmem_cols = cols;
  const int64_t wblocks = (wrows + BM - 1) / BM;
  a.oob_block = (int)wblocks;
  CUtensorMap tmW, tmH;
  if (!make_weight_map(&tmW, w, tiled, wrows, d) || !make_map(&tmH, hidden, (uint64_t)d, (uint64_t)rows, (uint32_t)a.npad))
    return fail(MEDUSA_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed", fn);
  const size_t smem = 1024 + a.part_off + part_bytes;  // ring | barriers | residuals | partial records
  auto kern = a.stat_mode ? lm_head_tc_kernel<true, false> : lm_head_tc_kernel<false, false>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  // balanced: every CTA gets ceil or floor of items / grid work items
  const int items = a.ngroups * a.nchunks;
  const int per_cta = (items + sm_count() - 1) / sm_count();
  const int grid = (items + per_cta - 1) / per_cta;
  launch_kernel(kern, dim3(grid), dim3(kThreads), smem, s, tmW, tmH, tmW, a);
  return check_launch(fn);
}

// Joint plan: the fewest CTAs (at most one per SM) whose shares of the W and
// W1 tiles add up to at most nt tiles, for the smallest nt that has one.
// Fewer CTAs leave SMs free for concurrent work; every CTA streams at most nt
// tiles over one shared pass of the hidden k-blocks.  False if none fits.
bool plan_joint(int lm_tiles, int w1_tiles, int npad, int& nt, int& grid) {
  for (nt = 2; nt <= kMaxTiles; ++nt) {
    if (nt * npad > 512) break;  // one accumulator of nt tiles in TMEM
    for (grid = 1; grid <= sm_count(); ++grid)
      if ((lm_tiles + grid - 1) / grid + (w1_tiles + grid - 1) / grid <= nt) return true;
  }
  return false;
}

// f32 heads projection: one warp per (row, used head, output j).
__global__ void __launch_bounds__(256) heads_hidden_f32_kernel(const float* hidden, const float* w1, const float* b1,
                                                               float* u, int rows, int d, int K, int nused,
                                                               HeadSlots hs) {
  const int64_t g = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (g >= (int64_t)rows * nused * d) return;
  const int j = (int)(g % d);
  const int slot = (int)((g / d) % nused);
  const int r = (int)(g / ((int64_t)d * nused));
  const int k = hs.id[slot];
  const float* h = hidden + (int64_t)r * d;
  const float* wr = w1 + ((int64_t)k * d + j) * d;
  float acc = 0.f;
  for (int i = lane; i < d; i += 32) acc += h[i] * wr[i];
  acc = warp_sum(acc);
  if (lane == 0) {
    const float y = acc + (b1 ? b1[(int64_t)k * d + j] : 0.f);
    u[((int64_t)r * K + k) * d + j] = y / (1.f + expf(-y)) + h[j];
  }
}

}  // namespace
}  // namespace medusa

extern "C" int medusa_lm_head_verify(const void* hidden, const void* w_lm, float* logits, int rows, int d,
                                     int V, medusa_dtype dtype, medusa_w_layout w_layout, void* workspace,
                                     size_t workspace_bytes, int32_t* err, void* stream) {
  const char* fn = "medusa_lm_head_verify";
  (void)workspace; (void)workspace_bytes;
  if (!hidden || !w_lm || !logits) return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (rows < 1 || d < 1 || V < 1) return fail(MEDUSA_ERR_INVALID, "%s: rows=%d d=%d V=%d", fn, rows, d, V);
  if (w_layout != MEDUSA_W_ROWS && w_layout != MEDUSA_W_TILES)
    return fail(MEDUSA_ERR_INVALID, "%s: w_layout=%d", fn, (int)w_layout);
  cudaStream_t s = as_stream(stream);
  if (dtype == MEDUSA_BF16) {
    if (d % BK) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: d=%d not a multiple of %d", fn, d, BK);
    if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(w_lm)) % 16)
      return fail(MEDUSA_ERR_INVALID, "%s: hidden / w_lm not 16-byte aligned", fn);
    LmArgs a{};
    a.logits = logits; a.V = V; a.err = err;
    a.mode = 0;
    a.write_logits = 1;
    a.ntiles = (V + BM - 1) / BM;
    return launch_tc(a, w_lm, w_layout == MEDUSA_W_TILES, V, hidden, rows, d, s, fn);
  }
  if (dtype != MEDUSA_F32) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: dtype", fn);
  if (w_layout != MEDUSA_W_ROWS) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: f32 takes MEDUSA_W_ROWS only", fn);
  const int64_t total = (int64_t)rows * V;
  launch_kernel(lm_head_f32_kernel, dim3((unsigned)((total + 7) / 8)), dim3(256), 0, s,
             static_cast<const float*>(hidden), static_cast<const float*>(w_lm), logits, rows, d, V);
  return check_launch(fn);
}

extern "C" int medusa_heads_hidden(const void* hidden, int rows, const void* w1, medusa_w_layout w1_layout,
                                   const void* b1, const int32_t* s_k, int K, int d, medusa_dtype dtype, void* u,
                                   int32_t* err, void* stream) {
  const char* fn = "medusa_heads_hidden";
  if (!hidden || !w1 || !s_k || !u) return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (rows < 1 || K < 1 || d < 1) return fail(MEDUSA_ERR_INVALID, "%s: rows=%d K=%d d=%d", fn, rows, K, d);
  if (K > MEDUSA_MAX_K) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: K=%d above the maximum", fn, K);
  if (w1_layout != MEDUSA_W_ROWS && w1_layout != MEDUSA_W_TILES)
    return fail(MEDUSA_ERR_INVALID, "%s: w1_layout=%d", fn, (int)w1_layout);
  HeadSlots hs{};
  int nused = 0;
  for (int k = 0; k < K; ++k) {
    if (s_k[k] < 0) return fail(MEDUSA_ERR_INVALID, "%s: s[%d]=%d", fn, k, s_k[k]);
    if (s_k[k] > 0) hs.id[nused++] = k;
  }
  if (nused == 0) return MEDUSA_OK;
  cudaStream_t s = as_stream(stream);
  if (dtype == MEDUSA_BF16) {
    if (d % BM) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: d=%d not a multiple of %d", fn, d, BM);
    if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(w1) | reinterpret_cast<uintptr_t>(u)) %
        16)
      return fail(MEDUSA_ERR_INVALID, "%s: hidden / w1 / u not 16-byte aligned", fn);
    LmArgs a{};
    a.mode = 1;
    a.V = nused * d;
    a.ntiles = nused * (d / BM);
    a.tpr = d / BM;
    a.K = K;
    for (int i = 0; i < nused; ++i) a.heads[i] = hs.id[i];
    a.hidden = static_cast<const uint16_t*>(hidden);
    a.b1 = static_cast<const uint16_t*>(b1);
    a.u = static_cast<uint16_t*>(u);
    a.err = err;
    return launch_tc(a, w1, w1_layout == MEDUSA_W_TILES, (int64_t)K * d, hidden, rows, d, s, fn);
  }
  if (dtype != MEDUSA_F32) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: dtype", fn);
  if (w1_layout != MEDUSA_W_ROWS) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: f32 takes MEDUSA_W_ROWS only", fn);
  const int64_t warps = (int64_t)rows * nused * d;
  launch_kernel(heads_hidden_f32_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s,
                static_cast<const float*>(hidden), static_cast<const float*>(w1), static_cast<const float*>(b1),
                static_cast<float*>(u), rows, d, K, nused, hs);
  return check_launch(fn);
}

extern "C" int medusa_lm_head_verify_heads_hidden(const void* hidden, int rows, int d, const void* w_lm,
                                                  medusa_w_layout w_layout, int V, float* logits, const void* w1,
                                                  medusa_w_layout w1_layout, const void* b1, const int32_t* s_k,
                                                  int K, void* u, medusa_dtype dtype, int32_t* err, void* stream) {
  const char* fn = "medusa_lm_head_verify_heads_hidden";
  if (!hidden || !w_lm || !logits || !w1 || !s_k || !u) return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (rows < 1 || d < 1 || V < 1 || K < 1)
    return fail(MEDUSA_ERR_INVALID, "%s: rows=%d d=%d V=%d K=%d", fn, rows, d, V, K);
  if (K > MEDUSA_MAX_K) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: K=%d above the maximum", fn, K);
  for (medusa_w_layout l : {w_layout, w1_layout})
    if (l != MEDUSA_W_ROWS && l != MEDUSA_W_TILES) return fail(MEDUSA_ERR_INVALID, "%s: layout=%d", fn, (int)l);
  if (dtype != MEDUSA_BF16) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: bf16 only", fn);
  if (d % BM) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: d=%d not a multiple of %d", fn, d, BM);
  if (rows > kMaxN) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: rows=%d above %d", fn, rows, kMaxN);
  if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(w_lm) | reinterpret_cast<uintptr_t>(w1) |
       reinterpret_cast<uintptr_t>(u)) % 16)
    return fail(MEDUSA_ERR_INVALID, "%s: hidden / w_lm / w1 / u not 16-byte aligned", fn);
  LmArgs a{};
  int nused = 0;
  for (int k = 0; k < K; ++k) {
    if (s_k[k] < 0) return fail(MEDUSA_ERR_INVALID, "%s: s[%d]=%d", fn, k, s_k[k]);
    if (s_k[k] > 0) a.heads[nused++] = k;
  }
  cudaStream_t s = as_stream(stream);
  if (nused == 0)
    return medusa_lm_head_verify(hidden, w_lm, logits, rows, d, V, dtype, w_layout, nullptr, 0, err, stream);
  a.logits = logits; a.V = V; a.err = err; a.rows = rows; a.d = d;
  a.mode = 0; a.write_logits = 1;
  a.hidden = static_cast<const uint16_t*>(hidden);
  a.b1 = static_cast<const uint16_t*>(b1);
  a.u = static_cast<uint16_t*>(u);
  a.K = K; a.tpr = d / BM;
  a.lm_tiles = (V + BM - 1) / BM;
  a.w1_tiles = nused * (d / BM);
  a.Vu = nused * d;
  a.tiled = w_layout == MEDUSA_W_TILES;
  a.tiled1 = w1_layout == MEDUSA_W_TILES;
  a.nchunks = 1;
  a.npad = (rows + 15) / 16 * 16;
  a.cpi = 1;
  a.ncol = a.npad;
  a.nacc = 1;  // one work item per CTA
  a.ntiles = a.lm_tiles;
  a.oob_block = a.lm_tiles;  // a block past W: its loads read zeros
  int grid = 0;
  if (!plan_joint(a.lm_tiles, a.w1_tiles, a.npad, a.nt, grid))
    return fail(MEDUSA_ERR_UNSUPPORTED, "%s: no joint plan for %d + %d tiles", fn, a.lm_tiles, a.w1_tiles);
  a.ngroups = grid;
  const size_t stage_bytes = (size_t)a.nt * BM * BK * 2 + (size_t)a.npad * BK * 2;
  const size_t res_bytes = (size_t)((a.w1_tiles + grid - 1) / grid) * a.npad * BM * 2;
  a.stages = (int)std::min<size_t>(8, (kSmemBudget - 1024 - 256 - res_bytes) / stage_bytes);
  if (a.stages < 2) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: shared memory for %d tiles", fn, a.nt);
  a.part_off = (uint32_t)align_up((size_t)a.stages * stage_bytes + 1024 + res_bytes, 16);
  uint32_t cols = 32;
  while (cols < (uint32_t)(a.nt * a.npad)) cols <<= 1;  // one accumulator: one work item per CTA
  a.tmem_cols = cols;
  CUtensorMap tmW, tmH, tmW1;
  if (!make_weight_map(&tmW, w_lm, a.tiled, V, d) || !make_weight_map(&tmW1, w1, a.tiled1, (int64_t)K * d, d) ||
      !make_map(&tmH, hidden, (uint64_t)d, (uint64_t)rows, (uint32_t)a.npad))
    return fail(MEDUSA_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed", fn);
  const size_t smem = 1024 + a.part_off;
  cudaFuncSetAttribute(lm_head_tc_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_kernel(lm_head_tc_kernel<false, true>, dim3(grid), dim3(kThreads), smem, s, tmW, tmH, tmW1, a);
  return check_launch(fn);
}

extern "C" int medusa_lm_head_ctas(int rows, int V) {
  if (rows < 1 || V < 1) return 0;
  LmArgs a{};
  a.ntiles = (V + BM - 1) / BM;
  if (use_pair(a, rows)) return pair_grid(plan_pair(rows, a.ntiles));
  if (use_xrows(a, rows)) return plan_xrows(a.ntiles).grid;
  const LmPlan p = plan_tc(rows, (V + BM - 1) / BM, false, false);
  if (p.stages < 2) return 0;
  const int items = p.ngroups * p.nchunks;
  const int per_cta = (items + sm_count() - 1) / sm_count();
  return (items + per_cta - 1) / per_cta;
}

extern "C" int medusa_lm_head_stat_groups(int rows, int V) {
  if (rows < 1 || V < 1) return 0;
  return plan_tc(rows, (V + BM - 1) / BM, false, true).ngroups;
}

extern "C" int medusa_lm_head_verify_stats(const void* hidden, const void* w_lm, float* logits, int rows, int d,
                                           int V, medusa_dtype dtype, medusa_w_layout w_layout, int mode,
                                           float temperature, void* stats, size_t stats_bytes, int32_t* err,
                                           void* stream) {
  const char* fn = "medusa_lm_head_verify_stats";
  if (!hidden || !w_lm || !stats) return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (rows < 1 || d < 1 || V < 1) return fail(MEDUSA_ERR_INVALID, "%s: rows=%d d=%d V=%d", fn, rows, d, V);
  if (mode != 0 && mode != 1) return fail(MEDUSA_ERR_INVALID, "%s: mode %d", fn, mode);
  if (mode == 1 && !(temperature > 0.f)) return fail(MEDUSA_ERR_INVALID, "%s: temperature must be > 0", fn);
  if (mode == 1 && !logits) return fail(MEDUSA_ERR_INVALID, "%s: typical acceptance needs the logits", fn);
  if (w_layout != MEDUSA_W_ROWS && w_layout != MEDUSA_W_TILES)
    return fail(MEDUSA_ERR_INVALID, "%s: w_layout=%d", fn, (int)w_layout);
  if (dtype != MEDUSA_BF16) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: bf16 only", fn);
  if (d % BK) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: d=%d not a multiple of %d", fn, d, BK);
  if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(w_lm) |
       reinterpret_cast<uintptr_t>(stats)) % 16)
    return fail(MEDUSA_ERR_INVALID, "%s: hidden / w_lm / stats not 16-byte aligned", fn);
  const size_t need = (size_t)medusa_lm_head_stat_groups(rows, V) * rows * 16;
  if (stats_bytes < need) return fail(MEDUSA_ERR_CAPACITY, "%s: stats %zu < %zu bytes", fn, stats_bytes, need);
  LmArgs a{};
  a.logits = logits; a.V = V; a.err = err;
  a.mode = 0;
  a.write_logits = logits != nullptr;
  a.stats = static_cast<float4*>(stats);
  a.stat_mode = 1 + mode;
  a.inv_temp = mode == 1 ? 1.f / temperature : 1.f;
  a.ntiles = (V + BM - 1) / BM;
  return launch_tc(a, w_lm, w_layout == MEDUSA_W_TILES, V, hidden, rows, d, as_stream(stream), fn);
}
