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
// bf16: swap-AB tensor-core GEMM (vocabulary rows are the M dimension, tree
// rows the N dimension).  One persistent CTA per SM owns a contiguous slice of
// the vocabulary, so every weight byte is read once and no partial sums are
// exchanged; the slice streams through a 4-stage cp.async pipeline while the
// few hundred tree rows are re-read from L2.
// f32: a plain CUDA-core kernel (one warp per output element).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace medusa {
namespace {

constexpr int KB = 64;           // k per pipeline stage (128 bytes of bf16)
constexpr int STAGES = 4;
constexpr int NWARP = 8;
constexpr int WM = 32;           // vocabulary rows per warp (two m16 tiles)
constexpr int CM = NWARP * WM;   // vocabulary rows per CTA pass
constexpr int NT = 9;            // n8 tiles per pass: 72 tree rows
constexpr int CN = NT * 8;
constexpr int W_STAGE = CM * KB;  // elements
constexpr int H_STAGE = CN * KB;
constexpr size_t SMEM = (size_t)STAGES * (W_STAGE + H_STAGE) * sizeof(uint16_t);

struct LmArgs {
  const uint16_t* hidden;
  const uint16_t* w;
  float* logits;
  int rows, d, V, nblk;
};

__global__ void __launch_bounds__(NWARP * 32, 1) lm_head_mma_kernel(LmArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* ws = reinterpret_cast<uint16_t*>(smem);
  uint16_t* hs = ws + STAGES * W_STAGE;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // contiguous vocabulary slice of this CTA, in multiples of 16 rows
  const int v16 = (a.V + 15) / 16;
  const int v_lo = (int)((long)blockIdx.x * v16 / a.nblk) * 16;
  const int v_hi = min(a.V, (int)((long)(blockIdx.x + 1) * v16 / a.nblk) * 16);
  const int nkb = a.d / KB;

  for (int vp = v_lo; vp < v_hi; vp += CM) {
    for (int np = 0; np < a.rows; np += CN) {
      auto load = [&](int stage, int kb) {
        uint16_t* wst = ws + stage * W_STAGE;
        uint16_t* hst = hs + stage * H_STAGE;
        const int k0 = kb * KB;
        for (int e = threadIdx.x; e < CM * 8; e += blockDim.x) {
          const int rr = e >> 3, c = e & 7;
          const int v = vp + rr;
          const bool ok = v < v_hi;
          const uint16_t* src = a.w + (int64_t)(ok ? v : v_lo) * a.d + k0 + c * 8;
          cp_async16(smem_u32(wst + rr * KB + ((c ^ (rr & 7)) * 8)), src, ok ? 16 : 0);
        }
        for (int e = threadIdx.x; e < CN * 8; e += blockDim.x) {
          const int rr = e >> 3, c = e & 7;
          const int r = np + rr;
          const bool ok = r < a.rows;
          const uint16_t* src = a.hidden + (int64_t)(ok ? r : 0) * a.d + k0 + c * 8;
          cp_async16(smem_u32(hst + rr * KB + ((c ^ (rr & 7)) * 8)), src, ok ? 16 : 0);
        }
      };
      float acc[2][NT][4];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[m][n][0] = acc[m][n][1] = acc[m][n][2] = acc[m][n][3] = 0.f;

#pragma unroll
      for (int s = 0; s < STAGES - 1; ++s) {
        if (s < nkb) load(s, s);
        cp_async_commit();
      }
      for (int kb = 0; kb < nkb; ++kb) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        if (kb + STAGES - 1 < nkb) load((kb + STAGES - 1) % STAGES, kb + STAGES - 1);
        cp_async_commit();
        const uint16_t* wst = ws + (kb % STAGES) * W_STAGE;
        const uint16_t* hst = hs + (kb % STAGES) * H_STAGE;
#pragma unroll
        for (int kk = 0; kk < KB / 16; ++kk) {
          uint32_t af[2][4];
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const int rr = warp * WM + m * 16 + (lane & 15);
            const int c = kk * 2 + (lane >> 4);
            ldmatrix_x4(af[m], smem_u32(wst + rr * KB + ((c ^ (rr & 7)) * 8)));
          }
#pragma unroll
          for (int n = 0; n + 1 < NT; n += 2) {
            const int rr = n * 8 + (lane & 7) + ((lane >> 4) << 3);
            const int c = kk * 2 + ((lane >> 3) & 1);
            uint32_t bf[4];
            ldmatrix_x4(bf, smem_u32(hst + rr * KB + ((c ^ (rr & 7)) * 8)));
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              mma_bf16_16816(acc[m][n], af[m], bf[0], bf[1]);
              mma_bf16_16816(acc[m][n + 1], af[m], bf[2], bf[3]);
            }
          }
          if (NT & 1) {
            // last n8 tile: lanes 16..31 repeat rows of lanes 0..15
            const int n = NT - 1;
            const int rr = n * 8 + (lane & 7);
            const int c = kk * 2 + ((lane >> 3) & 1);
            uint32_t bf[4];
            ldmatrix_x4(bf, smem_u32(hst + rr * KB + ((c ^ (rr & 7)) * 8)));
#pragma unroll
            for (int m = 0; m < 2; ++m) mma_bf16_16816(acc[m][n], af[m], bf[0], bf[1]);
          }
        }
      }
      cp_async_wait<0>();
      __syncthreads();
      // epilogue: fp32 logits
#pragma unroll
      for (int m = 0; m < 2; ++m) {
#pragma unroll
        for (int n = 0; n < NT; ++n) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int v = vp + warp * WM + m * 16 + (lane >> 2) + (e >= 2 ? 8 : 0);
            const int r = np + n * 8 + (lane & 3) * 2 + (e & 1);
            if (v < v_hi && r < a.rows) a.logits[(int64_t)r * a.V + v] = acc[m][n][e];
          }
        }
      }
    }
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

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_lm_head_workspace_size(int rows, int d, int V) {
  (void)rows; (void)d; (void)V;
  return 0;
}

extern "C" int medusa_lm_head_verify(const void* hidden, const void* w_lm, float* logits, int rows,
                                     int d, int V, medusa_dtype dtype, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  const char* fn = "medusa_lm_head_verify";
  (void)workspace; (void)workspace_bytes;
  if (!hidden || !w_lm || !logits) return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (rows < 1 || d < 1 || V < 1) return fail(MEDUSA_ERR_INVALID, "%s: rows=%d d=%d V=%d", fn, rows, d, V);
  cudaStream_t s = as_stream(stream);
  if (dtype == MEDUSA_BF16) {
    if (d % KB) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: d=%d not a multiple of %d", fn, d, KB);
    if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(w_lm)) % 16)
      return fail(MEDUSA_ERR_INVALID, "%s: hidden / w_lm not 16-byte aligned", fn);
    LmArgs a{static_cast<const uint16_t*>(hidden), static_cast<const uint16_t*>(w_lm), logits, rows, d, V, 0};
    a.nblk = std::min(sm_count(), (V + 15) / 16);
    cudaFuncSetAttribute(lm_head_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
    lm_head_mma_kernel<<<a.nblk, NWARP * 32, SMEM, s>>>(a);
    return check_launch(fn);
  }
  if (dtype != MEDUSA_F32) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: dtype", fn);
  const int64_t total = (int64_t)rows * V;
  lm_head_f32_kernel<<<(unsigned)((total + 7) / 8), 256, 0, s>>>(
      static_cast<const float*>(hidden), static_cast<const float*>(w_lm), logits, rows, d, V);
  return check_launch(fn);
}
