// KV-cache compaction to the accepted path.
//
// "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
// Heads", decoding-step box (step 6) and Pitfalls: after acceptance, the
// accepted path's KV entries are copied into contiguous cache slots after the
// prefix.  The copy is a gather (the accepted nodes are not contiguous in the
// flattened tree), and it is done in place: slot L+j receives slot
// L+accepted[j], and since accepted[i] may equal j for some i < j, every
// source is read before any destination is written.
//
// One CTA per sequence.  Each thread owns a set of 16-byte columns of the
// (K, V) rows; it loads all A+1 source vectors of its columns into registers
// and only then stores them, so no column is written before it is read and no
// barrier is needed between CTAs.
#include "common.cuh"
#include "internal.h"

namespace medusa {
namespace {

__global__ void __launch_bounds__(256) kv_compact_kernel(uint8_t* k_cache, uint8_t* v_cache,
                                                          const int64_t* seq_start, int32_t* prefix_len,
                                                          const int32_t* accepted_nodes,
                                                          const int32_t* accept_len, int row_bytes,
                                                          int Kmax, int32_t* src_slots, int32_t* err) {
  const int b = blockIdx.x;
  const int L = prefix_len[b];
  const int64_t st = seq_start[b];
  const int A = accept_len[b];
  const int32_t* an = accepted_nodes + (int64_t)b * (Kmax + 1);
  __shared__ int src[MEDUSA_MAX_K + 1];
  __shared__ int bad;
  if (threadIdx.x == 0) {
    bad = (A < 0 || A > Kmax || L < 0) ? MEDUSA_DEVERR_LENGTH : 0;
    if (!bad) {
      for (int j = 0; j <= A; ++j) {
        const int a = an[j];
        if (a < j || a >= MEDUSA_MAX_T) bad = MEDUSA_DEVERR_NODE;
        src[j] = a;
      }
    }
    if (bad) set_err(err, bad);
  }
  __syncthreads();
  if (bad) return;
  const int vecs = row_bytes / 16;  // 16-byte columns per K (or V) row
  constexpr int MAXR = MEDUSA_MAX_K + 1;
  for (int col = threadIdx.x; col < 2 * vecs; col += blockDim.x) {
    uint8_t* base = col < vecs ? k_cache : v_cache;
    const int c = col < vecs ? col : col - vecs;
    uint4 tmp[MAXR];
#pragma unroll
    for (int j = 0; j < MAXR; ++j)
      if (j <= A && src[j] != j)
        tmp[j] = *reinterpret_cast<const uint4*>(base + (st + L + src[j]) * row_bytes + (int64_t)c * 16);
#pragma unroll
    for (int j = 0; j < MAXR; ++j)
      if (j <= A && src[j] != j)
        *reinterpret_cast<uint4*>(base + (st + L + j) * row_bytes + (int64_t)c * 16) = tmp[j];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (src_slots)
      for (int j = 0; j <= Kmax; ++j) src_slots[(int64_t)b * (Kmax + 1) + j] = j <= A ? L + src[j] : -1;
    prefix_len[b] = L + A + 1;
  }
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" int medusa_kv_compact(void* k_cache, void* v_cache, const int64_t* seq_start,
                                 int32_t* prefix_len, const int32_t* accepted_nodes,
                                 const int32_t* accept_len, int B, int H, int Dh, int Kmax,
                                 medusa_dtype dtype, int32_t* src_slots, int32_t* err, void* stream) {
  const char* fn = "medusa_kv_compact";
  if (!k_cache || !v_cache || !seq_start || !prefix_len || !accepted_nodes || !accept_len)
    return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (B < 1 || B > MEDUSA_MAX_B || H < 1 || Dh < 1 || Kmax < 0)
    return fail(MEDUSA_ERR_INVALID, "%s: B=%d H=%d Dh=%d Kmax=%d", fn, B, H, Dh, Kmax);
  if (Kmax > MEDUSA_MAX_K) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: Kmax=%d > %d", fn, Kmax, MEDUSA_MAX_K);
  if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: dtype", fn);
  const int row_bytes = H * Dh * (dtype == MEDUSA_BF16 ? 2 : 4);
  if (row_bytes % 16) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: H*Dh row of %d bytes is not a multiple of 16", fn, row_bytes);
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) % 16)
    return fail(MEDUSA_ERR_INVALID, "%s: caches not 16-byte aligned", fn);
  kv_compact_kernel<<<B, 256, 0, as_stream(stream)>>>(
      static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), seq_start, prefix_len,
      accepted_nodes, accept_len, row_bytes, Kmax, src_slots, err);
  return check_launch(fn);
}
