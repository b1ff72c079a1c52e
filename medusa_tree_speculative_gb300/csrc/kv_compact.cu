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
// One CTA per sequence (it alone reads and then advances prefix_len[b]).
// Each thread owns 16-byte columns of the (K, V) rows; it loads all A+1
// source vectors of its columns into registers and only then stores them, so
// no column is written before it is read and no barrier is needed.
#include "common.cuh"
#include "internal.h"

namespace medusa {
namespace {

template <int MAXR, int CPT>
__global__ void __launch_bounds__(512) kv_compact_kernel(uint8_t* k_cache, uint8_t* v_cache,
                                                          const int64_t* seq_start, int32_t* prefix_len,
                                                          const int32_t* accepted_nodes,
                                                          const int32_t* accept_len, int row_bytes,
                                                          int Kmax, int T, int32_t* src_slots, int32_t* err) {
  const int b = blockIdx.x;
  const int L = prefix_len[b];
  const int64_t st = seq_start[b];
  const int A = accept_len[b];
  const int32_t* an = accepted_nodes + (int64_t)b * (Kmax + 1);
  __shared__ int src[MEDUSA_MAX_K + 1];
  __shared__ int64_t soff[MEDUSA_MAX_K + 1], doff[MEDUSA_MAX_K + 1];  // byte offsets of moved rows
  __shared__ int bad, nmove;
  if (threadIdx.x == 0) {
    bad = (A < 0 || A > Kmax || L < 0) ? MEDUSA_DEVERR_LENGTH : 0;
    int n = 0;
    if (!bad) {
      for (int j = 0; j <= A; ++j) {
        const int a = an[j];
        // a node at depth j has index >= j (breadth-first order) and lies
        // inside the tree, whose rows were appended at slots L .. L + T - 1
        if (a < j || a >= T) bad = MEDUSA_DEVERR_NODE;
        src[j] = a;
        if (a != j) {  // row j moves: slot L+a -> slot L+j
          soff[n] = (st + L + a) * (int64_t)row_bytes;
          doff[n] = (st + L + j) * (int64_t)row_bytes;
          ++n;
        }
      }
    }
    nmove = n;
    if (bad) set_err(err, bad);
  }
  __syncthreads();
  if (bad) return;
  const int vecs = row_bytes / 16;  // 16-byte columns per K (or V) row; CPT per thread per pass
  const int nm = nmove;
  for (int col0 = threadIdx.x; col0 < 2 * vecs; col0 += CPT * blockDim.x) {
    uint4 tmp[CPT][MAXR];
#pragma unroll
    for (int q = 0; q < CPT; ++q) {
      const int col = col0 + q * blockDim.x;
      if (col >= 2 * vecs) continue;
      const uint8_t* base = (col < vecs ? k_cache : v_cache) + (int64_t)(col < vecs ? col : col - vecs) * 16;
#pragma unroll
      for (int t = 0; t < MAXR; ++t)
        if (t < nm) tmp[q][t] = *reinterpret_cast<const uint4*>(base + soff[t]);
    }
#pragma unroll
    for (int q = 0; q < CPT; ++q) {
      const int col = col0 + q * blockDim.x;
      if (col >= 2 * vecs) continue;
      uint8_t* base = (col < vecs ? k_cache : v_cache) + (int64_t)(col < vecs ? col : col - vecs) * 16;
#pragma unroll
      for (int t = 0; t < MAXR; ++t)
        if (t < nm) *reinterpret_cast<uint4*>(base + doff[t]) = tmp[q][t];
    }
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
                                 const int32_t* accept_len, int B, int H, int Dh, int Kmax, int T,
                                 medusa_dtype dtype, int32_t* src_slots, int32_t* err, void* stream) {
  const char* fn = "medusa_kv_compact";
  if (!k_cache || !v_cache || !seq_start || !prefix_len || !accepted_nodes || !accept_len)
    return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (B < 1 || B > MEDUSA_MAX_B || H < 1 || Dh < 1 || Kmax < 0)
    return fail(MEDUSA_ERR_INVALID, "%s: B=%d H=%d Dh=%d Kmax=%d", fn, B, H, Dh, Kmax);
  if (Kmax > MEDUSA_MAX_K) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: Kmax=%d > %d", fn, Kmax, MEDUSA_MAX_K);
  if (T < 1 || T > MEDUSA_MAX_T) return fail(MEDUSA_ERR_INVALID, "%s: T=%d outside 1..%d", fn, T, MEDUSA_MAX_T);
  if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: dtype", fn);
  const int row_bytes = H * Dh * (dtype == MEDUSA_BF16 ? 2 : 4);
  if (row_bytes % 16) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: H*Dh row of %d bytes is not a multiple of 16", fn, row_bytes);
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) % 16)
    return fail(MEDUSA_ERR_INVALID, "%s: caches not 16-byte aligned", fn);
  auto* kc = static_cast<uint8_t*>(k_cache);
  auto* vc = static_cast<uint8_t*>(v_cache);
  if (Kmax <= 4)
    launch_kernel(kv_compact_kernel<5, 2>, dim3(B), dim3(512), 0, as_stream(stream), kc, vc, seq_start, prefix_len,
               accepted_nodes, accept_len, row_bytes, Kmax, T, src_slots, err);
  else
    launch_kernel(kv_compact_kernel<MEDUSA_MAX_K + 1, 1>, dim3(B), dim3(512), 0, as_stream(stream), kc, vc,
               seq_start, prefix_len, accepted_nodes, accept_len, row_bytes, Kmax, T, src_slots, err);
  return check_launch(fn);
}
