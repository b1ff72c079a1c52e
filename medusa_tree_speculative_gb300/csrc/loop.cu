// The decode loop's glue on the device: appending each step's tokens to the
// output, and a stand-in for the backbone forward.
//
// "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
// Heads", decoding-step box, step 6: the step appends the root and the
// accepted tokens (1 + accept_len new tokens) and the next step starts from
// the accepted path.  medusa_append_tokens is that append.
//
// medusa_standin_embed has no counterpart in the paper: it stands in for the
// backbone forward over the tree (hidden state of each tree token = one row of
// an embedding table), so that the verify step can run in a closed loop on the
// device without a transformer.  It is the whole "model" of the stand-in.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace medusa {
namespace {

__global__ void __launch_bounds__(32) append_tokens_kernel(const int32_t* tokens, const int32_t* accepted_nodes,
                                                           const int32_t* accept_len, int T, int Kmax,
                                                           int32_t* out, int32_t* out_len, int out_cap,
                                                           int32_t* err) {
  const int b = blockIdx.x, lane = threadIdx.x;
  const int n = accept_len[b];
  const int L0 = out_len[b];
  if (n < 0 || n > Kmax) {
    if (lane == 0) set_err(err, MEDUSA_DEVERR_LENGTH);
    return;
  }
  if (L0 < 0 || L0 + n + 1 > out_cap) {
    if (lane == 0) set_err(err, MEDUSA_DEVERR_CAPACITY);
    return;
  }
  bool bad = false;
  for (int j = lane; j <= n; j += 32) {
    const int node = accepted_nodes[(int64_t)b * (Kmax + 1) + j];
    if (node < 0 || node >= T) {
      bad = true;
      continue;
    }
    out[(int64_t)b * out_cap + L0 + j] = tokens[(int64_t)b * T + node];
  }
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) set_err(err, MEDUSA_DEVERR_NODE);
    return;  // out_len unchanged: the step's tokens are not counted
  }
  __syncwarp();
  if (lane == 0) out_len[b] = L0 + n + 1;
}

// hidden[r] = emb[tokens[r]] (16-byte chunks); an out-of-range token gives a
// zero row and raises the error bit.
__global__ void __launch_bounds__(256) standin_embed_kernel(const int32_t* tokens, const uint4* emb, int V,
                                                            int rows, int chunks, uint4* hidden, int32_t* err) {
  const int64_t total = (int64_t)rows * chunks;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(g / chunks), c = (int)(g % chunks);
    const int t = tokens[r];
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (t >= 0 && t < V)
      v = __ldg(emb + (int64_t)t * chunks + c);
    else if (c == 0)
      set_err(err, MEDUSA_DEVERR_TOKEN);
    hidden[g] = v;
  }
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" int medusa_append_tokens(const int32_t* tokens, const int32_t* accepted_nodes,
                                    const int32_t* accept_len, int B, int T, int Kmax, int32_t* out,
                                    int32_t* out_len, int out_cap, int32_t* err, void* stream) {
  const char* fn = "medusa_append_tokens";
  if (!tokens || !accepted_nodes || !accept_len || !out || !out_len)
    return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (B < 1 || B > MEDUSA_MAX_B || T < 1 || Kmax < 0 || Kmax > MEDUSA_MAX_K || out_cap < 1)
    return fail(MEDUSA_ERR_INVALID, "%s: B=%d T=%d Kmax=%d out_cap=%d", fn, B, T, Kmax, out_cap);
  launch_kernel(append_tokens_kernel, dim3(B), dim3(32), 0, as_stream(stream), tokens, accepted_nodes, accept_len,
                T, Kmax, out, out_len, out_cap, err);
  return check_launch(fn);
}

extern "C" int medusa_standin_embed(const int32_t* tokens, int rows, const void* emb, int V, int d,
                                    medusa_dtype dtype, void* hidden, int32_t* err, void* stream) {
  const char* fn = "medusa_standin_embed";
  if (!tokens || !emb || !hidden) return fail(MEDUSA_ERR_INVALID, "%s: NULL tensor", fn);
  if (rows < 1 || V < 1 || d < 1) return fail(MEDUSA_ERR_INVALID, "%s: rows=%d V=%d d=%d", fn, rows, V, d);
  if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: dtype", fn);
  const int esize = dtype == MEDUSA_BF16 ? 2 : 4;
  if (((int64_t)d * esize) % 16) return fail(MEDUSA_ERR_UNSUPPORTED, "%s: rows of %d bytes", fn, d * esize);
  if ((reinterpret_cast<uintptr_t>(emb) | reinterpret_cast<uintptr_t>(hidden)) % 16)
    return fail(MEDUSA_ERR_INVALID, "%s: emb / hidden not 16-byte aligned", fn);
  const int chunks = d * esize / 16;
  const int64_t total = (int64_t)rows * chunks;
  const int grid = (int)std::min<int64_t>((total + 255) / 256, (int64_t)sm_count() * 4);
  launch_kernel(standin_embed_kernel, dim3(grid), dim3(256), 0, as_stream(stream), tokens,
                static_cast<const uint4*>(emb), V, rows, chunks, static_cast<uint4*>(hidden), err);
  return check_launch(fn);
}
