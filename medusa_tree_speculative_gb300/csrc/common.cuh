// Device helpers shared by the libmedusa kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "medusa.h"

#define MDEV __device__ __forceinline__

namespace medusa {

// ---------------------------------------------------------------- numbers --

MDEV float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
MDEV float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Eight bf16 packed in 16 bytes -> eight floats.
MDEV void unpack8_bf16(const uint4& v, float* f) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

MDEV uint32_t pack2_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&h);
}

MDEV uint16_t f32_to_bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&h);
}

MDEV float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

template <typename T> MDEV float to_f32(T x);
template <> MDEV float to_f32<float>(float x) { return x; }
template <> MDEV float to_f32<uint16_t>(uint16_t x) { return bf16_bits_to_f32(x); }

template <typename T> MDEV T from_f32(float x);
template <> MDEV float from_f32<float>(float x) { return x; }
template <> MDEV uint16_t from_f32<uint16_t>(float x) { return f32_to_bf16_bits(x); }

// ------------------------------------------------------------ memory ops --

// Streaming 16-byte load that bypasses L1 (weights are read exactly once).
MDEV uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

MDEV uint4 ldg_v4(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

MDEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// cp.async 16 bytes global -> shared; src_bytes = 0 writes zeros.
MDEV void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
MDEV void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N> MDEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// --------------------------------------------------------- tensor cores --
// Warp-level m16n8k16 bf16 MMA with fp32 accumulation (legacy mma.sync path).

MDEV void ldmatrix_x4(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
MDEV void ldmatrix_x4_trans(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
MDEV void mma_bf16_16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ----------------------------------------------------------- reductions --

MDEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
MDEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// (value, index) ordered by value descending, then index ascending.
MDEV bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

MDEV void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ranks_before(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

// Counter arrival that publishes the block's earlier writes and, for the
// thread that sees the final count, acquires every other block's: call it
// from one thread after a __syncthreads() that follows the block's writes,
// and have the block read the others' data after another __syncthreads().
MDEV int arrive_acq_rel(int* counter) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;\n" : "=r"(old) : "l"(counter) : "memory");
  return old;
}

MDEV void set_err(int32_t* err, int code) {
  if (err) atomicOr(err, code);
}

}  // namespace medusa
