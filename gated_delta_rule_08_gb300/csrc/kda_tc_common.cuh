// Shared definitions of the tensor-core prefill kernels: the per-(chunk, head) record
// exchanged between the chunk-parallel kernel and the scan, swizzled shared-memory
// addressing, and thin wrappers over tcgen05 / TMEM / named barriers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kda_device.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace tcx {

using namespace tc;

// ----------------------------------------------------------------- record layout (bytes)
constexpr uint32_t kRecWT = 0;          // W^T   [128 dk][64 r] fp16, row format (MN-major B of D_U)
constexpr uint32_t kRecQH = 16384;      // Q_hat [64 r][128 dk] fp16, token-row blocks (K-major B of D_O)
constexpr uint32_t kRecKB = 32768;      // K_bar [64 r][128 dk] fp16, token-row blocks (MN-major B of D_S)
constexpr uint32_t kRecMM = 49152;      // M     [64 r][64 s]   fp16, row format (K-major B of D_O)
constexpr uint32_t kRecGC = 57344;      // e^{G_C} [128] fp32
constexpr uint32_t kRecStage = 57856;   // bytes the scan kernel stages in shared memory
constexpr uint32_t kRecUT = 59392;      // U_hat^T [128 dv][64 r] fp16, row format (read from global)
constexpr uint32_t kRecBytes = 75776;   // 74 KB

// ----------------------------------------------------------------- swizzled addressing
// fp16/bf16 [64 rows][128 channels] as two 64-channel blocks of 64 x 128 B (128-byte swizzle):
// byte offset of the 16-byte chunk holding channels 8j..8j+7 of row r.
__device__ __forceinline__ uint32_t trow_chunk(int r, int c8) {
  return (uint32_t)(c8 >> 3) * 8192u + (uint32_t)r * 128u + ((((uint32_t)c8 & 7u) ^ ((uint32_t)r & 7u)) << 4);
}
// fp32 [64 rows][128 channels] as four 32-channel blocks of 64 x 128 B: chunk of channels 4j..4j+3.
__device__ __forceinline__ uint32_t g_chunk(int r, int c4) {
  return (uint32_t)(c4 >> 3) * 8192u + (uint32_t)r * 128u + ((((uint32_t)c4 & 7u) ^ ((uint32_t)r & 7u)) << 4);
}
// tf32 [R rows][32 channels] (one 128-byte K block): chunk of channels 4j..4j+3 of row r.
__device__ __forceinline__ uint32_t op_chunk(int r, int c4) {
  return (uint32_t)r * 128u + ((((uint32_t)c4 & 7u) ^ ((uint32_t)r & 7u)) << 4);
}
// fp16 [R rows][64 cols] row format: chunk j (cols 8j..8j+7) of row r.
__device__ __forceinline__ uint32_t row_chunk(int r, int j) {
  return (uint32_t)r * 128u + ((((uint32_t)j ^ (uint32_t)r) & 7u) << 4);
}

__device__ __forceinline__ float to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_h2(uint32_t u) {
  __half2 h = *reinterpret_cast<__half2*>(&u);
  return __half22float2(h);
}
__device__ __forceinline__ float2 unpack_bf2(uint32_t u) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(h);
}
__device__ __forceinline__ uint4 pack8_h(const float* v) {
  uint4 w;
  w.x = pack_h2(v[0], v[1]);
  w.y = pack_h2(v[2], v[3]);
  w.z = pack_h2(v[4], v[5]);
  w.w = pack_h2(v[6], v[7]);
  return w;
}
// 64 floats -> one fp16 row (row format) at `dst` (shared or global memory).
__device__ __forceinline__ void store_row64(uint8_t* dst, int r, const float* v) {
#pragma unroll
  for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(dst + row_chunk(r, j)) = pack8_h(v + 8 * j);
}

constexpr uint32_t idesc_f16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  mma_bf16_ss(d, a, b, idesc, acc);  // same instruction form; the descriptor selects f16
}
__device__ __forceinline__ void mma_tf32(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc ? 1u : 0u)
      : "memory");
}
// A shared-memory descriptor advanced by `bytes` (start-address field, 16-byte units;
// shared addresses stay below 256 KB, so the 14-bit field never carries).
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

__device__ __forceinline__ uint32_t tmem_lane(uint32_t base, int warp) {
  return base + ((uint32_t)((warp & 3) * 32) << 16);
}
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float t[16];
    tmem_ld16(taddr + 16 * q, t);
#pragma unroll
    for (int j = 0; j < 16; ++j) v[16 * q + j] = t[j];
  }
  tmem_wait_ld();
}
// Named barrier over `n` threads returning the AND of `v` across them.
__device__ __forceinline__ bool group_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void group_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}


}  // namespace tcx
}  // namespace kda
