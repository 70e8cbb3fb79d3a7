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
// Every operand block is fp16 in "row format": 128-byte rows of 64 values, 8-row atoms with the
// 128-byte swizzle (row_chunk below).  The scan feeds two fused products from the staged part:
//   [D_U | D_O] = S^T [W^T | Q_hat^T]  (B MN-major: two 64-column blocks 16 KB apart)
//   [D_O | S^T] += U^T [M ; K_bar^T]^T (B K-major: 192 rows, M directly followed by K_bar^T)
constexpr uint32_t kRecWT = 0;          // W^T     [128 dk][64 r]
constexpr uint32_t kRecQT = 16384;      // Q_hat^T [128 dk][64 r]
constexpr uint32_t kRecMM = 32768;      // M       [64 r][64 s]
constexpr uint32_t kRecKT = 40960;      // K_bar^T [128 dk][64 r]
constexpr uint32_t kRecGC = 57344;      // e^{G_C} [128] fp32
constexpr uint32_t kRecStage = 57856;   // bytes the scan kernel stages in shared memory
constexpr uint32_t kRecUT = 59392;      // U_hat^T [128 dv][64 r] (read from global)
constexpr uint32_t kRecBytes = 75776;   // 74 KB

// ----------------------------------------------------------------- swizzled addressing
// fp16 [R rows][64 cols] row format: chunk j (cols 8j..8j+7) of row r.
__device__ __forceinline__ uint32_t row_chunk(int r, int j) {
  return (uint32_t)r * 128u + ((((uint32_t)j ^ (uint32_t)r) & 7u) << 4);
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

constexpr uint32_t idesc_f16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  mma_bf16_ss(d, a, b, idesc, acc);  // same instruction form; the descriptor selects f16
}
// A shared-memory descriptor advanced by `bytes` (start-address field, 16-byte units;
// shared addresses stay below 256 KB, so the 14-bit field never carries).
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

__device__ __forceinline__ uint32_t tmem_lane(uint32_t base, int warp) {
  return base + ((uint32_t)((warp & 3) * 32) << 16);
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


// MMA with the A operand in TMEM (lane = row, fp16 pairs packed two per 32-bit column, the
// even K index in the low half) and B from a shared-memory descriptor.
__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc ? 1u : 0u)
      : "memory");
}
// 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
// Bounded mbarrier wait that also gives up once another role has raised the CTA's abort flag;
// a wait that runs out raises the flag itself.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              uint32_t max_spins = 20000000u) {
  for (uint32_t i = 0; i < max_spins; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u && *abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}
// The same wait in a kernel variant built to test the abort path: with kGiveUp it gives up at
// once (raises the abort flag without polling), which is what a wait that runs out does.
template <bool kGiveUp>
__device__ __forceinline__ bool wait_or_abort_t(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if constexpr (kGiveUp) {
    *abort_flag = 1;
    return false;
  } else {
    return wait_or_abort(bar, parity, abort_flag);
  }
}

}  // namespace tcx
}  // namespace kda
