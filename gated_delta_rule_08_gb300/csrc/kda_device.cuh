// Small device helpers shared by the KDA kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define KDA_DEVERR_BAD_SLOT 0x1u
#define KDA_DEVERR_BAD_SEQLENS 0x2u
#define KDA_DEVERR_WAIT_TIMEOUT 0x4u
#define KDA_DEVERR_BAD_COUNT 0x8u
#define KDA_DEVERR_NONFINITE 0x10u
#define KDA_DEVERR_PRECONDITION 0x20u

namespace kda {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// sigmoid; the reciprocal by the fast divide (about 2 ulp; 0 once e^-x overflows)
__device__ __forceinline__ float sigmoidf_(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

__device__ __forceinline__ float4 f4_fma(float a, float4 b, float4 c) {
  return make_float4(fmaf(a, b.x, c.x), fmaf(a, b.y, c.y), fmaf(a, b.z, c.z), fmaf(a, b.w, c.w));
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// plan (built on the device from cu_seqlens): plan[0..B] exclusive chunk offsets (plan[B] = all
// chunks), plan[B+1] = 1 if cu_seqlens was valid, plan[B+2+r] = the sequence of rank r by
// decreasing length (ties by index; the identity for large B).
// Sequence of rank r in the serial pass's launch order: the longest chains start first.
// bytes (a multiple of 16) from a 16-byte aligned global address into L2, without waiting
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

constexpr int kOrderMaxB = 512;  // beyond this many sequences the order is the identity
__device__ __forceinline__ int sequence_of_rank(int r, const int32_t* plan, const int32_t* cu, int B) {
  return cu == nullptr ? r : plan[B + 2 + r];
}

// Resolve a global chunk index into (sequence b, token start t0, valid rows n).
// Without cu_seqlens: B sequences of T tokens each.  Returns false for a chunk
// index beyond the last chunk (grid over-provisioning) or an invalid plan.
__device__ __forceinline__ bool resolve_chunk(int64_t chunk, const int32_t* plan,
                                              const int32_t* cu, int B, int64_t T,
                                              int& b, int64_t& t0, int& n, int64_t& c_in_seq) {
  if (cu == nullptr) {
    const int64_t nc = (T + 63) / 64;
    if (nc == 0) return false;
    b = (int)(chunk / nc);
    if (b >= B) return false;
    c_in_seq = chunk % nc;
    t0 = (int64_t)b * T + c_in_seq * 64;
    const int64_t rem = T - c_in_seq * 64;
    n = (int)(rem < 64 ? rem : 64);
    return true;
  }
  if (plan[B + 1] == 0) return false;
  if (chunk >= plan[B]) return false;
  int lo = 0, hi = B - 1;  // largest b with plan[b] <= chunk
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (plan[mid] <= chunk) lo = mid; else hi = mid - 1;
  }
  b = lo;
  c_in_seq = chunk - plan[b];
  t0 = (int64_t)cu[b] + c_in_seq * 64;
  const int64_t rem = (int64_t)cu[b + 1] - t0;
  n = (int)(rem < 64 ? rem : 64);
  return n > 0;
}

// Sequence bounds for the serial pass.  Returns the number of chunks of sequence b
// and its first global chunk index / first token.
__device__ __forceinline__ int64_t sequence_chunks(int b, const int32_t* plan, const int32_t* cu,
                                                   int B, int64_t T, int64_t& first_chunk,
                                                   int64_t& t_begin, int64_t& len) {
  if (cu == nullptr) {
    const int64_t nc = (T + 63) / 64;
    first_chunk = (int64_t)b * nc;
    t_begin = (int64_t)b * T;
    len = T;
    return nc;
  }
  if (plan[B + 1] == 0) { first_chunk = 0; t_begin = 0; len = 0; return 0; }
  first_chunk = plan[b];
  t_begin = cu[b];
  len = (int64_t)cu[b + 1] - cu[b];
  return (int64_t)plan[b + 1] - plan[b];
}

// Index of the first state checkpoint of sequence b when every sequence stores one after each
// `span` of its tokens (span = 64 x checkpoint interval in chunks): the checkpoints of the
// sequences before b, floor(len / span) each.
__device__ __forceinline__ int64_t checkpoint_base(int b, const int32_t* cu, int64_t T, int64_t span) {
  if (cu == nullptr) return (int64_t)b * (T / span);
  int64_t s = 0;
  for (int i = 0; i < b; ++i) s += ((int64_t)cu[i + 1] - cu[i]) / span;
  return s;
}

}  // namespace kda
