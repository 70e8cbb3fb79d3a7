// KDA chunked prefill on the tcgen05 tensor cores (bf16 inputs, dk = dv = 128).
//
// Kimi K3: Open Frontier Intelligence (kimi-k3-paper.pages.dev), section 2.5 / Eq. 4:
// per 64-token chunk a parallel intra-chunk part and a serial inter-chunk state pass.
// With chunk-start state S0, G_r the inclusive cumulative log-decay of the chunk,
//   A_rs = beta_r sum_c k_rc k_sc e^{G_rc - G_sc} (s < r),  M_rs = sum_c q_rc k_sc e^{G_rc - G_sc} (s <= r)
//   T = (I + A)^-1 Diag(beta),  W = T K_hat,  U_hat = T V                 (WY / UT transform)
//   U = U_hat - W S0,  O = Q_hat S0 + M U,  S_C = Diag(e^{G_C}) S0 + K_bar^T U
// Section 3.2 / Eq. 5 (g > -5) bounds every reference-scaled factor used below by e^{+-80}.
//
// Two kernels, both written with tcgen05 MMAs, TMEM accumulators and bulk (TMA-engine) copies:
//
//  kda_tc_chunk_prep  (grid = chunks x heads, fully parallel)
//    - cumulative log-decay G (fp32), reference-scaled operands (two centred references per
//      chunk, 15 and 47, and 47 for the off-diagonal block);
//    - one split-tf32 product (three tf32 MMAs per K step, fp32 accumulation), M=128 (64 key rows
//      + 64 query rows) x N=96 x K=128, yields both A and M: N columns 0..63 are the two diagonal
//      32x32 blocks, 64..95 the off-diagonal block;
//    - the unit-lower solve T = (I + A)^-1 Diag(beta) in fp32 on the CUDA cores;
//    - fp16 MMAs W^T = K_hat^T T^T and U_hat^T = V^T T^T (M=128, N=64, K=64);
//    - writes one 74 KB record per (chunk, head) laid out exactly as the scan kernel's shared
//      memory operands want them (W^T, Q_hat, K_bar, M, U_hat^T in fp16, e^{G_C} in fp32).
//
//  kda_tc_chunk_scan  (grid = sequences x heads; serial over the chunks of a sequence)
//    - S^T (dv x dk, fp32) lives in TMEM for the whole sequence; an fp16 copy in shared memory
//      is the A operand of the two state products;
//    - per chunk: D_U = S^T W^T, D_O = S^T Q_hat^T (MMA), U^T = U_hat^T - D_U (CUDA cores, fp16),
//      S^T = S^T Diag(e^{G_C}) (TMEM ld/st) + U^T K_bar (MMA), D_O += U^T M^T (MMA);
//    - records are double-buffered with bulk copies so the next chunk's operands arrive while
//      the current chunk runs; the optional RMSNorm + sigmoid-gate epilogue is fused in.
//
// Precision: bf16 operands cannot meet the parity bound on these workloads (see the design
// notes); fp16 has the bf16 MMA rate with 3 more significand bits, and every fp16 operand here is
// bounded (decayed keys/queries <= 1, values and states well inside the fp16 range).  The
// reference-scaled A/M operands need fp32 range; plain tf32 is enough for A but not for M (it
// feeds the read-out directly), so the A/M product is split-tf32.  Accumulation is fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kda_device.cuh"
#include "kda_internal.h"
#include "tc_ptx.cuh"

namespace kda {
namespace {

using namespace tc;

// ----------------------------------------------------------------- record layout (bytes)
constexpr uint32_t kRecWT = 0;        // W^T   [128 dk][64 r] fp16, row format (MN-major B of D_U)
constexpr uint32_t kRecQH = 16384;    // Q_hat [64 r][128 dk] fp16, token-row blocks (K-major B of D_O)
constexpr uint32_t kRecKB = 32768;    // K_bar [64 r][128 dk] fp16, token-row blocks (MN-major B of D_S)
constexpr uint32_t kRecMM = 49152;    // M     [64 r][64 s]   fp16, row format (K-major B of D_O)
constexpr uint32_t kRecUT = 57344;    // U_hat^T [128 dv][64 r] fp16, row format (read by threads)
constexpr uint32_t kRecGC = 73728;    // e^{G_C} [128] fp32
constexpr uint32_t kRecBytes = 75776; // 74 KB, multiple of 1024

// ----------------------------------------------------------------- swizzled addressing
// fp16 [64 rows][128 channels] as two 64-channel blocks of 64 x 128 B, 128-byte swizzle.
__device__ __forceinline__ uint32_t trow_f16(int r, int c) {
  return (uint32_t)(c >> 6) * 8192u + (uint32_t)r * 128u + ((((uint32_t)(c >> 3) & 7u) ^ ((uint32_t)r & 7u)) << 4) +
         ((uint32_t)(c & 7) << 1);
}
// fp16 [R rows][64 cols], one 128-byte row each, 128-byte swizzle.
__device__ __forceinline__ uint32_t row64_f16(int r, int j) {
  return (uint32_t)r * 128u + ((((uint32_t)(j >> 3) ^ (uint32_t)r) & 7u) << 4) + ((uint32_t)(j & 7) << 1);
}
// tf32 (fp32 container) [R rows][128 channels] K-major: four 32-channel blocks of R x 128 B.
__device__ __forceinline__ uint32_t kmaj_tf32(int r, int c, int R) {
  return (uint32_t)(c >> 5) * (uint32_t)(R * 128) + (uint32_t)r * 128u +
         ((((uint32_t)(c >> 2) & 7u) ^ ((uint32_t)r & 7u)) << 4) + ((uint32_t)(c & 3) << 2);
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
// Write one 64-element fp16 row (row format) from 64 floats.
__device__ __forceinline__ void store_row64(uint8_t* base, int r, const float* v) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint4 w;
    w.x = pack_h2(v[8 * j + 0], v[8 * j + 1]);
    w.y = pack_h2(v[8 * j + 2], v[8 * j + 3]);
    w.z = pack_h2(v[8 * j + 4], v[8 * j + 5]);
    w.w = pack_h2(v[8 * j + 6], v[8 * j + 7]);
    *reinterpret_cast<uint4*>(base + (uint32_t)r * 128u + ((((uint32_t)j ^ (uint32_t)r) & 7u) << 4)) = w;
  }
}

// Instruction descriptors.
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

__device__ __forceinline__ uint32_t tmem_lane(uint32_t base, int warp) {
  return base + ((uint32_t)((warp & 3) * 32) << 16);
}

// Load 64 consecutive TMEM columns of this thread's lane.
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

// =================================================================== prep kernel
constexpr int kPrepThreads = 256;
// shared-memory map (offsets from a 1024-aligned base)
// A/M pass operands (one 64-channel pass at a time), tf32 K-major, 112 KB in total:
constexpr uint32_t P_XH = 0;          // X hi [128 rows][64 ch] 32 KB
constexpr uint32_t P_XL = 32768;      // X lo 32 KB
constexpr uint32_t P_YH = 65536;      // Y hi [96 rows][64 ch] 24 KB
constexpr uint32_t P_YL = 90112;      // Y lo 24 KB
// ... reused after the A/M product:
constexpr uint32_t P_WT = 0;          // fp16 W^T [128][64] 16 KB
constexpr uint32_t P_UT = 16384;      // fp16 U_hat^T [128][64] 16 KB
constexpr uint32_t P_SA = 65536;      // fp32 A [64][65] for the solve
constexpr uint32_t P_KH = 114688;     // fp16 K_hat token-row blocks 16 KB
constexpr uint32_t P_VV = 131072;     // fp16 V token-row blocks 16 KB
constexpr uint32_t P_QH = 147456;     // fp16 Q_hat 16 KB
constexpr uint32_t P_KB = 163840;     // fp16 K_bar 16 KB
constexpr uint32_t P_TT = 180224;     // fp16 T [64 r][64 s] 8 KB
constexpr uint32_t P_MM = 188416;     // fp16 M [64 r][64 s] 8 KB
constexpr uint32_t P_GC = 196608;     // fp32 [128]
constexpr uint32_t P_BETA = 197120;   // fp32 [64]
constexpr uint32_t P_REF = 197376;    // fp32 [4][128]: G_15, G_31, G_47, G_63
constexpr uint32_t P_BAR = 199424;    // 2 mbarriers + TMEM address
constexpr uint32_t P_END = 199488;
constexpr uint32_t kPrepSmem = P_END + 1024;

constexpr uint32_t T_AM = 0;     // TMEM columns: A/M accumulator [128 x 96]
constexpr uint32_t T_W = 96;     // W^T accumulator [128 x 64]
constexpr uint32_t T_U = 160;    // U_hat^T accumulator [128 x 64]

__global__ void __launch_bounds__(kPrepThreads, 1)
kda_tc_chunk_prep(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                  const __nv_bfloat16* __restrict__ v, const float* __restrict__ g, const float* __restrict__ beta,
                  const int32_t* __restrict__ plan, const int32_t* __restrict__ cu, int B, int64_t T, int H,
                  uint8_t* __restrict__ records, unsigned int* __restrict__ err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_am = reinterpret_cast<uint64_t*>(sm + P_BAR);
  uint64_t* bar_wu = bar_am + 1;
  uint64_t* bar_fin = bar_am + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + P_BAR + 32);
  float* sGC = reinterpret_cast<float*>(sm + P_GC);
  float* sBeta = reinterpret_cast<float*>(sm + P_BETA);
  float* sRef = reinterpret_cast<float*>(sm + P_REF);

  const int64_t chunk = blockIdx.x;
  const int h = blockIdx.y;
  int b, n;
  int64_t t0, cseq;
  if (!resolve_chunk(chunk, plan, cu, B, T, b, t0, n, cseq)) return;
  uint8_t* rec = records + ((size_t)chunk * H + h) * kRecBytes;

  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  if (tid == 32) {
    mbar_init(bar_am, 1);
    mbar_init(bar_wu, 1);
    mbar_init(bar_fin, 1);
    mbar_fence_init();
  }

  // ---- 1. cumulative log-decay: thread (channel c, half) owns rows 32*half .. 32*half+31
  const int c = tid & 127, half = tid >> 7, r0 = 32 * half;
  float G[32];
  {
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int r = r0 + i;
      const float gv = (r < n) ? g[((size_t)(t0 + r) * H + h) * 128 + c] : 0.f;
      acc += gv;
      G[i] = acc;
    }
  }
  if (tid < 64) sBeta[tid] = (tid < n) ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
  if (half == 0) {
    sRef[0 * 128 + c] = G[15];
    sRef[1 * 128 + c] = G[31];
  }
  __syncthreads();
  if (half == 1) {
    const float base = sRef[1 * 128 + c];
#pragma unroll
    for (int i = 0; i < 32; ++i) G[i] += base;
    sRef[2 * 128 + c] = G[15];
    sRef[3 * 128 + c] = G[31];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- 2. operands
  {
    const float G63 = sRef[3 * 128 + c];
    if (half == 0) sGC[c] = __expf(G63);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int r = r0 + i;
      const size_t gi = ((size_t)(t0 + r) * H + h) * 128 + c;
      float kv = 0.f, qv = 0.f, vv = 0.f;
      if (r < n) {
        kv = __bfloat162float(k[gi]);
        qv = __bfloat162float(q[gi]);
        vv = __bfloat162float(v[gi]);
      }
      const float Gr = G[i];
      const float eG = __expf(Gr);
      *reinterpret_cast<__half*>(sm + P_KH + trow_f16(r, c)) = __float2half_rn(kv * eG);
      *reinterpret_cast<__half*>(sm + P_QH + trow_f16(r, c)) = __float2half_rn(qv * eG);
      *reinterpret_cast<__half*>(sm + P_KB + trow_f16(r, c)) = __float2half_rn(kv * __expf(G63 - Gr));
      *reinterpret_cast<__half*>(sm + P_VV + trow_f16(r, c)) = __float2half_rn(vv);
    }
  }
  // ---- 3. A and M: D[128 x 96] = X[128 x 128] Y[96 x 128]^T with X = [k e^{G-R}; q e^{G-R}],
  // Y = [k e^{R-G}; k e^{G_47-G} (s < 32)], as split-tf32 products (x = x_hi + x_lo, three MMAs:
  // hi*hi + hi*lo + lo*hi, fp32 accumulation; ~fp32 accuracy, which M needs for the read-out).
  // The operands of both splits do not fit at once, so the 128 channels go in two passes of 64.
  bool ok = true;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    if (pass == 1) ok = __syncthreads_and(ok && mbar_wait(bar_am, 0)) != 0;  // pass 0 MMAs done
    if ((c >> 6) == pass) {
      const int cc = c & 63;
      const float R = sRef[(half == 0 ? 0 : 2) * 128 + c];
      const float G47 = sRef[2 * 128 + c];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int r = r0 + i;
        const size_t gi = ((size_t)(t0 + r) * H + h) * 128 + c;
        float kv = 0.f, qv = 0.f;
        if (r < n) {
          kv = __bfloat162float(k[gi]);
          qv = __bfloat162float(q[gi]);
        }
        const float Gr = G[i];
        const float e1 = __expf(Gr - R), e2 = __expf(R - Gr);
        float x, hi;
        x = kv * e1; hi = to_tf32(x);
        *reinterpret_cast<float*>(sm + P_XH + kmaj_tf32(r, cc, 128)) = hi;
        *reinterpret_cast<float*>(sm + P_XL + kmaj_tf32(r, cc, 128)) = to_tf32(x - hi);
        x = qv * e1; hi = to_tf32(x);
        *reinterpret_cast<float*>(sm + P_XH + kmaj_tf32(64 + r, cc, 128)) = hi;
        *reinterpret_cast<float*>(sm + P_XL + kmaj_tf32(64 + r, cc, 128)) = to_tf32(x - hi);
        x = kv * e2; hi = to_tf32(x);
        *reinterpret_cast<float*>(sm + P_YH + kmaj_tf32(r, cc, 96)) = hi;
        *reinterpret_cast<float*>(sm + P_YL + kmaj_tf32(r, cc, 96)) = to_tf32(x - hi);
        if (half == 0) {
          x = kv * __expf(G47 - Gr); hi = to_tf32(x);
          *reinterpret_cast<float*>(sm + P_YH + kmaj_tf32(64 + r, cc, 96)) = hi;
          *reinterpret_cast<float*>(sm + P_YL + kmaj_tf32(64 + r, cc, 96)) = to_tf32(x - hi);
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_tf32(128, 96);
#pragma unroll
      for (int k0 = 0; k0 < 64; k0 += 8) {
        const uint32_t kb = k0 >> 5, kk = (k0 & 31) * 4;
        const uint64_t xh = smem_desc_sw128(smem_u32(sm + P_XH) + kb * 128 * 128 + kk, 16, 1024);
        const uint64_t xl = smem_desc_sw128(smem_u32(sm + P_XL) + kb * 128 * 128 + kk, 16, 1024);
        const uint64_t yh = smem_desc_sw128(smem_u32(sm + P_YH) + kb * 96 * 128 + kk, 16, 1024);
        const uint64_t yl = smem_desc_sw128(smem_u32(sm + P_YL) + kb * 96 * 128 + kk, 16, 1024);
        mma_tf32(tmem + T_AM, xh, yh, idesc, pass > 0 || k0 > 0);
        mma_tf32(tmem + T_AM, xh, yl, idesc, true);
        mma_tf32(tmem + T_AM, xl, yh, idesc, true);
      }
      mma_commit(bar_am);
    }
  }
  ok = __syncthreads_and(ok && mbar_wait(bar_am, 1)) != 0;
  tc_fence_after();

  // ---- 4. TMEM -> A (fp32, smem, beta-scaled strict lower) and M (fp16 record operand)
  float* sA = reinterpret_cast<float*>(sm + P_SA);  // [64][65]
  if (ok && warp < 4) {
    const int lane_row = warp * 32 + (tid & 31);  // 0..63: key rows (A); 64..127: query rows (M)
    const int r = lane_row & 63;
    float d[96];
#pragma unroll
    for (int q4 = 0; q4 < 6; ++q4) {
      float t[16];
      tmem_ld16(tmem_lane(tmem + T_AM, warp) + 16 * q4, t);
#pragma unroll
      for (int j = 0; j < 16; ++j) d[16 * q4 + j] = t[j];
    }
    tmem_wait_ld();
    if (lane_row < 64) {
      const float br = sBeta[r];
#pragma unroll
      for (int s = 0; s < 64; ++s) {
        const bool same = (s >> 5) == (r >> 5);
        const float raw = same ? d[s] : ((r >= 32 && s < 32) ? d[64 + (s & 31)] : 0.f);
        sA[r * 65 + s] = (s < r) ? br * raw : 0.f;  // select, never multiply a mask
      }
    } else {
      float m[64];
#pragma unroll
      for (int s = 0; s < 64; ++s) {
        const bool same = (s >> 5) == (r >> 5);
        const float raw = same ? d[s] : ((r >= 32 && s < 32) ? d[64 + (s & 31)] : 0.f);
        m[s] = (s <= r) ? raw : 0.f;
      }
      store_row64(sm + P_MM, r, m);
    }
  }
  __syncthreads();

  // ---- 5. T = (I + A)^-1 Diag(beta): forward substitution, 4 threads per column
  if (ok) {
    const int s = tid >> 2, part = tid & 3;
    float x[16];
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) x[jj] = 0.f;
#pragma unroll
    for (int r = 0; r < 64; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int j = 4 * jj + part;
        if (j < r) acc = fmaf(sA[r * 65 + j], x[jj], acc);
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      const float xv = (r == s) ? 1.f : ((r < s) ? 0.f : -acc);
      if (part == (r & 3)) x[r >> 2] = xv;
    }
    const float bs = sBeta[s];
#pragma unroll
    for (int jj = 0; jj < 16; ++jj)
      *reinterpret_cast<__half*>(sm + P_TT + row64_f16(4 * jj + part, s)) = __float2half_rn(x[jj] * bs);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();

  // ---- 6. W^T = K_hat^T T^T, U_hat^T = V^T T^T (fp16, M=128, N=64, K=64)
  if (tid == 0 && ok) {
    tc_fence_after();
    const uint32_t idesc = idesc_f16(128, 64, /*a_mn=*/true, /*b_mn=*/false);
#pragma unroll
    for (int k0 = 0; k0 < 64; k0 += 16) {
      const uint64_t bd = smem_desc_sw128(smem_u32(sm + P_TT) + k0 * 2, 16, 1024);
      const uint64_t ak = smem_desc_sw128(smem_u32(sm + P_KH) + (k0 >> 3) * 1024, 8192, 1024);
      const uint64_t av = smem_desc_sw128(smem_u32(sm + P_VV) + (k0 >> 3) * 1024, 8192, 1024);
      mma_f16(tmem + T_W, ak, bd, idesc, k0 > 0);
      mma_f16(tmem + T_U, av, bd, idesc, k0 > 0);
    }
    mma_commit(bar_wu);
  }
  ok = __syncthreads_and(ok && mbar_wait(bar_wu, 0)) != 0;
  tc_fence_after();

  // ---- 7. TMEM -> fp16 W^T (warps 0-3) and U_hat^T (warps 4-7) rows, into the old XA region
  if (ok) {
    const int row = (warp & 3) * 32 + (tid & 31);  // dk row (W^T) or dv row (U_hat^T)
    float vrow[64];
    tmem_ld64(tmem_lane(tmem + (warp < 4 ? T_W : T_U), warp), vrow);
    store_row64(sm + (warp < 4 ? P_WT : P_UT), row, vrow);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();

  // ---- 8. record -> global (bulk copies), then release TMEM
  if (tid == 0 && ok) {
    bulk_s2g(rec + kRecWT, sm + P_WT, 16384);
    bulk_s2g(rec + kRecQH, sm + P_QH, 16384);
    bulk_s2g(rec + kRecKB, sm + P_KB, 16384);
    bulk_s2g(rec + kRecMM, sm + P_MM, 8192);
    bulk_s2g(rec + kRecUT, sm + P_UT, 16384);
    bulk_s2g(rec + kRecGC, sm + P_GC, 512);
    bulk_commit();
    bulk_wait_all();
  }
  if (tid == 0 && !ok) {
    // a wait ran out: record it, let this thread's issued MMAs drain (bounded), then free TMEM
    atomicOr(err, KDA_DEVERR_WAIT_TIMEOUT);
    mma_commit(bar_fin);
    mbar_wait(bar_fin, 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// =================================================================== scan kernel
constexpr int kScanThreads = 128;
constexpr uint32_t S_STAGE0 = 0;
constexpr uint32_t S_STAGE1 = kRecBytes;
constexpr uint32_t S_SA = 2 * kRecBytes;          // fp16 S^T [128 dv][128 dk], two 16 KB K-blocks
constexpr uint32_t S_UA = S_SA + 32768;           // fp16 U^T [128 dv][64 r]
constexpr uint32_t S_BAR = S_UA + 16384;          // full[2], bar_u, bar_s, bar_o, bar_fin, tmem slot
constexpr uint32_t S_END = S_BAR + 64;
constexpr uint32_t kScanSmem = S_END + 1024;

constexpr uint32_t T_S = 0;      // TMEM: S^T fp32 [128 x 128]
constexpr uint32_t T_DU = 128;   // D_U [128 x 64]
constexpr uint32_t T_DO = 192;   // D_O [128 x 64]

// fp16 S^T element address: two K-blocks (dk 0..63, 64..127) of [128 rows][128 B]
__device__ __forceinline__ void store_srow(uint8_t* sa, int row, const float* s) {
#pragma unroll
  for (int kb = 0; kb < 2; ++kb)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float* p = s + 64 * kb + 8 * j;
      uint4 w;
      w.x = pack_h2(p[0], p[1]);
      w.y = pack_h2(p[2], p[3]);
      w.z = pack_h2(p[4], p[5]);
      w.w = pack_h2(p[6], p[7]);
      *reinterpret_cast<uint4*>(sa + kb * 16384 + (uint32_t)row * 128u + ((((uint32_t)j ^ (uint32_t)row) & 7u) << 4)) = w;
    }
}

template <typename Tout>
__global__ void __launch_bounds__(kScanThreads, 1)
kda_tc_chunk_scan(const uint8_t* __restrict__ records, const int32_t* __restrict__ plan,
                  const int32_t* __restrict__ cu, int B, int64_t T, int H, const float* __restrict__ h0,
                  float* __restrict__ hT, Tout* __restrict__ out, const __nv_bfloat16* __restrict__ gate,
                  const float* __restrict__ norm_w, float eps, unsigned int* __restrict__ err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + S_BAR);  // [2]
  uint64_t* bar_u = full + 2;
  uint64_t* bar_s = full + 3;
  uint64_t* bar_o = full + 4;
  uint64_t* bar_fin = full + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S_BAR + 48);

  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
  if (cu != nullptr && plan[B + 1] == 0) return;  // invalid cu_seqlens: sequence skipped
  int64_t first_chunk, t_begin, len;
  const int64_t nchunks = sequence_chunks(b, plan, cu, B, T, first_chunk, t_begin, len);

  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (tid == 32) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(bar_u, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init(bar_fin, 1);
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tl = tmem_lane(tmem, warp);  // this warp's lane quadrant
  const int row = tid;                         // dv row owned by this thread (TMEM lane)

  // initial state: S^T[row][dk] = h0[dk][row]
  {
    const size_t soff = ((size_t)b * H + h) * 128 * 128;
    float s[128];
#pragma unroll
    for (int c = 0; c < 128; ++c) s[c] = h0 ? h0[soff + (size_t)c * 128 + row] : 0.f;
#pragma unroll
    for (int q4 = 0; q4 < 8; ++q4) {
      float t[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) t[j] = s[16 * q4 + j];
      tmem_st16(tl + T_S + 16 * q4, t);
    }
    tmem_wait_st();
    store_srow(sm + S_SA, row, s);
  }
  if (tid == 0 && nchunks > 0) {
    mbar_arrive_expect_tx(&full[0], kRecBytes);
    bulk_g2s(sm + S_STAGE0, records + ((size_t)first_chunk * H + h) * kRecBytes, kRecBytes, &full[0]);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();

  bool ok = true;
  int64_t pending = nchunks > 0 ? 0 : -1;  // chunk whose record load is in flight / unconsumed
  for (int64_t c = 0; c < nchunks && ok; ++c) {
    const int st = (int)(c & 1);
    uint8_t* stage = sm + (st ? S_STAGE1 : S_STAGE0);
    const uint32_t ph = (uint32_t)(c & 1);
    // prefetch the next record into the other stage (freed at the end of chunk c-1)
    if (tid == 0 && c + 1 < nchunks) {
      uint8_t* nst = sm + (st ? S_STAGE0 : S_STAGE1);
      mbar_arrive_expect_tx(&full[st ^ 1], kRecBytes);
      bulk_g2s(nst, records + ((size_t)(first_chunk + c + 1) * H + h) * kRecBytes, kRecBytes, &full[st ^ 1]);
    }
    if (!__syncthreads_and(mbar_wait(&full[st], (uint32_t)((c >> 1) & 1)))) { ok = false; break; }
    pending = c + 1 < nchunks ? c + 1 : -1;
    tc_fence_after();

    // MMA: D_U = S^T W^T ; D_O = S^T Q_hat^T
    if (tid == 0) {
      const uint32_t id_u = idesc_f16(128, 64, false, true);
      const uint32_t id_o = idesc_f16(128, 64, false, false);
#pragma unroll
      for (int k0 = 0; k0 < 128; k0 += 16) {
        const uint32_t kb = k0 >> 6, kk = (k0 & 63) * 2;
        const uint64_t ad = smem_desc_sw128(smem_u32(sm + S_SA) + kb * 16384 + kk, 16, 1024);
        const uint64_t bw = smem_desc_sw128(smem_u32(stage + kRecWT) + (k0 >> 3) * 1024, 8192, 1024);
        mma_f16(tmem + T_DU, ad, bw, id_u, k0 > 0);
      }
      mma_commit(bar_u);
#pragma unroll
      for (int k0 = 0; k0 < 128; k0 += 16) {
        const uint32_t kb = k0 >> 6, kk = (k0 & 63) * 2;
        const uint64_t ad = smem_desc_sw128(smem_u32(sm + S_SA) + kb * 16384 + kk, 16, 1024);
        const uint64_t bq = smem_desc_sw128(smem_u32(stage + kRecQH) + kb * 8192 + kk, 16, 1024);
        mma_f16(tmem + T_DO, ad, bq, id_o, k0 > 0);
      }
    }
    __syncwarp();

    // while the MMAs run: S^T <- S^T Diag(e^{G_C}) in TMEM (the MMAs read the fp16 copy)
    {
      const float* gc = reinterpret_cast<const float*>(stage + kRecGC);
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        float t[16];
        tmem_ld16(tl + T_S + 16 * q4, t);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) t[j] *= gc[16 * q4 + j];
        tmem_st16(tl + T_S + 16 * q4, t);
      }
      tmem_wait_st();
    }

    // U^T = U_hat^T - D_U  -> fp16 A operand
    if (!__syncthreads_and(mbar_wait(bar_u, ph))) { ok = false; break; }
    tc_fence_after();
    {
      float u[64];
      tmem_ld64(tl + T_DU, u);
      const uint8_t* ut = stage + kRecUT + (uint32_t)row * 128u;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 w = *reinterpret_cast<const uint4*>(ut + ((((uint32_t)j ^ (uint32_t)row) & 7u) << 4));
        const float2 a0 = unpack_h2(w.x), a1 = unpack_h2(w.y), a2 = unpack_h2(w.z), a3 = unpack_h2(w.w);
        u[8 * j + 0] = a0.x - u[8 * j + 0]; u[8 * j + 1] = a0.y - u[8 * j + 1];
        u[8 * j + 2] = a1.x - u[8 * j + 2]; u[8 * j + 3] = a1.y - u[8 * j + 3];
        u[8 * j + 4] = a2.x - u[8 * j + 4]; u[8 * j + 5] = a2.y - u[8 * j + 5];
        u[8 * j + 6] = a3.x - u[8 * j + 6]; u[8 * j + 7] = a3.y - u[8 * j + 7];
      }
      store_row64(sm + S_UA, row, u);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // MMA: S^T += U^T K_bar ; D_O += U^T M^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id_s = idesc_f16(128, 128, false, true);
      const uint32_t id_o = idesc_f16(128, 64, false, false);
#pragma unroll
      for (int k0 = 0; k0 < 64; k0 += 16) {
        const uint64_t au = smem_desc_sw128(smem_u32(sm + S_UA) + k0 * 2, 16, 1024);
        const uint64_t bk = smem_desc_sw128(smem_u32(stage + kRecKB) + (k0 >> 3) * 1024, 8192, 1024);
        mma_f16(tmem + T_S, au, bk, id_s, true);
      }
      mma_commit(bar_s);
#pragma unroll
      for (int k0 = 0; k0 < 64; k0 += 16) {
        const uint64_t au = smem_desc_sw128(smem_u32(sm + S_UA) + k0 * 2, 16, 1024);
        const uint64_t bm = smem_desc_sw128(smem_u32(stage + kRecMM) + k0 * 2, 16, 1024);
        mma_f16(tmem + T_DO, au, bm, id_o, true);
      }
      mma_commit(bar_o);
    }
    __syncwarp();

    // new state -> fp16 A operand for the next chunk
    if (!__syncthreads_and(mbar_wait(bar_s, ph))) { ok = false; break; }
    tc_fence_after();
    {
      float s[128];
      tmem_ld64(tl + T_S, s);
      tmem_ld64(tl + T_S + 64, s + 64);
      store_srow(sm + S_SA, row, s);
    }

    // outputs: D_O -> fp32 [r][dv] in this stage (its operands are consumed) -> epilogue -> global
    if (!__syncthreads_and(mbar_wait(bar_o, ph))) { ok = false; break; }
    tc_fence_after();
    {
      float o[64];
      tmem_ld64(tl + T_DO, o);
      float* ost = reinterpret_cast<float*>(stage);
#pragma unroll
      for (int r = 0; r < 64; ++r) ost[r * 128 + row] = o[r];
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    {
      const int64_t rem = len - 64 * c;
      const int n = (int)(rem < 64 ? rem : 64);
      const int64_t t0 = t_begin + 64 * c;
      const float* ost = reinterpret_cast<const float*>(stage);
      const int lane = tid & 31;
      for (int r = warp; r < n; r += 4) {
        float4 y = *reinterpret_cast<const float4*>(ost + r * 128 + 4 * lane);
        const size_t orow = ((size_t)(t0 + r) * H + h) * 128 + 4 * lane;
        if (gate != nullptr) {
          float ss = y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
          ss = warp_sum(ss);
          const float inv = rsqrtf(ss * (1.f / 128.f) + eps);
          float w0 = 1.f, w1 = 1.f, w2 = 1.f, w3 = 1.f;
          if (norm_w) { w0 = norm_w[4 * lane]; w1 = norm_w[4 * lane + 1]; w2 = norm_w[4 * lane + 2]; w3 = norm_w[4 * lane + 3]; }
          y.x = y.x * inv * w0 * sigmoidf_(__bfloat162float(gate[orow + 0]));
          y.y = y.y * inv * w1 * sigmoidf_(__bfloat162float(gate[orow + 1]));
          y.z = y.z * inv * w2 * sigmoidf_(__bfloat162float(gate[orow + 2]));
          y.w = y.w * inv * w3 * sigmoidf_(__bfloat162float(gate[orow + 3]));
        }
        out[orow + 0] = from_f32<Tout>(y.x);
        out[orow + 1] = from_f32<Tout>(y.y);
        out[orow + 2] = from_f32<Tout>(y.z);
        out[orow + 3] = from_f32<Tout>(y.w);
      }
    }
    tc_fence_before();
    __syncthreads();  // stage free for the prefetch issued at the start of chunk c+1
  }

  if (!ok) {
    // a wait ran out: record it, let the in-flight record load and this thread's MMAs drain
    // (each wait bounded), then free TMEM and return
    if (tid == 0) {
      atomicOr(err, KDA_DEVERR_WAIT_TIMEOUT);
      if (pending >= 0) mbar_wait(&full[pending & 1], (uint32_t)((pending >> 1) & 1));
      mma_commit(bar_fin);
      mbar_wait(bar_fin, 0);
    }
  } else if (hT != nullptr) {
    tc_fence_after();
    float s[128];
    tmem_ld64(tl + T_S, s);
    tmem_ld64(tl + T_S + 64, s + 64);
    const size_t soff = ((size_t)b * H + h) * 128 * 128;
#pragma unroll
    for (int c = 0; c < 128; ++c) hT[soff + (size_t)c * 128 + row] = s[c];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

template <typename Tout>
cudaError_t launch_tc(const PrefillArgs& a, cudaStream_t st) {
  static bool attr_done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kda_tc_chunk_prep, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kPrepSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_tc_chunk_scan<Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScanSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const bool has_cu = a.cu_seqlens != nullptr;
  const int64_t nchunks = max_chunks(a.B, a.T, has_cu);
  int32_t* plan = static_cast<int32_t*>(a.workspace);
  uint8_t* records = static_cast<uint8_t*>(a.workspace) + plan_bytes(a.B);
  if (has_cu) {
    TraceScope ts("kda_plan", st);
    cudaError_t e = plan_launch(a.cu_seqlens, a.B, a.T_tot, plan, a.err, st);
    if (e != cudaSuccess) return e;
  }
  if (nchunks > 0) {
    TraceScope ts("kda_tc_chunk_prep", st);
    kda_tc_chunk_prep<<<dim3((unsigned)nchunks, (unsigned)a.H), kPrepThreads, kPrepSmem, st>>>(
        static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
        static_cast<const __nv_bfloat16*>(a.v), a.g, a.beta, plan, a.cu_seqlens, a.B, a.T, a.H, records, a.err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  TraceScope ts("kda_tc_chunk_scan", st);
  kda_tc_chunk_scan<Tout><<<dim3((unsigned)a.B, (unsigned)a.H), kScanThreads, kScanSmem, st>>>(
      records, plan, a.cu_seqlens, a.B, a.T, a.H, a.h0, a.hT, static_cast<Tout*>(a.out),
      static_cast<const __nv_bfloat16*>(a.epi.gate), a.epi.norm_weight, a.epi.eps, a.err);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_tc_blob_bytes(int, int) { return kRecBytes; }
bool prefill_tc_supported(int dk, int dv) { return dk == 128 && dv == 128; }
cudaError_t prefill_tc_launch(const PrefillArgs& a, cudaStream_t st) {
  if (!a.bf16 || !prefill_tc_supported(a.dk, a.dv)) return cudaErrorNotSupported;
  return a.out_bf16 ? launch_tc<__nv_bfloat16>(a, st) : launch_tc<float>(a, st);
}

}  // namespace kda
