// KDA chunked prefill on the tcgen05 tensor cores (bf16 inputs, dk = dv = 128): the
// chunk-parallel part.
//
// Kimi K3: Open Frontier Intelligence (kimi-k3-paper.pages.dev), section 2.5 / Eq. 4:
// per 64-token chunk a parallel intra-chunk part and a serial inter-chunk state pass.
// With chunk-start state S0, G_r the inclusive cumulative log-decay of the chunk,
//   A_rs = beta_r sum_c k_rc k_sc e^{G_rc - G_sc} (s < r),  M_rs = sum_c q_rc k_sc e^{G_rc - G_sc} (s <= r)
//   T = (I + A)^-1 Diag(beta),  W = T K_hat,  U_hat = T V                 (WY / UT transform)
//   U = U_hat - W S0,  O = Q_hat S0 + M U,  S_C = Diag(e^{G_C}) S0 + K_bar^T U
// Section 3.2 / Eq. 5 (g > -5) bounds every reference-scaled factor used below by e^{+-80}.
//
//  kda_tc_chunk_prep (persistent, two CTAs per SM, each looping over (chunk, head) tasks)
//    warp 8 stages the raw q, k, v tiles by TMA (128-byte swizzle; the next task's tiles once the
//      current task's last MMAs have read k and v, which the passes overwrite in place) and beta by
//      plain loads, and issues every MMA;
//    warps 0-7, per task:
//    - four 32-channel passes; thread = (channel pair, 4 rows): the cumulative log-decay is a
//      running sum over the thread's rows plus the sums of the row groups above it (exchanged in
//      shared memory); g is read straight from global memory one pass ahead;
//    - each pass writes the reference-scaled keys/queries as a three-way bf16 split
//      (x = hi + lo, hi = x with its low 16 bits cleared, lo = x - hi rounded): A and M come from
//      X_h [Y_h ; Y_l]^T (N = 192) + X_l Y_h^T (N = 96), fp32 accumulation, M = 128 rows (64 key
//      rows for A, 64 query rows for M) x 96 columns (two diagonal 32 x 32 blocks with centred
//      references 15 and 47, plus the off-diagonal block with reference 47).  Pass p fills half
//      (p & 1) of every 128-byte operand row, so it only waits for the MMAs of pass p - 2;
//    - the passes also emit Q_hat^T and K_bar^T (channel-major) and e^{G_C} into the record, and
//      Diag(beta) K_hat and Diag(beta) V (fp16) in place of the raw tiles;
//    - X = (I + A)^-1: 16 x 16 diagonal blocks by forward substitution (fp32), then two
//      levels of block merges (16 -> 32 -> 64 rows) by warp-level tf32 MMAs with a three-term split
//      (~fp32), one 16 x 8 half-tile per warp;
//    - fp16 MMAs W^T = (Diag(beta) K_hat)^T X^T and U_hat^T = (Diag(beta) V)^T X^T with
//      X = (I + A)^-1 (M = 128, N = 64, K = 64), then W^T, M and U_hat^T into the record.
//
// Precision: bf16 operands cannot meet the parity bound on these workloads; fp16 has the bf16
// MMA rate with 3 more significand bits, and every fp16 operand here is bounded (decayed
// keys/queries <= 1) except those that scale with the values (Diag(beta) V, U_hat) and the
// inverse X; one of those past 65504 becomes inf, which the state pass meets in what it writes
// (KDA_DEVERR_NONFINITE).  The reference-scaled A/M operands need fp32 range and ~16 significant
// bits (M feeds the read-out directly, and a head-wise RMSNorm amplifies its error on rows of small
// norm: a single tf32 product measured 0.031 max|err|/RMS there): hence the split.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kda_internal.h"
#include "kda_tc_common.cuh"

namespace kda {
namespace {

using namespace tcx;

// =================================================================== prep kernel
constexpr int kPrepThreads = 288;   // warps 0-7 compute, warp 8 stages inputs and issues the MMAs
constexpr int kCompute = 256;
constexpr int kIssuer = 8;
// raw tiles: k | q | v (bf16 token-row blocks, two 64-channel blocks each)
constexpr uint32_t R_K = 0, R_Q = 16384, R_V = 32768, R_BYTES = 49152;
constexpr uint32_t P_OPS = R_BYTES;      // 56 KB: one 64-channel K block of split-bf16 operands
constexpr uint32_t O_XH = 0, O_XL = 16384, O_YH = 32768, O_YL = 45056, O_BYTES = 57344;
// after the A/M product the operand region holds the solve:
constexpr uint32_t O_SA = 0;             // fp32 A [64][68]
constexpr uint32_t O_SX = 17408;         // fp32 X = (I + A)^-1 [64][64], columns permuted per row (swx)
constexpr uint32_t O_SY = 33792;         // fp32 scratch: four 16 x 16 tiles, row stride 24
constexpr uint32_t O_TT = 40960;         // fp16 X [64 r][64 s] row format (1024-aligned)
constexpr uint32_t O_MST = 49152;        // M staged for its bulk copy to the record (8 KB)
static_assert(O_SY + 4 * 16 * 24 * 4 <= O_TT && O_MST + 8192 <= O_BYTES, "solve region");
// after the W / U_hat MMAs: W^T at 0 and U_hat^T at 16384 staged for their bulk copies
constexpr uint32_t P_MISC = P_OPS + O_BYTES;
constexpr uint32_t M_BETA = 0;           // fp32 [2 tasks][64]
constexpr uint32_t M_TOT = 512;          // float2 [2][8 warps][16 channel pairs]: decay sums of row-group pairs
constexpr uint32_t M_BAR = 4608;         // barriers, tmem slot, abort flag
constexpr uint32_t M_END = 4736;
constexpr uint32_t kPrepSmem = P_MISC + M_END + 1024;
constexpr uint32_t kPrepTmemCols = 256;

constexpr uint32_t T_AM = 0;    // TMEM: [X_h Y_h + X_l Y_h | X_h Y_l] [128 x 192]
constexpr uint32_t T_W = 0;     // W^T [128 x 64]      } reuse the A/M columns once they are read
constexpr uint32_t T_U = 64;    // U_hat^T [128 x 64]  }

// x (2 floats) -> bf16 hi (x with its low 16 bits cleared, exact in bf16) and lo = x - hi
// rounded to bf16, each as a packed pair.
// two fp32 lanes per instruction (each lane rounded exactly as the scalar operation)
#define KDA_F32X2_OP(name, op)                                                                        \
  __device__ __forceinline__ float2 name(float2 a, float2 b) {                                        \
    float2 d;                                                                                         \
    asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n " op            \
        " rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"                                                       \
        : "=f"(d.x), "=f"(d.y)                                                                        \
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));                                                    \
    return d;                                                                                         \
  }
KDA_F32X2_OP(fadd2, "add.rn.f32x2")
KDA_F32X2_OP(fsub2, "sub.rn.f32x2")
KDA_F32X2_OP(fmul2, "mul.rn.f32x2")
#undef KDA_F32X2_OP

__device__ __forceinline__ void split_bf16x2(float2 x, uint32_t& hi, uint32_t& lo) {
  const uint32_t a = __float_as_uint(x.x) & 0xFFFF0000u, b = __float_as_uint(x.y) & 0xFFFF0000u;
  hi = (a >> 16) | b;
  const float2 r = fsub2(x, make_float2(__uint_as_float(a), __uint_as_float(b)));
  const __nv_bfloat162 t = __floats2bfloat162_rn(r.x, r.y);
  lo = *reinterpret_cast<const uint32_t*>(&t);
}

// ---- warp-level tf32 MMA (mma.sync m16n8k8) for the 16 x 16 blocks of the triangular solve.
// Fragments: A (16 x 8) a0 (g, t), a1 (g+8, t), a2 (g, t+4), a3 (g+8, t+4); B (8 x 8, k x n) b0 (t, g),
// b1 (t+4, g); C (16 x 8) c0 (g, 2t), c1 (g, 2t+1), c2 (g+8, 2t), c3 (g+8, 2t+1); g = lane / 4, t = lane % 4.
// x = hi + lo with hi = x with its low 13 mantissa bits cleared (exact in tf32) and lo = x - hi
// (exact in fp32); the MMA reads lo's top 19 bits, so lo carries about 10 more significant bits
// and hi*hi + hi*lo + lo*hi is ~2^-20 relative, with fp32 range.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = __float_as_uint(x) & 0xFFFFE000u;
  lo = __float_as_uint(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma_tf32_m16n8k8(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Shared-memory layouts of the solve, chosen so that the fragment loads below are free of bank
// conflicts: A (fragment rows g, columns t) at row stride 68; X with its columns XOR-permuted per
// row (swx), which serves both fragment shapes (rows g / columns t and rows t / columns g); the
// 16 x 16 scratch tiles, read as k x n operands only, at row stride 24.
constexpr int kLdA = 68, kLdY = 24;
__device__ __forceinline__ int swx(int r) {
  const int x = r & 7;
  return (((x & 3) << 1) | (x >> 2)) << 2;
}
struct LayA {
  const float* p;
  __device__ __forceinline__ float operator()(int r, int c) const { return p[r * kLdA + c]; }
};
struct LayX {
  float* p;
  __device__ __forceinline__ float& operator()(int r, int c) const { return p[r * 64 + (c ^ swx(r))]; }
};
struct LayY {
  float* p;
  __device__ __forceinline__ float& operator()(int r, int c) const { return p[r * kLdY + c]; }
};

// acc[term] += M1[r1.., c1..] (16 x 16) * M2[r2.., c2..] (16 x 8, k rows x n columns), with each
// operand split as x = hi + lo (both tf32): the terms hi*hi, hi*lo, lo*hi accumulate separately
// (independent MMA chains) and sum to ~fp32 accuracy with fp32 range.
template <class L1, class L2>
__device__ __forceinline__ void warp_gemm16x8_acc(float (&acc)[3][4], const L1& m1, int r1, int c1, const L2& m2,
                                                  int r2, int c2, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    const int ca = c1 + 8 * ks + t, rb = r2 + 8 * ks + t;
    const float af[4] = {m1(r1 + g, ca), m1(r1 + g + 8, ca), m1(r1 + g, ca + 4), m1(r1 + g + 8, ca + 4)};
    const float b0 = m2(rb, c2 + g), b1 = m2(rb + 4, c2 + g);
    uint32_t ah[4], al[4], bh0, bl0, bh1, bl1;
#pragma unroll
    for (int i = 0; i < 4; ++i) split_tf32(af[i], ah[i], al[i]);
    split_tf32(b0, bh0, bl0);
    split_tf32(b1, bh1, bl1);
    mma_tf32_m16n8k8(acc[0], ah, bh0, bh1);
    mma_tf32_m16n8k8(acc[1], ah, bl0, bl1);
    mma_tf32_m16n8k8(acc[2], al, bh0, bh1);
  }
}
// s * (acc[0] + (acc[1] + acc[2])) into dst[r0.., c0..] (16 x 8; every layout keeps columns 2j, 2j + 1
// adjacent)
template <class L>
__device__ __forceinline__ void store_acc16x8(const float (&acc)[3][4], float s, const L& dst, int r0, int c0,
                                              int lane) {
  const int g = lane >> 2, t = lane & 3;
  float v[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) v[e] = s * (acc[0][e] + (acc[1][e] + acc[2][e]));
  *reinterpret_cast<float2*>(&dst(r0 + g, c0 + 2 * t)) = make_float2(v[0], v[1]);
  *reinterpret_cast<float2*>(&dst(r0 + g + 8, c0 + 2 * t)) = make_float2(v[2], v[3]);
}

struct PrepMaps {
  CUtensorMap k, q, v;
};

// Next valid task index >= t (tasks: chunk-major, head-minor), or -1.  Task and chunk indices and
// sequence lengths below 2^31 (every practical problem) take 32-bit divisions.
__device__ __forceinline__ int64_t next_task(int64_t t, int64_t ntask, int64_t stride, const int32_t* plan,
                                             const int32_t* cu, int B, int64_t T, int H, int& h, int64_t& t0,
                                             int& n, int64_t& chunk) {
  const bool narrow = ntask < (int64_t(1) << 31) && T < (int64_t(1) << 31);
  for (; t < ntask; t += stride) {
    if (narrow) {
      const uint32_t c32 = (uint32_t)t / (uint32_t)H;
      chunk = c32;
      h = (int)((uint32_t)t - c32 * (uint32_t)H);
      if (cu == nullptr) {
        const uint32_t nc = (uint32_t)((T + 63) / 64);
        if (nc == 0) continue;
        const uint32_t b = c32 / nc, cs = c32 - b * nc;
        if ((int)b >= B) continue;
        t0 = (int64_t)b * T + (int64_t)cs * 64;
        const int64_t rem = T - (int64_t)cs * 64;
        n = (int)(rem < 64 ? rem : 64);
        return t;
      }
    } else {
      chunk = t / H;
      h = (int)(t - chunk * H);
    }
    int b;
    int64_t cseq;
    if (resolve_chunk(chunk, plan, cu, B, T, b, t0, n, cseq)) return t;
  }
  return -1;
}

// 2^x (the decays below are carried in log2 units: e^G = 2^(G log2 e))
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;

// g of this thread's 4 rows x 2 channels for one pass (rows past the sequence end read as 0).  Only
// the next pass consumes these registers, so the loads stay in flight through the current one.
__device__ __forceinline__ void load_g(float2 (&gv)[4], const float* __restrict__ g, int64_t t0, int n, int H, int h,
                                       int c, int rg) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 4 * rg + i;
    const float2 x = r < n ? __ldg(reinterpret_cast<const float2*>(g + ((size_t)(t0 + r) * H + h) * 128 + c))
                           : make_float2(0.f, 0.f);
    gv[i] = x;
  }
}

// Raw q, k, v tiles of a task (one transaction-counted arrival on `bar`).
__device__ __forceinline__ void tma_qkv(const PrepMaps& m, uint8_t* raw, uint64_t* bar, int h, int64_t t0) {
  mbar_arrive_expect_tx(bar, R_BYTES);
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    tma_load_2d(raw + R_K + 8192 * b, &m.k, h * 128 + 64 * b, (int)t0, bar);
    tma_load_2d(raw + R_Q + 8192 * b, &m.q, h * 128 + 64 * b, (int)t0, bar);
    tma_load_2d(raw + R_V + 8192 * b, &m.v, h * 128 + 64 * b, (int)t0, bar);
  }
}
// beta of a task into shared memory (whole issuer warp), then one arrival on `bar`.
__device__ __forceinline__ void stage_beta(const float* beta, float* sbeta, uint64_t* bar, int h, int64_t t0, int n,
                                           int H, int lane) {
  const float b0 = lane < n ? beta[(size_t)(t0 + lane) * H + h] : 0.f;
  const float b1 = lane + 32 < n ? beta[(size_t)(t0 + lane + 32) * H + h] : 0.f;
  sbeta[lane] = b0;
  sbeta[lane + 32] = b1;
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

template <bool GIVEUP>
__global__ void __launch_bounds__(kPrepThreads, 2)
kda_tc_chunk_prep(const __grid_constant__ PrepMaps maps, const float* __restrict__ g, const float* __restrict__ beta,
                  const int32_t* __restrict__ plan, const int32_t* __restrict__ cu, int B, int64_t T, int H,
                  int64_t ntask, uint8_t* __restrict__ records, unsigned int* __restrict__ err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* raw = sm;
  uint8_t* ops = sm + P_OPS;
  uint8_t* misc = sm + P_MISC;
  float* sBetaAll = reinterpret_cast<float*>(misc + M_BETA);
  float2* sTot = reinterpret_cast<float2*>(misc + M_TOT);      // [2][8][16]
  uint64_t* full = reinterpret_cast<uint64_t*>(misc + M_BAR);  // raw tiles landed + beta staged
  uint64_t* ops_ready = full + 1;                              // [2] pass operands written (256 arrivals)
  uint64_t* bar_ops = full + 3;                                // [2] pass MMAs done
  uint64_t* tt_ready = full + 5;                               // X written, A/M read (256 arrivals)
  uint64_t* bar_wu = full + 6;                                 // W / U_hat MMAs done
  uint64_t* bar_fin = full + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + M_BAR + 80);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + M_BAR + 84);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t stride = gridDim.x;
  int h, n;
  int64_t t0, chunk;
  griddep_launch_dependents();  // the state pass may be scheduled on SMs this grid leaves
  int64_t task = next_task(blockIdx.x, ntask, stride, plan, cu, B, T, H, h, t0, n, chunk);
  if (task < 0) return;

  if (warp == 0) {
    tmem_alloc(tmem_slot, kPrepTmemCols);
    tmem_relinquish();
  }
  if (tid == 32) {
    mbar_init(full, 2);
    mbar_init(&ops_ready[0], kCompute);
    mbar_init(&ops_ready[1], kCompute);
    mbar_init(&bar_ops[0], 1);
    mbar_init(&bar_ops[1], 1);
    mbar_init(tt_ready, kCompute);
    mbar_init(bar_wu, 1);
    mbar_init(bar_fin, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kIssuer) {
    // ======================== issuer warp
    // full: the raw tiles of a task (one transaction-counted arrival) and its beta (one arrival).
    // The tiles of the next task are loaded once the current task's last MMAs have read them;
    // the other CTA on the SM covers that latency.
    bool load_pending = false;  // a tile load has been issued and not yet waited for by the compute warps
    if (lane == 0) tma_qkv(maps, raw, full, h, t0);
    stage_beta(beta, sBetaAll, full, h, t0, n, H, lane);
    load_pending = true;
    bool ok = true;
    const uint32_t id_hh = idesc_bf16_f32(128, 192, false, false);  // X_h [Y_h ; Y_l]^T
    const uint32_t id_lh = idesc_bf16_f32(128, 96, false, false);   // X_l Y_h^T
    const uint32_t id_wu = idesc_f16(128, 64, /*a_mn=*/true, /*b_mn=*/false);
    const uint64_t dxh = smem_desc_sw128(smem_u32(ops + O_XH), 16, 1024);
    const uint64_t dxl = smem_desc_sw128(smem_u32(ops + O_XL), 16, 1024);
    const uint64_t dyh = smem_desc_sw128(smem_u32(ops + O_YH), 16, 1024);
    const uint64_t dtt = smem_desc_sw128(smem_u32(ops + O_TT), 16, 1024);
    const uint64_t dkh = smem_desc_sw128(smem_u32(raw + R_K), 8192, 1024);
    const uint64_t dvv = smem_desc_sw128(smem_u32(raw + R_V), 8192, 1024);
    uint32_t it = 0;
    while (task >= 0 && ok) {
      int nh = 0, nn = 0;
      int64_t nt0 = 0, nchunk = 0;
      const int64_t ntask_idx = next_task(task + stride, ntask, stride, plan, cu, B, T, H, nh, nt0, nn, nchunk);
      if (lane == 0) {
        for (int pass = 0; pass < 4 && ok; ++pass) {
          ok = wait_or_abort_t<GIVEUP>(&ops_ready[pass & 1], (uint32_t)((pass >> 1) & 1), abort_flag);
          if (!ok) break;
          if (pass == 0) load_pending = false;  // the compute warps have consumed this task's tiles
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint32_t off = (uint32_t)(32 * (pass & 1) + 16 * kk) * 2u;
            mma_bf16_ss(tmem + T_AM, desc_add(dxh, off), desc_add(dyh, off), id_hh, pass > 0 || kk > 0);
            mma_bf16_ss(tmem + T_AM, desc_add(dxl, off), desc_add(dyh, off), id_lh, true);
          }
          mma_commit(&bar_ops[pass & 1]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      if (ntask_idx >= 0) stage_beta(beta, sBetaAll + 64 * ((it + 1) & 1), full, nh, nt0, nn, H, lane);
      if (lane == 0) {
        ok = wait_or_abort_t<GIVEUP>(tt_ready, it & 1, abort_flag);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int k0 = 0; k0 < 64; k0 += 16) {
            mma_f16(tmem + T_W, desc_add(dkh, (k0 >> 3) * 1024), desc_add(dtt, k0 * 2), id_wu, k0 > 0);
            mma_f16(tmem + T_U, desc_add(dvv, (k0 >> 3) * 1024), desc_add(dtt, k0 * 2), id_wu, k0 > 0);
          }
          mma_commit(bar_wu);
          if (ntask_idx >= 0) {
            // the next task's tiles once these MMAs have read the current k and v
            ok = wait_or_abort_t<GIVEUP>(bar_wu, it & 1, abort_flag);
            if (ok) {
              tma_qkv(maps, raw, full, nh, nt0);
              load_pending = true;
            }
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      task = ntask_idx;
      h = nh; n = nn; t0 = nt0; chunk = nchunk;
      ++it;
    }
    if (lane == 0 && (!ok || *abort_flag)) {
      *abort_flag = 1;
      // let staged copies and issued MMAs drain (bounded) before TMEM is released
      if (load_pending) mbar_wait(full, it & 1);
      mma_commit(bar_fin);
      mbar_wait(bar_fin, 0);
    }
  } else {
    // ======================== compute warps
    const int cp = tid & 15, rg = tid >> 4;  // channel pair within a 32-channel pass, row group (4 rows)
    const int cl = 2 * cp;
    bool ok = true;
    uint32_t it = 0;
    float2 gcur[4];
    load_g(gcur, g, t0, n, H, h, cl, rg);
    while (task >= 0 && ok) {
      const float* sBeta = sBetaAll + 64 * (it & 1);
      uint8_t* rec = records + ((size_t)chunk * H + h) * kRecBytes;
      int nh = 0, nn = 0;
      int64_t nt0 = 0, nchunk = 0;
      const int64_t ntask_idx = next_task(task + stride, ntask, stride, plan, cu, B, T, H, nh, nt0, nn, nchunk);
      // the previous task's bulk copies out of the operand region have read it
      if (tid == 0) bulk_wait_read_all();
      // every break decision of the compute warps is made together (named barriers follow)
      ok = group_and(1, kCompute, wait_or_abort_t<GIVEUP>(full, it & 1, abort_flag));
      if (!ok) break;
      if (n < 64) {
        // a tail chunk: rows n..63 of the raw tiles (the next sequence's tokens, or the tensor's
        // zero fill) become zeros once, so that the passes need no per-row test
        const int nz = (64 - n) * 6 * 8;  // 16-byte pieces: rows x (k, q, v) x (two blocks) x 8
        for (int i = tid; i < nz; i += kCompute) {
          const int piece = i & 7, tile = (i >> 3) % 6, r = n + (i >> 3) / 6;
          *reinterpret_cast<uint4*>(raw + (uint32_t)tile * 8192u + (uint32_t)r * 128u + (uint32_t)piece * 16u) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        group_sync(1, kCompute);
      }

      // ---- four 32-channel passes
#pragma unroll 1
      for (int pass = 0; pass < 4; ++pass) {
        const int c = 32 * pass + cl;  // first of this thread's two channels
        float2 gnext[4];
        if (pass < 3) load_g(gnext, g, t0, n, H, h, c + 32, rg);
        else if (ntask_idx >= 0) load_g(gnext, g, nt0, nn, H, nh, cl, rg);
        float2 L[4], prev;
        {
          float2 run = make_float2(0.f, 0.f);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            run.x = fmaf(gcur[i].x, kLog2e, run.x);  // log2 units
            run.y = fmaf(gcur[i].y, kLog2e, run.y);
            L[i] = run;
          }
          // row groups 2w and 2w + 1 sit in lanes cp and cp + 16 of warp w: one exchange gives
          // the pair's total and, for the odd group, the sum of the group above it
          prev = make_float2(__shfl_xor_sync(0xffffffffu, run.x, 16), __shfl_xor_sync(0xffffffffu, run.y, 16));
          if (lane < 16) sTot[(pass & 1) * 128 + warp * 16 + cp] = make_float2(run.x + prev.x, run.y + prev.y);
        }
        if (pass >= 2) ok = wait_or_abort_t<GIVEUP>(&bar_ops[pass & 1], 0, abort_flag);
        ok = group_and(1, kCompute, ok);
        if (!ok) break;
        float2 off = lane < 16 ? make_float2(0.f, 0.f) : prev, cum = make_float2(0.f, 0.f), G15, G47, G63;
#pragma unroll
        for (int wi = 0; wi < 8; ++wi) {
          const float2 t = sTot[(pass & 1) * 128 + wi * 16 + cp];
          if (wi < warp) {
            off.x += t.x;
            off.y += t.y;
          }
          cum.x += t.x;
          cum.y += t.y;
          if (wi == 1) G15 = cum;
          if (wi == 5) G47 = cum;
        }
        G63 = cum;
        const bool first = rg < 8;  // rows < 32: reference row 15, else 47
        const float2 R = first ? G15 : G47;
        const float2 eR = make_float2(ex2(R.x), ex2(R.y));
        const float2 c3 = make_float2(ex2(G63.x - G47.x), ex2(G63.y - G47.y));
        if (rg == 0)
          *reinterpret_cast<float2*>(rec + kRecGC + c * 4) = make_float2(ex2(G63.x), ex2(G63.y));
        uint32_t qh2[4], kb2[4];
        const uint32_t kbyte = (uint32_t)(c & 63) * 2u;  // byte of channel c within its 128-byte row
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 4 * rg + i;
          const float2 G = fadd2(off, L[i]);
          const uint32_t ob = (uint32_t)r * 128u + ((((kbyte >> 4) ^ (uint32_t)r) & 7u) << 4) + (kbyte & 15u);
          const uint32_t toff = (uint32_t)(c >> 6) * 8192u + ob;
          uint32_t* pk = reinterpret_cast<uint32_t*>(raw + R_K + toff);
          uint32_t* pq = reinterpret_cast<uint32_t*>(raw + R_Q + toff);
          uint32_t* pv = reinterpret_cast<uint32_t*>(raw + R_V + toff);
          const float2 k2 = unpack_bf2(*pk), q2 = unpack_bf2(*pq), v2 = unpack_bf2(*pv);
          const float2 d1 = fsub2(G, R), d2 = fsub2(R, G);
          const float2 e1 = make_float2(ex2(d1.x), ex2(d1.y)), e2 = make_float2(ex2(d2.x), ex2(d2.y));
          uint32_t hi, lo;
          const uint32_t ob64 = ob + 64u * 128u;  // row 64 + r (same swizzle phase)
          const float2 ke1 = fmul2(k2, e1), qe1 = fmul2(q2, e1), ke2 = fmul2(k2, e2);
          split_bf16x2(ke1, hi, lo);
          *reinterpret_cast<uint32_t*>(ops + O_XH + ob) = hi;
          *reinterpret_cast<uint32_t*>(ops + O_XL + ob) = lo;
          split_bf16x2(qe1, hi, lo);
          *reinterpret_cast<uint32_t*>(ops + O_XH + ob64) = hi;
          *reinterpret_cast<uint32_t*>(ops + O_XL + ob64) = lo;
          split_bf16x2(ke2, hi, lo);
          *reinterpret_cast<uint32_t*>(ops + O_YH + ob) = hi;
          *reinterpret_cast<uint32_t*>(ops + O_YL + ob) = lo;
          float2 kb;
          if (first) {
            // rows < 32: k e^{G_47 - G} and k e^{G_C - G} from one exponential each (a factored
            // form can underflow while the product it feeds is O(1))
            const float2 d3 = fsub2(G47, G), d4 = fsub2(G63, G);
            split_bf16x2(fmul2(k2, make_float2(ex2(d3.x), ex2(d3.y))), hi, lo);
            *reinterpret_cast<uint32_t*>(ops + O_YH + ob64) = hi;
            *reinterpret_cast<uint32_t*>(ops + O_YL + ob64) = lo;
            kb = fmul2(k2, make_float2(ex2(d4.x), ex2(d4.y)));
          } else {
            kb = fmul2(ke2, c3);  // e^{G_C - G_47} >= e^{-80}: no underflow
          }
          const float2 qh = fmul2(qe1, eR);
          qh2[i] = pack_h2(qh.x, qh.y);  // q e^{G}
          kb2[i] = pack_h2(kb.x, kb.y);
          // Diag(beta) K_hat and Diag(beta) V as fp16, in place (T = X Diag(beta) is applied
          // through its right factor, so the solve's X is used as is)
          const float br = sBeta[r];
          const float2 b2 = make_float2(br, br);
          const float2 kh = fmul2(fmul2(ke1, eR), b2), vb = fmul2(v2, b2);
          *pk = pack_h2(kh.x, kh.y);
          *pv = pack_h2(vb.x, vb.y);
        }
        // Q_hat^T / K_bar^T rows (channel-major): lanes l and l ^ 16 hold rows 8w..8w+3 and
        // 8w+4..8w+7 of the same two channels; after one exchange each writes a full 16-byte
        // chunk (8 rows) of one channel.
        {
          const bool lower = lane < 16;
          const int ch = lower ? c : c + 1;
          const uint32_t chunk_off = row_chunk(ch, rg >> 1);
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            const uint32_t* x = a == 0 ? qh2 : kb2;
            const uint32_t c0a = __byte_perm(x[0], x[1], 0x5410), c0b = __byte_perm(x[2], x[3], 0x5410);  // channel c
            const uint32_t c1a = __byte_perm(x[0], x[1], 0x7632), c1b = __byte_perm(x[2], x[3], 0x7632);  // channel c+1
            const uint32_t s0 = lower ? c1a : c0a, s1 = lower ? c1b : c0b;
            const uint32_t r0 = __shfl_xor_sync(0xffffffffu, s0, 16), r1 = __shfl_xor_sync(0xffffffffu, s1, 16);
            const uint4 v = lower ? make_uint4(c0a, c0b, r0, r1) : make_uint4(r0, r1, c1a, c1b);
            *reinterpret_cast<uint4*>(rec + (a == 0 ? kRecQT : kRecKT) + chunk_off) = v;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&ops_ready[pass & 1]);
#pragma unroll
        for (int i = 0; i < 4; ++i) gcur[i] = gnext[i];
      }
      if (!ok) break;
      ok = group_and(1, kCompute, wait_or_abort_t<GIVEUP>(&bar_ops[1], 1, abort_flag));  // pass 3 (and all before) done
      if (!ok) break;
      tc_fence_after();

      // ---- TMEM -> A (fp32, beta-scaled strict lower) and M (fp16, into the record).
      // D[:, 0..95] + D[:, 96..191]; columns 0..63 hold the two diagonal 32 x 32 blocks, 64..95 the
      // off-diagonal block (rows >= 32, columns < 32).  Warp w: TMEM lane quadrant w & 3, s-half w >> 2.
      float* sA = reinterpret_cast<float*>(ops + O_SA);
      {
        const int q = warp & 3, hh = warp >> 2;
        const int lrow = 32 * q + lane;
        const int r = lrow & 63;
        const bool zero_half = (q & 1) == 0 && hh == 1;  // upper off-diagonal block
        const uint32_t c1 = (q & 1) == 0 ? 0u : (hh == 0 ? 64u : 32u);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          float val[16];
          if (zero_half) {
#pragma unroll
            for (int j = 0; j < 16; ++j) val[j] = 0.f;
          } else {
            float a1[16], a2[16];
            tmem_ld16(tmem_lane(tmem + T_AM, warp) + c1 + 16 * part, a1);
            tmem_ld16(tmem_lane(tmem + T_AM, warp) + c1 + 96u + 16 * part, a2);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) val[j] = a1[j] + a2[j];
          }
          const int s0 = 32 * hh + 16 * part;
          if (lrow < 64) {
            const float br = sBeta[r];
#pragma unroll
            for (int j = 0; j < 16; j += 4) {  // select, not mask-multiply
              float4 w;
              w.x = (s0 + j < r) ? br * val[j] : 0.f;
              w.y = (s0 + j + 1 < r) ? br * val[j + 1] : 0.f;
              w.z = (s0 + j + 2 < r) ? br * val[j + 2] : 0.f;
              w.w = (s0 + j + 3 < r) ? br * val[j + 3] : 0.f;
              *reinterpret_cast<float4*>(sA + r * kLdA + s0 + j) = w;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) val[j] = (s0 + j <= r) ? val[j] : 0.f;
            *reinterpret_cast<uint4*>(ops + O_MST + row_chunk(r, s0 >> 3)) = pack8_h(val);
            *reinterpret_cast<uint4*>(ops + O_MST + row_chunk(r, (s0 >> 3) + 1)) = pack8_h(val + 8);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      group_sync(1, kCompute);
      if (tid == 0) {  // M to the record in one bulk copy
        bulk_s2g(rec + kRecMM, ops + O_MST, 8192);
        bulk_commit();
      }

      // ---- X = (I + A)^-1: 16 x 16 diagonal blocks, then two levels of block merges
      {
        const LayA la{sA};
        const LayX lx{reinterpret_cast<float*>(ops + O_SX)};
        float* sY = reinterpret_cast<float*>(ops + O_SY);
        // diagonal blocks: one thread per column, substitution inside its 16 x 16 block
        if (tid < 64) {
          const int s_ = tid, r0 = s_ & ~15;
          float x[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int r = r0 + i;
            float acc0 = 0.f, acc1 = 0.f;  // two independent chains
#pragma unroll
            for (int j = 0; j < i; j += 2) {
              acc0 = fmaf(la(r, r0 + j), x[j], acc0);
              if (j + 1 < i) acc1 = fmaf(la(r, r0 + j + 1), x[j + 1], acc1);
            }
            x[i] = (r == s_) ? 1.f : ((r < s_) ? 0.f : -(acc0 + acc1));
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) lx(r0 + i, s_) = x[i];
        }
        group_sync(1, kCompute);
        // With X_[ii] the inverses of two adjacent diagonal blocks of (I + A), the block below them is
        //   X_[10] = -X_[11] A_[10] X_[00].
        // Level 1 merges the 16 x 16 pairs (0, 1) and (2, 3) (warps 0-3); level 2 merges the two
        // 32 x 32 halves, first Y = A[32:64, 0:32] X[0:32, 0:32], then X[32:64, 0:32] = -X[32:64, 32:64] Y
        // (warps 0-7).  Each warp computes one 8-column half of a 16 x 16 tile with warp-level tf32
        // MMAs and the three-term split.
        if (warp < 4) {
          const int b = 32 * (warp & 1), hn = 8 * (warp >> 1);
          const LayY ly{sY + (warp & 1) * 16 * kLdY};
          float acc[3][4] = {};
          warp_gemm16x8_acc(acc, la, b + 16, b, lx, b, b + hn, lane);
          store_acc16x8(acc, 1.f, ly, 0, hn, lane);
          __syncwarp();
          float z[3][4] = {};
          warp_gemm16x8_acc(z, lx, b + 16, b + 16, ly, 0, hn, lane);
          store_acc16x8(z, -1.f, lx, b + 16, b + hn, lane);
        }
        group_sync(1, kCompute);
        {
          const int tile = warp & 3, ti = tile >> 1, tj = tile & 1, hn = 8 * (warp >> 2);
          float acc[3][4] = {};
          if (tj == 0) warp_gemm16x8_acc(acc, la, 32 + 16 * ti, 0, lx, 0, hn, lane);
          warp_gemm16x8_acc(acc, la, 32 + 16 * ti, 16, lx, 16, 16 * tj + hn, lane);
          store_acc16x8(acc, 1.f, LayY{sY + tile * 16 * kLdY}, 0, hn, lane);
        }
        group_sync(1, kCompute);
        {
          const int tile = warp & 3, ti = tile >> 1, tj = tile & 1, hn = 8 * (warp >> 2);
          float acc[3][4] = {};
          if (ti == 1) warp_gemm16x8_acc(acc, lx, 48, 32, LayY{sY + tj * 16 * kLdY}, 0, hn, lane);
          warp_gemm16x8_acc(acc, lx, 32 + 16 * ti, 32 + 16 * ti, LayY{sY + tile * 16 * kLdY}, 0, hn, lane);
          store_acc16x8(acc, -1.f, lx, 32 + 16 * ti, 16 * tj + hn, lane);
        }
        group_sync(1, kCompute);
        // X -> fp16 row format [r][s] (zero above the diagonal)
        {
          const int r = tid >> 2, j0 = (tid & 3) * 2;  // two 8-column chunks per thread
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int j = j0 + jj;
            const float4 xa = *reinterpret_cast<const float4*>(&lx(r, 8 * j));
            const float4 xb = *reinterpret_cast<const float4*>(&lx(r, 8 * j + 4));
            const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int s_ = 8 * j + e;
              v[e] = (s_ <= r) ? xv[e] : 0.f;
            }
            *reinterpret_cast<uint4*>(ops + O_TT + row_chunk(r, j)) = pack8_h(v);
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(tt_ready);

      // ---- W^T = K_hat^T T^T, U_hat^T = V^T T^T (issued by the issuer warp) -> the record
      ok = group_and(1, kCompute, wait_or_abort_t<GIVEUP>(bar_wu, it & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      {
        // staged in the operand region (free now), then two bulk copies to the record
        const int row = (warp & 3) * 32 + lane;  // dk row (W^T, warps 0-3) or dv row (U_hat^T, warps 4-7)
        const uint32_t ta = tmem_lane(tmem + (warp < 4 ? T_W : T_U), warp);
        uint8_t* dst = ops + (warp < 4 ? 0 : 16384);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          float v[32];
          tmem_ld32(ta + 32 * part, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(dst + row_chunk(row, 4 * part + j)) = pack8_h(v + 8 * j);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      group_sync(1, kCompute);
      if (tid == 0) {
        bulk_s2g(rec + kRecWT, ops, 16384);
        bulk_s2g(rec + kRecUT, ops + 16384, 16384);
        bulk_commit();
      }
      task = ntask_idx;
      h = nh; n = nn; t0 = nt0; chunk = nchunk;
      ++it;
    }
    if (!ok) *abort_flag = 1;
    if (tid == 0) bulk_wait_all();  // record bulk copies complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) atomicOr(err, KDA_DEVERR_WAIT_TIMEOUT);
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kPrepTmemCols);
}

// ----------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D map over [rows = T_tot][cols = H * 128] with a {box_x, 64} box and 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int64_t rows, int H, int box_x) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)H * 128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)H * 128 * esize};
  cuuint32_t box[2] = {(cuuint32_t)box_x, 64};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <typename Tout>
cudaError_t launch_tc(const PrefillArgs& a, cudaStream_t st) {
  static DeviceOnce once;
  static int sm_count[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  cudaError_t e0 = once.run(dev, [dev] {
    cudaError_t e = cudaFuncSetAttribute(kda_tc_chunk_prep<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kPrepSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_tc_chunk_prep<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem);
    if (e != cudaSuccess) return e;
    return cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
  });
  if (e0 != cudaSuccess) return e0;
  const bool has_cu = a.cu_seqlens != nullptr;
  const int64_t nchunks = max_chunks(a.B, a.T, has_cu);
  int32_t* plan = static_cast<int32_t*>(a.workspace);
  uint8_t* records = static_cast<uint8_t*>(a.workspace) + plan_bytes(a.B);
  if (has_cu) {
    TraceScope ts("kda_plan", st);
    cudaError_t e = plan_launch(a.cu_seqlens, a.B, a.T_tot, plan, a.err, st);
    if (e != cudaSuccess) return e;
  }
  if (nchunks > 0 && a.T_tot > 0) {
    PrepMaps maps;
    if (!make_map(&maps.k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T_tot, a.H, 64) ||
        !make_map(&maps.q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T_tot, a.H, 64) ||
        !make_map(&maps.v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T_tot, a.H, 64))
      return cudaErrorInvalidValue;
    const int64_t ntask = nchunks * a.H;
    const int64_t slots = 2 * (int64_t)sm_count[dev];  // two CTAs per SM
    const int grid = (int)(ntask < slots ? ntask : slots);
    TraceScope ts("kda_tc_chunk_prep", st);
    auto* kernel = a.give_up ? kda_tc_chunk_prep<true> : kda_tc_chunk_prep<false>;
    kernel<<<grid, kPrepThreads, kPrepSmem, st>>>(maps, a.g, a.beta, plan, a.cu_seqlens, a.B, a.T, a.H, ntask, records,
                                                  a.err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // state pass, split into sequence segments when there are too few (sequence, head) chains (a
  // segment map runs its range as one segment)
  const int nseg = a.seg_P != nullptr ? 1 : prefill_tc_cp_segments(a.B, a.T, a.H);
  const int64_t maxc = (a.T + kChunk - 1) / kChunk;  // chunks of the longest possible sequence
  const int64_t seg_len = (maxc + nseg - 1) / nseg;
  float* cp = reinterpret_cast<float*>(records + align_up((size_t)nchunks * a.H * kRecBytes, 256));
  return scan_tc_launch(a, records, plan, cp, nseg, seg_len > 0 ? seg_len : 1, st);
}

}  // namespace

constexpr int64_t kCpMinChunks = 96;       // sequences shorter than this are never split
constexpr int64_t kCpMinSegChunks = 32;    // smallest segment
constexpr int64_t kCpLongChunks = 2048;    // from this length on, transitions may take two waves

int prefill_tc_cp_segments(int B, int64_t T, int H) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 1;
  const int64_t maxc = (T + kChunk - 1) / kChunk;
  const int64_t chains = (int64_t)B * H;
  // Worth it only when the chains leave at least half of the SMs idle and the sequences span
  // several minimum-size segments.  n segments cost 2 n - 3 transition runs of segment length per
  // chain (one run of segment 0 from h0, then P and b of every later segment but the last); for
  // moderate lengths keep them to one wave of CTAs, for very long sequences a second wave is
  // repaid by the shorter read-out pass.
  if (maxc < kCpMinChunks || chains * 2 > sms) return 1;
  int64_t n = maxc >= kCpLongChunks ? sms / chains : (sms / chains + 3) / 2;
  if (n > maxc / kCpMinSegChunks) n = maxc / kCpMinSegChunks;
  return n < 1 ? 1 : (int)n;
}

size_t prefill_tc_cp_bytes(int B, int64_t T, int H) {
  const int nseg = prefill_tc_cp_segments(B, T, H);
  return nseg > 1 ? (size_t)B * H * nseg * 3 * 128 * 128 * sizeof(float) : 0;
}

size_t prefill_tc_blob_bytes(int, int) { return kRecBytes; }
bool prefill_tc_supported(int dk, int dv) { return dk == 128 && dv == 128; }
cudaError_t prefill_tc_launch(const PrefillArgs& a, cudaStream_t st) {
  if (!a.bf16 || !prefill_tc_supported(a.dk, a.dv)) return cudaErrorNotSupported;
  return a.out_bf16 ? launch_tc<__nv_bfloat16>(a, st) : launch_tc<float>(a, st);
}

}  // namespace kda
