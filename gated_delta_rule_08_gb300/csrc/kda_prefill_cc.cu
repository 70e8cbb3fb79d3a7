// KDA chunked prefill for fp32 inputs and 64-dim heads: fp32 arithmetic on the CUDA cores, with
// the chunk products on the warp-level tensor cores as three-term tf32 MMAs (fp32-level accuracy).
//
// Kimi K3 report walk-through (kimi-k3-paper.pages.dev), section 2.5 / Eq. 4: the
// sequence is cut into chunks of C = 64 tokens; a parallel intra-chunk part is
// followed by a serial inter-chunk state pass.  Per chunk (positions r = 0..63,
// chunk-start state S0, G_r = cumulative log-decay inside the chunk):
//   A_rs  = beta_r sum_c k_rc k_sc exp(G_rc - G_sc)   (s < r)
//   M_rs  =        sum_c q_rc k_sc exp(G_rc - G_sc)   (s <= r)
//   T     = (I + A)^-1 Diag(beta),  W = T K_hat,  U_hat = T V,   K_hat = K * exp(G)
//   U     = U_hat - W S0
//   O     = Q_hat S0 + M U,                                       Q_hat = Q * exp(G)
//   S_C   = Diag(exp G_last) S0 + K_bar^T U,                      K_bar = K * exp(G_last - G)
//
// Decay numerics (section 3.1-3.2, Eq. 5: g > -5): a pairwise factor exp(G_r - G_s)
// is split as exp(G_r - R) exp(R - G_s) around a reference R so that A and M are
// plain matrix products.  One reference per 64-token chunk could need exp(+-320)
// (fp32 overflows past exp(88.7)), so the chunk uses two 32-token halves with centred
// references (positions 15 and 47: every factor within exp(+-80)) for the two
// diagonal 32x32 blocks, and the reference 47 for the off-diagonal block (its
// key-side factor exp(G_47 - G_s) <= 1 never overflows).  Entries outside the causal
// mask can overflow to inf and are discarded by selection, never multiplied by 0.
//
// Two kernels:
//   chunk_prep_cc : one CTA per (chunk, head), fully parallel; writes the chunk's
//                   W, U_hat, Q_hat, K_bar, M and exp(G_last) into the workspace.
//   chunk_scan_cc : one cluster of dv / 16 CTAs per (sequence, head), each walking the
//                   chunks in order with 16 value columns of the state (registers, and a
//                   transposed copy in shared memory); writes outputs (with the optional
//                   RMSNorm + sigmoid gate epilogue) and the final state.
#include <algorithm>

#include "kda_device.cuh"
#include "kda_internal.h"
#include "tc_ptx.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;

// One (chunk, head) record of the chunkwise operands in the workspace, laid out as the serial
// pass's shared-memory image: row pitches of 4 floats past a multiple of 32 keep that pass's MMA
// fragment loads free of bank conflicts, and one bulk copy moves W .. Gamma while a second moves
// the CTA's 16-column slice of U_hat (stored slice-major).
template <int DK, int DV>
struct CcBlob {
  static constexpr int NC = 16, NS = DV / NC;             // value-column slices of the serial pass
  static constexpr int PK = DK + 4, PR = 68, PC = NC + 4;  // row pitches in floats (16-byte multiples)
  static constexpr int W = 0;                              // [64][PK]
  static constexpr int QH = W + 64 * PK;                   // [64][PK]
  static constexpr int KBT = QH + 64 * PK;                 // K_bar transposed: [DK][PR]
  static constexpr int M = KBT + DK * PR;                  // [64][PR], lower triangular
  static constexpr int GC = M + 64 * PR;                   // exp(G_last): [DK]
  static constexpr int HEAD = GC + DK;                     // floats of the first bulk copy
  static constexpr int UH = HEAD;                          // [NS][64][PC]
  static constexpr int SLICE = 64 * PC;
  static constexpr int FLOATS = (UH + NS * SLICE + 63) / 64 * 64;
};


// ---- warp-level tf32 MMA (mma.sync m16n8k8).  Fragments (g = lane / 4, t = lane % 4):
// A (16 x 8) a0 (g, t), a1 (g+8, t), a2 (g, t+4), a3 (g+8, t+4); B (8 x 8, k x n) b0 (t, g), b1 (t+4, g);
// C (16 x 8) c0 (g, 2t), c1 (g, 2t+1), c2 (g+8, 2t), c3 (g+8, 2t+1).
__device__ __forceinline__ void mma_tf32(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// x = hi + lo: hi = x with its low 13 mantissa bits cleared (exact in tf32), lo = x - hi (exact in
// fp32, of which the MMA reads the top 19 bits): hi*hi + hi*lo + lo*hi is ~2^-20 relative
struct Tf32x2 {
  uint32_t hi, lo;
};
__device__ __forceinline__ Tf32x2 split_tf32(float x) {
  const uint32_t h = __float_as_uint(x) & 0xFFFFE000u;
  return {h, __float_as_uint(x - __uint_as_float(h))};
}
// D += A B with A (16 x 8) and B (8 x 8) given by their fp32 fragment values, three-term split
__device__ __forceinline__ void mma3(float (&c)[4], const float (&a)[4], const float (&bv)[2]) {
  const Tf32x2 a0 = split_tf32(a[0]), a1 = split_tf32(a[1]), a2 = split_tf32(a[2]), a3 = split_tf32(a[3]);
  const Tf32x2 b0 = split_tf32(bv[0]), b1 = split_tf32(bv[1]);
  mma_tf32(c, a0.lo, a1.lo, a2.lo, a3.lo, b0.hi, b1.hi);
  mma_tf32(c, a0.hi, a1.hi, a2.hi, a3.hi, b0.lo, b1.lo);
  mma_tf32(c, a0.hi, a1.hi, a2.hi, a3.hi, b0.hi, b1.hi);
}

template <int DK, int DV>
constexpr int prep_smem_floats() {
  constexpr int PM = (DK > DV ? DK : DV) + 4;
  return 64 * PM * 4 + 32 * PM + 64 * 65 + 3 * DK + 64;
}

// 2^x: the decays are carried in log2 units (e^G = 2^(G log2 e)), so every factor is one ex2
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;

// 16 bytes of raw input elements -> fp32 in shared memory
__device__ __forceinline__ void store_f32(float* dst, const uint4& raw, float) {
  *reinterpret_cast<float4*>(dst) = *reinterpret_cast<const float4*>(&raw);
}
__device__ __forceinline__ void store_f32(float* dst, const uint4& raw, __nv_bfloat16) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&raw);
  const float2 a = __bfloat1622float2(p[0]), b = __bfloat1622float2(p[1]);
  const float2 c = __bfloat1622float2(p[2]), d = __bfloat1622float2(p[3]);
  *reinterpret_cast<float4*>(dst) = make_float4(a.x, a.y, b.x, b.y);
  *reinterpret_cast<float4*>(dst + 4) = make_float4(c.x, c.y, d.x, d.y);
}

template <int DK, int DV, typename Tin>
__global__ void __launch_bounds__(kThreads, 1)
chunk_prep_cc(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
              const float* __restrict__ g, const float* __restrict__ beta,
              const int32_t* __restrict__ plan, const int32_t* __restrict__ cu, int B, int64_t T,
              int H, float* __restrict__ blob_base) {
  using L = CcBlob<DK, DV>;
  constexpr int PM = (DK > DV ? DK : DV) + 4;
  constexpr int VE = 16 / (int)sizeof(Tin);          // input elements per 16-byte load
  constexpr int NLK = 64 * DK / VE / kThreads;       // loads of k (and of q) per thread
  constexpr int NLV = 64 * DV / VE / kThreads;
  constexpr int NLG = 64 * DK / 4 / kThreads;
  extern __shared__ float4 smem4[];
  float* sG = reinterpret_cast<float*>(smem4);  // [64][PM] g, then G (log2 units), then K_hat
  float* sK = sG + 64 * PM;                      // [64][PM] k, then k * 2^(G - R(r))
  float* sQ = sK + 64 * PM;                      // [64][PM] q, then q * 2^(G - R(r)), then V
  float* sKR = sQ + 64 * PM;                     // [64][PM] k * 2^(R(s) - G), then T (pitch 65)
  float* sKX = sKR + 64 * PM;                    // [32][PM] k * 2^(G_47 - G), s < 32
  float* sA = sKX + 32 * PM;                     // [64][65]; first the cumulative sums' part totals
  float* sRef = sA + 64 * 65;                    // [3][DK] G at rows 15, 47, 63
  float* sBeta = sRef + 3 * DK;                  // [64]

  const int64_t chunk = blockIdx.x;
  const int h = blockIdx.y;
  int b, n;
  int64_t t0, cseq;
  if (!resolve_chunk(chunk, plan, cu, B, T, b, t0, n, cseq)) return;
  float* blob = blob_base + ((size_t)chunk * H + h) * L::FLOATS;
  const int tid = threadIdx.x;

  // 1. the raw tiles (rows n..63 zero; g = 0 there keeps G flat), every load issued before use;
  //    v stays in registers until its shared-memory buffer is free
  float4 rg[NLG];
  uint4 rk[NLK], rq[NLK], rv[NLV];
#pragma unroll
  for (int j = 0; j < NLG; ++j) {
    const int i = tid + j * kThreads, r = i / (DK / 4), c4 = (i % (DK / 4)) * 4;
    rg[j] = r < n ? __ldg(reinterpret_cast<const float4*>(g + ((size_t)(t0 + r) * H + h) * DK + c4))
                  : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int j = 0; j < NLK; ++j) {
    const int i = tid + j * kThreads, r = i / (DK / VE), e0 = (i % (DK / VE)) * VE;
    const size_t gi = ((size_t)(t0 + r) * H + h) * DK + e0;
    rk[j] = r < n ? __ldg(reinterpret_cast<const uint4*>(k + gi)) : make_uint4(0u, 0u, 0u, 0u);
    rq[j] = r < n ? __ldg(reinterpret_cast<const uint4*>(q + gi)) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int j = 0; j < NLV; ++j) {
    const int i = tid + j * kThreads, r = i / (DV / VE), e0 = (i % (DV / VE)) * VE;
    rv[j] = r < n ? __ldg(reinterpret_cast<const uint4*>(v + ((size_t)(t0 + r) * H + h) * DV + e0))
                  : make_uint4(0u, 0u, 0u, 0u);
  }
  if (tid < 64) sBeta[tid] = (tid < n) ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
#pragma unroll
  for (int j = 0; j < NLG; ++j) {
    const int i = tid + j * kThreads, r = i / (DK / 4), c4 = (i % (DK / 4)) * 4;
    *reinterpret_cast<float4*>(&sG[r * PM + c4]) =
        make_float4(rg[j].x * kLog2e, rg[j].y * kLog2e, rg[j].z * kLog2e, rg[j].w * kLog2e);
  }
#pragma unroll
  for (int j = 0; j < NLK; ++j) {
    const int i = tid + j * kThreads, r = i / (DK / VE), e0 = (i % (DK / VE)) * VE;
    store_f32(&sK[r * PM + e0], rk[j], Tin());
    store_f32(&sQ[r * PM + e0], rq[j], Tin());
  }
  __syncthreads();

  // 2. cumulative log-decay per channel: each of the 256 / DK parts of a channel's rows sums its
  //    own rows, then adds the totals of the parts above it
  {
    constexpr int P = kThreads / DK, RP = 64 / P;
    const int c = tid % DK, part = tid / DK;
    float run = 0.f;
#pragma unroll
    for (int i = 0; i < RP; ++i) {
      float& x = sG[(part * RP + i) * PM + c];
      run += x;
      x = run;
    }
    sA[part * DK + c] = run;
    __syncthreads();
    float off = 0.f;
    for (int p = 0; p < part; ++p) off += sA[p * DK + c];
    if (part > 0)
#pragma unroll
      for (int i = 0; i < RP; ++i) sG[(part * RP + i) * PM + c] += off;
    __syncthreads();
    if (tid < DK) {
      sRef[tid] = sG[15 * PM + tid];
      sRef[DK + tid] = sG[47 * PM + tid];
      sRef[2 * DK + tid] = sG[63 * PM + tid];
    }
    __syncthreads();
  }

  // 3. K_bar^T = (k * 2^(G_63 - G))^T into the record (rows fastest, for coalesced stores) and
  //    exp(G_last); then the reference-scaled operands of A and M, K_hat and Q_hat, each element
  //    in place by the one thread that owns it
  for (int idx = tid; idx < 64 * DK; idx += kThreads) {
    const int r = idx % 64, c = idx / 64;
    blob[L::KBT + c * L::PR + r] = sK[r * PM + c] * ex2(sRef[2 * DK + c] - sG[r * PM + c]);
  }
  if (tid < DK) blob[L::GC + tid] = ex2(sRef[2 * DK + tid]);
  __syncthreads();
  for (int idx = tid; idx < 64 * DK; idx += kThreads) {
    const int r = idx / DK, c = idx % DK;
    const float G = sG[r * PM + c], R = sRef[(r < 32 ? 0 : DK) + c];
    const float kv = sK[r * PM + c], qv = sQ[r * PM + c];
    const float ef = ex2(G - R), eG = ex2(G);
    sK[r * PM + c] = kv * ef;
    sQ[r * PM + c] = qv * ef;
    sKR[r * PM + c] = kv * ex2(R - G);
    if (r < 32) sKX[r * PM + c] = kv * ex2(sRef[DK + c] - G);
    sG[r * PM + c] = kv * eG;
    blob[L::QH + r * L::PK + c] = qv * eG;
  }
  __syncthreads();

  // 4. A (strict lower, row-scaled by beta) and M (lower incl. diagonal) as three-term tf32 MMAs:
  //    A = K_L K_R^T and M = Q_L K_R^T, with K_X in place of K_R for the off-diagonal block (rows
  //    >= 32, columns < 32); the upper off-diagonal block is masked and neither computed nor read.
  //    Warps 0-3 take A's 24 tiles of 16 x 8, warps 4-7 M's.
  const int warp = tid >> 5, lane = tid & 31, fg = lane >> 2, ft = lane & 3;  // MMA fragment row / column
  {
    const bool isM = warp >= 4;
    const float* X = isM ? sQ : sK;
    for (int q = 0; q < 6; ++q) {
      const int ti = (warp & 3) + 4 * q;  // tiles 0..7: rows 0-31, columns 0-31; 8..23: rows 32-63
      const int mi = ti < 8 ? (ti >> 2) : 2 + ((ti - 8) >> 3);
      const int ni = ti < 8 ? (ti & 3) : ((ti - 8) & 7);
      const float* Y = (mi >= 2 && ni < 4) ? sKX : sKR;
      const int ra = 16 * mi + fg, sb = 8 * ni + fg;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int kk = 0; kk < DK; kk += 8) {
        const float a[4] = {X[ra * PM + kk + ft], X[(ra + 8) * PM + kk + ft], X[ra * PM + kk + ft + 4],
                            X[(ra + 8) * PM + kk + ft + 4]};
        const float bv[2] = {Y[sb * PM + kk + ft], Y[sb * PM + kk + ft + 4]};
        mma3(acc, a, bv);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = ra + 8 * (e >> 1), sc = 8 * ni + 2 * ft + (e & 1);
        if (isM) blob[L::M + r * L::PR + sc] = (sc <= r) ? acc[e] : 0.f;
        else sA[r * 65 + sc] = (sc < r) ? sBeta[r] * acc[e] : 0.f;
      }
    }
  }
  __syncthreads();

  // 5. V into shared memory (over q * 2^(G - R)), and T = (I + A)^-1 Diag(beta) by blocks:
  //    X = (I + A)^-1 is unit lower triangular; its four 16 x 16 diagonal blocks come from forward
  //    substitution, and each off-diagonal block from the two above it on the diagonal,
  //    X_10 = -X_11 A_10 X_00, first for the 16-row pairs (0, 1) and (2, 3), then for the 32-row
  //    halves.  X and then T sit over k * 2^(R - G) (pitch 65); the products' intermediate
  //    Y = A_10 X_00 over k * 2^(G_47 - G) (pitch 33).
  float* sV = sQ;
#pragma unroll
  for (int j = 0; j < NLV; ++j) {
    const int i = tid + j * kThreads, r = i / (DV / VE), e0 = (i % (DV / VE)) * VE;
    store_f32(&sV[r * PM + e0], rv[j], Tin());
  }
  float* sT = sKR;
  float* sY = sKX;
  {
    // diagonal blocks: thread = (block bi, column s, part p); X[b + r][b + s] for the rows r of the
    // block, the sum over j split four ways (j = 4 p .. 4 p + 3) and combined by two shuffles
    const int p = tid & 3, s = (tid >> 2) & 15, bi = tid >> 6, b = 16 * bi;
    float x[4] = {0.f, 0.f, 0.f, 0.f};  // x[jj] = X[b + 4 p + jj][b + s]
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
        if (4 * p + jj < r) acc = fmaf(sA[(b + r) * 65 + b + 4 * p + jj], x[jj], acc);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      const float xv = (r == s) ? 1.f : ((r < s) ? 0.f : -acc);
      if (p == (r >> 2)) x[r & 3] = xv;
    }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) sT[(b + 4 * p + jj) * 65 + b + s] = x[jj];
    // the blocks above the diagonal are zero
    for (int i = tid; i < 64 * 64; i += kThreads) {
      const int r = i >> 6, c = i & 63;
      if ((c >> 4) > (r >> 4)) sT[r * 65 + c] = 0.f;
    }
  }
  __syncthreads();
  {
    // 16-row pairs q = 0, 1 (blocks 2q, 2q + 1): Y_q = A[16(2q+1) + r][16(2q) + k] X[16(2q) + k][16(2q) + c]
    const int q = tid >> 7, r = tid & 15, c2 = ((tid >> 4) & 7) * 2;
    const int r0 = 16 * (2 * q + 1), c0 = 16 * (2 * q);
    float y0 = 0.f, y1 = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float a = sA[(r0 + r) * 65 + c0 + k];
      y0 = fmaf(a, sT[(c0 + k) * 65 + c0 + c2], y0);
      y1 = fmaf(a, sT[(c0 + k) * 65 + c0 + c2 + 1], y1);
    }
    sY[q * 16 * 33 + r * 33 + c2] = y0;
    sY[q * 16 * 33 + r * 33 + c2 + 1] = y1;
    __syncthreads();
    // X[16(2q+1) + r][16(2q) + c] = -X[16(2q+1) + r][16(2q+1) + k] Y_q[k][c]
    float z0 = 0.f, z1 = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float xr = sT[(r0 + r) * 65 + r0 + k];
      z0 = fmaf(xr, sY[q * 16 * 33 + k * 33 + c2], z0);
      z1 = fmaf(xr, sY[q * 16 * 33 + k * 33 + c2 + 1], z1);
    }
    sT[(r0 + r) * 65 + c0 + c2] = -z0;
    sT[(r0 + r) * 65 + c0 + c2 + 1] = -z1;
  }
  __syncthreads();
  {
    // 32-row halves: Y = A[32 + r][k] X[k][c] (k, c < 32), then X[32 + r][c] = -X[32 + r][32 + k] Y[k][c];
    // thread = (row r = lane, four columns of a warp-uniform group)
    const int r = tid & 31, c4 = (tid >> 5) * 4;
    float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      const float a = sA[(32 + r) * 65 + k];
#pragma unroll
      for (int e = 0; e < 4; ++e) y[e] = fmaf(a, sT[k * 65 + c4 + e], y[e]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) sY[r * 33 + c4 + e] = y[e];
    __syncthreads();
    float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      const float xr = sT[(32 + r) * 65 + 32 + k];
#pragma unroll
      for (int e = 0; e < 4; ++e) z[e] = fmaf(xr, sY[k * 33 + c4 + e], z[e]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) sT[(32 + r) * 65 + c4 + e] = -z[e];
  }
  __syncthreads();
  // T = X Diag(beta), re-laid at row pitch 68 over k * 2^(G - R) (free after the A/M products)
  float* sT2 = sK;
  for (int i = tid; i < 64 * 64; i += kThreads) {
    const int r = i >> 6, c = i & 63;
    sT2[r * 68 + c] = sT[r * 65 + c] * sBeta[c];
  }
  __syncthreads();

  // 6. [W | U_hat] = T [K_hat | V] as three-term tf32 MMAs (T lower triangular: tile row block mi
  //    stops at column 16 mi + 15); warp w takes every eighth 16 x 8 tile
  {
    constexpr int NT = 4 * (DK + DV) / 8;
    for (int q = 0; q < NT / 8; ++q) {
      const int ti = warp + 8 * q;
      const int mi = ti & 3, nj = ti >> 2;
      const bool isW = nj < DK / 8;
      const float* Bm = isW ? sG : sV;
      const int nb = isW ? nj : nj - DK / 8;
      const int ra = 16 * mi + fg;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int kk = 0; kk < 16 * mi + 16; kk += 8) {
        const float a[4] = {sT2[ra * 68 + kk + ft], sT2[(ra + 8) * 68 + kk + ft], sT2[ra * 68 + kk + ft + 4],
                            sT2[(ra + 8) * 68 + kk + ft + 4]};
        const float bv[2] = {Bm[(kk + ft) * PM + 8 * nb + fg], Bm[(kk + ft + 4) * PM + 8 * nb + fg]};
        mma3(acc, a, bv);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = ra + 8 * (e >> 1), j = 8 * nb + 2 * ft + (e & 1);
        if (isW) blob[L::W + r * L::PK + j] = acc[e];
        else blob[L::UH + (j / L::NC) * L::SLICE + r * L::PC + j % L::NC] = acc[e];
      }
    }
  }
}

// ------------------------------------------------------------------ serial state pass
// The recurrence is separable in the value columns: column j of U, O and S involves only column
// j of U_hat and of S.  A chain therefore runs as a thread-block cluster of NS = dv / 16 CTAs,
// each owning 16 value columns of the state; every CTA reads the chunk's W, Q_hat, K_bar^T and M
// (the repeats hit L2).  The one exchange is the RMSNorm's sum of squares over a token's dv
// outputs (gate epilogue only): each CTA stores its 16-column partial sums into every CTA of the
// cluster (distributed shared memory) by st.async, whose bytes complete the peer's mbarrier
// phase, and normalises a chunk's outputs one chunk later, so that the exchange overlaps the next
// chunk's products.  The next chunk's record arrives by bulk copy while the current one is used
// (two stages where shared memory allows).
template <int DK, int DV>
struct CcScan {
  using L = CcBlob<DK, DV>;
  static constexpr int NSLOT = 4;   // partial-sum slots in flight (a peer runs at most 2 chunks ahead)
  static constexpr int PST = DK + 4, PUT = 68;        // pitches of the transposed state and U
  static constexpr int STAGE = L::HEAD + L::SLICE;    // record image + this CTA's U_hat slice
  // state, U, partial sums, slots, and the gate tiles of two chunks (room for fp32 gates)
  static constexpr int EXTRA = L::NC * PST + L::NC * PUT + 4 * 64 + NSLOT * L::NS * 64 + 2 * 64 * L::NC;
  static constexpr size_t bytes(int stages) {
    return ((size_t)stages * STAGE + EXTRA) * sizeof(float) + (2 + NSLOT) * sizeof(uint64_t);
  }
  static constexpr int STAGES = bytes(2) <= 227 * 1024 ? 2 : 1;
  static constexpr size_t SMEM = bytes(STAGES);
};


__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// the address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// an asynchronous 4-byte store into a peer's shared memory that, once it lands, counts its bytes
// against the peer's mbarrier (both addresses in the peer CTA); the sender does not wait for it
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(addr), "f"(v),
               "r"(bar)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(tc::smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int DK, int DV, typename Tin, typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
chunk_scan_cc(const float* __restrict__ blob_base, const int32_t* __restrict__ plan,
              const int32_t* __restrict__ cu, int B, int64_t T, int H, const float* __restrict__ h0,
              float* __restrict__ hT, Tout* __restrict__ out, const Tin* __restrict__ gate,
              const float* __restrict__ norm_w, float eps, float* __restrict__ ckpt, int64_t ckpt_chunks,
              unsigned int* __restrict__ err) {
  using L = CcBlob<DK, DV>;
  using Sc = CcScan<DK, DV>;
  constexpr int NC = L::NC, NS = L::NS, PK = L::PK, PR = L::PR, PC = L::PC, KR = DK / 64;
  constexpr int PST = Sc::PST, PUT = Sc::PUT, NSLOT = Sc::NSLOT, STAGES = Sc::STAGES;
  extern __shared__ float4 smem4[];
  float* stages = reinterpret_cast<float*>(smem4);
  float* sST = stages + STAGES * Sc::STAGE;  // [NC][PST] this CTA's 16 state columns, transposed
  float* sUT = sST + NC * PST;               // [NC][PUT] U, transposed
  float* sPart = sUT + NC * PUT;             // [2][64] sums of squares of each 8-column half
  float* sSlot = sPart + 4 * 64;             // [NSLOT][NS][64] 16-column sums from each CTA
  Tin* sGate = reinterpret_cast<Tin*>(sSlot + NSLOT * NS * 64);          // [2][64][NC] gate tiles
  uint64_t* full = reinterpret_cast<uint64_t*>(sSlot + NSLOT * NS * 64 + 2 * 64 * NC);  // [2] stage landed
  uint64_t* slot_bar = full + 2;                                         // [NSLOT] slot filled

  const int tid = threadIdx.x;
  if (cu != nullptr && plan[B + 1] == 0) return;  // invalid cu_seqlens: every CTA returns
  const int slice = (int)cluster_ctarank();       // = blockIdx.x % NS
  const int h = blockIdx.y;
  const int b = sequence_of_rank(blockIdx.x / NS, plan, cu, B);
  int64_t first_chunk, t_begin, len;
  const int64_t nchunks = sequence_chunks(b, plan, cu, B, T, first_chunk, t_begin, len);
  const bool epi = gate != nullptr;
  const int col0 = slice * NC;

  if (tid == 0) {
    tc::mbar_init(&full[0], 1);
    tc::mbar_init(&full[1], 1);
    for (int i = 0; i < NSLOT; ++i) tc::mbar_init(&slot_bar[i], 1);  // armed per chunk, filled by st.async
    tc::mbar_fence_init();
  }
  if (epi) cluster_sync_all();  // every CTA's barriers exist before the first remote arrival
  else __syncthreads();

  // Warp w owns the 16 x 8 output tile (rows 16 m .. 16 m + 15 of the chunk, columns 8 n .. 8 n + 7
  // of the slice), m = w / 2, n = w % 2, of W S, Q_hat S, M U and U, and the state tiles (rows
  // 16 (m + 4 j), the same columns) of the update K_bar^T U, j < dk / 64.
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int m = warp >> 1, n = warp & 1;
  const int rA = 16 * m + g, cA = 8 * n + 2 * t;  // this lane's first C element (row, slice column)
  const size_t soff = ((size_t)b * H + h) * DK * DV;
  float sreg[KR][4];  // state tiles, C layout
#pragma unroll
  for (int j = 0; j < KR; ++j) {
    const int k0 = 16 * (m + 4 * j) + g;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = k0 + 8 * (e >> 1), c = cA + (e & 1);
      sreg[j][e] = h0 ? h0[soff + (size_t)k * DV + col0 + c] : 0.f;
      sST[c * PST + k] = sreg[j][e];
    }
  }
  const int64_t ck_base = ckpt != nullptr ? checkpoint_base(b, cu, T, 64 * ckpt_chunks) : 0;
  float nw[2] = {1.f, 1.f};
  if (epi && norm_w != nullptr) {
    nw[0] = norm_w[col0 + cA];
    nw[1] = norm_w[col0 + cA + 1];
  }

  // one thread stages chunk c's record image and U_hat slice
  auto issue = [&](int64_t c) {
    const int st = STAGES == 2 ? (int)(c & 1) : 0;
    const float* blob = blob_base + ((size_t)(first_chunk + c) * H + h) * L::FLOATS;
    float* d = stages + st * Sc::STAGE;
    tc::fence_proxy_async_smem();
    tc::mbar_arrive_expect_tx(&full[st], Sc::STAGE * sizeof(float));
    tc::bulk_g2s(d, blob, L::HEAD * sizeof(float), &full[st]);
    tc::bulk_g2s(d + L::HEAD, blob + L::UH + slice * L::SLICE, L::SLICE * sizeof(float), &full[st]);
  };

  bool waits_ok = true;
  auto wait_bar = [&](uint64_t* bar, uint32_t parity, bool cluster_scope) {
    if (!waits_ok) return;
    bool ok = false;
    for (uint32_t i = 0; i < 20000000u && !ok; ++i)
      ok = cluster_scope ? mbar_try_wait_cluster(bar, parity) : tc::mbar_try_wait(bar, parity);
    if (!ok) {
      atomicOr(err, KDA_DEVERR_WAIT_TIMEOUT);
      waits_ok = false;
    }
  };
  auto rows_of = [&](int64_t c) {
    const int64_t rem = len - 64 * c;
    return (int)(rem < 64 ? rem : 64);
  };
  // epilogue: the 16-column sum of squares of chunk c's row tid (both 8-column halves) into slot
  // c % NSLOT of every CTA of the cluster; one thread per row
  auto send = [&](int64_t c) {
    const float ss = sPart[tid] + sPart[64 + tid];
    const int sl = (int)(c % NSLOT);
    const uint32_t slot = tc::smem_u32(&sSlot[(sl * NS + slice) * 64 + tid]);
    const uint32_t bar = tc::smem_u32(&slot_bar[sl]);
#pragma unroll
    for (int p = 0; p < NS; ++p) st_async_f32(cluster_map(slot, (uint32_t)p), ss, cluster_map(bar, (uint32_t)p));
  };
  // epilogue: chunk c's gate tile (this CTA's 16 columns) into slot c & 1, by cp.async
  constexpr int PPR = NC * (int)sizeof(Tin) / 16;  // 16-byte pieces per row
  auto stage_gate = [&](int64_t c) {
    if (tid < 64 * PPR) {
      const int rr = tid / PPR, pc = tid % PPR;
      if (rr < rows_of(c))
        cp_async16(reinterpret_cast<char*>(sGate + ((int)(c & 1) * 64 + rr) * NC) + pc * 16,
                   reinterpret_cast<const char*>(gate + ((size_t)(t_begin + 64 * c + rr) * H + h) * DV + col0) +
                       pc * 16);
    }
    cp_async_commit();
  };
  // chunk c's outputs (this lane's rows rA, rA + 8 and columns cA, cA + 1), normalised with every
  // CTA's partial sums (epilogue) or as they are
  auto store = [&](int64_t c, const float (&o)[4]) {
    const int nrows = rows_of(c);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = rA + 8 * hr;
      float y0 = o[2 * hr], y1 = o[2 * hr + 1];
      if (epi) {
        const int sl = (int)(c % NSLOT);
        if (hr == 0) wait_bar(&slot_bar[sl], (uint32_t)((c / NSLOT) & 1), true);
        float tot = 0.f;
#pragma unroll
        for (int p = 0; p < NS; ++p) tot += sSlot[(sl * NS + p) * 64 + r];
        const float scale = rsqrtf(tot / (float)DV + eps);
        const Tin* gr = sGate + ((int)(c & 1) * 64 + r) * NC + cA;
        y0 = y0 * scale * nw[0] * sigmoidf_(to_f32(gr[0]));
        y1 = y1 * scale * nw[1] * sigmoidf_(to_f32(gr[1]));
      }
      if (r < nrows) {
        Tout* po = out + ((size_t)(t_begin + 64 * c + r) * H + h) * DV + col0 + cA;
        po[0] = from_f32<Tout>(y0);
        po[1] = from_f32<Tout>(y1);
      }
    }
  };

  if (tid == 0 && nchunks > 0) issue(0);
  float o_prev[4] = {0.f, 0.f, 0.f, 0.f};
  for (int64_t c = 0; c < nchunks; ++c) {
    const int st = STAGES == 2 ? (int)(c & 1) : 0;
    const float* d = stages + st * Sc::STAGE;
    __syncthreads();  // chunk c - 1 is done with the state, U, the partial sums and (one stage) the record
    if (tid == 0) {
      if (STAGES == 2 && c + 1 < nchunks) issue(c + 1);
      if (STAGES == 1 && c > 0) issue(c);
    }
    if (epi) {
      stage_gate(c);  // read when chunk c's outputs leave, at the end of chunk c + 1
      if (c > 0) {
        // slot (c - 1) % NSLOT expects 64 rows from each of the NS CTAs (bytes counted on arrival)
        if (tid == 0) tc::mbar_arrive_expect_tx(&slot_bar[(c - 1) % NSLOT], 64 * NS * (uint32_t)sizeof(float));
        if (tid < 64) send(c - 1);
      }
    }
    wait_bar(&full[st], (uint32_t)((c / STAGES) & 1), false);

    // W S and Q_hat S for this warp's tile; B = S (k x slice column) from the transposed state
    float ws[4] = {0.f, 0.f, 0.f, 0.f}, o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
    for (int kk = 0; kk < DK; kk += 8) {
      const float bv[2] = {sST[(8 * n + g) * PST + kk + t], sST[(8 * n + g) * PST + kk + t + 4]};
      const float aw[4] = {d[L::W + rA * PK + kk + t], d[L::W + (rA + 8) * PK + kk + t],
                           d[L::W + rA * PK + kk + t + 4], d[L::W + (rA + 8) * PK + kk + t + 4]};
      const float aq[4] = {d[L::QH + rA * PK + kk + t], d[L::QH + (rA + 8) * PK + kk + t],
                           d[L::QH + rA * PK + kk + t + 4], d[L::QH + (rA + 8) * PK + kk + t + 4]};
      mma3(ws, aw, bv);
      mma3(o, aq, bv);
    }
    // U = U_hat - W S, transposed into shared memory
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = rA + 8 * (e >> 1), cl = cA + (e & 1);
      sUT[cl * PUT + r] = d[L::HEAD + r * PC + cl] - ws[e];
    }
    if (epi) cp_async_wait<1>();  // this thread's copies of chunk c - 1's gate have landed
    __syncthreads();  // U complete; every read of the state done; the gate of chunk c - 1 in place

    // O += M U (M lower triangular: tile m stops at column 16 m + 15) and
    // S = Diag(exp G_last) S + K_bar^T U, B = U (s x slice column) from the transposed U
    float acc[KR][4];
#pragma unroll
    for (int j = 0; j < KR; ++j) {
      const int k0 = 16 * (m + 4 * j) + g;
      const float gm0 = d[L::GC + k0], gm1 = d[L::GC + k0 + 8];
      acc[j][0] = sreg[j][0] * gm0;
      acc[j][1] = sreg[j][1] * gm0;
      acc[j][2] = sreg[j][2] * gm1;
      acc[j][3] = sreg[j][3] * gm1;
    }
#pragma unroll 2
    for (int kk = 0; kk < 64; kk += 8) {
      const float bv[2] = {sUT[(8 * n + g) * PUT + kk + t], sUT[(8 * n + g) * PUT + kk + t + 4]};
      if (kk < 16 * m + 16) {  // warp-uniform
        const float am[4] = {d[L::M + rA * PR + kk + t], d[L::M + (rA + 8) * PR + kk + t],
                             d[L::M + rA * PR + kk + t + 4], d[L::M + (rA + 8) * PR + kk + t + 4]};
        mma3(o, am, bv);
      }
#pragma unroll
      for (int j = 0; j < KR; ++j) {
        const int k0 = 16 * (m + 4 * j) + g;
        const float ak[4] = {d[L::KBT + k0 * PR + kk + t], d[L::KBT + (k0 + 8) * PR + kk + t],
                             d[L::KBT + k0 * PR + kk + t + 4], d[L::KBT + (k0 + 8) * PR + kk + t + 4]};
        mma3(acc[j], ak, bv);
      }
    }
#pragma unroll
    for (int j = 0; j < KR; ++j) {
      const int k0 = 16 * (m + 4 * j) + g;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sreg[j][e] = acc[j][e];
        sST[(cA + (e & 1)) * PST + k0 + 8 * (e >> 1)] = acc[j][e];
      }
    }

    // state checkpoint after every ckpt_chunks full chunks (this lane's own elements)
    if (ckpt != nullptr && (c + 1) % ckpt_chunks == 0 && (c + 1) * 64 <= len) {
      float* dst = ckpt + ((size_t)(ck_base + (c + 1) / ckpt_chunks - 1) * H + h) * DK * DV;
#pragma unroll
      for (int j = 0; j < KR; ++j) {
        const int k0 = 16 * (m + 4 * j) + g;
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[(size_t)(k0 + 8 * (e >> 1)) * DV + col0 + cA + (e & 1)] = sreg[j][e];
      }
    }

    if (epi) {
      // this tile's 8-column sums of squares of rows rA and rA + 8 (over the four lanes of a row)
      float s0 = o[0] * o[0] + o[1] * o[1], s1 = o[2] * o[2] + o[3] * o[3];
      s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
      s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
      if (t == 0) {
        sPart[n * 64 + rA] = s0;
        sPart[n * 64 + rA + 8] = s1;
      }
      if (c > 0) store(c - 1, o_prev);
#pragma unroll
      for (int e = 0; e < 4; ++e) o_prev[e] = o[e];
    } else {
      store(c, o);
    }
  }
  if (epi && nchunks > 0) {
    const int64_t c = nchunks - 1;
    cp_async_wait<0>();
    __syncthreads();  // every column half's partial sums and the gate of the last chunk are in place
    if (tid == 0) tc::mbar_arrive_expect_tx(&slot_bar[c % NSLOT], 64 * NS * (uint32_t)sizeof(float));
    if (tid < 64) send(c);
    store(c, o_prev);
  }

  if (hT != nullptr)
#pragma unroll
    for (int j = 0; j < KR; ++j) {
      const int k0 = 16 * (m + 4 * j) + g;
#pragma unroll
      for (int e = 0; e < 4; ++e) hT[soff + (size_t)(k0 + 8 * (e >> 1)) * DV + col0 + cA + (e & 1)] = sreg[j][e];
    }
  if (epi) cluster_sync_all();  // no CTA leaves while a peer may still write into its shared memory
}

__global__ void plan_kernel(const int32_t* __restrict__ cu, int B, int64_t T_tot, int32_t* __restrict__ plan,
                            unsigned int* __restrict__ err) {
  // One block of 1024 threads: each thread owns a contiguous range of sequences.
  __shared__ int64_t part[32];
  __shared__ int bad;
  const int tid = threadIdx.x, nt = blockDim.x;
  if (tid == 0) bad = (cu[0] != 0);
  __syncthreads();
  const int per = (B + nt - 1) / nt;
  const int b0 = tid * per, b1 = min(B, b0 + per);
  int64_t local = 0;
  bool lbad = false;
  for (int b = b0; b < b1; ++b) {
    const int64_t a = cu[b], e = cu[b + 1];
    if (a < 0 || e < a || e > T_tot) lbad = true;
    else local += (e - a + 63) / 64;
  }
  if (lbad) atomicOr(&bad, 1);
  // exclusive scan of the per-thread chunk counts: within each warp by shuffles, then over the
  // warp totals
  const int lane = tid & 31, wid = tid >> 5, nw = nt >> 5;
  int64_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) part[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int64_t w = lane < nw ? part[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) part[lane] = w;  // inclusive totals of warps 0..lane
  }
  __syncthreads();
  if (tid == 0) {
    plan[B] = (int32_t)part[nw - 1];
    plan[B + 1] = bad ? 0 : 1;
    if (bad) atomicOr(err, KDA_DEVERR_BAD_SEQLENS);
  }
  int64_t acc = incl - local + (wid > 0 ? part[wid - 1] : 0);
  for (int b = b0; b < b1; ++b) {
    plan[b] = (int32_t)acc;
    const int64_t a = cu[b], e = cu[b + 1];
    if (a >= 0 && e >= a) acc += (e - a + 63) / 64;
  }
  // the sequences by decreasing length (ties by index), so that the serial pass starts its
  // longest chains first; O(B^2) rank count, the identity for large B
  __shared__ int32_t scu[kOrderMaxB + 1];
  const bool order = B <= kOrderMaxB;
  if (order)
    for (int i = tid; i <= B; i += nt) scu[i] = cu[i];
  __syncthreads();
  if (bad) return;  // the kernels that read the order return before it
  for (int b = b0; b < b1; ++b) {
    int r = b;
    if (order) {
      const int32_t lb = scu[b + 1] - scu[b];
      r = 0;
      for (int j = 0; j < B; ++j) {
        const int32_t lj = scu[j + 1] - scu[j];
        r += (lj > lb || (lj == lb && j < b)) ? 1 : 0;
      }
    }
    plan[B + 2 + r] = b;
  }
}

template <int DK, int DV, typename Tin, typename Tout>
cudaError_t launch_cc(const PrefillArgs& a, cudaStream_t st) {
  using Sc = CcScan<DK, DV>;
  const size_t prep_smem = prep_smem_floats<DK, DV>() * sizeof(float);
  static DeviceOnce once;  // per instantiation
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const cudaError_t e0 = once.run(dev, [prep_smem] {
    cudaError_t e = cudaFuncSetAttribute(chunk_prep_cc<DK, DV, Tin>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)prep_smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(chunk_scan_cc<DK, DV, Tin, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)Sc::SMEM);
  });
  if (e0 != cudaSuccess) return e0;
  const bool has_cu = a.cu_seqlens != nullptr;
  const int64_t nchunks = max_chunks(a.B, a.T, has_cu);
  int32_t* plan = static_cast<int32_t*>(a.workspace);
  float* blob = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + plan_bytes(a.B));
  if (has_cu) {
    TraceScope ts("kda_plan", st);
    cudaError_t e = plan_launch(a.cu_seqlens, a.B, a.T_tot, plan, a.err, st);
    if (e != cudaSuccess) return e;
  }
  if (nchunks > 0) {
    dim3 grid((unsigned)nchunks, (unsigned)a.H);
    TraceScope ts("kda_chunk_prep_cc", st);
    chunk_prep_cc<DK, DV, Tin><<<grid, kThreads, prep_smem, st>>>(
        static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v), a.g, a.beta,
        plan, a.cu_seqlens, a.B, a.T, a.H, blob);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // one cluster of NS CTAs (the value-column slices) per (sequence, head)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(CcBlob<DK, DV>::NS * a.B), (unsigned)a.H, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Sc::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CcBlob<DK, DV>::NS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  TraceScope ts("kda_chunk_scan_cc", st);
  return cudaLaunchKernelEx(&cfg, chunk_scan_cc<DK, DV, Tin, Tout>, static_cast<const float*>(blob),
                            static_cast<const int32_t*>(plan), a.cu_seqlens, a.B, a.T, a.H, a.h0, a.hT,
                            static_cast<Tout*>(a.out), static_cast<const Tin*>(a.epi.gate), a.epi.norm_weight,
                            a.epi.eps, a.ckpt, a.ckpt_chunks, a.err);
}

template <typename Tin, typename Tout>
cudaError_t launch_cc_dims(const PrefillArgs& a, cudaStream_t st) {
  if (a.dk == 128 && a.dv == 128) return launch_cc<128, 128, Tin, Tout>(a, st);
  if (a.dk == 64 && a.dv == 64) return launch_cc<64, 64, Tin, Tout>(a, st);
  if (a.dk == 128 && a.dv == 64) return launch_cc<128, 64, Tin, Tout>(a, st);
  if (a.dk == 64 && a.dv == 128) return launch_cc<64, 128, Tin, Tout>(a, st);
  return cudaErrorInvalidValue;
}

template <typename Tin>
cudaError_t launch_cc_out(const PrefillArgs& a, cudaStream_t st) {
  return a.out_bf16 ? launch_cc_dims<Tin, __nv_bfloat16>(a, st) : launch_cc_dims<Tin, float>(a, st);
}

}  // namespace

size_t prefill_cc_blob_bytes(int dk, int dv) {
  if (dk == 128 && dv == 128) return CcBlob<128, 128>::FLOATS * sizeof(float);
  if (dk == 64 && dv == 64) return CcBlob<64, 64>::FLOATS * sizeof(float);
  if (dk == 128 && dv == 64) return CcBlob<128, 64>::FLOATS * sizeof(float);
  if (dk == 64 && dv == 128) return CcBlob<64, 128>::FLOATS * sizeof(float);
  return 0;
}

cudaError_t plan_launch(const int32_t* cu_seqlens, int B, int64_t T_tot, int32_t* plan, unsigned int* err,
                        cudaStream_t st) {
  plan_kernel<<<1, 1024, 0, st>>>(cu_seqlens, B, T_tot, plan, err);
  return cudaGetLastError();
}

cudaError_t prefill_cc_launch(const PrefillArgs& a, cudaStream_t st) {
  return a.bf16 ? launch_cc_out<__nv_bfloat16>(a, st) : launch_cc_out<float>(a, st);
}

}  // namespace kda
