// KDA backward, chunkwise (products on the tensor cores as three-term tf32 warp MMAs, everything else
// in fp32): gradients of L = sum_t <dout_t, o_t> + <dhT, hT> with
// respect to q, k, v, g, beta and h0, for the prefill recurrence without epilogue.
//
// Kimi K3: Open Frontier Intelligence (kimi-k3-paper.pages.dev), section 2.5 / Eq. 4 gives the
// chunk form of the forward: with chunk-start state S0, G the chunk's inclusive cumulative decay,
//   A_rs = beta_r sum_c k_rc k_sc e^{G_rc - G_sc} (s < r),  M_rs = sum_c q_rc k_sc e^{G_rc - G_sc} (s <= r)
//   X = (I + A)^-1,  T = X Diag(beta),  W = T K_hat,  U_hat = T V,  U = U_hat - W S0
//   O = Q_hat S0 + M U,  S_C = Diag(e^{G_C}) S0 + K_bar^T U
// (K_hat = K e^{G}, Q_hat = Q e^{G}, K_bar = K e^{G_C - G}).  Its reverse mode, per chunk, given
// dO and dS_C (dL/dS at the chunk end):
//   dU = M^T dO + K_bar dS_C,   dS0 = Q_hat^T dO + Diag(e^{G_C}) dS_C - W^T dU   (the serial pass)
//   dQ_hat = dO S0^T, dM = dO U^T, dK_bar = U dS_C^T, dW = -dU S0^T,
//   dT = dU V^T + dW K_hat^T, dK_hat = T^T dW, dV = T^T dU,
//   dX = dT Diag(beta), dbeta += colsum(X (.) dT), dA = -X^T dX X^T (strict lower),
//   dbeta += rowsum(dA (.) A_tilde) (A_tilde: A without beta), P = Diag(beta) dA,
//   and the A / M terms reach dq, dk and dG through e^{G_r - G_s} with the same reference points as
//   the forward; dg is the reverse cumulative sum of dG over the chunk.
//
// Kernels (fp32 data; the products by warp_mma below):
//   bwd_rec    per (chunk, head): the chunk's records (T, X, A_tilde, M, W, W^T, U_hat, K_bar,
//              K_bar^T, Q_hat, e^{G_C});
//   bwd_fwd    per (sequence, head, value-column slice), serial over chunks: S0 and U per chunk;
//   bwd_rev    the same, reverse: dS_C and dU per chunk, dh0;
//   bwd_dvsums per (chunk, head): the products summed over the value columns, and dv;
//   bwd_grads  per (chunk, head): the parameter gradients.
// Global memory is written row by row: a transposed copy is assembled in shared memory first.
#include <type_traits>

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kC = 64;         // chunk length
constexpr int kThreads = 256;  // every kernel here
static_assert(kThreads == 4 * kC, "the diagonal inverses in bwd_rec give each column four lanes");

// ---- warp-level tensor-core products (mma.sync m16n8k8, tf32) with a three-term split: each operand
// x = hi + lo with hi = x truncated to tf32 (its low 13 mantissa bits cleared) and lo = x - hi (exact
// in fp32), and hi*hi + hi*lo + lo*hi accumulated in fp32.  The tensor core reads only the tf32 part
// of lo, so the dropped terms are about 2^-20 of each product: fp32-level results for the backward's
// tolerance, with two integer/float instructions per element instead of conversions.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = __float_as_uint(x) & 0xffffe000u;
  lo = __float_as_uint(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// acc (a 16 x 8 NT tile at rows m0.., columns n0..) += sum_{k < K} At[k * lda + m] B[k * ldb + n] for one
// warp; both operands k-major in shared memory, K a multiple of 8.  The three terms accumulate
// separately (no MMA waits on the one before it in the same k step) and are added at the end.
// Lane (g = lane / 4, t = lane % 4) holds acc[nt][0..1] at row m0 + g, columns n0 + 8 nt + 2t, +1,
// and acc[nt][2..3] eight rows below.
// With AT = false the left operand is given row-major instead (A[m * lda + k]).  AX (BX) declares every
// value of the left (right) operand exact in tf32, a widened bf16 input: its low part is zero, so the
// product term that would multiply it is skipped (the result is bit-identical).
template <int NT, bool AT = true, bool AX = false, bool BX = false>
__device__ __forceinline__ void warp_mma(float (&acc)[NT][4], const float* At, int lda, int m0, const float* B,
                                         int ldb, int n0, int K, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const auto a = [&](int m, int k) { return AT ? At[k * lda + m] : At[m * lda + k]; };
  float hl[NT][4] = {}, lh[NT][4] = {};
#pragma unroll 4
  for (int k0 = 0; k0 < K; k0 += 8) {
    uint32_t ah[4], al[4];
    split_tf32(a(m0 + g, k0 + t), ah[0], al[0]);
    split_tf32(a(m0 + g + 8, k0 + t), ah[1], al[1]);
    split_tf32(a(m0 + g, k0 + t + 4), ah[2], al[2]);
    split_tf32(a(m0 + g + 8, k0 + t + 4), ah[3], al[3]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      uint32_t bh0, bl0, bh1, bl1;
      split_tf32(B[(k0 + t) * ldb + n0 + 8 * nt + g], bh0, bl0);
      split_tf32(B[(k0 + t + 4) * ldb + n0 + 8 * nt + g], bh1, bl1);
      mma_tf32(acc[nt], ah, bh0, bh1);
      if constexpr (!BX) mma_tf32(hl[nt], ah, bl0, bl1);
      if constexpr (!AX) mma_tf32(lh[nt], al, bh0, bh1);
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] += hl[nt][e] + lh[nt][e];
}
// inputs stored as bf16 (8 significant bits) are exact in tf32 once widened to fp32
template <typename Tin>
constexpr bool kExactInput = std::is_same<Tin, __nv_bfloat16>::value;
// the fragment element e of tile nt of a warp_mma accumulator: its row and column
__device__ __forceinline__ int frag_row(int m0, int lane, int e) { return m0 + (lane >> 2) + 8 * (e >> 1); }
__device__ __forceinline__ int frag_col(int n0, int lane, int nt, int e) { return n0 + 8 * nt + 2 * (lane & 3) + (e & 1); }
// rows r < rmax of a warp_mma result, times scale, into a row-major array (row stride ld)
template <int NT>
__device__ __forceinline__ void frag_store(float* dst, size_t ld, const float (&acc)[NT][4], int m0, int n0, int lane,
                                           float scale, int rmax = kC) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int r = m0 + g + 8 * hf;
      if (r < rmax)
        *reinterpret_cast<float2*>(dst + (size_t)r * ld + n0 + 8 * nt + 2 * t) =
            make_float2(scale * acc[nt][2 * hf], scale * acc[nt][2 * hf + 1]);
    }
}
// Warp tiling of a ROWS x ES product over the eight warps: warp w takes the 16-row tile w mod
// (ROWS / 16) and NT eight-column tiles starting at column n0.
template <int ROWS, int ES>
struct WarpTiles {
  static constexpr int MT = ROWS / 16, WPM = 8 / MT, NT = ES / 8 / WPM;
  static_assert(8 % MT == 0 && NT >= 1, "tiling");
  __device__ static void at(int warp, int& m0, int& n0) {
    m0 = 16 * (warp % MT);
    n0 = (warp / MT) * (ES / WPM);
  }
};

// for (i = tid; i < n; i += kThreads) put(i, get(i)), with eight loads in flight per thread before
// their stores (the gets are global loads, the puts shared-memory stores)
template <class Get, class Put>
__device__ __forceinline__ void batched(int n, int tid, Get get, Put put) {
  for (int base = tid; base < n; base += 8 * kThreads) {
    decltype(get(0)) x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + u * kThreads;
      if (i < n) x[u] = get(i);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + u * kThreads;
      if (i < n) put(i, x[u]);
    }
  }
}

// the D (or E) values of rows t0 .. t0+n-1 of head h of a [T][H][D] array into L2, thread tid0 + r
// taking row r (rows are 16-byte aligned: D * sizeof(T) is a multiple of 16)
template <typename Tp>
__device__ __forceinline__ void prefetch_rows_l2(const Tp* x, int64_t t0, int n, int H, int h, int D, int tid, int tid0) {
  const int r = tid - tid0;
  if (r >= 0 && r < n) prefetch_l2(x + ((size_t)(t0 + r) * H + h) * D, (uint32_t)(D * sizeof(Tp)));
}

// The (chunk, head) task that this CTA takes next: true with its rows when it exists.
__device__ __forceinline__ bool next_task(int64_t task, int64_t ntask, int H, const int32_t* plan, const int32_t* cu,
                                          int B, int64_t T, int& h, int64_t& t0, int& n) {
  const int64_t nt = task + gridDim.x;
  int b;
  int64_t cseq;
  if (nt >= ntask || !resolve_chunk(nt / H, plan, cu, B, T, b, t0, n, cseq)) return false;
  h = (int)(nt % H);
  return true;
}

// Per-(chunk, head) record layout in the workspace (floats).
struct RecLayout {
  int D, E;
  __host__ __device__ size_t T() const { return 0; }                     // [C][C]
  __host__ __device__ size_t X() const { return (size_t)kC * kC; }       // [C][C]
  __host__ __device__ size_t At() const { return 2 * (size_t)kC * kC; }  // [C][C] A without beta, strict lower
  __host__ __device__ size_t M() const { return 3 * (size_t)kC * kC; }   // [C][C] lower incl. diagonal
  __host__ __device__ size_t W() const { return 4 * (size_t)kC * kC; }   // [C][D]
  __host__ __device__ size_t WT() const { return W() + (size_t)kC * D; }  // [D][C]
  __host__ __device__ size_t Uh() const { return WT() + (size_t)kC * D; }  // [C][E]
  __host__ __device__ size_t Kb() const { return Uh() + (size_t)kC * E; }  // [C][D]
  __host__ __device__ size_t KbT() const { return Kb() + (size_t)kC * D; }  // [D][C]
  __host__ __device__ size_t Qh() const { return KbT() + (size_t)kC * D; }  // [C][D]
  __host__ __device__ size_t GC() const { return Qh() + (size_t)kC * D; }   // [D]
  __host__ __device__ size_t size() const { return GC() + (size_t)D; }
};
// Per-(chunk, head) states of the two serial passes (floats): S0^T and dS_C^T [E][D], U^T and dU^T [E][C].
struct StateLayout {
  int D, E;
  __host__ __device__ size_t S0T() const { return 0; }
  __host__ __device__ size_t UT() const { return (size_t)E * D; }
  __host__ __device__ size_t dST() const { return UT() + (size_t)E * kC; }
  __host__ __device__ size_t dUT() const { return dST() + (size_t)E * D; }
  __host__ __device__ size_t size() const { return dUT() + (size_t)E * kC; }
};

// rows x C floats from shared memory (row stride sld) to a dense [rows][C] block of global memory,
// 16-byte coalesced stores
__device__ __forceinline__ void copy_out(float* dst, const float* src, int sld, int rows, int tid) {
  for (int i = tid; i < rows * (kC / 4); i += kThreads) {
    const int r = i / (kC / 4), c = 4 * (i % (kC / 4));
    *reinterpret_cast<float4*>(dst + (size_t)r * kC + c) = *reinterpret_cast<const float4*>(src + r * sld + c);
  }
}

// ---------------------------------------------------------------- per-chunk records
// Shared floats of bwd_rec: k, q, G [C][D+4]; scratch (A/M operands, later V and T^T); A_tilde, M, X
// [C][C+4]; beta [C].
template <int D, int E>
struct RecSmem {
  static constexpr int LD = D + 4, LE = E + 4, LC = kC + 4, L32 = 32 + 4;
  static constexpr int SC0 = 3 * D * L32, SC1 = kC * LE + kC * LC;
  static constexpr int SC = SC0 > SC1 ? SC0 : SC1;
  static constexpr int floats = 3 * kC * LD + SC + 3 * kC * LC + kC;
};

// 16-byte pieces (16 / sizeof(Tp) values) of a [C][D] tile of head h, rows n.. reading as zero, widened
// to fp32 in shared memory (row stride ld, a multiple of 4)
template <int D, typename Tp>
struct TileLoad {
  static constexpr int V = 16 / sizeof(Tp), PER_ROW = D / V, PIECES = kC * PER_ROW;
  static_assert(PIECES % kThreads == 0, "whole pieces per thread");
  static constexpr int N = PIECES / kThreads;
  uint4 x[N];
  __device__ __forceinline__ void load(const Tp* a, int64_t t0, int n, int H, int h, int tid) {
#pragma unroll
    for (int u = 0; u < N; ++u) {
      const int i = tid + u * kThreads, r = i / PER_ROW;
      x[u] = r < n ? *reinterpret_cast<const uint4*>(a + ((size_t)(t0 + r) * H + h) * D + V * (i % PER_ROW))
                   : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  __device__ __forceinline__ void store(float* dst, int ld, int tid) const {
#pragma unroll
    for (int u = 0; u < N; ++u) {
      const int i = tid + u * kThreads;
      float* o = dst + (i / PER_ROW) * ld + V * (i % PER_ROW);
      const Tp* e = reinterpret_cast<const Tp*>(&x[u]);
#pragma unroll
      for (int w = 0; w < V; w += 4)
        *reinterpret_cast<float4*>(o + w) = make_float4(to_f32(e[w]), to_f32(e[w + 1]), to_f32(e[w + 2]), to_f32(e[w + 3]));
    }
  }
};
// k, q and g of one chunk into shared memory (row stride ld); rows n..C-1 are zero.  Every load is
// issued before the first store.
template <int D, typename Tin>
__device__ __forceinline__ void load_kqg(const Tin* k, const Tin* q, const float* g, int64_t t0, int n, int H, int h,
                                         float* kS, float* qS, float* gS, int ld, int tid) {
  TileLoad<D, Tin> tk, tq;
  TileLoad<D, float> tg;
  tk.load(k, t0, n, H, h, tid);
  tq.load(q, t0, n, H, h, tid);
  tg.load(g, t0, n, H, h, tid);
  tk.store(kS, ld, tid);
  tq.store(qS, ld, tid);
  tg.store(gS, ld, tid);
}

template <int D, int E, typename Tin>
__global__ void __launch_bounds__(kThreads, 1)
bwd_rec(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v, const float* __restrict__ g,
        const float* __restrict__ beta, const int32_t* __restrict__ plan, const int32_t* __restrict__ cu, int B,
        int64_t T, int H, int64_t ntask, float* __restrict__ recs) {
  using SM = RecSmem<D, E>;
  constexpr int LD = SM::LD, LE = SM::LE, LC = SM::LC, L32 = SM::L32;
  extern __shared__ __align__(16) float sm[];
  float* kS = sm;                 // k, later K_hat
  float* qS = kS + kC * LD;
  float* gS = qS + kC * LD;       // g, then G
  float* sc = gS + kC * LD;
  float* AtS = sc + SM::SC;
  float* MS = AtS + kC * LC;
  float* XS = MS + kC * LC;
  float* bS = XS + kC * LC;
  const int tid = threadIdx.x;
  const RecLayout L{D, E};
  for (int64_t task = blockIdx.x; task < ntask; task += gridDim.x) {
    const int64_t chunk = task / H;
    const int h = (int)(task - chunk * H);
    int b, n;
    int64_t t0, cseq;
    if (!resolve_chunk(chunk, plan, cu, B, T, b, t0, n, cseq)) continue;  // same for the whole CTA
    float* rec = recs + (size_t)task * L.size();
    {  // the next task's inputs into L2 while this one runs
      int h2, n2;
      int64_t t2;
      if (next_task(task, ntask, H, plan, cu, B, T, h2, t2, n2)) {
        prefetch_rows_l2(k, t2, n2, H, h2, D, tid, 0);
        prefetch_rows_l2(q, t2, n2, H, h2, D, tid, 64);
        prefetch_rows_l2(g, t2, n2, H, h2, D, tid, 128);
        prefetch_rows_l2(v, t2, n2, H, h2, E, tid, 192);
      }
    }
    // inputs of the chunk (rows past the sequence end: k = q = 0, g = 0, beta = 0)
    load_kqg<D>(k, q, g, t0, n, H, h, kS, qS, gS, LD, tid);
    if (tid < kC) bS[tid] = tid < n ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
    for (int i = tid; i < kC * LC; i += kThreads) {
      AtS[i] = 0.f;
      MS[i] = 0.f;
    }
    __syncthreads();
    if (tid < D) {  // G: inclusive cumulative decay over the chunk
      float run = 0.f;
      for (int r = 0; r < kC; ++r) {
        run += gS[r * LD + tid];
        gS[r * LD + tid] = run;
      }
    }
    __syncthreads();
    // e^{G_C}, K_bar = k e^{G_C - G} (and its transpose, through the scratch), Q_hat = q e^{G}
    for (int i = tid; i < kC * D; i += kThreads) {
      const int r = i / D, c = i % D;
      const float G = gS[r * LD + c], Gc = gS[(kC - 1) * LD + c];
      const float kb = kS[r * LD + c] * __expf(Gc - G);
      rec[L.Kb() + (size_t)r * D + c] = kb;
      sc[c * LC + r] = kb;
      rec[L.Qh() + (size_t)r * D + c] = qS[r * LD + c] * __expf(G);
      if (r == 0) rec[L.GC() + c] = __expf(Gc);
    }
    __syncthreads();
    copy_out(rec + L.KbT(), sc, LC, D, tid);
    __syncthreads();
    // A_tilde (strict lower) and M (lower incl. diagonal) by 32 x 32 blocks, each with a reference
    // point R that keeps every factor within e^{+-80} (g > -5): the diagonal blocks use the centred
    // rows 15 and 47, the block below the diagonal row 47 (its key-side factor is then <= 1)
    for (int blk = 0; blk < 3; ++blk) {
      const int ra = blk == 0 ? 0 : 32, sb = blk == 1 ? 32 : 0, ref = blk == 0 ? 15 : 47;
      float* XkT = sc;
      float* XqT = sc + D * L32;
      float* YT = sc + 2 * D * L32;
      for (int i = tid; i < D * 32; i += kThreads) {
        const int c = i / 32, r = i % 32;
        const float R = gS[ref * LD + c];
        const float er = __expf(gS[(ra + r) * LD + c] - R);
        XkT[c * L32 + r] = kS[(ra + r) * LD + c] * er;
        XqT[c * L32 + r] = qS[(ra + r) * LD + c] * er;
        YT[c * L32 + r] = kS[(sb + r) * LD + c] * __expf(R - gS[(sb + r) * LD + c]);
      }
      __syncthreads();
      {  // warp w: the A (w < 4) or M block, rows 16 ((w >> 1) & 1).., columns 16 (w & 1)..
        const int warp = tid >> 5, lane = tid & 31;
        const bool isM = warp >= 4;
        const int m0 = 16 * ((warp >> 1) & 1), n0 = 16 * (warp & 1);
        float acc[2][4] = {};
        warp_mma<2>(acc, isM ? XqT : XkT, L32, m0, YT, L32, n0, D, lane);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = ra + frag_row(m0, lane, e), s = sb + frag_col(n0, lane, nt, e);
            if (isM) MS[r * LC + s] = r >= s ? acc[nt][e] : 0.f;  // select, not mask-multiply
            else AtS[r * LC + s] = r > s ? acc[nt][e] : 0.f;
          }
      }
      __syncthreads();
    }
    // X = (I + A)^-1 with A = Diag(beta) A_tilde strictly lower, by blocks.  First the four diagonal
    // 16 x 16 inverses by forward substitution, X_rs = -beta_r sum_{s <= j < r} A_tilde_rj X_js: each
    // column is owned by four adjacent lanes, lane p summing the terms j = s + p (mod 4).
    {
      const int o = 16 * (tid >> 6), s = (tid >> 2) & 15, p = tid & 3;
      for (int r = 0; r < 16; ++r) {
        float part = 0.f;
        for (int j = s + p; j < r; j += 4) part = fmaf(AtS[(o + r) * LC + o + j], XS[(o + j) * LC + o + s], part);
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        if (p == 0) XS[(o + r) * LC + o + s] = r > s ? -bS[o + r] * part : (r == s ? 1.f : 0.f);
        __syncwarp();  // column s of the block is read back only by its own four lanes
      }
      for (int i = tid; i < kC * kC; i += kThreads)  // the blocks above the diagonal
        if ((i / kC) >> 4 < (i % kC) >> 4) XS[(i / kC) * LC + i % kC] = 0.f;
    }
    __syncthreads();
    // Then pairs of diagonal blocks of size m are merged into blocks of size 2m: with
    // [[X11, 0], [X21, X22]] the inverse of [[I + A11, 0], [A21, I + A22]], X21 = -X22 A21 X11.
    for (int m = 16; m < kC; m *= 2) {
      constexpr int LY = 32 + 4;
      float* Y = sc;  // [kC / 2][LY]: A21 X11 of every merged block, stacked
      const int outs = (kC / 2) * m;
      for (int i = tid; i < outs; i += kThreads) {
        const int bi = i / (m * m), rr = (i / m) % m, cc = i % m, o = 2 * m * bi;
        float acc = 0.f;
        for (int j = cc; j < m; ++j)  // X11 is lower triangular
          acc = fmaf(AtS[(o + m + rr) * LC + o + j], XS[(o + j) * LC + o + cc], acc);
        Y[(bi * m + rr) * LY + cc] = bS[o + m + rr] * acc;
      }
      __syncthreads();
      for (int i = tid; i < outs; i += kThreads) {
        const int bi = i / (m * m), rr = (i / m) % m, cc = i % m, o = 2 * m * bi;
        float acc = 0.f;
        for (int j = 0; j <= rr; ++j)  // X22 is lower triangular
          acc = fmaf(XS[(o + m + rr) * LC + o + m + j], Y[(bi * m + j) * LY + cc], acc);
        XS[(o + m + rr) * LC + o + cc] = -acc;
      }
      __syncthreads();
    }
    // T = X Diag(beta) (also transposed for the products below); records T, X, A_tilde, M
    float* vS = sc;               // [C][LE]
    float* TT = sc + kC * LE;     // [C][LC]
    for (int i = tid; i < kC * kC; i += kThreads) {
      const int r = i / kC, s = i % kC;
      const float x = XS[r * LC + s], t = x * bS[s];
      rec[L.T() + i] = t;
      rec[L.X() + i] = x;
      rec[L.At() + i] = AtS[r * LC + s];
      rec[L.M() + i] = MS[r * LC + s];
      TT[s * LC + r] = t;
    }
    for (int i = tid; i < kC * D; i += kThreads) {  // K_hat = k e^{G}, in place
      const int r = i / D, c = i % D;
      kS[r * LD + c] *= __expf(gS[r * LD + c]);
    }
    batched(kC * E, tid, [&](int i) { const int r = i / E; return r < n ? to_f32(v[((size_t)(t0 + r) * H + h) * E + i % E]) : 0.f; },
            [&](int i, float x) { vS[(i / E) * LE + i % E] = x; });
    __syncthreads();
    float* WTs = qS;  // [D][LC] over q and G (free now)
    static_assert(D * LC <= 2 * kC * LD, "W^T fits over q and G");
    {  // W = T K_hat (and its transpose, through shared memory)
      using TD = WarpTiles<kC, D>;
      const int warp = tid >> 5, lane = tid & 31;
      int m0, n0;
      TD::at(warp, m0, n0);
      float acc[TD::NT][4] = {};
      warp_mma<TD::NT>(acc, TT, LC, m0, kS, LD, n0, kC, lane);
      frag_store<TD::NT>(rec + L.W(), D, acc, m0, n0, lane, 1.f);
#pragma unroll
      for (int nt = 0; nt < TD::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) WTs[frag_col(n0, lane, nt, e) * LC + frag_row(m0, lane, e)] = acc[nt][e];
    }
    {  // U_hat = T V
      using TE = WarpTiles<kC, E>;
      const int warp = tid >> 5, lane = tid & 31;
      int m0, n0;
      TE::at(warp, m0, n0);
      float acc[TE::NT][4] = {};
      warp_mma<TE::NT, true, false, kExactInput<Tin>>(acc, TT, LC, m0, vS, LE, n0, kC, lane);
      frag_store<TE::NT>(rec + L.Uh(), E, acc, m0, n0, lane, 1.f);
    }
    __syncthreads();
    copy_out(rec + L.WT(), WTs, LC, D, tid);
    __syncthreads();  // shared memory is rewritten by the next task
  }
}

// ---------------------------------------------------------------- the two serial passes
// Each CTA: one (sequence, head) chain and ES of its value columns (the recurrence is separable in
// the columns of the state).  Per chunk, 64 x ES and D x ES products on the tensor cores (warp_mma,
// three-term tf32), each warp owning whole tiles of the result.

// rows x cols floats from global (row stride gld) into shared memory (row stride sld), 16-byte
// copies through registers, eight per thread in flight (measured faster than the asynchronous
// copies below for the serial passes' L2-resident records)
__device__ __forceinline__ void stage(float* dst, int sld, const float* src, size_t gld, int rows, int cols, int tid) {
  const int q = cols / 4;
  batched(rows * q, tid,
          [&](int i) { return *reinterpret_cast<const float4*>(src + (size_t)(i / q) * gld + 4 * (i % q)); },
          [&](int i, float4 x) { *reinterpret_cast<float4*>(dst + (i / q) * sld + 4 * (i % q)) = x; });
}
// the same as asynchronous 16-byte copies, all in flight at once; stage_wait() before the barrier
// that publishes them
__device__ __forceinline__ void stage_async(float* dst, int sld, const float* src, size_t gld, int rows, int cols,
                                            int tid) {
  const int q = cols / 4;
  for (int i = tid; i < rows * q; i += kThreads) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst + (i / q) * sld + 4 * (i % q)));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src + (size_t)(i / q) * gld + 4 * (i % q))
                 : "memory");
  }
}
__device__ __forceinline__ void stage_wait() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The transpose of a rows x cols block of global memory (row stride gld; rows a multiple of 8, cols
// of 16) into shared memory, dst[c * sld + r] (sld = 4 mod 32).  Each warp moves 8 rows x 16
// columns: 64 contiguous bytes of each row, and shared stores at most two-way conflicted.
__device__ __forceinline__ void stage_t(float* dst, int sld, const float* src, size_t gld, int rows, int cols,
                                        int tid) {
  const int rb = rows / 8;
  const auto row = [&](int i) { return 8 * ((i >> 5) % rb) + (i & 7); };
  const auto grp = [&](int i) { return 4 * ((i >> 5) / rb) + ((i & 31) >> 3); };  // 4-column group
  batched(rows * (cols / 4), tid,
          [&](int i) { return *reinterpret_cast<const float4*>(src + (size_t)row(i) * gld + 4 * grp(i)); },
          [&](int i, float4 x) {
            float* o = dst + 4 * grp(i) * sld + row(i);
            o[0] = x.x;
            o[sld] = x.y;
            o[2 * sld] = x.z;
            o[3 * sld] = x.w;
          });
}

template <int D, int E, int ES>
struct FwdSmem {
  static constexpr int LC = kC + 4, LD = D + 4, LS = ES + 4;
  static constexpr int floats = D * LC + kC * LD + kC * LS + D + D * LS + kC * LS;
};


template <int D, int E, int ES>
__global__ void __launch_bounds__(kThreads, 1)
bwd_fwd(const float* __restrict__ recs, const float* __restrict__ h0, const int32_t* __restrict__ plan,
        const int32_t* __restrict__ cu, int B, int64_t T, int H, float* __restrict__ states) {
  using SM = FwdSmem<D, E, ES>;
  using TU = WarpTiles<kC, ES>;
  using TS = WarpTiles<D, ES>;
  constexpr int LC = SM::LC, LD = SM::LD, LS = SM::LS;
  extern __shared__ __align__(16) float sm[];
  float* WTs = sm;              // W^T [D][LC]
  float* Kbs = WTs + D * LC;    // K_bar [C][LD]
  float* Uhs = Kbs + kC * LD;   // U_hat slice [C][LS]
  float* GCs = Uhs + kC * LS;   // e^{G_C} [D]
  float* S = GCs + D;           // [D][LS]
  float* U = S + D * LS;        // [C][LS]
  const int b = blockIdx.x, h = blockIdx.y, j0 = blockIdx.z * ES, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (cu != nullptr && plan[B + 1] == 0) return;
  int64_t first_chunk, t_begin, len;
  const int64_t nch = sequence_chunks(b, plan, cu, B, T, first_chunk, t_begin, len);
  const RecLayout L{D, E};
  const StateLayout SL{D, E};
  for (int i = tid; i < D * ES; i += kThreads) {
    const int c = i / ES, j = i % ES;
    S[c * LS + j] = h0 != nullptr ? h0[(((size_t)b * H + h) * D + c) * E + j0 + j] : 0.f;
  }
  for (int64_t ci = 0; ci < nch; ++ci) {
    const size_t task = (size_t)(first_chunk + ci) * H + h;
    const float* rec = recs + task * L.size();
    float* st = states + task * SL.size();
    if (tid == 0 && ci + 1 < nch) {  // the next chunk's records: W^T, U_hat, K_bar (adjacent) and e^{G_C}
      const float* nx = rec + (size_t)H * L.size();
      prefetch_l2(nx + L.WT(), (uint32_t)((L.Kb() + (size_t)kC * D - L.WT()) * 4));
      prefetch_l2(nx + L.GC(), D * 4);
    }
    stage(WTs, LC, rec + L.WT(), kC, D, kC, tid);
    stage(Kbs, LD, rec + L.Kb(), D, kC, D, tid);
    stage(Uhs, LS, rec + L.Uh() + j0, E, kC, ES, tid);
    stage(GCs, D, rec + L.GC(), D, 1, D, tid);
    __syncthreads();
    for (int i = tid; i < D * ES; i += kThreads) {  // S0^T, coalesced along dk
      const int j = i / D, c = i % D;
      st[SL.S0T() + (size_t)(j0 + j) * D + c] = S[c * LS + j];
    }
    {  // U = U_hat - W S
      int m0, n0;
      TU::at(warp, m0, n0);
      float acc[TU::NT][4] = {};
      warp_mma<TU::NT>(acc, WTs, LC, m0, S, LS, n0, D, lane);
#pragma unroll
      for (int nt = 0; nt < TU::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = frag_row(m0, lane, e), c = frag_col(n0, lane, nt, e);
          U[r * LS + c] = Uhs[r * LS + c] - acc[nt][e];
        }
    }
    __syncthreads();
    for (int i = tid; i < kC * ES; i += kThreads) {  // U^T, coalesced along the chunk
      const int j = i / kC, r = i % kC;
      st[SL.UT() + (size_t)(j0 + j) * kC + r] = U[r * LS + j];
    }
    {  // S <- Diag(e^{G_C}) S + K_bar^T U (each warp reads and writes only its own tile of S)
      int m0, n0;
      TS::at(warp, m0, n0);
      float acc[TS::NT][4] = {};
      warp_mma<TS::NT>(acc, Kbs, LD, m0, U, LS, n0, kC, lane);
#pragma unroll
      for (int nt = 0; nt < TS::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = frag_row(m0, lane, e), c = frag_col(n0, lane, nt, e);
          float& sv = S[r * LS + c];
          sv = fmaf(GCs[r], sv, acc[nt][e]);
        }
    }
    __syncthreads();
  }
}

template <int D, int E, int ES>
struct RevSmem {
  static constexpr int LC = kC + 4, LD = D + 4, LS = ES + 4;
  static constexpr int floats = kC * LC + D * LC + 2 * kC * LD + D + D * LS + 2 * kC * LS;
};

template <int D, int E, int ES, typename Tin>
__global__ void __launch_bounds__(kThreads, 1)
bwd_rev(const float* __restrict__ recs, const Tin* __restrict__ dout, const float* __restrict__ dhT,
        const int32_t* __restrict__ plan, const int32_t* __restrict__ cu, int B, int64_t T, int H,
        float* __restrict__ states, float* __restrict__ dh0) {
  using SM = RevSmem<D, E, ES>;
  using TU = WarpTiles<kC, ES>;
  using TS = WarpTiles<D, ES>;
  constexpr int LC = SM::LC, LD = SM::LD, LS = SM::LS;
  extern __shared__ __align__(16) float sm[];
  float* Ms = sm;               // M [C][LC]
  float* KbTs = Ms + kC * LC;   // K_bar^T [D][LC]
  float* Qhs = KbTs + D * LC;   // Q_hat [C][LD]
  float* Ws = Qhs + kC * LD;    // W [C][LD]
  float* GCs = Ws + kC * LD;    // [D]
  float* dS = GCs + D;          // [D][LS]
  float* dO = dS + D * LS;      // [C][LS]
  float* dU = dO + kC * LS;     // [C][LS]
  const int b = blockIdx.x, h = blockIdx.y, j0 = blockIdx.z * ES, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (cu != nullptr && plan[B + 1] == 0) return;
  int64_t first_chunk, t_begin, len;
  const int64_t nch = sequence_chunks(b, plan, cu, B, T, first_chunk, t_begin, len);
  const RecLayout L{D, E};
  const StateLayout SL{D, E};
  for (int i = tid; i < D * ES; i += kThreads) {
    const int c = i / ES, j = i % ES;
    dS[c * LS + j] = dhT != nullptr ? dhT[(((size_t)b * H + h) * D + c) * E + j0 + j] : 0.f;
  }
  for (int64_t ci = nch - 1; ci >= 0; --ci) {
    const size_t task = (size_t)(first_chunk + ci) * H + h;
    const float* rec = recs + task * L.size();
    float* st = states + task * SL.size();
    const int64_t t0 = t_begin + 64 * ci;
    const int n = (int)(len - 64 * ci < 64 ? len - 64 * ci : 64);
    if (ci > 0) {  // the previous chunk's records (M and W; K_bar^T, Q_hat and e^{G_C}) and dout rows
      const float* nx = rec - (size_t)H * L.size();
      if (tid == 0) {
        prefetch_l2(nx + L.M(), (uint32_t)((L.W() + (size_t)kC * D - L.M()) * 4));
        prefetch_l2(nx + L.KbT(), (uint32_t)((L.size() - L.KbT()) * 4));
      } else if (tid >= 64 && tid < 64 + kC) {
        const Tin* row = dout + ((size_t)(t0 - 64 + tid - 64) * H + h) * E + j0;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(row) : "memory");
      }
    }
    stage(Ms, LC, rec + L.M(), kC, kC, kC, tid);
    stage(KbTs, LC, rec + L.KbT(), kC, D, kC, tid);
    stage(Qhs, LD, rec + L.Qh(), D, kC, D, tid);
    stage(Ws, LD, rec + L.W(), D, kC, D, tid);
    stage(GCs, D, rec + L.GC(), D, 1, D, tid);
    batched(kC * ES, tid,
            [&](int i) { return i / ES < n ? to_f32(dout[((size_t)(t0 + i / ES) * H + h) * E + j0 + i % ES]) : 0.f; },
            [&](int i, float x) { dO[(i / ES) * LS + i % ES] = x; });
    __syncthreads();
    for (int i = tid; i < D * ES; i += kThreads) {  // dS_C^T, coalesced along dk
      const int j = i / D, c = i % D;
      st[SL.dST() + (size_t)(j0 + j) * D + c] = dS[c * LS + j];
    }
    {  // dU = M^T dO + K_bar dS
      int m0, n0;
      TU::at(warp, m0, n0);
      float acc[TU::NT][4] = {};
      warp_mma<TU::NT, true, false, kExactInput<Tin>>(acc, Ms, LC, m0, dO, LS, n0, kC, lane);
      warp_mma<TU::NT>(acc, KbTs, LC, m0, dS, LS, n0, D, lane);
#pragma unroll
      for (int nt = 0; nt < TU::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) dU[frag_row(m0, lane, e) * LS + frag_col(n0, lane, nt, e)] = acc[nt][e];
    }
    __syncthreads();
    for (int i = tid; i < kC * ES; i += kThreads) {  // dU^T, coalesced along the chunk
      const int j = i / kC, r = i % kC;
      st[SL.dUT() + (size_t)(j0 + j) * kC + r] = dU[r * LS + j];
    }
    {  // dS <- Q_hat^T dO + Diag(e^{G_C}) dS - W^T dU (each warp reads and writes only its own tile of dS)
      int m0, n0;
      TS::at(warp, m0, n0);
      float a1[TS::NT][4] = {}, a2[TS::NT][4] = {};
      warp_mma<TS::NT, true, false, kExactInput<Tin>>(a1, Qhs, LD, m0, dO, LS, n0, kC, lane);
      warp_mma<TS::NT>(a2, Ws, LD, m0, dU, LS, n0, kC, lane);
#pragma unroll
      for (int nt = 0; nt < TS::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = frag_row(m0, lane, e), c = frag_col(n0, lane, nt, e);
          float& sv = dS[r * LS + c];
          sv = fmaf(GCs[r], sv, a1[nt][e] - a2[nt][e]);
        }
    }
    __syncthreads();
  }
  if (dh0 != nullptr)
    for (int i = tid; i < D * ES; i += kThreads) {
      const int c = i / ES, j = i % ES;
      dh0[(((size_t)b * H + h) * D + c) * E + j0 + j] = dS[c * LS + j];
    }
}

// ---------------------------------------------------------------- gradients, part 1: sums over dv
// Per (chunk, head) scratch written here and read by bwd_grads (floats).
struct GradLayout {
  int D;
  __host__ __device__ size_t dQh() const { return 0; }                       // [C][D]
  __host__ __device__ size_t dW() const { return (size_t)kC * D; }           // [C][D]
  __host__ __device__ size_t dKb() const { return 2 * (size_t)kC * D; }      // [C][D]
  __host__ __device__ size_t dM() const { return 3 * (size_t)kC * D; }       // [C][C] (on M's support)
  __host__ __device__ size_t dT1() const { return dM() + (size_t)kC * kC; }  // [C][C]: dU V^T
  __host__ __device__ size_t dGam() const { return dT1() + (size_t)kC * kC; }  // [D]: rowsum(dS_C (.) S0)
  __host__ __device__ size_t size() const { return dGam() + (size_t)D; }
};

// Shared floats of bwd_dvsums: dO^T, V^T and dU^T [E][C+4]; S0^T, later dS_C^T [E][D+4]; dU
// [C][E+4], later U^T [E][C+4]; T [C][C+4].
template <int D, int E>
struct DvSmem {
  static constexpr int LC = kC + 4, LE = E + 4, LD = D + 4;
  static constexpr int CT = E * LC, UR = kC * LE > CT ? kC * LE : CT;
  static constexpr int floats = 3 * CT + E * LD + UR + kC * LC;
};

// 16-byte pieces of a [C][E] tile of head h (rows n.. reading as zero), widened to fp32 and stored
// transposed, [E][ld]; consecutive threads take consecutive rows so that the stores do not conflict
template <int E, typename Tp>
struct TileLoadT {
  static constexpr int V = 16 / sizeof(Tp), PIECES = kC * (E / V);
  static_assert(PIECES % kThreads == 0, "whole pieces per thread");
  static constexpr int N = PIECES / kThreads;
  uint4 x[N];
  __device__ __forceinline__ void load(const Tp* a, int64_t t0, int n, int H, int h, int tid) {
#pragma unroll
    for (int u = 0; u < N; ++u) {
      const int i = tid + u * kThreads, r = i % kC;
      x[u] = r < n ? *reinterpret_cast<const uint4*>(a + ((size_t)(t0 + r) * H + h) * E + V * (i / kC))
                   : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  __device__ __forceinline__ void store(float* dst, int ld, int tid) const {
#pragma unroll
    for (int u = 0; u < N; ++u) {
      const int i = tid + u * kThreads, r = i % kC, c = V * (i / kC);
      const Tp* e = reinterpret_cast<const Tp*>(&x[u]);
#pragma unroll
      for (int w = 0; w < V; ++w) dst[(c + w) * ld + r] = to_f32(e[w]);
    }
  }
};

// dQ_hat = dO S0^T, dW = -dU S0^T, dK_bar = U dS_C^T, dM = dO U^T, dU V^T, rowsum(dS_C (.) S0) into
// the scratch; dv = T^T dU into the output.  Every product reads both operands from shared memory.
template <int D, int E, typename Tin>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dvsums(const Tin* __restrict__ v, const Tin* __restrict__ dout, const int32_t* __restrict__ plan,
           const int32_t* __restrict__ cu, int B, int64_t T, int H, int64_t ntask, const float* __restrict__ recs,
           const float* __restrict__ states, float* __restrict__ grads, float* __restrict__ dv) {
  using SM = DvSmem<D, E>;
  constexpr int LC = SM::LC, LE = SM::LE, LD = SM::LD;
  extern __shared__ __align__(16) float sm[];
  float* dOT = sm;              // [E][LC]
  float* VT = dOT + SM::CT;     // [E][LC]
  float* dUT = VT + SM::CT;     // [E][LC]
  float* S0T = dUT + SM::CT;    // [E][LD]: S0^T, then dS_C^T
  float* dUr = S0T + E * LD;    // [C][LE]: dU, then U^T [E][LC]
  float* TS = dUr + SM::UR;     // [C][LC]
  const int tid = threadIdx.x;
  const RecLayout L{D, E};
  const StateLayout SL{D, E};
  const GradLayout GL{D};
  for (int64_t task = blockIdx.x; task < ntask; task += gridDim.x) {
    const int64_t chunk = task / H;
    const int h = (int)(task - chunk * H);
    int b, n;
    int64_t t0, cseq;
    if (!resolve_chunk(chunk, plan, cu, B, T, b, t0, n, cseq)) continue;
    const float* rec = recs + (size_t)task * L.size();
    const float* st = states + (size_t)task * SL.size();
    float* gr = grads + (size_t)task * GL.size();
    {  // the next task's operands into L2 while this one runs
      int h2, n2;
      int64_t t2;
      if (next_task(task, ntask, H, plan, cu, B, T, h2, t2, n2)) {
        const size_t nt = (size_t)task + gridDim.x;
        if (tid == 0) prefetch_l2(states + nt * SL.size(), (uint32_t)(SL.size() * 4));
        if (tid == 1) prefetch_l2(recs + nt * L.size() + L.T(), kC * kC * 4);
        prefetch_rows_l2(v, t2, n2, H, h2, E, tid, 64);
        prefetch_rows_l2(dout, t2, n2, H, h2, E, tid, 128);
      }
    }
    {
      stage_async(dUT, LC, st + SL.dUT(), kC, E, kC, tid);
      stage_async(S0T, LD, st + SL.S0T(), D, E, D, tid);
      stage_async(TS, LC, rec + L.T(), kC, kC, kC, tid);
      TileLoadT<E, Tin> tdo, tv;
      tdo.load(dout, t0, n, H, h, tid);
      tv.load(v, t0, n, H, h, tid);
      tdo.store(dOT, LC, tid);
      tv.store(VT, LC, tid);
    }
    stage_wait();
    __syncthreads();
    for (int i = tid; i < kC * E; i += kThreads) dUr[(i % kC) * LE + i / kC] = dUT[(i / kC) * LC + i % kC];
    __syncthreads();
    using TD = WarpTiles<kC, D>;
    using TE = WarpTiles<kC, E>;
    using TC = WarpTiles<kC, kC>;
    const int warp = tid >> 5, lane = tid & 31;
    {
      int m0, n0;
      TD::at(warp, m0, n0);
      float acc[TD::NT][4] = {};
      warp_mma<TD::NT, true, kExactInput<Tin>>(acc, dOT, LC, m0, S0T, LD, n0, E, lane);  // dO S0^T
      frag_store<TD::NT>(gr + GL.dQh(), D, acc, m0, n0, lane, 1.f);
      float acc2[TD::NT][4] = {};
      warp_mma<TD::NT>(acc2, dUT, LC, m0, S0T, LD, n0, E, lane);  // dU S0^T
      frag_store<TD::NT>(gr + GL.dW(), D, acc2, m0, n0, lane, -1.f);
    }
    {  // dv = T^T dU (rows of the sequence only)
      int m0, n0;
      TE::at(warp, m0, n0);
      float acc[TE::NT][4] = {};
      warp_mma<TE::NT>(acc, TS, LC, m0, dUr, LE, n0, kC, lane);
      frag_store<TE::NT>(dv + ((size_t)t0 * H + h) * E, (size_t)H * E, acc, m0, n0, lane, 1.f, n);
    }
    if (tid < D) {  // rowsum(dS_C (.) S0), dS_C^T from global
      float s0 = 0.f, s1 = 0.f;
      for (int j = 0; j < E; j += 2) {
        s0 = fmaf(st[SL.dST() + (size_t)j * D + tid], S0T[j * LD + tid], s0);
        s1 = fmaf(st[SL.dST() + (size_t)(j + 1) * D + tid], S0T[(j + 1) * LD + tid], s1);
      }
      gr[GL.dGam() + tid] = s0 + s1;
    }
    __syncthreads();  // S0^T and dU are no longer read
    float* UT = dUr;
    stage_async(S0T, LD, st + SL.dST(), D, E, D, tid);
    stage_async(UT, LC, st + SL.UT(), kC, E, kC, tid);
    stage_wait();
    __syncthreads();
    {
      int m0, n0;
      TD::at(warp, m0, n0);
      float acc[TD::NT][4] = {};
      warp_mma<TD::NT>(acc, UT, LC, m0, S0T, LD, n0, E, lane);  // U dS_C^T
      frag_store<TD::NT>(gr + GL.dKb(), D, acc, m0, n0, lane, 1.f);
    }
    {
      int m0, n0;
      TC::at(warp, m0, n0);
      float acc[TC::NT][4] = {};
      warp_mma<TC::NT, true, kExactInput<Tin>>(acc, dOT, LC, m0, UT, LC, n0, E, lane);  // dO U^T, on M's support
#pragma unroll
      for (int nt = 0; nt < TC::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (frag_row(m0, lane, e) < frag_col(n0, lane, nt, e)) acc[nt][e] = 0.f;
      frag_store<TC::NT>(gr + GL.dM(), kC, acc, m0, n0, lane, 1.f);
      float acc2[TC::NT][4] = {};
      warp_mma<TC::NT, true, false, kExactInput<Tin>>(acc2, dUT, LC, m0, VT, LC, n0, E, lane);  // dU V^T
      frag_store<TC::NT>(gr + GL.dT1(), kC, acc2, m0, n0, lane, 1.f);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- gradients, part 2
template <int D>
struct GradSmem {
  static constexpr int LD = D + 4, LC = kC + 4;
  static constexpr int base = 3 * kC * LD;  // k, q, G
  static constexpr int R1 = 3 * kC * LC;    // P, P^T, dA / dM^T (and dT, dX^T before them)
  static constexpr int R2a = 3 * 32 * LD, R2b = D * LC, R2c = 2 * kC * LC;
  static constexpr int R2 = R2a > R2b ? (R2a > R2c ? R2a : R2c) : (R2b > R2c ? R2b : R2c);
  static constexpr int floats = base + R1 + R2 + kC * LC + 2 * kC;  // + dM [C][LC], dbeta, beta
};

template <int D, int E, typename Tin>
__global__ void __launch_bounds__(kThreads, 1)
bwd_grads(const Tin* __restrict__ q, const Tin* __restrict__ k, const float* __restrict__ g,
          const float* __restrict__ beta, const int32_t* __restrict__ plan, const int32_t* __restrict__ cu, int B,
          int64_t T, int H, int64_t ntask, const float* __restrict__ recs, const float* __restrict__ grads,
          float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dg, float* __restrict__ dbeta) {
  using SM = GradSmem<D>;
  constexpr int LD = SM::LD, LC = SM::LC;
  extern __shared__ __align__(16) float sm[];
  float* kS = sm;
  float* qS = kS + kC * LD;  // q; rows of a finished half then hold that half's dG
  float* gS = qS + kC * LD;  // G
  float* s0 = gS + kC * LD;  // R1: three [C][LC]
  float* s1 = s0 + kC * LC;
  float* s2 = s1 + kC * LC;
  float* r2 = s0 + SM::R1;   // R2
  float* dMs = r2 + SM::R2;  // dM [C][LC]
  float* dbS = dMs + kC * LC;  // dbeta of the chunk's rows
  float* bS = dbS + kC;        // beta of the chunk's rows
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const RecLayout L{D, E};
  const GradLayout GL{D};
  for (int64_t task = blockIdx.x; task < ntask; task += gridDim.x) {
    const int64_t chunk = task / H;
    const int h = (int)(task - chunk * H);
    int b, n;
    int64_t t0, cseq;
    if (!resolve_chunk(chunk, plan, cu, B, T, b, t0, n, cseq)) continue;
    const float* rec = recs + (size_t)task * L.size();
    const float* gr = grads + (size_t)task * GL.size();
    {  // the next task's operands into L2 while this one runs
      int h2, n2;
      int64_t t2;
      if (next_task(task, ntask, H, plan, cu, B, T, h2, t2, n2)) {
        const size_t nt = (size_t)task + gridDim.x;
        if (tid == 0) prefetch_l2(grads + nt * GL.size(), (uint32_t)(GL.size() * 4));
        if (tid == 1) prefetch_l2(recs + nt * L.size() + L.T(), 3 * kC * kC * 4);  // T, X, A_tilde
        prefetch_rows_l2(k, t2, n2, H, h2, D, tid, 64);
        prefetch_rows_l2(q, t2, n2, H, h2, D, tid, 128);
        prefetch_rows_l2(g, t2, n2, H, h2, D, tid, 192);
      }
    }
    load_kqg<D>(k, q, g, t0, n, H, h, kS, qS, gS, LD, tid);
    if (tid < kC) {
      dbS[tid] = 0.f;
      bS[tid] = tid < n ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
    }
    __syncthreads();
    if (tid < D) {
      float run = 0.f;
      for (int r = 0; r < kC; ++r) {
        run += gS[r * LD + tid];
        gS[r * LD + tid] = run;
      }
    }
    __syncthreads();
    // ---- dT = dU V^T + dW K_hat^T
    float* KhT = r2;  // [D][LC]
    float* dWT = s1;  // [D][LC] over s1 and s2 (free until dX)
    static_assert(D * LC <= 2 * kC * LC, "dW^T fits in two C x C tiles");
    stage_t(dWT, LC, gr + GL.dW(), D, kC, D, tid);
    for (int i = tid; i < kC * D; i += kThreads) {
      const int s = i / D, c = i % D;
      KhT[c * LC + s] = kS[s * LD + c] * __expf(gS[s * LD + c]);
    }
    __syncthreads();
    float* dTS = s0;
    using TC = WarpTiles<kC, kC>;
    {
      int m0, n0;
      TC::at(warp, m0, n0);
      float acc[TC::NT][4] = {};
      warp_mma<TC::NT>(acc, dWT, LC, m0, KhT, LC, n0, D, lane);
#pragma unroll
      for (int nt = 0; nt < TC::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = frag_row(m0, lane, e), c = frag_col(n0, lane, nt, e);
          dTS[r * LC + c] = acc[nt][e] + gr[GL.dT1() + (size_t)r * kC + c];
        }
    }
    __syncthreads();
    // ---- T = X Diag(beta): dbeta_s += sum_r X_rs dT_rs; dX = dT Diag(beta) (stored transposed); X^T
    float* dXT = s1;
    float* XT = r2;           // [C][LC] (K_hat^T is no longer needed)
    float* YS = r2 + kC * LC;  // [C][LC]
    for (int i = tid; i < kC * kC; i += kThreads) {
      const int s = i / kC, j = i % kC;
      XT[j * LC + s] = rec[L.X() + i];
      dXT[j * LC + s] = dTS[s * LC + j] * bS[j];
    }
    __syncthreads();
    {  // four lanes per column s, lane p summing the rows r = p (mod 4)
      const int s = tid >> 2, p = tid & 3;
      float acc = 0.f;
      for (int r = p; r < kC; r += 4) acc = fmaf(XT[s * LC + r], dTS[r * LC + s], acc);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (p == 0) dbS[s] = acc;
    }
    // ---- dA = -X^T dX X^T on the strict lower triangle (Y = dX X^T first)
    {
      int m0, n0;
      TC::at(warp, m0, n0);
      float acc[TC::NT][4] = {};
      warp_mma<TC::NT>(acc, dXT, LC, m0, XT, LC, n0, kC, lane);
#pragma unroll
      for (int nt = 0; nt < TC::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) YS[frag_row(m0, lane, e) * LC + frag_col(n0, lane, nt, e)] = acc[nt][e];
    }
    __syncthreads();
    float* PS = s0;   // P = Diag(beta) dA
    float* PT = s1;   // P^T
    float* dAS = s2;  // dA, then dM^T
    {
      int m0, n0;
      TC::at(warp, m0, n0);
      float acc[TC::NT][4] = {};
      warp_mma<TC::NT, false>(acc, XT, LC, m0, YS, LC, n0, kC, lane);  // X^T Y: XT read row-major
#pragma unroll
      for (int nt = 0; nt < TC::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = frag_row(m0, lane, e), s = frag_col(n0, lane, nt, e);
          const float da = r > s ? -acc[nt][e] : 0.f;
          dAS[r * LC + s] = da;
          PS[r * LC + s] = bS[r] * da;
          PT[s * LC + r] = bS[r] * da;
        }
    }
    __syncthreads();
    if (tid < kC) {  // dbeta_r += sum_s dA_rs A_tilde_rs
      const int r = tid;
      float acc = 0.f;
      for (int s = 0; s < r; ++s) acc = fmaf(dAS[r * LC + s], rec[L.At() + (size_t)r * kC + s], acc);
      dbS[r] += acc;
    }
    __syncthreads();
    float* dMT = s2;
    for (int i = tid; i < kC * kC; i += kThreads) {
      const int r = i / kC, s = i % kC;
      const float x = gr[GL.dM() + i];
      dMT[s * LC + r] = x;
      dMs[r * LC + s] = x;
    }
    __syncthreads();
    // ---- the A / M terms and the elementwise terms, one 32-row output half at a time; warp w owns
    // 16-row tile w mod 2 and columns (w / 2) D/4.. of the half's dq, dk and dG (warp_mma fragments)
    float* Xk = r2;               // [32][LD] k e^{G - R} of the block's row half
    float* Xq = r2 + 32 * LD;     // [32][LD] q e^{G - R}
    float* Yk = r2 + 64 * LD;     // [32][LD] k e^{R - G} of the block's column half
    using TH = WarpTiles<32, D>;
    constexpr int NT = TH::NT;
    int hm0, hn0;
    TH::at(warp, hm0, hn0);
    for (int ho = 0; ho < 2; ++ho) {
      float aq[NT][4] = {}, ak[NT][4] = {}, aG[NT][4] = {};
      for (int blk = 0; blk < 3; ++blk) {
        const int a = blk == 0 ? 0 : 1, bb = blk == 1 ? 1 : 0, ref = blk == 0 ? 15 : 47;
        const bool rows_side = a == ho, cols_side = bb == ho;
        if (!rows_side && !cols_side) continue;  // same for every thread
        for (int i = tid; i < 32 * D; i += kThreads) {
          const int r = i / D, c = i % D;
          const float R = gS[ref * LD + c];
          const float er = __expf(gS[(32 * a + r) * LD + c] - R);
          Xk[r * LD + c] = kS[(32 * a + r) * LD + c] * er;
          Xq[r * LD + c] = qS[(32 * a + r) * LD + c] * er;
          Yk[r * LD + c] = kS[(32 * bb + r) * LD + c] * __expf(R - gS[(32 * bb + r) * LD + c]);
        }
        __syncthreads();
        if (rows_side) {  // rows r of half a: sum_s P_rs k_s e^{G_r - G_s}, sum_s dM_rs k_s e^{G_r - G_s}
          float t1[NT][4] = {}, t2[NT][4] = {};
          warp_mma<NT>(t1, PT + 32 * bb * LC, LC, 32 * a + hm0, Yk, LD, hn0, 32, lane);
          warp_mma<NT>(t2, dMT + 32 * bb * LC, LC, 32 * a + hm0, Yk, LD, hn0, 32, lane);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int r = 32 * a + frag_row(hm0, lane, e), c = frag_col(hn0, lane, nt, e);
              const float f = __expf(gS[r * LD + c] - gS[ref * LD + c]);
              const float pa = f * t1[nt][e], pm = f * t2[nt][e];
              ak[nt][e] += pa;
              aq[nt][e] += pm;
              aG[nt][e] += kS[r * LD + c] * pa + qS[r * LD + c] * pm;
            }
        }
        if (cols_side) {  // rows s of half bb: sum_r P_rs k_r e^{G_r - G_s}, sum_r dM_rs q_r e^{G_r - G_s}
          float t3[NT][4] = {}, t4[NT][4] = {};
          warp_mma<NT>(t3, PS + 32 * a * LC, LC, 32 * bb + hm0, Xk, LD, hn0, 32, lane);
          warp_mma<NT>(t4, dMs + 32 * a * LC, LC, 32 * bb + hm0, Xq, LD, hn0, 32, lane);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int s_ = 32 * bb + frag_row(hm0, lane, e), c = frag_col(hn0, lane, nt, e);
              const float f = __expf(gS[ref * LD + c] - gS[s_ * LD + c]);
              const float pa = f * t3[nt][e], pm = f * t4[nt][e];
              ak[nt][e] += pa + pm;
              aG[nt][e] -= kS[s_ * LD + c] * (pa + pm);
            }
        }
        __syncthreads();
      }
      // dK_hat = T^T dW (columns 32 ho.. of T and all of dW staged over the operand tiles), and the
      // terms through Q_hat, K_hat and K_bar
      constexpr int L36 = 32 + 4;
      float* Tsl = r2;            // [C][36]: T[k][32 ho + m]
      float* dWs = r2 + kC * L36;  // [C][LD]
      static_assert(kC * L36 + kC * LD <= SM::R2, "T slab and dW fit over the operand tiles");
      stage_async(Tsl, L36, rec + L.T() + 32 * ho, kC, kC, 32, tid);
      stage_async(dWs, LD, gr + GL.dW(), D, kC, D, tid);
      stage_wait();
      __syncthreads();
      {
        float t5[NT][4] = {};
        warp_mma<NT>(t5, Tsl, L36, hm0, dWs, LD, hn0, kC, lane);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = 32 * ho + frag_row(hm0, lane, e), c = frag_col(hn0, lane, nt, e);
            const float G = gS[r * LD + c], Gc = gS[(kC - 1) * LD + c];
            const float gam = __expf(G), eb = __expf(Gc - G), kv = kS[r * LD + c], qv = qS[r * LD + c];
            const float dqh = gr[GL.dQh() + (size_t)r * D + c], dkb = gr[GL.dKb() + (size_t)r * D + c];
            aq[nt][e] += dqh * gam;
            ak[nt][e] += t5[nt][e] * gam + dkb * eb;
            aG[nt][e] += dqh * qv * gam + t5[nt][e] * kv * gam - dkb * kv * eb;
          }
      }
      frag_store<NT>(dq + ((size_t)(t0 + 32 * ho) * H + h) * D, (size_t)H * D, aq, hm0, hn0, lane, 1.f, n - 32 * ho);
      frag_store<NT>(dk + ((size_t)(t0 + 32 * ho) * H + h) * D, (size_t)H * D, ak, hm0, hn0, lane, 1.f, n - 32 * ho);
      __syncthreads();  // q rows of this half and the staged tiles are no longer read
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          qS[(32 * ho + frag_row(hm0, lane, e)) * LD + frag_col(hn0, lane, nt, e)] = aG[nt][e];
      __syncthreads();
    }
    // ---- dg: reverse cumulative sum of dG, with G_C's terms on the last row
    if (tid < D) {
      const int c = tid;
      const float Gc = gS[(kC - 1) * LD + c];
      float last = gr[GL.dGam() + c] * __expf(Gc);
      for (int r = 0; r < kC; ++r)
        last = fmaf(gr[GL.dKb() + (size_t)r * D + c], kS[r * LD + c] * __expf(Gc - gS[r * LD + c]), last);
      float run = last;
      for (int r = kC - 1; r >= 0; --r) {
        run += qS[r * LD + c];
        if (r < n) dg[((size_t)(t0 + r) * H + h) * D + c] = run;
      }
    }
    if (tid < n) dbeta[(size_t)(t0 + tid) * H + h] = dbS[tid];
    __syncthreads();
  }
}

// ---------------------------------------------------------------- host side
int serial_slices(int B, int H, int E) {  // value-column slices of the two serial passes
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 1;
  const int64_t chains = (int64_t)B * H;
  for (int n = 8; n > 1; n /= 2)
    if (chains * n <= (int64_t)sms && E / n >= 16) return n;
  return E > 64 ? 2 : 1;  // at most 64 columns per slice (shared memory)
}

template <int D, int E, int ES, typename Tin>
cudaError_t launch_serial(const BackwardArgs& a, const float* recs, float* states, cudaStream_t st) {
  constexpr size_t fs = FwdSmem<D, E, ES>::floats * sizeof(float), rs = RevSmem<D, E, ES>::floats * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(bwd_fwd<D, E, ES>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fs);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_rev<D, E, ES, Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rs);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)a.B, (unsigned)a.H, (unsigned)(E / ES));
  bwd_fwd<D, E, ES><<<grid, kThreads, fs, st>>>(recs, a.h0, a.plan, a.cu_seqlens, a.B, a.T, a.H, states);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_rev<D, E, ES, Tin><<<grid, kThreads, rs, st>>>(recs, static_cast<const Tin*>(a.dout), a.dhT, a.plan,
                                                       a.cu_seqlens, a.B, a.T, a.H, states, a.dh0);
  return cudaGetLastError();
}

template <int D, int E, typename Tin>
cudaError_t launch_chunked(const BackwardArgs& a, float* ws, cudaStream_t st) {
  static DeviceOnce once;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return cudaErrorInvalidDevice;
  constexpr size_t rec_smem = RecSmem<D, E>::floats * sizeof(float);
  constexpr size_t dv_smem = DvSmem<D, E>::floats * sizeof(float);
  constexpr size_t gr_smem = GradSmem<D>::floats * sizeof(float);
  const cudaError_t e0 = once.run(dev, [] {
    cudaError_t e = cudaFuncSetAttribute(bwd_rec<D, E, Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rec_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(bwd_dvsums<D, E, Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dv_smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(bwd_grads<D, E, Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gr_smem);
    return e;
  });
  if (e0 != cudaSuccess) return e0;
  const int64_t ntask = max_chunks(a.B, a.T, a.cu_seqlens != nullptr) * a.H;
  if (ntask == 0) return cudaSuccess;
  float* recs = ws;
  float* states = recs + (size_t)ntask * RecLayout{D, E}.size();
  float* grads = states + (size_t)ntask * StateLayout{D, E}.size();
  const int grid = (int)(ntask < sms ? ntask : sms);
  const Tin* q = static_cast<const Tin*>(a.q);
  const Tin* k = static_cast<const Tin*>(a.k);
  const Tin* v = static_cast<const Tin*>(a.v);
  {
    TraceScope ts("kda_bwd_records", st);
    bwd_rec<D, E, Tin><<<grid, kThreads, rec_smem, st>>>(q, k, v, a.g, a.beta, a.plan, a.cu_seqlens, a.B, a.T, a.H,
                                                          ntask, recs);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    TraceScope ts("kda_bwd_state_passes", st);
    const int nsl = serial_slices(a.B, a.H, E);
    // (serial_slices keeps every slice at 16 columns or more)
    cudaError_t e = nsl == 8   ? launch_serial<D, E, (E / 8 < 16 ? 16 : E / 8), Tin>(a, recs, states, st)
                    : nsl == 4 ? launch_serial<D, E, E / 4, Tin>(a, recs, states, st)
                    : nsl == 2 ? launch_serial<D, E, E / 2, Tin>(a, recs, states, st)
                               : launch_serial<D, E, (E > 64 ? 64 : E), Tin>(a, recs, states, st);
    if (e != cudaSuccess) return e;
  }
  TraceScope ts("kda_bwd_chunk_grads", st);
  bwd_dvsums<D, E, Tin><<<grid, kThreads, dv_smem, st>>>(v, static_cast<const Tin*>(a.dout), a.plan, a.cu_seqlens, a.B,
                                                          a.T, a.H, ntask, recs, states, grads, a.dv);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_grads<D, E, Tin><<<grid, kThreads, gr_smem, st>>>(q, k, a.g, a.beta, a.plan, a.cu_seqlens, a.B, a.T, a.H, ntask,
                                                         recs, grads, a.dq, a.dk, a.dg, a.dbeta);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_chunked_dims(const BackwardArgs& a, float* ws, cudaStream_t st) {
  if (a.dim_k == 128 && a.dim_v == 128) return launch_chunked<128, 128, Tin>(a, ws, st);
  if (a.dim_k == 64 && a.dim_v == 64) return launch_chunked<64, 64, Tin>(a, ws, st);
  if (a.dim_k == 128 && a.dim_v == 64) return launch_chunked<128, 64, Tin>(a, ws, st);
  if (a.dim_k == 64 && a.dim_v == 128) return launch_chunked<64, 128, Tin>(a, ws, st);
  return cudaErrorInvalidValue;
}

}  // namespace

size_t backward_chunked_bytes(int B, int64_t T, int H, int dk, int dv, bool has_cu) {
  const int64_t ntask = max_chunks(B, T, has_cu) * H;
  const size_t per = RecLayout{dk, dv}.size() + StateLayout{dk, dv}.size() + GradLayout{dk}.size();
  return (size_t)ntask * per * sizeof(float);
}

cudaError_t backward_chunked_launch(const BackwardArgs& a, float* ws, cudaStream_t st) {
  return a.bf16 ? launch_chunked_dims<__nv_bfloat16>(a, ws, st) : launch_chunked_dims<float>(a, ws, st);
}

}  // namespace kda
