// KDA chunked prefill on CUDA cores in fp32 (the fp32-input path).
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
// plain dot products.  One reference per 64-token chunk could need exp(+-320)
// (fp32 overflows past exp(88.7)), so the chunk uses two 32-token halves with centred
// references (positions 15 and 47: every factor within exp(+-80)) for the two
// diagonal 32x32 blocks, and the reference 47 for the off-diagonal block (its
// key-side factor exp(G_47 - G_s) <= 1 never overflows).  Entries outside the causal
// mask can overflow to inf and are discarded by selection, never multiplied by 0.
//
// Two kernels:
//   chunk_prep_cc : one CTA per (chunk, head), fully parallel; writes the chunk's
//                   W, U_hat, Q_hat, K_bar, M and exp(G_last) into the workspace.
//   chunk_scan_cc : one CTA per (sequence, head); walks the chunks in order keeping
//                   the dk x dv state in shared memory; writes outputs (with the
//                   optional RMSNorm + sigmoid gate epilogue) and the final state.
#include <algorithm>

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 256;

template <int DK, int DV>
struct CcBlob {  // fp32 offsets inside one (chunk, head) record
  static constexpr size_t W = 0;
  static constexpr size_t UH = W + 64 * DK;
  static constexpr size_t QH = UH + 64 * DV;
  static constexpr size_t KB = QH + 64 * DK;
  static constexpr size_t M = KB + 64 * DK;
  static constexpr size_t GC = M + 64 * 64;
  static constexpr size_t FLOATS = (GC + DK + 63) / 64 * 64;
};

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}
__device__ __forceinline__ float comp(const float4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// C[64][N] (global, row-major) = T[64][64] (smem, pitch 65) x Bm[64][N] (smem, pitch PB)
template <int N>
__device__ __forceinline__ void tmul_store(const float* sT, const float* sB, int PB, float* outg) {
  const int rr = threadIdx.x / 16, cc = (threadIdx.x % 16) * 4;
  constexpr int JB = N / 64;
  float4 acc[4][JB];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int jb = 0; jb < JB; ++jb) acc[i][jb] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < 64; ++s) {
    float t[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) t[i] = sT[(rr + 16 * i) * 65 + s];
#pragma unroll
    for (int jb = 0; jb < JB; ++jb) {
      const float4 bv = *reinterpret_cast<const float4*>(&sB[s * PB + cc + 64 * jb]);
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i][jb] = f4_fma(t[i], bv, acc[i][jb]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int jb = 0; jb < JB; ++jb)
      *reinterpret_cast<float4*>(&outg[(size_t)(rr + 16 * i) * N + cc + 64 * jb]) = acc[i][jb];
}

template <int DK, int DV>
constexpr int prep_smem_floats() {
  constexpr int PM = (DK > DV ? DK : DV) + 4;
  return 64 * PM * 4 + 32 * PM + 64 * 65 + 64;
}

template <int DK, int DV, typename Tin>
__global__ void __launch_bounds__(kThreads, 1)
chunk_prep_cc(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
              const float* __restrict__ g, const float* __restrict__ beta,
              const int32_t* __restrict__ plan, const int32_t* __restrict__ cu, int B, int64_t T,
              int H, float* __restrict__ blob_base) {
  using L = CcBlob<DK, DV>;
  constexpr int PM = (DK > DV ? DK : DV) + 4;
  extern __shared__ float4 smem4[];
  float* sG = reinterpret_cast<float*>(smem4);  // [64][PM] cumulative log-decay
  float* sKL = sG + 64 * PM;                     // [64][PM] k * exp(G - R(r)); later K_hat
  float* sQL = sKL + 64 * PM;                    // [64][PM] q * exp(G - R(r)); later V
  float* sKR = sQL + 64 * PM;                    // [64][PM] k * exp(R(s) - G); later T
  float* sKX = sKR + 64 * PM;                    // [32][PM] k * exp(G_47 - G), s < 32
  float* sA = sKX + 32 * PM;                     // [64][65]
  float* sBeta = sA + 64 * 65;                   // [64]

  const int64_t chunk = blockIdx.x;
  const int h = blockIdx.y;
  int b, n;
  int64_t t0, cseq;
  if (!resolve_chunk(chunk, plan, cu, B, T, b, t0, n, cseq)) return;
  float* blob = blob_base + ((size_t)chunk * H + h) * L::FLOATS;
  const int tid = threadIdx.x;

  // 1. cumulative log-decay per key channel (padding rows: g = 0, so G stays flat)
  for (int c = tid; c < DK; c += kThreads) {
    float acc = 0.f;
    for (int r = 0; r < 64; ++r) {
      const float gv = (r < n) ? g[((size_t)(t0 + r) * H + h) * DK + c] : 0.f;
      acc += gv;
      sG[r * PM + c] = acc;
    }
  }
  if (tid < 64) sBeta[tid] = (tid < n) ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
  __syncthreads();

  // 2. reference-scaled operands for A and M
  for (int idx = tid; idx < 64 * DK; idx += kThreads) {
    const int r = idx / DK, c = idx % DK;
    const size_t gi = ((size_t)(t0 + r) * H + h) * DK + c;
    const float kv = (r < n) ? to_f32(k[gi]) : 0.f;
    const float qv = (r < n) ? to_f32(q[gi]) : 0.f;
    const float G = sG[r * PM + c];
    const float R = sG[(r < 32 ? 15 : 47) * PM + c];
    const float ef = expf(G - R), eb = expf(R - G);
    sKL[r * PM + c] = kv * ef;
    sQL[r * PM + c] = qv * ef;
    sKR[r * PM + c] = kv * eb;
    if (r < 32) sKX[r * PM + c] = kv * expf(sG[47 * PM + c] - G);
  }
  __syncthreads();

  // 3. A (strict lower, row-scaled by beta) and M (lower incl. diagonal)
  {
    const int rr = tid / 16, ss = tid % 16;
    float accA[4][4], accM[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) accA[i][j] = accM[i][j] = 0.f;
    for (int c = 0; c < DK; c += 4) {
      float4 kl[4], ql[4], kr[4], kx[2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        kl[i] = *reinterpret_cast<const float4*>(&sKL[(rr + 16 * i) * PM + c]);
        ql[i] = *reinterpret_cast<const float4*>(&sQL[(rr + 16 * i) * PM + c]);
        kr[i] = *reinterpret_cast<const float4*>(&sKR[(ss + 16 * i) * PM + c]);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) kx[j] = *reinterpret_cast<const float4*>(&sKX[(ss + 16 * j) * PM + c]);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (i < 2 && j >= 2) continue;  // upper off-diagonal block: always masked
          const float4 bb = (i >= 2 && j < 2) ? kx[j] : kr[j];
          accA[i][j] += dot4(kl[i], bb);
          accM[i][j] += dot4(ql[i], bb);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = rr + 16 * i, s = ss + 16 * j;
        sA[r * 65 + s] = (s < r) ? sBeta[r] * accA[i][j] : 0.f;
        blob[L::M + r * 64 + s] = (s <= r) ? accM[i][j] : 0.f;
      }
  }
  __syncthreads();

  // 4. K_hat and V into shared memory; Q_hat, K_bar, exp(G_last) into the blob
  float* sKH = sKL;
  float* sV = sQL;
  for (int idx = tid; idx < 64 * DK; idx += kThreads) {
    const int r = idx / DK, c = idx % DK;
    const size_t gi = ((size_t)(t0 + r) * H + h) * DK + c;
    const float kv = (r < n) ? to_f32(k[gi]) : 0.f;
    const float qv = (r < n) ? to_f32(q[gi]) : 0.f;
    const float G = sG[r * PM + c];
    const float eG = expf(G);
    sKH[r * PM + c] = kv * eG;
    blob[L::QH + r * DK + c] = qv * eG;
    blob[L::KB + r * DK + c] = kv * expf(sG[63 * PM + c] - G);
  }
  for (int idx = tid; idx < 64 * DV; idx += kThreads) {
    const int r = idx / DV, j = idx % DV;
    sV[r * PM + j] = (r < n) ? to_f32(v[((size_t)(t0 + r) * H + h) * DV + j]) : 0.f;
  }
  for (int c = tid; c < DK; c += kThreads) blob[L::GC + c] = expf(sG[63 * PM + c]);

  // 5. T = (I + A)^-1 Diag(beta): forward substitution, 4 threads per column s
  float* sT = sKR;
  {
    const int s = tid >> 2, part = tid & 3;
    float x[16];  // x[jj] = X[4 jj + part][s]
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
    for (int jj = 0; jj < 16; ++jj) sT[(4 * jj + part) * 65 + s] = x[jj] * bs;
  }
  __syncthreads();

  // 6. W = T K_hat, U_hat = T V
  tmul_store<DK>(sT, sKH, PM, blob + L::W);
  tmul_store<DV>(sT, sV, PM, blob + L::UH);
}

template <int DK, int DV>
constexpr int scan_smem_floats() {
  return DK * (DV + 4) + 64 * (DV + 4) + 64 * (DK + 4) + 64 * 68 + DK;
}

template <int DK, int DV, typename Tin, typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
chunk_scan_cc(const float* __restrict__ blob_base, const int32_t* __restrict__ plan,
              const int32_t* __restrict__ cu, int B, int64_t T, int H, const float* __restrict__ h0,
              float* __restrict__ hT, Tout* __restrict__ out, const Tin* __restrict__ gate,
              const float* __restrict__ norm_w, float eps, float* __restrict__ ckpt, int64_t ckpt_chunks) {
  using L = CcBlob<DK, DV>;
  constexpr int PSV = DV + 4, PSK = DK + 4, JB = DV / 64, SI = DK / 16;
  extern __shared__ float4 smem4[];
  float* sS = reinterpret_cast<float*>(smem4);  // [DK][PSV] state
  float* sU = sS + DK * PSV;                     // [64][PSV] U_hat, then U
  float* sX = sU + 64 * PSV;                     // [64][PSK] W, then Q_hat, then K_bar
  float* sM = sX + 64 * PSK;                     // [64][68]
  float* sGam = sM + 64 * 68;                    // [DK]

  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  if (cu != nullptr && plan[B + 1] == 0) return;  // invalid cu_seqlens: sequence skipped
  int64_t first_chunk, t_begin, len;
  const int64_t nchunks = sequence_chunks(b, plan, cu, B, T, first_chunk, t_begin, len);

  const size_t soff = ((size_t)b * H + h) * DK * DV;
  const int64_t ck_base = ckpt != nullptr ? checkpoint_base(b, cu, T, 64 * ckpt_chunks) : 0;
  for (int idx = tid; idx < DK * DV; idx += kThreads) {
    const int r = idx / DV, j = idx % DV;
    sS[r * PSV + j] = h0 ? h0[soff + idx] : 0.f;
  }
  __syncthreads();

  const int rr = tid / 16, cc = (tid % 16) * 4;
  for (int64_t c = 0; c < nchunks; ++c) {
    const float* blob = blob_base + ((size_t)(first_chunk + c) * H + h) * L::FLOATS;
    const int64_t rem = len - 64 * c;
    const int n = (int)(rem < 64 ? rem : 64);
    const int64_t t0 = t_begin + 64 * c;

    // a. W -> sX, U_hat -> sU, exp(G_last) -> sGam
    for (int idx = tid; idx < 64 * DK / 4; idx += kThreads) {
      const int r = idx / (DK / 4), c4 = (idx % (DK / 4)) * 4;
      *reinterpret_cast<float4*>(&sX[r * PSK + c4]) = *reinterpret_cast<const float4*>(&blob[L::W + r * DK + c4]);
    }
    for (int idx = tid; idx < 64 * DV / 4; idx += kThreads) {
      const int r = idx / (DV / 4), c4 = (idx % (DV / 4)) * 4;
      *reinterpret_cast<float4*>(&sU[r * PSV + c4]) = *reinterpret_cast<const float4*>(&blob[L::UH + r * DV + c4]);
    }
    for (int i = tid; i < DK; i += kThreads) sGam[i] = blob[L::GC + i];
    __syncthreads();

    // b. U = U_hat - W S
    {
      float4 acc[4][JB];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jb = 0; jb < JB; ++jb)
          acc[i][jb] = *reinterpret_cast<const float4*>(&sU[(rr + 16 * i) * PSV + cc + 64 * jb]);
      for (int c4 = 0; c4 < DK; c4 += 4) {
        float4 w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = *reinterpret_cast<const float4*>(&sX[(rr + 16 * i) * PSK + c4]);
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int jb = 0; jb < JB; ++jb) {
            const float4 sv = *reinterpret_cast<const float4*>(&sS[(c4 + u) * PSV + cc + 64 * jb]);
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i][jb] = f4_fma(-comp(w[i], u), sv, acc[i][jb]);
          }
      }
      __syncthreads();  // all reads of sX (W) done
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jb = 0; jb < JB; ++jb)
          *reinterpret_cast<float4*>(&sU[(rr + 16 * i) * PSV + cc + 64 * jb]) = acc[i][jb];
    }
    // c. Q_hat -> sX, M -> sM
    for (int idx = tid; idx < 64 * DK / 4; idx += kThreads) {
      const int r = idx / (DK / 4), c4 = (idx % (DK / 4)) * 4;
      *reinterpret_cast<float4*>(&sX[r * PSK + c4]) = *reinterpret_cast<const float4*>(&blob[L::QH + r * DK + c4]);
    }
    for (int idx = tid; idx < 64 * 16; idx += kThreads) {
      const int r = idx / 16, c4 = (idx % 16) * 4;
      *reinterpret_cast<float4*>(&sM[r * 68 + c4]) = *reinterpret_cast<const float4*>(&blob[L::M + r * 64 + c4]);
    }
    __syncthreads();

    // d. O = Q_hat S + M U
    float4 o[4][JB];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int jb = 0; jb < JB; ++jb) o[i][jb] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c4 = 0; c4 < DK; c4 += 4) {
      float4 qq[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) qq[i] = *reinterpret_cast<const float4*>(&sX[(rr + 16 * i) * PSK + c4]);
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int jb = 0; jb < JB; ++jb) {
          const float4 sv = *reinterpret_cast<const float4*>(&sS[(c4 + u) * PSV + cc + 64 * jb]);
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i][jb] = f4_fma(comp(qq[i], u), sv, o[i][jb]);
        }
    }
    for (int s4 = 0; s4 < 64; s4 += 4) {
      float4 mm[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) mm[i] = *reinterpret_cast<const float4*>(&sM[(rr + 16 * i) * 68 + s4]);
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int jb = 0; jb < JB; ++jb) {
          const float4 uv = *reinterpret_cast<const float4*>(&sU[(s4 + u) * PSV + cc + 64 * jb]);
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i][jb] = f4_fma(comp(mm[i], u), uv, o[i][jb]);
        }
    }

    // e. optional epilogue, store valid rows
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = rr + 16 * i;
      const size_t orow = ((size_t)(t0 + r) * H + h) * DV;
      float scale = 1.f;
      if (gate != nullptr) {
        float ss = 0.f;
#pragma unroll
        for (int jb = 0; jb < JB; ++jb) ss += dot4(o[i][jb], o[i][jb]);
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        ss += __shfl_xor_sync(0xffffffffu, ss, 4);
        ss += __shfl_xor_sync(0xffffffffu, ss, 8);
        scale = rsqrtf(ss / (float)DV + eps);
      }
      if (r < n) {
#pragma unroll
        for (int jb = 0; jb < JB; ++jb)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int col = cc + 64 * jb + e;
            float y = comp(o[i][jb], e);
            if (gate != nullptr) {
              const float wj = norm_w ? norm_w[col] : 1.f;
              y = y * scale * wj * sigmoidf_(to_f32(gate[orow + col]));
            }
            out[orow + col] = from_f32<Tout>(y);
          }
      }
    }
    __syncthreads();  // all reads of sX (Q_hat) done

    // f. K_bar -> sX
    for (int idx = tid; idx < 64 * DK / 4; idx += kThreads) {
      const int r = idx / (DK / 4), c4 = (idx % (DK / 4)) * 4;
      *reinterpret_cast<float4*>(&sX[r * PSK + c4]) = *reinterpret_cast<const float4*>(&blob[L::KB + r * DK + c4]);
    }
    __syncthreads();

    // g. S = Diag(exp G_last) S + K_bar^T U
    {
      float4 acc[SI][JB];
#pragma unroll
      for (int i = 0; i < SI; ++i) {
        const float gm = sGam[rr + 16 * i];
#pragma unroll
        for (int jb = 0; jb < JB; ++jb) {
          float4 sv = *reinterpret_cast<const float4*>(&sS[(rr + 16 * i) * PSV + cc + 64 * jb]);
          sv.x *= gm; sv.y *= gm; sv.z *= gm; sv.w *= gm;
          acc[i][jb] = sv;
        }
      }
      for (int r = 0; r < 64; ++r) {
        float4 uv[JB];
#pragma unroll
        for (int jb = 0; jb < JB; ++jb) uv[jb] = *reinterpret_cast<const float4*>(&sU[r * PSV + cc + 64 * jb]);
#pragma unroll
        for (int i = 0; i < SI; ++i) {
          const float kb = sX[r * PSK + rr + 16 * i];
#pragma unroll
          for (int jb = 0; jb < JB; ++jb) acc[i][jb] = f4_fma(kb, uv[jb], acc[i][jb]);
        }
      }
#pragma unroll
      for (int i = 0; i < SI; ++i)
#pragma unroll
        for (int jb = 0; jb < JB; ++jb)
          *reinterpret_cast<float4*>(&sS[(rr + 16 * i) * PSV + cc + 64 * jb]) = acc[i][jb];
    }
    __syncthreads();
    // state checkpoint after every ckpt_chunks full chunks (sS is next written by step g of a
    // later chunk, after further barriers)
    if (ckpt != nullptr && (c + 1) % ckpt_chunks == 0 && (c + 1) * 64 <= len) {
      float* dst = ckpt + ((size_t)(ck_base + (c + 1) / ckpt_chunks - 1) * H + h) * DK * DV;
      for (int idx = tid; idx < DK * DV; idx += kThreads) dst[idx] = sS[(idx / DV) * PSV + idx % DV];
    }
  }

  if (hT != nullptr)
    for (int idx = tid; idx < DK * DV; idx += kThreads) {
      const int r = idx / DV, j = idx % DV;
      hT[soff + idx] = sS[r * PSV + j];
    }
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
  using L = CcBlob<DK, DV>;
  const size_t prep_smem = prep_smem_floats<DK, DV>() * sizeof(float);
  const size_t scan_smem = scan_smem_floats<DK, DV>() * sizeof(float);
  static DeviceOnce once;  // per instantiation
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const cudaError_t e0 = once.run(dev, [prep_smem, scan_smem] {
    cudaError_t e = cudaFuncSetAttribute(chunk_prep_cc<DK, DV, Tin>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)prep_smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(chunk_scan_cc<DK, DV, Tin, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)scan_smem);
  });
  if (e0 != cudaSuccess) return e0;
  const bool has_cu = a.cu_seqlens != nullptr;
  const int64_t nchunks = max_chunks(a.B, a.T, has_cu);
  int32_t* plan = static_cast<int32_t*>(a.workspace);
  float* blob = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + plan_bytes(a.B));
  (void)L::FLOATS;
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
  dim3 grid2((unsigned)a.B, (unsigned)a.H);
  TraceScope ts("kda_chunk_scan_cc", st);
  chunk_scan_cc<DK, DV, Tin, Tout><<<grid2, kThreads, scan_smem, st>>>(
      blob, plan, a.cu_seqlens, a.B, a.T, a.H, a.h0, a.hT, static_cast<Tout*>(a.out),
      static_cast<const Tin*>(a.epi.gate), a.epi.norm_weight, a.epi.eps, a.ckpt, a.ckpt_chunks);
  return cudaGetLastError();
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
  return (((size_t)64 * (3 * dk + dv) + 64 * 64 + dk + 63) / 64 * 64) * sizeof(float);
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
