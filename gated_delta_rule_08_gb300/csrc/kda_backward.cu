// KDA backward: gradients of L = sum_t <dout_t, o_t> + <dhT, hT> with respect to q, k, v, g, beta
// and h0, for the recurrence of the prefill (no epilogue).
//
// Kimi K3: Open Frontier Intelligence (kimi-k3-paper.pages.dev), section 2.2 Eq. 1 and section
// 2.4 Eq. 3, per (sequence, head), with P_t = Diag(alpha_t) S_{t-1}, alpha_t = exp(g_t):
//   u_t = v_t - P_t^T k_t,   S_t = P_t + beta_t k_t u_t^T,   o_t = S_t^T q_t.
// Reverse-mode, token by token (dS = dL/dS_t, accumulated from later tokens):
//   dS   += q_t dout_t^T                      dq_t    = S_t dout_t
//   w     = dS u_t                            dbeta_t = k_t . w
//   du    = beta_t dS^T k_t                   dv_t    = du
//   dk_t  = beta_t w - P_t du
//   dP    = dS - k_t du^T                     dg_t    = alpha_t (.) rowsum(dP (.) S_{t-1})
//   dS_{t-1} = Diag(alpha_t) dP               dh0     = dS_0
// (section 5.1 names a training kernel for KDA; this one is a plain, exact-arithmetic-faithful
// fp32 form, not a chunkwise one).
//
//  kda_bwd_token<DK, DV, NSL, Tin> (one CTA per (sequence, head, value-column slice), 256
//  threads): the recurrence is separable in the value columns of the state, so NSL CTAs each take
//  DV / NSL columns; their contributions to dq, dk, dg, dbeta (sums over the columns) meet by
//  atomic adds onto zeroed outputs — with NSL <= 2 that sum is order-independent, so the result
//  is deterministic.  The state slice lives in registers as in the decode kernel (thread = 4
//  value columns x DK/NG rows).  A forward sweep
//  stores the state at every chunk start; then, chunk by chunk from the end, the 64 token states
//  of the chunk are recomputed into scratch and the chunk's tokens are walked backwards.  Column
//  sums go through shared memory, row sums through a segmented butterfly of warp shuffles.
#include <cstdlib>
#include <cstring>

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kBwdThreads = 256;  // one or two value-column slices per chain
constexpr int kBwdThreads4 = 128;  // four slices per chain: each thread keeps the same share of its slice

// Sums, over the L lanes of a lane segment, R per-row partials per lane (R <= L, powers of two).
// Afterwards vals[0] holds the full sum of local row `row_of(lane)`; the lanes that share a row all
// hold it, and `owner` is true for exactly one of them.
template <int R, int L>
__device__ __forceinline__ float seg_row_reduce(float (&vals)[R], int lane, int& row, bool& owner) {
  int m = R, base = 0;
#pragma unroll
  for (int o = L / 2; o >= 1; o >>= 1) {
    if (m > 1) {
      const int h = m / 2;
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int k = 0; k < R / 2; ++k) {
        if (k < h) {
          const float send = up ? vals[k] : vals[h + k];
          const float recv = __shfl_xor_sync(0xffffffffu, send, o);
          vals[k] = (up ? vals[h + k] : vals[k]) + recv;
        }
      }
      if (up) base += h;
      m = h;
    } else {
      vals[0] += __shfl_xor_sync(0xffffffffu, vals[0], o);
    }
  }
  row = base;
  owner = (lane & (L / R - 1)) == 0;
  return vals[0];
}

__device__ __forceinline__ float dot4(float4 a, float4 b) { return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w; }
__device__ __forceinline__ float4 f4_axpy(float a, float4 x, float4 y) {  // a x + y
  return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}
__device__ __forceinline__ float4 f4_scale(float a, float4 x) { return make_float4(a * x.x, a * x.y, a * x.z, a * x.w); }
__device__ __forceinline__ float4 f4_sub(float4 a, float4 b) { return make_float4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w); }

template <int DK, int DV, int THREADS>
struct BwdShared {
  static constexpr int TPR = DV / 4, NG = THREADS / TPR;
  float k[DK], q[DK], al[DK], v[DV], dout[DV];
  float beta;
  float4 partA[NG][TPR], partB[NG][TPR];
  float dbeta[THREADS / 32];
};

template <int DK, int DV, int NSL, typename Tin, int THREADS = NSL == 4 ? kBwdThreads4 : kBwdThreads>
__global__ void __launch_bounds__(THREADS, 1)
kda_bwd_token(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
              const float* __restrict__ g, const float* __restrict__ beta, const float* __restrict__ h0,
              const int32_t* __restrict__ plan, const int32_t* __restrict__ cu, int B, int64_t T, int H,
              const Tin* __restrict__ dout, const float* __restrict__ dhT, float* __restrict__ dq,
              float* __restrict__ dk, float* __restrict__ dv, float* __restrict__ dg, float* __restrict__ dbeta,
              float* __restrict__ dh0, float* __restrict__ ckpt, float* __restrict__ tokbuf,
              float* __restrict__ side) {
  constexpr int DVS = DV / NSL;  // value columns of this CTA's slice
  using SH = BwdShared<DK, DVS, THREADS>;
  constexpr int TPR = SH::TPR, NG = SH::NG, RPG = DK / NG;
  // each output element receives at most two addends onto zero (order-independent); with four
  // slices, slices 2 and 3 add into `side` (dq, dk, dg, dbeta in the same layout), summed after
  static_assert(NSL == 1 || NSL == 2 || NSL == 4, "slices");
  static_assert(DK % NG == 0 && RPG <= TPR, "layout");
  __shared__ SH sh;
  const int b = blockIdx.x, h = blockIdx.y, slice = blockIdx.z, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j0 = slice * DVS;
  const int cg = tid % TPR, rg = tid / TPR;
  const int seg_lane = lane % TPR;  // lane within this row's lane segment
  if (cu != nullptr && plan[B + 1] == 0) return;  // invalid cu_seqlens: sequence skipped
  int64_t first_chunk, t_begin, len;
  const int64_t nch = sequence_chunks(b, plan, cu, B, T, first_chunk, t_begin, len);
  constexpr size_t MAT = (size_t)DK * DVS;  // one state slice in scratch
  const size_t soff = ((size_t)b * H + h) * DK * DV + j0;  // this slice in [B, H, DK, DV] states
  float* tb = tokbuf + (((size_t)b * H + h) * NSL + slice) * 64 * MAT;
  auto ck = [&](int64_t c) { return ckpt + (((size_t)(first_chunk + c) * H + h) * NSL + slice) * MAT; };
  // this thread's elements: rows rg + i NG, columns 4 cg .. 4 cg + 3 of the slice (row stride ld)
  auto ld_state = [&](const float* src, float4 (&s)[RPG], int ld) {
#pragma unroll
    for (int i = 0; i < RPG; ++i) s[i] = __ldcg(reinterpret_cast<const float4*>(src + (size_t)(rg + i * NG) * ld) + cg);
  };
  auto st_state = [&](float* dst, const float4 (&s)[RPG], int ld) {
#pragma unroll
    for (int i = 0; i < RPG; ++i) __stcg(reinterpret_cast<float4*>(dst + (size_t)(rg + i * NG) * ld) + cg, s[i]);
  };
  const size_t rows_tot = (size_t)(cu != nullptr ? T : (int64_t)B * T) * H;
  // one column slice's share of a row gradient; `dst` points into dq, dk or dg ([rows][DK]) or
  // dbeta ([rows]), whose copies in `side` follow each other: dq, dk, dg, dbeta
  auto out_row = [&](float* dst, size_t side_off, float x) {
    if (NSL == 1) *dst = x;
    else if (NSL == 2 || slice < 2) atomicAdd(dst, x);
    else atomicAdd(side + side_off, x);
  };
  // token vectors into shared memory (rows past the sequence end never occur here)
  auto load_token = [&](int64_t t, bool with_q) {
    const size_t row = (size_t)t * H + h;
    for (int i = tid; i < DK; i += THREADS) {
      sh.k[i] = to_f32(k[row * DK + i]);
      sh.al[i] = __expf(g[row * DK + i]);
      if (with_q) sh.q[i] = to_f32(q[row * DK + i]);
    }
    for (int j = tid; j < DVS; j += THREADS) {
      sh.v[j] = to_f32(v[row * DV + j0 + j]);
      if (with_q) sh.dout[j] = to_f32(dout[row * DV + j0 + j]);
    }
    if (tid == 0) sh.beta = beta[row];
  };
  // S <- (I - beta k k^T) Diag(alpha) S + beta k v^T for token t
  auto fwd_step = [&](int64_t t, float4 (&s)[RPG]) {
    load_token(t, false);
    __syncthreads();
    float4 pa = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
      const int r = rg + i * NG;
      s[i] = f4_scale(sh.al[r], s[i]);
      pa = f4_axpy(sh.k[r], s[i], pa);
    }
    sh.partA[rg][cg] = pa;
    __syncthreads();
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      const float4 x = sh.partA[gi][cg];
      a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
    }
    const float4 v4 = reinterpret_cast<const float4*>(sh.v)[cg];
    const float4 d4 = f4_scale(sh.beta, f4_sub(v4, a));
#pragma unroll
    for (int i = 0; i < RPG; ++i) s[i] = f4_axpy(sh.k[rg + i * NG], d4, s[i]);
    __syncthreads();  // shared token vectors are rewritten by the next step
  };

  // ---- forward sweep: the state at every chunk start
  {
    float4 s[RPG];
    if (h0 != nullptr) ld_state(h0 + soff, s, DV);
    else
#pragma unroll
      for (int i = 0; i < RPG; ++i) s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t c = 0; c < nch; ++c) {
      st_state(ck(c), s, DVS);
      const int64_t t0 = t_begin + 64 * c, n = len - 64 * c < 64 ? len - 64 * c : 64;
      for (int64_t t = t0; t < t0 + n; ++t) fwd_step(t, s);
    }
  }

  // ---- backward sweep, chunk by chunk from the end
  float4 ds[RPG];
  if (dhT != nullptr) ld_state(dhT + soff, ds, DV);
  else
#pragma unroll
    for (int i = 0; i < RPG; ++i) ds[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t c = nch - 1; c >= 0; --c) {
    const int64_t t0 = t_begin + 64 * c, n = len - 64 * c < 64 ? len - 64 * c : 64;
    {  // the chunk's token states S_{t-1}, recomputed from its start
      float4 s[RPG];
      ld_state(ck(c), s, DVS);
      for (int64_t j = 0; j < n; ++j) {
        st_state(tb + (size_t)j * MAT, s, DVS);
        if (j + 1 < n) fwd_step(t0 + j, s);
      }
    }
    for (int64_t j = n - 1; j >= 0; --j) {
      const int64_t t = t0 + j;
      const size_t row = (size_t)t * H + h;
      float4 sp[RPG];  // S_{t-1}
      ld_state(tb + (size_t)j * MAT, sp, DVS);
      load_token(t, true);
      __syncthreads();
      const float bt = sh.beta;
      const float4 do4 = reinterpret_cast<const float4*>(sh.dout)[cg];
      // u = v - P^T k (column sums); dS += q dout^T
      {
        float4 pa = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < RPG; ++i) {
          const int r = rg + i * NG;
          pa = f4_axpy(sh.k[r], f4_scale(sh.al[r], sp[i]), pa);
          ds[i] = f4_axpy(sh.q[r], do4, ds[i]);
        }
        sh.partA[rg][cg] = pa;
      }
      __syncthreads();
      float4 u4 = reinterpret_cast<const float4*>(sh.v)[cg];
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) u4 = f4_sub(u4, sh.partA[gi][cg]);
      // row sums dq = S_t dout, w = dS u; column sums dS^T k
      float rq[RPG], rw[RPG];
      {
        float4 pb = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < RPG; ++i) {
          const int r = rg + i * NG;
          const float4 st = f4_axpy(bt * sh.k[r], u4, f4_scale(sh.al[r], sp[i]));  // S_t = P + beta k u^T
          rq[i] = dot4(st, do4);
          rw[i] = dot4(ds[i], u4);
          pb = f4_axpy(sh.k[r], ds[i], pb);
        }
        sh.partB[rg][cg] = pb;
      }
      int rrow;
      bool owner;
      const float dq_row = seg_row_reduce<RPG, TPR>(rq, seg_lane, rrow, owner);
      const int my_row = rg + rrow * NG;
      if (owner) out_row(&dq[row * DK + my_row], row * DK + my_row, dq_row);
      const float w_row = seg_row_reduce<RPG, TPR>(rw, seg_lane, rrow, owner);
      __syncthreads();
      float4 du4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        const float4 x = sh.partB[gi][cg];
        du4.x += x.x; du4.y += x.y; du4.z += x.z; du4.w += x.w;
      }
      du4 = f4_scale(bt, du4);
      if (rg == 0) reinterpret_cast<float4*>(dv + row * DV + j0)[cg] = du4;
      // row sums P du and (dP (.) S_{t-1}); dS <- Diag(alpha) dP
      float rp[RPG], ra[RPG];
#pragma unroll
      for (int i = 0; i < RPG; ++i) {
        const int r = rg + i * NG;
        rp[i] = sh.al[r] * dot4(sp[i], du4);
        const float4 dP = f4_axpy(-sh.k[r], du4, ds[i]);
        ra[i] = dot4(dP, sp[i]);
        ds[i] = f4_scale(sh.al[r], dP);
      }
      const float pdu_row = seg_row_reduce<RPG, TPR>(rp, seg_lane, rrow, owner);
      const float da_row = seg_row_reduce<RPG, TPR>(ra, seg_lane, rrow, owner);
      float kw = 0.f;
      if (owner) {
        out_row(&dk[row * DK + my_row], rows_tot * DK + row * DK + my_row, bt * w_row - pdu_row);
        out_row(&dg[row * DK + my_row], 2 * rows_tot * DK + row * DK + my_row, sh.al[my_row] * da_row);
        kw = sh.k[my_row] * w_row;
      }
      kw = warp_sum(kw);
      if (lane == 0) sh.dbeta[warp] = kw;
      __syncthreads();
      if (tid == 0) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < THREADS / 32; ++w) s += sh.dbeta[w];
        out_row(&dbeta[row], 3 * rows_tot * DK + row, s);
      }
      __syncthreads();  // shared token vectors and partials are rewritten by the next token
    }
  }
  if (dh0 != nullptr) st_state(dh0 + soff, ds, DV);
}

// out += side for the four slices' second pair of addends (dq, dk, dg: n = rows x DK each; dbeta: rows)
__global__ void bwd_add_side(float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dg,
                             float* __restrict__ dbeta, const float* __restrict__ side, size_t n, size_t rows) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    dq[i] += side[i];
    dk[i] += side[n + i];
    dg[i] += side[2 * n + i];
  }
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < rows; i += stride) dbeta[i] += side[3 * n + i];
}

template <int DK, int DV, typename Tin>
cudaError_t launch_bwd_typed(const BackwardArgs& a, float* ckpt, float* tokbuf, float* side, cudaStream_t st) {
  const int nsl = backward_slices(a.B, a.H, a.dim_v);
  const int64_t T_tot = a.cu_seqlens ? a.T : (int64_t)a.B * a.T;
  const size_t rows = (size_t)T_tot * a.H;
  if (nsl > 1) {  // the slices' contributions are added onto zeros
    cudaError_t e = cudaMemsetAsync(a.dq, 0, rows * DK * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dk, 0, rows * DK * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dg, 0, rows * DK * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dbeta, 0, rows * sizeof(float), st);
    if (e == cudaSuccess && nsl == 4) e = cudaMemsetAsync(side, 0, (3 * rows * DK + rows) * sizeof(float), st);
    if (e != cudaSuccess) return e;
  }
  TraceScope ts("kda_bwd_token", st);
  const dim3 grid((unsigned)a.B, (unsigned)a.H, (unsigned)nsl);
#define KDA_BWD_ARGS                                                                                               \
  static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v), a.g, a.beta, a.h0,     \
      a.plan, a.cu_seqlens, a.B, a.T, a.H, static_cast<const Tin*>(a.dout), a.dhT, a.dq, a.dk, a.dv, a.dg, a.dbeta, \
      a.dh0, ckpt, tokbuf, side
  if (nsl == 4) {
    kda_bwd_token<DK, DV, 4, Tin><<<grid, kBwdThreads4, 0, st>>>(KDA_BWD_ARGS);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_add_side<<<1024, 256, 0, st>>>(a.dq, a.dk, a.dg, a.dbeta, side, rows * DK, rows);
  } else if (nsl == 2) {
    kda_bwd_token<DK, DV, 2, Tin><<<grid, kBwdThreads, 0, st>>>(KDA_BWD_ARGS);
  } else {
    kda_bwd_token<DK, DV, 1, Tin><<<grid, kBwdThreads, 0, st>>>(KDA_BWD_ARGS);
  }
#undef KDA_BWD_ARGS
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_bwd_dims(const BackwardArgs& a, float* ckpt, float* tokbuf, float* side, cudaStream_t st) {
  if (a.dim_k == 128 && a.dim_v == 128) return launch_bwd_typed<128, 128, Tin>(a, ckpt, tokbuf, side, st);
  if (a.dim_k == 64 && a.dim_v == 64) return launch_bwd_typed<64, 64, Tin>(a, ckpt, tokbuf, side, st);
  if (a.dim_k == 128 && a.dim_v == 64) return launch_bwd_typed<128, 64, Tin>(a, ckpt, tokbuf, side, st);
  if (a.dim_k == 64 && a.dim_v == 128) return launch_bwd_typed<64, 128, Tin>(a, ckpt, tokbuf, side, st);
  return cudaErrorInvalidValue;
}

}  // namespace

// Value-column slices per chain: as many (1, 2 or 4) as keep one CTA per chain slice within one
// wave of the device's SMs.
int backward_slices(int B, int H, int dv) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 1;
  const int64_t chains = (int64_t)B * H;
  if (chains * 4 <= sms && dv % 64 == 0) return 4;
  if (chains * 2 <= sms) return 2;
  return 1;
}

// The chunkwise backward keeps about 0.6 MB of fp32 scratch per (chunk, head) (dk = dv = 128); up to
// this much scratch it is used, beyond it the token sweep below (whose scratch is per chain).
constexpr size_t kChunkedMaxBytes = size_t(48) << 30;

// KDA_BACKWARD_PATH=token or =chunked in the environment forces one path (read at every call, so
// the workspace size and the call agree while it is unchanged).
bool use_chunked(int B, int64_t T, int H, int dk, int dv) {
  const char* forced = std::getenv("KDA_BACKWARD_PATH");
  if (forced != nullptr && std::strcmp(forced, "token") == 0) return false;
  if (forced != nullptr && std::strcmp(forced, "chunked") == 0) return true;
  return backward_chunked_bytes(B, T, H, dk, dv, true) <= kChunkedMaxBytes &&
         backward_chunked_bytes(B, T, H, dk, dv, false) <= kChunkedMaxBytes;
}

size_t backward_scratch_bytes(int B, int64_t T, int H, int dk, int dv, bool has_cu) {
  if (use_chunked(B, T, H, dk, dv)) return backward_chunked_bytes(B, T, H, dk, dv, has_cu);
  const size_t mat = (size_t)dk * dv * sizeof(float);
  size_t bytes = align_up((size_t)max_chunks(B, T, has_cu) * H * mat, 256) + align_up((size_t)B * H * 64 * mat, 256);
  if (backward_slices(B, H, dv) == 4) {  // the second pair of addends of dq, dk, dg, dbeta
    const size_t rows = (size_t)(has_cu ? T : (int64_t)B * T) * H;
    bytes += (3 * rows * dk + rows) * sizeof(float);
  }
  return bytes;
}

cudaError_t backward_launch(const BackwardArgs& a, cudaStream_t st) {
  uint8_t* ws = static_cast<uint8_t*>(a.workspace) + plan_bytes(a.B);
  if (use_chunked(a.B, a.T, a.H, a.dim_k, a.dim_v)) return backward_chunked_launch(a, reinterpret_cast<float*>(ws), st);
  const size_t mat = (size_t)a.dim_k * a.dim_v * sizeof(float);
  const size_t ck_bytes = align_up((size_t)max_chunks(a.B, a.T, a.cu_seqlens != nullptr) * a.H * mat, 256);
  float* ckpt = reinterpret_cast<float*>(ws);
  float* tokbuf = reinterpret_cast<float*>(ws + ck_bytes);
  float* side = reinterpret_cast<float*>(ws + ck_bytes + align_up((size_t)a.B * a.H * 64 * mat, 256));
  return a.bf16 ? launch_bwd_dims<__nv_bfloat16>(a, ckpt, tokbuf, side, st)
                : launch_bwd_dims<float>(a, ckpt, tokbuf, side, st);
}

}  // namespace kda
