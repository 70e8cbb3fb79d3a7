// KDA recurrent decode over a pool of fp32 states (in place), one or several tokens per request.
//
// Kimi K3 report walk-through (kimi-k3-paper.pages.dev): section 2.2 Eq. 1 (the
// per-token update), section 2.4 Eq. 3 (read-out), section 3.3 Eq. 6 (RMSNorm then
// sigmoid gate), section 13.10 (decode as one fused kernel: state update and
// read-out in a single call), section 13.9 (one fixed-size state per request in a
// pooled layout).
//
// Per (request n, head h) with S = pool[slot_idx[n], h] (dk x dv, rows = key channels):
//   S'    = Diag(exp g) S
//   a     = S'^T k,  b = S'^T q                  (reductions over dk)
//   delta = beta (v - a)
//   S_new = S' + k delta^T                       (== (I - beta k k^T) S' + beta k v^T)
//   o     = S_new^T q = b + (k . q) delta
//
// Multi-token form (section 13.4, the state problem of speculative decoding: an in-place update
// cannot be rolled back, so the verify pass must not overwrite the pooled state): a request may
// carry several tokens, applied in order to the state held in registers; the state is written
// back only when asked (commit), after exactly the request's own token count.  Verify = all
// draft tokens, no write-back; accept = the accepted prefix recomputed from the cached inputs,
// with write-back.  One token with write-back is the plain decode step.
//
// The kernel is bound by HBM bandwidth: it streams the 64 KB state in and out once.
// One CTA per (n, h); each thread owns 4 contiguous value columns (one float4) of
// DK / NG consecutive rows (so its rows' k, q and decay come four per 16-byte shared load),
// and a warp reads/writes whole 512-byte rows with 128-bit accesses;
// the whole state slice lives in registers between the load and the store.  The
// column reductions over dk are a register partial sum per thread followed by one
// shared-memory pass across the row groups.
#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kDecodeThreads = 256;

// two fp32 lanes per instruction (each lane rounded as fmaf / a plain product)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
constexpr int kStageTok = 4;  // tokens whose inputs are staged in shared memory together (multi-token calls)

template <int DK, int DV, int NST, typename Tin, typename Tout>
__global__ void __launch_bounds__(kDecodeThreads, 2)
decode_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
              const float* __restrict__ g, const float* __restrict__ beta, float* __restrict__ pool,
              const int32_t* __restrict__ slot_idx, Tout* __restrict__ out, int H, int num_slots, int n_tok,
              const int32_t* __restrict__ ntok_per_req, int commit, const Tin* __restrict__ gate,
              const float* __restrict__ norm_w, float eps, unsigned int* __restrict__ err) {
  constexpr int TPR = DV / 4;               // threads per state row
  constexpr int NG = kDecodeThreads / TPR;  // row groups
  constexpr int RPG = DK / NG;              // rows per thread
  static_assert(DK % NG == 0 && (DK / NG) % 4 == 0, "rows must split evenly, four per thread at least");

  const int nh = blockIdx.x;  // n * H + h
  const int n = nh / H, h = nh - (nh / H) * H;
  const int tid = threadIdx.x;
  const int cg = tid % TPR, rg = tid / TPR;

  const int slot = slot_idx[n];
  if (slot < 0 || slot >= num_slots) {
    if (tid == 0 && h == 0) atomicOr(err, KDA_DEVERR_BAD_SLOT);
    return;
  }
  int count = n_tok;
  if (ntok_per_req != nullptr) {
    count = ntok_per_req[n];
    if (count < 0 || count > n_tok) {
      if (tid == 0 && h == 0) atomicOr(err, KDA_DEVERR_BAD_COUNT);
      return;
    }
  }
  if (count == 0) return;  // nothing to apply: outputs and state untouched
  float* S = pool + ((size_t)slot * H + h) * (size_t)(DK * DV);

  // Several tokens per request: the inputs of a stage of up to NST tokens as raw values in
  // registers (loaded together, converted when stored to shared memory).  The first stage's are
  // issued before the state, so that they land first and their conversion overlaps the state's
  // arrival.
  constexpr int NLK = NST > 1 ? (NST * DK + kDecodeThreads - 1) / kDecodeThreads : 1;
  constexpr int VPT = 16 / (int)sizeof(Tin);  // elements per 16-byte copy of v or the gate
  __shared__ __align__(16) Tin sv_raw[NST > 1 ? NST : 1][NST > 1 ? DV : 8], sg_raw[NST > 1 ? NST : 1][NST > 1 ? DV : 8];
  struct StageRegs {
    Tin k[NLK], q[NLK];
    float g[NLK], b;
  };
  auto load_stage = [&](int t, StageRegs& R) {
    const int nst = count - t < NST ? count - t : NST;
    const size_t row0 = ((size_t)n * n_tok + t) * H + h;
#pragma unroll
    for (int j = 0; j < NLK; ++j) {
      const int i = tid + j * kDecodeThreads;
      if (i < nst * DK) {
        const int w = i / DK, c = i - w * DK;
        const size_t rk = (row0 + (size_t)w * H) * DK + c;
        R.k[j] = k[rk];
        R.q[j] = q[rk];
        R.g[j] = g[rk];
      }
    }
    // v and the gate: raw 16-byte pieces straight into shared memory (converted where used)
    if (tid < nst * DV / VPT) {
      const int w = tid / (DV / VPT), c = (tid % (DV / VPT)) * VPT;
      const size_t rw = (row0 + (size_t)w * H) * DV + c;
      cp_async16(&sv_raw[w][c], v + rw);
      if (gate != nullptr) cp_async16(&sg_raw[w][c], gate + rw);
    }
    cp_async_commit();
    R.b = tid < nst ? beta[row0 + (size_t)tid * H] : 0.f;
  };
  StageRegs R;
  if constexpr (NST > 1) load_stage(0, R);

  // Issue the state loads next: they are the longest-latency traffic.
  float4 s[RPG];
#pragma unroll
  for (int i = 0; i < RPG; ++i)
    s[i] = __ldcs(reinterpret_cast<const float4*>(S + (size_t)(rg * RPG + i) * DV) + cg);

  // the inputs of up to NST tokens, loaded together so that their latency is paid once
  __shared__ __align__(16) float sk[NST][DK], sq[NST][DK], salpha[NST][DK], sv[1][NST > 1 ? 1 : DV];
  __shared__ float sbeta[NST];
  __shared__ float4 part_a[NG][TPR], part_b[NG][TPR];
  __shared__ float sdelta[DV], so[NST][DV];
  __shared__ float red[kDecodeThreads / 32];
  __shared__ float s_kq, s_kq_st[NST];

  for (int t = 0; t < count; ++t) {
    const int u = t % NST;
    const size_t row = ((size_t)n * n_tok + t) * H + h;  // token row of [N, n_tok, H]
    const size_t rv = row * DV;
    float b_r;
    if constexpr (NST == 1) {  // one token per request (the launch for n_tok = 1)
      const size_t rk = row * DK;
      for (int i = tid; i < DK; i += kDecodeThreads) {
        sk[0][i] = to_f32(k[rk + i]);
        sq[0][i] = to_f32(q[rk + i]);
        salpha[0][i] = __expf(g[rk + i]);
      }
      for (int j = tid; j < DV; j += kDecodeThreads) sv[0][j] = to_f32(v[rv + j]);
      b_r = beta[row];
      __syncthreads();
    } else if (u == 0) {
      if (t > 0) {
        __syncthreads();  // the previous stage is no longer read
        load_stage(t, R);
      }
      const int nst = count - t < NST ? count - t : NST;
#pragma unroll
      for (int j = 0; j < NLK; ++j) {
        const int i = tid + j * kDecodeThreads;
        if (i < nst * DK) {
          const int w = i / DK, c = i - w * DK;
          sk[w][c] = to_f32(R.k[j]);
          sq[w][c] = to_f32(R.q[j]);
          salpha[w][c] = __expf(R.g[j]);
        }
      }
      if (tid < nst) sbeta[tid] = R.b;
      cp_async_wait_all();  // this thread's v and gate pieces
      __syncthreads();
      // k . q of every staged token, one warp each, read after the token's first barrier
      if (tid < 32 * nst) {
        const int w = tid >> 5;
        float acc = 0.f;
        for (int i = tid & 31; i < DK; i += 32) acc = fmaf(sk[w][i], sq[w][i], acc);
        acc = warp_sum(acc);
        if ((tid & 31) == 0) s_kq_st[w] = acc;
      }
    }
    if constexpr (NST > 1) b_r = sbeta[u];

    if (NST == 1 && tid < 32) {  // k . q
      float acc = 0.f;
      for (int i = tid; i < DK; i += 32) acc = fmaf(sk[u][i], sq[u][i], acc);
      acc = warp_sum(acc);
      if (tid == 0) s_kq = acc;
    }

    float2 pa01 = make_float2(0.f, 0.f), pa23 = pa01, pb01 = pa01, pb23 = pa01;
#pragma unroll
    for (int i4 = 0; i4 < RPG; i4 += 4) {  // this thread's rows rg RPG + i: four per 16-byte load
      const float4 al4 = *reinterpret_cast<const float4*>(&salpha[u][rg * RPG + i4]);
      const float4 k4 = *reinterpret_cast<const float4*>(&sk[u][rg * RPG + i4]);
      const float4 q4 = *reinterpret_cast<const float4*>(&sq[u][rg * RPG + i4]);
      const float al[4] = {al4.x, al4.y, al4.z, al4.w}, kk[4] = {k4.x, k4.y, k4.z, k4.w},
                  qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float4& x = s[i4 + e];
        const float2 a2 = make_float2(al[e], al[e]), k2 = make_float2(kk[e], kk[e]), q2 = make_float2(qq[e], qq[e]);
        const float2 x01 = fmul2(make_float2(x.x, x.y), a2), x23 = fmul2(make_float2(x.z, x.w), a2);
        x = make_float4(x01.x, x01.y, x23.x, x23.y);
        pa01 = ffma2(k2, x01, pa01);
        pa23 = ffma2(k2, x23, pa23);
        pb01 = ffma2(q2, x01, pb01);
        pb23 = ffma2(q2, x23, pb23);
      }
    }
    const float4 pa = make_float4(pa01.x, pa01.y, pa23.x, pa23.y), pb = make_float4(pb01.x, pb01.y, pb23.x, pb23.y);
    part_a[rg][cg] = pa;
    part_b[rg][cg] = pb;
    __syncthreads();

    if (tid < DV) {
      const int c4 = tid >> 2, e = tid & 3;
      float a = 0.f, b = 0.f;
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        a += reinterpret_cast<const float*>(&part_a[gi][c4])[e];
        b += reinterpret_cast<const float*>(&part_b[gi][c4])[e];
      }
      float vv;
      if constexpr (NST > 1) vv = to_f32(sv_raw[u][tid]);
      else vv = sv[0][tid];
      const float d = b_r * (vv - a);
      sdelta[tid] = d;
      so[u][tid] = fmaf(NST == 1 ? s_kq : s_kq_st[u], d, b);
    }
    __syncthreads();

    const float4 d4 = reinterpret_cast<const float4*>(sdelta)[cg];
    const float2 d01 = make_float2(d4.x, d4.y), d23 = make_float2(d4.z, d4.w);
#pragma unroll
    for (int i4 = 0; i4 < RPG; i4 += 4) {
      const float4 k4 = *reinterpret_cast<const float4*>(&sk[u][rg * RPG + i4]);
      const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float4& x = s[i4 + e];
        const float2 k2 = make_float2(kk[e], kk[e]);
        const float2 x01 = ffma2(k2, d01, make_float2(x.x, x.y)), x23 = ffma2(k2, d23, make_float2(x.z, x.w));
        x = make_float4(x01.x, x01.y, x23.x, x23.y);
      }
    }

    // Read-out (+ optional RMSNorm over dv and sigmoid gate).
    if constexpr (NST == 1) {
      float o = 0.f;
      if (tid < DV) o = so[0][tid];
      if (gate != nullptr) {
        float sq_sum = (tid < DV) ? o * o : 0.f;
        sq_sum = warp_sum(sq_sum);
        if ((tid & 31) == 0) red[tid >> 5] = sq_sum;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < (DV + 31) / 32; ++w) tot += red[w];
        if (tid < DV) {
          const float inv = rsqrtf(tot / (float)DV + eps);
          const float wj = norm_w ? norm_w[tid] : 1.f;
          o = o * inv * wj * sigmoidf_(to_f32(gate[rv + tid]));
        }
      }
      if (tid < DV) out[rv + tid] = from_f32<Tout>(o);
    } else if (u == NST - 1 || t + 1 == count) {
      // the stage's read-outs together, one warp per token: no barrier per token for the norm
      __syncthreads();
      const int w = tid >> 5, lane = tid & 31;
      if (w <= u) {
        float ov[DV / 32], ss = 0.f;
#pragma unroll
        for (int j = 0; j < DV / 32; ++j) {
          ov[j] = so[w][lane + 32 * j];
          ss = fmaf(ov[j], ov[j], ss);
        }
        const float inv = gate != nullptr ? rsqrtf(warp_sum(ss) / (float)DV + eps) : 1.f;
        const size_t rw = (((size_t)n * n_tok + (t - u + w)) * H + h) * DV;
#pragma unroll
        for (int j = 0; j < DV / 32; ++j) {
          const int c = lane + 32 * j;
          float o = ov[j];
          if (gate != nullptr) o = o * inv * (norm_w ? norm_w[c] : 1.f) * sigmoidf_(to_f32(sg_raw[w][c]));
          out[rw + c] = from_f32<Tout>(o);
        }
      }
    }
    // no barrier between tokens: what a token writes to shared memory before its first barrier was
    // last read before the previous token's second barrier (and red, written after the second,
    // was last read before this point)
  }

  if (commit) {
#pragma unroll
    for (int i = 0; i < RPG; ++i)
      __stcs(reinterpret_cast<float4*>(S + (size_t)(rg * RPG + i) * DV) + cg, s[i]);
  }
}

template <int DK, int DV, typename Tin, typename Tout>
cudaError_t launch_typed(const DecodeArgs& a, cudaStream_t st) {
  const int rows = a.N * a.H;
  if (rows == 0) return cudaSuccess;
  TraceScope ts("kda_decode", st);
  auto kern = a.n_tok == 1 ? decode_kernel<DK, DV, 1, Tin, Tout> : decode_kernel<DK, DV, kStageTok, Tin, Tout>;
  kern<<<rows, kDecodeThreads, 0, st>>>(
      static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v), a.g,
      a.beta, a.state_pool, a.slot_idx, static_cast<Tout*>(a.out), a.H, a.num_slots, a.n_tok, a.ntok_per_req,
      a.commit ? 1 : 0, static_cast<const Tin*>(a.epi.gate), a.epi.norm_weight, a.epi.eps, a.err);
  return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t launch_dims(const DecodeArgs& a, cudaStream_t st) {
  if (a.dk == 128 && a.dv == 128) return launch_typed<128, 128, Tin, Tout>(a, st);
  if (a.dk == 64 && a.dv == 64) return launch_typed<64, 64, Tin, Tout>(a, st);
  if (a.dk == 128 && a.dv == 64) return launch_typed<128, 64, Tin, Tout>(a, st);
  if (a.dk == 64 && a.dv == 128) return launch_typed<64, 128, Tin, Tout>(a, st);
  return cudaErrorInvalidValue;
}

template <typename Tin>
cudaError_t launch_out(const DecodeArgs& a, cudaStream_t st) {
  return a.out_bf16 ? launch_dims<Tin, __nv_bfloat16>(a, st) : launch_dims<Tin, float>(a, st);
}

}  // namespace

cudaError_t decode_launch(const DecodeArgs& a, cudaStream_t st) {
  return a.bf16 ? launch_out<__nv_bfloat16>(a, st) : launch_out<float>(a, st);
}

}  // namespace kda
