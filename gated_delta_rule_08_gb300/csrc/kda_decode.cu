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
// carry several tokens, applied in groups of up to four in the chunk form (decode_group_kernel
// below) to the state held in registers; the state is written back only when asked (commit),
// after exactly the request's own token count.  Verify = all draft tokens, no write-back;
// accept = the accepted prefix recomputed from the cached inputs, with write-back.  One token
// with write-back is the plain decode step.
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
constexpr int kStageTok = 4;  // tokens per group of the multi-token kernel

// One token per request (the decode step, and multi-token calls with n_tok = 1).
template <int DK, int DV, typename Tin, typename Tout>
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

  // Issue the state loads first: they are the longest-latency traffic.
  float4 s[RPG];
#pragma unroll
  for (int i = 0; i < RPG; ++i)
    s[i] = __ldcs(reinterpret_cast<const float4*>(S + (size_t)(rg * RPG + i) * DV) + cg);

  __shared__ __align__(16) float sk[DK], sq[DK], salpha[DK], sv[DV];
  __shared__ float4 part_a[NG][TPR], part_b[NG][TPR];
  __shared__ float sdelta[DV], so[DV];
  __shared__ float red[kDecodeThreads / 32];
  __shared__ float s_kq;

  for (int t = 0; t < count; ++t) {
    const size_t row = ((size_t)n * n_tok + t) * H + h;  // token row of [N, n_tok, H]
    const size_t rv = row * DV;
    const size_t rk = row * DK;
    for (int i = tid; i < DK; i += kDecodeThreads) {
      sk[i] = to_f32(k[rk + i]);
      sq[i] = to_f32(q[rk + i]);
      salpha[i] = __expf(g[rk + i]);
    }
    for (int j = tid; j < DV; j += kDecodeThreads) sv[j] = to_f32(v[rv + j]);
    const float b_r = beta[row];
    __syncthreads();

    if (tid < 32) {  // k . q
      float acc = 0.f;
      for (int i = tid; i < DK; i += 32) acc = fmaf(sk[i], sq[i], acc);
      acc = warp_sum(acc);
      if (tid == 0) s_kq = acc;
    }

    float2 pa01 = make_float2(0.f, 0.f), pa23 = pa01, pb01 = pa01, pb23 = pa01;
#pragma unroll
    for (int i4 = 0; i4 < RPG; i4 += 4) {  // this thread's rows rg RPG + i: four per 16-byte load
      const float4 al4 = *reinterpret_cast<const float4*>(&salpha[rg * RPG + i4]);
      const float4 k4 = *reinterpret_cast<const float4*>(&sk[rg * RPG + i4]);
      const float4 q4 = *reinterpret_cast<const float4*>(&sq[rg * RPG + i4]);
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
    part_a[rg][cg] = make_float4(pa01.x, pa01.y, pa23.x, pa23.y);
    part_b[rg][cg] = make_float4(pb01.x, pb01.y, pb23.x, pb23.y);
    __syncthreads();

    if (tid < DV) {
      const int c4 = tid >> 2, e = tid & 3;
      float a = 0.f, b = 0.f;
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        a += reinterpret_cast<const float*>(&part_a[gi][c4])[e];
        b += reinterpret_cast<const float*>(&part_b[gi][c4])[e];
      }
      const float d = b_r * (sv[tid] - a);
      sdelta[tid] = d;
      so[tid] = fmaf(s_kq, d, b);
    }
    __syncthreads();

    const float4 d4 = reinterpret_cast<const float4*>(sdelta)[cg];
    const float2 d01 = make_float2(d4.x, d4.y), d23 = make_float2(d4.z, d4.w);
#pragma unroll
    for (int i4 = 0; i4 < RPG; i4 += 4) {
      const float4 k4 = *reinterpret_cast<const float4*>(&sk[rg * RPG + i4]);
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
    float o = 0.f;
    if (tid < DV) o = so[tid];
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
  }

  if (commit) {
#pragma unroll
    for (int i = 0; i < RPG; ++i)
      __stcs(reinterpret_cast<float4*>(S + (size_t)(rg * RPG + i) * DV) + cg, s[i]);
  }
}

// Several tokens per request (verify / accept) in groups of up to kStageTok tokens, each group in
// the chunk form of section 2.5 / Eq. 4 restated for m tokens, with the group's initial state S
// and per-channel cumulative log-decays G_t = sum_{s <= t} g_s inside the group:
//   a_t = S^T (k_t e^{G_t}),  b_t = S^T (q_t e^{G_t})           (one pass over S for all 2 m vectors)
//   delta_t = beta_t (v_t - a_t) - sum_{s < t} A_ts delta_s,    A_ts = beta_t sum_c k_tc k_sc e^{G_tc - G_sc}
//   o_t = b_t + sum_{s <= t} M_ts delta_s,                      M_ts = sum_c q_tc k_sc e^{G_tc - G_sc}
//   S_new = Diag(e^{G_{m-1}}) S + sum_s (k_s e^{G_{m-1} - G_s}) delta_s^T
// which is the token recurrence (delta_t is the token's beta (v - S'^T k)) with every state-sized
// product fused into one reduction and one rank-m update (the update only when the state is kept
// or written back).  g > -5 keeps e^{-G_s} below e^{20} over a group, so k_s e^{-G_s} stays in fp32
// range; every factor applied to the state is at most 1.
template <int DK, int DV, typename Tin, typename Tout>
__global__ void __launch_bounds__(kDecodeThreads, 2)
decode_group_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                    const float* __restrict__ g, const float* __restrict__ beta, float* __restrict__ pool,
                    const int32_t* __restrict__ slot_idx, Tout* __restrict__ out, int H, int num_slots, int n_tok,
                    const int32_t* __restrict__ ntok_per_req, int commit, const Tin* __restrict__ gate,
                    const float* __restrict__ norm_w, float eps, unsigned int* __restrict__ err, int pf_lead) {
  constexpr int NST = kStageTok;
  constexpr int TPR = DV / 4;               // threads per state row
  constexpr int NG = kDecodeThreads / TPR;  // row groups
  constexpr int RPG = DK / NG;              // rows per thread
  static_assert(DK % NG == 0 && (DK / NG) % 4 == 0, "rows must split evenly, four per thread at least");
  static_assert(2 * NST * TPR <= kDecodeThreads, "one thread per (vector, column group) in the combine");

  const int nh = blockIdx.x;  // n * H + h
  const int n = nh / H, h = nh - (nh / H) * H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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

  // a group's inputs: k, q and g as raw values in registers (converted when stored to shared
  // memory); v and the gate straight into shared memory by cp.async.  The first group's are
  // issued before the state, so that they land first.
  constexpr int NLK = (NST * DK + kDecodeThreads - 1) / kDecodeThreads;
  constexpr int VPT = 16 / (int)sizeof(Tin);
  __shared__ __align__(16) Tin sv_raw[NST][DV], sg_raw[NST][DV];
  Tin rk[NLK], rq[NLK];
  float rg_[NLK], rb = 0.f;
  auto load_group = [&](int t0) {
    const int m = count - t0 < NST ? count - t0 : NST;
    const size_t row0 = ((size_t)n * n_tok + t0) * H + h;
#pragma unroll
    for (int j = 0; j < NLK; ++j) {
      const int i = tid + j * kDecodeThreads;
      if (i < m * DK) {
        const int w = i / DK, c = i - w * DK;
        const size_t rkk = (row0 + (size_t)w * H) * DK + c;
        rk[j] = k[rkk];
        rq[j] = q[rkk];
        rg_[j] = g[rkk];
      }
    }
    if (tid < m * DV / VPT) {
      const int w = tid / (DV / VPT), c = (tid % (DV / VPT)) * VPT;
      const size_t rw = (row0 + (size_t)w * H) * DV + c;
      cp_async16(&sv_raw[w][c], v + rw);
      if (gate != nullptr) cp_async16(&sg_raw[w][c], gate + rw);
    }
    cp_async_commit();
    rb = tid < m ? beta[row0 + (size_t)tid * H] : 0.f;
  };
  load_group(0);

  float4 s[RPG];
#pragma unroll
  for (int i = 0; i < RPG; ++i)
    s[i] = __ldcs(reinterpret_cast<const float4*>(S + (size_t)(rg * RPG + i) * DV) + cg);

  // Warm L2 with the state and inputs of the CTA that will take this one's place (pf_lead = the
  // number of CTAs resident at once), so that HBM keeps streaming while the resident CTAs compute:
  // the state by four bulk prefetches (the pool is 16-byte aligned), each input row line by line.
  if (pf_lead > 0 && nh + pf_lead < (int)gridDim.x) {
    const int nh2 = nh + pf_lead;
    const int n2 = nh2 / H, h2 = nh2 - (nh2 / H) * H;
    if (tid >= kDecodeThreads - 4) {
      const int slot2 = slot_idx[n2];
      if (slot2 >= 0 && slot2 < num_slots)
        prefetch_l2(pool + ((size_t)slot2 * H + h2) * (size_t)(DK * DV) + (tid - (kDecodeThreads - 4)) * (DK * DV / 4),
                    DK * DV);
    }
    for (int i = tid; i < 5 * n_tok; i += kDecodeThreads) {
      const int t = i / 5, a = i - 5 * t;
      const size_t r2 = ((size_t)n2 * n_tok + t) * H + h2;
      const char* p = nullptr;
      int bytes = 0;
      if (a == 0) {
        p = reinterpret_cast<const char*>(k + r2 * DK), bytes = DK * (int)sizeof(Tin);
      } else if (a == 1) {
        p = reinterpret_cast<const char*>(q + r2 * DK), bytes = DK * (int)sizeof(Tin);
      } else if (a == 2) {
        p = reinterpret_cast<const char*>(g + r2 * DK), bytes = DK * 4;
      } else if (a == 3) {
        p = reinterpret_cast<const char*>(v + r2 * DV), bytes = DV * (int)sizeof(Tin);
      } else if (gate != nullptr) {
        p = reinterpret_cast<const char*>(gate + r2 * DV), bytes = DV * (int)sizeof(Tin);
      }
      for (int o = 0; o < bytes; o += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(p + o));
    }
  }

  extern __shared__ float4 dsm4[];
  float4* part = dsm4;  // [2 NST][NG][TPR]: per-row-group partial reductions (a_t, then b_t)
  __shared__ __align__(16) float sgv[NST][DK], skv[NST][DK], sqv[NST][DK];
  __shared__ __align__(16) float khat[NST][DK], qhat[NST][DK], ktil[NST][DK], kbar[NST][DK], gam_last[DK];
  __shared__ __align__(16) float red_a[NST][DV], red_b[NST][DV], sdelta[NST][DV], so[NST][DV];
  __shared__ float sbeta[NST], sA[NST][NST], sM[NST][NST];

  for (int t0 = 0; t0 < count; t0 += NST) {
    const int m = count - t0 < NST ? count - t0 : NST;
    const size_t row0 = ((size_t)n * n_tok + t0) * H + h;  // token row of [N, n_tok, H]
    if (t0 > 0) {
      __syncthreads();  // the previous group's shared arrays are no longer read
      load_group(t0);
    }
#pragma unroll
    for (int j = 0; j < NLK; ++j) {
      const int i = tid + j * kDecodeThreads;
      if (i < m * DK) {
        const int w = i / DK, c = i - w * DK;
        skv[w][c] = to_f32(rk[j]);
        sqv[w][c] = to_f32(rq[j]);
        sgv[w][c] = rg_[j];
      }
    }
    if (tid < m) sbeta[tid] = rb;
    cp_async_wait_all();  // this thread's v and gate pieces
    __syncthreads();
    // per channel: the group's cumulative decays and the four scaled key / query forms
    for (int c = tid; c < DK; c += kDecodeThreads) {
      float G[NST];
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < NST; ++w) {
        if (w < m) acc += sgv[w][c];
        G[w] = acc;
      }
#pragma unroll
      for (int w = 0; w < NST; ++w) {
        if (w >= m) break;
        const float kk = skv[w][c], qq = sqv[w][c], e = __expf(G[w]);
        khat[w][c] = kk * e;
        qhat[w][c] = qq * e;
        ktil[w][c] = kk * __expf(-G[w]);
        kbar[w][c] = kk * __expf(G[m - 1] - G[w]);
      }
      gam_last[c] = __expf(G[m - 1]);
    }
    __syncthreads();

    // the small matrices M_ts (s <= t) and A_ts (s < t), one dot product over dk per warp
    for (int d = warp; d < NST * NST; d += kDecodeThreads / 32) {
      const int t = d / NST, s2 = d % NST;
      if (t < m && s2 <= t) {
        float am = 0.f, aa = 0.f;
        for (int c = lane; c < DK; c += 32) {
          const float kt = ktil[s2][c];
          am = fmaf(qhat[t][c], kt, am);
          aa = fmaf(khat[t][c], kt, aa);
        }
        am = warp_sum(am);
        aa = warp_sum(aa);
        if (lane == 0) {
          sM[t][s2] = am;
          sA[t][s2] = s2 < t ? sbeta[t] * aa : 0.f;
        }
      }
    }
    // a_t and b_t over this thread's rows: every state element read once for all 2 m vectors
    {
      float2 pa01[NST], pa23[NST], pb01[NST], pb23[NST];
#pragma unroll
      for (int w = 0; w < NST; ++w) pa01[w] = pa23[w] = pb01[w] = pb23[w] = make_float2(0.f, 0.f);
#pragma unroll
      for (int i4 = 0; i4 < RPG; i4 += 4) {
#pragma unroll
        for (int w = 0; w < NST; ++w) {
          if (w >= m) break;
          const float4 k4 = *reinterpret_cast<const float4*>(&khat[w][rg * RPG + i4]);
          const float4 q4 = *reinterpret_cast<const float4*>(&qhat[w][rg * RPG + i4]);
          const float kk[4] = {k4.x, k4.y, k4.z, k4.w}, qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4& x = s[i4 + e];
            const float2 x01 = make_float2(x.x, x.y), x23 = make_float2(x.z, x.w);
            const float2 k2 = make_float2(kk[e], kk[e]), q2 = make_float2(qq[e], qq[e]);
            pa01[w] = ffma2(k2, x01, pa01[w]);
            pa23[w] = ffma2(k2, x23, pa23[w]);
            pb01[w] = ffma2(q2, x01, pb01[w]);
            pb23[w] = ffma2(q2, x23, pb23[w]);
          }
        }
      }
#pragma unroll
      for (int w = 0; w < NST; ++w) {
        if (w >= m) break;
        part[((size_t)w * NG + rg) * TPR + cg] = make_float4(pa01[w].x, pa01[w].y, pa23[w].x, pa23[w].y);
        part[((size_t)(NST + w) * NG + rg) * TPR + cg] = make_float4(pb01[w].x, pb01[w].y, pb23[w].x, pb23[w].y);
      }
    }
    __syncthreads();
    // sum over the row groups: one thread per (vector, column group)
    if (tid < 2 * NST * TPR) {
      const int j = tid / TPR, c4 = tid % TPR, w = j % NST;
      if (w < m) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
          const float4 x = part[((size_t)j * NG + gi) * TPR + c4];
          acc.x += x.x;
          acc.y += x.y;
          acc.z += x.z;
          acc.w += x.w;
        }
        *reinterpret_cast<float4*>(j < NST ? &red_a[w][4 * c4] : &red_b[w][4 * c4]) = acc;
      }
    }
    __syncthreads();
    // per value column: forward substitution for delta, then the read-outs
    for (int c = tid; c < DV; c += kDecodeThreads) {
      float dl[NST];
#pragma unroll
      for (int t = 0; t < NST; ++t) {
        if (t >= m) break;
        float d = sbeta[t] * (to_f32(sv_raw[t][c]) - red_a[t][c]);
#pragma unroll
        for (int s2 = 0; s2 < t; ++s2) d = fmaf(-sA[t][s2], dl[s2], d);
        dl[t] = d;
        sdelta[t][c] = d;
        float o = red_b[t][c];
#pragma unroll
        for (int s2 = 0; s2 <= t; ++s2) o = fmaf(sM[t][s2], dl[s2], o);
        so[t][c] = o;
      }
    }
    __syncthreads();
    // the state after the group (kept for the next group, written back on commit)
    if (t0 + m < count || commit) {
#pragma unroll
      for (int i4 = 0; i4 < RPG; i4 += 4) {
        const float4 gl = *reinterpret_cast<const float4*>(&gam_last[rg * RPG + i4]);
        const float gle[4] = {gl.x, gl.y, gl.z, gl.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float4& x = s[i4 + e];
          const float2 g2 = make_float2(gle[e], gle[e]);
          float2 x01 = fmul2(make_float2(x.x, x.y), g2), x23 = fmul2(make_float2(x.z, x.w), g2);
#pragma unroll
          for (int w = 0; w < NST; ++w) {
            if (w >= m) break;
            const float4 d4 = reinterpret_cast<const float4*>(sdelta[w])[cg];
            const float kb = kbar[w][rg * RPG + i4 + e];
            const float2 kb2 = make_float2(kb, kb);
            x01 = ffma2(kb2, make_float2(d4.x, d4.y), x01);
            x23 = ffma2(kb2, make_float2(d4.z, d4.w), x23);
          }
          x = make_float4(x01.x, x01.y, x23.x, x23.y);
        }
      }
    }
    // the group's read-outs, one warp per token (+ optional RMSNorm over dv and sigmoid gate)
    if (warp < m) {
      float ov[DV / 32], ss = 0.f;
#pragma unroll
      for (int j = 0; j < DV / 32; ++j) {
        ov[j] = so[warp][lane + 32 * j];
        ss = fmaf(ov[j], ov[j], ss);
      }
      const float inv = gate != nullptr ? rsqrtf(warp_sum(ss) / (float)DV + eps) : 1.f;
      const size_t rw = (row0 + (size_t)warp * H) * DV;
#pragma unroll
      for (int j = 0; j < DV / 32; ++j) {
        const int c = lane + 32 * j;
        float o = ov[j];
        if (gate != nullptr) o = o * inv * (norm_w ? norm_w[c] : 1.f) * sigmoidf_(to_f32(sg_raw[warp][c]));
        out[rw + c] = from_f32<Tout>(o);
      }
    }
  }

  if (commit) {
#pragma unroll
    for (int i = 0; i < RPG; ++i)
      __stcs(reinterpret_cast<float4*>(S + (size_t)(rg * RPG + i) * DV) + cg, s[i]);
  }
}

template <int DK, int DV>
constexpr size_t group_smem() {
  return (size_t)2 * kStageTok * (kDecodeThreads / (DV / 4)) * (DV / 4) * sizeof(float4);
}

template <int DK, int DV, typename Tin, typename Tout>
cudaError_t launch_typed(const DecodeArgs& a, cudaStream_t st) {
  const int rows = a.N * a.H;
  if (rows == 0) return cudaSuccess;
  TraceScope ts("kda_decode", st);
  if (a.n_tok > 1) {  // several tokens per request: the grouped chunk form
    static DeviceOnce once;
    static int lead[kMaxDevices];  // CTAs resident at once, written under the once-lock
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const cudaError_t e = once.run(dev, [dev] {
      auto kern = decode_group_kernel<DK, DV, Tin, Tout>;
      cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)group_smem<DK, DV>());
      int per_sm = 0, sms = 0;
      if (r == cudaSuccess)
        r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecodeThreads, group_smem<DK, DV>());
      if (r == cudaSuccess) r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (r == cudaSuccess) lead[dev] = per_sm * sms;
      return r;
    });
    if (e != cudaSuccess) return e;
    decode_group_kernel<DK, DV, Tin, Tout><<<rows, kDecodeThreads, group_smem<DK, DV>(), st>>>(
        static_cast<const Tin*>(a.q), static_cast<const Tin*>(a.k), static_cast<const Tin*>(a.v), a.g, a.beta,
        a.state_pool, a.slot_idx, static_cast<Tout*>(a.out), a.H, a.num_slots, a.n_tok, a.ntok_per_req,
        a.commit ? 1 : 0, static_cast<const Tin*>(a.epi.gate), a.epi.norm_weight, a.epi.eps, a.err, lead[dev]);
    return cudaGetLastError();
  }
  auto kern = decode_kernel<DK, DV, Tin, Tout>;
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
