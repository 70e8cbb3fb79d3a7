// KDA prefill: the serial inter-chunk state pass on the tcgen05 tensor cores, and the
// intra-device context parallelism that splits it into sequence segments.
//
// Kimi K3: Open Frontier Intelligence (kimi-k3-paper.pages.dev), section 2.5 / Eq. 4: per
// chunk, with chunk-start state S0 and the chunk record (W, U_hat, Q_hat, K_bar, M, e^{G_C}):
//   U = U_hat - W S0,  O = Q_hat S0 + M U,  S_C = Diag(e^{G_C}) S0 + K_bar^T U.
// Section 13.3.1 (intra-device CP): the SMs of one device each take a segment of a sequence,
// evaluate the segment's transition independently, then merge to recover every segment's
// initial state.  A chunk maps S0 affinely, S_C = (Diag(e^{G_C}) - K_bar^T W) S0 + K_bar^T U_hat,
// so a segment of chunks maps S_in to S_out = P S_in + b with
//   b = the segment's final state from S_in = 0,
//   P = the segment's final state from S_in = I with U_hat = 0 (a dk x dk state);
// both are ordinary runs of the same state pass.  The first segment's input is known (h0), so it
// needs neither: one run from h0 gives S_in(1) itself.  The merge then walks the remaining
// segments, S_in(p+1) = P_p S_in(p) + b_p for p >= 1, and a last pass re-runs every segment from
// its S_in with outputs.
//
//  kda_tc_chunk_scan<Tout, MODE> (grid = sequences x heads x segments, 16 warps):
//    the state^T (dv x dk, fp32) lives in TMEM for the whole segment, next to an fp16 copy that
//    is the A operand (read from TMEM) of the first fused product
//      [D_U | D_O] = S^T [W^T | Q_hat^T]                      (8 MMAs, N = 128)
//    and U^T (fp16, also in TMEM) is the A operand of the second
//      [D_O | S^T] += U^T [M ; K_bar^T]^T                     (4 MMAs, N = 192),
//    with S^T already scaled by Diag(e^{G_C}) in place.
//    warp 12 (one lane) stages the records with bulk copies and issues every MMA;
//    warps 0-7 (two per TMEM lane quadrant, each owning half of the columns) convert
//      D_U -> U^T and the updated state -> its fp16 copy, and apply the decay;
//    MODE 0 (read-out): warps 8-11 drain D_O off the serial path: a full chunk without the
//      epilogue straight from registers (each store writes 32 consecutive dv of a token), else
//      through a staging buffer with the optional RMSNorm + gate epilogue, whose rows warps
//      13-15 share with them (seven warps on a chunk's 64 rows);
//    MODE 1 (transition): z = 0 runs segment 0 from h0 (its final state is S_in(1)); for p >= 1,
//      z = 2 p - 1 + kind, kind 0 runs b_p and kind 1 runs P_p; no read-out.
//    segment map (context parallelism across devices, section 13.3.2): MODE 1 over one token range
//      with z = 2 p + kind for every segment p, both runs starting from 0 (kind 0, with U_hat) or I
//      (kind 1, U_hat = 0); with one segment the runs' final states are the range's b and P.
//  kda_cp_merge (grid = sequences x heads x 4 column slices): the sequential segment merge in fp32.
//
//  Non-finite results: an fp16 operand past 65504 (a value, an intra-chunk term or the state copy)
//  becomes inf and reaches the state (through U = U_hat - W S and S += K_bar^T U) as well as the
//  outputs, so the state warps test every run's final state (written or not) and the checkpoints
//  they write (a sum is finite exactly when its terms are) and set KDA_DEVERR_NONFINITE; nothing on
//  the serial path or in the output warps is checked.
#include <cuda_bf16.h>

#include <type_traits>

#include "kda_internal.h"
#include "kda_tc_common.cuh"

namespace kda {
namespace {

using namespace tcx;

// sigmoid(x) = (1 + tanh(x / 2)) / 2 with the hardware tanh approximation (relative error about
// 2^-11): one special-function operation instead of an exponential and a reciprocal
__device__ __forceinline__ float sigmoid_tanh(float x) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * x));
  return fmaf(0.5f, t, 0.5f);
}

constexpr int kScanThreads = 512;
constexpr int kEpiWarps = 7;                     // warps 8-11 and 13-15 (with the epilogue)
constexpr int kStateThreads = 256;               // warps 0-7
constexpr int kIssuerWarp = 12;
constexpr int kStages = 3;                       // records staged up to two chunks ahead
constexpr uint32_t kStage = 59392;               // staged record bytes, 1024-aligned
constexpr uint32_t S_OUT = kStages * kStage;     // fp32 read-out staging [64 r][128 dv]
constexpr uint32_t S_GATE = S_OUT + 32768;       // gate logits of a chunk: [64 rows][32 lanes] x 8 B
constexpr uint32_t S_BAR = S_GATE + 16384;       // barriers + tmem slot + abort flag
constexpr uint32_t S_END = S_BAR + 128;
constexpr uint32_t kScanSmem = S_END + 1024;

constexpr uint32_t T_DU = 0;     // TMEM: D_U [128 x 64]
constexpr uint32_t T_DO = 64;    // D_O [128 x 64]   (directly after D_U and directly before S)
constexpr uint32_t T_S = 128;    // state^T fp32 [128 x 128]
constexpr uint32_t T_S16 = 256;  // state^T fp16 pairs [128 x 64 columns]
constexpr uint32_t T_U16 = 320;  // U^T fp16 pairs [128 x 32 columns]

constexpr size_t kCpMat = 128 * 128;  // floats per CP matrix

struct ScanParams {
  const uint8_t* records;
  const int32_t* plan;
  const int32_t* cu;
  int B;
  int64_t T;
  int H;
  const float* h0;
  float* hT;
  void* out;
  const __nv_bfloat16* gate;
  const float* norm_w;
  float eps;
  unsigned int* err;
  int nseg;
  int64_t seg_len;  // chunks per segment
  float* cp;        // [B][H][nseg][3][128][128]: P_p, b_p, S_in(p)
  float* ckpt;      // state checkpoints [n][H][128][128] fp32, or null (read-out pass only)
  int64_t ckpt_chunks;
  float* seg_P;         // segment map: the range's transition [H][128][128] (MODE 1), or null
  float* seg_b;         // segment map: the range's offset [H][128][128] (MODE 1)
};

// 8 bytes global -> shared without registers (completion: cp_async_wait_all by the same thread)
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// four consecutive outputs (16-byte fp32 or 8-byte bf16 store)
__device__ __forceinline__ void store_row(float* dst, const float4& y) { *reinterpret_cast<float4*>(dst) = y; }
__device__ __forceinline__ void store_row(__nv_bfloat16* dst, const float4& y) {
  __nv_bfloat162 a = __floats2bfloat162_rn(y.x, y.y), b = __floats2bfloat162_rn(y.z, y.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&a);
  pk.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(dst) = pk;
}

__device__ __forceinline__ void tmem_ld64b(uint32_t taddr, float* v) {
  float a[32], b[32];
  tmem_ld32(taddr, a);
  tmem_ld32(taddr + 32, b);
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = a[i];
    v[32 + i] = b[i];
  }
}
// 64 fp32 columns -> TMEM (as raw bits)
__device__ __forceinline__ void tmem_st64f(uint32_t taddr, const float* v) {
  uint32_t a[32], b[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    a[i] = __float_as_uint(v[i]);
    b[i] = __float_as_uint(v[32 + i]);
  }
  tmem_st32u(taddr, a);
  tmem_st32u(taddr + 32, b);
}
// 64 fp32 values -> 32 fp16 pairs -> TMEM
__device__ __forceinline__ void tmem_st64h(uint32_t taddr, const float* v) {
  uint32_t a[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) a[i] = pack_h2(v[2 * i], v[2 * i + 1]);
  tmem_st32u(taddr, a);
}

template <typename Tout, int MODE, bool CKPT, bool GIVEUP = false>
__global__ void __launch_bounds__(kScanThreads, 1) kda_tc_chunk_scan(const ScanParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + S_BAR);  // [3] record staged (bulk copy)
  uint64_t* bar_u = full + 3;                                // [D_U | D_O] product done
  uint64_t* bar_s = full + 4;                                // [D_O | S] product done
  uint64_t* s16_ready = full + 5;                            // fp16 state copy written (256 arrivals)
  uint64_t* u16_ready = full + 6;                            // U^T written, decay applied (256 arrivals)
  uint64_t* do_free = full + 7;                              // D_O read by the output warps
  uint64_t* bar_fin = full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S_BAR + 80);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + S_BAR + 84);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H;
  griddep_launch_dependents();
  // A CTA that has nothing to do still waits for the predecessor grid before it exits, so that
  // no grid of the chain completes before the one it follows (a successor's griddep_wait covers
  // only its immediate predecessor).
  if (p.cu != nullptr && p.plan[p.B + 1] == 0) {  // invalid cu_seqlens: sequence skipped
    griddep_wait();
    return;
  }
  // blockIdx.x = rank x H + head: all heads of the longest sequence are dispatched first
  const int h = (int)(blockIdx.x % (unsigned)H);
  const int b = sequence_of_rank((int)(blockIdx.x / (unsigned)H), p.plan, p.cu, p.B);
  int64_t first_chunk, t_begin, len;
  const int64_t nchunks = sequence_chunks(b, p.plan, p.cu, p.B, p.T, first_chunk, t_begin, len);
  const int64_t p_last = nchunks > 0 ? (nchunks - 1) / p.seg_len : 0;
  // MODE 1: kind 0 = offset b (from h0 for segment 0), 1 = transition P; a segment map runs both
  // kinds for every segment, from 0 and from I
  const bool segmap = MODE == 1 && p.seg_P != nullptr;
  const uint32_t z = blockIdx.z;
  const int seg = segmap ? (int)(z >> 1) : (MODE == 0 || z == 0 ? (int)z : (int)((z + 1) >> 1));
  const int kind = segmap ? (int)(z & 1) : (MODE == 0 || z == 0 ? 0 : (int)((z + 1) & 1));
  if ((MODE == 0 && seg > p_last) || (MODE == 1 && !segmap && seg >= p_last) || (segmap && seg > p_last)) {
    griddep_wait();
    return;
  }
  const int64_t c_begin = (int64_t)seg * p.seg_len;
  const int64_t c_end = nchunks < c_begin + p.seg_len ? nchunks : c_begin + p.seg_len;
  const int64_t ncs = c_end > c_begin ? c_end - c_begin : 0;
  float* cpb = p.cp + ((size_t)(b * H + h) * p.nseg + seg) * 3 * kCpMat;

  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int i = 0; i < kStages; ++i) mbar_init(&full[i], 1);
    mbar_init(bar_u, 1);
    mbar_init(bar_s, 1);
    mbar_init(s16_ready, kStateThreads);
    mbar_init(u16_ready, kStateThreads);
    mbar_init(do_free, 1);
    mbar_init(bar_fin, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // everything above overlaps the predecessor's tail; its records and segment states are read below
  griddep_wait();
  const uint32_t tl = tmem_lane(tmem, warp);
  const int row = (warp & 3) * 32 + lane;  // TMEM lane = state column (dv for S, dk for P)
  const size_t soff = ((size_t)b * H + h) * kCpMat;
  const uint8_t* rec0 = p.records + ((size_t)(first_chunk + c_begin) * H + h) * kRecBytes;
  const size_t rec_stride = (size_t)H * kRecBytes;

  if (warp == kIssuerWarp) {
    // ======================== issuer: record staging + all MMAs (one lane)
    if (lane == 0) {
      int64_t last_load = -1, consumed = -1;
      bool ok = true;
      // the read-out pass stages the whole operand part of a record; the transitions use only
      // W^T, K_bar^T and e^{G_C}
      auto stage_record = [&](int64_t c) {
        const int s2 = (int)(c % kStages);
        const uint8_t* src = rec0 + (size_t)c * rec_stride;
        uint8_t* dst = sm + s2 * kStage;
        if (MODE == 0) {
          mbar_arrive_expect_tx(&full[s2], kRecStage);
          bulk_g2s(dst, src, kRecStage, &full[s2]);
        } else {
          mbar_arrive_expect_tx(&full[s2], (kRecQT - kRecWT) + (kRecStage - kRecKT));
          bulk_g2s(dst + kRecWT, src + kRecWT, kRecQT - kRecWT, &full[s2]);
          bulk_g2s(dst + kRecKT, src + kRecKT, kRecStage - kRecKT, &full[s2]);
        }
        last_load = c;
      };
      for (int64_t c = 0; c < 2 && c < ncs; ++c) stage_record(c);
      const uint32_t id1 = MODE == 0 ? idesc_f16(128, 128, false, true) : idesc_f16(128, 64, false, true);
      const uint32_t id2 = MODE == 0 ? idesc_f16(128, 192, false, false) : idesc_f16(128, 128, false, false);
      for (int64_t c = 0; c < ncs && ok; ++c) {
        const int st = (int)(c % kStages);
        uint8_t* stage = sm + st * kStage;
        if (c + 2 < ncs) {
          // chunk c+2 goes where chunk c-1 was: free once that chunk's products are done
          if (c >= 1) ok = wait_or_abort_t<GIVEUP>(bar_s, (uint32_t)((c - 1) & 1), abort_flag);
          if (!ok) break;
          stage_record(c + 2);
        }
        ok = wait_or_abort_t<GIVEUP>(&full[st], (uint32_t)((c / kStages) & 1), abort_flag);
        if (ok) consumed = c;
        ok = ok && wait_or_abort_t<GIVEUP>(s16_ready, (uint32_t)(c & 1), abort_flag);
        if (MODE == 0 && ok && c >= 1) ok = wait_or_abort_t<GIVEUP>(do_free, (uint32_t)((c - 1) & 1), abort_flag);
        if (!ok) break;
        tc_fence_after();
        {
          const uint64_t db = smem_desc_sw128(smem_u32(stage + kRecWT), kRecQT - kRecWT, 1024);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_f16_ts(tmem + T_DU, tmem + T_S16 + 8 * ks, desc_add(db, ks * 2048), id1, ks > 0);
          mma_commit(bar_u);
        }
        ok = wait_or_abort_t<GIVEUP>(u16_ready, (uint32_t)(c & 1), abort_flag);
        if (!ok) break;
        tc_fence_after();
        {
          const uint64_t db = smem_desc_sw128(smem_u32(stage + (MODE == 0 ? kRecMM : kRecKT)), 16, 1024);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_f16_ts(tmem + (MODE == 0 ? T_DO : T_S), tmem + T_U16 + 8 * ks, desc_add(db, ks * 32), id2, true);
          mma_commit(bar_s);
        }
      }
      if (!ok || *abort_flag) {
        *abort_flag = 1;
        // let this thread's copies and MMAs drain (bounded) before TMEM is released
        for (int64_t l = consumed + 1; l <= last_load; ++l) mbar_wait(&full[l % kStages], (uint32_t)((l / kStages) & 1));
        mma_commit(bar_fin);
        mbar_wait(bar_fin, 0);
      }
    }
  } else if (warp < 8) {
    // ======================== state warps: TMEM lane quadrant warp & 3, column half hc
    const int hc = warp >> 2;
    // state checkpoints (CKPT): after every ckpt_chunks full chunks of the sequence
    const int64_t ck_base = CKPT ? checkpoint_base(b, p.cu, p.T, 64 * p.ckpt_chunks) : 0;
    int64_t ck_next = CKPT ? (c_begin / p.ckpt_chunks + 1) * p.ckpt_chunks : 0;  // next boundary (chunks done)
    bool ok = true;
    float fsum = 0.f;  // sum over this run's final state and its checkpoints (finite iff each entry is)
    {
      // segment 0 starts from h0 in both modes (a segment map's from 0); the read-out of a later
      // segment from S_in(seg)
      const bool from_state = MODE == 0 || (seg == 0 && !segmap);
      const float* init = nullptr;
      if (from_state) init = seg == 0 ? (p.h0 ? p.h0 + soff : nullptr) : cpb + 2 * kCpMat;
      float s[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const int col = 64 * hc + c;
        if (from_state) s[c] = init ? init[(size_t)col * 128 + row] : 0.f;
        else s[c] = (kind == 1 && col == row) ? 1.f : 0.f;
      }
      tmem_st64h(tl + T_S16 + 32 * hc, s);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(s16_ready);
      if (ncs > 0) {
        ok = wait_or_abort_t<GIVEUP>(&full[0], 0, abort_flag);
        if (ok) {
          const float* gc = reinterpret_cast<const float*>(sm + kRecGC) + 64 * hc;
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] *= gc[c];
        }
      }
      tmem_st64f(tl + T_S + 64 * hc, s);
      tmem_wait_st();
    }
    // this thread's half of the U_hat^T row (r = 32 hc .. 32 hc + 31), fetched one chunk ahead
    const bool use_uh = MODE == 0 || kind == 0;
    uint4 uh[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) uh[j] = make_uint4(0u, 0u, 0u, 0u);
    if (use_uh && ncs > 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j) uh[j] = *reinterpret_cast<const uint4*>(rec0 + kRecUT + row_chunk(row, 4 * hc + j));
    }
    for (int64_t c = 0; c < ncs && ok; ++c) {
      uint4 uh_next[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) uh_next[j] = make_uint4(0u, 0u, 0u, 0u);
      if (use_uh && c + 1 < ncs) {
        const uint8_t* ut = rec0 + (size_t)(c + 1) * rec_stride + kRecUT;
#pragma unroll
        for (int j = 0; j < 4; ++j) uh_next[j] = *reinterpret_cast<const uint4*>(ut + row_chunk(row, 4 * hc + j));
      }
      // U^T = U_hat^T - D_U on this thread's 32 columns
      ok = wait_or_abort_t<GIVEUP>(bar_u, (uint32_t)(c & 1), abort_flag);
      if (!ok) break;
      tc_fence_after();
      {
        float u[32];
        tmem_ld32(tl + T_DU + 32 * hc, u);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w4[4] = {uh[j].x, uh[j].y, uh[j].z, uh[j].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 a = unpack_h2(w4[e]);
            pk[4 * j + e] = pack_h2(a.x - u[8 * j + 2 * e], a.y - u[8 * j + 2 * e + 1]);
          }
        }
        tmem_st16u(tl + T_U16 + 16 * hc, pk);
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(u16_ready);
      // updated state -> fp16 copy (next chunk's A operand), then the next chunk's decay in place
      ok = wait_or_abort_t<GIVEUP>(bar_s, (uint32_t)(c & 1), abort_flag);
      if (!ok) break;
      tc_fence_after();
      bool ckpt_now = false;
      if constexpr (CKPT) {
        const int64_t cg1 = c_begin + c + 1;  // chunks of the sequence done
        if (cg1 == ck_next) {
          ckpt_now = cg1 * 64 <= len;  // full chunks only
          ck_next += p.ckpt_chunks;
        }
      }
      if (c + 1 < ncs || ckpt_now) {
        float s[64];
        tmem_ld64b(tl + T_S + 64 * hc, s);
        if (c + 1 < ncs) {
          tmem_st64h(tl + T_S16 + 32 * hc, s);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(s16_ready);
        }
        if (ckpt_now) {
          float* dst = p.ckpt + ((size_t)(ck_base + (ck_next - p.ckpt_chunks) / p.ckpt_chunks - 1) * H + h) * kCpMat;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            dst[(size_t)(64 * hc + j) * 128 + row] = s[j];
            fsum += s[j];
          }
        }
        if (c + 1 < ncs) {
          const int st1 = (int)((c + 1) % kStages);
          ok = wait_or_abort_t<GIVEUP>(&full[st1], (uint32_t)(((c + 1) / kStages) & 1), abort_flag);
          if (!ok) break;
          const float* gc = reinterpret_cast<const float*>(sm + st1 * kStage + kRecGC) + 64 * hc;
#pragma unroll
          for (int j = 0; j < 64; ++j) s[j] *= gc[j];
          tmem_st64f(tl + T_S + 64 * hc, s);
          tmem_wait_st();
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) uh[j] = uh_next[j];
    }
    // final state of this (sequence, head, segment)
    float* dst = nullptr;
    if (MODE == 0 && seg == p_last) dst = p.hT ? p.hT + soff : nullptr;
    if (MODE == 1) dst = seg == 0 ? cpb + (3 + 2) * kCpMat : cpb + (kind == 1 ? 0 : kCpMat);  // S_in(1), or P_p / b_p
    if (segmap) dst = p.nseg == 1 ? (kind == 1 ? p.seg_P : p.seg_b) + (size_t)h * kCpMat : cpb + (kind == 1 ? 0 : kCpMat);
    if (ok && !*abort_flag) {
      tc_fence_after();
      float s[64];
      tmem_ld64b(tl + T_S + 64 * hc, s);
#pragma unroll
      for (int c = 0; c < 64; ++c) fsum += s[c];
      if (dst != nullptr) {
#pragma unroll
        for (int c = 0; c < 64; ++c) dst[(size_t)(64 * hc + c) * 128 + row] = s[c];
      }
    }
    if (!ok) *abort_flag = 1;
    if (!isfinite(fsum)) atomicOr(p.err, KDA_DEVERR_NONFINITE);
  } else if (MODE == 0) {
    // ======================== output warps 8-11: D_O -> staging -> epilogue -> global; with the
    // epilogue, warps 13-15 join them on the staged rows (seven warps share a chunk's 64 rows)
    // (two specialisations: without the epilogue, and with it; the gate's global loads of the
    // latter are copied into shared memory while D_O is produced)
    float* ost = reinterpret_cast<float*>(sm + S_OUT);
    const bool tw = warp < kIssuerWarp;       // reads D_O from TMEM lane quadrant warp & 3
    const int ow = tw ? warp - 8 : warp - 9;  // 0-3 the TMEM warps, 4-6 the epilogue helpers
    Tout* out = static_cast<Tout*>(p.out);
    bool ok = true;
    auto readout = [&](auto epi_tag) {
      constexpr bool EPI = decltype(epi_tag)::value;
      if (!EPI && !tw) return;
      constexpr int kEw = kEpiWarps, kRows = (64 + kEpiWarps - 1) / kEpiWarps;
      uint2* sgate = reinterpret_cast<uint2*>(sm + S_GATE) + lane;  // [64 rows][32 lanes]
      float4 wv = make_float4(1.f, 1.f, 1.f, 1.f);  // RMSNorm weight of this lane's four dv
      if (EPI && p.norm_w != nullptr)
        wv = make_float4(p.norm_w[4 * lane], p.norm_w[4 * lane + 1], p.norm_w[4 * lane + 2], p.norm_w[4 * lane + 3]);
      for (int64_t c = 0; c < ncs; ++c) {
        const int64_t cg = c_begin + c;
        const int64_t rem = len - 64 * cg;
        const int n = (int)(rem < 64 ? rem : 64);
        const int64_t t0 = t_begin + 64 * cg;
        if constexpr (!EPI) {
          ok = group_and(2, 128, wait_or_abort_t<GIVEUP>(bar_s, (uint32_t)(c & 1), abort_flag));
          if (!ok) break;
          tc_fence_after();
          float o[64];
          tmem_ld64b(tl + T_DO, o);
          tc_fence_before();
          group_sync(2, 128);
          if (ow == 0 && lane == 0) mbar_arrive(do_free);
          if (n == 64 && sizeof(Tout) == 2) {
            // full chunk, plain bf16 output: each warp instruction writes 32 consecutive dv of a token
            __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(out) + (size_t)t0 * H * 128 + (size_t)h * 128 + row;
#pragma unroll
            for (int r = 0; r < 64; ++r) {
              ob[(size_t)r * H * 128] = __float2bfloat16_rn(o[r]);
              if ((r & 7) == 7) __nanosleep(64);  // spread the stores over the chunk period
            }
            continue;
          }
#pragma unroll
          for (int r = 0; r < 64; ++r) ost[r * 128 + row] = o[r];
          group_sync(2, 128);
          for (int r = ow; r < n; r += 4) {
            const float4 y = *reinterpret_cast<const float4*>(ost + r * 128 + 4 * lane);
            store_row(out + ((size_t)(t0 + r) * H + h) * 128 + 4 * lane, y);
          }
          group_sync(2, 128);  // staging buffer free for the next chunk
        } else {
          {
            // the gate logits of this warp's rows, each lane its own 8 bytes
            const __nv_bfloat16* gp = p.gate + ((size_t)(t0 + ow) * H + h) * 128 + 4 * lane;
            const size_t gstep = (size_t)kEw * H * 128;
#pragma unroll 1
            for (int r = ow, i = 0; r < n; r += kEw, ++i) cp_async8(sgate + r * 32, gp + i * gstep);
            cp_async_commit();
            // the next chunk's rows of this warp into L2, one 128-byte line per lane
            if (c + 1 < ncs) {
              const int64_t rem1 = len - 64 * (cg + 1);
              const int n1 = (int)(rem1 < 64 ? rem1 : 64);
              const int r1 = ow + kEw * (lane >> 1);
              if (r1 < n1)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(p.gate + ((size_t)(t0 + 64 + r1) * H + h) * 128 + 64 * (lane & 1)));
            }
          }
          if (tw) {
            ok = group_and(2, 128, wait_or_abort_t<GIVEUP>(bar_s, (uint32_t)(c & 1), abort_flag));
            if (ok) {
              tc_fence_after();
              float o[64];
              tmem_ld64b(tl + T_DO, o);
              tc_fence_before();
              group_sync(2, 128);
              if (ow == 0 && lane == 0) mbar_arrive(do_free);
#pragma unroll
              for (int r = 0; r < 64; ++r) ost[r * 128 + row] = o[r];
            }
          }
          cp_async_wait_all();  // this lane's gate copies
          // the staged chunk (and every warp's decision to go on) to all seven warps
          ok = group_and(3, 32 * kEw, ok);
          if (!ok) break;
          // the sums of squares of this warp's rows first, reduced together (independent chains)
          float ss[kRows];
#pragma unroll
          for (int i = 0; i < kRows; ++i) {
            const int r = ow + kEw * i;
            const float4 y = r < n ? *reinterpret_cast<const float4*>(ost + r * 128 + 4 * lane)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            ss[i] = y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
          }
#pragma unroll
          for (int m = 16; m > 0; m >>= 1)
#pragma unroll
            for (int i = 0; i < kRows; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], m);
#pragma unroll
          for (int i = 0; i < kRows; ++i) {
            const int r = ow + kEw * i;
            if (r >= n) break;
            float4 y = *reinterpret_cast<const float4*>(ost + r * 128 + 4 * lane);
            const size_t orow = ((size_t)(t0 + r) * H + h) * 128 + 4 * lane;
            const float inv = rsqrtf(ss[i] * (1.f / 128.f) + p.eps);
            const uint2 gw = sgate[r * 32];
            const float2 g01 = unpack_bf2(gw.x), g23 = unpack_bf2(gw.y);
            y.x = y.x * inv * wv.x * sigmoid_tanh(g01.x);
            y.y = y.y * inv * wv.y * sigmoid_tanh(g01.y);
            y.z = y.z * inv * wv.z * sigmoid_tanh(g23.x);
            y.w = y.w * inv * wv.w * sigmoid_tanh(g23.y);
            store_row(out + orow, y);
          }
          group_sync(3, 32 * kEw);  // staging buffer and gate rows free for the next chunk
        }
      }
    };
    if (p.gate != nullptr) readout(std::true_type{});
    else readout(std::false_type{});
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) atomicOr(p.err, KDA_DEVERR_WAIT_TIMEOUT);
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// Segment merge: S_in(p+1) = P_p S_in(p) + b_p for 1 <= p < p_last (S_in(1) comes from the
// transitions), fp32, on a 32-column slice of the state per CTA.  P_p (64 KB) is staged into shared memory by bulk copies one step ahead; warp w
// computes rows 16 w .. 16 w + 15 of the slice, lane = column, so P is read as broadcast float4s
// and the state slice column-wise without bank conflicts.
constexpr int kMergeThreads = 256;
constexpr int kMergeCols = 32;
constexpr uint32_t kMergeSmem = 2 * 65536 + 128 * kMergeCols * 4 + 64;
__global__ void __launch_bounds__(kMergeThreads, 1) kda_cp_merge(const ScanParams p) {
  extern __shared__ __align__(128) uint8_t msm[];
  float* sP = reinterpret_cast<float*>(msm);                        // [2][128][128]
  float* sS = reinterpret_cast<float*>(msm + 2 * 65536);            // [128][kMergeCols]
  uint64_t* bar = reinterpret_cast<uint64_t*>(msm + 2 * 65536 + 128 * kMergeCols * 4);  // [2]
  const int b = blockIdx.x, h = blockIdx.y, j0 = kMergeCols * blockIdx.z, tid = threadIdx.x;
  const int lane = tid & 31, rg = tid >> 5;
  griddep_launch_dependents();
  griddep_wait();  // the transitions' P, b and S_in(1); every CTA waits (see the state pass)
  if (p.cu != nullptr && p.plan[p.B + 1] == 0) return;
  int64_t first_chunk, t_begin, len;
  const int64_t nchunks = sequence_chunks(b, p.plan, p.cu, p.B, p.T, first_chunk, t_begin, len);
  const int64_t p_last = nchunks > 0 ? (nchunks - 1) / p.seg_len : 0;
  const int64_t nsteps = p_last - 1;  // step i composes segment i + 1
  if (nsteps <= 0) return;
  float* cp = p.cp + (size_t)(b * p.H + h) * p.nseg * 3 * kCpMat;
  int64_t issued = 0;
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_fence_init();
    for (; issued < 2 && issued < nsteps; ++issued) {
      mbar_arrive_expect_tx(&bar[issued], 65536);
      bulk_g2s(sP + issued * 16384, cp + (size_t)(issued + 1) * 3 * kCpMat, 65536, &bar[issued]);
    }
  }
  // S_in(1) slice and the first b slice: all loads in flight before any is used
  constexpr int kPer = 128 * kMergeCols / kMergeThreads;
  {
    const float* sin1 = cp + (size_t)(3 + 2) * kCpMat;
    float x[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = tid + i * kMergeThreads;
      x[i] = sin1[(size_t)(e / kMergeCols) * 128 + j0 + e % kMergeCols];
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) sS[tid + i * kMergeThreads] = x[i];
  }
  float acc[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] = cp[(size_t)(3 + 1) * kCpMat + (size_t)(rg * 16 + j) * 128 + j0 + lane];
  __syncthreads();
  bool ok = true;
  for (int64_t step = 0; step < nsteps; ++step) {
    const int64_t s = step + 1;
    const int buf = (int)(step & 1);
    ok = __syncthreads_and(mbar_wait(&bar[buf], (uint32_t)((step >> 1) & 1))) != 0;
    if (!ok) break;
    const float* P = sP + buf * 16384 + (rg * 16) * 128;
#pragma unroll 2
    for (int k = 0; k < 128; k += 4) {
      const float s0 = sS[k * kMergeCols + lane], s1 = sS[(k + 1) * kMergeCols + lane];
      const float s2 = sS[(k + 2) * kMergeCols + lane], s3 = sS[(k + 3) * kMergeCols + lane];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float4 pv = *reinterpret_cast<const float4*>(P + j * 128 + k);
        acc[j] = fmaf(pv.x, s0, fmaf(pv.y, s1, fmaf(pv.z, s2, fmaf(pv.w, s3, acc[j]))));
      }
    }
    fence_proxy_async_smem();  // reads of this P buffer precede the next bulk copy into it
    __syncthreads();
    if (tid == 0 && issued < nsteps) {
      mbar_arrive_expect_tx(&bar[buf], 65536);
      bulk_g2s(sP + buf * 16384, cp + (size_t)(issued + 1) * 3 * kCpMat, 65536, &bar[buf]);
      ++issued;
    }
    float* sin_next = cp + ((size_t)(s + 1) * 3 + 2) * kCpMat;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int r = rg * 16 + j;
      sS[r * kMergeCols + lane] = acc[j];
      sin_next[(size_t)r * 128 + j0 + lane] = acc[j];
    }
    if (step + 1 < nsteps) {  // the next step's b slice
      const float* bo = cp + ((size_t)(s + 1) * 3 + 1) * kCpMat;
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[j] = bo[(size_t)(rg * 16 + j) * 128 + j0 + lane];
    }
    __syncthreads();
  }
  if (!ok && tid == 0) {
    atomicOr(p.err, KDA_DEVERR_WAIT_TIMEOUT);
    // let the copies in flight land before the CTA's shared memory is released (each completes on
    // its own; the wait keeps the default bound)
    for (int64_t s = 0; s < issued; ++s) mbar_wait(&bar[s & 1], (uint32_t)((s >> 1) & 1));
  }
}

// Launch with programmatic stream serialization: the kernel may start while its predecessor on
// the stream drains (it calls griddep_wait() before reading that predecessor's results).
template <typename... KArgs, typename... Args>
cudaError_t launch_after(void (*kernel)(KArgs...), dim3 grid, int threads, size_t smem, cudaStream_t st,
                         Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename Tout>
cudaError_t launch_scan(const PrefillArgs& a, const uint8_t* records, const int32_t* plan, float* cp, int nseg,
                        int64_t seg_len, cudaStream_t st) {
  static DeviceOnce once;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  cudaError_t e0 = once.run(dev, [] {
    void (*kernels[])(const ScanParams) = {kda_tc_chunk_scan<Tout, 0, false>, kda_tc_chunk_scan<Tout, 1, false>,
                                           kda_tc_chunk_scan<Tout, 0, true>, kda_tc_chunk_scan<Tout, 0, false, true>,
                                           kda_tc_chunk_scan<Tout, 1, false, true>};
    for (auto* k : kernels) {
      const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScanSmem);
      if (e != cudaSuccess) return e;
    }
    return cudaFuncSetAttribute(kda_cp_merge, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMergeSmem);
  });
  if (e0 != cudaSuccess) return e0;
  // the variants whose waits give up at once (abort-path tests) are used when asked for; the
  // checkpointing pass has none
  auto* mode0 = a.give_up ? kda_tc_chunk_scan<Tout, 0, false, true> : kda_tc_chunk_scan<Tout, 0, false>;
  auto* mode1 = a.give_up ? kda_tc_chunk_scan<Tout, 1, false, true> : kda_tc_chunk_scan<Tout, 1, false>;
  ScanParams p;
  p.records = records; p.plan = plan; p.cu = a.cu_seqlens; p.B = a.B; p.T = a.T; p.H = a.H;
  p.h0 = a.h0; p.hT = a.hT; p.out = a.out; p.gate = static_cast<const __nv_bfloat16*>(a.epi.gate);
  p.norm_w = a.epi.norm_weight; p.eps = a.epi.eps; p.err = a.err;
  p.nseg = nseg; p.seg_len = seg_len; p.cp = cp;
  p.ckpt = a.ckpt; p.ckpt_chunks = a.ckpt_chunks;
  p.seg_P = a.seg_P; p.seg_b = a.seg_b;
  if (a.seg_P != nullptr) {
    // segment map of one token range: both runs of every segment (one segment: P and b directly)
    TraceScope ts("kda_tc_chunk_scan_segmap", st);
    return launch_after(mode1, dim3((unsigned)a.H, 1, (unsigned)(2 * nseg)), kScanThreads, kScanSmem, st, p);
  }
  if (nseg > 1) {
    {
      // segment 0 from h0, then b_p and P_p for 1 <= p <= nseg - 2
      TraceScope ts("kda_tc_chunk_scan_transition", st);
      cudaError_t e = launch_after(mode1, dim3((unsigned)(a.B * a.H), 1, (unsigned)(2 * nseg - 3)), kScanThreads,
                                   kScanSmem, st, p);
      if (e != cudaSuccess) return e;
    }
    if (nseg > 2) {
      TraceScope ts("kda_cp_merge", st);
      cudaError_t e = launch_after(kda_cp_merge, dim3((unsigned)a.B, (unsigned)a.H, 128 / kMergeCols), kMergeThreads,
                                   kMergeSmem, st, p);
      if (e != cudaSuccess) return e;
    }
  }
  TraceScope ts("kda_tc_chunk_scan", st);
  const dim3 grid((unsigned)(a.B * a.H), 1, (unsigned)nseg);
  if (a.ckpt != nullptr) return launch_after(kda_tc_chunk_scan<Tout, 0, true>, grid, kScanThreads, kScanSmem, st, p);
  return launch_after(mode0, grid, kScanThreads, kScanSmem, st, p);
}

}  // namespace

cudaError_t scan_tc_launch(const PrefillArgs& a, const uint8_t* records, const int32_t* plan, float* cp, int nseg,
                           int64_t seg_len, cudaStream_t st) {
  return a.out_bf16 ? launch_scan<__nv_bfloat16>(a, records, plan, cp, nseg, seg_len, st)
                    : launch_scan<float>(a, records, plan, cp, nseg, seg_len, st);
}

}  // namespace kda
