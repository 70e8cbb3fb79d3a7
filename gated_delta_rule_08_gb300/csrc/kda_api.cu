// C-ABI entry points of libkda: argument validation, dispatch, device error word.
// The public contract is include/kda.h.
#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "../../include/kda.h"
#include "kda_internal.h"

#define KDA_API extern "C" __attribute__((visibility("default")))

namespace kda {
namespace {

// Device error word (KDA_DEVERR_* bits), one per device that loads the library.
// Host code only uses its address, obtained per device with cudaGetSymbolAddress.
__device__ unsigned int g_device_error = 0u;

std::mutex g_mu;
unsigned int* g_err_ptr[kMaxDevices] = {};
int g_cc_major[kMaxDevices] = {}, g_cc_minor[kMaxDevices] = {};

// Error-word address and compute capability of the current device.
kda_status device_state(unsigned int** err, int* major, int* minor) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return KDA_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return KDA_ERR_CUDA;
    g_cc_major[dev] = prop.major;
    g_cc_minor[dev] = prop.minor;
    g_err_ptr[dev] = static_cast<unsigned int*>(p);
  }
  *err = g_err_ptr[dev];
  if (major) *major = g_cc_major[dev];
  if (minor) *minor = g_cc_minor[dev];
  return KDA_OK;
}

bool dims_ok(int dk, int dv) { return (dk == 64 || dk == 128) && (dv == 64 || dv == 128); }

// ---- precondition checks (KDA_DEBUG_CHECKS): one pass over the inputs, flag on the device
__global__ void check_decay_beta(const float4* __restrict__ g, int64_t n_g4, const float* __restrict__ beta,
                                 int64_t n_beta, unsigned int* err) {
  bool bad = false;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_g4; i += stride) {
    const float4 x = g[i];
    bad |= !(x.x > -5.f && x.x <= 0.f) || !(x.y > -5.f && x.y <= 0.f) || !(x.z > -5.f && x.z <= 0.f) ||
           !(x.w > -5.f && x.w <= 0.f);
  }
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_beta; i += stride) {
    const float x = beta[i];
    bad |= !(x >= 0.f && x <= 1.f);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(err, KDA_DEVERR_PRECONDITION);
}
// distinct decode slots: every in-range slot index compared with the ones after it (O(N^2) work,
// spread over the grid; a debugging aid)
__global__ void check_distinct_slots(const int32_t* __restrict__ slot, int N, int num_slots, unsigned int* err) {
  bool bad = false;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < N; i += gridDim.x * blockDim.x) {
    const int si = slot[i];
    if (si < 0 || si >= num_slots) continue;  // reported by the decode kernel itself
    for (int j = i + 1; j < N; ++j) bad |= slot[j] == si;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(err, KDA_DEVERR_PRECONDITION);
}

cudaError_t launch_checks(const float* g, int64_t n_g, const float* beta, int64_t n_beta, const int32_t* slot, int N,
                          int num_slots, unsigned int* err, cudaStream_t st) {
  TraceScope ts("kda_debug_checks", st);
  if (n_g > 0 || n_beta > 0) {
    const int64_t work = (n_g / 4 > n_beta ? n_g / 4 : n_beta);
    const int grid = (int)((work + 255) / 256 < 1184 ? (work + 255) / 256 : 1184);
    check_decay_beta<<<grid > 0 ? grid : 1, 256, 0, st>>>(reinterpret_cast<const float4*>(g), n_g / 4, beta,
                                                          n_beta, err);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (slot != nullptr && N > 1) {
    check_distinct_slots<<<(N + 255) / 256, 256, 0, st>>>(slot, N, num_slots, err);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t blob_bytes(kda_dtype dtype, int dk, int dv) {
  if (dtype == KDA_DTYPE_BF16 && prefill_tc_supported(dk, dv)) return prefill_tc_blob_bytes(dk, dv);
  return prefill_cc_blob_bytes(dk, dv);
}

}  // namespace

bool test_wait_timeout() {
  const char* e = getenv("KDA_TEST_WAIT_TIMEOUT");
  return e != nullptr && *e != '\0' && strcmp(e, "0") != 0;
}

bool debug_checks() {
  const char* e = getenv("KDA_DEBUG_CHECKS");
  return e != nullptr && *e != '\0' && strcmp(e, "0") != 0;
}
}  // namespace kda

using namespace kda;

KDA_API const char* kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    case KDA_ERR_DEVICE: return "KDA_ERR_DEVICE";
    case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
  }
  return "KDA_STATUS_UNKNOWN";
}

KDA_API size_t kda_chunk_fwd_workspace_size(int B, int64_t T, int H, int dk, int dv, int C, kda_dtype dtype) {
  if (B <= 0 || T < 0 || H <= 0 || C != kChunk || !dims_ok(dk, dv)) return 0;
  if (dtype != KDA_DTYPE_BF16 && dtype != KDA_DTYPE_FP32) return 0;
  // Sized for the cu_seqlens case (the larger bound), so one size serves both.
  const int64_t chunks = max_chunks(B, T, true) > max_chunks(B, T, false) ? max_chunks(B, T, true)
                                                                           : max_chunks(B, T, false);
  size_t bytes = plan_bytes(B) + align_up((size_t)chunks * (size_t)H * blob_bytes(dtype, dk, dv), 256);
  if (dtype == KDA_DTYPE_BF16 && prefill_tc_supported(dk, dv)) bytes += prefill_tc_cp_bytes(B, T, H);
  return bytes;
}

namespace {
kda_status chunk_fwd_common(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            const float* h0, const int32_t* cu_seqlens, void* out, float* hT, float* states,
                            int64_t ckpt_chunks, int B, int64_t T, int H, int dk, int dv, int C, kda_dtype dtype,
                            kda_dtype out_dtype, const kda_epilogue* epi, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (B <= 0 || T < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  if (states && (ckpt_chunks <= 0 || !aligned16(states))) return KDA_ERR_INVALID_ARG;
  if (dtype != KDA_DTYPE_BF16 && dtype != KDA_DTYPE_FP32) return KDA_ERR_UNSUPPORTED;
  if (out_dtype != KDA_DTYPE_BF16 && out_dtype != KDA_DTYPE_FP32) return KDA_ERR_UNSUPPORTED;
  if (C != kChunk || !dims_ok(dk, dv)) return KDA_ERR_UNSUPPORTED;
  const int64_t T_tot = cu_seqlens ? T : (int64_t)B * T;
  if (T_tot > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_INVALID_ARG;
  if (epi && T_tot > 0 && !epi->gate_logits) return KDA_ERR_INVALID_ARG;
  if (epi && !(epi->eps >= 0.f)) return KDA_ERR_INVALID_ARG;
  if (T_tot > ((int64_t)1 << 31) * 64 / H) return KDA_ERR_UNSUPPORTED;  // chunk index fits int32
  if (out && (out == q || out == k || out == v || out == (const void*)g || out == (const void*)beta))
    return KDA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(out) ||
      !aligned16(h0) || !aligned16(hT) || (epi && (!aligned16(epi->gate_logits) || !aligned16(epi->norm_weight))))
    return KDA_ERR_INVALID_ARG;
  const size_t need = kda_chunk_fwd_workspace_size(B, T, H, dk, dv, C, dtype);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return KDA_ERR_WORKSPACE;

  unsigned int* err = nullptr;
  int major = 0, minor = 0;
  kda_status st = device_state(&err, &major, &minor);
  if (st != KDA_OK) return st;
  if (major != 10 || minor != 3) return KDA_ERR_UNSUPPORTED;  // built for sm_103a only

  PrefillArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = h0; a.cu_seqlens = cu_seqlens;
  a.out = out; a.hT = hT; a.B = B; a.T = T; a.T_tot = T_tot; a.H = H; a.dk = dk; a.dv = dv;
  a.bf16 = (dtype == KDA_DTYPE_BF16);
  a.out_bf16 = (out_dtype == KDA_DTYPE_BF16);
  a.epi.gate = epi ? epi->gate_logits : nullptr;
  a.epi.norm_weight = epi ? epi->norm_weight : nullptr;
  a.epi.eps = epi ? epi->eps : 0.f;
  a.workspace = workspace; a.workspace_bytes = workspace_bytes; a.err = err;
  a.ckpt = states; a.ckpt_chunks = states ? ckpt_chunks : 0;
  a.give_up = test_wait_timeout();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (debug_checks() &&
      launch_checks(g, T_tot * H * dk, beta, T_tot * H, nullptr, 0, 0, err, s) != cudaSuccess)
    return KDA_ERR_CUDA;
  cudaError_t e = (a.bf16 && prefill_tc_supported(dk, dv)) ? prefill_tc_launch(a, s) : prefill_cc_launch(a, s);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
}  // namespace

KDA_API kda_status kda_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                                 const float* beta, const float* h0, const int32_t* cu_seqlens, void* out,
                                 float* hT, int B, int64_t T, int H, int dk, int dv, int C, kda_dtype dtype,
                                 kda_dtype out_dtype, const kda_epilogue* epi, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  return chunk_fwd_common(q, k, v, g, beta, h0, cu_seqlens, out, hT, nullptr, 0, B, T, H, dk, dv, C, dtype,
                          out_dtype, epi, workspace, workspace_bytes, stream);
}

KDA_API kda_status kda_chunk_fwd_checkpoints(const void* q, const void* k, const void* v, const float* g,
                                             const float* beta, const float* h0, const int32_t* cu_seqlens,
                                             void* out, float* hT, float* states, int64_t ckpt_chunks, int B,
                                             int64_t T, int H, int dk, int dv, int C, kda_dtype dtype,
                                             kda_dtype out_dtype, const kda_epilogue* epi, void* workspace,
                                             size_t workspace_bytes, void* stream) {
  if (!states) return KDA_ERR_INVALID_ARG;
  return chunk_fwd_common(q, k, v, g, beta, h0, cu_seqlens, out, hT, states, ckpt_chunks, B, T, H, dk, dv, C, dtype,
                          out_dtype, epi, workspace, workspace_bytes, stream);
}

KDA_API kda_status kda_chunk_fwd_segment_map(const void* k, const void* v, const float* g, const float* beta,
                                             float* P, float* b, int64_t T, int H, int dk, int dv, int C,
                                             kda_dtype dtype, void* workspace, size_t workspace_bytes,
                                             void* stream) {
  if (T < 0 || H <= 0 || !P || !b) return KDA_ERR_INVALID_ARG;
  if (dtype != KDA_DTYPE_BF16 && dtype != KDA_DTYPE_FP32) return KDA_ERR_UNSUPPORTED;
  if (C != kChunk || !dims_ok(dk, dv)) return KDA_ERR_UNSUPPORTED;
  if (dtype != KDA_DTYPE_BF16 || !prefill_tc_supported(dk, dv)) return KDA_ERR_UNSUPPORTED;
  if (T > 0 && (!k || !v || !g || !beta)) return KDA_ERR_INVALID_ARG;
  if (T > ((int64_t)1 << 31) * 64 / H) return KDA_ERR_UNSUPPORTED;
  if (!aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(P) || !aligned16(b)) return KDA_ERR_INVALID_ARG;
  const size_t need = kda_chunk_fwd_workspace_size(1, T, H, dk, dv, C, dtype);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return KDA_ERR_WORKSPACE;
  unsigned int* err = nullptr;
  int major = 0, minor = 0;
  kda_status st = device_state(&err, &major, &minor);
  if (st != KDA_OK) return st;
  if (major != 10 || minor != 3) return KDA_ERR_UNSUPPORTED;
  PrefillArgs a{};
  a.q = k; a.k = k; a.v = v; a.g = g; a.beta = beta;  // the read-out operands are not used
  a.B = 1; a.T = T; a.T_tot = T; a.H = H; a.dk = dk; a.dv = dv;
  a.bf16 = true; a.out_bf16 = true;
  a.workspace = workspace; a.workspace_bytes = workspace_bytes; a.err = err;
  a.give_up = test_wait_timeout();
  a.seg_P = P; a.seg_b = b;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (debug_checks() && launch_checks(g, T * H * dk, beta, T * H, nullptr, 0, 0, err, s) != cudaSuccess)
    return KDA_ERR_CUDA;
  return prefill_tc_launch(a, s) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

KDA_API kda_status kda_state_compose(const float* P, const float* b, const float* S0, float* S_out, int n, int H,
                                     int dk, int dv, void* stream) {
  if (n < 0 || H <= 0 || !S_out || (n > 0 && (!P || !b))) return KDA_ERR_INVALID_ARG;
  if (!dims_ok(dk, dv)) return KDA_ERR_UNSUPPORTED;
  if (!aligned16(P) || !aligned16(b) || !aligned16(S0) || !aligned16(S_out)) return KDA_ERR_INVALID_ARG;
  unsigned int* err = nullptr;
  int major = 0, minor = 0;
  kda_status st = device_state(&err, &major, &minor);
  if (st != KDA_OK) return st;
  if (major != 10 || minor != 3) return KDA_ERR_UNSUPPORTED;
  return state_compose_launch(P, b, S0, S_out, n, H, dk, dv, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KDA_OK
             : KDA_ERR_CUDA;
}

KDA_API size_t kda_chunk_bwd_workspace_size(int B, int64_t T, int H, int dk, int dv) {
  if (B <= 0 || T < 0 || H <= 0 || !dims_ok(dk, dv)) return 0;
  // sized for the larger of the two chunk bounds (with and without cu_seqlens)
  const size_t a = backward_scratch_bytes(B, T, H, dk, dv, true), b = backward_scratch_bytes(B, T, H, dk, dv, false);
  return plan_bytes(B) + (a > b ? a : b);
}

KDA_API kda_status kda_chunk_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                 const float* h0, const int32_t* cu_seqlens, const void* dout, const float* dhT,
                                 float* dq, float* dk_, float* dv_, float* dg, float* dbeta, float* dh0, int B,
                                 int64_t T, int H, int dk, int dv, kda_dtype dtype, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (B <= 0 || T < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  if (dtype != KDA_DTYPE_BF16 && dtype != KDA_DTYPE_FP32) return KDA_ERR_UNSUPPORTED;
  if (!dims_ok(dk, dv)) return KDA_ERR_UNSUPPORTED;
  const int64_t T_tot = cu_seqlens ? T : (int64_t)B * T;
  if (T_tot > 0 && (!q || !k || !v || !g || !beta || !dout || !dq || !dk_ || !dv_ || !dg || !dbeta))
    return KDA_ERR_INVALID_ARG;
  if (T_tot > ((int64_t)1 << 31) * 64 / H) return KDA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(dout) || !aligned16(h0) ||
      !aligned16(dhT) || !aligned16(dq) || !aligned16(dk_) || !aligned16(dv_) || !aligned16(dg) || !aligned16(dh0))
    return KDA_ERR_INVALID_ARG;
  const size_t need = kda_chunk_bwd_workspace_size(B, T, H, dk, dv);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return KDA_ERR_WORKSPACE;
  unsigned int* err = nullptr;
  int major = 0, minor = 0;
  kda_status st = device_state(&err, &major, &minor);
  if (st != KDA_OK) return st;
  if (major != 10 || minor != 3) return KDA_ERR_UNSUPPORTED;
  if (T_tot == 0 && dh0 == nullptr) return KDA_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* plan = static_cast<int32_t*>(workspace);
  if (cu_seqlens) {
    TraceScope ts("kda_plan", s);
    if (plan_launch(cu_seqlens, B, T_tot, plan, err, s) != cudaSuccess) return KDA_ERR_CUDA;
  }
  BackwardArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = h0; a.cu_seqlens = cu_seqlens; a.plan = plan;
  a.dout = dout; a.dhT = dhT; a.dq = dq; a.dk = dk_; a.dv = dv_; a.dg = dg; a.dbeta = dbeta; a.dh0 = dh0;
  a.B = B; a.T = T; a.H = H; a.dim_k = dk; a.dim_v = dv; a.bf16 = (dtype == KDA_DTYPE_BF16);
  a.workspace = workspace;
  return backward_launch(a, s) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

namespace {
kda_status decode_common(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         float* state_pool, const int32_t* slot_idx, const int32_t* ntok_per_req, void* out, int N,
                         int n_tok, int H, int dk, int dv, int num_slots, bool commit, kda_dtype dtype,
                         kda_dtype out_dtype, const kda_epilogue* epi, void* stream) {
  if (N < 0 || n_tok < 0 || H <= 0 || num_slots < 0) return KDA_ERR_INVALID_ARG;
  if (dtype != KDA_DTYPE_BF16 && dtype != KDA_DTYPE_FP32) return KDA_ERR_UNSUPPORTED;
  if (out_dtype != KDA_DTYPE_BF16 && out_dtype != KDA_DTYPE_FP32) return KDA_ERR_UNSUPPORTED;
  if (!dims_ok(dk, dv)) return KDA_ERR_UNSUPPORTED;
  const bool work = N > 0 && n_tok > 0;
  if (work && (!q || !k || !v || !g || !beta || !state_pool || !slot_idx || !out)) return KDA_ERR_INVALID_ARG;
  if (epi && work && !epi->gate_logits) return KDA_ERR_INVALID_ARG;
  if (epi && !(epi->eps >= 0.f)) return KDA_ERR_INVALID_ARG;
  if ((int64_t)N * H > 0x7fffffff || (int64_t)N * n_tok * H > 0x7fffffff) return KDA_ERR_UNSUPPORTED;
  // v and the gate logits are staged into shared memory by 16-byte asynchronous copies
  if (!aligned16(state_pool) || !aligned16(v) || (epi && !aligned16(epi->gate_logits))) return KDA_ERR_INVALID_ARG;
  unsigned int* err = nullptr;
  int major = 0, minor = 0;
  kda_status st = device_state(&err, &major, &minor);
  if (st != KDA_OK) return st;
  if (major != 10 || minor != 3) return KDA_ERR_UNSUPPORTED;
  if (!work) return KDA_OK;
  DecodeArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.state_pool = state_pool; a.slot_idx = slot_idx;
  a.out = out; a.N = N; a.H = H; a.dk = dk; a.dv = dv; a.num_slots = num_slots;
  a.n_tok = n_tok; a.ntok_per_req = ntok_per_req; a.commit = commit;
  a.bf16 = (dtype == KDA_DTYPE_BF16);
  a.out_bf16 = (out_dtype == KDA_DTYPE_BF16);
  a.epi.gate = epi ? epi->gate_logits : nullptr;
  a.epi.norm_weight = epi ? epi->norm_weight : nullptr;
  a.epi.eps = epi ? epi->eps : 0.f;
  a.err = err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t rows = (int64_t)N * n_tok * H;
  if (debug_checks() && launch_checks(g, rows * dk, beta, rows, slot_idx, N, num_slots, err, s) != cudaSuccess)
    return KDA_ERR_CUDA;
  cudaError_t e = decode_launch(a, s);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
}  // namespace

KDA_API kda_status kda_decode_step(const void* q, const void* k, const void* v, const float* g,
                                   const float* beta, float* state_pool, const int32_t* slot_idx, void* out,
                                   int N, int H, int dk, int dv, int num_slots, kda_dtype dtype,
                                   kda_dtype out_dtype, const kda_epilogue* epi, void* stream) {
  return decode_common(q, k, v, g, beta, state_pool, slot_idx, nullptr, out, N, 1, H, dk, dv, num_slots, true, dtype,
                       out_dtype, epi, stream);
}

KDA_API kda_status kda_decode_multi(const void* q, const void* k, const void* v, const float* g,
                                    const float* beta, float* state_pool, const int32_t* slot_idx,
                                    const int32_t* ntok_per_req, void* out, int N, int n_tok, int H, int dk, int dv,
                                    int num_slots, int commit, kda_dtype dtype, kda_dtype out_dtype,
                                    const kda_epilogue* epi, void* stream) {
  return decode_common(q, k, v, g, beta, state_pool, slot_idx, ntok_per_req, out, N, n_tok, H, dk, dv, num_slots,
                       commit != 0, dtype, out_dtype, epi, stream);
}

KDA_API kda_status kda_get_device_error(void* stream, uint32_t* flags) {
  if (!flags) return KDA_ERR_INVALID_ARG;
  unsigned int* err = nullptr;
  kda_status st = device_state(&err, nullptr, nullptr);
  if (st != KDA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return KDA_ERR_CUDA;
  if (v != 0 && cudaMemset(err, 0, sizeof(v)) != cudaSuccess) return KDA_ERR_CUDA;
  *flags = v;
  return KDA_OK;
}

// ----------------------------------------------------------------------------- tracing
#include <string.h>

#include <string>
#include <vector>

namespace kda {
namespace {
struct TraceRec {
  const char* name;
  cudaEvent_t a, b;
};
std::mutex g_tmu;
bool g_trace_on = false;
std::vector<TraceRec> g_recs;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
}  // namespace

bool trace_enabled() { return g_trace_on; }

void trace_begin(const char* name, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_tmu);
  TraceRec r{name, take_event(), nullptr};
  if (r.a) cudaEventRecord(r.a, s);
  g_recs.push_back(r);
}

void trace_end(cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_tmu);
  if (g_recs.empty()) return;
  TraceRec& r = g_recs.back();
  r.b = take_event();
  if (r.b) cudaEventRecord(r.b, s);
}
}  // namespace kda

KDA_API kda_status kda_trace_enable(int enable) {
  std::lock_guard<std::mutex> lk(g_tmu);
  g_trace_on = enable != 0;
  return KDA_OK;
}

KDA_API kda_status kda_trace_collect(int max_entries, char* names, int* launches, double* total_ms,
                                     int* n_entries) {
  if (max_entries < 0 || !n_entries || (max_entries > 0 && (!names || !launches || !total_ms)))
    return KDA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_tmu);
  std::vector<std::string> keys;
  std::vector<int> cnt;
  std::vector<double> ms;
  kda_status st = KDA_OK;
  for (TraceRec& r : g_recs) {
    float t = 0.f;
    if (!r.a || !r.b || cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
      st = KDA_ERR_CUDA;
    size_t i = 0;
    while (i < keys.size() && keys[i] != r.name) ++i;
    if (i == keys.size()) { keys.emplace_back(r.name); cnt.push_back(0); ms.push_back(0.0); }
    cnt[i] += 1;
    ms[i] += t;
    if (r.a) g_event_pool.push_back(r.a);
    if (r.b) g_event_pool.push_back(r.b);
  }
  g_recs.clear();
  const int n = (int)keys.size() < max_entries ? (int)keys.size() : max_entries;
  for (int i = 0; i < n; ++i) {
    strncpy(names + 64 * i, keys[i].c_str(), 63);
    names[64 * i + 63] = '\0';
    launches[i] = cnt[i];
    total_ms[i] = ms[i];
  }
  *n_entries = n;
  return st;
}
