// Internal declarations shared by the host-side translation units of libkda.
// Not part of the public ABI (include/kda.h is).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

namespace kda {

constexpr int kChunk = 64;  // tokens per chunk (C)
constexpr int kMaxDevices = 64;

// One-time per-device set-up (kernel attributes, device properties), safe to call from several
// host threads: `init` runs under a lock until it has succeeded once on the device, and whatever it
// wrote is visible to every caller that returns cudaSuccess.
struct DeviceOnce {
  std::mutex mu;
  bool done[kMaxDevices] = {};
  template <class F>
  cudaError_t run(int dev, F&& init) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (done[dev]) return cudaSuccess;
    const cudaError_t e = init();
    if (e == cudaSuccess) done[dev] = true;
    return e;
  }
};

// The tensor-core kernels' bounded waits on work of their own CTA (mbarrier phases of copies, MMAs
// and hand-overs between warps) give up after ~2e7 polls.  With the environment variable
// KDA_TEST_WAIT_TIMEOUT set (any value but "" or "0"; read at every call) the launches use kernel
// variants whose waits give up at once, so that a test can make them run out on purpose and check
// that the kernels report KDA_DEVERR_WAIT_TIMEOUT and leave the device usable.  Waits for a CTA's own
// copies and MMAs to drain before it exits keep their bound in both variants.
bool test_wait_timeout();

// KDA_DEBUG_CHECKS (environment variable, read at every call; any value but "" or "0" enables it):
// before the hot-path kernels, a check kernel tests the documented preconditions on the device
// (g in (-5, 0], beta in [0, 1], distinct decode slots) and sets KDA_DEVERR_PRECONDITION.
bool debug_checks();

// Epilogue arguments as the kernels see them (gate == nullptr: no epilogue).
struct Epilogue {
  const void* gate;
  const float* norm_weight;
  float eps;
};

struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* h0;            // may be null
  const int32_t* cu_seqlens;  // may be null (equal lengths)
  void* out;
  float* hT;                  // may be null
  int B;
  int64_t T;                  // per-sequence length if cu_seqlens == null, else T_tot
  int64_t T_tot;
  int H, dk, dv;
  bool bf16;       // q, k, v, gate are bf16 (else fp32)
  bool out_bf16;   // out is bf16 (else fp32)
  Epilogue epi;
  void* workspace;
  size_t workspace_bytes;
  unsigned int* err;          // device error word
  float* ckpt;                // state checkpoints [n][H][dk][dv] fp32, or null
  int64_t ckpt_chunks;        // a checkpoint after every ckpt_chunks full chunks of a sequence
  bool give_up;               // launch the kernel variants whose waits give up at once (tests)
  // segment map (context parallelism across devices): instead of out / hT, the transition P
  // [H][dk][dk] and the offset b [H][dk][dv] of the whole token range (B == 1, no cu_seqlens)
  float* seg_P;
  float* seg_b;
};

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  float* state_pool;
  const int32_t* slot_idx;
  void* out;
  int N, H, dk, dv, num_slots;
  int n_tok;                     // tokens per request in the input arrays ([N, n_tok, H, ..])
  const int32_t* ntok_per_req;   // device [N] tokens to apply per request, or null (= n_tok)
  bool commit;                   // write the state back after the request's tokens
  bool bf16;
  bool out_bf16;
  Epilogue epi;
  unsigned int* err;
};

// Backward (kda_backward.cu): gradients of sum_t <dout_t, o_t> + <dhT, hT>.
struct BackwardArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* h0;            // may be null
  const int32_t* cu_seqlens;  // may be null
  const int32_t* plan;        // chunk offsets (written by plan_launch when cu_seqlens is given)
  const void* dout;           // [T_tot, H, dv] (input dtype)
  const float* dhT;           // [B, H, dk, dv] or null
  float* dq;                  // [T_tot, H, dk] fp32
  float* dk;                  // [T_tot, H, dk] fp32
  float* dv;                  // [T_tot, H, dv] fp32
  float* dg;                  // [T_tot, H, dk] fp32
  float* dbeta;               // [T_tot, H] fp32
  float* dh0;                 // [B, H, dk, dv] fp32 or null
  int B;
  int64_t T;                  // per-sequence length if cu_seqlens == null, else T_tot
  int H, dim_k, dim_v;
  bool bf16;
  void* workspace;            // plan region, then the backward scratch
};
int backward_slices(int B, int H, int dv);  // value-column slices per chain (1, 2 or 4)
size_t backward_scratch_bytes(int B, int64_t T, int H, int dk, int dv, bool has_cu);
// chunkwise backward (kda_backward_chunk.cu): per-chunk records, states and gradient scratch
size_t backward_chunked_bytes(int B, int64_t T, int H, int dk, int dv, bool has_cu);
cudaError_t backward_chunked_launch(const BackwardArgs& a, float* workspace, cudaStream_t stream);
cudaError_t backward_launch(const BackwardArgs& a, cudaStream_t stream);

// Upper bound on the number of 64-token chunks of a packed batch:
// sum_b ceil(len_b / 64) <= ceil(T_tot / 64) + B.
inline int64_t max_chunks(int B, int64_t T, bool has_cu) {
  if (!has_cu) return (int64_t)B * ((T + kChunk - 1) / kChunk);
  return (T + kChunk - 1) / kChunk + B;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Plan region at the start of the workspace: int32 chunk offsets [B+1] + one valid flag.
// plan: [B] exclusive chunk offsets, [B] total chunks, [B+1] cu_seqlens valid, [B+2 .. 2B+1] the
// sequences by decreasing length (see kda_device.cuh)
inline size_t plan_bytes(int B) { return align_up((size_t)(2 * B + 2) * sizeof(int32_t), 256); }

// fp32 CUDA-core path (kda_prefill_cc.cu)
size_t prefill_cc_blob_bytes(int dk, int dv);
cudaError_t prefill_cc_launch(const PrefillArgs& a, cudaStream_t stream);

// bf16 tensor-core path (kda_prefill_tc.cu, kda_scan_tc.cu)
size_t prefill_tc_blob_bytes(int dk, int dv);
bool prefill_tc_supported(int dk, int dv);
cudaError_t prefill_tc_launch(const PrefillArgs& a, cudaStream_t stream);
// Intra-device context parallelism: sequence segments of the state pass (1 = none), chosen
// from the problem shape and the current device's SM count, and the scratch it needs.
int prefill_tc_cp_segments(int B, int64_t T, int H);
size_t prefill_tc_cp_bytes(int B, int64_t T, int H);
cudaError_t scan_tc_launch(const PrefillArgs& a, const uint8_t* records, const int32_t* plan, float* cp, int nseg,
                           int64_t seg_len, cudaStream_t stream);

// context parallelism across devices (kda_kcp.cu): S_out = P[n-1](... (P[0] S0 + b[0]) ...) + b[n-1]
cudaError_t state_compose_launch(const float* P, const float* b, const float* S0, float* S_out, int n, int H, int dk,
                                 int dv, cudaStream_t stream);

// plan kernel (kda_prefill_cc.cu): chunk offsets per sequence + cu_seqlens validation
cudaError_t plan_launch(const int32_t* cu_seqlens, int B, int64_t T_tot, int32_t* plan,
                        unsigned int* err, cudaStream_t stream);

// decode (kda_decode.cu)
cudaError_t decode_launch(const DecodeArgs& a, cudaStream_t stream);

// Kernel tracing (kda_trace_enable): brackets internal launches with CUDA events.
bool trace_enabled();
void trace_begin(const char* name, cudaStream_t s);
void trace_end(cudaStream_t s);

struct TraceScope {
  cudaStream_t s;
  bool on;
  TraceScope(const char* name, cudaStream_t st) : s(st), on(trace_enabled()) {
    if (on) trace_begin(name, s);
  }
  ~TraceScope() {
    if (on) trace_end(s);
  }
};

}  // namespace kda
