/*
 * libkda — Kimi Delta Attention (KDA) hot path for GB300 (sm_103a).
 *
 * The operation (Kimi K3 technical-report walk-through, kimi-k3-paper.pages.dev):
 *   per (sequence, head), tokens t = 1..T, state S in R^{dk x dv} (rows = key channels)
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T      (section 2.2, Eq. 1)
 *     o_t = S_t^T q_t                                                        (section 2.4, Eq. 3)
 *   with a channel-wise decay exp(g_t), g_t in (-5, 0] (sections 2.3 and 3.2, Eq. 5), and
 *   an optional epilogue y_t = o_t / sqrt(mean(o_t^2) + eps) * w * sigmoid(gate_t)
 *   (section 3.3, Eq. 6: head-wise RMSNorm, then the sigmoid output gate).
 *
 * General conventions for every entry point:
 *   - All tensor pointers are caller-owned DEVICE memory, dense, row-major, in the
 *     layouts stated per argument, and 16-byte aligned (KDA_ERR_INVALID_ARG otherwise;
 *     for decode only the state pool, v and the gate logits must be).  The library never allocates device memory and
 *     never frees anything it is given.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL means
 *     the legacy default stream).  The call returns after validation and launch.
 *   - Argument errors are detected synchronously on the host: nothing is launched and
 *     the corresponding status is returned.  Conditions that only the device can see
 *     (an out-of-range slot index, inconsistent cu_seqlens, a device wait that ran out)
 *     are recorded in a per-device error word read by kda_get_device_error(); the
 *     affected rows are skipped, never trapped on.
 *   - dk, dv must each be 64 or 128 and C must be 64 (KDA_ERR_UNSUPPORTED otherwise).
 *   - `dtype` is the element type of q, k, v and the gate logits; `out_dtype` that of out
 *     (either may be bf16 or fp32).  bf16 prefill inputs with dk = dv = 128 run on the tcgen05
 *     tensor-core path.  fp32 inputs, and bf16 inputs with dk or dv = 64, run on a path with
 *     fp32 arithmetic whose chunk products are three-term tf32 warp MMAs (fp32-level accuracy:
 *     about 3e-5 max|err|/RMS against an fp64 reference over 8192 tokens).  The read-out is
 *     computed in fp32 and rounded once when stored in out_dtype.
 *   - Value range of the bf16 tensor-core path (prefill with dk = dv = 128): the values, the
 *     intra-chunk terms built from them (beta v, U_hat = T V, U = U_hat - W S) and the running
 *     state (h0 included) enter fp16 tensor-core operands, so each of |beta v|, |h0| and the
 *     state's entries must stay below 65504 (keep them below ~1e4 for margin; accumulation is
 *     fp32).  Past it the operand becomes inf, which reaches out and the state; the state pass
 *     tests every final state it reaches (and each checkpoint) and sets KDA_DEVERR_NONFINITE (the
 *     results are not valid; nothing traps).  Non-finite inputs set it too.  Values far below 1 (under ~6e-5 relative to the state) lose precision as fp16
 *     subnormals.  The recurrence is linear in (v, h0) jointly, so a caller with larger or tiny
 *     values can scale v and h0 by one factor and divide out and hT by it.  Keys and queries
 *     (unit norm) and the decays need no such care.  The fp32 paths have fp32 range.
 *   - Debugging: with the environment variable KDA_DEBUG_CHECKS set (any value but "" or "0";
 *     read at every call), kda_chunk_fwd*, kda_chunk_fwd_segment_map and kda_decode_* first run
 *     a check kernel over the inputs and set KDA_DEVERR_PRECONDITION when g is outside (-5, 0],
 *     beta outside [0, 1], or (decode) two requests name the same slot.  The check reads every
 *     g and beta once (decode: O(N^2) slot comparisons); it is off by default.
 *   - Testing: with the environment variable KDA_TEST_WAIT_TIMEOUT set (any value but "" or "0";
 *     read at every call) the prefill launches kernel variants whose bounded waits on work of
 *     their own CTA give up at once, so that a test can make them run out and see
 *     KDA_DEVERR_WAIT_TIMEOUT reported with the device left usable.  Not for production use.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent sizes          */
  KDA_ERR_UNSUPPORTED = 2,   /* dk/dv not in {64,128}, C != 64, unknown dtype, no sm_103a */
  KDA_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch, attribute, sync)      */
  KDA_ERR_DEVICE = 4,        /* the device error word is non-zero (kda_get_device_error)  */
  KDA_ERR_WORKSPACE = 5      /* workspace pointer NULL or smaller than required           */
} kda_status;

typedef enum {
  KDA_DTYPE_BF16 = 0,
  KDA_DTYPE_FP32 = 1
} kda_dtype;

/* Bits of the device error word. */
#define KDA_DEVERR_BAD_SLOT     0x1u  /* decode: slot_idx[n] outside [0, num_slots)        */
#define KDA_DEVERR_BAD_SEQLENS  0x2u  /* prefill: cu_seqlens not non-decreasing in [0, T]  */
#define KDA_DEVERR_WAIT_TIMEOUT 0x4u  /* a bounded device-side wait gave up                */
#define KDA_DEVERR_BAD_COUNT    0x8u  /* decode_multi: ntok_per_req[n] outside [0, n_tok]   */
#define KDA_DEVERR_NONFINITE   0x10u /* tensor-core path wrote a non-finite out / state value */
#define KDA_DEVERR_PRECONDITION 0x20u /* KDA_DEBUG_CHECKS: g, beta or slot_idx broke a precondition */

/* Optional fused epilogue (section 3.3, Eq. 6): RMSNorm over dv per (token, head), then
 * the sigmoid output gate.  The norm is taken on the fp32 read-out before rounding.
 *   gate_logits : [rows, H, dv] in the call's dtype (rows = T_tot or N)   — required
 *   norm_weight : [dv] fp32, shared by all heads; NULL means weight 1
 *   eps         : added to mean(o^2) before the square root (typical 1e-6) */
typedef struct {
  const void* gate_logits;
  const float* norm_weight;
  float eps;
} kda_epilogue;

/* Bytes of device scratch kda_chunk_fwd needs for this problem (0 on bad arguments).
 * T has the same meaning as in kda_chunk_fwd.  The scratch holds per-chunk operands
 * of the chunkwise form (~72.5 KB per 64-token chunk and head for bf16 at dk=dv=128)
 * plus a small plan. */
size_t kda_chunk_fwd_workspace_size(int B, int64_t T, int H, int dk, int dv, int C,
                                    kda_dtype dtype);

/* Chunked prefill over a packed batch of B variable-length sequences
 * (section 2.5, Eq. 4: serial inter-chunk state pass + parallel intra-chunk term).
 *   q, k      : [T_tot, H, dk]  (dtype)      L2-normalised upstream; not re-normalised
 *   v         : [T_tot, H, dv]  (dtype)
 *   g         : [T_tot, H, dk]  fp32         log-decay; precondition g in (-5, 0]
 *   beta      : [T_tot, H]      fp32         write strength, precondition in [0, 1]
 *   h0        : [B, H, dk, dv]  fp32 or NULL (zero initial states)
 *   cu_seqlens: [B+1] int32 device token offsets (cu[0] = 0, cu[B] = T_tot, non-decreasing),
 *               or NULL meaning B sequences of exactly T tokens each
 *   out       : [T_tot, H, dv]  (out_dtype)  must not alias any input
 *   hT        : [B, H, dk, dv]  fp32 or NULL (final states not written); may alias h0
 *   T         : tokens per sequence if cu_seqlens == NULL, else T_tot
 *   C         : chunk size, must be 64.  Chunks start at each sequence's first token.
 *   epi       : NULL or the fused epilogue
 *   workspace : device scratch of at least kda_chunk_fwd_workspace_size(...) bytes,
 *               256-byte aligned; contents on entry are ignored, on exit undefined.
 * Errors: KDA_ERR_INVALID_ARG / _UNSUPPORTED / _WORKSPACE before any launch; KDA_ERR_CUDA
 * if a launch fails.  Bad cu_seqlens set KDA_DEVERR_BAD_SEQLENS and the affected
 * sequences are skipped. */
kda_status kda_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* h0, const int32_t* cu_seqlens,
                         void* out, float* hT, int B, int64_t T, int H, int dk, int dv, int C,
                         kda_dtype dtype, kda_dtype out_dtype, const kda_epilogue* epi,
                         void* workspace, size_t workspace_bytes, void* stream);

/* kda_chunk_fwd that also stores intermediate states for a prefix cache (section 13.9: the KDA
 * path of the prefix cache can only resume at checkpoints stored at the 512-token hash-block
 * endpoints, i.e. ckpt_chunks = 8).  Sequence b stores its fp32 state after each
 * span = 64 * ckpt_chunks of its tokens: after tokens span, 2 span, ..., floor(len_b / span) span
 * (a checkpoint at the sequence end equals hT).
 *   states      : [n_ckpt, H, dk, dv] fp32 device, 16-byte aligned, written (not read), where
 *                 n_ckpt = sum_b floor(len_b / span); sequence b's checkpoints start at index
 *                 sum_{b' < b} floor(len_b' / span), in token order
 *   ckpt_chunks : >= 1
 * Every other argument, result and error is that of kda_chunk_fwd (states == NULL or
 * ckpt_chunks < 1: KDA_ERR_INVALID_ARG). */
kda_status kda_chunk_fwd_checkpoints(const void* q, const void* k, const void* v, const float* g,
                                     const float* beta, const float* h0, const int32_t* cu_seqlens,
                                     void* out, float* hT, float* states, int64_t ckpt_chunks, int B,
                                     int64_t T, int H, int dk, int dv, int C, kda_dtype dtype,
                                     kda_dtype out_dtype, const kda_epilogue* epi, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* One recurrent decode step for N requests, one token each, on a pool of fp32 states
 * updated in place (section 13.9 prefix cache: one fixed-size state per request in a
 * pooled layout; section 13.10: state update and read-out in a single fused kernel).
 *   q, k       : [N, H, dk] (dtype);  v : [N, H, dv] (dtype)
 *   g          : [N, H, dk] fp32;     beta : [N, H] fp32
 *   state_pool : [num_slots, H, dk, dv] fp32, read and written in place
 *   slot_idx   : [N] int32 device; request n uses state_pool[slot_idx[n]].  Slots must be
 *                distinct (duplicates race; not checked).  An index outside
 *                [0, num_slots) sets KDA_DEVERR_BAD_SLOT and leaves that request's out rows
 *                and every slot untouched.
 *   out        : [N, H, dv] (out_dtype)
 * Slots not named in slot_idx are never read or written. */
kda_status kda_decode_step(const void* q, const void* k, const void* v, const float* g,
                           const float* beta, float* state_pool, const int32_t* slot_idx,
                           void* out, int N, int H, int dk, int dv, int num_slots,
                           kda_dtype dtype, kda_dtype out_dtype, const kda_epilogue* epi,
                           void* stream);

/* Several tokens per request on the pooled states: the verify and accept steps of speculative
 * decoding (section 13.4: an in-place update cannot be rolled back once a draft token is
 * rejected, so verification must leave the pooled state untouched and the accepted tokens are
 * applied afterwards from their cached inputs).
 *   q, k       : [N, n_tok, H, dk] (dtype);  v : [N, n_tok, H, dv] (dtype)
 *   g          : [N, n_tok, H, dk] fp32;     beta : [N, n_tok, H] fp32
 *   gate (epi) : [N, n_tok, H, dv] (dtype)
 *   state_pool, slot_idx : as for kda_decode_step
 *   ntok_per_req : device int32 [N], tokens to apply to request n (its first ntok_per_req[n]
 *                tokens, in order), or NULL meaning all n_tok.  A value outside [0, n_tok] sets
 *                KDA_DEVERR_BAD_COUNT and that request is skipped (out and state untouched).
 *   out        : [N, n_tok, H, dv] (out_dtype); rows of tokens not applied are not written
 *   commit     : 0 = verify: the pool is only read; 1 = accept: the state of each request after
 *                its applied tokens is written back to its slot (a request with 0 tokens keeps
 *                its state).  Token t of a request sees exactly the state after its tokens < t,
 *                so outputs of a verify call and of the accepting call agree on the tokens both
 *                apply.
 * kda_decode_step(...) is kda_decode_multi(..., ntok_per_req = NULL, N, n_tok = 1, ..., commit = 1). */
kda_status kda_decode_multi(const void* q, const void* k, const void* v, const float* g,
                            const float* beta, float* state_pool, const int32_t* slot_idx,
                            const int32_t* ntok_per_req, void* out, int N, int n_tok, int H, int dk,
                            int dv, int num_slots, int commit, kda_dtype dtype, kda_dtype out_dtype,
                            const kda_epilogue* epi, void* stream);

/* Backward of the prefill recurrence (no epilogue): the gradients of
 *   L = sum_t <dout_t, o_t> + <dhT, hT>
 * with respect to q, k, v, g, beta and h0 (section 2.2 Eq. 1, section 2.4 Eq. 3; section 5.1 names
 * a KDA training kernel), to fp32 accuracy.  Two paths give the same gradients within rounding:
 * the chunkwise reverse mode of the section 2.5 / Eq. 4 chunk form (per-chunk records, serial
 * state passes over chunks, per-chunk gradients, its products as tensor-core MMAs with a
 * three-term tf32 split; used while its scratch, about 0.6 MB per (chunk, head) at dk = dv = 128,
 * stays within 48 GB), else an fp32 reverse-time sweep over the tokens with the state recomputed
 * from per-chunk checkpoints.  The environment variable
 * KDA_BACKWARD_PATH=token or =chunked forces one of them; it is read at every call, including by
 * kda_chunk_bwd_workspace_size, so query the size under the same setting.
 *   q, k, v, g, beta, h0, cu_seqlens, B, T, H, dk, dv, dtype : as for kda_chunk_fwd
 *   dout       : [T_tot, H, dv] (dtype)
 *   dhT        : [B, H, dk, dv] fp32 or NULL (zero)
 *   dq, dk_, dg: [T_tot, H, dk] fp32;  dv_ : [T_tot, H, dv] fp32;  dbeta : [T_tot, H] fp32
 *   dh0        : [B, H, dk, dv] fp32 or NULL (not written)
 *   workspace  : at least kda_chunk_bwd_workspace_size(B, T, H, dk, dv) bytes, 256-byte aligned
 * Every pointer 16-byte aligned (beta, dbeta exempt).  Errors as for kda_chunk_fwd. */
size_t kda_chunk_bwd_workspace_size(int B, int64_t T, int H, int dk, int dv);
kda_status kda_chunk_bwd(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* h0, const int32_t* cu_seqlens,
                         const void* dout, const float* dhT, float* dq, float* dk_, float* dv_,
                         float* dg, float* dbeta, float* dh0, int B, int64_t T, int H, int dk,
                         int dv, kda_dtype dtype, void* workspace, size_t workspace_bytes,
                         void* stream);

/* Context parallelism across devices (section 13.3.2, KCP; open-day article section 5.2).  A long
 * sequence is split into consecutive token ranges, one per device.  Over a range the state pass is
 * affine in the range's initial state: S_out = P S_in + b, with P the range's accumulated transition
 * and b its final state from a zero initial state.  Each device computes the map of its range, the
 * devices exchange these fixed-size maps (an all-gather of H * (dk*dk + dk*dv) fp32 values each),
 * each folds the maps of the ranges before its own into its initial state with kda_state_compose,
 * then runs kda_chunk_fwd on its range from that state.
 *
 * kda_chunk_fwd_segment_map: the map (P, b) of one token range of one sequence, all H heads.
 *   k, v, g, beta : the range's tokens: [T, H, dk], [T, H, dv] (dtype), [T, H, dk] fp32, [T, H] fp32
 *                   (no q: the map does not depend on it)
 *   P             : [H, dk, dk] fp32, written: S_out = P S_in + b for every initial state S_in
 *   b             : [H, dk, dv] fp32, written: the range's final state from S_in = 0
 *   workspace     : at least kda_chunk_fwd_workspace_size(1, T, H, dk, dv, C, dtype) bytes, 256-byte
 *                   aligned
 * T = 0 gives P = I and b = 0.  Supported: bf16 inputs with dk = dv = 128 (else KDA_ERR_UNSUPPORTED).
 * The range runs as one serial pass per head (two runs: from 0 and, for P, from I).
 * Other errors as for kda_chunk_fwd. */
kda_status kda_chunk_fwd_segment_map(const void* k, const void* v, const float* g, const float* beta,
                                     float* P, float* b, int64_t T, int H, int dk, int dv, int C,
                                     kda_dtype dtype, void* workspace, size_t workspace_bytes,
                                     void* stream);

/* kda_state_compose: the initial state of the range that follows n ranges with maps (P[i], b[i]),
 *   S_out = P[n-1] ( ... (P[0] S0 + b[0]) ... ) + b[n-1],
 * in fp32 on the device.
 *   P     : [n, H, dk, dk] fp32;  b : [n, H, dk, dv] fp32   (maps in token order)
 *   S0    : [H, dk, dv] fp32, or NULL for a zero state;  S_out : [H, dk, dv] fp32, may alias S0
 * n = 0 copies S0 (or writes zeros).  dk, dv in {64, 128}; all pointers 16-byte aligned device
 * memory (KDA_ERR_INVALID_ARG otherwise). */
kda_status kda_state_compose(const float* P, const float* b, const float* S0, float* S_out, int n, int H,
                             int dk, int dv, void* stream);

/* Synchronises `stream`, then reads and clears the current device's error word into
 * *flags (KDA_DEVERR_* bits).  Returns KDA_OK, or KDA_ERR_CUDA if the sync failed. */
kda_status kda_get_device_error(void* stream, uint32_t* flags);

/* Kernel-level timing for profilers; not needed for normal use.  While enabled, each
 * internal kernel launch made by kda_chunk_fwd / kda_decode_step is bracketed by two CUDA
 * events recorded on the call's stream (a few microseconds of host overhead per launch).
 * kda_trace_collect synchronises on those events and reports, per kernel name, the number
 * of launches and their summed device time in milliseconds since the previous collect:
 *   names    : caller buffer of max_entries * 64 bytes (NUL-terminated names)
 *   launches : [max_entries];  total_ms : [max_entries];  *n_entries : entries written
 * Both return KDA_ERR_CUDA if an event call fails.  Not thread-safe against concurrent
 * enable/disable; recording itself is serialised internally. */
kda_status kda_trace_enable(int enable);
kda_status kda_trace_collect(int max_entries, char* names, int* launches, double* total_ms,
                             int* n_entries);

/* kda_chunk_fwd for callers that cannot allocate device memory.  The method itself has
 * no counterpart to this: it is an interface variant for deployment.  Callers such as
 * code running under an allocator that owns all device memory, or hosts whose execution
 * path forbids cudaMalloc, cannot provide kda_chunk_fwd's workspace; this entry point
 * takes no workspace and allocates nothing (no cudaMalloc/cudaFree, no allocating
 * library call).  Its scratch is a fixed library-owned device array of
 * kda_noalloc_scratch_bytes() bytes (64 MiB), reserved on every device that loads the
 * library until the process exits.
 *   - Arguments, layouts, results and errors are those of kda_chunk_fwd.
 *   - Problems with kda_chunk_fwd_workspace_size(...) above the scratch size return
 *     KDA_ERR_WORKSPACE before any launch.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress);
 *     make that first call outside any stream capture.
 *   - All calls on a device share the one array and it keeps the last call's contents
 *     (nothing in it needs to start at zero).  Calls whose GPU work overlaps in time, e.g.
 *     on two unordered streams, race on it: order them. */
kda_status kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                 const float* beta, const float* h0, const int32_t* cu_seqlens,
                                 void* out, float* hT, int B, int64_t T, int H, int dk, int dv,
                                 int C, kda_dtype dtype, kda_dtype out_dtype,
                                 const kda_epilogue* epi, void* stream);

/* Size in bytes of the library-owned scratch used by kda_chunk_fwd_noalloc. */
size_t kda_noalloc_scratch_bytes(void);

/* Static, human-readable name of a status code. */
const char* kda_status_string(kda_status status);

#ifdef __cplusplus
}
#endif
#endif /* KDA_H_ */
