/*
 * KDA oracle: a plain, slow fp64 token-by-token evaluation of the Kimi Delta
 * Attention recurrence.  TEST INFRASTRUCTURE ONLY: nothing in the product path
 * (the CUDA library and its Python binding) may link, load or call this file.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 *
 * What it follows (Kimi K3 technical-report walk-through, kimi-k3-paper.pages.dev):
 *   - section 2.2, Eq. 1 ("decay first, then erase"): per token t
 *         S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     with beta_t scaling both the erase and the write;
 *   - section 2.3: alpha_t is a d_k-vector in (0,1), one decay per key channel,
 *     i.e. Diag(alpha_t) scales the ROWS of S (S is d_k x d_v);
 *   - section 2.4, Eq. 3: read-out o_t = S_t^T q_t (no extra scale);
 *   - section 3.3, Eq. 6: optional epilogue, head-wise RMSNorm of o_t followed by
 *     the sigmoid output gate, y = o / sqrt(mean(o^2) + eps) * w * sigmoid(gate).
 * alpha_t = exp(g_t); g is an input (section 3.2 / Eq. 5 bound it to (-5, 0)).
 *
 * Each step is written out in the order the pages give it: decay, erase, write,
 * read.  No chunking, blocking, fusion or reordering.  Sequences of a packed
 * batch are independent chains; OpenMP runs the (sequence, head) chains in
 * parallel, each chain strictly sequential over its tokens.
 *
 * Layouts (all row-major, fp64):
 *   q, k, g : [T_tot, H, dk]     v : [T_tot, H, dv]     beta : [T_tot, H]
 *   h0, hT  : [B, H, dk, dv]     out : [T_tot, H, dv]   gate : [T_tot, H, dv]
 *   norm_weight : [dv]           cu_seqlens : [B+1] token offsets
 *   state pool (decode) : [num_slots, H, dk, dv], slot_idx : [N]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Optional epilogue on one read-out vector o[dv] (in place). */
static void epilogue(double* o, const double* gate, const double* w, double eps, int dv) {
  double ms = 0.0;
  for (int j = 0; j < dv; ++j) ms += o[j] * o[j];
  ms /= (double)dv;
  const double inv_rms = 1.0 / sqrt(ms + eps);
  for (int j = 0; j < dv; ++j) {
    const double wj = w ? w[j] : 1.0;
    const double sig = 1.0 / (1.0 + exp(-gate[j]));
    o[j] = o[j] * inv_rms * wj * sig;
  }
}

/* One recurrence step on S[dk][dv] for one token of one head; writes o[dv].
 * kS is caller scratch of length dv. */
static void kda_token_step(double* S, const double* q, const double* k, const double* v,
                           const double* g, double beta, double* o, double* kS,
                           int dk, int dv) {
  /* decay: S <- Diag(alpha) S, alpha = exp(g) per key channel (row) */
  for (int i = 0; i < dk; ++i) {
    const double a = exp(g[i]);
    for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= a;
  }
  /* erase: S <- (I - beta k k^T) S  =  S - beta k (k^T S) */
  for (int j = 0; j < dv; ++j) kS[j] = 0.0;
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j) kS[j] += k[i] * S[(size_t)i * dv + j];
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] -= beta * k[i] * kS[j];
  /* write: S <- S + beta k v^T */
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += beta * k[i] * v[j];
  /* read-out: o = S^T q */
  for (int j = 0; j < dv; ++j) o[j] = 0.0;
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j) o[j] += S[(size_t)i * dv + j] * q[i];
}

/* Prefill over a packed batch.  Returns 0 on success, -1 on bad arguments.
 * h0 may be NULL (zero initial state); hT may be NULL; gate == NULL disables the
 * epilogue; norm_weight may be NULL (weight 1). */
int oracle_kda_prefill(const double* q, const double* k, const double* v, const double* g,
                       const double* beta, const double* h0, const int64_t* cu_seqlens,
                       int B, int H, int dk, int dv, const double* gate,
                       const double* norm_weight, double eps, double* out, double* hT,
                       int num_threads) {
  if (B < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return -1;
  for (int b = 0; b < B; ++b)
    if (cu_seqlens[b + 1] < cu_seqlens[b]) return -1;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#else
  (void)num_threads;
#endif
  const long nchains = (long)B * H;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (long chain = 0; chain < nchains; ++chain) {
    const int b = (int)(chain / H), h = (int)(chain % H);
    const size_t ssz = (size_t)dk * dv;
    double* S = (double*)malloc(ssz * sizeof(double));
    double* kS = (double*)malloc((size_t)dv * sizeof(double));
    if (!S || !kS) { free(S); free(kS); bad |= 1; continue; }
    if (h0) memcpy(S, h0 + ((size_t)b * H + h) * ssz, ssz * sizeof(double));
    else memset(S, 0, ssz * sizeof(double));
    for (int64_t t = cu_seqlens[b]; t < cu_seqlens[b + 1]; ++t) {
      const size_t rk = ((size_t)t * H + h) * dk, rv = ((size_t)t * H + h) * dv;
      double* o = out + rv;
      kda_token_step(S, q + rk, k + rk, v + rv, g + rk, beta[(size_t)t * H + h], o, kS, dk, dv);
      if (gate) epilogue(o, gate + rv, norm_weight, eps, dv);
    }
    if (hT) memcpy(hT + ((size_t)b * H + h) * ssz, S, ssz * sizeof(double));
    free(S);
    free(kS);
  }
  return bad ? -1 : 0;
}

/* One decode step over a pool of states, updated in place.  Rows whose slot is
 * outside [0, num_slots) are skipped (out untouched) and counted in the return
 * value (>= 0); -1 on bad arguments. */
int oracle_kda_decode(const double* q, const double* k, const double* v, const double* g,
                      const double* beta, double* state_pool, const int64_t* slot_idx,
                      int N, int H, int dk, int dv, int num_slots, const double* gate,
                      const double* norm_weight, double eps, double* out, int num_threads) {
  if (N < 0 || H <= 0 || dk <= 0 || dv <= 0 || num_slots < 0 || !slot_idx) return -1;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#else
  (void)num_threads;
#endif
  const size_t ssz = (size_t)dk * dv;
  int skipped = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : skipped)
  for (long row = 0; row < (long)N * H; ++row) {
    const int n = (int)(row / H), h = (int)(row % H);
    const int64_t slot = slot_idx[n];
    if (slot < 0 || slot >= num_slots) { if (h == 0) skipped += 1; continue; }
    double* kS = (double*)malloc((size_t)dv * sizeof(double));
    if (!kS) continue;
    double* S = state_pool + ((size_t)slot * H + h) * ssz;
    const size_t rk = ((size_t)n * H + h) * dk, rv = ((size_t)n * H + h) * dv;
    kda_token_step(S, q + rk, k + rk, v + rv, g + rk, beta[(size_t)n * H + h], out + rv, kS, dk, dv);
    if (gate) epilogue(out + rv, gate + rv, norm_weight, eps, dv);
    free(kS);
  }
  return skipped;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
