/*
 * gdn_oracle.c -- plain, slow, sequential fp64 reference of the gated
 * delta-net (GDN) recurrence.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this library. It shares no code, header,
 * table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * What it computes. Per sequence s and head h, starting from that sequence's
 * input state S (D_k x D_v, row i = key index, column j = value index), for
 * each token t of the sequence in order:
 *
 *   decay    S <- exp(g_t) * S                      (GDA: one gate per head)
 *            S[i,:] <- exp(g_t[i]) * S[i,:]         (KDA: one gate per row i)
 *   read     u_j = sum_i S[i,j] * k_t[i]
 *   correct  d_j = beta_t * (v_t[j] - u_j)
 *   write    S[i,j] <- S[i,j] + k_t[i] * d_j
 *   query    o_t[j] = scale * sum_i S[i,j] * q_t[i]   (the updated state)
 *   snapshot if t >= T_s - K:  slot[t - (T_s - K)] <- S   (bit copy)
 *
 * Sources. The recurrence is the gated delta rule of "Gated Delta Networks:
 * Improving Mamba2 with Delta Rule" (Yang, Kautz, Hatamizadeh, ICLR 2025),
 * i.e. the op GGML_OP_GATED_DELTA_NET of the llama.cpp commit "metal : add
 * GDN kernel (#20361)" (llama.cpp commits, tag b9752, src/models/qwen35.cpp),
 * whose two gate modes are GDA (scalar gate) and KDA (per-row gate). The
 * snapshot slots follow "metal: add GDN partial rollback" (koboldcpp commits,
 * tag v1.113.1): the input state is read once, the intermediate states of the
 * token loop go to distinct slots, and K = 1 keeps the single-slot behaviour.
 * Readings where the pages are silent: the input state is a separate buffer
 * that is never written; slot j holds the state after token T_s-K+j, so slot
 * K-1 is the final state; when T_s < K the slots j < K-T_s are left
 * untouched; the query reads the state after the write; g is a log-decay
 * applied as exp(g) with no clamp; beta is used as given (no sigmoid).
 *
 * Layouts (all dense, innermost index last, fp64):
 *   q, k   [Ntok][H][Dk]      v, out  [Ntok][H][Dv]
 *   g      [Ntok][H] (GDA) or [Ntok][H][Dk] (KDA)       beta [Ntok][H]
 *   state_in, state_out  [n_seqs][H][Dk][Dv]
 *   slots  [n_seqs][n_slots][H][Dk][Dv]
 * Sequence s covers tokens seq_start[s] .. seq_start[s]+seq_len[s]-1.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_ROLLBACK_RANGE 3

/* One (sequence, head) chain: the token loop written out step by step. */
static void run_chain(int64_t t0, int64_t T, int h, int H, int Dk, int Dv,
                      int kda, const double *q, const double *k,
                      const double *v, const double *g, const double *beta,
                      double scale, double *S, double *u, double *out,
                      int n_slots, double *slots_s /* slot 0 of this seq */) {
  const int64_t slot_stride = (int64_t)H * Dk * Dv; /* one slot, all heads */
  for (int64_t t = 0; t < T; ++t) {
    const int64_t row = (t0 + t) * H + h; /* (token, head) row index */
    const double *kt = k + row * Dk;
    const double *qt = q + row * Dk;
    const double *vt = v + row * Dv;
    const double b = beta[row];

    /* decay */
    if (kda) {
      const double *gt = g + row * Dk;
      for (int i = 0; i < Dk; ++i) {
        const double a = exp(gt[i]);
        for (int j = 0; j < Dv; ++j) S[i * Dv + j] *= a;
      }
    } else {
      const double a = exp(g[row]);
      for (int i = 0; i < Dk; ++i)
        for (int j = 0; j < Dv; ++j) S[i * Dv + j] *= a;
    }

    /* read: u = S^T k */
    for (int j = 0; j < Dv; ++j) {
      double acc = 0.0;
      for (int i = 0; i < Dk; ++i) acc += S[i * Dv + j] * kt[i];
      u[j] = acc;
    }

    /* correct: d = beta (v - u), kept in u */
    for (int j = 0; j < Dv; ++j) u[j] = b * (vt[j] - u[j]);

    /* write: S += k d^T */
    for (int i = 0; i < Dk; ++i)
      for (int j = 0; j < Dv; ++j) S[i * Dv + j] += kt[i] * u[j];

    /* query: o = scale S^T q */
    double *ot = out + row * Dv;
    for (int j = 0; j < Dv; ++j) {
      double acc = 0.0;
      for (int i = 0; i < Dk; ++i) acc += S[i * Dv + j] * qt[i];
      ot[j] = scale * acc;
    }

    /* snapshot */
    if (n_slots > 0 && slots_s != NULL && t >= T - n_slots) {
      const int64_t slot = t - (T - n_slots);
      double *dst = slots_s + slot * slot_stride + (int64_t)h * Dk * Dv;
      memcpy(dst, S, sizeof(double) * (size_t)Dk * (size_t)Dv);
    }
  }
}

/*
 * Runs the recurrence over every (sequence, head) chain. n_threads <= 0 uses
 * the OpenMP default; chains are independent, so the result does not depend
 * on the thread count. Returns ORACLE_OK or ORACLE_ERR_ARG.
 */
int gdn_oracle_forward(int n_seqs, const int64_t *seq_start,
                       const int64_t *seq_len, int H, int Dk, int Dv, int kda,
                       const double *q, const double *k, const double *v,
                       const double *g, const double *beta, double scale,
                       const double *state_in, double *out, double *state_out,
                       int n_slots, double *slots, int n_threads) {
  if (n_seqs < 0 || H <= 0 || Dk <= 0 || Dv <= 0 || n_slots < 0) return ORACLE_ERR_ARG;
  if (n_seqs > 0 && (!seq_start || !seq_len || !q || !k || !v || !g || !beta ||
                     !state_in || !out))
    return ORACLE_ERR_ARG;
  if (n_slots > 0 && !slots) return ORACLE_ERR_ARG;
  for (int s = 0; s < n_seqs; ++s)
    if (seq_len[s] < 0 || seq_start[s] < 0) return ORACLE_ERR_ARG;

  const int64_t n_chains = (int64_t)n_seqs * H;
  const int64_t state_sz = (int64_t)Dk * Dv;
  int err = 0;

#ifdef _OPENMP
  if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
#endif
  {
    double *S = (double *)malloc(sizeof(double) * (size_t)state_sz);
    double *u = (double *)malloc(sizeof(double) * (size_t)Dv);
    if (!S || !u) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      err = 1;
    }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t c = 0; c < n_chains; ++c) {
      if (!S || !u) continue;
      const int s = (int)(c / H);
      const int h = (int)(c % H);
      const double *src = state_in + ((int64_t)s * H + h) * state_sz;
      memcpy(S, src, sizeof(double) * (size_t)state_sz);
      double *slots_s =
          n_slots > 0 ? slots + (int64_t)s * n_slots * H * state_sz : NULL;
      run_chain(seq_start[s], seq_len[s], h, H, Dk, Dv, kda, q, k, v, g, beta,
                scale, S, u, out, n_slots, slots_s);
      if (state_out)
        memcpy(state_out + ((int64_t)s * H + h) * state_sz, S,
               sizeof(double) * (size_t)state_sz);
    }
    free(S);
    free(u);
  }
  return err ? ORACLE_ERR_ARG : ORACLE_OK;
}

/*
 * Which stored state holds the result of accepting the first n_accepted of
 * the T tokens of the last forward, when that forward kept K slots
 * ("llama: allow partial seq_rm for GDN models for speculative decoding",
 * koboldcpp commits, tag v1.113.1: rollback up to draft_max reads a stored
 * intermediate instead of re-running the target).
 *   n_accepted == 0            -> *slot = -1 (the input state is unchanged)
 *   token n_accepted-1 was snapshotted -> *slot = its slot index
 *   otherwise                  -> ORACLE_ERR_ROLLBACK_RANGE (must recompute)
 */
int gdn_oracle_rollback_slot(int T, int K, int n_accepted, int *slot) {
  if (!slot || T < 0 || K < 1) return ORACLE_ERR_ARG;
  if (n_accepted < 0 || n_accepted > T) return ORACLE_ERR_ROLLBACK_RANGE;
  if (n_accepted == 0) {
    *slot = -1;
    return ORACLE_OK;
  }
  /* the state after token t (0-based) sits in slot t-(T-K) when t >= T-K */
  const int t = n_accepted - 1;
  const int first_snapshotted = T - K > 0 ? T - K : 0;
  if (t < first_snapshotted) return ORACLE_ERR_ROLLBACK_RANGE;
  *slot = t - (T - K);
  return ORACLE_OK;
}

int gdn_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
