/* gdn_forward used from C with device memory: 3 sequences x 5 tokens, H=2,
 * D_k=D_v=64, fp32 inputs, GDA, 2 snapshot slots, checked against the fp64
 * oracle's C entry point (test infrastructure, linked only here). Built and
 * run by tests/test_c_abi.py on a GPU. Exit status 0 = within 1e-5 rel-L2. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "gdn.h"

int gdn_oracle_forward(int n_seqs, const int64_t *seq_start, const int64_t *seq_len, int H,
                       int Dk, int Dv, int kda, const double *q, const double *k,
                       const double *v, const double *g, const double *beta, double scale,
                       const double *state_in, double *out, double *state_out, int n_slots,
                       double *slots, int n_threads);

enum { N = 3, T = 5, H = 2, D = 64, K = 2, NTOK = N * T };

static uint64_t lcg = 12345;
static double uni(void) { /* uniform in (0, 1) */
  lcg = lcg * 6364136223846793005ull + 1442695040888963407ull;
  return ((lcg >> 11) + 0.5) / 9007199254740992.0;
}
static double gauss(void) { return sqrt(-2 * log(uni())) * cos(6.283185307179586 * uni()); }

static double rel_l2(const float *x, const double *ref, size_t n) {
  double num = 0, den = 0;
  for (size_t i = 0; i < n; ++i) {
    num += (x[i] - ref[i]) * (x[i] - ref[i]);
    den += ref[i] * ref[i];
  }
  return sqrt(num / (den > 0 ? den : 1));
}

#define CUDA_OK(x)                                                    \
  do {                                                                \
    if ((x) != cudaSuccess) {                                         \
      fprintf(stderr, "CUDA error at %s:%d\n", __FILE__, __LINE__);   \
      return 2;                                                       \
    }                                                                 \
  } while (0)

int main(void) {
  const size_t nqk = (size_t)NTOK * H * D, nst = (size_t)N * H * D * D;
  float *hq = malloc(nqk * 4), *hk = malloc(nqk * 4), *hv = malloc(nqk * 4);
  float *hg = malloc(NTOK * H * 4), *hb = malloc(NTOK * H * 4), *hs = malloc(nst * 4);
  double *dq = malloc(nqk * 8), *dk = malloc(nqk * 8), *dv = malloc(nqk * 8);
  double *dg = malloc(NTOK * H * 8), *db = malloc(NTOK * H * 8), *ds = malloc(nst * 8);
  for (size_t row = 0; row < (size_t)NTOK * H; ++row) { /* q, k unit rows */
    double nq = 0, nk = 0, tq[D], tk[D];
    for (int i = 0; i < D; ++i) {
      tq[i] = gauss(); tk[i] = gauss();
      nq += tq[i] * tq[i]; nk += tk[i] * tk[i];
    }
    for (int i = 0; i < D; ++i) {
      hq[row * D + i] = (float)(tq[i] / sqrt(nq));
      hk[row * D + i] = (float)(tk[i] / sqrt(nk));
      hv[row * D + i] = (float)gauss();
    }
    hg[row] = (float)-log(1 + exp(gauss())); /* -softplus */
    hb[row] = (float)(1 / (1 + exp(-gauss())));
  }
  for (size_t i = 0; i < nst; ++i) hs[i] = (float)(0.05 * gauss());
  for (size_t i = 0; i < nqk; ++i) { dq[i] = hq[i]; dk[i] = hk[i]; dv[i] = hv[i]; }
  for (size_t i = 0; i < (size_t)NTOK * H; ++i) { dg[i] = hg[i]; db[i] = hb[i]; }
  for (size_t i = 0; i < nst; ++i) ds[i] = hs[i];

  float *q, *k, *v, *g, *b, *st, *slots, *out;
  const float **ptrs;
  CUDA_OK(cudaMalloc((void **)&q, nqk * 4));
  CUDA_OK(cudaMalloc((void **)&k, nqk * 4));
  CUDA_OK(cudaMalloc((void **)&v, nqk * 4));
  CUDA_OK(cudaMalloc((void **)&g, NTOK * H * 4));
  CUDA_OK(cudaMalloc((void **)&b, NTOK * H * 4));
  CUDA_OK(cudaMalloc((void **)&st, nst * 4));
  CUDA_OK(cudaMalloc((void **)&slots, (size_t)N * K * H * D * D * 4));
  CUDA_OK(cudaMalloc((void **)&out, nqk * 4));
  CUDA_OK(cudaMalloc((void **)&ptrs, N * sizeof(float *)));
  CUDA_OK(cudaMemcpy(q, hq, nqk * 4, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(k, hk, nqk * 4, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(v, hv, nqk * 4, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(g, hg, NTOK * H * 4, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(b, hb, NTOK * H * 4, cudaMemcpyHostToDevice));
  CUDA_OK(cudaMemcpy(st, hs, nst * 4, cudaMemcpyHostToDevice));
  const float *hp[N];
  for (int s = 0; s < N; ++s) hp[s] = st + (size_t)s * H * D * D;
  CUDA_OK(cudaMemcpy(ptrs, hp, sizeof hp, cudaMemcpyHostToDevice));

  gdn_shape sh;
  memset(&sh, 0, sizeof sh);
  sh.n_seqs = N; sh.T = T; sh.H = H; sh.D_k = D; sh.D_v = D; sh.in_dtype = GDN_F32;
  if (gdn_forward(&sh, q, k, v, g, b, ptrs, slots, out, K, GDN_MODE_GDA, NULL) != GDN_OK ||
      gdn_check_device_error(NULL) != GDN_OK) {
    fprintf(stderr, "gdn_forward: %s\n", gdn_last_error());
    return 3;
  }
  float *ho = malloc(nqk * 4), *hsl = malloc((size_t)N * K * H * D * D * 4);
  CUDA_OK(cudaMemcpy(ho, out, nqk * 4, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(hsl, slots, (size_t)N * K * H * D * D * 4, cudaMemcpyDeviceToHost));

  int64_t start[N], len[N];
  for (int s = 0; s < N; ++s) { start[s] = (int64_t)s * T; len[s] = T; }
  double *ro = malloc(nqk * 8), *rfin = malloc(nst * 8);
  double *rsl = malloc((size_t)N * K * H * D * D * 8);
  if (gdn_oracle_forward(N, start, len, H, D, D, 0, dq, dk, dv, dg, db, 1 / sqrt((double)D),
                         ds, ro, rfin, K, rsl, 1) != 0) {
    fprintf(stderr, "oracle failed\n");
    return 4;
  }
  const double e_out = rel_l2(ho, ro, nqk);
  const double e_sl = rel_l2(hsl, rsl, (size_t)N * K * H * D * D);
  printf("out rel-L2 %.3e, slots rel-L2 %.3e\n", e_out, e_sl);
  return (e_out <= 1e-5 && e_sl <= 1e-5) ? 0 : 1;
}
