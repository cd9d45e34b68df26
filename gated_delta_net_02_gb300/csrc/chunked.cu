// chunked.cu -- chunked (chunk 64, WY/UT-transform) GDN prefill of varlen
// sequences on sm_103a tensor cores ("llama : enable chunked fused GDN path",
// llama.cpp commits, tag b9752; the chunkwise form of the delta rule of
// "Parallelizing Linear Transformers with the Delta Rule over Sequence
// Length", Yang et al., NeurIPS 2024, with the gates of "Gated Delta
// Networks", Yang, Kautz, Hatamizadeh, ICLR 2025).
//
// Within a chunk of C = 64 tokens r = 0..63 with start state S0 (D_k x D_v),
// g_r the log-gate (a scalar for GDA, a D_k-vector for KDA) and
// gamma_r = g_0 + ... + g_r:
//   A[r][j] = beta_r sum_i k_ri k_ji exp(gamma_ri - gamma_ji)   (j < r)
//   T       = (I + A)^-1 diag(beta)
//   W       = T (exp(gamma) . K)          U = T V
//   D       = U - W S0                    (row r of D is d_r of the token loop)
//   O       = scale [ (exp(gamma) . Q) S0 + P D ],
//             P[r][j] = sum_i q_ri k_ji exp(gamma_ri - gamma_ji)   (j <= r)
//   S_C     = exp(gamma_C) . S0 + (exp(gamma_C - gamma) . K)^T D
// A partial last chunk is padded with rows that have k = q = v = 0,
// beta = 0 and g = 0, which leave S unchanged.
//
// Three kernels run per call, all on the caller's stream:
//  1. worklist_kernel: validates cu_seqlens and lays out the chunks of every
//     sequence's chunked part [0, L_s - K) plus the K-token tails.
//  2. chunk_prep_kernel (one CTA per chunk and head, fully parallel):
//     G = [K; Q] K^T on the tensor cores (tcgen05, accumulator in TMEM),
//     then A and P with their decays, then T by forward substitution in
//     fp32; T and P are stored as bf16 in the workspace.
//  3. chunk_scan_kernel (one CTA per sequence and head, sequential over the
//     chunks): W^T = (e^g.K)^T T^T, then [D; Q^S0] = [-W; Q^] S0 + [T; 0] V,
//     then S = e^gC.S0 + K~^T D~ and O += [0; P] D, all on tcgen05 with the
//     fp32 master state in registers and bf16 copies as MMA operands.
// The last K tokens of each sequence then run through the recurrent kernel,
// which writes the snapshot slots.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int CH = 64;  // chunk length

// ---- workspace layout --------------------------------------------------------

struct WsLayout {
  size_t hdr, chunk_seq, chunk_tok, chunk_len, seq_chunk0, seq_nch, tail_start,
      tail_len, order, state_ptrs, states, T, P, total;
  long long max_chunks;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WsLayout ws_layout(int n_seqs, int total_tokens, int H, int Dk, int Dv) {
  WsLayout w{};
  w.max_chunks = (long long)total_tokens / CH + n_seqs;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  w.hdr = take(64);
  w.chunk_seq = take(sizeof(int) * (size_t)w.max_chunks);
  w.chunk_tok = take(sizeof(int) * (size_t)w.max_chunks);
  w.chunk_len = take(sizeof(int) * (size_t)w.max_chunks);
  w.seq_chunk0 = take(sizeof(int) * (size_t)n_seqs);
  w.seq_nch = take(sizeof(int) * (size_t)n_seqs);
  w.tail_start = take(sizeof(int) * (size_t)n_seqs);
  w.tail_len = take(sizeof(int) * (size_t)n_seqs);
  w.order = take(sizeof(int) * (size_t)n_seqs);
  w.state_ptrs = take(sizeof(float *) * (size_t)n_seqs);
  w.states = take(sizeof(float) * (size_t)n_seqs * H * Dk * Dv);
  w.T = take(2 * (size_t)w.max_chunks * H * CH * CH);
  w.P = take(2 * (size_t)w.max_chunks * H * CH * CH);
  w.total = off;
  return w;
}

struct WsPtrs {
  int *hdr, *chunk_seq, *chunk_tok, *chunk_len, *seq_chunk0, *seq_nch, *tail_start,
      *tail_len, *order;
  const float **state_ptrs;
  float *states;
  __nv_bfloat16 *T, *P;
};

WsPtrs ws_ptrs(void *base, const WsLayout &w) {
  char *b = static_cast<char *>(base);
  WsPtrs p;
  p.hdr = reinterpret_cast<int *>(b + w.hdr);
  p.chunk_seq = reinterpret_cast<int *>(b + w.chunk_seq);
  p.chunk_tok = reinterpret_cast<int *>(b + w.chunk_tok);
  p.chunk_len = reinterpret_cast<int *>(b + w.chunk_len);
  p.seq_chunk0 = reinterpret_cast<int *>(b + w.seq_chunk0);
  p.seq_nch = reinterpret_cast<int *>(b + w.seq_nch);
  p.tail_start = reinterpret_cast<int *>(b + w.tail_start);
  p.tail_len = reinterpret_cast<int *>(b + w.tail_len);
  p.order = reinterpret_cast<int *>(b + w.order);
  p.state_ptrs = reinterpret_cast<const float **>(b + w.state_ptrs);
  p.states = reinterpret_cast<float *>(b + w.states);
  p.T = reinterpret_cast<__nv_bfloat16 *>(b + w.T);
  p.P = reinterpret_cast<__nv_bfloat16 *>(b + w.P);
  return p;
}

// ---- 1. work list ---------------------------------------------------------------

constexpr int WL_THREADS = 1024;

// One block. Validates cu_seqlens (cu[0] = 0, non-decreasing, cu[N] = Ntok);
// on failure every sequence gets zero chunks and zero tail tokens, and the
// error word is set. Otherwise sequence s gets Lc_s = max(L_s - K, 0) chunked
// tokens in ceil(Lc_s / 64) chunks and a tail of L_s - Lc_s tokens, and the
// chunk scan visits sequences longest first.
__global__ void __launch_bounds__(WL_THREADS)
    worklist_kernel(const int32_t *__restrict__ cu, int N, int total, int K, int H,
                    long long state_elems, const float *const *state_in, WsPtrs w,
                    int *err) {
  __shared__ int bad;
  __shared__ int part[WL_THREADS];
  const int tid = threadIdx.x;
  if (tid == 0) bad = (cu[0] != 0 || cu[N] != total) ? 1 : 0;
  __syncthreads();
  for (int s = tid; s < N; s += WL_THREADS)
    if (cu[s + 1] < cu[s]) bad = 1;
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      set_error(err, kDevBadSeqlens);
      w.hdr[0] = 0;
    }
    for (int s = tid; s < N; s += WL_THREADS) {
      w.seq_nch[s] = 0;
      w.seq_chunk0[s] = 0;
      w.tail_len[s] = 0;
      w.tail_start[s] = 0;
      w.order[s] = s;
      w.state_ptrs[s] = nullptr;
    }
    return;
  }
  // per-thread contiguous segment of sequences, then a block scan of counts
  const int per = (N + WL_THREADS - 1) / WL_THREADS;
  const int s0 = min(N, tid * per), s1 = min(N, s0 + per);
  int cnt = 0;
  for (int s = s0; s < s1; ++s) {
    const int L = cu[s + 1] - cu[s];
    const int Lc = max(L - K, 0);
    cnt += (Lc + CH - 1) / CH;
  }
  part[tid] = cnt;
  __syncthreads();
  for (int off = 1; off < WL_THREADS; off <<= 1) {  // Hillis-Steele inclusive scan
    const int v = tid >= off ? part[tid - off] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int base = part[tid] - cnt;
  for (int s = s0; s < s1; ++s) {
    const int L = cu[s + 1] - cu[s];
    const int Lc = max(L - K, 0);
    const int nch = (Lc + CH - 1) / CH;
    w.seq_chunk0[s] = base;
    w.seq_nch[s] = nch;
    w.tail_start[s] = cu[s] + Lc;
    w.tail_len[s] = L - Lc;
    w.state_ptrs[s] = nch > 0 ? w.states + (long long)s * state_elems : state_in[s];
    for (int j = 0; j < nch; ++j) {
      w.chunk_seq[base + j] = s;
      w.chunk_tok[base + j] = cu[s] + j * CH;
      w.chunk_len[base + j] = min(CH, Lc - j * CH);
    }
    base += nch;
  }
  if (tid == WL_THREADS - 1) w.hdr[0] = part[WL_THREADS - 1];
  // longest chunk count first (ties by index); identity beyond 4096 sequences
  for (int s = tid; s < N; s += WL_THREADS) {
    if (N > 4096) {
      w.order[s] = s;
      continue;
    }
    const int L = cu[s + 1] - cu[s];
    const int ns = (max(L - K, 0) + CH - 1) / CH;
    int rank = 0;
    for (int t = 0; t < N; ++t) {
      const int Lt = cu[t + 1] - cu[t];
      const int nt = (max(Lt - K, 0) + CH - 1) / CH;
      rank += (nt > ns) || (nt == ns && t < s);
    }
    w.order[rank] = s;
  }
}

// ---- 2. chunk preparation: T = (I + A)^-1 diag(beta) and P ------------------

constexpr int PREP_THREADS = 128;
constexpr int AF_LD = 68;  // fp32 row stride of A in shared memory (16-byte rows)
// shared memory: KQ [128 x 128] bf16 (2 swizzled atom columns of 16 KB),
// KB [64 x 128] bf16 (KDA B operand), A fp32 [64][AF_LD], gamma, beta, barrier
constexpr int PREP_KQ = 0, PREP_KB = 32768, PREP_AF = 49152;
constexpr int PREP_GAM = PREP_AF + 64 * AF_LD * 4, PREP_BETA = PREP_GAM + 256;
constexpr int PREP_BAR = PREP_BETA + 256, PREP_TSLOT = PREP_BAR + 8;
constexpr int PREP_SMEM = PREP_TSLOT + 8 + 1024;  // + alignment slack

__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
  return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
}

// One CTA per (chunk, head). Rows r of the chunk are tokens chunk_tok + r,
// r < len; the rest are padding (k = q = 0, beta = 0, g = 0).
template <bool KDA>
__global__ void __launch_bounds__(PREP_THREADS)
    chunk_prep_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                      const float *__restrict__ g, const float *__restrict__ beta, int H,
                      WsPtrs w, int *err) {
  constexpr int DK = 128;
  const int c = blockIdx.x / H, h = blockIdx.x % H;
  if (c >= w.hdr[0]) return;
  const int t0 = w.chunk_tok[c], len = w.chunk_len[c];
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = align1024(smem_raw);
  unsigned char *KQ = sm + PREP_KQ, *KB = sm + PREP_KB;
  float *Af = reinterpret_cast<float *>(sm + PREP_AF);
  float *sgam = reinterpret_cast<float *>(sm + PREP_GAM);
  float *sbeta = reinterpret_cast<float *>(sm + PREP_BETA);
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + PREP_BAR);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + PREP_TSLOT);
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid < CH) {
    const long long row = (long long)(t0 + tid) * H + h;
    sbeta[tid] = tid < len ? beta[row] : 0.f;
    if constexpr (!KDA) sgam[tid] = tid < len ? g[row] : 0.f;
  }
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if constexpr (!KDA) {
    if (tid == 0) {  // inclusive cumulative gate of the chunk
      float acc = 0.f;
      for (int r = 0; r < CH; ++r) {
        acc += sgam[r];
        sgam[r] = acc;
      }
    }
  }
  // Operand tiles: thread i fills column i of every row.
  {
    const int i = tid;
    const uint32_t aoff = (uint32_t)(i >> 6) * 16384u, boff = (uint32_t)(i >> 6) * 8192u;
    const __nv_bfloat16 zero = __float2bfloat16(0.f);
    if constexpr (KDA) {
      // decays are split around the middle row so that each factor stays
      // within exp(+-half the chunk's cumulative decay)
      float gref = 0.f;
      for (int r = 0; r < CH / 2; ++r)
        if (r < len) gref += g[((long long)(t0 + r) * H + h) * DK + i];
      float gam = 0.f;
      for (int r = 0; r < CH; ++r) {
        const long long row = (long long)(t0 + r) * H + h;
        __nv_bfloat16 kq = zero, qq = zero, kb = zero;
        if (r < len) {
          gam += g[row * DK + i];
          const float e1 = expf(gam - gref), e2 = expf(gref - gam);
          const float kv = __bfloat162float(k[row * DK + i]);
          const float qv = __bfloat162float(q[row * DK + i]);
          kq = __float2bfloat16(kv * e1);
          qq = __float2bfloat16(qv * e1);
          kb = __float2bfloat16(kv * e2);
        }
        *reinterpret_cast<__nv_bfloat16 *>(KQ + aoff + sw128_offset(r, i & 63)) = kq;
        *reinterpret_cast<__nv_bfloat16 *>(KQ + aoff + sw128_offset(CH + r, i & 63)) = qq;
        *reinterpret_cast<__nv_bfloat16 *>(KB + boff + sw128_offset(r, i & 63)) = kb;
      }
    } else {
      for (int r = 0; r < CH; ++r) {
        const long long row = (long long)(t0 + r) * H + h;
        const __nv_bfloat16 kv = r < len ? k[row * DK + i] : zero;
        const __nv_bfloat16 qv = r < len ? q[row * DK + i] : zero;
        *reinterpret_cast<__nv_bfloat16 *>(KQ + aoff + sw128_offset(r, i & 63)) = kv;
        *reinterpret_cast<__nv_bfloat16 *>(KQ + aoff + sw128_offset(CH + r, i & 63)) = qv;
      }
    }
  }
  fence_proxy_async();
  if (warp == 0) {
    tmem_alloc(tslot, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  // G = [K'; Q'] K''^T : M = 128, N = 64, K = 128 (8 steps of 16)
  if (tid == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
    const uint32_t a0 = smem_u32(KQ);
    const uint32_t b0 = KDA ? smem_u32(KB) : smem_u32(KQ);
    const uint32_t bcol = KDA ? 8192u : 16384u;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint64_t ad = sdesc_kmajor(a0 + (s >> 2) * 16384u + (s & 3) * 32u);
      const uint64_t bd = sdesc_kmajor(b0 + (s >> 2) * bcol + (s & 3) * 32u);
      umma_bf16(tbase, ad, bd, idesc, s > 0);
    }
    umma_commit(bar);
    if (!mbar_wait(bar, 0, err)) abort_flag = 1;
  }
  __syncthreads();
  tc_fence_after();
  if (!abort_flag) {
    // thread = accumulator row: rows 0..63 give A, rows 64..127 give P
    float G[CH];
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      float v[16];
      tmem_ld16(tbase + ((uint32_t)(32 * warp) << 16) + 16 * cc, v);
#pragma unroll
      for (int e = 0; e < 16; ++e) G[16 * cc + e] = v[e];
    }
    if (tid < CH) {
      const int r = tid;
      const float br = sbeta[r];
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        float a = 0.f;
        if (j < r) {
          a = br * G[j];
          if constexpr (!KDA) a *= expf(sgam[r] - sgam[j]);
        }
        Af[r * AF_LD + j] = a;
      }
    } else {
      const int r = tid - CH;
      uint32_t packed[CH / 2];
#pragma unroll
      for (int j = 0; j < CH; j += 2) {
        float p0 = 0.f, p1 = 0.f;
        if (r < len) {
          if (j <= r) {
            p0 = G[j];
            if constexpr (!KDA) p0 *= expf(sgam[r] - sgam[j]);
          }
          if (j + 1 <= r) {
            p1 = G[j + 1];
            if constexpr (!KDA) p1 *= expf(sgam[r] - sgam[j + 1]);
          }
        }
        packed[j / 2] = pack_bf16(p0, p1);
      }
      uint4 *dst = reinterpret_cast<uint4 *>(w.P + (((long long)c * H + h) * CH + r) * CH);
#pragma unroll
      for (int e = 0; e < CH / 8; ++e)
        dst[e] = make_uint4(packed[4 * e], packed[4 * e + 1], packed[4 * e + 2],
                            packed[4 * e + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 64);
  if (abort_flag) return;

  // T = (I + A)^-1 diag(beta): thread j solves column j by forward
  // substitution, x_r = [r == j] - sum_{m < r} A[r][m] x_m, in fp32.
  if (tid < CH) {
    const int j = tid;
    float x[CH];
#pragma unroll
    for (int r = 0; r < CH; ++r) x[r] = 0.f;
#pragma unroll
    for (int r = 0; r < CH; ++r) {
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
      const float4 *row = reinterpret_cast<const float4 *>(Af + r * AF_LD);
#pragma unroll
      for (int m4 = 0; m4 < (r + 3) / 4; ++m4) {
        const float4 av = row[m4];
        a0 = fmaf(av.x, x[4 * m4 + 0], a0);
        a1 = fmaf(av.y, x[4 * m4 + 1], a1);
        a2 = fmaf(av.z, x[4 * m4 + 2], a2);
        a3 = fmaf(av.w, x[4 * m4 + 3], a3);
      }
      x[r] = (r == j ? 1.f : 0.f) - ((a0 + a1) + (a2 + a3));
    }
    const float bj = sbeta[j];
    __nv_bfloat16 *dst = w.T + ((long long)c * H + h) * CH * CH + j;
#pragma unroll
    for (int r = 0; r < CH; ++r) dst[r * CH] = __float2bfloat16(x[r] * bj);
  }
}

// ---- 3. chunk scan ---------------------------------------------------------------

constexpr int SCAN_THREADS = 256;
// Shared-memory tiles (offsets from a 1024-aligned base). Every tile is made
// of 128-byte swizzled rows; "rows x cols" below, cols split into 64-wide
// atom columns stored one after the other.
constexpr int SC_S = 0;          // S0 bf16 [128 i][128 v]   (B of X, MN-major)
constexpr int SC_KQ = 32768;     // [K; Q] bf16 [128][128 i] (TMA; K is A of the S update)
constexpr int SC_V = 65536;      // V bf16 [64 j][128 v]     (TMA; B of X, MN-major)
constexpr int SC_TZP = 81920;    // T [64 r][64 j] | zeros [64][64] | P [64 r][64 j]
constexpr int SC_KH = 106496;    // K^ = e^gamma . K [64 j][128 i] (A of W^T, MN-major)
constexpr int SC_WQ = 122880;    // [-W; Q^] bf16 [128][128 i] (A of X, K-major)
constexpr int SC_D = 155648;     // D bf16 [64 r][128 v]     (B of the O update)
constexpr int SC_DT = 172032;    // D~ = e^(gC-gamma) . D    (B of the S update, GDA)
constexpr int SC_KT = 188416;    // K~ = e^(gC-gamma) . K    (A of the S update, KDA)
constexpr int SC_SMALL = 204800; // gate scalars, barriers, TMEM address
constexpr int SC_GAM = SC_SMALL;              // 64 f32: gamma_r (GDA)
constexpr int SC_EG = SC_GAM + 256;           // 64 f32: exp(gamma_r) (GDA)
constexpr int SC_EDC = SC_EG + 256;           // 64 f32: exp(gamma_C - gamma_r) (GDA)
constexpr int SC_GC = SC_EDC + 256;           // 128 f32: exp(gamma_C,i)
constexpr int SC_BAR = SC_GC + 512;           // 2 mbarriers
constexpr int SC_TSLOT = SC_BAR + 16;
constexpr int SCAN_SMEM = SC_TSLOT + 16 + 1024;  // + alignment slack
constexpr int SC_GAMK = SC_D;    // KDA gamma f32 [64][128] aliases D and D~ (dead then)
constexpr uint32_t COL_W = 0, COL_X = 64, COL_S = 192;  // TMEM columns (512 allocated)

struct ScanMaps {
  CUtensorMap q, k, v, T, P;
};

__device__ __forceinline__ uint32_t chunk16(int row, int cj) {
  return (uint32_t)(row * 128 + ((cj ^ (row & 7)) << 4));
}

// One CTA per (sequence, head): all chunks of the sequence in order.
template <bool KDA>
__global__ void __launch_bounds__(SCAN_THREADS, 1)
    chunk_scan_kernel(const __grid_constant__ CUtensorMap map_q,
                      const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v,
                      const __grid_constant__ CUtensorMap map_T,
                      const __grid_constant__ CUtensorMap map_P, const float *__restrict__ g,
                      const float *const *state_in, float *__restrict__ out, int H,
                      float scale, WsPtrs w, int *err) {
  constexpr int DK = 128, DV = 128;
  const int s = w.order[blockIdx.x / H];
  const int h = blockIdx.x % H;
  const int nch = w.seq_nch[s];
  if (nch == 0) return;
  const int chunk0 = w.seq_chunk0[s];

  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = align1024(smem_raw);
  float *sgam = reinterpret_cast<float *>(sm + SC_GAM);
  float *seg = reinterpret_cast<float *>(sm + SC_EG);
  float *sedc = reinterpret_cast<float *>(sm + SC_EDC);
  float *sgc = reinterpret_cast<float *>(sm + SC_GC);
  float *sgamk = reinterpret_cast<float *>(sm + SC_GAMK);
  uint64_t *bar_tma = reinterpret_cast<uint64_t *>(sm + SC_BAR);
  uint64_t *bar_mma = bar_tma + 1;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + SC_TSLOT);
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3, hv = warp >> 2;
  const int row = 32 * qd + lane;  // TMEM lane this thread reads
  const uint32_t lane_off = (uint32_t)(32 * qd) << 16;

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
    prefetch_tmap(&map_q);
    prefetch_tmap(&map_k);
    prefetch_tmap(&map_v);
    prefetch_tmap(&map_T);
    prefetch_tmap(&map_P);
  }
  // zero tile between T and P (rows 64..127 of the [T; 0] operand and rows
  // 0..63 of the [0; P] operand)
  for (int e = tid; e < 8192 / 16; e += SCAN_THREADS)
    reinterpret_cast<uint4 *>(sm + SC_TZP + 8192)[e] = make_uint4(0, 0, 0, 0);

  // fp32 master state: this thread owns S[row][64 hv .. 64 hv + 63]
  float Sm[64];
  {
    const float *src = state_in[s];
    if (src) {
      const float4 *p4 =
          reinterpret_cast<const float4 *>(src + ((long long)h * DK + row) * DV + 64 * hv);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float4 v4 = p4[e];
        Sm[4 * e] = v4.x; Sm[4 * e + 1] = v4.y; Sm[4 * e + 2] = v4.z; Sm[4 * e + 3] = v4.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 64; ++e) Sm[e] = 0.f;
    }
    unsigned char *st = sm + SC_S + hv * 16384;
#pragma unroll
    for (int cj = 0; cj < 8; ++cj) {
      uint4 u;
      u.x = pack_bf16(Sm[8 * cj], Sm[8 * cj + 1]);
      u.y = pack_bf16(Sm[8 * cj + 2], Sm[8 * cj + 3]);
      u.z = pack_bf16(Sm[8 * cj + 4], Sm[8 * cj + 5]);
      u.w = pack_bf16(Sm[8 * cj + 6], Sm[8 * cj + 7]);
      *reinterpret_cast<uint4 *>(st + chunk16(row, cj)) = u;
    }
  }
  fence_proxy_async();
  if (warp == 0) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  uint32_t mma_phase = 0;

  // single waiter, then a block barrier that publishes the outcome
  auto wait_mma = [&]() {
    if (tid == 0 && !mbar_wait(bar_mma, mma_phase, err)) abort_flag = 1;
    mma_phase ^= 1;
    __syncthreads();
    tc_fence_after();
  };

  for (int jc = 0; jc < nch && !abort_flag; ++jc) {
    const int gc = chunk0 + jc;
    const int t0 = w.chunk_tok[gc], len = w.chunk_len[gc];
    // B0: TMA loads of K, Q, V, T, P
    if (tid == 0) {
      mbar_arrive_expect_tx(bar_tma, 65536);
      tma_load_3d(sm + SC_KQ, &map_k, 0, h, t0, bar_tma);
      tma_load_3d(sm + SC_KQ + 16384, &map_k, 64, h, t0, bar_tma);
      tma_load_3d(sm + SC_KQ + 8192, &map_q, 0, h, t0, bar_tma);
      tma_load_3d(sm + SC_KQ + 16384 + 8192, &map_q, 64, h, t0, bar_tma);
      tma_load_3d(sm + SC_V, &map_v, 0, h, t0, bar_tma);
      tma_load_3d(sm + SC_V + 8192, &map_v, 64, h, t0, bar_tma);
      const int trow = (gc * H + h) * CH;
      tma_load_2d(sm + SC_TZP, &map_T, 0, trow, bar_tma);
      tma_load_2d(sm + SC_TZP + 16384, &map_P, 0, trow, bar_tma);
    }
    // cumulative gates of the chunk (padding rows have g = 0)
    if constexpr (KDA) {
      if (tid < DK) {
        const int i = tid;
        float gam = 0.f;
        for (int r = 0; r < CH; ++r) {
          if (r < len) gam += g[((long long)(t0 + r) * H + h) * DK + i];
          sgamk[r * DK + i] = gam;
        }
        sgc[i] = expf(gam);
      }
    } else {
      if (tid < CH) sgam[tid] = tid < len ? g[(long long)(t0 + tid) * H + h] : 0.f;
    }
    __syncthreads();
    if constexpr (!KDA) {
      if (tid == 0) {
        float acc = 0.f;
        for (int r = 0; r < CH; ++r) {
          acc += sgam[r];
          sgam[r] = acc;
        }
        sgc[0] = expf(acc);
      }
      __syncthreads();
      if (tid < CH) {
        seg[tid] = expf(sgam[tid]);
        sedc[tid] = expf(sgam[CH - 1] - sgam[tid]);
      }
    }
    if (tid == 0 && !mbar_wait(bar_tma, jc & 1, err)) abort_flag = 1;
    __syncthreads();
    if (abort_flag) break;

    // B1: padding rows of K, Q, V are zero
    if (len < CH) {
      const int nz = (CH - len) * 8;  // 16-byte chunks per 64-wide atom row set
      for (int e = tid; e < nz * 2; e += SCAN_THREADS) {
        const int a = e / nz, rem = e % nz;
        const int r = len + rem / 8, cj = rem % 8;
        const uint4 z = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(sm + SC_KQ + a * 16384 + r * 128 + cj * 16) = z;
        *reinterpret_cast<uint4 *>(sm + SC_KQ + a * 16384 + (CH + r) * 128 + cj * 16) = z;
        *reinterpret_cast<uint4 *>(sm + SC_V + a * 8192 + r * 128 + cj * 16) = z;
      }
      __syncthreads();
    }
    // B2: K^ = e^gamma . K, Q^ = e^gamma . Q (into WQ rows 64..127), K~ (KDA)
    for (int e = tid; e < CH * 16; e += SCAN_THREADS) {
      const int r = e >> 4, cc = e & 15, a = cc >> 3, cj = cc & 7;
      const uint32_t o = chunk16(r, cj);
      const uint4 ku = *reinterpret_cast<const uint4 *>(sm + SC_KQ + a * 16384 + o);
      const uint4 qu = *reinterpret_cast<const uint4 *>(sm + SC_KQ + a * 16384 + CH * 128 + o);
      const __nv_bfloat16 *kb = reinterpret_cast<const __nv_bfloat16 *>(&ku);
      const __nv_bfloat16 *qb = reinterpret_cast<const __nv_bfloat16 *>(&qu);
      float kh[8], qh[8], kt[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const float kv = __bfloat162float(kb[x]), qv = __bfloat162float(qb[x]);
        if constexpr (KDA) {
          const int i = a * 64 + cj * 8 + x;
          const float gm = sgamk[r * DK + i];
          const float eg = expf(gm);
          kh[x] = kv * eg;
          qh[x] = qv * eg;
          kt[x] = kv * expf(sgamk[(CH - 1) * DK + i] - gm);
        } else {
          kh[x] = kv * seg[r];
          qh[x] = qv * seg[r];
          kt[x] = 0.f;
        }
      }
      uint4 o1, o2;
      o1.x = pack_bf16(kh[0], kh[1]); o1.y = pack_bf16(kh[2], kh[3]);
      o1.z = pack_bf16(kh[4], kh[5]); o1.w = pack_bf16(kh[6], kh[7]);
      o2.x = pack_bf16(qh[0], qh[1]); o2.y = pack_bf16(qh[2], qh[3]);
      o2.z = pack_bf16(qh[4], qh[5]); o2.w = pack_bf16(qh[6], qh[7]);
      *reinterpret_cast<uint4 *>(sm + SC_KH + a * 8192 + o) = o1;
      *reinterpret_cast<uint4 *>(sm + SC_WQ + a * 16384 + CH * 128 + o) = o2;
      if constexpr (KDA) {
        uint4 o3;
        o3.x = pack_bf16(kt[0], kt[1]); o3.y = pack_bf16(kt[2], kt[3]);
        o3.z = pack_bf16(kt[4], kt[5]); o3.w = pack_bf16(kt[6], kt[7]);
        *reinterpret_cast<uint4 *>(sm + SC_KT + a * 8192 + o) = o3;
      }
    }
    fence_proxy_async();
    __syncthreads();

    // B3: W^T = K^^T T^T  (M = i 128, N = r 64, K = j 64)
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16_f32(128, 64, true, false);
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        const uint64_t ad = sdesc_mnmajor(smem_u32(sm + SC_KH) + st * 2048, 8192);
        const uint64_t bd = sdesc_kmajor(smem_u32(sm + SC_TZP) + st * 32);
        umma_bf16(tbase + COL_W, ad, bd, idesc, st > 0);
      }
      umma_commit(bar_mma);
    }
    wait_mma();
    if (abort_flag) break;
    // B4: -W (rows r) into WQ rows 0..63, column i = row
    {
      float wv[32];
      float t16[16];
      tmem_ld16(tbase + lane_off + COL_W + 32 * hv, t16);
#pragma unroll
      for (int x = 0; x < 16; ++x) wv[x] = t16[x];
      tmem_ld16(tbase + lane_off + COL_W + 32 * hv + 16, t16);
#pragma unroll
      for (int x = 0; x < 16; ++x) wv[16 + x] = t16[x];
      const int i = row;
      unsigned char *base = sm + SC_WQ + (i >> 6) * 16384;
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        const int r = 32 * hv + x;
        *reinterpret_cast<__nv_bfloat16 *>(base + sw128_offset(r, i & 63)) =
            __float2bfloat16(-wv[x]);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // B5: X = [-W; Q^] S0 + [T; 0] V  (M = 128, N = 128, K = 128 + 64)
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
      for (int st = 0; st < 8; ++st) {
        const uint64_t ad =
            sdesc_kmajor(smem_u32(sm + SC_WQ) + (st >> 2) * 16384 + (st & 3) * 32);
        const uint64_t bd = sdesc_mnmajor(smem_u32(sm + SC_S) + st * 2048, 16384);
        umma_bf16(tbase + COL_X, ad, bd, idesc_s, st > 0);
      }
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        const uint64_t ad = sdesc_kmajor(smem_u32(sm + SC_TZP) + st * 32);
        const uint64_t bd = sdesc_mnmajor(smem_u32(sm + SC_V) + st * 2048, 8192);
        umma_bf16(tbase + COL_X, ad, bd, idesc_s, true);
      }
      umma_commit(bar_mma);
    }
    wait_mma();
    if (abort_flag) break;
    // B6: D rows (TMEM lanes 0..63) -> D and D~ tiles
    if (qd < 2) {
      const int r = row;
      float dv[64];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float t16[16];
        tmem_ld16(tbase + lane_off + COL_X + 64 * hv + 16 * cc, t16);
#pragma unroll
        for (int x = 0; x < 16; ++x) dv[16 * cc + x] = t16[x];
      }
      unsigned char *dbase = sm + SC_D + hv * 8192;
      unsigned char *tbase_d = sm + SC_DT + hv * 8192;
      const float dec = KDA ? 1.f : sedc[r];
#pragma unroll
      for (int cj = 0; cj < 8; ++cj) {
        uint4 u;
        u.x = pack_bf16(dv[8 * cj], dv[8 * cj + 1]);
        u.y = pack_bf16(dv[8 * cj + 2], dv[8 * cj + 3]);
        u.z = pack_bf16(dv[8 * cj + 4], dv[8 * cj + 5]);
        u.w = pack_bf16(dv[8 * cj + 6], dv[8 * cj + 7]);
        *reinterpret_cast<uint4 *>(dbase + chunk16(r, cj)) = u;
        if constexpr (!KDA) {
          uint4 t;
          t.x = pack_bf16(dv[8 * cj] * dec, dv[8 * cj + 1] * dec);
          t.y = pack_bf16(dv[8 * cj + 2] * dec, dv[8 * cj + 3] * dec);
          t.z = pack_bf16(dv[8 * cj + 4] * dec, dv[8 * cj + 5] * dec);
          t.w = pack_bf16(dv[8 * cj + 6] * dec, dv[8 * cj + 7] * dec);
          *reinterpret_cast<uint4 *>(tbase_d + chunk16(r, cj)) = t;
        }
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // B7: S_acc = K~^T D~ (M = i, N = v, K = r); X += [0; P] D (K = r')
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idesc_u = idesc_bf16_f32(128, 128, true, true);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, 128, false, true);
      const uint32_t a_s = KDA ? smem_u32(sm + SC_KT) : smem_u32(sm + SC_KQ);
      const uint32_t a_lbo = KDA ? 8192u : 16384u;
      const uint32_t b_s = KDA ? smem_u32(sm + SC_D) : smem_u32(sm + SC_DT);
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        const uint64_t ad = sdesc_mnmajor(a_s + st * 2048, a_lbo);
        const uint64_t bd = sdesc_mnmajor(b_s + st * 2048, 8192);
        umma_bf16(tbase + COL_S, ad, bd, idesc_u, st > 0);
      }
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        const uint64_t ad = sdesc_kmajor(smem_u32(sm + SC_TZP) + 8192 + st * 32);
        const uint64_t bd = sdesc_mnmajor(smem_u32(sm + SC_D) + st * 2048, 8192);
        umma_bf16(tbase + COL_X, ad, bd, idesc_o, true);
      }
      umma_commit(bar_mma);
    }
    wait_mma();
    if (abort_flag) break;
    // B8: S = e^gC . S + S_acc (fp32 master, bf16 operand copy); O rows out
    {
      const float gcs = KDA ? sgc[row] : sgc[0];
      unsigned char *st = sm + SC_S + hv * 16384;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float t16[16];
        tmem_ld16(tbase + lane_off + COL_S + 64 * hv + 16 * cc, t16);
#pragma unroll
        for (int x = 0; x < 16; ++x) Sm[16 * cc + x] = fmaf(gcs, Sm[16 * cc + x], t16[x]);
      }
#pragma unroll
      for (int cj = 0; cj < 8; ++cj) {
        uint4 u;
        u.x = pack_bf16(Sm[8 * cj], Sm[8 * cj + 1]);
        u.y = pack_bf16(Sm[8 * cj + 2], Sm[8 * cj + 3]);
        u.z = pack_bf16(Sm[8 * cj + 4], Sm[8 * cj + 5]);
        u.w = pack_bf16(Sm[8 * cj + 6], Sm[8 * cj + 7]);
        *reinterpret_cast<uint4 *>(st + chunk16(row, cj)) = u;
      }
      if (qd >= 2) {
        const int r = row - CH;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          float t16[16];
          tmem_ld16(tbase + lane_off + COL_X + 64 * hv + 16 * cc, t16);
          if (r < len) {
            float4 *dst = reinterpret_cast<float4 *>(
                out + ((long long)(t0 + r) * H + h) * DV + 64 * hv + 16 * cc);
#pragma unroll
            for (int x = 0; x < 4; ++x)
              dst[x] = make_float4(scale * t16[4 * x], scale * t16[4 * x + 1],
                                   scale * t16[4 * x + 2], scale * t16[4 * x + 3]);
          }
        }
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
  }

  if (!abort_flag) {  // state after the chunked part, read by the tail
    float4 *dst = reinterpret_cast<float4 *>(
        w.states + (((long long)s * H + h) * DK + row) * DV + 64 * hv);
#pragma unroll
    for (int e = 0; e < 16; ++e)
      dst[e] = make_float4(Sm[4 * e], Sm[4 * e + 1], Sm[4 * e + 2], Sm[4 * e + 3]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

}  // namespace
}  // namespace gdn

// ---- host side ------------------------------------------------------------------

namespace gdn {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 [Ntok][H][D] viewed as (D, H, Ntok); 64 x 1 x 64 boxes, 128-byte swizzle
bool map_tokens(CUtensorMap *m, const void *base, int ntok, int H, int D) {
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)ntok};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  const cuuint32_t box[3] = {64, 1, 64}, es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [rows][64]; 64 x 64 boxes, 128-byte swizzle
bool map_rows64(CUtensorMap *m, const void *base, long long rows) {
  const cuuint64_t dims[2] = {64, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {64, 64}, es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Opt-in shared-memory sizes, once per device.
std::mutex g_attr_mu;
bool g_attr_done[64] = {};

cudaError_t set_attributes() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (dev >= 0 && dev < 64 && g_attr_done[dev]) return cudaSuccess;
  const void *fns[] = {(const void *)chunk_prep_kernel<false>,
                       (const void *)chunk_prep_kernel<true>};
  for (const void *f : fns) {
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, PREP_SMEM);
    if (e != cudaSuccess) return e;
  }
  const void *sfns[] = {(const void *)chunk_scan_kernel<false>,
                        (const void *)chunk_scan_kernel<true>};
  for (const void *f : sfns) {
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SCAN_SMEM);
    if (e != cudaSuccess) return e;
  }
  if (dev >= 0 && dev < 64) g_attr_done[dev] = true;
  return cudaSuccess;
}

}  // namespace

size_t chunked_workspace_size(int n_seqs, int total_tokens, int H, int Dk, int Dv, int) {
  return ws_layout(n_seqs, total_tokens, H, Dk, Dv).total;
}

cudaError_t launch_chunked(const ChunkedArgs &a, cudaStream_t stream) {
  if (a.Dk != 128 || a.Dv != 128) return cudaErrorInvalidValue;
  if (!encode_fn()) return cudaErrorNotSupported;
  cudaError_t e = set_attributes();
  if (e != cudaSuccess) return e;
  const WsLayout lay = ws_layout(a.n_seqs, a.total_tokens, a.H, a.Dk, a.Dv);
  if (a.workspace_bytes < lay.total) return cudaErrorInvalidValue;
  const WsPtrs w = ws_ptrs(a.workspace, lay);
  const long long state_elems = (long long)a.H * a.Dk * a.Dv;

  worklist_kernel<<<1, WL_THREADS, 0, stream>>>(a.cu_seqlens, a.n_seqs, a.total_tokens,
                                                a.n_slots, a.H, state_elems, a.state_in, w,
                                                a.err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  if (a.total_tokens > 0) {
    const long long prep_grid = lay.max_chunks * a.H;
    const auto *q = static_cast<const __nv_bfloat16 *>(a.q);
    const auto *k = static_cast<const __nv_bfloat16 *>(a.k);
    if (a.kda)
      chunk_prep_kernel<true><<<(unsigned)prep_grid, PREP_THREADS, PREP_SMEM, stream>>>(
          q, k, a.g, a.beta, a.H, w, a.err);
    else
      chunk_prep_kernel<false><<<(unsigned)prep_grid, PREP_THREADS, PREP_SMEM, stream>>>(
          q, k, a.g, a.beta, a.H, w, a.err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    CUtensorMap mq, mk, mv, mT, mP;
    const long long trows = lay.max_chunks * a.H * CH;
    if (!map_tokens(&mq, a.q, a.total_tokens, a.H, a.Dk) ||
        !map_tokens(&mk, a.k, a.total_tokens, a.H, a.Dk) ||
        !map_tokens(&mv, a.v, a.total_tokens, a.H, a.Dv) || !map_rows64(&mT, w.T, trows) ||
        !map_rows64(&mP, w.P, trows))
      return cudaErrorInvalidValue;
    const unsigned scan_grid = (unsigned)((long long)a.n_seqs * a.H);
    if (a.kda)
      chunk_scan_kernel<true><<<scan_grid, SCAN_THREADS, SCAN_SMEM, stream>>>(
          mq, mk, mv, mT, mP, a.g, a.state_in, a.out, a.H, a.scale, w, a.err);
    else
      chunk_scan_kernel<false><<<scan_grid, SCAN_THREADS, SCAN_SMEM, stream>>>(
          mq, mk, mv, mT, mP, a.g, a.state_in, a.out, a.H, a.scale, w, a.err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }

  // the last n_slots tokens of every sequence: token loop with snapshots
  RecurrentArgs r{};
  r.q = a.q; r.k = a.k; r.v = a.v; r.g = a.g; r.beta = a.beta;
  r.state_in = w.state_ptrs;
  r.slots = a.slots; r.out = a.out;
  r.tok_start = w.tail_start; r.seq_len = w.tail_len;
  r.n_seqs = a.n_seqs; r.T = 0; r.H = a.H; r.Dk = a.Dk; r.Dv = a.Dv;
  r.n_slots = a.n_slots; r.kda = a.kda; r.bf16 = true; r.scale = a.scale; r.err = a.err;
  return launch_recurrent(r, stream);
}

}  // namespace gdn

// ---- allocation-free variant (gdn_forward_chunked_noalloc) -----------------------
//
// Some callers cannot hand this library a workspace: code that runs inside a
// host application which owns all device memory through its own pool, or
// latency-critical loops where a cudaMalloc (which may synchronise the whole
// device) is not acceptable. For them the chunked path can run from a fixed
// scratch area compiled into the library. It is a plain device array, so
// every GPU that loads this library's chunked kernels keeps it (64 MiB)
// until the process exits.
namespace gdn {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {
std::mutex g_scratch_mu;
void *g_scratch_addr[64] = {};
}  // namespace

size_t static_scratch_bytes() { return kStaticScratchBytes; }

// *need = workspace bytes this shape needs. Returns cudaErrorInvalidValue
// (and launches nothing) when *need exceeds the static area. The first call
// on a device looks up the area's device address with that device current.
cudaError_t launch_chunked_static(ChunkedArgs a, cudaStream_t stream, size_t *need) {
  *need = chunked_workspace_size(a.n_seqs, a.total_tokens, a.H, a.Dk, a.Dv, a.n_slots);
  if (*need > kStaticScratchBytes) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void *base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
      void *p = nullptr;
      e = cudaGetSymbolAddress(&p, g_static_scratch);
      if (e != cudaSuccess) return e;
      g_scratch_addr[dev] = p;
    }
    base = g_scratch_addr[dev];
  }
  a.workspace = base;
  a.workspace_bytes = kStaticScratchBytes;
  return launch_chunked(a, stream);
}

}  // namespace gdn
