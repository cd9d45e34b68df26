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
//  2. chunk_prep_kernel (one CTA per chunk and head, fully parallel): all
//     the state-independent work of a chunk. G = [K^; Q^] K~^T on the tensor
//     cores (tcgen05, accumulator in TMEM) gives A and P; T comes from a
//     blocked fp32 inverse; W = [T'; 0] K is a second tcgen05 product (T' =
//     T diag(e^g) and raw K for GDA; T and K^ = e^g . K for KDA). T, P and -W
//     go to the workspace as bf16, and for KDA also Q^ = e^g . Q and
//     K~ = e^(gC - g) . K; the gate factors the scan needs go there in fp32.
//  3. chunk_scan_kernel (one CTA per sequence, head and half of the value
//     columns, sequential over the chunks): only the state-dependent chain,
//     [D; Q^ S0] = [-W; Q^] S0 + [T; 0] V, then S = e^gC . S0 + K~^T D~ and
//     O = Q^ S0 + [0; P] D on tcgen05, with the fp32 master state in
//     registers and a bf16 copy as the MMA operand; the next chunk's tiles
//     stream in by TMA meanwhile.
// The last K tokens of each sequence then run through the recurrent kernel,
// which writes the snapshot slots.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int CH = 64;  // chunk length

// ---- workspace layout --------------------------------------------------------
//
// Per (chunk, head) tiles, bf16 row-major: T and P [64][64], -W [64][128];
// KDA adds Q^ and K~ [64][128]. Per (chunk, head) gate factors, fp32 [256]:
// GDA e^gamma_r [0, 64), e^(gamma_C - gamma_r) [64, 128), e^gamma_C [128, 256);
// KDA e^gamma_C,i [128, 256) (the rest 1).

struct WsLayout {
  size_t hdr, chunk_seq, chunk_tok, chunk_len, seq_chunk0, seq_nch, tail_start,
      tail_len, tail_pos, order, state_ptrs, states, ready, T, P, W, Qh, Kt, gs, total;
  long long max_chunks;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// with_tiles = false: the token-loop route (fp32 inputs or head sizes other
// than 128), which needs only the per-sequence work list.
WsLayout ws_layout(int n_seqs, int total_tokens, int H, int Dk, int Dv, bool kda,
                   bool with_tiles = true) {
  WsLayout w{};
  w.max_chunks = with_tiles ? (long long)total_tokens / CH + n_seqs : 0;
  const size_t tiles = (size_t)w.max_chunks * H;
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
  w.tail_pos = take(sizeof(int) * (size_t)n_seqs);
  w.order = take(sizeof(int) * (size_t)n_seqs);
  w.state_ptrs = take(sizeof(float *) * (size_t)n_seqs);
  w.states = take(with_tiles ? sizeof(float) * (size_t)n_seqs * H * Dk * Dv : 0);
  w.ready = take(sizeof(int) * tiles);
  w.T = take(2 * tiles * CH * CH);
  w.P = take(2 * tiles * CH * CH);
  w.W = take(2 * tiles * CH * Dk);
  w.Qh = kda ? take(2 * tiles * CH * Dk) : w.W;
  w.Kt = kda ? take(2 * tiles * CH * Dk) : w.W;
  w.gs = take(4 * tiles * 256);
  w.total = off;
  return w;
}

struct WsPtrs {
  int *hdr, *chunk_seq, *chunk_tok, *chunk_len, *seq_chunk0, *seq_nch, *tail_start,
      *tail_len, *tail_pos, *order;
  int *ready;  // per (chunk, head) tile: 1 once chunk prep has written it
  const float **state_ptrs;
  float *states;
  __nv_bfloat16 *T, *P, *W, *Qh, *Kt;
  float *gs;
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
  p.tail_pos = reinterpret_cast<int *>(b + w.tail_pos);
  p.order = reinterpret_cast<int *>(b + w.order);
  p.state_ptrs = reinterpret_cast<const float **>(b + w.state_ptrs);
  p.states = reinterpret_cast<float *>(b + w.states);
  p.ready = reinterpret_cast<int *>(b + w.ready);
  p.T = reinterpret_cast<__nv_bfloat16 *>(b + w.T);
  p.P = reinterpret_cast<__nv_bfloat16 *>(b + w.P);
  p.W = reinterpret_cast<__nv_bfloat16 *>(b + w.W);
  p.Qh = reinterpret_cast<__nv_bfloat16 *>(b + w.Qh);
  p.Kt = reinterpret_cast<__nv_bfloat16 *>(b + w.Kt);
  p.gs = reinterpret_cast<float *>(b + w.gs);
  return p;
}

__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
  return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
}

// Byte offset of 16-byte chunk cj (8 bf16) of row `row` in a tile of
// 128-byte swizzled rows.
__device__ __forceinline__ uint32_t chunk16(int row, int cj) {
  return (uint32_t)(row * 128 + ((cj ^ (row & 7)) << 4));
}

// In-place 4 x 4 transpose of 16-byte pieces inside each group of 4 lanes:
// lane 4a + b holding pieces 0..3 of row 4a + b ends up with p[u] = piece b
// of row 4a + u, so that store u of the group writes 64 contiguous bytes of
// one row. Two xor-shuffle steps.
__device__ __forceinline__ void transpose4x4(uint4 (&p)[4], int lane) {
#pragma unroll
  for (int m = 2; m >= 1; m >>= 1) {
    const bool hi = (lane & m) != 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      if (b & m) continue;
      const uint4 snd = hi ? p[b] : p[b | m];
      uint4 rcv;
      rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, m);
      rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, m);
      rcv.z = __shfl_xor_sync(0xffffffffu, snd.z, m);
      rcv.w = __shfl_xor_sync(0xffffffffu, snd.w, m);
      if (hi) p[b] = rcv;
      else p[b | m] = rcv;
    }
  }
}

__device__ __forceinline__ uint2 pack4(const float *x) {
  return make_uint2(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]));
}

__device__ __forceinline__ uint4 pack8(const float *x) {
  uint4 u;
  u.x = pack_bf16(x[0], x[1]);
  u.y = pack_bf16(x[2], x[3]);
  u.z = pack_bf16(x[4], x[5]);
  u.w = pack_bf16(x[6], x[7]);
  return u;
}

// bf16 high parts of (x0, x1) and the bf16 roundings of the rests, packed in
// pairs (x0 in the low half): x = hi + lo to about 2^-16 relative.
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}

// Warp-level D (16 x 8, fp32) += A (16 x 16, bf16, row-major) * B (16 x 8,
// bf16), fragments as the PTX ISA lays out mma.m16n8k16 (g = lane / 4,
// t = lane % 4; each register a pair of consecutive K indices):
// a = A[g][2t..], A[g+8][2t..], A[g][2t+8..], A[g+8][2t+8..];
// b = B[2t..][g], B[2t+8..][g]; d = D[g][2t], D[g][2t+1], D[g+8][2t], D[g+8][2t+1].
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// ---- 1. work list ---------------------------------------------------------------

constexpr int WL_THREADS = 1024;
constexpr int WL_SMEM_SEQS = 4096;  // cu_seqlens read into shared memory up to this many sequences

// One block. Validates cu_seqlens (cu[0] = 0, non-decreasing, cu[N] = Ntok);
// hdr[0] = chunks in use, hdr[1] = chunk prep's tile counter (zeroed here);
// on failure every sequence gets zero chunks and zero tail tokens, and the
// error word is set. Otherwise sequence s gets Lc_s = max(L_s - K, 0) chunked
// tokens in ceil(Lc_s / 64) chunks and a tail of L_s - Lc_s tokens, and the
// chunk scan visits sequences longest first.
__global__ void __launch_bounds__(WL_THREADS)
    worklist_kernel(const int32_t *__restrict__ cu, int N, int total, int K, int H,
                    long long state_elems, const float *const *state_in, WsPtrs w,
                    long long n_ready, int *err) {
  // The kernels after this one are programmatic dependents: they may start
  // their set-up now and wait for this grid before reading what it writes.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ int bad;
  __shared__ int wsum[WL_THREADS / 32];
  __shared__ int scu[WL_SMEM_SEQS + 1];
  __shared__ int sbase[WL_SMEM_SEQS + 1];  // first chunk of each sequence, then the count
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool in_smem = N <= WL_SMEM_SEQS;
  auto CU = [&](int i) { return in_smem ? scu[i] : cu[i]; };
  // chunk prep's tile counter, and the per-tile ready flags when the scan
  // runs beside the prep
  if (tid == 0) {
    w.hdr[1] = 0;
    bad = 0;
  }
  for (long long e = tid; e < n_ready; e += WL_THREADS) w.ready[e] = 0;
  if (in_smem)
    for (int i = tid; i <= N; i += WL_THREADS) scu[i] = cu[i];
  __syncthreads();
  if (tid == 0 && (CU(0) != 0 || CU(N) != total)) bad = 1;
  for (int s = tid; s < N; s += WL_THREADS)
    if (CU(s + 1) < CU(s)) bad = 1;
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
      w.tail_pos[s] = 0;
      w.order[s] = s;
      w.state_ptrs[s] = nullptr;
    }
    return;
  }
  // per-thread contiguous segment of sequences, then a block scan of counts
  // (inclusive scans within each warp, then over the warps' totals)
  const int per = (N + WL_THREADS - 1) / WL_THREADS;
  const int s0 = min(N, tid * per), s1 = min(N, s0 + per);
  int cnt = 0;
  for (int s = s0; s < s1; ++s) {
    const int L = CU(s + 1) - CU(s);
    const int Lc = max(L - K, 0);
    cnt += (Lc + CH - 1) / CH;
  }
  int incl = cnt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = wsum[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += y;
    }
    wsum[lane] = v;
  }
  __syncthreads();
  if (warp > 0) incl += wsum[warp - 1];
  int base = incl - cnt;
  for (int s = s0; s < s1; ++s) {
    const int L = CU(s + 1) - CU(s);
    const int Lc = max(L - K, 0);
    const int nch = (Lc + CH - 1) / CH;
    w.seq_chunk0[s] = base;
    w.seq_nch[s] = nch;
    w.tail_start[s] = CU(s) + Lc;
    w.tail_len[s] = L - Lc;
    w.tail_pos[s] = Lc;  // position of the first tail token within the sequence
    w.state_ptrs[s] = nch > 0 ? w.states + (long long)s * state_elems : state_in[s];
    if (in_smem) {
      sbase[s] = base;
    } else {
      for (int j = 0; j < nch; ++j) {
        w.chunk_seq[base + j] = s;
        w.chunk_tok[base + j] = CU(s) + j * CH;
        w.chunk_len[base + j] = min(CH, Lc - j * CH);
      }
    }
    base += nch;
  }
  if (tid == WL_THREADS - 1) {
    w.hdr[0] = incl;
    if (in_smem) sbase[N] = incl;
  }
  if (in_smem) {
    // every thread fills chunks: chunk gc belongs to the last sequence whose
    // first chunk is at most gc (sequences without chunks share their base
    // with the next one)
    __syncthreads();
    const int nchunks = sbase[N];
    for (int gc = tid; gc < nchunks; gc += WL_THREADS) {
      int lo = 0, hi = N;  // sbase[lo] <= gc < sbase[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sbase[mid] <= gc) lo = mid;
        else hi = mid;
      }
      const int j = gc - sbase[lo];
      const int Lc = max(CU(lo + 1) - CU(lo) - K, 0);
      w.chunk_seq[gc] = lo;
      w.chunk_tok[gc] = CU(lo) + j * CH;
      w.chunk_len[gc] = min(CH, Lc - j * CH);
    }
  }
  // longest chunk count first (ties by index); identity beyond 4096 sequences
  for (int s = tid; s < N; s += WL_THREADS) {
    if (N > 4096) {
      w.order[s] = s;
      continue;
    }
    const int L = CU(s + 1) - CU(s);
    const int ns = (max(L - K, 0) + CH - 1) / CH;
    int rank = 0;
    for (int t = 0; t < N; ++t) {
      const int Lt = CU(t + 1) - CU(t);
      const int nt = (max(Lt - K, 0) + CH - 1) / CH;
      rank += (nt > ns) || (nt == ns && t < s);
    }
    w.order[rank] = s;
  }
}

// ---- 2. chunk preparation (all state-independent products) -------------------

constexpr int PREP_THREADS = 256;
constexpr int XS_LD = 68;  // fp32 row stride of X (16-byte rows, conflict-free row reads)
// Shared memory, offsets from a 1024-aligned base:
//  KQ [128][128] bf16 in two 64-column halves of 16 KB: K rows 0..63, Q rows
//     64..127 (TMA; KDA scales them in place to K^ = e^g . K and Q^ = e^g . Q).
//     A of G; its K rows are also B of W. Once G is done the Q rows hold A
//     (fp32, rows 0..31 in half 0 and rows 32..63 in half 1, see af_off).
//  TZ [64][64] bf16: T', written after the solve into the Q rows of half 0
//     (free by then); rows 0..63 of the A operand of W (rows 64..127 of that
//     operand read the next 8 KB, K rows, whose products are never used).
//  KB [64][128] bf16: KDA e^-g . K (B of G); afterwards X fp32 [64][XS_LD].
constexpr int PREP_KQ = 0, PREP_TZ = 8192, PREP_KB = 32768;
constexpr int PREP_GAM = PREP_KB + 64 * XS_LD * 4;  // [64] f32 gamma (GDA)
constexpr int PREP_TF = PREP_GAM + 256;             // [64] f32 column factor of T'
constexpr int PREP_BETA = PREP_TF + 256;            // [64] f32
constexpr int PREP_HSUM = PREP_BETA + 256;          // [64] f32 GDA running gate minimum (1 KB)
constexpr int PREP_LAST = PREP_HSUM + 1024;         // [64] int GDA last reset row (-1: none)
constexpr int PREP_FAC = PREP_LAST + 256;           // GDA [64] row, [64] column decay factors,
                                                    // [4] gate range, [1] factored flag
constexpr int PREP_BAR = PREP_FAC + 512 + 32;       // 3 mbarriers
constexpr int PREP_TSLOT = PREP_BAR + 24;
constexpr int PREP_SMEM = PREP_TSLOT + 8 + 1024;    // + alignment slack
constexpr int PREP_KTOT = (PREP_TSLOT + 8 + 15) & ~15;  // KDA [8 warps][128] f32 gate sums
constexpr int PREP_SMEM_KDA = PREP_KTOT + 4096 + 1024;
constexpr uint32_t PCOL_G = 0, PCOL_W = 0;          // TMEM columns (128 allocated; W reuses G's)
static_assert(PREP_TZ % 1024 == 0 && PREP_KB % 1024 == 0, "swizzled atoms are 1024-aligned");
static_assert(64 * XS_LD * 4 >= 16384, "X region also holds KB");

// Byte offset of A(r, j) (fp32) inside KQ once G is done: rows 0..31 in the
// Q rows of half 0, rows 32..63 in those of half 1; 64 floats (16 pieces of
// 16 bytes) per row with the piece index XOR-ed by (r & 15): a thread
// writes 4 consecutive columns of its row as one 16-byte store, 32 threads
// storing the same columns of 32 consecutive rows take the minimum 4
// wavefronts, and the tensor-core fragment reads of the solve (rows g, g+8,
// columns t, t+4 of a 16 x 8 tile) touch 32 different banks.
__device__ __forceinline__ uint32_t af_off(int r, int j) {
  return (uint32_t)((r >> 5) * 16384 + 8192 + (r & 31) * 256 + ((((j >> 2) ^ (r & 15))) << 4) +
                    ((j & 3) << 2));
}

// One CTA per (chunk, head). Rows r of the chunk are tokens chunk_tok + r,
// r < len; the rest are padding (k = q = 0, beta = 0, g = 0).
template <bool KDA>
__global__ void __launch_bounds__(PREP_THREADS, KDA ? 3 : 4)
    chunk_prep_kernel(const __grid_constant__ CUtensorMap map_q,
                      const __grid_constant__ CUtensorMap map_k, const float *__restrict__ g,
                      const float *__restrict__ beta, int H, int Hqk, int qk_grouped,
                      WsPtrs w, int publish, int handoff_sms, int num_sms, int *err) {
  constexpr int DK = 128;
  // This grid is a programmatic dependent of the work list: wait for it
  // before reading what it wrote. The chunk scan, launched after this grid as
  // a programmatic dependent, may then start once every CTA here has passed
  // this point (so the work list is complete for it too).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int ntiles = w.hdr[0] * H;  // (chunks in use) x heads, chunk-major
  if ((int)blockIdx.x >= ntiles) return;
  // Hand-off: the CTAs on about handoff_sms of the SMs leave at once, so that
  // the scan's CTAs (one per SM) take those SMs, set up and wait for their
  // first tiles while the rest of the prep goes on beside them.
  if (handoff_sms > 0) {
    uint32_t smid, nsmid;
    asm("mov.u32 %0, %%smid;" : "=r"(smid));
    asm("mov.u32 %0, %%nsmid;" : "=r"(nsmid));
    if ((long long)smid * num_sms < (long long)handoff_sms * nsmid) return;
  }
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = align1024(smem_raw);
  unsigned char *KQ = sm + PREP_KQ, *KB = sm + PREP_KB, *TZ = sm + PREP_TZ;
  float *Xs = reinterpret_cast<float *>(sm + PREP_KB);  // [64][XS_LD], after G
  float *sgam = reinterpret_cast<float *>(sm + PREP_GAM);
  float *stf = reinterpret_cast<float *>(sm + PREP_TF);
  float *sbeta = reinterpret_cast<float *>(sm + PREP_BETA);
  float *hsum = reinterpret_cast<float *>(sm + PREP_HSUM);
  int *slast = reinterpret_cast<int *>(sm + PREP_LAST);
  float *smin = hsum;  // GDA: running minimum of the cumulative gate [64]
  float *srowf = reinterpret_cast<float *>(sm + PREP_FAC), *scolf = srowf + 64;
  float *srange = scolf + 64;
  int *sfact = reinterpret_cast<int *>(srange + 4);
  float4 *ktot = reinterpret_cast<float4 *>(sm + PREP_KTOT);  // KDA only
  uint64_t *bar_tma = reinterpret_cast<uint64_t *>(sm + PREP_BAR);
  uint64_t *bar_g = bar_tma + 1, *bar_w = bar_tma + 2;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + PREP_TSLOT);
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // K and Q rows of tile tl (first token lt) into KQ, completing on bar_tma
  // (one thread)
  auto load_tile = [&](int tl, int lt) {
    const int lh = tl % H;
    const int lq = qk_grouped ? lh / (H / Hqk) : lh % Hqk;
    mbar_arrive_expect_tx(bar_tma, 32768);
    tma_load_3d(KQ, &map_k, 0, lq, lt, bar_tma);
    tma_load_3d(KQ + 16384, &map_k, 64, lq, lt, bar_tma);
    tma_load_3d(KQ + 8192, &map_q, 0, lq, lt, bar_tma);
    tma_load_3d(KQ + 16384 + 8192, &map_q, 64, lq, lt, bar_tma);
  };
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(bar_tma, 1);
    mbar_init(bar_g, 1);
    mbar_init(bar_w, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  // Persistent: every CTA takes the next unclaimed tile (tiles go in chunk
  // order) from the counter in hdr[1]; the copies of its next tile are issued
  // as soon as the current one's last product has read K and Q. Thread 0
  // claims, and counts the loads issued and waited for; the first token and
  // length of the next tile's chunk are read with the claim and handed over
  // in shared memory.
  __shared__ int next_tile, next_tok, next_len, s_claim[3];
  int loads_issued = 0, loads_done = 0;
  if (tid == 0) {
    const int t = atomicAdd(&w.hdr[1], 1);
    next_tile = t;
    if (t < ntiles) {
      next_tok = w.chunk_tok[t / H];
      next_len = w.chunk_len[t / H];
      load_tile(t, next_tok);
      loads_issued = 1;
    }
  }
  __syncthreads();
  for (int it = 0, tl = next_tile; tl < ntiles; ++it) {
  const uint32_t par = (uint32_t)(it & 1);
  const int h = tl % H;
  const int t0 = next_tok, len = next_len;
  const long long tile = tl;
  // gates and beta while the tiles are in flight (padding rows: g = beta = 0)
  // KDA gates: warp = 8 consecutive rows, lane = 4 consecutive channels, so
  // that every load (and every store of Q^ and K~ below) is one whole row
  float gk[KDA ? 8 : 1][4];
  if constexpr (KDA) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int r = 8 * warp + k;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < len)
        a = *reinterpret_cast<const float4 *>(g + ((long long)(t0 + r) * H + h) * DK + 4 * lane);
      gk[k][0] = a.x; gk[k][1] = a.y; gk[k][2] = a.z; gk[k][3] = a.w;
    }
  }
  if (tid < CH) {
    const long long row = (long long)(t0 + tid) * H + h;
    sbeta[tid] = tid < len ? beta[row] : 0.f;
    if constexpr (!KDA) {
      // A gate of -inf resets the state: every decay across that token is
      // exactly zero. The cumulative gate sums the other (finite) gates, and
      // slast[r] is the last reset row <= r (-1: none), so the decay from
      // row j to row r >= j is zero when slast[r] > j and e^(sgam[r] -
      // sgam[j]) otherwise, never inf - inf. Inclusive shuffle scans (sum
      // and max) in each warp, then warp 1 adds warp 0's totals.
      float x = tid < len ? g[row] : 0.f;
      int li = -1;
      if (x == -INFINITY) {
        x = 0.f;
        li = tid;
      }
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, off);
        const int l = __shfl_up_sync(0xffffffffu, li, off);
        if (lane >= off) {
          x += y;
          li = max(li, l);
        }
      }
      // running minimum of the cumulative gate (warp 0 also counts the chunk
      // start, 0), for the growth check below
      float mn = tid < 32 ? fminf(x, 0.f) : x;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, mn, off);
        if (lane >= off) mn = fminf(mn, y);
      }
      sgam[tid] = x;
      slast[tid] = li;
      smin[tid] = mn;
    }
  }
  // thread 0 waits for this tile's copies; thread 64 (idle until the barrier
  // below) claims the tile after this one, so that the two latencies overlap
  // and the claim is known long before its copies are issued (kept in shared
  // memory: no registers live across the tile)
  if (tid == 0) {
    if (mbar_wait(bar_tma, par, err, kSitePrepLoad)) ++loads_done;
    else abort_flag = 1;
  }
  if (tid == 64) s_claim[0] = atomicAdd(&w.hdr[1], 1);
  __syncthreads();
  if constexpr (!KDA) {
    if (tid >= 32 && tid < CH) {
      smin[tid] = fminf(smin[31], smin[tid] + sgam[31]);
      sgam[tid] += sgam[31];
      slast[tid] = max(slast[tid], slast[31]);
    }
  }
  if (abort_flag) break;
  if constexpr (KDA) {
    // cumulative gates: prefix over the warp's 8 rows here, the sums of the
    // warps before it after the barrier below
#pragma unroll
    for (int k = 1; k < 8; ++k)
#pragma unroll
      for (int c = 0; c < 4; ++c) gk[k][c] += gk[k - 1][c];
    ktot[warp * 32 + lane] = make_float4(gk[7][0], gk[7][1], gk[7][2], gk[7][3]);
  }
  if (len < CH) {  // padding rows of K and Q are zero
    const int nz = (CH - len) * 8;
    for (int e = tid; e < nz * 2; e += PREP_THREADS) {
      const int a = e / nz, rem = e % nz;
      const int r = len + rem / 8, cj = rem % 8;
      const uint4 z = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4 *>(KQ + a * 16384 + r * 128 + cj * 16) = z;
      *reinterpret_cast<uint4 *>(KQ + a * 16384 + (CH + r) * 128 + cj * 16) = z;
    }
  }
  __syncthreads();
  if constexpr (KDA) {
    // Per-row decays inside the operands, relative to the chunk start:
    // K^ = e^g K and Q^ = e^g Q (A of G; K^ is also B of W), e^-g K (B of G),
    // and for the scan Q^, K~ = e^(gC - g) K and e^gC. The sums of the warps
    // before this one complete the cumulative gates; all eight give gC.
    float ex[4] = {0.f, 0.f, 0.f, 0.f}, gC[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w2 = 0; w2 < 8; ++w2) {
      const float4 t = ktot[w2 * 32 + lane];
      if (w2 < warp) {
        ex[0] += t.x; ex[1] += t.y; ex[2] += t.z; ex[3] += t.w;
      }
      gC[0] += t.x; gC[1] += t.y; gC[2] += t.z; gC[3] += t.w;
    }
    // out of range (NaN included): |gamma| > 80 at the chunk end or any row
    bool bad = false;
    float eC[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      bad |= !(fabsf(gC[c]) <= kMaxChunkLogDecay);
      eC[c] = __expf(gC[c]);
    }
    // channels 4 lane .. 4 lane + 3: 64-column half, 16-byte piece, 8-byte half
    const uint32_t half = (uint32_t)(lane >> 4), piece = (uint32_t)((lane & 15) >> 1);
    const uint32_t sub = (uint32_t)(lane & 1) << 3;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int r = 8 * warp + k;
      const uint32_t sw = (uint32_t)r * 128u + ((piece ^ (uint32_t)(r & 7)) << 4) + sub;
      uint2 *pk = reinterpret_cast<uint2 *>(KQ + half * 16384u + sw);
      uint2 *pq = reinterpret_cast<uint2 *>(KQ + half * 16384u + 8192u + sw);
      const uint2 ku = *pk, qu = *pq;
      const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&ku);
      const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&qu);
      float kh[4], qh[4], kb[4], kt[4];
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const float2 kf = __bfloat1622float2(k2[c2]), qf = __bfloat1622float2(q2[c2]);
        const float kv[2] = {kf.x, kf.y}, qv[2] = {qf.x, qf.y};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = 2 * c2 + e;
          const float gam = gk[k][c] + ex[c];
          bad |= !(fabsf(gam) <= kMaxChunkLogDecay);
          // |gamma| <= 80 inside a chunk (checked), so e^gC e^-gamma does not
          // overflow and stands in for e^(gC - gamma)
          const float e1 = __expf(gam), e2 = __expf(-gam);
          kh[c] = kv[e] * e1;
          qh[c] = qv[e] * e1;
          kb[c] = kv[e] * e2;
          kt[c] = kv[e] * (eC[c] * e2);
        }
      }
      const uint2 qhu = pack4(qh);
      *pk = pack4(kh);
      *pq = qhu;
      *reinterpret_cast<uint2 *>(KB + half * 8192u + sw) = pack4(kb);
      *reinterpret_cast<uint2 *>(w.Qh + (tile * CH + r) * DK + 4 * lane) = qhu;
      *reinterpret_cast<uint2 *>(w.Kt + (tile * CH + r) * DK + 4 * lane) = pack4(kt);
    }
    if (warp == 0) {
      reinterpret_cast<float4 *>(w.gs + tile * 256 + 128)[lane] =
          make_float4(expf(gC[0]), expf(gC[1]), expf(gC[2]), expf(gC[3]));
      reinterpret_cast<float4 *>(w.gs + tile * 256)[lane] = make_float4(1.f, 1.f, 1.f, 1.f);
    }
    if (bad) set_error(err, kDevGateRange);
  } else {  // gate factors of the scan
    const float gCs = sgam[CH - 1];
    const int lastC = slast[CH - 1];
    float *gs = w.gs + tile * 256;
    if (tid < CH) {
      // decay from the chunk start to row tid, and from row tid to the end
      gs[tid] = slast[tid] >= 0 ? 0.f : expf(sgam[tid]);
      gs[CH + tid] = lastC > tid ? 0.f : expf(gCs - sgam[tid]);
      // Decays are pairwise differences; only growth can overflow. The
      // largest growth over rows (j, tid] is sgam[tid] minus smin[tid], the
      // smallest cumulative gate up to it (0 at the chunk start); a NaN or
      // +inf gate fails the test too.
      if (!(sgam[tid] - smin[tid] <= kMaxChunkLogDecay)) set_error(err, kDevGateRange);
      // range of the cumulative gate over the chunk, for the factored decays
      float hi = sgam[tid], lo = hi;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off));
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
      }
      if (lane == 0) {
        srange[2 * warp] = hi;
        srange[2 * warp + 1] = lo;
      }
    } else if (tid < CH + 128) {
      gs[128 + tid - CH] = lastC >= 0 ? 0.f : expf(gCs);
    }
  }
  if (tid < CH) {  // column factor of T' = T diag(e^gamma) (GDA) or T (KDA)
    float f = sbeta[tid];
    if constexpr (!KDA) f = slast[tid] >= 0 ? 0.f : f * __expf(sgam[tid]);
    stf[tid] = f;
  }
  fence_proxy_async();
  __syncthreads();
  if constexpr (!KDA) {
    // Decay from row j to row r: e^(gamma_r - gamma_j) = e^(gamma_r - m) e^(m - gamma_j)
    // with m the middle of the chunk's gate range. When that range is at most
    // 160 both factors stay within e^(+-80) (no overflow, no flush to zero of a
    // factor whose partner is large), and A and P take two multiplies per
    // element instead of an exponential; wider ranges keep the pairwise form.
    if (tid < CH) {
      const float hi = fmaxf(srange[0], srange[2]), lo = fminf(srange[1], srange[3]);
      const float m = 0.5f * (hi + lo);
      srowf[tid] = __expf(sgam[tid] - m);
      scolf[tid] = __expf(m - sgam[tid]);
      if (tid == 0) *sfact = hi - lo <= 2.f * kMaxChunkLogDecay ? 1 : 0;
    }
  }

  // G = [K'; Q'] K''^T : M = 128, N = 64, K = 128 (8 steps of 16)
  if (tid == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
    const uint32_t a0 = smem_u32(KQ);
    const uint32_t b0 = KDA ? smem_u32(KB) : smem_u32(KQ);
    const uint32_t bcol = KDA ? 8192u : 16384u;
#pragma unroll
    for (int s = 0; s < 8; ++s)
      umma_bf16(tbase + PCOL_G, sdesc_kmajor(a0 + (s >> 2) * 16384u + (s & 3) * 32u),
                sdesc_kmajor(b0 + (s >> 2) * bcol + (s & 3) * 32u), idesc, s > 0);
    umma_commit(bar_g);
    if (s_claim[0] < ntiles) {
      s_claim[1] = w.chunk_tok[s_claim[0] / H];
      s_claim[2] = w.chunk_len[s_claim[0] / H];
    }
    if (!mbar_wait(bar_g, par, err, kSitePrepG)) abort_flag = 1;
  }
  __syncthreads();
  tc_fence_after();
  if (!abort_flag) {
    // thread = accumulator row (TMEM lane group warp & 3) and 32 columns
    // (warp >> 2): rows 0..63 give A (into the Q rows, dead once G is done),
    // rows 64..127 give P
    const int row = 32 * (warp & 3) + lane, j0 = 32 * (warp >> 2);
    float G[32];
    tmem_ld32(tbase + ((uint32_t)(32 * (warp & 3)) << 16) + PCOL_G + j0, G);
    if (row < CH) {
      const int r = row;
      const float br = sbeta[r];
      const float gr = KDA ? 0.f : sgam[r];
      const int lr = KDA ? -1 : slast[r];  // decays across a reset row are zero
      if (KDA || !*sfact) {
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int j = j0 + u;
          float a = 0.f;
          if (j < r && j >= lr) {
            a = br * G[u];
            if constexpr (!KDA) a *= __expf(gr - sgam[j]);
          }
          G[u] = a;
        }
        unsigned char *arow = KQ + af_off(r, 0) - ((r & 15) << 4);  // row base
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          *reinterpret_cast<float4 *>(arow + ((((j0 >> 2) + c4) ^ (r & 15)) << 4)) =
              make_float4(G[4 * c4], G[4 * c4 + 1], G[4 * c4 + 2], G[4 * c4 + 3]);
      } else {
        const float brf = br * srowf[r];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int j = j0 + u;
          G[u] = j < r && j >= lr ? brf * G[u] * scolf[j] : 0.f;
        }
        unsigned char *arow = KQ + af_off(r, 0) - ((r & 15) << 4);  // row base
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          *reinterpret_cast<float4 *>(arow + ((((j0 >> 2) + c4) ^ (r & 15)) << 4)) =
              make_float4(G[4 * c4], G[4 * c4 + 1], G[4 * c4 + 2], G[4 * c4 + 3]);
      }
    } else {
      const int r = row - CH;
      const float gr = KDA ? 0.f : sgam[r];
      const int lr = KDA ? -1 : slast[r];
      uint32_t packed[16];
      if (KDA || !*sfact) {
#pragma unroll
        for (int u = 0; u < 32; u += 2) {
          const int j = j0 + u;
          float p0 = 0.f, p1 = 0.f;
          if (r < len) {
            if (j <= r && j >= lr) {
              p0 = G[u];
              if constexpr (!KDA) p0 *= __expf(gr - sgam[j]);
            }
            if (j + 1 <= r && j + 1 >= lr) {
              p1 = G[u + 1];
              if constexpr (!KDA) p1 *= __expf(gr - sgam[j + 1]);
            }
          }
          packed[u / 2] = pack_bf16(p0, p1);
        }
      } else {
        const float rf = r < len ? srowf[r] : 0.f;
#pragma unroll
        for (int u = 0; u < 32; u += 2) {
          const int j = j0 + u;
          const float p0 = j <= r && j >= lr ? rf * G[u] * scolf[j] : 0.f;
          const float p1 = j + 1 <= r && j + 1 >= lr ? rf * G[u + 1] * scolf[j + 1] : 0.f;
          packed[u / 2] = pack_bf16(p0, p1);
        }
      }
      uint4 pc[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        pc[e] = make_uint4(packed[4 * e], packed[4 * e + 1], packed[4 * e + 2], packed[4 * e + 3]);
      transpose4x4(pc, lane);  // each store: 64 contiguous bytes of 8 rows
      const int rb = r - (lane & 3);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        reinterpret_cast<uint4 *>(w.P + (tile * CH + rb + u) * CH + j0)[lane & 3] = pc[u];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (abort_flag) break;

  // X = (I + A)^-1 by 16 x 16 blocks (A strictly lower triangular):
  //   X[R][R] = (I + A[R][R])^-1,
  //   X[R][K] = -X[R][R] sum_{M=K..R-1} A[R][M] X[M][K]      (K < R),
  // one block row after another. The four diagonal inverses are forward
  // substitutions on the CUDA cores (thread = block and column); the block
  // products run on the tensor cores as warp-level bf16 MMAs with every
  // operand split into a bf16 high and low part (hi*hi + hi*lo + lo*hi),
  // about 2^-16 relative, far below the bf16 rounding T and T' get next.
  // X goes to Xs (fp32, row stride XS_LD).
  {
    if (tid < CH) {  // diagonal block R, column c: right-looking substitution
      const int R = tid >> 4, c = tid & 15, r0 = 16 * R;
      // A(r0 + u2, r0 + u) sits at ablk[u2 >> 2] + 256 u2 + 16 ((u >> 2) ^ (u2 & 3))
      // + 4 (u & 3): four bases per thread, the rest compile-time offsets
      const unsigned char *arow = KQ + (R >> 1) * 16384 + 8192 + (R & 1) * 4096;
      const unsigned char *ablk[4] = {arow + 64 * (R ^ 0), arow + 64 * (R ^ 1),
                                      arow + 64 * (R ^ 2), arow + 64 * (R ^ 3)};
      float *xcol = Xs + r0 * XS_LD + r0 + c;
      float acc[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) acc[u] = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float xu = (u == c ? 1.f : 0.f) - acc[u];
        xcol[u * XS_LD] = xu;
#pragma unroll
        for (int u2 = u + 1; u2 < 16; ++u2)
          acc[u2] = fmaf(*reinterpret_cast<const float *>(ablk[u2 >> 2] + 256 * u2 +
                                                          16 * ((u >> 2) ^ (u2 & 3)) +
                                                          4 * (u & 3)),
                         xu, acc[u2]);
      }
    } else {  // zero blocks above the diagonal
      for (int e = tid - CH; e < 6 * 256; e += PREP_THREADS - CH) {
        const int blk = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
        // upper blocks (R, K), K > R: (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
        const int R = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int K = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        Xs[(16 * R + rr) * XS_LD + 16 * K + cc] = 0.f;
      }
    }
    __syncthreads();
    const int g = lane >> 2, t = lane & 3;
    auto Af = [&](int r, int j) { return *reinterpret_cast<const float *>(KQ + af_off(r, j)); };
    // fragments of a 16 x 16 A tile (rows r0.., columns k0..) and of a 16 x 8
    // B tile of Xs (rows k0.., columns c0..), split into bf16 high and low parts
    auto a_frags = [&](auto ld, int r0, int k0, uint32_t (&ah)[4], uint32_t (&al)[4]) {
      split_bf16x2(ld(r0 + g, k0 + 2 * t), ld(r0 + g, k0 + 2 * t + 1), ah[0], al[0]);
      split_bf16x2(ld(r0 + g + 8, k0 + 2 * t), ld(r0 + g + 8, k0 + 2 * t + 1), ah[1], al[1]);
      split_bf16x2(ld(r0 + g, k0 + 2 * t + 8), ld(r0 + g, k0 + 2 * t + 9), ah[2], al[2]);
      split_bf16x2(ld(r0 + g + 8, k0 + 2 * t + 8), ld(r0 + g + 8, k0 + 2 * t + 9), ah[3], al[3]);
    };
    auto Xf = [&](int r, int j) { return Xs[r * XS_LD + j]; };
    auto b_frags = [&](int k0, int c0, uint32_t (&bh)[2], uint32_t (&bl)[2]) {
      split_bf16x2(Xf(k0 + 2 * t, c0 + g), Xf(k0 + 2 * t + 1, c0 + g), bh[0], bl[0]);
      split_bf16x2(Xf(k0 + 2 * t + 8, c0 + g), Xf(k0 + 2 * t + 9, c0 + g), bh[1], bl[1]);
    };
    for (int R = 1; R < 4; ++R) {
      if (warp < 2 * R) {  // output X[R][K], columns 8 nh .. 8 nh + 7 of block K
        const int K = warp >> 1, c0 = 16 * K + 8 * (warp & 1), r0 = 16 * R;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int M = K; M < R; ++M) {
          uint32_t ah[4], al[4], bh[2], bl[2];
          a_frags(Af, r0, 16 * M, ah, al);
          b_frags(16 * M, c0, bh, bl);
          mma_bf16_16816(acc, al, bh);
          mma_bf16_16816(acc, ah, bl);
          mma_bf16_16816(acc, ah, bh);
        }
        // the sum over M goes where X[R][K] will be (this warp alone reads
        // and writes these 16 x 8 values), then X[R][K] = -X[R][R] (sum)
        Xs[(r0 + g) * XS_LD + c0 + 2 * t] = acc[0];
        Xs[(r0 + g) * XS_LD + c0 + 2 * t + 1] = acc[1];
        Xs[(r0 + g + 8) * XS_LD + c0 + 2 * t] = acc[2];
        Xs[(r0 + g + 8) * XS_LD + c0 + 2 * t + 1] = acc[3];
        __syncwarp();
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        {
          uint32_t ah[4], al[4], bh[2], bl[2];
          a_frags(Xf, r0, r0, ah, al);
          b_frags(r0, c0, bh, bl);
          mma_bf16_16816(o, al, bh);
          mma_bf16_16816(o, ah, bl);
          mma_bf16_16816(o, ah, bh);
        }
        __syncwarp();  // every lane has read the sum before it is overwritten
        Xs[(r0 + g) * XS_LD + c0 + 2 * t] = -o[0];
        Xs[(r0 + g) * XS_LD + c0 + 2 * t + 1] = -o[1];
        Xs[(r0 + g + 8) * XS_LD + c0 + 2 * t] = -o[2];
        Xs[(r0 + g + 8) * XS_LD + c0 + 2 * t + 1] = -o[3];
      }
      __syncthreads();
    }
  }
  // T[r][j] = X[r][j] beta_j (to the workspace) and T'[r][j] = X[r][j] f_j
  // into TZ; thread = (row r = tid / 4, columns 8q..8q+7 and 8q+32..8q+39 with
  // q = tid % 4), so that each store of a warp writes 64 contiguous bytes of
  // each of 8 rows
  {
    const int r = tid >> 2, q = tid & 3;
    float tv[16], tp[16];
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      const float4 *xr = reinterpret_cast<const float4 *>(Xs + r * XS_LD + 8 * q + 32 * hlf);
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        const float4 x4 = xr[v];
        const float xv[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int j = 8 * q + 32 * hlf + 4 * v + b;
          tv[8 * hlf + 4 * v + b] = xv[b] * sbeta[j];
          tp[8 * hlf + 4 * v + b] = xv[b] * stf[j];
        }
      }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(w.T + (tile * CH + r) * CH);
    dst[q] = pack8(tv);
    dst[q + 4] = pack8(tv + 8);
    *reinterpret_cast<uint4 *>(TZ + chunk16(r, q)) = pack8(tp);
    *reinterpret_cast<uint4 *>(TZ + chunk16(r, q + 4)) = pack8(tp + 8);
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // W (lanes r, columns i) = T'(r, j) K(i, j), K (or K^) as the MN-major K
  // rows of KQ: M = 128 (rows 64..127 unused), N = 128, K = 64
  if (tid == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
    for (int s = 0; s < 4; ++s)
      umma_bf16(tbase + PCOL_W, sdesc_kmajor(smem_u32(TZ) + s * 32),
                sdesc_mnmajor(smem_u32(KQ) + s * 2048, 16384), idesc, s > 0);
    umma_commit(bar_w);
    if (!mbar_wait(bar_w, par, err, kSitePrepW)) {
      abort_flag = 1;
    } else {  // K and Q are free: the next tile's copies
      next_tile = s_claim[0];
      if (s_claim[0] < ntiles) {
        next_tok = s_claim[1];
        next_len = s_claim[2];
        load_tile(s_claim[0], s_claim[1]);
        ++loads_issued;
      }
    }
  }
  __syncthreads();
  tc_fence_after();
  if (!abort_flag && (warp & 3) < 2) {  // -W: rows r (lanes 0..63), 64 columns per warp
    const int r = 32 * (warp & 3) + lane, c0 = 64 * (warp >> 2);
    const int rb = r - (lane & 3);
#pragma unroll
    for (int q32 = 0; q32 < 2; ++q32) {
      float v[32];
      tmem_ld32(tbase + ((uint32_t)(32 * (warp & 3)) << 16) + PCOL_W + c0 + 32 * q32, v);
#pragma unroll
      for (int u = 0; u < 32; ++u) v[u] = -v[u];
      uint4 pc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) pc[q] = pack8(v + 8 * q);
      transpose4x4(pc, lane);  // each store: 64 contiguous bytes of 8 rows
#pragma unroll
      for (int u = 0; u < 4; ++u)
        reinterpret_cast<uint4 *>(w.W + (tile * CH + rb + u) * DK + c0 + 32 * q32)[lane & 3] =
            pc[u];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (abort_flag) break;
  if (publish && tid == 0) {
    // every thread's stores of this tile precede the barrier above; the
    // release makes them visible before the flag (the scan acquires it)
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(w.ready + tile), "r"(1) : "memory");
  }
  tl = next_tile;
  }  // tiles
  // after an abort, copies still in flight land before the CTA exits
  if (tid == 0 && loads_issued > loads_done)
    mbar_wait(bar_tma, (uint32_t)(loads_done & 1), nullptr);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 128);
}

// ---- 3. chunk scan (warp-specialised, two-stage pipelined) --------------------
//
// One CTA per (sequence, head, half of the value columns): NV = 64 state
// columns, all chunks of the sequence in order. Roles:
//   warps 0..STATE_WARPS-1 "state": thread (key row i = 32 (w & 3) + lane,
//             CPT columns from CPT (w >> 2)) owns that part of the fp32
//             state; turns X into D and D~, applies the state update, writes
//             outputs (a warp reads TMEM lanes 32 (w & 3) .. + 31 only);
//   warp STATE_WARPS "producer": TMA loads of each chunk's tiles into a
//             two-stage ring (and zero padding rows of a partial last chunk);
//   warp STATE_WARPS + 1 "mma": lane 0 issues every tcgen05.mma.
// Per chunk the state-dependent chain is: X += [-W; Q] S0 (mma) -> D (state)
// -> S_acc = K~^T D~ (mma) -> S = e^gC . S0 + S_acc (state) -> next chunk.
// Off that chain: [T; 0] V of the next chunk is issued right behind the
// state update, [0; P] D right behind the next chunk's [-W; Q] S0, and the
// outputs of a chunk are stored while the next chunk's state update runs.
constexpr int NV = 64;
constexpr int STATE_WARPS = 8;  // a multiple of 4 (one warp per TMEM lane quadrant)
constexpr int STATE_THREADS = 32 * STATE_WARPS;
constexpr int PRODUCER_WARP = STATE_WARPS, MMA_WARP = STATE_WARPS + 1;
constexpr int SCAN_WARPS = STATE_WARPS + 2;
constexpr int SCAN_THREADS = SCAN_WARPS * 32;
// state columns per state thread (of the CTA's NV) and their 8-column pieces
constexpr int CPT = NV / (STATE_WARPS / 4), PPT = CPT / 8;
static_assert(STATE_WARPS % 4 == 0 && (CPT == 16 || CPT == 32), "state split");
// stage: K (GDA) or K~ (KDA) [64 r][128 i] | [-W; Q or Q^] [128][128 i] |
//        V [64 j][64 v] | T [64 r][64 j] | zeros [64][64] | P [64 r][64 j] |
//        gate factors fp32 [256]
constexpr int ST_K = 0, ST_WQ = 16384, ST_V = 49152, ST_T = 57344, ST_Z = 65536,
              ST_P = 73728, ST_G = 81920, ST_BYTES = 82944;
constexpr int ST_TX = 16384 + 32768 + 8192 + 8192 + 8192 + 1024;  // bytes TMA brings
constexpr int SC_S = 2 * ST_BYTES;       // S0 bf16 [128 i][64 v] (B of X, MN-major)
constexpr int SC_D = SC_S + 16384;       // D [2][64 r][64 v] (double-buffered)
constexpr int SC_DT = SC_D + 16384;      // D~ [64 r][64 v] (GDA)
constexpr int SC_OUT = SC_DT + 8192;    // output staging fp32 [2][64 r][32 v], 128-byte swizzle
constexpr int SC_BARS = SC_OUT + 16384;  // 11 mbarriers
constexpr int SC_RFLAGS = SC_BARS + 11 * 8;
constexpr int SC_TSLOT = SC_RFLAGS + 8;
constexpr int SCAN_SMEM = SC_TSLOT + 8 + 1024;  // + alignment slack
static_assert(ST_BYTES % 1024 == 0 && SC_S % 1024 == 0, "swizzled tiles are 1024-aligned");
// TMEM columns (512 allocated): X triple-buffered (a chunk's Q S0 rows are
// read after the next chunk's X is issued), state update, O double-buffered
constexpr uint32_t COL_X0 = 0, COL_S = 192, COL_O0 = 256;
// polls of the clean-up waits before exit (a healthy one ends at once)
constexpr uint32_t kDrainPolls = 1u << 22;

// TMEM -> registers, CPT consecutive columns of the thread's lane.
template <int N>
__device__ __forceinline__ void tmem_ld_cpt(uint32_t taddr, float (&v)[N]) {
  if constexpr (N == 32) tmem_ld32(taddr, v);
  else tmem_ld16(taddr, v);
}

// Barrier over the state threads (id 1). The non-aligned form counts
// threads, so lanes that reach it at different times are fine; __syncwarp
// first reconverges the warp after a single-lane wait.
__device__ __forceinline__ void named_bar(int id) {
  __syncwarp();
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "n"(STATE_THREADS) : "memory");
}

// In-place 8 x 8 transpose of 16-byte pieces inside each group of 8 lanes:
// lane 8g + a holding piece b of row 8g + a (x[4b .. 4b+3]) ends up holding
// piece a of row 8g + b. Three xor-shuffle steps; applying it twice restores x.
__device__ __forceinline__ void transpose8x8(float (&x)[32], int lane) {
#pragma unroll
  for (int m = 4; m >= 1; m >>= 1) {
    const bool hi = (lane & m) != 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      if (b & m) continue;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float snd = hi ? x[4 * b + c] : x[4 * (b | m) + c];
        const float rcv = __shfl_xor_sync(0xffffffffu, snd, m);
        if (hi) x[4 * b + c] = rcv;
        else x[4 * (b | m) + c] = rcv;
      }
    }
  }
}

// Stores the 32 x 32 fp32 block a warp holds (lane l: row l, 32 consecutive
// floats) to rows `ld` floats apart starting at dst: after transpose8x8 each
// store instruction writes four whole 128-byte rows instead of 32 scattered
// 16-byte pieces; a second transpose gives x back. Every lane must call it.
__device__ __forceinline__ void store_rows32(float (&x)[32], float *dst, long long ld,
                                             int lane) {
  transpose8x8(x, lane);
  const int g = lane >> 3, p = lane & 7;
#pragma unroll
  for (int u = 0; u < 8; ++u)
    *reinterpret_cast<float4 *>(dst + (long long)(8 * g + u) * ld + 4 * p) =
        make_float4(x[4 * u], x[4 * u + 1], x[4 * u + 2], x[4 * u + 3]);
  transpose8x8(x, lane);
}

// Stores the 32 x 16 fp32 block a warp holds (lane l: row l, 16 consecutive
// floats) to rows `ld` floats apart starting at dst: after a 4 x 4 transpose
// of 16-byte pieces inside each group of 4 lanes, each store instruction
// writes 64 contiguous bytes of 8 rows; a second transpose gives x back.
[[maybe_unused]] __device__ __forceinline__ void store_rows16(float (&x)[16], float *dst,
                                                              long long ld, int lane) {
  uint4 p[4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
    p[u] = make_uint4(__float_as_uint(x[4 * u]), __float_as_uint(x[4 * u + 1]),
                      __float_as_uint(x[4 * u + 2]), __float_as_uint(x[4 * u + 3]));
  transpose4x4(p, lane);
  const int rb = lane & ~3, a = lane & 3;
#pragma unroll
  for (int u = 0; u < 4; ++u)
    *reinterpret_cast<uint4 *>(dst + (long long)(rb + u) * ld + 4 * a) = p[u];
}

template <int N>
__device__ __forceinline__ void store_rows_cpt(float (&x)[N], float *dst, long long ld,
                                               int lane) {
  if constexpr (N == 32) store_rows32(x, dst, ld, lane);
  else store_rows16(x, dst, ld, lane);
}

// Bounded wait that also gives up early once another role has aborted. On
// a timeout the error word records the site (bits 8..15) and chunk (16..).
__device__ __forceinline__ bool wait_ab(uint64_t *bar, uint32_t parity,
                                        volatile int *abort_flag, int *err, int site,
                                        int jc) {
  for (uint32_t i = 0; i < kMaxPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return !*abort_flag;
    if ((i & 1023u) == 1023u && *abort_flag) return false;
  }
  set_error(err, kDevTimeout | (site << 8) | ((jc & 0x7fff) << 16));
  *abort_flag = 1;
  return false;
}

// Wait of at most kReadyWaitNs for a tile's ready flag (set by chunk prep
// with a release); then orders the async-proxy (TMA) reads of that tile after
// the acquire. On a timeout the error word records the site and chunk.
constexpr unsigned long long kReadyWaitNs = 2000000000ull;
__device__ __forceinline__ bool wait_ready_flag(const int *flag, volatile int *abort_flag,
                                                int *err, int jc) {
  unsigned long long t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (uint32_t i = 0;; ++i) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      return !*abort_flag;
    }
    if ((i & 255u) == 255u) {
      if (*abort_flag) return false;
      unsigned long long t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > kReadyWaitNs) break;
    }
  }
  set_error(err, kDevTimeout | (kSiteScanReady << 8) | ((jc & 0x7fff) << 16));
  *abort_flag = 1;
  return false;
}

// Wait used only while shutting down: bounded, ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kDrainPolls; ++i)
    if (mbar_try_wait(bar, parity)) return;
}

// One role's wait: its first thread polls, then the role's barrier publishes
// the outcome through a flag slot that alternates per call, so every thread
// of the role takes the same branch even if another role aborts meanwhile.
struct RoleSync {
  int id;            // named barrier id
  int *flags;        // 2 ints in shared memory
  int calls;         // waits made so far (same in every thread of the role)
  __device__ bool wait(bool elected, uint64_t *bar, uint32_t parity,
                       volatile int *abort_flag, int *err, int site, int jc) {
    int *slot = flags + (calls & 1);
    ++calls;
    if (elected) *slot = wait_ab(bar, parity, abort_flag, err, site, jc) ? 0 : 1;
    named_bar(id);
    return *reinterpret_cast<volatile int *>(slot) == 0;
  }
};

// CKPT: also store the checkpoints (a separate instance, so that the plain
// prefill's chunk loop carries no trace of them)
template <bool KDA, bool CKPT>
__global__ void __launch_bounds__(SCAN_THREADS, 1)
    chunk_scan_kernel(const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_q,
                      const __grid_constant__ CUtensorMap map_v,
                      const __grid_constant__ CUtensorMap map_T,
                      const __grid_constant__ CUtensorMap map_P,
                      const __grid_constant__ CUtensorMap map_W,
                      const __grid_constant__ CUtensorMap map_out,
                      const float *const *state_in, float *__restrict__ out, int H,
                      int Hqk, int qk_grouped, float scale, WsPtrs w, float *ckpt,
                      int ckpt_every, int max_ckpts, int wait_ready, int *err) {
  constexpr int DK = 128, DV = 128;
  // This grid is a programmatic dependent of the chunk prep. The work list
  // is complete when it starts (every prep CTA waited for it before this
  // grid could start), and nothing here reads what the prep writes except
  // the producer's copies of the prep's tiles: with wait_ready (the prep
  // still running beside this grid) each chunk's tiles are copied only after
  // their ready flags; otherwise the producer waits for the whole prep before
  // its first copy, while the other roles set up. (The recurrent tail is
  // launched normally and starts after this grid has completed.)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int vs = blockIdx.x & 1;  // value-column half
  const int h = (blockIdx.x >> 1) % H;
  const int hq = qk_grouped ? h / (H / Hqk) : h % Hqk;  // q/k head of value head h
  const int s = w.order[(blockIdx.x >> 1) / H];
  const int nch = w.seq_nch[s];
  if (nch == 0) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // see the end
    return;
  }
  const int chunk0 = w.seq_chunk0[s];
  // chunk j of the sequence starts at token tok0 + 64 j, and only the last
  // one can be partial (work-list layout): no per-chunk metadata loads
  const int tok0 = w.chunk_tok[chunk0], last_len = w.chunk_len[chunk0 + nch - 1];
  auto chunk_len_of = [&](int j) { return j == nch - 1 ? last_len : CH; };

  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = align1024(smem_raw);
  // full[st]: stage st landed; empty[st]: the products reading stage st are
  // done; E1: padding of a partial last chunk zeroed; E4: S0 in shared
  // memory; E5: X done; E6: D and D~ in shared memory; E7: S_acc done;
  // E8[j & 1]: O of chunk j done (one per parity: on the last chunk O can
  // finish before the previous chunk's O is waited for); E9: every product
  // issued so far done (shutdown).
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + SC_BARS);
  uint64_t *full = bars, *empty = bars + 2;  // [2] each
  uint64_t *bE1 = bars + 4, *bE4 = bars + 5, *bE5 = bars + 6, *bE6 = bars + 7,
           *bE7 = bars + 8, *bE8 = bars + 9;  // bE8 [2]
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + SC_TSLOT);
  __shared__ int abort_flag_s;
  __shared__ uint64_t bE9_s;
  volatile int *abort_flag = &abort_flag_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    abort_flag_s = 0;
    for (int b = 0; b < 11; ++b) mbar_init(&bars[b], 1);
    mbar_init(&bE9_s, 1);
    fence_mbar_init();
  }
  for (int e = tid; e < 8192 / 16; e += SCAN_THREADS) {  // zero tiles of both stages
    reinterpret_cast<uint4 *>(sm + ST_Z)[e] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4 *>(sm + ST_BYTES + ST_Z)[e] = make_uint4(0, 0, 0, 0);
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    int issued = 0;
    if (lane == 0) {
      prefetch_tmap(&map_k);
      prefetch_tmap(&map_q);
      prefetch_tmap(&map_v);
      prefetch_tmap(&map_T);
      prefetch_tmap(&map_P);
      prefetch_tmap(&map_W);
    }
    if (!wait_ready) asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int jc = 0; jc < nch; ++jc) {
      const int st = jc & 1;
      if (jc >= 2) {  // the products of chunk jc - 2 have released the stage
        int ok = 1;
        if (lane == 0) ok = wait_ab(&empty[st], ((jc >> 1) - 1) & 1, abort_flag, err, kSiteScanEmpty, jc);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      unsigned char *base = sm + st * ST_BYTES;
      const int gc = chunk0 + jc;
      const int t0 = tok0 + CH * jc, len = chunk_len_of(jc);
      const int trow = (gc * H + h) * CH;
      if (wait_ready) {  // the tiles of chunk gc, head h are written
        int ok = 1;
        if (lane == 0) ok = wait_ready_flag(w.ready + gc * H + h, abort_flag, err, jc);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      if (lane == 0) {
        uint64_t *fb = &full[st];
        mbar_arrive_expect_tx(fb, ST_TX);
        if constexpr (KDA) {  // K~ and Q^ tiles from the workspace
          tma_load_2d(base + ST_K, &map_k, 0, trow, fb);
          tma_load_2d(base + ST_K + 8192, &map_k, 64, trow, fb);
          tma_load_2d(base + ST_WQ + 8192, &map_q, 0, trow, fb);
          tma_load_2d(base + ST_WQ + 16384 + 8192, &map_q, 64, trow, fb);
        } else {  // raw K and Q rows of the packed token tensors
          tma_load_3d(base + ST_K, &map_k, 0, hq, t0, fb);
          tma_load_3d(base + ST_K + 8192, &map_k, 64, hq, t0, fb);
          tma_load_3d(base + ST_WQ + 8192, &map_q, 0, hq, t0, fb);
          tma_load_3d(base + ST_WQ + 16384 + 8192, &map_q, 64, hq, t0, fb);
        }
        tma_load_2d(base + ST_WQ, &map_W, 0, trow, fb);
        tma_load_2d(base + ST_WQ + 16384, &map_W, 64, trow, fb);
        tma_load_3d(base + ST_V, &map_v, NV * vs, h, t0, fb);
        tma_load_2d(base + ST_T, &map_T, 0, trow, fb);
        tma_load_2d(base + ST_P, &map_P, 0, trow, fb);
        bulk_g2s(base + ST_G, w.gs + ((long long)gc * H + h) * 256, 1024, fb);
        if (jc + 2 < nch) {  // chunk jc + 2 loads into this stage two chunks later: warm L2
          const int gp = gc + 2, tp = tok0 + CH * (jc + 2), prow = (gp * H + h) * CH;
          if constexpr (KDA) {
            tma_prefetch_2d(&map_k, 0, prow);
            tma_prefetch_2d(&map_k, 64, prow);
            tma_prefetch_2d(&map_q, 0, prow);
            tma_prefetch_2d(&map_q, 64, prow);
          } else {
            tma_prefetch_3d(&map_k, 0, hq, tp);
            tma_prefetch_3d(&map_k, 64, hq, tp);
            tma_prefetch_3d(&map_q, 0, hq, tp);
            tma_prefetch_3d(&map_q, 64, hq, tp);
          }
          tma_prefetch_2d(&map_W, 0, prow);
          tma_prefetch_2d(&map_W, 64, prow);
          tma_prefetch_3d(&map_v, NV * vs, h, tp);
          tma_prefetch_2d(&map_T, 0, prow);
          tma_prefetch_2d(&map_P, 0, prow);
        }
      }
      ++issued;
      if (len < CH) {
        // Only the last chunk can be partial. Its padding rows hold the next
        // tokens, whose values must not reach this chunk's results even as
        // 0 * inf: zero those of V (rows of T V) and, for GDA, of the raw K
        // (rows of K^T D~). Padding rows of Q only reach outputs that are
        // not stored; KDA's K~ and Q^ come from the workspace, already padded.
        int ok = 1;
        if (lane == 0) ok = wait_ab(&full[st], (jc >> 1) & 1, abort_flag, err, kSiteScanPad, jc);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        constexpr int per_row = KDA ? 8 : 24;  // 16-byte pieces per padding row
        for (int e = lane; e < (CH - len) * per_row; e += 32) {
          const int r = len + e / per_row, c = e % per_row;
          unsigned char *dst;
          if (c < 8)
            dst = base + ST_V + r * 128 + c * 16;
          else
            dst = base + ST_K + ((c - 8) >> 3) * 8192 + r * 128 + ((c - 8) & 7) * 16;
          *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(bE1);
      }
    }
    // copies still in flight (after an abort) land before the CTA exits
    if (lane == 0)
      for (int j = issued >= 2 ? issued - 2 : 0; j < issued; ++j)
        drain_wait(&full[j & 1], (j >> 1) & 1);
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ mma
    if (lane == 0) {
      constexpr uint32_t id_x = idesc_bf16_f32(128, 64, false, true);
      constexpr uint32_t id_s = idesc_bf16_f32(128, 64, true, true);
      // stage of chunk j usable: landed, or for a partial last chunk padded
      auto stage_bar = [&](int j, uint32_t *parity) -> uint64_t * {
        if (chunk_len_of(j) < CH) {
          *parity = 0;
          return bE1;
        }
        *parity = (j >> 1) & 1;
        return &full[j & 1];
      };
      // X(j) = [T; 0] V (state-free) into X buffer j % 3
      // shared-memory descriptors of both stages, built once; a K step
      // advances the start-address field (bytes >> 4) by a plain add
      const uint32_t sm0 = smem_u32(sm);
      auto kdesc = [&](uint32_t off) { return sdesc_kmajor(sm0 + off); };
      auto mdesc = [&](uint32_t off, uint32_t lbo) { return sdesc_mnmajor(sm0 + off, lbo); };
      const uint64_t dT[2] = {kdesc(ST_T), kdesc(ST_BYTES + ST_T)};
      const uint64_t dV[2] = {mdesc(ST_V, 8192), mdesc(ST_BYTES + ST_V, 8192)};
      const uint64_t dWQ[2] = {kdesc(ST_WQ), kdesc(ST_BYTES + ST_WQ)};
      const uint64_t dK[2] = {mdesc(ST_K, 8192), mdesc(ST_BYTES + ST_K, 8192)};
      const uint64_t dZ[2] = {kdesc(ST_Z), kdesc(ST_BYTES + ST_Z)};
      const uint64_t dS = mdesc(SC_S, 8192);
      const uint64_t dD[2] = {mdesc(SC_D, 8192), mdesc(SC_D + 8192, 8192)};
      const uint64_t dDT = mdesc(SC_DT, 8192);
      auto issue_x1 = [&](int j) {
        const uint32_t colx = COL_X0 + 64u * (uint32_t)(j % 3);
        tc_fence_after();
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          umma_bf16(tbase + colx, dT[j & 1] + 2 * k4, dV[j & 1] + 128 * k4, id_x, k4 > 0);
      };
      // X(j) += [-W; Q] S0, once S0 is in shared memory
      auto issue_x2 = [&](int j) -> bool {
        const uint32_t colx = COL_X0 + 64u * (uint32_t)(j % 3);
        if (!wait_ab(bE4, j & 1, abort_flag, err, kSiteScanS0, j)) return false;
        tc_fence_after();
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8)
          umma_bf16(tbase + colx, dWQ[j & 1] + (k8 >> 2) * 1024 + (k8 & 3) * 2, dS + 128 * k8,
                    id_x, true);
        umma_commit(bE5);
        return true;
      };
      uint32_t par;
      uint64_t *sb = stage_bar(0, &par);
      bool ok = wait_ab(sb, par, abort_flag, err, kSiteScanStage, 0);
      if (ok) {
        issue_x1(0);
        ok = issue_x2(0);
      }
      for (int jc = 0; ok && jc < nch; ++jc) {
        const int st = jc & 1;
        // D(jc) in shared memory (the next chunk's state-free product is issued
        // only behind this chunk's S and O products, so that nothing stands
        // between D(jc) and S(jc) in the in-order tensor pipe)
        if (!wait_ab(bE6, jc & 1, abort_flag, err, kSiteScanD, jc)) break;
        tc_fence_after();
        // S_acc = K~^T D~
        const uint64_t dB = KDA ? dD[jc & 1] : dDT;
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          umma_bf16(tbase + COL_S, dK[st] + 128 * k4, dB + 128 * k4, id_s, k4 > 0);
        umma_commit(bE7);
        // O = [0; P] D, then the stage is free
        const uint32_t colo = COL_O0 + 64u * (jc & 1);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          umma_bf16(tbase + colo, dZ[st] + 2 * k4, dD[jc & 1] + 128 * k4, id_x, k4 > 0);
        umma_commit(&bE8[jc & 1]);
        umma_commit(&empty[st]);
        if (jc + 1 < nch) {
          uint64_t *nb = stage_bar(jc + 1, &par);
          if (!wait_ab(nb, par, abort_flag, err, kSiteScanStage, jc + 1)) break;
          issue_x1(jc + 1);
          if (!issue_x2(jc + 1)) break;
        }
      }
      umma_commit(&bE9_s);  // tracks every product issued above
      drain_wait(&bE9_s, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ state
    const int i = 32 * (warp & 3) + lane;  // key row / TMEM lane
    const int ch = warp >> 2;              // which CPT of the CTA's 64 columns
    const int c0 = CPT * ch;               // first of them
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    RoleSync rs{1, reinterpret_cast<int *>(sm + SC_RFLAGS), 0};
    float Sm[CPT];
    {
      const float *src = state_in[s];
      if (src) {
        const float4 *p4 = reinterpret_cast<const float4 *>(
            src + ((long long)h * DK + i) * DV + NV * vs + c0);
#pragma unroll
        for (int e = 0; e < CPT / 4; ++e) {
          const float4 v4 = p4[e];
          Sm[4 * e] = v4.x; Sm[4 * e + 1] = v4.y; Sm[4 * e + 2] = v4.z; Sm[4 * e + 3] = v4.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < CPT; ++e) Sm[e] = 0.f;
      }
#pragma unroll
      for (int q = 0; q < PPT; ++q)
        *reinterpret_cast<uint4 *>(sm + SC_S + chunk16(i, PPT * ch + q)) = pack8(Sm + 8 * q);
    }
    fence_proxy_async();
    named_bar(1);
    if (tid == 0) mbar_arrive(bE4);
    // outputs of chunk j: rows 64..127 of X (Q S0) and of O (P D). A full
    // chunk goes through a shared-memory tile and two TMA stores (thread 0
    // issues them; it waits for the previous pair to have read the tile
    // before the barrier that precedes the next writes); a partial last
    // chunk is stored row by row, so no token past its end is touched.
    auto store_out = [&](int j, float qf) {
      const int t0 = tok0 + CH * j, len = chunk_len_of(j);
      if ((warp & 3) >= 2) {
        const int r = i - CH;
        float xv[CPT], ov[CPT];
        tmem_ld_cpt(tbase + lane_off + COL_X0 + 64u * (uint32_t)(j % 3) + c0, xv);
        tmem_ld_cpt(tbase + lane_off + COL_O0 + 64u * (uint32_t)(j & 1) + c0, ov);
        float4 o4[CPT / 4];
#pragma unroll
        for (int u = 0; u < CPT / 4; ++u)
          o4[u] = make_float4(scale * fmaf(qf, xv[4 * u], ov[4 * u]),
                              scale * fmaf(qf, xv[4 * u + 1], ov[4 * u + 1]),
                              scale * fmaf(qf, xv[4 * u + 2], ov[4 * u + 2]),
                              scale * fmaf(qf, xv[4 * u + 3], ov[4 * u + 3]));
        if (len == CH) {
          // staging tile c0 / 32 (32 columns, 128-byte rows), pieces from (c0 % 32) / 4
          unsigned char *tile = sm + SC_OUT + (c0 >> 5) * 8192 + r * 128;
          const int pc0 = (c0 & 31) >> 2;
#pragma unroll
          for (int u = 0; u < CPT / 4; ++u)
            *reinterpret_cast<float4 *>(tile + (((pc0 + u) ^ (r & 7)) << 4)) = o4[u];
        } else if (r < len) {
          float4 *dst = reinterpret_cast<float4 *>(out + ((long long)(t0 + r) * H + h) * DV +
                                                   NV * vs + c0);
#pragma unroll
          for (int u = 0; u < CPT / 4; ++u) dst[u] = o4[u];
        }
      }
      if (len == CH) {
        fence_proxy_async();
        named_bar(1);
        if (tid == 0) {
          tma_store_3d(&map_out, NV * vs, h, t0, sm + SC_OUT);
          tma_store_3d(&map_out, NV * vs + 32, h, t0, sm + SC_OUT + 8192);
          bulk_commit();
        }
      }
    };
    for (int jc = 0; jc < nch; ++jc) {
      const int st = jc & 1;
      const uint32_t colx = COL_X0 + 64u * (uint32_t)(jc % 3);
      if (!rs.wait(tid == 0, bE5, jc & 1, abort_flag, err, kSiteScanX, jc)) break;
      tc_fence_after();
      // gate factors of this chunk: the stage landed before X could finish;
      // the wait gives each thread its own view of it (never blocks here)
      drain_wait(&full[st], (jc >> 1) & 1);
      const float *gs = reinterpret_cast<const float *>(sm + st * ST_BYTES + ST_G);
      const float gcs = gs[128 + i];
      float dec = 1.f, qf = 1.f;
      if constexpr (!KDA) {
        if (i < CH) dec = gs[64 + i];
        else qf = gs[i - CH];
      }
      // D rows (TMEM lanes 0..63) -> D and D~ tiles
      if ((warp & 3) < 2) {
        float dv[CPT];
        tmem_ld_cpt(tbase + lane_off + colx + c0, dv);
        unsigned char *dbuf = sm + SC_D + (jc & 1) * 8192;
#pragma unroll
        for (int q = 0; q < PPT; ++q)
          *reinterpret_cast<uint4 *>(dbuf + chunk16(i, PPT * ch + q)) = pack8(dv + 8 * q);
        if constexpr (!KDA) {
#pragma unroll
          for (int e = 0; e < CPT; ++e) dv[e] *= dec;
#pragma unroll
          for (int q = 0; q < PPT; ++q)
            *reinterpret_cast<uint4 *>(sm + SC_DT + chunk16(i, PPT * ch + q)) =
                pack8(dv + 8 * q);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      named_bar(1);
      if (tid == 0) mbar_arrive(bE6);
      // state update, handed to the next chunk
      if (!rs.wait(tid == 0, bE7, jc & 1, abort_flag, err, kSiteScanS, jc)) break;
      tc_fence_after();
      {
        float v[CPT];
        tmem_ld_cpt(tbase + lane_off + COL_S + c0, v);
#pragma unroll
        for (int u = 0; u < CPT; ++u) Sm[u] = fmaf(gcs, Sm[u], v[u]);
      }
#pragma unroll
      for (int q = 0; q < PPT; ++q)
        *reinterpret_cast<uint4 *>(sm + SC_S + chunk16(i, PPT * ch + q)) = pack8(Sm + 8 * q);
      fence_proxy_async();
      tc_fence_before();
      named_bar(1);
      if (tid == 0 && jc + 1 < nch) mbar_arrive(bE4);
      // checkpoint: the state after a full chunk that ends on a multiple of
      // ckpt_every tokens (chunks start at multiples of 64 in the sequence)
      if (CKPT && chunk_len_of(jc) == CH) {
        const int pos = (jc + 1) * CH, c = pos / ckpt_every - 1;
        if (pos % ckpt_every == 0 && c < max_ckpts)
          store_rows_cpt(Sm,
                         ckpt + ((((long long)s * max_ckpts + c) * H + h) * DK +
                                 32 * (warp & 3)) * DV + NV * vs + c0,
                         DV, lane);
      }
      // this chunk's outputs, while the next chunk's X is computed (the
      // staging tile is free once thread 0's earlier stores have read it)
      if (tid == 0) bulk_wait_read();
      if (!rs.wait(tid == 0, &bE8[jc & 1], (jc >> 1) & 1, abort_flag, err, kSiteScanO, jc)) break;
      tc_fence_after();
      store_out(jc, qf);
      tc_fence_before();
    }
    if (tid == 0) bulk_wait_all();
    if (!*abort_flag) {  // state after the chunked part: read by the tail, or the slot itself
      float4 *dst = reinterpret_cast<float4 *>(
          w.states + (((long long)s * H + h) * DK + i) * DV + NV * vs + c0);
#pragma unroll
      for (int e = 0; e < CPT / 4; ++e)
        dst[e] = make_float4(Sm[4 * e], Sm[4 * e + 1], Sm[4 * e + 2], Sm[4 * e + 3]);
    }
  }
  // Only the producer may have waited for the prep so far (with wait_ready,
  // nobody): every thread waits for it here (it has long finished), so that
  // the grid's completion implies the prep's and whatever runs after this
  // grid in the stream finds the prep complete as well.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    __syncwarp();
    tmem_dealloc(tbase, 512);
  }
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

// bf16 [rows][width] workspace tiles (width 64 or 128); 64 x 64 boxes,
// 128-byte swizzle
bool map_rows(CUtensorMap *m, const void *base, long long rows, int width) {
  const cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)width * 2};
  const cuuint32_t box[2] = {64, 64}, es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [Ntok][H][D] viewed as (D, H, Ntok); 32 x 1 x 64 boxes, 128-byte swizzle
bool map_out_f32(CUtensorMap *m, void *base, int ntok, int H, int D) {
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)ntok};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)H * D * 4};
  const cuuint32_t box[3] = {32, 1, 64}, es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Opt-in shared-memory sizes and the SM count, once per device.
std::mutex g_attr_mu;
bool g_attr_done[64] = {};
int g_num_sms[64] = {};

cudaError_t set_attributes(int *num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (g_attr_done[dev]) {
    *num_sms = g_num_sms[dev];
    return cudaSuccess;
  }
  e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  *num_sms = g_num_sms[dev];
  const void *fns[] = {(const void *)chunk_prep_kernel<false>,
                       (const void *)chunk_prep_kernel<true>};
  for (const void *f : fns) {
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, PREP_SMEM_KDA);
    if (e != cudaSuccess) return e;
    // the whole unified L1 as shared memory, so that four CTAs fit per SM
    e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  const void *sfns[] = {(const void *)chunk_scan_kernel<false, false>,
                        (const void *)chunk_scan_kernel<true, false>,
                        (const void *)chunk_scan_kernel<false, true>,
                        (const void *)chunk_scan_kernel<true, true>};
  for (const void *f : sfns) {
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SCAN_SMEM);
    if (e != cudaSuccess) return e;
  }
  g_attr_done[dev] = true;
  return cudaSuccess;
}

}  // namespace

// The public size query has no gate mode, so it returns the larger (KDA)
// layout; a GDA call needs less and fits in it.
size_t chunked_workspace_size(int n_seqs, int total_tokens, int H, int Dk, int Dv, bool bf16) {
  return ws_layout(n_seqs, total_tokens, H, Dk, Dv, true, tensor_core_route(bf16, Dk, Dv)).total;
}

size_t chunked_workspace_need(int n_seqs, int total_tokens, int H, int Dk, int Dv, bool kda,
                              bool bf16) {
  return ws_layout(n_seqs, total_tokens, H, Dk, Dv, kda, tensor_core_route(bf16, Dk, Dv)).total;
}

// fp32 inputs and head sizes other than 128: every token of every sequence
// through the recurrent kernel (which also writes the slots), from the work
// list with no chunked part.
static cudaError_t launch_token_loop(const ChunkedArgs &a, cudaStream_t stream) {
  const WsLayout lay = ws_layout(a.n_seqs, a.total_tokens, a.H, a.Dk, a.Dv, a.kda, false);
  if (a.workspace_bytes < lay.total) return cudaErrorInvalidValue;
  const WsPtrs w = ws_ptrs(a.workspace, lay);
  worklist_kernel<<<1, WL_THREADS, 0, stream>>>(a.cu_seqlens, a.n_seqs, a.total_tokens,
                                                0x7fffffff, a.H, 0, a.state_in, w, 0, a.err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  RecurrentArgs r{};
  r.q = a.q; r.k = a.k; r.v = a.v; r.g = a.g; r.beta = a.beta;
  r.state_in = w.state_ptrs;
  r.slots = a.slots; r.out = a.out;
  r.tok_start = w.tail_start; r.seq_len = w.tail_len;
  r.n_seqs = a.n_seqs; r.T = 0; r.H = a.H; r.Dk = a.Dk; r.Dv = a.Dv;
  r.Hqk = a.Hqk > 0 ? a.Hqk : a.H; r.qk_grouped = a.qk_grouped;
  r.n_slots = a.n_slots; r.kda = a.kda; r.bf16 = a.bf16; r.scale = a.scale; r.err = a.err;
  r.ckpt = a.ckpt; r.pos0 = w.tail_pos; r.ckpt_every = a.ckpt_every; r.max_ckpts = a.max_ckpts;
  r.long_chains = true;
  return launch_recurrent(r, stream);
}

cudaError_t launch_chunked(const ChunkedArgs &a, cudaStream_t stream) {
  if (!tensor_core_route(a.bf16, a.Dk, a.Dv)) return launch_token_loop(a, stream);
  if (!encode_fn()) return cudaErrorNotSupported;
  int num_sms = 0;
  cudaError_t e = set_attributes(&num_sms);
  if (e != cudaSuccess) return e;
  const WsLayout lay = ws_layout(a.n_seqs, a.total_tokens, a.H, a.Dk, a.Dv, a.kda);
  if (a.workspace_bytes < lay.total) return cudaErrorInvalidValue;
  const WsPtrs w = ws_ptrs(a.workspace, lay);
  const long long state_elems = (long long)a.H * a.Dk * a.Dv;
  // With one slot, the slot is the final state: the chunked part takes every
  // token, the scan writes its final state straight into the slot (same
  // [N][H][D_k][D_v] layout as the workspace states), and no tail runs.
  const bool direct = a.n_slots == 1;
  WsPtrs ws = w;
  if (direct) ws.states = a.slots;

  worklist_kernel<<<1, WL_THREADS, 0, stream>>>(a.cu_seqlens, a.n_seqs, a.total_tokens,
                                                direct ? 0 : a.n_slots, a.H, state_elems,
                                                a.state_in, w, lay.max_chunks * a.H, a.err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  if (a.total_tokens > 0) {
    CUtensorMap mq, mk, mv, mT, mP, mW, mQh, mKt, mo;
    const long long trows = lay.max_chunks * a.H * CH;
    if (trows >= (1LL << 31)) return cudaErrorInvalidValue;  // TMA row coordinates are int32
    const int Hqk = a.Hqk > 0 ? a.Hqk : a.H;
    if (!map_tokens(&mq, a.q, a.total_tokens, Hqk, a.Dk) ||
        !map_tokens(&mk, a.k, a.total_tokens, Hqk, a.Dk) ||
        !map_tokens(&mv, a.v, a.total_tokens, a.H, a.Dv) ||
        !map_rows(&mT, w.T, trows, CH) || !map_rows(&mP, w.P, trows, CH) ||
        !map_rows(&mW, w.W, trows, a.Dk) ||
        !map_out_f32(&mo, a.out, a.total_tokens, a.H, a.Dv))
      return cudaErrorInvalidValue;
    if (a.kda && (!map_rows(&mQh, w.Qh, trows, a.Dk) || !map_rows(&mKt, w.Kt, trows, a.Dk)))
      return cudaErrorInvalidValue;
    const int qg = a.qk_grouped ? 1 : 0;
    // persistent prep CTAs: as many as fit at once (registers allow three per
    // SM for per-row gates, four for scalar gates; four use all of TMEM)
    const int per_sm = a.kda ? 3 : 4;
    // The prep and the scan are programmatic dependent launches behind the
    // work list: each one's launch and set-up overlap the previous kernel's
    // drain, and each waits (griddepcontrol.wait) before reading what that
    // one wrote. The work list and the recurrent tail are launched normally
    // (programmatic launches of those two measured 4-5% slower).
    auto launch_prep = [&](int publish, int handoff) -> cudaError_t {
      const dim3 g3((unsigned)std::min<long long>(lay.max_chunks * a.H,
                                                  (long long)num_sms * per_sm));
      if (a.kda)
        return launch_pdl(chunk_prep_kernel<true>, g3, dim3(PREP_THREADS), PREP_SMEM_KDA,
                          stream, mq, mk, a.g, a.beta, a.H, Hqk, qg, w, publish, handoff,
                          num_sms, a.err);
      return launch_pdl(chunk_prep_kernel<false>, g3, dim3(PREP_THREADS), PREP_SMEM, stream, mq,
                        mk, a.g, a.beta, a.H, Hqk, qg, w, publish, handoff, num_sms, a.err);
    };
    const long long scan_grid = (long long)a.n_seqs * a.H * 2;
    auto launch_scan = [&](int wait_ready) -> cudaError_t {
      const dim3 sg((unsigned)scan_grid), st(SCAN_THREADS);
      const int ce = a.ckpt ? a.ckpt_every : 1, cm = a.ckpt ? a.max_ckpts : 0;
      if (a.kda && a.ckpt)
        return launch_pdl(chunk_scan_kernel<true, true>, sg, st, SCAN_SMEM, stream, mKt, mQh, mv,
                          mT, mP, mW, mo, a.state_in, a.out, a.H, Hqk, qg, a.scale, ws, a.ckpt,
                          ce, cm, wait_ready, a.err);
      if (a.kda)
        return launch_pdl(chunk_scan_kernel<true, false>, sg, st, SCAN_SMEM, stream, mKt, mQh,
                          mv, mT, mP, mW, mo, a.state_in, a.out, a.H, Hqk, qg, a.scale, ws,
                          (float *)nullptr, ce, cm, wait_ready, a.err);
      if (a.ckpt)
        return launch_pdl(chunk_scan_kernel<false, true>, sg, st, SCAN_SMEM, stream, mk, mq, mv,
                          mT, mP, mW, mo, a.state_in, a.out, a.H, Hqk, qg, a.scale, ws, a.ckpt,
                          ce, cm, wait_ready, a.err);
      return launch_pdl(chunk_scan_kernel<false, false>, sg, st, SCAN_SMEM, stream, mk, mq, mv,
                        mT, mP, mW, mo, a.state_in, a.out, a.H, Hqk, qg, a.scale, ws,
                        (float *)nullptr, ce, cm, wait_ready, a.err);
    };
    // The prep runs first, on every SM. When the scan (one CTA per SM) needs
    // at most half of the SMs, it is launched right behind the prep as a
    // programmatic dependent ("hand-off"): the prep CTAs on as many SMs as the
    // scan has CTAs leave at once, the scan's CTAs take those SMs and wait for
    // each tile's ready flag while the rest of the prep goes on. The scan can start only once every prep CTA has started, and the
    // prep never waits on the scan, so the prep always finishes. With more
    // scan CTAs the prep left on the other SMs cannot keep up with the chains
    // (a schedule model with the measured rates puts the break-even between
    // 80 and 96 scan CTAs for either gate mode, and a 128-CTA scan 3x slower
    // beside the prep than after it), so the scan simply runs after the prep.
    const bool handoff = 2 * scan_grid <= num_sms;
    if ((e = launch_prep(handoff ? 1 : 0, handoff ? (int)scan_grid : 0)) != cudaSuccess)
      return e;
    if ((e = launch_scan(handoff ? 1 : 0)) != cudaSuccess) return e;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }

  if (direct) return cudaSuccess;
  // the last n_slots tokens of every sequence: token loop with snapshots
  RecurrentArgs r{};
  r.q = a.q; r.k = a.k; r.v = a.v; r.g = a.g; r.beta = a.beta;
  r.state_in = w.state_ptrs;
  r.slots = a.slots; r.out = a.out;
  r.tok_start = w.tail_start; r.seq_len = w.tail_len;
  r.n_seqs = a.n_seqs; r.T = 0; r.H = a.H; r.Dk = a.Dk; r.Dv = a.Dv;
  r.Hqk = a.Hqk > 0 ? a.Hqk : a.H; r.qk_grouped = a.qk_grouped;
  r.n_slots = a.n_slots; r.kda = a.kda; r.bf16 = true; r.scale = a.scale; r.err = a.err;
  r.ckpt = a.ckpt; r.pos0 = w.tail_pos; r.ckpt_every = a.ckpt_every; r.max_ckpts = a.max_ckpts;
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
// every GPU that loads this library's chunked kernels keeps it (256 MiB)
// until the process exits.
namespace gdn {

constexpr size_t kStaticScratchBytes = size_t(256) << 20;
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
  *need = chunked_workspace_need(a.n_seqs, a.total_tokens, a.H, a.Dk, a.Dv, a.kda, a.bf16);
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
