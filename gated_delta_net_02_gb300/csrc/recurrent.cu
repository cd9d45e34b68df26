// recurrent.cu -- token-loop GDN kernel for decode, speculative verify and
// the snapshot tail of chunked prefill.
//
// Computes, per (sequence, head, token), decay -> read -> correct -> write ->
// query on a D_k x D_v fp32 state held in registers, and writes the state
// after each of the last K tokens to its snapshot slot (gated delta rule of
// "Gated Delta Networks", Yang, Kautz, Hatamizadeh, ICLR 2025; GDA/KDA gates
// of "metal : add GDN kernel (#20361)" and the K-slot snapshots of "metal: add
// GDN partial rollback", llama.cpp / koboldcpp commit pages).
//
// Design (sm_103a):
//  * The state columns of a head are independent given k, q, the gate and
//    beta, so each warp owns a slice of WCOLS columns over all D_k rows
//    (columns sharded across warps, as in "CUDA: AR gated delta net
//    improvements (#20391)"). Lane = (row group rg, column group cg): a lane
//    holds 4 adjacent columns of rows rg, rg+ROWG, rg+2*ROWG, ... so one
//    128-bit load of a warp covers ROWG rows x 4*CG contiguous floats.
//  * S^T k and S^T q reduce within the lane over its rows, then across the
//    ROWG row groups with xor-shuffles: no shared memory, no block barrier.
//  * The reduction order is fixed by (D_k, D_v) alone, never by T, K or the
//    grid, so re-running a prefix reproduces every snapshot bit for bit.
//  * q/k/v rows of a tile of TT tokens are staged in shared memory by bulk
//    (TMA) copies on an mbarrier, double-buffered, and issued before the
//    state loads so both are in flight together.
//  * State loads bypass L1 (streamed once); the decay is applied in the read
//    pass; outputs and snapshots are 128-bit stores.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

struct RecParams {
  const void *q, *k, *v;
  const float *g, *beta;
  const float *const *state_in;
  float *slots, *out;
  const int *tok_start, *seq_len;
  long long slots_elems;
  int n_seqs, T, H, n_slots;
  int Hqk, qk_grouped;  // q/k heads and the value-head -> q/k-head map
  float *ckpt;          // optional checkpoints, [n_seqs][max_ckpts][H][Dk][Dv]
  int pdl;              // launched programmatically (tok_start, seq_len, ckpt NULL)
  int long_chains;      // see RecurrentArgs
  int host_io;          // see RecurrentArgs
  const int *pos0;      // position of each sequence's first token (NULL = 0)
  int ckpt_every, max_ckpts;
  float scale;
  int *err;
};

template <int DK_, int DV_, int ROWG_, int WPC_, bool KDA_, typename Tin_>
struct RecCfg {
  static constexpr int DK = DK_, DV = DV_, ROWG = ROWG_, WPC = WPC_;
  static constexpr bool KDA = KDA_;
  using Tin = Tin_;
  static constexpr int CG = 32 / ROWG;       // lanes across columns
  static constexpr int WCOLS = 4 * CG;       // columns per warp
  static constexpr int RPT = DK / ROWG;      // rows per thread
  static constexpr int CCOLS = WCOLS * WPC;  // columns per CTA
  static constexpr int CTAS_PER_HEAD = DV / CCOLS;
  static constexpr int NT = 32 * WPC;
  static constexpr int TT = 8;               // tokens per staged tile
  // raw staging (one buffer): q[TT][DK], k[TT][DK], v[TT][CCOLS] in Tin,
  // then (KDA) g[TT][DK] fp32
  static constexpr int RAW_QK = TT * DK * (int)sizeof(Tin);
  static constexpr int RAW_V = TT * CCOLS * (int)sizeof(Tin);
  static constexpr int RAW_G = KDA ? TT * DK * 4 : 0;
  static constexpr int RAW_BYTES = 2 * RAW_QK + RAW_V + RAW_G;
  // converted fp32: q, k [TT][DK], v [TT][CCOLS], alpha [TT][DK or 1], beta
  static constexpr int F_ALPHA = KDA ? DK : 1;
  static constexpr int F_FLOATS = TT * (2 * DK + CCOLS + F_ALPHA + 1);
  static constexpr size_t SMEM = 2 * RAW_BYTES + F_FLOATS * 4 + 64;
  // 16-byte pieces of one token's raw rows (q, k, v, then the KDA gates) and
  // of a whole tile per thread, when the tile is read with ordinary loads
  static constexpr int P_QK = DK * (int)sizeof(Tin) / 16;
  static constexpr int P_V = CCOLS * (int)sizeof(Tin) / 16;
  static constexpr int P_G = KDA ? DK * 4 / 16 : 0;
  static constexpr int P_TOK = 2 * P_QK + P_V + P_G;
  static constexpr int P_THREAD = (TT * P_TOK + NT - 1) / NT;
  static_assert(ROWG * CG == 32, "lane split");
  static_assert(DK % ROWG == 0 && DV % CCOLS == 0, "shape split");
  static_assert(RAW_QK % 16 == 0 && RAW_V % 16 == 0, "bulk copy alignment");
};

// One token on a lane's slice of the state (rows rg + ROWG*m, 4 columns):
// decay, read u = (aS)^T k, correct d = beta (v - u), write S += k d^T,
// query o = S^T q. Returns the lane's 4 outputs summed over the row groups
// (before the output scale). The order of the arithmetic is fixed by the
// configuration alone, never by T, K or the grid.
template <class C>
__device__ __forceinline__ float4 token_update(float4 (&st)[C::RPT], const float *kr,
                                               const float *qr, const float *ar, float a_h,
                                               float beta, float4 vv, int rg) {
  constexpr int ROWG = C::ROWG, CG = C::CG, RPT = C::RPT;
  float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
  for (int m = 0; m < RPT; ++m) {
    const int i = rg + ROWG * m;
    float a = a_h;
    if constexpr (C::KDA) a = ar[i];
    const float kv = kr[i];
    st[m].x *= a; st[m].y *= a; st[m].z *= a; st[m].w *= a;
    u0 = fmaf(st[m].x, kv, u0);
    u1 = fmaf(st[m].y, kv, u1);
    u2 = fmaf(st[m].z, kv, u2);
    u3 = fmaf(st[m].w, kv, u3);
  }
#pragma unroll
  for (int off = CG; off < 32; off <<= 1) {
    u0 += __shfl_xor_sync(0xffffffffu, u0, off);
    u1 += __shfl_xor_sync(0xffffffffu, u1, off);
    u2 += __shfl_xor_sync(0xffffffffu, u2, off);
    u3 += __shfl_xor_sync(0xffffffffu, u3, off);
  }
  const float d0 = beta * (vv.x - u0), d1 = beta * (vv.y - u1);
  const float d2 = beta * (vv.z - u2), d3 = beta * (vv.w - u3);
  float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
  for (int m = 0; m < RPT; ++m) {
    const int i = rg + ROWG * m;
    const float kv = kr[i], qv = qr[i];
    st[m].x = fmaf(kv, d0, st[m].x);
    st[m].y = fmaf(kv, d1, st[m].y);
    st[m].z = fmaf(kv, d2, st[m].z);
    st[m].w = fmaf(kv, d3, st[m].w);
    o0 = fmaf(st[m].x, qv, o0);
    o1 = fmaf(st[m].y, qv, o1);
    o2 = fmaf(st[m].z, qv, o2);
    o3 = fmaf(st[m].w, qv, o3);
  }
#pragma unroll
  for (int off = CG; off < 32; off <<= 1) {
    o0 += __shfl_xor_sync(0xffffffffu, o0, off);
    o1 += __shfl_xor_sync(0xffffffffu, o1, off);
    o2 += __shfl_xor_sync(0xffffffffu, o2, off);
    o3 += __shfl_xor_sync(0xffffffffu, o3, off);
  }
  return make_float4(o0, o1, o2, o3);
}

// CKPT: also store the checkpoints of p.ckpt (a separate instance, so the
// decode and verify instances carry no trace of it). HOSTIO: the token tiles
// are read with ordinary loads instead of bulk copies, so q, k, v, g, beta
// (and out, always written with ordinary stores) may be page-locked host
// memory mapped into the device's address space. The HOSTIO instance is
// held to 512 threads' worth of CTAs per SM (the register budget the other
// instances reach on their own); a minimum of 0 leaves those unbounded.
template <class C, bool CKPT, bool HOSTIO = false>
__global__ void __launch_bounds__(C::NT, HOSTIO ? 512 / C::NT : 0)
    recurrent_kernel(const RecParams p) {
  using Tin = typename C::Tin;
  constexpr int DK = C::DK, DV = C::DV, ROWG = C::ROWG, CG = C::CG;
  constexpr int RPT = C::RPT, TT = C::TT, CCOLS = C::CCOLS;

  // The next kernel of the stream (if launched programmatically) may be
  // scheduled once every block of this one has started.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ __align__(128) unsigned char smem[];
  float *fq = reinterpret_cast<float *>(smem + 2 * C::RAW_BYTES);
  float *fk = fq + TT * DK;
  float *fv = fk + TT * DK;
  float *fa = fv + TT * CCOLS;
  float *fb = fa + TT * C::F_ALPHA;
  uint64_t *bar = reinterpret_cast<uint64_t *>(fb + TT + (TT & 1));
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int rg = lane / CG, cg = lane % CG;

  const int part = blockIdx.x % C::CTAS_PER_HEAD;
  const int sh = blockIdx.x / C::CTAS_PER_HEAD;
  const int h = sh % p.H;
  const int s = sh / p.H;
  if (s >= p.n_seqs) return;
  const int hq = p.qk_grouped ? h / (p.H / p.Hqk) : h % p.Hqk;  // q/k head of h
  const int T_s = p.seq_len ? p.seq_len[s] : p.T;
  const long long t0 = p.tok_start ? (long long)p.tok_start[s] : (long long)s * p.T;
  if (T_s <= 0) return;

  const int col_base = part * CCOLS;
  const int wcol = col_base + warp * C::WCOLS + cg * 4;  // first column of lane
  const int ntiles = (T_s + TT - 1) / TT;

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();

  const Tin *q = static_cast<const Tin *>(p.q);
  const Tin *k = static_cast<const Tin *>(p.k);
  const Tin *v = static_cast<const Tin *>(p.v);

  // Warp 0 stages tile `tile` into raw buffer `b`: lane r copies token r.
  auto issue = [&](int tile, int b) {
    const int n = min(TT, T_s - tile * TT);
    unsigned char *rb = smem + b * C::RAW_BYTES;
    if (lane == 0) {
      const uint32_t bytes =
          n * (2 * DK * (int)sizeof(Tin) + CCOLS * (int)sizeof(Tin) + (C::KDA ? DK * 4 : 0));
      mbar_arrive_expect_tx(&bar[b], bytes);
    }
    __syncwarp();
    if (lane < n) {
      const long long row = (t0 + tile * TT + lane) * p.H + h;
      const long long row_qk = (t0 + tile * TT + lane) * p.Hqk + hq;
      bulk_g2s(rb + lane * DK * sizeof(Tin), q + row_qk * DK, DK * sizeof(Tin), &bar[b]);
      bulk_g2s(rb + C::RAW_QK + lane * DK * sizeof(Tin), k + row_qk * DK,
               DK * sizeof(Tin), &bar[b]);
      bulk_g2s(rb + 2 * C::RAW_QK + lane * CCOLS * sizeof(Tin),
               v + row * DV + col_base, CCOLS * sizeof(Tin), &bar[b]);
      if constexpr (C::KDA)
        bulk_g2s(rb + 2 * C::RAW_QK + C::RAW_V + lane * DK * 4, p.g + row * DK,
                 DK * 4, &bar[b]);
    }
  };
  // HOSTIO: the same raw layout, filled by 16-byte loads spread over the
  // CTA (piece e: token e / P_TOK, then q, k, v and the KDA gates in turn).
  // A tile's loads are issued into registers early (before the state loads
  // for the first tile, before the previous tile's tokens otherwise) and
  // stored to shared memory later, so that the latency of the host link
  // overlaps other work.
  uint4 hreg[HOSTIO ? C::P_THREAD : 1];
  auto piece_dst = [&](int e) -> uint32_t {
    const int r = e / C::P_TOK, c = e - r * C::P_TOK;
    if (c < C::P_QK) return r * DK * (int)sizeof(Tin) + c * 16;
    if (c < 2 * C::P_QK) return C::RAW_QK + r * DK * (int)sizeof(Tin) + (c - C::P_QK) * 16;
    if (c < 2 * C::P_QK + C::P_V)
      return 2 * C::RAW_QK + r * CCOLS * (int)sizeof(Tin) + (c - 2 * C::P_QK) * 16;
    return 2 * C::RAW_QK + C::RAW_V + r * DK * 4 + (c - 2 * C::P_QK - C::P_V) * 16;
  };
  auto piece_src = [&](int tile, int e) -> const void * {
    const int r = e / C::P_TOK, c = e - r * C::P_TOK;
    const long long tok = t0 + tile * TT + r;
    const long long row = tok * p.H + h, row_qk = tok * p.Hqk + hq;
    if (c < C::P_QK) return reinterpret_cast<const uint4 *>(q + row_qk * DK) + c;
    if (c < 2 * C::P_QK) return reinterpret_cast<const uint4 *>(k + row_qk * DK) + (c - C::P_QK);
    if (c < 2 * C::P_QK + C::P_V)
      return reinterpret_cast<const uint4 *>(v + row * DV + col_base) + (c - 2 * C::P_QK);
    return reinterpret_cast<const uint4 *>(p.g + row * DK) + (c - 2 * C::P_QK - C::P_V);
  };
  auto host_load = [&](int tile) {
    const int np = min(TT, T_s - tile * TT) * C::P_TOK;
#pragma unroll
    for (int j = 0; j < C::P_THREAD; ++j) {
      const int e = tid + j * C::NT;
      if (e < np) hreg[j] = ld_u4(piece_src(tile, e));
    }
  };
  auto host_store = [&](int tile, int b) {
    const int np = min(TT, T_s - tile * TT) * C::P_TOK;
    unsigned char *rb = smem + b * C::RAW_BYTES;
#pragma unroll
    for (int j = 0; j < C::P_THREAD; ++j) {
      const int e = tid + j * C::NT;
      if (e < np) *reinterpret_cast<uint4 *>(rb + piece_dst(e)) = hreg[j];
    }
  };
  // gate and beta scalars of a tile (the GDA gate is one value per token),
  // loaded into registers ahead of the tile's wait
  auto gate_scalars = [&](int tile, float &gv, float &bv) {
    const int n = min(TT, T_s - tile * TT);
    gv = 0.f;
    bv = 0.f;
    if (tid < n) {
      const long long row = (t0 + tile * TT + tid) * p.H + h;
      if constexpr (!C::KDA) gv = p.g[row];
      bv = p.beta[row];
    }
  };

  // Launched programmatically (gdn_forward), this grid may have been scheduled
  // while the previous kernel of the stream runs: nothing in global memory
  // has been read or written up to here (T and the token offsets are launch
  // parameters then), and nothing is before that kernel completes, not even
  // an address to prefetch from (that kernel may be writing the state_in
  // pointer array). Without a programmatic launch the wait returns at once.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // token copies and gate scalars first, then the state pointer
  if constexpr (HOSTIO) host_load(0);
  else if (warp == 0) issue(0, 0);
  float g_cur, b_cur;
  gate_scalars(0, g_cur, b_cur);

  const float *Sin = p.state_in[s];
  if (Sin) {
    const float *lo = p.slots, *hi = p.slots + p.slots_elems;
    const float *a = Sin, *b = Sin + (long long)p.H * DK * DV;
    if (a < hi && b > lo) {  // overlaps the slot buffer: refuse this sequence
      if (tid == 0) {
        set_error(p.err, kDevOverlap);
        if (!HOSTIO) mbar_wait(&bar[0], 0, nullptr);  // the first tile's copies land before exit
      }
      return;
    }
    Sin += (long long)h * DK * DV;
  }

  // State slice into registers: st[m] = S[rg + ROWG*m][wcol .. wcol+3].
  float4 st[RPT];
  if (Sin) {
#pragma unroll
    for (int m = 0; m < RPT; ++m)
      st[m] = ld_stream_f4(Sin + (rg + ROWG * m) * DV + wcol);
  } else {
#pragma unroll
    for (int m = 0; m < RPT; ++m) st[m] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if constexpr (HOSTIO) host_store(0, 0);

  const int first_snap = T_s - p.n_slots;  // tokens t >= first_snap are stored
  int pos0 = 0;
  if constexpr (CKPT) pos0 = p.pos0 ? p.pos0[s] : 0;
  float *slot_base = p.slots + ((long long)s * p.n_slots * p.H + h) * DK * DV;
  const long long slot_stride = (long long)p.H * DK * DV;

  for (int tile = 0; tile < ntiles; ++tile) {
    const int b = tile & 1;
    const uint32_t parity = (tile >> 1) & 1;
    const int n = min(TT, T_s - tile * TT);
    if constexpr (HOSTIO) {
      if (tile + 1 < ntiles) host_load(tile + 1);
    } else if (warp == 0 && tile + 1 < ntiles) {
      issue(tile + 1, b ^ 1);
    }
    float g_nxt = 0.f, b_nxt = 0.f;
    if (tile + 1 < ntiles) gate_scalars(tile + 1, g_nxt, b_nxt);
    if (!HOSTIO && tid == 0 && !mbar_wait(&bar[b], parity, p.err, kSiteRecTile)) abort_flag = 1;
    if (tid < n) {
      if constexpr (!C::KDA) fa[tid] = expf(g_cur);
      fb[tid] = b_cur;
    }
    g_cur = g_nxt;
    b_cur = b_nxt;
    __syncthreads();
    if (abort_flag) {
      // Let a copy still in flight for the next tile land before exiting.
      if (!HOSTIO && tid == 0 && tile + 1 < ntiles)
        mbar_wait(&bar[b ^ 1], ((tile + 1) >> 1) & 1, nullptr);
      return;
    }
    {  // convert the raw tile to fp32
      const unsigned char *rb = smem + b * C::RAW_BYTES;
      const Tin *rq = reinterpret_cast<const Tin *>(rb);
      const Tin *rk = reinterpret_cast<const Tin *>(rb + C::RAW_QK);
      const Tin *rv = reinterpret_cast<const Tin *>(rb + 2 * C::RAW_QK);
      for (int e = tid; e < n * DK; e += C::NT) {
        fq[e] = to_f32(rq[e]);
        fk[e] = to_f32(rk[e]);
      }
      for (int e = tid; e < n * CCOLS; e += C::NT) fv[e] = to_f32(rv[e]);
      if constexpr (C::KDA) {
        const float *rg_ = reinterpret_cast<const float *>(rb + 2 * C::RAW_QK + C::RAW_V);
        for (int e = tid; e < n * DK; e += C::NT) fa[e] = expf(rg_[e]);
      }
    }
    __syncthreads();

    for (int r = 0; r < n; ++r) {
      const int t = tile * TT + r;  // token index within the sequence
      const float *kr = fk + r * DK;
      const float *qr = fq + r * DK;
      const float beta = fb[r];
      float a_h = 1.f;
      if constexpr (!C::KDA) a_h = fa[r];

      const float4 vv =
          *reinterpret_cast<const float4 *>(fv + r * CCOLS + (wcol - col_base));
      const float4 o = token_update<C>(st, kr, qr, C::KDA ? fa + r * DK : nullptr, a_h, beta,
                                       vv, rg);
      const float o0 = o.x, o1 = o.y, o2 = o.z, o3 = o.w;
      if (rg == 0) {
        float *orow = p.out + ((t0 + t) * p.H + h) * DV + wcol;
        st_f4(orow, make_float4(p.scale * o0, p.scale * o1, p.scale * o2, p.scale * o3));
      }
      // snapshot
      if (t >= first_snap) {
        float *dst = slot_base + (long long)(t - first_snap) * slot_stride;
#pragma unroll
        for (int m = 0; m < RPT; ++m) st_f4(dst + (rg + ROWG * m) * DV + wcol, st[m]);
      }
      // checkpoint at a multiple of ckpt_every tokens of the sequence
      if constexpr (CKPT) {
        const int pos = pos0 + t + 1;
        const int c = pos / p.ckpt_every - 1;
        if (pos % p.ckpt_every == 0 && c < p.max_ckpts) {
          float *dst = p.ckpt + (((long long)s * p.max_ckpts + c) * p.H + h) * DK * DV;
#pragma unroll
          for (int m = 0; m < RPT; ++m) st_f4(dst + (rg + ROWG * m) * DV + wcol, st[m]);
        }
      }
    }
    if constexpr (HOSTIO) {
      if (tile + 1 < ntiles) host_store(tile + 1, b ^ 1);
    }
    __syncthreads();  // fp32 tile buffers are rewritten by the next tile
  }
}

// Kernel configuration per head size. Fixed per (D_k, D_v) and input type so
// that the arithmetic order never depends on T, K or the batch (the chunked
// call's fp32 token loop, 128 x 128 heads, takes its own fixed configuration:
// see launch_d).
template <int DK, int DV, bool KDA, typename Tin>
struct RecPick;
template <bool KDA, typename Tin>
struct RecPick<128, 128, KDA, Tin> { using C = RecCfg<128, 128, 8, 4, KDA, Tin>; };
template <bool KDA, typename Tin>
struct RecPick<128, 64, KDA, Tin> { using C = RecCfg<128, 64, 8, 4, KDA, Tin>; };
template <bool KDA, typename Tin>
struct RecPick<64, 128, KDA, Tin> { using C = RecCfg<64, 128, 4, 2, KDA, Tin>; };
template <bool KDA, typename Tin>
struct RecPick<64, 64, KDA, Tin> { using C = RecCfg<64, 64, 4, 2, KDA, Tin>; };

template <typename C>
cudaError_t launch_c(const RecParams &p, cudaStream_t stream) {
  const long long n_items = (long long)p.n_seqs * p.H * C::CTAS_PER_HEAD;
  if (n_items == 0) return cudaSuccess;
  if (n_items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  static_assert(C::SMEM <= 48 * 1024, "fits the default shared-memory window");
  if (p.pdl)  // gdn_forward: overlaps the previous kernel's tail with this prologue
    return launch_pdl(recurrent_kernel<C, false>, dim3((unsigned)n_items), dim3(C::NT), C::SMEM,
                      stream, p);
  if (p.ckpt)
    recurrent_kernel<C, true><<<(unsigned)n_items, C::NT, C::SMEM, stream>>>(p);
  else
    recurrent_kernel<C, false><<<(unsigned)n_items, C::NT, C::SMEM, stream>>>(p);
  return cudaGetLastError();
}

template <int DK, int DV, bool KDA, typename Tin>
cudaError_t launch_t(const RecParams &p, cudaStream_t stream) {
  return launch_c<typename RecPick<DK, DV, KDA, Tin>::C>(p, stream);
}

// gdn_forward_host: the configuration of gdn_forward (same arithmetic), with
// the token tiles read by ordinary loads; a programmatic launch like it.
template <int DK, int DV, bool KDA, typename Tin>
cudaError_t launch_host_io(const RecParams &p, cudaStream_t stream) {
  using C = typename RecPick<DK, DV, KDA, Tin>::C;
  const long long n_items = (long long)p.n_seqs * p.H * C::CTAS_PER_HEAD;
  if (n_items == 0) return cudaSuccess;
  if (n_items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(recurrent_kernel<C, false, true>, dim3((unsigned)n_items), dim3(C::NT),
                    C::SMEM, stream, p);
}

template <int DK, int DV>
cudaError_t launch_d(const RecParams &p, bool kda, bool bf16, cudaStream_t s) {
  if (p.host_io) {
    if (kda)
      return bf16 ? launch_host_io<DK, DV, true, __nv_bfloat16>(p, s)
                  : launch_host_io<DK, DV, true, float>(p, s);
    return bf16 ? launch_host_io<DK, DV, false, __nv_bfloat16>(p, s)
                : launch_host_io<DK, DV, false, float>(p, s);
  }
  if constexpr (DK == 128 && DV == 128) {
    // long fp32 chains: a token's step is latency-bound, and a narrower slice
    // per CTA shortens it (about 10% on the varlen fp32 prefill)
    if (p.long_chains && !bf16)
      return kda ? launch_c<RecCfg<128, 128, 16, 4, true, float>>(p, s)
                 : launch_c<RecCfg<128, 128, 16, 4, false, float>>(p, s);
  }
  if (kda)
    return bf16 ? launch_t<DK, DV, true, __nv_bfloat16>(p, s)
                : launch_t<DK, DV, true, float>(p, s);
  return bf16 ? launch_t<DK, DV, false, __nv_bfloat16>(p, s)
              : launch_t<DK, DV, false, float>(p, s);
}

}  // namespace

cudaError_t launch_recurrent(const RecurrentArgs &a, cudaStream_t stream) {
  RecParams p;
  p.q = a.q; p.k = a.k; p.v = a.v; p.g = a.g; p.beta = a.beta;
  p.state_in = a.state_in; p.slots = a.slots; p.out = a.out;
  p.tok_start = a.tok_start; p.seq_len = a.seq_len;
  p.slots_elems = (long long)a.n_seqs * a.n_slots * a.H * a.Dk * a.Dv;
  p.n_seqs = a.n_seqs; p.T = a.T; p.H = a.H; p.n_slots = a.n_slots;
  p.Hqk = a.Hqk > 0 ? a.Hqk : a.H;
  p.qk_grouped = a.qk_grouped ? 1 : 0;
  p.ckpt = a.ckpt; p.pos0 = a.pos0;
  p.pdl = a.pdl && !a.tok_start && !a.seq_len && !a.ckpt ? 1 : 0;
  p.long_chains = a.long_chains ? 1 : 0;
  p.host_io = a.host_io && p.pdl ? 1 : 0;
  p.ckpt_every = a.ckpt_every > 0 ? a.ckpt_every : 1; p.max_ckpts = a.max_ckpts;
  p.scale = a.scale; p.err = a.err;
  if (a.Dk == 128 && a.Dv == 128) return launch_d<128, 128>(p, a.kda, a.bf16, stream);
  if (a.Dk == 128 && a.Dv == 64) return launch_d<128, 64>(p, a.kda, a.bf16, stream);
  if (a.Dk == 64 && a.Dv == 128) return launch_d<64, 128>(p, a.kda, a.bf16, stream);
  if (a.Dk == 64 && a.Dv == 64) return launch_d<64, 64>(p, a.kda, a.bf16, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
