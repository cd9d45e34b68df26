// api.cu -- the C ABI of libgdn (declared in include/gdn.h): argument
// validation, dispatch to the kernels, error reporting, the per-device error
// word and the host-side rollback table.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "gdn.h"
#include "kernels.h"

namespace {

thread_local std::string g_msg;

__attribute__((format(printf, 2, 3))) gdn_status fail(gdn_status st, const char *fmt, ...);
gdn_status fail(gdn_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_msg = buf;
  return st;
}

gdn_status ok() { return GDN_OK; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool head_size_ok(int d) { return d == 64 || d == 128; }

}  // namespace

// One error word per device; kernels receive its device address.
__device__ int g_gdn_err_word;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_err_mu;
int *g_err_ptr[kMaxDevices] = {};

// Device address of the current device's error word, looked up once per
// device with that device current.
gdn_status device_err_ptr(int **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return fail(GDN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(GDN_ERR_UNSUPPORTED, "device ordinal %d above %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_err_mu);
  if (!g_err_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_gdn_err_word);
    if (e != cudaSuccess)
      return fail(GDN_ERR_CUDA, "cudaGetSymbolAddress(error word): %s",
                  cudaGetErrorString(e));
    g_err_ptr[dev] = static_cast<int *>(p);
  }
  *out = g_err_ptr[dev];
  return GDN_OK;
}

gdn_status check_launch(cudaError_t e, const char *what) {
  if (e != cudaSuccess)
    return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return GDN_OK;
}

}  // namespace

extern "C" {

const char *gdn_last_error(void) { return g_msg.c_str(); }

const char *gdn_version(void) { return "libgdn 0.2.0 (sm_103a)"; }

// Resolves the grouped-query fields: H_qk = 0 means H; H_qk must divide H.
static gdn_status qk_heads(const char *fn, int H, int H_qk, int qk_map, int *hq) {
  *hq = H_qk == 0 ? H : H_qk;
  if (*hq <= 0 || *hq > H || H % *hq != 0)
    return fail(GDN_ERR_INVALID_ARG, "%s: H_qk=%d must divide H=%d", fn, H_qk, H);
  if (qk_map != GDN_QK_TILED && qk_map != GDN_QK_GROUPED)
    return fail(GDN_ERR_INVALID_ARG, "%s: qk_map %d", fn, qk_map);
  return GDN_OK;
}

// True when the device can dereference p: device or managed memory, or
// page-locked host memory mapped into the device's address space at the same
// address (unified addressing). Pageable host memory is refused.
static bool device_reachable(const void *p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // clear the (non-sticky) error the query reported
    return false;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return true;
  return at.type == cudaMemoryTypeHost && at.devicePointer == p;
}

// gdn_forward and gdn_forward_host: the same checks and kernel arithmetic;
// host_io reads the token rows with ordinary loads (host memory allowed).
static gdn_status forward_impl(const char *fn, const gdn_shape *shape, const void *q,
                               const void *k, const void *v, const float *g,
                               const float *beta, const float *const *state_in,
                               float *state_slots, float *out, int n_slots, gdn_mode mode,
                               gdn_stream_t stream, bool host_io) {
  if (!shape) return fail(GDN_ERR_INVALID_ARG, "%s: shape is NULL", fn);
  const gdn_shape &s = *shape;
  if (s.n_seqs < 0 || s.T < 0 || s.H <= 0)
    return fail(GDN_ERR_INVALID_ARG, "%s: n_seqs=%d T=%d H=%d", fn, s.n_seqs, s.T, s.H);
  if (mode != GDN_MODE_GDA && mode != GDN_MODE_KDA)
    return fail(GDN_ERR_INVALID_ARG, "%s: mode %d", fn, (int)mode);
  if (s.in_dtype != GDN_F32 && s.in_dtype != GDN_BF16)
    return fail(GDN_ERR_INVALID_ARG, "%s: in_dtype %d", fn, (int)s.in_dtype);
  if (n_slots < 1)
    return fail(GDN_ERR_INVALID_ARG, "%s: n_slots=%d (need >= 1)", fn, n_slots);
  if (s.D_k <= 0 || s.D_v <= 0)
    return fail(GDN_ERR_INVALID_ARG, "%s: D_k=%d D_v=%d", fn, s.D_k, s.D_v);
  if (!head_size_ok(s.D_k) || !head_size_ok(s.D_v))
    return fail(GDN_ERR_UNSUPPORTED, "%s: head sizes D_k=%d D_v=%d (supported: 64, 128)", fn,
                s.D_k, s.D_v);
  if (!std::isfinite(s.scale))
    return fail(GDN_ERR_INVALID_ARG, "%s: scale is not finite", fn);
  int hq = 0;
  if (qk_heads(fn, s.H, s.H_qk, (int)s.qk_map, &hq) != GDN_OK) return GDN_ERR_INVALID_ARG;
  const long long ntok = (long long)s.n_seqs * s.T;
  if (ntok > (1LL << 31) / s.H)
    return fail(GDN_ERR_UNSUPPORTED, "%s: %lld tokens x %d heads too large", fn, ntok, s.H);
  if (s.n_seqs == 0) return ok();
  if (!state_in || !state_slots)
    return fail(GDN_ERR_INVALID_ARG, "%s: state_in/state_slots is NULL", fn);
  if (!aligned16(state_in) || !aligned16(state_slots))
    return fail(GDN_ERR_INVALID_ARG, "%s: state buffers must be 16-byte aligned", fn);
  if (ntok == 0) return ok();
  const void *ptrs[] = {q, k, v, g, beta, out};
  const char *names[] = {"q", "k", "v", "g", "beta", "out"};
  for (int i = 0; i < 6; ++i) {
    if (!ptrs[i]) return fail(GDN_ERR_INVALID_ARG, "%s: %s is NULL", fn, names[i]);
    if (!aligned16(ptrs[i]))
      return fail(GDN_ERR_INVALID_ARG, "%s: %s is not 16-byte aligned", fn, names[i]);
  }
  if (host_io)
    for (int i = 0; i < 6; ++i)
      if (!device_reachable(ptrs[i]))
        return fail(GDN_ERR_INVALID_ARG,
                    "%s: %s is neither device memory nor page-locked host memory mapped at "
                    "the same address", fn, names[i]);
  int *err = nullptr;
  gdn_status st = device_err_ptr(&err);
  if (st != GDN_OK) return st;

  gdn::RecurrentArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.state_in = state_in; a.slots = state_slots; a.out = out;
  a.tok_start = nullptr; a.seq_len = nullptr;
  a.n_seqs = s.n_seqs; a.T = s.T; a.H = s.H; a.Dk = s.D_k; a.Dv = s.D_v;
  a.Hqk = hq; a.qk_grouped = s.qk_map == GDN_QK_GROUPED;
  a.n_slots = n_slots;
  a.kda = mode == GDN_MODE_KDA;
  a.bf16 = s.in_dtype == GDN_BF16;
  a.scale = s.scale != 0.f ? s.scale : 1.0f / std::sqrt((float)s.D_k);
  a.err = err;
  a.pdl = true;  // prologue overlaps the previous kernel of the stream
  a.host_io = host_io;
  return check_launch(gdn::launch_recurrent(a, reinterpret_cast<cudaStream_t>(stream)),
                      host_io ? "gdn_forward_host launch" : "gdn_forward launch");
}

gdn_status gdn_forward(const gdn_shape *shape, const void *q, const void *k,
                       const void *v, const float *g, const float *beta,
                       const float *const *state_in, float *state_slots,
                       float *out, int n_slots, gdn_mode mode,
                       gdn_stream_t stream) {
  return forward_impl("gdn_forward", shape, q, k, v, g, beta, state_in, state_slots, out,
                      n_slots, mode, stream, false);
}

gdn_status gdn_forward_host(const gdn_shape *shape, const void *q, const void *k,
                            const void *v, const float *g, const float *beta,
                            const float *const *state_in, float *state_slots,
                            float *out, int n_slots, gdn_mode mode,
                            gdn_stream_t stream) {
  return forward_impl("gdn_forward_host", shape, q, k, v, g, beta, state_in, state_slots,
                      out, n_slots, mode, stream, true);
}

size_t gdn_chunked_workspace_size(const gdn_varlen_shape *shape, int n_slots) {
  if (!shape || shape->n_seqs <= 0 || shape->total_tokens < 0 || shape->H <= 0 ||
      n_slots < 1)
    return 0;
  return gdn::chunked_workspace_size(shape->n_seqs, shape->total_tokens, shape->H,
                                     shape->D_k, shape->D_v, shape->in_dtype == GDN_BF16);
}

// Argument checks shared by every chunked entry point, and the launch
// arguments they imply (all but the workspace and the checkpoints).
static gdn_status chunked_args(const char *fn, const gdn_varlen_shape *shape,
                               const int32_t *cu_seqlens, const void *q, const void *k,
                               const void *v, const float *g, const float *beta,
                               const float *const *state_in, float *state_slots, float *out,
                               int n_slots, gdn_mode mode, gdn::ChunkedArgs *a) {
  if (!shape) return fail(GDN_ERR_INVALID_ARG, "%s: shape is NULL", fn);
  const gdn_varlen_shape &s = *shape;
  if (s.n_seqs <= 0 || s.total_tokens < 0 || s.H <= 0)
    return fail(GDN_ERR_INVALID_ARG, "%s: n_seqs=%d total_tokens=%d H=%d", fn,
                s.n_seqs, s.total_tokens, s.H);
  if (mode != GDN_MODE_GDA && mode != GDN_MODE_KDA)
    return fail(GDN_ERR_INVALID_ARG, "%s: mode %d", fn, (int)mode);
  if (s.in_dtype != GDN_F32 && s.in_dtype != GDN_BF16)
    return fail(GDN_ERR_INVALID_ARG, "%s: in_dtype %d", fn, (int)s.in_dtype);
  if (n_slots < 1)
    return fail(GDN_ERR_INVALID_ARG, "%s: n_slots=%d (need >= 1)", fn, n_slots);
  if (!head_size_ok(s.D_k) || !head_size_ok(s.D_v))
    return fail(GDN_ERR_UNSUPPORTED,
                "%s: head sizes D_k=%d D_v=%d (supported: 64, 128)", fn, s.D_k,
                s.D_v);
  if (!std::isfinite(s.scale))
    return fail(GDN_ERR_INVALID_ARG, "%s: scale is not finite", fn);
  int hq = 0;
  if (qk_heads(fn, s.H, s.H_qk, (int)s.qk_map, &hq) != GDN_OK)
    return GDN_ERR_INVALID_ARG;
  if ((long long)s.total_tokens * s.H > (1LL << 31))
    return fail(GDN_ERR_UNSUPPORTED, "%s: too many token-heads", fn);
  const void *ptrs[] = {cu_seqlens, state_in, state_slots};
  const char *names[] = {"cu_seqlens", "state_in", "state_slots"};
  for (int i = 0; i < 3; ++i)
    if (!ptrs[i]) return fail(GDN_ERR_INVALID_ARG, "%s: %s is NULL", fn, names[i]);
  if (s.total_tokens > 0) {
    const void *tp[] = {q, k, v, g, beta, out};
    const char *tn[] = {"q", "k", "v", "g", "beta", "out"};
    for (int i = 0; i < 6; ++i) {
      if (!tp[i]) return fail(GDN_ERR_INVALID_ARG, "%s: %s is NULL", fn, tn[i]);
      if (!aligned16(tp[i]))
        return fail(GDN_ERR_INVALID_ARG, "%s: %s is not 16-byte aligned", fn, tn[i]);
    }
  }
  if (!aligned16(state_in) || !aligned16(state_slots) || !aligned16(cu_seqlens))
    return fail(GDN_ERR_INVALID_ARG, "%s: buffers must be 16-byte aligned", fn);

  *a = gdn::ChunkedArgs{};
  a->cu_seqlens = cu_seqlens;
  a->q = q; a->k = k; a->v = v; a->g = g; a->beta = beta;
  a->state_in = state_in; a->slots = state_slots; a->out = out;
  a->n_seqs = s.n_seqs; a->total_tokens = s.total_tokens; a->H = s.H;
  a->Hqk = hq; a->qk_grouped = s.qk_map == GDN_QK_GROUPED;
  a->bf16 = s.in_dtype == GDN_BF16;
  a->Dk = s.D_k; a->Dv = s.D_v; a->n_slots = n_slots;
  a->kda = mode == GDN_MODE_KDA;
  a->scale = s.scale != 0.f ? s.scale : 1.0f / std::sqrt((float)s.D_k);
  return GDN_OK;
}

// Validation and launch shared by gdn_forward_chunked (ckpt = NULL) and
// gdn_forward_chunked_checkpointed.
static gdn_status chunked_call(const char *fn, const gdn_varlen_shape *shape,
                               const int32_t *cu_seqlens, const void *q, const void *k,
                               const void *v, const float *g, const float *beta,
                               const float *const *state_in, float *state_slots, float *out,
                               int n_slots, gdn_mode mode, float *ckpt, int ckpt_every,
                               int max_ckpts, void *workspace, size_t workspace_bytes,
                               gdn_stream_t stream) {
  gdn::ChunkedArgs a;
  gdn_status st = chunked_args(fn, shape, cu_seqlens, q, k, v, g, beta, state_in, state_slots,
                               out, n_slots, mode, &a);
  if (st != GDN_OK) return st;
  if (!workspace) return fail(GDN_ERR_INVALID_ARG, "%s: workspace is NULL", fn);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(GDN_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", fn);
  const size_t need = gdn_chunked_workspace_size(shape, n_slots);
  if (workspace_bytes < need)
    return fail(GDN_ERR_INVALID_ARG, "%s: workspace %zu bytes < %zu needed", fn,
                workspace_bytes, need);
  if ((st = device_err_ptr(&a.err)) != GDN_OK) return st;
  a.workspace = workspace; a.workspace_bytes = workspace_bytes;
  a.ckpt = ckpt; a.ckpt_every = ckpt_every; a.max_ckpts = max_ckpts;
  return check_launch(gdn::launch_chunked(a, reinterpret_cast<cudaStream_t>(stream)),
                      fn);
}

gdn_status gdn_forward_chunked(const gdn_varlen_shape *shape,
                               const int32_t *cu_seqlens, const void *q,
                               const void *k, const void *v, const float *g,
                               const float *beta, const float *const *state_in,
                               float *state_slots, float *out, int n_slots,
                               gdn_mode mode, void *workspace,
                               size_t workspace_bytes, gdn_stream_t stream) {
  return chunked_call("gdn_forward_chunked", shape, cu_seqlens, q, k, v, g, beta, state_in,
                      state_slots, out, n_slots, mode, nullptr, 0, 0, workspace,
                      workspace_bytes, stream);
}

static bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

gdn_status gdn_forward_chunked_checkpointed(
    const gdn_varlen_shape *shape, const int32_t *cu_seqlens, const void *q, const void *k,
    const void *v, const float *g, const float *beta, const float *const *state_in,
    float *state_slots, float *out, int n_slots, gdn_mode mode, float *checkpoints,
    int ckpt_every, int max_ckpts, void *workspace, size_t workspace_bytes,
    gdn_stream_t stream) {
  const char *fn = "gdn_forward_chunked_checkpointed";
  if (!checkpoints) return fail(GDN_ERR_INVALID_ARG, "%s: checkpoints is NULL", fn);
  if (!aligned16(checkpoints))
    return fail(GDN_ERR_INVALID_ARG, "%s: checkpoints is not 16-byte aligned", fn);
  if (ckpt_every <= 0 || ckpt_every % 64 != 0)
    return fail(GDN_ERR_INVALID_ARG, "%s: ckpt_every=%d (need a positive multiple of 64)", fn,
                ckpt_every);
  if (max_ckpts < 1) return fail(GDN_ERR_INVALID_ARG, "%s: max_ckpts=%d (need >= 1)", fn,
                                 max_ckpts);
  if (shape && shape->n_seqs > 0 && shape->H > 0 && shape->D_k > 0 && shape->D_v > 0 &&
      shape->total_tokens >= 0 && n_slots >= 1) {
    const size_t st = sizeof(float) * (size_t)shape->H * shape->D_k * shape->D_v;
    const size_t nck = st * (size_t)shape->n_seqs * (size_t)max_ckpts;
    if (state_slots &&
        ranges_overlap(checkpoints, nck, state_slots, st * (size_t)shape->n_seqs * n_slots))
      return fail(GDN_ERR_INVALID_ARG, "%s: checkpoints overlap state_slots", fn);
    if (out && ranges_overlap(checkpoints, nck, out,
                              sizeof(float) * (size_t)shape->total_tokens * shape->H *
                                  shape->D_v))
      return fail(GDN_ERR_INVALID_ARG, "%s: checkpoints overlap out", fn);
  }
  return chunked_call(fn, shape, cu_seqlens, q, k, v, g, beta, state_in, state_slots, out,
                      n_slots, mode, checkpoints, ckpt_every, max_ckpts, workspace,
                      workspace_bytes, stream);
}

gdn_status gdn_checkpoint_select(int n_keep, int L, int n_slots, int ckpt_every,
                                 int max_ckpts, int *source, int *index, int *replay_from) {
  const char *fn = "gdn_checkpoint_select";
  if (!source || !index || !replay_from)
    return fail(GDN_ERR_INVALID_ARG, "%s: NULL output pointer", fn);
  if (L < 0 || n_keep < 0 || n_keep > L)
    return fail(GDN_ERR_INVALID_ARG, "%s: n_keep=%d L=%d (need 0 <= n_keep <= L)", fn, n_keep,
                L);
  if (n_slots < 1 || max_ckpts < 1 || ckpt_every <= 0 || ckpt_every % 64 != 0)
    return fail(GDN_ERR_INVALID_ARG, "%s: n_slots=%d ckpt_every=%d max_ckpts=%d", fn, n_slots,
                ckpt_every, max_ckpts);
  // slot j holds the state after token L - n_slots + j (slots before the
  // sequence's first token are not written)
  const int slot = n_keep - 1 - (L - n_slots);
  if (n_keep >= 1 && slot >= 0) {
    *source = 2; *index = slot; *replay_from = n_keep;
    return GDN_OK;
  }
  const int m = (n_keep / ckpt_every < max_ckpts ? n_keep / ckpt_every : max_ckpts) - 1;
  if (m >= 0) {
    *source = 1; *index = m; *replay_from = (m + 1) * ckpt_every;
    return GDN_OK;
  }
  *source = 0; *index = -1; *replay_from = 0;
  return GDN_OK;
}

// Same computation as gdn_forward_chunked, but the scratch it needs lives in
// a fixed device array inside the library instead of a caller workspace, so
// the call allocates nothing. For callers that cannot allocate device memory
// themselves (hosts that own every byte through their own pool, loops that
// must not pay for a device allocation).
gdn_status gdn_forward_chunked_noalloc(const gdn_varlen_shape *shape,
                                       const int32_t *cu_seqlens, const void *q,
                                       const void *k, const void *v, const float *g,
                                       const float *beta, const float *const *state_in,
                                       float *state_slots, float *out, int n_slots,
                                       gdn_mode mode, gdn_stream_t stream) {
  const char *fn = "gdn_forward_chunked_noalloc";
  gdn::ChunkedArgs a;
  gdn_status st = chunked_args(fn, shape, cu_seqlens, q, k, v, g, beta, state_in, state_slots,
                               out, n_slots, mode, &a);
  if (st != GDN_OK) return st;
  const size_t need = gdn::chunked_workspace_need(a.n_seqs, a.total_tokens, a.H, a.Dk, a.Dv,
                                                  a.kda, a.bf16);
  if (need > gdn::static_scratch_bytes())
    return fail(GDN_ERR_UNSUPPORTED,
                "%s: this shape needs %zu bytes of scratch; the built-in area holds %zu "
                "(use gdn_forward_chunked with a workspace)",
                fn, need, gdn::static_scratch_bytes());
  if ((st = device_err_ptr(&a.err)) != GDN_OK) return st;
  size_t need2 = 0;
  return check_launch(
      gdn::launch_chunked_static(a, reinterpret_cast<cudaStream_t>(stream), &need2), fn);
}

size_t gdn_noalloc_scratch_bytes(void) { return gdn::static_scratch_bytes(); }

// ---- rollback table --------------------------------------------------------

struct gdn_seq_table {
  int n_seqs;
  int n_slots;
  std::vector<int> T_last;  // tokens of each sequence's last forward
};

gdn_status gdn_seq_table_create(int n_seqs, int n_slots, gdn_seq_table **out) {
  if (!out) return fail(GDN_ERR_INVALID_ARG, "gdn_seq_table_create: out is NULL");
  *out = nullptr;
  if (n_seqs < 0 || n_slots < 1)
    return fail(GDN_ERR_INVALID_ARG, "gdn_seq_table_create: n_seqs=%d n_slots=%d", n_seqs, n_slots);
  gdn_seq_table *t = new (std::nothrow) gdn_seq_table;
  if (!t) return fail(GDN_ERR_INVALID_ARG, "gdn_seq_table_create: out of host memory");
  t->n_seqs = n_seqs;
  t->n_slots = n_slots;
  t->T_last.assign((size_t)n_seqs, 0);
  *out = t;
  return GDN_OK;
}

void gdn_seq_table_destroy(gdn_seq_table *table) { delete table; }

gdn_status gdn_seq_table_record(gdn_seq_table *t, int seq, int T_last) {
  if (!t) return fail(GDN_ERR_INVALID_ARG, "gdn_seq_table_record: table is NULL");
  if (seq < 0 || seq >= t->n_seqs || T_last < 0)
    return fail(GDN_ERR_INVALID_ARG, "gdn_seq_table_record: seq=%d T_last=%d", seq, T_last);
  t->T_last[(size_t)seq] = T_last;
  return GDN_OK;
}

gdn_status gdn_seq_table_clear(gdn_seq_table *t, int seq) {
  if (!t) return fail(GDN_ERR_INVALID_ARG, "gdn_seq_table_clear: table is NULL");
  if (seq < 0 || seq >= t->n_seqs)
    return fail(GDN_ERR_INVALID_ARG, "gdn_seq_table_clear: seq=%d", seq);
  t->T_last[(size_t)seq] = 0;
  return GDN_OK;
}

gdn_status gdn_rollback(const gdn_seq_table *t, int seq, int n_accepted, int *slot) {
  if (!t || !slot) return fail(GDN_ERR_INVALID_ARG, "gdn_rollback: NULL argument");
  if (seq < 0 || seq >= t->n_seqs)
    return fail(GDN_ERR_INVALID_ARG, "gdn_rollback: seq=%d of %d", seq, t->n_seqs);
  const int T = t->T_last[(size_t)seq];
  const int K = t->n_slots;
  if (n_accepted < 0 || n_accepted > T)
    return fail(GDN_ERR_ROLLBACK_RANGE, "gdn_rollback: n_accepted=%d outside [0, %d]",
                n_accepted, T);
  if (n_accepted == 0) {
    *slot = -1;
    return GDN_OK;
  }
  // The state after token n_accepted-1 was stored iff that token is one of
  // the last K tokens of the forward.
  const int j = (n_accepted - 1) - (T - K);
  if (j < 0)
    return fail(GDN_ERR_ROLLBACK_RANGE,
                "gdn_rollback: state after %d of %d tokens was not stored (K=%d)",
                n_accepted, T, K);
  *slot = j;
  return GDN_OK;
}

gdn_status gdn_slot_state_ptr(const float *state_slots, int seq, int slot,
                              int n_slots, int H, int D_k, int D_v,
                              const float **out) {
  if (!out) return fail(GDN_ERR_INVALID_ARG, "gdn_slot_state_ptr: out is NULL");
  if (slot == -1) {
    *out = nullptr;
    return GDN_OK;
  }
  if (!state_slots || seq < 0 || slot < 0 || slot >= n_slots || H <= 0 || D_k <= 0 || D_v <= 0)
    return fail(GDN_ERR_INVALID_ARG, "gdn_slot_state_ptr: seq=%d slot=%d n_slots=%d", seq,
                slot, n_slots);
  const long long per = (long long)H * D_k * D_v;
  *out = state_slots + ((long long)seq * n_slots + slot) * per;
  return GDN_OK;
}

static const char *wait_site_name(int site) {
  switch (site) {
    case gdn::kSiteRecTile: return "recurrent kernel, token tile copies";
    case gdn::kSitePrepLoad: return "chunk prep, K/Q tile copies";
    case gdn::kSitePrepG: return "chunk prep, G product";
    case gdn::kSitePrepW: return "chunk prep, W product";
    case gdn::kSiteScanX: return "chunk scan, X product";
    case gdn::kSiteScanS: return "chunk scan, state-update product";
    case gdn::kSiteScanO: return "chunk scan, output product";
    case gdn::kSiteScanEmpty: return "chunk scan, stage release";
    case gdn::kSiteScanPad: return "chunk scan, partial-chunk copies";
    case gdn::kSiteScanReady: return "chunk scan, ready flag of a prepared tile";
    case gdn::kSiteScanStage: return "chunk scan, stage copies";
    case gdn::kSiteScanS0: return "chunk scan, state operand";
    case gdn::kSiteScanD: return "chunk scan, D tile";
    default: return "unnamed wait";
  }
}

gdn_status gdn_decode_device_error(int word) {
  if (word == 0) return GDN_OK;
  switch (word & 0xff) {
    case gdn::kDevTimeout: {
      const int site = (word >> 8) & 0xff;
      return fail(GDN_ERR_TIMEOUT,
                  "a device-side wait ran out (kernel abandoned its work; site %d: %s; "
                  "chunk %d)",
                  site, wait_site_name(site), (word >> 16) & 0x7fff);
    }
    case gdn::kDevBadSeqlens:
      return fail(GDN_ERR_DEVICE_ARG, "cu_seqlens is not a valid offset table");
    case gdn::kDevOverlap:
      return fail(GDN_ERR_DEVICE_ARG, "a state_in pointer points into state_slots");
    case gdn::kDevGateRange:
      return fail(GDN_ERR_DEVICE_ARG,
                  "a gate decays (or grows) by more than e^80 inside one 64-token chunk, or "
                  "is NaN; the chunked path cannot represent that decay, run these "
                  "sequences through gdn_forward");
    default:
      return fail(GDN_ERR_DEVICE_ARG, "device error word %d", word);
  }
}

gdn_status gdn_device_error_word(int **word) {
  if (!word) return fail(GDN_ERR_INVALID_ARG, "gdn_device_error_word: word is NULL");
  return device_err_ptr(word);
}

gdn_status gdn_check_device_error(gdn_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(GDN_ERR_CUDA, "gdn_check_device_error: %s", cudaGetErrorString(e));
  int *dummy = nullptr;
  gdn_status st = device_err_ptr(&dummy);
  if (st != GDN_OK) return st;
  int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_gdn_err_word, sizeof(int));
  if (e != cudaSuccess)
    return fail(GDN_ERR_CUDA, "gdn_check_device_error: %s", cudaGetErrorString(e));
  if (word == 0) return GDN_OK;
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_gdn_err_word, &zero, sizeof(int));
  if (e != cudaSuccess)
    return fail(GDN_ERR_CUDA, "gdn_check_device_error: %s", cudaGetErrorString(e));
  return gdn_decode_device_error(word);
}

}  // extern "C"
