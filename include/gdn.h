/*
 * gdn.h -- C ABI of libgdn, the gated delta-net (GDN) recurrence on NVIDIA
 * GB300 (sm_103a).
 *
 * The op. Per sequence s, head h and token t, the D_k x D_v fp32 state S of
 * that head (row i = key index, column j = value index) is
 *   decayed    S <- exp(g) S               (GDA: one gate per head and token)
 *              S[i,:] <- exp(g_i) S[i,:]   (KDA: one gate per key row)
 *   read       u = S^T k
 *   corrected  d = beta (v - u)
 *   written    S <- S + k d^T
 *   queried    o = scale S^T q             (after the write)
 * This is the gated delta rule of "Gated Delta Networks" (Yang, Kautz,
 * Hatamizadeh, ICLR 2025); the op is GGML_OP_GATED_DELTA_NET with the GDA and
 * KDA modes and head sizes 64/128 of "metal : add GDN kernel (#20361)"
 * (llama.cpp commits, tag b9752, src/models/qwen35.cpp). g is a log-decay used
 * as exp(g) with no clamp; beta is used as given (the caller applies any
 * sigmoid); q and k are used as given (the caller normalises them).
 *
 * Snapshots and rollback ("metal: add GDN partial rollback" and "llama: allow
 * partial seq_rm for GDN models for speculative decoding", koboldcpp commits,
 * tag v1.113.1): a forward keeps K = n_slots states per sequence. After token
 * t of a T-token sequence with t >= T-K the state goes to slot t-(T-K), so
 * slot K-1 is the final state and K = 1 is the plain single-state forward.
 * When T < K, slots j < K-T are not written. The input state is a separate
 * buffer and is never written. Rolling back to n accepted tokens is a slot
 * select (gdn_rollback), not a recompute.
 *
 * Conventions for every call below.
 *  - Ownership: the caller allocates and owns every buffer and the stream.
 *    The library allocates no device memory on these calls and never
 *    synchronises the stream, except gdn_check_device_error.
 *  - Layouts: dense, row-major, innermost index last, exactly as written in
 *    each comment; no strides. Ntok is the number of packed tokens.
 *  - Alignment: every device buffer must be 16-byte aligned.
 *  - Supported shapes: D_k, D_v in {64, 128}. Anything else returns
 *    GDN_ERR_UNSUPPORTED; there is no fallback path of any kind.
 *  - Errors: every call returns a gdn_status; gdn_last_error() gives the
 *    calling thread's last message. Kernel launches are asynchronous: a
 *    condition only the device can see (a bad cu_seqlens entry, a bounded
 *    wait that ran out) sets a per-device error word that
 *    gdn_check_device_error reads and clears.
 *  - Streams: gdn_stream_t is a cudaStream_t (NULL = the legacy default).
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *gdn_stream_t; /* same type as cudaStream_t */

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misaligned buffer, overlap */
  GDN_ERR_UNSUPPORTED = 2,    /* valid but not implemented (e.g. D_k = 32) */
  GDN_ERR_ROLLBACK_RANGE = 3, /* the requested state was not stored */
  GDN_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
  GDN_ERR_TIMEOUT = 5,        /* a bounded device-side wait ran out */
  GDN_ERR_DEVICE_ARG = 6      /* the device found a bad argument (cu_seqlens, or a
                                 gate range the chunked path cannot represent) */
} gdn_status;

typedef enum { GDN_MODE_GDA = 0, GDN_MODE_KDA = 1 } gdn_mode;
typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Grouped-query heads: q and k may carry H_qk heads for H value heads (H a
 * multiple of H_qk), and the op reads them per value head instead of the
 * caller repeating them ("models : avoid Q and K repeats when using fused
 * GDA", llama.cpp commits page, tag b9752). Value head h reads q/k head
 *   GDN_QK_TILED:   h % H_qk            (heads repeated as a whole block)
 *   GDN_QK_GROUPED: h / (H / H_qk)      (each q/k head repeated in place)
 * Both orders occur ("reorder v heads for linear attention to avoid
 * expensive interleaved repeat", same page, "support qwen3.5 series"). */
typedef enum { GDN_QK_TILED = 0, GDN_QK_GROUPED = 1 } gdn_qk_map;

/* Message of the calling thread's last failed call ("" if none). */
const char *gdn_last_error(void);

/* Version string of the library. */
const char *gdn_version(void);

/* ------------------------------------------------------------------------
 * Uniform-length forward: decode (T = 1) and speculative verify
 * (T = draft_max + 1). Runs the token recurrence on the recurrent kernel.
 * ---------------------------------------------------------------------- */
typedef struct {
  int n_seqs;         /* N >= 0 independent sequences */
  int T;              /* tokens per sequence, >= 0 */
  int H;              /* value heads (v, g, beta, out and the state have H heads) */
  int D_k, D_v;       /* head sizes, each 64 or 128 */
  gdn_dtype in_dtype; /* dtype of q, k, v; g and beta are always fp32 */
  float scale;        /* output scale; 0 means 1/sqrt(D_k) */
  int H_qk;           /* heads of q and k; 0 means H; must divide H */
  gdn_qk_map qk_map;  /* value head -> q/k head when H_qk < H */
} gdn_shape;

/*
 * q, k        device [N*T][H_qk][D_k]  in_dtype (token n*T+t is token t of seq n)
 * v           device [N*T][H][D_v]  in_dtype
 * g           device fp32 [N*T][H] (GDA) or [N*T][H][D_k] (KDA)
 * beta        device fp32 [N*T][H]
 * state_in    device array of N device pointers; state_in[s] -> fp32
 *             [H][D_k][D_v], the state before this call (any slot a rollback
 *             chose). A NULL entry means a zero state. Read only.
 * state_slots device fp32 [N][n_slots][H][D_k][D_v]; slot j of sequence s
 *             receives the state after token T-n_slots+j. No state_in[s] may
 *             point into it: the kernel checks each pointer, leaves that
 *             sequence unwritten and reports GDN_ERR_DEVICE_ARG through
 *             gdn_check_device_error.
 * out         device fp32 [N*T][H][D_v]
 * n_slots     K >= 1
 * Returns GDN_OK once the kernel is enqueued on `stream`.
 * The kernel is a programmatic dependent launch: its blocks may be scheduled
 * while the previous kernel of `stream` is still running, but they read and
 * write no memory until that kernel has completed, so stream order holds for
 * every argument as for an ordinary launch.
 */
gdn_status gdn_forward(const gdn_shape *shape, const void *q, const void *k,
                       const void *v, const float *g, const float *beta,
                       const float *const *state_in, float *state_slots,
                       float *out, int n_slots, gdn_mode mode,
                       gdn_stream_t stream);

/*
 * gdn_forward with the per-token buffers in host memory (no counterpart on
 * the pages): q, k, v, g, beta and out may each be page-locked host memory
 * (cudaMallocHost / cudaHostAlloc / cudaHostRegister, mapped into the
 * device's address space at the same address, as unified addressing does)
 * or device memory. The kernel reads the token rows and writes the outputs
 * over the host link itself, so no separate copy (and no event between a copy
 * stream and the launch stream) stands between consecutive calls; the state
 * pointers and slots stay device memory. Layouts, results (bit for bit) and
 * the programmatic launch are those of gdn_forward.
 * Errors: GDN_ERR_INVALID_ARG when one of the six pointers is pageable host
 * memory or unknown to CUDA (each is checked with cudaPointerGetAttributes
 * before anything is enqueued), otherwise as gdn_forward. The host memory
 * must stay valid and unmodified until the call has completed on `stream`.
 */
gdn_status gdn_forward_host(const gdn_shape *shape, const void *q, const void *k,
                            const void *v, const float *g, const float *beta,
                            const float *const *state_in, float *state_slots,
                            float *out, int n_slots, gdn_mode mode,
                            gdn_stream_t stream);

/* ------------------------------------------------------------------------
 * Varlen chunked prefill ("llama : enable chunked fused GDN path", llama.cpp
 * commits, tag b9752). Sequence s covers packed tokens
 * [cu_seqlens[s], cu_seqlens[s+1]). Routing:
 *  - bf16 inputs with D_k = D_v = 128: tokens [0, L_s - n_slots) of each
 *    sequence run through the chunked (chunk 64, WY/UT-transform)
 *    tensor-core kernels, with the last partial chunk padded by no-op rows;
 *    the last n_slots tokens run through the recurrent kernel, which writes
 *    the slots. With n_slots = 1 the slot is the final state, so every token
 *    runs through the chunked kernels, which write it. The result equals the
 *    token recurrence up to rounding (bf16 tensor-core operands, fp32
 *    accumulation and fp32 state).
 *  - fp32 inputs (whose 1e-5 accuracy bf16 operands cannot meet) and head
 *    sizes of 64: every token runs through the recurrent kernel on the GPU,
 *    as the pages' chunked path also falls back to the token loop ("Enable
 *    GDN also for prefill, move TODO for chunked_GDN", llama.cpp commits).
 * ---------------------------------------------------------------------- */
typedef struct {
  int n_seqs;         /* N >= 1 */
  int total_tokens;   /* Ntok = cu_seqlens[N] */
  int H;              /* value heads */
  int D_k, D_v;       /* each 64 or 128 */
  gdn_dtype in_dtype; /* GDN_BF16 or GDN_F32 (see the routing note below) */
  float scale;        /* 0 means 1/sqrt(D_k) */
  int H_qk;           /* heads of q and k; 0 means H; must divide H */
  gdn_qk_map qk_map;  /* value head -> q/k head when H_qk < H */
} gdn_varlen_shape;

/* Bytes of device workspace gdn_forward_chunked needs for this shape in either
 * gate mode (the per-row gate mode needs more; this is its figure). */
size_t gdn_chunked_workspace_size(const gdn_varlen_shape *shape, int n_slots);

/*
 * cu_seqlens  device int32 [N+1], non-decreasing, cu_seqlens[0] = 0,
 *             cu_seqlens[N] = total_tokens (checked on the device)
 * q, k, v, g, beta, out: as gdn_forward with Ntok = total_tokens (q, k with
 *             H_qk heads)
 * state_in    device array of N device pointers (NULL entry = zero state)
 * state_slots device fp32 [N][n_slots][H][D_k][D_v]
 * workspace   device buffer of at least gdn_chunked_workspace_size bytes,
 *             256-byte aligned; its contents on entry do not matter.
 * Gate range: inside each 64-token chunk the cumulative log-gate from the
 * chunk's first token must stay within [-80, 80] for per-row gates. For
 * scalar gates only growth is limited (no interval of the chunk may grow by
 * more than e^80); any decay is computed, and a gate of -inf resets the state
 * exactly. The chunk form keeps its decay factors e^(+-gamma) in bf16/fp32,
 * whose range ends near e^88. A chunk outside the range (a NaN gate too)
 * leaves its outputs undefined and makes gdn_check_device_error return
 * GDN_ERR_DEVICE_ARG; gdn_forward (the token loop) has no such limit, and
 * the last n_slots tokens of each sequence, which run through it, neither.
 */
gdn_status gdn_forward_chunked(const gdn_varlen_shape *shape,
                               const int32_t *cu_seqlens, const void *q,
                               const void *k, const void *v, const float *g,
                               const float *beta, const float *const *state_in,
                               float *state_slots, float *out, int n_slots,
                               gdn_mode mode, void *workspace,
                               size_t workspace_bytes, gdn_stream_t stream);

/* ------------------------------------------------------------------------
 * Allocation-free chunked prefill. The pages describe no counterpart: this is
 * a convenience of this library. Some callers cannot give the chunked call a
 * workspace because they may not allocate device memory at all: a host
 * application that owns every device byte through its own pool, or a loop
 * that must never pay for a device allocation (cudaMalloc can synchronise the
 * whole device). This entry point computes exactly what gdn_forward_chunked
 * computes, with the same arguments minus the workspace; its scratch is a
 * fixed 256 MiB device array inside the library, which every GPU that loads
 * the chunked kernels holds until the process exits.
 *  - Limit: shapes whose workspace for the given mode exceeds
 *    gdn_noalloc_scratch_bytes() are rejected with GDN_ERR_UNSUPPORTED and a
 *    message naming both sizes. The scalar-gate mode needs about 33 KB per
 *    (chunk of 64 tokens, head), the per-row mode about 65 KB, plus 64 KB of
 *    fp32 state per (sequence, head): 1 x 4096 tokens x 32 heads needs about
 *    140 MB per-row and fits; 8 x ~4k tokens x 16 heads does not.
 *  - The first call on a device looks up the array's device address with
 *    that device current and keeps it for the life of the process; make that
 *    first call before any stream capture. A cudaDeviceReset invalidates the
 *    kept address (as it does the error word's): do not call this entry
 *    point after resetting a device it was used on.
 *  - Every call on a device shares the one array and it keeps the previous
 *    call's contents; nothing in it needs to start at zero (the work list
 *    rewrites what the later kernels read). Calls that can overlap on the
 *    GPU (different streams without ordering) race on it: serialise them.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine.
 * ---------------------------------------------------------------------- */
gdn_status gdn_forward_chunked_noalloc(const gdn_varlen_shape *shape,
                                       const int32_t *cu_seqlens, const void *q,
                                       const void *k, const void *v, const float *g,
                                       const float *beta, const float *const *state_in,
                                       float *state_slots, float *out, int n_slots,
                                       gdn_mode mode, gdn_stream_t stream);

/* Size in bytes of the built-in scratch array of gdn_forward_chunked_noalloc. */
size_t gdn_noalloc_scratch_bytes(void);

/* ------------------------------------------------------------------------
 * Chunked prefill with state checkpoints ("llama-memory: enable
 * checkpointing with partial rollback", koboldcpp commits page, tag
 * v1.113.1): the slots keep only the last n_slots states of a call, so a
 * caller that may later keep fewer tokens (a shared prompt prefix, a
 * rejected continuation) also wants states at regular positions. Computes
 * exactly what gdn_forward_chunked computes and in addition stores
 *   checkpoints[s][m] = state after token (m+1)*ckpt_every - 1 of sequence s
 * (0-based within the sequence) for every m < max_ckpts with
 * (m+1)*ckpt_every <= L_s. Entries a sequence does not reach are not
 * written.
 * checkpoints  device fp32 [N][max_ckpts][H][D_k][D_v], 16-byte aligned;
 *              must not overlap state_in, state_slots or out
 * ckpt_every   positive multiple of 64 (a chunk boundary)
 * max_ckpts    >= 1
 * The other arguments are those of gdn_forward_chunked.
 * ---------------------------------------------------------------------- */
gdn_status gdn_forward_chunked_checkpointed(
    const gdn_varlen_shape *shape, const int32_t *cu_seqlens, const void *q, const void *k,
    const void *v, const float *g, const float *beta, const float *const *state_in,
    float *state_slots, float *out, int n_slots, gdn_mode mode, float *checkpoints,
    int ckpt_every, int max_ckpts, void *workspace, size_t workspace_bytes,
    gdn_stream_t stream);

/*
 * Where to restart a sequence of L tokens, last run with n_slots slots and
 * checkpoints every ckpt_every tokens (max_ckpts of them), that keeps only
 * its first n_keep tokens (0 <= n_keep <= L):
 *   *source = 0: start from that call's state_in and replay tokens
 *                [0, n_keep) (*index = -1, *replay_from = 0);
 *   *source = 1: start from checkpoint *index and replay tokens
 *                [*replay_from, n_keep);
 *   *source = 2: the state is slot *index, nothing to replay
 *                (*replay_from = n_keep).
 * A slot is chosen whenever one holds the state; otherwise the latest
 * checkpoint at or before n_keep. GDN_ERR_INVALID_ARG for bad arguments.
 * Host only.
 */
gdn_status gdn_checkpoint_select(int n_keep, int L, int n_slots, int ckpt_every,
                                 int max_ckpts, int *source, int *index,
                                 int *replay_from);

/* ------------------------------------------------------------------------
 * Rollback bookkeeping: a host-side table with one entry per sequence (the
 * recurrent memory's per-sequence record of which stored state is live,
 * "llama-memory-recurrent: clear rs_idx in clear", koboldcpp commits, tag
 * v1.113.1). No device work.
 * ---------------------------------------------------------------------- */
typedef struct gdn_seq_table gdn_seq_table;

gdn_status gdn_seq_table_create(int n_seqs, int n_slots, gdn_seq_table **out);
void gdn_seq_table_destroy(gdn_seq_table *table);

/* Records that the last forward ran T_last tokens of sequence `seq`. */
gdn_status gdn_seq_table_record(gdn_seq_table *table, int seq, int T_last);

/* Forgets the last forward of `seq` (only n_accepted = 0 is valid after). */
gdn_status gdn_seq_table_clear(gdn_seq_table *table, int seq);

/*
 * Which state holds sequence `seq` after accepting the first n_accepted
 * tokens of its last forward: *slot = -1 means "the state_in of that forward
 * is unchanged"; otherwise the slot index. GDN_ERR_ROLLBACK_RANGE when
 * n_accepted is outside [0, T_last] or the token was not snapshotted (the
 * caller must recompute). The table is not modified.
 */
gdn_status gdn_rollback(const gdn_seq_table *table, int seq, int n_accepted,
                        int *slot);

/*
 * Device address of slot `slot` of sequence `seq` in a state_slots buffer of
 * the layout above, for building the next call's state_in array. Pure
 * address arithmetic; *out = NULL for slot = -1.
 */
gdn_status gdn_slot_state_ptr(const float *state_slots, int seq, int slot,
                              int n_slots, int H, int D_k, int D_v,
                              const float **out);

/* ------------------------------------------------------------------------
 * Device error word of the current device: synchronises `stream`, then
 * reads and clears the word. GDN_OK if no kernel reported a problem since
 * the last check; else GDN_ERR_TIMEOUT or GDN_ERR_DEVICE_ARG with a message.
 * ---------------------------------------------------------------------- */
gdn_status gdn_check_device_error(gdn_stream_t stream);

/*
 * Maps a value of the device error word to the status gdn_check_device_error
 * returns for it, and sets the calling thread's gdn_last_error message to the
 * text it would give: GDN_OK for 0; GDN_ERR_TIMEOUT for a bounded wait that
 * ran out (the message names the wait site, bits 8..15, and the chunk, bits
 * 16..30); GDN_ERR_DEVICE_ARG for the argument conditions above. Host only,
 * no device access.
 */
gdn_status gdn_decode_device_error(int word);

/*
 * Device address of the current device's error word (one int), for a
 * caller's own kernels that want to report through gdn_check_device_error:
 * they set it with atomicCAS(word, 0, value) so that the first condition
 * wins, as the library's kernels do. The address is looked up once per
 * device and is not valid after cudaDeviceReset.
 */
gdn_status gdn_device_error_word(int **word);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
