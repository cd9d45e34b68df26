// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernels. Host-only declarations; no CUDA types beyond cudaStream_t.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

// Recurrent (token-loop) forward over n_seqs sequences of one head group.
struct RecurrentArgs {
  const void *q, *k, *v;        // q, k [Ntok][Hqk][Dk]; v [Ntok][H][Dv]; bf16 or fp32
  const float *g, *beta;        // [Ntok][H](x Dk for KDA), [Ntok][H]
  const float *const *state_in; // device [n_seqs] pointers, NULL = zero
  float *slots;                 // [n_seqs][n_slots][H][Dk][Dv]
  float *out;                   // [Ntok][H][Dv]
  const int *tok_start;         // device [n_seqs] first token, or NULL (s*T)
  const int *seq_len;           // device [n_seqs] tokens, or NULL (T)
  int n_seqs, T, H, Dk, Dv, n_slots;
  int Hqk;                      // q/k heads (divides H)
  bool qk_grouped;              // value head h reads q/k head h / (H / Hqk), else h % Hqk
  bool kda, bf16;
  float scale;
  int *err;                     // device error word
  // optional checkpoints: the state after sequence position p (1-based count
  // of tokens) goes to ckpt[s][p / ckpt_every - 1] when p % ckpt_every == 0
  float *ckpt = nullptr;        // [n_seqs][max_ckpts][H][Dk][Dv]
  const int *pos0 = nullptr;    // device [n_seqs] position of the first token (NULL = 0)
  int ckpt_every = 0, max_ckpts = 0;
  // programmatic launch (gdn_forward only: tok_start and seq_len must be NULL,
  // since the kernel reads its scalars before waiting for its predecessor)
  bool pdl = false;
  // long serial chains (the chunked call's token-loop route): 128 x 128
  // heads with fp32 inputs take a narrower slice per CTA (16 lanes across
  // the key rows, 32 columns), which shortens each token's step
  bool long_chains = false;
  // q, k, v, g, beta and out may be page-locked host memory (mapped into the
  // device's address space): the token tiles are read with ordinary loads,
  // not bulk copies (gdn_forward_host); requires pdl
  bool host_io = false;
};

cudaError_t launch_recurrent(const RecurrentArgs &a, cudaStream_t stream);

// Chunked (tensor-core) prefill of varlen sequences; see chunked.cu.
struct ChunkedArgs {
  const int32_t *cu_seqlens;    // device [n_seqs + 1]
  const void *q, *k, *v;        // bf16 (tensor-core route) or fp32
  const float *g, *beta;
  const float *const *state_in; // device [n_seqs]
  float *slots;
  float *out;
  int n_seqs, total_tokens, H, Dk, Dv, n_slots;
  int Hqk;                      // q/k heads (divides H)
  bool qk_grouped;              // value head -> q/k head map (see RecurrentArgs)
  bool bf16;                    // q, k, v dtype (else fp32)
  bool kda;
  float scale;
  void *workspace;
  size_t workspace_bytes;
  int *err;
  float *ckpt = nullptr;        // optional checkpoints (see RecurrentArgs)
  int ckpt_every = 0, max_ckpts = 0;
};

// bf16 inputs with 128 x 128 heads run on the tensor cores; anything else
// goes through the recurrent kernel, token by token.
inline bool tensor_core_route(bool bf16, int Dk, int Dv) { return bf16 && Dk == 128 && Dv == 128; }
size_t chunked_workspace_size(int n_seqs, int total_tokens, int H, int Dk, int Dv, bool bf16);
// Bytes one call of the given gate mode needs (at most the size above).
size_t chunked_workspace_need(int n_seqs, int total_tokens, int H, int Dk, int Dv, bool kda,
                              bool bf16);
cudaError_t launch_chunked(const ChunkedArgs &a, cudaStream_t stream);

// The chunked path on the library's fixed scratch area (no workspace
// argument); see gdn_forward_chunked_noalloc in gdn.h.
size_t static_scratch_bytes();
cudaError_t launch_chunked_static(ChunkedArgs a, cudaStream_t stream, size_t *need);

}  // namespace gdn
