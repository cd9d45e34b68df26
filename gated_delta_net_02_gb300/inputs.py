"""Seeded synthetic inputs shaped like the GDN workloads.

This module is shared by the tests, the benchmark and the smoke check, and
feeds both the CUDA path and the fp64 oracle. It holds no GDN arithmetic: only
the input recipe (random draws, the q/k L2 normalisation and the gate and
beta activations the caller applies before the op).

Recipe (all draws from ``torch.Generator('cpu')`` seeded per workload, in a
fixed order; "N(0, s)" has standard deviation s):
  q, k   ~ N(0,1), then L2-normalised over D_k per (token, head), then cast to
         the input dtype (bf16 or fp32)
  v      ~ N(0,1), cast to the input dtype
  beta   = sigmoid(N(0,1)), fp32 [Ntok, H]
  g      = -softplus(N(0,1)), fp32 [Ntok, H]          (GDA, scalar gate)
         = -softplus(N(0,1)) * 0.1, fp32 [Ntok, H, D_k] (KDA, per-row gate)
  state  zeros, or ~ N(0, 0.05) fp32 [N, H, D_k, D_v]
Tokens of all sequences are packed: token row n, head h is q[n, h, :].
"""
from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass
class GDNBatch:
    q: torch.Tensor            # [Ntok, H_qk, Dk] (H_qk = H unless grouped-query)
    k: torch.Tensor            # [Ntok, H_qk, Dk]
    v: torch.Tensor            # [Ntok, H, Dv]
    g: torch.Tensor            # [Ntok, H] or [Ntok, H, Dk], fp32
    beta: torch.Tensor         # [Ntok, H], fp32
    state: torch.Tensor        # [N, H, Dk, Dv], fp32
    mode: str                  # "gda" | "kda"
    scale: float
    seq_len: torch.Tensor      # int64 [N]
    n_slots: int = 1
    meta: dict = field(default_factory=dict)
    qk_map: str = "tiled"      # value head -> q/k head when H_qk < H: "tiled" | "grouped"

    @property
    def n_seqs(self) -> int:
        return int(self.state.shape[0])

    @property
    def cu_seqlens(self) -> torch.Tensor:
        cu = torch.zeros(self.n_seqs + 1, dtype=torch.int64)
        cu[1:] = torch.cumsum(self.seq_len, 0)
        return cu


def _tokens(gen, ntok, H, Dk, Dv, dtype, mode, kda_gate_scale=0.1, H_qk=None):
    Hq = H if H_qk is None else H_qk
    q = torch.randn(ntok, Hq, Dk, generator=gen)
    k = torch.randn(ntok, Hq, Dk, generator=gen)
    v = torch.randn(ntok, H, Dv, generator=gen)
    q = q / q.norm(dim=-1, keepdim=True)
    k = k / k.norm(dim=-1, keepdim=True)
    beta = torch.sigmoid(torch.randn(ntok, H, generator=gen))
    if mode == "gda":
        g = -torch.nn.functional.softplus(torch.randn(ntok, H, generator=gen))
    elif mode == "kda":
        g = -torch.nn.functional.softplus(
            torch.randn(ntok, H, Dk, generator=gen)) * kda_gate_scale
    else:
        raise ValueError(mode)
    return (q.to(dtype).contiguous(), k.to(dtype).contiguous(),
            v.to(dtype).contiguous(), g.float().contiguous(),
            beta.float().contiguous())


def _state(gen, N, H, Dk, Dv, std):
    if std == 0.0:
        return torch.zeros(N, H, Dk, Dv, dtype=torch.float32)
    return (torch.randn(N, H, Dk, Dv, generator=gen) * std).float().contiguous()


def make_batch(seed: int, seq_len, H: int, Dk: int, Dv: int, *,
               dtype=torch.bfloat16, mode: str = "gda", state_std: float = 0.05,
               n_slots: int = 1, scale: Optional[float] = None,
               kda_gate_scale: float = 0.1, H_qk: Optional[int] = None,
               qk_map: str = "tiled") -> GDNBatch:
    """A packed batch of len(seq_len) sequences drawn with the recipe above.
    H_qk < H gives q and k H_qk heads (grouped-query layout, read per value
    head through qk_map)."""
    gen = torch.Generator("cpu")
    gen.manual_seed(seed)
    seq_len = torch.as_tensor(seq_len, dtype=torch.int64)
    N = int(seq_len.numel())
    ntok = int(seq_len.sum())
    state = _state(gen, N, H, Dk, Dv, state_std)
    q, k, v, g, beta = _tokens(gen, ntok, H, Dk, Dv, dtype, mode, kda_gate_scale, H_qk)
    if scale is None:
        scale = Dk ** -0.5
    return GDNBatch(q, k, v, g, beta, state, mode, float(scale), seq_len, n_slots,
                    qk_map=qk_map)


# ---- the five workloads ---------------------------------------------------

def tiny_gda(seed: int = 0) -> GDNBatch:
    """1 sequence, H=4, D_k=D_v=64, T=32, fp32 everything, K=1, zero state."""
    return make_batch(seed, [32], 4, 64, 64, dtype=torch.float32, mode="gda",
                      state_std=0.0, n_slots=1)


def decode_state(seed: int = 1, N: int = 64, H: int = 16, D: int = 128) -> torch.Tensor:
    """Decode start state [N, H, D, D] ~ N(0, 0.05)."""
    gen = torch.Generator("cpu")
    gen.manual_seed(seed)
    return _state(gen, N, H, D, D, 0.05)


def decode_tokens(seed: int, step: int, N: int = 64, H: int = 16, D: int = 128,
                  dtype=torch.bfloat16):
    """Fresh tokens for decode step ``step``: one token per sequence.
    Returns (q, k, v, g, beta) with Ntok = N."""
    gen = torch.Generator("cpu")
    gen.manual_seed(seed * 1_000_003 + step + 1)
    return _tokens(gen, N, H, D, D, dtype, "gda")


def verify_batch(seed: int = 2, N: int = 32, T: int = 8, H: int = 16,
                 D: int = 128, n_slots: int = 8) -> GDNBatch:
    """Speculative verify: N sequences of T = draft_max + 1 tokens, K slots,
    plus n_accepted ~ U{0..T} per sequence in meta['n_accepted']."""
    b = make_batch(seed, [T] * N, H, D, D, dtype=torch.bfloat16, mode="gda",
                   state_std=0.05, n_slots=n_slots)
    gen = torch.Generator("cpu")
    gen.manual_seed(seed + 7919)
    b.meta["n_accepted"] = torch.randint(0, T + 1, (N,), generator=gen)
    return b


def kda_prefill(seed: int = 3, T: int = 4096, H: int = 32, D: int = 128,
                n_slots: int = 1) -> GDNBatch:
    """One long KDA sequence (per-row gate), bf16 q/k/v."""
    return make_batch(seed, [T], H, D, D, dtype=torch.bfloat16, mode="kda",
                      state_std=0.05, n_slots=n_slots)


def varlen_lengths(seed: int = 4, N: int = 8, lo: int = 512, hi: int = 8192):
    gen = torch.Generator("cpu")
    gen.manual_seed(seed)
    return torch.randint(lo, hi + 1, (N,), generator=gen)


def varlen_prefill(seed: int = 4, N: int = 8, H: int = 16, D: int = 128,
                   n_slots: int = 8, lo: int = 512, hi: int = 8192) -> GDNBatch:
    """N packed GDA sequences with lengths ~ U[lo, hi], K slots each."""
    lens = varlen_lengths(seed, N, lo, hi)
    return make_batch(seed + 1, lens, H, D, D, dtype=torch.bfloat16, mode="gda",
                      state_std=0.05, n_slots=n_slots)


def to_f64(t: torch.Tensor):
    """Exact widening to a float64 numpy array (bf16 and fp32 widen exactly)."""
    return t.detach().to("cpu").double().numpy()
