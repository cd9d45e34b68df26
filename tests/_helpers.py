"""Shared test helpers: run the CUDA path and the oracle on one batch, and
compare them with the tolerances of the op.

Tolerance metric: relative L2 error ||x - x_ref|| / ||x_ref|| over a whole
tensor, in fp64, against the fp64 oracle: 1e-5 for fp32 inputs and 5e-3 for
bf16 inputs.
"""
import numpy as np
import torch

import oracle
from gated_delta_net_02_gb300 import inputs

TOL = {torch.float32: 1e-5, torch.bfloat16: 5e-3}


def rel_l2(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def oracle_run(b: inputs.GDNBatch, n_slots=None, threads=0):
    n_slots = b.n_slots if n_slots is None else n_slots
    cu = b.cu_seqlens.numpy()
    return oracle.forward(
        inputs.to_f64(b.q), inputs.to_f64(b.k), inputs.to_f64(b.v), inputs.to_f64(b.g),
        inputs.to_f64(b.beta), inputs.to_f64(b.state), mode=b.mode, scale=b.scale,
        n_slots=n_slots, seq_start=cu[:-1], seq_len=b.seq_len.numpy(), threads=threads,
        qk_map=b.qk_map)


def to_dev(b: inputs.GDNBatch, dev="cuda"):
    return {name: getattr(b, name).to(dev).contiguous()
            for name in ("q", "k", "v", "g", "beta", "state")}


def gpu_forward(b: inputs.GDNBatch, n_slots=None, state_ptrs=None, slots=None,
                out=None, stream=None, check=True, dev_tensors=None):
    """Runs gdn_forward (uniform T) on cuda:0 and returns (out, slots) as
    torch tensors on the device."""
    from gated_delta_net_02_gb300 import gdn
    n_slots = b.n_slots if n_slots is None else n_slots
    N = b.n_seqs
    T = int(b.seq_len[0]) if N else 0
    assert bool((b.seq_len == T).all()), "gdn_forward needs uniform lengths"
    d = dev_tensors or to_dev(b)
    H, Dk = b.v.shape[1], b.q.shape[2]
    Dv = b.v.shape[2]
    if slots is None:
        slots = torch.full((N, n_slots, H, Dk, Dv), float("nan"), device="cuda")
    if out is None:
        out = torch.full((N * T, H, Dv), float("nan"), device="cuda")
    if state_ptrs is None:
        state_ptrs = gdn.state_ptr_array(gdn.per_seq_state_ptrs(d["state"], N), "cuda")
    shape = gdn.gdn_shape(N, T, H, Dk, Dv, gdn.dtype_code(b.q.dtype), b.scale,
                          b.q.shape[1], gdn.QK_MAPS[b.qk_map])
    gdn.gdn_forward(shape, d["q"], d["k"], d["v"], d["g"], d["beta"], state_ptrs, slots, out,
                    n_slots, b.mode, stream)
    if check:
        gdn.gdn_check_device_error(stream)
    return out, slots
