"""fp64 CPU oracle of the gated delta-net recurrence.

TEST INFRASTRUCTURE: only ``tests/``, the package smoke check and the
benchmark's CPU-baseline leg may import this module. The CUDA path never
imports it and shares no code with it.

The arithmetic lives in ``gdn_oracle.c`` (plain sequential fp64 C); this module
only marshals numpy arrays. What the recurrence computes, and the sources it
follows, are stated at the top of that file.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(_build.build())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int64)
        lib.gdn_oracle_forward.restype = ctypes.c_int
        lib.gdn_oracle_forward.argtypes = [
            ctypes.c_int, ip, ip, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, dp, dp, dp, dp, dp, ctypes.c_double, dp, dp, dp,
            ctypes.c_int, dp, ctypes.c_int]
        lib.gdn_oracle_rollback_slot.restype = ctypes.c_int
        lib.gdn_oracle_rollback_slot.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.POINTER(ctypes.c_int)]
        lib.gdn_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a, name):
    a = np.asarray(a)
    if a.dtype != np.float64:
        raise TypeError(f"{name}: oracle inputs are float64, got {a.dtype}")
    return np.ascontiguousarray(a)


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_load().gdn_oracle_max_threads())


class RollbackRangeError(ValueError):
    """The accepted prefix ends at a token whose state was not snapshotted."""


def qk_head_index(H, H_qk, qk_map="tiled"):
    """Which q/k head each of the H value heads reads when q and k carry
    H_qk <= H heads (grouped-query layout: the op broadcasts q and k instead
    of the caller repeating them, "models : avoid Q and K repeats when using
    fused GDA", llama.cpp commits page, tag b9752). Two head orders exist
    ("reorder v heads for linear attention to avoid expensive interleaved
    repeat", same page, "support qwen3.5 series"): "tiled" reads head
    h mod H_qk, "grouped" reads head h // (H // H_qk)."""
    if H_qk <= 0 or H % H_qk:
        raise ValueError(f"H={H} is not a multiple of H_qk={H_qk}")
    h = np.arange(H)
    if qk_map == "tiled":
        return h % H_qk
    if qk_map == "grouped":
        return h // (H // H_qk)
    raise ValueError(f"qk_map {qk_map!r}")


def forward(q, k, v, g, beta, state_in, *, mode="gda", scale=None, n_slots=0,
            seq_start=None, seq_len=None, threads=0, want_state=True, qk_map="tiled"):
    """Runs the token recurrence in fp64.

    q, k: [Ntok, H_qk, Dk] with H_qk dividing H (value head h reads q/k head
    qk_head_index(H, H_qk, qk_map)[h]); v: [Ntok, H, Dv]; g: [Ntok, H] (gda) or
    [Ntok, H, Dk] (kda); beta: [Ntok, H]; state_in: [N, H, Dk, Dv].
    Sequences are either uniform (seq_start/seq_len omitted: N equal runs of
    Ntok/N tokens) or given by seq_start/seq_len (int64 [N]).
    scale=None means 1/sqrt(Dk).
    Returns (out [Ntok,H,Dv], state_out [N,H,Dk,Dv] or None,
    slots [N,n_slots,H,Dk,Dv] or None). Slots a short sequence does not reach
    are NaN.
    """
    q, k, v = _f64(q, "q"), _f64(k, "k"), _f64(v, "v")
    g, beta, state_in = _f64(g, "g"), _f64(beta, "beta"), _f64(state_in, "state_in")
    if q.shape[1] != v.shape[1]:  # broadcast the q/k heads to the value heads
        idx = qk_head_index(v.shape[1], q.shape[1], qk_map)
        q = np.ascontiguousarray(q[:, idx])
        k = np.ascontiguousarray(k[:, idx])
    ntok, H, Dk = q.shape
    Dv = v.shape[2]
    N = state_in.shape[0]
    assert k.shape == (ntok, H, Dk) and v.shape == (ntok, H, Dv)
    assert beta.shape == (ntok, H) and state_in.shape == (N, H, Dk, Dv)
    kda = {"gda": 0, "kda": 1}[mode]
    assert g.shape == ((ntok, H, Dk) if kda else (ntok, H))
    if seq_start is None:
        assert N > 0 and ntok % N == 0
        T = ntok // N
        seq_start = np.arange(N, dtype=np.int64) * T
        seq_len = np.full(N, T, dtype=np.int64)
    seq_start = np.ascontiguousarray(seq_start, dtype=np.int64)
    seq_len = np.ascontiguousarray(seq_len, dtype=np.int64)
    assert seq_start.shape == (N,) and seq_len.shape == (N,)
    if scale is None:
        scale = 1.0 / np.sqrt(Dk)
    out = np.zeros((ntok, H, Dv), dtype=np.float64)
    state_out = np.empty((N, H, Dk, Dv), dtype=np.float64) if want_state else None
    slots = (np.full((N, n_slots, H, Dk, Dv), np.nan, dtype=np.float64)
             if n_slots > 0 else None)
    ip = ctypes.POINTER(ctypes.c_int64)
    rc = _load().gdn_oracle_forward(
        N, seq_start.ctypes.data_as(ip), seq_len.ctypes.data_as(ip), H, Dk, Dv,
        kda, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
        _ptr(state_in), _ptr(out), _ptr(state_out), int(n_slots), _ptr(slots),
        int(threads))
    if rc != 0:
        raise ValueError(f"gdn_oracle_forward failed with code {rc}")
    return out, state_out, slots


def rollback_slot(T: int, K: int, n_accepted: int) -> int:
    """Slot index holding the state after n_accepted tokens, or -1 for
    "keep the input state". Raises RollbackRangeError when that state was
    not stored."""
    slot = ctypes.c_int(-2)
    rc = _load().gdn_oracle_rollback_slot(int(T), int(K), int(n_accepted),
                                          ctypes.byref(slot))
    if rc == 3:
        raise RollbackRangeError(f"n_accepted={n_accepted} with T={T}, K={K}")
    if rc != 0:
        raise ValueError(f"gdn_oracle_rollback_slot failed with code {rc}")
    return slot.value


__all__ = ["forward", "rollback_slot", "max_threads", "qk_head_index", "RollbackRangeError"]
