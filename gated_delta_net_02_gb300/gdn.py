"""Thin ctypes binding of libgdn (include/gdn.h): same names, argument
marshalling only. Every step of the op runs in the library's CUDA kernels.

Device buffers may be passed as torch tensors (their data_ptr is used) or as
integer addresses. A non-OK status raises GDNError carrying the status code
and the library's message. If the library is missing this module raises at
import time: there is no fallback.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libgdn.so")

GDN_OK = 0
GDN_ERR_INVALID_ARG = 1
GDN_ERR_UNSUPPORTED = 2
GDN_ERR_ROLLBACK_RANGE = 3
GDN_ERR_CUDA = 4
GDN_ERR_TIMEOUT = 5
GDN_ERR_DEVICE_ARG = 6

GDN_MODE_GDA = 0
GDN_MODE_KDA = 1
GDN_F32 = 0
GDN_BF16 = 1

_MODES = {"gda": GDN_MODE_GDA, "kda": GDN_MODE_KDA,
          GDN_MODE_GDA: GDN_MODE_GDA, GDN_MODE_KDA: GDN_MODE_KDA}


class GDNError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"[gdn status {status}] {message}")
        self.status = status


GDN_QK_TILED, GDN_QK_GROUPED = 0, 1
QK_MAPS = {"tiled": GDN_QK_TILED, "grouped": GDN_QK_GROUPED}


class gdn_shape(ctypes.Structure):
    # H_qk = 0 (the default) means q and k have H heads
    _fields_ = [("n_seqs", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("D_k", ctypes.c_int), ("D_v", ctypes.c_int),
                ("in_dtype", ctypes.c_int), ("scale", ctypes.c_float),
                ("H_qk", ctypes.c_int), ("qk_map", ctypes.c_int)]


class gdn_varlen_shape(ctypes.Structure):
    _fields_ = [("n_seqs", ctypes.c_int), ("total_tokens", ctypes.c_int),
                ("H", ctypes.c_int), ("D_k", ctypes.c_int), ("D_v", ctypes.c_int),
                ("in_dtype", ctypes.c_int), ("scale", ctypes.c_float),
                ("H_qk", ctypes.c_int), ("qk_map", ctypes.c_int)]


if not os.path.exists(LIB_PATH):
    raise ImportError(f"libgdn.so is not built ({LIB_PATH}); run "
                      "gated_delta_net_02_gb300/build.py or __graft_entry__.build()")
lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_i = ctypes.c_int
_st = ctypes.c_int

lib.gdn_last_error.restype = ctypes.c_char_p
lib.gdn_version.restype = ctypes.c_char_p
lib.gdn_forward.restype = _st
lib.gdn_forward.argtypes = [ctypes.POINTER(gdn_shape), _vp, _vp, _vp, _vp, _vp, _vp,
                            _vp, _vp, _i, _i, _vp]
lib.gdn_forward_host.restype = _st
lib.gdn_forward_host.argtypes = lib.gdn_forward.argtypes
lib.gdn_chunked_workspace_size.restype = ctypes.c_size_t
lib.gdn_chunked_workspace_size.argtypes = [ctypes.POINTER(gdn_varlen_shape), _i]
lib.gdn_forward_chunked.restype = _st
lib.gdn_forward_chunked.argtypes = [ctypes.POINTER(gdn_varlen_shape), _vp, _vp, _vp, _vp,
                                    _vp, _vp, _vp, _vp, _vp, _i, _i, _vp, ctypes.c_size_t,
                                    _vp]
lib.gdn_forward_chunked_noalloc.restype = _st
lib.gdn_forward_chunked_noalloc.argtypes = [ctypes.POINTER(gdn_varlen_shape), _vp, _vp, _vp,
                                            _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _vp]
lib.gdn_forward_chunked_checkpointed.restype = _st
lib.gdn_forward_chunked_checkpointed.argtypes = [
    ctypes.POINTER(gdn_varlen_shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i,
    _vp, _i, _i, _vp, ctypes.c_size_t, _vp]
lib.gdn_checkpoint_select.restype = _st
lib.gdn_checkpoint_select.argtypes = [_i, _i, _i, _i, _i, ctypes.POINTER(_i),
                                      ctypes.POINTER(_i), ctypes.POINTER(_i)]
lib.gdn_noalloc_scratch_bytes.restype = ctypes.c_size_t
lib.gdn_noalloc_scratch_bytes.argtypes = []
lib.gdn_seq_table_create.restype = _st
lib.gdn_seq_table_create.argtypes = [_i, _i, ctypes.POINTER(_vp)]
lib.gdn_seq_table_destroy.restype = None
lib.gdn_seq_table_destroy.argtypes = [_vp]
lib.gdn_seq_table_record.restype = _st
lib.gdn_seq_table_record.argtypes = [_vp, _i, _i]
lib.gdn_seq_table_clear.restype = _st
lib.gdn_seq_table_clear.argtypes = [_vp, _i]
lib.gdn_rollback.restype = _st
lib.gdn_rollback.argtypes = [_vp, _i, _i, ctypes.POINTER(_i)]
lib.gdn_slot_state_ptr.restype = _st
lib.gdn_slot_state_ptr.argtypes = [_vp, _i, _i, _i, _i, _i, _i, ctypes.POINTER(_vp)]
lib.gdn_check_device_error.restype = _st
lib.gdn_check_device_error.argtypes = [_vp]
lib.gdn_decode_device_error.restype = _st
lib.gdn_decode_device_error.argtypes = [_i]
lib.gdn_device_error_word.restype = _st
lib.gdn_device_error_word.argtypes = [ctypes.POINTER(_vp)]


def _addr(x):
    """Device address of a tensor argument (or a raw integer address). The C
    ABI takes packed row-major buffers, so a strided view is refused here
    rather than read as if it were packed."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("gdn: tensor arguments must be contiguous (packed row-major)")
    return x.data_ptr()


def _check(status):
    if status != GDN_OK:
        raise GDNError(status, lib.gdn_last_error().decode(errors="replace"))


def _stream(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream  # torch.cuda.Stream


def gdn_version() -> str:
    return lib.gdn_version().decode()


def gdn_last_error() -> str:
    return lib.gdn_last_error().decode(errors="replace")


def gdn_forward(shape: gdn_shape, q, k, v, g, beta, state_in, state_slots, out,
                n_slots: int, mode, stream=None) -> None:
    """state_in: device array of n_seqs state pointers (e.g. an int64 tensor
    built with state_ptr_array)."""
    _check(lib.gdn_forward(ctypes.byref(shape), _addr(q), _addr(k), _addr(v), _addr(g),
                           _addr(beta), _addr(state_in), _addr(state_slots), _addr(out),
                           int(n_slots), _MODES[mode], _stream(stream)))


def gdn_forward_host(shape: gdn_shape, q, k, v, g, beta, state_in, state_slots, out,
                     n_slots: int, mode, stream=None) -> None:
    """gdn_forward whose q, k, v, g, beta and out may be pinned host tensors
    (or device tensors): the kernel reads and writes them over the host link."""
    _check(lib.gdn_forward_host(ctypes.byref(shape), _addr(q), _addr(k), _addr(v), _addr(g),
                                _addr(beta), _addr(state_in), _addr(state_slots), _addr(out),
                                int(n_slots), _MODES[mode], _stream(stream)))


def gdn_chunked_workspace_size(shape: gdn_varlen_shape, n_slots: int) -> int:
    return int(lib.gdn_chunked_workspace_size(ctypes.byref(shape), int(n_slots)))


def gdn_forward_chunked(shape: gdn_varlen_shape, cu_seqlens, q, k, v, g, beta, state_in,
                        state_slots, out, n_slots: int, mode, workspace,
                        workspace_bytes: int, stream=None) -> None:
    _check(lib.gdn_forward_chunked(ctypes.byref(shape), _addr(cu_seqlens), _addr(q),
                                   _addr(k), _addr(v), _addr(g), _addr(beta),
                                   _addr(state_in), _addr(state_slots), _addr(out),
                                   int(n_slots), _MODES[mode], _addr(workspace),
                                   int(workspace_bytes), _stream(stream)))


def gdn_forward_chunked_noalloc(shape: gdn_varlen_shape, cu_seqlens, q, k, v, g, beta,
                                state_in, state_slots, out, n_slots: int, mode,
                                stream=None) -> None:
    """gdn_forward_chunked without a workspace: the library's built-in
    scratch array is used (for callers that cannot allocate device memory)."""
    _check(lib.gdn_forward_chunked_noalloc(ctypes.byref(shape), _addr(cu_seqlens), _addr(q),
                                           _addr(k), _addr(v), _addr(g), _addr(beta),
                                           _addr(state_in), _addr(state_slots), _addr(out),
                                           int(n_slots), _MODES[mode], _stream(stream)))


def gdn_forward_chunked_checkpointed(shape: gdn_varlen_shape, cu_seqlens, q, k, v, g, beta,
                                     state_in, state_slots, out, n_slots: int, mode,
                                     checkpoints, ckpt_every: int, max_ckpts: int,
                                     workspace, workspace_bytes: int, stream=None) -> None:
    """gdn_forward_chunked that also stores checkpoints[s][m], the state
    after (m+1)*ckpt_every tokens of sequence s (fp32 [N][max_ckpts][H][D_k][D_v])."""
    _check(lib.gdn_forward_chunked_checkpointed(
        ctypes.byref(shape), _addr(cu_seqlens), _addr(q), _addr(k), _addr(v), _addr(g),
        _addr(beta), _addr(state_in), _addr(state_slots), _addr(out), int(n_slots),
        _MODES[mode], _addr(checkpoints), int(ckpt_every), int(max_ckpts), _addr(workspace),
        int(workspace_bytes), _stream(stream)))


CKPT_SOURCES = ("state_in", "checkpoint", "slot")


def gdn_checkpoint_select(n_keep: int, L: int, n_slots: int, ckpt_every: int,
                          max_ckpts: int):
    """(source, index, replay_from) for keeping the first n_keep of L tokens;
    source is one of CKPT_SOURCES."""
    src, idx, rep = _i(), _i(), _i()
    _check(lib.gdn_checkpoint_select(int(n_keep), int(L), int(n_slots), int(ckpt_every),
                                     int(max_ckpts), ctypes.byref(src), ctypes.byref(idx),
                                     ctypes.byref(rep)))
    return CKPT_SOURCES[src.value], idx.value, rep.value


def gdn_noalloc_scratch_bytes() -> int:
    return int(lib.gdn_noalloc_scratch_bytes())


def gdn_check_device_error(stream=None) -> None:
    _check(lib.gdn_check_device_error(_stream(stream)))


def gdn_decode_device_error(word: int):
    """(status, message) the library gives for a device error-word value."""
    st = int(lib.gdn_decode_device_error(int(word)))
    return st, (lib.gdn_last_error().decode(errors="replace") if st != GDN_OK else "")


def gdn_device_error_word() -> int:
    """Device address of the current device's error word."""
    out = _vp()
    _check(lib.gdn_device_error_word(ctypes.byref(out)))
    return out.value or 0


class SeqTable:
    """Owner of a gdn_seq_table (host-side rollback bookkeeping)."""

    def __init__(self, n_seqs: int, n_slots: int):
        h = _vp()
        _check(lib.gdn_seq_table_create(int(n_seqs), int(n_slots), ctypes.byref(h)))
        self._h = h
        self.n_seqs, self.n_slots = n_seqs, n_slots

    def record(self, seq: int, T_last: int) -> None:
        _check(lib.gdn_seq_table_record(self._h, int(seq), int(T_last)))

    def clear(self, seq: int) -> None:
        _check(lib.gdn_seq_table_clear(self._h, int(seq)))

    def rollback(self, seq: int, n_accepted: int) -> int:
        """gdn_rollback: slot index, or -1 for "input state unchanged"."""
        slot = _i(-2)
        _check(lib.gdn_rollback(self._h, int(seq), int(n_accepted), ctypes.byref(slot)))
        return slot.value

    def close(self):
        if self._h:
            lib.gdn_seq_table_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def gdn_slot_state_ptr(state_slots, seq: int, slot: int, n_slots: int, H: int, D_k: int,
                       D_v: int) -> int:
    out = _vp()
    _check(lib.gdn_slot_state_ptr(_addr(state_slots), int(seq), int(slot), int(n_slots),
                                  int(H), int(D_k), int(D_v), ctypes.byref(out)))
    return out.value or 0


def state_ptr_array(ptrs, device):
    """Device int64 tensor holding the given state addresses (0 = zero state)."""
    import torch
    return torch.tensor([int(p) if p else 0 for p in ptrs], dtype=torch.int64, device=device)


def per_seq_state_ptrs(state, n_seqs: int):
    """Addresses of state[s] for a contiguous [N, H, D_k, D_v] fp32 tensor."""
    per = state[0].numel() * state.element_size()
    base = state.data_ptr()
    return [base + s * per for s in range(n_seqs)]


def dtype_code(torch_dtype) -> int:
    import torch
    if torch_dtype == torch.bfloat16:
        return GDN_BF16
    if torch_dtype == torch.float32:
        return GDN_F32
    raise ValueError(f"unsupported input dtype {torch_dtype}")
