"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every symbol include/gdn.h declares, validates arguments before touching the
device, and implements the rollback bookkeeping exactly as the oracle's slot
choice defines it."""
import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_net_02_gb300 import build
    build.build()
    from gated_delta_net_02_gb300 import gdn as mod
    return mod


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(gdn):
    names = declared_functions()
    assert "gdn_forward" in names and "gdn_rollback" in names and "gdn_forward_chunked" in names
    for name in names:
        assert hasattr(gdn.lib, name), name
        assert ctypes.cast(getattr(gdn.lib, name), ctypes.c_void_p).value


def test_version(gdn):
    assert "sm_103a" in gdn.gdn_version()


def shape(gdn, **kw):
    base = dict(n_seqs=2, T=3, H=2, D_k=128, D_v=128, in_dtype=gdn.GDN_BF16, scale=0.0)
    base.update(kw)
    return gdn.gdn_shape(**base)


FAKE = 1 << 20  # 16-byte aligned non-null address; never dereferenced here


def call_forward(gdn, sh, n_slots=1, mode="gda", **ptrs):
    p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state_in=FAKE, state_slots=FAKE,
             out=FAKE)
    p.update(ptrs)
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_forward(sh, p["q"], p["k"], p["v"], p["g"], p["beta"], p["state_in"],
                        p["state_slots"], p["out"], n_slots, mode)
    return e.value.status


def test_forward_argument_errors(gdn):
    assert call_forward(gdn, shape(gdn, D_k=32)) == gdn.GDN_ERR_UNSUPPORTED
    assert call_forward(gdn, shape(gdn, D_v=96)) == gdn.GDN_ERR_UNSUPPORTED
    assert call_forward(gdn, shape(gdn), n_slots=0) == gdn.GDN_ERR_INVALID_ARG
    assert call_forward(gdn, shape(gdn, H=0)) == gdn.GDN_ERR_INVALID_ARG
    assert call_forward(gdn, shape(gdn, T=-1)) == gdn.GDN_ERR_INVALID_ARG
    assert call_forward(gdn, shape(gdn, in_dtype=7)) == gdn.GDN_ERR_INVALID_ARG
    assert call_forward(gdn, shape(gdn, scale=float("nan"))) == gdn.GDN_ERR_INVALID_ARG
    assert call_forward(gdn, shape(gdn), q=0) == gdn.GDN_ERR_INVALID_ARG
    assert call_forward(gdn, shape(gdn), beta=FAKE + 4) == gdn.GDN_ERR_INVALID_ARG
    assert call_forward(gdn, shape(gdn), state_in=0) == gdn.GDN_ERR_INVALID_ARG
    rc = gdn.lib.gdn_forward(ctypes.byref(shape(gdn)), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                             FAKE, FAKE, 1, 9, None)
    assert rc == gdn.GDN_ERR_INVALID_ARG
    assert "mode" in gdn.gdn_last_error()


def test_forward_host_argument_errors(gdn):
    """gdn_forward_host makes gdn_forward's checks (under its own name), then
    refuses a pointer CUDA does not know as device or page-locked host memory
    before anything is enqueued (here: an address nothing allocated)."""
    def call(sh, n_slots=1, **ptrs):
        p = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state_in=FAKE, state_slots=FAKE,
                 out=FAKE)
        p.update(ptrs)
        with pytest.raises(gdn.GDNError) as e:
            gdn.gdn_forward_host(sh, p["q"], p["k"], p["v"], p["g"], p["beta"], p["state_in"],
                                 p["state_slots"], p["out"], n_slots, "gda")
        return e.value.status, gdn.gdn_last_error()

    assert call(shape(gdn, D_k=32))[0] == gdn.GDN_ERR_UNSUPPORTED
    st, msg = call(shape(gdn), n_slots=0)
    assert st == gdn.GDN_ERR_INVALID_ARG and msg.startswith("gdn_forward_host: n_slots")
    st, msg = call(shape(gdn), beta=FAKE + 4)
    assert st == gdn.GDN_ERR_INVALID_ARG and "beta is not 16-byte aligned" in msg
    st, msg = call(shape(gdn))
    assert st == gdn.GDN_ERR_INVALID_ARG
    assert msg == ("gdn_forward_host: q is neither device memory nor page-locked host "
                   "memory mapped at the same address")
    assert gdn.lib.gdn_forward_host(None, 0, 0, 0, 0, 0, 0, 0, 0, 1, 0, None) == \
        gdn.GDN_ERR_INVALID_ARG
    gdn.gdn_forward_host(shape(gdn, n_seqs=0), 0, 0, 0, 0, 0, 0, 0, 0, 1, "gda")


def test_null_shape(gdn):
    assert gdn.lib.gdn_forward(None, 0, 0, 0, 0, 0, 0, 0, 0, 1, 0, None) == gdn.GDN_ERR_INVALID_ARG


def test_empty_batch_is_a_no_op(gdn):
    # no sequences: nothing to validate or launch, no device needed
    gdn.gdn_forward(shape(gdn, n_seqs=0), 0, 0, 0, 0, 0, 0, 0, 0, 1, "gda")


def vshape(gdn, **kw):
    base = dict(n_seqs=2, total_tokens=100, H=2, D_k=128, D_v=128, in_dtype=gdn.GDN_BF16,
                scale=0.0)
    base.update(kw)
    return gdn.gdn_varlen_shape(**base)


def call_chunked(gdn, sh, n_slots=1, ws_bytes=None, **ptrs):
    p = dict(cu=FAKE, q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state_in=FAKE,
             state_slots=FAKE, out=FAKE, ws=FAKE)
    p.update(ptrs)
    if ws_bytes is None:
        ws_bytes = gdn.gdn_chunked_workspace_size(sh, n_slots)
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_forward_chunked(sh, p["cu"], p["q"], p["k"], p["v"], p["g"], p["beta"],
                                p["state_in"], p["state_slots"], p["out"], n_slots, "gda",
                                p["ws"], ws_bytes)
    return e.value.status


def test_chunked_argument_errors(gdn):
    assert call_chunked(gdn, vshape(gdn, D_k=32)) == gdn.GDN_ERR_UNSUPPORTED
    assert call_chunked(gdn, vshape(gdn, D_v=96)) == gdn.GDN_ERR_UNSUPPORTED
    assert call_chunked(gdn, vshape(gdn, in_dtype=7)) == gdn.GDN_ERR_INVALID_ARG
    assert call_chunked(gdn, vshape(gdn, n_seqs=0)) == gdn.GDN_ERR_INVALID_ARG
    assert call_chunked(gdn, vshape(gdn), n_slots=0, ws_bytes=1 << 30) == gdn.GDN_ERR_INVALID_ARG
    assert call_chunked(gdn, vshape(gdn), cu=0) == gdn.GDN_ERR_INVALID_ARG
    assert call_chunked(gdn, vshape(gdn), ws=FAKE + 16) == gdn.GDN_ERR_INVALID_ARG
    assert call_chunked(gdn, vshape(gdn), ws_bytes=1) == gdn.GDN_ERR_INVALID_ARG
    assert call_chunked(gdn, vshape(gdn), out=FAKE + 8) == gdn.GDN_ERR_INVALID_ARG


def test_workspace_size_grows_with_tokens(gdn):
    a = gdn.gdn_chunked_workspace_size(vshape(gdn, total_tokens=1000), 8)
    b = gdn.gdn_chunked_workspace_size(vshape(gdn, total_tokens=100000), 8)
    assert 0 < a <= b
    assert gdn.gdn_chunked_workspace_size(vshape(gdn), 0) == 0


@pytest.mark.parametrize("T,K", [(8, 8), (8, 3), (1, 1), (5, 1), (3, 6), (0, 2)])
def test_rollback_matches_oracle_slot_choice(gdn, T, K):
    t = gdn.SeqTable(3, K)
    t.record(1, T)
    for n in range(-2, T + 3):
        try:
            want = oracle.rollback_slot(T, K, n)
        except oracle.RollbackRangeError:
            want = None
        if want is None:
            with pytest.raises(gdn.GDNError) as e:
                t.rollback(1, n)
            assert e.value.status == gdn.GDN_ERR_ROLLBACK_RANGE
        else:
            assert t.rollback(1, n) == want
    t.close()


def test_seq_table_record_clear_and_bounds(gdn):
    t = gdn.SeqTable(2, 4)
    assert t.rollback(0, 0) == -1          # never ran: only "keep the input"
    with pytest.raises(gdn.GDNError):
        t.rollback(0, 1)
    t.record(0, 4)
    assert t.rollback(0, 4) == 3 and t.rollback(0, 1) == 0
    t.clear(0)                              # a cleared sequence has no slots
    with pytest.raises(gdn.GDNError) as e:
        t.rollback(0, 1)
    assert e.value.status == gdn.GDN_ERR_ROLLBACK_RANGE
    for bad in [(-1, 0), (2, 0)]:
        with pytest.raises(gdn.GDNError) as e:
            t.rollback(*bad)
        assert e.value.status == gdn.GDN_ERR_INVALID_ARG
    with pytest.raises(gdn.GDNError):
        t.record(0, -1)
    with pytest.raises(gdn.GDNError):
        gdn.SeqTable(1, 0)


def test_slot_state_ptr_arithmetic(gdn):
    base = 1 << 30
    H, Dk, Dv, K = 3, 64, 128, 5
    p = gdn.gdn_slot_state_ptr(base, 2, 4, K, H, Dk, Dv)
    assert p == base + ((2 * K + 4) * H * Dk * Dv) * 4
    assert gdn.gdn_slot_state_ptr(base, 2, -1, K, H, Dk, Dv) == 0
    with pytest.raises(gdn.GDNError):
        gdn.gdn_slot_state_ptr(base, 0, K, K, H, Dk, Dv)


def test_grouped_query_heads_are_validated_on_the_host(gdn):
    # H_qk must divide H (0 means H); qk_map is tiled (0) or grouped (1)
    assert call_forward(gdn, shape(gdn, H=4, H_qk=3)) == gdn.GDN_ERR_INVALID_ARG
    assert "H_qk" in gdn.gdn_last_error()
    assert call_forward(gdn, shape(gdn, H=4, H_qk=8)) == gdn.GDN_ERR_INVALID_ARG
    assert call_forward(gdn, shape(gdn, H=4, H_qk=-2)) == gdn.GDN_ERR_INVALID_ARG
    assert call_forward(gdn, shape(gdn, H=4, H_qk=2, qk_map=5)) == gdn.GDN_ERR_INVALID_ARG
    assert "qk_map" in gdn.gdn_last_error()
    assert call_chunked(gdn, vshape(gdn, H=6, H_qk=4)) == gdn.GDN_ERR_INVALID_ARG
    assert call_chunked(gdn, vshape(gdn, H=6, H_qk=3, qk_map=2)) == gdn.GDN_ERR_INVALID_ARG
    # valid grouped-query fields pass validation (the next failure is a NULL input)
    assert call_forward(gdn, shape(gdn, H=4, H_qk=2, qk_map=gdn.GDN_QK_GROUPED), q=0) \
        == gdn.GDN_ERR_INVALID_ARG
    assert "q is NULL" in gdn.gdn_last_error()


def test_binding_refuses_strided_views(gdn):
    # the C ABI has no strides: a transposed view must not reach it
    import torch
    x = torch.zeros(4, 8)
    with pytest.raises(ValueError):
        gdn._addr(x.t())
    assert gdn._addr(x) == x.data_ptr()
    assert gdn._addr(None) is None and gdn._addr(1 << 20) == 1 << 20


def wait_sites():
    src = open(os.path.join(ROOT, "gated_delta_net_02_gb300", "csrc", "common.cuh")).read()
    return {name: int(v) for name, v in re.findall(r"(kSite\w+) = (\d+)", src)}


def test_device_error_word_decoding(gdn):
    """Every value the kernels can put in the error word maps to its status
    and message, with no device access: timeouts name their wait site
    (bits 8..15) and chunk (bits 16..30); each named site has its own name."""
    assert gdn.gdn_decode_device_error(0) == (gdn.GDN_OK, "")
    sites = wait_sites()
    assert len(sites) >= 10 and len(set(sites.values())) == len(sites)
    names = set()
    for site in sites.values():
        st, msg = gdn.gdn_decode_device_error(1 | (site << 8) | (37 << 16))
        assert st == gdn.GDN_ERR_TIMEOUT
        assert f"site {site}: " in msg and "chunk 37" in msg and "unnamed" not in msg
        names.add(msg.split(f"site {site}: ")[1].split(";")[0])
    assert len(names) == len(sites)
    st, msg = gdn.gdn_decode_device_error(1 | (250 << 8))
    assert st == gdn.GDN_ERR_TIMEOUT and "site 250: unnamed wait" in msg
    assert gdn.gdn_decode_device_error(2) == (gdn.GDN_ERR_DEVICE_ARG,
                                              "cu_seqlens is not a valid offset table")
    st, msg = gdn.gdn_decode_device_error(3)
    assert st == gdn.GDN_ERR_DEVICE_ARG and "state_slots" in msg
    st, msg = gdn.gdn_decode_device_error(4)
    assert st == gdn.GDN_ERR_DEVICE_ARG and "e^80" in msg and "gdn_forward" in msg
    st, msg = gdn.gdn_decode_device_error(9)
    assert st == gdn.GDN_ERR_DEVICE_ARG and "device error word 9" in msg
