"""gdn_forward_chunked_noalloc: the chunked prefill for callers that cannot
allocate device memory (for example a host program that hands out every
device byte from its own pool, or a loop that must never pay for a
cudaMalloc, which can synchronise the whole device). Instead of a caller
workspace it uses a fixed scratch array built into the library.

These tests run it through the C ABI twice in a row and check each result
against gdn_forward_chunked with a caller workspace, within the bf16
tolerance the other chunked tests use, and check that a shape too large for
the built-in array is refused with a clear error. The file is named so that
pytest collects it last."""
import pytest
import torch

from gated_delta_net_02_gb300 import inputs

from _helpers import rel_l2, to_dev

pytestmark = pytest.mark.gpu

TOL_BF16 = 5e-3


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_net_02_gb300 import build
    build.build()
    from gated_delta_net_02_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


def _run(gdn, b, noalloc):
    d = to_dev(b)
    N, ntok = b.n_seqs, b.q.shape[0]
    H = b.q.shape[1]
    cu = b.cu_seqlens.to(torch.int32).cuda()
    shape = gdn.gdn_varlen_shape(N, ntok, H, 128, 128, gdn.GDN_BF16, b.scale)
    slots = torch.full((N, b.n_slots, H, 128, 128), float("nan"), device="cuda")
    out = torch.full((ntok, H, 128), float("nan"), device="cuda")
    ptrs = gdn.state_ptr_array(gdn.per_seq_state_ptrs(d["state"], N), "cuda")
    if noalloc:
        gdn.gdn_forward_chunked_noalloc(shape, cu, d["q"], d["k"], d["v"], d["g"], d["beta"],
                                        ptrs, slots, out, b.n_slots, b.mode)
    else:
        ws_bytes = gdn.gdn_chunked_workspace_size(shape, b.n_slots)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        gdn.gdn_forward_chunked(shape, cu, d["q"], d["k"], d["v"], d["g"], d["beta"], ptrs,
                                slots, out, b.n_slots, b.mode, ws, ws_bytes)
    gdn.gdn_check_device_error()
    return out, slots


def _close(a, b):
    a = a.double().cpu().nan_to_num(0.0).numpy()
    b = b.double().cpu().nan_to_num(0.0).numpy()
    return rel_l2(a, b)


def test_noalloc_matches_workspace_path_on_two_calls_in_a_row(gdn):
    first = inputs.make_batch(77, [300, 70, 5], 2, 128, 128, mode="kda", n_slots=4)
    second = inputs.make_batch(78, [129, 400], 3, 128, 128, mode="gda", n_slots=2)
    ref1 = _run(gdn, first, noalloc=False)
    ref2 = _run(gdn, second, noalloc=False)
    got1 = _run(gdn, first, noalloc=True)    # first call on this device: sets up
    got2 = _run(gdn, second, noalloc=True)   # second call reuses the array as left
    for got, ref in ((got1, ref1), (got2, ref2)):
        assert not torch.isnan(got[0]).any()
        assert _close(got[0], ref[0]) <= TOL_BF16
        assert _close(got[1], ref[1]) <= TOL_BF16
        # the same slots are written (NaN marks the untouched ones)
        assert torch.equal(torch.isnan(got[1]), torch.isnan(ref[1]))


def test_noalloc_refuses_shapes_beyond_its_scratch(gdn):
    cap = gdn.gdn_noalloc_scratch_bytes()
    big = gdn.gdn_varlen_shape(8, 40000, 16, 128, 128, gdn.GDN_BF16, 0.0)
    assert gdn.gdn_chunked_workspace_size(big, 8) > cap
    fake = 1 << 20  # aligned, never dereferenced: the size check comes first
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_forward_chunked_noalloc(big, fake, fake, fake, fake, fake, fake, fake, fake,
                                        fake, 8, "gda")
    assert e.value.status == gdn.GDN_ERR_UNSUPPORTED
    assert str(cap) in str(e.value)
