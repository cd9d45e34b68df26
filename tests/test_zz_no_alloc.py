"""gdn_forward_chunked_noalloc: the chunked prefill for callers that cannot
allocate device memory (for example a host program that hands out every
device byte from its own pool, or a loop that must never pay for a
cudaMalloc, which can synchronise the whole device). Instead of a caller
workspace it uses a fixed scratch array built into the library.

These tests run it through the C ABI twice in a row and require each result
to equal gdn_forward_chunked with a caller workspace bit for bit (both run the
same kernels on the same workspace layout, so the scratch array left over by
the previous call must change nothing), and to match the fp64 oracle within
the tolerance of the input dtype: the tensor-core route (bf16, 5e-3) and the
token-loop route (fp32, 1e-5). A shape too large for the built-in array is
refused with a clear error. The file is named so that pytest collects it
last."""
import pytest
import torch

from gated_delta_net_02_gb300 import inputs

from _helpers import oracle_run, rel_l2, to_dev

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 5e-3, torch.float32: 1e-5}
SENTINEL = -12345.0   # stands for NaN (an unwritten slot) in exact comparisons


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
    H, D = b.v.shape[1], b.v.shape[2]
    cu = b.cu_seqlens.to(torch.int32).cuda()
    shape = gdn.gdn_varlen_shape(N, ntok, H, D, D, gdn.dtype_code(b.q.dtype), b.scale)
    slots = torch.full((N, b.n_slots, H, D, D), float("nan"), device="cuda")
    out = torch.full((ntok, H, D), float("nan"), device="cuda")
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


def _same(a, b):
    return torch.equal(a.nan_to_num(SENTINEL), b.nan_to_num(SENTINEL))


def _check_oracle(b, out, slots):
    o_ref, s_ref, _ = oracle_run(b)
    tol = TOL[b.q.dtype]
    assert not torch.isnan(out).any()
    assert rel_l2(out.double().cpu().numpy(), o_ref) <= tol
    ran = b.seq_len.numpy() > 0
    assert rel_l2(slots[:, -1].double().cpu().numpy()[ran], s_ref[ran]) <= tol


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_workspace_path_on_two_calls_in_a_row(gdn, dtype):
    # bf16 runs the tensor-core kernels, fp32 the token-loop route; both use
    # the built-in array for their work list
    first = inputs.make_batch(77, [300, 70, 5], 2, 128, 128, dtype=dtype, mode="kda",
                              n_slots=4)
    second = inputs.make_batch(78, [129, 400], 3, 128, 128, dtype=dtype, mode="gda",
                               n_slots=2)
    ref1 = _run(gdn, first, noalloc=False)
    ref2 = _run(gdn, second, noalloc=False)
    got1 = _run(gdn, first, noalloc=True)    # first call on this device: sets up
    got2 = _run(gdn, second, noalloc=True)   # second call reuses the array as left
    for b, got, ref in ((first, got1, ref1), (second, got2, ref2)):
        assert _same(got[0], ref[0])
        assert _same(got[1], ref[1])
        _check_oracle(b, *got)


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
