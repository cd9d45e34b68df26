"""GPU tests of gdn_forward_host: the uniform-length forward whose q, k, v,
g, beta and out sit in page-locked host memory (read and written by the
kernel over the host link). Its results must equal gdn_forward's bit for bit
(same configuration and arithmetic), whatever mix of host and device buffers
is passed, over one and several token tiles; and the oracle bounds hold."""
import numpy as np
import pytest
import torch

from gated_delta_net_02_gb300 import inputs

from _helpers import TOL, gpu_forward, oracle_run, rel_l2, to_dev

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "g", "beta")


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_net_02_gb300 import build
    build.build()
    from gated_delta_net_02_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


def host_forward(gdn, b, on_host, stream=None):
    """gdn_forward_host with the tensors named in on_host (and "out") pinned
    on the host, the others on the device; returns (out, slots) on the device."""
    N, T = b.n_seqs, int(b.seq_len[0])
    H, Dk, Dv = b.v.shape[1], b.q.shape[2], b.v.shape[2]
    d = to_dev(b)
    args = {n: (getattr(b, n).contiguous().pin_memory() if n in on_host else d[n])
            for n in NAMES}
    for n in on_host:
        if n != "out":
            assert args[n].is_pinned() and not args[n].is_cuda
    slots = torch.full((N, b.n_slots, H, Dk, Dv), float("nan"), device="cuda")
    if "out" in on_host:
        out = torch.full((N * T, H, Dv), float("nan")).pin_memory()
    else:
        out = torch.full((N * T, H, Dv), float("nan"), device="cuda")
    ptrs = gdn.state_ptr_array(gdn.per_seq_state_ptrs(d["state"], N), "cuda")
    shape = gdn.gdn_shape(N, T, H, Dk, Dv, gdn.dtype_code(b.q.dtype), b.scale,
                          b.q.shape[1], gdn.QK_MAPS[b.qk_map])
    gdn.gdn_forward_host(shape, args["q"], args["k"], args["v"], args["g"], args["beta"],
                         ptrs, slots, out, b.n_slots, b.mode, stream)
    gdn.gdn_check_device_error(stream)
    torch.cuda.synchronize()
    return out.cuda(), slots


ALL_HOST = NAMES + ("out",)


@pytest.mark.parametrize("T", [1, 8, 37])
@pytest.mark.parametrize("mode", ["gda", "kda"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_host_buffers_equal_device_call(gdn, T, mode, dtype):
    """decode (T=1), verify (T=8: one full tile) and T=37 (five tiles, the
    last one ragged: the next tile's loads are in flight over the token loop)."""
    b = inputs.make_batch(40 + T, [T] * 5, 4, 128, 128, dtype=dtype, mode=mode,
                          n_slots=min(T, 4))
    out_d, slots_d = gpu_forward(b)
    out_h, slots_h = host_forward(gdn, b, ALL_HOST)
    assert torch.equal(out_h, out_d)
    assert torch.equal(slots_h.nan_to_num(7.0), slots_d.nan_to_num(7.0))


@pytest.mark.parametrize("Dk,Dv", [(64, 64), (64, 128), (128, 64)])
def test_host_buffers_other_head_sizes(gdn, Dk, Dv):
    b = inputs.make_batch(7 + Dk + Dv, [11] * 3, 3, Dk, Dv, dtype=torch.bfloat16,
                          mode="kda", n_slots=3)
    out_d, slots_d = gpu_forward(b)
    out_h, slots_h = host_forward(gdn, b, ALL_HOST)
    assert torch.equal(out_h, out_d)
    assert torch.equal(slots_h.nan_to_num(7.0), slots_d.nan_to_num(7.0))


@pytest.mark.parametrize("on_host", [("v", "g", "beta", "out"), ("q", "k"), ()])
def test_mixed_host_and_device_buffers(gdn, on_host):
    b = inputs.make_batch(77, [9] * 4, 4, 128, 128, dtype=torch.bfloat16, mode="gda",
                          n_slots=2)
    out_d, slots_d = gpu_forward(b)
    out_h, slots_h = host_forward(gdn, b, on_host)
    assert torch.equal(out_h, out_d)
    assert torch.equal(slots_h.nan_to_num(7.0), slots_d.nan_to_num(7.0))


def test_grouped_query_heads_from_host(gdn):
    b = inputs.make_batch(91, [8] * 3, 8, 128, 128, dtype=torch.bfloat16, mode="gda",
                          n_slots=2, H_qk=2, qk_map="grouped")
    out_d, slots_d = gpu_forward(b)
    out_h, slots_h = host_forward(gdn, b, ALL_HOST)
    assert torch.equal(out_h, out_d)
    assert torch.equal(slots_h.nan_to_num(7.0), slots_d.nan_to_num(7.0))


def test_decode_workload_from_host_against_oracle(gdn):
    """The batched decode shape (64 sequences x 1 token, H=16, D=128, bf16,
    GDA, state ~N(0, 0.05)) with every token buffer and the output on the
    host, against the fp64 oracle."""
    N, H, D = 64, 16, 128
    q, k, v, g, beta = inputs.decode_tokens(1, 3, N, H, D)
    state = inputs.decode_state(1, N, H, D)
    b = inputs.GDNBatch(q, k, v, g, beta, state, "gda", D ** -0.5,
                        torch.ones(N, dtype=torch.int64), 1)
    out_h, slots_h = host_forward(gdn, b, ALL_HOST)
    o_ref, s_ref, _ = oracle_run(b)
    assert rel_l2(out_h.double().cpu().numpy(), o_ref) <= TOL[torch.bfloat16]
    assert rel_l2(slots_h[:, 0].double().cpu().numpy(), s_ref) < 1e-5


def test_pageable_host_memory_is_refused(gdn):
    """An ordinary (pageable) host tensor is refused before anything is
    enqueued, and the outputs stay untouched."""
    b = inputs.make_batch(5, [2] * 2, 2, 128, 128, dtype=torch.bfloat16, n_slots=1)
    d = to_dev(b)
    pageable_v = b.v.contiguous()
    assert not pageable_v.is_pinned()
    slots = torch.full((2, 1, 2, 128, 128), float("nan"), device="cuda")
    out = torch.full((4, 2, 128), float("nan"), device="cuda")
    ptrs = gdn.state_ptr_array(gdn.per_seq_state_ptrs(d["state"], 2), "cuda")
    shape = gdn.gdn_shape(2, 2, 2, 128, 128, gdn.GDN_BF16, 0.0)
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_forward_host(shape, d["q"], d["k"], pageable_v, d["g"], d["beta"], ptrs,
                             slots, out, 1, "gda")
    assert e.value.status == gdn.GDN_ERR_INVALID_ARG
    assert "gdn_forward_host: v" in str(e.value)
    torch.cuda.synchronize()
    assert torch.isnan(out).all() and torch.isnan(slots).all()
    gdn.gdn_check_device_error()


def test_host_calls_in_a_cuda_graph(gdn):
    """Consecutive decode steps captured in one graph, each reading its own
    pinned host tokens and writing its own pinned host output, each step's
    state feeding the next: equal to the same chain through gdn_forward."""
    N, H, D, STEPS = 16, 4, 128, 6
    state0 = inputs.decode_state(2, N, H, D)
    toks = [inputs.decode_tokens(2, s, N, H, D) for s in range(STEPS)]
    host_toks = [[t.contiguous().pin_memory() for t in tk] for tk in toks]
    dev_toks = [[t.cuda() for t in tk] for tk in toks]
    shape = gdn.gdn_shape(N, 1, H, D, D, gdn.GDN_BF16, 0.0)

    def chain(use_host, outs, stream):
        bank = [state0.cuda(), torch.empty(N, H, D, D, device="cuda")]
        ptrs = [gdn.state_ptr_array(gdn.per_seq_state_ptrs(x, N), "cuda") for x in bank]
        torch.cuda.synchronize()
        fn = gdn.gdn_forward_host if use_host else gdn.gdn_forward
        src = host_toks if use_host else dev_toks

        def run():
            for s in range(STEPS):
                q, k, v, g, beta = src[s]
                fn(shape, q, k, v, g, beta, ptrs[s % 2], bank[(s + 1) % 2], outs[s], 1,
                   "gda", stream)
        return bank, run

    stream = torch.cuda.Stream()
    outs_h = [torch.empty(N, H, D).pin_memory() for _ in range(STEPS)]
    bank_h, run_h = chain(True, outs_h, stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            run_h()
    graph.replay()
    torch.cuda.synchronize()
    outs_d = [torch.empty(N, H, D, device="cuda") for _ in range(STEPS)]
    bank_d, run_d = chain(False, outs_d, stream)
    with torch.cuda.stream(stream):
        run_d()
    torch.cuda.synchronize()
    gdn.gdn_check_device_error()
    for s in range(STEPS):
        assert torch.equal(outs_h[s].cuda(), outs_d[s]), s
    assert torch.equal(bank_h[STEPS % 2], bank_d[STEPS % 2])


@pytest.mark.parametrize("T", [1, 12])
def test_host_call_refuses_state_in_inside_slots(gdn, T):
    """A state pointer into the slot buffer is refused by the device for that
    sequence (GDN_ERR_DEVICE_ARG); the other sequence still runs and matches
    the device-buffer call, and the error word clears."""
    b = inputs.make_batch(15 + T, [T] * 2, 2, 128, 128, n_slots=2)
    N, H = 2, 2
    slots_h = torch.full((N, 2, H, 128, 128), float("nan"), device="cuda")
    slots_d = slots_h.clone()
    d = to_dev(b)
    shape = gdn.gdn_shape(N, T, H, 128, 128, gdn.GDN_BF16, 0.0)
    h = {n: getattr(b, n).contiguous().pin_memory() for n in NAMES}
    out_h = torch.full((N * T, H, 128), float("nan")).pin_memory()
    out_d = torch.full((N * T, H, 128), float("nan"), device="cuda")
    ptrs_h = gdn.state_ptr_array([slots_h[1, 0].data_ptr(), d["state"][1].data_ptr()], "cuda")
    ptrs_d = gdn.state_ptr_array([slots_d[1, 0].data_ptr(), d["state"][1].data_ptr()], "cuda")
    gdn.gdn_forward_host(shape, h["q"], h["k"], h["v"], h["g"], h["beta"], ptrs_h, slots_h,
                         out_h, 2, "gda")
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_check_device_error()
    assert e.value.status == gdn.GDN_ERR_DEVICE_ARG
    gdn.gdn_forward(shape, d["q"], d["k"], d["v"], d["g"], d["beta"], ptrs_d, slots_d, out_d,
                    2, "gda")
    with pytest.raises(gdn.GDNError):
        gdn.gdn_check_device_error()
    gdn.gdn_check_device_error()  # cleared
    torch.cuda.synchronize()
    assert torch.equal(out_h.cuda()[T:], out_d[T:])          # sequence 1 ran
    assert torch.equal(slots_h[1].nan_to_num(7.0), slots_d[1].nan_to_num(7.0))
    assert torch.isnan(out_h[:T]).all()                        # sequence 0 did not
