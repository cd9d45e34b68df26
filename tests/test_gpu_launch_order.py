"""Stream order under programmatic dependent launch, on the GPU.

gdn_forward's kernel may be scheduled while the previous kernel of the
stream still runs; it must read and write nothing before that kernel has
completed. These tests enqueue chains of dependent calls with no host
synchronisation in between and require bit-identical results to the same
chains with a device synchronisation after every call:
- decode steps whose state_in is the previous step's slot buffer (ping-pong),
  all writing the same `out`;
- a chunked prefill whose slots feed decode steps directly.
"""
import pytest
import torch

from gated_delta_net_02_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_net_02_gb300 import build
    build.build()
    from gated_delta_net_02_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


def decode_chain(gdn, toks, state0, steps, sync, stream):
    N, H, D = state0.shape[0], state0.shape[1], state0.shape[2]
    bank = [state0.clone(), torch.empty_like(state0)]
    ptrs = [gdn.state_ptr_array(gdn.per_seq_state_ptrs(b, N), "cuda") for b in bank]
    out = torch.full((N, H, D), float("nan"), device="cuda")
    shape = gdn.gdn_shape(N, 1, H, D, D, gdn.GDN_BF16, D ** -0.5)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(steps):
            q, k, v, g, beta = (t[i % len(t)] for t in toks)
            gdn.gdn_forward(shape, q, k, v, g, beta, ptrs[i % 2], bank[(i + 1) % 2], out, 1,
                            "gda", stream)
            if sync:
                torch.cuda.synchronize()
    torch.cuda.synchronize()
    gdn.gdn_check_device_error(stream)
    return out, bank[steps % 2]


def test_back_to_back_dependent_decode_steps(gdn):
    N, H, D, steps = 64, 16, 128, 16
    state0 = inputs.decode_state(5, N, H, D).cuda()
    pool = [inputs.decode_tokens(5, s, N, H, D) for s in range(4)]
    toks = [torch.stack([p[j] for p in pool]).cuda() for j in range(5)]
    stream = torch.cuda.Stream()
    out_a, st_a = decode_chain(gdn, toks, state0, steps, False, stream)
    out_b, st_b = decode_chain(gdn, toks, state0, steps, True, stream)
    assert not torch.isnan(out_a).any()
    assert torch.equal(out_a, out_b)
    assert torch.equal(st_a, st_b)


def test_decode_right_after_chunked_prefill(gdn):
    # prefill writes K slots; decode steps start from the last slot at once
    N, H, D, K = 4, 16, 128, 2
    b = inputs.make_batch(6, [300, 64, 129, 200], H, D, D, mode="gda", n_slots=K)
    d = {n: getattr(b, n).cuda().contiguous() for n in ("q", "k", "v", "g", "beta", "state")}
    cu = b.cu_seqlens.to(torch.int32).cuda()
    vshape = gdn.gdn_varlen_shape(N, b.q.shape[0], H, D, D, gdn.GDN_BF16, b.scale)
    ws_bytes = gdn.gdn_chunked_workspace_size(vshape, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    pool = [inputs.decode_tokens(7, s, N, H, D) for s in range(3)]
    toks = [[t.cuda() for t in p] for p in pool]
    dshape = gdn.gdn_shape(N, 1, H, D, D, gdn.GDN_BF16, D ** -0.5)
    stream = torch.cuda.Stream()

    def run(sync):
        slots = torch.full((N, K, H, D, D), float("nan"), device="cuda")
        pre_out = torch.full((b.q.shape[0], H, D), float("nan"), device="cuda")
        bank = [torch.empty(N, H, D, D, device="cuda") for _ in range(2)]
        out = torch.empty(N, H, D, device="cuda")
        in_ptrs = gdn.state_ptr_array(gdn.per_seq_state_ptrs(d["state"], N), "cuda")
        last = gdn.state_ptr_array([gdn.gdn_slot_state_ptr(slots, s, K - 1, K, H, D, D)
                                    for s in range(N)], "cuda")
        bptrs = [gdn.state_ptr_array(gdn.per_seq_state_ptrs(x, N), "cuda") for x in bank]
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            gdn.gdn_forward_chunked(vshape, cu, d["q"], d["k"], d["v"], d["g"], d["beta"],
                                    in_ptrs, slots, pre_out, K, "gda", ws, ws_bytes, stream)
            if sync:
                torch.cuda.synchronize()
            for i, (q, k, v, g, beta) in enumerate(toks):
                src = last if i == 0 else bptrs[(i + 1) % 2]
                gdn.gdn_forward(dshape, q, k, v, g, beta, src, bank[i % 2], out, 1, "gda",
                                stream)
                if sync:
                    torch.cuda.synchronize()
        torch.cuda.synchronize()
        gdn.gdn_check_device_error(stream)
        return pre_out, slots, out, bank[(len(toks) - 1) % 2]

    a = run(False)
    b_ = run(True)
    for x, y in zip(a, b_):
        assert torch.equal(x.nan_to_num(3.0), y.nan_to_num(3.0))
    assert not torch.isnan(a[2]).any()
