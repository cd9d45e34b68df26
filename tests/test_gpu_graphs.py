"""Both entry points enqueue work only on the caller's stream and never
synchronise, so a caller can capture them in a CUDA graph (after one eager
call per device, which sets up per-device state). A replay must reproduce
the eager call bit for bit."""
import pytest
import torch

from gated_delta_net_02_gb300 import inputs

from _helpers import gpu_forward, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_net_02_gb300 import build
    build.build()
    from gated_delta_net_02_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


def test_decode_step_in_a_graph(gdn):
    b = inputs.make_batch(250, [1] * 16, 4, 128, 128, n_slots=1)
    d = to_dev(b)
    eager_out, eager_slots = gpu_forward(b, dev_tensors=d)
    out = torch.full_like(eager_out, float("nan"))
    slots = torch.full_like(eager_slots, float("nan"))
    ptrs = gdn.state_ptr_array(gdn.per_seq_state_ptrs(d["state"], 16), "cuda")
    shape = gdn.gdn_shape(16, 1, 4, 128, 128, gdn.GDN_BF16, b.scale)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s), torch.cuda.graph(g, stream=s):
        gdn.gdn_forward(shape, d["q"], d["k"], d["v"], d["g"], d["beta"], ptrs, slots, out, 1,
                        "gda", s)
    g.replay()
    torch.cuda.synchronize()
    gdn.gdn_check_device_error()
    assert torch.equal(out, eager_out) and torch.equal(slots, eager_slots)


@pytest.mark.parametrize("mode", ["gda", "kda"])
def test_chunked_prefill_in_a_graph(gdn, mode):
    b = inputs.make_batch(251, [300, 70, 5], 2, 128, 128, mode=mode, n_slots=3)
    d = to_dev(b)
    N, ntok, H = 3, b.q.shape[0], 2
    cu = b.cu_seqlens.to(torch.int32).cuda()
    shape = gdn.gdn_varlen_shape(N, ntok, H, 128, 128, gdn.GDN_BF16, b.scale)
    ws_bytes = gdn.gdn_chunked_workspace_size(shape, 3)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ptrs = gdn.state_ptr_array(gdn.per_seq_state_ptrs(d["state"], N), "cuda")

    def run(out, slots, stream=None):
        gdn.gdn_forward_chunked(shape, cu, d["q"], d["k"], d["v"], d["g"], d["beta"], ptrs,
                                slots, out, 3, mode, ws, ws_bytes, stream)

    eager_out = torch.full((ntok, H, 128), float("nan"), device="cuda")
    eager_slots = torch.full((N, 3, H, 128, 128), float("nan"), device="cuda")
    run(eager_out, eager_slots)
    torch.cuda.synchronize()
    out = torch.full_like(eager_out, float("nan"))
    slots = torch.full_like(eager_slots, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s), torch.cuda.graph(g, stream=s):
        run(out, slots, s)
    for _ in range(2):  # replays reuse the workspace as the previous one left it
        g.replay()
    torch.cuda.synchronize()
    gdn.gdn_check_device_error()
    assert torch.equal(out, eager_out)
    assert torch.equal(slots.nan_to_num(0.0), eager_slots.nan_to_num(0.0))


def test_checkpointed_prefill_in_a_graph(gdn):
    # the checkpoint instance of the scan kernel and the tail's checkpoint
    # stores, captured and replayed, equal an eager call bit for bit
    b = inputs.make_batch(252, [300, 140, 5], 2, 128, 128, mode="gda", n_slots=3)
    d = to_dev(b)
    N, ntok, H = 3, b.q.shape[0], 2
    cu = b.cu_seqlens.to(torch.int32).cuda()
    shape = gdn.gdn_varlen_shape(N, ntok, H, 128, 128, gdn.GDN_BF16, b.scale)
    ws_bytes = gdn.gdn_chunked_workspace_size(shape, 3)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ptrs = gdn.state_ptr_array(gdn.per_seq_state_ptrs(d["state"], N), "cuda")

    def run(out, slots, cks, stream=None):
        gdn.gdn_forward_chunked_checkpointed(shape, cu, d["q"], d["k"], d["v"], d["g"],
                                             d["beta"], ptrs, slots, out, 3, "gda", cks, 64, 4,
                                             ws, ws_bytes, stream)

    def bufs():
        return (torch.full((ntok, H, 128), float("nan"), device="cuda"),
                torch.full((N, 3, H, 128, 128), float("nan"), device="cuda"),
                torch.full((N, 4, H, 128, 128), float("nan"), device="cuda"))

    eager = bufs()
    run(*eager)
    torch.cuda.synchronize()
    got = bufs()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s), torch.cuda.graph(g, stream=s):
        run(*got, s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    gdn.gdn_check_device_error()
    for x, y in zip(got, eager):
        assert torch.equal(x.nan_to_num(0.0), y.nan_to_num(0.0))
    assert not torch.isnan(got[2][0]).any()  # L=300 reaches all 4 checkpoints
