"""GPU parity of the chunked (tensor-core) prefill against the fp64 oracle,
through the C ABI: varlen batches with ragged last chunks, sequences shorter
than one chunk or than K, GDA and KDA, K snapshot slots from the recurrent
tail, the full-size KDA and varlen workloads, zero-state pointers and a bad
cu_seqlens table reported by the device."""
import numpy as np
import pytest
import torch

from gated_delta_net_02_gb300 import inputs

from _helpers import gpu_forward, oracle_run, rel_l2, to_dev

pytestmark = pytest.mark.gpu

TOL_BF16 = 5e-3


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_net_02_gb300 import build
    build.build()
    from gated_delta_net_02_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


def chunked_forward(gdn, b, n_slots=None, state_ptrs=None, cu=None, check=True,
                    dev_tensors=None):
    n_slots = b.n_slots if n_slots is None else n_slots
    d = dev_tensors or to_dev(b)
    N = b.n_seqs
    H, Dk, Dv = b.v.shape[1], b.q.shape[2], b.v.shape[2]
    ntok = b.q.shape[0]
    cu_dev = (b.cu_seqlens if cu is None else cu).to(torch.int32).cuda()
    shape = gdn.gdn_varlen_shape(N, ntok, H, Dk, Dv, gdn.dtype_code(b.q.dtype), b.scale,
                                 b.q.shape[1], gdn.QK_MAPS[b.qk_map])
    ws_bytes = gdn.gdn_chunked_workspace_size(shape, n_slots)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    slots = torch.full((N, n_slots, H, Dk, Dv), float("nan"), device="cuda")
    out = torch.full((ntok, H, Dv), float("nan"), device="cuda")
    if state_ptrs is None:
        state_ptrs = gdn.state_ptr_array(gdn.per_seq_state_ptrs(d["state"], N), "cuda")
    gdn.gdn_forward_chunked(shape, cu_dev, d["q"], d["k"], d["v"], d["g"], d["beta"], state_ptrs,
                            slots, out, n_slots, b.mode, ws, ws_bytes)
    if check:
        gdn.gdn_check_device_error()
    return out, slots


def compare(b, out, slots, n_slots=None, tol=TOL_BF16):
    n_slots = b.n_slots if n_slots is None else n_slots
    o_ref, s_ref, sl_ref = oracle_run(b, n_slots=n_slots)
    out = out.double().cpu().numpy()
    slots = slots.double().cpu().numpy()
    assert not np.isnan(out).any(), "unwritten outputs"
    e_out = rel_l2(out, o_ref)
    ran = b.seq_len.numpy() > 0    # an empty sequence writes no slot
    e_fin = rel_l2(slots[ran, -1], s_ref[ran])
    assert e_out <= tol, f"out rel-L2 {e_out}"
    assert e_fin <= tol, f"final state rel-L2 {e_fin}"
    for j in range(n_slots):
        written = ~np.isnan(sl_ref[:, j, 0, 0, 0])
        if written.any():
            e = rel_l2(slots[written, j], sl_ref[written, j])
            assert e <= tol, f"slot {j} rel-L2 {e}"
        assert np.isnan(slots[~written, j]).all()
    return e_out, e_fin


@pytest.mark.parametrize("mode", ["gda", "kda"])
def test_varlen_ragged_small(gdn, mode):
    # chunk-multiple, ragged, one-chunk, shorter-than-K and empty sequences
    lens = [200, 64, 131, 9, 1, 0, 65]
    b = inputs.make_batch(41, lens, 2, 128, 128, mode=mode, n_slots=4)
    out, slots = chunked_forward(gdn, b)
    compare(b, out, slots)


@pytest.mark.parametrize("n_seqs", [300, 4100])
def test_many_sequences_work_list(gdn, n_seqs):
    """Many short sequences (0 to 150 tokens: empty, shorter than K, one and
    several chunks), H=1: 300 sequences (the work list keeps cu_seqlens in
    shared memory and all its threads fill the chunk table) and 4100 (past its
    shared-memory capacity: each thread fills its own sequences' chunks)"""
    gen = np.random.default_rng(n_seqs)
    lens = gen.integers(0, 151, n_seqs)
    lens[:5] = [0, 64, 0, 0, 129]  # runs of empty sequences between chunked ones
    b = inputs.make_batch(48, lens.tolist(), 1, 128, 128, mode="gda", n_slots=2)
    out, slots = chunked_forward(gdn, b)
    compare(b, out, slots)


@pytest.mark.parametrize("mode", ["gda", "kda"])
@pytest.mark.parametrize("K", [1, 8])
def test_single_long_sequence(gdn, mode, K):
    b = inputs.make_batch(42 + K, [777], 3, 128, 128, mode=mode, n_slots=K)
    out, slots = chunked_forward(gdn, b)
    compare(b, out, slots)


def test_kda_prefill_full_size(gdn):
    """1 sequence, T=4096, H=32, D=128, KDA gate, bf16 q/k/v, K=1, seed 3."""
    b = inputs.kda_prefill(3)
    out, slots = chunked_forward(gdn, b)
    e_out, e_fin = compare(b, out, slots)
    print(f"kda prefill: out rel-L2 {e_out:.2e}, state rel-L2 {e_fin:.2e}")


def test_varlen_prefill_full_size(gdn):
    """8 sequences, lengths ~U[512, 8192], H=16, D=128, GDA, K=8, seed 4."""
    b = inputs.varlen_prefill(4)
    out, slots = chunked_forward(gdn, b)
    e_out, e_fin = compare(b, out, slots)
    print(f"varlen prefill: out rel-L2 {e_out:.2e}, state rel-L2 {e_fin:.2e}")


@pytest.mark.parametrize("mode", ["gda", "kda"])
@pytest.mark.parametrize("n_slots", [1, 64, 65])
def test_slot_counts_around_one_chunk(gdn, mode, n_slots):
    # the recurrent tail covers the last n_slots tokens: a whole chunk's
    # worth and more; lengths below, at and above n_slots, so the chunked
    # part ends on and off chunk boundaries
    lens = [300, 64, 130, 40, 65, 1]
    b = inputs.make_batch(47, lens, 2, 128, 128, mode=mode, n_slots=n_slots)
    out, slots = chunked_forward(gdn, b)
    compare(b, out, slots)


def test_matches_recurrent_path(gdn):
    b = inputs.make_batch(43, [300, 300], 2, 128, 128, mode="gda", n_slots=2)
    out_c, sl_c = chunked_forward(gdn, b)
    out_r, sl_r = gpu_forward(b)
    assert rel_l2(out_c.double().cpu().numpy(), out_r.double().cpu().numpy()) < TOL_BF16
    assert rel_l2(sl_c.double().cpu().numpy(), sl_r.double().cpu().numpy()) < TOL_BF16


def test_zero_state_pointers(gdn):
    b = inputs.make_batch(44, [150, 70], 2, 128, 128, state_std=0.0, n_slots=2)
    out_a, sl_a = chunked_forward(gdn, b)
    ptrs = gdn.state_ptr_array([0, 0], "cuda")
    out_b, sl_b = chunked_forward(gdn, b, state_ptrs=ptrs)
    assert torch.equal(out_a, out_b) and torch.equal(sl_a, sl_b)


def test_bad_cu_seqlens_reported_by_device(gdn):
    b = inputs.make_batch(45, [100, 50], 2, 128, 128, n_slots=1)
    bad = torch.tensor([0, 120, 150], dtype=torch.int64)   # non-matching split is fine
    chunked_forward(gdn, b, cu=bad)                           # valid table: no error
    for cu in ([0, 160, 150], [5, 100, 150], [0, 100, 149]):
        chunked_forward(gdn, b, cu=torch.tensor(cu), check=False)
        with pytest.raises(gdn.GDNError) as e:
            gdn.gdn_check_device_error()
        assert e.value.status == gdn.GDN_ERR_DEVICE_ARG
    gdn.gdn_check_device_error()


def test_repeated_calls_reuse_dirty_workspace(gdn):
    b = inputs.make_batch(46, [257, 90], 2, 128, 128, mode="kda", n_slots=3)
    out1, sl1 = chunked_forward(gdn, b)
    out2, sl2 = chunked_forward(gdn, b)
    assert torch.equal(out1, out2) and torch.equal(sl1, sl2)


def test_kda_strong_decay_inside_range(gdn):
    # per-row gates ~ -softplus(N(0,1)): a chunk's cumulative log-gate reaches
    # about -50 to -70 per channel, inside the range the chunk form accepts
    b = inputs.make_batch(47, [200, 130], 2, 128, 128, mode="kda", n_slots=2,
                          kda_gate_scale=1.0)
    gmin = float(torch.cumsum(b.g[:64], dim=0).min())
    assert -80.0 < gmin < -40.0
    out, slots = chunked_forward(gdn, b)
    compare(b, out, slots)


def test_kda_decay_beyond_range_reported(gdn):
    # gates 3x stronger leave [-80, 80] inside the first chunk: the device
    # reports it, and the token-loop entry point still matches the oracle
    b = inputs.make_batch(48, [200], 2, 128, 128, mode="kda", n_slots=1, kda_gate_scale=3.0)
    assert float(torch.cumsum(b.g[:64], dim=0).min()) < -80.0
    chunked_forward(gdn, b, check=False)
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_check_device_error()
    assert e.value.status == gdn.GDN_ERR_DEVICE_ARG
    assert "e^80" in str(e.value)
    out, slots = gpu_forward(b)
    o_ref, s_ref, _ = oracle_run(b, n_slots=1)
    assert rel_l2(out.double().cpu().numpy(), o_ref) <= TOL_BF16
    assert rel_l2(slots[:, -1].double().cpu().numpy(), s_ref) <= TOL_BF16


@pytest.mark.parametrize("qk_map", ["tiled", "grouped"])
@pytest.mark.parametrize("mode", ["gda", "kda"])
def test_grouped_query_heads(gdn, qk_map, mode):
    # 4 value heads reading 2 q/k heads, ragged varlen batch with a short tail
    b = inputs.make_batch(230, [300, 70, 5], 4, 128, 128, mode=mode, n_slots=4, H_qk=2,
                          qk_map=qk_map)
    out, slots = chunked_forward(gdn, b)
    compare(b, out, slots)


@pytest.mark.parametrize("mode", ["gda", "kda"])
@pytest.mark.parametrize("dtype,D", [(torch.float32, 128), (torch.float32, 64),
                                     (torch.bfloat16, 64)])
def test_token_loop_route(gdn, mode, dtype, D):
    """fp32 inputs and 64-wide heads take the recurrent kernel for every
    token: fp32 must then meet the fp32 tolerance."""
    b = inputs.make_batch(240, [150, 3, 0, 70], 2, D, D, dtype=dtype, mode=mode, n_slots=4)
    out, slots = chunked_forward(gdn, b)
    tol = 1e-5 if dtype == torch.float32 else TOL_BF16
    compare(b, out, slots, tol=tol)


def test_token_loop_route_needs_only_the_work_list(gdn):
    big = gdn.gdn_varlen_shape(8, 40000, 16, 128, 128, gdn.GDN_BF16, 0.0)
    f32 = gdn.gdn_varlen_shape(8, 40000, 16, 128, 128, gdn.GDN_F32, 0.0)
    assert gdn.gdn_chunked_workspace_size(f32, 8) < 4096 < gdn.gdn_chunked_workspace_size(big, 8)


def worst_head(x, ref):
    """Largest rel-L2 over the (sequence, head) pairs of [N, H, ...] arrays."""
    worst, where = 0.0, None
    for s in range(x.shape[0]):
        for h in range(x.shape[1]):
            e = rel_l2(x[s, h], ref[s, h])
            if e > worst:
                worst, where = e, (s, h)
    return worst, where


@pytest.mark.parametrize("T,seed", [(4096, 3), (4096, 30), (4096, 300),
                                    (8192, 3), (8192, 30), (8192, 300)])
def test_kda_precision_margin(gdn, T, seed):
    """The KDA prefill workload (1 sequence, H=32, D=128, per-row gates
    -softplus(N(0,1)) * 0.1, bf16 q/k/v) at its length and at twice it, on
    three seeds: the whole-tensor rel-L2 of out, state and slot stays within
    the 5e-3 bf16 budget, and the worst (sequence, head) is printed."""
    b = inputs.kda_prefill(seed, T=T)
    out, slots = chunked_forward(gdn, b)
    e_out, e_fin = compare(b, out, slots)
    o_ref, s_ref, _ = oracle_run(b)
    H = b.v.shape[1]
    o = out.double().cpu().numpy().reshape(1, T, H, -1).transpose(0, 2, 1, 3)
    w_out, at_out = worst_head(o, o_ref.reshape(1, T, H, -1).transpose(0, 2, 1, 3))
    w_st, at_st = worst_head(slots[:, -1].double().cpu().numpy(), s_ref)
    print(f"KDA T={T} seed={seed}: out {e_out:.3e} (worst head {w_out:.3e} at {at_out}), "
          f"state {e_fin:.3e} (worst head {w_st:.3e} at {at_st})")


@pytest.mark.parametrize("mode", ["gda", "kda"])
def test_prep_beside_scan_equals_prep_before_scan(gdn, mode):
    """A batch of 8 sequences x 16 heads needs 256 scan CTAs, more than the SMs,
    so chunk prep runs before the scan; one sequence alone (32 scan CTAs) runs
    the prep beside the scan on the free SMs, the scan waiting for each tile's
    ready flag. Per tile and per chain the arithmetic is the same, so every
    sequence's outputs and slots must agree bit for bit between the two."""
    lens = [200, 330, 64, 129, 257, 70, 300, 191]
    b = inputs.make_batch(250, lens, 16, 128, 128, mode=mode, n_slots=3)
    assert torch.cuda.get_device_properties(0).multi_processor_count < 256
    out_all, slots_all = chunked_forward(gdn, b)
    cu = b.cu_seqlens.tolist()
    for s in range(len(lens)):
        sl = slice(cu[s], cu[s + 1])
        one = inputs.GDNBatch(b.q[sl], b.k[sl], b.v[sl], b.g[sl], b.beta[sl],
                              b.state[s:s + 1], mode, b.scale, torch.tensor([lens[s]]), 3)
        out_one, slots_one = chunked_forward(gdn, one)
        assert torch.equal(out_one, out_all[sl]), f"sequence {s}"
        assert torch.equal(slots_one[0], slots_all[s]), f"sequence {s}"
    compare(b, out_all, slots_all)
