"""GPU parity of the recurrent (token-loop) kernel against the fp64 oracle,
through the C ABI: decode, speculative verify with K slots, rollback and
prefix re-runs (bit-exact), GDA/KDA, fp32/bf16, every head-size pair, ragged
token tiles, zero-state pointers, and device-side argument checks."""
import numpy as np
import pytest
import torch

from gated_delta_net_02_gb300 import inputs

from _helpers import TOL, gpu_forward, oracle_run, rel_l2, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_net_02_gb300 import build
    build.build()
    from gated_delta_net_02_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


def check_against_oracle(b, out, slots, n_slots=None, tol=None):
    n_slots = b.n_slots if n_slots is None else n_slots
    o_ref, s_ref, sl_ref = oracle_run(b, n_slots=n_slots)
    tol = TOL[b.q.dtype] if tol is None else tol
    out = out.double().cpu().numpy()
    slots = slots.double().cpu().numpy()
    assert not np.isnan(out).any()
    e_out = rel_l2(out, o_ref)
    assert e_out <= tol, f"out rel-L2 {e_out}"
    ran = b.seq_len.numpy() > 0    # an empty sequence writes no slot
    e_fin = rel_l2(slots[ran, -1], s_ref[ran]) if ran.any() else 0.0
    assert e_fin <= tol, f"final state rel-L2 {e_fin}"
    for j in range(n_slots):
        written = ~np.isnan(sl_ref[:, j, 0, 0, 0])
        if written.any():
            e = rel_l2(slots[written, j], sl_ref[written, j])
            assert e <= tol, f"slot {j} rel-L2 {e}"
        # slots the sequence never reaches stay untouched (NaN-filled here)
        assert np.isnan(slots[~written, j]).all()
    return e_out, e_fin


def test_tiny_gda_fp32(gdn):
    """1 sequence, H=4, D=64, T=32, fp32, K=1, zero state, seed 0."""
    b = inputs.tiny_gda(0)
    out, slots = gpu_forward(b)
    e_out, e_fin = check_against_oracle(b, out, slots)
    assert e_out < 1e-5 and e_fin < 1e-5


@pytest.mark.parametrize("Dk,Dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("mode", ["gda", "kda"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_head_sizes_modes_dtypes(gdn, Dk, Dv, mode, dtype):
    # T = 19 spans three staged tiles of 8 tokens with a ragged tail
    b = inputs.make_batch(100 + Dk + Dv, [19] * 3, 3, Dk, Dv, dtype=dtype, mode=mode,
                          n_slots=4)
    out, slots = gpu_forward(b)
    check_against_oracle(b, out, slots)


def test_decode_full_size_chained_steps(gdn):
    """64 sequences x 1 token, H=16, D=128, bf16, GDA; 4 chained steps with
    fresh tokens, each step's slot feeding the next step's state_in."""
    N, H, D = 64, 16, 128
    state0 = inputs.decode_state(1, N, H, D)
    S_ref = inputs.to_f64(state0)
    bank = [state0.cuda(), torch.empty_like(state0, device="cuda")]
    import oracle
    for step in range(4):
        q, k, v, g, beta = inputs.decode_tokens(1, step, N, H, D)
        b = inputs.GDNBatch(q, k, v, g, beta, state0, "gda", D ** -0.5,
                            torch.ones(N, dtype=torch.int64), 1)
        src, dst = bank[step % 2], bank[(step + 1) % 2]
        ptrs = gdn.state_ptr_array(gdn.per_seq_state_ptrs(src, N), "cuda")
        out, _ = gpu_forward(b, state_ptrs=ptrs, slots=dst.view(N, 1, H, D, D),
                             dev_tensors=dict(q=q.cuda(), k=k.cuda(), v=v.cuda(),
                                              g=g.cuda(), beta=beta.cuda(), state=src))
        o_ref, S_ref, _ = oracle.forward(inputs.to_f64(q), inputs.to_f64(k), inputs.to_f64(v),
                                         inputs.to_f64(g), inputs.to_f64(beta), S_ref,
                                         scale=D ** -0.5)
        assert rel_l2(out.double().cpu().numpy(), o_ref) <= 5e-3
        assert rel_l2(dst.double().cpu().numpy(), S_ref) <= 5e-3
    # the recurrent kernel itself computes in fp32: far inside the bf16 budget
    assert rel_l2(dst.double().cpu().numpy(), S_ref) < 1e-5


def test_decode_1000_step_chain_against_oracle(gdn):
    """The batched decode workload in full: 64 sequences x 1 token, H=16,
    D=128, bf16 q/k/v, GDA, state ~N(0, 0.05), 1000 consecutive steps with
    fresh tokens, each step reading the state the previous step wrote. The
    oracle runs the same chain (the 1000 steps of a sequence are its tokens),
    100 steps per call; every step's output and the state after every 100th
    step are compared."""
    import oracle
    N, H, D, STEPS, BLOCK = 64, 16, 128, 1000, 100
    state0 = inputs.decode_state(1, N, H, D)
    bank = [state0.cuda(), torch.empty(N, H, D, D, device="cuda")]
    ptrs = [gdn.state_ptr_array(gdn.per_seq_state_ptrs(b_, N), "cuda") for b_ in bank]
    shape = gdn.gdn_shape(N, 1, H, D, D, gdn.GDN_BF16, D ** -0.5)
    S_ref = inputs.to_f64(state0)
    worst_out = worst_state = 0.0
    for blk in range(STEPS // BLOCK):
        toks = [inputs.decode_tokens(1, blk * BLOCK + t, N, H, D) for t in range(BLOCK)]
        dev = [[x.cuda() for x in tk] for tk in toks]
        outs = torch.empty(BLOCK, N, H, D, device="cuda")
        for t in range(BLOCK):
            i = blk * BLOCK + t
            q, k, v, g, beta = dev[t]
            gdn.gdn_forward(shape, q, k, v, g, beta, ptrs[i % 2], bank[(i + 1) % 2], outs[t],
                            1, "gda")
        gdn.gdn_check_device_error()
        # the oracle: sequence s's tokens are steps t of this block, packed
        # sequence by sequence
        seq = [torch.stack([tk[j] for tk in toks], dim=1) for j in range(5)]   # [N, T, ...]
        q, k, v, g, beta = (inputs.to_f64(x.reshape(N * BLOCK, *x.shape[2:])) for x in seq)
        o_ref, S_ref, _ = oracle.forward(q, k, v, g, beta, S_ref, scale=D ** -0.5,
                                         seq_start=np.arange(N) * BLOCK,
                                         seq_len=np.full(N, BLOCK))
        got = outs.permute(1, 0, 2, 3).reshape(N * BLOCK, H, D).double().cpu().numpy()
        e_out = rel_l2(got, o_ref)
        e_st = rel_l2(bank[((blk + 1) * BLOCK) % 2].double().cpu().numpy(), S_ref)
        worst_out, worst_state = max(worst_out, e_out), max(worst_state, e_st)
        assert e_out <= 5e-3 and e_st <= 5e-3, (blk, e_out, e_st)
    print(f"decode 1000-step chain: worst out rel-L2 {worst_out:.2e}, "
          f"worst state rel-L2 {worst_state:.2e}")
    # fp32 arithmetic on exact bf16 inputs: far inside the bf16 budget
    assert worst_state < 1e-5


def test_verify_full_size_and_rollback_bit_exact(gdn):
    """32 sequences x T=8, K=8, H=16, D=128, bf16: parity, then rollback to
    n_accepted ~ U{0..8} and a re-run of only the accepted prefix from the
    same state_in; the chosen slot must equal the re-run bit for bit."""
    b = inputs.verify_batch(2)
    N, T, K = 32, 8, 8
    d = to_dev(b)
    out, slots = gpu_forward(b, dev_tensors=d)
    check_against_oracle(b, out, slots)

    table = gdn.SeqTable(N, K)
    for s in range(N):
        table.record(s, T)
    n_acc = b.meta["n_accepted"].tolist()
    H, D = 16, 128
    for s in range(N):
        n = n_acc[s]
        slot = table.rollback(s, n)
        chosen = d["state"][s] if slot == -1 else slots[s, slot]
        if n == 0:
            assert slot == -1
            continue
        sl = slice(s * T, s * T + n)
        sub = inputs.GDNBatch(b.q[sl], b.k[sl], b.v[sl], b.g[sl], b.beta[sl],
                              b.state[s:s + 1], "gda", b.scale,
                              torch.tensor([n]), 1)
        ptr = gdn.state_ptr_array([d["state"][s].data_ptr()], "cuda")
        _, re_slots = gpu_forward(sub, state_ptrs=ptr,
                                  dev_tensors=dict(q=d["q"][sl], k=d["k"][sl], v=d["v"][sl],
                                                   g=d["g"][sl], beta=d["beta"][sl],
                                                   state=d["state"][s:s + 1]))
        assert torch.equal(re_slots[0, 0], chosen), f"seq {s} n_accepted {n}"


def test_single_slot_equals_final_of_multi_slot(gdn):
    b = inputs.make_batch(7, [8] * 4, 2, 128, 128, n_slots=8)
    _, slots8 = gpu_forward(b)
    _, slots1 = gpu_forward(b, n_slots=1)
    assert torch.equal(slots8[:, -1], slots1[:, 0])


def test_forward_after_rollback_reads_only_selected_slot(gdn):
    """A forward that starts from a rolled-back slot must not depend on the
    other slots ("loading into a dirty ctx")."""
    b = inputs.make_batch(8, [8] * 2, 2, 128, 128, n_slots=8)
    d = to_dev(b)
    _, slots = gpu_forward(b, dev_tensors=d)
    table = gdn.SeqTable(2, 8)
    table.record(0, 8)
    table.record(1, 8)
    picks = [table.rollback(0, 3), table.rollback(1, 6)]
    nxt = inputs.make_batch(9, [5] * 2, 2, 128, 128, n_slots=2)
    dn = to_dev(nxt)
    base = [gdn.gdn_slot_state_ptr(slots, s, picks[s], 8, 2, 128, 128) for s in range(2)]
    ptrs = gdn.state_ptr_array(base, "cuda")
    out1, sl1 = gpu_forward(nxt, state_ptrs=ptrs, dev_tensors=dn)
    # scribble over every slot that was not chosen, then run again
    for s in range(2):
        for j in range(8):
            if j != picks[s]:
                slots[s, j].fill_(1e30)
    out2, sl2 = gpu_forward(nxt, state_ptrs=ptrs, dev_tensors=dn)
    assert torch.equal(out1, out2) and torch.equal(sl1, sl2)


def test_zero_state_pointer_and_empty(gdn):
    b = inputs.make_batch(10, [6] * 2, 2, 64, 64, state_std=0.0, n_slots=2)
    out_a, sl_a = gpu_forward(b)                                  # explicit zeros
    ptrs = gdn.state_ptr_array([0, 0], "cuda")                     # NULL entries
    out_b, sl_b = gpu_forward(b, state_ptrs=ptrs)
    assert torch.equal(out_a, out_b) and torch.equal(sl_a, sl_b)
    # T = 0: nothing written, no error
    e = inputs.make_batch(11, [0] * 2, 2, 64, 64, n_slots=2)
    _, sl = gpu_forward(e)
    assert torch.isnan(sl).all()


def test_short_sequence_leaves_leading_slots(gdn):
    b = inputs.make_batch(12, [3] * 2, 2, 128, 128, n_slots=6)
    out, slots = gpu_forward(b)
    check_against_oracle(b, out, slots)
    assert torch.isnan(slots[:, :3]).all()


def test_state_in_inside_slots_is_refused_on_device(gdn):
    b = inputs.make_batch(13, [4] * 2, 2, 64, 64, n_slots=2)
    slots = torch.zeros(2, 2, 2, 64, 64, device="cuda")
    ptrs = gdn.state_ptr_array([slots[1, 0].data_ptr(), 0], "cuda")
    gpu_forward(b, state_ptrs=ptrs, slots=slots, check=False)
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_check_device_error()
    assert e.value.status == gdn.GDN_ERR_DEVICE_ARG
    gdn.gdn_check_device_error()  # the word was cleared


def test_many_sequences_ragged_grid(gdn):
    # 37 sequences x 5 heads: the grid is not a multiple of anything
    b = inputs.make_batch(14, [9] * 37, 5, 128, 64, mode="kda", n_slots=3)
    out, slots = gpu_forward(b)
    check_against_oracle(b, out, slots)


def test_runs_on_a_side_stream(gdn):
    b = inputs.make_batch(15, [8] * 4, 2, 128, 128, n_slots=2)
    s = torch.cuda.Stream()
    d = to_dev(b)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        out, slots = gpu_forward(b, stream=s, dev_tensors=d)
    s.synchronize()
    check_against_oracle(b, out, slots)


@pytest.mark.parametrize("mode", ["gda", "kda"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n_slots", [1, 3])
def test_decode_step_bitwise_equals_first_token_of_longer_run(gdn, mode, dtype, n_slots):
    """A decode step (T = 1) must reproduce, bit for bit, token 0 of a T = 2
    run from the same state: the recurrent kernel's per-token arithmetic and
    its reduction order do not depend on T or on the number of slots."""
    b2 = inputs.make_batch(200 + n_slots, [2] * 5, 3, 128, 128, dtype=dtype, mode=mode,
                           n_slots=2)
    d2 = to_dev(b2)
    out2, slots2 = gpu_forward(b2, dev_tensors=d2)
    first = [2 * s for s in range(5)]
    b1 = inputs.GDNBatch(b2.q[first], b2.k[first], b2.v[first], b2.g[first], b2.beta[first],
                         b2.state, mode, b2.scale, torch.ones(5, dtype=torch.int64), n_slots)
    d1 = {n: t[first] if n != "state" else t for n, t in d2.items()}
    out1, slots1 = gpu_forward(b1, dev_tensors={n: t.contiguous() for n, t in d1.items()})
    assert torch.equal(out1, out2[first])
    assert torch.equal(slots1[:, -1], slots2[:, 0])
    if n_slots > 1:  # a single token writes only the last slot
        assert torch.isnan(slots1[:, :-1]).all()


def test_decode_step_null_state_and_few_items(gdn):
    # 1 sequence x 1 head (a grid of two CTAs); NULL state pointer
    b = inputs.make_batch(210, [1], 1, 128, 128, state_std=0.0, n_slots=1)
    out_a, sl_a = gpu_forward(b)
    out_b, sl_b = gpu_forward(b, state_ptrs=gdn.state_ptr_array([0], "cuda"))
    assert torch.equal(out_a, out_b) and torch.equal(sl_a, sl_b)
    check_against_oracle(b, out_a, sl_a)


def test_decode_step_state_in_inside_slots_is_refused(gdn):
    b = inputs.make_batch(211, [1] * 2, 2, 128, 128, n_slots=2)
    slots = torch.zeros(2, 2, 2, 128, 128, device="cuda")
    ptrs = gdn.state_ptr_array([slots[1, 0].data_ptr(), 0], "cuda")
    gpu_forward(b, state_ptrs=ptrs, slots=slots, check=False)
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_check_device_error()
    assert e.value.status == gdn.GDN_ERR_DEVICE_ARG
    gdn.gdn_check_device_error()


@pytest.mark.parametrize("qk_map", ["tiled", "grouped"])
@pytest.mark.parametrize("mode", ["gda", "kda"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_grouped_query_heads(gdn, qk_map, mode, dtype):
    # 6 value heads reading 2 q/k heads; T = 19 spans three token tiles
    b = inputs.make_batch(220, [19] * 2, 6, 128, 128, dtype=dtype, mode=mode, n_slots=3,
                          H_qk=2, qk_map=qk_map)
    out, slots = gpu_forward(b)
    check_against_oracle(b, out, slots)


def test_grouped_query_decode_step(gdn):
    b = inputs.make_batch(221, [1] * 8, 8, 128, 128, n_slots=1, H_qk=2, qk_map="grouped")
    out, slots = gpu_forward(b)
    check_against_oracle(b, out, slots)
