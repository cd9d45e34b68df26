"""GPU parity of the checkpointed prefill (gdn_forward_chunked_checkpointed)
against the fp64 oracle, through the C ABI.

- Every checkpoint a sequence reaches equals the oracle's state after that
  many tokens (tolerance of the input dtype); entries it does not reach stay
  untouched. Checkpoints inside the chunked part come from the chunk scan,
  those among the last n_slots tokens from the token loop; the fp32 and
  64-wide routes write all of them from the token loop.
- A checkpoint in the token-loop tail is bit-identical to the snapshot slot
  that holds the same state, and a scan checkpoint does not depend on the
  tokens after it (bit-identical when the sequences are cut short).
- Restarting from what gdn_checkpoint_select chooses and replaying the rest
  with gdn_forward_chunked gives the oracle's state after n_keep tokens.
- Outputs and slots are those of gdn_forward_chunked, bit for bit.
"""
import numpy as np
import pytest
import torch

from gated_delta_net_02_gb300 import inputs

import oracle

from _helpers import rel_l2, to_dev, TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_net_02_gb300 import build
    build.build()
    from gated_delta_net_02_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


def run(gdn, b, every, max_ckpts, ckpt=True, d=None):
    """One call; returns (out, slots, checkpoints) on the device (checkpoints
    prefilled with NaN, so unwritten entries stay NaN)."""
    d = d or to_dev(b)
    N, n_slots = b.n_seqs, b.n_slots
    H, Dk, Dv = b.v.shape[1], b.q.shape[2], b.v.shape[2]
    ntok = b.q.shape[0]
    cu_dev = b.cu_seqlens.to(torch.int32).cuda()
    shape = gdn.gdn_varlen_shape(N, ntok, H, Dk, Dv, gdn.dtype_code(b.q.dtype), b.scale,
                                 b.q.shape[1], gdn.QK_MAPS[b.qk_map])
    ws_bytes = gdn.gdn_chunked_workspace_size(shape, n_slots)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    slots = torch.full((N, n_slots, H, Dk, Dv), float("nan"), device="cuda")
    out = torch.full((ntok, H, Dv), float("nan"), device="cuda")
    cks = torch.full((N, max_ckpts, H, Dk, Dv), float("nan"), device="cuda")
    ptrs = gdn.state_ptr_array(gdn.per_seq_state_ptrs(d["state"], N), "cuda")
    if ckpt:
        gdn.gdn_forward_chunked_checkpointed(shape, cu_dev, d["q"], d["k"], d["v"], d["g"],
                                             d["beta"], ptrs, slots, out, n_slots, b.mode,
                                             cks, every, max_ckpts, ws, ws_bytes)
    else:
        gdn.gdn_forward_chunked(shape, cu_dev, d["q"], d["k"], d["v"], d["g"], d["beta"],
                                ptrs, slots, out, n_slots, b.mode, ws, ws_bytes)
    gdn.gdn_check_device_error()
    torch.cuda.synchronize()
    return out, slots, cks


def oracle_prefix_state(b, counts):
    """State of every sequence after counts[s] of its tokens (fp64 oracle)."""
    lens = np.minimum(np.asarray(counts, dtype=np.int64), b.seq_len.numpy())
    f = inputs.to_f64
    return oracle.forward(f(b.q), f(b.k), f(b.v), f(b.g), f(b.beta), f(b.state),
                          mode=b.mode, scale=b.scale, seq_start=b.cu_seqlens.numpy()[:-1],
                          seq_len=lens, qk_map=b.qk_map)[1]


def check_checkpoints(b, cks, every, max_ckpts, tol):
    cks = cks.double().cpu().numpy()
    L = b.seq_len.numpy()
    n_written = 0
    for m in range(max_ckpts):
        p = (m + 1) * every
        reach = L >= p
        if reach.any():
            ref = oracle_prefix_state(b, [p] * b.n_seqs)
            e = rel_l2(cks[reach, m], ref[reach])
            assert e <= tol, f"checkpoint {m} (after {p} tokens) rel-L2 {e}"
            n_written += int(reach.sum())
        assert np.isnan(cks[~reach, m]).all(), f"checkpoint {m} written past a sequence end"
    return n_written


# lengths: several boundaries inside the chunked part (700), a boundary in the
# token-loop tail (257, 320: 4 slots cover tokens 253..256 and 316..319), a
# ragged last chunk ending just before a boundary (191), short and empty
# sequences, and one exactly one chunk long
LENS = [700, 257, 64, 191, 9, 0, 320]


@pytest.mark.parametrize("mode", ["gda", "kda"])
def test_one_slot_checkpoints(gdn, mode):
    """One slot: the chunk scan covers every token and writes the slot itself
    (no token-loop tail), so a checkpoint on a sequence's last token comes from
    the scan too. Lengths ending on a boundary (320, 256, 64), ragged (257,
    191, 9) and empty."""
    lens = [320, 257, 256, 191, 64, 9, 0]
    every, max_ckpts = 64, 6
    b = inputs.make_batch(77, lens, 2, 128, 128, mode=mode, n_slots=1)
    out, slots, cks = run(gdn, b, every, max_ckpts)
    assert check_checkpoints(b, cks, every, max_ckpts, TOL[torch.bfloat16]) > 0
    final = oracle_prefix_state(b, b.seq_len.numpy())
    L = b.seq_len.numpy()
    have = L > 0
    sl = slots.double().cpu().numpy()
    assert rel_l2(sl[have, 0], final[have]) <= TOL[torch.bfloat16]
    assert np.isnan(sl[~have]).all()
    for s, n in enumerate(L):  # a checkpoint on the last token is the slot itself
        if n > 0 and n % every == 0 and n // every <= max_ckpts:
            assert torch.equal(cks[s, n // every - 1], slots[s, 0])
    out0, slots0, _ = run(gdn, b, every, max_ckpts, ckpt=False)
    assert torch.equal(out.nan_to_num(7.0), out0.nan_to_num(7.0))
    assert torch.equal(slots.nan_to_num(7.0), slots0.nan_to_num(7.0))


@pytest.mark.parametrize("mode", ["gda", "kda"])
@pytest.mark.parametrize("every,max_ckpts", [(64, 12), (128, 2)])
def test_checkpoints_match_oracle_bf16(gdn, mode, every, max_ckpts):
    b = inputs.make_batch(71, LENS, 2, 128, 128, mode=mode, n_slots=4)
    out, slots, cks = run(gdn, b, every, max_ckpts)
    assert check_checkpoints(b, cks, every, max_ckpts, TOL[torch.bfloat16]) > 0
    # outputs and slots: those of the plain call, bit for bit
    out0, slots0, _ = run(gdn, b, every, max_ckpts, ckpt=False)
    assert torch.equal(out.nan_to_num(7.0), out0.nan_to_num(7.0))
    assert torch.equal(slots.nan_to_num(7.0), slots0.nan_to_num(7.0))


@pytest.mark.parametrize("mode", ["gda", "kda"])
def test_checkpoints_with_a_long_tail(gdn, mode):
    # 70 slots: the last 70 tokens go through the recurrent kernel, which
    # writes the boundaries among them (L=257: 192 and 256; L=320: 256, 320)
    b = inputs.make_batch(76, [700, 257, 320, 30], 2, 128, 128, mode=mode, n_slots=70)
    _, _, cks = run(gdn, b, 64, 12)
    assert check_checkpoints(b, cks, 64, 12, TOL[torch.bfloat16]) == 10 + 4 + 5


@pytest.mark.parametrize("dtype,D", [(torch.float32, 128), (torch.bfloat16, 64)])
def test_checkpoints_token_loop_route(gdn, dtype, D):
    b = inputs.make_batch(72, [300, 130, 64, 5], 2, D, D, mode="gda", n_slots=3, dtype=dtype)
    _, _, cks = run(gdn, b, 64, 8)
    assert check_checkpoints(b, cks, 64, 8, TOL[dtype]) == 4 + 2 + 1


def test_tail_checkpoint_equals_slot(gdn):
    # L=257, 4 slots: slot j holds the state after 254 + j tokens, so
    # checkpoint 3 (after 256) is slot 2; L=320: checkpoint 4 is slot 3
    b = inputs.make_batch(73, [257, 320], 2, 128, 128, mode="gda", n_slots=4)
    _, slots, cks = run(gdn, b, 64, 5)
    assert torch.equal(cks[0, 3], slots[0, 2])
    assert torch.equal(cks[1, 4], slots[1, 3])


@pytest.mark.parametrize("mode", ["gda", "kda"])
def test_scan_checkpoints_ignore_later_tokens(gdn, mode):
    # cut every sequence to 256 + 4 tokens: the chunked part of both calls
    # covers tokens [0, 256) with the same chunks, so the checkpoints there
    # are the same bits
    b = inputs.make_batch(74, [700, 500, 300], 2, 128, 128, mode=mode, n_slots=4)
    _, _, full = run(gdn, b, 64, 4)
    keep = [260, 260, 260]
    idx = np.concatenate([np.arange(c, c + n) for c, n in
                          zip(b.cu_seqlens.numpy()[:-1], keep)])
    cut = inputs.GDNBatch(**{**b.__dict__,
                             "q": b.q[idx], "k": b.k[idx], "v": b.v[idx], "g": b.g[idx],
                             "beta": b.beta[idx],
                             "seq_len": torch.tensor(keep, dtype=torch.int64)})
    _, _, short = run(gdn, cut, 64, 4)
    assert torch.equal(full[:, :4], short[:, :4])


@pytest.mark.parametrize("mode", ["gda", "kda"])
def test_restart_from_selected_state(gdn, mode):
    n_slots, every, M = 4, 64, 6
    lens = [700, 257, 191, 320]
    b = inputs.make_batch(75, lens, 2, 128, 128, mode=mode, n_slots=n_slots)
    _, slots, cks = run(gdn, b, every, M)
    # keep counts that land on a slot, on a checkpoint, between checkpoints,
    # before the first checkpoint and past the last one
    n_keep = [450, 255, 130, 40]
    starts, seg_lo, seg_hi, sources = [], [], [], []
    for s, (L, nk) in enumerate(zip(lens, n_keep)):
        src, idx, rep = gdn.gdn_checkpoint_select(nk, L, n_slots, every, M)
        sources.append(src)
        if src == "slot":
            starts.append(slots[s, idx])
        elif src == "checkpoint":
            starts.append(cks[s, idx])
        else:
            starts.append(b.state[s].cuda())
        seg_lo.append(rep)
        seg_hi.append(nk)
    assert set(sources) >= {"checkpoint", "state_in"}
    # replay [replay_from, n_keep) of each sequence in one chunked call
    cu = b.cu_seqlens.numpy()
    idx = np.concatenate([np.arange(cu[s] + lo, cu[s] + hi) for s, (lo, hi)
                          in enumerate(zip(seg_lo, seg_hi))]).astype(np.int64)
    seg = np.asarray(seg_hi) - np.asarray(seg_lo)
    rb = inputs.GDNBatch(**{**b.__dict__,
                            "q": b.q[idx], "k": b.k[idx], "v": b.v[idx], "g": b.g[idx],
                            "beta": b.beta[idx],
                            "state": torch.stack([x.cpu() for x in starts]).contiguous(),
                            "seq_len": torch.from_numpy(seg)})
    _, rslots, _ = run(gdn, rb, every, 1, ckpt=False)
    got = rslots[:, -1].double().cpu().numpy()
    for s in range(len(lens)):  # nothing replayed: the start state is the answer
        if seg[s] == 0:
            got[s] = starts[s].double().cpu().numpy()
    ref = oracle_prefix_state(b, n_keep)
    e = rel_l2(got, ref)
    assert e <= TOL[torch.bfloat16], f"restarted state rel-L2 {e}"


@pytest.mark.parametrize("mode", ["gda", "kda"])
@pytest.mark.parametrize("qk_map", ["tiled", "grouped"])
def test_checkpoints_with_grouped_query_heads(gdn, mode, qk_map):
    # 4 value heads reading 2 q/k heads; boundaries in the scan and (L=257)
    # in the tail: 6 + 2 + 4 checkpoints reached
    b = inputs.make_batch(77, [400, 130, 257], 4, 128, 128, mode=mode, n_slots=4, H_qk=2,
                          qk_map=qk_map)
    _, _, cks = run(gdn, b, 64, 8)
    assert check_checkpoints(b, cks, 64, 8, TOL[torch.bfloat16]) == 6 + 2 + 4
