"""GPU parity of the gate reset, g = -inf, against the fp64 oracle.

A log-gate of -inf decays the state by exp(-inf) = 0 before the token's own
read and write: everything before that token is forgotten (the oracle pins
this in tests/test_oracle_pins.py). Every path must compute it, element by
element within the tolerance of its input dtype:
- gdn_forward (the recurrent kernel): decode (T = 1) and verify (T = 8),
  scalar (GDA) and per-row (KDA) gates, bf16 and fp32 inputs;
- gdn_forward_chunked, GDA, on the tensor-core route with resets on the first,
  a middle and the last row of a chunk, on the last row of a partial chunk,
  twice in one chunk, on a sequence's first token and inside the recurrent
  tail; and on the token-loop route (fp32 inputs);
- gdn_forward_chunked, KDA: the chunk form keeps per-row decays inside its
  operands and refuses a -inf gate in the chunked part with
  GDN_ERR_DEVICE_ARG (as documented); a reset inside the recurrent tail and
  the token-loop route are computed.
"""
import math

import numpy as np
import pytest
import torch

from gated_delta_net_02_gb300 import inputs

from _helpers import TOL, gpu_forward, oracle_run, rel_l2, to_dev

pytestmark = pytest.mark.gpu

NEG_INF = -math.inf


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_net_02_gb300 import build
    build.build()
    from gated_delta_net_02_gb300 import gdn as mod
    assert torch.cuda.is_available()
    return mod


def chunked_forward(gdn, b, check=True):
    d = to_dev(b)
    N, ntok = b.n_seqs, b.q.shape[0]
    H, Dk, Dv = b.v.shape[1], b.q.shape[2], b.v.shape[2]
    cu = b.cu_seqlens.to(torch.int32).cuda()
    shape = gdn.gdn_varlen_shape(N, ntok, H, Dk, Dv, gdn.dtype_code(b.q.dtype), b.scale)
    ws_bytes = gdn.gdn_chunked_workspace_size(shape, b.n_slots)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    slots = torch.full((N, b.n_slots, H, Dk, Dv), float("nan"), device="cuda")
    out = torch.full((ntok, H, Dv), float("nan"), device="cuda")
    ptrs = gdn.state_ptr_array(gdn.per_seq_state_ptrs(d["state"], N), "cuda")
    gdn.gdn_forward_chunked(shape, cu, d["q"], d["k"], d["v"], d["g"], d["beta"], ptrs, slots,
                            out, b.n_slots, b.mode, ws, ws_bytes)
    if check:
        gdn.gdn_check_device_error()
    return out, slots


def compare(b, out, slots, tol):
    o_ref, s_ref, sl_ref = oracle_run(b)
    out = out.double().cpu().numpy()
    slots = slots.double().cpu().numpy()
    assert np.isfinite(out).all(), "non-finite outputs"
    e_out = rel_l2(out, o_ref)
    e_fin = rel_l2(slots[:, -1], s_ref)
    assert e_out <= tol, f"out rel-L2 {e_out}"
    assert e_fin <= tol, f"final state rel-L2 {e_fin}"
    for j in range(b.n_slots):
        written = ~np.isnan(sl_ref[:, j, 0, 0, 0])
        if written.any():
            e = rel_l2(slots[written, j], sl_ref[written, j])
            assert e <= tol, f"slot {j} rel-L2 {e}"
    return e_out, e_fin


def set_resets(b, where):
    """g = -inf at (packed token, head) pairs; for KDA the whole gate row
    of that token and head unless a channel list is given."""
    for item in where:
        t, h = item[0], item[1]
        if b.mode == "gda":
            b.g[t, h] = NEG_INF
        else:
            ch = item[2] if len(item) > 2 else slice(None)
            b.g[t, h, ch] = NEG_INF
    return b


@pytest.mark.parametrize("mode", ["gda", "kda"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_step_reset(gdn, mode, dtype):
    # 8 sequences x 1 token: a reset in some (sequence, head) pairs; KDA also
    # resets only a few rows of one head
    b = inputs.make_batch(300, [1] * 8, 4, 128, 128, dtype=dtype, mode=mode, n_slots=1)
    where = [(0, 0), (3, 2), (7, 3)]
    if mode == "kda":
        where.append((5, 1, [0, 17, 127]))
    set_resets(b, where)
    out, slots = gpu_forward(b)
    compare(b, out, slots, TOL[dtype])


@pytest.mark.parametrize("mode", ["gda", "kda"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_verify_reset_first_middle_last_token(gdn, mode, dtype):
    # 6 sequences x T = 8 with K = 8 slots: resets on token 0, 3 and 7
    T = 8
    b = inputs.make_batch(301, [T] * 6, 4, 128, 128, dtype=dtype, mode=mode, n_slots=8)
    where = [(0 * T + 0, 0), (1 * T + 3, 1), (2 * T + 7, 2), (3 * T + 3, 3), (3 * T + 5, 3)]
    if mode == "kda":
        where.append((4 * T + 2, 0, list(range(0, 128, 5))))
    set_resets(b, where)
    out, slots = gpu_forward(b)
    compare(b, out, slots, TOL[dtype])


def chunk_positions(lens, K):
    """Resets for a batch of GDA sequences (packed tokens, head): first,
    middle and last row of the second chunk, the last row of a partial last
    chunk, two in one chunk, a sequence's first token, and one in the tail."""
    cu = np.concatenate([[0], np.cumsum(lens)])
    s0, s1 = int(cu[0]), int(cu[1])
    L1 = lens[1]
    last_partial = s1 + (L1 - K) - 1        # last chunked token of sequence 1
    return [(s0 + 64, 0), (s0 + 95, 1), (s0 + 127, 2), (s0 + 140, 3), (s0 + 150, 3),
            (s1 + 0, 0), (last_partial, 1), (s1 + L1 - 2, 2)]


def test_chunked_gda_tensor_core_route(gdn):
    lens, K = [300, 200, 130], 4
    assert (lens[1] - K) % 64 != 0          # sequence 1 ends on a partial chunk
    b = inputs.make_batch(302, lens, 4, 128, 128, mode="gda", n_slots=K)
    set_resets(b, chunk_positions(lens, K))
    out, slots = chunked_forward(gdn, b)
    e_out, e_fin = compare(b, out, slots, TOL[torch.bfloat16])
    print(f"gda reset, chunked: out {e_out:.2e}, state {e_fin:.2e}")


def test_chunked_gda_every_token_of_a_chunk_reset(gdn):
    # every gate of the second chunk is -inf: each row keeps only its own write
    b = inputs.make_batch(303, [260], 2, 128, 128, mode="gda", n_slots=2)
    b.g[64:128, 0] = NEG_INF
    out, slots = chunked_forward(gdn, b)
    compare(b, out, slots, TOL[torch.bfloat16])


def test_chunked_gda_token_loop_route(gdn):
    lens, K = [300, 200, 130], 4
    b = inputs.make_batch(304, lens, 4, 128, 128, dtype=torch.float32, mode="gda", n_slots=K)
    set_resets(b, chunk_positions(lens, K))
    out, slots = chunked_forward(gdn, b)
    compare(b, out, slots, TOL[torch.float32])


def test_chunked_kda_reset_in_chunk_part_refused(gdn):
    b = inputs.make_batch(305, [200], 2, 128, 128, mode="kda", n_slots=2)
    set_resets(b, [(70, 1, [3])])
    chunked_forward(gdn, b, check=False)
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_check_device_error()
    assert e.value.status == gdn.GDN_ERR_DEVICE_ARG
    gdn.gdn_check_device_error()   # the word was cleared


def test_chunked_kda_reset_in_tail_computed(gdn):
    # the last K tokens run through the recurrent kernel, which takes -inf
    K = 4
    b = inputs.make_batch(306, [200, 150], 2, 128, 128, mode="kda", n_slots=K)
    set_resets(b, [(198, 0), (200 + 147, 1, [0, 64])])
    out, slots = chunked_forward(gdn, b)
    compare(b, out, slots, TOL[torch.bfloat16])


def test_chunked_kda_token_loop_route(gdn):
    b = inputs.make_batch(307, [150, 70], 2, 128, 128, dtype=torch.float32, mode="kda",
                          n_slots=2)
    set_resets(b, [(64, 0), (100, 1, [5, 6, 7]), (150 + 3, 0)])
    out, slots = chunked_forward(gdn, b)
    compare(b, out, slots, TOL[torch.float32])
