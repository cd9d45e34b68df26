"""Host-side checks of the checkpointed prefill (no GPU needed): argument
validation of gdn_forward_chunked_checkpointed, and gdn_checkpoint_select
against a brute-force choice over every state that one call stores.

A call over a sequence of L tokens with n_slots slots and checkpoints every
E tokens (at most M of them) keeps the state after these token counts:
  - 0 (the call's input state, always available);
  - (m+1)*E for m < M with (m+1)*E <= L (checkpoint m);
  - L - n_slots + j + 1 >= 1 for slot j < n_slots (the snapshot slots).
To keep the first n_keep tokens, the cheapest restart is the stored state
with the largest count <= n_keep (fewest tokens to replay); when a slot and
a checkpoint hold the same count, the slot is chosen.
"""
import ctypes

import pytest


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_net_02_gb300 import build
    build.build()
    from gated_delta_net_02_gb300 import gdn as mod
    return mod


def stored_states(L, n_slots, E, M):
    """(count, source, index) of every state one call keeps."""
    states = [(0, "state_in", -1)]
    for m in range(M):
        if (m + 1) * E <= L:
            states.append(((m + 1) * E, "checkpoint", m))
    for j in range(n_slots):
        c = L - n_slots + j + 1
        if c >= 1:
            states.append((c, "slot", j))
    return states


def brute_force(n_keep, L, n_slots, E, M):
    rank = {"slot": 2, "checkpoint": 1, "state_in": 0}
    best = max((s for s in stored_states(L, n_slots, E, M) if s[0] <= n_keep),
               key=lambda s: (s[0], rank[s[1]]))
    return best[1], best[2], best[0]


@pytest.mark.parametrize("L", [0, 1, 5, 63, 64, 65, 130, 256, 300, 1000])
@pytest.mark.parametrize("n_slots", [1, 4, 8])
@pytest.mark.parametrize("E,M", [(64, 1), (64, 3), (128, 100), (192, 2)])
def test_select_matches_brute_force(gdn, L, n_slots, E, M):
    for n_keep in range(L + 1):
        got = gdn.gdn_checkpoint_select(n_keep, L, n_slots, E, M)
        assert got == brute_force(n_keep, L, n_slots, E, M), (n_keep, L, n_slots, E, M)


def test_select_replays_only_kept_tokens(gdn):
    # the restart state never lies past n_keep, and a slot restart replays nothing
    for n_keep in range(0, 500, 7):
        src, idx, rep = gdn.gdn_checkpoint_select(n_keep, 500, 8, 64, 5)
        assert 0 <= rep <= n_keep
        if src == "slot":
            assert rep == n_keep and 0 <= idx < 8
        elif src == "checkpoint":
            assert rep == (idx + 1) * 64 and idx < 5
        else:
            assert (idx, rep) == (-1, 0)


@pytest.mark.parametrize("args", [
    (5, 4, 1, 64, 1),     # n_keep > L
    (-1, 4, 1, 64, 1),    # negative n_keep
    (0, -1, 1, 64, 1),    # negative L
    (1, 4, 0, 64, 1),     # no slots
    (1, 4, 1, 0, 1),      # ckpt_every 0
    (1, 4, 1, 96, 1),     # not a chunk boundary
    (1, 4, 1, 64, 0),     # no checkpoints
])
def test_select_argument_errors(gdn, args):
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_checkpoint_select(*args)
    assert e.value.status == gdn.GDN_ERR_INVALID_ARG
    i = ctypes.c_int()
    assert gdn.lib.gdn_checkpoint_select(1, 4, 1, 64, 1, None, ctypes.byref(i),
                                         ctypes.byref(i)) == gdn.GDN_ERR_INVALID_ARG


FAKE = 1 << 20  # 16-byte aligned non-null address; never dereferenced here
FAR = 1 << 40   # far from FAKE: no overlap with the other buffers


def call_ckpt(gdn, sh, n_slots=1, ckpt=FAR, every=64, max_ckpts=2, **ptrs):
    p = dict(cu=FAKE, q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state_in=FAKE,
             state_slots=FAKE, out=FAKE, ws=FAKE)
    p.update(ptrs)
    ws_bytes = gdn.gdn_chunked_workspace_size(sh, n_slots)
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_forward_chunked_checkpointed(
            sh, p["cu"], p["q"], p["k"], p["v"], p["g"], p["beta"], p["state_in"],
            p["state_slots"], p["out"], n_slots, "gda", ckpt, every, max_ckpts, p["ws"],
            ws_bytes)
    return e.value.status, gdn.gdn_last_error()


def vshape(gdn, **kw):
    base = dict(n_seqs=2, total_tokens=100, H=2, D_k=128, D_v=128, in_dtype=gdn.GDN_BF16,
                scale=0.0)
    base.update(kw)
    return gdn.gdn_varlen_shape(**base)


def test_checkpointed_argument_errors(gdn):
    E = gdn.GDN_ERR_INVALID_ARG
    assert call_ckpt(gdn, vshape(gdn), ckpt=0)[0] == E
    assert call_ckpt(gdn, vshape(gdn), ckpt=FAR + 8)[0] == E
    assert call_ckpt(gdn, vshape(gdn), every=0)[0] == E
    assert call_ckpt(gdn, vshape(gdn), every=100)[0] == E
    assert call_ckpt(gdn, vshape(gdn), max_ckpts=0)[0] == E
    st, msg = call_ckpt(gdn, vshape(gdn), ckpt=FAKE)  # same address as the slots
    assert st == E and "overlap" in msg
    # the checks shared with gdn_forward_chunked, under this entry point's name
    st, msg = call_ckpt(gdn, vshape(gdn, D_k=32))
    assert st == gdn.GDN_ERR_UNSUPPORTED and "gdn_forward_chunked_checkpointed" in msg
    assert call_ckpt(gdn, vshape(gdn), cu=0)[0] == E
    assert call_ckpt(gdn, vshape(gdn), n_slots=0)[0] == E
