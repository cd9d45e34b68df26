"""Pins of the fp64 oracle against what the mathematics of the gated delta
rule fixes, independent of the oracle's own code.

Each test states a property that a plausible mistake in the oracle (a dropped
decay, a wrong sign, a transposed state, gating columns instead of rows, the
query reading the pre-write state, a slot off by one) would break. The
formulations used as references here (the transition-matrix form, the
chunked WY/UT form, orthonormal retrieval) are written independently of the
oracle's step-by-step loop.

Sources: the gated delta rule S_t = a_t (I - b_t k_t k_t^T) S_{t-1}
+ b_t k_t v_t^T of "Gated Delta Networks" (Yang, Kautz, Hatamizadeh, ICLR
2025, Eq. for the gated delta rule) and its chunkwise WY/UT form ("Parallelizing
Linear Transformers with the Delta Rule over Sequence Length", Yang et al.,
NeurIPS 2024, Sec. 3); gate modes GDA/KDA from "metal : add GDN kernel
(#20361)" (llama.cpp commits, tag b9752, src/models/qwen35.cpp); snapshot slots
and rollback from "metal: add GDN partial rollback" and "llama: allow partial
seq_rm for GDN models for speculative decoding" (koboldcpp commits, tag
v1.113.1).
"""
import numpy as np
import pytest

import oracle


def rng(seed):
    return np.random.default_rng(seed)


def unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def random_case(seed, T, H=2, Dk=8, Dv=6, mode="gda", N=1, s0_std=0.3):
    r = rng(seed)
    ntok = N * T
    q = unit_rows(r.standard_normal((ntok, H, Dk)))
    k = unit_rows(r.standard_normal((ntok, H, Dk)))
    v = r.standard_normal((ntok, H, Dv))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((ntok, H))))
    gshape = (ntok, H) if mode == "gda" else (ntok, H, Dk)
    g = -np.log1p(np.exp(r.standard_normal(gshape))) * (1.0 if mode == "gda" else 0.3)
    S0 = r.standard_normal((N, H, Dk, Dv)) * s0_std
    return q, k, v, g, beta, S0


def transition_form(q, k, v, g, beta, S0, scale, mode):
    """S_t = (I - b k k^T) Dg_t S_{t-1} + b k v^T with explicit matrices."""
    T, H, Dk = q.shape
    out = np.zeros((T, H, v.shape[2]))
    S_all = []
    for h in range(H):
        S = S0[h].copy()
        for t in range(T):
            kk = k[t, h][:, None]
            if mode == "gda":
                Dg = np.exp(g[t, h]) * np.eye(Dk)
            else:
                Dg = np.diag(np.exp(g[t, h]))
            S = (np.eye(Dk) - beta[t, h] * kk @ kk.T) @ Dg @ S \
                + beta[t, h] * kk @ v[t, h][None, :]
            out[t, h] = scale * S.T @ q[t, h]
        S_all.append(S)
    return out, np.stack(S_all)


def chunked_wy(q, k, v, g, beta, S0, scale, C, mode):
    """Chunkwise WY/UT form of one head (q,k [T,Dk], v [T,Dv], g [T] or
    [T,Dk], beta [T]); pairwise decays, explicit triangular solve."""
    T = q.shape[0]
    S = S0.copy()
    outs = []
    for c0 in range(0, T, C):
        Q, K, V, G, B = q[c0:c0 + C], k[c0:c0 + C], v[c0:c0 + C], g[c0:c0 + C], beta[c0:c0 + C]
        n = Q.shape[0]
        gam = np.cumsum(G, axis=0)
        low = np.tril(np.ones((n, n)), -1).astype(bool)
        lowd = np.tril(np.ones((n, n))).astype(bool)
        if mode == "kda":
            diff = gam[:, None, :] - gam[None, :, :]           # (r, j, i)
            diff = np.where(lowd[:, :, None], diff, -np.inf)
            Dr = np.exp(diff)
            KK = np.einsum("ri,ji,rji->rj", K, K, Dr)
            QK = np.einsum("ri,ji,rji->rj", Q, K, Dr)
            Kg = K * np.exp(gam)
            Qg = Q * np.exp(gam)
            Kt = K * np.exp(gam[-1][None, :] - gam)
            S_dec = np.exp(gam[-1])[:, None] * S
        else:
            diff = np.where(lowd, gam[:, None] - gam[None, :], -np.inf)
            Dr = np.exp(diff)
            KK = (K @ K.T) * Dr
            QK = (Q @ K.T) * Dr
            Kg = K * np.exp(gam)[:, None]
            Qg = Q * np.exp(gam)[:, None]
            Kt = K * np.exp(gam[-1] - gam)[:, None]
            S_dec = np.exp(gam[-1]) * S
        A = np.where(low, B[:, None] * KK, 0.0)
        Tm = np.linalg.solve(np.eye(n) + A, np.diag(B))
        W = Tm @ Kg
        U = Tm @ V
        D = U - W @ S
        P = np.where(lowd, QK, 0.0)
        outs.append(scale * (Qg @ S + P @ D))
        S = S_dec + Kt.T @ D
    return np.concatenate(outs), S


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# ---------------------------------------------------------------- single token

@pytest.mark.parametrize("mode", ["gda", "kda"])
def test_single_token_matrix_form(mode):
    q, k, v, g, beta, S0 = random_case(1, T=1, mode=mode)
    scale = 0.37
    out, S1, _ = oracle.forward(q, k, v, g, beta, S0, mode=mode, scale=scale)
    for h in range(q.shape[1]):
        kk = k[0, h][:, None]
        Dg = np.exp(g[0, h]) * np.eye(8) if mode == "gda" else np.diag(np.exp(g[0, h]))
        exp_S = (np.eye(8) - beta[0, h] * kk @ kk.T) @ Dg @ S0[0, h] + beta[0, h] * kk @ v[0, h][None]
        assert np.allclose(S1[0, h], exp_S, rtol=0, atol=1e-14)
        assert np.allclose(out[0, h], scale * exp_S.T @ q[0, h], rtol=0, atol=1e-14)


def test_single_token_zero_state_closed_form():
    # S0 = 0: o = scale * beta * (k . q) * v, independent of the gate
    q, k, v, g, beta, S0 = random_case(2, T=1)
    S0[:] = 0.0
    out, _, _ = oracle.forward(q, k, v, g, beta, S0, scale=0.5)
    for h in range(q.shape[1]):
        expect = 0.5 * beta[0, h] * np.dot(k[0, h], q[0, h]) * v[0, h]
        assert np.allclose(out[0, h], expect, rtol=1e-14, atol=1e-15)


def test_default_scale_is_inverse_sqrt_dk():
    q, k, v, g, beta, S0 = random_case(3, T=3, Dk=16)
    a, _, _ = oracle.forward(q, k, v, g, beta, S0)
    b, _, _ = oracle.forward(q, k, v, g, beta, S0, scale=0.25)
    assert np.array_equal(a, b)


# ------------------------------------------------------------ independent forms

@pytest.mark.parametrize("mode", ["gda", "kda"])
def test_transition_matrix_form(mode):
    q, k, v, g, beta, S0 = random_case(4, T=13, H=3, Dk=8, Dv=5, mode=mode)
    out, S, _ = oracle.forward(q, k, v, g, beta, S0, mode=mode, scale=0.3)
    out_ref, S_ref = transition_form(q, k, v, g, beta, S0[0], 0.3, mode)
    assert rel(out, out_ref) < 1e-13
    assert rel(S[0], S_ref) < 1e-13


@pytest.mark.parametrize("mode", ["gda", "kda"])
@pytest.mark.parametrize("C,T", [(4, 13), (8, 21), (64, 150), (64, 64)])
def test_chunked_wy_form_equals_token_loop(mode, C, T):
    Dk, Dv = (16, 12) if C < 64 else (32, 24)
    q, k, v, g, beta, S0 = random_case(5 + C + T, T=T, H=2, Dk=Dk, Dv=Dv, mode=mode)
    out, S, _ = oracle.forward(q, k, v, g, beta, S0, mode=mode, scale=0.2)
    for h in range(2):
        o_ref, S_ref = chunked_wy(q[:, h], k[:, h], v[:, h], g[:, h], beta[:, h],
                                  S0[0, h], 0.2, C, mode)
        assert rel(out[:, h], o_ref) < 1e-10
        assert rel(S[0, h], S_ref) < 1e-10


# ------------------------------------------------------------ read / write

def test_orthonormal_key_retrieval():
    # g = 0, beta = 1, S0 = 0, orthonormal keys: reading key i returns v_i
    r = rng(6)
    Dk, Dv, T = 64, 40, 16
    Qm, _ = np.linalg.qr(r.standard_normal((Dk, Dk)))
    keys = Qm[:, :T].T                                     # T orthonormal rows
    vals = r.standard_normal((T, Dv))
    # T write tokens, then T read tokens that write nothing (k = 0)
    q = np.concatenate([r.standard_normal((T, Dk)), keys])[:, None, :]
    k = np.concatenate([keys, np.zeros((T, Dk))])[:, None, :]
    v = np.concatenate([vals, r.standard_normal((T, Dv))])[:, None, :]
    g = np.zeros((2 * T, 1))
    beta = np.ones((2 * T, 1))
    S0 = np.zeros((1, 1, Dk, Dv))
    out, S, _ = oracle.forward(q, k, v, g, beta, S0, scale=1.0)
    assert np.abs(out[T:, 0] - vals).max() < 1e-13
    # the state is exactly sum_t k_t v_t^T
    assert np.abs(S[0, 0] - keys.T @ vals).max() < 1e-13


def test_delta_rule_overwrites_same_key():
    r = rng(7)
    Dk, Dv = 16, 8
    key = unit_rows(r.standard_normal(Dk))
    v1, v2 = r.standard_normal(Dv), r.standard_normal(Dv)
    q = np.stack([r.standard_normal(Dk), r.standard_normal(Dk), key])[:, None]
    k = np.stack([key, key, np.zeros(Dk)])[:, None]
    v = np.stack([v1, v2, np.zeros(Dv)])[:, None]
    g = np.zeros((3, 1))
    beta = np.ones((3, 1))
    S0 = r.standard_normal((1, 1, Dk, Dv))
    out, _, _ = oracle.forward(q, k, v, g, beta, S0, scale=1.0)
    assert np.abs(out[2, 0] - v2).max() < 1e-13


def test_query_reads_updated_state():
    # a token's own write is visible to its own query: with S0 = 0 and q = k
    # (unit), o = beta * v
    r = rng(8)
    k = unit_rows(r.standard_normal((1, 1, 8)))
    v = r.standard_normal((1, 1, 5))
    out, _, _ = oracle.forward(k.copy(), k, v, np.zeros((1, 1)), np.full((1, 1), 0.7),
                               np.zeros((1, 1, 8, 5)), scale=1.0)
    assert np.allclose(out[0, 0], 0.7 * v[0, 0], rtol=1e-14, atol=1e-15)


# ------------------------------------------------------------ gates

@pytest.mark.parametrize("mode", ["gda", "kda"])
def test_minus_infinity_gate_resets_state(mode):
    q, k, v, g, beta, S0 = random_case(9, T=12, mode=mode)
    t = 5
    g[t] = -np.inf
    out, S, _ = oracle.forward(q, k, v, g, beta, S0, mode=mode, scale=0.4)
    out2, S2, _ = oracle.forward(q[t:], k[t:], v[t:], np.where(np.isinf(g[t:]), 0.0, g[t:]),
                                 beta[t:], np.zeros_like(S0), mode=mode, scale=0.4)
    assert rel(out[t:], out2) < 1e-14
    assert rel(S, S2) < 1e-14


def test_zero_gate_zero_beta_keeps_state():
    q, k, v, g, beta, S0 = random_case(10, T=9)
    g[:] = 0.0
    beta[:] = 0.0
    out, S, _ = oracle.forward(q, k, v, g, beta, S0, scale=0.6)
    assert np.array_equal(S, S0)
    for t in range(9):
        for h in range(2):
            assert np.allclose(out[t, h], 0.6 * S0[0, h].T @ q[t, h], rtol=1e-14, atol=1e-15)


def test_kda_with_equal_rows_equals_gda_bitwise():
    q, k, v, g, beta, S0 = random_case(11, T=10, Dk=8)
    g_kda = np.repeat(g[:, :, None], 8, axis=2)
    a = oracle.forward(q, k, v, g, beta, S0, mode="gda", n_slots=3)
    b = oracle.forward(q, k, v, g_kda, beta, S0, mode="kda", n_slots=3)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_kda_gates_rows_not_columns():
    # a per-row gate of -inf on key rows R zeroes exactly those rows of S
    # before the read; it must equal a plain run from S0 with rows R zeroed
    q, k, v, g, beta, S0 = random_case(12, T=6, Dk=8, Dv=5, mode="kda")
    g[:] = 0.0
    rows = [1, 4, 6]
    g[0, :, rows] = -np.inf
    out, S, _ = oracle.forward(q, k, v, g, beta, S0, mode="kda", scale=0.3)
    S0z = S0.copy()
    S0z[:, :, rows, :] = 0.0
    out2, S2, _ = oracle.forward(q, k, v, np.zeros(g.shape[:2]), beta, S0z, mode="gda", scale=0.3)
    assert rel(out, out2) < 1e-14 and rel(S, S2) < 1e-14


# ------------------------------------------------------------ Householder

def test_householder_reflection_preserves_norm():
    q, k, v, g, beta, S0 = random_case(13, T=7)
    g[:] = 0.0
    beta[:] = 2.0
    v[:] = 0.0
    _, S, _ = oracle.forward(q, k, v, g, beta, S0)
    for h in range(2):
        assert abs(np.linalg.norm(S[0, h]) - np.linalg.norm(S0[0, h])) < 1e-13


def test_projection_removes_key_direction():
    q, k, v, g, beta, S0 = random_case(14, T=1)
    g[:] = 0.0
    beta[:] = 1.0
    v[:] = 0.0
    _, S, _ = oracle.forward(q, k, v, g, beta, S0)
    for h in range(2):
        assert np.abs(S[0, h].T @ k[0, h]).max() < 1e-14


# ------------------------------------------------------------ linearity

def test_linear_in_state_and_values():
    q, k, v, g, beta, S0 = random_case(15, T=11)
    _, _, v2, _, _, S02 = random_case(16, T=11)
    a, b = 0.7, -1.3
    o1, s1, _ = oracle.forward(q, k, v, g, beta, S0)
    o2, s2, _ = oracle.forward(q, k, v2, g, beta, S02)
    o3, s3, _ = oracle.forward(q, k, a * v + b * v2, g, beta, a * S0 + b * S02)
    assert rel(o3, a * o1 + b * o2) < 1e-12
    assert rel(s3, a * s1 + b * s2) < 1e-12


# ------------------------------------------------------------ slots / rollback

def test_single_slot_is_final_state_bitwise():
    q, k, v, g, beta, S0 = random_case(17, T=9, N=3)
    _, S, slots = oracle.forward(q, k, v, g, beta, S0, n_slots=1)
    assert np.array_equal(slots[:, 0], S)


@pytest.mark.parametrize("T,K", [(8, 8), (8, 3), (5, 1), (1, 1)])
def test_slots_equal_prefix_runs_bitwise(T, K):
    N = 2
    q, k, v, g, beta, S0 = random_case(18 + T + K, T=T, N=N)
    _, _, slots = oracle.forward(q, k, v, g, beta, S0, n_slots=K)
    for s in range(N):
        sl = slice(s * T, (s + 1) * T)
        for j in range(K):
            n = T - K + j + 1          # tokens consumed when slot j is written
            _, Sp, _ = oracle.forward(q[sl][:n], k[sl][:n], v[sl][:n], g[sl][:n],
                                      beta[sl][:n], S0[s:s + 1])
            assert np.array_equal(slots[s, j], Sp[0])


def test_short_sequence_leaves_leading_slots_untouched():
    q, k, v, g, beta, S0 = random_case(19, T=3)
    _, S, slots = oracle.forward(q, k, v, g, beta, S0, n_slots=5)
    assert np.isnan(slots[0, :2]).all()            # never written
    assert np.array_equal(slots[0, 4], S[0])       # last slot = final state


@pytest.mark.parametrize("T,K", [(8, 8), (8, 3), (4, 6)])
def test_rollback_selects_state_of_accepted_prefix(T, K):
    q, k, v, g, beta, S0 = random_case(20 + K, T=T)
    _, _, slots = oracle.forward(q, k, v, g, beta, S0, n_slots=K)
    for n in range(T + 1):
        _, Sp, _ = oracle.forward(q[:n], k[:n], v[:n], g[:n], beta[:n], S0) if n else (None, S0, None)
        if n > 0 and n - 1 < T - K:
            with pytest.raises(oracle.RollbackRangeError):
                oracle.rollback_slot(T, K, n)
            continue
        slot = oracle.rollback_slot(T, K, n)
        chosen = S0[0] if slot == -1 else slots[0, slot]
        assert np.array_equal(chosen, Sp[0])
    with pytest.raises(oracle.RollbackRangeError):
        oracle.rollback_slot(T, K, T + 1)
    with pytest.raises(oracle.RollbackRangeError):
        oracle.rollback_slot(T, K, -1)


# ------------------------------------------------------------ varlen / threads

def test_varlen_equals_separate_runs():
    r = rng(21)
    lens = [5, 1, 9, 3]
    H, Dk, Dv = 2, 8, 4
    ntok = sum(lens)
    q = unit_rows(r.standard_normal((ntok, H, Dk)))
    k = unit_rows(r.standard_normal((ntok, H, Dk)))
    v = r.standard_normal((ntok, H, Dv))
    g = -np.abs(r.standard_normal((ntok, H)))
    beta = r.uniform(0, 1, (ntok, H))
    S0 = r.standard_normal((4, H, Dk, Dv))
    start = np.cumsum([0] + lens[:-1])
    out, S, slots = oracle.forward(q, k, v, g, beta, S0, seq_start=start,
                                   seq_len=np.array(lens), n_slots=2)
    for s, (a, n) in enumerate(zip(start, lens)):
        o1, S1, sl1 = oracle.forward(q[a:a + n], k[a:a + n], v[a:a + n], g[a:a + n],
                                     beta[a:a + n], S0[s:s + 1], n_slots=2)
        assert np.array_equal(out[a:a + n], o1)
        assert np.array_equal(S[s], S1[0])
        assert np.array_equal(slots[s], sl1[0], equal_nan=True)


def test_thread_count_does_not_change_bits():
    q, k, v, g, beta, S0 = random_case(22, T=7, N=5, H=3)
    a = oracle.forward(q, k, v, g, beta, S0, n_slots=2, threads=1)
    b = oracle.forward(q, k, v, g, beta, S0, n_slots=2, threads=4)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_empty_sequence_returns_input_state():
    r = rng(23)
    S0 = r.standard_normal((2, 1, 4, 4))
    q = np.zeros((3, 1, 4)); k = np.zeros((3, 1, 4)); v = np.zeros((3, 1, 4))
    g = np.zeros((3, 1)); beta = np.zeros((3, 1))
    _, S, _ = oracle.forward(q, k, v, g, beta, S0, seq_start=np.array([0, 0]),
                             seq_len=np.array([0, 3]))
    assert np.array_equal(S[0], S0[0])


def test_grouped_query_head_maps():
    # tiled repeats the H_qk heads as a block, grouped repeats each head in place
    assert oracle.qk_head_index(6, 2, "tiled").tolist() == [0, 1, 0, 1, 0, 1]
    assert oracle.qk_head_index(6, 2, "grouped").tolist() == [0, 0, 0, 1, 1, 1]
    assert oracle.qk_head_index(4, 4, "grouped").tolist() == [0, 1, 2, 3]
    with pytest.raises(ValueError):
        oracle.qk_head_index(6, 4, "tiled")


@pytest.mark.parametrize("mode", ["gda", "kda"])
@pytest.mark.parametrize("qk_map,expand", [
    ("tiled", lambda x, r: np.tile(x, (1, r, 1))),     # the heads as a repeated block
    ("grouped", lambda x, r: np.repeat(x, r, axis=1)),  # each head repeated in place
])
def test_grouped_query_equals_explicitly_repeated_heads(mode, qk_map, expand):
    """Broadcasting H_qk q/k heads to H value heads equals running the plain
    op on q, k repeated to H heads by numpy's tile / repeat."""
    rng = np.random.default_rng(31)
    ntok, H, Hqk, Dk, Dv = 12, 6, 2, 16, 8
    q = rng.standard_normal((ntok, Hqk, Dk))
    k = rng.standard_normal((ntok, Hqk, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((ntok, H, Dv))
    g = -np.log1p(np.exp(rng.standard_normal((ntok, H, Dk) if mode == "kda" else (ntok, H))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((ntok, H))))
    S0 = 0.05 * rng.standard_normal((2, H, Dk, Dv))
    kw = dict(mode=mode, n_slots=2, seq_start=np.array([0, 7]), seq_len=np.array([7, 5]))
    o1, s1, sl1 = oracle.forward(q, k, v, g, beta, S0, qk_map=qk_map, **kw)
    o2, s2, sl2 = oracle.forward(expand(q, 3), expand(k, 3), v, g, beta, S0, **kw)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)
    assert np.array_equal(sl1, sl2, equal_nan=True)
    # and the two head orders really differ
    other = "grouped" if qk_map == "tiled" else "tiled"
    o3, _, _ = oracle.forward(q, k, v, g, beta, S0, qk_map=other, **kw)
    assert not np.allclose(o1, o3)
