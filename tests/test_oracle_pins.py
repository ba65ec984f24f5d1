"""Self-pins of the fp64 oracle against what the pages and the mathematics fix.

Each test ties one part of the oracle to something other than the oracle's own
formula: closed forms, brute-force dense products on tiny inputs, algebraic
invariants, special cases, and constants the pages print
(tests/golden/pages_constants.json).  A plausible mistake in the oracle (a
dropped term, a wrong sign or index, a transposed operand, an exclusive /
inclusive decay mix-up) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_constants.json")
G_MIN = -5.0


def rnd_inputs(T, H, dk, dv, seed, z_mean=0.0, z_std=1.0, beta_mean=0.0, A_std=0.5):
    r = np.random.default_rng(seed)
    q = r.standard_normal((T, H, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = r.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((T, H, dv))
    z = z_mean + z_std * r.standard_normal((T, H, dk))
    A = A_std * r.standard_normal(H)
    beta = 1.0 / (1.0 + np.exp(-(beta_mean + r.standard_normal((T, H)))))
    return q, k, v, z, A, beta


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# ---------------------------------------------------------------- gate (P10)

def test_gate_special_values_and_symmetry():
    # z = 0: sigmoid(0) = 1/2 exactly, for every A.
    for A in (-1.0, 0.0, 0.7):
        assert oracle._load().oracle_gate(G_MIN, A, 0.0) == G_MIN / 2
    # sigmoid(x) + sigmoid(-x) = 1  ->  g(z) + g(-z) = g_min.
    for z in (0.3, 1.7, -2.2, 6.0):
        s = oracle._load().oracle_gate(G_MIN, 0.4, z) + oracle._load().oracle_gate(G_MIN, 0.4, -z)
        assert abs(s - G_MIN) < 1e-14
    # A only rescales the abscissa: g(A, z) = g(0, e^A z).
    for A, z in ((0.5, 1.3), (-0.8, -2.0)):
        assert abs(oracle._load().oracle_gate(G_MIN, A, z)
                   - oracle._load().oracle_gate(G_MIN, 0.0, math.exp(A) * z)) < 1e-14
    # slope at 0 is g_min * e^A / 4 (sigmoid'(0) = 1/4), sign and scale pinned.
    A, h = 0.3, 1e-6
    d = (oracle._load().oracle_gate(G_MIN, A, h) - oracle._load().oracle_gate(G_MIN, A, -h)) / (2 * h)
    assert abs(d - G_MIN * math.exp(A) / 4) < 1e-8


def test_gate_bounds_match_pages():
    gold = json.load(open(GOLDEN))
    g_min = gold["gate_lower_bound"]["value"]
    z = np.linspace(-30, 30, 2001).reshape(1, 1, -1)
    g = oracle.gate(z, np.array([0.0]), g_min)
    assert np.all(g < 0) and np.all(g > g_min)
    assert np.all(np.diff(g.ravel()) <= 0)  # decreasing in z
    # limits: z -> +inf pins to g_min, z -> -inf pins to 0
    assert abs(oracle.gate(np.full((1, 1, 1), 60.0), np.array([0.0]), g_min)[0, 0, 0] - g_min) < 1e-12
    assert abs(oracle.gate(np.full((1, 1, 1), -60.0), np.array([0.0]), g_min)[0, 0, 0]) < 1e-12
    # fastest forgetting: alpha > e^{g_min} ~ 0.67 % per step (printed on the page)
    m = gold["min_alpha_per_step"]
    assert abs(math.exp(g_min) - m["value"]) / m["value"] < m["rel_tol"]
    # 16-token sub-tile: accumulated log decay > 16 * g_min = -80, e^80 ~ 5.5e34 < bf16 max
    n = gold["subtile_tokens"]["value"]
    assert n * g_min == gold["subtile_log_decay_bound"]["value"]
    e80 = gold["exp80"]
    assert abs(math.exp(-n * g_min) - e80["value"]) / e80["value"] < e80["rel_tol"]
    assert math.exp(-n * g_min) < gold["bf16_max"]["value"]


# ---------------------------------------------------------------- P1: beta = 0

def test_beta_zero_is_pure_channel_decay():
    T, H, dk, dv = 37, 2, 16, 12
    q, k, v, z, A, beta = rnd_inputs(T, H, dk, dv, 1)
    beta[:] = 0.0
    S0 = np.random.default_rng(2).standard_normal((1, H, dk, dv))
    o, fin = oracle.recurrent(q, k, v, z, A, beta, init_state=S0)
    g = oracle.gate(z, A)
    cum = np.cumsum(g, axis=0)  # [T, H, dk], inclusive
    for h in range(H):
        for t in range(T):
            St = np.exp(cum[t, h])[:, None] * S0[0, h]
            assert rel(o[t, h], St.T @ q[t, h]) < 1e-12
        assert rel(fin[0, h], np.exp(cum[-1, h])[:, None] * S0[0, h]) < 1e-12


# ---------------------------------------------------------------- P2: brute force, T <= 16

@pytest.mark.parametrize("T", [1, 5, 16])
def test_recurrence_equals_dense_transition_products(T):
    H, dk, dv = 2, 8, 6
    q, k, v, z, A, beta = rnd_inputs(T, H, dk, dv, 10 + T)
    S0 = np.random.default_rng(3).standard_normal((1, H, dk, dv))
    o, fin = oracle.recurrent(q, k, v, z, A, beta, init_state=S0)
    for h in range(H):
        Ms = oracle.transition_matrices(k, z, A, beta, h)
        S = S0[0, h].copy()
        for t in range(T):
            S = Ms[t] @ S + beta[t, h] * np.outer(k[t, h], v[t, h])  # eq. (1), dense
            assert rel(o[t, h], S.T @ q[t, h]) < 1e-12
        P, Hm = oracle.brute_P_H(k, v, z, A, beta, h)
        assert rel(fin[0, h], P @ S0[0, h] + Hm) < 1e-12
        assert rel(S, fin[0, h]) < 1e-12


@pytest.mark.parametrize("T", [2, 7, 16])
def test_wy_and_ut_match_brute_force(T):
    """WY (P = Diag(gamma) - sum Diag(gamma^{i->r}) k w^T, H = sum Diag(..) k u^T) and the
    UT transform M = (I + StrictTril(Diag(beta)(Gamma.K)(K/Gamma)^T))^-1 Diag(beta),
    W = M (Gamma.K), U = M V, against dense products.  The decay between i and r is
    gamma^r / gamma^i; the inclusive reading (gamma^r / gamma^{i-1}) fails here."""
    H, dk, dv = 1, 8, 5
    q, k, v, z, A, beta = rnd_inputs(T, H, dk, dv, 20 + T)
    h = 0
    w, u, gam, Gc = oracle.wy_vectors(k, v, z, A, beta, h)
    P, Hm = oracle.brute_P_H(k, v, z, A, beta, h)
    Pw = np.diag(gam[-1]).copy()
    Hw = np.zeros((dk, dv))
    for i in range(T):
        d = np.exp(Gc[-1] - Gc[i])
        Pw -= np.outer(d * k[i, h], w[i])
        Hw += np.outer(d * k[i, h], u[i])
    assert rel(Pw, P) < 1e-12
    assert rel(Hw, Hm) < 1e-12
    # UT transform
    GK = gam * k[:, h]
    KG = k[:, h] / gam
    Lm = np.tril(np.diag(beta[:, h]) @ GK @ KG.T, -1)
    M = np.linalg.solve(np.eye(T) + Lm, np.diag(beta[:, h]))
    assert rel(M @ GK, w) < 1e-12
    assert rel(M @ v[:, h], u) < 1e-12


# ---------------------------------------------------------------- P3: chunk form == recurrence

@pytest.mark.parametrize("C", [16, 32, 64])
def test_chunk_form_equals_recurrence(C):
    T, H, dk, dv = 203, 2, 32, 24
    q, k, v, z, A, beta = rnd_inputs(T, H, dk, dv, 30 + C)
    cu = np.array([0, 70, 71, 203])  # includes a one-token document
    S0 = 0.1 * np.random.default_rng(4).standard_normal((3, H, dk, dv))
    o_r, f_r = oracle.recurrent(q, k, v, z, A, beta, cu_seqlens=cu, init_state=S0)
    o_c, f_c = oracle.chunk_form(q, k, v, z, A, beta, C, cu_seqlens=cu, init_state=S0)
    assert rel(o_c, o_r) < 1e-12
    assert rel(f_c, f_r) < 1e-12


def test_chunk_form_strong_gate_range():
    """Gate near its lower bound over a whole 64-token chunk: |G| up to 320, still exact in fp64."""
    T, H, dk, dv = 128, 1, 16, 16
    q, k, v, z, A, beta = rnd_inputs(T, H, dk, dv, 5, z_mean=8.0)
    o_r, f_r = oracle.recurrent(q, k, v, z, A, beta)
    o_c, f_c = oracle.chunk_form(q, k, v, z, A, beta, 64)
    assert rel(o_c, o_r) < 1e-11
    assert rel(f_c, f_r) < 1e-11


# ---------------------------------------------------------------- P4: eq. (17) composition

def _stress(T, H, dk, dv, seed):
    # slow decay (z ~ N(-10, 1): g ~ -2e-4) and small beta keep M far from zero
    return rnd_inputs(T, H, dk, dv, seed, z_mean=-10.0, beta_mean=-4.0)


@pytest.mark.parametrize("stress", [False, True])
def test_segment_composition_equals_unsplit(stress):
    T, H, dk, dv = 300, 2, 16, 12
    gen = _stress if stress else (lambda *a: rnd_inputs(*a))
    q, k, v, z, A, beta = gen(T, H, dk, dv, 40)
    S0 = np.random.default_rng(5).standard_normal((1, H, dk, dv))
    o_ref, f_ref = oracle.recurrent(q, k, v, z, A, beta, init_state=S0)
    cuts = [0, 64, 77, 200, 300]
    for h in range(H):
        S = S0[0, h]
        for a, b in zip(cuts[:-1], cuts[1:]):
            M, St = oracle.pair(k, v, z, A, beta, a, b, h)
            # matrix-free check of M: the recurrence from X with v = 0 gives M X
            X = np.random.default_rng(a).standard_normal((1, 1, dk, dv))
            _, fx = oracle.recurrent(q[a:b, h:h + 1], k[a:b, h:h + 1], np.zeros((b - a, 1, dv)),
                                     z[a:b, h:h + 1], A[h:h + 1], beta[a:b, h:h + 1], init_state=X)
            assert rel(M @ X[0, 0], fx[0, 0]) < 1e-12
            S_next = M @ S + St
            if stress:
                # non-vacuous: the carried-in part is a large share of the exit state
                assert np.linalg.norm(M @ S) / np.linalg.norm(S_next) > 0.1
            # re-running the segment from the composed entering state reproduces o
            o_seg, f_seg = oracle.recurrent(q[a:b, h:h + 1], k[a:b, h:h + 1], v[a:b, h:h + 1],
                                            z[a:b, h:h + 1], A[h:h + 1], beta[a:b, h:h + 1],
                                            init_state=S[None, None])
            assert rel(o_seg[:, 0], o_ref[a:b, h]) < 1e-11
            S = S_next
        assert rel(S, f_ref[0, h]) < 1e-11


def test_composition_associative_not_commutative():
    r = np.random.default_rng(6)
    dk, dv = 8, 5
    ps = [(r.standard_normal((dk, dk)), r.standard_normal((dk, dv))) for _ in range(3)]
    (M1, S1), (M2, S2), (M3, S3) = ps
    a = oracle.compose(*oracle.compose(M3, S3, M2, S2), M1, S1)
    b = oracle.compose(M3, S3, *oracle.compose(M2, S2, M1, S1))
    assert rel(a[0], b[0]) < 1e-13 and rel(a[1], b[1]) < 1e-13
    c = oracle.compose(M1, S1, M2, S2)
    d = oracle.compose(M2, S2, M1, S1)
    assert rel(c[1], d[1]) > 1e-3
    # the page's formula, written out: (M2 M1, M2 S1 + S2)
    assert rel(d[0], M2 @ M1) < 1e-14 and rel(d[1], M2 @ S1 + S2) < 1e-14


def test_linear_attention_limit_is_addition():
    """M = I (plain linear attention): composition adds and commutes ([K3-7] step 2)."""
    r = np.random.default_rng(7)
    dk, dv = 6, 4
    S1, S2 = r.standard_normal((dk, dv)), r.standard_normal((dk, dv))
    I = np.eye(dk)
    a = oracle.compose(I, S2, I, S1)
    b = oracle.compose(I, S1, I, S2)
    assert rel(a[1], S1 + S2) < 1e-15 and rel(a[1], b[1]) < 1e-15


def test_identity_pair_when_nothing_happens():
    """beta = 0 and alpha -> 1 (z = -50): the pair is (I, 0), the unit of composition."""
    T, H, dk, dv = 40, 1, 8, 8
    q, k, v, z, A, beta = rnd_inputs(T, H, dk, dv, 8)
    z[:] = -50.0
    A[:] = 0.0
    beta[:] = 0.0
    M, St = oracle.pair(k, v, z, A, beta, 0, T, 0)
    assert np.array_equal(M, np.eye(dk)) and np.all(St == 0)


def test_document_start_inside_segment_resets_pair():
    T, H, dk, dv = 120, 1, 8, 8
    q, k, v, z, A, beta = rnd_inputs(T, H, dk, dv, 9)
    cu = np.array([0, 50, 120])
    init = np.random.default_rng(10).standard_normal((2, H, dk, dv))
    M, St = oracle.pair(k, v, z, A, beta, 30, 120, 0, cu_seqlens=cu, init_state=init)
    assert np.all(M == 0)
    _, f = oracle.recurrent(q, k, v, z, A, beta, cu_seqlens=cu, init_state=init)
    assert rel(St, f[1, 0]) < 1e-12


# ---------------------------------------------------------------- P5: delta rule exactness

def test_delta_rule_recalls_orthonormal_keys():
    T, H, dk, dv = 24, 1, 32, 10
    r = np.random.default_rng(11)
    Qm, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    k = Qm[:, :T].T.reshape(T, 1, dk).copy()
    k[20, 0] = k[3, 0]  # a repeated key overwrites its slot
    v = r.standard_normal((T, H, dv))
    q = k.copy()
    z = np.full((T, H, dk), -50.0)  # alpha = 1 to double precision
    A = np.zeros(H)
    beta = np.ones((T, H))
    o, fin = oracle.recurrent(q, k, v, z, A, beta)
    S = fin[0, 0]
    for j in range(T):
        expect = v[20, 0] if j == 3 else v[j, 0]
        assert rel(S.T @ k[j, 0], expect) < 1e-12
        assert rel(o[j, 0], v[j, 0]) < 1e-12  # the token reads its own write


# ---------------------------------------------------------------- P7 / P8: linearity, resume, varlen

def test_linearity_in_values_and_state():
    T, H, dk, dv = 90, 2, 16, 8
    q, k, v, z, A, beta = rnd_inputs(T, H, dk, dv, 12)
    r = np.random.default_rng(13)
    v2 = r.standard_normal(v.shape)
    S1 = r.standard_normal((1, H, dk, dv))
    S2 = r.standard_normal((1, H, dk, dv))
    o1, f1 = oracle.recurrent(q, k, v, z, A, beta, init_state=S1)
    o2, f2 = oracle.recurrent(q, k, v2, z, A, beta, init_state=S2)
    o3, f3 = oracle.recurrent(q, k, v + v2, z, A, beta, init_state=S1 + S2)
    assert rel(o3, o1 + o2) < 1e-12 and rel(f3, f1 + f2) < 1e-12
    o4, f4 = oracle.recurrent(q, k, 2.5 * v, z, A, beta, init_state=2.5 * S1)
    assert rel(o4, 2.5 * o1) < 1e-13 and rel(f4, 2.5 * f1) < 1e-13


def test_resume_and_packed_documents():
    T, H, dk, dv = 150, 2, 16, 8
    q, k, v, z, A, beta = rnd_inputs(T, H, dk, dv, 14)
    S0 = np.random.default_rng(15).standard_normal((1, H, dk, dv))
    o, f = oracle.recurrent(q, k, v, z, A, beta, init_state=S0)
    t = 61
    oa, fa = oracle.recurrent(q[:t], k[:t], v[:t], z[:t], A, beta[:t], init_state=S0)
    ob, fb = oracle.recurrent(q[t:], k[t:], v[t:], z[t:], A, beta[t:], init_state=fa)
    assert rel(np.concatenate([oa, ob]), o) < 1e-13 and rel(fb, f) < 1e-13
    # packed = separate runs with their own initial states
    cu = np.array([0, 40, 41, 150])
    S = np.random.default_rng(16).standard_normal((3, H, dk, dv))
    op, fp = oracle.recurrent(q, k, v, z, A, beta, cu_seqlens=cu, init_state=S)
    for d in range(3):
        a, b = cu[d], cu[d + 1]
        od, fd = oracle.recurrent(q[a:b], k[a:b], v[a:b], z[a:b], A, beta[a:b],
                                  init_state=S[d:d + 1])
        assert rel(op[a:b], od) < 1e-14 and rel(fp[d], fd[0]) < 1e-14


def test_empty_document_keeps_initial_state():
    T, H, dk, dv = 20, 1, 8, 8
    q, k, v, z, A, beta = rnd_inputs(T, H, dk, dv, 17)
    cu = np.array([0, 10, 10, 20])
    S = np.random.default_rng(18).standard_normal((3, H, dk, dv))
    _, fp = oracle.recurrent(q, k, v, z, A, beta, cu_seqlens=cu, init_state=S)
    assert np.array_equal(fp[1], S[1])


# ---------------------------------------------------------------- P9: decode replay

def test_decode_replay_equals_committed_stream():
    N, W, H, dk, dv = 5, 5, 2, 16, 8
    r = np.random.default_rng(19)

    def window():
        q = r.standard_normal((N, W, H, dk))
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k = r.standard_normal((N, W, H, dk))
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        return (q, k, r.standard_normal((N, W, H, dv)), r.standard_normal((N, W, H, dk)),
                1 / (1 + np.exp(-r.standard_normal((N, W, H)))))

    A = 0.3 * r.standard_normal(H)
    S0 = 0.05 * r.standard_normal((N, H, dk, dv))
    cache = (np.zeros((N, W - 1, H, dk)), np.zeros((N, W - 1, H, dk)), np.zeros((N, W - 1, H, dv)),
             np.zeros((N, W - 1, H, dk)), np.zeros((N, W - 1, H)))
    w1 = window()
    o1, S1, cache = oracle.decode_step(S0, *w1, A, *cache, num_accepted=None)
    w2 = window()
    nacc = np.array([0, 4, 2, 1, 3])
    o2, S2, cache2 = oracle.decode_step(S1, *w2, A, *cache, num_accepted=nacc)
    for b in range(N):
        n = nacc[b]
        # committed stream: t0 of window 1, its first n drafts, t0 of window 2
        idx1 = list(range(0, n + 1))
        seqs = [np.concatenate([w1[i][b, idx1], w2[i][b, :1]]) for i in range(5)]
        # then the speculative drafts of window 2
        seqs = [np.concatenate([s, w2[i][b, 1:]]) for s, i in zip(seqs, range(5))]
        q, k, v, z, beta = seqs
        o_ref, _ = oracle.recurrent(q, k, v, z, A, beta, init_state=S0[b:b + 1])
        # committed state = recurrence over t0(1), d1..dn(1), t0(2)
        _, f_ref = oracle.recurrent(q[:n + 2], k[:n + 2], v[:n + 2], z[:n + 2], A, beta[:n + 2],
                                    init_state=S0[b:b + 1])
        assert rel(S2[b], f_ref[0]) < 1e-12
        # window-2 outputs: t0 then drafts continue the committed stream
        assert rel(o2[b], o_ref[n + 1:]) < 1e-12
        # window-1 outputs: t0 and all drafts in order
        o1_ref, _ = oracle.recurrent(w1[0][b], w1[1][b], w1[2][b], w1[3][b], A, w1[4][b],
                                     init_state=S0[b:b + 1])
        assert rel(o1[b], o1_ref) < 1e-12
    # the cache now holds window 2's drafts
    assert np.array_equal(cache2[1], w2[1][:, 1:])


def test_decode_replay_equals_snapshot_rollback():
    """Replaying the accepted prefix equals keeping a state snapshot after every draft and
    rolling back to the one at the accepted length ([K3-7] decode paragraph)."""
    N, W, H, dk, dv = 3, 5, 1, 8, 8
    r = np.random.default_rng(21)
    q = r.standard_normal((N, W, H, dk)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = r.standard_normal((N, W, H, dk)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((N, W, H, dv)); z = r.standard_normal((N, W, H, dk))
    beta = 1 / (1 + np.exp(-r.standard_normal((N, W, H))))
    A = np.zeros(H)
    S0 = r.standard_normal((N, H, dk, dv))
    empty = (np.zeros((N, W - 1, H, dk)),) * 2 + (np.zeros((N, W - 1, H, dv)),
                                                  np.zeros((N, W - 1, H, dk)), np.zeros((N, W - 1, H)))
    _, S1, cache = oracle.decode_step(S0, q, k, v, z, beta, A, *empty)
    nacc = np.array([4, 0, 2])
    w2 = [x.copy() for x in (q, k, v, z, beta)]
    _, S2, _ = oracle.decode_step(S1, *w2, A, *cache, num_accepted=nacc)
    for b in range(N):
        snaps = [S1[b]]
        for j in range(1, W):
            _, f = oracle.recurrent(q[b, j:j + 1], k[b, j:j + 1], v[b, j:j + 1], z[b, j:j + 1], A,
                                    beta[b, j:j + 1], init_state=snaps[-1][None])
            snaps.append(f[0])
        _, f = oracle.recurrent(w2[0][b, :1], w2[1][b, :1], w2[2][b, :1], w2[3][b, :1], A,
                                w2[4][b, :1], init_state=snaps[nacc[b]][None])
        assert rel(S2[b], f[0]) < 1e-13


# ---------------------------------------------------------------- in-kernel input options

def test_input_prep_l2norm_closed_forms():
    r = np.random.default_rng(11)
    q = r.standard_normal((5, 3, 128)) * 3.0
    k = r.standard_normal((5, 3, 128)) * 0.2
    qn, kn, _ = oracle.input_prep(q, k, np.zeros((5, 3)), qk_l2norm=True)
    # unit rows (up to the eps under the root), same directions
    assert np.allclose(np.linalg.norm(qn, axis=-1), 1.0, atol=1e-6)
    assert np.allclose(np.linalg.norm(kn, axis=-1), 1.0, atol=1e-4)
    assert np.allclose(qn * np.linalg.norm(q, axis=-1, keepdims=True), q, atol=1e-6)
    # scale invariance over the key dimension only (a norm over the wrong axis breaks it)
    qs, _, _ = oracle.input_prep(q * np.arange(1, 6).reshape(5, 1, 1), k, np.zeros((5, 3)), qk_l2norm=True)
    assert np.allclose(qs, qn, atol=1e-9)
    # eps sits under the root: a row of squared norm eps comes out with norm 1/sqrt(2)
    e = oracle.L2NORM_EPS
    tiny = np.zeros((1, 1, 128))
    tiny[0, 0, 7] = math.sqrt(e)
    t, _, _ = oracle.input_prep(tiny, tiny, np.zeros((1, 1)), qk_l2norm=True)
    assert abs(np.linalg.norm(t) - 1 / math.sqrt(2)) < 1e-12
    # the zero row stays zero; flags off leave everything unchanged
    z0, _, _ = oracle.input_prep(np.zeros((1, 1, 128)), tiny, np.zeros((1, 1)), qk_l2norm=True)
    assert not z0.any()
    q2, k2, b2 = oracle.input_prep(q, k, np.ones((5, 3)))
    assert np.array_equal(q2, q) and np.array_equal(k2, k) and np.array_equal(b2, np.ones((5, 3)))


def test_input_prep_q_scale_closed_forms():
    """q times dk^-1/2 = 1/sqrt(128) = 0.08838834764831845 (a closed value), after the
    L2 norm (so a normalised q has norm 1/sqrt(128)); k and beta untouched; and, o
    being linear in q, the recurrence's outputs scale by the same factor while the
    state does not change."""
    r = np.random.default_rng(12)
    q = r.standard_normal((6, 2, 128)) * 2.0
    k = r.standard_normal((6, 2, 128))
    b = r.random((6, 2))
    qs, ks, bs = oracle.input_prep(q, k, b, q_scale=True)
    assert abs(1.0 / math.sqrt(128) - 0.08838834764831845) < 1e-16
    assert np.allclose(qs, q * 0.08838834764831845, rtol=1e-15, atol=0)
    assert np.array_equal(ks, k) and np.array_equal(bs, b)
    qn, _, _ = oracle.input_prep(q, k, b, qk_l2norm=True, q_scale=True)
    assert np.allclose(np.linalg.norm(qn, axis=-1), 0.08838834764831845, rtol=1e-6)
    v, z = r.standard_normal((6, 2, 128)), r.standard_normal((6, 2, 128))
    A = np.zeros(2)
    o1, s1 = oracle.recurrent(q, k, v, z, A, b)
    o2, s2 = oracle.recurrent(qs, k, v, z, A, b)
    assert np.allclose(o2, o1 * 0.08838834764831845, rtol=1e-12, atol=1e-14)
    assert np.array_equal(s1, s2)


def test_input_prep_beta_sigmoid_closed_forms():
    x = np.array([[-30.0, -2.0, 0.0, 0.5, 3.0, 30.0]])
    _, _, b = oracle.input_prep(np.zeros((1, 1, 4)), np.zeros((1, 1, 4)), x, beta_sigmoid=True)
    assert b[0, 2] == 0.5
    assert np.allclose(b + oracle.input_prep(np.zeros((1, 1, 4)), np.zeros((1, 1, 4)), -x, beta_sigmoid=True)[2], 1.0)
    assert abs(b[0, 4] - 1 / (1 + math.exp(-3.0))) < 1e-15
    assert 0 < b[0, 0] < 1e-12 and 1 - b[0, 5] < 1e-12


# ---------------------------------------------------------------- fused decode step

def test_short_conv_equals_numpy_convolve():
    """The depthwise causal convolution against numpy's discrete convolution per channel."""
    r = np.random.default_rng(31)
    C, n = 6, 9
    hist, x, w = r.standard_normal((3, C)), r.standard_normal((n, C)), r.standard_normal((C, 4))
    y = oracle.short_conv(hist, x, w)
    s = np.concatenate([hist, x])
    for c in range(C):
        # numpy flips its second operand: reversed taps give tap 3 on the current token
        assert np.allclose(y[:, c], np.convolve(s[:, c], w[c, ::-1], mode="valid"), rtol=0, atol=1e-13)
    # causal: a later input leaves earlier outputs unchanged
    x2 = x.copy()
    x2[5] += 1.0
    y2 = oracle.short_conv(hist, x2, w)
    assert np.array_equal(y2[:5], y[:5]) and not np.allclose(y2[5], y[5])
    # a unit impulse on the last tap copies the input; on the first, the input three tokens back
    e = np.zeros((C, 4))
    e[:, 3] = 1.0
    assert np.array_equal(oracle.short_conv(hist, x, e), x)
    e = np.zeros((C, 4))
    e[:, 0] = 1.0
    assert np.array_equal(oracle.short_conv(hist, x, e), s[:n])


def test_short_conv_silu_closed_forms():
    """SiLU option: silu(0) = 0, silu(y) - silu(-y) = y, silu(1) = 1 / (1 + 1/e)."""
    C = 4
    e = np.zeros((C, 4))
    e[:, 3] = 1.0
    x = np.array([[0.0, 1.0, -2.5, 7.0]])
    hist = np.zeros((3, C))
    yp = oracle.short_conv(hist, x, e, silu=True)
    ym = oracle.short_conv(hist, -x, e, silu=True)
    assert yp[0, 0] == 0.0
    assert np.allclose(yp - ym, x, rtol=0, atol=1e-14)
    assert abs(yp[0, 1] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert 0 < -ym[0, 3] < 7.0 * 1e-3  # large negative inputs are nearly cut off


def test_gated_output_norm_invariants():
    """o / rms(o) * w * sigmoid(gate) per (token, head): unit RMS with w = 1 and gate = 0 (up
    to the factor 1/2), direction kept, scale invariance, gate odds e^g, eps under the root."""
    r = np.random.default_rng(33)
    o = r.standard_normal((5, 3, 32)) * 4.0
    one = np.ones(32)
    zero = np.zeros((5, 3, 32))
    y = oracle.rms_norm_gated(o, zero, one, 0.0) * 2.0
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, atol=1e-13)
    ratio = y / o
    assert np.allclose(ratio, ratio[..., :1], rtol=1e-12) and (ratio > 0).all()
    assert np.allclose(oracle.rms_norm_gated(o * 17.0, zero, one, 0.0), y / 2.0, rtol=1e-13)
    # per-row scaling: the norm is over the d_v channels of one (token, head) only
    sc = r.uniform(0.1, 10.0, (5, 3, 1))
    assert np.allclose(oracle.rms_norm_gated(o * sc, zero, one, 0.0), y / 2.0, rtol=1e-12)
    w = r.uniform(0.5, 1.5, 32)
    assert np.allclose(oracle.rms_norm_gated(o, zero, w, 0.0), y / 2.0 * w, rtol=1e-13)
    g = r.standard_normal((5, 3, 32))
    odds = oracle.rms_norm_gated(o, g, one, 0.0) / oracle.rms_norm_gated(o, -g, one, 0.0)
    assert np.allclose(odds, np.exp(g), rtol=1e-12)
    row = np.zeros((1, 1, 32))
    row[0, 0, 3] = math.sqrt(32 * 1e-3)  # mean square 1e-3
    t = oracle.rms_norm_gated(row, np.zeros((1, 1, 32)), one, 1e-3) * 2.0
    assert abs(np.sqrt(np.mean(t * t)) - 1 / math.sqrt(2)) < 1e-12


def _fused_setup(N, W, H, d, seed):
    r = np.random.default_rng(seed)

    def window():
        return dict(q=r.standard_normal((N, W, H, d)), k=r.standard_normal((N, W, H, d)),
                    v=r.standard_normal((N, W, H, d)), z=r.standard_normal((N, W, H, d)),
                    beta=r.standard_normal((N, W, H)), o_gate=r.standard_normal((N, W, H, d)))

    A = 0.3 * r.standard_normal(H)
    S0 = 0.05 * r.standard_normal((N, H, d, d))
    cs0 = r.standard_normal((N, H, 3, 3, d))
    conv_w = r.uniform(-0.5, 0.5, (3, H, d, 4))
    norm_w = 1.0 + 0.1 * r.standard_normal(d)
    empty = (np.zeros((N, W - 1, H, d)),) * 4 + (np.zeros((N, W - 1, H)),)
    return r, window, A, S0, cs0, conv_w, norm_w, empty


def _fused(S, w, A, conv_w, cs, norm_w, cache, nacc, **opt):
    return oracle.decode_step_fused(S, w["q"], w["k"], w["v"], w["z"], w["beta"], A, conv_w, cs,
                                    w["o_gate"], norm_w, 1e-6, *cache, num_accepted=nacc,
                                    return_prenorm=True, **opt)


def test_fused_decode_with_unit_conv_is_plain_decode():
    """With the convolution a unit impulse on the current token and no input options the
    fused step's recurrence is the plain decode step, over two steps with replay."""
    N, W, H, d = 4, 4, 2, 16
    _, window, A, S0, cs0, _, norm_w, empty = _fused_setup(N, W, H, d, 35)
    unit = np.zeros((3, H, d, 4))
    unit[..., 3] = 1.0
    w1, w2 = window(), window()
    for w in (w1, w2):
        w["beta"] = 1.0 / (1.0 + np.exp(-w["beta"]))
    nacc = np.array([0, 3, 1, 2])
    o1, S1, c1, cs1, p1 = _fused(S0, w1, A, unit, cs0, norm_w, empty, None)
    o2, S2, c2, cs2, p2 = _fused(S1, w2, A, unit, cs1, norm_w, c1, nacc)
    r1, T1, k1 = oracle.decode_step(S0, w1["q"], w1["k"], w1["v"], w1["z"], w1["beta"], A, *empty)
    r2, T2, k2 = oracle.decode_step(T1, w2["q"], w2["k"], w2["v"], w2["z"], w2["beta"], A, *k1,
                                    num_accepted=nacc)
    assert rel(p1, r1) < 1e-13 and rel(S1, T1) < 1e-13
    assert rel(p2, r2) < 1e-13 and rel(S2, T2) < 1e-13
    for a, b in zip(c2, k2):
        assert np.array_equal(a, b)


def test_fused_decode_equals_convolved_committed_stream():
    """Two fused steps equal numpy's convolution of the committed stream (convolution state,
    t0, the accepted drafts, the next t0, then the new drafts) followed by the plain
    recurrence; the convolution state then holds the last three committed inputs."""
    N, W, H, d = 4, 5, 2, 16
    _, window, A, S0, cs0, conv_w, norm_w, empty = _fused_setup(N, W, H, d, 37)
    w1, w2 = window(), window()
    nacc = np.array([0, 4, 2, 1])
    opt = dict(qk_l2norm=True, beta_sigmoid=True, conv_silu=True)
    _, S1, c1, cs1, _ = _fused(S0, w1, A, conv_w, cs0, norm_w, empty, None, **opt)
    _, S2, _, cs2, p2 = _fused(S1, w2, A, conv_w, cs1, norm_w, c1, nacc, **opt)
    for b in range(N):
        n = nacc[b]
        raw = {}
        for i, name in enumerate(("q", "k", "v")):
            s = np.concatenate([cs0[b, :, i].transpose(1, 0, 2), w1[name][b, :n + 1], w2[name][b]])
            y = np.zeros((len(s) - 3, H, d))
            for h in range(H):
                for c in range(d):
                    y[:, h, c] = np.convolve(s[:, h, c], conv_w[i, h, c, ::-1], mode="valid")
            raw[name] = y * np.exp(y) / (1.0 + np.exp(y))  # SiLU as x / (1 + e^-x), rewritten
            # the state after step 2 holds the inputs at t0(1) d1..dn, t0(2): the last three
            assert np.array_equal(cs2[b, :, i], s[n + 2:n + 5].transpose(1, 0, 2))
        z = np.concatenate([w1["z"][b, :n + 1], w2["z"][b]])
        beta = np.concatenate([w1["beta"][b, :n + 1], w2["beta"][b]])
        q, k, beta = oracle.input_prep(raw["q"], raw["k"], beta, qk_l2norm=True, beta_sigmoid=True)
        o_ref, _ = oracle.recurrent(q, k, raw["v"], z, A, beta, init_state=S0[b:b + 1])
        _, f_ref = oracle.recurrent(q[:n + 2], k[:n + 2], raw["v"][:n + 2], z[:n + 2], A, beta[:n + 2],
                                    init_state=S0[b:b + 1])
        assert rel(S2[b], f_ref[0]) < 1e-12
        assert rel(p2[b], o_ref[n + 1:]) < 1e-12


def test_fused_decode_output_is_normalised_prenorm():
    """The fused outputs are the pre-norm outputs through the gated per-head norm; the new
    cache holds the window's drafts as given (before the convolution)."""
    N, W, H, d = 3, 3, 2, 16
    _, window, A, S0, cs0, conv_w, norm_w, empty = _fused_setup(N, W, H, d, 39)
    w1 = window()
    w1["o_gate"][:] = 0.0
    o, _, c, _, p = _fused(S0, w1, A, conv_w, cs0, np.ones(d), empty, None)
    y = o * 2.0  # gate 0: sigmoid 1/2
    assert np.allclose(y * np.sqrt(np.mean(p * p, axis=-1, keepdims=True) + 1e-6), p, rtol=1e-12)
    for a, name in zip(c, ("q", "k", "v", "z", "beta")):
        assert np.array_equal(a, w1[name][:, 1:])
