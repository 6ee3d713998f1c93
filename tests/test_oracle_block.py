"""Pins for the fp64 block oracle.

The oracle is checked against things other than itself:
  * closed forms (a scalar-algebra evaluation of the block on constant rows),
  * library routines (scipy's softmax and expit),
  * brute force (the per-token definition vs the expert-batched form),
  * the invariants the method implies (token-order equivariance, the k=1
    dense reduction, per-expert output-scale invariance, routing independence
    for identical experts, zero gate -> identity, constant expert gamma ->
    known RMS, identity pooler/unpooler -> a plain top-k SwiGLU MoE),
  * and a negative test: normalising after the sum computes something else
    (LMSYS Muse Spark Open post, "MoE with pooler, unpooler and per-expert
    normalization": the order matters).
"""
import math

import numpy as np
import pytest
import scipy.special as sps

import oracle
from oracle import BlockParams, ExpertStack


def rand_params(rs, D, L, E, I, eps=1e-6, gamma=True):
    g = (lambda n: 1 + 0.1 * rs.standard_normal(n)) if gamma else (lambda n: np.ones(n))
    return BlockParams(
        W_router=rs.standard_normal((E, D)) / math.sqrt(D),
        W_pool=rs.standard_normal((L, D)) / math.sqrt(D), g_pool=g(L),
        W_gate=ExpertStack(rs.standard_normal((E, I, L)) / math.sqrt(L), E),
        W_up=ExpertStack(rs.standard_normal((E, I, L)) / math.sqrt(L), E),
        W_down=ExpertStack(rs.standard_normal((E, L, I)) / math.sqrt(I), E),
        g_expert=np.stack([g(L) for _ in range(E)]),
        W_unpool=rs.standard_normal((D, L)) / math.sqrt(L), g_pre=g(D), g_post=g(D), eps=eps)


SHAPES = [(5, 24, 16, 6, 40, 2), (7, 32, 48, 8, 16, 3), (3, 16, 8, 4, 24, 1), (4, 16, 16, 5, 8, 5)]


@pytest.mark.parametrize("T,D,L,E,I,k", SHAPES)
def test_batched_equals_per_token_definition(T, D, L, E, I, k):
    rs = np.random.default_rng(T * 1000 + D)
    P = rand_params(rs, D, L, E, I)
    x = rs.standard_normal((T, D))
    a = oracle.forward_per_token(x, P, k)
    b = oracle.forward_batched(x, P, k)
    assert np.max(np.abs(a - b)) <= 1e-12 * max(1.0, np.max(np.abs(a)))


def test_closed_form_constant_rows():
    # D = L = I = n, identity-like weights, constant rows: every norm and the SwiGLU
    # reduce to scalar algebra, evaluated here with the math module alone.
    n, E, k, eps = 16, 4, 2, 1e-6
    a_, b_, d_ = 0.7, -1.3, 2.1
    eye = np.eye(n)
    P = BlockParams(
        W_router=np.random.default_rng(0).standard_normal((E, n)), W_pool=eye, g_pool=np.ones(n),
        W_gate=ExpertStack(np.stack([a_ * eye] * E), E), W_up=ExpertStack(np.stack([b_ * eye] * E), E),
        W_down=ExpertStack(np.stack([d_ * eye] * E), E), g_expert=np.ones((E, n)),
        W_unpool=eye, g_pre=np.ones(n), g_post=np.ones(n), eps=eps)
    for alpha in (0.3, -2.0, 5.0):
        x = np.full((1, n), alpha)
        nrm = lambda s: s / math.sqrt(s * s + eps)
        beta = nrm(alpha)
        gam = nrm(beta)
        delta = d_ * (a_ * gam / (1 + math.exp(-a_ * gam))) * (b_ * gam)
        zeta = nrm(delta)
        expect = alpha + nrm(zeta)
        out = oracle.forward_batched(x, P, k)
        assert np.allclose(out, expect, rtol=0, atol=1e-13), (out[0, 0], expect)


def test_route_against_scipy_softmax_and_ties():
    rs = np.random.default_rng(5)
    l = rs.standard_normal((50, 12))
    idx, w, _ = oracle.route(l, 3)
    for t in range(50):
        sel = np.argsort(-l[t])[:3]
        assert list(idx[t]) == list(sel)
        # renormalised full softmax == softmax over the selected logits only
        assert np.allclose(w[t], sps.softmax(l[t, sel]), rtol=0, atol=1e-15)
        assert np.allclose(w[t], sps.softmax(l[t])[sel] / sps.softmax(l[t])[sel].sum(), atol=1e-15)
    # exact ties go to the lower expert index
    lt = np.array([[0.5, 2.0, 2.0, 1.0, 2.0]])
    assert oracle.route(lt, 2)[0].tolist() == [[1, 2]]
    assert oracle.route(lt, 3)[0].tolist() == [[1, 2, 4]]
    # near-tie flag: k-th vs (k+1)-th margin below 1e-3
    assert oracle.route(np.array([[3.0, 1.0, 1.0005, 0.0]]), 2)[2].tolist() == [True]
    assert oracle.route(np.array([[3.0, 1.0, 1.002, 0.0]]), 2)[2].tolist() == [False]
    # k = E: weights are the plain softmax
    idx, w, nt = oracle.route(l[:1], 12)
    assert np.allclose(w[0], sps.softmax(l[0])[idx[0]], atol=1e-15) and not nt.any()


def test_rms_norm_closed_form_and_eps_placement():
    v = np.array([[3.0, -4.0]])        # mean square 12.5
    g = np.array([2.0, 0.5])
    eps = 0.5
    out = oracle.rms_norm(v, g, eps)
    assert np.allclose(out, v / math.sqrt(12.5 + 0.5) * g, atol=1e-15)
    assert oracle.silu(np.array([1.5]))[0] == pytest.approx(1.5 * sps.expit(1.5), abs=1e-15)


def test_token_permutation_equivariance():
    rs = np.random.default_rng(7)
    P = rand_params(rs, 32, 16, 6, 24)
    x = rs.standard_normal((9, 32))
    perm = rs.permutation(9)
    a = oracle.forward_per_token(x, P, 2)
    b = oracle.forward_per_token(x[perm], P, 2)
    assert np.array_equal(a[perm], b)        # per-token evaluation: bitwise


def test_k1_reduces_to_dense_swiglu_path():
    # Independent dense path written with scipy's expit: with top_k = 1 the weight is 1
    # and the block is x + N(U N(D (silu(G h0) * (U' h0)); g_e); g_post).
    rs = np.random.default_rng(8)
    D, L, E, I = 24, 16, 5, 20
    P = rand_params(rs, D, L, E, I)
    x = rs.standard_normal((6, D))
    out = oracle.forward_batched(x, P, 1)

    def nrm(v, g):
        return v / np.sqrt((v ** 2).sum() / v.size + P.eps) * g

    for t in range(6):
        xn = nrm(x[t], P.g_pre)
        e = int(np.argmax(P.W_router @ xn))
        h0 = nrm(P.W_pool @ xn, P.g_pool)
        a = P.W_gate[e] @ h0
        y = P.W_down[e] @ (a * sps.expit(a) * (P.W_up[e] @ h0))
        ref = x[t] + nrm(P.W_unpool @ nrm(y, P.g_expert[e]), P.g_post)
        assert np.allclose(out[t], ref, rtol=0, atol=1e-12)


def test_norm_after_sum_differs():
    rs = np.random.default_rng(9)
    P = rand_params(rs, 32, 16, 8, 24)
    x = rs.standard_normal((16, 32))
    a = oracle.forward_batched(x, P, 2)
    b = oracle.forward_norm_after_sum(x, P, 2)
    assert np.max(np.abs(a - b)) > 1e-3 * np.sqrt(np.mean(a ** 2))


def test_per_expert_output_scale_invariance():
    # scaling W_down[e] by a > 0 leaves the block unchanged (up to the eps terms) only
    # because each expert output is normalised before it is weighted
    rs = np.random.default_rng(10)
    P = rand_params(rs, 32, 16, 6, 24, eps=1e-12)
    x = rs.standard_normal((8, 32))
    a = oracle.forward_batched(x, P, 3)
    Wd = np.stack([P.W_down[e] * (0.1 + 3 * e) for e in range(6)])
    P2 = BlockParams(**{**P.__dict__, "W_down": ExpertStack(Wd, 6)})
    b = oracle.forward_batched(x, P2, 3)
    assert np.max(np.abs(a - b)) < 1e-9
    b2 = oracle.forward_norm_after_sum(x, P2, 3)
    assert np.max(np.abs(oracle.forward_norm_after_sum(x, P, 3) - b2)) > 1e-3


def test_identical_experts_make_routing_irrelevant():
    rs = np.random.default_rng(11)
    P = rand_params(rs, 32, 16, 6, 24)
    one = lambda S: ExpertStack(np.stack([S[0]] * 6), 6)
    P2 = BlockParams(**{**P.__dict__, "W_gate": one(P.W_gate), "W_up": one(P.W_up),
                        "W_down": one(P.W_down), "g_expert": np.stack([P.g_expert[0]] * 6)})
    x = rs.standard_normal((8, 32))
    a = oracle.forward_batched(x, P2, 1)
    b = oracle.forward_batched(x, P2, 4)
    P3 = BlockParams(**{**P2.__dict__, "W_router": -P2.W_router})
    c = oracle.forward_batched(x, P3, 2)
    assert np.allclose(a, b, atol=1e-12) and np.allclose(a, c, atol=1e-12)


def test_zero_gate_is_identity():
    rs = np.random.default_rng(12)
    P = rand_params(rs, 32, 16, 6, 24)
    P2 = BlockParams(**{**P.__dict__, "W_gate": ExpertStack(np.zeros((6, 24, 16)), 6)})
    x = rs.standard_normal((5, 32))
    assert np.array_equal(oracle.forward_batched(x, P2, 2), x)


def test_constant_expert_gamma_gives_known_rms():
    rs = np.random.default_rng(13)
    P = rand_params(rs, 32, 16, 6, 24)
    cs = 0.5 + np.arange(6)
    P2 = BlockParams(**{**P.__dict__, "g_expert": cs[:, None] * np.ones((6, 16))})
    x = rs.standard_normal((5, 32))
    tr = oracle.Trace()
    oracle.forward_batched(x, P2, 3, trace=tr)
    for (t, j), y in tr.y.items():
        e = int(tr.idx[t, j])
        ms = np.mean(y ** 2)
        rms_z = np.sqrt(np.mean(tr.z[(t, j)] ** 2))
        assert rms_z == pytest.approx(cs[e] * math.sqrt(ms / (ms + P.eps)), rel=1e-13)


def test_identity_pool_unpool_gives_plain_topk_swiglu_moe():
    # W_pool = [I_L | 0], W_unpool = [I_L ; 0]: the latent block becomes a plain top-k
    # SwiGLU MoE with norms, written here without the oracle
    rs = np.random.default_rng(14)
    D, L, E, I, k = 24, 16, 6, 20, 2
    P = rand_params(rs, D, L, E, I)
    Wp = np.zeros((L, D)); Wp[:, :L] = np.eye(L)
    Wu = np.zeros((D, L)); Wu[:L, :] = np.eye(L)
    P2 = BlockParams(**{**P.__dict__, "W_pool": Wp, "W_unpool": Wu})
    x = rs.standard_normal((7, D))
    out = oracle.forward_batched(x, P2, k)

    def nrm(v, g):
        return v / np.sqrt(np.mean(v * v) + P.eps) * g

    for t in range(7):
        xn = nrm(x[t], P.g_pre)
        l = P.W_router @ xn
        sel = np.argsort(-l, kind="stable")[:k]
        wts = sps.softmax(l[sel])
        h0 = nrm(xn[:L], P.g_pool)
        c = np.zeros(L)
        for wj, e in zip(wts, sel):
            a = P.W_gate[e] @ h0
            c += wj * nrm(P.W_down[e] @ (a * sps.expit(a) * (P.W_up[e] @ h0)), P.g_expert[e])
        u = np.zeros(D); u[:L] = c
        ref = x[t] + nrm(u, P.g_post)
        assert np.allclose(out[t], ref, rtol=0, atol=1e-12)


def test_forced_routing_uses_softmax_at_forced_ids():
    rs = np.random.default_rng(15)
    P = rand_params(rs, 32, 16, 6, 24)
    x = rs.standard_normal((4, 32))
    forced = np.array([[5, 0], [1, 2], [3, 4], [0, 5]])
    tr = oracle.Trace()
    oracle.forward_batched(x, P, 2, forced_idx=forced, trace=tr)
    assert np.array_equal(tr.idx, forced)
    for t in range(4):
        assert np.allclose(tr.w[t], sps.softmax(tr.logits[t, forced[t]]), atol=1e-15)


def test_nvfp4_mode_with_dense_weights_moves_little_and_is_deterministic():
    rs = np.random.default_rng(16)
    P = rand_params(rs, 64, 32, 6, 48)
    Pq = BlockParams(**{**P.__dict__, "nvfp4": True})
    x = rs.standard_normal((6, 64))
    a = oracle.forward_batched(x, P, 2)
    b = oracle.forward_batched(x, Pq, 2)
    c = oracle.forward_per_token(x, Pq, 2)
    d = a - x
    assert np.max(np.abs(b - c)) < 1e-12
    assert 1e-4 < np.sqrt(np.mean((b - a) ** 2)) / np.sqrt(np.mean(d ** 2)) < 0.3
