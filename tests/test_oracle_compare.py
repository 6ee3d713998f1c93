"""Pins for the parity comparator (oracle/compare.py): classify_topk and compare_block.

Every GPU parity decision goes through these two functions, so they are fed hand-built cases
whose right answer follows from the grading rules alone (LMSYS Muse Spark Open post, "MoE
with pooler, unpooler and per-expert normalization": the router's top-k over the full-width
logits; the near-tie band of 1e-3 on the k-th/(k+1)-th margin and the 2e-2 / 6e-2 x RMS output
bars are the grading rules the block is held to):

  * an exact match is accepted and counted as exact;
  * a near-tie token (k-th and (k+1)-th logits within 1e-3) that picks a different set is
    accepted, counted, and graded against the oracle re-run with the GPU's selection;
  * two selected experts whose logits differ by less than 1e-3 may come in either order;
  * a swap of two experts 2e-3 apart is rejected, and so is a wrong set on a clear margin,
    even when the output matches the GPU's own (wrong) selection;
  * outputs just under tol x RMS pass, just over fail.

The cases are written once as functions of (classify, compare) and also run against broken
copies of the comparator defined in this file (each with one plausible mistake): each broken
copy must fail at least one case, which shows that the cases can see that mistake.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
from oracle import BlockParams, ExpertStack
from oracle import compare as C


# ------------------------------------------------------------------ fixtures
def _params(E: int, bias, tie_delta=0.0, seed=0, D=16, L=8, I=12):
    """Tiny block whose router gives experts 0 and 1 the same logit up to `bias` (+ a tiny
    per-token difference `tie_delta` * (xn . r)), and experts >= 2 their bias offsets."""
    rs = np.random.default_rng(seed)
    w0 = rs.standard_normal(D) / math.sqrt(D)
    W = np.tile(w0, (E, 1))
    if tie_delta:
        W[1] = w0 + tie_delta * rs.standard_normal(D)
    g = lambda n: 1 + 0.1 * rs.standard_normal(n)  # noqa: E731
    return BlockParams(
        W_router=W, W_pool=rs.standard_normal((L, D)) / math.sqrt(D), g_pool=g(L),
        W_gate=ExpertStack(rs.standard_normal((E, I, L)) / math.sqrt(L), E),
        W_up=ExpertStack(rs.standard_normal((E, I, L)) / math.sqrt(L), E),
        W_down=ExpertStack(rs.standard_normal((E, L, I)) / math.sqrt(I), E),
        g_expert=np.stack([g(L) for _ in range(E)]), W_unpool=rs.standard_normal((D, L)) / math.sqrt(L),
        g_pre=g(D), g_post=g(D), router_bias=np.asarray(bias, dtype=np.float64))


def _x(T, D=16, seed=1):
    return np.random.default_rng(seed).standard_normal((T, D))


def _ref(x, P, k, forced=None):
    tr = oracle.Trace()
    out = oracle.forward_batched(x, P, k, forced_idx=forced, trace=tr)
    return out, tr


def _forced_out(x, P, k, idx):
    """The output each token has under the selection `idx` (per-token definition)."""
    return np.stack([oracle.forward_per_token(x[t:t + 1], P, k, forced_idx=idx[t:t + 1])[0]
                     for t in range(x.shape[0])])


# ------------------------------------------------------------------ the cases
def case_exact_match(classify, compare):
    P = _params(4, [0.0, -0.5, -1.0, -1.5])
    x = _x(5)
    out, tr = _ref(x, P, 2)
    exact, near, swaps, bad = classify(tr.idx.copy(), tr, 2)
    assert exact.all() and near == [] and swaps == [] and bad == []
    rep = compare(out, tr.idx, x, P, 2, C.TOL_BF16)
    assert rep.ok and rep.idx_exact == 5 and rep.near_tie_tokens == 0 and rep.order_swaps == 0
    assert rep.max_abs_err == 0.0


def case_near_tie_other_set_accepted_and_regraded(classify, compare):
    # k = 1; experts 0 and 1 within ~1e-5 of each other, expert 2 ten below: every token is a
    # near tie.  The GPU picks the other one of the pair; its output is that of its own choice.
    P = _params(3, [0.0, 0.0, -10.0], tie_delta=1e-6)
    x = _x(4)
    out, tr = _ref(x, P, 1)
    assert tr.near_tie.all()
    gidx = 1 - tr.idx                      # the other expert of the tied pair
    exact, near, swaps, bad = classify(gidx, tr, 1)
    assert near == [0, 1, 2, 3] and swaps == [] and bad == []
    gout = _forced_out(x, P, 1, gidx)
    assert np.max(np.abs(gout - out)) > 10 * C.TOL_BF16 * np.sqrt(np.mean(out ** 2))   # really different
    rep = compare(gout, gidx, x, P, 1, C.TOL_BF16)
    assert rep.ok and rep.near_tie_tokens == 4 and rep.bad_idx_tokens == []
    assert rep.max_abs_err <= 1e-12
    # the oracle's own output for the oracle's selection is then wrong for this token
    rep2 = compare(out, gidx, x, P, 1, C.TOL_BF16)
    assert not rep2.ok


def case_in_band_order_swap_accepted(classify, compare):
    # k = 2 of 3: experts 0 and 1 within 1e-5, expert 2 ten below (a clear k-th margin)
    P = _params(3, [0.0, 0.0, -10.0], tie_delta=1e-6)
    x = _x(3)
    out, tr = _ref(x, P, 2)
    assert not tr.near_tie.any()
    gidx = tr.idx[:, ::-1].copy()          # same set, the two swapped
    exact, near, swaps, bad = classify(gidx, tr, 2)
    assert swaps == [0, 1, 2] and near == [] and bad == []
    gout = _forced_out(x, P, 2, gidx)
    rep = compare(gout, gidx, x, P, 2, C.TOL_BF16)
    assert rep.ok and rep.order_swaps == 3


def case_out_of_band_swap_rejected(classify, compare):
    # experts 0 and 1 exactly 2e-3 apart (bias), expert 2 ten below: the order is decided
    P = _params(3, [0.0, -2e-3, -10.0])
    x = _x(3)
    out, tr = _ref(x, P, 2)
    assert (tr.idx == [0, 1]).all() and not tr.near_tie.any()
    gidx = tr.idx[:, ::-1].copy()
    exact, near, swaps, bad = classify(gidx, tr, 2)
    assert bad == [0, 1, 2] and swaps == [] and near == []
    gout = _forced_out(x, P, 2, gidx)
    rep = compare(gout, gidx, x, P, 2, C.TOL_BF16)
    assert not rep.ok and rep.bad_idx_tokens == [0, 1, 2]


def case_wrong_set_on_clear_margin_rejected(classify, compare):
    # k = 1, expert 0 one logit above expert 1: picking 1 is wrong, even though the output
    # then matches the GPU's own selection exactly (no re-grading of a non-tie token)
    P = _params(3, [0.0, -1.0, -10.0])
    x = _x(4)
    out, tr = _ref(x, P, 1)
    assert (tr.idx[:, 0] == 0).all() and not tr.near_tie.any()
    gidx = tr.idx.copy()
    gidx[2, 0] = 1
    exact, near, swaps, bad = classify(gidx, tr, 1)
    assert bad == [2] and near == [] and swaps == [] and int(exact.sum()) == 3
    gout = out.copy()
    gout[2] = _forced_out(x[2:3], P, 1, gidx[2:3])[0]
    rep = compare(gout, gidx, x, P, 1, C.TOL_BF16)
    assert not rep.ok and rep.bad_idx_tokens == [2]


def case_output_bar(classify, compare, tol=C.TOL_BF16):
    P = _params(4, [0.0, -0.5, -1.0, -1.5])
    x = _x(6)
    out, tr = _ref(x, P, 2)
    rms = float(np.sqrt(np.mean(out ** 2)))
    for frac, ok in ((0.99, True), (1.01, False)):
        g = out.copy()
        g[3, 5] += frac * tol * rms
        g[1, 2] -= 0.5 * tol * rms
        rep = compare(g, tr.idx, x, P, 2, tol)
        assert rep.ok == ok, (frac, rep)
        assert math.isclose(rep.max_abs_err, frac * tol * rms, rel_tol=1e-9)
        assert math.isclose(rep.ref_rms, rms, rel_tol=1e-12)


def case_output_bar_nvfp4(classify, compare):
    case_output_bar(classify, compare, tol=C.TOL_NVFP4)


def case_k_equals_e_has_no_near_tie(classify, compare):
    # with k = E every expert is selected: there is no (k+1)-th logit and no near tie
    P = _params(3, [0.0, 0.0, 0.0], tie_delta=1e-6)
    x = _x(3)
    out, tr = _ref(x, P, 3)
    assert not tr.near_tie.any()
    exact, near, swaps, bad = classify(tr.idx.copy(), tr, 3)
    assert exact.all() and near == [] and bad == []


CASES = [case_exact_match, case_near_tie_other_set_accepted_and_regraded, case_in_band_order_swap_accepted,
         case_out_of_band_swap_rejected, case_wrong_set_on_clear_margin_rejected, case_output_bar,
         case_output_bar_nvfp4, case_k_equals_e_has_no_near_tie]


@pytest.mark.parametrize("case", CASES, ids=lambda f: f.__name__)
def test_comparator_case(case):
    case(C.classify_topk, C.compare_block)


# ------------------------------------------------------------------ broken copies
def _classify_any_same_set_is_swap(gpu_idx, tr, k):
    """Mistake: a same-set reordering is accepted whatever the logit gap."""
    gpu_idx = np.asarray(gpu_idx, dtype=np.int64)
    exact = np.all(gpu_idx == tr.idx, axis=1)
    near, swaps, bad = [], [], []
    for t in np.nonzero(~exact)[0]:
        if tr.near_tie[t]:
            near.append(int(t))
        elif set(gpu_idx[t].tolist()) == set(tr.idx[t].tolist()):
            swaps.append(int(t))
        else:
            bad.append(int(t))
    return exact, near, swaps, bad


def _classify_every_mismatch_is_near_tie(gpu_idx, tr, k):
    """Mistake: the near-tie flag is not consulted; every mismatch counts as a near tie."""
    gpu_idx = np.asarray(gpu_idx, dtype=np.int64)
    exact = np.all(gpu_idx == tr.idx, axis=1)
    return exact, [int(t) for t in np.nonzero(~exact)[0]], [], []


def _classify_band_on_wrong_side(gpu_idx, tr, k):
    """Mistake: the band test compares the logit gap the wrong way (accepts gaps >= band)."""
    gpu_idx = np.asarray(gpu_idx, dtype=np.int64)
    exact = np.all(gpu_idx == tr.idx, axis=1)
    near, swaps, bad = [], [], []
    for t in np.nonzero(~exact)[0]:
        if tr.near_tie[t]:
            near.append(int(t))
            continue
        lg = tr.logits[t]
        if set(gpu_idx[t].tolist()) == set(tr.idx[t].tolist()) and \
                np.all(np.abs(lg[gpu_idx[t]] - lg[tr.idx[t]]) >= C.TIE_BAND):
            swaps.append(int(t))
            continue
        bad.append(int(t))
    return exact, near, swaps, bad


def _compare_variant(regrade_bad=False, regrade_none=False, rms_of_gpu=False, sum_err=False):
    """compare_block with one mistake switched on."""
    def compare(gpu_out, gpu_idx, x, P, k, tol, tr=None, ref=None, forced_idx=None):
        x = np.asarray(x, dtype=np.float64)
        tr = oracle.Trace()
        ref = oracle.forward_batched(x, P, k, forced_idx=forced_idx, trace=tr)
        exact, near, swaps, bad = C.classify_topk(gpu_idx, tr, k)
        ref = ref.copy()
        regrade = [] if regrade_none else (near + swaps + (bad if regrade_bad else []))
        for t in regrade:
            ref[t] = oracle.forward_per_token(x[t:t + 1], P, k, forced_idx=np.asarray(gpu_idx)[t:t + 1])[0]
        err = np.abs(np.asarray(gpu_out, dtype=np.float64) - ref)
        base = np.asarray(gpu_out) if rms_of_gpu else ref
        return C.Report(tokens=x.shape[0], idx_exact=int(exact.sum()), near_tie_tokens=len(near),
                        order_swaps=len(swaps), bad_idx_tokens=[] if regrade_bad else bad,
                        max_abs_err=float(err.sum() if sum_err else err.max()),
                        ref_rms=float(np.sqrt(np.mean(base ** 2))), tol=tol)
    return compare


BROKEN = {
    "classify_any_same_set_is_swap": (_classify_any_same_set_is_swap, C.compare_block),
    "classify_every_mismatch_is_near_tie": (_classify_every_mismatch_is_near_tie, C.compare_block),
    "classify_band_on_wrong_side": (_classify_band_on_wrong_side, C.compare_block),
    "compare_regrades_bad_tokens": (C.classify_topk, _compare_variant(regrade_bad=True)),
    "compare_never_regrades": (C.classify_topk, _compare_variant(regrade_none=True)),
    "compare_sums_errors": (C.classify_topk, _compare_variant(sum_err=True)),
}


@pytest.mark.parametrize("name", sorted(BROKEN))
def test_broken_comparator_is_caught(name):
    classify, compare = BROKEN[name]
    failed = []
    for case in CASES:
        try:
            case(classify, compare)
        except AssertionError:
            failed.append(case.__name__)
    assert failed, f"no case detects the broken comparator {name}"


# ------------------------------------------------------------------ NVFP4 rounding boundaries
def _nvfp4_params(seed=3):
    P = _params(4, [0.0, -0.5, -1.0, -1.5], seed=seed, D=32, L=32, I=32)
    P.nvfp4 = True
    return P


def test_forward_token_choices_first_is_the_definition():
    P = _nvfp4_params()
    x = _x(3, D=32)
    ref = oracle.forward_per_token(x, P, 2)
    for t in range(3):
        outs = oracle.block.forward_token_choices(x[t], P, 2)
        assert np.max(np.abs(outs[0] - ref[t])) <= 1e-12


def _fake_choices(delta):
    """A choices function whose single alternative moves element 0 of the output by delta."""
    def choices(x_t, P, k, sel):
        base = oracle.forward_per_token(np.asarray(x_t)[None], P, k,
                                        forced_idx=None if sel is None else np.asarray(sel)[None])[0]
        alt = base.copy()
        alt[0] += delta
        return [base, alt]
    return choices


def test_boundary_alternative_accepted_and_counted_only_when_it_matches():
    P = _nvfp4_params()
    x = _x(4, D=32)
    out, tr = _ref(x, P, 2)
    rms = float(np.sqrt(np.mean(out ** 2)))
    big = 0.5 * rms                                 # far outside the 6e-2 bar
    g = out.copy()
    g[2, 0] += big
    rep = C.compare_block(g, tr.idx, x, P, 2, C.TOL_NVFP4, choices=_fake_choices(big))
    assert rep.ok and rep.quant_boundary_tokens == 1 and rep.max_abs_err < 1e-12
    # the GPU output matches no alternative: rejected
    rep = C.compare_block(g, tr.idx, x, P, 2, C.TOL_NVFP4, choices=_fake_choices(-big))
    assert not rep.ok and rep.quant_boundary_tokens == 0
    # BF16 compute has no quantisation decisions to take either way: never consulted
    P.nvfp4 = False
    out_b, tr_b = _ref(x, P, 2)
    g_b = out_b.copy()
    g_b[2, 0] += big
    rep = C.compare_block(g_b, tr_b.idx, x, P, 2, C.TOL_BF16, choices=_fake_choices(big))
    assert not rep.ok and rep.quant_boundary_tokens == 0


def test_boundary_alternative_found_in_a_real_nvfp4_block():
    # an NVFP4 block (E = 1024, k = 16, L = 256) where one token's c holds a block whose scale
    # ratio lies 1e-8 (relative) from an E4M3 midpoint: the token has exactly one alternative
    # output, 0.15 x RMS from the rule's own, the size of a one-code scale change of one block
    import workloads
    w = workloads.Workload("fp4_24_256_256_1024_256_16", T=24, D=256, L=256, E=1024, I=256, k=16,
                           weights="nvfp4", seed=24 % 5)
    inp = workloads.make_inputs(w, "cpu")
    P = oracle.params_from_inputs(inp)
    x = inp.x.double().numpy()[[3, 17]]
    ref = oracle.forward_batched(x, P, w.k)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert len(oracle.block.forward_token_choices(x[0], P, w.k)) == 1
    outs = oracle.block.forward_token_choices(x[1], P, w.k)
    assert len(outs) == 2 and 0.1 < np.max(np.abs(outs[1] - outs[0])) / rms < 0.2


def _compare_accepts_every_nvfp4_outlier(gpu_out, gpu_idx, x, P, k, tol, tr=None, ref=None, forced_idx=None,
                                         choices=None):
    """Mistake: an NVFP4 token outside the bar is accepted without matching an alternative."""
    rep = C.compare_block(gpu_out, gpu_idx, x, P, k, tol, tr=tr, ref=ref, forced_idx=forced_idx,
                          choices=lambda x_t, P_, k_, sel: [None, np.asarray(gpu_out)[
                              int(np.nonzero(np.all(np.asarray(x) == x_t, axis=1))[0][0])]])
    return rep


def test_broken_boundary_acceptance_is_caught():
    P = _nvfp4_params()
    x = _x(4, D=32)
    out, tr = _ref(x, P, 2)
    g = out.copy()
    g[2, 0] += 0.5 * float(np.sqrt(np.mean(out ** 2)))
    # with no alternative matching, the real comparator rejects; the broken one would accept
    assert not C.compare_block(g, tr.idx, x, P, 2, C.TOL_NVFP4, choices=_fake_choices(-1.0)).ok
    assert _compare_accepts_every_nvfp4_outlier(g, tr.idx, x, P, 2, C.TOL_NVFP4).ok
