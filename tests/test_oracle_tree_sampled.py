"""Pins for the oracle's sampled token tree (sequential over siblings).

Source: EAGLE-3 review, "EAGLE-3 inference" step 4 (sampling keeps min(1, p/q)
acceptance and residual correction, which preserves the target distribution)
and the review's identity min(p, q) + max(0, p - q) = p; the sibling rule is
the reading stated in the oracle (test children in order, replace p' by
norm(max(0, p' - q)) after each rejection, draw from p' when none is accepted).

What fixes it from outside the oracle:
  * the output law: with children drawn i.i.d. from q, the first token has law
    p of the root and, given that a child was accepted, the second token has
    the law of that child's row (chi-square, as the pages ask for the chain);
  * which sibling is accepted: P(child j first accepted) = S_{j-1} - S_j and
    P(none) = S_m, where S_j = sum_x max(0, p(x) - T_j q(x)), T_0 = 0, S_0 = 1,
    T_{j+1} = T_j + S_j (the j-fold residual written in closed form);
  * a tree with one child per level is the chain;
  * q = p accepts every child; q(x) = 0 accepts; out-of-range children are
    rejected and the draw follows the closed-form residual (numpy cumsum +
    searchsorted).
"""
import numpy as np
import pytest
from scipy import stats

from speculative_decoding_verification_chain_gb300 import workloads as W

from test_oracle_pins import _softmax64


def closed_form_masses(p, q, m):
    """S_0..S_m and T_0..T_m of the j-fold residual max(0, p - T_j q)."""
    S, T = [1.0], [0.0]
    for _ in range(m):
        T.append(T[-1] + S[-1])
        S.append(float(np.maximum(0.0, p - T[-1] * q).sum()))
    return np.array(S), np.array(T)


def law_case(seed=41, trials=1_000_000, V=6, m=3, m2=2, Temp=1.0):
    """Root with m children, each with m2 children.  Logits of a level-1 node
    are a function of its token (table[token]); children are drawn i.i.d. from
    their parent's q (q_root at the root, q1[token] below)."""
    g = np.random.default_rng(seed)
    z0 = g.standard_normal(V).astype(np.float32) * 1.5
    table = (g.standard_normal((V, V)) * 1.5).astype(np.float32)
    zleaf = (g.standard_normal(V) * 1.5).astype(np.float32)
    q0 = _softmax64(z0 + g.standard_normal(V) * 1.2, 1.0).astype(np.float32)
    q1 = _softmax64(table + g.standard_normal((V, V)) * 1.2, 1.0).astype(np.float32)
    parent = W.parents_in_order((m, m2))
    N = parent.shape[0] - 1
    B = trials
    c0 = np.cumsum(q0.astype(np.float64))
    t1 = np.minimum(np.searchsorted(c0, g.random((B, m)) * c0[-1], side="right"), V - 1).astype(np.int32)
    c1 = np.cumsum(q1.astype(np.float64), axis=1)
    t2 = np.empty((B, m * m2), np.int32)
    r2 = g.random((B, m * m2))
    for j in range(m * m2):
        rows = c1[t1[:, j // m2]]
        t2[:, j] = np.minimum((rows < (r2[:, j] * rows[:, -1])[:, None]).sum(axis=1), V - 1)
    toks = np.concatenate([t1, t2], axis=1)
    z = np.empty((B, N + 1, V), np.float32)
    z[:, 0] = z0
    z[:, 1:m + 1] = table[t1]
    z[:, m + 1:] = zleaf
    q = np.zeros((B, N + 1, V), np.float32)
    q[:, 0] = q0
    q[:, 1:m + 1] = q1[t1]
    ua = W.method_uniforms(g, (B, N))
    us = W.method_uniforms(g, (B, N + 1))
    return dict(z=z, q=q, toks=toks, parent=parent, T=np.full(B, Temp, np.float32), ua=ua, us=us,
                z0=z0, table=table, q0=q0, m=m, V=V, Temp=Temp)


def run(O, c, lib=None):
    return O.verify_tree_sampled(c["z"], W.FP32, c["toks"], c["parent"], c["T"], c["ua"], c["us"], c["q"],
                                 lib=lib)


def law_pvalues(c, r):
    """p-values: first token vs p_root; which root child is accepted vs the
    closed form; second token given the first vs that child's row."""
    V, m, Temp = c["V"], c["m"], c["Temp"]
    B = r["tokens"].shape[0]
    out = {}
    p0 = _softmax64(c["z0"], Temp)
    out["first"] = stats.chisquare(np.bincount(r["tokens"][:, 0], minlength=V), p0 * B).pvalue
    S, _ = closed_form_masses(p0, c["q0"].astype(np.float64), m)
    which = r["path"][:, 1]
    obs = np.array([(which == j).sum() for j in range(1, m + 1)] + [(which < 0).sum()])
    exp = np.concatenate([S[:-1] - S[1:], S[-1:]]) * B
    out["sibling"] = stats.chisquare(obs, exp).pvalue
    pv = []
    for t in range(V):
        sel = (r["length"] >= 2) & (r["tokens"][:, 0] == t)
        if sel.sum() < 2000:
            continue
        pt = _softmax64(c["table"][t], Temp)
        pv.append(stats.chisquare(np.bincount(r["tokens"][sel, 1], minlength=V), pt * sel.sum()).pvalue)
    out["second"] = min(pv)
    out["n_second"] = len(pv)
    return out


def test_output_law_and_sibling_law(oracle_mod):
    c = law_case()
    r = run(oracle_mod, c)
    pv = law_pvalues(c, r)
    assert pv["n_second"] >= 4
    assert pv["first"] > 0.01, pv
    assert pv["sibling"] > 0.01, pv
    # several conditional laws: Bonferroni over them
    assert pv["second"] > 0.01 / pv["n_second"], pv


def test_temperature_enters_the_law(oracle_mod):
    c = law_case(seed=42, trials=100_000, Temp=0.6)
    r = run(oracle_mod, c)
    pv = law_pvalues(c, r)
    assert pv["first"] > 0.01 and pv["sibling"] > 0.01, pv


def test_one_child_per_level_is_the_chain(oracle_mod):
    O = oracle_mod
    x = W.chain_sampled(seed=43, B=300, k=4, V=257, temperature=0.8, lam=0.4, dtype=W.FP32)
    k = 4
    parent = W.parents_in_order((1,) * k)
    q = np.zeros((x.B, k + 1, x.V), np.float32)
    q[:, :k] = x.draft_probs
    rt = O.verify_tree_sampled(x.logits, x.dtype, x.draft_tokens, parent, x.temperature, x.u_accept, x.u_sample, q)
    rc = O.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample, x.draft_probs, x.u_accept)
    assert ((rt["length"] - 1) == rc["num_accepted"]).all()
    assert (rt["path"] == np.where(np.arange(k + 1)[None, :] <= rc["num_accepted"][:, None],
                                   np.arange(k + 1)[None, :], -1)).all()
    flagged = rt["flag_sample"].astype(bool) | rc["flag_sample"].astype(bool)
    same = (rt["tokens"] == rc["out_tokens"]).all(axis=1)
    assert (same | flagged).all()
    assert same.sum() >= 0.95 * x.B


def q_equal_p_mismatches(O, lib=None):
    """q = p: every child is accepted (ratio 1 > u), so the walk takes the first
    child at each level and draws from the leaf's p with u_sample[leaf].
    Returns the number of requests that break this."""
    g = np.random.default_rng(44)
    B, V, Temp = 50, 97, 0.9
    parent = W.parents_in_order((3, 2, 1))
    N = parent.shape[0] - 1
    z = (g.standard_normal((B, N + 1, V)) * 2).astype(np.float32)
    q = _softmax64(z, Temp).astype(np.float32)
    toks = g.integers(0, V, size=(B, N)).astype(np.int32)
    ua = W.method_uniforms(g, (B, N))
    us = W.method_uniforms(g, (B, N + 1))
    r = O.verify_tree_sampled(z, W.FP32, toks, parent, np.full(B, Temp, np.float32), ua, us, q, lib=lib)
    first = np.array([0, 1, 4, 10])           # first child at every level of (3, 2, 1)
    bad = 0
    for b in range(B):
        p = _softmax64(z[b, 10], Temp)
        cdf = np.cumsum(p)
        j = int(np.searchsorted(cdf, float(us[b, 10]) * cdf[-1], side="right"))
        ok = (r["path"][b] == first).all() and r["length"][b] == 4
        ok = ok and (r["tokens"][b, :3] == toks[b, [0, 3, 9]]).all()
        ok = ok and (r["tokens"][b, 3] == j or bool(r["flag_sample"][b]))
        bad += int(not ok)
    return bad


def test_q_equal_p_accepts_every_child_and_draws_from_the_leaf(oracle_mod):
    assert q_equal_p_mismatches(oracle_mod) == 0


def zero_q_violations(O, lib=None):
    """Two children under the root: the first is out of range (p(x) = 0, so it
    is rejected at any u), the second has q(x) = 0 (accepted even at the
    largest uniform).  Returns the requests whose walk does not end at the
    second child with its token."""
    g = np.random.default_rng(45)
    B, V = 40, 31
    parent = W.parents_in_order((2,))
    z = (g.standard_normal((B, 3, V)) * 2).astype(np.float32)
    q = _softmax64(g.standard_normal((B, 3, V)), 1.0).astype(np.float32)
    toks = g.integers(0, V, size=(B, 2)).astype(np.int32)
    q[np.arange(B), 0, toks[:, 1]] = 0.0       # second child has q = 0; first child is out of range
    toks[:, 0] = V
    ua = np.full((B, 2), np.float32(1.0 - 2 ** -24))
    us = W.method_uniforms(g, (B, 3))
    r = O.verify_tree_sampled(z, W.FP32, toks, parent, np.ones(B, np.float32), ua, us, q, lib=lib)
    return int(((r["path"][:, 1] != 2) | (r["length"] != 2) | (r["tokens"][:, 0] != toks[:, 1])).sum())


def test_zero_draft_probability_accepts(oracle_mod):
    assert zero_q_violations(oracle_mod) == 0


def closed_form_residual_mismatches(O, lib=None):
    """Out-of-range children are rejected one after another; the draw then
    follows max(0, p - T_m q) / S_m (closed form of the m-fold residual).
    Returns (requests that break this, flagged draws)."""
    g = np.random.default_rng(46)
    B, V, m, Temp = 200, 211, 4, 0.8
    parent = W.parents_in_order((m,))
    z = (g.standard_normal((B, m + 1, V)) * 2).astype(np.float32)
    q = _softmax64(z + g.standard_normal((B, m + 1, V)) * 0.8, 1.0).astype(np.float32)
    toks = np.where(g.random((B, m)) < 0.5, -1, V).astype(np.int32)
    ua = W.method_uniforms(g, (B, m))
    us = W.method_uniforms(g, (B, m + 1))
    r = O.verify_tree_sampled(z, W.FP32, toks, parent, np.full(B, Temp, np.float32), ua, us, q, lib=lib)
    bad = int(((r["length"] != 1) | (r["path"][:, 1] != -1)).sum())
    for b in range(B):
        p = _softmax64(z[b, 0], Temp)
        qb = q[b, 0].astype(np.float64)
        S, T = closed_form_masses(p, qb, m)
        w = np.maximum(0.0, p - T[-1] * qb) if S[-1] > 0 else p
        cdf = np.cumsum(w)
        j = int(np.searchsorted(cdf, float(us[b, 0]) * cdf[-1], side="right"))
        bad += int(r["tokens"][b, 0] != j and not r["flag_sample"][b])
    return bad, int(r["flag_sample"].sum())


def test_all_rejected_draws_from_closed_form_residual(oracle_mod):
    bad, flagged = closed_form_residual_mismatches(oracle_mod)
    assert bad == 0
    assert flagged <= 10


def test_full_size_workload_runs_and_flags_are_rare(oracle_mod):
    x = W.tree_sampled(seed=47, B=4, V=4096)
    r = oracle_mod.verify_tree_sampled(x.logits, x.dtype, x.node_tokens, x.parent, x.temperature,
                                       x.u_accept, x.u_sample, x.draft_probs)
    assert ((r["length"] >= 1) & (r["length"] <= 6)).all()
    # path consistency: parents chain, tokens are the path's node tokens
    for b in range(x.B):
        L = r["length"][b]
        for i in range(1, L):
            n = r["path"][b, i]
            assert x.parent[n] == r["path"][b, i - 1]
            assert r["tokens"][b, i - 1] == x.node_tokens[b, n - 1]
        assert (r["path"][b, L:] == -1).all() and (r["tokens"][b, L:] == -1).all()


def test_argument_checks(oracle_mod):
    c = law_case(trials=4)
    with pytest.raises(ValueError):
        oracle_mod.verify_tree_sampled(c["z"], W.FP32, c["toks"], c["parent"], np.zeros(4, np.float32),
                                       c["ua"], c["us"], c["q"])
    bad_parent = c["parent"].copy()
    bad_parent[3] = 5
    with pytest.raises(ValueError):
        oracle_mod.verify_tree_sampled(c["z"], W.FP32, c["toks"], bad_parent, c["T"], c["ua"], c["us"], c["q"])


def test_bench_bytes_from_path_match_the_oracle(oracle_mod):
    """The benchmark derives a walk's algorithmic bytes from its path alone;
    on the same walks that equals the oracle's own count."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    x = W.tree_sampled(seed=48, B=40, V=3001, children_per_level=(3, 2, 2), lam=0.5)
    r = oracle_mod.verify_tree_sampled(x.logits, x.dtype, x.node_tokens, x.parent, x.temperature,
                                       x.u_accept, x.u_sample, x.draft_probs)
    for b in range(x.B):
        got = bench.tree_sampled_bytes(x.parent, r["path"][b:b + 1], r["length"][b:b + 1], x.V, 2)
        assert got == r["b_alg"][b], b
