"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these re-types the oracle's own formulas: each checks a closed form, a
special case, a brute-force enumeration, a library routine (numpy argmax /
cumsum + searchsorted) or a statistical law the pages state.
"""
import os

import numpy as np
import pytest
from scipy import stats

from speculative_decoding_verification_chain_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _softmax64(z, T):
    s = np.asarray(z, np.float64) / float(T)
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


# ---------------------------------------------------------------- greedy ----
def test_greedy_always_wrong_emits_row0_argmax(oracle_mod):
    """EAGLE-3 review, greedy rule: a draft that never matches yields a = 0 and
    the target's own argmax (the output equals plain greedy decoding)."""
    x = W.chain_greedy(seed=11, B=16, k=5, V=3001)
    zf = W.logits_as_f32(x.logits, x.dtype)
    am = np.argmax(zf, axis=-1)
    x.draft_tokens = ((am[:, :5] + 1) % x.V).astype(np.int32)
    r = oracle_mod.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample)
    assert (r["num_accepted"] == 0).all()
    assert (r["out_tokens"][:, 0] == am[:, 0]).all()
    assert (r["out_tokens"][:, 1:] == -1).all()


def test_greedy_always_right_accepts_all_plus_bonus(oracle_mod):
    x = W.chain_greedy(seed=12, B=16, k=5, V=3001, p_match=1.0)
    zf = W.logits_as_f32(x.logits, x.dtype)
    am = np.argmax(zf, axis=-1)
    r = oracle_mod.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample)
    assert (r["num_accepted"] == 5).all()
    assert (r["out_tokens"] == am).all()


@pytest.mark.parametrize("dtype", [W.BF16, W.FP32])
def test_greedy_matches_bruteforce_numpy(oracle_mod, dtype):
    """Brute force with numpy argmax (first occurrence) on the same data."""
    x = W.chain_greedy(seed=13, B=40, k=6, V=777, p_match=0.7, dtype=dtype)
    zf = W.logits_as_f32(x.logits, dtype)
    am = np.argmax(zf, axis=-1)
    r = oracle_mod.verify_chain(x.logits, dtype, x.draft_tokens, x.temperature, x.u_sample)
    for b in range(x.B):
        a = 0
        while a < x.k and x.draft_tokens[b, a] == am[b, a]:
            a += 1
        assert r["num_accepted"][b] == a
        exp = np.full(x.k + 1, -1)
        exp[:a] = x.draft_tokens[b, :a]
        exp[a] = am[b, a]
        assert (r["out_tokens"][b] == exp).all()
        assert r["b_alg"][b] == (a + 1) * x.V * (2 if dtype == W.BF16 else 4)


def test_greedy_ties_go_to_lowest_index(oracle_mod):
    V = 64
    z = np.zeros((3, 3, V), np.float32)
    z[:, :, 5] = 7.0
    z[:, :, 40] = 7.0     # same maximum later in the row
    z[1, :, 2] = 7.0      # and earlier in request 1
    tok = np.array([[5, 5], [5, 2], [40, 5]], np.int32)
    r = oracle_mod.verify_chain(z, W.FP32, tok, np.zeros(3, np.float32), np.zeros((3, 3), np.float32))
    assert list(r["num_accepted"]) == [2, 0, 0]
    assert list(r["out_tokens"][0]) == [5, 5, 5]
    assert list(r["out_tokens"][1]) == [2, -1, -1]
    assert list(r["out_tokens"][2]) == [5, -1, -1]
    # -0.0 and +0.0 are the same value: the first one wins
    z2 = np.full((1, 2, 4), -1.0, np.float32)
    z2[0, :, 1] = -0.0
    z2[0, :, 3] = 0.0
    r2 = oracle_mod.verify_chain(z2, W.FP32, np.array([[3]], np.int32), np.zeros(1, np.float32),
                                 np.zeros((1, 2), np.float32))
    assert r2["num_accepted"][0] == 0 and r2["out_tokens"][0, 0] == 1


def test_greedy_out_of_range_token_is_a_rejection(oracle_mod):
    x = W.chain_greedy(seed=14, B=4, k=3, V=100, p_match=1.0, dtype=W.FP32)
    x.draft_tokens[:, 1] = np.array([-1, 100, 1 << 30, -(1 << 30)], np.int32)
    r = oracle_mod.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample)
    assert (r["num_accepted"] == 1).all()


# --------------------------------------------------------------- sampled ----
def test_q_equal_p_accepts_everything(oracle_mod):
    """p/q = 1 > u for every u in [0, 1): every draft is accepted (modulo the
    |u - p/q| < 1e-6 window where fp32 storage of q can tip the comparison)."""
    g = np.random.default_rng(21)
    B, k, V, T = 200, 4, 50, 0.9
    z = (g.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    q = _softmax64(z[:, :k], T).astype(np.float32)
    tok = np.stack([[g.choice(V, p=q[b, i] / q[b, i].sum()) for i in range(k)] for b in range(B)]).astype(np.int32)
    ua = W.method_uniforms(g, (B, k))
    ua[:5, :] = np.float32(1.0 - 2.0 ** -24)   # the largest possible uniform
    us = W.method_uniforms(g, (B, k + 1))
    r = oracle_mod.verify_chain(z, W.FP32, tok, np.full(B, T, np.float32), us, q, ua)
    ok = (r["num_accepted"] == k) | (r["flag_accept"].sum(axis=1) > 0)
    assert ok.all()
    assert (r["num_accepted"] == k).mean() > 0.9


def test_accept_probability_is_overlap_mass(oracle_mod):
    """EAGLE-3 review: q(x) A(x) = min(p(x), q(x)), so P(accept) = sum_x min(p, q)."""
    g = np.random.default_rng(22)
    V, T, n = 6, 1.0, 200000
    zp = g.standard_normal(V) * 1.5
    zq = zp + g.standard_normal(V)
    p = _softmax64(zp, T)
    q = _softmax64(zq, 1.0).astype(np.float32)
    x = W.chain_fixed_rows(23, n, np.stack([zp, zp]).astype(np.float32), q[None, :], temperature=T)
    r = oracle_mod.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample,
                                x.draft_probs, x.u_accept)
    alpha = np.minimum(p, q.astype(np.float64)).sum()
    acc = (r["num_accepted"] >= 1).mean()
    se = np.sqrt(alpha * (1 - alpha) / n)
    assert abs(acc - alpha) < 4 * se


def _residual_token_numpy(z, T, q, u):
    """numpy cumsum + searchsorted(side='right') on max(0, p - q)."""
    p = _softmax64(z, T)
    r = np.maximum(0.0, p - q.astype(np.float64))
    if r.sum() == 0.0:
        r = p
    c = np.cumsum(r)
    return int(np.searchsorted(c, u * c[-1], side="right")), c, u * c[-1]


def test_residual_sampler_is_inverse_cdf(oracle_mod):
    """The resample at the rejected row reduces to numpy's cumsum + searchsorted."""
    g = np.random.default_rng(24)
    B, k, V, T = 300, 3, 257, 0.8
    z = (g.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    q = _softmax64(z[:, :k] + g.standard_normal((B, k, V)), 1.0).astype(np.float32)
    tok = g.integers(0, V, size=(B, k)).astype(np.int32)
    ua = W.method_uniforms(g, (B, k))
    us = W.method_uniforms(g, (B, k + 1))
    r = oracle_mod.verify_chain(z, W.FP32, tok, np.full(B, T, np.float32), us, q, ua)
    checked = 0
    for b in range(B):
        a = r["num_accepted"][b]
        if a == k:
            continue
        j, c, t = _residual_token_numpy(z[b, a], T, q[b, a], float(us[b, a]))
        if not r["flag_sample"][b]:
            assert r["out_tokens"][b, a] == j
            checked += 1
    assert checked > 200


def test_bonus_sampler_is_inverse_cdf(oracle_mod):
    """u_accept = 0 accepts every draft (0 < p/q); the bonus is then the inverse
    CDF of p at row k with u_sample[b, k]."""
    g = np.random.default_rng(25)
    B, k, V, T = 200, 2, 300, 1.3
    z = (g.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    q = _softmax64(z[:, :k], 1.0).astype(np.float32)
    tok = g.integers(0, V, size=(B, k)).astype(np.int32)
    ua = np.zeros((B, k), np.float32)
    us = W.method_uniforms(g, (B, k + 1))
    r = oracle_mod.verify_chain(z, W.FP32, tok, np.full(B, T, np.float32), us, q, ua)
    assert (r["num_accepted"] == k).all()
    for b in range(B):
        p = _softmax64(z[b, k], T)
        c = np.cumsum(p)
        j = int(np.searchsorted(c, float(us[b, k]) * c[-1], side="right"))
        assert r["flag_sample"][b] or r["out_tokens"][b, k] == j
        assert (r["out_tokens"][b, :k] == tok[b]).all()


def sampled_edge_violations(O, lib=None):
    """Sampled drafts at the edges of the accept rule.  A draft with q(x) = 0
    and p(x) > 0 has p/q = inf > u: accepted, even at the largest uniform.  A
    draft outside [0, V) has p(x) = 0, so p/q = 0 and it is rejected for any u
    (here u = 0); the token at that position is the residual draw, numpy
    cumsum + searchsorted on max(0, p - q).  Returns the number of requests
    that break either rule."""
    g = np.random.default_rng(27)
    B, k, V, T = 40, 2, 64, 1.0
    z = (g.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    q = _softmax64(z[:, :k] + g.standard_normal((B, k, V)), 1.0).astype(np.float32)
    tok = g.integers(0, V, size=(B, k)).astype(np.int32)
    ua = W.method_uniforms(g, (B, k))
    us = W.method_uniforms(g, (B, k + 1))
    h = B // 2
    q[np.arange(h), 0, tok[:h, 0]] = 0.0            # first half: q(x) = 0 at position 0
    ua[:h, 0] = np.float32(1.0 - 2.0 ** -24)
    tok[h:, 0] = np.array([V, -1, V + 7, 1 << 30] * (B // 8), np.int32)[:B - h]
    ua[h:, 0] = 0.0                                 # second half: out of range at position 0
    r = O.verify_chain(z, W.FP32, tok, np.full(B, T, np.float32), us, q, ua, lib=lib)
    bad = int((r["num_accepted"][:h] < 1).sum())
    for b in range(h, B):
        j, _, _ = _residual_token_numpy(z[b, 0], T, q[b, 0], float(us[b, 0]))
        bad += int(r["num_accepted"][b] != 0 or (not r["flag_sample"][b] and r["out_tokens"][b, 0] != j))
    return bad


def test_sampled_q_zero_accepts_and_out_of_range_rejects(oracle_mod):
    assert sampled_edge_violations(oracle_mod) == 0


def u_zero_violations(O, lib=None):
    """u = 0 gives t = 0, and the inverse CDF takes the smallest j whose prefix
    exceeds t: the first token with mass, never a zero-mass token before it.
    Bonus draws (first half): row 1's first five logits are -inf, so p = 0
    there.  Residual draws (second half): q puts 0.2 on each of tokens 0..4,
    above p, so max(0, p - q) is 0 there; the draft (token 0) is rejected at
    the largest uniform.  Both must give token 5, as numpy searchsorted does."""
    g = np.random.default_rng(28)
    B, k, V, T = 16, 1, 40, 1.0
    h = B // 2
    z = g.standard_normal((B, k + 1, V)).astype(np.float32)
    z[:h, 1, :5] = -np.inf
    q = np.zeros((B, k, V), np.float32)
    q[:, 0, 10] = 1.0                              # first half: the draft (10) is accepted at u = 0
    q[h:, 0, :] = 0.0
    q[h:, 0, :5] = 0.2
    tok = np.full((B, k), 10, np.int32)
    tok[h:, 0] = 0
    ua = np.zeros((B, k), np.float32)
    ua[h:, 0] = np.float32(1.0 - 2.0 ** -24)
    us = np.zeros((B, k + 1), np.float32)
    r = O.verify_chain(z, W.FP32, tok, np.full(B, T, np.float32), us, q, ua, lib=lib)
    bad = int((r["num_accepted"][:h] != 1).sum() + (r["num_accepted"][h:] != 0).sum())
    for b in range(B):
        a = 1 if b < h else 0
        if b < h:
            c = np.cumsum(_softmax64(z[b, 1], T))
            j = int(np.searchsorted(c, 0.0, side="right"))
        else:
            j, _, _ = _residual_token_numpy(z[b, 0], T, q[b, 0], 0.0)
        bad += int(j != 5 or r["out_tokens"][b, a] != 5)
    return bad


def test_draws_at_u_zero_skip_zero_mass_tokens(oracle_mod):
    assert u_zero_violations(oracle_mod) == 0


@pytest.mark.parametrize("lam", [0.1, 0.6])
def test_bench_chain_bytes_match_the_oracle(oracle_mod, lam):
    """The benchmark's algorithmic bytes come from num_accepted and the
    temperatures alone; on a mixed greedy / sampled batch they equal the
    oracle's own count, request by request."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    x = W.chain_mixed(seed=91, B=24, k=4, V=3001, lam=lam)
    r = oracle_mod.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample,
                                x.draft_probs, x.u_accept)
    assert 0 < (x.temperature > 0).sum() < x.B
    for b in range(x.B):
        alg, _, _ = bench.chain_bytes(r["num_accepted"][b:b + 1], x.temperature[b:b + 1], x.k, x.V, 2)
        assert alg == r["b_alg"][b], b


def test_bench_greedy_tree_bytes_match_the_oracle(oracle_mod):
    """The benchmark's greedy-tree algorithmic bytes (root, accepted nodes with
    children, the chosen node) equal the oracle's own count."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    t = W.tree_greedy(seed=57, B=24, V=501, children_per_level=(4, 2, 2, 1, 1), p_match=0.7)
    r = oracle_mod.verify_tree(t.logits, t.dtype, t.node_tokens, t.parent)
    g = np.argmax(W.logits_as_f32(t.logits, t.dtype), axis=-1)
    assert (r["length"] > 2).any()
    for b in range(t.B):
        got = bench.tree_greedy_bytes(t.parent, t.node_tokens[b:b + 1], g[b:b + 1], r["path"][b:b + 1],
                                      r["length"][b:b + 1], t.V, 2)
        assert got == r["b_alg"][b], b


def test_zero_drafts_emit_the_row0_token(oracle_mod):
    """A request with no drafts (k = 0, ragged batches) accepts nothing and emits
    the bonus token of row 0: numpy argmax when greedy, else the inverse CDF of
    p_0 (numpy cumsum + searchsorted) at u_sample[b, 0]."""
    g = np.random.default_rng(26)
    B, V, T = 64, 333, 0.9
    z = (g.standard_normal((B, 1, V)) * 2).astype(np.float32)
    us = W.method_uniforms(g, (B, 1))
    tok = np.zeros((B, 0), np.int32)
    r = oracle_mod.verify_chain(z, W.FP32, tok, np.zeros(B, np.float32), us)
    assert (r["num_accepted"] == 0).all()
    assert (r["out_tokens"][:, 0] == np.argmax(z[:, 0], axis=-1)).all()
    r = oracle_mod.verify_chain(z, W.FP32, tok, np.full(B, T, np.float32), us, np.zeros((B, 0, V), np.float32),
                                np.zeros((B, 0), np.float32))
    assert (r["num_accepted"] == 0).all()
    for b in range(B):
        c = np.cumsum(_softmax64(z[b, 0], T))
        j = int(np.searchsorted(c, float(us[b, 0]) * c[-1], side="right"))
        assert r["flag_sample"][b] or r["out_tokens"][b, 0] == j


def _lossless_case(seed, V=8, k=4, T=1.0):
    g = np.random.default_rng(seed)
    zp = (g.standard_normal((k + 1, V)) * 1.2).astype(np.float32)
    zq = zp[:k] + g.standard_normal((k, V)) * 1.0
    q = _softmax64(zq, 1.0).astype(np.float32)
    return zp, q


def _chi2_pvalues(out_tokens, num_accepted, zp, T):
    k1, V = zp.shape
    pv = []
    for i in range(k1):
        sel = num_accepted >= i
        obs = np.bincount(out_tokens[sel, i], minlength=V)[:V]
        p = _softmax64(zp[i], T)
        pv.append(stats.chisquare(obs, p * sel.sum()).pvalue)
    return pv


def test_lossless_chi_square(oracle_mod):
    """EAGLE-3 review (identity min(p,q) + max(0,p-q) = p) and the serving-book
    acceptance rule: the emitted token at every output index follows p of that
    row.  10^6 trials on V = 8, k = 4; chi-square p-value > 0.01 per index."""
    zp, q = _lossless_case(31)
    x = W.chain_fixed_rows(32, 1_000_000, zp, q, temperature=1.0)
    r = oracle_mod.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample,
                                x.draft_probs, x.u_accept, nthreads=os.cpu_count() or 1)
    pv = _chi2_pvalues(r["out_tokens"], r["num_accepted"], zp, 1.0)
    assert min(pv) > 0.01, pv


# ---------------------------------------------------------------- counts ----
def _expected_tokens(alpha, k):
    return (1 - alpha ** (k + 1)) / (1 - alpha)


def _golden_table():
    rows = {}
    with open(os.path.join(GOLDEN, "expected_tokens_table.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            a, *v = line.split()
            rows[float(a)] = dict(zip((2, 4, 8), map(float, v)))
    return rows


def test_expected_tokens_formula_matches_printed_table():
    for alpha, row in _golden_table().items():
        for k, v in row.items():
            assert round(_expected_tokens(alpha, k), 2) == pytest.approx(v, abs=1e-9)
    assert _expected_tokens(0.8, 4) == pytest.approx(3.3616, abs=1e-12)


@pytest.mark.parametrize("alpha", [0.6, 0.8, 0.9])
@pytest.mark.parametrize("k", [2, 4, 8])
def test_mean_tokens_per_step_matches_table(oracle_mod, alpha, k):
    """V = 2, p = (1/2, 1/2), q = (1/2 + d, 1/2 - d): per-token acceptance is
    sum min(p, q) = 1 - d = alpha, so E[a + 1] = (1 - alpha^(k+1)) / (1 - alpha)."""
    d = 1.0 - alpha
    zp = np.zeros((k + 1, 2), np.float32)
    q = np.tile(np.array([0.5 + d, 0.5 - d], np.float32), (k, 1))
    n = 200_000
    x = W.chain_fixed_rows(40 + k, n, zp, q, temperature=1.0)
    r = oracle_mod.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample,
                                x.draft_probs, x.u_accept, nthreads=os.cpu_count() or 1)
    t = r["num_accepted"].astype(np.float64) + 1
    se = t.std(ddof=1) / np.sqrt(n)
    alpha_eff = np.minimum(0.5, q[0].astype(np.float64)).sum()
    assert abs(t.mean() - _expected_tokens(alpha_eff, k)) < 4 * se
    assert abs(t.mean() - _golden_table()[alpha][k]) < 4 * se + 0.005


def test_tiny_chain_tokens_per_step(oracle_mod):
    """Fixed rows: E[a + 1] = sum_i prod_{j<i} alpha_j with alpha_j = sum min(p_j, q_j)."""
    x = W.chain_tiny(seed=1, trials=1000)
    p = _softmax64(x.meta["target_rows"], 1.0)
    q = x.meta["q_rows"].astype(np.float64)
    al = np.minimum(p[:x.k], q).sum(axis=1)
    expect = sum(np.prod(al[:i]) for i in range(x.k + 1))
    r = oracle_mod.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample,
                                x.draft_probs, x.u_accept)
    t = r["num_accepted"] + 1.0
    se = t.std(ddof=1) / np.sqrt(len(t))
    assert abs(t.mean() - expect) < 4 * se
    assert (t >= 1).all()                 # at least one token per step


# ------------------------------------------------------------------ tree ----
def _tree_bruteforce(zf, toks, parent):
    """Enumerate every root-to-node path and keep the deepest one whose every
    edge matches the parent's argmax (first one found at that depth)."""
    N = len(parent) - 1
    g = np.argmax(zf, axis=-1)
    best_path = [0]
    for n in range(1, N + 1):
        path = [n]
        while path[-1] != 0:
            path.append(int(parent[path[-1]]))
        path = path[::-1]
        if all(toks[c - 1] == g[path[i]] for i, c in enumerate(path[1:])):
            if len(path) > len(best_path):
                best_path = path
    out = [int(toks[c - 1]) for c in best_path[1:]] + [int(g[best_path[-1]])]
    return best_path, out


def test_tree_metadata_matches_worked_example(oracle_mod):
    vals = {}
    with open(os.path.join(GOLDEN, "tree_levels.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *v = line.split()
            vals[key] = [int(t) for t in v]
    choices = W.level_tree_choices((4, 2, 2, 1, 1))
    m = oracle_mod.tree_level_metadata(choices)
    assert m["num_drafts_per_level"] == vals["num_drafts_per_level"]
    assert m["cu_drafts_per_level"] == vals["cu_drafts_per_level"]
    assert m["child_drafts_per_level"] == vals["child_drafts_per_level"]
    assert m["depth"] == vals["depth"][0]
    assert (oracle_mod.parent_from_choices(choices) == W.parents_in_order((4, 2, 2, 1, 1))).all()


@pytest.mark.parametrize("shape", [(4, 2, 2, 1, 1), (3, 3, 1), (1, 1, 1, 1), (5,)])
def test_tree_matches_bruteforce(oracle_mod, shape):
    t = W.tree_greedy(seed=50 + len(shape), B=12, V=97, children_per_level=shape, p_match=0.75)
    r = oracle_mod.verify_tree(t.logits, t.dtype, t.node_tokens, t.parent)
    zf = W.logits_as_f32(t.logits, t.dtype)
    D = len(shape)
    for b in range(t.B):
        path, out = _tree_bruteforce(zf[b], t.node_tokens[b], t.parent)
        assert r["length"][b] == len(path)
        assert list(r["path"][b, :len(path)]) == path
        assert (r["path"][b, len(path):] == -1).all()
        assert list(r["tokens"][b, :len(path)]) == out
        assert (r["tokens"][b, len(path):] == -1).all()
        assert r["path"].shape[1] == D + 1


def test_tree_sibling_tie_takes_smallest_index(oracle_mod):
    parent = W.parents_in_order((3, 1))       # root -> 1,2,3 ; 1->4, 2->5, 3->6
    V = 10
    z = np.zeros((1, 7, V), np.float32)
    z[0, 0, 7] = 1.0     # root argmax 7
    z[0, 1, 2] = 1.0
    z[0, 2, 2] = 1.0
    z[0, 3, 2] = 1.0
    toks = np.array([[9, 7, 7, 2, 2, 2]], np.int32)   # nodes 2 and 3 match; 5 and 6 match
    r = oracle_mod.verify_tree(z, W.FP32, toks, parent)
    assert list(r["path"][0]) == [0, 2, 5]
    assert list(r["tokens"][0]) == [7, 2, 0]


def test_chain_is_a_tree_with_one_child_per_level(oracle_mod):
    """Cross-check: a chain equals a tree with parent[n] = n - 1 on the same data."""
    x = W.chain_greedy(seed=60, B=30, k=6, V=500, p_match=0.8)
    rc = oracle_mod.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample)
    parent = np.arange(-1, x.k, dtype=np.int32)
    rt = oracle_mod.verify_tree(x.logits, x.dtype, x.draft_tokens, parent)
    assert (rt["length"] == rc["num_accepted"] + 1).all()
    assert (rt["tokens"] == rc["out_tokens"]).all()


# ----------------------------------------------------------------- slots ----
def test_slot_fixup_chain_and_tree(oracle_mod):
    g = np.random.default_rng(70)
    B, P = 9, 7
    s = W.slot_map(g, B, P)
    a = np.array([0, 1, 2, 3, 4, 5, 6, 0, 6], np.int32)
    out = oracle_mod.fixup_slots(s, num_accepted=a, pad=-1)
    for b in range(B):
        assert (out[b, :a[b] + 1] == s[b, :a[b] + 1]).all()       # kept bit-exact
        assert (out[b, a[b] + 1:] == -1).all()
    path = np.full((B, 3), -1, np.int32)
    path[:, 0] = 0
    path[1, 1:] = [3, 5]
    path[2, 1] = 6
    out = oracle_mod.fixup_slots(s, path=path, pad=-7)
    assert (out[0] == np.r_[s[0, 0], [-7] * 6]).all()
    assert (out[1] == np.array([s[1, 0], -7, -7, s[1, 3], -7, s[1, 5], -7])).all()
    assert (out[2, 6] == s[2, 6]) and (out[2, 1:6] == -7).all()
