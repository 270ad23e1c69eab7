"""The pins must catch plausible mistakes in the oracle.

Each case copies spec_oracle.c, plants one mistake (a flipped sign, a dropped
clip, a wrong row or index, a reversed comparison, a dropped ancestor term),
compiles the copy on the CPU and checks that the corresponding pin fails on it
while passing on the real oracle.
"""
import os
import subprocess

import numpy as np
import pytest

from speculative_decoding_verification_chain_gb300 import workloads as W

import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "spec_oracle.c")


def _mutant(tmp_path, old, new, tag):
    src = open(SRC).read()
    assert src.count(old) == 1, old
    path = tmp_path / ("mut_%s.c" % tag)
    path.write_text(src.replace(old, new))
    so = tmp_path / ("libmut_%s.so" % tag)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           "-o", str(so), str(path), "-lm", "-lpthread"])
    from oracle import oracle as O
    return O.load_library(str(so))


def _lossless(O, lib):
    zp, q = pins._lossless_case(31)
    x = W.chain_fixed_rows(32, 300_000, zp, q, temperature=1.0)
    r = O.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample,
                       x.draft_probs, x.u_accept, nthreads=os.cpu_count() or 1, lib=lib)
    return min(pins._chi2_pvalues(r["out_tokens"], r["num_accepted"], zp, 1.0))


def _residual_mismatches(O, lib):
    g = np.random.default_rng(24)
    B, k, V, T = 120, 3, 257, 0.8
    z = (g.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    q = pins._softmax64(z[:, :k] + g.standard_normal((B, k, V)), 1.0).astype(np.float32)
    tok = g.integers(0, V, size=(B, k)).astype(np.int32)
    ua = W.method_uniforms(g, (B, k))
    us = W.method_uniforms(g, (B, k + 1))
    r = O.verify_chain(z, W.FP32, tok, np.full(B, T, np.float32), us, q, ua, lib=lib)
    bad = 0
    for b in range(B):
        a = r["num_accepted"][b]
        if a < k:
            j, _, _ = pins._residual_token_numpy(z[b, a], T, q[b, a], float(us[b, a]))
            bad += int(r["out_tokens"][b, a] != j)
    return bad


def _bonus_mismatches(O, lib):
    g = np.random.default_rng(25)
    B, k, V, T = 100, 2, 300, 1.3
    z = (g.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    q = pins._softmax64(z[:, :k], 1.0).astype(np.float32)
    tok = g.integers(0, V, size=(B, k)).astype(np.int32)
    us = W.method_uniforms(g, (B, k + 1))
    r = O.verify_chain(z, W.FP32, tok, np.full(B, T, np.float32), us, q,
                       np.zeros((B, k), np.float32), lib=lib)
    bad = 0
    for b in range(B):
        c = np.cumsum(pins._softmax64(z[b, k], T))
        bad += int(r["out_tokens"][b, k] != np.searchsorted(c, float(us[b, k]) * c[-1], side="right"))
    return bad


def _accept_rate_z(O, lib):
    g = np.random.default_rng(22)
    V, n = 6, 100000
    zp = g.standard_normal(V) * 1.5
    q = pins._softmax64(zp + g.standard_normal(V), 1.0).astype(np.float32)
    x = W.chain_fixed_rows(23, n, np.stack([zp, zp]).astype(np.float32), q[None, :])
    r = O.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample,
                       x.draft_probs, x.u_accept, lib=lib)
    alpha = np.minimum(pins._softmax64(zp, 1.0), q.astype(np.float64)).sum()
    acc = (r["num_accepted"] >= 1).mean()
    return abs(acc - alpha) / np.sqrt(alpha * (1 - alpha) / n)


def _tie_ok(O, lib):
    z = np.zeros((1, 2, 16), np.float32)
    z[0, :, 3] = 5.0
    z[0, :, 9] = 5.0
    r = O.verify_chain(z, W.FP32, np.array([[9]], np.int32), np.zeros(1, np.float32),
                       np.zeros((1, 2), np.float32), lib=lib)
    return r["num_accepted"][0] == 0 and r["out_tokens"][0, 0] == 3


def _tree_mismatches(O, lib):
    t = W.tree_greedy(seed=55, B=12, V=97, children_per_level=(4, 2, 2, 1, 1), p_match=0.75)
    r = O.verify_tree(t.logits, t.dtype, t.node_tokens, t.parent, lib=lib)
    zf = W.logits_as_f32(t.logits, t.dtype)
    bad = 0
    for b in range(t.B):
        path, out = pins._tree_bruteforce(zf[b], t.node_tokens[b], t.parent)
        bad += int(list(r["tokens"][b, :len(path)]) != out or r["length"][b] != len(path)
                   or r["path"][b, :len(path)].tolist() != list(path))
    return bad


def _ngram_mismatches(O, lib):
    import test_oracle_ngram as ng
    g = np.random.default_rng(72)
    B, Lmax = 200, 50
    t = g.integers(0, 3, size=(B, Lmax)).astype(np.int32)
    ln = g.integers(0, Lmax + 1, size=B).astype(np.int32)
    r = O.ngram_propose(t, ln, 1, 5, 4, lib=lib)
    bad = 0
    for b in range(B):
        s = t[b, :ln[b]]
        n, e = ng._numpy_search(s, 1, 5)
        draft = [int(v) for v in s[e + 1:e + 5]] if e >= 0 else []
        bad += int((r["match_len"][b], r["match_end"][b]) != (n, e) or r["count"][b] != len(draft)
                   or r["draft"][b].tolist() != draft + [-1] * (4 - len(draft)))
    return bad


def _tree_law(O, lib):
    import test_oracle_tree_sampled as ts
    c = ts.law_case(seed=52, trials=200_000)
    pv = ts.law_pvalues(c, ts.run(O, c, lib=lib))
    return min(pv["first"], pv["sibling"], pv["second"])


def _tree_closed_form(O, lib):
    import test_oracle_tree_sampled as ts
    return ts.closed_form_residual_mismatches(O, lib)[0]


def _tree_q_equal_p(O, lib):
    import test_oracle_tree_sampled as ts
    return ts.q_equal_p_mismatches(O, lib)


def _tree_zero_q(O, lib):
    import test_oracle_tree_sampled as ts
    return ts.zero_q_violations(O, lib)


def _next_step_bad(O, lib):
    import test_oracle_next_step as ns
    g = ns.golden_case()
    r = O.prepare_next_step(g["out_tokens"], g["a"], g["pos"], g["bt"], 4, 3, rows_per_req=4, lib=lib)
    return int((r["next_position"] != g["next_position"]).sum() + (r["next_slots"] != g["slots"]).any(axis=1).sum()
               + (r["last_row"] != g["last_row"]).sum() + (r["next_token"] != g["next_token"]).sum())


def _hidden_bad(O, lib):
    """The gathered hidden row is the last accepted position's row, found by
    numpy indexing (padded and ragged row layouts)."""
    import test_oracle_next_step as ns
    out_tokens, a, pos, bt, hid = ns.random_case(52, B=64)
    k1 = out_tokens.shape[1]
    r = O.prepare_next_step(out_tokens, a, pos, bt, 16, 2, rows_per_req=k1, hidden=hid, lib=lib)
    bad = int((r["hidden_out"] != hid[np.arange(len(a)) * k1 + a]).any(axis=1).sum())
    g = np.random.default_rng(62)
    ks = g.integers(0, 8, size=40)
    cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    ot = g.integers(0, 1000, size=(40, 9)).astype(np.int32)
    aa = np.array([g.integers(0, kk + 1) for kk in ks], np.int32)
    hh = g.standard_normal((int(cu[-1]) + 40, 8)).astype(np.float32)
    r = O.prepare_next_step(ot, aa, np.zeros(40, np.int32), np.zeros((40, 1), np.int32), 64, 0, cu=cu,
                            hidden=hh, lib=lib)
    return bad + int((r["hidden_out"] != hh[cu[:-1] + np.arange(40) + aa]).any(axis=1).sum())


def _compaction_bad(O, lib):
    import test_oracle_next_step as ns
    parent = W.parents_in_order((4, 2, 2))
    paths = np.array([[0, 2, 7, 16], [0, 3, 4, 13], [0, 1, 2, -1], [0, 4, 12, 28]], np.int32)
    return ns.compaction_mismatches(O, paths, parent, lib=lib)


def _greedy_bad(O, lib):
    """Greedy chains against brute force (numpy first-occurrence argmax): drafts
    that never, always and sometimes match."""
    bad = 0
    for seed, p_match in ((11, 0.0), (12, 1.0), (13, 0.7)):
        x = W.chain_greedy(seed=seed, B=16, k=5, V=3001, p_match=p_match)
        am = np.argmax(W.logits_as_f32(x.logits, x.dtype), axis=-1)
        r = O.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample, lib=lib)
        for b in range(x.B):
            a = 0
            while a < x.k and x.draft_tokens[b, a] == am[b, a]:
                a += 1
            want = [int(t) for t in x.draft_tokens[b, :a]] + [int(am[b, a])] + [-1] * (x.k - a)
            bad += int(r["num_accepted"][b] != a) + int(r["out_tokens"][b].tolist() != want)
    return bad


def _fixup_bad(O, lib):
    """Slot fix-up by its meaning: a chain keeps slots 0..a, a tree keeps the
    root and its path's nodes; everything else becomes the pad value."""
    g = np.random.default_rng(70)
    B, P = 9, 7
    s = W.slot_map(g, B, P)
    a = np.array([0, 1, 2, 3, 4, 5, 6, 0, 6], np.int32)
    keep = np.arange(P)[None, :] <= a[:, None]
    out = O.fixup_slots(s, num_accepted=a, pad=-1, lib=lib)
    bad = int((out != np.where(keep, s, -1)).any(axis=1).sum())
    path = np.full((B, 3), -1, np.int32)
    path[:, 0] = 0
    path[1, 1:] = [3, 5]
    path[2, 1] = 6
    keep = np.zeros((B, P), bool)
    keep[:, 0] = True
    keep[1, [3, 5]] = True
    keep[2, 6] = True
    out = O.fixup_slots(s, path=path, pad=-7, lib=lib)
    return bad + int((out != np.where(keep, s, -7)).any(axis=1).sum())


_SNAPSHOT_LOOP = """        for (int i = 1; i < L; ++i) {
            const int node = path[(size_t)b * path_stride + i];"""


CASES = [
    ("greedy_emits_draft", "                out[i] = g;\n                a = i;",
     "                out[i] = x;\n                a = i;", lambda O, lib: _greedy_bad(O, lib) > 0),
    ("greedy_accept_reversed", "if (x != g) {", "if (x == g) {", lambda O, lib: _greedy_bad(O, lib) > 0),
    ("fixup_off_by_one", "keep = j <= num_accepted[b];", "keep = j < num_accepted[b];",
     lambda O, lib: _fixup_bad(O, lib) > 0),
    ("fixup_tree_path_stride", "keep = path[(size_t)b * path_stride + i] == j;", "keep = path[(size_t)b + i] == j;",
     lambda O, lib: _fixup_bad(O, lib) > 0),
    ("tree_tie_last", "if (acc[n] && depth[n] > depth[best])", "if (acc[n] && depth[n] >= depth[best])",
     lambda O, lib: _tree_mismatches(O, lib) > 0),
    ("ngram_draft_offset", "v = s[best_e + 1 + j];", "v = s[best_e + j];",
     lambda O, lib: _ngram_mismatches(O, lib) > 0),
    ("next_slot_offset", "slot = (int64_t)e * block_size + pos % block_size;", "slot = (int64_t)e * block_size;",
     lambda O, lib: _next_step_bad(O, lib) > 0),
    ("next_negative_block", "if (e >= 0)\n", "if (1)\n", lambda O, lib: _next_step_bad(O, lib) > 0),
    ("next_hidden_row", "hidden_in + (size_t)r * (size_t)row_bytes", "hidden_in + (size_t)r0 * (size_t)row_bytes",
     lambda O, lib: _hidden_bad(O, lib) > 0),
    ("cdf_ties_inclusive", "        if (c > t) {", "        if (c >= t) {", lambda O, lib: pins.u_zero_violations(O, lib) > 0),
    ("tree_sampled_q_zero_rejects", "if (qh == 0.0) {\n                        accept = 1;",
     "if (qh == 0.0) {\n                        accept = 0;", lambda O, lib: _tree_zero_q(O, lib) > 0),
    ("tree_sampled_out_of_range_accepts", "int accept = 0;", "int accept = 1;",
     lambda O, lib: _tree_zero_q(O, lib) > 0),
    ("q_zero_rejects", "if (qh == 0.0) {\n                    accept = 1;", "if (qh == 0.0) {\n                    accept = 0;",
     lambda O, lib: pins.sampled_edge_violations(O, lib) > 0),
    ("sampled_out_of_range_accepts", "accept = 0; /* out-of-range draft: p(x) = 0 */", "accept = 1;",
     lambda O, lib: pins.sampled_edge_violations(O, lib) > 0),
    ("accept_row_shift", "row_softmax(J->logits, J->dtype, zbase + (size_t)i * row, V, T, p);",
     "row_softmax(J->logits, J->dtype, zbase + (size_t)(i + 1) * row, V, T, p);",
     lambda O, lib: _residual_mismatches(O, lib) > 10),
    ("residual_sign", "double d = p[j] - (double)qi[j];", "double d = (double)qi[j] - p[j];",
     lambda O, lib: _lossless(O, lib) < 1e-6),
    ("residual_noclip", "r[j] = d > 0.0 ? d : 0.0;", "r[j] = d > 0.0 ? d : -d;",
     lambda O, lib: _lossless(O, lib) < 1e-6),
    ("bonus_row", "row_softmax(J->logits, J->dtype, zbase + (size_t)k * row, V, T, p);",
     "row_softmax(J->logits, J->dtype, zbase + (size_t)(k - 1) * row, V, T, p);",
     lambda O, lib: _bonus_mismatches(O, lib) > 10),
    ("accept_reversed", "accept = u < ratio;", "accept = u > ratio;",
     lambda O, lib: _accept_rate_z(O, lib) > 10),
    ("sample_uniform_index", "J->u_sample[(size_t)b * (k + 1) + sampled_row]",
     "J->u_sample[(size_t)b * (k + 1)]", lambda O, lib: _residual_mismatches(O, lib) > 10),
    ("no_temperature", "p[j] = logit_at(z, dtype, off + (size_t)j) / T;",
     "p[j] = logit_at(z, dtype, off + (size_t)j);", lambda O, lib: _bonus_mismatches(O, lib) > 10),
    ("tie_last", "if (v > bv) {", "if (v >= bv) {", lambda O, lib: not _tie_ok(O, lib)),
    ("tree_no_ancestor", "acc[n] = acc[parent[n]] && x == g[parent[n]];",
     "acc[n] = x == g[parent[n]];", lambda O, lib: _tree_mismatches(O, lib) > 0),
    ("tree_parent_row", "acc[n] = acc[parent[n]] && x == g[parent[n]];",
     "acc[n] = acc[parent[n]] && x == g[n];", lambda O, lib: _tree_mismatches(O, lib) > 0),
    ("ngram_earliest", "for (int e = L - 2; e >= n - 1; --e) {", "for (int e = n - 1; e <= L - 2; ++e) {",
     lambda O, lib: _ngram_mismatches(O, lib) > 0),
    ("ngram_shortest_first", "for (int n = n_max; n >= n_min && best_e < 0; --n) {",
     "for (int n = n_min; n <= n_max && best_e < 0; ++n) {", lambda O, lib: _ngram_mismatches(O, lib) > 0),
    ("ngram_self_match", "for (int e = L - 2; e >= n - 1; --e) {", "for (int e = L - 1; e >= n - 1; --e) {",
     lambda O, lib: _ngram_mismatches(O, lib) > 0),
    ("tree_sampled_no_normalise", "w[j] = r / Z;", "w[j] = r;", lambda O, lib: _tree_closed_form(O, lib) > 10),
    ("tree_sampled_no_clip", "Z += r > 0.0 ? r : 0.0;", "Z += r;", lambda O, lib: _tree_closed_form(O, lib) > 10),
    ("tree_sampled_first_sibling_only",
     "                        }\n                    }\n            }\n            if (next < 0)\n",
     "                        }\n                    }\n                n = N;\n            }\n            if (next < 0)\n",
     lambda O, lib: _tree_law(O, lib) < 1e-6),
    ("tree_sampled_child_q_row", "+ (size_t)c) * row : NULL;", "+ (size_t)(c < N ? c + 1 : c)) * row : NULL;",
     lambda O, lib: _tree_law(O, lib) < 1e-6),
    ("tree_sampled_accept_reversed", "accept = ratio > u;", "accept = ratio < u;",
     lambda O, lib: _tree_law(O, lib) < 1e-6),
    ("tree_sampled_uniform_index", "u_sample[(size_t)b * (size_t)(N + 1) + (size_t)c]",
     "u_sample[(size_t)b * (size_t)(N + 1)]", lambda O, lib: _tree_q_equal_p(O, lib) > 10),
    ("next_position_no_bonus", "const int64_t np = (int64_t)positions[b] + a + 1;",
     "const int64_t np = (int64_t)positions[b] + a;", lambda O, lib: _next_step_bad(O, lib) > 0),
    ("next_block_index", "const int64_t blk = pos / block_size;", "const int64_t blk = (pos + 1) / block_size;",
     lambda O, lib: _next_step_bad(O, lib) > 0),
    ("next_last_row", "const int64_t r = r0 + a;", "const int64_t r = r0;", lambda O, lib: _next_step_bad(O, lib) > 0),
    ("next_token_row", "next_token[b] = out_tokens[(size_t)b * out_stride + a];",
     "next_token[b] = out_tokens[(size_t)b * out_stride + (a > 0 ? a - 1 : 0)];",
     lambda O, lib: _next_step_bad(O, lib) > 0),
    ("compaction_descending_in_place", _SNAPSHOT_LOOP,
     """        for (int i = L - 1; i >= 1; --i) {
            const int node = path[(size_t)b * path_stride + i];
            if (node > 0 && node < slot_stride && node != i && slot_mapping[(size_t)b * slot_stride + node] >= 0)
                memmove(kv + (size_t)slot_mapping[(size_t)b * slot_stride + i] * (size_t)row_bytes,
                        kv + (size_t)slot_mapping[(size_t)b * slot_stride + node] * (size_t)row_bytes,
                        (size_t)row_bytes);
            continue;""", lambda O, lib: _compaction_bad(O, lib) > 0),
    ("compaction_wrong_destination", "const int64_t s_dst = slot_mapping[(size_t)b * slot_stride + i];",
     "const int64_t s_dst = slot_mapping[(size_t)b * slot_stride + i - 1];",
     lambda O, lib: _compaction_bad(O, lib) > 0),
]


def test_real_oracle_passes_the_mutation_checks(oracle_mod):
    O = oracle_mod
    lib = O._load()
    assert _lossless(O, lib) > 0.01
    assert _residual_mismatches(O, lib) == 0
    assert _bonus_mismatches(O, lib) == 0
    assert _accept_rate_z(O, lib) < 4
    assert _tie_ok(O, lib)
    assert _tree_mismatches(O, lib) == 0
    assert _ngram_mismatches(O, lib) == 0
    assert _tree_law(O, lib) > 0.01
    assert _tree_closed_form(O, lib) == 0
    assert _tree_q_equal_p(O, lib) == 0
    assert _next_step_bad(O, lib) == 0
    assert _compaction_bad(O, lib) == 0
    assert _greedy_bad(O, lib) == 0
    assert _fixup_bad(O, lib) == 0
    assert pins.sampled_edge_violations(O, lib) == 0
    assert _hidden_bad(O, lib) == 0
    assert pins.u_zero_violations(O, lib) == 0
    assert _tree_zero_q(O, lib) == 0


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_planted_mistake_is_caught(oracle_mod, tmp_path, case):
    tag, old, new, caught = case
    lib = _mutant(tmp_path, old, new, tag)
    assert caught(oracle_mod, lib)
