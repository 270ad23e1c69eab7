"""Pins of the oracle's n-gram lookup drafting (serving-book chapter, table of
draft sources, row "n-gram lookup": propose what follows an earlier copy of the
text's current ending).

None of these re-types the oracle's loops: hand-worked examples (golden file),
numpy's sliding-window comparison as an independent search, and invariants any
correct answer satisfies.
"""
import os

import numpy as np
import pytest
from numpy.lib.stride_tricks import sliding_window_view

from speculative_decoding_verification_chain_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ngram_examples.txt")


def _golden():
    out = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        a, b, c, d = [x.strip() for x in line.split("|")]
        toks = [] if a == "-" else [int(v) for v in a.split()]
        nmin, nmax, k = map(int, b.split())
        out.append((toks, nmin, nmax, k, [int(v) for v in c.split()], tuple(map(int, d.split()))))
    return out


def test_hand_worked_examples(oracle_mod):
    cases = _golden()
    assert len(cases) >= 8
    for toks, nmin, nmax, k, draft, (ml, me) in cases:
        t = np.zeros((1, max(1, len(toks))), np.int32)
        t[0, :len(toks)] = toks
        r = oracle_mod.ngram_propose(t, np.array([len(toks)], np.int32), nmin, nmax, k)
        assert r["draft"][0].tolist() == draft, toks
        assert (r["match_len"][0], r["match_end"][0]) == (ml, me), toks
        assert r["count"][0] == sum(1 for v in draft if v >= 0)


def _numpy_search(s, nmin, nmax):
    """Longest ending with an earlier copy, then its latest copy, via numpy's
    sliding windows over the text before the last token."""
    L = len(s)
    for n in range(min(nmax, L - 1), nmin - 1, -1):
        win = sliding_window_view(s[:L - 1], n)          # windows ending at e = i + n - 1 <= L - 2
        hits = np.flatnonzero((win == s[L - n:]).all(axis=1))
        if hits.size:
            return n, int(hits[-1]) + n - 1
    return 0, -1


@pytest.mark.parametrize("V", [2, 3, 50])
def test_matches_numpy_sliding_windows(oracle_mod, V):
    g = np.random.default_rng(70 + V)
    B, Lmax = 300, 60
    t = g.integers(0, V, size=(B, Lmax)).astype(np.int32)
    ln = g.integers(0, Lmax + 1, size=B).astype(np.int32)
    for nmin, nmax, k in ((1, 4, 5), (2, 6, 3), (3, 3, 8)):
        r = oracle_mod.ngram_propose(t, ln, nmin, nmax, k)
        for b in range(B):
            s = t[b, :ln[b]]
            n, e = _numpy_search(s, nmin, nmax)
            assert (r["match_len"][b], r["match_end"][b]) == (n, e)
            exp = list(s[e + 1:e + 1 + k]) if e >= 0 else []
            assert r["draft"][b].tolist() == exp + [-1] * (k - len(exp))


def test_invariants_on_copy_heavy_texts(oracle_mod):
    t, ln = W.ngram_texts(seed=71, B=40, Lmax=3000, V=500)
    nmin, nmax, k = 2, 8, 6
    r = oracle_mod.ngram_propose(t, ln, nmin, nmax, k)
    found = 0
    for b in range(40):
        s, L = t[b], int(ln[b])
        n, e, c = int(r["match_len"][b]), int(r["match_end"][b]), int(r["count"][b])
        if e < 0:
            assert n == 0 and c == 0 and (r["draft"][b] == -1).all()
            continue
        found += 1
        assert nmin <= n <= nmax and n - 1 <= e <= L - 2
        assert (s[e - n + 1:e + 1] == s[L - n:L]).all()        # the copy matches the ending
        assert c == min(k, L - 1 - e) and (r["draft"][b, :c] == s[e + 1:e + 1 + c]).all()
        for e2 in range(e + 1, L - 1):                         # no later copy of this length
            assert not (e2 - n + 1 >= 0 and (s[e2 - n + 1:e2 + 1] == s[L - n:L]).all())
    assert found >= 12   # endings inside copied spans
