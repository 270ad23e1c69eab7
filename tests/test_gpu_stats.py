"""Statistical laws the pages state, checked on the CUDA path itself.

* Lossless (EAGLE-3 review: min(p,q) + max(0,p-q) = p; serving-book acceptance
  rule): the emitted token at each output index follows p of that row,
  chi-square over 10^6 trials on V = 8, k = 4, p-value > 0.01.
* Expected tokens per step (serving-book "expected number of tokens"):
  (1 - alpha^(k+1)) / (1 - alpha) under constant acceptance alpha.
"""
import numpy as np
import pytest
from scipy import stats

from speculative_decoding_verification_chain_gb300 import workloads as W

from helpers import run_chain

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for gpu-marked tests")
    return torch.device("cuda", 0)


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_chain_gb300 as m
    m.load_library()
    return m


@pytest.fixture(autouse=True, params=[0, 1, 2], ids=["auto", "persistent", "cluster"])
def chain_path(request, sv):
    """The kernel that verifies: path 0 (automatic) sends sampled padded chains
    whose per-request clusters fit on the GPU to the chain cluster kernel, and
    greedy trees and small greedy padded chains to the greedy cluster kernel;
    path 1 sends every batch to the persistent kernel; path 2 is path 0 with
    every greedy padded chain on the greedy cluster kernel.  Tests of ragged batches, the separate fix-up, n-gram
    lookup and next-step preparation do not depend on it and run once; trees
    run on paths 0 and 1."""
    path = request.param
    name = request.node.name
    if path != 0 and any(w in name for w in ("fixup_slots", "ragged", "ngram", "next_step", "kv")):
        pytest.skip("the path applies to padded chains and trees only")
    if path == 2 and "tree" in name:
        pytest.skip("trees take the same kernel on paths 0 and 2")
    sv.set_tuning(0, 0, path)
    yield path
    sv.set_tuning(0, 0, 0)


def _softmax64(z, T):
    s = np.asarray(z, np.float64) / T
    e = np.exp(s - s.max(-1, keepdims=True))
    return e / e.sum(-1, keepdims=True)


def test_lossless_chi_square_on_gpu(sv, dev):
    g = np.random.default_rng(131)
    V, k = 8, 4
    zp = (g.standard_normal((k + 1, V)) * 1.2).astype(np.float32)
    q = _softmax64(zp[:k] + g.standard_normal((k, V)), 1.0).astype(np.float32)
    x = W.chain_fixed_rows(132, 1_000_000, zp, q, temperature=1.0)
    got_t, got_a = run_chain(sv, x, dev)
    for i in range(k + 1):
        sel = got_a >= i
        obs = np.bincount(got_t[sel, i], minlength=V)[:V]
        pv = stats.chisquare(obs, _softmax64(zp[i], 1.0) * sel.sum()).pvalue
        assert pv > 0.01, (i, pv)


@pytest.mark.parametrize("alpha", [0.6, 0.8, 0.9])
@pytest.mark.parametrize("k", [2, 4, 8])
def test_mean_tokens_per_step_on_gpu(sv, dev, alpha, k):
    d = 1.0 - alpha
    zp = np.zeros((k + 1, 2), np.float32)
    q = np.tile(np.array([0.5 + d, 0.5 - d], np.float32), (k, 1))
    n = 200_000
    x = W.chain_fixed_rows(140 + k, n, zp, q, temperature=1.0)
    got_t, got_a = run_chain(sv, x, dev)
    t = got_a.astype(np.float64) + 1
    a_eff = np.minimum(0.5, q[0].astype(np.float64)).sum()
    expect = (1 - a_eff ** (k + 1)) / (1 - a_eff)
    assert abs(t.mean() - expect) < 4 * t.std(ddof=1) / np.sqrt(n)
