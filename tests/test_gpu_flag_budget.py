"""Flag budget of the sampled paths, measured at full size.

Sampled tokens may differ from the oracle's only at positions the oracle
flags: an accept test with |u - p(x)/q(x)| below 1e-6, or an inverse-CDF
threshold t within 1e-5 (relative) of a bucket edge (EAGLE-3 review,
"Speculative Decoding": accept with min(1, p/q), resample from
norm(max(0, p - q)); serving-book chapter, acceptance rule).  Here the GPU
path runs over many independent trials of each full-size sampled workload
(the same rows, fresh draft tokens and uniforms per trial) and the run counts,
over all positions (B x (k+1) target rows, or B x (N+1) tree nodes):

  flagged  positions the oracle flags (a property of the workload and the
           windows, not of the kernel);
  differ   positions where the GPU's result differs from the oracle's.

Every difference must sit at the flag of the decision that made it, and the
differences over all positions of all these workloads together must stay
below 1e-4 of them (per workload the counts are too small for a rate of that
size to be tested on its own: a few thousand positions each).  Both fractions,
and the achieved acceptance rate per lambda, are printed per workload in the
run's summary.
"""
import numpy as np
import pytest

from speculative_decoding_verification_chain_gb300 import workloads as W

from helpers import count_chain, count_tree_sampled, cuda, oracle_chain

pytestmark = pytest.mark.gpu

BUDGET = 1e-4   # differences per position
_ALL = {}       # counts over every workload run in this module


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for gpu-marked tests")
    return torch.device("cuda", 0)


@pytest.fixture(scope="module")
def O(oracle_mod):
    return oracle_mod


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_chain_gb300 as m
    m.load_library()
    return m


def _add(tot, c):
    for key, v in c.items():
        tot[key] = tot.get(key, 0) + v


def _chain_trials(sv, O, dev, x, trials, seed0):
    """GPU and oracle over `trials` redraws of x (the rows uploaded once)."""
    z, q, T = cuda(x.logits, dev), cuda(x.draft_probs, dev), cuda(x.temperature, dev)
    tot = {}
    for t in range(trials):
        xt = x if t == 0 else W.redraw(x, seed0 + t)
        ot, na = sv.verify_chain(z, cuda(xt.draft_tokens, dev), T, cuda(xt.u_accept, dev), cuda(xt.u_sample, dev), q)
        _add(tot, count_chain(ot.cpu().numpy(), na.cpu().numpy(), oracle_chain(O, xt)))
    return tot


def _check(report, name, tot):
    P = tot["positions"]
    line = "%-46s positions %7d  flagged %5d (%.2e)  differ %d (%.2e)" % (
        name, P, tot["flagged"], tot["flagged"] / P, tot["differ"], tot["differ"] / P)
    if "tested" in tot:
        line += "  alpha %.3f" % (tot["accepted"] / max(1, tot["tested"]))
    report(line)
    _add(_ALL, {"positions": P, "flagged": tot["flagged"], "differ": tot["differ"], "unflagged": tot["unflagged"]})
    assert tot["unflagged"] == 0, (name, tot)


def test_flag_budget_tiny_chain(sv, O, dev, report):
    """B = 1000 trials of one fixed k = 4, V = 1000 fp32 chain."""
    x = W.chain_tiny(seed=1, trials=1000)
    _check(report, "tiny chain B=1000 k=4 V=1000", _chain_trials(sv, O, dev, x, 12, 7100))


@pytest.mark.parametrize("path", [0, 1], ids=["cluster", "persistent"])
@pytest.mark.parametrize("lam", [0.1, 0.3, 0.6])
def test_flag_budget_sampled_chain(sv, O, dev, report, lam, path):
    """B = 32, k = 4, V = 128256, T = 0.7, Zipf-shaped logits; on the cluster
    kernel (the default for this batch) and on the persistent kernel."""
    x = W.chain_sampled(seed=3, B=32, k=4, V=128256, temperature=0.7, lam=lam)
    sv.set_tuning(0, 0, path)
    try:
        tot = _chain_trials(sv, O, dev, x, 60, 7200 + int(lam * 10))
    finally:
        sv.set_tuning(0, 0, 0)
    _check(report, "sampled chain B=32 k=4 V=128256 lambda=%.1f %s" % (lam, ("cluster", "persistent")[path]), tot)


def test_flag_budget_sweep(sv, O, dev, report):
    """B = 256, k = 8, V = 152064, T = 1, lambda = 0.3, whole batch; and its
    first 64 requests as the B = 64 launch."""
    x = W.named("sweep", B=256)
    _check(report, "sweep B=256 k=8 V=152064 lambda=0.3", _chain_trials(sv, O, dev, x, 6, 7300))
    x64 = W.ChainInputs(logits=x.logits[:64], dtype=x.dtype, draft_tokens=x.draft_tokens[:64],
                        temperature=x.temperature[:64], u_sample=x.u_sample[:64],
                        draft_probs=x.draft_probs[:64], u_accept=x.u_accept[:64])
    _check(report, "sweep B=64 k=8 V=152064 lambda=0.3", _chain_trials(sv, O, dev, x64, 16, 7400))


def test_flag_budget_sampled_tree(sv, O, dev, report):
    """B = 16, 60-node level tree (4, 2, 2, 1, 1), V = 128256, T = 0.7."""
    import torch
    x = W.tree_sampled(seed=920, B=16, V=128256)
    z = cuda(x.logits, dev)
    z = z.view(torch.bfloat16) if x.dtype == W.BF16 else z
    q, T = cuda(x.draft_probs, dev), cuda(x.temperature, dev)
    tot = {}
    for t in range(40):
        xt = x if t == 0 else W.redraw(x, 7500 + t)
        p, tk, n = sv.verify_tree_sampled(z, q, cuda(xt.node_tokens, dev), xt.parent, T, cuda(xt.u_accept, dev),
                                          cuda(xt.u_sample, dev))
        got = dict(path=p.cpu().numpy(), tokens=tk.cpu().numpy(), length=n.cpu().numpy())
        ref = O.verify_tree_sampled(xt.logits, xt.dtype, xt.node_tokens, xt.parent, xt.temperature, xt.u_accept,
                                    xt.u_sample, xt.draft_probs)
        _add(tot, count_tree_sampled(np.asarray(x.parent), got, ref))
    _check(report, "sampled tree B=16 N=60 V=128256 lambda=0.3", tot)


def test_flag_budget_all_positions(report):
    """Differences over all positions of the workloads above: below 1e-4."""
    if not _ALL:
        pytest.skip("no flag-budget workload ran")
    P = _ALL["positions"]
    report("%-46s positions %7d  flagged %5d (%.2e)  differ %d (%.2e)" % (
        "all sampled workloads", P, _ALL["flagged"], _ALL["flagged"] / P, _ALL["differ"], _ALL["differ"] / P))
    assert _ALL["unflagged"] == 0
    assert _ALL["differ"] < BUDGET * P, _ALL
