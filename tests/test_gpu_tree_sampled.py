"""Sampled token trees on the GPU against the oracle.

Paths, lengths and tokens are compared request by request; where they differ,
the first difference must sit at a decision the oracle flags (an accept test
within its window among the children of the node where the walks part, or
the final draw near a bucket edge).  The output and sibling laws are checked
on the GPU path itself by chi-square.  Every call goes through the C ABI via
the binding.
"""
import numpy as np
import pytest

from speculative_decoding_verification_chain_gb300 import workloads as W

from helpers import cuda, tree_divergence

pytestmark = pytest.mark.gpu


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


def _logits_dev(x, dev):
    import torch
    t = cuda(x.logits, dev)
    return t.view(torch.bfloat16) if x.dtype == W.BF16 else t


def run_gpu(sv, dev, x, status=None):
    import torch
    p, t, n = sv.verify_tree_sampled(_logits_dev(x, dev), cuda(x.draft_probs, dev), cuda(x.node_tokens, dev),
                                     x.parent, cuda(x.temperature, dev), cuda(x.u_accept, dev),
                                     cuda(x.u_sample, dev), status=status)
    torch.cuda.synchronize(dev)
    return dict(path=p.cpu().numpy(), tokens=t.cpu().numpy(), length=n.cpu().numpy())


def run_oracle(O, x):
    return O.verify_tree_sampled(x.logits, x.dtype, x.node_tokens, x.parent, x.temperature, x.u_accept,
                                 x.u_sample, x.draft_probs)


def compare(x, got, ref):
    """(exact requests, flagged differences, unexplained differences).  A
    difference is excused only by the oracle's flag on the decision that made
    it: the test of the first child on which the two walks disagree, or the
    final draw when the walks are the same."""
    exact = flagged = bad = 0
    for b in range(x.B):
        d = tree_divergence(x.parent, got, ref, b)
        if d is None:
            exact += 1
            continue
        kind, n = d
        ok = (kind == "accept" and bool(ref["flag_accept"][b, n - 1])) or (
            kind == "sample" and bool(ref["flag_sample"][b]))
        if ok:
            flagged += 1
        else:
            bad += 1
    return exact, flagged, bad


@pytest.mark.parametrize("dtype", [W.FP32, W.BF16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("V", [1000, 4099, 32000])
def test_parity_level_tree(sv, O, dev, dtype, V):
    x = W.tree_sampled(seed=900 + V, B=64, V=V, dtype=dtype)
    got, ref = run_gpu(sv, dev, x), run_oracle(O, x)
    exact, flagged, bad = compare(x, got, ref)
    assert bad == 0, (exact, flagged, bad)
    assert exact >= 60


@pytest.mark.parametrize("lam,T", [(0.1, 1.0), (0.6, 0.7), (0.9, 0.5)])
def test_parity_acceptance_regimes(sv, O, dev, lam, T):
    x = W.tree_sampled(seed=910, B=48, V=5003, children_per_level=(3, 3, 2), temperature=T, lam=lam)
    got, ref = run_gpu(sv, dev, x), run_oracle(O, x)
    exact, flagged, bad = compare(x, got, ref)
    assert bad == 0 and exact >= 44, (exact, flagged, bad)


def test_parity_full_size_bf16(sv, O, dev):
    x = W.tree_sampled(seed=920, B=16, V=128256)
    got, ref = run_gpu(sv, dev, x), run_oracle(O, x)
    exact, flagged, bad = compare(x, got, ref)
    assert bad == 0 and exact >= 15, (exact, flagged, bad)


@pytest.mark.parametrize("V", [1, 2, 7, 9, 152064, 262144])
def test_parity_vocabulary_edges(sv, O, dev, V):
    """Tiny vocabularies (one CTA, partial chunks), the sweep vocabulary, and a
    vocabulary that needs a 16-CTA cluster."""
    B = 24 if V < 100000 else 4
    x = W.tree_sampled(seed=930 + V, B=B, V=V, children_per_level=(2, 2), dtype=W.FP32)
    got, ref = run_gpu(sv, dev, x), run_oracle(O, x)
    exact, flagged, bad = compare(x, got, ref)
    assert bad == 0 and exact >= B - 2, (exact, flagged, bad)


def test_root_only_tree_draws_from_root(sv, O, dev):
    x = W.tree_sampled(seed=940, B=32, V=3000, parent=np.array([-1], np.int32))
    got, ref = run_gpu(sv, dev, x), run_oracle(O, x)
    assert (got["length"] == 1).all() and (got["path"][:, 0] == 0).all()
    exact, flagged, bad = compare(x, got, ref)
    assert bad == 0 and exact >= 30


def test_irregular_tree(sv, O, dev):
    parent = np.array([-1, 0, 0, 1, 1, 1, 2, 3, 3, 6, 7, 7, 7, 9], np.int32)
    x = W.tree_sampled(seed=941, B=64, V=2048, parent=parent, lam=0.6)
    got, ref = run_gpu(sv, dev, x), run_oracle(O, x)
    exact, flagged, bad = compare(x, got, ref)
    assert bad == 0 and exact >= 60, (exact, flagged, bad)


def test_status_bits(sv, O, dev):
    import torch
    x = W.tree_sampled(seed=942, B=8, V=500, children_per_level=(2,))
    x.node_tokens[:, 0] = 500                 # out of range: rejected
    x.node_tokens[0, 1] = -3
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    got = run_gpu(sv, dev, x, status=st)
    assert int(st.item()) & sv.STATUS_TOKEN_RANGE
    ref = run_oracle(O, x)
    assert compare(x, got, ref)[2] == 0
    x.temperature[3] = 0.0
    st.zero_()
    run_gpu(sv, dev, x, status=st)
    assert int(st.item()) & sv.STATUS_BAD_TEMPERATURE


def test_law_on_gpu(sv, O, dev):
    """The GPU path's own output law and sibling law (chi-square, as for the oracle)."""
    import test_oracle_tree_sampled as ts
    c = ts.law_case(seed=52, trials=200_000)
    x = W.TreeInputs(logits=c["z"], dtype=W.FP32, node_tokens=c["toks"], parent=c["parent"], tree_choices=[],
                     draft_probs=c["q"], temperature=c["T"], u_accept=c["ua"], u_sample=c["us"])
    got = run_gpu(sv, dev, x)
    pv = ts.law_pvalues(c, got)
    assert pv["first"] > 0.01 and pv["sibling"] > 0.01, pv
    assert pv["second"] > 0.01 / pv["n_second"], pv


def test_host_checks(sv, dev):
    import torch
    x = W.tree_sampled(seed=943, B=2, V=64, children_per_level=(2,))
    with pytest.raises(Exception):
        sv.verify_tree_sampled(_logits_dev(x, dev), cuda(x.draft_probs, dev), cuda(x.node_tokens, dev),
                               [-1, 0, 2], cuda(x.temperature, dev), cuda(x.u_accept, dev), cuda(x.u_sample, dev))
    with pytest.raises(Exception):
        sv.verify_tree_sampled(_logits_dev(x, dev), cuda(x.draft_probs, dev), cuda(x.node_tokens, dev),
                               x.parent, cuda(x.temperature, dev), cuda(x.u_accept, dev), cuda(x.u_sample, dev),
                               max_depth=0)
    assert torch.cuda.is_available()


def test_one_child_per_level_equals_the_sampled_chain_kernel(sv, O, dev):
    """Two separate GPU paths on the same inputs: the sampled tree with one child
    per level and the chain verify agree (tokens, counts), except where the
    oracle flags the deciding test or draw."""
    import torch
    x = W.chain_sampled(seed=950, B=40, k=4, V=20011, temperature=0.8, lam=0.3, dtype=W.FP32)
    k = x.k
    parent = W.parents_in_order((1,) * k)
    q = np.zeros((x.B, k + 1, x.V), np.float32)
    q[:, :k] = x.draft_probs
    p, t, n = sv.verify_tree_sampled(cuda(x.logits, dev), cuda(q, dev), cuda(x.draft_tokens, dev), parent,
                                     cuda(x.temperature, dev), cuda(x.u_accept, dev), cuda(x.u_sample, dev))
    ot, na = sv.verify_chain(cuda(x.logits, dev), cuda(x.draft_tokens, dev), cuda(x.temperature, dev),
                             cuda(x.u_accept, dev), cuda(x.u_sample, dev), cuda(x.draft_probs, dev))
    torch.cuda.synchronize(dev)
    ref = O.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample, x.draft_probs, x.u_accept)
    tl, tt, ca, ct = n.cpu().numpy(), t.cpu().numpy(), na.cpu().numpy(), ot.cpu().numpy()
    same = 0
    for b in range(x.B):
        a, c = int(tl[b]) - 1, int(ca[b])
        if a == c and (tt[b] == ct[b]).all():
            same += 1
            continue
        # both walks accepted every test below j = min(a, c); at j one accepted and
        # the other rejected (or, with equal counts, their draws differ).  Each walk
        # agrees with the oracle up to its first flagged decision, so the oracle
        # flags an accept test at or below j, or, with equal counts, the draw
        j = min(a, c)
        tests_flagged = bool(ref["flag_accept"][b, :min(j + 1, k)].any())
        assert tests_flagged or (a == c and ref["flag_sample"][b]), b
    assert same >= x.B - 2
