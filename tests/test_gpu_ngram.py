"""n-gram lookup drafting on the GPU against the oracle (bit-exact: drafts,
counts, match lengths and match ends are integers).  Every call goes through
the C ABI via the package binding."""
import numpy as np
import pytest

from speculative_decoding_verification_chain_gb300 import workloads as W

from helpers import cuda

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


def _run(sv, dev, t, ln, nmin, nmax, k):
    d, c, ml, me = sv.ngram_propose(cuda(t, dev), cuda(ln, dev), nmin, nmax, k)
    return dict(draft=d.cpu().numpy(), count=c.cpu().numpy(), match_len=ml.cpu().numpy(),
                match_end=me.cpu().numpy())


def _same(got, ref):
    for key in ("draft", "count", "match_len", "match_end"):
        assert (got[key] == ref[key]).all(), key


@pytest.mark.parametrize("V", [2, 3, 50, 128256])
@pytest.mark.parametrize("cfg", [(1, 4, 5), (2, 6, 3), (3, 3, 8), (1, 64, 16)], ids=str)
def test_random_texts_bit_exact(sv, O, dev, V, cfg):
    g = np.random.default_rng(800 + V)
    B, Lmax = 96, 700
    t = g.integers(0, V, size=(B, Lmax)).astype(np.int32)
    ln = g.integers(0, Lmax + 1, size=B).astype(np.int32)
    nmin, nmax, k = cfg
    _same(_run(sv, dev, t, ln, nmin, nmax, k), O.ngram_propose(t, ln, nmin, nmax, k))


def test_copy_heavy_texts_full_size(sv, O, dev):
    t, ln = W.ngram_texts(seed=801, B=64, Lmax=8192, V=128256)
    got = _run(sv, dev, t, ln, 2, 8, 8)
    _same(got, O.ngram_propose(t, ln, 2, 8, 8))
    assert (got["count"] > 0).sum() >= 16


def test_edge_cases(sv, O, dev):
    # empty, one token, all equal (overlapping copies), no repeat at all,
    # repeats that only a short n finds, k = 0, n_min above what fits
    Lmax = 40
    t = np.zeros((6, Lmax), np.int32)
    ln = np.array([0, 1, 40, 40, 17, 40], np.int32)
    t[2] = 7
    t[3] = np.arange(Lmax)
    t[4, :17] = [1, 2, 3, 1, 2, 3, 1, 2, 3, 4, 1, 2, 3, 1, 2, 3, 4]
    t[5] = np.tile([9, 8, 7, 6, 5], 8)
    for nmin, nmax, k in ((1, 8, 6), (2, 3, 0), (4, 64, 12)):
        _same(_run(sv, dev, t, ln, nmin, nmax, k), O.ngram_propose(t, ln, nmin, nmax, k))
    # lengths outside [0, Lmax] are clamped by the kernel
    bad = np.array([-3, 1, 99, 40, 17, 41], np.int32)
    _same(_run(sv, dev, t, bad, 1, 8, 6), O.ngram_propose(t, np.clip(bad, 0, Lmax).astype(np.int32), 1, 8, 6))


def test_golden_examples_on_gpu(sv, dev):
    import test_oracle_ngram as ng
    for toks, nmin, nmax, k, draft, (ml, me) in ng._golden():
        t = np.zeros((1, max(1, len(toks))), np.int32)
        t[0, :len(toks)] = toks
        got = _run(sv, dev, t, np.array([len(toks)], np.int32), nmin, nmax, k)
        assert got["draft"][0].tolist() == draft, toks
        assert (got["match_len"][0], got["match_end"][0]) == (ml, me), toks
