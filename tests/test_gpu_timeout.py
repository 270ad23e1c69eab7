"""The wait time-out path, driven without faulting or hanging anything.

Every wait a kernel makes on other blocks, warps or cluster peers is bounded;
a wait that runs out sets SPEC_STATUS_WAIT_TIMEOUT and the kernel finishes
early instead of hanging.  spec_set_wait_limit_ns(0) makes every wait give up
at its first unsuccessful try, so the path runs on ordinary inputs.  The tests
check that such a call returns with the status bit set, and that the next call
at the default limit, on the same workspace, is bit-exact against the oracle
(so the time-out left the workspace counters clean).
"""
import pytest

from speculative_decoding_verification_chain_gb300 import workloads as W

from helpers import compare_chain, cuda, oracle_chain

pytestmark = pytest.mark.gpu

TIMEOUT = 4   # SPEC_STATUS_WAIT_TIMEOUT


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


@pytest.fixture
def no_wait(sv):
    """Sets the wait limit to 0 for the test body's first phase; the test calls
    restore() itself, and the default is put back whatever happens."""
    prev = sv.set_wait_limit_ns(0)
    state = {"prev": prev}
    yield lambda: sv.set_wait_limit_ns(state["prev"])
    sv.set_wait_limit_ns(prev)


def _chain_args(x, dev):
    sampled = x.draft_probs is not None
    a = [cuda(x.logits, dev), cuda(x.draft_tokens, dev)]
    if sampled:
        a += [cuda(x.temperature, dev), cuda(x.u_accept, dev), cuda(x.u_sample, dev), cuda(x.draft_probs, dev)]
    return a


@pytest.mark.parametrize("kind", ["greedy", "sampled", "tree"])
def test_verify_kernel_times_out_and_leaves_the_workspace_clean(sv, O, dev, no_wait, kind):
    import torch
    if kind == "greedy":
        x = W.chain_greedy(seed=801, B=48, k=5, V=128256, p_match=0.8)
        rows = x.k + 1
    elif kind == "sampled":
        x = W.chain_sampled(seed=802, B=32, k=4, V=60000, temperature=0.8, lam=0.3)
        rows = x.k + 1
    else:
        x = W.tree_greedy(seed=803, B=8, V=128256)
        rows = x.N + 1
    ws = torch.zeros(sv.workspace_bytes(x.B, rows, x.V), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    if kind == "tree":
        call = lambda status: sv.verify_tree(cuda(x.logits, dev), cuda(x.node_tokens, dev), x.parent,
                                             workspace=ws, status=status)
    else:
        args = _chain_args(x, dev)
        call = lambda status: sv.verify_chain(*args, workspace=ws, status=status)
    call(st)
    torch.cuda.synchronize(dev)
    assert int(st.item()) & TIMEOUT, "no wait ran out at limit 0"
    no_wait()   # back to the default limit, same workspace
    st2 = torch.zeros(1, dtype=torch.int32, device=dev)
    out = call(st2)
    torch.cuda.synchronize(dev)
    assert int(st2.item()) == 0
    if kind == "tree":
        path, toks, ln = out
        ref = O.verify_tree(x.logits, x.dtype, x.node_tokens, x.parent)
        assert (ln.cpu().numpy() == ref["length"]).all()
        assert (path.cpu().numpy() == ref["path"]).all() and (toks.cpu().numpy() == ref["tokens"]).all()
    else:
        ot, na = out
        ref = oracle_chain(O, x)
        got_t, got_a = ot.cpu().numpy(), na.cpu().numpy()
        if kind == "greedy":
            assert (got_a == ref["num_accepted"]).all() and (got_t == ref["out_tokens"]).all()
        else:
            compare_chain(got_t, got_a, ref)


@pytest.mark.parametrize("V", [60000, 7])
def test_sampled_tree_kernel_times_out(sv, O, dev, no_wait, V):
    """Row copies (V = 60000: the first copy is still in flight) and cluster
    exchanges (V = 7: rows too short for bulk copies, so the first wait is an
    exchange) of the sampled-tree kernel: at limit 0 the walks end early with
    the status bit; the next call is right."""
    import torch
    x = W.tree_sampled(seed=804, B=8, V=V, dtype=W.FP32 if V < 16 else W.BF16)
    args = (cuda(x.logits, dev), cuda(x.draft_probs, dev), cuda(x.node_tokens, dev), x.parent,
            cuda(x.temperature, dev), cuda(x.u_accept, dev), cuda(x.u_sample, dev))
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    sv.verify_tree_sampled(*args, status=st)
    torch.cuda.synchronize(dev)
    assert int(st.item()) & TIMEOUT, "no wait ran out at limit 0"
    no_wait()
    st2 = torch.zeros(1, dtype=torch.int32, device=dev)
    p, t, n = sv.verify_tree_sampled(*args, status=st2)
    torch.cuda.synchronize(dev)
    assert int(st2.item()) == 0
    got = dict(path=p.cpu().numpy(), tokens=t.cpu().numpy(), length=n.cpu().numpy())
    ref = O.verify_tree_sampled(x.logits, x.dtype, x.node_tokens, x.parent, x.temperature, x.u_accept,
                                x.u_sample, x.draft_probs)
    from helpers import count_tree_sampled
    assert count_tree_sampled(x.parent, got, ref)["unflagged"] == 0


def test_default_limit_is_restored(sv):
    prev = sv.set_wait_limit_ns(123)
    assert sv.set_wait_limit_ns(prev) == 123
    assert prev == 500_000_000
