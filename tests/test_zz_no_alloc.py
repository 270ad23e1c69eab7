"""spec_verify_chain_noalloc: the entry point for callers that cannot allocate
device memory (they have no allocator of their own to create the workspace
that spec_verify_chain needs, e.g. a plugin whose runtime owns and budgets all
device memory).  It must give the same results as spec_verify_chain, call
after call, using the library's fixed scratch array instead of a workspace.

This file is collected last on purpose; it runs alone in a fresh process too.
"""

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
def sv():
    import speculative_decoding_verification_chain_gb300 as m
    m.load_library()
    return m


def _noalloc_call(sv, lib, x, dev):
    """One call through the C ABI; returns host copies of the outputs."""
    import torch
    sampled = x.draft_probs is not None
    z = cuda(x.logits, dev)
    tok = cuda(x.draft_tokens, dev)
    T = cuda(x.temperature, dev) if sampled else None
    ua = cuda(x.u_accept, dev) if sampled else None
    us = cuda(x.u_sample, dev) if sampled else None
    q = cuda(x.draft_probs, dev) if sampled else None
    out = torch.full((x.B, x.k + 1), -7, dtype=torch.int32, device=dev)
    na = torch.full((x.B,), -7, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ptr = lambda t: None if t is None else t.data_ptr()
    code = sv.SPEC_BF16 if x.dtype == W.BF16 else sv.SPEC_FP32
    rc = lib.spec_verify_chain_noalloc(ptr(z), code, ptr(q), ptr(tok), ptr(T), ptr(ua), ptr(us), x.B, x.k, x.V,
                                       ptr(out), ptr(na), ptr(st), torch.cuda.current_stream(dev).cuda_stream)
    assert rc == 0, lib.spec_last_error()
    torch.cuda.synchronize(dev)
    return out.cpu().numpy(), na.cpu().numpy(), int(st.item())


CASES = [
    ("greedy", lambda: W.chain_greedy(seed=501, B=24, k=5, V=50000, p_match=0.8)),
    ("sampled", lambda: W.chain_sampled(seed=502, B=16, k=4, V=30011, temperature=0.8, lam=0.3)),
    ("greedy_small_fp32", lambda: W.chain_greedy(seed=503, B=5, k=3, V=777, dtype=W.FP32)),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_workspace_entry_point_twice(sv, dev, name, make):
    x = make()
    sampled = x.draft_probs is not None
    ref_t, ref_a = sv.verify_chain(cuda(x.logits, dev), cuda(x.draft_tokens, dev),
                                   cuda(x.temperature, dev) if sampled else None,
                                   cuda(x.u_accept, dev) if sampled else None,
                                   cuda(x.u_sample, dev) if sampled else None,
                                   cuda(x.draft_probs, dev) if sampled else None)
    ref_t, ref_a = ref_t.cpu().numpy(), ref_a.cpu().numpy()
    lib = sv.load_library()
    for _ in range(2):   # two calls in a row share (and must clean up) the scratch
        got_t, got_a, st = _noalloc_call(sv, lib, x, dev)
        assert st == 0
        # same kernel, same inputs: identical results (tighter than the
        # flagged-position tolerance the oracle comparisons use)
        assert (got_a == ref_a).all()
        assert (got_t == ref_t).all()


def test_noalloc_alternating_sizes_and_python_wrapper(sv, dev):
    xs = [W.chain_greedy(seed=511, B=9, k=2, V=20000), W.chain_greedy(seed=512, B=40, k=6, V=9000)]
    refs = []
    for x in xs:
        t, a = sv.verify_chain(cuda(x.logits, dev), cuda(x.draft_tokens, dev))
        refs.append((t.cpu().numpy(), a.cpu().numpy()))
    for _ in range(2):
        for x, (rt, ra) in zip(xs, refs):
            t, a = sv.verify_chain_noalloc(cuda(x.logits, dev), cuda(x.draft_tokens, dev))
            assert (a.cpu().numpy() == ra).all() and (t.cpu().numpy() == rt).all()


def test_noalloc_rejects_sizes_beyond_the_scratch(sv, dev):
    lib = sv.load_library()
    cap = lib.spec_noalloc_scratch_bytes()
    assert cap == 16 << 20
    B, k, V = 1024, 8, 152064
    assert lib.spec_workspace_bytes(B, k + 1, V, 0) > cap
    rc = lib.spec_verify_chain_noalloc(0x10000, 0, None, 0x20000, None, None, None, B, k, V, 0x30000, 0x40000,
                                       None, None)
    assert rc == 1
    assert b"scratch" in lib.spec_last_error()


def test_noalloc_calls_take_no_device_memory(sv, dev):
    """The point of the entry point: a call allocates nothing.  With inputs and
    outputs made beforehand, the device's free memory is the same before and
    after several calls (the first call on the device, which sets up the
    kernels and looks up the scratch address, is made before the reading)."""
    import torch
    x = W.chain_sampled(seed=521, B=8, k=4, V=30011, temperature=0.8, lam=0.3)
    args = [cuda(a, dev) for a in (x.logits, x.draft_tokens, x.temperature, x.u_accept, x.u_sample, x.draft_probs)]
    out = torch.empty((x.B, x.k + 1), dtype=torch.int32, device=dev)
    na = torch.empty((x.B,), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    sv.verify_chain_noalloc(*args, out_tokens=out, out_num_accepted=na, status=st)
    torch.cuda.synchronize(dev)
    free0, _ = torch.cuda.mem_get_info(dev)
    for _ in range(4):
        sv.verify_chain_noalloc(*args, out_tokens=out, out_num_accepted=na, status=st)
    torch.cuda.synchronize(dev)
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0, (free0, free1)
    assert int(st.item()) == 0
