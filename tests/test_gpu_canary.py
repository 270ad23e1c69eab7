"""Guard regions around every output buffer (a stand-in for a memory checker).

Each output (and the workspace) lives inside a larger device buffer whose
first and last 4 KiB hold a fixed byte pattern.  The edge shapes run through
the C ABI -- V = 1, V not a multiple of 8, k = 1, k = 255, B = 1, ragged
batches with requests that have no drafts, root-only trees, 14-byte hidden
rows, KV rows next to the moved ones -- and the results are compared with the
oracle; afterwards every guard must still hold its pattern, so no kernel wrote
before or past a buffer it was given.
"""
import numpy as np
import pytest

from speculative_decoding_verification_chain_gb300 import workloads as W

from helpers import compare_chain, count_tree_sampled, cuda, oracle_chain

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


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


class Guarded:
    """Device buffers with GUARD pattern bytes before and after."""

    def __init__(self, dev):
        self.dev = dev
        self.bufs = []

    def make(self, name, shape, dtype, init=None):
        import torch
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        buf = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device=self.dev)
        view = buf[GUARD:GUARD + n].view(dtype).view(tuple(shape))
        if isinstance(init, (int, float)):
            view.fill_(init)
        elif init is not None:
            view.copy_(init)
        self.bufs.append((name, buf, n))
        return view

    def check(self):
        import torch
        torch.cuda.synchronize(self.dev)
        for name, buf, n in self.bufs:
            assert (buf[:GUARD] == PATTERN).all(), "%s: bytes written before the buffer" % name
            assert (buf[GUARD + n:] == PATTERN).all(), "%s: bytes written past the buffer" % name


CHAINS = [("greedy", 1, 1, 1, W.BF16), ("greedy", 3, 1, 13, W.BF16), ("greedy", 2, 255, 300, W.FP32),
          ("greedy", 1, 4, 128256, W.BF16), ("greedy", 5, 3, 1001, W.FP32),
          ("sampled", 1, 1, 1, W.FP32), ("sampled", 4, 3, 4099, W.BF16), ("sampled", 2, 255, 129, W.FP32),
          ("sampled", 1, 4, 128256, W.BF16), ("sampled", 3, 2, 13, W.BF16)]


@pytest.mark.parametrize("kind,B,k,V,dtype", CHAINS,
                         ids=["%s-B%d-k%d-V%d-%s" % (c[0], c[1], c[2], c[3], "bf16" if c[4] == W.BF16 else "fp32")
                              for c in CHAINS])
def test_chain_outputs_stay_inside_their_buffers(sv, O, dev, kind, B, k, V, dtype):
    import torch
    if kind == "greedy":
        x = W.chain_greedy(seed=4000 + B * 31 + k + V, B=B, k=k, V=V, p_match=0.8, dtype=dtype)
    else:
        x = W.chain_sampled(seed=4100 + B * 31 + k + V, B=B, k=k, V=V, temperature=0.9, lam=0.3, dtype=dtype)
    g = Guarded(dev)
    code = sv.SPEC_BF16 if dtype == W.BF16 else sv.SPEC_FP32
    ws = g.make("workspace", (sv.workspace_bytes(B, k + 1, V, code),), torch.uint8, 0)
    out = g.make("out_tokens", (B, k + 1), torch.int32)
    na = g.make("num_accepted", (B,), torch.int32)
    st = g.make("status", (1,), torch.int32, 0)
    slots = g.make("slot_mapping", (B, k + 1), torch.int64, torch.from_numpy(x.slot_mapping))
    sampled = x.draft_probs is not None
    args = [cuda(x.logits, dev), cuda(x.draft_tokens, dev)]
    if sampled:
        args += [cuda(x.temperature, dev), cuda(x.u_accept, dev), cuda(x.u_sample, dev), cuda(x.draft_probs, dev)]
    sv.verify_chain(*args, out_tokens=out, out_num_accepted=na, status=st, workspace=ws, slot_mapping=slots)
    g.check()
    ref = oracle_chain(O, x)
    got_t, got_a = out.cpu().numpy(), na.cpu().numpy()
    if sampled:
        compare_chain(got_t, got_a, ref)
    else:
        assert (got_a == ref["num_accepted"]).all() and (got_t == ref["out_tokens"]).all()
    assert (slots.cpu().numpy() == O.fixup_slots(x.slot_mapping, num_accepted=got_a)).all()
    assert int(st.item()) == 0


@pytest.mark.parametrize("mode,max_k,V", [("mixed", 4, 1), ("mixed", 6, 13), ("greedy", 0, 300),
                                          ("sampled", 3, 4099)])
def test_ragged_outputs_stay_inside_their_buffers(sv, O, dev, mode, max_k, V):
    """Ragged batches with requests that have no drafts (k_b = 0)."""
    import torch
    x = W.chain_ragged(seed=4200 + max_k + V, B=7, max_k=max_k, V=V, mode=mode, min_k=0)
    B = x.B
    g = Guarded(dev)
    ws = g.make("workspace", (sv.workspace_bytes(B, max_k + 1, V, sv.SPEC_BF16),), torch.uint8, 0)
    out = g.make("out_tokens", (B, max_k + 1), torch.int32)
    na = g.make("num_accepted", (B,), torch.int32)
    slots = g.make("slot_mapping", x.slot_mapping.shape, torch.int64, torch.from_numpy(x.slot_mapping))
    sampled = x.draft_probs is not None
    sv.verify_chain_ragged(cuda(x.logits, dev), cuda(x.draft_tokens, dev), cuda(x.cu, dev), max_k,
                           cuda(x.temperature, dev) if sampled else None, cuda(x.u_accept, dev) if sampled else None,
                           cuda(x.u_sample, dev) if sampled else None, cuda(x.draft_probs, dev) if sampled else None,
                           out_tokens=out, out_num_accepted=na, workspace=ws, slot_mapping=slots)
    g.check()
    got_t, got_a = out.cpu().numpy(), na.cpu().numpy()
    for b, part in enumerate(x.parts):
        ref = O.verify_chain(part.logits, part.dtype, part.draft_tokens, part.temperature, part.u_sample,
                             part.draft_probs, part.u_accept)
        compare_chain(got_t[b:b + 1, :part.k + 1], got_a[b:b + 1], ref)
        assert (got_t[b, part.k + 1:] == -1).all()
    # the separate ragged fix-up on guarded slots as well
    slots2 = g.make("slot_mapping (separate fix-up)", x.slot_mapping.shape, torch.int64,
                    torch.from_numpy(x.slot_mapping))
    sv.fixup_slots_ragged(slots2, cuda(x.cu, dev), na)
    g.check()
    assert (slots2.cpu().numpy() == slots.cpu().numpy()).all()


@pytest.mark.parametrize("shape,V", [(None, 1), ((2,), 7), ((3, 2, 1), 13), ((4, 2, 2, 1, 1), 1001)])
def test_tree_outputs_stay_inside_their_buffers(sv, O, dev, shape, V):
    """Greedy trees (root-only when shape is None) and the tree-mode fix-up."""
    import torch
    if shape is None:
        t = W.tree_greedy(seed=4300, B=3, V=V, parent=np.array([-1], np.int32))
    else:
        t = W.tree_greedy(seed=4300 + V, B=5, V=V, children_per_level=shape, p_match=0.75)
    B, N, D = t.B, t.N, int(max(1, len(shape))) if shape else 0
    g = Guarded(dev)
    ws = g.make("workspace", (sv.workspace_bytes(B, N + 1, V, sv.SPEC_BF16),), torch.uint8, 0)
    path = g.make("out_path", (B, D + 1), torch.int32)
    toks = g.make("out_tokens", (B, D + 1), torch.int32)
    ln = g.make("out_len", (B,), torch.int32)
    sv.verify_tree(cuda(t.logits, dev), cuda(t.node_tokens, dev), t.parent, D,
                   out_path=path, out_tokens=toks, out_len=ln, workspace=ws)
    g.check()
    ref = O.verify_tree(t.logits, t.dtype, t.node_tokens, t.parent)
    assert (ln.cpu().numpy() == ref["length"]).all()
    assert (path.cpu().numpy() == ref["path"]).all() and (toks.cpu().numpy() == ref["tokens"]).all()
    slots = g.make("slot_mapping", (B, N + 1), torch.int64, torch.from_numpy(t.slot_mapping))
    sv.fixup_slots(slots, path=path)
    g.check()
    assert (slots.cpu().numpy() == O.fixup_slots(t.slot_mapping, path=ref["path"])).all()


@pytest.mark.parametrize("V", [1, 7, 4099])
def test_sampled_tree_outputs_stay_inside_their_buffers(sv, O, dev, V):
    import torch
    x = W.tree_sampled(seed=4400 + V, B=6, V=V, children_per_level=(3, 2), dtype=W.FP32)
    B, D = x.B, 2
    g = Guarded(dev)
    path = g.make("out_path", (B, D + 1), torch.int32)
    toks = g.make("out_tokens", (B, D + 1), torch.int32)
    ln = g.make("out_len", (B,), torch.int32)
    st = g.make("status", (1,), torch.int32, 0)
    sv.verify_tree_sampled(cuda(x.logits, dev), cuda(x.draft_probs, dev), cuda(x.node_tokens, dev), x.parent,
                           cuda(x.temperature, dev), cuda(x.u_accept, dev), cuda(x.u_sample, dev), D,
                           out_path=path, out_tokens=toks, out_len=ln, status=st)
    g.check()
    got = dict(path=path.cpu().numpy(), tokens=toks.cpu().numpy(), length=ln.cpu().numpy())
    ref = O.verify_tree_sampled(x.logits, x.dtype, x.node_tokens, x.parent, x.temperature, x.u_accept,
                                x.u_sample, x.draft_probs)
    assert count_tree_sampled(np.asarray(x.parent), got, ref)["unflagged"] == 0


@pytest.mark.parametrize("row_bytes,ragged", [(14, False), (4096, True), (16, False)])
def test_next_step_outputs_stay_inside_their_buffers(sv, O, dev, row_bytes, ragged):
    """spec_prepare_next_step through the C ABI with every output guarded."""
    import torch
    rng = np.random.default_rng(4500 + row_bytes)
    B, k, bs, P_next, max_blocks = 5, 4, 8, 6, 4
    if ragged:
        ks = rng.integers(0, k + 1, size=B)
        cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
        rows = int(cu[-1]) + B
        a = np.array([rng.integers(0, kb + 1) for kb in ks], np.int32)
    else:
        cu = None
        rows = B * (k + 1)
        a = rng.integers(0, k + 1, size=B).astype(np.int32)
    ot = rng.integers(0, 50000, size=(B, k + 1)).astype(np.int32)
    pos = rng.integers(0, 20, size=B).astype(np.int32)
    bt = rng.integers(-1, 30, size=(B, max_blocks)).astype(np.int32)
    hid = rng.integers(0, 256, size=(rows, row_bytes)).astype(np.uint8)
    g = Guarded(dev)
    nt = g.make("next_token", (B,), torch.int32)
    npos = g.make("next_position", (B,), torch.int32)
    ns = g.make("next_slots", (B, P_next), torch.int64)
    lr = g.make("last_row", (B,), torch.int32)
    ho = g.make("hidden_out", (B, row_bytes), torch.uint8)
    st = g.make("status", (1,), torch.int32, 0)
    lib = sv.load_library()
    d_ot, d_a, d_pos, d_bt, d_hid = (cuda(ot, dev), cuda(a, dev), cuda(pos, dev), cuda(bt, dev), cuda(hid, dev))
    d_cu = cuda(cu, dev) if ragged else None
    ptr = lambda t: None if t is None else t.data_ptr()
    rc = lib.spec_prepare_next_step(ptr(d_ot), k + 1, ptr(d_a), ptr(d_pos), ptr(d_bt), max_blocks, bs, B, P_next,
                                    0 if ragged else k + 1, ptr(d_cu), ptr(d_hid), row_bytes, -1, ptr(nt),
                                    ptr(npos), ptr(ns), ptr(lr), ptr(ho), ptr(st),
                                    torch.cuda.current_stream(dev).cuda_stream)
    assert rc == 0, lib.spec_last_error()
    g.check()
    ref = O.prepare_next_step(ot, a, pos, bt, bs, P_next, rows_per_req=0 if ragged else k + 1, cu=cu, hidden=hid)
    assert (nt.cpu().numpy() == ref["next_token"]).all() and (npos.cpu().numpy() == ref["next_position"]).all()
    assert (ns.cpu().numpy() == ref["next_slots"]).all() and (lr.cpu().numpy() == ref["last_row"]).all()
    assert (ho.cpu().numpy() == ref["hidden_out"]).all()
    # the oracle reports the slot-range case as its own bit 1
    assert bool(int(st.item()) & sv.STATUS_SLOT_RANGE) == bool(int(ref["status"][0]) & 1)


def test_kv_compaction_touches_only_destination_rows(sv, O, dev):
    """KV rows next to the moved ones, and the bytes around the cache, keep
    their values; the destinations get their sources' rows."""
    import torch
    t = W.tree_greedy(seed=4600, B=4, V=3001, children_per_level=(3, 2, 2), p_match=0.9)
    path, toks, ln = sv.verify_tree(cuda(t.logits, dev), cuda(t.node_tokens, dev), t.parent)
    rng = np.random.default_rng(4601)
    num_slots, row_bytes = t.B * (t.N + 1) * 3, 48
    kv = rng.integers(0, 256, size=(num_slots, row_bytes)).astype(np.uint8)
    smap = rng.permutation(num_slots)[: t.B * (t.N + 1)].reshape(t.B, t.N + 1).astype(np.int64)
    g = Guarded(dev)
    kvd = g.make("kv", kv.shape, torch.uint8, torch.from_numpy(kv))
    st = g.make("status", (1,), torch.int32, 0)
    sv.compact_tree_kv(kvd, cuda(smap, dev), path, ln, status=st)
    g.check()
    exp = O.compact_tree_kv(kv, smap, path.cpu().numpy(), ln.cpu().numpy())["kv"]
    assert (kvd.cpu().numpy() == exp).all()


@pytest.mark.parametrize("k", [0, 1, 7])
def test_ngram_outputs_stay_inside_their_buffers(sv, O, dev, k):
    import torch
    tt, tl = W.ngram_texts(seed=4700 + k, B=6, Lmax=200)
    tl[0], tl[1] = 0, 1   # an empty text and a one-token text
    B = tt.shape[0]
    g = Guarded(dev)
    d = g.make("out_draft", (B, k), torch.int32)
    c = g.make("out_count", (B,), torch.int32)
    ml = g.make("out_match_len", (B,), torch.int32)
    me = g.make("out_match_end", (B,), torch.int32)
    sv.ngram_propose(cuda(tt, dev), cuda(tl, dev), 2, 6, k, out_draft=d, out_count=c, out_match_len=ml,
                     out_match_end=me)
    g.check()
    r = O.ngram_propose(tt, tl, 2, 6, k)
    assert (d.cpu().numpy() == r["draft"]).all() and (c.cpu().numpy() == r["count"]).all()
    assert (ml.cpu().numpy() == r["match_len"]).all() and (me.cpu().numpy() == r["match_end"]).all()
