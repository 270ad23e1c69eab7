"""Next-step preparation and tree KV compaction on the GPU against the oracle
(bit-exact: integers and byte copies).  Every call goes through the C ABI via
the binding."""
import numpy as np
import pytest

from speculative_decoding_verification_chain_gb300 import workloads as W

from helpers import cuda

import test_oracle_next_step as ns

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


def gpu_prepare(sv, dev, ot, a, pos, bt, bs, P_next, status=None, **kw):
    t, p, s, r, h = sv.prepare_next_step(cuda(ot, dev), cuda(a, dev), cuda(pos, dev), cuda(bt, dev), bs, P_next,
                                         status=status, **kw)
    return dict(next_token=t.cpu().numpy(), next_position=p.cpu().numpy(), next_slots=s.cpu().numpy(),
                last_row=r.cpu().numpy(), hidden_out=None if h is None else h.cpu().numpy())


def same_prepare(got, ref):
    for key in ("next_token", "next_position", "next_slots", "last_row"):
        assert (got[key] == ref[key]).all(), key
    if ref["hidden_out"] is not None:
        assert (got["hidden_out"].view(np.uint8) == ref["hidden_out"].view(np.uint8)).all()


def test_golden_examples(sv, dev):
    import torch
    g = ns.golden_case()
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    got = gpu_prepare(sv, dev, g["out_tokens"], g["a"], g["pos"], g["bt"], 4, 3, rows_per_req=4, status=st)
    assert (got["next_token"] == g["next_token"]).all()
    assert (got["next_position"] == g["next_position"]).all()
    assert (got["next_slots"] == g["slots"]).all()
    assert (got["last_row"] == g["last_row"]).all()
    assert int(st.item()) & sv.STATUS_SLOT_RANGE


@pytest.mark.parametrize("P_next", [0, 1, 6, 9, 300])
def test_prepare_parity(sv, O, dev, P_next):
    import torch
    ot, a, pos, bt, hid = ns.random_case(500 + P_next, B=257, k=5, max_blocks=40, block_size=16, hidden=4096)
    ref = O.prepare_next_step(ot, a, pos, bt, 16, P_next, rows_per_req=6, hidden=hid)
    got = gpu_prepare(sv, dev, ot, a, pos, bt, 16, P_next, rows_per_req=6, hidden=cuda(hid, dev))
    same_prepare(got, ref)


def test_prepare_ragged_and_odd_rows(sv, O, dev):
    g = np.random.default_rng(510)
    B = 70
    ks = g.integers(0, 8, size=B)
    cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    ot = g.integers(0, 1000, size=(B, 9)).astype(np.int32)
    a = np.array([g.integers(0, kk + 1) for kk in ks], np.int32)
    pos = g.integers(0, 500, size=B).astype(np.int32)
    bt = g.integers(-1, 300, size=(B, 64)).astype(np.int32)
    hid = g.integers(-30000, 30000, size=(int(cu[-1]) + B, 7)).astype(np.int16)   # 14-byte rows: byte copies
    ref = O.prepare_next_step(ot, a, pos, bt, 8, 9, cu=cu, hidden=hid)
    got = gpu_prepare(sv, dev, ot, a, pos, bt, 8, 9, cu_num_draft_tokens=cuda(cu, dev), hidden=cuda(hid, dev))
    same_prepare(got, ref)


def test_prepare_clamps_accepted_counts(sv, dev):
    import torch
    ot = np.arange(12, dtype=np.int32).reshape(2, 6)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    got = gpu_prepare(sv, dev, ot, np.array([9, -2], np.int32), np.zeros(2, np.int32), np.zeros((2, 2), np.int32),
                      16, 1, rows_per_req=6, status=st)
    assert got["next_token"].tolist() == [5, 6]
    assert int(st.item()) & sv.STATUS_BAD_OFFSETS


def gpu_compact(sv, dev, kv, slots, paths, out_len, status=None):
    t = cuda(kv, dev)
    sv.compact_tree_kv(t, cuda(slots, dev), cuda(paths, dev), cuda(out_len, dev), status=status)
    return t.cpu().numpy()


def compact_case(seed, parent, B, row, paths=None):
    g = np.random.default_rng(seed)
    N1 = parent.shape[0]
    if paths is None:
        paths = ns.random_paths(parent, B, seed + 1)
    num_slots = B * N1 + 37
    slots = g.permutation(num_slots)[:B * N1].reshape(B, N1).astype(np.int64)
    kv = g.integers(0, 256, size=(num_slots, row)).astype(np.uint8)
    out_len = (paths >= 0).sum(axis=1).astype(np.int32)
    return kv, slots, paths, out_len


@pytest.mark.parametrize("row", [16, 96, 4096 + 16])
def test_compaction_parity(sv, O, dev, row):
    parent = W.parents_in_order((4, 2, 2, 1, 1))
    kv, slots, paths, out_len = compact_case(520 + row, parent, 300, row)
    ref = O.compact_tree_kv(kv, slots, paths, out_len)["kv"]
    assert (gpu_compact(sv, dev, kv, slots, paths, out_len) == ref).all()


def test_compaction_sources_that_are_destinations(sv, O, dev):
    parent = W.parents_in_order((4, 2, 2))
    paths = np.array([[0, 2, 7, 16], [0, 3, 4, 13], [0, 1, 2, -1], [0, 4, 12, 28], [0, -1, -1, -1]], np.int32)
    kv, slots, paths, out_len = compact_case(530, parent, 5, 64, paths=paths)
    ref = O.compact_tree_kv(kv, slots, paths, out_len)["kv"]
    assert (gpu_compact(sv, dev, kv, slots, paths, out_len) == ref).all()


def test_compaction_deep_chain_groups(sv, O, dev):
    """Depth 40 with nodes shifted by one: every group of eight copies reads
    rows the next group overwrites."""
    parent = np.concatenate([[-1], np.arange(0, 60)]).astype(np.int32)   # a chain of 60 nodes
    paths = np.full((3, 61), -1, np.int32)
    paths[0, :41] = np.arange(41)
    paths[1, :41] = np.concatenate([[0], np.arange(2, 42)])
    paths[2, :31] = np.concatenate([[0], np.arange(20, 50)])
    kv, slots, paths, out_len = compact_case(531, parent, 3, 32, paths=paths)
    ref = O.compact_tree_kv(kv, slots, paths, out_len)["kv"]
    assert (gpu_compact(sv, dev, kv, slots, paths, out_len) == ref).all()


def test_compaction_status(sv, dev):
    import torch
    parent = W.parents_in_order((2, 2))
    kv = np.arange(160, dtype=np.uint8).reshape(10, 16)
    slots = np.array([[0, 1, 2, 3, 4, 5, 6], [0, 1, 2, 3, 4, 5, 6]], np.int64)
    slots[1, 5] = 99                                                   # outside the cache
    paths = np.array([[0, 2, 1], [0, 2, 5]], np.int32)                 # request 0 does not increase
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out = gpu_compact(sv, dev, kv, slots, paths, np.array([3, 3], np.int32), status=st)
    assert int(st.item()) & sv.STATUS_BAD_OFFSETS and int(st.item()) & sv.STATUS_SLOT_RANGE
    want = kv.copy()
    want[1] = kv[2]                                                    # request 1, depth 1; depth 2 skipped
    assert (out == want).all()


def test_tree_verify_then_compact(sv, O, dev):
    """The sampled tree's own paths drive the compaction."""
    import torch
    x = W.tree_sampled(seed=540, B=24, V=3000)
    p, t, n = sv.verify_tree_sampled(cuda(x.logits, dev), cuda(x.draft_probs, dev), cuda(x.node_tokens, dev),
                                     x.parent, cuda(x.temperature, dev), cuda(x.u_accept, dev), cuda(x.u_sample, dev))
    g = np.random.default_rng(541)
    num_slots = x.B * (x.N + 1) + 11
    slots = g.permutation(num_slots)[:x.B * (x.N + 1)].reshape(x.B, x.N + 1).astype(np.int64)
    kv = g.integers(0, 256, size=(num_slots, 256)).astype(np.uint8)
    ref = O.compact_tree_kv(kv, slots, p.cpu().numpy(), n.cpu().numpy())["kv"]
    kt = cuda(kv, dev)
    sv.compact_tree_kv(kt, cuda(slots, dev), p, n)
    assert (kt.cpu().numpy() == ref).all()
    torch.cuda.synchronize(dev)
