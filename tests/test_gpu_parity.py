"""GPU parity: the CUDA path against the CPU oracle on the same seeded inputs.

Greedy chains, trees, accepted counts and slot maps must be bit-exact.  Sampled
tokens must be bit-exact except at positions the oracle flags (|u - p/q| < 1e-6
for an accept test, or the inverse-CDF threshold within 1e-5 relative of a
bucket edge).  Every call goes through the C ABI via the package binding.
"""
import numpy as np
import pytest

from speculative_decoding_verification_chain_gb300 import workloads as W

from helpers import compare_chain, cuda, oracle_chain, run_chain

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


@pytest.fixture(scope="module")
def O(oracle_mod):
    return oracle_mod


# ------------------------------------------------------------------ greedy --
GREEDY_SHAPES = [
    (1, 1, 1), (1, 1, 7), (3, 2, 255), (2, 3, 256), (4, 5, 257), (5, 4, 8191), (6, 3, 8192),
    (7, 2, 8193), (16, 5, 20011), (4, 8, 40000), (3, 31, 1000), (2, 255, 300),
]


@pytest.mark.parametrize("dtype", [W.BF16, W.FP32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("shape", GREEDY_SHAPES, ids=[str(s) for s in GREEDY_SHAPES])
def test_greedy_chain_bit_exact(sv, O, dev, shape, dtype):
    B, k, V = shape
    x = W.chain_greedy(seed=1000 + B * 7 + k, B=B, k=k, V=V, p_match=0.8, dtype=dtype)
    got_t, got_a = run_chain(sv, x, dev)
    ref = oracle_chain(O, x)
    assert (got_a == ref["num_accepted"]).all()
    assert (got_t == ref["out_tokens"]).all()


@pytest.mark.parametrize("p_match", [0.0, 1.0])
def test_greedy_always_wrong_and_always_right(sv, O, dev, p_match):
    x = W.chain_greedy(seed=31, B=8, k=5, V=128256, p_match=p_match)
    zf = W.logits_as_f32(x.logits, x.dtype)
    am = np.argmax(zf, axis=-1)
    if p_match == 0.0:
        x.draft_tokens = ((am[:, :5] + 1) % x.V).astype(np.int32)
    got_t, got_a = run_chain(sv, x, dev)
    if p_match == 0.0:
        assert (got_a == 0).all() and (got_t[:, 0] == am[:, 0]).all() and (got_t[:, 1:] == -1).all()
    else:
        assert (got_a == 5).all() and (got_t == am).all()


def test_greedy_ties_across_chunks_take_lowest_index(sv, O, dev):
    B, k, V = 6, 3, 3 * 8192 + 100
    g = np.random.default_rng(5)
    z = (g.standard_normal((B, k + 1, V)) * 0.5).astype(np.float32)
    top = np.float32(9.0)
    for b in range(B):
        for i in range(k + 1):
            pos = np.sort(g.choice(V, size=4, replace=False))
            z[b, i, pos] = top
    bits = W.f32_to_bf16_bits(z)
    zf = W.bf16_bits_to_f32(bits)
    am = np.argmax(zf, axis=-1).astype(np.int32)
    tok = am[:, :k].copy()
    tok[1, 1] = (tok[1, 1] + 1) % V
    x = W.ChainInputs(logits=bits, dtype=W.BF16, draft_tokens=tok, temperature=np.zeros(B, np.float32),
                      u_sample=np.zeros((B, k + 1), np.float32))
    got_t, got_a = run_chain(sv, x, dev)
    ref = oracle_chain(O, x)
    assert (got_a == ref["num_accepted"]).all() and (got_t == ref["out_tokens"]).all()


def test_greedy_full_size_chain(sv, O, dev):
    x = W.chain_greedy(seed=2, B=64, k=5, V=128256, p_match=0.8)
    got_t, got_a = run_chain(sv, x, dev)
    ref = oracle_chain(O, x)
    assert (got_a == ref["num_accepted"]).all()
    assert (got_t == ref["out_tokens"]).all()


def test_out_of_range_tokens_are_rejections_and_flagged(sv, O, dev):
    import torch
    x = W.chain_greedy(seed=41, B=4, k=3, V=5000, p_match=1.0)
    x.draft_tokens[:, 1] = np.array([-1, 5000, 1 << 29, -(1 << 29)], np.int32)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    got_t, got_a = run_chain(sv, x, dev, status=st)
    ref = oracle_chain(O, x)
    assert (got_a == ref["num_accepted"]).all() and (got_t == ref["out_tokens"]).all()
    assert int(st.item()) & sv.STATUS_TOKEN_RANGE


def test_nonfinite_logit_sets_status(sv, dev):
    import torch
    x = W.chain_greedy(seed=42, B=2, k=2, V=3000, p_match=1.0, dtype=W.FP32)
    x.logits[1, 0, 17] = np.nan
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    run_chain(sv, x, dev, status=st)
    assert int(st.item()) & sv.STATUS_NONFINITE


def _mask_vocab(x, V):
    """-inf over whole 256-element blocks, a ragged stretch and the row tail
    (a masked vocabulary: those tokens have probability 0)."""
    neg = np.uint16(0xFF80) if x.dtype == W.BF16 else np.float32(-np.inf)
    spans = [(256, 256 + 3 * 256), (3000, 3000 + 777), (V - 1100, V)]
    for lo, hi in spans:
        x.logits[:, :, lo:hi] = neg
    return x


@pytest.mark.parametrize("dtype", [W.BF16, W.FP32], ids=["bf16", "fp32"])
def test_masked_vocabulary_greedy(sv, O, dev, dtype):
    import torch
    x = _mask_vocab(W.chain_greedy(seed=43, B=12, k=4, V=20011, p_match=0.8, dtype=dtype), 20011)
    x.draft_tokens[0, 0] = 300     # a masked draft token is rejected
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    got_t, got_a = run_chain(sv, x, dev, status=st)
    ref = oracle_chain(O, x)
    assert int(st.item()) == 0
    assert (got_a == ref["num_accepted"]).all() and (got_t == ref["out_tokens"]).all()
    assert got_a[0] == 0


@pytest.mark.parametrize("dtype", [W.BF16, W.FP32], ids=["bf16", "fp32"])
def test_masked_vocabulary_sampled(sv, O, dev, dtype):
    import torch
    V = 20011
    x = _mask_vocab(W.chain_sampled(seed=44, B=12, k=4, V=V, temperature=0.8, lam=0.3, dtype=dtype), V)
    x.draft_tokens[0, 0] = 300     # p = 0 at a masked token: always rejected
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    got_t, got_a = run_chain(sv, x, dev, status=st)
    ref = oracle_chain(O, x)
    assert int(st.item()) == 0
    compare_chain(got_t, got_a, ref)
    masked = np.zeros(V, bool)
    for lo, hi in [(256, 1024), (3000, 3777), (V - 1100, V)]:
        masked[lo:hi] = True
    # no emitted token (accepted draft, residual or bonus sample) is masked
    emitted = got_t[got_t >= 0]
    assert not masked[emitted].any()
    assert got_a[0] == 0


def test_all_masked_row_sets_status(sv, dev):
    import torch
    x = W.chain_sampled(seed=45, B=3, k=2, V=3000, temperature=1.0, lam=0.3, dtype=W.FP32)
    x.logits[2, 1, :] = -np.inf
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    run_chain(sv, x, dev, status=st)
    assert int(st.item()) & sv.STATUS_NONFINITE


# ----------------------------------------------------------------- sampled --
SAMPLED = [
    dict(B=16, k=4, V=5000, temperature=0.7, lam=0.3),
    dict(B=16, k=4, V=20011, temperature=1.0, lam=0.1),
    dict(B=12, k=6, V=8193, temperature=0.5, lam=0.6),
    dict(B=8, k=1, V=257, temperature=1.3, lam=0.3),
    dict(B=8, k=3, V=1, temperature=1.0, lam=0.3),
    dict(B=9, k=8, V=30000, temperature=0.9, lam=0.3, dtype=W.FP32),
]


@pytest.mark.parametrize("cfg", SAMPLED, ids=[str(i) for i in range(len(SAMPLED))])
def test_sampled_chain_matches_oracle_modulo_flags(sv, O, dev, cfg):
    x = W.chain_sampled(seed=2000 + cfg["V"], **cfg)
    got_t, got_a = run_chain(sv, x, dev)
    ref = oracle_chain(O, x)
    res = compare_chain(got_t, got_a, ref)
    assert res["mismatch"] <= res["flagged"]


def test_tiny_chain_trials(sv, O, dev):
    x = W.chain_tiny(seed=1, trials=1000)
    got_t, got_a = run_chain(sv, x, dev)
    ref = oracle_chain(O, x)
    compare_chain(got_t, got_a, ref)


def test_q_equal_p_accepts_every_draft(sv, O, dev):
    g = np.random.default_rng(7)
    B, k, V, T = 64, 4, 3000, 0.9
    z = (g.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    s = z[:, :k].astype(np.float64) / T
    q = np.exp(s - s.max(-1, keepdims=True))
    q = (q / q.sum(-1, keepdims=True)).astype(np.float32)
    tok = np.stack([[g.choice(V, p=q[b, i] / q[b, i].sum()) for i in range(k)] for b in range(B)]).astype(np.int32)
    x = W.ChainInputs(logits=z, dtype=W.FP32, draft_tokens=tok, temperature=np.full(B, T, np.float32),
                      u_sample=W.method_uniforms(g, (B, k + 1)), draft_probs=q,
                      u_accept=W.method_uniforms(g, (B, k)))
    got_t, got_a = run_chain(sv, x, dev)
    ref = oracle_chain(O, x)
    compare_chain(got_t, got_a, ref)
    assert ((got_a == k) | (ref["flag_accept"].sum(1) > 0)).all()


def test_zero_draft_probability_accepts(sv, O, dev):
    x = W.chain_sampled(seed=77, B=8, k=3, V=4000, temperature=1.0, lam=0.3)
    for b in range(x.B):
        x.draft_probs[b, 0, x.draft_tokens[b, 0]] = 0.0
    got_t, got_a = run_chain(sv, x, dev)
    ref = oracle_chain(O, x)
    compare_chain(got_t, got_a, ref)
    assert (got_a >= 1).all()


def test_sampled_out_of_range_drafts_are_rejections(sv, O, dev):
    """p(x) = 0 outside the vocabulary: rejected even at u = 0, the token at
    that position is the residual draw, and the status word says so."""
    import torch
    x = W.chain_sampled(seed=79, B=8, k=3, V=4000, temperature=1.0, lam=0.3)
    x.u_accept[:, 0] = 0.0
    x.draft_tokens[:, 0] = np.array([-1, 4000, 1 << 29, -(1 << 29)] * 2, np.int32)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    got_t, got_a = run_chain(sv, x, dev, status=st)
    ref = oracle_chain(O, x)
    compare_chain(got_t, got_a, ref)
    assert (got_a == 0).all() and (ref["num_accepted"] == 0).all()
    assert int(st.item()) & sv.STATUS_TOKEN_RANGE


def test_mixed_greedy_and_sampled_batch(sv, O, dev):
    x = W.chain_mixed(seed=88, B=24, k=4, V=12000)
    got_t, got_a = run_chain(sv, x, dev)
    ref = oracle_chain(O, x)
    compare_chain(got_t, got_a, ref)
    greedy = x.temperature == 0
    assert (got_a[greedy] == ref["num_accepted"][greedy]).all()
    assert (got_t[greedy] == ref["out_tokens"][greedy]).all()


@pytest.mark.parametrize("lam", [0.1, 0.3, 0.6])
def test_sampled_full_size_zipf(sv, O, dev, lam):
    x = W.chain_sampled(seed=3, B=32, k=4, V=128256, temperature=0.7, lam=lam)
    got_t, got_a = run_chain(sv, x, dev)
    ref = oracle_chain(O, x)
    res = compare_chain(got_t, got_a, ref)
    print("lam", lam, res)


@pytest.mark.parametrize("B", [1, 8, 64, 256])
def test_sweep_full_size_with_slot_fixup(sv, O, dev, B):
    import torch
    x = W.named("sweep", B=B)
    got_t, got_a = run_chain(sv, x, dev)
    rows = np.arange(B) if B <= 64 else np.random.default_rng(9).choice(B, 48, replace=False)
    ref = oracle_chain(O, x, rows=rows)
    compare_chain(got_t[rows], got_a[rows], ref)
    slots = cuda(x.slot_mapping, dev)
    sv.fixup_slots(slots, num_accepted=torch.from_numpy(got_a).to(dev))
    exp = O.fixup_slots(x.slot_mapping, num_accepted=got_a)
    assert (slots.cpu().numpy() == exp).all()


# ------------------------------------------------- fused slot fix-up --
FUSED = [("greedy", dict(B=64, k=5, V=128256)), ("greedy", dict(B=7, k=31, V=1000)),
         ("greedy", dict(B=3, k=255, V=300)), ("sampled", dict(B=32, k=4, V=128256)),
         ("sampled", dict(B=9, k=8, V=5003)), ("mixed", dict(B=24, k=6, V=20011))]


@pytest.mark.parametrize("kind,cfg", FUSED, ids=["%s-%d-%d-%d" % (k_, c["B"], c["k"], c["V"]) for k_, c in FUSED])
def test_fused_fixup_matches_the_separate_fixup(sv, O, dev, kind, cfg):
    """spec_verify_chain_fused: the same tokens and counts as spec_verify_chain,
    and the slot map the oracle's fix-up writes for those counts."""
    import torch
    if kind == "greedy":
        x = W.chain_greedy(seed=60 + cfg["k"], **cfg)
    elif kind == "sampled":
        x = W.chain_sampled(seed=61 + cfg["k"], temperature=0.8, lam=0.4, **cfg)
    else:
        x = W.chain_mixed(seed=62, **cfg)
    sampled = x.draft_probs is not None
    args = [cuda(x.logits, dev), cuda(x.draft_tokens, dev)]
    if sampled:
        args += [cuda(x.temperature, dev), cuda(x.u_accept, dev), cuda(x.u_sample, dev), cuda(x.draft_probs, dev)]
    slots = cuda(x.slot_mapping, dev)
    ot, na = sv.verify_chain(*args, slot_mapping=slots, padding_slot_id=-7)
    ot2, na2 = sv.verify_chain(*args)
    torch.cuda.synchronize(dev)
    got_a = na.cpu().numpy()
    assert (ot.cpu().numpy() == ot2.cpu().numpy()).all() and (got_a == na2.cpu().numpy()).all()
    ref = oracle_chain(O, x)
    compare_chain(ot.cpu().numpy(), got_a, ref)
    assert (slots.cpu().numpy() == O.fixup_slots(x.slot_mapping, num_accepted=got_a, pad=-7)).all()


# -------------------------------------------------------------------- tree --
TREES = [(4, 2, 2, 1, 1), (3, 3, 1), (1, 1, 1, 1), (5,), (2, 2, 2, 2, 2, 2)]


@pytest.mark.parametrize("dtype", [W.BF16, W.FP32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("shape", TREES, ids=[str(t) for t in TREES])
def test_tree_bit_exact(sv, O, dev, shape, dtype):
    t = W.tree_greedy(seed=300 + len(shape), B=12, V=9001, children_per_level=shape, p_match=0.75, dtype=dtype)
    path, toks, ln = sv.verify_tree(cuda(t.logits, dev), cuda(t.node_tokens, dev), t.parent)
    ref = O.verify_tree(t.logits, t.dtype, t.node_tokens, t.parent)
    assert (path.cpu().numpy() == ref["path"]).all()
    assert (toks.cpu().numpy() == ref["tokens"]).all()
    assert (ln.cpu().numpy() == ref["length"]).all()


def test_tree_root_only(sv, O, dev):
    t = W.tree_greedy(seed=5, B=3, V=777, parent=np.array([-1], np.int32))
    path, toks, ln = sv.verify_tree(cuda(t.logits, dev), cuda(np.zeros((3, 0), np.int32), dev), [-1])
    ref = O.verify_tree(t.logits, t.dtype, np.zeros((3, 0), np.int32), np.array([-1], np.int32))
    assert (toks.cpu().numpy() == ref["tokens"]).all() and (ln.cpu().numpy() == 1).all()


def test_tree_full_size_with_slot_fixup(sv, O, dev):
    t = W.tree_greedy(seed=4, B=16, V=128256)
    path, toks, ln = sv.verify_tree(cuda(t.logits, dev), cuda(t.node_tokens, dev), t.parent)
    ref = O.verify_tree(t.logits, t.dtype, t.node_tokens, t.parent)
    assert (path.cpu().numpy() == ref["path"]).all()
    assert (toks.cpu().numpy() == ref["tokens"]).all()
    assert (ln.cpu().numpy() == ref["length"]).all()
    slots = cuda(t.slot_mapping, dev)
    sv.fixup_slots(slots, path=path)
    assert (slots.cpu().numpy() == O.fixup_slots(t.slot_mapping, path=ref["path"])).all()


def test_chain_equals_tree_with_unit_fanout(sv, dev):
    x = W.chain_greedy(seed=61, B=20, k=6, V=30000, p_match=0.8)
    got_t, got_a = run_chain(sv, x, dev)
    parent = np.arange(-1, x.k, dtype=np.int32)
    path, toks, ln = sv.verify_tree(cuda(x.logits, dev), cuda(x.draft_tokens, dev), parent)
    assert (ln.cpu().numpy() == got_a + 1).all()
    assert (toks.cpu().numpy() == got_t).all()


# ----------------------------------------------------------------- fix-up --
def test_fixup_slots_chain_and_tree_modes(sv, O, dev):
    import torch
    g = np.random.default_rng(3)
    B, P = 33, 9
    s = W.slot_map(g, B, P)
    a = g.integers(0, P, size=B).astype(np.int32)
    st = cuda(s, dev)
    sv.fixup_slots(st, num_accepted=cuda(a, dev))
    assert (st.cpu().numpy() == O.fixup_slots(s, num_accepted=a)).all()
    path = np.full((B, 4), -1, np.int32)
    path[:, 0] = 0
    for b in range(B):
        d = g.integers(0, 4)
        path[b, 1:1 + d] = np.sort(g.choice(np.arange(1, P), d, replace=False))
    st = cuda(s, dev)
    sv.fixup_slots(st, path=cuda(path, dev), padding_slot_id=-5)
    assert (st.cpu().numpy() == O.fixup_slots(s, path=path, pad=-5)).all()


# ------------------------------------------------------------- workspace --
def test_workspace_is_left_clean_between_calls(sv, O, dev):
    """Back-to-back calls of different kinds and sizes on one workspace give the
    same answers as fresh calls (the kernel clears its own counters)."""
    xs = [W.chain_greedy(seed=90, B=5, k=4, V=20000),
          W.chain_sampled(seed=91, B=7, k=3, V=9000, temperature=0.8, lam=0.3),
          W.chain_greedy(seed=92, B=9, k=2, V=777)]
    t = W.tree_greedy(seed=93, B=4, V=5000)
    refs = [oracle_chain(O, x) for x in xs]
    tref = O.verify_tree(t.logits, t.dtype, t.node_tokens, t.parent)
    for rep in range(3):
        for x, ref in zip(xs, refs):
            got_t, got_a = run_chain(sv, x, dev)
            compare_chain(got_t, got_a, ref)
            if x.draft_probs is None:
                assert (got_t == ref["out_tokens"]).all()
        path, toks, ln = sv.verify_tree(cuda(t.logits, dev), cuda(t.node_tokens, dev), t.parent)
        assert (toks.cpu().numpy() == tref["tokens"]).all()


# ------------------------------------------- skipped rows, producer run-ahead --
@pytest.fixture
def tuning(sv):
    """spec_set_tuning for one test, put back to automatic afterwards."""
    yield sv.set_tuning
    sv.set_tuning(0, 0, 0)


@pytest.mark.parametrize("ahead,splits", [(2, 0), (3, 0), (3, 3), (2, 1)])
def test_results_do_not_depend_on_producer_run_ahead(sv, O, dev, ahead, splits, tuning):
    """How many stages the producer keeps in flight, and how finely rows are
    split, change the timing of claims and so which rows are skipped; the
    answers must not change."""
    tuning(splits, ahead, 1)
    x = W.chain_greedy(seed=61 + ahead, B=16, k=5, V=128256, p_match=0.5)
    got_t, got_a = run_chain(sv, x, dev)
    ref = oracle_chain(O, x)
    assert (got_a == ref["num_accepted"]).all() and (got_t == ref["out_tokens"]).all()
    t = W.tree_greedy(seed=62 + ahead + splits, B=4, V=50000)
    path, toks, ln = sv.verify_tree(cuda(t.logits, dev), cuda(t.node_tokens, dev), t.parent)
    r = O.verify_tree(t.logits, t.dtype, t.node_tokens, t.parent)
    assert (ln.cpu().numpy() == r["length"]).all()
    assert (path.cpu().numpy() == r["path"]).all() and (toks.cpu().numpy() == r["tokens"]).all()
    xs = W.chain_sampled(seed=63 + ahead, B=8, k=4, V=30000, temperature=0.8, lam=0.3)
    got_t, got_a = run_chain(sv, xs, dev)
    compare_chain(got_t, got_a, oracle_chain(O, xs))


def test_rejected_first_drafts_skip_later_rows(sv, O, dev, tuning):
    """Every first draft wrong: rows 1..k are never needed.  Many are skipped
    at claim (the first stage of row 0 already shows the rejection), and the
    counters stay consistent."""
    import torch
    tuning(0, 3, 1)
    x = W.chain_greedy(seed=64, B=32, k=5, V=128256, p_match=0.0)
    z, tok = cuda(x.logits, dev), cuda(x.draft_tokens, dev)
    ws = torch.zeros(sv.workspace_bytes(x.B, x.k + 1, x.V), dtype=torch.uint8, device=dev)
    ot, na = sv.verify_chain(z, tok, workspace=ws)
    c = sv.workspace_counters(ws)
    ref = oracle_chain(O, x)
    assert (na.cpu().numpy() == 0).all()
    assert (na.cpu().numpy() == ref["num_accepted"]).all() and (ot.cpu().numpy() == ref["out_tokens"]).all()
    units = c["a_loaded"] + c["a_skipped"]   # rows x splits per row
    assert units >= x.B * (x.k + 1) and units % (x.B * (x.k + 1)) == 0
    assert c["a_skipped"] > 0
    print("counters", c)
