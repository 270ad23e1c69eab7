"""The C-ABI library: it loads, exports every declared symbol, and its host-side
checks and host helper work without a GPU (no device work is requested here)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_chain_gb300 import build
    build.build()
    import speculative_decoding_verification_chain_gb300 as sv
    return sv.load_library()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"spec_verify_chain", "spec_verify_tree", "spec_fixup_slots", "spec_workspace_bytes",
            "spec_tree_from_choices"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_bytes(lib):
    a = lib.spec_workspace_bytes(64, 6, 128256, 0)
    b = lib.spec_workspace_bytes(128, 6, 128256, 0)
    assert 0 < a < b
    assert lib.spec_workspace_bytes(0, 6, 100, 0) == 0
    assert lib.spec_workspace_bytes(1, 257, 100, 0) == 0
    assert lib.spec_workspace_bytes(1, 2, 0, 0) == 0


def _chain(lib, **kw):
    args = dict(z=0x10000, dtype=0, q=None, tok=0x20000, T=None, ua=None, us=None, B=2, k=3, V=100,
                out=0x30000, na=0x40000, st=None, ws=0x50000, wsb=1 << 30, stream=None)
    args.update(kw)
    return lib.spec_verify_chain(args["z"], args["dtype"], args["q"], args["tok"], args["T"], args["ua"],
                                 args["us"], args["B"], args["k"], args["V"], args["out"], args["na"],
                                 args["st"], args["ws"], args["wsb"], args["stream"])


@pytest.mark.parametrize("bad", [
    dict(B=0), dict(k=0), dict(k=256), dict(V=0), dict(V=1 << 30), dict(dtype=7), dict(z=None),
    dict(tok=None), dict(out=None), dict(na=None), dict(z=0x10008),
    dict(T=0x60000),                                   # sampled pointers given only partly
    dict(q=0x70004, T=0x60000, ua=0x80000, us=0x90000),  # misaligned draft_probs
    dict(ws=None), dict(wsb=16), dict(ws=0x50004),
])
def test_chain_host_checks_reject_bad_arguments(lib, bad):
    assert _chain(lib, **bad) == 1
    assert lib.spec_last_error() != b""


def _ragged(lib, **kw):
    args = dict(z=0x10000, dtype=0, q=None, tok=0x20000, cu=0x28000, total=5, T=None, ua=None, us=None, B=2,
                max_k=3, V=100, out=0x30000, na=0x40000, st=None, ws=0x50000, wsb=1 << 30, stream=None)
    args.update(kw)
    return lib.spec_verify_chain_ragged(args["z"], args["dtype"], args["q"], args["tok"], args["cu"], args["total"],
                                        args["T"], args["ua"], args["us"], args["B"], args["max_k"], args["V"],
                                        args["out"], args["na"], args["st"], args["ws"], args["wsb"], args["stream"])


@pytest.mark.parametrize("bad", [
    dict(B=0), dict(max_k=-1), dict(max_k=256), dict(V=0), dict(total=-1), dict(total=7),   # 7 > B * max_k
    dict(cu=None), dict(tok=None), dict(z=None), dict(out=None), dict(z=0x10008), dict(dtype=3),
    dict(T=0x60000), dict(ws=None), dict(wsb=16),
])
def test_ragged_host_checks_reject_bad_arguments(lib, bad):
    assert _ragged(lib, **bad) == 1
    assert lib.spec_last_error() != b""


def test_ragged_fixup_host_checks(lib):
    assert lib.spec_fixup_slots_ragged(None, 2, 0x1000, 3, 0x2000, -1, None) == 1
    assert lib.spec_fixup_slots_ragged(0x3000, 2, None, 3, 0x2000, -1, None) == 1
    assert lib.spec_fixup_slots_ragged(0x3000, 2, 0x1000, 3, None, -1, None) == 1
    assert lib.spec_fixup_slots_ragged(0x3000, -1, 0x1000, 3, 0x2000, -1, None) == 1
    assert lib.spec_fixup_slots_ragged(None, 0, None, 0, None, -1, None) == 0


def test_tree_sampled_host_checks(lib):
    import ctypes
    par = (ctypes.c_int32 * 4)(-1, 0, 0, 1)
    bad_par = (ctypes.c_int32 * 4)(-1, 0, 3, 1)

    def call(B=2, N=3, V=100, depth=2, z=0x1000, q=0x2000, tok=0x3000, parent=par, T=0x4000, ua=0x5000,
             us=0x6000, op=0x7000, ot=0x8000, ol=0x9000, dtype=0):
        return lib.spec_verify_tree_sampled(z, dtype, q, tok, parent, T, ua, us, B, N, V, depth, op, ot, ol,
                                            None, None)
    for bad in (dict(B=0), dict(N=-1), dict(N=256), dict(V=0), dict(V=409601), dict(depth=1), dict(depth=-1),
                dict(parent=bad_par), dict(z=None), dict(q=None), dict(tok=None), dict(T=None), dict(ua=None),
                dict(us=None), dict(op=None), dict(ot=None), dict(ol=None), dict(z=0x1008), dict(q=0x2004),
                dict(dtype=7)):
        assert call(**bad) == 1, bad
        assert lib.spec_last_error() != b""


def test_fused_chain_host_checks(lib):
    # slot_mapping is required; the rest is checked as for spec_verify_chain
    rc = lib.spec_verify_chain_fused(0x1000, 0, None, 0x2000, None, None, None, 2, 3, 100, 0x3000, 0x4000,
                                     None, -1, None, 0x5000, 1 << 20, None)
    assert rc == 1 and lib.spec_last_error() != b""
    rc = lib.spec_verify_chain_fused(0x1000, 0, None, 0x2000, None, None, None, 0, 3, 100, 0x3000, 0x4000,
                                     0x6000, -1, None, 0x5000, 1 << 20, None)
    assert rc == 1


def test_next_step_host_checks(lib):
    def call(ot=0x1000, stride=4, na=0x2000, pos=0x3000, bt=0x4000, mb=4, bs=16, B=2, P=3, rpr=4, cu=None,
             hid=None, rb=0, nt=0x5000, npos=0x6000, ns=0x7000):
        return lib.spec_prepare_next_step(ot, stride, na, pos, bt, mb, bs, B, P, rpr, cu, hid, rb, -1, nt, npos,
                                          ns, None, None, None, None)
    for bad in (dict(B=-1), dict(stride=0), dict(mb=-1), dict(bs=0), dict(P=-1), dict(rpr=0), dict(ot=None),
                dict(na=None), dict(pos=None), dict(nt=None), dict(npos=None), dict(bt=None), dict(ns=None),
                dict(hid=0x8000, rb=0)):
        assert call(**bad) == 1, bad
        assert lib.spec_last_error() != b""
    assert call(B=0) == 0


def test_compact_host_checks(lib):
    def call(kv=0x1000, ns=100, rb=64, sm=0x2000, ss=7, pa=0x3000, ps=4, ol=0x4000, B=2):
        return lib.spec_compact_tree_kv(kv, ns, rb, sm, ss, pa, ps, ol, B, None, None)
    for bad in (dict(B=-1), dict(ns=-1), dict(rb=8), dict(rb=40), dict(ss=0), dict(ps=0), dict(ps=257),
                dict(kv=None), dict(sm=None), dict(pa=None), dict(ol=None), dict(kv=0x1008)):
        assert call(**bad) == 1, bad
        assert lib.spec_last_error() != b""
    assert call(B=0) == 0 and call(ns=0) == 0


def test_ngram_host_checks(lib):
    def call(B=2, Lmax=10, nmin=1, nmax=4, k=3, tok=0x1000, ln=0x2000, d=0x3000, c=0x4000):
        return lib.spec_ngram_propose(tok, ln, B, Lmax, nmin, nmax, k, d, c, None, None, None)
    for bad in (dict(B=-1), dict(Lmax=-1), dict(nmin=0), dict(nmax=0), dict(nmin=3, nmax=2), dict(nmax=65),
                dict(k=-1), dict(tok=None), dict(ln=None), dict(d=None), dict(c=None)):
        assert call(**bad) == 1, bad
        assert lib.spec_last_error() != b""
    assert call(B=0, tok=None, ln=None, d=None, c=None) == 0


def test_tree_host_checks(lib):
    par = np.array([-1, 0, 0, 1], np.int32)
    bad_par = np.array([-1, 0, 2, 1], np.int32)
    P = ctypes.c_void_p

    def call(parent, N=3, max_depth=2, z=0x10000):
        return lib.spec_verify_tree(z, 0, 0x20000, parent.ctypes.data, 2, N, 50, max_depth, 0x30000, 0x40000,
                                    0x50000, None, 0x60000, 1 << 30, None)
    assert call(bad_par) == 1
    assert call(par, max_depth=1) == 1
    assert call(np.array([0, 0, 0, 1], np.int32)) == 1
    assert call(par, z=0x10002) == 1


def test_fixup_host_checks(lib):
    assert lib.spec_fixup_slots(0x1000, 2, 3, None, None, 0, -1, None) == 1
    assert lib.spec_fixup_slots(None, 2, 3, 0x2000, None, 0, -1, None) == 1
    assert lib.spec_fixup_slots(0x1000, -1, 3, 0x2000, None, 0, -1, None) == 1
    assert lib.spec_fixup_slots(0x1000, 2, 3, None, 0x3000, 0, -1, None) == 1
    assert lib.spec_fixup_slots(None, 0, 3, None, None, 0, -1, None) == 0


def test_tree_from_choices_matches_oracle(lib, oracle_mod):
    import speculative_decoding_verification_chain_gb300 as sv
    from speculative_decoding_verification_chain_gb300 import workloads as W
    for shape in [(4, 2, 2, 1, 1), (3, 1), (1,), (2, 2, 2, 2)]:
        choices = W.level_tree_choices(shape)
        got = sv.tree_from_choices(choices)
        meta = oracle_mod.tree_level_metadata(choices)
        assert (got["parent"] == oracle_mod.parent_from_choices(choices)).all()
        assert got["cu_drafts_per_level"] == meta["cu_drafts_per_level"]
        assert got["child_drafts_per_level"] == meta["child_drafts_per_level"]
        assert got["depth"] == meta["depth"]
    # an irregular tree (per-branch fan-out differs)
    choices = [(0,), (1,), (0, 0), (0, 1), (1, 0), (0, 0, 0)]
    got = sv.tree_from_choices(choices)
    assert list(got["parent"]) == list(oracle_mod.parent_from_choices(choices))
    with pytest.raises(sv.SpecError):
        sv.tree_from_choices([(0, 0), (0,)])          # not level order
    with pytest.raises(sv.SpecError):
        sv.tree_from_choices([(0,), (1, 0)])          # prefix (1,) missing
