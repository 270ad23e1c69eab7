"""Pins for the oracle's next-step preparation and tree KV compaction.

Source: vLLM EAGLE walkthrough, "slot mapping and KV-cache management" (the
next-step helpers are named there), and the EAGLE-3 review, "EAGLE-3
inference" step 5 (only the accepted path's KV is kept; drafting restarts
from the confirmed prefix).  The readings are stated in the golden file and
in the oracle.

Pinned by: hand-worked examples (golden file); the slot lookup against an
independent formulation (every request's block table expanded into the slot
of every position, then indexed); the hidden-row gather against numpy
indexing; compaction by its meaning (each path row is found at the depth's
slot afterwards, every other row unchanged), including paths whose nodes are
both a source and a destination.
"""
import os

import numpy as np
import pytest

from speculative_decoding_verification_chain_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "next_step_examples.txt")


def golden_case():
    rows = [l for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    out_tokens, a, pos, bt, nt, npos, slots, last = [], [], [], [], [], [], [], []
    for line in rows:
        f = [x.strip() for x in line.split("|")]
        out_tokens.append([int(v) for v in f[1].split()])
        a.append(int(f[2]))
        pos.append(int(f[3]))
        bt.append([int(v) for v in f[4].split()])
        t, p = map(int, f[5].split())
        nt.append(t)
        npos.append(p)
        slots.append([int(v) for v in f[6].split()])
        last.append(int(f[7]))
    arr = lambda v, dt=np.int32: np.array(v, dt)
    return dict(out_tokens=arr(out_tokens), a=arr(a), pos=arr(pos), bt=arr(bt), next_token=arr(nt),
                next_position=arr(npos), slots=arr(slots, np.int64), last_row=arr(last))


def test_hand_worked_examples(oracle_mod):
    g = golden_case()
    r = oracle_mod.prepare_next_step(g["out_tokens"], g["a"], g["pos"], g["bt"], 4, 3, rows_per_req=4)
    assert (r["next_token"] == g["next_token"]).all()
    assert (r["next_position"] == g["next_position"]).all()
    assert (r["next_slots"] == g["slots"]).all()
    assert (r["last_row"] == g["last_row"]).all()
    assert r["status"][0] & 1                    # two requests ran past their tables


def expanded_slots(block_table, block_size):
    """Slot of every position 0 .. max_blocks*block_size - 1 of each request,
    -1 where the table entry is negative."""
    bt = block_table.astype(np.int64)
    s = bt[:, :, None] * block_size + np.arange(block_size)[None, None, :]
    s = np.where(bt[:, :, None] >= 0, s, -1)
    return s.reshape(bt.shape[0], -1)


def random_case(seed, B=200, k=5, max_blocks=12, block_size=16, hidden=64):
    g = np.random.default_rng(seed)
    out_tokens = g.integers(0, 128256, size=(B, k + 1)).astype(np.int32)
    a = g.integers(0, k + 1, size=B).astype(np.int32)
    pos = g.integers(0, max_blocks * block_size - 2, size=B).astype(np.int32)
    bt = g.integers(0, 5000, size=(B, max_blocks)).astype(np.int32)
    bt[g.random((B, max_blocks)) < 0.05] = -1
    hid = g.standard_normal((B * (k + 1), hidden)).astype(np.float32)
    return out_tokens, a, pos, bt, hid


@pytest.mark.parametrize("P_next", [1, 6, 9])
def test_slots_match_the_expanded_block_table(oracle_mod, P_next):
    out_tokens, a, pos, bt, hid = random_case(50 + P_next)
    k1 = out_tokens.shape[1]
    r = oracle_mod.prepare_next_step(out_tokens, a, pos, bt, 16, P_next, rows_per_req=k1, hidden=hid)
    table = expanded_slots(bt, 16)
    for b in range(out_tokens.shape[0]):
        npos = int(pos[b]) + int(a[b]) + 1
        want = [int(table[b, x]) if x < table.shape[1] else -1 for x in range(npos, npos + P_next)]
        assert r["next_slots"][b].tolist() == want
        assert r["next_token"][b] == out_tokens[b, a[b]]
        assert r["next_position"][b] == npos
    assert (r["last_row"] == np.arange(len(a)) * k1 + a).all()
    assert (r["hidden_out"] == hid[r["last_row"]]).all()


def test_ragged_rows(oracle_mod):
    g = np.random.default_rng(61)
    B = 50
    ks = g.integers(0, 8, size=B)
    cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    out_tokens = g.integers(0, 1000, size=(B, 9)).astype(np.int32)
    a = np.array([g.integers(0, kk + 1) for kk in ks], np.int32)
    hid = g.standard_normal((int(cu[-1]) + B, 8)).astype(np.float32)
    r = oracle_mod.prepare_next_step(out_tokens, a, np.zeros(B, np.int32), np.zeros((B, 1), np.int32), 64, 0,
                                     cu=cu, hidden=hid)
    assert (r["last_row"] == cu[:-1] + np.arange(B) + a).all()
    assert (r["hidden_out"] == hid[r["last_row"]]).all()


# ------------------------------------------------------------ compaction --
def compaction_mismatches(O, paths, parent, lib=None, seed=70, row=48):
    """Rows of every request carry their own random bytes; after compaction the
    slot of depth i must hold what the slot of path[i] held before, and every
    other row must be unchanged.  Returns the number of broken rows."""
    g = np.random.default_rng(seed)
    B, D1 = paths.shape
    N1 = parent.shape[0]
    num_slots = B * N1 + 37
    slots = g.permutation(num_slots)[:B * N1].reshape(B, N1).astype(np.int64)
    kv = g.integers(0, 256, size=(num_slots, row)).astype(np.uint8)
    out_len = (paths >= 0).sum(axis=1).astype(np.int32)
    r = O.compact_tree_kv(kv, slots, paths, out_len, lib=lib)
    want = kv.copy()
    for b in range(B):
        for i in range(1, out_len[b]):
            want[slots[b, i]] = kv[slots[b, paths[b, i]]]
    return int((r["kv"] != want).any(axis=1).sum())


def random_paths(parent, B, seed):
    """Random root-to-node walks (each stops with probability 1/4 per level)."""
    g = np.random.default_rng(seed)
    depth = 0
    kids = [np.flatnonzero(parent == c) for c in range(parent.shape[0])]
    d = np.zeros(parent.shape[0], int)
    for n in range(1, parent.shape[0]):
        d[n] = d[parent[n]] + 1
    depth = d.max()
    out = -np.ones((B, depth + 1), np.int32)
    for b in range(B):
        c, i = 0, 0
        out[b, 0] = 0
        while kids[c].size and g.random() > 0.25:
            c = int(g.choice(kids[c]))
            i += 1
            out[b, i] = c
    return out


def test_compaction_moves_every_path_row(oracle_mod):
    parent = W.parents_in_order((4, 2, 2, 1, 1))
    paths = random_paths(parent, 300, 71)
    assert compaction_mismatches(oracle_mod, paths, parent) == 0


def test_compaction_with_nodes_that_are_source_and_destination(oracle_mod):
    """Path 0, 2, 7, 16 in the (4, 2, 2) tree: node 2 is the source of depth 1
    and the destination of depth 2, so depth 1 must get node 2's old row."""
    parent = W.parents_in_order((4, 2, 2))
    paths = np.array([[0, 2, 7, 16], [0, 3, 4, 13], [0, 1, 2, -1], [0, 4, 12, 28], [0, -1, -1, -1]], np.int32)
    assert compaction_mismatches(oracle_mod, paths, parent) == 0


def test_compaction_status_for_bad_slots(oracle_mod):
    parent = W.parents_in_order((2, 2))
    kv = np.arange(40, dtype=np.uint8).reshape(10, 4)
    slots = np.array([[0, 1, 2, 3, 4, 5, 6]], np.int64)
    slots[0, 4] = -1                                  # node 4 (a source) has no slot
    r = oracle_mod.compact_tree_kv(kv, slots, np.array([[0, 2, 4]], np.int32), np.array([3], np.int32))
    assert r["status"][0] & 1
    assert (r["kv"][1] == kv[2]).all() and (r["kv"][2] == kv[2]).all()
