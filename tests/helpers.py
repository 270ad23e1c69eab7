"""Shared helpers for the GPU parity tests: host arrays to CUDA tensors and the
comparison rules (bit-exact for integers; sampled tokens bit-exact except at
positions the oracle flags)."""
import numpy as np


def cuda(a, dev):
    import torch
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def run_chain(sv, x, dev, status=None, **kw):
    sampled = x.draft_probs is not None
    ot, na = sv.verify_chain(
        cuda(x.logits, dev), cuda(x.draft_tokens, dev),
        cuda(x.temperature, dev) if sampled else None,
        cuda(x.u_accept, dev) if sampled else None,
        cuda(x.u_sample, dev) if sampled else None,
        cuda(x.draft_probs, dev) if sampled else None, status=status, **kw)
    return ot.cpu().numpy(), na.cpu().numpy()


def oracle_chain(O, x, nthreads=8, rows=None):
    if rows is None:
        return O.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample,
                              x.draft_probs, x.u_accept, nthreads=nthreads)
    sl = lambda a: None if a is None else a[rows]
    return O.verify_chain(x.logits[rows], x.dtype, x.draft_tokens[rows], x.temperature[rows],
                          x.u_sample[rows], sl(x.draft_probs), sl(x.u_accept), nthreads=nthreads)


def compare_chain(got_tokens, got_a, ref, greedy_exact=True):
    """Returns dict(mismatch=..., flagged=..., positions=...) and asserts that
    every mismatch sits at a flagged position (greedy: no mismatch at all)."""
    B, k1 = got_tokens.shape
    k = k1 - 1
    mism = 0
    flagged = int(ref["flag_accept"].sum() + ref["flag_sample"].sum())
    for b in range(B):
        ra = int(ref["num_accepted"][b])
        ga = int(got_a[b])
        if ga != ra:
            lo = min(ga, ra)
            assert ref["flag_accept"][b, lo] == 1, (
                "request %d: accepted %d vs oracle %d with no flag at %d" % (b, ga, ra, lo))
            mism += 1
            continue
        assert (got_tokens[b, :ra] == ref["out_tokens"][b, :ra]).all(), "request %d: accepted drafts differ" % b
        assert (got_tokens[b, ra + 1:] == -1).all(), "request %d: padding" % b
        if got_tokens[b, ra] != ref["out_tokens"][b, ra]:
            assert ref["flag_sample"][b] == 1, (
                "request %d: token %d vs oracle %d at row %d, not flagged"
                % (b, got_tokens[b, ra], ref["out_tokens"][b, ra], ra))
            mism += 1
    return dict(mismatch=mism, flagged=flagged, positions=B * (k + 1))


def count_chain(got_tokens, got_a, ref):
    """Counts for the flag budget, without asserting: positions (B x (k+1)
    target rows), positions the oracle flags, requests whose GPU result differs
    from the oracle's (an accept decision or the drawn token), and differences
    not explained by the flag on the decision that made them.  Also the drafts
    tested and accepted (achieved acceptance rate)."""
    B, k1 = got_tokens.shape
    c = dict(positions=B * k1, flagged=int(ref["flag_accept"].sum() + ref["flag_sample"].sum()),
             differ=0, unflagged=0, tested=0, accepted=0)
    k = k1 - 1
    for b in range(B):
        ra, ga = int(ref["num_accepted"][b]), int(got_a[b])
        c["accepted"] += ra
        c["tested"] += ra + (1 if ra < k else 0)
        if ga != ra:
            c["differ"] += 1
            c["unflagged"] += int(not (0 <= min(ga, ra) < k and ref["flag_accept"][b, min(ga, ra)]))
            continue
        if (got_tokens[b, :ra] != ref["out_tokens"][b, :ra]).any() or (got_tokens[b, ra + 1:] != -1).any():
            c["differ"] += 1
            c["unflagged"] += 1
        elif got_tokens[b, ra] != ref["out_tokens"][b, ra]:
            c["differ"] += 1
            c["unflagged"] += int(not ref["flag_sample"][b])
    return c


def tree_divergence(parent, got, ref, b):
    """Sampled trees: where request b's GPU walk leaves the oracle's, and the
    oracle flag that would excuse it.  Returns None when the two agree, else
    (kind, index): ("accept", n) when the walks part below a node because the
    test of child n went the other way (n is the lower of the two children
    they moved to, or the one child either moved to: the first test on which
    they disagree), ("sample", b) when the walks are the same and only the
    drawn token differs, ("invalid", -1) when the GPU's walk is not a walk."""
    gp, rp = got["path"][b], ref["path"][b]
    gl, rl = int(got["length"][b]), int(ref["length"][b])
    if gl == rl and (gp == rp).all() and (got["tokens"][b] == ref["tokens"][b]).all():
        return None
    if gl < 1 or gl > gp.shape[0] or gp[0] != 0:
        return ("invalid", -1)
    i = 1
    while i < min(gl, rl) and gp[i] == rp[i]:
        i += 1
    node = int(rp[i - 1])
    rc = int(rp[i]) if i < rl else -1
    gc = int(gp[i]) if i < gl else -1
    if rc < 0 and gc < 0:
        same = (gp[:gl] == rp[:rl]).all() and (got["tokens"][b, :gl - 1] == ref["tokens"][b, :rl - 1]).all()
        return ("sample", b) if same else ("invalid", -1)
    for c in (rc, gc):
        if c >= 0 and (c >= len(parent) or int(parent[c]) != node):
            return ("invalid", -1)
    return ("accept", min(c for c in (rc, gc) if c >= 0))


def count_tree_sampled(parent, got, ref):
    """Flag-budget counts for a sampled-tree batch: positions (B x (N+1)),
    oracle-flagged positions, requests whose result differs, and differences
    the flag on the deciding test (or draw) does not excuse."""
    B, N1 = got["path"].shape[0], len(parent)
    c = dict(positions=B * N1, flagged=int(ref["flag_accept"].sum() + ref["flag_sample"].sum()),
             differ=0, unflagged=0)
    for b in range(B):
        d = tree_divergence(parent, got, ref, b)
        if d is None:
            continue
        c["differ"] += 1
        kind, n = d
        if kind == "accept":
            c["unflagged"] += int(not ref["flag_accept"][b, n - 1])
        elif kind == "sample":
            c["unflagged"] += int(not ref["flag_sample"][b])
        else:
            c["unflagged"] += 1
    return c
