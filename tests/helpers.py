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
