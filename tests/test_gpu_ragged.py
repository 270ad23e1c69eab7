"""Ragged chains on the GPU (a different number of drafts per request, packed
by cu_num_draft_tokens offsets), against the oracle run request by request.

Greedy tokens and counts are bit-exact; sampled tokens are bit-exact except at
positions the oracle flags.  Every call goes through the C ABI via the binding.
"""
import numpy as np
import pytest

from speculative_decoding_verification_chain_gb300 import workloads as W

from helpers import compare_chain, cuda

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


def run_ragged(sv, x, dev, max_k=None, status=None):
    sampled = x.draft_probs is not None
    max_k = x.max_k if max_k is None else max_k
    ot, na = sv.verify_chain_ragged(
        cuda(x.logits, dev), cuda(x.draft_tokens, dev), cuda(x.cu, dev), max_k,
        cuda(x.temperature, dev) if sampled else None,
        cuda(x.u_accept, dev) if sampled else None,
        cuda(x.u_sample, dev) if sampled else None,
        cuda(x.draft_probs, dev) if sampled else None, status=status)
    return ot.cpu().numpy(), na.cpu().numpy()


def check_against_oracle(O, x, got_t, got_a):
    """Per request: the oracle on that request alone (B = 1, k = k_b)."""
    mism = flagged = 0
    for b, part in enumerate(x.parts):
        k = part.k
        ref = O.verify_chain(part.logits, part.dtype, part.draft_tokens, part.temperature, part.u_sample,
                             part.draft_probs, part.u_accept)
        if part.temperature[0] == 0:
            assert got_a[b] == ref["num_accepted"][0], b
            assert (got_t[b, :k + 1] == ref["out_tokens"][0]).all(), b
        else:
            r = compare_chain(got_t[b:b + 1, :k + 1], got_a[b:b + 1], ref)
            mism += r["mismatch"]
            flagged += r["flagged"]
        assert (got_t[b, k + 1:] == -1).all(), b
    return mism, flagged


@pytest.mark.parametrize("dtype", [W.BF16, W.FP32], ids=["bf16", "fp32"])
def test_ragged_greedy_bit_exact(sv, O, dev, dtype):
    x = W.chain_ragged(seed=901, B=24, max_k=6, V=20011, mode="greedy", dtype=dtype)
    got_t, got_a = run_ragged(sv, x, dev)
    check_against_oracle(O, x, got_t, got_a)


def test_ragged_sampled_matches_oracle_modulo_flags(sv, O, dev):
    x = W.chain_ragged(seed=902, B=20, max_k=5, V=30011, mode="sampled", temperature=0.8, lam=0.3)
    got_t, got_a = run_ragged(sv, x, dev)
    mism, flagged = check_against_oracle(O, x, got_t, got_a)
    assert mism <= flagged


def test_ragged_mixed_greedy_and_sampled(sv, O, dev):
    x = W.chain_ragged(seed=903, B=32, max_k=7, V=12007, mode="mixed")
    got_t, got_a = run_ragged(sv, x, dev)
    check_against_oracle(O, x, got_t, got_a)


def test_ragged_full_size_greedy(sv, O, dev):
    x = W.chain_ragged(seed=904, B=64, max_k=8, V=128256, mode="greedy")
    got_t, got_a = run_ragged(sv, x, dev)
    check_against_oracle(O, x, got_t, got_a)


def test_ragged_with_uniform_k_equals_padded_chain(sv, dev):
    """Every k_b = k: the ragged call and spec_verify_chain on the same rows agree."""
    x = W.chain_sampled(seed=905, B=16, k=4, V=9001, temperature=0.9, lam=0.3)
    B, k, V = x.B, x.k, x.V
    r = W.RaggedChainInputs(
        logits=x.logits.reshape(B * (k + 1), V), dtype=x.dtype,
        cu=np.arange(0, (B + 1) * k, k, dtype=np.int32), draft_tokens=x.draft_tokens.reshape(-1),
        temperature=x.temperature, u_sample=x.u_sample.reshape(-1), draft_probs=x.draft_probs.reshape(B * k, V),
        u_accept=x.u_accept.reshape(-1), slot_mapping=x.slot_mapping.reshape(-1), parts=[])
    got_t, got_a = run_ragged(sv, r, dev, max_k=k)
    pad_t, pad_a = sv.verify_chain(cuda(x.logits, dev), cuda(x.draft_tokens, dev), cuda(x.temperature, dev),
                                   cuda(x.u_accept, dev), cuda(x.u_sample, dev), cuda(x.draft_probs, dev))
    assert (got_a == pad_a.cpu().numpy()).all() and (got_t == pad_t.cpu().numpy()).all()


def test_ragged_all_requests_without_drafts(sv, O, dev):
    x = W.chain_ragged(seed=906, B=9, max_k=0, V=5003, mode="mixed")
    got_t, got_a = run_ragged(sv, x, dev, max_k=0)
    assert (got_a == 0).all()
    check_against_oracle(O, x, got_t, got_a)


def test_ragged_slot_fixup(sv, O, dev):
    x = W.chain_ragged(seed=907, B=16, max_k=5, V=4001, mode="greedy")
    got_t, got_a = run_ragged(sv, x, dev)
    import torch
    slots = cuda(x.slot_mapping, dev)
    sv.fixup_slots_ragged(slots, cuda(x.cu, dev), torch.from_numpy(got_a).to(dev))
    exp = x.slot_mapping.copy()
    for b in range(x.B):
        lo = int(x.cu[b]) + b
        kb = int(x.cu[b + 1] - x.cu[b])
        ref = O.fixup_slots(x.slot_mapping[lo:lo + kb + 1][None, :], num_accepted=got_a[b:b + 1])
        exp[lo:lo + kb + 1] = ref[0]
    assert (slots.cpu().numpy() == exp).all()


@pytest.mark.parametrize("mode", ["greedy", "mixed"])
def test_ragged_fused_slot_fixup(sv, O, dev, mode):
    """spec_verify_chain_ragged_fused: the verify's results and, in the same
    launch, the slot map the oracle's fix-up writes for those counts."""
    import torch
    x = W.chain_ragged(seed=908, B=24, max_k=6, V=4001, mode=mode, min_k=0)
    sampled = x.draft_probs is not None
    slots = cuda(x.slot_mapping, dev)
    ot, na = sv.verify_chain_ragged(
        cuda(x.logits, dev), cuda(x.draft_tokens, dev), cuda(x.cu, dev), x.max_k,
        cuda(x.temperature, dev) if sampled else None, cuda(x.u_accept, dev) if sampled else None,
        cuda(x.u_sample, dev) if sampled else None, cuda(x.draft_probs, dev) if sampled else None,
        slot_mapping=slots, padding_slot_id=-3)
    torch.cuda.synchronize(dev)
    got_t, got_a = ot.cpu().numpy(), na.cpu().numpy()
    ref_t, ref_a = run_ragged(sv, x, dev)
    assert (got_t == ref_t).all() and (got_a == ref_a).all()
    check_against_oracle(O, x, got_t, got_a)
    exp = x.slot_mapping.copy()
    for b in range(x.B):
        lo = int(x.cu[b]) + b
        kb = int(x.cu[b + 1] - x.cu[b])
        exp[lo:lo + kb + 1] = O.fixup_slots(x.slot_mapping[lo:lo + kb + 1][None, :], num_accepted=got_a[b:b + 1],
                                            pad=-3)[0]
    assert (slots.cpu().numpy() == exp).all()


def test_ragged_offsets_out_of_order_are_flagged_not_faulted(sv, dev):
    """Offsets that break the rules are clamped inside the packed inputs and
    reported in the status word; the call completes."""
    import torch
    x = W.chain_ragged(seed=908, B=3, max_k=5, V=3001, mode="greedy", min_k=2)
    bad = x.cu.copy()
    bad[1], bad[2] = bad[2], bad[1]   # not non-decreasing
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ot, na = sv.verify_chain_ragged(cuda(x.logits, dev), cuda(x.draft_tokens, dev), cuda(bad, dev), x.max_k,
                                    status=st)
    torch.cuda.synchronize(dev)
    assert int(st.item()) & sv.STATUS_BAD_OFFSETS
