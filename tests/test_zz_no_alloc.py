"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory
(a plugin inside a host application that owns every device allocation, or a
runtime that forbids allocation after start-up).  Its scratch is a fixed array
inside the library, shared by every call.

It runs the same kernels as fa_bwd with the dK/dV Q-range split off, so with
that split forced off in fa_bwd too the two must agree bit for bit, on two
calls in a row that reuse the shared scratch; both are also held to the oracle
tolerances.  The odd-row case (G = 1, T = S = 77, segment ids) puts the
segment-range table after an odd number of fp32 D rows.  Collected last on
purpose (file name), so a run that stops at the first failure has already run
every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from flash_attention_gqa_gb300 import binding, inputs
from _parity import check_grad, to_np

pytestmark = pytest.mark.gpu

CASES = [
    # seed, B, K, G, T, H, causal, segments (lo, hi) or None
    (31, 1, 2, 8, 512, 256, True, None),
    (32, 2, 2, 4, 1024, 128, True, (64, 300)),
    (33, 1, 1, 1, 77, 128, True, (5, 30)),
    (34, 1, 1, 1, 77, 256, False, (5, 30)),
]


def _case(seed, B, K, G, T, H, causal, segments):
    dev = torch.device("cuda")
    seg = None
    if segments is not None:
        seg = inputs.document_segment_ids(B, T, seed=seed, lo=segments[0], hi=segments[1])
    x = inputs.make_tensors(B, K, G, T, T, H, seed=seed, backward=True, seg_q=seg, seg_kv=seg)
    q, k, v, dO = (t.to(dev) for t in (x.q, x.k, x.v, x.dO))
    sq = None if x.seg_q is None else x.seg_q.to(dev)
    o, lse = binding.attention_forward(q, k, v, causal=causal, seg_q=sq, seg_kv=sq)
    assert binding.fa_set_bwd_q_splits(1) == binding.FA_OK
    try:
        ref = binding.attention_backward(q, k, v, o, lse, dO, causal=causal, seg_q=sq, seg_kv=sq)
    finally:
        binding.fa_set_bwd_q_splits(0)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    want = oracle.attention_backward(x.q, x.k, x.v, x.dO, causal=causal, seg_q=x.seg_q,
                                     seg_kv=x.seg_kv)
    return (q, k, v, o, lse, dO, sq), ref, want


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"G{c[3]}_T{c[4]}_H{c[5]}")
def test_noalloc_matches_fa_bwd_bitwise_on_two_calls_in_a_row(case):
    seed, B, K, G, T, H, causal, segments = case
    (q, k, v, o, lse, dO, sq), ref, want = _case(seed, B, K, G, T, H, causal, segments)
    for call in range(2):
        # poison the outputs so a gradient the call failed to write cannot pass
        dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
        binding.fa_bwd_noalloc(q, k, v, o, lse, dO, sq, sq, causal, dq, dk, dv)
        torch.cuda.synchronize()
        assert binding.fa_check_status() == binding.FA_OK
        for name, got, r, w in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, want):
            assert torch.equal(got, r), f"{name} differs from fa_bwd (call {call})"
            check_grad(to_np(got), w, f"{name} vs oracle (call {call})")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = binding.load()
    P = ctypes.c_void_p
    # 1 x 1 x 128 heads x 32768 rows needs 16 MiB of fp32 D rows: over the fixed 8 MiB
    rc = lib.fa_bwd_noalloc(P(16), P(16), P(16), P(16), P(16), P(16), None, None, 1,
                            P(16), P(16), P(16), 1, 1, 128, 32768, 32768, 128, None)
    assert rc == binding.FA_ERR_UNSUPPORTED
