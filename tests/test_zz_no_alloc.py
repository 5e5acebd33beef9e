"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory
(its scratch is a fixed array inside the library).  It must give what fa_bwd
gives, on consecutive calls that reuse the shared scratch, and refuse sizes
whose scratch would not fit.  Collected last on purpose (file name)."""
import ctypes

import numpy as np
import pytest
import torch

from flash_attention_gqa_gb300 import binding, inputs
from _parity import GRAD_REL_FRO, rel_fro, to_np

pytestmark = pytest.mark.gpu


def _case(seed, B, K, G, T, H, causal, segments):
    dev = torch.device("cuda")
    seg = inputs.document_segment_ids(B, T, seed=seed, lo=64, hi=300) if segments else None
    x = inputs.make_tensors(B, K, G, T, T, H, seed=seed, backward=True, seg_q=seg, seg_kv=seg)
    q, k, v, dO = (t.to(dev) for t in (x.q, x.k, x.v, x.dO))
    sq = None if x.seg_q is None else x.seg_q.to(dev)
    o, lse = binding.attention_forward(q, k, v, causal=causal, seg_q=sq, seg_kv=sq)
    ref = binding.attention_backward(q, k, v, o, lse, dO, causal=causal, seg_q=sq, seg_kv=sq)
    return q, k, v, o, lse, dO, sq, ref


def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row():
    cases = [(_case(31, 1, 2, 8, 512, 256, True, False), True),
             (_case(32, 2, 2, 4, 1024, 128, True, True), True)]
    for (q, k, v, o, lse, dO, sq, ref), causal in cases:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        binding.fa_bwd_noalloc(q, k, v, o, lse, dO, sq, sq, causal, dq, dk, dv)
        torch.cuda.synchronize()
        assert binding.fa_check_status() == binding.FA_OK
        for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            g, w = to_np(got), to_np(want)
            assert np.all(np.isfinite(g)), name
            assert rel_fro(g, w) <= GRAD_REL_FRO, name


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = binding.load()
    P = ctypes.c_void_p
    # 1 x 1 x 128 heads x 32768 rows needs 16 MiB of fp32 D rows: over the fixed 8 MiB
    rc = lib.fa_bwd_noalloc(P(16), P(16), P(16), P(16), P(16), P(16), None, None, 1,
                            P(16), P(16), P(16), 1, 1, 128, 32768, 32768, 128, None)
    assert rc == binding.FA_ERR_UNSUPPORTED
