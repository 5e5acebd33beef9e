"""Block-sparse masks on the GPU (fa_fwd_masked / fa_bwd_masked through the C
ABI) against the oracle with the same mask in dense form."""
import numpy as np
import pytest
import torch

import oracle
from flash_attention_gqa_gb300 import binding, inputs
from _parity import check_grad, check_lse, check_o, to_np

pytestmark = pytest.mark.gpu


def block_structured_mask(heads, T, S, seed):
    """Each 128 x 128 block empty, full, or random at a random density."""
    rng = np.random.default_rng(seed)
    m = np.zeros((heads, T, S), dtype=bool)
    for h in range(heads):
        for t0 in range(0, T, 128):
            for s0 in range(0, S, 128):
                kind = rng.integers(0, 3)
                blk = m[h, t0:t0 + 128, s0:s0 + 128]
                if kind == 1:
                    blk[:] = True
                elif kind == 2:
                    blk[:] = rng.random(blk.shape) < rng.uniform(0.2, 0.9)
    return m


def run_masked(B, K, G, T, S, H, heads, causal=False, segs=False, seed=0, backward=True):
    seg = inputs.document_segment_ids(B, T, seed=seed, lo=60, hi=250) if (segs and T == S) else None
    x = inputs.make_tensors(B, K, G, T, S, H, seed=seed, backward=backward, seg_q=seg, seg_kv=seg)
    dense = block_structured_mask(heads, T, S, seed)
    dev = torch.device("cuda")
    meta = binding.block_mask_from_dense(dense, device=dev)
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    sq = None if x.seg_q is None else x.seg_q.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, K, G, T), dtype=torch.float32, device=dev)
    binding.fa_fwd_masked(q, k, v, sq, sq, causal, meta, o, lse)
    assert binding.fa_check_status() == binding.FA_OK
    kw = dict(causal=causal, seg_q=x.seg_q, seg_kv=x.seg_kv, mask=dense)
    o_ref, l_ref = oracle.attention_forward(x.q, x.k, x.v, **kw)
    check_o(to_np(o), o_ref)
    check_lse(lse.cpu().numpy().astype(np.float64), l_ref)
    if not backward:
        return
    dO = x.dO.to(dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(max(256, binding.fa_bwd_workspace_size(B, K, G, T, S, H)), dtype=torch.uint8,
                     device=dev)
    binding.fa_bwd_masked(q, k, v, o, lse, dO, sq, sq, causal, meta, dq, dk, dv, ws)
    assert binding.fa_check_status() == binding.FA_OK
    g_ref = oracle.attention_backward(x.q, x.k, x.v, x.dO, **kw)
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), g_ref):
        check_grad(to_np(got), want, name)


@pytest.mark.parametrize("per_head", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,G", [(128, 4), (256, 8)])
def test_block_sparse(per_head, causal, H, G):
    K = 2
    run_masked(1, K, G, 512, 512, H, K * G if per_head else 1, causal=causal, seed=H + G)


def test_block_sparse_with_segments_and_ragged():
    run_masked(2, 2, 4, 300, 300, 128, 8, causal=True, segs=True, seed=3)
    run_masked(1, 2, 8, 200, 333, 256, 1, causal=False, seed=4)


def test_block_sparse_forward_h64_and_rectangular_causal():
    run_masked(1, 1, 4, 256, 384, 64, 4, causal=True, seed=5, backward=False)


@pytest.mark.parametrize("rows", [64, 128])
def test_block_sparse_h128_both_kv_tile_sizes(rows):
    assert binding.fa_set_bwd_kv_rows(rows) == binding.FA_OK
    try:
        run_masked(1, 2, 4, 512, 512, 128, 8, causal=True, seed=rows)
        run_masked(2, 2, 4, 300, 300, 128, 8, causal=True, segs=True, seed=rows + 1)
    finally:
        binding.fa_set_bwd_kv_rows(0)


@pytest.mark.parametrize("mode", [1, 2])
def test_block_sparse_forward_both_grids(mode):
    assert binding.fa_set_fwd_schedule(mode) == binding.FA_OK
    try:
        run_masked(2, 4, 4, 1024, 1024, 128, 16, causal=True, seed=mode, backward=False)
        run_masked(1, 1, 4, 256, 384, 64, 4, causal=True, seed=mode + 2, backward=False)
    finally:
        binding.fa_set_fwd_schedule(0)
