"""Backward parity: fa_fwd + fa_bwd (through the C ABI) against the fp64
oracle's analytic gradients on the same seeded bf16 inputs.  GPU only."""
import numpy as np
import pytest
import torch

import oracle
from flash_attention_gqa_gb300 import binding, inputs
from _parity import check_grad, check_lse, check_o, to_np

pytestmark = pytest.mark.gpu


def run_case(B, K, G, T, S, H, causal=False, seg_q=None, seg_kv=None, seed=0):
    x = inputs.make_tensors(B, K, G, T, S, H, seed=seed, backward=True, seg_q=seg_q,
                            seg_kv=seg_kv)
    dev = torch.device("cuda")
    q, k, v, dO = (t.to(dev) for t in (x.q, x.k, x.v, x.dO))
    sq = None if x.seg_q is None else x.seg_q.to(dev)
    skv = None if x.seg_kv is None else x.seg_kv.to(dev)
    o, lse = binding.attention_forward(q, k, v, causal=causal, seg_q=sq, seg_kv=skv)
    dq, dk, dv = binding.attention_backward(q, k, v, o, lse, dO, causal=causal, seg_q=sq,
                                            seg_kv=skv)
    assert binding.fa_check_status() == binding.FA_OK
    kw = dict(causal=causal, seg_q=x.seg_q, seg_kv=x.seg_kv)
    o_ref, l_ref = oracle.attention_forward(x.q, x.k, x.v, **kw)
    g_ref = oracle.attention_backward(x.q, x.k, x.v, x.dO, **kw)
    check_o(to_np(o), o_ref)
    check_lse(lse.cpu().numpy().astype(np.float64), l_ref)
    errs = {}
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), g_ref):
        errs[name] = check_grad(to_np(g), r, name)
    return (dq, dk, dv), g_ref, errs


@pytest.mark.parametrize("H", [64, 128, 256])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_shapes(H, G, causal):
    run_case(1, 2, G, 384, 384, H, causal=causal, seed=100 + H + G)


@pytest.mark.parametrize("G", [16, 64])
def test_wide_groups(G):
    run_case(1, 1, G, 256, 256, 128, causal=True, seed=G)


def test_rectangular_noncausal():
    run_case(2, 1, 4, 128, 640, 128, causal=False, seed=13)
    run_case(1, 2, 2, 512, 128, 256, causal=False, seed=14)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H", [128, 256])
def test_random_nonmonotone_segments(causal, H):
    B, T = 2, 512
    seg = inputs.random_segment_ids(B, T, 3, seed=17)
    run_case(B, 2, 4, T, T, H, causal=causal, seg_q=seg, seg_kv=seg, seed=15)


def test_document_segments_causal():
    B, T = 3, 1024
    seg = inputs.document_segment_ids(B, T, seed=0, lo=50, hi=400)
    run_case(B, 2, 4, T, T, 128, causal=True, seg_q=seg, seg_kv=seg, seed=16)


def test_fully_masked_rows_get_zero_gradient():
    B, T = 1, 256
    seg_q = np.zeros((B, T), dtype=np.int32)
    seg_kv = np.zeros((B, T), dtype=np.int32)
    seg_q[0, 100:140] = 7
    (dq, _, _), _, _ = run_case(B, 1, 4, T, T, 128, causal=False, seg_q=seg_q,
                                seg_kv=seg_kv, seed=18)
    assert torch.all(dq[0, 0, :, 100:140] == 0)


@pytest.mark.parametrize("T,S", [(300, 300), (77, 77), (1000, 1000)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,G", [(128, 4), (256, 8)])
def test_ragged_lengths(T, S, causal, H, G):
    run_case(1, 2, G, T, S, H, causal=causal, seed=T + H)


@pytest.mark.parametrize("T,S", [(100, 300), (300, 100), (1, 500), (5, 3)])
@pytest.mark.parametrize("H", [128, 256])
def test_rectangular_causal(T, S, H):
    run_case(2, 1, 4, T, S, H, causal=True, seed=T + S)


def test_ragged_segments():
    T = 333
    seg = inputs.document_segment_ids(2, T, seed=5, lo=40, hi=200)
    run_case(2, 2, 4, T, T, 128, causal=True, seg_q=seg, seg_kv=seg, seed=7)
    seg_q = inputs.random_segment_ids(1, T, 3, seed=3)
    seg_kv = inputs.random_segment_ids(1, T + 5, 3, seed=4)
    run_case(1, 1, 8, T, T + 5, 256, causal=False, seg_q=seg_q, seg_kv=seg_kv, seed=8)


@pytest.mark.parametrize("H", [128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_odd_row_count_with_segments(H, causal):
    # B*K*G*T = 77 rows: the segment-range table follows an odd number of fp32
    # D rows in the workspace, so its 8-byte pairs need their own alignment
    seg = inputs.document_segment_ids(1, 77, seed=9, lo=5, hi=30)
    run_case(1, 1, 1, 77, 77, H, causal=causal, seg_q=seg, seg_kv=seg, seed=41 + H)
    seg_q = inputs.random_segment_ids(1, 77, 3, seed=10)
    seg_kv = inputs.random_segment_ids(1, 91, 3, seed=11)
    run_case(1, 1, 1, 77, 91, H, causal=False, seg_q=seg_q, seg_kv=seg_kv, seed=43 + H)


def test_causal_workload_h128_t1024_full():
    w = inputs.WORKLOADS["gqa_causal_h128_t1024"]
    run_case(w.B, w.K, w.G, w.T, w.S, w.H, causal=True, seed=w.seed)


def test_backward_is_deterministic():
    x = inputs.make_tensors(1, 2, 8, 512, 512, 256, seed=19, backward=True)
    dev = torch.device("cuda")
    q, k, v, dO = (t.to(dev) for t in (x.q, x.k, x.v, x.dO))
    o, lse = binding.attention_forward(q, k, v, causal=True)
    a = binding.attention_backward(q, k, v, o, lse, dO, causal=True)
    b = binding.attention_backward(q, k, v, o, lse, dO, causal=True)
    for x1, x2 in zip(a, b):
        assert torch.equal(x1, x2)


# H = 64 runs the H = 128 kernels over zero-filled upper head dims: ragged
# sizes, segment ids, both KV tile sizes and the dK/dV split must all hold.
@pytest.mark.parametrize("T,S,causal", [(77, 77, True), (300, 300, False), (100, 300, True),
                                        (1000, 1000, True)])
def test_h64_ragged_and_rectangular(T, S, causal):
    run_case(1, 2, 4, T, S, 64, causal=causal, seed=T + S + 64)


def test_h64_segments():
    seg = inputs.document_segment_ids(2, 640, seed=12, lo=40, hi=300)
    run_case(2, 2, 4, 640, 640, 64, causal=True, seg_q=seg, seg_kv=seg, seed=64)
    seg = inputs.random_segment_ids(1, 333, 3, seed=13)
    run_case(1, 1, 8, 333, 333, 64, causal=False, seg_q=seg, seg_kv=seg, seed=65)


@pytest.mark.parametrize("rows", [64, 128])
@pytest.mark.parametrize("splits", [1, 3])
def test_h64_kv_tile_sizes_and_splits(rows, splits):
    assert binding.fa_set_bwd_kv_rows(rows) == binding.FA_OK
    assert binding.fa_set_bwd_q_splits(splits) == binding.FA_OK
    try:
        run_case(1, 2, 4, 640, 640, 64, causal=True, seed=rows + splits)
    finally:
        binding.fa_set_bwd_kv_rows(0)
        binding.fa_set_bwd_q_splits(0)


# ----------------------------------------------- both KV tile sizes at H = 128

@pytest.fixture
def forced_kv_rows(request):
    assert binding.fa_set_bwd_kv_rows(request.param) == binding.FA_OK
    yield request.param
    binding.fa_set_bwd_kv_rows(0)


def _doc_segs(B, T, seed):
    return inputs.document_segment_ids(B, T, seed=seed, lo=40, hi=300)


KV_TILE_CASES = {
    "causal": dict(B=1, K=2, G=4, T=384, S=384, causal=True),
    "full_g8_ragged": dict(B=1, K=2, G=8, T=1000, S=1000, causal=False),
    "causal_ragged": dict(B=2, K=1, G=4, T=300, S=300, causal=True),
    "rect_causal": dict(B=2, K=2, G=4, T=100, S=300, causal=True),
    "doc_segments": dict(B=2, K=2, G=4, T=640, S=640, causal=True, segs=True),
}


@pytest.mark.parametrize("forced_kv_rows", [64, 128], indirect=True)
@pytest.mark.parametrize("name", sorted(KV_TILE_CASES))
def test_h128_both_kv_tile_sizes(forced_kv_rows, name):
    c = dict(KV_TILE_CASES[name])
    seg = _doc_segs(c["B"], c["T"], 3) if c.pop("segs", False) else None
    run_case(c["B"], c["K"], c["G"], c["T"], c["S"], 128, causal=c["causal"], seg_q=seg,
             seg_kv=seg, seed=len(name) + forced_kv_rows)


# --------------------------------- Q-range split of dK/dV grids under the GPU

@pytest.fixture
def forced_q_splits(request):
    assert binding.fa_set_bwd_q_splits(request.param) == binding.FA_OK
    yield request.param
    binding.fa_set_bwd_q_splits(0)


# Small grids, so the split applies; T > S and T < S give splits with no tile.
Q_SPLIT_CASES = {
    "causal_h128": dict(B=1, K=2, G=4, T=640, S=640, H=128, causal=True),
    "causal_h256": dict(B=1, K=1, G=8, T=512, S=512, H=256, causal=True),
    "full_ragged_h256": dict(B=1, K=1, G=4, T=333, S=300, H=256, causal=False),
    "rect_causal_t_lt_s": dict(B=1, K=2, G=4, T=100, S=700, H=128, causal=True),
    "rect_causal_t_gt_s": dict(B=1, K=1, G=8, T=700, S=200, H=256, causal=True),
    "doc_segments": dict(B=2, K=1, G=4, T=640, S=640, H=128, causal=True, segs=True),
}


@pytest.mark.parametrize("forced_q_splits", [1, 2, 3, 4], indirect=True)
@pytest.mark.parametrize("name", sorted(Q_SPLIT_CASES))
def test_dkdv_q_splits(forced_q_splits, name):
    c = dict(Q_SPLIT_CASES[name])
    seg = _doc_segs(c["B"], c["T"], 5) if c.pop("segs", False) else None
    run_case(c["B"], c["K"], c["G"], c["T"], c["S"], c["H"], causal=c["causal"], seg_q=seg,
             seg_kv=seg, seed=len(name) + 10 * forced_q_splits)


def _bwd_inputs(B, K, G, T, H, seed):
    x = inputs.make_tensors(B, K, G, T, T, H, seed=seed, backward=True)
    dev = torch.device("cuda")
    q, k, v, dO = (t.to(dev) for t in (x.q, x.k, x.v, x.dO))
    o, lse = binding.attention_forward(q, k, v, causal=True)
    return q, k, v, o, lse, dO


@pytest.mark.parametrize("H", [128, 256])
def test_split_backward_is_repeatable_and_matches_unsplit(H):
    q, k, v, o, lse, dO = _bwd_inputs(1, 2, 4, 1024, H, seed=23)
    split = [binding.attention_backward(q, k, v, o, lse, dO, causal=True) for _ in range(2)]
    for x1, x2 in zip(*split):
        assert torch.equal(x1, x2)       # the partials are added in a fixed order
    assert binding.fa_set_bwd_q_splits(1) == binding.FA_OK
    try:
        whole = binding.attention_backward(q, k, v, o, lse, dO, causal=True)
    finally:
        binding.fa_set_bwd_q_splits(0)
    assert torch.equal(split[0][0], whole[0])    # dQ does not take part in the split
    for name, a, b in zip(("dk", "dv"), split[0][1:], whole[1:]):
        a, b = to_np(a), to_np(b)
        # only the fp32 summation order differs: at most about one bf16 unit
        assert np.linalg.norm(a - b) <= 2.0 ** -8 * np.linalg.norm(b), name


def test_backward_runs_unsplit_in_a_base_size_workspace():
    B, K, G, T, H = 1, 2, 4, 640, 128
    q, k, v, o, lse, dO = _bwd_inputs(B, K, G, T, H, seed=29)
    up = lambda n: (n + 255) // 256 * 256
    # D rows, the per-tile segment ranges, one segment-run byte per 64-key tile
    base = up(B * K * G * T * 4) + up(B * (T // (128 // G) + -(-T // 64)) * 8) + up(B * -(-T // 64))
    assert binding.fa_bwd_workspace_size(B, K, G, T, T, H) > base   # the split part exists here
    dev = q.device
    outs = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    binding.fa_bwd(q, k, v, o, lse, dO, None, None, True, *outs,
                   torch.empty(base, device=dev, dtype=torch.uint8))
    assert binding.fa_check_status() == binding.FA_OK
    assert binding.fa_set_bwd_q_splits(1) == binding.FA_OK
    try:
        whole = binding.attention_backward(q, k, v, o, lse, dO, causal=True)
    finally:
        binding.fa_set_bwd_q_splits(0)
    for a, b in zip(outs, whole):
        assert torch.equal(a, b)         # no split part: the one-CTA-per-KV-tile result
