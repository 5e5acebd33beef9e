"""Forward parity: fa_fwd (through the C ABI) against the fp64 oracle on the
same seeded bf16 inputs.  GPU only."""
import numpy as np
import pytest
import torch

import oracle
from flash_attention_gqa_gb300 import binding, inputs
from _parity import check_lse, check_o, to_np

pytestmark = pytest.mark.gpu


def run_case(B, K, G, T, S, H, causal=False, seg_q=None, seg_kv=None, seed=0, heads=None):
    x = inputs.make_tensors(B, K, G, T, S, H, seed=seed, backward=False, seg_q=seg_q,
                            seg_kv=seg_kv)
    dev = torch.device("cuda")
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    sq = None if x.seg_q is None else x.seg_q.to(dev)
    skv = None if x.seg_kv is None else x.seg_kv.to(dev)
    o, lse = binding.attention_forward(q, k, v, causal=causal, seg_q=sq, seg_kv=skv)
    assert binding.fa_check_status() == binding.FA_OK
    o_ref, l_ref = oracle.attention_forward(x.q, x.k, x.v, causal=causal, seg_q=x.seg_q,
                                            seg_kv=x.seg_kv, heads=heads)
    og, lg = to_np(o), lse.cpu().numpy().astype(np.float64)
    if heads is not None:
        sel = tuple(zip(*heads))
        og, o_ref, lg, l_ref = og[sel], o_ref[sel], lg[sel], l_ref[sel]
    check_o(og, o_ref)
    check_lse(lg, l_ref)
    return og, o_ref


def test_small_workload_h64_t128():
    w = inputs.WORKLOADS["gqa_h64_t128_fwd"]
    run_case(w.B, w.K, w.G, w.T, w.S, w.H, causal=w.causal, seed=w.seed)


@pytest.mark.parametrize("H", [64, 128, 256])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_shapes(H, G, causal):
    run_case(1, 2, G, 384, 384, H, causal=causal, seed=H + G)


@pytest.mark.parametrize("G", [16, 32, 128])
def test_wide_groups(G):
    run_case(1, 1, G, 256, 256, 128, causal=True, seed=G)


def test_rectangular_noncausal():
    run_case(2, 1, 4, 128, 640, 128, causal=False, seed=3)
    run_case(1, 2, 2, 512, 128, 64, causal=False, seed=4)


@pytest.mark.parametrize("causal", [False, True])
def test_random_nonmonotone_segments(causal):
    B, T = 2, 512
    seg = inputs.random_segment_ids(B, T, 3, seed=7)
    run_case(B, 2, 4, T, T, 128, causal=causal, seg_q=seg, seg_kv=seg, seed=5)


def test_document_segments_causal():
    B, T = 3, 1024
    seg = inputs.document_segment_ids(B, T, seed=0, lo=50, hi=400)
    run_case(B, 2, 4, T, T, 128, causal=True, seg_q=seg, seg_kv=seg, seed=6)


def test_fully_masked_rows_give_zero():
    B, T = 1, 256
    seg_q = np.zeros((B, T), dtype=np.int32)
    seg_kv = np.zeros((B, T), dtype=np.int32)
    seg_q[0, 100:140] = 7      # id 7 never appears among the keys
    og, _ = run_case(B, 1, 4, T, T, 64, causal=False, seg_q=seg_q, seg_kv=seg_kv, seed=8)
    assert np.all(og[0, 0, :, 100:140] == 0.0)


def test_segments_with_distinct_key_ids():
    # keys and queries carry different id sequences; whole tiles are empty
    B, T = 2, 512
    seg_q = np.repeat(np.arange(4, dtype=np.int32), 128)[None].repeat(B, 0)
    seg_kv = np.repeat(np.array([3, 2, 1, 0], dtype=np.int32), 128)[None].repeat(B, 0)
    run_case(B, 1, 8, T, T, 256, causal=False, seg_q=seg_q, seg_kv=seg_kv, seed=9)


def test_large_logits_are_stable():
    # scale q up so logits span tens of units: exercises the running-max rescale
    B, K, G, T, H = 1, 1, 4, 512, 128
    x = inputs.make_tensors(B, K, G, T, T, H, seed=11, backward=False, scale=1.0)
    dev = torch.device("cuda")
    o, lse = binding.attention_forward(x.q.to(dev), x.k.to(dev), x.v.to(dev), causal=True)
    o_ref, l_ref = oracle.attention_forward(x.q, x.k, x.v, causal=True)
    check_o(to_np(o), o_ref)
    check_lse(lse.cpu().numpy().astype(np.float64), l_ref)


@pytest.mark.parametrize("T,S", [(300, 300), (200, 200), (1000, 1000), (77, 77)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,G", [(64, 4), (128, 8), (256, 1)])
def test_ragged_lengths(T, S, causal, H, G):
    run_case(1, 2, G, T, S, H, causal=causal, seed=T + H + G)


@pytest.mark.parametrize("T,S", [(100, 300), (300, 100), (128, 1000), (1, 1000), (1, 1), (5, 3)])
@pytest.mark.parametrize("causal", [False, True])
def test_rectangular_and_decode_shapes(T, S, causal):
    # causal with T != S keeps s <= t + (S - T); T = 1 is a decode step
    run_case(2, 2, 8, T, S, 128, causal=causal, seed=T * 7 + S)


@pytest.mark.parametrize("T", [333, 1001])
def test_ragged_segments(T):
    # T not a multiple of 4: segment-id rows are not 16-byte aligned
    seg = inputs.document_segment_ids(2, T, seed=T, lo=40, hi=200)
    run_case(2, 2, 4, T, T, 128, causal=True, seg_q=seg, seg_kv=seg, seed=T)
    seg_q = inputs.random_segment_ids(1, T, 3, seed=1)
    seg_kv = inputs.random_segment_ids(1, T + 5, 3, seed=2)
    run_case(1, 1, 8, T, T + 5, 256, causal=False, seg_q=seg_q, seg_kv=seg_kv, seed=T + 1)


def test_causal_workload_h128_t1024_full():
    w = inputs.WORKLOADS["gqa_causal_h128_t1024"]
    run_case(w.B, w.K, w.G, w.T, w.S, w.H, causal=True, seed=w.seed)


def test_empty_inputs():
    dev = torch.device("cuda")
    # no keys: o = 0, lse = -inf
    q = torch.randn(1, 1, 4, 128, 64, device=dev).to(torch.bfloat16)
    k = torch.empty(1, 1, 0, 64, device=dev, dtype=torch.bfloat16)
    o = torch.full_like(q, 3.0)
    lse = torch.zeros(1, 1, 4, 128, device=dev)
    binding.fa_fwd(q, k, k, None, None, False, o, lse)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    # no queries: nothing to do
    q0 = torch.empty(1, 1, 4, 0, 64, device=dev, dtype=torch.bfloat16)
    k1 = torch.randn(1, 1, 128, 64, device=dev).to(torch.bfloat16)
    binding.fa_fwd(q0, k1, k1, None, None, False, torch.empty_like(q0),
                   torch.empty(1, 1, 4, 0, device=dev))
    assert binding.fa_check_status() == binding.FA_OK


def test_repeatable():
    x = inputs.make_tensors(1, 2, 4, 512, 512, 128, seed=12, backward=False)
    dev = torch.device("cuda")
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    o1, l1 = binding.attention_forward(q, k, v, causal=True)
    o2, l2 = binding.attention_forward(q, k, v, causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ------------------------------------------------------------- split-KV

def run_split(B, K, G, T, S, H, n_splits, causal=False, seg_q=None, seg_kv=None, seed=0):
    x = inputs.make_tensors(B, K, G, T, S, H, seed=seed, backward=False, seg_q=seg_q,
                            seg_kv=seg_kv)
    dev = torch.device("cuda")
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    sq = None if x.seg_q is None else x.seg_q.to(dev)
    skv = None if x.seg_kv is None else x.seg_kv.to(dev)
    o, lse = binding.attention_forward_splitkv(q, k, v, causal=causal, seg_q=sq, seg_kv=skv,
                                               n_splits=n_splits)
    assert binding.fa_check_status() == binding.FA_OK
    o_ref, l_ref = oracle.attention_forward(x.q, x.k, x.v, causal=causal, seg_q=x.seg_q,
                                            seg_kv=x.seg_kv)
    check_o(to_np(o), o_ref)
    check_lse(lse.cpu().numpy().astype(np.float64), l_ref)


@pytest.mark.parametrize("H", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n_splits", [2, 7, 40])
def test_splitkv_decode(H, causal, n_splits):
    run_split(2, 2, 8, 1, 3000, H, n_splits, causal=causal, seed=H + n_splits)


@pytest.mark.parametrize("T,S", [(16, 4096), (100, 1000), (300, 300)])
def test_splitkv_small_t(T, S):
    run_split(1, 2, 4, T, S, 128, 5, causal=True, seed=T)


def test_splitkv_segments_and_more_splits_than_tiles():
    T = 200
    seg = inputs.document_segment_ids(2, T, seed=2, lo=20, hi=90)
    run_split(2, 1, 4, T, T, 128, 3, causal=True, seg_q=seg, seg_kv=seg, seed=4)
    run_split(1, 1, 8, 1, 300, 128, 9, causal=False, seed=5)   # 9 splits, 3 kv tiles


def test_splitkv_default_splits():
    n = binding.fa_fwd_splitkv_default_splits(1, 8, 8, 1, 32768, 128)
    assert 1 <= n <= 64
    assert binding.fa_fwd_splitkv_default_splits(1, 2, 8, 8192, 8192, 256) == 1
    run_split(1, 8, 8, 1, 8192, 128, None, causal=True, seed=6)


# ------------------------------------- both forward grids (H <= 128 choices)

@pytest.fixture
def fwd_schedule(request):
    assert binding.fa_set_fwd_schedule(request.param) == binding.FA_OK
    yield request.param
    binding.fa_set_fwd_schedule(0)


def _distinct_key_ids(B, T):
    # query ids 0..3 by 128-position block, key ids reversed: whole Q tiles see no key
    seg_q = np.repeat(np.arange(4, dtype=np.int32), T // 4)[None].repeat(B, 0)
    seg_kv = np.repeat(np.array([3, 2, 1, 0], dtype=np.int32), T // 4)[None].repeat(B, 0)
    seg_q[:, : T // 8] = 7  # ids no key carries
    return seg_q, seg_kv


GRID_CASES = {
    "h64_causal": dict(B=1, K=2, G=4, T=384, S=384, H=64, causal=True),
    "h128_ragged_full": dict(B=1, K=2, G=8, T=1000, S=1000, H=128, causal=False),
    "h128_rect_causal": dict(B=2, K=2, G=4, T=100, S=300, H=128, causal=True),
    "h128_decode": dict(B=2, K=2, G=8, T=1, S=1000, H=128, causal=True),
    "h128_many_items": dict(B=2, K=8, G=4, T=2048, S=2048, H=128, causal=True),
    "h128_docs_many_items": dict(B=4, K=8, G=4, T=1024, S=1024, H=128, causal=True, segs="docs"),
    "h128_empty_q_tiles": dict(B=2, K=4, G=4, T=512, S=512, H=128, causal=False, segs="distinct"),
}


@pytest.mark.parametrize("fwd_schedule", [1, 2], indirect=True)
@pytest.mark.parametrize("name", sorted(GRID_CASES))
def test_both_forward_grids(fwd_schedule, name):
    c = dict(GRID_CASES[name])
    kind = c.pop("segs", None)
    seg_q = seg_kv = None
    if kind == "docs":
        seg_q = seg_kv = inputs.document_segment_ids(c["B"], c["T"], seed=5, lo=40, hi=300)
    elif kind == "distinct":
        seg_q, seg_kv = _distinct_key_ids(c["B"], c["T"])
    run_case(c["B"], c["K"], c["G"], c["T"], c["S"], c["H"], causal=c["causal"], seg_q=seg_q,
             seg_kv=seg_kv, seed=len(name))
