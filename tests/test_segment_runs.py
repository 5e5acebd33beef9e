"""Parity of the segment-id masks on layouts built to reach every branch of the
per-tile run byte (the classifiers record, per KV tile, where its segment id
changes when it changes at most once; such tiles mask one contiguous key range
per query row, others compare ids key by key):

- ids changing on the first, second, last and second-to-last key of a tile and
  on tile edges (one run, two runs with the change anywhere);
- three or more runs in one tile (the key-by-key path);
- key ids that no query carries next to ones that some do (a row matching
  neither run of a two-run tile);
- a ragged last tile (S not a multiple of the tile) with two runs.

fa_fwd + fa_bwd through the C ABI against the fp64 oracle, causal and not, at
H = 128 (both backward KV tile sizes) and H = 256.  GPU only."""
import numpy as np
import pytest
import torch

import oracle
from flash_attention_gqa_gb300 import binding, inputs
from _parity import check_grad, check_lse, check_o, to_np

pytestmark = pytest.mark.gpu

T = 400  # three full 128-key tiles and a ragged one of 16 keys


def ids_from_boundaries(length, starts):
    """Segment ids that go up by one at every position in `starts`."""
    ids = np.zeros(length, dtype=np.int32)
    for s in sorted(starts):
        ids[s:] += 1
    return ids


LAYOUTS = {
    # changes on the first, second, last and second-to-last key of a tile
    "edges": ids_from_boundaries(T, [1, 127, 128, 129, 254, 256, 383, 384]),
    # three runs in the first tile, four in the second, two in the ragged tail
    "many_runs": ids_from_boundaries(T, [10, 20, 140, 141, 200, 390]),
    # long documents: most tiles hold one run
    "long_docs": ids_from_boundaries(T, [150, 330]),
}


def run(seg_q, seg_kv, H, G, causal, seed, kv_rows=0):
    B, K = 2, 2
    sq = np.stack([seg_q, seg_q[::-1].copy()]).astype(np.int32)
    skv = np.stack([seg_kv, seg_kv[::-1].copy()]).astype(np.int32)
    x = inputs.make_tensors(B, K, G, T, T, H, seed=seed, backward=True, seg_q=sq, seg_kv=skv)
    dev = torch.device("cuda")
    q, k, v, dO = (t.to(dev) for t in (x.q, x.k, x.v, x.dO))
    dsq, dskv = x.seg_q.to(dev), x.seg_kv.to(dev)
    assert binding.fa_set_bwd_kv_rows(kv_rows) == binding.FA_OK
    try:
        o, lse = binding.attention_forward(q, k, v, causal=causal, seg_q=dsq, seg_kv=dskv)
        grads = binding.attention_backward(q, k, v, o, lse, dO, causal=causal, seg_q=dsq,
                                           seg_kv=dskv)
        torch.cuda.synchronize()
    finally:
        binding.fa_set_bwd_kv_rows(0)
    assert binding.fa_check_status() == binding.FA_OK
    kw = dict(causal=causal, seg_q=x.seg_q, seg_kv=x.seg_kv)
    o_ref, l_ref = oracle.attention_forward(x.q, x.k, x.v, **kw)
    check_o(to_np(o), o_ref)
    check_lse(lse.cpu().numpy().astype(np.float64), l_ref)
    for name, g, r in zip(("dq", "dk", "dv"), grads, oracle.attention_backward(x.q, x.k, x.v, x.dO, **kw)):
        check_grad(to_np(g), r, name)


@pytest.mark.parametrize("layout", sorted(LAYOUTS))
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,G,kv_rows", [(128, 4, 128), (128, 4, 64), (256, 8, 0)])
def test_same_ids(layout, causal, H, G, kv_rows):
    ids = LAYOUTS[layout]
    run(ids, ids, H, G, causal, seed=len(layout) + H + G, kv_rows=kv_rows)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,G,kv_rows", [(128, 4, 128), (128, 2, 64), (256, 8, 0)])
def test_key_ids_no_query_carries(causal, H, G, kv_rows):
    # keys 128-255 take ids 100 and 101 (two runs) that no query has: the rows of
    # those tiles match neither run; elsewhere keys and queries agree
    seg_q = LAYOUTS["edges"]
    seg_kv = seg_q.copy()
    seg_kv[128:200] = 100
    seg_kv[200:256] = 101
    run(seg_q, seg_kv, H, G, causal, seed=7 + H, kv_rows=kv_rows)
