"""Parity at the full sizes of the three long workloads, launched as bench.py
times them.

The timed step is one fa_fwd and one fa_bwd call on one stream (the dQ grid
may start while the dK/dV grid drains); bench.py's per-kernel loop runs
fa_bwd_stage 0, 1, 2 with events between them.  Both launch orders run here
and must give the same bits.

* causal H=256, T=S=8192 (model_dim 4096, 16 query heads, 2 kv heads) and the
  packed-document workload (causal + segment ids, H=128, T=S=4096): every
  element of O, lse, dq, dk and dv against the full oracle.
* the 1024-key causal sliding window (H=128, T=S=8192) as a block-sparse mask:
  every element of O, lse, dq, dk and dv against the oracle's dense mask.
* one decode step (T=1, S=32768, split-KV): every element of O and lse.
* causal H=256, T=S=32768: O and lse at one query row of every Q tile of every
  head (the row within the tile rotates from tile to tile), and dk, dv over
  three whole 64-key tiles (the first, one in the middle, the last) of both kv
  heads, with dq at sampled query rows.

The oracle runs on the host in spawned worker processes, one (b, kv head) or
one head per worker: minutes of fp64 time.  GPU only."""
import numpy as np
import pytest
import torch

import _oracle_pool as pool
from flash_attention_gqa_gb300 import binding, inputs
from _parity import GRAD_REL_FRO, LSE_ABS, O_MAX_ABS, O_REL_FRO

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def run_bench_launch(w):
    """fa_fwd + fa_bwd (one call), then the staged backward into fresh
    outputs; returns the workload's CPU tensors and the GPU results (CPU)."""
    x = inputs.make_workload(w)
    dev = torch.device("cuda")
    q, k, v, dO = (t.to(dev) for t in (x.q, x.k, x.v, x.dO))
    sq = None if x.seg_q is None else x.seg_q.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.K, w.G, w.T), dtype=torch.float32, device=dev)
    ws = torch.empty(max(256, binding.fa_bwd_workspace_size(w.B, w.K, w.G, w.T, w.S, w.H)),
                     dtype=torch.uint8, device=dev)
    binding.fa_fwd(q, k, v, sq, sq, w.causal, o, lse)
    grads = [torch.empty_like(t) for t in (q, k, v)]
    binding.fa_bwd(q, k, v, o, lse, dO, sq, sq, w.causal, *grads, ws)
    staged = [torch.empty_like(t) for t in (q, k, v)]
    for st in range(3):
        binding.fa_bwd_stage(st, q, k, v, o, lse, dO, sq, sq, w.causal, *staged, ws)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    for name, a, b in zip(("dq", "dk", "dv"), grads, staged):
        assert torch.equal(a, b), f"{name}: fa_bwd and fa_bwd_stage 0-2 differ"
    del staged, ws
    return x, o.cpu(), lse.cpu(), [t.cpu() for t in grads]


def f32(t):
    return t.float().numpy()


def seg_slice(x, b):
    return (None, None) if x.seg_q is None else (x.seg_q[b:b + 1].numpy(),
                                                 x.seg_kv[b:b + 1].numpy())


def assert_results(res, grads=("dq", "dk", "dv")):
    o = pool.merge([r["o"] for r in res if "o" in r])
    lse = pool.merge([r["lse"] for r in res if "lse" in r])
    if o["n"]:
        assert o["inf_mismatch"] == 0 and o["nonfinite_gpu"] == 0, o
        assert o["max_abs"] <= O_MAX_ABS, f"O max abs {o['max_abs']:.3e}"
        assert o["rel_fro"] <= O_REL_FRO, f"O rel Frobenius {o['rel_fro']:.3e}"
    if lse["n"]:
        assert lse["inf_mismatch"] == 0 and lse["nonfinite_gpu"] == 0, lse
        assert lse["max_abs"] <= LSE_ABS, f"lse max abs {lse['max_abs']:.3e}"
    for name in grads:
        g = pool.merge([r[name] for r in res if name in r])
        assert g["n"] > 0
        assert g["inf_mismatch"] == 0 and g["nonfinite_gpu"] == 0, (name, g)
        assert g["rel_fro"] <= GRAD_REL_FRO, f"{name} rel Frobenius {g['rel_fro']:.3e}"
    return o, lse


def check_every_element(name):
    w = inputs.WORKLOADS[name]
    x, o, lse, (dq, dk, dv) = run_bench_launch(w)
    jobs = []
    for b in range(w.B):
        sq, skv = seg_slice(x, b)
        for kh in range(w.K):
            u = np.s_[b:b + 1, kh:kh + 1]
            common = dict(q=f32(x.q[u]), k=f32(x.k[u]), v=f32(x.v[u]), seg_q=sq, seg_kv=skv,
                          causal=w.causal)
            jobs.append(dict(common, part="fwd", o_gpu=f32(o[u]), lse_gpu=lse[u].numpy()))
            jobs.append(dict(common, part="bwd", dO=f32(x.dO[u]), dq_gpu=f32(dq[u]),
                             dk_gpu=f32(dk[u]), dv_gpu=f32(dv[u])))
    res = pool.run(pool.full_unit, jobs)
    o_res, l_res = assert_results(res)
    assert o_res["n"] == x.q.numel() and l_res["n"] == lse.numel()


def test_window1024_h128_t8192_every_element():
    """The 1024-key causal sliding window given as a block-sparse mask: fa_fwd_masked
    and fa_bwd_masked with the block metadata built from the dense mask, as bench.py
    runs them; every element of O, lse, dq, dk, dv against the oracle's dense mask."""
    w = inputs.WORKLOADS["gqa_window1024_h128_t8192"]
    x = inputs.make_workload(w)
    dev = torch.device("cuda")
    meta = binding.block_mask_from_dense(inputs.window_mask(w.T, w.S, w.window), device=dev)
    q, k, v, dO = (t.to(dev) for t in (x.q, x.k, x.v, x.dO))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.K, w.G, w.T), dtype=torch.float32, device=dev)
    binding.fa_fwd_masked(q, k, v, None, None, w.causal, meta, o, lse)
    grads = [torch.empty_like(t) for t in (q, k, v)]
    ws = torch.empty(max(256, binding.fa_bwd_workspace_size(w.B, w.K, w.G, w.T, w.S, w.H)),
                     dtype=torch.uint8, device=dev)
    binding.fa_bwd_masked(q, k, v, o, lse, dO, None, None, w.causal, meta, *grads, ws)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    o, lse, (dq, dk, dv) = o.cpu(), lse.cpu(), [t.cpu() for t in grads]
    jobs = []
    for b in range(w.B):
        for kh in range(w.K):
            u = np.s_[b:b + 1, kh:kh + 1]
            common = dict(q=f32(x.q[u]), k=f32(x.k[u]), v=f32(x.v[u]), seg_q=None, seg_kv=None,
                          causal=w.causal, window=(w.T, w.S, w.window))
            jobs.append(dict(common, part="fwd", o_gpu=f32(o[u]), lse_gpu=lse[u].numpy()))
            jobs.append(dict(common, part="bwd", dO=f32(x.dO[u]), dq_gpu=f32(dq[u]),
                             dk_gpu=f32(dk[u]), dv_gpu=f32(dv[u])))
    o_res, l_res = assert_results(pool.run(pool.full_unit, jobs))
    assert o_res["n"] == x.q.numel() and l_res["n"] == lse.numel()


def test_causal_h256_t8192_every_element():
    check_every_element("gqa_causal_h256_t8192")


def test_packed_docs_h128_t4096_every_element():
    check_every_element("gqa_packed_docs_h128_t4096")


def test_causal_h256_t32768_every_q_tile_and_three_key_tiles():
    w = inputs.WORKLOADS["gqa_causal_h256_t32768"]
    x, o, lse, (dq, dk, dv) = run_bench_launch(w)
    Tb = 128 // w.G                      # query positions per packed Q tile
    n_qt = -(-w.T // Tb)
    # forward: one row in every Q tile of every (kv head, g)
    jobs = []
    for kh in range(w.K):
        for g in range(w.G):
            rows = np.minimum(np.arange(n_qt) * Tb + (np.arange(n_qt) * 5 + 3 * g + kh) % Tb,
                              w.T - 1)
            jobs.append(dict(q=f32(x.q[0:1, kh:kh + 1, g:g + 1]), k=f32(x.k[0:1, kh:kh + 1]),
                             v=f32(x.v[0:1, kh:kh + 1]), seg_q=None, seg_kv=None,
                             causal=w.causal, rows=rows, o_gpu=f32(o[0, kh, g, rows]),
                             lse_gpu=lse[0, kh, g, rows].numpy()))
    o_res, l_res = assert_results(pool.run(pool.rows_unit, jobs), grads=())
    assert o_res["n"] == w.K * w.G * n_qt * w.H and l_res["n"] == w.K * w.G * n_qt
    # backward: whole 64-key tiles at the start, middle and end of S; dq at sampled rows
    kv = 64
    s_rows = np.concatenate([np.arange(0, kv), np.arange(w.S // 2, w.S // 2 + kv),
                             np.arange(w.S - kv, w.S)])
    rng = np.random.default_rng(4)
    t_rows = np.unique(np.concatenate([[0, 1, w.T // 2, w.T - 1], rng.integers(0, w.T, 60)]))
    jobs = []
    for kh in range(w.K):
        jobs.append(dict(q=f32(x.q[0:1, kh:kh + 1]), k=f32(x.k[0:1, kh:kh + 1]),
                         v=f32(x.v[0:1, kh:kh + 1]), dO=f32(x.dO[0:1, kh:kh + 1]),
                         seg_q=None, seg_kv=None, causal=w.causal, t_rows=t_rows, s_rows=s_rows,
                         dq_gpu=f32(dq[0, kh][:, t_rows]), dk_gpu=f32(dk[0, kh][s_rows]),
                         dv_gpu=f32(dv[0, kh][s_rows])))
    assert_results(pool.run(pool.keys_unit, jobs))


def test_decode_h128_s32768_every_element():
    """One decode step (T=1) against a 32768-key cache, B=8 K=8 G=8 H=128, through
    fa_fwd_splitkv with the default split count, as bench.py runs it: every element
    of O and lse against the full oracle."""
    w = inputs.WORKLOADS["gqa_decode_h128_s32768"]
    x = inputs.make_workload(w)
    dev = torch.device("cuda")
    o, lse = binding.attention_forward_splitkv(x.q.to(dev), x.k.to(dev), x.v.to(dev),
                                               causal=w.causal)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    o, lse = o.cpu(), lse.cpu()
    jobs = []
    for b in range(w.B):
        for kh in range(w.K):
            u = np.s_[b:b + 1, kh:kh + 1]
            jobs.append(dict(q=f32(x.q[u]), k=f32(x.k[u]), v=f32(x.v[u]), seg_q=None, seg_kv=None,
                             causal=w.causal, part="fwd", o_gpu=f32(o[u]), lse_gpu=lse[u].numpy()))
    o_res, l_res = assert_results(pool.run(pool.full_unit, jobs), grads=())
    assert o_res["n"] == x.q.numel() and l_res["n"] == lse.numel()
