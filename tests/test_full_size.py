"""Parity at the full sizes of the three large workloads, launched the way
bench.py times them (fa_fwd, then fa_bwd_stage 0, 1, 2 on one stream), checked
on sampled outputs the oracle computes one by one: O and lse rows, dq rows, and
dk / dv rows (whose oracle needs every row's lse and rowsum(W dP) first).
GPU only; a few tens of seconds of fp64 oracle time on the host."""
import numpy as np
import pytest
import torch

import oracle
from flash_attention_gqa_gb300 import binding, inputs
from _parity import LSE_ABS, O_MAX_ABS, check_grad, rel_fro, to_np

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def run_bench_launch(w):
    x = inputs.make_workload(w)
    dev = torch.device("cuda")
    q, k, v, dO = (t.to(dev) for t in (x.q, x.k, x.v, x.dO))
    sq = None if x.seg_q is None else x.seg_q.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.K, w.G, w.T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(binding.fa_bwd_workspace_size(w.B, w.K, w.G, w.T, w.S, w.H),
                     dtype=torch.uint8, device=dev)
    binding.fa_fwd(q, k, v, sq, sq, w.causal, o, lse)
    for st in range(3):
        binding.fa_bwd_stage(st, q, k, v, o, lse, dO, sq, sq, w.causal, dq, dk, dv, ws)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    return x, o.cpu(), lse.cpu(), dq.cpu(), dk.cpu(), dv.cpu()


def sample_rows(T, n, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, T // 2, T - 1]
    return np.unique(np.concatenate([fixed, rng.integers(0, T, n)]))


def check_workload(name, bwd_heads, n_rows=12, n_keys=12, late_keys=0):
    w = inputs.WORKLOADS[name]
    x, o, lse, dq, dk, dv = run_bench_launch(w)
    kw = dict(causal=w.causal, seg_q=x.seg_q, seg_kv=x.seg_kv)
    # forward: sampled rows of every (b, kv head, g)
    og, orf, lg, lrf = [], [], [], []
    for b in range(w.B):
        for kh in range(w.K):
            for g in range(w.G):
                rows = sample_rows(w.T, 3, seed=b * 131 + kh * 17 + g)
                o_ref, l_ref = oracle.attention_rows(x.q, x.k, x.v, b, kh, g, rows, **kw)
                og.append(to_np(o[b, kh, g, rows])); orf.append(o_ref)
                lg.append(lse[b, kh, g, rows].numpy().astype(np.float64)); lrf.append(l_ref)
    og, orf = np.concatenate(og), np.concatenate(orf)
    lg, lrf = np.concatenate(lg), np.concatenate(lrf)
    assert np.max(np.abs(og - orf)) <= O_MAX_ABS
    assert rel_fro(og, orf) <= 5e-3
    fin = np.isfinite(lrf)
    assert np.array_equal(fin, np.isfinite(lg))
    assert np.max(np.abs(lg[fin] - lrf[fin])) <= LSE_ABS
    # backward: sampled query rows (dq) and key rows (dk, dv) of the chosen heads
    for b, kh in bwd_heads:
        t_rows = sample_rows(w.T, n_rows, seed=7 + kh)
        s_rows = sample_rows(w.S, n_keys, seed=11 + kh)
        if late_keys:   # keys near the end: only the rows that can see them matter
            s_rows = np.unique(np.concatenate([s_rows[s_rows >= w.S - late_keys], [w.S - 1]]))
        gq, gk, gv, _, _ = oracle.attention_backward_rows(
            x.q, x.k, x.v, x.dO, b, kh, t_rows=t_rows, s_rows=s_rows, row_block=256, **kw)
        check_grad(to_np(dq[b, kh][:, t_rows]), gq, f"dq[{b},{kh}]")
        check_grad(to_np(dk[b, kh][s_rows]), gk, f"dk[{b},{kh}]")
        check_grad(to_np(dv[b, kh][s_rows]), gv, f"dv[{b},{kh}]")


def test_causal_h256_t8192_full_size():
    check_workload("gqa_causal_h256_t8192", bwd_heads=[(0, 0), (0, 1)])


def test_causal_h256_t32768_full_size():
    check_workload("gqa_causal_h256_t32768", bwd_heads=[(0, 1)], n_rows=8, n_keys=64,
                   late_keys=4096)


def test_packed_docs_h128_t4096_full_size():
    check_workload("gqa_packed_docs_h128_t4096", bwd_heads=[(0, 3), (3, 7)])
