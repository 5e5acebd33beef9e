"""Pins for the CPU oracle: invariants, closed forms, brute force, finite
differences and an independent library routine.  CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa
from flash_attention_gqa_gb300 import inputs


def rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def small(B=1, K=2, G=2, T=7, S=7, H=5, seed=0):
    q = rand((B, K, G, T, H), seed, H ** -0.5)
    k = rand((B, K, S, H), seed + 1)
    v = rand((B, K, S, H), seed + 2)
    dO = rand((B, K, G, T, H), seed + 3)
    return q, k, v, dO


# ----------------------------------------------------------------- softmax

def test_rows_sum_to_one():
    rng = np.random.default_rng(1)
    L = rng.standard_normal((3, 9, 11)) * 5
    M = rng.random((9, 11)) < 0.6
    M[:, 0] = True
    W, _ = oracle.masked_softmax(L, M[None])
    assert np.all(np.abs(W.sum(-1) - 1.0) <= 1e-12)
    assert np.all(W[:, ~M] == 0.0)
    assert np.all(W >= 0)


def test_shift_invariance():
    rng = np.random.default_rng(2)
    L = rng.standard_normal((4, 13)) * 3
    M = rng.random((4, 13)) < 0.7
    M[:, 3] = True
    W1, l1 = oracle.masked_softmax(L, M)
    W2, l2 = oracle.masked_softmax(L + 7.25, M)
    assert np.max(np.abs(W1 - W2)) <= 1e-14
    assert np.max(np.abs((l2 - l1) - 7.25)) <= 1e-12


def test_lse_is_log_sum_exp():
    rng = np.random.default_rng(3)
    L = rng.standard_normal((5, 8))
    M = np.ones((5, 8), dtype=bool)
    _, l = oracle.masked_softmax(L, M)
    assert np.allclose(l, np.log(np.exp(L).sum(-1)), rtol=0, atol=1e-13)


def test_large_logits_do_not_overflow():
    # exp of raw logits overflows; subtracting the row maximum must not
    L = np.array([[1000.0, 999.0, -1000.0]])
    W, l = oracle.masked_softmax(L, np.ones_like(L, dtype=bool))
    e = math.exp(-1.0)
    assert np.allclose(W[0], [1 / (1 + e), e / (1 + e), 0.0], atol=1e-15)
    assert abs(l[0] - (1000.0 + math.log1p(e))) < 1e-12


# ----------------------------------------------------------- closed forms

def test_two_key_closed_form():
    # q.k logits a, b -> W = (sigmoid(a-b), sigmoid(b-a)); O = W . v
    q = np.array([1.0, 2.0]).reshape(1, 1, 1, 2, 1)
    k = np.array([1.0, 0.0]).reshape(1, 1, 2, 1)
    v = np.array([1.0, 3.0]).reshape(1, 1, 2, 1)
    o, lse = oracle.attention_forward(q, k, v)
    for t, qt in enumerate([1.0, 2.0]):
        a, b = qt * 1.0, 0.0
        w0 = 1.0 / (1.0 + math.exp(b - a))
        assert abs(o[0, 0, 0, t, 0] - (w0 * 1.0 + (1 - w0) * 3.0)) < 1e-15
        assert abs(lse[0, 0, 0, t] - math.log(math.exp(a) + math.exp(b))) < 1e-14
    # causal: row 0 sees key 0 only
    o, lse = oracle.attention_forward(q, k, v, causal=True)
    assert o[0, 0, 0, 0, 0] == 1.0 and lse[0, 0, 0, 0] == 1.0


def test_single_key_returns_v_exactly():
    q, k, v, _ = small(S=1, T=4)
    o, lse = oracle.attention_forward(q, k, v)
    assert np.array_equal(o, np.broadcast_to(v[:, :, None, :, :], o.shape))
    expect = np.einsum("bkgth,bksh->bkgt", q, k)
    assert np.allclose(lse, expect, atol=1e-14)


def test_causal_row_zero_returns_v0_exactly():
    q, k, v, _ = small(T=6, S=6)
    o, _ = oracle.attention_forward(q, k, v, causal=True)
    assert np.array_equal(o[:, :, :, 0, :],
                          np.broadcast_to(v[:, :, None, 0, :], o[:, :, :, 0, :].shape))


def test_identical_keys_give_mean_of_v():
    q, k, v, _ = small(T=6, S=6)
    k[:] = k[:, :, :1, :]                       # every key equal
    o, _ = oracle.attention_forward(q, k, v)
    assert np.allclose(o, v.mean(axis=2)[:, :, None, None, :], atol=1e-14)
    o, _ = oracle.attention_forward(q, k, v, causal=True)
    for t in range(6):
        mean = v[:, :, : t + 1, :].mean(axis=2)
        assert np.allclose(o[:, :, :, t, :], mean[:, :, None, :], atol=1e-14)


def test_segments_equal_separate_attentions():
    B, K, G, T, H = 2, 2, 2, 12, 4
    q, k, v, dO = small(B, K, G, T, T, H, seed=5)
    seg = np.array([[0] * 5 + [1] * 3 + [2] * 4, [0] * 2 + [1] * 10], dtype=np.int32)
    for causal in (False, True):
        o, lse = oracle.attention_forward(q, k, v, causal=causal, seg_q=seg, seg_kv=seg)
        dq, dk, dv = oracle.attention_backward(q, k, v, dO, causal=causal,
                                               seg_q=seg, seg_kv=seg)
        for b in range(B):
            for i in np.unique(seg[b]):
                idx = np.nonzero(seg[b] == i)[0]
                lo, hi = idx[0], idx[-1] + 1
                sub = lambda x, ax: np.take(x[b:b + 1], np.arange(lo, hi), axis=ax)
                o2, l2 = oracle.attention_forward(sub(q, 3), sub(k, 2), sub(v, 2),
                                                  causal=causal)
                g2 = oracle.attention_backward(sub(q, 3), sub(k, 2), sub(v, 2),
                                               sub(dO, 3), causal=causal)
                assert np.allclose(o[b, :, :, lo:hi], o2[0], atol=1e-13)
                assert np.allclose(lse[b, :, :, lo:hi], l2[0], atol=1e-13)
                assert np.allclose(dq[b, :, :, lo:hi], g2[0][0], atol=1e-13)
                assert np.allclose(dk[b, :, lo:hi], g2[1][0], atol=1e-13)
                assert np.allclose(dv[b, :, lo:hi], g2[2][0], atol=1e-13)


def test_fully_masked_rows_are_zero():
    q, k, v, dO = small(B=1, K=1, G=2, T=4, S=4, H=3)
    seg_q = np.array([[0, 1, 9, 1]], dtype=np.int32)   # id 9 absent from keys
    seg_kv = np.array([[0, 1, 1, 1]], dtype=np.int32)
    o, lse = oracle.attention_forward(q, k, v, seg_q=seg_q, seg_kv=seg_kv)
    assert np.all(o[0, 0, :, 2] == 0.0) and np.all(np.isneginf(lse[0, 0, :, 2]))
    dq, dk, dv = oracle.attention_backward(q, k, v, dO, seg_q=seg_q, seg_kv=seg_kv)
    assert np.all(dq[0, 0, :, 2] == 0.0)
    ref = oracle.attention_bruteforce(q, k, v, dO, seg_q=seg_q, seg_kv=seg_kv)
    for a, r in zip((o, dq, dk, dv), (ref[0], ref[2], ref[3], ref[4])):
        assert np.max(np.abs(a - r)) <= 1e-12
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref[1]))
    fin = np.isfinite(lse)
    assert np.max(np.abs(lse[fin] - ref[1][fin])) <= 1e-12


# ----------------------------------------------------------- brute force

@pytest.mark.parametrize("causal,segs", [(False, False), (True, False),
                                         (False, True), (True, True)])
def test_blocked_matches_bruteforce(causal, segs):
    B, K, G, T, S, H = 2, 2, 3, 6, 6, 4
    q, k, v, dO = small(B, K, G, T, S, H, seed=11)
    sq = skv = None
    if segs:
        sq = inputs.random_segment_ids(B, T, 2, seed=4, sorted_runs=False)
        skv = inputs.random_segment_ids(B, S, 2, seed=9, sorted_runs=False)
    o, lse = oracle.attention_forward(q, k, v, causal=causal, seg_q=sq,
                                      seg_kv=skv, row_block=4)
    dq, dk, dv = oracle.attention_backward(q, k, v, dO, causal=causal, seg_q=sq,
                                           seg_kv=skv, row_block=4)
    ref = oracle.attention_bruteforce(q, k, v, dO, causal=causal, seg_q=sq, seg_kv=skv)
    for a, r in zip((o, dq, dk, dv), (ref[0], ref[2], ref[3], ref[4])):
        assert np.max(np.abs(a - r)) <= 1e-12
    fin = np.isfinite(ref[1])
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.max(np.abs(lse[fin] - ref[1][fin])) <= 1e-12


@pytest.mark.parametrize("T,S", [(3, 8), (8, 3), (5, 5), (1, 7)])
@pytest.mark.parametrize("segs", [False, True])
def test_rectangular_causal_bruteforce(T, S, segs):
    # causal with T != S: queries aligned to the end of the keys (s <= t + S - T)
    q, k, v, dO = small(B=1, K=2, G=2, T=T, S=S, H=4, seed=22 + T + S)
    sq = skv = None
    if segs:
        sq = inputs.random_segment_ids(1, T, 2, seed=5)
        skv = inputs.random_segment_ids(1, S, 2, seed=6)
    kw = dict(causal=True, seg_q=sq, seg_kv=skv)
    o, lse = oracle.attention_forward(q, k, v, row_block=2, **kw)
    dq, dk, dv = oracle.attention_backward(q, k, v, dO, row_block=2, **kw)
    ref = oracle.attention_bruteforce(q, k, v, dO, **kw)
    for a, r in zip((o, dq, dk, dv), (ref[0], ref[2], ref[3], ref[4])):
        assert np.max(np.abs(a - r)) <= 1e-12
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref[1]))
    fin = np.isfinite(lse)
    assert np.max(np.abs(lse[fin] - ref[1][fin]), initial=0.0) <= 1e-12
    # the last query sees every key (when T <= S), the first S - T + 1 keys... etc.
    if T <= S and not segs:
        m = oa.attention_mask(np.arange(T), np.arange(S), True, None, None, S - T)
        assert m[-1].all() and m[0].sum() == S - T + 1


def test_rectangular_noncausal_bruteforce():
    q, k, v, dO = small(B=1, K=2, G=2, T=3, S=8, H=4, seed=21)
    o, lse = oracle.attention_forward(q, k, v)
    dq, dk, dv = oracle.attention_backward(q, k, v, dO)
    ref = oracle.attention_bruteforce(q, k, v, dO)
    for a, r in zip((o, lse, dq, dk, dv), ref):
        assert np.max(np.abs(a - r)) <= 1e-12


# ------------------------------------------------------ finite differences

@pytest.mark.parametrize("causal,segs", [(False, False), (True, False),
                                         (True, True), (False, True)])
def test_gradients_match_finite_differences(causal, segs):
    B, K, G, T, S, H = 1, 1, 2, 5, 5, 3
    q, k, v, dO = small(B, K, G, T, S, H, seed=31)
    sq = skv = None
    if segs:
        sq = np.array([[0, 0, 1, 1, 1]], dtype=np.int32)
        skv = sq.copy()
    kw = dict(causal=causal, seg_q=sq, seg_kv=skv)
    dq, dk, dv = oracle.attention_backward(q, k, v, dO, **kw)

    def loss(qq, kk, vv):
        o, _ = oracle.attention_forward(qq, kk, vv, **kw)
        return float((o * dO).sum())

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            xp = x.copy(); xp[i] += h
            xm = x.copy(); xm[i] -= h
            args = {"q": (q, k, v), "k": (q, k, v), "v": (q, k, v)}[name]
            ap = list(args); am = list(args)
            idx = "qkv".index(name)
            ap[idx] = xp; am[idx] = xm
            fd[i] = (loss(*ap) - loss(*am)) / (2 * h)
        rel = np.linalg.norm(fd - g) / max(np.linalg.norm(g), 1e-30)
        assert rel <= 1e-6, (name, rel)


# ------------------------------------------- independent library routine

def _sdpa_reference(q, k, v, dO, causal, seg, seg_kv=None):
    """torch scaled_dot_product_attention in fp64 with autograd (scale 1 because
    q is pre-scaled); the kv heads are repeated over the G query heads."""
    B, K, G, T, H = q.shape
    S = k.shape[2]
    qt = torch.tensor(q.reshape(B, K * G, T, H), requires_grad=True)
    kt = torch.tensor(k, requires_grad=True)
    vt = torch.tensor(v, requires_grad=True)
    ke = kt.repeat_interleave(G, dim=1)
    ve = vt.repeat_interleave(G, dim=1)
    mask = None
    if causal or seg is not None:
        m = torch.ones(B, 1, T, S, dtype=torch.bool)
        if causal:
            # end-aligned causal mask: keep s <= t + (S - T)
            m &= torch.ones(T, S, dtype=torch.bool).tril(diagonal=S - T)
        if seg is not None:
            sq = torch.tensor(seg)
            sk = torch.tensor(seg if seg_kv is None else seg_kv)
            m &= (sq[:, :, None] == sk[:, None, :])[:, None]
        mask = m
    o = torch.nn.functional.scaled_dot_product_attention(qt, ke, ve, attn_mask=mask,
                                                         scale=1.0)
    o.backward(torch.tensor(dO.reshape(B, K * G, T, H)))
    return (o.detach().numpy().reshape(B, K, G, T, H),
            qt.grad.numpy().reshape(B, K, G, T, H), kt.grad.numpy(), vt.grad.numpy())


@pytest.mark.parametrize("causal,segs", [(False, False), (True, False), (True, True)])
def test_matches_torch_sdpa_fp64(causal, segs):
    B, K, G, T, H = 2, 2, 4, 40, 16
    q, k, v, dO = small(B, K, G, T, T, H, seed=41)
    seg = inputs.document_segment_ids(B, T, seed=3, lo=5, hi=17) if segs else None
    o, _ = oracle.attention_forward(q, k, v, causal=causal, seg_q=seg, seg_kv=seg,
                                    row_block=16)
    dq, dk, dv = oracle.attention_backward(q, k, v, dO, causal=causal, seg_q=seg,
                                           seg_kv=seg, row_block=16)
    ro, rdq, rdk, rdv = _sdpa_reference(q, k, v, dO, causal, seg)
    for a, r in ((o, ro), (dq, rdq), (dk, rdk), (dv, rdv)):
        assert np.max(np.abs(a - r)) <= 1e-12


@pytest.mark.parametrize("T,S", [(24, 40), (40, 24)])
def test_rectangular_causal_matches_torch_sdpa(T, S):
    B, K, G, H = 1, 2, 2, 8
    rng = np.random.default_rng(7)
    q = rng.standard_normal((B, K, G, T, H)) * H ** -0.5
    k = rng.standard_normal((B, K, S, H))
    v = rng.standard_normal((B, K, S, H))
    dO = rng.standard_normal((B, K, G, T, H))
    o, _ = oracle.attention_forward(q, k, v, causal=True, row_block=7)
    dq, dk, dv = oracle.attention_backward(q, k, v, dO, causal=True, row_block=7)
    ro, rdq, rdk, rdv = _sdpa_reference(q, k, v, dO, True, None)
    rows = slice(max(0, T - S), T)   # rows with at least one key (SDPA gives NaN otherwise)
    assert np.max(np.abs(o[:, :, :, rows] - ro[:, :, :, rows])) <= 1e-12
    assert np.max(np.abs(dq[:, :, :, rows] - rdq[:, :, :, rows])) <= 1e-12
    if T <= S:
        assert np.max(np.abs(dk - rdk)) <= 1e-12 and np.max(np.abs(dv - rdv)) <= 1e-12


# ----------------------------------------------- sampled-row entry points

def test_sampled_rows_match_full():
    B, K, G, T, H = 2, 2, 2, 64, 8
    q, k, v, dO = small(B, K, G, T, T, H, seed=51)
    seg = inputs.document_segment_ids(B, T, seed=1, lo=5, hi=30)
    kw = dict(causal=True, seg_q=seg, seg_kv=seg)
    o, lse = oracle.attention_forward(q, k, v, **kw)
    dq, dk, dv = oracle.attention_backward(q, k, v, dO, **kw)
    rows = [0, 5, 31, 63]
    o2, l2 = oracle.attention_rows(q, k, v, 1, 0, 1, rows, **kw)
    assert np.max(np.abs(o2 - o[1, 0, 1, rows])) <= 1e-13
    assert np.max(np.abs(l2 - lse[1, 0, 1, rows])) <= 1e-13
    srows = [0, 7, 40, 63]
    gq, gk, gv, l3, _ = oracle.attention_backward_rows(q, k, v, dO, 1, 1, t_rows=rows,
                                                       s_rows=srows, row_block=16, **kw)
    assert np.max(np.abs(gq - dq[1, 1][:, rows])) <= 1e-12
    assert np.max(np.abs(gk - dk[1, 1][srows])) <= 1e-12
    assert np.max(np.abs(gv - dv[1, 1][srows])) <= 1e-12
    assert np.max(np.abs(l3 - lse[1, 1])) <= 1e-12


def test_sampled_late_keys_skip_rows_exactly():
    # with only late sampled keys, rows that cannot see them are skipped; the
    # sampled dk / dv / dq must not change
    B, K, G, T, H = 1, 1, 2, 96, 8
    q, k, v, dO = small(B, K, G, T, T, H, seed=53)
    dq, dk, dv = oracle.attention_backward(q, k, v, dO, causal=True)
    rows, srows = [3, 50, 95], [70, 80, 95]
    gq, gk, gv, lse, _ = oracle.attention_backward_rows(q, k, v, dO, 0, 0, t_rows=rows,
                                                        s_rows=srows, row_block=16, causal=True)
    assert np.max(np.abs(gq - dq[0, 0][:, rows])) <= 1e-12
    assert np.max(np.abs(gk - dk[0, 0][srows])) <= 1e-12
    assert np.max(np.abs(gv - dv[0, 0][srows])) <= 1e-12
    assert np.isneginf(lse[:, 20]).all()        # a skipped row (no sampled key visible)


def test_row_block_size_does_not_matter():
    q, k, v, dO = small(B=1, K=1, G=3, T=33, S=33, H=6, seed=61)
    a = oracle.attention_backward(q, k, v, dO, causal=True, row_block=1)
    b = oracle.attention_backward(q, k, v, dO, causal=True, row_block=512)
    for x, y in zip(a, b):
        assert np.max(np.abs(x - y)) <= 1e-13


# -------------------------------------------- planted mistakes are caught

def _fd_grads(q, k, v, dO, causal, h=1e-6):
    """Central differences of sum(O * dO) through the oracle forward."""
    def loss(qq, kk, vv):
        o, _ = oracle.attention_forward(qq, kk, vv, causal=causal)
        return float((o * dO).sum())
    out = []
    for idx, x in enumerate((q, k, v)):
        fd = np.zeros_like(x)
        for i in np.ndindex(x.shape):
            args_p, args_m = [q, k, v], [q, k, v]
            xp = x.copy(); xp[i] += h
            xm = x.copy(); xm[i] -= h
            args_p[idx], args_m[idx] = xp, xm
            fd[i] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        out.append(fd)
    return out


def _slipped_backward(q, k, v, dO, slip):
    """The backward with one deliberate slip (planted on the CPU only)."""
    B, K, G, T, H = q.shape
    S = k.shape[2]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    M = oa.attention_mask(np.arange(T), np.arange(S), True, None, None)
    for b in range(B):
        for kh in range(K):
            qb, dOb = q[b, kh], dO[b, kh]
            W, _ = oracle.masked_softmax(qb @ k[b, kh].T, M[None])
            dP = dOb @ v[b, kh].T
            if slip == "dropped_rowsum":
                dS = W * dP
            elif slip == "wrong_sign":
                dS = W * (dP + (W * dP).sum(-1, keepdims=True))
            else:
                dS = W * (dP - (W * dP).sum(-1, keepdims=True))
            dq[b, kh] = dS @ (v[b, kh] if slip == "wrong_operand" else k[b, kh])
            gs = [0] if slip == "no_group_sum" else range(G)
            for g in gs:
                dk[b, kh] += dS[g].T @ qb[g]
                dv[b, kh] += (W[g] if slip != "transposed_w" else W[g][::-1, ::-1]).T @ dOb[g]
    return dq, dk, dv


def test_planted_mistakes_fail_the_finite_difference_pin():
    q, k, v, dO = small(B=1, K=1, G=2, T=4, S=4, H=4, seed=71)
    fd = _fd_grads(q, k, v, dO, causal=True)

    def worst(grads):
        return max(np.linalg.norm(a - f) / np.linalg.norm(f) for a, f in zip(grads, fd))

    assert worst(oracle.attention_backward(q, k, v, dO, causal=True)) <= 1e-6
    assert worst(_slipped_backward(q, k, v, dO, None)) <= 1e-6
    for slip in ("dropped_rowsum", "wrong_sign", "wrong_operand", "no_group_sum",
                 "transposed_w"):
        assert worst(_slipped_backward(q, k, v, dO, slip)) > 1e-3, slip


def test_planted_unmasked_softmax_fails_bruteforce(monkeypatch):
    q, k, v, _ = small(B=1, K=1, G=2, T=4, S=4, H=3, seed=72)
    real = oa.masked_softmax
    monkeypatch.setattr(oa, "masked_softmax", lambda L, M: real(L, np.ones_like(M)))
    o_bad, _ = oa.attention_forward(q, k, v, causal=True)
    monkeypatch.setattr(oa, "masked_softmax", real)
    o_ref = oracle.attention_bruteforce(q, k, v, causal=True)[0]
    assert np.max(np.abs(o_bad - o_ref)) > 1e-3


def test_unmasked_pair_count():
    seg = inputs.document_segment_ids(2, 300, seed=0, lo=10, hi=90)
    n = inputs.unmasked_pairs(300, 300, True, seg, seg)
    brute = 0
    for b in range(2):
        m = oa.attention_mask(np.arange(300), np.arange(300), True, seg[b], seg[b])
        brute += int(m.sum())
    assert n == brute
    assert inputs.unmasked_pairs(7, 7, True, None, None) == 28
    assert inputs.unmasked_pairs(7, 5, False, None, None) == 35
    for T, S in ((3, 9), (9, 3)):
        m = oa.attention_mask(np.arange(T), np.arange(S), True, None, None, S - T)
        assert inputs.unmasked_pairs(T, S, True, None, None) == int(m.sum())


# ------------------------------------------------------ explicit masks

def test_explicit_mask_matches_bruteforce_per_head():
    B, K, G, T, S, H = 1, 2, 2, 6, 7, 3
    q, k, v, dO = small(B, K, G, T, S, H, seed=81)
    rng = np.random.default_rng(3)
    mask = rng.random((K * G, T, S)) < 0.6
    for causal in (False, True):
        o, lse = oracle.attention_forward(q, k, v, causal=causal, mask=mask, row_block=4)
        g = oracle.attention_backward(q, k, v, dO, causal=causal, mask=mask, row_block=4)
        ref = oracle.attention_bruteforce(q, k, v, dO, causal=causal, mask=mask)
        for a, r in zip((o, *g), (ref[0], ref[2], ref[3], ref[4])):
            assert np.max(np.abs(a - r)) <= 1e-12
        assert np.array_equal(np.isneginf(lse), np.isneginf(ref[1]))


def test_explicit_mask_equal_to_causal_gives_causal():
    q, k, v, dO = small(B=1, K=2, G=2, T=9, S=9, H=4, seed=82)
    tri = np.tril(np.ones((9, 9), dtype=bool))[None]
    a = oracle.attention_forward(q, k, v, mask=tri)
    b = oracle.attention_forward(q, k, v, causal=True)
    assert np.max(np.abs(a[0] - b[0])) <= 1e-14
    ga = oracle.attention_backward(q, k, v, dO, mask=tri)
    gb = oracle.attention_backward(q, k, v, dO, causal=True)
    for x, y in zip(ga, gb):
        assert np.max(np.abs(x - y)) <= 1e-13
    full = np.ones((1, 9, 9), dtype=bool)
    c = oracle.attention_forward(q, k, v, mask=full)
    d = oracle.attention_forward(q, k, v)
    assert np.max(np.abs(c[0] - d[0])) <= 1e-15
