"""CPU oracle for blocked GQA flash attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
reference legs of ``bench.py`` may import or run this module.  The product
(the CUDA library and its Python binding) never calls it, and it shares no
code with the CUDA path.

What it computes is the plain definition of masked softmax attention, in
float64, on the bf16-rounded inputs:

  * Logits  L[b,k,g,t,s] = sum_h q[b,k,g,t,h] * k[b,k,s,h]; q arrives already
    multiplied by H**-0.5, so no further scale is applied ("What is wrong with
    naive attention?", danielwatson6.github.io/fa/fa.html: the naive GQA
    attention with pre-scaled queries and the bkgth,bksh->bkgts contraction).
  * Mask    M[t,s] = (s <= t if causal) and (seg_q[b,t] == seg_kv[b,s] if
    segment ids are given) -- SegmentIds docs (a token attends only to tokens
    carrying the same segment id; pallas_operations.flash_attention.tpu.
    jax_flash_attn_tpu, section "SegmentIds"); causal as the lower-triangular mask of the axlearn
    PR "Optimize TPU Flash Attention (400x speed-up on 32k long context)".
  * Softmax over the kept keys with the maximum subtracted (the tutorial's
    "Chunked attention" section: softmax(l) = softmax(l + c)), then
    O = W . v (bkgts,bksh->bkgth) and lse = max + log(sum exp(L - max)).
  * Backward (not on the pages; textbook derivative of the same formula):
      dP = dO . v^T,  dS = W * (dP - rowsum(W * dP)),  dq = dS . k,
      dk = sum_g dS^T . q,  dv = sum_g W^T . dO.

Readings where the pages are silent (all listed with the design notes):
  * causal keeps s <= t + (S - T): queries are aligned to the end of the keys,
    so the last query sees every key; for T == S this is s <= t with the same
    absolute index for queries and keys (the pages only use T == S);
  * an optional explicit mask ``mask[h, t, s]`` (h = k*G + g, the query head
    within a batch row, or a single head shared by all) is ANDed with the causal and segment
    masks: the dense form of the block-sparse mask metadata the kernels take
    (splash attention's MultiHeadMask / process_mask in the tutorial's
    "Our first kernel" baseline);
  * a query row with no kept key has O = 0, lse = -inf and contributes no
    gradient (with attention limited to equal ids, such a row has nothing to
    attend to);
  * natural exp/log throughout; lse is in natural-log units.

Everything is blocked over query rows only, so long sequences fit in memory;
there is no other blocking, fusion or reordering.  ``attention_bruteforce`` is
a pure-Python triple loop for tiny shapes.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

NEG_INF = -np.inf


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor (any dtype): exact widening
        x = x.detach().cpu().float().numpy()
    return np.asarray(x, dtype=np.float64)


def _i32(x) -> Optional[np.ndarray]:
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.asarray(x, dtype=np.int64)


def attention_mask(t_idx: np.ndarray, s_idx: np.ndarray, causal: bool,
                   seg_q_row: Optional[np.ndarray],
                   seg_kv_row: Optional[np.ndarray], offset: int = 0) -> np.ndarray:
    """Boolean keep-mask M[t, s] for the given query and key positions.

    ``offset`` is S - T: with ``causal`` a query t keeps the keys s <= t + offset."""
    m = np.ones((len(t_idx), len(s_idx)), dtype=bool)
    if causal:
        m &= s_idx[None, :] <= t_idx[:, None] + offset
    if seg_q_row is not None:
        m &= seg_q_row[t_idx][:, None] == seg_kv_row[s_idx][None, :]
    return m


def masked_softmax(L: np.ndarray, M: np.ndarray):
    """Explicit softmax of logits ``L[..., s]`` over the keys kept by ``M``.

    Returns (W, lse).  The row maximum over kept keys is subtracted before the
    exponential; rows with no kept key get W = 0 and lse = -inf."""
    Lm = np.where(M, L, NEG_INF)
    mx = Lm.max(axis=-1, keepdims=True)
    empty = ~np.isfinite(mx)
    mx_safe = np.where(empty, 0.0, mx)
    E = np.where(M, np.exp(Lm - mx_safe), 0.0)
    den = E.sum(axis=-1, keepdims=True)
    W = np.where(empty, 0.0, E / np.where(empty, 1.0, den))
    lse = np.where(empty, NEG_INF, mx_safe + np.log(np.where(empty, 1.0, den)))
    return W, lse[..., 0]


def _row_blocks(T: int, rb: int):
    for t0 in range(0, T, rb):
        yield t0, min(T, t0 + rb)


def _key_range(t1: int, S: int, causal: bool, offset: int = 0) -> int:
    # keys s >= t1 + offset are masked for every row t < t1 when causal; they
    # would only contribute exact zeros, so the logits are not evaluated there.
    return max(0, min(S, t1 + offset)) if causal else S


def _head_mask(mask, kh, G, t_idx, s_idx):
    """[G, rows, keys] slice of the explicit mask for kv head kh (or None)."""
    if mask is None:
        return None
    m = np.asarray(mask, dtype=bool)
    if m.shape[0] == 1:
        return np.broadcast_to(m[0][np.ix_(t_idx, s_idx)][None], (G, len(t_idx), len(s_idx)))
    return np.stack([m[kh * G + g][np.ix_(t_idx, s_idx)] for g in range(G)])


def attention_forward(q, k, v, *, causal: bool = False, seg_q=None,
                      seg_kv=None, row_block: int = 512,
                      heads: Optional[Sequence[tuple]] = None, mask=None):
    """Masked GQA attention.  q [B,K,G,T,H], k/v [B,K,S,H] -> (o, lse).

    ``o`` is [B,K,G,T,H] float64 and ``lse`` [B,K,G,T] float64.  ``heads``
    restricts the work to the listed (b, kv_head) pairs (others stay zero)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    sq, skv = _i32(seg_q), _i32(seg_kv)
    B, K, G, T, H = q.shape
    S = k.shape[2]
    o = np.zeros((B, K, G, T, H))
    lse = np.full((B, K, G, T), NEG_INF)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(K)]
    s_all = np.arange(S)
    off = S - T
    for b, kh in pairs:
        for t0, t1 in _row_blocks(T, row_block):
            ns = _key_range(t1, S, causal, off)
            if ns == 0:       # no key is visible to these rows: O = 0, lse = -inf
                continue
            t_idx = np.arange(t0, t1)
            M = attention_mask(t_idx, s_all[:ns], causal,
                               None if sq is None else sq[b],
                               None if skv is None else skv[b], off)[None]
            hm = _head_mask(mask, kh, G, t_idx, s_all[:ns])
            if hm is not None:
                M = M & hm
            L = q[b, kh, :, t0:t1, :] @ k[b, kh, :ns, :].T       # [G, rb, ns]
            W, l = masked_softmax(L, M)
            o[b, kh, :, t0:t1, :] = W @ v[b, kh, :ns, :]
            lse[b, kh, :, t0:t1] = l
    return o, lse


def attention_backward(q, k, v, dO, *, causal: bool = False, seg_q=None,
                       seg_kv=None, row_block: int = 512,
                       heads: Optional[Sequence[tuple]] = None, mask=None):
    """Gradients of sum(O * dO) with respect to q, k, v (float64)."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    sq, skv = _i32(seg_q), _i32(seg_kv)
    B, K, G, T, H = q.shape
    S = k.shape[2]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(K)]
    s_all = np.arange(S)
    off = S - T
    for b, kh in pairs:
        for t0, t1 in _row_blocks(T, row_block):
            ns = _key_range(t1, S, causal, off)
            if ns == 0:       # rows with no visible key contribute no gradient
                continue
            t_idx = np.arange(t0, t1)
            M = attention_mask(t_idx, s_all[:ns], causal,
                               None if sq is None else sq[b],
                               None if skv is None else skv[b], off)[None]
            hm = _head_mask(mask, kh, G, t_idx, s_all[:ns])
            if hm is not None:
                M = M & hm
            qb = q[b, kh, :, t0:t1, :]                            # [G, rb, H]
            dOb = dO[b, kh, :, t0:t1, :]
            L = qb @ k[b, kh, :ns, :].T                           # [G, rb, ns]
            W, _ = masked_softmax(L, M)
            dP = dOb @ v[b, kh, :ns, :].T                         # [G, rb, ns]
            dS = W * (dP - (W * dP).sum(axis=-1, keepdims=True))
            dq[b, kh, :, t0:t1, :] = dS @ k[b, kh, :ns, :]
            dk[b, kh, :ns, :] += np.einsum("grs,grh->sh", dS, qb)
            dv[b, kh, :ns, :] += np.einsum("grs,grh->sh", W, dOb)
    return dq, dk, dv


def attention_rows(q, k, v, b: int, kh: int, g: int, t_rows, *,
                   causal: bool = False, seg_q=None, seg_kv=None):
    """O and lse of the listed query rows of one (b, kv_head, g) only."""
    q, k, v = _f64(q[b, kh, g]), _f64(k[b, kh]), _f64(v[b, kh])
    sq, skv = _i32(seg_q), _i32(seg_kv)
    t_idx = np.asarray(t_rows)
    S = k.shape[0]
    M = attention_mask(t_idx, np.arange(S), causal,
                       None if sq is None else sq[b],
                       None if skv is None else skv[b], S - q.shape[0])
    W, l = masked_softmax(q[t_idx] @ k.T, M)
    return W @ v, l


def attention_backward_rows(q, k, v, dO, b: int, kh: int, *, t_rows, s_rows,
                            causal: bool = False, seg_q=None, seg_kv=None,
                            row_block: int = 1024):
    """Sampled gradients of one (b, kv_head): dq at query rows ``t_rows`` (all
    G heads) and dk, dv at key rows ``s_rows``.

    dk/dv at a key need the softmax normaliser and rowsum(W * dP) of every
    query that sees the key, so those two per-row statistics are computed
    first (blocked over query rows, the same definition as
    ``attention_backward``) for the rows that matter."""
    qh, kk, vv, dOh = _f64(q[b, kh]), _f64(k[b, kh]), _f64(v[b, kh]), _f64(dO[b, kh])
    sq, skv = _i32(seg_q), _i32(seg_kv)
    G, T, H = qh.shape
    S = kk.shape[0]
    sqb = None if sq is None else sq[b]
    skb = None if skv is None else skv[b]
    t_rows = np.asarray(t_rows)
    s_rows = np.asarray(s_rows)
    off = S - T
    # Rows whose statistics are needed: the sampled query rows, and every row
    # that can see a sampled key.  Under the causal mask a row t sees key s
    # only if s <= t + off, so rows t < min(s_rows) - off contribute exactly
    # zero to the sampled dk / dv and are skipped (lse stays -inf there).
    need = np.zeros(T, dtype=bool)
    need[t_rows] = True
    if causal:
        need[max(0, int(s_rows.min()) - off):] = True
    else:
        need[:] = True
    lse = np.full((G, T), NEG_INF)
    delta = np.zeros((G, T))
    s_all = np.arange(S)
    for t0, t1 in _row_blocks(T, row_block):
        if not need[t0:t1].any():
            continue
        ns = _key_range(t1, S, causal, off)
        if ns == 0:
            continue
        M = attention_mask(np.arange(t0, t1), s_all[:ns], causal, sqb, skb, off)
        W, l = masked_softmax(qh[:, t0:t1] @ kk[:ns].T, M[None])
        dP = dOh[:, t0:t1] @ vv[:ns].T
        lse[:, t0:t1] = l
        delta[:, t0:t1] = (W * dP).sum(axis=-1)
    # dq rows: full key range for the sampled query rows
    M = attention_mask(t_rows, s_all, causal, sqb, skb, off)
    Wt, _ = masked_softmax(qh[:, t_rows] @ kk.T, M[None])
    dPt = dOh[:, t_rows] @ vv.T
    dSt = Wt * (dPt - delta[:, t_rows][..., None])
    dq = dSt @ kk                                                   # [G, nt, H]
    # dk / dv rows: all queries against the sampled keys
    M = attention_mask(np.arange(T), s_rows, causal, sqb, skb, off)  # [T, ns]
    L = qh @ kk[s_rows].T                                           # [G, T, ns]
    fin = np.isfinite(lse)[..., None]
    Ws = np.where(M[None] & fin, np.exp(L - np.where(fin, lse[..., None], 0.0)), 0.0)
    dPs = dOh @ vv[s_rows].T
    dSs = Ws * (dPs - delta[..., None])
    dk = np.einsum("gts,gth->sh", dSs, qh)
    dv = np.einsum("gts,gth->sh", Ws, dOh)
    return dq, dk, dv, lse, delta


def attention_bruteforce(q, k, v, dO=None, *, causal: bool = False,
                         seg_q=None, seg_kv=None, mask=None):
    """Pure-Python loops over every (b, kv_head, g, t, s, h); tiny shapes only.

    Returns (o, lse) and, when ``dO`` is given, also (dq, dk, dv)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    dOa = None if dO is None else _f64(dO)
    sq, skv = _i32(seg_q), _i32(seg_kv)
    B, K, G, T, H = q.shape
    S = k.shape[2]
    o = np.zeros((B, K, G, T, H))
    lse = np.full((B, K, G, T), NEG_INF)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for kh in range(K):
            for g in range(G):
                for t in range(T):
                    keep = []
                    for s in range(S):
                        ok = (not causal) or s <= t + (S - T)
                        if sq is not None:
                            ok = ok and sq[b, t] == skv[b, s]
                        if mask is not None:
                            mh = 0 if len(mask) == 1 else kh * G + g
                            ok = ok and bool(mask[mh][t][s])
                        if ok:
                            keep.append(s)
                    if not keep:
                        continue
                    logit = {}
                    for s in keep:
                        acc = 0.0
                        for h in range(H):
                            acc += float(q[b, kh, g, t, h]) * float(k[b, kh, s, h])
                        logit[s] = acc
                    mx = max(logit.values())
                    den = sum(math.exp(logit[s] - mx) for s in keep)
                    w = {s: math.exp(logit[s] - mx) / den for s in keep}
                    lse[b, kh, g, t] = mx + math.log(den)
                    for h in range(H):
                        o[b, kh, g, t, h] = sum(w[s] * float(v[b, kh, s, h]) for s in keep)
                    if dOa is None:
                        continue
                    dp = {s: sum(float(dOa[b, kh, g, t, h]) * float(v[b, kh, s, h])
                                 for h in range(H)) for s in keep}
                    dlt = sum(w[s] * dp[s] for s in keep)
                    for s in keep:
                        ds = w[s] * (dp[s] - dlt)
                        for h in range(H):
                            dq[b, kh, g, t, h] += ds * float(k[b, kh, s, h])
                            dk[b, kh, s, h] += ds * float(q[b, kh, g, t, h])
                            dv[b, kh, s, h] += w[s] * float(dOa[b, kh, g, t, h])
    if dOa is None:
        return o, lse
    return o, lse, dq, dk, dv
