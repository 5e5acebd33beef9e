"""Seeded synthetic workloads for blocked GQA flash attention.

This module only draws random numbers and builds segment-id layouts.  It holds
none of the attention arithmetic, so both the CPU oracle (through the tests)
and the CUDA path can be fed from it without sharing any of the method.

Tensor layout (notation of "Notation" on the flash-attention tutorial page,
danielwatson6.github.io/fa/fa.html):
  q  [B, K, G, T, H]  pre-scaled by H**-0.5, rounded to bf16 once
  k  [B, K, S, H]
  v  [B, K, S, H]
  dO [B, K, G, T, H]  (backward workloads only)
  seg_q [B, T], seg_kv [B, S] int32 (packed-sequence workload only)

Recipe: a CPU ``torch.Generator`` seeded with ``seed`` draws fp32 N(0, 1)
tensors in the order q, k, v, dO; q is multiplied by H**-0.5 in fp32 and every
tensor is rounded to bf16 exactly once.  Document lengths for the packed
workload come from ``numpy.random.default_rng(seed)``: for each batch row in
turn, integer lengths uniform on [lo, hi] are drawn until they cover the row,
the last one truncated; ids count 0, 1, 2, ... within a row.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    K: int
    G: int
    T: int
    S: int
    H: int
    causal: bool
    segments: bool = False
    backward: bool = True
    seed: int = 0
    doc_len: tuple = (128, 2048)
    kind: str = "dense"      # "dense", "decode" (split-KV forward) or "window" (block-sparse)
    window: int = 0          # "window": keys t - window < s <= t (with causal)

    @property
    def scale(self) -> float:
        return float(self.H) ** -0.5


# The five workloads the method is measured on.  The three long causal ones are
# model_dim 4096 / 16 query heads / 2 kv heads (the axlearn TPU flash-attention
# benchmark shape) and the packed-document mix.
WORKLOADS = {
    "gqa_h64_t128_fwd": Workload("gqa_h64_t128_fwd", 1, 1, 4, 128, 128, 64,
                                 causal=False, backward=False),
    "gqa_causal_h128_t1024": Workload("gqa_causal_h128_t1024", 2, 2, 4, 1024,
                                      1024, 128, causal=True),
    "gqa_causal_h256_t8192": Workload("gqa_causal_h256_t8192", 1, 2, 8, 8192,
                                      8192, 256, causal=True),
    "gqa_causal_h256_t32768": Workload("gqa_causal_h256_t32768", 1, 2, 8,
                                       32768, 32768, 256, causal=True),
    "gqa_packed_docs_h128_t4096": Workload("gqa_packed_docs_h128_t4096", 4, 8,
                                           4, 4096, 4096, 128, causal=True,
                                           segments=True),
    # One decode step (T = 1) against a 32k-key cache: memory-bound.
    "gqa_decode_h128_s32768": Workload("gqa_decode_h128_s32768", 8, 8, 8, 1, 32768, 128,
                                       causal=True, backward=False, kind="decode"),
    # Causal sliding window of 1024 keys given as a block-sparse mask.
    "gqa_window1024_h128_t8192": Workload("gqa_window1024_h128_t8192", 1, 8, 4, 8192, 8192,
                                          128, causal=True, kind="window", window=1024),
}


def window_mask(T: int, S: int, window: int) -> np.ndarray:
    """Dense [1, T, S] keep-mask of a causal sliding window: t - window < s <= t + (S - T).

    A mask *layout* (which pairs exist), not attention arithmetic."""
    off = S - T
    t = np.arange(T)[:, None]
    s = np.arange(S)[None, :]
    return ((s <= t + off) & (s > t + off - window))[None]


def document_segment_ids(batch: int, length: int, seed: int,
                         lo: int = 128, hi: int = 2048) -> np.ndarray:
    """Consecutive documents per row, lengths uniform on [lo, hi] (inclusive),
    the last one truncated at ``length``.  Returns int32 [batch, length]."""
    rng = np.random.default_rng(seed)
    ids = np.empty((batch, length), dtype=np.int32)
    for b in range(batch):
        pos, doc = 0, 0
        while pos < length:
            n = int(rng.integers(lo, hi + 1))
            ids[b, pos:pos + n] = doc
            pos += n
            doc += 1
    return ids


def random_segment_ids(batch: int, length: int, n_ids: int, seed: int,
                       sorted_runs: bool = False) -> np.ndarray:
    """Arbitrary (non-monotone unless ``sorted_runs``) int32 ids in [0, n_ids)."""
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, n_ids, size=(batch, length)).astype(np.int32)
    if sorted_runs:
        ids = np.sort(ids, axis=1)
    return ids


@dataclasses.dataclass
class Tensors:
    """bf16 CPU tensors of one workload plus optional int32 segment ids."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    dO: Optional[torch.Tensor]
    seg_q: Optional[torch.Tensor]
    seg_kv: Optional[torch.Tensor]

    def f64(self, name: str) -> np.ndarray:
        """Exact fp64 copy of a bf16 tensor (bf16 -> fp32 -> fp64 is exact)."""
        t = getattr(self, name)
        return t.float().numpy().astype(np.float64)


def make_tensors(B: int, K: int, G: int, T: int, S: int, H: int, *,
                 seed: int = 0, backward: bool = True,
                 seg_q: Optional[np.ndarray] = None,
                 seg_kv: Optional[np.ndarray] = None,
                 scale: Optional[float] = None) -> Tensors:
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    sc = float(H) ** -0.5 if scale is None else scale
    q = torch.randn((B, K, G, T, H), generator=gen, dtype=torch.float32)
    q = (q * sc).to(torch.bfloat16)
    k = torch.randn((B, K, S, H), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((B, K, S, H), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    dO = None
    if backward:
        dO = torch.randn((B, K, G, T, H), generator=gen,
                         dtype=torch.float32).to(torch.bfloat16)
    sq = None if seg_q is None else torch.from_numpy(np.ascontiguousarray(seg_q, dtype=np.int32))
    skv = None if seg_kv is None else torch.from_numpy(np.ascontiguousarray(seg_kv, dtype=np.int32))
    return Tensors(q, k, v, dO, sq, skv)


def make_workload(w: Workload) -> Tensors:
    seg = None
    if w.segments:
        seg = document_segment_ids(w.B, w.T, w.seed, *w.doc_len)
    return make_tensors(w.B, w.K, w.G, w.T, w.S, w.H, seed=w.seed,
                        backward=w.backward, seg_q=seg, seg_kv=seg)


def unmasked_pairs(T: int, S: int, causal: bool,
                   seg_q: Optional[np.ndarray], seg_kv: Optional[np.ndarray],
                   B: int = 1) -> int:
    """Number of (b, t, s) query/key pairs the mask keeps, summed over batch.

    This is bookkeeping for FLOP accounting (the mask-adjusted FLOP count),
    computed by counting, not by the attention arithmetic."""
    off = S - T
    if seg_q is None:
        if causal:
            # keep s <= t + (S - T): queries aligned to the end of the keys
            per = sum(max(0, min(t + off + 1, S)) for t in range(T))
        else:
            per = T * S
        return per * B
    total = 0
    for b in range(seg_q.shape[0]):
        sq, sk = seg_q[b], seg_kv[b]
        ids = np.union1d(sq, sk)
        for i in ids:
            tq = np.nonzero(sq == i)[0]
            ts = np.nonzero(sk == i)[0]
            if causal:
                total += int(np.searchsorted(ts, tq + off, side="right").sum())
            else:
                total += len(tq) * len(ts)
    return total
