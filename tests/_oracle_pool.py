"""Runs the fp64 oracle on independent units of a full-size workload in spawned
worker processes and compares each unit with the GPU's results there, so only
error sums travel back.  A unit is one (batch row, kv head) for the full
checks, or one head's sampled rows / one kv head's sampled keys for the
32768-key workload.

Workers are started with ``spawn`` (never forked from a process that has used
CUDA) and import only numpy and the oracle.  Each gets an equal share of the
host's cores for its BLAS threads."""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np

_BLAS_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def err_sums(g: np.ndarray, r: np.ndarray) -> dict:
    """max |g - r|, sum (g - r)^2 and sum r^2 (finite entries of r only for
    lse, where -inf rows must match exactly)."""
    g = np.asarray(g, dtype=np.float64).ravel()
    r = np.asarray(r, dtype=np.float64).ravel()
    assert g.shape == r.shape, (g.shape, r.shape)
    fin = np.isfinite(r)
    gf, rf = g[fin], r[fin]
    ok = np.isfinite(gf)
    d = gf[ok] - rf[ok]
    return {"inf_mismatch": int(np.count_nonzero(np.isfinite(g) != fin)),
            "nonfinite_gpu": int(np.count_nonzero(~ok)),
            "max_abs": float(np.max(np.abs(d))) if d.size else 0.0,
            "num2": float(np.dot(d, d)), "den2": float(np.dot(rf, rf)), "n": int(g.size)}


def merge(parts: list[dict]) -> dict:
    out = {"inf_mismatch": 0, "nonfinite_gpu": 0, "max_abs": 0.0, "num2": 0.0, "den2": 0.0, "n": 0}
    for p in parts:
        for key in ("inf_mismatch", "nonfinite_gpu", "num2", "den2", "n"):
            out[key] += p[key]
        out["max_abs"] = max(out["max_abs"], p["max_abs"])
    out["rel_fro"] = float(np.sqrt(out["num2"] / out["den2"])) if out["den2"] > 0 else 0.0
    return out


# ------------------------------------------------------------------ units

def full_unit(job: dict) -> dict:
    """Every element of one (b, kv head): O and lse (job["part"] == "fwd") or
    dq, dk and dv (job["part"] == "bwd").

    Inputs are the unit's slices as [1, 1, G, T, H] / [1, 1, S, H] float32
    arrays (bf16 values, exact) and [1, T] / [1, S] segment ids; job["window"]
    (T, S, window), if given, adds a causal sliding-window mask."""
    import oracle
    kw = dict(causal=job["causal"], seg_q=job["seg_q"], seg_kv=job["seg_kv"], row_block=256)
    if job.get("window"):
        # causal sliding window t - window < s <= t + (S - T), as a dense [1, T, S]
        # keep-mask (a layout: which pairs exist)
        T, S, window = job["window"]
        t = np.arange(T)[:, None]
        s = np.arange(S)[None, :]
        kw["mask"] = ((s <= t + (S - T)) & (s > t + (S - T) - window))[None]
    if job["part"] == "fwd":
        o, lse = oracle.attention_forward(job["q"], job["k"], job["v"], **kw)
        return {"o": err_sums(job["o_gpu"], o), "lse": err_sums(job["lse_gpu"], lse)}
    dq, dk, dv = oracle.attention_backward(job["q"], job["k"], job["v"], job["dO"], **kw)
    return {"dq": err_sums(job["dq_gpu"], dq), "dk": err_sums(job["dk_gpu"], dk),
            "dv": err_sums(job["dv_gpu"], dv)}


def rows_unit(job: dict) -> dict:
    """O and lse at the listed query rows of one (b, kv head, g), in chunks."""
    import oracle
    rows = np.asarray(job["rows"])
    o_parts, l_parts = [], []
    for i in range(0, len(rows), 256):
        o, lse = oracle.attention_rows(job["q"], job["k"], job["v"], 0, 0, 0, rows[i:i + 256],
                                       causal=job["causal"], seg_q=job["seg_q"],
                                       seg_kv=job["seg_kv"])
        o_parts.append(o)
        l_parts.append(lse)
    return {"o": err_sums(job["o_gpu"], np.concatenate(o_parts)),
            "lse": err_sums(job["lse_gpu"], np.concatenate(l_parts))}


def keys_unit(job: dict) -> dict:
    """dq at sampled query rows and dk, dv at the listed key rows of one
    (b, kv head)."""
    import oracle
    dq, dk, dv, _, _ = oracle.attention_backward_rows(
        job["q"], job["k"], job["v"], job["dO"], 0, 0, t_rows=job["t_rows"],
        s_rows=job["s_rows"], causal=job["causal"], seg_q=job["seg_q"], seg_kv=job["seg_kv"],
        row_block=128)
    return {"dq": err_sums(job["dq_gpu"], dq), "dk": err_sums(job["dk_gpu"], dk),
            "dv": err_sums(job["dv_gpu"], dv)}


def run(fn, jobs: list[dict], max_workers: int | None = None) -> list[dict]:
    """fn over jobs in spawned workers; each worker's BLAS pool gets
    cores / workers threads."""
    cores = os.cpu_count() or 1
    n = max(1, min(len(jobs), max_workers or cores))
    saved = {k: os.environ.get(k) for k in _BLAS_VARS}
    for k in _BLAS_VARS:
        os.environ[k] = str(max(1, cores // n))
    try:
        with ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn")) as ex:
            return list(ex.map(fn, jobs))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
