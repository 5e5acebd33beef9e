"""Shared comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (stated for the method's bf16-in / fp32-accumulate arithmetic):
  O        max |err| <= 2e-2 and relative Frobenius error <= 5e-3
  lse      max |err| <= 1e-3 (natural-log units; -inf must match exactly)
  dq/dk/dv relative Frobenius error <= 1e-2
"""
import numpy as np
import torch

O_MAX_ABS = 2e-2
O_REL_FRO = 5e-3
LSE_ABS = 1e-3
GRAD_REL_FRO = 1e-2


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_fro(a: np.ndarray, r: np.ndarray) -> float:
    den = np.linalg.norm(r)
    num = np.linalg.norm(a - r)
    if den == 0:
        return float(num)
    return float(num / den)


def check_o(o_gpu: np.ndarray, o_ref: np.ndarray, what: str = "O"):
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite values"
    err = float(np.max(np.abs(o_gpu - o_ref))) if o_ref.size else 0.0
    rf = rel_fro(o_gpu, o_ref)
    assert err <= O_MAX_ABS, f"{what}: max abs err {err:.3e} > {O_MAX_ABS}"
    assert rf <= O_REL_FRO, f"{what}: rel Frobenius err {rf:.3e} > {O_REL_FRO}"
    return err, rf


def check_lse(l_gpu: np.ndarray, l_ref: np.ndarray):
    inf_g, inf_r = np.isneginf(l_gpu), np.isneginf(l_ref)
    assert np.array_equal(inf_g, inf_r), "lse: -inf rows differ"
    fin = ~inf_r
    assert np.all(np.isfinite(l_gpu[fin])), "lse: non-finite values"
    err = float(np.max(np.abs(l_gpu[fin] - l_ref[fin]))) if fin.any() else 0.0
    assert err <= LSE_ABS, f"lse: max abs err {err:.3e} > {LSE_ABS}"
    return err


def check_grad(g_gpu: np.ndarray, g_ref: np.ndarray, what: str):
    assert np.all(np.isfinite(g_gpu)), f"{what}: non-finite values"
    rf = rel_fro(g_gpu, g_ref)
    assert rf <= GRAD_REL_FRO, f"{what}: rel Frobenius err {rf:.3e} > {GRAD_REL_FRO}"
    return rf
