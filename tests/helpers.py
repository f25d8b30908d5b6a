"""Shared test helpers: build-once fixture logic and comparison utilities."""

import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cpattn.h")

# Tolerances for floating point parity (max-abs), from the stated acceptance bars.
TOL_F32 = 1e-5
TOL_BF16_O = 2e-2
TOL_BF16_LSE = 1e-3


def ensure_built():
    from context_blockwise_attention_gb300 import build as b
    if not os.path.exists(b.LIB):
        b.build()
    return b.LIB


def header_functions():
    """Names of the functions declared in include/cpattn.h."""
    with open(HEADER) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cp_[a-z_0-9]+)\s*\(", src)))


def max_abs(a, b, mask=None):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if mask is not None:
        a = a[mask]
        b = b[mask]
    if a.size == 0:
        return 0.0
    return float(np.abs(a - b).max())


def compare_partial(o_gpu, l_gpu, o_ref, l_ref, tol_o, tol_l, what=""):
    """O and LSE parity; rows with no visible key must be exactly O=0, LSE=-inf."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    l_gpu = np.asarray(l_gpu, dtype=np.float64)
    empty = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(l_gpu), empty), f"{what}: empty-row pattern differs"
    assert np.all(o_gpu[empty] == 0.0), f"{what}: empty rows must have O = 0"
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    eo = max_abs(o_gpu, o_ref)
    el = max_abs(l_gpu, l_ref, ~empty)
    assert eo <= tol_o, f"{what}: max|dO| = {eo:.3e} > {tol_o}"
    assert el <= tol_l, f"{what}: max|dLSE| = {el:.3e} > {tol_l}"
    return eo, el


# Gradients (backward pass): max-abs error relative to the tensor's own scale, max(1, max|ref|).
# fp32 inputs: fp32 accumulation only.  bf16 inputs: P and dS are rounded to bf16 (relative
# 2^-9 each) before the dV, dK and dQ products.
TOL_GRAD_F32 = 1e-5
TOL_GRAD_BF16 = 1e-2
# bf16 inputs, also per row: every gradient row (one token and head, all D columns) is checked
# against its own scale, max|ref row|, so an error in a row far smaller than the tensor's peak
# cannot hide under the tensor-wide bound.  The rounding of P and dS bounds a row's error by 2^-9
# of the magnitudes of the terms it sums, not of its value: a row whose terms cancel (a causal
# query's first keys, where sum_j dS_ij = 0 holds with few terms) can be far below them, so rows
# below 1e-2 of the tensor's scale are held to that floor (1e-4 of the tensor's scale).
# Observed worst over the parity cases: 4.3e-3.
TOL_GRAD_BF16_ROW = 1e-2
ROW_FLOOR = 1e-2


def compare_grad(g_gpu, g_ref, tol, what="", rows=True):
    g_gpu = np.asarray(g_gpu, dtype=np.float64)
    g_ref = np.asarray(g_ref, dtype=np.float64)
    assert g_gpu.shape == g_ref.shape, f"{what}: shape {g_gpu.shape} != {g_ref.shape}"
    assert np.all(np.isfinite(g_gpu)), f"{what}: non-finite gradient"
    scale = max(1.0, float(np.abs(g_ref).max()) if g_ref.size else 1.0)
    err = float(np.abs(g_gpu - g_ref).max()) / scale if g_ref.size else 0.0
    assert err <= tol, f"{what}: max|err|/scale = {err:.3e} > {tol} (scale {scale:.3g})"
    if rows and tol == TOL_GRAD_BF16 and g_ref.size:
        rows_err = np.abs(g_gpu - g_ref).max(axis=-1)
        rows_scale = np.maximum(np.abs(g_ref).max(axis=-1), ROW_FLOOR * float(np.abs(g_ref).max()))
        live = rows_scale > 0
        rel = float((rows_err[live] / rows_scale[live]).max()) if live.any() else 0.0
        assert np.all(rows_err[~live] == 0.0), f"{what}: rows with a zero reference must be exactly zero"
        assert rel <= TOL_GRAD_BF16_ROW, f"{what}: worst row max|err|/max|ref row| = {rel:.3e} > {TOL_GRAD_BF16_ROW}"
    return err

