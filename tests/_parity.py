"""Comparison helpers for the CUDA-vs-oracle parity tests.

Tolerances (the parity bar: codes and signs near-exact, dequantized rows within
1e-4 relative L2, attention within 2e-3 max-abs in fp32, plus the relative-L2 and
needle checks that keep the attention bar meaningful at long contexts):
  codes   bit-exact except where the oracle's rotated unit coordinate lies within
          CODE_WINDOW of a decision boundary; mismatch rate ≤ MAX_MISMATCH.
  signs   bit-exact except where |(S r)_i| / ‖S_i‖ < CODE_WINDOW (the residual's
          coordinate along the unit direction of S's row i, same unit-sphere
          scale as the codes), compared against the oracle's signs computed from
          the GPU's own codes; mismatch rate ≤ MAX_MISMATCH.
  norms   relative 1e-5 (‖x‖) and 1e-4 (‖r‖): float32 accumulation.
  dequant relative L2 ≤ 1e-4 per row.
  attn    max-abs ≤ 2e-3 and relative L2 ≤ 1e-3 (fp32 output).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O

CODE_WINDOW = 1e-5
MAX_MISMATCH = 1e-4
NORM_RTOL = 1e-5
RNORM_RTOL = 1e-4
DEQUANT_REL_L2 = 1e-4
ATTN_MAX_ABS = 2e-3
ATTN_REL_L2 = 1e-3


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def oracle_params(qz) -> O.Params:
    return O.make_params(qz.d, qz.bits, qz.variant, qz.seed, getattr(qz, "rotation", "qr"))


def boundary_margin(p: O.Params, y_unit: np.ndarray) -> np.ndarray:
    if p.bounds.size == 0:
        return np.full(y_unit.shape, np.inf)
    return np.min(np.abs(y_unit[..., None] - p.bounds[None, None, :]), axis=-1)


def check_quantize(p: O.Params, X: np.ndarray, planes: dict, rows=None, report: dict | None = None):
    """Compare GPU planes (all rows, or the given row indices) with the oracle on X[rows]."""
    sel = np.arange(X.shape[0]) if rows is None else np.asarray(rows)
    Xs = X[sel]
    ref = O.quantize(p, Xs)
    g_norm = to_np(planes["norm"])[sel].astype(np.float64)
    o_norm = ref["norm"].astype(np.float64)
    assert np.allclose(g_norm, o_norm, rtol=NORM_RTOL, atol=0), np.max(np.abs(g_norm - o_norm) / np.maximum(o_norm, 1e-30))
    if p.b_mse > 0:
        g_idx = O.unpack_codes(to_np(planes["codes"])[sel], p.d, p.b_mse)
        mism = g_idx != ref["idx"]
        margin = boundary_margin(p, ref["y_unit"])
        outside = mism & (margin >= CODE_WINDOW)
        assert not outside.any(), f"{outside.sum()} code mismatches outside the {CODE_WINDOW} window"
        rate = mism.mean()
        assert rate <= MAX_MISMATCH, f"code mismatch rate {rate}"
    else:
        g_idx = np.zeros_like(ref["idx"])
        rate = 0.0
    srate = 0.0
    if p.variant == "prod":
        ref2 = O.qjl_of_residual(p, Xs, g_idx)
        g_z = O.unpack_signs(to_np(planes["signs"])[sel], p.d)
        smism = g_z != ref2["z"]
        smargin = np.abs(ref2["sr"]) / np.linalg.norm(p.S, axis=1)[None, :]
        outside = smism & (smargin >= CODE_WINDOW)
        assert not outside.any(), f"{outside.sum()} sign mismatches outside the window"
        srate = smism.mean()
        assert srate <= MAX_MISMATCH, f"sign mismatch rate {srate}"
        g_rn = to_np(planes["rnorm"])[sel].astype(np.float64)
        o_rn = ref2["rnorm"].astype(np.float64)
        assert np.allclose(g_rn, o_rn, rtol=RNORM_RTOL, atol=1e-7)
    if report is not None:
        report.update(code_mismatch_rate=float(rate), sign_mismatch_rate=float(srate))
    return g_idx


def planes_to_oracle_rows(p: O.Params, planes: dict, rows=None) -> dict:
    """Unpack GPU planes into the oracle's row dict (idx, norm[, z, rnorm])."""
    def take(t):
        a = to_np(t)
        return a if rows is None else a[rows]
    out = {"idx": O.unpack_codes(take(planes["codes"]), p.d, p.b_mse) if p.b_mse > 0
           else np.zeros((len(take(planes["norm"])), p.d), dtype=np.int64),
           "norm": take(planes["norm"])}
    if p.variant == "prod":
        out["z"] = O.unpack_signs(take(planes["signs"]), p.d)
        out["rnorm"] = take(planes["rnorm"])
    return out


def check_dequant(p: O.Params, planes: dict, gpu_rows: torch.Tensor, rows=None):
    r = planes_to_oracle_rows(p, planes, rows)
    ref = O.dequantize(p, r["idx"], r["norm"], r.get("z"), r.get("rnorm"))
    g = f64(gpu_rows) if rows is None else f64(gpu_rows)[rows]
    num = np.linalg.norm(g - ref, axis=1)
    den = np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    rel = num / den
    zero = np.linalg.norm(ref, axis=1) == 0
    assert np.all(np.abs(g[zero]) == 0)
    assert np.max(rel[~zero], initial=0.0) <= DEQUANT_REL_L2, np.max(rel[~zero])
    return float(np.max(rel[~zero], initial=0.0))


def check_attention(gpu_out: np.ndarray, ref_out: np.ndarray):
    diff = np.abs(gpu_out - ref_out)
    mx = float(diff.max(initial=0.0))
    rel = float(np.linalg.norm(gpu_out - ref_out) / max(np.linalg.norm(ref_out), 1e-30))
    assert mx <= ATTN_MAX_ABS, mx
    assert rel <= ATTN_REL_L2 or np.linalg.norm(ref_out) == 0, rel
    return mx, rel
