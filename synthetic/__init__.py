"""Seeded synthetic inputs shared by the tests, the oracle runs and bench.py.

This module holds no TurboQuant arithmetic: it only draws random rows, queries
and sequence lengths with NumPy's ``default_rng`` and rounds them to the storage
dtype with PyTorch's CPU cast.  The pages measure on real Llama KV caches
(LongBench / Needle-in-a-Haystack); those models and datasets are not available,
so these shapes and distributions stand in for them.

The host generators return CPU ``torch`` tensors in the storage dtype; callers
copy them to the device for the CUDA path and call ``.double().numpy()`` for the
oracle, so both sides see bit-identical inputs.  The ``*_cuda`` generators draw
inputs too large for the host on the device; the oracle then reads sampled rows
of that same device tensor.
"""
from __future__ import annotations

import numpy as np
import torch

_DT = {"bf16": torch.bfloat16, "f32": torch.float32, "f16": torch.float16}


def _cast(a: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(_DT[dtype])


def gaussian(shape, seed: int, dtype: str = "bf16") -> torch.Tensor:
    """i.i.d. N(0,1)."""
    return _cast(np.random.default_rng(seed).standard_normal(shape, dtype=np.float32), dtype)


def gaussian_cuda(shape, seed: int, dtype=torch.bfloat16) -> torch.Tensor:
    """I.i.d. N(0, 1) drawn on the current CUDA device by a generator seeded with
    `seed` (for inputs too large to draw on the host; the oracle reads sampled
    rows of the same tensor)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randn(tuple(shape), generator=g, device="cuda", dtype=torch.float32).to(dtype)


def student_t_unit_var(shape, seed: int, nu: float = 4.0, dtype: str = "bf16") -> torch.Tensor:
    """Heavy-tailed rows: Student-t with ν degrees of freedom scaled to unit variance
    (variance of t_ν is ν/(ν−2), so ν=4 is scaled by 1/√2)."""
    a = np.random.default_rng(seed).standard_t(nu, size=shape).astype(np.float64)
    return _cast(a * np.sqrt((nu - 2.0) / nu), dtype)


def student_t_unit_var_cuda(shape, seed: int, nu: int = 4, dtype=torch.bfloat16) -> torch.Tensor:
    """Heavy-tailed rows drawn on the current CUDA device (for inputs too large to
    draw on the host): Student-t with an integer ν degrees of freedom as
    z / √(χ²_ν / ν), χ²_ν the sum of ν squared standard normals, scaled by
    √((ν − 2)/ν) to unit variance; every normal comes from one generator seeded
    with `seed`."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    z = torch.randn(tuple(shape), generator=g, device="cuda", dtype=torch.float32)
    chi2 = torch.zeros_like(z)
    for _ in range(int(nu)):
        e = torch.randn(tuple(shape), generator=g, device="cuda", dtype=torch.float32)
        chi2.addcmul_(e, e)
    t = z * torch.rsqrt(chi2 / nu) * float(np.sqrt((nu - 2.0) / nu))
    return t.to(dtype)


def outlier_channels(d: int, count: int, seed: int) -> np.ndarray:
    """``count`` distinct channel indices in [0, d), the same for every head."""
    return np.sort(np.random.default_rng(seed).choice(d, size=count, replace=False))


def kv_with_outliers(heads: int, tokens: int, d: int, seed: int, channels, factor: float = 10.0,
                     dtype: str = "bf16") -> torch.Tensor:
    """[heads, tokens, d] N(0,1) with the given channels multiplied by ``factor``."""
    a = np.random.default_rng(seed).standard_normal((heads, tokens, d), dtype=np.float32)
    a[..., channels] *= factor
    return _cast(a, dtype)


def seq_lens_uniform(batch: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """Per-sequence lengths uniform on the integers [lo, hi]."""
    return torch.from_numpy(np.random.default_rng(seed).integers(lo, hi + 1, size=batch).astype(np.int32))


def unit_rows(n: int, d: int, seed: int) -> np.ndarray:
    """Rows uniform on the unit sphere (float64), for distortion statistics."""
    a = np.random.default_rng(seed).standard_normal((n, d))
    return a / np.linalg.norm(a, axis=1, keepdims=True)


def plant_needles(keys: torch.Tensor, q: torch.Tensor, positions, strength: float, group: int) -> torch.Tensor:
    """Return a copy of ``keys`` [B, Hkv, T, d] in which, for every (b, kv head), the
    rows at ``positions`` are replaced by ``strength`` times the unit direction of
    the first query head of that group (q is [B, Hq, d]).  Makes the softmax peak."""
    k = keys.clone().float()
    B, Hkv, T, d = k.shape
    qf = q.float()
    for b in range(B):
        for h in range(Hkv):
            u = qf[b, h * group]
            u = u / u.norm()
            for t in positions:
                if t < T:
                    k[b, h, t] = strength * u
    return k.to(keys.dtype)


# ---------------------------------------------------------------------------
# The five workload shapes (sizes as stated for each; dtype of the stored rows)
# ---------------------------------------------------------------------------
WORKLOADS = {
    "small_mse_b2": dict(d=128, rows=4096, queries=64, bits=2, variant="mse", dtype="f32"),
    "llama70b_layer_kv_quant": dict(heads=8, tokens=32768, d=128, bits=3, variant="mse",
                                    outliers=4, outlier_factor=10.0, hq=64, dtype="bf16"),
    "decode_131k": dict(B=1, Hq=64, Hkv=8, d=128, T=131072, k_bits=3, k_variant="prod",
                        v_bits=3, v_variant="mse", dtype="bf16"),
    "batched_decode_32k": dict(B=16, Hq=32, Hkv=8, d=128, T=32768, lo=8192, k_bits=4, k_variant="prod",
                               v_bits=2, v_variant="mse", dtype="bf16"),
    "sweep": dict(rows=1 << 20, bits=(1, 2, 3, 4), variants=("mse", "prod"), d=(64, 128, 256),
                  queries=1024, dtype="bf16"),
}
