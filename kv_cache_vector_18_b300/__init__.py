"""TurboQuant KV-cache codec and compressed-cache decode attention on B300.

Thin Python binding over the C ABI of ``libtq.so`` (include/tq.h).  It only
marshals arguments: every step of quantization, dequantization and attention
runs in the library's CUDA kernels.  PyTorch provides device memory and streams.
There is no CPU fallback: without the built library, importing the compute
entry points raises ImportError.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
import torch

from . import _lib
from ._lib import TQ_BF16, TQ_F32, TQ_MSE, TQ_PROD, TQError, check

__all__ = ["Quantizer", "MixedQuantizer", "quantize_kv", "mixed_quantize_kv", "decode_attention", "decode_append_attention", "mixed_decode_attention",
           "mixed_decode_workspace_bytes", "select_outlier_channels", "decode_workspace_bytes", "build_params_host", "TQError",
           "library_path"]

_VARIANTS = {"mse": TQ_MSE, "prod": TQ_PROD}
_ROTATIONS = {"qr": _lib.TQ_ROT_QR, "hadamard": _lib.TQ_ROT_HADAMARD}
_DTYPES = {torch.bfloat16: TQ_BF16, torch.float32: TQ_F32}


def library_path() -> str:
    return _lib.LIB_PATH


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


try:  # the raw current-stream handle without building a torch.cuda.Stream object
    _raw_stream = torch._C._cuda_getCurrentRawStream
    _cur_device = torch._C._cuda_getDevice
except AttributeError:  # pragma: no cover - older torch
    _raw_stream = None


def _stream(stream) -> int | None:
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(_cur_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def build_params_host(d: int, bits: int, variant: str = "mse", seed: int = 0, rotation: str = "qr") -> dict:
    """Float64 Π, S, centroids and boundaries exactly as tq_init_ex builds them (host only, no GPU)."""
    L = _lib.lib()
    b_m = bits if variant == "mse" else bits - 1
    Pi = np.zeros(d * d)
    S = np.zeros(d * d)
    c = np.zeros(1 << b_m)
    t = np.zeros(max((1 << b_m) - 1, 1))
    dp = ctypes.POINTER(ctypes.c_double)
    check(L.tq_build_params_host_ex(d, bits, _VARIANTS[variant], _ROTATIONS[rotation], seed, Pi.ctypes.data_as(dp),
                                    S.ctypes.data_as(dp), c.ctypes.data_as(dp), t.ctypes.data_as(dp)))
    out = {"Pi": Pi.reshape(d, d), "centroids": c, "bounds": t[: (1 << b_m) - 1]}
    if variant == "prod":
        out["S"] = S.reshape(d, d)
    return out


class Quantizer:
    """One TurboQuant quantizer (tq_init_ex handle) on the current CUDA device.

    rotation: "qr" (Π from the QR factor of a Gaussian matrix) or "hadamard"
    (randomised Walsh–Hadamard, d a power of two).
    """

    def __init__(self, d: int, bits: int, variant: str = "mse", seed: int = 0, rotation: str = "qr"):
        L = _lib.lib()
        h = ctypes.c_void_p()
        check(L.tq_init_ex(d, bits, _VARIANTS[variant], _ROTATIONS[rotation], seed, ctypes.byref(h)))
        self._h = h
        self.d, self.bits, self.variant, self.seed, self.rotation = d, bits, variant, seed, rotation
        self.b_mse = bits if variant == "mse" else bits - 1
        cb, sb = ctypes.c_int(), ctypes.c_int()
        check(L.tq_row_bytes(h, ctypes.byref(cb), ctypes.byref(sb)))
        self.code_bytes, self.sign_bytes = cb.value, sb.value
        self.device = torch.cuda.current_device()

    @property
    def handle(self) -> ctypes.c_void_p:
        return self._h

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.lib().tq_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def params(self) -> dict:
        d, lv = self.d, 1 << self.b_mse
        Pi, S, c, t = np.zeros(d * d), np.zeros(d * d), np.zeros(lv), np.zeros(max(lv - 1, 1))
        dp = ctypes.POINTER(ctypes.c_double)
        check(_lib.lib().tq_get_params(self._h, Pi.ctypes.data_as(dp), S.ctypes.data_as(dp),
                                       c.ctypes.data_as(dp), t.ctypes.data_as(dp)))
        out = {"Pi": Pi.reshape(d, d), "centroids": c, "bounds": t[: lv - 1]}
        if self.variant == "prod":
            out["S"] = S.reshape(d, d)
        return out

    def device_status(self, clear: bool = True) -> int:
        """Non-zero when a kernel pipeline wait timed out since the last clear."""
        st = ctypes.c_int()
        check(_lib.lib().tq_device_status(self._h, ctypes.byref(st), int(clear)))
        return st.value

    def check_wait_timeout(self, code: int, limit_ns: int, stream=None) -> None:
        """Enqueue a block whose bounded wait expires and records `code` (tq_check_wait_timeout)."""
        check(_lib.lib().tq_check_wait_timeout(self._h, int(code), int(limit_ns), _stream(stream)))

    def empty_planes(self, n_rows: int, device=None) -> dict:
        """Allocate packed planes for n_rows rows (see include/tq.h for the layout)."""
        dev = device if device is not None else torch.device("cuda", self.device)
        p = {"codes": torch.empty((n_rows, self.code_bytes), dtype=torch.uint8, device=dev),
             "norm": torch.empty((n_rows,), dtype=torch.float32, device=dev)}
        if self.variant == "prod":
            p["signs"] = torch.empty((n_rows, self.sign_bytes), dtype=torch.uint8, device=dev)
            p["rnorm"] = torch.empty((n_rows,), dtype=torch.float32, device=dev)
        return p

    @staticmethod
    def planes_struct(p: dict) -> _lib.Planes:
        return _lib.Planes(_ptr(p.get("codes")) if p.get("codes") is not None and p["codes"].numel() else None,
                           _ptr(p.get("signs")), _ptr(p.get("norm")), _ptr(p.get("rnorm")))

    def quantize(self, x: torch.Tensor, out: dict | None = None, stream=None) -> dict:
        """tq_quantize over the rows of x ([..., d], bf16 or fp32, on the device)."""
        if x.dim() < 2:
            raise ValueError("x must have shape [..., d]")
        x2 = x.reshape(-1, x.shape[-1])
        n = x2.shape[0]
        if out is None:
            out = self.empty_planes(n, x.device)
        if n == 0:
            return out
        if x2.stride(-1) != 1:
            raise ValueError("x rows must be contiguous")
        check(_lib.lib().tq_quantize(self._h, _ptr(x2), _DTYPES[x.dtype], n, x2.stride(0),
                                     self.planes_struct(out), _stream(stream)))
        return out

    def dequantize(self, planes: dict, n_rows: int | None = None, dtype=torch.float32, stream=None) -> torch.Tensor:
        n = planes["norm"].shape[0] if n_rows is None else n_rows
        y = torch.empty((n, self.d), dtype=dtype, device=planes["norm"].device)
        check(_lib.lib().tq_dequantize(self._h, self.planes_struct(planes), n, _ptr(y), _DTYPES[dtype],
                                       _stream(stream)))
        return y


def quantize_kv(kq: Quantizer, vq: Quantizer, k: torch.Tensor, v: torch.Tensor, k_out: dict | None = None,
                v_out: dict | None = None, stream=None) -> tuple[dict, dict]:
    """tq_quantize_kv: the rows of k with kq and the rows of v with vq in one call
    (one launch when both are mse with the same d, b and rotation kind).  k and v
    are [..., d] with the same dtype (bf16 or fp32) on the device."""
    if k.dtype != v.dtype:
        raise ValueError("k and v must have the same dtype")
    k2, v2 = k.reshape(-1, k.shape[-1]), v.reshape(-1, v.shape[-1])
    nk, nv = k2.shape[0], v2.shape[0]
    k_out = kq.empty_planes(nk, k.device) if k_out is None else k_out
    v_out = vq.empty_planes(nv, v.device) if v_out is None else v_out
    if (nk and k2.stride(-1) != 1) or (nv and v2.stride(-1) != 1):
        raise ValueError("k and v rows must be contiguous")
    check(_lib.lib().tq_quantize_kv(kq.handle, vq.handle, _ptr(k2) if nk else None, _ptr(v2) if nv else None,
                                    _DTYPES[k.dtype], nk, nv, k2.stride(0) if nk else kq.d,
                                    v2.stride(0) if nv else vq.d, Quantizer.planes_struct(k_out),
                                    Quantizer.planes_struct(v_out), _stream(stream)))
    return k_out, v_out


def decode_workspace_bytes(kq: Quantizer, vq: Quantizer, B: int, Hq: int, Hkv: int, T_max: int) -> int:
    n = ctypes.c_size_t()
    check(_lib.lib().tq_decode_workspace_bytes(kq.handle, vq.handle, B, Hq, Hkv, T_max, ctypes.byref(n)))
    return n.value


def decode_attention(kq: Quantizer, vq: Quantizer, q: torch.Tensor, kcache: dict, vcache: dict,
                     seq_lens: torch.Tensor, Hkv: int, T_max: int, scale: float | None = None,
                     return_scores: bool = False, workspace: torch.Tensor | None = None,
                     out: torch.Tensor | None = None, stream=None):
    """tq_decode_attention.  q: [B, Hq, d] (bf16/fp32), caches hold B·Hkv·T_max rows
    ordered [B][Hkv][T_max], seq_lens: int32 [B] on the device.  Returns out
    [B, Hq, d] fp32 (and the pre-softmax scores [B, Hq, T_max] when asked)."""
    B, Hq, d = q.shape
    if not q.is_contiguous():
        raise ValueError("q must be contiguous")
    if seq_lens.dtype != torch.int32:
        raise ValueError("seq_lens must be int32")
    if workspace is None:  # a caller-provided workspace is size-checked by the library
        need = decode_workspace_bytes(kq, vq, B, Hq, Hkv, T_max)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    scores = torch.full((B, Hq, T_max), float("nan"), dtype=torch.float32, device=q.device) if return_scores else None
    check(_lib.lib().tq_decode_attention(
        kq.handle, vq.handle, _ptr(q), _DTYPES[q.dtype], Quantizer.planes_struct(kcache),
        Quantizer.planes_struct(vcache), _ptr(seq_lens), B, Hq, Hkv, T_max,
        float(scale) if scale is not None else 0.0, _ptr(out), _ptr(scores), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return (out, scores) if return_scores else out


def decode_append_attention(kq: Quantizer, vq: Quantizer, q: torch.Tensor, k_new: torch.Tensor,
                            v_new: torch.Tensor, kcache: dict, vcache: dict, seq_lens: torch.Tensor, Hkv: int,
                            T_max: int, scale: float | None = None, workspace: torch.Tensor | None = None,
                            out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """tq_decode_append_attention.  k_new, v_new: [B, Hkv, d] (bf16/fp32, same dtype)
    appended at token seq_lens[b] of each (b, KV head) slab; seq_lens (int32 [B] on
    the device) is incremented in place; returns out [B, Hq, d] fp32 over the
    updated cache."""
    B, Hq, d = q.shape
    for name, t in (("q", q), ("k_new", k_new), ("v_new", v_new)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if k_new.shape != (B, Hkv, d) or v_new.shape != (B, Hkv, d) or k_new.dtype != v_new.dtype:
        raise ValueError("k_new and v_new must both be [B, Hkv, d] of one dtype")
    if seq_lens.dtype != torch.int32:
        raise ValueError("seq_lens must be int32")
    if workspace is None:  # a caller-provided workspace is size-checked by the library
        need = decode_workspace_bytes(kq, vq, B, Hq, Hkv, T_max)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    check(_lib.lib().tq_decode_append_attention(
        kq.handle, vq.handle, _ptr(q), _DTYPES[q.dtype], _ptr(k_new), _ptr(v_new), _DTYPES[k_new.dtype],
        Quantizer.planes_struct(kcache), Quantizer.planes_struct(vcache), _ptr(seq_lens), B, Hq, Hkv, T_max,
        float(scale) if scale is not None else 0.0, _ptr(out), _ptr(workspace), workspace.numel(),
        _stream(stream)))
    return out


def select_outlier_channels(x: torch.Tensor, d_o: int, stream=None):
    """tq_select_outlier_channels.  x: [n, d] (bf16/fp32, unit stride along d).
    Returns (perm int32 [d]: the d_o channels of largest energy ascending, then the
    rest ascending; energy float64 [d])."""
    n, d = x.shape
    if x.stride(1) != 1:
        raise ValueError("x must have unit stride along channels")
    perm = torch.empty(d, dtype=torch.int32, device=x.device)
    energy = torch.empty(d, dtype=torch.float64, device=x.device)
    check(_lib.lib().tq_select_outlier_channels(_ptr(x), _DTYPES[x.dtype], n, x.stride(0), d, d_o, _ptr(energy),
                                                _ptr(perm), _stream(stream)))
    return perm, energy


class MixedQuantizer:
    """Outlier-channel mixed precision: channels perm[:d_o] quantized by one handle
    (bits_o), the others by a second (bits_n), both of one variant; perm is an
    int32 permutation of range(d) on the device.  Planes come as {"o": …, "n": …}."""

    def __init__(self, perm: torch.Tensor, d_o: int, bits_o: int, bits_n: int, variant: str = "mse",
                 seed_o: int = 0, seed_n: int = 1, rotation: str = "qr"):
        if perm.dtype != torch.int32 or perm.dim() != 1 or not perm.is_cuda:
            raise ValueError("perm must be a 1-D int32 CUDA tensor")
        self.d = perm.numel()
        self.perm = perm.contiguous()
        self.qo = Quantizer(d_o, bits_o, variant, seed=seed_o, rotation=rotation)
        self.qn = Quantizer(self.d - d_o, bits_n, variant, seed=seed_n, rotation=rotation)
        self.d_o, self.variant = d_o, variant
        # scratch for the combined rotation operand of the tensor-core path (room
        # for two, so mixed_quantize_kv can put keys and values in one launch)
        self.scratch = torch.empty(2 * _lib.lib().tq_mixed_quantize_scratch_bytes(), dtype=torch.uint8,
                                   device=self.perm.device)

    def empty_planes(self, n_rows: int) -> dict:
        return {"o": self.qo.empty_planes(n_rows), "n": self.qn.empty_planes(n_rows)}

    def quantize(self, x: torch.Tensor, out: dict | None = None, stream=None) -> dict:
        n, d = x.shape
        if d != self.d or x.stride(1) != 1:
            raise ValueError("x must be [n, d] with unit stride along channels")
        out = out if out is not None else self.empty_planes(n)
        check(_lib.lib().tq_mixed_quantize(self.qo.handle, self.qn.handle, _ptr(self.perm), _ptr(x),
                                           _DTYPES[x.dtype], n, x.stride(0), Quantizer.planes_struct(out["o"]),
                                           Quantizer.planes_struct(out["n"]), _ptr(self.scratch), self.scratch.numel(),
                                           _stream(stream)))
        return out

    def dequantize(self, planes: dict, dtype=torch.float32, stream=None) -> torch.Tensor:
        n = planes["o"]["norm"].shape[0]
        y = torch.empty((n, self.d), dtype=dtype, device=self.perm.device)
        check(_lib.lib().tq_mixed_dequantize(self.qo.handle, self.qn.handle, _ptr(self.perm),
                                             Quantizer.planes_struct(planes["o"]), Quantizer.planes_struct(planes["n"]),
                                             n, _ptr(y), _DTYPES[dtype], _stream(stream)))
        return y


def mixed_quantize_kv(mk: MixedQuantizer, mv: MixedQuantizer, k: torch.Tensor, v: torch.Tensor,
                      k_out: dict | None = None, v_out: dict | None = None, stream=None) -> tuple[dict, dict]:
    """tq_mixed_quantize_kv: k with mk and v with mv in one call (one launch on the
    tensor cores when both splits have the same d_o and bits); the scratch is mk's.
    k and v are [n, d] with unit stride along channels and the same dtype."""
    if k.dtype != v.dtype:
        raise ValueError("k and v must have the same dtype")
    for x, m in ((k, mk), (v, mv)):
        if x.dim() != 2 or x.shape[1] != m.d or (x.shape[0] and x.stride(1) != 1):
            raise ValueError("k and v must be [n, d] with unit stride along channels")
    nk, nv = k.shape[0], v.shape[0]
    k_out = mk.empty_planes(nk) if k_out is None else k_out
    v_out = mv.empty_planes(nv) if v_out is None else v_out
    P = Quantizer.planes_struct
    check(_lib.lib().tq_mixed_quantize_kv(
        mk.qo.handle, mk.qn.handle, mv.qo.handle, mv.qn.handle, _ptr(mk.perm), _ptr(mv.perm),
        _ptr(k) if nk else None, _ptr(v) if nv else None, _DTYPES[k.dtype], nk, nv, k.stride(0) if nk else mk.d,
        v.stride(0) if nv else mv.d, P(k_out["o"]), P(k_out["n"]), P(v_out["o"]), P(v_out["n"]), _ptr(mk.scratch),
        mk.scratch.numel(), _stream(stream)))
    return k_out, v_out


def mixed_decode_workspace_bytes(mk: MixedQuantizer, mv: MixedQuantizer, B: int, Hq: int, Hkv: int, T_max: int) -> int:
    n = ctypes.c_size_t()
    check(_lib.lib().tq_mixed_decode_workspace_bytes(mk.qo.handle, mk.qn.handle, mv.qo.handle, mv.qn.handle, B, Hq,
                                                     Hkv, T_max, ctypes.byref(n)))
    return n.value


def mixed_decode_attention(mk: MixedQuantizer, mv: MixedQuantizer, q: torch.Tensor, kcache: dict, vcache: dict,
                           seq_lens: torch.Tensor, Hkv: int, T_max: int, scale: float | None = None,
                           return_scores: bool = False, workspace: torch.Tensor | None = None,
                           out: torch.Tensor | None = None, stream=None):
    """tq_mixed_decode_attention; arguments as decode_attention with MixedQuantizer
    handles and {"o", "n"} caches."""
    B, Hq, d = q.shape
    if not q.is_contiguous():
        raise ValueError("q must be contiguous")
    if seq_lens.dtype != torch.int32:
        raise ValueError("seq_lens must be int32")
    need = mixed_decode_workspace_bytes(mk, mv, B, Hq, Hkv, T_max)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    scores = torch.full((B, Hq, T_max), float("nan"), dtype=torch.float32, device=q.device) if return_scores else None
    P = Quantizer.planes_struct
    check(_lib.lib().tq_mixed_decode_attention(
        mk.qo.handle, mk.qn.handle, mv.qo.handle, mv.qn.handle, _ptr(mk.perm), _ptr(mv.perm), _ptr(q),
        _DTYPES[q.dtype], P(kcache["o"]), P(kcache["n"]), P(vcache["o"]), P(vcache["n"]), _ptr(seq_lens), B, Hq,
        Hkv, T_max, float(scale) if scale is not None else 0.0, _ptr(out), _ptr(scores), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return (out, scores) if return_scores else out


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)
