"""tq_decode_attention_noalloc: decode attention whose scratch is a static device
array inside the library, for callers that cannot allocate device memory (for
example a serving loop whose memory another allocator has fully reserved, or a
thin foreign binding with no device allocator).

Checked against tq_decode_attention with a caller-owned workspace over a
sequence of calls that reuse the shared scratch: each call's split partials and
merge tickets land on bytes an earlier call left behind with another layout —
including a call whose query is NaN, so that its partials are NaN.  Also checks
that a warmed-up call leaves the device's free memory unchanged.  Collected last
on purpose.
"""
import numpy as np
import pytest
import torch

import synthetic
from _parity import check_attention

pytestmark = pytest.mark.gpu


def _case(tq, B, Hq, Hkv, T, d, kb, kv, vb, vv, lens, seed):
    K = synthetic.gaussian((B, Hkv, T, d), seed=seed + 1).cuda().reshape(-1, d)
    V = synthetic.gaussian((B, Hkv, T, d), seed=seed + 2).cuda().reshape(-1, d)
    q = synthetic.gaussian((B, Hq, d), seed=seed + 3).cuda()
    kq = tq.Quantizer(d, kb, kv, seed=seed + 11)
    vq = tq.Quantizer(d, vb, vv, seed=seed + 12)
    kc, vc = kq.quantize(K), vq.quantize(V)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    return kq, vq, q, kc, vc, sl


def _noalloc(tq, kq, vq, q, kc, vc, sl, Hkv, T, scores=False, out=None):
    from kv_cache_vector_18_b300 import _lib
    B, Hq, d = q.shape
    if out is None:
        out = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device="cuda")
    sc = torch.full((B, Hq, T), float("nan"), dtype=torch.float32, device="cuda") if scores else None
    rc = _lib.lib().tq_decode_attention_noalloc(
        kq.handle, vq.handle, q.data_ptr(), _lib.TQ_BF16, tq.Quantizer.planes_struct(kc),
        tq.Quantizer.planes_struct(vc), sl.data_ptr(), B, Hq, Hkv, T, 0.0, out.data_ptr(),
        None if sc is None else sc.data_ptr(), torch.cuda.current_stream().cuda_stream)
    _lib.check(rc)
    return out, sc


# Run in this order: a many-split layout, then a call whose NaN query leaves NaN
# partials and used tickets all over the scratch, then layouts whose partials
# and tickets sit at other offsets (a CUDA-core head dimension, fewer splits, a
# larger one again).
CASES = [
    dict(B=4, Hq=32, Hkv=4, T=3000, d=128, kb=3, kv="prod", vb=3, vv="mse", lens=[3000, 1, 2999, 1500], seed=0),
    dict(B=2, Hq=16, Hkv=2, T=2000, d=128, kb=3, kv="prod", vb=3, vv="mse", lens=[2000, 777], seed=10, nan=True),
    dict(B=1, Hq=8, Hkv=1, T=5000, d=64, kb=2, kv="mse", vb=4, vv="mse", lens=[4999], seed=50),
    dict(B=2, Hq=16, Hkv=2, T=2000, d=128, kb=3, kv="prod", vb=3, vv="mse", lens=[2000, 777], seed=20),
    dict(B=1, Hq=64, Hkv=8, T=4096, d=128, kb=4, kv="prod", vb=2, vv="mse", lens=[4096], seed=30),
]


def test_noalloc_matches_workspace_entry_point_over_dirty_scratch():
    import kv_cache_vector_18_b300 as tq
    for i, c in enumerate(CASES):
        c = dict(c)
        nan = c.pop("nan", False)
        kq, vq, q, kc, vc, sl = _case(tq, **c)
        if nan:
            q = torch.full_like(q, float("nan"))
            _noalloc(tq, kq, vq, q, kc, vc, sl, c["Hkv"], c["T"])
            torch.cuda.synchronize()
            continue
        ref, ref_sc = tq.decode_attention(kq, vq, q, kc, vc, sl, c["Hkv"], c["T"], return_scores=True)
        got, got_sc = _noalloc(tq, kq, vq, q, kc, vc, sl, c["Hkv"], c["T"], scores=True)
        torch.cuda.synchronize()
        g, r = got.double().cpu().numpy(), ref.double().cpu().numpy()
        assert np.all(np.isfinite(g)), f"call {i}: non-finite output"
        check_attention(g, r)
        gs, rs = got_sc.cpu().numpy(), ref_sc.cpu().numpy()
        valid = ~np.isnan(rs)
        assert np.array_equal(np.isnan(gs), np.isnan(rs))
        assert np.max(np.abs(gs[valid] - rs[valid])) <= 2e-3


def test_noalloc_call_leaves_free_memory_unchanged():
    import kv_cache_vector_18_b300 as tq
    kq, vq, q, kc, vc, sl = _case(tq, **{k: v for k, v in CASES[0].items()})
    out = torch.empty((4, 32, 128), dtype=torch.float32, device="cuda")
    for _ in range(2):  # warm-up: module loading, first symbol lookup
        _noalloc(tq, kq, vq, q, kc, vc, sl, 4, 3000, out=out)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _noalloc(tq, kq, vq, q, kc, vc, sl, 4, 3000, out=out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes across no-alloc calls"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import kv_cache_vector_18_b300 as tq
    from kv_cache_vector_18_b300 import _lib
    kq = tq.Quantizer(128, 3, "prod", seed=1)
    vq = tq.Quantizer(128, 3, "mse", seed=2)
    B, Hq, Hkv, T = 64, 64, 8, 131072
    assert tq.decode_workspace_bytes(kq, vq, B, Hq, Hkv, T) > _lib.NOALLOC_WORKSPACE_BYTES
    q = torch.zeros((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((B, Hq, 128), dtype=torch.float32, device="cuda")
    sl = torch.zeros((B,), dtype=torch.int32, device="cuda")
    empty = _lib.Planes(None, None, None, None)
    rc = _lib.lib().tq_decode_attention_noalloc(kq.handle, vq.handle, q.data_ptr(), _lib.TQ_BF16, empty, empty,
                                                sl.data_ptr(), B, Hq, Hkv, T, 0.0, out.data_ptr(), None, None)
    assert rc == _lib.TQ_EWORKSPACE
    assert b"static buffer" in _lib.lib().tq_last_error()
    torch.cuda.synchronize()
    assert torch.all(out == 0)
