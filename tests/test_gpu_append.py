"""Decode step with append (tq_decode_append_attention) vs the oracle (needs a GPU).

Each step quantizes the new key and value row of every (batch, KV head) into the
next free token of its slab, bumps the length, and attends over the cache with
the new token.  Checked: the appended rows against the oracle's quantization of
the new rows, every other cache row untouched, the lengths, the attention output
against the oracle over the GPU's cache, and a full slab left alone and flagged.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from _parity import check_attention, check_quantize, f64, oracle_params, planes_to_oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    import kv_cache_vector_18_b300 as m
    return m


def _rows(planes: dict, rows) -> dict:
    idx = torch.as_tensor(np.asarray(rows), device="cuda")
    return {k: (v.index_select(0, idx) if v.numel() else v) for k, v in planes.items()}


def _clone(planes: dict) -> dict:
    return {k: v.clone() for k, v in planes.items()}


def _setup(tq, B, Hq, Hkv, T, d, kb, kv, vb, vv, lens, seed, rotation="qr"):
    K = synthetic.gaussian((B, Hkv, T, d), seed=seed + 1)
    V = synthetic.gaussian((B, Hkv, T, d), seed=seed + 2)
    kq = tq.Quantizer(d, kb, kv, seed=seed + 11, rotation=rotation)
    vq = tq.Quantizer(d, vb, vv, seed=seed + 12, rotation=rotation)
    kc = kq.quantize(K.cuda().reshape(-1, d))
    vc = vq.quantize(V.cuda().reshape(-1, d))
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    return kq, vq, kc, vc, sl


def _step_and_check(tq, kq, vq, kc, vc, sl, B, Hq, Hkv, T, d, seed, kv_dtype="bf16"):
    lens0 = sl.cpu().numpy().copy()
    k_new = synthetic.gaussian((B, Hkv, d), seed=seed + 100, dtype=kv_dtype)
    v_new = synthetic.gaussian((B, Hkv, d), seed=seed + 101, dtype=kv_dtype)
    q = synthetic.gaussian((B, Hq, d), seed=seed + 102)
    kc0, vc0 = _clone(kc), _clone(vc)
    out = tq.decode_append_attention(kq, vq, q.cuda(), k_new.cuda(), v_new.cuda(), kc, vc, sl, Hkv, T)
    torch.cuda.synchronize()
    lens1 = sl.cpu().numpy()
    room = (lens0 >= 0) & (lens0 < T)
    assert np.array_equal(lens1, np.where(room, lens0 + 1, lens0))
    # appended rows: the oracle's quantization of the new rows
    src, dst = [], []
    for b in range(B):
        for h in range(Hkv):
            if room[b]:
                src.append(b * Hkv + h)
                dst.append((b * Hkv + h) * T + lens0[b])
    pk, pv = oracle_params(kq), oracle_params(vq)
    if src:
        check_quantize(pk, f64(k_new.reshape(-1, d))[src], _rows(kc, dst))
        check_quantize(pv, f64(v_new.reshape(-1, d))[src], _rows(vc, dst))
    # every other row untouched
    keep = np.setdiff1d(np.arange(B * Hkv * T), np.asarray(dst, dtype=np.int64))
    for new, old in ((kc, kc0), (vc, vc0)):
        for name in new:
            if new[name].numel():
                a, b_ = _rows(new, keep)[name], _rows(old, keep)[name]
                assert torch.equal(a, b_), name
    ref, _ = O.decode_attention(pk, pv, f64(q), planes_to_oracle_rows(pk, kc), planes_to_oracle_rows(pv, vc),
                                lens1.tolist(), Hkv, T)
    check_attention(f64(out), ref)
    return out


@pytest.mark.parametrize("kv,kb,vv,vb", [("prod", 3, "mse", 3), ("mse", 3, "mse", 3), ("prod", 4, "mse", 2),
                                         ("prod", 3, "prod", 3)])
def test_append_step(tq, kv, kb, vv, vb):
    B, Hq, Hkv, T, d = 3, 16, 2, 300, 128
    kq, vq, kc, vc, sl = _setup(tq, B, Hq, Hkv, T, d, kb, kv, vb, vv, [0, 150, 299], seed=kb * 10 + vb)
    _step_and_check(tq, kq, vq, kc, vc, sl, B, Hq, Hkv, T, d, seed=7)
    assert kq.device_status() == 0


@pytest.mark.parametrize("kv,kb,vv,vb", [("prod", 3, "mse", 3), ("mse", 3, "mse", 3)])
def test_append_long_context_streams_stable_prefix(tq, kv, kb, vv, vb):
    # 131072-token slabs: the decode's CTAs take chunks long enough to stream
    # their rows below the pre-append length before waiting for the append, and
    # the append runs on the SMs the decode grid leaves free.  Checked: the
    # appended rows against the oracle, the output bit for bit against the plain
    # decode over the updated cache (same plan, same arithmetic), and five steps
    # enqueued without synchronisation against the same steps synchronised one
    # by one.
    B, Hq, Hkv, T, d = 1, 64, 8, 131072, 128
    kq = tq.Quantizer(d, kb, kv, seed=31)
    vq = tq.Quantizer(d, vb, vv, seed=32)
    kc = kq.quantize(synthetic.gaussian_cuda((B * Hkv * T, d), seed=33))
    vc = vq.quantize(synthetic.gaussian_cuda((B * Hkv * T, d), seed=34))
    sl = torch.tensor([T - 100], dtype=torch.int32, device="cuda")
    new = [(synthetic.gaussian((B, Hkv, d), seed=200 + i), synthetic.gaussian((B, Hkv, d), seed=300 + i),
            synthetic.gaussian((B, Hq, d), seed=400 + i)) for i in range(6)]
    kn, vn, qn = new[0]
    out = tq.decode_append_attention(kq, vq, qn.cuda(), kn.cuda(), vn.cuda(), kc, vc, sl, Hkv, T)
    plain = tq.decode_attention(kq, vq, qn.cuda(), kc, vc, sl, Hkv, T)
    torch.cuda.synchronize()
    assert sl.tolist() == [T - 99]
    assert torch.equal(out, plain)
    dst = [h * T + T - 100 for h in range(Hkv)]
    check_quantize(oracle_params(kq), f64(kn.reshape(-1, d)), _rows(kc, dst))
    check_quantize(oracle_params(vq), f64(vn.reshape(-1, d)), _rows(vc, dst))
    kc0, vc0, sl0 = _clone(kc), _clone(vc), sl.clone()
    dev = [(k.cuda(), v.cuda(), q.cuda()) for k, v, q in new[1:]]
    torch.cuda.synchronize()
    free = [tq.decode_append_attention(kq, vq, q, k, v, kc, vc, sl, Hkv, T) for k, v, q in dev]
    torch.cuda.synchronize()
    for i, (k, v, q) in enumerate(dev):
        ref = tq.decode_append_attention(kq, vq, q, k, v, kc0, vc0, sl0, Hkv, T)
        torch.cuda.synchronize()
        assert torch.equal(free[i], ref), i
    assert torch.equal(sl, sl0) and sl.tolist() == [T - 94]
    for a_, b_ in ((kc, kc0), (vc, vc0)):
        for name in a_:
            assert torch.equal(a_[name], b_[name]), name
    assert kq.device_status() == 0


@pytest.mark.parametrize("Hq", [64, 32])  # 8 query heads per KV head, and 4 (the keys-as-A step)
def test_append_long_context_ragged_and_full(tq, Hq):
    # as above with two ragged slabs and a full one in the batch: chunks that end
    # before a slab's length, one that holds it, ones past it, and a slab that
    # takes no row (its status flagged, its length unchanged)
    B, Hkv, T, d = 3, 8, 65536, 128
    kq = tq.Quantizer(d, 3, "prod", seed=41)
    vq = tq.Quantizer(d, 3, "mse", seed=42)
    kc = kq.quantize(synthetic.gaussian_cuda((B * Hkv * T, d), seed=43))
    vc = vq.quantize(synthetic.gaussian_cuda((B * Hkv * T, d), seed=44))
    lens0 = [65000, 30001, T]
    sl = torch.tensor(lens0, dtype=torch.int32, device="cuda")
    kn, vn, qn = (synthetic.gaussian((B, Hkv, d), seed=45), synthetic.gaussian((B, Hkv, d), seed=46),
                  synthetic.gaussian((B, Hq, d), seed=47))
    out = tq.decode_append_attention(kq, vq, qn.cuda(), kn.cuda(), vn.cuda(), kc, vc, sl, Hkv, T)
    plain = tq.decode_attention(kq, vq, qn.cuda(), kc, vc, sl, Hkv, T)
    torch.cuda.synchronize()
    assert sl.tolist() == [65001, 30002, T]
    assert torch.equal(out, plain)
    assert kq.device_status(clear=True) == _lib_status()
    src = [b * Hkv + h for b in range(2) for h in range(Hkv)]
    dst = [(b * Hkv + h) * T + lens0[b] for b in range(2) for h in range(Hkv)]
    check_quantize(oracle_params(kq), f64(kn.reshape(-1, d))[src], _rows(kc, dst))
    check_quantize(oracle_params(vq), f64(vn.reshape(-1, d))[src], _rows(vc, dst))


@pytest.mark.parametrize("d", [64, 256])
def test_append_other_head_dims_and_fp32_rows(tq, d):
    B, Hq, Hkv, T = 2, 8, 2, 200
    kq, vq, kc, vc, sl = _setup(tq, B, Hq, Hkv, T, d, 3, "prod", 3, "mse", [17, 0], seed=d)
    _step_and_check(tq, kq, vq, kc, vc, sl, B, Hq, Hkv, T, d, seed=d + 1, kv_dtype="f32")


def test_append_several_steps_hadamard(tq):
    B, Hq, Hkv, T, d = 2, 8, 1, 130, 128
    kq, vq, kc, vc, sl = _setup(tq, B, Hq, Hkv, T, d, 3, "prod", 3, "mse", [125, 3], seed=5, rotation="hadamard")
    for step in range(6):  # batch 0 fills up at step 5 and is left alone after that
        _step_and_check(tq, kq, vq, kc, vc, sl, B, Hq, Hkv, T, d, seed=40 + step)
    assert sl.tolist() == [130, 9]
    assert kq.device_status() == _lib_status()


def _lib_status():
    from kv_cache_vector_18_b300 import _lib
    return _lib.TQ_STATUS_APPEND_FULL


def test_append_full_slab_flagged_and_untouched(tq):
    B, Hq, Hkv, T, d = 2, 8, 2, 64, 128
    kq, vq, kc, vc, sl = _setup(tq, B, Hq, Hkv, T, d, 3, "prod", 3, "mse", [64, 10], seed=9)
    assert kq.device_status() == 0
    _step_and_check(tq, kq, vq, kc, vc, sl, B, Hq, Hkv, T, d, seed=11)
    assert kq.device_status(clear=True) == _lib_status()
    assert kq.device_status() == 0


def test_append_rejects_bad_arguments(tq):
    from kv_cache_vector_18_b300 import _lib
    B, Hq, Hkv, T, d = 1, 8, 1, 16, 128
    kq, vq, kc, vc, sl = _setup(tq, B, Hq, Hkv, T, d, 3, "mse", 3, "mse", [3], seed=1)
    q = torch.zeros((B, Hq, d), dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros((B, Hkv, d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        tq.decode_append_attention(kq, vq, q, kn, kn.float(), kc, vc, sl, Hkv, T)
    L = _lib.lib()
    ws = torch.empty(tq.decode_workspace_bytes(kq, vq, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    P = tq.Quantizer.planes_struct
    args = [kq.handle, vq.handle, q.data_ptr(), 0, kn.data_ptr(), kn.data_ptr(), 0, P(kc), P(vc), sl.data_ptr(),
            B, Hq, Hkv, T, 0.0, out.data_ptr(), ws.data_ptr(), ws.numel(), None]
    bad = list(args)
    bad[6] = 9  # kv dtype
    assert L.tq_decode_append_attention(*bad) == _lib.TQ_EINVAL
    bad = list(args)
    bad[4] = None  # k_new
    assert L.tq_decode_append_attention(*bad) == _lib.TQ_EINVAL
    bad = list(args)
    bad[17] = 16  # workspace too small
    assert L.tq_decode_append_attention(*bad) == _lib.TQ_EWORKSPACE
    torch.cuda.synchronize()
    assert sl.tolist() == [3]  # nothing was launched
