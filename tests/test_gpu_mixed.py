"""Outlier-channel mixed precision vs the oracle (needs a GPU).

The page's experiments keep 32 "outlier" channels at 3 bits and the other 96 at
2 bits.  Each part is an ordinary quantizer of its own dimension over a channel
permutation; attention sums the parts' scores.  Checked against the oracle's
mixed_* functions: channel selection, both parts' codes, the scattered
dequantization, attention outputs and scores, and a bad permutation entry
turned into a status code.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic
from _parity import check_attention, check_dequant, check_quantize, f64, oracle_params, planes_to_oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    import kv_cache_vector_18_b300 as m
    return m


def _hot_rows(n, d, hot, seed, dtype="bf16"):
    X = synthetic.gaussian((n, d), seed=seed, dtype="f32")
    X[:, torch.as_tensor(hot)] *= 6.0
    return X.to(torch.bfloat16) if dtype == "bf16" else X


def _mixed_params(mq):
    return O.MixedParams(oracle_params(mq.qo), oracle_params(mq.qn), mq.perm.cpu().numpy())


@pytest.mark.parametrize("d,d_o", [(128, 32), (64, 32), (256, 64)])
def test_outlier_channel_selection(tq, d, d_o):
    hot = np.random.default_rng(d).choice(d, d_o, replace=False)
    X = _hot_rows(3000, d, hot, seed=d)
    perm, energy = tq.select_outlier_channels(X.cuda(), d_o)
    torch.cuda.synchronize()
    Xf = f64(X)
    assert np.allclose(energy.cpu().numpy(), np.sum(Xf * Xf, axis=0), rtol=1e-12)
    assert np.array_equal(perm.cpu().numpy(), O.outlier_channel_perm(Xf, d_o))
    assert np.array_equal(perm.cpu().numpy()[:d_o], np.sort(hot))


@pytest.mark.parametrize("variant,bo,bn", [("mse", 3, 2), ("mse", 4, 3), ("prod", 3, 2), ("prod", 4, 3)])
def test_mixed_quantize_dequantize(tq, variant, bo, bn):
    d, d_o, n = 128, 32, 1500
    hot = np.random.default_rng(1).choice(d, d_o, replace=False)
    X = _hot_rows(n, d, hot, seed=2)
    perm, _ = tq.select_outlier_channels(X.cuda(), d_o)
    mq = tq.MixedQuantizer(perm, d_o, bo, bn, variant, seed_o=5, seed_n=6)
    planes = mq.quantize(X.cuda())
    y = mq.dequantize(planes)
    torch.cuda.synchronize()
    assert mq.qo.device_status() == 0 and mq.qn.device_status() == 0
    mp = _mixed_params(mq)
    Xf = f64(X)
    check_quantize(mp.po, Xf[:, mp.out], planes["o"])
    check_quantize(mp.pn, Xf[:, mp.rest], planes["n"])
    ro = planes_to_oracle_rows(mp.po, planes["o"])
    rn = planes_to_oracle_rows(mp.pn, planes["n"])
    ref = O.mixed_dequantize(mp, ro, rn)
    rel = np.linalg.norm(f64(y) - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert rel.max() <= 1e-4, rel.max()
    # each part on its own equals the single-part path on the gathered sub-rows
    sub = X.cuda()[:, perm[:d_o].long()].contiguous()
    alone = mq.qo.quantize(sub)
    torch.cuda.synchronize()
    check_dequant(mp.po, alone, mq.qo.dequantize(alone))


@pytest.mark.parametrize("d_o,bo,bn", [(32, 3, 2), (64, 4, 2), (32, 2, 2), (64, 3, 1)])
def test_mixed_tensor_core_and_cuda_core_paths(tq, d_o, bo, bn):
    # bf16 mse rows at d = 128 take the tensor-core path when a scratch is given and
    # the per-part CUDA-core path without one; both against the oracle, over enough
    # rows for several tiles per SM, a ragged tail, and rows with one part all zero
    from kv_cache_vector_18_b300 import _lib
    d, n = 128, 148 * 128 * 2 + 77
    hot = np.random.default_rng(d_o + bo).choice(d, d_o, replace=False)
    X = _hot_rows(n, d, hot, seed=bo * 10 + bn)
    perm, _ = tq.select_outlier_channels(X.cuda(), d_o)
    hot_sorted = perm[:d_o].long().cpu()
    X[5, hot_sorted] = 0                        # outlier part zero
    rest = torch.as_tensor(np.setdiff1d(np.arange(d), hot_sorted.numpy()))
    X[n - 3, rest] = 0                          # other part zero
    X[n - 1] = 0                                # whole row zero
    mq = tq.MixedQuantizer(perm, d_o, bo, bn, "mse", seed_o=41, seed_n=42)
    xd = X.cuda()
    tc = mq.quantize(xd)
    cc = mq.empty_planes(n)
    P = tq.Quantizer.planes_struct
    assert _lib.lib().tq_mixed_quantize(mq.qo.handle, mq.qn.handle, mq.perm.data_ptr(), xd.data_ptr(), 0, n, d,
                                        P(cc["o"]), P(cc["n"]), None, 0, None) == 0
    torch.cuda.synchronize()
    assert mq.qo.device_status() == 0 and mq.qn.device_status() == 0
    mp = _mixed_params(mq)
    Xf = f64(X)
    rows = np.unique(np.concatenate([np.arange(300), np.arange(n - 300, n),
                                     np.random.default_rng(2).choice(n, 3000, replace=False)]))
    for planes in (tc, cc):
        check_quantize(mp.po, Xf[:, mp.out], planes["o"], rows=rows)
        check_quantize(mp.pn, Xf[:, mp.rest], planes["n"], rows=rows)
    assert float(tc["o"]["norm"][5]) == 0 and float(tc["n"]["norm"][n - 3]) == 0
    assert not tc["o"]["codes"][5].any() and not tc["n"]["codes"][n - 1].any()


def test_mixed_fp32_strided_input(tq):
    d, d_o = 128, 32
    perm = torch.as_tensor(np.random.default_rng(3).permutation(d), dtype=torch.int32, device="cuda")
    base = synthetic.gaussian((700, 256), seed=9, dtype="f32").cuda()
    x = base[:, 32:160]
    mq = tq.MixedQuantizer(perm, d_o, 3, 2, "mse", seed_o=1, seed_n=2)
    planes = mq.quantize(x)
    torch.cuda.synchronize()
    mp = _mixed_params(mq)
    Xf = f64(x)
    check_quantize(mp.po, Xf[:, mp.out], planes["o"])
    check_quantize(mp.pn, Xf[:, mp.rest], planes["n"])


@pytest.mark.parametrize("d,kdo,vdo,kv,kb,vv,vb,Hq", [
    (128, 32, 32, "mse", (3, 2), "mse", (3, 2), 32),   # 16 query heads per KV head: two head blocks
    (128, 32, 32, "mse", (3, 2), "mse", (3, 2), 8),
    (128, 32, 64, "prod", (4, 3), "mse", (3, 2), 8),
    (128, 64, 32, "prod", (3, 2), "prod", (4, 3), 8),
    (64, 32, 32, "mse", (4, 2), "mse", (3, 2), 8),
    (256, 64, 96, "mse", (3, 2), "prod", (3, 3), 24),  # 12 heads per KV head: 3 blocks of 4
])
def test_mixed_decode_attention(tq, d, kdo, vdo, kv, kb, vv, vb, Hq):
    B, Hkv, T = 2, 2, 333
    lens = [333, 120]
    rng = np.random.default_rng(d + kdo + vdo)
    hot_k = rng.choice(d, kdo, replace=False)
    hot_v = rng.choice(d, vdo, replace=False)
    K = _hot_rows(B * Hkv * T, d, hot_k, seed=11)
    V = _hot_rows(B * Hkv * T, d, hot_v, seed=12)
    q = synthetic.gaussian((B, Hq, d), seed=13)
    pk, _ = tq.select_outlier_channels(K.cuda(), kdo)
    pv, _ = tq.select_outlier_channels(V.cuda(), vdo)
    mk = tq.MixedQuantizer(pk, kdo, kb[0], kb[1], kv, seed_o=21, seed_n=22)
    mv = tq.MixedQuantizer(pv, vdo, vb[0], vb[1], vv, seed_o=23, seed_n=24)
    kc, vc = mk.quantize(K.cuda()), mv.quantize(V.cuda())
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out, sc = tq.mixed_decode_attention(mk, mv, q.cuda(), kc, vc, sl, Hkv, T, return_scores=True)
    torch.cuda.synchronize()
    assert mk.qo.device_status() == 0
    a, b = _mixed_params(mk), _mixed_params(mv)
    ref, ref_sc = O.mixed_decode_attention(
        a, b, f64(q), planes_to_oracle_rows(a.po, kc["o"]), planes_to_oracle_rows(a.pn, kc["n"]),
        planes_to_oracle_rows(b.po, vc["o"]), planes_to_oracle_rows(b.pn, vc["n"]), lens, Hkv, T)
    check_attention(f64(out), ref)
    g = f64(sc)
    mask = ~np.isnan(ref_sc)
    assert np.max(np.abs(g[mask] - ref_sc[mask])) <= 1e-3 * max(1.0, np.max(np.abs(ref_sc[mask])))


def test_bad_channel_entry_is_flagged(tq):
    from kv_cache_vector_18_b300 import _lib
    d, d_o = 128, 32
    perm = torch.arange(d, dtype=torch.int32, device="cuda")
    perm[40] = 1000  # outside [0, d): read as channel 0, flagged, never dereferenced
    mq = tq.MixedQuantizer(perm, d_o, 3, 2, "mse", seed_o=1, seed_n=2)
    x = synthetic.gaussian((64, d), seed=1).cuda()
    mq.quantize(x)
    torch.cuda.synchronize()
    assert mq.qo.device_status() == 0
    assert mq.qn.device_status(clear=True) == _lib.TQ_STATUS_BAD_CHANNEL
    assert mq.qn.device_status() == 0


def test_mixed_rejects_bad_arguments(tq):
    from kv_cache_vector_18_b300 import _lib
    L = _lib.lib()
    perm = torch.arange(128, dtype=torch.int32, device="cuda")
    a = tq.Quantizer(32, 3, "mse", seed=1)
    b = tq.Quantizer(96, 2, "prod", seed=2)
    x = torch.zeros((8, 128), dtype=torch.bfloat16, device="cuda")
    P = tq.Quantizer.planes_struct
    pa, pb = a.empty_planes(8), b.empty_planes(8)
    # parts of different variants
    assert L.tq_mixed_quantize(a.handle, b.handle, perm.data_ptr(), x.data_ptr(), 0, 8, 128, P(pa), P(pb),
                               None, 0, None) == _lib.TQ_EINVAL
    c = tq.Quantizer(96, 2, "mse", seed=2)
    pc = c.empty_planes(8)
    # row stride below d
    assert L.tq_mixed_quantize(a.handle, c.handle, perm.data_ptr(), x.data_ptr(), 0, 8, 64, P(pa), P(pc),
                               None, 0, None) == _lib.TQ_EINVAL
    assert L.tq_mixed_quantize(a.handle, c.handle, None, x.data_ptr(), 0, 8, 128, P(pa), P(pc),
                               None, 0, None) == _lib.TQ_EINVAL
    e = torch.empty(128, dtype=torch.float64, device="cuda")
    assert L.tq_select_outlier_channels(x.data_ptr(), 0, 8, 128, 128, 100, e.data_ptr(), perm.data_ptr(),
                                        None) == _lib.TQ_EINVAL
    torch.cuda.synchronize()


def _mixed_case(tq, B, Hq, Hkv, T, bo, bn, seed, q_dtype="bf16", kv="mse"):
    d = 128
    rng = np.random.default_rng(seed)
    hot_k = rng.choice(d, 32, replace=False)
    hot_v = rng.choice(d, 32, replace=False)
    K = _hot_rows(B * Hkv * T, d, hot_k, seed=seed + 1)
    V = _hot_rows(B * Hkv * T, d, hot_v, seed=seed + 2)
    q = synthetic.gaussian((B, Hq, d), seed=seed + 3, dtype=q_dtype)
    pk, _ = tq.select_outlier_channels(K.cuda(), 32)
    pv, _ = tq.select_outlier_channels(V.cuda(), 32)
    mk = tq.MixedQuantizer(pk, 32, bo, bn, kv, seed_o=seed + 21, seed_n=seed + 22)
    mv = tq.MixedQuantizer(pv, 32, bo, bn, "mse", seed_o=seed + 23, seed_n=seed + 24)
    kc, vc = mk.quantize(K.cuda()), mv.quantize(V.cuda())
    return mk, mv, q, kc, vc


def _mixed_ref(mk, mv, q, kc, vc, lens, Hkv, T):
    a, b = _mixed_params(mk), _mixed_params(mv)
    return O.mixed_decode_attention(
        a, b, f64(q), planes_to_oracle_rows(a.po, kc["o"]), planes_to_oracle_rows(a.pn, kc["n"]),
        planes_to_oracle_rows(b.po, vc["o"]), planes_to_oracle_rows(b.pn, vc["n"]), lens, Hkv, T)


@pytest.mark.parametrize("bo,bn,B,Hq,Hkv,T,lens,q_dtype", [
    (3, 2, 3, 16, 2, 1028, [1028, 17, 1], "bf16"),      # the page's split; two head blocks; ragged tails
    (3, 2, 2, 8, 1, 700, [0, 699], "f32"),               # an empty sequence, an fp32 query
    (4, 3, 2, 12, 3, 512, [512, 300], "bf16"),           # G = 4: a partial head block
    (4, 2, 1, 8, 1, 8192, [8191], "bf16"),               # 128 splits: several merge rounds
])
def test_mixed_decode_tensor_core_path(tq, bo, bn, B, Hq, Hkv, T, lens, q_dtype):
    # T_max % 4 == 0, 32 outlier channels, mse parts: the tensor-core mixed decode
    mk, mv, q, kc, vc = _mixed_case(tq, B, Hq, Hkv, T, bo, bn, seed=bo * 10 + bn + T, q_dtype=q_dtype)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out, sc = tq.mixed_decode_attention(mk, mv, q.cuda(), kc, vc, sl, Hkv, T, return_scores=True)
    torch.cuda.synchronize()
    assert mk.qo.device_status() == 0
    ref, ref_sc = _mixed_ref(mk, mv, q, kc, vc, lens, Hkv, T)
    check_attention(f64(out), ref)
    g = f64(sc)
    mask = ~np.isnan(ref_sc)
    assert np.array_equal(np.isnan(g), ~mask)
    assert np.max(np.abs(g[mask] - ref_sc[mask])) <= 1e-3 * max(1.0, np.max(np.abs(ref_sc[mask])))
    if 0 in lens:
        assert np.all(f64(out)[lens.index(0)] == 0)


@pytest.mark.parametrize("bo,bn,B,Hq,Hkv,T,lens,q_dtype", [
    (3, 2, 3, 16, 2, 1028, [1028, 17, 1], "bf16"),      # the page's split; two head blocks; ragged tails
    (4, 3, 2, 8, 1, 700 + 32, [0, 731], "f32"),          # an empty sequence, an fp32 query
    (4, 2, 1, 8, 1, 8192, [8191], "bf16"),               # many splits: several merge rounds
])
def test_mixed_decode_tensor_core_prod_keys(tq, bo, bn, B, Hq, Hkv, T, lens, q_dtype):
    # prod key parts (codes of b − 1 bits and QJL signs per part) with mse values of
    # the same bits: the tensor-core mixed decode (its workspace is the one the mse
    # keys of the same shape take, not the CUDA-core path's)
    mk, mv, q, kc, vc = _mixed_case(tq, B, Hq, Hkv, T, bo, bn, seed=bo * 10 + bn + T + 1, q_dtype=q_dtype,
                                    kv="prod")
    mse_k = tq.MixedQuantizer(mk.perm, 32, bo, bn, "mse", seed_o=1, seed_n=2)
    assert tq.mixed_decode_workspace_bytes(mk, mv, B, Hq, Hkv, T) == \
        tq.mixed_decode_workspace_bytes(mse_k, mv, B, Hq, Hkv, T)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out, sc = tq.mixed_decode_attention(mk, mv, q.cuda(), kc, vc, sl, Hkv, T, return_scores=True)
    torch.cuda.synchronize()
    assert mk.qo.device_status() == 0
    ref, ref_sc = _mixed_ref(mk, mv, q, kc, vc, lens, Hkv, T)
    check_attention(f64(out), ref)
    g = f64(sc)
    mask = ~np.isnan(ref_sc)
    assert np.array_equal(np.isnan(g), ~mask)
    assert np.max(np.abs(g[mask] - ref_sc[mask])) <= 1e-3 * max(1.0, np.max(np.abs(ref_sc[mask])))
    if 0 in lens:
        assert np.all(f64(out)[lens.index(0)] == 0)


def test_mixed_decode_tensor_core_bad_channel_flagged(tq):
    # a permutation entry outside [0, d) in the decode's key or value map is read
    # as channel 0 and recorded in the outlier key handle's status word
    from kv_cache_vector_18_b300 import _lib
    mk, mv, q, kc, vc = _mixed_case(tq, 1, 8, 1, 256, 3, 2, seed=5)
    sl = torch.tensor([256], dtype=torch.int32, device="cuda")
    pk_bad = mk.perm.clone()
    pk_bad[77] = -3
    mk.perm = pk_bad
    out = tq.mixed_decode_attention(mk, mv, q.cuda(), kc, vc, sl, 1, 256)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    assert mk.qo.device_status(clear=True) == _lib.TQ_STATUS_BAD_CHANNEL
    assert mk.qo.device_status() == 0


@pytest.mark.parametrize("case", [
    # (key d_o, key bits, value d_o, value bits, key rows, value rows, dtype)
    (32, (3, 2), 32, (3, 2), 148 * 128 + 77, 2 * 148 * 128 + 5, "bf16"),   # one launch, ragged tails
    (64, (4, 2), 64, (4, 2), 3000, 1, "bf16"),                            # one launch, 1-row side
    (32, (4, 3), 32, (4, 3), 1, 129, "bf16"),                              # one launch on two CTAs
    (32, (3, 2), 64, (3, 2), 900, 700, "bf16"),                            # d_o differs: two launches
    (32, (3, 2), 32, (4, 2), 900, 700, "bf16"),                            # bits differ: two launches
    (32, (3, 2), 32, (3, 2), 0, 500, "bf16"),                              # no keys
    (32, (3, 2), 32, (3, 2), 500, 0, "bf16"),                              # no values
    (32, (3, 2), 32, (3, 2), 400, 300, "f32"),                             # CUDA-core parts
])
def test_mixed_quantize_kv_matches_separate_calls(tq, case):
    # tq_mixed_quantize_kv writes the bytes the two tq_mixed_quantize calls write
    # (each checked against the oracle elsewhere); the value side is also checked
    # against the oracle directly on sampled rows
    kdo, kb, vdo, vb, nk, nv, dt = case
    d = 128
    K = _hot_rows(max(nk, 1), d, np.arange(0, 128, 4)[:kdo], seed=21, dtype=dt)[:nk]
    V = _hot_rows(max(nv, 1), d, np.arange(1, 128, 4)[:vdo], seed=22, dtype=dt)[:nv]
    pk = torch.as_tensor(np.random.default_rng(5).permutation(d), dtype=torch.int32, device="cuda")
    pv = torch.as_tensor(np.random.default_rng(6).permutation(d), dtype=torch.int32, device="cuda")
    mk = tq.MixedQuantizer(pk, kdo, kb[0], kb[1], "mse", seed_o=51, seed_n=52)
    mv = tq.MixedQuantizer(pv, vdo, vb[0], vb[1], "mse", seed_o=53, seed_n=54)
    kd, vd = K.cuda().contiguous(), V.cuda().contiguous()
    kc, vc = tq.mixed_quantize_kv(mk, mv, kd, vd)
    ks = mk.quantize(kd) if nk else mk.empty_planes(0)
    vs = mv.quantize(vd) if nv else mv.empty_planes(0)
    torch.cuda.synchronize()
    for m in (mk, mv):
        assert m.qo.device_status() == 0 and m.qn.device_status() == 0
    for got, ref in ((kc, ks), (vc, vs)):
        for part in ("o", "n"):
            for name in ref[part]:
                assert torch.equal(got[part][name], ref[part][name]), (part, name)
    if nv:
        mp = _mixed_params(mv)
        Xf = f64(V)
        rows = np.unique(np.concatenate([np.arange(min(nv, 150)), np.arange(max(nv - 150, 0), nv)]))
        check_quantize(mp.po, Xf[:, mp.out], vc["o"], rows=rows)
        check_quantize(mp.pn, Xf[:, mp.rest], vc["n"], rows=rows)


def test_mixed_quantize_kv_rejects_bad_arguments(tq):
    from kv_cache_vector_18_b300 import _lib
    perm = torch.arange(128, dtype=torch.int32, device="cuda")
    mk = tq.MixedQuantizer(perm, 32, 3, 2, "mse", seed_o=1, seed_n=2)
    mv = tq.MixedQuantizer(perm, 32, 3, 2, "mse", seed_o=3, seed_n=4)
    x = torch.zeros((16, 128), dtype=torch.bfloat16, device="cuda")
    kp, vp = mk.empty_planes(16), mv.empty_planes(16)
    P = tq.Quantizer.planes_struct
    L = _lib.lib()

    def call(hvo=mv.qo.handle, v_stride=128, scratch_bytes=mk.scratch.numel()):
        return L.tq_mixed_quantize_kv(mk.qo.handle, mk.qn.handle, hvo, mv.qn.handle, perm.data_ptr(),
                                      perm.data_ptr(), x.data_ptr(), x.data_ptr(), 0, 16, 16, 128, v_stride,
                                      P(kp["o"]), P(kp["n"]), P(vp["o"]), P(vp["n"]), mk.scratch.data_ptr(),
                                      scratch_bytes, None)
    assert call(hvo=None) == _lib.TQ_EINVAL
    assert call(v_stride=100) == _lib.TQ_EINVAL
    assert call(v_stride=132) == _lib.TQ_EALIGN
    assert "value" in L.tq_last_error().decode()
    # one operand's worth of scratch: the sides run one after the other, same bytes
    assert call(scratch_bytes=L.tq_mixed_quantize_scratch_bytes()) == 0
    torch.cuda.synchronize()
    assert mk.qo.device_status() == 0 and mv.qo.device_status() == 0
