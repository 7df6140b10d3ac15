"""Parity at the full sizes of the workloads (needs a GPU).

Each case runs the library at the size and in the launch configuration that
bench.py times (same shapes, same seeds, same quantizer seeds, same calls), and
checks sampled outputs against the oracle one by one: packed rows of the codec
on a sample of rows, and the attention outputs of whole (batch, KV head)
groups, which the oracle recomputes from the dequantized cache of that group.
The bit-width / head-dimension sweep adds what holds at any size: the
distortion over all 2^20 rows against the oracle's D_mse, and unbiased inner
products for the prod variant.
"""
import math

import numpy as np
import pytest
import torch

import bench
import oracle as O
import synthetic
from _parity import (check_attention, check_dequant, check_quantize, f64, oracle_params,
                     planes_to_oracle_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    import kv_cache_vector_18_b300 as m
    return m


def _sample_rows(n: int, k: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    rows = np.concatenate([np.arange(0, min(256, n)), np.arange(max(n - 256, 0), n), rng.choice(n, min(k, n), replace=False)])
    return np.unique(rows)


def _slice(planes: dict, rows: np.ndarray) -> dict:
    idx = torch.as_tensor(rows, device="cuda")
    return {k: (v.index_select(0, idx) if v.numel() else v) for k, v in planes.items()}


def _group_rows(b: int, kvh: int, Hkv: int, T: int, L: int) -> np.ndarray:
    base = (b * Hkv + kvh) * T
    return np.arange(base, base + L)


@pytest.mark.parametrize("workload,groups", [
    ("llama70b_layer_kv_quant", [(0, 0), (0, 5)]),
    ("decode_131k", [(0, 0), (0, 7)]),
    ("batched_decode_32k", "shortest,longest,mid"),
])
def test_workload_full_size(tq, workload, groups):
    spec = bench.workload_spec(workload)
    K, V, q, lens = bench.make_inputs(spec)
    d, B, Hq, Hkv, T = spec["d"], spec["B"], spec["Hq"], spec["Hkv"], spec["T"]
    G = Hq // Hkv
    kq = tq.Quantizer(d, spec["k_bits"], spec["k_variant"], seed=10)
    vq = tq.Quantizer(d, spec["v_bits"], spec["v_variant"], seed=11)
    Kf, Vf = K.reshape(-1, d), V.reshape(-1, d)
    Kd, Vd, qd, ld = Kf.cuda(), Vf.cuda(), q.cuda(), lens.cuda()
    kc, vc = kq.quantize(Kd), vq.quantize(Vd)
    out = tq.decode_attention(kq, vq, qd, kc, vc, ld, Hkv, T)
    torch.cuda.synchronize()
    assert kq.device_status() == 0 and vq.device_status() == 0
    pk, pv = oracle_params(kq), oracle_params(vq)

    # codec: sampled rows of both caches
    n = Kf.shape[0]
    rows = _sample_rows(n, 4096, seed=len(workload))
    check_quantize(pk, f64(Kf[torch.as_tensor(rows)]), _slice(kc, rows))
    check_quantize(pv, f64(Vf[torch.as_tensor(rows)]), _slice(vc, rows))

    # attention: whole (batch, KV head) groups against the oracle on the GPU's packed cache
    L = lens.tolist()
    if groups == "shortest,longest,mid":
        order = np.argsort(L)
        groups = [(int(order[0]), 1), (int(order[-1]), 6), (int(order[len(order) // 2]), 3)]
    out_np = f64(out)
    for b, kvh in groups:
        r = _group_rows(b, kvh, Hkv, T, L[b])
        k_rows = planes_to_oracle_rows(pk, kc, rows=r)
        v_rows = planes_to_oracle_rows(pv, vc, rows=r)
        qg = f64(q)[b:b + 1, kvh * G:(kvh + 1) * G]
        ref, _ = O.decode_attention(pk, pv, qg, k_rows, v_rows, [L[b]], 1, L[b])
        check_attention(out_np[b:b + 1, kvh * G:(kvh + 1) * G], ref)


def test_small_config_fp32_rows_full(tq):
    # 4096 fp32 N(0,1) rows, mse b = 2: quantize + dequantize all rows, then 64 fp32
    # queries scored against all 4096 keys
    w = synthetic.WORKLOADS["small_mse_b2"]
    n, d, nq = w["rows"], w["d"], w["queries"]
    X = synthetic.gaussian((n, d), seed=0, dtype="f32")
    qz = tq.Quantizer(d, w["bits"], w["variant"], seed=0)
    planes = qz.quantize(X.cuda())
    y = qz.dequantize(planes)
    q = synthetic.gaussian((1, nq, d), seed=1, dtype="f32")
    sl = torch.tensor([n], dtype=torch.int32, device="cuda")
    out, sc = tq.decode_attention(qz, qz, q.cuda(), planes, planes, sl, 1, n, return_scores=True)
    torch.cuda.synchronize()
    p = oracle_params(qz)
    check_quantize(p, f64(X), planes)
    check_dequant(p, planes, y)
    rows = planes_to_oracle_rows(p, planes)
    ref, ref_sc = O.decode_attention(p, p, f64(q), rows, rows, [n], 1, n)
    check_attention(f64(out), ref)
    rs = ref_sc[0]
    assert np.max(np.abs(f64(sc)[0] - rs)) <= 1e-3 * max(1.0, np.max(np.abs(rs)))


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("variant", ["mse", "prod"])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_sweep_point_full_size(tq, d, variant, bits):
    w = synthetic.WORKLOADS["sweep"]
    n, nq = w["rows"], w["queries"]
    seed = 100 * d + 10 * bits + (variant == "prod")
    X = synthetic.gaussian_cuda((n, d), seed=seed)  # bf16 on the device
    qz = tq.Quantizer(d, bits, variant, seed=seed)
    planes = qz.quantize(X)
    Y = qz.dequantize(planes)
    torch.cuda.synchronize()
    assert qz.device_status() == 0
    p = oracle_params(qz)
    # sampled rows, bit-exact codes / signs and dequantized rows against the oracle
    rows = _sample_rows(n, 2048, seed=seed)
    ridx = torch.as_tensor(rows, device="cuda")
    sub = _slice(planes, rows)
    check_quantize(p, f64(X.index_select(0, ridx)), sub)
    check_dequant(p, sub, Y.index_select(0, ridx))
    # what holds at any size, over all 2^20 rows and 1024 random queries:
    #   mse   D = E‖x − x̃‖²/‖x‖² equals the oracle's d·C(f_X, b); inner products
    #         shrink by 1 − D (the centroid condition makes x̃ ⟂ x − x̃ on average)
    #         and their error, relative to E⟨y, x⟩², is D
    #   prod  E‖r‖² = D_mse(b − 1) for the stored residual norms; inner products are
    #         unbiased (slope 1) with relative error at most (π/2)·D_mse(b − 1)
    Xf = X.float()
    dm = O.mse_distortion_theory(d, 1 << p.b_mse) if p.b_mse > 0 else 1.0
    if variant == "mse":
        err = ((Xf - Y.float()) ** 2).sum(1) / (Xf ** 2).sum(1).clamp_min(1e-30)
        D = float(err.double().mean())
        assert abs(D - dm) <= 0.02 * dm, (D, dm)
    else:
        r2 = float((planes["rnorm"].double() ** 2).mean())
        assert abs(r2 - dm) <= 0.02 * dm, (r2, dm)
    Q = synthetic.gaussian_cuda((nq, d), seed=seed + 1, dtype=torch.float32)
    m = 1 << 16
    ip_true = (Q @ Xf[:m].T).double()
    ip_est = (Q @ Y.float()[:m].T).double()
    beta = float((ip_est * ip_true).sum() / (ip_true ** 2).sum())
    rel = float(((ip_est - ip_true) ** 2).mean() / (ip_true ** 2).mean())
    if variant == "mse":
        assert abs(beta - (1 - dm)) <= 0.02, (beta, dm)
        assert abs(rel - dm) <= 0.05 * dm + 1e-4, (rel, dm)
    else:
        assert abs(beta - 1.0) <= 0.02, beta
        assert rel <= 1.1 * (math.pi / 2) * dm, (rel, dm)
