"""Walsh–Hadamard rotation option (tq_init_ex) vs the oracle (needs a GPU).

The page's community findings (#3) recommend a Walsh–Hadamard transform for the
MSE stage with an independent transform for QJL.  The tensor-core quantize path
takes the ±1 matrix √d·Π in one MMA pass; every other kernel reads Π itself.
"""
import math

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


def test_device_params_match_oracle(tq):
    for d, b, v in [(32, 2, "mse"), (128, 3, "prod"), (256, 4, "mse")]:
        qz = tq.Quantizer(d, b, v, seed=77, rotation="hadamard")
        p = O.make_params(d, b, v, 77, rotation="hadamard")
        assert np.max(np.abs(qz.params()["Pi"] - p.Pi)) <= 1e-15


def test_rejects_non_power_of_two(tq):
    with pytest.raises(tq.TQError, match="power of two"):
        tq.Quantizer(96, 2, "mse", seed=0, rotation="hadamard")


@pytest.mark.parametrize("variant", ["mse", "prod"])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_quantize_dequantize_parity(tq, d, bits, variant):
    n = 1000  # several 128-row tiles and a ragged tail
    qz = tq.Quantizer(d, bits, variant, seed=2000 + d + bits, rotation="hadamard")
    x = synthetic.gaussian((n, d), seed=d * 10 + bits + 5, dtype="bf16").cuda()
    planes = qz.quantize(x)
    y = qz.dequantize(planes)
    torch.cuda.synchronize()
    p = oracle_params(qz)
    assert p.rotation == "hadamard"
    check_quantize(p, f64(x), planes)
    check_dequant(p, planes, y)
    assert qz.device_status() == 0


@pytest.mark.parametrize("variant", ["mse", "prod"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_tensor_core_path_many_tiles(tq, d, bits, variant):
    # several tiles per CTA on every SM, a ragged tail, zero rows and one-hot rows
    # (every rotated coordinate of a one-hot row is ±‖x‖/√d)
    n = 148 * 128 * 3 + 77
    qz = tq.Quantizer(d, bits, variant, seed=31 + bits, rotation="hadamard")
    x = synthetic.gaussian((n, d), seed=bits + d + 1).cuda()
    x[5] = 0
    x[n - 2] = 0
    for r, k in [(10, 0), (11, d - 1), (n - 1, d // 2)]:
        x[r] = 0
        x[r, k] = 2.5
    planes = qz.quantize(x)
    torch.cuda.synchronize()
    assert qz.device_status() == 0
    rows = np.concatenate([np.arange(0, 300), np.arange(n - 300, n),
                           np.random.default_rng(1).choice(n, 3000, replace=False)])
    p = oracle_params(qz)
    check_quantize(p, f64(x), planes, rows=rows)
    y = qz.dequantize(planes)
    torch.cuda.synchronize()
    check_dequant(p, planes, y, rows=np.array([5, 10, 11, n - 2, n - 1]))


def test_fp32_input_and_strided_rows(tq):
    qz = tq.Quantizer(128, 3, "mse", seed=8, rotation="hadamard")
    base = synthetic.gaussian((600, 256), seed=6, dtype="f32").cuda()
    x = base[:, 64:192]
    planes = qz.quantize(x)
    torch.cuda.synchronize()
    check_quantize(oracle_params(qz), f64(x), planes)


@pytest.mark.parametrize("kv,kb,vv,vb", [("prod", 3, "mse", 3), ("mse", 4, "mse", 2), ("prod", 2, "prod", 3)])
def test_decode_attention(tq, kv, kb, vv, vb):
    B, Hq, Hkv, T, d = 2, 16, 2, 700, 128
    lens = [700, 291]
    K = synthetic.gaussian((B, Hkv, T, d), seed=41)
    V = synthetic.gaussian((B, Hkv, T, d), seed=42)
    q = synthetic.gaussian((B, Hq, d), seed=43)
    kq = tq.Quantizer(d, kb, kv, seed=51, rotation="hadamard")
    vq = tq.Quantizer(d, vb, vv, seed=52, rotation="hadamard")
    kc = kq.quantize(K.cuda().reshape(-1, d))
    vc = vq.quantize(V.cuda().reshape(-1, d))
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = tq.decode_attention(kq, vq, q.cuda(), kc, vc, sl, Hkv, T)
    torch.cuda.synchronize()
    pk, pv = oracle_params(kq), oracle_params(vq)
    ref, _ = O.decode_attention(pk, pv, f64(q), planes_to_oracle_rows(pk, kc), planes_to_oracle_rows(pv, vc),
                                lens, Hkv, T)
    check_attention(f64(out), ref)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_distortion_at_full_size(tq, d, bits):
    # 2^20 Gaussian rows: Π_H is orthogonal, so D_mse = d·C(f_X, b) holds for them
    # exactly in expectation, as for the QR rotation
    n = 1 << 20
    seed = 500 + 10 * d + bits
    X = synthetic.gaussian_cuda((n, d), seed=seed)
    qz = tq.Quantizer(d, bits, "mse", seed=seed, rotation="hadamard")
    planes = qz.quantize(X)
    Y = qz.dequantize(planes)
    torch.cuda.synchronize()
    assert qz.device_status() == 0
    Xf = X.float()
    err = ((Xf - Y.float()) ** 2).sum(1) / (Xf ** 2).sum(1).clamp_min(1e-30)
    D = float(err.double().mean())
    dm = O.mse_distortion_theory(d, 1 << bits)
    se = float(err.double().std()) / math.sqrt(n)
    assert abs(D - dm) <= 4 * se + 2e-3 * dm, (D, dm)
    rows = np.unique(np.concatenate([np.arange(256), np.random.default_rng(seed).choice(n, 1024, replace=False)]))
    ridx = torch.as_tensor(rows, device="cuda")
    sub = {k: (v.index_select(0, ridx) if v.numel() else v) for k, v in planes.items()}
    check_quantize(oracle_params(qz), f64(X.index_select(0, ridx)), sub)
