"""CUDA quantize / dequantize vs the oracle, through the C ABI (needs a GPU)."""
import numpy as np
import pytest
import torch

import synthetic
from _parity import check_dequant, check_quantize, f64, oracle_params

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    import kv_cache_vector_18_b300 as m
    return m


@pytest.mark.parametrize("variant", ["mse", "prod"])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_quantize_dequantize_parity(tq, d, bits, variant):
    n = 1000  # several 128-row tiles and a ragged tail
    qz = tq.Quantizer(d, bits, variant, seed=1000 + d + bits)
    x = synthetic.gaussian((n, d), seed=d * 10 + bits, dtype="bf16").cuda()
    planes = qz.quantize(x)
    y = qz.dequantize(planes)
    torch.cuda.synchronize()
    p = oracle_params(qz)
    X = f64(x)
    check_quantize(p, X, planes)
    check_dequant(p, planes, y)
    assert qz.device_status() == 0


@pytest.mark.parametrize("variant", ["mse", "prod"])
def test_fp32_input(tq, variant):
    qz = tq.Quantizer(128, 2, variant, seed=5)
    x = synthetic.gaussian((4096, 128), seed=0, dtype="f32").cuda()
    planes = qz.quantize(x)
    torch.cuda.synchronize()
    check_quantize(oracle_params(qz), f64(x), planes)


@pytest.mark.parametrize("n", [1, 127, 128, 129, 255, 4097])
def test_ragged_row_counts(tq, n):
    qz = tq.Quantizer(128, 3, "prod", seed=3)
    x = synthetic.gaussian((n, 128), seed=n, dtype="bf16").cuda()
    planes = qz.quantize(x)
    y = qz.dequantize(planes)
    torch.cuda.synchronize()
    p = oracle_params(qz)
    check_quantize(p, f64(x), planes)
    check_dequant(p, planes, y)


def test_zero_rows_and_strided_input(tq):
    qz = tq.Quantizer(64, 3, "prod", seed=9)
    base = synthetic.gaussian((300, 128), seed=4, dtype="bf16").cuda()
    base[7] = 0
    base[200] = 0
    x = base[:, :64]  # row stride 128 elements
    planes = qz.quantize(x)
    torch.cuda.synchronize()
    p = oracle_params(qz)
    check_quantize(p, f64(x), planes)
    codes = planes["codes"].cpu().numpy()
    assert np.all(codes[7] == 0) and np.all(planes["signs"].cpu().numpy()[7] == 255)
    assert planes["norm"][200].item() == 0 and planes["rnorm"][200].item() == 0
    y = qz.dequantize(planes)
    assert torch.all(y[7] == 0)


def test_outlier_channels_and_heavy_tails(tq):
    ch = synthetic.outlier_channels(128, 4, seed=4)
    x = synthetic.kv_with_outliers(2, 1024, 128, seed=0, channels=ch).reshape(-1, 128).cuda()
    t = synthetic.student_t_unit_var((2048, 128), seed=3).cuda()
    for data in (x, t):
        qz = tq.Quantizer(128, 3, "mse", seed=10)
        planes = qz.quantize(data)
        torch.cuda.synchronize()
        check_quantize(oracle_params(qz), f64(data), planes)


def test_empty_and_bf16_dequant(tq):
    qz = tq.Quantizer(128, 4, "mse", seed=2)
    x = synthetic.gaussian((0, 128), seed=1).cuda()
    planes = qz.quantize(x)
    assert planes["norm"].numel() == 0
    x = synthetic.gaussian((257, 128), seed=1).cuda()
    planes = qz.quantize(x)
    y32 = qz.dequantize(planes)
    y16 = qz.dequantize(planes, dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.allclose(y16.float(), y32, rtol=1e-2, atol=1e-2)


def test_params_match_oracle(tq):
    for d, b, v in [(128, 3, "prod"), (256, 4, "mse"), (64, 1, "prod")]:
        qz = tq.Quantizer(d, b, v, seed=77)
        got = qz.params()
        p = oracle_params(qz)
        assert np.max(np.abs(got["Pi"] - p.Pi)) <= 1e-12
        assert np.max(np.abs(got["centroids"] - p.centroids)) <= 1e-12
        if v == "prod":
            assert np.max(np.abs(got["S"] - p.S)) <= 1e-12


def test_abi_rejects_bad_arguments(tq):
    from kv_cache_vector_18_b300 import _lib
    qz = tq.Quantizer(128, 3, "mse", seed=1)
    x = torch.zeros((16, 128), dtype=torch.bfloat16, device="cuda")
    planes = qz.empty_planes(16)
    L = _lib.lib()
    st = qz.planes_struct(planes)
    # host pointer instead of device memory
    hx = torch.zeros((16, 128), dtype=torch.bfloat16)
    assert L.tq_quantize(qz.handle, hx.data_ptr(), 0, 16, 128, st, None) == _lib.TQ_EINVAL
    # misaligned pointer
    assert L.tq_quantize(qz.handle, x.data_ptr() + 2, 0, 15, 128, st, None) == _lib.TQ_EALIGN
    # stride smaller than d, bad dtype, negative rows
    assert L.tq_quantize(qz.handle, x.data_ptr(), 0, 16, 64, st, None) == _lib.TQ_EINVAL
    assert L.tq_quantize(qz.handle, x.data_ptr(), 7, 16, 128, st, None) == _lib.TQ_EINVAL
    assert L.tq_quantize(qz.handle, x.data_ptr(), 0, -1, 128, st, None) == _lib.TQ_EINVAL
    # missing plane
    bad = _lib.Planes(planes["codes"].data_ptr(), None, None, None)
    assert L.tq_quantize(qz.handle, x.data_ptr(), 0, 16, 128, bad, None) == _lib.TQ_EINVAL
    assert L.tq_quantize(None, x.data_ptr(), 0, 16, 128, st, None) == _lib.TQ_EINVAL
    assert len(L.tq_last_error()) > 0
    torch.cuda.synchronize()


def test_bounded_wait_timeout_reports_status(tq):
    # A block waits on an mbarrier that nothing completes.  The bounded wait (the one
    # every quantize pipeline stage uses) gives up after 50 ms, records the code in the
    # status word and returns; the context stays usable and later work is unaffected.
    from kv_cache_vector_18_b300 import _lib
    qz = tq.Quantizer(128, 3, "mse", seed=3)
    assert qz.device_status() == 0
    L = _lib.lib()
    assert L.tq_check_wait_timeout(qz.handle, 0, 50_000_000, None) == _lib.TQ_EINVAL
    assert L.tq_check_wait_timeout(qz.handle, 99, 0, None) == _lib.TQ_EINVAL
    assert L.tq_check_wait_timeout(qz.handle, 99, 2_000_000_000, None) == _lib.TQ_EINVAL
    assert L.tq_check_wait_timeout(None, 99, 50_000_000, None) == _lib.TQ_EINVAL
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    qz.check_wait_timeout(99, 50_000_000)
    t1.record()
    torch.cuda.synchronize()
    assert 45.0 <= t0.elapsed_time(t1) < 1000.0
    assert qz.device_status(clear=False) == 99
    assert qz.device_status(clear=True) == 99
    assert qz.device_status() == 0
    # the handle still quantizes correctly after the timeout
    n = 148 * 128 + 33
    x = synthetic.gaussian((n, 128), seed=5).cuda()
    planes = qz.quantize(x)
    torch.cuda.synchronize()
    assert qz.device_status() == 0
    rows = np.concatenate([np.arange(0, 200), np.arange(n - 200, n)])
    check_quantize(oracle_params(qz), f64(x), planes, rows=rows)


@pytest.mark.parametrize("variant", ["mse", "prod"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_tensor_core_path_many_tiles(tq, d, bits, variant):
    # enough rows for several tiles per CTA on every SM, plus a ragged tail
    n = 148 * 128 * 3 + 77
    qz = tq.Quantizer(d, bits, variant, seed=7 + bits)
    x = synthetic.gaussian((n, d), seed=bits + d).cuda()
    planes = qz.quantize(x)
    torch.cuda.synchronize()
    assert qz.device_status() == 0
    rows = np.concatenate([np.arange(0, 300), np.arange(n - 300, n),
                           np.random.default_rng(0).choice(n, 3000, replace=False)])
    check_quantize(oracle_params(qz), f64(x), planes, rows=rows)
    # repeat into the same planes: results must be identical
    codes0 = planes["codes"].clone()
    signs0 = planes["signs"].clone() if variant == "prod" else None
    qz.quantize(x, out=planes)
    torch.cuda.synchronize()
    assert torch.equal(codes0, planes["codes"])
    if variant == "prod":
        assert torch.equal(signs0, planes["signs"])


@pytest.mark.parametrize("rotation", ["qr", "hadamard"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_tensor_core_path_fp32_rows(tq, d, bits, rotation):
    # fp32 rows on the tensor-core mse path (each row split into bf16 hi + lo on
    # the device): several tiles per CTA, a ragged tail, a row stride wider than
    # d and two all-zero rows
    n = 148 * 128 * 2 + 45
    qz = tq.Quantizer(d, bits, "mse", seed=31 + bits, rotation=rotation)
    base = synthetic.student_t_unit_var((n, d + 32), seed=bits * 3 + d, dtype="f32").cuda()
    base[5] = 0
    base[n - 1] = 0
    x = base[:, :d]
    planes = qz.quantize(x)
    torch.cuda.synchronize()
    assert qz.device_status() == 0
    rows = np.concatenate([np.arange(0, 300), np.arange(n - 300, n),
                           np.random.default_rng(1).choice(n, 3000, replace=False)])
    check_quantize(oracle_params(qz), f64(x), planes, rows=rows)
    codes = planes["codes"].cpu().numpy()
    assert np.all(codes[5] == 0) and np.all(codes[n - 1] == 0)
    assert planes["norm"][5].item() == 0


@pytest.mark.parametrize("case", [
    # (d, bits K, variant K, bits V, variant V, rotation, dtype, K rows, V rows): one launch
    (128, 3, "mse", 3, "mse", "qr", "bf16", 148 * 128 * 2 + 77, 148 * 128 * 2 + 77),
    (64, 2, "mse", 2, "mse", "hadamard", "bf16", 5000, 300001),
    (128, 4, "mse", 4, "mse", "qr", "f32", 20000, 777),
    (128, 1, "mse", 1, "mse", "qr", "bf16", 1, 1),
    (128, 3, "mse", 3, "mse", "qr", "bf16", 0, 4000),
    # two launches: prod keys, d = 256, different bits
    (128, 3, "prod", 3, "mse", "qr", "bf16", 3000, 3000),
    (256, 2, "mse", 2, "mse", "qr", "bf16", 1000, 1000),
    (128, 4, "mse", 2, "mse", "qr", "bf16", 2000, 2000),
])
def test_quantize_kv_matches_separate_calls(tq, case):
    # tq_quantize_kv (K and V in one launch where the pair allows it) writes the
    # same bytes as two tq_quantize calls; those are checked against the oracle
    d, bk, vk, bv, vv, rot, dt, nk, nv = case
    kq = tq.Quantizer(d, bk, vk, seed=101, rotation=rot)
    vq = tq.Quantizer(d, bv, vv, seed=102, rotation=rot)
    K = synthetic.gaussian((nk, d), seed=11, dtype=dt).cuda()
    V = synthetic.student_t_unit_var((nv, d), seed=12, dtype=dt).cuda()
    kc, vc = tq.quantize_kv(kq, vq, K, V)
    ks, vs = kq.quantize(K), vq.quantize(V)
    torch.cuda.synchronize()
    assert kq.device_status() == 0 and vq.device_status() == 0
    for got, ref in ((kc, ks), (vc, vs)):
        for name in ref:
            assert torch.equal(got[name], ref[name]), name
    rows = np.unique(np.concatenate([np.arange(0, min(nv, 200)), np.arange(max(nv - 200, 0), nv)]))
    if nv:
        check_quantize(oracle_params(vq), f64(V), vc, rows=rows)


def test_quantize_kv_rejects_bad_arguments(tq):
    from kv_cache_vector_18_b300 import _lib
    kq = tq.Quantizer(128, 3, "mse", seed=1)
    vq = tq.Quantizer(128, 3, "mse", seed=2)
    x = torch.zeros((16, 128), dtype=torch.bfloat16, device="cuda")
    kp, vp = kq.empty_planes(16), vq.empty_planes(16)
    L = _lib.lib()
    ks, vs = kq.planes_struct(kp), vq.planes_struct(vp)
    assert L.tq_quantize_kv(kq.handle, vq.handle, x.data_ptr(), x.data_ptr() + 2, 0, 16, 15, 128, 128, ks, vs,
                            None) == _lib.TQ_EALIGN
    assert L.tq_quantize_kv(kq.handle, None, x.data_ptr(), x.data_ptr(), 0, 16, 16, 128, 128, ks, vs,
                            None) == _lib.TQ_EINVAL
    assert L.tq_quantize_kv(kq.handle, vq.handle, x.data_ptr(), x.data_ptr(), 0, 16, 16, 128, 64, ks, vs,
                            None) == _lib.TQ_EINVAL
    torch.cuda.synchronize()
