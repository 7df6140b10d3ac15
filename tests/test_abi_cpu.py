"""C ABI checks that need no GPU: the library loads, exports every declared
symbol, and builds the same parameters as the oracle on the host."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    syms = set()
    for name in os.listdir(os.path.join(ROOT, "include")):
        if name.endswith(".h"):
            text = open(os.path.join(ROOT, "include", name)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            syms |= set(re.findall(r"\b(tq_\w+)\s*\(", text))
    return syms


@pytest.fixture(scope="module")
def lib():
    from kv_cache_vector_18_b300 import _lib
    return _lib.lib()


def test_library_exports_every_declared_symbol(lib):
    syms = _declared_symbols()
    assert {"tq_init", "tq_quantize", "tq_dequantize", "tq_decode_attention"} <= syms
    for s in sorted(syms):
        assert hasattr(lib, s), s


def test_binding_declares_every_symbol():
    from kv_cache_vector_18_b300 import _lib
    assert _declared_symbols() == set(_lib.EXPORTED)


@pytest.mark.parametrize("d,b,v", [(32, 1, "mse"), (64, 2, "prod"), (128, 3, "mse"), (128, 3, "prod"),
                                   (128, 4, "prod"), (256, 4, "mse"), (96, 2, "mse"), (128, 1, "prod")])
def test_host_params_match_oracle(d, b, v):
    import kv_cache_vector_18_b300 as tq
    got = tq.build_params_host(d, b, v, seed=1234)
    p = O.make_params(d, b, v, 1234)
    assert np.max(np.abs(got["Pi"] - p.Pi)) <= 1e-12
    assert np.max(np.abs(got["centroids"] - p.centroids)) <= 1e-12
    assert np.max(np.abs(got["bounds"] - p.bounds), initial=0.0) <= 1e-12
    if v == "prod":
        assert np.max(np.abs(got["S"] - p.S)) <= 1e-12


def test_host_params_reject_bad_shapes(lib):
    from kv_cache_vector_18_b300 import _lib
    dp = ctypes.POINTER(ctypes.c_double)
    buf = np.zeros(256 * 256)
    p = buf.ctypes.data_as(dp)
    assert lib.tq_build_params_host(33, 2, 0, 0, p, p, p, p) == _lib.TQ_EUNSUPPORTED
    assert lib.tq_build_params_host(512, 2, 0, 0, p, p, p, p) == _lib.TQ_EUNSUPPORTED
    assert lib.tq_build_params_host(128, 5, 0, 0, p, p, p, p) == _lib.TQ_EUNSUPPORTED
    assert lib.tq_build_params_host(128, 0, 1, 0, p, p, p, p) == _lib.TQ_EUNSUPPORTED
    assert lib.tq_build_params_host(128, 2, 2, 0, p, p, p, p) == _lib.TQ_EINVAL
    assert b"variant" in lib.tq_last_error()


def test_seed_changes_rotation_and_sketch():
    import kv_cache_vector_18_b300 as tq
    a = tq.build_params_host(64, 2, "prod", seed=1)
    b = tq.build_params_host(64, 2, "prod", seed=2)
    assert np.max(np.abs(a["Pi"] - b["Pi"])) > 0.1 and np.max(np.abs(a["S"] - b["S"])) > 0.1
    # Π and S drawn from independent streams of the same seed
    assert abs(np.corrcoef(a["Pi"].ravel(), a["S"].ravel())[0, 1]) < 0.1


@pytest.mark.parametrize("d,b,v", [(32, 1, "mse"), (64, 2, "prod"), (128, 3, "mse"), (128, 3, "prod"),
                                   (256, 4, "mse"), (128, 1, "prod")])
def test_host_hadamard_params_match_oracle(d, b, v):
    # the library builds (H_d)_ji from popcount parity, the oracle by Sylvester recursion
    import kv_cache_vector_18_b300 as tq
    got = tq.build_params_host(d, b, v, seed=99, rotation="hadamard")
    p = O.make_params(d, b, v, 99, rotation="hadamard")
    assert np.max(np.abs(got["Pi"] - p.Pi)) <= 1e-15
    assert np.max(np.abs(got["centroids"] - p.centroids)) <= 1e-12
    if v == "prod":
        assert np.max(np.abs(got["S"] - p.S)) <= 1e-12


def test_host_hadamard_rejects_bad_arguments(lib):
    from kv_cache_vector_18_b300 import _lib
    dp = ctypes.POINTER(ctypes.c_double)
    buf = np.zeros(256 * 256)
    p = buf.ctypes.data_as(dp)
    # not a power of two
    assert lib.tq_build_params_host_ex(96, 2, 0, _lib.TQ_ROT_HADAMARD, 0, p, p, p, p) == _lib.TQ_EUNSUPPORTED
    assert b"power of two" in lib.tq_last_error()
    assert lib.tq_build_params_host_ex(128, 2, 0, 2, 0, p, p, p, p) == _lib.TQ_EINVAL
    assert lib.tq_build_params_host_ex(96, 2, 0, _lib.TQ_ROT_QR, 0, p, p, p, p) == _lib.TQ_OK
    # the plain entry point is the QR rotation
    a, b = np.zeros(64 * 64), np.zeros(64 * 64)
    assert lib.tq_build_params_host(64, 2, 0, 5, a.ctypes.data_as(dp), None, None, None) == _lib.TQ_OK
    assert lib.tq_build_params_host_ex(64, 2, 0, _lib.TQ_ROT_QR, 5, b.ctypes.data_as(dp), None, None, None) == _lib.TQ_OK
    assert np.array_equal(a, b)


def test_new_entry_points_reject_bad_arguments_on_the_host(lib):
    # argument checks run before any CUDA call, so they hold without a GPU
    from kv_cache_vector_18_b300 import _lib
    h = ctypes.c_void_p()
    assert lib.tq_init_ex(128, 3, 0, 7, 0, ctypes.byref(h)) == _lib.TQ_EINVAL       # unknown rotation
    assert lib.tq_init_ex(96, 3, 0, _lib.TQ_ROT_HADAMARD, 0, ctypes.byref(h)) == _lib.TQ_EUNSUPPORTED
    assert not h.value
    assert lib.tq_check_wait_timeout(None, 99, 1000, None) == _lib.TQ_EINVAL
    assert lib.tq_select_outlier_channels(None, 0, 10, 128, 48, 32, None, None, None) == _lib.TQ_EUNSUPPORTED
    assert lib.tq_select_outlier_channels(None, 0, 10, 128, 128, 40, None, None, None) == _lib.TQ_EINVAL
    assert lib.tq_select_outlier_channels(None, 0, 10, 128, 128, 128, None, None, None) == _lib.TQ_EINVAL
    assert lib.tq_select_outlier_channels(None, 5, 10, 128, 128, 32, None, None, None) == _lib.TQ_EINVAL
    P = _lib.Planes()
    assert lib.tq_mixed_quantize(None, None, None, None, 0, 8, 128, P, P, None, 0, None) == _lib.TQ_EINVAL
    assert lib.tq_mixed_dequantize(None, None, None, P, P, 8, None, 0, None) == _lib.TQ_EINVAL
    n = ctypes.c_size_t()
    assert lib.tq_mixed_decode_workspace_bytes(None, None, None, None, 1, 8, 1, 16, ctypes.byref(n)) == _lib.TQ_EINVAL
    assert lib.tq_decode_append_attention(None, None, None, 0, None, None, 0, P, P, None, 1, 8, 1, 16, 0.0, None,
                                          None, 0, None) == _lib.TQ_EINVAL
    assert lib.tq_mixed_quantize_scratch_bytes() == 2 * 128 * 128 * 2
    assert len(lib.tq_last_error()) > 0


def test_binding_constants_match_the_header():
    from kv_cache_vector_18_b300 import _lib
    text = open(os.path.join(ROOT, "include", "tq.h")).read()
    defines = {m.group(1): int(m.group(2))
               for m in re.finditer(r"^#define\s+(TQ_\w+)\s+\(?(-?\d+)\)?\s*(?:/\*.*)?$", text, flags=re.M)}
    assert {"TQ_OK", "TQ_EWORKSPACE", "TQ_STATUS_APPEND_FULL", "TQ_STATUS_BAD_CHANNEL"} <= set(defines)
    for name, value in defines.items():
        assert getattr(_lib, name) == value, name
    assert "#define TQ_NOALLOC_WORKSPACE_BYTES (4u << 20)" in text and _lib.NOALLOC_WORKSPACE_BYTES == 4 << 20
    enums = {}
    for body in re.findall(r"enum\s*\{([^}]*)\}", text):
        for name, value in re.findall(r"(TQ_\w+)\s*=\s*(\d+)", body):
            enums[name] = int(value)
    assert {"TQ_MSE", "TQ_PROD", "TQ_BF16", "TQ_F32", "TQ_ROT_QR", "TQ_ROT_HADAMARD"} <= set(enums)
    for name, value in enums.items():
        assert getattr(_lib, name) == value, name
