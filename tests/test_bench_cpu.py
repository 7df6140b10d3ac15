"""bench.py host logic that needs no GPU: record sizes, the algorithmic byte
model of a step, workload shapes and the traffic records' source check."""
import json
import os

import pytest

import bench
import oracle as O


@pytest.mark.parametrize("variant,sizes", [("mse", [20, 36, 52, 68]), ("prod", [24, 40, 56, 72])])
def test_row_bytes_at_d128(variant, sizes):
    # codes b_m·d/8 + float32 norm (+ signs d/8 + float32 residual norm for prod)
    assert [bench.row_bytes(b, variant, 128) for b in (1, 2, 3, 4)] == sizes
    for b in (1, 2, 3, 4):
        p = O.make_params(128, b, variant, 0)
        extra = 4 + (4 if variant == "prod" else 0)
        assert bench.row_bytes(b, variant, 128) == O.code_bytes_per_row(p) + O.sign_bytes_per_row(p) + extra


def test_traffic_model_of_the_layer_step():
    spec = bench.workload_spec("llama70b_layer_kv_quant")
    assert (spec["B"], spec["Hkv"], spec["T"], spec["d"], spec["Hq"]) == (1, 8, 32768, 128, 64)
    tm = bench.traffic_model(spec, [spec["T"]])
    rows = 8 * 32768
    # quantize: bf16 in (256 B) + 52-byte records out, for K and for V
    assert tm["quant_k"] == tm["quant_v"] == rows * (256 + 52)
    # decode: both records of every cached token, bf16 q in, fp32 out
    assert tm["decode"] == rows * 104 + 64 * 128 * 6
    assert tm["total"] == 188792832
    assert tm["ctx_rows"] == rows


def test_traffic_model_counts_only_live_tokens():
    spec = bench.workload_spec("batched_decode_32k")
    lens = [100, 2000] + [0] * (spec["B"] - 2)
    tm = bench.traffic_model(spec, lens)
    krb, vrb = bench.row_bytes(spec["k_bits"], spec["k_variant"], 128), bench.row_bytes(spec["v_bits"], spec["v_variant"], 128)
    assert (krb, vrb) == (72, 36)
    assert tm["decode"] == 2100 * spec["Hkv"] * (krb + vrb) + spec["B"] * spec["Hq"] * 128 * 6


def test_recorded_traffic_requires_the_same_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps({"k": {"source_hash": "abc", "dram_bytes_per_unit": 2.5}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("k", "abc", 4) == 10.0
    assert bench.recorded_traffic("k", "other", 4) is None
    assert bench.recorded_traffic("missing", "abc", 4) is None


def test_committed_traffic_records_name_their_capture():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for key, r in rec.items():
        assert r["capture"].startswith("ncu ") and "--clock-control none" in r["capture"], key
        assert r["unit"] in ("row", "token-head") and r["dram_bytes_per_unit"] > 0


def test_source_hash_is_stable_and_sensitive(tmp_path, monkeypatch):
    (tmp_path / "a.cu").write_text("x")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.source_hash(["a.cu"])
    assert h == bench.source_hash(["a.cu"]) and len(h) == 16
    (tmp_path / "a.cu").write_text("y")
    assert bench.source_hash(["a.cu"]) != h
