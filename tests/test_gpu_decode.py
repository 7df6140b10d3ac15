"""CUDA decode attention over the packed cache vs the oracle (needs a GPU).

The oracle gets the GPU's own packed cache (unpacked) so that the comparison
checks the attention path alone; the codec itself is checked in test_gpu_codec.
"""
import math

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


def _run(tq, B, Hq, Hkv, T, d, kb, kv, vb, vv, lens, seed=0, dist="gauss", needle=None, q_dtype="bf16",
         scale=None, return_scores=False):
    gen = synthetic.gaussian if dist == "gauss" else synthetic.student_t_unit_var
    K = gen((B, Hkv, T, d), seed=seed + 1)
    V = gen((B, Hkv, T, d), seed=seed + 2)
    q = gen((B, Hq, d), seed=seed + 3, dtype=q_dtype)
    if needle is not None:
        K = synthetic.plant_needles(K, q, needle["pos"], needle["strength"], Hq // Hkv)
    kq = tq.Quantizer(d, kb, kv, seed=seed + 11)
    vq = tq.Quantizer(d, vb, vv, seed=seed + 12)
    kc = kq.quantize(K.cuda().reshape(-1, d))
    vc = vq.quantize(V.cuda().reshape(-1, d))
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    res = tq.decode_attention(kq, vq, q.cuda(), kc, vc, sl, Hkv, T, scale=scale, return_scores=return_scores)
    torch.cuda.synchronize()
    pk, pv = oracle_params(kq), oracle_params(vq)
    ref_out, ref_sc = O.decode_attention(pk, pv, f64(q), planes_to_oracle_rows(pk, kc),
                                         planes_to_oracle_rows(pv, vc), lens, Hkv, T, scale=scale)
    if return_scores:
        out, sc = res
        return f64(out), ref_out, f64(sc), ref_sc
    return f64(res), ref_out


@pytest.mark.parametrize("kv,kb", [("prod", 3), ("mse", 3), ("prod", 4), ("mse", 2), ("prod", 1)])
@pytest.mark.parametrize("vv,vb", [("mse", 3), ("mse", 2), ("prod", 3)])
def test_decode_variants(tq, kv, kb, vv, vb):
    g, r = _run(tq, B=2, Hq=8, Hkv=2, T=700, d=128, kb=kb, kv=kv, vb=vb, vv=vv, lens=[700, 333], seed=kb * 7 + vb)
    check_attention(g, r)


@pytest.mark.parametrize("d", [32, 64, 256])
def test_decode_head_dims(tq, d):
    g, r = _run(tq, B=1, Hq=4, Hkv=1, T=513, d=d, kb=3, kv="prod", vb=3, vv="mse", lens=[513], seed=d)
    check_attention(g, r)


@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (16, 1), (32, 8), (12, 4)])
def test_decode_group_sizes(tq, Hq, Hkv):
    g, r = _run(tq, B=1, Hq=Hq, Hkv=Hkv, T=300, d=128, kb=4, kv="prod", vb=2, vv="mse", lens=[300], seed=Hq)
    check_attention(g, r)


def test_decode_edge_lengths(tq):
    # empty context, one token, a partial chunk, full capacity
    g, r = _run(tq, B=4, Hq=8, Hkv=2, T=1000, d=128, kb=3, kv="prod", vb=3, vv="mse", lens=[0, 1, 65, 1000])
    check_attention(g, r)
    assert np.all(g[0] == 0)


@pytest.mark.parametrize("T,lens", [(701, [701, 333, 1, 0]), (1002, [1002, 999, 16, 17])])
def test_decode_slabs_not_16_byte_aligned(tq, T, lens):
    # T_max % 4 != 0: slab norm rows start off 16-byte boundaries, so tiles are
    # staged by per-lane copies instead of bulk copies; prod values on the second
    g, r = _run(tq, B=4, Hq=16, Hkv=2, T=T, d=128, kb=3, kv="prod", vb=3, vv="mse" if T == 701 else "prod",
                lens=lens, seed=T)
    check_attention(g, r)


@pytest.mark.parametrize("vv", ["mse", "prod"])
def test_decode_bulk_staging_tail_rows(tq, vv):
    # T_max % 16 == 4: the last tile of a slab copies only 4 rows; lengths end
    # inside tiles so the rows past each chunk are masked
    g, r = _run(tq, B=3, Hq=8, Hkv=2, T=1028, d=128, kb=4, kv="prod", vb=2, vv=vv, lens=[1028, 1027, 515],
                seed=11)
    check_attention(g, r)


def test_decode_needle(tq):
    # planted keys aligned with the query make the softmax peak, so 2e-3 max-abs bites
    g, r = _run(tq, B=1, Hq=8, Hkv=1, T=4096, d=128, kb=3, kv="prod", vb=3, vv="mse", lens=[4096],
                needle={"pos": [17, 2500], "strength": 40.0}, seed=5)
    check_attention(g, r)
    assert np.max(np.abs(r)) > 0.2  # the needle dominates


def test_decode_heavy_tailed_fp32_query_and_scale(tq):
    g, r = _run(tq, B=2, Hq=4, Hkv=2, T=400, d=128, kb=4, kv="prod", vb=2, vv="mse", lens=[400, 250],
                dist="t", q_dtype="f32", scale=0.2, seed=8)
    check_attention(g, r)


def test_scores_output_small_config(tq):
    # 64 fp32 queries scored against 4096 keys (mse b=2, d=128)
    g, r, gs, rs = _run(tq, B=1, Hq=64, Hkv=1, T=4096, d=128, kb=2, kv="mse", vb=2, vv="mse", lens=[4096],
                        q_dtype="f32", return_scores=True, seed=0)
    check_attention(g, r)
    assert np.max(np.abs(gs - rs)) <= 1e-3 * max(1.0, np.max(np.abs(rs)))


@pytest.mark.parametrize("Hq,Hkv,T,lens,vv", [
    (8, 2, 1002, [1002, 517], "mse"),    # four query heads per KV head, per-lane staging (T % 4 != 0)
    (6, 2, 1000, [999, 20], "prod"),      # three, bulk staging, prod values
    (2, 2, 701, [701, 1], "mse"),         # one
])
def test_scores_output_small_groups(tq, Hq, Hkv, T, lens, vv):
    # pre-softmax scores and outputs of the keys-as-A step (at most four query heads
    # per KV head), fp32 queries, ragged tails
    g, r, gs, rs = _run(tq, B=2, Hq=Hq, Hkv=Hkv, T=T, d=128, kb=3, kv="prod", vb=3, vv=vv, lens=lens,
                        q_dtype="f32", return_scores=True, seed=Hq + T)
    check_attention(g, r)
    for b, L in enumerate(lens):
        assert np.max(np.abs(gs[b, :, :L] - rs[b, :, :L])) <= 1e-3 * max(1.0, np.max(np.abs(rs[b, :, :L])))


@pytest.mark.parametrize("kb", [1, 2])
def test_decode_low_bit_prod_keys_heavy_tailed(tq, kb):
    # prod keys of 1 and 2 bits, where the QJL term is all or most of the score,
    # on heavy-tailed rows with eight query heads per KV head: the score path's
    # precision (Q″ as f16 hi + lo) is what keeps these inside the bound
    g, r = _run(tq, B=2, Hq=16, Hkv=2, T=2000, d=128, kb=kb, kv="prod", vb=3, vv="mse", lens=[2000, 1500],
                dist="t", seed=kb * 10)
    check_attention(g, r)


def test_decode_workspace_too_small(tq):
    from kv_cache_vector_18_b300 import _lib
    kq = tq.Quantizer(128, 3, "prod", seed=1)
    vq = tq.Quantizer(128, 3, "mse", seed=2)
    K = synthetic.gaussian((256, 128), seed=1).cuda()
    kc, vc = kq.quantize(K), vq.quantize(K)
    q = synthetic.gaussian((1, 8, 128), seed=2).cuda()
    sl = torch.tensor([256], dtype=torch.int32, device="cuda")
    need = tq.decode_workspace_bytes(kq, vq, 1, 8, 1, 256)
    ws = torch.empty(need // 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(tq.TQError) as e:
        tq.decode_attention(kq, vq, q, kc, vc, sl, 1, 256, workspace=ws)
    assert e.value.code == _lib.TQ_EWORKSPACE
    with pytest.raises(tq.TQError):
        tq.decode_attention(kq, vq, q, kc, vc, sl, 3, 256)  # Hq not a multiple of Hkv


def test_end_to_end_against_oracle_codes(tq):
    # The oracle quantizes the raw K and V rows itself and attends over its own
    # codes; the GPU quantizes and attends over its packed cache.  Reported next to
    # the comparison on the GPU's packed cache.  The two differ only where a
    # coordinate lies within the code window of a boundary and the two precisions
    # decide it differently; for a prod key such a code also changes its residual,
    # so about a fifth of that row's sketch signs flip with it and that key's score
    # moves by up to a few tenths.  So the bound here is loose: what is checked
    # exactly is that every disagreement is such a near-boundary decision.
    B, Hq, Hkv, T, d = 2, 16, 2, 1500, 128
    lens = [1500, 977]
    K = synthetic.gaussian((B, Hkv, T, d), seed=71)
    V = synthetic.gaussian((B, Hkv, T, d), seed=72)
    q = synthetic.gaussian((B, Hq, d), seed=73)
    kq = tq.Quantizer(d, 3, "prod", seed=81)
    vq = tq.Quantizer(d, 3, "mse", seed=82)
    kc = kq.quantize(K.cuda().reshape(-1, d))
    vc = vq.quantize(V.cuda().reshape(-1, d))
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = f64(tq.decode_attention(kq, vq, q.cuda(), kc, vc, sl, Hkv, T))
    pk, pv = oracle_params(kq), oracle_params(vq)
    ref_cache, _ = O.decode_attention(pk, pv, f64(q), planes_to_oracle_rows(pk, kc), planes_to_oracle_rows(pv, vc),
                                      lens, Hkv, T)
    check_attention(out, ref_cache)
    Kf, Vf = f64(K).reshape(-1, d), f64(V).reshape(-1, d)
    check_quantize(pk, Kf, kc)  # every code and sign disagreement is inside the window
    check_quantize(pv, Vf, vc)
    ko = O.quantize(pk, Kf)
    vo = O.quantize(pv, Vf)
    ref_own, _ = O.decode_attention(pk, pv, f64(q), ko, vo, lens, Hkv, T)
    gk, gv = planes_to_oracle_rows(pk, kc), planes_to_oracle_rows(pv, vc)
    k_rows = int(np.sum(np.any(gk["idx"] != ko["idx"], axis=1)))
    s_rows = int(np.sum(np.any(gk["z"] != ko["z"], axis=1)))
    v_rows = int(np.sum(np.any(gv["idx"] != vo["idx"], axis=1)))
    e_cache = np.max(np.abs(out - ref_cache))
    e_own = np.max(np.abs(out - ref_own))
    l2_own = np.linalg.norm(out - ref_own) / np.linalg.norm(ref_own)
    print(f"end to end: max-abs {e_cache:.2e} against the oracle on the GPU's packed cache, {e_own:.2e} "
          f"(rel-L2 {l2_own:.2e}) against the oracle on its own codes; rows whose codes differ: K {k_rows}, "
          f"K signs {s_rows}, V {v_rows} of {K.shape[0] * K.shape[1] * K.shape[2]}")
    assert e_own <= 5e-2 and l2_own <= 5e-2


def test_decode_launched_behind_quantize_reads_its_codes(tq):
    # The decode is a programmatic dependent (through the ticket clearing kernel)
    # of the quantize launched just before it, so its prologue overlaps the
    # quantize; it must still read only what that quantize wrote.  Outputs of
    # unsynchronised quantize → decode sequences equal those of the same calls
    # with a synchronisation in between, bit for bit (the decode's arithmetic and
    # merge order are fixed).
    B, Hq, Hkv, T, d = 1, 64, 8, 32768, 128
    kq = tq.Quantizer(d, 3, "mse", seed=91)
    vq = tq.Quantizer(d, 3, "mse", seed=92)
    X = [synthetic.gaussian((B * Hkv * T, d), seed=s).cuda() for s in (1, 2, 3, 4)]
    q = synthetic.gaussian((B, Hq, d), seed=5).cuda()
    sl = torch.tensor([T], dtype=torch.int32, device="cuda")
    kc, vc = kq.empty_planes(B * Hkv * T), vq.empty_planes(B * Hkv * T)

    def step(k, v, sync):
        tq.quantize_kv(kq, vq, k, v, k_out=kc, v_out=vc)
        if sync:
            torch.cuda.synchronize()
        return tq.decode_attention(kq, vq, q, kc, vc, sl, Hkv, T)

    ref_a = step(X[0], X[1], True)
    ref_b = step(X[2], X[3], True)
    torch.cuda.synchronize()
    outs = [step(X[2 * (i % 2)], X[2 * (i % 2) + 1], False) for i in range(6)]
    torch.cuda.synchronize()
    assert kq.device_status() == 0 and vq.device_status() == 0
    assert not torch.equal(ref_a, ref_b)
    for i, o in enumerate(outs):
        assert torch.equal(o, ref_a if i % 2 == 0 else ref_b), i


def test_mixed_decode_launched_behind_quantize_reads_its_codes(tq):
    # as above for the mixed-precision pair (one-launch K+V quantize, tensor-core decode)
    B, Hq, Hkv, T, d = 1, 64, 8, 32768, 128
    X = [synthetic.gaussian((B * Hkv * T, d), seed=s).cuda() for s in (11, 12, 13, 14)]
    pk = torch.as_tensor(np.random.default_rng(1).permutation(d), dtype=torch.int32, device="cuda")
    pv = torch.as_tensor(np.random.default_rng(2).permutation(d), dtype=torch.int32, device="cuda")
    mk = tq.MixedQuantizer(pk, 32, 3, 2, "mse", seed_o=1, seed_n=2)
    mv = tq.MixedQuantizer(pv, 32, 3, 2, "mse", seed_o=3, seed_n=4)
    q = synthetic.gaussian((B, Hq, d), seed=15).cuda()
    sl = torch.tensor([T], dtype=torch.int32, device="cuda")
    kc, vc = mk.empty_planes(B * Hkv * T), mv.empty_planes(B * Hkv * T)

    def step(k, v, sync):
        tq.mixed_quantize_kv(mk, mv, k, v, kc, vc)
        if sync:
            torch.cuda.synchronize()
        return tq.mixed_decode_attention(mk, mv, q, kc, vc, sl, Hkv, T)

    ref_a = step(X[0], X[1], True)
    ref_b = step(X[2], X[3], True)
    torch.cuda.synchronize()
    outs = [step(X[2 * (i % 2)], X[2 * (i % 2) + 1], False) for i in range(6)]
    torch.cuda.synchronize()
    assert mk.qo.device_status() == 0 and mv.qo.device_status() == 0
    assert not torch.equal(ref_a, ref_b)
    for i, o in enumerate(outs):
        assert torch.equal(o, ref_a if i % 2 == 0 else ref_b), i
