"""Pins for the CPU oracle (no GPU): the oracle is checked against things other
than itself -- torch's float8_e4m3fn / bfloat16 conversions (library
routines), the E4M3 format's special values, the scatter worked example of the
scatter_pa_kv_cache_with_k_scale page, brute-force FP64 attention, closed
forms, invariances and a separately written single-pass softmax."""
import dataclasses
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# E4M3 / BF16 codec
# ---------------------------------------------------------------------------

def _torch_e4m3_decode(codes):
    t = torch.from_numpy(np.asarray(codes, dtype=np.uint8).copy())
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_e4m3_encode(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32).copy()).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = _torch_e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(mine[~nan], ref[~nan])
    # signed zero and the largest finite value
    assert math.copysign(1.0, mine[0x80]) == -1.0
    assert mine[0x7E] == 448.0 and mine[0xFE] == -448.0


def test_e4m3_special_values_golden():
    d = json.load(open(os.path.join(GOLDEN, "e4m3_special_values.json")))
    xs = np.array([c["x"] for c in d["cases"]], dtype=np.float32)
    want = np.array([c["code"] for c in d["cases"]], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(xs), want)
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F
    assert oracle.e4m3_encode(np.array([np.inf, -np.inf], np.float32)).tolist() == [0x7E, 0xFE]


def _boundary_floats():
    """Floats with exponents -14..8 whose mantissas sit on, just off and
    exactly between E4M3 grid points (and the subnormal grid)."""
    lows = np.array([0, 1, 0x3FFFF, 0x40000, 0x40001, 0x7FFFF, 0x20000, 0x60000], np.uint32)
    tops = np.arange(16, dtype=np.uint32) << 19
    mant = (tops[:, None] | lows[None, :]).reshape(-1)
    exps = np.arange(127 - 14, 127 + 9, dtype=np.uint32)
    bits = (exps[:, None] << 23 | mant[None, :]).reshape(-1)
    bits = np.concatenate([bits, bits | np.uint32(0x80000000)])
    return bits.view(np.float32)


def test_e4m3_encode_matches_torch_on_grid_boundaries():
    x = _boundary_floats()
    x = x[np.abs(x) < 464.0]   # torch's cast does not saturate; compare below it
    assert np.array_equal(oracle.e4m3_encode(x), _torch_e4m3_encode(x))


def test_e4m3_encode_matches_torch_random():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(400000) * np.exp2(rng.uniform(-14, 9, 400000))).astype(np.float32)
    x = x[np.abs(x) < 464.0]
    assert np.array_equal(oracle.e4m3_encode(x), _torch_e4m3_encode(x))


def test_e4m3_encode_saturates():
    x = np.array([464.0001, 479.9, 480.0, 1000.0, 3.0e38], np.float32)
    assert oracle.e4m3_encode(x).tolist() == [0x7E] * 5
    assert oracle.e4m3_encode(-x).tolist() == [0xFE] * 5


def test_bf16_matches_torch():
    rng = np.random.default_rng(6)
    x = np.concatenate([
        (rng.standard_normal(200000) * np.exp2(rng.uniform(-30, 30, 200000))).astype(np.float32),
        _boundary_floats(),
        np.array([0.0, -0.0, 1.0, 65504.0, 3.0e38], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_from_float(x), ref)


# ---------------------------------------------------------------------------
# Quantisers
# ---------------------------------------------------------------------------

def test_quant_rows_definition():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((300, 128)).astype(np.float32)
    x[7] *= 1e-3
    x[8] = 0.0
    codes, scale = oracle.quant_rows(x)
    amax = np.abs(x).max(axis=1)
    # dequant scale is amax / 448 in FP32 (IEEE division)
    assert np.array_equal(scale, (amax / np.float32(448.0)).astype(np.float32))
    nz = amax > 0
    # the amax element encodes to +-448
    i = np.abs(x).argmax(axis=1)
    top = codes[np.arange(300), i]
    assert np.all((top[nz] & 0x7F) == 0x7E)
    # every code is the library's nearest E4M3 of x / scale
    ref = _torch_e4m3_encode(x[nz] / scale[nz, None])
    assert np.array_equal(codes[nz], ref)
    # all-zero row: scale 0, codes 0
    assert scale[8] == 0.0 and not codes[8].any()


def test_value_channel_scale_and_codes():
    rng = np.random.default_rng(8)
    cu = np.array([0, 5, 5, 40], np.int64)
    v = rng.standard_normal((40, 2, 128)).astype(np.float32)
    vs = oracle.value_channel_scale(v, cu, 3)
    for b in range(3):
        seg = v[cu[b]:cu[b + 1]]
        amax = np.abs(seg).max(axis=0) if len(seg) else np.zeros((2, 128), np.float32)
        assert np.array_equal(vs[b], (amax / np.float32(448.0)).astype(np.float32))
    tb = np.repeat(np.arange(3, dtype=np.int32), np.diff(cu))
    codes = oracle.quant_channels(v, tb, vs)
    ref = _torch_e4m3_encode(v / vs[tb])
    assert np.array_equal(codes, ref)
    # per channel the amax element hits 448 exactly
    seg = codes[5:40]
    mx = (seg & 0x7F).max(axis=0)
    assert np.all(mx == 0x7E)


# ---------------------------------------------------------------------------
# Scatter
# ---------------------------------------------------------------------------

def test_scatter_worked_example():
    d = json.load(open(os.path.join(GOLDEN, "scatter_worked_example.json")))
    T, H, Dk, Dv = d["num_tokens"], d["num_head"], d["k_head_size"], d["v_head_size"]
    NB, BS = d["num_blocks"], d["block_size"]
    rng = np.random.default_rng(9)
    key = rng.integers(1, 255, (T, H, Dk), dtype=np.uint8)
    val = rng.integers(1, 255, (T, H, Dv), dtype=np.uint8)
    ks = rng.standard_normal((T, H)).astype(np.float32)
    kc = np.zeros((NB, H, BS, Dk), np.uint8)
    vc = np.zeros((NB, H, BS, Dv), np.uint8)
    ksc = np.zeros((NB, H, BS, 1), np.float32)
    oracle.cache_scatter(key, val, kc, vc, np.array(d["slot_mapping"]), ks, ksc,
                         layout=oracle.LAYOUT_BNBD)
    written = np.zeros((NB, BS), bool)
    for i, (blk, off) in enumerate(d["expected_block_offset"]):
        assert np.array_equal(kc[blk, :, off, :], key[i])
        assert np.array_equal(vc[blk, :, off, :], val[i])
        assert np.array_equal(ksc[blk, :, off, 0], ks[i])
        written[blk, off] = True
    for blk in range(NB):
        for off in range(BS):
            if not written[blk, off]:
                assert not kc[blk, :, off].any() and not vc[blk, :, off].any()
                assert not ksc[blk, :, off].any()


@pytest.mark.parametrize("layout", [oracle.LAYOUT_BSND, oracle.LAYOUT_BNBD])
def test_scatter_skips_invalid_slots_and_keeps_rest(layout):
    rng = np.random.default_rng(10)
    T, H, D, NB, BS = 6, 3, 16, 3, 8
    key = rng.integers(0, 256, (T, H, D), dtype=np.uint8)
    val = rng.integers(0, 256, (T, H, D), dtype=np.uint8)
    ks_full = rng.standard_normal((T, 2 * H)).astype(np.float32)
    ks = ks_full[:, ::2]               # non-contiguous tail
    shape = (NB, H, BS, D) if layout == oracle.LAYOUT_BNBD else (NB, BS, H, D)
    kc = rng.integers(0, 256, shape, dtype=np.uint8)
    vc = rng.integers(0, 256, shape, dtype=np.uint8)
    ksc = rng.standard_normal(shape[:3] + (1,)).astype(np.float32)
    kc0, vc0, ksc0 = kc.copy(), vc.copy(), ksc.copy()
    slots = np.array([-1, 3, NB * BS, 17, -5, NB * BS - 1], np.int64)
    oracle.cache_scatter(key, val, kc, vc, slots, ks, ksc, layout=layout)
    expect_k, expect_v, expect_s = kc0.copy(), vc0.copy(), ksc0.copy()
    for i, s in enumerate(slots):
        if s < 0 or s >= NB * BS:
            continue
        blk, off = s // BS, s % BS
        for j in range(H):
            idx = (blk, j, off) if layout == oracle.LAYOUT_BNBD else (blk, off, j)
            expect_k[idx] = key[i, j]
            expect_v[idx] = val[i, j]
            expect_s[idx] = ks[i, j]
    assert np.array_equal(kc, expect_k)
    assert np.array_equal(vc, expect_v)
    assert np.array_equal(ksc, expect_s)


def test_quant_scatter_matches_quant_then_scatter():
    rng = np.random.default_rng(11)
    T, H, D, NB, BS = 5, 2, 128, 2, 16
    k = torch.from_numpy(rng.standard_normal((T, H, D)).astype(np.float32)).to(
        torch.bfloat16).float().numpy()
    v = torch.from_numpy(rng.standard_normal((T, H, D)).astype(np.float32)).to(
        torch.bfloat16).float().numpy()
    vscale = (np.abs(rng.standard_normal((3, H, D))) / 200).astype(np.float32)
    tb = np.array([0, 1, 2, 1, 0], np.int32)
    slots = np.array([3, -1, 20, 31, 0], np.int64)
    kc = np.zeros((NB, H, BS, D), np.uint8)
    vc = np.zeros((NB, H, BS, D), np.uint8)
    ksc = np.zeros((NB, H, BS, 1), np.float32)
    oracle.cache_quant_scatter(k, v, kc, vc, slots, ksc, vscale, tb)
    # independent composition: library E4M3 cast of k / (amax/448), v / vscale
    for i, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = s // BS, s % BS
        for j in range(H):
            amax = np.abs(k[i, j]).max()
            sc = np.float32(amax) / np.float32(448.0)
            assert ksc[blk, j, off, 0] == sc
            assert np.array_equal(kc[blk, j, off], _torch_e4m3_encode(k[i, j] / sc))
            want_v = np.clip(v[i, j] / vscale[tb[i], j], -448, 448)
            assert np.array_equal(vc[blk, j, off], _torch_e4m3_encode(want_v))
    assert not kc[0, :, 1].any()   # untouched slot


# ---------------------------------------------------------------------------
# Decode attention
# ---------------------------------------------------------------------------

def build_inputs(case):
    """Quantise a workload with the oracle and lay it out in the paged cache
    (cache placement done here with numpy indexing, not by the oracle)."""
    q32 = case.q()
    k32, v32 = case.kv()
    q8, qs = oracle.quant_rows(q32)
    k8, ks = oracle.quant_rows(k32)
    vs = oracle.value_channel_scale(v32, case.cu_seqlens, case.B)
    v8 = oracle.quant_channels(v32, case.token_batch, vs)
    NB, BS, H, D = case.num_blocks, case.BS, case.NKV, case.D
    slots = case.slots
    blk, off = slots // BS, slots % BS
    if case.layout == workloads.LAYOUT_BSND:
        kc = np.zeros((NB, BS, H, D), np.uint8)
        vc = np.zeros((NB, BS, H, D), np.uint8)
        ksc = np.zeros((NB, BS, H), np.float32)
        kc[blk, off] = k8
        vc[blk, off] = v8
        ksc[blk, off] = ks
    else:
        kc = np.zeros((NB, H, BS, D), np.uint8)
        vc = np.zeros((NB, H, BS, D), np.uint8)
        ksc = np.zeros((NB, H, BS), np.float32)
        kc[blk, :, off] = k8
        vc[blk, :, off] = v8
        ksc[blk, :, off] = ks
    return dict(q8=q8, qs=qs, kc=kc, ksc=ksc, vc=vc, vs=vs, k8=k8, ks=ks, v8=v8)


def run_oracle(case, inp, **kw):
    return oracle.pa_decode(inp["q8"], inp["qs"], inp["kc"], inp["ksc"], inp["vc"], inp["vs"],
                            case.block_table, case.act, S1=case.S1, NKV=case.NKV,
                            layout=case.layout, s2_tile=kw.pop("s2_tile", case.s2_tile),
                            softmax_scale=case.softmax_scale, **kw)


def brute_force(case, q, k, v, with_abs=False):
    """FP64 softmax(q k^T * scale) v per row, from per-token arrays. With
    ``with_abs`` also returns softmax(...) |v| (the weight of |v| per row)."""
    cu = case.cu_seqlens
    B, S1, NQ, G = case.B, case.S1, case.NQ, case.group
    out = np.zeros((B * S1, NQ, case.D))
    wabs = np.zeros((B * S1, NQ, case.D))
    for b in range(B):
        kb = k[cu[b]:cu[b + 1]].astype(np.float64)
        vb = v[cu[b]:cu[b + 1]].astype(np.float64)
        if len(kb) == 0:
            continue
        for s in range(S1):
            for h in range(NQ):
                n2 = h // G
                sc = kb[:, n2] @ q[b * S1 + s, h].astype(np.float64) * case.softmax_scale
                p = np.exp(sc - sc.max())
                out[b * S1 + s, h] = (p / p.sum()) @ vb[:, n2]
                wabs[b * S1 + s, h] = (p / p.sum()) @ np.abs(vb[:, n2])
    return (out, wabs) if with_abs else out


def p_quant_bound(ref, wabs):
    """Error bound of the quantised pipeline against exact attention on the
    dequantised inputs: each P_j is rounded to E4M3 with relative error at
    most 2^-4 (3 mantissa bits, round to nearest) while the sum uses the
    unrounded P, so |err| <= 2^-4 * sum_j p_j |v_j|; plus the BF16 cast
    (2^-8 relative) and FP32 slack."""
    return wabs / 16.0 + np.abs(ref) * 2.0 ** -8 + 1e-6


def small_gqa(layout=workloads.LAYOUT_BSND, s2_tile=128):
    return workloads.custom("small", 2, 1, 8, 2, [200, 517], max_blocks=6, layout=layout,
                            s2_tile=s2_tile)


@pytest.mark.parametrize("mk", [lambda: workloads.tiny(s2_tile=128),
                                lambda: workloads.tiny(s2_tile=512),
                                lambda: small_gqa(workloads.LAYOUT_BSND),
                                lambda: small_gqa(workloads.LAYOUT_BNBD, 256)])
def test_decode_vs_bruteforce_fp64(mk):
    case = mk()
    inp = build_inputs(case)
    out = oracle.bf16_to_float(run_oracle(case, inp)).astype(np.float64)
    k32, v32 = case.kv()
    # (a) unquantised FP64 attention: the quantised pipeline stays within 6e-2
    ref = brute_force(case, case.q(), k32, v32)
    assert np.abs(out - ref).max() < 6e-2
    # (b) FP64 attention on the dequantised inputs: only the P quantisation
    # and the BF16 cast remain
    qd = oracle.e4m3_decode(inp["q8"]) * inp["qs"][..., None]
    kd = oracle.e4m3_decode(inp["k8"]) * inp["ks"][..., None]
    vd = oracle.e4m3_decode(inp["v8"]) * inp["vs"][case.token_batch]
    ref2, wabs = brute_force(case, qd, kd, vd, with_abs=True)
    err = np.abs(out - ref2)
    assert np.all(err <= p_quant_bound(ref2, wabs))


def test_decode_all_equal_keys_gives_mean_of_values():
    case = small_gqa(s2_tile=128)
    inp = build_inputs(case)
    k32, _ = case.kv()
    row = k32[0].copy()
    k8, ks = oracle.quant_rows(np.broadcast_to(row, k32.shape))
    blk, off = case.slots // case.BS, case.slots % case.BS
    inp["kc"][blk, off] = k8
    inp["ksc"][blk, off] = ks
    out, o32 = run_oracle(case, inp, want_f32=True)
    vd = oracle.e4m3_decode(inp["v8"]) * inp["vs"][case.token_batch].astype(np.float64)
    cu = case.cu_seqlens
    for b in range(case.B):
        mean = vd[cu[b]:cu[b + 1]].mean(axis=0)        # [NKV, D]
        for h in range(case.NQ):
            np.testing.assert_allclose(o32[b, h], mean[h // case.group], rtol=2e-5, atol=1e-6)


def test_decode_single_token_gives_that_value_row():
    case = workloads.custom("one", 3, 1, 6, 3, [1, 1, 1], max_blocks=2)
    inp = build_inputs(case)
    out, o32 = run_oracle(case, inp, want_f32=True)
    vd = oracle.e4m3_decode(inp["v8"]) * inp["vs"][case.token_batch].astype(np.float64)
    for b in range(3):
        for h in range(6):
            np.testing.assert_allclose(o32[b, h], vd[b, h // 2], rtol=3e-7, atol=0)


def test_decode_zero_length_gives_zeros():
    case = workloads.custom("zero", 2, 1, 4, 2, [0, 130], max_blocks=2)
    inp = build_inputs(case)
    out = run_oracle(case, inp)
    assert not out[0].any() and out[1].any()


def test_decode_block_table_permutation_invariance():
    case = small_gqa(s2_tile=128)
    inp = build_inputs(case)
    base = run_oracle(case, inp)
    rng = np.random.default_rng(12)
    perm = rng.permutation(case.num_blocks)          # new position of each block
    kc = np.empty_like(inp["kc"]); vc = np.empty_like(inp["vc"]); ksc = np.empty_like(inp["ksc"])
    kc[perm] = inp["kc"]; vc[perm] = inp["vc"]; ksc[perm] = inp["ksc"]
    bt = np.where(case.block_table >= 0, perm[np.maximum(case.block_table, 0)], -1).astype(np.int32)
    inp2 = dict(inp, kc=kc, vc=vc, ksc=ksc)
    case2 = dataclasses.replace(case, block_table=bt)
    assert np.array_equal(run_oracle(case2, inp2), base)


def test_decode_gqa_identical_queries_identical_outputs():
    case = workloads.custom("gqa", 2, 2, 8, 2, [90, 300], max_blocks=3)
    inp = build_inputs(case)
    q8 = inp["q8"].copy(); qs = inp["qs"].copy()
    q8[:, 1:4] = q8[:, :1]; qs[:, 1:4] = qs[:, :1]        # heads 0-3 share kv head 0
    q8[1] = q8[0]; qs[1] = qs[0]                          # s1 rows of batch 0 equal
    out = run_oracle(case, dict(inp, q8=q8, qs=qs))
    for h in range(1, 4):
        assert np.array_equal(out[:, h], out[:, 0])
    assert np.array_equal(out[1], out[0])


def one_pass_reference(case, inp, row):
    """Single-pass (one s2 tile) softmax with per-row FP8 P quantisation,
    written with numpy FP32 arithmetic and torch's E4M3 cast."""
    b, h = divmod(row, case.NQ)
    b //= case.S1
    n2 = h // case.group
    n = int(case.act[b])
    j = np.arange(n)
    blk = np.maximum(case.block_table[b, j // case.BS], 0)
    off = j % case.BS
    kv_idx = (blk, off, n2) if case.layout == workloads.LAYOUT_BSND else (blk, n2, off)
    K = _torch_e4m3_decode(inp["kc"][kv_idx])
    V = _torch_e4m3_decode(inp["vc"][kv_idx])
    ksc = inp["ksc"][kv_idx]
    qd = _torch_e4m3_decode(inp["q8"].reshape(-1, case.D)[row])
    acc = (K @ qd).astype(np.float32)                   # exact sums, one rounding
    S = ((acc * inp["qs"].reshape(-1)[row]) * ksc) * np.float32(case.softmax_scale)
    P = np.exp((S - S.max()).astype(np.float64)).astype(np.float32)
    L = np.float32(0)
    for p in P:
        L = np.float32(L + p)
    qsc = np.float32(448.0) / P.max()
    P8 = _torch_e4m3_decode(_torch_e4m3_encode(P * qsc))
    ot = (P8 @ V).astype(np.float32)
    O = (ot * (np.float32(1.0) / qsc)) * inp["vs"][b, n2]
    return (O / L).astype(np.float32)


def test_decode_one_tile_matches_single_pass_softmax():
    case = workloads.custom("onetile", 3, 1, 4, 2, [37, 129, 300], max_blocks=3)
    inp = build_inputs(case)
    _, o32 = run_oracle(case, inp, s2_tile=512, want_f32=True)
    for row in range(case.B * case.NQ):
        ref = one_pass_reference(case, inp, row)
        np.testing.assert_allclose(o32.reshape(-1, case.D)[row], ref, rtol=2e-6, atol=1e-7)


def test_decode_late_large_score_needs_rescale():
    """A token in the last tile with a much larger score: the running output
    must be rescaled by exp(M_old - M_new) (a dropped rescale gives a grossly
    wrong answer here)."""
    case = workloads.custom("late", 1, 1, 2, 1, [400], max_blocks=4, s2_tile=128)
    inp = build_inputs(case)
    k32, v32 = case.kv()
    k32 = k32.copy()
    k32[350, 0] = case.q()[0, 0] * 3.0
    k8, ks = oracle.quant_rows(k32)
    blk, off = case.slots // case.BS, case.slots % case.BS
    inp["kc"][blk, off] = k8
    inp["ksc"][blk, off] = ks
    inp["k8"], inp["ks"] = k8, ks
    out = oracle.bf16_to_float(run_oracle(case, inp)).astype(np.float64)
    qd = oracle.e4m3_decode(inp["q8"]) * inp["qs"][..., None]
    kd = oracle.e4m3_decode(k8) * ks[..., None]
    vd = oracle.e4m3_decode(inp["v8"]) * inp["vs"][case.token_batch]
    ref, wabs = brute_force(case, qd, kd, vd, with_abs=True)
    assert np.all(np.abs(out - ref) <= p_quant_bound(ref, wabs))


def test_decode_rows_subset_matches_full():
    case = small_gqa(s2_tile=256)
    inp = build_inputs(case)
    full = run_oracle(case, inp)
    rows = np.array([0, 5, 11, 15])
    part = run_oracle(case, inp, rows=rows)
    flat_f, flat_p = full.reshape(-1, 128), part.reshape(-1, 128)
    assert np.array_equal(flat_p[rows], flat_f[rows])
    mask = np.ones(len(flat_p), bool); mask[rows] = False
    assert not flat_p[mask].any()


# ---------------------------------------------------------------------------
# KV compress epilog, modes 0/1 ("CANN ops-transformer aclnnKvCompressEpilog
# 算子详解": 计算公式 场景 1/2, 约束说明, kvCacheCol 的源码级解读)
# ---------------------------------------------------------------------------

def _kvc_run(x, mode, round_scale, *, head_dim=None, block_num=3, block_size=4, slots=None,
             fill=0xA5, stride_pad=0):
    """Run the oracle on rows x (float32 of BF16 values) into a pre-filled
    cache; return the cache and its layout."""
    bs, d = x.shape
    head_dim = head_dim or oracle.kvc_min_head_dim(d, mode)
    stride = block_size * head_dim + stride_pad
    cache = np.full(block_num * stride, fill, np.uint8)
    slots = np.arange(bs) if slots is None else np.asarray(slots)
    oracle.kv_compress_epilog(x, cache, block_num, block_size, stride, head_dim, slots, mode,
                              round_scale)
    return cache, head_dim, stride, block_size


def _kvc_row(cache, slot, head_dim, stride, block_size):
    base = (slot // block_size) * stride + (slot % block_size) * head_dim
    return cache[base:base + head_dim]


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def test_kvc_row_widths_printed_on_the_page():
    """约束说明: d=256 and d=512 with quantMode=1 need headDim >= 323 and 583
    (the page's own examples); mode 0 rounds the row up to 32 bytes."""
    assert oracle.kvc_min_head_dim(256, 1) == 323
    assert oracle.kvc_min_head_dim(512, 1) == 583
    # concatCol = (d-64) + 64*2 + groups * scale bytes
    assert oracle.kvc_concat_bytes(256, 0) == 192 + 128 + 3 * 2
    assert oracle.kvc_min_head_dim(256, 0) == 352


@pytest.mark.parametrize("mode", [0, 1])
def test_kvc_constant_group_closed_form(mode):
    """A group of equal values c: scale c/448, every code E4M3(448) = 0x7E
    (mode 0); with a power-of-two scale 2^ceil(log2(c/448)) the code is
    E4M3(c / 2^k) (mode 1). The rope part is the last 64 columns as BF16."""
    d = 192
    x = np.zeros((1, d), np.float32)
    x[0, :64] = 3.0          # group 0
    x[0, 64:128] = -0.25     # group 1
    x[0, 128:] = _bf16(np.linspace(-2, 2, 64))   # rope
    cache, hd, st, bsz = _kvc_run(x, mode, True)
    row = _kvc_row(cache, 0, hd, st, bsz)
    rope = row[:128].view(np.uint16)
    assert np.array_equal(rope, oracle.bf16_from_float(x[0, 128:]))
    codes = row[128:128 + 128]
    if mode == 0:
        assert np.all(codes[:64] == 0x7E) and np.all(codes[64:] == 0xFE)
        sc = row[256:260].view(np.uint16)
        assert np.array_equal(sc, oracle.bf16_from_float(np.array([3.0 / 448, 0.25 / 448], np.float32)))
    else:
        # 3/448 -> 2^-7 (3 * 128 = 384, code 0x7C); 0.25/448 -> 2^-10 (-256, code 0xF8)
        assert np.all(codes[:64] == 0x7C) and np.all(codes[64:] == 0xF8)
        assert list(row[256:258]) == [127 - 7, 127 - 10]
    assert np.all(row[oracle.kvc_concat_bytes(d, mode):] == 0xA5)   # bytes past the row


def test_kvc_spike_and_zero_groups():
    """[v, 0, ...] encodes v as 448 and the rest as 0; an all-zero group has
    scale 0 and zero codes in both modes."""
    d = 256
    x = np.zeros((1, d), np.float32)
    x[0, 5] = -7.5
    for mode in (0, 1):
        cache, hd, st, bsz = _kvc_run(x, mode, True)
        row = _kvc_row(cache, 0, hd, st, bsz)
        codes = row[128:128 + 192]
        if mode == 0:
            assert codes[5] == 0xFE and np.count_nonzero(codes) == 1
            assert list(row[320:326]) == list(oracle.bf16_from_float(
                np.array([7.5 / 448, 0, 0], np.float32)).view(np.uint8))
        else:
            # 7.5/448 -> 2^-5: 7.5 * 32 = 240 (code 0xF7)
            assert codes[5] == 0xF7 and np.count_nonzero(codes) == 1
            assert list(row[320:323]) == [127 - 5, 0, 0]


@pytest.mark.parametrize("round_scale", [True, False])
def test_kvc_mode1_power_of_two_bounds(round_scale):
    """Mode 1: every group scale is a power of two within a factor 2 of
    amax/448 (at or above it with roundScale, at or below it without), so the
    largest decoded |code| lies in [224, 448] with roundScale and is 448
    (saturated or exact) without; codes times the scale reproduce x within
    E4M3's half-ulp."""
    rng = np.random.default_rng(5)
    d, bs = 512, 6
    x = _bf16(rng.standard_normal((bs, d)) * np.exp2(rng.uniform(-30, 30, (bs, 1))))
    cache, hd, st, bsz = _kvc_run(x, 1, round_scale, block_num=2, block_size=4)
    nope = d - 64
    for i in range(bs):
        row = _kvc_row(cache, i, hd, st, bsz)
        codes = row[128:128 + nope].reshape(-1, 64)
        k = row[128 + nope:128 + nope + nope // 64].astype(np.int64) - 127
        dec = oracle.e4m3_decode(codes)
        xg = x[i, :nope].reshape(-1, 64)
        amax = np.abs(xg).max(axis=1)
        s = np.exp2(k.astype(np.float64))
        exact = amax.astype(np.float64) / 448
        if round_scale:
            assert np.all(s >= exact) and np.all(s < 2 * exact)
            top = np.abs(dec).max(axis=1)
            assert np.all(top <= 448) and np.all(top >= 224)   # amax/s in (224, 448], rounded
        else:
            assert np.all(s <= exact) and np.all(s > exact / 2)
            assert np.all(np.abs(dec).max(axis=1) == 448)
        deq = dec * s[:, None]
        inrange = np.abs(xg / s[:, None]) <= 448
        err = np.abs(deq - xg)[inrange]
        bound = np.maximum(np.abs(xg) * 2.0 ** -4, (s[:, None] * 2.0 ** -10 + 0 * xg))[inrange]
        assert np.all(err <= bound * (1 + 1e-12))


def test_kvc_mode0_error_bound_and_scale_definition():
    """Mode 0: the stored BF16 scale is BF16(amax/448) and codes times the
    FP32 scale reproduce x within E4M3's half-ulp (subnormal step for tiny
    values)."""
    rng = np.random.default_rng(6)
    d, bs = 1024, 4
    x = _bf16(rng.standard_normal((bs, d)) * 3.0)
    cache, hd, st, bsz = _kvc_run(x, 0, True, block_num=2, block_size=2)
    nope = d - 64
    for i in range(bs):
        row = _kvc_row(cache, i, hd, st, bsz)
        xg = x[i, :nope].reshape(-1, 64)
        scale = (np.abs(xg).max(axis=1).astype(np.float32) / np.float32(448)).astype(np.float32)
        sc = row[128 + nope:128 + nope + 2 * (nope // 64)].view(np.uint16)
        assert np.array_equal(sc, oracle.bf16_from_float(scale))
        dec = oracle.e4m3_decode(row[128:128 + nope].reshape(-1, 64))
        err = np.abs(dec * scale[:, None].astype(np.float64) - xg)
        bound = np.maximum(np.abs(xg) * 2.0 ** -4, scale[:, None] * 2.0 ** -10)
        assert np.all(err <= bound * (1 + 1e-6))


def test_kvc_slots_skip_and_untouched_bytes():
    """Slot -1 and out-of-range slots are skipped; rows not addressed and the
    bytes past each written row keep their values; rows land at
    block * block_stride + offset * head_dim (non-contiguous blocks)."""
    rng = np.random.default_rng(8)
    d = 256
    x = _bf16(rng.standard_normal((5, d)))
    slots = np.array([3, -1, 10, 99, 6])
    cache, hd, st, bsz = _kvc_run(x, 1, True, head_dim=400, block_num=3, block_size=4,
                                  slots=slots, stride_pad=77)
    ref = np.full_like(cache, 0xA5)
    for i, s in enumerate(slots):
        if 0 <= s < 12:
            one, *_ = _kvc_run(x[i:i + 1], 1, True, head_dim=400, block_num=1, block_size=1,
                               slots=[0])
            base = (s // 4) * st + (s % 4) * 400
            ref[base:base + 400] = one[:400]
    assert np.array_equal(cache, ref)
