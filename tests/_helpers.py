"""Shared test helpers: the same seeded workload turned into inputs twice --
once by the CPU oracle's quantisers (numpy placement into the paged cache)
and once by the library's CUDA kernels -- plus the parity comparison.

Tolerance of the BF16 attention output against the oracle (element-wise):
max |gpu - oracle| <= 3e-2 and mean |gpu - oracle| <= 2e-3. FP8 codes,
scales and scattered bytes must match bit for bit."""
from __future__ import annotations

import numpy as np

import oracle
import workloads

MAX_ABS_TOL = 3e-2
MEAN_ABS_TOL = 2e-3


def oracle_inputs(case, batches=None):
    """Quantise ``case`` with the oracle and place it in a paged cache with
    numpy indexing. With ``batches`` only those sequences are filled (the
    rest of the cache stays zero), which is all the oracle reads for their
    rows."""
    q8, qs = oracle.quant_rows(case.q())
    k32, v32 = case.kv()
    cu = case.cu_seqlens
    sel = range(case.B) if batches is None else sorted(set(int(b) for b in batches))
    NB, BS, H, D = case.num_blocks, case.BS, case.NKV, case.D
    if case.layout == workloads.LAYOUT_BSND:
        kc = np.zeros((NB, BS, H, D), np.uint8)
        ksc = np.zeros((NB, BS, H), np.float32)
    else:
        kc = np.zeros((NB, H, BS, D), np.uint8)
        ksc = np.zeros((NB, H, BS), np.float32)
    vc = np.zeros_like(kc)
    vs = np.zeros((case.B, H, D), np.float32)
    slots_all = case.slots
    for b in sel:
        lo, hi = int(cu[b]), int(cu[b + 1])
        if hi == lo:
            continue
        k8, ks = oracle.quant_rows(k32[lo:hi])
        vsb = oracle.value_channel_scale(v32[lo:hi], np.array([0, hi - lo]), 1)
        v8 = oracle.quant_channels(v32[lo:hi], np.zeros(hi - lo, np.int32), vsb)
        vs[b] = vsb[0]
        sl = slots_all[lo:hi]
        blk, off = sl // BS, sl % BS
        if case.layout == workloads.LAYOUT_BSND:
            kc[blk, off] = k8
            vc[blk, off] = v8
            ksc[blk, off] = ks
        else:
            kc[blk, :, off] = k8
            vc[blk, :, off] = v8
            ksc[blk, :, off] = ks
    return dict(q8=q8, qs=qs, kc=kc, vc=vc, ksc=ksc, vs=vs, batches=list(sel))


def oracle_decode(case, inp, rows=None, s2_tile=None):
    return oracle.pa_decode(inp["q8"], inp["qs"], inp["kc"], inp["ksc"], inp["vc"], inp["vs"],
                            case.block_table, case.act, S1=case.S1, NKV=case.NKV,
                            layout=case.layout, s2_tile=s2_tile or case.s2_tile,
                            softmax_scale=case.softmax_scale, rows=rows)


def device_inputs(case, device="cuda"):
    """The same workload quantised and paged by the library's kernels."""
    import torch
    import fp8_paged_kv_block_gb300 as pa
    from fp8_paged_kv_block_gb300 import paged

    q32 = torch.from_numpy(case.q()).to(device)
    q8, qs = paged.quantize_queries(q32)
    k32, v32 = case.kv()
    cache = paged.build_cache(
        torch.from_numpy(k32).to(device), torch.from_numpy(v32).to(device),
        torch.from_numpy(case.cu_seqlens).to(device), torch.from_numpy(case.slots).to(device),
        torch.from_numpy(case.token_batch).to(device), case.num_blocks, case.layout)
    return dict(q8=q8, qs=qs, cache=cache,
                block_table=torch.from_numpy(case.block_table).to(device),
                act=torch.from_numpy(case.act).to(device), pa=pa)


def gpu_decode(case, dev, *, s2_tile=None, num_ctas=0, workspace=None, out=None):
    import torch
    pa = dev["pa"]
    c = dev["cache"]
    if out is None:
        out = torch.empty((case.B * case.S1, case.NQ, case.D), dtype=torch.bfloat16,
                          device=dev["q8"].device)
    pa.decode(dev["q8"], dev["qs"], c.k_cache, c.k_scale, c.v_cache, c.v_scale,
              dev["block_table"], dev["act"], out, S1=case.S1, layout=case.layout,
              s2_tile=s2_tile or case.s2_tile, softmax_scale=case.softmax_scale,
              workspace=workspace, num_ctas=num_ctas)
    return out


def to_u16(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def compare_bf16(gpu_u16, ref_u16, rows=None):
    """Element-wise parity of BF16 outputs (flat rows x D)."""
    g = oracle.bf16_to_float(gpu_u16).reshape(-1, gpu_u16.shape[-1]).astype(np.float64)
    r = oracle.bf16_to_float(ref_u16).reshape(-1, ref_u16.shape[-1]).astype(np.float64)
    if rows is not None:
        g, r = g[rows], r[rows]
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    err = np.abs(g - r)
    stats = dict(max_abs=float(err.max()), mean_abs=float(err.mean()))
    assert stats["max_abs"] <= MAX_ABS_TOL, stats
    assert stats["mean_abs"] <= MEAN_ABS_TOL, stats
    return stats


def check_cache_bitexact(case, dev, inp):
    """GPU-built cache (codes, key scales, value scales) == oracle-built, over
    the sequences the oracle filled."""
    c = dev["cache"]
    vs = c.v_scale.cpu().numpy()
    for b in inp["batches"]:
        assert np.array_equal(vs[b], inp["vs"][b]), "v_scale mismatch in batch %d" % b
    if len(inp["batches"]) == case.B:
        assert np.array_equal(c.k_cache.cpu().numpy(), inp["kc"])
        assert np.array_equal(c.v_cache.cpu().numpy(), inp["vc"])
        assert np.array_equal(c.k_scale.cpu().numpy(), inp["ksc"])
    else:
        cu = case.cu_seqlens
        sl_all = case.slots
        kc, vc, ks = c.k_cache.cpu().numpy(), c.v_cache.cpu().numpy(), c.k_scale.cpu().numpy()
        for b in inp["batches"]:
            sl = sl_all[cu[b]:cu[b + 1]]
            blk, off = sl // case.BS, sl % case.BS
            if case.layout == workloads.LAYOUT_BSND:
                idx = (blk, off)
            else:
                idx = (blk, slice(None), off)
            assert np.array_equal(kc[idx], inp["kc"][idx])
            assert np.array_equal(vc[idx], inp["vc"][idx])
            assert np.array_equal(ks[idx], inp["ksc"][idx])
