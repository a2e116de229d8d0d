"""GPU parity of the FP8 cache append: pass-through scatter and
quantise-on-append, bit-exact against the oracle, then decode attention over
the updated cache (the append + attend step)."""
import json
import os

import numpy as np
import pytest

import oracle
import workloads
from tests import _helpers as H

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    import fp8_paged_kv_block_gb300 as pa
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pa.lib()
    return torch


def test_scatter_worked_example(torch_cuda):
    torch = torch_cuda
    import fp8_paged_kv_block_gb300 as pa
    d = json.load(open(os.path.join(GOLDEN, "scatter_worked_example.json")))
    T, Hh, Dk, Dv = d["num_tokens"], d["num_head"], d["k_head_size"], d["v_head_size"]
    NB, BS = d["num_blocks"], d["block_size"]
    rng = np.random.default_rng(41)
    key = rng.integers(1, 255, (T, Hh, Dk), dtype=np.uint8)
    val = rng.integers(1, 255, (T, Hh, Dv), dtype=np.uint8)
    ks = rng.standard_normal((T, Hh)).astype(np.float32)
    kc = torch.zeros((NB, Hh, BS, Dk), dtype=torch.uint8, device="cuda")
    vc = torch.zeros((NB, Hh, BS, Dv), dtype=torch.uint8, device="cuda")
    ksc = torch.zeros((NB, Hh, BS, 1), dtype=torch.float32, device="cuda")
    pa.cache_scatter(torch.from_numpy(key).cuda(), torch.from_numpy(val).cuda(), kc, vc,
                     torch.tensor(d["slot_mapping"], dtype=torch.int32, device="cuda"),
                     torch.from_numpy(ks).cuda(), ksc, layout=pa.LAYOUT_BNBD)
    kc, vc, ksc = kc.cpu().numpy(), vc.cpu().numpy(), ksc.cpu().numpy()
    written = np.zeros((NB, BS), bool)
    for i, (blk, off) in enumerate(d["expected_block_offset"]):
        assert np.array_equal(kc[blk, :, off], key[i])
        assert np.array_equal(vc[blk, :, off], val[i])
        assert np.array_equal(ksc[blk, :, off, 0], ks[i])
        written[blk, off] = True
    assert not kc.transpose(0, 2, 1, 3)[~written].any()
    assert not vc.transpose(0, 2, 1, 3)[~written].any()


@pytest.mark.parametrize("layout", [workloads.LAYOUT_BSND, workloads.LAYOUT_BNBD])
@pytest.mark.parametrize("slot_dtype", ["int32", "int64"])
@pytest.mark.parametrize("dims", [(128, 128), (64, 32), (24, 40)])
def test_scatter_bitexact(torch_cuda, layout, slot_dtype, dims):
    """Random slots (unique) with invalid ones mixed in, non-contiguous
    key_scale, pre-filled caches: bytes equal the oracle's."""
    torch = torch_cuda
    import fp8_paged_kv_block_gb300 as pa
    Dk, Dv = dims
    rng = np.random.default_rng(42 + Dk + layout)
    T, Hh, NB, BS = 300, 4, 9, 128
    key = rng.integers(0, 256, (T, Hh, Dk), dtype=np.uint8)
    val = rng.integers(0, 256, (T, Hh, Dv), dtype=np.uint8)
    ks_full = rng.standard_normal((T, 3 * Hh)).astype(np.float32)
    slots = rng.choice(NB * BS, T, replace=False).astype(np.int64)
    slots[::17] = -1
    slots[5] = NB * BS
    slots[6] = -7
    shape_k = (NB, Hh, BS, Dk) if layout == workloads.LAYOUT_BNBD else (NB, BS, Hh, Dk)
    shape_v = shape_k[:3] + (Dv,)
    kc0 = rng.integers(0, 256, shape_k, dtype=np.uint8)
    vc0 = rng.integers(0, 256, shape_v, dtype=np.uint8)
    ksc0 = rng.standard_normal(shape_k[:3] + (1,)).astype(np.float32)
    kc, vc, ksc = kc0.copy(), vc0.copy(), ksc0.copy()
    oracle.cache_scatter(key, val, kc, vc, slots, ks_full[:, ::3], ksc, layout=layout)
    gk = torch.from_numpy(kc0).cuda()
    gv = torch.from_numpy(vc0).cuda()
    gs = torch.from_numpy(ksc0).cuda()
    ks_dev = torch.from_numpy(ks_full).cuda()[:, ::3]
    pa.cache_scatter(torch.from_numpy(key).cuda(), torch.from_numpy(val).cuda(), gk, gv,
                     torch.from_numpy(slots.astype(slot_dtype)).cuda(), ks_dev, gs, layout=layout)
    assert np.array_equal(gk.cpu().numpy(), kc)
    assert np.array_equal(gv.cpu().numpy(), vc)
    assert np.array_equal(gs.cpu().numpy(), ksc)


def _append_context():
    ap = workloads.append()
    return ap, ap.ctx


def test_append_quant_scatter_bitexact_and_attend(torch_cuda):
    """The append + attend step: 64 BF16 K/V rows quantised per token-head
    (key_scale = amax/448) and scattered (5% slots -1) into a BNBD cache over
    contexts of 512-8192 tokens, then GQA decode over the updated cache."""
    torch = torch_cuda
    import fp8_paged_kv_block_gb300 as pa
    ap, ctx = _append_context()
    rng = np.random.default_rng(43)
    bsel = np.sort(rng.choice(ctx.B, 12, replace=False))
    # context caches, both paths (the oracle fills the sampled sequences)
    inp = H.oracle_inputs(ctx, batches=bsel)
    dev = H.device_inputs(ctx)
    H.check_cache_bitexact(ctx, dev, inp)
    # new tokens
    k_new, v_new = ap.new_kv_f32()
    kb, vb = ap.new_kv_bf16()
    slot = ap.slot_mapping
    c = dev["cache"]
    pa.cache_quant_scatter(kb.cuda(), vb.cuda(), c.k_cache, c.v_cache,
                           torch.from_numpy(slot).cuda(), c.k_scale, c.v_scale,
                           torch.from_numpy(ap.token_batch).cuda(), layout=ctx.layout)
    # oracle append for every new token (its cache holds only the sampled
    # sequences' contexts; the appended rows are compared for all tokens)
    kc, vc, ksc = inp["kc"], inp["vc"], inp["ksc"]
    vs_all = c.v_scale.cpu().numpy()          # compared bit-exact below for bsel
    for b in inp["batches"]:
        assert np.array_equal(vs_all[b], inp["vs"][b])
    vs_or = inp["vs"].copy()
    # sequences outside bsel: the oracle computes their channel scales itself
    k32, v32 = ctx.kv()
    cu = ctx.cu_seqlens
    for b in range(ctx.B):
        if b not in set(bsel.tolist()):
            vs_or[b] = oracle.value_channel_scale(v32[cu[b]:cu[b + 1]],
                                                  np.array([0, cu[b + 1] - cu[b]]), 1)[0]
    assert np.array_equal(vs_all, vs_or)
    oracle.cache_quant_scatter(k_new, v_new, kc, vc, slot.astype(np.int64), ksc, vs_or,
                               ap.token_batch, layout=ctx.layout)
    gk, gv, gs = c.k_cache.cpu().numpy(), c.v_cache.cpu().numpy(), c.k_scale.cpu().numpy()
    BS = ctx.BS
    for i, s in enumerate(slot):
        if s < 0:
            continue
        blk, off = s // BS, s % BS
        assert np.array_equal(gk[blk, :, off], kc[blk, :, off]), i
        assert np.array_equal(gv[blk, :, off], vc[blk, :, off]), i
        assert np.array_equal(gs[blk, :, off], ksc[blk, :, off]), i
    # skipped tokens left their slots untouched (still zero)
    for b in np.nonzero(slot < 0)[0]:
        a = int(ctx.act[b])
        s = int(ctx.block_table[b, a // BS]) * BS + a % BS
        assert not gk[s // BS, :, s % BS].any() and not gv[s // BS, :, s % BS].any()
    # attend over the updated cache
    act_after = ap.act_after
    import dataclasses
    ctx2 = dataclasses.replace(ctx, act=act_after)
    out = torch.empty((ctx.B, ctx.NQ, ctx.D), dtype=torch.bfloat16, device="cuda")
    ws = pa.DecodeWorkspace(ctx.B, 1, ctx.NQ, ctx.NKV)
    pa.decode(dev["q8"], dev["qs"], c.k_cache, c.k_scale, c.v_cache, c.v_scale,
              dev["block_table"], torch.from_numpy(act_after).cuda(), out, S1=1,
              layout=ctx.layout, workspace=ws)
    rows = np.sort(np.concatenate([b * ctx.NQ + rng.choice(ctx.NQ, 6, replace=False)
                                   for b in bsel]))
    ref = oracle.pa_decode(inp["q8"], inp["qs"], kc, ksc, vc, vs_or, ctx.block_table, act_after,
                           S1=1, NKV=ctx.NKV, layout=ctx.layout, s2_tile=512,
                           softmax_scale=ctx.softmax_scale, rows=rows)
    H.compare_bf16(H.to_u16(out), ref, rows=rows)
    assert ws.error_flags() == 0


@pytest.mark.parametrize("overlap", [False, True])
@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("D", [64, 128, 200, 384, 640])
def test_quant_scatter_head_sizes(torch_cuda, D, dtype, overlap):
    """Quantise-on-append for head sizes that take each kernel form (one, two
    or four groups of 128 channels per warp in registers, and the looped form
    above 512, with ragged last groups), FP32 and BF16 inputs, plain and with
    programmatic serialisation: pre-filled BSND caches equal the oracle's
    byte for byte, including a zero v_scale channel and a zero key row."""
    torch = torch_cuda
    import fp8_paged_kv_block_gb300 as pa
    T, Hh, NB, BS, NBT = 37, 3, 5, 16, 5
    rng = np.random.default_rng(1000 + D)
    k = rng.standard_normal((T, Hh, D)).astype(np.float32) * 3.0
    v = rng.standard_normal((T, Hh, D)).astype(np.float32)
    k[4, 1] = 0.0                                          # all-zero key row
    tdt = getattr(torch, dtype)
    kt, vt = torch.from_numpy(k).to(tdt), torch.from_numpy(v).to(tdt)
    k32, v32 = kt.float().numpy(), vt.float().numpy()      # the values the kernel sees
    slot = rng.choice(NB * BS, T, replace=False).astype(np.int64)
    slot[rng.random(T) < 0.15] = -1
    slot[0] = NB * BS + 3                                  # out of range: skipped
    tb = rng.integers(0, NBT, T).astype(np.int32)
    vs = (np.abs(rng.standard_normal((NBT, Hh, D))) / 100.0 + 1e-3).astype(np.float32)
    vs[1, 2, 7] = 0.0
    kc0 = rng.integers(0, 256, (NB, BS, Hh, D), dtype=np.uint8)
    vc0 = rng.integers(0, 256, (NB, BS, Hh, D), dtype=np.uint8)
    ks0 = rng.standard_normal((NB, BS, Hh)).astype(np.float32)
    kc, vc, ks = (torch.from_numpy(a.copy()).cuda() for a in (kc0, vc0, ks0))
    pa.cache_quant_scatter(kt.cuda(), vt.cuda(), kc, vc, torch.from_numpy(slot).cuda(), ks,
                           torch.from_numpy(vs).cuda(), torch.from_numpy(tb).cuda(),
                           layout=pa.LAYOUT_BSND, overlap_prologue=overlap)
    torch.cuda.synchronize()
    okc, ovc, oks = kc0.copy(), vc0.copy(), ks0.copy()
    oracle.cache_quant_scatter(k32, v32, okc, ovc, slot, oks, vs, tb, layout=workloads.LAYOUT_BSND)
    assert np.array_equal(kc.cpu().numpy(), okc)
    assert np.array_equal(vc.cpu().numpy(), ovc)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), oks.view(np.uint32))


@pytest.mark.parametrize("mode", [1, 2])
def test_step_chain_overlap_in_graph(torch_cuda, mode):
    """decode -> append -> decode with programmatic serialisation on all three
    launches (decode mode 1: prologue only; mode 2: also the cache blocks
    below each sequence's newest position), eagerly and captured in a CUDA
    graph: the append's stores wait for the first decode, the second decode
    sees the appended token, both outputs and the cache match the oracle."""
    torch = torch_cuda
    import fp8_paged_kv_block_gb300 as pa
    case = workloads.custom("chain", 6, 1, 24, 2, [1, 127, 700, 1300, 2049, 3000], max_blocks=25)
    inp = H.oracle_inputs(case)
    dev = H.device_inputs(case)
    ref0 = H.oracle_decode(case, inp)
    knew, vnew, slot, act_after = workloads.step_tokens(case)
    import dataclasses
    case1 = dataclasses.replace(case, act=act_after)
    oracle.cache_quant_scatter(knew.float().numpy(), vnew.float().numpy(), inp["kc"], inp["vc"],
                               slot.astype(np.int64), inp["ksc"], inp["vs"],
                               np.arange(case.B, dtype=np.int32), layout=case.layout)
    ref1 = H.oracle_decode(case1, inp)
    c = dev["cache"]
    snap = [t.clone() for t in (c.k_cache, c.v_cache, c.k_scale)]
    ws = pa.DecodeWorkspace(case.B, case.S1, case.NQ, case.NKV, s2_tile=case.s2_tile)
    shape = (case.B * case.S1, case.NQ, case.D)
    o0 = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    o1 = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    kn, vn = knew.cuda(), vnew.cuda()
    sl = torch.from_numpy(slot).cuda()
    tb = torch.arange(case.B, dtype=torch.int32, device="cuda")
    act0 = dev["act"]
    act1 = torch.from_numpy(act_after).cuda()

    def chain():
        for act, out in ((act0, o0), (None, None), (act1, o1)):
            if act is None:
                pa.cache_quant_scatter(kn, vn, c.k_cache, c.v_cache, sl, c.k_scale, c.v_scale, tb,
                                       layout=case.layout, overlap_prologue=True)
                continue
            pa.decode(dev["q8"], dev["qs"], c.k_cache, c.k_scale, c.v_cache, c.v_scale,
                      dev["block_table"], act, out, S1=case.S1, layout=case.layout,
                      s2_tile=case.s2_tile, softmax_scale=case.softmax_scale, workspace=ws,
                      overlap_prologue=mode)

    def check():
        torch.cuda.synchronize()
        assert ws.error_flags() == 0
        H.compare_bf16(H.to_u16(o0), ref0)
        H.compare_bf16(H.to_u16(o1), ref1)
        assert np.array_equal(c.k_cache.cpu().numpy(), inp["kc"])
        assert np.array_equal(c.v_cache.cpu().numpy(), inp["vc"])
        assert np.array_equal(c.k_scale.cpu().numpy(), inp["ksc"])

    tick = torch.zeros(1, device="cuda")

    def restore():
        for t, s in zip((c.k_cache, c.v_cache, c.k_scale), snap):
            t.copy_(s)
        o0.fill_(float("nan"))
        o1.fill_(float("nan"))
        # the first decode may read old cache blocks while its predecessor
        # runs (mode 2): that predecessor is a kernel that writes no cache
        tick.add_(1)

    chain()
    check()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        restore()
        chain()
    torch.cuda.current_stream().wait_stream(s)
    check()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        restore()
        chain()
    for _ in range(2):
        g.replay()
        check()


def test_prepared_step_calls(torch_cuda):
    """prepare_cache_quant_scatter and prepare_decode: the step's two calls
    validated and marshalled once, then launched (programmatic serialisation,
    decode mode 2) eagerly on the prepared stream, on another stream, and
    captured in a CUDA graph; output against the oracle, cache bit-exact."""
    torch = torch_cuda
    import dataclasses
    import fp8_paged_kv_block_gb300 as pa
    case = workloads.custom("prep", 6, 1, 24, 2, [1, 127, 700, 1300, 2049, 3000], max_blocks=25)
    inp = H.oracle_inputs(case)
    dev = H.device_inputs(case)
    knew, vnew, slot, act_after = workloads.step_tokens(case)
    oracle.cache_quant_scatter(knew.float().numpy(), vnew.float().numpy(), inp["kc"], inp["vc"],
                               slot.astype(np.int64), inp["ksc"], inp["vs"],
                               np.arange(case.B, dtype=np.int32), layout=case.layout)
    ref = H.oracle_decode(dataclasses.replace(case, act=act_after), inp)
    c = dev["cache"]
    snap = [t.clone() for t in (c.k_cache, c.v_cache, c.k_scale)]
    out = torch.empty((case.B * case.S1, case.NQ, case.D), dtype=torch.bfloat16, device="cuda")
    kn, vn = knew.cuda(), vnew.cuda()
    sl = torch.from_numpy(slot).cuda()
    tb = torch.arange(case.B, dtype=torch.int32, device="cuda")
    act1 = torch.from_numpy(act_after).cuda()
    append = pa.prepare_cache_quant_scatter(kn, vn, c.k_cache, c.v_cache, sl, c.k_scale,
                                            c.v_scale, tb, layout=case.layout,
                                            overlap_prologue=True)
    attend = pa.prepare_decode(dev["q8"], dev["qs"], c.k_cache, c.k_scale, c.v_cache, c.v_scale,
                               dev["block_table"], act1, out, S1=case.S1, layout=case.layout,
                               s2_tile=case.s2_tile, softmax_scale=case.softmax_scale,
                               overlap_prologue=2)

    def restore():
        for t, sn in zip((c.k_cache, c.v_cache, c.k_scale), snap):
            t.copy_(sn)
        out.fill_(float("nan"))

    def check():
        torch.cuda.synchronize()
        H.compare_bf16(H.to_u16(out), ref)
        assert np.array_equal(c.k_cache.cpu().numpy(), inp["kc"])
        assert np.array_equal(c.v_scale.cpu().numpy(), inp["vs"])
        assert np.array_equal(c.k_scale.cpu().numpy(), inp["ksc"])

    append()
    attend()
    check()
    restore()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    append(s)
    attend(s)
    torch.cuda.current_stream().wait_stream(s)
    check()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        restore()
        cur = torch.cuda.current_stream()
        append(cur)
        attend(cur)
    for _ in range(2):
        g.replay()
        check()


@pytest.mark.parametrize("round_scale", [True, False])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("d", [128, 256, 576, 1024])
def test_kv_compress_epilog_bitexact(torch_cuda, d, mode, round_scale):
    """KV compress epilog, modes 0/1: BF16 rows with a wide dynamic range,
    zero and one-spike groups, int32/int64 slots with -1 and out-of-range
    entries, blocks at a stride larger than the block (non-contiguous) and an
    odd row pitch: every cache byte equals the oracle's."""
    torch = torch_cuda
    import fp8_paged_kv_block_gb300 as pa
    rng = np.random.default_rng(900 + d + 10 * mode + int(round_scale))
    bs, NB, BS = 45, 7, 8
    x = (rng.standard_normal((bs, d)) * np.exp2(rng.uniform(-40, 40, (bs, 1)))).astype(np.float32)
    x[3, :64] = 0.0                          # zero group
    x[4, :] = 0.0
    x[4, 70] = -3.5                          # one spike
    xb = torch.from_numpy(x).to(torch.bfloat16)
    xf = xb.float().numpy()
    head_dim = oracle.kvc_min_head_dim(d, mode) + 3          # odd pitch
    pitch = (BS + 2) * head_dim                              # strided blocks
    slots = rng.choice(NB * BS, bs, replace=False).astype(np.int64)
    slots[rng.random(bs) < 0.1] = -1
    slots[7] = NB * BS + 5
    for slot_dtype in (torch.int32, torch.int64):
        base = torch.from_numpy(rng.integers(0, 256, NB * pitch, dtype=np.uint8)).cuda()
        ref = base.cpu().numpy().copy()
        cache = base.view(NB, BS + 2, 1, head_dim)[:, :BS]
        pa.kv_compress_epilog(cache, xb.cuda(), torch.from_numpy(slots).to(slot_dtype).cuda(),
                              quant_mode=mode, round_scale=round_scale)
        torch.cuda.synchronize()
        oracle.kv_compress_epilog(xf, ref, NB, BS, pitch, head_dim, slots, mode, round_scale)
        got = base.cpu().numpy()
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, (slot_dtype, bad[:10], got[bad[:10]], ref[bad[:10]])


def test_step_chain_all_slots_skipped(torch_cuda):
    """decode -> append -> decode -> append -> ... with programmatic
    serialisation on every launch, where every slot of each append is -1 (a
    legal input: skipped slots): no thread of the append stores anything, yet
    the append must still complete only after the decode before it, so that
    the next decode (same workspace, same output buffer) cannot start writing
    while the previous one runs. Replayed back to back from a CUDA graph;
    every output matches the oracle and the cache is unchanged."""
    torch = torch_cuda
    import fp8_paged_kv_block_gb300 as pa
    case = workloads.custom("skipchain", 6, 1, 24, 2, [1, 127, 700, 1300, 2049, 3000], max_blocks=25)
    inp = H.oracle_inputs(case)
    dev = H.device_inputs(case)
    ref = H.oracle_decode(case, inp)
    knew, vnew, slot, _ = workloads.step_tokens(case)
    c = dev["cache"]
    snap = [t.clone() for t in (c.k_cache, c.v_cache, c.k_scale)]
    ws = pa.DecodeWorkspace(case.B, case.S1, case.NQ, case.NKV, s2_tile=case.s2_tile)
    shape = (case.B * case.S1, case.NQ, case.D)
    outs = [torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    kn, vn = knew.cuda(), vnew.cuda()
    skipped = torch.full((case.B,), -1, dtype=torch.int32, device="cuda")
    tb = torch.arange(case.B, dtype=torch.int32, device="cuda")

    def chain():
        for out in outs:
            pa.decode(dev["q8"], dev["qs"], c.k_cache, c.k_scale, c.v_cache, c.v_scale,
                      dev["block_table"], dev["act"], out, S1=case.S1, layout=case.layout,
                      s2_tile=case.s2_tile, softmax_scale=case.softmax_scale, workspace=ws,
                      overlap_prologue=2)
            pa.cache_quant_scatter(kn, vn, c.k_cache, c.v_cache, skipped, c.k_scale, c.v_scale, tb,
                                   layout=case.layout, overlap_prologue=True)

    def check():
        torch.cuda.synchronize()
        assert ws.error_flags() == 0
        for out in outs:
            H.compare_bf16(H.to_u16(out), ref)
        for t, s in zip((c.k_cache, c.v_cache, c.k_scale), snap):
            assert torch.equal(t, s)

    chain()
    check()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        chain()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for out in outs:
            out.fill_(float("nan"))
        chain()
    for _ in range(5):
        g.replay()
        check()
