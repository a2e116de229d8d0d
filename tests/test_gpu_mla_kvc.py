"""MLA sparse FP8 decode over KV compress epilog rows on the GPU, against the oracle.

The rows are those the CANN aclnnKvCompressEpilog page's operator writes for d = 576
(BF16 rope first, E4M3 nope in groups of 64, one BF16 or E8M0 scale per group), read
with the DeepSeek V32 MLA page's dequantisation. Cases: rows drawn in that layout, and
the append-then-attend chain where pa_fp8_kv_compress_epilog writes the cache on the
GPU from BF16 key rows and pa_mla_sparse_decode_kvc reads it. Criteria as for the
page-format decode (tests/test_gpu_mla.py): the page's count of elements outside atol
1e-4 + rtol 5e-3, the per-element arithmetic bound, max-abs 3e-2 and mean-abs 2e-3.
"""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DN, DR = 512, 64
KVC = {0: workloads.MLA_FORMAT_KVC_BF16, 1: workloads.MLA_FORMAT_KVC_E8M0}


@pytest.fixture(scope="module")
def pa():
    import fp8_paged_kv_block_gb300 as m
    m.build()
    m.lib()
    return m


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def small(B=2, S1=2, NQ=128, act=(300, 41), topk=256, seed=1, frac_invalid=0.0):
    return workloads.mla("gpu_kvc", B, S1, list(act), NQ=NQ, topk=topk,
                         seed=workloads.BASE_SEED + 500 + seed, frac_invalid=frac_invalid)


def run_gpu(pa, case, cache, mode, topk=None):
    dev = torch.device("cuda")
    qn, qr = case.q_bf16()
    c = cache if torch.is_tensor(cache) else torch.from_numpy(np.ascontiguousarray(cache)).to(dev)
    tk = torch.from_numpy(case.topk_indices() if topk is None else topk).to(dev)
    out = torch.full((case.T, case.NQ, DN), float("nan"), dtype=torch.bfloat16, device=dev)
    st = pa.MlaStatus()
    pa.mla_sparse_decode_kvc(qn.to(dev), qr.to(dev), c, tk,
                             torch.from_numpy(case.block_table).to(dev),
                             torch.from_numpy(case.act).to(dev), out, quant_mode=mode,
                             S1=case.S1, status=st, block_size=case.BS,
                             softmax_scale=case.softmax_scale)
    torch.cuda.synchronize()
    assert st.value() == 0, "MLA decode kernel reported a wait timeout"
    return out.cpu().view(torch.int16).numpy().view(np.uint16)


def run_oracle(case, cache, mode, rows=None):
    qn, qr = case.q_bits()
    return oracle.mla_sparse_decode(qn, qr, cache, case.topk_indices(), case.block_table,
                                    case.act, S1=case.S1, block_size=case.BS,
                                    s2_tile=case.s2_tile, softmax_scale=case.softmax_scale,
                                    rows=rows, want_f32=True, row_format=KVC[mode])


def abs_weighted(case, cache, mode, tokens=None):
    """float64 [T, NQ, 512]: sum_j w_j |V_j[c]| with w the FP64 softmax weights over each
    token's valid selected keys, the keys dequantised from the KV compress rows with torch
    (E4M3 codes at bytes 128..639 times each 64 channels' scale, rounded to BF16)."""
    tk = case.topk_indices()
    qn, qr = case.q_bf16()
    q = torch.cat([qn, qr], dim=-1).double()
    out = np.zeros((case.T, case.NQ, DN))
    cur = case.cur()
    for t in (range(case.T) if tokens is None else tokens):
        b = t // case.S1
        idx = tk[t, :cur[t]].astype(np.int64)
        idx = idx[(idx >= 0) & (idx < case.act[b])]
        if idx.size == 0:
            continue
        rows = torch.from_numpy(cache[case.physical_rows(idx, np.full(idx.shape, b))].copy())
        codes = rows[:, 2 * DR:2 * DR + DN].contiguous().view(torch.float8_e4m3fn).float()
        if mode == 0:
            sc = rows[:, 640:656].contiguous().view(torch.bfloat16).float()
        else:
            sc = torch.pow(2.0, rows[:, 640:648].float() - 127.0)
        kn = (codes * sc.repeat_interleave(64, dim=1)).to(torch.bfloat16).double()
        kr = rows[:, :2 * DR].contiguous().view(torch.bfloat16).double()
        s = (q[t] @ torch.cat([kn, kr], dim=1).T) * case.softmax_scale
        w = torch.softmax(s, dim=1)
        out[t] = (w @ kn.abs()).numpy()
    return out


def check_close(gpu_bits, ref_f32, wabs):
    g = bf16_bits_to_f32(gpu_bits)
    r = np.asarray(ref_f32, dtype=np.float32)
    assert np.isfinite(g).all()
    d = np.abs(g.astype(np.float64) - r)
    page_bad = d > 1e-4 + 5e-3 * np.abs(r)
    assert int(page_bad.sum()) <= 100, (int(page_bad.sum()), float(d.max()))
    bound = 2.0 ** -8 * np.abs(r) + 2.0 ** -7 * wabs + 1e-6
    over = d > bound
    assert not over.any(), (int(over.sum()), float((d - bound).max()))
    assert d.max() <= 3e-2 and d.mean() <= 2e-3, (float(d.max()), float(d.mean()))
    return d


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("NQ", [64, 128])
def test_mla_kvc_drawn_rows(pa, mode, NQ):
    """Rows drawn in the KV compress layout; visible counts 256, 40 and 41 (two full tiles,
    ragged tiles), 5% masked entries."""
    case = small(NQ=NQ, seed=NQ + mode, frac_invalid=0.05)
    cache = case.cache(fmt=KVC[mode])
    gpu = run_gpu(pa, case, cache, mode)
    _, ref = run_oracle(case, cache, mode)
    check_close(gpu, ref, abs_weighted(case, cache, mode))


@pytest.mark.parametrize("mode,round_scale", [(0, False), (1, True), (1, False)])
def test_mla_kvc_after_gpu_compress_epilog(pa, mode, round_scale):
    """Append then attend: the GPU's KV compress epilog writes BF16 key rows [nope | rope]
    into a paged cache of 672-byte rows (bit for bit the oracle's epilog), and the decode
    over that cache matches the oracle's decode over the oracle's cache."""
    case = small(B=2, S1=2, NQ=128, act=(1000, 333), topk=512, seed=20 + mode + 2 * round_scale)
    rows = case.rows_used()
    x = case.key_rows(rows)
    dev = torch.device("cuda")
    nrows = case.num_blocks * case.BS
    RB = workloads.MLA_ROW_BYTES
    cache_d = torch.zeros((case.num_blocks, case.BS, 1, RB), dtype=torch.uint8, device=dev)
    pa.kv_compress_epilog(cache_d, torch.from_numpy(x).to(torch.bfloat16).to(dev),
                          torch.from_numpy(rows.astype(np.int64)).to(dev), quant_mode=mode,
                          round_scale=round_scale)
    host = np.zeros((nrows, RB), dtype=np.uint8)
    oracle.kv_compress_epilog(x, host, case.num_blocks, case.BS, case.BS * RB, RB,
                              rows.astype(np.int64), quant_mode=mode, round_scale=round_scale)
    assert np.array_equal(cache_d.cpu().numpy().reshape(nrows, RB), host)
    gpu = run_gpu(pa, case, cache_d.view(nrows, RB), mode)
    _, ref = run_oracle(case, host, mode)
    check_close(gpu, ref, abs_weighted(case, host, mode))


@pytest.mark.parametrize("mode", [0, 1])
def test_mla_kvc_strided_blocks(pa, mode):
    """The epilog's cache with blocks 4 KB further apart than their rows need (block_stride
    = block_size * head_dim + 4096): the GPU epilog writes it, the decode reads it, and the
    output equals, bit for bit, the decode over the same rows in contiguous blocks, and the
    oracle's within the criteria."""
    case = small(B=2, S1=2, NQ=64, act=(700, 257), topk=384, seed=40 + mode, frac_invalid=0.05)
    rows = case.rows_used()
    x = torch.from_numpy(case.key_rows(rows)).to(torch.bfloat16).cuda()
    slots = torch.from_numpy(rows.astype(np.int64)).cuda()
    NB, BS, RB = case.num_blocks, case.BS, workloads.MLA_ROW_BYTES
    pitch = BS * RB + 4096
    big = torch.full((NB, pitch), 0x7F, dtype=torch.uint8, device="cuda")
    strided = big.as_strided((NB, BS, 1, RB), (pitch, RB, RB, 1))
    compact = torch.zeros((NB, BS, 1, RB), dtype=torch.uint8, device="cuda")
    for c in (strided, compact):
        pa.kv_compress_epilog(c, x, slots, quant_mode=mode, round_scale=True)
    a = run_gpu(pa, case, strided, mode)
    b = run_gpu(pa, case, compact, mode)
    assert np.array_equal(a, b)
    host = compact.cpu().numpy().reshape(NB * BS, RB)
    _, ref = run_oracle(case, host, mode)
    check_close(a, ref, abs_weighted(case, host, mode))


@pytest.mark.parametrize("mode", [0, 1])
def test_mla_kvc_same_keys_as_the_page_format(pa, mode):
    """Page-format rows whose scales the KV compress row holds exactly (BF16 values, powers
    of two), moved byte by byte into the KV compress layout: the GPU gives the same output
    through either entry point, bit for bit (both dequantise to the same BF16 keys, and the
    kernel's arithmetic order is fixed)."""
    case = small(seed=30 + mode)
    page = case.cache()
    s4 = page[:, 640:656].copy().view(np.uint32)
    if mode == 0:
        s4 &= np.uint32(0xFFFF0000)
    else:
        k = np.random.default_rng(2).integers(-9, -6, size=s4.shape)
        s4[:] = np.ldexp(1.0, k).astype(np.float32).view(np.uint32)
    page[:, 640:656] = s4.view(np.uint8).reshape(-1, 16)
    kvc = np.full_like(page, 0xFF)
    kvc[:, :2 * DR] = page[:, DN:DN + 2 * DR]
    kvc[:, 2 * DR:2 * DR + DN] = page[:, :DN]
    s8 = np.repeat(page[:, 640:656].copy().view(np.float32), 2, axis=1)
    if mode == 0:
        kvc[:, 640:656] = (s8.view(np.uint32) >> 16).astype(np.uint16).view(np.uint8).reshape(-1, 16)
    else:
        kvc[:, 640:648] = (np.frexp(s8.astype(np.float64))[1] - 1 + 127).astype(np.uint8)
    dev = torch.device("cuda")
    qn, qr = case.q_bf16()
    out = torch.empty((case.T, case.NQ, DN), dtype=torch.bfloat16, device=dev)
    st = pa.MlaStatus()
    pa.mla_sparse_decode(qn.to(dev), qr.to(dev), torch.from_numpy(page).to(dev),
                         torch.from_numpy(case.topk_indices()).to(dev),
                         torch.from_numpy(case.block_table).to(dev),
                         torch.from_numpy(case.act).to(dev), out, S1=case.S1, status=st)
    torch.cuda.synchronize()
    a = out.cpu().view(torch.int16).numpy().view(np.uint16)
    b = run_gpu(pa, case, kvc, mode)
    assert st.value() == 0
    assert np.array_equal(a, b)


def test_mla_kvc_page_b64_sampled(pa):
    """The MLA page's default decode case (b=64, s_q=2, 65536-long sequences, top-k 2048,
    128 heads) over KV compress rows (quant mode 0), as the benchmark runs it: all heads of
    6 tokens, spread over the batch, against the oracle."""
    case = workloads.mla_page_b64()
    used = case.rows_used()
    dev = torch.device("cuda")
    nrows = case.num_blocks * case.BS
    RB = workloads.MLA_ROW_BYTES
    rb = case.row_bytes(used, KVC[0])
    cache_d = torch.zeros((nrows, RB), dtype=torch.uint8, device=dev)
    cache_d[torch.from_numpy(used).to(dev)] = torch.from_numpy(rb).to(dev)
    gpu = run_gpu(pa, case, cache_d, 0)
    del cache_d
    toks = np.array([0, 1, 37, 64, 100, 127])
    rows = (toks[:, None] * case.NQ + np.arange(case.NQ)[None, :]).reshape(-1)
    host = np.zeros((nrows, RB), dtype=np.uint8)
    host[used] = rb
    _, ref = run_oracle(case, host, 0, rows=rows)
    wabs = abs_weighted(case, host, 0, tokens=toks)
    check_close(gpu[toks], ref[toks], wabs[toks])
