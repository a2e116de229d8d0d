"""MLA sparse FP8 decode on the GPU against the oracle.

The GPU's BF16 output is compared with the oracle's FP32 output before its
BF16 cast:
  - the DeepSeek V32 MLA sparse attention page's criterion: at most 100
    elements outside atol 1e-4 + rtol 5e-3 (its max_error_count);
  - every element within the bound the arithmetic gives: the GPU's own BF16
    rounding (2^-9 relative, taken as 2^-8) plus one BF16 step in every P_j
    (P is rounded to BF16 on both sides, from FP32 scores summed in a
    different order and exponentials of different accuracy, so a P_j near a
    rounding boundary may land one step apart: at most 2^-7 P_j), i.e.
    2^-7 * sum_j w_j |V_j[c]| with w the softmax weights;
  - max-abs 3e-2 and mean-abs 2e-3 for BF16 attention outputs.
"""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DN = 512


@pytest.fixture(scope="module")
def pa():
    import fp8_paged_kv_block_gb300 as m
    m.build()
    m.lib()
    return m


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def run_gpu(pa, case, cache_np, *, topk=None, row_bytes=None, status=None):
    dev = torch.device("cuda")
    qn, qr = case.q_bf16()
    cache = torch.from_numpy(np.ascontiguousarray(cache_np)).to(dev)
    tk = torch.from_numpy(case.topk_indices() if topk is None else topk).to(dev)
    bt = torch.from_numpy(case.block_table).to(dev)
    act = torch.from_numpy(case.act).to(dev)
    out = torch.full((case.T, case.NQ, DN), float("nan"), dtype=torch.bfloat16, device=dev)
    st = status or pa.MlaStatus()
    pa.mla_sparse_decode(qn.to(dev), qr.to(dev), cache, tk, bt, act, out, S1=case.S1,
                         status=st, block_size=case.BS, softmax_scale=case.softmax_scale)
    torch.cuda.synchronize()
    assert st.value() == 0, "MLA decode kernel reported a wait timeout"
    return out.cpu().view(torch.int16).numpy().view(np.uint16)


def run_oracle(case, cache_np, *, topk=None, rows=None):
    qn, qr = case.q_bits()
    return oracle.mla_sparse_decode(qn, qr, cache_np,
                                    case.topk_indices() if topk is None else topk,
                                    case.block_table, case.act, S1=case.S1, block_size=case.BS,
                                    s2_tile=case.s2_tile, softmax_scale=case.softmax_scale,
                                    rows=rows, want_f32=True)


def abs_weighted(case, cache, topk=None, tokens=None):
    """float64 [T, NQ, 512]: sum_j w_j |V_j[c]| with w the FP64 softmax
    weights over each token's valid selected keys (zeros where none)."""
    tk = case.topk_indices() if topk is None else topk
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
        codes = rows[:, :DN].contiguous().view(torch.float8_e4m3fn).float()
        sc = rows[:, 640:656].contiguous().view(torch.float32)
        kn = (codes * sc.repeat_interleave(128, dim=1)).to(torch.bfloat16).double()
        kr = rows[:, DN:640].contiguous().view(torch.bfloat16).double()
        s = (q[t] @ torch.cat([kn, kr], dim=1).T) * case.softmax_scale
        w = torch.softmax(s, dim=1)
        out[t] = (w @ kn.abs()).numpy()
    return out


def check_close(gpu_bits, ref_f32, wabs, sel=None):
    g = bf16_bits_to_f32(gpu_bits)
    r = np.asarray(ref_f32, dtype=np.float32)
    if sel is not None:
        g, r, wabs = g[sel], r[sel], wabs[sel]
    assert np.isfinite(g).all()
    d = np.abs(g.astype(np.float64) - r)
    page_bad = d > 1e-4 + 5e-3 * np.abs(r)
    assert int(page_bad.sum()) <= 100, (int(page_bad.sum()), float(d.max()))
    bound = 2.0 ** -8 * np.abs(r) + 2.0 ** -7 * wabs + 1e-6
    over = d > bound
    assert not over.any(), (int(over.sum()), float((d - bound).max()))
    assert d.max() <= 3e-2 and d.mean() <= 2e-3, (float(d.max()), float(d.mean()))
    return d


def small(B=2, S1=2, NQ=128, act=(300, 41), topk=256, seed=1, frac_invalid=0.0, BS=128):
    return workloads.mla("gpu_small", B, S1, list(act), NQ=NQ, topk=topk,
                         seed=workloads.BASE_SEED + 400 + seed, frac_invalid=frac_invalid, BS=BS)


@pytest.mark.parametrize("NQ", [64, 128, 256])
def test_mla_small_several_tiles_and_ragged_tail(pa, NQ):
    """Visible counts 256 (two full tiles), 40 and 41 (one ragged tile)."""
    case = small(NQ=NQ, act=(300, 41), topk=256, seed=NQ)
    cache = case.cache()
    gpu = run_gpu(pa, case, cache)
    _, ref = run_oracle(case, cache)
    check_close(gpu, ref, abs_weighted(case, cache))


def test_mla_masked_entries_and_long_lists(pa):
    """5% of the selected entries are -1; visible counts 1000, 999 (8 tiles,
    a ragged last one)."""
    case = small(B=1, S1=2, act=(1000,), topk=1024, seed=7, frac_invalid=0.05)
    cache = case.cache()
    gpu = run_gpu(pa, case, cache)
    _, ref = run_oracle(case, cache)
    check_close(gpu, ref, abs_weighted(case, cache))


def test_mla_no_visible_key_gives_zeros(pa):
    """Tokens whose visible count is 0 (a sequence shorter than S1 - s) and
    tokens whose every selected entry is masked get all-zero rows."""
    case = small(B=3, S1=3, act=(200, 2, 1), topk=128, seed=3)
    cache = case.cache()
    tk = case.topk_indices().copy()
    tk[1, :] = -1                                   # token (0, 1): every entry masked
    gpu = run_gpu(pa, case, cache, topk=tk)
    _, ref = run_oracle(case, cache, topk=tk)
    zero = case.cur() == 0
    zero[1] = True
    assert not gpu[zero].any()
    check_close(gpu, ref, abs_weighted(case, cache, topk=tk))


def test_mla_page_ragged_case_full(pa):
    """The page's decode case b=4, s_q=2, lengths [65536, 16381, 666, 15],
    topk 2048, 128 heads: every output element against the oracle."""
    case = workloads.mla_page_ragged()
    used = case.rows_used()
    cache = case.cache(rows=used)
    gpu = run_gpu(pa, case, cache)
    _, ref = run_oracle(case, cache)
    d = check_close(gpu, ref, abs_weighted(case, cache))
    # most outputs round to the very same BF16 value, and the mean error is
    # within half a BF16 step (2^-8 relative) of the mean magnitude
    same = (gpu == oracle.bf16_from_float(ref.reshape(-1)).reshape(gpu.shape)).mean()
    assert same > 0.95, same
    assert d.mean() <= 2.0 ** -8 * np.abs(ref).mean(), (d.mean(), np.abs(ref).mean())


def test_mla_row_pitch_and_block_size(pa):
    """Unpadded 656-byte rows and 64-token blocks address the same keys."""
    case = small(B=2, S1=1, act=(700, 130), topk=512, seed=9, BS=64)
    full = case.cache()
    cache = np.ascontiguousarray(full[:, :656])
    gpu = run_gpu(pa, case, cache)
    _, ref = run_oracle(case, cache)
    check_close(gpu, ref, abs_weighted(case, cache))
    wide = np.zeros((full.shape[0], 688), dtype=np.uint8)
    wide[:, :672] = full
    wide[:, 656:] = 0x7F
    assert np.array_equal(run_gpu(pa, case, wide), gpu)


def test_mla_deterministic(pa):
    case = small(seed=11)
    cache = case.cache()
    a = run_gpu(pa, case, cache)
    b = run_gpu(pa, case, cache)
    assert np.array_equal(a, b)


def test_mla_page_b64_sampled(pa):
    """The page's default decode case b=64, s_q=2, every sequence 65536 long
    (2 x 64 query tokens x 2048 selected keys): all heads of 6 tokens, spread
    over the batch, against the oracle."""
    case = workloads.mla_page_b64()
    used = case.rows_used()
    dev = torch.device("cuda")
    nrows = case.num_blocks * case.BS
    cache_d = torch.zeros((nrows, workloads.MLA_ROW_BYTES), dtype=torch.uint8, device=dev)
    rb = case.row_bytes(used)
    cache_d[torch.from_numpy(used).to(dev)] = torch.from_numpy(rb).to(dev)
    qn, qr = case.q_bf16()
    out = torch.empty((case.T, case.NQ, DN), dtype=torch.bfloat16, device=dev)
    st = pa.MlaStatus()
    pa.mla_sparse_decode(qn.to(dev), qr.to(dev), cache_d,
                         torch.from_numpy(case.topk_indices()).to(dev),
                         torch.from_numpy(case.block_table).to(dev),
                         torch.from_numpy(case.act).to(dev), out, S1=case.S1, status=st)
    torch.cuda.synchronize()
    assert st.value() == 0
    gpu = out.cpu().view(torch.int16).numpy().view(np.uint16)
    del cache_d
    toks = np.array([0, 1, 37, 64, 100, 127])
    rows = (toks[:, None] * case.NQ + np.arange(case.NQ)[None, :]).reshape(-1)
    host = np.zeros((nrows, workloads.MLA_ROW_BYTES), dtype=np.uint8)
    host[used] = rb
    _, ref = run_oracle(case, host, rows=rows)
    wabs = abs_weighted(case, host, tokens=toks)
    check_close(gpu[toks], ref[toks], wabs[toks])
