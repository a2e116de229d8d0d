"""Pins for the MLA sparse FP8 decode oracle (no GPU).

The oracle (``oracle.mla_sparse_decode``) follows the steps of the DeepSeek
V3.2 MLA sparse attention FP8 anti-quantisation page. Here it is checked
against things other than itself: brute-force FP64 attention, closed forms
computed with torch's float8_e4m3fn / bfloat16 conversions, the online merge
written out for keys in separate tiles, and invariances (padding bytes,
physical block placement, entries past the visible count, masked entries,
key order within a tile).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads

DN, DR = 512, 64


def small_case(B=2, S1=2, NQ=4, act=(300, 41), topk=64, seed=7, frac_invalid=0.0, BS=128):
    return workloads.mla("small", B, S1, list(act), NQ=NQ, topk=topk,
                         seed=workloads.BASE_SEED + 300 + seed, frac_invalid=frac_invalid, BS=BS)


def run(case, cache=None, topk=None, s2_tile=None, bt=None, want_f32=True, rows=None):
    qn, qr = case.q_bits()
    return oracle.mla_sparse_decode(
        qn, qr, case.cache() if cache is None else cache,
        case.topk_indices() if topk is None else topk,
        case.block_table if bt is None else bt, case.act, S1=case.S1, block_size=case.BS,
        s2_tile=case.s2_tile if s2_tile is None else s2_tile, softmax_scale=case.softmax_scale,
        rows=rows, want_f32=want_f32)


# ---- independent dequantisation with torch ---------------------------------

def torch_keys(case, cache, rows):
    """(kn BF16 values as float64 [n, 512], kr float64 [n, 64]) of the given
    physical rows, dequantised with torch: E4M3 -> float32, times the FP32
    scale of each 128-channel group, rounded to BF16."""
    r = torch.from_numpy(cache[np.asarray(rows)].copy())
    codes = r[:, :DN].contiguous().view(torch.float8_e4m3fn).to(torch.float32)
    scale = r[:, DN + 2 * DR:DN + 2 * DR + 16].contiguous().view(torch.float32)
    kn = (codes * scale.repeat_interleave(128, dim=1)).to(torch.bfloat16).to(torch.float64)
    kr = r[:, DN:DN + 2 * DR].contiguous().view(torch.bfloat16).to(torch.float64)
    return kn.numpy(), kr.numpy()


def torch_query(case, t, h):
    qn, qr = case.q_bf16()
    return np.concatenate([qn[t, h].double().numpy(), qr[t, h].double().numpy()])


def selected(case, t):
    """Physical rows of token t's valid selected keys, in list order."""
    b, s = divmod(t, case.S1)
    n = int(case.cur()[t])
    idx = case.topk_indices()[t, :n].astype(np.int64)
    idx = idx[(idx >= 0) & (idx < case.act[b])]
    return case.physical_rows(idx, np.full(idx.shape, b))


# ---- brute force ------------------------------------------------------------

@pytest.mark.parametrize("s2_tile", [128, 16, 5])
def test_mla_vs_bruteforce_fp64(s2_tile):
    """Unquantised-softmax FP64 attention over the dequantised keys: the
    oracle differs only by the BF16 casts of the keys and P."""
    case = small_case(frac_invalid=0.1)
    cache = case.cache()
    _, out32 = run(case, cache=cache, s2_tile=s2_tile)
    worst = 0.0
    for t in range(case.T):
        rows = selected(case, t)
        for h in range(case.NQ):
            if rows.size == 0:
                assert not out32[t, h].any()
                continue
            codes = cache[rows, :DN]
            sc = cache[rows, DN + 2 * DR:DN + 2 * DR + 16].copy().view(np.float32)
            kn = oracle.e4m3_decode(codes) * np.repeat(sc.astype(np.float64), 128, axis=1)
            kr = cache[rows, DN:DN + 2 * DR].copy().view(np.uint16).astype(np.uint32) << 16
            kr = kr.view(np.float32).astype(np.float64)
            q = torch_query(case, t, h)
            s = (np.concatenate([kn, kr], axis=1) @ q) * case.softmax_scale
            w = np.exp(s - s.max())
            ref = (w / w.sum()) @ kn
            worst = max(worst, float(np.abs(out32[t, h] - ref).max()))
    # BF16 keys and P carry 2^-9 relative error each
    assert worst < 2e-2, worst


# ---- closed forms -----------------------------------------------------------

def test_mla_single_key_gives_its_bf16_nope_row():
    """One visible key: P = 1 and L = 1, so every head outputs that key's
    dequantised, BF16-rounded nope row, bit for bit."""
    case = small_case(act=(1, 1), S1=1, B=2, topk=8)
    cache = case.cache()
    out = run(case, cache=cache, want_f32=False)
    for t in range(case.T):
        rows = selected(case, t)
        assert rows.size == 1
        kn, _ = torch_keys(case, cache, rows)
        want = torch.from_numpy(kn[0]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        for h in range(case.NQ):
            assert np.array_equal(out[t, h], want)


def _two_key_case(gap):
    """One token, two visible keys; the second key's rope part is shifted so
    that its score is `gap` below the first's."""
    case = small_case(B=1, S1=1, NQ=2, act=(2,), topk=2)
    cache = case.cache()
    rows = selected(case, 0)
    return case, cache, rows


def test_mla_two_keys_one_tile_closed_form():
    """Two keys in one tile: O = (P_1 kn_1 + P_2 kn_2) / (p_1 + p_2) with
    p = exp(S - max S) and P = BF16(p) (the numerator uses the BF16 P, the sum
    the FP32 p). Scores include the rope part."""
    case, cache, rows = _two_key_case(0.0)
    _, out32 = run(case, cache=cache, s2_tile=128)
    kn, kr = torch_keys(case, cache, rows)
    for h in range(case.NQ):
        q = torch_query(case, 0, h)
        s = (np.concatenate([kn, kr], axis=1) @ q) * np.float64(np.float32(case.softmax_scale))
        p = np.exp(s - s.max())
        P = torch.from_numpy(p.astype(np.float32)).to(torch.bfloat16).double().numpy()
        want = (P @ kn) / p.sum()
        np.testing.assert_allclose(out32[0, h], want, rtol=2e-5, atol=1e-6)
        # dropping the rope part would change the weights
        s_nr = (kn @ q[:DN]) * case.softmax_scale
        assert abs((s - s.max())[0] - (s_nr - s_nr.max())[0]) > 1e-3 or \
            abs((s - s.max())[1] - (s_nr - s_nr.max())[1]) > 1e-3


def test_mla_two_keys_two_tiles_online_merge():
    """Keys in separate tiles (s2_tile 1): each tile has P = 1 exactly, so the
    merge O = a o_1 + b o_2, L = a + b with a = exp(m_1 - M), b = exp(m_2 - M)
    gives the exact softmax weighting of the two BF16 nope rows."""
    case, cache, rows = _two_key_case(0.0)
    _, out32 = run(case, cache=cache, s2_tile=1)
    kn, kr = torch_keys(case, cache, rows)
    for h in range(case.NQ):
        q = torch_query(case, 0, h)
        s = (np.concatenate([kn, kr], axis=1) @ q) * np.float64(np.float32(case.softmax_scale))
        w = np.exp(s - s.max())
        want = (w @ kn) / w.sum()
        np.testing.assert_allclose(out32[0, h], want, rtol=2e-5, atol=1e-6)


def test_mla_tile_size_changes_only_the_bf16_rounding_of_p():
    """Tile-local P: with one tile per key there is no BF16 rounding of P at
    all; with one tile for all keys there is. The two agree to BF16 accuracy
    but not bit for bit."""
    case = small_case(B=1, S1=1, act=(60,), topk=64)
    cache = case.cache()
    _, a = run(case, cache=cache, s2_tile=1)
    _, b = run(case, cache=cache, s2_tile=128)
    assert not np.array_equal(a, b)
    np.testing.assert_allclose(a, b, atol=2e-3 * np.abs(a).max())


# ---- the visible count, masking and addressing --------------------------------

def test_mla_visible_count_rule():
    """Token s of a sequence of length n attends to min(n - S1 + 1 + s, topk)
    selected keys: entries past that count are never read, and a token with
    no visible key gets zeros."""
    case = small_case(B=3, S1=3, act=(200, 2, 1), topk=64)
    assert case.cur().tolist() == [64, 64, 64, 0, 1, 2, 0, 0, 1]
    cache = case.cache()
    tk = case.topk_indices().copy()
    base = run(case, cache=cache, topk=tk, want_f32=False)
    cur = case.cur()
    t2 = tk.copy()
    for t in range(case.T):
        # fill the unread tail with valid positions of the sequence
        b = t // case.S1
        t2[t, cur[t]:] = np.arange(case.topk - cur[t]) % max(int(case.act[b]), 1)
    assert np.array_equal(run(case, cache=cache, topk=t2, want_f32=False), base)
    for t in np.nonzero(cur == 0)[0]:
        assert not base[t].any()


def test_mla_masked_entries_take_no_part():
    """Within one tile, entries that are -1 or past kv_act_seqs contribute
    nothing: the output equals that of the list with them removed."""
    case = small_case(B=1, S1=1, act=(100,), topk=64)
    cache = case.cache()
    tk = case.topk_indices().copy()
    n = int(case.cur()[0])
    bad = tk.copy()
    bad[0, 3] = -1
    bad[0, 10] = case.act[0]          # one past the end
    bad[0, 20] = case.act[0] + 500
    keep = [j for j in range(n) if j not in (3, 10, 20)]
    comp = np.full_like(tk, -1)
    comp[0, :len(keep)] = tk[0, keep]
    _, a = run(case, cache=cache, topk=bad)
    _, b = run(case, cache=cache, topk=comp)
    np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-7)


def test_mla_key_order_within_a_tile():
    """Permuting the selected entries of a one-tile list changes only the
    order of FP32 sums."""
    case = small_case(B=1, S1=1, act=(120,), topk=64)
    cache = case.cache()
    tk = case.topk_indices().copy()
    n = int(case.cur()[0])
    perm = tk.copy()
    perm[0, :n] = tk[0, np.random.default_rng(3).permutation(n)]
    _, a = run(case, cache=cache, topk=tk)
    _, b = run(case, cache=cache, topk=perm)
    np.testing.assert_allclose(a, b, rtol=1e-5, atol=1e-7)


def test_mla_block_placement_invariance():
    """Moving the physical blocks and rewriting the block table accordingly
    leaves every output bit unchanged."""
    case = small_case(B=2, S1=2, act=(300, 130), topk=64)
    cache = case.cache()
    base = run(case, cache=cache, want_f32=False)
    nb = case.num_blocks
    perm = np.random.default_rng(11).permutation(nb)      # old block i -> new perm[i]
    moved = np.empty_like(cache).reshape(nb, case.BS, -1)
    moved[perm] = cache.reshape(nb, case.BS, -1)
    bt = np.where(case.block_table >= 0, perm[np.maximum(case.block_table, 0)], -1).astype(np.int32)
    assert np.array_equal(run(case, cache=moved.reshape(cache.shape), bt=bt, want_f32=False), base)


def test_mla_padding_and_unread_bytes_are_not_read():
    """Bytes 656..671 of every row, and every row no valid entry selects, may
    hold anything."""
    case = small_case(B=2, S1=2, act=(300, 130), topk=64, frac_invalid=0.05)
    cache = case.cache()
    base = run(case, cache=cache, want_f32=False)
    noisy = cache.copy()
    noisy[:, 656:] = np.random.default_rng(5).integers(0, 256, size=noisy[:, 656:].shape)
    used = case.rows_used()
    unused = np.setdiff1d(np.arange(cache.shape[0]), used)
    noisy[unused] = 0x7F        # E4M3 NaN codes
    assert np.array_equal(run(case, cache=noisy, want_f32=False), base)
    # and the generator's own sparse cache gives the same result
    assert np.array_equal(run(case, cache=case.cache(rows=used), want_f32=False), base)


def test_mla_group_scale_assignment():
    """The scale of group g multiplies exactly channels 128g..128g+127 of kn:
    doubling one group's scale of the single visible key doubles (before the
    BF16 cast, exactly) that group's output channels only."""
    case = small_case(B=1, S1=1, act=(1,), topk=4)
    cache = case.cache()
    row = selected(case, 0)[0]
    _, a = run(case, cache=cache)
    for g in range(4):
        c2 = cache.copy()
        sc = c2[row, 640:656].copy().view(np.float32)
        sc[g] *= 2
        c2[row, 640:656] = sc.view(np.uint8)
        _, b = run(case, cache=c2)
        sel = np.zeros(DN, bool)
        sel[128 * g:128 * (g + 1)] = True
        np.testing.assert_array_equal(b[0, :, ~sel], a[0, :, ~sel])
        np.testing.assert_allclose(b[0, :, sel], 2 * a[0, :, sel], rtol=2 ** -8)


def test_mla_rows_subset_matches_full():
    case = small_case(frac_invalid=0.05)
    cache = case.cache()
    full = run(case, cache=cache, want_f32=False)
    rows = np.array([0, 5, 7, case.T * case.NQ - 1], dtype=np.int64)
    part = run(case, cache=cache, rows=rows, want_f32=False)
    flat_f, flat_p = full.reshape(-1, DN), part.reshape(-1, DN)
    assert np.array_equal(flat_p[rows], flat_f[rows])
    others = np.setdiff1d(np.arange(flat_p.shape[0]), rows)
    assert not flat_p[others].any()


def test_mla_page_cases_shapes():
    """The page's decode cases: b=4 s_q=2 lengths [65536, 16381, 666, 15] and
    b=64 s_q=2 lengths 65536; topk 2048, 128 heads, block size 128."""
    c = workloads.mla_page_ragged()
    assert (c.B, c.S1, c.NQ, c.topk, c.BS) == (4, 2, 128, 2048, 128)
    assert c.cur().tolist() == [2048, 2048, 2048, 2048, 665, 666, 14, 15]
    tk = c.topk_indices()
    for t in range(c.T):
        n = int(c.cur()[t])
        b, s = divmod(t, c.S1)
        sel = tk[t, :n]
        assert len(np.unique(sel)) == n and sel.min() >= 0
        assert sel.max() < c.act[b] - c.S1 + 1 + s
        assert (tk[t, n:] == -1).all()
    c64 = workloads.mla_page_b64()
    assert (c64.B, c64.S1, int(c64.act.min()), int(c64.act.max())) == (64, 2, 65536, 65536)


# ---- rows written by the KV compress epilog (quant modes 0 and 1) ----------------------
# The CANN aclnnKvCompressEpilog page's row for d = 576: the rope part first as BF16, the nope
# part as E4M3 in groups of 64 channels, one scale per group (BF16 in quant mode 0, an E8M0
# power of two in quant mode 1). The decode dequantises it with the MLA page's rule
# (BF16(FP32(code) * scale)), each group by its own scale.

KVC_FORMATS = [workloads.MLA_FORMAT_KVC_BF16, workloads.MLA_FORMAT_KVC_E8M0]


def run_fmt(case, cache, fmt, want_f32=True, s2_tile=None):
    qn, qr = case.q_bits()
    return oracle.mla_sparse_decode(qn, qr, cache, case.topk_indices(), case.block_table,
                                    case.act, S1=case.S1, block_size=case.BS,
                                    s2_tile=case.s2_tile if s2_tile is None else s2_tile,
                                    softmax_scale=case.softmax_scale, want_f32=want_f32,
                                    row_format=fmt)


def kvc_rows_from_page_rows(page, fmt):
    """The same keys moved into the KV compress row: rope bytes first, then the codes, then
    each 128-channel FP32 scale twice as two 64-channel scales (BF16 bits, or the E8M0 byte
    of a power of two). Only scales that the KV compress format holds exactly are allowed."""
    out = np.full_like(page, 0xFF)
    out[:, :2 * DR] = page[:, DN:DN + 2 * DR]
    out[:, 2 * DR:2 * DR + DN] = page[:, :DN]
    s4 = page[:, 640:656].copy().view(np.float32)
    s8 = np.repeat(s4, 2, axis=1)
    if fmt == workloads.MLA_FORMAT_KVC_BF16:
        bits = s8.view(np.uint32)
        assert not (bits & 0xFFFF).any(), "scale not exact in BF16"
        out[:, 640:656] = (bits >> 16).astype(np.uint16).view(np.uint8).reshape(-1, 16)
    else:
        m, e = np.frexp(s8.astype(np.float64))
        assert (m == 0.5).all(), "scale not a power of two"
        out[:, 640:648] = (e - 1 + 127).astype(np.uint8)
    return out


@pytest.mark.parametrize("fmt", KVC_FORMATS)
def test_mla_kvc_row_equals_the_page_row_holding_the_same_keys(fmt):
    """Page-format rows whose scales the KV compress row can hold exactly (BF16 values; powers
    of two) are moved byte by byte into the KV compress layout: the outputs are bit-identical,
    so the new layout is read as the same keys through the pinned page-format path."""
    case = small_case(frac_invalid=0.1, act=(300, 141))
    page = case.cache()
    s4 = page[:, 640:656].copy().view(np.uint32)
    if fmt == workloads.MLA_FORMAT_KVC_BF16:
        s4 &= np.uint32(0xFFFF0000)
    else:
        k = np.random.default_rng(2).integers(-9, -6, size=s4.shape)
        s4[:] = (np.ldexp(1.0, k).astype(np.float32)).view(np.uint32)
    page[:, 640:656] = s4.view(np.uint8).reshape(-1, 16)
    kvc = kvc_rows_from_page_rows(page, fmt)
    a, a32 = run(case, cache=page)
    b, b32 = run_fmt(case, kvc, fmt)
    assert np.array_equal(a, b) and np.array_equal(a32, b32)
    assert np.abs(a32).max() > 0.1


@pytest.mark.parametrize("fmt", KVC_FORMATS)
def test_mla_kvc_single_key_gives_its_dequantised_row(fmt):
    """One visible key: every head outputs that key's nope row dequantised with torch (E4M3
    codes at bytes 128..639 to float32, times the scale of each 64 channels, to BF16), bit for
    bit."""
    case = small_case(act=(1, 1), S1=1, B=2, topk=8)
    cache = case.cache(fmt=fmt)
    out = run_fmt(case, cache, fmt, want_f32=False)
    for t in range(case.T):
        rows = selected(case, t)
        assert rows.size == 1
        r = torch.from_numpy(cache[rows].copy())
        codes = r[:, 2 * DR:2 * DR + DN].contiguous().view(torch.float8_e4m3fn).to(torch.float32)
        if fmt == workloads.MLA_FORMAT_KVC_BF16:
            sc = r[:, 640:656].contiguous().view(torch.bfloat16).to(torch.float32)
        else:
            sc = torch.pow(2.0, r[:, 640:648].to(torch.float32) - 127.0)
        kn = (codes * sc.repeat_interleave(64, dim=1)).to(torch.bfloat16)
        want = kn[0].view(torch.int16).numpy().view(np.uint16)
        for h in range(case.NQ):
            assert np.array_equal(out[t, h], want)


@pytest.mark.parametrize("fmt", KVC_FORMATS)
def test_mla_kvc_padding_after_the_scales_is_not_used(fmt):
    case = small_case(act=(300, 41))
    cache = case.cache(fmt=fmt)
    end = 656 if fmt == workloads.MLA_FORMAT_KVC_BF16 else 648
    other = cache.copy()
    other[:, end:] = np.random.default_rng(4).integers(0, 256, size=other[:, end:].shape,
                                                       dtype=np.uint8)
    a, a32 = run_fmt(case, cache, fmt)
    b, b32 = run_fmt(case, other, fmt)
    assert np.array_equal(a, b) and np.array_equal(a32, b32)


@pytest.mark.parametrize("mode,round_scale", [(0, False), (1, True)])
def test_mla_kvc_reads_what_the_compress_epilog_wrote(mode, round_scale):
    """The append-then-attend chain on the CPU: BF16 key rows x = [nope 512 | rope 64] go
    through the KV compress epilog oracle into a paged cache, and the decode over that cache
    matches FP64 softmax attention over x itself (keys [nope, rope], values the nope part)
    within the quantisation error: E4M3 codes carry up to 2^-4 relative error per channel
    (an E8M0 scale rounded up doubles it), BF16 keys and P 2^-9; measured worst 0.025 (mode
    0) and 0.033 (mode 1), a layout or scale mistake gives errors of order 1. Quant mode 1
    without roundScale is left out: its power of two at or below max|x|/448 saturates the
    group's largest values at 448 by design (pinned with the epilog oracle itself)."""
    case = small_case(B=2, S1=2, NQ=4, act=(300, 141), topk=96, frac_invalid=0.1)
    rows = case.rows_used()
    x = torch.from_numpy(case.key_rows(rows))
    assert torch.equal(x.to(torch.bfloat16).float(), x)
    cache = np.zeros((case.num_blocks * case.BS, workloads.MLA_ROW_BYTES), dtype=np.uint8)
    oracle.kv_compress_epilog(x.numpy(), cache,
                              case.num_blocks, case.BS, case.BS * workloads.MLA_ROW_BYTES,
                              workloads.MLA_ROW_BYTES, rows.astype(np.int64), quant_mode=mode,
                              round_scale=round_scale)
    fmt = workloads.MLA_FORMAT_KVC_BF16 if mode == 0 else workloads.MLA_FORMAT_KVC_E8M0
    _, out32 = run_fmt(case, cache, fmt)
    key_of_row = {int(r): i for i, r in enumerate(rows)}
    xd = x.double().numpy()
    assert abs(xd.std() - 1.0) < 0.05
    worst = 0.0
    for t in range(case.T):
        sel = selected(case, t)
        for h in range(case.NQ):
            if sel.size == 0:
                assert not out32[t, h].any()
                continue
            k = xd[[key_of_row[int(r)] for r in sel]]
            s = (k @ torch_query(case, t, h)) * case.softmax_scale
            w = np.exp(s - s.max())
            ref = (w / w.sum()) @ k[:, :DN]
            worst = max(worst, float(np.abs(out32[t, h] - ref).max()))
    assert worst < 0.1, worst


def test_mla_kvc_e8m0_extreme_exponents():
    """E8M0 scale bytes at the ends of what the epilog writes: byte 0 is 2^-127 (an FP32
    subnormal, kept, not flushed) and small bytes give subnormal products; one visible key
    outputs its row dequantised with torch, bit for bit."""
    case = small_case(act=(1, 1), S1=1, B=2, topk=8)
    cache = case.cache(fmt=workloads.MLA_FORMAT_KVC_E8M0)
    rows = [int(selected(case, t)[0]) for t in range(case.T)]
    cache[rows[0], 640:648] = [0, 1, 2, 127, 0, 3, 1, 0]
    cache[rows[1], 640:648] = [126, 127, 128, 130, 0, 0, 2, 1]
    out = run_fmt(case, cache, workloads.MLA_FORMAT_KVC_E8M0, want_f32=False)
    for t in range(case.T):
        r = torch.from_numpy(cache[rows[t]:rows[t] + 1].copy())
        codes = r[:, 2 * DR:2 * DR + DN].contiguous().view(torch.float8_e4m3fn).to(torch.float32)
        sc = torch.tensor([np.ldexp(1.0, int(e) - 127) for e in cache[rows[t], 640:648]],
                          dtype=torch.float64).to(torch.float32)
        kn = (codes * sc.repeat_interleave(64)).to(torch.bfloat16)
        want = kn[0].view(torch.int16).numpy().view(np.uint16)
        if t == 0:
            assert (want[:64] != 0).any() and (np.abs(kn[0, :64].float().numpy()) < 2.0 ** -126).any()
        for h in range(case.NQ):
            assert np.array_equal(out[t, h], want)
