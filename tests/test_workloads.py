"""The seeded input recipe (no GPU): the generators are deterministic, a cache
row's bytes depend on its id alone (so any subset can be drawn), the KV compress
layouts hold the same codes and rope values as the page's packed rows, and the
shapes and ranges match the recipe."""
import numpy as np

import workloads


def test_decode_inputs_are_deterministic():
    a, b = workloads.glm(), workloads.glm()
    assert np.array_equal(a.act, b.act) and np.array_equal(a.block_table, b.block_table)
    assert np.array_equal(a.q(), b.q())
    ka, va = a.kv()
    kb, vb = b.kv()
    assert np.array_equal(ka, kb) and np.array_equal(va, vb)


def test_decode_block_tables_are_a_permutation_of_the_pool():
    for case in (workloads.tiny(), workloads.glm(), workloads.ragged()):
        used = case.block_table[case.block_table >= 0]
        assert np.unique(used).size == used.size                  # no block shared
        assert used.max() < case.num_blocks
        need = np.ceil(np.maximum(case.act, 0) / case.BS).astype(int)
        assert ((case.block_table >= 0).sum(axis=1) >= need).all()
        slots = case.slots
        assert np.unique(slots).size == slots.size


def test_recipe_ranges():
    g = workloads.glm()
    assert g.B == 16 and g.NQ == 96 and g.NKV == 8 and g.S1 == 1
    assert g.act.min() >= 1 and g.act.max() <= 4096
    r = workloads.ragged()
    assert r.B == 256 and r.S1 == 2 and r.act.min() >= 1 and r.act.max() <= 16384
    assert 700 < np.median(r.act) < 1400
    lc = workloads.long_ctx()
    assert lc.act.min() >= 32768 and lc.act.max() <= 131072


def test_mla_rows_depend_on_their_id_alone():
    case = workloads.mla_page_ragged()
    rows = np.array([5, 17, 123456, 9, 17], dtype=np.int64)
    for fmt in (workloads.MLA_FORMAT_PAGE, workloads.MLA_FORMAT_KVC_BF16,
                workloads.MLA_FORMAT_KVC_E8M0):
        together = case.row_bytes(rows, fmt)
        alone = np.stack([case.row_bytes(rows[i:i + 1], fmt)[0] for i in range(rows.size)])
        assert np.array_equal(together, alone)
        assert np.array_equal(together[1], together[4])


def test_mla_formats_hold_the_same_codes_and_rope():
    case = workloads.mla_page_ragged()
    rows = np.arange(0, 4000, 37, dtype=np.int64)
    page = case.row_bytes(rows, workloads.MLA_FORMAT_PAGE)
    for fmt in (workloads.MLA_FORMAT_KVC_BF16, workloads.MLA_FORMAT_KVC_E8M0):
        kvc = case.row_bytes(rows, fmt)
        assert np.array_equal(kvc[:, 128:640], page[:, :512])     # E4M3 codes
        assert np.array_equal(kvc[:, :128], page[:, 512:640])     # BF16 rope values
    # no code is the E4M3 NaN pattern; scales in the stated ranges
    assert not ((page[:, :512] & 0x7F) == 0x7F).any()
    s4 = page[:, 640:656].copy().view(np.float32)
    assert (s4 >= 0.004).all() and (s4 <= 0.009).all()
    b8 = (case.row_bytes(rows, workloads.MLA_FORMAT_KVC_BF16)[:, 640:656].copy()
          .view(np.uint16).astype(np.uint32) << 16).view(np.float32)
    assert (b8 >= 0.0039).all() and (b8 <= 0.009).all()
    e8 = case.row_bytes(rows, workloads.MLA_FORMAT_KVC_E8M0)[:, 640:648]
    assert set(np.unique(e8).tolist()) <= {119, 120}


def test_mla_key_rows_are_bf16_values_by_row_id():
    case = workloads.mla_page_ragged()
    rows = np.array([3, 1000, 3], dtype=np.int64)
    x = case.key_rows(rows)
    assert x.shape == (3, 576) and x.dtype == np.float32
    assert not (x.view(np.uint32) & 0xFFFF).any()                 # BF16-representable
    assert np.array_equal(x[0], x[2])
    assert np.array_equal(x[1], case.key_rows(np.array([1000]))[0])
