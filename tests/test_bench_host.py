"""Host-side helpers of bench.py (no GPU): how the oracle's sample is dealt to
threads, the host's thread count, and the MLA row-format table."""
import sys

import numpy as np

import bench
import fp8_paged_kv_block_gb300 as pa
import workloads


def test_deal_units_keeps_whole_units_round_robin():
    case = workloads.glm()
    G = case.group
    rows = [b * case.NQ + n2 * G + g for b in range(3) for n2 in range(case.NKV) for g in range(G)]
    for threads in (1, 5, 8, 64):
        chunks = bench.deal_units(case, rows, threads)
        flat = sorted(r for c in chunks for r in c)
        assert flat == sorted(rows)                                  # every row once
        for c in chunks:
            assert len(c) % G == 0
            for i in range(0, len(c), G):                            # whole units
                u = c[i:i + G]
                assert u == list(range(u[0], u[0] + G)) and u[0] % G == 0
        sizes = [len(c) // G for c in chunks]
        assert max(sizes) - min(sizes) <= 1 and len(chunks) == min(threads, len(rows) // G)


def test_host_threads_is_positive():
    assert bench.host_threads() >= 1


def test_mla_format_table(monkeypatch):
    for name, (fmt, mode, entry, rows) in bench.MLA_FORMATS.items():
        assert fmt in (workloads.MLA_FORMAT_PAGE, workloads.MLA_FORMAT_KVC_BF16,
                       workloads.MLA_FORMAT_KVC_E8M0)
        assert (mode is None) == (fmt == workloads.MLA_FORMAT_PAGE)
        assert hasattr(pa, entry)
        monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", "mla", "--mla-format", name])
        args = bench.parse_args()
        assert bench.mla_workload_name(args, 64).startswith(entry + ": b=64 ")
    # the traffic record belongs to one format only
    assert bench.MLA_TRAFFIC["format"] in bench.MLA_FORMATS


def test_configs_cover_every_decode_workload():
    names = [c[0] for c in bench.CONFIGS]
    assert names == ["tiny", "glm45", "long", "ragged", "append"]
    for _, make, _ in bench.CONFIGS:
        made = make()
        case = getattr(made, "ctx", made)
        assert case.algorithmic_bytes() > 0 and np.all(case.act >= 0)
