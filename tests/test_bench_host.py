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
    assert names == ["tiny", "glm45", "long", "ragged", "append"] + [
        "page%d" % i for i in range(len(workloads.PAGE_CASES))]
    for name, make, desc in bench.CONFIGS:
        made = make()
        case = getattr(made, "ctx", made)
        assert case.algorithmic_bytes() > 0 and np.all(case.act >= 0)
        assert case.s2_tile == 0, name            # the library's automatic tile
    for i, (b, s1, s2, nq, nkv) in enumerate(workloads.PAGE_CASES):
        case = bench.CONFIGS[5 + i][1]()
        assert (case.B, case.S1, case.NQ, case.NKV) == (b, s1, nq, nkv)
        assert np.all(case.act == s2)


def test_percentiles():
    d = bench.percentiles(list(range(1, 102)))
    assert d == {"median": 51.0, "p10": 11.0, "p90": 91.0, "samples": 101}


def test_unit_rows_and_parity_units():
    case = workloads.custom("u", 3, 2, 12, 2, [5, 0, 9])
    # S1 = 2, group 6: rows (b*2 + s)*12 + n2*6 + g
    assert bench.unit_rows(case, 1, 1) == [30, 31, 32, 33, 34, 35, 42, 43, 44, 45, 46, 47]
    every = bench.parity_units(case, case.act, 1e9, 1e-9)
    assert sorted(every) == [(b, n) for b in range(3) for n in range(2)]
    one = bench.parity_units(case, case.act, 0.0, 1.0)
    assert len(one) == 1
    assert bench.parity_units(case, case.act, 0.0, 1.0) == one      # seeded


def test_config_oracle_leg_reports_the_error_of_the_gpu_rows():
    """The configs sweep's oracle leg on a small case: fed the oracle's own
    output it reports zero error; one planted BF16 change shows as that
    row's difference."""
    import oracle
    from tests import _helpers as H
    case = workloads.custom("leg", 3, 1, 8, 2, [40, 300, 129], s2_tile=256)
    leg = bench.ConfigOracleLeg(case, None, case.act, 30.0)
    assert sorted(leg.units) == [(b, n) for b in range(3) for n in range(2)]
    full = H.oracle_decode(case, H.oracle_inputs(case))
    cpu, acc = leg.run(full)
    assert acc["max_abs"] == 0.0 and acc["within_tol"] and acc["rows"] == 3 * 8
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["value"] > 0
    bad = full.copy().reshape(-1, case.D)
    x = oracle.bf16_to_float(bad[5:6, 7:8]).astype(np.float64)[0, 0]
    bad[5, 7] = np.uint16(int(bad[5, 7]) ^ 0x0100)   # flip the lowest exponent bit
    y = oracle.bf16_to_float(bad[5:6, 7:8]).astype(np.float64)[0, 0]
    _, acc = leg.run(bad.reshape(full.shape))
    assert acc["max_abs"] == abs(x - y) > 0
    assert acc["mean_abs"] == abs(x - y) / (3 * 8 * case.D)


def test_host_cpu_record():
    rec = bench.host_cpu()
    assert isinstance(rec["cpu_model"], str) and rec["cpu_model"]
    assert rec["nproc"] >= 1
