"""Planted mistakes in the oracle: each must fail at least one pin.

The oracle is trusted only because its pins (tests/test_oracle.py and
tests/test_oracle_mla.py) tie it to the pages and to the mathematics. This
file checks that the pins are strong enough: for each plausible mistake (a
dropped rescale, a wrong index, a swapped operand, a skipped step) it edits
a copy of oracle/pa_oracle.c, compiles the copy with the oracle's own flags,
and runs the pins of that file against it in a separate process
(PA_ORACLE_LIB points the oracle module at the copy). A mistake that every
pin passes is a hole in the pins and fails here. Every edit keeps the copy's
memory accesses inside the buffers it is given, so a mutant can only give
wrong numbers, never crash.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pa_oracle.c")
DECODE_PINS = "tests/test_oracle.py"
MLA_PINS = "tests/test_oracle_mla.py"

# (name, pins file, [(text in pa_oracle.c, replacement), ...]); each text must
# occur exactly once in the oracle source.
MUTANTS = [
    # paged decode ([PA] 计算流程 steps 1-10)
    ("decode: O not rescaled by exp(M_old - M_new)", DECODE_PINS,
     [("O[d] = O[d] * alpha + (ot * ps)", "O[d] = O[d] + (ot * ps)")]),
    ("decode: running sum not rescaled", DECODE_PINS,
     [("L = L * alpha + sumP;", "L = L + sumP;")]),
    ("decode: sum taken over the quantised P", DECODE_PINS,
     [("L = L * alpha + sumP;", "L = L * alpha;"),
      ("            /* steps 7-9: MM2, dequant, accumulate */",
       "            for (j = 0; j < j1 - j0; ++j)\n"
       "                L += (float)or_e4m3_decode(P8[j]) * ps;\n")]),
    ("decode: GQA head map h % NKV instead of h / group", DECODE_PINS,
     [("n2 = h / group;", "n2 = h % NKV;")]),
    ("decode: softmax scale dropped", DECODE_PINS,
     [("* k_scale[krow]) * softmax_scale;", "* k_scale[krow]);")]),
    ("decode: P scale inverted (qs instead of 1/qs)", DECODE_PINS,
     [("ps = 1.0f / qs;", "ps = qs;")]),
    ("decode: value channel scale dropped", DECODE_PINS,
     [("(ot * ps) * v_scale[((int64_t)b * NKV + n2) * D + d];", "(ot * ps);")]),
    ("cache: PA_BSND and BNBD addressing swapped", DECODE_PINS,
     [("    if (layout == 0)\n        return (blk * BS + off) * H + h;",
       "    if (layout != 0)\n        return (blk * BS + off) * H + h;")]),
    ("decode: tokens past kv_act_seqs up to the block end not masked", DECODE_PINS,
     [("int j1 = (j0 + s2_tile < n) ? j0 + s2_tile : n;",
       "int nb = (n + BS - 1) / BS * BS;\n"
       "            int j1 = (j0 + s2_tile < nb) ? j0 + s2_tile : nb;")]),
    ("codec: E4M3 encode truncates instead of rounding to nearest even", DECODE_PINS,
     [("q = rne_nonneg(ldexp(a, 3 - e));", "q = floor(ldexp(a, 3 - e));")]),
    # MLA sparse decode ([MS] 计算流程, 在线反量化与 Online Softmax)
    ("mla: P not rounded to BF16 before C2", MLA_PINS,
     [("P[j] = or_bf16_to_float(or_bf16_from_float(p));", "P[j] = p;")]),
    ("mla: sum taken over the BF16 P", MLA_PINS,
     [("l += p;", "l += or_bf16_to_float(or_bf16_from_float(p));")]),
    ("mla: rope part left out of C1", MLA_PINS,
     [("acc += q[DN + c] * (double)kr[(int64_t)j * DR + c];", "acc += 0.0;")]),
    ("mla: merge factors of the running and the tile state swapped", MLA_PINS,
     [("O[c] = any ? O[c] * a + o * bb : o;", "O[c] = any ? O[c] * bb + o * a : o;"),
      ("L = any ? L * a + l * bb : l;", "L = any ? L * bb + l * a : l;")]),
    ("mla: tile sum merged without its factor", MLA_PINS,
     [("L = any ? L * a + l * bb : l;", "L = any ? L * a + l : l;")]),
    ("mla: scale groups of 64 channels instead of 128", MLA_PINS,
     [("sc[c] = s4[c / 2];", "sc[c] = s4[c % 4];")]),
    ("mla: visible count off by one", MLA_PINS,
     [("cur = act - S1 + 1 + s;", "cur = act - S1 + s;")]),
    ("mla: dequantised keys not rounded to BF16", MLA_PINS,
     [("kn[(int64_t)j * DN + c] = or_bf16_to_float(or_bf16_from_float(f));",
       "kn[(int64_t)j * DN + c] = f;")]),
    ("mla: positions read as physical rows (no block-table lookup)", MLA_PINS,
     [("blk = block_table[(int64_t)b * max_blocks + idx / BS];", "blk = idx / BS;")]),
    ("mla: positions masked by the table size, not by kv_act_seqs", MLA_PINS,
     [("ok[j] = (uint8_t)(idx >= 0 && idx < act);",
       "ok[j] = (uint8_t)(idx >= 0 && idx < max_blocks * BS);")]),
    ("mla: softmax scale dropped", MLA_PINS,
     [("S[j] = (float)acc * softmax_scale;", "S[j] = (float)acc;")]),
    # MLA decode of rows written by the KV compress epilog ([KC] 计算公式 场景 1 / 场景 2)
    ("mla kvc: group scales per 128 channels instead of 64", MLA_PINS,
     [("float f = (float)or_e4m3_decode(code[c]) * sc[c / 64];",
       "float f = (float)or_e4m3_decode(code[c]) * sc[row_format == 0 ? c / 64 : c / 128];")]),
    ("mla kvc: E8M0 exponent bias 128 instead of 127", MLA_PINS,
     [("(int)kv[640 + c] - 127)", "(int)kv[640 + c] - 128)")]),
    ("mla kvc: BF16 scale bytes read big-endian", MLA_PINS,
     [("(kv[640 + 2 * c] |\n", "(kv[640 + 2 * c + 1] |\n"),
      ("(kv[640 + 2 * c + 1] << 8)))", "(kv[640 + 2 * c] << 8)))")]),
    ("mla kvc: rope read where the page row keeps it", MLA_PINS,
     [("rope = kv;", "rope = kv + DN;")]),
    ("mla kvc: codes read from the row start", MLA_PINS,
     [("code = kv + 2 * DR;", "code = kv;")]),
    ("mla kvc: E8M0 byte 0 read as a zero scale", MLA_PINS,
     [("(float)ldexp(1.0, (int)kv[640 + c] - 127)",
       "(kv[640 + c] ? (float)ldexp(1.0, (int)kv[640 + c] - 127) : 0.0f)")]),
]


def _mutate(text, edits):
    for old, new in edits:
        n = text.count(old)
        assert n == 1, "edit target occurs %d times in pa_oracle.c: %r" % (n, old)
        text = text.replace(old, new)
    return text


def _run_pins(lib, pins):
    env = dict(os.environ, PA_ORACLE_LIB=lib)
    return subprocess.run([sys.executable, "-m", "pytest", pins, "-q", "-x", "-p",
                           "no:cacheprovider", "-m", "not gpu"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_every_planted_mistake_fails_a_pin(tmp_path):
    with open(SRC) as fh:
        text = fh.read()
    jobs = []
    for i, (name, pins, edits) in enumerate(MUTANTS):
        src = tmp_path / ("mutant%02d.c" % i)
        src.write_text(_mutate(text, edits))
        lib = oracle.compile_source(str(src), str(tmp_path / ("libmutant%02d.so" % i)))
        jobs.append((name, pins, lib))
    # the unmutated oracle passes both files of pins through the same route
    clean = oracle.build()
    jobs.append(("(none)", DECODE_PINS, clean))
    jobs.append(("(none)", MLA_PINS, clean))
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda j: (j, _run_pins(j[2], j[1])), jobs))
    survivors, errors = [], []
    for (name, pins, _), r in results:
        if name == "(none)":
            if r.returncode != 0:
                errors.append("unmutated oracle fails %s:\n%s" % (pins, r.stdout[-2000:]))
        elif r.returncode == 0:
            survivors.append(name)
        elif r.returncode != 1:      # 1 = some pin failed; anything else is not a pin
            errors.append("%s: pytest exit %d\n%s%s" % (name, r.returncode, r.stdout[-1500:],
                                                         r.stderr[-1500:]))
    assert not errors, "\n\n".join(errors)
    assert not survivors, "planted mistakes that pass every pin: %s" % survivors


@pytest.mark.parametrize("name,pins,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_applies_once(name, pins, edits):
    with open(SRC) as fh:
        text = fh.read()
    assert _mutate(text, edits) != text
