"""Host-side checks of the C-ABI library (no GPU needed): it builds, loads,
exports every function declared in include/pa_fp8.h, and rejects bad
arguments before touching the device."""
import ctypes

import numpy as np
import os
import re
import subprocess

import pytest

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa_fp8.h")


_KEEP = []


def _buf():
    """A small real buffer (64 KiB) for an argument that validation must reject
    before any use: device memory when a GPU is present, so that a regression
    that launched anyway would still touch valid memory; host memory otherwise
    (no kernel can run without a device)."""
    try:
        import torch
        if torch.cuda.is_available():
            t = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
            _KEEP.append(t)
            return ctypes.c_void_p(t.data_ptr())
    except ImportError:
        pass
    a = np.zeros(1 << 16, dtype=np.uint8)
    _KEEP.append(a)
    return ctypes.c_void_p(a.ctypes.data)


@pytest.fixture(scope="module")
def L():
    import fp8_paged_kv_block_gb300 as pa
    pa.build()
    return pa.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = declared_functions()
    for need in ("pa_fp8_decode", "pa_fp8_decode_workspace_size", "pa_fp8_cache_scatter",
                 "pa_fp8_cache_quant_scatter", "pa_fp8_quantize_rows",
                 "pa_fp8_value_channel_scale", "pa_fp8_kv_compress_epilog",
                 "pa_mla_sparse_decode", "pa_status_string",
                 "pa_last_error"):
        assert need in names


def test_library_exports_every_declared_symbol(L):
    import fp8_paged_kv_block_gb300 as pa
    out = subprocess.run(["nm", "-D", "--defined-only", pa.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(L, name)


def test_header_compiles_as_c():
    src = '#include "pa_fp8.h"\nint main(void){ pa_decode_config c = {0}; (void)c; return 0; }\n'
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER),
                        "-x", "c", "-", "-o", os.devnull], input=src, text=True,
                       capture_output=True)
    assert r.returncode == 0, r.stderr


def test_status_strings(L):
    for code in range(6):
        assert L.pa_status_string(code)
    assert b"PA_ERR_WORKSPACE" in L.pa_status_string(3)


def test_scatter_rejects_bad_arguments_without_launching(L):
    P = ctypes.c_void_p
    fake = _buf()  # never dereferenced: validation fails first
    st = L.pa_fp8_cache_scatter(None, fake, fake, fake, fake, 0, fake, 1, 1, fake, 4, 8, 128, 128,
                                2, 16, 1, None)
    assert st == 1 and b"NULL" in L.pa_last_error()
    st = L.pa_fp8_cache_scatter(fake, fake, fake, fake, fake, 0, fake, 1, 1, fake, 0, 8, 128, 128,
                                2, 16, 1, None)
    assert st == 2
    st = L.pa_fp8_cache_scatter(fake, fake, fake, fake, fake, 0, fake, 1, 1, fake, 4, 8, 128, 128,
                                2, 16, 7, None)
    assert st == 2 and b"layout" in L.pa_last_error()
    st = L.pa_fp8_cache_scatter(fake, fake, fake, fake, fake, 3, fake, 1, 1, fake, 4, 8, 128, 128,
                                2, 16, 1, None)
    assert st == 2


def test_decode_rejects_bad_arguments_without_launching(L):
    import fp8_paged_kv_block_gb300 as pa
    n = ctypes.c_size_t(0)
    assert L.pa_fp8_decode_workspace_size(16, 1, 96, 8, 64, None, ctypes.byref(n)) == 5
    assert b"head size" in L.pa_last_error()
    assert L.pa_fp8_decode_workspace_size(16, 1, 96, 7, 128, None, ctypes.byref(n)) == 2
    assert L.pa_fp8_decode_workspace_size(0, 1, 96, 8, 128, None, ctypes.byref(n)) == 2
    cfg = pa.pa_decode_config()
    cfg.s2_tile = 100
    assert L.pa_fp8_decode_workspace_size(16, 1, 96, 8, 128, ctypes.byref(cfg),
                                          ctypes.byref(n)) == 2
    cfg.s2_tile = 2048
    assert L.pa_fp8_decode_workspace_size(16, 1, 96, 8, 128, ctypes.byref(cfg),
                                          ctypes.byref(n)) == 5
    cfg.s2_tile = 1024   # built for up to 16 query rows per kv head
    cfg.num_ctas = 152   # no device query (no GPU here)
    assert L.pa_fp8_decode_workspace_size(16, 1, 96, 8, 128, ctypes.byref(cfg),
                                          ctypes.byref(n)) == 0
    assert L.pa_fp8_decode_workspace_size(16, 2, 96, 8, 128, ctypes.byref(cfg),
                                          ctypes.byref(n)) == 5
    assert b"1024" in L.pa_last_error()
    cfg.s2_tile = 512
    cfg.num_ctas = 0
    cfg.overlap_prologue = 3
    assert L.pa_fp8_decode_workspace_size(16, 1, 96, 8, 128, ctypes.byref(cfg),
                                          ctypes.byref(n)) == 2
    assert b"overlap_prologue" in L.pa_last_error()
    P = ctypes.c_void_p
    fake = _buf()
    st = L.pa_fp8_decode(fake, fake, None, fake, fake, fake, fake, fake, fake, 16, 1, 96, 8, 128,
                         128, 10, 4, 0, ctypes.c_float(0.088), None, fake, 1 << 20, None)
    assert st == 1


def test_quantizers_reject_bad_arguments(L):
    P = ctypes.c_void_p
    fake = _buf()
    assert L.pa_fp8_quantize_rows(fake, 0, 10, 6, fake, fake, None) == 5
    assert L.pa_fp8_quantize_rows(fake, 9, 10, 128, fake, fake, None) == 2
    assert L.pa_fp8_quantize_rows(None, 0, 10, 128, fake, fake, None) == 1
    assert L.pa_fp8_value_channel_scale(fake, 0, fake, 0, 10, 8, 128, fake, None) == 2
    assert L.pa_fp8_cache_quant_scatter(fake, fake, 0, fake, fake, fake, 0, fake, fake, fake, 1,
                                        4, 8, 126, 2, 16, 1, 0, None) == 5


def test_product_path_has_no_oracle_dependency():
    """The package must not import, load or call the oracle."""
    pkg = os.path.join(ROOT, "fp8_paged_kv_block_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text and "pa_oracle" not in text, f


def test_kv_compress_epilog_rejects_bad_arguments(L):
    P = ctypes.c_void_p
    fake = _buf()
    f = L.pa_fp8_kv_compress_epilog
    f.restype = ctypes.c_int
    f.argtypes = [P, ctypes.c_int64, ctypes.c_int, ctypes.c_int64, ctypes.c_int, P, ctypes.c_int64,
                  ctypes.c_int, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
    # cache, NB, BS, stride, head_dim, x, bs, d, slots, slot type, group, mode, round, stream
    assert f(None, 8, 16, 16 * 384, 384, fake, 4, 256, fake, 0, 64, 1, 1, None) == 1
    assert f(fake, 8, 16, 16 * 384, 384, fake, 4, 200, fake, 0, 64, 1, 1, None) == 2   # d % 64
    assert f(fake, 8, 16, 16 * 384, 384, fake, 4, 64, fake, 0, 64, 1, 1, None) == 2    # d > 64
    assert f(fake, 8, 16, 16 * 384, 384, fake, 4, 256, fake, 0, 32, 1, 1, None) == 2   # group 64
    assert f(fake, 8, 16, 16 * 384, 384, fake, 4, 256, fake, 0, 64, 2, 1, None) == 5   # HiF8/FP4
    assert f(fake, 8, 16, 16 * 322, 322, fake, 4, 256, fake, 0, 64, 1, 1, None) == 2   # 323 bytes
    assert b"323" in L.pa_last_error()
    assert f(fake, 8, 16, 16 * 326, 326, fake, 4, 256, fake, 0, 64, 0, 1, None) == 2   # mode 0: 352
    assert f(fake, 8, 16, 15 * 384, 384, fake, 4, 256, fake, 0, 64, 1, 1, None) == 2   # block stride


def test_mla_sparse_decode_rejects_bad_arguments(L):
    """Host validation of the MLA decode: every rejection happens before a
    launch (no GPU is needed to reach these answers)."""
    P = ctypes.c_void_p
    fake = _buf()
    f = L.pa_mla_sparse_decode
    scale = ctypes.c_float(1.0 / 24.0)

    def call(**kw):
        a = dict(qn=fake, qr=fake, cache=fake, row_bytes=672, tk=fake, bt=fake, act=fake, out=fake,
                 B=4, S1=2, NQ=128, n_kv=1, topk=2048, bs=128, nb=100, mb=512, s2=128, status=fake)
        a.update(kw)
        return f(a["qn"], a["qr"], a["cache"], a["row_bytes"], a["tk"], a["bt"], a["act"], a["out"],
                 a["B"], a["S1"], a["NQ"], a["n_kv"], a["topk"], a["bs"], a["nb"], a["mb"], scale,
                 a["s2"], a["status"], None)

    assert call(cache=None) == 1
    assert call(status=None) == 1
    assert call(row_bytes=640) == 2          # the 656 used bytes do not fit
    assert call(row_bytes=660) == 2          # not a multiple of 16
    assert call(topk=0) == 2
    assert call(S1=0) == 2
    assert call(n_kv=2) == 5                 # one latent KV head
    assert call(NQ=96) == 5                  # heads in groups of 64
    assert call(s2=512) == 5
    assert b"s2_tile" in L.pa_last_error()
    assert call(out=P(258)) == 2             # alignment
    assert call(B=0) == 0                    # nothing to do, nothing enqueued


def test_mla_sparse_decode_kvc_rejects_bad_arguments(L):
    """Host validation of the MLA decode over KV compress epilog rows: the
    shared checks, plus the quant mode (0 and 1 are built, 2 is HiFloat8)."""
    P = ctypes.c_void_p
    fake = _buf()
    f = L.pa_mla_sparse_decode_kvc
    scale = ctypes.c_float(1.0 / 24.0)

    def call(**kw):
        a = dict(qn=fake, qr=fake, cache=fake, row_bytes=672, stride=0, mode=0, tk=fake, bt=fake,
                 act=fake, out=fake, B=4, S1=2, NQ=128, n_kv=1, topk=2048, bs=128, nb=100, mb=512,
                 s2=128, status=fake)
        a.update(kw)
        return f(a["qn"], a["qr"], a["cache"], ctypes.c_int64(a["row_bytes"]),
                 ctypes.c_int64(a["stride"]), a["mode"], a["tk"],
                 a["bt"], a["act"], a["out"], a["B"], a["S1"], a["NQ"], a["n_kv"], a["topk"],
                 a["bs"], ctypes.c_int64(a["nb"]), a["mb"], scale, a["s2"], a["status"], None)

    assert call(mode=2) == 5                 # HiFloat8 / FP4 rows
    assert b"quant_mode" in L.pa_last_error()
    assert call(mode=3) == 2
    assert call(mode=-1) == 2
    assert call(cache=None) == 1
    assert call(row_bytes=648) == 2          # the minimum mode-1 row is not 16-byte aligned
    assert call(mode=1, row_bytes=648) == 2
    assert call(n_kv=2) == 5
    assert call(NQ=96) == 5
    assert call(s2=64) == 5
    assert call(qn=P(264)) == 2              # alignment
    assert call(stride=128 * 672 - 16) == 2  # blocks overlap
    assert b"block_stride" in L.pa_last_error()
    assert call(stride=128 * 672 + 8) == 2   # not a multiple of 16
    assert call(B=0) == 0
    assert call(mode=1, B=0) == 0
    assert call(B=0, stride=128 * 672 + 4096) == 0


def _c_kind(param):
    """The ctypes class a C parameter of the header needs."""
    p = " ".join(param.split())
    if "*" in p:
        return "ptr"
    base = p.rsplit(" ", 1)[0].replace("const ", "")
    return {"int": "i32", "int32_t": "i32", "pa_status": "i32", "int64_t": "i64",
            "size_t": "u64", "float": "f32"}[base]


def _ctypes_kind(t):
    if t is ctypes.c_void_p or t is ctypes.c_char_p or hasattr(t, "_type_") and \
            isinstance(getattr(t, "_type_"), type):
        return "ptr"
    if t is ctypes.c_float:
        return "f32"
    if issubclass(t, ctypes._SimpleCData):
        size, signed = ctypes.sizeof(t), t(-1).value == -1
        return {(4, True): "i32", (8, True): "i64", (8, False): "u64"}[(size, signed)]
    raise AssertionError(t)


def test_binding_argtypes_match_the_header(L):
    """Every entry point the Python binding declares to ctypes takes the
    header's parameters in order, with the same widths (a mismatch would pass
    garbage to the library without any error)."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    checked = 0
    for m in re.finditer(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(([^)]*)\)\s*;", text):
        name, params = m.group(1), [p for p in m.group(2).split(",") if p.strip() != "void"]
        argtypes = getattr(L, name).argtypes
        if argtypes is None:          # not marshalled by the binding (called directly in tests)
            continue
        want = [_c_kind(p) for p in params]
        got = [_ctypes_kind(t) for t in argtypes]
        assert got == want, (name, got, want)
        checked += 1
    assert checked >= 11


def test_auto_s2_tile_rule(L):
    """s2_tile 0: [PA] 配置说明's long-sequence tile of 1024 from s2 = 8192
    on (s2 = the block table's capacity), where at most 16 query rows share a
    kv head (the rows a 1024-token tile is built for); 512 otherwise."""
    import fp8_paged_kv_block_gb300 as pa
    f = L.pa_fp8_decode_auto_s2_tile
    assert f(1, 96, 8, 33 * 128) == 512          # GLM-4.5 bench shape: U[1, 4096]
    assert f(1, 96, 8, 8191) == 512
    assert f(1, 96, 8, 8192) == 1024             # the page's threshold
    assert f(1, 96, 8, 1025 * 128) == 1024       # 32K-131K contexts
    assert f(2, 96, 8, 129 * 128) == 512         # 24 rows per kv head: 1024 not built
    assert f(1, 128, 4, 1 << 20) == 512          # 32 rows per kv head
    assert f(1, 16, 1, 8192) == 1024             # 16 rows: still built
    for i, (b, s1, s2, nq, nkv) in enumerate(workloads.PAGE_CASES):
        cap = -(-s2 // 128) * 128
        want = 1024 if cap >= 8192 and s1 * nq // nkv <= 16 else 512
        assert pa.auto_s2_tile(s1, nq, nkv, cap) == want, i
    assert [pa.auto_s2_tile(s1, nq, nkv, -(-s2 // 128) * 128)
            for b, s1, s2, nq, nkv in workloads.PAGE_CASES] == [512, 1024, 1024, 1024, 512, 512]
    for bad in ((0, 8, 1, 100), (1, 0, 1, 100), (1, 8, 0, 100), (1, 12, 5, 100), (1, 8, 1, -1)):
        assert f(*bad) == 0
    with pytest.raises(ValueError):
        pa.auto_s2_tile(1, 12, 5, 100)
    # the workspace size does not depend on the tile, so s2_tile 0 sizes it
    assert (pa.decode_workspace_size(16, 1, 96, 8, num_ctas=152)
            == pa.decode_workspace_size(16, 1, 96, 8, s2_tile=512, num_ctas=152)
            == pa.decode_workspace_size(16, 1, 96, 8, s2_tile=128, num_ctas=152))


def test_prepared_calls_validate_before_touching_a_device(L):
    """prepare_decode / prepare_cache_quant_scatter check their tensors as
    decode() and cache_quant_scatter() do, before anything reaches the
    library: host tensors are refused."""
    torch = pytest.importorskip("torch")
    import fp8_paged_kv_block_gb300 as pa
    u8 = torch.zeros((2, 4, 128), dtype=torch.uint8)
    f32 = torch.zeros((2, 4), dtype=torch.float32)
    kc = torch.zeros((4, 128, 1, 128), dtype=torch.uint8)
    ks = torch.zeros((4, 128, 1), dtype=torch.float32)
    vs = torch.zeros((2, 1, 128), dtype=torch.float32)
    bt = torch.zeros((2, 1), dtype=torch.int32)
    act = torch.ones(2, dtype=torch.int32)
    out = torch.zeros((2, 4, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pa.prepare_decode(u8, f32, kc, ks, kc, ks, bt, act, out)
    kn = torch.zeros((2, 1, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pa.prepare_cache_quant_scatter(kn, kn, kc, kc, act, ks, vs, act)
