"""CPU oracle for FP8 paged decode attention and the FP8 cache-append scatter.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this package. The
product path (``fp8_paged_kv_block_gb300``) never imports it and shares no code
with it. The arithmetic lives in ``pa_oracle.c`` (plain C, single-threaded),
compiled with gcc on first use; this module only marshals numpy arrays.

Each function cites the page section it follows in ``pa_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

LAYOUT_BSND = 0
LAYOUT_BNBD = 1


def compile_source(src: str, out: str) -> str:
    """Compile one C source of the oracle into the shared library ``out``
    (gcc, C11, -O2, no fast-math, no FMA contraction)."""
    tmp = out + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off",
           "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into _build/liboracle.so (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # PA_ORACLE_LIB names another compiled copy of the oracle: the
        # planted-mistake tests load mutated copies this way, each in a
        # process of its own.
        lib = ctypes.CDLL(os.environ.get("PA_ORACLE_LIB") or build())
        P = ctypes.c_void_p
        i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.or_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.or_e4m3_decode.restype = ctypes.c_double
        lib.or_e4m3_encode.argtypes = [f32]
        lib.or_e4m3_encode.restype = ctypes.c_uint8
        lib.or_bf16_from_float.argtypes = [f32]
        lib.or_bf16_from_float.restype = ctypes.c_uint16
        lib.or_e4m3_encode_array.argtypes = [P, i64, P]
        lib.or_e4m3_encode_array.restype = None
        lib.or_bf16_from_float_array.argtypes = [P, i64, P]
        lib.or_bf16_from_float_array.restype = None
        lib.or_quant_rows.argtypes = [P, i64, i32, P, P]
        lib.or_quant_rows.restype = None
        lib.or_value_channel_scale.argtypes = [P, P, i32, i32, i32, P]
        lib.or_value_channel_scale.restype = None
        lib.or_quant_channels.argtypes = [P, P, i64, i32, i32, P, P]
        lib.or_quant_channels.restype = None
        lib.or_cache_scatter.argtypes = [P, P, P, P, P, P, i64, i64, P, i64, i32, i32,
                                         i32, i64, i32, i32]
        lib.or_cache_scatter.restype = None
        lib.or_cache_quant_scatter.argtypes = [P, P, P, P, P, P, P, P, i64, i32, i32, i32,
                                               i64, i32, i32]
        lib.or_cache_quant_scatter.restype = None
        lib.or_kvc_concat_bytes.argtypes = [i32, i32]
        lib.or_kvc_concat_bytes.restype = i64
        lib.or_kvc_min_head_dim.argtypes = [i32, i32]
        lib.or_kvc_min_head_dim.restype = i64
        lib.or_kv_compress_epilog.argtypes = [P, i64, i32, P, i64, i32, i64, i32, P, i32, i32]
        lib.or_kv_compress_epilog.restype = None
        lib.or_pa_decode.argtypes = [P, P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                     i32, i64, i32, i32, i32, f32, P, i64]
        lib.or_pa_decode.restype = ctypes.c_int
        lib.or_mla_sparse_decode.argtypes = [P, P, P, i64, P, i32, P, P, P, P, i32, i32, i32,
                                             i32, i64, i32, i32, f32, P, i64, i32]
        lib.or_mla_sparse_decode.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    """Contiguous array of exactly ``dtype`` (a copy only when needed)."""
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# Codec
# --------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """E4M3 code bytes -> float64 values (NaN for the NaN code)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib.or_e4m3_decode(i) for i in range(256)], dtype=np.float64)
    return table[c]


def e4m3_encode(x) -> np.ndarray:
    """float32 values -> E4M3 codes (RNE, saturating to +-448, NaN -> 0x7F)."""
    lib = _load()
    xs = _c(x, np.float32)
    out = np.empty(xs.shape, dtype=np.uint8)
    lib.or_e4m3_encode_array(_ptr(xs), xs.size, _ptr(out))
    return out


def bf16_from_float(x) -> np.ndarray:
    """float32 -> BF16 bit patterns (round to nearest even)."""
    lib = _load()
    xs = _c(x, np.float32)
    out = np.empty(xs.shape, dtype=np.uint16)
    lib.or_bf16_from_float_array(_ptr(xs), xs.size, _ptr(out))
    return out


def bf16_to_float(h) -> np.ndarray:
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# Quantisers
# --------------------------------------------------------------------------

def quant_rows(x):
    """x[..., D] float32 -> (codes uint8 [..., D], dequant scale float32 [...])."""
    lib = _load()
    x = _c(x, np.float32)
    D = x.shape[-1]
    rows = x.size // D
    codes = np.empty(x.shape, dtype=np.uint8)
    scale = np.empty(x.shape[:-1], dtype=np.float32)
    lib.or_quant_rows(_ptr(x), rows, D, _ptr(codes), _ptr(scale))
    return codes, scale


def value_channel_scale(v, cu_seqlens, B):
    """v[Ttot, H, D] float32, cu_seqlens[B+1] -> vscale[B, H, D] float32."""
    lib = _load()
    v = _c(v, np.float32)
    cu = _c(cu_seqlens, np.int64)
    _, H, D = v.shape
    out = np.empty((B, H, D), dtype=np.float32)
    lib.or_value_channel_scale(_ptr(v), _ptr(cu), B, H, D, _ptr(out))
    return out


def quant_channels(v, token_batch, vscale):
    """v[T, H, D] float32 with per-token batch ids -> codes uint8 [T, H, D]."""
    lib = _load()
    v = _c(v, np.float32)
    tb = _c(token_batch, np.int32)
    vs = _c(vscale, np.float32)
    T, H, D = v.shape
    codes = np.empty(v.shape, dtype=np.uint8)
    lib.or_quant_channels(_ptr(v), _ptr(tb), T, H, D, _ptr(vs), _ptr(codes))
    return codes


# --------------------------------------------------------------------------
# Scatter
# --------------------------------------------------------------------------

def cache_scatter(key, value, key_cache, value_cache, slot_mapping, key_scale,
                  key_scale_cache, layout=LAYOUT_BNBD):
    """In-place FP8 cache append. key/value uint8 [T, H, D*]; caches uint8,
    key_scale float32 [T, H] (any strides), key_scale_cache float32."""
    lib = _load()
    key = _c(key, np.uint8)
    value = _c(value, np.uint8)
    slot = _c(slot_mapping, np.int64)
    ks = np.asarray(key_scale, dtype=np.float32)
    assert key_cache.flags.c_contiguous and value_cache.flags.c_contiguous
    assert key_scale_cache.flags.c_contiguous
    T, H, Dk = key.shape
    Dv = value.shape[2]
    if layout == LAYOUT_BNBD:
        NB, _, BS, _ = key_cache.shape
    else:
        NB, BS, _, _ = key_cache.shape
    s0, s1 = ks.strides[0] // 4, ks.strides[1] // 4
    base = ks
    lib.or_cache_scatter(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                         _ptr(slot), ctypes.c_void_p(base.__array_interface__["data"][0]),
                         s0, s1, _ptr(key_scale_cache), T, H, Dk, Dv, NB, BS, layout)


def cache_quant_scatter(key, value, key_cache, value_cache, slot_mapping,
                        key_scale_cache, vscale, token_batch, layout=LAYOUT_BNBD):
    """In-place quantise-on-append. key/value float32 [T, H, D*] (BF16 sources
    are passed as their exact float32 values)."""
    lib = _load()
    key = _c(key, np.float32)
    value = _c(value, np.float32)
    slot = _c(slot_mapping, np.int64)
    vs = _c(vscale, np.float32)
    tb = _c(token_batch, np.int32)
    T, H, Dk = key.shape
    Dv = value.shape[2]
    if layout == LAYOUT_BNBD:
        NB, _, BS, _ = key_cache.shape
    else:
        NB, BS, _, _ = key_cache.shape
    lib.or_cache_quant_scatter(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                               _ptr(slot), _ptr(key_scale_cache), _ptr(vs), _ptr(tb),
                               T, H, Dk, Dv, NB, BS, layout)


def kvc_concat_bytes(d, quant_mode):
    """Bytes one KV-compress-epilog row writes (rope + nope codes + scales)."""
    return int(_load().or_kvc_concat_bytes(d, quant_mode))


def kvc_min_head_dim(d, quant_mode):
    """Smallest cache row pitch for KV compress epilog rows of width d."""
    return int(_load().or_kvc_min_head_dim(d, quant_mode))


def kv_compress_epilog(x, cache, block_num, block_size, block_stride, head_dim, slot_mapping,
                       quant_mode, round_scale):
    """In-place KV compress epilog (modes 0/1). x: float32 [bs, d] holding BF16
    values; cache: uint8 array of block_num * block_stride bytes."""
    lib = _load()
    x = _c(x, np.float32)
    slot = _c(slot_mapping, np.int64)
    assert cache.dtype == np.uint8 and cache.flags["C_CONTIGUOUS"]
    assert cache.size >= block_num * block_stride
    bs, d = x.shape
    lib.or_kv_compress_epilog(_ptr(x), bs, d, _ptr(cache), block_num, block_size, block_stride,
                              head_dim, _ptr(slot), quant_mode, int(bool(round_scale)))


# --------------------------------------------------------------------------
# Decode attention
# --------------------------------------------------------------------------

def pa_decode(q, q_scale, k_cache, k_scale, v_cache, v_scale, block_table, kv_act_seqs,
              *, S1, NKV, layout=LAYOUT_BSND, s2_tile=512, softmax_scale=None,
              rows=None, want_f32=False):
    """Paged FP8 decode attention.

    q uint8 [B*S1, NQ, D], q_scale float32 [B*S1, NQ], caches uint8 in
    ``layout``, k_scale float32 (cache shape with D=1), v_scale float32
    [B, NKV, D], block_table int32 [B, max_blocks], kv_act_seqs int32 [B].
    Returns BF16 bits uint16 [B*S1, NQ, D] (and the float32 values before the
    cast when ``want_f32``). ``rows`` restricts the work to the listed flat
    rows ``(b*S1+s)*NQ + h``; other rows are left zero.
    """
    lib = _load()
    q = _c(q, np.uint8)
    qs = _c(q_scale, np.float32)
    kc = _c(k_cache, np.uint8)
    ks = _c(k_scale, np.float32)
    vc = _c(v_cache, np.uint8)
    vs = _c(v_scale, np.float32)
    bt = _c(block_table, np.int32)
    act = _c(kv_act_seqs, np.int32)
    BS1, NQ, D = q.shape
    B = act.shape[0]
    assert BS1 == B * S1
    if layout == LAYOUT_BSND:
        NB, BS = kc.shape[0], kc.shape[1]
    else:
        NB, BS = kc.shape[0], kc.shape[2]
    max_blocks = bt.shape[1]
    if softmax_scale is None:
        softmax_scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    out = np.zeros((BS1, NQ, D), dtype=np.uint16)
    out32 = np.zeros((BS1, NQ, D), dtype=np.float32) if want_f32 else None
    r = None if rows is None else _c(rows, np.int64)
    nrows = 0 if r is None else r.size
    rc = lib.or_pa_decode(_ptr(q), _ptr(qs), _ptr(kc), _ptr(ks), _ptr(vc), _ptr(vs), _ptr(bt),
                          _ptr(act), _ptr(out), _ptr(out32), B, S1, NQ, NKV, D, BS, NB,
                          max_blocks, layout, s2_tile, softmax_scale, _ptr(r), nrows)
    if rc != 0:
        raise ValueError("or_pa_decode rejected its arguments")
    return (out, out32) if want_f32 else out


# --------------------------------------------------------------------------
# MLA sparse attention with FP8 anti-quantisation (decode)
# --------------------------------------------------------------------------

MLA_DN = 512
MLA_DR = 64
MLA_ROW_USED = 656


MLA_FORMAT_PAGE = 0        # [MS]: E4M3 kn | BF16 kr | 4 FP32 scales (per 128 channels)
MLA_FORMAT_KVC_BF16 = 1    # [KC] quant mode 0: BF16 kr | E4M3 kn | 8 BF16 scales (per 64)
MLA_FORMAT_KVC_E8M0 = 2    # [KC] quant mode 1: BF16 kr | E4M3 kn | 8 E8M0 scales (per 64)


def mla_sparse_decode(q_nope, q_rope, cache, topk_indices, block_table, kv_act_seqs, *, S1,
                      block_size=128, s2_tile=128, softmax_scale=None, rows=None,
                      want_f32=False, row_format=MLA_FORMAT_PAGE):
    """MLA sparse FP8 decode (the steps are listed in ``pa_oracle.c``).

    q_nope uint16 (BF16 bits) [T, NQ, 512], q_rope uint16 [T, NQ, 64] with
    T = B*S1; cache uint8 [num_blocks*block_size, row_bytes >= 656] packed rows
    in the layout ``row_format`` names (MLA_FORMAT_*); topk_indices int32 [T, topk];
    block_table int32 [B, max_blocks]; kv_act_seqs int32 [B]. Returns BF16 bits
    uint16 [T, NQ, 512] (and the float32 values before the cast when
    ``want_f32``). ``rows`` restricts the work to the flat rows ``t*NQ + h``;
    other rows are left zero.
    """
    lib = _load()
    qn = _c(q_nope, np.uint16)
    qr = _c(q_rope, np.uint16)
    kv = _c(cache, np.uint8)
    tk = _c(topk_indices, np.int32)
    bt = _c(block_table, np.int32)
    act = _c(kv_act_seqs, np.int32)
    T, NQ, dn = qn.shape
    assert dn == MLA_DN and qr.shape == (T, NQ, MLA_DR)
    B = act.shape[0]
    assert T == B * S1 and tk.shape[0] == T
    rows_total, row_bytes = kv.shape
    assert rows_total % block_size == 0
    num_blocks = rows_total // block_size
    if softmax_scale is None:
        softmax_scale = float(np.float32(1.0) / np.sqrt(np.float32(MLA_DN + MLA_DR)))
    out = np.zeros((T, NQ, MLA_DN), dtype=np.uint16)
    out32 = np.zeros((T, NQ, MLA_DN), dtype=np.float32) if want_f32 else None
    r = None if rows is None else _c(rows, np.int64)
    nrows = 0 if r is None else r.size
    rc = lib.or_mla_sparse_decode(_ptr(qn), _ptr(qr), _ptr(kv), row_bytes, _ptr(tk),
                                  tk.shape[1], _ptr(bt), _ptr(act), _ptr(out), _ptr(out32), B,
                                  S1, NQ, block_size, num_blocks, bt.shape[1], s2_tile,
                                  softmax_scale, _ptr(r), nrows, row_format)
    if rc != 0:
        raise ValueError("or_mla_sparse_decode rejected its arguments")
    return (out, out32) if want_f32 else out
