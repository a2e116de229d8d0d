"""GB300 (sm_103a) FP8 paged-KV decode attention and cache append.

Thin ctypes binding over the C ABI declared in ``include/pa_fp8.h``
(``libpa_fp8.so``). This module only marshals arguments: every step runs in
the library's CUDA kernels. PyTorch supplies device memory and the current
stream. There is no fallback: if the library is missing, calls raise.

Functions take torch CUDA tensors and work in place (outputs are arguments):
  decode(...)              paged FP8 decode attention -> BF16
  cache_scatter(...)       FP8 K/V (+ key_scale) append by slot_mapping
  cache_quant_scatter(...) BF16/FP32 K/V quantised to E4M3 on append
  kv_compress_epilog(...)  BF16 rows to rope (BF16) + grouped E4M3 nope (modes 0/1)
  quantize_rows(...)       per-token E4M3 quantiser (Q, K)
  value_channel_scale(...) per-channel V dequant scale
  mla_sparse_decode(...)   MLA sparse attention over a packed FP8 latent cache
  mla_sparse_decode_kvc(...) the same over rows the KV compress epilog wrote
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from . import _build

LAYOUT_BSND = 0
LAYOUT_BNBD = 1
DTYPE_F32 = 0
DTYPE_BF16 = 1
INDEX_I32 = 0
INDEX_I64 = 1

PA_OK = 0
_STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_NULLPTR", 2: "PA_ERR_INVALID", 3: "PA_ERR_WORKSPACE",
                 4: "PA_ERR_CUDA", 5: "PA_ERR_UNSUPPORTED"}

LIB_PATH = _build.LIB_PATH
_lock = threading.Lock()
_lib = None


class PaError(RuntimeError):
    """A non-PA_OK status from the library."""

    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__("%s: %s (%s)" % (where, _STATUS_NAMES.get(status, status), detail))


class pa_decode_config(ctypes.Structure):
    _fields_ = [("s2_tile", ctypes.c_int), ("num_ctas", ctypes.c_int),
                ("overlap_prologue", ctypes.c_int), ("merge_wait_ns", ctypes.c_int),
                ("wait_limit_ns", ctypes.c_int), ("reserved", ctypes.c_int * 3)]


def build(force: bool = False) -> str:
    """Compile libpa_fp8.so (nvcc, sm_103a) if it is stale."""
    return _build.build(force=force)


def lib():
    """The loaded ctypes library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libpa_fp8.so is not built (%s); run "
                               "fp8_paged_kv_block_gb300.build() first" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                ctypes.c_size_t)
        L.pa_status_string.argtypes = [i32]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_last_error.argtypes = []
        L.pa_last_error.restype = ctypes.c_char_p
        L.pa_fp8_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, P,
                                                   ctypes.POINTER(sz)]
        L.pa_fp8_decode_workspace_size.restype = i32
        L.pa_fp8_decode_auto_s2_tile.argtypes = [i32, i32, i32, i64]
        L.pa_fp8_decode_auto_s2_tile.restype = i32
        L.pa_fp8_decode.argtypes = [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64,
                                    i32, i32, f32, P, P, sz, P]
        L.pa_fp8_decode.restype = i32
        L.pa_fp8_cache_scatter.argtypes = [P, P, P, P, P, i32, P, i64, i64, P, i64, i32, i32, i32,
                                           i64, i32, i32, P]
        L.pa_fp8_cache_scatter.restype = i32
        L.pa_fp8_cache_quant_scatter.argtypes = [P, P, i32, P, P, P, i32, P, P, P, i32, i64, i32,
                                                 i32, i64, i32, i32, i32, P]
        L.pa_fp8_cache_quant_scatter.restype = i32
        L.pa_fp8_kv_compress_epilog.argtypes = [P, i64, i32, i64, i32, P, i64, i32, P, i32, i32,
                                                i32, i32, P]
        L.pa_fp8_kv_compress_epilog.restype = i32
        L.pa_fp8_quantize_rows.argtypes = [P, i32, i64, i32, P, P, P]
        L.pa_fp8_quantize_rows.restype = i32
        L.pa_fp8_value_channel_scale.argtypes = [P, i32, P, i32, i64, i32, i32, P, P]
        L.pa_fp8_value_channel_scale.restype = i32
        L.pa_mla_sparse_decode.argtypes = [P, P, P, i64, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                           i64, i32, f32, i32, P, P]
        L.pa_mla_sparse_decode.restype = i32
        L.pa_mla_sparse_decode_kvc.argtypes = [P, P, P, i64, i64, i32, P, P, P, P, i32, i32, i32,
                                               i32, i32, i32, i64, i32, f32, i32, P, P]
        L.pa_mla_sparse_decode_kvc.restype = i32
        _lib = L
        return L


def _check(status: int, where: str):
    if status != PA_OK:
        detail = lib().pa_last_error().decode(errors="replace")
        raise PaError(status, where, detail)


def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, name, dtype=None, contiguous=True):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError("%s has dtype %s, expected %s" % (name, t.dtype, dtype))
    if contiguous and not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _fp8_types():
    torch = _torch()
    return (torch.uint8, torch.float8_e4m3fn, torch.float8_e5m2)


def _in_dtype(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError("expected float32 or bfloat16, got %s" % t.dtype)


# --------------------------------------------------------------------------
# Decode attention
# --------------------------------------------------------------------------

_configs = {}


def _config(s2_tile: int, num_ctas: int, overlap_prologue=0, merge_wait_ns=0, wait_limit_ns=0):
    key = (s2_tile, num_ctas, int(overlap_prologue), int(merge_wait_ns), int(wait_limit_ns))
    c = _configs.get(key)
    if c is None:
        c = pa_decode_config()
        c.s2_tile = s2_tile
        c.num_ctas = num_ctas
        c.overlap_prologue = int(overlap_prologue)
        c.merge_wait_ns = int(merge_wait_ns)
        c.wait_limit_ns = int(wait_limit_ns)
        _configs[key] = c
    return c


def auto_s2_tile(S1: int, NQ: int, NKV: int, s2: int) -> int:
    """The s2_tile that s2_tile=0 selects for sequences of capacity s2 (the
    block table's width x block_size): 1024 from 8192 tokens on where at most
    16 query rows share a kv head, else 512 (pa_fp8_decode_auto_s2_tile)."""
    t = lib().pa_fp8_decode_auto_s2_tile(S1, NQ, NKV, s2)
    if t == 0:
        raise ValueError("auto_s2_tile: invalid shape S1=%d NQ=%d NKV=%d s2=%d" % (S1, NQ, NKV, s2))
    return t


def decode_workspace_size(B: int, S1: int, NQ: int, NKV: int, D: int = 128, *,
                          s2_tile: int = 0, num_ctas: int = 0) -> int:
    n = ctypes.c_size_t(0)
    cfg = _config(s2_tile, num_ctas)
    _check(lib().pa_fp8_decode_workspace_size(B, S1, NQ, NKV, D, ctypes.byref(cfg),
                                              ctypes.byref(n)), "pa_fp8_decode_workspace_size")
    return n.value


class DecodeWorkspace:
    """Zero-initialised device scratch for pa_fp8_decode (reusable: every call
    leaves its counters at zero)."""

    def __init__(self, B, S1, NQ, NKV, D=128, *, s2_tile=0, num_ctas=0, device=None):
        torch = _torch()
        self.nbytes = decode_workspace_size(B, S1, NQ, NKV, D, s2_tile=s2_tile, num_ctas=num_ctas)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device or "cuda")

    def error_flags(self) -> int:
        """Non-zero if a kernel wait gave up (bitmask of the wait sites)."""
        return int(self.buf[:4].view(_torch().int32).item())

    def clear_error_flags(self) -> None:
        """Zero the error word (on the current stream); the kernel only ever
        sets bits in it."""
        self.buf[:4].zero_()


def decode(q, q_scale, k_cache, k_scale, v_cache, v_scale, block_table, kv_act_seqs, out, *,
           S1: int = 1, layout: int = LAYOUT_BSND, s2_tile: int = 0, softmax_scale=None,
           workspace: DecodeWorkspace | None = None, num_ctas: int = 0, stream=None,
           overlap_prologue: int = 0, merge_wait_ns: int = 0, wait_limit_ns: int = 0):
    """Paged FP8 decode attention (in place into ``out``).

    q [B*S1, NQ, D] E4M3 (uint8 or float8_e4m3fn), q_scale float32 [B*S1, NQ],
    k_cache/v_cache E4M3 in ``layout`` ([NB, BS, NKV, D] for BSND,
    [NB, NKV, BS, D] for BNBD), k_scale float32 (cache shape without D),
    v_scale float32 [B, NKV, D], block_table int32 [B, max_blocks],
    kv_act_seqs int32 [B], out bfloat16 [B*S1, NQ, D].
    s2_tile: 0 (automatic, see auto_s2_tile), 128, 256, 512 or 1024.
    overlap_prologue: 1 (or True) lets the kernel's prologue overlap the
    preceding kernel in the stream (that kernel must not write kv_act_seqs,
    block_table, q, q_scale or v_scale); 2 also lets it load the cache blocks
    below each sequence's S1 newest positions early (that kernel must not
    write the cache there); see pa_decode_config.overlap_prologue.
    merge_wait_ns, wait_limit_ns: test and diagnostic knobs, see
    pa_decode_config.
    """
    args, keep = _decode_args(q, q_scale, k_cache, k_scale, v_cache, v_scale, block_table,
                              kv_act_seqs, out, S1, layout, s2_tile, softmax_scale, workspace,
                              num_ctas, overlap_prologue, merge_wait_ns, wait_limit_ns)
    _check(lib().pa_fp8_decode(*args, _stream(stream)), "pa_fp8_decode")
    del keep   # (a workspace made here lives until the launch is enqueued)
    return out


def _decode_args(q, q_scale, k_cache, k_scale, v_cache, v_scale, block_table, kv_act_seqs, out,
                 S1, layout, s2_tile, softmax_scale, workspace, num_ctas, overlap_prologue,
                 merge_wait_ns, wait_limit_ns):
    """pa_fp8_decode's arguments but the stream, validated, and the objects
    they point into."""
    torch = _torch()
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, _fp8_types())
    _need(q_scale, "q_scale", torch.float32)
    _need(k_scale, "k_scale", torch.float32)
    _need(v_scale, "v_scale", torch.float32)
    _need(block_table, "block_table", torch.int32)
    _need(kv_act_seqs, "kv_act_seqs", torch.int32)
    _need(out, "out", torch.bfloat16)
    B = kv_act_seqs.shape[0]
    BS1, NQ, D = q.shape
    if layout == LAYOUT_BSND:
        NB, BS, NKV, _ = k_cache.shape
    else:
        NB, NKV, BS, _ = k_cache.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if workspace is None:
        workspace = DecodeWorkspace(B, S1, NQ, NKV, D, s2_tile=s2_tile, num_ctas=num_ctas,
                                    device=q.device)
    cfg = _config(s2_tile, num_ctas, overlap_prologue, merge_wait_ns, wait_limit_ns)
    args = (_ptr(q), _ptr(q_scale), _ptr(k_cache), _ptr(k_scale), _ptr(v_cache), _ptr(v_scale),
            _ptr(block_table), _ptr(kv_act_seqs), _ptr(out), B, S1, NQ, NKV, D, BS, NB,
            block_table.shape[1], layout, float(softmax_scale), ctypes.byref(cfg),
            _ptr(workspace.buf), workspace.nbytes)
    keep = (q, q_scale, k_cache, k_scale, v_cache, v_scale, block_table, kv_act_seqs, out,
            workspace, cfg)
    return args, keep


class _Prepared:
    """A library call whose arguments were validated and marshalled once, for
    a loop that makes the same call every step (the buffers' contents may
    change between calls, not their addresses, shapes or dtypes). Runs on the
    stream given when it was made (default: the current stream then), or on
    the stream passed to the call."""

    def __init__(self, fn, where, args, keep, stream):
        self._fn, self._where, self._args, self._keep = fn, where, args, keep
        self._stream = _stream(stream)

    def __call__(self, stream=None):
        st = self._fn(*self._args, self._stream if stream is None else _stream(stream))
        if st != PA_OK:
            _check(st, self._where)


def prepare_decode(q, q_scale, k_cache, k_scale, v_cache, v_scale, block_table, kv_act_seqs, out,
                   *, S1: int = 1, layout: int = LAYOUT_BSND, s2_tile: int = 0,
                   softmax_scale=None, workspace: DecodeWorkspace | None = None,
                   num_ctas: int = 0, overlap_prologue: int = 0, stream=None):
    """decode() prepared once: returns a callable that launches the same
    decode on the same buffers (arguments as for decode())."""
    args, keep = _decode_args(q, q_scale, k_cache, k_scale, v_cache, v_scale, block_table,
                              kv_act_seqs, out, S1, layout, s2_tile, softmax_scale, workspace,
                              num_ctas, overlap_prologue, 0, 0)
    return _Prepared(lib().pa_fp8_decode, "pa_fp8_decode", args, keep, stream)


# --------------------------------------------------------------------------
# Cache append
# --------------------------------------------------------------------------

def _cache_dims(key_cache, layout):
    if layout == LAYOUT_BNBD:
        NB, H, BS, _ = key_cache.shape
    else:
        NB, BS, H, _ = key_cache.shape
    return NB, H, BS


def _slot_type(slot_mapping):
    torch = _torch()
    if slot_mapping.dtype == torch.int32:
        return INDEX_I32
    if slot_mapping.dtype == torch.int64:
        return INDEX_I64
    raise TypeError("slot_mapping must be int32 or int64")


def cache_scatter(key, value, key_cache, value_cache, slot_mapping, key_scale, key_scale_cache,
                  *, layout: int = LAYOUT_BNBD, stream=None):
    """FP8 K/V + key_scale append by slot_mapping (in place). key_scale may
    have a non-contiguous tail (any 2-D strides)."""
    torch = _torch()
    for t, n in ((key, "key"), (value, "value"), (key_cache, "key_cache"),
                 (value_cache, "value_cache")):
        _need(t, n, _fp8_types())
    _need(slot_mapping, "slot_mapping", (torch.int32, torch.int64))
    _need(key_scale, "key_scale", torch.float32, contiguous=False)
    _need(key_scale_cache, "key_scale_cache", torch.float32)
    T, H, Dk = key.shape
    Dv = value.shape[2]
    NB, _, BS = _cache_dims(key_cache, layout)
    st = lib().pa_fp8_cache_scatter(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                                    _ptr(slot_mapping), _slot_type(slot_mapping), _ptr(key_scale),
                                    key_scale.stride(0), key_scale.stride(1),
                                    _ptr(key_scale_cache), T, H, Dk, Dv, NB, BS, layout,
                                    _stream(stream))
    _check(st, "pa_fp8_cache_scatter")


def cache_quant_scatter(key, value, key_cache, value_cache, slot_mapping, key_scale_cache,
                        v_scale, token_batch, *, layout: int = LAYOUT_BNBD,
                        overlap_prologue: bool = False, stream=None):
    """BF16/FP32 K/V quantised to E4M3 on append (in place): key per
    (token, head) with scale amax/448 stored to key_scale_cache, value against
    v_scale[token_batch[i]]. overlap_prologue=True launches it with
    programmatic stream serialisation: the inputs are read while the preceding
    kernel may still run (it must not write them), the caches are written after
    it has completed."""
    args, keep = _quant_scatter_args(key, value, key_cache, value_cache, slot_mapping,
                                     key_scale_cache, v_scale, token_batch, layout,
                                     overlap_prologue)
    _check(lib().pa_fp8_cache_quant_scatter(*args, _stream(stream)), "pa_fp8_cache_quant_scatter")
    del keep


def _quant_scatter_args(key, value, key_cache, value_cache, slot_mapping, key_scale_cache,
                        v_scale, token_batch, layout, overlap_prologue):
    torch = _torch()
    _need(key, "key", (torch.float32, torch.bfloat16))
    _need(value, "value", (key.dtype,))
    for t, n in ((key_cache, "key_cache"), (value_cache, "value_cache")):
        _need(t, n, _fp8_types())
    _need(slot_mapping, "slot_mapping", (torch.int32, torch.int64))
    _need(key_scale_cache, "key_scale_cache", torch.float32)
    _need(v_scale, "v_scale", torch.float32)
    _need(token_batch, "token_batch", torch.int32)
    T, H, D = key.shape
    NB, _, BS = _cache_dims(key_cache, layout)
    args = (_ptr(key), _ptr(value), _in_dtype(key), _ptr(key_cache), _ptr(value_cache),
            _ptr(slot_mapping), _slot_type(slot_mapping), _ptr(key_scale_cache), _ptr(v_scale),
            _ptr(token_batch), v_scale.shape[0], T, H, D, NB, BS, layout,
            int(bool(overlap_prologue)))
    keep = (key, value, key_cache, value_cache, slot_mapping, key_scale_cache, v_scale,
            token_batch)
    return args, keep


def prepare_cache_quant_scatter(key, value, key_cache, value_cache, slot_mapping,
                                key_scale_cache, v_scale, token_batch, *,
                                layout: int = LAYOUT_BNBD, overlap_prologue: bool = False,
                                stream=None):
    """cache_quant_scatter() prepared once: returns a callable that launches the
    same append on the same buffers."""
    args, keep = _quant_scatter_args(key, value, key_cache, value_cache, slot_mapping,
                                     key_scale_cache, v_scale, token_batch, layout,
                                     overlap_prologue)
    return _Prepared(lib().pa_fp8_cache_quant_scatter, "pa_fp8_cache_quant_scatter", args, keep,
                     stream)


def kv_compress_epilog(cache, x, slot_mapping, *, quant_group_size: int = 64, quant_mode: int = 1,
                       round_scale: bool = True, stream=None):
    """KV compress epilog (modes 0 and 1), in place: cache uint8
    [block_num, block_size, 1, head_dim] (blocks may be strided), x bfloat16
    [bs, d], slot_mapping int32/int64 [bs]. Each row is written as the rope
    part (last 64 values) in BF16, the rest in E4M3 groups of 64, then the
    group scales (BF16 in mode 0, E8M0 in mode 1)."""
    torch = _torch()
    _need(cache, "cache", (torch.uint8,), contiguous=False)
    _need(x, "x", (torch.bfloat16,))
    _need(slot_mapping, "slot_mapping", (torch.int32, torch.int64))
    if cache.dim() != 4 or cache.shape[2] != 1:
        raise ValueError("cache must be [block_num, block_size, 1, head_dim]")
    NB, BS, _, HD = cache.shape
    if cache.stride(3) != 1 or cache.stride(1) != HD:
        raise ValueError("cache rows must be contiguous within a block")
    bs, d = x.shape
    st = lib().pa_fp8_kv_compress_epilog(_ptr(cache), NB, BS, cache.stride(0), HD, _ptr(x), bs, d,
                                         _ptr(slot_mapping), _slot_type(slot_mapping),
                                         quant_group_size, quant_mode, int(bool(round_scale)),
                                         _stream(stream))
    _check(st, "pa_fp8_kv_compress_epilog")


def quantize_rows(x, codes, scale, *, stream=None):
    """Per-row E4M3 quantiser: x [..., D] float32/bfloat16 -> codes [..., D],
    dequant scale [...] = amax / 448."""
    torch = _torch()
    _need(x, "x", (torch.float32, torch.bfloat16))
    _need(codes, "codes", _fp8_types())
    _need(scale, "scale", torch.float32)
    D = x.shape[-1]
    rows = x.numel() // D
    st = lib().pa_fp8_quantize_rows(_ptr(x), _in_dtype(x), rows, D, _ptr(codes), _ptr(scale),
                                    _stream(stream))
    _check(st, "pa_fp8_quantize_rows")


def value_channel_scale(v, cu_seqlens, v_scale, *, stream=None):
    """v [Ttot, H, D] float32/bfloat16, cu_seqlens int64 [B+1] (device) ->
    v_scale [B, H, D] = per-channel max |v| over each sequence / 448."""
    torch = _torch()
    _need(v, "v", (torch.float32, torch.bfloat16))
    _need(cu_seqlens, "cu_seqlens", torch.int64)
    _need(v_scale, "v_scale", torch.float32)
    T, H, D = v.shape
    B = cu_seqlens.shape[0] - 1
    st = lib().pa_fp8_value_channel_scale(_ptr(v), _in_dtype(v), _ptr(cu_seqlens), B, T, H, D,
                                          _ptr(v_scale), _stream(stream))
    _check(st, "pa_fp8_value_channel_scale")


__all__ = [
    "LAYOUT_BSND", "LAYOUT_BNBD", "PaError", "build", "lib", "decode", "decode_workspace_size",
    "auto_s2_tile", "prepare_decode", "prepare_cache_quant_scatter",
    "DecodeWorkspace", "cache_scatter", "cache_quant_scatter", "quantize_rows",
    "value_channel_scale",
]


MLA_ROW_USED = 656


class MlaStatus:
    """A device int the MLA decode kernel ORs a bit into when one of its
    bounded waits gives up (zeroed at creation)."""

    def __init__(self, device=None):
        torch = _torch()
        self.buf = torch.zeros(1, dtype=torch.int32,
                               device=device if device is not None else torch.cuda.current_device())

    def value(self) -> int:
        return int(self.buf.item())


def _mla_args(q_nope, q_rope, topk_indices, block_table, kv_act_seqs, out, S1, softmax_scale):
    torch = _torch()
    _need(q_nope, "q_nope", torch.bfloat16)
    _need(q_rope, "q_rope", torch.bfloat16)
    _need(topk_indices, "topk_indices", torch.int32)
    _need(block_table, "block_table", torch.int32)
    _need(kv_act_seqs, "kv_act_seqs", torch.int32)
    _need(out, "out", torch.bfloat16)
    T, NQ, dn = q_nope.shape
    if dn != 512 or tuple(q_rope.shape) != (T, NQ, 64) or tuple(out.shape) != (T, NQ, 512):
        raise ValueError("q_nope/out must be [T, NQ, 512] and q_rope [T, NQ, 64]")
    B = kv_act_seqs.shape[0]
    if T != B * S1 or topk_indices.shape[0] != T:
        raise ValueError("B*S1 must equal the query token count of q_nope and topk_indices")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(576.0)
    return B, NQ, float(softmax_scale)


def mla_sparse_decode(q_nope, q_rope, nope_cache, topk_indices, block_table, kv_act_seqs, out, *,
                      S1: int, status: MlaStatus, block_size: int = 128, softmax_scale=None,
                      s2_tile: int = 128, stream=None):
    """MLA sparse attention with FP8 anti-quantisation (decode), in place.

    q_nope bfloat16 [B*S1, NQ, 512], q_rope bfloat16 [B*S1, NQ, 64];
    nope_cache uint8 [num_blocks*block_size, row_bytes] packed rows (E4M3 kn |
    BF16 kr | 4 FP32 scales, row_bytes >= 656); topk_indices int32
    [B*S1, topk]; block_table int32 [B, max_blocks]; kv_act_seqs int32 [B];
    out bfloat16 [B*S1, NQ, 512]."""
    torch = _torch()
    B, NQ, sc = _mla_args(q_nope, q_rope, topk_indices, block_table, kv_act_seqs, out, S1,
                          softmax_scale)
    _need(nope_cache, "nope_cache", torch.uint8)
    rows, row_bytes = nope_cache.shape
    if rows % block_size:
        raise ValueError("nope_cache rows must be a multiple of block_size")
    st = lib().pa_mla_sparse_decode(_ptr(q_nope), _ptr(q_rope), _ptr(nope_cache), row_bytes,
                                    _ptr(topk_indices), _ptr(block_table), _ptr(kv_act_seqs),
                                    _ptr(out), B, S1, NQ, 1, topk_indices.shape[1], block_size,
                                    rows // block_size, block_table.shape[1], sc,
                                    s2_tile, _ptr(status.buf), _stream(stream))
    _check(st, "pa_mla_sparse_decode")


def mla_sparse_decode_kvc(q_nope, q_rope, kv_cache, topk_indices, block_table, kv_act_seqs, out,
                          *, quant_mode: int, S1: int, status: MlaStatus, block_size: int = 128,
                          softmax_scale=None, s2_tile: int = 128, stream=None):
    """The MLA sparse decode of ``mla_sparse_decode`` over cache rows written by
    ``kv_compress_epilog`` with d = 576 and the given quant_mode (0: BF16 group
    scales, 1: E8M0 group scales). kv_cache is the epilog's cache, uint8
    [block_num, block_size, 1, head_dim] (blocks may be strided, rows within a
    block contiguous), or [block_num * block_size, head_dim]; head_dim >= 656
    and a multiple of 16."""
    torch = _torch()
    B, NQ, sc = _mla_args(q_nope, q_rope, topk_indices, block_table, kv_act_seqs, out, S1,
                          softmax_scale)
    _need(kv_cache, "kv_cache", torch.uint8, contiguous=False)
    if kv_cache.dim() == 4:
        nb, bs, one, row_bytes = kv_cache.shape
        if one != 1 or bs != block_size or kv_cache.stride(3) != 1 or kv_cache.stride(1) != row_bytes:
            raise ValueError("kv_cache must be [block_num, block_size, 1, head_dim] with "
                             "contiguous rows inside a block")
        stride = kv_cache.stride(0)
    elif kv_cache.dim() == 2 and kv_cache.is_contiguous():
        rows, row_bytes = kv_cache.shape
        if rows % block_size:
            raise ValueError("kv_cache rows must be a multiple of block_size")
        nb, stride = rows // block_size, block_size * row_bytes
    else:
        raise ValueError("kv_cache must be [block_num, block_size, 1, head_dim] or a contiguous "
                         "[block_num * block_size, head_dim]")
    st = lib().pa_mla_sparse_decode_kvc(_ptr(q_nope), _ptr(q_rope), _ptr(kv_cache), row_bytes,
                                        stride, int(quant_mode), _ptr(topk_indices),
                                        _ptr(block_table), _ptr(kv_act_seqs), _ptr(out), B, S1,
                                        NQ, 1, topk_indices.shape[1], block_size, nb,
                                        block_table.shape[1], sc, s2_tile, _ptr(status.buf),
                                        _stream(stream))
    _check(st, "pa_mla_sparse_decode_kvc")
