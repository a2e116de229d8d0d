"""pa_fp8_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (a plugin handed only tensor pointers and a stream, or
a serving loop with a pre-planned memory budget that must not call
cudaMalloc mid-step). Its scratch is a fixed array inside the library.

Called through the C ABI (ctypes) twice in a row and compared with
pa_fp8_decode on a caller-allocated workspace, within the parity tolerance of
the other GPU tests. This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

import workloads
from tests import _helpers as H

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    import fp8_paged_kv_block_gb300 as pa
    L = pa.lib()
    fn = L.pa_fp8_decode_noalloc
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    fn.argtypes = [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, i32, i32, f32, P,
                   P]
    fn.restype = i32
    return fn


def _call_noalloc(fn, case, dev, out, num_ctas=0):
    import torch
    import fp8_paged_kv_block_gb300 as pa
    c = dev["cache"]
    cfg = pa.pa_decode_config()
    cfg.s2_tile = case.s2_tile
    cfg.num_ctas = num_ctas
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    NB = c.k_cache.shape[0]
    st = fn(p(dev["q8"]), p(dev["qs"]), p(c.k_cache), p(c.k_scale), p(c.v_cache), p(c.v_scale),
            p(dev["block_table"]), p(dev["act"]), p(out), case.B, case.S1, case.NQ, case.NKV,
            case.D, case.BS, NB, case.max_blocks, case.layout, case.softmax_scale,
            ctypes.byref(cfg), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, pa.lib().pa_last_error()


@pytest.mark.parametrize("mk,num_ctas", [(workloads.glm, 0),
                                         (lambda: workloads.custom(
                                             "split", 5, 1, 24, 2, [1, 127, 128, 513, 1300]), 7)])
def test_noalloc_matches_workspace_decode_twice(mk, num_ctas):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_paged_kv_block_gb300 as pa
    fn = _noalloc_fn()
    case = mk()
    dev = H.device_inputs(case)
    ws = pa.DecodeWorkspace(case.B, case.S1, case.NQ, case.NKV, s2_tile=case.s2_tile,
                            num_ctas=num_ctas)
    ref = H.to_u16(H.gpu_decode(case, dev, num_ctas=num_ctas, workspace=ws))
    assert ws.error_flags() == 0
    for _ in range(2):
        out = torch.full((case.B * case.S1, case.NQ, case.D), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        _call_noalloc(fn, case, dev, out, num_ctas)
        torch.cuda.synchronize()
        H.compare_bf16(H.to_u16(out), ref)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_paged_kv_block_gb300 as pa
    fn = _noalloc_fn()
    need = pa.decode_workspace_size(1024, 1, 96, 8)
    assert need > (16 << 20)
    fake = ctypes.c_void_p(256)   # rejected on the host before any use
    st = fn(fake, fake, fake, fake, fake, fake, fake, fake, fake, 1024, 1, 96, 8, 128, 128, 100,
            4, 0, 0.088, None, None)
    assert st == 3
    assert b"scratch" in pa.lib().pa_last_error()
