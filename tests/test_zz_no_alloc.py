"""pa_fp8_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (a plugin handed only tensor pointers and a stream, or
a serving loop with a pre-planned memory budget that must not call
cudaMalloc mid-step). Its scratch is a fixed array inside the library.

Called through the C ABI (ctypes): twice in a row against pa_fp8_decode on a
caller-allocated workspace and against the CPU oracle, within the parity
tolerance of the other GPU tests; after an append with overlap_prologue 2;
two shapes back to back on the shared array; and its error word read back
with pa_fp8_decode_noalloc_error. This file is collected last on purpose."""
import ctypes
import dataclasses

import numpy as np
import pytest

import oracle
import workloads
from tests import _helpers as H

pytestmark = pytest.mark.gpu


def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _fns():
    import fp8_paged_kv_block_gb300 as pa
    L = pa.lib()
    fn = L.pa_fp8_decode_noalloc
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    fn.argtypes = [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, i32, i32, f32, P,
                   P]
    fn.restype = i32
    err = L.pa_fp8_decode_noalloc_error
    err.argtypes = [ctypes.POINTER(ctypes.c_int32), i32, P]
    err.restype = i32
    return fn, err


def _call_noalloc(fn, case, dev, out, num_ctas=0, **cfg_fields):
    import torch
    import fp8_paged_kv_block_gb300 as pa
    c = dev["cache"]
    cfg = pa.pa_decode_config()
    cfg.s2_tile = case.s2_tile
    cfg.num_ctas = num_ctas
    for k, v in cfg_fields.items():
        setattr(cfg, k, v)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    NB = c.k_cache.shape[0]
    st = fn(p(dev["q8"]), p(dev["qs"]), p(c.k_cache), p(c.k_scale), p(c.v_cache), p(c.v_scale),
            p(dev["block_table"]), p(dev["act"]), p(out), case.B, case.S1, case.NQ, case.NKV,
            case.D, case.BS, NB, case.max_blocks, case.layout, case.softmax_scale,
            ctypes.byref(cfg), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, pa.lib().pa_last_error()


def _read_error(err, clear=False):
    import torch
    flags = ctypes.c_int32(-1)
    st = err(ctypes.byref(flags), 1 if clear else 0,
             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    return flags.value


def _split_case():
    return workloads.custom("split", 5, 1, 24, 2, [1, 127, 128, 513, 1300])


def _empty_out(case):
    import torch
    return torch.full((case.B * case.S1, case.NQ, case.D), float("nan"), dtype=torch.bfloat16,
                      device="cuda")


@pytest.mark.parametrize("mk,num_ctas", [(workloads.glm, 0), (_split_case, 7)])
def test_noalloc_matches_workspace_decode_twice(mk, num_ctas):
    torch = _cuda()
    import fp8_paged_kv_block_gb300 as pa
    fn, err = _fns()
    case = mk()
    dev = H.device_inputs(case)
    ws = pa.DecodeWorkspace(case.B, case.S1, case.NQ, case.NKV, s2_tile=case.s2_tile,
                            num_ctas=num_ctas)
    ref = H.to_u16(H.gpu_decode(case, dev, num_ctas=num_ctas, workspace=ws))
    assert ws.error_flags() == 0
    for _ in range(2):
        out = _empty_out(case)
        _call_noalloc(fn, case, dev, out, num_ctas)
        torch.cuda.synchronize()
        H.compare_bf16(H.to_u16(out), ref)
    assert _read_error(err) == 0


def test_noalloc_matches_oracle_twice():
    """Directly against the CPU oracle (split sequences merged across CTAs)."""
    torch = _cuda()
    fn, err = _fns()
    case = _split_case()
    inp = H.oracle_inputs(case)
    dev = H.device_inputs(case)
    ref = H.oracle_decode(case, inp)
    for _ in range(2):
        out = _empty_out(case)
        _call_noalloc(fn, case, dev, out, num_ctas=7)
        torch.cuda.synchronize()
        H.compare_bf16(H.to_u16(out), ref)
    assert _read_error(err) == 0


def test_noalloc_two_shapes_back_to_back():
    """The split case then the GLM-4.5 case on the shared array, on one
    stream without synchronising in between: each call finds the counters it
    uses at zero (the previous shape left them so)."""
    torch = _cuda()
    fn, err = _fns()
    small, big = _split_case(), workloads.glm()
    dev_s, dev_b = H.device_inputs(small), H.device_inputs(big)
    ref_s = H.oracle_decode(small, H.oracle_inputs(small))
    rows = np.random.default_rng(5).choice(big.B * big.S1 * big.NQ, 96, replace=False)
    inp_b = H.oracle_inputs(big, batches=np.unique(rows // (big.S1 * big.NQ)))
    ref_b = H.oracle_decode(big, inp_b, rows=rows)
    outs = []
    for case, dev, n in ((small, dev_s, 7), (big, dev_b, 0), (small, dev_s, 3)):
        out = _empty_out(case)
        _call_noalloc(fn, case, dev, out, num_ctas=n)
        outs.append(out)
    torch.cuda.synchronize()
    H.compare_bf16(H.to_u16(outs[0]), ref_s)
    H.compare_bf16(H.to_u16(outs[1]), ref_b, rows=rows)
    H.compare_bf16(H.to_u16(outs[2]), ref_s)
    assert _read_error(err) == 0


def test_noalloc_after_append_with_overlap_prologue_2():
    """append (programmatic serialisation) -> allocation-free decode with
    overlap_prologue 2: the decode may read older cache blocks while the
    append runs and sees the appended token; output against the oracle."""
    torch = _cuda()
    import fp8_paged_kv_block_gb300 as pa
    fn, err = _fns()
    case = workloads.custom("chain", 6, 1, 24, 2, [1, 127, 700, 1300, 2049, 3000], max_blocks=25)
    inp = H.oracle_inputs(case)
    dev = H.device_inputs(case)
    knew, vnew, slot, act_after = workloads.step_tokens(case)
    oracle.cache_quant_scatter(knew.float().numpy(), vnew.float().numpy(), inp["kc"], inp["vc"],
                               slot.astype(np.int64), inp["ksc"], inp["vs"],
                               np.arange(case.B, dtype=np.int32), layout=case.layout)
    case1 = dataclasses.replace(case, act=act_after)
    ref = H.oracle_decode(case1, inp)
    c = dev["cache"]
    dev["act"] = torch.from_numpy(act_after).cuda()
    out = _empty_out(case)
    torch.cuda.synchronize()
    pa.cache_quant_scatter(knew.cuda(), vnew.cuda(), c.k_cache, c.v_cache, torch.from_numpy(slot).cuda(),
                           c.k_scale, c.v_scale, torch.arange(case.B, dtype=torch.int32, device="cuda"),
                           layout=case.layout, overlap_prologue=True)
    _call_noalloc(fn, case1, dev, out, overlap_prologue=2)
    torch.cuda.synchronize()
    H.compare_bf16(H.to_u16(out), ref)
    assert _read_error(err) == 0


def test_noalloc_error_word_reports_and_clears():
    """With every wait's limit at 1 ns the kernel's waits run out on a valid
    input: the call returns, the error word (read through
    pa_fp8_decode_noalloc_error) is non-zero and keeps its bits until
    cleared; a default call afterwards matches the oracle."""
    torch = _cuda()
    fn, err = _fns()
    case = _split_case()
    inp = H.oracle_inputs(case)
    dev = H.device_inputs(case)
    out = _empty_out(case)
    _call_noalloc(fn, case, dev, out, num_ctas=7, wait_limit_ns=1)
    first = _read_error(err)
    assert first != 0
    assert _read_error(err, clear=True) == first      # still set; cleared after the copy
    assert _read_error(err) == 0
    out = _empty_out(case)
    _call_noalloc(fn, case, dev, out, num_ctas=7)
    torch.cuda.synchronize()
    H.compare_bf16(H.to_u16(out), H.oracle_decode(case, inp))
    assert _read_error(err) == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    torch = _cuda()
    import fp8_paged_kv_block_gb300 as pa
    fn, _ = _fns()
    need = pa.decode_workspace_size(1024, 1, 96, 8)
    assert need > (16 << 20)
    # small real allocations: rejected on the host before any use
    bufs = [torch.zeros(1 << 16, dtype=torch.uint8, device="cuda") for _ in range(9)]
    ptrs = [ctypes.c_void_p(b.data_ptr()) for b in bufs]
    st = fn(*ptrs, 1024, 1, 96, 8, 128, 128, 100, 4, 0, 0.088, None, None)
    assert st == 3
    assert b"scratch" in pa.lib().pa_last_error()
