"""The byte and flop counts that every GB/s, TFLOP/s and roofline fraction of the
benchmark divides by, recounted independently (no GPU).

Decode: the bytes a decode must move at minimum are the valid tokens' K and V
codes and key scales, the query codes and scales, the value channel scales, the
BF16 output, the block table and the lengths; here they are summed from the
sizes of the arrays the oracle's inputs actually hold (cache bytes only at the
slots of valid tokens). MLA: the valid selected (token, key) pairs are counted
by a plain loop over the top-k lists with the visible-count and masking rules,
and bytes / flops follow from them.
"""
import dataclasses

import numpy as np
import pytest

import bench
import workloads
from tests import _helpers as H


@pytest.mark.parametrize("mk", [workloads.tiny,
                                lambda: workloads.custom("acct", 3, 2, 24, 2, [1, 0, 700]),
                                lambda: workloads.tiny(layout=workloads.LAYOUT_BNBD)])
def test_decode_algorithmic_bytes_from_the_inputs(mk):
    case = mk()
    inp = H.oracle_inputs(case)
    slots = case.slots                                   # one per valid context token
    NB, BS = case.num_blocks, case.BS
    occupied = np.zeros(NB * BS, dtype=bool)
    occupied[slots] = True
    assert occupied.sum() == slots.size                 # every valid token has its own slot
    per_slot = (inp["kc"].nbytes + inp["vc"].nbytes + inp["ksc"].nbytes) // (NB * BS)
    kv = int(occupied.sum()) * per_slot                 # K, V codes and key scale at used slots
    out = inp["q8"].size * 2                            # BF16 output, one per query element
    want = (kv + inp["q8"].nbytes + inp["qs"].nbytes + inp["vs"].nbytes + out
            + case.block_table.nbytes + case.act.astype(np.int32).nbytes)
    assert case.algorithmic_bytes() == want


def test_append_step_bytes():
    """The append's share of a step: BF16 K and V rows in, E4M3 K and V codes
    and one FP32 key scale out per (token, head), and the int32 slot and batch
    id of each token."""
    case = workloads.tiny()
    knew, vnew, slot, act_after = workloads.step_tokens(case)
    dec, app = bench.step_bytes(case, act_after)
    codes_out = 2 * knew.numel()                         # one byte per K and V element
    scales_out = 4 * case.B * case.NKV
    want_app = (knew.numel() * knew.element_size() + vnew.numel() * vnew.element_size()
                + codes_out + scales_out + slot.astype(np.int32).nbytes + 4 * case.B)
    assert app == want_app
    assert dec == dataclasses.replace(case, act=act_after).algorithmic_bytes()
    assert (act_after - case.act).sum() == (slot >= 0).sum()


def _valid_pairs_by_loop(case, variant=0):
    tk = case.topk_indices(variant)
    n = 0
    for t in range(case.T):
        b, s = divmod(t, case.S1)
        visible = min(max(int(case.act[b]) - case.S1 + 1 + s, 0), case.topk)
        for j in range(visible):
            idx = int(tk[t, j])
            if 0 <= idx < int(case.act[b]):
                n += 1
    return n


@pytest.mark.parametrize("S1,act,frac", [(2, (300, 41, 1), 0.1), (1, (2048, 5), 0.0),
                                         (3, (2, 700), 0.05)])
def test_mla_keys_flops_and_bytes(S1, act, frac):
    case = workloads.mla("acct", len(act), S1, list(act), NQ=64, topk=256,
                         seed=workloads.BASE_SEED + 900, frac_invalid=frac)
    keys = _valid_pairs_by_loop(case)
    assert case.keys_read() == keys
    assert case.flops() == keys * case.NQ * 2 * (576 + 512)      # C1 over 576, C2 over 512
    qn, qr = case.q_bf16()
    out = qn.numel() * 2                                         # BF16 output, 512 per head
    indices = 4 * int(case.cur().sum())                          # the visible top-k entries
    want = (keys * 656 + qn.numel() * 2 + qr.numel() * 2 + out + indices
            + case.act.astype(np.int32).nbytes)
    assert case.algorithmic_bytes() == want


def test_mla_rows_used_are_the_rows_valid_entries_read():
    case = workloads.mla("acct", 2, 2, [300, 41], NQ=64, topk=128,
                         seed=workloads.BASE_SEED + 901, frac_invalid=0.1)
    tk = case.topk_indices()
    rows = set()
    for t in range(case.T):
        b, s = divmod(t, case.S1)
        visible = min(max(int(case.act[b]) - case.S1 + 1 + s, 0), case.topk)
        for j in range(visible):
            idx = int(tk[t, j])
            if 0 <= idx < int(case.act[b]):
                blk = max(int(case.block_table[b, idx // case.BS]), 0)
                rows.add(blk * case.BS + idx % case.BS)
    assert sorted(rows) == case.rows_used().tolist()
