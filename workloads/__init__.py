"""Seeded synthetic inputs for FP8 paged decode attention and cache append.

This module holds no step of the method: it draws raw FP32 tensors (N(0,1)),
sequence lengths, paged block tables and slot mappings. Quantisation to E4M3
and everything after it is done separately by the CUDA library and by the
CPU oracle. Both sides take their inputs from here.

Workloads (sizes from the GLM-4.5 decode setting; D = 128, block_size = 128):
  tiny     B=2,  S1=1, NQ=4,  NKV=1, kv lengths {37, 300}, 8 physical blocks
  glm      B=16, S1=1, NQ=96, NKV=8, lengths ~ U{1..4096}, s2_tile 512
  long     B=4,  S1=1, NQ=96, NKV=8, lengths ~ U{32768..131072}; every 64th
           K row scaled by 8 before quantisation (outlier tokens)
  ragged   B=256, S1=2, NQ=96, NKV=8, lengths lognormal(median 1024, sigma 1)
           clipped to [1, 16384]
  append   64 new tokens (one per sequence) over contexts ~ U{512..8192},
           BNBD cache; 5% of the new slots are -1 (skipped)
The block pool holds the needed blocks plus 10% spare; each sequence's block
table row is a slice of a random permutation of the pool, padded with -1.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

LAYOUT_BSND = 0
LAYOUT_BNBD = 1
BASE_SEED = 20261202


def _rng(seed: int, *stream) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *stream])))


@dataclasses.dataclass
class DecodeCase:
    """One paged decode workload. Raw tensors are drawn lazily and cached."""

    name: str
    B: int
    S1: int
    NQ: int
    NKV: int
    act: np.ndarray            # int32 [B] kv_act_seqs
    max_blocks: int
    num_blocks: int
    block_table: np.ndarray    # int32 [B, max_blocks], -1 padded
    seed: int
    D: int = 128
    BS: int = 128
    s2_tile: int = 512
    layout: int = LAYOUT_BSND
    k_outlier_every: int = 0   # every n-th token row of K is scaled by k_outlier_scale
    k_outlier_scale: float = 8.0

    def __post_init__(self):
        self._q = None
        self._kv = None

    # ---- derived integer structure ------------------------------------
    @property
    def group(self) -> int:
        return self.NQ // self.NKV

    @property
    def softmax_scale(self) -> float:
        return float(np.float32(1.0) / np.sqrt(np.float32(self.D)))

    @property
    def cu_seqlens(self) -> np.ndarray:
        cu = np.zeros(self.B + 1, dtype=np.int64)
        cu[1:] = np.cumsum(np.maximum(self.act, 0).astype(np.int64))
        return cu

    @property
    def total_tokens(self) -> int:
        return int(np.maximum(self.act, 0).astype(np.int64).sum())

    @property
    def token_batch(self) -> np.ndarray:
        """int32 [Ttot]: the batch of each context token."""
        return np.repeat(np.arange(self.B, dtype=np.int32),
                         np.maximum(self.act, 0).astype(np.int64))

    @property
    def token_pos(self) -> np.ndarray:
        """int64 [Ttot]: the position of each context token in its sequence."""
        cu = self.cu_seqlens
        tb = self.token_batch
        return np.arange(self.total_tokens, dtype=np.int64) - cu[tb]

    @property
    def slots(self) -> np.ndarray:
        """int64 [Ttot]: physical cache slot of each context token,
        block_table[b][j // BS] * BS + j % BS."""
        tb = self.token_batch
        j = self.token_pos
        return self.block_table[tb, j // self.BS].astype(np.int64) * self.BS + j % self.BS

    # ---- raw FP32 tensors ------------------------------------------------
    def q(self) -> np.ndarray:
        """float32 [B*S1, NQ, D], N(0,1)."""
        if self._q is None:
            self._q = _rng(self.seed, 1).standard_normal(
                (self.B * self.S1, self.NQ, self.D), dtype=np.float32)
        return self._q

    def kv(self):
        """(k, v) float32 [Ttot, NKV, D], N(0,1), sequences concatenated in
        batch order (cu_seqlens). Drawn per sequence from its own stream."""
        if self._kv is None:
            T = self.total_tokens
            k = np.empty((T, self.NKV, self.D), dtype=np.float32)
            v = np.empty((T, self.NKV, self.D), dtype=np.float32)
            cu = self.cu_seqlens
            for b in range(self.B):
                n = int(cu[b + 1] - cu[b])
                if n == 0:
                    continue
                r = _rng(self.seed, 2, b)
                kb = r.standard_normal((n, self.NKV, self.D), dtype=np.float32)
                vb = r.standard_normal((n, self.NKV, self.D), dtype=np.float32)
                if self.k_outlier_every:
                    kb[:: self.k_outlier_every] *= np.float32(self.k_outlier_scale)
                k[cu[b]:cu[b + 1]] = kb
                v[cu[b]:cu[b + 1]] = vb
            self._kv = (k, v)
        return self._kv

    def drop(self):
        """Forget the cached raw tensors."""
        self._q = None
        self._kv = None

    # ---- byte accounting (valid tokens only) -----------------------------
    def algorithmic_bytes(self) -> int:
        """Bytes one decode step must move at minimum: K, V and k_scale of the
        valid tokens, q and q_scale, v_scale, the BF16 output, block table and
        lengths."""
        B, S1, NQ, NKV, D = self.B, self.S1, self.NQ, self.NKV, self.D
        return (self.total_tokens * NKV * (2 * D + 4) + B * S1 * NQ * (D + 4)
                + B * NKV * D * 4 + B * S1 * NQ * D * 2 + 4 * (B * self.max_blocks + B))

    def flops(self) -> int:
        return 4 * self.D * self.total_tokens * self.S1 * self.NQ


def _paged(name, B, S1, NQ, NKV, act, max_blocks, seed, *, num_blocks=None, spare=0.10,
           room=0, **kw) -> DecodeCase:
    """Block pool and tables for sequences of lengths ``act`` with space for
    ``room`` more tokens each."""
    act = np.asarray(act, dtype=np.int32)
    BS = kw.get("BS", 128)
    need = [int(math.ceil((int(a) + room) / BS)) for a in act]
    total = sum(need)
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(total * (1.0 + spare))))
    assert num_blocks >= total and max(need) <= max_blocks
    perm = _rng(seed, 0).permutation(num_blocks).astype(np.int32)
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        bt[b, :need[b]] = perm[pos:pos + need[b]]
        pos += need[b]
    return DecodeCase(name=name, B=B, S1=S1, NQ=NQ, NKV=NKV, act=act, max_blocks=max_blocks,
                      num_blocks=num_blocks, block_table=bt, seed=seed, **kw)


def tiny(s2_tile: int = 512, layout: int = LAYOUT_BSND) -> DecodeCase:
    """B=2, NQ=4, NKV=1, lengths {37, 300}, 8 physical blocks."""
    return _paged("tiny", 2, 1, 4, 1, [37, 300], 4, BASE_SEED + 0, num_blocks=8,
                  s2_tile=s2_tile, layout=layout)


def glm(s2_tile: int = 512, layout: int = LAYOUT_BSND, seed_offset: int = 0) -> DecodeCase:
    """GLM-4.5 decode shape: B=16, NQ=96, NKV=8, lengths ~ U{1..4096}."""
    seed = BASE_SEED + 1 + 1000 * seed_offset
    act = _rng(seed, 9).integers(1, 4096, size=16, endpoint=True)
    return _paged("glm", 16, 1, 96, 8, act, 33, seed, s2_tile=s2_tile, layout=layout, room=1)


def long_ctx(s2_tile: int = 512, layout: int = LAYOUT_BSND) -> DecodeCase:
    """B=4, NQ=96, NKV=8, lengths ~ U{32768..131072}, K outlier rows x8."""
    seed = BASE_SEED + 2
    act = _rng(seed, 9).integers(32768, 131072, size=4, endpoint=True)
    return _paged("long", 4, 1, 96, 8, act, 1025, seed, s2_tile=s2_tile, layout=layout,
                  k_outlier_every=64, room=1)


def ragged(s2_tile: int = 512, layout: int = LAYOUT_BSND, sigma: float = 1.0) -> DecodeCase:
    """B=256, S1=2, NQ=96, NKV=8, lengths lognormal (median 1024), clip [1, 16384]."""
    seed = BASE_SEED + 3
    x = _rng(seed, 9).normal(math.log(1024.0), sigma, size=256)
    act = np.clip(np.rint(np.exp(x)), 1, 16384).astype(np.int32)
    return _paged("ragged", 256, 2, 96, 8, act, 129, seed, s2_tile=s2_tile, layout=layout,
                  room=1)


def custom(name, B, S1, NQ, NKV, act, *, max_blocks=None, seed=BASE_SEED + 7, **kw):
    act = np.asarray(act, dtype=np.int32)
    BS = kw.get("BS", 128)
    if max_blocks is None:
        max_blocks = max(1, int(math.ceil(max(int(act.max()), 1) / BS)))
    return _paged(name, B, S1, NQ, NKV, act, max_blocks, seed, **kw)


# The six (b, s1, s2, nq, nkv) shapes of the GLM-4.5 paged FP8 page's test
# table (every sequence at its full s2).
PAGE_CASES = [
    (1, 2, 2048, 48, 8),
    (16, 1, 8195, 12, 2),
    (16, 1, 8192, 12, 1),
    (16, 1, 8192, 12, 2),
    (2, 1, 1024, 12, 1),
    (16, 1, 256, 16, 4),
]


def page_case(i: int, s2_tile: int = 512) -> DecodeCase:
    b, s1, s2, nq, nkv = PAGE_CASES[i]
    return custom("page%d" % i, b, s1, nq, nkv, [s2] * b, seed=BASE_SEED + 100 + i,
                  s2_tile=s2_tile)


def step_tokens(case: DecodeCase, seed_offset: int = 0):
    """One new token per sequence for a decode step: (key, value) BF16 torch
    CPU tensors [B, NKV, D] drawn N(0,1), the int32 slot of position
    kv_act_seqs[b] in each sequence's block table (-1 where the table has no
    room), and the lengths after the append."""
    import torch  # BF16 rounding by the library routine
    r = _rng(case.seed, 4, seed_offset)
    shape = (case.B, case.NKV, case.D)
    k = torch.from_numpy(r.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(r.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)
    a = case.act.astype(np.int64)
    bi = a // case.BS
    ok = bi < case.max_blocks
    blk = np.where(ok, case.block_table[np.arange(case.B), np.minimum(bi, case.max_blocks - 1)], -1)
    slot = np.where(blk >= 0, blk.astype(np.int64) * case.BS + a % case.BS, -1).astype(np.int32)
    act_after = (case.act + (slot >= 0)).astype(np.int32)
    return k, v, slot, act_after


@dataclasses.dataclass
class AppendCase:
    """Append one new token per sequence, then decode over the updated cache."""

    ctx: DecodeCase            # the existing contexts (BNBD cache)
    slot_mapping: np.ndarray   # int32 [T] slot of each new token (-1 = skipped)
    seed: int

    def __post_init__(self):
        self._new = None

    @property
    def T(self) -> int:
        return self.ctx.B

    def new_kv_f32(self):
        """(key, value) float32 [T, NKV, D] N(0,1), rounded to BF16 values."""
        import torch  # BF16 rounding by the library routine
        if self._new is None:
            r = _rng(self.seed, 3)
            shape = (self.T, self.ctx.NKV, self.ctx.D)
            k = torch.from_numpy(r.standard_normal(shape, dtype=np.float32))
            v = torch.from_numpy(r.standard_normal(shape, dtype=np.float32))
            self._new = (k.to(torch.bfloat16), v.to(torch.bfloat16))
        k, v = self._new
        return k.float().numpy(), v.float().numpy()

    def new_kv_bf16(self):
        """(key, value) as torch.bfloat16 CPU tensors [T, NKV, D]."""
        self.new_kv_f32()
        return self._new

    @property
    def token_batch(self) -> np.ndarray:
        return np.arange(self.T, dtype=np.int32)

    @property
    def act_after(self) -> np.ndarray:
        """kv_act_seqs after the append: +1 where the token was written."""
        return (self.ctx.act + (self.slot_mapping >= 0)).astype(np.int32)


def append(frac_skip: float = 0.05, B: int = 64, lo: int = 512, hi: int = 8192,
           s2_tile: int = 512) -> AppendCase:
    """64 new BF16 K/V rows into contexts ~ U{512..8192}, NQ=96, NKV=8, BNBD."""
    seed = BASE_SEED + 4
    r = _rng(seed, 9)
    act = r.integers(lo, hi, size=B, endpoint=True).astype(np.int32)
    BS = 128
    # room for one more token in every sequence
    max_blocks = int(math.ceil((hi + 1) / BS))
    need = [int(math.ceil((int(a) + 1) / BS)) for a in act]
    num_blocks = int(math.ceil(sum(need) * 1.1))
    perm = _rng(seed, 0).permutation(num_blocks).astype(np.int32)
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        bt[b, :need[b]] = perm[pos:pos + need[b]]
        pos += need[b]
    ctx = DecodeCase(name="append", B=B, S1=1, NQ=96, NKV=8, act=act, max_blocks=max_blocks,
                     num_blocks=num_blocks, block_table=bt, seed=seed, layout=LAYOUT_BNBD,
                     s2_tile=s2_tile)
    slot = (bt[np.arange(B), act // BS].astype(np.int64) * BS + act % BS).astype(np.int32)
    nskip = int(round(frac_skip * B))
    skip = r.choice(B, size=nskip, replace=False)
    slot[skip] = -1
    return AppendCase(ctx=ctx, slot_mapping=slot, seed=seed)


# --------------------------------------------------------------------------
# MLA sparse decode (DeepSeek-V3.2 shape): 128 query heads sharing one latent
# KV head of 512 "nope" + 64 rope channels; each query token selects `topk`
# positions of its sequence through top-k indices.
# --------------------------------------------------------------------------

MLA_DN = 512
MLA_DR = 64
MLA_ROW_BYTES = 672     # 656 used bytes padded to 672
# Cache row formats the MLA decode reads: the MLA page's packed row, and the
# KV compress epilog's row for d = 576 (rope first; 64-channel group scales,
# BF16 for its quant mode 0, E8M0 for quant mode 1).
MLA_FORMAT_PAGE = 0
MLA_FORMAT_KVC_BF16 = 1
MLA_FORMAT_KVC_E8M0 = 2


def _mix64(x: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser (a counter-based hash) on uint64 arrays."""
    x = (x ^ (x >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    x = (x ^ (x >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return x ^ (x >> np.uint64(31))


def _hashed_words(seed: int, rows: np.ndarray, nwords: int, lane: int) -> np.ndarray:
    """uint64 [len(rows), nwords]: hashed (seed, lane, row, word) counters, so
    a row's content depends on its id alone, whatever subset is drawn."""
    key = _mix64(np.array([seed * 1000003 + lane], dtype=np.uint64))[0]
    ctr = (np.asarray(rows, dtype=np.uint64)[:, None] * np.uint64(nwords)
           + np.arange(nwords, dtype=np.uint64)[None, :])
    with np.errstate(over="ignore"):
        return _mix64(ctr ^ key)


def _code_of_byte() -> np.ndarray:
    """Random byte -> E4M3 code: its sign bit, exponent field 6 + (bits 3..6
    scaled to 0..9), its low 3 bits as mantissa; the NaN pattern becomes the
    largest finite magnitude's neighbour."""
    b = np.arange(256, dtype=np.int64)
    e = 6 + (((b >> 3) & 15) * 10 >> 4)
    m = b & 7
    m = np.where((e == 15) & (m == 7), 6, m)
    return ((b & 0x80) | (e << 3) | m).astype(np.uint8)


_CODE_OF_BYTE = _code_of_byte()


def _uniform01(words: np.ndarray) -> np.ndarray:
    """float64 in (0, 1) from the top 53 bits."""
    return ((words >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / (1 << 53))


@dataclasses.dataclass
class MlaCase:
    """One MLA sparse decode workload. Cache rows are drawn as raw bytes:
    E4M3 codes with a random sign, exponent field uniform in [6, 15] (values
    2^-1 .. 448, the upper range an amax/448 group quantiser fills) and a
    random mantissa; 64 BF16 rope values N(0,1) (truncated to BF16); group
    scales: 4 FP32 uniform in [0.004, 0.009] (page format), 8 BF16 of the
    same range truncated to BF16 (KV compress quant mode 0), or 8 E8M0 bytes
    for 2^-8 or 2^-7 (quant mode 1). The bytes after the scales are 0xFF
    padding, which no step may use."""

    name: str
    B: int
    S1: int
    NQ: int
    topk: int
    act: np.ndarray            # int32 [B] kv_act_seqs
    max_blocks: int
    num_blocks: int
    block_table: np.ndarray    # int32 [B, max_blocks], -1 padded
    seed: int
    BS: int = 128
    s2_tile: int = 128
    frac_invalid: float = 0.0  # share of selected entries replaced by -1

    def __post_init__(self):
        self._q = None
        self._topk = {}

    @property
    def T(self) -> int:
        return self.B * self.S1

    @property
    def softmax_scale(self) -> float:
        return float(np.float32(1.0) / np.sqrt(np.float32(MLA_DN + MLA_DR)))

    def cur(self) -> np.ndarray:
        """int64 [T]: selected keys each query token attends to,
        clamp(kv_act_seqs[b] - S1 + 1 + s, 0, topk)."""
        t = np.arange(self.T)
        c = self.act[t // self.S1].astype(np.int64) - self.S1 + 1 + t % self.S1
        return np.clip(c, 0, self.topk)

    def topk_indices(self, variant: int = 0) -> np.ndarray:
        """int32 [T, topk]: for token (b, s) the first cur entries are distinct
        positions of its visible prefix [0, kv_act_seqs[b] - S1 + 1 + s) in
        random order (a share frac_invalid of them replaced by -1); the rest -1.
        Each variant is an independent draw (a different selection)."""
        if variant not in self._topk:
            out = np.full((self.T, self.topk), -1, dtype=np.int32)
            cur = self.cur()
            for t in range(self.T):
                n = int(cur[t])
                if n == 0:
                    continue
                b, s = divmod(t, self.S1)
                prefix = int(self.act[b]) - self.S1 + 1 + s
                r = _rng(self.seed, 5, t) if variant == 0 else _rng(self.seed, 5, t, variant)
                sel = r.permutation(prefix)[:n] if prefix <= 4 * n else \
                    r.choice(prefix, size=n, replace=False)
                if self.frac_invalid > 0:
                    sel = np.where(r.random(n) < self.frac_invalid, -1, sel)
                out[t, :n] = sel
            self._topk[variant] = out
        return self._topk[variant]

    def q_bf16(self):
        """(q_nope, q_rope) BF16 torch CPU tensors [T, NQ, 512] / [T, NQ, 64],
        N(0,1) rounded to BF16 by the library routine."""
        import torch
        if self._q is None:
            r = _rng(self.seed, 1)
            qn = r.standard_normal((self.T, self.NQ, MLA_DN), dtype=np.float32)
            qr = r.standard_normal((self.T, self.NQ, MLA_DR), dtype=np.float32)
            self._q = (torch.from_numpy(qn).to(torch.bfloat16),
                       torch.from_numpy(qr).to(torch.bfloat16))
        return self._q

    def q_bits(self):
        """(q_nope, q_rope) as uint16 BF16 bit patterns."""
        import torch
        qn, qr = self.q_bf16()
        return (qn.view(torch.int16).numpy().view(np.uint16),
                qr.view(torch.int16).numpy().view(np.uint16))

    def physical_rows(self, idx: np.ndarray, b: np.ndarray) -> np.ndarray:
        """int64 physical cache rows of sequence positions idx of batches b
        (a -1 block is read as block 0)."""
        blk = self.block_table[b, idx // self.BS].astype(np.int64)
        return np.maximum(blk, 0) * self.BS + idx % self.BS

    def _valid(self, variant: int):
        """(flat positions, batch of each) of the valid visible selected entries."""
        tk = self.topk_indices(variant)
        cur = self.cur()
        t = np.repeat(np.arange(self.T), self.topk)
        j = np.tile(np.arange(self.topk), self.T)
        idx = tk.reshape(-1).astype(np.int64)
        b = t // self.S1
        ok = (j < cur[t]) & (idx >= 0) & (idx < self.act[b])
        return idx[ok], b[ok]

    def rows_used(self, variants=(0,)) -> np.ndarray:
        """Sorted unique physical rows that valid selected keys read."""
        parts = [self.physical_rows(*self._valid(v)) for v in variants]
        return np.unique(np.concatenate(parts))

    def keys_read(self, variant: int = 0) -> int:
        """Valid selected (token, key) pairs: the packed rows one decode reads."""
        return int(self._valid(variant)[0].size)

    def row_bytes(self, rows: np.ndarray, fmt: int = MLA_FORMAT_PAGE) -> np.ndarray:
        """uint8 [len(rows), 672]: the cache rows with these ids in row format
        fmt (MLA_FORMAT_*). The codes and rope values of a row are the same
        draw in every format; only their places and the scales differ."""
        rows = np.asarray(rows, dtype=np.int64)
        n = rows.size
        code_at, rope_at = (0, MLA_DN) if fmt == MLA_FORMAT_PAGE else (2 * MLA_DR, 0)
        out = np.empty((n, MLA_ROW_BYTES), dtype=np.uint8)
        w = _hashed_words(self.seed, rows, MLA_DN // 8, 0).view(np.uint8).reshape(n, MLA_DN)
        out[:, code_at:code_at + MLA_DN] = _CODE_OF_BYTE[w]
        h = _hashed_words(self.seed, rows, MLA_DR, 1)
        u = ((h & np.uint64(0xFFFFFFFF)).astype(np.float32) + 0.5) * np.float32(2.0 ** -32)
        v = ((h >> np.uint64(32)).astype(np.float32) + 0.5) * np.float32(2.0 ** -32)
        rope = np.sqrt(np.float32(-2.0) * np.log(u)) * np.cos(np.float32(2.0 * np.pi) * v)
        out[:, rope_at:rope_at + 2 * MLA_DR] = (rope.view(np.uint32) >> np.uint32(16)).astype(
            np.uint16).view(np.uint8).reshape(n, 2 * MLA_DR)
        s0 = MLA_DN + 2 * MLA_DR
        if fmt == MLA_FORMAT_PAGE:
            h = _hashed_words(self.seed, rows, 2, 2)
            s4 = np.stack([h & np.uint64(0xFFFFFFFF), h >> np.uint64(32)], axis=-1).reshape(n, 4)
            sc = (np.float32(0.004) + np.float32(0.005 * 2.0 ** -32) * s4.astype(np.float32))
            out[:, s0:s0 + 16] = sc.astype(np.float32).view(np.uint8).reshape(n, 16)
            end = s0 + 16
        elif fmt == MLA_FORMAT_KVC_BF16:
            h = _hashed_words(self.seed, rows, 4, 3)
            s8 = np.stack([h & np.uint64(0xFFFFFFFF), h >> np.uint64(32)], axis=-1).reshape(n, 8)
            sc = (np.float32(0.004) + np.float32(0.005 * 2.0 ** -32) * s8.astype(np.float32))
            out[:, s0:s0 + 16] = (sc.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(
                np.uint16).view(np.uint8).reshape(n, 16)
            end = s0 + 16
        elif fmt == MLA_FORMAT_KVC_E8M0:
            h = _hashed_words(self.seed, rows, 1, 4).view(np.uint8).reshape(n, 8)
            out[:, s0:s0 + 8] = (np.uint8(119) + (h & np.uint8(1))).astype(np.uint8)
            end = s0 + 8
        else:
            raise ValueError("unknown MLA row format %r" % (fmt,))
        out[:, end:] = 0xFF
        return out

    def key_rows(self, rows: np.ndarray) -> np.ndarray:
        """float32 [len(rows), 576] holding BF16 values: unquantised key rows
        [nope 512 | rope 64] of these physical rows, N(0,1) truncated to BF16,
        for an append step (the KV compress epilog) to write into the cache.
        A row's values depend on its id alone."""
        rows = np.asarray(rows, dtype=np.int64)
        n = rows.size
        h = _hashed_words(self.seed, rows, (MLA_DN + MLA_DR) // 2, 5)
        u = ((h & np.uint64(0xFFFFFFFF)).astype(np.float32) + 0.5) * np.float32(2.0 ** -32)
        v = ((h >> np.uint64(32)).astype(np.float32) + 0.5) * np.float32(2.0 ** -32)
        r = np.sqrt(np.float32(-2.0) * np.log(u))
        x = np.concatenate([r * np.cos(np.float32(2.0 * np.pi) * v),
                            r * np.sin(np.float32(2.0 * np.pi) * v)], axis=1).astype(np.float32)
        return (x.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).reshape(n, -1)

    def cache(self, rows=None, fmt: int = MLA_FORMAT_PAGE) -> np.ndarray:
        """uint8 [num_blocks*BS, 672]: every row drawn (rows=None), or only the
        listed rows drawn and the others zero."""
        total = self.num_blocks * self.BS
        if rows is None:
            return self.row_bytes(np.arange(total), fmt)
        c = np.zeros((total, MLA_ROW_BYTES), dtype=np.uint8)
        c[rows] = self.row_bytes(rows, fmt)
        return c

    def flops(self, variant: int = 0) -> int:
        """2 * NQ * (576 + 512) per valid selected key of every query token:
        the two contractions."""
        return self.keys_read(variant) * 2 * self.NQ * (MLA_DN + MLA_DR + MLA_DN)

    def algorithmic_bytes(self, variant: int = 0) -> int:
        """Bytes one decode must move at minimum: the 656 used bytes of every
        selected row, the BF16 queries and output, the selected indices, the
        lengths (block-table reads are not counted)."""
        return (self.keys_read(variant) * 656 + self.T * self.NQ * (MLA_DN + MLA_DR) * 2
                + self.T * self.NQ * MLA_DN * 2 + int(self.cur().sum()) * 4 + self.B * 4)


def mla(name: str, B: int, S1: int, act, *, NQ: int = 128, topk: int = 2048, seed: int,
        spare: float = 0.10, frac_invalid: float = 0.0, BS: int = 128) -> MlaCase:
    act = np.asarray(act, dtype=np.int32)
    need = [max(1, int(math.ceil(int(a) / BS))) for a in act]
    max_blocks = max(need)
    num_blocks = max(1, int(math.ceil(sum(need) * (1.0 + spare))))
    perm = _rng(seed, 0).permutation(num_blocks).astype(np.int32)
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        bt[b, :need[b]] = perm[pos:pos + need[b]]
        pos += need[b]
    return MlaCase(name=name, B=B, S1=S1, NQ=NQ, topk=topk, act=act, max_blocks=max_blocks,
                   num_blocks=num_blocks, block_table=bt, seed=seed, BS=BS,
                   frac_invalid=frac_invalid)


def mla_page_ragged() -> MlaCase:
    """The MLA page's first decode case: b=4, nq=128, n_kv=1, s_q=2, actual
    sequence lengths [65536, 16381, 666, 15]."""
    return mla("mla_ragged", 4, 2, [65536, 16381, 666, 15], seed=BASE_SEED + 200)


def mla_page_b64(B: int = 64) -> MlaCase:
    """The MLA page's default decode case: b=64, nq=128, n_kv=1, s_q=2, every
    sequence 65536 long (B other than 64: the same case with fewer or more
    sequences)."""
    return mla("mla_b%d" % B, B, 2, [65536] * B, seed=BASE_SEED + 201)


WORKLOADS = {
    "tiny": tiny,
    "glm": glm,
    "long": long_ctx,
    "ragged": ragged,
}
