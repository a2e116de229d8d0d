// decode.cu -- paged FP8 decode attention (split-KV flash decoding) for sm_103a.
//
// What it computes: "PyPTO 实现 GLM-4.5 Paged Attention FP8 量化算子 ... Kernel
// 实战解析", 计算流程 steps 1-10 (gather K/V blocks through block_table, MM1
// Q_fp8.K_fp8^T -> FP32, dequant by q_scale and k_scale, online softmax with
// FP32 running max / sum / output, per-row FP8 quantisation of P over each
// s2 tile, MM2 P_fp8.V_fp8 -> FP32, dequant by P_scale and v_scale, final
// O / Sum cast to BF16); tensor signature from Kernel 签名与源码对应关系.
//
// GPU design (GB300, 152 SMs, HBM-bound: every K/V byte is read once):
//  * Work unit = (batch b, kv head n2, chunk of <= 32 query rows). A unit's
//    rows are all S1 x group query rows that share kv head n2, so each K/V
//    byte is read once for all of them. The unit's KV is walked in s2 tiles.
//  * Persistent grid, one CTA per SM. The flattened (unit, tile) sequence is
//    cut into contiguous per-CTA ranges balanced by token count (plus a fixed
//    per-tile cost); ranges start and end on tile boundaries so the
//    P-quantisation groups are those of the sequential walk. A unit split
//    across CTAs is merged by whichever CTA finishes its part last
//    (log-sum-exp combine through the workspace; no waiting on other CTAs).
//  * One thread of warp 8 is the producer. Per 128-token block it issues one
//    2-D TMA load (128 rows x 128 bytes, 128-byte swizzle) of K or V into a
//    shared-memory ring, plus one TMA of the block's key scales with K; the
//    unit's Q rows arrive by 1-D bulk copies. Block ids are loaded one tile
//    ahead, so no global load sits between two copies.
//  * Warps 0-7 consume. MM1: warp w takes s2_tile/8 tokens, FP8 mma.sync
//    m16n8k32 with Q as A (rows padded to 16/32) and K rows (ldmatrix) as B.
//    Row maxima meet in shared memory; P = exp2(S*log2e - M), its sum, and the
//    E4M3 quantisation (cvt.rn.satfinite) stay in registers, written once to
//    shared memory already in mma A-fragment order. MM2: warp w owns 16 of
//    the 128 output channels over the whole tile; V comes in through
//    ldmatrix.trans + byte permutes so no transpose pass is needed.
//  * Masked tokens (beyond kv_act_seqs) get S = -inf, P = 0, and their V
//    bytes are zeroed in registers (a stale E4M3 NaN code times 0 is NaN).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <mutex>

#include "common.cuh"

namespace pa {
namespace {

constexpr int kD = 128;
constexpr int kBS = 128;
constexpr int kNCW = 8;                      // consumer warps
constexpr int kThreads = (kNCW + 1) * 32;    // + one producer warp
constexpr int kSlotBytes = kBS * kD;         // one 128-token block of one head
constexpr int kKsFloats = 512;               // key-scale area per ring slot
constexpr int kMaxB = 1024;
// Work-balancing cost model in token units: a unit (batch, kv head, row
// chunk) costs kCU + tokens + tiles * kC0 (fixed per-unit and per-tile costs).
constexpr int kC0 = 512;
constexpr int kCU = 1024;
constexpr int kPartFloats = 32 * kD + 64;    // O[32][128], M[32], L[32]
constexpr size_t kWsHeader = 256;            // error flag + padding

// How one block's 128 key scales of one head arrive.
enum : int {
    KS_CONTIG = 0,   // BNBD: 128 contiguous floats, one 512-byte bulk copy
    KS_QUAD = 1,     // BSND, NKV % 4 == 0: 2-D TMA box of 4 heads x 128 rows
    KS_WHOLE = 2     // BSND, NKV <= 3: the block's whole [128][NKV] region
};

template <int MT, int S2T>
struct DecodeCfg {
    static constexpr int NSLOT = (MT == 2 && S2T == 512) ? 9 : 10;
};

template <int MT, int S2T>
struct __align__(1024) DecodeSmem {
    static constexpr int NSLOT = DecodeCfg<MT, S2T>::NSLOT;
    alignas(1024) uint8_t ring[NSLOT][kSlotBytes];
    alignas(1024) float kscale[NSLOT][kKsFloats];
    // P8 A-fragments (two-row-tile path only)
    alignas(128) uint32_t pfrag[MT == 1 ? 1 : 2][MT == 1 ? 1 : S2T / 32][MT][32][4];
    // P8 swap between paired warps / cross-warp output sum (one-row-tile path)
    alignas(128) float obuf[MT == 1 ? kNCW * 512 : 4];
    alignas(128) uint8_t q[2][32][kD];
    alignas(128) float vsc[2][kD];
    float red_max[2][kNCW][32];
    float red_l[kNCW][32];
    float rrow[32];
    float lrow[32];
    float mrow[32];
    int scan[kThreads];
    int bpre[kMaxB + 1];
    int slen[kMaxB];
    uint64_t full_bar[NSLOT];
    uint64_t empty_bar[NSLOT];
    uint64_t hdr_full[2];
    uint64_t hdr_empty[2];
    int flag;
    int abort;
};

struct DecodeParams {
    const uint8_t* q;
    const float* q_scale;
    const float* k_scale;
    const float* v_scale;
    const int32_t* block_table;
    const int32_t* act;
    __nv_bfloat16* out;
    float* part;
    int* counters;
    int* err;
    int64_t num_blocks;
    int B, S1, NQ, NKV, G, R, NRC, max_blocks, layout, grid, maxlen, ks_mode;
    float sscale;  // softmax_scale * log2(e)
};

struct Pos {
    int b, i, t;
};

__device__ __forceinline__ bool pos_eq(const Pos& a, const Pos& b)
{
    return a.b == b.b && a.i == b.i && a.t == b.t;
}

__device__ __forceinline__ int clamp_len(const DecodeParams& p, int n)
{
    return n < 0 ? 0 : (n > p.maxlen ? p.maxlen : n);
}

template <int S2T>
__device__ __forceinline__ int tiles_of(int len)
{
    return (len + S2T - 1) / S2T;
}

// First batch >= b with work (B if none).
__device__ __forceinline__ int next_nonempty(const int* bpre, int b, int B)
{
    while (b < B && bpre[b + 1] == bpre[b]) ++b;
    return b;
}

template <int S2T>
__device__ __forceinline__ Pos pos_next(const int* slen, const int* bpre, int B, Pos x, int W)
{
    if (++x.t >= tiles_of<S2T>(slen[x.b])) {
        x.t = 0;
        if (++x.i == W) {
            x.i = 0;
            x.b = next_nonempty(bpre, x.b + 1, B);
        }
    }
    return x;
}

// First tile whose start cost is >= lo (END = {B, 0, 0} if none).
template <int S2T>
__device__ Pos find_pos(const int* slen, const int* bpre, int B, int64_t lo, int64_t Ctot, int W)
{
    constexpr int TC = S2T + kC0;  // tile t of a unit starts at unit start + kCU + t * TC
    Pos end{B, 0, 0};
    if (lo >= Ctot) return end;
    int lb = 0, hb = B - 1;
    while (lb < hb) {
        const int mid = (lb + hb + 1) >> 1;
        if (static_cast<int64_t>(bpre[mid]) * W <= lo) lb = mid; else hb = mid - 1;
    }
    const int b = lb;
    const int64_t cost = bpre[b + 1] - bpre[b];
    const int64_t rem = lo - static_cast<int64_t>(bpre[b]) * W;
    int i = static_cast<int>(rem / cost);
    const int64_t r2 = rem - static_cast<int64_t>(i) * cost - kCU;
    int t = r2 <= 0 ? 0 : static_cast<int>((r2 + TC - 1) / TC);
    Pos x{b, i, t};
    if (t >= tiles_of<S2T>(slen[b])) {
        x.t = 0;
        if (++x.i == W) {
            x.i = 0;
            x.b = next_nonempty(bpre, b + 1, B);
        }
    }
    return x;
}

__device__ __forceinline__ int cta_of(int64_t s, int64_t Ctot, int grid)
{
    const int64_t c = (s * grid) / Ctot;
    return c >= grid ? grid - 1 : static_cast<int>(c);
}

__device__ __forceinline__ int64_t q_row(const DecodeParams& p, int b, int n2, int r)
{
    const int s = r / p.G, g = r - s * p.G;
    return (static_cast<int64_t>(b) * p.S1 + s) * p.NQ + n2 * p.G + g;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void zero_rows(const DecodeParams& p, int b, int tid, int nthreads)
{
    const int64_t row0 = static_cast<int64_t>(b) * p.S1 * p.NQ;
    const int64_t n16 = static_cast<int64_t>(p.S1) * p.NQ * kD * 2 / 16;
    uint4* dst = reinterpret_cast<uint4*>(p.out + row0 * kD);
    for (int64_t k = tid; k < n16; k += nthreads) dst[k] = make_uint4(0, 0, 0, 0);
}

template <int MT, int S2T>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmKS, const DecodeParams p)
{
    constexpr int NSLOT = DecodeCfg<MT, S2T>::NSLOT;
    constexpr int RCH = MT * 16;      // rows per unit chunk (padded)
    constexpr int NBT = S2T / kBS;    // blocks per tile
    constexpr int TPW = S2T / kNCW;   // MM1 tokens per warp
    constexpr int NT8 = TPW / 8;      // n8 tiles per warp
    constexpr int TC = S2T + kC0;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    auto& sm = *reinterpret_cast<DecodeSmem<MT, S2T>*>(smem_raw + ((1024u - (raw & 1023u)) & 1023u));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int W = p.NKV * p.NRC;

    if (tid == 0) {
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(&sm.full_bar[i], 1);
            mbar_init(&sm.empty_bar[i], kNCW);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.hdr_full[i], 1);
            mbar_init(&sm.hdr_empty[i], kNCW);
        }
        sm.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // Rows of a query chunk shorter than 32 are never copied in: start from
    // zeros (later such rows hold earlier finite Q codes, and their q_scale
    // is taken as 0).
    for (int k = tid; k < 2 * 32 * kD / 16; k += kThreads)
        reinterpret_cast<uint4*>(&sm.q[0][0][0])[k] = make_uint4(0, 0, 0, 0);

    // ---- per-batch lengths and cost prefix: cost(b) = kCU + len_b + tiles_b * kC0 --
    {
        const int per = (p.B + kThreads - 1) / kThreads;
        const int b0 = min(tid * per, p.B), b1 = min(b0 + per, p.B);
        int local = 0;
        for (int b = b0; b < b1; ++b) {
            const int n = clamp_len(p, __ldg(p.act + b));
            sm.slen[b] = n;
            local += n > 0 ? kCU + n + tiles_of<S2T>(n) * kC0 : 0;
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) sm.scan[warp] = incl;
        __syncthreads();
        if (tid == 0) {
            int run = 0;
            for (int w = 0; w < kThreads / 32; ++w) {
                const int v = sm.scan[w];
                sm.scan[w] = run;
                run += v;
            }
            sm.bpre[p.B] = run;
        }
        __syncthreads();
        int run = sm.scan[warp] + incl - local;
        for (int b = b0; b < b1; ++b) {
            sm.bpre[b] = run;
            run += sm.slen[b] > 0 ? kCU + sm.slen[b] + tiles_of<S2T>(sm.slen[b]) * kC0 : 0;
        }
        __syncthreads();
    }

    const int64_t Ctot = static_cast<int64_t>(sm.bpre[p.B]) * W;
    const int cta = blockIdx.x;
    // Effective grid: at most Ctot / (TC + kCU) CTAs, so every CTA's share is
    // at least the largest gap between consecutive tile starts. Then
    // consecutive tiles land in the same or the next CTA, and the CTAs holding
    // a unit's tiles are a contiguous run [first, last] (what the split
    // combine counts on).
    const int64_t gcap = Ctot / (TC + kCU);
    const int grid = static_cast<int>(gcap < 1 ? 1 : (gcap < p.grid ? gcap : p.grid));

    if (cta >= grid) {
        // no tiles for this CTA; it may still owe zero rows for empty sequences
        if (warp < kNCW)
            for (int b = cta; b < p.B; b += p.grid)
                if (sm.slen[b] == 0) zero_rows(p, b, tid, kNCW * 32);
        return;
    }
    const Pos start = find_pos<S2T>(sm.slen, sm.bpre, p.B,
                                    (static_cast<int64_t>(cta) * Ctot + grid - 1) / grid, Ctot, W);
    const Pos end = find_pos<S2T>(sm.slen, sm.bpre, p.B,
                                  (static_cast<int64_t>(cta + 1) * Ctot + grid - 1) / grid, Ctot, W);

    if (warp == kNCW) {
        // =============================== producer ===============================
        if (lane != 0) return;
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmK) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmV) : "memory");
        if (p.ks_mode == KS_QUAD) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmKS) : "memory");
        const uint64_t pol = l2_evict_first_policy();
        const int ks_bytes = p.ks_mode == KS_CONTIG ? kBS * 4
                                                    : (p.ks_mode == KS_QUAD ? kBS * 16 : kBS * 4 * p.NKV);
        int slot = 0;
        uint32_t ph = 0;
        int hcount = 0;
        bool first = true;
        // block ids of the current and the next tile (loaded one tile ahead)
        int cid[NBT], nid[NBT];
#pragma unroll
        for (int j = 0; j < NBT; ++j) nid[j] = 0;
        auto load_ids = [&](const Pos& x, int (&ids)[NBT]) {
            const int nbx = min(NBT, (sm.slen[x.b] - x.t * S2T + kBS - 1) / kBS);
            const int* row = p.block_table + static_cast<int64_t>(x.b) * p.max_blocks + x.t * NBT;
#pragma unroll
            for (int j = 0; j < NBT; ++j) ids[j] = j < nbx ? __ldg(row + j) : 0;
        };
        load_ids(start, cid);
        for (Pos x = start; !pos_eq(x, end);) {
            const Pos nx = pos_next<S2T>(sm.slen, sm.bpre, p.B, x, W);
            if (!pos_eq(nx, end)) load_ids(nx, nid);
            const int b = x.b, n2 = x.i / p.NRC, rc = x.i - (x.i / p.NRC) * p.NRC, t = x.t;
            const int len = sm.slen[b];
            if (first || t == 0) {
                // this unit's Q rows: one bulk copy per run of consecutive rows
                const int hs = hcount & 1;
                mbar_wait(&sm.hdr_empty[hs], ((hcount >> 1) & 1) ^ 1, p.err, 2, &sm.abort);
                const int r0 = rc * RCH, r1 = min(p.R, r0 + RCH);
                mbar_arrive_expect_tx(&sm.hdr_full[hs], static_cast<uint32_t>((r1 - r0) * kD + kD * 4));
                bulk_load_1d(&sm.vsc[hs][0], p.v_scale + (static_cast<int64_t>(b) * p.NKV + n2) * kD,
                             kD * 4, &sm.hdr_full[hs]);
                for (int r = r0; r < r1;) {
                    const int s = r / p.G, g0 = r - s * p.G;
                    const int n = min(p.G - g0, r1 - r);
                    bulk_load_1d(&sm.q[hs][r - r0][0], p.q + q_row(p, b, n2, r) * kD,
                                 static_cast<uint32_t>(n * kD), &sm.hdr_full[hs]);
                    r += n;
                }
                ++hcount;
                first = false;
            }
            const int nb = min(NBT, (len - t * S2T + kBS - 1) / kBS);
            for (int kind = 0; kind < 2; ++kind) {
#pragma unroll
                for (int j = 0; j < NBT; ++j) {
                    if (j >= nb) break;
                    mbar_wait(&sm.empty_bar[slot], ph ^ 1, p.err, 4, &sm.abort);
                    int blk = cid[j];
                    if (blk < 0 || blk >= p.num_blocks) blk = 0;
                    int x0, y0;
                    if (p.layout == PA_LAYOUT_BSND) {
                        x0 = n2 * kD;
                        y0 = blk * kBS;
                    } else {
                        x0 = 0;
                        y0 = (blk * p.NKV + n2) * kBS;
                    }
                    if (kind == 0) {
                        mbar_arrive_expect_tx(&sm.full_bar[slot], kSlotBytes + ks_bytes);
                        tma_load_2d(sm.ring[slot], &tmK, x0, y0, &sm.full_bar[slot], pol);
                        if (p.ks_mode == KS_CONTIG)
                            bulk_load_1d(sm.kscale[slot],
                                         p.k_scale + (static_cast<int64_t>(blk) * p.NKV + n2) * kBS,
                                         kBS * 4, &sm.full_bar[slot]);
                        else if (p.ks_mode == KS_QUAD)
                            tma_load_2d_nohint(sm.kscale[slot], &tmKS, n2 & ~3, blk * kBS,
                                               &sm.full_bar[slot]);
                        else
                            bulk_load_1d(sm.kscale[slot],
                                         p.k_scale + static_cast<int64_t>(blk) * kBS * p.NKV,
                                         static_cast<uint32_t>(ks_bytes), &sm.full_bar[slot]);
                    } else {
                        mbar_arrive_expect_tx(&sm.full_bar[slot], kSlotBytes);
                        tma_load_2d(sm.ring[slot], &tmV, x0, y0, &sm.full_bar[slot], pol);
                    }
                    if (++slot == NSLOT) {
                        slot = 0;
                        ph ^= 1;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < NBT; ++j) cid[j] = nid[j];
            x = nx;
        }
        return;
    }

    // ================================ consumers ================================
    const int g = lane >> 2, tq = lane & 3;

    // sequences of length 0 produce zero rows (no tile ever covers them)
    for (int b = cta; b < p.B; b += p.grid)
        if (sm.slen[b] == 0) zero_rows(p, b, tid, kNCW * 32);

    if constexpr (MT == 1) {
        // ------------------------------------------------------------------
        // One row tile (<= 16 query rows per kv head). Warps form 4 token
        // groups x 2 channel halves: warp w runs MM1 on its own s2_tile/8
        // tokens, keeps its P8 in registers in mma A-fragment order, swaps
        // it with its partner warp (w ^ 1) through shared memory, and runs
        // MM2 over the pair's tokens for 64 of the 128 channels. Per tile the
        // only CTA-wide exchange is the row maximum. The accumulator holds
        // O*448 / r, where r (per row) is the P-quantisation reference (max P
        // of the last tile that contributed); a new tile rescales it by
        // f = r * alpha / a (alpha = exp(M_old - M_new), a = max P of the
        // tile). The four token groups' partial outputs are summed once per
        // unit in shared memory.
        // ------------------------------------------------------------------
        constexpr int GT = 2 * TPW;           // tokens per group (pair of warps)
        constexpr int KSG = GT / 32;          // MM2 k-steps per group: 4 / 2 / 1
        constexpr int HU = TPW / 16;          // 16-token half k-steps per warp: 4 / 2 / 1
        constexpr float kMinA = 5.421010862427522e-20f;  // 2^-64
        const int tg = warp >> 1, dh = warp & 1;
        uint32_t* xbuf = reinterpret_cast<uint32_t*>(&sm.obuf[0]);   // [warp][lane][2*HU]
        int ks_st = 1, ks_off = 0;
        int slot = 0;
        uint32_t ph = 0;
        int hcount = 0, tcount = 0, hs = 0;
        bool first = true;
        uint32_t qa[4][4];
        float qsc[2], M[2], Lp[2], rsc[2];
        float Oh[4][2][4];

        for (Pos x = start; !pos_eq(x, end);) {
            const int b = x.b, n2 = x.i / p.NRC, rc = x.i - (x.i / p.NRC) * p.NRC, t = x.t;
            const int len = sm.slen[b];
            const int T = tiles_of<S2T>(len);

            if (first || t == 0) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = rc * RCH + g + 8 * h;
                    qsc[h] = r < p.R ? __ldg(p.q_scale + q_row(p, b, n2, r)) * p.sscale : 0.f;
                }
                if (p.ks_mode == KS_CONTIG) {
                    ks_st = 1;
                    ks_off = 0;
                } else if (p.ks_mode == KS_QUAD) {
                    ks_st = 4;
                    ks_off = n2 & 3;
                } else {
                    ks_st = p.NKV;
                    ks_off = n2;
                }
                hs = hcount & 1;
                mbar_wait(&sm.hdr_full[hs], (hcount >> 1) & 1, p.err, 8, &sm.abort);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint8_t* r0 = &sm.q[hs][g][kk * 32 + 4 * tq];
                    const uint8_t* r8 = &sm.q[hs][g + 8][kk * 32 + 4 * tq];
                    qa[kk][0] = *reinterpret_cast<const uint32_t*>(r0);
                    qa[kk][1] = *reinterpret_cast<const uint32_t*>(r8);
                    qa[kk][2] = *reinterpret_cast<const uint32_t*>(r0 + 16);
                    qa[kk][3] = *reinterpret_cast<const uint32_t*>(r8 + 16);
                }
                ++hcount;
                first = false;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    M[h] = -INFINITY;
                    Lp[h] = 0.f;
                    rsc[h] = 1.f;
                }
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
#pragma unroll
                        for (int i = 0; i < 4; ++i) Oh[c][e][i] = 0.f;
            }

            // ------------------------------ one s2 tile ------------------------------
            const int valid = min(S2T, len - t * S2T);
            const int nb = (valid + kBS - 1) / kBS;
            const int buf = tcount & 1;
            const int wtok0 = warp * TPW;
            const int wblk = wtok0 / kBS;
            const int wrow0 = wtok0 - wblk * kBS;
            const int gtok0 = tg * GT;
            const int gblk = gtok0 / kBS;
            const int grow0 = gtok0 - gblk * kBS;
            const bool active = wtok0 < valid;
            const bool gactive = gtok0 < valid;

            float s[NT8][4];
            float rmax[2] = {-INFINITY, -INFINITY};
            if (active) {
                int ks_slot = slot + wblk;
                uint32_t ks_par = ph;
                if (ks_slot >= NSLOT) {
                    ks_slot -= NSLOT;
                    ks_par ^= 1;
                }
                mbar_wait(&sm.full_bar[ks_slot], ks_par, p.err, 16, &sm.abort);
                const uint32_t kbase = smem_u32(sm.ring[ks_slot]);
                const float* ksm = sm.kscale[ks_slot];
                const bool full = wtok0 + TPW <= valid;
                // key scales first (their latency overlaps the MMAs)
                float kv0[NT8], kv1[NT8];
#pragma unroll
                for (int j = 0; j < NT8; ++j) {
                    const int trow = wrow0 + 8 * j + 2 * tq;
                    kv0[j] = ksm[trow * ks_st + ks_off];
                    kv1[j] = ksm[(trow + 1) * ks_st + ks_off];
                }
                // K fragments double-buffered one n8 tile ahead of the MMAs
                uint32_t bb[2][8];
                auto load_k = [&](int j, uint32_t (&dst)[8]) {
                    const int row = wrow0 + 8 * j + (lane & 7);
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int chunk = hf * 4 + (lane >> 3);
                        ldsm_x4(kbase + row * 128 + ((chunk ^ (row & 7)) << 4), dst[4 * hf], dst[4 * hf + 1],
                                dst[4 * hf + 2], dst[4 * hf + 3]);
                    }
                };
                load_k(0, bb[0]);
#pragma unroll
                for (int j = 0; j < NT8; ++j) {
                    if (j + 1 < NT8) load_k(j + 1, bb[(j + 1) & 1]);
                    float c4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) mma_e4m3(c4, qa[kk], bb[j & 1][2 * kk], bb[j & 1][2 * kk + 1]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[j][e] = c4[e];
                }
#pragma unroll
                for (int j = 0; j < NT8; ++j) {
                    const float k0 = kv0[j];
                    const float k1 = kv1[j];
                    const int tk = wtok0 + 8 * j + 2 * tq;
                    const bool v0 = full || tk < valid, v1 = full || tk + 1 < valid;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float x0 = v0 ? (s[j][2 * h] * qsc[h]) * k0 : -INFINITY;
                        const float x1 = v1 ? (s[j][2 * h + 1] * qsc[h]) * k1 : -INFINITY;
                        s[j][2 * h] = x0;
                        s[j][2 * h + 1] = x1;
                        rmax[h] = fmaxf(rmax[h], fmaxf(x0, x1));
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v = rmax[h];
                v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
                v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
                if (tq == 0) sm.red_max[buf][warp][g + 8 * h] = v;
            }
            __syncwarp();
            if (lane == 0)
                for (int j = 0; j < nb; ++j) {
                    int sl = slot + j;
                    if (sl >= NSLOT) sl -= NSLOT;
                    mbar_arrive(&sm.empty_bar[sl]);
                }
            named_bar_sync(1, kNCW * 32);

            // tile max -> running max, P quantisation scale, accumulator rescale
            float Mn[2], alpha[2], qs[2], f[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int rr = g + 8 * h;
                float m = sm.red_max[buf][0][rr];
#pragma unroll
                for (int w = 1; w < kNCW; ++w) m = fmaxf(m, sm.red_max[buf][w][rr]);
                const float mn = fmaxf(M[h], m);
                Mn[h] = mn;
                alpha[h] = ex2(M[h] - mn);
                const float a = ex2(m - mn);  // max_j P_j of this tile
                const bool use = a >= kMinA;
                qs[h] = use ? __fdividef(448.0f, a) : 0.f;
                f[h] = use ? __fdividef(rsc[h] * alpha[h], a) : 1.f;
                rsc[h] = use ? a : rsc[h] * alpha[h];
                M[h] = mn;
            }

            // P, its sum, and this warp's P8 as 16-token half k-steps
            // (own[u][0]: row g, own[u][1]: row g+8; tokens 16u .. 16u+15)
            uint32_t own[HU][2];
            if (active) {
                float lsum[2] = {0.f, 0.f};
#pragma unroll
                for (int j = 0; j < NT8; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = e >> 1;
                        const float pv = ex2(s[j][e] - Mn[h]);
                        lsum[h] += pv;
                        s[j][e] = pv * qs[h];
                    }
#pragma unroll
                for (int h = 0; h < 2; ++h) Lp[h] = Lp[h] * alpha[h] + lsum[h];
#pragma unroll
                for (int u = 0; u < HU; ++u) {
                    own[u][0] = e4m3x4(s[2 * u][0], s[2 * u][1], s[2 * u + 1][0], s[2 * u + 1][1]);
                    own[u][1] = e4m3x4(s[2 * u][2], s[2 * u][3], s[2 * u + 1][2], s[2 * u + 1][3]);
                }
            } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) Lp[h] = Lp[h] * alpha[h];
#pragma unroll
                for (int u = 0; u < HU; ++u) own[u][0] = own[u][1] = 0u;
            }
            // swap P8 with the partner warp of the token group
            {
                uint32_t* mine = xbuf + (warp * 32 + lane) * (2 * HU);
#pragma unroll
                for (int u = 0; u < HU; ++u)
                    *reinterpret_cast<uint2*>(mine + 2 * u) = make_uint2(own[u][0], own[u][1]);
            }
            named_bar_sync(2 + tg, 64);
            uint32_t par[HU][2];
            {
                const uint32_t* theirs = xbuf + (((warp ^ 1) * 32) + lane) * (2 * HU);
#pragma unroll
                for (int u = 0; u < HU; ++u) {
                    const uint2 v = *reinterpret_cast<const uint2*>(theirs + 2 * u);
                    par[u][0] = v.x;
                    par[u][1] = v.y;
                }
            }
            // A fragments of the group's k-steps: half k-steps 0..HU-1 belong
            // to warp 2tg, HU..2HU-1 to warp 2tg+1
            uint32_t pa[KSG][4];
#pragma unroll
            for (int kk = 0; kk < KSG; ++kk)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int uu = 2 * kk + hh;
                    const int owner = uu / HU, loc = uu - owner * HU;
                    const bool mineu = owner == dh;
                    pa[kk][2 * hh] = mineu ? own[loc][0] : par[loc][0];
                    pa[kk][2 * hh + 1] = mineu ? own[loc][1] : par[loc][1];
                }
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int e = 0; e < 2; ++e)
#pragma unroll
                    for (int i = 0; i < 4; ++i) Oh[c][e][i] *= f[i >> 1];

            if (gactive) {
                int vs_slot = slot + nb + gblk;
                uint32_t vs_par = ph;
                if (vs_slot >= NSLOT) {
                    vs_slot -= NSLOT;
                    vs_par ^= 1;
                }
                mbar_wait(&sm.full_bar[vs_slot], vs_par, p.err, 32, &sm.abort);
                const uint32_t vbase = smem_u32(sm.ring[vs_slot]);
#pragma unroll
                for (int kk = 0; kk < KSG; ++kk) {
                    const int tb = gtok0 + 32 * kk;
                    if (tb >= valid) break;
                    const int lim = valid - tb;
                    const int row = grow0 + 32 * kk + lane;
                    const int tk = 2 * tq;
                    const uint32_t m0 = (tk < lim ? 0x0000FFFFu : 0u) | (tk + 1 < lim ? 0xFFFF0000u : 0u);
                    const uint32_t m1 = (tk + 8 < lim ? 0x0000FFFFu : 0u) | (tk + 9 < lim ? 0xFFFF0000u : 0u);
                    const uint32_t m2 = (tk + 16 < lim ? 0x0000FFFFu : 0u) | (tk + 17 < lim ? 0xFFFF0000u : 0u);
                    const uint32_t m3 = (tk + 24 < lim ? 0x0000FFFFu : 0u) | (tk + 25 < lim ? 0xFFFF0000u : 0u);
                    // all four channel chunks of this k-step in flight at once
                    uint32_t rv[4][4];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        ldsm_x4_t(vbase + row * 128 + (((4 * dh + c) ^ (row & 7)) << 4), rv[c][0], rv[c][1],
                                  rv[c][2], rv[c][3]);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t r0 = rv[c][0], r1 = rv[c][1], r2 = rv[c][2], r3 = rv[c][3];
                        if (lim < 32) {  // zero V bytes of tokens past the sequence end
                            r0 &= m0;
                            r1 &= m1;
                            r2 &= m2;
                            r3 &= m3;
                        }
                        const uint32_t b0e0 = prmt(r0, r1, 0x6420), b1e0 = prmt(r2, r3, 0x6420);
                        const uint32_t b0e1 = prmt(r0, r1, 0x7531), b1e1 = prmt(r2, r3, 0x7531);
                        mma_e4m3(Oh[c][0], pa[kk], b0e0, b1e0);
                        mma_e4m3(Oh[c][1], pa[kk], b0e1, b1e1);
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                for (int j = 0; j < nb; ++j) {
                    int sl = slot + nb + j;
                    if (sl >= NSLOT) sl -= NSLOT;
                    mbar_arrive(&sm.empty_bar[sl]);
                }
            slot += 2 * nb;
            if (slot >= NSLOT) {
                slot -= NSLOT;
                ph ^= 1;
            }
            ++tcount;

            const Pos nx = pos_next<S2T>(sm.slen, sm.bpre, p.B, x, W);
            if (t == T - 1 || pos_eq(nx, end)) {
                // ------------------------------ unit end ------------------------------
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float l = Lp[h];
                    l += __shfl_xor_sync(0xffffffffu, l, 1);
                    l += __shfl_xor_sync(0xffffffffu, l, 2);
                    if (tq == 0) sm.red_l[warp][g + 8 * h] = l;
                }
                named_bar_sync(1, kNCW * 32);  // every warp is past its MM2 (xbuf free)
                if (warp == 0 && tq == 0) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float l = 0.f;
#pragma unroll
                        for (int w = 0; w < kNCW; ++w) l += sm.red_l[w][g + 8 * h];
                        sm.lrow[g + 8 * h] = l;
                        sm.rrow[g + 8 * h] = rsc[h];
                        sm.mrow[g + 8 * h] = M[h];
                    }
                }
                const int64_t u = static_cast<int64_t>(b) * W + x.i;
                const int64_t cost = sm.bpre[b + 1] - sm.bpre[b];
                const int64_t pu = static_cast<int64_t>(sm.bpre[b]) * W + static_cast<int64_t>(x.i) * cost;
                const int cf = cta_of(pu + kCU, Ctot, grid);
                const int cl = cta_of(pu + kCU + static_cast<int64_t>(T - 1) * TC, Ctot, grid);
                float* part = p.part + (u + cta) * kPartFloats;
                // Sum of the 4 token groups, rows 0-7 then 8-15. Accumulator
                // (c, e, i) of lane (g, tq) is channel 64dh + 16c + 4tq + e +
                // 2(i & 1) of row g + 8(i >> 1); it is stored in fragment order.
#pragma unroll
                for (int ih = 0; ih < 2; ++ih) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int e = 0; e < 2; ++e)
#pragma unroll
                            for (int il = 0; il < 2; ++il)
                                sm.obuf[warp * 512 + ((c * 2 + e) * 2 + il) * 32 + lane] = Oh[c][e][2 * ih + il];
                    named_bar_sync(1, kNCW * 32);
                    const int orow = 8 * ih + (tid >> 5);
                    const int d0 = (tid & 31) * 4;
                    const float rr = sm.rrow[orow] * (1.0f / 448.0f);
                    float ov[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int col = d0 + k;
                        const int dhh = col >> 6, cc = (col >> 4) & 3, r16 = col & 15;
                        const int src = ((cc * 2 + (r16 & 1)) * 2 + ((r16 >> 1) & 1)) * 32 + (orow & 7) * 4 + (r16 >> 2);
                        float acc = 0.f;
#pragma unroll
                        for (int gq = 0; gq < 4; ++gq) acc += sm.obuf[(2 * gq + dhh) * 512 + src];
                        ov[k] = acc * rr * sm.vsc[hs][col];
                    }
                    named_bar_sync(1, kNCW * 32);  // obuf free for the next round / unit
                    const int r = rc * RCH + orow;
                    if (cf == cl) {
                        if (r < p.R) {
                            const float L = sm.lrow[orow];
                            uint2 o;
                            o.x = pack_bf16x2(__fdiv_rn(ov[0], L), __fdiv_rn(ov[1], L));
                            o.y = pack_bf16x2(__fdiv_rn(ov[2], L), __fdiv_rn(ov[3], L));
                            *reinterpret_cast<uint2*>(p.out + q_row(p, b, n2, r) * kD + d0) = o;
                        }
                    } else {
                        *reinterpret_cast<float4*>(part + orow * kD + d0) = make_float4(ov[0], ov[1], ov[2], ov[3]);
                        if ((tid & 31) == 0) {
                            part[32 * kD + orow] = sm.mrow[orow];
                            part[32 * kD + 32 + orow] = sm.lrow[orow];
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.hdr_empty[hs]);
                if (cf != cl) {
                    __threadfence();
                    named_bar_sync(1, kNCW * 32);
                    if (tid == 0) {
                        const int old = atomicAdd(p.counters + u, 1);
                        const int last = (old == cl - cf);
                        if (last) p.counters[u] = 0;
                        sm.flag = last;
                    }
                    named_bar_sync(1, kNCW * 32);
                    if (sm.flag) {
                        __threadfence();
                        const int n = cl - cf + 1;
                        const int orow = tid >> 4, d0 = (tid & 15) * 8;
                        const int r = rc * RCH + orow;
                        if (r < p.R) {
                            float mx = -INFINITY;
                            for (int k = 0; k < n; ++k)
                                mx = fmaxf(mx, __ldcg(p.part + (u + cf + k) * kPartFloats + 32 * kD + orow));
                            float ls = 0.f;
                            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                            for (int k = 0; k < n; ++k) {
                                const float* pp = p.part + (u + cf + k) * kPartFloats;
                                const float sc = ex2(__ldcg(pp + 32 * kD + orow) - mx);
                                ls += __ldcg(pp + 32 * kD + 32 + orow) * sc;
                                const float4 o4a = __ldcg(reinterpret_cast<const float4*>(pp + orow * kD + d0));
                                const float4 o4b = __ldcg(reinterpret_cast<const float4*>(pp + orow * kD + d0 + 4));
                                acc[0] += o4a.x * sc;
                                acc[1] += o4a.y * sc;
                                acc[2] += o4a.z * sc;
                                acc[3] += o4a.w * sc;
                                acc[4] += o4b.x * sc;
                                acc[5] += o4b.y * sc;
                                acc[6] += o4b.z * sc;
                                acc[7] += o4b.w * sc;
                            }
                            uint4 o;
                            o.x = pack_bf16x2(__fdiv_rn(acc[0], ls), __fdiv_rn(acc[1], ls));
                            o.y = pack_bf16x2(__fdiv_rn(acc[2], ls), __fdiv_rn(acc[3], ls));
                            o.z = pack_bf16x2(__fdiv_rn(acc[4], ls), __fdiv_rn(acc[5], ls));
                            o.w = pack_bf16x2(__fdiv_rn(acc[6], ls), __fdiv_rn(acc[7], ls));
                            *reinterpret_cast<uint4*>(p.out + q_row(p, b, n2, r) * kD + d0) = o;
                        }
                    }
                }
            }
            x = nx;
        }
        return;
    }


    // key scale of row r of this CTA's head inside a slot: kscale[r*ks_st + ks_off]
    int ks_st = 1, ks_off = 0;

    int slot = 0;
    uint32_t ph = 0;
    int hcount = 0, tcount = 0;
    bool first = true;

    uint32_t qa[MT][4][4];
    float qsc[MT][2];
    float4 vsc = make_float4(0.f, 0.f, 0.f, 0.f);
    float M[MT][2], Lp[MT][2], O[MT][2][4];

    for (Pos x = start; !pos_eq(x, end);) {
        const int b = x.b, n2 = x.i / p.NRC, rc = x.i - (x.i / p.NRC) * p.NRC, t = x.t;
        const int len = sm.slen[b];
        const int T = tiles_of<S2T>(len);

        if (first || t == 0) {
            // per-unit scales: loads issued here, first used after MM1 / MM2
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = rc * RCH + mt * 16 + g + 8 * h;
                    qsc[mt][h] = r < p.R ? __ldg(p.q_scale + q_row(p, b, n2, r)) * p.sscale : 0.f;
                }
            vsc = __ldg(reinterpret_cast<const float4*>(p.v_scale +
                                                        (static_cast<int64_t>(b) * p.NKV + n2) * kD +
                                                        16 * warp + 4 * tq));
            if (p.ks_mode == KS_CONTIG) {
                ks_st = 1;
                ks_off = 0;
            } else if (p.ks_mode == KS_QUAD) {
                ks_st = 4;
                ks_off = n2 & 3;
            } else {
                ks_st = p.NKV;
                ks_off = n2;
            }
            const int hs = hcount & 1;
            mbar_wait(&sm.hdr_full[hs], (hcount >> 1) & 1, p.err, 8, &sm.abort);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint8_t* r0 = &sm.q[hs][mt * 16 + g][kk * 32 + 4 * tq];
                    const uint8_t* r8 = &sm.q[hs][mt * 16 + g + 8][kk * 32 + 4 * tq];
                    qa[mt][kk][0] = *reinterpret_cast<const uint32_t*>(r0);
                    qa[mt][kk][1] = *reinterpret_cast<const uint32_t*>(r8);
                    qa[mt][kk][2] = *reinterpret_cast<const uint32_t*>(r0 + 16);
                    qa[mt][kk][3] = *reinterpret_cast<const uint32_t*>(r8 + 16);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.hdr_empty[hs]);
            ++hcount;
            first = false;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    M[mt][h] = -INFINITY;
                    Lp[mt][h] = 0.f;
#pragma unroll
                    for (int c = 0; c < 4; ++c) O[mt][h][c] = 0.f;
                }
        }

        // --------------------------------- one s2 tile ---------------------------------
        const int tok0 = t * S2T;
        const int valid = min(S2T, len - tok0);
        const int nb = (valid + kBS - 1) / kBS;
        const int buf = tcount & 1;
        const int wtok0 = warp * TPW;
        const int wblk = wtok0 / kBS;
        const int wrow0 = wtok0 - wblk * kBS;

        float s[MT][NT8][4];
        float rmax[MT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) rmax[mt][0] = rmax[mt][1] = -INFINITY;

        if (wtok0 < valid) {
            int ks_slot = slot + wblk;
            uint32_t ks_par = ph;
            if (ks_slot >= NSLOT) {
                ks_slot -= NSLOT;
                ks_par ^= 1;
            }
            mbar_wait(&sm.full_bar[ks_slot], ks_par, p.err, 16, &sm.abort);
            const uint32_t kbase = smem_u32(sm.ring[ks_slot]);
            const float* ksm = sm.kscale[ks_slot];
            const bool full = wtok0 + TPW <= valid;
#pragma unroll
            for (int j = 0; j < NT8; ++j) {
                uint32_t bb[8];
                const int row = wrow0 + 8 * j + (lane & 7);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int chunk = hf * 4 + (lane >> 3);
                    ldsm_x4(kbase + row * 128 + ((chunk ^ (row & 7)) << 4), bb[4 * hf], bb[4 * hf + 1],
                            bb[4 * hf + 2], bb[4 * hf + 3]);
                }
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) mma_e4m3(c, qa[mt][kk], bb[2 * kk], bb[2 * kk + 1]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[mt][j][e] = c[e];
                }
            }
            // dequant (q_scale * softmax_scale * log2e, and k_scale), mask, row max
#pragma unroll
            for (int j = 0; j < NT8; ++j) {
                const int trow = wrow0 + 8 * j + 2 * tq;
                const float k0 = ksm[trow * ks_st + ks_off];
                const float k1 = ksm[(trow + 1) * ks_st + ks_off];
                const int tk = wtok0 + 8 * j + 2 * tq;
                const bool v0 = full || tk < valid, v1 = full || tk + 1 < valid;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float x0 = v0 ? (s[mt][j][2 * h] * qsc[mt][h]) * k0 : -INFINITY;
                        const float x1 = v1 ? (s[mt][j][2 * h + 1] * qsc[mt][h]) * k1 : -INFINITY;
                        s[mt][j][2 * h] = x0;
                        s[mt][j][2 * h + 1] = x1;
                        rmax[mt][h] = fmaxf(rmax[mt][h], fmaxf(x0, x1));
                    }
            }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v = rmax[mt][h];
                v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
                v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
                if (tq == 0) sm.red_max[0][warp][mt * 16 + g + 8 * h] = v;
            }
        __syncwarp();
        if (lane == 0)
            for (int j = 0; j < nb; ++j) {
                int sl = slot + j;
                if (sl >= NSLOT) sl -= NSLOT;
                mbar_arrive(&sm.empty_bar[sl]);
            }
        named_bar_sync(1, kNCW * 32);

        // tile row max -> running max, rescale factor, P quantisation scale
        float Mn[MT][2], alpha[MT][2], qs[MT][2], ps[MT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int rr = mt * 16 + g + 8 * h;
                float m = sm.red_max[0][0][rr];
#pragma unroll
                for (int w = 1; w < kNCW; ++w) m = fmaxf(m, sm.red_max[0][w][rr]);
                const float mn = fmaxf(M[mt][h], m);
                Mn[mt][h] = mn;
                alpha[mt][h] = ex2(M[mt][h] - mn);
                const float a = ex2(m - mn);  // max_j P_j of this tile
                qs[mt][h] = a > 0.f ? __fdividef(448.0f, a) : 0.f;
                ps[mt][h] = a * (1.0f / 448.0f);
            }

        if (wtok0 < valid) {
            float lsum[MT][2];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) lsum[mt][0] = lsum[mt][1] = 0.f;
#pragma unroll
            for (int j = 0; j < NT8; ++j)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = e >> 1;
                        const float pv = ex2(s[mt][j][e] - Mn[mt][h]);
                        lsum[mt][h] += pv;
                        s[mt][j][e] = pv * qs[mt][h];
                    }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) Lp[mt][h] = Lp[mt][h] * alpha[mt][h] + lsum[mt][h];
        } else {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) Lp[mt][h] = Lp[mt][h] * alpha[mt][h];
        }
        // P8 into shared memory in mma A-fragment order. Tokens 8j..8j+15 of the
        // warp (n8 tiles j, j+1) fill half of one 32-token k-step.
#pragma unroll
        for (int jp = 0; jp < NT8 / 2; ++jp) {
            const int j = 2 * jp;
            const int tb = wtok0 + 8 * j;
            const int ksi = tb >> 5, half = (tb >> 4) & 1;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint2 wv = make_uint2(0u, 0u);
                if (wtok0 < valid) {
                    wv.x = e4m3x4(s[mt][j][0], s[mt][j][1], s[mt][j + 1][0], s[mt][j + 1][1]);
                    wv.y = e4m3x4(s[mt][j][2], s[mt][j][3], s[mt][j + 1][2], s[mt][j + 1][3]);
                }
                *reinterpret_cast<uint2*>(&sm.pfrag[buf][ksi][mt][lane][2 * half]) = wv;
            }
        }
        named_bar_sync(1, kNCW * 32);

        // MM2 over the tile's valid k-steps for this warp's 16 channels; two
        // accumulator sets (even / odd k-step) halve the dependent mma chain.
        float ot[MT][2][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
                    for (int c = 0; c < 4; ++c) ot[mt][e][a2][c] = 0.f;
        {
            const int nks = (valid + 31) >> 5;
#pragma unroll
            for (int bi = 0; bi < NBT; ++bi) {
                if (bi >= nb) break;
                int vs_slot = slot + nb + bi;
                uint32_t vs_par = ph;
                if (vs_slot >= NSLOT) {
                    vs_slot -= NSLOT;
                    vs_par ^= 1;
                }
                mbar_wait(&sm.full_bar[vs_slot], vs_par, p.err, 32, &sm.abort);
                const uint32_t vbase = smem_u32(sm.ring[vs_slot]);
#pragma unroll
                for (int kb = 0; kb < 4; ++kb) {
                    const int ksi = bi * 4 + kb;
                    if (ksi >= nks) break;
                    const int row = (kb << 5) + lane;
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4_t(vbase + row * 128 + ((warp ^ (row & 7)) << 4), r0, r1, r2, r3);
                    const int lim = valid - (ksi << 5);
                    if (lim < 32) {  // zero V bytes of tokens past the sequence end
                        const int tk = 2 * tq;
                        r0 &= (tk < lim ? 0x0000FFFFu : 0u) | (tk + 1 < lim ? 0xFFFF0000u : 0u);
                        r1 &= (tk + 8 < lim ? 0x0000FFFFu : 0u) | (tk + 9 < lim ? 0xFFFF0000u : 0u);
                        r2 &= (tk + 16 < lim ? 0x0000FFFFu : 0u) | (tk + 17 < lim ? 0xFFFF0000u : 0u);
                        r3 &= (tk + 24 < lim ? 0x0000FFFFu : 0u) | (tk + 25 < lim ? 0xFFFF0000u : 0u);
                    }
                    const uint32_t b0e0 = prmt(r0, r1, 0x6420), b1e0 = prmt(r2, r3, 0x6420);
                    const uint32_t b0e1 = prmt(r0, r1, 0x7531), b1e1 = prmt(r2, r3, 0x7531);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        const uint4 af = *reinterpret_cast<const uint4*>(&sm.pfrag[buf][ksi][mt][lane][0]);
                        const uint32_t a[4] = {af.x, af.y, af.z, af.w};
                        mma_e4m3(ot[mt][0][kb & 1], a, b0e0, b1e0);
                        mma_e4m3(ot[mt][1][kb & 1], a, b0e1, b1e1);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            for (int j = 0; j < nb; ++j) {
                int sl = slot + nb + j;
                if (sl >= NSLOT) sl -= NSLOT;
                mbar_arrive(&sm.empty_bar[sl]);
            }
        // O = O * alpha + (O_t * P_scale) * v_scale. Channel of (e, c):
        // 16*warp + 4*tq + e + 2*(c & 1).
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int h = c >> 1;
                    const float vs = (c & 1) ? (e ? vsc.w : vsc.z) : (e ? vsc.y : vsc.x);
                    const float o_t = ot[mt][e][0][c] + ot[mt][e][1][c];
                    O[mt][e][c] = O[mt][e][c] * alpha[mt][h] + (o_t * ps[mt][h]) * vs;
                }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            M[mt][0] = Mn[mt][0];
            M[mt][1] = Mn[mt][1];
        }
        slot += 2 * nb;
        if (slot >= NSLOT) {
            slot -= NSLOT;
            ph ^= 1;
        }
        ++tcount;

        const Pos nx = pos_next<S2T>(sm.slen, sm.bpre, p.B, x, W);
        if (t == T - 1 || pos_eq(nx, end)) {
            // ------------------------------ unit end ------------------------------
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float l = Lp[mt][h];
                    l += __shfl_xor_sync(0xffffffffu, l, 1);
                    l += __shfl_xor_sync(0xffffffffu, l, 2);
                    if (tq == 0) sm.red_l[warp][mt * 16 + g + 8 * h] = l;
                }
            named_bar_sync(1, kNCW * 32);
            float Lr[MT][2];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float l = 0.f;
#pragma unroll
                    for (int w = 0; w < kNCW; ++w) l += sm.red_l[w][mt * 16 + g + 8 * h];
                    Lr[mt][h] = l;
                }
            const int64_t u = static_cast<int64_t>(b) * W + x.i;
            const int64_t cost = sm.bpre[b + 1] - sm.bpre[b];
            const int64_t pu = static_cast<int64_t>(sm.bpre[b]) * W + static_cast<int64_t>(x.i) * cost;
            const int cf = cta_of(pu + kCU, Ctot, grid);
            const int cl = cta_of(pu + kCU + static_cast<int64_t>(T - 1) * TC, Ctot, grid);
            if (cf == cl) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int r = rc * RCH + mt * 16 + g + 8 * h;
                        if (r >= p.R) continue;
                        const float L = Lr[mt][h];
                        uint2 o;
                        o.x = pack_bf16x2(__fdiv_rn(O[mt][0][2 * h], L), __fdiv_rn(O[mt][1][2 * h], L));
                        o.y = pack_bf16x2(__fdiv_rn(O[mt][0][2 * h + 1], L), __fdiv_rn(O[mt][1][2 * h + 1], L));
                        *reinterpret_cast<uint2*>(p.out + q_row(p, b, n2, r) * kD + 16 * warp + 4 * tq) = o;
                    }
            } else {
                float* part = p.part + (u + cta) * kPartFloats;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int rr = mt * 16 + g + 8 * h;
                        *reinterpret_cast<float4*>(part + rr * kD + 16 * warp + 4 * tq) =
                            make_float4(O[mt][0][2 * h], O[mt][1][2 * h], O[mt][0][2 * h + 1],
                                        O[mt][1][2 * h + 1]);
                        if (warp == 0 && tq == 0) {
                            part[32 * kD + rr] = M[mt][h];
                            part[32 * kD + 32 + rr] = Lr[mt][h];
                        }
                    }
                __threadfence();
                named_bar_sync(1, kNCW * 32);
                if (tid == 0) {
                    const int old = atomicAdd(p.counters + u, 1);
                    const int last = (old == cl - cf);
                    if (last) p.counters[u] = 0;
                    sm.flag = last;
                }
                named_bar_sync(1, kNCW * 32);
                if (sm.flag) {
                    __threadfence();
                    const int n = cl - cf + 1;
                    for (int item = tid; item < RCH * 32; item += kNCW * 32) {
                        const int rr = item >> 5, cg = item & 31, r = rc * RCH + rr;
                        if (r >= p.R) continue;
                        float mx = -INFINITY;
                        for (int k = 0; k < n; ++k)
                            mx = fmaxf(mx, __ldcg(p.part + (u + cf + k) * kPartFloats + 32 * kD + rr));
                        float ls = 0.f;
                        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int k = 0; k < n; ++k) {
                            const float* pp = p.part + (u + cf + k) * kPartFloats;
                            const float sc = ex2(__ldcg(pp + 32 * kD + rr) - mx);
                            ls += __ldcg(pp + 32 * kD + 32 + rr) * sc;
                            const float4 o4 = __ldcg(reinterpret_cast<const float4*>(pp + rr * kD + 4 * cg));
                            acc.x += o4.x * sc;
                            acc.y += o4.y * sc;
                            acc.z += o4.z * sc;
                            acc.w += o4.w * sc;
                        }
                        uint2 o;
                        o.x = pack_bf16x2(__fdiv_rn(acc.x, ls), __fdiv_rn(acc.y, ls));
                        o.y = pack_bf16x2(__fdiv_rn(acc.z, ls), __fdiv_rn(acc.w, ls));
                        *reinterpret_cast<uint2*>(p.out + q_row(p, b, n2, r) * kD + 4 * cg) = o;
                    }
                }
            }
        }
        x = nx;
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 2-D byte view of a paged cache: rows of `inner` bytes, box 128 x 128.
pa_status make_cache_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows)
{
    auto enc = tensor_map_encoder();
    PA_REQUIRE(enc != nullptr, PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kD), static_cast<cuuint32_t>(kBS)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    PA_REQUIRE(r == CUDA_SUCCESS, PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return PA_OK;
}

// 2-D float view of PA_BSND key scales [num_blocks*128 rows][NKV] with a box
// of 4 heads x 128 rows (NKV % 4 == 0).
pa_status make_kscale_map(CUtensorMap* map, const float* base, int NKV, uint64_t rows)
{
    auto enc = tensor_map_encoder();
    PA_REQUIRE(enc != nullptr, PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(NKV), rows};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(NKV) * 4};
    cuuint32_t box[2] = {4, static_cast<cuuint32_t>(kBS)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    PA_REQUIRE(r == CUDA_SUCCESS, PA_ERR_CUDA, "cuTensorMapEncodeTiled (key scales) failed (%d)",
               static_cast<int>(r));
    return PA_OK;
}

struct Plan {
    int S2T, MT, RCH, NRC, R, G, grid;
    int64_t U;
    size_t counters_bytes, part_bytes, total;
};

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

pa_status make_plan(int B, int S1, int NQ, int NKV, int D, const pa_decode_config* cfg, Plan* pl)
{
    PA_REQUIRE(B > 0 && S1 > 0 && NQ > 0 && NKV > 0 && D > 0, PA_ERR_INVALID,
               "pa_fp8_decode: empty or negative shape (B=%d S1=%d NQ=%d NKV=%d D=%d)", B, S1, NQ, NKV, D);
    PA_REQUIRE(NQ % NKV == 0, PA_ERR_INVALID, "pa_fp8_decode: NQ %d is not a multiple of NKV %d", NQ, NKV);
    PA_REQUIRE(D == kD, PA_ERR_UNSUPPORTED, "pa_fp8_decode: head size %d (only 128 is built)", D);
    PA_REQUIRE(B <= kMaxB, PA_ERR_UNSUPPORTED, "pa_fp8_decode: batch %d > %d", B, kMaxB);
    pl->S2T = (cfg && cfg->s2_tile) ? cfg->s2_tile : 512;
    PA_REQUIRE(pl->S2T > 0 && pl->S2T % kBS == 0, PA_ERR_INVALID,
               "pa_fp8_decode: s2_tile %d is not a multiple of block_size 128", pl->S2T);
    PA_REQUIRE(pl->S2T == 128 || pl->S2T == 256 || pl->S2T == 512, PA_ERR_UNSUPPORTED,
               "pa_fp8_decode: s2_tile %d (128, 256 and 512 are built)", pl->S2T);
    pl->G = NQ / NKV;
    pl->R = S1 * pl->G;
    pl->MT = pl->R <= 16 ? 1 : 2;
    pl->RCH = pl->MT * 16;
    pl->NRC = (pl->R + pl->RCH - 1) / pl->RCH;
    pl->U = static_cast<int64_t>(B) * NKV * pl->NRC;
    int grid = (cfg && cfg->num_ctas > 0) ? cfg->num_ctas : device_sm_count();
    PA_REQUIRE(grid > 0, PA_ERR_CUDA, "pa_fp8_decode: cannot query the device");
    pl->grid = grid;
    pl->counters_bytes = round256(static_cast<size_t>(pl->U) * sizeof(int));
    pl->part_bytes = static_cast<size_t>(pl->U + grid) * kPartFloats * sizeof(float);
    pl->total = kWsHeader + pl->counters_bytes + pl->part_bytes;
    return PA_OK;
}

template <int MT, int S2T>
pa_status launch(const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tks,
                 const DecodeParams& prm, cudaStream_t st)
{
    const size_t smem = sizeof(DecodeSmem<MT, S2T>) + 1024;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [&] {
        attr = cudaFuncSetAttribute(decode_kernel<MT, S2T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem));
    });
    PA_REQUIRE(attr == cudaSuccess, PA_ERR_CUDA, "pa_fp8_decode: smem attribute: %s", cudaGetErrorString(attr));
    decode_kernel<MT, S2T><<<prm.grid, kThreads, smem, st>>>(tk, tv, tks, prm);
    return check_launch("pa_fp8_decode");
}

// Bulk-copy / TMA destinations must be 16-byte aligned (128 for the tensor
// loads of key scales, 1024 for the 128-byte-swizzled K/V tiles).
template <int MT, int S2T>
struct SmemLayoutChecks {
    using S = DecodeSmem<MT, S2T>;
    static_assert(offsetof(S, ring) % 1024 == 0, "ring alignment");
    static_assert(offsetof(S, kscale) % 128 == 0, "kscale alignment");
    static_assert(offsetof(S, q) % 16 == 0, "q alignment");
    static_assert(offsetof(S, vsc) % 16 == 0, "vsc alignment");
    static_assert(offsetof(S, pfrag) % 16 == 0, "pfrag alignment");
    static_assert(offsetof(S, obuf) % 16 == 0, "obuf alignment");
    static_assert(sizeof(S) + 1024 <= 232448, "decode shared memory over budget");
    static constexpr bool ok = true;
};
static_assert(SmemLayoutChecks<1, 128>::ok && SmemLayoutChecks<1, 256>::ok && SmemLayoutChecks<1, 512>::ok &&
                  SmemLayoutChecks<2, 128>::ok && SmemLayoutChecks<2, 256>::ok && SmemLayoutChecks<2, 512>::ok,
              "shared memory layout");
static_assert(sizeof(DecodeSmem<2, 512>) + 1024 <= 232448, "decode shared memory over budget");
static_assert(sizeof(DecodeSmem<1, 512>) + 1024 <= 232448, "decode shared memory over budget");
static_assert(sizeof(DecodeSmem<2, 256>) + 1024 <= 232448, "decode shared memory over budget");

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_fp8_decode_workspace_size(int B, int S1, int NQ, int NKV, int D,
                                                  const pa_decode_config* cfg, size_t* bytes)
{
    PA_REQUIRE(bytes != nullptr, PA_ERR_NULLPTR, "pa_fp8_decode_workspace_size: bytes is NULL");
    Plan pl;
    pa_status st = make_plan(B, S1, NQ, NKV, D, cfg, &pl);
    if (st != PA_OK) return st;
    *bytes = pl.total;
    return PA_OK;
}

extern "C" pa_status pa_fp8_decode(const void* q, const float* q_scale, const void* k_cache,
                                   const float* k_scale, const void* v_cache, const float* v_scale,
                                   const int32_t* block_table, const int32_t* kv_act_seqs, void* out,
                                   int B, int S1, int NQ, int NKV, int D, int block_size,
                                   int64_t num_blocks, int max_blocks_per_seq, int layout,
                                   float softmax_scale, const pa_decode_config* cfg, void* workspace,
                                   size_t workspace_bytes, void* stream)
{
    PA_REQUIRE(q && q_scale && k_cache && k_scale && v_cache && v_scale && block_table &&
                   kv_act_seqs && out,
               PA_ERR_NULLPTR, "pa_fp8_decode: NULL tensor pointer");
    Plan pl;
    pa_status st = make_plan(B, S1, NQ, NKV, D, cfg, &pl);
    if (st != PA_OK) return st;
    PA_REQUIRE(block_size == kBS, PA_ERR_UNSUPPORTED, "pa_fp8_decode: block_size %d (only 128 is built)", block_size);
    PA_REQUIRE(num_blocks > 0 && max_blocks_per_seq > 0, PA_ERR_INVALID,
               "pa_fp8_decode: empty cache or block table");
    PA_REQUIRE(layout == PA_LAYOUT_BSND || layout == PA_LAYOUT_BNBD, PA_ERR_INVALID,
               "pa_fp8_decode: unknown layout %d", layout);
    PA_REQUIRE(aligned(q, 16) && aligned(k_cache, 16) && aligned(v_cache, 16) && aligned(v_scale, 16) &&
                   aligned(k_scale, 16) && aligned(out, 16),
               PA_ERR_INVALID,
               "pa_fp8_decode: misaligned pointer (q, caches, key/value scales and out need 16 bytes)");
    int ks_mode = KS_CONTIG;
    if (layout == PA_LAYOUT_BSND) {
        PA_REQUIRE(NKV % 4 == 0 || NKV <= 3, PA_ERR_UNSUPPORTED,
                   "pa_fp8_decode: PA_BSND key scales with NKV=%d (multiples of 4 and 1-3 are built)", NKV);
        ks_mode = NKV % 4 == 0 ? KS_QUAD : KS_WHOLE;
    }
    const int64_t rows = num_blocks * kBS * (layout == PA_LAYOUT_BNBD ? NKV : 1);
    PA_REQUIRE(rows < (int64_t(1) << 31), PA_ERR_UNSUPPORTED, "pa_fp8_decode: cache too large for 32-bit TMA rows");
    const int64_t maxlen = static_cast<int64_t>(max_blocks_per_seq) * kBS;
    const int64_t per_b = kCU + maxlen + (maxlen + pl.S2T - 1) / pl.S2T * kC0;
    PA_REQUIRE(per_b * B < (int64_t(1) << 31), PA_ERR_UNSUPPORTED,
               "pa_fp8_decode: B * max_blocks_per_seq too large for the 32-bit schedule");
    PA_REQUIRE(workspace != nullptr && aligned(workspace, 256), PA_ERR_WORKSPACE,
               "pa_fp8_decode: workspace missing or not 256-byte aligned");
    PA_REQUIRE(workspace_bytes >= pl.total, PA_ERR_WORKSPACE,
               "pa_fp8_decode: workspace %zu bytes < %zu required", workspace_bytes, pl.total);

    CUtensorMap tk, tv, tks;
    const uint64_t inner = layout == PA_LAYOUT_BSND ? static_cast<uint64_t>(NKV) * kD : kD;
    st = make_cache_map(&tk, k_cache, inner, static_cast<uint64_t>(rows));
    if (st != PA_OK) return st;
    st = make_cache_map(&tv, v_cache, inner, static_cast<uint64_t>(rows));
    if (st != PA_OK) return st;
    if (ks_mode == KS_QUAD) {
        st = make_kscale_map(&tks, k_scale, NKV, static_cast<uint64_t>(num_blocks) * kBS);
        if (st != PA_OK) return st;
    } else {
        tks = tk;  // not read by the kernel in this mode
    }

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    DecodeParams prm;
    prm.q = static_cast<const uint8_t*>(q);
    prm.q_scale = q_scale;
    prm.k_scale = k_scale;
    prm.v_scale = v_scale;
    prm.block_table = block_table;
    prm.act = kv_act_seqs;
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.err = reinterpret_cast<int*>(ws);
    prm.counters = reinterpret_cast<int*>(ws + kWsHeader);
    prm.part = reinterpret_cast<float*>(ws + kWsHeader + pl.counters_bytes);
    prm.num_blocks = num_blocks;
    prm.B = B;
    prm.S1 = S1;
    prm.NQ = NQ;
    prm.NKV = NKV;
    prm.G = pl.G;
    prm.R = pl.R;
    prm.NRC = pl.NRC;
    prm.max_blocks = max_blocks_per_seq;
    prm.layout = layout;
    prm.grid = pl.grid;
    prm.maxlen = static_cast<int>(maxlen);
    prm.ks_mode = ks_mode;
    prm.sscale = softmax_scale * 1.4426950408889634f;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pl.MT == 1) {
        if (pl.S2T == 128) return launch<1, 128>(tk, tv, tks, prm, s);
        if (pl.S2T == 256) return launch<1, 256>(tk, tv, tks, prm, s);
        return launch<1, 512>(tk, tv, tks, prm, s);
    }
    if (pl.S2T == 128) return launch<2, 128>(tk, tv, tks, prm, s);
    if (pl.S2T == 256) return launch<2, 256>(tk, tv, tks, prm, s);
    return launch<2, 512>(tk, tv, tks, prm, s);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of pa_fp8_decode: the same kernel, with its scratch
// (split partials, per-sequence counters, error flag) in a fixed array that
// is part of the library's device image instead of a caller workspace.
// ---------------------------------------------------------------------------
namespace pa {
namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(PA_FP8_DECODE_NOALLOC_MAX_SCRATCH);

// One array per device that loads the library, alive until process exit.
__device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

// Device address of g_decode_scratch on the current device. The host-side
// name is only a stand-in for the symbol, so the address is looked up once
// per device (with that device current) and cached.
pa_status decode_scratch_address(void** out)
{
    static std::mutex mu;
    static void* cache[64] = {nullptr};
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    PA_REQUIRE(e == cudaSuccess, PA_ERR_CUDA, "pa_fp8_decode_noalloc: cudaGetDevice: %s",
               cudaGetErrorString(e));
    PA_REQUIRE(dev >= 0 && dev < 64, PA_ERR_UNSUPPORTED, "pa_fp8_decode_noalloc: device %d", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        PA_REQUIRE(e == cudaSuccess && p != nullptr, PA_ERR_CUDA,
                   "pa_fp8_decode_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        cache[dev] = p;
    }
    *out = cache[dev];
    return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_fp8_decode_noalloc(const void* q, const float* q_scale, const void* k_cache,
                                           const float* k_scale, const void* v_cache,
                                           const float* v_scale, const int32_t* block_table,
                                           const int32_t* kv_act_seqs, void* out, int B, int S1,
                                           int NQ, int NKV, int D, int block_size,
                                           int64_t num_blocks, int max_blocks_per_seq, int layout,
                                           float softmax_scale, const pa_decode_config* cfg,
                                           void* stream)
{
    PA_REQUIRE(q && q_scale && k_cache && k_scale && v_cache && v_scale && block_table &&
                   kv_act_seqs && out,
               PA_ERR_NULLPTR, "pa_fp8_decode_noalloc: NULL tensor pointer");
    Plan pl;
    pa_status st = make_plan(B, S1, NQ, NKV, D, cfg, &pl);
    if (st != PA_OK) return st;
    PA_REQUIRE(pl.total <= kStaticScratchBytes, PA_ERR_WORKSPACE,
               "pa_fp8_decode_noalloc: this shape needs %zu bytes of scratch, more than the "
               "built-in %zu; use pa_fp8_decode with a caller workspace",
               pl.total, kStaticScratchBytes);
    void* ws = nullptr;
    st = decode_scratch_address(&ws);
    if (st != PA_OK) return st;
    // The array keeps the previous call's contents: the error flag and the
    // per-sequence counters must start at zero.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(ws, 0, kWsHeader + pl.counters_bytes, s);
    PA_REQUIRE(e == cudaSuccess, PA_ERR_CUDA, "pa_fp8_decode_noalloc: clearing scratch: %s",
               cudaGetErrorString(e));
    return pa_fp8_decode(q, q_scale, k_cache, k_scale, v_cache, v_scale, block_table, kv_act_seqs,
                         out, B, S1, NQ, NKV, D, block_size, num_blocks, max_blocks_per_seq, layout,
                         softmax_scale, cfg, ws, kStaticScratchBytes, stream);
}
