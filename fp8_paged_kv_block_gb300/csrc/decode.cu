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
//  * Warp 8 is the producer: TMA 2-D tile loads (128 tokens x 128 bytes,
//    128-byte swizzle) of K then V blocks of each tile into a 10-slot
//    shared-memory ring, k_scale and the per-unit Q / q_scale / v_scale
//    header via cp.async, all tracked by mbarriers.
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

#include <mutex>

#include "common.cuh"

namespace pa {
namespace {

constexpr int kD = 128;
constexpr int kBS = 128;
constexpr int kNCW = 8;                      // consumer warps
constexpr int kThreads = (kNCW + 1) * 32;    // + one producer warp
constexpr int kNSlot = 10;                   // ring slots of one 128x128 block
constexpr int kSlotBytes = kBS * kD;
constexpr int kQStride = 144;                // padded Q row (bank-conflict free)
constexpr int kMaxB = 2048;
constexpr int kC0 = 64;                      // per-tile fixed cost (token units)
constexpr int kPartFloats = 32 * kD + 64;    // O[32][128], M[32], L[32]
constexpr size_t kWsHeader = 256;            // error flag + padding

template <int MT, int S2T>
struct __align__(1024) DecodeSmem {
    uint8_t ring[kNSlot][kSlotBytes];
    float kscale[kNSlot][kBS];
    uint32_t pfrag[2][S2T / 32][MT][32][4];
    uint8_t q[2][32][kQStride];
    float qscale[2][32];
    float vscale[2][kD];
    float red_max[kNCW][32];
    float red_l[kNCW][32];
    int scan[kThreads];
    int bpre[kMaxB + 1];
    uint64_t full_bar[kNSlot];
    uint64_t empty_bar[kNSlot];
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
    int B, S1, NQ, NKV, G, R, NRC, max_blocks, layout, grid, maxlen;
    float sscale;  // softmax_scale * log2(e)
};

struct Pos {
    int b, i, t;
};

__device__ __forceinline__ bool pos_eq(const Pos& a, const Pos& b)
{
    return a.b == b.b && a.i == b.i && a.t == b.t;
}

__device__ __forceinline__ int len_of(const DecodeParams& p, int b)
{
    int n = __ldg(p.act + b);
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
__device__ __forceinline__ Pos pos_next(const DecodeParams& p, const int* bpre, Pos x, int W)
{
    const int T = tiles_of<S2T>(len_of(p, x.b));
    if (++x.t >= T) {
        x.t = 0;
        if (++x.i == W) {
            x.i = 0;
            x.b = next_nonempty(bpre, x.b + 1, p.B);
        }
    }
    return x;
}

// First tile whose start cost is >= lo (END = {B, 0, 0} if none).
template <int S2T>
__device__ Pos find_pos(const DecodeParams& p, const int* bpre, int64_t lo, int64_t Ctot, int W)
{
    constexpr int TC = S2T + kC0;
    Pos end{p.B, 0, 0};
    if (lo >= Ctot) return end;
    int lb = 0, hb = p.B - 1;
    while (lb < hb) {
        const int mid = (lb + hb + 1) >> 1;
        if (static_cast<int64_t>(bpre[mid]) * W <= lo) lb = mid; else hb = mid - 1;
    }
    const int b = lb;
    const int64_t cost = bpre[b + 1] - bpre[b];
    const int64_t rem = lo - static_cast<int64_t>(bpre[b]) * W;
    int i = static_cast<int>(rem / cost);
    const int64_t r2 = rem - static_cast<int64_t>(i) * cost;
    int t = static_cast<int>((r2 + TC - 1) / TC);
    Pos x{b, i, t};
    if (t >= tiles_of<S2T>(len_of(p, b))) {
        x.t = 0;
        if (++x.i == W) {
            x.i = 0;
            x.b = next_nonempty(bpre, b + 1, p.B);
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

template <int MT, int S2T>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecodeParams p)
{
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
        for (int i = 0; i < kNSlot; ++i) {
            mbar_init(&sm.full_bar[i], 33);
            mbar_init(&sm.empty_bar[i], kNCW);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.hdr_full[i], 32);
            mbar_init(&sm.hdr_empty[i], kNCW);
        }
        sm.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }

    // ---- per-batch cost prefix: cost(b) = len_b + tiles_b * kC0 --------------
    {
        const int per = (p.B + kThreads - 1) / kThreads;
        const int b0 = min(tid * per, p.B), b1 = min(b0 + per, p.B);
        int local = 0;
        for (int b = b0; b < b1; ++b) {
            const int n = len_of(p, b);
            local += n + tiles_of<S2T>(n) * kC0;
        }
        // block-wide exclusive scan of `local`
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
            const int n = len_of(p, b);
            run += n + tiles_of<S2T>(n) * kC0;
        }
        __syncthreads();
    }

    const int64_t Ctot = static_cast<int64_t>(sm.bpre[p.B]) * W;
    const int cta = blockIdx.x;
    // Effective grid: at most Ctot / TC CTAs, so every CTA's share is at
    // least one full tile's cost. Then consecutive tiles of a unit land in
    // the same or the next CTA, and the CTAs holding a unit's tiles are a
    // contiguous run [first, last] (what the split combine counts on).
    const int64_t gcap = Ctot / TC;
    const int grid = static_cast<int>(gcap < 1 ? 1 : (gcap < p.grid ? gcap : p.grid));
    const Pos start = find_pos<S2T>(p, sm.bpre, (static_cast<int64_t>(cta) * Ctot + grid - 1) / grid, Ctot, W);
    const Pos end = find_pos<S2T>(p, sm.bpre, (static_cast<int64_t>(cta + 1) * Ctot + grid - 1) / grid, Ctot, W);

    if (cta >= grid) {
        // no tiles for this CTA; it may still owe zero rows for empty sequences
        if (warp < kNCW)
            for (int b = cta; b < p.B; b += p.grid) {
                if (len_of(p, b) != 0) continue;
                const int64_t row0 = static_cast<int64_t>(b) * p.S1 * p.NQ;
                const int64_t n16 = static_cast<int64_t>(p.S1) * p.NQ * kD * 2 / 16;
                uint4* dst = reinterpret_cast<uint4*>(p.out + row0 * kD);
                for (int64_t k = tid; k < n16; k += kNCW * 32) dst[k] = make_uint4(0, 0, 0, 0);
            }
        return;
    }

    if (warp == kNCW) {
        // =============================== producer ===============================
        const uint64_t pol = l2_evict_first_policy();
        int slot = 0;
        uint32_t ph = 0;
        int hcount = 0;
        bool first = true;
        for (Pos x = start; !pos_eq(x, end); x = pos_next<S2T>(p, sm.bpre, x, W)) {
            const int b = x.b, n2 = x.i / p.NRC, rc = x.i - (x.i / p.NRC) * p.NRC, t = x.t;
            const int len = len_of(p, b);
            if (first || t == 0) {
                const int hs = hcount & 1;
                mbar_wait(&sm.hdr_empty[hs], ((hcount >> 1) & 1) ^ 1, p.err, 2, &sm.abort);
                for (int ch = lane; ch < RCH * 8; ch += 32) {
                    const int rr = ch >> 3, part = ch & 7, r = rc * RCH + rr;
                    const uint8_t* src = p.q;
                    uint32_t nbytes = 0;
                    if (r < p.R) {
                        src = p.q + q_row(p, b, n2, r) * kD + part * 16;
                        nbytes = 16;
                    }
                    cp_async16(&sm.q[hs][rr][part * 16], src, nbytes);
                }
                if (lane < RCH) {
                    const int r = rc * RCH + lane;
                    const float* src = p.q_scale;
                    uint32_t nbytes = 0;
                    if (r < p.R) {
                        src = p.q_scale + q_row(p, b, n2, r);
                        nbytes = 4;
                    }
                    cp_async4(&sm.qscale[hs][lane], src, nbytes);
                }
                cp_async16(&sm.vscale[hs][lane * 4],
                           p.v_scale + (static_cast<int64_t>(b) * p.NKV + n2) * kD + lane * 4, 16);
                cp_async_arrive_noinc(&sm.hdr_full[hs]);
                ++hcount;
                first = false;
            }
            const int tok0 = t * S2T;
            const int nb = min(NBT, (len - tok0 + kBS - 1) / kBS);
            for (int kind = 0; kind < 2; ++kind) {
                for (int j = 0; j < nb; ++j) {
                    mbar_wait(&sm.empty_bar[slot], ph ^ 1, p.err, 4, &sm.abort);
                    int blk = __ldg(p.block_table + static_cast<int64_t>(b) * p.max_blocks + t * NBT + j);
                    if (blk < 0 || blk >= p.num_blocks) blk = 0;
                    int x0, y0;
                    if (p.layout == PA_LAYOUT_BSND) {
                        x0 = n2 * kD;
                        y0 = blk * kBS;
                    } else {
                        x0 = 0;
                        y0 = (blk * p.NKV + n2) * kBS;
                    }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&sm.full_bar[slot], kSlotBytes);
                        tma_load_2d(sm.ring[slot], kind ? &tmV : &tmK, x0, y0, &sm.full_bar[slot], pol);
                    }
                    if (kind == 0) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int off = lane * 4 + k;
                            const int64_t idx = p.layout == PA_LAYOUT_BSND
                                                    ? (static_cast<int64_t>(blk) * kBS + off) * p.NKV + n2
                                                    : (static_cast<int64_t>(blk) * p.NKV + n2) * kBS + off;
                            cp_async4(&sm.kscale[slot][off], p.k_scale + idx, 4);
                        }
                    }
                    cp_async_arrive_noinc(&sm.full_bar[slot]);
                    if (++slot == kNSlot) {
                        slot = 0;
                        ph ^= 1;
                    }
                }
            }
        }
        return;
    }

    // ================================ consumers ================================
    const int g = lane >> 2, tq = lane & 3;

    // sequences of length 0 produce zero rows (no tile ever covers them)
    for (int b = cta; b < p.B; b += p.grid) {
        if (len_of(p, b) != 0) continue;
        const int64_t row0 = static_cast<int64_t>(b) * p.S1 * p.NQ;
        const int64_t n16 = static_cast<int64_t>(p.S1) * p.NQ * kD * 2 / 16;
        uint4* dst = reinterpret_cast<uint4*>(p.out + row0 * kD);
        for (int64_t k = tid; k < n16; k += kNCW * 32) dst[k] = make_uint4(0, 0, 0, 0);
    }

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
        const int len = len_of(p, b);
        const int T = tiles_of<S2T>(len);

        if (first || t == 0) {
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
                qsc[mt][0] = sm.qscale[hs][mt * 16 + g] * p.sscale;
                qsc[mt][1] = sm.qscale[hs][mt * 16 + g + 8] * p.sscale;
            }
            vsc = *reinterpret_cast<const float4*>(&sm.vscale[hs][16 * warp + 4 * tq]);
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
            if (ks_slot >= kNSlot) {
                ks_slot -= kNSlot;
                ks_par ^= 1;
            }
            mbar_wait(&sm.full_bar[ks_slot], ks_par, p.err, 16, &sm.abort);
            const uint32_t kbase = smem_u32(sm.ring[ks_slot]);
            const float* ksm = sm.kscale[ks_slot];
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
                // dequant (q_scale * softmax_scale * log2e folded into qsc), mask, row max
                const int trow = wrow0 + 8 * j + 2 * tq;
                const float2 kk2 = *reinterpret_cast<const float2*>(ksm + trow);
                const int tk = wtok0 + 8 * j + 2 * tq;
                const bool v0 = tk < valid, v1 = tk + 1 < valid;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float x0 = v0 ? (s[mt][j][2 * h] * qsc[mt][h]) * kk2.x : -INFINITY;
                        const float x1 = v1 ? (s[mt][j][2 * h + 1] * qsc[mt][h]) * kk2.y : -INFINITY;
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
                if (tq == 0) sm.red_max[warp][mt * 16 + g + 8 * h] = v;
            }
        __syncwarp();
        if (lane == 0)
            for (int j = 0; j < nb; ++j) {
                int sl = slot + j;
                if (sl >= kNSlot) sl -= kNSlot;
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
                float m = sm.red_max[0][rr];
#pragma unroll
                for (int w = 1; w < kNCW; ++w) m = fmaxf(m, sm.red_max[w][rr]);
                const float mn = fmaxf(M[mt][h], m);
                Mn[mt][h] = mn;
                alpha[mt][h] = ex2(M[mt][h] - mn);
                const float a = ex2(m - mn);  // max_j P_j of this tile
                qs[mt][h] = a > 0.f ? __fdiv_rn(448.0f, a) : 0.f;
                ps[mt][h] = a > 0.f ? __frcp_rn(qs[mt][h]) : 0.f;
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

        // MM2 over the tile's valid k-steps for this warp's 16 channels
        float ot[MT][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int c = 0; c < 4; ++c) ot[mt][e][c] = 0.f;
        {
            const int nks = (valid + 31) >> 5;
            int cur = -1;
            uint32_t vbase = 0;
            for (int ksi = 0; ksi < nks; ++ksi) {
                const int bi = ksi >> 2;
                if (bi != cur) {
                    int vs_slot = slot + nb + bi;
                    uint32_t vs_par = ph;
                    if (vs_slot >= kNSlot) {
                        vs_slot -= kNSlot;
                        vs_par ^= 1;
                    }
                    mbar_wait(&sm.full_bar[vs_slot], vs_par, p.err, 32, &sm.abort);
                    vbase = smem_u32(sm.ring[vs_slot]);
                    cur = bi;
                }
                const int row = ((ksi & 3) << 5) + lane;
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
                    mma_e4m3(ot[mt][0], a, b0e0, b1e0);
                    mma_e4m3(ot[mt][1], a, b0e1, b1e1);
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            for (int j = 0; j < nb; ++j) {
                int sl = slot + nb + j;
                if (sl >= kNSlot) sl -= kNSlot;
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
                    O[mt][e][c] = O[mt][e][c] * alpha[mt][h] + (ot[mt][e][c] * ps[mt][h]) * vs;
                }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            M[mt][0] = Mn[mt][0];
            M[mt][1] = Mn[mt][1];
        }
        slot += 2 * nb;
        if (slot >= kNSlot) {
            slot -= kNSlot;
            ph ^= 1;
        }
        ++tcount;

        const Pos nx = pos_next<S2T>(p, sm.bpre, x, W);
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
            const int cf = cta_of(pu, Ctot, grid);
            const int cl = cta_of(pu + static_cast<int64_t>(T - 1) * TC, Ctot, grid);
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
pa_status launch(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& prm, cudaStream_t st)
{
    const size_t smem = sizeof(DecodeSmem<MT, S2T>) + 1024;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [&] {
        attr = cudaFuncSetAttribute(decode_kernel<MT, S2T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem));
    });
    PA_REQUIRE(attr == cudaSuccess, PA_ERR_CUDA, "pa_fp8_decode: smem attribute: %s", cudaGetErrorString(attr));
    decode_kernel<MT, S2T><<<prm.grid, kThreads, smem, st>>>(tk, tv, prm);
    return check_launch("pa_fp8_decode");
}

static_assert(sizeof(DecodeSmem<2, 512>) + 1024 <= 232448, "decode shared memory over budget");

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
                   aligned(out, 16),
               PA_ERR_INVALID, "pa_fp8_decode: misaligned pointer (q/k/v/v_scale need 16 bytes, out 16)");
    const int64_t rows = num_blocks * kBS * (layout == PA_LAYOUT_BNBD ? NKV : 1);
    PA_REQUIRE(rows < (int64_t(1) << 31), PA_ERR_UNSUPPORTED, "pa_fp8_decode: cache too large for 32-bit TMA rows");
    const int64_t maxlen = static_cast<int64_t>(max_blocks_per_seq) * kBS;
    const int64_t per_b = maxlen + (maxlen + pl.S2T - 1) / pl.S2T * kC0;
    PA_REQUIRE(per_b * B < (int64_t(1) << 31), PA_ERR_UNSUPPORTED,
               "pa_fp8_decode: B * max_blocks_per_seq too large for the 32-bit schedule");
    PA_REQUIRE(workspace != nullptr && aligned(workspace, 256), PA_ERR_WORKSPACE,
               "pa_fp8_decode: workspace missing or not 256-byte aligned");
    PA_REQUIRE(workspace_bytes >= pl.total, PA_ERR_WORKSPACE,
               "pa_fp8_decode: workspace %zu bytes < %zu required", workspace_bytes, pl.total);

    CUtensorMap tk, tv;
    const uint64_t inner = layout == PA_LAYOUT_BSND ? static_cast<uint64_t>(NKV) * kD : kD;
    st = make_cache_map(&tk, k_cache, inner, static_cast<uint64_t>(rows));
    if (st != PA_OK) return st;
    st = make_cache_map(&tv, v_cache, inner, static_cast<uint64_t>(rows));
    if (st != PA_OK) return st;

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
    prm.sscale = softmax_scale * 1.4426950408889634f;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pl.MT == 1) {
        if (pl.S2T == 128) return launch<1, 128>(tk, tv, prm, s);
        if (pl.S2T == 256) return launch<1, 256>(tk, tv, prm, s);
        return launch<1, 512>(tk, tv, prm, s);
    }
    if (pl.S2T == 128) return launch<2, 128>(tk, tv, prm, s);
    if (pl.S2T == 256) return launch<2, 256>(tk, tv, prm, s);
    return launch<2, 512>(tk, tv, prm, s);
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
