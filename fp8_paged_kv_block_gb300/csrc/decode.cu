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
//    cut into contiguous per-CTA ranges balanced by token count (plus fixed
//    per-unit and per-tile costs); ranges start and end on tile boundaries so
//    the P-quantisation groups are those of the sequential walk. A unit split
//    across CTAs is merged (log-sum-exp) by its first CTA, which reaches it
//    last; the other parts are published through the workspace with a
//    release count, and a bounded wait falls back to last-arriver merging.
//  * Warp 8 (one thread) feeds the K ring: per 128-token block one 2-D TMA
//    load (128 rows x 128 bytes, 128-byte swizzle); per unit the Q rows,
//    q_scale and v_scale. Warp 9 (one thread) feeds the V ring the same way.
//  * Warps 0-7 consume. Warp w owns tokens [w S2T/8, (w+1) S2T/8) of every
//    tile (one block, or part of one). For those tokens it
//      MM1  S[row][token] = Q_fp8 . K_fp8^T   warp-level mma.sync m16n8k32
//           E4M3 x E4M3 -> F32, Q fragments held in registers for the unit,
//           K fragments read with ldmatrix from the swizzled ring slot;
//    scales by q_scale * k_scale, masks past kv_act_seqs, finds the tile's
//    row maxima (in-thread, over the lane quad, then over the warps through
//    shared memory), P = 2^(x - tile max), the row sums and the E4M3 codes
//    P8 = 448 P, written as the MM2 operand; then one lane issues its
//      MM2  O^T[chan][row] = V_blk^T (MN-major: the V ring slot)
//                            x P8^T (K-major, 128-byte swizzle)
//    on the tensor cores (tcgen05.mma kind::f8f6f4, accumulator in tensor
//    memory, one accumulator per warp). A tcgen05.mma costs ~100 issue cycles
//    whatever its N, so the group-sized MM1 (N = query rows) runs faster as
//    warp MMAs next to the softmax; MM2 reads the V slot straight from the
//    ring. The warps' accumulators are summed in a fixed order when a tile is
//    folded into registers with the running-max rescale (double-buffered by
//    tile parity), so results do not depend on the order MMAs complete in.
//    Quantising against the tile's own maximum gives the same codes as
//    quantising exp(S - running max) against its tile maximum (the ratio
//    cancels the running max); the running max only weights whole tiles.
//  * Masked tokens get S = -inf (selected, never multiplied) and P = 0; the
//    V rows of a partial last block are zeroed in shared memory before MM2
//    (a stale E4M3 NaN code times 0 is NaN).
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
constexpr int kKProducerWarp = kNCW;        // K blocks and the per-unit header
constexpr int kVProducerWarp = kNCW + 1;    // V blocks
// Three full warpgroups: the consumers' two and the producers' (warps 10 and
// 11 only hand their registers over and exit), so that the register split
// below is made per warpgroup.
constexpr int kThreads = (kNCW + 4) * 32;
// Registers per thread after the split: the launch gives every thread 168
// (three warps share a sub-partition's register file); the producer
// warpgroup gives back down to kProdRegs and the consumers take the rest:
// 8 x kConsRegs + 4 x kProdRegs = 12 x 168.
constexpr int kProdRegs = 72;
constexpr int kConsRegs = 216;
static_assert(kNCW * kConsRegs + 4 * kProdRegs <= (kThreads / 32) * 168, "register split over the launch budget");
constexpr int kKSlots = 4;                   // K ring (one s2 tile of 512); the V ring takes the other slots
constexpr int kSlotBytes = kBS * kD;         // one 128-token block of one head
constexpr int kMaxB = 1024;
// Work-balancing cost model in token units: a unit (batch, kv head, row
// chunk) costs kCU + tokens + tiles * kC0 (fixed per-unit and per-tile costs).
constexpr int kC0 = 512;
constexpr int kCU = 1024;
constexpr int kPartFloats = 32 * kD + 64;    // O[32][128], M[32], L[32]
constexpr size_t kWsHeader = 256;            // error flag + padding
constexpr uint64_t kMergeWaitNs = 100000;     // the merging CTA's wait for the other parts

__host__ __device__ constexpr uint32_t tmem_cols(int need)
{
    uint32_t c = 32;
    while (c < static_cast<uint32_t>(need)) c <<= 1;
    return c;
}

// How an s2 tile is shared by the consumer warps.
template <int S2T>
struct TileSplit {
    static constexpr int NBT = S2T / kBS;                      // 128-token blocks per tile
    static constexpr int TPW = S2T / kNCW;                     // tokens per consumer warp
    static constexpr int NT = TPW / 8;                         // MM1 n-tiles (8 tokens) per warp
    static constexpr bool PAIRS = TPW < 32;                    // two warps share one 32-token MM2 k-step
    static constexpr int GT = PAIRS ? 32 : TPW;                // tokens per MM2 accumulator group
    static constexpr int OCW = S2T / GT;                       // accumulator groups (MMA-issuing warps)
    static constexpr int KW = kBS / TPW;                       // warps that read one block's K
    static constexpr int VW = kBS / GT;                        // warps whose MMAs read one block's V
    static constexpr int KSL = TPW >= 32 ? TPW / 32 : 1;       // key scales loaded per lane and tile
    static constexpr int MMS = GT / 32;                        // MM2 k-steps per issuing warp
    static_assert(TPW >= 16 && TPW <= kBS && TPW % 16 == 0, "tokens per warp");
};

struct Pos {
    int b, i, t;
};

// NR: padded query rows per unit (16 or 32); S2T: s2 tile; NS: ring slots (as
// many as fit): slots 0 .. NK-1 hold K blocks, the rest V blocks, each ring
// with its own producer.
template <int NR, int S2T, int NS>
struct __align__(1024) DecodeSmemT {
    static constexpr int NSLOT = NS;
    alignas(1024) uint8_t ring[NS][kSlotBytes];
    // P8 as the K-major MM2 operand, one 128-byte-swizzled atom per block:
    // token t of block a, row r at a * NR * 128 + r * 128 + (((t / 16) ^ (r % 8)) * 16) + t % 16
    // (also the BF16 staging of a unit's output rows, NR x 128 x 2 bytes)
    alignas(1024) uint8_t pbuf[S2T * NR > NR * kD * 2 ? S2T * NR : NR * kD * 2];
    alignas(16) uint8_t qb[2][NR][kD];    // the unit's Q rows (plain rows), by unit parity
    alignas(16) float vsc[2][kD];
    alignas(16) float qs[2][32];
    alignas(16) float ks[kNCW][TileSplit<S2T>::TPW];   // key scales of each warp's tokens
    alignas(16) float red[2][NR][kNCW];   // per-warp row maxima, double-buffered by tile
    alignas(16) float redl[kNCW][32];     // per-warp row sums at unit end
    alignas(16) float wst[kNCW][2][32];   // per-warp copies: [0] tile max, [1] q_scale or row sum
    alignas(16) float wfold[2][kNCW][2][32];   // per-warp fold weights c1, c2 by tile parity
    int scan[kThreads / 32];
    int bpre[kMaxB + 1];
    int slen[kMaxB];
    // A slot's uses alternate between two full barriers (use u on bank u & 1,
    // phase u / 2), so that a consumer waiting for a slot's second use within
    // a tile cannot mistake the first use's phase for it: consumer warps wait
    // for their own blocks in any order.
    uint64_t full_bar[NS][2];
    uint64_t empty_bar[NS];
    uint64_t hdr_full[2];
    uint64_t hdr_empty[2];
    uint64_t o_full;
    uint64_t done_bar;
    uint32_t tmem;
    Pos range[2];               // this CTA's first tile and the tile after its last
    int owner[2];               // first CTA of the range's first unit, last CTA of its last unit
    alignas(16) int64_t orow[2][32];   // output row of each query row of the unit (by unit parity)
    int k_tiles;                // tiles whose K blocks the K producer has requested
    int flag;
    int abort;
};

constexpr size_t kSmemOptIn = 232448;   // per-block opt-in maximum (the +1024 is alignment slack)

template <int NR, int S2T>
constexpr int pick_slots()
{
    return sizeof(DecodeSmemT<NR, S2T, 12>) + 1024 <= kSmemOptIn   ? 12
           : sizeof(DecodeSmemT<NR, S2T, 11>) + 1024 <= kSmemOptIn ? 11
           : sizeof(DecodeSmemT<NR, S2T, 10>) + 1024 <= kSmemOptIn ? 10
                                                                    : 9;
}

template <int NR, int S2T>
using DecodeSmem = DecodeSmemT<NR, S2T, pick_slots<NR, S2T>()>;

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
    int overlap;   // programmatic stream serialisation: 0 off, 1 prologue, 2 also older cache blocks
    float sscale;  // softmax_scale * log2(e)
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

// kv head of unit index i (i = n2 * NRC + row chunk); one chunk per head is
// the common case and needs no division
__device__ __forceinline__ int head_of(const DecodeParams& p, int i)
{
    return p.NRC == 1 ? i : i / p.NRC;
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

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float* v)
{
    if constexpr (N == 8) {
        tmem_ld8(taddr, v);
    } else {
#pragma unroll
        for (int c = 0; c < N; c += 16) tmem_ld16(taddr + c, v + c);
    }
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v)
{
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

template <int NR, int S2T>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecodeParams p)
{
    using TS = TileSplit<S2T>;
    constexpr int NBT = TS::NBT, TPW = TS::TPW, NT = TS::NT, GT = TS::GT, OCW = TS::OCW;
    constexpr int KSL = TS::KSL, MMS = TS::MMS;
    constexpr bool PAIRS = TS::PAIRS;
    constexpr int MT = NR / 16;                  // MM1 m-tiles of 16 query rows
    constexpr int HR = NR / 2;                   // O^T columns (query rows) per folding thread
    constexpr uint32_t TCOLS = tmem_cols(2 * OCW * NR);   // two O^T buffers of OCW accumulators
    constexpr int TC = S2T + kC0;
    constexpr int NSLOT = DecodeSmem<NR, S2T>::NSLOT;
    // K ring of kKSlots (one tile up to s2 tile 512), the V ring the rest. A
    // ring slot is used at most twice within one tile (two full-barrier banks)
    constexpr int NK = kKSlots, NV = NSLOT - NK;
    static_assert(NBT <= 2 * NK && NBT <= 2 * NV, "a ring slot would be used more than twice in a tile");
    static_assert(2 * OCW * NR <= 512, "tensor memory columns");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    auto& sm = *reinterpret_cast<DecodeSmem<NR, S2T>*>(smem_raw + ((1024u - (raw & 1023u)) & 1023u));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int W = p.NKV * p.NRC;
    // The next kernel of the stream may be scheduled now (it waits for this
    // one before touching anything this one writes).
    grid_launch_dependents();

    if (tid == 0) {
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(&sm.full_bar[i][0], 1);
            mbar_init(&sm.full_bar[i][1], 1);
            // K blocks are released by every consumer warp that reads them,
            // V blocks by the MM2 commits of the warps whose MMAs read them
            mbar_init(&sm.empty_bar[i], i < NK ? TS::KW : TS::VW);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.hdr_full[i], 2);           // byte-counted copies + the q_scale cp.async
            mbar_init(&sm.hdr_empty[i], kNCW);       // every consumer warp at the unit's end
        }
        mbar_init(&sm.o_full, OCW);                  // every accumulator group's MM2 share
        mbar_init(&sm.done_bar, kNCW);               // every consumer warp's last MMAs
        sm.abort = 0;
        sm.k_tiles = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // warm L2 with the block table; the producer reads it once its range is known
    {
        const int64_t bt_bytes = static_cast<int64_t>(p.B) * p.max_blocks * 4;
        if (static_cast<int64_t>(tid) * 128 < bt_bytes)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const uint8_t*>(p.block_table) +
                                                          static_cast<size_t>(tid) * 128));
    }

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
        grid_dependency_wait();
        if (warp < kNCW)
            for (int b = cta; b < p.B; b += p.grid)
                if (sm.slen[b] == 0) zero_rows(p, b, tid, kNCW * 32);
        return;
    }
    // this CTA's range: two lanes of the K producer warp find its ends (the
    // other warps get them through shared memory with the barrier below)
    if (warp == kKProducerWarp && lane < 2) {
        const Pos x = find_pos<S2T>(sm.slen, sm.bpre, p.B,
                                    (static_cast<int64_t>(cta + lane) * Ctot + grid - 1) / grid, Ctot, W);
        sm.range[lane] = x;
        // Only the range's first and last units can be shared with other CTAs:
        // the CTA holding the first unit's first tile, and the one holding the
        // last unit's last tile (for the split combine).
        int own = cta;
        if (x.b < p.B && x.t > 0) {
            const int64_t cost = sm.bpre[x.b + 1] - sm.bpre[x.b];
            const int64_t pu = static_cast<int64_t>(sm.bpre[x.b]) * W + static_cast<int64_t>(x.i) * cost;
            own = lane == 0 ? cta_of(pu + kCU, Ctot, grid)
                            : cta_of(pu + kCU + static_cast<int64_t>(tiles_of<S2T>(sm.slen[x.b]) - 1) * TC, Ctot,
                                     grid);
        }
        sm.owner[lane] = own;
    }

    // tensor memory (the MM2 accumulators): allocated by consumer warp 0,
    // address published in shared memory
    if (warp == 0) tmem_alloc(&sm.tmem, TCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem;
    const Pos start = sm.range[0];
    const Pos end = sm.range[1];

    if (warp >= kNCW) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProdRegs));
        if (warp > kVProducerWarp) return;
        // ============================== producers ==============================
        // The K producer fills the K ring (plus the per-unit header), the V
        // producer the V ring; each runs ahead of the consumers as far as its
        // own ring allows, so V tiles waiting for their P never hold back the
        // next tile's K.
        if (lane != 0) return;
        const bool isK = warp == kKProducerWarp;
        const CUtensorMap* tm = isK ? &tmK : &tmV;
        asm volatile("prefetch.tensormap [%0];" ::"l"(tm) : "memory");
        const uint64_t pol = l2_evict_first_policy();
        const int base = isK ? 0 : NK, nring = isK ? NK : NV;
        int hcount = 0, fills = 0, tcount = 0;   // fills: blocks issued into this ring so far
        bool first = true;
        // block ids, loaded two tiles ahead of their use
        int id0[NBT], id1[NBT], id2[NBT];
        auto load_ids = [&](const Pos& x, int (&ids)[NBT]) {
            if (pos_eq(x, end)) return;
            const int nbx = min(NBT, (sm.slen[x.b] - x.t * S2T + kBS - 1) / kBS);
            const int* row = p.block_table + static_cast<int64_t>(x.b) * p.max_blocks + x.t * NBT;
#pragma unroll
            for (int j = 0; j < NBT; ++j) ids[j] = j < nbx ? __ldg(row + j) : 0;
        };
#pragma unroll
        for (int j = 0; j < NBT; ++j) id0[j] = id1[j] = id2[j] = 0;
        // the unit's Q rows (one bulk copy per run of consecutive rows), its
        // q_scale values and its v_scale row
        auto issue_header = [&](int b, int n2, int rc) {
            const int hs = hcount & 1;
            mbar_wait(&sm.hdr_empty[hs], ((hcount >> 1) & 1) ^ 1, p.err, 2, &sm.abort);
            const int r0 = rc * NR, r1 = min(p.R, r0 + NR);
            mbar_arrive_expect_tx(&sm.hdr_full[hs], static_cast<uint32_t>((r1 - r0) * kD + kD * 4));
            bulk_load_1d(&sm.vsc[hs][0], p.v_scale + (static_cast<int64_t>(b) * p.NKV + n2) * kD,
                         kD * 4, &sm.hdr_full[hs]);
            for (int r = r0; r < r1;) {
                const int s = r / p.G, g0 = r - s * p.G;
                const int n = min(p.G - g0, r1 - r);
                const int64_t row = q_row(p, b, n2, r);
                bulk_load_1d(&sm.qb[hs][r - r0][0], p.q + row * kD, static_cast<uint32_t>(n * kD),
                             &sm.hdr_full[hs]);
                for (int k = 0; k < n; ++k) cp_async4(&sm.qs[hs][r - r0 + k], p.q_scale + row + k, 4);
                r += n;
            }
            cp_async_arrive_noinc(&sm.hdr_full[hs]);
            ++hcount;
        };
        bool waited = false;
        Pos x1 = start;
        load_ids(start, id0);
        if (!pos_eq(start, end)) {
            x1 = pos_next<S2T>(sm.slen, sm.bpre, p.B, start, W);
            load_ids(x1, id1);
        }
        for (Pos x = start; !pos_eq(x, end);) {
            const Pos nx = x1;
            if (!pos_eq(nx, end)) {
                x1 = pos_next<S2T>(sm.slen, sm.bpre, p.B, nx, W);
                load_ids(x1, id2);
            }
            const int b = x.b, n2 = head_of(p, x.i), rc = x.i - n2 * p.NRC, t = x.t;
            const int len = sm.slen[b];
            const bool need_hdr = isK && (first || t == 0);
            bool hdr_done = false;
            // MM1 needs the header; when the K ring is shorter than a tile the
            // tile's later K blocks wait for the consumers to read its first
            // ones, so the header goes out before them
            if (need_hdr && NK < NBT) {
                issue_header(b, n2, rc);
                hdr_done = true;
            }
            if (!waited) {
                // inputs not written by the preceding kernel may be read before
                // it ends; the KV cache only after (with overlap 2, only the
                // blocks that hold one of a sequence's S1 newest positions)
                if (need_hdr && !hdr_done && p.overlap) {
                    issue_header(b, n2, rc);
                    hdr_done = true;
                }
                if (p.overlap < 2) {
                    grid_dependency_wait();
                    waited = true;
                }
            }
            const int nb = min(NBT, (len - t * S2T + kBS - 1) / kBS);
            // V blocks of a tile are requested only after its K blocks: K is
            // needed first (MM1, softmax), V only once P is known
            if (!isK) {
                const volatile int* kt = &sm.k_tiles;
                if (*kt <= tcount) {
                    const uint64_t t0 = globaltimer_ns();
                    volatile int* ab = &sm.abort;
                    while (*kt <= tcount) {
                        __nanosleep(64);
                        if (*ab) break;
                        if (globaltimer_ns() - t0 > kWaitLimitNs) {
                            *ab = 1;
                            atomicOr(p.err, 2048);
                            break;
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < NBT; ++j) {
                if (j >= nb) break;
                // slot and use of this ring's fills-th block
                const int u = isK ? fills / NK : fills / NV;
                const int sl = base + (isK ? fills % NK : fills % NV);
                if (!waited && t * S2T + (j + 1) * kBS > len - p.S1) {
                    grid_dependency_wait();
                    waited = true;
                }
                mbar_wait(&sm.empty_bar[sl], (static_cast<uint32_t>(u) & 1u) ^ 1u, p.err, 4, &sm.abort);
                int blk = id0[j];
                if (blk < 0 || blk >= p.num_blocks) blk = 0;
                int x0, y0;
                if (p.layout == PA_LAYOUT_BSND) {
                    x0 = n2 * kD;
                    y0 = blk * kBS;
                } else {
                    x0 = 0;
                    y0 = (blk * p.NKV + n2) * kBS;
                }
                mbar_arrive_expect_tx(&sm.full_bar[sl][u & 1], kSlotBytes);
                tma_load_2d(sm.ring[sl], tm, x0, y0, &sm.full_bar[sl][u & 1], pol);
                ++fills;
            }
#pragma unroll
            for (int j = 0; j < NBT; ++j) {
                id0[j] = id1[j];
                id1[j] = id2[j];
            }
            if (isK) {
                __threadfence_block();
                *reinterpret_cast<volatile int*>(&sm.k_tiles) = tcount + 1;
            }
            // the unit's header after its first K blocks (K is the long pole; MM1
            // needs both), unless it went out before the dependency wait
            if (need_hdr && !hdr_done) issue_header(b, n2, rc);
            first = false;
            ++tcount;
            x = nx;
        }
        // every copy issued here lands before the CTA may exit
        for (int s = 0; s < nring; ++s) {
            const int n = fills / nring + (s < fills % nring ? 1 : 0);   // uses of slot s
            for (int u = n - 2 < 0 ? 0 : n - 2; u < n; ++u)
                mbar_wait_drain(&sm.full_bar[base + s][u & 1], static_cast<uint32_t>(u >> 1) & 1u, p.err, 1024);
        }
        if (isK) {
            for (int h = 0; h < 2; ++h) {
                const int n = hcount / 2 + (h < hcount % 2 ? 1 : 0);
                if (n > 0) mbar_wait_drain(&sm.hdr_full[h], static_cast<uint32_t>(n - 1) & 1u, p.err, 1024);
            }
        }
        return;
    }

    // ================================ consumers ================================
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsRegs));
    // MM1 / softmax: warp w owns tokens [w TPW, (w+1) TPW) of the tile: block
    // wblk, tokens tok0 .. tok0 + TPW - 1 of it. In the m16n8 fragments, lane
    // (g = lane / 4, t4 = lane % 4) holds rows g + 8 h + 16 m and tokens
    // 8 j + 2 t4 + {0, 1} of n-tile j.
    // Fold: warp w reads tensor-memory lanes 32 (w % 4) .. +31 (channels) and
    // O^T columns (query rows) hh * HR .. +HR - 1, hh = w / 4.
    const int g = lane >> 2, t4 = lane & 3;
    const int wblk = (warp * TPW) / kBS, tok0 = (warp * TPW) % kBS;
    const int grp = PAIRS ? (warp >> 1) : warp;           // this warp's MM2 accumulator group
    const bool issuer = !PAIRS || (warp & 1) == 0;        // the group's MMA-issuing warp
    const int q4 = warp & 3, hh = warp >> 2;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);

    int kpos = 0, vpos = 0;     // blocks of this CTA's walk before the current tile (ring positions)
    int hcount = 0, tcount = 0, hs = 0, nrows = 0;
    bool first = true;
    uint32_t qa[MT][4][4];      // Q fragments of the unit (m-tile, k-step, register)
    float Lp[MT][2];            // this thread's share of the row sums (running-max units)
    float Oa[HR];               // O^T[32 q4 + lane][hh * HR + k], times 448
    float Mref = -INFINITY;     // running max of row `lane` (lanes < NR; scaled log2 units)
#pragma unroll
    for (int m = 0; m < MT; ++m) Lp[m][0] = Lp[m][1] = 0.f;
#pragma unroll
    for (int k = 0; k < HR; ++k) Oa[k] = 0.f;
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) qa[m][kk][0] = qa[m][kk][1] = qa[m][kk][2] = qa[m][kk][3] = 0u;

    // Tile k's O^T (buffer k & 1: the accumulators of the groups that had
    // valid tokens, summed in group order) folded into Oa once its MM2 has
    // completed, with the weights of tile k.
    auto fold = [&](int k, int kvalid) {
        mbar_wait(&sm.o_full, k & 1, p.err, 512, &sm.abort);
        tc_fence_after();
        const int nact = min(OCW, (kvalid + GT - 1) / GT);
        constexpr int FC = HR == 8 ? 4 : 2;   // accumulators read per batch
        float acc[HR];
#pragma unroll
        for (int c = 0; c < HR; ++c) acc[c] = 0.f;
        const uint32_t cb = tl + static_cast<uint32_t>((k & 1) * OCW * NR + hh * HR);
#pragma unroll
        for (int a0 = 0; a0 < OCW; a0 += FC) {
            if (a0 >= nact) break;
            float ot[FC][HR];
#pragma unroll
            for (int i = 0; i < FC; ++i)
                if (a0 + i < nact) tmem_ld_cols<HR>(cb + static_cast<uint32_t>((a0 + i) * NR), ot[i]);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < FC; ++i)
                if (a0 + i < nact)
#pragma unroll
                    for (int c = 0; c < HR; ++c) acc[c] += ot[i][c];
        }
#pragma unroll
        for (int c4 = 0; c4 < HR / 4; ++c4) {
            const float4 a4 = *reinterpret_cast<const float4*>(&sm.wfold[k & 1][warp][0][hh * HR + 4 * c4]);
            const float4 b4 = *reinterpret_cast<const float4*>(&sm.wfold[k & 1][warp][1][hh * HR + 4 * c4]);
            Oa[4 * c4 + 0] = Oa[4 * c4 + 0] * a4.x + acc[4 * c4 + 0] * b4.x;
            Oa[4 * c4 + 1] = Oa[4 * c4 + 1] * a4.y + acc[4 * c4 + 1] * b4.y;
            Oa[4 * c4 + 2] = Oa[4 * c4 + 2] * a4.z + acc[4 * c4 + 2] * b4.z;
            Oa[4 * c4 + 3] = Oa[4 * c4 + 3] * a4.w + acc[4 * c4 + 3] * b4.w;
        }
        // buffer k & 1 is written again by tile k + 2's MMAs, which come
        // after that tile's row-maximum barrier
        tc_fence_before();
    };
    int pend = -1, pvalid = 0;   // tile whose O^T has not been folded yet, and its valid tokens
    // Key scales of this warp's tokens, read from global memory through L2
    // one tile ahead of their use (the block id one tile before that), staged
    // in shared memory per tile; no copy engine is used.
    auto tile_id = [&](const Pos& y) {
        const int nby = min(NBT, (sm.slen[y.b] - y.t * S2T + kBS - 1) / kBS);   // y.b < B here
        return wblk < nby ? __ldg(p.block_table + static_cast<int64_t>(y.b) * p.max_blocks + y.t * NBT + wblk)
                          : -1;
    };
    auto tile_ks = [&](const Pos& y, int id, float (&dst)[KSL]) {
        const int n2y = head_of(p, y.i);
        int blk = id;
        if (blk < 0 || blk >= p.num_blocks) blk = 0;
#pragma unroll
        for (int q = 0; q < KSL; ++q) {
            const int tok = tok0 + min(lane + 32 * q, TPW - 1);
            const int64_t idx = p.layout == PA_LAYOUT_BSND
                                    ? (static_cast<int64_t>(blk) * kBS + tok) * p.NKV + n2y
                                    : (static_cast<int64_t>(blk) * p.NKV + n2y) * kBS + tok;
            dst[q] = __ldcg(p.k_scale + idx);
        }
    };
    float ksn[KSL];   // key scales of the next tile
    int idn = -1;     // block id of the tile after it
#pragma unroll
    for (int q = 0; q < KSL; ++q) ksn[q] = 0.f;
    // The walk is carried in registers: the current tile, the next two, and
    // their sequence lengths (a tile's successor needs only its own length).
    auto advance = [&](Pos y, int leny, int& lnext) {
        if (++y.t < tiles_of<S2T>(leny)) {
            lnext = leny;
            return y;
        }
        y.t = 0;
        if (++y.i < W) {
            lnext = leny;
            return y;
        }
        y.i = 0;
        y.b = next_nonempty(sm.bpre, y.b + 1, p.B);
        lnext = y.b < p.B ? sm.slen[y.b] : 0;
        return y;
    };
    int lenx = pos_eq(start, end) ? 0 : sm.slen[start.b];
    int len1 = 0, len2 = 0;
    Pos x1 = end, x2 = end;
    if (!pos_eq(start, end)) x1 = advance(start, lenx, len1);
    if (!pos_eq(x1, end)) x2 = advance(x1, len1, len2);
    // block ids (not written by the preceding kernel) before its end; key
    // scales, out and the workspace only after it
    int id0 = -1;
    if (!pos_eq(start, end)) {
        id0 = tile_id(start);
        if (!pos_eq(x1, end)) idn = tile_id(x1);
    }
    grid_dependency_wait();
    if (!pos_eq(start, end)) tile_ks(start, id0, ksn);
    // sequences of length 0 produce zero rows (no tile ever covers them)
    for (int b = cta; b < p.B; b += p.grid)
        if (sm.slen[b] == 0) zero_rows(p, b, tid, kNCW * 32);

    constexpr uint32_t kIdescO = idesc_e4m3(128, NR, 1, 0);   // MN-major V^T, K-major P8^T

    for (Pos x = start; !pos_eq(x, end);) {
        const Pos nx = x1;
        const int b = x.b, n2 = head_of(p, x.i), rc = x.i - n2 * p.NRC, t = x.t;
        const int len = lenx;
        const int T = tiles_of<S2T>(len);

        if (first || t == 0) {
            hs = hcount & 1;
            mbar_wait(&sm.hdr_full[hs], (hcount >> 1) & 1, p.err, 8, &sm.abort);
            nrows = min(p.R - rc * NR, NR);
            if (warp == 0 && lane < NR) sm.orow[hcount & 1][lane] = q_row(p, b, n2, rc * NR + lane);
            // this warp's copy of q_scale * softmax_scale * log2(e) per row (0
            // past the chunk's rows); the slot holds the row sums at unit end
            if (lane < NR) sm.wst[warp][1][lane] = lane < nrows ? sm.qs[hs][lane] * p.sscale : 0.f;
            // Q fragments (rows past the chunk's end are zeros)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const int r0 = 16 * m + g, r1 = r0 + 8;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint8_t* a = &sm.qb[hs][r0][32 * kk + 4 * t4];
                    const uint8_t* c = &sm.qb[hs][r1][32 * kk + 4 * t4];
                    qa[m][kk][0] = r0 < nrows ? *reinterpret_cast<const uint32_t*>(a) : 0u;
                    qa[m][kk][1] = r1 < nrows ? *reinterpret_cast<const uint32_t*>(c) : 0u;
                    qa[m][kk][2] = r0 < nrows ? *reinterpret_cast<const uint32_t*>(a + 16) : 0u;
                    qa[m][kk][3] = r1 < nrows ? *reinterpret_cast<const uint32_t*>(c + 16) : 0u;
                }
            }
            __syncwarp();
#pragma unroll
            for (int m = 0; m < MT; ++m) Lp[m][0] = Lp[m][1] = 0.f;
#pragma unroll
            for (int k = 0; k < HR; ++k) Oa[k] = 0.f;
            Mref = -INFINITY;
            ++hcount;
            first = false;
        }

        const int valid = min(S2T, len - t * S2T);
        const int nb = (valid + kBS - 1) / kBS;
        const bool hasblk = wblk < nb;
        const int wvalid = min(max(valid - warp * TPW, 0), TPW);   // this warp's valid tokens
        const int gvalid = min(max(valid - grp * GT, 0), GT);      // its accumulator group's
        // this tile's key scales to shared memory; the next tile's requested
#pragma unroll
        for (int q = 0; q < KSL; ++q)
            if (lane + 32 * q < TPW) sm.ks[warp][lane + 32 * q] = ksn[q];
        __syncwarp();
        if (!pos_eq(nx, end)) {
            tile_ks(nx, idn, ksn);
            if (!pos_eq(x2, end)) idn = tile_id(x2);
        }
        // the walk moves on by one tile
        lenx = len1;
        x1 = x2;
        len1 = len2;
        if (!pos_eq(x2, end)) x2 = advance(x2, len2, len2);

        // ---- MM1: S = Q . K^T for this warp's tokens (mma.sync, K via ldmatrix) ----
        float sc[MT][NT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int j = 0; j < NT; ++j) sc[m][j][0] = sc[m][j][1] = sc[m][j][2] = sc[m][j][3] = 0.f;
        if (hasblk) {
            const int ku = (kpos + wblk) / NK, ksl = (kpos + wblk) % NK;
            mbar_wait(&sm.full_bar[ksl][ku & 1], static_cast<uint32_t>(ku >> 1) & 1u, p.err, 16, &sm.abort);
            if (wvalid > 0) {
                // lane L addresses row L % 8 of matrix L / 8; the 16-byte chunk c
                // of a token row sits at (c ^ row % 8) * 16 (128-byte swizzle)
                const int r7 = lane & 7, qm = lane >> 3;
                const uint32_t kb = smem_u32(sm.ring[ksl]) + static_cast<uint32_t>((tok0 + r7) * 128);
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    uint32_t kf[8];
                    const uint32_t row = kb + static_cast<uint32_t>(j * 8 * 128);
                    ldsm_x4(row + static_cast<uint32_t>((qm ^ r7) << 4), kf[0], kf[1], kf[2], kf[3]);
                    ldsm_x4(row + static_cast<uint32_t>(((4 + qm) ^ r7) << 4), kf[4], kf[5], kf[6], kf[7]);
#pragma unroll
                    for (int m = 0; m < MT; ++m)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) mma_e4m3(sc[m][j], qa[m][kk], kf[2 * kk], kf[2 * kk + 1]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty_bar[ksl]);
        }

        // ---- scores x = S * q_scale * scale * log2(e) * k_scale; tile row maxima ----
        float mx[MT][2];
        {
            float qsc[MT][2];
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                qsc[m][0] = sm.wst[warp][1][16 * m + g];
                qsc[m][1] = sm.wst[warp][1][16 * m + g + 8];
                mx[m][0] = mx[m][1] = -INFINITY;
            }
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int tk = 8 * j + 2 * t4;
                const float2 kv = *reinterpret_cast<const float2*>(&sm.ks[warp][tk]);
                const bool ok0 = tk < wvalid, ok1 = tk + 1 < wvalid;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    sc[m][j][0] = ok0 ? (sc[m][j][0] * qsc[m][0]) * kv.x : -INFINITY;
                    sc[m][j][1] = ok1 ? (sc[m][j][1] * qsc[m][0]) * kv.y : -INFINITY;
                    sc[m][j][2] = ok0 ? (sc[m][j][2] * qsc[m][1]) * kv.x : -INFINITY;
                    sc[m][j][3] = ok1 ? (sc[m][j][3] * qsc[m][1]) * kv.y : -INFINITY;
                    mx[m][0] = fmaxf(mx[m][0], fmaxf(sc[m][j][0], sc[m][j][1]));
                    mx[m][1] = fmaxf(mx[m][1], fmaxf(sc[m][j][2], sc[m][j][3]));
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                mx[m][h] = fmaxf(mx[m][h], __shfl_xor_sync(0xffffffffu, mx[m][h], 1));
                mx[m][h] = fmaxf(mx[m][h], __shfl_xor_sync(0xffffffffu, mx[m][h], 2));
            }
        const int rb = tcount & 1;
        if (t4 == 0)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                sm.red[rb][16 * m + g][warp] = mx[m][0];
                sm.red[rb][16 * m + g + 8][warp] = mx[m][1];
            }
        named_bar_sync(1, kNCW * 32);
        // lane r (< NR) combines row r's maxima over the warps, updates the
        // running max and publishes this warp's copies of the tile max and the
        // fold weights c1 = 2^(M_old - M_new), c2 = 2^(m_t - M_new)
        if (lane < NR) {
            const float4 a = *reinterpret_cast<const float4*>(&sm.red[rb][lane][0]);
            const float4 c = *reinterpret_cast<const float4*>(&sm.red[rb][lane][4]);
            const float mt =
                fmaxf(fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)), fmaxf(fmaxf(c.x, c.y), fmaxf(c.z, c.w)));
            const float Mn = fmaxf(Mref, mt);
            sm.wst[warp][0][lane] = mt;
            sm.wfold[tcount & 1][warp][0][lane] = ex2(Mref - Mn);
            sm.wfold[tcount & 1][warp][1][lane] = ex2(mt - Mn);
            Mref = Mn;
        }
        __syncwarp();
        // the previous tile's MM2 ran while this tile's maxima were found
        if (pend >= 0) fold(pend, pvalid);

        // ---- P = 2^(x - tile max), row sums, P8 = E4M3(448 P) as the MM2 operand ----
        float ls[MT][2];
#pragma unroll
        for (int m = 0; m < MT; ++m) ls[m][0] = ls[m][1] = 0.f;
        if (gvalid > 0) {   // the group's MMA reads this warp's codes (zeros past the end)
            const uint32_t pb = smem_u32(sm.pbuf) + static_cast<uint32_t>(wblk * NR * 128);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float mt0 = sm.wst[warp][0][16 * m + g], mt1 = sm.wst[warp][0][16 * m + g + 8];
                const uint32_t r0a = pb + static_cast<uint32_t>((16 * m + g) * 128);
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const float e0 = ex2(sc[m][j][0] - mt0), e1 = ex2(sc[m][j][1] - mt0);
                    const float e2 = ex2(sc[m][j][2] - mt1), e3 = ex2(sc[m][j][3] - mt1);
                    ls[m][0] += e0 + e1;
                    ls[m][1] += e2 + e3;
                    const int tb = tok0 + 8 * j + 2 * t4;   // token within the block
                    const uint32_t off = static_cast<uint32_t>((((tb >> 4) ^ g) << 4) | (tb & 15));
                    st_shared_u16(r0a + off, e4m3x2(448.f * e0, 448.f * e1));
                    st_shared_u16(r0a + 8 * 128 + off, e4m3x2(448.f * e2, 448.f * e3));
                }
            }
        }
        // ---- MM2: O^T[chan][row] = V^T[chan][tok] . P8^T[tok][row] over this
        // group's tokens, into the group's own accumulator. V rows of tokens
        // past the sequence end are zeroed first: P is 0 there, and a stale
        // NaN code times 0 would still be NaN. ----
        if (hasblk) {
            const int vu = (vpos + wblk) / NV, vsl = NK + (vpos + wblk) % NV;
            const uint32_t vpar = static_cast<uint32_t>(vu >> 1) & 1u;
            if (gvalid > 0 && wvalid < TPW) {
                mbar_wait(&sm.full_bar[vsl][vu & 1], vpar, p.err, 32, &sm.abort);
                for (int rr = wvalid + lane; rr < TPW; rr += 32) {
                    uint4* vr = reinterpret_cast<uint4*>(sm.ring[vsl] + (tok0 + rr) * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c) vr[c] = make_uint4(0, 0, 0, 0);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if constexpr (PAIRS) named_bar_sync(3 + (warp >> 1), 64);   // both warps' P8 and zeroed rows
            if (issuer && lane == 0) {
                mbar_wait(&sm.full_bar[vsl][vu & 1], vpar, p.err, 32, &sm.abort);
                if (gvalid > 0) {
                    tc_fence_after();
                    const uint64_t vd = smem_desc(smem_u32(sm.ring[vsl]), 1024, 1024, kSmem128BSwizzle);
                    const uint64_t pd = smem_desc(smem_u32(sm.pbuf) + static_cast<uint32_t>(wblk * NR * 128), 16,
                                                  1024, kSmem128BSwizzle);
                    const uint32_t d = tmem + static_cast<uint32_t>(((tcount & 1) * OCW + grp) * NR);
                    const int gt0 = (grp * GT) % kBS;   // the group's first token within the block
#pragma unroll
                    for (int s = 0; s < MMS; ++s) {
                        if (grp * GT + 32 * s >= valid) break;
                        const int tk = gt0 + 32 * s;
                        umma_e4m3(d, vd + static_cast<uint64_t>(tk * 8), pd + static_cast<uint64_t>(tk >> 4),
                                  kIdescO, s > 0 ? 1u : 0u);
                    }
                    umma_commit(&sm.empty_bar[vsl]);
                    umma_commit(&sm.o_full);
                } else {
                    // nothing valid in this group: release the slot once its copy landed
                    mbar_arrive(&sm.empty_bar[vsl]);
                    mbar_arrive(&sm.o_full);
                }
            }
            __syncwarp();
        } else if (issuer && lane == 0) {
            mbar_arrive(&sm.o_full);
        }

        // ---- running sums; this tile's O^T is folded with the next tile ----
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = 16 * m + 8 * h + g;
                Lp[m][h] = Lp[m][h] * sm.wfold[tcount & 1][warp][0][r] + ls[m][h] * sm.wfold[tcount & 1][warp][1][r];
            }
        pend = tcount;
        pvalid = valid;
        kpos += nb;
        vpos += nb;
        ++tcount;

        if (t == T - 1 || pos_eq(nx, end)) {
            // ------------------------------ unit end ------------------------------
            fold(pend, pvalid);
            pend = -1;
            // row sums: over the lane quad, then over the warps
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float v = Lp[m][h];
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    if (t4 == 0) sm.redl[warp][16 * m + 8 * h + g] = v;
                }
            named_bar_sync(1, kNCW * 32);
            float L = 0.f;
            if (lane < NR) {
#pragma unroll
                for (int w = 0; w < kNCW; ++w) L += sm.redl[w][lane];
                sm.wst[warp][1][lane] = L;
            }
            __syncwarp();
            const int ch = 32 * q4 + lane;
            const float vs = sm.vsc[hs][ch] * (1.0f / 448.0f);
            const int64_t u = static_cast<int64_t>(b) * W + x.i;
            const bool first_unit = b == start.b && x.i == start.i;
            const bool last_unit = b == end.b && x.i == end.i;
            const int cf = first_unit ? sm.owner[0] : cta;
            const int cl = last_unit ? sm.owner[1] : cta;
            if (cf == cl) {
                // BF16 rows staged in shared memory, then written 16 bytes per thread
                __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(sm.pbuf);
#pragma unroll
                for (int k = 0; k < HR; ++k) {
                    const int rr = hh * HR + k;
                    stage[rr * kD + ch] = __float2bfloat16_rn(Oa[k] * vs * (1.0f / sm.wst[warp][1][rr]));
                }
                named_bar_sync(1, kNCW * 32);
                const int64_t* orow = sm.orow[(hcount - 1) & 1];
#pragma unroll
                for (int it = 0; it < NR * 16 / (kNCW * 32); ++it) {
                    const int item = it * kNCW * 32 + tid;
                    const int rr = item >> 4, c8 = (item & 15) * 8;
                    if (rr < nrows)
                        *reinterpret_cast<uint4*>(p.out + orow[rr] * kD + c8) =
                            *reinterpret_cast<const uint4*>(stage + rr * kD + c8);
                }
                named_bar_sync(1, kNCW * 32);   // staging free before the next tile's P8
            }
            // A split unit's first CTA holds the range's last unit: it merges,
            // normally without publishing its own part
            const bool merger = cf != cl && cta == cf;
            auto write_part = [&]() {
                float* part = p.part + (u + cta) * kPartFloats;
#pragma unroll
                for (int k = 0; k < HR; ++k) part[(hh * HR + k) * kD + ch] = Oa[k] * vs;
                if (warp == 0 && lane < NR) {
                    part[32 * kD + lane] = Mref;
                    part[32 * kD + 32 + lane] = L;
                }
            };
            if (cf != cl && !merger) write_part();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.hdr_empty[hs]);
            // rows of the unit combined from its parts (own: this CTA's part in
            // shared memory when non-null, else every part from the workspace)
            auto merge = [&](const float* own) {
                const int n = cl - cf + 1;
                for (int item = tid; item < NR * 16; item += kNCW * 32) {
                    const int orow = item >> 4, d0 = (item & 15) * 8;
                    const int r = rc * NR + orow;
                    if (orow >= nrows) continue;
                    // one pass over the parts, four at a time with every load
                    // issued first, rescaling to the running maximum
                    float mxv = -INFINITY, lsm = 0.f;
                    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    int kfirst = 0;
                    if (own != nullptr) {
                        mxv = own[32 * kD + orow];
                        lsm = own[32 * kD + 32 + orow];
                        const float4 a = *reinterpret_cast<const float4*>(own + orow * kD + d0);
                        const float4 c = *reinterpret_cast<const float4*>(own + orow * kD + d0 + 4);
                        acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
                        acc[4] = c.x; acc[5] = c.y; acc[6] = c.z; acc[7] = c.w;
                        kfirst = 1;
                    }
                    for (int k0 = kfirst; k0 < n; k0 += 4) {
                        float mk[4], lk[4];
                        float4 oa[4], ob[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if (k0 + q < n) {
                                const float* pp = p.part + (u + cf + k0 + q) * kPartFloats;
                                mk[q] = __ldcg(pp + 32 * kD + orow);
                                lk[q] = __ldcg(pp + 32 * kD + 32 + orow);
                                oa[q] = __ldcg(reinterpret_cast<const float4*>(pp + orow * kD + d0));
                                ob[q] = __ldcg(reinterpret_cast<const float4*>(pp + orow * kD + d0 + 4));
                            } else {
                                mk[q] = -INFINITY;
                                lk[q] = 0.f;
                                oa[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                                ob[q] = oa[q];
                            }
                        }
                        const float mn = fmaxf(fmaxf(mxv, fmaxf(mk[0], mk[1])), fmaxf(mk[2], mk[3]));
                        const float c = ex2(mxv - mn);
                        lsm *= c;
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[e] *= c;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float scq = ex2(mk[q] - mn);
                            lsm += lk[q] * scq;
                            acc[0] += oa[q].x * scq;
                            acc[1] += oa[q].y * scq;
                            acc[2] += oa[q].z * scq;
                            acc[3] += oa[q].w * scq;
                            acc[4] += ob[q].x * scq;
                            acc[5] += ob[q].y * scq;
                            acc[6] += ob[q].z * scq;
                            acc[7] += ob[q].w * scq;
                        }
                        mxv = mn;
                    }
                    uint4 o;
                    o.x = pack_bf16x2(__fdiv_rn(acc[0], lsm), __fdiv_rn(acc[1], lsm));
                    o.y = pack_bf16x2(__fdiv_rn(acc[2], lsm), __fdiv_rn(acc[3], lsm));
                    o.z = pack_bf16x2(__fdiv_rn(acc[4], lsm), __fdiv_rn(acc[5], lsm));
                    o.w = pack_bf16x2(__fdiv_rn(acc[6], lsm), __fdiv_rn(acc[7], lsm));
                    *reinterpret_cast<uint4*>(p.out + q_row(p, b, n2, r) * kD + d0) = o;
                }
            };
            if (cf != cl) {
                bool done = false;
                if (merger) {
                    // the other parts are normally complete by now (their CTAs
                    // reach them at the start of their ranges): an acquire load
                    // of their count, bounded so that a part whose CTA is not
                    // running yet cannot hold this one
                    if (tid == 0) {
                        const int want = cl - cf;
                        int ok = 0;
                        const uint64_t t0 = globaltimer_ns();
                        for (;;) {
                            int v;
                            asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p.counters + u) : "memory");
                            if (v == want) {
                                ok = 1;
                                break;
                            }
                            if (globaltimer_ns() - t0 > kMergeWaitNs) break;
                            __nanosleep(64);
                        }
                        if (ok) p.counters[u] = 0;
                        sm.flag = ok;
                    }
                    named_bar_sync(1, kNCW * 32);
                    done = sm.flag != 0;
                    if (done) {
                        // this CTA's part staged in the ring (its last tile's
                        // loads and MMAs are complete)
                        float* own = reinterpret_cast<float*>(sm.ring[0]);
#pragma unroll
                        for (int k = 0; k < HR; ++k) own[(hh * HR + k) * kD + ch] = Oa[k] * vs;
                        if (warp == 0 && lane < NR) {
                            own[32 * kD + lane] = Mref;
                            own[32 * kD + 32 + lane] = L;
                        }
                        named_bar_sync(1, kNCW * 32);
                        merge(own);
                    } else {
                        write_part();
                    }
                }
                if (!done) {
                    // every consumer thread's partial stores precede the barrier; one
                    // thread then releases them with the count (and acquires the
                    // other parts when it is the last to arrive)
                    named_bar_sync(1, kNCW * 32);
                    if (tid == 0) {
                        int old;
                        asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;"
                                     : "=r"(old)
                                     : "l"(p.counters + u)
                                     : "memory");
                        const int last = (old == cl - cf);
                        if (last) p.counters[u] = 0;
                        sm.flag = last;
                    }
                    named_bar_sync(1, kNCW * 32);
                    if (sm.flag) merge(nullptr);
                }
            }
        }
        x = nx;
    }
    // every MMA issued by this warp has completed before the tensor memory is
    // released (normally already true: each unit end folds its last tile)
    if (lane == 0) {
        umma_commit(&sm.done_bar);
        mbar_wait_drain(&sm.done_bar, 0, p.err, 1024);
    }
    __syncwarp();
    tc_fence_before();
    named_bar_sync(1, kNCW * 32);
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TCOLS);
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
    // L2 promotion to 128 bytes, the row size: with PA_BSND a row is one head's
    // 128 bytes of a token, and a larger promotion would also fetch the next
    // head's bytes, which another CTA reads at another time
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    PA_REQUIRE(r == CUDA_SUCCESS, PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return PA_OK;
}

struct Plan {
    int S2T, NR, NRC, R, G, grid;
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
    PA_REQUIRE(pl->S2T == 128 || pl->S2T == 256 || pl->S2T == 512 || pl->S2T == 1024, PA_ERR_UNSUPPORTED,
               "pa_fp8_decode: s2_tile %d (128, 256, 512 and 1024 are built)", pl->S2T);
    PA_REQUIRE(!cfg || (cfg->overlap_prologue >= 0 && cfg->overlap_prologue <= 2), PA_ERR_INVALID,
               "pa_fp8_decode: overlap_prologue %d (0, 1 or 2)", cfg ? cfg->overlap_prologue : 0);
    pl->G = NQ / NKV;
    pl->R = S1 * pl->G;
    pl->NR = pl->R <= 16 ? 16 : 32;
    // 1024-token tiles: each consumer warp holds the scores of 128 tokens for
    // every query row of the unit in registers; 16 rows fit, 32 do not
    PA_REQUIRE(pl->S2T < 1024 || pl->NR == 16, PA_ERR_UNSUPPORTED,
               "pa_fp8_decode: s2_tile 1024 needs at most 16 query rows per kv head (S1 x group = %d)", pl->R);
    pl->NRC = (pl->R + pl->NR - 1) / pl->NR;
    pl->U = static_cast<int64_t>(B) * NKV * pl->NRC;
    int grid = (cfg && cfg->num_ctas > 0) ? cfg->num_ctas : device_sm_count();
    PA_REQUIRE(grid > 0, PA_ERR_CUDA, "pa_fp8_decode: cannot query the device");
    pl->grid = grid;
    pl->counters_bytes = round256(static_cast<size_t>(pl->U) * sizeof(int));
    pl->part_bytes = static_cast<size_t>(pl->U + grid) * kPartFloats * sizeof(float);
    pl->total = kWsHeader + pl->counters_bytes + pl->part_bytes;
    return PA_OK;
}

template <int NR, int S2T>
pa_status launch(const CUtensorMap& tk, const CUtensorMap& tv,
                 const DecodeParams& prm, cudaStream_t st)
{
    const size_t smem = sizeof(DecodeSmem<NR, S2T>) + 1024;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    static int nregs = 0;
    std::call_once(once, [&] {
        attr = cudaFuncSetAttribute(decode_kernel<NR, S2T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem));
        cudaFuncAttributes fa;
        if (attr == cudaSuccess) attr = cudaFuncGetAttributes(&fa, decode_kernel<NR, S2T>);
        if (attr == cudaSuccess) nregs = fa.numRegs;
    });
    PA_REQUIRE(attr == cudaSuccess, PA_ERR_CUDA, "pa_fp8_decode: kernel attributes: %s", cudaGetErrorString(attr));
    // The consumers' setmaxnreg.inc takes registers the producers gave back;
    // it could only wait forever if the launch held fewer than the split needs.
    PA_REQUIRE(nregs * (kThreads / 32) >= kNCW * kConsRegs + 4 * kProdRegs, PA_ERR_CUDA,
               "pa_fp8_decode: kernel built with %d registers per thread, below the register split", nregs);
    if (prm.overlap) {
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(static_cast<unsigned>(prm.grid));
        lc.blockDim = dim3(kThreads);
        lc.dynamicSmemBytes = smem;
        lc.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        lc.attrs = at;
        lc.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&lc, decode_kernel<NR, S2T>, tk, tv, prm);
        PA_REQUIRE(e == cudaSuccess, PA_ERR_CUDA, "pa_fp8_decode: launch: %s", cudaGetErrorString(e));
        return PA_OK;
    }
    decode_kernel<NR, S2T><<<prm.grid, kThreads, smem, st>>>(tk, tv, prm);
    return check_launch("pa_fp8_decode");
}

// Bulk-copy / TMA destinations must be 16-byte aligned; the 128-byte-swizzled
// K/V tiles and the P8 operand sit on 1024-byte boundaries (the swizzle atom
// the ldmatrix addressing and the MMA descriptors assume).
template <int NR, int S2T>
struct SmemLayoutChecks {
    using S = DecodeSmem<NR, S2T>;
    static_assert(offsetof(S, ring) % 1024 == 0, "ring alignment");
    static_assert(offsetof(S, qb) % 16 == 0, "Q rows alignment");
    static_assert(offsetof(S, pbuf) % 1024 == 0, "P operand alignment");
    static_assert(offsetof(S, vsc) % 16 == 0, "vsc alignment");
    static_assert(offsetof(S, wst) % 16 == 0, "wst alignment");
    static_assert(sizeof(S) + 1024 <= 232448, "decode shared memory over budget");
    static constexpr bool ok = true;
};
static_assert(SmemLayoutChecks<16, 128>::ok && SmemLayoutChecks<16, 256>::ok && SmemLayoutChecks<16, 512>::ok &&
                  SmemLayoutChecks<16, 1024>::ok &&
                  SmemLayoutChecks<32, 128>::ok && SmemLayoutChecks<32, 256>::ok && SmemLayoutChecks<32, 512>::ok,
              "shared memory layout");

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
                   aligned(k_scale, 4) && aligned(out, 16),
               PA_ERR_INVALID,
               "pa_fp8_decode: misaligned pointer (q, caches, v_scale and out need 16 bytes, k_scale 4)");
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
    prm.overlap = cfg ? cfg->overlap_prologue : 0;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pl.NR == 16) {
        if (pl.S2T == 128) return launch<16, 128>(tk, tv, prm, s);
        if (pl.S2T == 256) return launch<16, 256>(tk, tv, prm, s);
        if (pl.S2T == 512) return launch<16, 512>(tk, tv, prm, s);
        return launch<16, 1024>(tk, tv, prm, s);
    }
    if (pl.S2T == 128) return launch<32, 128>(tk, tv, prm, s);
    if (pl.S2T == 256) return launch<32, 256>(tk, tv, prm, s);
    return launch<32, 512>(tk, tv, prm, s);
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
