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
//  * Warp 10 owns the tensor memory and issues MM1 from one thread
//    (tcgen05.mma kind::f8f6f4, E4M3 x E4M3 -> F32, M = 128):
//      MM1  S^T[token][row]   = K_blk (K-major, the ring slot as loaded)
//                               x Q^T (K-major, 128-byte swizzled rows)
//    S^T lives in tensor memory, up to 4 tiles ahead of the consumers.
//  * Warps 0-7 consume: tcgen05.ld of S^T (a lane = a token, a column = a
//    query row), scaling by q_scale * k_scale (each thread loads its token's
//    key scales a tile ahead), masking past kv_act_seqs, the tile's row
//    maxima (butterfly over lanes, then over warps through shared memory),
//    P = 2^(x - tile max), the row sums, E4M3 P8 = 448 * P written as the
//    MM2 operand; each warp then issues the MM2 k-step of its own tokens:
//      MM2  O^T[chan][row]   += V_blk^T (MN-major: the V ring slot)
//                               x P8^T (MN-major)
//    O^T is double-buffered by tile parity and folded into registers with the
//    running-max rescale while the next tile's maxima are found. Quantising
//    against the tile's own maximum gives the same codes as quantising
//    exp(S - running max) against its tile maximum (the ratio cancels the
//    running max); the running max only weights whole tiles.
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
constexpr int kKProducerWarp = kNCW;        // K blocks, key scales, per-unit header
constexpr int kVProducerWarp = kNCW + 1;    // V blocks
constexpr int kMmaWarp = kNCW + 2;          // tensor memory owner; issues MM1
constexpr int kThreads = (kNCW + 3) * 32;
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

// S^T buffers in tensor memory (MM1 may run that many tiles ahead of the
// consumers): as many as fit next to O^T in the 512 columns, at most 4.
__host__ __device__ constexpr int s_buffers(int sc, int nr)
{
    return (4 * sc + 2 * nr <= 512) ? 4 : ((3 * sc + 2 * nr <= 512) ? 3 : 2);
}

struct Pos {
    int b, i, t;
};

// NR: padded query rows per unit (16 or 32, the MMA N); S2T: s2 tile; NS:
// ring slots (as many as fit): slots 0 .. kKSlots-1 hold K blocks, the rest
// V blocks, each ring with its own producer.
template <int NR, int S2T, int NS>
struct __align__(1024) DecodeSmemT {
    static constexpr int NSLOT = NS;
    alignas(1024) uint8_t ring[NS][kSlotBytes];
    // Q rows: bulk-copied as plain rows, then swizzled in place into the
    // 128-byte-swizzled K-major operand layout
    alignas(1024) uint8_t qb[2][NR][kD];
    // P8^T, MN-major without swizzle: token t, row r at
    // (t / 8) * 8 * NR + (r / 16) * 128 + (t % 8) * 16 + r % 16
    // (also the BF16 staging of a unit's output rows, NR x 128 x 2 bytes)
    alignas(1024) uint8_t pbuf[S2T * NR > NR * kD * 2 ? S2T * NR : NR * kD * 2];
    // key scales of one tile's blocks, double-buffered by tile parity
    alignas(16) float vsc[2][kD];
    alignas(16) float qs[2][32];
    alignas(16) float red[2][32][kNCW];   // per-warp row maxima (row-major), double-buffered by tile
    float redl[kNCW][32];       // per-warp row sums at unit end
    alignas(16) float wst[kNCW][4][32];   // per-warp copies of row values
    alignas(16) float wfold[2][kNCW][2][32];   // per-warp fold weights c1, c2 by tile parity
    int scan[kThreads / 32];
    int bpre[kMaxB + 1];
    int slen[kMaxB];
    uint64_t full_bar[NS];
    uint64_t empty_bar[NS];
    uint64_t hdr_full[2];
    uint64_t hdr_empty[2];
    uint64_t s_full[4];
    uint64_t s_empty[4];
    uint64_t o_full;
    uint64_t done_bar;
    uint64_t cdrain;            // every consumer warp's MMAs complete (before tensor memory is freed)
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
    int64_t merge_wait_ns;   // the merging CTA's wait for the other parts (< 0: none)
    uint64_t wait_ns;        // limit of the bounded waits
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

// Butterfly sum over the 32 lanes of a warp of N per-lane values (one per
// query row): on return lane L holds the sum of row (N == 16 ? L / 2 : L)
// over all lanes. `a` is clobbered.
template <int N>
__device__ __forceinline__ float lane_sum(float (&a)[N], int lane)
{
#pragma unroll
    for (int s = 0; s < 5; ++s) {
        const int h = N >> (s + 1);
        if (h == 0) break;
        const int o = 16 >> s;
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float keep = up ? a[i + h] : a[i];
            const float send = up ? a[i] : a[i + h];
            a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float v = a[0];
    if (N == 16) v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v;
}

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float* v)
{
    if constexpr (N == 8) {
        tmem_ld8(taddr, v);
    } else {
#pragma unroll
        for (int c = 0; c + 16 <= N; c += 16) tmem_ld16(taddr + c, v + c);
        if constexpr (N % 16 == 8) tmem_ld8(taddr + N - 8, v + N - 8);
    }
}

// Slot and phase parity of the j-th block (j < NBT) after (slot, ph) in a ring
// of NSLOT; a ring that holds a tile wraps at most once.
template <int NSLOT, int NBT>
__device__ __forceinline__ int ring_slot(int slot, uint32_t ph, int j, uint32_t* par)
{
    if constexpr (NBT <= NSLOT) {
        int s = slot + j;
        *par = ph;
        if (s >= NSLOT) {
            s -= NSLOT;
            *par ^= 1u;
        }
        return s;
    } else {
        const int k = slot + j;
        *par = ph ^ static_cast<uint32_t>((k / NSLOT) & 1);
        return k % NSLOT;
    }
}

// Advance (slot, ph) by n <= NBT blocks in a ring of NSLOT.
template <int NSLOT, int NBT>
__device__ __forceinline__ void ring_advance(int& slot, uint32_t& ph, int n)
{
    slot += n;
    if constexpr (NBT <= NSLOT) {
        if (slot >= NSLOT) {
            slot -= NSLOT;
            ph ^= 1u;
        }
    } else {
        ph ^= static_cast<uint32_t>((slot / NSLOT) & 1);
        slot %= NSLOT;
    }
}

// NRV: the query rows of a chunk that are computed (a multiple of 4, at most
// NR); rows NRV..NR-1 are MMA padding whose scores, exponentials and P codes
// are skipped (only used where every chunk has exactly NRV rows: 12 or 24).
template <int NR, int S2T, int NRV = NR>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecodeParams p)
{
    static_assert(NRV % 4 == 0 && NRV <= NR, "computed rows");
    constexpr int NBT = S2T / kBS;               // 128-token blocks (MMA M-blocks) per tile
    constexpr int MBW = NBT >= 2 ? NBT / 2 : 1;  // blocks per consumer warp
    constexpr int SC = NBT * NR;                 // tensor-memory columns of one S^T buffer
    constexpr int NSB = s_buffers(SC, NR);       // S^T buffers
    constexpr int OCOL = NSB * SC;               // first column of O^T (two buffers of NR columns)
    constexpr uint32_t TCOLS = tmem_cols(NSB * SC + 2 * NR);
    constexpr int HR = NR / 2;                   // O^T columns (query rows) per consumer warp
    constexpr int TC = S2T + kC0;
    constexpr int NSLOT = DecodeSmem<NR, S2T>::NSLOT;
    // K ring: one tile up to s2 tile 512; with longer tiles the V ring takes a
    // whole tile (MM2 needs every block of the tile) and K the rest
    constexpr int NK = NBT <= kKSlots ? kKSlots : NSLOT - NBT, NV = NSLOT - NK;
    static_assert(NV >= NBT, "the V ring must hold one tile");
    static_assert(NK >= 1, "no K ring slot left");

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
            mbar_init(&sm.full_bar[i], 1);
            // the MMAs reading the slot completed: K blocks are read by the MM1
            // thread, V blocks by one MMA of each of the 4 consumer warps that
            // hold the block's tokens
            mbar_init(&sm.empty_bar[i], i < NK ? 1 : 4);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.hdr_full[i], 2);           // byte-counted copies + the q_scale cp.async
            mbar_init(&sm.hdr_empty[i], 1 + kNCW);   // last MM1 of the unit + every consumer warp
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&sm.s_full[i], 1);
            mbar_init(&sm.s_empty[i], kNCW);
        }
        mbar_init(&sm.o_full, kNCW);                 // every consumer warp's MM2 share
        mbar_init(&sm.done_bar, 1);
        mbar_init(&sm.cdrain, kNCW);
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

    // tensor memory: allocated by the MMA warp, address published in shared memory
    if (warp == kMmaWarp) tmem_alloc(&sm.tmem, TCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem;
    const Pos start = sm.range[0];
    const Pos end = sm.range[1];

    if (warp == kKProducerWarp || warp == kVProducerWarp) {
        // ============================== producers ==============================
        // The K producer fills the K ring (plus key scales and the per-unit
        // header), the V producer the V ring; each runs ahead of the MMAs as
        // far as its own ring allows, so V tiles waiting for their P never
        // hold back the next tile's K.
        if (lane != 0) return;
        const bool isK = warp == kKProducerWarp;
        const CUtensorMap* tm = isK ? &tmK : &tmV;
        asm volatile("prefetch.tensormap [%0];" ::"l"(tm) : "memory");
        const uint64_t pol = l2_evict_first_policy();
        const int base = isK ? 0 : NK, nring = isK ? NK : NV;
        int slot = 0;
        uint32_t ph = 0;
        int hcount = 0, fills = 0, tcount = 0;
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
        // After a wait that gave up nothing more is issued (no copy may land in
        // a slot whose previous copy or MMA is still running, and no barrier
        // may see more arrivals than its count); the loop ends.
        bool stop = false;
        auto issue_header = [&](int b, int n2, int rc) {
            const int hs = hcount & 1;
            if (!mbar_wait(&sm.hdr_empty[hs], ((hcount >> 1) & 1) ^ 1, p.err, 2, &sm.abort, p.wait_ns)) {
                stop = true;
                return;
            }
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
        for (Pos x = start; !pos_eq(x, end) && !stop;) {
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
            // tile's later K blocks wait for MM1 on its first ones, so the
            // header goes out before them
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
                        if (globaltimer_ns() - t0 > p.wait_ns) {
                            *ab = 1;
                            atomicOr(p.err, 2048);
                            break;
                        }
                    }
                    if (*ab) break;
                }
            }
#pragma unroll
            for (int j = 0; j < NBT; ++j) {
                if (j >= nb) break;
                const int sl = base + slot;
                if (!waited && t * S2T + (j + 1) * kBS > len - p.S1) {
                    grid_dependency_wait();
                    waited = true;
                }
                if (!mbar_wait(&sm.empty_bar[sl], ph ^ 1, p.err, 4, &sm.abort, p.wait_ns)) {
                    stop = true;
                    break;
                }
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
                mbar_arrive_expect_tx(&sm.full_bar[sl], kSlotBytes);
                tma_load_2d(sm.ring[sl], tm, x0, y0, &sm.full_bar[sl], pol);
                ++fills;
                if (++slot == nring) {
                    slot = 0;
                    ph ^= 1;
                }
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
            const int n = fills / nring + (s < fills % nring ? 1 : 0);
            if (n > 0) mbar_wait_drain(&sm.full_bar[base + s], static_cast<uint32_t>(n - 1) & 1u, p.err, 1024);
        }
        if (isK) {
            for (int h = 0; h < 2; ++h) {
                const int n = hcount / 2 + (h < hcount % 2 ? 1 : 0);
                if (n > 0) mbar_wait_drain(&sm.hdr_full[h], static_cast<uint32_t>(n - 1) & 1u, p.err, 1024);
            }
        }
        return;
    }

    if (warp == kMmaWarp) {
        // ============================== MM1 issue ==============================
        // One thread issues MM1 as soon as a K block lands (up to NSB tiles
        // ahead of the consumers). MM2 is issued by the consumer warps.
        constexpr uint32_t kIdescS = idesc_e4m3(128, NR, 0, 0);   // K-major K and Q
        constexpr bool mm1 = true;
        int slot = 0;
        uint32_t ph = 0;
        int hcount = 0, tcount = 0, hs = 0;
        bool first = true;
        for (Pos x = start; !pos_eq(x, end);) {
            const Pos nx = pos_next<S2T>(sm.slen, sm.bpre, p.B, x, W);
            const int rc = x.i - head_of(p, x.i) * p.NRC, t = x.t;
            const int len = sm.slen[x.b];
            const int valid = min(S2T, len - t * S2T);
            const int nb = (valid + kBS - 1) / kBS;
            if (mm1) {
                if (first || t == 0) {
                    hs = hcount & 1;
                    mbar_wait(&sm.hdr_full[hs], (hcount >> 1) & 1, p.err, 8, &sm.abort, p.wait_ns);
                    // Q rows into the 128-byte-swizzled K-major layout (16-byte
                    // chunk c of row r goes to position c ^ (r % 8)); rows past
                    // the chunk's end become zeros
                    if (lane < NR) {
                        const int nrows = min(p.R - rc * NR, NR);
                        uint4* row = reinterpret_cast<uint4*>(&sm.qb[hs][lane][0]);
                        uint4 v[8];
#pragma unroll
                        for (int c = 0; c < 8; ++c) v[c] = lane < nrows ? row[c] : make_uint4(0, 0, 0, 0);
#pragma unroll
                        for (int c = 0; c < 8; ++c) row[c ^ (lane & 7)] = v[c];
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    ++hcount;
                }
                const int sb = tcount % NSB;
                if (lane == 0 && !*reinterpret_cast<volatile int*>(&sm.abort)) {
                    // MM1: S^T[token][row] for each block of the tile (nothing
                    // is issued after a wait gave up)
                    bool ok = mbar_wait(&sm.s_empty[sb], ((tcount / NSB) & 1) ^ 1, p.err, 64, &sm.abort, p.wait_ns);
                    tc_fence_after();
                    const uint64_t qd = smem_desc(smem_u32(&sm.qb[hs][0][0]), 16, 1024, kSmem128BSwizzle);
                    for (int j = 0; j < nb && ok; ++j) {
                        uint32_t par;
                        const int s = ring_slot<NK, NBT>(slot, ph, j, &par);
                        if (!mbar_wait(&sm.full_bar[s], par, p.err, 16, &sm.abort, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t kd = smem_desc(smem_u32(sm.ring[s]), 16, 1024, kSmem128BSwizzle);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)   // 32 bytes of head dim per MMA
                            umma_e4m3(tmem + sb * SC + j * NR, kd + 2 * kk, qd + 2 * kk, kIdescS, kk);
                        umma_commit(&sm.empty_bar[s]);
                    }
                    if (ok) {
                        umma_commit(&sm.s_full[sb]);
                        if (t == tiles_of<S2T>(len) - 1 || pos_eq(nx, end)) umma_commit(&sm.hdr_empty[hs]);
                    }
                }
                __syncwarp();
                if (__shfl_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&sm.abort), 0)) break;
                ring_advance<NK, NBT>(slot, ph, nb);
            }
            first = false;
            ++tcount;
            x = nx;
        }
        // all MMAs complete before the tensor memory is released
        if (lane == 0) {
            umma_commit(&sm.done_bar);
            mbar_wait_drain(&sm.done_bar, 0, p.err, 1024);
        }
        __syncwarp();
        named_bar_sync(2, (kNCW + 1) * 32);
        tc_fence_after();
        tmem_dealloc(tmem, TCOLS);
        return;
    }

    // ================================ consumers ================================
    // Warp w reads tensor-memory lanes 32 (w % 4) .. +31: tokens of its blocks
    // (S^T) and channels (O^T). Warps 0-3 take the first half of the tile's
    // blocks and O^T rows 0 .. NR/2-1, warps 4-7 the rest.
    const int q4 = warp & 3, hh = warp >> 2;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    const int rho = NR == 16 ? (lane >> 1) : lane;   // query row whose reductions this lane holds
    const bool rep = NR == 32 || (lane & 1) == 0;    // lane that publishes row rho

    int vslot = 0;
    uint32_t vph = 0;
    int hcount = 0, tcount = 0, hs = 0, nrows = 0;
    bool first = true;
    // Row sums (running-max units). 16 rows: this thread's share of every row,
    // reduced over the lanes at unit end. 32 rows: reduced over the lanes
    // every tile into one value per lane (row rho), which frees the registers
    // that let a 24-row unit keep its scores across the row-maximum barrier.
    constexpr bool kRowSumPerTile = NR == 32;
    float Lp[kRowSumPerTile ? 1 : NR];
    float Lr = 0.f;
    float Oa[HR];               // O^T[32 q4 + lane][hh * HR + k], times 448
    float Mref = -INFINITY;     // running max of row rho (scaled log2 units)
#pragma unroll
    for (int r = 0; r < (kRowSumPerTile ? 1 : NR); ++r) Lp[r] = 0.f;
#pragma unroll
    for (int k = 0; k < HR; ++k) Oa[k] = 0.f;
    {
        // O^T starts at zero: every MM2 MMA accumulates
        const float zero8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < HR; c += 8) {
            tmem_st8(tl + OCOL + hh * HR + c, zero8);
            tmem_st8(tl + OCOL + NR + hh * HR + c, zero8);
        }
        tmem_wait_st();
        tc_fence_before();
    }
    // Tile k's O^T (buffer k & 1) folded into Oa once its MM2 has completed,
    // with the weights of tile k, then zeroed for tile k + 2.
    auto fold = [&](int k) {
        mbar_wait(&sm.o_full, k & 1, p.err, 512, &sm.abort, p.wait_ns);
        tc_fence_after();
        float ot[HR];
        tmem_ld_cols<HR>(tl + OCOL + (k & 1) * NR + hh * HR, ot);
        tmem_wait_ld();
#pragma unroll
        for (int c4 = 0; c4 < HR / 4; ++c4) {
            const float4 a4 = *reinterpret_cast<const float4*>(&sm.wfold[k & 1][warp][0][hh * HR + 4 * c4]);
            const float4 b4 = *reinterpret_cast<const float4*>(&sm.wfold[k & 1][warp][1][hh * HR + 4 * c4]);
            Oa[4 * c4 + 0] = Oa[4 * c4 + 0] * a4.x + ot[4 * c4 + 0] * b4.x;
            Oa[4 * c4 + 1] = Oa[4 * c4 + 1] * a4.y + ot[4 * c4 + 1] * b4.y;
            Oa[4 * c4 + 2] = Oa[4 * c4 + 2] * a4.z + ot[4 * c4 + 2] * b4.z;
            Oa[4 * c4 + 3] = Oa[4 * c4 + 3] * a4.w + ot[4 * c4 + 3] * b4.w;
        }
        // zeroed for the MMAs of tile k + 2, which come after that tile's
        // row-maximum barrier
        const float zero8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < HR; c += 8) tmem_st8(tl + OCOL + (k & 1) * NR + hh * HR + c, zero8);
        tmem_wait_st();
        tc_fence_before();
    };
    int pend = -1;   // tile whose O^T has not been folded yet
    // Key scales of this thread's token (lane) in each of its blocks, read
    // from global memory through L2 one tile ahead of their use (the block
    // ids one tile before that), so that the loads are in flight while the
    // current tile is processed and no copy engine or shared memory is used.
    const int ktok = 32 * q4 + lane;
    auto tile_ids = [&](const Pos& y, int (&ids)[MBW]) {
        const int nby = min(NBT, (sm.slen[y.b] - y.t * S2T + kBS - 1) / kBS);   // y.b < B here
        const int* row = p.block_table + static_cast<int64_t>(y.b) * p.max_blocks + y.t * NBT;
#pragma unroll
        for (int jj = 0; jj < MBW; ++jj) {
            const int mb = hh * MBW + jj;
            ids[jj] = mb < nby ? __ldg(row + mb) : -1;
        }
    };
    auto tile_ks = [&](const Pos& y, const int (&ids)[MBW], float (&dst)[MBW]) {
        const int n2y = head_of(p, y.i);
#pragma unroll
        for (int jj = 0; jj < MBW; ++jj) {
            int blk = ids[jj];
            if (blk < 0 || blk >= p.num_blocks) blk = 0;
            const int64_t idx = p.layout == PA_LAYOUT_BSND
                                    ? (static_cast<int64_t>(blk) * kBS + ktok) * p.NKV + n2y
                                    : (static_cast<int64_t>(blk) * p.NKV + n2y) * kBS + ktok;
            dst[jj] = __ldcg(p.k_scale + idx);
        }
    };
    float ksn[MBW];   // key scales of the next tile
    int idn[MBW];     // block ids of the tile after it
#pragma unroll
    for (int jj = 0; jj < MBW; ++jj) {
        ksn[jj] = 0.f;
        idn[jj] = -1;
    }
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
    int id0[MBW];
    if (!pos_eq(start, end)) {
        tile_ids(start, id0);
        if (!pos_eq(x1, end)) tile_ids(x1, idn);
    }
    grid_dependency_wait();
    if (!pos_eq(start, end)) tile_ks(start, id0, ksn);
    // sequences of length 0 produce zero rows (no tile ever covers them)
    for (int b = cta; b < p.B; b += p.grid)
        if (sm.slen[b] == 0) zero_rows(p, b, tid, kNCW * 32);

    for (Pos x = start; !pos_eq(x, end);) {
        const Pos nx = x1;
        const int b = x.b, n2 = head_of(p, x.i), rc = x.i - n2 * p.NRC, t = x.t;
        const int len = lenx;
        const int T = tiles_of<S2T>(len);

        if (first || t == 0) {
            hs = hcount & 1;
            mbar_wait(&sm.hdr_full[hs], (hcount >> 1) & 1, p.err, 8, &sm.abort, p.wait_ns);
            nrows = min(p.R - rc * NR, NR);
            if (warp == 0 && lane < NR) sm.orow[hcount & 1][lane] = q_row(p, b, n2, rc * NR + lane);
            // this warp's copy of q_scale * softmax_scale * log2(e) per row (0
            // past the chunk's rows); the slot holds the row sums at unit end
            if (lane < NR) sm.wst[warp][3][lane] = lane < nrows ? sm.qs[hs][lane] * p.sscale : 0.f;
            __syncwarp();
#pragma unroll
            for (int r = 0; r < (kRowSumPerTile ? 1 : NR); ++r) Lp[r] = 0.f;
            Lr = 0.f;
#pragma unroll
            for (int k = 0; k < HR; ++k) Oa[k] = 0.f;
            Mref = -INFINITY;
            ++hcount;
            first = false;
        }

        const int valid = min(S2T, len - t * S2T);
        const int nb = (valid + kBS - 1) / kBS;
        const int sb = tcount % NSB;
        float ksv[MBW];
#pragma unroll
        for (int jj = 0; jj < MBW; ++jj) ksv[jj] = ksn[jj];
        if (!pos_eq(nx, end)) {
            tile_ks(nx, idn, ksn);
            if (!pos_eq(x2, end)) tile_ids(x2, idn);
        }
        // the walk moves on by one tile
        lenx = len1;
        x1 = x2;
        len1 = len2;
        if (!pos_eq(x2, end)) x2 = advance(x2, len2, len2);

        // ---- S^T of this warp's blocks and their key scales ----
        // With 32 query rows and two blocks per warp, the scores of both blocks
        // do not fit in registers next to the rest of the state (they spill):
        // each block is read from tensor memory twice instead, once for the
        // row maxima and once for P, and the S^T buffer is released after the
        // second read. With 24 computed rows they fit and are read once.
        constexpr bool kReload = NR == 32 && MBW > 1 && NRV == NR;
        constexpr int SVB = kReload ? 1 : MBW;
        mbar_wait(&sm.s_full[sb], (tcount / NSB) & 1, p.err, 256, &sm.abort, p.wait_ns);
        tc_fence_after();
        float sv[SVB][NR];
        if constexpr (!kReload) {
#pragma unroll
            for (int jj = 0; jj < MBW; ++jj) {
                const int mb = hh * MBW + jj;
                if (mb < nb) tmem_ld_cols<(NRV % 8 == 0 ? NRV : NR)>(tl + sb * SC + mb * NR, sv[jj]);
            }
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.s_empty[sb]);
        }

        // ---- scores x = S * q_scale * scale * log2(e) * k_scale; tile row maxima ----
        float mloc[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) mloc[r] = r < NRV ? -INFINITY : 0.f;   // padding rows stay finite
        if constexpr (!kReload) {
            float qsc[NR];
#pragma unroll
            for (int r4 = 0; r4 < NRV / 4; ++r4) {
                const float4 q4v = *reinterpret_cast<const float4*>(&sm.wst[warp][3][4 * r4]);
                qsc[4 * r4 + 0] = q4v.x;
                qsc[4 * r4 + 1] = q4v.y;
                qsc[4 * r4 + 2] = q4v.z;
                qsc[4 * r4 + 3] = q4v.w;
            }
#pragma unroll
            for (int jj = 0; jj < MBW; ++jj) {
                const int mb = hh * MBW + jj;
                if (mb < nb) {
                    const bool ok = mb * kBS + 32 * q4 + lane < valid;
#pragma unroll
                    for (int r = 0; r < NRV; ++r) {
                        const float xv = ok ? (sv[jj][r] * qsc[r]) * ksv[jj] : -INFINITY;
                        sv[jj][r] = xv;
                        mloc[r] = fmaxf(mloc[r], xv);
                    }
                }
            }
        } else {
#pragma unroll
            for (int jj = 0; jj < MBW; ++jj) {
                const int mb = hh * MBW + jj;
                if (mb < nb) {
                    tmem_ld_cols<NR>(tl + sb * SC + mb * NR, sv[0]);
                    tmem_wait_ld();
                    const bool ok = mb * kBS + 32 * q4 + lane < valid;
#pragma unroll
                    for (int r4 = 0; r4 < NRV / 4; ++r4) {
                        const float4 q4v = *reinterpret_cast<const float4*>(&sm.wst[warp][3][4 * r4]);
                        const float qv[4] = {q4v.x, q4v.y, q4v.z, q4v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int r = 4 * r4 + e;
                            const float xv = ok ? (sv[0][r] * qv[e]) * ksv[jj] : -INFINITY;
                            mloc[r] = fmaxf(mloc[r], xv);
                        }
                    }
                }
            }
        }
        // each row's maximum over the warp's tokens (one warp reduction per
        // computed row), kept by the lanes that hold row rho
        float wmax = 0.f;
#pragma unroll
        for (int r = 0; r < NRV; ++r) {
            const float m = warp_max_f32(mloc[r]);
            wmax = rho == r ? m : wmax;
        }
        const int rb = tcount & 1;
        if (rep) sm.red[rb][rho][warp] = wmax;
        named_bar_sync(1, kNCW * 32);
        float mt;
        {
            const float4 a = *reinterpret_cast<const float4*>(&sm.red[rb][rho][0]);
            const float4 c = *reinterpret_cast<const float4*>(&sm.red[rb][rho][4]);
            mt = fmaxf(fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)), fmaxf(fmaxf(c.x, c.y), fmaxf(c.z, c.w)));
        }
        {
            const float Mn = fmaxf(Mref, mt);
            const float c1 = ex2(Mref - Mn), c2 = ex2(mt - Mn);
            Mref = Mn;
            if (rep) {
                sm.wst[warp][0][rho] = mt;
                sm.wfold[tcount & 1][warp][0][rho] = c1;
                sm.wfold[tcount & 1][warp][1][rho] = c2;
            }
        }
        __syncwarp();
        // the previous tile's MM2 ran while this tile's maxima were found
        if (pend >= 0) fold(pend);

        // ---- P = 2^(x - tile max), row sums, P8 = E4M3(448 P) as the MM2 operand ----
        float ls[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) ls[r] = r < NRV ? 0.f : 1.f;   // padding rows: a non-zero sum
#pragma unroll
        for (int jj = 0; jj < MBW; ++jj) {
            const int mb = hh * MBW + jj;
            if (mb < nb) {
                const int tok = mb * kBS + 32 * q4 + lane;
                float* x = sv[kReload ? 0 : jj];
                if constexpr (kReload) {
                    // the same scores as in the first pass, bit for bit
                    tmem_ld_cols<NR>(tl + sb * SC + mb * NR, x);
                    tmem_wait_ld();
                    const bool ok = tok < valid;
#pragma unroll
                    for (int r4 = 0; r4 < NRV / 4; ++r4) {
                        const float4 q4v = *reinterpret_cast<const float4*>(&sm.wst[warp][3][4 * r4]);
                        x[4 * r4 + 0] = ok ? (x[4 * r4 + 0] * q4v.x) * ksv[jj] : -INFINITY;
                        x[4 * r4 + 1] = ok ? (x[4 * r4 + 1] * q4v.y) * ksv[jj] : -INFINITY;
                        x[4 * r4 + 2] = ok ? (x[4 * r4 + 2] * q4v.z) * ksv[jj] : -INFINITY;
                        x[4 * r4 + 3] = ok ? (x[4 * r4 + 3] * q4v.w) * ksv[jj] : -INFINITY;
                    }
                }
                uint32_t pk[NR / 4];
#pragma unroll
                for (int r4 = NRV / 4; r4 < NR / 4; ++r4) pk[r4] = 0u;
#pragma unroll
                for (int r4 = 0; r4 < NRV / 4; ++r4) {
                    const float4 m4 = *reinterpret_cast<const float4*>(&sm.wst[warp][0][4 * r4]);
                    const float e0 = ex2(x[4 * r4 + 0] - m4.x);
                    const float e1 = ex2(x[4 * r4 + 1] - m4.y);
                    const float e2 = ex2(x[4 * r4 + 2] - m4.z);
                    const float e3 = ex2(x[4 * r4 + 3] - m4.w);
                    ls[4 * r4 + 0] += e0;
                    ls[4 * r4 + 1] += e1;
                    ls[4 * r4 + 2] += e2;
                    ls[4 * r4 + 3] += e3;
                    pk[r4] = e4m3x4(448.f * e0, 448.f * e1, 448.f * e2, 448.f * e3);
                }
                uint8_t* dst = sm.pbuf + (tok >> 3) * (8 * NR) + (tok & 7) * 16;
#pragma unroll
                for (int a = 0; a < NR / 16; ++a)
                    *reinterpret_cast<uint4*>(dst + a * 128) =
                        make_uint4(pk[4 * a], pk[4 * a + 1], pk[4 * a + 2], pk[4 * a + 3]);
            }
        }
        if constexpr (kReload) {
            // both reads of this tile's S^T are done: MM1 may reuse the buffer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.s_empty[sb]);
        }
        // ---- this warp's share of MM2: the k-step of its 32 tokens in each of
        // its blocks, O^T[chan][row] += V^T[chan][tok] . P8^T[tok][row] (O^T
        // was zeroed when the previous tile was folded). V rows of tokens
        // past the sequence end are zeroed first: P is 0 there, and a stale
        // NaN code times 0 would still be NaN. ----
        {
            constexpr uint32_t kIdescO = idesc_e4m3(128, NR, 1, 1);   // MN-major V^T and P8^T
            int vsl[MBW];
            uint32_t vpar[MBW];
#pragma unroll
            for (int jj = 0; jj < MBW; ++jj) {
                const int mb = hh * MBW + jj;
                vsl[jj] = NK + ring_slot<NV, NBT>(vslot, vph, mb, &vpar[jj]);
                if (mb < nb && (mb + 1) * kBS > valid) {
                    mbar_wait(&sm.full_bar[vsl[jj]], vpar[jj], p.err, 32, &sm.abort, p.wait_ns);
                    const int row = 32 * q4 + lane;
                    if (mb * kBS + row >= valid) {
                        uint4* vr = reinterpret_cast<uint4*>(sm.ring[vsl[jj]] + row * 128);
#pragma unroll
                        for (int c = 0; c < 8; ++c) vr[c] = make_uint4(0, 0, 0, 0);
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const uint64_t pd = smem_desc(smem_u32(sm.pbuf), 8 * NR, 128, kSmemNoSwizzle);
                bool any = false;
#pragma unroll
                for (int jj = 0; jj < MBW; ++jj) {
                    const int mb = hh * MBW + jj;
                    if (mb < nb) {
                        mbar_wait(&sm.full_bar[vsl[jj]], vpar[jj], p.err, 32, &sm.abort, p.wait_ns);
                        tc_fence_after();
                        const uint64_t vd = smem_desc(smem_u32(sm.ring[vsl[jj]]), 1024, 1024, kSmem128BSwizzle);
                        umma_e4m3(tmem + OCOL + (tcount & 1) * NR, vd + 256 * q4,
                                  pd + static_cast<uint64_t>(((mb * kBS + 32 * q4) * NR) >> 4), kIdescO, 1);
                        umma_commit(&sm.empty_bar[vsl[jj]]);
                        any = true;
                    }
                }
                if (any)
                    umma_commit(&sm.o_full);
                else
                    mbar_arrive(&sm.o_full);
            }
            __syncwarp();
        }

        // ---- running sums; this tile's O^T is folded with the next tile ----
        if constexpr (kRowSumPerTile) {
            const float wls = lane_sum<NR>(ls, lane);
            Lr = Lr * sm.wfold[tcount & 1][warp][0][rho] + wls * sm.wfold[tcount & 1][warp][1][rho];
        } else {
#pragma unroll
            for (int r4 = 0; r4 < NR / 4; ++r4) {
                const float4 a4 = *reinterpret_cast<const float4*>(&sm.wfold[tcount & 1][warp][0][4 * r4]);
                const float4 b4 = *reinterpret_cast<const float4*>(&sm.wfold[tcount & 1][warp][1][4 * r4]);
                Lp[4 * r4 + 0] = Lp[4 * r4 + 0] * a4.x + ls[4 * r4 + 0] * b4.x;
                Lp[4 * r4 + 1] = Lp[4 * r4 + 1] * a4.y + ls[4 * r4 + 1] * b4.y;
                Lp[4 * r4 + 2] = Lp[4 * r4 + 2] * a4.z + ls[4 * r4 + 2] * b4.z;
                Lp[4 * r4 + 3] = Lp[4 * r4 + 3] * a4.w + ls[4 * r4 + 3] * b4.w;
            }
        }
        pend = tcount;
        ring_advance<NV, NBT>(vslot, vph, nb);
        ++tcount;

        if (t == T - 1 || pos_eq(nx, end)) {
            // ------------------------------ unit end ------------------------------
            fold(pend);
            pend = -1;
            float wl = Lr;
            if constexpr (!kRowSumPerTile) {
                float lsum[NR];
#pragma unroll
                for (int r = 0; r < NR; ++r) lsum[r] = Lp[r];
                wl = lane_sum<NR>(lsum, lane);
            }
            if (rep) sm.redl[warp][rho] = wl;
            named_bar_sync(1, kNCW * 32);
            float L = 0.f;
#pragma unroll
            for (int w = 0; w < kNCW; ++w) L += sm.redl[w][rho];
            if (rep) sm.wst[warp][3][rho] = L;
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
                    stage[rr * kD + ch] = __float2bfloat16_rn(Oa[k] * vs * (1.0f / sm.wst[warp][3][rr]));
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
                if (warp == 0 && rep) {
                    part[32 * kD + rho] = Mref;
                    part[32 * kD + 32 + rho] = L;
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
                    float mx = -INFINITY, lsm = 0.f;
                    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    int kfirst = 0;
                    if (own != nullptr) {
                        mx = own[32 * kD + orow];
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
                        const float mn = fmaxf(fmaxf(mx, fmaxf(mk[0], mk[1])), fmaxf(mk[2], mk[3]));
                        const float c = ex2(mx - mn);
                        lsm *= c;
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[e] *= c;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float sc = ex2(mk[q] - mn);
                            lsm += lk[q] * sc;
                            acc[0] += oa[q].x * sc;
                            acc[1] += oa[q].y * sc;
                            acc[2] += oa[q].z * sc;
                            acc[3] += oa[q].w * sc;
                            acc[4] += ob[q].x * sc;
                            acc[5] += ob[q].y * sc;
                            acc[6] += ob[q].z * sc;
                            acc[7] += ob[q].w * sc;
                        }
                        mx = mn;
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
                        // (a negative wait hands the merge to the last part at once)
                        for (; p.merge_wait_ns >= 0;) {
                            int v;
                            asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p.counters + u) : "memory");
                            if (v == want) {
                                ok = 1;
                                break;
                            }
                            if (globaltimer_ns() - t0 > static_cast<uint64_t>(p.merge_wait_ns)) break;
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
                        if (warp == 0 && rep) {
                            own[32 * kD + rho] = Mref;
                            own[32 * kD + 32 + rho] = L;
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
    // the MM2 MMAs this warp issued have completed (already true unless a wait
    // gave up) before the tensor memory is released
    if (lane == 0 && *(volatile int*)&sm.abort) {
        umma_commit(&sm.cdrain);
        mbar_wait_drain(&sm.cdrain, 0, p.err, 1024);
    }
    __syncwarp();
    tc_fence_before();
    named_bar_sync(2, (kNCW + 1) * 32);
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

// s2_tile 0 picks the tile from the sequences' capacity s2 (the block table's
// width x block_size, the longest a sequence can be): the GLM-4.5 paged FP8
// page's configuration notes give 1024-token tiles to sequences of 8192 and
// more; that tile is built for up to 16 query rows per kv head. Everything
// else gets 512, this kernel's measured best at short lengths (the page's
// short tile of 128 follows its own hardware's tiling).
constexpr int64_t kLongS2 = 8192;

int auto_s2_tile(int S1, int G, int64_t s2)
{
    return (s2 >= kLongS2 && static_cast<int64_t>(S1) * G <= 16) ? 1024 : 512;
}

pa_status make_plan(int B, int S1, int NQ, int NKV, int D, const pa_decode_config* cfg, Plan* pl,
                    int64_t s2 = 0)
{
    PA_REQUIRE(B > 0 && S1 > 0 && NQ > 0 && NKV > 0 && D > 0, PA_ERR_INVALID,
               "pa_fp8_decode: empty or negative shape (B=%d S1=%d NQ=%d NKV=%d D=%d)", B, S1, NQ, NKV, D);
    PA_REQUIRE(NQ % NKV == 0, PA_ERR_INVALID, "pa_fp8_decode: NQ %d is not a multiple of NKV %d", NQ, NKV);
    PA_REQUIRE(D == kD, PA_ERR_UNSUPPORTED, "pa_fp8_decode: head size %d (only 128 is built)", D);
    PA_REQUIRE(B <= kMaxB, PA_ERR_UNSUPPORTED, "pa_fp8_decode: batch %d > %d", B, kMaxB);
    pl->S2T = (cfg && cfg->s2_tile) ? cfg->s2_tile : auto_s2_tile(S1, NQ / NKV, s2);
    PA_REQUIRE(pl->S2T > 0 && pl->S2T % kBS == 0, PA_ERR_INVALID,
               "pa_fp8_decode: s2_tile %d is not a multiple of block_size 128", pl->S2T);
    PA_REQUIRE(pl->S2T == 128 || pl->S2T == 256 || pl->S2T == 512 || pl->S2T == 1024, PA_ERR_UNSUPPORTED,
               "pa_fp8_decode: s2_tile %d (128, 256, 512 and 1024 are built)", pl->S2T);
    PA_REQUIRE(!cfg || (cfg->overlap_prologue >= 0 && cfg->overlap_prologue <= 2), PA_ERR_INVALID,
               "pa_fp8_decode: overlap_prologue %d (0, 1 or 2)", cfg ? cfg->overlap_prologue : 0);
    PA_REQUIRE(!cfg || cfg->wait_limit_ns >= 0, PA_ERR_INVALID, "pa_fp8_decode: wait_limit_ns %d < 0",
               cfg ? cfg->wait_limit_ns : 0);
    pl->G = NQ / NKV;
    pl->R = S1 * pl->G;
    pl->NR = pl->R <= 16 ? 16 : 32;
    // 1024-token tiles: three S^T buffers of 8 x 16 columns fit the tensor
    // memory next to O^T, 8 x 32 do not
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

template <int NR, int S2T, int NRV = NR>
pa_status launch(const CUtensorMap& tk, const CUtensorMap& tv,
                 const DecodeParams& prm, cudaStream_t st)
{
    const size_t smem = sizeof(DecodeSmem<NR, S2T>) + 1024;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [&] {
        attr = cudaFuncSetAttribute(decode_kernel<NR, S2T, NRV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem));
    });
    PA_REQUIRE(attr == cudaSuccess, PA_ERR_CUDA, "pa_fp8_decode: smem attribute: %s", cudaGetErrorString(attr));
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
        const cudaError_t e = cudaLaunchKernelEx(&lc, decode_kernel<NR, S2T, NRV>, tk, tv, prm);
        PA_REQUIRE(e == cudaSuccess, PA_ERR_CUDA, "pa_fp8_decode: launch: %s", cudaGetErrorString(e));
        return PA_OK;
    }
    decode_kernel<NR, S2T, NRV><<<prm.grid, kThreads, smem, st>>>(tk, tv, prm);
    return check_launch("pa_fp8_decode");
}

// Bulk-copy / TMA destinations must be 16-byte aligned (128 for the tensor
// loads of key scales); the 128-byte-swizzled K/V tiles and the Q operand sit
// on 1024-byte boundaries (the swizzle atom the MMA descriptors assume).
template <int NR, int S2T>
struct SmemLayoutChecks {
    using S = DecodeSmem<NR, S2T>;
    static_assert(offsetof(S, ring) % 1024 == 0, "ring alignment");
    static_assert(offsetof(S, qb) % 1024 == 0, "Q operand alignment");
    static_assert(offsetof(S, pbuf) % 128 == 0, "P operand alignment");
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

extern "C" int pa_fp8_decode_auto_s2_tile(int S1, int NQ, int NKV, int64_t s2)
{
    if (S1 <= 0 || NQ <= 0 || NKV <= 0 || NQ % NKV != 0 || s2 < 0) return 0;
    return auto_s2_tile(S1, NQ / NKV, s2);
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
    pa_status st = make_plan(B, S1, NQ, NKV, D, cfg, &pl, static_cast<int64_t>(max_blocks_per_seq) * block_size);
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
    // Units of 32 padded query rows are launched in plain stream order: with
    // programmatic serialisation that kernel hung on the 256-sequence, 24-row
    // workload, for a reason not yet found (the 16-row kernels are unaffected).
    prm.overlap = (cfg && pl.NR == 16) ? cfg->overlap_prologue : 0;
    prm.merge_wait_ns = (cfg && cfg->merge_wait_ns != 0) ? (cfg->merge_wait_ns < 0 ? -1 : cfg->merge_wait_ns)
                                                        : static_cast<int64_t>(kMergeWaitNs);
    prm.wait_ns = (cfg && cfg->wait_limit_ns > 0) ? static_cast<uint64_t>(cfg->wait_limit_ns) : kWaitLimitNs;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pl.NR == 16) {
        if (pl.S2T == 128) return launch<16, 128>(tk, tv, prm, s);
        if (pl.S2T == 256) return launch<16, 256>(tk, tv, prm, s);
        // 12 rows per kv head (the GLM-4.5 group at S1 = 1): the 4 padding
        // rows' softmax work is skipped
        if (pl.S2T == 512) return pl.R == 12 ? launch<16, 512, 12>(tk, tv, prm, s) : launch<16, 512>(tk, tv, prm, s);
        return pl.R == 12 ? launch<16, 1024, 12>(tk, tv, prm, s) : launch<16, 1024>(tk, tv, prm, s);
    }
    if (pl.S2T == 128) return launch<32, 128>(tk, tv, prm, s);
    if (pl.S2T == 256) return launch<32, 256>(tk, tv, prm, s);
    // 24 rows per kv head (S1 = 2 at a group of 12) in one chunk: the 8
    // padding rows' softmax work is skipped
    if (pl.R == 24) return launch<32, 512, 24>(tk, tv, prm, s);
    return launch<32, 512>(tk, tv, prm, s);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of pa_fp8_decode: the same kernel, with its scratch
// (split partials, per-sequence counters, error word) in a fixed array that
// is part of the library's device image instead of a caller workspace.
// ---------------------------------------------------------------------------
namespace pa {
namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(PA_FP8_DECODE_NOALLOC_MAX_SCRATCH);

// One array per device that loads the library, alive until process exit.
__device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current()
{
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
    });
    return fn;
}

// Device address of g_decode_scratch on the current device. The host-side
// name is only a stand-in for the symbol, so the address is looked up with
// that device current and cached per device together with the context it
// was found in: after a device reset the library's image is loaded again
// (possibly elsewhere), the context differs, and the address is looked up
// anew. The first lookup in a context also clears the whole array on
// `stream` (every call leaves the counters zero after that; the error word
// keeps its bits until the caller clears it).
pa_status decode_scratch_address(void** out, cudaStream_t stream)
{
    static std::mutex mu;
    static void* cache[64] = {nullptr};
    static CUcontext ctx_of[64] = {nullptr};
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    PA_REQUIRE(e == cudaSuccess, PA_ERR_CUDA, "pa_fp8_decode_noalloc: cudaGetDevice: %s",
               cudaGetErrorString(e));
    PA_REQUIRE(dev >= 0 && dev < 64, PA_ERR_UNSUPPORTED, "pa_fp8_decode_noalloc: device %d", dev);
    auto get = ctx_get_current();
    PA_REQUIRE(get != nullptr, PA_ERR_CUDA, "pa_fp8_decode_noalloc: cuCtxGetCurrent is not available");
    CUcontext ctx = nullptr;   // none yet before the runtime's first call on this thread
    PA_REQUIRE(get(&ctx) == CUDA_SUCCESS, PA_ERR_CUDA, "pa_fp8_decode_noalloc: cannot read the current context");
    std::lock_guard<std::mutex> lock(mu);
    if (ctx == nullptr || cache[dev] == nullptr || ctx_of[dev] != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);   // makes the device's context current
        PA_REQUIRE(e == cudaSuccess && p != nullptr, PA_ERR_CUDA,
                   "pa_fp8_decode_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        PA_REQUIRE(get(&ctx) == CUDA_SUCCESS && ctx != nullptr, PA_ERR_CUDA,
                   "pa_fp8_decode_noalloc: no current context");
        if (p != cache[dev] || ctx != ctx_of[dev]) {
            e = cudaMemsetAsync(p, 0, kStaticScratchBytes, stream);
            PA_REQUIRE(e == cudaSuccess, PA_ERR_CUDA, "pa_fp8_decode_noalloc: clearing scratch: %s",
                       cudaGetErrorString(e));
            cache[dev] = p;
            ctx_of[dev] = ctx;
        }
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
    st = decode_scratch_address(&ws, static_cast<cudaStream_t>(stream));
    if (st != PA_OK) return st;
    // Every call leaves the counters zero (also one whose waits gave up), so
    // nothing is cleared here and the decode is the only work enqueued: with
    // overlap_prologue it overlaps the preceding kernel as pa_fp8_decode does.
    return pa_fp8_decode(q, q_scale, k_cache, k_scale, v_cache, v_scale, block_table, kv_act_seqs,
                         out, B, S1, NQ, NKV, D, block_size, num_blocks, max_blocks_per_seq, layout,
                         softmax_scale, cfg, ws, kStaticScratchBytes, stream);
}

extern "C" pa_status pa_fp8_decode_noalloc_error(int32_t* flags, int clear, void* stream)
{
    PA_REQUIRE(flags != nullptr, PA_ERR_NULLPTR, "pa_fp8_decode_noalloc_error: flags is NULL");
    void* ws = nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    pa_status st = decode_scratch_address(&ws, s);
    if (st != PA_OK) return st;
    cudaError_t e = cudaMemcpyAsync(flags, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    PA_REQUIRE(e == cudaSuccess, PA_ERR_CUDA, "pa_fp8_decode_noalloc_error: copy: %s", cudaGetErrorString(e));
    if (clear) {
        e = cudaMemsetAsync(ws, 0, sizeof(int32_t), s);
        PA_REQUIRE(e == cudaSuccess, PA_ERR_CUDA, "pa_fp8_decode_noalloc_error: clear: %s",
                   cudaGetErrorString(e));
    }
    return PA_OK;
}
