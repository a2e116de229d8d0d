// mla.cu -- MLA sparse attention with FP8 anti-quantisation (decode) on
// sm_103a: the DeepSeek-V3.2 shape of "PyPTO-Gym 算子实战：DeepSeek V32 MLA 的
// Sparse Attention FP8 反量化算子（Ascend 950PR）解析与验证" (sections 核心参数与
// KV Cache 布局, 计算流程：5 层嵌套循环, 关键实现细节, 在线反量化与 Online Softmax
// 的实现细节).
//
// One CTA per (query token, group of 64 query heads). The token's selected
// keys are walked in tiles of 128:
//   producers (7 warps)  gather half of the selected rows (top-k index -> block
//                        table -> 656-byte packed row), dequantise the E4M3 nope
//                        part by its 128-channel group scale to BF16 and write
//                        the 576-wide BF16 key rows into shared memory as nine
//                        64-channel chunks in the 128-byte-swizzled layout (the
//                        consumers do the other half between their softmax steps);
//   MMA warp (1 thread)  C1: S^T[key][head] = K[key][576] . Q[head][576]^T
//                        (tcgen05 kind::f16, M = 128 keys, N = 64 heads, FP32 in
//                        tensor memory); C2: O^T[chan][head] += V^T[chan][key] .
//                        P^T[key][head] with V = the nope chunks of the same
//                        tile read MN-major (M = 128 channels, four groups);
//   consumers (8 warps)  per tile and head: max over the tile's keys, P =
//                        exp(S - max), its sum, BF16 P^T for C2; the running
//                        max / sum and the rescale of O^T in tensor memory;
//                        finally out = BF16(O / L).
// The softmax is tile-local as on the page: P is taken against the tile's
// own max and cast to BF16, and tiles are merged with exp(m_old - m_new) and
// exp(m_tile - m_new). O^T is kept as O / beta, beta being the last merged
// tile's exp(m_tile - m_new), so that C2 can accumulate into it directly.
//
// The same kernel also reads the rows that the KV compress epilog ("CANN
// ops-transformer aclnnKvCompressEpilog 算子详解", 计算公式 场景 1 / 场景 2)
// writes for d = 576: rope first, the nope codes in groups of 64 channels,
// one BF16 or E8M0 scale per group. Only where the producers find the codes,
// the rope bytes and the scale of a group differs (a template parameter).
#include "common.cuh"

#include <cuda_fp8.h>

#include <cmath>
#include <cstddef>
#include <mutex>

namespace pa {
namespace {

constexpr int kDn = 512;            // kv_lora_rank: the nope part, also V
constexpr int kDr = 64;             // rope part
constexpr int kRowUsed = 656;       // kn 512 B | kr 128 B | 4 FP32 scales
// Row formats. Page: the MLA page's packed row (E4M3 kn at byte 0, BF16 kr at
// 512, four FP32 scales, one per 128 channels, at 640). KvcBf16 / KvcE8m0: the
// KV compress epilog's row for d = 576 with quant mode 0 / 1 (BF16 kr at 0,
// E4M3 kn at 128, at 640 one scale per 64 channels: 8 BF16 values / 8 E8M0
// bytes e for 2^(e - 127)). Every format lies within bytes [0, 656).
constexpr int kFmtPage = 0;
constexpr int kFmtKvcBf16 = 1;
constexpr int kFmtKvcE8m0 = 2;
constexpr int kScaleOff = kDn + 2 * kDr;
template <int F>
constexpr int kCodeOff = F == kFmtPage ? 0 : 2 * kDr;
template <int F>
constexpr int kRopeOff = F == kFmtPage ? kDn : 0;
constexpr int kHG = 64;             // query heads per CTA (N of C1 and C2)
constexpr int kNK = 128;            // keys per tile (M of C1)
constexpr int kNC = 9;              // 64-channel chunks of a 576-wide row
constexpr int kKChunk = kNK * 128;  // bytes per key chunk (128 rows x 128 B)
constexpr int kQChunk = kHG * 128;
constexpr int kConsWarps = 8;
constexpr int kProdWarps = 7;       // 16 warps in all: 4 per SM sub-partition, 128 registers each
constexpr int kRowGroups = kNK / 4;   // 4 key rows per group
// Row groups 0..15 of a tile are dequantised by the 7 producer warps (group
// rg by warp rg % 7, up to 3 each), 16..31 by the 8 consumer warps (group rg
// by consumer warp (rg - 16) % 8, 2 each) once they have handed P^T to C2.
constexpr int kProdGroups = kRowGroups / 2;
constexpr int kGroupsPerProd = (kProdGroups + kProdWarps - 1) / kProdWarps;
constexpr int kGroupsPerCons = (kRowGroups - kProdGroups) / kConsWarps;
constexpr int kProdWarp0 = kConsWarps;
constexpr int kMmaWarp = kConsWarps + kProdWarps;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 2 * kHG;   // O^T group g at columns kOCol + 64 g; S^T double buffer below
// A tile whose max lies more than 2^30 below the running max adds under
// 2^-30 * 128 of the running sum: it is left out for that head, which keeps
// O / beta finite.
constexpr float kNegligibleLog2 = -30.0f;

struct MlaSmem {
    uint8_t kt[kNC][kKChunk];         // key tile; chunk 8 holds kr, then P^T
    uint8_t qt[kNC][kQChunk];         // the 64 heads' queries
    float red[2][4][kHG];             // per lane quarter: column max / column sum
    float wrow[kConsWarps][32];       // per consumer warp: one broadcast row
    // k_full[i] (i < 4): chunks 2i, 2i+1 of the tile written; k_full[4]: the rope
    // chunk. k_empty[g]: C2's channel group g (chunks 2g, 2g+1) done; after
    // group 3 P^T in chunk 8 is free too.
    uint64_t q_full, k_full[5], k_empty[4], s_full[2], s_empty[2], p_full, o_done, drain;
    uint32_t tmem_base;
    int abort;
};

struct MlaParams {
    const uint16_t* q_nope;
    const uint16_t* q_rope;
    const uint8_t* cache;
    const int32_t* topk_idx;
    const int32_t* block_table;
    const int32_t* act;
    uint16_t* out;
    int* err;
    int64_t row_bytes;
    int64_t block_stride;             // bytes from one block to the next (>= BS * row_bytes)
    int64_t num_blocks;
    int S1, NQ, topk, BS, max_blocks;
    float scale_log2;                 // softmax_scale * log2(e)
};

// ---- 16-bit tcgen05 operands, 32-column tensor memory transfers, cp.async drain ----
// Instruction descriptor of kind::f16 with BF16 A and B (format 1 in both
// operand-type fields), F32 accumulator; a_mn / b_mn select MN-major (1)
// instead of K-major (0) operands.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
           (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// D(tmem) (+)= A(smem) * B(smem) with 16-bit operands (K = 16 per MMA).
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v)
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

// Blocks until every cp.async of this thread has landed.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Position of 16-byte unit u of row r in a 128-byte-swizzled chunk.
__device__ __forceinline__ uint32_t sw128(int r, int u)
{
    return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((u ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint4 ldg_nc16(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Two E4M3 codes (low byte first) times an FP32 scale, each product rounded
// to BF16, packed low element first.
__device__ __forceinline__ uint32_t dq2(uint32_t two, float s)
{
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
    const __nv_bfloat162 r = __floats2bfloat162_rn(f.x * s, f.y * s);
    return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&r);
}

// Warp transpose-sum of a 32 x 32 block (lane = row, v[c] = column c):
// returns, in lane l, the sum of column l over the 32 lanes. v is destroyed.
__device__ __forceinline__ float col_sum(float (&v)[32], int lane)
{
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = up ? v[i] : v[i + s];
            const float keep = up ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return v[0];
}

// ---- key rows: a warp handles row groups rg = rg0 + step * gi (gi < NG, rg <
// lim); lane (rr, cu) handles row 4 rg + rr and its 16-byte units cu + 8 i:
// unit U holds channels 16U..16U+15, i.e. chunk U / 4 and scale group i ----

// Byte offset of each row in the cache, -1 for an entry that takes no part
// (past the visible count, -1, or past the sequence end).
template <int NG>
__device__ __forceinline__ void rows_locate(const MlaParams& p, int t, int cur, int act, int b, int64_t tk_base,
                                            int rg0, int step, int lim, int rr, int64_t (&ro)[NG])
{
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
        const int rg = rg0 + step * gi;
        ro[gi] = -1;
        if (rg < lim) {
            const int j = t * kNK + 4 * rg + rr;
            const int idx = j < cur ? __ldg(p.topk_idx + tk_base + j) : -1;
            if (idx >= 0 && idx < act) {
                const int bi = idx / p.BS;   // past the table's width: out of contract, block 0
                int blk = bi < p.max_blocks ? __ldg(p.block_table + static_cast<int64_t>(b) * p.max_blocks + bi)
                                            : 0;
                if (blk < 0 || blk >= p.num_blocks) blk = 0;
                ro[gi] = static_cast<int64_t>(blk) * p.block_stride + static_cast<int64_t>(idx % p.BS) * p.row_bytes;
            }
        }
    }
}

// The codes and the scale unit of each row into registers (zeros for rows
// that take no part); the rope bytes are brought to L2 for the later copy.
template <int F, int NG>
__device__ __forceinline__ void rows_load(const MlaParams& p, const int64_t (&ro)[NG], int cu, uint4 (&kn)[NG][4],
                                          uint4 (&sc)[NG])
{
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
        if (ro[gi] >= 0) {
            const uint8_t* src = p.cache + ro[gi];
#pragma unroll
            for (int i = 0; i < 4; ++i) kn[gi][i] = ldg_nc16(src + kCodeOff<F> + 16 * (cu + 8 * i));
            sc[gi] = ldg_nc16(src + kScaleOff);
            asm volatile("prefetch.global.L2 [%0];" ::"l"(src + kRopeOff<F> + 16 * cu));
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) kn[gi][i] = make_uint4(0, 0, 0, 0);
            sc[gi] = make_uint4(0, 0, 0, 0);
        }
    }
}

// Whole rows (656 bytes, at most six 128-byte lines) to L2 ahead of time.
template <int NG>
__device__ __forceinline__ void rows_prefetch_l2(const MlaParams& p, const int64_t (&ro)[NG], int cu)
{
#pragma unroll
    for (int gi = 0; gi < NG; ++gi)
        if (ro[gi] >= 0 && cu < 6) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.cache + ro[gi] + 128 * cu));
}

// Dequant scale of a lane's code unit i (channels 128 i + 16 cu .. + 15) from
// the row's 16-byte scale unit: the page row's FP32 scale of 128 channels i,
// or the KV compress row's scale of 64 channels 2 i + cu / 4.
template <int F>
__device__ __forceinline__ float unit_scale(const uint4& s, int i, int cu)
{
    const uint32_t w = i == 0 ? s.x : i == 1 ? s.y : i == 2 ? s.z : s.w;
    if constexpr (F == kFmtPage) {
        return __uint_as_float(w);
    } else if constexpr (F == kFmtKvcBf16) {
        // BF16 scale 2 i + cu / 4: half cu / 4 of word i (little-endian)
        return __uint_as_float(cu < 4 ? w << 16 : w & 0xFFFF0000u);
    } else {
        // E8M0 byte 2 i + cu / 4 of the first 8 bytes: 2^(e - 127), e = 0
        // being the FP32 subnormal 2^-127
        const uint32_t w8 = i < 2 ? s.x : s.y;
        const uint32_t e = (w8 >> (8 * (2 * (i & 1) + (cu >> 2)))) & 0xFFu;
        return __uint_as_float(e != 0 ? e << 23 : 0x00400000u);
    }
}

// Dequantise the rows' unit i (channels 128 i + 16 cu .. + 15 of each row)
// into chunk pair i, and the rope chunk; each step is announced on k_full
// once the previous tile's C2 has released the chunks.
template <int F, int NG>
__device__ __forceinline__ void rows_produce(MlaSmem& sm, const MlaParams& p, int t, const int64_t (&ro)[NG],
                                             const uint4 (&kn)[NG][4], const uint4 (&sc)[NG], int rg0, int step,
                                             int lim, int rr, int cu, int lane)
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (t > 0) mbar_wait(&sm.k_empty[i], static_cast<uint32_t>(t - 1) & 1u, p.err, 2, &sm.abort);
        uint8_t* chunk = sm.kt[(cu >> 2) + 2 * i];
        const int u0 = 2 * (cu & 3);
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            const int rg = rg0 + step * gi;
            if (rg >= lim) continue;
            const int k = 4 * rg + rr;
            const uint4 c8 = kn[gi][i];
            const float f = unit_scale<F>(sc[gi], i, cu);
            uint4 lo, hi;
            lo.x = dq2(c8.x & 0xFFFFu, f);
            lo.y = dq2(c8.x >> 16, f);
            lo.z = dq2(c8.y & 0xFFFFu, f);
            lo.w = dq2(c8.y >> 16, f);
            hi.x = dq2(c8.z & 0xFFFFu, f);
            hi.y = dq2(c8.z >> 16, f);
            hi.z = dq2(c8.w & 0xFFFFu, f);
            hi.w = dq2(c8.w >> 16, f);
            *reinterpret_cast<uint4*>(chunk + sw128(k, u0)) = lo;
            *reinterpret_cast<uint4*>(chunk + sw128(k, u0 + 1)) = hi;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.k_full[i]);
    }
    // the rope chunk: free once the previous C2's last group is done, which
    // the wait for pair 3 covered
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
        const int rg = rg0 + step * gi;
        if (rg < lim) {
            const int k = 4 * rg + rr;
            uint8_t* dst = sm.kt[8] + sw128(k, cu);
            if (ro[gi] >= 0)
                cp_async16(dst, p.cache + ro[gi] + kRopeOff<F> + 16 * cu, 16);
            else
                *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.k_full[4]);
}

template <int F>
__global__ void __launch_bounds__(kThreads, 1) mla_decode_kernel(const MlaParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
    MlaSmem& sm = *reinterpret_cast<MlaSmem*>(smem_raw + ((1024u - (raw & 1023u)) & 1023u));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ngroups = p.NQ / kHG;
    const int tok = blockIdx.x / ngroups;
    const int hg = blockIdx.x - tok * ngroups;
    const int b = tok / p.S1, s = tok - b * p.S1;
    const int act = __ldg(p.act + b);
    // keys this token attends to: clamp(kv_act_seqs - S1 + 1 + s, 0, topk)
    const int cur = min(max(act - p.S1 + 1 + s, 0), p.topk);
    const int ntiles = (cur + kNK - 1) / kNK;
    uint16_t* const outp = p.out + (static_cast<int64_t>(tok) * p.NQ + hg * kHG) * kDn;
    if (ntiles == 0) {
        for (int i = threadIdx.x; i < kHG * kDn / 8; i += kThreads)
            reinterpret_cast<uint4*>(outp)[i] = make_uint4(0, 0, 0, 0);
        return;
    }

    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, kProdWarps);
        for (int i = 0; i < 5; ++i) mbar_init(&sm.k_full[i], kProdWarps + kConsWarps);
        for (int i = 0; i < 4; ++i) mbar_init(&sm.k_empty[i], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.s_full[i], 1);
            mbar_init(&sm.s_empty[i], kConsWarps);
        }
        mbar_init(&sm.p_full, kConsWarps);
        mbar_init(&sm.o_done, 1);
        mbar_init(&sm.drain, 1);
        sm.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) tmem_alloc(&sm.tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const int64_t tk_base = static_cast<int64_t>(tok) * p.topk;

    if (warp >= kProdWarp0 && warp < kMmaWarp) {
        // ================================ producers ================================
        const int pw = warp - kProdWarp0;
        {
            // the 64 heads' 576-wide queries: 72 16-byte units per head
            const int64_t row0 = static_cast<int64_t>(tok) * p.NQ + hg * kHG;
            for (int i = threadIdx.x - kProdWarp0 * 32; i < kHG * 72; i += kProdWarps * 32) {
                const int h = i / 72, u = i - h * 72;
                uint4 v;
                int c, cu;
                if (u < 64) {
                    v = ldg_nc16(p.q_nope + (row0 + h) * kDn + u * 8);
                    c = u >> 3;
                    cu = u & 7;
                } else {
                    v = ldg_nc16(p.q_rope + (row0 + h) * kDr + (u - 64) * 8);
                    c = 8;
                    cu = u - 64;
                }
                *reinterpret_cast<uint4*>(sm.qt[c] + sw128(h, cu)) = v;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.q_full);
        }
        const int rr = lane >> 3, cu = lane & 7;
        for (int t = 0; t < ntiles; ++t) {
            int64_t ro[kGroupsPerProd];
            uint4 kn[kGroupsPerProd][4], sc[kGroupsPerProd];
            rows_locate<kGroupsPerProd>(p, t, cur, act, b, tk_base, pw, kProdWarps, kProdGroups, rr, ro);
            rows_load<F, kGroupsPerProd>(p, ro, cu, kn, sc);
            rows_produce<F, kGroupsPerProd>(sm, p, t, ro, kn, sc, pw, kProdWarps, kProdGroups, rr, cu, lane);
        }
    } else if (warp == kMmaWarp) {
        // ================================ MMA issue ================================
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16(128, kHG, 0, 0);   // K-major keys and queries
            constexpr uint32_t kIdescO = idesc_bf16(128, kHG, 1, 1);   // MN-major V^T and P^T
            mbar_wait(&sm.q_full, 0, p.err, 1, &sm.abort);
            for (int t = 0; t < ntiles; ++t) {
                mbar_wait(&sm.s_empty[t & 1], (static_cast<uint32_t>(t >> 1) & 1u) ^ 1u, p.err, 32, &sm.abort);
                const uint32_t d = tmem + static_cast<uint32_t>((t & 1) * kHG);
                for (int c = 0; c < kNC; ++c) {
                    if ((c & 1) == 0) {   // chunks 2i, 2i+1 (and the rope chunk 8) as they land
                        mbar_wait(&sm.k_full[c >> 1], static_cast<uint32_t>(t) & 1u, p.err, 16, &sm.abort);
                        tc_fence_after();
                    }
                    const uint64_t ad = smem_desc(smem_u32(sm.kt[c]), 16, 1024, kSmem128BSwizzle);
                    const uint64_t bd = smem_desc(smem_u32(sm.qt[c]), 16, 1024, kSmem128BSwizzle);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)   // 16 channels (32 bytes) per MMA
                        umma_bf16(d, ad + 2 * kk, bd + 2 * kk, kIdescS, (c | kk) != 0);
                }
                umma_commit(&sm.s_full[t & 1]);
                mbar_wait(&sm.p_full, static_cast<uint32_t>(t) & 1u, p.err, 64, &sm.abort);
                tc_fence_after();
                for (int g = 0; g < 4; ++g) {
                    // channels 128g..128g+127 = key chunks 2g and 2g+1 (LBO: the
                    // next 64 channels); 16 keys per MMA (SBO: the next 8 keys)
                    for (int ks = 0; ks < kNK / 16; ++ks) {
                        const uint64_t ad = smem_desc(smem_u32(sm.kt[2 * g]) + ks * 2048, kKChunk, 1024,
                                                      kSmem128BSwizzle);
                        const uint64_t bd = smem_desc(smem_u32(sm.kt[8]) + ks * 2048, kKChunk, 1024,
                                                      kSmem128BSwizzle);
                        umma_bf16(tmem + kOCol + 64 * g, ad, bd, kIdescO, (t > 0 || ks > 0) ? 1u : 0u);
                    }
                    umma_commit(&sm.k_empty[g]);
                }
                umma_commit(&sm.o_done);
            }
            umma_commit(&sm.drain);
            mbar_wait_drain(&sm.drain, 0, p.err, 128);
        }
        __syncwarp();
    } else {
        // ================================ consumers ================================
        const int q4 = warp & 3, hf = warp >> 2;
        const int key = 32 * q4 + lane;                 // tensor memory lane of S^T / O^T
        // this warp's share of the key rows (row groups 16 + warp, 24 + warp):
        // tile 0 now, tile t+1 once P^T of tile t is handed to C2
        const int rr = lane >> 3, cu = lane & 7;
        const int crg0 = kProdGroups + warp;
        int64_t cro[kGroupsPerCons];
        rows_locate<kGroupsPerCons>(p, 0, cur, act, b, tk_base, crg0, kConsWarps, kRowGroups, rr, cro);
        {
            uint4 kn[kGroupsPerCons][4], sc[kGroupsPerCons];
            rows_load<F, kGroupsPerCons>(p, cro, cu, kn, sc);
            rows_produce<F, kGroupsPerCons>(sm, p, 0, cro, kn, sc, crg0, kConsWarps, kRowGroups, rr, cu, lane);
        }
        if (ntiles > 1) {
            rows_locate<kGroupsPerCons>(p, 1, cur, act, b, tk_base, crg0, kConsWarps, kRowGroups, rr, cro);
            rows_prefetch_l2<kGroupsPerCons>(p, cro, cu);
        }
        const uint32_t lanes = static_cast<uint32_t>(32 * q4) << 16;
        float Mrun = -INFINITY, Lrun = 0.f, sig = 1.f;   // head hf*32 + lane (log2 units)
        bool any = false;
        int idx_next = key < cur ? __ldg(p.topk_idx + tk_base + key) : -1;
        for (int t = 0; t < ntiles; ++t) {
            const int j = t * kNK + key;
            const int idx = idx_next;
            if (t + 1 < ntiles) idx_next = j + kNK < cur ? __ldg(p.topk_idx + tk_base + j + kNK) : -1;
            const bool ok = j < cur && idx >= 0 && idx < act;

            mbar_wait(&sm.s_full[t & 1], static_cast<uint32_t>(t >> 1) & 1u, p.err, 4, &sm.abort);
            tc_fence_after();
            float v[32];
            tmem_ld32(tmem + lanes + static_cast<uint32_t>((t & 1) * kHG + hf * 32), v);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.s_empty[t & 1]);
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = ok ? v[c] * p.scale_log2 : -INFINITY;

            // ---- tile max per head ----
            float w[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) w[c] = v[c];
            {
                // column c's maximum over the warp's 32 keys (one warp reduction
                // per head column), kept by lane c
                float cm = 0.f;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float m = warp_max_f32(w[c]);
                    cm = lane == c ? m : cm;
                }
                sm.red[0][q4][hf * 32 + lane] = cm;
            }
            named_bar_sync(1, kConsWarps * 32);
            const int hc = hf * 32 + lane;
            const float m_t = fmaxf(fmaxf(sm.red[0][0][hc], sm.red[0][1][hc]),
                                    fmaxf(sm.red[0][2][hc], sm.red[0][3][hc]));
            bool drop = m_t == -INFINITY;
            float Mn = m_t;
            if (!drop && any) {
                Mn = fmaxf(Mrun, m_t);
                drop = m_t - Mn < kNegligibleLog2;
            }
            sm.wrow[warp][lane] = drop ? INFINITY : m_t;
            __syncwarp();
            // ---- P = 2^(S - m), its BF16 copy and its sum per head ----
            uint32_t pk[16];
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                const float4 m4 = reinterpret_cast<const float4*>(sm.wrow[warp])[c4];
                w[4 * c4 + 0] = ex2(v[4 * c4 + 0] - m4.x);
                w[4 * c4 + 1] = ex2(v[4 * c4 + 1] - m4.y);
                w[4 * c4 + 2] = ex2(v[4 * c4 + 2] - m4.z);
                w[4 * c4 + 3] = ex2(v[4 * c4 + 3] - m4.w);
            }
#pragma unroll
            for (int c2 = 0; c2 < 16; ++c2) pk[c2] = pack_bf16(w[2 * c2], w[2 * c2 + 1]);
            __syncwarp();
            sm.red[1][q4][hc] = col_sum(w, lane);
            named_bar_sync(1, kConsWarps * 32);
            const float l_t = (sm.red[1][0][hc] + sm.red[1][1][hc]) + (sm.red[1][2][hc] + sm.red[1][3][hc]);
            // ---- running state of head hc and the factor for O^T ----
            float gamma = 1.f;
            if (!drop) {
                if (!any) {
                    gamma = 0.f;
                    Mrun = m_t;
                    Lrun = l_t;
                    sig = 1.f;
                    any = true;
                } else {
                    const float a = ex2(Mrun - Mn), be = ex2(m_t - Mn);
                    Lrun = Lrun * a + l_t * be;
                    gamma = a * sig / be;
                    sig = be;
                    Mrun = Mn;
                }
            }
            sm.wrow[warp][lane] = gamma;
            __syncwarp();
            if (t > 0) {
                // the previous tile's C2 is complete: rescale O^T, then P^T may
                // replace the previous P^T
                mbar_wait(&sm.o_done, static_cast<uint32_t>(t - 1) & 1u, p.err, 8, &sm.abort);
                tc_fence_after();
                if (__any_sync(0xffffffffu, gamma != 1.f)) {
                    float gc[32];
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const float4 g4 = reinterpret_cast<const float4*>(sm.wrow[warp])[c4];
                        gc[4 * c4 + 0] = g4.x;
                        gc[4 * c4 + 1] = g4.y;
                        gc[4 * c4 + 2] = g4.z;
                        gc[4 * c4 + 3] = g4.w;
                    }
#pragma unroll 1
                    for (int g = 0; g < 4; ++g) {
                        const uint32_t a = tmem + lanes + kOCol + static_cast<uint32_t>(64 * g + hf * 32);
                        float o[32];
                        tmem_ld32(a, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] *= gc[c];
                        tmem_st32(a, o);
                    }
                    tmem_wait_st();
                }
            }
            // P^T row `key`: heads hf*32 .. hf*32+31 are 16-byte units 4 hf .. 4 hf + 3
            uint8_t* prow = sm.kt[8];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                *reinterpret_cast<uint4*>(prow + sw128(key, 4 * hf + u)) =
                    make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.p_full);
            if (t + 1 < ntiles) {
                {
                    uint4 kn[kGroupsPerCons][4], sc[kGroupsPerCons];
                    rows_load<F, kGroupsPerCons>(p, cro, cu, kn, sc);
                    rows_produce<F, kGroupsPerCons>(sm, p, t + 1, cro, kn, sc, crg0, kConsWarps, kRowGroups, rr,
                                                    cu, lane);
                }
                if (t + 2 < ntiles) {
                    rows_locate<kGroupsPerCons>(p, t + 2, cur, act, b, tk_base, crg0, kConsWarps, kRowGroups, rr,
                                                cro);
                    rows_prefetch_l2<kGroupsPerCons>(p, cro, cu);
                }
            }
        }
        // ---- out = BF16(O / L) = BF16(O^T * sig / L) ----
        mbar_wait(&sm.o_done, static_cast<uint32_t>(ntiles - 1) & 1u, p.err, 8, &sm.abort);
        tc_fence_after();
        sm.wrow[warp][lane] = any ? sig / Lrun : 0.f;
        __syncwarp();
        float fc[32];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
            const float4 f4 = reinterpret_cast<const float4*>(sm.wrow[warp])[c4];
            fc[4 * c4 + 0] = f4.x;
            fc[4 * c4 + 1] = f4.y;
            fc[4 * c4 + 2] = f4.z;
            fc[4 * c4 + 3] = f4.w;
        }
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
            float o[32];
            tmem_ld32(tmem + lanes + kOCol + static_cast<uint32_t>(64 * g + hf * 32), o);
            tmem_wait_ld();
            uint16_t* dst = outp + static_cast<int64_t>(hf * 32) * kDn + 128 * g + key;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const __nv_bfloat16 h = __float2bfloat16_rn(o[c] * fc[c]);
                dst[static_cast<int64_t>(c) * kDn] = *reinterpret_cast<const uint16_t*>(&h);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

static_assert(offsetof(MlaSmem, kt) % 1024 == 0 && offsetof(MlaSmem, qt) % 1024 == 0, "operand alignment");
static_assert(offsetof(MlaSmem, wrow) % 16 == 0, "broadcast row alignment");
static_assert(kProdGroups <= kGroupsPerProd * kProdWarps && kGroupsPerCons * kConsWarps + kProdGroups == kRowGroups,
              "every row group has one warp");
static_assert(sizeof(MlaSmem) + 1024 <= 232448, "MLA decode shared memory over budget");

inline bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// Validation and launch shared by the entry points; F is the row format.
template <int F>
pa_status mla_launch(const char* name, const void* q_nope, const void* q_rope, const void* cache, int64_t row_bytes,
                     int64_t block_stride, const int32_t* topk_indices, const int32_t* block_table, const int32_t* kv_act_seqs, void* out,
                     int B, int S1, int NQ, int n_kv, int topk, int block_size, int64_t num_blocks,
                     int max_blocks_per_seq, float softmax_scale, int s2_tile, int* status, void* stream)
{
    PA_REQUIRE(q_nope && q_rope && cache && topk_indices && block_table && kv_act_seqs && out && status,
               PA_ERR_NULLPTR, "%s: null pointer argument", name);
    PA_REQUIRE(B >= 0 && S1 >= 1 && NQ >= 1 && topk >= 1 && block_size >= 1 && num_blocks >= 1 &&
                   max_blocks_per_seq >= 1,
               PA_ERR_INVALID, "%s: bad sizes (B=%d S1=%d NQ=%d topk=%d block_size=%d)", name, B, S1, NQ, topk,
               block_size);
    PA_REQUIRE(row_bytes >= kRowUsed && row_bytes % 16 == 0, PA_ERR_INVALID,
               "%s: row_bytes %lld must be >= 656 and a multiple of 16", name, static_cast<long long>(row_bytes));
    PA_REQUIRE(block_stride >= block_size * row_bytes && block_stride % 16 == 0, PA_ERR_INVALID,
               "%s: block_stride %lld must be >= block_size * row_bytes and a multiple of 16", name,
               static_cast<long long>(block_stride));
    PA_REQUIRE(std::isfinite(softmax_scale), PA_ERR_INVALID, "%s: softmax_scale not finite", name);
    PA_REQUIRE(num_blocks * block_size <= 0x7FFFFFFF, PA_ERR_UNSUPPORTED, "%s: more than 2^31 - 1 cache rows", name);
    PA_REQUIRE(n_kv == 1, PA_ERR_UNSUPPORTED, "%s: n_kv %d (one latent KV head is built)", name, n_kv);
    PA_REQUIRE(NQ % kHG == 0, PA_ERR_UNSUPPORTED, "%s: NQ %d (a multiple of 64 is built)", name, NQ);
    PA_REQUIRE(s2_tile == kNK, PA_ERR_UNSUPPORTED, "%s: s2_tile %d (128 is built)", name, s2_tile);
    PA_REQUIRE(aligned16(q_nope) && aligned16(q_rope) && aligned16(cache) && aligned16(out) &&
                   (reinterpret_cast<uintptr_t>(status) & 3u) == 0,
               PA_ERR_INVALID, "%s: q_nope, q_rope, the cache and out must be 16-byte aligned", name);
    const int64_t grid = static_cast<int64_t>(B) * S1 * (NQ / kHG);
    PA_REQUIRE(grid <= 0x7FFFFFFF, PA_ERR_INVALID, "%s: too many CTAs", name);
    if (grid == 0) return PA_OK;

    MlaParams prm;
    prm.q_nope = static_cast<const uint16_t*>(q_nope);
    prm.q_rope = static_cast<const uint16_t*>(q_rope);
    prm.cache = static_cast<const uint8_t*>(cache);
    prm.topk_idx = topk_indices;
    prm.block_table = block_table;
    prm.act = kv_act_seqs;
    prm.out = static_cast<uint16_t*>(out);
    prm.err = status;
    prm.row_bytes = row_bytes;
    prm.block_stride = block_stride;
    prm.num_blocks = num_blocks;
    prm.S1 = S1;
    prm.NQ = NQ;
    prm.topk = topk;
    prm.BS = block_size;
    prm.max_blocks = max_blocks_per_seq;
    prm.scale_log2 = softmax_scale * 1.4426950408889634f;

    const size_t smem = sizeof(MlaSmem) + 1024;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [&] {
        attr = cudaFuncSetAttribute(mla_decode_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem));
    });
    PA_REQUIRE(attr == cudaSuccess, PA_ERR_CUDA, "%s: smem attribute: %s", name, cudaGetErrorString(attr));
    mla_decode_kernel<F><<<static_cast<unsigned>(grid), kThreads, smem, static_cast<cudaStream_t>(stream)>>>(prm);
    return check_launch(name);
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_mla_sparse_decode(const void* q_nope, const void* q_rope, const void* nope_cache,
                                          int64_t row_bytes, const int32_t* topk_indices,
                                          const int32_t* block_table, const int32_t* kv_act_seqs, void* out,
                                          int B, int S1, int NQ, int n_kv, int topk, int block_size,
                                          int64_t num_blocks, int max_blocks_per_seq, float softmax_scale,
                                          int s2_tile, int* status, void* stream)
{
    return mla_launch<kFmtPage>("pa_mla_sparse_decode", q_nope, q_rope, nope_cache, row_bytes,
                                static_cast<int64_t>(block_size) * row_bytes, topk_indices, block_table,
                                kv_act_seqs, out, B, S1, NQ, n_kv, topk, block_size, num_blocks, max_blocks_per_seq,
                                softmax_scale, s2_tile, status, stream);
}

extern "C" pa_status pa_mla_sparse_decode_kvc(const void* q_nope, const void* q_rope, const void* kv_cache,
                                              int64_t row_bytes, int64_t block_stride, int quant_mode,
                                              const int32_t* topk_indices, const int32_t* block_table,
                                              const int32_t* kv_act_seqs, void* out, int B, int S1, int NQ,
                                              int n_kv, int topk, int block_size, int64_t num_blocks,
                                              int max_blocks_per_seq, float softmax_scale, int s2_tile,
                                              int* status, void* stream)
{
    PA_REQUIRE(quant_mode != 2, PA_ERR_UNSUPPORTED,
               "pa_mla_sparse_decode_kvc: quant_mode 2 (HiFloat8 / FP4 rows) is not built");
    PA_REQUIRE(quant_mode == 0 || quant_mode == 1, PA_ERR_INVALID, "pa_mla_sparse_decode_kvc: quant_mode %d",
               quant_mode);
    if (block_stride == 0) block_stride = static_cast<int64_t>(block_size) * row_bytes;
    if (quant_mode == 0)
        return mla_launch<kFmtKvcBf16>("pa_mla_sparse_decode_kvc", q_nope, q_rope, kv_cache, row_bytes,
                                       block_stride, topk_indices, block_table, kv_act_seqs, out, B, S1, NQ,
                                       n_kv, topk, block_size, num_blocks, max_blocks_per_seq, softmax_scale,
                                       s2_tile, status, stream);
    return mla_launch<kFmtKvcE8m0>("pa_mla_sparse_decode_kvc", q_nope, q_rope, kv_cache, row_bytes, block_stride,
                                   topk_indices, block_table, kv_act_seqs, out, B, S1, NQ, n_kv, topk, block_size,
                                   num_blocks, max_blocks_per_seq, softmax_scale, s2_tile, status, stream);
}
