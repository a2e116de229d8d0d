// cache.cu -- FP8 paged-cache append (scatter and quantise-on-append) and the
// per-token / per-channel E4M3 quantisers.
//
// Pages:
//  "CANN ops-transformer 中的 FP8 KV Cache 更新算子 scatter_pa_kv_cache_with_k_scale
//   使用指南": 功能说明与计算公式 (block_idx = slot / block_size, block_offset =
//   slot % block_size, rows copied per head), 参数说明 (shapes, int32/int64
//   slots, non-contiguous key_scale tail), Kernel 实现 (out-of-range slots
//   skipped).
//  "CANN ops-transformer aclnnKvCompressEpilog 算子详解": 计算公式 场景 1
//   (scale = max|x| / FP8_MAX, q = round(x / scale), FP8_E4M3FN max 448).
//  "PyPTO 实现 GLM-4.5 Paged Attention FP8 量化算子 ...": 量化策略 (Q/K per
//   token, V per channel with the maximum over the sequence).
//
// GPU design: the append moves a few hundred KB, so each kernel is a flat grid
// of independent warps/threads with 16-byte (copy) or 4-byte-per-lane (encode)
// coalesced accesses; no shared memory, no inter-block communication except
// the atomicMax reduction of the per-channel scale.
#include "common.cuh"

namespace pa {
namespace {

constexpr float kE4M3Max = 448.0f;

__device__ __forceinline__ int64_t cache_row(int layout, int64_t blk, int64_t off, int64_t h,
                                             int BS, int H)
{
    return layout == PA_LAYOUT_BSND ? (blk * BS + off) * H + h : (blk * H + h) * BS + off;
}

__device__ __forceinline__ int64_t load_slot(const void* slots, int slot_type, int64_t i)
{
    return slot_type == PA_INDEX_I64 ? __ldg(static_cast<const long long*>(slots) + i)
                                     : static_cast<int64_t>(__ldg(static_cast<const int*>(slots) + i));
}

template <typename T>
__device__ __forceinline__ void load4(const T* p, float (&x)[4]);

template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&x)[4])
{
    float4 v = __ldg(reinterpret_cast<const float4*>(p));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}

template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[4])
{
    uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    x[0] = __uint_as_float(v.x << 16);
    x[1] = __uint_as_float(v.x & 0xFFFF0000u);
    x[2] = __uint_as_float(v.y << 16);
    x[3] = __uint_as_float(v.y & 0xFFFF0000u);
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Codes of x / scale for four values (scale 0 -> code 0).
__device__ __forceinline__ uint32_t encode4_div(const float (&x)[4], float scale)
{
    if (scale == 0.0f) return 0u;
    return e4m3x4(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale), __fdiv_rn(x[2], scale),
                  __fdiv_rn(x[3], scale));
}

// One warp quantises one row of D values (D % 4 == 0): returns the dequant
// scale amax / 448 and writes the codes.
template <typename T>
__device__ __forceinline__ float quant_row_warp(const T* x, int D, uint8_t* codes, int lane)
{
    float amax = 0.0f;
    for (int d = 4 * lane; d < D; d += 128) {
        float v[4];
        load4(x + d, v);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
    }
    amax = warp_max(amax);
    const float scale = __fdiv_rn(amax, kE4M3Max);
    for (int d = 4 * lane; d < D; d += 128) {
        float v[4];
        load4(x + d, v);
        *reinterpret_cast<uint32_t*>(codes + d) = encode4_div(v, scale);
    }
    return scale;
}

// ---- FP8 pass-through scatter ------------------------------------------------
// One thread per (token, head, 16-byte chunk of the K row or V row).
__global__ void scatter16_kernel(const uint8_t* __restrict__ key, const uint8_t* __restrict__ value,
                                 uint8_t* __restrict__ key_cache, uint8_t* __restrict__ value_cache,
                                 const void* __restrict__ slots, int slot_type,
                                 const float* __restrict__ key_scale, int64_t ks0, int64_t ks1,
                                 float* __restrict__ key_scale_cache, int64_t T, int H, int Dk,
                                 int Dv, int64_t num_blocks, int BS, int layout)
{
    const int ck = Dk >> 4, cv = Dv >> 4, per = ck + cv;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= T * H * per) return;
    const int64_t th = idx / per;
    const int c = static_cast<int>(idx - th * per);
    const int64_t i = th / H;
    const int j = static_cast<int>(th - i * H);
    const int64_t s = load_slot(slots, slot_type, i);
    if (s < 0 || s >= num_blocks * BS) return;  // out-of-range slot: skipped
    const int64_t row = cache_row(layout, s / BS, s % BS, j, BS, H);
    if (c < ck) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(key + th * Dk) + c);
        reinterpret_cast<uint4*>(key_cache + row * Dk)[c] = v;
        if (c == 0) key_scale_cache[row] = __ldg(key_scale + i * ks0 + j * ks1);
    } else {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(value + th * Dv) + (c - ck));
        reinterpret_cast<uint4*>(value_cache + row * Dv)[c - ck] = v;
    }
}

// Byte-wise fallback for head sizes that are not multiples of 16 bytes or
// unaligned pointers: one thread per (token, head).
__global__ void scatter_bytes_kernel(const uint8_t* __restrict__ key, const uint8_t* __restrict__ value,
                                     uint8_t* __restrict__ key_cache, uint8_t* __restrict__ value_cache,
                                     const void* __restrict__ slots, int slot_type,
                                     const float* __restrict__ key_scale, int64_t ks0, int64_t ks1,
                                     float* __restrict__ key_scale_cache, int64_t T, int H, int Dk,
                                     int Dv, int64_t num_blocks, int BS, int layout)
{
    const int64_t th = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (th >= T * H) return;
    const int64_t i = th / H;
    const int j = static_cast<int>(th - i * H);
    const int64_t s = load_slot(slots, slot_type, i);
    if (s < 0 || s >= num_blocks * BS) return;
    const int64_t row = cache_row(layout, s / BS, s % BS, j, BS, H);
    for (int d = 0; d < Dk; ++d) key_cache[row * Dk + d] = key[th * Dk + d];
    for (int d = 0; d < Dv; ++d) value_cache[row * Dv + d] = value[th * Dv + d];
    key_scale_cache[row] = key_scale[i * ks0 + j * ks1];
}

// ---- quantise-on-append ----------------------------------------------------------
// One warp per (token, head): key row -> per-row scale and codes, value row ->
// codes against the sequence's per-channel scale.
//
// For D <= 128 * NC every lane keeps its NC groups of four values in
// registers, so all loads (K/V rows, slot, batch, value scales) are issued and
// every code is computed before griddepcontrol.wait; only the cache stores
// follow it. Launched with programmatic stream serialisation the kernel thus
// runs beside the tail of the preceding kernel and writes once that kernel has
// completed; launched plainly the wait returns at once. Threads that store
// nothing (a skipped slot, or past the last token) wait too before they exit:
// the kernel must not complete before its predecessor, or a kernel chained
// after it (a decode) would start writing while that predecessor still runs
// -- with every slot skipped, no thread would otherwise wait at all.
// Blocks are two warps (kAppendThreads) so that they fit on an SM beside a
// resident decode CTA.
constexpr int kAppendThreads = 64;

template <typename T, int NC>
__global__ void __launch_bounds__(kAppendThreads)
quant_scatter_kernel(const T* __restrict__ key, const T* __restrict__ value,
                     uint8_t* __restrict__ key_cache, uint8_t* __restrict__ value_cache,
                     const void* __restrict__ slots, int slot_type,
                     float* __restrict__ key_scale_cache, const float* __restrict__ v_scale,
                     const int* __restrict__ token_batch, int num_batches, int64_t ntok, int H,
                     int D, int64_t num_blocks, int BS, int layout)
{
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t th = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (th >= ntok * H) {
        grid_dependency_wait();
        return;
    }
    const int64_t i = th / H;
    const int j = static_cast<int>(th - i * H);
    const T* krow = key + th * D;
    const T* vrow = value + th * D;
    float k[NC][4] = {}, v[NC][4] = {};
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const int d = 128 * c + 4 * lane;
        if (d < D) {
            load4(krow + d, k[c]);
            load4(vrow + d, v[c]);
        }
    }
    const int64_t s = load_slot(slots, slot_type, i);
    if (s < 0 || s >= num_blocks * BS) {
        grid_dependency_wait();
        return;
    }
    int tb = __ldg(token_batch + i);
    tb = tb < 0 ? 0 : (tb >= num_batches ? num_batches - 1 : tb);
    const float* vs = v_scale + (static_cast<int64_t>(tb) * H + j) * D;
    float4 sc[NC] = {};
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const int d = 128 * c + 4 * lane;
        if (d < D) {
            sc[c] = __ldg(reinterpret_cast<const float4*>(vs + d));
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(k[c][0]), fabsf(k[c][1])),
                                     fmaxf(fabsf(k[c][2]), fabsf(k[c][3]))));
        }
    }
    amax = warp_max(amax);
    const float ks = __fdiv_rn(amax, kE4M3Max);
    uint32_t kc[NC], vc[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        kc[c] = encode4_div(k[c], ks);
        const float q0 = sc[c].x == 0.0f ? 0.0f : __fdiv_rn(v[c][0], sc[c].x);
        const float q1 = sc[c].y == 0.0f ? 0.0f : __fdiv_rn(v[c][1], sc[c].y);
        const float q2 = sc[c].z == 0.0f ? 0.0f : __fdiv_rn(v[c][2], sc[c].z);
        const float q3 = sc[c].w == 0.0f ? 0.0f : __fdiv_rn(v[c][3], sc[c].w);
        vc[c] = e4m3x4(q0, q1, q2, q3);
    }
    const int64_t row = cache_row(layout, s / BS, s % BS, j, BS, H);
    grid_dependency_wait();
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const int d = 128 * c + 4 * lane;
        if (d < D) {
            *reinterpret_cast<uint32_t*>(key_cache + row * D + d) = kc[c];
            *reinterpret_cast<uint32_t*>(value_cache + row * D + d) = vc[c];
        }
    }
    if (lane == 0) key_scale_cache[row] = ks;
}

// Head sizes above 512: the same encoding in loops over the row, everything
// after griddepcontrol.wait.
template <typename T>
__global__ void __launch_bounds__(kAppendThreads)
quant_scatter_wide_kernel(const T* __restrict__ key, const T* __restrict__ value,
                          uint8_t* __restrict__ key_cache, uint8_t* __restrict__ value_cache,
                          const void* __restrict__ slots, int slot_type,
                          float* __restrict__ key_scale_cache, const float* __restrict__ v_scale,
                          const int* __restrict__ token_batch, int num_batches, int64_t ntok,
                          int H, int D, int64_t num_blocks, int BS, int layout)
{
    grid_launch_dependents();
    grid_dependency_wait();
    const int lane = threadIdx.x & 31;
    const int64_t th = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (th >= ntok * H) return;
    const int64_t i = th / H;
    const int j = static_cast<int>(th - i * H);
    const int64_t s = load_slot(slots, slot_type, i);
    if (s < 0 || s >= num_blocks * BS) return;
    int tb = __ldg(token_batch + i);
    tb = tb < 0 ? 0 : (tb >= num_batches ? num_batches - 1 : tb);
    const int64_t row = cache_row(layout, s / BS, s % BS, j, BS, H);
    const float ks = quant_row_warp(key + th * D, D, key_cache + row * D, lane);
    if (lane == 0) key_scale_cache[row] = ks;
    const T* vrow = value + th * D;
    const float* vs = v_scale + (static_cast<int64_t>(tb) * H + j) * D;
    for (int d = 4 * lane; d < D; d += 128) {
        float v[4];
        load4(vrow + d, v);
        const float4 sc = __ldg(reinterpret_cast<const float4*>(vs + d));
        const float q0 = sc.x == 0.0f ? 0.0f : __fdiv_rn(v[0], sc.x);
        const float q1 = sc.y == 0.0f ? 0.0f : __fdiv_rn(v[1], sc.y);
        const float q2 = sc.z == 0.0f ? 0.0f : __fdiv_rn(v[2], sc.z);
        const float q3 = sc.w == 0.0f ? 0.0f : __fdiv_rn(v[3], sc.w);
        *reinterpret_cast<uint32_t*>(value_cache + row * D + d) = e4m3x4(q0, q1, q2, q3);
    }
}

// ---- KV compress epilog (modes 0 and 1) ---------------------------------------------
// One warp per row of x (d BF16 values): the last 64 values (rope) are stored
// first as BF16, the first d - 64 (nope) as E4M3 in groups of 64 with one scale
// per group after them: BF16(amax / 448) in mode 0, a power of two 2^k stored
// as the E8M0 byte k + 127 in mode 1 (k rounded up from amax / 448 with
// round_scale, the exponent of amax / 448 without). The row pitch may be odd,
// so the stores are bytes.
constexpr int kKvcThreads = 128;

// floor(log2(s)) of a positive finite float and whether s is a power of two.
__device__ __forceinline__ int floor_log2_pos(float s, bool* pow2)
{
    const uint32_t u = __float_as_uint(s);
    const int e = static_cast<int>((u >> 23) & 0xFF);
    const uint32_t m = u & 0x7FFFFFu;
    if (e != 0) {
        *pow2 = m == 0;
        return e - 127;
    }
    *pow2 = (m & (m - 1)) == 0;            // subnormal: s = m * 2^-149
    return (31 - __clz(static_cast<int>(m))) - 149;
}

// 2^k as a float for k in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2f(int k)
{
    return k >= -126 ? __uint_as_float(static_cast<uint32_t>(k + 127) << 23) : __uint_as_float(0x00400000u);
}

__global__ void __launch_bounds__(kKvcThreads)
kv_compress_epilog_kernel(uint8_t* __restrict__ cache, int64_t block_num, int block_size,
                          int64_t block_stride, int head_dim, const __nv_bfloat16* __restrict__ x,
                          int64_t bs, int d, const void* __restrict__ slots, int slot_type,
                          int quant_mode, int round_scale)
{
    const int lane = threadIdx.x & 31;
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (r >= bs) return;
    const int64_t s = load_slot(slots, slot_type, r);
    if (s < 0 || s >= block_num * block_size) return;
    uint8_t* row = cache + (s / block_size) * block_stride + (s % block_size) * static_cast<int64_t>(head_dim);
    const uint32_t* xr = reinterpret_cast<const uint32_t*>(x + r * d);   // BF16 pairs
    const int nope = d - 64;
    // rope: 64 BF16 = 128 bytes, 4 per lane
    {
        const uint32_t v = __ldg(xr + (nope >> 1) + lane);
        uint8_t* dst = row + 4 * lane;
        dst[0] = static_cast<uint8_t>(v);
        dst[1] = static_cast<uint8_t>(v >> 8);
        dst[2] = static_cast<uint8_t>(v >> 16);
        dst[3] = static_cast<uint8_t>(v >> 24);
    }
    const int groups = nope / 64;
    for (int g = 0; g < groups; ++g) {
        const uint32_t v = __ldg(xr + 32 * g + lane);
        const float x0 = __uint_as_float(v << 16), x1 = __uint_as_float(v & 0xFFFF0000u);
        const float amax = warp_max(fmaxf(fabsf(x0), fabsf(x1)));
        const float scale = __fdiv_rn(amax, kE4M3Max);
        uint16_t codes;
        if (quant_mode == 0) {
            codes = scale == 0.0f ? 0 : e4m3x2(__fdiv_rn(x0, scale), __fdiv_rn(x1, scale));
            if (lane == 0) {
                // BF16 of the (finite, non-negative) scale: round to nearest even
                // on the FP32 bit pattern
                const uint32_t u = __float_as_uint(scale);
                const uint32_t hb = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
                uint8_t* sc = row + 128 + nope + 2 * g;
                sc[0] = static_cast<uint8_t>(hb);
                sc[1] = static_cast<uint8_t>(hb >> 8);
            }
        } else {
            int k = 0;
            if (scale != 0.0f) {
                bool p2;
                k = floor_log2_pos(scale, &p2);
                if (round_scale && !p2) ++k;
                k = k < -127 ? -127 : (k > 127 ? 127 : k);
                const float p = pow2f(k);
                codes = e4m3x2(__fdiv_rn(x0, p), __fdiv_rn(x1, p));
            } else {
                codes = 0;
                k = -127;
            }
            if (lane == 0) row[128 + nope + g] = static_cast<uint8_t>(k + 127);
        }
        uint8_t* dst = row + 128 + 64 * g + 2 * lane;
        dst[0] = static_cast<uint8_t>(codes);
        dst[1] = static_cast<uint8_t>(codes >> 8);
    }
}

// ---- per-row quantiser -------------------------------------------------------------
template <typename T>
__global__ void quantize_rows_kernel(const T* __restrict__ x, int64_t rows, int D,
                                     uint8_t* __restrict__ codes, float* __restrict__ scale)
{
    const int lane = threadIdx.x & 31;
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (r >= rows) return;
    const float s = quant_row_warp(x + r * D, D, codes + r * D, lane);
    if (lane == 0) scale[r] = s;
}

// ---- per-channel value scale ----------------------------------------------------------
// amax over each sequence's tokens, per (head, channel); bits of the
// non-negative float maxima are combined with atomicMax into v_scale (zeroed
// first), then divided by 448 in place.
constexpr int kVsTokens = 64;

template <typename T>
__global__ void value_amax_kernel(const T* __restrict__ v, const long long* __restrict__ cu,
                                  int B, int64_t total, int HD, unsigned int* __restrict__ amax_bits)
{
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kVsTokens;
    if (t0 >= total) return;
    const int64_t t1 = min(t0 + kVsTokens, total);
    // batch of token t0: last b with cu[b] <= t0
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= t0) lo = mid; else hi = mid - 1;
    }
    for (int g = threadIdx.x; 4 * g < HD; g += blockDim.x) {
        int b = lo;
        int64_t bend = __ldg(cu + b + 1);
        float m[4] = {0.f, 0.f, 0.f, 0.f};
        for (int64_t t = t0; t < t1; ++t) {
            while (t >= bend) {  // flush and move to the next sequence
                unsigned int* dst = amax_bits + static_cast<int64_t>(b) * HD + 4 * g;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (m[k] > 0.f) atomicMax(dst + k, __float_as_uint(m[k]));
                    m[k] = 0.f;
                }
                ++b;
                bend = __ldg(cu + b + 1);
            }
            float x[4];
            load4(v + t * HD + 4 * g, x);
#pragma unroll
            for (int k = 0; k < 4; ++k) m[k] = fmaxf(m[k], fabsf(x[k]));
        }
        unsigned int* dst = amax_bits + static_cast<int64_t>(b) * HD + 4 * g;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (m[k] > 0.f) atomicMax(dst + k, __float_as_uint(m[k]));
    }
}

__global__ void value_scale_finalize_kernel(float* __restrict__ vs, int64_t n)
{
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n) vs[i] = __fdiv_rn(__uint_as_float(reinterpret_cast<unsigned int*>(vs)[i]), kE4M3Max);
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline unsigned int blocks_for(int64_t n, int per) { return static_cast<unsigned int>((n + per - 1) / per); }

// Launches the quantise-on-append kernel for this head size, with
// programmatic stream serialisation when `overlap` is set.
template <typename T>
cudaError_t launch_quant_scatter(const T* key, const T* value, unsigned int grid, cudaStream_t st,
                                 bool overlap, void* key_cache, void* value_cache,
                                 const void* slots, int slot_type, float* key_scale_cache,
                                 const float* v_scale, const int32_t* token_batch,
                                 int num_batches, int64_t ntok, int H, int D, int64_t num_blocks,
                                 int BS, int layout)
{
    using Kern = void (*)(const T*, const T*, uint8_t*, uint8_t*, const void*, int, float*,
                          const float*, const int*, int, int64_t, int, int, int64_t, int, int);
    const Kern k = D <= 128   ? quant_scatter_kernel<T, 1>
                   : D <= 256 ? quant_scatter_kernel<T, 2>
                   : D <= 512 ? quant_scatter_kernel<T, 4>
                              : quant_scatter_wide_kernel<T>;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3(kAppendThreads);
    lc.dynamicSmemBytes = 0;
    lc.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = overlap ? 1 : 0;
    return cudaLaunchKernelEx(&lc, k, key, value, static_cast<uint8_t*>(key_cache),
                              static_cast<uint8_t*>(value_cache), slots, slot_type,
                              key_scale_cache, v_scale, token_batch, num_batches, ntok, H, D,
                              num_blocks, BS, layout);
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_fp8_cache_scatter(const void* key, const void* value, void* key_cache,
                                          void* value_cache, const void* slot_mapping,
                                          int slot_type, const float* key_scale,
                                          int64_t ks_stride0, int64_t ks_stride1,
                                          float* key_scale_cache, int64_t num_tokens, int num_head,
                                          int k_head_size, int v_head_size, int64_t num_blocks,
                                          int block_size, int layout, void* stream)
{
    PA_REQUIRE(key && value && key_cache && value_cache && slot_mapping && key_scale &&
                   key_scale_cache,
               PA_ERR_NULLPTR, "pa_fp8_cache_scatter: NULL tensor pointer");
    PA_REQUIRE(num_tokens > 0 && num_head > 0 && k_head_size > 0 && v_head_size > 0 &&
                   num_blocks > 0 && block_size > 0,
               PA_ERR_INVALID, "pa_fp8_cache_scatter: empty or negative size");
    PA_REQUIRE(layout == PA_LAYOUT_BSND || layout == PA_LAYOUT_BNBD, PA_ERR_INVALID,
               "pa_fp8_cache_scatter: unknown layout %d", layout);
    PA_REQUIRE(slot_type == PA_INDEX_I32 || slot_type == PA_INDEX_I64, PA_ERR_INVALID,
               "pa_fp8_cache_scatter: unknown slot type %d", slot_type);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool vec = (k_head_size % 16 == 0) && (v_head_size % 16 == 0) && aligned(key, 16) &&
                     aligned(value, 16) && aligned(key_cache, 16) && aligned(value_cache, 16);
    if (vec) {
        const int64_t n = num_tokens * num_head * (k_head_size / 16 + v_head_size / 16);
        scatter16_kernel<<<blocks_for(n, 256), 256, 0, st>>>(
            static_cast<const uint8_t*>(key), static_cast<const uint8_t*>(value),
            static_cast<uint8_t*>(key_cache), static_cast<uint8_t*>(value_cache), slot_mapping,
            slot_type, key_scale, ks_stride0, ks_stride1, key_scale_cache, num_tokens, num_head,
            k_head_size, v_head_size, num_blocks, block_size, layout);
    } else {
        const int64_t n = num_tokens * num_head;
        scatter_bytes_kernel<<<blocks_for(n, 128), 128, 0, st>>>(
            static_cast<const uint8_t*>(key), static_cast<const uint8_t*>(value),
            static_cast<uint8_t*>(key_cache), static_cast<uint8_t*>(value_cache), slot_mapping,
            slot_type, key_scale, ks_stride0, ks_stride1, key_scale_cache, num_tokens, num_head,
            k_head_size, v_head_size, num_blocks, block_size, layout);
    }
    return check_launch("pa_fp8_cache_scatter");
}

extern "C" pa_status pa_fp8_cache_quant_scatter(const void* key, const void* value, int in_dtype,
                                                void* key_cache, void* value_cache,
                                                const void* slot_mapping, int slot_type,
                                                float* key_scale_cache, const float* v_scale,
                                                const int32_t* token_batch, int num_batches,
                                                int64_t num_tokens, int num_head, int head_size,
                                                int64_t num_blocks, int block_size, int layout,
                                                int overlap_prologue, void* stream)
{
    PA_REQUIRE(key && value && key_cache && value_cache && slot_mapping && key_scale_cache &&
                   v_scale && token_batch,
               PA_ERR_NULLPTR, "pa_fp8_cache_quant_scatter: NULL tensor pointer");
    PA_REQUIRE(num_tokens > 0 && num_head > 0 && head_size > 0 && num_blocks > 0 &&
                   block_size > 0 && num_batches > 0,
               PA_ERR_INVALID, "pa_fp8_cache_quant_scatter: empty or negative size");
    PA_REQUIRE(head_size % 4 == 0, PA_ERR_UNSUPPORTED,
               "pa_fp8_cache_quant_scatter: head_size %d is not a multiple of 4", head_size);
    PA_REQUIRE(layout == PA_LAYOUT_BSND || layout == PA_LAYOUT_BNBD, PA_ERR_INVALID,
               "pa_fp8_cache_quant_scatter: unknown layout %d", layout);
    PA_REQUIRE(slot_type == PA_INDEX_I32 || slot_type == PA_INDEX_I64, PA_ERR_INVALID,
               "pa_fp8_cache_quant_scatter: unknown slot type %d", slot_type);
    PA_REQUIRE(in_dtype == PA_DTYPE_F32 || in_dtype == PA_DTYPE_BF16, PA_ERR_INVALID,
               "pa_fp8_cache_quant_scatter: unknown input dtype %d", in_dtype);
    const uintptr_t in_align = in_dtype == PA_DTYPE_F32 ? 16 : 8;
    PA_REQUIRE(aligned(key, in_align) && aligned(value, in_align) && aligned(key_cache, 4) &&
                   aligned(value_cache, 4) && aligned(v_scale, 16),
               PA_ERR_INVALID, "pa_fp8_cache_quant_scatter: misaligned pointer");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t warps = num_tokens * num_head;
    const unsigned int grid = blocks_for(warps * 32, kAppendThreads);
    cudaError_t e;
    if (in_dtype == PA_DTYPE_F32)
        e = launch_quant_scatter(static_cast<const float*>(key), static_cast<const float*>(value),
                                 grid, st, overlap_prologue != 0, key_cache, value_cache,
                                 slot_mapping, slot_type, key_scale_cache, v_scale, token_batch,
                                 num_batches, num_tokens, num_head, head_size, num_blocks,
                                 block_size, layout);
    else
        e = launch_quant_scatter(static_cast<const __nv_bfloat16*>(key),
                                 static_cast<const __nv_bfloat16*>(value), grid, st,
                                 overlap_prologue != 0, key_cache, value_cache, slot_mapping,
                                 slot_type, key_scale_cache, v_scale, token_batch, num_batches,
                                 num_tokens, num_head, head_size, num_blocks, block_size, layout);
    PA_REQUIRE(e == cudaSuccess, PA_ERR_CUDA, "pa_fp8_cache_quant_scatter: launch: %s",
               cudaGetErrorString(e));
    return PA_OK;
}

extern "C" pa_status pa_fp8_kv_compress_epilog(void* cache, int64_t block_num, int block_size,
                                               int64_t block_stride, int head_dim, const void* x,
                                               int64_t bs, int d, const void* slot_mapping,
                                               int slot_type, int quant_group_size, int quant_mode,
                                               int round_scale, void* stream)
{
    PA_REQUIRE(cache && x && slot_mapping, PA_ERR_NULLPTR, "pa_fp8_kv_compress_epilog: NULL tensor pointer");
    PA_REQUIRE(bs > 0 && block_num > 0 && block_size > 0 && head_dim > 0, PA_ERR_INVALID,
               "pa_fp8_kv_compress_epilog: empty or negative size");
    PA_REQUIRE(d % 64 == 0 && d > 64 && d <= 8192, PA_ERR_INVALID,
               "pa_fp8_kv_compress_epilog: d %d (a multiple of 64 in (64, 8192])", d);
    PA_REQUIRE(quant_mode == 0 || quant_mode == 1, quant_mode == 2 ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID,
               "pa_fp8_kv_compress_epilog: quant_mode %d (0 and 1 are built)", quant_mode);
    PA_REQUIRE(quant_group_size == 64, PA_ERR_INVALID,
               "pa_fp8_kv_compress_epilog: quant_group_size %d (modes 0 and 1 use 64)", quant_group_size);
    PA_REQUIRE(slot_type == PA_INDEX_I32 || slot_type == PA_INDEX_I64, PA_ERR_INVALID,
               "pa_fp8_kv_compress_epilog: unknown slot type %d", slot_type);
    const int64_t concat = (d - 64) + 128 + static_cast<int64_t>((d - 64) / 64) * (quant_mode == 0 ? 2 : 1);
    const int64_t min_col = quant_mode == 0 ? (concat + 31) / 32 * 32 : concat;
    PA_REQUIRE(head_dim >= min_col, PA_ERR_INVALID,
               "pa_fp8_kv_compress_epilog: head_dim %d < %lld bytes a row needs", head_dim,
               static_cast<long long>(min_col));
    PA_REQUIRE(block_stride >= static_cast<int64_t>(block_size) * head_dim, PA_ERR_INVALID,
               "pa_fp8_kv_compress_epilog: block_stride %lld < block_size * head_dim",
               static_cast<long long>(block_stride));
    PA_REQUIRE(aligned(x, 4), PA_ERR_INVALID, "pa_fp8_kv_compress_epilog: misaligned x");
    kv_compress_epilog_kernel<<<blocks_for(bs * 32, kKvcThreads), kKvcThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint8_t*>(cache), block_num, block_size, block_stride, head_dim,
        static_cast<const __nv_bfloat16*>(x), bs, d, slot_mapping, slot_type, quant_mode, round_scale);
    return check_launch("pa_fp8_kv_compress_epilog");
}

extern "C" pa_status pa_fp8_quantize_rows(const void* x, int in_dtype, int64_t rows, int D,
                                          void* codes, float* scale, void* stream)
{
    PA_REQUIRE(x && codes && scale, PA_ERR_NULLPTR, "pa_fp8_quantize_rows: NULL tensor pointer");
    PA_REQUIRE(rows > 0 && D > 0, PA_ERR_INVALID, "pa_fp8_quantize_rows: empty tensor");
    PA_REQUIRE(D % 4 == 0, PA_ERR_UNSUPPORTED, "pa_fp8_quantize_rows: D %d not a multiple of 4", D);
    PA_REQUIRE(in_dtype == PA_DTYPE_F32 || in_dtype == PA_DTYPE_BF16, PA_ERR_INVALID,
               "pa_fp8_quantize_rows: unknown input dtype %d", in_dtype);
    PA_REQUIRE(aligned(x, in_dtype == PA_DTYPE_F32 ? 16 : 8) && aligned(codes, 4), PA_ERR_INVALID,
               "pa_fp8_quantize_rows: misaligned pointer");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const unsigned int grid = blocks_for(rows * 32, 256);
    if (in_dtype == PA_DTYPE_F32)
        quantize_rows_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(x), rows, D,
                                                          static_cast<uint8_t*>(codes), scale);
    else
        quantize_rows_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
            static_cast<const __nv_bfloat16*>(x), rows, D, static_cast<uint8_t*>(codes), scale);
    return check_launch("pa_fp8_quantize_rows");
}

extern "C" pa_status pa_fp8_value_channel_scale(const void* v, int in_dtype,
                                                const int64_t* cu_seqlens, int B,
                                                int64_t total_tokens, int H, int D,
                                                float* v_scale, void* stream)
{
    PA_REQUIRE(v && cu_seqlens && v_scale, PA_ERR_NULLPTR,
               "pa_fp8_value_channel_scale: NULL tensor pointer");
    PA_REQUIRE(B > 0 && H > 0 && D > 0 && total_tokens >= 0, PA_ERR_INVALID,
               "pa_fp8_value_channel_scale: empty or negative size");
    PA_REQUIRE((static_cast<int64_t>(H) * D) % 4 == 0, PA_ERR_UNSUPPORTED,
               "pa_fp8_value_channel_scale: H*D not a multiple of 4");
    PA_REQUIRE(in_dtype == PA_DTYPE_F32 || in_dtype == PA_DTYPE_BF16, PA_ERR_INVALID,
               "pa_fp8_value_channel_scale: unknown input dtype %d", in_dtype);
    PA_REQUIRE(aligned(v, in_dtype == PA_DTYPE_F32 ? 16 : 8), PA_ERR_INVALID,
               "pa_fp8_value_channel_scale: misaligned pointer");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t n = static_cast<int64_t>(B) * H * D;
    if (cudaMemsetAsync(v_scale, 0, n * sizeof(float), st) != cudaSuccess)
        return check_launch("pa_fp8_value_channel_scale: memset");
    const int HD = H * D;
    const int threads = HD / 4 >= 256 ? 256 : ((HD / 4 + 31) / 32) * 32;
    if (total_tokens > 0) {
        const unsigned int grid = blocks_for(total_tokens, kVsTokens);
        if (in_dtype == PA_DTYPE_F32)
            value_amax_kernel<float><<<grid, threads, 0, st>>>(
                static_cast<const float*>(v), reinterpret_cast<const long long*>(cu_seqlens), B,
                total_tokens, HD, reinterpret_cast<unsigned int*>(v_scale));
        else
            value_amax_kernel<__nv_bfloat16><<<grid, threads, 0, st>>>(
                static_cast<const __nv_bfloat16*>(v), reinterpret_cast<const long long*>(cu_seqlens),
                B, total_tokens, HD, reinterpret_cast<unsigned int*>(v_scale));
    }
    value_scale_finalize_kernel<<<blocks_for(n, 256), 256, 0, st>>>(v_scale, n);
    return check_launch("pa_fp8_value_channel_scale");
}
