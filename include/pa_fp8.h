/*
 * pa_fp8.h -- C ABI of the GB300 (sm_103a) FP8 paged-KV library.
 *
 * Two operations sit on the decode hot path:
 *   pa_fp8_decode        grouped-query paged decode attention over an FP8
 *                        E4M3 KV cache (split-KV flash decoding, BF16 out);
 *   pa_fp8_cache_scatter the FP8 cache append by slot_mapping, with its
 *                        quantise-on-append form pa_fp8_cache_quant_scatter.
 * Two small quantisers prepare FP8 inputs the way the decode page describes
 * (per-token Q/K, per-channel V): pa_fp8_quantize_rows and
 * pa_fp8_value_channel_scale.
 *
 * Conventions shared by every entry point:
 *  - Every tensor pointer is CUDA device memory owned by the caller (or
 *    memory the device can address, e.g. managed memory). The library keeps
 *    no pointer after a call returns.
 *  - The library never allocates or frees device memory and never waits
 *    for the device: each call validates its arguments on the host, enqueues
 *    its kernels on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and returns. Results are ready when the stream reaches them.
 *  - Shapes are explicit integers; tensors are dense row-major unless a
 *    stride argument says otherwise. FP8 tensors are bytes (E4M3 codes).
 *  - Errors: argument problems found on the host return a status without
 *    enqueuing anything; a failed launch returns PA_ERR_CUDA.
 *    pa_last_error() gives a one-line description of the last failure on the
 *    calling thread. Device-side data (block ids, slots, lengths) is not
 *    validated on the host; the kernels guard memory safety as documented
 *    per call.
 *
 * Page references name the page title and section:
 *  [PA] "PyPTO 实现 GLM-4.5 Paged Attention FP8 量化算子 ... Kernel 实战解析"
 *  [SC] "CANN ops-transformer 中的 FP8 KV Cache 更新算子
 *        scatter_pa_kv_cache_with_k_scale 使用指南"
 *  [KC] "CANN ops-transformer aclnnKvCompressEpilog 算子详解"
 */
#ifndef PA_FP8_H
#define PA_FP8_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_NULLPTR = 1,     /* a required pointer is NULL                      */
    PA_ERR_INVALID = 2,     /* bad shape, size, layout, dtype or empty tensor  */
    PA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required      */
    PA_ERR_CUDA = 4,        /* a CUDA runtime/driver call or launch failed     */
    PA_ERR_UNSUPPORTED = 5  /* valid, but not built (e.g. head_size != 128)    */
} pa_status;

/* Paged cache layouts.
 * PA_LAYOUT_BSND: [num_blocks, block_size, num_heads, head_size] -- the
 *   "PA_BSND" layout of [PA] (Kernel 签名: k [num_blocks, block_size, NKV, D]).
 * PA_LAYOUT_BNBD: [num_blocks, num_heads, block_size, head_size] -- the
 *   "BNBD" cache_layout of [SC] (参数说明).
 * Scale caches use the same shapes with head_size 1. */
typedef enum pa_kv_layout {
    PA_LAYOUT_BSND = 0,
    PA_LAYOUT_BNBD = 1
} pa_kv_layout;

/* Element type of floating-point inputs to the quantisers. */
typedef enum pa_dtype {
    PA_DTYPE_F32 = 0,
    PA_DTYPE_BF16 = 1
} pa_dtype;

/* Element type of slot_mapping ([SC] 参数说明: int32 or int64). */
typedef enum pa_index_type {
    PA_INDEX_I32 = 0,
    PA_INDEX_I64 = 1
} pa_index_type;

/* Tuning knobs of pa_fp8_decode. Zero-initialise and set only what you
 * need; 0 means "default". */
typedef struct pa_decode_config {
    int s2_tile;   /* KV tile of the online softmax and the P-quantisation
                      group ([PA] 配置说明: s2_tile). Multiple of block_size;
                      128, 256 and 512 are built, and 1024 (the pages' tile
                      for long sequences) when S1 x NQ/NKV <= 16. 0 (default):
                      pa_fp8_decode_auto_s2_tile() of the block table's
                      capacity max_blocks_per_seq x block_size.              */
    int num_ctas;  /* persistent grid size. Default: SM count x resident
                      CTAs per SM.                                            */
    int overlap_prologue; /* 1: launch with programmatic stream serialisation
                      so that the kernel's prologue (schedule, block ids, Q
                      rows and scales) overlaps the tail of the preceding
                      kernel in the stream. The kernel then reads
                      kv_act_seqs, block_table, q, q_scale and v_scale
                      before that kernel has finished -- the caller
                      guarantees the preceding kernel does not write them --
                      and waits for it before touching k_cache, v_cache,
                      k_scale, out and the workspace. 0 (default): ordinary
                      stream order.
                      2: as 1, and the K/V cache blocks that hold only
                      positions below kv_act_seqs[b] - S1 of their sequence
                      are also loaded (and MM1 run on them) before the
                      preceding kernel has finished; the caller guarantees
                      that kernel writes no K/V cache entry there (it may
                      write each sequence's S1 newest positions, as the
                      append of a decode step does). Key scales, the newest
                      blocks, out and the workspace still wait for it.
                      Units of more than 16 query rows per kv head
                      (S1 x NQ/NKV > 16) are always launched in plain
                      stream order: 1 and 2 act as 0 there.
                      Other values return PA_ERR_INVALID.                     */
    int merge_wait_ns; /* test and diagnostic knob. A sequence whose tiles are
                      spread over several CTAs is merged by its first CTA,
                      which waits (bounded) for the other parts' count; when
                      that wait runs out, the last part to arrive merges
                      instead. 0: default wait (100 us); negative: no wait, so
                      the last-arriving part always merges. Same result either
                      way, up to FP32 rounding order.                         */
    int wait_limit_ns; /* test and diagnostic knob: time limit of the kernel's
                      bounded waits (a wait that runs out sets a bit of the
                      workspace error word and the kernel finishes, its output
                      undefined; the workspace stays usable). 0: default
                      (about 2 s). Waits that keep issued copies and MMAs from
                      outliving the CTA keep the default. Negative values
                      return PA_ERR_INVALID.                                  */
    int reserved[3];
} pa_decode_config;

/* Text of a status code (static storage). */
PA_API const char* pa_status_string(pa_status status);

/* One-line description of the last non-PA_OK status returned on the calling
 * thread (static thread-local storage; "" if none). */
PA_API const char* pa_last_error(void);

/* ------------------------------------------------------------------------
 * Paged FP8 decode attention ([PA] 计算流程 steps 1-10; signature from
 * [PA] Kernel 签名与源码对应关系).
 *
 * For every batch b, query row s < S1 and query head h (kv head
 * n2 = h / (NQ / NKV), grouped-query attention), over the kv_act_seqs[b]
 * tokens of sequence b, walked in s2_tile-sized tiles:
 *   S_j  = ((Q_fp8 . K_fp8,j) * q_scale) * k_scale_j * softmax_scale
 *   M    = running max, P_j = exp(S_j - M),
 *   Sum  = Sum * exp(M_old - M) + sum_j P_j                (FP32 state)
 *   P_fp8 = E4M3(P * 448 / max_j P_j) per row and tile, P_scale = max P / 448
 *   O    = O * exp(M_old - M) + ((P_fp8 . V_fp8) * P_scale) * v_scale
 *   out  = BF16(O / Sum)
 * The tiles of one sequence may be processed by several CTAs (split-KV) and
 * merged with a log-sum-exp combine; splits fall on s2_tile boundaries so
 * the P-quantisation groups are those of the sequential walk.
 *
 * Arguments (device pointers; shapes in elements):
 *   q            E4M3 [B*S1, NQ, D], row (b*S1 + s)*NQ + h.
 *   q_scale      float [B*S1, NQ] dequant scale per query token and head.
 *   k_cache      E4M3 paged cache in `layout`, num_blocks blocks of
 *                block_size tokens, NKV heads of D bytes.
 *   k_scale      float, the k_cache shape with D = 1 (per token and head).
 *   v_cache      E4M3, same shape as k_cache.
 *   v_scale      float [B, NKV, D] per-channel dequant scale.
 *   block_table  int32 [B, max_blocks_per_seq]; entry i of row b is the
 *                physical block of tokens [i*block_size, (i+1)*block_size).
 *                -1 (and any id outside [0, num_blocks)) is read as block 0
 *                ([PA] 注意事项); entries past the sequence end are not read.
 *   kv_act_seqs  int32 [B] sequence lengths. Values above
 *                max_blocks_per_seq*block_size are clamped to it; values
 *                <= 0 give an all-zero output row.
 *   out          BF16 [B*S1, NQ, D].
 *   D, block_size  128 and 128 are built; anything else is
 *                PA_ERR_UNSUPPORTED. NQ must be a multiple of NKV.
 *   softmax_scale  usually 1/sqrt(D).
 *   cfg          optional (NULL = defaults).
 *   workspace    device scratch of at least pa_fp8_decode_workspace_size()
 *                bytes, 256-byte aligned. Its first bytes are per-sequence
 *                counters that must be zero before the FIRST call that uses
 *                this workspace (e.g. cudaMemset once after allocation);
 *                every call leaves them zero again. Calls that share a
 *                workspace must not overlap in time (same stream is fine).
 * Limits: B <= 1024; s2_tile (cfg) 0 (automatic), 128, 256, 512 or 1024
 * (1024 needs S1 x NQ/NKV <= 16). Other values return PA_ERR_UNSUPPORTED
 * before anything is enqueued.
 * Alignment: q, k_cache, v_cache, v_scale and out 16-byte aligned, k_scale
 * 4-byte aligned (PA_ERR_INVALID otherwise).
 * Errors on the device: every wait inside the kernel is bounded (about 2 s);
 * a wait that gives up sets a non-zero word at the start of the workspace
 * and the output is undefined. The call itself has returned PA_OK by then:
 * callers that want to detect it read that word after the stream completes.
 * ------------------------------------------------------------------------ */
PA_API pa_status pa_fp8_decode_workspace_size(int B, int S1, int NQ, int NKV, int D,
                                       const pa_decode_config* cfg, size_t* bytes);

/* ------------------------------------------------------------------------
 * pa_fp8_decode_auto_s2_tile -- the s2_tile that s2_tile 0 selects.
 * [PA] 配置说明 (s2_tile): a 1024-token tile for long sequences (its
 * threshold 8192; the comparator is lost in the page, read here as s2 >=
 * 8192), a short tile otherwise. Returns 1024 when s2 >= 8192 and
 * S1 x NQ/NKV <= 16 (the query rows a 1024-token tile is built for), else
 * 512; 0 for an invalid shape (S1, NQ or NKV < 1, NQ not a multiple of NKV,
 * s2 < 0). s2 is the longest a sequence can be: pa_fp8_decode passes
 * max_blocks_per_seq x block_size. Host-only; touches no device.
 * ------------------------------------------------------------------------ */
PA_API int pa_fp8_decode_auto_s2_tile(int S1, int NQ, int NKV, int64_t s2);

PA_API pa_status pa_fp8_decode(const void* q, const float* q_scale,
                        const void* k_cache, const float* k_scale,
                        const void* v_cache, const float* v_scale,
                        const int32_t* block_table, const int32_t* kv_act_seqs,
                        void* out,
                        int B, int S1, int NQ, int NKV, int D, int block_size,
                        int64_t num_blocks, int max_blocks_per_seq, int layout,
                        float softmax_scale, const pa_decode_config* cfg,
                        void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * pa_fp8_decode_noalloc: the same decode as pa_fp8_decode for callers that
 * cannot allocate device memory. The pages have no counterpart to it; it
 * exists for callers that are handed tensor pointers and a stream but own no
 * allocator -- for example a plugin inside another framework's runtime, or
 * a serving loop whose device memory is planned up front and which must not
 * call cudaMalloc in the middle of a step (cudaMalloc can synchronise the
 * device and can fail under memory pressure).
 *
 * It takes the arguments of pa_fp8_decode except the workspace. Its scratch
 * is a fixed array of PA_FP8_DECODE_NOALLOC_MAX_SCRATCH bytes compiled into
 * the library; every GPU that loads the library holds that array until the
 * process exits. Shapes whose pa_fp8_decode_workspace_size() exceeds it are
 * rejected with PA_ERR_WORKSPACE (nothing is enqueued).
 *  - No cudaMalloc, cudaFree or allocating library routine is called.
 *  - The first call on each device (and the first after a device reset)
 *    looks up the array's device address (cudaGetSymbolAddress, with that
 *    device current) and clears the array with cudaMemsetAsync on `stream`;
 *    make that first call before any stream capture. Later calls enqueue the
 *    decode kernel only (so overlap_prologue works as for pa_fp8_decode):
 *    every call leaves the array's counters zero again.
 *  - All calls on a device share the one array: calls whose execution
 *    overlaps on the GPU (different streams without ordering) race and give
 *    wrong results. Calls ordered on one stream are safe.
 *  - Errors on the device: the array's first word is the error word of
 *    pa_fp8_decode (a bit set when a kernel wait gave up, output undefined);
 *    it keeps its bits across calls until cleared. Read it with
 *    pa_fp8_decode_noalloc_error.
 * ------------------------------------------------------------------------ */
#define PA_FP8_DECODE_NOALLOC_MAX_SCRATCH (16u << 20)

PA_API pa_status pa_fp8_decode_noalloc(const void* q, const float* q_scale,
                                       const void* k_cache, const float* k_scale,
                                       const void* v_cache, const float* v_scale,
                                       const int32_t* block_table,
                                       const int32_t* kv_act_seqs, void* out,
                                       int B, int S1, int NQ, int NKV, int D,
                                       int block_size, int64_t num_blocks,
                                       int max_blocks_per_seq, int layout,
                                       float softmax_scale, const pa_decode_config* cfg,
                                       void* stream);

/* pa_fp8_decode_noalloc_error: enqueues on `stream` a copy of the allocation-
 * free decode's error word (of the current device) into *flags (host memory;
 * the value is valid once the stream has completed the copy: after a stream
 * or event synchronisation), and, if `clear` is non-zero, then zeroes the
 * word. Like the decode itself it allocates nothing; the pages have no
 * counterpart to it. */
PA_API pa_status pa_fp8_decode_noalloc_error(int32_t* flags, int clear, void* stream);

/* ------------------------------------------------------------------------
 * FP8 cache append scatter ([SC] 功能说明与计算公式, 参数说明, 约束说明).
 * In place. For token i < num_tokens and head j < num_head, with
 * s = slot_mapping[i]:
 *   if s < 0 or s >= num_blocks*block_size: skip ([SC] Kernel 实现, 边界防御)
 *   blk = s / block_size, off = s % block_size
 *   key_cache[blk][j][off][:]   = key[i][j][:]          (BNBD indexing)
 *   value_cache[blk][j][off][:] = value[i][j][:]
 *   key_scale_cache[blk][j][off][0] = key_scale[i][j]
 * key, value     FP8 bytes [num_tokens, num_head, k_head_size / v_head_size]
 *                (E4M3 or E5M2: bytes are copied unchanged).
 * key_cache, value_cache  FP8 bytes in `layout`.
 * slot_mapping   int32 or int64 [num_tokens] (slot_type). Slots should be
 *                unique; with duplicates which write wins is undefined.
 * key_scale      float, element (i, j) at key_scale[i*ks_stride0 +
 *                j*ks_stride1] (the tail may be non-contiguous).
 * key_scale_cache float, the cache shape with head size 1 (contiguous).
 * num_tokens, num_head, head sizes > 0 (empty tensors are PA_ERR_INVALID).
 * ------------------------------------------------------------------------ */
PA_API pa_status pa_fp8_cache_scatter(const void* key, const void* value,
                               void* key_cache, void* value_cache,
                               const void* slot_mapping, int slot_type,
                               const float* key_scale, int64_t ks_stride0,
                               int64_t ks_stride1, float* key_scale_cache,
                               int64_t num_tokens, int num_head, int k_head_size,
                               int v_head_size, int64_t num_blocks, int block_size,
                               int layout, void* stream);

/* ------------------------------------------------------------------------
 * Quantise-on-append scatter: like pa_fp8_cache_scatter, but key and value
 * arrive in FP32 or BF16 (in_dtype) and are encoded on the way in.
 *   key:   per (token, head) dequant scale ks = max_d |k| / 448 (FP32 IEEE
 *          division), codes E4M3(k / ks) round-to-nearest-even, saturating;
 *          ks is stored to key_scale_cache ([KC] 计算公式 场景 1 applied to
 *          the whole head; the per-token-head key_scale of [SC]).
 *   value: codes E4M3(v / v_scale[token_batch[i]][j][d]) against the
 *          sequence's per-channel scale (saturating). A zero scale gives
 *          code 0, as does an all-zero key row (ks = 0).
 * v_scale      float [num_batches, num_head, head_size].
 * token_batch  int32 [num_tokens], the sequence of each new token, in
 *              [0, num_batches).
 * overlap_prologue  0: ordinary stream order. Non-zero: the kernel is
 *              launched with programmatic stream serialisation; it reads key,
 *              value, slot_mapping, token_batch and v_scale and computes all
 *              codes while the preceding kernel of the stream may still run,
 *              and writes the caches only after that kernel has completed
 *              (griddepcontrol.wait). The caller guarantees that the preceding
 *              kernel does not write those five inputs. It also lets the next
 *              kernel launch early (a decode with overlap_prologue set then
 *              overlaps this one the same way).
 * Slots, alignment and errors as above; head_size a multiple of 4; key and
 * value 16-byte (FP32) or 8-byte (BF16) aligned, caches 4-byte, v_scale
 * 16-byte aligned, else PA_ERR_INVALID.
 * ------------------------------------------------------------------------ */
PA_API pa_status pa_fp8_cache_quant_scatter(const void* key, const void* value, int in_dtype,
                                     void* key_cache, void* value_cache,
                                     const void* slot_mapping, int slot_type,
                                     float* key_scale_cache, const float* v_scale,
                                     const int32_t* token_batch, int num_batches,
                                     int64_t num_tokens, int num_head, int head_size,
                                     int64_t num_blocks, int block_size, int layout,
                                     int overlap_prologue, void* stream);

/* ------------------------------------------------------------------------
 * KV compress epilog, modes 0 and 1 ([KC] 功能说明, 计算公式 场景 1 and 场景 2,
 * 约束说明, kvCacheCol 的源码级解读). In place. For each row i < bs of x with
 * s = slot_mapping[i] (skipped if s < 0 or s >= block_num * block_size), the
 * cache row at byte offset (s / block_size) * block_stride +
 * (s % block_size) * head_dim receives, in this order:
 *   bytes [0, 128)           x[i][d-64 .. d) (the rope part) as BF16,
 *   bytes [128, 128 + d-64)  x[i][0 .. d-64) (the nope part) as E4M3 codes,
 *                            quantised in groups of 64: scale_g =
 *                            max|x_g| / 448 (FP32 IEEE division),
 *                            code = E4M3(x / scale_g) round-to-nearest-even,
 *                            saturating (all-zero group: scale 0, codes 0);
 *   then one scale per group: mode 0 BF16(scale_g) (2 bytes, little-endian);
 *   mode 1 one E8M0 byte k + 127 for the power of two 2^k used instead of
 *   scale_g: the one at or above scale_g with round_scale, the one at or
 *   below it (scale_g's exponent) without, k clamped to [-127, 127]; codes
 *   are E4M3(x / 2^k) (an all-zero group stores byte 0).
 * Other bytes of the row, and rows no slot names, are left unchanged.
 * cache       uint8, block_num blocks of block_stride bytes (>= block_size *
 *             head_dim; blocks need not be contiguous), rows of head_dim bytes.
 * head_dim    >= (d - 64) + 128 + (d - 64) / 64 * (2 or 1) bytes, rounded
 *             up to 32 for mode 0 (d = 256, mode 1: 323).
 * x           BF16 [bs, d], d a multiple of 64 in (64, 8192], 4-byte aligned.
 * slot_mapping int32 or int64 [bs] (slot_type); slots should be unique.
 * quant_group_size must be 64. quant_mode 2 (HiFloat8 rope, FP4 nope) returns
 * PA_ERR_UNSUPPORTED; other invalid arguments PA_ERR_INVALID.
 * ------------------------------------------------------------------------ */
PA_API pa_status pa_fp8_kv_compress_epilog(void* cache, int64_t block_num, int block_size,
                                    int64_t block_stride, int head_dim, const void* x,
                                    int64_t bs, int d, const void* slot_mapping, int slot_type,
                                    int quant_group_size, int quant_mode, int round_scale,
                                    void* stream);

/* ------------------------------------------------------------------------
 * Per-token quantiser ([PA] 量化策略: Query/Key per-token): each row of D
 * values gets dequant scale s = max|x| / 448 and codes E4M3(x / s)
 * (round-to-nearest-even, saturating; an all-zero row gives s = 0, codes 0).
 * x      FP32 or BF16 [rows, D];  codes  E4M3 [rows, D];  scale float [rows].
 * ------------------------------------------------------------------------ */
PA_API pa_status pa_fp8_quantize_rows(const void* x, int in_dtype, int64_t rows, int D,
                               void* codes, float* scale, void* stream);

/* ------------------------------------------------------------------------
 * Per-channel value scale ([PA] 量化策略: Value per-channel, maximum over
 * the sequence): v_scale[b][h][d] = max over the tokens of sequence b of
 * |v[t][h][d]|, divided by 448.
 * v           FP32 or BF16 [total_tokens, H, D], sequences concatenated.
 * cu_seqlens  int64 [B + 1] device array of token offsets (non-decreasing,
 *             cu_seqlens[0] = 0, cu_seqlens[B] = total_tokens).
 * v_scale     float [B, H, D] (written; also used as scratch).
 * ------------------------------------------------------------------------ */
PA_API pa_status pa_fp8_value_channel_scale(const void* v, int in_dtype,
                                     const int64_t* cu_seqlens, int B,
                                     int64_t total_tokens, int H, int D,
                                     float* v_scale, void* stream);

/* ------------------------------------------------------------------------
 * MLA sparse attention with FP8 anti-quantisation, decode ([MS] 核心参数与
 * KV Cache 布局, API 签名与 Decode / Prefill 差异, 计算流程：5 层嵌套循环,
 * 关键实现细节, 在线反量化与 Online Softmax 的实现细节). [MS] = the page
 * "PyPTO-Gym 算子实战：DeepSeek V32 MLA 的 Sparse Attention FP8 反量化算子
 * （Ascend 950PR）解析与验证".
 *
 * NQ query heads share one latent KV head (n_kv = 1) of 512 "nope" channels
 * (kv_lora_rank) plus 64 rope channels. For query token t = b*S1 + s and head
 * h, over the first cur = clamp(kv_act_seqs[b] - S1 + 1 + s, 0, topk)
 * entries of topk_indices[t], walked in tiles of s2_tile entries:
 *   idx  = topk_indices[t][j], a position in sequence b; the packed row
 *          block_table[b][idx / block_size] * block_size + idx % block_size
 *          of nope_cache is read (an entry outside [0, kv_act_seqs[b]) takes
 *          no part; a block id of -1 or outside [0, num_blocks) reads block 0)
 *   kn   = BF16(FP32(E4M3 code) * scale[channel / 128]), k = [kn, kr] (576)
 *   S_j  = ([q_nope, q_rope] . k_j) * softmax_scale           (FP32)
 *   per tile: m = max S_j, p_j = exp(S_j - m), l = sum p_j, P = BF16(p)
 *             o = P . kn                                       (FP32, 512)
 *   merge:    M' = max(M, m); O = O exp(M - M') + o exp(m - M');
 *             L = L exp(M - M') + l exp(m - M')    (the first tile sets them)
 *   out  = BF16(O / L); a token with no valid entry gets zeros.
 *
 * Arguments (device pointers):
 *   q_nope        BF16 [B*S1, NQ, 512], row t*NQ + h.
 *   q_rope        BF16 [B*S1, NQ, 64].
 *   nope_cache    bytes [num_blocks*block_size, row_bytes]: per row 512 E4M3
 *                 codes, 64 BF16 rope values, 4 FP32 scales (bytes 0..655);
 *                 the rest of the row is padding and is not read. row_bytes
 *                 >= 656 and a multiple of 16 ([MS] pads rows to 672); at
 *                 most 2^31 - 1 rows (PA_ERR_UNSUPPORTED otherwise). E4M3
 *                 NaN codes are out of contract.
 *   topk_indices  int32 [B*S1, topk].
 *   block_table   int32 [B, max_blocks_per_seq].
 *   kv_act_seqs   int32 [B]; only the entries the visible count lets through
 *                 are read, so the table needs no room past each sequence.
 *   out           BF16 [B*S1, NQ, 512].
 *   n_kv          1 (anything else is PA_ERR_UNSUPPORTED).
 *   NQ            a multiple of 64 (PA_ERR_UNSUPPORTED otherwise).
 *   s2_tile       128, the kernel's tile of selected entries (the tile is a
 *                 tuning knob on the page; it decides which keys share one
 *                 tile max, i.e. the BF16 rounding of P). Other values are
 *                 PA_ERR_UNSUPPORTED.
 *   status        device int, zeroed by the caller before the first call;
 *                 a wait inside the kernel that gives up (about 2 s) ORs a
 *                 non-zero bit into it and the output is undefined.
 * Alignment: q_nope, q_rope, nope_cache, out 16-byte aligned; status 4-byte.
 * B = 0 enqueues nothing. Nothing is allocated; the call is asynchronous on
 * `stream`.
 * ------------------------------------------------------------------------ */
PA_API pa_status pa_mla_sparse_decode(const void* q_nope, const void* q_rope,
                                      const void* nope_cache, int64_t row_bytes,
                                      const int32_t* topk_indices,
                                      const int32_t* block_table,
                                      const int32_t* kv_act_seqs, void* out,
                                      int B, int S1, int NQ, int n_kv, int topk,
                                      int block_size, int64_t num_blocks,
                                      int max_blocks_per_seq, float softmax_scale,
                                      int s2_tile, int* status, void* stream);

/* ------------------------------------------------------------------------
 * The MLA sparse decode above over cache rows that pa_fp8_kv_compress_epilog
 * wrote with d = 576 (nope 512, rope 64): the decode side of the KV compress
 * epilog ("CANN ops-transformer aclnnKvCompressEpilog 算子详解", 计算公式
 * 场景 1 / 场景 2) read with [MS]'s dequantisation rule (在线反量化:
 * BF16(FP32(code) * scale)), each 64-channel group by its own scale.
 *
 * Row layout (bytes; the rest of the row is not used):
 *   [0, 128)    kr, 64 BF16 values;
 *   [128, 640)  kn, 512 E4M3 codes;
 *   quant_mode 0: [640, 656) eight BF16 scales s_g, one per 64 channels;
 *   quant_mode 1: [640, 648) eight E8M0 bytes e_g for s_g = 2^(e_g - 127)
 *                 (byte 255 is out of contract; the epilog writes <= 254).
 * kn[c] = BF16(FP32(E4M3 code c) * s_{c / 64}); everything else (gather,
 * visible count, masking, C1, tile-local softmax, BF16 P, C2, merge, output)
 * is the same as pa_mla_sparse_decode.
 *
 * Arguments: as pa_mla_sparse_decode, with
 *   kv_cache      bytes: num_blocks blocks of block_stride bytes, row r of a
 *                 block at r * row_bytes (the epilog's cache, block_stride and
 *                 head_dim); position idx of sequence b is row idx % block_size
 *                 of block block_table[b][idx / block_size].
 *   row_bytes     the epilog's head_dim, >= 656 and a multiple of 16 (mode 1
 *                 rows of the minimum 648 bytes do not qualify: pad to 656).
 *   block_stride  >= block_size * row_bytes and a multiple of 16; 0 means
 *                 block_size * row_bytes (contiguous blocks).
 *   quant_mode    0 or 1 as given to the epilog; 2 (HiFloat8 rope, FP4 nope)
 *                 returns PA_ERR_UNSUPPORTED, anything else PA_ERR_INVALID.
 * Nothing is allocated; the call is asynchronous on `stream`.
 * ------------------------------------------------------------------------ */
PA_API pa_status pa_mla_sparse_decode_kvc(const void* q_nope, const void* q_rope,
                                          const void* kv_cache, int64_t row_bytes,
                                          int64_t block_stride, int quant_mode,
                                          const int32_t* topk_indices,
                                          const int32_t* block_table,
                                          const int32_t* kv_act_seqs, void* out,
                                          int B, int S1, int NQ, int n_kv, int topk,
                                          int block_size, int64_t num_blocks,
                                          int max_blocks_per_seq, float softmax_scale,
                                          int s2_tile, int* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_FP8_H */
