/*
 * kvq.h -- C ABI of libkvq: group-quantised KV-cache attention on GB300 (sm_103a).
 *
 * The method (source pages: 《分块稀疏注意力与KV Cache量化：长文本推理显存优化实践》,
 * xdnf.cn, here "P4"; and 《一只"兔子"如何搅动大模型推理赛道的底层逻辑》, m.xxqk.cn, "P1"):
 *   - the KV cache is stored as integer codes, quantised in groups of 32
 *     adjacent head_dim channels, each group with its own scale and zero point
 *     (P4 §2.4 "KV Cache分组量化"; group size 32 from the hook in P4 §3.2);
 *   - attention softmax(Q K^T / sqrt(d)) V (P1 §3.1) is computed tile by tile
 *     with an online softmax whose running max and normaliser are merged
 *     across tiles (P4 §2.2);
 *   - dequantisation happens inside the attention read, not as a separate pass
 *     (P4 §1.3);
 *   - prefill may skip whole key tiles with a block-sparse mask (P4 §1.3, §2.3).
 *
 * Conventions for every call:
 *   - Ownership: the caller owns every buffer.  The library never allocates or
 *     frees the caller's memory, never synchronises, and launches only on
 *     `stream` (a cudaStream_t; NULL = the legacy default stream).  All calls
 *     are asynchronous with respect to the host.  The one exception to "no
 *     allocation" is kvq_decode_step_host, which keeps up to 16 CUDA graphs
 *     (driver resources) to replay repeated steps; see that call.
 *   - Errors: argument problems are detected on the host; the call returns a
 *     status and launches nothing.  A failed launch returns KVQ_ERR_CUDA.
 *   - Device status: conditions only the device can see (non-finite input,
 *     fp16 scale overflow, a sequence length beyond capacity, a bounded wait
 *     that timed out) are written to the optional device word `dev_status`
 *     (first error wins; the caller zeroes it and reads it after its own
 *     synchronisation).  NULL disables the report.
 *   - bf16 tensors are raw 16-bit bfloat16 values; fp16 values are IEEE binary16.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned buffer, ... */
  KVQ_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. D not 64/128) */
  KVQ_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
  KVQ_ERR_WORKSPACE = 4,     /* workspace missing or too small */
  KVQ_ERR_TIMEOUT = 5,       /* (device) a bounded wait gave up */
  KVQ_ERR_NONFINITE = 6,     /* (device) non-finite input or fp16 overflow */
  KVQ_ERR_BOUNDS = 7         /* (device, libkvq_debug.so only) an index check failed; the access was skipped */
} kvq_status;

#define KVQ_GROUP 32          /* channels per quantisation group (P4 §3.2) */
#define KVQ_MAX_HKV 64        /* most KV heads a cache may have */
#define KVQ_TILE_TOKENS 64    /* cache capacity granularity */
#define KVQ_OUT_F32 0
#define KVQ_OUT_BF16 1

/*
 * A quantised KV cache (one for K, one for V).  Group quantisation of P4 §2.4:
 * per (sequence b, KV head h, token t, group g of 32 channels) one fp16 scale
 * s and one fp16 integer zero point z; each channel value x is stored as the
 * code c with x_hat = (c - z) * s.  Per-head bit-width (P4 §2.4: sensitive
 * heads keep more bits) is 8 (one code per byte) or 4 (two codes per byte,
 * even channel in the low nibble).
 *
 * Layout (fixed by the library; all device memory, 16-byte aligned):
 *   codes: one plane per KV head.  Planes of 8-bit heads come first, in head
 *          order, then planes of 4-bit heads, in head order.  A plane is
 *          [B][Tcap][D*bits/8] bytes, row-major.  kvq_cache_head_offset()
 *          gives a plane's byte offset; kvq_cache_codes_bytes() the total.
 *   sz:    [Hkv][B][Tcap][D/32] 32-bit words; low 16 bits = fp16 scale,
 *          high 16 bits = fp16 zero point.  kvq_cache_sz_bytes() is the size.
 * head_bits is a HOST array of Hkv entries, each 4 or 8; it must stay valid
 * for the duration of each call that takes the cache.  Tcap must be a
 * multiple of KVQ_TILE_TOKENS; D is 64 or 128.
 */
typedef struct kvq_cache {
  uint8_t* codes;
  uint32_t* sz;
  const int8_t* head_bits;
  int32_t B, Hkv, Tcap, D;
} kvq_cache;

/* Total bytes of the code planes / the scale-zero words; -1 on invalid shape. */
KVQ_API int64_t kvq_cache_codes_bytes(const kvq_cache* cache);
KVQ_API int64_t kvq_cache_sz_bytes(const kvq_cache* cache);
/* Byte offset of KV head h's code plane within `codes`; -1 on invalid input. */
KVQ_API int64_t kvq_cache_head_offset(const kvq_cache* cache, int32_t h);

/*
 * kvq_quantize -- quantise-on-write (P4 §2.4, group 32 per P4 §3.2).
 *
 * x: device bf16, element (b, h, t, d) at x[b*sx_b + h*sx_h + t*sx_t + d]
 *    (element strides; channels contiguous; every row 16-byte aligned), for
 *    b < dst->B, h < dst->Hkv, t < nt.
 * Writes cache positions t0 .. t0+nt-1 of every (b, h) of `dst`.
 * Per group of 32 channels, qmax = 2^bits - 1, all arithmetic IEEE fp32:
 *   lo = min(0, min x), hi = max(0, max x), r = hi - lo;
 *   r == 0: s = 1, z = 0, codes 0;
 *   else s = fp16 rounded up from r / qmax, z = clamp(rne(-lo / s), 0, qmax),
 *        c = clamp(rne(x / s) + z, 0, qmax)   (rne = round half to even).
 * A non-finite input or a scale beyond fp16 range reports KVQ_ERR_NONFINITE
 * in dev_status; that group's stored values are then unspecified.
 */
KVQ_API kvq_status kvq_quantize(const void* x, int64_t sx_b, int64_t sx_h, int64_t sx_t,
                        int32_t t0, int32_t nt, const kvq_cache* dst,
                        int32_t* dev_status, void* stream);

/*
 * Workspace bytes kvq_decode_attention needs for this shape on the CURRENT
 * device (the split count depends on its SM count).  0 on invalid shape.
 */
KVQ_API size_t kvq_decode_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D);

/*
 * kvq_decode_attention -- one query token per (sequence, query head) over the
 * quantised cache, dequantised inside the attention read (P4 §1.3), tiled
 * online softmax (P4 §2.2) split across CTAs, then a log-sum-exp merge.
 *
 * q:        device bf16 [B][Hq][D], contiguous, 16-byte aligned.
 * k, v:     caches with identical B, Hkv, Tcap, D and head_bits.
 * seq_lens: device int32 [B]; sequence b attends cache tokens 0 .. len_b-1.
 *           len_b == 0 gives a zero output row; len_b outside [0, Tcap]
 *           reports KVQ_ERR_INVALID_ARG in dev_status and is clamped.
 * Hq:       query heads; Hq % Hkv == 0 and Hq / Hkv <= 8.  Query head h
 *           reads KV head h / (Hq / Hkv).
 * softmax_scale: multiplies Q.K; <= 0 selects 1/sqrt(D).
 * out:      device [B][Hq][D], fp32 (out_dtype KVQ_OUT_F32) or bf16 (KVQ_OUT_BF16).
 * workspace: device scratch of >= kvq_decode_workspace_bytes(B, Hq, Hkv, D)
 *           bytes, 16-byte aligned.  Zero-fill it once before its first use
 *           (e.g. cudaMemsetAsync): it holds per-segment arrival counters that
 *           every successful call leaves at zero again.  After a call that
 *           reported a device error, zero-fill it again.  Calls that share a
 *           workspace must be ordered on the GPU.
 * q values must lie within fp16 range (|q| < 65504): the kernel's tensor-core
 * products take Q in fp16 (exact for bf16 values in that range).
 */
KVQ_API kvq_status kvq_decode_attention(const void* q, const kvq_cache* k, const kvq_cache* v,
                                const int32_t* seq_lens, int32_t Hq, float softmax_scale,
                                void* out, int32_t out_dtype,
                                void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, void* stream);

/*
 * kvq_prefill_attention -- prefill (causal or not) over a group-quantised KV cache.
 *
 * Quantises K and V into k_cache / v_cache (positions 0 .. S-1, exactly as
 * kvq_quantize), then computes, per query head h and query position i,
 *   O[i] = softmax_j(scale * Q[i] . K_hat[j]) V_hat[j]
 * over keys j <= i when causal == 1 (P1 §3.1 with the causal rule), over all
 * keys j < S when causal == 0, where K_hat, V_hat are the dequantised cache
 * rows, tile by tile with an online softmax (P4 §2.2).
 * With a tile mask (P4 §1.3, §2.3: skipped blocks are not computed), an
 * off-diagonal key tile kt of query tile qt takes part only if
 * tile_mask[qt * nT + kt] != 0, where nT = S / tile; the keys of a skipped
 * tile are left out of the softmax.  Causal prefill reads only kt < qt of the
 * mask; non-causal reads every off-diagonal entry.  Diagonal tiles are always
 * computed (element-wise causal rule when causal == 1, whole when 0).
 *
 * q:    device bf16 [B][Hq][S][D]; k, v: device bf16 [B][Hkv][S][D];
 *       contiguous, 16-byte aligned.
 * causal 0 or 1; tile must be 128; S a multiple of 128; D 64 or 128;
 * Hq % Hkv == 0; caches with any per-head bits (8 or 4, e.g. from
 * kvq_allocate_head_bits), Tcap >= S.
 * tile_mask: device uint8 [nT][nT] or NULL (every tile kept); with a mask,
 *       nT * nT must stay below 2^31 (S up to 5,931,520), else
 *       KVQ_ERR_UNSUPPORTED.
 * out:  device [B][Hq][S][D], fp32 or bf16.
 */
KVQ_API kvq_status kvq_prefill_attention(const void* q, const void* k, const void* v,
                                 int32_t B, int32_t Hq, int32_t Hkv, int32_t S, int32_t D,
                                 int32_t causal, float softmax_scale,
                                 const uint8_t* tile_mask, int32_t tile,
                                 const kvq_cache* k_cache, const kvq_cache* v_cache,
                                 void* out, int32_t out_dtype,
                                 int32_t* dev_status, void* stream);

/*
 * kvq_head_error_stats -- per-head quantisation-error statistics, the input
 * of a sensitivity-driven per-head bit allocation (P4 §2.4: every attention
 * head gets a sensitivity score; sensitive heads are stored at the higher
 * bit-width, the rest at the lower one).
 *
 * For each head h, with x_hat the dequantised value that kvq_quantize would
 * store at `bits` bits (the same codes, bit for bit):
 *   stats[h][0] = sum_{b, t < len_b} w[b][h][t] * sum_d (x - x_hat)^2
 *   stats[h][1] = sum_{b, t < len_b} w[b][h][t] * sum_d x^2
 * x:        device bf16 [B][H][T][D], contiguous, 16-byte aligned; D 64 or 128.
 * seq_lens: device int32 [B] or NULL (every sequence T tokens); tokens
 *           t >= len_b are left out.
 * weights:  device float [B][H][T] or NULL (1): a per-token attention mass,
 *           expected >= 0.
 * bits:     4 or 8.
 * stats:    device double [H][2], written whole.
 * workspace: device, at least kvq_head_error_stats_workspace_bytes(H) bytes,
 *           16-byte aligned, else KVQ_ERR_WORKSPACE.
 * The sums are fp32 within a 32-channel group and fp64 beyond it, in an order
 * fixed by the sizes and the device (the same result on every call).
 * Non-finite input reports KVQ_ERR_NONFINITE in dev_status.  Two launches.
 */
KVQ_API size_t kvq_head_error_stats_workspace_bytes(int32_t H);
KVQ_API kvq_status kvq_head_error_stats(const void* x, int32_t B, int32_t H, int32_t T, int32_t D,
                                const int32_t* seq_lens, const float* weights, int32_t bits,
                                double* stats, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, void* stream);

/*
 * kvq_allocate_head_bits -- per-head bit-widths from K and V error statistics
 * (host function; P4 §2.4, and P4 §3.4: keeping more heads at high precision
 * trades compression, about 4x down to 2.5x, for accuracy).
 *
 * score[h] = k_stats[h][0] / k_stats[h][1] + v_stats[h][0] / v_stats[h][1]
 * (a term with a zero norm counts 0): the relative error of the head's K and
 * V at the low bit-width.  The n_high heads with the largest scores get 8
 * bits, ties going to the smaller head index; the others get low_bits.
 * k_stats, v_stats: host double [H][2] (kvq_head_error_stats, copied back);
 * head_bits: host int8 [H], written; score: host double [H] or NULL.
 * 0 <= n_high <= H; low_bits 4 or 8.  A non-finite score returns
 * KVQ_ERR_NONFINITE and writes nothing.
 */
KVQ_API kvq_status kvq_allocate_head_bits(const double* k_stats, const double* v_stats, int32_t H,
                                  int32_t n_high, int32_t low_bits, int8_t* head_bits, double* score);

/*
 * kvq_prefill_attention_varlen -- kvq_prefill_attention over a batch of
 * sequences of different lengths, padded to S.
 *
 * seq_lens: device int32 [B], sequence b's length L_b (0 <= L_b <= S; a value
 *   outside that range reports KVQ_ERR_INVALID_ARG in dev_status and is
 *   clamped).  Rows i < L_b of q, k, v hold the sequence; rows L_b .. S-1 are
 *   padding and are never read into the result (they may hold anything,
 *   non-finite values included).
 * Cache positions 0 .. L_b-1 get the codes kvq_quantize would write;
 * positions from L_b to the end of its 128-token tile are cleared (codes and
 * scale/zero words 0); positions past that keep their contents.  Output rows
 * i < L_b are the attention of query i over keys j <= i (causal == 1) or
 * j < L_b (causal == 0), with the tile mask as in kvq_prefill_attention;
 * rows L_b .. S-1 of out are written as zeros.  Query tiles wholly past L_b
 * cost one store of zeros.  Other arguments, layouts and errors as in
 * kvq_prefill_attention.
 */
KVQ_API kvq_status kvq_prefill_attention_varlen(const void* q, const void* k, const void* v,
                                        int32_t B, int32_t Hq, int32_t Hkv, int32_t S, int32_t D,
                                        const int32_t* seq_lens, int32_t causal, float softmax_scale,
                                        const uint8_t* tile_mask, int32_t tile,
                                        const kvq_cache* k_cache, const kvq_cache* v_cache,
                                        void* out, int32_t out_dtype,
                                        int32_t* dev_status, void* stream);

/*
 * kvq_build_tile_mask -- a block-sparse tile mask for kvq_prefill_attention
 * (P4 §2.3: tiles judged unnecessary are skipped, the skipped share capped so
 * that no query block is starved), built on the GPU.
 *
 * mask: device uint8 [nT][nT], written whole.  For query tile qt the
 *   candidates are key tiles kt in [1, qt); the row skips
 *   floor(max(qt - 1, 0) * skip_num / skip_den) of them (0 <= skip_num <=
 *   skip_den; integer arithmetic, so each row's cap is exact): those with the
 *   smallest keys SplitMix64(seed, qt * nT + kt + 1) -- output number
 *   qt * nT + kt + 1 of the SplitMix64 generator (Steele, Lea and Flood,
 *   2014) seeded with `seed` -- ties to the smaller kt.  Entries are 1 for kept
 *   tiles, key tile 0 and the diagonal, 0 for skipped tiles and above the
 *   diagonal.  1 <= nT <= 16384.  One launch on `stream`.
 */
KVQ_API kvq_status kvq_build_tile_mask(uint8_t* mask, int32_t nT, int32_t skip_num, int32_t skip_den,
                                       uint64_t seed, void* stream);

/*
 * kvq_decode_attention_noalloc -- kvq_decode_attention for callers that may
 * not allocate device memory (for example code running inside another
 * framework's memory pool, or a plugin whose host forbids cudaMalloc at call
 * time).  The source pages have no counterpart to this call.
 *
 * Arguments and results are those of kvq_decode_attention, minus the
 * workspace: the split scratch is a fixed array of 4 MiB compiled into the
 * library, present on every GPU that loads it until the process exits.  A
 * shape whose kvq_decode_workspace_bytes() exceeds 4 MiB returns
 * KVQ_ERR_WORKSPACE and launches nothing.  The call allocates nothing; it
 * clears the array's arrival counters with an asynchronous memset on `stream`
 * before the decode launch.
 *
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * Every call on a device shares the one array, so calls whose executions
 * overlap on the GPU (different streams, no ordering between them) race and
 * give wrong results; order them.
 */
KVQ_API kvq_status kvq_decode_attention_noalloc(const void* q, const kvq_cache* k, const kvq_cache* v,
                                                const int32_t* seq_lens, int32_t Hq, float softmax_scale,
                                                void* out, int32_t out_dtype,
                                                int32_t* dev_status, void* stream);

/*
 * kvq_decode_step -- one step of a decode loop over the quantised cache (the
 * decode phase of P4 §1.3: each new token's K/V is quantised on write, then
 * the new query attends the cache with dequantisation inside the read).
 *
 * Appends the new token of every (sequence b, KV head) to both caches at
 * position seq_lens[b] - 1, quantised exactly as kvq_quantize writes it, then
 * computes kvq_decode_attention over positions 0 .. seq_lens[b] - 1.
 *
 * k_new, v_new: device bf16 [B][Hkv][D], contiguous, 16-byte aligned.
 * seq_lens: device int32 [B], each length INCLUDING the new token.  A length
 *           outside [1, Tcap] reports KVQ_ERR_INVALID_ARG in dev_status and
 *           that sequence appends nothing (decode then treats the length as
 *           kvq_decode_attention does).
 * q, k, v, Hq, softmax_scale, out, out_dtype, workspace, dev_status, stream:
 *           as kvq_decode_attention; the workspace is required.
 * Two launches on `stream`: the append kernel (K and V together) and the
 * decode kernel, whose prologue overlaps the append kernel's end
 * (programmatic dependent launch); the decode waits for the append before
 * reading memory.  All arguments are checked before the first launch.
 */
KVQ_API kvq_status kvq_decode_step(const void* q, const void* k_new, const void* v_new,
                                   const kvq_cache* k, const kvq_cache* v, const int32_t* seq_lens,
                                   int32_t Hq, float softmax_scale, void* out, int32_t out_dtype,
                                   void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                   void* stream);

/*
 * Device staging bytes kvq_decode_step_host needs: q, k_new, v_new and the
 * output, each rounded up to 256 bytes.  0 on invalid shape.
 */
KVQ_API size_t kvq_decode_step_staging_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t out_dtype);

/*
 * kvq_decode_step_host -- kvq_decode_step with the step's inputs and output in
 * HOST memory: q_host bf16 [B][Hq][D], k_new_host / v_new_host bf16
 * [B][Hkv][D], out_host [B][Hq][D] of out_dtype, all 16-byte aligned.
 * When all four host buffers are pinned (page-locked, so mapped into the
 * GPU's address space) the call makes no copy calls: the append launch reads
 * the new K/V rows in place over the host link and stages q in `staging`,
 * and the decode launch writes the output straight into out_host.  Otherwise
 * it enqueues three host-to-device copies into `staging`, the two launches of
 * kvq_decode_step and a device-to-host copy of the output (with pageable
 * memory the copies may block the host).  Either way everything goes to
 * `stream` and the call returns once it is enqueued; out_host holds the
 * result after the caller synchronises the stream, and the host inputs and
 * `staging` must stay untouched until then.
 * Repeated steps (pinned buffers): the second call whose arguments all match
 * an earlier call's -- every pointer and size, Hq, softmax_scale, out_dtype,
 * both caches' fields and per-head bit widths, the current device -- captures
 * the two launches into a CUDA graph on an internal stream, and every later
 * matching call launches that graph on `stream` (one launch call, no
 * tensor-map encoding).  The kernels read the lengths, the new rows and the
 * caches at run time, so those may change between calls.  Up to 16 graphs
 * are kept for the life of the process; other steps launch directly, and so
 * does any call on a stream that is being captured.
 * staging: device scratch of >= kvq_decode_step_staging_bytes(B, Hq, Hkv, D,
 * out_dtype) bytes, 256-byte aligned.  The caches, seq_lens, workspace and
 * dev_status are device memory as in kvq_decode_step.
 */
KVQ_API kvq_status kvq_decode_step_host(const void* q_host, const void* k_new_host, const void* v_new_host,
                                        const kvq_cache* k, const kvq_cache* v, const int32_t* seq_lens,
                                        int32_t Hq, float softmax_scale, void* out_host, int32_t out_dtype,
                                        void* staging, size_t staging_bytes,
                                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                        void* stream);

/*
 * Paged caches: the block-table layout of the serving systems the pages
 * compare against (PagedAttention with an INT8 cache), here for the
 * group-quantised cache.  A page POOL is a kvq_cache whose B counts pages and
 * whose Tcap is KVQ_TILE_TOKENS (64): page p holds 64 consecutive tokens of
 * one sequence, in every head's code plane and in the scale/zero words, in
 * exactly the kvq_cache layout.  A block table maps sequence b's token t to
 * page pages[b * max_pages + t / 64], slot t % 64.  Pages are the caller's to
 * allocate; two sequences may share a page only while no call writes it.
 */
typedef struct kvq_block_table {
  const int32_t* pages;   /* device int32 [B][max_pages], 4-byte aligned */
  int32_t B;              /* sequences */
  int32_t max_pages;      /* pages per sequence: capacity max_pages * 64 tokens */
} kvq_block_table;

/*
 * kvq_quantize into a page pool: x's rows are (sequence b < table->B, KV
 * head, position t0 + t) with the strides of kvq_quantize, and each row is
 * written to its page and slot, quantised exactly as kvq_quantize does.
 * t0 + nt <= max_pages * 64.  A page id outside [0, pool->B) reports
 * KVQ_ERR_INVALID_ARG in dev_status and that row is not written.
 */
KVQ_API kvq_status kvq_quantize_paged(const void* x, int64_t sx_b, int64_t sx_h, int64_t sx_t,
                                      int32_t t0, int32_t nt, const kvq_cache* pool,
                                      const kvq_block_table* table, int32_t* dev_status, void* stream);

/*
 * kvq_decode_attention over page pools: q [table->B][Hq][D]; sequence b
 * attends its tokens 0 .. seq_lens[b] - 1 through the block table
 * (seq_lens[b] <= max_pages * 64, else KVQ_ERR_INVALID_ARG in dev_status and
 * the length is clamped).  A page id outside the pool reports
 * KVQ_ERR_INVALID_ARG and that tile reads page 0 instead.  The workspace is
 * kvq_decode_workspace_bytes(table->B, Hq, Hkv, D).  Other arguments as
 * kvq_decode_attention.
 */
KVQ_API kvq_status kvq_decode_attention_paged(const void* q, const kvq_cache* k_pool, const kvq_cache* v_pool,
                                              const kvq_block_table* table, const int32_t* seq_lens,
                                              int32_t Hq, float softmax_scale, void* out, int32_t out_dtype,
                                              void* workspace, size_t workspace_bytes,
                                              int32_t* dev_status, void* stream);

/*
 * kvq_decode_step over page pools: the new token of sequence b goes to page
 * pages[b * max_pages + (seq_lens[b] - 1) / 64], slot (seq_lens[b] - 1) % 64,
 * then kvq_decode_attention_paged.  A length outside [1, max_pages * 64] or a
 * page id outside the pool reports KVQ_ERR_INVALID_ARG and that sequence
 * appends nothing.
 */
KVQ_API kvq_status kvq_decode_step_paged(const void* q, const void* k_new, const void* v_new,
                                         const kvq_cache* k_pool, const kvq_cache* v_pool,
                                         const kvq_block_table* table, const int32_t* seq_lens,
                                         int32_t Hq, float softmax_scale, void* out, int32_t out_dtype,
                                         void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                         void* stream);

/*
 * kvq_policy -- per-call settings for the two phases (P4 §5.3: prefill and
 * decode want different settings -- prefill has no history to re-read and is
 * compute-bound, so its tile mask may skip more; decode re-reads the whole
 * cache for every token and is memory-bound, so it gains from fetching the
 * cache further ahead).  The prefill phase's sparsity is its tile mask
 * (kvq_build_tile_mask's skip ratio); the decode phase's prefetch width is
 * set here.  kvq_policy_default() fills the values every other call uses.
 *
 *   decode_ring_tiles     64-token tiles of K and V that each decode CTA keeps
 *                         in flight into shared memory, 2 or 4 (default 4).
 *   decode_l2_warm_tiles  tiles per CTA requested into L2 before the decode
 *                         waits for the previous kernel in the stream to
 *                         finish, 0 .. 16 (default 5).
 *   wait_limit_us         every bounded wait inside the decode and prefill
 *                         kernels gives up after this long and reports
 *                         KVQ_ERR_TIMEOUT in dev_status, 1 .. 60,000,000
 *                         (default 2,000,000 = 2 s).
 *   test_issue_limit      FOR TESTS OF THE TIMEOUT PATH ONLY; negative (the
 *                         default) = off.  Decode: each CTA's copy issuer
 *                         streams only its first test_issue_limit tiles, so
 *                         the waits for the rest run out.  Prefill: 0
 *                         withholds the query load, so every role's first
 *                         wait runs out (other values: no effect).  Nothing
 *                         is left in flight; the call reports KVQ_ERR_TIMEOUT
 *                         and its outputs are unspecified.
 * An out-of-range field returns KVQ_ERR_INVALID_ARG and launches nothing.
 */
typedef struct kvq_policy {
  int32_t decode_ring_tiles;
  int32_t decode_l2_warm_tiles;
  uint32_t wait_limit_us;
  int32_t test_issue_limit;
} kvq_policy;

KVQ_API void kvq_policy_default(kvq_policy* policy);

/* kvq_decode_attention with a policy (NULL = kvq_policy_default). */
KVQ_API kvq_status kvq_decode_attention_ex(const void* q, const kvq_cache* k, const kvq_cache* v,
                                           const int32_t* seq_lens, int32_t Hq, float softmax_scale,
                                           void* out, int32_t out_dtype,
                                           void* workspace, size_t workspace_bytes,
                                           const kvq_policy* policy, int32_t* dev_status, void* stream);

/* kvq_prefill_attention_varlen with a policy (NULL = kvq_policy_default);
 * seq_lens may be NULL (every sequence S long, as kvq_prefill_attention). */
KVQ_API kvq_status kvq_prefill_attention_ex(const void* q, const void* k, const void* v,
                                            int32_t B, int32_t Hq, int32_t Hkv, int32_t S, int32_t D,
                                            const int32_t* seq_lens, int32_t causal, float softmax_scale,
                                            const uint8_t* tile_mask, int32_t tile,
                                            const kvq_cache* k_cache, const kvq_cache* v_cache,
                                            void* out, int32_t out_dtype, const kvq_policy* policy,
                                            int32_t* dev_status, void* stream);

/* Static, human-readable name of a status code. */
KVQ_API const char* kvq_status_str(kvq_status status);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
