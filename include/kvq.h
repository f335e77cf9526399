/*
 * kvq.h -- C ABI of libkvq: FP8 paged KV cache for NVIDIA GB300 (sm_103a).
 *
 * Two operations make the hot path of a quantized-KV-cache decoder:
 *
 *   kvq_write        quantize bf16 K/V with cast_fp8(x / s) and scatter the
 *                    codes into a paged cache ("10.4 KV Cache quantization:
 *                    INT8, KIVI 2-bit, FP8 KV", section 10.4.5; the INT8
 *                    analogue of the write is section 10.4.2).
 *   kvq_decode_attn  decode attention straight off that cache with the
 *                    dequantization fused in: P = softmax(Q K^T / sqrt(dh)),
 *                    O = P V^, K^ = cast_float(K_fp8) * sK, V^ likewise
 *                    (section 10.4.2 "efficient path", section 10.4.5).
 *
 * plus the unfused ablation (kvq_dequant_cache, section 10.4.2 "inefficient
 * path": a separate dequant kernel that materialises a bf16 cache) and the
 * host helpers that mirror the configuration surface described in the
 * "vLLM FP8 quantized KV cache guide" (kv_cache_dtype strings, per-tensor
 * and per-attention-head scales, skip layers).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All pointers passed to the compute calls are DEVICE pointers on the
 *   current CUDA device, except where a parameter says "host".  The caller
 *   owns every buffer (inputs, caches, scales, workspace, outputs, status).
 *   The library keeps no state between calls and allocates no device memory.
 * - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *   stream).  Calls do not synchronize and never read device memory on the
 *   host: scale values are only read on the device.
 * - Return value: KVQ_OK (0), or a negative kvq_status.  Host-detectable
 *   errors are returned BEFORE anything is enqueued.  KVQ_ERR_CUDA reports a
 *   launch error (cudaGetLastError after the launch).
 * - Device-detected bad indices (a slot past the cache, a block id outside
 *   [0, num_blocks), a sequence length outside [0, max_blocks_per_seq *
 *   block_size]) never trap: the offending work item is skipped (its tokens
 *   are masked out of attention, or not written) and a KVQ_DEV_* bit is OR-ed
 *   into *dev_status when dev_status is not NULL.  The caller reads the word
 *   after synchronizing.  Bounded waits inside the kernels that run out set
 *   KVQ_DEV_WAIT_TIMEOUT and the kernel returns early.
 * - Cache layout, per layer and per tensor (K and V separately):
 *     [num_blocks][num_kv_heads][block_size][head_dim]
 *   elements are uint8 FP8 codes (fmt E4M3 / E5M2) or bf16 (fmt BF16, the
 *   layout used for layers skipped from quantization).  A token at slot s
 *   lives in block s / block_size at offset s % block_size.
 * - Supported shapes: head_dim in {64, 128}; block_size == 16;
 *   num_q_heads % num_kv_heads == 0 with num_q_heads / num_kv_heads <= 8.
 *   All device pointers must be 16-byte aligned.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* kvq_stream_t;

/* Cache element format (the kv_cache_dtype of the layer). */
typedef enum {
  KVQ_FMT_BF16 = 0, /* not quantized: bf16 cache ("auto" for a bf16 model)  */
  KVQ_FMT_E4M3 = 1, /* FP8 E4M3 (OCP, max 448, no inf); "fp8" is an alias   */
  KVQ_FMT_E5M2 = 2  /* FP8 E5M2 (OCP, max 57344)                            */
} kvq_fmt;

/* Scale granularity: per tensor (shape [1]), per attention head (k/v scale
 * shape [num_kv_heads], q scale shape [num_q_heads]), or per (token, KV head)
 * ("10.4 KV Cache quantization", section 10.4.3, per-token granularity):
 * k/v scale caches [num_blocks][num_kv_heads][block_size] fp32 beside the
 * pages, written by kvq_write_token_head. */
typedef enum {
  KVQ_SCALE_PER_TENSOR = 0,
  KVQ_SCALE_PER_HEAD = 1,
  KVQ_SCALE_PER_TOKEN_HEAD = 2
} kvq_gran;

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_NULL = -1,        /* a required pointer is NULL                         */
  KVQ_ERR_SHAPE = -2,       /* inconsistent sizes, or a scale length off its shape */
  KVQ_ERR_ALIGN = -3,       /* a pointer or stride is not 16-byte aligned         */
  KVQ_ERR_UNSUPPORTED = -4, /* head_dim, block_size, group size, fmt or flag      */
  KVQ_ERR_WORKSPACE = -5,   /* workspace smaller than kvq_decode_workspace_size   */
  KVQ_ERR_CUDA = -6,        /* CUDA runtime error at launch                       */
  KVQ_ERR_ARG = -7          /* other invalid argument (negative count, bad enum)  */
} kvq_status;

/* Bits OR-ed into *dev_status by the kernels. */
#define KVQ_DEV_BAD_SLOT 1u     /* slot >= num_blocks * block_size: token not written */
#define KVQ_DEV_BAD_BLOCK 2u    /* block id outside [0, num_blocks): page masked out  */
#define KVQ_DEV_BAD_SEQLEN 4u   /* seq_len < 0 or > max_blocks_per_seq * block_size   */
#define KVQ_DEV_WAIT_TIMEOUT 8u /* a bounded pipeline wait ran out; output is invalid */
#define KVQ_DEV_INTERNAL 16u    /* an internal index guard failed (bits 16..31 name it); */
                                /* the access was skipped and the output is invalid      */
#define KVQ_DEV_BAD_QLEN 32u    /* prefill: a chunk longer than max_q_len; its rows past */
                                /* the first max_q_len (rounded up to whole tiles) were  */
                                /* not written                                           */

/* Bytes at the start of every decode workspace that must be zero before the
 * first call: the arrival counters of kvq_decode_attn, one 32-bit word per
 * (sequence, KV head), in a fixed-size table whatever the batch shape. */
#define KVQ_WS_COUNTER_BYTES ((size_t)65536 * 4u)

/* Flags of kvq_decode_attn. */
#define KVQ_Q_FP8 1u /* FP8-domain attention: Q quantized with q_scale; see kvq_decode_attn */
#define KVQ_CACHE_READY 2u /* start before the preceding kernel ends; see kvq_decode_attn */

/*
 * kvq_write -- quantize and scatter K and V into the paged cache.
 *
 * For every token t with slot = slot_mapping[t] >= 0, every KV head h and
 * every d < head_dim:
 *   k_cache[slot / bs][h][slot % bs][d] = cast_fp8(float(k[t][h][d]) / sK[h])
 * and likewise for V with sV.  The quotient is the IEEE binary32 quotient
 * (round to nearest even); cast_fp8 rounds to nearest even and saturates
 * finite overflow and +-inf to +-max ("10.4 KV Cache quantization",
 * section 10.4.5: cast_fp8(K / sK) is stored).  With fmt == KVQ_FMT_BF16 the
 * bf16 bits are copied unchanged and the scales are ignored (may be NULL).
 *
 *   k, v            bf16 [num_tokens][num_kv_heads][head_dim], consecutive
 *                   tokens `token_stride` elements apart (token_stride >=
 *                   num_kv_heads * head_dim, a multiple of 8).
 *   slot_mapping    int64 [num_tokens]; negative = padding, skipped.
 *                   Slots must be distinct (duplicates race).
 *   k_cache,v_cache the layer's caches, layout above, num_blocks blocks.
 *   k_scale,v_scale fp32 device arrays of k_scale_len / v_scale_len floats:
 *                   1 for KVQ_SCALE_PER_TENSOR, num_kv_heads for
 *                   KVQ_SCALE_PER_HEAD; values finite and > 0.
 *   dev_status      optional (NULL allowed); receives KVQ_DEV_BAD_SLOT.
 * num_tokens == 0 is a no-op.
 */
KVQ_API int kvq_write(const void* k, const void* v, int64_t token_stride, const int64_t* slot_mapping,
              int64_t num_tokens, int num_kv_heads, int head_dim, void* k_cache, void* v_cache,
              int64_t num_blocks, int block_size, const float* k_scale, int k_scale_len,
              const float* v_scale, int v_scale_len, int scale_granularity, int fmt,
              uint32_t* dev_status, kvq_stream_t stream);

/*
 * kvq_write_token_head -- quantize and scatter with per-(token, KV head)
 * scales ("10.4 KV Cache quantization", section 10.4.3: one scale per token
 * along dh, so every new token is quantized on its own and appended; vLLM's
 * fp8_per_token_head).  Each written row k[t][h][:] gets
 *   s = amax / fmt_max   (amax = largest magnitude among the row's finite
 *                         values, NaN and +-inf ignored; binary32 division;
 *                         fmt_max = 448 for E4M3, 57344 for E5M2),
 * s = 1 where that quotient is 0, stored at
 *   k_scale_cache[slot / bs][h][slot % bs],
 * and its codes are cast_fp8(float(x) / s) exactly as kvq_write forms them
 * (V likewise).  The row's largest finite value thus lands on the format's
 * largest code.  kvq_decode_attn and kvq_dequant_cache read the scale caches
 * with scale_granularity KVQ_SCALE_PER_TOKEN_HEAD.
 *
 *   k, v, slot_mapping, caches   as for kvq_write.
 *   k_scale_cache, v_scale_cache fp32 [num_blocks][num_kv_heads][block_size],
 *                   16-byte aligned; only the written rows' entries change.
 *   fmt             KVQ_FMT_E4M3 or KVQ_FMT_E5M2 (BF16: KVQ_ERR_UNSUPPORTED).
 * Cache metadata: 4 bytes per row beside dh code bytes (264 bytes per
 * (token, KV head) at dh = 128 for K and V together, against 512 in bf16).
 */
KVQ_API int kvq_write_token_head(const void* k, const void* v, int64_t token_stride,
                                 const int64_t* slot_mapping, int64_t num_tokens,
                                 int num_kv_heads, int head_dim, void* k_cache, void* v_cache,
                                 int64_t num_blocks, int block_size, float* k_scale_cache,
                                 float* v_scale_cache, int fmt, uint32_t* dev_status,
                                 kvq_stream_t stream);

/*
 * kvq_calibrate_scales -- per-tensor or per-KV-head scales from the data
 * ("vLLM FP8 quantized KV cache guide", scale calibration, way two: scales
 * estimated from statistics of the K/V activations).  The statistic is the
 * absolute maximum over the finite values of the given tokens (NaN and +-inf
 * are ignored), of one KV head or of the whole tensor:
 *   s = amax / fmt_max   (binary32 division, round to nearest even;
 *                         fmt_max = 448 for E4M3, 57344 for E5M2),
 * and s = 1 where that quotient is 0.  Quantizing the same tokens with s
 * (kvq_write) maps amax onto the format's largest finite value.
 *
 *   k, v            bf16 [num_tokens][num_kv_heads][head_dim], consecutive
 *                   tokens token_stride elements apart (as for kvq_write).
 *   k_scale,v_scale fp32 device arrays, outputs: 1 float for
 *                   KVQ_SCALE_PER_TENSOR, num_kv_heads for KVQ_SCALE_PER_HEAD
 *                   (4-byte aligned).  Overwritten on the stream (three
 *                   kernels: zero, reduce, divide).
 *   fmt             KVQ_FMT_E4M3 or KVQ_FMT_E5M2 (else KVQ_ERR_UNSUPPORTED).
 *   dev_status      optional; an internal guard bit if a load index fails.
 * num_tokens == 0 gives scales of 1.
 */
KVQ_API int kvq_calibrate_scales(const void* k, const void* v, int64_t token_stride,
                                 int64_t num_tokens, int num_kv_heads, int head_dim,
                                 int scale_granularity, int fmt, float* k_scale, float* v_scale,
                                 uint32_t* dev_status, kvq_stream_t stream);

/*
 * kvq_decode_workspace_size -- bytes of device workspace kvq_decode_attn
 * needs for these sizes.  num_sms <= 0 queries the current device (the value
 * depends on the device's SM count).  Returns 0 for invalid sizes.
 */
KVQ_API size_t kvq_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int num_sms);

/*
 * kvq_decode_attn -- grouped-query decode attention over the paged cache,
 * dequantization fused ("10.4 KV Cache quantization", section 10.4.2:
 * P = softmax(Q K^T / sqrt(dh) + mask), O = P V^; section 10.4.5:
 * K^ = cast_float(K_fp8) * sK).
 *
 * Sequence b attends to its tokens [lo_b, L_b), L_b = seq_lens[b] (the
 * token being decoded included, so write it first on the same stream) and
 * lo_b = L_b - sliding_window when 0 < sliding_window < L_b, else 0.  Query
 * head h reads KV head h / (num_q_heads / num_kv_heads).  Token t of
 * sequence b lives in block block_tables[b][t / block_size].
 *
 *   q               bf16 [num_seqs][num_q_heads][head_dim], any finite values
 *                   (for the FP8 caches each head's query is scaled by a power
 *                   of two, exactly, before its f16 tensor-core conversion).
 *   block_tables    int32 [num_seqs][max_blocks_per_seq]; entries past
 *                   ceil(L_b / block_size) are never read.
 *   seq_lens        int32 [num_seqs]; 0 gives a zero output row.
 *   q_scale         fp32, q_scale_len 1 (KVQ_SCALE_PER_TENSOR) or
 *                   num_q_heads (KVQ_SCALE_PER_HEAD); 1 or num_q_heads
 *                   with KVQ_SCALE_PER_TOKEN_HEAD.  Used only with
 *                   KVQ_Q_FP8; otherwise optional and only shape-checked.
 *   k_scale,v_scale as for kvq_write (ignored and may be NULL for BF16);
 *                   with KVQ_SCALE_PER_TOKEN_HEAD the scale caches of
 *                   kvq_write_token_head (k/v_scale_len = num_blocks *
 *                   num_kv_heads * block_size, 16-byte aligned): token t of
 *                   head g uses the scale stored beside its row, the logit
 *                   x_t = q . K_codes_t * sK_t / sqrt(dh) and V^_t = V_t sV_t.
 *   sliding_window  0 = none.
 *   flags           KVQ_Q_FP8: the FP8-domain mode ("vLLM FP8 quantized KV
 *                   cache guide", FlashAttention 3 note: the query is
 *                   quantized to FP8 like K and V).  Each query value is
 *                   divided by its head's q_scale (binary32) and encoded in
 *                   the cache's FP8 format as kvq_write encodes K; QK^T then
 *                   runs on the FP8 codes (m16n8k32 FP8 MMA), the logits
 *                   scaled by sQ sK / sqrt(dh).  Needs an FP8 cache
 *                   (KVQ_ERR_UNSUPPORTED for BF16) and q_scale
 *                   (KVQ_ERR_NULL).
 *                   KVQ_CACHE_READY (combinable with KVQ_Q_FP8): the kernel
 *                   is launched as a
 *                   programmatic dependent of the kernel before it on the
 *                   stream.  Without the flag it waits for that kernel to
 *                   complete before reading anything.  With KVQ_CACHE_READY
 *                   it reads block_tables, seq_lens, k_scale, v_scale and
 *                   every cache page (with its per-token scales) except the
 *                   one holding each sequence's last token (L_b - 1) while
 *                   that kernel may still run,
 *                   and waits only before reading q or those last pages and
 *                   before writing anything: the caller promises that the
 *                   preceding kernel writes none of the early inputs (true
 *                   when it is the kvq_write of one new token per sequence,
 *                   or a decode of another layer).
 *   workspace       device scratch of at least
 *                   kvq_decode_workspace_size(num_seqs, ...) bytes, 256-byte
 *                   aligned.  Its first KVQ_WS_COUNTER_BYTES bytes are
 *                   per-(sequence, KV head) arrival counters: zero them
 *                   once before the first call (for instance
 *                   cudaMemsetAsync of the whole buffer); every completed
 *                   call leaves them zero again (re-zero after a
 *                   KVQ_DEV_WAIT_TIMEOUT).  The rest needs no initialisation.
 *                   Successive calls on one stream may share it (each call
 *                   writes it only after the kernel before it has completed,
 *                   with or without KVQ_CACHE_READY); calls that may run
 *                   concurrently on different streams must not.
 *   out             bf16 [num_seqs][num_q_heads][head_dim] (fp32
 *                   accumulation, round to nearest even).
 *   dev_status      optional; KVQ_DEV_BAD_BLOCK, KVQ_DEV_BAD_SEQLEN,
 *                   KVQ_DEV_WAIT_TIMEOUT.
 * Limits: num_seqs <= 4096; num_seqs * num_kv_heads <= 65536;
 * num_seqs * (max_blocks_per_seq + 16) * num_kv_heads < 2^31;
 * num_blocks * num_kv_heads * block_size < 2^31 (cache rows); beyond them
 * KVQ_ERR_UNSUPPORTED.
 */
KVQ_API int kvq_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                    int64_t num_blocks, int block_size, const float* q_scale, int q_scale_len,
                    const float* k_scale, int k_scale_len, const float* v_scale, int v_scale_len,
                    int scale_granularity, int fmt, int sliding_window, unsigned flags,
                    void* workspace, size_t workspace_bytes, void* out, uint32_t* dev_status,
                    kvq_stream_t stream);

/*
 * kvq_decode_attn_static -- kvq_decode_attn without a caller-provided
 * workspace.  The pages this library is written from have no counterpart of
 * this entry point; it exists for callers that cannot allocate device
 * memory: a plugin handed only input and output pointers by its host
 * program, with no allocator to call, or a serving loop whose device-memory
 * plan is fixed at start-up and which may not call cudaMalloc (it can block
 * until the device is idle) on the decode path.
 *
 * Same arguments, semantics and errors as kvq_decode_attn, minus workspace
 * and workspace_bytes; the caller still passes every input and the output.
 * The scratch is one array of KVQ_STATIC_SCRATCH_BYTES bytes compiled into
 * the library's device image: every GPU on which the library's device code
 * is loaded holds it until the process exits.  Sizes whose workspace
 * (kvq_decode_workspace_size) exceeds it return KVQ_ERR_WORKSPACE before
 * anything is enqueued.  Nothing is allocated: no cudaMalloc, cudaFree or
 * allocating library routine is called.
 *
 * The first call on a device, made with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) and keeps it; make that
 * first call before any stream capture.  All calls on a device share the
 * one array, which keeps the last call's contents.  Its counters start at
 * zero (device variables are zero-initialized when the library's device
 * code is loaded) and every completed call leaves them zero, so nothing
 * needs clearing unless a call reported KVQ_DEV_WAIT_TIMEOUT: then call
 * kvq_decode_static_reset before the next kvq_decode_attn_static on that
 * device.  Calls on one stream are ordered; calls that
 * may overlap on the GPU (different streams, or different host threads)
 * race on it: serialize them, or give each its own workspace through
 * kvq_decode_attn.
 */
#define KVQ_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
KVQ_API int kvq_decode_attn_static(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* seq_lens, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int head_dim, int64_t num_blocks,
                                   int block_size, const float* q_scale, int q_scale_len,
                                   const float* k_scale, int k_scale_len, const float* v_scale,
                                   int v_scale_len, int scale_granularity, int fmt,
                                   int sliding_window, unsigned flags, void* out,
                                   uint32_t* dev_status, kvq_stream_t stream);

/*
 * kvq_decode_static_reset -- clear the counter table (the first
 * KVQ_WS_COUNTER_BYTES bytes) of the current device's static scratch array,
 * asynchronously on `stream` (a cudaMemsetAsync on the array's own address:
 * nothing is allocated).  Needed only after a kvq_decode_attn_static call
 * reported KVQ_DEV_WAIT_TIMEOUT, whose aborted CTAs may leave counts behind;
 * enqueue it on the stream of the next static call, or order the two.
 * Returns KVQ_OK or KVQ_ERR_CUDA (no device, or the array's address could
 * not be looked up).
 */
KVQ_API int kvq_decode_static_reset(kvq_stream_t stream);

/*
 * kvq_prefill_attn -- prefill, chunked-prefill and prefix-hit attention over
 * the paged cache, dequantization fused ("10.4 KV Cache quantization",
 * section 10.4.2: prefill, decode and prefix-hit paths all read the same
 * compressed cache).  Sequence b holds L_b = seq_lens[b] tokens in the cache
 * (write the chunk's K/V first, on the same stream); its last
 * n_b = cu_q_lens[b+1] - cu_q_lens[b] tokens are the queries.  Query row
 * cu_q_lens[b] + j is the token at position pos = L_b - n_b + j and attends
 * to the tokens [lo, pos] of its sequence, lo = pos + 1 - sliding_window when
 * 0 < sliding_window <= pos, else 0:
 *   O = softmax(q K^T / sqrt(dh) over [lo, pos]) V^,  K^ = cast_float(K) sK.
 * The tokens before the chunk are a cached prefix (a prefix hit, or the
 * earlier chunks of a chunked prefill); n_b = 1 is the decode.
 *
 *   q               bf16 [num_q_tokens][num_q_heads][head_dim].  With the
 *                   FP8 caches each element is converted to f16 for the MMAs:
 *                   |q| must stay below 65504 (elements below 2^-24 flush to
 *                   zero).
 *   cu_q_lens       int32 [num_seqs + 1], device: 0 = cu_q_lens[0] <= ... <=
 *                   cu_q_lens[num_seqs] = num_q_tokens.
 *   max_q_len       host: an upper bound of every n_b (sets the grid; the
 *                   rows of a longer chunk past it are left unwritten and
 *                   KVQ_DEV_BAD_QLEN is raised).
 *   block_tables, seq_lens, caches, q_scale, k_scale, v_scale,
 *   scale_granularity, fmt   as for kvq_decode_attn, every granularity
 *                   included: KVQ_SCALE_PER_TOKEN_HEAD reads the scale caches
 *                   that kvq_write_token_head fills (a prefix hit on such a
 *                   cache); q_scale is read only with KVQ_Q_FP8.
 *   flags           0 or KVQ_Q_FP8 (FP8 caches only): each query element is
 *                   encoded to the cache's format as cast_fp8(q / sQ) and
 *                   attends as its decoded value times sQ, as in
 *                   kvq_decode_attn.
 *   out             bf16 [num_q_tokens][num_q_heads][head_dim].
 *   dev_status      optional; KVQ_DEV_BAD_BLOCK (page masked out),
 *                   KVQ_DEV_BAD_SEQLEN (L_b < n_b or L_b > max_blocks_per_seq
 *                   * block_size: the sequence's rows are zero),
 *                   KVQ_DEV_BAD_QLEN (n_b > max_q_len), KVQ_DEV_WAIT_TIMEOUT.
 * Group size num_q_heads / num_kv_heads in {1, 2, 4, 8}; num_seqs <= 65535.
 * No workspace.  The FP8 caches run one CTA per (sequence, KV head, one or
 * two tiles of 128 query rows -- two when that needs fewer waves of CTAs),
 * the bf16 cache one per 64 query rows; a short chunk over a long prefix
 * keeps few SMs busy.  Precision: each probability reaches the PV MMA as one
 * f16 (the decode uses two f16 parts), so an output element may differ from
 * exact arithmetic over the dequantized cache by up to 2^-12 times the
 * largest |V| the row attends to, beyond its bf16 rounding.
 */
KVQ_API int kvq_prefill_attn(const void* q, const int32_t* cu_q_lens, int64_t num_q_tokens,
                             int max_q_len, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, int max_blocks_per_seq,
                             const int32_t* seq_lens, int num_seqs, int num_q_heads,
                             int num_kv_heads, int head_dim, int64_t num_blocks,
                             int block_size, const float* q_scale, int q_scale_len,
                             const float* k_scale, int k_scale_len, const float* v_scale,
                             int v_scale_len, int scale_granularity, int fmt,
                             int sliding_window, unsigned flags, void* out,
                             uint32_t* dev_status, kvq_stream_t stream);

/*
 * kvq_dequant_cache -- the unfused path's separate dequant kernel
 * ("10.4 KV Cache quantization", section 10.4.2: read the quantized KV,
 * dequantize in an independent kernel, write a 16-bit KV back to HBM).
 * dst_bf16[i] = bf16(fp32(cast_float(src[i]) * s_h)) over the whole cache
 * [num_blocks][num_kv_heads][block_size][head_dim]; the product is rounded to
 * binary32 (exact whenever s_h is a power of two), then to bf16 (nearest
 * even).  kvq_decode_attn with fmt KVQ_FMT_BF16 then reads the result.
 * fmt must be E4M3 or E5M2; scale as for kvq_write, or with
 * KVQ_SCALE_PER_TOKEN_HEAD the scale cache of kvq_write_token_head
 * (scale_len = num_blocks * num_kv_heads * block_size; row r of the cache
 * uses scale[r]).
 */
KVQ_API int kvq_dequant_cache(const void* src, void* dst_bf16, int64_t num_blocks, int num_kv_heads,
                      int block_size, int head_dim, const float* scale, int scale_len,
                      int scale_granularity, int fmt, kvq_stream_t stream);

/*
 * Host helpers (no device work).
 *
 * kvq_parse_dtype: kv_cache_dtype string -> kvq_fmt ("vLLM FP8 quantized KV
 * cache guide", choosing kv_cache_dtype): "fp8" and "fp8_e4m3" -> E4M3,
 * "fp8_e5m2" -> E5M2, "auto" / "bfloat16" / "bf16" -> BF16 (this library's
 * model dtype).  Anything else -> KVQ_ERR_UNSUPPORTED; NULL -> KVQ_ERR_NULL.
 *
 * kvq_layer_fmt: the skip-layer rule of the same guide ("per-layer
 * exemption of quantization-sensitive layers"): a layer keeps the model
 * dtype (returns KVQ_FMT_BF16) when it is a sliding-window layer
 * (is_sliding != 0) and the skip list holds "sliding_window", or when the
 * decimal string of layer_idx is in the skip list; otherwise returns fmt.
 * skip is a host array of n_skip C strings.  Errors: KVQ_ERR_NULL,
 * KVQ_ERR_ARG (bad fmt / negative index or count).
 *
 * kvq_status_string: static text for a kvq_status.
 * kvq_version: 10000 * major + 100 * minor + patch.
 */
KVQ_API int kvq_parse_dtype(const char* s);
KVQ_API int kvq_layer_fmt(int fmt, int layer_idx, int is_sliding, const char* const* skip, int n_skip);
KVQ_API const char* kvq_status_string(int status);
KVQ_API int kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
