/*
 * kvarn.h -- C ABI of the GB300 (sm_103a) KVarN 2-bit KV-cache library
 * (3- and 4-bit codes as options of the same format).
 *
 * KVarN stores the K and V caches at 2 bits per element without calibration
 * data: each block of tokens is rotated by a randomised Hadamard matrix over
 * head_dim, normalised along the token axis and the channel axis in turn
 * until both have unit variance, and quantised in 32-channel groups; the
 * scales are kept and applied again when the cache is read. Decode attention
 * reads the packed cache directly, with the query rotated by the same matrix
 * and the inverse rotation applied once to the output.
 *
 * Sources (page title, section):
 *   "KVarN: cuantizacion de KV-Cache normalizada por varianza mitiga la
 *    acumulacion de errores en tareas de razonamiento" -- English abstract:
 *    Hadamard rotation then dual-scaling variance normalisation over both
 *    axes of K and V, calibration-free, 2-bit.
 *   "KVarN：方差归一化让 2-bit KV 缓存扛住长链推理" -- section 三, 3.1
 *    (randomised Hadamard on K and V; q multiplied by the same matrix so
 *    Q K^T is unchanged) and 3.2 (token-axis then channel-axis variance to 1,
 *    repeated 2-3 times; grouped scales kept for dequantisation; statistics
 *    computed at decode time and fusable into the KV write kernel).
 *
 * Conventions for every entry point
 *   - Pointers marked "device" must be device memory of the current CUDA
 *     device; "host" pointers are host memory. Nothing is allocated, freed or
 *     synchronised by the library except where stated (kvarn_read_error).
 *   - stream is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). All device work is enqueued on it, in order.
 *   - The caller owns every buffer. Buffers written by a call must not be
 *     read or written by other work until that call's stream work completes.
 *   - Return value: KVARN_OK, or a negative kvarn_status when the arguments
 *     are rejected on the host (nothing enqueued) or a launch fails.
 *     Data-dependent faults found on the device (a block id outside the
 *     pool, a position beyond the block table, non-finite input, a wait that
 *     ran out of time) never trap: the kernel skips the affected unit and
 *     ORs a KVARN_DEVERR_* flag into the workspace error word, which
 *     kvarn_read_error returns. Outputs of a call that raised a flag are
 *     unspecified.
 *
 * Data layouts (little-endian; fp16/bf16 are IEEE binary16 / bfloat16)
 *   Head-block: one (physical block, kv head, K or V): B tokens x 128
 *   channels with `bits` (2, 3 or 4) bits per code, packed as (X = 16*bits*B)
 *     [0, X)             codes, in 8*bits-byte records (order below)
 *     [X, X+8B)          s: fp16 [4][B]   per (group, token) step
 *     [X+8B, X+16B)      z: fp16 [4][B]   per (group, token) zero (lowest level)
 *     [X+16B, X+18B)     R: fp16 [B]      per-token factor
 *     [X+18B, X+18B+256) C: fp16 [128]    per-channel factor
 *   = 1856 / 3456 bytes for 2 bits at B = 32 / 64, 2368 / 4480 for 3 bits,
 *   2880 / 5504 for 4 bits.
 *   The value of element (t, c) in the rotated space is
 *   (code * s[g][t] + z[g][t]) * R[t] * C[c] with g = c / 32 and code in
 *   0 .. 2^bits - 1. Code records: record r = 32*sb + 4a + b (sb = t / 32)
 *   holds 2*bits little-endian 32-bit words; a code sits at bit position p
 *   of word w of its record:
 *     kind K: a = (t%32)/4, i = t%4, g = c/32, b = (c%32)/8, e = c%8;
 *             2 bits: w = 2i + g/2, p = 2*(4*(g%2) + e/2) + 16*(e%2)
 *             4 bits: w = 4i + g,   p = 4*(e/2) + 16*(e%2)
 *     kind V: b = (t%32)/8, d = t%8, g = c/32, a = (c%32)/4, f = c%4;
 *             2 bits: w = 2g + f/2, p = 2*(4*(d/4) + 2*((d%4)/2) + f%2) + 16*(d%2)
 *             4 bits: w = 4g + f,   p = 4*(d/2) + 16*(d%2)
 *   3 bits: words 0..7 of a 12-word record hold each code's low two bits
 *           at its 2-bit (w, p); words 8..11 hold its high bit at word
 *           8 + w/2, bit 8*(w%2) + j + 16*h, where p = 2j + 16h
 *   (each lane of the attention kernel's warp reads exactly one record per
 *   32 tokens and turns it into tensor-core operands with one mask and one
 *   fp16 multiply per pair of codes).
 *   Pool: physical block p holds its head-blocks at
 *     pool + p*kvarn_block_bytes + (2*h + kind)*kvarn_head_block_bytes,
 *   kind 0 = K, 1 = V. pool must be 16-byte aligned.
 *   Staging (the incomplete tail block, raw unrotated values):
 *     bf16 [max_seqs][n_kv][2][B][128]; token t of sequence b is row t % B.
 *   Block table: int32 [batch][max_blocks_per_seq], logical -> physical.
 */
#ifndef KVARN_H_
#define KVARN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVARN_OK = 0,
    KVARN_ERR_INVALID_ARG = -1,   /* null/misaligned pointer, bad size or config field */
    KVARN_ERR_UNSUPPORTED = -2,   /* a valid config this build does not implement */
    KVARN_ERR_CUDA = -3,          /* a CUDA runtime call or launch failed */
    KVARN_ERR_WORKSPACE = -4      /* workspace_bytes below kvarn_workspace_bytes */
} kvarn_status;

/* device error word flags (sticky, OR-ed) */
#define KVARN_DEVERR_BLOCK_ID 0x1u      /* physical block id < 0 or >= n_pool_blocks */
#define KVARN_DEVERR_POSITION 0x2u      /* pos / seq_len outside [0, max_blocks*B] */
#define KVARN_DEVERR_NONFINITE 0x4u     /* NaN or Inf in a block being quantised */
#define KVARN_DEVERR_WAIT_TIMEOUT 0x8u  /* a shared-memory copy wait hit its limit */

typedef enum { KVARN_BF16 = 0, KVARN_FP32 = 1 } kvarn_dtype;
typedef enum { KVARN_KIND_K = 0, KVARN_KIND_V = 1 } kvarn_kind;

typedef struct kvarn_config {
    int32_t head_dim;       /* must be 128 */
    int32_t block_size;     /* tokens per block B: 32 or 64 */
    int32_t group_size;     /* channels per quantisation group: must be 32 */
    int32_t bits;           /* bits per code: 2 (the method), 3 or 4 */
    int32_t varn_iters;     /* VarN iterations (token pass then channel pass): 0..8 */
    int32_t n_q_heads;      /* query heads */
    int32_t n_kv_heads;     /* kv heads; n_q_heads / n_kv_heads in 1..4 */
    float sm_scale;         /* softmax scale; 0 means 1/sqrt(head_dim) */
    uint32_t sign_bits[4];  /* rotation signs: bit c set => channel c negated */
    uint32_t flags;         /* 0 for the method; KVARN_FLAG_* bits select an ablation */
} kvarn_config;

/*
 * Ablation switches (section 五 of the method page, its ablation list: the
 * full method against Hadamard only, VarN only, and VarN along one axis).
 * They change what is stored, so a cache must be read with the flags it was
 * written with. Hadamard only = flags 0 with varn_iters 0.
 *   KVARN_FLAG_NO_ROTATION      no Hadamard rotation (R = I): keys, values and
 *                               queries stay in the original space and the
 *                               output is not rotated back
 *   KVARN_FLAG_NO_TOKEN_PASS    VarN without its token-axis pass (R_t = 1)
 *   KVARN_FLAG_NO_CHANNEL_PASS  VarN without its channel-axis pass (C_c = 1)
 */
#define KVARN_FLAG_NO_ROTATION 0x1u
#define KVARN_FLAG_NO_TOKEN_PASS 0x2u
#define KVARN_FLAG_NO_CHANNEL_PASS 0x4u
/*
 * Test switch (no counterpart in the paper): with it, every warp of
 * kvarn_decode_attn's split kernel gives up its first shared-memory copy
 * wait at once, so the wait-timeout path runs without anything hanging:
 * KVARN_DEVERR_WAIT_TIMEOUT is raised, the copies already in flight are
 * waited for, the warp stops, the call's outputs are unspecified and the
 * workspace stays usable (clear the error word and call again). Ignored by
 * the other entry points; never set it outside tests.
 */
#define KVARN_FLAG_TEST_WAIT_TIMEOUT 0x100u

/* Library version string, e.g. "kvarn 0.1 sm_103a". */
const char* kvarn_version(void);

/* Human-readable text for a kvarn_status value. */
const char* kvarn_status_string(int status);

/* Bytes of one packed head-block: (16*bits + 18)*B + 256 (50*B + 256 at 2
 * bits). 0 for an invalid config. */
size_t kvarn_head_block_bytes(const kvarn_config* cfg);

/* Bytes of one physical block: n_kv_heads * 2 * kvarn_head_block_bytes. */
size_t kvarn_block_bytes(const kvarn_config* cfg);

/* Bytes of the bf16 staging buffer for max_seqs sequences:
 * max_seqs * n_kv * 2 * B * 128 * 2. */
size_t kvarn_staging_bytes(const kvarn_config* cfg, int32_t max_seqs);

/* Minimum workspace for kvarn_decode_attn / kvarn_decode_attn_bf16 with this
 * batch on the CURRENT device (the split-K partial results depend on its SM
 * count): 256 header bytes (the error word is the first uint32), one
 * partial (max, sum, 128 accumulators per query head) per (sequence, kv
 * head) and per resident warp, then 8 bytes per (sequence, kv head) in
 * which the split kernel records the first and last warp of each for the
 * merge. batch = 0 gives the 256 bytes that kvarn_quantize_block and
 * kvarn_append need. 0 on a bad config. */
size_t kvarn_workspace_bytes(const kvarn_config* cfg, int32_t batch, int32_t max_blocks_per_seq);

/* Workspace with which kvarn_prefill_attn runs at full speed for this batch
 * and chunk on the CURRENT device: at least kvarn_workspace_bytes(cfg,
 * batch * chunk, ...), and room for several partials per row when there are
 * too few (sequence, kv head, row tile) units to fill the GPU (2-bit caches;
 * the block split adapts to the workspace actually passed). 0 on a bad
 * config. */
size_t kvarn_prefill_workspace_bytes(const kvarn_config* cfg, int32_t batch, int32_t chunk,
                                     int32_t max_blocks_per_seq);

/*
 * kvarn_quantize_block -- bulk quantise-on-write of complete head-blocks
 * (prefill). Passage: abstract (rotation then dual-axis normalisation, 2-bit);
 * section 三 3.1-3.2 of the method page.
 *
 * For each n in [0, n_head_blocks): reads the B x 128 block
 *   src[n*src_block_stride + t*src_token_stride + c]  (elements, dtype
 *   src_dtype: KVARN_BF16 or KVARN_FP32; device)
 * rotates each token by H diag(sigma)/sqrt(128), runs varn_iters passes of
 * token-axis then channel-axis variance normalisation, rounds the factors to
 * fp16, quantises each (token, 32-channel group) to `bits` bits
 * (2^bits - 1 steps) with an fp16 step and zero, and writes one packed head-block of `kind` layout to
 *   dst_base + dst_offsets[n]   (bytes; device int64 array, NULL means
 *                               n * kvarn_head_block_bytes)
 * dst_base + offset must be 16-byte aligned. workspace: >= 256 bytes of
 * device memory whose first uint32 is the error word (KVARN_DEVERR_NONFINITE).
 */
int kvarn_quantize_block(const kvarn_config* cfg, int32_t kind, const void* src, int32_t src_dtype,
                         int64_t n_head_blocks, int64_t src_block_stride,
                         int64_t src_token_stride, void* dst_base, const int64_t* dst_offsets,
                         void* workspace, void* stream);

/*
 * kvarn_append -- one decode step's KV write (quantise-on-append). Passage:
 * section 三 3.2 of the method page (scales computed at decode time from the
 * data itself, fused into the KV write kernel).
 *
 * For each sequence b < batch and kv head h, the new token's K and V
 * (k_new, v_new: device bf16 [batch][n_kv][128]) are written to staging row
 * pos[b] % B (pos: device int32 [batch], the index of the new token, i.e.
 * the length before this step). When that row completes the block
 * (pos[b] % B == B - 1), the whole block is quantised exactly as
 * kvarn_quantize_block does and written to physical block
 * block_table[b][pos[b] / B] of the pool (n_pool_blocks blocks); the staging
 * rows are left as they are. Nothing is re-quantised later. Device faults:
 * KVARN_DEVERR_POSITION (pos < 0 or pos >= max_blocks_per_seq * B),
 * KVARN_DEVERR_BLOCK_ID, KVARN_DEVERR_NONFINITE.
 */
int kvarn_append(const kvarn_config* cfg, void* pool, int64_t n_pool_blocks, void* staging,
                 const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* pos,
                 const void* k_new, const void* v_new, int32_t batch, void* workspace,
                 void* stream);

/*
 * kvarn_decode_attn -- decode attention over the packed cache. Passage:
 * section 三 3.1 of the method page (the query is multiplied by the same
 * Hadamard matrix, so q.k is unchanged).
 *
 * q: device [batch][n_q][128], dtype q_dtype (KVARN_BF16 or KVARN_FP32).
 * seq_lens: device int32 [batch], tokens per sequence including the newest.
 * For query head j of sequence b (kv head h = j / (n_q / n_kv)):
 *   out[b][j][:] = sum_t softmax_t(sm_scale * q.k_t) v_t
 * over the first floor(L/B)*B tokens from the pool (dequantised on the fly)
 * and the remaining L % B tokens from staging (raw bf16). out: device fp32
 * [batch][n_q][128]. L = 0 gives zeros. workspace: device, at least
 * kvarn_workspace_bytes(cfg, batch, max_blocks_per_seq) bytes, 16-byte
 * aligned, passed as workspace_bytes. The work is split evenly over the
 * GPU's resident warps (split-K over each sequence's blocks) and merged by a
 * second kernel on the same stream. n_pool_blocks must be below 2^31
 * (KVARN_ERR_INVALID_ARG otherwise). Device faults: KVARN_DEVERR_BLOCK_ID,
 * KVARN_DEVERR_POSITION, KVARN_DEVERR_WAIT_TIMEOUT.
 */
int kvarn_decode_attn(const kvarn_config* cfg, const void* q, int32_t q_dtype, const void* pool,
                      int64_t n_pool_blocks, const void* staging, const int32_t* block_table,
                      int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch,
                      float* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * kvarn_prefill_attn -- chunked prefill attention over the same packed cache
 * (the pages describe only the decode step; this is its causal extension,
 * with the query multiplied by the same Hadamard matrix, section 三 3.1).
 *
 * The last `chunk` tokens of every sequence have already been appended
 * (kvarn_append / kvarn_quantize_block); q: device [batch][chunk][n_q][128]
 * (q_dtype KVARN_BF16 or KVARN_FP32) holds their queries. Query row r of
 * sequence b sits at position p = seq_lens[b] - chunk + r and, for query
 * head j (kv head j / (n_q / n_kv)),
 *   out[b][r][j][:] = sum_{t <= p} softmax_t(sm_scale * q.k_t) v_t
 * with every token read from the cache as it stands: tokens below
 * floor(L/B)*B dequantised from the pool, the rest raw bf16 from staging. A
 * row with p < 0 (seq_lens[b] < chunk) gives zeros. out: device fp32
 * [batch][chunk][n_q][128]. chunk >= 1; chunk = 1 is kvarn_decode_attn.
 * workspace: at least kvarn_workspace_bytes(cfg, batch * chunk,
 * max_blocks_per_seq) bytes; kvarn_prefill_workspace_bytes gives the size
 * with which short chunks split each sequence's blocks over enough warps.
 * One warp scores 8 query vectors (8 / G rows x G heads) against each
 * block, building each code's tensor-core operand once for all 8. Device
 * faults as kvarn_decode_attn.
 */
int kvarn_prefill_attn(const kvarn_config* cfg, const void* q, int32_t q_dtype, const void* pool,
                       int64_t n_pool_blocks, const void* staging, const int32_t* block_table,
                       int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch, int32_t chunk,
                       float* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * kvarn_dequantize -- packed head-blocks back to fp32 values. Passage:
 * section 三 3.2 of the method page (the kept scales restore the data).
 * Reads n_head_blocks head-blocks of `kind` layout at src_base +
 * src_offsets[n] (device int64 bytes; NULL = contiguous) and writes out
 * (device fp32 [n][B][128]): rotated != 0 gives the rotated-space values
 * (code*s + z)*R*C; rotated == 0 also applies the inverse rotation.
 */
int kvarn_dequantize(const kvarn_config* cfg, int32_t kind, const void* src_base,
                     const int64_t* src_offsets, int64_t n_head_blocks, int32_t rotated,
                     float* out, void* stream);

/*
 * kvarn_error_decomposition -- the magnitude / direction split of each
 * token's quantisation error. Passage: section 二 of the method page: with
 * x^ = x + eps, eps = E_M + E_D, E_M = (|x^| - |x|) x/|x| (length error) and
 * E_D = |x^| (x^/|x^| - x/|x|) (direction error).
 * src: the values before quantisation, laid out as for kvarn_quantize_block
 * (n_head_blocks blocks of B rows, strides in elements, dtype src_dtype);
 * packed_base + packed_offsets[n] (device int64 bytes; NULL = contiguous):
 * the head-blocks of `kind` layout written from them with the same cfg.
 * out: device fp32 [n][B][4] = (|x|, |x^|, |E_M|, |E_D|) per token. A zero
 * token (direction undefined) reports all of its error as |E_M|. Read-only
 * on its inputs; no error word.
 */
int kvarn_error_decomposition(const kvarn_config* cfg, int32_t kind, const void* src, int32_t src_dtype,
                              int64_t n_head_blocks, int64_t src_block_stride, int64_t src_token_stride,
                              const void* packed_base, const int64_t* packed_offsets, float* out,
                              void* stream);

/*
 * kvarn_decode_attn_bf16 -- the same decode attention over a plain bf16
 * paged cache (the comparison point for the 2-bit path; no rotation, no
 * staging). kv_pool: device bf16 [n_pool_blocks][n_kv][2][B][128]; every
 * token of a sequence, the last block partly filled, is in the pool.
 * Other arguments as kvarn_decode_attn.
 */
int kvarn_decode_attn_bf16(const kvarn_config* cfg, const void* q, int32_t q_dtype,
                           const void* kv_pool, int64_t n_pool_blocks,
                           const int32_t* block_table, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, int32_t batch, float* out, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * kvarn_decode_attn_noalloc -- kvarn_decode_attn for callers that cannot
 * allocate device memory. (The paper has no counterpart; this is a library
 * convenience.) Some callers can only hand over their inputs and outputs: a
 * plug-in interface with no workspace argument, a runtime whose memory
 * planner owns all device memory, or a loop that must not call cudaMalloc
 * because allocation can synchronise the device. This entry point allocates
 * nothing: its split-K scratch is a 16 MiB array compiled into the library
 * (held on every GPU that loads the library until the process exits).
 *
 * Arguments and results are those of kvarn_decode_attn, without the
 * workspace. error_word (device uint32, may be NULL) receives this call's
 * KVARN_DEVERR_* flags (0 when none). The scratch must hold
 * kvarn_workspace_bytes(cfg, batch, max_blocks_per_seq) bytes (256 + (batch *
 * n_kv + resident warps) * G * 528 + batch * n_kv * 8); larger problems are refused with
 * KVARN_ERR_WORKSPACE before anything is enqueued.
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it; make that first call before any stream
 * capture. Every call shares the one array: calls whose GPU work overlaps
 * (other streams, other host threads) race on it and must be serialised by
 * the caller. Each call clears the error word it uses before its kernels run.
 */
int kvarn_decode_attn_noalloc(const kvarn_config* cfg, const void* q, int32_t q_dtype,
                              const void* pool, int64_t n_pool_blocks, const void* staging,
                              const int32_t* block_table, int32_t max_blocks_per_seq,
                              const int32_t* seq_lens, int32_t batch, float* out,
                              uint32_t* error_word, void* stream);

/* Copies the workspace error word to *code (host) after synchronising
 * stream. Returns KVARN_OK or KVARN_ERR_CUDA. */
int kvarn_read_error(const void* workspace, uint32_t* code, void* stream);

/* Zeroes the workspace error word (enqueued on stream). */
int kvarn_clear_error(void* workspace, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVARN_H_ */
