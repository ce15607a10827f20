// api.cu -- the extern "C" entry points declared in include/kvarn.h: host-side
// validation, sizes, and kernel launches on the caller's stream.
#include "host_checks.h"

namespace kvarn {
cudaError_t launch_quantize_blocks(const kvarn_config& cfg, int kind, const void* src, int dtype, int64_t n,
                                   int64_t block_stride, int64_t token_stride, void* dst_base,
                                   const int64_t* dst_offsets, uint32_t* err, cudaStream_t st);
cudaError_t launch_append(const kvarn_config& cfg, void* pool, int64_t n_pool_blocks, int64_t block_bytes,
                          void* staging, const int32_t* block_table, int max_blocks, const int32_t* pos,
                          const void* k_new, const void* v_new, int batch, uint32_t* err, cudaStream_t st);
cudaError_t launch_dequantize(const kvarn_config& cfg, int kind, const void* src_base, const int64_t* src_offsets,
                              int64_t n, int rotated, float* out, cudaStream_t st);
cudaError_t launch_error_split(const kvarn_config& cfg, int kind, const void* src, int dtype, int64_t n,
                               int64_t block_stride, int64_t token_stride, const void* packed_base,
                               const int64_t* packed_offsets, float* out, cudaStream_t st);
cudaError_t launch_decode_attn(const kvarn_config& cfg, const void* q, int q_dtype, const void* pool,
                               int64_t n_pool_blocks, int64_t block_bytes, const void* staging,
                               const int32_t* block_table, int max_blocks, const int32_t* seq_lens, int batch,
                               float* out, void* workspace, int nw, cudaStream_t st);
cudaError_t launch_decode_attn_bf16(const kvarn_config& cfg, const void* q, int q_dtype, const void* kv_pool,
                                    int64_t n_pool_blocks, const int32_t* block_table, int max_blocks,
                                    const int32_t* seq_lens, int batch, float* out, void* workspace, int nw,
                                    cudaStream_t st);
cudaError_t launch_prefill_attn(const kvarn_config& cfg, const void* q, int q_dtype, const void* pool,
                                int64_t n_pool_blocks, int64_t block_bytes, const void* staging,
                                const int32_t* block_table, int max_blocks, const int32_t* seq_lens, int batch,
                                int chunk, float* out, void* workspace, int64_t max_slots, int64_t splits,
                                cudaStream_t st);
int64_t prefill_splits(const kvarn_config& cfg, int64_t batch, int64_t chunk, int device);
}  // namespace kvarn

using namespace kvarn;

namespace {

size_t ws_bytes(const kvarn_config& c, int32_t batch) { return decode_ws_bytes(c, batch); }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? KVARN_OK : KVARN_ERR_CUDA; }

}  // namespace

extern "C" {

const char* kvarn_version(void) { return "kvarn 0.1 sm_103a"; }

const char* kvarn_status_string(int status) {
    switch (status) {
        case KVARN_OK: return "ok";
        case KVARN_ERR_INVALID_ARG: return "invalid argument";
        case KVARN_ERR_UNSUPPORTED: return "unsupported configuration";
        case KVARN_ERR_CUDA: return "CUDA error";
        case KVARN_ERR_WORKSPACE: return "workspace too small";
        default: return "unknown status";
    }
}

size_t kvarn_head_block_bytes(const kvarn_config* cfg) {
    kvarn_config c;
    if (check_config(cfg, &c) != KVARN_OK) return 0;
    return (size_t)head_block_bytes(c.block_size, c.bits);
}

size_t kvarn_block_bytes(const kvarn_config* cfg) {
    kvarn_config c;
    if (check_config(cfg, &c) != KVARN_OK) return 0;
    return (size_t)c.n_kv_heads * 2 * head_block_bytes(c.block_size, c.bits);
}

size_t kvarn_staging_bytes(const kvarn_config* cfg, int32_t max_seqs) {
    kvarn_config c;
    if (check_config(cfg, &c) != KVARN_OK || max_seqs < 0) return 0;
    return (size_t)max_seqs * c.n_kv_heads * 2 * c.block_size * 128 * 2;
}

// Warps the 2-bit prefill kernel aims for: half the resident warps (measured
// on the Llama-3.1-8B layer: more block splits than that cost more in partials
// and merging than they gain in occupancy).
size_t kvarn_prefill_workspace_bytes(const kvarn_config* cfg, int32_t batch, int32_t chunk,
                                     int32_t max_blocks_per_seq) {
    kvarn_config c;
    if (check_config(cfg, &c) != KVARN_OK || batch < 0 || chunk < 1 || max_blocks_per_seq < 0) return 0;
    if ((int64_t)batch * chunk > 0x7fffffff / c.n_q_heads) return 0;
    const size_t base = ws_bytes(c, batch * chunk);
    if (base == 0 || batch == 0 || chunk == 1) return base;
    const int64_t rows = (int64_t)batch * chunk * c.n_kv_heads;
    const size_t split = kWsHeader + (size_t)(rows * prefill_splits(c, batch, chunk, current_device())) *
                                         (size_t)(c.n_q_heads / c.n_kv_heads) * 132 * sizeof(float);
    return split > base ? split : base;
}

size_t kvarn_workspace_bytes(const kvarn_config* cfg, int32_t batch, int32_t max_blocks_per_seq) {
    kvarn_config c;
    if (check_config(cfg, &c) != KVARN_OK || batch < 0 || max_blocks_per_seq < 0) return 0;
    return ws_bytes(c, batch);
}

int kvarn_quantize_block(const kvarn_config* cfg, int32_t kind, const void* src, int32_t src_dtype,
                         int64_t n_head_blocks, int64_t src_block_stride, int64_t src_token_stride,
                         void* dst_base, const int64_t* dst_offsets, void* workspace, void* stream) {
    kvarn_config c;
    int r = check_config(cfg, &c);
    if (r != KVARN_OK) return r;
    if (kind != KVARN_KIND_K && kind != KVARN_KIND_V) return KVARN_ERR_INVALID_ARG;
    if (src_dtype != KVARN_BF16 && src_dtype != KVARN_FP32) return KVARN_ERR_INVALID_ARG;
    if (n_head_blocks < 0 || n_head_blocks > 0x7fffffff) return KVARN_ERR_INVALID_ARG;
    if (n_head_blocks == 0) return KVARN_OK;
    if (!src || !dst_base || !workspace) return KVARN_ERR_INVALID_ARG;
    const size_t esz = src_dtype == KVARN_FP32 ? 4 : 2;
    if (!aligned(src, 4 * esz) || (src_block_stride % 4) || (src_token_stride % 4)) return KVARN_ERR_INVALID_ARG;
    if (src_token_stride < 128 || src_block_stride < 0) return KVARN_ERR_INVALID_ARG;
    if (!aligned(dst_base, 16) || !aligned(workspace, 16) || (dst_offsets && !aligned(dst_offsets, 8)))
        return KVARN_ERR_INVALID_ARG;
    return cuda_status(launch_quantize_blocks(c, kind, src, src_dtype, n_head_blocks, src_block_stride,
                                              src_token_stride, dst_base, dst_offsets, (uint32_t*)workspace,
                                              (cudaStream_t)stream));
}

int kvarn_append(const kvarn_config* cfg, void* pool, int64_t n_pool_blocks, void* staging,
                 const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* pos, const void* k_new,
                 const void* v_new, int32_t batch, void* workspace, void* stream) {
    kvarn_config c;
    int r = check_config(cfg, &c);
    if (r != KVARN_OK) return r;
    if (batch < 0 || max_blocks_per_seq < 0 || n_pool_blocks < 0) return KVARN_ERR_INVALID_ARG;
    if (batch == 0) return KVARN_OK;
    if (batch > 0x7fffffff / 1 || c.n_kv_heads > 65535) return KVARN_ERR_INVALID_ARG;
    if (!pool || !staging || !block_table || !pos || !k_new || !v_new || !workspace) return KVARN_ERR_INVALID_ARG;
    if (!aligned(pool, 16) || !aligned(staging, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) ||
        !aligned(workspace, 16) || !aligned(block_table, 4) || !aligned(pos, 4))
        return KVARN_ERR_INVALID_ARG;
    if ((int64_t)max_blocks_per_seq * c.block_size > 0x7fffffff) return KVARN_ERR_INVALID_ARG;
    return cuda_status(launch_append(c, pool, n_pool_blocks, (int64_t)kvarn_block_bytes(&c), staging, block_table,
                                     max_blocks_per_seq, pos, k_new, v_new, batch, (uint32_t*)workspace,
                                     (cudaStream_t)stream));
}

namespace {
// Decode (chunk = 1) and chunked prefill share one split-K launch: every query
// row of a chunk is a virtual sequence with its own causal prefix.
int packed_attn(const kvarn_config* cfg, const void* q, int32_t q_dtype, const void* pool, int64_t n_pool_blocks,
                const void* staging, const int32_t* block_table, int32_t max_blocks_per_seq,
                const int32_t* seq_lens, int32_t batch, int32_t chunk, float* out, void* workspace,
                size_t workspace_bytes, void* stream) {
    kvarn_config c;
    int r = check_config(cfg, &c);
    if (r != KVARN_OK) return r;
    r = check_packed_attn_args(c, q, q_dtype, pool, n_pool_blocks, staging, block_table, max_blocks_per_seq,
                               seq_lens, batch, chunk, out);
    if (r != KVARN_OK || batch == 0) return r;
    if (!workspace || !aligned(workspace, 16)) return KVARN_ERR_INVALID_ARG;
    const size_t need = ws_bytes(c, batch * chunk);
    if (need == 0) return KVARN_ERR_CUDA;
    if (workspace_bytes < need) return KVARN_ERR_WORKSPACE;
    if (chunk > 1) {   // rows of a chunk share each block's operands
        // partial slots the caller's workspace holds: the block splits adapt to it
        const int64_t slots = (int64_t)((workspace_bytes - kWsHeader) /
                                        ((size_t)(c.n_q_heads / c.n_kv_heads) * 132 * sizeof(float)));
        return cuda_status(launch_prefill_attn(c, q, q_dtype, pool, n_pool_blocks, (int64_t)kvarn_block_bytes(&c),
                                               staging, block_table, max_blocks_per_seq, seq_lens, batch, chunk,
                                               out, workspace, slots, prefill_splits(c, batch, chunk, current_device()),
                                               (cudaStream_t)stream));
    }
    const int nw = attn_grid_warps(c.block_size, c.bits, current_device());
    if (nw <= 0) return KVARN_ERR_CUDA;
    return cuda_status(launch_decode_attn(c, q, q_dtype, pool, n_pool_blocks, (int64_t)kvarn_block_bytes(&c),
                                          staging, block_table, max_blocks_per_seq, seq_lens, batch, out,
                                          workspace, nw, (cudaStream_t)stream));
}
}  // namespace

int kvarn_decode_attn(const kvarn_config* cfg, const void* q, int32_t q_dtype, const void* pool,
                      int64_t n_pool_blocks, const void* staging, const int32_t* block_table,
                      int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch, float* out,
                      void* workspace, size_t workspace_bytes, void* stream) {
    return packed_attn(cfg, q, q_dtype, pool, n_pool_blocks, staging, block_table, max_blocks_per_seq, seq_lens,
                       batch, 1, out, workspace, workspace_bytes, stream);
}

int kvarn_prefill_attn(const kvarn_config* cfg, const void* q, int32_t q_dtype, const void* pool,
                       int64_t n_pool_blocks, const void* staging, const int32_t* block_table,
                       int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch, int32_t chunk,
                       float* out, void* workspace, size_t workspace_bytes, void* stream) {
    return packed_attn(cfg, q, q_dtype, pool, n_pool_blocks, staging, block_table, max_blocks_per_seq, seq_lens,
                       batch, chunk, out, workspace, workspace_bytes, stream);
}

int kvarn_dequantize(const kvarn_config* cfg, int32_t kind, const void* src_base, const int64_t* src_offsets,
                     int64_t n_head_blocks, int32_t rotated, float* out, void* stream) {
    kvarn_config c;
    int r = check_config(cfg, &c);
    if (r != KVARN_OK) return r;
    if (kind != KVARN_KIND_K && kind != KVARN_KIND_V) return KVARN_ERR_INVALID_ARG;
    if (n_head_blocks < 0 || n_head_blocks > 0x7fffffff) return KVARN_ERR_INVALID_ARG;
    if (n_head_blocks == 0) return KVARN_OK;
    if (!src_base || !out) return KVARN_ERR_INVALID_ARG;
    if (!aligned(src_base, 16) || !aligned(out, 16) || (src_offsets && !aligned(src_offsets, 8)))
        return KVARN_ERR_INVALID_ARG;
    return cuda_status(launch_dequantize(c, kind, src_base, src_offsets, n_head_blocks, rotated ? 1 : 0, out,
                                         (cudaStream_t)stream));
}

int kvarn_error_decomposition(const kvarn_config* cfg, int32_t kind, const void* src, int32_t src_dtype,
                              int64_t n_head_blocks, int64_t src_block_stride, int64_t src_token_stride,
                              const void* packed_base, const int64_t* packed_offsets, float* out, void* stream) {
    kvarn_config c;
    int r = check_config(cfg, &c);
    if (r != KVARN_OK) return r;
    if (kind != KVARN_KIND_K && kind != KVARN_KIND_V) return KVARN_ERR_INVALID_ARG;
    if (src_dtype != KVARN_BF16 && src_dtype != KVARN_FP32) return KVARN_ERR_INVALID_ARG;
    if (n_head_blocks < 0 || n_head_blocks > 0x7fffffff) return KVARN_ERR_INVALID_ARG;
    if (n_head_blocks == 0) return KVARN_OK;
    if (!src || !packed_base || !out) return KVARN_ERR_INVALID_ARG;
    const size_t esz = src_dtype == KVARN_FP32 ? 4 : 2;
    if (!aligned(src, 4 * esz) || (src_block_stride % 4) || (src_token_stride % 4)) return KVARN_ERR_INVALID_ARG;
    if (src_token_stride < 128 || src_block_stride < 0) return KVARN_ERR_INVALID_ARG;
    if (!aligned(packed_base, 16) || !aligned(out, 16) || (packed_offsets && !aligned(packed_offsets, 8)))
        return KVARN_ERR_INVALID_ARG;
    return cuda_status(launch_error_split(c, kind, src, src_dtype, n_head_blocks, src_block_stride,
                                          src_token_stride, packed_base, packed_offsets, out,
                                          (cudaStream_t)stream));
}

int kvarn_decode_attn_bf16(const kvarn_config* cfg, const void* q, int32_t q_dtype, const void* kv_pool,
                           int64_t n_pool_blocks, const int32_t* block_table, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, int32_t batch, float* out, void* workspace,
                           size_t workspace_bytes, void* stream) {
    kvarn_config c;
    int r = check_config(cfg, &c);
    if (r != KVARN_OK) return r;
    if (q_dtype != KVARN_BF16 && q_dtype != KVARN_FP32) return KVARN_ERR_INVALID_ARG;
    if (batch < 0 || max_blocks_per_seq < 0 || n_pool_blocks < 1) return KVARN_ERR_INVALID_ARG;
    if (batch == 0) return KVARN_OK;
    if (!q || !kv_pool || !block_table || !seq_lens || !out || !workspace) return KVARN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(kv_pool, 16) || !aligned(out, 16) || !aligned(workspace, 16) ||
        !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return KVARN_ERR_INVALID_ARG;
    if ((int64_t)max_blocks_per_seq * c.block_size > 0x7fffffff) return KVARN_ERR_INVALID_ARG;
    const size_t need = ws_bytes(c, batch);
    if (need == 0) return KVARN_ERR_CUDA;
    if (workspace_bytes < need) return KVARN_ERR_WORKSPACE;
    const int nw = attn_bf16_grid_warps(c.block_size, current_device());
    if (nw <= 0) return KVARN_ERR_CUDA;
    return cuda_status(launch_decode_attn_bf16(c, q, q_dtype, kv_pool, n_pool_blocks, block_table,
                                               max_blocks_per_seq, seq_lens, batch, out, workspace, nw,
                                               (cudaStream_t)stream));
}

int kvarn_read_error(const void* workspace, uint32_t* code, void* stream) {
    if (!workspace || !code) return KVARN_ERR_INVALID_ARG;
    cudaError_t e = cudaMemcpyAsync(code, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    return cuda_status(e);
}

int kvarn_clear_error(void* workspace, void* stream) {
    if (!workspace) return KVARN_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(workspace, 0, sizeof(uint32_t), (cudaStream_t)stream));
}

}  // extern "C"
