// host_checks.h -- host-side argument rules shared by every entry point that
// launches the decode attention (api.cu with a caller's workspace, noalloc.cu
// with the library's fixed scratch): one definition of the configuration
// check, the argument checks and the workspace size rule, so the two entry
// points cannot drift apart.
#pragma once
#include <math.h>

#include "common.cuh"

namespace kvarn {

int attn_grid_warps(int block_size, int bits, int device);
int attn_bf16_grid_warps(int block_size, int device);

constexpr int kMaxGroup = 4;   // query heads per kv head

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Validates cfg and returns a copy with defaults applied (sm_scale).
inline int check_config(const kvarn_config* cfg, kvarn_config* out) {
    if (!cfg) return KVARN_ERR_INVALID_ARG;
    if (cfg->head_dim != 128 || cfg->group_size != 32 || (cfg->bits < 2 || cfg->bits > 4))
        return KVARN_ERR_UNSUPPORTED;
    if (cfg->block_size != 32 && cfg->block_size != 64) return KVARN_ERR_UNSUPPORTED;
    if (cfg->varn_iters < 0 || cfg->varn_iters > 8) return KVARN_ERR_INVALID_ARG;
    if (cfg->flags & ~(KVARN_FLAG_NO_ROTATION | KVARN_FLAG_NO_TOKEN_PASS | KVARN_FLAG_NO_CHANNEL_PASS |
                       KVARN_FLAG_TEST_WAIT_TIMEOUT))
        return KVARN_ERR_INVALID_ARG;
    if (cfg->n_kv_heads < 1 || cfg->n_q_heads < cfg->n_kv_heads) return KVARN_ERR_INVALID_ARG;
    if (cfg->n_q_heads % cfg->n_kv_heads != 0) return KVARN_ERR_INVALID_ARG;
    if (cfg->n_q_heads / cfg->n_kv_heads > kMaxGroup) return KVARN_ERR_UNSUPPORTED;
    if (!(cfg->sm_scale >= 0.0f) || isinf(cfg->sm_scale)) return KVARN_ERR_INVALID_ARG;
    *out = *cfg;
    if (out->sm_scale == 0.0f) out->sm_scale = 1.0f / sqrtf(128.0f);
    return KVARN_OK;
}

inline int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return d;
}

// Packed bytes of one physical block (every kv head, K and V).
inline int64_t block_bytes_of(const kvarn_config& c) {
    return (int64_t)c.n_kv_heads * 2 * head_block_bytes(c.block_size, c.bits);
}

// Workspace bytes the decode kernels need for `batch` query rows on the
// current device: the header, one partial slot per (row, kv head) and one
// per resident warp of the larger of the 2-bit and bf16 split kernels, then
// the 2-bit kernel's unit map (first and last warp of every (row, kv head),
// 8 bytes each). 0 when the device cannot be queried.
inline size_t decode_ws_bytes(const kvarn_config& c, int32_t batch) {
    if (batch <= 0) return kWsHeader;
    const int d = current_device();
    if (d < 0) return 0;
    const int a = attn_grid_warps(c.block_size, c.bits, d);
    const int b = attn_bf16_grid_warps(c.block_size, d);
    const int nw = a > b ? a : b;
    if (a <= 0 || b <= 0) return 0;
    const size_t G = (size_t)(c.n_q_heads / c.n_kv_heads);
    const size_t slots = (size_t)batch * c.n_kv_heads + (size_t)nw;
    // header, split-K partials, then the (first, last) warp of every unit
    return kWsHeader + slots * G * 132 * sizeof(float) + (size_t)batch * c.n_kv_heads * 2 * sizeof(int32_t);
}

// Arguments of a packed-cache attention call (decode: chunk = 1; chunked
// prefill: chunk > 1), everything but the workspace. KVARN_OK means the call
// may launch; batch == 0 is valid and launches nothing.
inline int check_packed_attn_args(const kvarn_config& c, const void* q, int32_t q_dtype, const void* pool,
                                  int64_t n_pool_blocks, const void* staging, const int32_t* block_table,
                                  int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch,
                                  int32_t chunk, const float* out) {
    if (q_dtype != KVARN_BF16 && q_dtype != KVARN_FP32) return KVARN_ERR_INVALID_ARG;
    if (batch < 0 || chunk < 1 || max_blocks_per_seq < 0 || n_pool_blocks < 1) return KVARN_ERR_INVALID_ARG;
    if ((int64_t)batch * chunk > 0x7fffffff / c.n_q_heads) return KVARN_ERR_INVALID_ARG;
    if (batch == 0) return KVARN_OK;
    if (!q || !pool || !staging || !block_table || !seq_lens || !out) return KVARN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(pool, 16) || !aligned(staging, 16) || !aligned(out, 16) ||
        !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return KVARN_ERR_INVALID_ARG;
    if ((int64_t)max_blocks_per_seq * c.block_size > 0x7fffffff) return KVARN_ERR_INVALID_ARG;
    if (n_pool_blocks > 0x7fffffff || block_bytes_of(c) > 0x7fffffff) return KVARN_ERR_INVALID_ARG;
    return KVARN_OK;
}

}  // namespace kvarn
