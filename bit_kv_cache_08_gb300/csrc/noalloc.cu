// noalloc.cu -- decode attention for callers that cannot allocate device
// memory.
//
// kvarn_decode_attn needs a caller-provided workspace for its split-K partial
// results and its error word. Some callers have no way to provide one: a
// plug-in interface that hands a custom operator only its input and output
// buffers, a runtime whose memory planner owns every device allocation and
// forbids others, or a latency-critical loop that must never call cudaMalloc
// because an allocation can synchronise the device. kvarn_decode_attn_noalloc
// serves them: its scratch is a fixed array compiled into this library, so
// the call allocates nothing.
//
// The array (kNoAllocScratchBytes) lives in every GPU that loads the library
// until the process exits. Host code never dereferences its symbol: the
// device address is fetched once per device with cudaGetSymbolAddress, on the
// first call made while that device is current, and cached.
#include <mutex>

#include "common.cuh"

namespace kvarn {
cudaError_t launch_decode_attn(const kvarn_config& cfg, const void* q, int q_dtype, const void* pool,
                               int64_t n_pool_blocks, int64_t block_bytes, const void* staging,
                               const int32_t* block_table, int max_blocks, const int32_t* seq_lens, int batch,
                               float* out, void* workspace, int nw, cudaStream_t st);
int attn_grid_warps(int block_size, int bits, int device);
int attn_bf16_grid_warps(int block_size, int device);
}  // namespace kvarn

using namespace kvarn;

namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;   // 16 MiB: header + split-K partials
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set up once).
int scratch_for_current_device(void** addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVARN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KVARN_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return KVARN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int kvarn_decode_attn_noalloc(const kvarn_config* cfg, const void* q, int32_t q_dtype,
                                         const void* pool, int64_t n_pool_blocks, const void* staging,
                                         const int32_t* block_table, int32_t max_blocks_per_seq,
                                         const int32_t* seq_lens, int32_t batch, float* out,
                                         uint32_t* error_word, void* stream) {
    if (!cfg) return KVARN_ERR_INVALID_ARG;
    if (cfg->head_dim != 128 || cfg->group_size != 32 || (cfg->bits < 2 || cfg->bits > 4) ||
        (cfg->block_size != 32 && cfg->block_size != 64))
        return KVARN_ERR_UNSUPPORTED;
    if (cfg->varn_iters < 0 || cfg->varn_iters > 8 || cfg->n_kv_heads < 1 || cfg->n_q_heads < cfg->n_kv_heads ||
        cfg->n_q_heads % cfg->n_kv_heads != 0 || !(cfg->sm_scale >= 0.0f) || isinf(cfg->sm_scale) ||
        (cfg->flags & ~(KVARN_FLAG_NO_ROTATION | KVARN_FLAG_NO_TOKEN_PASS | KVARN_FLAG_NO_CHANNEL_PASS)))
        return KVARN_ERR_INVALID_ARG;
    if (cfg->n_q_heads / cfg->n_kv_heads > 4) return KVARN_ERR_UNSUPPORTED;
    kvarn_config c = *cfg;
    if (c.sm_scale == 0.0f) c.sm_scale = 1.0f / sqrtf(128.0f);
    if (q_dtype != KVARN_BF16 && q_dtype != KVARN_FP32) return KVARN_ERR_INVALID_ARG;
    if (batch < 0 || max_blocks_per_seq < 0 || n_pool_blocks < 1) return KVARN_ERR_INVALID_ARG;
    if (n_pool_blocks > 0x7fffffff) return KVARN_ERR_INVALID_ARG;
    if (batch == 0) return KVARN_OK;
    if (!q || !pool || !staging || !block_table || !seq_lens || !out) return KVARN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(pool) || !aligned16(staging) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(error_word) & 3u))
        return KVARN_ERR_INVALID_ARG;
    if ((int64_t)max_blocks_per_seq * c.block_size > 0x7fffffff) return KVARN_ERR_INVALID_ARG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVARN_ERR_CUDA;
    const int nw = attn_grid_warps(c.block_size, c.bits, dev);
    const int nw_any = nw > attn_bf16_grid_warps(c.block_size, dev) ? nw : attn_bf16_grid_warps(c.block_size, dev);
    if (nw <= 0 || nw_any <= 0) return KVARN_ERR_CUDA;
    // same size rule as kvarn_workspace_bytes; beyond the fixed array: refuse
    const size_t G = (size_t)(c.n_q_heads / c.n_kv_heads);
    const size_t need = kWsHeader + ((size_t)batch * c.n_kv_heads + (size_t)nw_any) * G * 132 * sizeof(float);
    if (need > kNoAllocScratchBytes) return KVARN_ERR_WORKSPACE;

    void* scratch = nullptr;
    const int r = scratch_for_current_device(&scratch);
    if (r != KVARN_OK) return r;
    cudaStream_t st = (cudaStream_t)stream;
    // the error word is the only part of the scratch that must start at zero
    if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), st) != cudaSuccess) return KVARN_ERR_CUDA;
    const int64_t block_bytes = (int64_t)c.n_kv_heads * 2 * head_block_bytes(c.block_size, c.bits);
    if (launch_decode_attn(c, q, q_dtype, pool, n_pool_blocks, block_bytes, staging, block_table,
                           max_blocks_per_seq, seq_lens, batch, out, scratch, nw, st) != cudaSuccess)
        return KVARN_ERR_CUDA;
    if (error_word &&
        cudaMemcpyAsync(error_word, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return KVARN_ERR_CUDA;
    return KVARN_OK;
}
