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

#include "host_checks.h"

namespace kvarn {
cudaError_t launch_decode_attn(const kvarn_config& cfg, const void* q, int q_dtype, const void* pool,
                               int64_t n_pool_blocks, int64_t block_bytes, const void* staging,
                               const int32_t* block_table, int max_blocks, const int32_t* seq_lens, int batch,
                               float* out, void* workspace, int nw, cudaStream_t st);
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

}  // namespace

extern "C" int kvarn_decode_attn_noalloc(const kvarn_config* cfg, const void* q, int32_t q_dtype,
                                         const void* pool, int64_t n_pool_blocks, const void* staging,
                                         const int32_t* block_table, int32_t max_blocks_per_seq,
                                         const int32_t* seq_lens, int32_t batch, float* out,
                                         uint32_t* error_word, void* stream) {
    kvarn_config c;
    int r = check_config(cfg, &c);
    if (r != KVARN_OK) return r;
    r = check_packed_attn_args(c, q, q_dtype, pool, n_pool_blocks, staging, block_table, max_blocks_per_seq,
                               seq_lens, batch, 1, out);
    if (r != KVARN_OK || batch == 0) return r;
    if (!aligned(error_word, 4)) return KVARN_ERR_INVALID_ARG;
    // the workspace the same call with a caller's buffer would need; beyond
    // the fixed array: refuse
    const size_t need = decode_ws_bytes(c, batch);
    if (need == 0) return KVARN_ERR_CUDA;
    if (need > kNoAllocScratchBytes) return KVARN_ERR_WORKSPACE;
    const int nw = attn_grid_warps(c.block_size, c.bits, current_device());
    if (nw <= 0) return KVARN_ERR_CUDA;

    void* scratch = nullptr;
    r = scratch_for_current_device(&scratch);
    if (r != KVARN_OK) return r;
    cudaStream_t st = (cudaStream_t)stream;
    // the error word is the only part of the scratch that must start at zero
    if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), st) != cudaSuccess) return KVARN_ERR_CUDA;
    if (launch_decode_attn(c, q, q_dtype, pool, n_pool_blocks, block_bytes_of(c), staging, block_table,
                           max_blocks_per_seq, seq_lens, batch, out, scratch, nw, st) != cudaSuccess)
        return KVARN_ERR_CUDA;
    if (error_word &&
        cudaMemcpyAsync(error_word, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return KVARN_ERR_CUDA;
    return KVARN_OK;
}
