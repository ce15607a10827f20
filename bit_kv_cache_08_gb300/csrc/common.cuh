// common.cuh -- device helpers shared by the KVarN kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvarn.h"

namespace kvarn {

constexpr int kD = 128;          // head_dim
constexpr int kGroups = 4;       // 32-channel quantisation groups per token
constexpr int kGroupSize = 32;
constexpr float kInvSqrtD = 0.08838834764831845f;   // 1/sqrt(128)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kF16Max = 65504.0f;
constexpr float kF16MinNormal = 6.103515625e-05f;   // 2^-14
constexpr uint32_t kFull = 0xffffffffu;

// Head-block sections for codes of `bits` bits: codes (16 B bits bytes), then
// s, z (fp16 [4][B] each), R (fp16 [B]), C (fp16 [128]).
__host__ __device__ constexpr int off_s(int B, int bits) { return 16 * bits * B; }
__host__ __device__ constexpr int off_z(int B, int bits) { return off_s(B, bits) + 8 * B; }
__host__ __device__ constexpr int off_R(int B, int bits) { return off_s(B, bits) + 16 * B; }
__host__ __device__ constexpr int off_C(int B, int bits) { return off_s(B, bits) + 18 * B; }
__host__ __device__ constexpr int head_block_bytes(int B, int bits) { return off_C(B, bits) + 256; }

// Workspace header: the first uint32 is the sticky device error word.
constexpr size_t kWsHeader = 256;

__device__ __forceinline__ void raise_error(uint32_t* err, uint32_t flag) {
    if (err) atomicOr(err, flag);
}

__device__ __forceinline__ float sign_of(const uint32_t (&sb)[4], int c) {
    return ((sb[c >> 5] >> (c & 31)) & 1u) ? -1.0f : 1.0f;
}
// Same, from four scalar words (keeps kernel parameters out of local memory).
__device__ __forceinline__ float sign_of4(uint32_t s0, uint32_t s1, uint32_t s2, uint32_t s3, int c) {
    const int w = c >> 5;
    const uint32_t word = w == 0 ? s0 : (w == 1 ? s1 : (w == 2 ? s2 : s3));
    return ((word >> (c & 31)) & 1u) ? -1.0f : 1.0f;
}

// ---------------------------------------------------------------- warp reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, m));
    return v;
}

// ---------------------------------------------------------------- FWHT-128
// Lane l holds channels 4l..4l+3 in v[0..3]. Computes the unnormalised
// Sylvester-Hadamard transform (H x)_i = sum_j (-1)^popcount(i&j) x_j with
// butterflies: channel bits 0-1 inside the thread, bits 2-6 across lanes
// (lane bit k-2 = channel bit k).
__device__ __forceinline__ void fwht128(float (&v)[4], int lane) {
    float a0 = v[0] + v[1], a1 = v[0] - v[1];
    float a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2; v[2] = a0 - a2;
    v[1] = a1 + a3; v[3] = a1 - a3;
#pragma unroll
    for (int m = 1; m <= 16; m <<= 1) {
        // lower lane: v + o; upper lane: o - v (one fma with a +-1 factor, exact)
        const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float o = __shfl_xor_sync(kFull, v[k], m);
            v[k] = fmaf(sgn, v[k], o);
        }
    }
}

// ---------------------------------------------------------------- launches
// Programmatic dependent launch: every kernel of this library is launched with
// programmatic stream serialization and begins with a wait on the grids ahead
// of it in the stream. Its CTAs may then be scheduled while the previous
// kernel drains, and its memory accesses still see everything that kernel
// wrote (the wait returns once those grids have completed and flushed).
__device__ __forceinline__ void wait_prior_grids() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
    cudaLaunchConfig_t c = {};
    c.gridDim = grid;
    c.blockDim = block;
    c.dynamicSmemBytes = smem;
    c.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    c.attrs = at;
    c.numAttrs = 1;
    return cudaLaunchKernelEx(&c, kernel, args...);
}

// ---------------------------------------------------------------- fp16 helpers
__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }
__device__ __forceinline__ uint16_t f2h_rn(float f) { return __half_as_ushort(__float2half_rn(f)); }

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// ---------------------------------------------------------------- error-bounded mbarrier wait
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
// Returns true once the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Bounded wait: gives up after `limit` polls (each try_wait may itself
// suspend for a hardware-defined time) and reports false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

}  // namespace kvarn

namespace kvarn {
__device__ __forceinline__ int64_t warp_sum_i64(int64_t v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
    return v;
}
}  // namespace kvarn
