// attn_common.cuh -- pieces shared by the decode-attention kernels: the
// argument block, tensor-core and exponent helpers, and the kernels that
// merge the split-K partials (one warp per query row, or eight) with the
// launch that picks between them.
#pragma once
#include "split.cuh"

namespace kvarn {

constexpr uint32_t kWaitLimit = 1u << 22;
// Cost of one 2-bit block per token of block size, in units of merging one
// partial; see split_active_warps. Chosen from batch-1 timings of the
// Llama-shaped cache (8K-128K tokens) with the wide merge, where 2 beat 0.5,
// 1 and 4 (0.5 had been best while one warp merged a row's partials).
constexpr float kSplitRatio2bit = 2.0f;

struct AttnArgs {
    const void* q;
    const uint8_t* pool;
    const uint16_t* staging;
    const int32_t* block_table;
    const int32_t* seq_lens;
    float* partials;
    float* out;
    uint32_t* err;
    int64_t n_pool_blocks;
    int64_t block_bytes;
    int q_dtype;
    int max_blocks;
    int batch;
    int n_q, n_kv, G;
    int nw;
    int chunk;        // query rows per sequence (1: decode); batch counts batch * chunk rows
    int single;       // > 0: that many partials per (row, kv head) unit u, in slots u * single ..
    float sm_scale;
    uint32_t flags;   // KVARN_FLAG_*: the cache's ablation switches
    uint32_t first_wait_limit;   // polls of each warp's first stage wait (kWaitLimit; less only in tests)
    uint32_t sb[4];
    // (first, last) warp of each (sequence, kv head) unit, written by the split
    // kernel for the merge; nullptr: the merge finds them from the split arithmetic
    int32_t* unit_map;
};

// ---------------------------------------------------------------- small helpers
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = A B when `first` (a zero C: no zeroing of d), else d += A B; `first`
// is a compile-time constant at every call
__device__ __forceinline__ void mma16816_acc(float (&d)[4], bool first, uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
    if (first)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%10,%10,%10,%10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
    else
        mma16816(d, a0, a1, a2, a3, b0, b1);
}

// Scaled-subnormal code operands (decode and prefill). A code field masked out of a
// record word in place is an fp16 subnormal, its value the code times a
// power of two set by the field's bit position; one multiply by the inverse
// power brings every code to the same exact normal value code * 2^-9. One
// LOP3 (the mask) on the ALU pipe and one HMUL2 on the fp16 pipe per pair,
// no shift: fields j >= 4 come from w8 = w >> 8, taken once per word.
constexpr float kCodeScale = 1.0f / 512.0f;   // an operand holds code * 2^-9
constexpr uint32_t kCodeScaleH2 = 0x18001800u;   // 2^-9 as fp16x2

__device__ __forceinline__ uint32_t scale_sub(uint32_t x, uint32_t pow2_h2) {
    return h2_as_u32(__hmul2(u32_as_h2(x), u32_as_h2(pow2_h2)));
}
// fp16x2 2^(15 - 2k) for k = 0..3: 2^15, 2^13, 2^11, 2^9
__device__ __forceinline__ constexpr uint32_t pow2_for_field2(int k) {
    return k == 0 ? 0x78007800u : (k == 1 ? 0x70007000u : (k == 2 ? 0x68006800u : 0x60006000u));
}
// 2-bit pair j (0..7): bits 2j, 2j + 1 of each half of w -> (c_lo, c_hi) * 2^-9
__device__ __forceinline__ uint32_t code2_s(uint32_t w, uint32_t w8, int j) {
    const int k = j & 3;
    return scale_sub((j < 4 ? w : w8) & (0x00030003u << (2 * k)), pow2_for_field2(k));
}
// 3-bit pair: the low two bits at 2-bit pair j of w, the high bit at bit jh
// of each half of the 1-bit plane word hw, joined into a 3-bit field at bits
// 2k..2k+2 (k = j & 3) and scaled by 2^(15 - 2k): (c_lo, c_hi) * 2^-9
__device__ __forceinline__ uint32_t code3_s(uint32_t w, uint32_t w8, uint32_t hw, int j, int jh) {
    const int k = j & 3, d = 2 * k + 2 - jh;
    const uint32_t hs = d >= 0 ? (hw << d) : (hw >> (-d));
    const uint32_t x = ((j < 4 ? w : w8) & (0x00030003u << (2 * k))) | (hs & (0x00040004u << (2 * k)));
    return scale_sub(x, pow2_for_field2(k));
}
// 4-bit pair j (0..3): bits 4j..4j+3 of each half of w (w8 for j >= 2),
// scaled by 2^15 or 2^11: (c_lo, c_hi) * 2^-9
__device__ __forceinline__ uint32_t code4_s(uint32_t w, uint32_t w8, int j) {
    const int k = j & 1;
    return scale_sub((j < 2 ? w : w8) & (0x000F000Fu << (4 * k)), k == 0 ? 0x78007800u : 0x68006800u);
}

// Raw subnormal code operands (2-bit decode). mma.m16n8k16 keeps full
// precision for subnormal fp16 A operands whose set bits sit at 6 and above:
// measured against exact sums on the GB300, the worst error is 2^-19.8 of the
// largest product for a 2-bit field at bits 6..7 and 2^-20 at bits 8..9, as
// for normal operands, against 2^-13 at bits 0..1 and 2^-18.3 at 4..5. So
// each 2-bit field j of a record word is brought to bits 8..9 (even j: the
// operand is code * 2^-16) or 6..7 (odd j: code * 2^-18) of its half by one
// of four views of the word, and one LOP3 keeps it: the word itself (fields
// 3, 4), w << 4 (fields 1, 2), w >> 4 (fields 5, 6) and the byte swap inside
// each half (fields 7 and 0). Three shifts or permutes per word and one mask
// per pair, all on the ALU pipe, no fp16 multiply. The factor 4 between odd
// and even fields is carried by the other operand (QK) or by the output row
// (PV); the common 2^-16 by the fp32 epilogue.
constexpr float kRawScale = 1.0f / 65536.0f;    // even fields' operands, code * 2^-16
constexpr uint32_t kRawOneEven = 0x01000100u;   // code 1 at bits 8..9 of both halves: 2^-16
constexpr uint32_t kRawOneOdd = 0x00400040u;    // code 1 at bits 6..7 of both halves: 2^-18
// which view of the word holds field j (0..7) at bits 6..9
__device__ __forceinline__ constexpr int code2_view_of(int j) {
    return (j == 0 || j == 7) ? 0 : (j <= 2 ? 1 : (j <= 4 ? 2 : 3));
}
__device__ __forceinline__ uint32_t code2_view(uint32_t w, int v) {
    return v == 0 ? __byte_perm(w, 0u, 0x2301u) : (v == 1 ? (w << 4) : (v == 2 ? w : (w >> 4)));
}
// field j of both halves of the word, from its view code2_view(w, code2_view_of(j))
__device__ __forceinline__ uint32_t code2_r(uint32_t view, int j) {
    return view & ((j & 1) ? 0x00C000C0u : 0x03000300u);
}

// 2^k as a float for k in [-126, 127]
__device__ __forceinline__ float exp2i(int k) {
    k = max(-126, min(127, k));
    return __int_as_float((127 + k) << 23);
}
// ceil(log2(x)) for finite x > 0 (normal)
__device__ __forceinline__ int ceil_log2(float x) {
    const uint32_t u = __float_as_uint(x);
    return (int)((u >> 23) & 0xff) - 127 + ((u & 0x7fffff) != 0);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    return h2_as_u32(__floats2half2_rn(lo, hi));
}

__device__ __forceinline__ void load_q4(const void* q, int q_dtype, int64_t row, int lane, float (&v)[4]) {
    if (q_dtype == KVARN_FP32) {
        float4 f = reinterpret_cast<const float4*>(static_cast<const float*>(q) + row * kD)[lane];
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    } else {
        uint2 u = reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(q) + row * kD)[lane];
        v[0] = __uint_as_float(u.x << 16);
        v[1] = __uint_as_float(u.x & 0xffff0000u);
        v[2] = __uint_as_float(u.y << 16);
        v[3] = __uint_as_float(u.y & 0xffff0000u);
    }
}

__device__ __forceinline__ void prefetch_l1(const void* p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// ---------------------------------------------------------------- merge
// LSE merge of np >= 1 partials starting at p0, pstride floats apart: the
// common maximum m, the weighted sum l and this lane's 4 weighted
// accumulators (channels 4 lane .. 4 lane + 3).
__device__ __forceinline__ void lse_partials(const float* p0, int np, int64_t pstride, int lane, float& m, float& l,
                                             float (&acc)[4]) {
    if (np <= 16) {
        // one round trip: lane i holds partial i's (m, l); every lane loads its
        // 4 channels of all partials at once, then weighs them
        const float pm = lane < np ? __ldcg(p0 + lane * pstride) : -INFINITY;
        const float pl = lane < np ? __ldcg(p0 + lane * pstride + 1) : 0.f;
        float4 pa[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (i < np) pa[i] = __ldcg(reinterpret_cast<const float4*>(p0 + i * pstride + 4) + lane);
        m = warp_max(pm);
        if (m != -INFINITY) {
            const float wl = lane < np ? exp2f(pm - m) : 0.f;
            l = warp_sum(pl * wl);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (i < np) {
                    const float wgt = __shfl_sync(kFull, wl, i);
                    acc[0] = fmaf(wgt, pa[i].x, acc[0]);
                    acc[1] = fmaf(wgt, pa[i].y, acc[1]);
                    acc[2] = fmaf(wgt, pa[i].z, acc[2]);
                    acc[3] = fmaf(wgt, pa[i].w, acc[3]);
                }
            }
        }
    } else {
        // the common maximum and the weighted sum of l, lanes over partials
        float mx = -INFINITY;
        for (int i = lane; i < np; i += 32) mx = fmaxf(mx, __ldcg(p0 + i * pstride));
        m = warp_max(mx);
        if (m != -INFINITY) {
            float ls = 0.f;
            for (int i = lane; i < np; i += 32) ls += __ldcg(p0 + i * pstride + 1) * exp2f(__ldcg(p0 + i * pstride) - m);
            l = warp_sum(ls);
            // every lane its 4 channels over all partials (independent loads; a
            // deep unroll keeps many in flight when one unit has hundreds of partials)
#pragma unroll 16
            for (int i = 0; i < np; ++i) {
                const float* bp = p0 + i * pstride;
                const float wgt = exp2f(__ldcg(bp) - m);
                const float4 pa = __ldcg(reinterpret_cast<const float4*>(bp + 4) + lane);
                acc[0] = fmaf(wgt, pa.x, acc[0]);
                acc[1] = fmaf(wgt, pa.y, acc[1]);
                acc[2] = fmaf(wgt, pa.z, acc[2]);
                acc[3] = fmaf(wgt, pa.w, acc[3]);
            }
        }
    }
}

// The same LSE merge in batches of NB partials with a running rescale, for
// the wide merge's warps (fewer registers than lse_partials); m, l and acc
// start at -inf, 0 and 0.
template <int NB>
__device__ __forceinline__ void lse_stream(const float* p0, int np, int64_t pstride, int lane, float& m, float& l,
                                           float (&acc)[4]) {
    for (int i0 = 0; i0 < np; i0 += NB) {
        const int cnt = min(NB, np - i0);
        const float* q = p0 + i0 * pstride;
        const float pm = lane < cnt ? __ldcg(q + lane * pstride) : -INFINITY;
        const float pl = lane < cnt ? __ldcg(q + lane * pstride + 1) : 0.f;
        float4 pa[NB];
#pragma unroll
        for (int i = 0; i < NB; ++i)
            if (i < cnt) pa[i] = __ldcg(reinterpret_cast<const float4*>(q + i * pstride + 4) + lane);
        const float bm = warp_max(pm);
        if (bm == -INFINITY) continue;
        const float mn = fmaxf(m, bm);
        const float fa = m == -INFINITY ? 0.f : exp2f(m - mn);
        const float wl = lane < cnt ? exp2f(pm - mn) : 0.f;
        l = l * fa + warp_sum(pl * wl);
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] *= fa;
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            if (i < cnt) {
                const float wgt = __shfl_sync(kFull, wl, i);
                acc[0] = fmaf(wgt, pa[i].x, acc[0]);
                acc[1] = fmaf(wgt, pa[i].y, acc[1]);
                acc[2] = fmaf(wgt, pa[i].z, acc[2]);
                acc[3] = fmaf(wgt, pa[i].w, acc[3]);
            }
        }
        m = mn;
    }
}

// The same merge over the per-warp results (m, l, acc[128], at 0, 1 and 4 of
// each kPartialStride-float row) of the n <= 32 warps of a wide merge.
__device__ __forceinline__ void combine_slices(const float* sl, int n, int lane, float& m, float& l, float (&acc)[4]) {
    const float pm = lane < n ? sl[lane * kPartialStride] : -INFINITY;
    const float pl = lane < n ? sl[lane * kPartialStride + 1] : 0.f;
    m = warp_max(pm);
    if (m == -INFINITY) return;
    const float wl = (lane < n && pm != -INFINITY) ? exp2f(pm - m) : 0.f;
    l = warp_sum(pl * wl);
    for (int i = 0; i < n; ++i) {
        const float wgt = __shfl_sync(kFull, wl, i);
        const float4 pa = *reinterpret_cast<const float4*>(sl + i * kPartialStride + 4 + 4 * lane);
        acc[0] = fmaf(wgt, pa.x, acc[0]);
        acc[1] = fmaf(wgt, pa.y, acc[1]);
        acc[2] = fmaf(wgt, pa.z, acc[2]);
        acc[3] = fmaf(wgt, pa.w, acc[3]);
    }
}

// LSE slice of the raw tail rows r = first, first + step, ... < ntail (at most
// 64 / step of them) of one (row, query head): unrotated q (times sm_scale
// log2 e, this lane's 4 channels in qv) against the bf16 staging rows. Each
// lane scores its 4 channels of every row, a warp sum gives the score; m, l
// and acc (this lane's 4 channels) start at -inf, 0 and 0.
template <int B, int STEP>
__device__ __forceinline__ void tail_slice(const uint16_t* kst, int ntail, int first, const float (&qv)[4], int lane,
                                           float& m, float& l, float (&acc)[4]) {
    constexpr int R = (B + STEP - 1) / STEP;   // rows of this slice at most
    const uint16_t* vst = kst + B * kD;
    uint2 ku[R], vu[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int r = first + i * STEP;
        if (r < ntail) {
            ku[i] = reinterpret_cast<const uint2*>(kst + (int64_t)r * kD)[lane];
            vu[i] = reinterpret_cast<const uint2*>(vst + (int64_t)r * kD)[lane];
        }
    }
    float sc[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        float d = 0.f;
        if (first + i * STEP < ntail) {
            d = fmaf(qv[0], __uint_as_float(ku[i].x << 16), d);
            d = fmaf(qv[1], __uint_as_float(ku[i].x & 0xffff0000u), d);
            d = fmaf(qv[2], __uint_as_float(ku[i].y << 16), d);
            d = fmaf(qv[3], __uint_as_float(ku[i].y & 0xffff0000u), d);
        }
        sc[i] = d;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
        for (int i = 0; i < R; ++i) sc[i] += __shfl_xor_sync(kFull, sc[i], o);
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < R; ++i)
        if (first + i * STEP < ntail) mx = fmaxf(mx, sc[i]);
    if (mx == -INFINITY) return;
    m = mx;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        if (first + i * STEP < ntail) {
            const float p = exp2f(sc[i] - mx);
            l += p;
            acc[0] = fmaf(p, __uint_as_float(vu[i].x << 16), acc[0]);
            acc[1] = fmaf(p, __uint_as_float(vu[i].x & 0xffff0000u), acc[1]);
            acc[2] = fmaf(p, __uint_as_float(vu[i].y << 16), acc[2]);
            acc[3] = fmaf(p, __uint_as_float(vu[i].y & 0xffff0000u), acc[3]);
        }
    }
}

// One (row, query head) output: LSE-merge the np partials of its unit
// (p0: the first, consecutive partials G * kPartialStride floats apart; np =
// 0 when the unit has no pool blocks), add the raw tail rows, normalise and
// store. For the 2-bit cache (ROT = true) the merged accumulator is in the
// rotated space: it is rotated back once and the raw bf16 tail tokens
// (unrotated) are added; the bf16 cache (ROT = false) has every token in its
// pages. qsh: 128 floats of this warp's shared memory. gw = row * n_q +
// query head. With NWIDE > 0 (the wide merge's warp 0) the partials and the
// tail rows arrive as NWIDE per-warp LSE slices in shared memory (wide, tails).
template <int B, bool ROT, int NWIDE = 0>
__device__ __forceinline__ void merge_row(const AttnArgs& a, int64_t gw, int np, const float* p0, float* qsh,
                                          int lane, const float* wide = nullptr, const float* tails = nullptr) {
    const int b = (int)(gw / a.n_q), hq = (int)(gw % a.n_q);   // b: a (virtual) row sequence
    const int h = hq / a.G;
    const int rb = a.chunk == 1 ? b : b / a.chunk;              // its real sequence
    const int L = a.seq_lens[rb];
    float* out = a.out + gw * kD;
    if (L < 0 || L > a.max_blocks * B) {
        if (lane == 0) raise_error(a.err, KVARN_DEVERR_POSITION);
        reinterpret_cast<float4*>(out)[lane] = make_float4(NAN, NAN, NAN, NAN);
        return;
    }
    const SplitArgs sp{a.seq_lens, a.batch, a.n_kv, a.max_blocks, B, ROT ? 0 : 1, a.chunk};
    const int nb = split_nblocks(sp, b);
    // raw rows in staging (< B <= 64): the visible tokens past the pool blocks
    const int ntail = ROT ? max(0, split_visible(sp, b, L) - nb * B) : 0;
    float qt[4] = {0.f, 0.f, 0.f, 0.f};   // the query for the tail rows, loaded with them
    if (NWIDE == 0 && ntail > 0) {   // start the tail rows on their way to L1 while the partials merge
        load_q4(a.q, a.q_dtype, gw, lane, qt);
        const uint16_t* kst = a.staging + (((int64_t)rb * a.n_kv + h) * 2 + 0) * B * kD;
        for (int r = lane; r < ntail; r += 32) {
            prefetch_l1(kst + (int64_t)r * kD);
            prefetch_l1(kst + (int64_t)r * kD + 64);
            prefetch_l1(kst + (int64_t)(B + r) * kD);
            prefetch_l1(kst + (int64_t)(B + r) * kD + 64);
        }
    }
    float m = -INFINITY, l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (nb > 0 && np > 0) {
        if constexpr (NWIDE > 0) combine_slices(wide, NWIDE, lane, m, l, acc);
        else lse_partials(p0, np, (int64_t)a.G * kPartialStride, lane, m, l, acc);
        if (ROT && !(a.flags & KVARN_FLAG_NO_ROTATION)) {
            // rotate back: x = sigma . H(acc) / sqrt(128)
            fwht128(acc, lane);
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[k] *= kInvSqrtD * sign_of4(a.sb[0], a.sb[1], a.sb[2], a.sb[3], 4 * lane + k);
        }
    }
    if constexpr (NWIDE > 0) {
        // the wide merge's warps scored the tail rows: fold their slices in (the
        // slices are unrotated, like the accumulator after the inverse FWHT)
        float mt = -INFINITY, lt = 0.f, at[4] = {0.f, 0.f, 0.f, 0.f};
        if (ntail > 0) combine_slices(tails, NWIDE, lane, mt, lt, at);
        if (mt != -INFINITY) {
            const float mn = fmaxf(m, mt);
            const float fa = m == -INFINITY ? 0.f : exp2f(m - mn), ft = exp2f(mt - mn);
            l = l * fa + lt * ft;
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[k] = acc[k] * fa + at[k] * ft;
            m = mn;
        }
    } else if (ntail > 0) {
        // this warp's query (unrotated, times sm_scale log2 e) in shared memory, so
        // that lane r can score tail row r (and r + 32) over all 128 channels
        // with its loads issued at once
        __syncwarp();
        {
            const float qs = a.sm_scale * kLog2e;
            *reinterpret_cast<float4*>(qsh + 4 * lane) = make_float4(qt[0] * qs, qt[1] * qs, qt[2] * qs, qt[3] * qs);
        }
        __syncwarp();
        const uint16_t* kst = a.staging + (((int64_t)rb * a.n_kv + h) * 2 + 0) * B * kD;
        const uint16_t* vst = kst + B * kD;
        float mine[2] = {-INFINITY, -INFINITY};   // scores of rows lane, lane + 32
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = lane + 32 * half;
            if (half * 32 < ntail && r < ntail) {
                const uint4* kr = reinterpret_cast<const uint4*>(kst + (int64_t)r * kD);
                float d = 0.f;
#pragma unroll
                for (int c0 = 0; c0 < 16; c0 += 8) {
                uint4 ku[16];
#pragma unroll
                for (int c = c0; c < c0 + 8; ++c) ku[c] = kr[c];
#pragma unroll
                for (int c = c0; c < c0 + 8; ++c) {
                    const float4 qa = *reinterpret_cast<const float4*>(qsh + 8 * c);
                    const float4 qb = *reinterpret_cast<const float4*>(qsh + 8 * c + 4);
                    d = fmaf(qa.x, __uint_as_float(ku[c].x << 16), d);
                    d = fmaf(qa.y, __uint_as_float(ku[c].x & 0xffff0000u), d);
                    d = fmaf(qa.z, __uint_as_float(ku[c].y << 16), d);
                    d = fmaf(qa.w, __uint_as_float(ku[c].y & 0xffff0000u), d);
                    d = fmaf(qb.x, __uint_as_float(ku[c].z << 16), d);
                    d = fmaf(qb.y, __uint_as_float(ku[c].z & 0xffff0000u), d);
                    d = fmaf(qb.z, __uint_as_float(ku[c].w << 16), d);
                    d = fmaf(qb.w, __uint_as_float(ku[c].w & 0xffff0000u), d);
                }
                }
                mine[half] = d;
            }
        }
        const float mt = warp_max(fmaxf(mine[0], mine[1]));
        const float mn = fmaxf(m, mt);                      // finite: ntail > 0
        const float fa = (m == -INFINITY) ? 0.f : exp2f(m - mn);
        const float p0t = exp2f(mine[0] - mn), p1t = exp2f(mine[1] - mn);   // 0 for empty slots
        l = l * fa + warp_sum(p0t + p1t);
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] *= fa;
        m = mn;
        // values: 8 rows per step, their loads independent of each other
        for (int r0 = 0; r0 < ntail; r0 += 8) {
            uint2 vu[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (r0 + k < ntail) vu[k] = reinterpret_cast<const uint2*>(vst + (int64_t)(r0 + k) * kD)[lane];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int r = r0 + k;
                if (r < ntail) {
                    const float p = __shfl_sync(kFull, (r < 32) ? p0t : p1t, r & 31);
                    acc[0] = fmaf(p, __uint_as_float(vu[k].x << 16), acc[0]);
                    acc[1] = fmaf(p, __uint_as_float(vu[k].x & 0xffff0000u), acc[1]);
                    acc[2] = fmaf(p, __uint_as_float(vu[k].y << 16), acc[2]);
                    acc[3] = fmaf(p, __uint_as_float(vu[k].y & 0xffff0000u), acc[3]);
                }
            }
        }
    }
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
    reinterpret_cast<float4*>(out)[lane] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
}

// The partials of row gw's unit: their count np and the first p0 (np = 0
// when the unit has no pool blocks or the row's length is out of range).
template <int B, bool ROT>
__device__ __forceinline__ void merge_locate(const AttnArgs& a, int64_t gw, int lane, int& np, const float*& p0) {
    np = 0;
    p0 = nullptr;
    const int b = (int)(gw / a.n_q), hq = (int)(gw % a.n_q);
    const int h = hq / a.G, jq = hq % a.G;
    const int rb = a.chunk == 1 ? b : b / a.chunk;
    const int64_t u = (int64_t)b * a.n_kv + h;
    // the unit map entry does not depend on the length: both loads in flight at once
    int2 wm = make_int2(-1, -1);
    if (a.unit_map != nullptr) wm = __ldcg(reinterpret_cast<const int2*>(a.unit_map) + u);
    const int L = a.seq_lens[rb];
    if (L < 0 || L > a.max_blocks * B) return;
    const SplitArgs sp{a.seq_lens, a.batch, a.n_kv, a.max_blocks, B, ROT ? 0 : 1, a.chunk};
    const int nb = split_nblocks(sp, b);
    if (nb <= 0) return;
    if (a.unit_map != nullptr) {
        // a range outside the grid (a warp gave up before recording it, its
        // error flag set) merges nothing rather than reading out of bounds
        if (wm.x >= 0 && wm.y >= wm.x && wm.y < a.nw) {
            np = wm.y - wm.x + 1;
            p0 = a.partials + ((u + wm.x) * a.G + jq) * kPartialStride;
        }
    } else if (a.single > 0) {
        np = a.single;
        p0 = a.partials + (u * a.single * a.G + jq) * kPartialStride;
    } else {
        int64_t before, total;
        split_prefix(sp, b, lane, before, total);
        const int64_t W = total * a.n_kv;
        const int64_t nwe = split_active_warps(W, a.nw, (int64_t)a.batch * a.n_kv, ROT ? kSplitRatio2bit * B : 0.f);
        const int64_t Su = before * a.n_kv + (int64_t)h * nb;
        const int64_t w0 = split_last_warp_at(Su, W, nwe), w1 = split_last_warp_at(Su + nb - 1, W, nwe);
        np = (int)(w1 - w0 + 1);
        p0 = a.partials + ((u + w0) * a.G + jq) * kPartialStride;
    }
}

// The merge kernel: one warp per (row, query head), which finds its unit's
// partials from the split arithmetic or the split kernel's unit map.
template <int B, bool ROT>
__global__ void __launch_bounds__(128) merge_kernel(AttnArgs a) {
    wait_prior_grids();
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (gw >= (int64_t)a.batch * a.n_q) return;
    __shared__ __align__(16) float q_all[4][kD];
    int np;
    const float* p0;
    merge_locate<B, ROT>(a, gw, lane, np, p0);
    merge_row<B, ROT>(a, gw, np, p0, q_all[threadIdx.x >> 5], lane);
}

// The wide merge, for units cut into many partials (few long sequences) or
// few enough rows for one wave of its CTAs: one CTA of kWideWarps warps per
// (row, query head). Warp k LSE-merges its
// share of the unit's partials and scores its share of the raw tail rows
// (rows k, k + kWideWarps, ...); the shares meet in shared memory and warp 0
// combines the partials, rotates them back, folds in the tail shares and
// finishes the row.
// NB: partials per load round trip of a warp's LSE merge. With 8 the kernel
// needs 110 registers (2 CTAs per SM); with 4, 64 (4 CTAs per SM).
constexpr int kWideWarps = 8;
template <int B, bool ROT, int NB>
__global__ void __launch_bounds__(32 * kWideWarps, NB == 8 ? 2 : 4) merge_wide_kernel(AttnArgs a) {
    wait_prior_grids();
    const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
    const int64_t gw = blockIdx.x;
    if (gw >= (int64_t)a.batch * a.n_q) return;   // (uniform over the CTA)
    __shared__ __align__(16) float slices[kWideWarps][kPartialStride];
    __shared__ __align__(16) float tails[kWideWarps][kPartialStride];
    __shared__ __align__(16) float qsh[kD];
    // q (for the raw tail rows) and the unit's length and partial range are
    // independent loads: issue them together
    float qv[4] = {0.f, 0.f, 0.f, 0.f};
    if (ROT) load_q4(a.q, a.q_dtype, gw, lane, qv);
    int np;
    const float* p0;
    merge_locate<B, ROT>(a, gw, lane, np, p0);
    // this warp's share of the raw tail rows (2-bit cache): rows wp, wp + 8, ...;
    // their lines are requested now and read after the partials' LSE merge
    int ntail = 0;
    const uint16_t* kst = nullptr;
    if (ROT) {
        const int b = (int)(gw / a.n_q), h = (int)(gw % a.n_q) / a.G;
        const int rb = a.chunk == 1 ? b : b / a.chunk;
        const int L = a.seq_lens[rb];
        if (L >= 0 && L <= a.max_blocks * B) {
            const SplitArgs sp{a.seq_lens, a.batch, a.n_kv, a.max_blocks, B, 0, a.chunk};
            ntail = max(0, split_visible(sp, b, L) - split_nblocks(sp, b) * B);
            kst = a.staging + (((int64_t)rb * a.n_kv + h) * 2 + 0) * B * kD;
            // lane: row wp + 8 (lane / 4), K or V (bit 1), first or second 128-byte line (bit 0)
            constexpr int R = (B + kWideWarps - 1) / kWideWarps;
            const int r = wp + kWideWarps * (lane >> 2);
            if ((lane >> 2) < R && r < ntail)
                prefetch_l1(kst + ((lane & 2) ? B * kD : 0) + (int64_t)r * kD + (lane & 1) * 64);
        }
    }
    float m = -INFINITY, l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    const int i0 = (int)((int64_t)np * wp / kWideWarps), i1 = (int)((int64_t)np * (wp + 1) / kWideWarps);
    const int64_t pstride = (int64_t)a.G * kPartialStride;
    if (i1 > i0) lse_stream<NB>(p0 + i0 * pstride, i1 - i0, pstride, lane, m, l, acc);
    float tm = -INFINITY, tl = 0.f, tacc[4] = {0.f, 0.f, 0.f, 0.f};
    if (wp < ntail) {
        const float qs = a.sm_scale * kLog2e;
#pragma unroll
        for (int k = 0; k < 4; ++k) qv[k] *= qs;
        tail_slice<B, kWideWarps>(kst, ntail, wp, qv, lane, tm, tl, tacc);
    }
    if (lane == 0) {
        slices[wp][0] = m;
        slices[wp][1] = l;
        tails[wp][0] = tm;
        tails[wp][1] = tl;
    }
    *reinterpret_cast<float4*>(&slices[wp][4 + 4 * lane]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(&tails[wp][4 + 4 * lane]) = make_float4(tacc[0], tacc[1], tacc[2], tacc[3]);
    __syncthreads();
    if (wp == 0) merge_row<B, ROT, kWideWarps>(a, gw, np, p0, qsh, lane, &slices[0][0], &tails[0][0]);
}

// Whether the merge of a launch with nw split warps over `units` (sequence,
// kv head) units and `rows` query rows takes the wide kernel: 16 or more
// partials per unit on average, or no more rows than wide_rows (the 2-bit
// cache: one wave of wide CTAs, so that 8 warps share each row's raw tail
// rows; 0 for the bf16 cache, which has no tail rows).
inline bool merge_wide(int64_t nw, int64_t units, int64_t rows, int64_t wide_rows) {
    return nw >= 16 * units || rows <= wide_rows;
}

// The wide merge's partials per round trip: 8 when its warps average more
// than 4 partials each and the rows fit one wave at 2 CTAs per SM (few long
// sequences), else 4.
inline int wide_merge_batch(int64_t nw, int64_t units, int64_t rows, int64_t sms) {
    return (nw > 4 * kWideWarps * units && rows <= 2 * sms) ? 8 : 4;
}

// SMs of the current device (cached per device; 0 when it cannot be queried).
inline int64_t current_device_sms() {
    static int cache[64];
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return 0;
    if (cache[d] <= 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return 0;
        cache[d] = sms;
    }
    return cache[d];
}

// Launches the merge of a split launch with nw warps: the wide kernel (with
// its batch) or the one-warp-per-row kernel. wide_ctas_per_sm > 0 also takes
// the wide kernel for up to that many rows per SM.
template <int B, bool ROT>
cudaError_t launch_merge(const AttnArgs& a, int64_t nw, int wide_ctas_per_sm, cudaStream_t st) {
    const int64_t units = (int64_t)a.batch * a.n_kv, rows = (int64_t)a.batch * a.n_q;
    const int64_t sms = current_device_sms();
    if (merge_wide(nw, units, rows, wide_ctas_per_sm * sms)) {
        if (wide_merge_batch(nw, units, rows, sms) == 8)
            return launch_pdl(merge_wide_kernel<B, ROT, 8>, (unsigned)rows, 32 * kWideWarps, 0, st, a);
        return launch_pdl(merge_wide_kernel<B, ROT, 4>, (unsigned)rows, 32 * kWideWarps, 0, st, a);
    }
    return launch_pdl(merge_kernel<B, ROT>, (unsigned)((rows + 3) / 4), 128, 0, st, a);
}

}  // namespace kvarn
