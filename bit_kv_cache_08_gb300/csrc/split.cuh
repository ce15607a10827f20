// split.cuh -- balanced split-K partition shared by the decode-attention
// kernels, and the per-row block counts the merge uses for chunked prefill
// (every query row of a chunk is a virtual sequence of its own: virtual
// v = b * chunk + r sees the causal prefix of real sequence b). The (sequence, kv head) units are laid end to end, block by block
// (sequence-major, then head, then block); warp w of the nw active warps
// (nw = min(resident warps, W)) takes global blocks [floor(w*W/nw),
// floor((w+1)*W/nw)), at least one. A unit's partial from warp w lives in slot
// (unit + w), which is unique because a later unit's warps never come before
// an earlier unit's; the warps of one unit are consecutive.
#pragma once
#include "common.cuh"

namespace kvarn {

constexpr int kPartialStride = 132;   // floats per (slot, head): m, l, pad, pad, acc[128]

struct SplitArgs {
    const int32_t* seq_lens;
    int batch;
    int n_kv;
    int max_blocks;
    int B;
    int ceil_blocks;   // 1: a partial last block counts (bf16 pages); 0: full blocks only
    int chunk;         // query rows per real sequence (1: decode); batch counts virtual sequences
};

// Tokens virtual sequence v may see: the causal prefix 0 .. L - chunk + r of
// its real sequence (L itself when chunk = 1); <= 0 sees nothing.
__device__ __forceinline__ int split_visible(const SplitArgs& s, int v, int L) {
    if (s.chunk == 1) return L;
    const int b = v / s.chunk;
    return L - s.chunk + 1 + (v - b * s.chunk);
}

// Pool blocks a (virtual) sequence reads: its complete blocks (all blocks for
// bf16 pages), cut at the last one holding a visible token.
__device__ __forceinline__ int split_nblocks(const SplitArgs& s, int v) {
    const int L = s.seq_lens[s.chunk == 1 ? v : v / s.chunk];
    if (L < 0 || L > s.max_blocks * s.B) return 0;   // flagged by the merge kernel
    const int full = s.ceil_blocks ? (L + s.B - 1) / s.B : L / s.B;
    if (s.chunk == 1) return full;
    const int vis = split_visible(s, v, L);
    const int cap = vis > 0 ? (vis + s.B - 1) / s.B : 0;
    return cap < full ? cap : full;
}

// Warp-cooperative: returns W (total blocks over all units); if x < W, sets
// (b, h, j) of global position x.
__device__ __forceinline__ int64_t split_locate(const SplitArgs& s, int64_t x, int lane, int& b_out,
                                       int& h_out, int& j_out) {
    int64_t prefix = 0;
    int found_b = -1;
    int64_t found_base = 0;
    for (int b0 = 0; b0 < s.batch; b0 += 32) {
        const int b = b0 + lane;
        const int64_t nb = (b < s.batch) ? (int64_t)split_nblocks(s, b) * s.n_kv : 0;
        int64_t inc = nb;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const int64_t o = __shfl_up_sync(kFull, inc, m);
            if (lane >= m) inc += o;
        }
        const int64_t excl = prefix + inc - nb;
        const bool hit = found_b < 0 && nb > 0 && x >= excl && x < excl + nb;
        const uint32_t ball = __ballot_sync(kFull, hit);
        if (ball) {
            const int src = __ffs(ball) - 1;
            found_b = b0 + src;
            found_base = __shfl_sync(kFull, excl, src);
        }
        prefix += __shfl_sync(kFull, inc, 31);
    }
    if (found_b >= 0) {
        const int nb = split_nblocks(s, found_b);
        const int64_t local = x - found_base;
        b_out = found_b;
        h_out = (int)(local / nb);
        j_out = (int)(local % nb);
    }
    return prefix;
}

struct Cursor {
    int b, h, j, nb;
};

__device__ __forceinline__ void split_advance(const SplitArgs& s, Cursor& c) {
    if (++c.j < c.nb) return;
    c.j = 0;
    if (++c.h < s.n_kv) return;
    c.h = 0;
    do {
        ++c.b;
        c.nb = (c.b < s.batch) ? split_nblocks(s, c.b) : 1;
    } while (c.nb == 0);
}

// Blocks of all sequences before b, and of all sequences (warp-cooperative).
__device__ __forceinline__ void split_prefix(const SplitArgs& s, int b, int lane, int64_t& before,
                                    int64_t& total) {
    before = 0;
    total = 0;
#pragma unroll 4
    for (int b0 = 0; b0 < s.batch; b0 += 32) {
        const int bb = b0 + lane;
        const int64_t nb = (bb < s.batch) ? (int64_t)split_nblocks(s, bb) : 0;
        total += warp_sum_i64(nb);
        before += warp_sum_i64(bb < b ? nb : 0);
    }
}

// Warps that take part in a split of W blocks (units = sequences x kv heads)
// over at most nw warps. Never more than there are blocks, so that every
// active warp owns at least one block and a unit's partials sit in
// consecutive slots. With ratio > 0, also at most sqrt(ratio * W * units):
// a warp's time grows with its blocks (W / n) while the merge of a unit
// grows with its partials (n / units); their sum is least near
// n = sqrt(ratio * W * units), ratio being the cost of a block over that of
// merging one partial. This only bites when few long units would otherwise
// be cut into hundreds of single-block partials (batch 1, long contexts).
__host__ __device__ __forceinline__ int64_t split_active_warps(int64_t W, int64_t nw, int64_t units,
                                                               float ratio) {
    int64_t n = W < nw ? W : nw;
    if (ratio > 0.f) {
        const int64_t c = (int64_t)sqrtf(ratio * (float)W * (float)units);
        if (c < n) n = c > 1 ? c : 1;
    }
    return n;
}

// Largest w in [0, nw) with floor(w*W/nw) <= x.
__host__ __device__ __forceinline__ int64_t split_last_warp_at(int64_t x, int64_t W, int64_t nw) {
    const int64_t r = ((x + 1) * nw - 1) / W;
    return r < nw - 1 ? r : nw - 1;
}

}  // namespace kvarn
