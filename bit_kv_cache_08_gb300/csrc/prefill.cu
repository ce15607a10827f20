// prefill.cu -- chunked prefill attention over the KVarN paged cache (2-, 3-
// or 4-bit codes; sm_103a): the query rows of a chunk share one pass over
// each cache block.
//
// Method: "KVarN：方差归一化让 2-bit KV 缓存扛住长链推理", section 三 3.1 (the
// query multiplied by the same randomised Hadamard matrix as K and V) and 3.2
// (the stored scales applied again when the cache is read), extended from the
// decode step to the rows of a chunk: row r of a chunk of C rows sits at
// position L - C + r of its sequence and sees tokens 0 .. L - C + r, read from
// the cache as it stands.
//
// One warp owns 8 query vectors of one (sequence, kv head): P = 8 / G chunk
// rows x G query heads (vector v = row v / G, head v % G). Unlike the decode
// kernel (keys as MMA rows, the 4 heads of one row as columns), the vectors
// are the MMA rows and the keys the columns, so every 2-bit code is turned
// into a tensor-core operand once for all 8 vectors:
//   QK  A = q' (vector gq in row gq as fp16 hi, row gq + 8 as lo), B = the
//       K codes straight from the lane's record as raw fp16 subnormals (a
//       shifted or byte-swapped view of the word and one mask: even fields
//       code * 2^-16 at bits 8..9, odd fields code * 2^-18 at bits 6..7,
//       exact on the tensor cores at those positions; q' of the odd k-slots
//       x 4; n-tile i holds tokens 4n + i of a 32-token sub-block); one
//       accumulator per 32-channel group
//   the score accumulator layout leaves lane (gq, tq) with tokens
//   8tq .. 8tq + 7 of each sub-block for vector gq, which is exactly the
//   A-operand layout of the PV product, so P never leaves registers
//   PV  A = P'_g = p R s_g lam (hi rows, lo rows), B = the V codes
//       (n = channel, k = token; the odd fields' output columns x 4), one
//       group at a time; the block's result is folded into O with the
//       per-channel factor C / (kA lam) at once.
//       P' is an fp16 two-product of P'' = p R lam (hi | lo once per token)
//       with the group's steps; the zero-point sums of all groups come from
//       two MMAs per 32 tokens (B columns z_0..z_3 | s_0..s_3).
// K and V head-blocks stream through a shared-memory ring filled by 1-D bulk
// copies (lane 0) counted on mbarriers with bounded waits. Each (sequence,
// kv head, row tile) unit's blocks are split over 1 to 16 warps, chosen from
// the unit count and the kernel's resident warps (prefill_splits). Each vector's (max,
// sum, 128 rotated accumulators) per split goes to one workspace partial;
// the merge kernel combines a row's partials, adds the raw bf16 tail rows,
// rotates back once and normalises. 3- and 4-bit codes take the same path with 48- and 64-byte
// records, their operands code * 2^-9 (a mask and one fp16 multiply per pair).
#include <algorithm>

#include "attn_common.cuh"

namespace kvarn {

namespace {

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// halves i and i + 4 (i = 0..3) of 8 fp16 at a 16-byte aligned shared address,
// as an fp32 pair
__device__ __forceinline__ float2 pair_i4(const uint4& u, int i) {
    const __half2 a = u32_as_h2(i < 2 ? u.x : u.y), b = u32_as_h2(i < 2 ? u.z : u.w);
    return __half22float2((i & 1) ? __highs2half2(a, b) : __lows2half2(a, b));
}

}  // namespace

constexpr int kPrefillVecs = 8;   // query vectors per warp

template <int B>
constexpr int prefill_stages() { return B == 32 ? 4 : 2; }

template <int B, int BITS>
constexpr size_t prefill_smem_bytes() {
    return (size_t)prefill_stages<B>() * 2 * head_block_bytes(B, BITS) + 64 + 2 * kPrefillVecs * kD * 2 +
           kPrefillVecs * 4;
}

template <int B, int BITS, int S>
__global__ void __launch_bounds__(32) prefill_attn_kernel(AttnArgs a) {
    static_assert(BITS >= 2 && BITS <= 4, "2-, 3- or 4-bit codes");
    wait_prior_grids();
    constexpr int HB = head_block_bytes(B, BITS);
    constexpr int NSB = B / 32;
    constexpr int RW = 4 * BITS;              // 32-bit words per lane record
    // kA: the operand scale of a code (2-bit: even fields' raw subnormals)
    constexpr float kA = BITS == 2 ? kRawScale : kCodeScale;
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t* stages = smem;                                                    // S x (K, V)
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * 2 * HB);           // S mbarriers
    uint16_t* qh_s = reinterpret_cast<uint16_t*>(smem + S * 2 * HB + 64);      // [8][128] fp16 hi
    uint16_t* ql_s = qh_s + kPrefillVecs * kD;                                 // [8][128] fp16 lo
    float* kmul_s = reinterpret_cast<float*>(ql_s + kPrefillVecs * kD);        // [8]

    const int lane = threadIdx.x;
    const int gq = lane >> 2, tq = lane & 3;

    const int G = a.G, n_kv = a.n_kv, n_q = a.n_q, chunk = a.chunk, max_blocks = a.max_blocks;
    const int P = kPrefillVecs / G;                       // chunk rows per warp
    const int tiles = (chunk + P - 1) / P;
    const int NS = a.single;                              // block ranges per (row tile, kv head)
    const int64_t w = blockIdx.x;
    const int split = (int)(w % NS);
    const int64_t wu = w / NS;
    const int tile = (int)(wu % tiles);
    const int h = (int)((wu / tiles) % n_kv);
    const int b = (int)(wu / tiles / n_kv);
    if (b >= a.batch) return;
    const int L = a.seq_lens[b];
    if (L < 0 || L > max_blocks * B) return;               // flagged by the merge kernel
    const int r0 = tile * P;
    const uint8_t* __restrict__ pool = a.pool;
    uint32_t* err = a.err;
    const int64_t n_pool_blocks = a.n_pool_blocks, block_bytes = a.block_bytes;

    // this lane's vector (row gq of the MMAs) and the tokens it may see
    const int my_row = r0 + gq / G;
    const bool my_ok = gq < P * G && my_row < chunk;
    const int my_vis = my_ok ? L - chunk + my_row + 1 : 0;
    // the warp's last row sees the most
    const int last_row = min(chunk - 1, r0 + P - 1);
    const int max_vis = L - chunk + last_row + 1;
    const int nvis = max_vis > 0 ? min(L / B, (max_vis + B - 1) / B) : 0;
    // this warp's share of those blocks (possibly none: its partial is then empty)
    const int jb = (int)((int64_t)split * nvis / NS), je = (int)((int64_t)(split + 1) * nvis / NS);
    const int nblk = je - jb;

    // ---- queries: rotate, scale to 2^12, fp16 hi | lo in shared memory
    {
        const bool rotate = !(a.flags & KVARN_FLAG_NO_ROTATION);
        const float sgn[4] = {sign_of4(a.sb[0], a.sb[1], a.sb[2], a.sb[3], 4 * lane),
                              sign_of4(a.sb[0], a.sb[1], a.sb[2], a.sb[3], 4 * lane + 1),
                              sign_of4(a.sb[0], a.sb[1], a.sb[2], a.sb[3], 4 * lane + 2),
                              sign_of4(a.sb[0], a.sb[1], a.sb[2], a.sb[3], 4 * lane + 3)};
        for (int v = 0; v < kPrefillVecs; ++v) {
            const int row = r0 + v / G;
            float x[4] = {0.f, 0.f, 0.f, 0.f};
            float km = 0.f;
            if (v < P * G && row < chunk) {
                load_q4(a.q, a.q_dtype, ((int64_t)b * chunk + row) * n_q + (int64_t)h * G + v % G, lane, x);
                if (rotate) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) x[k] *= sgn[k];
                    fwht128(x, lane);
#pragma unroll
                    for (int k = 0; k < 4; ++k) x[k] *= kInvSqrtD;
                }
                float amax = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fabsf(x[k]));
                amax = warp_max(amax);
                const int e = (amax > 0.f && isfinite(amax)) ? ceil_log2(amax) : 0;
                const float sc = exp2i(12 - e);
#pragma unroll
                for (int k = 0; k < 4; ++k) x[k] *= sc;
                km = (1.0f / kA) * exp2i(e - 12) * a.sm_scale * kLog2e;
            }
            uint16_t hi[4], lo[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const __half hh = __float2half_rn(x[k]);
                hi[k] = __half_as_ushort(hh);
                lo[k] = f2h_rn(x[k] - __half2float(hh));
            }
            *reinterpret_cast<uint2*>(qh_s + v * kD + 4 * lane) =
                make_uint2(hi[0] | ((uint32_t)hi[1] << 16), hi[2] | ((uint32_t)hi[3] << 16));
            *reinterpret_cast<uint2*>(ql_s + v * kD + 4 * lane) =
                make_uint2(lo[0] | ((uint32_t)lo[1] << 16), lo[2] | ((uint32_t)lo[3] << 16));
            if (lane == 0) kmul_s[v] = km;
        }
    }
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const float kmul = my_ok ? kmul_s[gq] : 0.f;

    // ---- block ring
    const int32_t* __restrict__ btab = a.block_table + (int64_t)b * max_blocks;
    uint32_t okmask = 0;
    auto issue = [&](int j, int stage) {
        int64_t phys = btab[jb + j];
        const bool ok = phys >= 0 && phys < n_pool_blocks;
        if (!ok) phys = 0;   // read a valid block, result discarded below
        if (lane == 0) {
            const uint8_t* src = pool + phys * block_bytes + (int64_t)(2 * h) * HB;
            mbar_arrive_expect_tx(&bars[stage], 2 * HB);
            bulk_g2s(stages + stage * 2 * HB, src, 2 * HB, &bars[stage]);
        }
        return ok;
    };
    for (int s = 0; s < S && s < nblk; ++s)
        if (issue(s, s)) okmask |= 1u << s;

    float m_run = -INFINITY, l_part = 0.f;
    float2 O[4][4];   // vector gq, channels 32g + 8tq + f and + 4 + f
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int f = 0; f < 4; ++f) O[g][f] = make_float2(0.f, 0.f);

    int stage = 0;
    uint32_t phase = 0;
    for (int j = 0; j < nblk; ++j) {
        if (!mbar_wait_bounded(&bars[stage], phase, kWaitLimit)) {
            if (lane == 0) raise_error(err, KVARN_DEVERR_WAIT_TIMEOUT);
            uint32_t ph = phase;
            for (int k = 0, st2 = stage; k < S && j + k < nblk; ++k) {
                mbar_wait_bounded(&bars[st2], ph, kWaitLimit);
                if (++st2 == S) { st2 = 0; ph ^= 1u; }
            }
            return;
        }
        const uint8_t* Kb = stages + stage * 2 * HB;
        const uint8_t* Vb = Kb + HB;
        const bool valid = (okmask >> stage) & 1u;
        if (!valid && lane == 0) raise_error(err, KVARN_DEVERR_BLOCK_ID);

        if (valid) {
            const uint16_t* KC = reinterpret_cast<const uint16_t*>(Kb + off_C(B, BITS));
            // ---- per-block power of two bringing max C to (1/2, 1]
            float cmax;
            {
                const uint2 c2 = *reinterpret_cast<const uint2*>(KC + 4 * lane);
                const __half2 m2 = __hmax2(u32_as_h2(c2.x), u32_as_h2(c2.y));
                cmax = warp_max(fmaxf(__low2float(m2), __high2float(m2)));
            }
            const int ec = ceil_log2(fmaxf(cmax, kF16MinNormal));
            const __half2 cinv = __float2half2_rn(exp2i(-ec));
            // 2-bit: the odd k-slot of each pair meets codes at 2^-18, so its q' is x 4
            const __half2 cinv_o = BITS == 2 ? __float2half2_rn(exp2i(2 - ec)) : cinv;
            const float kmb = kmul * exp2i(ec);
            // ---- QK A operand for vector gq: q' = q_s * C * 2^-ec, hi (row gq) | lo (row gq + 8)
            uint32_t qa_h[16], qa_l[16];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const uint4 c4 = *reinterpret_cast<const uint4*>(KC + 32 * g + 8 * tq);
                const uint4 h4 = *reinterpret_cast<const uint4*>(qh_s + gq * kD + 32 * g + 8 * tq);
                const uint4 l4 = *reinterpret_cast<const uint4*>(ql_s + gq * kD + 32 * g + 8 * tq);
                const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
                const uint32_t hw[4] = {h4.x, h4.y, h4.z, h4.w};
                const uint32_t lw[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const __half2 C2 = __hmul2(u32_as_h2(cw[e2]), (e2 & 1) ? cinv_o : cinv);
                    const __half2 qh = u32_as_h2(hw[e2]);
                    const __half2 hi = __hmul2(qh, C2);
                    __half2 lo = __hfma2(qh, C2, __hneg2(hi));
                    lo = __hfma2(u32_as_h2(lw[e2]), C2, lo);
                    qa_h[4 * g + e2] = h2_as_u32(hi);
                    qa_l[4 * g + e2] = h2_as_u32(lo);
                }
            }
            // ---- Q'_g * kA of vector gq: the same A against a B of codes of 1
            constexpr uint32_t kOneE = BITS == 2 ? kRawOneEven : kCodeScaleH2;
            constexpr uint32_t kOneO = BITS == 2 ? kRawOneOdd : kCodeScaleH2;
            float Qq[4];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                float d[4];
                mma16816_acc(d, true, qa_h[4 * g], qa_l[4 * g], qa_h[4 * g + 1], qa_l[4 * g + 1], kOneE, kOneO);
                mma16816(d, qa_h[4 * g + 2], qa_l[4 * g + 2], qa_h[4 * g + 3], qa_l[4 * g + 3], kOneE, kOneO);
                Qq[g] = d[0] + d[2];
            }
            const uint16_t* Ks = reinterpret_cast<const uint16_t*>(Kb + off_s(B, BITS));
            const uint16_t* Kz = reinterpret_cast<const uint16_t*>(Kb + off_z(B, BITS));
            const uint16_t* KR = reinterpret_cast<const uint16_t*>(Kb + off_R(B, BITS));

            // ---------------- QK: scores of tokens 32sb + 8tq + {0..7} for vector gq
            float sc[NSB][8];
#pragma unroll
            for (int sb = 0; sb < NSB; ++sb) {
                uint32_t kw[RW], kw8[RW];
                {
                    const uint4* rec = reinterpret_cast<const uint4*>(Kb) + (RW / 4) * (32 * sb + lane);
#pragma unroll
                    for (int r = 0; r < RW / 4; ++r) {
                        const uint4 rr = rec[r];
                        kw[4 * r] = rr.x; kw[4 * r + 1] = rr.y; kw[4 * r + 2] = rr.z; kw[4 * r + 3] = rr.w;
                    }
                }
#pragma unroll
                for (int k = 0; k < RW; ++k) kw8[k] = kw[k] >> 8;
                const int t0 = 32 * sb + 8 * tq;
                // R, s and z of tokens (t0 + i, t0 + 4 + i) as fp32 pairs
                float2 Rv[4], sv[4][4], zv[4][4];
                {
                    const uint4 r4 = *reinterpret_cast<const uint4*>(KR + t0);
#pragma unroll
                    for (int i = 0; i < 4; ++i) Rv[i] = pair_i4(r4, i);
                }
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const uint4 s4 = *reinterpret_cast<const uint4*>(Ks + g * B + t0);
                    const uint4 z4 = *reinterpret_cast<const uint4*>(Kz + g * B + t0);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        sv[g][i] = pair_i4(s4, i);
                        zv[g][i] = pair_i4(z4, i);
                    }
                }
                const float2 kmb2 = make_float2(kmb, kmb);
#pragma unroll
                for (int i = 0; i < 4; ++i) {   // n-tile i: tokens 4n + i; this lane's columns 2tq, 2tq + 1
                    float acc[4][4];
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            uint32_t b0, b1;
                            if (BITS == 2) {   // word 2i + g/2, pair 4(g%2) + e/2
                                const int wi = 2 * i + (g >> 1), jj = 4 * (g & 1) + 2 * kk;
                                b0 = code2_r(code2_view(kw[wi], code2_view_of(jj)), jj);
                                b1 = code2_r(code2_view(kw[wi], code2_view_of(jj + 1)), jj + 1);
                            } else if (BITS == 3) {   // + the high bit: word 8 + i, bit 8(g/2) + pair
                                const int wi = 2 * i + (g >> 1), jj = 4 * (g & 1) + 2 * kk, wh = 8 + i;
                                const int jh = 8 * (g >> 1) + jj;
                                b0 = code3_s(kw[wi], kw8[wi], kw[wh], jj, jh);
                                b1 = code3_s(kw[wi], kw8[wi], kw[wh], jj + 1, jh + 1);
                            } else {           // word 4i + g, field e/2
                                const int wi = 4 * i + g;
                                b0 = code4_s(kw[wi], kw8[wi], 2 * kk);
                                b1 = code4_s(kw[wi], kw8[wi], 2 * kk + 1);
                            }
                            const int qi = 4 * g + 2 * kk;
                            mma16816_acc(acc[g], kk == 0, qa_h[qi], qa_l[qi], qa_h[qi + 1], qa_l[qi + 1], b0, b1);
                        }
                    }
                    // column 2tq: token t0 + i; column 2tq + 1: token t0 + 4 + i (hi + lo rows)
                    float2 s_ = make_float2(0.f, 0.f);
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const float2 d = __fadd2_rn(make_float2(acc[g][0], acc[g][1]), make_float2(acc[g][2], acc[g][3]));
                        s_ = __ffma2_rn(sv[g][i], d, s_);
                        s_ = __ffma2_rn(zv[g][i], make_float2(Qq[g], Qq[g]), s_);
                    }
                    const float2 v = __fmul2_rn(__fmul2_rn(s_, Rv[i]), kmb2);
                    sc[sb][i] = v.x;
                    sc[sb][i + 4] = v.y;
                }
            }
            // causal cut: tokens at or past this vector's visible length
            const int lim = my_vis - (jb + j) * B;
            if (__any_sync(kFull, lim < B)) {
#pragma unroll
                for (int sb = 0; sb < NSB; ++sb)
#pragma unroll
                    for (int tt = 0; tt < 8; ++tt)
                        if (32 * sb + 8 * tq + tt >= lim) sc[sb][tt] = -INFINITY;
            }

            // ---------------- online softmax of vector gq (its 4 lanes hold the block)
            float bm = -INFINITY;
#pragma unroll
            for (int sb = 0; sb < NSB; ++sb)
#pragma unroll
                for (int tt = 0; tt < 8; ++tt) bm = fmaxf(bm, sc[sb][tt]);
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 1));
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 2));
            const float m_new = fmaxf(m_run, bm);
            const float alpha = (m_new == -INFINITY) ? 1.f : ex2(m_run - m_new);
            const uint16_t* Vs = reinterpret_cast<const uint16_t*>(Vb + off_s(B, BITS));
            const uint16_t* Vz = reinterpret_cast<const uint16_t*>(Vb + off_z(B, BITS));
            const uint16_t* VR = reinterpret_cast<const uint16_t*>(Vb + off_R(B, BITS));
            float2 pR[NSB][4];   // tokens 8tq + 2k, + 1
            float psum = 0.f, pmax = 0.f;
#pragma unroll
            for (int sb = 0; sb < NSB; ++sb) {
                const uint4 r4 = *reinterpret_cast<const uint4*>(VR + 32 * sb + 8 * tq);
                const uint32_t rw[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float2 p;
                    p.x = (m_new == -INFINITY) ? 0.f : ex2(sc[sb][2 * k] - m_new);
                    p.y = (m_new == -INFINITY) ? 0.f : ex2(sc[sb][2 * k + 1] - m_new);
                    psum += p.x;
                    psum += p.y;
                    pR[sb][k] = __fmul2_rn(p, __half22float2(u32_as_h2(rw[k])));
                    pmax = fmaxf(pmax, fmaxf(pR[sb][k].x, pR[sb][k].y));
                }
            }
            l_part = l_part * alpha + psum;
            m_run = m_new;
            {
                const float2 al2 = make_float2(alpha, alpha);
#pragma unroll
                for (int g = 0; g < 4; ++g)
#pragma unroll
                    for (int f = 0; f < 4; ++f) O[g][f] = __fmul2_rn(O[g][f], al2);
            }
            pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, 1));
            pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, 2));
            float smax;
            if (B == 32) {
                const uint2 s2 = *reinterpret_cast<const uint2*>(Vs + 4 * lane);
                const __half2 m2 = __hmax2(u32_as_h2(s2.x), u32_as_h2(s2.y));
                smax = fmaxf(__low2float(m2), __high2float(m2));
            } else {
                const uint4 s4 = *reinterpret_cast<const uint4*>(Vs + 8 * lane);
                const __half2 m2 = __hmax2(__hmax2(u32_as_h2(s4.x), u32_as_h2(s4.y)),
                                           __hmax2(u32_as_h2(s4.z), u32_as_h2(s4.w)));
                smax = fmaxf(__low2float(m2), __high2float(m2));
            }
            smax = warp_max(smax);
            // power of two lam with p R lam <= 2^14 and p R s lam <= 2^12 (fp16 range
            // of P' and of its hi | lo halves); undone in the update of O
            float lam = 1.f;
            if (pmax > 0.f) {
                int k = 14 - ceil_log2(pmax);
                if (smax > 0.f) k = min(k, 12 - ceil_log2(pmax * smax));
                lam = exp2i(k);
            }
            // P'' = p R lam per token as fp16 hi | lo pairs (tokens 8tq + 2k, + 1 of
            // each sub-block): the A operand of the zero-point MMA, and the
            // factor of every group's P' = P'' s two-product
            uint32_t ph[NSB][4], pl[NSB][4];
#pragma unroll
            for (int sb = 0; sb < NSB; ++sb)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 v = __fmul2_rn(pR[sb][k], make_float2(lam, lam));
                    const __half2 hh = __float22half2_rn(v);
                    ph[sb][k] = h2_as_u32(hh);
                    pl[sb][k] = h2_as_u32(__float22half2_rn(__ffma2_rn(__half22float2(hh), make_float2(-1.f, -1.f), v)));
                }
            const float il4 = (1.0f / kA) / lam;
            const uint16_t* VC = reinterpret_cast<const uint16_t*>(Vb + off_C(B, BITS));

            // ---------------- zero-point sums by MMA: A = P'' (hi rows, lo rows), B columns
            // 0..3 = z of groups 0..3, 4..7 = s of groups 0..3, k = tokens
            float Dz[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int sb = 0; sb < NSB; ++sb) {
                const uint16_t* src = (gq < 4 ? Vz : Vs) + (gq & 3) * B + 32 * sb + 8 * tq;
                const uint4 zs4 = *reinterpret_cast<const uint4*>(src);
                mma16816(Dz, ph[sb][0], pl[sb][0], ph[sb][1], pl[sb][1], zs4.x, zs4.y);
                mma16816(Dz, ph[sb][2], pl[sb][2], ph[sb][3], pl[sb][3], zs4.z, zs4.w);
            }
            // this lane: columns 2tq, 2tq + 1 of vector gq (hi + lo rows): tq < 2 holds
            // Z of groups 2tq, 2tq + 1; zq[g] = Z_g * kA for the 4 lanes of vector gq
            float zq[4];
            {
                const float c0 = Dz[0] + Dz[2], c1 = Dz[1] + Dz[3];
                const float zA = c0 * kA, zB = c1 * kA;   // valid at tq < 2
                const int base = lane & ~3;
                zq[0] = __shfl_sync(kFull, zA, base);
                zq[1] = __shfl_sync(kFull, zB, base);
                zq[2] = __shfl_sync(kFull, zA, base + 1);
                zq[3] = __shfl_sync(kFull, zB, base + 1);
            }

            // ---------------- PV, one 32-channel group at a time
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                float Ob[4][4];   // n-tile f: channels 32g + 4n + f
#pragma unroll
                for (int f = 0; f < 4; ++f) Ob[f][0] = Ob[f][1] = Ob[f][2] = Ob[f][3] = 0.f;
#pragma unroll
                for (int sb = 0; sb < NSB; ++sb) {
                    // P' = P'' s_g as fp16 hi | lo (two-product), tokens 8tq + 2k, + 1
                    const uint4 s4 = *reinterpret_cast<const uint4*>(Vs + g * B + 32 * sb + 8 * tq);
                    const uint32_t sw[4] = {s4.x, s4.y, s4.z, s4.w};
                    uint32_t Ph[4], Pl[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const __half2 s2 = u32_as_h2(sw[k]), hp = u32_as_h2(ph[sb][k]);
                        const __half2 hi = __hmul2(hp, s2);
                        __half2 lo = __hfma2(hp, s2, __hneg2(hi));
                        lo = __hfma2(u32_as_h2(pl[sb][k]), s2, lo);
                        Ph[k] = h2_as_u32(hi);
                        Pl[k] = h2_as_u32(lo);
                    }
                    // this group's record words: 2g + f/2 at 2 bits (and the high-bit
                    // word 8 + g at 3 bits), 4g + f at 4 bits
                    const uint32_t* rec = reinterpret_cast<const uint32_t*>(Vb) + RW * (32 * sb + lane);
                    constexpr int NV = BITS == 4 ? 4 : 3;
                    uint32_t vw[NV], vw8[NV];
#pragma unroll
                    for (int k = 0; k < NV; ++k) {
                        vw[k] = BITS == 4 ? rec[4 * g + k] : (k < 2 ? rec[2 * g + k] : rec[8 + g]);
                        vw8[k] = vw[k] >> 8;
                    }
#pragma unroll
                    for (int kt = 0; kt < 2; ++kt) {
                        // A: P' of tokens 8tq + 4kt + {0, 1 | 2, 3}, hi row gq, lo row gq + 8
                        const uint32_t a0 = Ph[2 * kt], a1 = Pl[2 * kt], a2 = Ph[2 * kt + 1], a3 = Pl[2 * kt + 1];
#pragma unroll
                        for (int f = 0; f < 4; ++f) {
                            if (BITS == 2) {   // pair 4(d/4) + 2((d%4)/2) + f%2
                                const uint32_t w = vw[f >> 1];
                                const int j0 = 4 * kt + (f & 1), j1 = j0 + 2;
                                mma16816(Ob[f], a0, a1, a2, a3, code2_r(code2_view(w, code2_view_of(j0)), j0),
                                         code2_r(code2_view(w, code2_view_of(j1)), j1));
                            } else if (BITS == 3) {   // + the high bit at 8(f/2) + pair in word 8 + g
                                const uint32_t w = vw[f >> 1], w8 = vw8[f >> 1];
                                const int j0 = 4 * kt + (f & 1), j1 = j0 + 2, hb = 8 * (f >> 1);
                                mma16816(Ob[f], a0, a1, a2, a3, code3_s(w, w8, vw[2], j0, hb + j0),
                                         code3_s(w, w8, vw[2], j1, hb + j1));
                            } else {           // field d/2
                                mma16816(Ob[f], a0, a1, a2, a3, code4_s(vw[f], vw8[f], 2 * kt),
                                         code4_s(vw[f], vw8[f], 2 * kt + 1));
                            }
                        }
                    }
                }
                // O += C_c / (kA lam) * (Ob + Z * kA): lane holds channels 32g + 8tq + f (column 2tq)
                // and 32g + 8tq + 4 + f (column 2tq + 1)
                const uint4 c4 = *reinterpret_cast<const uint4*>(VC + 32 * g + 8 * tq);
                const float2 il42 = make_float2(il4, il4), zq2 = make_float2(zq[g], zq[g]);
#pragma unroll
                for (int f = 0; f < 4; ++f) {
                    // 2-bit: odd f columns hold odd fields at kA / 4
                    const float wf = (BITS == 2 && (f & 1)) ? 4.f : 1.f;
                    const float2 t = __ffma2_rn(__fadd2_rn(make_float2(Ob[f][0], Ob[f][1]), make_float2(Ob[f][2], Ob[f][3])),
                                                make_float2(wf, wf), zq2);
                    O[g][f] = __ffma2_rn(__fmul2_rn(pair_i4(c4, f), il42), t, O[g][f]);
                }
            }
        }
        // ---- retire the stage and refill it
        __syncwarp();
        okmask &= ~(1u << stage);
        if (j + S < nblk && issue(j + S, stage)) okmask |= 1u << stage;
        if (++stage == S) {
            stage = 0;
            phase ^= 1u;
        }
    }

    // ---- this vector's partial: (max, sum, rotated accumulators) in its row's slot
    float l = l_part;
    l += __shfl_xor_sync(kFull, l, 1);
    l += __shfl_xor_sync(kFull, l, 2);
    if (my_ok) {
        const int64_t vrow = (int64_t)b * chunk + my_row;
        float* base = a.partials + (((vrow * n_kv + h) * NS + split) * G + gq % G) * kPartialStride;
        if (tq == 0) {
            base[0] = m_run;
            base[1] = l;
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            float4* dst = reinterpret_cast<float4*>(base + 4 + 32 * g + 8 * tq);
            dst[0] = make_float4(O[g][0].x, O[g][1].x, O[g][2].x, O[g][3].x);
            dst[1] = make_float4(O[g][0].y, O[g][1].y, O[g][2].y, O[g][3].y);
        }
    }
}

// ---------------------------------------------------------------- host side
// Resident one-warp CTAs of the prefill kernel on `device` (cached per
// device and configuration).
static int prefill_grid_warps(int block_size, int bits, int device) {
    static int cache[2][3][64];
    const int bi = block_size == 32 ? 0 : 1, wi = bits - 2;
    if (device < 0 || device >= 64 || wi < 0 || wi > 2) return 0;
    if (cache[bi][wi][device] > 0) return cache[bi][wi][device];
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
    auto occ = [&](auto kernel, size_t smem) { return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 32, smem); };
    cudaError_t e;
    if (block_size == 32)
        e = bits == 4   ? occ(prefill_attn_kernel<32, 4, prefill_stages<32>()>, prefill_smem_bytes<32, 4>())
            : bits == 3 ? occ(prefill_attn_kernel<32, 3, prefill_stages<32>()>, prefill_smem_bytes<32, 3>())
                        : occ(prefill_attn_kernel<32, 2, prefill_stages<32>()>, prefill_smem_bytes<32, 2>());
    else
        e = bits == 4   ? occ(prefill_attn_kernel<64, 4, prefill_stages<64>()>, prefill_smem_bytes<64, 4>())
            : bits == 3 ? occ(prefill_attn_kernel<64, 3, prefill_stages<64>()>, prefill_smem_bytes<64, 3>())
                        : occ(prefill_attn_kernel<64, 2, prefill_stages<64>()>, prefill_smem_bytes<64, 2>());
    if (e != cudaSuccess || per_sm <= 0) return 0;
    cache[bi][wi][device] = sms * per_sm;
    return cache[bi][wi][device];
}

// Block splits per (sequence, kv head, row tile) unit, 1..16. With at most
// half a wave of units the split just fills one wave; with more it aims at
// about two and a half waves, where the last wave's remainder costs little
// (measured on the Llama-8B layer, 4096 cached tokens: chunks of 4, 16 and
// 64 rows ran fastest at 0.9, 2.45 and 2.45 waves).
int64_t prefill_splits(const kvarn_config& cfg, int64_t batch, int64_t chunk, int device) {
    const int G = cfg.n_q_heads / cfg.n_kv_heads, P = kPrefillVecs / G;
    const int64_t units = batch * cfg.n_kv_heads * ((chunk + P - 1) / P);
    const int64_t R = prefill_grid_warps(cfg.block_size, cfg.bits, device);
    if (units <= 0 || R <= 0) return 1;
    const int64_t ns = 2 * units <= R ? R / units : (5 * R + units) / (2 * units);
    return ns < 1 ? 1 : (ns > 16 ? 16 : ns);
}

cudaError_t launch_prefill_attn(const kvarn_config& cfg, const void* q, int q_dtype, const void* pool,
                                int64_t n_pool_blocks, int64_t block_bytes, const void* staging,
                                const int32_t* block_table, int max_blocks, const int32_t* seq_lens, int batch,
                                int chunk, float* out, void* workspace, int64_t max_slots, int64_t splits,
                                cudaStream_t st) {
    AttnArgs a = {};
    a.q = q;
    a.q_dtype = q_dtype;
    a.pool = (const uint8_t*)pool;
    a.staging = (const uint16_t*)staging;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.err = (uint32_t*)workspace;
    a.partials = (float*)((uint8_t*)workspace + kWsHeader);
    a.out = out;
    a.n_pool_blocks = n_pool_blocks;
    a.block_bytes = block_bytes;
    a.max_blocks = max_blocks;
    a.batch = batch;   // real sequences here; the merge below runs over the batch * chunk rows
    a.n_q = cfg.n_q_heads;
    a.n_kv = cfg.n_kv_heads;
    a.G = cfg.n_q_heads / cfg.n_kv_heads;
    a.nw = 0;
    a.chunk = chunk;
    a.sm_scale = cfg.sm_scale;
    a.flags = cfg.flags;
    for (int i = 0; i < 4; ++i) a.sb[i] = cfg.sign_bits[i];
    const int P = kPrefillVecs / a.G;
    const int64_t tiles = (chunk + P - 1) / P;
    const int64_t units = (int64_t)batch * a.n_kv * tiles;
    // split each unit's blocks (prefill_splits); the partials of a row must fit
    // the workspace slots and one merge round trip (16)
    const int64_t rows = (int64_t)batch * chunk * a.n_kv;
    int64_t ns = splits;
    ns = std::min<int64_t>(ns, std::min<int64_t>(16, rows > 0 ? max_slots / rows : 1));
    a.single = (int)std::max<int64_t>(ns, 1);
    const int64_t warps = units * a.single;
    if (warps > 0x7fffffff) return cudaErrorInvalidValue;
    cudaError_t e;
    auto go = [&](auto kernel, size_t smem) { return launch_pdl(kernel, (unsigned)warps, 32, smem, st, a); };
    if (cfg.block_size == 32) {
        e = cfg.bits == 4   ? go(prefill_attn_kernel<32, 4, prefill_stages<32>()>, prefill_smem_bytes<32, 4>())
            : cfg.bits == 3 ? go(prefill_attn_kernel<32, 3, prefill_stages<32>()>, prefill_smem_bytes<32, 3>())
                            : go(prefill_attn_kernel<32, 2, prefill_stages<32>()>, prefill_smem_bytes<32, 2>());
    } else {
        e = cfg.bits == 4   ? go(prefill_attn_kernel<64, 4, prefill_stages<64>()>, prefill_smem_bytes<64, 4>())
            : cfg.bits == 3 ? go(prefill_attn_kernel<64, 3, prefill_stages<64>()>, prefill_smem_bytes<64, 3>())
                            : go(prefill_attn_kernel<64, 2, prefill_stages<64>()>, prefill_smem_bytes<64, 2>());
    }
    if (e != cudaSuccess) return e;
    a.batch = batch * chunk;
    const unsigned mgrid = (unsigned)(((int64_t)a.batch * a.n_q + 3) / 4);
    return cfg.block_size == 32 ? launch_pdl(merge_kernel<32, true>, mgrid, 128, 0, st, a)
                                : launch_pdl(merge_kernel<64, true>, mgrid, 128, 0, st, a);
}

}  // namespace kvarn
