// attention.cu -- split-K decode attention over the KVarN 2-bit paged cache
// (sm_103a), and the merge kernel that finishes it.
//
// Method: "KVarN：方差归一化让 2-bit KV 缓存扛住长链推理", section 三 3.1: the
// query is multiplied by the same randomised Hadamard matrix as K and V, so
// q.k is unchanged; section 三 3.2: the stored scales are applied again when
// the cache is read. Because V is stored rotated, the attention output is
// rotated back once, after the merge.
//
// Work split. The (sequence, kv head) units are laid end to end, block by
// block; the grid is the GPU's resident warps (one warp per CTA), and warp w
// takes blocks [w*W/nw, (w+1)*W/nw) of the W blocks in total, so ragged
// lengths stay balanced. A warp writes one partial (running max, sum and 128
// rotated accumulators per query head) for every unit its range touches, in
// slot unit + w; the merge kernel finds the warps of a unit by the same
// arithmetic.
//
// Per warp: lane 0 streams each block's K and V head-blocks into a ring of
// shared-memory stages with 1-D bulk copies (cp.async.bulk) counted on
// mbarriers; all lanes wait with a bounded try_wait. Each lane reads one
// 32-byte code record per 32 tokens and turns every pair of 2-bit codes into
// an fp16x2 tensor-core operand a = 1 + code/4 (exact) with one shift and
// one LOP3. The contractions run on mma.sync m16n8k16 (f16 in, f32
// accumulate); since code*s + z = 4s*a + (z - 4s):
//   QK: D[token][col] = sum_c a[t][c] * q'[c][col], per 32-channel group,
//       col = (query head, hi|lo) with q' = q_rot*C split into two fp16s, so
//       the scores keep fp32 accuracy; then
//       score[t][h] = R_t*(sum_g 4 s_tg*acc_g + (z_tg - 4 s_tg)*Q'_g[h]),
//       Q'_g = sum_{c in g} q'_c
//   PV: O^T[c][col] = sum_t a[t][c] * P'[t][col],  P' = p_t*R_t*s_tg*lam (hi|lo),
//       plus the zero term sum_t p_t R_t lam (z_tg - 4 s_tg) in fp32; the
//       running accumulator gets C_c/lam*(4 O_blk + zero term) per block.
// Operand order inside each MMA (which token is row r, which channel is
// k-slot j) is chosen so that the packed record order gives every lane its
// operands directly; the writer packs codes in that order.
#include "attn_common.cuh"

namespace kvarn {

// ---------------------------------------------------------------- the split-K kernel
template <int B, int S>
__global__ void __launch_bounds__(32) decode_attn_2bit_kernel(AttnArgs a) {
    constexpr int HB = head_block_bytes(B);
    constexpr int NSB = B / 32;
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t* stages = smem;                                              // S x (K, V)
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * 2 * HB);     // S mbarriers
    float* qsm = reinterpret_cast<float*>(smem + S * 2 * HB + 64);       // [4][128]
    uint16_t* pex = reinterpret_cast<uint16_t*>(qsm + 4 * kD);           // [2][4][32]: hi, lo

    const int lane = threadIdx.x;
    const int gq = lane >> 2, tq = lane & 3;   // mma groupID, thread-in-group
    const int w = blockIdx.x;

    const SplitArgs sp{a.seq_lens, a.batch, a.n_kv, a.max_blocks, B, 0};
    Cursor cc;
    cc.b = cc.h = cc.j = 0;
    const int64_t W = split_locate(sp, 0, lane, cc.b, cc.h, cc.j);
    const int64_t s_beg = (int64_t)w * W / a.nw, s_end = (int64_t)(w + 1) * W / a.nw;
    if (s_beg >= s_end) return;
    split_locate(sp, s_beg, lane, cc.b, cc.h, cc.j);
    cc.nb = split_nblocks(sp, cc.b);
    Cursor ic = cc;   // issue cursor

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    // block-table chunk cache for the issue cursor
    int bt_b = -1, bt_j0 = 0, bt_val = 0;
    auto issue = [&](int64_t x, int stage) {
        if (ic.b != bt_b || ic.j < bt_j0 || ic.j >= bt_j0 + 32) {
            bt_b = ic.b;
            bt_j0 = ic.j;
            const int jj = bt_j0 + lane;
            bt_val = (jj < a.max_blocks) ? a.block_table[(int64_t)bt_b * a.max_blocks + jj] : -1;
        }
        int64_t phys = __shfl_sync(kFull, bt_val, ic.j - bt_j0);
        const bool ok = phys >= 0 && phys < a.n_pool_blocks;
        if (!ok) phys = 0;   // read a valid block, result discarded below
        if (lane == 0) {
            const uint8_t* src = a.pool + phys * a.block_bytes + (int64_t)(2 * ic.h) * HB;
            mbar_arrive_expect_tx(&bars[stage], 2 * HB);
            bulk_g2s(stages + stage * 2 * HB, src, 2 * HB, &bars[stage]);
        }
        split_advance(sp, ic);
        return ok;
    };
    uint32_t okmask = 0;   // bit s: the block in stage s had a valid id
    {
        int64_t x = s_beg;
        for (int s = 0; s < S && x < s_end; ++s, ++x)
            if (issue(x, s)) okmask |= 1u << s;
    }

    // per-unit state
    uint32_t Qh[16], Qlm[16], Qhm[16];
    float qsQ[16];
    float kmul = 0.f;
    float m_run = -INFINITY, l_part = 0.f;
    float O[8][4];
    const float sgn4[4] = {sign_of(a.sb, 4 * lane), sign_of(a.sb, 4 * lane + 1),
                           sign_of(a.sb, 4 * lane + 2), sign_of(a.sb, 4 * lane + 3)};
    const bool head_ok = tq < a.G;          // this lane's score/accumulator head
    const int hbq = gq >> 1, part = gq & 1;  // this lane's B-fragment column: (head, hi|lo)
    const bool bcol_ok = hbq < a.G;

    auto unit_setup = [&]() {
        __syncwarp();
        for (int j = 0; j < a.G; ++j) {
            float v[4];
            load_q4(a, (int64_t)cc.b * a.n_q + (int64_t)cc.h * a.G + j, lane, v);
#pragma unroll
            for (int k = 0; k < 4; ++k) v[k] *= sgn4[k];
            fwht128(v, lane);
            float amax = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                v[k] *= kInvSqrtD;
                amax = fmaxf(amax, fabsf(v[k]));
            }
            amax = warp_max(amax);
            const int e = (amax > 0.f && isfinite(amax)) ? ceil_log2(amax) : 0;
            const float sc = exp2i(-e);
            *reinterpret_cast<float4*>(&qsm[j * kD + 4 * lane]) =
                make_float4(v[0] * sc, v[1] * sc, v[2] * sc, v[3] * sc);
            if (j == tq) kmul = exp2i(e) * a.sm_scale * kLog2e;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int c0 = 32 * (i >> 2) + 8 * tq + 2 * (i & 3);
            uint32_t hv = 0, lv = 0;
            if (bcol_ok) {
                const float v0 = qsm[hbq * kD + c0], v1 = qsm[hbq * kD + c0 + 1];
                const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
                hv = h2_as_u32(__halves2half2(h0, h1));
                lv = pack_h2(v0 - __half2float(h0), v1 - __half2float(h1));
            }
            Qh[i] = hv;
            Qlm[i] = part ? lv : 0u;
            Qhm[i] = part ? hv : 0u;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k)
            qsQ[k] = head_ok ? qsm[tq * kD + 32 * (gq >> 1) + 16 * (gq & 1) + k] : 0.f;
        if (!head_ok) kmul = 0.f;
        m_run = -INFINITY;
        l_part = 0.f;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int r = 0; r < 4; ++r) O[mt][r] = 0.f;
    };

    auto unit_flush = [&]() {
        float l = l_part;
        l += __shfl_xor_sync(kFull, l, 4);
        l += __shfl_xor_sync(kFull, l, 8);
        l += __shfl_xor_sync(kFull, l, 16);
        if (head_ok) {
            const int64_t slot = (int64_t)cc.b * a.n_kv + cc.h + w;
            float* base = a.partials + (slot * a.G + tq) * kPartialStride;
            if (gq == 0) {
                base[0] = m_run;
                base[1] = l;
            }
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                // rows gq / gq+8 of m-tiles 2g, 2g+1 -> channels 32g + 4gq + {0,1,2,3}
                float4 o;
                o.x = O[2 * g][0] + O[2 * g][1];
                o.y = O[2 * g][2] + O[2 * g][3];
                o.z = O[2 * g + 1][0] + O[2 * g + 1][1];
                o.w = O[2 * g + 1][2] + O[2 * g + 1][3];
                *reinterpret_cast<float4*>(base + 4 + 32 * g + 4 * gq) = o;
            }
        }
    };

    unit_setup();
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t x = s_beg; x < s_end; ++x) {
        if (!mbar_wait_bounded(&bars[stage], phase, kWaitLimit)) {
            if (lane == 0) raise_error(a.err, KVARN_DEVERR_WAIT_TIMEOUT);
            // let every copy still in flight into this CTA's shared memory land
            // (again with a limit) before the CTA exits
            uint32_t ph = phase;
            for (int k = 0, st2 = stage; k < S && x + k < s_end; ++k) {
                mbar_wait_bounded(&bars[st2], ph, kWaitLimit);
                if (++st2 == S) { st2 = 0; ph ^= 1u; }
            }
            return;
        }
        const uint8_t* Kb = stages + stage * 2 * HB;
        const uint8_t* Vb = Kb + HB;
        const bool valid = (okmask >> stage) & 1u;
        if (!valid && lane == 0) raise_error(a.err, KVARN_DEVERR_BLOCK_ID);

        if (valid) {
            // ---- QK B operand for this block: q' = q_rot * C, split hi|lo
            uint32_t bq[16];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const uint4 c4 = *reinterpret_cast<const uint4*>(Kb + off_C(B) + 2 * (32 * g + 8 * tq));
                const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const int i = 4 * g + e2;
                    const __half2 C2 = u32_as_h2(cw[e2]);
                    const __half2 mhi = __hmul2(u32_as_h2(Qhm[i]), C2);
                    __half2 r = __hfma2(u32_as_h2(Qh[i]), C2, __hneg2(mhi));
                    r = __hfma2(u32_as_h2(Qlm[i]), C2, r);
                    bq[i] = h2_as_u32(r);
                }
            }
            // ---- Q'_g for this lane's head: sum over the group of q_rot * C (fp32)
            float Qp[4];
            {
                const uint4* cp = reinterpret_cast<const uint4*>(Kb + off_C(B) + 2 * (32 * (gq >> 1) + 16 * (gq & 1)));
                float qp = 0.f;
#pragma unroll
                for (int v4 = 0; v4 < 2; ++v4) {
                    const uint4 c4 = cp[v4];
                    const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) {
                        const float2 cf = __half22float2(u32_as_h2(cw[e2]));
                        qp = fmaf(qsQ[8 * v4 + 2 * e2], cf.x, qp);
                        qp = fmaf(qsQ[8 * v4 + 2 * e2 + 1], cf.y, qp);
                    }
                }
                qp += __shfl_xor_sync(kFull, qp, 4);
#pragma unroll
                for (int g = 0; g < 4; ++g) Qp[g] = __shfl_sync(kFull, qp, 8 * g + tq);
            }
            const uint16_t* Ks = reinterpret_cast<const uint16_t*>(Kb + off_s(B));
            const uint16_t* Kz = reinterpret_cast<const uint16_t*>(Kb + off_z(B));
            const uint16_t* KR = reinterpret_cast<const uint16_t*>(Kb + off_R(B));
            const uint16_t* Vs = reinterpret_cast<const uint16_t*>(Vb + off_s(B));
            const uint16_t* Vz = reinterpret_cast<const uint16_t*>(Vb + off_z(B));
            const uint16_t* VR = reinterpret_cast<const uint16_t*>(Vb + off_R(B));

#pragma unroll
            for (int sb = 0; sb < NSB; ++sb) {
                // ---------------- QK
                uint32_t kw[8];
                {
                    const uint4* rec = reinterpret_cast<const uint4*>(Kb) + 2 * (32 * sb + lane);
                    const uint4 r0 = rec[0], r1 = rec[1];
                    kw[0] = r0.x; kw[1] = r0.y; kw[2] = r0.z; kw[3] = r0.w;
                    kw[4] = r1.x; kw[5] = r1.y; kw[6] = r1.z; kw[7] = r1.w;
                }
                float acc[4][2][4];
#pragma unroll
                for (int g = 0; g < 4; ++g)
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                        for (int r = 0; r < 4; ++r) acc[g][mt][r] = 0.f;
#pragma unroll
                for (int g = 0; g < 4; ++g)
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const uint32_t b0 = bq[4 * g + 2 * kk], b1 = bq[4 * g + 2 * kk + 1];
                        const int j = 4 * (g & 1) + 2 * kk;
#pragma unroll
                        for (int mt = 0; mt < 2; ++mt) {
                            const uint32_t w0 = kw[2 * (2 * mt) + (g >> 1)];
                            const uint32_t w1 = kw[2 * (2 * mt + 1) + (g >> 1)];
                            mma16816(acc[g][mt], code_pair(w0, j), code_pair(w1, j),
                                     code_pair(w0, j + 1), code_pair(w1, j + 1), b0, b1);
                        }
                    }
                // scores of tokens 32sb + 4gq + i, head tq
                const int t0 = 32 * sb + 4 * gq;
                float sc[4];
                {
                    const uint2 Rr = *reinterpret_cast<const uint2*>(KR + t0);
                    const float2 R01 = __half22float2(u32_as_h2(Rr.x)), R23 = __half22float2(u32_as_h2(Rr.y));
                    const float Rv[4] = {R01.x, R01.y, R23.x, R23.y};
                    float sv[4][4], zv[4][4];   // [group][token]
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const uint2 s2 = *reinterpret_cast<const uint2*>(Ks + g * B + t0);
                        const uint2 z2 = *reinterpret_cast<const uint2*>(Kz + g * B + t0);
                        const float2 s01 = __half22float2(u32_as_h2(s2.x)), s23 = __half22float2(u32_as_h2(s2.y));
                        const float2 z01 = __half22float2(u32_as_h2(z2.x)), z23 = __half22float2(u32_as_h2(z2.y));
                        sv[g][0] = s01.x; sv[g][1] = s01.y; sv[g][2] = s23.x; sv[g][3] = s23.y;
                        zv[g][0] = z01.x; zv[g][1] = z01.y; zv[g][2] = z23.x; zv[g][3] = z23.y;
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int mt = i >> 1, rh = i & 1;
                        float s = 0.f;
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            const float ag = acc[g][mt][2 * rh] + acc[g][mt][2 * rh + 1];
                            const float s4 = 4.0f * sv[g][i];
                            s = fmaf(s4, ag, s);
                            s = fmaf(zv[g][i] - s4, Qp[g], s);
                        }
                        sc[i] = s * Rv[i] * kmul;
                    }
                }
                // ---------------- online softmax (head tq, 32 tokens over 8 lanes)
                float bm = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
                bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 4));
                bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 8));
                bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
                const float m_new = fmaxf(m_run, bm);
                const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
                float pv[4], psum = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    pv[i] = (m_new == -INFINITY) ? 0.f : exp2f(sc[i] - m_new);
                    psum += pv[i];
                }
                l_part = l_part * alpha + psum;
                m_run = m_new;
                if (__any_sync(kFull, alpha != 1.f)) {
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                        for (int r = 0; r < 4; ++r) O[mt][r] *= alpha;
                }
                // ---------------- P' = p * R_v * s_v, normalised per (head, 32 tokens)
                float pR[4];
                {
                    const uint2 Rr = *reinterpret_cast<const uint2*>(VR + t0);
                    const float2 R01 = __half22float2(u32_as_h2(Rr.x)), R23 = __half22float2(u32_as_h2(Rr.y));
                    pR[0] = pv[0] * R01.x; pR[1] = pv[1] * R01.y; pR[2] = pv[2] * R23.x; pR[3] = pv[3] * R23.y;
                }
                // largest step of this V sub-block (all groups)
                float smax;
                {
                    const uint2 s2 = *reinterpret_cast<const uint2*>(Vs + (lane >> 3) * B + 32 * sb + 4 * (lane & 7));
                    const __half2 m2 = __hmax2(u32_as_h2(s2.x), u32_as_h2(s2.y));
                    smax = fmaxf(__low2float(m2), __high2float(m2));
                    smax = warp_max(smax);
                }
                float pmax = fmaxf(fmaxf(pR[0], pR[1]), fmaxf(pR[2], pR[3]));
                pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, 4));
                pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, 8));
                pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, 16));
                // power-of-two scale so that p*R <= 2^14 and p*R*s <= 2^12 (fp16
                // range for P' and its hi|lo split); undone in the update of O
                float lam = 1.f;
                if (pmax > 0.f) {
                    int k = 14 - ceil_log2(pmax);
                    if (smax > 0.f) k = min(k, 12 - ceil_log2(pmax * smax));
                    lam = exp2i(k);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) pR[i] *= lam;
                {
                    uint16_t* ph = pex + tq * 32 + 4 * gq;            // [hi][head][token]
                    uint16_t* pl = pex + 128 + tq * 32 + 4 * gq;      // [lo][head][token]
                    float hi[4], lo[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        hi[i] = __half2float(__float2half_rn(pR[i]));
                        lo[i] = pR[i] - hi[i];
                    }
                    *reinterpret_cast<uint2*>(ph) = make_uint2(pack_h2(hi[0], hi[1]), pack_h2(hi[2], hi[3]));
                    *reinterpret_cast<uint2*>(pl) = make_uint2(pack_h2(lo[0], lo[1]), pack_h2(lo[2], lo[3]));
                }
                // zero term per group for head tq over this sub-block (fp32):
                // sum_t p R lam (z - 4 s)
                float zs[4];
                {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const uint2 z2 = *reinterpret_cast<const uint2*>(Vz + g * B + t0);
                        const uint2 s2 = *reinterpret_cast<const uint2*>(Vs + g * B + t0);
                        const float2 z01 = __half22float2(u32_as_h2(z2.x)), z23 = __half22float2(u32_as_h2(z2.y));
                        const float2 s01 = __half22float2(u32_as_h2(s2.x)), s23 = __half22float2(u32_as_h2(s2.y));
                        float zz = pR[0] * fmaf(-4.0f, s01.x, z01.x);
                        zz = fmaf(pR[1], fmaf(-4.0f, s01.y, z01.y), zz);
                        zz = fmaf(pR[2], fmaf(-4.0f, s23.x, z23.x), zz);
                        zz = fmaf(pR[3], fmaf(-4.0f, s23.y, z23.y), zz);
                        zz += __shfl_xor_sync(kFull, zz, 4);
                        zz += __shfl_xor_sync(kFull, zz, 8);
                        zz += __shfl_xor_sync(kFull, zz, 16);
                        zs[g] = zz;
                    }
                }
                __syncwarp();
                // ---------------- PV B operand: tokens 8tq..8tq+7, column (hbq, part)
                uint32_t bv[4][4];   // [group][token pair]
                {
                    uint4 phv = make_uint4(0, 0, 0, 0), plv = make_uint4(0, 0, 0, 0);
                    if (bcol_ok) {
                        phv = *reinterpret_cast<const uint4*>(pex + hbq * 32 + 8 * tq);
                        plv = *reinterpret_cast<const uint4*>(pex + 128 + hbq * 32 + 8 * tq);
                    }
                    const uint32_t ph[4] = {phv.x, phv.y, phv.z, phv.w};
                    const uint32_t pl[4] = {plv.x, plv.y, plv.z, plv.w};
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const uint4 s4 = *reinterpret_cast<const uint4*>(Vs + g * B + 32 * sb + 8 * tq);
                        const uint32_t sw[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const __half2 s2 = u32_as_h2(sw[k]);
                            const __half2 hp = u32_as_h2(ph[k]);
                            const __half2 mhi = __hmul2(hp, s2);
                            if (part == 0) {
                                bv[g][k] = h2_as_u32(mhi);
                            } else {
                                __half2 r = __hfma2(hp, s2, __hneg2(mhi));
                                r = __hfma2(u32_as_h2(pl[k]), s2, r);
                                bv[g][k] = h2_as_u32(r);
                            }
                        }
                    }
                }
                __syncwarp();
                // ---------------- PV: O_blk^T[c][col] over this sub-block's 32 tokens
                uint32_t vw[8];
                {
                    const uint4* rec = reinterpret_cast<const uint4*>(Vb) + 2 * (32 * sb + lane);
                    const uint4 r0 = rec[0], r1 = rec[1];
                    vw[0] = r0.x; vw[1] = r0.y; vw[2] = r0.z; vw[3] = r0.w;
                    vw[4] = r1.x; vw[5] = r1.y; vw[6] = r1.z; vw[7] = r1.w;
                }
                float Ob[8][4];
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
                    for (int r = 0; r < 4; ++r) Ob[mt][r] = 0.f;
                    const int g = mt >> 1, m = mt & 1;
                    const uint32_t wd = vw[2 * g + m];
#pragma unroll
                    for (int kt = 0; kt < 2; ++kt) {
                        mma16816(Ob[mt], code_pair(wd, 4 * kt + 0), code_pair(wd, 4 * kt + 1),
                                 code_pair(wd, 4 * kt + 2), code_pair(wd, 4 * kt + 3),
                                 bv[g][2 * kt], bv[g][2 * kt + 1]);
                    }
                }
                // ---------------- O += C_c / lam * (4 O_blk + zs_g)
                {
                    const float il = 1.f / lam;
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const uint2 c2 = *reinterpret_cast<const uint2*>(Vb + off_C(B) + 2 * (32 * g + 4 * gq));
                        const float2 c01 = __half22float2(u32_as_h2(c2.x)), c23 = __half22float2(u32_as_h2(c2.y));
                        const float cf[4] = {c01.x, c01.y, c23.x, c23.y};   // channels 32g+4gq+{0..3}
#pragma unroll
                        for (int m = 0; m < 2; ++m) {
                            const int mt = 2 * g + m;
#pragma unroll
                            for (int rh = 0; rh < 2; ++rh) {
                                const float cs = cf[2 * m + rh] * il;
                                O[mt][2 * rh] = fmaf(cs, fmaf(Ob[mt][2 * rh], 4.0f, zs[g]), O[mt][2 * rh]);
                                O[mt][2 * rh + 1] = fmaf(cs * 4.0f, Ob[mt][2 * rh + 1], O[mt][2 * rh + 1]);
                            }
                        }
                    }
                }
            }
        }
        // ---- retire the stage and refill it
        __syncwarp();
        const int64_t xn = x + S;
        okmask &= ~(1u << stage);
        if (xn < s_end && issue(xn, stage)) okmask |= 1u << stage;
        if (++stage == S) {
            stage = 0;
            phase ^= 1u;
        }
        // ---- unit boundary
        const int pb = cc.b, ph_ = cc.h;
        split_advance(sp, cc);
        if (x + 1 == s_end || cc.b != pb || cc.h != ph_) {
            Cursor done = cc;
            cc.b = pb;
            cc.h = ph_;
            unit_flush();
            cc = done;
            if (x + 1 < s_end) unit_setup();
        }
    }
}

// ---------------------------------------------------------------- host side
template <int B>
constexpr int stages_for() { return B == 32 ? 4 : 3; }

template <int B>
size_t attn_smem_bytes() {
    return (size_t)stages_for<B>() * 2 * head_block_bytes(B) + 64 + 4 * kD * sizeof(float) + 256 * sizeof(uint16_t);
}

// Resident warps of the split-K kernel on `device` (cached per device).
int attn_grid_warps(int block_size, int device) {
    static int cache[2][64];
    const int bi = block_size == 32 ? 0 : 1;
    if (device < 0 || device >= 64) return 0;
    if (cache[bi][device] > 0) return cache[bi][device];
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
    cudaError_t e;
    if (block_size == 32)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_attn_2bit_kernel<32, stages_for<32>()>, 32,
                                                          attn_smem_bytes<32>());
    else
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_attn_2bit_kernel<64, stages_for<64>()>, 32,
                                                          attn_smem_bytes<64>());
    if (e != cudaSuccess || per_sm <= 0) return 0;
    cache[bi][device] = sms * per_sm;
    return cache[bi][device];
}

cudaError_t launch_decode_attn(const kvarn_config& cfg, const void* q, int q_dtype, const void* pool,
                               int64_t n_pool_blocks, int64_t block_bytes, const void* staging,
                               const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                               int batch, float* out, void* workspace, int nw, cudaStream_t st) {
    AttnArgs a;
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
    a.batch = batch;
    a.n_q = cfg.n_q_heads;
    a.n_kv = cfg.n_kv_heads;
    a.G = cfg.n_q_heads / cfg.n_kv_heads;
    a.nw = nw;
    a.sm_scale = cfg.sm_scale;
    for (int i = 0; i < 4; ++i) a.sb[i] = cfg.sign_bits[i];
    const unsigned mgrid = (unsigned)(((int64_t)batch * a.n_q + 3) / 4);
    if (cfg.block_size == 32) {
        decode_attn_2bit_kernel<32, stages_for<32>()><<<nw, 32, attn_smem_bytes<32>(), st>>>(a);
        merge_kernel<32, true><<<mgrid, 128, 0, st>>>(a);
    } else {
        decode_attn_2bit_kernel<64, stages_for<64>()><<<nw, 32, attn_smem_bytes<64>(), st>>>(a);
        merge_kernel<64, true><<<mgrid, 128, 0, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace kvarn
