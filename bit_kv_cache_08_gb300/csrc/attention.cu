// attention.cu -- split-K decode attention over the KVarN 2-bit paged cache
// (sm_103a); the merge kernel that finishes it is in attn_common.cuh.
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
// slot unit + w, and records in the workspace's unit map whether it took the
// unit's first or last block, so that the merge kernel reads the unit's
// consecutive slots without redoing the split arithmetic.
//
// Per warp: lane 0 streams each block's K and V head-blocks into a ring of
// shared-memory stages with 1-D bulk copies (cp.async.bulk) counted on
// mbarriers; all lanes wait with a bounded try_wait. Each lane reads one
// 32-byte code record per 32 tokens and turns every pair of 2-bit codes into
// an fp16x2 tensor-core operand without a multiply: a shifted or byte-swapped
// view of the record word holds the pair's field at bits 8..9 (even fields:
// an fp16 subnormal a = code * 2^-16) or 6..7 (odd fields: code * 2^-18) of
// each half, and one LOP3 keeps it; the tensor cores keep full precision for
// subnormal operands at those bit positions. The factor 4 between the two is
// put into q' for QK (odd k-slots x 4) and into the output rows for PV.
// Below, "a" is the operand at the even fields' scale (code * 2^-16 =
// code * kA). Everything runs on mma.sync m16n8k16 (f16 in,
// f32 accumulate) with fp32 epilogues; code * s + z = s a / kA + z.
//   q'  = q_rot * C per block, as two fp16 halves (hi | lo) so the tensor
//         cores keep fp32 accuracy; q_rot is scaled to 2^12 per unit and C by
//         a power of two per block so both halves stay normal fp16 (fp16
//         subnormal operands lose precision on the tensor cores).
//   Q'_g = sum_{c in g} q'_c * kA      (MMA with code-1 A operands)
//   QK:  acc_g[t][h] = sum_{c in g} a[t][c] q'[c][h]  (one accumulator per
//        32-channel group, hi and lo columns), then
//        score[t][h] = R_t / kA sum_g (s_tg acc_g + z_tg Q'_g)
//   softmax over the block (running max and sum per head, log2 domain)
//   PV:  P'[t][h,g] = p_t R_t s_tg lam (hi | lo), lam a power of two per
//        (head, block) keeping P' inside fp16;
//        Ob[c][h] = sum_t a[t][c] P'[t][h, g(c)]
//        zs[h][g] = sum_t p_t R_t lam z_tg  (MMA with p as A, z | s as B)
//        O[c][h] += C_c / (kA lam) * (Ob[c][h] + zs[h][g(c)] * kA)  once per block.
// Operand order inside each MMA (which token is row r, which channel is
// k-slot j) is chosen so that the packed record order gives every lane its
// operands directly; the writer packs codes in that order.
// 3- and 4-bit codes (BITS = 3, 4) take the same path with a lane record of
// 48 or 64 bytes, but their operands are a = code * 2^-9 for every field
// (kA = 2^-9): a field masked in place is scaled to that value by one HMUL2
// (a 3-bit field is first joined from the 2-bit word and the 1-bit plane by
// one shift and two LOP3s). The kernel's name keeps the method's width.
// q's hi | lo halves are read from shared memory per block rather than held
// in 32 registers per lane.
#include "attn_common.cuh"

namespace kvarn {

// 2^x by the MUFU instruction (relative error ~2^-22; results below 2^-126,
// i.e. softmax weights that cannot move an fp32 sum, flush to 0)
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- the split-K kernel
// Shared memory for q: the fp16 planes hi, -hi, lo ([4][128] each, written
// over the fp32 copy of q) and a zero line, at byte offsets 0, 1088, 2176 and
// 3264 (in fp16 elements below): a lane reading the hi | lo column of the B
// operand and its neighbour reading the other part of the same head then hit
// opposite halves of the banks (offsets 64 bytes apart mod 128). The 192
// bytes this adds keep a B = 64 CTA at 18 432 bytes, 12 per SM. Keeping q in
// shared memory rather than in 32 registers per lane lets B = 32 run 16 warps
// per SM (128 registers) instead of 12.
constexpr int kQHi = 0, kQNegHi = 544, kQLo = 1088, kQZero = 1632;
__host__ __device__ constexpr int attn_q_bytes(int) { return 2 * kQZero + 2 * kD; }
// P'' exchange rows [hi|lo][4 heads][B] fp16: row r holds its tokens rotated
// by pex_rot(r) elements (mod B), so that the four heads' rows written by one
// store instruction fall on different banks without padding
__host__ __device__ constexpr int pex_rot(int B, int r) { return B == 64 ? 16 * r : 16 * (r >> 1); }

template <int B, int BITS, int S>
__device__ __forceinline__ void decode_attn_2bit_body(const AttnArgs& a) {
    static_assert(BITS >= 2 && BITS <= 4, "2-, 3- or 4-bit codes");
    wait_prior_grids();
    constexpr int HB = head_block_bytes(B, BITS);
    constexpr int RW = 4 * BITS;             // 32-bit words per lane record
    constexpr int NSB = B / 32;
    // kA: the operand scale of a code (2-bit: even fields' raw subnormals)
    constexpr float kA = BITS == 2 ? kRawScale : kCodeScale;
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t* stages = smem;                                              // S x (K, V)
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * 2 * HB);     // S mbarriers
    float* qsm = reinterpret_cast<float*>(smem + S * 2 * HB + 64);       // [4][128] fp32 q, then the fp16 planes below
    uint16_t* pex = reinterpret_cast<uint16_t*>(smem + S * 2 * HB + 64 + attn_q_bytes(B));   // [hi|lo][4 heads][B]

    const int lane = threadIdx.x;
    const int gq = lane >> 2, tq = lane & 3;   // mma groupID, thread-in-group
    const int w = blockIdx.x;

    // scalar copies of the arguments (the lambdas below must not take the
    // address of the kernel parameter block)
    const uint8_t* __restrict__ pool = a.pool;
    const int32_t* __restrict__ btab = a.block_table;
    const int max_blocks = a.max_blocks, G = a.G, n_q = a.n_q, n_kv = a.n_kv, q_dtype = a.q_dtype;
    const int64_t n_pool_blocks = a.n_pool_blocks, block_bytes = a.block_bytes;
    const void* qptr = a.q;
    float* partials = a.partials;
    int32_t* umap = a.unit_map;
    uint32_t* err = a.err;
    const float sm_scale = a.sm_scale;
    const uint32_t sb0 = a.sb[0], sb1 = a.sb[1], sb2 = a.sb[2], sb3 = a.sb[3];
    const bool rotate_q = !(a.flags & KVARN_FLAG_NO_ROTATION);

    const SplitArgs sp{a.seq_lens, a.batch, n_kv, max_blocks, B, 0, 1};
    Cursor cc;
    cc.b = cc.h = cc.j = 0;
    const int64_t W = split_locate(sp, 0, lane, cc.b, cc.h, cc.j);
    const int64_t nwe = split_active_warps(W, a.nw, (int64_t)a.batch * n_kv, kSplitRatio2bit * B);
    if (w >= nwe) return;
    const int64_t s_beg = (int64_t)w * W / nwe, s_end = (int64_t)(w + 1) * W / nwe;
    if (s_beg >= s_end) return;
    split_locate(sp, s_beg, lane, cc.b, cc.h, cc.j);
    cc.nb = split_nblocks(sp, cc.b);
    Cursor ic = cc;   // issue cursor
    {
        // the first unit's query rows on their way to L1 while the block table
        // and the first copies are fetched (unit_setup reads them)
        const int qbytes = q_dtype == KVARN_FP32 ? 4 : 2, lines = qbytes;   // 128-byte lines per row
        if (lane < G * lines) {
            const int64_t row = (int64_t)cc.b * n_q + (int64_t)cc.h * G + lane / lines;
            prefetch_l1(static_cast<const uint8_t*>(qptr) + row * kD * qbytes + 128 * (lane % lines));
        }
    }

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    // block-table chunk cache for the issue cursor
    int bt_b = -1, bt_j0 = 0, bt_val = 0;
    auto issue = [&](int stage) {
        if (ic.b != bt_b || ic.j < bt_j0 || ic.j >= bt_j0 + 32) {
            bt_b = ic.b;
            bt_j0 = ic.j;
            const int jj = bt_j0 + lane;
            bt_val = (jj < max_blocks) ? btab[(int64_t)bt_b * max_blocks + jj] : -1;
        }
        int64_t phys = __shfl_sync(kFull, bt_val, ic.j - bt_j0);
        const bool ok = phys >= 0 && phys < n_pool_blocks;
        if (!ok) phys = 0;   // read a valid block, result discarded below
        if (lane == 0) {
            const uint8_t* src = pool + phys * block_bytes + (int64_t)(2 * ic.h) * HB;
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
            if (issue(s)) okmask |= 1u << s;
    }

    // per-unit state
    float kmul = 0.f;          // 2^(e-12) * sm_scale * log2(e) / kA for this lane's head tq
    float m_run = -INFINITY, l_part = 0.f;
    float2 O[8];               // rotated output, channels 32g + 4gq + 2m + {0, 1}, head tq
    const float sgn4[4] = {sign_of4(sb0, sb1, sb2, sb3, 4 * lane), sign_of4(sb0, sb1, sb2, sb3, 4 * lane + 1),
                           sign_of4(sb0, sb1, sb2, sb3, 4 * lane + 2), sign_of4(sb0, sb1, sb2, sb3, 4 * lane + 3)};
    const bool head_ok = tq < G;            // this lane's score / accumulator head
    const int hbq = gq >> 1, part = gq & 1;  // this lane's B-fragment column: (head, hi|lo)
    const bool bcol_ok = hbq < G;
    // The same two-products in three operations: t = RN(x * y) negated on the
    // lo-column lanes, then fma(x_z, y, t) with x_z = x there and 0 on the hi
    // ones (-RN(xy) + xy exact | RN(xy)), then + lo * y.
    const __half2 pneg = part ? __float2half2_rn(-1.f) : __float2half2_rn(1.f);
    const __half2 pone = part ? __float2half2_rn(1.f) : __float2half2_rn(0.f);
    // q's fp16 planes [4][128] each (hi, -hi, lo) and a zero line; this lane
    // reads (hi | -hi), (0 | hi), (0 | lo) for its B-fragment column
    const uint16_t* qpl = reinterpret_cast<const uint16_t*>(qsm);
    const uint16_t* q_n = qpl + (part ? kQNegHi : kQHi) + hbq * kD + 8 * tq;
    const uint16_t* q_z = part ? qpl + kQHi + hbq * kD + 8 * tq : qpl + kQZero + 8 * tq;
    const uint16_t* q_l = part ? qpl + kQLo + hbq * kD + 8 * tq : qpl + kQZero + 8 * tq;
    reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(qsm) + kQZero)[lane] = make_uint2(0u, 0u);
    // this lane's P'' hi | lo rows of pex (the zero line for heads >= G)
    const uint16_t* px_h = bcol_ok ? pex + hbq * B : qpl + kQZero;
    const uint16_t* px_l = bcol_ok ? pex + (4 + hbq) * B : qpl + kQZero;
    // this lane's P'' element offsets in those rows (rotated, see pex_rot): the
    // store of tokens 32 sb + 4 gq .. in row tq, the loads of 32 sb + 8 tq .. in row hbq
    int px_st[NSB], px_ld[NSB];
#pragma unroll
    for (int sb = 0; sb < NSB; ++sb) {
        px_st[sb] = (32 * sb + 4 * gq + pex_rot(B, tq)) % B;
        px_ld[sb] = bcol_ok ? (32 * sb + 8 * tq + pex_rot(B, hbq)) % B : 32 * sb + 8 * tq;
    }

    // the merge finds a unit's partials from its first and last warp, which
    // unit_flush records: this warp is the first if it took the unit's block 0
    bool u_first = false;
    auto unit_setup = [&]() {
        u_first = cc.j == 0;
        __syncwarp();
        for (int j = 0; j < G; ++j) {
            float v[4];
            load_q4(qptr, q_dtype, (int64_t)cc.b * n_q + (int64_t)cc.h * G + j, lane, v);
            if (rotate_q) {   // q_rot = H (sigma . q) / sqrt(128), as the cache was rotated
#pragma unroll
                for (int k = 0; k < 4; ++k) v[k] *= sgn4[k];
                fwht128(v, lane);
#pragma unroll
                for (int k = 0; k < 4; ++k) v[k] *= kInvSqrtD;
            }
            float amax = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fabsf(v[k]));
            amax = warp_max(amax);
            const int e = (amax > 0.f && isfinite(amax)) ? ceil_log2(amax) : 0;
            const float sc = exp2i(12 - e);
            *reinterpret_cast<float4*>(&qsm[j * kD + 4 * lane]) =
                make_float4(v[0] * sc, v[1] * sc, v[2] * sc, v[3] * sc);
            if (j == tq) kmul = (1.0f / kA) * exp2i(e - 12) * sm_scale * kLog2e;
        }
        __syncwarp();
        {
            // fp16 hi, -hi and lo planes [4][128] each, over the fp32 copy (rows of heads >= G zero)
            float4 qv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                qv[j] = j < G ? *reinterpret_cast<const float4*>(&qsm[j * kD + 4 * lane])
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            __syncwarp();
            uint16_t* qhp = reinterpret_cast<uint16_t*>(qsm) + kQHi;
            uint16_t* qnp = reinterpret_cast<uint16_t*>(qsm) + kQNegHi;
            uint16_t* qlp = reinterpret_cast<uint16_t*>(qsm) + kQLo;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float v[4] = {qv[j].x, qv[j].y, qv[j].z, qv[j].w};
                uint32_t hw[2], lw[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const __half h0 = __float2half_rn(v[2 * k]), h1 = __float2half_rn(v[2 * k + 1]);
                    hw[k] = h2_as_u32(__halves2half2(h0, h1));
                    lw[k] = pack_h2(v[2 * k] - __half2float(h0), v[2 * k + 1] - __half2float(h1));
                }
                *reinterpret_cast<uint2*>(qhp + j * kD + 4 * lane) = make_uint2(hw[0], hw[1]);
                *reinterpret_cast<uint2*>(qnp + j * kD + 4 * lane) =
                    make_uint2(hw[0] ^ 0x80008000u, hw[1] ^ 0x80008000u);
                *reinterpret_cast<uint2*>(qlp + j * kD + 4 * lane) = make_uint2(lw[0], lw[1]);
            }
        }
        if (!head_ok) kmul = 0.f;
        m_run = -INFINITY;
        l_part = 0.f;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) O[mt] = make_float2(0.f, 0.f);
    };

    auto unit_flush = [&](bool last) {
        float l = l_part;
        l += __shfl_xor_sync(kFull, l, 4);
        l += __shfl_xor_sync(kFull, l, 8);
        l += __shfl_xor_sync(kFull, l, 16);
        if (head_ok) {
            const int64_t slot = (int64_t)cc.b * n_kv + cc.h + w;
            float* base = partials + (slot * G + tq) * kPartialStride;
            if (gq == 0) {
                base[0] = m_run;
                base[1] = l;
            }
#pragma unroll
            for (int g = 0; g < 4; ++g)   // channels 32g + 4gq + {0,1,2,3}
                *reinterpret_cast<float4*>(base + 4 + 32 * g + 4 * gq) =
                    make_float4(O[2 * g].x, O[2 * g].y, O[2 * g + 1].x, O[2 * g + 1].y);
        }
        if (lane == 0) {
            const int64_t u = (int64_t)cc.b * n_kv + cc.h;
            if (u_first) umap[2 * u] = w;
            if (last) umap[2 * u + 1] = w;
        }
    };

    unit_setup();
    int stage = 0;
    uint32_t phase = 0;
    // A wait that runs out raises the error flag, lets every copy still in
    // flight into this CTA's shared memory land (again with a limit) and ends
    // the warp. The first wait is taken here, outside the block loop, with the
    // launch's limit for it (kWaitLimit; zero under the test switch).
    auto give_up = [&](int64_t x0) {
        if (lane == 0) raise_error(err, KVARN_DEVERR_WAIT_TIMEOUT);
        uint32_t ph = phase;
        for (int k = 0, st2 = stage; k < S && x0 + k < s_end; ++k) {
            mbar_wait_bounded(&bars[st2], ph, kWaitLimit);
            if (++st2 == S) { st2 = 0; ph ^= 1u; }
        }
    };
    if (!mbar_wait_bounded(&bars[0], 0, a.first_wait_limit)) {
        give_up(s_beg);
        return;
    }
    for (int64_t x = s_beg; x < s_end; ++x) {
        if (!mbar_wait_bounded(&bars[stage], phase, kWaitLimit)) {
            give_up(x);
            return;
        }
        const uint8_t* Kb = stages + stage * 2 * HB;
        const uint8_t* Vb = Kb + HB;
        const bool valid = (okmask >> stage) & 1u;
        if (!valid && lane == 0) raise_error(err, KVARN_DEVERR_BLOCK_ID);

        if (valid) {
            const uint16_t* KC = reinterpret_cast<const uint16_t*>(Kb + off_C(B, BITS));
            // ---- largest K channel factor (for a per-block power of two bringing
            // it to (1/2, 1]) and largest V step, in one fp16x2 warp reduction
            float cmax, smax;
            {
                const uint2 c2 = *reinterpret_cast<const uint2*>(KC + 4 * lane);
                const __half2 mc = __hmax2(u32_as_h2(c2.x), u32_as_h2(c2.y));
                __half2 ms;
                if (B == 32) {
                    const uint2 s2 = *reinterpret_cast<const uint2*>(Vb + off_s(B, BITS) + 8 * lane);
                    ms = __hmax2(u32_as_h2(s2.x), u32_as_h2(s2.y));
                } else {
                    const uint4 s4 = *reinterpret_cast<const uint4*>(Vb + off_s(B, BITS) + 16 * lane);
                    ms = __hmax2(__hmax2(u32_as_h2(s4.x), u32_as_h2(s4.y)), __hmax2(u32_as_h2(s4.z), u32_as_h2(s4.w)));
                }
                // (C max, s max) of this lane; both non-negative, so their fp16 bit
                // patterns order as integers and one redux each finds the warp's maxima
                const uint32_t m2 = h2_as_u32(__hmax2(__lows2half2(mc, ms), __highs2half2(mc, ms)));
                cmax = __half2float(__ushort_as_half((uint16_t)__reduce_max_sync(kFull, m2 & 0xffffu)));
                smax = __half2float(__ushort_as_half((uint16_t)__reduce_max_sync(kFull, m2 >> 16)));
            }
            const int ec = ceil_log2(fmaxf(cmax, kF16MinNormal));
            const __half2 cinv = __float2half2_rn(exp2i(-ec));
            // 2-bit: the odd k-slot of each pair meets codes at 2^-18, so its q' is x 4
            const __half2 cinv_o = BITS == 2 ? __float2half2_rn(exp2i(2 - ec)) : cinv;
            const float kmb = kmul * exp2i(ec);
            // ---- QK B operand: q' = q_s * C * 2^-ec as fp16 hi | lo (two-product)
            uint32_t bq[16];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const uint4 c4 = *reinterpret_cast<const uint4*>(KC + 32 * g + 8 * tq);
                const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
                const uint4 n4 = *reinterpret_cast<const uint4*>(q_n + 32 * g);
                const uint4 z4 = *reinterpret_cast<const uint4*>(q_z + 32 * g);
                const uint4 l4 = *reinterpret_cast<const uint4*>(q_l + 32 * g);
                const uint32_t nw[4] = {n4.x, n4.y, n4.z, n4.w};
                const uint32_t zw[4] = {z4.x, z4.y, z4.z, z4.w};
                const uint32_t lw[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const __half2 C2 = __hmul2(u32_as_h2(cw[e2]), (e2 & 1) ? cinv_o : cinv);
                    __half2 r = __hfma2(u32_as_h2(zw[e2]), C2, __hmul2(u32_as_h2(nw[e2]), C2));
                    r = __hfma2(u32_as_h2(lw[e2]), C2, r);
                    bq[4 * g + e2] = h2_as_u32(r);
                }
            }
            // ---- Q'_g * kA for this lane's head: an MMA whose A operand is a code of
            // 1 everywhere sums each group (hi + lo columns), at the codes' scale
            constexpr uint32_t kOneE = BITS == 2 ? kRawOneEven : kCodeScaleH2;
            constexpr uint32_t kOneO = BITS == 2 ? kRawOneOdd : kCodeScaleH2;
            float Qq[4];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                float cq[4];
                mma16816_acc(cq, true, kOneE, kOneE, kOneO, kOneO, bq[4 * g], bq[4 * g + 1]);
                mma16816(cq, kOneE, kOneE, kOneO, kOneO, bq[4 * g + 2], bq[4 * g + 3]);
                Qq[g] = cq[0] + cq[1];
            }
            const uint16_t* Ks = reinterpret_cast<const uint16_t*>(Kb + off_s(B, BITS));
            const uint16_t* Kz = reinterpret_cast<const uint16_t*>(Kb + off_z(B, BITS));
            const uint16_t* KR = reinterpret_cast<const uint16_t*>(Kb + off_R(B, BITS));
            const uint16_t* Vs = reinterpret_cast<const uint16_t*>(Vb + off_s(B, BITS));
            const uint16_t* Vz = reinterpret_cast<const uint16_t*>(Vb + off_z(B, BITS));
            const uint16_t* VR = reinterpret_cast<const uint16_t*>(Vb + off_R(B, BITS));

            // ---------------- QK for every 32-token sub-block
            float2 sc[NSB][2];   // tokens 32sb + 4gq + 2mt + {0, 1}
#pragma unroll
            for (int sb = 0; sb < NSB; ++sb) {
                // the score combine's steps, zero points and R, loaded ahead of the MMAs
                const int t0 = 32 * sb + 4 * gq;
                uint2 s2h[4], z2h[4];
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    s2h[g] = *reinterpret_cast<const uint2*>(Ks + g * B + t0);
                    z2h[g] = *reinterpret_cast<const uint2*>(Kz + g * B + t0);
                }
                const uint2 Rr = *reinterpret_cast<const uint2*>(KR + t0);
                uint32_t kw[RW], kw8[RW];
                {
                    const uint4* rec = reinterpret_cast<const uint4*>(Kb) + (RW / 4) * (32 * sb + lane);
#pragma unroll
                    for (int r = 0; r < RW / 4; ++r) {
                        const uint4 rr = rec[r];
                        kw[4 * r] = rr.x; kw[4 * r + 1] = rr.y; kw[4 * r + 2] = rr.z; kw[4 * r + 3] = rr.w;
                    }
                }
                if (BITS != 2) {
#pragma unroll
                    for (int k = 0; k < RW; ++k) kw8[k] = kw[k] >> 8;
                }
                float acc[4][2][4];   // one chain per (group, 16-token tile)
#pragma unroll
                for (int g = 0; g < 4; ++g)
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const uint32_t b0 = bq[4 * g + 2 * kk], b1 = bq[4 * g + 2 * kk + 1];
#pragma unroll
                        for (int mt = 0; mt < 2; ++mt) {
                            uint32_t a0, a1, a2, a3;
                            if (BITS == 2) {   // word 2i + g/2, pair 4(g%2) + e/2
                                const int j = 4 * (g & 1) + 2 * kk;
                                const int i0 = 2 * (2 * mt) + (g >> 1), i1 = 2 * (2 * mt + 1) + (g >> 1);
                                const int ve = code2_view_of(j), vo = code2_view_of(j + 1);
                                a0 = code2_r(code2_view(kw[i0], ve), j);
                                a1 = code2_r(code2_view(kw[i1], ve), j);
                                a2 = code2_r(code2_view(kw[i0], vo), j + 1);
                                a3 = code2_r(code2_view(kw[i1], vo), j + 1);
                            } else if (BITS == 3) {   // 2-bit word 2i + g/2; high bits in word 8 + i
                                const int j = 4 * (g & 1) + 2 * kk, jh = 8 * (g >> 1) + j;
                                const int i0 = 2 * (2 * mt) + (g >> 1), i1 = 2 * (2 * mt + 1) + (g >> 1);
                                const int h0 = 8 + 2 * mt, h1 = 8 + 2 * mt + 1;
                                a0 = code3_s(kw[i0], kw8[i0], kw[h0], j, jh);
                                a1 = code3_s(kw[i1], kw8[i1], kw[h1], j, jh);
                                a2 = code3_s(kw[i0], kw8[i0], kw[h0], j + 1, jh + 1);
                                a3 = code3_s(kw[i1], kw8[i1], kw[h1], j + 1, jh + 1);
                            } else {           // word 4i + g, field e/2
                                const int j = 2 * kk;
                                const int i0 = 4 * (2 * mt) + g, i1 = 4 * (2 * mt + 1) + g;
                                a0 = code4_s(kw[i0], kw8[i0], j);
                                a1 = code4_s(kw[i1], kw8[i1], j);
                                a2 = code4_s(kw[i0], kw8[i0], j + 1);
                                a3 = code4_s(kw[i1], kw8[i1], j + 1);
                            }
                            mma16816_acc(acc[g][mt], kk == 0, a0, a1, a2, a3, b0, b1);
                        }
                    }
                // scores of tokens 32sb + 4gq + 2mt + {0, 1}, head tq, as fp32 pairs
                const float2 Rv[2] = {__half22float2(u32_as_h2(Rr.x)), __half22float2(u32_as_h2(Rr.y))};
                float2 s_[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const uint2 s2 = s2h[g], z2 = z2h[g];
                    const float2 sv[2] = {__half22float2(u32_as_h2(s2.x)), __half22float2(u32_as_h2(s2.y))};
                    const float2 zv[2] = {__half22float2(u32_as_h2(z2.x)), __half22float2(u32_as_h2(z2.y))};
                    const float2 qq = make_float2(Qq[g], Qq[g]);
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) {   // hi + lo column of rows gq, gq + 8
                        const float2 d = make_float2(acc[g][mt][0] + acc[g][mt][1], acc[g][mt][2] + acc[g][mt][3]);
                        s_[mt] = __ffma2_rn(sv[mt], d, s_[mt]);
                        s_[mt] = __ffma2_rn(zv[mt], qq, s_[mt]);
                    }
                }
                const float2 kmb2 = make_float2(kmb, kmb);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) sc[sb][mt] = __fmul2_rn(__fmul2_rn(s_[mt], Rv[mt]), kmb2);
            }
            // ---------------- online softmax over the block (head tq: 8 lanes x 4 tokens per sub-block)
            float bm = -INFINITY;
#pragma unroll
            for (int sb = 0; sb < NSB; ++sb)
                bm = fmaxf(bm, fmaxf(fmaxf(sc[sb][0].x, sc[sb][0].y), fmaxf(sc[sb][1].x, sc[sb][1].y)));
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 4));
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 8));
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
            const float m_new = fmaxf(m_run, bm);
            const bool none = m_new == -INFINITY;
            const float alpha = none ? 1.f : fast_exp2(m_run - m_new);
            const float2 nm2 = make_float2(-m_new, -m_new);
            float2 pR[NSB][2];
            float psum = 0.f, pmax = 0.f;
#pragma unroll
            for (int sb = 0; sb < NSB; ++sb) {
                const uint2 Rr = *reinterpret_cast<const uint2*>(VR + 32 * sb + 4 * gq);
                const float2 Rv[2] = {__half22float2(u32_as_h2(Rr.x)), __half22float2(u32_as_h2(Rr.y))};
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const float2 e = __fadd2_rn(sc[sb][mt], nm2);
                    const float2 p = none ? make_float2(0.f, 0.f) : make_float2(fast_exp2(e.x), fast_exp2(e.y));
                    psum += p.x;
                    psum += p.y;
                    pR[sb][mt] = __fmul2_rn(p, Rv[mt]);
                    pmax = fmaxf(pmax, fmaxf(pR[sb][mt].x, pR[sb][mt].y));
                }
            }
            l_part = l_part * alpha + psum;
            m_run = m_new;
            {   // (unconditional: cheaper than testing alpha == 1)
                const float2 al2 = make_float2(alpha, alpha);
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) O[mt] = __fmul2_rn(O[mt], al2);
            }
            pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, 4));
            pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, 8));
            pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, 16));
            // power of two lam so that p*R*lam <= 2^14 and p*R*s*lam <= 2^12 (fp16 range
            // of P' and of its hi | lo halves); undone in the update of O
            float lam = 1.f;
            if (pmax > 0.f) {
                int k = 14 - ceil_log2(pmax);
                if (smax > 0.f) k = min(k, 12 - ceil_log2(pmax * smax));
                lam = exp2i(k);
            }
            const float2 lam2 = make_float2(lam, lam);
#pragma unroll
            for (int sb = 0; sb < NSB; ++sb) {
                uint32_t hw[2], lw[2];
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const float2 v = __fmul2_rn(pR[sb][mt], lam2);
                    const __half2 h = __float22half2_rn(v);
                    const float2 hf = __half22float2(h);
                    hw[mt] = h2_as_u32(h);
                    lw[mt] = h2_as_u32(__float22half2_rn(__fadd2_rn(v, make_float2(-hf.x, -hf.y))));
                }
                uint16_t* ph = pex + (0 * 4 + tq) * B + px_st[sb];
                uint16_t* pl = pex + (1 * 4 + tq) * B + px_st[sb];
                *reinterpret_cast<uint2*>(ph) = make_uint2(hw[0], hw[1]);
                *reinterpret_cast<uint2*>(pl) = make_uint2(lw[0], lw[1]);
            }
            __syncwarp();

            // ---------------- PV over the block's tokens
            float Ob[8][4], Dz[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            // unrolled, each accumulator chain started by its first MMA from a zero C
#pragma unroll
            for (int sb = 0; sb < NSB; ++sb) {
                // this lane's B column (head hbq, part) for tokens 32sb + 8tq .. +7
                const uint4 phv = *reinterpret_cast<const uint4*>(px_h + px_ld[sb]);
                const uint4 plv = *reinterpret_cast<const uint4*>(px_l + px_ld[sb]);
                const uint32_t ph[4] = {phv.x, phv.y, phv.z, phv.w};
                const uint32_t pl[4] = {plv.x, plv.y, plv.z, plv.w};
                uint32_t plm[4], pa[4], hpn[4], hpz[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    plm[k] = h2_as_u32(__hmul2(u32_as_h2(pl[k]), pone));
                    pa[k] = part ? pl[k] : ph[k];
                    hpn[k] = h2_as_u32(__hmul2(u32_as_h2(ph[k]), pneg));
                    hpz[k] = h2_as_u32(__hmul2(u32_as_h2(ph[k]), pone));
                }
                uint32_t bv[4][4];   // [group][token pair]
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const uint4 s4 = *reinterpret_cast<const uint4*>(Vs + g * B + 32 * sb + 8 * tq);
                    const uint32_t sw[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const __half2 s2 = u32_as_h2(sw[k]);
                        __half2 r = __hfma2(u32_as_h2(hpz[k]), s2, __hmul2(u32_as_h2(hpn[k]), s2));
                        r = __hfma2(u32_as_h2(plm[k]), s2, r);
                        bv[g][k] = h2_as_u32(r);
                    }
                }
                // zero-point sums: rows (head, part) x columns z_0..z_3, s_0..s_3
                {
                    const uint16_t* src = (gq < 4 ? Vz : Vs) + (gq & 3) * B + 32 * sb + 8 * tq;
                    const uint4 z4 = *reinterpret_cast<const uint4*>(src);
                    mma16816(Dz, pa[0], 0u, pa[1], 0u, z4.x, z4.y);
                    mma16816(Dz, pa[2], 0u, pa[3], 0u, z4.z, z4.w);
                }
                uint32_t vw[RW], vw8[RW];
                {
                    const uint4* rec = reinterpret_cast<const uint4*>(Vb) + (RW / 4) * (32 * sb + lane);
#pragma unroll
                    for (int r = 0; r < RW / 4; ++r) {
                        const uint4 rr = rec[r];
                        vw[4 * r] = rr.x; vw[4 * r + 1] = rr.y; vw[4 * r + 2] = rr.z; vw[4 * r + 3] = rr.w;
                    }
                }
                if (BITS != 2) {
#pragma unroll
                    for (int k = 0; k < RW; ++k) vw8[k] = vw[k] >> 8;
                }
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    const int g = mt >> 1, m = mt & 1;
                    if (BITS == 2) {   // word 2g + f/2, pair 4(d/4) + 2((d%4)/2) + f%2
                        // rows gq take the even fields (code * 2^-16), rows gq + 8 the odd ones (2^-18)
                        const uint32_t wd = vw[2 * g + m];
#pragma unroll
                        for (int kt = 0; kt < 2; ++kt) {
                            const int f = 4 * kt;
                            mma16816_acc(Ob[mt], sb == 0 && kt == 0, code2_r(code2_view(wd, code2_view_of(f)), f),
                                         code2_r(code2_view(wd, code2_view_of(f + 1)), f + 1),
                                         code2_r(code2_view(wd, code2_view_of(f + 2)), f + 2),
                                         code2_r(code2_view(wd, code2_view_of(f + 3)), f + 3), bv[g][2 * kt],
                                         bv[g][2 * kt + 1]);
                        }
                    } else if (BITS == 3) {   // 2-bit word 2g + f/2; high bits in word 8 + g, bit 8(f/2) + j
                        const int wl = 2 * g + m, wh = 8 + g;
#pragma unroll
                        for (int kt = 0; kt < 2; ++kt)
                            mma16816_acc(Ob[mt], sb == 0 && kt == 0,
                                         code3_s(vw[wl], vw8[wl], vw[wh], 4 * kt + 0, 8 * m + 4 * kt + 0),
                                         code3_s(vw[wl], vw8[wl], vw[wh], 4 * kt + 1, 8 * m + 4 * kt + 1),
                                         code3_s(vw[wl], vw8[wl], vw[wh], 4 * kt + 2, 8 * m + 4 * kt + 2),
                                         code3_s(vw[wl], vw8[wl], vw[wh], 4 * kt + 3, 8 * m + 4 * kt + 3),
                                         bv[g][2 * kt], bv[g][2 * kt + 1]);
                    } else {           // word 4g + f, field d/2
                        const int w0 = 4 * g + 2 * m, w1 = w0 + 1;
#pragma unroll
                        for (int kt = 0; kt < 2; ++kt)
                            mma16816_acc(Ob[mt], sb == 0 && kt == 0, code4_s(vw[w0], vw8[w0], 2 * kt),
                                         code4_s(vw[w1], vw8[w1], 2 * kt), code4_s(vw[w0], vw8[w0], 2 * kt + 1),
                                         code4_s(vw[w1], vw8[w1], 2 * kt + 1), bv[g][2 * kt], bv[g][2 * kt + 1]);
                    }
                }
            }
            __syncwarp();   // pex is rewritten by the next block
            // zs[h][g] = the z-sum, hi + lo rows, at the codes' scale; delivered to the
            // lanes of head tq
            float zq[4];
            {
                const float zA = Dz[0] + __shfl_xor_sync(kFull, Dz[0], 4);   // valid where tq < 2:
                const float zB = Dz[1] + __shfl_xor_sync(kFull, Dz[1], 4);   // groups 2tq, 2tq+1 of head gq/2
                zq[0] = kA * __shfl_sync(kFull, zA, 8 * tq);
                zq[1] = kA * __shfl_sync(kFull, zB, 8 * tq);
                zq[2] = kA * __shfl_sync(kFull, zA, 8 * tq + 1);
                zq[3] = kA * __shfl_sync(kFull, zB, 8 * tq + 1);
            }
            // ---------------- O += C_c / (kA lam) * (Ob + zs * kA)
            {
                const float il4 = (1.0f / kA) / lam;
                // 2-bit: rows gq + 8 (y) hold odd fields at kA / 4
                const float2 rw2 = BITS == 2 ? make_float2(1.f, 4.f) : make_float2(1.f, 1.f);
                const float2 il42 = make_float2(il4, il4);
                const uint16_t* VC = reinterpret_cast<const uint16_t*>(Vb + off_C(B, BITS));
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const uint2 c2 = *reinterpret_cast<const uint2*>(VC + 32 * g + 4 * gq);
                    const float2 c01 = __half22float2(u32_as_h2(c2.x)), c23 = __half22float2(u32_as_h2(c2.y));
                    const float2 zq2 = make_float2(zq[g], zq[g]);
#pragma unroll
                    for (int m = 0; m < 2; ++m) {   // channels 32g + 4gq + 2m + {0, 1}
                        const int mt = 2 * g + m;
                        const float2 t = __ffma2_rn(make_float2(Ob[mt][0] + Ob[mt][1], Ob[mt][2] + Ob[mt][3]), rw2, zq2);
                        O[mt] = __ffma2_rn(__fmul2_rn(m ? c23 : c01, il42), t, O[mt]);
                    }
                }
            }
        }
        // ---- retire the stage and refill it
        __syncwarp();
        okmask &= ~(1u << stage);
        if (x + S < s_end && issue(stage)) okmask |= 1u << stage;
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
            unit_flush(done.b != pb || done.h != ph_);
            cc = done;
            if (x + 1 < s_end) unit_setup();
        }
    }
}

// The split kernel at ptxas's own register target, and with a minimum of
// MINB resident CTAs per SM (at most 65536 / (32 MINB) registers a thread).
template <int B, int BITS, int S>
__global__ void __launch_bounds__(32) decode_attn_2bit_kernel(AttnArgs a) {
    decode_attn_2bit_body<B, BITS, S>(a);
}
template <int B, int BITS, int S, int MINB>
__global__ void __launch_bounds__(32, MINB) decode_attn_2bit_kernel_minb(AttnArgs a) {
    decode_attn_2bit_body<B, BITS, S>(a);
}

// ---------------------------------------------------------------- host side
template <int B, int BITS>
constexpr int stages_for() { return 2; }

// Minimum resident CTAs per SM that the split kernel is compiled for (0: the
// plain kernel), chosen by timing each instantiation on the 64 x 8192-token
// Llama-shaped cache. 3-bit, B = 64: shared memory holds 9 CTAs per SM
// whatever the registers, and with the bound at 1 ptxas takes 191 registers
// instead of 156 (237 -> 200 us). 3-bit, B = 32: 16 gives 128 registers
// without spills, 15 warps per SM (shared memory) instead of 12 (218 -> 207
// us). The 2- and 4-bit instantiations were fastest plain (bounds of 1, 10,
// 11 at 2 bits, B = 64: 142, 129.5, 129.4 against 128.7 us).
template <int B, int BITS>
constexpr int attn_min_ctas() { return BITS != 3 ? 0 : (B == 64 ? 1 : 16); }

template <int B, int BITS>
constexpr auto attn_kernel_fn() {
    constexpr int S = stages_for<B, BITS>(), M = attn_min_ctas<B, BITS>();
    if constexpr (M > 0) return decode_attn_2bit_kernel_minb<B, BITS, S, M>;
    else return decode_attn_2bit_kernel<B, BITS, S>;
}

template <int B, int BITS>
size_t attn_smem_bytes() {
    return (size_t)stages_for<B, BITS>() * 2 * head_block_bytes(B, BITS) + 64 + attn_q_bytes(B) +
           2 * 4 * B * sizeof(uint16_t);
}

template <int B, int BITS>
struct AttnKernel {
    static constexpr int kB = B;
    static constexpr auto fn = attn_kernel_fn<B, BITS>();
    static size_t smem() { return attn_smem_bytes<B, BITS>(); }
};

template <typename F>
auto with_attn_kernel(int block_size, int bits, F&& f) {
    if (block_size == 32)
        return bits == 4 ? f(AttnKernel<32, 4>{}) : (bits == 3 ? f(AttnKernel<32, 3>{}) : f(AttnKernel<32, 2>{}));
    return bits == 4 ? f(AttnKernel<64, 4>{}) : (bits == 3 ? f(AttnKernel<64, 3>{}) : f(AttnKernel<64, 2>{}));
}

// Resident warps of the split-K kernel for (block size, code width) on
// `device` (cached per device).
int attn_grid_warps(int block_size, int bits, int device) {
    static int cache[2][3][64];
    const int bi = block_size == 32 ? 0 : 1, wi = bits - 2;
    if (device < 0 || device >= 64) return 0;
    if (cache[bi][wi][device] > 0) return cache[bi][wi][device];
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
    const cudaError_t e = with_attn_kernel(block_size, bits, [&](auto k) {
        using K = decltype(k);
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, K::fn, 32, K::smem());
    });
    if (e != cudaSuccess || per_sm <= 0) return 0;
    cache[bi][wi][device] = sms * per_sm;
    return cache[bi][wi][device];
}

cudaError_t launch_decode_attn(const kvarn_config& cfg, const void* q, int q_dtype, const void* pool,
                               int64_t n_pool_blocks, int64_t block_bytes, const void* staging,
                               const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                               int batch, float* out, void* workspace, int nw, cudaStream_t st) {
    AttnArgs a = {};
    a.q = q;
    a.q_dtype = q_dtype;
    a.pool = (const uint8_t*)pool;
    a.staging = (const uint16_t*)staging;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.err = (uint32_t*)workspace;
    a.partials = (float*)((uint8_t*)workspace + kWsHeader);
    // the unit map follows this launch's partial slots (the workspace size
    // counts the largest grid's slots, then the map)
    a.unit_map = (int32_t*)((uint8_t*)a.partials + ((size_t)batch * cfg.n_kv_heads + (size_t)nw) *
                                                       (size_t)(cfg.n_q_heads / cfg.n_kv_heads) * kPartialStride *
                                                       sizeof(float));
    a.out = out;
    a.n_pool_blocks = n_pool_blocks;
    a.block_bytes = block_bytes;
    a.max_blocks = max_blocks;
    a.batch = batch;
    a.chunk = 1;
    a.single = 0;
    a.n_q = cfg.n_q_heads;
    a.n_kv = cfg.n_kv_heads;
    a.G = cfg.n_q_heads / cfg.n_kv_heads;
    a.nw = nw;
    a.sm_scale = cfg.sm_scale;
    a.flags = cfg.flags;
    // test switch: every warp's first copy wait gives up at once (the
    // wait-timeout path, run without a hang)
    a.first_wait_limit = (cfg.flags & KVARN_FLAG_TEST_WAIT_TIMEOUT) ? 0u : kWaitLimit;
    for (int i = 0; i < 4; ++i) a.sb[i] = cfg.sign_bits[i];
    return with_attn_kernel(cfg.block_size, cfg.bits, [&](auto k) {
        using K = decltype(k);
        cudaError_t e = launch_pdl(K::fn, nw, 32, K::smem(), st, a);
        // up to one wave of wide CTAs (4 per SM), so that 8 warps share each
        // row's raw tail rows
        if (e == cudaSuccess) e = launch_merge<K::kB, true>(a, nw, 4, st);
        return e;
    });
}

}  // namespace kvarn
