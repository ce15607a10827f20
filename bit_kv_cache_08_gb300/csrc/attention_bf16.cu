// attention_bf16.cu -- decode attention over a plain bf16 paged KV cache:
// the comparison point for the 2-bit path, with the same balanced split-K
// partition and merge, no rotation and no staging.
//
// The split unit is a 16-token chunk of a page (4 KB of K and 4 KB of V).
// Each lane copies one 256-byte row (lanes 0-15 K, 16-31 V) with a 1-D bulk
// copy into a 3-stage shared-memory ring whose rows are padded to 272 bytes,
// so that ldmatrix reads of 8 rows hit 32 distinct banks. Both contractions
// run on mma.sync m16n8k16 (bf16 in, f32 accumulate):
//   QK  A = K chunk (16 tokens x 16 channels per k-step, ldmatrix),
//       B = q as bf16 hi | lo per head (exact for a bf16 query);
//   PV  A = V^T (16 channels x 16 tokens per m-tile, ldmatrix.trans),
//       B = p as bf16 hi | lo per head, so p keeps ~16 bits.
// Accumulator columns are (head, hi | lo); the online softmax runs per chunk
// in the log2 domain and rescales the PV accumulators in place. Rows past the
// sequence end are zero-filled instead of copied (0 * garbage could be NaN).
#include "attn_common.cuh"

namespace kvarn {

constexpr int kChunk = 16;
constexpr int kBfStages = 3;
constexpr int kRowPitch = kD * 2 + 16;                 // 272 bytes
constexpr int kStageBytes = 2 * kChunk * kRowPitch;    // K rows then V rows

__device__ __forceinline__ void mma16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(const void* p, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x4_trans(const void* p, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_addr(p)));
}

// (hi, lo) bf16 pairs of two floats: hi = RN(v), lo = RN(v - hi)
__device__ __forceinline__ void split_bf16x2(float v0, float v1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

template <int B>
__global__ void __launch_bounds__(32) decode_attn_bf16_kernel(AttnArgs a) {
    wait_prior_grids();
    constexpr int CPB = B / kChunk;   // chunks per page
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBfStages * kStageBytes);
    const int lane = threadIdx.x;
    const int gq = lane >> 2, tq = lane & 3;
    const int w = blockIdx.x;
    const int max_pages = a.max_blocks / CPB;
    const int G = a.G;

    // positions are 16-token chunks; a partial last chunk counts
    const SplitArgs sp{a.seq_lens, a.batch, a.n_kv, a.max_blocks, kChunk, 1, 1};
    Cursor cc;
    cc.b = cc.h = cc.j = 0;
    const int64_t W = split_locate(sp, 0, lane, cc.b, cc.h, cc.j);
    const int64_t nwe = split_active_warps(W, a.nw, (int64_t)a.batch * a.n_kv, 0.f);   // >= 1 chunk per warp
    if (w >= nwe) return;
    const int64_t s_beg = (int64_t)w * W / nwe, s_end = (int64_t)(w + 1) * W / nwe;
    if (s_beg >= s_end) return;
    split_locate(sp, s_beg, lane, cc.b, cc.h, cc.j);
    cc.nb = split_nblocks(sp, cc.b);
    Cursor ic = cc;

    if (lane == 0) {
        for (int s = 0; s < kBfStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    // every lane moves one row: lanes 0-15 K, 16-31 V; rows past the end are zeroed
    auto issue = [&](int stage) {
        const int page = ic.j / CPB, sub = ic.j % CPB;
        int64_t phys = a.block_table[(int64_t)ic.b * max_pages + page];
        const bool ok = phys >= 0 && phys < a.n_pool_blocks;
        if (!ok) phys = 0;
        const int nv = min(kChunk, a.seq_lens[ic.b] - ic.j * kChunk);
        const int kind = lane >> 4, row = lane & 15;
        uint8_t* dst = stages + stage * kStageBytes + (kind * kChunk + row) * kRowPitch;
        if (row >= nv) {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int i = 0; i < kD * 2 / 16; ++i) d4[i] = make_uint4(0, 0, 0, 0);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (lane == 0) mbar_arrive_expect_tx(&bars[stage], 2 * nv * kD * 2);
        __syncwarp();
        if (row < nv) {
            const uint8_t* src = a.pool + phys * a.block_bytes + (int64_t)(2 * ic.h + kind) * B * kD * 2 +
                                 (int64_t)(sub * kChunk + row) * kD * 2;
            bulk_g2s(dst, src, kD * 2, &bars[stage]);
        }
        split_advance(sp, ic);
        return ok;
    };
    uint32_t okmask = 0;
    {
        int64_t x = s_beg;
        for (int s = 0; s < kBfStages && x < s_end; ++s, ++x)
            if (issue(s)) okmask |= 1u << s;
    }

    const int hb = gq >> 1, part = gq & 1;   // this lane's B column: (head, hi | lo)
    const float qs = a.sm_scale * kLog2e;
    uint32_t qb[16];                          // QK B fragments, k-steps 0..7
    float O[8][4];                            // PV accumulators: channels 16mt + gq (+8), head tq hi | lo
    float m_run = -INFINITY, l_part = 0.f;

    auto unit_setup = [&]() {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int c = 16 * (i >> 1) + 8 * (i & 1) + 2 * tq;
            float v0 = 0.f, v1 = 0.f;
            if (hb < G) {
                const int64_t row = (int64_t)cc.b * a.n_q + (int64_t)cc.h * G + hb;
                if (a.q_dtype == KVARN_FP32) {
                    const float2 f = *reinterpret_cast<const float2*>(static_cast<const float*>(a.q) + row * kD + c);
                    v0 = f.x; v1 = f.y;
                } else {
                    const uint32_t u = *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(a.q) + row * kD + c);
                    v0 = __uint_as_float(u << 16);
                    v1 = __uint_as_float(u & 0xffff0000u);
                }
            }
            uint32_t hi, lo;
            split_bf16x2(v0, v1, hi, lo);
            qb[i] = part ? lo : hi;
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) O[mt][0] = O[mt][1] = O[mt][2] = O[mt][3] = 0.f;
        m_run = -INFINITY;
        l_part = 0.f;
    };
    auto unit_flush = [&]() {
        float l = l_part;
        l += __shfl_xor_sync(kFull, l, 4);
        l += __shfl_xor_sync(kFull, l, 8);
        l += __shfl_xor_sync(kFull, l, 16);
        if (tq < G) {
            const int64_t slot = (int64_t)cc.b * a.n_kv + cc.h + w;
            float* base = a.partials + (slot * G + tq) * kPartialStride;
            if (gq == 0) {
                base[0] = m_run;
                base[1] = l;
            }
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                base[4 + 16 * mt + gq] = O[mt][0] + O[mt][1];
                base[4 + 16 * mt + gq + 8] = O[mt][2] + O[mt][3];
            }
        }
    };

    unit_setup();
    int stage = 0;
    uint32_t phase = 0;
    // ldmatrix row addresses: lane supplies row (lane & 7) of matrix (lane >> 3)
    const int mi = lane >> 3, mr = lane & 7;
    const int k_row = 8 * (mi & 1) + mr, k_col = 8 * (mi >> 1);   // QK A: rows = tokens
    const int v_row = 8 * (mi >> 1) + mr, v_col = 8 * (mi & 1);   // PV A (trans): rows = tokens
    for (int64_t x = s_beg; x < s_end; ++x) {
        if (!mbar_wait_bounded(&bars[stage], phase, kWaitLimit)) {
            if (lane == 0) raise_error(a.err, KVARN_DEVERR_WAIT_TIMEOUT);
            uint32_t ph = phase;
            for (int k = 0, st2 = stage; k < kBfStages && x + k < s_end; ++k) {
                mbar_wait_bounded(&bars[st2], ph, kWaitLimit);
                if (++st2 == kBfStages) { st2 = 0; ph ^= 1u; }
            }
            return;
        }
        const bool valid = (okmask >> stage) & 1u;
        if (!valid && lane == 0) raise_error(a.err, KVARN_DEVERR_BLOCK_ID);
        const int nvalid = min(kChunk, a.seq_lens[cc.b] - cc.j * kChunk);
        if (valid) {
            const uint8_t* Kc = stages + stage * kStageBytes;
            const uint8_t* Vc = Kc + kChunk * kRowPitch;
            // ---- scores: tokens gq and gq + 8, head tq (hi + lo columns)
            float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(Kc + k_row * kRowPitch + (16 * ks + k_col) * 2, a0, a1, a2, a3);
                mma16816_bf16(sacc, a0, a1, a2, a3, qb[2 * ks], qb[2 * ks + 1]);
            }
            float s0 = (sacc[0] + sacc[1]) * qs, s1 = (sacc[2] + sacc[3]) * qs;
            if (gq >= nvalid) s0 = -INFINITY;
            if (gq + 8 >= nvalid) s1 = -INFINITY;
            float bm = fmaxf(s0, s1);
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 4));
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 8));
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
            const float m_new = fmaxf(m_run, bm);
            const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
            const float p0 = (m_new == -INFINITY) ? 0.f : exp2f(s0 - m_new);
            const float p1 = (m_new == -INFINITY) ? 0.f : exp2f(s1 - m_new);
            l_part = l_part * alpha + (p0 + p1);
            m_run = m_new;
            if (__any_sync(kFull, alpha != 1.f)) {
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    O[mt][0] *= alpha; O[mt][1] *= alpha; O[mt][2] *= alpha; O[mt][3] *= alpha;
                }
            }
            // ---- PV B fragments: p of tokens 2tq, 2tq+1 (b0) and 2tq+8, 2tq+9 (b1), head hb
            const int sA = 8 * tq + hb, sB = 8 * tq + 4 + hb;
            const float pa0 = __shfl_sync(kFull, p0, sA), pa1 = __shfl_sync(kFull, p0, sB);
            const float pb0 = __shfl_sync(kFull, p1, sA), pb1 = __shfl_sync(kFull, p1, sB);
            uint32_t h0, l0, h1, l1;
            split_bf16x2(pa0, pa1, h0, l0);
            split_bf16x2(pb0, pb1, h1, l1);
            const uint32_t b0 = part ? l0 : h0, b1 = part ? l1 : h1;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_trans(Vc + v_row * kRowPitch + (16 * mt + v_col) * 2, a0, a1, a2, a3);
                mma16816_bf16(O[mt], a0, a1, a2, a3, b0, b1);
            }
        }
        __syncwarp();
        okmask &= ~(1u << stage);
        if (x + kBfStages < s_end && issue(stage)) okmask |= 1u << stage;
        if (++stage == kBfStages) {
            stage = 0;
            phase ^= 1u;
        }
        const int pb = cc.b, ph_ = cc.h;
        split_advance(sp, cc);
        if (x + 1 == s_end || cc.b != pb || cc.h != ph_) {
            Cursor nxt = cc;
            cc.b = pb;
            cc.h = ph_;
            unit_flush();
            cc = nxt;
            if (x + 1 < s_end) unit_setup();
        }
    }
}

size_t attn_bf16_smem_bytes() { return (size_t)kBfStages * kStageBytes + 64; }

int attn_bf16_grid_warps(int block_size, int device) {
    static int cache[2][64];
    const int bi = block_size == 32 ? 0 : 1;
    if (device < 0 || device >= 64) return 0;
    if (cache[bi][device] > 0) return cache[bi][device];
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
    cudaError_t e = block_size == 32
                        ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_attn_bf16_kernel<32>, 32,
                                                                        attn_bf16_smem_bytes())
                        : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_attn_bf16_kernel<64>, 32,
                                                                        attn_bf16_smem_bytes());
    if (e != cudaSuccess || per_sm <= 0) return 0;
    cache[bi][device] = sms * per_sm;
    return cache[bi][device];
}

cudaError_t launch_decode_attn_bf16(const kvarn_config& cfg, const void* q, int q_dtype, const void* kv_pool,
                                    int64_t n_pool_blocks, const int32_t* block_table, int max_blocks,
                                    const int32_t* seq_lens, int batch, float* out, void* workspace, int nw,
                                    cudaStream_t st) {
    AttnArgs a = {};
    a.q = q;
    a.q_dtype = q_dtype;
    a.pool = (const uint8_t*)kv_pool;
    a.staging = nullptr;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.err = (uint32_t*)workspace;
    a.partials = (float*)((uint8_t*)workspace + kWsHeader);
    a.out = out;
    a.n_pool_blocks = n_pool_blocks;
    a.block_bytes = (int64_t)cfg.n_kv_heads * 2 * cfg.block_size * kD * 2;
    a.max_blocks = max_blocks * (cfg.block_size / kChunk);   // in 16-token chunks
    a.batch = batch;
    a.chunk = 1;
    a.single = 0;
    a.n_q = cfg.n_q_heads;
    a.n_kv = cfg.n_kv_heads;
    a.G = cfg.n_q_heads / cfg.n_kv_heads;
    a.nw = nw;
    a.sm_scale = cfg.sm_scale;
    a.flags = cfg.flags;
    for (int i = 0; i < 4; ++i) a.sb[i] = cfg.sign_bits[i];
    cudaError_t e;
    if (cfg.block_size == 32)
        e = launch_pdl(decode_attn_bf16_kernel<32>, nw, 32, attn_bf16_smem_bytes(), st, a);
    else
        e = launch_pdl(decode_attn_bf16_kernel<64>, nw, 32, attn_bf16_smem_bytes(), st, a);
    // (no raw tail rows: the wide kernel only for many partials per unit)
    if (e == cudaSuccess) e = launch_merge<kChunk, false>(a, nw, 0, st);
    return e;
}

}  // namespace kvarn
