// attention_bf16.cu -- decode attention over a plain bf16 paged KV cache:
// the comparison point for the 2-bit path, with the same balanced split-K
// partition and merge, no rotation and no staging.
//
// The split unit is a 16-token chunk of a page (4 KB of K and 4 KB of V),
// streamed into a 3-stage shared-memory ring with 1-D bulk copies. Lane l
// owns channels 4l..4l+3; the 16 x G partial dot products of a chunk are
// summed across lanes with a transposing butterfly (each of 5 levels halves
// the values a lane carries), which leaves lane l with the scores of token
// l/2 for heads 2(l%2) and 2(l%2)+1. All arithmetic is fp32.
#include "attn_common.cuh"

namespace kvarn {

constexpr int kChunk = 16;
constexpr int kBfStages = 3;
constexpr int kChunkBytes = kChunk * kD * 2;   // one of K or V

template <int B>
__global__ void __launch_bounds__(32) decode_attn_bf16_kernel(AttnArgs a) {
    constexpr int CPB = B / kChunk;   // chunks per page
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBfStages * 2 * kChunkBytes);
    const int lane = threadIdx.x;
    const int w = blockIdx.x;
    const int max_pages = a.max_blocks / CPB;

    // positions are 16-token chunks; a partial last chunk counts
    const SplitArgs sp{a.seq_lens, a.batch, a.n_kv, a.max_blocks, kChunk, 1};
    Cursor cc;
    cc.b = cc.h = cc.j = 0;
    const int64_t W = split_locate(sp, 0, lane, cc.b, cc.h, cc.j);
    const int64_t s_beg = (int64_t)w * W / a.nw, s_end = (int64_t)(w + 1) * W / a.nw;
    if (s_beg >= s_end) return;
    split_locate(sp, s_beg, lane, cc.b, cc.h, cc.j);
    cc.nb = split_nblocks(sp, cc.b);
    Cursor ic = cc;

    if (lane == 0) {
        for (int s = 0; s < kBfStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    auto issue = [&](int stage) {
        const int page = ic.j / CPB, sub = ic.j % CPB;
        int64_t phys = a.block_table[(int64_t)ic.b * max_pages + page];
        const bool ok = phys >= 0 && phys < a.n_pool_blocks;
        if (!ok) phys = 0;
        if (lane == 0) {
            const uint8_t* kp = a.pool + phys * a.block_bytes + (int64_t)(2 * ic.h) * B * kD * 2 +
                                (int64_t)sub * kChunkBytes;
            mbar_arrive_expect_tx(&bars[stage], 2 * kChunkBytes);
            bulk_g2s(stages + stage * 2 * kChunkBytes, kp, kChunkBytes, &bars[stage]);
            bulk_g2s(stages + stage * 2 * kChunkBytes + kChunkBytes, kp + (int64_t)B * kD * 2, kChunkBytes,
                     &bars[stage]);
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

    float qv[4][4], O[4][4], m_run[4], l_run[4];
    auto unit_setup = [&]() {
        const float qs = a.sm_scale * kLog2e;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (h < a.G) load_q4(a.q, a.q_dtype, (int64_t)cc.b * a.n_q + (int64_t)cc.h * a.G + h, lane, v);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                qv[h][k] = v[k] * qs;
                O[h][k] = 0.f;
            }
            m_run[h] = -INFINITY;
            l_run[h] = 0.f;
        }
    };
    auto unit_flush = [&]() {
        const int64_t slot = (int64_t)cc.b * a.n_kv + cc.h + w;
        for (int h = 0; h < a.G; ++h) {
            float* base = a.partials + (slot * a.G + h) * kPartialStride;
            if (lane == 0) {
                base[0] = m_run[h];
                base[1] = l_run[h];
            }
            reinterpret_cast<float4*>(base + 4)[lane] = make_float4(O[h][0], O[h][1], O[h][2], O[h][3]);
        }
    };

    unit_setup();
    int stage = 0;
    uint32_t phase = 0;
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
            const uint8_t* Kc = stages + stage * 2 * kChunkBytes;
            const uint8_t* Vc = Kc + kChunkBytes;
            float v[64];   // [token][head] partial dots
#pragma unroll
            for (int t = 0; t < kChunk; ++t) {
                const uint2 ku = *reinterpret_cast<const uint2*>(Kc + t * kD * 2 + 8 * lane);
                const float k0 = __uint_as_float(ku.x << 16), k1 = __uint_as_float(ku.x & 0xffff0000u);
                const float k2 = __uint_as_float(ku.y << 16), k3 = __uint_as_float(ku.y & 0xffff0000u);
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    v[4 * t + h] = fmaf(qv[h][3], k3, fmaf(qv[h][2], k2, fmaf(qv[h][1], k1, qv[h][0] * k0)));
            }
            // transposing butterfly: lane ends with entries 2*lane, 2*lane+1
#pragma unroll
            for (int lvl = 0, m = 16, half = 32; lvl < 5; ++lvl, m >>= 1, half >>= 1) {
                const bool up = (lane & m) != 0;
#pragma unroll
                for (int i = 0; i < half; ++i) {
                    const float send = up ? v[i] : v[i + half];
                    const float keep = up ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(kFull, send, m);
                }
            }
            const int tok = lane >> 1, hp = 2 * (lane & 1);   // heads hp, hp+1
            float s0 = (tok < nvalid) ? v[0] : -INFINITY;
            float s1 = (tok < nvalid) ? v[1] : -INFINITY;
            float b0 = s0, b1 = s1;
#pragma unroll
            for (int mm = 2; mm <= 16; mm <<= 1) {
                b0 = fmaxf(b0, __shfl_xor_sync(kFull, b0, mm));
                b1 = fmaxf(b1, __shfl_xor_sync(kFull, b1, mm));
            }
            float mn[2], p[2];
            const float mo0 = (hp == 0) ? m_run[0] : m_run[2];
            const float mo1 = (hp == 0) ? m_run[1] : m_run[3];
            mn[0] = fmaxf(mo0, b0);
            mn[1] = fmaxf(mo1, b1);
            p[0] = (mn[0] == -INFINITY) ? 0.f : exp2f(s0 - mn[0]);
            p[1] = (mn[1] == -INFINITY) ? 0.f : exp2f(s1 - mn[1]);
            float ps0 = p[0], ps1 = p[1];
#pragma unroll
            for (int mm = 2; mm <= 16; mm <<= 1) {
                ps0 += __shfl_xor_sync(kFull, ps0, mm);
                ps1 += __shfl_xor_sync(kFull, ps1, mm);
            }
            // every lane: new max and chunk sum of all four heads
            float mnew[4], psum[4];
            mnew[0] = __shfl_sync(kFull, mn[0], 0);
            mnew[1] = __shfl_sync(kFull, mn[1], 0);
            mnew[2] = __shfl_sync(kFull, mn[0], 1);
            mnew[3] = __shfl_sync(kFull, mn[1], 1);
            psum[0] = __shfl_sync(kFull, ps0, 0);
            psum[1] = __shfl_sync(kFull, ps1, 0);
            psum[2] = __shfl_sync(kFull, ps0, 1);
            psum[3] = __shfl_sync(kFull, ps1, 1);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float al = (m_run[h] == -INFINITY) ? 0.f : exp2f(m_run[h] - mnew[h]);
                l_run[h] = l_run[h] * al + psum[h];
#pragma unroll
                for (int k = 0; k < 4; ++k) O[h][k] *= al;
                m_run[h] = mnew[h];
            }
#pragma unroll
            for (int t = 0; t < kChunk; ++t) {
                if (t >= nvalid) break;   // rows past the length may hold anything
                const uint2 vu = *reinterpret_cast<const uint2*>(Vc + t * kD * 2 + 8 * lane);
                const float v0 = __uint_as_float(vu.x << 16), v1 = __uint_as_float(vu.x & 0xffff0000u);
                const float v2 = __uint_as_float(vu.y << 16), v3 = __uint_as_float(vu.y & 0xffff0000u);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float ph = __shfl_sync(kFull, p[h & 1], 2 * t + (h >> 1));
                    O[h][0] = fmaf(ph, v0, O[h][0]);
                    O[h][1] = fmaf(ph, v1, O[h][1]);
                    O[h][2] = fmaf(ph, v2, O[h][2]);
                    O[h][3] = fmaf(ph, v3, O[h][3]);
                }
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

size_t attn_bf16_smem_bytes() { return (size_t)kBfStages * 2 * kChunkBytes + 64; }

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
    AttnArgs a;
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
    a.n_q = cfg.n_q_heads;
    a.n_kv = cfg.n_kv_heads;
    a.G = cfg.n_q_heads / cfg.n_kv_heads;
    a.nw = nw;
    a.sm_scale = cfg.sm_scale;
    for (int i = 0; i < 4; ++i) a.sb[i] = cfg.sign_bits[i];
    const unsigned mgrid = (unsigned)(((int64_t)batch * a.n_q + 3) / 4);
    if (cfg.block_size == 32)
        decode_attn_bf16_kernel<32><<<nw, 32, attn_bf16_smem_bytes(), st>>>(a);
    else
        decode_attn_bf16_kernel<64><<<nw, 32, attn_bf16_smem_bytes(), st>>>(a);
    merge_kernel<kChunk, false><<<mgrid, 128, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kvarn
