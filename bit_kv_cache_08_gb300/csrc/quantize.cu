// quantize.cu -- KVarN quantise-on-write (bulk and fused into the decode-step
// KV append) and dequantisation, hand-written for sm_103a.
//
// Method: abstract of "KVarN: cuantizacion de KV-Cache normalizada por
// varianza mitiga la acumulacion de errores en tareas de razonamiento"
// (Hadamard rotation, then dual-scaling variance normalisation over both axes
// of K and V, 2-bit) and "KVarN：方差归一化让 2-bit KV 缓存扛住长链推理"
// section 三 3.1 (randomised Hadamard) and 3.2 (token axis then channel axis
// to variance 1, repeated; grouped scales kept for dequantisation; computed
// at decode time inside the KV write kernel).
//
// One CTA of 8B threads (B/4 warps) owns one head-block of B tokens x 128
// channels. Warp w holds tokens 4w .. 4w+3, lane l channels 4l..4l+3, all in
// registers:
//   rotation   sign flip + FWHT-128 (2 in-register + 5 shuffle stages), *1/sqrt(128)
//   VarN       each pass sets a factor from the rotated tile directly: scaling a
//              row by a constant scales its spread by the same constant, so after
//              a token pass R_t = std_c(x_rot[t][c] / C_c) and after a channel
//              pass C_c = std_t(x_rot[t][c] / R_t) -- the values the pages'
//              divide-and-accumulate iteration reaches, without keeping the
//              normalised tile. Token pass: two-pass mean/variance by warp
//              reduction; channel pass: per-warp partial sums through shared memory
//   factors    sqrt(v) as v * rsqrt(v) (a few fp32 ulps; the factors only feed
//              statistics and an fp16 rounding), then fp16 round-to-nearest of
//              the clamped factors
//   quantise   y = x_rot * (1/R16) * (1/C16) (correctly rounded reciprocals;
//              a few fp32 ulps from the quotient), per (token, 32-channel group):
//              z = fp16 round-down of the
//              minimum, s = least fp16 with z + L s >= maximum, L = 2^bits - 1
//              (directed-rounding candidate plus one exact check), code = nearest
//              level, ties even (3 compares at 2 bits, a 4-step binary search
//              over the 15 boundaries at 4 bits)
//   pack       codes OR-ed into the shared-memory image of the head-block in
//              the attention kernel's record order, then 16-byte stores.
#include "common.cuh"

namespace kvarn {

constexpr int kRowsPerWarp = 4;
template <int B> constexpr int quant_warps() { return B / kRowsPerWarp; }
template <int B> constexpr int quant_threads() { return 32 * quant_warps<B>(); }

template <int B, int BITS>
struct QuantSmem {
    alignas(16) uint8_t image[head_block_bytes(B, BITS)];   // exact global layout
    alignas(16) float part[quant_warps<B>()][kD + 4]; // per-warp column partial sums (padded rows)
    alignas(16) float tot[2][kD];                     // column totals (double-buffered)
};

// Sums over the tile's rows of one value per (row, channel), given each
// thread's partial over its warp's rows for channels 4 lane .. 4 lane + 3.
// Warp w reduces channels [w*CPW, (w+1)*CPW) over all warps (4 shared loads
// per thread plus a shuffle tree), then every thread reads back its 4 totals.
// `buf` alternates between calls so that one barrier per call suffices.
template <int B, int BITS>
__device__ __forceinline__ float4 column_totals(QuantSmem<B, BITS>& q, const float (&cs)[4], int warp, int lane,
                                                int buf) {
    constexpr int NW = quant_warps<B>(), CPW = kD / NW, SUB = 32 / CPW;   // SUB warp subsets of 4 warps
    *reinterpret_cast<float4*>(&q.part[warp][4 * lane]) = make_float4(cs[0], cs[1], cs[2], cs[3]);
    __syncthreads();
    const int c = warp * CPW + (lane % CPW), sub = lane / CPW;
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < NW / SUB; ++k) t += q.part[sub * (NW / SUB) + k][c];
#pragma unroll
    for (int m = CPW; m < 32; m <<= 1) t += __shfl_xor_sync(kFull, t, m);
    if (sub == 0) q.tot[buf][c] = t;
    __syncthreads();
    return *reinterpret_cast<const float4*>(&q.tot[buf][4 * lane]);
}

// Row sums of a warp's rows at once (v[i]: this lane's partial of row i): a
// transposing butterfly leaves each lane with the total of one row (selected
// by its top lane bits), then one shuffle per row hands every lane all totals.
template <int RPW>
__device__ __forceinline__ void row_totals(float (&v)[RPW], int lane) {
    static_assert(RPW == 2 || RPW == 4, "two or four rows per warp");
    float k;
    if constexpr (RPW == 4) {
        const bool u16 = lane & 16, u8 = lane & 8;
        float k0 = u16 ? v[2] : v[0], k1 = u16 ? v[3] : v[1];
        const float s0 = u16 ? v[0] : v[2], s1 = u16 ? v[1] : v[3];
        k0 += __shfl_xor_sync(kFull, s0, 16);
        k1 += __shfl_xor_sync(kFull, s1, 16);
        k = u8 ? k1 : k0;
        const float s = u8 ? k0 : k1;
        k += __shfl_xor_sync(kFull, s, 8);
    } else {
        const bool u16 = lane & 16;
        k = u16 ? v[1] : v[0];
        const float s = u16 ? v[0] : v[1];
        k += __shfl_xor_sync(kFull, s, 16);
        k += __shfl_xor_sync(kFull, k, 8);
    }
    k += __shfl_xor_sync(kFull, k, 4);
    k += __shfl_xor_sync(kFull, k, 2);
    k += __shfl_xor_sync(kFull, k, 1);
#pragma unroll
    for (int i = 0; i < RPW; ++i) v[i] = __shfl_sync(kFull, k, (32 / RPW) * i);
}

struct QuantParams {
    int kind;          // 0 = K record order, 1 = V record order
    int iters;
    uint32_t flags;    // KVARN_FLAG_* ablation switches
    uint32_t sb[4];    // rotation signs
};

// A variance that is zero up to rounding (v <= 2^-30 mu^2), not positive or
// not finite leaves its row/column factor unchanged (a constant column keeps C).
// (v > 2^-30 mu^2 already rules out v <= 0, and a NaN fails both comparisons.)
__device__ __forceinline__ bool usable_variance(float v, float mu) {
    return v > 0x1p-30f * (mu * mu) && v < INFINITY;
}

// Least fp16 s >= 0 with z + L s >= M (L = 2^bits - 1 steps), for fp16 z <= M
// (all exact comparisons).
template <int L>
__device__ __forceinline__ float step_for(float zf, float M) {
    static_assert(L == 3 || L == 7 || L == 15, "2-, 3- or 4-bit codes");
    if (zf >= M) return 0.0f;
    // >= exact (M - z)/L: every step rounds up; RU(1/3) = 0x1.555556p-2f,
    // RU(1/7) = 0x1.24924ap-3f, RU(1/15) = 0x1.111112p-4f
    constexpr float kInvL = L == 3 ? 0x1.555556p-2f : (L == 7 ? 0x1.24924ap-3f : 0x1.111112p-4f);
    float t = __fmul_ru(__fsub_ru(M, zf), kInvL);
    __half s = __float2half_ru(t);                         // >= exact minimum
    float sf = __half2float(s);
    if (!(sf <= kF16Max)) { s = __float2half_rn(kF16Max); sf = kF16Max; }
    // the directed roundings may overshoot by one fp16 step: check the one below
    uint16_t bits = __half_as_ushort(s);
    if (bits > 0) {
        float pf = __half2float(__ushort_as_half((uint16_t)(bits - 1)));
        if (__fadd_rd(zf, (float)L * pf) >= M) sf = pf;     // L pf exact; rd-sum >= M <=> exact sum >= M
    }
    return sf;
}

// Quantise the tile held in x (rows of this warp) into q.image.
// fwht128 with the five cross-lane butterfly stages as packed fp32 pairs: the
// same operations on every value (bit-identical), fewer instructions
__device__ __forceinline__ void fwht128_x2(float (&v)[4], int lane) {
    float a0 = v[0] + v[1], a1 = v[0] - v[1];
    float a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2; v[2] = a0 - a2;
    v[1] = a1 + a3; v[3] = a1 - a3;
#pragma unroll
    for (int m = 1; m <= 16; m <<= 1) {
        const float sgn = (lane & m) ? -1.0f : 1.0f;
        const float2 s2 = make_float2(sgn, sgn);
        const float2 o01 = make_float2(__shfl_xor_sync(kFull, v[0], m), __shfl_xor_sync(kFull, v[1], m));
        const float2 o23 = make_float2(__shfl_xor_sync(kFull, v[2], m), __shfl_xor_sync(kFull, v[3], m));
        const float2 r01 = __ffma2_rn(s2, make_float2(v[0], v[1]), o01);
        const float2 r23 = __ffma2_rn(s2, make_float2(v[2], v[3]), o23);
        v[0] = r01.x; v[1] = r01.y; v[2] = r23.x; v[3] = r23.y;
    }
}

template <int B, int BITS>
__device__ void quantize_tile(float (&x)[kRowsPerWarp][4], const QuantParams& p, QuantSmem<B, BITS>& q,
                              int warp, int lane) {
    constexpr int RPW = kRowsPerWarp, NW = quant_warps<B>();
    uint32_t* words = reinterpret_cast<uint32_t*>(q.image);
    uint16_t* s_sec = reinterpret_cast<uint16_t*>(q.image + off_s(B, BITS));
    uint16_t* z_sec = reinterpret_cast<uint16_t*>(q.image + off_z(B, BITS));
    uint16_t* R_sec = reinterpret_cast<uint16_t*>(q.image + off_R(B, BITS));
    uint16_t* C_sec = reinterpret_cast<uint16_t*>(q.image + off_C(B, BITS));

    // ---- rotation: x_rot = H (sigma . x) / sqrt(128) (identity in the no-rotation ablation)
    uint32_t sw = p.sb[lane >> 3] >> (4 * (lane & 7));    // this lane's 4 sign bits
    const bool rotate = !(p.flags & KVARN_FLAG_NO_ROTATION);
#pragma unroll
    for (int i = 0; i < RPW && rotate; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) x[i][k] = ((sw >> k) & 1u) ? -x[i][k] : x[i][k];
        fwht128_x2(x[i], lane);
        const float2 r2 = make_float2(kInvSqrtD, kInvSqrtD);
        const float2 a = __fmul2_rn(make_float2(x[i][0], x[i][1]), r2), b = __fmul2_rn(make_float2(x[i][2], x[i][3]), r2);
        x[i][0] = a.x; x[i][1] = a.y; x[i][2] = b.x; x[i][3] = b.y;
    }

    // ---- VarN: token pass then channel pass, p.iters times
    float Rf[RPW], rR[RPW], Cf[4] = {1.f, 1.f, 1.f, 1.f}, rCf[4] = {1.f, 1.f, 1.f, 1.f};
#pragma unroll
    for (int i = 0; i < RPW; ++i) { Rf[i] = 1.f; rR[i] = 1.f; }
    int buf = 0;
    for (int it = 0; it < p.iters; ++it) {
        // token pass: R_t = population std over channels of x_rot[t][c] / C_c
        if (!(p.flags & KVARN_FLAG_NO_TOKEN_PASS)) {
            float2 u[RPW][2];   // channels (0, 1), (2, 3) of this lane's 4
            float mu[RPW], var[RPW];
            const float2 rc01 = make_float2(rCf[0], rCf[1]), rc23 = make_float2(rCf[2], rCf[3]);
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                u[i][0] = __fmul2_rn(make_float2(x[i][0], x[i][1]), rc01);
                u[i][1] = __fmul2_rn(make_float2(x[i][2], x[i][3]), rc23);
                mu[i] = (u[i][0].x + u[i][0].y) + (u[i][1].x + u[i][1].y);
            }
            row_totals<RPW>(mu, lane);
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                // every product, sum and multiply-add of the statistics is an explicit
                // fp32 operation (packed in pairs where the channels pair up): nothing is
                // left for the compiler to contract, so the bytes are the same in every
                // kernel and build
                mu[i] = __fmul_rn(mu[i], 1.0f / kD);
                const float2 nmu = make_float2(-mu[i], -mu[i]);
                const float2 d01 = __fadd2_rn(u[i][0], nmu), d23 = __fadd2_rn(u[i][1], nmu);
                const float d0 = d01.x, d1 = d01.y, d2 = d23.x, d3 = d23.y;
                var[i] = fmaf(d0, d0, __fmul_rn(d1, d1)) + fmaf(d2, d2, __fmul_rn(d3, d3));
            }
            row_totals<RPW>(var, lane);
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const float v = __fmul_rn(var[i], 1.0f / kD);
                const float r = rsqrtf(v);    // within 2 ulp; the factor is rounded to fp16 below
                const bool ok = usable_variance(v, mu[i]);
                rR[i] = ok ? r : rR[i];
                Rf[i] = ok ? v * r : Rf[i];
            }
        }
        if (p.flags & KVARN_FLAG_NO_CHANNEL_PASS) continue;   // (uniform over the CTA)
        // channel pass: C_c = population std over tokens of x_rot[t][c] / R_t
        float cs[4];
        {
            float2 c01 = make_float2(0.f, 0.f), c23 = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const float2 r2 = make_float2(rR[i], rR[i]);
                c01 = __ffma2_rn(make_float2(x[i][0], x[i][1]), r2, c01);
                c23 = __ffma2_rn(make_float2(x[i][2], x[i][3]), r2, c23);
            }
            cs[0] = c01.x; cs[1] = c01.y; cs[2] = c23.x; cs[3] = c23.y;
        }
        const float4 m4 = column_totals<B, BITS>(q, cs, warp, lane, buf);
        buf ^= 1;
        const float cmu[4] = {__fmul_rn(m4.x, 1.0f / B), __fmul_rn(m4.y, 1.0f / B), __fmul_rn(m4.z, 1.0f / B),
                              __fmul_rn(m4.w, 1.0f / B)};
        {
            float2 c01 = make_float2(0.f, 0.f), c23 = make_float2(0.f, 0.f);
            const float2 n01 = make_float2(-cmu[0], -cmu[1]), n23 = make_float2(-cmu[2], -cmu[3]);
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const float2 r2 = make_float2(rR[i], rR[i]);
                const float2 d01 = __ffma2_rn(make_float2(x[i][0], x[i][1]), r2, n01);
                const float2 d23 = __ffma2_rn(make_float2(x[i][2], x[i][3]), r2, n23);
                c01 = __ffma2_rn(d01, d01, c01);
                c23 = __ffma2_rn(d23, d23, c23);
            }
            cs[0] = c01.x; cs[1] = c01.y; cs[2] = c23.x; cs[3] = c23.y;
        }
        const float4 v4 = column_totals<B, BITS>(q, cs, warp, lane, buf);
        buf ^= 1;
        const float cvar[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float vk = __fmul_rn(cvar[k], 1.0f / B);
            const float r = rsqrtf(vk);
            const bool ok = usable_variance(vk, cmu[k]);
            rCf[k] = ok ? r : rCf[k];
            Cf[k] = ok ? vk * r : Cf[k];
        }
    }

    // ---- fp16 factors (clamped to the normal range) and normalised values
    float C16[4], rC[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        C16[k] = __half2float(__float2half_rn(fminf(fmaxf(Cf[k], kF16MinNormal), kF16Max)));
        rC[k] = __frcp_rn(C16[k]);
    }
    const int g = lane >> 3;   // this lane's 32-channel group
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int t = warp * RPW + i;
        const float R16 = __half2float(__float2half_rn(fminf(fmaxf(Rf[i], kF16MinNormal), kF16Max)));
        const float rRq = __frcp_rn(R16);
        float yq[4];
        {
            const float2 r2 = make_float2(rRq, rRq);
            const float2 y01 = __fmul2_rn(__fmul2_rn(make_float2(x[i][0], x[i][1]), r2), make_float2(rC[0], rC[1]));
            const float2 y23 = __fmul2_rn(__fmul2_rn(make_float2(x[i][2], x[i][3]), r2), make_float2(rC[2], rC[3]));
            yq[0] = y01.x; yq[1] = y01.y; yq[2] = y23.x; yq[3] = y23.y;
        }
        float mn = fminf(fminf(yq[0], yq[1]), fminf(yq[2], yq[3]));
        float mx = fmaxf(fmaxf(yq[0], yq[1]), fmaxf(yq[2], yq[3]));
#pragma unroll
        for (int m = 1; m <= 4; m <<= 1) {
            mn = fminf(mn, __shfl_xor_sync(kFull, mn, m));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, m));
        }
        const __half zh = __float2half_rd(fminf(fmaxf(mn, -kF16Max), kF16Max));
        const float zf = __half2float(zh);
        const float sf = step_for<(1 << BITS) - 1>(zf, mx);
        uint32_t code[4];
        if (sf == 0.0f) {
            code[0] = code[1] = code[2] = code[3] = 0u;
        } else if (BITS == 2) {
            const float b0 = zf + 0.5f * sf, b1 = zf + 1.5f * sf, b2 = zf + 2.5f * sf;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                code[k] = (uint32_t)(yq[k] > b0) + (uint32_t)(yq[k] >= b1) + (uint32_t)(yq[k] > b2);
        } else {
            // binary search over the 2^BITS - 1 boundaries z + (c - 1/2) s (each one
            // fma, rounded once like the 2-bit ones); a tie goes to the even level,
            // so the candidate steps above 1 (even candidates) test >=, step 1 tests >
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t c = 0;
#pragma unroll
                for (int st = 1 << (BITS - 1); st >= 1; st >>= 1) {
                    const float b = fmaf((float)(c + st) - 0.5f, sf, zf);
                    const bool up = (st == 1) ? (yq[k] > b) : (yq[k] >= b);
                    c = up ? c + st : c;
                }
                code[k] = c;
            }
        }
        // ---- pack into the record order of this kind
        const int sb = t >> 5;
        if (BITS == 3) {
            // low two bits at the 2-bit positions of a 12-word record, the high bit
            // in the record's 1-bit plane: word 8 + w2/2, bit 8(w2%2) + j + 16h
            if (p.kind == KVARN_KIND_K) {   // w2 = 2i + g/2, j = 4(g%2) + e/2, h = e%2
                const int a = (t & 31) >> 2, ii = t & 3, bq = (lane & 7) >> 1, eh = lane & 1;
                const int rec = 32 * sb + 4 * a + bq;
                uint32_t lo = 0, hi = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int e = 4 * eh + k, j = 4 * (g & 1) + (e >> 1), h = e & 1;
                    lo |= (code[k] & 3u) << (2 * j + 16 * h);
                    hi |= (code[k] >> 2) << (8 * (g >> 1) + j + 16 * h);
                }
                atomicOr(&words[rec * 12 + 2 * ii + (g >> 1)], lo);
                atomicOr(&words[rec * 12 + 8 + ii], hi);
            } else {                        // w2 = 2g + f/2, j = 4(d/4) + 2((d%4)/2) + f%2, h = d%2
                const int a = lane & 7, bq = (t & 31) >> 3, d = t & 7;
                const int rec = 32 * sb + 4 * a + bq;
                const int jb = 4 * (d >> 2) + 2 * ((d & 3) >> 1), h = d & 1;
                uint32_t hi = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) hi |= (code[k] >> 2) << (8 * (k >> 1) + jb + (k & 1) + 16 * h);
                atomicOr(&words[rec * 12 + 2 * g + 0],
                         ((code[0] & 3u) << (2 * jb + 16 * h)) | ((code[1] & 3u) << (2 * jb + 2 + 16 * h)));
                atomicOr(&words[rec * 12 + 2 * g + 1],
                         ((code[2] & 3u) << (2 * jb + 16 * h)) | ((code[3] & 3u) << (2 * jb + 2 + 16 * h)));
                atomicOr(&words[rec * 12 + 8 + g], hi);
            }
        } else if (BITS == 4) {
            if (p.kind == KVARN_KIND_K) {   // word 4i + g, bit 4(e/2) + 16(e%2)
                const int a = (t & 31) >> 2, ii = t & 3, bq = (lane & 7) >> 1, eh = lane & 1;
                uint32_t contrib = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int e = 4 * eh + k;
                    contrib |= code[k] << (4 * (e >> 1) + 16 * (e & 1));
                }
                atomicOr(&words[(32 * sb + 4 * a + bq) * 16 + 4 * ii + g], contrib);
            } else {                        // word 4g + f, bit 4(d/2) + 16(d%2)
                const int a = lane & 7, bq = (t & 31) >> 3, d = t & 7;
                const int rec = 32 * sb + 4 * a + bq, bit = 4 * (d >> 1) + 16 * (d & 1);
#pragma unroll
                for (int k = 0; k < 4; ++k) atomicOr(&words[rec * 16 + 4 * g + k], code[k] << bit);
            }
        } else if (p.kind == KVARN_KIND_K) {
            const int a = (t & 31) >> 2, ii = t & 3, bq = (lane & 7) >> 1, eh = lane & 1;
            const int word = (32 * sb + 4 * a + bq) * 8 + 2 * ii + (g >> 1);
            uint32_t contrib = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int e = 4 * eh + k;
                contrib |= code[k] << (2 * (4 * (g & 1) + (e >> 1)) + 16 * (e & 1));
            }
            atomicOr(&words[word], contrib);
        } else {
            const int a = lane & 7, bq = (t & 31) >> 3, d = t & 7;
            const int rec = 32 * sb + 4 * a + bq;
            const int base = 2 * (4 * (d >> 2) + 2 * ((d & 3) >> 1)) + 16 * (d & 1);
            atomicOr(&words[rec * 8 + 2 * g + 0], (code[0] << base) | (code[1] << (base + 2)));
            atomicOr(&words[rec * 8 + 2 * g + 1], (code[2] << base) | (code[3] << (base + 2)));
        }
        if ((lane & 7) == 0) {
            s_sec[g * B + t] = __half_as_ushort(__float2half_rn(sf));   // sf is an fp16 value
            z_sec[g * B + t] = __half_as_ushort(zh);
        }
        if (lane == 0) R_sec[t] = __half_as_ushort(__float2half_rn(R16));
    }
    if (warp == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) C_sec[4 * lane + k] = __half_as_ushort(__float2half_rn(C16[k]));
    }
    __syncthreads();
}

template <int B, int BITS>
__device__ __forceinline__ void zero_code_words(QuantSmem<B, BITS>& q, int tid) {
    uint32_t* words = reinterpret_cast<uint32_t*>(q.image);
    for (int i = tid; i < B * 4 * BITS; i += quant_threads<B>()) words[i] = 0u;
}

template <int B, int BITS>
__device__ __forceinline__ void store_image(const QuantSmem<B, BITS>& q, uint8_t* dst, int tid) {
    const uint4* src = reinterpret_cast<const uint4*>(q.image);
    uint4* d = reinterpret_cast<uint4*>(dst);
    for (int i = tid; i < head_block_bytes(B, BITS) / 16; i += quant_threads<B>()) d[i] = src[i];
}

__device__ __forceinline__ void load4(const void* src, int dtype, int64_t elem_off, float (&v)[4]) {
    if (dtype == KVARN_FP32) {
        float4 f = *reinterpret_cast<const float4*>(static_cast<const float*>(src) + elem_off);
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    } else {
        uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(src) + elem_off);
        v[0] = __uint_as_float(u.x << 16);
        v[1] = __uint_as_float(u.x & 0xffff0000u);
        v[2] = __uint_as_float(u.y << 16);
        v[3] = __uint_as_float(u.y & 0xffff0000u);
    }
}

// ---------------------------------------------------------------- bulk quantise
template <int B, int BITS>
__global__ void __launch_bounds__(quant_threads<B>(), 3) quantize_blocks_kernel(
    const void* __restrict__ src, int dtype, int64_t block_stride, int64_t token_stride,
    uint8_t* __restrict__ dst_base, const int64_t* __restrict__ dst_offsets, QuantParams p,
    uint32_t* err) {
    wait_prior_grids();
    __shared__ QuantSmem<B, BITS> q;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n = blockIdx.x;
    zero_code_words<B, BITS>(q, tid);
    float x[kRowsPerWarp][4];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int t = warp * kRowsPerWarp + i;
        load4(src, dtype, n * block_stride + (int64_t)t * token_stride + 4 * lane, x[i]);
#pragma unroll
        for (int k = 0; k < 4; ++k) bad |= !isfinite(x[i][k]);
    }
    if (__syncthreads_or(bad) && tid == 0) raise_error(err, KVARN_DEVERR_NONFINITE);
    quantize_tile<B, BITS>(x, p, q, warp, lane);
    const int64_t off = dst_offsets ? dst_offsets[n] : n * (int64_t)head_block_bytes(B, BITS);
    store_image<B, BITS>(q, dst_base + off, tid);
}

// ---------------------------------------------------------------- fused append
// grid (batch, n_kv, 2): one CTA per (sequence, kv head, K|V).
template <int B, int BITS>
__global__ void __launch_bounds__(quant_threads<B>(), 3) append_kernel(
    uint8_t* __restrict__ pool, int64_t n_pool_blocks, int64_t block_bytes,
    uint16_t* __restrict__ staging, const int32_t* __restrict__ block_table, int max_blocks,
    const int32_t* __restrict__ pos_arr, const uint16_t* __restrict__ k_new,
    const uint16_t* __restrict__ v_new, int n_kv, QuantParams p, uint32_t* err) {
    wait_prior_grids();
    __shared__ QuantSmem<B, BITS> q;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x, h = blockIdx.y, kv = blockIdx.z;
    const int pos = pos_arr[b];
    if (pos < 0 || pos >= max_blocks * B) {
        if (tid == 0 && h == 0 && kv == 0) raise_error(err, KVARN_DEVERR_POSITION);
        return;
    }
    const int row = pos % B;
    const uint16_t* newrow = (kv ? v_new : k_new) + ((int64_t)b * n_kv + h) * kD;
    uint16_t* stage = staging + (((int64_t)b * n_kv + h) * 2 + kv) * B * kD;
    if (tid < 16)   // 256 bytes, 16 per thread
        reinterpret_cast<uint4*>(stage + row * kD)[tid] = reinterpret_cast<const uint4*>(newrow)[tid];
    if (row != B - 1) return;

    const int64_t phys = block_table[(int64_t)b * max_blocks + pos / B];
    if (phys < 0 || phys >= n_pool_blocks) {
        if (tid == 0) raise_error(err, KVARN_DEVERR_BLOCK_ID);
        return;
    }
    p.kind = kv;
    zero_code_words<B, BITS>(q, tid);
    float x[kRowsPerWarp][4];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int t = warp * kRowsPerWarp + i;
        const uint16_t* r = (t == B - 1) ? newrow : stage + t * kD;
        load4(r, KVARN_BF16, 4 * lane, x[i]);
#pragma unroll
        for (int k = 0; k < 4; ++k) bad |= !isfinite(x[i][k]);
    }
    if (__syncthreads_or(bad) && tid == 0) raise_error(err, KVARN_DEVERR_NONFINITE);
    quantize_tile<B, BITS>(x, p, q, warp, lane);
    store_image<B, BITS>(q, pool + phys * block_bytes + (int64_t)(2 * h + kv) * head_block_bytes(B, BITS), tid);
}

// ---------------------------------------------------------------- dequantise
// Token row t of a head-block image in shared memory: this lane's 4 channels
// 4 lane .. 4 lane + 3 of (code*s + z)*R*C (rotated space).
template <int B, int BITS>
__device__ __forceinline__ void dequant_row4(const uint8_t* img, int kind, int t, int lane, float (&v)[4]) {
    const uint32_t* words = reinterpret_cast<const uint32_t*>(img);
    const uint16_t* s_sec = reinterpret_cast<const uint16_t*>(img + off_s(B, BITS));
    const uint16_t* z_sec = reinterpret_cast<const uint16_t*>(img + off_z(B, BITS));
    const uint16_t* R_sec = reinterpret_cast<const uint16_t*>(img + off_R(B, BITS));
    const uint16_t* C_sec = reinterpret_cast<const uint16_t*>(img + off_C(B, BITS));
    const int g = lane >> 3, sb = t >> 5;
    const float s = h2f(s_sec[g * B + t]), z = h2f(z_sec[g * B + t]), R = h2f(R_sec[t]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int c = 4 * lane + k;
        int word, bit;
        if (BITS == 3) {   // low two bits in the 2-bit layout, the high bit in the 1-bit plane
            int rec, w2, j, h;
            if (kind == KVARN_KIND_K) {
                const int a = (t & 31) >> 2, ii = t & 3, bq = (c & 31) >> 3, e = c & 7;
                rec = 32 * sb + 4 * a + bq;
                w2 = 2 * ii + (g >> 1);
                j = 4 * (g & 1) + (e >> 1);
                h = e & 1;
            } else {
                const int bq = (t & 31) >> 3, d = t & 7, a = (c & 31) >> 2, f = c & 3;
                rec = 32 * sb + 4 * a + bq;
                w2 = 2 * g + (f >> 1);
                j = 4 * (d >> 2) + 2 * ((d & 3) >> 1) + (f & 1);
                h = d & 1;
            }
            const uint32_t lo = (words[rec * 12 + w2] >> (2 * j + 16 * h)) & 3u;
            const uint32_t hb = (words[rec * 12 + 8 + (w2 >> 1)] >> (8 * (w2 & 1) + j + 16 * h)) & 1u;
            v[k] = fmaf((float)(lo | (hb << 2)), s, z) * R * h2f(C_sec[c]);
            continue;
        }
        if (kind == KVARN_KIND_K) {
            const int a = (t & 31) >> 2, ii = t & 3, bq = (c & 31) >> 3, e = c & 7;
            if (BITS == 4) {
                word = (32 * sb + 4 * a + bq) * 16 + 4 * ii + g;
                bit = 4 * (e >> 1) + 16 * (e & 1);
            } else {
                word = (32 * sb + 4 * a + bq) * 8 + 2 * ii + (g >> 1);
                bit = 2 * (4 * (g & 1) + (e >> 1)) + 16 * (e & 1);
            }
        } else {
            const int bq = (t & 31) >> 3, d = t & 7, a = (c & 31) >> 2, f = c & 3;
            if (BITS == 4) {
                word = (32 * sb + 4 * a + bq) * 16 + 4 * g + f;
                bit = 4 * (d >> 1) + 16 * (d & 1);
            } else {
                word = (32 * sb + 4 * a + bq) * 8 + 2 * g + (f >> 1);
                bit = 2 * (4 * (d >> 2) + 2 * ((d & 3) >> 1) + (f & 1)) + 16 * (d & 1);
            }
        }
        const float code = (float)((words[word] >> bit) & ((1u << BITS) - 1u));
        v[k] = fmaf(code, s, z) * R * h2f(C_sec[c]);
    }
}

template <int B, int BITS>
__device__ __forceinline__ void load_image(uint8_t* img, const uint8_t* src, int tid) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    for (int i = tid; i < head_block_bytes(B, BITS) / 16; i += 256) reinterpret_cast<uint4*>(img)[i] = s4[i];
}

template <int B, int BITS>
__global__ void __launch_bounds__(256) dequantize_kernel(
    const uint8_t* __restrict__ src_base, const int64_t* __restrict__ src_offsets, int kind,
    int rotated, QuantParams p, float* __restrict__ out) {
    wait_prior_grids();
    __shared__ alignas(16) uint8_t img[head_block_bytes(B, BITS)];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n = blockIdx.x;
    const int64_t off = src_offsets ? src_offsets[n] : n * (int64_t)head_block_bytes(B, BITS);
    load_image<B, BITS>(img, src_base + off, tid);
    __syncthreads();
    for (int i = 0; i < B / 8; ++i) {
        const int t = warp * (B / 8) + i;
        float v[4];
        dequant_row4<B, BITS>(img, kind, t, lane, v);
        if (!rotated && !(p.flags & KVARN_FLAG_NO_ROTATION)) {
            fwht128(v, lane);
#pragma unroll
            for (int k = 0; k < 4; ++k) v[k] *= kInvSqrtD * sign_of(p.sb, 4 * lane + k);
        }
        *reinterpret_cast<float4*>(out + (n * B + t) * kD + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
    }
}

// ---------------------------------------------------------------- error decomposition
// Per token: (|x|, |x^|, |E_M|, |E_D|) with E_M = (|x^| - |x|) x/|x| and
// E_D = |x^| (x^/|x^| - x/|x|), x the values before quantisation and x^ the
// dequantised ones. Norms and the angle do not change under the rotation, so
// both are taken in the rotated space (x rotated like the quantiser does).
template <int B, int BITS>
__global__ void __launch_bounds__(256) error_split_kernel(
    const void* __restrict__ src, int dtype, int64_t block_stride, int64_t token_stride,
    const uint8_t* __restrict__ packed_base, const int64_t* __restrict__ packed_offsets, int kind,
    QuantParams p, float* __restrict__ out) {
    wait_prior_grids();
    __shared__ alignas(16) uint8_t img[head_block_bytes(B, BITS)];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n = blockIdx.x;
    const int64_t off = packed_offsets ? packed_offsets[n] : n * (int64_t)head_block_bytes(B, BITS);
    load_image<B, BITS>(img, packed_base + off, tid);
    __syncthreads();
    const uint32_t sw = p.sb[lane >> 3] >> (4 * (lane & 7));
    for (int i = 0; i < B / 8; ++i) {
        const int t = warp * (B / 8) + i;
        float x[4], xh[4];
        load4(src, dtype, n * block_stride + (int64_t)t * token_stride + 4 * lane, x);
        if (!(p.flags & KVARN_FLAG_NO_ROTATION)) {
#pragma unroll
            for (int k = 0; k < 4; ++k) x[k] = ((sw >> k) & 1u) ? -x[k] : x[k];
            fwht128(x, lane);
#pragma unroll
            for (int k = 0; k < 4; ++k) x[k] *= kInvSqrtD;
        }
        dequant_row4<B, BITS>(img, kind, t, lane, xh);
        const float nx = sqrtf(warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]));
        const float nh = sqrtf(warp_sum(xh[0] * xh[0] + xh[1] * xh[1] + xh[2] * xh[2] + xh[3] * xh[3]));
        float em, ed = 0.f;
        if (nx == 0.f) {
            em = nh;                 // direction undefined: all of the error is magnitude
        } else {
            em = fabsf(nh - nx);
            if (nh > 0.f) {
                const float ix = 1.0f / nx, ih = 1.0f / nh;
                float d = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float u = xh[k] * ih - x[k] * ix;
                    d = fmaf(u, u, d);
                }
                ed = nh * sqrtf(warp_sum(d));
            }
        }
        if (lane == 0) *reinterpret_cast<float4*>(out + (n * B + t) * 4) = make_float4(nx, nh, em, ed);
    }
}

// ---------------------------------------------------------------- host launchers
static QuantParams make_params(const kvarn_config& cfg, int kind) {
    QuantParams p;
    p.kind = kind;
    p.iters = cfg.varn_iters;
    p.flags = cfg.flags;
    for (int i = 0; i < 4; ++i) p.sb[i] = cfg.sign_bits[i];
    return p;
}

// The (block size, code width) instantiation for a config: f(int_constant<B>, int_constant<BITS>).
template <int V> struct ic { static constexpr int value = V; };
template <typename F>
cudaError_t dispatch(const kvarn_config& cfg, F&& f) {
    if (cfg.block_size == 32)
        return cfg.bits == 4 ? f(ic<32>{}, ic<4>{}) : (cfg.bits == 3 ? f(ic<32>{}, ic<3>{}) : f(ic<32>{}, ic<2>{}));
    return cfg.bits == 4 ? f(ic<64>{}, ic<4>{}) : (cfg.bits == 3 ? f(ic<64>{}, ic<3>{}) : f(ic<64>{}, ic<2>{}));
}

cudaError_t launch_quantize_blocks(const kvarn_config& cfg, int kind, const void* src, int dtype,
                                   int64_t n, int64_t block_stride, int64_t token_stride,
                                   void* dst_base, const int64_t* dst_offsets, uint32_t* err,
                                   cudaStream_t st) {
    QuantParams p = make_params(cfg, kind);
    return dispatch(cfg, [&](auto b, auto w) {
        constexpr int B = decltype(b)::value, BITS = decltype(w)::value;
        return launch_pdl(quantize_blocks_kernel<B, BITS>, (unsigned)n, quant_threads<B>(), 0, st, src, dtype,
                          block_stride, token_stride, (uint8_t*)dst_base, dst_offsets, p, err);
    });
}

cudaError_t launch_append(const kvarn_config& cfg, void* pool, int64_t n_pool_blocks,
                          int64_t block_bytes, void* staging, const int32_t* block_table,
                          int max_blocks, const int32_t* pos, const void* k_new, const void* v_new,
                          int batch, uint32_t* err, cudaStream_t st) {
    QuantParams p = make_params(cfg, 0);
    const dim3 grid(batch, cfg.n_kv_heads, 2);
    return dispatch(cfg, [&](auto b, auto w) {
        constexpr int B = decltype(b)::value, BITS = decltype(w)::value;
        return launch_pdl(append_kernel<B, BITS>, grid, quant_threads<B>(), 0, st, (uint8_t*)pool, n_pool_blocks,
                          block_bytes, (uint16_t*)staging, block_table, max_blocks, pos, (const uint16_t*)k_new,
                          (const uint16_t*)v_new, cfg.n_kv_heads, p, err);
    });
}

cudaError_t launch_error_split(const kvarn_config& cfg, int kind, const void* src, int dtype, int64_t n,
                               int64_t block_stride, int64_t token_stride, const void* packed_base,
                               const int64_t* packed_offsets, float* out, cudaStream_t st) {
    QuantParams p = make_params(cfg, kind);
    return dispatch(cfg, [&](auto b, auto w) {
        constexpr int B = decltype(b)::value, BITS = decltype(w)::value;
        return launch_pdl(error_split_kernel<B, BITS>, (unsigned)n, 256, 0, st, src, dtype, block_stride,
                          token_stride, (const uint8_t*)packed_base, packed_offsets, kind, p, out);
    });
}

cudaError_t launch_dequantize(const kvarn_config& cfg, int kind, const void* src_base,
                              const int64_t* src_offsets, int64_t n, int rotated, float* out,
                              cudaStream_t st) {
    QuantParams p = make_params(cfg, kind);
    return dispatch(cfg, [&](auto b, auto w) {
        constexpr int B = decltype(b)::value, BITS = decltype(w)::value;
        return launch_pdl(dequantize_kernel<B, BITS>, (unsigned)n, 256, 0, st, (const uint8_t*)src_base,
                          src_offsets, kind, rotated, p, out);
    });
}

}  // namespace kvarn
