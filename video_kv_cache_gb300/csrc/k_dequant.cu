// Fused reconstruction: dequantize the final residual and add back every stage's
// assigned centroid in one pass, in registers.
//
// Method step: X^(T) = deQ(X_INT, S_x), then X^(t-1) = X^(t) + C^(t)_{pi_i} for t = T..1
// (review page "Quant VideoGen: 基于2-Bit KV缓存量化的自回归长视频生成", pipeline paragraph;
// "Quant VideoGen" notes page, sections Progressive Residual Quantization and
// Algorithm-System Co-design, the fused dequantization kernel).
//
// Design (HBM-bound for one or two stages; beyond that bound by the shared-memory reads of
// the tables, T fp32 values per output element):
//   * The T tables of a tensor are staged in shared memory one channel slice of W channels
//     at a time (T x C x W fp32; W is the widest of 128, 64 and 32 that fits 200 KB: 64
//     for T = 2, 32 for T = 4 with C = 256).  The S = 128 / W slices of a token range are
//     taken by S CTAs side by side: CTA b holds slice b % S and the (b / S)-th equal share
//     of the flattened (tensor, token) space, so the S CTAs of a share walk the same
//     tokens at about the same time, and the code, scale and index sectors they share come
//     from DRAM once (the others hit L2).  A CTA restages only when its share moves to
//     another tensor or centroid table.
//   * A lane rebuilds 16 contiguous channels of a token (four 4-channel chunks): one 4- or
//     8-byte code load, one scale byte (the 16 channels lie in one scale group) and T
//     cluster-index bytes, loaded two tokens ahead of the one being computed.
//   * Conflict-free table reads without a swizzle: the 8 lanes of a quarter-warp read 16
//     bytes each from up to 8 different table rows; a row's chunk c sits in bank group
//     c mod 8.  Lane (token q of the quarter, part u of the token) reads its four chunks in
//     the order k -> 4u + ((k + rot) mod 4), rot = (q * LPT / 2 + u / 2) mod 4 (LPT lanes
//     per token), so at every step the 8 lanes hit 8 different bank groups whatever rows
//     they read.  The codes are rotated the same way (a funnel shift), the arithmetic runs
//     in that order, and two rounds of selects put the results back in channel order before
//     the store.
//   * Arithmetic per element: the code u is masked in place into the mantissa of the float
//     2^23 (one logic op), one subtraction gives (u - 2^(b-1)) * 2^k exactly, and
//     y = fma(s_q * 2^-k, that, C^(T)) (s_q * q is exact, so this equals adding C^(T) to
//     the dequantized value); then one add per further stage, T - 1 down to 1, in fp32,
//     rounded once to the output type.  The subtraction, the fma and the adds run on f32x2
//     pairs of neighbouring channels (each half rounds as the scalar operation does).
//   * A lane writes its 16 outputs with one 32-byte store (two for fp32) when the output
//     is 32-byte aligned, so every store instruction fills whole sectors.
#include <cuda_fp8.h>

#include <algorithm>
#include <type_traits>

#include "internal.cuh"

namespace qvg {

namespace {
constexpr int kDqThreads = 1024;
constexpr size_t kDqTableBytes = 200 * 1024;  // largest table slice staged by one CTA

// 32-byte store (sm_100 and later), 32-byte aligned address.
__device__ __forceinline__ void st_v8(void *ptr, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3);
    return __half2float(__half(h));
}

__device__ __forceinline__ uint32_t sel(bool c, uint32_t a, uint32_t b) { return c ? a : b; }
}  // namespace

template <int BITS, int OUT, int TT, int SH>  // SH: 1 for the mid-rise grid, else 0
__global__ void __launch_bounds__(kDqThreads, 1)
    k_dequant(DPlan p, int W, int S, int64_t n_chunks, int smem_tables, int wide_stores) {
    pdl_begin();
    extern __shared__ __align__(16) float smem_f[];
    constexpr int MID = 1 << (BITS - 1);
    constexpr int PER16 = 16 / BITS;  // codes in a 16-bit half-word
    constexpr int OW = OUT == DT_F32 ? 4 : 2;  // output words per 4-channel chunk
    const int T = TT >= 0 ? TT : p.T;
    const int C = p.C;
    float *tab = smem_f;  // [T][C][W]
    constexpr int sh = SH;  // code shift of the level trick
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int LPT = W / 16;        // lanes per token
    const int TPW = 32 / LPT;      // tokens per warp and pass
    const int sub = lane % LPT;    // part of the token's slice
    const int tq = (lane & 7) / LPT;  // token within the quarter-warp
    const int rot = (tq * (LPT >> 1) + (sub >> 1)) & 3;
    const int tpc = (kDqThreads / 32) * TPW;  // tokens per CTA pass
    const int row_bytes = kD * BITS / 8;
    const int ngroups = kD / p.group;
    const int s = blockIdx.x % S;
    const int G = gridDim.x / S, g = blockIdx.x / S;
    const int ch0 = s * W + sub * 16;  // the lane's first channel
    // float offsets in a staged row of the chunk read at step k
    int roff[4];
#pragma unroll
    for (int k = 0; k < 4; k++) roff[k] = sub * 16 + 4 * ((k + rot) & 3);

    const int64_t total = (int64_t)p.H * p.N;
    const int64_t wb = total * g / G, we = total * (g + 1) / G;
    int64_t staged = -1;
    bool bad_index = false;

    for (int64_t pos = wb; pos < we;) {
        const int h = (int)(pos / p.N);
        const int64_t i0 = pos - (int64_t)h * p.N;
        const int64_t c = min(i0 / p.chunk_len, n_chunks - 1);
        // the chunk's tokens (the last chunk's run to N), within the share
        const int64_t i1 = min(min(p.N, (c + 1) * p.chunk_len), i0 + (we - pos));
        pos += i1 - i0;
        const int64_t hc = (int64_t)h * n_chunks + c;
        const float *tbl = p.cent + ((int64_t)h * p.n_tables + c) * T * C * kD;
        if (smem_tables && T > 0 && hc != staged) {
            __syncthreads();
            const int wq = W >> 2;
            const int nvec = T * C * wq;
            for (int x = tid; x < nvec; x += kDqThreads) {
                const int rr = x / wq, cc = x - rr * wq;
                reinterpret_cast<float4 *>(tab)[x] =
                    __ldg(reinterpret_cast<const float4 *>(tbl + (int64_t)rr * kD + s * W) + cc);
            }
            __syncthreads();
            staged = hc;
        }
        int64_t i = i0 + warp * TPW + lane / LPT;
        // running pointers of token i; they advance by tpc tokens per pass
        const uint8_t *cp = p.codes + ((int64_t)h * p.cap + i) * row_bytes + ch0 * BITS / 8;
        const uint8_t *sp = p.scales + ((int64_t)h * p.cap + i) * ngroups + ch0 / p.group;
        const uint8_t *pp = p.pi + (int64_t)h * T * p.cap + i;
        char *op = static_cast<char *>(p.out) +
                   ((int64_t)h * p.out_stride + i * kD + ch0) * (OUT == DT_F32 ? 4 : 2);
        const int64_t cstep = (int64_t)tpc * row_bytes, sstep = (int64_t)tpc * ngroups;
        const int64_t ostep = (int64_t)tpc * kD * (OUT == DT_F32 ? 4 : 2);
        int64_t poff[TT > 0 ? TT : 1];  // offsets of the stages' index planes
#pragma unroll
        for (int t = 0; t < (TT > 0 ? TT : 1); t++) poff[t] = (int64_t)t * p.cap;

        // cluster indices of up to four stages fit one word
        using PK = typename std::conditional<(TT >= 0 && TT <= 4), uint32_t, uint64_t>::type;
        struct Meta {
            uint32_t code[BITS / 2];  // 16 codes, channel 0 in the low bits
            uint32_t sbyte;
            PK pk;                    // pi^(1..T), one byte per stage
        };
        auto fetch = [&](Meta &m) {
            if constexpr (BITS == 2) {
                m.code[0] = __ldg(reinterpret_cast<const uint32_t *>(cp));
            } else {
                const uint2 v = __ldg(reinterpret_cast<const uint2 *>(cp));
                m.code[0] = v.x;
                m.code[1] = v.y;
            }
            m.sbyte = __ldg(sp);
            m.pk = 0;
            if (TT >= 0) {
#pragma unroll
                for (int t = 0; t < TT; t++) m.pk |= (PK)__ldg(pp + poff[t]) << (8 * t);
            } else {
                for (int t = 0; t < T; t++) m.pk |= (uint64_t)__ldg(pp + (int64_t)t * p.cap) << (8 * t);
            }
        };
        // a stored index >= C is reported and clamped (one compare per stage for the flag,
        // one min for the clamp)
        auto stage_j = [&](const Meta &m, int t) {
            const int j = (int)((m.pk >> (8 * t)) & 0xFFu);
            bad_index |= j >= C;
            return min(j, C - 1);
        };
        // stage-t centroid values of the lane's four chunks, cluster j, in read order
        auto table16 = [&](int t, int j, float4 (&a)[4]) {
            if (smem_tables) {
                const float *row = tab + (t * C + j) * W;
#pragma unroll
                for (int k = 0; k < 4; k++) a[k] = *reinterpret_cast<const float4 *>(row + roff[k]);
            } else {
                const float *row = tbl + ((int64_t)t * C + j) * kD + s * W;
#pragma unroll
                for (int k = 0; k < 4; k++) a[k] = __ldg(reinterpret_cast<const float4 *>(row + roff[k]));
            }
        };

        // two tokens of metadata in flight ahead of the one being computed
        Meta cur, nxt;
        if (i < i1) fetch(cur);
        cp += cstep;
        sp += sstep;
        pp += tpc;
        if (i + tpc < i1) fetch(nxt);
        while (i < i1) {
            const int64_t inext = i + tpc;
            Meta nxt2;
            cp += cstep;
            sp += sstep;
            pp += tpc;
            if (inext + tpc < i1) fetch(nxt2);
            // the codes in read order: chunk (k + rot) mod 4 at position k
            uint32_t cw[BITS / 2];
            if constexpr (BITS == 2) {
                cw[0] = __funnelshift_r(cur.code[0], cur.code[0], 8 * rot);
            } else {
                const uint32_t a0 = sel(rot & 2, cur.code[1], cur.code[0]);
                const uint32_t a1 = sel(rot & 2, cur.code[0], cur.code[1]);
                cw[0] = sel(rot & 1, __funnelshift_r(a0, a1, 16), a0);
                cw[1] = sel(rot & 1, __funnelshift_r(a1, a0, 16), a1);
            }
            // Code e of a 16-bit half-word sits at bits BITS*e; shifted left by sh (0, or 1
            // for the mid-rise grid) and kept inside the mantissa of 2^23, the float is
            // 2^23 + u * 2^(BITS*e + sh).  Subtracting 2^23 + (MID * 2^sh - sh) * 2^(BITS*e)
            // leaves (u * 2^sh - MID * 2^sh + sh) * 2^(BITS*e) exactly, and
            // sq * 2^-(BITS*e + sh) (exact: a power-of-two rescaling) turns it into the
            // level: sq * (u - MID), or sq * (u - MID + 1/2) for the mid-rise grid.
            const float sq = e4m3_to_float(cur.sbyte & 0xFFu);
            constexpr int NP = PER16 / 2;
            float2 se[NP], nk[NP];
#pragma unroll
            for (int e2 = 0; e2 < NP; e2++) {
                float s2[2], k2[2];
#pragma unroll
                for (int o = 0; o < 2; o++) {
                    const int e = 2 * e2 + o;
                    s2[o] = __fmul_rn(sq, __uint_as_float((uint32_t)(127 - BITS * e - sh) << 23));
                    k2[o] = -(__uint_as_float(0x4B000000u) + (float)(((MID << sh) - sh) << (BITS * e)));
                }
                se[e2] = make_float2(s2[0], s2[1]);
                nk[e2] = make_float2(k2[0], k2[1]);
            }
            // y[2k], y[2k + 1]: the four channels of the chunk read at step k
            float2 y[8];
#pragma unroll
            for (int hw = 0; hw < 16 / PER16; hw++) {
                const uint32_t word = (cw[hw >> 1] >> (16 * (hw & 1))) << sh;
#pragma unroll
                for (int e = 0; e < PER16; e += 2) {
                    const uint32_t m0 = (word & (((1u << BITS) - 1u) << (BITS * e + sh))) | 0x4B000000u;
                    const uint32_t m1 = (word & (((1u << BITS) - 1u) << (BITS * (e + 1) + sh))) | 0x4B000000u;
                    y[(hw * PER16 + e) / 2] =
                        __fadd2_rn(make_float2(__uint_as_float(m0), __uint_as_float(m1)), nk[e / 2]);
                }
            }
            if (T == 0) {
#pragma unroll
                for (int x = 0; x < 8; x++) y[x] = __fmul2_rn(se[x % NP], y[x]);
            } else {
                float4 a[4];
                table16(T - 1, stage_j(cur, T - 1), a);
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    y[2 * k] = __ffma2_rn(se[(2 * k) % NP], y[2 * k], make_float2(a[k].x, a[k].y));
                    y[2 * k + 1] = __ffma2_rn(se[(2 * k + 1) % NP], y[2 * k + 1], make_float2(a[k].z, a[k].w));
                }
                for (int t = T - 2; t >= 0; t--) {
                    table16(t, stage_j(cur, t), a);
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        y[2 * k] = __fadd2_rn(y[2 * k], make_float2(a[k].x, a[k].y));
                        y[2 * k + 1] = __fadd2_rn(y[2 * k + 1], make_float2(a[k].z, a[k].w));
                    }
                }
            }
            // output words of the chunk read at step k, then back in channel order: chunk c
            // was read at step (c - rot) mod 4
            uint32_t w[4][OW];
#pragma unroll
            for (int k = 0; k < 4; k++) {
                if constexpr (OUT == DT_F32) {
                    w[k][0] = __float_as_uint(y[2 * k].x);
                    w[k][1] = __float_as_uint(y[2 * k].y);
                    w[k][2] = __float_as_uint(y[2 * k + 1].x);
                    w[k][3] = __float_as_uint(y[2 * k + 1].y);
                } else if constexpr (OUT == DT_BF16) {
                    const __nv_bfloat162 v0 = __floats2bfloat162_rn(y[2 * k].x, y[2 * k].y);
                    const __nv_bfloat162 v1 = __floats2bfloat162_rn(y[2 * k + 1].x, y[2 * k + 1].y);
                    w[k][0] = *reinterpret_cast<const uint32_t *>(&v0);
                    w[k][1] = *reinterpret_cast<const uint32_t *>(&v1);
                } else {
                    const __half2 v0 = __floats2half2_rn(y[2 * k].x, y[2 * k].y);
                    const __half2 v1 = __floats2half2_rn(y[2 * k + 1].x, y[2 * k + 1].y);
                    w[k][0] = *reinterpret_cast<const uint32_t *>(&v0);
                    w[k][1] = *reinterpret_cast<const uint32_t *>(&v1);
                }
            }
            uint32_t o[4 * OW];
#pragma unroll
            for (int q = 0; q < OW; q++) {
                const bool r2 = rot & 2, r1 = rot & 1;
                const uint32_t a0 = sel(r2, w[2][q], w[0][q]), a1 = sel(r2, w[3][q], w[1][q]);
                const uint32_t a2 = sel(r2, w[0][q], w[2][q]), a3 = sel(r2, w[1][q], w[3][q]);
                o[0 * OW + q] = sel(r1, a3, a0);
                o[1 * OW + q] = sel(r1, a0, a1);
                o[2 * OW + q] = sel(r1, a1, a2);
                o[3 * OW + q] = sel(r1, a2, a3);
            }
            if (wide_stores) {
#pragma unroll
                for (int k = 0; k < OW / 2; k++) {
                    uint32_t v8[8];
#pragma unroll
                    for (int x = 0; x < 8; x++) v8[x] = o[8 * k + x];
                    st_v8(op + 32 * k, v8);
                }
            } else {
                uint4 *dst = reinterpret_cast<uint4 *>(op);
#pragma unroll
                for (int k = 0; k < OW; k++)
                    dst[k] = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
            }
            op += ostep;
            cur = nxt;
            nxt = nxt2;
            i = inext;
        }
    }
    if (__any_sync(0xffffffffu, bad_index) && lane == 0) or_status(p.status, QVG_DEV_BAD_INDEX);
}

namespace {

template <int BITS, int OUT, int TT>
cudaError_t launch_dq(const DPlan &p, int num_sms, int W, size_t table_bytes, bool smem_tables,
                      cudaStream_t st) {
    auto kern = p.qscheme == QVG_QSCHEME_MIDRISE ? k_dequant<BITS, OUT, TT, 1> : k_dequant<BITS, OUT, TT, 0>;
    const size_t smem = smem_tables ? table_bytes : 16;
    // 32-byte stores need a 32-byte aligned output and tensor stride
    const size_t eb = p.out_dtype == DT_F32 ? 4 : 2;
    const int wide = (reinterpret_cast<uintptr_t>(p.out) % 32 == 0 &&
                      (p.out_stride * eb) % 32 == 0) ? 1 : 0;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t n_chunks = (p.N + p.chunk_len - 1) / p.chunk_len;
    // S CTAs (one per slice) per share of the tokens; at least one share
    const int S = kD / W;
    const int grid = std::max(1, num_sms / S) * S;
    return launch_kernel(kern, dim3(grid), dim3(kDqThreads), smem, st, p, W, S, n_chunks,
                         smem_tables ? 1 : 0, wide);
}

template <int BITS, int OUT>
cudaError_t launch_dq_T(const DPlan &p, int num_sms, int W, size_t tb, bool sm, cudaStream_t st) {
    switch (p.T) {
        case 0: return launch_dq<BITS, OUT, 0>(p, num_sms, W, tb, sm, st);
        case 1: return launch_dq<BITS, OUT, 1>(p, num_sms, W, tb, sm, st);
        case 2: return launch_dq<BITS, OUT, 2>(p, num_sms, W, tb, sm, st);
        case 3: return launch_dq<BITS, OUT, 3>(p, num_sms, W, tb, sm, st);
        case 4: return launch_dq<BITS, OUT, 4>(p, num_sms, W, tb, sm, st);
        default: return launch_dq<BITS, OUT, -1>(p, num_sms, W, tb, sm, st);
    }
}

template <int BITS>
cudaError_t launch_dq_out(const DPlan &p, int num_sms, int W, size_t tb, bool sm, cudaStream_t st) {
    if (p.out_dtype == DT_BF16) return launch_dq_T<BITS, DT_BF16>(p, num_sms, W, tb, sm, st);
    if (p.out_dtype == DT_F16) return launch_dq_T<BITS, DT_F16>(p, num_sms, W, tb, sm, st);
    return launch_dq_T<BITS, DT_F32>(p, num_sms, W, tb, sm, st);
}

}  // namespace

cudaError_t launch_dequant(const DPlan &p, int num_sms, cudaStream_t st) {
    // slice width: the widest whose T x C x W fp32 tables fit the staging budget
    const size_t per_ch = (size_t)p.T * p.C * 4;  // bytes per channel of all tables
    int W = 128;
    bool smem_tables = p.T > 0;
    if (smem_tables) {
        W = 0;
        for (int w : {128, 64, 32})
            if (per_ch * w <= kDqTableBytes) {
                W = w;
                break;
            }
        if (W == 0) {
            W = 128;
            smem_tables = false;
        }
    }
    const size_t tb = smem_tables ? per_ch * W : 0;
    if (p.bits == 2) return launch_dq_out<2>(p, num_sms, W, tb, smem_tables, st);
    return launch_dq_out<4>(p, num_sms, W, tb, smem_tables, st);
}

}  // namespace qvg
