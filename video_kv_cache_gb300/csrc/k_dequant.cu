// Fused reconstruction: dequantize the final residual and add back every stage's
// assigned centroid in one pass, in registers.
//
// Method step: X^(T) = deQ(X_INT, S_x), then X^(t-1) = X^(t) + C^(t)_{pi_i} for t = T..1
// (review page "Quant VideoGen: 基于2-Bit KV缓存量化的自回归长视频生成", pipeline paragraph;
// "Quant VideoGen" notes page, sections Progressive Residual Quantization and
// Algorithm-System Co-design, the fused dequantization kernel).
//
// Design (HBM-bound for one or two stages; bound by shared-memory reads of the tables
// beyond that, since every output element reads T fp32 table values):
//   * One CTA of 640 threads per SM takes an equal contiguous share of the flattened
//     (tensor, token) space and walks it in blocks of up to kDqBlock tokens inside one
//     centroid table.  The T tables are staged in shared memory one channel slice of W
//     channels at a time (T x C x W fp32: W is the widest of 128, 64 and 32 that fits
//     200 KB -- 64 for T = 2, 32 for T = 4 with C = 256); beyond that they are read
//     through L1 / L2 without slicing.  Every slice of a block is done before the next
//     block, so the block's codes, scales and indices, which each slice reads again, are
//     still in L2.
//   * A lane rebuilds 16 contiguous channels of a token, in four groups of four: one 4- or
//     8-byte code load, one scale byte and T cluster-index bytes per token; the W / 16
//     lanes of a token cover the slice.
//   * Arithmetic per element: the code u is masked in place into the mantissa of the float
//     2^23 (one logic op), one subtraction gives (u - 2^(b-1)) * 2^k exactly, and
//     y = fma(s_q * 2^-k, that, C^(T)) (s_q * q is exact, so this equals adding C^(T) to
//     the dequantized value); then one add per further stage, T - 1 down to 1, in fp32,
//     rounded once to the output type.  The subtraction, the fma and the adds run on f32x2
//     pairs of neighbouring channels (each half rounds as the scalar operation does).
//   * Bank-conflict-free table reads.  A 16-byte chunk c of a staged row sits at chunk
//     c ^ ((c >> 3) & 3) of the row, and the lanes of one token visit their four groups
//     in an order rotated by the token's slot in its quarter-warp, so that the eight lanes
//     of a quarter-warp (the unit of a 16-byte shared load) always read eight distinct
//     bank groups, whichever rows their tokens' clusters select.
//   * The lane puts its four groups back in channel order with two conditional swaps and
//     writes its 16 outputs with one 32-byte store (two for fp32) when the output is
//     32-byte aligned, so every store instruction fills whole sectors.
//   * The codes, scale and indices of the next two tokens are loaded before the current
//     token is computed, to keep reads in flight.
#include <cuda_fp8.h>

#include <algorithm>

#include "internal.cuh"

namespace qvg {

namespace {
constexpr int kDqThreads = 640;
constexpr size_t kDqTableBytes = 200 * 1024;  // largest table slice staged by one CTA
constexpr int kLaneCh = 16;                   // channels a lane rebuilds per token
constexpr int64_t kDqBlock = 8192;            // tokens whose slices are done together

// 32-byte store (sm_100 and later), 32-byte aligned address.
__device__ __forceinline__ void st_v8(void *ptr, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// Physical position of 16-byte chunk c in a staged table row.
__device__ __forceinline__ int phys_chunk(int c) { return c ^ ((c >> 3) & 3); }

__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3);
    return __half2float(__half(h));
}
}  // namespace

template <int BITS, int OUT, int TT, int SH>  // SH: 1 for the mid-rise grid, else 0
__global__ void __launch_bounds__(kDqThreads, 1)
    k_dequant(DPlan p, int W, int64_t n_chunks, int smem_tables, int wide_stores) {
    pdl_begin();
    extern __shared__ __align__(16) float smem_f[];
    constexpr int MID = 1 << (BITS - 1);
    constexpr int sh = SH;  // code shift of the level trick
    const int T = TT >= 0 ? TT : p.T;
    const int C = p.C;
    const float4 *tab = reinterpret_cast<const float4 *>(smem_f);  // [T][C][W / 4] chunks
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int LPT = W / kLaneCh;  // lanes per token
    const int TPW = 32 / LPT;     // tokens per warp and pass
    const int sub = lane % LPT;
    const int tpc = (kDqThreads / 32) * TPW;  // tokens per CTA pass
    const int slices = kD / W;
    const int row_bytes = kD * BITS / 8;
    const int ngroups = kD / p.group;
    const int wq = W >> 2;  // 16-byte chunks per staged row
    constexpr int eb = OUT == DT_F32 ? 4 : 2;
    // the lane visits its groups k = 0..3 as group k ^ xr: xr rotates the order by the
    // token's slot in its quarter-warp (W = 32: four tokens, W = 64: two, W = 128: one)
    const int xr = ((lane & 7) / LPT) * ((4 * LPT) / 8);
    int poff[4];  // staged chunk of the group visited at step k
#pragma unroll
    for (int k = 0; k < 4; k++) poff[k] = phys_chunk(4 * sub + (k ^ xr));

    const int64_t total = p.N * p.H;
    const int64_t wb = total * blockIdx.x / gridDim.x;
    const int64_t we = total * (blockIdx.x + 1) / gridDim.x;
    int64_t staged = -1;
    bool bad_index = false;

    for (int64_t pos = wb; pos < we;) {
        const int h = (int)(pos / p.N);
        const int64_t b0 = pos - (int64_t)h * p.N;              // first token of the block
        const int64_t c = min(b0 / p.chunk_len, n_chunks - 1);  // its centroid table
        const int64_t cend = min(p.N, (c + 1) * p.chunk_len);
        const int64_t b1 = min(min(cend, b0 + kDqBlock), b0 + (we - pos));
        pos += b1 - b0;
        const float *tbl = p.cent + ((int64_t)h * p.n_tables + c) * T * C * kD;
        for (int s = 0; s < slices; s++) {
            const int64_t hcs = ((int64_t)h * n_chunks + c) * slices + s;
            if (smem_tables && T > 0 && hcs != staged) {
                __syncthreads();
                const int nvec = T * C * wq;
                for (int x = tid; x < nvec; x += kDqThreads) {
                    const int rr = x / wq, cc = x - rr * wq;
                    reinterpret_cast<float4 *>(smem_f)[rr * wq + phys_chunk(cc)] =
                        __ldg(reinterpret_cast<const float4 *>(tbl + (int64_t)rr * kD + s * W) + cc);
                }
                __syncthreads();
                staged = hcs;
            }
            const int ch0 = s * W + sub * kLaneCh;  // the lane's first channel
            int64_t i = b0 + warp * TPW + lane / LPT;
            // running pointers of token i; they advance by tpc tokens per pass
            const uint8_t *cp = p.codes + ((int64_t)h * p.cap + i) * row_bytes + ch0 * BITS / 8;
            const uint8_t *sp = p.scales + ((int64_t)h * p.cap + i) * ngroups + ch0 / p.group;
            const uint8_t *pp = p.pi + (int64_t)h * T * p.cap + i;
            char *op = static_cast<char *>(p.out) + ((int64_t)h * p.out_stride + i * kD + ch0) * eb;
            const int64_t cstep = (int64_t)tpc * row_bytes, sstep = (int64_t)tpc * ngroups;
            const int64_t ostep = (int64_t)tpc * kD * eb;

            struct Meta {
                uint32_t code[BITS / 2];  // 16 codes, channel 0 in the low bits
                uint32_t sbyte;
                uint64_t pk;              // pi^(1..T), one byte per stage
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
                    for (int t = 0; t < TT; t++) m.pk |= (uint64_t)__ldg(pp + (int64_t)t * p.cap) << (8 * t);
                } else {
                    for (int t = 0; t < T; t++) m.pk |= (uint64_t)__ldg(pp + (int64_t)t * p.cap) << (8 * t);
                }
            };
            auto stage_j = [&](const Meta &m, int t) {
                int j = (int)((m.pk >> (8 * t)) & 0xFFu);
                if (j >= C) {
                    j = C - 1;
                    bad_index = true;
                }
                return j;
            };
            // the four stage-t centroid values of the group visited at step k, cluster j
            auto table4 = [&](int t, int j, int k) {
                if (smem_tables) return tab[(t * C + j) * wq + poff[k]];
                return __ldg(reinterpret_cast<const float4 *>(tbl + ((int64_t)t * C + j) * kD + ch0) +
                             (k ^ xr));
            };

            // two tokens of metadata in flight ahead of the one being computed
            Meta cur, nxt;
            if (i < b1) fetch(cur);
            cp += cstep;
            sp += sstep;
            pp += tpc;
            if (i + tpc < b1) fetch(nxt);
            while (i < b1) {
                const int64_t inext = i + tpc;
                Meta nxt2;
                cp += cstep;
                sp += sstep;
                pp += tpc;
                if (inext + tpc < b1) fetch(nxt2);
                // Code e of a group's four sits at bits BITS*e once the group is shifted
                // down; shifted left by sh (0, or 1 for the mid-rise grid) and kept inside
                // the mantissa of 2^23, the float is 2^23 + u * 2^(BITS*e + sh).
                // Subtracting 2^23 + (MID * 2^sh - sh) * 2^(BITS*e) leaves
                // (u * 2^sh - MID * 2^sh + sh) * 2^(BITS*e) exactly, and
                // sq * 2^-(BITS*e + sh) (exact: a power-of-two rescaling) turns it into the
                // level: sq * (u - MID), or sq * (u - MID + 1/2) for the mid-rise grid.
                const float sq = e4m3_to_float(cur.sbyte & 0xFFu);
                float2 se[2], nk[2];
#pragma unroll
                for (int e2 = 0; e2 < 2; e2++) {
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
                int js[TT > 0 ? TT : 1];
                if constexpr (TT > 0) {
#pragma unroll
                    for (int t = 0; t < TT; t++) js[t] = stage_j(cur, t);
                }
                // res[k] holds the 4 outputs of group k ^ xr, packed as the output type
                constexpr int WPG = OUT == DT_F32 ? 4 : 2;  // 32-bit words per group
                uint32_t res[4][WPG];
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int g = k ^ xr;  // channels 4g .. 4g + 3 of the lane's 16
                    uint32_t cw;
                    if constexpr (BITS == 2)
                        cw = (cur.code[0] >> (8 * g)) << sh;
                    else
                        cw = (((g & 2) ? cur.code[1] : cur.code[0]) >> (16 * (g & 1))) << sh;
                    float m[4];
#pragma unroll
                    for (int e = 0; e < 4; e++)
                        m[e] = __uint_as_float((cw & (((1u << BITS) - 1u) << (BITS * e + sh))) | 0x4B000000u);
                    float2 y0 = __fadd2_rn(make_float2(m[0], m[1]), nk[0]);
                    float2 y1 = __fadd2_rn(make_float2(m[2], m[3]), nk[1]);
                    if (T == 0) {
                        y0 = __fmul2_rn(se[0], y0);
                        y1 = __fmul2_rn(se[1], y1);
                    } else {
                        float4 a = table4(T - 1, TT > 0 ? js[TT > 0 ? T - 1 : 0] : stage_j(cur, T - 1), k);
                        y0 = __ffma2_rn(se[0], y0, make_float2(a.x, a.y));
                        y1 = __ffma2_rn(se[1], y1, make_float2(a.z, a.w));
#pragma unroll
                        for (int t = T - 2; t >= 0; t--) {
                            a = table4(t, TT > 0 ? js[TT > 0 ? t : 0] : stage_j(cur, t), k);
                            y0 = __fadd2_rn(y0, make_float2(a.x, a.y));
                            y1 = __fadd2_rn(y1, make_float2(a.z, a.w));
                        }
                    }
                    if constexpr (OUT == DT_F32) {
                        res[k][0] = __float_as_uint(y0.x);
                        res[k][1] = __float_as_uint(y0.y);
                        res[k][2] = __float_as_uint(y1.x);
                        res[k][3] = __float_as_uint(y1.y);
                    } else if constexpr (OUT == DT_BF16) {
                        const __nv_bfloat162 v0 = __floats2bfloat162_rn(y0.x, y0.y);
                        const __nv_bfloat162 v1 = __floats2bfloat162_rn(y1.x, y1.y);
                        res[k][0] = *reinterpret_cast<const uint32_t *>(&v0);
                        res[k][1] = *reinterpret_cast<const uint32_t *>(&v1);
                    } else {
                        const __half2 v0 = __floats2half2_rn(y0.x, y0.y);
                        const __half2 v1 = __floats2half2_rn(y1.x, y1.y);
                        res[k][0] = *reinterpret_cast<const uint32_t *>(&v0);
                        res[k][1] = *reinterpret_cast<const uint32_t *>(&v1);
                    }
                }
                // back to channel order: res[k] holds group k ^ xr, so swapping the pairs
                // (k, k ^ 1) when bit 0 of xr is set and then (k, k ^ 2) when bit 1 is set
                // leaves group k in res[k]
#pragma unroll
                for (int b = 1; b <= 2; b <<= 1) {
                    const bool sw = (xr & b) != 0;
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        if (k & b) continue;
#pragma unroll
                        for (int x = 0; x < WPG; x++) {
                            const uint32_t lo = res[k][x], hi = res[k | b][x];
                            res[k][x] = sw ? hi : lo;
                            res[k | b][x] = sw ? lo : hi;
                        }
                    }
                }
                // 32-byte stores where the output allows them, else 16-byte ones
                if constexpr (OUT == DT_F32) {
#pragma unroll
                    for (int half = 0; half < 2; half++) {
                        const uint32_t w[8] = {res[2 * half][0], res[2 * half][1], res[2 * half][2],
                                               res[2 * half][3], res[2 * half + 1][0], res[2 * half + 1][1],
                                               res[2 * half + 1][2], res[2 * half + 1][3]};
                        if (wide_stores) {
                            st_v8(op + 32 * half, w);
                        } else {
                            reinterpret_cast<uint4 *>(op + 32 * half)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                            reinterpret_cast<uint4 *>(op + 32 * half)[1] = make_uint4(w[4], w[5], w[6], w[7]);
                        }
                    }
                } else {
                    const uint32_t w[8] = {res[0][0], res[0][1], res[1][0], res[1][1],
                                           res[2][0], res[2][1], res[3][0], res[3][1]};
                    if (wide_stores) {
                        st_v8(op, w);
                    } else {
                        reinterpret_cast<uint4 *>(op)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        reinterpret_cast<uint4 *>(op)[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
                op += ostep;
                cur = nxt;
                nxt = nxt2;
                i = inext;
            }
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
    const int wide = (reinterpret_cast<uintptr_t>(p.out) % 32 == 0 && (p.out_stride * eb) % 32 == 0) ? 1 : 0;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t n_chunks = (p.N + p.chunk_len - 1) / p.chunk_len;
    return launch_kernel(kern, dim3(num_sms), dim3(kDqThreads), smem, st, p, W, n_chunks,
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
