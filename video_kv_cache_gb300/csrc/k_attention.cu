// Attention read straight from the compressed cache: keys and values are rebuilt in
// registers from their codes, scales, cluster indices and centroid tables, used, and
// dropped, so the reconstructed cache never goes to memory.
//
// Method step: the fused reconstruction X^(T) = deQ(X_INT, S_x), X^(t-1) = X^(t) + C^(t)_{pi_i}
// ("Quant VideoGen" notes page, Algorithm-System Co-design, the fused dequantization that
// feeds attention on the fly; review page "Quant VideoGen: 基于2-Bit KV缓存量化的自回归长视频生成",
// pipeline paragraph).  Attention itself is the standard scaled dot-product softmax form:
// o = sum_j p_j v_j, p = softmax_j(scale * q.k_j).
//
// Design (one query block per head; the reads of the compressed rows are latency-bound, so
// the kernel is built to keep many of them in flight):
//   * The N keys of a head are cut into S splits of equal length, a multiple of 32 keys and
//     at least 64, chosen so that all heads together have about 2048 splits.  One warp
//     takes one split and walks it in 32-key tiles with a running maximum and weight sum per
//     query (online softmax); k_attn_combine merges the splits of a head.
//   * A rebuilt row is the value qvg_dequantize writes in fp32: the code's level times the
//     E4M3 scale, plus the stage-T centroid, then stages T-1 .. 1, each add rounded in fp32.
//     A tile's 32 rows are rebuilt together in shared memory (rows padded to 132 floats):
//     lane k reads key k's codes, scale bytes and cluster indices (one pass of coalesced
//     reads for the whole tile), writes its dequantized row and looks up, once, where
//     each stage's centroid row of the key lies (a small shared table); then for each
//     stage the warp adds the keys' centroid rows (lane l: channels 4l .. 4l+3), with the
//     rows of 8 keys loaded before any is added.
//   * Keys: lane j scores key j against every query (queries in shared memory, broadcast
//     reads) with 128 sequential fp32 FMAs.
//   * Values: the tile's value rows are rebuilt the same way into the same buffer; lane l
//     adds channels 4l .. 4l+3 of each, weighted by the key's softmax numerator, into its
//     M x 4 accumulators.
#include <cuda_fp8.h>

#include <algorithm>

#include "internal.cuh"

namespace qvg {

namespace {
constexpr int kAttnWarps = 4;   // warps (splits) per CTA
constexpr int kAttnTile = 32;   // keys per tile
constexpr int kKRow = 132;      // padded staged key row, floats

__device__ __forceinline__ float e4m3_value(uint32_t b) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3);
    return __half2float(__half(h));
}

// Rows [t0, t0 + cnt) of compressed tensor ti, rebuilt as qvg_dequantize's fp32 output has
// them, into rows[k * kKRow + c] (k < cnt).  The reads are issued in bulk, not one key at a
// time: lane k first reads key t0 + k's codes, scale bytes and cluster indices (coalesced
// across the warp), writes its dequantized row and, for each stage, the index of the key's
// centroid row within tensor ti's tables into srow[t * kAttnTile + k]; then, stage by
// stage from T down to 1, the warp adds each key's centroid row (lane l: channels
// 4l .. 4l+3), the rows of KB keys loaded together before they are added.  Each element
// gets the same fp32 operations, in the same order, as in qvg_dequantize.
// (Kept out of line: inlined twice into the split kernel it pushed that kernel's register
// count past what fits several warps per SM.)  Returns true if a stored index was out of
// range.
template <int BITS, int SH, int KB>
__device__ __noinline__ bool rebuild_tile(const APlan &p, const uint8_t *codes,
                                          const uint8_t *scales, const uint8_t *pi,
                                          const float *cent, int64_t ti, int64_t t0, int cnt,
                                          int lane, float *rows, int *srow) {
    bool bad = false;
    constexpr int MID = 1 << (BITS - 1);
    constexpr int WORDS = kD * BITS / 32;  // code words of a row
    constexpr int PER = 32 / BITS;         // codes in a word
    const int ngroups = kD / p.group;
    if (lane < cnt) {
        const int64_t row = ti * p.cap + t0 + lane;
        const uint32_t *cwp = reinterpret_cast<const uint32_t *>(codes + row * (kD * BITS / 8));
        const int tbl = (int)min((t0 + lane) / p.chunk_len, (int64_t)p.n_tables - 1);
        for (int t = 0; t < p.T; t++) {
            int j = __ldg(pi + (ti * p.T + t) * p.cap + t0 + lane);
            bad |= j >= p.C;
            j = min(j, p.C - 1);
            srow[t * kAttnTile + lane] = (tbl * p.T + t) * p.C + j;
        }
        // the row's scale bytes (ngroups = 8, 4 or 2 of them, naturally aligned)
        const uint8_t *sr = scales + row * ngroups;
        const uint64_t sw = ngroups == 8   ? __ldg(reinterpret_cast<const unsigned long long *>(sr))
                            : ngroups == 4 ? (uint64_t)__ldg(reinterpret_cast<const uint32_t *>(sr))
                                           : (uint64_t)__ldg(reinterpret_cast<const unsigned short *>(sr));
        const int gsh = 31 - __clz(p.group);  // log2 of the group size
        float *dst = rows + lane * kKRow;
        // Every code word is read first; code u of a word goes into the mantissa of 2^23
        // (one logic op) and one subtraction leaves u - MID exactly, the level of the
        // symmetric grid (plus 1/2 on the mid-rise grid).
        uint32_t cw[WORDS];
#pragma unroll
        for (int w = 0; w < WORDS; w++) cw[w] = __ldg(cwp + w);
#pragma unroll
        for (int w = 0; w < WORDS; w++) {
#pragma unroll
            for (int c4 = 0; c4 < PER; c4 += 4) {
                const int c = w * PER + c4;
                const float sq = e4m3_value((uint32_t)(sw >> (8 * (c >> gsh))) & 0xFFu);
                float y[4];
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const uint32_t u = (cw[w] >> (BITS * (c4 + k))) & ((1u << BITS) - 1u);
                    float lv = __fsub_rn(__uint_as_float(0x4B000000u | u), 8388608.0f + (float)MID);
                    if (SH) lv = __fadd_rn(lv, 0.5f);
                    y[k] = __fmul_rn(sq, lv);
                }
                *reinterpret_cast<float4 *>(dst + c) = make_float4(y[0], y[1], y[2], y[3]);
            }
        }
    }
    __syncwarp();
    for (int t = p.T - 1; t >= 0; t--) {
        const float *tbase = cent + ti * p.n_tables * p.T * p.C * kD + 4 * lane;  // tensor ti
        const int *sr = srow + t * kAttnTile;
        for (int k0 = 0; k0 < cnt; k0 += KB) {
            float4 c4[KB];
#pragma unroll
            for (int u = 0; u < KB; u++) {
                const int k = k0 + u;
                if (k < cnt) c4[u] = __ldg(reinterpret_cast<const float4 *>(tbase + (int64_t)sr[k] * kD));
            }
#pragma unroll
            for (int u = 0; u < KB; u++) {
                const int k = k0 + u;
                if (k < cnt) {
                    float4 *r = reinterpret_cast<float4 *>(rows + k * kKRow + 4 * lane);
                    const float4 y = *r;
                    *r = make_float4(__fadd_rn(y.x, c4[u].x), __fadd_rn(y.y, c4[u].y),
                                     __fadd_rn(y.z, c4[u].z), __fadd_rn(y.w, c4[u].w));
                }
            }
        }
    }
    __syncwarp();
    return bad;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
}  // namespace

// grid (ceil(S / kAttnWarps), H), block 32 * kAttnWarps; warp w of CTA x takes split
// x * kAttnWarps + w of head blockIdx.y.  MQ >= M queries are held (the rest are zero).
template <int BITS, int SH, int MQ>
__global__ void __launch_bounds__(32 * kAttnWarps, MQ > 4 ? 2 : 4) k_attn_split(APlan p) {
    constexpr int KB = 8;  // centroid rows in flight per lane
    pdl_begin();
    extern __shared__ __align__(16) float sm_attn[];
    float *sQ = sm_attn;  // [MQ][d]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *sK = sm_attn + MQ * kD + warp * (kAttnTile * kKRow + MQ * kAttnTile + p.T * kAttnTile);
    float *sP = sK + kAttnTile * kKRow;                                     // [MQ][32]
    int *sRow = reinterpret_cast<int *>(sP + MQ * kAttnTile);               // [T][32]
    const int h = blockIdx.y;
    for (int x = threadIdx.x; x < MQ * kD; x += blockDim.x) {
        const int m = x / kD;
        sQ[x] = m < p.M ? load_x1(p.Q, p.q_dtype, ((int64_t)h * p.M + m) * kD + (x - m * kD)) : 0.f;
    }
    __syncthreads();
    const int s = blockIdx.x * kAttnWarps + warp;
    if (s >= p.S) return;
    const int64_t n0 = (int64_t)s * p.split_len;
    const int64_t n1 = min(p.N, n0 + p.split_len);
    const int64_t tk = p.k_first + (int64_t)h * p.step, tv = p.v_first + (int64_t)h * p.step;

    float mrun[MQ], lrun[MQ], o[MQ][4];
#pragma unroll
    for (int m = 0; m < MQ; m++) {
        mrun[m] = -INFINITY;
        lrun[m] = 0.f;
        o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.f;
    }
    bool bad = false;
    for (int64_t t0 = n0; t0 < n1; t0 += kAttnTile) {
        const int cnt = (int)min((int64_t)kAttnTile, n1 - t0);
        bad |= rebuild_tile<BITS, SH, KB>(p, p.kc, p.ks, p.kp, p.kcent, tk, t0, cnt, lane, sK, sRow);
        float sc[MQ];
#pragma unroll
        for (int m = 0; m < MQ; m++) sc[m] = 0.f;
        if (lane < cnt) {
            const float4 *kr = reinterpret_cast<const float4 *>(sK + lane * kKRow);
            for (int c = 0; c < kD / 4; c++) {
                const float4 kv = kr[c];
#pragma unroll
                for (int m = 0; m < MQ; m++) {
                    const float4 qv = reinterpret_cast<const float4 *>(sQ + m * kD)[c];
                    sc[m] = __fmaf_rn(qv.x, kv.x, sc[m]);
                    sc[m] = __fmaf_rn(qv.y, kv.y, sc[m]);
                    sc[m] = __fmaf_rn(qv.z, kv.z, sc[m]);
                    sc[m] = __fmaf_rn(qv.w, kv.w, sc[m]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MQ; m++) {
            const float sv = lane < cnt ? __fmul_rn(sc[m], p.scale) : -INFINITY;
            const float mnew = fmaxf(mrun[m], warp_max(sv));  // finite: the tile has a key
            const float corr = expf(mrun[m] - mnew);            // 0 on the first tile
            const float pj = expf(sv - mnew);                   // 0 past the tile's keys
            lrun[m] = __fmaf_rn(lrun[m], corr, warp_sum(pj));
            mrun[m] = mnew;
#pragma unroll
            for (int c = 0; c < 4; c++) o[m][c] = __fmul_rn(o[m][c], corr);
            sP[m * kAttnTile + lane] = pj;
        }
        __syncwarp();  // every lane has scored its key: the value rows can overwrite sK
        bad |= rebuild_tile<BITS, SH, KB>(p, p.vc, p.vs, p.vp, p.vcent, tv, t0, cnt, lane, sK, sRow);
        // four keys at a time (their weights read as one vector per query), then the rest
        // one by one; each accumulator adds the keys in order
        int kk = 0;
        for (; kk + 4 <= cnt; kk += 4) {
            float4 v4[4];
#pragma unroll
            for (int u = 0; u < 4; u++) v4[u] = *reinterpret_cast<const float4 *>(sK + (kk + u) * kKRow + 4 * lane);
#pragma unroll
            for (int m = 0; m < MQ; m++) {
                const float4 w4 = *reinterpret_cast<const float4 *>(sP + m * kAttnTile + kk);
                const float w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    o[m][0] = __fmaf_rn(w[u], v4[u].x, o[m][0]);
                    o[m][1] = __fmaf_rn(w[u], v4[u].y, o[m][1]);
                    o[m][2] = __fmaf_rn(w[u], v4[u].z, o[m][2]);
                    o[m][3] = __fmaf_rn(w[u], v4[u].w, o[m][3]);
                }
            }
        }
        for (; kk < cnt; kk++) {
            const float4 v4 = *reinterpret_cast<const float4 *>(sK + kk * kKRow + 4 * lane);
#pragma unroll
            for (int m = 0; m < MQ; m++) {
                const float w = sP[m * kAttnTile + kk];
                o[m][0] = __fmaf_rn(w, v4.x, o[m][0]);
                o[m][1] = __fmaf_rn(w, v4.y, o[m][1]);
                o[m][2] = __fmaf_rn(w, v4.z, o[m][2]);
                o[m][3] = __fmaf_rn(w, v4.w, o[m][3]);
            }
        }
        __syncwarp();  // the next tile overwrites sK and sP
    }
#pragma unroll
    for (int m = 0; m < MQ; m++) {
        if (m < p.M) {
            const int64_t r = ((int64_t)h * p.S + s) * p.M + m;
            *reinterpret_cast<float4 *>(p.part + r * kD + 4 * lane) =
                make_float4(o[m][0], o[m][1], o[m][2], o[m][3]);
            if (lane == 0) {
                p.ml[2 * r] = mrun[m];
                p.ml[2 * r + 1] = lrun[m];
            }
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) or_status(p.status, QVG_DEV_BAD_INDEX);
}

// One warp per (head, query): the splits' partial outputs rescaled to the largest maximum,
// summed, and divided by the summed weights.  Lane l writes channels 4l .. 4l+3.
__global__ void __launch_bounds__(256) k_attn_combine(APlan p) {
    pdl_begin();
    const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (w >= p.H * p.M) return;
    const int h = w / p.M, m = w - h * p.M;
    float mx = -INFINITY;
    for (int s = lane; s < p.S; s += 32) mx = fmaxf(mx, p.ml[2 * (((int64_t)h * p.S + s) * p.M + m)]);
    mx = warp_max(mx);
    float l = 0.f, a[4] = {0.f, 0.f, 0.f, 0.f};
    // the splits in order, eight at a time: their partial rows and (max, sum) pairs are read
    // before any is added
    constexpr int SB = 8;
    for (int s0 = 0; s0 < p.S; s0 += SB) {
        float2 ml[SB];
        float4 po[SB];
#pragma unroll
        for (int u = 0; u < SB; u++) {
            if (s0 + u < p.S) {
                const int64_t r = ((int64_t)h * p.S + s0 + u) * p.M + m;
                ml[u] = *reinterpret_cast<const float2 *>(p.ml + 2 * r);
                po[u] = *reinterpret_cast<const float4 *>(p.part + r * kD + 4 * lane);
            }
        }
#pragma unroll
        for (int u = 0; u < SB; u++) {
            if (s0 + u < p.S) {
                const float wgt = expf(ml[u].x - mx);
                l = __fmaf_rn(wgt, ml[u].y, l);
                a[0] = __fmaf_rn(wgt, po[u].x, a[0]);
                a[1] = __fmaf_rn(wgt, po[u].y, a[1]);
                a[2] = __fmaf_rn(wgt, po[u].z, a[2]);
                a[3] = __fmaf_rn(wgt, po[u].w, a[3]);
            }
        }
    }
    const int64_t off = ((int64_t)h * p.M + m) * kD + 4 * lane;
#pragma unroll
    for (int c = 0; c < 4; c++) {
        const float v = __fdiv_rn(a[c], l);
        if (p.out_dtype == DT_F32)
            static_cast<float *>(p.O)[off + c] = v;
        else if (p.out_dtype == DT_BF16)
            static_cast<__nv_bfloat16 *>(p.O)[off + c] = __float2bfloat16_rn(v);
        else
            static_cast<__half *>(p.O)[off + c] = __float2half_rn(v);
    }
}

namespace {
template <int BITS, int SH, int MQ>
cudaError_t launch_split(const APlan &p, cudaStream_t st) {
    const size_t smem =
        (size_t)(MQ * kD + kAttnWarps * (kAttnTile * kKRow + MQ * kAttnTile + p.T * kAttnTile)) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(k_attn_split<BITS, SH, MQ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(k_attn_split<BITS, SH, MQ>,
                         dim3((unsigned)((p.S + kAttnWarps - 1) / kAttnWarps), p.H),
                         dim3(32 * kAttnWarps), smem, st, p);
}

template <int BITS, int SH>
cudaError_t launch_split_m(const APlan &p, cudaStream_t st) {
    if (p.M <= 1) return launch_split<BITS, SH, 1>(p, st);
    if (p.M <= 4) return launch_split<BITS, SH, 4>(p, st);
    return launch_split<BITS, SH, kMaxAttnQ>(p, st);
}
}  // namespace

cudaError_t launch_attention(const APlan &p, cudaStream_t st) {
    const bool mr = p.qscheme == QVG_QSCHEME_MIDRISE;
    cudaError_t e = p.bits == 2 ? (mr ? launch_split_m<2, 1>(p, st) : launch_split_m<2, 0>(p, st))
                                : (mr ? launch_split_m<4, 1>(p, st) : launch_split_m<4, 0>(p, st));
    if (e != cudaSuccess) return e;
    return launch_kernel(k_attn_combine, dim3((unsigned)((p.H * p.M + 7) / 8)), dim3(256), 0, st, p);
}

}  // namespace qvg
