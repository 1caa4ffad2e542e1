// Fused reconstruction: dequantize the final residual and add back every stage's
// assigned centroid in one pass, in registers.
//
// Method step: X^(T) = deQ(X_INT, S_x), then X^(t-1) = X^(t) + C^(t)_{pi_i} for t = T..1
// (review page "Quant VideoGen: 基于2-Bit KV缓存量化的自回归长视频生成", pipeline paragraph;
// "Quant VideoGen" notes page, sections Progressive Residual Quantization and
// Algorithm-System Co-design, the fused dequantization kernel).
//
// Design (HBM-bound: the output write is most of the bytes):
//   * One CTA of 1024 threads per SM.  A work unit is (tensor, centroid table, channel
//     slice of W channels, token block); the CTA stages that W-channel slice of all T
//     tables (T x C x W fp32) in shared memory once per unit.  W is the widest of 128,
//     64 and 32 whose slice fits in 200 KB (64 for T = 2, C = 256); beyond that the
//     tables are read through L1 / L2.
//   * A lane rebuilds 16 contiguous channels of a token: one 4- or 8-byte code load, one
//     scale byte and T cluster-index bytes; the W / 16 lanes of a token write its W
//     channels as one contiguous run.
//   * Arithmetic per element: the code u is masked in place into the mantissa of the float
//     2^23 (one logic op), one subtraction gives (u - 2^(b-1)) * 2^k exactly, and
//     y = fma(s_q * 2^-k, that, C^(T)) (s_q * q is exact, so this equals adding C^(T) to
//     the dequantized value); then one add per further stage, T - 1 down to 1, in fp32,
//     rounded once to the output type.
//   * A staged table row's 16-byte chunks are stored XOR-swizzled, so a quarter-warp's
//     16-byte reads hit distinct bank groups.
//   * The next token's codes, scale and indices are loaded before the current token is
//     computed, to keep reads in flight.
#include <cuda_fp8.h>

#include <algorithm>

#include "internal.cuh"

namespace qvg {

namespace {
constexpr int kDqThreads = 1024;
constexpr size_t kDqTableBytes = 200 * 1024;  // largest table slice staged by one CTA
constexpr int kLaneCh = 16;                   // channels a lane rebuilds per token

// Physical 16-byte chunk of logical chunk c in a staged table row: bits 3-4 of c are
// XOR-ed into its low bits, so the lanes of a quarter-warp reading chunk 4l + k
// (l = 0..7) hit 8 distinct bank groups.
__device__ __forceinline__ int swz(int c) { return c ^ ((c >> 3) & 3); }
}  // namespace

template <int BITS, int OUT, int TT>
__global__ void __launch_bounds__(kDqThreads, 1)
    k_dequant(DPlan p, int W, int64_t n_chunks, int64_t blocks_per_chunk, int64_t blk,
              int64_t total_units, int smem_tables) {
    extern __shared__ __align__(16) float smem_f[];
    constexpr int MID = 1 << (BITS - 1);
    constexpr int PER16 = 16 / BITS;  // codes in a 16-bit half-word
    const int T = TT >= 0 ? TT : p.T;
    const int C = p.C;
    float *lut = smem_f;        // [256] E4M3 -> fp32
    float *tab = smem_f + 256;  // [T][C][W], swizzled 16-byte chunks
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int LPT = W / kLaneCh;  // lanes per token
    const int TPW = 32 / LPT;     // tokens per warp and pass
    const int sub = lane % LPT;
    const int tpc = (kDqThreads / 32) * TPW;  // tokens per CTA pass
    const int slices = kD / W;
    const int row_bytes = kD * BITS / 8;
    const int ngroups = kD / p.group;
    const int wq = W >> 2;  // 16-byte chunks per staged row

    if (tid < 256)
        lut[tid] = __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)tid, __NV_E4M3)));

    const int64_t per = total_units / gridDim.x, rem = total_units % gridDim.x;
    const int64_t ub = blockIdx.x * per + min((int64_t)blockIdx.x, rem);
    const int64_t ue = ub + per + ((int64_t)blockIdx.x < rem ? 1 : 0);
    int64_t staged = -1;
    bool bad_index = false;
    __syncthreads();

    for (int64_t u = ub; u < ue; u++) {
        const int64_t b = u % blocks_per_chunk;
        const int64_t hcs = u / blocks_per_chunk;  // (h, chunk, slice)
        const int s = (int)(hcs % slices);
        const int64_t hc = hcs / slices;
        const int64_t c = hc % n_chunks;
        const int h = (int)(hc / n_chunks);
        const float *tbl = p.cent + ((int64_t)h * p.n_tables + c) * T * C * kD;
        if (smem_tables && T > 0 && hcs != staged) {
            __syncthreads();
            const int nvec = T * C * wq;
            for (int x = tid; x < nvec; x += kDqThreads) {
                const int r = x / wq, cc = x - r * wq;
                reinterpret_cast<float4 *>(tab)[r * wq + swz(cc)] =
                    __ldg(reinterpret_cast<const float4 *>(tbl + (int64_t)r * kD + s * W) + cc);
            }
            __syncthreads();
            staged = hcs;
        }
        const int64_t c_lo = c * p.chunk_len;
        const int64_t i0 = c_lo + b * blk;
        const int64_t i1 = min(min(c_lo + p.chunk_len, p.N), i0 + blk);
        const int ch0 = s * W + sub * kLaneCh;  // the lane's first channel
        int64_t i = i0 + warp * TPW + lane / LPT;
        // running pointers of token i; they advance by tpc tokens per pass
        const uint8_t *cp = p.codes + ((int64_t)h * p.cap + i) * row_bytes + ch0 * BITS / 8;
        const uint8_t *sp = p.scales + ((int64_t)h * p.cap + i) * ngroups + ch0 / p.group;
        const uint8_t *pp = p.pi + (int64_t)h * T * p.cap + i;
        char *op = static_cast<char *>(p.out) +
                   ((int64_t)h * p.out_stride + i * kD + ch0) * (OUT == DT_F32 ? 4 : 2);
        const int64_t cstep = (int64_t)tpc * row_bytes, sstep = (int64_t)tpc * ngroups;
        const int64_t ostep = (int64_t)tpc * kD * (OUT == DT_F32 ? 4 : 2);

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
        // stage-t centroid values of this lane's 16 channels, cluster j, into 4 float4
        auto table16 = [&](int t, int j, float4 (&a)[4]) {
            if (smem_tables) {
                const float4 *row = reinterpret_cast<const float4 *>(tab) + (t * C + j) * wq;
#pragma unroll
                for (int k = 0; k < 4; k++) a[k] = row[swz(4 * sub + k)];
            } else {
                const float4 *g =
                    reinterpret_cast<const float4 *>(tbl + ((int64_t)t * C + j) * kD + ch0);
#pragma unroll
                for (int k = 0; k < 4; k++) a[k] = __ldg(g + k);
            }
        };

        Meta cur;
        if (i < i1) fetch(cur);
        while (i < i1) {
            const int64_t inext = i + tpc;
            Meta nxt;
            cp += cstep;
            sp += sstep;
            pp += tpc;
            if (inext < i1) fetch(nxt);
            // Code e of a 16-bit half-word sits at bits BITS*e; kept in place inside the
            // mantissa of 2^23, the float is 2^23 + u * 2^(BITS*e), so subtracting
            // 2^23 + MID * 2^(BITS*e) leaves (u - MID) * 2^(BITS*e) exactly, and
            // sq * 2^-(BITS*e) (exact: a power-of-two rescaling) turns it into sq * q.
            const float sq = lut[cur.sbyte & 0xFFu];
            float se[PER16], ke[PER16];
#pragma unroll
            for (int e = 0; e < PER16; e++) {
                se[e] = __fmul_rn(sq, __uint_as_float((uint32_t)(127 - BITS * e) << 23));
                ke[e] = __uint_as_float(0x4B000000u) + (float)(MID << (BITS * e));
            }
            float y[16];
#pragma unroll
            for (int hw = 0; hw < 16 / PER16; hw++) {
                const uint32_t word = cur.code[hw >> 1] >> (16 * (hw & 1));
#pragma unroll
                for (int e = 0; e < PER16; e++) {
                    const uint32_t m = (word & (((1u << BITS) - 1u) << (BITS * e))) | 0x4B000000u;
                    y[hw * PER16 + e] = __fsub_rn(__uint_as_float(m), ke[e]);
                }
            }
            if (T == 0) {
#pragma unroll
                for (int x = 0; x < 16; x++) y[x] = __fmul_rn(se[x % PER16], y[x]);
            } else {
                float4 a[4];
                table16(T - 1, stage_j(cur, T - 1), a);
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const float cv[4] = {a[k].x, a[k].y, a[k].z, a[k].w};
#pragma unroll
                    for (int q = 0; q < 4; q++)
                        y[4 * k + q] = __fmaf_rn(se[(4 * k + q) % PER16], y[4 * k + q], cv[q]);
                }
                for (int t = T - 2; t >= 0; t--) {
                    table16(t, stage_j(cur, t), a);
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        const float cv[4] = {a[k].x, a[k].y, a[k].z, a[k].w};
#pragma unroll
                        for (int q = 0; q < 4; q++) y[4 * k + q] = __fadd_rn(y[4 * k + q], cv[q]);
                    }
                }
            }
            if constexpr (OUT == DT_F32) {
                float4 *dst = reinterpret_cast<float4 *>(op);
#pragma unroll
                for (int k = 0; k < 4; k++)
                    dst[k] = make_float4(y[4 * k], y[4 * k + 1], y[4 * k + 2], y[4 * k + 3]);
            } else {
                uint32_t w[8];
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    if constexpr (OUT == DT_BF16) {
                        const __nv_bfloat162 v2 = __floats2bfloat162_rn(y[2 * k], y[2 * k + 1]);
                        w[k] = *reinterpret_cast<const uint32_t *>(&v2);
                    } else {
                        const __half2 v2 = __floats2half2_rn(y[2 * k], y[2 * k + 1]);
                        w[k] = *reinterpret_cast<const uint32_t *>(&v2);
                    }
                }
                uint4 *dst = reinterpret_cast<uint4 *>(op);
                dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
            op += ostep;
            cur = nxt;
            i = inext;
        }
    }
    if (__any_sync(0xffffffffu, bad_index) && lane == 0) or_status(p.status, QVG_DEV_BAD_INDEX);
}

namespace {

template <int BITS, int OUT, int TT>
cudaError_t launch_dq(const DPlan &p, int num_sms, int W, size_t table_bytes, bool smem_tables,
                      cudaStream_t st) {
    auto kern = k_dequant<BITS, OUT, TT>;
    const size_t smem = 256 * 4 + (smem_tables ? table_bytes : 0);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t slices = kD / W;
    const int64_t n_chunks = (p.N + p.chunk_len - 1) / p.chunk_len;
    const int64_t base_units = (int64_t)p.H * n_chunks * slices;
    // split chunks into token blocks until there are a couple of units per SM
    int64_t bpc = std::max<int64_t>(1, ((int64_t)num_sms * 2 + base_units - 1) / base_units);
    const int64_t clen = std::min(p.chunk_len, p.N);
    int64_t blk = std::max<int64_t>(256, (clen + bpc - 1) / bpc);
    blk = (blk + 31) / 32 * 32;
    bpc = (clen + blk - 1) / blk;
    const int64_t total = base_units * bpc;
    const int grid = (int)std::min<int64_t>(total, num_sms);
    kern<<<grid, kDqThreads, smem, st>>>(p, W, n_chunks, bpc, blk, total, smem_tables ? 1 : 0);
    return cudaGetLastError();
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
