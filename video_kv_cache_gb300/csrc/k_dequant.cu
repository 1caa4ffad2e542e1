// Fused reconstruction: dequantize the final residual and add back every stage's
// assigned centroid in one pass, in registers.
//
// Method step: X^(T) = deQ(X_INT, S_x), then X^(t-1) = X^(t) + C^(t)_{pi_i} for t = T..1
// (review page "Quant VideoGen: 基于2-Bit KV缓存量化的自回归长视频生成", pipeline paragraph;
// "Quant VideoGen" notes page, sections Progressive Residual Quantization and
// Algorithm-System Co-design, the fused dequantization kernel).
//
// Design (HBM-bound; the output write dominates the bytes):
//   * Work unit = (tensor, centroid table, channel slice of W channels, token block).  The
//     CTA stages the T tables' W-channel slices (T x C x W fp32) in shared memory once per
//     unit, so centroid lookups never leave the SM in the token loop.
//   * A thread reconstructs 16 channels of one token: four 4-channel chunks spread W/4
//     channels apart, so the TPT = W/16 threads of a token cover the slice.  Per chunk it
//     reads one 16-byte table row piece per stage (LDS.128) and writes 4 outputs at once.
//   * Bank conflicts: one quarter-warp (8 threads) serves 8/TPT tokens whose table rows are
//     random.  A token's chunk j sits in bank group (j mod 4 for W = 32, j mod 2 for
//     W = 64); the token in quarter-warp slot k walks its chunks starting at j = k, so the
//     tokens sharing a quarter-warp always hit disjoint banks.
//   * The next token's codes, scales and cluster indices are loaded before the current
//     token is computed, to keep reads in flight.
//   * When even 32-channel slices of the tables do not fit in shared memory the kernel
//     reads them through L1/L2 instead.
#include <cuda_fp8.h>

#include <algorithm>
#include <cstdlib>

#include "internal.cuh"

namespace qvg {

namespace {
constexpr int kDqThreads = 512;

// Per-token state of one thread: the code bits of its 4 chunks (8 bits per chunk for INT2,
// 16 for INT4), their 4 E4M3 scale bytes, and pi^(1..T) one byte per stage.
template <int BITS>
struct TokMeta {
    uint32_t code[BITS / 2];
    uint32_t sbytes;
    uint64_t pk;
};
}  // namespace

// Two CTAs per SM where the state fits in 64 registers a thread; one otherwise.
template <int BITS, int OUT, int TT>
__global__ void __launch_bounds__(kDqThreads, (BITS == 2 && TT >= 0 && TT <= 2) ? 2 : 1)
    k_dequant(DPlan p, int W, int64_t n_chunks, int64_t blocks_per_chunk, int64_t blk,
              int64_t total_units, int table_floats, int smem_tables) {
    extern __shared__ __align__(16) float smem_f[];
    constexpr int MID = 1 << (BITS - 1);
    const int T = TT >= 0 ? TT : p.T;
    const int C = p.C;
    float *tab = smem_f;                  // [T][C][W]
    float *lut = smem_f + table_floats;   // [256] E4M3 -> fp32
    const int tid = threadIdx.x;
    const int TPT = W >> 4;               // threads per token
    const int q = tid & (TPT - 1);
    const int slot = (tid & 7) / TPT;     // token position within the quarter-warp
    const int tpc = kDqThreads / TPT;     // tokens per pass of the CTA
    const int tok = tid / TPT;
    const int slices = kD / W;
    const int row_bytes = kD * BITS / 8;
    const int ngroups = kD / p.group;

    if (tid < 256)
        lut[tid] = __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)tid, __NV_E4M3)));

    const int64_t per = total_units / gridDim.x, rem = total_units % gridDim.x;
    const int64_t ub = blockIdx.x * per + min((int64_t)blockIdx.x, rem);
    const int64_t ue = ub + per + ((int64_t)blockIdx.x < rem ? 1 : 0);
    int64_t staged = -1;
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
            const int nvec = T * C * (W / 4);
            for (int x = tid; x < nvec; x += kDqThreads) {
                const int r = x / (W / 4), qq = x - r * (W / 4);
                reinterpret_cast<float4 *>(tab)[x] =
                    __ldg(reinterpret_cast<const float4 *>(tbl + (int64_t)r * kD + s * W) + qq);
            }
            __syncthreads();
            staged = hcs;
        }
        const int64_t c_lo = c * p.chunk_len;
        const int64_t i0 = c_lo + b * blk;
        const int64_t i1 = min(min(c_lo + p.chunk_len, p.N), i0 + blk);
        // this thread's chunks (first channels), in the bank-rotated order
        int ch[4];
#pragma unroll
        for (int j = 0; j < 4; j++) ch[j] = s * W + 4 * (q + TPT * ((j + slot) & 3));
        const int gshift = 31 - __clz(p.group);
        const uint8_t *codes_h = p.codes + (int64_t)h * p.cap * row_bytes;
        const uint8_t *scales_h = p.scales + (int64_t)h * p.cap * ngroups;
        const uint8_t *pi_h = p.pi + (int64_t)h * T * p.cap;
        float *out32 = static_cast<float *>(p.out) + (int64_t)h * p.out_stride;
        uint16_t *out16 = static_cast<uint16_t *>(p.out) + (int64_t)h * p.out_stride;

        auto fetch = [&](int64_t i, TokMeta<BITS> &m) {
            const uint8_t *cp = codes_h + i * row_bytes;
            const uint8_t *sp = scales_h + i * ngroups;
            m.sbytes = 0;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                m.sbytes |= (uint32_t)__ldg(sp + (ch[j] >> gshift)) << (8 * j);
                if constexpr (BITS == 2) {
                    const uint32_t v = __ldg(cp + (ch[j] >> 2));
                    if (j == 0) m.code[0] = v; else m.code[0] |= v << (8 * j);
                } else {
                    const uint32_t v = __ldg(reinterpret_cast<const unsigned short *>(cp + (ch[j] >> 1)));
                    if ((j & 1) == 0) m.code[j >> 1] = v; else m.code[j >> 1] |= v << 16;
                }
            }
            m.pk = 0;
            if (TT >= 0) {
#pragma unroll
                for (int t = 0; t < (TT > 0 ? TT : 1); t++)
                    if (t < T) m.pk |= (uint64_t)__ldg(pi_h + (int64_t)t * p.cap + i) << (8 * t);
            } else {
                for (int t = 0; t < T; t++)
                    m.pk |= (uint64_t)__ldg(pi_h + (int64_t)t * p.cap + i) << (8 * t);
            }
        };

        int64_t i = i0 + tok;
        TokMeta<BITS> cur;
        if (i < i1) fetch(i, cur);
        while (i < i1) {
            const int64_t inext = i + tpc;
            TokMeta<BITS> nxt;
            if (inext < i1) fetch(inext, nxt);
            int rowoff[TT > 0 ? TT : 8];
            if (TT >= 0) {
#pragma unroll
                for (int t = 0; t < (TT > 0 ? TT : 1); t++)
                    if (t < T) rowoff[t] = (t * C + min((int)((cur.pk >> (8 * t)) & 0xFFu), C - 1)) * W;
            }
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const float sq = lut[(cur.sbytes >> (8 * j)) & 0xFFu];
                const uint32_t cbits = BITS == 2 ? (cur.code[0] >> (8 * j)) & 0xFFu
                                                 : (cur.code[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
                const float off = -sq * (float)MID;
                float y[4];
#pragma unroll
                for (int e = 0; e < 4; e++)
                    y[e] = __fmaf_rn(sq, (float)((cbits >> (e * BITS)) & ((1u << BITS) - 1u)), off);
                const int cw = ch[j] - s * W;  // channel offset within the slice
                if (TT >= 0) {
#pragma unroll
                    for (int t = (TT > 0 ? TT : 1) - 1; t >= 0; t--) {
                        if (t < T) {
                            float4 a;
                            if (smem_tables) {
                                a = *reinterpret_cast<const float4 *>(tab + rowoff[t] + cw);
                            } else {
                                const int pj = rowoff[t] / W - t * C;
                                a = __ldg(reinterpret_cast<const float4 *>(tbl + ((int64_t)t * C + pj) * kD + ch[j]));
                            }
                            y[0] += a.x; y[1] += a.y; y[2] += a.z; y[3] += a.w;
                        }
                    }
                } else {
                    for (int t = T - 1; t >= 0; t--) {
                        const int pj = min((int)((cur.pk >> (8 * t)) & 0xFFu), C - 1);
                        const float4 a = smem_tables
                            ? *reinterpret_cast<const float4 *>(tab + (t * C + pj) * W + cw)
                            : __ldg(reinterpret_cast<const float4 *>(tbl + ((int64_t)t * C + pj) * kD + ch[j]));
                        y[0] += a.x; y[1] += a.y; y[2] += a.z; y[3] += a.w;
                    }
                }
                const int64_t o = i * kD + ch[j];
                if constexpr (OUT == DT_F32) {
                    *reinterpret_cast<float4 *>(out32 + o) = make_float4(y[0], y[1], y[2], y[3]);
                } else if constexpr (OUT == DT_BF16) {
                    const __nv_bfloat162 lo2 = __floats2bfloat162_rn(y[0], y[1]);
                    const __nv_bfloat162 hi2 = __floats2bfloat162_rn(y[2], y[3]);
                    *reinterpret_cast<uint2 *>(out16 + o) =
                        make_uint2(*reinterpret_cast<const uint32_t *>(&lo2),
                                   *reinterpret_cast<const uint32_t *>(&hi2));
                } else {
                    const __half2 lo2 = __floats2half2_rn(y[0], y[1]);
                    const __half2 hi2 = __floats2half2_rn(y[2], y[3]);
                    *reinterpret_cast<uint2 *>(out16 + o) =
                        make_uint2(*reinterpret_cast<const uint32_t *>(&lo2),
                                   *reinterpret_cast<const uint32_t *>(&hi2));
                }
            }
            cur = nxt;
            i = inext;
        }
    }
}

namespace {

template <int BITS, int OUT, int TT>
cudaError_t launch_dq(const DPlan &p, int num_sms, int W, size_t table_bytes, bool smem_tables,
                      cudaStream_t st) {
    auto kern = k_dequant<BITS, OUT, TT>;
    const size_t smem = (smem_tables ? table_bytes : 0) + 256 * 4;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kDqThreads, smem);
    if (e != cudaSuccess) return e;
    occ = std::max(occ, 1);
    const int64_t resident = (int64_t)num_sms * occ;
    const int64_t slices = kD / W;
    const int64_t n_chunks = (p.N + p.chunk_len - 1) / p.chunk_len;
    const int64_t base_units = (int64_t)p.H * n_chunks * slices;
    // split chunks into token blocks until there are a couple of units per resident CTA
    int64_t bpc = std::max<int64_t>(1, (resident * 2 + base_units - 1) / base_units);
    const int64_t clen = std::min(p.chunk_len, p.N);
    int64_t blk = std::max<int64_t>(256, (clen + bpc - 1) / bpc);
    blk = (blk + 31) / 32 * 32;
    bpc = (clen + blk - 1) / blk;
    const int64_t total = base_units * bpc;
    const int grid = (int)std::min<int64_t>(total, resident);
    kern<<<grid, kDqThreads, smem, st>>>(p, W, n_chunks, bpc, blk, total,
                                         smem_tables ? (int)(table_bytes / 4) : 0, smem_tables ? 1 : 0);
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
    // Slice width: the widest W whose T x C x W fp32 tables stay within the budget (so that
    // several CTAs share an SM); 32-channel slices up to 160 KB of tables; tables through
    // L1/L2 beyond that.
    size_t budget = 64 * 1024;
    if (const char *env = std::getenv("QVG_DQ_TABLE_BYTES")) budget = (size_t)std::atol(env);
    const size_t per_ch = (size_t)p.T * p.C * 4;  // bytes per channel of all tables
    int W = 128;
    bool smem_tables = p.T > 0;
    if (smem_tables) {
        W = 0;
        for (int w : {128, 64, 32})
            if (per_ch * w <= budget) {
                W = w;
                break;
            }
        if (W == 0) {
            if (per_ch * 32 <= 160 * 1024) {
                W = 32;
            } else {
                W = 128;
                smem_tables = false;
            }
        }
    }
    const size_t tb = smem_tables ? per_ch * W : 0;
    if (p.bits == 2) return launch_dq_out<2>(p, num_sms, W, tb, smem_tables, st);
    return launch_dq_out<4>(p, num_sms, W, tb, smem_tables, st);
}

}  // namespace qvg
