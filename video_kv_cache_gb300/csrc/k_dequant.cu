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
//     unit, so centroid lookups never go to L2/HBM in the token loop.
//   * A warp takes 32 tokens at a time.  First every lane fetches one token's metadata (its
//     slice of codes, its scale bytes, its T cluster indices) with wide coalesced loads,
//     so 32 tokens' worth of reads are in flight per warp; the metadata goes to a per-warp
//     shared-memory buffer.  Then the warp reconstructs the 32 tokens one after another:
//     lane l owns CPL = W/32 consecutive channels, all lanes read the same table row
//     (consecutive words: no bank conflicts), and the warp writes one contiguous
//     W * sizeof(out) run per token.
//   * When even 32-channel slices of the tables do not fit in shared memory, the kernel
//     reads them through L1/L2 instead.
#include <cuda_fp8.h>

#include <algorithm>
#include <cstdlib>

#include "internal.cuh"

namespace qvg {

namespace {
constexpr int kDqThreads = 512;

// Bytes of per-token metadata staged for a W-channel slice: the slice's codes, its scale
// bytes (padded to 8) and the T cluster indices packed into 8 bytes.
template <int CPL, int BITS>
struct DqMeta {
    static constexpr int W = 32 * CPL;
    static constexpr int CODE_BYTES = W * BITS / 8;  // 8 .. 64
    static constexpr int BYTES = CODE_BYTES + 16;
};
}  // namespace

template <int CPL, int BITS, int OUT, bool SMEM>
__global__ void __launch_bounds__(kDqThreads)
    k_dequant(DPlan p, int64_t n_chunks, int64_t blocks_per_chunk, int64_t blk,
              int64_t total_units, int table_floats) {
    extern __shared__ __align__(16) float smem_f[];
    using Meta = DqMeta<CPL, BITS>;
    constexpr int W = Meta::W;
    constexpr int SLICES = kD / W;
    constexpr int CB = Meta::CODE_BYTES;
    constexpr int MB = Meta::BYTES;
    constexpr int CODE_BITS = CPL * BITS;  // codes of one lane: 2..16 bits
    constexpr int MID = 1 << (BITS - 1);
    constexpr int nw = kDqThreads / 32;
    float *tab = smem_f;                                                 // [T][C][W]
    float *lut = smem_f + table_floats;                                  // [256] E4M3 -> fp32
    unsigned char *meta = reinterpret_cast<unsigned char *>(lut + 256);  // [nw][32][MB]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int T = p.T, C = p.C;
    const int row_bytes = kD * BITS / 8;
    const int ngroups = kD / p.group;
    unsigned char *my_meta = meta + warp * 32 * MB;

    if (threadIdx.x < 256)
        lut[threadIdx.x] = __half2float(
            __half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)threadIdx.x, __NV_E4M3)));

    const int64_t per = total_units / gridDim.x, rem = total_units % gridDim.x;
    const int64_t ub = blockIdx.x * per + min((int64_t)blockIdx.x, rem);
    const int64_t ue = ub + per + ((int64_t)blockIdx.x < rem ? 1 : 0);
    int64_t staged = -1;
    __syncthreads();

    for (int64_t u = ub; u < ue; u++) {
        const int64_t b = u % blocks_per_chunk;
        const int64_t hcs = u / blocks_per_chunk;  // (h, chunk, slice)
        const int s = (int)(hcs % SLICES);
        const int64_t hc = hcs / SLICES;
        const int64_t c = hc % n_chunks;
        const int h = (int)(hc / n_chunks);
        const float *tbl = p.cent + ((int64_t)h * p.n_tables + c) * T * C * kD;
        if (SMEM && T > 0 && hcs != staged) {
            __syncthreads();
            const int nvec = T * C * (W / 4);
            for (int x = threadIdx.x; x < nvec; x += kDqThreads) {
                const int r = x / (W / 4), q = x - r * (W / 4);
                reinterpret_cast<float4 *>(tab)[x] =
                    __ldg(reinterpret_cast<const float4 *>(tbl + (int64_t)r * kD + s * W) + q);
            }
            __syncthreads();
            staged = hcs;
        }
        const int64_t c_lo = c * p.chunk_len;
        const int64_t i0 = c_lo + b * blk;
        const int64_t i1 = min(min(c_lo + p.chunk_len, p.N), i0 + blk);
        const uint8_t *codes_h = p.codes + (int64_t)h * p.cap * row_bytes + s * CB;
        // scale bytes of this slice: its W/group groups, or the one group that holds it
        const int sgroups = W >= p.group ? W / p.group : 1;
        const uint8_t *scales_h = p.scales + (int64_t)h * p.cap * ngroups + (s * W) / p.group;
        const uint8_t *pi_h = p.pi + (int64_t)h * T * p.cap;
        float *out32 = static_cast<float *>(p.out);
        uint16_t *out16 = static_cast<uint16_t *>(p.out);
        const int64_t out_h = (int64_t)h * p.out_stride + s * W + lane * CPL;
        // this lane's place inside a token's slice metadata
        const int code_byte = (lane * CODE_BITS) >> 3, code_shift = (lane * CODE_BITS) & 7;
        const int scale_byte = W >= p.group ? (lane * CPL) / p.group : 0;

        for (int64_t base = i0 + (int64_t)warp * 32; base < i1; base += (int64_t)nw * 32) {
            // phase 1: lane l fetches the metadata of token base + l
            const int64_t il = base + lane;
            if (il < i1) {
                const uint8_t *cp = codes_h + il * row_bytes;
                unsigned char *mp = my_meta + lane * MB;
                if constexpr (CB == 8) {
                    *reinterpret_cast<uint2 *>(mp) = __ldg(reinterpret_cast<const uint2 *>(cp));
                } else {
#pragma unroll
                    for (int q = 0; q < CB / 16; q++)
                        reinterpret_cast<uint4 *>(mp)[q] = __ldg(reinterpret_cast<const uint4 *>(cp) + q);
                }
                uint64_t sc = 0, pk = 0;
                for (int g = 0; g < sgroups; g++)
                    sc |= (uint64_t)__ldg(scales_h + il * ngroups + g) << (8 * g);
#pragma unroll
                for (int t = 0; t < kMaxT; t++)
                    if (t < T) pk |= (uint64_t)__ldg(pi_h + (int64_t)t * p.cap + il) << (8 * t);
                *reinterpret_cast<uint64_t *>(mp + CB) = sc;
                *reinterpret_cast<uint64_t *>(mp + CB + 8) = pk;
            }
            __syncwarp();
            // phase 2: the warp reconstructs the W-channel slice of each of those tokens
            const int nt = (int)min((int64_t)32, i1 - base);
#pragma unroll 2
            for (int j = 0; j < nt; j++) {
                const unsigned char *mp = my_meta + j * MB;
                uint32_t cw;
                if constexpr (CODE_BITS <= 8)
                    cw = (uint32_t)(mp[code_byte] >> code_shift);
                else
                    cw = *reinterpret_cast<const uint16_t *>(mp + code_byte);
                const float sq = lut[mp[CB + scale_byte]];
                const float off = -sq * (float)MID;
                const uint64_t pk = *reinterpret_cast<const uint64_t *>(mp + CB + 8);
                float y[CPL];
#pragma unroll
                for (int q = 0; q < CPL; q++)
                    y[q] = __fmaf_rn(sq, (float)((cw >> (q * BITS)) & ((1u << BITS) - 1u)), off);
                for (int t = T - 1; t >= 0; t--) {
                    const int pjt = min((int)((pk >> (8 * t)) & 0xFFu), C - 1);
                    if constexpr (SMEM) {
                        const float *trow = tab + (t * C + pjt) * W + lane * CPL;
                        if constexpr (CPL == 4) {
                            const float4 a = *reinterpret_cast<const float4 *>(trow);
                            y[0] += a.x; y[1] += a.y; y[2] += a.z; y[3] += a.w;
                        } else if constexpr (CPL == 2) {
                            const float2 a = *reinterpret_cast<const float2 *>(trow);
                            y[0] += a.x; y[1] += a.y;
                        } else {
                            y[0] += trow[0];
                        }
                    } else {
                        const float *trow = tbl + ((int64_t)t * C + pjt) * kD + s * W + lane * CPL;
#pragma unroll
                        for (int q = 0; q < CPL; q++) y[q] += __ldg(trow + q);
                    }
                }
                const int64_t o = out_h + (base + j) * kD;
                if constexpr (OUT == DT_F32) {
                    if constexpr (CPL == 4)
                        *reinterpret_cast<float4 *>(out32 + o) = make_float4(y[0], y[1], y[2], y[3]);
                    else if constexpr (CPL == 2)
                        *reinterpret_cast<float2 *>(out32 + o) = make_float2(y[0], y[1]);
                    else
                        out32[o] = y[0];
                } else {
                    uint32_t hv[CPL];
#pragma unroll
                    for (int q = 0; q < CPL; q++)
                        hv[q] = OUT == DT_BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(y[q]))
                                               : __half_as_ushort(__float2half_rn(y[q]));
                    if constexpr (CPL == 4)
                        *reinterpret_cast<uint2 *>(out16 + o) =
                            make_uint2(hv[0] | (hv[1] << 16), hv[2] | (hv[3] << 16));
                    else if constexpr (CPL == 2)
                        *reinterpret_cast<uint32_t *>(out16 + o) = hv[0] | (hv[1] << 16);
                    else
                        out16[o] = (uint16_t)hv[0];
                }
            }
            __syncwarp();
        }
    }
}

namespace {

template <int CPL, int BITS, int OUT, bool SMEM>
cudaError_t launch_dq(const DPlan &p, int num_sms, size_t table_bytes, cudaStream_t st) {
    auto kern = k_dequant<CPL, BITS, OUT, SMEM>;
    const size_t smem =
        table_bytes + 256 * 4 + (size_t)(kDqThreads / 32) * 32 * DqMeta<CPL, BITS>::BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kDqThreads, smem);
    if (e != cudaSuccess) return e;
    occ = std::max(occ, 1);
    const int64_t resident = (int64_t)num_sms * occ;
    constexpr int W = 32 * CPL;
    const int64_t slices = kD / W;
    const int64_t n_chunks = (p.N + p.chunk_len - 1) / p.chunk_len;
    const int64_t base_units = (int64_t)p.H * n_chunks * slices;
    // split chunks into token blocks until there are a few units per resident CTA
    int64_t bpc = std::max<int64_t>(1, (resident * 2 + base_units - 1) / base_units);
    const int64_t clen = std::min(p.chunk_len, p.N);
    int64_t blk = std::max<int64_t>(256, (clen + bpc - 1) / bpc);
    blk = (blk + 31) / 32 * 32;
    bpc = (clen + blk - 1) / blk;
    const int64_t total = base_units * bpc;
    const int grid = (int)std::min<int64_t>(total, resident);
    kern<<<grid, kDqThreads, smem, st>>>(p, n_chunks, bpc, blk, total, (int)(table_bytes / 4));
    return cudaGetLastError();
}

template <int CPL, int BITS>
cudaError_t launch_dq_out(const DPlan &p, int num_sms, size_t tbytes, bool use_smem, cudaStream_t st) {
    if (use_smem) {
        if (p.out_dtype == DT_BF16) return launch_dq<CPL, BITS, DT_BF16, true>(p, num_sms, tbytes, st);
        if (p.out_dtype == DT_F16) return launch_dq<CPL, BITS, DT_F16, true>(p, num_sms, tbytes, st);
        return launch_dq<CPL, BITS, DT_F32, true>(p, num_sms, tbytes, st);
    }
    if (p.out_dtype == DT_BF16) return launch_dq<CPL, BITS, DT_BF16, false>(p, num_sms, 0, st);
    if (p.out_dtype == DT_F16) return launch_dq<CPL, BITS, DT_F16, false>(p, num_sms, 0, st);
    return launch_dq<CPL, BITS, DT_F32, false>(p, num_sms, 0, st);
}

template <int CPL>
cudaError_t launch_dq_bits(const DPlan &p, int num_sms, size_t tbytes, bool use_smem, cudaStream_t st) {
    if (p.bits == 2) return launch_dq_out<CPL, 2>(p, num_sms, tbytes, use_smem, st);
    return launch_dq_out<CPL, 4>(p, num_sms, tbytes, use_smem, st);
}

}  // namespace

cudaError_t launch_dequant(const DPlan &p, int num_sms, cudaStream_t st) {
    // Slice width: the widest W whose T x C x W fp32 tables stay within the budget; 32-
    // channel slices up to 160 KB of tables; tables through L1/L2 beyond that.
    size_t budget = 128 * 1024;
    if (const char *env = std::getenv("QVG_DQ_TABLE_BYTES")) budget = (size_t)std::atol(env);
    const size_t per_ch = (size_t)p.T * p.C * 4;  // bytes per channel of all tables
    int W = 128;
    bool use_smem = p.T > 0;
    if (use_smem) {
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
                use_smem = false;
            }
        }
    }
    const size_t tbytes = use_smem ? per_ch * W : 0;
    if (W == 128) return launch_dq_bits<4>(p, num_sms, tbytes, use_smem, st);
    if (W == 64) return launch_dq_bits<2>(p, num_sms, tbytes, use_smem, st);
    return launch_dq_bits<1>(p, num_sms, tbytes, use_smem, st);
}

}  // namespace qvg
