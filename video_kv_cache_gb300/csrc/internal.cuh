// Internal declarations shared by the CUDA translation units of libqvg.
//
// Numerics used on the device (the oracle works in fp64; these are the GPU's choices):
//   * Residuals r = x - C^(1)[pi^(1)] - ... are formed with an error-free TwoSum chain and
//     rounded once to fp32, so r is the fp32 value nearest the exact residual.
//   * Centroid sums are exact: every residual is turned into a 64-bit fixed-point integer
//     with a per-(tensor, stage) power-of-two scale 2^Q chosen from max|r| and N, then added
//     with integer atomics.  The result does not depend on summation order, and the mean
//     is the exact sum divided by the count, rounded once to fp32.
//   * Distances for the assignment come from a tensor-core GEMM on a two-term bf16 split of
//     the centred operands (hi*hi + hi*lo + lo*hi, fp32 accumulate).  Every cluster whose
//     GEMM score lies within a rigorous error margin of the best one is re-scored with a
//     direct fp32 sum of squared differences, ties going to the lowest cluster index.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "qvg.h"

namespace qvg {

constexpr int kD = 128;            // channels per token
constexpr int kMaxT = 8;           // most smoothing stages
constexpr int kMaxC = 256;         // most clusters (pi is uint8)

enum : int { DT_F16 = 0, DT_BF16 = 1, DT_F32 = 2 };

// Everything a quantize call's kernels need, resolved on the host.
struct QPlan {
    int H;
    int64_t N;
    int C, Cpad, T, bits, group, iters, in_dtype;
    int64_t x_stride;      // elements between tensors of X
    int64_t cap, tok_off;  // token slots per tensor in codes/scales/pi, first slot written
    int64_t cent_tstride;  // floats between tensors in the centroid tables
    int64_t cent_off;      // floats to this call's table slot inside a tensor
    const void *X;
    uint8_t *codes, *scales, *pi;
    float *cent;
    const float *warm;
    int64_t warm_stride;
    // workspace
    float *R32;            // [H][N][128] residual R^(t-1), stages t >= 2
    __nv_bfloat16 *A;      // [H][2][N][128] bf16 hi / lo planes of the centred residual
    float *rnorm;          // [H][N] norm of the centred residual row
    __nv_bfloat16 *B;      // [H][2][Cpad][128] bf16 hi / lo planes of the centred centroids
    float *cn;             // [H][Cpad] squared norm of the centred centroids
    float *mu;             // [H][128] centring vector of the current stage
    int *counts;           // [H][C] cluster sizes of the current assignment
    int *offs;             // [H][C] first position of each cluster in `ids`
    int *blockoff;         // [H][nsb][C] per token block: its first position per cluster
    int *ids;              // [H][N] token indices grouped by cluster, increasing in a cluster
    uint8_t *cid;          // [H][N] cluster of each sorted position
    float *psum;           // [H][nchunk][2][2][128] (sum, error) of the runs that cross a
                           // chunk boundary: [0] the run at the chunk start, [1] the last run
    float *wsum;           // [H][C][2][128] (sum, error) of clusters inside one chunk
    int nsb, nchunk;       // token blocks of the sort, 64-position chunks per tensor
    unsigned *maxabs;      // [H] max |r| of the current stage, as float bits
    int *init_idx;         // [H][T][C] cold-start rows
    unsigned *stats;       // [16] counters (see kStat*)
    int *rq_count;         // number of queued near-tie re-scoring requests
    struct RefineReq *rq;  // [H*N] near-tie re-scoring requests
    uint32_t *status;      // caller's device status word (may be NULL)
};

enum { kStatRefineRows = 0, kStatRefineCands = 1 };

// A token whose GEMM scores leave more than one cluster within the error margin of the
// best: cand holds one bit per cluster to re-score exactly.
struct RefineReq {
    int h;
    int i;
    uint32_t cand[8];
};

// ------------------------------------------------------------------------------------
// Small device helpers
// ------------------------------------------------------------------------------------

__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// 8 consecutive input channels of X as fp32 (exact for fp16 / bf16).
__device__ __forceinline__ void load_x8(const void *X, int dt, int64_t off, float v[8]) {
    if (dt == DT_F32) {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(X) + off);
        float4 a = __ldg(p), b = __ldg(p + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        uint4 raw = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(X) + off));
        uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int q = 0; q < 4; q++) {
            if (dt == DT_BF16) {
                v[2 * q] = __uint_as_float(w[q] << 16);
                v[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
            } else {
                __half2 h = *reinterpret_cast<__half2 *>(&w[q]);
                float2 f = __half22float2(h);
                v[2 * q] = f.x;
                v[2 * q + 1] = f.y;
            }
        }
    }
}

__device__ __forceinline__ float load_x1(const void *X, int dt, int64_t off) {
    if (dt == DT_F32) return __ldg(static_cast<const float *>(X) + off);
    uint16_t b = __ldg(static_cast<const unsigned short *>(X) + off);
    if (dt == DT_BF16) return __uint_as_float(static_cast<uint32_t>(b) << 16);
    return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ void load_f8(const float *p, float v[8]) {
    float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Fixed-point exponent for sums of n <= N values bounded by the float whose bits are
// `maxabs_bits`: |sum * 2^Q| < 2^62.
__device__ __forceinline__ int fixed_q(unsigned maxabs_bits, int64_t N) {
    unsigned eb = (maxabs_bits >> 23) & 0xFFu;
    if (maxabs_bits == 0u || eb == 0xFFu) return 0;
    int e = (int)(eb < 1u ? 1u : eb) - 126;  // maxabs < 2^e
    int L = 64 - __clzll((unsigned long long)N);  // N < 2^L
    int q = 62 - L - e;
    return q < -100 ? -100 : (q > 120 ? 120 : q);
}

__device__ __forceinline__ float pow2f(int q) { return __int_as_float((q + 127) << 23); }

// x * 2^q rounded to nearest (ties to even) as a 64-bit integer, for |x * 2^q| < 2^62.
// Integer-only: a float -> int64 conversion instruction would run on the FP64 pipe, which
// is narrow on this GPU.
__device__ __forceinline__ long long f2fix(float x, int q) {
    const uint32_t b = __float_as_uint(x);
    const int e = (int)((b >> 23) & 0xFFu);
    const uint32_t m = (b & 0x7FFFFFu) | (e ? 0x800000u : 0u);
    const int sh = (e ? e : 1) - 150 + q;  // |x| = m * 2^(e - 150) for normals
    unsigned long long v;
    if (sh >= 0) {
        v = (unsigned long long)m << (sh < 63 ? sh : 63);
    } else {
        const int s = -sh < 31 ? -sh : 31;
        const uint32_t kept = m >> s;
        const uint32_t rem = m - (kept << s);
        const uint32_t half = 1u << (s - 1);
        v = kept + ((rem > half) || (rem == half && (kept & 1u)) ? 1u : 0u);
    }
    return (b >> 31) ? -(long long)v : (long long)v;
}

__device__ __forceinline__ void or_status(uint32_t *status, uint32_t bits) {
    if (status) atomicOr(status, bits);
}

// ------------------------------------------------------------------------------------
// Launchers (each enqueues on `st`; returns the CUDA error of the launch)
// ------------------------------------------------------------------------------------

cudaError_t launch_init_centroids(const QPlan &p, int t, cudaStream_t st);
cudaError_t launch_centre(const QPlan &p, int t, cudaStream_t st);
cudaError_t launch_prep(const QPlan &p, int t, cudaStream_t st);
cudaError_t launch_centroid_planes(const QPlan &p, int t, cudaStream_t st);
cudaError_t launch_cluster_means(const QPlan &p, int t, bool planes, cudaStream_t st);
constexpr int kSortBlock = 256;  // tokens per block of the counting sort
constexpr int kChunk = 64;       // sorted positions summed by one warp
cudaError_t launch_encode(const QPlan &p, cudaStream_t st);

// TMA tensor maps of the assignment GEMM: A = residual planes, B = centroid planes.
struct AssignMaps {
    CUtensorMap a;
    CUtensorMap b;
};
// Encodes the maps for plan p into caller-provided storage (no allocation).
cudaError_t assign_encode(const QPlan &p, AssignMaps *maps);
// Heap-allocates the maps and encodes them; free with assign_release.
cudaError_t assign_prepare(const QPlan &p, AssignMaps **maps);
void assign_release(AssignMaps *maps);
cudaError_t launch_assign(const QPlan &p, const AssignMaps *maps, int t, int num_sms,
                          cudaStream_t st);
cudaError_t launch_refine(const QPlan &p, int t, int num_sms, cudaStream_t st);
size_t assign_smem_bytes(int Cpad);

struct DPlan {
    int H;
    int64_t N;
    int C, T, bits, group, out_dtype;
    int64_t chunk_len, cap;
    int n_tables;
    int64_t out_stride;
    const uint8_t *codes, *scales, *pi;
    const float *cent;
    void *out;
    uint32_t *status;
};
cudaError_t launch_dequant(const DPlan &p, int num_sms, cudaStream_t st);

}  // namespace qvg
