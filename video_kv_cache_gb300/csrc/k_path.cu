// Bandwidth-bound kernels of the quantize path: cold/warm start, centring, residual
// preparation, the exact centroid-mean update, and the final group encoding.
//
// Method steps (pages about Quant VideoGen, arXiv 2602.02958):
//   * residual R^(t-1) = X - C^(1)[pi^(1)] - ... - C^(t-1)[pi^(t-1)]: review page, pipeline
//     paragraph (R^(0) = X, stage t works on R^(t-1)); notes page, section Progressive
//     Residual Quantization.
//   * centroid = mean of the group's members: notes page, section Semantic-Aware Smoothing;
//     review page, pipeline step (b).
//   * Q(R^(T)): symmetric group INT2/INT4 with FP8 E4M3 scales: review page, pipeline
//     paragraph; notes page, section Algorithm-System Co-design; explainer, Step-by-step.
//   * warm start from the previous chunk's centroids: notes page, section
//     Algorithm-System Co-design.
#include <cuda_fp8.h>

#include <atomic>
#include <type_traits>

#include "internal.cuh"

namespace qvg {

// --------------------------------------------------------------------------------------
// Cold-start rows: for each (tensor, stage) the first C picks of a partial Fisher-Yates
// shuffle of 0..N-1 driven by SplitMix64 (Steele, Lea and Flood, 2014, with the constants
// Vigna published), state seed ^ (tensor_id * 0x9E3779B97F4A7C15) ^ t.  Only the touched
// positions of the permutation are stored: positions < C directly, the others in a small
// open-addressing table.  The k-th SplitMix64 output depends only on state + k * gamma, so
// the warp draws all C picks and their modulo reductions in parallel first; lane 0 then
// applies the swaps in order.   grid (T, H), one warp.
// --------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t splitmix64_next(uint64_t &state) {
    uint64_t z = (state += 0x9E3779B97F4A7C15ULL);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

constexpr int kHashSlots = 1024;

__global__ void k_init_indices(QPlan p, uint64_t seed, int64_t tid_base) {
    pdl_begin();
    const int t = blockIdx.x + 1, h = blockIdx.y, lane = threadIdx.x;
    __shared__ int lo[kMaxC];
    __shared__ int pick[kMaxC];  // position swapped with position j at step j
    __shared__ int keys[kHashSlots];
    __shared__ int vals[kHashSlots];
    const uint64_t state0 = seed ^ ((uint64_t)(tid_base + h) * 0x9E3779B97F4A7C15ULL) ^ (uint64_t)t;
    for (int x = lane; x < p.C; x += 32) {
        lo[x] = x;
        uint64_t st = state0 + (uint64_t)x * 0x9E3779B97F4A7C15ULL;  // state before draw x
        const uint64_t r = splitmix64_next(st);
        pick[x] = x + (int)(r % (uint64_t)(p.N - x));
    }
    for (int x = lane; x < kHashSlots; x += 32) keys[x] = -1;
    __syncwarp();
    if (lane != 0) return;
    int *out = p.init_idx + (int64_t)(h * p.T + (t - 1)) * p.C;
    for (int j = 0; j < p.C; j++) {
        const int k = pick[j];
        int vk;
        int slot = -1;
        if (k < p.C) {
            vk = lo[k];
        } else {
            slot = (int)(((uint32_t)k * 2654435761u) >> 22);  // 10-bit hash
            while (keys[slot] != -1 && keys[slot] != k) slot = (slot + 1) & (kHashSlots - 1);
            vk = keys[slot] == k ? vals[slot] : k;
        }
        const int vj = lo[j];  // position j is never read again after this step
        out[j] = vk;
        if (k < p.C) {
            lo[k] = vj;
        } else {
            keys[slot] = k;
            vals[slot] = vj;
        }
    }
}

cudaError_t launch_init_indices(const QPlan &p, uint64_t seed, int64_t tid_base, cudaStream_t st) {
    return launch_kernel(k_init_indices, dim3(p.T, p.H), dim3(32), 0, st, p, seed, tid_base);
}

// A centroid value in the stored format (qvg_centroid_format): v + rem, with v a faithful
// fp32 rounding of it, rounded once to nearest even in binary16 or bfloat16.  The midpoint
// of the two format neighbours lo <= hi of v is an fp32 number, so v + rem lies on the same
// side of it as v unless v is that midpoint; then the sign of rem decides.  The midpoint of two
// neighbouring 16-bit values has at most 12 significant bits, so it is exact in fp32 (away
// from fp32's subnormal range, which no centroid of these inputs reaches).
__device__ __forceinline__ float store_centroid_value(float v, float rem, int fmt) {
    if (fmt == QVG_CENTROIDS_F32) return v;
    float lo, hi, rn;
    if (fmt == QVG_CENTROIDS_F16) {
        lo = __half2float(__float2half_rd(v));
        hi = __half2float(__float2half_ru(v));
        rn = __half2float(__float2half_rn(v));
    } else {
        lo = __bfloat162float(__float2bfloat16_rd(v));
        hi = __bfloat162float(__float2bfloat16_ru(v));
        rn = __bfloat162float(__float2bfloat16_rn(v));
    }
    if (lo == hi || isinf(lo) || isinf(hi) || v != 0.5f * (lo + hi) || rem == 0.f) return rn;
    return rem > 0.f ? hi : lo;
}

// --------------------------------------------------------------------------------------
// Stage-t initial centroids: rows of R^(t-1) picked by the seeded shuffle, or the caller's
// warm-start table.   grid (C, H), block 128 (one thread per channel).
// --------------------------------------------------------------------------------------
__global__ void k_init_centroids(QPlan p, int t) {
    pdl_begin();
    const int j = blockIdx.x, h = blockIdx.y, k = threadIdx.x;
    float *dst = p.cent + h * p.cent_tstride + p.cent_off + (int64_t)(t - 1) * p.C * kD +
                 (int64_t)j * kD;
    float v, rem = 0.f;
    if (p.warm) {
        v = __ldg(p.warm + h * p.warm_stride + (int64_t)(t - 1) * p.C * kD + (int64_t)j * kD + k);
    } else {
        const int64_t row = p.init_idx[(h * p.T + (t - 1)) * p.C + j];
        v = load_x1(p.X, p.in_dtype, h * p.x_stride + row * kD + k);
        if (t > 1) {  // the row of R^(t-1), by the residual kernels' TwoSum chain
            float e = 0.f;
            for (int st = 1; st < t; st++) {
                const int pj = min((int)p.pi[(int64_t)(h * p.T + st - 1) * p.cap + p.tok_off + row],
                                   p.C - 1);
                const float c = p.cent[h * p.cent_tstride + p.cent_off + (int64_t)(st - 1) * p.C * kD +
                                       (int64_t)pj * kD + k];
                float err;
                two_sum(v, -c, v, err);
                e = __fadd_rn(e, err);
            }
            const float r = __fadd_rn(v, e);
            rem = __fadd_rn(__fsub_rn(v, r), e);  // |e| is far below |v|: v - r is exact
            v = r;
        }
    }
    dst[k] = store_centroid_value(v, rem, p.cfmt);
}

cudaError_t launch_init_centroids(const QPlan &p, int t, cudaStream_t st) {
    return launch_kernel(k_init_centroids, dim3(p.C, p.H), dim3(kD), 0, st, p, t);
}

// --------------------------------------------------------------------------------------
// Centring vector for the GEMM operands.  Squared distances do not change when both
// operands are shifted by the same vector; shifting by a point near the data's centre
// keeps the fp16 operands small, and their rounding error is relative to their size.
// Stage 1 uses the mean of the initial centroids (C sample rows of X, or the warm-start
// table); later stages work on residuals whose mean is already ~0 and use 0.
// grid H, block 128.
// --------------------------------------------------------------------------------------
__global__ void k_centre(QPlan p, int t) {
    pdl_begin();
    const int h = blockIdx.x, k = threadIdx.x;
    float m = 0.f;
    if (t == 1) {
        const float *c = p.cent + h * p.cent_tstride + p.cent_off + k;
        float s = 0.f;
        for (int j = 0; j < p.C; j++) s += c[(int64_t)j * kD];
        m = s / (float)p.C;
    }
    p.mu[h * kD + k] = m;
}

cudaError_t launch_centre(const QPlan &p, int t, cudaStream_t st) {
    return launch_kernel(k_centre, dim3(p.H), dim3(kD), 0, st, p, t);
}

// --------------------------------------------------------------------------------------
// The stage input of channels 8*c8 .. 8*c8+7 of G tokens: x minus the earlier stages'
// assigned centroid rows C^(1)[pi^(1)_i], ..., C^(n)[pi^(n)_i], subtracted in that order by
// a packed TwoSum chain whose collected rounding errors are added back at the end, so each
// value is the fp32 number nearest the exact residual (the same value every kernel that
// rebuilds the stage input forms).  v holds X's values on entry.  NST: the number of earlier
// stages when it is fixed at compile time (every token's cluster indices, then every
// centroid row, are loaded before any arithmetic), or -1 for n given at run time.  An index
// >= C is clamped to C - 1 and reported through bad_index.
// --------------------------------------------------------------------------------------
template <int G, int NST>
__device__ __forceinline__ void stage_input8(const QPlan &p, int h, const int64_t (&i)[G],
                                             const bool (&valid)[G], int c8, int n,
                                             float2 (&v)[G][4], bool &bad_index) {
    if constexpr (NST != 0) {
        const float *tab = p.cent + h * p.cent_tstride + p.cent_off + c8 * 8;
        auto index = [&](int g, int st) {
            int j = 0;
            if (valid[g]) {
                j = p.pi[(int64_t)(h * p.T + st) * p.cap + p.tok_off + i[g]];
                if (j >= p.C) {
                    j = p.C - 1;
                    bad_index = true;
                }
            }
            return j;
        };
        float2 e[G][4];
#pragma unroll
        for (int g = 0; g < G; g++)
#pragma unroll
            for (int q = 0; q < 4; q++) e[g][q] = make_float2(0.f, 0.f);
        auto sub_row = [&](int g, float4 a, float4 b) {
            const float2 c[4] = {make_float2(a.x, a.y), make_float2(a.z, a.w), make_float2(b.x, b.y),
                                 make_float2(b.z, b.w)};
#pragma unroll
            for (int q = 0; q < 4; q++) {
                float2 t;
                v[g][q] = two_diff2(v[g][q], c[q], t);
                e[g][q] = __fadd2_rn(e[g][q], t);
            }
        };
        if constexpr (NST > 0) {
            int pj[G][NST];
#pragma unroll
            for (int g = 0; g < G; g++)
#pragma unroll
                for (int st = 0; st < NST; st++) pj[g][st] = index(g, st);
            float4 ca[G][NST], cb[G][NST];
#pragma unroll
            for (int g = 0; g < G; g++)
#pragma unroll
                for (int st = 0; st < NST; st++) {
                    const float4 *r = reinterpret_cast<const float4 *>(tab + ((int64_t)st * p.C + pj[g][st]) * kD);
                    ca[g][st] = __ldg(r);
                    cb[g][st] = __ldg(r + 1);
                }
#pragma unroll
            for (int st = 0; st < NST; st++)
#pragma unroll
                for (int g = 0; g < G; g++) sub_row(g, ca[g][st], cb[g][st]);
        } else {
            for (int st = 0; st < n; st++) {
#pragma unroll
                for (int g = 0; g < G; g++) {
                    const float4 *r = reinterpret_cast<const float4 *>(tab + ((int64_t)st * p.C + index(g, st)) * kD);
                    sub_row(g, __ldg(r), __ldg(r + 1));
                }
            }
        }
#pragma unroll
        for (int g = 0; g < G; g++)
#pragma unroll
            for (int q = 0; q < 4; q++) v[g][q] = __fadd2_rn(v[g][q], e[g][q]);
    }
}

// 8 channels of X as four pairs; the probe becomes NaN if one of them is not finite
// (x * 0 is NaN exactly for an infinity or a NaN)
__device__ __forceinline__ void load_x8_pairs(const QPlan &p, int64_t off, float2 (&v)[4], float2 &probe) {
    float x[8];
    load_x8(p.X, p.in_dtype, off, x);
#pragma unroll
    for (int q = 0; q < 4; q++) {
        v[q] = make_float2(x[2 * q], x[2 * q + 1]);
        probe = __ffma2_rn(v[q], make_float2(0.f, 0.f), probe);
    }
}

// --------------------------------------------------------------------------------------
// Residual preparation for stage t.  One thread per (token, 8 channels).
//   r      = fp32(x - sum_{s<t} C^(s)[pi^(s)_i]) via the TwoSum chain (one final rounding);
//            not stored: the kernels that need r again rebuild it by the same chain
//   A      = fp16(r - mu)                (tensor-core operand of the assignment)
//   rnorm  = ||r - mu||, fp32            (for the assignment's error margin)
//   dnorm  = ||A - (r - mu)||, fp32      (the same)
// grid (blocks per tensor, H), block 256 = 16 tokens x 16 chunks of 8 channels.
// --------------------------------------------------------------------------------------
constexpr int kPrepTokens = 64;

// G tokens per thread (16 threads per token, 8 channels each): all of a thread's loads are
// issued before its arithmetic, so that G rows are in flight per thread.  NST: earlier
// stages (0 at stage 1), -1 when given at run time (t - 1).
template <int G, int NST>
__global__ void __launch_bounds__(256) k_prep(QPlan p, int t) {
    pdl_begin();
    const int h = blockIdx.y;
    const int c8 = threadIdx.x & 15;
    const int64_t i0 = (int64_t)blockIdx.x * kPrepTokens;
    const int64_t i1 = min(p.N, i0 + kPrepTokens);
    float2 mu[4];
    {
        float m8[8];
        load_f8(p.mu + h * kD + c8 * 8, m8);
#pragma unroll
        for (int q = 0; q < 4; q++) mu[q] = make_float2(m8[2 * q], m8[2 * q + 1]);
    }
    float2 probe = make_float2(0.f, 0.f);
    bool bad_index = false;
#pragma unroll 1
    for (int64_t ib = i0; ib < i1; ib += 16 * G) {
        // the loop bound is uniform over the block, so every lane reaches the shuffles
        float2 v[G][4];
        int64_t ii[G];
        bool valid[G];
#pragma unroll
        for (int g = 0; g < G; g++) {
            ii[g] = ib + 16 * g + (threadIdx.x >> 4);
            valid[g] = ii[g] < i1;
            if (valid[g]) {
                load_x8_pairs(p, h * p.x_stride + ii[g] * kD + c8 * 8, v[g], probe);
            } else {
#pragma unroll
                for (int q = 0; q < 4; q++) v[g][q] = make_float2(0.f, 0.f);
            }
        }
        stage_input8<G, NST>(p, h, ii, valid, c8, t - 1, v, bad_index);
#pragma unroll
        for (int g = 0; g < G; g++) {
            // a = r - mu, its fp16 copy and the fp16 rounding error (exact), on pairs
            float2 ss = make_float2(0.f, 0.f), dd = ss;
            __align__(16) __half2 a16[4];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const float2 x = sub2(v[g][q], mu[q]);
                a16[q] = __float22half2_rn(x);
                const float2 dx = sub2(x, __half22float2(a16[q]));
                ss = __ffma2_rn(x, x, ss);
                dd = __ffma2_rn(dx, dx, dd);
            }
            if (valid[g])
                *reinterpret_cast<uint4 *>(p.A + ((int64_t)h * p.N + ii[g]) * kD + c8 * 8) =
                    *reinterpret_cast<uint4 *>(a16);
            float sss = __fadd_rn(ss.x, ss.y), ddd = __fadd_rn(dd.x, dd.y);
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) {
                sss += __shfl_xor_sync(0xffffffffu, sss, o);
                ddd += __shfl_xor_sync(0xffffffffu, ddd, o);
            }
            if (valid[g] && c8 == 0) {
                p.rnorm[h * p.N + ii[g]] = sqrtf(sss);
                p.dnorm[h * p.N + ii[g]] = sqrtf(ddd);
            }
        }
    }
    const bool finite = probe.x == probe.x && probe.y == probe.y;
    // one status update per block
    __shared__ int bad, bad_idx;
    if (threadIdx.x == 0) bad = 0, bad_idx = 0;
    __syncthreads();
    if (!finite) bad = 1;
    if (bad_index) bad_idx = 1;
    __syncthreads();
    if (threadIdx.x == 0) {
        if (bad) or_status(p.status, QVG_DEV_NONFINITE);
        if (bad_idx) or_status(p.status, QVG_DEV_BAD_INDEX);
    }
}

// Later stages: one token per 16-thread group and pass, passes software-pipelined: a pass
// issues its tokens' earlier centroid rows (their cluster indices are already in registers)
// together with the next pass's X rows and cluster indices, then does its own arithmetic,
// so that each pass waits on one round of loads instead of two in a row.
constexpr int kPrepPipeTokens = 256;

template <int NST>
__global__ void __launch_bounds__(256) k_prep_pipe(QPlan p, int t) {
    pdl_begin();
    static_assert(NST > 0, "stage 1 has nothing to subtract");
    const int h = blockIdx.y;
    const int c8 = threadIdx.x & 15;
    const int64_t i0 = (int64_t)blockIdx.x * kPrepPipeTokens;
    const int64_t i1 = min(p.N, i0 + kPrepPipeTokens);
    float2 mu[4];
    {
        float m8[8];
        load_f8(p.mu + h * kD + c8 * 8, m8);
#pragma unroll
        for (int q = 0; q < 4; q++) mu[q] = make_float2(m8[2 * q], m8[2 * q + 1]);
    }
    const float *tab = p.cent + h * p.cent_tstride + p.cent_off + c8 * 8;
    float2 probe = make_float2(0.f, 0.f);
    bool bad_index = false;
    struct Pass {
        int64_t i;
        bool valid;
        float2 x[4];
        int pj[NST];
    };
    auto load_pass = [&](int64_t ib, Pass &q) {
        q.i = ib + (threadIdx.x >> 4);
        q.valid = q.i < i1;
        if (q.valid) {
            load_x8_pairs(p, h * p.x_stride + q.i * kD + c8 * 8, q.x, probe);
        } else {
#pragma unroll
            for (int k = 0; k < 4; k++) q.x[k] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int st = 0; st < NST; st++) {
            int j = 0;
            if (q.valid) {
                j = p.pi[(int64_t)(h * p.T + st) * p.cap + p.tok_off + q.i];
                bad_index |= j >= p.C;
                j = min(j, p.C - 1);
            }
            q.pj[st] = j;
        }
    };
    Pass cur;
    load_pass(i0, cur);
#pragma unroll 1
    for (int64_t ib = i0; ib < i1; ib += 16) {
        // this pass's earlier centroid rows, then the next pass's inputs
        float4 ca[NST], cb[NST];
#pragma unroll
        for (int st = 0; st < NST; st++) {
            const float4 *r = reinterpret_cast<const float4 *>(tab + ((int64_t)st * p.C + cur.pj[st]) * kD);
            ca[st] = __ldg(r);
            cb[st] = __ldg(r + 1);
        }
        const bool more = ib + 16 < i1;  // uniform over the block
        Pass nxt;
        if (more) load_pass(ib + 16, nxt);
        // r = x - C^(1)[pi^(1)] - ... by the TwoSum chain, one final rounding
        float2 v[4], e[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            v[k] = cur.x[k];
            e[k] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int st = 0; st < NST; st++) {
            const float2 c[4] = {make_float2(ca[st].x, ca[st].y), make_float2(ca[st].z, ca[st].w),
                                 make_float2(cb[st].x, cb[st].y), make_float2(cb[st].z, cb[st].w)};
#pragma unroll
            for (int k = 0; k < 4; k++) {
                float2 tt;
                v[k] = two_diff2(v[k], c[k], tt);
                e[k] = __fadd2_rn(e[k], tt);
            }
        }
        // a = r - mu, its fp16 copy and the fp16 rounding error (exact), on pairs
        float2 ss = make_float2(0.f, 0.f), dd = ss;
        __align__(16) __half2 a16[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const float2 x = sub2(__fadd2_rn(v[k], e[k]), mu[k]);
            a16[k] = __float22half2_rn(x);
            const float2 dx = sub2(x, __half22float2(a16[k]));
            ss = __ffma2_rn(x, x, ss);
            dd = __ffma2_rn(dx, dx, dd);
        }
        if (cur.valid)
            *reinterpret_cast<uint4 *>(p.A + ((int64_t)h * p.N + cur.i) * kD + c8 * 8) =
                *reinterpret_cast<uint4 *>(a16);
        float sss = __fadd_rn(ss.x, ss.y), ddd = __fadd_rn(dd.x, dd.y);
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) {
            sss += __shfl_xor_sync(0xffffffffu, sss, o);
            ddd += __shfl_xor_sync(0xffffffffu, ddd, o);
        }
        if (cur.valid && c8 == 0) {
            p.rnorm[h * p.N + cur.i] = sqrtf(sss);
            p.dnorm[h * p.N + cur.i] = sqrtf(ddd);
        }
        if (more) cur = nxt;
    }
    const bool finite = probe.x == probe.x && probe.y == probe.y;
    // one status update per block
    __shared__ int bad, bad_idx;
    if (threadIdx.x == 0) bad = 0, bad_idx = 0;
    __syncthreads();
    if (!finite) bad = 1;
    if (bad_index) bad_idx = 1;
    __syncthreads();
    if (threadIdx.x == 0) {
        if (bad) or_status(p.status, QVG_DEV_NONFINITE);
        if (bad_idx) or_status(p.status, QVG_DEV_BAD_INDEX);
    }
}

cudaError_t launch_prep(const QPlan &p, int t, cudaStream_t st) {
    const dim3 grid((unsigned)((p.N + kPrepTokens - 1) / kPrepTokens), p.H);
    const dim3 pgrid((unsigned)((p.N + kPrepPipeTokens - 1) / kPrepPipeTokens), p.H);
    switch (t - 1) {
        case 0: return launch_kernel(k_prep<4, 0>, grid, dim3(256), 0, st, p, t);
        case 1: return launch_kernel(k_prep_pipe<1>, pgrid, dim3(256), 0, st, p, t);
        case 2: return launch_kernel(k_prep_pipe<2>, pgrid, dim3(256), 0, st, p, t);
        case 3: return launch_kernel(k_prep_pipe<3>, pgrid, dim3(256), 0, st, p, t);
        default: return launch_kernel(k_prep<1, -1>, grid, dim3(256), 0, st, p, t);
    }
}

// --------------------------------------------------------------------------------------
// Assignment operands of the stage's initial centroids, per centroid j (c = C_j - mu):
//   B[j]   = fp16(c), the tensor-core operand;
//   Bx[j]  = the offset -||c||^2 / 2 as three tf32 parts (h, m, l, 0, ...);
//   cnd[j] = (||c||^2, ||fp16(c) - c||), for the assignment's error bound.
// The padded rows j in [C, Cpad) get the offset -2^100, so their scores never win.
// grid (Cpad, H), block 128 (one thread per channel).
// --------------------------------------------------------------------------------------
__device__ __forceinline__ void write_offset_row(const QPlan &p, int h, int j, int lane, float cn) {
    float oh, om, ol;
    tf32_split3(-0.5f * cn, oh, om, ol);
    p.Bx[((int64_t)h * p.Cpad + j) * kOffsetRow + lane] =
        lane == 0 ? oh : lane == 1 ? om : lane == 2 ? ol : 0.f;
}

__global__ void k_centroid_planes(QPlan p, int t) {
    pdl_begin();
    const int j = blockIdx.x, h = blockIdx.y, k = threadIdx.x;
    if (j >= p.C) {  // a padded column (the whole block takes this branch)
        if (k < kOffsetRow) p.Bx[((int64_t)h * p.Cpad + j) * kOffsetRow + k] = k == 0 ? -0x1p100f : 0.f;
        return;
    }
    const float v = p.cent[h * p.cent_tstride + p.cent_off + (int64_t)(t - 1) * p.C * kD +
                           (int64_t)j * kD + k];
    __shared__ float red[4][2];
    const float ct = __fsub_rn(v, p.mu[h * kD + k]);
    const __half hi = __float2half_rn(ct);
    p.B[((int64_t)h * p.Cpad + j) * kD + k] = hi;
    const float dv = __fsub_rn(ct, __half2float(hi));  // exact
    float ss = ct * ct, dd = dv * dv;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
        dd += __shfl_xor_sync(0xffffffffu, dd, o);
    }
    if ((k & 31) == 0) {
        red[k >> 5][0] = ss;
        red[k >> 5][1] = dd;
    }
    __syncthreads();
    if (k < 32) {
        const float cn = (red[0][0] + red[1][0]) + (red[2][0] + red[3][0]);
        write_offset_row(p, h, j, k, cn);
        if (k == 0)
            p.cnd[(int64_t)h * p.Cpad + j] =
                make_float2(cn, sqrtf((red[0][1] + red[1][1]) + (red[2][1] + red[3][1])));
    }
}

cudaError_t launch_centroid_planes(const QPlan &p, int t, cudaStream_t st) {
    return launch_kernel(k_centroid_planes, dim3(p.Cpad, p.H), dim3(kD), 0, st, p, t);
}

// --------------------------------------------------------------------------------------
// Centroid update: C_j = mean of the residual rows assigned to j, for every non-empty j.
//
// 1. A stable counting sort groups the token indices by cluster, increasing within a
//    cluster (histogram per block of 256 tokens, scans, scatter with in-block ranks).
// 2. The sorted positions are cut into chunks of 32; one warp adds each run of equal
//    cluster inside its chunk with error-free TwoSum accumulation (sum + running error,
//    both fp32) in sorted order (lane l holds channels 4l..4l+3).
// 3. One warp per cluster adds its pieces (one, or one per chunk it spans) in chunk
//    order, forms the mean, and writes the centroid with the fp16 GEMM planes of
//    C_j - mu and ||C_j - mu||^2 for the next assignment; empty clusters keep their
//    centroid.
// Every reduction has a fixed order, so repeated runs give identical bits; the
// compensated sums carry about twice fp32's precision.
// --------------------------------------------------------------------------------------
__device__ __forceinline__ void acc_two_sum(float &s, float &e, float x) {
    float err;
    two_sum(s, x, s, err);
    e = __fadd_rn(e, err);
}

// The sort's items.  delta = 0 (a stage's first round): every token, keyed by its cluster.
// delta = 1 (later rounds): for every token whose cluster changed since the previous round,
// a leave item keyed by its old cluster and an enter item keyed by its new one; within a
// token block and cluster the leave items come first, each kind in token order, so the
// order is fixed.
struct SortKeys {
    int leave, enter;  // cluster keys of the token's items (-1: none)
    bool changed;
    bool bad;          // the stored index is out of range
};
__device__ __forceinline__ SortKeys sort_keys(const QPlan &p, int h, int t, int64_t i, int delta) {
    SortKeys k{-1, -1, false, false};
    if (i >= p.N) return k;
    const int j = p.pi[(int64_t)(h * p.T + t - 1) * p.cap + p.tok_off + i];
    if (j >= p.C) {  // reported by the histogram; the token takes no part
        k.bad = true;
        return k;
    }
    if (!delta) {
        k.enter = j;
        return k;
    }
    const int jo = p.pi_prev[(int64_t)h * p.N + i];
    // (an earlier round's index is < C unless that round had an out-of-range index, which
    // is reported; keys stay < C so that no position leaves its tensor's items)
    if (jo != j && jo < p.C) {
        k.leave = jo;
        k.enter = j;
        k.changed = true;
    }
    return k;
}

// Sort blocks per CTA of the histogram: each thread reads its token's indices in all of
// them before any is counted, so those reads overlap.
constexpr int kSortSB = 4;

// Block histograms (one per sort block of kSortBlock tokens), and the cluster totals: one
// atomic per cluster per CTA, the sum over its blocks.
__global__ void __launch_bounds__(kSortBlock) k_sort_hist(QPlan p, int t, int delta) {
    pdl_begin();
    __shared__ int hist[kSortSB][kMaxC];
    __shared__ int lsum[kMaxC];  // leave items of the CTA's blocks per cluster
    const int h = blockIdx.y, tl = threadIdx.x;
    const int bb = blockIdx.x * kSortSB;  // the CTA's first sort block
    for (int x = tl; x < kSortSB * kMaxC; x += kSortBlock) (&hist[0][0])[x] = 0;
    for (int j = tl; j < kMaxC; j += kSortBlock) lsum[j] = 0;
    SortKeys k[kSortSB];
    bool bad = false;
#pragma unroll
    for (int u = 0; u < kSortSB; u++) {
        k[u] = sort_keys(p, h, t, (int64_t)(bb + u) * kSortBlock + tl, delta);
        bad |= k[u].bad;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kSortSB; u++) {
        if (k[u].enter >= 0) atomicAdd(&hist[u][k[u].enter], 1);
        if (k[u].leave >= 0) {
            atomicAdd(&hist[u][k[u].leave], 1);
            atomicAdd(&lsum[k[u].leave], 1);
        }
    }
    if (__any_sync(0xffffffffu, bad) && (tl & 31) == 0) or_status(p.status, QVG_DEV_BAD_INDEX);
    __syncthreads();
    for (int j = tl; j < p.C; j += kSortBlock) {
        int tot = 0;
#pragma unroll
        for (int u = 0; u < kSortSB; u++) {
            const int v = hist[u][j];
            if (bb + u < p.nsb) p.blockoff[((int64_t)h * p.nsb + bb + u) * p.C + j] = v;
            tot += v;
        }
        if (tot) atomicAdd(p.counts + h * p.C + j, tot);  // cluster totals (zero on entry)
        if (lsum[j]) atomicAdd(p.dleave + h * p.C + j, lsum[j]);
    }
}

// Offsets of the counting sort.  grid (C/32 cluster groups, H), block 256: lane = cluster
// of the group, warp w = a slice of the token blocks.  offs[j] = sum of the totals of the
// clusters before j; blockoff[b][j] (in place, over the block histogram) = offs[j] + the
// items of cluster j in the blocks before b; items = the tensor's total.
__global__ void __launch_bounds__(256) k_sort_scan(QPlan p) {
    pdl_begin();
    constexpr int NW = 8;
    __shared__ int tot[kMaxC];
    __shared__ int wsum[NW][32];
    const int h = blockIdx.y, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int j = blockIdx.x * 32 + lane;
    // inclusive scan of the cluster totals of this tensor
    const int x = threadIdx.x;
    tot[x] = x < p.C ? p.counts[h * p.C + x] : 0;
    __syncthreads();
    for (int o = 1; o < kMaxC; o <<= 1) {
        const int a1 = x >= o ? tot[x - o] : 0;
        __syncthreads();
        tot[x] += a1;
        __syncthreads();
    }
    if (blockIdx.x == 0 && x == 0) p.items[h] = tot[kMaxC - 1];
    int *bh = p.blockoff + (int64_t)h * p.nsb * p.C;
    const int per = (p.nsb + NW - 1) / NW;
    const int b0 = w * per, b1 = min(p.nsb, b0 + per);
    int local = 0;
    if (j < p.C) {
#pragma unroll 8
        for (int b = b0; b < b1; b++) local += bh[(int64_t)b * p.C + j];
    }
    wsum[w][lane] = local;
    __syncthreads();
    if (j < p.C) {
        const int off = tot[j] - (j < p.C ? p.counts[h * p.C + j] : 0);
        if (w == 0) p.offs[h * p.C + j] = off;
        int run = off;
        for (int w2 = 0; w2 < w; w2++) run += wsum[w2][lane];
        for (int b = b0; b < b1; b++) {
            const int v = bh[(int64_t)b * p.C + j];
            bh[(int64_t)b * p.C + j] = run;
            run += v;
        }
    }
}

// Writes the block's items to their sorted positions (the leave items of a cluster before
// its enter items, each in token order), and the round's assignment into pi_prev.
// A CTA holds kScatterGroups sort blocks, one per group of kSortBlock threads.
constexpr int kScatterGroups = 2;
__global__ void __launch_bounds__(kSortBlock * kScatterGroups) k_sort_scatter(QPlan p, int t, int delta) {
    pdl_begin();
    constexpr int NW = kSortBlock / 32;
    // leave / enter items of each cluster per warp, per group (at most 32: one byte each)
    __shared__ __align__(16) uint8_t wl_s[kScatterGroups][NW][kMaxC], we_s[kScatterGroups][NW][kMaxC];
    __shared__ int bo_s[kScatterGroups][kMaxC];  // the block's first position per cluster
    const int h = blockIdx.y, g = threadIdx.x / kSortBlock, tl = threadIdx.x % kSortBlock;
    const int b = blockIdx.x * kScatterGroups + g;
    uint8_t (*wl)[kMaxC] = wl_s[g], (*we)[kMaxC] = we_s[g];
    // the block's offsets, read beside its tokens' indices (neither waits for the other)
    if (tl < p.C && b < p.nsb) bo_s[g][tl] = p.blockoff[((int64_t)h * p.nsb + b) * p.C + tl];
    const int lane = tl & 31, w = tl >> 5;
    const int64_t i = (int64_t)b * kSortBlock + tl;  // >= N for a group past the last block
    const SortKeys k = sort_keys(p, h, t, i, delta);
    static_assert(2 * NW * kMaxC == kSortBlock * 16, "one 16-byte store per thread");
    constexpr int kVec = NW * kMaxC / 16;  // 16-byte pieces of one array
    reinterpret_cast<uint4 *>(tl < kVec ? &wl[0][0] : &we[0][0])[tl % kVec] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    const unsigned sl = __match_any_sync(0xffffffffu, k.leave);
    const unsigned se = __match_any_sync(0xffffffffu, k.enter);
    const unsigned below = (1u << lane) - 1u;
    const int rl = __popc(sl & below), re = __popc(se & below);  // earlier lanes, same key
    if (k.leave >= 0 && rl == 0) wl[w][k.leave] = (uint8_t)__popc(sl);
    if (k.enter >= 0 && re == 0) we[w][k.enter] = (uint8_t)__popc(se);
    __syncthreads();
    const int *bo = bo_s[g];
    int *ids = p.ids + (int64_t)h * p.icap;
    uint8_t *cid = p.cid + (int64_t)h * p.icap;
    if (k.leave >= 0) {
        int pos = bo[k.leave] + rl;
        for (int w2 = 0; w2 < w; w2++) pos += wl[w2][k.leave];
        ids[pos] = (int)i | (int)0x80000000u;
        cid[pos] = (uint8_t)k.leave;
    }
    if (k.enter >= 0) {
        int pos = bo[k.enter] + re;
        for (int w2 = 0; w2 < NW; w2++) pos += wl[w2][k.enter];  // the block's leave items first
        for (int w2 = 0; w2 < w; w2++) pos += we[w2][k.enter];
        ids[pos] = (int)i;
        cid[pos] = (uint8_t)k.enter;
        if (!delta || k.changed) p.pi_prev[(int64_t)h * p.N + i] = (uint8_t)k.enter;
    }
}

// Mean of S + E over n rows: the quotient of S corrected by the remainder and by E.
__device__ __forceinline__ float mean_of(float S, float E, float n) {
    const float q0 = __fdiv_rn(S, n);
    const float r = __fadd_rn(__fmaf_rn(-q0, n, S), E);
    return __fadd_rn(q0, __fdiv_rn(r, n));
}

// The mean of a compensated sum (S, E) over n members in the stored format: the fp32 mean
// and the sign of what it leaves out decide the rounding.
__device__ __forceinline__ float stored_mean(float S, float E, float n, int fmt) {
    const float m = mean_of(S, E, n);
    if (fmt == QVG_CENTROIDS_F32) return m;
    return store_centroid_value(m, __fadd_rn(__fmaf_rn(-m, n, S), E), fmt);
}

// New centroid row j (lane l: channels 4l..4l+3), and its assignment operands (as
// k_centroid_planes writes them) if requested.
__device__ __forceinline__ void write_centroid(const QPlan &p, int h, int t, int j, int lane,
                                               bool set, float4 cv, bool planes, float4 mu) {
    float *c = p.cent + h * p.cent_tstride + p.cent_off + (int64_t)(t - 1) * p.C * kD +
               (int64_t)j * kD + 4 * lane;
    if (set)
        *reinterpret_cast<float4 *>(c) = cv;
    else
        cv = *reinterpret_cast<float4 *>(c);
    if (!planes) return;
    const float ct[4] = {__fsub_rn(cv.x, mu.x), __fsub_rn(cv.y, mu.y), __fsub_rn(cv.z, mu.z),
                         __fsub_rn(cv.w, mu.w)};
    __align__(8) __half hi[4];
    float ss = 0.f, dd = 0.f;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        hi[k] = __float2half_rn(ct[k]);
        const float dv = __fsub_rn(ct[k], __half2float(hi[k]));  // exact
        ss = __fmaf_rn(ct[k], ct[k], ss);
        dd = __fmaf_rn(dv, dv, dd);
    }
    *reinterpret_cast<uint2 *>(p.B + ((int64_t)h * p.Cpad + j) * kD + 4 * lane) =
        *reinterpret_cast<uint2 *>(hi);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
        dd += __shfl_xor_sync(0xffffffffu, dd, o);
    }
    write_offset_row(p, h, j, lane, ss);
    if (lane == 0) p.cnd[(int64_t)h * p.Cpad + j] = make_float2(ss, sqrtf(dd));
}

// Cluster sums over chunks of 32 cluster-sorted items.  The rows of each run (same
// cluster) are added with TwoSum in sorted order, a leave item's row negated (exactly).  A run that is a whole cluster leaves its
// (sum, error) in the cluster's slot; a run that crosses the chunk's start or end leaves it
// in the chunk's first / last slot.  k_cluster_finalize turns them into means.  Stage 1
// (nothing to subtract) fits 64 registers, so four CTAs share an SM; the second stage (one
// subtraction) three, later ones, with the longer chain, two.
//
// The summed rows are the stage input R^(t-1): X itself at stage 1, later a residual that
// is not stored but rebuilt here from X and the earlier stages' centroid rows (L2-resident)
// by a TwoSum chain.  The chain's running difference and its collected rounding errors both
// enter the compensated sum, so a mean is that of the exact residuals and rounds as the
// fp64 reference's does (not the mean of fp32-rounded residuals, which is off by up to half
// an fp32 ulp of the largest member and can flip a near tie).  Reaching a row takes
// three dependent loads (its id from the sort, its earlier clusters, then X and the
// centroid rows), so the kernel is built to keep many of them in flight:
//   * persistent warps, each striding over the chunks of all tensors; lane m holds sorted
//     position m of a chunk (its token, cluster and earlier clusters), and the next chunk's
//     ids and pi bytes are read while the current chunk is summed;
//   * the X rows reach shared memory by TMA gathers (or bulk copies that each lane issues
//     for its own position), eight rows to a group on one mbarrier, two groups in flight
//     ahead of the sums, running on from one chunk into the next;
//   * a lane reads its four channels of each earlier stage's centroid row (16 bytes, from
//     L2, where the tables stay) with one vector load while it sums, so the shared-memory
//     ring holds X rows only and more warps fit on an SM to keep those loads in flight.
constexpr int kBulkGroup = 8;  // rows a group (one mbarrier phase)
__host__ __device__ constexpr int bulk_xbytes(int src) { return src == 1 ? 512 : 256; }
// warps per CTA: as many as fit 96 KB of row slots (two groups a warp), at most 8
__host__ __device__ inline int bulk_warps(int src) {
    const int w = 98304 / (2 * kBulkGroup * bulk_xbytes(src));
    return w > 8 ? 8 : (w < 1 ? 1 : w);
}

__device__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t n = 0; n < (1u << 22); n++) {
        if (mbar_try_suspend(bar, parity)) return true;
        if ((n & 15u) == 15u && global_ns() - t0 > 2000000000ull) break;
    }
    return false;
}

// one chunk as the warp holds it: lane m's values are those of sorted position m
struct SumChunk {
    int h, k, nk;           // tensor, chunk, positions in the chunk
    int id, cl;             // the lane's token and cluster (cl = -1 past the end)
    uint32_t neg;           // bit m: position m is a leave item (its row is subtracted)
    int xrow, crow;         // row of the token in the X row view; first row of the tables
    int c_prev, c_next;     // clusters just before and after the chunk (-1: none)
    uint32_t pk0, pk1;      // the token's earlier clusters, 8 bits a stage
    uint32_t brk;           // bit m: position m begins a new run
};

template <int SRC, int TP>  // SRC: X dtype (0 bf16, 1 fp32, 3 fp16); TP: t - 1 (0..3), or -1
__global__ void __launch_bounds__(256, TP == 0 ? 4 : (TP == 1 ? 3 : 2))
    k_chunk_sums(const __grid_constant__ CUtensorMap tmX, QPlan p, int t, int gather) {
    pdl_begin();
    static_assert(kChunk == 32, "one sorted position per lane");
    constexpr int XB = bulk_xbytes(SRC);
    extern __shared__ __align__(128) uint8_t bulk_smem[];
    const int tp = TP >= 0 ? TP : t - 1;
    constexpr int row_bytes = XB;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int wpc = blockDim.x >> 5;
    const int total = p.H * p.nchunk;
    const int nw = gridDim.x * wpc;
    // the warp's chunks: every nw-th of all tensors' chunk slots, skipping those past the
    // tensor's item count (in a stage's first round half the slots, in later ones most)
    auto next_chunk = [&](int c) {
        while (c < total) {
            const int h = c / p.nchunk;
            if ((int64_t)(c - h * p.nchunk) * kChunk < (int64_t)p.items[h]) break;
            // the rest of tensor h is empty too: on to this warp's first slot in tensor h + 1
            c += ((h + 1) * p.nchunk - c + nw - 1) / nw * nw;
        }
        return c;
    };
    int ci = next_chunk(blockIdx.x * wpc + wid);
    if (ci >= total) return;  // no CTA-wide barrier below
    const uint32_t bars = smem_u32(bulk_smem) + wid * 16;  // group n waits on bars + 8 (n & 1)
    const uint32_t ring = smem_u32(bulk_smem) + 128 + wid * 2 * kBulkGroup * row_bytes;
    const uint8_t *ring_g = bulk_smem + 128 + wid * 2 * kBulkGroup * row_bytes;
    if (lane == 0) {
        mbar_init(bars, 1);
        mbar_init(bars + 8, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();

    auto fetch = [&](int c, SumChunk &m) {
        m.h = c / p.nchunk;
        m.k = c - m.h * p.nchunk;
        const int64_t c0 = (int64_t)m.k * kChunk;
        const int64_t n_items = p.items[m.h];
        m.nk = (int)min((int64_t)kChunk, n_items - c0);
        const int64_t base = (int64_t)m.h * p.icap + c0;
        const bool mine = lane < m.nk;
        const int raw = mine ? p.ids[base + lane] : 0;
        m.id = raw & 0x7FFFFFFF;
        m.neg = __ballot_sync(0xffffffffu, raw < 0);
        m.cl = mine ? (int)p.cid[base + lane] : -1;
        m.xrow = (int)(m.h * (p.x_stride / kD)) + m.id;
        m.crow = (int)((m.h * p.cent_tstride + p.cent_off) / kD);
        m.c_prev = m.k > 0 ? (int)p.cid[base - 1] : -1;
        m.c_next = c0 + m.nk < n_items ? (int)p.cid[base + m.nk] : -1;
    };
    auto fetch_pi = [&](SumChunk &m) {  // needs m.id; also finds the run starts
        m.pk0 = m.pk1 = 0u;
        if (lane < m.nk) {
            for (int st = 0; st < tp; st++) {
                const uint32_t b = p.pi[(int64_t)(m.h * p.T + st) * p.cap + p.tok_off + m.id];
                if (st < 4) m.pk0 |= b << (8 * st);
                else m.pk1 |= b << (8 * (st - 4));
            }
        }
        int pc = __shfl_up_sync(0xffffffffu, m.cl, 1);
        if (lane == 0) pc = -2;
        m.brk = __ballot_sync(0xffffffffu, lane < m.nk && m.cl != pc);
    };
    auto n_groups = [](const SumChunk &m) { return (m.nk + kBulkGroup - 1) / kBulkGroup; };

    uint32_t n_issued = 0, n_done = 0;  // groups issued / summed by this warp so far
    // Group g of chunk m (positions 8g..8g+7) goes to half (n_issued & 1) of the warp's
    // slots: its X rows (XB bytes each).
    auto issue = [&](const SumChunk &m, int g) {
        const int n_rows = min(kBulkGroup, m.nk - g * kBulkGroup);
        const int half = n_issued & 1;
        const uint32_t bar = bars + 8 * half;
        const uint32_t hb = ring + half * kBulkGroup * row_bytes;
        if (gather) {
            // four rows per TMA gather; a short last group repeats its last row
            const int n4 = (n_rows + 3) >> 2;
            if (lane == 0) mbar_expect_tx(bar, (uint32_t)(n4 * 4 * row_bytes));
            __syncwarp();
            for (int u4 = 0; u4 < n4; u4++) {
                int src[4];
#pragma unroll
                for (int k = 0; k < 4; k++) src[k] = min(g * kBulkGroup + 4 * u4 + k, m.nk - 1);
                int r[4];
#pragma unroll
                for (int k = 0; k < 4; k++) r[k] = __shfl_sync(0xffffffffu, m.xrow, src[k]);
                if (lane == 0) tma_gather4(hb + 4 * u4 * XB, &tmX, 0, r[0], r[1], r[2], r[3], bar);
            }
        } else {
            // one bulk copy per row, issued by the lane that holds the row
            if (lane == 0) mbar_expect_tx(bar, (uint32_t)(n_rows * row_bytes));
            __syncwarp();
            if (lane >= g * kBulkGroup && lane < g * kBulkGroup + n_rows) {
                const int u = lane & (kBulkGroup - 1);
                bulk_g2s(hb + u * XB,
                         static_cast<const char *>(p.X) + (m.h * p.x_stride + (int64_t)m.id * kD) * (XB / kD),
                         XB, bar);
            }
        }
        n_issued++;
    };

    SumChunk cur, nxt;
    fetch(ci, cur);
    fetch_pi(cur);
    bool has_next = false;
    // the issue pointer: group ip_g of the current (ip_next = 0) or the next chunk
    int ip_next = 0, ip_g = 0;
    auto issue_next = [&]() {
        if (!ip_next) {
            if (ip_g < n_groups(cur)) {
                issue(cur, ip_g++);
                return;
            }
            ip_next = 1;
            ip_g = 0;
        }
        if (has_next && ip_g < n_groups(nxt)) issue(nxt, ip_g++);
    };
    issue_next();
    issue_next();
    for (;;) {
        const int cn = next_chunk(ci + nw);
        has_next = cn < total;
        if (has_next) {
            fetch(cn, nxt);
            fetch_pi(nxt);
        }
        // keep two groups in flight (the current chunk may have had fewer than two)
        while (n_issued < n_done + 2) {
            const uint32_t before = n_issued;
            issue_next();
            if (n_issued == before) break;
        }
        // the running (sum, error) pair of the current run, channels (0,1) and (2,3)
        float2 s01 = make_float2(0.f, 0.f), s23 = s01, e01 = s01, e23 = s01;
        int run_c = __shfl_sync(0xffffffffu, cur.cl, 0), run_start = 0;
        auto stash = [&](int end) {
            const bool whole = (run_start > 0 || cur.c_prev != run_c) && (end < cur.nk || cur.c_next != run_c);
            float *dst = whole ? p.wsum + ((int64_t)cur.h * p.C + run_c) * 2 * kD
                               : p.psum + (((int64_t)cur.h * p.nchunk + cur.k) * 2 + (run_start == 0 ? 0 : 1)) * 2 * kD;
            reinterpret_cast<float4 *>(dst)[lane] = make_float4(s01.x, s01.y, s23.x, s23.y);
            reinterpret_cast<float4 *>(dst + kD)[lane] = make_float4(e01.x, e01.y, e23.x, e23.y);
        };
        // Adds the lane's four channels of the row in slot u, as the stage input, to the
        // running (sum, error) pair.  From the second stage on the stage input is
        // x - C^(1)[pi^(1)] - ..., formed by a TwoSum chain as d + r with d the running
        // fp32 difference and r the sum of the chain's rounding errors; d goes through the
        // compensated sum and r is added to its error term, so the sum is that of the exact
        // residuals (to about twice fp32's precision), not of their fp32 roundings.
        auto add_row = [&](const uint8_t *hs, int u, uint32_t q0, uint32_t q1, uint32_t sg) {
            const uint8_t *slot = hs + u * XB;  // the X row
            float2 v01, v23;
            if constexpr (SRC == 0) {
                const uint2 w = *reinterpret_cast<const uint2 *>(slot + lane * 8);
                v01 = make_float2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u));
                v23 = make_float2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
            } else if constexpr (SRC == 3) {
                const uint2 w = *reinterpret_cast<const uint2 *>(slot + lane * 8);
                v01 = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
                v23 = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
            } else {
                const float4 w = *reinterpret_cast<const float4 *>(slot + lane * 16);
                v01 = make_float2(w.x, w.y);
                v23 = make_float2(w.z, w.w);
            }
            auto flip = [sg](float2 a) {  // negation of a leave item's values (exact)
                return make_float2(__uint_as_float(__float_as_uint(a.x) ^ sg),
                                   __uint_as_float(__float_as_uint(a.y) ^ sg));
            };
            if constexpr (TP == 0) {
                acc_two_sum2(s01, e01, flip(v01));
                acc_two_sum2(s23, e23, flip(v23));
            } else {
                float2 r01 = make_float2(0.f, 0.f), r23 = r01;
                auto chain = [&](int st) {  // subtract the row of stage st + 1
                    const int pj = min((int)(((st < 4 ? q0 : q1) >> (8 * (st & 3))) & 255u), p.C - 1);
                    const float4 c = __ldg(reinterpret_cast<const float4 *>(
                        p.cent + (int64_t)(cur.crow + st * p.C + pj) * kD) + lane);
                    float2 t01, t23;
                    v01 = two_diff2(v01, make_float2(c.x, c.y), t01);
                    v23 = two_diff2(v23, make_float2(c.z, c.w), t23);
                    r01 = __fadd2_rn(r01, t01);
                    r23 = __fadd2_rn(r23, t23);
                };
                if constexpr (TP > 0) {
#pragma unroll
                    for (int st = 0; st < TP; st++) chain(st);
                } else {
                    for (int st = 0; st < tp; st++) chain(st);
                }
                acc_two_sum2(s01, e01, flip(v01));
                acc_two_sum2(s23, e23, flip(v23));
                e01 = __fadd2_rn(e01, flip(r01));
                e23 = __fadd2_rn(e23, flip(r23));
            }
        };
        const uint32_t starts = cur.brk & ~1u;  // position 0 opens the first run above
        const int ng = n_groups(cur);
        for (int g = 0; g < ng; g++) {
            const int half = n_done & 1;
            if (!mbar_wait_bounded(bars + 8 * half, (n_done >> 1) & 1)) {
                // a copy that never landed: report it, let the other group's copies finish
                if (lane == 0) or_status(p.status, QVG_DEV_TIMEOUT);
                if (n_issued > n_done + 1) mbar_wait_bounded(bars + 8 * (half ^ 1), ((n_done + 1) >> 1) & 1);
                return;
            }
            const int n_rows = min(kBulkGroup, cur.nk - g * kBulkGroup);
            const uint8_t *gslots = ring_g + half * kBulkGroup * row_bytes;
            if (n_rows == kBulkGroup && ((starts >> (g * kBulkGroup)) & 0xFFu) == 0u) {
                // a full group inside one run (the usual case)
#pragma unroll
                for (int u = 0; u < kBulkGroup; u++) {
                    const int m = g * kBulkGroup + u;
                    add_row(gslots, u, TP != 0 ? __shfl_sync(0xffffffffu, cur.pk0, m) : 0u,
                            TP < 0 ? __shfl_sync(0xffffffffu, cur.pk1, m) : 0u,
                            ((cur.neg >> m) & 1u) << 31);
                }
            } else {
#pragma unroll 1
                for (int u = 0; u < n_rows; u++) {
                    const int m = g * kBulkGroup + u;
                    if ((starts >> m) & 1u) {  // warp-uniform
                        stash(m);
                        run_c = __shfl_sync(0xffffffffu, cur.cl, m);
                        run_start = m;
                        s01 = s23 = e01 = e23 = make_float2(0.f, 0.f);
                    }
                    add_row(gslots, u, TP != 0 ? __shfl_sync(0xffffffffu, cur.pk0, m) : 0u,
                            TP < 0 ? __shfl_sync(0xffffffffu, cur.pk1, m) : 0u,
                            ((cur.neg >> m) & 1u) << 31);
                }
            }
            n_done++;
            __syncwarp();  // every lane has read the group's slots before they are refilled
            issue_next();
        }
        stash(cur.nk);
        if (!has_next) break;
        cur = nxt;
        ci = cn;
        if (!ip_next) ip_g = 0;  // every group of the old chunk was issued
        ip_next = 0;
        has_next = false;
    }
}

template <int SRC, int TP>
static cudaError_t launch_sums(const QPlan &p, const AssignMaps *maps, int t, int num_sms,
                               cudaStream_t st) {
    const int tp = TP >= 0 ? TP : t - 1;
    const int wpc = bulk_warps(SRC);
    const int smem = 128 + wpc * 2 * kBulkGroup * bulk_xbytes(SRC);
    cudaError_t e = cudaFuncSetAttribute(k_chunk_sums<SRC, TP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // resident CTAs per SM, looked up once per stage count (the kernel's resources are fixed)
    static std::atomic<int> per_sm_of[kMaxT];
    int per_sm = per_sm_of[tp].load(std::memory_order_relaxed);
    if (per_sm == 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_chunk_sums<SRC, TP>, 32 * wpc, smem);
        if (e != cudaSuccess) return e;
        per_sm = std::max(per_sm, 1);
        per_sm_of[tp].store(per_sm, std::memory_order_relaxed);
    }
    const int64_t need = ((int64_t)p.H * p.nchunk + wpc - 1) / wpc;
    const int grid = (int)std::min<int64_t>(need, (int64_t)per_sm * num_sms);
    return launch_kernel(k_chunk_sums<SRC, TP>, dim3(grid), dim3(32 * wpc), smem, st, maps->x_rows,
                         p, t, maps->gather);
}

// One warp per cluster.  The round's items of the cluster come from its own slot or, when
// they span several chunks, from their pieces added in chunk order.  In a stage's first
// round they are all its members; in a delta round they are the tokens that left (negated)
// and entered it, added to the total the previous round kept.  The total is kept,
// renormalised, for the next round, and the mean of the members written with its GEMM
// operands.  A cluster with no members keeps its centroid.  Each warp waits on a few
// dependent reads (its counts, then its pieces), so the kernel is built for four blocks per
// SM (64 registers): 0.06 ms less per quantize at the 13B-class shape than at three.
__global__ void __launch_bounds__(256, 4) k_cluster_finalize(QPlan p, int t, int planes, int delta) {
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int j = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int h = blockIdx.y;
    if (j >= p.C) return;
    const int64_t hj = (int64_t)h * p.C + j;
    // the item count and offset load together (the offset is unused without items)
    const int cnt = p.counts[hj];
    const int off = p.offs[hj];
    if (delta && cnt == 0) return;  // no member moved: the centroid and its operands stand
    float S[4] = {0.f, 0.f, 0.f, 0.f}, E[4] = {0.f, 0.f, 0.f, 0.f};
    float *tt = p.tot + hj * 2 * kD;
    int n = cnt;
    if (delta) {
        n = p.ccount[hj] + cnt - 2 * p.dleave[hj];
        const float4 ta = reinterpret_cast<const float4 *>(tt)[lane];
        const float4 tb = reinterpret_cast<const float4 *>(tt + kD)[lane];
        S[0] = ta.x; S[1] = ta.y; S[2] = ta.z; S[3] = ta.w;
        E[0] = tb.x; E[1] = tb.y; E[2] = tb.z; E[3] = tb.w;
    }
    const float4 mu = *reinterpret_cast<const float4 *>(p.mu + h * kD + 4 * lane);
    if (cnt > 0) {
        const int a = off / kChunk, b = (off + cnt - 1) / kChunk;
        if (a == b) {
            // all of the cluster's items were one run of one chunk
            const float *ws = p.wsum + hj * 2 * kD;
            const float4 sa = reinterpret_cast<const float4 *>(ws)[lane];
            const float4 sb = reinterpret_cast<const float4 *>(ws + kD)[lane];
            const float av[4] = {sa.x, sa.y, sa.z, sa.w}, bv[4] = {sb.x, sb.y, sb.z, sb.w};
#pragma unroll
            for (int k = 0; k < 4; k++) {
                acc_two_sum(S[k], E[k], av[k]);
                E[k] = __fadd_rn(E[k], bv[k]);
            }
        }
        const int np = a == b ? 0 : b - a + 1;
        for (int q0 = 0; q0 < np; q0 += 4) {
            float4 sa[4], sb[4];  // 4 pieces' loads in flight, added in chunk order
#pragma unroll
            for (int u = 0; u < 4; u++)
                if (q0 + u < np) {
                    const int kk = a + q0 + u;
                    // in its first chunk the cluster's run is the chunk's last run unless
                    // it starts exactly at the chunk start; in later chunks it is the first
                    const int slot = (kk == a && off != (int64_t)a * kChunk) ? 1 : 0;
                    const float *ps = p.psum + (((int64_t)h * p.nchunk + kk) * 2 + slot) * 2 * kD;
                    sa[u] = reinterpret_cast<const float4 *>(ps)[lane];
                    sb[u] = reinterpret_cast<const float4 *>(ps + kD)[lane];
                }
#pragma unroll
            for (int u = 0; u < 4; u++)
                if (q0 + u < np) {
                    const float av[4] = {sa[u].x, sa[u].y, sa[u].z, sa[u].w};
                    const float bv[4] = {sb[u].x, sb[u].y, sb[u].z, sb[u].w};
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        acc_two_sum(S[k], E[k], av[k]);
                        E[k] = __fadd_rn(E[k], bv[k]);
                    }
                }
        }
    }
    // every lane has read the counters; they restart at zero for the next round's sort
    __syncwarp();
    if (lane == 0) {
        p.counts[hj] = 0;
        p.dleave[hj] = 0;
        p.ccount[hj] = n;
    }
    if (n <= 0) {
        // no members: the total restarts at zero and the centroid stays (in the first
        // round its operands are written again from it)
        reinterpret_cast<float4 *>(tt)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
        reinterpret_cast<float4 *>(tt + kD)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (!delta) write_centroid(p, h, t, j, lane, false, make_float4(0.f, 0.f, 0.f, 0.f), planes != 0, mu);
        return;
    }
    // renormalise: S + E exactly as fl(S + E) plus its rounding error
#pragma unroll
    for (int k = 0; k < 4; k++) {
        float sum = S[k], err = 0.f;
        acc_two_sum(sum, err, E[k]);
        S[k] = sum;
        E[k] = err;
    }
    reinterpret_cast<float4 *>(tt)[lane] = make_float4(S[0], S[1], S[2], S[3]);
    reinterpret_cast<float4 *>(tt + kD)[lane] = make_float4(E[0], E[1], E[2], E[3]);
    const float fn = (float)n;
    write_centroid(p, h, t, j, lane, true,
                   make_float4(stored_mean(S[0], E[0], fn, p.cfmt), stored_mean(S[1], E[1], fn, p.cfmt),
                               stored_mean(S[2], E[2], fn, p.cfmt), stored_mean(S[3], E[3], fn, p.cfmt)),
                   planes != 0, mu);
}

cudaError_t launch_cluster_means(const QPlan &p, const AssignMaps *maps, int t, bool planes,
                                 bool delta, int num_sms, cudaStream_t st) {
    const int dl = delta ? 1 : 0;
    cudaError_t e = launch_kernel(k_sort_hist, dim3((unsigned)((p.nsb + kSortSB - 1) / kSortSB), p.H),
                                  dim3(kSortBlock), 0, st, p, t, dl);
    if (e == cudaSuccess)
        e = launch_kernel(k_sort_scan, dim3((unsigned)((p.C + 31) / 32), p.H), dim3(256), 0, st, p);
    if (e == cudaSuccess)
        e = launch_kernel(k_sort_scatter, dim3((unsigned)((p.nsb + kScatterGroups - 1) / kScatterGroups), p.H),
                          dim3(kSortBlock * kScatterGroups), 0, st, p, t, dl);
    if (e != cudaSuccess) return e;
    auto sums = [&](auto src) {
        constexpr int S = decltype(src)::value;
        switch (t - 1) {
            case 0: return launch_sums<S, 0>(p, maps, t, num_sms, st);
            case 1: return launch_sums<S, 1>(p, maps, t, num_sms, st);
            case 2: return launch_sums<S, 2>(p, maps, t, num_sms, st);
            case 3: return launch_sums<S, 3>(p, maps, t, num_sms, st);
            default: return launch_sums<S, -1>(p, maps, t, num_sms, st);
        }
    };
    e = p.in_dtype == DT_F32   ? sums(std::integral_constant<int, 1>())
        : p.in_dtype == DT_F16 ? sums(std::integral_constant<int, 3>())
                               : sums(std::integral_constant<int, 0>());
    if (e != cudaSuccess) return e;
    return launch_kernel(k_cluster_finalize, dim3((unsigned)((p.C + 7) / 8), p.H), dim3(256), 0, st, p, t,
                         planes ? 1 : 0, dl);
}

// --------------------------------------------------------------------------------------
// Final encoding of R^(T).  One thread per (token, 8 channels); the G = group/8 threads of
// a scale group reduce their absmax with shuffles.
//   a = max|r|, s = a / qmax (IEEE fp32), s_q = E4M3(s) (round to nearest even, saturate to
//   finite), q = clamp(rne(r / s_q), -qmax, qmax), u = q + 2^(b-1); s_q == 0 gives u = 2^(b-1).
// grid-stride over tokens, block 256 = 16 tokens x 16 chunks.
// --------------------------------------------------------------------------------------
constexpr int kEncTokens = 32;
constexpr int kEncG = 1;  // tokens per thread whose loads are in flight together

// TT: the number of stages when it is 0..4 (the stage loop unrolled), -1 for any T.
template <int BITS, int TT>
__global__ void __launch_bounds__(256) k_encode(QPlan p) {
    pdl_begin();
    constexpr int QMAX = (1 << (BITS - 1)) - 1, MID = 1 << (BITS - 1);
    const int T = TT >= 0 ? TT : p.T;
    const int h = blockIdx.y;
    const int c8 = threadIdx.x & 15;
    const int lpg = p.group >> 3;  // lanes per scale group (2, 4, 8)
    const bool midrise = p.qscheme == QVG_QSCHEME_MIDRISE;
    const int64_t i0 = (int64_t)blockIdx.x * kEncTokens;
    const int64_t i1 = min(p.N, i0 + kEncTokens);
    float nanprobe = 0.f;  // becomes NaN if any input is NaN or infinite (x * 0)
    bool bad_index = false;
#pragma unroll 1
    for (int64_t ib = i0; ib < i1; ib += 16 * kEncG) {
        // the loop bound is uniform over the block, so every lane reaches the shuffles;
        // rows past the end compute on zeros and store nothing.  The kEncG tokens of a
        // thread load together: X, then their cluster indices, then the centroid rows.
        float2 v[kEncG][4];
        int64_t ii[kEncG];
        bool ok[kEncG];
#pragma unroll
        for (int g = 0; g < kEncG; g++) {
            ii[g] = ib + 16 * g + (threadIdx.x >> 4);
            ok[g] = ii[g] < i1;
            if (ok[g]) {
                float x[8];
                load_x8(p.X, p.in_dtype, h * p.x_stride + ii[g] * kD + c8 * 8, x);
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    v[g][q] = make_float2(x[2 * q], x[2 * q + 1]);
                    nanprobe = __fmaf_rn(x[2 * q], 0.f, __fmaf_rn(x[2 * q + 1], 0.f, nanprobe));
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; q++) v[g][q] = make_float2(0.f, 0.f);
            }
        }
        // r = x - C^(1)[pi^(1)] - ... - C^(T)[pi^(T)] rounded once (the TwoSum chain)
        stage_input8<kEncG, TT>(p, h, ii, ok, c8, T, v, bad_index);
#pragma unroll
        for (int g = 0; g < kEncG; g++) {
            const int64_t i = ii[g];
            const bool valid = ok[g];
            float r[8], a = 0.f;
#pragma unroll
            for (int q = 0; q < 8; q++) {
                r[q] = q & 1 ? v[g][q >> 1].y : v[g][q >> 1].x;
                a = fmaxf(a, fabsf(r[q]));
            }
            for (int o = 1; o < lpg; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            // a / (the outermost level), IEEE: qmax, or 2^(b-1) - 1/2 for the mid-rise grid
            const float sc = midrise ? __fdiv_rn(a, (float)MID - 0.5f)
                                     : (QMAX == 1 ? a : __fdiv_rn(a, (float)QMAX));
            const __nv_fp8_storage_t sb = __nv_cvt_float_to_fp8(sc, __NV_SATFINITE, __NV_E4M3);
            const float sq = __half2float(__half(__nv_cvt_fp8_to_halfraw(sb, __NV_E4M3)));
            uint32_t word = 0;
            if (BITS == 2 && sq != 0.f) {
                // INT2: the code is decided by comparing r with exact multiples of s_q (s_q/2
                // and s_q are exact in fp32), which is the code of the exact quotient r / s_q:
                //   symmetric: q = clamp(rne(r / s_q), -1, 1) is 1 when r > s_q / 2, -1 when
                //     r < -s_q / 2, else 0 (an exact half rounds to the even 0);
                //   mid-rise: u = floor(r / s_q) + 2 clamped to [0, 3] steps at -s_q, 0, s_q.
                const float hq = midrise ? sq : 0.5f * sq;
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    uint32_t u;
                    if (midrise)
                        u = r[q] >= 0.f ? (r[q] >= hq ? 3u : 2u) : (r[q] >= -hq ? 1u : 0u);
                    else
                        u = r[q] > hq ? 3u : (r[q] < -hq ? 1u : 2u);
                    word |= u << (q * BITS);
                }
            } else if (sq != 0.f && midrise) {
                // u = floor(r / s_q) + 2^(b-1), clamped.  r times an approximate reciprocal
                // (a few ulps) has the same floor except close to an integer; there the
                // quotient is recomputed with a correctly rounded division.
                float inv;
                asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(sq));
                float fq[8];
                uint32_t close = 0;
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    const float v = __fmul_rn(r[q], inv);
                    fq[q] = floorf(v);
                    close |= (fabsf(__fsub_rn(v, rintf(v))) < 0x1p-17f * fmaxf(1.f, fabsf(v)) ? 1u : 0u) << q;
                }
                if (close) {  // rare
#pragma unroll
                    for (int q = 0; q < 8; q++)
                        if ((close >> q) & 1u) fq[q] = floorf(__fdiv_rn(r[q], sq));
                }
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    const float u = fminf(fmaxf(fq[q] + (float)MID, 0.f), (float)(2 * MID - 1));
                    word |= (uint32_t)u << (q * BITS);
                }
            } else if (sq != 0.f) {
                // q = clamp(rne(r / s_q)) with the IEEE quotient.  r times an approximate
                // reciprocal (a few ulps) gives the same rounding except close to a
                // half-integer; there the quotient is recomputed with a correctly rounded
                // division.  Adding 1.5 * 2^23 to the clamped quotient rounds it to an
                // integer (half to even) and leaves that integer in the low mantissa bits.
                constexpr float kRound = 12582912.f;  // 1.5 * 2^23
                float inv;
                asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(sq));
                float tq[8];
                uint32_t close = 0;  // elements whose quotient is near a half-integer
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    const float v = fminf(fmaxf(__fmul_rn(r[q], inv), (float)-QMAX), (float)QMAX);
                    tq[q] = __fadd_rn(v, kRound);
                    const float d = __fsub_rn(v, __fsub_rn(tq[q], kRound));  // v - rne(v)
                    close |= (fabsf(d) > 0.5f - 0x1p-17f ? 1u : 0u) << q;
                }
                if (close) {  // rare
#pragma unroll
                    for (int q = 0; q < 8; q++)
                        if ((close >> q) & 1u)
                            tq[q] = __fadd_rn(fminf(fmaxf(__fdiv_rn(r[q], sq), (float)-QMAX), (float)QMAX),
                                              kRound);
                }
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    const int qi = (int)(__float_as_uint(tq[q]) - 0x4B400000u);  // rne(v)
                    word |= (uint32_t)(qi + MID) << (q * BITS);
                }
            } else {
#pragma unroll
                for (int q = 0; q < 8; q++) word |= (uint32_t)MID << (q * BITS);
            }
            if (valid) {
                const int64_t orow = (int64_t)h * p.cap + p.tok_off + i;
                if constexpr (BITS == 2)
                    *reinterpret_cast<uint16_t *>(p.codes + orow * (kD / 4) + c8 * 2) = (uint16_t)word;
                else
                    *reinterpret_cast<uint32_t *>(p.codes + orow * (kD / 2) + c8 * 4) = word;
                if ((c8 & (lpg - 1)) == 0) p.scales[orow * (kD / p.group) + c8 / lpg] = sb;
            }
        }
    }
    if (__any_sync(0xffffffffu, nanprobe != nanprobe) && (threadIdx.x & 31) == 0)
        or_status(p.status, QVG_DEV_NONFINITE);
    if (__any_sync(0xffffffffu, bad_index) && (threadIdx.x & 31) == 0) or_status(p.status, QVG_DEV_BAD_INDEX);
}

template <int BITS>
static cudaError_t launch_encode_b(const QPlan &p, cudaStream_t st) {
    const dim3 grid((unsigned)((p.N + kEncTokens - 1) / kEncTokens), p.H);
    switch (p.T) {
        case 0: return launch_kernel(k_encode<BITS, 0>, grid, dim3(256), 0, st, p);
        case 1: return launch_kernel(k_encode<BITS, 1>, grid, dim3(256), 0, st, p);
        case 2: return launch_kernel(k_encode<BITS, 2>, grid, dim3(256), 0, st, p);
        case 3: return launch_kernel(k_encode<BITS, 3>, grid, dim3(256), 0, st, p);
        case 4: return launch_kernel(k_encode<BITS, 4>, grid, dim3(256), 0, st, p);
        default: return launch_kernel(k_encode<BITS, -1>, grid, dim3(256), 0, st, p);
    }
}

cudaError_t launch_encode(const QPlan &p, cudaStream_t st) {
    return p.bits == 2 ? launch_encode_b<2>(p, st) : launch_encode_b<4>(p, st);
}

}  // namespace qvg
