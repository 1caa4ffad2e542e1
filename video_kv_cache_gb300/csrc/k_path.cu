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

#include "internal.cuh"

namespace qvg {

// --------------------------------------------------------------------------------------
// Cold-start rows: for each (tensor, stage) the first C picks of a partial Fisher-Yates
// shuffle of 0..N-1 driven by SplitMix64 (Steele, Lea and Flood, 2014, with the constants
// Vigna published), state seed ^ (tensor_id * 0x9E3779B97F4A7C15) ^ t.  Only the touched
// positions of the permutation are stored: positions < C directly, the others in a small
// open-addressing table.   grid (T, H), one warp; lane 0 runs the sequential shuffle.
// --------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t splitmix64_next(uint64_t &state) {
    uint64_t z = (state += 0x9E3779B97F4A7C15ULL);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

constexpr int kHashSlots = 1024;

__global__ void k_init_indices(QPlan p, uint64_t seed, int64_t tid_base) {
    const int t = blockIdx.x + 1, h = blockIdx.y, lane = threadIdx.x;
    __shared__ int lo[kMaxC];
    __shared__ int keys[kHashSlots];
    __shared__ int vals[kHashSlots];
    for (int x = lane; x < p.C; x += 32) lo[x] = x;
    for (int x = lane; x < kHashSlots; x += 32) keys[x] = -1;
    __syncwarp();
    if (lane != 0) return;
    uint64_t state = seed ^ ((uint64_t)(tid_base + h) * 0x9E3779B97F4A7C15ULL) ^ (uint64_t)t;
    int *out = p.init_idx + (int64_t)(h * p.T + (t - 1)) * p.C;
    for (int j = 0; j < p.C; j++) {
        const uint64_t r = splitmix64_next(state);
        const int k = j + (int)(r % (uint64_t)(p.N - j));
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
    k_init_indices<<<dim3(p.T, p.H), 32, 0, st>>>(p, seed, tid_base);
    return cudaGetLastError();
}

// --------------------------------------------------------------------------------------
// Stage-t initial centroids: rows of R^(t-1) picked by the seeded shuffle, or the caller's
// warm-start table.   grid (C, H), block 128 (one thread per channel).
// --------------------------------------------------------------------------------------
__global__ void k_init_centroids(QPlan p, int t) {
    const int j = blockIdx.x, h = blockIdx.y, k = threadIdx.x;
    float *dst = p.cent + h * p.cent_tstride + p.cent_off + (int64_t)(t - 1) * p.C * kD +
                 (int64_t)j * kD;
    float v;
    if (p.warm) {
        v = __ldg(p.warm + h * p.warm_stride + (int64_t)(t - 1) * p.C * kD + (int64_t)j * kD + k);
    } else {
        const int64_t row = p.init_idx[(h * p.T + (t - 1)) * p.C + j];
        if (t == 1)
            v = load_x1(p.X, p.in_dtype, h * p.x_stride + row * kD + k);
        else
            v = p.R32[(h * p.N + row) * kD + k];
    }
    dst[k] = v;
}

cudaError_t launch_init_centroids(const QPlan &p, int t, cudaStream_t st) {
    k_init_centroids<<<dim3(p.C, p.H), kD, 0, st>>>(p, t);
    return cudaGetLastError();
}

// --------------------------------------------------------------------------------------
// Centring vector for the GEMM operands.  Squared distances do not change when both
// operands are shifted by the same vector; shifting by a point near the data's centre
// keeps the bf16 split's error small.  Stage 1 uses the mean of the initial centroids
// (C sample rows of X, or the warm-start table); later stages work on residuals whose
// mean is already ~0 and use 0.   grid H, block 128.
// --------------------------------------------------------------------------------------
__global__ void k_centre(QPlan p, int t) {
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
    k_centre<<<p.H, kD, 0, st>>>(p, t);
    return cudaGetLastError();
}

// --------------------------------------------------------------------------------------
// Residual preparation for stage t.  One thread per (token, 8 channels).
//   r      = fp32(x - sum_{s<t} C^(s)[pi^(s)_i]) via a TwoSum chain (one final rounding)
//   R32    = r                           (stages t >= 2; stage 1 reads X directly)
//   A hi/lo = bf16 split of r - mu       (tensor-core operand of the assignment)
//   rnorm  = ||r - mu||                  (for the assignment's error margin)
//   maxabs = max |r| over the tensor     (fixed-point scale of the centroid sums)
// grid (blocks per tensor, H), block 256 = 16 tokens x 16 chunks of 8 channels.
// --------------------------------------------------------------------------------------
constexpr int kPrepTokens = 512;

__global__ void __launch_bounds__(256) k_prep(QPlan p, int t) {
    const int h = blockIdx.y;
    const int c8 = threadIdx.x & 15;
    const int64_t i0 = (int64_t)blockIdx.x * kPrepTokens;
    const int64_t i1 = min(p.N, i0 + kPrepTokens);
    float mu[8];
    load_f8(p.mu + h * kD + c8 * 8, mu);
    float mx = 0.f;
    bool finite = true, bad_index = false;
    for (int64_t ib = i0; ib < i1; ib += 16) {
        // the loop bound is uniform over the block, so every lane reaches the shuffles
        const int64_t i = ib + (threadIdx.x >> 4);
        const bool valid = i < i1;
        float x[8], s[8], e[8];
        if (valid) {
            load_x8(p.X, p.in_dtype, h * p.x_stride + i * kD + c8 * 8, x);
        } else {
#pragma unroll
            for (int q = 0; q < 8; q++) x[q] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < 8; q++) {
            finite &= isfinite(x[q]);
            s[q] = x[q];
            e[q] = 0.f;
        }
        for (int st = 1; valid && st < t; st++) {
            int pj = p.pi[(int64_t)(h * p.T + st - 1) * p.cap + p.tok_off + i];
            if (pj >= p.C) {
                pj = p.C - 1;
                bad_index = true;
            }
            float c[8];
            load_f8(p.cent + h * p.cent_tstride + p.cent_off + (int64_t)(st - 1) * p.C * kD +
                        (int64_t)pj * kD + c8 * 8, c);
#pragma unroll
            for (int q = 0; q < 8; q++) {
                float err;
                two_sum(s[q], -c[q], s[q], err);
                e[q] = __fadd_rn(e[q], err);
            }
        }
        float r[8];
#pragma unroll
        for (int q = 0; q < 8; q++) r[q] = __fadd_rn(s[q], e[q]);
        if (valid && t >= 2) {
            float4 *dst = reinterpret_cast<float4 *>(p.R32 + (h * p.N + i) * kD + c8 * 8);
            dst[0] = make_float4(r[0], r[1], r[2], r[3]);
            dst[1] = make_float4(r[4], r[5], r[6], r[7]);
        }
        float ss = 0.f;
        __align__(16) __nv_bfloat16 hi[8], lo[8];
#pragma unroll
        for (int q = 0; q < 8; q++) {
            float v = __fsub_rn(r[q], mu[q]);
            hi[q] = __float2bfloat16_rn(v);
            lo[q] = __float2bfloat16_rn(__fsub_rn(v, __bfloat162float(hi[q])));
            ss = __fmaf_rn(v, v, ss);
            mx = fmaxf(mx, fabsf(r[q]));
        }
        if (valid) {
            *reinterpret_cast<uint4 *>(p.A + ((int64_t)(h * 2 + 0) * p.N + i) * kD + c8 * 8) =
                *reinterpret_cast<uint4 *>(hi);
            *reinterpret_cast<uint4 *>(p.A + ((int64_t)(h * 2 + 1) * p.N + i) * kD + c8 * 8) =
                *reinterpret_cast<uint4 *>(lo);
        }
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (valid && c8 == 0) p.rnorm[h * p.N + i] = sqrtf(ss);
    }
    // block max -> one atomic per block
    __shared__ float red[8];
    __shared__ int bad, bad_idx;
    if (threadIdx.x == 0) bad = 0, bad_idx = 0;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    __syncthreads();
    if (!finite) bad = 1;
    if (bad_index) bad_idx = 1;
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = red[0];
        for (int w = 1; w < 8; w++) m = fmaxf(m, red[w]);
        if (m == m) atomicMax(p.maxabs + h, __float_as_uint(m));
        if (bad) or_status(p.status, QVG_DEV_NONFINITE);
        if (bad_idx) or_status(p.status, QVG_DEV_BAD_INDEX);
    }
}

cudaError_t launch_prep(const QPlan &p, int t, cudaStream_t st) {
    dim3 grid((unsigned)((p.N + kPrepTokens - 1) / kPrepTokens), p.H);
    k_prep<<<grid, 256, 0, st>>>(p, t);
    return cudaGetLastError();
}

// --------------------------------------------------------------------------------------
// Centroid finalisation and GEMM planes.   grid (C, H), block 128.
//   from_sums: C_j = fp32(exact fixed-point sum / count) for non-empty clusters (empty ones
//              keep their value); the sums and counts are cleared for the next round.
//   planes:    bf16 hi / lo split of C_j - mu and ||C_j - mu||^2 for the next assignment.
// --------------------------------------------------------------------------------------
__global__ void k_centroid_planes(QPlan p, int t, int from_sums, int planes) {
    const int j = blockIdx.x, h = blockIdx.y, k = threadIdx.x;
    float *c = p.cent + h * p.cent_tstride + p.cent_off + (int64_t)(t - 1) * p.C * kD +
               (int64_t)j * kD;
    float v = c[k];
    __shared__ double inv_s;
    __shared__ int cnt_s;
    __shared__ float red[4];
    if (from_sums) {
        if (k == 0) {
            const int cnt = p.counts[h * p.C + j];
            cnt_s = cnt;
            if (cnt > 0) inv_s = ldexp(1.0, -fixed_q(p.maxabs[h], p.N)) / (double)cnt;
            p.counts[h * p.C + j] = 0;
        }
        __syncthreads();
        long long *sp = p.sums + ((int64_t)h * p.C + j) * kD + k;
        if (cnt_s > 0) {
            v = (float)((double)(*sp) * inv_s);
            c[k] = v;
        }
        *sp = 0;
    }
    if (planes) {
        const float ct = __fsub_rn(v, p.mu[h * kD + k]);
        const __nv_bfloat16 hi = __float2bfloat16_rn(ct);
        const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(ct, __bfloat162float(hi)));
        p.B[((int64_t)(h * 2 + 0) * p.Cpad + j) * kD + k] = hi;
        p.B[((int64_t)(h * 2 + 1) * p.Cpad + j) * kD + k] = lo;
        float ss = ct * ct;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if ((k & 31) == 0) red[k >> 5] = ss;
        __syncthreads();
        if (k == 0) p.cn[(int64_t)h * p.Cpad + j] = (red[0] + red[1]) + (red[2] + red[3]);
    }
}

cudaError_t launch_centroid_planes(const QPlan &p, int t, bool from_sums, bool planes,
                                   cudaStream_t st) {
    k_centroid_planes<<<dim3(p.C, p.H), kD, 0, st>>>(p, t, from_sums ? 1 : 0, planes ? 1 : 0);
    return cudaGetLastError();
}

// --------------------------------------------------------------------------------------
// Centroid sums.  Each CTA owns a token range of one tensor and a slab of CH = 32*CPL
// channels, keeps int64 fixed-point bins [C][CH] in shared memory, and adds them to the
// global bins once at the end.  A warp walks its tokens in order with lane l holding
// channels l*CPL..; consecutive tokens of a run with the same cluster (frequent: the
// grouping follows the video's spatial layout) are summed in registers and flushed to the
// shared bins only when the cluster changes.  Integer adds make every order give the
// same bits.
//   SRC: 0 = X as 16-bit (fp16 / bf16), 1 = X as fp32, 2 = R32 (stages t >= 2)
// grid (units per tensor, channel slabs, H), block 512.
// --------------------------------------------------------------------------------------
constexpr int kUpdThreads = 512;
constexpr int kUpdBatch = 16;  // tokens whose loads are in flight per warp

template <int CPL, int SRC>
__global__ void __launch_bounds__(kUpdThreads) k_update(QPlan p, int t, int64_t toks) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int CH = 32 * CPL;
    long long *bins = reinterpret_cast<long long *>(smem_raw);
    unsigned *cnt = reinterpret_cast<unsigned *>(bins + (size_t)p.C * CH);
    const int h = blockIdx.z, slab = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int nw = kUpdThreads / 32;
    for (int x = threadIdx.x; x < p.C * CH; x += kUpdThreads) bins[x] = 0;
    for (int x = threadIdx.x; x < p.C; x += kUpdThreads) cnt[x] = 0;
    __syncthreads();

    const float scale = pow2f(fixed_q(p.maxabs[h], p.N));
    const int64_t t0 = (int64_t)blockIdx.x * toks;
    const int64_t t1 = min(p.N, t0 + toks);
    const int64_t span = (t1 - t0 + nw - 1) / nw;
    const int64_t w0 = min(t1, t0 + warp * span), w1 = min(t1, w0 + span);
    // lane l owns channels slab*CH + l + 32*c: every access of a warp is one contiguous run
    const int ch = slab * CH + lane;
    const uint8_t *pis = p.pi + (int64_t)(h * p.T + t - 1) * p.cap + p.tok_off;
    const float *rsrc = SRC == 2 ? p.R32 + (int64_t)h * p.N * kD + ch : nullptr;
    const float *xsrc32 = SRC == 1 ? static_cast<const float *>(p.X) + h * p.x_stride + ch : nullptr;
    const uint16_t *xsrc16 = SRC == 0 ? static_cast<const uint16_t *>(p.X) + h * p.x_stride + ch : nullptr;

    int run_p = -1;
    unsigned run_n = 0;
    long long acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; c++) acc[c] = 0;

    auto flush = [&]() {
        if (run_p >= 0) {
#pragma unroll
            for (int c = 0; c < CPL; c++)
                atomicAdd(reinterpret_cast<unsigned long long *>(bins + run_p * CH + lane + 32 * c),
                          static_cast<unsigned long long>(acc[c]));
            if (lane == 0) atomicAdd(cnt + run_p, run_n);
        }
    };

    for (int64_t base = w0; base < w1; base += 32) {
        const int n = (int)min((int64_t)32, w1 - base);
        int my_p = lane < n ? (int)pis[base + lane] : 0;
        if (my_p >= p.C) {  // never produced by the assignment; counted, not accumulated
            or_status(p.status, QVG_DEV_BAD_INDEX);
            my_p = -1;
        }
        for (int jj = 0; jj < n; jj += kUpdBatch) {
            float val[kUpdBatch][CPL];
#pragma unroll
            for (int u = 0; u < kUpdBatch; u++) {
                const int64_t i = base + jj + u;
                if (jj + u < n) {
#pragma unroll
                    for (int c = 0; c < CPL; c++) {
                        if constexpr (SRC == 2) {
                            val[u][c] = __ldg(rsrc + i * kD + 32 * c);
                        } else if constexpr (SRC == 1) {
                            val[u][c] = __ldg(xsrc32 + i * kD + 32 * c);
                        } else {
                            const uint32_t b = __ldg(reinterpret_cast<const unsigned short *>(xsrc16) + i * kD + 32 * c);
                            val[u][c] = p.in_dtype == DT_BF16 ? __uint_as_float(b << 16)
                                                              : __half2float(__ushort_as_half((unsigned short)b));
                        }
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kUpdBatch; u++) {
                if (jj + u < n) {
                    const int pj = __shfl_sync(0xffffffffu, my_p, jj + u);
                    if (pj < 0) continue;
                    if (pj != run_p) {
                        flush();
                        run_p = pj;
                        run_n = 0;
#pragma unroll
                        for (int c = 0; c < CPL; c++) acc[c] = 0;
                    }
                    run_n++;
#pragma unroll
                    for (int c = 0; c < CPL; c++) acc[c] += __float2ll_rn(val[u][c] * scale);
                }
            }
        }
    }
    flush();
    __syncthreads();
    long long *gs = p.sums + (int64_t)h * p.C * kD + slab * CH;
    for (int x = threadIdx.x; x < p.C * CH; x += kUpdThreads) {
        const int j = x / CH;
        if (cnt[j] != 0u)
            atomicAdd(reinterpret_cast<unsigned long long *>(gs + (int64_t)j * kD + (x - j * CH)),
                      static_cast<unsigned long long>(bins[x]));
    }
    if (slab == 0)
        for (int j = threadIdx.x; j < p.C; j += kUpdThreads)
            if (cnt[j] != 0u) atomicAdd(p.counts + h * p.C + j, (int)cnt[j]);
}

template <int CPL>
static cudaError_t launch_update_cpl(const QPlan &p, int t, int num_sms, cudaStream_t st) {
    constexpr int CH = 32 * CPL;
    const size_t smem = (size_t)p.C * CH * 8 + (size_t)p.C * 4;
    const int slabs = kD / CH;
    // one wave of CTAs (one per SM): few CTAs keep the final flush of the shared-memory
    // bins to the global sums small; at least 512 tokens per CTA
    const int64_t per_tensor = std::max<int64_t>(1, num_sms / ((int64_t)p.H * slabs));
    int64_t toks = std::max<int64_t>(512, (p.N + per_tensor - 1) / per_tensor);
    toks = (toks + 31) / 32 * 32;
    const unsigned units = (unsigned)((p.N + toks - 1) / toks);
    dim3 grid(units, slabs, p.H);
    cudaError_t e;
    if (t >= 2) {
        e = cudaFuncSetAttribute(k_update<CPL, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k_update<CPL, 2><<<grid, kUpdThreads, smem, st>>>(p, t, toks);
    } else if (p.in_dtype == DT_F32) {
        e = cudaFuncSetAttribute(k_update<CPL, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k_update<CPL, 1><<<grid, kUpdThreads, smem, st>>>(p, t, toks);
    } else {
        e = cudaFuncSetAttribute(k_update<CPL, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k_update<CPL, 0><<<grid, kUpdThreads, smem, st>>>(p, t, toks);
    }
    return cudaGetLastError();
}

cudaError_t launch_update(const QPlan &p, int t, int num_sms, cudaStream_t st) {
    // 128-channel bins when they fit comfortably in shared memory, else 64-channel slabs.
    if ((size_t)p.C * kD * 8 <= 100 * 1024) return launch_update_cpl<4>(p, t, num_sms, st);
    return launch_update_cpl<2>(p, t, num_sms, st);
}

// --------------------------------------------------------------------------------------
// Final encoding of R^(T).  One thread per (token, 8 channels); the G = group/8 threads of
// a scale group reduce their absmax with shuffles.
//   a = max|r|, s = a / qmax (IEEE fp32), s_q = E4M3(s) (round to nearest even, saturate to
//   finite), q = clamp(rne(r / s_q), -qmax, qmax), u = q + 2^(b-1); s_q == 0 gives u = 2^(b-1).
// grid-stride over tokens, block 256 = 16 tokens x 16 chunks.
// --------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_encode(QPlan p) {
    const int c8 = threadIdx.x & 15;
    const int lpg = p.group >> 3;  // lanes per scale group (2, 4, 8)
    const int qmax = (1 << (p.bits - 1)) - 1, mid = 1 << (p.bits - 1);
    const int64_t total = (int64_t)p.H * p.N;
    bool finite = true, bad_index = false;
    for (int64_t rb = (int64_t)blockIdx.x * 16; rb < total; rb += (int64_t)gridDim.x * 16) {
        // the loop bound is uniform over the block, so every lane reaches the shuffles;
        // rows past the end compute on zeros and store nothing
        const int64_t row = rb + (threadIdx.x >> 4);
        const bool valid = row < total;
        const int h = valid ? (int)(row / p.N) : 0;
        const int64_t i = valid ? row - (int64_t)h * p.N : 0;
        float x[8], s[8], e[8];
        if (valid) {
            load_x8(p.X, p.in_dtype, h * p.x_stride + i * kD + c8 * 8, x);
        } else {
#pragma unroll
            for (int q = 0; q < 8; q++) x[q] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < 8; q++) {
            finite &= isfinite(x[q]);
            s[q] = x[q];
            e[q] = 0.f;
        }
        for (int st = 1; valid && st <= p.T; st++) {
            int pj = p.pi[(int64_t)(h * p.T + st - 1) * p.cap + p.tok_off + i];
            if (pj >= p.C) {
                pj = p.C - 1;
                bad_index = true;
            }
            float c[8];
            load_f8(p.cent + h * p.cent_tstride + p.cent_off + (int64_t)(st - 1) * p.C * kD +
                        (int64_t)pj * kD + c8 * 8, c);
#pragma unroll
            for (int q = 0; q < 8; q++) {
                float err;
                two_sum(s[q], -c[q], s[q], err);
                e[q] = __fadd_rn(e[q], err);
            }
        }
        float r[8], a = 0.f;
#pragma unroll
        for (int q = 0; q < 8; q++) {
            r[q] = __fadd_rn(s[q], e[q]);
            a = fmaxf(a, fabsf(r[q]));
        }
        for (int o = 1; o < lpg; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const float sc = __fdiv_rn(a, (float)qmax);
        const __nv_fp8_storage_t sb = __nv_cvt_float_to_fp8(sc, __NV_SATFINITE, __NV_E4M3);
        const float sq = __half2float(__half(__nv_cvt_fp8_to_halfraw(sb, __NV_E4M3)));
        // q = rne(r / s_q) with the IEEE quotient.  r * (1/s_q) is within 1.5 ulp of that
        // quotient, so it gives the same rounding except within a few ulps of a half-integer;
        // there the quotient is recomputed with a correctly rounded division.
        const float inv = sq != 0.f ? __frcp_rn(sq) : 0.f;
        uint32_t word = 0;
#pragma unroll
        for (int q = 0; q < 8; q++) {
            int u = mid;
            if (sq != 0.f) {
                float v = __fmul_rn(r[q], inv);
                if (fabsf(fabsf(v - rintf(v)) - 0.5f) < 0x1p-17f) v = __fdiv_rn(r[q], sq);
                const float qq = fminf(fmaxf(rintf(v), (float)-qmax), (float)qmax);
                u = (int)qq + mid;
            }
            word |= (uint32_t)u << (q * p.bits);
        }
        if (valid) {
            const int64_t orow = (int64_t)h * p.cap + p.tok_off + i;
            if (p.bits == 2)
                *reinterpret_cast<uint16_t *>(p.codes + orow * (kD / 4) + c8 * 2) = (uint16_t)word;
            else
                *reinterpret_cast<uint32_t *>(p.codes + orow * (kD / 2) + c8 * 4) = word;
            if ((c8 & (lpg - 1)) == 0) p.scales[orow * (kD / p.group) + c8 / lpg] = sb;
        }
    }
    if (!finite) or_status(p.status, QVG_DEV_NONFINITE);
    if (bad_index) or_status(p.status, QVG_DEV_BAD_INDEX);
}

cudaError_t launch_encode(const QPlan &p, cudaStream_t st) {
    const int64_t rows = (int64_t)p.H * p.N;
    int64_t blocks = (rows + 15) / 16;
    if (blocks > 65535LL * 16) blocks = 65535LL * 16;
    k_encode<<<(unsigned)blocks, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace qvg
