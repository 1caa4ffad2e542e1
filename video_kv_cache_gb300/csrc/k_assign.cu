// k-means assignment on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// Method step: pi_i = argmin_j ||R_i - C_j||^2 over the C centroids of the current stage,
// ties to the lowest j ("Quant VideoGen" notes page, section Semantic-Aware Smoothing, step
// 1; review page, pipeline step (a)).
//
// Since ||R_i - C_j||^2 = ||R_i||^2 - 2 R_i.C_j + ||C_j||^2, the argmin only needs the
// score s_ij = ||C_j||^2 - 2 R_i.C_j, and R.C^T is a [N x 128] x [128 x C] GEMM.  Both
// operands are first shifted by a common centring vector mu (distances do not change) and
// split into two bf16 terms, x = hi + lo.  The GEMM accumulates hi.hi + hi.lo + lo.hi in
// fp32 TMEM, which carries ~16 significant bits of each operand.  The epilogue then finds
// the best score; every cluster whose score is within a bound on the GEMM's error of the
// best one is re-scored exactly (direct fp32 sum of squared differences on the fp32
// residual and centroid), so the chosen index is that of the true nearest centroid up to
// fp32 rounding.
//
// Kernel structure (one persistent CTA per SM, 192 threads):
//   warp 0   TMA producer: B (centroid planes, C x 128 x 2 planes) once per tensor, A
//            (residual planes of 128 tokens, four 16 KB blocks of 64 channels per tile)
//            into a ring of smem slots.
//   warp 1   TMEM allocator and MMA issuer (one thread): 3 x 8 tcgen05.mma of
//            M=128, N=Cpad, K=16 per tile into one of two TMEM accumulators.
//   warps 2-5 epilogue: warp w reads TMEM lanes 32*(w%4).. (one token row per thread),
//            computes the argmin, releases the accumulator, re-scores near ties, writes pi.
// Every mbarrier wait is bounded; on timeout the kernel sets QVG_DEV_TIMEOUT, stops, waits
// for its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>

#include <algorithm>

#include "internal.cuh"

namespace qvg {

namespace {

constexpr int kEpiGroups = 2;                      // epilogue groups of 8 warps
constexpr int kThreads = 64 + kEpiGroups * 8 * 32;  // producer, MMA, 16 epilogue warps
constexpr int kTileM = 128;
constexpr uint32_t kKBlockBytes = kTileM * 64 * 2;  // 16 KB: 64 channels of that plane
constexpr uint32_t kSpinLimit = 1u << 22;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0u;
}

// Bounded wait on a phase.  Gives up when another role already gave up, or after the
// spin limit (then it raises the abort flag itself).
__device__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    for (uint32_t n = 0; n < kSpinLimit; n++) {
        if (mbar_try(bar, parity)) return true;
        if (*abort_flag) return false;
        if (n >= 1024) __nanosleep(128);
    }
    *abort_flag = 1;
    return false;
}
// Bounded wait used during teardown, which must not stop at the abort flag.
__device__ void mbar_wait_final(uint32_t bar, uint32_t parity) {
    for (uint32_t n = 0; n < kSpinLimit; n++) {
        if (mbar_try(bar, parity)) return;
        if (n >= 1024) __nanosleep(128);
    }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float v[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int q = 0; q < 32; q++) v[q] = __uint_as_float(r[q]);
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of 128 bytes,
// 8-row groups 1024 bytes apart (the layout a TMA box of 64 bf16 x rows writes with
// CU_TENSOR_MAP_SWIZZLE_128B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4)   // start address
           | ((uint64_t)1 << 16)                 // leading-dimension offset (unused here)
           | ((uint64_t)(1024 >> 4) << 32)       // stride between 8-row groups
           | ((uint64_t)1 << 46)                 // descriptor version
           | ((uint64_t)2 << 61);                // 128-byte swizzle
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both K-major.
__device__ __forceinline__ uint32_t make_idesc(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(kTileM >> 4) << 24);
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    k_assign(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
             QPlan p, int t, int tiles_per_tensor, int nslots, uint32_t tmem_cols,
             uint32_t acc_stride) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int Cpad = p.Cpad;
    const uint32_t bsub = (uint32_t)Cpad * 128u;  // one (plane, 64-channel block) of B
    unsigned char *sB = sm;
    unsigned char *sA = sm + 4 * bsub;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sA + (size_t)nslots * kKBlockBytes);
    uint64_t *a_full = bars, *a_empty = bars + nslots;
    uint64_t *b_full = bars + 2 * nslots, *b_empty = b_full + 1;
    uint64_t *acc_full = b_full + 2, *acc_empty = acc_full + kEpiGroups, *fin = acc_empty + kEpiGroups;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // per epilogue group: ||c||^2 of its current tensor and the column-half exchange
    // 16-byte aligned: the epilogue reads it with 16-byte vector loads
    float *cn_s = reinterpret_cast<float *>(
        (reinterpret_cast<uintptr_t>(tmem_slot + 4) + 15) & ~static_cast<uintptr_t>(15));  // [kEpiGroups][Cpad]
    float *x_best = cn_s + kEpiGroups * Cpad;                     // [kEpiGroups][128]
    float *x_second = x_best + kEpiGroups * kTileM;
    int *x_idx = reinterpret_cast<int *>(x_second + kEpiGroups * kTileM);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t total = (int64_t)p.H * tiles_per_tensor;
    const int64_t per = total / gridDim.x, rem = total % gridDim.x;
    const int64_t tb = blockIdx.x * per + min((int64_t)blockIdx.x, rem);
    const int64_t te = tb + per + ((int64_t)blockIdx.x < rem ? 1 : 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < nslots; s++) {
            mbar_init(smem_u32(a_full + s), 1);
            mbar_init(smem_u32(a_empty + s), 1);
        }
        mbar_init(smem_u32(b_full), 1);
        mbar_init(smem_u32(b_empty), 1);
        for (int g = 0; g < kEpiGroups; g++) {
            mbar_init(smem_u32(acc_full + g), 1);
            mbar_init(smem_u32(acc_empty + g), 8);
        }
        mbar_init(smem_u32(fin), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int cur_h = -1;
            uint32_t nb = 0, issued = 0;
            for (int64_t tile = tb, lt = 0; tile < te && !*abort_flag; tile++, lt++) {
                const int h = (int)(tile / tiles_per_tensor);
                const int m0 = (int)(tile - (int64_t)h * tiles_per_tensor) * kTileM;
                if (h != cur_h) {
                    if (nb > 0 && !mbar_wait(smem_u32(b_empty), (nb - 1) & 1, abort_flag)) break;
                    mbar_expect_tx(smem_u32(b_full), 4 * bsub);
                    for (int pl = 0; pl < 2; pl++)
                        for (int kb = 0; kb < 2; kb++)
                            tma_load_3d(smem_u32(sB + (pl * 2 + kb) * bsub), &tmB, kb * 64, 0,
                                        2 * h + pl, smem_u32(b_full));
                    nb++;
                    cur_h = h;
                }
                // four 16 KB loads per tile: hi plane channels 0-63, 64-127, then lo plane
                bool ok = true;
                for (int k = 0; k < 4; k++) {
                    const uint32_t q = 4u * (uint32_t)lt + k, s = q % nslots, ph = (q / nslots) & 1u;
                    if (!mbar_wait(smem_u32(a_empty + s), ph ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(smem_u32(a_full + s), kKBlockBytes);
                    tma_load_3d(smem_u32(sA + s * kKBlockBytes), &tmA, (k & 1) * 64, m0,
                                2 * h + (k >> 1), smem_u32(a_full + s));
                    issued = q + 1;
                }
                if (!ok) break;
            }
            // make sure every copy this CTA started has landed before the CTA can exit
            if (nb > 0) mbar_wait_final(smem_u32(b_full), (nb - 1) & 1);
            const uint32_t first = issued > (uint32_t)nslots ? issued - nslots : 0u;
            for (uint32_t q = first; q < issued; q++)
                mbar_wait_final(smem_u32(a_full + q % nslots), (q / nslots) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = make_idesc(Cpad);
            int cur_h = -1;
            uint32_t nb = 0;
            const uint64_t dB0 = sw128_desc(smem_u32(sB));
            for (int64_t tile = tb, lt = 0; tile < te; tile++, lt++) {
                const int h = (int)(tile / tiles_per_tensor);
                if (h != cur_h) {
                    if (nb > 0) tc_commit(smem_u32(b_empty));
                    if (!mbar_wait(smem_u32(b_full), nb & 1, abort_flag)) break;
                    nb++;
                    cur_h = h;
                }
                // tile lt goes to accumulator and epilogue group lt % 2, free once the
                // group released its previous tile
                const uint32_t buf = (uint32_t)lt & 1u, grp = buf, use = (uint32_t)lt >> 1;
                if (!mbar_wait(smem_u32(acc_empty + grp), (use & 1u) ^ 1u, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem + buf * acc_stride;
                // k = 0, 1: hi plane blocks against B hi and B lo; k = 2, 3: lo plane against
                // B hi.  Each A block's slot is released as soon as its MMAs complete.
                bool ok = true;
                for (int k = 0; k < 4 && ok; k++) {
                    const uint32_t q = 4u * (uint32_t)lt + k, s = q % nslots;
                    if (!mbar_wait(smem_u32(a_full + s), (q / nslots) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t dA = sw128_desc(smem_u32(sA + s * kKBlockBytes));
                    const int kb = k & 1;
                    const int nbp = k < 2 ? 2 : 1;
                    for (int bp = 0; bp < nbp; bp++)
                        for (int kk = 0; kk < 4; kk++)
                            tc_mma(d, dA + (uint64_t)((kk * 32) >> 4),
                                   dB0 + (uint64_t)(((bp * 2 + kb) * bsub + kk * 32) >> 4), idesc,
                                   (k | bp | kk) != 0);
                    tc_commit(smem_u32(a_empty + s));
                }
                if (!ok) break;
                tc_commit(smem_u32(acc_full + grp));
            }
            // every MMA issued so far completes before TMEM is released
            tc_commit(smem_u32(fin));
            mbar_wait_final(smem_u32(fin), 0);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Two groups of 8 warps take turns: group g handles the tiles with lt % 2 == g, found
        // in TMEM accumulator g.  Warp w reads TMEM lanes 32*(w%4).. (its 32 rows); the two
        // warps of a group with the same lanes split the columns, and the lower-column warp
        // merges the pair's results through shared memory.
        const int e = warp - 2;
        const int grp = e >> 3, half = (e >> 2) & 1, quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int C = p.C;
        const int nchunks = (Cpad + 31) >> 5;
        const int split = (nchunks + 1) >> 1;
        const int ch_lo = half ? split : 0, ch_hi = half ? nchunks : split;
        const int pair_bar = 1 + grp * 4 + quarter;  // named barrier of the two warps of a row block
        const int grp_bar = 9 + grp;                  // named barrier of the group's 8 warps
        float *cns = cn_s + grp * Cpad;
        float *xb = x_best + grp * kTileM, *xs = x_second + grp * kTileM;
        int *xi = x_idx + grp * kTileM;
        int cur_h = -1;
        float cmax = 0.f, cmax2 = 0.f;
        unsigned n_ref_rows = 0;
        for (int64_t tile = tb + grp, lt = grp; tile < te; tile += kEpiGroups, lt += kEpiGroups) {
            const int h = (int)(tile / tiles_per_tensor);
            const int64_t i = (tile - (int64_t)h * tiles_per_tensor) * kTileM + row;
            const bool valid = i < p.N;
            const uint32_t buf = (uint32_t)grp, use = (uint32_t)lt >> 1;
            const float rn = (half == 0 && valid) ? __ldg(p.rnorm + (int64_t)h * p.N + i) : 0.f;
            const bool ok = mbar_wait(smem_u32(acc_full + grp), use & 1u, abort_flag);
            // every warp of the group takes the same branch after the bounded wait; this is
            // also the group barrier that ends the previous tile's reads of ||c||^2
            uint32_t any_fail;
            asm volatile(
                "{\n\t.reg .pred p, q;\n\tsetp.eq.u32 p, %1, 0;\n\t"
                "bar.red.or.pred q, %2, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}\n"
                : "=r"(any_fail)
                : "r"((uint32_t)(ok ? 1 : 0)), "r"(grp_bar)
                : "memory");
            if (any_fail) break;
            if (h != cur_h) {
                // the group's private copy of ||c||^2 for this tensor
                cur_h = h;
                const float *cn = p.cn + (int64_t)h * Cpad;
                for (int j = e * 32 + lane - grp * 256; j < Cpad; j += 256) cns[j] = __ldg(cn + j);
                asm volatile("bar.sync %0, 256;" ::"r"(grp_bar) : "memory");
                cmax2 = 0.f;
                for (int j = lane; j < C; j += 32) cmax2 = fmaxf(cmax2, cns[j]);
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1)
                    cmax2 = fmaxf(cmax2, __shfl_xor_sync(0xffffffffu, cmax2, o));
                cmax = sqrtf(cmax2);
            }
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + buf * acc_stride;
            float best = INFINITY, second = INFINITY;
            int bj = 0;
#pragma unroll 1
            for (int cb = ch_lo; cb < ch_hi; cb++) {
                float v[32];
                tc_ld32(taddr + cb * 32, v);
#pragma unroll
                for (int q = 0; q < 32; q += 4) {
                    const float4 c4 = *reinterpret_cast<const float4 *>(cns + cb * 32 + q);
                    const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                    for (int u = 0; u < 4; u++) {
                        const int j = cb * 32 + q + u;
                        const float s = j < C ? __fmaf_rn(-2.f, v[q + u], cc[u]) : INFINITY;
                        second = fminf(second, fmaxf(s, best));
                        if (s < best) bj = j;
                        best = fminf(best, s);
                    }
                }
            }
            if (half == 1) {
                xb[row] = best;
                xs[row] = second;
                xi[row] = bj;
            }
            asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
            if (half == 0) {
                const float ob = xb[row], os = xs[row];
                const int oj = xi[row];
                second = fminf(fminf(second, os), fmaxf(best, ob));
                if (ob < best) bj = oj;  // the lower half wins ties: lowest cluster index
                best = fminf(best, ob);
            }
            // |error of a score| <= 2^-12 ||r|| ||c_j|| + 2^-17 ||c_j||^2; two scores differ
            // from their exact values by at most twice that.
            const float margin = 2.f * (ldexpf(rn * cmax, -12) + ldexpf(cmax2, -17)) + 1e-30f;
            const float lim = best + margin;
            const bool need = half == 0 && valid && second <= lim;
            uint32_t cand[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            if (half == 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int cb = 0; cb < 8; cb++) {
                    if (cb < nchunks) {
                        float v[32];
                        tc_ld32(taddr + cb * 32, v);
#pragma unroll
                        for (int q = 0; q < 32; q++) {
                            const int j = cb * 32 + q;
                            const float s = __fmaf_rn(-2.f, v[q], cns[j]);
                            if (need && j < C && s <= lim) cand[cb] |= 1u << q;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(acc_empty + grp));
            if (half == 0 && valid) {
                p.pi[(int64_t)(h * p.T + t - 1) * p.cap + p.tok_off + i] = (uint8_t)bj;
                if (need) {
                    n_ref_rows++;
                    const int slot = atomicAdd(p.rq_count, 1);
                    RefineReq *rq = p.rq + slot;
                    rq->h = h;
                    rq->i = (int)i;
#pragma unroll
                    for (int cb = 0; cb < 8; cb++) rq->cand[cb] = cand[cb];
                }
            }
        }
        if (p.stats && half == 0) {
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                n_ref_rows += __shfl_xor_sync(0xffffffffu, n_ref_rows, o);
            if (lane == 0 && n_ref_rows) atomicAdd(p.stats + kStatRefineRows, n_ref_rows);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) or_status(p.status, QVG_DEV_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(tmem_cols)
                     : "memory");
    }
}

// --------------------------------------------------------------------------------------
// Exact re-scoring of near ties.  One warp per queued token: lane l holds channels
// 4l..4l+3 of the fp32 residual; each candidate's squared distance is a 4-term partial sum
// per lane reduced over the warp in a fixed order.  Candidates are visited in increasing
// cluster order and only a strictly smaller distance replaces the best, so ties go to the
// lowest index.   grid-stride over the queue, block 256.
// --------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_refine(QPlan p, int t) {
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nw = (gridDim.x * blockDim.x) >> 5;
    const int count = *p.rq_count;
    unsigned n_cands = 0;
    for (int r = gw; r < count; r += nw) {
        const RefineReq rq = p.rq[r];
        const int h = rq.h;
        const int64_t i = rq.i;
        float4 x;
        if (t == 1) {
            float v8[8];
            load_x8(p.X, p.in_dtype, h * p.x_stride + i * kD + (lane >> 1) * 8, v8);
            const int o = (lane & 1) * 4;
            x = make_float4(v8[o], v8[o + 1], v8[o + 2], v8[o + 3]);
        } else {
            x = __ldg(reinterpret_cast<const float4 *>(p.R32 + ((int64_t)h * p.N + i) * kD) + lane);
        }
        const float *c0 = p.cent + h * p.cent_tstride + p.cent_off + (int64_t)(t - 1) * p.C * kD;
        float bestD = INFINITY;
        int bestj = 0;
#pragma unroll
        for (int cb = 0; cb < 8; cb++) {
            uint32_t m = rq.cand[cb];
            while (m) {
                const int j = cb * 32 + __ffs(m) - 1;
                m &= m - 1u;
                n_cands++;
                const float4 c = __ldg(reinterpret_cast<const float4 *>(c0 + (int64_t)j * kD) + lane);
                const float d0 = __fsub_rn(x.x, c.x), d1 = __fsub_rn(x.y, c.y);
                const float d2 = __fsub_rn(x.z, c.z), d3 = __fsub_rn(x.w, c.w);
                float D = __fmaf_rn(d3, d3, __fmaf_rn(d2, d2, __fmaf_rn(d1, d1, __fmul_rn(d0, d0))));
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) D = __fadd_rn(D, __shfl_xor_sync(0xffffffffu, D, o));
                if (D < bestD) {
                    bestD = D;
                    bestj = j;
                }
            }
        }
        if (lane == 0) p.pi[(int64_t)(h * p.T + t - 1) * p.cap + p.tok_off + i] = (uint8_t)bestj;
    }
    if (p.stats && lane == 0 && n_cands) atomicAdd(p.stats + kStatRefineCands, n_cands);
}

// --------------------------------------------------------------------------------------
// Host side
// --------------------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    // Resolved once per process; the pointer never changes afterwards.
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(ptr);
    }();
    return fn;
}

static const int kMaxSmem = 232448;  // opt-in shared memory per block on sm_100-class GPUs

// barriers, TMEM slot, abort flag, and per epilogue group ||c||^2 and the column-half
// exchange (best, second, index per row)
static size_t assign_tail_bytes(int nslots, int Cpad) {
    return (size_t)(2 * nslots + 3 + 2 * kEpiGroups) * 8 + 16 + 16 /* alignment */ +
           (size_t)kEpiGroups * (Cpad + 3 * kTileM) * 4;
}

static int assign_slots(int Cpad) {
    for (int n = 12; n >= 4; n--)
        if ((size_t)1024 + 4 * (size_t)Cpad * 128 + (size_t)n * kKBlockBytes +
                assign_tail_bytes(n, Cpad) <= (size_t)kMaxSmem)
            return n;
    return 4;
}

size_t assign_smem_bytes(int Cpad) {
    const int nslots = assign_slots(Cpad);
    return (size_t)1024 + 4 * (size_t)Cpad * 128 + (size_t)nslots * kKBlockBytes +
           assign_tail_bytes(nslots, Cpad);
}

cudaError_t assign_encode(const QPlan &p, AssignMaps *m) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint32_t estr[3] = {1, 1, 1};
    {
        const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)p.N, (cuuint64_t)(2 * p.H)};
        const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)p.N * kD * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)kTileM, 1};
        if (enc(&m->a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.A, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)p.C, (cuuint64_t)(2 * p.H)};
        const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)p.Cpad * kD * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)p.Cpad, 1};
        if (enc(&m->b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.B, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

cudaError_t assign_prepare(const QPlan &p, AssignMaps **out) {
    *out = nullptr;
    if (!encode_fn()) return cudaErrorNotSupported;
    AssignMaps *m = new AssignMaps;
    const cudaError_t e = assign_encode(p, m);
    if (e != cudaSuccess) {
        delete m;
        return e;
    }
    *out = m;
    return cudaSuccess;
}

void assign_release(AssignMaps *maps) { delete maps; }

cudaError_t launch_assign(const QPlan &p, const AssignMaps *maps, int t, int num_sms,
                          cudaStream_t st) {
    const int tiles = (int)((p.N + kTileM - 1) / kTileM);
    const int64_t total = (int64_t)tiles * p.H;
    const int grid = (int)std::min<int64_t>(total, num_sms);
    const int nslots = assign_slots(p.Cpad);
    const size_t smem = assign_smem_bytes(p.Cpad);
    // two accumulators of Cpad fp32 columns, each at least 32 columns wide so that the
    // epilogue's 32-column loads stay inside the allocation
    uint32_t stride = 32;
    while (stride < (uint32_t)p.Cpad) stride <<= 1;
    const uint32_t cols = 2 * stride;
    cudaError_t e = cudaFuncSetAttribute(k_assign, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    k_assign<<<grid, kThreads, smem, st>>>(maps->a, maps->b, p, t, tiles, nslots, cols, stride);
    return cudaGetLastError();
}

cudaError_t launch_refine(const QPlan &p, int t, int num_sms, cudaStream_t st) {
    k_refine<<<num_sms * 2, 256, 0, st>>>(p, t);
    return cudaGetLastError();
}

}  // namespace qvg
