// k-means assignment on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// Method step: pi_i = argmin_j ||R_i - C_j||^2 over the C centroids of the current stage,
// ties to the lowest j ("Quant VideoGen" notes page, section Semantic-Aware Smoothing, step
// 1; review page, pipeline step (a)).
//
// Both operands are first shifted by a common centring vector mu (distances do not change):
// a = R_i - mu and c_j = C_j - mu.  Then
//   ||R_i - C_j||^2 = ||a||^2 - 2 (a.c_j - ||c_j||^2 / 2),
// so the nearest centroid is the one with the largest score t_j = a.c_j - ||c_j||^2 / 2, and
// the scores of a tile of 128 tokens are one [128 x 128] x [128 x C] product plus a per-column
// offset.  Both parts run on the tensor cores into one fp32 TMEM accumulator:
//   * the offset: one kind::tf32 MMA (K = 8) of a constant A block (every row 1, 1, 1, 0, ...)
//     with B rows (h_j, m_j, l_j, 0, ...), the exact three-part tf32 split of the fp32 value
//     -||c_j||^2 / 2, issued first (it initialises the accumulator);
//   * the product: eight kind::f16 MMAs (K = 16) of fp16(a) with fp16(c_j), accumulated.
// The epilogue reads finished scores: a maximum per 32-column chunk and candidate bits.
//
// Error bound.  Let A^ = fp16(a), B^_j = fp16(c_j) and dn = ||A^ - a||, dc_j = ||B^_j - c_j||,
// both measured exactly in fp32 by the kernels that write the fp16 copies (typically about
// 0.6 * 2^-11 of the norm).  With rn = ||a||, cmax = max_j ||c_j||, dcmax = max_j dc_j:
//   |A^.B^_j - a.c_j| <= dn (cmax + dcmax) + rn dcmax               (Cauchy-Schwarz)
//   fp32 accumulation of the offset and 128 exact products, at most 144 roundings of at
//   most 2^-23 of the running magnitude: <= 2^-15 ((rn + dn)(cmax + dcmax) + cmax^2 / 2)
//   the offset: ||c_j||^2 summed in fp32 (four fused terms a lane, a five-level butterfly)
//   is within 2^-20 of itself, and its tf32 split is exact: <= 2^-21 cmax^2
// so every score is within E of a.c_j - ||c_j||^2 / 2 computed exactly on the fp32 operands,
//   E = 1.01 dn (cmax + dcmax) + 1.01 rn dcmax + 2^-15 (rn + dn)(cmax + dcmax)
//       + 2^-15 cmax^2 + 2^-20 (rn + dn),
// the last term a margin for the fp32 rounding of the centred operands and of the stage
// input itself (at most 2^-24 of each component).  Any cluster whose score is within 2E of
// the best score may be the true nearest one; those clusters are re-scored by k_refine, in
// fp64 on the stage input rebuilt in fp64 wherever fp32 cannot separate them, so the chosen
// index is that of the nearest centroid up to fp64 rounding: the same choice as an fp64
// reference, ties to the lowest index.  A row with ||a|| >= 60000, or a centroid set with
// cmax >= 60000, could overflow fp16: all of its clusters are re-scored.
//
// Kernel structure (one persistent CTA per SM, 576 threads):
//   warp 0   TMA producer: B (the fp16 centroid plane, C x 128) and the offset rows
//            (C x 32 fp32) once per tensor, then A (128 tokens x 128 channels fp16 per tile,
//            as two 16 KB blocks of 64 channels) into a ring of smem slots.
//   warp 1   TMEM allocator and MMA issuer (one thread): per tile one tf32 MMA and 2 x 4
//            f16 MMAs of M = 128, N = Cpad into one of two TMEM accumulators.
//   warps 2-17 epilogue, two groups of 8 warps taking alternate tiles: a warp reads 32
//            TMEM lanes (one token row per thread) and half of the columns, 64 columns per
//            TMEM load, once.  For each 32-column chunk it takes the largest score, updates
//            the row's running best and sets one candidate bit per score at or above the
//            running limit best - 2E (the sign of score - limit, shifted in).  The pair of
//            warps on the same rows exchanges their bests for the row's; chunks whose
//            largest score is below the row's limit are cleared (see the epilogue for why
//            the rest is exact where it matters).  Then the accumulator is released; a row
//            with one candidate gets it as pi, a row with several is queued for k_refine.
// Every mbarrier wait is bounded (2 s by default, a launch argument); on timeout the kernel
// sets QVG_DEV_TIMEOUT, stops, waits for its own copies and MMAs, frees TMEM and returns.
// A self-test withholds the centroid operand's load so that the MMA warp's first wait runs
// out (qvg_selftest_assign_timeout).
#include <cuda.h>

#include <algorithm>

#include "internal.cuh"

namespace qvg {

namespace {

constexpr int kEpiGroups = 2;                      // epilogue groups of 8 warps
constexpr int kThreads = 64 + kEpiGroups * 8 * 32;  // producer, MMA, 16 epilogue warps
constexpr int kTileM = kAssignTileM;
constexpr uint32_t kKBlockBytes = kTileM * 64 * 2;  // 16 KB: 64 fp16 channels of 128 rows
constexpr int kABlocks = 2;                           // A blocks per tile (128 channels)
constexpr uint32_t kAuxABytes = kTileM * 128;         // the constant tf32 block: 128 rows of 128 B
constexpr uint32_t kSpinLimit = 1u << 22;
// maximum of three fp32 values (one instruction on sm_100-class GPUs; NaN inputs are
// ignored unless all three are NaN, as with fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// coefficients of the bound (see the error bound above)
constexpr float kDnRel = 0x1.03p0f;   // 1.01
constexpr float kAccRel = 0x1p-15f;

// Bounded wait on a phase.  Gives up when another role already gave up, or after
// kSpinLimit tries or limit_ns of wall time, whichever comes first (then it raises the
// abort flag itself).
__device__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                          uint64_t limit_ns) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t n = 0; n < kSpinLimit; n++) {
        if (mbar_try_suspend(bar, parity)) return true;
        if (*abort_flag) return false;
        if ((n & 15u) == 15u && global_ns() - t0 > limit_ns) break;
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
// The offset MMA: tf32 operands; accumulate = 0 overwrites the accumulator.
__device__ __forceinline__ void tc_mma_tf32(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane; the wait is in the same asm
// statement, so no use of the values can be scheduled before the data has arrived.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float v[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int q = 0; q < 32; q++) v[q] = __uint_as_float(r[q]);
}

// 64 consecutive fp32 columns (two chunks) in one load.
__device__ __forceinline__ void tc_ld64(uint32_t taddr, float v[64]) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]),
          "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]),
          "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
          "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]),
          "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]),
          "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int q = 0; q < 64; q++) v[q] = __uint_as_float(r[q]);
}

// (tensor, tile within the tensor) of a flat tile index, advanced by a fixed step without a
// 64-bit division per tile (one division when the walk starts).
struct TileWalk {
    int h, ti, tpt;
    __device__ TileWalk(int64_t tile, int tiles_per_tensor) : tpt(tiles_per_tensor) {
        h = (int)(tile / tiles_per_tensor);
        ti = (int)(tile - (int64_t)h * tiles_per_tensor);
    }
    __device__ void advance(int step) {  // step <= tiles_per_tensor is not required
        ti += step;
        while (ti >= tpt) {
            ti -= tpt;
            h++;
        }
    }
};

// Largest of 32 scores, in two independent chains.
__device__ __forceinline__ float chunk_max(const float *v) {
    float ma = fmaxf(v[0], v[1]), mb = fmaxf(v[2], v[3]);
#pragma unroll
    for (int q = 4; q < 32; q += 4) {
        ma = fmax3(ma, v[q], v[q + 1]);
        mb = fmax3(mb, v[q + 2], v[q + 3]);
    }
    return fmaxf(ma, mb);
}

// (hi:lo << 1) >> 32 = (hi << 1) | (lo >> 31): shifts the sign bit of lo into hi.
__device__ __forceinline__ uint32_t shift_in_sign(uint32_t hi, float lo) {
    uint32_t r;
    asm("shf.l.wrap.b32 %0, %1, %2, 1;" : "=r"(r) : "r"(__float_as_uint(lo)), "r"(hi));
    return r;
}

// Candidate bits of a chunk: bit q set when v[q] >= lim (v[q] - lim rounds to a number of
// the same sign as the exact difference, and to +0 when they are equal).
__device__ __forceinline__ uint32_t chunk_cands(const float *v, float lim) {
    const float2 nl = make_float2(-lim, -lim);
    uint32_t w = 0u;  // sign bits, score 31 shifted in first
#pragma unroll
    for (int q = 31; q > 0; q -= 2) {
        const float2 d = __fadd2_rn(make_float2(v[q], v[q - 1]), nl);
        w = shift_in_sign(w, d.x);
        w = shift_in_sign(w, d.y);
    }
    return ~w;
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of 128 bytes,
// 8-row groups 1024 bytes apart (the layout a TMA box of 128-byte rows writes with
// CU_TENSOR_MAP_SWIZZLE_128B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4)   // start address
           | ((uint64_t)1 << 16)                 // leading-dimension offset (unused here)
           | ((uint64_t)(1024 >> 4) << 32)       // stride between 8-row groups
           | ((uint64_t)1 << 46)                 // descriptor version
           | ((uint64_t)2 << 61);                // 128-byte swizzle
}

// Instruction descriptors: fp32 accumulator (bits 4-5 = 1), A and B formats at bits 7-9 and
// 10-12 (kind::f16: 0 = fp16; kind::tf32: 2 = tf32), both K-major, N >> 3 at bit 17,
// M >> 4 at bit 24.
__device__ __forceinline__ uint32_t make_idesc(int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTileM >> 4) << 24);
}
__device__ __forceinline__ uint32_t make_idesc_tf32(int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(kTileM >> 4) << 24);
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    k_assign(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
             const __grid_constant__ CUtensorMap tmBx, QPlan p, int t, int tiles_per_tensor,
             int nslots, uint32_t tmem_cols, uint32_t acc_stride, uint64_t wait_ns,
             int withhold_b) {
    pdl_begin();
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int Cpad = p.Cpad;
    const uint32_t bsub = (uint32_t)Cpad * 128u;  // one 64-channel block of B, or the offset rows
    unsigned char *sB = sm;                       // two blocks of fp16 B
    unsigned char *sBx = sm + 2 * bsub;           // offset rows (tf32, 32 a row)
    unsigned char *sAx = sm + 3 * bsub;           // the constant tf32 A block
    unsigned char *sA = sAx + kAuxABytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sA + (size_t)nslots * kKBlockBytes);
    uint64_t *a_full = bars, *a_empty = bars + nslots;
    uint64_t *b_full = bars + 2 * nslots, *b_empty = b_full + 1;
    uint64_t *acc_full = b_full + 2, *acc_empty = acc_full + kEpiGroups, *fin = acc_empty + kEpiGroups;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *q_count = reinterpret_cast<int *>(tmem_slot + 2);  // requests this CTA queued
    // per epilogue group: the column-half exchange (best score and candidate words per row)
    float *x_best = reinterpret_cast<float *>(
        (reinterpret_cast<uintptr_t>(tmem_slot + 4) + 15) & ~static_cast<uintptr_t>(15));  // [kEpiGroups][2][128]
    uint32_t *x_cand = reinterpret_cast<uint32_t *>(x_best + kEpiGroups * 2 * kTileM);  // [kEpiGroups][128][4]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t total = (int64_t)p.H * tiles_per_tensor;
    const int64_t per = total / gridDim.x, rem = total % gridDim.x;
    const int64_t tb = blockIdx.x * per + min((int64_t)blockIdx.x, rem);
    const int64_t te = tb + per + ((int64_t)blockIdx.x < rem ? 1 : 0);

    // The constant A block of the offset MMA: every row (1, 1, 1, 0, ..., 0) as tf32, in the
    // 128-byte swizzled layout (16-byte chunk c of row r stored at chunk c ^ (r & 7)).
    for (int x = threadIdx.x; x < kTileM * 32; x += kThreads) {
        const int r = x >> 5, col = x & 31;
        const int logical_chunk = (col >> 2) ^ (r & 7);
        reinterpret_cast<float *>(sAx)[x] = (logical_chunk == 0 && (col & 3) < 3) ? 1.f : 0.f;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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
        *q_count = 0;
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
            TileWalk tw(tb, tiles_per_tensor);
            for (int64_t tile = tb, lt = 0; tile < te && !*abort_flag; tile++, lt++, tw.advance(1)) {
                const int h = tw.h;
                const int m0 = tw.ti * kTileM;
                if (h != cur_h) {
                    if (nb > 0 && !mbar_wait(smem_u32(b_empty), (nb - 1) & 1, abort_flag, wait_ns)) break;
                    // (withhold_b: the failure self-test; b_full then never completes)
                    if (!withhold_b) {
                        mbar_expect_tx(smem_u32(b_full), 3 * bsub);
                        for (int kb = 0; kb < 2; kb++)
                            tma_load_3d(smem_u32(sB + kb * bsub), &tmB, kb * 64, 0, h, smem_u32(b_full));
                        tma_load_3d(smem_u32(sBx), &tmBx, 0, 0, h, smem_u32(b_full));
                    }
                    nb++;
                    cur_h = h;
                }
                // two 16 KB loads per tile: channels 0-63, then 64-127
                bool ok = true;
                for (int k = 0; k < kABlocks; k++) {
                    const uint32_t q = kABlocks * (uint32_t)lt + k, s = q % nslots,
                                   ph = (q / nslots) & 1u;
                    if (!mbar_wait(smem_u32(a_empty + s), ph ^ 1u, abort_flag, wait_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(smem_u32(a_full + s), kKBlockBytes);
                    tma_load_3d(smem_u32(sA + s * kKBlockBytes), &tmA, k * 64, m0, h,
                                smem_u32(a_full + s));
                    issued = q + 1;
                }
                if (!ok) break;
            }
            // make sure every copy this CTA started has landed before the CTA can exit
            if (nb > 0 && !withhold_b) mbar_wait_final(smem_u32(b_full), (nb - 1) & 1);
            const uint32_t first = issued > (uint32_t)nslots ? issued - nslots : 0u;
            for (uint32_t q = first; q < issued; q++)
                mbar_wait_final(smem_u32(a_full + q % nslots), (q / nslots) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = make_idesc(Cpad), idesc32 = make_idesc_tf32(Cpad);
            int cur_h = -1;
            uint32_t nb = 0;
            const uint64_t dB0 = sw128_desc(smem_u32(sB));
            const uint64_t dBx = sw128_desc(smem_u32(sBx));
            const uint64_t dAx = sw128_desc(smem_u32(sAx));
            TileWalk tw(tb, tiles_per_tensor);
            for (int64_t tile = tb, lt = 0; tile < te; tile++, lt++, tw.advance(1)) {
                const int h = tw.h;
                if (h != cur_h) {
                    if (nb > 0) tc_commit(smem_u32(b_empty));
                    if (!mbar_wait(smem_u32(b_full), nb & 1, abort_flag, wait_ns)) break;
                    nb++;
                    cur_h = h;
                }
                // tile lt goes to accumulator and epilogue group lt % 2, free once the
                // group released its previous tile
                const uint32_t buf = (uint32_t)lt & 1u, grp = buf, use = (uint32_t)lt >> 1;
                if (!mbar_wait(smem_u32(acc_empty + grp), (use & 1u) ^ 1u, abort_flag, wait_ns)) break;
                tc_fence_after();
                const uint32_t d = tmem + buf * acc_stride;
                // the per-column offset -||c_j||^2 / 2 first: it initialises the accumulator
                tc_mma_tf32(d, dAx, dBx, idesc32, 0u);
                // A block k (channels 64k..64k+63) against the same channels of B; each A
                // block's slot is released as soon as its MMAs complete.
                bool ok = true;
                for (int k = 0; k < kABlocks && ok; k++) {
                    const uint32_t q = kABlocks * (uint32_t)lt + k, s = q % nslots;
                    if (!mbar_wait(smem_u32(a_full + s), (q / nslots) & 1u, abort_flag, wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t dA = sw128_desc(smem_u32(sA + s * kKBlockBytes));
                    for (int kk = 0; kk < 4; kk++)
                        tc_mma(d, dA + (uint64_t)((kk * 32) >> 4),
                               dB0 + (uint64_t)((k * bsub + kk * 32) >> 4), idesc, 1u);
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
        const int nchunks = Cpad >> 5;  // Cpad is a multiple of 32
        const int split = (nchunks + 1) >> 1;
        const int ch_lo = half ? split : 0, ch_hi = half ? nchunks : split;
        const int nc = ch_hi - ch_lo;   // 0 .. 4 chunks for this warp
        const int pair_bar = 1 + grp * 4 + quarter;  // named barrier of the two warps of a row block
        const int grp_bar = 9 + grp;                  // named barrier of the group's 8 warps
        float *xb = x_best + grp * 2 * kTileM;
        uint32_t *xc = x_cand + grp * 4 * kTileM;
        int cur_h = -1;
        float cmax = 0.f, cmax2 = 0.f, dcmax = 0.f;
        unsigned n_ref_rows = 0;
        TileWalk tw(tb + grp, tiles_per_tensor);
        for (int64_t tile = tb + grp, lt = grp; tile < te;
             tile += kEpiGroups, lt += kEpiGroups, tw.advance(kEpiGroups)) {
            const int h = tw.h;
            const int64_t i = (int64_t)tw.ti * kTileM + row;
            const bool valid = i < p.N;
            const uint32_t buf = (uint32_t)grp, use = (uint32_t)lt >> 1;
            const float rn = valid ? __ldg(p.rnorm + (int64_t)h * p.N + i) : 0.f;
            const float dn = valid ? __ldg(p.dnorm + (int64_t)h * p.N + i) : 0.f;
            if (h != cur_h) {
                // the tensor's largest centroid norm and fp16 rounding error (each warp
                // reduces them itself)
                cur_h = h;
                const float2 *cd = p.cnd + (int64_t)h * Cpad;
                float m2 = 0.f, md = 0.f;
                for (int j = lane; j < C; j += 32) {
                    const float2 v = __ldg(cd + j);
                    m2 = fmaxf(m2, v.x);
                    md = fmaxf(md, v.y);
                }
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) {
                    m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, o));
                    md = fmaxf(md, __shfl_xor_sync(0xffffffffu, md, o));
                }
                cmax2 = m2;
                cmax = sqrtf(m2) * 1.000001f;
                dcmax = md;
            }
            const bool ok = mbar_wait(smem_u32(acc_full + grp), use & 1u, abort_flag, wait_ns);
            // every warp of the group takes the same branch after the bounded wait
            uint32_t any_fail;
            asm volatile(
                "{\n\t.reg .pred p, q;\n\tsetp.eq.u32 p, %1, 0;\n\t"
                "bar.red.or.pred q, %2, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}\n"
                : "=r"(any_fail)
                : "r"((uint32_t)(ok ? 1 : 0)), "r"(grp_bar)
                : "memory");
            if (any_fail) break;
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + buf * acc_stride +
                                   (uint32_t)(ch_lo * 32);
            // The row's margin: every cluster whose score is within twice the error bound of
            // the best may be the nearest one (bound in the file header).
            const float cm1 = cmax + dcmax;
            const float two_err = 2.f * (kDnRel * dn * cm1 + kDnRel * rn * dcmax +
                                         kAccRel * ((rn + dn) * cm1 + cmax2) + 0x1p-20f * (rn + dn)) +
                                  1e-30f;
            // An untrusted row (fp16 operands may have overflowed, so its scores may be inf
            // or NaN) takes every cluster as a candidate.
            const bool trusted = rn < kFp16Safe && cmax < kFp16Safe;
            // One pass over this warp's chunks, two per TMEM load: each chunk's largest score,
            // the running best of the row, and candidate bits against the running limit
            // best - 2E.  A chunk read before the row's final best gets its bits against a
            // lower limit, a superset of its true candidates; below, a chunk whose largest
            // score is under the final limit is cleared, and one above it holds a true
            // candidate, so its row goes to exact re-scoring anyway.  The chunk holding the
            // best is always read with the final limit, so a row's single candidate is exact.
            float cm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            uint32_t cand[4] = {0u, 0u, 0u, 0u};
            float own = -INFINITY;
            {
                float v[64];
                if (nc >= 2) {
                    tc_ld64(taddr, v);
                    cm[0] = chunk_max(v);
                    cm[1] = chunk_max(v + 32);
                    own = fmaxf(cm[0], cm[1]);
                    const float lim = own - two_err;
                    cand[0] = chunk_cands(v, lim);
                    cand[1] = chunk_cands(v + 32, lim);
                }
                if (nc == 4) {
                    tc_ld64(taddr + 64, v);
                    cm[2] = chunk_max(v);
                    cm[3] = chunk_max(v + 32);
                    own = fmax3(own, cm[2], cm[3]);
                    const float lim = own - two_err;
                    cand[2] = chunk_cands(v, lim);
                    cand[3] = chunk_cands(v + 32, lim);
                } else if (nc & 1) {
                    const int c = nc - 1;  // 0 or 2
                    tc_ld32(taddr + c * 32, v);
                    const float m = chunk_max(v);
                    own = fmaxf(own, m);
                    const uint32_t w = chunk_cands(v, own - two_err);
                    if (c == 0) {
                        cm[0] = m;
                        cand[0] = w;
                    } else {
                        cm[2] = m;
                        cand[2] = w;
                    }
                }
            }
            // the row's best score over both column halves
            xb[half * kTileM + row] = own;
            asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
            const float best = fmaxf(own, xb[(half ^ 1) * kTileM + row]);
            const float lim = trusted ? best - two_err : -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; c++) {
                uint32_t w = trusted ? (cm[c] < lim ? 0u : cand[c]) : 0xFFFFFFFFu;
                // only real clusters (padded columns score -2^100, but an untrusted row's
                // padded columns are set above)
                const int live = C - (ch_lo + c) * 32;
                if (c >= nc) w = 0u;
                else if (live < 32) w &= (1u << live) - 1u;
                cand[c] = w;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(acc_empty + grp));
            // the upper half hands its candidate words to the lower half, which decides
            if (half == 1)
                *reinterpret_cast<uint4 *>(xc + row * 4) = make_uint4(cand[0], cand[1], cand[2], cand[3]);
            asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
            if (half == 0) {
                // candidate words in chunk order: chunk c belongs to the lower half when
                // c < split
                const uint4 up = *reinterpret_cast<const uint4 *>(xc + row * 4);
                auto word_of = [&](int c) {  // c is a compile-time constant below
                    const uint32_t up_w[4] = {up.x, up.y, up.z, up.w};
                    uint32_t w = 0u;
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        if (c == k && c < split) w = cand[k];
                        if (c == split + k && c < nchunks) w = up_w[k];
                    }
                    return w;
                };
                // words past a half's chunks are zero, so the count and the lowest candidate
                // need no chunk mapping: the lower half's chunks come first
                const int n_cand = __popc(cand[0]) + __popc(cand[1]) + __popc(cand[2]) +
                                   __popc(cand[3]) + __popc(up.x) + __popc(up.y) + __popc(up.z) +
                                   __popc(up.w);
                int bj;
                if (cand[0] | cand[1] | cand[2] | cand[3]) {
                    const int c = cand[0] ? 0 : cand[1] ? 1 : cand[2] ? 2 : 3;
                    const uint32_t w = cand[0] ? cand[0] : cand[1] ? cand[1] : cand[2] ? cand[2] : cand[3];
                    bj = c * 32 + __ffs(w) - 1;
                } else {
                    const int k = up.x ? 0 : up.y ? 1 : up.z ? 2 : 3;
                    const uint32_t w = up.x ? up.x : up.y ? up.y : up.z ? up.z : up.w;
                    bj = (split + k) * 32 + __ffs(w) - 1;
                }
                const bool need = valid && n_cand > 1;
                const unsigned m = __ballot_sync(0xffffffffu, need);
                if (m) {
                    // this CTA's region of the queue: one slot per row of its tiles
                    int base = 0;
                    if (lane == 0) base = atomicAdd(q_count, __popc(m));
                    base = __shfl_sync(0xffffffffu, base, 0);
                    if (need) {
                        n_ref_rows++;
                        RefineReq *rq = p.rq + tb * kTileM + base + __popc(m & ((1u << lane) - 1u));
                        rq->h = h;
                        rq->i = (int)i;
#pragma unroll
                        for (int c = 0; c < 8; c++) rq->cand[c] = word_of(c);
                    }
                }
                // a row with several candidates gets its lowest one here; k_refine
                // overwrites it with the exact choice
                if (valid) p.pi[(int64_t)(h * p.T + t - 1) * p.cap + p.tok_off + i] = (uint8_t)bj;
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
    if (threadIdx.x == 0) {
        if (*abort_flag) or_status(p.status, QVG_DEV_TIMEOUT);
        p.rq_cta[2 * blockIdx.x] = (int)(tb * kTileM);
        p.rq_cta[2 * blockIdx.x + 1] = *q_count;
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(tmem_cols)
                     : "memory");
    }
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

// barriers, TMEM slot, abort flag, and per epilogue group the column-half exchange (best
// score and candidate words per row)
static size_t assign_tail_bytes(int nslots) {
    return (size_t)(2 * nslots + 3 + 2 * kEpiGroups) * 8 + 16 + 16 /* alignment */ +
           (size_t)kEpiGroups * (2 * kTileM + 4 * kTileM) * 4;
}

// the fp16 centroid plane (two 64-channel blocks), the offset rows and the constant block
static size_t assign_fixed_bytes(int Cpad) { return (size_t)3 * Cpad * 128 + kAuxABytes; }

static int assign_slots(int Cpad, size_t max_smem) {
    for (int n = 12; n >= 4; n--)
        if ((size_t)1024 + assign_fixed_bytes(Cpad) + (size_t)n * kKBlockBytes +
                assign_tail_bytes(n) <= max_smem)
            return n;
    return 0;
}

// Opt-in shared memory per block of the current device.
static cudaError_t max_smem_optin(size_t *bytes) {
    int dev = 0, v = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    *bytes = (size_t)v;
    return e;
}

size_t assign_smem_bytes(int Cpad, int nslots) {
    return (size_t)1024 + assign_fixed_bytes(Cpad) + (size_t)nslots * kKBlockBytes +
           assign_tail_bytes(nslots);
}

cudaError_t assign_encode(const QPlan &p, AssignMaps *m) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint32_t estr[3] = {1, 1, 1};
    {
        const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)p.N, (cuuint64_t)p.H};
        const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)p.N * kD * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)kTileM, 1};
        if (enc(&m->a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, p.A, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // the C real rows of each tensor's plane; the padded rows of a box read as zeros
        const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)p.C, (cuuint64_t)p.H};
        const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)p.Cpad * kD * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)p.Cpad, 1};
        if (enc(&m->b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, p.B, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // the offset rows: all Cpad rows (the padded ones hold -2^100, written by
        // k_centroid_planes), 32 fp32 = 128 bytes each
        const cuuint64_t dims[3] = {(cuuint64_t)kOffsetRow, (cuuint64_t)p.Cpad, (cuuint64_t)p.H};
        const cuuint64_t strides[2] = {(cuuint64_t)kOffsetRow * 4,
                                       (cuuint64_t)p.Cpad * kOffsetRow * 4};
        const cuuint32_t box[3] = {(cuuint32_t)kOffsetRow, (cuuint32_t)p.Cpad, 1};
        if (enc(&m->bx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.Bx, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // the row view of X for the cluster sums (a box of one row of 128 elements, as gathers
    // need)
    m->gather = 0;
    if (p.x_stride % kD == 0) {
        const size_t eb = p.in_dtype == DT_F32 ? 4 : 2;
        const CUtensorMapDataType dt = p.in_dtype == DT_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : p.in_dtype == DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        const cuuint64_t xrows = (cuuint64_t)(p.H - 1) * (p.x_stride / kD) + (cuuint64_t)p.N;
        const cuuint32_t box[2] = {(cuuint32_t)kD, 1};
        const cuuint32_t estr2[2] = {1, 1};
        const cuuint64_t xdims[2] = {(cuuint64_t)kD, xrows}, xstr[1] = {(cuuint64_t)kD * eb};
        if (xrows < (1ull << 31) &&
            enc(&m->x_rows, dt, 2, const_cast<void *>(p.X), xdims, xstr, box, estr2,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
            m->gather = 1;
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
                          cudaStream_t st, uint64_t wait_ns, int withhold_b) {
    const int tiles = (int)((p.N + kTileM - 1) / kTileM);
    const int64_t total = (int64_t)tiles * p.H;
    const int grid = (int)std::min<int64_t>(std::min<int64_t>(total, num_sms), kMaxAssignCtas);
    size_t max_smem = 0;
    cudaError_t e = max_smem_optin(&max_smem);
    if (e != cudaSuccess) return e;
    const int nslots = assign_slots(p.Cpad, max_smem);
    if (nslots == 0) return cudaErrorInvalidConfiguration;
    const size_t smem = assign_smem_bytes(p.Cpad, nslots);
    // two accumulators of Cpad fp32 columns, each at least 32 columns wide so that the
    // epilogue's 32-column loads stay inside the allocation
    uint32_t stride = 32;
    while (stride < (uint32_t)p.Cpad) stride <<= 1;
    const uint32_t cols = 2 * stride;
    e = cudaFuncSetAttribute(k_assign, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(k_assign, dim3(grid), dim3(kThreads), smem, st, maps->a, maps->b, maps->bx,
                         p, t, tiles, nslots, cols, stride, wait_ns, withhold_b);
}

}  // namespace qvg
