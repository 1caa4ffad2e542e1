// Internal declarations shared by the CUDA translation units of libqvg.
//
// Numerics used on the device (the oracle works in fp64; these are the GPU's choices):
//   * Residuals r = x - C^(1)[pi^(1)] - ... are formed with an error-free TwoSum chain and
//     rounded once to fp32, so r is the fp32 value nearest the exact residual.
//   * Centroid sums run in a fixed order over the tokens grouped by cluster (a stable
//     counting sort), with TwoSum-compensated fp32 accumulation of the exact stage input
//     (from the second stage on, each residual enters as its fp32 value plus the rounding
//     error of the chain that formed it); the mean is rounded once to fp32.  Repeated runs
//     give identical bits.
//   * Distances for the assignment come from tensor-core MMAs: fp16 copies of the centred
//     operands plus a tf32 per-centroid offset, accumulated in fp32.  Every cluster whose
//     score lies within a rigorous bound on its error of the best one is re-scored exactly
//     (fp32, then fp64 where fp32 cannot separate them), ties going to the lowest index.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <utility>

#include "qvg.h"

namespace qvg {

constexpr int kD = 128;            // channels per token
constexpr int kMaxT = 8;           // most smoothing stages
constexpr int kMaxC = 256;         // most clusters (pi is uint8)
// fp32 values per row of the assignment's offset table (one 128-byte TMA row)
constexpr int kOffsetRow = 32;
// Largest |component| that the fp16 GEMM operands are trusted with; a residual row or a
// centroid set with a larger norm sends every cluster of the row to the exact re-scoring.
constexpr float kFp16Safe = 60000.f;

enum : int { DT_F16 = 0, DT_BF16 = 1, DT_F32 = 2 };

// Everything a quantize call's kernels need, resolved on the host.
struct QPlan {
    int H;
    int64_t N;
    int C, Cpad, T, bits, group, iters, in_dtype;  // Cpad: C rounded up to a multiple of 32
    int qscheme;           // qvg_qscheme of the codes
    int cfmt;              // qvg_centroid_format of the stored centroids
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
    __half *A;             // [H][N][128] fp16 copy of the centred residual r - mu
    float *rnorm;          // [H][N] norm of the centred residual row (fp32)
    float *dnorm;          // [H][N] norm of its fp16 rounding error, ||fp16(r - mu) - (r - mu)||
    __half *B;             // [H][Cpad][128] fp16(c - mu) of the centred centroids
    float *Bx;             // [H][Cpad][kOffsetRow] the offset -||c - mu||^2 / 2 as three tf32
                           // parts (h, m, l, 0, ...); -2^100 in the padded rows
    float2 *cnd;           // [H][Cpad] (||c - mu||^2, ||fp16(c - mu) - (c - mu)||) per centroid
    float *mu;             // [H][128] centring vector of the current stage
    // The mean update sorts items by cluster: in a stage's first round every token, in
    // later rounds two events per token whose cluster changed (it leaves its old cluster,
    // enters the new one), so the item capacity per tensor is icap = 2N.
    int *counts;           // [H][C] items of each cluster this round
    int *offs;             // [H][C] first position of each cluster's items in `ids`
    int *blockoff;         // [H][nsb][C] per token block: its first position per cluster
    int *ids;              // [H][icap] token index of each sorted item, bit 31 set for an item
                           // that leaves its cluster; increasing within a cluster's enters
                           // (and leaves) of one token block
    uint8_t *cid;          // [H][icap] cluster of each sorted item
    int *items;            // [H] items sorted this round
    float *psum;           // [H][nchunk][2][2][128] (sum, error) of the runs that cross a
                           // chunk boundary: [0] the run at the chunk start, [1] the last run
    float *wsum;           // [H][C][2][128] (sum, error) of clusters inside one chunk
    float *tot;            // [H][C][2][128] (sum, error) of each cluster's members, kept
                           // from round to round of a stage (renormalised: |error| <= ulp/2)
    int *ccount;           // [H][C] members of each cluster, kept from round to round
    int *dleave;           // [H][C] leave events of each cluster this round
    uint8_t *pi_prev;      // [H][N] the previous round's assignment of the stage
    int64_t icap;          // item capacity per tensor (2N)
    int nsb, nchunk;       // token blocks of the sort, 32-position chunks per tensor (of icap)
    int *init_idx;         // [H][T][C] cold-start rows
    unsigned *stats;       // [16] counters (see kStat*)
    int *rq_cta;           // [2 * kMaxAssignCtas] per assignment CTA: first slot of its
                           // region of rq, requests queued there
    struct RefineReq *rq;  // [H * tiles * kAssignTileM] near-tie re-scoring requests
    uint32_t *status;      // caller's device status word (may be NULL)
};

enum { kStatRefineRows = 0, kStatRefineCands = 1 };
// Most CTAs of one assignment launch (its grid is min(tiles, SMs), capped to this).
constexpr int kMaxAssignCtas = 1024;
// Tokens per assignment tile.  The near-tie queue has one slot per row of every tile (a
// tensor's last tile may be ragged), and each assignment CTA owns the slots of its tiles.
constexpr int kAssignTileM = 128;

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

// The fp32 value v as three tf32 parts, v = h + m + l exactly: h is v rounded to tf32
// (11 significant bits), m the remainder rounded to tf32, l what is left (at most two
// significant bits).  Each difference is exact in fp32.
__device__ __forceinline__ float tf32_round(float x) {
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}
__device__ __forceinline__ void tf32_split3(float v, float &h, float &m, float &l) {
    h = tf32_round(v);
    const float r = __fsub_rn(v, h);
    m = tf32_round(r);
    l = __fsub_rn(r, m);
}

// Two lanes of fp32 at once (packed f32x2 instructions).  a - b is taken as fma(b, -1, a),
// which rounds the same exact difference once, so every result equals the scalar form's.
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    return __ffma2_rn(b, make_float2(-1.f, -1.f), a);
}
// s + x on a pair, its exact rounding error added to e (compensated accumulation)
__device__ __forceinline__ void acc_two_sum2(float2 &s, float2 &e, float2 x) {
    const float2 sn = __fadd2_rn(s, x);
    const float2 bb = sub2(sn, s);
    const float2 err = __fadd2_rn(sub2(s, sub2(sn, bb)), sub2(x, bb));
    e = __fadd2_rn(e, err);
    s = sn;
}
// a - c on a pair with its exact rounding error: a - c = d + err exactly (TwoSum of a and
// -c, the negation folded into the last step)
__device__ __forceinline__ float2 two_diff2(float2 a, float2 c, float2 &err) {
    const float2 d = sub2(a, c);
    const float2 bb = sub2(d, a);
    err = sub2(sub2(a, sub2(d, bb)), __fadd2_rn(c, bb));
    return d;
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

__device__ __forceinline__ void or_status(uint32_t *status, uint32_t bits) {
    if (status) atomicOr(status, bits);
}

// ------------------------------------------------------------------------------------
// mbarrier and bulk-copy primitives (inline PTX)
// ------------------------------------------------------------------------------------

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

// try_wait that may suspend the thread until the phase completes, for at most the hinted
// time (the hardware wakes it as soon as the phase completes).
constexpr uint32_t kSuspendHintNs = 20000;  // longest single suspension in a wait
__device__ __forceinline__ bool mbar_try_suspend(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0u;
}

// TMA gather of four rows (2D tensor map whose box is one row high) into consecutive
// shared memory, counted on the mbarrier's transaction count.  col * element size must be
// a multiple of 16 bytes.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap *map, int col, int r0,
                                            int r1, int r2, int r3, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bulk copy (the TMA unit's untiled form) of `bytes` from global to shared memory, counted
// on the mbarrier's transaction count.  Both addresses 16-byte aligned, bytes a multiple
// of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// ------------------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation and begins with pdl_begin(): it lets the next kernel
// in the stream launch (its CTAs take SM slots as this grid's CTAs retire) and then waits
// until the previous kernel has completed and its writes are visible.  Kernel boundaries
// then cost no launch latency and no empty ramp; the order of memory effects is that of
// plain stream order.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_begin() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------------------------------------
// Launchers (each enqueues on `st`; returns the CUDA error of the launch)
// ------------------------------------------------------------------------------------

cudaError_t launch_init_centroids(const QPlan &p, int t, cudaStream_t st);
cudaError_t launch_centre(const QPlan &p, int t, cudaStream_t st);
cudaError_t launch_prep(const QPlan &p, int t, cudaStream_t st);
cudaError_t launch_centroid_planes(const QPlan &p, int t, cudaStream_t st);
struct AssignMaps;
// Stage t's new centroids from its assignment; planes: also their assignment operands;
// delta: fold the tokens whose cluster changed since the previous round into the cluster
// totals that round kept (otherwise sum every member afresh).
cudaError_t launch_cluster_means(const QPlan &p, const AssignMaps *maps, int t, bool planes,
                                 bool delta, int num_sms, cudaStream_t st);
constexpr int kSortBlock = 256;  // tokens per block of the counting sort
constexpr int kChunk = 32;       // sorted positions summed by one warp
cudaError_t launch_encode(const QPlan &p, cudaStream_t st);

// TMA tensor maps of the assignment GEMM: A = residual planes, B = centroid planes.
struct AssignMaps {
    CUtensorMap a;
    CUtensorMap b;
    CUtensorMap bx;  // the offset rows
    // row view for the cluster sums' gathers: X as [rows][128] (when every tensor starts on
    // a whole row, x_stride % 128 == 0; gather = 0 otherwise)
    CUtensorMap x_rows;
    int gather;
};
// Encodes the maps for plan p into caller-provided storage (no allocation).
cudaError_t assign_encode(const QPlan &p, AssignMaps *maps);
// Heap-allocates the maps and encodes them; free with assign_release.
cudaError_t assign_prepare(const QPlan &p, AssignMaps **maps);
void assign_release(AssignMaps *maps);
// A pipeline wait in the assignment kernel gives up after this long (then it sets
// QVG_DEV_TIMEOUT and the kernel unwinds); withhold_b only for the failure self-test.
constexpr uint64_t kAssignWaitNs = 2000000000ull;
cudaError_t launch_assign(const QPlan &p, const AssignMaps *maps, int t, int num_sms,
                          cudaStream_t st, uint64_t wait_ns = kAssignWaitNs, int withhold_b = 0);
cudaError_t launch_refine(const QPlan &p, int t, int num_sms, cudaStream_t st);
size_t assign_smem_bytes(int Cpad, int nslots);

struct DPlan {
    int H;
    int64_t N;
    int C, T, bits, group, out_dtype, qscheme;
    int64_t chunk_len, cap;
    int n_tables;
    int64_t out_stride;
    const uint8_t *codes, *scales, *pi;
    const float *cent;
    void *out;
    uint32_t *status;
};
cudaError_t launch_dequant(const DPlan &p, int num_sms, cudaStream_t st);

// Attention read straight from two compressed caches (keys and values).
constexpr int kMaxAttnQ = 16;  // most queries per head
struct APlan {
    int H, M;                  // heads, queries per head
    int64_t N;                 // keys per head
    int C, T, bits, group, qscheme;
    int64_t chunk_len, cap;
    int n_tables;
    int q_dtype, out_dtype;
    float scale;
    int64_t k_first, v_first, step;  // tensor of head h: first + h * step
    int S;                     // key splits per head
    int64_t split_len;         // keys per split (a multiple of 32)
    const void *Q;             // [H][M][d]
    const uint8_t *kc, *ks, *kp;
    const float *kcent;
    const uint8_t *vc, *vs, *vp;
    const float *vcent;
    float *part;               // [H][S][M][d] unnormalised partial outputs
    float *ml;                 // [H][S][M][2] running maximum and weight sum of each split
    void *O;                   // [H][M][d]
    uint32_t *status;
};
// Keys per split: about 2048 splits over all heads (a warp each, enough to cover the SMs
// with several warps apiece), at least 64 keys and a multiple of the 32-key tile.  Every
// split s < S = ceil(N / split_len) holds a key.
inline int64_t attn_split_len(int64_t N, int64_t heads) {
    const int64_t target = std::max<int64_t>(2048 / std::max<int64_t>(heads, 1), 1);
    const int64_t len = std::max<int64_t>((N + target - 1) / target, 64);
    return (len + 31) / 32 * 32;
}
cudaError_t launch_attention(const APlan &p, cudaStream_t st);

}  // namespace qvg
