// Exact re-scoring of the rows the tensor-core assignment left with near ties, sm_103a.
//
// Method step: pi_i = argmin_j ||R_i - C_j||^2 over the C centroids of the current stage,
// ties to the lowest j ("Quant VideoGen" notes page, section Semantic-Aware Smoothing, step
// 1; review page, pipeline step (a)).  The assignment kernel (k_assign.cu) decides every row
// whose best score is further than twice its error bound from all others; the rest are
// queued, with one bit per candidate cluster, and settled here.
#include <algorithm>

#include "internal.cuh"

namespace qvg {

// --------------------------------------------------------------------------------------
// Re-scoring of near ties.  One half-warp per queued token, two tokens a warp; lane l of a
// half holds channels 8l..8l+7.  First every candidate's squared distance is summed in fp32
// on the fp32 stage input (an 8-term fused chain per lane, reduced over the half-warp in a
// fixed order).  If the best two are further apart than fp32 can blur, that decides.
// Otherwise (a tie at fp32 resolution, rare) the stage input is rebuilt in fp64 from X and
// the earlier stages' centroids, by the same subtraction chain as the fp64 reference, and
// the candidates are scored again in fp64.  Candidates are visited in increasing cluster
// order and only a strictly smaller distance replaces the best, so ties go to the lowest
// index.  Blocks of 256 threads; several blocks share each assignment CTA's region of the
// queue.  The kernel is bound by the latency of each request's dependent reads, so it is
// built for four blocks per SM (64 registers, a few spilled): 96 us per stage-4 launch at
// the 13B-class shape against 102 us at three blocks (80 registers) and 135 us at two.
// --------------------------------------------------------------------------------------
template <int TP>  // t - 1 (0..3), or -1: any stage, with the earlier rows read one at a time
__global__ void __launch_bounds__(256, 4) k_refine(QPlan p, int t, int n_regions, int split) {
    pdl_begin();
    const int lane = threadIdx.x & 31, hl = lane & 15;
    const unsigned hmask = lane < 16 ? 0x0000FFFFu : 0xFFFF0000u;  // this half-warp
    // blocks b, b + n_regions, ... share region b % n_regions of the queue (one region per
    // assignment CTA); their half-warps stride over its requests
    const int region = blockIdx.x % n_regions;
    const int gh = ((blockIdx.x / n_regions) * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 2 + (lane >> 4);
    const int nh = split * (blockDim.x >> 5) * 2;
    int first = p.rq_cta[2 * region], count = p.rq_cta[2 * region + 1];
    // The queue is the one the assignment of this call wrote.  A region outside the queue's
    // capacity (the re-scoring step run with no assignment before it) is skipped and
    // reported, and so is a request for a row outside the problem; candidate bits at or past
    // C are ignored.  None of these occur when the steps run in order.
    const int64_t rq_cap = (int64_t)p.H * ((p.N + kAssignTileM - 1) / kAssignTileM) * kAssignTileM;
    if (first < 0 || count < 0 || (int64_t)first + count > rq_cap) {
        if (threadIdx.x == 0 && blockIdx.x < n_regions) or_status(p.status, QVG_DEV_BAD_INDEX);
        first = count = 0;
    }
    auto cand_word = [&](const RefineReq *rq, int w) {  // bits of clusters < C only
        const int live = p.C - 32 * w;
        const uint32_t keep = live >= 32 ? 0xFFFFFFFFu : (live <= 0 ? 0u : (1u << live) - 1u);
        return rq->cand[w] & keep;
    };
    auto hsum = [&](float v) {  // the half-warp's sum, the same in every lane of it
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(hmask, v, o));
        return v;
    };
    unsigned n_cands = 0;
    // A request's reads are issued together, not one after another: the next request is
    // read while this one is scored; this one's X row, earlier clusters and first two
    // candidates' rows go out together, then every earlier stage's centroid row at once,
    // then any further candidates two at a time.
    int cur_h = 0, cur_i = 0;
    if (gh < count) {
        cur_h = p.rq[first + gh].h;
        cur_i = p.rq[first + gh].i;
    }
    for (int r = gh; r < count; r += nh) {
        const RefineReq *rqp = p.rq + first + r;  // its candidate words are in L1 by now
        const bool has_next = r + nh < count;
        int nxt_h = 0, nxt_i = 0;
        if (has_next) {
            nxt_h = rqp[nh].h;
            nxt_i = rqp[nh].i;
        }
        const int h = cur_h;
        const int64_t i = cur_i;
        cur_h = nxt_h;
        cur_i = nxt_i;
        if ((unsigned)h >= (unsigned)p.H || i < 0 || i >= p.N) {  // the same in the half-warp
            if (hl == 0) or_status(p.status, QVG_DEV_BAD_INDEX);
            continue;
        }
        const float *ct = p.cent + h * p.cent_tstride + p.cent_off;
        const float *c0 = ct + (int64_t)(t - 1) * p.C * kD;
        constexpr int NB = TP > 0 ? TP : 1;  // earlier stages batched
        auto earlier = [&](int s2) {            // cluster of stage s2 + 1
            return min((int)p.pi[(int64_t)(h * p.T + s2) * p.cap + p.tok_off + i], p.C - 1);
        };
        int js[NB];
#pragma unroll
        for (int s2 = 0; s2 < NB; s2++) js[s2] = TP > 0 ? earlier(s2) : 0;
        // X's channels 8*hl..8*hl+7
        float xs[8];
        load_x8(p.X, p.in_dtype, h * p.x_stride + i * kD + hl * 8, xs);
        // candidates in increasing cluster order, two at a time; the first two rows now
        constexpr int KB = 2;
        int cb = 0;
        uint32_t m = cand_word(rqp, 0);
        int jj[KB], nb = 0;
        float4 ca[KB], cc[KB];
        auto next_batch = [&]() {
            nb = 0;
#pragma unroll
            for (int u = 0; u < KB; u++) {
                while (m == 0u && cb < 7) m = cand_word(rqp, ++cb);
                jj[u] = -1;
                if (m) {
                    jj[u] = cb * 32 + __ffs(m) - 1;
                    m &= m - 1u;
                    nb++;
                }
            }
#pragma unroll
            for (int u = 0; u < KB; u++)
                if (jj[u] >= 0) {
                    const float4 *cr = reinterpret_cast<const float4 *>(c0 + (int64_t)jj[u] * kD) + 2 * hl;
                    ca[u] = __ldg(cr);
                    cc[u] = __ldg(cr + 1);
                }
        };
        next_batch();
        // fp32 pass on the fp32 stage input: X itself at stage 1, later the residual formed
        // by the same TwoSum chain (one final rounding) as the GEMM operand's preparation
        float2 x[4];
#pragma unroll
        for (int q = 0; q < 4; q++) x[q] = make_float2(xs[2 * q], xs[2 * q + 1]);
        auto row8 = [&](int s2, int j, float4 &a, float4 &b) {  // stage s2 + 1's row j
            const float4 *cr = reinterpret_cast<const float4 *>(ct + ((int64_t)s2 * p.C + j) * kD) + 2 * hl;
            a = __ldg(cr);
            b = __ldg(cr + 1);
        };
        if (TP != 0) {
            float2 e[4];
#pragma unroll
            for (int q = 0; q < 4; q++) e[q] = make_float2(0.f, 0.f);
            auto sub_row = [&](const float4 &a, const float4 &b) {
                const float2 c[4] = {make_float2(a.x, a.y), make_float2(a.z, a.w), make_float2(b.x, b.y),
                                     make_float2(b.z, b.w)};
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    float2 err;
                    x[q] = two_diff2(x[q], c[q], err);
                    e[q] = __fadd2_rn(e[q], err);
                }
            };
            if (TP > 0) {
                float4 cra[NB], crb[NB];
#pragma unroll
                for (int s2 = 0; s2 < NB; s2++) row8(s2, js[s2], cra[s2], crb[s2]);
#pragma unroll
                for (int s2 = 0; s2 < NB; s2++) sub_row(cra[s2], crb[s2]);
            } else {
                for (int s2 = 0; s2 + 1 < t; s2++) {
                    float4 a, b;
                    row8(s2, earlier(s2), a, b);
                    sub_row(a, b);
                }
            }
#pragma unroll
            for (int q = 0; q < 4; q++) x[q] = __fadd2_rn(x[q], e[q]);
        }
        float bestD = INFINITY, secondD = INFINITY;
        int bestj = 0;
        for (;;) {
            if (nb == 0) break;
#pragma unroll
            for (int u = 0; u < KB; u++)
                if (jj[u] >= 0) {
                    n_cands++;
                    const float cv[8] = {ca[u].x, ca[u].y, ca[u].z, ca[u].w, cc[u].x, cc[u].y, cc[u].z, cc[u].w};
                    float D = 0.f;
#pragma unroll
                    for (int q = 0; q < 8; q++) {
                        const float d = __fsub_rn(q & 1 ? x[q >> 1].y : x[q >> 1].x, cv[q]);
                        D = q == 0 ? __fmul_rn(d, d) : __fmaf_rn(d, d, D);
                    }
                    D = hsum(D);
                    if (D < bestD) {
                        secondD = bestD;
                        bestD = D;
                        bestj = jj[u];
                    } else {
                        secondD = fminf(secondD, D);
                    }
                }
            if (nb < KB) break;
            next_batch();
        }
        bool close = secondD - bestD <= 0x1p-18f * secondD;
        if (!close && t > 1) {
            float xx = 0.f;
#pragma unroll
            for (int q = 0; q < 4; q++) xx = __fmaf_rn(x[q].y, x[q].y, __fmaf_rn(x[q].x, x[q].x, xx));
            const float xn = sqrtf(hsum(xx));
            if (xn > 0.f)
                close = secondD - bestD <= 0x1p-18f * secondD + 0x1.1p-22f * xn * sqrtf(secondD);
        }
        if (close) {
            // the stage input rebuilt in fp64: x - C^(1)[pi^(1)] - ... - C^(t-1)[pi^(t-1)],
            // subtracted in that order
            double xd[8];
            load_x8(p.X, p.in_dtype, h * p.x_stride + i * kD + hl * 8, xs);
#pragma unroll
            for (int k = 0; k < 8; k++) xd[k] = (double)xs[k];
            for (int s2 = 0; s2 + 1 < t; s2++) {
                float4 ca, cb2;
                row8(s2, earlier(s2), ca, cb2);
                const float cv[8] = {ca.x, ca.y, ca.z, ca.w, cb2.x, cb2.y, cb2.z, cb2.w};
#pragma unroll
                for (int k = 0; k < 8; k++) xd[k] -= (double)cv[k];
            }
            double bestDd = INFINITY;
            for (int cw = 0; cw < 8; cw++) {
                uint32_t mm = cand_word(rqp, cw);
                while (mm) {
                    const int j = cw * 32 + __ffs(mm) - 1;
                    mm &= mm - 1u;
                    const float4 *cr = reinterpret_cast<const float4 *>(c0 + (int64_t)j * kD) + 2 * hl;
                    const float4 ca = __ldg(cr), cc = __ldg(cr + 1);
                    const float cv[8] = {ca.x, ca.y, ca.z, ca.w, cc.x, cc.y, cc.z, cc.w};
                    double D = 0.0;
#pragma unroll
                    for (int k = 0; k < 8; k++) {
                        const double e = xd[k] - (double)cv[k];
                        D = __fma_rn(e, e, D);
                    }
#pragma unroll
                    for (int o = 8; o >= 1; o >>= 1) D += __shfl_xor_sync(hmask, D, o);
                    if (D < bestDd) {
                        bestDd = D;
                        bestj = j;
                    }
                }
            }
        }
        if (hl == 0) p.pi[(int64_t)(h * p.T + t - 1) * p.cap + p.tok_off + i] = (uint8_t)bestj;
    }
    if (p.stats && hl == 0 && n_cands) atomicAdd(p.stats + kStatRefineCands, n_cands);
}

// The assignment's grid for plan p (the number of queue regions it leaves).
static int assign_grid(const QPlan &p, int num_sms) {
    const int64_t total = (int64_t)((p.N + kAssignTileM - 1) / kAssignTileM) * p.H;
    return (int)std::min<int64_t>(std::min<int64_t>(total, num_sms), kMaxAssignCtas);
}

cudaError_t launch_refine(const QPlan &p, int t, int num_sms, cudaStream_t st) {
    const int regions = assign_grid(p, num_sms);
    const int split = std::max(1, (num_sms * 8 + regions - 1) / regions);
    const dim3 grid(regions * split);
    switch (t - 1) {
        case 0: return launch_kernel(k_refine<0>, grid, dim3(256), 0, st, p, t, regions, split);
        case 1: return launch_kernel(k_refine<1>, grid, dim3(256), 0, st, p, t, regions, split);
        case 2: return launch_kernel(k_refine<2>, grid, dim3(256), 0, st, p, t, regions, split);
        case 3: return launch_kernel(k_refine<3>, grid, dim3(256), 0, st, p, t, regions, split);
        default: return launch_kernel(k_refine<-1>, grid, dim3(256), 0, st, p, t, regions, split);
    }
}

}  // namespace qvg
