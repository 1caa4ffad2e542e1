// C ABI of libqvg: argument checks, workspace layout and the stage / Lloyd-round loop of
// the quantize path, plus the dequantize and attention entry points.  Declarations and their contracts
// are in include/qvg.h.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.cuh"
#include "qvg.h"

namespace qvg {

cudaError_t launch_init_indices(const QPlan &p, uint64_t seed, int64_t tid_base, cudaStream_t st);

namespace {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// GEMM columns: a multiple of 32, so that the MMA writes every TMEM column the epilogue's
// 32-column loads read.
inline int cpad_of(int C) { return (C + 31) / 32 * 32; }

struct WsLayout {
    size_t A, rnorm, dnorm, B, Bx, cnd, mu, counts, offs, blockoff, ids, cid, items, psum, wsum, tot,
        ccount, dleave, pi_prev, init_idx, stats, rq_cta, rq, total;
    int nsb, nchunk;
};

WsLayout ws_layout(int64_t H, int64_t N, int C, int T) {
    WsLayout w{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    w.stats = take(64);
    if (T > 0) {
        const int Cpad = cpad_of(C);
        w.A = take((size_t)H * N * kD * 2);
        w.rnorm = take((size_t)H * N * 4);
        w.dnorm = take((size_t)H * N * 4);
        w.B = take((size_t)H * Cpad * kD * 2);
        w.Bx = take((size_t)H * Cpad * kOffsetRow * 4);
        w.cnd = take((size_t)H * Cpad * 8);
        w.mu = take((size_t)H * kD * 4);
        const int64_t icap = 2 * N;  // items: a token, or two events of a changed token
        w.nsb = (int)((N + kSortBlock - 1) / kSortBlock);
        w.nchunk = (int)((icap + kChunk - 1) / kChunk);
        w.counts = take((size_t)H * C * 4);
        w.offs = take((size_t)H * C * 4);
        w.blockoff = take((size_t)H * w.nsb * C * 4);
        w.ids = take((size_t)H * icap * 4);
        w.cid = take((size_t)H * icap);
        w.items = take((size_t)H * 4);
        w.psum = take((size_t)H * w.nchunk * 4 * kD * 4);
        w.wsum = take((size_t)H * C * 2 * kD * 4);
        w.tot = take((size_t)H * C * 2 * kD * 4);
        w.ccount = take((size_t)H * C * 4);
        w.dleave = take((size_t)H * C * 4);
        w.pi_prev = take((size_t)H * N);
        w.init_idx = take((size_t)H * T * C * 4);
        w.rq_cta = take((size_t)2 * kMaxAssignCtas * 4);
        w.rq = take((size_t)H * ((N + kAssignTileM - 1) / kAssignTileM) * kAssignTileM *
                    sizeof(RefineReq));
    }
    w.total = off;
    return w;
}

int elem_bytes(int dt) { return dt == QVG_F32 ? 4 : 2; }

qvg_status check_quant(const qvg_quant_params *p) {
    if (!p) return QVG_ERR_INVALID_ARG;
    if (p->n_tensors < 1 || p->N < 1 || p->N >= (int64_t(1) << 31)) return QVG_ERR_INVALID_ARG;
    if (p->d != kD) return QVG_ERR_UNSUPPORTED;
    if (p->bits != 2 && p->bits != 4) return QVG_ERR_UNSUPPORTED;
    if (p->group != 16 && p->group != 32 && p->group != 64) return QVG_ERR_UNSUPPORTED;
    if (p->qscheme != QVG_QSCHEME_SYMMETRIC && p->qscheme != QVG_QSCHEME_MIDRISE)
        return QVG_ERR_UNSUPPORTED;
    if (p->centroid_format < QVG_CENTROIDS_F32 || p->centroid_format > QVG_CENTROIDS_BF16)
        return QVG_ERR_UNSUPPORTED;
    if (p->T < 0 || p->T > kMaxT) return QVG_ERR_UNSUPPORTED;
    if (p->in_dtype < QVG_F16 || p->in_dtype > QVG_F32) return QVG_ERR_UNSUPPORTED;
    if (p->T > 0) {
        if (p->C < 1 || p->C > kMaxC) return QVG_ERR_UNSUPPORTED;
        if (p->C > p->N) return QVG_ERR_INVALID_ARG;
        if (p->iters < 1) return QVG_ERR_INVALID_ARG;
    }
    if (p->x_stride < 0 || p->token_offset < 0 || p->token_capacity < 0 || p->warm_stride < 0)
        return QVG_ERR_INVALID_ARG;
    if (p->x_stride != 0 && p->x_stride < p->N * kD) return QVG_ERR_INVALID_ARG;
    if (p->x_stride * elem_bytes(p->in_dtype) % 16 != 0) return QVG_ERR_INVALID_ARG;
    const int64_t cap = p->token_capacity ? p->token_capacity : p->N;
    if (p->token_offset + p->N > cap) return QVG_ERR_INVALID_ARG;
    const int n_tables = p->n_tables ? p->n_tables : 1;
    if (n_tables < 1 || p->table_index < 0 || p->table_index >= n_tables) return QVG_ERR_INVALID_ARG;
    if (p->warm_stride != 0 && p->warm_stride < (int64_t)p->T * p->C * kD) return QVG_ERR_INVALID_ARG;
    if (p->warm_stride % 4 != 0) return QVG_ERR_INVALID_ARG;
    return QVG_OK;
}

qvg_status check_quant_buffers(const qvg_quant_params *prm, const void *X, const float *warm,
                               const qvg_buffers *out) {
    if (!X || !out || !out->codes || !out->scales) return QVG_ERR_INVALID_ARG;
    if (prm->T > 0 && (!out->pi || !out->centroids)) return QVG_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(out->codes) || !aligned16(out->scales) ||
        (prm->T > 0 && !aligned16(out->centroids)) || (warm && !aligned16(warm)))
        return QVG_ERR_INVALID_ARG;
    return QVG_OK;
}

qvg_status device_info(int *num_sms) {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QVG_ERR_CUDA;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return QVG_ERR_CUDA;
    if (major != 10 || minor != 3) return QVG_ERR_DEVICE;
    return QVG_OK;
}

#define QVG_CUDA(call)                                \
    do {                                              \
        if ((call) != cudaSuccess) {                  \
            (void)cudaGetLastError();                 \
            return QVG_ERR_CUDA;                      \
        }                                             \
    } while (0)

// Host-side fault injection, for testing the callers' error paths without faulting a GPU:
// QVG_FAULT_INJECT=launch makes every call that would enqueue device work return
// QVG_ERR_CUDA once its arguments are checked, as a failed launch would (nothing is
// enqueued); =alloc makes qvg_quantize_static's scratch lookup fail the same way;
// =timeout runs every assignment launch of qvg_quantize with its centroid operand withheld
// and a 1 ms wait limit, the path qvg_selftest_assign_timeout exercises: the device status
// gets QVG_DEV_TIMEOUT and the results are unspecified; =assign makes the first assignment
// launch of qvg_quantize fail (it is not enqueued), after the kernels before it were
// enqueued, so the call returns QVG_ERR_CUDA from the middle of its sequence.  Read at
// every call.
enum FaultMode { kFaultNone = 0, kFaultAlloc, kFaultLaunch, kFaultTimeout, kFaultAssign };
FaultMode fault_mode() {
    const char *v = getenv("QVG_FAULT_INJECT");
    if (!v) return kFaultNone;
    if (!strcmp(v, "alloc")) return kFaultAlloc;
    if (!strcmp(v, "launch")) return kFaultLaunch;
    if (!strcmp(v, "timeout")) return kFaultTimeout;
    if (!strcmp(v, "assign")) return kFaultAssign;
    return kFaultNone;
}

// The T smoothing stages: cold-start or warm centroids, then `iters` Lloyd rounds each.
qvg_status run_stages(QPlan &p, const AssignMaps *maps, int num_sms, cudaStream_t st) {
    const FaultMode fm = fault_mode();
    const bool inject_timeout = fm == kFaultTimeout, inject_assign = fm == kFaultAssign;
    qvg_status rc = QVG_OK;
    // the sort's item and leave counts start at zero; each update leaves them at zero again
    if (cudaMemsetAsync(p.counts, 0, (size_t)p.H * p.C * 4, st) != cudaSuccess ||
        cudaMemsetAsync(p.dleave, 0, (size_t)p.H * p.C * 4, st) != cudaSuccess)
        return QVG_ERR_CUDA;
    // Each launch reads what the earlier ones wrote, so after a failed launch nothing more is
    // enqueued (a re-scoring launched after a failed assignment would read a queue no kernel
    // of this call wrote).
    auto step = [&](auto &&launch) {
        if (rc == QVG_OK && launch() != cudaSuccess) rc = QVG_ERR_CUDA;
    };
    for (int t = 1; t <= p.T && rc == QVG_OK; t++) {
        if (t == 1) step([&] { return launch_init_centroids(p, t, st); });
        step([&] { return launch_centre(p, t, st); });
        step([&] { return launch_prep(p, t, st); });
        if (t >= 2) step([&] { return launch_init_centroids(p, t, st); });
        step([&] { return launch_centroid_planes(p, t, st); });
        for (int it = 1; it <= p.iters && rc == QVG_OK; it++) {
            step([&] {
                if (inject_assign) return cudaErrorLaunchFailure;  // as if the launch failed
                return inject_timeout ? launch_assign(p, maps, t, num_sms, st, 1000000ull, 1)
                                      : launch_assign(p, maps, t, num_sms, st);
            });
            step([&] { return launch_refine(p, t, num_sms, st); });
            // The first round sums every member; the ones between fold in the tokens that
            // moved.  The last sums every member again, so the stage's centroids are means
            // of a fresh compensated sum, with no rounding carried over from earlier rounds.
            step([&] {
                return launch_cluster_means(p, maps, t, it < p.iters, it > 1 && it < p.iters, num_sms, st);
            });
        }
    }
    return rc;
}

qvg_status run_quantize(QPlan &p, const qvg_quant_params *prm, int num_sms, cudaStream_t st) {
    if (p.T > 0) {
        if (!p.warm) QVG_CUDA(launch_init_indices(p, prm->seed, prm->tensor_id_base, st));
        AssignMaps *maps = nullptr;
        QVG_CUDA(assign_prepare(p, &maps));
        const qvg_status rc = run_stages(p, maps, num_sms, st);
        assign_release(maps);
        if (rc != QVG_OK) {
            (void)cudaGetLastError();
            return rc;
        }
    }
    QVG_CUDA(launch_encode(p, st));
    return QVG_OK;
}

QPlan make_plan(const qvg_quant_params *prm, const void *X, const float *warm,
                     const qvg_buffers *out, void *workspace, const WsLayout &w,
                     uint32_t *dev_status) {
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    QPlan p{};
    p.H = prm->n_tensors;
    p.N = prm->N;
    p.C = prm->T > 0 ? prm->C : 1;
    p.Cpad = cpad_of(p.C);
    p.T = prm->T;
    p.bits = prm->bits;
    p.group = prm->group;
    p.qscheme = prm->qscheme;
    p.cfmt = prm->centroid_format;
    p.iters = prm->iters;
    p.in_dtype = prm->in_dtype;
    p.x_stride = prm->x_stride ? prm->x_stride : prm->N * kD;
    p.cap = prm->token_capacity ? prm->token_capacity : prm->N;
    p.tok_off = prm->token_offset;
    const int n_tables = prm->n_tables ? prm->n_tables : 1;
    p.cent_tstride = (int64_t)n_tables * p.T * p.C * kD;
    p.cent_off = (int64_t)prm->table_index * p.T * p.C * kD;
    p.X = X;
    p.codes = out->codes;
    p.scales = out->scales;
    p.pi = out->pi;
    p.cent = out->centroids;
    p.warm = warm;
    p.warm_stride = prm->warm_stride ? prm->warm_stride : (int64_t)p.T * p.C * kD;
    p.stats = reinterpret_cast<unsigned *>(ws + w.stats);
    if (p.T > 0) {
        p.A = reinterpret_cast<__half *>(ws + w.A);
        p.rnorm = reinterpret_cast<float *>(ws + w.rnorm);
        p.dnorm = reinterpret_cast<float *>(ws + w.dnorm);
        p.B = reinterpret_cast<__half *>(ws + w.B);
        p.Bx = reinterpret_cast<float *>(ws + w.Bx);
        p.cnd = reinterpret_cast<float2 *>(ws + w.cnd);
        p.mu = reinterpret_cast<float *>(ws + w.mu);
        p.counts = reinterpret_cast<int *>(ws + w.counts);
        p.offs = reinterpret_cast<int *>(ws + w.offs);
        p.blockoff = reinterpret_cast<int *>(ws + w.blockoff);
        p.ids = reinterpret_cast<int *>(ws + w.ids);
        p.cid = reinterpret_cast<uint8_t *>(ws + w.cid);
        p.psum = reinterpret_cast<float *>(ws + w.psum);
        p.wsum = reinterpret_cast<float *>(ws + w.wsum);
        p.items = reinterpret_cast<int *>(ws + w.items);
        p.tot = reinterpret_cast<float *>(ws + w.tot);
        p.ccount = reinterpret_cast<int *>(ws + w.ccount);
        p.dleave = reinterpret_cast<int *>(ws + w.dleave);
        p.pi_prev = reinterpret_cast<uint8_t *>(ws + w.pi_prev);
        p.icap = 2 * p.N;
        p.nsb = w.nsb;
        p.nchunk = w.nchunk;
        p.init_idx = reinterpret_cast<int *>(ws + w.init_idx);
        p.rq_cta = reinterpret_cast<int *>(ws + w.rq_cta);
        p.rq = reinterpret_cast<RefineReq *>(ws + w.rq);
    }
    p.status = dev_status;
    return p;
}

// Scratch area of qvg_quantize_static.  A __device__ variable exists once in every CUDA
// context that loads this module, so each device (and each further context a caller
// creates) has its own copy.
static __device__ __align__(256) unsigned char g_static_scratch[QVG_STATIC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

// cuCtxGetCurrent, resolved once through the runtime (no link-time dependence on libcuda).
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<CtxGetCurrentFn>(ptr);
    }();
    return fn;
}

// The area's device address, looked up once per context: the address belongs to the context
// whose copy of the module it points into, so it is keyed by the current context, not by the
// device ordinal (a caller may make a context of its own current on a device).
constexpr int kMaxContexts = 64;
std::mutex g_static_mu;
CUcontext g_static_ctx[kMaxContexts];
void *g_static_addr[kMaxContexts];
int g_static_n = 0;

qvg_status static_scratch(void **addr) {
    CtxGetCurrentFn get = ctx_get_current();
    if (!get) return QVG_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS) return QVG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_static_mu);
    for (int k = 0; ctx && k < g_static_n; k++)
        if (g_static_ctx[k] == ctx) {
            *addr = g_static_addr[k];
            return QVG_OK;
        }
    // not seen yet (or no context current: the runtime then binds the device's primary
    // context on this lookup, and that is the one to key)
    void *a = nullptr;
    if (cudaGetSymbolAddress(&a, g_static_scratch) != cudaSuccess || !a) {
        (void)cudaGetLastError();
        return QVG_ERR_CUDA;
    }
    if (!ctx && (get(&ctx) != CUDA_SUCCESS || !ctx)) return QVG_ERR_CUDA;
    if (g_static_n < kMaxContexts) {  // beyond that, look the address up on every call
        g_static_ctx[g_static_n] = ctx;
        g_static_addr[g_static_n] = a;
        g_static_n++;
    }
    *addr = a;
    return QVG_OK;
}

}  // namespace
}  // namespace qvg

using namespace qvg;

extern "C" {

size_t qvg_quantize_workspace_bytes(const qvg_quant_params *params) {
    if (check_quant(params) != QVG_OK) return 0;
    return ws_layout(params->n_tensors, params->N, params->C, params->T).total;
}

qvg_status qvg_quantize(const qvg_quant_params *prm, const void *X, const float *warm,
                        const qvg_buffers *out, void *workspace, size_t workspace_bytes,
                        uint32_t *dev_status, void *stream) {
    qvg_status rc = check_quant(prm);
    if (rc != QVG_OK) return rc;
    rc = check_quant_buffers(prm, X, warm, out);
    if (rc != QVG_OK) return rc;
    const WsLayout w = ws_layout(prm->n_tensors, prm->N, prm->C, prm->T);
    if (!workspace || workspace_bytes < w.total) return QVG_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return QVG_ERR_INVALID_ARG;
    if (fault_mode() == kFaultLaunch) return QVG_ERR_CUDA;
    int num_sms = 0;
    rc = device_info(&num_sms);
    if (rc != QVG_OK) return rc;

    QPlan p = make_plan(prm, X, warm, out, workspace, w, dev_status);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(p.stats, 0, 64, st) != cudaSuccess) {
        (void)cudaGetLastError();
        return QVG_ERR_CUDA;
    }
    return run_quantize(p, prm, num_sms, st);
}

qvg_status qvg_quantize_static(const qvg_quant_params *prm, const void *X, const float *warm,
                               const qvg_buffers *out, uint32_t *dev_status, void *stream) {
    qvg_status rc = check_quant(prm);
    if (rc != QVG_OK) return rc;
    const WsLayout w = ws_layout(prm->n_tensors, prm->N, prm->C, prm->T);
    if (w.total > QVG_STATIC_SCRATCH_BYTES) return QVG_ERR_SCRATCH_LIMIT;
    rc = check_quant_buffers(prm, X, warm, out);
    if (rc != QVG_OK) return rc;
    const FaultMode fm = fault_mode();
    if (fm == kFaultLaunch || fm == kFaultAlloc) return QVG_ERR_CUDA;
    int num_sms = 0;
    rc = device_info(&num_sms);
    if (rc != QVG_OK) return rc;
    void *workspace = nullptr;
    rc = static_scratch(&workspace);
    if (rc != QVG_OK) return rc;

    QPlan p = make_plan(prm, X, warm, out, workspace, w, dev_status);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    QVG_CUDA(cudaMemsetAsync(p.stats, 0, 64, st));
    if (p.T > 0) {
        if (!p.warm) QVG_CUDA(launch_init_indices(p, prm->seed, prm->tensor_id_base, st));
        AssignMaps maps;  // kernel parameters are copied at launch: stack storage is enough
        QVG_CUDA(assign_encode(p, &maps));
        rc = run_stages(p, &maps, num_sms, st);
        if (rc != QVG_OK) {
            (void)cudaGetLastError();
            return rc;
        }
    }
    QVG_CUDA(launch_encode(p, st));
    return QVG_OK;
}

qvg_status qvg_reassign_steps(const qvg_quant_params *prm, const void *X, const qvg_buffers *out,
                              void *workspace, size_t workspace_bytes, int32_t steps,
                              uint32_t *dev_status, void *stream) {
    qvg_status rc = check_quant(prm);
    if (rc != QVG_OK) return rc;
    if (prm->T < 1) return QVG_ERR_INVALID_ARG;
    if ((steps & ~(QVG_STEP_PLANES | QVG_STEP_GEMM | QVG_STEP_REFINE)) != 0)
        return QVG_ERR_INVALID_ARG;
    if (!X || !out || !out->pi || !out->centroids) return QVG_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(out->centroids)) return QVG_ERR_INVALID_ARG;
    const WsLayout w = ws_layout(prm->n_tensors, prm->N, prm->C, prm->T);
    if (!workspace || workspace_bytes < w.total) return QVG_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return QVG_ERR_INVALID_ARG;
    if (fault_mode() == kFaultLaunch) return QVG_ERR_CUDA;
    int num_sms = 0;
    rc = device_info(&num_sms);
    if (rc != QVG_OK) return rc;
    QPlan p = make_plan(prm, X, nullptr, out, workspace, w, dev_status);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    AssignMaps *maps = nullptr;
    if (assign_prepare(p, &maps) != cudaSuccess) {
        (void)cudaGetLastError();
        return QVG_ERR_CUDA;
    }
    cudaError_t e = cudaSuccess;
    if (steps & QVG_STEP_PLANES) e = launch_centroid_planes(p, p.T, st);
    if (e == cudaSuccess && (steps & QVG_STEP_GEMM)) e = launch_assign(p, maps, p.T, num_sms, st);
    if (e == cudaSuccess && (steps & QVG_STEP_REFINE)) e = launch_refine(p, p.T, num_sms, st);
    assign_release(maps);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return QVG_ERR_CUDA;
    }
    return QVG_OK;
}

qvg_status qvg_reassign(const qvg_quant_params *prm, const void *X, const qvg_buffers *out,
                        void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                        void *stream) {
    return qvg_reassign_steps(prm, X, out, workspace, workspace_bytes,
                              QVG_STEP_PLANES | QVG_STEP_GEMM | QVG_STEP_REFINE, dev_status, stream);
}

qvg_status qvg_selftest_assign_timeout(const qvg_quant_params *prm, const void *X,
                                       const qvg_buffers *out, void *workspace,
                                       size_t workspace_bytes, uint32_t *dev_status,
                                       void *stream) {
    qvg_status rc = check_quant(prm);
    if (rc != QVG_OK) return rc;
    if (prm->T < 1) return QVG_ERR_INVALID_ARG;
    if (!X || !out || !out->pi || !out->centroids) return QVG_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(out->centroids)) return QVG_ERR_INVALID_ARG;
    const WsLayout w = ws_layout(prm->n_tensors, prm->N, prm->C, prm->T);
    if (!workspace || workspace_bytes < w.total) return QVG_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return QVG_ERR_INVALID_ARG;
    if (fault_mode() == kFaultLaunch) return QVG_ERR_CUDA;
    int num_sms = 0;
    rc = device_info(&num_sms);
    if (rc != QVG_OK) return rc;
    QPlan p = make_plan(prm, X, nullptr, out, workspace, w, dev_status);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    AssignMaps *maps = nullptr;
    if (assign_prepare(p, &maps) != cudaSuccess) {
        (void)cudaGetLastError();
        return QVG_ERR_CUDA;
    }
    // the centroid operand's load withheld, a wait limit of one millisecond
    cudaError_t e = launch_centroid_planes(p, p.T, st);
    if (e == cudaSuccess) e = launch_assign(p, maps, p.T, num_sms, st, 1000000ull, 1);
    assign_release(maps);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return QVG_ERR_CUDA;
    }
    return QVG_OK;
}

qvg_status qvg_dequantize(const qvg_dequant_params *prm, const qvg_buffers *in, void *X_hat,
                          uint32_t *dev_status, void *stream) {
    if (!prm || !in || !X_hat || !in->codes || !in->scales) return QVG_ERR_INVALID_ARG;
    if (prm->n_tensors < 1 || prm->N < 1 || prm->N >= (int64_t(1) << 31)) return QVG_ERR_INVALID_ARG;
    if (prm->d != kD) return QVG_ERR_UNSUPPORTED;
    if (prm->bits != 2 && prm->bits != 4) return QVG_ERR_UNSUPPORTED;
    if (prm->group != 16 && prm->group != 32 && prm->group != 64) return QVG_ERR_UNSUPPORTED;
    if (prm->qscheme != QVG_QSCHEME_SYMMETRIC && prm->qscheme != QVG_QSCHEME_MIDRISE)
        return QVG_ERR_UNSUPPORTED;
    if (prm->T < 0 || prm->T > kMaxT) return QVG_ERR_UNSUPPORTED;
    if (prm->out_dtype < QVG_F16 || prm->out_dtype > QVG_F32) return QVG_ERR_UNSUPPORTED;
    if (prm->T > 0 && (prm->C < 1 || prm->C > kMaxC)) return QVG_ERR_UNSUPPORTED;
    if (prm->T > 0 && (!in->pi || !in->centroids)) return QVG_ERR_INVALID_ARG;
    if (prm->chunk_len < 0 || prm->token_capacity < 0 || prm->n_tables < 0 || prm->out_stride < 0)
        return QVG_ERR_INVALID_ARG;
    const int64_t cap = prm->token_capacity ? prm->token_capacity : prm->N;
    const int64_t chunk = prm->chunk_len ? prm->chunk_len : prm->N;
    const int n_tables = prm->n_tables ? prm->n_tables : 1;
    const int64_t ostride = prm->out_stride ? prm->out_stride : prm->N * kD;
    if (cap < prm->N || ostride < prm->N * kD) return QVG_ERR_INVALID_ARG;
    if (prm->T > 0 && (prm->N + chunk - 1) / chunk > n_tables) return QVG_ERR_INVALID_ARG;
    if (ostride * elem_bytes(prm->out_dtype) % 16 != 0) return QVG_ERR_INVALID_ARG;
    if (!aligned16(X_hat) || !aligned16(in->codes) || !aligned16(in->scales) ||
        (prm->T > 0 && !aligned16(in->centroids)))
        return QVG_ERR_INVALID_ARG;
    if (fault_mode() == kFaultLaunch) return QVG_ERR_CUDA;
    int num_sms = 0;
    qvg_status rc = device_info(&num_sms);
    if (rc != QVG_OK) return rc;
    DPlan p{};
    p.H = prm->n_tensors;
    p.N = prm->N;
    p.C = prm->T > 0 ? prm->C : 1;
    p.T = prm->T;
    p.bits = prm->bits;
    p.group = prm->group;
    p.out_dtype = prm->out_dtype;
    p.qscheme = prm->qscheme;
    p.chunk_len = chunk;
    p.cap = cap;
    p.n_tables = n_tables;
    p.out_stride = ostride;
    p.codes = in->codes;
    p.scales = in->scales;
    p.pi = in->pi;
    p.cent = in->centroids;
    p.out = X_hat;
    p.status = dev_status;
    if (launch_dequant(p, num_sms, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        (void)cudaGetLastError();
        return QVG_ERR_CUDA;
    }
    return QVG_OK;
}

namespace {
qvg_status check_attention(const qvg_attention_params *prm) {
    if (!prm) return QVG_ERR_INVALID_ARG;
    if (prm->n_heads < 1 || prm->N < 1 || prm->N >= (int64_t(1) << 31)) return QVG_ERR_INVALID_ARG;
    if (prm->M < 1 || prm->M > kMaxAttnQ) return QVG_ERR_UNSUPPORTED;
    if (prm->n_heads > 65535) return QVG_ERR_UNSUPPORTED;  // one grid row per head
    if (prm->d != kD) return QVG_ERR_UNSUPPORTED;
    if (prm->bits != 2 && prm->bits != 4) return QVG_ERR_UNSUPPORTED;
    if (prm->group != 16 && prm->group != 32 && prm->group != 64) return QVG_ERR_UNSUPPORTED;
    if (prm->qscheme != QVG_QSCHEME_SYMMETRIC && prm->qscheme != QVG_QSCHEME_MIDRISE)
        return QVG_ERR_UNSUPPORTED;
    if (prm->T < 0 || prm->T > kMaxT) return QVG_ERR_UNSUPPORTED;
    if (prm->T > 0 && (prm->C < 1 || prm->C > kMaxC)) return QVG_ERR_UNSUPPORTED;
    if (prm->q_dtype < QVG_F16 || prm->q_dtype > QVG_F32) return QVG_ERR_UNSUPPORTED;
    if (prm->out_dtype < QVG_F16 || prm->out_dtype > QVG_F32) return QVG_ERR_UNSUPPORTED;
    if (!std::isfinite(prm->scale)) return QVG_ERR_INVALID_ARG;
    if (prm->chunk_len < 0 || prm->token_capacity < 0 || prm->n_tables < 0 ||
        prm->k_first < 0 || prm->v_first < 0 || prm->tensor_step < 0)
        return QVG_ERR_INVALID_ARG;
    const int64_t cap = prm->token_capacity ? prm->token_capacity : prm->N;
    const int64_t chunk = prm->chunk_len ? prm->chunk_len : prm->N;
    const int n_tables = prm->n_tables ? prm->n_tables : 1;
    if (cap < prm->N) return QVG_ERR_INVALID_ARG;
    if (prm->T > 0 && (prm->N + chunk - 1) / chunk > n_tables) return QVG_ERR_INVALID_ARG;
    return QVG_OK;
}

struct AttnWs {
    size_t part, ml, total;
};

AttnWs attn_layout(const qvg_attention_params *prm) {
    const int64_t L = attn_split_len(prm->N, prm->n_heads);
    const int64_t S = (prm->N + L - 1) / L;
    const size_t rows = (size_t)prm->n_heads * S * prm->M;
    AttnWs w{};
    w.part = 0;
    w.ml = (rows * kD * sizeof(float) + 255) / 256 * 256;
    w.total = w.ml + (rows * 2 * sizeof(float) + 255) / 256 * 256;
    return w;
}
}  // namespace

size_t qvg_attention_workspace_bytes(const qvg_attention_params *prm) {
    if (check_attention(prm) != QVG_OK) return 0;
    return attn_layout(prm).total;
}

qvg_status qvg_attention(const qvg_attention_params *prm, const void *Q,
                         const qvg_buffers *k_cache, const qvg_buffers *v_cache, void *O,
                         void *workspace, size_t ws_bytes, uint32_t *dev_status, void *stream) {
    qvg_status rc = check_attention(prm);
    if (rc != QVG_OK) return rc;
    if (!Q || !O || !k_cache || !v_cache) return QVG_ERR_INVALID_ARG;
    for (const qvg_buffers *b : {k_cache, v_cache}) {
        if (!b->codes || !b->scales) return QVG_ERR_INVALID_ARG;
        if (prm->T > 0 && (!b->pi || !b->centroids)) return QVG_ERR_INVALID_ARG;
        if (!aligned16(b->codes) || !aligned16(b->scales) || (prm->T > 0 && !aligned16(b->centroids)))
            return QVG_ERR_INVALID_ARG;
    }
    if (!aligned16(Q) || !aligned16(O)) return QVG_ERR_INVALID_ARG;
    const AttnWs w = attn_layout(prm);
    if (!workspace || ws_bytes < w.total || !aligned16(workspace)) return QVG_ERR_WORKSPACE;
    if (fault_mode() == kFaultLaunch) return QVG_ERR_CUDA;
    int num_sms = 0;
    rc = device_info(&num_sms);
    if (rc != QVG_OK) return rc;
    APlan p{};
    p.H = prm->n_heads;
    p.M = prm->M;
    p.N = prm->N;
    p.C = prm->T > 0 ? prm->C : 1;
    p.T = prm->T;
    p.bits = prm->bits;
    p.group = prm->group;
    p.qscheme = prm->qscheme;
    p.chunk_len = prm->chunk_len ? prm->chunk_len : prm->N;
    p.cap = prm->token_capacity ? prm->token_capacity : prm->N;
    p.n_tables = prm->n_tables ? prm->n_tables : 1;
    p.q_dtype = prm->q_dtype;
    p.out_dtype = prm->out_dtype;
    p.scale = prm->scale;
    p.k_first = prm->k_first;
    p.v_first = prm->v_first;
    p.step = prm->tensor_step;
    p.split_len = attn_split_len(prm->N, prm->n_heads);
    p.S = (int)((prm->N + p.split_len - 1) / p.split_len);
    p.Q = Q;
    p.kc = k_cache->codes;
    p.ks = k_cache->scales;
    p.kp = k_cache->pi;
    p.kcent = k_cache->centroids;
    p.vc = v_cache->codes;
    p.vs = v_cache->scales;
    p.vp = v_cache->pi;
    p.vcent = v_cache->centroids;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    p.part = reinterpret_cast<float *>(ws + w.part);
    p.ml = reinterpret_cast<float *>(ws + w.ml);
    p.O = O;
    p.status = dev_status;
    if (launch_attention(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        (void)cudaGetLastError();
        return QVG_ERR_CUDA;
    }
    return QVG_OK;
}

const char *qvg_status_string(qvg_status s) {
    switch (s) {
        case QVG_OK: return "ok";
        case QVG_ERR_INVALID_ARG: return "invalid argument (null, misaligned or inconsistent size)";
        case QVG_ERR_UNSUPPORTED: return "unsupported shape or parameter value";
        case QVG_ERR_WORKSPACE: return "workspace missing or too small";
        case QVG_ERR_CUDA: return "CUDA error while enqueuing work";
        case QVG_ERR_DEVICE: return "current device is not an sm_103 GPU";
        case QVG_ERR_SCRATCH_LIMIT:
            return "problem needs more scratch than qvg_quantize_static's fixed area holds";
    }
    return "unknown status";
}

uint32_t qvg_version(void) { return (1u << 16) | 1u; }

}  // extern "C"
