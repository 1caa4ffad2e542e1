/*
 * qvg.h -- C ABI of libqvg, a GB300 (sm_103a) implementation of the KV-cache compression
 * path of Quant VideoGen (arXiv 2602.02958).
 *
 * The method, as the pages state it:
 *   - Semantic-Aware Smoothing ("Quant VideoGen" notes page, section Semantic-Aware
 *     Smoothing; review page "Quant VideoGen: 基于2-Bit KV缓存量化的自回归长视频生成",
 *     pipeline paragraph, steps (a)-(c)): the N tokens of a per-head tensor X in R^{N x d}
 *     are clustered by k-means along the token axis into C groups, and each token has its
 *     group's centroid (the group mean) subtracted.
 *   - Progressive Residual Quantization (notes page, section Progressive Residual
 *     Quantization; review page, pipeline paragraph): with R^(0) = X, stage t = 1..T
 *     re-applies the smoothing to R^(t-1), producing R^(t), centroids C^(t) and
 *     assignments pi^(t); only R^(T) is quantized.
 *   - Q(R^(T)) is symmetric group integer quantization, INT2 or INT4, with one scale per
 *     group stored as FP8 E4M3 (notes page, section Algorithm-System Co-design; explainer
 *     "Quant VideoGen: Auto-Regressive Long Video Generation via 2-Bit KV-Cache
 *     Quantization", section Step-by-step).
 *   - Reconstruction dequantizes and adds the stages' assigned centroids back from stage T
 *     down to stage 1, fused in one pass (notes page, sections Progressive Residual
 *     Quantization and Algorithm-System Co-design).
 *   - Streaming: the previous chunk's centroids initialise the next chunk's k-means
 *     (notes page, section Algorithm-System Co-design).
 *
 * Conventions for every call:
 *   - All data pointers are DEVICE pointers into memory the caller owns and keeps alive
 *     until the work on `stream` has finished.  The library allocates no device memory and
 *     keeps no mutable global state; scratch space is the caller's `workspace`.  The one
 *     exception is qvg_quantize_static, whose scratch is a fixed area inside the library.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Work
 *     is enqueued asynchronously; a call returns once it is enqueued.  qvg_quantize,
 *     qvg_reassign and qvg_dequantize enqueue only kernels and memsets on `stream`, so a
 *     caller may capture them in a CUDA graph and replay it with the same buffers.
 *   - The kernels are launched with programmatic dependent launch: each one may become
 *     resident before the previous kernel on `stream` has finished, and waits for it
 *     (griddepcontrol.wait) before touching memory, so the order of memory effects is plain
 *     stream order.  Each also lets its dependents launch early.  A kernel the caller
 *     launches next with programmatic serialisation allowed must itself wait
 *     (griddepcontrol.wait) before reading the results; one launched without it needs
 *     nothing.
 *   - Argument errors are detected on the host before anything is enqueued and returned as
 *     QVG_ERR_INVALID_ARG / QVG_ERR_UNSUPPORTED / QVG_ERR_WORKSPACE.  A CUDA error reported
 *     while enqueuing returns QVG_ERR_CUDA; work already enqueued may have run.
 *   - Conditions only the device can see are OR-ed into *dev_status (a device uint32, may
 *     be NULL) as QVG_DEV_* bits; read it after synchronising the stream.  No call aborts
 *     the process or traps the device.
 *   - Pointers must be 16-byte aligned.
 *   - Fault injection, for testing a caller's error handling without faulting a GPU (read
 *     from the environment at every call): QVG_FAULT_INJECT=launch makes every call that
 *     would enqueue device work return QVG_ERR_CUDA after its argument checks, with nothing
 *     enqueued; =alloc does the same for qvg_quantize_static alone (its scratch lookup);
 *     =timeout runs qvg_quantize's tensor-core assignments with their centroid operand
 *     withheld and a 1 ms wait limit (as qvg_selftest_assign_timeout does), so the call
 *     returns QVG_OK, the device status gets QVG_DEV_TIMEOUT and the results are
 *     unspecified; =assign makes qvg_quantize's first tensor-core assignment launch fail
 *     after the kernels before it were enqueued, so the call returns QVG_ERR_CUDA from the
 *     middle of its sequence (nothing after the failed launch is enqueued; the outputs are
 *     unspecified).  Unset, or any other value: no effect.
 *
 * Supported shapes: d = 128; group in {16, 32, 64}; bits in {2, 4}; 1 <= C <= 256 and
 * C <= N when T > 0; 0 <= T <= 8; iters >= 1; N >= 1.
 */
#ifndef QVG_H
#define QVG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QVG_OK = 0,
    QVG_ERR_INVALID_ARG = 1, /* NULL / misaligned pointer, negative or inconsistent size */
    QVG_ERR_UNSUPPORTED = 2, /* a value outside the supported shapes listed above */
    QVG_ERR_WORKSPACE = 3,   /* workspace NULL or smaller than qvg_quantize_workspace_bytes */
    QVG_ERR_CUDA = 4,        /* a CUDA runtime call failed while enqueuing (no device, launch) */
    QVG_ERR_DEVICE = 5,      /* the current device is not an sm_103 (GB300-class) GPU */
    QVG_ERR_SCRATCH_LIMIT = 6 /* qvg_quantize_static: the problem needs more scratch than
                                 QVG_STATIC_SCRATCH_BYTES */
} qvg_status;

/* Bits OR-ed into *dev_status by the device. */
#define QVG_DEV_NONFINITE 0x1u /* X held a NaN or an infinity */
#define QVG_DEV_TIMEOUT 0x2u   /* a pipeline wait in the assignment kernel gave up */
#define QVG_DEV_BAD_INDEX 0x4u /* a stored cluster index was >= C; it was clamped to C-1 */

typedef enum { QVG_F16 = 0, QVG_BF16 = 1, QVG_F32 = 2 } qvg_dtype;

/* Parameters of one qvg_quantize call: n_tensors independent tensors of N tokens each. */
/* Integer grid of the codes.
 *   QVG_QSCHEME_SYMMETRIC: q in [-qmax, qmax], qmax = 2^(bits-1) - 1 (INT2 is ternary);
 *     s = max|r| / qmax; q = r / s_q rounded half to even and clamped; u = q + 2^(bits-1);
 *     x = s_q * (u - 2^(bits-1)).
 *   QVG_QSCHEME_MIDRISE: the 2^bits levels sit at half-integers (4 levels at INT2, the
 *     reading of one critique page of the method); s = max|r| / (2^(bits-1) - 1/2);
 *     u = floor(r / s_q) + 2^(bits-1) clamped to [0, 2^bits - 1] (a value exactly between
 *     two levels takes the upper one); x = s_q * (u - 2^(bits-1) + 1/2).
 * Either way s_q = E4M3(s) and s_q = 0 stores every code as 2^(bits-1). */
typedef enum { QVG_QSCHEME_SYMMETRIC = 0, QVG_QSCHEME_MIDRISE = 1 } qvg_qscheme;

/* Value format of the stored centroids.  The tables stay float arrays; with a 16-bit format
 * every stored value is exactly representable in it, so a consumer may narrow the tables
 * without loss, and residuals, codes and reconstruction all use those rounded values.
 *   QVG_CENTROIDS_F32:  the fp32 mean (the default).
 *   QVG_CENTROIDS_F16:  IEEE binary16; QVG_CENTROIDS_BF16: bfloat16.  The cluster mean, a
 *     cold-start row and a warm-start value are each rounded once to nearest even in the
 *     format.  The mean is carried to about twice fp32's precision, so it rounds as the
 *     exact mean of the stage's inputs does (from the second stage on, the exact residuals
 *     against the stored earlier centroids), save within about 2^-38 of the members' size
 *     of a tie.
 * Quant VideoGen explainer page, compression and metadata overhead: the ratios it prints
 * count centroids in a 16-bit format. */
typedef enum { QVG_CENTROIDS_F32 = 0, QVG_CENTROIDS_F16 = 1, QVG_CENTROIDS_BF16 = 2 }
    qvg_centroid_format;

typedef struct {
    int32_t n_tensors;      /* H >= 1: independent (layer, head, K/V) tensors in this call */
    int32_t d;              /* channels per token; must be 128 */
    int64_t N;              /* tokens per tensor in this call */
    int32_t C;              /* clusters per stage */
    int32_t T;              /* smoothing stages (0 = plain group quantization) */
    int32_t bits;           /* 2 or 4 */
    int32_t group;          /* channels per scale group: 16, 32 or 64 */
    int32_t iters;          /* Lloyd rounds (assign + mean update) per stage */
    int32_t in_dtype;       /* qvg_dtype of X */
    uint64_t seed;          /* cold-start seed */
    int64_t tensor_id_base; /* tensor h of this call uses id tensor_id_base + h for seeding */
    int64_t x_stride;       /* elements between consecutive tensors of X (0 = N*d) */
    int64_t token_offset;   /* first token slot written in codes / scales / pi */
    int64_t token_capacity; /* token slots per tensor in codes / scales / pi (0 = N) */
    int32_t table_index;    /* centroid-table slot written by this call */
    int32_t n_tables;       /* centroid-table slots per tensor (0 = 1) */
    int64_t warm_stride;    /* floats between consecutive tensors of warm_centroids
                               (0 = T*C*d) */
    int32_t qscheme;        /* qvg_qscheme of the codes (zero-initialised = symmetric) */
    int32_t centroid_format; /* qvg_centroid_format of the stored centroids (0 = fp32) */
} qvg_quant_params;

/* The compressed cache.  Layouts (all row-major, caller-owned device memory):
 *   codes     uint8 [H][token_capacity][d*bits/8]  channel k of a token sits at bits
 *             (k*bits) mod 8 of byte (k*bits)/8 of its row; stored code u = q + 2^(bits-1)
 *   scales    uint8 [H][token_capacity][d/group]   FP8 E4M3 bit patterns
 *   pi        uint8 [H][T][token_capacity]         cluster index per stage and token
 *   centroids float [H][n_tables][T][C][d]         one table per chunk of tokens
 * For T = 0, pi and centroids are not touched and may be NULL. */
typedef struct {
    uint8_t *codes;
    uint8_t *scales;
    uint8_t *pi;
    float *centroids;
} qvg_buffers;

/* Bytes of device scratch qvg_quantize needs for these parameters (0 if they are invalid).
 * Depends only on n_tensors, N, C, T. */
size_t qvg_quantize_workspace_bytes(const qvg_quant_params *params);

/* Compress X: T smoothing stages of `iters` Lloyd rounds each, then group quantization of
 * the last residual.  Writes codes/scales for tokens [token_offset, token_offset + N),
 * pi^(1..T) for the same slots, and C^(1..T) into table slot table_index.
 *   X               [H][N][d] of in_dtype, tensor h at X + h*x_stride elements
 *   warm_centroids  NULL for a cold start (seeded distinct rows of R^(t-1) as the initial
 *                   centroids of stage t), or fp32 [H][T][C][d] (tensor stride warm_stride)
 *                   used as stage t's initial centroids -- the streaming warm start.  It
 *                   may point into out->centroids (another table slot than table_index).
 *   workspace       >= qvg_quantize_workspace_bytes(params) bytes, 256-byte aligned; its
 *                   contents on entry do not matter.  Once the call's work has finished,
 *                   its first two uint32 words count, over all stages and Lloyd rounds, the
 *                   token rows whose nearest centroid the tensor-core scores could not
 *                   settle and the candidate clusters re-scored exactly for them.
 * Calls that share a workspace must be ordered on one stream. */
qvg_status qvg_quantize(const qvg_quant_params *params, const void *X,
                        const float *warm_centroids, const qvg_buffers *out, void *workspace,
                        size_t workspace_bytes, uint32_t *dev_status, void *stream);

/* Size of the fixed scratch area behind qvg_quantize_static: 64 MiB per device.  The area is
 * part of libqvg's device code, so it is reserved on every device (in every CUDA context)
 * where that code is loaded -- whichever entry points the process calls, qvg_quantize,
 * qvg_dequantize and qvg_attention included.  A caller sizing a KV pool to the last
 * megabyte should count it. */
#define QVG_STATIC_SCRATCH_BYTES ((size_t)64 << 20)

/* qvg_quantize without a workspace argument, for callers that cannot allocate.
 *
 * The paper has no counterpart to this call: it is a convenience of this library.  It
 * runs the same kernels as qvg_quantize and gives the same results, but takes its scratch
 * from one area of QVG_STATIC_SCRATCH_BYTES compiled into the library (a separate copy on
 * each device) instead of from the caller, and allocates nothing itself: no cudaMalloc or
 * cudaFree, no allocating library, no host heap.
 *
 * Who needs it: a caller that may not or cannot allocate device memory at the moment it
 * compresses -- a server that has handed all free memory to its KV pool or to a caching
 * allocator, a latency-bound loop in which cudaMalloc / cudaFree (which can synchronise
 * the device) would stall the other streams, or a plain C host with no allocator of its
 * own.
 *
 * Limit: qvg_quantize_workspace_bytes(params) must not exceed QVG_STATIC_SCRATCH_BYTES;
 * otherwise the call returns QVG_ERR_SCRATCH_LIMIT before touching the device.  The
 * scratch is about 450 bytes per token row plus about 630 KB per tensor, whatever T: one
 * tensor of up to about 148 000 tokens fits, 24 tensors of up to about 4 800 each (116 000
 * rows), 100 tensors of up to about 250 each.
 *
 * First call in a context: the area's device address belongs to the CUDA context whose
 * copy of the library's device code holds it, so the first call made while a given context
 * is current (a device's primary context, or one the caller created and made current) looks
 * it up once (cudaGetSymbolAddress, which can load the library's device code in that
 * context); if that fails the call returns QVG_ERR_CUDA.  Make this first call before any
 * stream capture begins in that context.  Later calls in the same context reuse the
 * address.  After cudaDeviceReset, or once a context is destroyed, the address kept for it
 * is stale: do not call this function again in that process.
 *
 * Contents on entry do not matter: everything the path needs to start at zero is cleared
 * by the call itself, on `stream`, before it is used.
 *
 * Races: all calls on one device share the one area.  Two calls whose device work can
 * overlap -- on different streams with no event ordering them, e.g. from different host
 * threads -- overwrite each other's scratch and both results are wrong.  Issue them on
 * one stream, or order them with events.
 *
 * Arguments other than the workspace, layouts and the other errors are those of
 * qvg_quantize. */
qvg_status qvg_quantize_static(const qvg_quant_params *params, const void *X,
                               const float *warm_centroids, const qvg_buffers *out,
                               uint32_t *dev_status, void *stream);

/* Assign every token's stage-T residual R^(T-1) to its nearest centroid of C^(T) as stored
 * in out->centroids (table slot table_index), writing pi^(T).  This is one assignment step
 * of the Lloyd iteration (notes page, section Semantic-Aware Smoothing, step 1), run on the
 * state a preceding qvg_quantize call with the same params, X, out and workspace left
 * behind: the residual planes of stage T stay in the workspace.  It lets the tensor-core
 * assignment be timed and checked on its own.  Requires T >= 1.  The codes and scales
 * are not updated. */
qvg_status qvg_reassign(const qvg_quant_params *params, const void *X, const qvg_buffers *out,
                        void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                        void *stream);

/* The steps of qvg_reassign, for timing them one at a time: */
#define QVG_STEP_PLANES 1 /* the centroids' GEMM operands (fp16 plane, offsets, norms) */
#define QVG_STEP_GEMM 2   /* the tensor-core GEMM with its fused argmax epilogue: pi^(T)
                             for every row with one candidate, the lowest candidate and a
                             re-scoring request for the others */
#define QVG_STEP_REFINE 4 /* the exact re-scoring of the requested rows */
/* qvg_reassign with only the steps in the `steps` mask.  Each step reads what the earlier
 * ones wrote in the workspace: run them in order, on one stream (the GEMM after the planes
 * of the same centroids, the re-scoring after the GEMM).  A re-scoring step whose queue no
 * GEMM step wrote (a fresh workspace) reads no request outside the queue's capacity: it
 * skips what is out of range and ORs QVG_DEV_BAD_INDEX into *dev_status.
 * QVG_ERR_INVALID_ARG for other bits; otherwise as qvg_reassign. */
qvg_status qvg_reassign_steps(const qvg_quant_params *params, const void *X,
                              const qvg_buffers *out, void *workspace, size_t workspace_bytes,
                              int32_t steps, uint32_t *dev_status, void *stream);

/* Self-test of the assignment kernel's failure handling; no step of the method.  It runs the
 * tensor-core assignment of qvg_reassign once with the load of the centroid operand withheld
 * and a wait limit of one millisecond (2 s in normal calls), so that the kernel's first wait
 * on that operand never completes: the wait gives up, the kernel ORs QVG_DEV_TIMEOUT into
 * *dev_status, waits for the copies it did issue, frees its tensor memory and returns.  The
 * device stays usable, and later calls run normally.  Arguments as for qvg_reassign; pi^(T)
 * is left unspecified.  The device is never faulted or trapped. */
qvg_status qvg_selftest_assign_timeout(const qvg_quant_params *params, const void *X,
                                       const qvg_buffers *out, void *workspace,
                                       size_t workspace_bytes, uint32_t *dev_status,
                                       void *stream);

/* Parameters of one qvg_dequantize call. */
typedef struct {
    int32_t n_tensors;      /* H */
    int32_t d;              /* 128 */
    int64_t N;              /* tokens to reconstruct per tensor, slots [0, N) */
    int32_t C, T, bits, group;
    int32_t out_dtype;      /* qvg_dtype of X_hat */
    int64_t chunk_len;      /* tokens per centroid table: slot i uses table i / chunk_len
                               (0 = N, one table) */
    int64_t token_capacity; /* token slots per tensor in codes / scales / pi (0 = N) */
    int32_t n_tables;       /* centroid-table slots per tensor (0 = 1) */
    int64_t out_stride;     /* elements between consecutive tensors of X_hat (0 = N*d) */
    int32_t qscheme;        /* qvg_qscheme the codes were written with */
} qvg_dequant_params;

/* Reconstruct X_hat[h][i] = x(u) + C^(T)[pi^(T)_i] + ... + C^(1)[pi^(1)_i], x(u) the level
 * of the code's scheme, added in that order (stage T first) in fp32 registers, rounded
 * once to out_dtype. */
qvg_status qvg_dequantize(const qvg_dequant_params *params, const qvg_buffers *in,
                          void *X_hat, uint32_t *dev_status, void *stream);

/* Parameters of one qvg_attention call. */
typedef struct {
    int32_t n_heads;        /* H: 1 .. 65535 */
    int32_t d;              /* 128 */
    int32_t M;              /* queries per head: 1 .. 16 */
    int64_t N;              /* keys per head: cache slots [0, N) */
    int32_t C, T, bits, group, qscheme;  /* of both caches, as they were quantized */
    int64_t chunk_len;      /* tokens per centroid table (0 = N), as in qvg_dequant_params */
    int64_t token_capacity; /* token slots per tensor of both caches (0 = N) */
    int32_t n_tables;       /* centroid-table slots per tensor (0 = 1) */
    int32_t q_dtype;        /* qvg_dtype of Q */
    int32_t out_dtype;      /* qvg_dtype of O */
    float scale;            /* multiplies q.k before the softmax, e.g. 1/sqrt(d); finite */
    int64_t k_first;        /* head h reads key tensor k_first + h * tensor_step of k_cache */
    int64_t v_first;        /* and value tensor v_first + h * tensor_step of v_cache */
    int64_t tensor_step;    /* >= 0; keys and values interleaved in one cache: pass it as
                               both caches with k_first 0, v_first 1, tensor_step 2 */
} qvg_attention_params;

/* Workspace bytes qvg_attention needs for these parameters (0 if they are invalid). */
size_t qvg_attention_workspace_bytes(const qvg_attention_params *params);

/* Softmax attention read straight from the compressed cache.  For head h and query m:
 *   O[h][m] = sum_j p_j v_j,  p = softmax over j < N of (scale * Q[h][m] . k_j),
 * where k_j and v_j are token j of the head's key and value tensors rebuilt exactly as
 * qvg_dequantize writes them in fp32.  The rebuilt rows stay in registers and shared
 * memory; nothing of size N x d is written (the notes page's fused reconstruction,
 * section Algorithm-System Co-design, feeding attention on the fly).
 * Layouts: Q [H][M][d] of q_dtype, O [H][M][d] of out_dtype, both contiguous and 16-byte
 * aligned; the caches as qvg_buffers describes.  Scores, softmax and sums are fp32, the
 * output rounded once to out_dtype.  Tensor indices are not checked against the caches'
 * sizes: the caller guarantees them.  A cluster index >= C is clamped and reported as
 * QVG_DEV_BAD_INDEX. */
qvg_status qvg_attention(const qvg_attention_params *params, const void *Q,
                         const qvg_buffers *k_cache, const qvg_buffers *v_cache, void *O,
                         void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                         void *stream);

/* Static description of a status code. */
const char *qvg_status_string(qvg_status status);

/* Library version, (major << 16) | minor.
 *   1.0  quantize, reassign, dequantize, the static-scratch quantize.
 *   1.1  qvg_quant_params.qscheme and .centroid_format, qvg_dequant_params.qscheme (both
 *        structs grew: rebuild callers), qvg_attention. */
uint32_t qvg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QVG_H */
