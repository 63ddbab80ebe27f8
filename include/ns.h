/*
 * ns.h -- C ABI of libns, batched quintic Newton-Schulz orthogonalization on
 * one GB300 (sm_103a).
 *
 * The operation. For every matrix X (M x N, row-major) of a batch:
 *     X <- X / (||X||_F + eps)
 *     work on W = X^T when M > N (W is m x n, m = min(M,N), n = max(M,N))
 *     repeat `steps` times:  A = W W^T;  B = b*A + c*A*A;  W = a*W + B*W
 *     write W back into X (transposed back when M > N).
 * The three pages this library follows -- "Fix megabatch_orthogonalize_async
 * hang on empty FSDP2 shards" (microsoft/dion), "Balance LayerWise optimizer
 * shards by Newton-Schulz cost, not parameter size" (Megatron-LM) and the
 * xtuner Muon remainder-strategy PR -- run this iteration on stacks of
 * same-shape 2-D momentum matrices but never print it; the form and the
 * default coefficients (a,b,c) = (3.4445, -4.7750, 2.0315), 5 steps and
 * eps = 1e-7 are Muon's standard quintic Newton-Schulz. The megabatch layout
 * (a stack of same-shape matrices, per-rank zero padding) is the first page's
 * "Concrete repro" and "Fix" sections; its "Fix" section also states the
 * invariant that zero rows stay zero, which lets the library skip padded rows
 * and columns instead of computing them. The cost model is the second page's
 * "Changes" item 1.
 *
 * Conventions for every call:
 *  - Pointers named X / X_host are caller-owned. Device pointers must be on
 *    the current CUDA device. Nothing is retained after the call returns,
 *    except the library's internal workspace cache (see ns_release_workspace).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). All device work is stream-ordered on it; calls do not
 *    synchronise unless stated.
 *  - Return value: NS_OK (0) or a negative NS_E* code. Arguments are
 *    validated before anything is launched; on a validation error nothing
 *    runs and the matrices are untouched. No C++ exception crosses the ABI.
 *  - CUDA graphs: once ns_orthogonalize_batched (or _sched) has run with the
 *    same matrices, shapes, steps, coefficients and stream, a repeat call
 *    allocates nothing and uploads nothing, so it may be captured into a
 *    graph on that stream and replayed. The library keeps the descriptor
 *    tables of the last 8 distinct batches per stream on the device, so a
 *    caller alternating between a few batches (e.g. remainder batches) also
 *    uploads nothing after the first call of each.
 */
#ifndef NS_H_
#define NS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types of X */
#define NS_F32 0  /* float32 in, float32 out, fp32-accurate arithmetic throughout (see ns_set_f32_gemm) */
#define NS_BF16 1 /* bfloat16 in/out; bf16 tensor-core operands, fp32 accumulation */

/* status codes */
#define NS_OK 0
#define NS_EINVAL (-1)   /* null pointer, negative dims/count/steps, bad dtype, a side above
                            2^30 - 1 or a matrix above 2^40 elements, overlapping matrices */
#define NS_EALIGN (-2)   /* a matrix pointer is not aligned to its element size */
#define NS_ENOMEM (-3)   /* workspace allocation failed / caller workspace too small */
#define NS_ECUDA (-4)    /* a CUDA runtime or driver call failed */
#define NS_ETIMEOUT (-5) /* a bounded device-side wait gave up (reported by ns_get_status) */
#define NS_ENODEV (-6)   /* no CUDA driver or device, or the current device is not sm_100-family */
#define NS_ETOOBIG (-7)  /* batch needs more scratch than ns_orthogonalize_batched_noalloc holds */
#define NS_EBOUNDS (-8)  /* a debug build's bounds check caught a store (reported by ns_get_status) */

/*
 * ns_orthogonalize_batched -- Newton-Schulz of `count` matrices, in place.
 *   X       host array of `count` device pointers; X[i] points at a
 *           contiguous row-major matrix of shapes[2i] x shapes[2i+1]
 *           elements of `dtype`. Matrices may differ in shape; a zero
 *           dimension makes that matrix a no-op. Matrices must not overlap
 *           (checked: overlapping ranges give NS_EINVAL).
 *   shapes  host array of 2*count int64 (M, N) pairs, read before return.
 *   count   number of matrices (0 is valid and does nothing).
 *   steps   number of iterations (>= 0; 0 = normalisation only).
 *   coeffs  NULL for (3.4445, -4.7750, 2.0315), else a host array of three
 *           floats (a, b, c) used by every step.
 *   dtype   NS_F32 or NS_BF16.
 *   stream  cudaStream_t.
 * eps is 1e-7. Work is scheduled largest ns_cost first. Scratch memory comes
 * from an internal per-(device, stream) workspace that grows on demand with
 * stream-ordered allocation.
 */
int ns_orthogonalize_batched(void *const *X, const int64_t *shapes, int count, int steps,
                             const float *coeffs, int dtype, void *stream);

/*
 * ns_orthogonalize_batched_ex -- as above, with an explicit eps and an
 * explicit caller-owned device workspace of at least
 * ns_workspace_bytes(shapes, count, dtype) bytes (256-byte aligned). The
 * workspace must not be used by anything else until the stream has passed
 * this call's work. Returns NS_ENOMEM if it is too small.
 */
int ns_orthogonalize_batched_ex(void *const *X, const int64_t *shapes, int count, int steps,
                                const float *coeffs, float eps, int dtype, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * ns_orthogonalize_batched_sched -- as ns_orthogonalize_batched, but step s
 * uses its own coefficients: coeff_table is a host array of steps x 3 floats,
 * row s = (a, b, c) of step s, read before return; 1 <= steps <= 32 (0 steps
 * is normalisation only and reads no table). The pages print no schedule;
 * this serves coefficient schedules that change from step to step.
 * Returns NS_EINVAL for a NULL table or more than 32 steps.
 */
int ns_orthogonalize_batched_sched(void *const *X, const int64_t *shapes, int count, int steps,
                                   const float *coeff_table, int dtype, void *stream);

/* Device workspace bytes the _ex call needs for this batch (0 on bad input). */
size_t ns_workspace_bytes(const int64_t *shapes, int count, int dtype);

/*
 * ns_orthogonalize_batched_host -- the same operation on HOST matrices:
 * copies each X_host[i] to the device, runs the method, copies the results
 * back into X_host[i] and returns once they are there. The batch is split into
 * up to 8 contiguous groups of about equal bytes, each of at least 32 MiB
 * (a smaller batch is one group); the copies in of group g+1,
 * the Newton-Schulz of group g and the copies out of group g-1 overlap on
 * library-owned streams ordered by events (even groups compute on `stream`,
 * odd groups on a second library stream, so one group's last partial wave of
 * tiles overlaps the next group's first; under NS_SCHED_SINGLE every group
 * computes on `stream`). Host buffers may be
 * pageable or pinned (only pinned buffers let the copies overlap). Device
 * copies and workspaces are part of the internal per-(device, stream) cache.
 */
int ns_orthogonalize_batched_host(void *const *X_host, const int64_t *shapes, int count,
                                  int steps, const float *coeffs, int dtype, void *stream);

/*
 * ns_orthogonalize_batched_noalloc -- the same operation as
 * ns_orthogonalize_batched (same arguments, eps = 1e-7) for callers that
 * cannot allocate device memory: processes whose framework allocator has
 * already reserved nearly all of HBM, optimizer steps that cannot absorb an
 * allocator's synchronisation, runtimes that forbid allocation after
 * start-up. It calls no cudaMalloc, cudaFree or other allocating routine; its
 * scratch is one fixed 256 MiB device array inside the library, reserved on
 * every device that loads the library until the process exits.
 *   - A batch whose ns_workspace_bytes exceeds 256 MiB is rejected with
 *     NS_ETOOBIG before anything runs (e.g. one 4096 x 4096 bf16 matrix
 *     fits; one 8192 x 6144 does not).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call shares the one array and leaves its contents behind; each
 *     call clears what must start at zero itself. Calls that overlap on the
 *     GPU (other streams, other host threads) race on the array: serialise
 *     them.
 * The pages have no counterpart of this entry point; it exists for callers
 * of this library that cannot allocate.
 */
int ns_orthogonalize_batched_noalloc(void *const *X, const int64_t *shapes, int count, int steps,
                                     const float *coeffs, int dtype, void *stream);

/*
 * ns_muon_update_batched -- one optimizer step around the orthogonalization,
 * for `count` matrices: the momentum step, Newton-Schulz and a scaled write
 * of the result. The dion page's "Summary" names Muon, NorMuon and Dion2 as
 * the optimizers that run the megabatch Newton-Schulz on momentum matrices;
 * the pages do not print their updates, so every constant here is a
 * parameter. For each matrix i, with every buffer M x N row-major of `dtype`
 * on the current device:
 *     Mom[i] <- mu * Mom[i] + G[i]                       (stored in Mom[i])
 *     X      <- G[i] + mu * Mom[i]   if nesterov, else Mom[i]
 *     Out[i] <- scale * NS(X)         (NS as ns_orthogonalize_batched, eps 1e-7)
 *   G       host array of count device pointers: gradients, read only
 *   Mom     host array of count device pointers: momentum buffers, updated
 *   Out     host array of count device pointers: where the update is written;
 *           Out[i] may be G[i] itself (the gradient buffer is overwritten)
 *   shapes, count, steps, coeffs, dtype, stream: as ns_orthogonalize_batched
 *   mu, scale  finite floats; nesterov 0 or 1.
 * One element-wise kernel does the momentum step and writes X into Out (bf16:
 * Mom and X rounded to nearest even, arithmetic in fp32); the Newton-Schulz
 * call then works on Out in place, and `scale` is applied inside its last
 * step before the final rounding. Buffers of the batch must not overlap,
 * except Out[i] == G[i] (NS_EINVAL otherwise, before anything runs). Other
 * returns as ns_orthogonalize_batched.
 */
int ns_muon_update_batched(void *const *G, void *const *Mom, void *const *Out, const int64_t *shapes,
                           int count, int steps, const float *coeffs, float mu, int nesterov,
                           float scale, int dtype, void *stream);

/*
 * ns_cost -- Newton-Schulz cost of an M x N matrix, max(M,N) * min(M,N)^2
 * (second page, "Changes" item 1: the dominant term of the orthogonalization).
 * Returns -1 if M or N is negative.
 */
int64_t ns_cost(int64_t M, int64_t N);

/*
 * ns_plan_shards -- host-only planner that assigns whole matrices to
 * `nshards` shards (GPUs, streams or ranks) so that Newton-Schulz work is
 * balanced. It follows the second page's "Changes" items 1-3: matrices are
 * taken largest first and each goes to the least-loaded shard; with
 * order = NS_PLAN_COST "size" and "load" are the ns_cost of the matrices,
 * with order = NS_PLAN_NUMEL they are element counts (the numel heuristic that
 * page replaces, kept for comparison).
 *   shapes     host array of 2*count (M, N) of the matrices Newton-Schulz runs
 *              on; a 1-D parameter of n elements is passed as (1, n), whose
 *              cost equals its numel.
 *   numels     NULL (element counts are M*N), or count element counts a shard
 *              stores, when they differ from the shape Newton-Schulz sees
 *              (a tensor-parallel shard is stored locally but orthogonalised
 *              after an all-gather: the second page's GTP case).
 *   numel_eps  per-call numel cap: when >= 0, a shard is a candidate for a
 *              matrix only while the elements placed on it by this call plus
 *              the matrix's stay within ceil((1 + numel_eps) * total / nshards);
 *              if no shard qualifies the matrix goes to the shard with the
 *              fewest elements placed by this call (least-numel fallback).
 *              The page uses 0.3. A negative value disables the cap.
 *   loads      NULL, or nshards int64 loads that persist across calls (one
 *              call per bucket); read as the starting loads and updated.
 *   assign     out: count shard indices.
 * Ties go to the shard with fewer elements placed by this call, then to the
 * lower index. Returns NS_OK or NS_EINVAL. Touches no GPU.
 */
#define NS_PLAN_COST 0
#define NS_PLAN_NUMEL 1
int ns_plan_shards(const int64_t *shapes, const int64_t *numels, int count, int nshards, double numel_eps,
                   int order, int64_t *loads, int *assign);

/*
 * ns_get_status -- synchronise `stream`, then return and clear the device
 * status word of the current device: NS_OK, or NS_ETIMEOUT if a kernel's
 * bounded wait gave up (its outputs are then unspecified), NS_EBOUNDS if a
 * debug build's bounds check caught a store outside its buffer (the store was
 * not made; outputs unspecified), or NS_ECUDA if the synchronisation itself
 * failed or a CTA pair's tensor-memory allocations disagreed.
 */
int ns_get_status(void *stream);

/*
 * Debug builds. Compiled with NS_DEBUG_BOUNDS (e.g. NS_BUILD_TAG=debug
 * NS_EXTRA_NVCC_FLAGS=-DNS_DEBUG_BOUNDS with the package's build script),
 * every store of the library's kernels is checked against the buffer it
 * belongs to; a store outside it is not made and the device status word
 * records NS_EBOUNDS. Release builds compile the checks away.
 * ns_selftest_bounds_check exercises the mechanism without touching memory:
 * one thread asks whether a store one past the end of a 4-byte buffer is in
 * bounds. Synchronises `stream`. Returns NS_OK in a debug build (the status
 * word then reads NS_EBOUNDS), NS_EINVAL in a release build.
 */
int ns_selftest_bounds_check(void *stream);

/* ns_strerror -- static description of a status code. */
const char *ns_strerror(int code);

/*
 * ns_release_workspace -- synchronise the device and free the internal
 * workspace cache of the current device. Returns NS_OK or NS_ECUDA.
 */
int ns_release_workspace(void);

/* ns_num_kernel_launches -- kernels this library launched on this process
 * since load (for launch accounting in benchmarks). */
int64_t ns_num_kernel_launches(void);

/*
 * ns_set_workspace_limit -- cap, in bytes, on any one workspace the library's
 * internal cache allocates (per device, stream and use); 0 removes the cap
 * (the default). A call whose batch needs a larger workspace than the cap and
 * than the cache already holds returns NS_ENOMEM before anything is allocated
 * or launched, exactly as when the device allocation itself fails. Calls with
 * a caller workspace (_ex) and ns_orthogonalize_batched_noalloc are not
 * affected. Process-wide; returns NS_OK.
 */
int ns_set_workspace_limit(size_t bytes);

/* ns_set_nvtx -- NVTX ranges for profilers' timelines: with enable != 0 every
 * call is bracketed by a range "ns call" and every kernel launch by a range
 * naming its class ("ns gram", "ns apply", ...). Off by default, unless the
 * environment variable NS_NVTX=1 was set when the library first looked.
 * Process-wide; returns NS_OK. */
int ns_set_nvtx(int enable);

/* ns_num_workspace_allocations -- device allocations (workspace cache growth)
 * this library has requested in this process since load; calls that reuse the
 * cached workspace, calls given a caller workspace and
 * ns_orthogonalize_batched_noalloc leave it unchanged. */
int64_t ns_num_workspace_allocations(void);

/*
 * Per-kernel timing for measurement tools. While enabled, every kernel
 * launch of later calls is bracketed by a pair of CUDA events recorded on the
 * caller's stream (a few microseconds of overhead per launch).
 * ns_set_kernel_timing(1) enables and clears the record, (0) disables it.
 * ns_get_kernel_times synchronises on the recorded events and writes, for the
 * kernel classes 0 norm pass (the one read of the caller's matrices: bf16 tile
 * sums of squares and extents, plus a copy where the first step cannot read
 * them in place; fp32 the sums and extents), 1 norm finish (bf16: the
 * per-matrix scale from the tile sums), 2 gram, 3 square, 4 apply,
 * 5 resident, 6 gemm (the tensor-core kernel running every step and phase of
 * a call in one launch), 7 prep (fp32: the normalising copy, or its bf16
 * slices on the tensor cores), 8 momentum
 * (ns_muon_update_batched's element-wise step), the total milliseconds into
 * ms[k] and the launch count into launches[k] for k < n (n <= 9). Returns
 * NS_OK or NS_EINVAL / NS_ECUDA.
 */
int ns_set_kernel_timing(int enable);
int ns_get_kernel_times(double *ms, int64_t *launches, int n);

/*
 * ns_set_gemm_schedule -- how later calls launch the bf16 tensor-core GEMMs
 * (process-wide):
 *   NS_SCHED_PHASE   one persistent launch per step and phase (default);
 *   NS_SCHED_SINGLE  one persistent, cooperative launch per call running every
 *                    step and phase; an item waits, on a per-matrix completion
 *                    counter, until the earlier phases of its matrix are done,
 *                    so phases of different matrices overlap. On GB300 it
 *                    measured 0-3% slower than NS_SCHED_PHASE on the
 *                    8 x 8192x6144, 76 x 2048x6144 and mixed 120-matrix
 *                    batches, so it is not the default.
 * Results are the same in both. The fp32 tensor-core path (ns_set_f32_gemm)
 * always uses NS_SCHED_PHASE. Returns NS_OK or NS_EINVAL.
 */
#define NS_SCHED_PHASE 0
#define NS_SCHED_SINGLE 1
int ns_set_gemm_schedule(int mode);

/*
 * ns_set_f32_gemm -- how later calls compute the GEMMs of large fp32 matrices
 * (those not on the shared-memory resident path), process-wide:
 *   NS_F32_TENSOR  tcgen05 tensor cores (default): every fp32 tensor (the
 *                  iterate, A and B) is held as three bf16 slices
 *                  x = h + m + l, h = bf16(x), m = bf16(x - h),
 *                  l = bf16(x - h - m) (x to 2^-27 relative), and each
 *                  product is the fp32-accumulated sum of the six slice
 *                  products of weight 2^-18 or more, smallest first:
 *                  (h,l), (l,h), (m,m), (h,m), (m,h), (h,h). The dropped
 *                  products weigh 2^-27 or less. The tensor cores' fp32
 *                  accumulation loses up to about a unit in the last place
 *                  per instruction, so the error grows with the contraction
 *                  length: measured 2.2e-5 relative after 5 steps for
 *                  2048 x 6144 (fp32 CUDA cores: 5.0e-6). A call whose
 *                  largest fp32 matrix has max(M, N) > 16384 therefore runs
 *                  on the CUDA cores, keeping every result within fp32's
 *                  1e-4 bar.
 *   NS_F32_SIMT    CUDA-core fp32 FMA GEMMs.
 * Both follow the same definition (the quintic iteration in fp32 between
 * phases); their rounding differs, so their results differ in the last
 * bits. The workspace size (ns_workspace_bytes) depends on the mode in effect
 * when it is computed. Returns NS_OK or NS_EINVAL.
 */
#define NS_F32_TENSOR 0
#define NS_F32_SIMT 1
int ns_set_f32_gemm(int mode);

/*
 * ns_selftest_wait_timeout -- failure-detection self-test. Launches one CTA
 * that waits, with the library's bounded wait and a limit of `limit_us`
 * microseconds (1 .. 10^7), on an mbarrier nothing will ever arrive on. The
 * wait gives up, records NS_ETIMEOUT in the device status word (read it with
 * ns_get_status) and the kernel exits normally: no fault, no trap, no hang,
 * and the CUDA context stays usable. Synchronises `stream`. Returns NS_OK if
 * the wait gave up as designed, NS_EINVAL for a bad limit, NS_ECUDA otherwise.
 */
int ns_selftest_wait_timeout(int limit_us, void *stream);

/*
 * ns_selftest_dependency_timeout -- failure-detection self-test of the
 * tensor-core kernel's dependency waits (the per-matrix completion counters of
 * the NS_SCHED_SINGLE schedule). Runs a two-step call on two 512 x 768 bf16
 * matrices (allocated, filled and released by the call itself) in one
 * cooperative launch whose completion signals are held back, with every
 * bounded wait limited to `limit_us` microseconds (1 .. 10^7): the items that
 * depend on earlier phases wait on counters that never advance, give up,
 * record NS_ETIMEOUT in the device status word (read it with ns_get_status),
 * drain their in-flight copies and MMAs, free their TMEM and exit. No fault,
 * no trap, no hang; the context stays usable. Synchronises `stream`. Returns
 * NS_OK if the waits gave up as designed, NS_EINVAL for a bad limit, NS_ENOMEM
 * if the buffers could not be allocated, NS_ECUDA otherwise.
 */
int ns_selftest_dependency_timeout(int limit_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* NS_H_ */
