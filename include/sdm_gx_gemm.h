/*
 * sdm_gx_gemm.h -- C ABI of the GB300 (sm_103a) gx_gemm library: the deterministic FP32 per-step d_u update of a
 * chunked backward pass.
 *
 * The operation (sparse_delta_memory/cuda/gx_gemm_cuda.py, module docstring formula; gx_gemm_kernel's chain and
 * epilogue): for a step ti and every chunk n = ti*P + p (0 <= p < P), row i < C and column c < hd,
 *
 *     acc = +0;   acc = fmaf(x[n, j, i], d_dv[n, j, c], acc)   for j = 0, 1, .., C-1   (one rounding per fma)
 *     d_u[n, i, c] = d_u[n, i, c] + acc                                               (one more rounding)
 *
 * i.e. d_u(ti) += x(ti)^T d_dv(ti) with a FIXED reduction order. Every output element is produced by one GPU thread
 * with exactly that chain on the FP32 CUDA cores (no tensor cores, no flush-to-zero), so the bits do not depend on the
 * tiling, the launch geometry, the stream or the run, and equal a CPU evaluation of the same chain.
 *
 * Layout (contiguous form): x is [N, C, C] float32 with x[n, j, i] at x[(n*C + j)*C + i]; d_dv is N*C*hd float32 read
 * as [N, C, hd] with d_dv[n, j, c] at d_dv[(n*C + j)*hd + c]; d_u is [N, C, hd] float32, updated in place. The
 * strided entry points take element strides instead (innermost stride always 1).
 *
 * Kernels (the same bits on every one): strides that are multiples of 4 floats (16 bytes) take the TMA-fed path 1:
 * its aligned configurations when every base pointer is 16-byte aligned, its offset configurations when some base is
 * 4, 8 or 12 bytes past a 16-byte boundary (tensor maps encoded from the base rounded down, tiles read from the
 * offset on). Other layouts (rows of a stride that is not a multiple of 4 floats) take the generic path 0, as does
 * SDM_GX_FLAG_GENERIC.
 *
 * Ownership: the caller owns every device buffer and stream. The library never allocates or frees device memory.
 * A plan holds raw device pointers and host memory only; it is valid while the buffers it names live. A plan created
 * with a workspace (sdm_gx_gemm_plan_create_ws) uses that caller-owned device buffer as scratch for as long as it lives.
 *
 * Errors: every entry point returns 0 (SDM_GX_OK) or a negative sdm_gx_status. All argument checks run before any
 * CUDA call. An empty step (nothing to compute) returns 0 without a launch. Calls are asynchronous and
 * stream-ordered: a kernel-side failure (a bounded device wait that gave up) is reported later by
 * sdm_gx_device_error().
 *
 * Programmatic dependent launch (pdl != 0): the step kernel may start while the previous kernel on the stream is
 * still running. Before its grid-dependency wait it reads only x and d_u(ti) (and prefetches d_dv into L2, which has
 * no visible effect); d_dv is read, and d_u written, only after the wait. The caller vouches that the previous
 * kernel writes neither x nor d_u(ti) (the page's step(ti, pdl=True) contract in make_step).
 *
 * Thread safety: entry points may be called from several host threads; per-device attributes are set once under a
 * lock. A plan may be launched from several threads; it is not modified by launches.
 */
#ifndef SDM_GX_GEMM_H_
#define SDM_GX_GEMM_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SDM_GX_ABI_VERSION 1

#if defined(__GNUC__)
#define SDM_GX_API __attribute__((visibility("default")))
#else
#define SDM_GX_API
#endif

typedef enum sdm_gx_status {
    SDM_GX_OK = 0,
    SDM_GX_E_NULL = -1,          /* a required pointer argument is NULL                                          */
    SDM_GX_E_SHAPE = -2,         /* C outside [1, 256] or hd outside [1, 2^20)                                   */
    SDM_GX_E_RANGE = -3,         /* not 1 <= P <= N < 2^31, or not 0 <= ti < N / P (checked by division)        */
    SDM_GX_E_ALIGN = -4,         /* an operand pointer is not 4-byte aligned (a plan workspace: 256-byte)        */
    SDM_GX_E_OVERLAP = -5,       /* d_u overlaps x or d_dv (the in-place update needs disjoint operands), or a
                                    plan workspace overlaps an operand                                          */
    SDM_GX_E_STRIDE = -6,        /* strides do not describe a non-overlapping [N, rows, cols] layout, or overflow */
    SDM_GX_E_GRID = -7,          /* more than 2^31 - 1 tiles in one step                                         */
    SDM_GX_E_SMEM = -8,          /* the kernel's shared memory exceeds the device's opt-in limit                 */
    SDM_GX_E_DEVICE = -9,        /* an operand is not device memory of the current device                        */
    SDM_GX_E_PLAN = -10,         /* plan pointer NULL or corrupt (bad magic / size)                              */
    SDM_GX_E_PLAN_TI = -11,      /* ti outside [0, ti_max] of the plan                                           */
    SDM_GX_E_PLAN_DEVICE = -12,  /* the current device is not the plan's device                                  */
    SDM_GX_E_FLAGS = -13,        /* unknown flag bits or an invalid forced configuration                         */
    SDM_GX_E_CUDA = -14,         /* a CUDA runtime call failed: sdm_gx_last_cuda_error() has its cudaError_t     */
    SDM_GX_E_DEVICE_FAULT = -15, /* the device error word is set: a bounded wait inside a kernel gave up          */
    SDM_GX_E_UNSUPPORTED = -16,  /* the current device is not compute capability 10.3 (this build is sm_103a only),
                                    or the plan's kernel cannot do the request (sdm_gx_gemm_plan_set_trace)        */
    SDM_GX_E_ALLOC = -17,        /* host memory for a plan could not be allocated                                */
    SDM_GX_E_CAPTURE = -18       /* sdm_gx_gemm_step_noalloc: its first call on a device came during stream capture */
} sdm_gx_status;

/* Element strides of the three operands (innermost stride is 1 for all):
 *   x[n, j, i]    at x    + n*x_sn  + j*x_sj  + i
 *   d_dv[n, j, c] at d_dv + n*dv_sn + j*dv_sj + c
 *   d_u[n, i, c]  at d_u  + n*du_sn + i*du_si + c
 * Valid layouts: x_sj >= C, x_sn >= C*x_sj, dv_sj >= hd, dv_sn >= C*dv_sj, du_si >= hd, du_sn >= C*du_si. */
typedef struct sdm_gx_strides {
    int64_t x_sn, x_sj;
    int64_t dv_sn, dv_sj;
    int64_t du_sn, du_si;
} sdm_gx_strides;

/* Launch geometry of a plan (also what sdm_gx_gemm_geometry reports for a shape). */
typedef struct sdm_gx_geom {
    int32_t path;         /* 0: generic kernel (any layout), 1: TMA-fed pipelined kernel                       */
    int32_t config;       /* index of the tile configuration within the path                                  */
    int32_t TI;           /* rows i per tile                                                                   */
    int32_t TC;           /* columns c per tile                                                                */
    int32_t KB;           /* j values per shared-memory stage                                                  */
    int32_t stages;       /* pipeline stages (TMA path) or 1                                                   */
    int32_t threads;      /* threads per CTA                                                                   */
    int32_t smem_bytes;   /* dynamic shared memory per CTA                                                     */
    int64_t tiles;        /* tiles per step: P * ceil(C / TI) * ceil(hd / TC) (offset configurations on the
                             shifted grid: P * ceil((C + off_x) / TI) * ceil((hd + off_dv) / TC), off in floats)  */
    int32_t ctas;         /* CTAs launched per step (persistent: each loops over tiles)                        */
    int32_t ctas_per_sm;  /* resident CTAs per SM at this configuration                                        */
    int32_t sms;          /* SM count of the device                                                            */
    int32_t one_wave;     /* 1 if every tile gets its own resident CTA (tiles <= sms * ctas_per_sm)            */
} sdm_gx_geom;

typedef struct sdm_gx_plan sdm_gx_plan;   /* opaque; host memory only */

/* Flags (plan_create / step_ex). 0 selects everything automatically. */
#define SDM_GX_FLAG_GENERIC      0x100u   /* force the generic kernel                                         */
#define SDM_GX_FLAG_NO_PREFETCH  0x200u   /* TMA path: no L2 prefetch of d_dv before the dependency wait       */
#define SDM_GX_FLAG_CONFIG_MASK  0x0FFu   /* (index + 1) of a forced tile configuration of the chosen path     */
#define SDM_GX_FLAG_CTAS_SHIFT   12       /* bits 12..15: forced resident CTAs per SM (0 = automatic)          */
#define SDM_GX_FLAG_CTAS_MASK    0xF000u
/* Test hook for failure detection (TMA path only): the producer arms its first stage but never issues its copies, so
 * every wait on that stage runs out after ~20 ms instead of the normal 2 s bound. The launch then completes, leaves d_u
 * partly unwritten, sets the device error word (read it with sdm_gx_device_error), and the context stays usable. */
#define SDM_GX_FLAG_TEST_STALL   0x400u
/* Test hook for a late hand-off (stream kernel): every CTA stores its head's partial sums but never flags them, so
 * each tail's wait runs out after 1 ms and the CTA computes that tile's whole chain itself. The step's results stay
 * exact; the device error word gets its informational bit 3. */
#define SDM_GX_FLAG_TEST_NO_HANDOFF 0x20000u
/* x given transposed, as the page's baddbmm call sees it (x.transpose(1, 2)): stored as [n][i][j], so that
 * x[n, j, i] is at x + n*x_sn + i*x_sj + j (x_sj is then the stride between the stored rows i; the stride rules of
 * sdm_gx_strides are unchanged). step_ex, geometry and plans; the generic kernels serve it (small-tile kernels, with
 * j-fastest staging), the same chain and bits. */
#define SDM_GX_FLAG_X_TRANSPOSED 0x10000u
/* sdm_gx_gemm_geometry only (alone, contiguous operands): report the geometry sdm_gx_gemm_step_noalloc would use for
 * a step of this shape. It makes no set-up of the static workspace. */
#define SDM_GX_FLAG_NOALLOC      0x800u

/*
 * One step ti on contiguous operands (the page's gx_gemm launcher, minus torch). d_u, x, d_dv are device pointers of
 * the current device; the step reads x and d_dv chunks ti*P .. ti*P + P - 1 and updates the same d_u chunks.
 * N is not known here: the caller guarantees that those chunks exist (the strided/plan entries check ti < N / P).
 * Checks: pointers non-NULL and 4-byte aligned; 1 <= C <= 256; 1 <= hd < 2^20; P >= 1, ti >= 0 and
 * (ti + 1) * P < 2^31; the step's d_u span does not overlap its x or d_dv span.
 * stream: a cudaStream_t (NULL: the legacy default stream). pdl != 0: programmatic dependent launch (see above).
 */
SDM_GX_API int sdm_gx_gemm_step(float *d_u, const float *x, const float *d_dv, int64_t ti, int64_t P, int64_t C, int64_t hd,
                     cudaStream_t stream, int pdl);

/* One step on strided operands with the chunk count N (strides NULL: contiguous): the page's gx_gemm launcher, whose
 * checks (1 <= P <= N, ti < N / P, d_u disjoint from x and d_dv) it runs on whole tensors, extended to the strided
 * views of the baddbmm call in the page's module docstring. Checks 1 <= P <= N < 2^31 and
 * 0 <= ti < N / P, the stride rules of sdm_gx_strides, and that d_u's whole [N, C, hd] span overlaps neither x's
 * nor d_dv's. flags: SDM_GX_FLAG_*. */
SDM_GX_API int sdm_gx_gemm_step_ex(float *d_u, const float *x, const float *d_dv, int64_t ti, int64_t N, int64_t P, int64_t C,
                        int64_t hd, const sdm_gx_strides *strides, cudaStream_t stream, int pdl, unsigned flags);

/* The geometry a step of this shape and layout would use on the current device (no launch): the page's make_step
 * records its launch geometry in step.geom and LAST_GEOM (rows per CTA, CTA cap, minimum shared memory); this reports
 * the same facts for this library's kernels (path, tile, CTAs, one-wave check). */
SDM_GX_API int sdm_gx_gemm_geometry(const float *d_u, const float *x, const float *d_dv, int64_t N, int64_t P, int64_t C,
                         int64_t hd, const sdm_gx_strides *strides, unsigned flags, sdm_gx_geom *out);

/*
 * One step exactly as sdm_gx_gemm_step (same operands, checks, results and stream semantics), but the step may use the
 * stream kernel without a plan: its workspace is a static device array inside the library (about 10 MiB per device,
 * sized for devices of up to 160 SMs), so the call allocates nothing, ever. The pages have no counterpart to this
 * entry point; it exists for callers that must not allocate device memory and hold no plan.
 * Extra error: SDM_GX_E_RANGE also when the device has more than 160 SMs (the array is too small for it).
 * The first call on a device zero-fills the array's flags and launch counters and synchronises the device.
 * Races: every call on a device shares the one array. Calls whose kernels may overlap in time -- on different
 * streams without an ordering between them, or from several host threads onto unordered streams -- race on the
 * partial sums and flags and can return wrong results or report a device error. Order all calls of this entry point
 * on one device, e.g. issue them on one stream (with pdl as for sdm_gx_gemm_step: a step touches the array only after
 * its grid-dependency wait). Plans never use the array.
 */
SDM_GX_API int sdm_gx_gemm_step_noalloc(float *d_u, const float *x, const float *d_dv, int64_t ti, int64_t P, int64_t C,
                                        int64_t hd, cudaStream_t stream, int pdl);

/*
 * Plans (the page's gx_gemm_plan / gx_gemm_plan_launch): validate once, launch many steps with only ti changing.
 * plan_create runs every check of sdm_gx_gemm_step_ex for ti = ti_max (which covers every ti <= ti_max), picks the
 * kernel and tile configuration, sets the kernel attributes, and encodes the TMA descriptors of the whole tensors.
 * *out receives a plan allocated in host memory (free it with sdm_gx_gemm_plan_destroy). The plan is bound to the
 * current device.
 */
SDM_GX_API int sdm_gx_gemm_plan_create(sdm_gx_plan **out, float *d_u, const float *x, const float *d_dv, int64_t N, int64_t P,
                            int64_t C, int64_t hd, const sdm_gx_strides *strides, int64_t ti_max, unsigned flags);

/*
 * A plan with a workspace. With a large enough workspace the plan may pick the stream kernel: the step's work, in
 * units of (tile, j), split evenly over every resident CTA (one or two per SM, by tile shape) instead of in whole
 * tiles. A CTA then runs the first j of one
 * tile and another CTA continues those outputs' chains from the FP32 accumulators that the first one left in the
 * workspace. Each output still gets the one fixed chain acc = fmaf(x, d_dv, acc) for j = 0..C-1 from +0 and the one
 * final add, so the results are bit for bit those of every other kernel. The pages split work only in whole chunks;
 * this split is ours, for SM balance (e.g. 256 tiles on 152 SMs).
 *   workspace: device memory of the current device, 256-byte aligned, not overlapping d_u, x or d_dv, at least
 *   sdm_gx_gemm_plan_workspace_size() bytes; NULL (or too small) gives the plan of sdm_gx_gemm_plan_create.
 *   The call synchronises the device, zero-fills the workspace's control words and waits for that.
 *   The workspace belongs to the plan until it is destroyed: no other plan may use it, and the steps of this plan
 *   must run one after the other (stream-ordered, as sdm_gx_gemm_plan_run, the graph and the host driver launch
 *   them; with PDL each step touches the workspace only after its grid-dependency wait). Steps of one plan running
 *   concurrently on unordered streams would race on it.
 * The stream kernel runs one CTA per resident slot and expects all of them resident together (a whole GPU); under a
 * context limited to fewer SMs, create the plan without a workspace.
 * Errors as sdm_gx_gemm_plan_create, plus SDM_GX_E_ALIGN / SDM_GX_E_OVERLAP / SDM_GX_E_DEVICE for the workspace.
 */
SDM_GX_API int sdm_gx_gemm_plan_create_ws(sdm_gx_plan **out, float *d_u, const float *x, const float *d_dv, int64_t N,
                                          int64_t P, int64_t C, int64_t hd, const sdm_gx_strides *strides,
                                          int64_t ti_max, unsigned flags, void *workspace, size_t workspace_bytes);

/* No counterpart on the pages (their kernel keeps no state between CTAs). Bytes of workspace that lets a plan of this
 * shape and layout use the stream kernel on the current device (0: no
 * kernel of this shape uses one). About (resident CTAs) x TI x TC x 4 bytes: 9.5 MiB for 128 x 128 tiles on 152 SMs
 * (one CTA per SM), the same for 128 x 64 tiles (two per SM). */
SDM_GX_API int sdm_gx_gemm_plan_workspace_size(const float *d_u, const float *x, const float *d_dv, int64_t N,
                                               int64_t P, int64_t C, int64_t hd, const sdm_gx_strides *strides,
                                               unsigned flags, size_t *bytes);

/*
 * Measure instead of estimate. The page picks the tile height by a rule, and the plans here pick a configuration by an
 * estimate of the step time, which on some shapes is not the fastest. This call times every configuration of the
 * path that a plan of this shape and layout takes, and reports the fastest. Each configuration is forced in turn
 * (SDM_GX_FLAG_CONFIG_MASK) into a plan over the caller's buffers; the call skips those the shape, the device or the
 * workspace does not admit, and times the rest over 2 untimed steps and then `steps` timed steps (1 .. 4096). Steps
 * cycle over ti = 0 .. N/P - 1 and are chained with programmatic dependent launch, as sdm_gx_gemm_plan_run chains them.
 *   d_u: a scratch buffer with the shape and strides of the real d_u. The timed steps update it in place, so pass a
 *   copy, never the real d_u. x, d_dv, N, P, C, hd, strides, workspace: as for sdm_gx_gemm_plan_create_ws. A workspace
 *   lets the stream configurations take part; the plan created afterwards must then have one too.
 *   flags: base flags (SDM_GX_FLAG_GENERIC or SDM_GX_FLAG_NO_PREFETCH); a forced configuration or
 *   SDM_GX_FLAG_TEST_STALL in them is SDM_GX_E_FLAGS.
 *   *flags_out: flags | (index + 1) of the fastest configuration, for sdm_gx_gemm_plan_create[_ws] on buffers of
 *   the same shape and layout. *config_out and *us_out (each nullable): its index and its time per step.
 * Runs on `stream`, waits for it, and synchronises the device. Creating a plan for a stream configuration also
 * synchronises the device. No device memory is allocated.
 * Errors: those of sdm_gx_gemm_plan_create_ws; SDM_GX_E_NULL (flags_out NULL); SDM_GX_E_RANGE (steps out of range);
 * SDM_GX_E_CUDA; SDM_GX_E_DEVICE_FAULT when the device error word is set at the end.
 */
SDM_GX_API int sdm_gx_gemm_autotune(float *d_u, const float *x, const float *d_dv, int64_t N, int64_t P, int64_t C,
                                    int64_t hd, const sdm_gx_strides *strides, unsigned flags, void *workspace,
                                    size_t workspace_bytes, int steps, cudaStream_t stream, unsigned *flags_out,
                                    int32_t *config_out, float *us_out);

/* Launch step ti of a plan on `stream` (pdl as above): the page's gx_gemm_plan_launch, which sets ti in the recorded
 * launch and issues it, with its status codes -1 / -2 / -5 as the three plan errors below. Errors: SDM_GX_E_PLAN (NULL / corrupt plan),
 * SDM_GX_E_PLAN_TI (ti < 0 or ti > ti_max), SDM_GX_E_PLAN_DEVICE (current device differs), SDM_GX_E_CUDA. */
SDM_GX_API int sdm_gx_gemm_plan_step(const sdm_gx_plan *plan, int64_t ti, cudaStream_t stream, int pdl);

/* The multi-step driver (the page's C++ step loop bwd_steps_cuda over make_step's plan(nsteps), gx_gemm page section
 * "the backward's C++ step loop"): launch steps ti_begin, ti_begin +- 1, ... stopping before ti_end (descending when
 * ti_begin > ti_end, e.g. (T-1, -1) for the backward's reverse loop), back to back on `stream`. With pdl != 0 every
 * launch after the first uses programmatic dependent launch, so each step's prologue overlaps its predecessor. The
 * first launch uses pdl as given too (its predecessor is whatever the caller enqueued before). Every ti in the range
 * must lie in [0, ti_max]; nothing is launched otherwise. */
SDM_GX_API int sdm_gx_gemm_plan_run(const sdm_gx_plan *plan, int64_t ti_begin, int64_t ti_end, cudaStream_t stream, int pdl);

/* The same driver with the synthetic producer in the chain (the page's backward runs the step's GWR kernel, which
 * writes d_dv(ti), right before each step: module docstring, PDL paragraph; the producer stands in for it): before
 * each step ti it launches the producer, which
 * writes d_dv chunks of step ti from S (S has d_dv's shape and strides; see sdm_gx_producer_step). Producer and step
 * launches alternate on `stream`; with pdl != 0 each is a programmatic dependent launch of the one before. The steps
 * of this driver skip the L2 prefetch of d_dv before their dependency wait (the producer is about to rewrite it). */
SDM_GX_API int sdm_gx_gemm_plan_run_producer(const sdm_gx_plan *plan, const float *S, int64_t ti_begin, int64_t ti_end,
                                  cudaStream_t stream, int pdl);

/*
 * A step chain captured once into an instantiated CUDA graph (the page's per-backward plan and C++ step loop, with the
 * host launch cost of every step paid once): the launches sdm_gx_gemm_plan_run (S == NULL) or
 * sdm_gx_gemm_plan_run_producer (S != NULL) would issue for ti_begin .. ti_end, with the synthetic successor after
 * every step when succ_out != NULL (sdm_gx_gemm_plan_run_successor), captured on a private stream, with
 * programmatic-dependent-launch edges when pdl != 0. *out receives the graph (host-side handle). The graph holds the
 * plan's pointers; it is valid while those buffers live, and on the plan's device. Creating it makes no launch.
 */
typedef struct sdm_gx_graph sdm_gx_graph;
SDM_GX_API int sdm_gx_gemm_plan_graph_create(sdm_gx_graph **out, const sdm_gx_plan *plan, const float *S,
                                             float *succ_out, int64_t ti_begin, int64_t ti_end, int pdl);
/* Launch the whole captured chain on `stream` (stream-ordered, asynchronous), as the page's step loop issues its plan
 * launches. Errors: SDM_GX_E_PLAN (NULL / corrupt graph), SDM_GX_E_PLAN_DEVICE, SDM_GX_E_CUDA. */
SDM_GX_API int sdm_gx_graph_launch(const sdm_gx_graph *graph, cudaStream_t stream);
/* Free a graph (NULL or an already destroyed handle: no effect). No counterpart on the pages: their plan is a torch
 * tensor freed with it. */
SDM_GX_API void sdm_gx_graph_destroy(sdm_gx_graph *graph);

/*
 * The chain with a synthetic successor after every step: step ti, then a consumer of d_u(ti) launched with programmatic
 * dependent launch (the page's next kernel of the backward step, "Phase A", reads token rows of d_u after its own
 * dependency wait and lets the following kernel start early; its algorithm is not built here). For every chunk n of
 * step ti the successor writes out[n] = the sum of the chunk's leading row d_u[n, 0, :] in a fixed order (per lane
 * l: columns l, l + 32, ... left to right from +0; then an xor butterfly over the 32 lanes with offsets 16, 8, 4, 2, 1),
 * and it triggers its dependents before its wait. out: device float array of N elements, not overlapping d_u, x or
 * d_dv. It measures the step -> successor -> next step hand-off.
 */
SDM_GX_API int sdm_gx_gemm_plan_run_successor(const sdm_gx_plan *plan, float *out, int64_t ti_begin, int64_t ti_end,
                                              cudaStream_t stream, int pdl);
/*
 * No counterpart on the pages (their operands are device tensors already). The chain fed from host memory, with
 * copies and compute overlapped: for every step ti (in the order ti_begin,
 * ti_begin +- 1, .. as sdm_gx_gemm_plan_run) the step's slices of x, d_dv and d_u are copied from the host arrays into
 * the plan's device tensors on stream `h2d`, the step runs on `compute` once they have arrived, and the step's d_u
 * slice is copied back to d_u_host on stream `d2h` once the step is done (consecutive steps are copied together in
 * groups of about 16 MB). While a group computes, the next group's copies in and the previous group's copies out
 * proceed. A call's copies in start after the work already enqueued on `compute` and `d2h`. The host arrays have the plan's logical shapes, contiguous
 * (x_host [N][C][C], d_dv_host and d_u_host [N][C][hd]); the plan's device tensors must be contiguous too. Use pinned
 * host memory for the copies to run asynchronously. Returns once everything is enqueued; the caller synchronises on
 * `d2h` (which ends with the last copy back). The three streams must be distinct.
 */
SDM_GX_API int sdm_gx_gemm_plan_run_host(const sdm_gx_plan *plan, float *d_u_host, const float *x_host,
                                         const float *d_dv_host, int64_t ti_begin, int64_t ti_end,
                                         cudaStream_t compute, cudaStream_t h2d, cudaStream_t d2h);
/*
 * An optional timeline of a plan's launches, for measuring what the page's PDL design is about: the gap between
 * chained steps (the page's module docstring: the step's reads before griddepcontrol.wait overlap the previous
 * kernel) and the start and end of each step. No counterpart on the pages (they time with CUDA events and profilers).
 * buf: device memory of the plan's device, 8-byte aligned, launches * (*ctas) * 4 entries; NULL or launches == 0
 * turns the timeline off. With it on, every launch of step ti < launches writes, for each of its CTAs b,
 * buf[(ti * ctas + b) * 4 + k] = the GPU's global timer in ns: k = 0 when the CTA starts, 1 when its first consumer
 * warp is past the grid-dependency wait, 2 when that warp holds its first staged data (stream kernel; 0 elsewhere),
 * 3 when that warp is done with its last output. Launches of steps >= launches write nothing. The plan records the
 * buffer: launches and graphs made after the call use it, graphs made before do not. Call it between launches (it
 * modifies the plan). *ctas (nullable) receives the CTAs per launch (the plan's geometry ctas).
 * Errors: SDM_GX_E_PLAN / SDM_GX_E_PLAN_DEVICE as for plan launches; SDM_GX_E_UNSUPPORTED for a plan on the generic or
 * slab kernel; SDM_GX_E_RANGE (launches < 0 or the buffer's index past 2^31); SDM_GX_E_ALIGN; SDM_GX_E_DEVICE.
 */
SDM_GX_API int sdm_gx_gemm_plan_set_trace(sdm_gx_plan *plan, unsigned long long *buf, int64_t launches,
                                          int32_t *ctas);

/* The geometry a plan launches every step with (the page's step.geom / LAST_GEOM for the plan's make_step). Errors:
 * SDM_GX_E_NULL (out NULL), SDM_GX_E_PLAN (NULL / corrupt plan). Makes no CUDA call. */
SDM_GX_API int sdm_gx_gemm_plan_geometry(const sdm_gx_plan *plan, sdm_gx_geom *out);
/* Free a plan's host memory (the page's plan is a tensor freed by torch). NULL or a corrupt plan: no effect. */
SDM_GX_API void sdm_gx_gemm_plan_destroy(sdm_gx_plan *plan);

/*
 * The synthetic producer of the chained workload (not on the pages: it stands in for the kernel that writes d_dv(ti)
 * right before each step). For chunks n = ti*P .. ti*P + P - 1: d_dv[n, j, c] = S[n, j, c] if ti is even, else
 * -S[n, j, c] (an exact sign flip). S and d_dv are contiguous [N, C, hd] device arrays; S must not overlap d_dv.
 * Under pdl it reads S before its dependency wait and writes d_dv after it.
 */
SDM_GX_API int sdm_gx_producer_step(float *d_dv, const float *S, int64_t ti, int64_t P, int64_t C, int64_t hd,
                         cudaStream_t stream, int pdl);

/* Registers per thread, local (spill) bytes, static shared bytes and max threads per block of a kernel (the page's
 * gx_gemm_attrs, which fills the same four int64 values for the one kernel instance it builds): path 0 = generic
 * (config 0..2 = 16/32/64 x 64 tiles, 3 = the 128 x 64 large-tile kernel), path 1 = TMA (config index as in
 * sdm_gx_geom). This library builds one kernel per configuration, so the call names the kernel; out[4] is as on the
 * page. Errors: SDM_GX_E_NULL, SDM_GX_E_FLAGS (unknown path or config), SDM_GX_E_CUDA. */
SDM_GX_API int sdm_gx_gemm_kernel_attrs(int32_t path, int32_t config, int64_t out[4]);

/* Static description of configuration `config` of a path (for sweeps and tests; the page's kernel has one tile width
 * TC = 64 and a row count chosen per launch by _rows, this library a menu of tiles): out[0..7] = TI, TC, KB, stages,
 * threads per CTA, dynamic shared memory bytes, kind (0: tile kernel, 1: balanced slab kernel, 2: stream kernel, which
 * needs a plan workspace, 3: tile kernel for bases off a 16-byte boundary, its boxes 4 floats wider and read by
 * element loads or realigned once per stage, 4: the same on the shifted tile grid, which needs d_u and d_dv equally
 * far off), consumer warps. SDM_GX_E_FLAGS for an unknown path or index. */
SDM_GX_API int sdm_gx_gemm_config_info(int32_t path, int32_t config, int32_t out[8]);

/* The stream kernel's split of a step (no counterpart on the pages, which give every chunk's tile to one CTA; the
 * chain split at a j boundary keeps the page's fixed order, module docstring formula; host code shared with the
 * kernel, for tests and tools): the step's
 * ntiles x C units (tile t, j), ordered by (t, j), go to CTAs 0..G-1 in equal contiguous ranges (CTA b: units
 * [b W / G, (b + 1) W / G), W = ntiles x C). Needs 1 <= C <= 256 and 1 <= G <= ntiles < 2^31 (every range is then at
 * least one tile long), 0 <= b < G. With q < 0 it returns the number of pieces CTA b runs; otherwise it writes piece q
 * (in the order the CTA runs them) to out[0..3] = tile, j0, j1 (the piece covers j0 <= j < j1) and kind (0: a whole
 * tile; 1: the head of a tile, run first, whose accumulators CTA b + 1 continues; 2: the tail of a tile, run last,
 * continuing CTA b - 1's accumulators) and returns 0. SDM_GX_E_RANGE for arguments outside those bounds. */
SDM_GX_API int sdm_gx_gemm_stream_piece(int64_t ntiles, int32_t C, int32_t G, int32_t b, int32_t q, int32_t out[4]);

/* The configuration a plan would choose, for a DESCRIBED device (the counterpart of the page's _rows / one_wave rule,
 * which also takes the SM count as an input): the same rule as sdm_gx_gemm_plan_create, on the
 * SM count `sms`, the resident CTAs per SM of every configuration of `path` (occ[k], n_occ entries =
 * sdm_gx_gemm_num_configs(path)), whether the slab kernel's 4-D x view is available (slab_ok), and a plan workspace
 * of ws_bytes (0: none). Makes no CUDA call (a diagnostic for tests and tools; a device's own values come from
 * sdm_gx_gemm_geometry). Returns the configuration's index (>= 0), or SDM_GX_E_NULL (occ NULL), SDM_GX_E_FLAGS
 * (path not 0 / 1), SDM_GX_E_SHAPE (C or hd out of range), SDM_GX_E_RANGE (sms outside [1, 4096], n_occ wrong,
 * a negative occ, P outside [1, 2^31)), SDM_GX_E_SMEM (no configuration is usable). */
SDM_GX_API int sdm_gx_gemm_choose_config(int32_t path, int32_t sms, const int32_t *occ, int32_t n_occ, int32_t slab_ok,
                                         int64_t P, int64_t C, int64_t hd, size_t ws_bytes);

/* Number of tile configurations of a path (for sweeps and tests; the page's menu is its GX_GEMM rows instances). */
SDM_GX_API int sdm_gx_gemm_num_configs(int32_t path);

/* The device error word of the current device. The page reports failures through its launcher's checks and the
 * negative status codes of gx_gemm_plan_launch; its kernel has no waits that can expire, so this word has no
 * counterpart there: it reports the bounded waits of this library's pipelined kernels. Bits 0-2 mean a kernel gave up
 * a bounded wait and its step is incomplete (bit 0: a consumer waited too long for staged data, bit 1: the producer
 * waited too long for a free stage, bit 2: a drain wait gave up); the call then returns SDM_GX_E_DEVICE_FAULT. Bit 3 is
 * informational: a stream-kernel CTA waited more than 1 ms for the previous CTA's partial sums and computed that
 * tile's whole chain itself, so the step's results are exact (the call returns SDM_GX_OK). Synchronizes the device.
 * clear != 0 resets the word to 0 afterwards. */
SDM_GX_API int sdm_gx_device_error(uint32_t *word, int clear);
#define SDM_GX_ERR_FATAL_MASK         0x7u   /* bits 0-2: a bounded wait gave up, the step is incomplete            */
#define SDM_GX_ERR_HANDOFF_RECOMPUTED 0x8u   /* bit 3, informational: a tile's chain recomputed, results exact      */

/* Launches of the library's kernels since load (the page's PDL_LAUNCHES counters, split by kernel): out[0] = step
 * kernels, out[1] = producer kernels,
 * out[2] = launches with programmatic dependent launch, out[3] = successor kernels. */
SDM_GX_API void sdm_gx_launch_counts(int64_t out[4]);

/* The cudaError_t of the last SDM_GX_E_CUDA returned on this host thread, 0 if none (the page's launcher raises the
 * CUDA error itself through C10_CUDA_CHECK; a C ABI returns SDM_GX_E_CUDA and keeps the code here). */
SDM_GX_API int sdm_gx_last_cuda_error(void);

/* A static description of a status code: the messages of the page's launcher checks (gx_gemm's TORCH_CHECKs) and of
 * gx_gemm_plan_launch's status codes (-1 corrupt plan, -2 step outside ti_max, -5 device mismatch), restated for
 * sdm_gx_status. Never NULL; unknown codes give "unknown status". */
SDM_GX_API const char *sdm_gx_strerror(int status);

/* SDM_GX_ABI_VERSION of the loaded library (no counterpart on the pages: a C ABI's version check). */
SDM_GX_API int sdm_gx_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SDM_GX_GEMM_H_ */
