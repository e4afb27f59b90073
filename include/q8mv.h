/*
 * q8mv: Q8_0 decode matrix-vector product on one NVIDIA GB300 (sm_103a).
 *
 * Operation (Phobos docs, "Q8_0 matvec" example page, "The tensors" and
 * "Factoring out the scale"):
 *
 *     C[0, n] = sum over blocks b of  S[b, n] * ( sum over k in block b of A[0, k] * W[k, n] )
 *
 * with blocks of 32 rows along K: block b holds rows 32*b .. 32*b+31 of W and
 * is scaled by row b of S.  K need not be a multiple of 32 ("Bounds"): the
 * last block then holds K - 32*(KB-1) rows and rows at or past K are never
 * read.  N need not be a multiple of anything: columns at or past N are
 * neither read nor written.
 *
 * Tensors (all contiguous, row-major, in device memory of the plan's GPU):
 *     A  f32  [1, K]        activation row                         (4*K bytes)
 *     W  i8   [K, N]        quantized weights, W[k, n] at k*N + n  (K*N bytes)
 *     S  f32  [KB, N]       block scales, KB = ceil(K / 32),
 *                           S[b, n] at b*N + n                     (4*KB*N bytes)
 *     C  f32  [1, N]        output row, overwritten                (4*N bytes)
 *
 * Arithmetic: each weight byte is converted to f32 exactly (every value in
 * -128 .. 127), each block's dot product is accumulated in f32 on the raw
 * bytes, and the block's scale is applied once per block and column with a
 * fused multiply-add into an f32 accumulator.  Summation order is fixed by
 * the plan, so a plan gives bit-identical results run after run.
 *
 * Ownership: the caller owns A, W, S and C.  A plan owns a small device
 * workspace (split-K partial sums and per-tile counters) that it allocates in
 * q8mv_plan and frees in q8mv_destroy; q8mv_run never allocates.
 *
 * Concurrency: q8mv_run is asynchronous on the given stream.  Calls on one
 * plan share its workspace, so they must be ordered (same stream, or
 * otherwise serialised); use one plan per concurrent stream.
 *
 * Errors: every call returns a q8mv_status_t.  Arguments are validated on the
 * host before anything is launched; q8mv_run reports launch-time errors only
 * (it does not synchronise).  The register, rows and batched register kernels
 * never wait on anything.  The streaming and tcgen05 kernels wait on
 * shared-memory barriers for their copies and handoffs; every such wait is
 * bounded (about 2 s), and a wait that runs out is recorded in the plan's
 * device error word (q8mv_check) instead of hanging the GPU.
 */
#ifndef Q8MV_H
#define Q8MV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    Q8MV_OK = 0,
    Q8MV_ERR_INVALID_ARG = 1,        /* null/misaligned/overlapping pointer, bad size, bad option */
    Q8MV_ERR_UNSUPPORTED_DEVICE = 2, /* no device, or not an sm_103 GPU this library was built for */
    Q8MV_ERR_OUT_OF_MEMORY = 3,      /* host or device allocation for the plan failed */
    Q8MV_ERR_CUDA = 4,               /* any other CUDA runtime error (see q8mv_last_cuda_error) */
    Q8MV_ERR_SCRATCH_TOO_SMALL = 5   /* q8mv_run_noalloc: the shape needs more split-K scratch than
                                        Q8MV_NOALLOC_SCRATCH_BYTES */
} q8mv_status_t;

/* Kernel families a plan can pick. */
enum {
    Q8MV_KERNEL_AUTO = 0,
    Q8MV_KERNEL_REGS = 1, /* weights streamed through registers with vector loads; any alignment */
    Q8MV_KERNEL_STREAM = 2, /* weights and scales streamed by the tensor-memory accelerator into a
                               shared-memory ring, one CTA per SM taking at most half of it, so that
                               the next call's CTAs become resident beside the running call and fill
                               their rings while it computes (with overlap = 1); split-K summed through
                               a thread-block cluster.  Needs N % 16 == 0, K <= 65536 and 16-byte
                               aligned W and S, else the register kernel runs.  (Value 3 is retired.) */
    Q8MV_KERNEL_ROWS = 4,  /* weights stored one output row per row (q8mv_plan_transposed): a CTA owns
                              rows_per_cta outputs, its warps split K, lanes read 16 bytes of a row */
    Q8MV_KERNEL_ROWS_I8 = 5, /* as ROWS, with int8 activations: each 32-element block of A is quantized
                                in the kernel (q8mv_quantize_rows) and multiplied with dp4a */
    Q8MV_KERNEL_MMA = 6,     /* batched plans: the block products of 16 activation rows on the tensor
                                cores (mma.sync bf16, A split into three bf16 parts); needs N % 4 == 0
                                and a 4-byte aligned W, else the batched register kernel runs */
    Q8MV_KERNEL_TC = 7       /* batched plans: the block products of 16 activation rows on the
                                5th-generation tensor cores (tcgen05.mma bf16, accumulators in tensor
                                memory, A split once per call into three bf16 parts); needs
                                N % 16 == 0 and a 16-byte aligned W, else the batched register kernel
                                runs */
};

/*
 * Optional overrides for tuning sweeps and tests.  Zero means "let the plan
 * choose".  An override that cannot apply to the shape gives INVALID_ARG.
 */
typedef struct {
    int32_t kernel;    /* Q8MV_KERNEL_* */
    int32_t vec_bytes; /* weight load per thread and row: 16, 8, 4, 2 or 1, used whenever W's
                          address allows it (narrower loads only as a fallback); 0 lets the
                          planner pick the width it expects to be fastest */
    int32_t threads_n; /* threads along N in one CTA: 32, 64, 128 or 256 */
    int32_t split_k;   /* K ranges per column tile, each summed by one CTA (>= 1; the streaming
                          kernel takes 1 .. 16, the cluster size) */
    int32_t stages;    /* streaming kernel: ring depth, 8, 16 or 24 stages of one 32 x 256 block
                          (as shared memory allows) */
    int32_t overlap;   /* 1: launch with programmatic dependent launch, so a call starts while the
                          previous kernel in its stream finishes and reads W and S before that kernel
                          has completed (A is read and C written only after it).  Only for weights
                          that the preceding work in the stream does not write. */
    int32_t cta_threads; /* register kernel: 128 or 256 threads per CTA; transposed plans: 32, 64,
                            128 or 256 (the warps splitting K, at most one per 512-wide step) */
    int32_t rows_per_cta; /* transposed plans: output rows per CTA, 8 or 16 */
} q8mv_opts_t;

/* What a plan chose for 16-byte aligned tensors: the kernel family asked for
 * (the register kernel by default) and, for the register kernel, the weight
 * load width the planner expects to be fastest. */
typedef struct {
    int32_t kernel;           /* Q8MV_KERNEL_* the plan runs for 16-byte aligned tensors */
    int32_t vec_bytes;        /* weight bytes per thread per row */
    int32_t threads_n;        /* threads along N per CTA */
    int32_t groups_k;         /* thread groups along K per CTA (threads per CTA / threads_n) */
    int32_t threads_per_cta;
    int32_t split_k;          /* K ranges per column tile (partial rows summed in range order) */
    int32_t blocks_per_split; /* 32-row blocks in each K range */
    int32_t stages;           /* streaming kernel's ring depth (0 for the register kernel) */
    int32_t overlap;          /* programmatic dependent launch enabled */
    int32_t cluster;          /* split-K partial rows summed through a thread-block cluster's
                                 distributed shared memory (no workspace) */
    int64_t tile_n;           /* output columns per CTA */
    int64_t grid_x;           /* column tiles */
    int64_t grid_y;           /* = split_k */
    int64_t workspace_bytes;  /* device workspace the plan owns */
    int32_t sm_count;
    int32_t ctas_per_sm;      /* resident CTAs per SM for the chosen kernel */
    int32_t rows;             /* activation rows M of the plan (1 for q8mv_plan) */
    int32_t rows_per_pass;    /* activation rows one CTA serves (1, or 2, 4, 8, 16 when batched) */
    int64_t grid_z;           /* passes of rows_per_pass rows: ceil(rows / rows_per_pass) */
} q8mv_plan_info_t;

typedef struct q8mv_plan_s *q8mv_plan_t;

/*
 * Create a plan for C[1,N] = A[1,K] x (W[K,N], S[KB,N]) on `device`
 * (-1 = the current device).  Queries the SM count, picks the kernel, tile
 * and split, and allocates the workspace.  K >= 0, N >= 0, K < 2^31,
 * N < 2^31 and K*N < 2^62; otherwise INVALID_ARG.  `opts` may be NULL.
 * On success *out holds the plan; on failure *out is set to NULL.
 * The calling thread's current device is left unchanged.
 */
q8mv_status_t q8mv_plan(q8mv_plan_t *out, int64_t K, int64_t N, int device,
                        const q8mv_opts_t *opts);

/*
 * Weights stored one output row per row: a plan for C[1,N] = A[1,K] x (Wt, St)
 * where Wt is i8 [N, K] (Wt[n, k] at n*K + k, output n's bytes in row n) and
 * St is f32 [N, KB] (St[n, b] at n*KB + b, output n's block scales):
 *
 *     C[0, n] = sum_b St[n, b] * ( sum_{k in block b} A[0, k] * Wt[n, k] )
 *
 * the Q8_0 product above with W = Wt^T and S = St^T, in the layout that dot_t
 * contracts ("dot and tensor cores" page: the last axis of both operands, as a
 * linear layer stores its weights).  q8mv_run and q8mv_run_fused then take Wt
 * and St in place of W and S.  Limits as for q8mv_plan.  Accepted overrides:
 * vec_bytes (16, 4 or 1: load per lane and step, used when K and Wt's address
 * allow it, narrower loads as the fallback), rows_per_cta (8 or 16), cta_threads
 * (32, 64, 128 or 256: warps along K; by default the fewest, at least 2 with
 * int8 activations, that still give every SM 32 warps, 12 with int8
 * activations), overlap,
 * and kernel = Q8MV_KERNEL_ROWS_I8 for int8 activations (below); any other
 * non-zero field gives INVALID_ARG.  Each output's blocks are summed in order
 * within a fixed interleave, so a plan is bitwise repeatable.
 *
 * Int8 activations (kernel = Q8MV_KERNEL_ROWS_I8; "dot and tensor cores" page,
 * "Hardware paths": an i8 dot_t accumulates in i32, a single row takes dp4a):
 * the kernel quantizes each 32-element block b of A as q8mv_quantize_rows does
 * and computes
 *     C[0, n] = sum_b (d_b * St[n, b]) * ( sum_{k in block b} q[k] * Wt[n, k] )
 * with the block's dot product exact in i32 (four dp4a per 16 bytes) and one
 * f32 fold per block.  This is an approximation of the f32 product: the codes
 * carry about 7 bits of each activation.
 */
q8mv_status_t q8mv_plan_transposed(q8mv_plan_t *out, int64_t K, int64_t N, int device,
                                   const q8mv_opts_t *opts);

/*
 * Int8 codes of M activation rows: for each 32-element block b of row m (the
 * last block may be partial), in IEEE f32 arithmetic,
 *     amax = max |A[m, k]|,  d[m, b] = amax / 127,
 *     q[m, k] = rint(A[m, k] * (127 / amax))   (ties to even; 0 when amax = 0)
 * so that A[m, k] ~ q[m, k] * d[m, b].  A f32 [M, K], q i8 [M, K], d f32
 * [M, KB], all device memory, row-major; A and d 4-byte aligned, no overlaps.
 * 0 <= M <= 65535.  Asynchronous on `stream`; the current device is used.
 */
q8mv_status_t q8mv_quantize_rows(int64_t M, int64_t K, const float *A, int8_t *q, float *d,
                                 cudaStream_t stream);

/*
 * Batched decode: a plan for C[M,N] = A[M,K] x (W[K,N], S[KB,N]), each row of
 * C the matvec above of the same row of A (A and C contiguous, row-major:
 * A[m, k] at m*K + k, C[m, n] at m*N + n).  The Q8_0 matvec example page
 * ("The tensors") defines one activation row, A[1, K]; here M rows share one
 * pass over the weights, as a decode step of M sequences does.
 *
 * 1 <= M <= 2^19, otherwise INVALID_ARG; the other limits and the ownership
 * rules are those of q8mv_plan.  M == 1 gives exactly the plan of q8mv_plan.
 * For M >= 2 the plan uses the batched register kernel: rows are served
 * 2, 4, 8 or 16 at a time (M rounded up to one of them, or ceil(M/16) passes
 * of 16 that each stream the weights again).  Accepted overrides: vec_bytes
 * (8, 4 or 1; 8-byte loads exist for up to 4 rows per pass), threads_n,
 * split_k, overlap, and kernel = Q8MV_KERNEL_MMA or Q8MV_KERNEL_TC for the
 * tensor-core kernels (which take split_k and overlap); any other non-zero field gives
 * INVALID_ARG.  Without a kernel named (and without vec_bytes or
 * threads_n, which tune the register kernel), 16 rows per pass, and 8 rows
 * per pass on weights of K * N >= 2^25, use the tcgen05 kernel when N % 16
 * == 0 and W and S are 16-byte aligned; everything else uses the register
 * kernel.
 *
 * Per element the arithmetic is that of q8mv_plan: exact byte conversion,
 * the block's 32 products summed in f32 in row order, one scale fold per
 * block, column and activation row, and split-K partial sums added in range
 * order, so a row's result does not depend on the other rows.
 */
q8mv_status_t q8mv_plan_batched(q8mv_plan_t *out, int64_t M, int64_t K, int64_t N, int device,
                                const q8mv_opts_t *opts);

/*
 * Enqueue C = matvec(A, W, S) on `stream` (0 = the legacy default stream).
 * For a batched plan A is [M, K] and C is [M, N] (see q8mv_plan_batched).
 * The plan's device must be current.  A, S and C must be 4-byte aligned;
 * W may have any alignment (narrower loads are used when W, S or N do not
 * allow 16-byte ones).  C must not overlap A, W or S.  Null pointers are
 * allowed only for tensors of zero size.  K == 0 writes C = 0; N == 0 is a
 * no-op.  Returns after the launch; errors inside the kernel surface on the
 * next synchronising call, as for any CUDA kernel.
 */
q8mv_status_t q8mv_run(q8mv_plan_t plan, const float *A, const int8_t *W, const float *S,
                       float *C, cudaStream_t stream);

/*
 * Fused epilogue ("dot and tensor cores" page, "The fused epilogue"): an
 * elementwise statement applied to each output as it is written, instead of
 * storing the product and sweeping it again.  For output (m, n) of a call
 * whose product is x[m, n]:
 *
 *     y = alpha * x[m, n] + beta * C[m, n] + bias[n]     (f32; C's previous
 *                                                         contents are read only
 *                                                         if beta != 0)
 *     y = act(y)
 *     C[m, n] = y + residual[m, n]
 *
 * The page's two forms are alpha (s = s * scale) and beta (acc = acc * corr +
 * dot(p, v)); bias, activation and residual are those of a decode layer.
 * act: none, relu = max(y, 0), silu = y / (1 + exp(-y)), or the tanh form of
 * gelu, 0.5 y (1 + tanh(sqrt(2/pi) (y + 0.044715 y^3))), with CUDA's expf and
 * tanhf.
 */
enum {
    Q8MV_ACT_NONE = 0,
    Q8MV_ACT_RELU = 1,
    Q8MV_ACT_SILU = 2,
    Q8MV_ACT_GELU_TANH = 3
};

typedef struct {
    float alpha;           /* scale of the product (1 = the product itself) */
    float beta;            /* scale of C's previous contents (0 = C is not read) */
    const float *bias;     /* [N], the same for every row, added before the activation; NULL = none */
    const float *residual; /* [M, N] (M = 1 for q8mv_plan), added after the activation; NULL = none */
    int32_t act;           /* Q8MV_ACT_* */
} q8mv_epilogue_t;

/*
 * q8mv_run with the fused epilogue `epi` (NULL = q8mv_run).  Same rules as
 * q8mv_run; in addition bias and residual are 4-byte aligned device arrays of
 * the plan's device that do not overlap C, and act is one of Q8MV_ACT_*.
 * Every kernel applies the epilogue as it writes C; for K == 0 the register
 * (or batched register) kernel runs it on a product of 0, so
 * C = act(beta * C + bias) + residual.
 */
q8mv_status_t q8mv_run_fused(q8mv_plan_t plan, const float *A, const int8_t *W, const float *S,
                             float *C, const q8mv_epilogue_t *epi, cudaStream_t stream);

/*
 * Synchronise the plan's device and report in *device_error the error bits
 * its kernels recorded since the last check (0 = none).  Streaming kernel:
 * 1 = a ring stage's copies did not land in time, 2 = a ring stage was not
 * released in time, 4 = copies in flight did not land in time at the end.
 * tcgen05 kernel: 8 = a stage or handoff wait ran out, 16 = the MMAs did not
 * complete in time, 32 = its final wait for copies and MMAs ran out.  A
 * kernel that records an error stops waiting and finishes; its output is then
 * undefined.  The bits are cleared, and the plan's split-K counters are reset
 * when any was set.
 */
q8mv_status_t q8mv_check(q8mv_plan_t plan, int32_t *device_error);

/*
 * For tests of the bounded-wait path only.  Sets the bound on every
 * shared-memory barrier wait of the plan's streaming and tcgen05 kernels to
 * wait_ns nanoseconds (0 restores the default of 2 s) and makes every ring
 * stage's barrier expect extra_tx bytes more than its copies deliver (0 in
 * normal use).  With extra_tx > 0 no stage ever completes, so the kernel's
 * first wait runs out after wait_ns: it records its error bit (q8mv_check),
 * stops issuing, waits at most wait_ns for what it issued, releases what it
 * holds and returns, and the GPU stays usable.  Calls made after restoring
 * (0, 0) compute normally.  INVALID_ARG for a NULL plan or wait_ns above 10 s.
 */
q8mv_status_t q8mv_plan_set_waits(q8mv_plan_t plan, uint64_t wait_ns, uint32_t extra_tx);

/* Release the plan and its workspace.  NULL is accepted.  Synchronises the
 * plan's device first so that no launch still uses the workspace. */
q8mv_status_t q8mv_destroy(q8mv_plan_t plan);

/* Fill *info with the plan's choices (for the widest legal weight load). */
q8mv_status_t q8mv_plan_info(q8mv_plan_t plan, q8mv_plan_info_t *info);

/*
 * Host-only planning, no GPU needed: the configuration q8mv_plan would pick
 * for K, N on a GPU with `sm_count` SMs.  For the register kernel (opts NULL
 * or kernel REGS/AUTO): `ctas_per_sm` resident CTAs and weight loads of
 * `vec_bytes` (which must divide N).  For opts->kernel == Q8MV_KERNEL_STREAM
 * the last two are ignored and an SM is taken to hold 228 KiB of shared
 * memory with 1 KiB reserved per CTA.  For opts->kernel == Q8MV_KERNEL_ROWS or
 * Q8MV_KERNEL_ROWS_I8: the transposed plan's rows per CTA and warps along K
 * (which depend on sm_count, not on ctas_per_sm, which is only reported back)
 * for loads of `vec_bytes` (16, 4 or 1).  Fills *info (workspace_bytes of
 * partial rows).
 */
q8mv_status_t q8mv_choose_config(int64_t K, int64_t N, int32_t sm_count, int32_t ctas_per_sm,
                                 int32_t vec_bytes, const q8mv_opts_t *opts,
                                 q8mv_plan_info_t *info);

/*
 * Host-only planning for a batched plan of M rows: the configuration
 * q8mv_plan_batched would pick on a GPU with `sm_count` SMs, where registers
 * allow `ctas_per_sm` resident CTAs of the batched kernel, with weight loads
 * of `vec_bytes` (8, 4 or 1, dividing N).  Fills *info.  With opts->kernel ==
 * Q8MV_KERNEL_TC or Q8MV_KERNEL_MMA it plans that tensor-core kernel instead
 * (`ctas_per_sm` its resident CTAs, `vec_bytes` ignored); INVALID_ARG when the
 * shape cannot take it (TC: N % 16 != 0; MMA: N % 4 != 0).
 */
q8mv_status_t q8mv_choose_config_batched(int64_t M, int64_t K, int64_t N, int32_t sm_count,
                                         int32_t ctas_per_sm, int32_t vec_bytes,
                                         const q8mv_opts_t *opts, q8mv_plan_info_t *info);

/* Static, human-readable text for a status code. */
const char *q8mv_status_string(q8mv_status_t status);

/*
 * Feed-forward pair: the up and down matvecs of one feed-forward block, the
 * down product reading the up product's output,
 *
 *     H[n] = epi_up(   sum_b S_up[b, n]   * ( sum_{k in b} A[k] * W_up[k, n] ) )     n < N_mid
 *     C[n] = epi_down( sum_b S_down[b, n] * ( sum_{k in b} H[k] * W_down[k, n] ) )   n < N_out
 *
 * each product the Q8_0 matvec above ("Q8_0 matvec" page) and each epilogue
 * the fused epilogue of q8mv_run_fused ("dot and tensor cores" page, "The
 * fused epilogue"), fused into one launch ("fusing the matvec pair
 * up -> down" of a feed-forward block) or chained as two.
 *
 * Tensors (device memory of the pair's GPU, contiguous, row-major):
 *     A       f32 [K]                     activation row
 *     W_up    i8  [K, N_mid]   S_up   f32 [ceil(K/32), N_mid]
 *     H       f32 [N_mid]                 the up product's output (written, then read back)
 *     W_down  i8  [N_mid, N_out]  S_down f32 [ceil(N_mid/32), N_out]
 *     C       f32 [N_out]                 output, overwritten
 *
 * Modes.  Q8MV_PAIR_AUTO (0) and Q8MV_PAIR_TWO_LAUNCHES run the products as
 * two q8mv_run_fused calls of single-row plans, the second launched with
 * programmatic dependent launch when opts->overlap is 1 (its first weight
 * loads then overlap the first call's tail).  Q8MV_PAIR_ONE_LAUNCH runs both
 * in one cooperative launch of the pair kernel: every CTA is resident, takes
 * one item of the up product, loads the first weight block of its item of
 * the down product, waits at a grid-wide barrier for H to be complete, then
 * computes that item; it needs N_mid and N_out to be multiples of 8
 * (q8mv_pair_plan fails with INVALID_ARG otherwise) and, at run time, W_up and
 * W_down 8-byte and S_up, S_down 4-byte aligned (else the call takes two
 * launches).  AUTO takes two launches because they measured faster on GB300
 * (7B FFN pair: 24.3 us against 26.1 us).
 *
 * Rules: those of q8mv_run_fused for each product; in addition H may overlap
 * none of A, W_up, S_up, W_down, S_down, C, nor epi_down's bias and residual,
 * and C none of A, W_up, S_up.  The pair owns the workspace of both products
 * and of its barrier; calls on one pair must be ordered, as for a plan.  The
 * barrier's wait is bounded (about 2 s): if it runs out the kernel records
 * error bit 1 (q8mv_pair_check) and finishes with C undefined.
 */
enum {
    Q8MV_PAIR_AUTO = 0,
    Q8MV_PAIR_ONE_LAUNCH = 1,
    Q8MV_PAIR_TWO_LAUNCHES = 2
};

typedef struct q8mv_pair_s *q8mv_pair_t;

typedef struct {
    int32_t overlap;     /* 0 or 1: launches with programmatic dependent launch, as q8mv_opts_t */
    int32_t split_up;    /* K ranges per column tile of the up product; 0 = planner (at most 64) */
    int32_t split_down;  /* the same for the down product */
    int32_t cta_threads; /* 128 or 256; 0 = 256 */
    int32_t mode;        /* Q8MV_PAIR_* */
} q8mv_pair_opts_t;

typedef struct {
    int32_t one_launch;       /* 1: q8mv_pair_run launches the pair kernel (pointers allowing) */
    int32_t threads_per_cta;  /* the pair kernel's choices (0 when one_launch is 0) */
    int32_t grid;             /* CTAs: the larger product's tiles x split */
    int32_t ctas_per_sm;
    int32_t split_up, split_down;
    int32_t tiles_up, tiles_down;  /* 128-column tiles */
    int64_t workspace_bytes;
} q8mv_pair_info_t;

/* Plan a pair for K, N_mid, N_out on `device` (-1 = current); opts may be NULL. */
q8mv_status_t q8mv_pair_plan(q8mv_pair_t *out, int64_t K, int64_t N_mid, int64_t N_out, int device,
                             const q8mv_pair_opts_t *opts);

/* H = epi_up(A . W_up), then C = epi_down(H . W_down), asynchronously on
 * `stream`; epi_up and epi_down may be NULL (plain products). */
q8mv_status_t q8mv_pair_run(q8mv_pair_t pair, const float *A, const int8_t *W_up, const float *S_up, float *H,
                            const q8mv_epilogue_t *epi_up, const int8_t *W_down, const float *S_down, float *C,
                            const q8mv_epilogue_t *epi_down, cudaStream_t stream);

q8mv_status_t q8mv_pair_info(q8mv_pair_t pair, q8mv_pair_info_t *info);

/* As q8mv_check, for the pair kernel: bit 1 = its grid barrier's wait ran
 * out.  Clears the bits, and resets the pair's counters when any was set. */
q8mv_status_t q8mv_pair_check(q8mv_pair_t pair, int32_t *device_error);

/* For tests of the bounded wait only: the grid barrier's bound in
 * nanoseconds (0 restores about 2 s).  INVALID_ARG above 10 s. */
q8mv_status_t q8mv_pair_set_wait(q8mv_pair_t pair, uint64_t wait_ns);

/* Release the pair (synchronises its device first).  NULL is accepted. */
q8mv_status_t q8mv_pair_destroy(q8mv_pair_t pair);

/*
 * Host-only planning, no GPU needed: the one-launch configuration that
 * q8mv_pair_plan would pick (mode Q8MV_PAIR_ONE_LAUNCH) on a GPU with
 * `sm_count` SMs holding `ctas_per_sm` pair-kernel CTAs each.  Fills *info
 * (workspace_bytes: the split sums' partial rows and counters, without the
 * barrier words); INVALID_ARG if the shapes cannot use the pair kernel.
 */
q8mv_status_t q8mv_pair_choose_config(int64_t K, int64_t N_mid, int64_t N_out, int32_t sm_count,
                                      int32_t ctas_per_sm, const q8mv_pair_opts_t *opts,
                                      q8mv_pair_info_t *info);

/* The last CUDA runtime error code this library saw on the calling thread
 * (0 if none), for diagnosing Q8MV_ERR_CUDA. */
int q8mv_last_cuda_error(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int q8mv_version(void);

/*
 * Allocation-free matvec.  The pages have no counterpart to this call: it
 * exists only for callers that cannot allocate device memory and therefore
 * cannot own a plan.  Examples are an engine that reserves the GPU's memory for
 * its own pool at start-up (a cudaMalloc would fail, or bypass the pool's
 * accounting), code on a latency-critical path that must not call cudaMalloc
 * (it can synchronise the device and its latency is unbounded), and plug-in
 * hosts that let an extension enqueue work on a given stream but not create
 * resources.
 *
 * It computes exactly what q8mv_run computes with a default plan for (K, N)
 * on the current device: same kernel, same tile and split, same summation
 * order.  The split-K partial sums and counters live in one static device
 * array of Q8MV_NOALLOC_SCRATCH_BYTES bytes inside this library (2 MiB, held
 * by every GPU that loads the library until the process exits) instead of a
 * plan's workspace.
 *
 *   - Arguments, alignment and overlap rules are those of q8mv_run; the current
 *     device is used.
 *   - Returns Q8MV_ERR_SCRATCH_TOO_SMALL, before launching anything, when the
 *     split the planner picks needs more than that scratch: split_k * N floats
 *     of partial sums beyond the first 64 KiB, or more than 16384 column tiles
 *     of counters.  The 7B- and 70B-class projections and a 128256-row LM head
 *     all fit with aligned weights; 1-byte-aligned weights of 16 MiB or more
 *     can be refused.
 *   - The first call on each device looks up the scratch array's device
 *     address and the device's SM count and occupancy; make that first call
 *     before any stream capture begins on that device.  A first call that
 *     fails is not remembered: the next call repeats the set-up.  The address
 *     is kept for the life of the process, so cudaDeviceReset on a device
 *     after its first call here is not supported (later calls would use the
 *     old context's address).
 *   - No cudaMalloc, cudaFree or other allocating routine is called.  Each
 *     call clears the counters it uses with cudaMemsetAsync on `stream` before
 *     its kernel, so a call never depends on what an earlier call left behind.
 *   - All calls on a device share the one scratch array, and it keeps the last
 *     call's contents.  Calls whose kernels may overlap on the GPU (other
 *     streams, other host threads) race on it: order them, for example by
 *     issuing them on one stream.
 */
#define Q8MV_NOALLOC_SCRATCH_BYTES (2u * 1024u * 1024u)

q8mv_status_t q8mv_run_noalloc(int64_t K, int64_t N, const float *A, const int8_t *W,
                               const float *S, float *C, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* Q8MV_H */
