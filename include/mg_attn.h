/*
 * mg_attn.h -- C ABI of the fused exp-normalised GQA attention kernels for GB300 (sm_103a).
 *
 * Operation (Mirage documentation, tutorials/group-query-attention, "Define GQA
 * Computation Graph"; the same graph opens section 1 of the blog "Reading Mirage's
 * muGraph search and backend generation through the GQA example"):
 *
 *     A = matmul(Q, K); E = exp(A); S = reduction(E, 2); D = div(E, S); O = matmul(D, V)
 *
 * that is, for every batch b, query row m and column c,
 *
 *     O[b,m,c] = sum_n exp(A[b,m,n]) V[b,n,c] / sum_n exp(A[b,m,n]),
 *     A[b,m,n] = sum_k Q[b,m,k] K[b,k,n],
 *
 * with no max-subtraction and no 1/sqrt(d) scale, exactly as the graph is written.
 *
 * Tensors (all contiguous, row-major, IEEE fp16, device memory of the plan's device):
 *     Q (B, M, d)   query rows
 *     K (B, d, N)   keys, already transposed: d rows of N contiguous columns
 *     V (B, N, d)   values
 *     O (B, M, d)   output
 * The shape and stride metadata is fixed when the plan is made, like the graph's
 * input tensors, whose row-major strides are fixed when the graph is built (blog,
 * section 2).
 *
 * Arithmetic: A and P.V accumulate in fp32 on the tensor cores; exp and the row sums are
 * fp32; exp(A) is rounded to fp16 only as the operand of the second product; the final
 * divide is one IEEE fp32 division per element, then round-to-nearest-even to fp16.
 * Precondition: exp(A) must fit fp16, i.e. A <= ln(65504) ~ 11.09. Larger scores make the
 * fp16 graph itself overflow; the result is then inf/NaN and no error is reported. The opt-in
 * MG_FLAG_SAFE_SOFTMAX lifts it: each row's maximum score is subtracted before exp, which the
 * normalisation cancels, so the result is the same function with every fp16 weight <= 1.
 *
 * Status codes: the first four mirror the error enum of Mirage's CUDA transpiler
 * (blog, section 5.1: success, insufficient shared memory, layout error, config error).
 *
 * Threading: plans are independent objects. One plan must not run on two streams at
 * the same time (its split workspace is shared by its launches). No call prints,
 * aborts or exits the process.
 */
#ifndef MG_ATTN_H_
#define MG_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *mg_stream_t;

typedef struct mg_attn_plan *mg_attn_plan_t; /* opaque; owned by the library */

typedef enum {
    MG_OK = 0,
    MG_ERR_INSUFFICIENT_SMEM = 1, /* the tile configuration does not fit the device's shared memory */
    MG_ERR_LAYOUT = 2,            /* a pointer is not 16-byte aligned, or N % 8 != 0 */
    MG_ERR_CONFIG = 3,            /* an option is out of range (n_split, stages, timeout) */
    MG_ERR_INVALID_ARG = 4,       /* a dimension <= 0 or too large, a NULL pointer or NULL plan */
    MG_ERR_UNSUPPORTED = 5,       /* d not in {64, 128}, or the device is not compute capability 10.3 */
    MG_ERR_CUDA = 6,              /* a CUDA call failed; mg_attn_last_error() has the detail */
    MG_ERR_TIMEOUT = 7            /* a bounded in-kernel wait ran out (reported by mg_attn_get_status) */
} mg_status;

/* Flags for mg_attn_options.flags. */
#define MG_FLAG_NO_PDL 0x1         /* launch without programmatic dependent launch */
#define MG_FLAG_NO_CLUSTER 0x4     /* always combine split partials with the second kernel, never on chip */
#define MG_FLAG_SAFE_SOFTMAX 0x8   /* max-subtracted evaluation: P = exp(A - m) with m a per-row shift
                                      no smaller than the row's largest score minus 8, and the split
                                      partials combine with weights exp(m_j - max_j m_j). The result is
                                      the graph's (the normalisation cancels any per-row shift) without
                                      the A <= ln(65504) precondition. The one-tile kernel finds m (each
                                      row's largest score per split) in a first pass over K: Q.K computed
                                      twice and K read twice. The few-row specialisation (MG_FLAG_SWAP_AB)
                                      keeps m running in one pass: whenever a tile's score exceeds m by
                                      more than 8, m rises to the tile's maximum and the row's partial sum
                                      and O accumulator are scaled by exp(m_old - m_new). */
#define MG_FLAG_QK_NORM 0x10       /* QK-norm attention (Mirage documentation, tutorials/attention-with-kv-norm):
                                      Q = rms_norm(Q), K = rms_norm(K) before the graph, each query row and
                                      each key vector K[b,:,n] normalised over d: x / sqrt(mean(x^2) + eps),
                                      eps = MG_QKNORM_EPS, no weight. The fused kernel computes the scales
                                      1/rms in fp32 (a query row's from the Q tile it holds, a key vector's
                                      in the row-maximum pass from the K tile it streams, kept for the main
                                      pass in the CTA's shared memory where they fit beside the ring, head
                                      dim 64 with at most 33 column tiles per CTA, else in the plan's
                                      workspace) and applies them to the scores in fp32, so Q and K stay the
                                      fp16 MMA operands and K is read twice, as without the flag.
                                      Normalised scores reach +-d, past the fp16 range of exp, so
                                      the flag implies MG_FLAG_SAFE_SOFTMAX. Under the few-row
                                      specialisation (MG_FLAG_SWAP_AB) it runs in one pass (K read once):
                                      the key scales come from each K tile in shared memory. */
#define MG_QKNORM_EPS 1e-6
#define MG_FLAG_Q_PAIRS 0x20       /* use the two-Q-tile kernel wherever it applies (head dim 64, the graph as
                                      written, an even number of 128-row tiles per batch): each CTA holds
                                      two Q tiles of one batch, streams each K/V tile once for both, and
                                      each softmax warp group owns one tile's S, P and O. Opt-in: measured
                                      on GB300 it is slower than the default one-tile kernel (see
                                      info.q_tiles_per_cta) */
#define MG_FLAG_NO_Q_PAIRS 0x40    /* always use the one-tile kernel (the default) */
#define MG_FLAG_STREAM_K 0x80      /* use the stream-K schedule where it applies (the graph as written, at
                                      most 16 query rows per batch, no explicit n_split, runs of at most
                                      ceil(N/128) units, and no more tiles for the busiest CTA than the split
                                      schedule gives): the B x ceil(N/128) (batch, column tile) units form one
                                      sequence that the grid's CTAs share in equal contiguous runs, one CTA
                                      per SM; each run's part of a batch is a partial that the second kernel
                                      sums in a fixed order. Opt-in: measured on GB300 it is not faster than
                                      the default split schedule on the decode shapes; see info.schedule */
#define MG_FLAG_NO_STREAM_K 0x100  /* the split schedule (N split n_split ways per row tile; the default) */
#define MG_FLAG_SWAP_AB 0x200      /* few-row specialisation (the graph as written, or its max-subtracted
                                      or QK-norm evaluation in one pass; head dim 128, at most 16
                                      query rows per batch, the split schedule): per K/V tile the products run
                                      transposed, S^T = K^T Q^T and O^T += V^T P^T, so the MMA's 128 rows are
                                      keys (resp. output columns) instead of mostly-empty query rows; split
                                      partials combine on chip (fp32) when the cluster fits, else in the
                                      second kernel. The default where it applies
                                      (this flag only states it); see info.swap_ab */
#define MG_FLAG_NO_SWAP_AB 0x400   /* never use the few-row specialisation (the one-tile kernel instead) */
#define MG_FLAG_PUSH_COMBINE 0x800 /* on-chip combine, pushed form (the graph as written, head dim 64): each
                                      thread stores its row's values into the row owner's receive area as
                                      soon as it has formed them (asynchronous stores counted on the owner's
                                      barrier; one pipeline stage fewer), instead of the owners reading them
                                      out of every CTA's shared memory after a cluster barrier (the default,
                                      pulled form). Opt-in: measured on GB300 it is slower; see info.xchg_push */
#define MG_FLAG_ISOLATED 0x2000     /* plan for calls that do not overlap (each between kernels of other
                                      work, or after a call whose output it reads): keep the split count
                                      chosen for one call's latency instead of lowering it so that several
                                      back-to-back calls fit the device at once (see mg_attn_query) */
#define MG_FLAG_NO_EARLY_LOADS 0x1000 /* the fused kernel reads nothing before the previous kernel on the
                                      stream has completed and releases the next one only after that (see
                                      mg_attn_run: by default it may read Q, K and V earlier, and start the
                                      next call early, when no recent call of this library wrote them) */
#define MG_FLAG_INJECT_TIMEOUT 0x2 /* test hook: before issuing any copy, the load warp waits on a
                                      barrier nothing arrives on, so the bounded-wait path runs and
                                      the plan's status becomes MG_ERR_TIMEOUT; O is then undefined */

typedef struct {
    int32_t n_split;    /* CTAs sharing one 128-row tile along N; 0 = automatic. 1 <= n_split <= ceil(N/128).
                           2..16 splits combine on chip in a thread-block cluster when the device can
                           schedule the cluster (unless MG_FLAG_NO_CLUSTER); more use the second kernel */
    int32_t stages;     /* K/V shared-memory pipeline depth; 0 = automatic (the deepest); 2..6 (d = 128: 2..3) */
    int32_t flags;      /* MG_FLAG_* bits */
    int32_t reserved;   /* must be 0 */
    int64_t timeout_ns; /* bound on every in-kernel wait; 0 = 1 second; otherwise 1e3 .. 6e10 */
} mg_attn_options;

typedef struct {
    int64_t B, M, N, d;
    int32_t block_m;         /* rows of Q per CTA tile (128) */
    int32_t block_n;         /* columns of K per pipeline step (128) */
    int32_t m_tiles;         /* B * ceil(M / block_m) */
    int32_t n_tiles;         /* ceil(N / block_n) */
    int32_t n_split;         /* CTAs per row tile; CTA j takes the column tiles j, j + n_split, ... */
    int32_t stages;          /* K/V pipeline depth */
    int32_t threads;         /* threads per CTA of the fused kernel */
    int32_t grid_ctas;       /* m_tiles / q_tiles_per_cta * n_split */
    int32_t smem_bytes;      /* dynamic shared memory per CTA of the fused kernel */
    int32_t tmem_cols;       /* tensor-memory columns allocated per CTA */
    int32_t kernels_per_run; /* 1 when the fused kernel writes O itself (n_split == 1 or cluster_ctas > 0), else 2 */
    int32_t num_sms;         /* streaming multiprocessors the plan was sized for */
    int64_t workspace_bytes; /* device bytes owned by the plan (split partials + status words) */
    int32_t cluster_ctas;    /* > 0: the n_split CTAs of a row tile (or row-tile pair) run as one
                                thread-block cluster and combine their partials themselves after
                                one cluster barrier (no second kernel); 0: second kernel */
    int32_t q_tiles_per_cta; /* 128-row Q tiles per CTA: 1 (one-tile kernel) or 2 (two-Q-tile
                                kernel; m_tiles / 2 row-tile pairs, each split n_split ways) */
    int32_t schedule;        /* 0: split (CTA j of a row tile takes column tiles j, j + n_split, ...);
                                1: stream-K (grid_ctas CTAs share the m_tiles x n_tiles units in equal
                                contiguous runs; n_split is then the second kernel's partials per row) */
    int32_t swap_ab;         /* 1: the few-row specialisation (transposed products, MG_FLAG_SWAP_AB) */
    int32_t xchg_push;       /* with cluster_ctas > 0: 1 when the CTAs push each owner's rows into its
                                receive area (MG_FLAG_PUSH_COMBINE), 0 when the owners pull them */
} mg_attn_plan_info;

/*
 * Make a plan for one problem shape on the current CUDA device. This is the step the pages take
 * before a graph's first launch: the optimized graph is transpiled and compiled for its fixed
 * input shapes (documentation, tutorials/group-query-attention, "Launch Mirage-Generated GQA
 * Kernel"; blog, section 5: compile and profile after the search). Validates the shape,
 * chooses the tiling and the N split from the device's SM count, and allocates the
 * plan's device workspace (fp32 partial numerators n_split*B*M*d and row sums
 * n_split*B*M, plus two status words). Synchronous. On success *out owns the plan.
 * Errors: MG_ERR_INVALID_ARG (dims <= 0, B*M*d or d*N beyond 2^31, out == NULL),
 * MG_ERR_UNSUPPORTED (d not 64/128, device not cc 10.3), MG_ERR_LAYOUT (N % 8 != 0),
 * MG_ERR_INSUFFICIENT_SMEM, MG_ERR_CUDA (no device, allocation failed).
 */
mg_status mg_attn_plan(int64_t B, int64_t M, int64_t N, int64_t d, mg_attn_plan_t *out);

/* As mg_attn_plan, with explicit options (NULL = defaults). Adds MG_ERR_CONFIG. */
mg_status mg_attn_plan_ex(int64_t B, int64_t M, int64_t N, int64_t d,
                          const mg_attn_options *opts, mg_attn_plan_t *out);

/*
 * Enqueue O = attention(Q, K, V) on `stream`. Restates the generated host entry point of the
 * CUDA transpiler, _execute_mugraph(input_tensors, output_tensors, buf) (documentation,
 * cuda-transpiler, "Generated CUDA Code Example"), called as optimized_graph(input_tensors) in
 * the GQA tutorial ("Launch Mirage-Generated GQA Kernel"): the inputs are (Q, K, V) and the
 * output O, as device pointers; the scratch buffer `buf` is the plan's workspace, so it is not an
 * argument here. Asynchronous and stream-ordered: no
 * synchronisation, no allocation. Q, K, V, O are device pointers with the plan's shape
 * (see the top of this file), 16-byte aligned; O must not overlap the inputs. The caller
 * keeps ownership of all four. With programmatic dependent launch (the default) the
 * kernels wait for all prior work on `stream` before writing global memory. The fused kernel
 * may read Q, K and V before the kernels before it on the stream have completed, when the
 * library knows them: the previous call on the same stream (and the same stream capture) was
 * one of this library's, and none of Q, K and V shares bytes with the outputs of the last 16
 * calls on that stream or with O. Then, for grids of more than SMs / 16 CTAs (10 on a 152-SM
 * GB300: fewer than 16 such grids fit the device at once, one CTA per SM), it also releases the
 * next kernel at its start and computes everything before its wait (back-to-back calls
 * overlap); otherwise only its first copies go out early. A kernel of another origin that runs
 * right before the call and releases its dependents before it completes (programmatic
 * dependent launch) must not write Q, K or V, nor may calls on one stream be enqueued from
 * several host threads at once; MG_FLAG_NO_EARLY_LOADS turns the early reads off.
 * Errors: MG_ERR_INVALID_ARG (NULL plan or pointer), MG_ERR_LAYOUT (misaligned pointer),
 * MG_ERR_CUDA (descriptor encoding or launch failed; the plan's device must be current).
 * In-kernel timeouts are not visible here; see mg_attn_get_status.
 */
mg_status mg_attn_run(mg_attn_plan_t plan, const void *Q, const void *K, const void *V,
                      void *O, mg_stream_t stream);

/*
 * End-to-end variant for host buffers: copies Q, K, V from host memory into device
 * buffers owned by the plan, runs as mg_attn_run, and copies O back into host memory,
 * all enqueued on `stream`; the caller synchronises the stream before reading hO.
 * Page-locked host buffers that the device can address (cudaHostAlloc / pinned tensors,
 * 16-byte aligned) are read by a copy kernel through their device addresses, chained to the
 * attention kernels with programmatic dependent launch. That kernel loads the inputs as soon as
 * it starts, which can be while the previous kernel on `stream` still runs (this library's
 * kernels release their dependents early), and stores them into the staging only after that
 * kernel ends. So the inputs must hold their final values when the call is made, and no kernel
 * enqueued before it may write them, except as the output of an earlier call of this library on
 * the same stream (O of mg_attn_run or mg_attn_run_noalloc, hO of mg_attn_run_host): when an
 * input shares bytes with the previous call's output on that stream, or with this call's hO, the
 * loads wait for the previous kernel. When the plan splits N
 * (info.n_split > 1) the kernels write O straight into such a host buffer, and otherwise a
 * second copy kernel writes it back. Other host memory (pageable) goes through cudaMemcpyAsync. The plan's device staging buffers (the size of
 * Q, K, V and O) are allocated by the first call on that plan and reused after, so one
 * plan must not run two such calls at once on different streams.
 * Errors: as mg_attn_run, plus MG_ERR_CUDA if the staging allocation fails.
 */
mg_status mg_attn_run_host(mg_attn_plan_t plan, const void *hQ, const void *hK, const void *hV,
                           void *hO, mg_stream_t stream);

/*
 * Allocation-free variant of mg_attn_run, for callers that cannot call cudaMalloc: code that has
 * handed all device memory to another allocator (a framework's caching pool), code on a latency
 * path where cudaMalloc's implicit device synchronisation is not acceptable, and code under rules
 * that forbid dynamic allocation after start-up. (The pages have no counterpart: Mirage's
 * generated entry takes a caller-allocated buffer instead.)
 *
 * Same operation, tensors, tiling and kernels as a default plan for (B, M, N, d) run with
 * mg_attn_run, so the results are the same. No plan is needed and nothing is allocated: the
 * split partials and status words live in a file-scope device array of 8 MiB
 * (MG_ATTN_STATIC_SCRATCH_BYTES) that every GPU loading this library holds until the process
 * exits. Shapes whose split partials need more than that (e.g. d = 128 with a long N and few
 * row tiles) are rejected with MG_ERR_INVALID_ARG and a message from mg_attn_last_error().
 *
 * The first call on each device (with that device current) does a one-time set-up: it looks up
 * the array's device address and clears its status words. Make that first call before any
 * stream capture. Every call shares the one array and it keeps the last call's contents, so
 * calls that overlap on the GPU (other streams, other host threads) race: serialise them.
 * In-kernel timeouts are recorded in the array's status words and not reported.
 * Errors: as mg_attn_run and mg_attn_plan (shape validation, device checks).
 */
#define MG_ATTN_STATIC_SCRATCH_BYTES (8u << 20)
mg_status mg_attn_run_noalloc(int64_t B, int64_t M, int64_t N, int64_t d, const void *Q, const void *K,
                              const void *V, void *O, mg_stream_t stream);

/*
 * Synchronise the device, then free the plan's workspace (the scratch buffer `buf` that the
 * generated entry point takes from its caller: documentation, cuda-transpiler, "Generated CUDA
 * Code Example"), its host staging and the plan. NULL is MG_ERR_INVALID_ARG; MG_ERR_CUDA if the
 * synchronisation reports an error (the memory is freed all the same).
 */
mg_status mg_attn_destroy(mg_attn_plan_t plan);

/*
 * Sticky device-side status of the plan, reported in the codes above, whose first four restate
 * the CUDA transpiler's error enum (blog, section 5.1: CUDA_T_SUCCESS, CUDA_T_INSUFFICIENT_SMEM,
 * CUDA_T_LAYOUT_ERROR, CUDA_T_CONFIG_ERROR); the pages have no in-kernel timeout, so
 * MG_ERR_TIMEOUT is this library's. MG_OK, or MG_ERR_TIMEOUT once any in-kernel wait
 * of any run of this plan ran out (the kernels then stop early and O is undefined).
 * Synchronises the device to read it. MG_ERR_CUDA if the read itself fails.
 */
mg_status mg_attn_get_status(mg_attn_plan_t plan);

/*
 * Measurement hook. When both events are non-NULL, every later mg_attn_run / mg_attn_run_host
 * on this plan records ev_begin on its stream just before the fused kernel's launch and ev_end
 * just after it (before the combine kernel), so that cudaEventElapsedTime(ev_begin, ev_end)
 * times the fused kernel alone. The events are cudaEvent_t handles owned by the caller, who
 * keeps them alive while the hook is set; NULL, NULL removes it. A recorded event between two
 * launches suspends the programmatic-launch overlap of those two kernels, so leave the hook
 * off for throughput runs. Errors: MG_ERR_INVALID_ARG for a NULL plan or exactly one NULL event.
 */
mg_status mg_attn_set_timing_events(mg_attn_plan_t plan, void *ev_begin, void *ev_end);

/* Copy the plan's decisions into *info. */
mg_status mg_attn_get_info(mg_attn_plan_t plan, mg_attn_plan_info *info);

/*
 * Host-only: the decisions mg_attn_plan_ex would take for this shape on a device with
 * `num_sms` SMs and `max_smem_optin` bytes of opt-in shared memory per block, without
 * touching any GPU. Same validation and error codes as mg_attn_plan_ex (minus device errors).
 * The one decision it cannot take is the placement of the on-chip combine's clusters, which
 * mg_attn_plan_ex asks the device about: how many clusters of the chosen size it holds at once.
 * Without an explicit n_split (and without MG_FLAG_ISOLATED for the second step) the plan then
 * takes a smaller cluster when that lets the clusters
 * of two back-to-back calls be resident together (at most one more column tile per CTA), or
 * when the chosen clusters do not fit at all (at most two more), and otherwise falls back to
 * the second kernel;
 * the one-tile kernel's two-pass variants keep the chosen cluster whenever it fits.
 */
mg_status mg_attn_query(int64_t B, int64_t M, int64_t N, int64_t d, const mg_attn_options *opts,
                        int32_t num_sms, int32_t max_smem_optin, mg_attn_plan_info *info);

/* Static English text for a status code (never NULL). */
const char *mg_attn_status_string(mg_status s);

/* Detail of the last failure on the calling thread (e.g. the CUDA error name); "" if none. */
const char *mg_attn_last_error(void);

/* ABI version: major * 10000 + minor * 100 + patch. */
int32_t mg_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MG_ATTN_H_ */
