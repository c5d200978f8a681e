/*
 * sgp.h -- C ABI of the intra-GPU spatial-pipelining decode-layer library (libsgp.so).
 *
 * One LLM decode layer (MoE transformer, GPT-OSS-120B-shaped per-GPU slice) runs either
 *   - temporally: every kernel back to back on the whole GPU, one full-batch microbatch
 *     ("SubGPU Pipelining: Intra-GPU Fine-Grained Spatial Parallelism for LLM Inference",
 *     Section 5.1, the "Temporal" baseline), or
 *   - as a spatial pipeline: the layer's operator chain is cut into contiguous segments,
 *     the segments are bound to stages backed by disjoint SM pools, and microbatches stream
 *     through the stages (same paper, Section 3.1, Eq. 1-3; Section 3.2 for the task DAG).
 *
 * Operator chain of one layer (same paper, Fig. 3), with the op indices used by the cut:
 *   0 SGP_OP_RMSNORM_ATTN  a = RMSNorm(x; g_attn)
 *   1 SGP_OP_QKV           [q | k | v] = a W_qkv^T; k, v written to cache slot kv_len-1
 *   2 SGP_OP_ATTENTION     GQA decode attention over cache positions [lo, kv_len)
 *   3 SGP_OP_OPROJ         h = x + o W_o^T
 *   4 SGP_OP_ROUTER        u = RMSNorm(h; g_mlp); z = u W_r^T (+ bias); top-k; softmax over k
 *   5 SGP_OP_DISPATCH      group the (token, pick) pairs by local expert slot
 *   6 SGP_OP_EXPERT_UP     z_r = silu(u W_gate^T) * (u W_up^T) per routed row (SwiGLU)
 *   7 SGP_OP_EXPERT_DOWN   y_r = z_r W_down^T
 *   8 SGP_OP_COMBINE       x_next = h + sum_j w_j y_(t,j)
 * Stage A of the default two-stage cut is ops 0-2, stage B is ops 3-8.
 *
 * Conventions for every entry point:
 *   - Pointers named "device" are CUDA device pointers; the caller owns all of them
 *     (weights, KV cache, activations, outputs, workspace).  The library owns only the
 *     sgp_pipeline handle and what it allocates inside it.
 *   - bf16 tensors are IEEE bfloat16, row-major, innermost dimension contiguous.  Device
 *     pointers must be 16-byte aligned (SGP_ERR_INVALID_ARG otherwise).
 *   - Calls are asynchronous on the given stream (a cudaStream_t; NULL = legacy default
 *     stream) unless stated.  Argument errors are returned at once and nothing is launched.
 *     Errors detected on the device (a bounded wait that ran out, a failed handoff check,
 *     an out-of-range index) are recorded in a device status word and returned by
 *     sgp_status_from_workspace / sgp_pipeline_sync.  Nothing aborts, traps or throws.
 *   - Results do not depend on the number of SMs used or on the microbatch size: every
 *     reduction has a fixed order, so temporal and pipelined outputs are bit-identical.
 */
#ifndef SGP_H
#define SGP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* sgp_stream_t; /* same type as cudaStream_t */

/* ---- status codes -------------------------------------------------------------------- */
enum {
    SGP_OK = 0,
    SGP_ERR_INVALID_ARG = -1,   /* shape, alignment, split or microbatch not supported   */
    SGP_ERR_UNSUPPORTED = -2,   /* device is not sm_103 / no green contexts              */
    SGP_ERR_CUDA = -3,          /* a CUDA runtime/driver call failed (see sgp_last_error) */
    SGP_ERR_TIMEOUT = -4,       /* a device-side bounded wait ran out                    */
    SGP_ERR_OOM = -5,           /* the library could not allocate its own state          */
    SGP_ERR_HANDOFF = -6,       /* a stage task started before its producer published    */
    SGP_ERR_DEVICE_BOUNDS = -7  /* a kernel saw an index outside its buffers and skipped it */
};

/* ---- operator indices (see the table above) ----------------------------------------- */
enum {
    SGP_OP_RMSNORM_ATTN = 0, SGP_OP_QKV = 1, SGP_OP_ATTENTION = 2, SGP_OP_OPROJ = 3,
    SGP_OP_ROUTER = 4, SGP_OP_DISPATCH = 5, SGP_OP_EXPERT_UP = 6, SGP_OP_EXPERT_DOWN = 7,
    SGP_OP_COMBINE = 8, SGP_N_OPS = 9
};

/* ---- projection path policy (static: never chosen per microbatch) ------------------ */
enum {
    SGP_PATH_AUTO = 0,  /* tensor cores (tcgen05) when the full batch gives >= gemv_max_tokens
                           rows per weight matrix, else the CUDA-core GEMV                     */
    SGP_PATH_GEMV = 1,  /* always the vectorised CUDA-core GEMV                                 */
    SGP_PATH_TC = 2     /* always the tcgen05 tensor-core GEMM                                  */
};

/* Layer dimensions.  Up to 512 sequences per call.  Supported: head_dim == 64; hidden, inter
 * and n_q_heads*head_dim multiples of 64; hidden <= 4096 (the router keeps rows of H in shared
 * memory); n_q_heads a multiple of n_kv_heads with n_q_heads/n_kv_heads <= 16; top_k <= 8;
 * n_experts <= 1024; n_local_experts <= n_experts. */
typedef struct sgp_dims {
    int hidden;           /* H                                                       */
    int n_q_heads;        /* query heads                                             */
    int n_kv_heads;       /* KV heads; query head h reads KV head h / (n_q/n_kv)      */
    int head_dim;         /* d (64)                                                  */
    int n_experts;        /* E: router width (global experts)                        */
    int top_k;            /* k experts per token                                     */
    int n_local_experts;  /* E_local: expert weight slots held on this GPU           */
    int inter;            /* I: SwiGLU intermediate size                             */
    float rms_eps;        /* RMSNorm epsilon (1e-5)                                  */
    int slot_map;         /* 0: global expert g -> slot g % E_local;
                             1: g -> g * E_local / E (expert-parallel loopback)      */
    int path;             /* SGP_PATH_*                                              */
    int gemv_max_tokens;  /* threshold of SGP_PATH_AUTO; 2 is measured best for
                             temporal execution on GB300 (36 layers: the GEMV wins
                             at 1 sequence, the tcgen05 GEMM from 2 on)             */
    float rope_theta;     /* RoPE base for q and the new key at position kv_len-1
                             (half-split pairs i, i + d/2); 0 = no rotation.  Needs the
                             tensor-core QKV path (SGP_ERR_UNSUPPORTED otherwise)      */
    /* Virtual communication of a multi-GPU deployment emulated on this GPU ("SubGPU
     * Pipelining: Intra-GPU Fine-Grained Spatial Parallelism for LLM Inference", Section
     * 5.3): when both are > 0, every layer and microbatch runs three loopback kernels that
     * copy the payload of the attention all-reduce (after the output projection, b*H bf16),
     * the MoE dispatch (after the dispatch, b*k*H bf16) and the MoE combine (before the
     * combine, b*k*H bf16) into workspace scratch and last at least
     * comm_floor_us + payload / comm_gbps.  Results are unchanged.  0, 0 = off.        */
    float comm_floor_us;
    float comm_gbps;
} sgp_dims;

/* One layer's weights and KV cache (all device pointers, caller-owned).
 *   g_attn, g_mlp  bf16 [H]
 *   w_qkv          bf16 [(n_q + 2 n_kv) d][H]   rows: q heads, then k heads, then v heads
 *   w_o            bf16 [H][n_q d]
 *   w_router       bf16 [E][H]
 *   router_bias    fp32 [E] or NULL
 *   w_gate_up      bf16 [E_local][2 I][H]       per slot: I gate rows, then I up rows
 *   w_down         bf16 [E_local][H][I]
 *   k_cache,v_cache bf16 [n_tokens][n_kv][kv_cap][d]; written in place at kv_len[b]-1.
 * window: 0 = full attention over [0, L); W > 0 = sliding window over [max(0, L-W), L). */
typedef struct sgp_layer {
    const void* g_attn;
    const void* w_qkv;
    const void* w_o;
    const void* g_mlp;
    const void* w_router;
    const float* router_bias;
    const void* w_gate_up;
    const void* w_down;
    void* k_cache;
    void* v_cache;
    int kv_cap;
    int window;
} sgp_layer;

/* Optional copies of one layer's intermediates (device pointers, NULL = skip), written by
 * sgp_layer_temporal for tests.  Row r of a routed tensor is the r-th (token, pick) pair in
 * slot order; pair_pos[t*k + j] gives the row of pick j of token t.
 *   a,u,h bf16 [T][H]; q,o bf16 [T][n_q d]; logits fp32 [T][E];
 *   slot_offsets int32 [E_local+1]; pair_pos int32 [T k]; z bf16 [T k][I]; y fp32 [T k][H] */
typedef struct sgp_layer_dump {
    void* a;
    void* q;
    void* o;
    void* h;
    void* u;
    float* logits;
    int32_t* slot_offsets;
    int32_t* pair_pos;
    void* z;
    float* y;
} sgp_layer_dump;

/* ---- device and library info --------------------------------------------------------- */
typedef struct sgp_device_info {
    int sm_count;              /* streaming multiprocessors of the current device        */
    int cc_major, cc_minor;
    int green_ctx_supported;   /* 1 if SM-partitioned green contexts can be created       */
    int sm_min_partition;      /* smallest legal SM pool                                  */
    int sm_alignment;          /* pools are multiples of this many SMs                     */
    size_t l2_bytes;
} sgp_device_info;

/* Fills *info for the current device.  Synchronous, launches nothing.
 * Returns SGP_OK, SGP_ERR_INVALID_ARG (info NULL) or SGP_ERR_CUDA. */
int sgp_device_info_get(sgp_device_info* info);

/* Text of a status code.  Never NULL; static storage. */
const char* sgp_status_string(int status);

/* Text of the last CUDA error this library saw in this thread (static/thread storage). */
const char* sgp_last_error(void);

/* ---- temporal execution (Section 5.1 "Temporal" baseline) --------------------------- */

/* Bytes of workspace sgp_layer_temporal / sgp_stack_temporal need for n_tokens sequences
 * whose KV length never exceeds max_kv_len.  Returns 0 on invalid arguments. */
size_t sgp_workspace_bytes(const sgp_dims* dims, int n_tokens, int max_kv_len);

/* One decode layer, every kernel on the whole GPU, in stream order.
 *   kv_len    device int32 [n_tokens], 1 <= kv_len[b] <= layer->kv_cap, counts the current token
 *   x_in      device bf16 [n_tokens][H];  x_out device bf16 [n_tokens][H] (may equal x_in)
 *   topk_idx  device int32 [n_tokens][k] or NULL; topk_w device fp32 [n_tokens][k] or NULL
 *             (picks in descending-logit order, ties to the lower expert index)
 *   workspace device, >= sgp_workspace_bytes(dims, n_tokens, kv_cap) bytes, 256-byte
 *             aligned, not shared with a call that may run concurrently
 *   dump      NULL or intermediates to copy out (tests)
 * The first call with a given workspace clears its status word and counters; later calls
 * keep the status sticky until sgp_status_from_workspace reads and clears it.
 * Returns SGP_OK, SGP_ERR_INVALID_ARG or SGP_ERR_CUDA (launch failure). */
int sgp_layer_temporal(const sgp_dims* dims, const sgp_layer* layer, const int32_t* kv_len,
                       const void* x_in, void* x_out, int n_tokens, int32_t* topk_idx,
                       float* topk_w, void* workspace, size_t ws_bytes,
                       const sgp_layer_dump* dump, sgp_stream_t stream);

/* n_layers layers back to back (layer l's output feeds layer l+1), temporally.
 *   layers    host array [n_layers]; topk_idx/topk_w NULL or device [n_layers][n_tokens][k]
 * Other arguments as sgp_layer_temporal. */
int sgp_stack_temporal(const sgp_dims* dims, const sgp_layer* layers, int n_layers,
                       const int32_t* kv_len, const void* x_in, void* x_out, int n_tokens,
                       int32_t* topk_idx, float* topk_w, void* workspace, size_t ws_bytes,
                       sgp_stream_t stream);

/* Launches op `op` (SGP_OP_*) of one temporal layer alone, on `stream`.  Its inputs are what
 * `workspace` holds from an earlier sgp_layer_temporal with the same arguments (for example
 * the normalised activations of op 0), so a sequence of ops 0..8 equals one
 * sgp_layer_temporal call.  Used to time and profile single kernels.  The zeroed counters
 * of the workspace must hold zero, as every kernel leaves them.  Arguments and returns as
 * sgp_layer_temporal. */
int sgp_layer_op(const sgp_dims* dims, const sgp_layer* layer, int op, const int32_t* kv_len,
                 const void* x_in, void* x_out, int n_tokens, void* workspace, size_t ws_bytes,
                 sgp_stream_t stream);

/* Synchronises `stream`, returns the device status recorded in `workspace` since the last
 * read (SGP_OK, SGP_ERR_TIMEOUT, SGP_ERR_HANDOFF, SGP_ERR_DEVICE_BOUNDS) and clears it.
 * Returns SGP_ERR_CUDA if the copy fails. */
int sgp_status_from_workspace(const void* workspace, sgp_stream_t stream);

/* ---- router without device allocation ----------------------------------------------
 * Some callers cannot call cudaMalloc at all: code that runs while a CUDA graph is being
 * captured, or inside an engine whose memory pool owns every byte of the device, or a
 * plugin that is handed only its inputs and outputs.  This entry point serves them: it is
 * the router of op SGP_OP_ROUTER (RMSNorm of h, fp32 logits, top-k, softmax over the k
 * selected logits) for one layer, and it allocates nothing.  The paper has no counterpart;
 * it is an interface convenience.
 *
 * Its scratch (fp32 logits and arrival counters) is a fixed array inside the library: at most
 * 262,144 logits, i.e. n_tokens * n_experts <= 262144 (for example 256 tokens x 1024 experts),
 * about 1 MiB, which every GPU that loads the library keeps until the process exits.  The
 * first call on a device does a one-time set-up with that device current: it looks up the
 * array's device address and prepares both router kernel variants (their shared-memory
 * limit), and it caches both; make that first call before any stream capture.  Every call
 * shares the array: the counters are cleared on `stream` at the start of each call, the
 * logits keep the last call's values, and calls that overlap on the GPU (two streams, or two
 * host threads) race -- serialise them.
 *
 *   h          device bf16 [n_tokens][H]   residual stream after the attention block
 *   g_mlp      device bf16 [H];  w_router device bf16 [E][H];  router_bias device fp32 [E] or NULL
 *   u_out      device bf16 [n_tokens][H]   RMSNorm(h; g_mlp), as the layer computes it
 *   topk_idx   device int32 [n_tokens][k]; topk_w device fp32 [n_tokens][k]
 * Results equal those sgp_layer_temporal produces for the same h.  Returns SGP_OK,
 * SGP_ERR_INVALID_ARG (NULL or unaligned pointer, unsupported dims (hidden above 4096
 * included), or a size beyond the fixed scratch; nothing is launched) or SGP_ERR_CUDA.  The
 * return code is the whole error report: the router kernel has no device-side error path (it
 * waits on nothing and indexes only within the sizes checked here), so no status is deferred
 * to the device. */
int sgp_router_topk_noalloc(const sgp_dims* dims, const void* h, const void* g_mlp,
                            const void* w_router, const float* router_bias, int n_tokens,
                            void* u_out, int32_t* topk_idx, float* topk_w, sgp_stream_t stream);

/* ---- spatial pipeline (Section 3: cut, binding, SM allocation, microbatches) -------- */
typedef struct sgp_pipeline sgp_pipeline;

/* Options of a pipeline; zero-initialise, then set what differs from the defaults. */
typedef struct sgp_pipeline_opts {
    /* Stage of every op, for full-attention layers [0][op] and sliding-window layers [1][op],
     * used when custom_cut != 0.  Consecutive ops of one microbatch on the same stage form
     * one task (a segment instance); any assignment is legal, including a last segment that
     * shares stage 0 with the first (boundary reuse, Eq. 1 with w = 1).
     * Default (custom_cut == 0): 2 stages -> ops 0-2 | 3-8; 3 stages -> 0-2 | 3-4 | 5-8;
     * 1 stage -> everything on one pool (temporal). */
    int custom_cut;
    int stage_of_op[2][SGP_N_OPS];
    int use_green_contexts;     /* 0 = default (on for n_stages >= 2), -1 = off: all stages
                                   share every SM (streams only; no partition guarantee)   */
    int green_ctx_flags;        /* passed to the SM split (1 = ignore SM co-scheduling)      */
    int serpentine_experts;     /* 1: odd microbatches walk expert slots in reverse order   */
    uint64_t wait_timeout_ns;   /* device bounded-wait limit (0 = 2 s)                     */
    uint32_t fault_inject;      /* TEST ONLY: bit 0 = drop the handoff flag of the first
                                   task; bit 1 = drop one TMA load of the first projection
                                   (its bounded wait then runs out)                          */
    int fault_task;             /* task index for fault bit 0                                */
    int programmatic_launch;    /* programmatic dependent launch between consecutive kernels
                                   of a task (a kernel's launch and prologue overlap the
                                   previous kernel's tail; results are identical):
                                   0 = default: only into the kernels whose prologue does
                                   not read the predecessor's output: the projection
                                   kernels and their finishing passes (the weight stream
                                   starts early) and the attention (it builds its chunk
                                   table from kv_len first);
                                   1 = into every kernel; -1 = off                            */
    int trace;                  /* 1: every kernel records its first-CTA start and last-CTA
                                   end (%globaltimer ns); read with sgp_pipeline_trace      */
    int weight_reuse;           /* 1: projection weights read by a microbatch that is not the
                                   last are loaded with an L2 evict-last hint (the next
                                   microbatch rereads them), the last microbatch's with
                                   evict-first; 0 = default (off: every weight load is
                                   evict-first; the hint measured no faster here)           */
    int l2_prefetch_mb;         /* L2 prefetch of the next projection's weights, issued beside
                                   the chain (a prefetch kernel that no launch waits for) once
                                   a projection's main kernel completes, so that HBM moves
                                   them while the kernels in between leave it idle: QKV ->
                                   output projection, output projection -> expert gate/up,
                                   expert gate/up -> expert down, expert down -> the next
                                   layer's QKV.  Dense matrices are prefetched whole, expert
                                   matrices up to this many MB; 0 = default (off: measured
                                   slower on the 36-layer slice).  Only timing changes;
                                   results are bit-identical                                  */
    int stage_lanes;            /* FIFOs per stage: 0 or 1 = default, one (every task of a stage
                                   waits for the task before it on that stage, Section 3.2);
                                   2 = one per microbatch parity, i.e. two streams per SM pool
                                   (the pages' prototype runs two stream rows per green
                                   context, Section 5.3): tasks of the other parity may run
                                   beside them on the same SMs.  Results are identical        */
    int stage_times_shared;     /* sgp_pipeline_stage_times and the balancer: 0 = default, each
                                   stage timed alone on the GPU; 1 = all stages replay their
                                   tasks at the same time, so each is timed while the others
                                   share HBM and L2 with it (the contention a pipelined run
                                   sees)                                                      */
} sgp_pipeline_opts;

/* Creates a pipeline for up to max_tokens sequences with KV length <= max_kv_len.
 *   sm_split   host int[n_stages]: SMs per stage, sum <= SM count, each a multiple of the
 *              green-context alignment (sgp_device_info_get); ignored for n_stages == 1
 *   n_stages   1 (temporal on all SMs), 2 or 3
 *   microbatch sequences per microbatch b; must divide the n_tokens of every run
 *   opts       NULL for defaults
 * Allocates the handle, its device state (status word, flags, per-microbatch scratch) and,
 * for n_stages >= 2, one green context and stream per stage.
 * Returns SGP_OK, SGP_ERR_INVALID_ARG, SGP_ERR_UNSUPPORTED, SGP_ERR_OOM or SGP_ERR_CUDA. */
int sgp_pipeline_create(const sgp_dims* dims, const int* sm_split, int n_stages,
                        int microbatch, int max_tokens, int max_kv_len,
                        const sgp_pipeline_opts* opts, sgp_pipeline** out);

/* Runs n_layers layers over n_tokens sequences as the pipeline's task DAG: task (l, mu, s)
 * waits for its data predecessor (the previous segment of microbatch mu) and for the task
 * before it on stage s in the global dispatch order (Section 3.2).  The DAG is a CUDA graph
 * (built on the first run with these arguments, then replayed); it starts after the work
 * already queued on `stream` and `stream` waits for it.  Runs of one pipeline may use
 * different streams: each run is also ordered after the pipeline's previous run (an event
 * wait), since they share its flags and scratch.  The call does not wait for the GPU and
 * makes no host round trip inside a run; only a call whose arguments differ from the
 * previous run's (a graph rebuild, which may reallocate the scratch) first waits for the
 * previous run to complete.
 * Arguments as sgp_stack_temporal; layers is a host array read during this call only.
 * Returns SGP_OK, SGP_ERR_INVALID_ARG, SGP_ERR_CUDA, or the device status left by an earlier
 * run that has already completed (read from a host copy, without waiting; a run still in
 * flight reports through sgp_pipeline_sync or a later run). */
int sgp_pipeline_run(sgp_pipeline* p, const sgp_layer* layers, int n_layers,
                     const int32_t* kv_len, const void* x_in, void* x_out, int n_tokens,
                     int32_t* topk_idx, float* topk_w, sgp_stream_t stream);

/* Waits for the last run (its completion event) and returns the device status recorded since
 * the status was last read (then clears it). */
int sgp_pipeline_sync(sgp_pipeline* p);

/* Times each stage's tasks of one run on its own SM pool, CUDA events, median of `reps`
 * replays; writes n_stages values (microseconds) to t_us.  Alone on the GPU by default; with
 * opts.stage_times_shared all stages replay at the same time.  Data dependencies between
 * stages are dropped, so outputs are meaningless; the caller's buffers are written as by a
 * run.  Synchronous. */
int sgp_pipeline_stage_times(sgp_pipeline* p, const sgp_layer* layers, int n_layers,
                             const int32_t* kv_len, const void* x_in, void* x_out,
                             int n_tokens, int reps, float* t_us);

/* Launch trace of the last run (pipeline created with opts.trace = 1).  Waits for the run,
 * then writes n_pairs = n_layers * m * SGP_N_OPS * 2 pairs {start_ns, end_ns} to t_ns (host,
 * at most max_pairs pairs), indexed [layer][microbatch][op][part]: part 0 is the op's main
 * kernel, part 1 the kernel that finishes a tensor-core projection.  A pair of zeros means
 * no such launch.  Start = earliest CTA start, end = latest CTA end, on the GPU's global
 * timer; used to check the makespan model (Eq. 4-5) against the measured task spans.
 * t_ns may be NULL to query n_pairs.  Returns SGP_OK, SGP_ERR_INVALID_ARG or SGP_ERR_CUDA. */
int sgp_pipeline_trace(sgp_pipeline* p, uint64_t* t_ns, int max_pairs, int* n_pairs);

/* SMs of every launch of the last run (pipeline created with opts.trace = 1): every CTA of a
 * kernel sets bit %smid (the hardware SM index, below 256) of that launch's mask.  Waits for
 * the run, then writes n_entries = n_layers * m * SGP_N_OPS * 2 masks of 8 uint32 words
 * (256 bits) to `masks` (host, at most max_entries), indexed like sgp_pipeline_trace's pairs.
 * An all-zero mask means no such launch.  Checks the SM partition: the kernels of different
 * stages must run on disjoint sets of SMs, each no larger than its pool ("SubGPU Pipelining:
 * Intra-GPU Fine-Grained Spatial Parallelism for LLM Inference", Section 3.1: disjoint SM
 * pools).  masks may be NULL to query n_entries.
 * Returns SGP_OK, SGP_ERR_INVALID_ARG or SGP_ERR_CUDA. */
int sgp_pipeline_trace_sms(sgp_pipeline* p, uint32_t* masks, int max_entries, int* n_entries);

/* Measured span of every task of the last run (pipeline created with opts.trace = 1): the
 * earliest CTA start of the task's first kernel and the latest CTA end of its last kernel,
 * on the GPU's global timer (ns), as {start_ns, end_ns} pairs in task order (the order of
 * sgp_pipeline_tasks).  Waits for the run.  A cross-stage handoff costs the gap between a
 * task's start and the end of its data predecessor (same paper, Section 3.2, Eq. 4 takes it
 * as zero).  spans may be NULL to query n_tasks.
 * Returns SGP_OK, SGP_ERR_INVALID_ARG or SGP_ERR_CUDA. */
int sgp_pipeline_task_spans(sgp_pipeline* p, uint64_t* spans, int max_tasks, int* n_tasks);

/* The timing recurrence of "SubGPU Pipelining: Intra-GPU Fine-Grained Spatial Parallelism
 * for LLM Inference", Section 3.2, Eq. 4-5, on a task DAG given as arrays (host memory):
 * task i (in a topological order: every predecessor index is below i, -1 for none) starts at
 * A_i = max(C_{pred_data[i]} + handoff when stage[pred_data[i]] != stage[i],
 * C_{pred_stage[i]}), an empty maximum being 0, and finishes at C_i = A_i + tau[i];
 * *makespan = max_i C_i, and finish (host double[n_tasks] or NULL) receives every C_i.
 * Host only.  Returns SGP_OK or SGP_ERR_INVALID_ARG. */
int sgp_makespan(int n_tasks, const int32_t* pred_data, const int32_t* pred_stage,
                 const int32_t* stage, const double* tau, double handoff, double* makespan,
                 double* finish);

/* Predicts the makespan of a run with the timing recurrence of "SubGPU Pipelining:
 * Intra-GPU Fine-Grained Spatial Parallelism for LLM Inference", Section 3.2, Eq. 4-5, from
 * task durations measured under contention: all stages replay their tasks at the same time
 * (one stream each, data edges dropped, launch trace on), and a task's duration runs from its
 * start to the start of the next task of its stage FIFO (so it includes the gap between
 * tasks).  Then A_i = max(C of the data predecessor + handoff_us when it ran on another stage,
 * C of the stage predecessor), C_i = A_i + tau_i, and *t_pred_us = max C_i.  t_stage_us (host
 * float[n_stages] or NULL) receives each stage's summed task durations.  The caller's buffers
 * are written as by a run; outputs are meaningless.  Synchronous.
 * Returns SGP_OK, SGP_ERR_INVALID_ARG, SGP_ERR_CUDA or a device status of the replays. */
int sgp_pipeline_predict(sgp_pipeline* p, const sgp_layer* layers, int n_layers,
                         const int32_t* kv_len, const void* x_in, void* x_out, int n_tokens,
                         float handoff_us, float* t_pred_us, float* t_stage_us);

/* Number of tasks of the last run's DAG and, when stamps != NULL, per-task
 * {stage, layer_first, micro, pred_data, pred_stage} as int32[5] rows (host memory). */
int sgp_pipeline_tasks(sgp_pipeline* p, int* n_tasks, int32_t* rows, int max_rows);

/* Frees the handle, its device state, streams and green contexts.  NULL is a no-op. */
void sgp_pipeline_destroy(sgp_pipeline* p);

/* ---- balancer (steady state is set by the slowest stage: split SMs by measured time) -- */

/* Legal two-stage splits: writes p_A values (stage A's SMs) in increasing order for
 * p_A in [p_min, n_sm - p_min] stepping by `quantum` (rounded up to the device alignment).
 * Returns the count (which may exceed max_out; only max_out are written) or a negative
 * status.  Host only. */
int sgp_enumerate_splits(int n_sm, int quantum, int p_min, int* out, int max_out);

/* For every legal split of a two-stage pipeline (sgp_enumerate_splits with the device's
 * SM count), measures t_A(p_A) and t_B(N - p_A) with sgp_pipeline_stage_times and returns
 * the split minimising max(t_A, t_B) in *best_split_out (p_A), plus all measurements:
 * splits[i], t_us[2 i], t_us[2 i + 1] for i < *n_out (capacity max_out).  Synchronous. */
int sgp_pipeline_balance(const sgp_dims* dims, const sgp_layer* layers, int n_layers,
                         const int32_t* kv_len, const void* x_in, void* x_out, int n_tokens,
                         int microbatch, int max_kv_len, int quantum, int reps,
                         const sgp_pipeline_opts* opts, int* best_split_out, int* splits,
                         float* t_us, int max_out, int* n_out);

/* ---- SM-allocation refinement for any stage count ---------------------------------- */

/* Objective of an SM allocation p[0..n_stages-1] (each entry a stage's SMs): lower is better;
 * a negative (or NaN) value marks an allocation that cannot be evaluated (treated as
 * infinitely bad).  ctx is passed through. */
typedef double (*sgp_alloc_objective)(const int* p, int n_stages, void* ctx);

/* Pairwise-line SM-allocation refinement ("SubGPU Pipelining: Intra-GPU Fine-Grained
 * Spatial Parallelism for LLM Inference", Section 4.2, Algorithm 2).  A move hands z * quantum
 * SMs from a donor stage to a receiver stage; the total stays fixed.  Each pass evaluates
 * every legal one-quantum move, takes the best (the first in (donor, receiver) order on
 * ties); if it beats the current value, a line search along that pair doubles the step
 * while the objective keeps improving and halves it otherwise; the allocation then moves to
 * the best point found.  The search stops when no legal move improves or after pass_limit
 * passes (<= 0: no limit).  A legal allocation has every entry >= max(p_min, quantum).
 * Objective values are memoised per allocation.
 *   p_inout  host int[n_stages]: the initial allocation (legal), replaced by the refined one
 *   t_out    host, or NULL: the refined allocation's objective
 * Host only, no device work of its own.  Returns the number of distinct allocations
 * evaluated (>= 1), or SGP_ERR_INVALID_ARG (2 <= n_stages <= 8). */
int sgp_refine_allocation(int n_stages, int* p_inout, int quantum, int p_min, int pass_limit,
                          sgp_alloc_objective f, void* ctx, double* t_out);

/* Pairwise-line refinement (sgp_refine_allocation) of a pipeline's SM allocation against
 * measured time: the objective of an allocation is the median of `reps` full pipelined runs
 * of the given layers (after one warm-up run), each a fresh pipeline with that split, the
 * same microbatch and opts.  The quantum is raised to the device's green-context alignment
 * and the minimum pool to its minimum partition.  Splits the device cannot form count as
 * infeasible.  For any stage count (2 or 3 here; Section 4.2 uses it for D >= 3).
 *   split_inout  host int[n_stages]: a legal starting allocation, replaced by the refined one
 *   t_us_out     host or NULL: the refined allocation's measured time (us)
 *   n_evals      host or NULL: distinct allocations measured
 * Synchronous.  Returns SGP_OK, SGP_ERR_INVALID_ARG, SGP_ERR_UNSUPPORTED, SGP_ERR_CUDA or a
 * device status of a measured run. */
int sgp_pipeline_refine(const sgp_dims* dims, const sgp_layer* layers, int n_layers,
                        const int32_t* kv_len, const void* x_in, void* x_out, int n_tokens,
                        int n_stages, int microbatch, int max_kv_len, int quantum, int reps,
                        int pass_limit, const sgp_pipeline_opts* opts, int* split_inout,
                        float* t_us_out, int* n_evals);

#ifdef __cplusplus
}
#endif
#endif /* SGP_H */
