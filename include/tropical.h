/*
 * tropical.h -- C ABI of the device-resident tropical einsum library
 * (libtropical_gb300.so, sm_103a).
 *
 * What the library computes
 * -------------------------
 * Pairwise tropical-semiring einsum kept on the device end to end:
 *   unary diagonal/trace pre-pass -> operand permute -> strided-batched
 *   tropical GEMM with argmax -> output permute (value and argmax through one
 *   index mapping), driven by a contraction-tree executor whose intermediates
 *   never leave device memory.
 *
 * Sources (web pages this library follows; section names are the pages' own):
 *  [I52]  omeinsum-rs issue #52, "GPU tropical path: keep tensors
 *         device-resident + device-side permute": Summary; "Why Julia is
 *         naturally fast"; "Proposed plan" steps 1-3; "Resolved design for
 *         step 3" kernels (a) permute/strided gather and (b) diagonal/trace
 *         gather + max/min reduce; "Acceptance criteria".
 *  [PR35] tropical-gemm PR #35, "batched GPU ops with DLPack zero-copy
 *         output": Summary (batched max-plus / min-plus / maxmul f32 kernels
 *         with argmax; rejecting host memory; zero-sized dimension guards;
 *         same-device validation).
 *  [RT]   rustytorch commit adding native CUDA gather / scatter-add
 *         (ops::index): scatter-add over the adjoint of the selection, with
 *         no atomics and deterministic results with duplicate indices; the
 *         adjoint identity test.
 *  [WR]   tenferro-rs design note "cuTENSOR workspace retirement without a
 *         stream barrier": Proposal (event on the owning stream + retirement
 *         queue) and "Open decisions" 1-2 (drain before allocation, bound 16,
 *         event wait at capacity, leak rather than race).
 *
 * Semirings (PR35 names them; their neutral elements are not given on the
 * pages and follow the usual tropical definitions):
 *     TROP_MAXPLUS : a (+) b = max(a,b), a (x) b = a + b, zero = -inf
 *     TROP_MINPLUS : a (+) b = min(a,b), a (x) b = a + b, zero = +inf
 *     TROP_MAXTIMES: a (+) b = max(a,b), a (x) b = a * b, zero = 0
 * Each (x) rounds once in the operands' IEEE format, binary32 (TROP_F32) or
 * binary64 (TROP_F64) (round to nearest even, subnormals kept); each (+) is
 * exact, so results do not depend on evaluation order.  f64 operands: I52
 * "Resolved design for step 3" kernel (a) lists f32/f64 operands; PR35
 * "Summary of latest fixes" handles f32 and f64 on its CPU path.
 * Integer operands (TROP_I32, TROP_I64; I52 "Resolved design for step 3"
 * kernel (a) lists integer types, PR35 "Summary of latest fixes" handles
 * dtypes beyond f32): each (x) is the exact integer a + b (a * b for
 * max-times) and every product formed must fit the operand type -- the pages
 * fix no overflow policy, so this precondition is the library's reading (a
 * product outside the type wraps; not checked).  The zeros are the type's
 * min / max / 0 and only start the running (+).
 * Argmax: the smallest contracted linear index that reaches the result; 0
 * when no term beats the semiring zero (e.g. an empty contraction).
 * Preconditions (not checked): no NaN; no -0.0; max-plus operands below
 * +inf and min-plus operands above -inf; max-times operands finite and
 * nonnegative (negative products are clamped by the zero 0).
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Tensor data pointers are DEVICE pointers of the current device
 *    (cudaMalloc / torch CUDA storage, or managed memory).  Host pointers are
 *    rejected with TROP_ERR_HOST_POINTER [PR35 Summary "Reject CudaHost"];
 *    pointers of another device with TROP_ERR_DEVICE_MISMATCH.
 *  - Strides are in ELEMENTS and may be 0 (broadcast) for inputs.  Outputs
 *    must not overlap themselves or the inputs (not checked).
 *  - The caller owns every input, output and argmax buffer.  The library owns
 *    only its workspace.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call is asynchronous on it: results are valid once the
 *    stream reaches the point of the call.  No call synchronizes a stream.
 *  - Return value: TROP_OK (0) or a negative TROP_ERR_* code.  The message of
 *    the last failure on the calling thread is tropical_last_error().  No C++
 *    exception crosses this boundary.  Validation failures launch nothing.
 *  - Zero-sized dimensions are allowed [PR35 Summary]: an empty output is a
 *    no-op; an empty contraction writes the semiring zero and argmax 0.
 *  - Thread safety: calls may come from several host threads; library state
 *    (module set-up, workspace pool, counters) is internally locked.
 */
#ifndef TROPICAL_GB300_H
#define TROPICAL_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TROP_MAX_RANK 32

typedef enum { TROP_MAXPLUS = 0, TROP_MINPLUS = 1, TROP_MAXTIMES = 2 } trop_semiring;
typedef enum { TROP_F32 = 0, TROP_I32 = 1, TROP_I64 = 2, TROP_F64 = 3 } trop_dtype;

enum {
    TROP_OK = 0,
    TROP_ERR_INVALID_ARG = -1,     /* null pointer, bad enum, rank or id out of range */
    TROP_ERR_HOST_POINTER = -2,    /* a data pointer is host memory */
    TROP_ERR_DEVICE_MISMATCH = -3, /* a data pointer belongs to another device */
    TROP_ERR_DTYPE = -4,           /* unsupported or mismatched dtype */
    TROP_ERR_SHAPE = -5,           /* extents disagree with the spec or each other */
    TROP_ERR_SPEC = -6,            /* einsum spec does not parse / is inconsistent */
    TROP_ERR_OVERFLOW = -7,        /* contracted extent does not fit an int32 argmax */
    TROP_ERR_CUDA = -8,            /* a CUDA runtime call or launch failed */
    TROP_ERR_OOM = -9,             /* workspace allocation failed */
    TROP_ERR_UNSUPPORTED = -10     /* valid request this build does not handle */
};

/* A strided tensor view.  data: device pointer (may be NULL when an extent is
 * 0); shape/stride: first `rank` entries used, strides in elements. */
typedef struct {
    void* data;
    int32_t dtype; /* trop_dtype */
    int32_t rank;  /* 0 .. TROP_MAX_RANK */
    int64_t shape[TROP_MAX_RANK];
    int64_t stride[TROP_MAX_RANK];
} trop_tensor;

/* One node of a contraction tree (see tropical_contract_tree).  Operand ids:
 * 0 .. n_inputs-1 are the tree's inputs, n_inputs + j is node j's output
 * (j smaller than this node's index).  rhs = -1 makes a unary node (diagonal /
 * trace / permute of lhs).  Labels are integers in [0, 65535]; a label
 * repeated inside one operand is a diagonal, a label absent from out_labels
 * is reduced with (+). */
typedef struct {
    int32_t lhs, rhs;
    int32_t n_lhs, n_rhs, n_out;
    const int32_t* lhs_labels;
    const int32_t* rhs_labels;
    const int32_t* out_labels;
} trop_node;

/* Counters since load (or since tropical_reset_stats). */
typedef struct {
    int64_t module_inits;        /* per-device kernel set-ups (once per device) */
    int64_t kernel_launches;     /* kernels launched by this library */
    int64_t pool_allocs;         /* workspace requests */
    int64_t pool_hits;           /* requests served from cached blocks */
    int64_t pool_device_mallocs; /* cudaMalloc calls made by the pool */
    int64_t pool_retired;        /* blocks handed to the retirement queue */
    int64_t pool_released;       /* retired blocks whose event completed */
    int64_t pool_event_waits;    /* queue at capacity: waited on the oldest event */
    int64_t pool_leaked;         /* event record failed: block leaked, never reused */
    int64_t pool_bytes_cached;   /* bytes held by the pool (free + retiring) */
    int64_t stream_syncs;        /* stream synchronizations issued (stays 0) */
    int64_t plan_cache_hits;     /* pairwise einsums (eager calls and tree nodes) whose
                                    lowering came from the plan cache */
    int64_t plan_cache_misses;   /* ... that were lowered (and then cached) */
    int64_t gemm_early_starts;   /* argmax GEMMs (one-launch form) that began loading and
                                    computing before the GEMM just before them on the stream
                                    had finished: their operands were outside its outputs */
} trop_stats;

/* Set up the kernels for `device` once (kernel attributes, device
 * properties, workspace pool) [I52 "Proposed plan" step 1: the context and
 * module are created once, not per node].  Idempotent; every other entry
 * point calls it for the current device.  Errors: TROP_ERR_CUDA. */
int tropical_init(int device);

/* Unary op [I52 "Resolved design for step 3", kernels (a) and (b)]:
 *   spec "in->out" over letters a-z A-Z, e.g. "abcdef->fbdcae" (permute),
 *   "iijk->ijk" (diagonal gather), "iijk->jk" (diagonal + (+)-reduce over i).
 *   out[o] = (+) over the labels of `in` absent from the output of
 *   in[diagonal position], in the semiring `semiring`; with no such label
 *   this is a strided gather (any dtype; semiring only checked for range).
 * in, out:  same dtype (f32, f64, i32 or i64); out.shape must equal the output
 *           label extents; out may be strided.
 * argmax:   nullable int32 buffer, contiguous row-major in out's shape: the
 *           row-major linear index over the reduced labels (first-appearance
 *           order in `in`) of the winner, 0 if nothing is reduced.
 * Errors: INVALID_ARG, SPEC, SHAPE, DTYPE, HOST_POINTER, DEVICE_MISMATCH,
 *         OVERFLOW (reduced extent > INT32_MAX with argmax), CUDA, OOM. */
int tropical_permute_trace(const trop_tensor* in, const char* spec, int semiring,
                           const trop_tensor* out, int32_t* argmax, void* stream);

/* Allocation-free variant of tropical_permute_trace (no counterpart on the
 * pages this library follows; it exists for callers of this library that
 * cannot allocate device memory: hosts that own every device allocation,
 * loops that cannot absorb an allocation's implicit synchronisation, or
 * processes whose device memory is already handed to their own allocator).
 * Same arguments, results and errors as tropical_permute_trace.  A split
 * reduction keeps its partial results in one fixed 256 KiB device array
 * compiled into the library (resident on every GPU that loads it) instead of
 * pool workspace; no call allocates or frees memory.  A partial result takes
 * 8 bytes of index plus one element (12 bytes for f32/i32, 16 for f64/i64),
 * and a reduction splits into fewer than 16 x (SM count) partials, so on a
 * 152-SM GB300 a call needs at most about 39 KB of the array.  Requests
 * whose partials would need more than 256 KiB (only possible on GPUs with
 * more than about 1000 SMs) fail with TROP_ERR_UNSUPPORTED.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  The address is kept for the life of the process: after
 * cudaDeviceReset the library's per-device state (this address and the
 * workspace pool) is stale, so do not call the library on a device that was
 * reset in the same process.  Every call shares the one array: calls whose
 * kernels overlap on the GPU (other streams, other host threads) race on it,
 * so serialise them.  Nothing in it needs to start at zero: each call writes
 * every partial it reads. */
int tropical_permute_trace_noalloc(const trop_tensor* in, const char* spec, int semiring,
                                   const trop_tensor* out, int32_t* argmax, void* stream);

/* Output permute of a result and its argmax through ONE index mapping
 * [I52 "Resolved design for step 3": the float result and the argmax must be
 * permuted with bit-for-bit identical index mappings].  spec is a pure
 * permutation "abc->cab" (no repeated or dropped label).  val_in/val_out are
 * f32, f64, i32 or i64 of equal dtype; arg_in/arg_out are int32 tensors of the
 * same shapes as val_in/val_out (any strides).  One kernel launch moves both. */
int tropical_permute_pair(const trop_tensor* val_in, const trop_tensor* arg_in, const char* spec,
                          const trop_tensor* val_out, const trop_tensor* arg_out, void* stream);

/* Strided-batched tropical GEMM with argmax [PR35 Summary: the batched
 * max-plus / min-plus / maxmul f32 kernels with argmax]:
 *   C[b,m,n] = (+)_{k<K} A[b,m,k] (x) B[b,k,n]
 *   argmax[b,m,n] = smallest k reaching C[b,m,n] (0 if none beats zero).
 * Element (b,m,k) of A is A[b*sAb + m*sAm + k*sAk]; likewise B and C.
 * argmax (nullable, int32) uses C's strides.  dtype: TROP_F32, TROP_F64,
 * TROP_I32 or TROP_I64, shared by A, B and C (the pointers carry no type: the
 * caller guarantees it).  Integer operands must keep every product inside the
 * type (a + b, or a * b for max-times); then every result is exact.
 * Ordering is the stream's: a call's results are complete when the stream
 * reaches the call's end.  On the GPU an f32 argmax call that directly
 * follows another on the same stream and reads none of the bytes that one
 * writes may start loading and computing before it has finished; it stores
 * nothing before then (trop_stats.gemm_early_starts counts such calls).
 * Errors: INVALID_ARG (negative extent, null pointer with nonzero extent),
 *         DTYPE, OVERFLOW (K > INT32_MAX with argmax), HOST_POINTER,
 *         DEVICE_MISMATCH, CUDA. */
int tropical_gemm_strided_batched_argmax(int semiring, int dtype,
                                         int64_t batch, int64_t M, int64_t N, int64_t K,
                                         const void* A, int64_t sAb, int64_t sAm, int64_t sAk,
                                         const void* B, int64_t sBb, int64_t sBk, int64_t sBn,
                                         void* C, int64_t sCb, int64_t sCm, int64_t sCn,
                                         int32_t* argmax, void* stream);

/* Backward of the strided-batched tropical GEMM: the gradient routed through
 * the forward argmax ("winner routing") [I52 "Acceptance criteria": forward,
 * backward and argmax consistent with the CPU path; PR35: the batched
 * autograd functions send the gradient through the argmax with a
 * scatter-add; RT: scatter-add over the adjoint, deterministic, no atomics].
 * Given dC and argmax I of a forward call (I uses dC's strides):
 *   dA[b,m,k] = sum over n in increasing order with I[b,m,n] == k of g
 *   dB[b,k,n] = sum over m in increasing order with I[b,m,n] == k of g
 * where g = dC[b,m,n] for max-plus / min-plus, and for max-times
 * g = dC[b,m,n] * B[b,k,n] in dA and g = dC[b,m,n] * A[b,m,k] in dB.  Every
 * output routes to its argmax (including 0 when nothing beat the zero); an
 * index outside [0,K) routes nowhere.  Each product and each addition rounds
 * once in binary32, in the order stated, so results are bit-reproducible.
 * dA and dB are written entirely (zero where nothing routes); either may be
 * NULL (not wanted).  The two are computed concurrently, so they must not
 * overlap each other or any input.  A and B are read only for max-times (may
 * be NULL otherwise).  All pointers are device memory, f32 except the int32 argmax;
 * the caller owns every buffer.  Strides in elements, any sign-free layout.
 * Errors: INVALID_ARG (negative extent, missing pointer), OVERFLOW
 *         (K > INT32_MAX), HOST_POINTER, DEVICE_MISMATCH, CUDA. */
int tropical_gemm_backward(int semiring, int64_t batch, int64_t M, int64_t N, int64_t K,
                           const float* A, int64_t sAb, int64_t sAm, int64_t sAk,
                           const float* B, int64_t sBb, int64_t sBk, int64_t sBn,
                           const float* dC, int64_t sCb, int64_t sCm, int64_t sCn,
                           const int32_t* argmax,
                           float* dA, int64_t sdAb, int64_t sdAm, int64_t sdAk,
                           float* dB, int64_t sdBb, int64_t sdBk, int64_t sdBn, void* stream);

/* Pairwise tropical einsum [I52 Summary and "Resolved design for step 3";
 * PR35 Summary]:  spec "zacd,zdce->zea" over letters a-z A-Z.
 * Plan cache [WR "Problem": the einsum path caches one plan per contraction]:
 * the lowering (pre-passes and GEMM layout) is kept per layout -- labels,
 * extents, strides, dtype, semiring, whether argmax is written and the 16-byte
 * alignment of every buffer -- in a bounded LRU of 64 entries (the environment
 * variable TROP_PLAN_CACHE at load sets the bound; 0 disables it), so a
 * repeated call skips it; trop_stats counts hits and misses.  The contraction
 * tree executor's nodes use the same cache.
 *   out[o] = (+) over all assignments of the labels absent from the output
 *            of A[..] (x) B[..]   (A, B and out of one dtype: f32, f64, i32
 *            or i64)
 *   argmax[o] = row-major linear index over the CONTRACTED labels (present
 *            in both operands, absent from the output), ordered by first
 *            appearance in A's spec, of the smallest index reaching out[o].
 *            Labels present in only one operand and absent from the output
 *            are (+)-reduced first (a unary pre-pass) and are not part of
 *            the argmax.  No contracted label: argmax 0.
 * Lowering: diagonal/trace pre-pass per operand, permutes only where an
 * operand's strides cannot feed the GEMM directly, strided-batched GEMM
 * writing value and argmax through the output's own strides, or into a
 * workspace followed by the one-mapping pair permute.
 * argmax: nullable int32, contiguous row-major in out's shape.
 * Errors: as tropical_permute_trace, plus OVERFLOW when the contracted extent
 *         exceeds INT32_MAX with argmax. */
int tropical_einsum_pairwise(const char* spec, const trop_tensor* A, const trop_tensor* B,
                             int semiring, const trop_tensor* out, int32_t* argmax, void* stream);

/* Contraction-tree executor [I52 Summary, "Why Julia is naturally fast"
 * row 1, "Acceptance criteria" 1: intermediates stay in device memory across
 * the whole tree].  Runs nodes 0..n_nodes-1 in order; node j's output lives
 * in pool workspace (contiguous, row-major in its out_labels order) until
 * its last consumer has been enqueued, then is retired through an event on
 * `stream` [WR Proposal].  The last node writes `out` (strided allowed).
 * node_argmax: nullable array of n_nodes nullable int32 device buffers; entry
 *   j receives node j's argmax (contiguous, node output shape), with the
 *   meaning of tropical_einsum_pairwise (binary) or tropical_permute_trace
 *   (unary).
 * All inputs must share out's dtype (f32, f64, i32 or i64).
 * Errors: as the pairwise/unary calls, plus INVALID_ARG for bad operand ids.
 * Validation of the whole tree happens before the first launch. */
int tropical_contract_tree(int n_inputs, const trop_tensor* inputs, int n_nodes,
                           const trop_node* nodes, int semiring, const trop_tensor* out,
                           int32_t* const* node_argmax, void* stream);

/* Tree plans: a contraction tree lowered once and replayed as one CUDA graph.
 * [WR "Result": with the stream barriers gone, per-kernel launch latency is
 * the remaining gap; WR "Problem": the cuTENSOR path caches its plans per
 * contraction; I52 "Proposed plan" step 1: build the GPU context and module
 * once instead of per contraction.]
 *
 * tropical_tree_plan_create validates and lowers the tree exactly as
 * tropical_contract_tree does, then captures the resulting launches into a
 * CUDA graph.  The plan binds the buffers passed here: every run reads the
 * current contents of `inputs` and writes `out` and the non-NULL
 * `node_argmax` buffers, so callers refill inputs in place between runs.
 * Intermediates and all internal workspace live in one device allocation
 * owned by the plan (blocks reused along the tree as their last consumer
 * passes, as the pool does); the shape, strides and dtypes fixed at creation
 * decide every lowering choice, so a run does no host planning and no
 * allocation.  Creation synchronises nothing but allocates (cudaMalloc).
 * Errors of create: as tropical_contract_tree, plus OOM and CUDA (a capture
 * or graph call failed); *plan is NULL on failure.
 *
 * tropical_tree_plan_run launches the graph on `stream` (asynchronous, like
 * every call here).  Runs of one plan are ordered by CUDA (a graph cannot run
 * concurrently with itself); callers that share a plan across host threads
 * serialise their calls.  Errors: INVALID_ARG (NULL plan), DEVICE_MISMATCH
 * (current device is not the plan's), CUDA.
 *
 * tropical_tree_plan_info reports the kernels one run launches and the bytes
 * of the plan's workspace (either pointer may be NULL).
 *
 * tropical_tree_plan_destroy frees the graph and the workspace; call it once
 * no run of the plan is pending (cudaFree waits for the device).  NULL is a
 * no-op. */
typedef struct trop_tree_plan_s* trop_tree_plan;
int tropical_tree_plan_create(int n_inputs, const trop_tensor* inputs, int n_nodes,
                              const trop_node* nodes, int semiring, const trop_tensor* out,
                              int32_t* const* node_argmax, trop_tree_plan* plan);
int tropical_tree_plan_run(trop_tree_plan plan, void* stream);
int tropical_tree_plan_info(trop_tree_plan plan, int64_t* kernels, size_t* workspace_bytes);
int tropical_tree_plan_destroy(trop_tree_plan plan);

/* Argmax back-tracking through a contraction tree, on the device.  Given the
 * tree of tropical_contract_tree, every node's argmax buffer and the linear
 * index `root_index` of an element of the last node's output (0 for a scalar
 * root), writes assignment[l] = the value of label l in the optimal
 * configuration, for l in [0, n_labels); labels whose value no argmax
 * determines (one-operand labels reduced inside a binary node, or nodes
 * whose argmax buffer is NULL) are -1.  assignment: int32 device buffer of
 * n_labels entries.  One warp walks the nodes backwards, with the node,
 * label and extent tables in shared memory when they fit (one thread over
 * global memory otherwise); nothing is copied to the host. */
int tropical_tree_backtrack(int n_inputs, const trop_tensor* inputs, int n_nodes,
                            const trop_node* nodes, int32_t* const* node_argmax,
                            int64_t root_index, int n_labels, int32_t* assignment, void* stream);

/* Drain the workspace retirement queue: wait for every pending event and
 * return the blocks to the pool [WR "Open decisions" 1: explicit
 * synchronize() is a drain point].  The only call that may block the host. */
int tropical_sync_pool(void);

/* Drain, then free every cached workspace block and the per-stream arrival
 * counters of the GEMM's split tiles (teardown). */
int tropical_release_pool(void);

int tropical_stats(trop_stats* out);
void tropical_reset_stats(void);

/* Bounded waits inside kernels on the current device that gave up, since load
 * or since the last reset.  The TMA-fed GEMM waits for each operand copy on an
 * mbarrier for at most about 0.2 s.  A CTA whose wait gives up counts one here
 * and waits once more with the full bound: a copy that lands late still gives
 * exact results.  If it has not landed then either, the CTA waits (bounded) for
 * its copies in flight, abandons its tile (its argmax entries are set to 0, its
 * values left as they were) and sets a device error word in host-mapped memory;
 * the first library call made on the device after that kernel finished (or
 * tropical_sync_pool) returns TROP_ERR_CUDA naming the failure, once.  The
 * values and argmax of the call whose kernel abandoned a tile are undefined.
 * In the one-launch form (argmax, K <= 256) the resolve work of each batch
 * also waits, for at most about 1 s, until that batch's tiles are stored; a
 * wait that gives up there sets the same error word (it is not counted here).
 * Reads a device counter: blocks until the device is idle.  reset != 0 zeroes
 * the counter after reading it.  Returns TROP_OK, or TROP_ERR_INVALID_ARG for a
 * NULL count, or TROP_ERR_CUDA. */
int tropical_device_wait_timeouts(unsigned int* count, int reset);

/* Bounds violations recorded by the library's debug build (compiled with
 * TROP_DEBUG_BOUNDS=1): every global load, store and copy of its kernels is
 * first tested against the byte range of the tensor view it belongs to
 * (computed on the host from extents and strides); an access outside it is
 * skipped and counted, and the first one's location and address kept.
 * *line = (file id << 16) | source line, the file ids being 1 unary.cu, 2
 * gemm.cu, 3 gemm64.cu, 4 gemm_int.cu, 5 backward.cu, 6 backtrack.cu.
 * Reads the record of the current device without synchronising: call it once
 * the work to inspect has completed.  reset != 0 clears the record.  The
 * normal build returns TROP_ERR_UNSUPPORTED with *count = 0.  It stands in
 * for an external memory checker; TMA box copies are bounded by their tensor
 * maps instead and are not tested. */
int tropical_debug_bounds_report(unsigned int* count, int* line, uint64_t* addr, int reset);

/* Test hook of the debug build: every byte range made after this call is cut
 * short by `bytes` at its top, so that the last `bytes` of each tensor read
 * or written count as outside it (the access itself is skipped, and it was
 * inside the tensor's memory anyway).  It shows that the checks fire; 0
 * restores exact ranges.  Returns TROP_OK, TROP_ERR_INVALID_ARG for a negative
 * count, or TROP_ERR_UNSUPPORTED from the normal build. */
int tropical_debug_bounds_trim(int64_t bytes);

/* Test hook for the bounded waits above (host-side; it changes no device
 * setting): mode 1 makes the first operand wait of every CTA of the TMA-fed
 * GEMMs launched afterwards give up at once (then wait again with the full
 * bound, so results stay exact and the counter above grows); mode 2 does the
 * same and then treats that second wait as failed after it completed, so each
 * CTA takes the failure path with no copy in flight (the next call reports
 * TROP_ERR_CUDA).  0 restores normal waits; other values are taken as 0. */
void tropical_debug_set_wait_mode(int mode);

/* Message of the last failure on this host thread ("" if none). */
const char* tropical_last_error(void);

/* Library / ABI version (increments on incompatible changes; 2: trop_stats gained the plan
 * cache counters). */
int tropical_version(void);

/* Host-only planner inspection (no device work, no GPU needed): describes how
 * tropical_einsum_pairwise would lower `spec` for operands with the given
 * shapes/strides and a contiguous output, as one line of text in buf.
 * Returns TROP_OK or an error code (SPEC, SHAPE, INVALID_ARG). */
int tropical_plan_describe(const char* spec, int rank_a, const int64_t* shape_a, const int64_t* stride_a,
                           int rank_b, const int64_t* shape_b, const int64_t* stride_b,
                           char* buf, int buflen);

/* Test hook for the leak-rather-than-race path [WR "Open decisions" 2]:
 * the next `count` retirements behave as if recording their CUDA event had
 * failed (the block is then leaked, never reused).  Host-side only. */
void tropical_debug_fail_next_event_records(int count);

/* Set the retirement-queue bound (default 16, or TROP_POOL_CAPACITY from the
 * environment at load).  Values < 1 are clamped to 1. */
void tropical_set_pool_capacity(int capacity);

/* Set the bound of the pairwise einsum's plan cache (see tropical_einsum_pairwise;
 * default 64, or TROP_PLAN_CACHE from the environment at load).  0 disables the
 * cache and drops its entries; a smaller bound drops the least recently used. */
void tropical_set_plan_cache_capacity(int capacity);

#ifdef __cplusplus
}
#endif

#endif /* TROPICAL_GB300_H */
