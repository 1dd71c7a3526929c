// internal.h -- declarations shared by the library's translation units.
// Not part of the public ABI (that is include/tropical.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

#include <map>

#include "tropical.h"
#include "bounds.h"

namespace trop {

constexpr int MAXR = TROP_MAX_RANK;
constexpr int MAXB = 16;  // batch dims a GEMM launch can carry (after merging)

// ---------------------------------------------------------------- errors
int set_error(int code, const char* fmt, ...);
void clear_error();
int cuda_error(cudaError_t e, const char* what);  // TROP_ERR_CUDA with message

#define TROP_TRY(expr)                    \
    do {                                  \
        int trop_rc_ = (expr);            \
        if (trop_rc_ != TROP_OK) return trop_rc_; \
    } while (0)

// ---------------------------------------------------------------- device
struct DeviceInfo {
    int device;
    int sm_count;
    int max_threads_per_sm;
    size_t smem_per_sm;
    size_t l2_bytes;
};
// Set up the current device once; fills *info.  Also reports (once) an error word set by a
// kernel that abandoned its work, allocating that word on the device's first call unless a
// NoAllocScope is active on the calling thread (the allocation-free entry point).
int ensure_device(const DeviceInfo** info);
struct NoAllocScope {
    NoAllocScope();
    ~NoAllocScope();
};
// Validate a device pointer for the current device (nbytes > 0 only).
int check_device_pointer(const void* p, const char* name);
// Device address of the current device's error word (host-mapped; allocated on first use).
// A kernel that abandons its work sets it; ensure_device reports and clears it.
int device_error_word(uint32_t** dev_ptr);
// Test mode of the TMA-fed GEMM's bounded waits (tropical_debug_set_wait_mode): 0 normal.
int wait_test_mode();

// ---------------------------------------------------------------- counters
void count_launches(int64_t n);
// Kernels this library has launched (on any device or stream, captured or not), plus stream
// operations that end a chain of programmatic dependents (graph launches): a value that has
// not moved since a launch means nothing of this library was enqueued after it.
uint64_t launch_seq();
void note_stream_op();
void count_early_start();

// The last fused GEMM launched on a stream (gemm.cu): the launch_seq() right after it, the half
// of its stream tickets it used, and the byte ranges [lo, hi) of its two outputs.  A GEMM that
// follows it directly may read its operands before that grid has completed when they lie
// outside those ranges.
struct LaunchRecord {
    bool valid;
    uint64_t seq;
    int parity;
    uintptr_t lo[2], hi[2];
};
LaunchRecord stream_record(cudaStream_t s);
void set_stream_record(cudaStream_t s, const LaunchRecord& r);
void count_module_init();
void count_plan(bool hit);  // plan cache of the pairwise einsum (api.cpp)
void count_pool(int field, int64_t n);  // field: see pool.cu
enum { ST_ALLOC, ST_HIT, ST_MALLOC, ST_RETIRED, ST_RELEASED, ST_EVWAIT, ST_LEAKED, ST_BYTES };

// ---------------------------------------------------------------- pool
// Workspace blocks, released only after an event recorded on the stream
// that last used them completes (see pool.cu).
int pool_alloc(size_t bytes, cudaStream_t stream, void** out);
void pool_retire(void* ptr, cudaStream_t stream);

// Zeroed per-stream counters for atomic arrival tickets (the kernels reset them to zero).
int stream_tickets(cudaStream_t s, size_t count, uint32_t** out);

// ---------------------------------------------------------------- capture arena
// While a CaptureArena is installed on the calling thread (tree plans capture their launches
// into a CUDA graph, api.cpp), pool_alloc / pool_retire / stream_tickets take memory from it
// instead of the pool, and count_launches counts into it.  Blocks are placed first fit at
// 256-byte offsets from `base` and reused after release, so a capture's placement depends only
// on its sequence of requests: a measuring pass over a fake base (capacity unbounded) finds
// the high-water mark, and a second pass over real memory of that size places every block at
// the same offset.  The graph runs its nodes in capture order, so a block released by one node
// may serve a later node, as the pool does on one stream.
struct CaptureArena {
    uintptr_t base = 0;
    size_t capacity = 0;
    bool measuring = false;
    size_t top = 0, high = 0;
    int64_t launches = 0;
    std::map<size_t, size_t> free_;  // offset -> length of free extents below top
    std::map<size_t, size_t> used_;  // offset -> length of live blocks
    int alloc(size_t bytes, void** out);
    bool release(void* p);
};
void set_capture_arena(CaptureArena* a);
CaptureArena* capture_arena();

// ---------------------------------------------------------------- fast divmod
// Unsigned 32-bit division by a runtime-invariant divisor with a
// precomputed multiplier (Granlund & Montgomery, "Division by invariant
// integers using multiplication", PLDI 1994): q = umulhi(n, mul) >> shift.
struct FastDiv {
    uint32_t d, mul, shift;
};
FastDiv make_fastdiv(uint32_t d);

#ifdef __CUDACC__
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f)
{
    return f.mul == 0 ? (n >> f.shift) : (__umulhi(n, f.mul) >> f.shift);
}
#endif

#ifdef __CUDACC__
// Programmatic dependent launch.  A kernel launched with launch_pdl may start while the grid
// before it on the stream drains; it calls pdl_wait() before its first access to global
// memory (which waits for that grid to complete and its writes to be visible) and then
// pdl_signal(), which lets the grid after it start the same way.  Without the launch attribute
// both are no-ops.  Every access therefore keeps plain stream order; only launch latency is
// hidden.
__device__ __forceinline__ void pdl_signal() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// mbarriers of a CTA (phase parity waits, transaction counts) and the global timer that bounds
// every wait
__device__ __forceinline__ uint32_t smem_u32(const void* ptr) { return (uint32_t)__cvta_generic_to_shared(ptr); }
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase of `parity` to complete; give up after about 0.2 s.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > 200000000ull) return false;
    return true;
}


template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}
#endif

// ---------------------------------------------------------------- launches
// Gather / permute over `rank` dims (output order, last fastest).  Optional
// companion int32 tensor moved through the same index mapping.
struct GatherDesc {
    int rank;
    int64_t size[MAXR];
    int64_t s_in[MAXR];
    int64_t s_out[MAXR];
    int64_t s_in2[MAXR];
    int64_t s_out2[MAXR];
};
int launch_gather(const void* in, void* out, int elem_bytes, const int32_t* in2, int32_t* out2,
                  const GatherDesc& d, cudaStream_t s);

// (+)-reduction over `red` dims for every element of `out` dims.
struct ReduceDesc {
    int out_rank;
    int64_t out_size[MAXR];
    int64_t out_s_in[MAXR];
    int64_t out_s_out[MAXR];
    int64_t out_s_arg[MAXR];
    int red_rank;
    int64_t red_size[MAXR];
    int64_t red_s_in[MAXR];
};
// Where a split reduction keeps its partial results when `fixed` is given: a caller-provided
// block of `bytes` (the request fails with TROP_ERR_UNSUPPORTED when they do not fit); nothing
// is allocated.  Without it they go to pool workspace.
struct ReduceScratch {
    void* ptr;
    size_t bytes;
};
int launch_reduce(int semiring, int dtype, const void* in, void* out, int32_t* argmax,
                  const ReduceDesc& d, const ReduceScratch* fixed, cudaStream_t s);
// Fixed scratch of noalloc.cu: its device address on the current device (looked up once per device).
int noalloc_scratch(void** ptr, size_t* bytes);

// Strided-batched tropical GEMM with a multi-dimensional batch.
struct GemmDesc {
    int semiring;
    int dtype;  // TROP_F32 (gemm.cu), TROP_F64 (gemm64.cu), TROP_I32 / TROP_I64 (gemm_int.cu); A, B, C share it
    int64_t M, N, K;
    const void* A;
    const void* B;
    void* C;
    int32_t* I;  // nullable
    int64_t sAm, sAk, sBk, sBn, sCm, sCn, sIm, sIn;
    int nb;
    int64_t bsize[MAXB];
    int64_t sAb[MAXB], sBb[MAXB], sCb[MAXB], sIb[MAXB];
};
// The byte ranges of A, B, C (elements of elem_bytes) and I that g addresses, into sp[0..3]
// (bounds-checked build only; nothing in the normal build).
inline void gemm_spans(const GemmDesc& g, size_t elem_bytes, Span* sp)
{
#if TROP_DEBUG_BOUNDS
    int64_t sz[MAXB + 2], st[MAXB + 2];
    auto one = [&](const void* base, size_t eb, int64_t r, int64_t c, int64_t sr, int64_t sc, const int64_t* sb) {
        for (int i = 0; i < g.nb; ++i) sz[i] = g.bsize[i], st[i] = sb[i];
        sz[g.nb] = r, st[g.nb] = sr, sz[g.nb + 1] = c, st[g.nb + 1] = sc;
        return span_of(base, eb, g.nb + 2, sz, st);
    };
    sp[0] = one(g.A, elem_bytes, g.M, g.K, g.sAm, g.sAk, g.sAb);
    sp[1] = one(g.B, elem_bytes, g.K, g.N, g.sBk, g.sBn, g.sBb);
    sp[2] = one(g.C, elem_bytes, g.M, g.N, g.sCm, g.sCn, g.sCb);
    sp[3] = one(g.I, 4, g.M, g.N, g.sIm, g.sIn, g.sIb);
#else
    (void)g, (void)elem_bytes, (void)sp;
#endif
}
int launch_gemm(const GemmDesc& g, cudaStream_t s, const char** kernel_name);
// The binary64 GEMM (gemm64.cu); launch_gemm forwards TROP_F64 descriptors here.
int launch_gemm_f64(const GemmDesc& g, cudaStream_t s);
// The integer GEMM (gemm_int.cu); launch_gemm forwards TROP_I32 / TROP_I64 descriptors here.
int launch_gemm_int(const GemmDesc& g, cudaStream_t s);
// The route launch_gemm takes for g (kernel, operand swap, vector width, staging) as text.
void describe_gemm(const GemmDesc& g, char* buf, size_t n);

// Gradient of the tropical GEMM routed through its argmax (backward.cu).  Strides are
// {batch, row, column} of each 3-d operand; dA / dB nullable.
int launch_gemm_backward(int semiring, int64_t batch, int64_t M, int64_t N, int64_t K, const float* A,
                         const int64_t* sA, const float* B, const int64_t* sB, const float* dC, const int64_t* sC,
                         const int32_t* I, float* dA, const int64_t* sdA, float* dB, const int64_t* sdB,
                         cudaStream_t s);

// Tree back-tracking (backtrack.cu).
struct BtNode {
    const int32_t* argmax;  // nullable
    int n_out;              // output labels (row-major, last fastest)
    int n_k;                // argmax labels (row-major, last fastest)
    int lab_off;            // offset into the label table: n_out out labels then n_k argmax labels
};
int launch_backtrack(const BtNode* nodes_dev, int n_nodes, const int32_t* labels_dev, int n_labs,
                     const int64_t* sizes_dev, int64_t root_index, int n_labels,
                     int32_t* assignment, cudaStream_t s);

size_t dtype_bytes(int dtype);

}  // namespace trop
