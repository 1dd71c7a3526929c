// runtime.cpp -- once-per-device set-up, error state, counters, and the
// workspace pool whose blocks are released only through CUDA events.
//
// Workspace retirement follows the tenferro-rs design note "cuTENSOR
// workspace retirement without a stream barrier": a block that is no longer
// needed gets an event recorded on the stream that last used it and joins a
// bounded retirement queue (Proposal, items 2-4).  The queue is drained --
// events queried, completed blocks returned to the free lists -- right
// before every allocation and on an explicit tropical_sync_pool()
// ("Open decisions" 1).  At capacity (default 16) the oldest retirement is
// resolved with an event wait; if recording the event fails the block is
// leaked, never reused ("Open decisions" 2: leak rather than race).  Unlike
// that note there is no stream-barrier fallback at all: no code path here
// calls cudaStreamSynchronize or cudaDeviceSynchronize.
//
// One refinement: a retiring block may be handed to a new request on the
// SAME stream before its event completes, because stream order already puts
// the new work after the old (the usual stream-ordered caching rule).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <iterator>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <deque>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

namespace trop {

// ------------------------------------------------------------------ errors
static thread_local std::string g_last_error;

int set_error(int code, const char* fmt, ...)
{
    char buf[1024];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

void clear_error() { g_last_error.clear(); }

int cuda_error(cudaError_t e, const char* what)
{
    return set_error(TROP_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

size_t dtype_bytes(int dtype)
{
    switch (dtype) {
    case TROP_F32: return 4;
    case TROP_I32: return 4;
    case TROP_I64: return 8;
    case TROP_F64: return 8;
    default: return 0;
    }
}

// ------------------------------------------------------------------ counters
static std::atomic<int64_t> c_module_inits{0}, c_launches{0}, c_stream_syncs{0};
static std::atomic<int64_t> c_pool[8];

static thread_local CaptureArena* t_arena = nullptr;
void set_capture_arena(CaptureArena* a) { t_arena = a; }
CaptureArena* capture_arena() { return t_arena; }

static std::atomic<uint64_t> g_launch_seq{0};
void count_launches(int64_t n)
{
    if (t_arena) t_arena->launches += n;
    else c_launches += n;
    g_launch_seq.fetch_add(1, std::memory_order_acq_rel);
}
uint64_t launch_seq() { return g_launch_seq.load(std::memory_order_acquire); }
void note_stream_op() { g_launch_seq.fetch_add(1, std::memory_order_acq_rel); }
void count_module_init() { c_module_inits += 1; }
static std::atomic<int64_t> c_plan_hits{0}, c_plan_misses{0}, c_early{0};
void count_plan(bool hit) { (hit ? c_plan_hits : c_plan_misses) += 1; }
void count_early_start() { c_early += 1; }
void count_pool(int field, int64_t n) { c_pool[field] += n; }

// ------------------------------------------------------------------ fast divmod
FastDiv make_fastdiv(uint32_t d)
{
    FastDiv f{};
    f.d = d ? d : 1;
    uint32_t l = 0;
    while (l < 32 && (uint64_t(1) << l) < f.d) ++l;  // l = ceil(log2 d)
    if ((f.d & (f.d - 1)) == 0) {                     // power of two: plain shift
        f.mul = 0;
        f.shift = l;
        return f;
    }
    // m = floor(2^(32+l) / d) + 1 fits 33 bits; keep the low 32 and fold the
    // top bit into the formula q = (umulhi(n, m') + n) >> l ... to stay in 32-bit
    // arithmetic we instead use the 31-bit-safe variant with n < 2^31:
    //   mul = ceil(2^(31+l) / d), q = umulhi(n, mul) >> (l - 1)
    // which is exact for all n < 2^31 (all index arithmetic here is below 2^31).
    uint64_t m = ((uint64_t(1) << (31 + l)) + f.d - 1) / f.d;
    f.mul = (uint32_t)m;
    f.shift = l - 1;
    return f;
}

// ------------------------------------------------------------------ device error word
// One word per device in pinned host memory that kernels can write (device-mapped): set by a
// kernel that had to abandon its work -- the TMA-fed GEMM when an operand copy did not land
// within twice its bounded wait.  Allocated by the first call on the device that may
// allocate (the allocation-free entry point never does), read without any synchronisation at
// the start of every later call and reported once, then cleared.
static std::mutex g_err_mu;
static std::atomic<volatile uint32_t*> g_err_host[64];
static std::atomic<uint32_t*> g_err_dev[64];
static std::atomic<int> g_wait_mode{0};

int device_error_word(uint32_t** dev_ptr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return set_error(TROP_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    if (uint32_t* w = g_err_dev[dev].load(std::memory_order_acquire)) {
        *dev_ptr = w;
        return TROP_OK;
    }
    std::lock_guard<std::mutex> lk(g_err_mu);
    if (!g_err_dev[dev].load(std::memory_order_relaxed)) {
        void* h = nullptr;
        e = cudaHostAlloc(&h, 64, cudaHostAllocMapped | cudaHostAllocPortable);
        if (e != cudaSuccess) return cuda_error(e, "cudaHostAlloc (device error word)");
        std::memset(h, 0, 64);
        void* d = nullptr;
        e = cudaHostGetDevicePointer(&d, h, 0);
        if (e != cudaSuccess) {
            cudaFreeHost(h);
            return cuda_error(e, "cudaHostGetDevicePointer (device error word)");
        }
        g_err_host[dev].store(static_cast<volatile uint32_t*>(h), std::memory_order_release);
        g_err_dev[dev].store(static_cast<uint32_t*>(d), std::memory_order_release);
    }
    *dev_ptr = g_err_dev[dev].load(std::memory_order_relaxed);
    return TROP_OK;
}

// nonzero error word of `dev`: clear it and return the error to report
static int take_device_error(int dev)
{
    volatile uint32_t* w = g_err_host[dev].load(std::memory_order_acquire);
    if (!w || *w == 0) return TROP_OK;
    *w = 0;
    return set_error(TROP_ERR_CUDA,
                     "a kernel on device %d abandoned its work: an operand copy of the TMA-fed GEMM did not land "
                     "within its bounded waits, so the values and argmax of that earlier call are undefined",
                     dev);
}

int wait_test_mode() { return g_wait_mode.load(std::memory_order_relaxed); }

#if TROP_DEBUG_BOUNDS
// words 4..7 of the device's host-mapped block: the bounds-violation record (bounds.h)
unsigned* bounds_record()
{
    uint32_t* w = nullptr;
    if (device_error_word(&w) != TROP_OK) {
        clear_error();
        return nullptr;
    }
    return w + 4;
}

// test hook: bytes cut from the top of every span made from now on (0: exact ranges)
static std::atomic<int64_t> g_span_trim{0};
int64_t bounds_span_trim() { return g_span_trim.load(std::memory_order_relaxed); }
#endif

// ------------------------------------------------------------------ device set-up
static std::mutex g_dev_mu;
static DeviceInfo g_dev[64];
static bool g_dev_ready[64];

extern int register_kernels_for_device();  // kernels.cu: loads kernels once

static thread_local int t_no_alloc = 0;
NoAllocScope::NoAllocScope() { ++t_no_alloc; }
NoAllocScope::~NoAllocScope() { --t_no_alloc; }

static std::atomic<bool> g_dev_done[64];  // set up, with its error word (lock-free fast path)

int ensure_device(const DeviceInfo** info)
{
    const bool may_allocate = t_no_alloc == 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return set_error(TROP_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    if (g_dev_done[dev].load(std::memory_order_acquire)) {
        if (info) *info = &g_dev[dev];
        return take_device_error(dev);
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev_ready[dev]) {
        cudaDeviceProp p;
        e = cudaGetDeviceProperties(&p, dev);
        if (e != cudaSuccess) return cuda_error(e, "cudaGetDeviceProperties");
        if (p.major < 10)
            return set_error(TROP_ERR_UNSUPPORTED, "device %d is sm_%d%d; this build targets sm_103a", dev,
                             p.major, p.minor);
        DeviceInfo& d = g_dev[dev];
        d.device = dev;
        d.sm_count = p.multiProcessorCount;
        d.max_threads_per_sm = p.maxThreadsPerMultiProcessor;
        d.smem_per_sm = p.sharedMemPerMultiprocessor;
        d.l2_bytes = (size_t)p.l2CacheSize;
        int rc = register_kernels_for_device();
        if (rc != TROP_OK) return rc;
        g_dev_ready[dev] = true;
        count_module_init();
    }
    if (info) *info = &g_dev[dev];
    if (may_allocate && !g_err_dev[dev].load(std::memory_order_acquire)) {
        uint32_t* w = nullptr;
        TROP_TRY(device_error_word(&w));
    }
    if (g_err_dev[dev].load(std::memory_order_acquire)) g_dev_done[dev].store(true, std::memory_order_release);
    return take_device_error(dev);
}

int check_device_pointer(const void* p, const char* name)
{
    if (!p) return set_error(TROP_ERR_INVALID_ARG, "%s is NULL", name);
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return set_error(TROP_ERR_HOST_POINTER, "%s (%p) is not a CUDA device pointer (%s)", name, p,
                         cudaGetErrorString(e));
    }
    if (a.type == cudaMemoryTypeUnregistered || a.type == cudaMemoryTypeHost)
        return set_error(TROP_ERR_HOST_POINTER, "%s (%p) is host memory; device memory is required", name, p);
    int dev = 0;
    cudaGetDevice(&dev);
    if (a.type == cudaMemoryTypeDevice && a.device != dev)
        return set_error(TROP_ERR_DEVICE_MISMATCH, "%s lives on device %d, current device is %d", name,
                         a.device, dev);
    return TROP_OK;
}

// ------------------------------------------------------------------ pool
namespace {

struct Block {
    void* ptr;
    size_t bytes;
    int device;
};

struct Retiring {
    Block b;
    cudaEvent_t ev;
    cudaStream_t stream;
};

struct Pool {
    std::mutex mu;
    std::multimap<size_t, Block> free_;  // keyed by size
    std::map<void*, Block> live_;        // handed out, not yet retired
    std::deque<Retiring> retiring_;
    std::vector<cudaEvent_t> events_;    // idle events for reuse
    int capacity = 16;
    int fail_records = 0;                // test hook
    size_t cached_bytes = 0;

    cudaEvent_t get_event()
    {
        if (!events_.empty()) {
            cudaEvent_t e = events_.back();
            events_.pop_back();
            return e;
        }
        cudaEvent_t e = nullptr;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        return e;
    }

    void to_free(const Block& b) { free_.emplace(b.bytes, b); }

    // query pending events in order; release the completed prefix and any
    // completed entry behind an incomplete one
    void drain_locked()
    {
        for (auto it = retiring_.begin(); it != retiring_.end();) {
            cudaError_t q = cudaEventQuery(it->ev);
            if (q == cudaSuccess) {
                to_free(it->b);
                events_.push_back(it->ev);
                count_pool(ST_RELEASED, 1);
                it = retiring_.erase(it);
            } else {
                if (q != cudaErrorNotReady) cudaGetLastError();
                ++it;
            }
        }
    }

    int wait_oldest_locked()
    {
        Retiring r = retiring_.front();
        retiring_.pop_front();
        cudaError_t e = cudaEventSynchronize(r.ev);
        count_pool(ST_EVWAIT, 1);
        if (e != cudaSuccess) {
            // cannot prove completion: leak the block rather than race
            cudaGetLastError();
            cached_bytes -= r.b.bytes;
            count_pool(ST_LEAKED, 1);
            return TROP_OK;
        }
        to_free(r.b);
        events_.push_back(r.ev);
        count_pool(ST_RELEASED, 1);
        return TROP_OK;
    }
};

Pool& pool()
{
    static Pool* p = [] {
        Pool* q = new Pool();
        if (const char* env = std::getenv("TROP_POOL_CAPACITY")) {
            int c = std::atoi(env);
            q->capacity = c < 1 ? 1 : c;
        }
        return q;
    }();
    return *p;
}

size_t round_bytes(size_t n)
{
    const size_t g = n < (size_t(1) << 20) ? 512 : (size_t(1) << 16);
    return (n + g - 1) / g * g;
}

}  // namespace

int CaptureArena::alloc(size_t bytes, void** out)
{
    *out = nullptr;
    const size_t want = (std::max<size_t>(bytes, 1) + 255) / 256 * 256;
    size_t off = top;
    for (auto it = free_.begin(); it != free_.end(); ++it) {
        if (it->second < want) continue;
        off = it->first;
        const size_t rest = it->second - want;
        free_.erase(it);
        if (rest) free_.emplace(off + want, rest);
        break;
    }
    if (off == top) {
        if (!measuring && top + want > capacity)
            return set_error(TROP_ERR_OOM, "capture arena exhausted (%zu + %zu > %zu bytes)", top, want, capacity);
        top += want;
        high = std::max(high, top);
    }
    used_.emplace(off, want);
    *out = reinterpret_cast<void*>(base + off);
    return TROP_OK;
}

bool CaptureArena::release(void* p)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    if (a < base) return false;
    auto it = used_.find(a - base);
    if (it == used_.end()) return false;
    size_t off = it->first, len = it->second;
    used_.erase(it);
    // coalesce with the free neighbours, then give the tail back to top
    auto nx = free_.lower_bound(off);
    if (nx != free_.end() && off + len == nx->first) {
        len += nx->second;
        nx = free_.erase(nx);
    }
    if (nx != free_.begin()) {
        auto pv = std::prev(nx);
        if (pv->first + pv->second == off) {
            off = pv->first;
            len += pv->second;
            free_.erase(pv);
        }
    }
    if (off + len == top) top = off;
    else free_.emplace(off, len);
    return true;
}

int pool_alloc(size_t bytes, cudaStream_t stream, void** out)
{
    if (t_arena) return t_arena->alloc(bytes, out);
    *out = nullptr;
    if (bytes == 0) bytes = 1;
    const size_t want = round_bytes(bytes);
    int dev = 0;
    cudaGetDevice(&dev);
    Pool& P = pool();
    std::lock_guard<std::mutex> lk(P.mu);
    count_pool(ST_ALLOC, 1);
    P.drain_locked();
    // best fit among free blocks of this device, at most 2x the request
    for (auto it = P.free_.lower_bound(want); it != P.free_.end() && it->first <= 2 * want; ++it) {
        if (it->second.device != dev) continue;
        Block b = it->second;
        P.free_.erase(it);
        P.live_[b.ptr] = b;
        count_pool(ST_HIT, 1);
        *out = b.ptr;
        return TROP_OK;
    }
    // a block still retiring on this same stream is safe by stream order
    for (auto it = P.retiring_.begin(); it != P.retiring_.end(); ++it) {
        if (it->stream != stream || it->b.device != dev) continue;
        if (it->b.bytes < want || it->b.bytes > 2 * want) continue;
        Block b = it->b;
        P.events_.push_back(it->ev);
        P.retiring_.erase(it);
        P.live_[b.ptr] = b;
        count_pool(ST_HIT, 1);
        *out = b.ptr;
        return TROP_OK;
    }
    void* p = nullptr;
    cudaError_t e = cudaMalloc(&p, want);
    if (e != cudaSuccess) {
        cudaGetLastError();
        // give back everything cached on this device and retry once
        while (!P.retiring_.empty()) P.wait_oldest_locked();
        for (auto it = P.free_.begin(); it != P.free_.end();) {
            if (it->second.device == dev) {
                cudaFree(it->second.ptr);
                P.cached_bytes -= it->second.bytes;
                it = P.free_.erase(it);
            } else {
                ++it;
            }
        }
        e = cudaMalloc(&p, want);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return set_error(TROP_ERR_OOM, "workspace allocation of %zu bytes failed: %s", want,
                             cudaGetErrorString(e));
        }
    }
    count_pool(ST_MALLOC, 1);
    P.cached_bytes += want;
    Block b{p, want, dev};
    P.live_[p] = b;
    *out = p;
    return TROP_OK;
}

void pool_retire(void* ptr, cudaStream_t stream)
{
    if (!ptr) return;
    if (t_arena) {
        t_arena->release(ptr);
        return;
    }
    Pool& P = pool();
    std::lock_guard<std::mutex> lk(P.mu);
    auto it = P.live_.find(ptr);
    if (it == P.live_.end()) return;
    Block b = it->second;
    P.live_.erase(it);
    count_pool(ST_RETIRED, 1);
    cudaEvent_t ev = nullptr;
    bool ok = false;
    if (P.fail_records > 0) {
        --P.fail_records;  // injected failure
    } else {
        ev = P.get_event();
        if (ev) {
            cudaError_t e = cudaEventRecord(ev, stream);
            if (e == cudaSuccess) ok = true;
            else {
                cudaGetLastError();
                P.events_.push_back(ev);
            }
        }
    }
    if (!ok) {  // no completion witness: leak rather than race
        P.cached_bytes -= b.bytes;
        count_pool(ST_LEAKED, 1);
        return;
    }
    while ((int)P.retiring_.size() >= P.capacity) P.wait_oldest_locked();
    P.retiring_.push_back(Retiring{b, ev, stream});
}

}  // namespace trop

// ====================================================================== C ABI
using namespace trop;

extern "C" int tropical_init(int device)
{
    clear_error();
    int cur = 0;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (device != cur) {
        e = cudaSetDevice(device);
        if (e != cudaSuccess) return cuda_error(e, "cudaSetDevice");
    }
    int rc = ensure_device(nullptr);
    if (device != cur) cudaSetDevice(cur);
    return rc;
}

// ------------------------------------------------------------------ per-stream tile tickets
// One zeroed uint32 array per (device, stream) for kernels whose CTAs count arrivals on a
// tile with atomics and leave every counter at zero when they end.  Launches on one stream
// run in order, so an array is never shared by two running launches.  Created on first use
// (zeroed on that stream, so it is ready before the launch that follows), replaced by a
// larger one when a launch needs more (the old array is freed by tropical_release_pool).
namespace {
struct Tickets {
    std::mutex mu;
    std::map<std::pair<int, cudaStream_t>, std::pair<uint32_t*, size_t>> arrays;
    std::vector<std::pair<int, uint32_t*>> retired;
};
Tickets& tickets()
{
    static Tickets* t = new Tickets();
    return *t;
}
}  // namespace

namespace {
struct Records {
    std::mutex mu;
    std::map<std::pair<int, cudaStream_t>, trop::LaunchRecord> last;
};
Records& records()
{
    static Records* r = new Records();
    return *r;
}
}  // namespace

trop::LaunchRecord trop::stream_record(cudaStream_t s)
{
    LaunchRecord r{};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return r;
    }
    Records& R = records();
    std::lock_guard<std::mutex> lk(R.mu);
    auto it = R.last.find(std::make_pair(dev, s));
    if (it != R.last.end()) r = it->second;
    return r;
}

void trop::set_stream_record(cudaStream_t s, const LaunchRecord& r)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    Records& R = records();
    std::lock_guard<std::mutex> lk(R.mu);
    R.last[std::make_pair(dev, s)] = r;
}

int trop::stream_tickets(cudaStream_t s, size_t count, uint32_t** out)
{
    *out = nullptr;
    if (CaptureArena* a = capture_arena()) {
        // captured: counters of the plan's own, zeroed by a memset node ahead of their kernel
        void* p = nullptr;
        TROP_TRY(a->alloc(count * sizeof(uint32_t), &p));
        if (!a->measuring) {
            cudaError_t e = cudaMemsetAsync(p, 0, count * sizeof(uint32_t), s);
            if (e != cudaSuccess) return cuda_error(e, "cudaMemsetAsync (captured tickets)");
        }
        *out = static_cast<uint32_t*>(p);
        return TROP_OK;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    Tickets& T = tickets();
    std::lock_guard<std::mutex> lk(T.mu);
    auto key = std::make_pair(dev, s);
    auto it = T.arrays.find(key);
    if (it != T.arrays.end() && it->second.second >= count) {
        *out = it->second.first;
        return TROP_OK;
    }
    const size_t n = (count + 4095) / 4096 * 4096;
    uint32_t* p = nullptr;
    e = cudaMalloc(&p, n * sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_error(e, "cudaMalloc (tile tickets)");
    e = cudaMemsetAsync(p, 0, n * sizeof(uint32_t), s);
    if (e != cudaSuccess) {
        cudaFree(p);
        return cuda_error(e, "cudaMemsetAsync (tile tickets)");
    }
    if (it != T.arrays.end()) {
        T.retired.emplace_back(dev, it->second.first);
        it->second = std::make_pair(p, n);
    } else {
        T.arrays.emplace(key, std::make_pair(p, n));
    }
    *out = p;
    return TROP_OK;
}

extern "C" int tropical_sync_pool(void)
{
    clear_error();
    {
        Pool& P = pool();
        std::lock_guard<std::mutex> lk(P.mu);
        while (!P.retiring_.empty()) P.wait_oldest_locked();
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return TROP_OK;
    }
    return dev >= 0 && dev < 64 ? take_device_error(dev) : TROP_OK;
}

extern "C" int tropical_debug_bounds_report(unsigned int* count, int* line, uint64_t* addr, int reset)
{
    clear_error();
    if (!count) return set_error(TROP_ERR_INVALID_ARG, "count pointer is NULL");
    *count = 0;
    if (line) *line = 0;
    if (addr) *addr = 0;
#if TROP_DEBUG_BOUNDS
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return set_error(TROP_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    volatile uint32_t* h = g_err_host[dev].load(std::memory_order_acquire);
    if (!h) return TROP_OK;  // nothing launched with a record yet
    *count = h[4];
    if (line) *line = (int)h[5];
    if (addr) *addr = (uint64_t)h[6] | ((uint64_t)h[7] << 32);
    if (reset) h[4] = h[5] = h[6] = h[7] = 0;
    return TROP_OK;
#else
    (void)reset;
    return set_error(TROP_ERR_UNSUPPORTED, "this library was built without bounds checks (TROP_DEBUG_BOUNDS=0)");
#endif
}

extern "C" int tropical_debug_bounds_trim(int64_t bytes)
{
    clear_error();
    if (bytes < 0) return set_error(TROP_ERR_INVALID_ARG, "trim of %lld bytes", (long long)bytes);
#if TROP_DEBUG_BOUNDS
    g_span_trim.store(bytes, std::memory_order_relaxed);
    return TROP_OK;
#else
    return set_error(TROP_ERR_UNSUPPORTED, "this library was built without bounds checks (TROP_DEBUG_BOUNDS=0)");
#endif
}

extern "C" void tropical_debug_set_wait_mode(int mode)
{
    g_wait_mode.store(mode < 0 || mode > 2 ? 0 : mode, std::memory_order_relaxed);
}

extern "C" int tropical_release_pool(void)
{
    clear_error();
    Pool& P = pool();
    std::lock_guard<std::mutex> lk(P.mu);
    while (!P.retiring_.empty()) P.wait_oldest_locked();
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto& kv : P.free_) {
        cudaSetDevice(kv.second.device);
        cudaFree(kv.second.ptr);
        P.cached_bytes -= kv.second.bytes;
    }
    {
        // tile tickets: every launch that used them has finished (the caller synchronised)
        Tickets& T = tickets();
        std::lock_guard<std::mutex> lt(T.mu);
        for (auto& kv : T.arrays) {
            cudaSetDevice(kv.first.first);
            cudaFree(kv.second.first);
        }
        for (auto& r : T.retired) {
            cudaSetDevice(r.first);
            cudaFree(r.second);
        }
        T.arrays.clear();
        T.retired.clear();
    }
    cudaSetDevice(cur);
    P.free_.clear();
    for (cudaEvent_t e : P.events_) cudaEventDestroy(e);
    P.events_.clear();
    return TROP_OK;
}

extern "C" int tropical_stats(trop_stats* out)
{
    if (!out) return set_error(TROP_ERR_INVALID_ARG, "stats pointer is NULL");
    out->module_inits = c_module_inits.load();
    out->kernel_launches = c_launches.load();
    out->pool_allocs = c_pool[ST_ALLOC].load();
    out->pool_hits = c_pool[ST_HIT].load();
    out->pool_device_mallocs = c_pool[ST_MALLOC].load();
    out->pool_retired = c_pool[ST_RETIRED].load();
    out->pool_released = c_pool[ST_RELEASED].load();
    out->pool_event_waits = c_pool[ST_EVWAIT].load();
    out->pool_leaked = c_pool[ST_LEAKED].load();
    out->plan_cache_hits = c_plan_hits.load();
    out->plan_cache_misses = c_plan_misses.load();
    out->gemm_early_starts = c_early.load();
    {
        Pool& P = pool();
        std::lock_guard<std::mutex> lk(P.mu);
        out->pool_bytes_cached = (int64_t)P.cached_bytes;
    }
    out->stream_syncs = c_stream_syncs.load();
    return TROP_OK;
}

extern "C" void tropical_reset_stats(void)
{
    c_launches = 0;
    c_stream_syncs = 0;
    c_plan_hits = 0;
    c_plan_misses = 0;
    c_early = 0;
    for (int i = 0; i < 7; ++i) c_pool[i] = 0;  // ST_BYTES is derived, module_inits kept
}

extern "C" const char* tropical_last_error(void) { return g_last_error.c_str(); }

extern "C" int tropical_version(void) { return 2; }

extern "C" void tropical_debug_fail_next_event_records(int count)
{
    Pool& P = pool();
    std::lock_guard<std::mutex> lk(P.mu);
    P.fail_records = count < 0 ? 0 : count;
}

extern "C" void tropical_set_pool_capacity(int capacity)
{
    Pool& P = pool();
    std::lock_guard<std::mutex> lk(P.mu);
    P.capacity = capacity < 1 ? 1 : capacity;
}
