// bounds.h -- the bounds-checked debug build (TROP_DEBUG_BOUNDS=1).
//
// compute-sanitizer is not available to this library's tests, so a debug build of the library
// checks memory accesses itself: every launch carries, for each tensor a kernel touches, the
// byte range [lo, hi) its view can address (from extents and strides, computed on the host), and
// each global load, store or copy a kernel issues is tested against its tensor's range first.
// An access outside it is skipped (a load yields 0, a copy fills zeros, a store is dropped) and
// the first violation -- the source file and line of the check and the address -- is recorded
// in host-mapped memory with a count, which tropical_debug_bounds_report reads.  Nothing traps: a wrong index
// shows up as a report and as results that differ from the oracle's.
//
// In the normal build TROP_DEBUG_BOUNDS is 0: Span is an empty struct, the checks are the
// constant true, and the kernels compile exactly as without them.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#ifndef TROP_DEBUG_BOUNDS
#define TROP_DEBUG_BOUNDS 0
#endif

namespace trop {

#if TROP_DEBUG_BOUNDS
// The violation record lives in the device's host-mapped word block (runtime.cpp): count, then
// the first violation's source line and address (low, high word).  Every span carries it.
struct Span {
    const char* lo;
    const char* hi;  // one past the last addressable byte
    unsigned* rep;
};
unsigned* bounds_record();  // this device's record (host-mapped); nullptr if unavailable
int64_t bounds_span_trim();  // test hook: bytes cut from the top of each span (normally 0)
#else
struct Span {};
#endif

// The byte range of a strided view: base + [min offset, max offset] elements (strides may be
// negative or zero), or an empty range for an empty view.
inline Span span_of(const void* base, size_t elem_bytes, int rank, const int64_t* size, const int64_t* stride)
{
#if TROP_DEBUG_BOUNDS
    int64_t lo = 0, hi = 0;
    for (int i = 0; i < rank; ++i) {
        if (size[i] <= 0) return Span{nullptr, nullptr, bounds_record()};
        const int64_t e = (size[i] - 1) * stride[i];
        if (e < 0) lo += e;
        else hi += e;
    }
    const char* b = static_cast<const char*>(base);
    if (!b) return Span{nullptr, nullptr, bounds_record()};
    return Span{b + lo * (int64_t)elem_bytes, b + (hi + 1) * (int64_t)elem_bytes - bounds_span_trim(), bounds_record()};
#else
    (void)base, (void)elem_bytes, (void)rank, (void)size, (void)stride;
    return Span{};
#endif
}
// a contiguous block of `bytes` at p
inline Span span_bytes(const void* p, size_t bytes)
{
#if TROP_DEBUG_BOUNDS
    const char* b = static_cast<const char*>(p);
    return b ? Span{b, b + bytes - bounds_span_trim(), bounds_record()} : Span{nullptr, nullptr, bounds_record()};
#else
    (void)p, (void)bytes;
    return Span{};
#endif
}

#ifdef __CUDACC__
#if TROP_DEBUG_BOUNDS
__device__ __forceinline__ bool bounds_ok(const void* p, int bytes, const Span& s, int line)
{
    const char* c = static_cast<const char*>(p);
    if (c >= s.lo && c + bytes <= s.hi) return true;
    if (s.rep && atomicAdd_system(&s.rep[0], 1u) == 0u) {
        const unsigned long long a = (unsigned long long)(uintptr_t)p;
        s.rep[1] = (unsigned)line;
        s.rep[2] = (unsigned)a;
        s.rep[3] = (unsigned)(a >> 32);
        __threadfence_system();
    }
    return false;
}
// the record's location word: the translation unit's TROP_TU id (set before including this
// header) in the high half, the source line in the low half
#ifndef TROP_TU
#define TROP_TU 0
#endif
#define TROP_IN(ptr, bytes, span) ::trop::bounds_ok((ptr), (bytes), (span), (TROP_TU << 16) | __LINE__)
#else
#define TROP_IN(ptr, bytes, span) true
#endif
#endif

}  // namespace trop
