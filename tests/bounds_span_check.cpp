// Host check of the bounds-checked build's span arithmetic (csrc/bounds.h): the byte range a
// strided view can address, for positive, negative, zero and unit strides and empty views.
// Built with -DTROP_DEBUG_BOUNDS=1 and run by tests/test_bounds_host.py; prints "ok" or the
// first mismatch and exits non-zero.  No GPU is touched: bounds_record() is a stand-in here.
#include <cstdio>
#include <cstdint>

#include "bounds.h"

namespace trop {
static unsigned g_record[4];
unsigned* bounds_record() { return g_record; }
int64_t bounds_span_trim() { return 0; }
}  // namespace trop

static int check(const char* name, const trop::Span& s, const char* base, long lo, long hi)
{
    if (s.lo != base + lo || s.hi != base + hi || s.rep == nullptr) {
        std::printf("%s: got [%ld, %ld), want [%ld, %ld)\n", name, (long)(s.lo - base), (long)(s.hi - base), lo, hi);
        return 1;
    }
    return 0;
}

int main()
{
    alignas(16) static char buf[1 << 16];
    const char* b = buf + 4096;
    int bad = 0;
    {   // contiguous 3 x 4 x 5 floats: 60 elements
        const int64_t sz[3] = {3, 4, 5}, st[3] = {20, 5, 1};
        bad |= check("contiguous", trop::span_of(b, 4, 3, sz, st), b, 0, 240);
    }
    {   // transposed view of a 7 x 9 matrix (strides 1, 7): the last element is offset 62
        const int64_t sz[2] = {9, 7}, st[2] = {1, 9};
        bad |= check("transposed", trop::span_of(b, 8, 2, sz, st), b, 0, 8 * 63);
    }
    {   // negative stride: elements at 0, -3, -6, -9 (and a second axis of stride 10, 2 long)
        const int64_t sz[2] = {4, 2}, st[2] = {-3, 10};
        bad |= check("negative", trop::span_of(b, 4, 2, sz, st), b, -36, 44);
    }
    {   // broadcast (stride 0) axis and a unit axis
        const int64_t sz[3] = {5, 1, 6}, st[3] = {0, 1000, 2};
        bad |= check("broadcast", trop::span_of(b, 2, 3, sz, st), b, 0, 22);
    }
    {   // an empty view addresses nothing
        const int64_t sz[2] = {3, 0}, st[2] = {1, 3};
        const trop::Span s = trop::span_of(b, 4, 2, sz, st);
        if (s.lo != nullptr || s.hi != nullptr) {
            std::printf("empty: want a null range\n");
            bad = 1;
        }
    }
    {   // rank 0: one element
        bad |= check("scalar", trop::span_of(b, 8, 0, nullptr, nullptr), b, 0, 8);
    }
    bad |= check("bytes", trop::span_bytes(b, 100), b, 0, 100);
    if (trop::span_bytes(nullptr, 100).lo != nullptr) {
        std::printf("null block: want a null range\n");
        bad = 1;
    }
    if (!bad) std::printf("ok\n");
    return bad;
}
