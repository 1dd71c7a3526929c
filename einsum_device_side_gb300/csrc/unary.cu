// unary.cu -- device-side permute / diagonal gather / trace reduce.
//
// The two kernels of omeinsum-rs issue #52 ("GPU tropical path: keep tensors
// device-resident + device-side permute", section "Resolved design for step
// 3"): (a) an N-d permute / strided gather, and (b) a diagonal/trace gather
// with the tropical max/min fused into the gather.  A repeated label is a
// view whose stride is the sum of the repeated axes' strides, so (a) also
// performs diagonal gathers; (b) reduces the labels absent from the output.
//
// Kernel (a) comes in three shapes, chosen at launch after merging axes that
// stay adjacent:
//   * k_copy_rows   the output's fastest axis is also the input's: rows are
//                   copied with 16-byte vectors;
//   * k_transpose   the fastest axes differ: a tile of 4096 elements (2048
//                   for 8-byte types) spanning the input-fastest axis chain x
//                   the output-fastest chain, its shape fitted to short
//                   chains (16x256 for a 16^6 tensor), is staged transposed
//                   through shared memory whose rows are XOR-swizzled, so the
//                   reads and the 16-byte vector writes are both coalesced and
//                   free of bank conflicts (the tiled transpose the issue
//                   names as the later ~2.6x step);
//   * k_gather      anything else: one thread per output element, decoding
//                   its index against the shape (the GPUArrays.jl scheme the
//                   issue describes as the first cut).
// A second, int32 tensor (an argmax) can ride along through the same index
// computation, so a result and its argmax are permuted identically.
#include <cuda_runtime.h>

#include <cstdint>
#include <algorithm>
#include <cstring>

#define TROP_TU 1  // this file's id in a bounds-violation record
#include "internal.h"

namespace trop {

namespace {

constexpr int NT = 256;  // threads per block for the unary kernels

// The axes a row-copy or transpose block iterates over, at most R of them.  Kernels come in
// two capacities: REST_SMALL axes (nearly every merged layout) and MAXR; the small one keeps the
// launch's parameter block near 400 bytes instead of 1.4 KB, which is measurable host time per
// launch (about 0.25 us on GB300).
constexpr int REST_SMALL = 8;
template <int R>
struct RestDims {
    int rank;
    FastDiv div[R];
    int64_t s_in[R];
    int64_t s_out[R];
    int64_t s_in2[R];
    int64_t s_out2[R];
};

// decode idx (< 2^31) over rest dims, last fastest
template <int R>
__device__ __forceinline__ void decode_rest(const RestDims<R>& r, uint32_t idx, int64_t& oi, int64_t& oo,
                                            int64_t& oi2, int64_t& oo2)
{
    oi = oo = oi2 = oo2 = 0;
    for (int d = r.rank - 1; d >= 0; --d) {
        uint32_t q = fdiv(idx, r.div[d]);
        uint32_t c = idx - q * r.div[d].d;
        idx = q;
        oi += (int64_t)c * r.s_in[d];
        oo += (int64_t)c * r.s_out[d];
        oi2 += (int64_t)c * r.s_in2[d];
        oo2 += (int64_t)c * r.s_out2[d];
    }
}

// ------------------------------------------------------------------ gather
struct GatherParams {
    int rank;
    int64_t total;
    int64_t size[MAXR];
    int64_t s_in[MAXR], s_out[MAXR], s_in2[MAXR], s_out2[MAXR];
#if TROP_DEBUG_BOUNDS
    Span sp[4];  // in, out, in2, out2
#endif
};

template <typename T, bool PAIR>
__global__ void k_gather(const T* __restrict__ in, T* __restrict__ out, const int32_t* __restrict__ in2,
                         int32_t* __restrict__ out2, GatherParams p)
{
    pdl_wait();
    pdl_signal();
    for (int64_t o = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; o < p.total;
         o += (int64_t)gridDim.x * blockDim.x) {
        int64_t rem = o, oi = 0, oo = 0, oi2 = 0, oo2 = 0;
        for (int d = p.rank - 1; d >= 0; --d) {
            int64_t c = rem % p.size[d];
            rem /= p.size[d];
            oi += c * p.s_in[d];
            oo += c * p.s_out[d];
            if (PAIR) {
                oi2 += c * p.s_in2[d];
                oo2 += c * p.s_out2[d];
            }
        }
        if (TROP_IN(in + oi, sizeof(T), p.sp[0]) && TROP_IN(out + oo, sizeof(T), p.sp[1])) out[oo] = in[oi];
        if (PAIR && TROP_IN(in2 + oi2, 4, p.sp[2]) && TROP_IN(out2 + oo2, 4, p.sp[3])) out2[oo2] = in2[oi2];
    }
}

// ------------------------------------------------------------------ row copy
template <int R>
struct RowParams {
    uint32_t L;      // row length in elements
    uint32_t Lv;     // row length in vectors
    uint32_t total;  // rows * Lv
    FastDiv divLv;
    RestDims<R> rest;
#if TROP_DEBUG_BOUNDS
    Span sp[4];  // in, out, in2, out2
#endif
};

template <typename T, typename V, bool PAIR, int R>
__global__ void k_copy_rows(const T* __restrict__ in, T* __restrict__ out, const int32_t* __restrict__ in2,
                            int32_t* __restrict__ out2, RowParams<R> p)
{
    pdl_wait();
    pdl_signal();
    constexpr int W = sizeof(V) / sizeof(T);
    for (uint32_t e = blockIdx.x * blockDim.x + threadIdx.x; e < p.total; e += gridDim.x * blockDim.x) {
        uint32_t row = fdiv(e, p.divLv);
        uint32_t col = (e - row * p.Lv) * W;
        int64_t oi, oo, oi2, oo2;
        decode_rest(p.rest, row, oi, oo, oi2, oo2);
        if (TROP_IN(in + oi + col, sizeof(V), p.sp[0]) && TROP_IN(out + oo + col, sizeof(V), p.sp[1]))
            *reinterpret_cast<V*>(out + oo + col) = __ldg(reinterpret_cast<const V*>(in + oi + col));
        if (PAIR) {
            // the companion is int32: copy W of them element-wise
#pragma unroll
            for (int q = 0; q < W; ++q)
                if (TROP_IN(in2 + oi2 + col + q, 4, p.sp[2]) && TROP_IN(out2 + oo2 + col + q, 4, p.sp[3]))
                    out2[oo2 + col + q] = __ldg(in2 + oi2 + col + q);
        }
    }
}

// ------------------------------------------------------------------ transpose
// Tile over two axis chains: GI = input-fastest chain (contiguous in the
// input), GJ = output-fastest chain (contiguous in the output), and TB
// consecutive indices of the remaining axes.  A tile is TB x TJ x TI = TILE
// elements (powers of two); its shape adapts when a chain is short (16 x 256
// when the input's fastest axis has 16 elements; TB > 1 stacks several
// outer-axis slices when both chains are short), so every tile stays full.
template <int R>
struct TransParams {
    uint32_t nI, nJ, nR;         // flattened chain extents, remaining-axes count
    uint32_t TI, TJ, TB;         // tile shape (powers of two)
    uint32_t lTI, lTJ, lTB;      // their log2
    uint32_t tilesI, tilesJ, tilesR;
    uint32_t tiles;              // tilesI * tilesJ * tilesR
    FastDiv div_tilesI, div_tilesJ;
    int gi_rank, gj_rank;
    FastDiv gi_div[4], gj_div[4];
    int64_t gi_s_out[4], gi_s_out2[4];  // output strides of GI axes (last = fastest in input)
    int64_t gj_s_in[4], gj_s_in2[4];    // input strides of GJ axes (last = fastest in output)
    int vec_in;                          // input rows 16-byte aligned for vector loads
    int vec_out;                         // output rows 16-byte aligned for vector stores
    int sw;                              // shared-memory swizzle step (see tile_pos)
    RestDims<R> rest;
#if TROP_DEBUG_BOUNDS
    Span sp[4];  // in, out, in2, out2
#endif
};

// Shared-memory slot of tile element (x, c): x = slice * TJ + GJ index, in [0, L) with
// L = TB * TJ; c = GI index.  The tile is held transposed, in rows of L elements per GI
// index, and a row's x is XOR-ed with a multiple of the vector width W below 32 that grows
// with c / W.  The loader's scalar stores -- lanes spread over W-wide runs of c and over
// consecutive x -- then land in distinct banks, and the storer's W-wide reads along x stay
// contiguous and 16-byte aligned.
template <int W>
__device__ __forceinline__ int tile_pos(int x, int c, int L, int sw)
{
    return c * L + (x ^ (((c / W) * sw) & 31 & (L - 1)));
}

template <int T_BYTES>
struct TileCfg {
    static constexpr int TILE = T_BYTES == 8 ? 2048 : 4096;  // elements per tile
    static constexpr int TJMAX = 512;
    static constexpr int TIMAX = 64;
    static constexpr int TBMAX = 64;
};

// Residency of the transpose, which is bound by load latency: registers capped for 6 CTAs
// (48 warps) per SM and a shared-memory carveout that fits them while leaving L1 room for
// the loads in flight (measured on GB300: a 16^6 f32 'abcdef->afbcde' took 31.4 us at
// 4 CTAs/SM, 25.1 us here; the maximum carveout starved L1 and doubled the time).
#ifndef TROP_TRANSPOSE_MINB
#define TROP_TRANSPOSE_MINB 6
#endif
#ifndef TROP_TRANSPOSE_CARVEOUT
#define TROP_TRANSPOSE_CARVEOUT 60
#endif
template <typename T, bool PAIR, int R>
__global__ void __launch_bounds__(NT, PAIR ? 3 : TROP_TRANSPOSE_MINB) k_transpose(const T* __restrict__ in, T* __restrict__ out,
                                                  const int32_t* __restrict__ in2, int32_t* __restrict__ out2,
                                                  TransParams<R> p)
{
    pdl_wait();
    pdl_signal();
    using Cfg = TileCfg<sizeof(T)>;
    using V = typename std::conditional<sizeof(T) == 8, longlong2, int4>::type;
    constexpr int W = 16 / sizeof(T);
    constexpr int VPT = Cfg::TILE / W / NT;  // vectors per thread in a full tile
    __shared__ __align__(16) T tile[Cfg::TILE];  // TI rows of L = TB*TJ, swizzled (tile_pos)
    __shared__ __align__(16) int32_t tile2[PAIR ? Cfg::TILE : 1];
    __shared__ int64_t row_in[Cfg::TJMAX], row_in2[PAIR ? Cfg::TJMAX : 1];     // input offset of a GJ index
    __shared__ int64_t row_out[Cfg::TIMAX], row_out2[PAIR ? Cfg::TIMAX : 1];   // output offset of a GI index
    __shared__ int64_t bin_s[Cfg::TBMAX], bout_s[Cfg::TBMAX];                   // offsets of the TB outer slices
    __shared__ int64_t bin2_s[PAIR ? Cfg::TBMAX : 1], bout2_s[PAIR ? Cfg::TBMAX : 1];
    const int TI = (int)p.TI, TJ = (int)p.TJ, TB = (int)p.TB, L = TB * TJ, sw = p.sw;
    const int lTI = (int)p.lTI, lTJ = (int)p.lTJ;

    for (uint32_t t = blockIdx.x; t < p.tiles; t += gridDim.x) {
        const uint32_t q1 = fdiv(t, p.div_tilesI);
        const uint32_t ti = t - q1 * p.tilesI;
        const uint32_t q2 = fdiv(q1, p.div_tilesJ);
        const uint32_t tj = q1 - q2 * p.tilesJ;
        const uint32_t r0 = q2 << p.lTB;
        const uint32_t i0 = ti * TI, j0 = tj * TJ;
        for (int x = threadIdx.x; x < TJ + TI + TB; x += NT) {
            if (x < TJ) {
                uint32_t j = j0 + x, rem = j < p.nJ ? j : 0;
                int64_t off = 0, off2 = 0;
                for (int d = p.gj_rank - 1; d >= 0; --d) {
                    uint32_t q = fdiv(rem, p.gj_div[d]);
                    uint32_t c = rem - q * p.gj_div[d].d;
                    rem = q;
                    off += (int64_t)c * p.gj_s_in[d];
                    off2 += (int64_t)c * p.gj_s_in2[d];
                }
                row_in[x] = off;
                if (PAIR) row_in2[PAIR ? x : 0] = off2;
            } else if (x < TJ + TI) {
                int y = x - TJ;
                uint32_t i = i0 + y, rem = i < p.nI ? i : 0;
                int64_t off = 0, off2 = 0;
                for (int d = p.gi_rank - 1; d >= 0; --d) {
                    uint32_t q = fdiv(rem, p.gi_div[d]);
                    uint32_t c = rem - q * p.gi_div[d].d;
                    rem = q;
                    off += (int64_t)c * p.gi_s_out[d];
                    off2 += (int64_t)c * p.gi_s_out2[d];
                }
                row_out[y] = off;
                if (PAIR) row_out2[PAIR ? y : 0] = off2;
            } else {
                const int b = x - TJ - TI;
                const uint32_t rr = r0 + b;
                int64_t a, bb, c, d;
                decode_rest(p.rest, rr < p.nR ? rr : 0, a, bb, c, d);
                bin_s[b] = a;
                bout_s[b] = bb;
                if (PAIR) {
                    bin2_s[PAIR ? b : 0] = c;
                    bout2_s[PAIR ? b : 0] = d;
                }
            }
        }
        __syncthreads();
        const bool full = i0 + TI <= p.nI && j0 + TJ <= p.nJ && r0 + TB <= p.nR;
        const int lvi = lTI - (W == 4 ? 2 : 1);  // log2 of vectors per input row
        // load: rows = (slice, GJ index) (strided in the input), columns = GI index (contiguous)
        // (the int32 companion of a pair rides in the same vectors when T is 4 bytes wide)
        constexpr bool VPAIR = !PAIR || sizeof(T) == 4;
        if (VPAIR && full && p.vec_in && TI >= W && (TB << (lTJ + lTI)) == Cfg::TILE) {
            V v[VPT];
            int4 v2[PAIR ? VPT : 1];
#pragma unroll
            for (int u = 0; u < VPT; ++u) {  // all loads in flight before any shared store
                const int e = threadIdx.x + u * NT;
                const int c = (e & ((1 << lvi) - 1)) * W, rj = e >> lvi;
                const int r = rj & (TJ - 1), b = rj >> lTJ;
                const T* src = in + bin_s[b] + row_in[r] + i0 + c;
                v[u] = TROP_IN(src, sizeof(V), p.sp[0]) ? __ldg(reinterpret_cast<const V*>(src)) : V{};
                if (PAIR) {
                    const int32_t* src2 = in2 + bin2_s[PAIR ? b : 0] + row_in2[PAIR ? r : 0] + i0 + c;
                    v2[PAIR ? u : 0] = TROP_IN(src2, 16, p.sp[2]) ? __ldg(reinterpret_cast<const int4*>(src2)) : int4{};
                }
            }
#pragma unroll
            for (int u = 0; u < VPT; ++u) {
                const int e = threadIdx.x + u * NT;
                const int c = (e & ((1 << lvi) - 1)) * W, rj = e >> lvi;
                const T* pv = reinterpret_cast<const T*>(&v[u]);
#pragma unroll
                for (int q = 0; q < W; ++q) tile[tile_pos<W>(rj, c + q, L, sw)] = pv[q];
                if (PAIR) {
                    const int32_t* pv2 = reinterpret_cast<const int32_t*>(&v2[PAIR ? u : 0]);
#pragma unroll
                    for (int q = 0; q < W; ++q) tile2[PAIR ? tile_pos<W>(rj, c + q, L, sw) : 0] = pv2[q];
                }
            }
        } else {
            for (int e = threadIdx.x; e < TB * TJ * TI; e += NT) {
                const int c = e & (TI - 1), rj = e >> lTI;
                const int r = rj & (TJ - 1), b = rj >> lTJ;
                if (r0 + b < p.nR && j0 + r < p.nJ && i0 + c < p.nI) {
                    const T* src = in + bin_s[b] + row_in[r] + i0 + c;
                    tile[tile_pos<W>(rj, c, L, sw)] = TROP_IN(src, sizeof(T), p.sp[0]) ? __ldg(src) : T{};
                    if (PAIR) {
                        const int32_t* src2 = in2 + bin2_s[PAIR ? b : 0] + row_in2[PAIR ? r : 0] + i0 + c;
                        tile2[PAIR ? tile_pos<W>(rj, c, L, sw) : 0] = TROP_IN(src2, 4, p.sp[2]) ? __ldg(src2) : 0;
                    }
                }
            }
        }
        __syncthreads();
        // store: rows = (slice, GI index) (strided in the output), columns = GJ index (contiguous)
        if (VPAIR && full && p.vec_out && TJ >= W) {
            const int lvj = lTJ - (W == 4 ? 2 : 1);
            for (int e = threadIdx.x; e < (TB * TI) << lvj; e += NT) {
                const int c = (e & ((1 << lvj) - 1)) * W, ri = e >> lvj;
                const int r = ri & (TI - 1), b = ri >> lTI;
                const int at = tile_pos<W>((b << lTJ) + c, r, L, sw);
                const V v = *reinterpret_cast<const V*>(&tile[at]);
                T* dst = out + bout_s[b] + row_out[r] + j0 + c;
                if (TROP_IN(dst, sizeof(V), p.sp[1])) *reinterpret_cast<V*>(dst) = v;
                if (PAIR) {
                    int32_t* dst2 = out2 + bout2_s[PAIR ? b : 0] + row_out2[PAIR ? r : 0] + j0 + c;
                    if (TROP_IN(dst2, 16, p.sp[3]))
                        *reinterpret_cast<int4*>(dst2) = *reinterpret_cast<const int4*>(&tile2[PAIR ? at : 0]);
                }
            }
        } else {
            for (int e = threadIdx.x; e < TB * TJ * TI; e += NT) {
                const int c = e & (TJ - 1), ri = e >> lTJ;
                const int r = ri & (TI - 1), b = ri >> lTI;
                if (r0 + b < p.nR && i0 + r < p.nI && j0 + c < p.nJ) {
                    T* dst = out + bout_s[b] + row_out[r] + j0 + c;
                    if (TROP_IN(dst, sizeof(T), p.sp[1])) *dst = tile[tile_pos<W>((b << lTJ) + c, r, L, sw)];
                    if (PAIR) {
                        int32_t* dst2 = out2 + bout2_s[PAIR ? b : 0] + row_out2[PAIR ? r : 0] + j0 + c;
                        if (TROP_IN(dst2, 4, p.sp[3])) *dst2 = tile2[PAIR ? tile_pos<W>((b << lTJ) + c, r, L, sw) : 0];
                    }
                }
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ reduce
template <int SR, typename T>
struct Semi;

template <int SR>
struct Semi<SR, float> {
    __device__ static float zero() { return SR == TROP_MAXPLUS ? -INFINITY : SR == TROP_MINPLUS ? INFINITY : 0.0f; }
    __device__ static bool better(float a, float b) { return SR == TROP_MINPLUS ? a < b : a > b; }
};
template <int SR>
struct Semi<SR, int32_t> {
    __device__ static int32_t zero() { return SR == TROP_MAXPLUS ? INT32_MIN : SR == TROP_MINPLUS ? INT32_MAX : 0; }
    __device__ static bool better(int32_t a, int32_t b) { return SR == TROP_MINPLUS ? a < b : a > b; }
};
// binary64: compared through the order-preserving signed-integer image of the
// double (integer lanes, not the narrow binary64 pipe); exact for non-NaN values
template <int SR>
struct Semi<SR, double> {
    __device__ static double zero() { return SR == TROP_MAXPLUS ? -INFINITY : SR == TROP_MINPLUS ? INFINITY : 0.0; }
    __device__ static long long key(double x)
    {
        const long long b = __double_as_longlong(x);
        return b ^ (long long)((unsigned long long)(b >> 63) >> 1);
    }
    __device__ static bool better(double a, double b) { return SR == TROP_MINPLUS ? key(a) < key(b) : key(a) > key(b); }
};
template <int SR>
struct Semi<SR, int64_t> {
    __device__ static int64_t zero() { return SR == TROP_MAXPLUS ? INT64_MIN : SR == TROP_MINPLUS ? INT64_MAX : 0; }
    __device__ static bool better(int64_t a, int64_t b) { return SR == TROP_MINPLUS ? a < b : a > b; }
};

constexpr int64_t NO_INDEX = INT64_MAX;

struct RedParams {
    int64_t n_out;
    int64_t R;  // reduced extent
    int out_rank;
    int64_t out_size[MAXR], out_s_in[MAXR], out_s_out[MAXR], out_s_arg[MAXR];
    int red_rank;
    int64_t red_size[MAXR], red_s_in[MAXR];
    int64_t nsplit;  // chunks per output (block kernel)
    int64_t chunk;   // reduced elements per chunk
#if TROP_DEBUG_BOUNDS
    Span sp[5];  // in, out, arg, part_v, part_i
#endif
};

// checked forms of the reduce kernels' global accesses (plain accesses in the normal build)
template <typename T>
__device__ __forceinline__ T red_load(const T* at, const RedParams& p)
{
    return TROP_IN(at, sizeof(T), p.sp[0]) ? __ldg(at) : T{};
}
template <typename T>
__device__ __forceinline__ void red_store(T* out, int64_t oo, T v, int32_t* arg, int64_t oa, int32_t idx,
                                          const RedParams& p)
{
    if (TROP_IN(out + oo, sizeof(T), p.sp[1])) out[oo] = v;
    if (arg && TROP_IN(arg + oa, 4, p.sp[2])) arg[oa] = idx;
}
// a merged first index: NO_INDEX when nothing beat the zero, stored as 0
__device__ __forceinline__ int32_t final_index(int64_t idx) { return idx == NO_INDEX ? 0 : (int32_t)idx; }

__device__ __forceinline__ void out_offsets(const RedParams& p, int64_t o, int64_t& oi, int64_t& oo, int64_t& oa)
{
    oi = oo = oa = 0;
    for (int d = p.out_rank - 1; d >= 0; --d) {
        int64_t c = o % p.out_size[d];
        o /= p.out_size[d];
        oi += c * p.out_s_in[d];
        oo += c * p.out_s_out[d];
        oa += c * p.out_s_arg[d];
    }
}

__device__ __forceinline__ int64_t red_offset(const RedParams& p, int64_t r)
{
    if (p.red_rank == 1) return r * p.red_s_in[0];
    int64_t off = 0;
    for (int d = p.red_rank - 1; d >= 0; --d) {
        int64_t c = r % p.red_size[d];
        r /= p.red_size[d];
        off += c * p.red_s_in[d];
    }
    return off;
}

// one thread per output element, ascending reduced index, strict update
template <int SR, typename T>
__global__ void k_reduce_thread(const T* __restrict__ in, T* __restrict__ out, int32_t* __restrict__ arg,
                                RedParams p)
{
    pdl_wait();
    pdl_signal();
    using S = Semi<SR, T>;
    for (int64_t o = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; o < p.n_out;
         o += (int64_t)gridDim.x * blockDim.x) {
        int64_t oi, oo, oa;
        out_offsets(p, o, oi, oo, oa);
        T best = S::zero();
        int64_t idx = 0;
        for (int64_t r = 0; r < p.R; ++r) {
            T v = red_load(in + oi + red_offset(p, r), p);
            if (S::better(v, best)) {
                best = v;
                idx = r;
            }
        }
        red_store(out, oo, best, arg, oa, (int32_t)idx, p);
    }
}

// block per (output, chunk); writes the final result when nsplit == 1, else
// a partial (value, index) into the workspace at [o * nsplit + chunk]
template <int SR, typename T>
__global__ void __launch_bounds__(NT) k_reduce_block(const T* __restrict__ in, T* __restrict__ out,
                                                     int32_t* __restrict__ arg, T* __restrict__ part_v,
                                                     int64_t* __restrict__ part_i, RedParams p)
{
    pdl_wait();
    pdl_signal();
    using S = Semi<SR, T>;
    __shared__ T sv[NT];
    __shared__ int64_t si[NT];
    const int64_t work = p.n_out * p.nsplit;
    for (int64_t w = blockIdx.x; w < work; w += gridDim.x) {
        const int64_t o = w / p.nsplit, ch = w - o * p.nsplit;
        int64_t oi, oo, oa;
        out_offsets(p, o, oi, oo, oa);
        const int64_t r0 = ch * p.chunk;
        const int64_t r1 = r0 + p.chunk < p.R ? r0 + p.chunk : p.R;
        T best = S::zero();
        int64_t idx = NO_INDEX;
        for (int64_t r = r0 + threadIdx.x; r < r1; r += NT) {
            T v = red_load(in + oi + red_offset(p, r), p);
            if (S::better(v, best)) {
                best = v;
                idx = r;
            }
        }
        sv[threadIdx.x] = best;
        si[threadIdx.x] = idx;
        __syncthreads();
        for (int h = NT / 2; h > 0; h >>= 1) {
            if (threadIdx.x < h) {
                T bv = sv[threadIdx.x + h];
                int64_t bi = si[threadIdx.x + h];
                T av = sv[threadIdx.x];
                int64_t ai = si[threadIdx.x];
                if (S::better(bv, av) || (bv == av && bi < ai)) {
                    sv[threadIdx.x] = bv;
                    si[threadIdx.x] = bi;
                }
            }
            __syncthreads();
        }
        if (threadIdx.x == 0) {
            if (p.nsplit == 1) {
                red_store(out, oo, sv[0], arg, oa, final_index(si[0]), p);
            } else {
                if (TROP_IN(part_v + w, sizeof(T), p.sp[3])) part_v[w] = sv[0];
                if (TROP_IN(part_i + w, 8, p.sp[4])) part_i[w] = si[0];
            }
        }
        __syncthreads();
    }
}

// 32 consecutive outputs along the fastest output axis (unit stride in the input, so a slice's
// loads are coalesced) x RS slices of the reduced range per CTA: lane x of slice y takes
// r = y, y + RS, ...  The slices' partial (value, first index) pairs are merged in shared
// memory, pairwise in log2(RS) levels, a better value or an equal one with a smaller index
// winning: the strict left-to-right result.
template <int SR, typename T, int RS>
__global__ void __launch_bounds__(32 * RS) k_reduce_tile(const T* __restrict__ in, T* __restrict__ out,
                                                        int32_t* __restrict__ arg, RedParams p)
{
    pdl_wait();
    pdl_signal();
    using S = Semi<SR, T>;
    __shared__ T sv[RS][32];
    __shared__ int64_t si[RS][32];
    const int x = threadIdx.x & 31, y = threadIdx.x >> 5;
    const int64_t inner = p.out_size[p.out_rank - 1];
    const int64_t per_row = (inner + 31) / 32;
    const int64_t groups = p.n_out / inner * per_row;
    for (int64_t g = blockIdx.x; g < groups; g += gridDim.x) {
        const int64_t row = g / per_row, c = (g - row * per_row) * 32 + x;
        const bool valid = c < inner;
        int64_t oi = 0, oo = 0, oa = 0;
        if (valid) out_offsets(p, row * inner + c, oi, oo, oa);
        T best = S::zero();
        int64_t idx = NO_INDEX;
        if (valid) {
#pragma unroll 4
            for (int64_t r = y; r < p.R; r += RS) {
                const T v = red_load(in + oi + red_offset(p, r), p);
                if (S::better(v, best)) {
                    best = v;
                    idx = r;
                }
            }
        }
        sv[y][x] = best;
        si[y][x] = idx;
        __syncthreads();
        // pairwise, in log2(RS) levels: slice y takes slice y + h's pair (the merge is associative
        // and commutative: the better value, then the smaller index)
#pragma unroll
        for (int h = RS / 2; h > 0; h >>= 1) {
            if (y < h) {
                const T v = sv[y + h][x];
                const int64_t i = si[y + h][x];
                if (S::better(v, best) || (v == best && i < idx)) {
                    best = v;
                    idx = i;
                }
                sv[y][x] = best;
                si[y][x] = idx;
            }
            __syncthreads();
        }
        if (y == 0 && valid) red_store(out, oo, best, arg, oa, final_index(idx), p);
    }
}

// combine the chunks of each output in chunk order (strict: earliest wins)
template <int SR, typename T>
__global__ void k_reduce_combine(T* __restrict__ out, int32_t* __restrict__ arg, const T* __restrict__ part_v,
                                 const int64_t* __restrict__ part_i, RedParams p)
{
    pdl_wait();
    pdl_signal();
    using S = Semi<SR, T>;
    for (int64_t o = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; o < p.n_out;
         o += (int64_t)gridDim.x * blockDim.x) {
        int64_t oi, oo, oa;
        out_offsets(p, o, oi, oo, oa);
        T best = S::zero();
        int64_t idx = NO_INDEX;
        for (int64_t c = 0; c < p.nsplit; ++c) {
            const int64_t w = o * p.nsplit + c;
            T v = TROP_IN(part_v + w, sizeof(T), p.sp[3]) ? part_v[w] : S::zero();
            if (S::better(v, best)) {
                best = v;
                idx = TROP_IN(part_i + w, 8, p.sp[4]) ? part_i[w] : NO_INDEX;
            }
        }
        red_store(out, oo, best, arg, oa, final_index(idx), p);
    }
}

// ------------------------------------------------------------------ helpers
int grid_for(int64_t work, int per_block, int sm_count, int waves = 8)
{
    int64_t g = (work + per_block - 1) / per_block;
    int64_t cap = (int64_t)sm_count * waves;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (int)g;
}

int check_launch(const char* name)
{
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, name);
    count_launches(1);
    return TROP_OK;
}

template <typename T>
int launch_gather_typed(const void* in_, void* out_, const int32_t* in2, int32_t* out2, const GatherDesc& d0,
                        cudaStream_t s, const DeviceInfo* dev)
{
    const T* in = static_cast<const T*>(in_);
    T* out = static_cast<T*>(out_);
    const bool pair = in2 != nullptr;
    // drop unit axes, then merge axes that stay adjacent in both tensors
    GatherDesc d{};
    for (int i = 0; i < d0.rank; ++i) {
        if (d0.size[i] == 0) return TROP_OK;
        if (d0.size[i] == 1) continue;
        int r = d.rank;
        if (r > 0) {
            int q = r - 1;
            bool m = d.s_in[q] == d0.s_in[i] * d0.size[i] && d.s_out[q] == d0.s_out[i] * d0.size[i];
            if (pair) m = m && d.s_in2[q] == d0.s_in2[i] * d0.size[i] && d.s_out2[q] == d0.s_out2[i] * d0.size[i];
            if (m) {
                d.size[q] *= d0.size[i];
                d.s_in[q] = d0.s_in[i];
                d.s_out[q] = d0.s_out[i];
                d.s_in2[q] = d0.s_in2[i];
                d.s_out2[q] = d0.s_out2[i];
                continue;
            }
        }
        d.size[r] = d0.size[i];
        d.s_in[r] = d0.s_in[i];
        d.s_out[r] = d0.s_out[i];
        d.s_in2[r] = d0.s_in2[i];
        d.s_out2[r] = d0.s_out2[i];
        d.rank = r + 1;
    }
    int64_t total = 1;
    for (int i = 0; i < d.rank; ++i) total *= d.size[i];
    const bool same_map = !pair || [&] {
        for (int i = 0; i < d.rank; ++i)
            if (d.s_in2[i] != d.s_in[i] || d.s_out2[i] != d.s_out[i]) return false;
        return true;
    }();
    const bool small_idx = total < (int64_t(1) << 31);
    const int last = d.rank - 1;
    // the byte ranges the four views can address (bounds-checked build only)
    auto set_spans = [&](auto& p) {
#if TROP_DEBUG_BOUNDS
        p.sp[0] = span_of(in, sizeof(T), d.rank, d.size, d.s_in);
        p.sp[1] = span_of(out, sizeof(T), d.rank, d.size, d.s_out);
        p.sp[2] = span_of(in2, 4, d.rank, d.size, d.s_in2);
        p.sp[3] = span_of(out2, 4, d.rank, d.size, d.s_out2);
#else
        (void)p;
#endif
    };

    auto fill_rest = [&](auto& r, int skip_mask) {
        r.rank = 0;
        for (int i = 0; i < d.rank; ++i) {
            if (skip_mask & (1 << i)) continue;
            int k = r.rank++;
            r.div[k] = make_fastdiv((uint32_t)d.size[i]);
            r.s_in[k] = d.s_in[i];
            r.s_out[k] = d.s_out[i];
            r.s_in2[k] = d.s_in2[i];
            r.s_out2[k] = d.s_out2[i];
        }
    };

    if (d.rank >= 1 && small_idx && same_map && d.s_in[last] == 1 && d.s_out[last] == 1 && d.rank <= 31) {
        // ---- row copy
        auto launch_rows = [&](auto& p) {
            p.L = (uint32_t)d.size[last];
            constexpr int W = 16 / sizeof(T);
            bool vec = (p.L % W) == 0 && ((uintptr_t)in % 16) == 0 && ((uintptr_t)out % 16) == 0;
            for (int i = 0; i < last; ++i) vec = vec && (d.s_in[i] % W) == 0 && (d.s_out[i] % W) == 0;
            fill_rest(p.rest, 1 << last);
            set_spans(p);
            constexpr int R = sizeof(p.rest.div) / sizeof(p.rest.div[0]);
            const int64_t rows = total / p.L;
            if (vec) {
                p.Lv = p.L / W;
                p.total = (uint32_t)(rows * p.Lv);
                p.divLv = make_fastdiv(p.Lv);
                using V = typename std::conditional<sizeof(T) == 8, longlong2, int4>::type;
                int g = grid_for(p.total, NT, dev->sm_count);
                if (pair) (void)launch_pdl(k_copy_rows<T, V, true, R>, g, NT, 0, s, in, out, in2, out2, p);
                else (void)launch_pdl(k_copy_rows<T, V, false, R>, g, NT, 0, s, in, out, in2, out2, p);
            } else {
                p.Lv = p.L;
                p.total = (uint32_t)total;
                p.divLv = make_fastdiv(p.Lv);
                int g = grid_for(p.total, NT, dev->sm_count);
                if (pair) (void)launch_pdl(k_copy_rows<T, T, true, R>, g, NT, 0, s, in, out, in2, out2, p);
                else (void)launch_pdl(k_copy_rows<T, T, false, R>, g, NT, 0, s, in, out, in2, out2, p);
            }
            return check_launch("k_copy_rows");
        };
        if (d.rank - 1 <= REST_SMALL) {
            RowParams<REST_SMALL> p{};
            return launch_rows(p);
        }
        RowParams<MAXR> p{};
        return launch_rows(p);
    }

    int din = -1;
    for (int i = 0; i < d.rank; ++i)
        if (d.s_in[i] == 1) din = i;
    // ---- tiled transpose over two axis chains (the rest axes fit the small parameter block
    // whenever the whole layout has at most REST_SMALL axes); returns 1 when it does not apply
    auto try_transpose = [&](auto& p) -> int {
        constexpr int R = sizeof(p.rest.div) / sizeof(p.rest.div[0]);
        constexpr int CHAIN_I = TileCfg<sizeof(T)>::TIMAX, CHAIN_J = TileCfg<sizeof(T)>::TJMAX;
        int used = 0;
        // output-fastest chain
        int gj[4], ngj = 0;
        int64_t nJ = 1;
        {
            int cur = last;
            while (cur >= 0 && ngj < 4) {
                gj[ngj++] = cur;
                used |= 1 << cur;
                nJ *= d.size[cur];
                if (nJ >= CHAIN_J) break;
                int nxt = -1;
                for (int i = 0; i < d.rank; ++i)
                    if (!(used & (1 << i)) && i != din && d.s_out[i] == nJ) nxt = i;
                cur = nxt;
            }
        }
        // input-fastest chain
        int gi[4], ngi = 0;
        int64_t nI = 1;
        {
            int cur = din;
            while (cur >= 0 && ngi < 4) {
                gi[ngi++] = cur;
                used |= 1 << cur;
                nI *= d.size[cur];
                if (nI >= CHAIN_I) break;
                int nxt = -1;
                for (int i = 0; i < d.rank; ++i)
                    if (!(used & (1 << i)) && d.s_in[i] == nI) nxt = i;
                cur = nxt;
            }
        }
        // chain digits are stored slowest first (index 0 = slowest)
        p.gj_rank = ngj;
        for (int k = 0; k < ngj; ++k) {
            int ax = gj[ngj - 1 - k];
            p.gj_div[k] = make_fastdiv((uint32_t)d.size[ax]);
            p.gj_s_in[k] = d.s_in[ax];
            p.gj_s_in2[k] = d.s_in2[ax];
        }
        p.gi_rank = ngi;
        for (int k = 0; k < ngi; ++k) {
            int ax = gi[ngi - 1 - k];
            p.gi_div[k] = make_fastdiv((uint32_t)d.size[ax]);
            p.gi_s_out[k] = d.s_out[ax];
            p.gi_s_out2[k] = d.s_out2[ax];
        }
        fill_rest(p.rest, used);
        set_spans(p);
        int64_t nrest = 1;
        for (int i = 0; i < d.rank; ++i)
            if (!(used & (1 << i))) nrest *= d.size[i];
        using Cfg = TileCfg<sizeof(T)>;
        auto pow2ceil = [](int64_t v) {
            int64_t r = 1;
            while (r < v) r <<= 1;
            return r;
        };
        // tile: TI x TJ = TILE elements, fitted to short chains
        int64_t ti_ = std::min<int64_t>(Cfg::TIMAX, std::max<int64_t>(4, pow2ceil(nI)));
        int64_t tj_ = std::min<int64_t>(Cfg::TJMAX, Cfg::TILE / ti_);
        if (pow2ceil(nJ) < tj_) {
            tj_ = std::max<int64_t>(4, pow2ceil(nJ));
            ti_ = std::min<int64_t>(Cfg::TIMAX, std::max<int64_t>(4, std::min<int64_t>(pow2ceil(nI), Cfg::TILE / tj_)));
        }
        // stack outer slices when both chains are short
        int64_t tb_ = 1;
        while (tb_ * 2 * ti_ * tj_ <= Cfg::TILE && tb_ * 2 <= Cfg::TBMAX && tb_ < nrest) tb_ *= 2;
        p.TI = (uint32_t)ti_;
        p.TJ = (uint32_t)tj_;
        p.TB = (uint32_t)tb_;
        p.lTI = 0;
        while ((1u << p.lTI) < p.TI) ++p.lTI;
        p.lTJ = 0;
        while ((1u << p.lTJ) < p.TJ) ++p.lTJ;
        p.lTB = 0;
        while ((1u << p.lTB) < p.TB) ++p.lTB;
        p.nI = (uint32_t)nI;
        p.nJ = (uint32_t)nJ;
        p.nR = (uint32_t)nrest;
        p.tilesI = (uint32_t)((nI + ti_ - 1) / ti_);
        p.tilesJ = (uint32_t)((nJ + tj_ - 1) / tj_);
        p.tilesR = (uint32_t)((nrest + tb_ - 1) / tb_);
        int64_t tiles = (int64_t)p.tilesI * p.tilesJ * p.tilesR;
        if (tiles < (int64_t(1) << 31)) {
            p.tiles = (uint32_t)tiles;
            p.div_tilesI = make_fastdiv(p.tilesI);
            p.div_tilesJ = make_fastdiv(p.tilesJ);
            constexpr int W = 16 / sizeof(T);
            bool vec = ((uintptr_t)in % 16) == 0 && (nI % W) == 0 && (p.TI % W) == 0 &&
                       (!pair || ((uintptr_t)in2 % 16) == 0);
            for (int i = 0; i < d.rank; ++i)
                if (i != din) vec = vec && (d.s_in[i] % W) == 0;
            p.vec_in = vec ? 1 : 0;
            // vector stores: output rows start 16-byte aligned (every stride but the GJ chain's unit one)
            bool vo = ((uintptr_t)out % 16) == 0 && (nJ % W) == 0 && (!pair || ((uintptr_t)out2 % 16) == 0);
            for (int i = 0; i < d.rank; ++i)
                if (i != last) vo = vo && (d.s_out[i] % W) == 0;
            p.vec_out = vo ? 1 : 0;
            // swizzle step: the x values one warp's loads cover (32 lanes over TI / W vectors per row),
            // at least W so the storer's W-wide runs stay whole
            p.sw = (int)std::max<int64_t>(W, (int64_t)32 * W / ti_);
            const int g = (int)std::min<int64_t>(tiles, (int64_t)dev->sm_count * 64);
            if (pair) (void)launch_pdl(k_transpose<T, true, R>, g, NT, 0, s, in, out, in2, out2, p);
            else (void)launch_pdl(k_transpose<T, false, R>, g, NT, 0, s, in, out, in2, out2, p);
            return check_launch("k_transpose");
        }
        return 1;
    };
    if (d.rank >= 2 && small_idx && same_map && d.s_out[last] == 1 && din >= 0 && din != last) {
        int rc;
        if (d.rank <= REST_SMALL) {
            TransParams<REST_SMALL> p{};
            rc = try_transpose(p);
        } else {
            TransParams<MAXR> p{};
            rc = try_transpose(p);
        }
        if (rc != 1) return rc;
    }

    // ---- generic gather
    GatherParams p{};
    p.rank = d.rank;
    p.total = total;
    for (int i = 0; i < d.rank; ++i) {
        p.size[i] = d.size[i];
        p.s_in[i] = d.s_in[i];
        p.s_out[i] = d.s_out[i];
        p.s_in2[i] = d.s_in2[i];
        p.s_out2[i] = d.s_out2[i];
    }
    set_spans(p);
    int g = grid_for(total, NT, dev->sm_count);
    if (pair) (void)launch_pdl(k_gather<T, true>, g, NT, 0, s, in, out, in2, out2, p);
    else (void)launch_pdl(k_gather<T, false>, g, NT, 0, s, in, out, in2, out2, p);
    return check_launch("k_gather");
}

template <int SR, typename T>
int launch_reduce_typed(const void* in_, void* out_, int32_t* arg, const ReduceDesc& d, const ReduceScratch* fixed,
                        cudaStream_t s, const DeviceInfo* dev)
{
    const T* in = static_cast<const T*>(in_);
    T* out = static_cast<T*>(out_);
    RedParams p{};
    p.n_out = 1;
    p.out_rank = 0;
    for (int i = 0; i < d.out_rank; ++i) {
        if (d.out_size[i] == 0) return TROP_OK;
        if (d.out_size[i] == 1) continue;
        int k = p.out_rank++;
        p.out_size[k] = d.out_size[i];
        p.out_s_in[k] = d.out_s_in[i];
        p.out_s_out[k] = d.out_s_out[i];
        p.out_s_arg[k] = d.out_s_arg[i];
        p.n_out *= d.out_size[i];
    }
    // merge reduced axes that stay adjacent (keeps the row-major index)
    p.R = 1;
    p.red_rank = 0;
    for (int i = 0; i < d.red_rank; ++i) {
        p.R *= d.red_size[i];
        if (d.red_size[i] == 1) continue;
        int q = p.red_rank - 1;
        if (q >= 0 && p.red_s_in[q] == d.red_s_in[i] * d.red_size[i]) {
            p.red_size[q] *= d.red_size[i];
            p.red_s_in[q] = d.red_s_in[i];
            continue;
        }
        p.red_size[p.red_rank] = d.red_size[i];
        p.red_s_in[p.red_rank] = d.red_s_in[i];
        ++p.red_rank;
    }
    if (p.red_rank == 0) {
        p.red_rank = 1;
        p.red_size[0] = 1;
        p.red_s_in[0] = 0;
    }
#if TROP_DEBUG_BOUNDS
    {
        int64_t sz[2 * MAXR], st[2 * MAXR];
        for (int i = 0; i < p.out_rank; ++i) sz[i] = p.out_size[i], st[i] = p.out_s_in[i];
        for (int i = 0; i < p.red_rank; ++i) sz[p.out_rank + i] = p.red_size[i], st[p.out_rank + i] = p.red_s_in[i];
        p.sp[0] = span_of(in, sizeof(T), p.out_rank + p.red_rank, sz, st);
        p.sp[1] = span_of(out, sizeof(T), p.out_rank, p.out_size, p.out_s_out);
        p.sp[2] = span_of(arg, 4, p.out_rank, p.out_size, p.out_s_arg);
    }
#endif
    const int64_t threads_wanted = (int64_t)dev->sm_count * 1024;
    if (p.R <= 64 || p.n_out >= threads_wanted) {
        int g = grid_for(p.n_out, NT, dev->sm_count);
        (void)launch_pdl(k_reduce_thread<SR, T>, g, NT, 0, s, in, out, arg, p);
        return check_launch("k_reduce_thread");
    }
    if (p.out_rank >= 1 && p.out_s_in[p.out_rank - 1] == 1 && p.R <= (int64_t(1) << 24)) {
        // outputs contiguous in the input: coalesced slices, no workspace
        const int64_t inner = p.out_size[p.out_rank - 1];
        const int64_t groups = p.n_out / inner * ((inner + 31) / 32);
        const int g = (int)std::min<int64_t>(std::max<int64_t>(groups, 1), (int64_t)dev->sm_count * 16);
        if (p.R >= 64) (void)launch_pdl(k_reduce_tile<SR, T, 32>, g, 32 * 32, 0, s, in, out, arg, p);
        else (void)launch_pdl(k_reduce_tile<SR, T, 8>, g, 32 * 8, 0, s, in, out, arg, p);
        return check_launch("k_reduce_tile");
    }
    // split each output's reduced range so that enough blocks exist
    const int64_t blocks_wanted = (int64_t)dev->sm_count * 8;
    int64_t nsplit = (blocks_wanted + p.n_out - 1) / p.n_out;
    int64_t max_split = (p.R + 2047) / 2048;
    if (nsplit > max_split) nsplit = max_split;
    if (nsplit < 1) nsplit = 1;
    p.nsplit = nsplit;
    p.chunk = (p.R + nsplit - 1) / nsplit;
    T* part_v = nullptr;
    int64_t* part_i = nullptr;
    void* ws = nullptr;
    if (nsplit > 1) {
        // the partial results: pool workspace, or the caller's fixed block (never allocated)
        const size_t nb = (size_t)(p.n_out * nsplit);
        const size_t need = nb * (sizeof(T) + sizeof(int64_t));
        if (fixed) {
            if (!fixed->ptr || need > fixed->bytes)
                return set_error(TROP_ERR_UNSUPPORTED,
                                 "reduction needs %zu bytes of scratch for %lld partial results; the fixed scratch "
                                 "holds %zu bytes",
                                 need, (long long)nb, fixed->bytes);
            part_i = static_cast<int64_t*>(fixed->ptr);
        } else {
            TROP_TRY(pool_alloc(need, s, &ws));
            part_i = static_cast<int64_t*>(ws);
        }
        part_v = reinterpret_cast<T*>(part_i + nb);
#if TROP_DEBUG_BOUNDS
        p.sp[3] = span_bytes(part_v, nb * sizeof(T));
        p.sp[4] = span_bytes(part_i, nb * sizeof(int64_t));
#endif
    }
    int g = grid_for(p.n_out * nsplit, 1, dev->sm_count, 16);
    (void)launch_pdl(k_reduce_block<SR, T>, g, NT, 0, s, in, out, arg, part_v, part_i, p);
    int rc = check_launch("k_reduce_block");
    if (rc == TROP_OK && nsplit > 1) {
        int g2 = grid_for(p.n_out, NT, dev->sm_count);
        (void)launch_pdl(k_reduce_combine<SR, T>, g2, NT, 0, s, out, arg, part_v, part_i, p);
        rc = check_launch("k_reduce_combine");
    }
    if (ws) pool_retire(ws, s);
    return rc;
}

}  // namespace

int launch_gather(const void* in, void* out, int elem_bytes, const int32_t* in2, int32_t* out2,
                  const GatherDesc& d, cudaStream_t s)
{
    const DeviceInfo* dev = nullptr;
    TROP_TRY(ensure_device(&dev));
    if (elem_bytes == 4) return launch_gather_typed<int32_t>(in, out, in2, out2, d, s, dev);
    if (elem_bytes == 8) return launch_gather_typed<int64_t>(in, out, in2, out2, d, s, dev);
    return set_error(TROP_ERR_DTYPE, "gather: unsupported element size %d", elem_bytes);
}

int launch_reduce(int semiring, int dtype, const void* in, void* out, int32_t* argmax, const ReduceDesc& d,
                  const ReduceScratch* fixed, cudaStream_t s)
{
    const DeviceInfo* dev = nullptr;
    TROP_TRY(ensure_device(&dev));
#define TROP_RED(SR)                                                                                 \
    case SR:                                                                                         \
        if (dtype == TROP_F32) return launch_reduce_typed<SR, float>(in, out, argmax, d, fixed, s, dev);   \
        if (dtype == TROP_I32) return launch_reduce_typed<SR, int32_t>(in, out, argmax, d, fixed, s, dev); \
        if (dtype == TROP_I64) return launch_reduce_typed<SR, int64_t>(in, out, argmax, d, fixed, s, dev); \
        if (dtype == TROP_F64) return launch_reduce_typed<SR, double>(in, out, argmax, d, fixed, s, dev);  \
        break;
    switch (semiring) {
        TROP_RED(TROP_MAXPLUS)
        TROP_RED(TROP_MINPLUS)
        TROP_RED(TROP_MAXTIMES)
    default: break;
    }
#undef TROP_RED
    return set_error(TROP_ERR_DTYPE, "reduce: unsupported semiring %d / dtype %d", semiring, dtype);
}

// kernels touched once per device at set-up so that module loading happens
// there and not inside a measured call
int register_unary_kernels()
{
    cudaFuncAttributes a;
    const void* ks[] = {
        (const void*)k_gather<int32_t, false>, (const void*)k_gather<int64_t, false>,
        (const void*)k_gather<int32_t, true>, (const void*)k_gather<int64_t, true>,
        (const void*)k_copy_rows<int32_t, int4, false, REST_SMALL>, (const void*)k_copy_rows<int64_t, longlong2, false, REST_SMALL>,
        (const void*)k_copy_rows<int32_t, int4, true, REST_SMALL>, (const void*)k_copy_rows<int32_t, int32_t, false, REST_SMALL>,
        (const void*)k_transpose<int32_t, false, REST_SMALL>, (const void*)k_transpose<int64_t, false, REST_SMALL>,
        (const void*)k_transpose<int32_t, true, REST_SMALL>, (const void*)k_transpose<int64_t, true, REST_SMALL>,
        (const void*)k_reduce_thread<TROP_MAXPLUS, float>, (const void*)k_reduce_block<TROP_MAXPLUS, float>,
        (const void*)k_reduce_tile<TROP_MAXPLUS, float, 8>, (const void*)k_reduce_tile<TROP_MAXPLUS, float, 32>,
        (const void*)k_reduce_combine<TROP_MAXPLUS, float>,
    };
    for (const void* k : ks) {
        cudaError_t e = cudaFuncGetAttributes(&a, k);
        if (e != cudaSuccess) return cuda_error(e, "cudaFuncGetAttributes (unary kernels)");
    }
    // shared-memory carveout of the transpose (see TROP_TRANSPOSE_CARVEOUT)
    const void* kt[] = {(const void*)k_transpose<int32_t, false, REST_SMALL>, (const void*)k_transpose<int64_t, false, REST_SMALL>,
                        (const void*)k_transpose<int32_t, true, REST_SMALL>, (const void*)k_transpose<int64_t, true, REST_SMALL>,
                        (const void*)k_transpose<int32_t, false, MAXR>, (const void*)k_transpose<int64_t, false, MAXR>,
                        (const void*)k_transpose<int32_t, true, MAXR>, (const void*)k_transpose<int64_t, true, MAXR>};
    for (const void* k : kt) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, TROP_TRANSPOSE_CARVEOUT);
        if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute (transpose carveout)");
    }
    return TROP_OK;
}

}  // namespace trop
