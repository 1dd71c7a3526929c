// gemm.cu -- strided-batched tropical GEMM with argmax on CUDA cores.
//
// C[b,m,n] = (+)_k A[b,m,k] (x) B[b,k,n] over max-plus, min-plus and
// max-times, plus argmax[b,m,n] = the smallest k reaching C (tropical-gemm
// PR #35 "batched GPU ops with DLPack zero-copy output", Summary: the
// tropical_{maxplus,minplus,maxmul}_f32_nn_batched_with_argmax kernels).
// A max-plus product is not a multiply-accumulate, so tensor cores do not
// apply; the work runs on the FP32 pipes:
//   * (x) two outputs at a time with the packed add.rn.f32x2 / mul.rn.f32x2
//     (one rounding per product, as the scalar op);
//   * (+) folds two new products into the running result with one
//     three-input max.f32 / min.f32.
// Both are exact per element, so the result does not depend on the order in
// which k is visited.
//
// Argmax without a compare per term: k is walked in chunks of CH = 8.  At the
// end of a chunk each output compares its running result with the value it
// had at the chunk's start; a strict improvement records the chunk number.
// Because the running result only grows (shrinks for min-plus), the last
// improving chunk holds the first k that reaches the final value, and a
// second pass (k_argmax_resolve) recomputes just that chunk's CH products to
// find it.  If nothing beat the semiring zero the argmax is 0, which is what
// a strict left-to-right scan gives.
//
// Kernels:
//   k_gemm_tma       the argmax GEMM for one batch axis, K a multiple of 16 and
//                    16-byte rows: 64x64 tile per 128-thread CTA, 8x4 outputs
//                    per thread, A and B boxes by TMA into a 3-stage mbarrier
//                    ring, 4 CTAs per SM; a programmatic dependent of the
//                    kernel before it.
//   k_gemm_tiled     other layouts: 64x64 output tile, 8x8 per thread (8x4
//                    with argmax), A staged transposed through registers and
//                    B by cp.async; needs sAk == 1 and sBn == 1 (the planner
//                    permutes other layouts).  A thin last wave is cut along k
//                    (stream-K, see the schedule below).
//   k_gemm_tma_fused the TMA-fed tiles and their short-K resolve (K <= 256) in
//                    one launch: CTAs take GEMM tiles, then resolve items, from
//                    a counter; a resolve item waits for its batch's tiles, so
//                    the resolve starts in the GEMM's last, part-filled wave.
//   k_argmax_resolve_rows  chunk -> exact index for K <= 256: a warp reads a
//                    row of A once, one chunk per lane, and outputs take their
//                    chunk's values by shuffles.
//   k_argmax_resolve chunk -> exact index for longer contractions or other
//                    layouts, B staged per column panel.  Both resolve passes
//                    split the rows of all column panels evenly over resident
//                    CTAs and are programmatic dependents of the GEMM.
//   k_gemm_stream    few rows (M <= 8) and a short contraction (K <= 64):
//                    one thread per (batch, column vector), memory bound.
//   k_gemm_generic   anything else: one thread per output, sequential k.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstdio>

#define TROP_TU 2  // this file's id in a bounds-violation record
#include "internal.h"

namespace trop {

namespace {

// ------------------------------------------------------------------ semiring ops
template <int SR>
struct Ops {
    __device__ __forceinline__ static float zero()
    {
        return SR == TROP_MAXPLUS ? -INFINITY : SR == TROP_MINPLUS ? INFINITY : 0.0f;
    }
    // value used to pad the K tail of B (A's tail is the zero): zero (x) pad == zero
    __device__ __forceinline__ static float bpad() { return 0.0f; }
    __device__ __forceinline__ static float mul(float a, float b)
    {
        return SR == TROP_MAXTIMES ? __fmul_rn(a, b) : __fadd_rn(a, b);
    }
    __device__ __forceinline__ static float2 mul2(float2 a, float2 b)
    {
        return SR == TROP_MAXTIMES ? __fmul2_rn(a, b) : __fadd2_rn(a, b);
    }
    __device__ __forceinline__ static bool better(float a, float b) { return SR == TROP_MINPLUS ? a < b : a > b; }
    __device__ __forceinline__ static float fold3(float acc, float x, float y)
    {
        float r;
        if (SR == TROP_MINPLUS) asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(acc), "f"(x), "f"(y));
        else asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(acc), "f"(x), "f"(y));
        return r;
    }
};

struct Batch {
    int nb;
    FastDiv div[MAXB];
    int64_t sA[MAXB], sB[MAXB], sC[MAXB], sI[MAXB];
};

__device__ __forceinline__ void batch_offsets(const Batch& bt, uint32_t b, int64_t& oa, int64_t& ob, int64_t& oc,
                                              int64_t& oi)
{
    oa = ob = oc = oi = 0;
    for (int d = bt.nb - 1; d >= 0; --d) {
        uint32_t q = fdiv(b, bt.div[d]);
        uint32_t c = b - q * bt.div[d].d;
        b = q;
        oa += (int64_t)c * bt.sA[d];
        ob += (int64_t)c * bt.sB[d];
        oc += (int64_t)c * bt.sC[d];
        oi += (int64_t)c * bt.sI[d];
    }
}

// ------------------------------------------------------------------ tiled kernel
constexpr int BM = 64, BN = 64, BK = 16, TM = 8;
// Outputs per thread: TM rows x TN columns.  Without argmax TN = 8 (64 threads per tile);
// with argmax the two accumulator sets double the registers, so TN = 4 (128 threads per tile)
// keeps a thread near 128 registers and gives each SM twice the warps to hide latency with.
#ifndef TROP_ARG_TN
#define TROP_ARG_TN 4
#endif
template <bool ARG> __host__ __device__ constexpr int tile_tn() { return ARG ? TROP_ARG_TN : 8; }
template <int TN> __host__ __device__ constexpr int tile_threads() { return (BM / TM) * (BN / TN); }
constexpr int TILE_ELEMS = BM * BN;
constexpr int APAD = 4;                          // float pad per transposed A row (keeps 16-byte rows)
#ifndef TROP_ARG_CHUNK
#define TROP_ARG_CHUNK 8
#endif
constexpr int CH = TROP_ARG_CHUNK;               // k per argmax chunk (divides BK)
static_assert(BK % CH == 0 && CH % 2 == 0, "chunk must divide the k-tile and hold whole k pairs");

// Tile schedule.  Tiles are numbered t = (b * tiles_m + mt) * tiles_n + nt.  CTA t < T_dp
// computes tile t over the whole contraction.  When the last tiles would only part-fill a
// wave of resident CTAs, those R tiles are cut along k instead: their U = R * nkt k-tiles
// ("units", tile-major) are dealt out L at a time to the CTAs after the data-parallel ones,
// so the tail keeps every SM busy (the stream-K decomposition of Osama et al., "Stream-K:
// Work-centric Parallel Decomposition for Dense Matrix-Matrix Multiplication on the GPU",
// PPoPP 2023).  With L <= nkt the units of one CTA touch at most two tiles; the piece of a
// tile it computes (a "segment") goes to workspace slot [j][0] for the tile its range starts
// in and [j][1] for the next.  A tile's segments come from CTAs ua / L .. (ua + nkt - 1) / L,
// ua being its first unit; the first of them used slot 1 if its range began in the tile
// before.  Merging segments in k order, a later one winning only when strictly better,
// reproduces the single pass exactly: (+) is exact, and the strict compare keeps the
// first k that reaches the result.
struct TiledParams {
    int M, N, K;
    const float* A;
    const float* B;
    float* C;
    int32_t* I;
    int64_t sAm, sBk, sCm, sCn, sIm, sIn;
    uint32_t nbatch;
    Batch bt;
    int vecA, vecB;  // 16-byte loads allowed (alignment of every row start)
    int vecC, vecI;  // 16-byte stores allowed (unit column stride, aligned rows)
    uint32_t tiles_m, tiles_n, nkt;
    FastDiv div_tm, div_tn, div_nkt, div_L;
    uint32_t T_dp;     // data-parallel tiles: 0 .. T_dp-1
    uint32_t L, U;     // stream-K: k-tiles per CTA, k-tiles in all (0: no stream-K tiles)
    float* seg_v;      // [G_sk][2][BM*BN] segment values
    uint16_t* seg_c;   // [G_sk][2][BM*BN] chunk + 1 of each segment's first maximum, 0 if none (ARG)
    uint32_t* sk_cnt;  // [R] arrival tickets of the stream-K tiles (zero before and after a launch)
    uint64_t r_units;  // rows walked by the resolve pass: nbatch * tiles_n * M
    int sAm32, sCm32, sIm32;  // the row strides as 32-bit values (short-K resolve only)
    // resolve work split: CTA j walks rows [j * r_per + min(j, r_rem), + r_per + (j < r_rem));
    // with r32 (r_units < 2^31) a row unit splits into (panel, row) and a panel into (batch,
    // column panel) by the fast 32-bit divisions
    uint64_t r_per;
    uint32_t r_rem;
    int r32;
    FastDiv div_M, div_npan;
    // TMA-fed kernel only: where a wait that could not be completed is reported (a word in
    // host-mapped memory, read by the library's next call) and the test mode of its waits
    uint32_t* err;
    int wait_mode;
    // fused kernel only (k_gemm_tma_fused): its work items are the n_tiles GEMM tiles followed
    // by the resolve items, items_per_batch per batch (rblocks row blocks of each column panel).
    // sched[0] hands out items in order; sched[1 + b] counts the stored tiles of batch b and
    // sched[1 + nbatch + b] its finished resolve items (all zero between launches).
    uint32_t* sched;
    uint32_t n_tiles, n_items, tiles_per_batch, items_per_batch, rblocks;
    FastDiv div_ipb, div_rblocks;
    // 1: the grid before on the stream is a fused GEMM whose outputs this launch does not read,
    // so the wait for it comes only ahead of this launch's first global store; 0: at the start
    int late;
#if TROP_DEBUG_BOUNDS
    Span sp[8];  // A, B, C, I, seg_v, seg_c, sk_cnt, sched
#endif
};

// checked global accesses of the tiled kernels (plain accesses in the normal build): operand k
// of TiledParams::sp must hold `bytes` at ptr
#define T_IN(ptr, bytes, k) TROP_IN(ptr, bytes, p.sp[k])

__device__ __forceinline__ void tile_coord(const TiledParams& p, uint32_t t, uint32_t& b, int& m0, int& n0)
{
    const uint32_t q = fdiv(t, p.div_tn);
    b = fdiv(q, p.div_tm);
    m0 = (int)(q - b * p.tiles_m) * BM;
    n0 = (int)(t - q * p.tiles_n) * BN;
}

// the CTAs holding the segments of stream-K tile tl, and the slot the first one used
__device__ __forceinline__ void sk_segments(const TiledParams& p, uint32_t tl, uint32_t& j0, uint32_t& j1, int& slot0)
{
    const uint32_t ua = tl * p.nkt;
    j0 = fdiv(ua, p.div_L);
    j1 = fdiv(ua + p.nkt - 1, p.div_L);
    slot0 = j0 * p.L < ua ? 1 : 0;
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes)
{
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(sa), "l"(gmem), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::); }

// rows / columns of the 8x8 outputs a thread owns: two groups of 4, half a tile apart
__device__ __forceinline__ int row_of(int tm, int i) { return i < 4 ? tm * 4 + i : BM / 2 + tm * 4 + (i - 4); }

// Programmatic dependent launch: a kernel launched with programmatic stream serialisation
// may start once every CTA of the kernel before it has signalled (or exited); it must
// wait before touching that kernel's results.  Without the launch attribute both are no-ops.

// Rows of the resolve pass that this CTA walks, and the (batch, first column, row) of row
// unit u (units run over the rows of every column panel of every batch).
__device__ __forceinline__ void resolve_range(const TiledParams& p, uint64_t& ubeg, uint64_t& uend)
{
    const uint64_t j = blockIdx.x;
    ubeg = j * p.r_per + min(j, (uint64_t)p.r_rem);
    uend = ubeg + p.r_per + (j < p.r_rem ? 1 : 0);
}
__device__ __forceinline__ void resolve_unit(const TiledParams& p, uint64_t u, uint32_t npan, int pw, uint32_t& b,
                                             int& n0, int& mb)
{
    if (p.r32) {
        const uint32_t pn = fdiv((uint32_t)u, p.div_M);
        mb = (int)((uint32_t)u - pn * (uint32_t)p.M);
        b = fdiv(pn, p.div_npan);
        n0 = (int)(pn - b * npan) * pw;
    } else {
        const uint64_t pn = u / (uint64_t)p.M;
        mb = (int)(u - pn * (uint64_t)p.M);
        b = (uint32_t)(pn / npan);
        n0 = (int)(pn - (uint64_t)b * npan) * pw;
    }
}

// Merge the segments of stream-K tile tl in k order (a later one wins only when strictly
// better) and store the tile through C's strides; with ARG also -(chunk + 1), or 0, into I.
// The segments of other CTAs are read through L2 (ld.global.cg): they were written by
// other SMs during this launch.
constexpr int MERGE_BATCH = 8;  // runs of 4 columns whose loads are in flight together

template <int SR, bool ARG, int THREADS>
__device__ __forceinline__ void sk_merge(const TiledParams& p, uint32_t tl, int m0, int n0, int64_t oc,
                                         int64_t oi, int tid)
{
    using O = Ops<SR>;
    constexpr int MERGE_RUNS = TILE_ELEMS / 4 / THREADS;  // runs of 4 columns per thread
    static_assert(MERGE_RUNS % MERGE_BATCH == 0, "whole batches of runs");
    uint32_t j0, j1;
    int slot0;
    sk_segments(p, tl, j0, j1, slot0);
#pragma unroll 1
    for (int q0 = 0; q0 < MERGE_RUNS; q0 += MERGE_BATCH) {
        float v[MERGE_BATCH][4];
        int cd[MERGE_BATCH][4];
#pragma unroll
        for (int q = 0; q < MERGE_BATCH; ++q)
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                v[q][x] = O::zero();
                cd[q][x] = 0;
            }
        for (uint32_t jj = j0; jj <= j1; ++jj) {
            const size_t base = ((size_t)jj * 2 + (jj == j0 ? slot0 : 0)) * TILE_ELEMS;
            float4 sv[MERGE_BATCH];
            uint2 sc[MERGE_BATCH];
#pragma unroll
            for (int q = 0; q < MERGE_BATCH; ++q) {
                const int e = ((q0 + q) * THREADS + tid) * 4;
                sv[q] = T_IN(p.seg_v + base + e, 16, 4) ? __ldcg(reinterpret_cast<const float4*>(p.seg_v + base + e))
                                                        : make_float4(O::zero(), O::zero(), O::zero(), O::zero());
                if (ARG) sc[q] = T_IN(p.seg_c + base + e, 8, 5) ? __ldcg(reinterpret_cast<const uint2*>(p.seg_c + base + e))
                                                                : make_uint2(0u, 0u);
            }
#pragma unroll
            for (int q = 0; q < MERGE_BATCH; ++q) {
                const float s4[4] = {sv[q].x, sv[q].y, sv[q].z, sv[q].w};
                const int c4[4] = {ARG ? (int)(sc[q].x & 0xffffu) : 0, ARG ? (int)(sc[q].x >> 16) : 0,
                                   ARG ? (int)(sc[q].y & 0xffffu) : 0, ARG ? (int)(sc[q].y >> 16) : 0};
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    if (O::better(s4[x], v[q][x])) {
                        v[q][x] = s4[x];
                        cd[q][x] = c4[x];
                    }
            }
        }
#pragma unroll
        for (int q = 0; q < MERGE_BATCH; ++q) {
            const int e = ((q0 + q) * THREADS + tid) * 4;
            const int m = m0 + e / BN, n = n0 + e % BN;
            if (m >= p.M) continue;
            float* crow = p.C + oc + (int64_t)m * p.sCm;
            if (p.vecC && n + 3 < p.N) {
                if (T_IN(crow + n, 16, 2))
                    *reinterpret_cast<float4*>(crow + n) = make_float4(v[q][0], v[q][1], v[q][2], v[q][3]);
            } else {
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    if (n + x < p.N && T_IN(crow + (int64_t)(n + x) * p.sCn, 4, 2))
                        crow[(int64_t)(n + x) * p.sCn] = v[q][x];
            }
            if (ARG) {
                int32_t* irow = p.I + oi + (int64_t)m * p.sIm;
                if (p.vecI && n + 3 < p.N) {
                    if (T_IN(irow + n, 16, 3))
                        *reinterpret_cast<int4*>(irow + n) = make_int4(-cd[q][0], -cd[q][1], -cd[q][2], -cd[q][3]);
                } else {
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        if (n + x < p.N && T_IN(irow + (int64_t)(n + x) * p.sIn, 4, 3))
                            irow[(int64_t)(n + x) * p.sIn] = -cd[q][x];
                }
            }
        }
    }
}

// ARG: besides C, writes into I the chunk that holds each output's first maximum as
// -(chunk + 1), or 0 when no product beat the semiring zero; k_argmax_resolve then
// replaces the chunk by the exact index.  Stream-K segments go to the workspace instead.
// resident CTAs per SM the register allocation must allow (measured best on GB300)
#ifndef TROP_ARG_MINB
#define TROP_ARG_MINB 3
#endif
#ifndef TROP_PLAIN_MINB
#define TROP_PLAIN_MINB 1
#endif
template <int SR, bool ARG, int TN>
__global__ void __launch_bounds__(tile_threads<TN>(), ARG ? TROP_ARG_MINB : TROP_PLAIN_MINB) k_gemm_tiled(TiledParams p)
{
    using O = Ops<SR>;
    constexpr int THREADS = tile_threads<TN>();
    constexpr int NG = TN / 4;             // groups of 4 columns per thread, half a tile apart
    constexpr int NLA = BM * BK / 4 / THREADS, NLB = BK * BN / 4 / THREADS;  // float4 loads per k-tile
    static_assert(TN == 4 || TN == 8, "4 or 8 columns per thread");
    __shared__ __align__(16) float As[2][BK][BM + APAD];  // A transposed: As[k][m]
    __shared__ __align__(16) float Bs[2][BK][BN];
    __shared__ uint16_t sid[ARG ? TM * TN : 1][ARG ? THREADS : 1];

    __shared__ int s_last;

    pdl_wait();    // launched as a programmatic dependent: the grid before it has completed
    pdl_signal();  // the resolve pass may start filling SMs as this grid drains
    const int tid = threadIdx.x;
    const int tm = tid / (BN / TN), tn = tid % (BN / TN);
    const float zero = O::zero();
    const bool sk = blockIdx.x >= p.T_dp;
    const uint32_t j = sk ? blockIdx.x - p.T_dp : 0;
    uint32_t u = sk ? j * p.L : 0;
    const uint32_t ue = sk ? min(p.U, u + p.L) : 0;

    for (int pass = 0; pass < 2; ++pass) {
        uint32_t t;
        int kt0, kt1;
        if (!sk) {
            if (pass) break;
            t = blockIdx.x;
            kt0 = 0;
            kt1 = (int)p.nkt;
        } else {
            if (u >= ue) break;
            const uint32_t tl = fdiv(u, p.div_nkt);
            kt0 = (int)(u - tl * p.nkt);
            kt1 = (int)min(p.nkt, (uint32_t)kt0 + (ue - u));
            u += (uint32_t)(kt1 - kt0);
            t = p.T_dp + tl;
        }
        uint32_t b;
        int m0, n0;
        tile_coord(p, t, b, m0, n0);
        int64_t oa, ob, oc, oi;
        batch_offsets(p.bt, b, oa, ob, oc, oi);
        const float* __restrict__ A = p.A + oa;
        const float* __restrict__ B = p.B + ob;

        // loader roles: A: rows tid/4 + (THREADS/4)*r, k quad (tid%4)*4;
        //               B: rows tid/16 + (THREADS/16)*r, n quad (tid%16)*4
        const int la_m = tid / 4, la_k = (tid % 4) * 4;
        const int lb_k = tid / 16, lb_n = (tid % 16) * 4;

        float4 ra[NLA];
        auto load_a = [&](int kt) {
            const int k0 = kt * BK;
#pragma unroll
            for (int r = 0; r < NLA; ++r) {
                const int m = m0 + la_m + (THREADS / 4) * r, k = k0 + la_k;
                const float* src = A + (int64_t)m * p.sAm + k;
                if (m < p.M && k + 3 < p.K && p.vecA) {
                    ra[r] = T_IN(src, 16, 0) ? __ldg(reinterpret_cast<const float4*>(src)) : make_float4(zero, zero, zero, zero);
                } else {
                    float v[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        v[q] = (m < p.M && k + q < p.K && T_IN(src + q, 4, 0)) ? __ldg(src + q) : zero;
                    ra[r] = make_float4(v[0], v[1], v[2], v[3]);
                }
            }
        };
        auto store_a = [&](int buf) {
#pragma unroll
            for (int r = 0; r < NLA; ++r) {
                const int m = la_m + (THREADS / 4) * r;
                As[buf][la_k + 0][m] = ra[r].x;
                As[buf][la_k + 1][m] = ra[r].y;
                As[buf][la_k + 2][m] = ra[r].z;
                As[buf][la_k + 3][m] = ra[r].w;
            }
        };
        // B rows of a k-tile: cp.async with zero fill outside [0,K) x [0,N) (the K-tail pad of B is 0,
        // and zero (x) 0 is the semiring zero, so padded products never win)
        auto issue_b = [&](int kt, int buf) {
            const int k0 = kt * BK;
#pragma unroll
            for (int r = 0; r < NLB; ++r) {
                const int kk = lb_k + (THREADS / 16) * r, k = k0 + kk, n = n0 + lb_n;
                float* dst = &Bs[buf][kk][lb_n];
                if (p.vecB) {
                    int valid = (k < p.K) ? max(0, min(4, p.N - n)) : 0;
                    if (valid && !T_IN(B + (int64_t)k * p.sBk + n, valid * 4, 1)) valid = 0;
                    const float* src = valid ? B + (int64_t)k * p.sBk + n : B;
                    cp_async16(dst, src, valid * 4);
                } else {
                    const float* src = B + (int64_t)k * p.sBk + n;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[q] = (k < p.K && n + q < p.N && T_IN(src + q, 4, 1)) ? __ldg(src + q) : 0.0f;
                }
            }
            cp_async_commit();
        };

        float best[TM][TN];
        float snap[ARG ? TM : 1][ARG ? TN : 1];  // the second accumulator set (ARG)
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int jj = 0; jj < TN; ++jj) {
                best[i][jj] = zero;
                if constexpr (ARG) snap[i][jj] = zero;
            }

        // the stage buffers are free here: every thread passed the last loop barrier of the
        // previous pass after its final reads
        issue_b(kt0, 0);
        load_a(kt0);
        store_a(0);
        cp_async_wait_all();
        __syncthreads();
        for (int kt = kt0; kt < kt1; ++kt) {
            const int buf = (kt - kt0) & 1;
            if (kt + 1 < kt1) {
                issue_b(kt + 1, buf ^ 1);
                load_a(kt + 1);
            }
#pragma unroll
            for (int kk = 0; kk < BK; kk += 2) {
                float a0[TM], a1[TM], b0[TN], b1[TN];
                {
                    const float4 x = *reinterpret_cast<const float4*>(&As[buf][kk][tm * 4]);
                    const float4 y = *reinterpret_cast<const float4*>(&As[buf][kk][BM / 2 + tm * 4]);
                    const float4 x1 = *reinterpret_cast<const float4*>(&As[buf][kk + 1][tm * 4]);
                    const float4 y1 = *reinterpret_cast<const float4*>(&As[buf][kk + 1][BM / 2 + tm * 4]);
                    a0[0] = x.x; a0[1] = x.y; a0[2] = x.z; a0[3] = x.w;
                    a0[4] = y.x; a0[5] = y.y; a0[6] = y.z; a0[7] = y.w;
                    a1[0] = x1.x; a1[1] = x1.y; a1[2] = x1.z; a1[3] = x1.w;
                    a1[4] = y1.x; a1[5] = y1.y; a1[6] = y1.z; a1[7] = y1.w;
#pragma unroll
                    for (int h = 0; h < NG; ++h) {
                        const float4 uu = *reinterpret_cast<const float4*>(&Bs[buf][kk][h * (BN / 2) + tn * 4]);
                        const float4 u1 = *reinterpret_cast<const float4*>(&Bs[buf][kk + 1][h * (BN / 2) + tn * 4]);
                        b0[4 * h] = uu.x; b0[4 * h + 1] = uu.y; b0[4 * h + 2] = uu.z; b0[4 * h + 3] = uu.w;
                        b1[4 * h] = u1.x; b1[4 * h + 1] = u1.y; b1[4 * h + 2] = u1.z; b1[4 * h + 3] = u1.w;
                    }
                }
                if constexpr (!ARG) {
#pragma unroll
                    for (int i = 0; i < TM; ++i)
#pragma unroll
                        for (int jj = 0; jj < TN; jj += 2) {
                            const float2 t0 = O::mul2(make_float2(a0[i], a0[i]), make_float2(b0[jj], b0[jj + 1]));
                            const float2 t1 = O::mul2(make_float2(a1[i], a1[i]), make_float2(b1[jj], b1[jj + 1]));
                            best[i][jj] = O::fold3(best[i][jj], t0.x, t1.x);
                            best[i][jj + 1] = O::fold3(best[i][jj + 1], t0.y, t1.y);
                        }
                } else {
                    // The two accumulator sets swap roles every chunk: the first fold of a chunk
                    // reads the running result from one set and writes the other, so at the
                    // chunk's end the set it came from still holds the chunk-start value to
                    // compare against -- no snapshot copy.  Chunks per k-tile are even, so the
                    // running result is back in `best` at every k-tile boundary.
                    // (an odd number of chunks per k-tile keeps one set and copies it instead)
                    constexpr bool alternate = (BK / CH) % 2 == 0;
                    const bool odd = !alternate || ((kk / CH) & 1) != 0;
                    const bool first = alternate && (kk % CH) == 0;
                    float(&src_)[TM][TN] = odd ? snap : best;
                    float(&dst_)[TM][TN] = odd ? best : snap;
#pragma unroll
                    for (int i = 0; i < TM; ++i)
#pragma unroll
                        for (int jj = 0; jj < TN; jj += 2) {
                            const float2 t0 = O::mul2(make_float2(a0[i], a0[i]), make_float2(b0[jj], b0[jj + 1]));
                            const float2 t1 = O::mul2(make_float2(a1[i], a1[i]), make_float2(b1[jj], b1[jj + 1]));
                            dst_[i][jj] = O::fold3(first ? src_[i][jj] : dst_[i][jj], t0.x, t1.x);
                            dst_[i][jj + 1] = O::fold3(first ? src_[i][jj + 1] : dst_[i][jj + 1], t0.y, t1.y);
                        }
                    if ((kk + 2) % CH == 0) {
                        // end of a chunk: a strict improvement over the chunk-start value marks it
                        const uint16_t chunk = (uint16_t)((kt * BK + kk + 2) / CH - 1);
#pragma unroll
                        for (int i = 0; i < TM; ++i)
#pragma unroll
                            for (int jj = 0; jj < TN; ++jj) {
                                if (O::better(dst_[i][jj], src_[i][jj])) sid[i * TN + jj][tid] = chunk;
                                if (!alternate) src_[i][jj] = dst_[i][jj];
                            }
                    }
                }
            }
            if (kt + 1 < kt1) store_a(buf ^ 1);
            cp_async_wait_all();
            __syncthreads();
        }

        if (!sk) {
            // ---------------- store values (and -(chunk + 1)) through the output strides
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const int m = m0 + row_of(tm, i);
                if (m >= p.M) continue;
                float* crow = p.C + oc + (int64_t)m * p.sCm;
                int32_t* irow = ARG ? p.I + oi + (int64_t)m * p.sIm : nullptr;
                int32_t code[TN];
                if (ARG) {
#pragma unroll
                    for (int jj = 0; jj < TN; ++jj)
                        code[jj] = best[i][jj] != zero ? -((int32_t)sid[i * TN + jj][tid] + 1) : 0;
                }
#pragma unroll
                for (int h = 0; h < NG; ++h) {
                    const int n = n0 + h * (BN / 2) + tn * 4;
                    if (p.vecC && n + 3 < p.N) {
                        if (T_IN(crow + n, 16, 2))
                            *reinterpret_cast<float4*>(crow + n) =
                                make_float4(best[i][4 * h], best[i][4 * h + 1], best[i][4 * h + 2], best[i][4 * h + 3]);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (n + q < p.N && T_IN(crow + (int64_t)(n + q) * p.sCn, 4, 2))
                                crow[(int64_t)(n + q) * p.sCn] = best[i][4 * h + q];
                    }
                    if (ARG) {
                        if (p.vecI && n + 3 < p.N) {
                            if (T_IN(irow + n, 16, 3))
                                *reinterpret_cast<int4*>(irow + n) =
                                    make_int4(code[4 * h], code[4 * h + 1], code[4 * h + 2], code[4 * h + 3]);
                        } else {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                if (n + q < p.N && T_IN(irow + (int64_t)(n + q) * p.sIn, 4, 3))
                                    irow[(int64_t)(n + q) * p.sIn] = code[4 * h + q];
                        }
                    }
                }
            }
        } else {
            // ---------------- stream-K segment: the whole 64x64 tile, row-major, to workspace
            float* sv = p.seg_v + ((size_t)j * 2 + pass) * TILE_ELEMS;
            uint16_t* sc = ARG ? p.seg_c + ((size_t)j * 2 + pass) * TILE_ELEMS : nullptr;
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const int r = row_of(tm, i);
#pragma unroll
                for (int h = 0; h < NG; ++h) {
                    const int c = h * (BN / 2) + tn * 4;
                    if (T_IN(sv + r * BN + c, 16, 4))
                        *reinterpret_cast<float4*>(sv + r * BN + c) =
                            make_float4(best[i][4 * h], best[i][4 * h + 1], best[i][4 * h + 2], best[i][4 * h + 3]);
                    if (ARG) {
                        uint32_t cd[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            cd[q] = best[i][4 * h + q] != zero ? (uint32_t)sid[i * TN + 4 * h + q][tid] + 1u : 0u;
                        if (T_IN(sc + r * BN + c, 8, 5))
                            *reinterpret_cast<uint2*>(sc + r * BN + c) = make_uint2(cd[0] | (cd[1] << 16), cd[2] | (cd[3] << 16));
                    }
                }
            }
            // arrival ticket: the last CTA to finish a segment of this tile merges them
            const uint32_t tl = t - p.T_dp;
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                uint32_t j0, j1;
                int slot0;
                sk_segments(p, tl, j0, j1, slot0);
                const bool last = T_IN(p.sk_cnt + tl, 4, 6) && atomicAdd(&p.sk_cnt[tl], 1u) == j1 - j0;
                if (last) p.sk_cnt[tl] = 0;  // zero again for the next launch on this stream
                s_last = last;
            }
            __syncthreads();
            if (s_last) {
                __threadfence();
                sk_merge<SR, ARG, THREADS>(p, tl, m0, n0, oc, oi, tid);
            }
        }
    }
}

// ------------------------------------------------------------------ TMA-fed tiled kernel (argmax)
// The tile, thread layout and chunked argmax of k_gemm_tiled<SR, true, 4> for the common case:
// one batch axis, K a multiple of BK (every k-tile whole), 16-byte aligned rows and strides.
// A's [BM x BK] box and B's [BK x BN] box arrive by TMA (cp.async.bulk.tensor) in a ring of
// TMA_STAGES stages, each with an mbarrier that counts the bytes landed; one thread issues
// the copies, so the loads cost the other threads no address arithmetic or bounds tests.  A
// keeps its natural [m][k] layout: for every 4 k a thread reads its 4 B rows once (16 bytes
// each) and then 4 k of each of its rows with one 16-byte load.  Rows or columns past M and
// N arrive zero-filled and are never stored.
#ifndef TROP_TMA_STAGES
#define TROP_TMA_STAGES 3
#endif
#ifndef TROP_TMA_MINB
#define TROP_TMA_MINB 4
#endif
constexpr int TMA_STAGES = TROP_TMA_STAGES;
constexpr uint32_t TMA_STAGE_BYTES = (BM * BK + BK * BN) * sizeof(float);

struct TmaMaps {
    CUtensorMap a;   // A as [batch][M][K] (K fastest), box [1][BM][BK]
    CUtensorMap b;   // B as [batch][K][N] (N fastest), box [1][BK][BN]
    CUtensorMap bp;  // B again, box [1][K][FPW]: a resolve panel (fused kernel only)
};

// bounded waits on this device that gave up once (each then waited again with the full bound)
__device__ unsigned int g_wait_timeouts;

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_u32(dst)), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// shared memory of one TMA-fed tile
struct __align__(128) TmaTileSmem {
    float As[TMA_STAGES][BM][BK];
    float Bs[TMA_STAGES][BK][BN];
    uint64_t full[TMA_STAGES];  // operand boxes of a stage landed
    uint16_t sid[TM * 4][tile_threads<4>()];
    int s_fail, s_gaveup;
};

// Tile t of the TMA-fed argmax GEMM: values and -(chunk + 1) codes through the strides.  With
// PDL the programmatic-dependent wait (and the signal to the next grid) comes between the
// barrier set-up and the first copy.  *bat receives the tile's batch.
template <int SR, bool PDL, bool ARG = true>
__device__ __forceinline__ void tma_tile(const TmaMaps& maps, const TiledParams& p, uint32_t t, TmaTileSmem& sm,
                                         uint32_t* bat)
{
    using O = Ops<SR>;
    constexpr int TN = 4;
    static_assert(BK % 4 == 0 && CH % 4 == 0 && (BK / CH) % 2 == 0, "k quads, an even number of chunks per k-tile");
    auto& As = sm.As;
    auto& Bs = sm.Bs;
    auto& full = sm.full;
    auto& sid = sm.sid;
    int& s_fail = sm.s_fail;
    int& s_gaveup = sm.s_gaveup;

    const int tid = threadIdx.x;
    const int tm = tid / (BN / TN), tn = tid % (BN / TN);
    const float zero = O::zero();
    uint32_t b;
    int m0, n0;
    tile_coord(p, t, b, m0, n0);
    *bat = b;
    const int nkt = (int)p.nkt;
    if (tid == 0) {
        for (int s = 0; s < TMA_STAGES; ++s) mbar_init(&full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_fail = 0;
        s_gaveup = 0;
    }
    __syncthreads();
    if constexpr (PDL) {
        // Launched as a programmatic dependent of whatever precedes it on the stream: nothing in
        // global memory is touched before that grid has completed (the wait), so the launch only
        // hides its latency.  Then the resolve pass may start filling SMs as this grid drains.
        pdl_wait();
        pdl_signal();
    }
    auto issue = [&](int kt) {
        const int s = kt % TMA_STAGES;
        mbar_expect_tx(&full[s], TMA_STAGE_BYTES);
        tma_load_3d(&As[s][0][0], &maps.a, kt * BK, m0, (int)b, &full[s]);
        tma_load_3d(&Bs[s][0][0], &maps.b, n0, kt * BK, (int)b, &full[s]);
    };
    int issued = 0;  // k-tiles whose copies thread 0 has issued
    if (tid == 0)
        for (; issued < min(nkt, TMA_STAGES); ++issued) issue(issued);

    float best[TM][TN], snap[TM][TN];  // two accumulator sets, roles swapped every chunk
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int jj = 0; jj < TN; ++jj) best[i][jj] = snap[i][jj] = zero;

    for (int kt = 0; kt < nkt; ++kt) {
        const int s = kt % TMA_STAGES;
        const uint32_t ph = (uint32_t)(kt / TMA_STAGES) & 1u;
        // A wait that gives up is counted and waited once more with the full bound, so a copy
        // that lands late still gives exact results; if it has not landed then either, the
        // tile's results are abandoned and the failure reported (below).  Test modes 1 and 2
        // make the first wait give up at once; mode 2 then treats the second one as failed
        // after it completed, so nothing is in flight when the failure path runs.
        if (!((p.wait_mode == 0 || kt != 0) && mbar_wait(&full[s], ph))) {
            s_gaveup = 1;
            if (!mbar_wait(&full[s], ph) || p.wait_mode == 2) s_fail = 1;
        }
#pragma unroll
        for (int kq = 0; kq < BK; kq += 4) {
            // chunk parity and the first quad of a chunk are known at compile time (BK / CH even)
            const bool odd = ((kq / CH) & 1) != 0;
            const bool first = (kq % CH) == 0;
            float(&src_)[TM][TN] = odd ? snap : best;
            float(&dst_)[TM][TN] = odd ? best : snap;
            float bq[4][TN];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float4 v = *reinterpret_cast<const float4*>(&Bs[s][kq + r][tn * 4]);
                bq[r][0] = v.x; bq[r][1] = v.y; bq[r][2] = v.z; bq[r][3] = v.w;
            }
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const float4 a4 = *reinterpret_cast<const float4*>(&As[s][row_of(tm, i)][kq]);
                const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int kp = 0; kp < 4; kp += 2) {
                    const bool ff = first && kp == 0;
#pragma unroll
                    for (int jj = 0; jj < TN; jj += 2) {
                        const float2 t0 = O::mul2(make_float2(av[kp], av[kp]), make_float2(bq[kp][jj], bq[kp][jj + 1]));
                        const float2 t1 =
                            O::mul2(make_float2(av[kp + 1], av[kp + 1]), make_float2(bq[kp + 1][jj], bq[kp + 1][jj + 1]));
                        if constexpr (ARG) {
                            dst_[i][jj] = O::fold3(ff ? src_[i][jj] : dst_[i][jj], t0.x, t1.x);
                            dst_[i][jj + 1] = O::fold3(ff ? src_[i][jj + 1] : dst_[i][jj + 1], t0.y, t1.y);
                        } else {  // no argmax: one accumulator set, no chunk marks
                            best[i][jj] = O::fold3(best[i][jj], t0.x, t1.x);
                            best[i][jj + 1] = O::fold3(best[i][jj + 1], t0.y, t1.y);
                        }
                    }
                }
            }
            if (ARG && (kq + 4) % CH == 0) {
                // end of a chunk: a strict improvement over the chunk-start value marks it
                const uint16_t chunk = (uint16_t)((kt * BK + kq + 4) / CH - 1);
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int jj = 0; jj < TN; ++jj)
                        if (O::better(dst_[i][jj], src_[i][jj])) sid[i * TN + jj][tid] = chunk;
            }
        }
        __syncthreads();  // every thread is done with stage s (and sees the same s_fail)
        if (s_fail) break;
        if (tid == 0 && issued < nkt) issue(issued++);
    }
    int64_t oa, ob, oc, oi;
    batch_offsets(p.bt, b, oa, ob, oc, oi);
    // (fused kernel: the grid before may still run when its wait was left until the stores;
    // nothing is stored before it has completed)
    if constexpr (!PDL) pdl_wait();
    if (tid == 0 && s_gaveup) atomicAdd(&g_wait_timeouts, 1u);
    if (s_fail) {
        // Abandon the tile: wait (bounded) for every copy still in flight into this CTA's
        // shared memory, mark its outputs "nothing to resolve" so the resolve pass reads no
        // stale chunk codes, and report the failure in the host-mapped error word.
        if (tid == 0)
            for (int k2 = max(0, issued - TMA_STAGES); k2 < issued; ++k2)
                (void)mbar_wait(&full[k2 % TMA_STAGES], (uint32_t)(k2 / TMA_STAGES) & 1u);
        if constexpr (ARG) {
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const int m = m0 + row_of(tm, i);
                if (m >= p.M) continue;
                int32_t* irow = p.I + oi + (int64_t)m * p.sIm;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (n0 + tn * 4 + q < p.N && T_IN(irow + (int64_t)(n0 + tn * 4 + q) * p.sIn, 4, 3))
                        irow[(int64_t)(n0 + tn * 4 + q) * p.sIn] = 0;
            }
        }
        if (tid == 0 && p.err) {
            *(volatile uint32_t*)p.err = 1u;
            __threadfence_system();
        }
        return;
    }

    // ---------------- store values and -(chunk + 1) (0: nothing beat the zero) through the strides
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int m = m0 + row_of(tm, i);
        if (m >= p.M) continue;
        float* crow = p.C + oc + (int64_t)m * p.sCm;
        const int n = n0 + tn * 4;
        if (p.vecC && n + 3 < p.N) {
            if (T_IN(crow + n, 16, 2))
                *reinterpret_cast<float4*>(crow + n) = make_float4(best[i][0], best[i][1], best[i][2], best[i][3]);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (n + q < p.N && T_IN(crow + (int64_t)(n + q) * p.sCn, 4, 2)) crow[(int64_t)(n + q) * p.sCn] = best[i][q];
        }
        if constexpr (!ARG) continue;
        int32_t* irow = p.I + oi + (int64_t)m * p.sIm;
        int32_t code[TN];
#pragma unroll
        for (int jj = 0; jj < TN; ++jj) code[jj] = best[i][jj] != zero ? -((int32_t)sid[i * TN + jj][tid] + 1) : 0;
        if (p.vecI && n + 3 < p.N) {
            if (T_IN(irow + n, 16, 3)) *reinterpret_cast<int4*>(irow + n) = make_int4(code[0], code[1], code[2], code[3]);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (n + q < p.N && T_IN(irow + (int64_t)(n + q) * p.sIn, 4, 3)) irow[(int64_t)(n + q) * p.sIn] = code[q];
        }
    }
}

template <int SR>
__global__ void __launch_bounds__(tile_threads<4>(), TROP_TMA_MINB)
    k_gemm_tma(const __grid_constant__ TmaMaps maps, TiledParams p)
{
    __shared__ TmaTileSmem sm;
    uint32_t b;
    tma_tile<SR, true>(maps, p, blockIdx.x, sm, &b);
}

// The same TMA-fed tile without argmax (one accumulator set, no chunk marks, C only).  Like the
// one-launch argmax GEMM below it may start early behind a GEMM that wrote none of its operands
// (p.late): it then waits for the grid before only ahead of its stores.
#ifndef TROP_TMA_PLAIN_MINB
#define TROP_TMA_PLAIN_MINB 4
#endif
template <int SR>
__global__ void __launch_bounds__(tile_threads<4>(), TROP_TMA_PLAIN_MINB)
    k_gemm_tma_plain(const __grid_constant__ TmaMaps maps, TiledParams p)
{
    __shared__ TmaTileSmem sm;
    if (!p.late) pdl_wait();
    pdl_signal();
    uint32_t b;
    tma_tile<SR, false, false>(maps, p, blockIdx.x, sm, &b);
}

// ------------------------------------------------------------------ fused GEMM + short-K resolve
// One launch does both passes for K <= 256.  Its CTAs take work items in order from a counter:
// first the GEMM tiles (batch-major), then the resolve items, each a block of FRB rows of one
// FPW-column panel of one batch.  A resolve item waits (bounded) until every tile of its batch
// has been stored, so in the last, part-filled wave of tiles the CTAs left over already resolve
// the batches finished in the waves before -- the resolve fills the GEMM's tail instead of
// following it.  Items are handed out in order, so a resolve item is taken only after every
// tile has been taken by a running CTA: the tiles it waits for are resident and finish without
// waiting on anything, hence no deadlock whatever the block scheduler does.
//
// A resolve item stages B's panel [K][FPW] (32 KiB at K = 256) by one TMA copy, issued before
// the wait.  A warp takes rows r0 + w, r0 + w + 4, ...; lane l owns column n0 + l.  Lane l also
// loads chunk l of the row's A; an output pending in chunk c takes that chunk's values from
// lane c by shuffles and B's from the staged panel (lane l reads column l: no bank conflict),
// and the first k whose product attains the chunk's best product is the argmax.  FG rows are
// loaded per group, and the next group is in flight while one is searched.
// A lane's chunk of A: one 32-byte load when the rows are 32-byte aligned (V8), else two 16-byte ones
template <bool V8>
__device__ __forceinline__ void load_chunk(const float* p, float (&a)[CH])
{
    if constexpr (V8) {
        asm volatile("ld.global.nc.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=f"(a[0]), "=f"(a[1]), "=f"(a[2]), "=f"(a[3]), "=f"(a[4]), "=f"(a[5]), "=f"(a[6]), "=f"(a[7])
                     : "l"(p));
    } else {
        const float4 x = __ldg(reinterpret_cast<const float4*>(p));
        const float4 y = __ldg(reinterpret_cast<const float4*>(p + 4));
        a[0] = x.x, a[1] = x.y, a[2] = x.z, a[3] = x.w, a[4] = y.x, a[5] = y.y, a[6] = y.z, a[7] = y.w;
    }
}

constexpr int FPW = 32;  // resolve panel columns, one per lane
#ifndef TROP_FUSED_ROWS
#define TROP_FUSED_ROWS 256
#endif
constexpr int FRB = TROP_FUSED_ROWS;  // rows of a resolve item
#ifndef TROP_FUSED_FG
#define TROP_FUSED_FG 4
#endif
constexpr int FG = TROP_FUSED_FG;     // rows of a warp in one load group
constexpr int FWARPS = tile_threads<4>() / 32;

struct __align__(128) FusedResolveSmem {
    float EB[32 * CH][FPW];  // the panel's rows of B (K <= 32 chunks)
    uint64_t bar;
};
union FusedSmem {
    TmaTileSmem g;
    FusedResolveSmem r;
};

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* ptr)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}
// Wait until *ctr >= need (acquire); false after about one second without it.
__device__ __forceinline__ bool wait_count(const uint32_t* ctr, uint32_t need)
{
    if (ld_acquire_u32(ctr) >= need) return true;
    const uint64_t t0 = global_ns();
    while (ld_acquire_u32(ctr) < need) {
        if (global_ns() - t0 > 1000000000ull) return false;
        __nanosleep(256);
    }
    return true;
}

template <int SR, bool V8>
__device__ __forceinline__ void fused_resolve(const TmaMaps& maps, const TiledParams& p, uint32_t r,
                                              FusedResolveSmem& sm, int& s_ok)
{
    using O = Ops<SR>;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t b = fdiv(r, p.div_ipb);
    const uint32_t rem = r - b * p.items_per_batch;
    const uint32_t pn = fdiv(rem, p.div_rblocks);
    const int n0 = (int)pn * FPW;
    const int r0 = (int)(rem - pn * p.rblocks) * FRB;
    const int r1 = min(p.M, r0 + FRB);
    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (tid == 0) {
        // B's panel is an input of the GEMM, not a result: its copy overlaps the waits
        mbar_expect_tx(&sm.bar, (uint32_t)(p.K * FPW * sizeof(float)));
        tma_load_3d(&sm.EB[0][0], &maps.bp, n0, 0, (int)b, &sm.bar);
    }
    // the grid before has completed (when it was not waited for at the start): the counters of
    // this ticket half were last used two launches back, by a grid now complete
    pdl_wait();
    if (tid == 0)
        s_ok = T_IN(p.sched + 1 + b, 4, 7) && wait_count(p.sched + 1 + b, p.tiles_per_batch) ? 1 : 0;
    const bool landed = mbar_wait(&sm.bar, 0);
    // thread 0's acquire of the batch's count, then this barrier: the batch's codes are visible
    const bool all_landed = __syncthreads_and(landed ? 1 : 0) != 0;
    if (!s_ok || !all_landed) {
        // a wait gave up: leave the codes (the results are undefined), let the panel copy land
        // before the CTA exits, and report the failure in the host-mapped error word
        if (!landed) (void)mbar_wait(&sm.bar, 0);
        if (tid == 0 && p.err) {
            *(volatile uint32_t*)p.err = 1u;
            __threadfence_system();
        }
        return;
    }
    const int nchunks = p.K / CH;
    int64_t oa, ob, oc, oi;
    batch_offsets(p.bt, b, oa, ob, oc, oi);
    const int achunk = min(lane, nchunks - 1);  // lanes past the last chunk read it again (unused)
    const float* __restrict__ Al = p.A + oa + achunk * CH;
    const int ncl = p.N - 1 - n0;  // the panel's last column
    const bool colok = lane <= ncl;
    const int32_t* __restrict__ Ir = p.I + oi + n0 + min(lane, ncl);
    int32_t* __restrict__ Iw = p.I + oi + n0 + lane;
    const int sA = p.sAm32, sI = p.sIm32;
    const float* eb0 = &sm.EB[0][lane];
    struct Row {
        int32_t c;
        float a[CH];
    };
    constexpr int STEP = FWARPS * FG;  // rows between a warp's groups
    auto load = [&](Row (&g)[FG], int mb) {
#pragma unroll
        for (int j = 0; j < FG; ++j) {
            const int m = mb + j * FWARPS;
            const int mm = m < r1 ? m : r1 - 1;
            // codes were stored by other CTAs of this launch: read them through L2
            g[j].c = T_IN(Ir + (int64_t)mm * sI, 4, 3) ? __ldcg(Ir + (int64_t)mm * sI) : 0;
            if (T_IN(Al + (int64_t)mm * sA, 4 * CH, 0)) {
                load_chunk<V8>(Al + (int64_t)mm * sA, g[j].a);
            } else {
#pragma unroll
                for (int kk = 0; kk < CH; ++kk) g[j].a[kk] = 0.0f;
            }
        }
    };
    auto search = [&](const Row (&g)[FG], int mb) {
#pragma unroll
        for (int j = 0; j < FG; ++j) {
            const int m = mb + j * FWARPS;
            // code -(c + 1): chunk c pending; 0: final (nothing beat the zero)
            const bool live = m < r1 && colok && g[j].c < 0 && ~g[j].c < nchunks;
            const int c = live ? ~g[j].c : 0;
            float a[CH], t[CH];
#pragma unroll
            for (int kk = 0; kk < CH; ++kk) a[kk] = __shfl_sync(0xffffffffu, g[j].a[kk], c);
            const float* eb = eb0 + c * (CH * FPW);
#pragma unroll
            for (int kk = 0; kk < CH; ++kk) t[kk] = O::mul(a[kk], eb[kk * FPW]);
            // the chunk's best product is the output's value; its first k is the argmax
            const float p1 = O::fold3(t[0], t[1], t[1]);
            const float p3 = O::fold3(p1, t[2], t[3]);
            const float p5 = O::fold3(p3, t[4], t[5]);
            const float v = O::fold3(p5, t[6], t[7]);
            const bool s2 = p3 != v;
            const bool s1 = (s2 ? p5 : p1) != v;
            const float x = s2 ? (s1 ? t[6] : t[4]) : (s1 ? t[2] : t[0]);
            const int idx = (s2 ? 4 : 0) + (s1 ? 2 : 0) + (x != v ? 1 : 0);
            if (live && T_IN(Iw + (int64_t)m * sI, 4, 3)) Iw[(int64_t)m * sI] = c * CH + idx;
        }
    };
    Row g0[FG], g1[FG];
    int ms = r0 + warp;
    if (ms < r1) load(g0, ms);
    while (ms < r1) {
        if (ms + STEP < r1) load(g1, ms + STEP);
        search(g0, ms);
        ms += STEP;
        if (ms >= r1) break;
        if (ms + STEP < r1) load(g0, ms + STEP);
        search(g1, ms);
        ms += STEP;
    }
    __syncthreads();
    if (tid == 0 && T_IN(p.sched + 1 + p.nbatch + b, 4, 7) &&
        atomicAdd(p.sched + 1 + p.nbatch + b, 1u) == p.items_per_batch - 1) {
        // the batch's last resolve item: every item of it has passed its wait, so the batch's
        // counters can be zeroed for the next launch
        p.sched[1 + b] = 0;
        p.sched[1 + p.nbatch + b] = 0;
    }
}

template <int SR, bool V8>
__global__ void __launch_bounds__(tile_threads<4>(), TROP_TMA_MINB)
    k_gemm_tma_fused(const __grid_constant__ TmaMaps maps, TiledParams p)
{
    __shared__ FusedSmem sm;
    __shared__ uint32_t s_item;
    __shared__ int s_ok;
    // A programmatic dependent of the grid before.  Normally nothing starts before that grid
    // has completed.  With p.late (that grid is a fused GEMM whose outputs this launch does not
    // read) the tiles load and compute at once and wait only ahead of their stores, and the
    // resolve items ahead of their counters.  The item counter is the other half of the
    // stream's tickets: its last user is the launch two back, whose CTAs had all taken their
    // items (and the last one zeroed it) before the grid before was let start.
    if (!p.late) pdl_wait();
    if (threadIdx.x == 0) {
        const uint32_t it = T_IN(p.sched, 4, 7) ? atomicAdd(p.sched, 1u) : 0u;
        if (it == p.n_items - 1) {
            // the last item taken: zero the counter for the launch after next, performed before
            // this CTA lets the next launch start
            p.sched[0] = 0;
            __threadfence();
        }
        s_item = it;
    }
    __syncthreads();
    pdl_signal();  // after the claim: the next launch may reuse the counters this one left
    const uint32_t it = s_item;
    if (it < p.n_tiles) {
        uint32_t b;
        tma_tile<SR, false>(maps, p, it, sm.g, &b);
        // publish the tile: its values and codes are stored
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0 && T_IN(p.sched + 1 + b, 4, 7)) atomicAdd(p.sched + 1 + b, 1u);
    } else if (it < p.n_items) {
        fused_resolve<SR, V8>(maps, p, it - p.n_tiles, sm.r, s_ok);
    }
}

// ------------------------------------------------------------------ argmax resolve
// Replaces each pending chunk by the exact first index.  The CTAs split the rows of all
// 64-column panels (batch, column tile) evenly.  For each panel a CTA stages B's rows for
// those columns into shared memory, RGK rows at a time; warp w then takes rows in steps of
// RR, lane l owning columns l and l + 32 -- so the staged reads B[k][n] of a warp hit 32
// distinct banks whatever chunk each lane needs.  An output whose chunk lies in the staged
// group recomputes that chunk's CH products, A's contiguous segment coming through L1, and
// keeps the first k whose product equals the value.  The (C, I) loads of a warp's next row
// step are issued before the current step's search.  Launched as a programmatic dependent
// of the GEMM, a CTA stages its first B rows before waiting for the GEMM's results.
#ifndef TROP_RESOLVE_RR
#define TROP_RESOLVE_RR 4
#endif
#ifndef TROP_RESOLVE_MINB
#define TROP_RESOLVE_MINB 2
#endif
constexpr int RTHREADS = 256, RWARPS = RTHREADS / 32, RGK = 256;  // B rows staged per group (64 columns)
constexpr int RR = CH <= 8 ? TROP_RESOLVE_RR : 2;  // rows per warp step: RR x 2 outputs per lane
constexpr size_t SMEM_RESOLVE = sizeof(float) * RGK * BN;  // 64 KiB
static_assert(RGK % CH == 0, "a chunk never straddles two staged groups");

// The rows mb .. me-1 of one staged group of a PW-column panel, for the common layout: C
// and I with unit column stride, every chunk whole (K a multiple of CH) and A's segments
// 16-byte aligned.  A lane owns NCOL columns (l, l + 32 for PW = 64) of RSUB interleaved rows
// (lanes l and l + PW for PW = 16) per row slot, RRP row slots per step.  Branch free per
// output: a dead output (no pending chunk in this group) loads A's first segment, searches
// the first staged rows and stores nothing.
template <int PW>
struct PanelShape {
    static constexpr int NCOL = PW >= 64 ? PW / 32 : 1;  // columns per lane
    static constexpr int RSUB = PW >= 32 ? 1 : 32 / PW;  // rows sharing a row slot
    static constexpr int RRP = PW >= 64 ? RR : 2 * RR;   // row slots per lane and step
    static constexpr int ROWS = RRP * RSUB;              // rows per warp step
    static constexpr int GK = (int)(SMEM_RESOLVE / sizeof(float)) / PW;  // B rows per staged group
};

template <int SR, int PW>
__device__ __forceinline__ void resolve_rows_fast(const TiledParams& p, const float* __restrict__ EB,
                                                  const float* __restrict__ A, const float* __restrict__ Cb,
                                                  int32_t* __restrict__ Ib, int n0, int mb, int me, int k0,
                                                  int kn, int warp, int lane)
{
    using O = Ops<SR>;
    using S = PanelShape<PW>;
    constexpr int NCOL = S::NCOL, RSUB = S::RSUB, RRP = S::RRP, ROWS = S::ROWS;
    const int nchunks = p.K / CH;  // whole chunks on this path
    const int cl = PW >= 32 ? lane : lane % PW;  // column (of the first column group)
    const int rs = PW >= 32 ? 0 : lane / PW;     // row within a row slot
    bool colok[NCOL];
#pragma unroll
    for (int h = 0; h < NCOL; ++h) colok[h] = n0 + h * 32 + cl < p.N;
    const float* __restrict__ cb = Cb + n0 + cl;
    int32_t* __restrict__ ib = Ib + n0 + cl;
    float nval[RRP][NCOL];
    int32_t ncode[RRP][NCOL];
    auto load_step = [&](int ms) {
#pragma unroll
        for (int r = 0; r < RRP; ++r) {
            const int m = ms + r * RSUB + rs;
            const float* cr = cb + (int64_t)m * p.sCm;
            const int32_t* ir = ib + (int64_t)m * p.sIm;
#pragma unroll
            for (int h = 0; h < NCOL; ++h) {
                const bool ok = m < me && colok[h];
                nval[r][h] = ok && T_IN(cr + h * 32, 4, 2) ? cr[h * 32] : 0.0f;
                ncode[r][h] = ok && T_IN(ir + h * 32, 4, 3) ? ir[h * 32] : 0;
            }
        }
    };
    int ms = mb + warp * ROWS;
    if (ms < me) load_step(ms);
    for (; ms < me; ms += RWARPS * ROWS) {
        float val[RRP][NCOL];
        int ka[RRP][NCOL];
        bool live[RRP][NCOL];
#pragma unroll
        for (int r = 0; r < RRP; ++r)
#pragma unroll
            for (int h = 0; h < NCOL; ++h) {
                val[r][h] = nval[r][h];
                // a code is live when it names a chunk of this staged group (a code outside
                // the contraction is never followed, whatever the buffer held)
                const int ch = ncode[r][h] < 0 ? -(ncode[r][h] + 1) : INT_MAX;
                const int kc = ch < nchunks ? ch * CH : -1;
                live[r][h] = kc >= k0 && kc < k0 + kn;
                ka[r][h] = live[r][h] ? kc : k0;
            }
        if (ms + RWARPS * ROWS < me) load_step(ms + RWARPS * ROWS);
        float av[RRP][NCOL][CH];
#pragma unroll
        for (int r = 0; r < RRP; ++r) {
            const int m = ms + r * RSUB + rs;
            // a row past me (end of the range) reads row mb instead: always inside A
            const float* arow = A + (int64_t)(m < me ? m : mb) * p.sAm;
#pragma unroll
            for (int h = 0; h < NCOL; ++h)
#pragma unroll
                for (int kk = 0; kk < CH; kk += 4) {
                    const float4 x = T_IN(arow + ka[r][h] + kk, 16, 0)
                                         ? __ldg(reinterpret_cast<const float4*>(arow + ka[r][h] + kk))
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                    av[r][h][kk] = x.x;
                    av[r][h][kk + 1] = x.y;
                    av[r][h][kk + 2] = x.z;
                    av[r][h][kk + 3] = x.w;
                }
        }
#pragma unroll
        for (int r = 0; r < RRP; ++r)
#pragma unroll
            for (int h = 0; h < NCOL; ++h) {
                const float* eb = EB + (ka[r][h] - k0) * PW + h * 32 + cl;
                int idx = 0;
#pragma unroll
                for (int kk = CH - 2; kk >= 0; kk -= 2) {
                    const float2 t = O::mul2(make_float2(av[r][h][kk], av[r][h][kk + 1]),
                                             make_float2(eb[kk * PW], eb[(kk + 1) * PW]));
                    idx = t.y == val[r][h] ? kk + 1 : idx;
                    idx = t.x == val[r][h] ? kk : idx;
                }
                if (live[r][h] && T_IN(ib + (int64_t)(ms + r * RSUB + rs) * p.sIm + h * 32, 4, 3))
                    ib[(int64_t)(ms + r * RSUB + rs) * p.sIm + h * 32] = ka[r][h] + idx;
            }
    }
}

// PW: columns per panel.  A narrower panel stages more B rows in the same 64 KiB (GK = 256,
// 512, 1024 for PW = 64, 32, 16), so a long contraction needs fewer passes over the rows;
// only the common layout (resolve_rows_fast) runs with PW < 64.
template <int SR, int PW>
__global__ void __launch_bounds__(RTHREADS, TROP_RESOLVE_MINB) k_argmax_resolve(TiledParams p)
{
    pdl_signal();  // a programmatic dependent (the next GEMM) may take SMs as this grid drains
    using O = Ops<SR>;
    constexpr int GK = PanelShape<PW>::GK;
    static_assert(GK % CH == 0, "a chunk never straddles two staged groups");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* EBf = reinterpret_cast<float*>(smem_raw);
    float(*EB)[BN] = reinterpret_cast<float(*)[BN]>(smem_raw);  // the PW = 64 view
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t ubeg, uend;
    resolve_range(p, ubeg, uend);
    const int ngr = (p.K + GK - 1) / GK;
    const int nchunks = (p.K + CH - 1) / CH;
    const uint32_t npan = (uint32_t)((p.N + PW - 1) / PW);  // panels per batch
    // common layout: unit column strides, whole chunks, 16-byte aligned A segments
    const bool fast = p.vecA && p.K % CH == 0 && p.sCn == 1 && p.sIn == 1;
    bool waited = false;
    for (uint64_t u = ubeg; u < uend;) {
        // rows mb .. me-1 of panel pn
        uint32_t b;
        int n0, mb;
        resolve_unit(p, u, npan, PW, b, n0, mb);
        const int me = (int)min((uint64_t)p.M, (uint64_t)mb + (uend - u));
        u += (uint64_t)(me - mb);
        int64_t oa, ob, oc, oi;
        batch_offsets(p.bt, b, oa, ob, oc, oi);
        const float* __restrict__ A = p.A + oa;
        const float* __restrict__ B = p.B + ob;
        const float* __restrict__ Cb = p.C + oc;
        int32_t* __restrict__ Ib = p.I + oi;
        bool colok[2];
        int64_t offC[2], offI[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = n0 + h * 32 + lane;
            colok[h] = n < p.N;
            offC[h] = (int64_t)n * p.sCn;
            offI[h] = (int64_t)n * p.sIn;
        }
        for (int g = 0; g < ngr; ++g) {
            const int k0 = g * GK;
            const int kn = min(GK, p.K - k0);
            __syncthreads();  // every warp is done with the rows staged before
            for (int e = tid; e < kn * (PW / 4); e += RTHREADS) {
                const int kk = e / (PW / 4), nq = (e % (PW / 4)) * 4, gk = k0 + kk, gn = n0 + nq;
                float* dst = EBf + kk * PW + nq;
                if (p.vecB) {
                    int valid = max(0, min(4, p.N - gn));
                    if (valid && !T_IN(B + (int64_t)gk * p.sBk + gn, valid * 4, 1)) valid = 0;
                    cp_async16(dst, valid ? B + (int64_t)gk * p.sBk + gn : B, valid * 4);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[q] = (gn + q < p.N && T_IN(B + (int64_t)gk * p.sBk + gn + q, 4, 1))
                                     ? __ldg(B + (int64_t)gk * p.sBk + gn + q)
                                     : 0.0f;
                }
            }
            cp_async_commit();
            cp_async_wait_all();
            __syncthreads();
            if (!waited) {
                pdl_wait();  // C and I come from the GEMM grid (B above is its input)
                waited = true;
            }

            if (fast) {
                resolve_rows_fast<SR, PW>(p, EBf, A, Cb, Ib, n0, mb, me, k0, kn, warp, lane);
                continue;
            }
            if constexpr (PW != BN) continue;  // (the host sends other layouts to PW = 64)
            float nval[RR][2];
            int32_t ncode[RR][2];
            auto load_step = [&](int ms) {
#pragma unroll
                for (int r = 0; r < RR; ++r) {
                    const int m = ms + r;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const bool in = m < me && colok[h];
                        nval[r][h] = in && T_IN(Cb + (int64_t)m * p.sCm + offC[h], 4, 2) ? Cb[(int64_t)m * p.sCm + offC[h]] : 0.0f;
                        ncode[r][h] = in && T_IN(Ib + (int64_t)m * p.sIm + offI[h], 4, 3) ? Ib[(int64_t)m * p.sIm + offI[h]] : 0;
                    }
                }
            };
            int ms = mb + warp * RR;
            if (ms < me) load_step(ms);
            for (; ms < me; ms += RWARPS * RR) {
                float val[RR][2];
                int ka[RR][2];  // first k of the pending chunk, or -1
#pragma unroll
                for (int r = 0; r < RR; ++r)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        val[r][h] = nval[r][h];
                        // ncode < 0: chunk -ncode-1 (never followed outside the contraction)
                        const int ch = ncode[r][h] < 0 ? -(ncode[r][h] + 1) : INT_MAX;
                        const int kc = ch < nchunks ? ch * CH : -1;
                        ka[r][h] = (kc >= k0 && kc < k0 + kn) ? kc : -1;
                    }
                if (ms + RWARPS * RR < me) load_step(ms + RWARPS * RR);
                float av[RR][2][CH];
#pragma unroll
                for (int r = 0; r < RR; ++r) {
                    const float* arow = A + (int64_t)(ms + r) * p.sAm;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int kmax = ka[r][h] >= 0 ? min(CH, p.K - ka[r][h]) : 0;
                        const float* src = arow + (ka[r][h] >= 0 ? ka[r][h] : 0);
#pragma unroll
                        for (int kk = 0; kk < CH; ++kk)
                            av[r][h][kk] = kk < kmax && T_IN(src + kk, 4, 0) ? __ldg(src + kk) : 0.0f;
                    }
                }
#pragma unroll
                for (int r = 0; r < RR; ++r)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (ka[r][h] < 0) continue;
                        const int kl = ka[r][h] - k0, c = h * 32 + lane;
                        const int kmax = min(CH, p.K - ka[r][h]);
                        int idx = 0;
#pragma unroll
                        for (int kk = CH - 1; kk >= 0; --kk)
                            if (kk < kmax && O::mul(av[r][h][kk], EB[kl + kk][c]) == val[r][h]) idx = kk;
                        if (T_IN(Ib + (int64_t)(ms + r) * p.sIm + offI[h], 4, 3))
                            Ib[(int64_t)(ms + r) * p.sIm + offI[h]] = ka[r][h] + idx;
                    }
            }
        }
    }
    // every CTA waits once, so this grid ends after the GEMM grid whatever its row range
    if (!waited) pdl_wait();
}

// ------------------------------------------------------------------ argmax resolve, short K
// The same replacement for contractions of at most 32 chunks (K <= 256) in the common layout
// (unit column strides, whole chunks, 16-byte aligned A rows, row strides below 2^31).  A warp
// takes one row of a 64-column panel per step.  Lane l loads chunk l of the row (one 32-byte
// load when the rows are 32-byte aligned) -- the warp reads the row once, coalesced -- and an
// output whose pending chunk is c takes that chunk's CH values of A from lane c by shuffles;
// B's rows sit in shared memory as in the general pass (lane l owns columns l and l + 32, so
// the staged reads are free of bank conflicts).  The value C is not read: it is the best
// product of the pending chunk.  No global load waits on another, so the next row's codes and
// A are in flight while a row is searched; the two rows in flight live in two register sets
// used in turn.
#ifndef TROP_RESOLVE2_MINB
#define TROP_RESOLVE2_MINB 3
#endif
constexpr int SHORT_K = 32 * CH;  // one chunk per lane
static_assert(SHORT_K <= RGK, "the staged B rows cover a short contraction");
static_assert(CH == 8, "the short resolve searches a chunk of 8 by halving");

template <int SR, bool V8>
__global__ void __launch_bounds__(RTHREADS, TROP_RESOLVE2_MINB) k_argmax_resolve_rows(TiledParams p)
{
    pdl_signal();  // a programmatic dependent (the next GEMM) may take SMs as this grid drains
    using O = Ops<SR>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* EB = reinterpret_cast<float*>(smem_raw);  // [K][BN]: the panel's rows of B
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t ubeg, uend;
    resolve_range(p, ubeg, uend);
    const uint32_t npan = (uint32_t)((p.N + BN - 1) / BN);
    // lane l holds chunk l of every row; lanes past the last chunk read the last one (unused)
    const int achunk = min(lane, p.K / CH - 1);
    const int nchunks = p.K / CH;
    const int sA = p.sAm32, sI = p.sIm32;
    bool waited = false;
    for (uint64_t u = ubeg; u < uend;) {
        // rows mb .. me-1 of panel pn
        uint32_t b;
        int n0, mb;
        resolve_unit(p, u, npan, BN, b, n0, mb);
        const int me = (int)min((uint64_t)p.M, (uint64_t)mb + (uend - u));
        u += (uint64_t)(me - mb);
        int64_t oa, ob, oc, oi;
        batch_offsets(p.bt, b, oa, ob, oc, oi);
        // loads are never predicated: a column past N reads column N - 1 and a row past the
        // range reads its last row; neither is searched or stored
        const int ncl = p.N - 1 - n0;
        const int c0 = min(lane, ncl), c1 = min(lane + 32, ncl);
        const float* __restrict__ Al = p.A + oa + achunk * CH;
        const float* __restrict__ B = p.B + ob;
        const int32_t* __restrict__ Ib = p.I + oi + n0;
        int32_t* __restrict__ Il = p.I + oi + n0 + lane;

        __syncthreads();  // every warp is done with the previous panel's rows
        {
            // thread -> column quad tid % 16 of rows tid / 16 + 16 i; zero fill past N
            const int q = (tid % (BN / 4)) * 4, n = n0 + q;
            const int valid = max(0, min(4, p.N - n));
            const float* src = valid ? B + n : B;
            const int64_t step = valid ? p.sBk * (RTHREADS / (BN / 4)) : 0;
            src += valid ? (int64_t)(tid / (BN / 4)) * p.sBk : 0;
            if (p.vecB) {  // 16-byte aligned rows of B
                for (int k = tid / (BN / 4); k < p.K; k += RTHREADS / (BN / 4), src += step)
                    cp_async16(EB + k * BN + q, src, valid && T_IN(src, valid * 4, 1) ? valid * 4 : 0);
                cp_async_commit();
                cp_async_wait_all();
            } else {
                for (int k = tid / (BN / 4); k < p.K; k += RTHREADS / (BN / 4), src += step) {
                    float v[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[e] = e < valid && T_IN(src + e, 4, 1) ? __ldg(src + e) : 0.0f;
                    *reinterpret_cast<float4*>(EB + k * BN + q) = make_float4(v[0], v[1], v[2], v[3]);
                }
            }
        }
        __syncthreads();
        if (!waited) {
            pdl_wait();  // C and I come from the GEMM grid (B above is its input)
            waited = true;
        }

        const bool col0 = lane <= ncl, col1 = lane + 32 <= ncl;
        // one row per warp step, two register sets used in turn (no copy between steps)
        struct RowSet {
            int32_t c[2];
            float a[CH];
            bool ok[2];
        };
        auto load_row = [&](RowSet& s, int m) {
            const bool rok = m < me;
            const int mm = rok ? m : me - 1;
            const int32_t* ir = Ib + (int64_t)mm * sI;
            const float* ar = Al + (int64_t)mm * sA;
            s.c[0] = T_IN(ir + c0, 4, 3) ? ir[c0] : 0;
            s.c[1] = T_IN(ir + c1, 4, 3) ? ir[c1] : 0;
            if (T_IN(ar, 4 * CH, 0)) {
                load_chunk<V8>(ar, s.a);
            } else {
#pragma unroll
                for (int kk = 0; kk < CH; ++kk) s.a[kk] = 0.0f;
            }
            s.ok[0] = rok && col0;
            s.ok[1] = rok && col1;
        };
        auto search_row = [&](const RowSet& s, int m) {
            int32_t* irow = Il + (int64_t)m * sI;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                // code -(c + 1): chunk c pending; 0: final (nothing beat the zero)
                const bool live = s.ok[h] && s.c[h] < 0 && ~s.c[h] < nchunks;
                const int c = live ? ~s.c[h] : 0;
                float a[CH];
#pragma unroll
                for (int kk = 0; kk < CH; ++kk) a[kk] = __shfl_sync(0xffffffffu, s.a[kk], c);
                const float* eb = EB + c * (CH * BN) + h * 32 + lane;
                // Chunk c is the last one whose products strictly raised the running result, so
                // the largest of its products (smallest for min-plus) is the output's value v and
                // no product of the chunk passes it: the prefix (+) of the products first reaches
                // v at the first k that attains it.  Halve the range on the prefixes of 4 and then
                // 2 products, then test one product.
                float t[CH];
#pragma unroll
                for (int kk = 0; kk < CH; ++kk) t[kk] = O::mul(a[kk], eb[kk * BN]);
                const float p1 = O::fold3(t[0], t[1], t[1]);
                const float p3 = O::fold3(p1, t[2], t[3]);
                const float p5 = O::fold3(p3, t[4], t[5]);
                const float v = O::fold3(p5, t[6], t[7]);
                const bool s2 = p3 != v;
                const bool s1 = (s2 ? p5 : p1) != v;
                const float x = s2 ? (s1 ? t[6] : t[4]) : (s1 ? t[2] : t[0]);
                const int idx = (s2 ? 4 : 0) + (s1 ? 2 : 0) + (x != v ? 1 : 0);
                if (live && T_IN(irow + h * 32, 4, 3)) irow[h * 32] = c * CH + idx;
            }
        };
        constexpr int WSTEP = RWARPS;
        int ms = mb + warp;
        RowSet s0, s1;
        if (ms < me) load_row(s0, ms);
        while (ms < me) {
            if (ms + WSTEP < me) load_row(s1, ms + WSTEP);
            search_row(s0, ms);
            ms += WSTEP;
            if (ms >= me) break;
            if (ms + WSTEP < me) load_row(s0, ms + WSTEP);
            search_row(s1, ms);
            ms += WSTEP;
        }
    }
    // every CTA waits once, so this grid ends after the GEMM grid whatever its row range
    if (!waited) pdl_wait();
}

// ------------------------------------------------------------------ stream kernel
constexpr int MAXM_STREAM = 8;

struct StreamParams {
    int M, N, K;
    const float* A;
    const float* B;
    float* C;
    int32_t* I;
    int64_t sAm, sAk, sBk, sBn, sCm, sCn, sIm, sIn;
    uint32_t nvec;   // vectors per batch row (N / VEC)
    FastDiv div_nvec;
    uint32_t total;  // nbatch * nvec
    Batch bt;
    // binner > 0: the innermost batch axis (binner entries) varies fastest across threads, for
    // layouts where its strides are below the column stride (consecutive threads then touch
    // consecutive memory); 0: the columns vary fastest
    uint32_t binner;
    FastDiv div_binner;
#if TROP_DEBUG_BOUNDS
    Span sp[4];  // A, B, C, I
#endif
};

template <int SR, bool ARG, int VEC, int MAXM>
__global__ void __launch_bounds__(256) k_gemm_stream(StreamParams p)
{
    using O = Ops<SR>;
    pdl_wait();
    pdl_signal();
    for (uint32_t e = blockIdx.x * blockDim.x + threadIdx.x; e < p.total; e += gridDim.x * blockDim.x) {
        uint32_t b;
        int n;
        if (p.binner) {
            const uint32_t r = fdiv(e, p.div_binner);
            const uint32_t q = fdiv(r, p.div_nvec);
            n = (int)(r - q * p.nvec) * VEC;
            b = q * p.binner + (e - r * p.binner);
        } else {
            b = fdiv(e, p.div_nvec);
            n = (int)(e - b * p.nvec) * VEC;
        }
        int64_t oa, ob, oc, oi;
        batch_offsets(p.bt, b, oa, ob, oc, oi);
        float best[MAXM][VEC];
        int32_t idx[MAXM][VEC];
#pragma unroll
        for (int m = 0; m < MAXM; ++m)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                best[m][v] = O::zero();
                idx[m][v] = 0;
            }
        const float* Ab = p.A + oa;
        const float* Bb = p.B + ob + (int64_t)n * p.sBn;
        for (int k = 0; k < p.K; ++k) {
            float bv[VEC];
            if (VEC == 4) {
                float4 x = T_IN(Bb + (int64_t)k * p.sBk, 16, 1) ? __ldg(reinterpret_cast<const float4*>(Bb + (int64_t)k * p.sBk))
                                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                bv[0] = x.x;
                bv[VEC > 1 ? 1 : 0] = x.y;
                bv[VEC > 2 ? 2 : 0] = x.z;
                bv[VEC > 3 ? 3 : 0] = x.w;
            } else {
#pragma unroll
                for (int v = 0; v < VEC; ++v)
                    bv[v] = T_IN(Bb + (int64_t)k * p.sBk + (int64_t)v * p.sBn, 4, 1)
                                ? __ldg(Bb + (int64_t)k * p.sBk + (int64_t)v * p.sBn)
                                : 0.0f;
            }
#pragma unroll
            for (int m = 0; m < MAXM; ++m) {
                if (m < p.M) {
                    const float* ap = Ab + (int64_t)m * p.sAm + (int64_t)k * p.sAk;
                    const float a = T_IN(ap, 4, 0) ? __ldg(ap) : 0.0f;
#pragma unroll
                    for (int v = 0; v < VEC; ++v) {
                        const float t = O::mul(a, bv[v]);
                        if (O::better(t, best[m][v])) {
                            best[m][v] = t;
                            if (ARG) idx[m][v] = k;
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            if (m < p.M) {
                float* cp = p.C + oc + (int64_t)m * p.sCm + (int64_t)n * p.sCn;
                int32_t* ip = ARG ? p.I + oi + (int64_t)m * p.sIm + (int64_t)n * p.sIn : nullptr;
                if (VEC == 4) {
                    if (T_IN(cp, 16, 2))
                        *reinterpret_cast<float4*>(cp) =
                            make_float4(best[m][0], best[m][VEC > 1 ? 1 : 0], best[m][VEC > 2 ? 2 : 0],
                                        best[m][VEC > 3 ? 3 : 0]);
                    if (ARG && T_IN(ip, 16, 3))
                        *reinterpret_cast<int4*>(ip) = make_int4(idx[m][0], idx[m][VEC > 1 ? 1 : 0],
                                                                 idx[m][VEC > 2 ? 2 : 0], idx[m][VEC > 3 ? 3 : 0]);
                } else {
#pragma unroll
                    for (int v = 0; v < VEC; ++v) {
                        if (T_IN(cp + (int64_t)v * p.sCn, 4, 2)) cp[(int64_t)v * p.sCn] = best[m][v];
                        if (ARG && T_IN(ip + (int64_t)v * p.sIn, 4, 3)) ip[(int64_t)v * p.sIn] = idx[m][v];
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------------------ generic kernel
struct GenericParams {
    int64_t M, N, K, total;
    const float* A;
    const float* B;
    float* C;
    int32_t* I;
    int64_t sAm, sAk, sBk, sBn, sCm, sCn, sIm, sIn;
    int nb;
    int64_t bsize[MAXB], sA[MAXB], sB[MAXB], sC[MAXB], sI[MAXB];
#if TROP_DEBUG_BOUNDS
    Span sp[4];  // A, B, C, I
#endif
};

template <int SR, bool ARG>
__global__ void k_gemm_generic(GenericParams p)
{
    pdl_wait();
    pdl_signal();
    using O = Ops<SR>;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < p.total;
         e += (int64_t)gridDim.x * blockDim.x) {
        int64_t r = e;
        const int64_t n = r % p.N;
        r /= p.N;
        const int64_t m = r % p.M;
        r /= p.M;
        int64_t oa = 0, ob = 0, oc = 0, oi = 0;
        for (int d = p.nb - 1; d >= 0; --d) {
            int64_t c = r % p.bsize[d];
            r /= p.bsize[d];
            oa += c * p.sA[d];
            ob += c * p.sB[d];
            oc += c * p.sC[d];
            oi += c * p.sI[d];
        }
        const float* a = p.A + oa + m * p.sAm;
        const float* b = p.B + ob + n * p.sBn;
        float best = O::zero();
        int64_t idx = 0;
        for (int64_t k = 0; k < p.K; ++k) {
            const float t = O::mul(T_IN(a + k * p.sAk, 4, 0) ? __ldg(a + k * p.sAk) : 0.0f,
                                   T_IN(b + k * p.sBk, 4, 1) ? __ldg(b + k * p.sBk) : 0.0f);
            if (O::better(t, best)) {
                best = t;
                idx = k;
            }
        }
        if (T_IN(p.C + oc + m * p.sCm + n * p.sCn, 4, 2)) p.C[oc + m * p.sCm + n * p.sCn] = best;
        if (ARG && T_IN(p.I + oi + m * p.sIm + n * p.sIn, 4, 3)) p.I[oi + m * p.sIm + n * p.sIn] = (int32_t)idx;
    }
}

// ------------------------------------------------------------------ dispatch
int check_launch(const char* name)
{
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, name);
    count_launches(1);
    return TROP_OK;
}

Batch make_batch(const GemmDesc& g, int64_t& nbatch)
{
    Batch bt{};
    nbatch = 1;
    for (int d = 0; d < g.nb; ++d) {
        if (g.bsize[d] == 1) continue;
        int k = bt.nb++;
        bt.div[k] = make_fastdiv((uint32_t)g.bsize[d]);
        bt.sA[k] = g.sAb[d];
        bt.sB[k] = g.sBb[d];
        bt.sC[k] = g.sCb[d];
        bt.sI[k] = g.sIb[d];
        nbatch *= g.bsize[d];
    }
    return bt;
}

// Resident CTAs per SM of a kernel (looked up once per kernel).
int resident_ctas(const void* fn, int threads, size_t smem, std::atomic<int>& cache)
{
    int occ = cache.load(std::memory_order_relaxed);
    if (occ > 0) return occ;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, threads, smem);
    if (e != cudaSuccess || occ < 1) {
        cudaGetLastError();
        occ = 1;
    }
    cache.store(occ, std::memory_order_relaxed);
    return occ;
}

// The TMA-fed argmax kernel's layout conditions (the tensor maps may still refuse): one batch
// axis, whole k-tiles, 16-byte aligned operands with row and batch strides in 16-byte units.
bool tma_layout_ok(const GemmDesc& g, const Batch& bt, int64_t nbatch, bool need_argmax = true)
{
    if ((need_argmax && !g.I) || bt.nb > 1 || g.K % BK != 0) return false;
    if ((uintptr_t)g.A % 16 || (uintptr_t)g.B % 16 || g.sAm <= 0 || g.sAm % 4 || g.sBk <= 0 || g.sBk % 4) return false;
    if (nbatch > 1 && (bt.sA[0] <= 0 || bt.sA[0] % 4 || bt.sB[0] <= 0 || bt.sB[0] % 4)) return false;
    return true;
}

// Which argmax resolve pass follows the TMA-fed or tiled argmax kernel: "rows" (K <= 256, whole
// chunks, unit column strides, 32-bit row strides) or the panel pass of width 64 / 32 / 16.
const char* resolve_kind(const GemmDesc& g, bool vecA)
{
    const bool fast = vecA && g.K % CH == 0 && g.sCn == 1 && g.sIn == 1;
    const auto fits32 = [](int64_t v) { return v >= INT32_MIN && v <= INT32_MAX; };
    if (fast && g.K >= CH && g.K <= SHORT_K && fits32(g.sAm) && fits32(g.sCm) && fits32(g.sIm)) return "rows";
    if (!fast || g.K <= PanelShape<64>::GK) return "panel64";
    return g.K <= PanelShape<32>::GK ? "panel32" : "panel16";
}

// The fused GEMM + resolve launch (k_gemm_tma_fused) serves the layouts of the short-K row
// resolve once the TMA-fed kernel is chosen, when its item count fits 31 bits.
#ifndef TROP_TMA_FUSED
#define TROP_TMA_FUSED 1
#endif
// Counters of one launch: the item counter, then a tile count and a resolve count per batch.  A
// stream's two halves have this fixed size whatever the launch's batch count, so that two
// launches of different batch counts in turn never share a counter.
constexpr int64_t FUSED_MAX_BATCH = 4095;
constexpr size_t FUSED_HALF = 1 + 2 * (size_t)FUSED_MAX_BATCH;
bool fused_ok(const GemmDesc& g, bool vecA, uint64_t T, int64_t nbatch)
{
    if (!TROP_TMA_FUSED || resolve_kind(g, vecA)[0] != 'r' || nbatch > FUSED_MAX_BATCH) return false;
    const uint64_t items = T + (uint64_t)nbatch * (uint64_t)((g.N + FPW - 1) / FPW) * (uint64_t)((g.M + FRB - 1) / FRB);
    return items < (uint64_t(1) << 31);
}
// The byte range [lo, hi) a GEMM operand view addresses (batch axes, then rows and columns).
void view_range(const void* base, size_t eb, const GemmDesc& g, int64_t rows, int64_t cols, int64_t srow,
                int64_t scol, const int64_t* sb, uintptr_t& lo, uintptr_t& hi)
{
    int64_t a = 0, z = 0;
    bool empty = rows <= 0 || cols <= 0;
    auto add = [&](int64_t n, int64_t st) {
        if (n <= 0) empty = true;
        else (st < 0 ? a : z) += (n - 1) * st;
    };
    for (int d = 0; d < g.nb; ++d) add(g.bsize[d], sb[d]);
    add(rows, srow);
    add(cols, scol);
    const uintptr_t b = (uintptr_t)base;
    lo = empty ? b : b + a * (int64_t)eb;
    hi = empty ? b : b + (z + 1) * (int64_t)eb;
}
// the two outputs (values, argmax) of g, into a launch record
void output_ranges(const GemmDesc& g, LaunchRecord& r)
{
    view_range(g.C, sizeof(float), g, g.M, g.N, g.sCm, g.sCn, g.sCb, r.lo[0], r.hi[0]);
    view_range(g.I, sizeof(int32_t), g, g.M, g.N, g.sIm, g.sIn, g.sIb, r.lo[1], r.hi[1]);
}
// whether g reads (A or B) any byte the launch of r writes
bool reads_overlap(const GemmDesc& g, const LaunchRecord& r)
{
    uintptr_t lo[2], hi[2];
    view_range(g.A, sizeof(float), g, g.M, g.K, g.sAm, g.sAk, g.sAb, lo[0], hi[0]);
    view_range(g.B, sizeof(float), g, g.K, g.N, g.sBk, g.sBn, g.sBb, lo[1], hi[1]);
    for (int i = 0; i < 2; ++i)
        for (int j = 0; j < 2; ++j)
            if (lo[i] < r.hi[j] && r.lo[j] < hi[i]) return true;
    return false;
}

// every row of A starts 32-byte aligned: a resolve lane loads its chunk of A in one piece
bool a_rows_32b(const TiledParams& p)
{
    bool v8 = ((uintptr_t)p.A % 32) == 0 && p.sAm % 8 == 0;
    for (int d = 0; d < p.bt.nb; ++d) v8 = v8 && p.bt.sA[d] % 8 == 0;
    return v8;
}

void resolve_split(TiledParams& p, uint64_t grid, uint32_t npan)
{
    p.r_per = p.r_units / grid;
    p.r_rem = (uint32_t)(p.r_units % grid);
    p.r32 = p.r_units < (uint64_t(1) << 31);
    p.div_M = make_fastdiv((uint32_t)p.M);
    p.div_npan = make_fastdiv(npan);
}

template <int SR, int PW>
int launch_resolve_pw(TiledParams& p, int64_t M, int64_t nbatch, cudaStream_t s, const DeviceInfo* dev)
{
    static std::atomic<int> occ{0};
    const uint64_t npan = (uint64_t)((p.N + PW - 1) / PW);
    p.r_units = (uint64_t)nbatch * npan * (uint64_t)M;
    const uint64_t slots =
        (uint64_t)dev->sm_count * resident_ctas((const void*)k_argmax_resolve<SR, PW>, RTHREADS, SMEM_RESOLVE, occ);
    const uint64_t per_cta = (uint64_t)RWARPS * PanelShape<PW>::ROWS;
    const uint64_t want = (p.r_units + per_cta - 1) / per_cta;
    // programmatic dependent launch: its CTAs stage B while the GEMM drains
    const uint64_t grid = std::max<uint64_t>(1, std::min(slots, want));
    resolve_split(p, grid, (uint32_t)npan);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(RTHREADS);
    cfg.dynamicSmemBytes = SMEM_RESOLVE;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_argmax_resolve<SR, PW>, p);
    if (e != cudaSuccess) return cuda_error(e, "k_argmax_resolve");
    return check_launch("k_argmax_resolve");
}

// Panel width of the resolve pass: the widest whose staged group covers K (fewest passes over
// the rows), 64 columns for layouts outside the common one.
template <int SR>
int launch_resolve_short(TiledParams& p, int64_t M, int64_t nbatch, cudaStream_t s, const DeviceInfo* dev)
{
    static std::atomic<int> occ{0};
    const uint64_t npan = (uint64_t)((p.N + BN - 1) / BN);
    p.r_units = (uint64_t)nbatch * npan * (uint64_t)M;
    const uint64_t slots =
        (uint64_t)dev->sm_count * resident_ctas((const void*)k_argmax_resolve_rows<SR, false>, RTHREADS, SMEM_RESOLVE, occ);
    const uint64_t per_cta = (uint64_t)RWARPS;
    const uint64_t want = (p.r_units + per_cta - 1) / per_cta;
    const uint64_t grid = std::max<uint64_t>(1, std::min(slots, want));
    resolve_split(p, grid, (uint32_t)npan);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(RTHREADS);
    cfg.dynamicSmemBytes = sizeof(float) * (size_t)p.K * BN;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // A's chunks by one 32-byte load each when every row start is 32-byte aligned
    cudaError_t e = a_rows_32b(p) ? cudaLaunchKernelEx(&cfg, k_argmax_resolve_rows<SR, true>, p)
                       : cudaLaunchKernelEx(&cfg, k_argmax_resolve_rows<SR, false>, p);
    if (e != cudaSuccess) return cuda_error(e, "k_argmax_resolve_rows");
    return check_launch("k_argmax_resolve_rows");
}

template <int SR>
int launch_resolve(TiledParams& p, const GemmDesc& g, int64_t nbatch, cudaStream_t s, const DeviceInfo* dev)
{
    const char* kind = resolve_kind(g, p.vecA != 0);
    if (kind[0] == 'r') return launch_resolve_short<SR>(p, g.M, nbatch, s, dev);
    if (kind[5] == '6') return launch_resolve_pw<SR, 64>(p, g.M, nbatch, s, dev);
    if (kind[5] == '3') return launch_resolve_pw<SR, 32>(p, g.M, nbatch, s, dev);
    return launch_resolve_pw<SR, 16>(p, g.M, nbatch, s, dev);
}

// cuTensorMapEncodeTiled from the driver, looked up once (no link against libcuda)
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled()
{
    static std::atomic<int> state{0};  // 0: not looked up, 1: found, 2: unavailable
    static std::atomic<EncodeTiledFn> fn{nullptr};
    if (state.load(std::memory_order_acquire) == 0) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
        if (e == cudaSuccess && q == cudaDriverEntryPointSuccess && ptr) {
            fn.store(reinterpret_cast<EncodeTiledFn>(ptr), std::memory_order_relaxed);
            state.store(1, std::memory_order_release);
        } else {
            cudaGetLastError();
            state.store(2, std::memory_order_release);
        }
    }
    return state.load(std::memory_order_acquire) == 1 ? fn.load(std::memory_order_relaxed) : nullptr;
}

// A 3-D tensor map of a row-major f32 operand [batch][rows][cols] (cols contiguous) with a
// [1][box_rows][box_cols] box; false when TMA cannot describe it (the caller keeps the
// cp.async kernel).  Strides in elements.
bool make_map(CUtensorMap* map, const float* base, uint64_t cols, uint64_t rows, uint64_t batch, int64_t row_stride,
              int64_t batch_stride, uint32_t box_cols, uint32_t box_rows)
{
    const EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    if (((uintptr_t)base % 16) != 0 || row_stride <= 0 || row_stride % 4 != 0) return false;
    if (batch > 1 && (batch_stride <= 0 || batch_stride % 4 != 0)) return false;
    const cuuint64_t dims[3] = {cols, rows, batch};
    const cuuint64_t strides[2] = {(cuuint64_t)row_stride * sizeof(float),
                                   (cuuint64_t)(batch > 1 ? batch_stride : row_stride * (int64_t)rows) * sizeof(float)};
    const cuuint32_t box[3] = {box_cols, box_rows, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// the GEMM without argmax by TMA (k_gemm_tma_plain): the TMA layout, and a driver that encodes maps
#ifndef TROP_TMA_PLAIN
#define TROP_TMA_PLAIN 1
#endif
bool plain_tma_ok(const GemmDesc& g, const Batch& bt, int64_t nbatch)
{
    return TROP_TMA_PLAIN && tma_layout_ok(g, bt, nbatch, false) && encode_tiled() != nullptr;
}

// Stream-K only when the last wave would run at most this full (percent); each stream-K
// CTA gets at least SK_MIN_UNITS k-tiles (unless a tile has fewer) and a tile is cut into at
// most SK_MAX_SEGS segments.
#ifndef TROP_SK_MAX_FILL_PCT
#define TROP_SK_MAX_FILL_PCT 85
#endif
constexpr uint64_t SK_MAX_FILL_PCT = TROP_SK_MAX_FILL_PCT, SK_MIN_UNITS = 4, SK_MAX_SEGS = 32;

// The stream-K decision for T tiles of nkt k-tiles on G resident CTAs: whether the last R
// tiles are cut along k, and then L (k-tiles per stream-K CTA) and the number of those CTAs.
bool sk_split(uint64_t T, uint64_t G, uint64_t nkt, bool arg, uint64_t& R, uint64_t& L, uint64_t& n_sk)
{
    R = T % G;
    // With argmax the merge of a split tile sits on the tail's critical path; measured on
    // batched 256^3 problems it paid off only when the whole problem is under half a wave.
    const bool sk_ok = !arg || T * 2 <= G;
    if (!(sk_ok && R > 0 && R * 100 <= G * SK_MAX_FILL_PCT && R * nkt < (uint64_t(1) << 31))) return false;
    const uint64_t U = R * nkt;
    // at least SK_MIN_UNITS k-tiles and at most SK_MAX_SEGS segments per tile; L <= nkt as R < G
    L = std::max({(U + G - 1) / G, std::min<uint64_t>(SK_MIN_UNITS, nkt), (nkt + SK_MAX_SEGS - 1) / SK_MAX_SEGS});
    n_sk = (U + L - 1) / L;
    return n_sk > R;
}

template <int SR, bool ARG>
int run_tiled(const GemmDesc& g, cudaStream_t s, const DeviceInfo* dev)
{
    static std::atomic<int> occ_gemm{0};
    TiledParams p{};
#if TROP_DEBUG_BOUNDS
    gemm_spans(g, sizeof(float), p.sp);
#endif
    p.M = (int)g.M;
    p.N = (int)g.N;
    p.K = (int)g.K;
    p.A = static_cast<const float*>(g.A);
    p.B = static_cast<const float*>(g.B);
    p.C = static_cast<float*>(g.C);
    p.I = g.I;
    p.sAm = g.sAm;
    p.sBk = g.sBk;
    p.sCm = g.sCm;
    p.sCn = g.sCn;
    p.sIm = g.sIm;
    p.sIn = g.sIn;
    p.sAm32 = (int)g.sAm;
    p.sCm32 = (int)g.sCm;
    p.sIm32 = (int)g.sIm;
    int64_t nbatch = 1;
    p.bt = make_batch(g, nbatch);
    p.nbatch = (uint32_t)nbatch;
    bool va = ((uintptr_t)g.A % 16) == 0 && g.sAm % 4 == 0;
    bool vb = ((uintptr_t)g.B % 16) == 0 && g.sBk % 4 == 0;
    bool vc = ((uintptr_t)g.C % 16) == 0 && g.sCm % 4 == 0 && g.sCn == 1;
    bool vi = ARG && ((uintptr_t)g.I % 16) == 0 && g.sIm % 4 == 0 && g.sIn == 1;
    for (int d = 0; d < p.bt.nb; ++d) {
        va = va && p.bt.sA[d] % 4 == 0;
        vb = vb && p.bt.sB[d] % 4 == 0;
        vc = vc && p.bt.sC[d] % 4 == 0;
        vi = vi && p.bt.sI[d] % 4 == 0;
    }
    p.vecA = va;
    p.vecB = vb;
    p.vecC = vc;
    p.vecI = vi;
    p.tiles_m = (uint32_t)((g.M + BM - 1) / BM);
    p.tiles_n = (uint32_t)((g.N + BN - 1) / BN);
    p.nkt = (uint32_t)((g.K + BK - 1) / BK);
    p.div_tm = make_fastdiv(p.tiles_m);
    p.div_tn = make_fastdiv(p.tiles_n);
    p.div_nkt = make_fastdiv(p.nkt);
    const uint64_t T = (uint64_t)nbatch * p.tiles_m * p.tiles_n;  // < 2^31 (route check)

    // ---- schedule: whole tiles for the full waves, stream-K for a thin last wave
    constexpr int TN = tile_tn<ARG>(), THREADS = tile_threads<TN>();
    const uint64_t G = (uint64_t)dev->sm_count *
                       resident_ctas((const void*)k_gemm_tiled<SR, ARG, TN>, THREADS, 0, occ_gemm);
    uint64_t R = 0, L = 0, n_sk = 0;
    uint64_t G_sk = 0;
    void* ws = nullptr;
    // without argmax, whole tiles by TMA (k_gemm_tma_plain) where the layout allows, no k split
    const bool plain_tma = !ARG && plain_tma_ok(g, p.bt, nbatch);
    if (!plain_tma && sk_split(T, G, p.nkt, ARG, R, L, n_sk)) {
        const uint64_t U = R * p.nkt;
        {
            const size_t seg_elems = (size_t)n_sk * 2 * TILE_ELEMS;
            uint32_t* cnt = nullptr;
            if (stream_tickets(s, (size_t)R, &cnt) == TROP_OK &&
                pool_alloc(seg_elems * (sizeof(float) + (ARG ? sizeof(uint16_t) : 0)), s, &ws) == TROP_OK) {
                G_sk = n_sk;
                p.L = (uint32_t)L;
                p.U = (uint32_t)U;
                p.div_L = make_fastdiv(p.L);
                p.seg_v = static_cast<float*>(ws);
                p.seg_c = ARG ? reinterpret_cast<uint16_t*>(p.seg_v + seg_elems) : nullptr;
                p.sk_cnt = cnt;
#if TROP_DEBUG_BOUNDS
                p.sp[4] = span_bytes(p.seg_v, seg_elems * sizeof(float));
                p.sp[5] = span_bytes(p.seg_c, ARG ? seg_elems * sizeof(uint16_t) : 0);
                p.sp[6] = span_bytes(cnt, (size_t)R * sizeof(uint32_t));
#endif
            } else {
                clear_error();  // no workspace: whole tiles only
                ws = nullptr;
            }
        }
    }
    p.T_dp = (uint32_t)(G_sk ? T - R : T);

    int rc = TROP_OK;
    bool launched = false, fused = false;
    // Early start (k_gemm_tma_fused, k_gemm_tma_plain): the last such GEMM on this stream and
    // whether it is the library's launch just before this one.  Never while the stream is being
    // captured (by this library or by the caller): a captured launch replays after arbitrary work.
    bool capturing = capture_arena() != nullptr;
    if (!capturing) {
        cudaStreamCaptureStatus cst = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cst) != cudaSuccess) {
            cudaGetLastError();
            cst = cudaStreamCaptureStatusActive;
        }
        capturing = cst != cudaStreamCaptureStatusNone;
    }
    auto record = [&](int parity) {
        if (p.late) count_early_start();
        LaunchRecord cur{};
        cur.valid = !capturing;
        cur.seq = launch_seq();
        cur.parity = parity;
        output_ranges(g, cur);
        set_stream_record(s, cur);
    };
    if constexpr (!ARG) {
        TmaMaps maps;
        const int64_t sAb = p.bt.nb ? p.bt.sA[0] : 0, sBb = p.bt.nb ? p.bt.sB[0] : 0;
        if (plain_tma && make_map(&maps.a, p.A, (uint64_t)g.K, (uint64_t)g.M, (uint64_t)nbatch, g.sAm, sAb, BK, BM) &&
            make_map(&maps.b, p.B, (uint64_t)g.N, (uint64_t)g.K, (uint64_t)nbatch, g.sBk, sBb, BN, BK)) {
            TROP_TRY(device_error_word(&p.err));
            p.wait_mode = wait_test_mode();
            const LaunchRecord prev = capturing ? LaunchRecord{} : stream_record(s);
            const bool follows = prev.valid && prev.seq == launch_seq();
            p.late = follows && !reads_overlap(g, prev) ? 1 : 0;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)T);
            cfg.blockDim = dim3(tile_threads<4>());
            cfg.stream = s;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            const cudaError_t e = cudaLaunchKernelEx(&cfg, k_gemm_tma_plain<SR>, maps, p);
            rc = e != cudaSuccess ? cuda_error(e, "k_gemm_tma_plain") : check_launch("k_gemm_tma_plain");
            // (no counters of its own: the next one-launch argmax GEMM alternates from the last one's half)
            if (rc == TROP_OK) record(follows ? prev.parity : 0);
            launched = true;
        } else if (plain_tma) {
            clear_error();  // (no tensor map: the cp.async kernel, whole tiles)
        }
    }
    if constexpr (ARG) {
        // whole tiles, one batch axis, whole k-tiles: operands by TMA
        if (!G_sk && tma_layout_ok(g, p.bt, nbatch)) {
            TROP_TRY(device_error_word(&p.err));
            p.wait_mode = wait_test_mode();
            TmaMaps maps;
            const int64_t sAb = p.bt.nb ? p.bt.sA[0] : 0, sBb = p.bt.nb ? p.bt.sB[0] : 0;
            if (make_map(&maps.a, p.A, (uint64_t)g.K, (uint64_t)g.M, (uint64_t)nbatch, g.sAm, sAb, BK, BM) &&
                make_map(&maps.b, p.B, (uint64_t)g.N, (uint64_t)g.K, (uint64_t)nbatch, g.sBk, sBb, BN, BK)) {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3((unsigned)T);
                cfg.blockDim = dim3(tile_threads<4>());
                cfg.stream = s;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
                attr[0].val.programmaticStreamSerializationAllowed = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                const size_t half = FUSED_HALF;  // tickets of one launch (one half of the stream's two)
                if (fused_ok(g, p.vecA != 0, T, nbatch) &&
                    make_map(&maps.bp, p.B, (uint64_t)g.N, (uint64_t)g.K, (uint64_t)nbatch, g.sBk, sBb, FPW,
                             (uint32_t)g.K) &&
                    stream_tickets(s, 2 * half, &p.sched) == TROP_OK) {
                    // two halves of tickets used in turn by the fused GEMMs on a stream; start early
                    // when the GEMM just before is one of them and wrote nothing this one reads.
                    // Never while the stream is being captured (by this library or by the caller):
                    // a captured launch replays after arbitrary work.
                    const LaunchRecord prev = capturing ? LaunchRecord{} : stream_record(s);
                    const bool follows = prev.valid && prev.seq == launch_seq();
                    const int parity = follows ? prev.parity ^ 1 : 0;
                    p.late = follows && !reads_overlap(g, prev) ? 1 : 0;
                    p.sched += parity * half;
                    // GEMM and resolve in one launch (k_gemm_tma_fused)
                    const uint32_t npan = (uint32_t)((g.N + FPW - 1) / FPW);
                    p.rblocks = (uint32_t)((g.M + FRB - 1) / FRB);
                    p.items_per_batch = npan * p.rblocks;
                    p.tiles_per_batch = p.tiles_m * p.tiles_n;
                    p.n_tiles = (uint32_t)T;
                    p.n_items = (uint32_t)(T + (uint64_t)nbatch * p.items_per_batch);
                    p.div_ipb = make_fastdiv(p.items_per_batch);
                    p.div_rblocks = make_fastdiv(p.rblocks);
#if TROP_DEBUG_BOUNDS
                    p.sp[7] = span_bytes(p.sched, half * sizeof(uint32_t));
#endif
                    cfg.gridDim = dim3(p.n_items);
                    const cudaError_t e = a_rows_32b(p) ? cudaLaunchKernelEx(&cfg, k_gemm_tma_fused<SR, true>, maps, p)
                                                        : cudaLaunchKernelEx(&cfg, k_gemm_tma_fused<SR, false>, maps, p);
                    rc = e != cudaSuccess ? cuda_error(e, "k_gemm_tma_fused") : check_launch("k_gemm_tma_fused");
                    fused = true;
                    if (rc == TROP_OK) record(parity);
                } else {
                    clear_error();  // (no tickets: the two-pass form below)
                    const cudaError_t e = cudaLaunchKernelEx(&cfg, k_gemm_tma<SR>, maps, p);
                    rc = e != cudaSuccess ? cuda_error(e, "k_gemm_tma") : check_launch("k_gemm_tma");
                }
                launched = true;
            }
        }
    }
    if (!launched) {
        (void)launch_pdl(k_gemm_tiled<SR, ARG, TN>, dim3((unsigned)(p.T_dp + G_sk)), dim3(THREADS), 0, s, p);
        rc = check_launch("k_gemm_tiled");
    }
    if (rc == TROP_OK && ARG && !fused) rc = launch_resolve<SR>(p, g, nbatch, s, dev);
    if (ws) pool_retire(ws, s);
    return rc;
}

// 16-byte vectors along n for the stream kernel: every row of B, C (and I) aligned
bool stream_vec(const GemmDesc& g, bool arg)
{
    bool vec = g.N % 4 == 0 && g.sBn == 1 && g.sCn == 1 && (!arg || g.sIn == 1) && ((uintptr_t)g.B % 16) == 0 &&
               ((uintptr_t)g.C % 16) == 0 && (!arg || ((uintptr_t)g.I % 16) == 0) && g.sBk % 4 == 0 &&
               g.sCm % 4 == 0 && (!arg || g.sIm % 4 == 0);
    for (int d = 0; d < g.nb; ++d)
        if (g.bsize[d] != 1) vec = vec && g.sBb[d] % 4 == 0 && g.sCb[d] % 4 == 0 && (!arg || g.sIb[d] % 4 == 0);
    return vec;
}

template <int SR, bool ARG>
int run_stream(const GemmDesc& g, cudaStream_t s, const DeviceInfo* dev)
{
    StreamParams p{};
#if TROP_DEBUG_BOUNDS
    gemm_spans(g, sizeof(float), p.sp);
#endif
    p.M = (int)g.M;
    p.N = (int)g.N;
    p.K = (int)g.K;
    p.A = static_cast<const float*>(g.A);
    p.B = static_cast<const float*>(g.B);
    p.C = static_cast<float*>(g.C);
    p.I = g.I;
    p.sAm = g.sAm;
    p.sAk = g.sAk;
    p.sBk = g.sBk;
    p.sBn = g.sBn;
    p.sCm = g.sCm;
    p.sCn = g.sCn;
    p.sIm = g.sIm;
    p.sIn = g.sIn;
    int64_t nbatch = 1;
    p.bt = make_batch(g, nbatch);
    const bool vec = stream_vec(g, ARG);
    const int VEC = vec ? 4 : 1;
    p.nvec = (uint32_t)(g.N / VEC);
    p.div_nvec = make_fastdiv(p.nvec);
    p.total = (uint32_t)(nbatch * p.nvec);
    if (p.bt.nb > 0) {
        // the batch index's fastest axis is the last one of the decomposition
        const int d = p.bt.nb - 1;
        const auto mag = [](int64_t v) { return v < 0 ? -v : v; };
        const int64_t col = std::min(mag(g.sBn), mag(g.sCn)) * VEC;
        int64_t bs = std::max(mag(p.bt.sB[d]), mag(p.bt.sC[d]));
        if (ARG) bs = std::max(bs, mag(p.bt.sI[d]));
        if (bs < col) {
            p.binner = p.bt.div[d].d;
            p.div_binner = p.bt.div[d];
        }
    }
    int64_t blocks = ((int64_t)p.total + 255) / 256;
    int64_t cap = (int64_t)dev->sm_count * 16;
    int grid = (int)(blocks < cap ? (blocks < 1 ? 1 : blocks) : cap);
    // register arrays sized to the rows actually present keep occupancy high
    if (g.M <= 2) {
        if (vec) (void)launch_pdl(k_gemm_stream<SR, ARG, 4, 2>, grid, 256, 0, s, p);
        else (void)launch_pdl(k_gemm_stream<SR, ARG, 1, 2>, grid, 256, 0, s, p);
    } else if (g.M <= 4) {
        if (vec) (void)launch_pdl(k_gemm_stream<SR, ARG, 4, 4>, grid, 256, 0, s, p);
        else (void)launch_pdl(k_gemm_stream<SR, ARG, 1, 4>, grid, 256, 0, s, p);
    } else {
        if (vec) (void)launch_pdl(k_gemm_stream<SR, ARG, 4, MAXM_STREAM>, grid, 256, 0, s, p);
        else (void)launch_pdl(k_gemm_stream<SR, ARG, 1, MAXM_STREAM>, grid, 256, 0, s, p);
    }
    return check_launch("k_gemm_stream");
}

template <int SR, bool ARG>
int run_generic(const GemmDesc& g, cudaStream_t s, const DeviceInfo* dev)
{
    GenericParams p{};
#if TROP_DEBUG_BOUNDS
    gemm_spans(g, sizeof(float), p.sp);
#endif
    p.M = g.M;
    p.N = g.N;
    p.K = g.K;
    p.A = static_cast<const float*>(g.A);
    p.B = static_cast<const float*>(g.B);
    p.C = static_cast<float*>(g.C);
    p.I = g.I;
    p.sAm = g.sAm;
    p.sAk = g.sAk;
    p.sBk = g.sBk;
    p.sBn = g.sBn;
    p.sCm = g.sCm;
    p.sCn = g.sCn;
    p.sIm = g.sIm;
    p.sIn = g.sIn;
    p.nb = g.nb;
    int64_t nbatch = 1;
    for (int d = 0; d < g.nb; ++d) {
        p.bsize[d] = g.bsize[d];
        p.sA[d] = g.sAb[d];
        p.sB[d] = g.sBb[d];
        p.sC[d] = g.sCb[d];
        p.sI[d] = g.sIb[d];
        nbatch *= g.bsize[d];
    }
    p.total = nbatch * g.M * g.N;
    int64_t blocks = (p.total + 255) / 256;
    int64_t cap = (int64_t)dev->sm_count * 16;
    int grid = (int)(blocks < cap ? (blocks < 1 ? 1 : blocks) : cap);
    (void)launch_pdl(k_gemm_generic<SR, ARG>, grid, 256, 0, s, p);
    return check_launch("k_gemm_generic");
}

GemmDesc swapped(const GemmDesc& g)
{
    // C^T = B^T (x) A^T; (x) commutes exactly (IEEE add and multiply do)
    GemmDesc t = g;
    t.M = g.N;
    t.N = g.M;
    t.A = g.B;
    t.B = g.A;
    t.sAm = g.sBn;
    t.sAk = g.sBk;
    t.sBk = g.sAk;
    t.sBn = g.sAm;
    t.sCm = g.sCn;
    t.sCn = g.sCm;
    t.sIm = g.sIn;
    t.sIn = g.sIm;
    for (int d = 0; d < g.nb; ++d) {
        t.sAb[d] = g.sBb[d];
        t.sBb[d] = g.sAb[d];
    }
    return t;
}

enum Route { R_TILED, R_STREAM, R_GENERIC };

Route choose(const GemmDesc& g, bool& swap)
{
    swap = false;
    int64_t nbatch = 1;
    for (int d = 0; d < g.nb; ++d) nbatch *= g.bsize[d];
    const bool fits32 = g.M < (1 << 30) && g.N < (1 << 30) && g.K < (1 << 30) && nbatch < (int64_t(1) << 31);
    // the argmax epilogue keeps chunk numbers in 16 bits
    const bool big = g.M >= 16 && g.N >= 16 && g.K >= 8 && (!g.I || g.K <= (int64_t)CH * 65535);
    // tiles in a 1-D grid, with room for the stream-K CTAs
    const int64_t tiles = nbatch * ((g.M + BM - 1) / BM) * ((g.N + BN - 1) / BN);
    const bool grid_ok = tiles < (int64_t(1) << 30);
    const bool grid_ok_t = grid_ok;
    if (fits32 && big) {
        if (g.sAk == 1 && g.sBn == 1 && grid_ok) return R_TILED;
        if (g.sBk == 1 && g.sAm == 1 && grid_ok_t) {
            swap = true;
            return R_TILED;
        }
    }
    if (fits32 && g.K <= 64) {
        if (g.M <= MAXM_STREAM && nbatch * g.N < (int64_t(1) << 31) && g.M <= g.N) return R_STREAM;
        if (g.N <= MAXM_STREAM && nbatch * g.M < (int64_t(1) << 31)) {
            swap = true;
            return R_STREAM;
        }
    }
    return R_GENERIC;
}

// The tiled kernel writes 4-column runs of an output row; when the output's column stride is
// not 1 (a transposed or permuted output) those become scattered 4-byte stores, and the argmax
// pass reads them back the same way.  Such a product goes to a contiguous pool buffer first and
// is then moved, value and argmax through one index mapping, by the tiled transpose.
template <int SR, bool ARG>
int run_tiled_staged(const GemmDesc& g, cudaStream_t s, const DeviceInfo* dev)
{
    int64_t nbatch = 1;
    for (int d = 0; d < g.nb; ++d) nbatch *= g.bsize[d];
    const size_t elems = (size_t)nbatch * (size_t)g.M * (size_t)g.N;
    void* ws = nullptr;
    if (pool_alloc(elems * (sizeof(float) + (ARG ? sizeof(int32_t) : 0)), s, &ws) != TROP_OK) {
        clear_error();
        return run_tiled<SR, ARG>(g, s, dev);  // no workspace: write through the strides
    }
    GemmDesc t = g;
    t.C = ws;
    t.I = ARG ? reinterpret_cast<int32_t*>(static_cast<float*>(ws) + elems) : nullptr;
    t.sCm = t.sIm = g.N;
    t.sCn = t.sIn = 1;
    GatherDesc gd{};
    gd.rank = g.nb + 2;
    int64_t st = g.M * g.N;
    for (int d = g.nb - 1; d >= 0; --d) {
        t.sCb[d] = t.sIb[d] = st;
        gd.size[d] = g.bsize[d];
        gd.s_in[d] = gd.s_in2[d] = st;
        gd.s_out[d] = g.sCb[d];
        gd.s_out2[d] = g.sIb[d];
        st *= g.bsize[d];
    }
    const int m = g.nb, n = g.nb + 1;
    gd.size[m] = g.M;
    gd.size[n] = g.N;
    gd.s_in[m] = gd.s_in2[m] = g.N;
    gd.s_in[n] = gd.s_in2[n] = 1;
    gd.s_out[m] = g.sCm;
    gd.s_out[n] = g.sCn;
    gd.s_out2[m] = g.sIm;
    gd.s_out2[n] = g.sIn;
    {
        // axes in the output's order (slowest first), as the gather planner expects
        GatherDesc o = gd;
        int idx[MAXR];
        for (int i = 0; i < gd.rank; ++i) idx[i] = i;
        std::stable_sort(idx, idx + gd.rank, [&](int x, int y) { return gd.s_out[x] > gd.s_out[y]; });
        for (int i = 0; i < gd.rank; ++i) {
            o.size[i] = gd.size[idx[i]];
            o.s_in[i] = gd.s_in[idx[i]];
            o.s_out[i] = gd.s_out[idx[i]];
            o.s_in2[i] = gd.s_in2[idx[i]];
            o.s_out2[i] = gd.s_out2[idx[i]];
        }
        gd = o;
    }
    int rc = run_tiled<SR, ARG>(t, s, dev);
    if (rc == TROP_OK) rc = launch_gather(t.C, g.C, (int)sizeof(float), t.I, g.I, gd, s);
    pool_retire(ws, s);
    return rc;
}

template <int SR, bool ARG>
int run(const GemmDesc& g0, cudaStream_t s, const DeviceInfo* dev, const char** name)
{
    bool swap = false;
    Route r = choose(g0, swap);
    const GemmDesc g = swap ? swapped(g0) : g0;
    switch (r) {
    case R_TILED:
        if (name) *name = "k_gemm_tiled";
        if (g.sCn != 1 || (ARG && g.sIn != 1)) return run_tiled_staged<SR, ARG>(g, s, dev);
        return run_tiled<SR, ARG>(g, s, dev);
    case R_STREAM:
        if (name) *name = "k_gemm_stream";
        return run_stream<SR, ARG>(g, s, dev);
    default:
        if (name) *name = "k_gemm_generic";
        return run_generic<SR, ARG>(g, s, dev);
    }
}

}  // namespace

void describe_gemm(const GemmDesc& g1, char* buf, size_t n)
{
    // a description is about layouts: take every pointer as 256-byte aligned
    GemmDesc g0 = g1;
    const uintptr_t aligned = 256;
    g0.A = reinterpret_cast<const void*>(aligned);
    g0.B = reinterpret_cast<const void*>(aligned);
    g0.C = reinterpret_cast<void*>(aligned);
    if (g1.I) g0.I = reinterpret_cast<int32_t*>(aligned);
    if (g1.dtype == TROP_F64) {
        snprintf(buf, n, " route=tiled_f64");
        return;
    }
    if (g1.dtype == TROP_I32 || g1.dtype == TROP_I64) {
        snprintf(buf, n, " route=tiled_int");
        return;
    }
    bool swap = false;
    const Route r = choose(g0, swap);
    const GemmDesc g = swap ? swapped(g0) : g0;
    const bool arg = g.I != nullptr;
    if (r == R_TILED) {
        const bool staged = g.sCn != 1 || (arg && g.sIn != 1);
        char extra[128] = "";
        // the last wave's stream-K split depends on the SM count: the current device's when one
        // is visible (a host query), else a GB300's 152
        int sms = 152, dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            sms = 152;
        }
        uint64_t T = 1;
        for (int d = 0; d < g.nb; ++d) T *= (uint64_t)g.bsize[d];
        T *= (uint64_t)((g.M + BM - 1) / BM) * (uint64_t)((g.N + BN - 1) / BN);
        const uint64_t nkt = (uint64_t)((g.K + BK - 1) / BK);
        uint64_t R = 0, L = 0, n_sk = 0;
        bool split = sk_split(T, (uint64_t)sms * (arg ? TROP_ARG_MINB : TROP_PLAIN_MINB), nkt, arg, R, L, n_sk);
        if (!arg) {
            // whole tiles by TMA where the layout allows (no k split on that kernel)
            int64_t nbatch = 1;
            const Batch bt = make_batch(g, nbatch);
            const bool tma = TROP_TMA_PLAIN && tma_layout_ok(g, bt, nbatch, false);
            if (tma) split = false;
            snprintf(extra, sizeof(extra), " kernel=%s", tma ? "tma" : "tiled");
        }
        if (arg) {
            // the staged product is contiguous: describe the kernels on that layout
            GemmDesc gs = g;
            if (staged) {
                gs.sCn = gs.sIn = 1;
                gs.sCm = gs.sIm = gs.N;
            }
            int64_t nbatch = 1;
            const Batch bt = make_batch(gs, nbatch);
            bool va = ((uintptr_t)gs.A % 16) == 0 && gs.sAm % 4 == 0;
            for (int d = 0; d < bt.nb; ++d) va = va && bt.sA[d] % 4 == 0;
            const bool tma = !split && tma_layout_ok(gs, bt, nbatch);
            snprintf(extra, sizeof(extra), " kernel=%s resolve=%s", tma ? "tma" : "tiled",
                     tma && fused_ok(gs, va, T, nbatch) ? "fused" : resolve_kind(gs, va));
        }
        snprintf(buf, n, " route=tiled%s%s%s%s", swap ? " swap" : "", staged ? " staged" : "",
                 split ? " split_tail" : "", extra);
    }
    else if (r == R_STREAM)
        snprintf(buf, n, " route=stream%s vec=%d", swap ? " swap" : "", stream_vec(g, arg) ? 4 : 1);
    else
        snprintf(buf, n, " route=generic");
}

int launch_gemm(const GemmDesc& g, cudaStream_t s, const char** kernel_name)
{
    const DeviceInfo* dev = nullptr;
    TROP_TRY(ensure_device(&dev));
    if (g.M == 0 || g.N == 0) return TROP_OK;
    for (int d = 0; d < g.nb; ++d)
        if (g.bsize[d] == 0) return TROP_OK;
    if (g.dtype == TROP_F64) {
        if (kernel_name) *kernel_name = "k_gemm_tiled_f64";
        return launch_gemm_f64(g, s);
    }
    if (g.dtype == TROP_I32 || g.dtype == TROP_I64) {
        if (kernel_name) *kernel_name = "k_gemm_int";
        return launch_gemm_int(g, s);
    }
    if (g.dtype != TROP_F32) return set_error(TROP_ERR_DTYPE, "tropical GEMM: unsupported dtype %d", g.dtype);
    const bool arg = g.I != nullptr;
    switch (g.semiring) {
    case TROP_MAXPLUS: return arg ? run<TROP_MAXPLUS, true>(g, s, dev, kernel_name) : run<TROP_MAXPLUS, false>(g, s, dev, kernel_name);
    case TROP_MINPLUS: return arg ? run<TROP_MINPLUS, true>(g, s, dev, kernel_name) : run<TROP_MINPLUS, false>(g, s, dev, kernel_name);
    case TROP_MAXTIMES: return arg ? run<TROP_MAXTIMES, true>(g, s, dev, kernel_name) : run<TROP_MAXTIMES, false>(g, s, dev, kernel_name);
    default: return set_error(TROP_ERR_INVALID_ARG, "unknown semiring %d", g.semiring);
    }
}

int register_gemm_kernels()
{
    cudaFuncAttributes a;
    {
        const void* kr[] = {
            (const void*)k_argmax_resolve<TROP_MAXPLUS, 64>,  (const void*)k_argmax_resolve<TROP_MINPLUS, 64>,
            (const void*)k_argmax_resolve<TROP_MAXTIMES, 64>, (const void*)k_argmax_resolve<TROP_MAXPLUS, 32>,
            (const void*)k_argmax_resolve<TROP_MINPLUS, 32>,  (const void*)k_argmax_resolve<TROP_MAXTIMES, 32>,
            (const void*)k_argmax_resolve<TROP_MAXPLUS, 16>,  (const void*)k_argmax_resolve<TROP_MINPLUS, 16>,
            (const void*)k_argmax_resolve<TROP_MAXTIMES, 16>,  (const void*)k_argmax_resolve_rows<TROP_MAXPLUS, false>,
            (const void*)k_argmax_resolve_rows<TROP_MINPLUS, false>,   (const void*)k_argmax_resolve_rows<TROP_MAXTIMES, false>,
            (const void*)k_argmax_resolve_rows<TROP_MAXPLUS, true>,
            (const void*)k_argmax_resolve_rows<TROP_MINPLUS, true>,    (const void*)k_argmax_resolve_rows<TROP_MAXTIMES, true>};
        for (const void* k : kr) {
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_RESOLVE);
            if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute (argmax resolve smem)");
        }
    }
    const void* ks[] = {
        (const void*)k_gemm_tiled<TROP_MAXPLUS, true, tile_tn<true>()>,  (const void*)k_gemm_tiled<TROP_MINPLUS, true, tile_tn<true>()>,
        (const void*)k_gemm_tiled<TROP_MAXTIMES, true, tile_tn<true>()>, (const void*)k_gemm_tiled<TROP_MAXPLUS, false, tile_tn<false>()>,
        (const void*)k_gemm_stream<TROP_MAXPLUS, true, 4, 2>, (const void*)k_gemm_stream<TROP_MAXPLUS, true, 1, 2>,
        (const void*)k_gemm_generic<TROP_MAXPLUS, true>,
    };
    for (const void* k : ks) {
        cudaError_t e = cudaFuncGetAttributes(&a, k);
        if (e != cudaSuccess) return cuda_error(e, "cudaFuncGetAttributes (gemm kernels)");
    }
    return TROP_OK;
}

}  // namespace trop

extern "C" int tropical_device_wait_timeouts(unsigned int* count, int reset)
{
    using namespace trop;
    if (!count) return set_error(TROP_ERR_INVALID_ARG, "count pointer is NULL");
    const DeviceInfo* dev = nullptr;
    TROP_TRY(ensure_device(&dev));
    cudaError_t e = cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(unsigned int));
    if (e != cudaSuccess) return cuda_error(e, "reading the wait-timeout counter");
    if (reset) {
        const unsigned int z = 0;
        e = cudaMemcpyToSymbol(g_wait_timeouts, &z, sizeof(unsigned int));
        if (e != cudaSuccess) return cuda_error(e, "resetting the wait-timeout counter");
    }
    return TROP_OK;
}
