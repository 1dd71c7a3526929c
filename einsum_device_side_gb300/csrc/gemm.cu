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
// Argmax without a compare per term: k is walked in chunks of 16 (one
// shared-memory stage).  At the end of a chunk each output compares its
// running result with a snapshot taken at the chunk's start; a strict
// improvement stores the chunk number.  Because the running result only
// grows (shrinks for min-plus), the last improving chunk holds the first k
// that reaches the final value, and an epilogue recomputes just that chunk's
// 16 products to find it.  If nothing beat the semiring zero the argmax is 0,
// which is what a strict left-to-right scan gives.
//
// Kernels:
//   k_gemm_tiled   64x64 output tile per 64-thread CTA, 8x8 per thread,
//                  A staged transposed and duplicated ({a,a} pairs) so the
//                  packed add needs no register shuffles; needs sAk == 1
//                  and sBn == 1 (the planner permutes other layouts).
//   k_gemm_stream  few rows (M <= 8) and a short contraction (K <= 64):
//                  one thread per (batch, column vector), memory bound.
//   k_gemm_generic anything else: one thread per output, sequential k.
#include <cuda_runtime.h>

#include <cstdint>

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
constexpr int BM = 64, BN = 64, BK = 16, TM = 8, TN = 8;
constexpr int TTHREADS = (BM / TM) * (BN / TN);  // 64
constexpr int APAD = 4;                          // float pad per transposed A row (keeps 16-byte rows)
#ifndef TROP_ARG_CHUNK
#define TROP_ARG_CHUNK 8
#endif
constexpr int CH = TROP_ARG_CHUNK;               // k per argmax chunk (divides BK)
static_assert(BK % CH == 0 && CH % 2 == 0, "chunk must divide the k-tile and hold whole k pairs");

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
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes)
{
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(sa), "l"(gmem), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::); }

// rows / columns of the 8x8 outputs a thread owns: two groups of 4, half a tile apart
__device__ __forceinline__ int row_of(int tm, int i) { return i < 4 ? tm * 4 + i : BM / 2 + tm * 4 + (i - 4); }
__device__ __forceinline__ int col_of(int tn, int j) { return j < 4 ? tn * 4 + j : BN / 2 + tn * 4 + (j - 4); }

// ARG: besides C, writes into I the chunk (+1) that holds each output's first
// maximum, or 0 when no product beat the semiring zero; k_argmax_resolve then
// replaces the chunk by the exact index.
template <int SR, bool ARG>
__global__ void __launch_bounds__(TTHREADS) k_gemm_tiled(TiledParams p)
{
    using O = Ops<SR>;
    __shared__ __align__(16) float As[2][BK][BM + APAD];  // A transposed: As[k][m]
    __shared__ __align__(16) float Bs[2][BK][BN];
    __shared__ uint16_t sid[ARG ? TM * TN : 1][ARG ? TTHREADS : 1];

    const int tid = threadIdx.x;
    const int tm = tid / (BN / TN), tn = tid % (BN / TN);
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int nkt = (p.K + BK - 1) / BK;
    const float zero = O::zero();

    for (uint32_t b = blockIdx.z; b < p.nbatch; b += gridDim.z) {
        int64_t oa, ob, oc, oi;
        batch_offsets(p.bt, b, oa, ob, oc, oi);
        const float* __restrict__ A = p.A + oa;
        const float* __restrict__ B = p.B + ob;

        // loader roles: A: rows tid/4 + 16*r, k quad (tid%4)*4;  B: rows tid/16 + 4*r, n quad (tid%16)*4
        const int la_m = tid / 4, la_k = (tid % 4) * 4;
        const int lb_k = tid / 16, lb_n = (tid % 16) * 4;

        float4 ra[4];
        auto load_a = [&](int kt) {
            const int k0 = kt * BK;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int m = m0 + la_m + 16 * r, k = k0 + la_k;
                const float* src = A + (int64_t)m * p.sAm + k;
                if (m < p.M && k + 3 < p.K && p.vecA) {
                    ra[r] = __ldg(reinterpret_cast<const float4*>(src));
                } else {
                    float v[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) v[q] = (m < p.M && k + q < p.K) ? __ldg(src + q) : zero;
                    ra[r] = make_float4(v[0], v[1], v[2], v[3]);
                }
            }
        };
        auto store_a = [&](int buf) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int m = la_m + 16 * r;
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
            for (int r = 0; r < 4; ++r) {
                const int kk = lb_k + 4 * r, k = k0 + kk, n = n0 + lb_n;
                float* dst = &Bs[buf][kk][lb_n];
                if (p.vecB) {
                    const int valid = (k < p.K) ? max(0, min(4, p.N - n)) : 0;
                    const float* src = valid ? B + (int64_t)k * p.sBk + n : B;
                    cp_async16(dst, src, valid * 4);
                } else {
                    const float* src = B + (int64_t)k * p.sBk + n;
#pragma unroll
                    for (int q = 0; q < 4; ++q) dst[q] = (k < p.K && n + q < p.N) ? __ldg(src + q) : 0.0f;
                }
            }
            cp_async_commit();
        };

        float best[TM][TN];
        float snap[ARG ? TM : 1][ARG ? TN : 1];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                best[i][j] = zero;
                if (ARG) snap[ARG ? i : 0][ARG ? j : 0] = zero;
            }

        issue_b(0, 0);
        load_a(0);
        store_a(0);
        cp_async_wait_all();
        __syncthreads();
        for (int kt = 0; kt < nkt; ++kt) {
            const int buf = kt & 1;
            if (kt + 1 < nkt) {
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
                    const float4 u = *reinterpret_cast<const float4*>(&Bs[buf][kk][tn * 4]);
                    const float4 v = *reinterpret_cast<const float4*>(&Bs[buf][kk][BN / 2 + tn * 4]);
                    const float4 u1 = *reinterpret_cast<const float4*>(&Bs[buf][kk + 1][tn * 4]);
                    const float4 v1 = *reinterpret_cast<const float4*>(&Bs[buf][kk + 1][BN / 2 + tn * 4]);
                    a0[0] = x.x; a0[1] = x.y; a0[2] = x.z; a0[3] = x.w;
                    a0[4] = y.x; a0[5] = y.y; a0[6] = y.z; a0[7] = y.w;
                    a1[0] = x1.x; a1[1] = x1.y; a1[2] = x1.z; a1[3] = x1.w;
                    a1[4] = y1.x; a1[5] = y1.y; a1[6] = y1.z; a1[7] = y1.w;
                    b0[0] = u.x; b0[1] = u.y; b0[2] = u.z; b0[3] = u.w;
                    b0[4] = v.x; b0[5] = v.y; b0[6] = v.z; b0[7] = v.w;
                    b1[0] = u1.x; b1[1] = u1.y; b1[2] = u1.z; b1[3] = u1.w;
                    b1[4] = v1.x; b1[5] = v1.y; b1[6] = v1.z; b1[7] = v1.w;
                }
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; j += 2) {
                        const float2 t0 = O::mul2(make_float2(a0[i], a0[i]), make_float2(b0[j], b0[j + 1]));
                        const float2 t1 = O::mul2(make_float2(a1[i], a1[i]), make_float2(b1[j], b1[j + 1]));
                        best[i][j] = O::fold3(best[i][j], t0.x, t1.x);
                        best[i][j + 1] = O::fold3(best[i][j + 1], t0.y, t1.y);
                    }
                if (ARG && (kk + 2) % CH == 0) {
                    // end of a chunk: a strict improvement over the chunk-start value marks it
                    const uint16_t chunk = (uint16_t)((kt * BK + kk + 2) / CH - 1);
#pragma unroll
                    for (int i = 0; i < TM; ++i)
#pragma unroll
                        for (int j = 0; j < TN; ++j) {
                            float& s = snap[ARG ? i : 0][ARG ? j : 0];
                            if (O::better(best[i][j], s)) sid[i * TN + j][tid] = chunk;
                            s = best[i][j];
                        }
                }
            }
            if (kt + 1 < nkt) store_a(buf ^ 1);
            cp_async_wait_all();
            __syncthreads();
        }

        // ---------------- store values (and chunk + 1) through the output strides
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int m = m0 + row_of(tm, i);
            if (m >= p.M) continue;
            float* crow = p.C + oc + (int64_t)m * p.sCm;
            int32_t* irow = ARG ? p.I + oi + (int64_t)m * p.sIm : nullptr;
            int32_t code[TN];
            if (ARG) {
#pragma unroll
                for (int j = 0; j < TN; ++j) code[j] = best[i][j] != zero ? (int32_t)sid[i * TN + j][tid] + 1 : 0;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int n = n0 + (h ? BN / 2 : 0) + tn * 4;
                if (p.vecC && n + 3 < p.N) {
                    *reinterpret_cast<float4*>(crow + n) =
                        make_float4(best[i][4 * h], best[i][4 * h + 1], best[i][4 * h + 2], best[i][4 * h + 3]);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (n + q < p.N) crow[(int64_t)(n + q) * p.sCn] = best[i][4 * h + q];
                }
                if (ARG) {
                    if (p.vecI && n + 3 < p.N) {
                        *reinterpret_cast<int4*>(irow + n) =
                            make_int4(code[4 * h], code[4 * h + 1], code[4 * h + 2], code[4 * h + 3]);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (n + q < p.N) irow[(int64_t)(n + q) * p.sIn] = code[4 * h + q];
                    }
                }
            }
        }
        // no barrier needed: the next batch iteration starts by writing stage 0, which every
        // thread finished reading before the last loop barrier
    }
}

// ------------------------------------------------------------------ argmax resolve
// One CTA (256 threads) per 64x64 output tile.  Each thread holds 16 outputs of
// the tile (4 rows x 4 consecutive columns) in registers: value and chunk
// code.  B's rows are staged into shared memory 256 k at a time; for each of
// its outputs whose chunk lies in the staged group a thread recomputes the
// chunk's CH products -- A's contiguous row segment through L1, B's column
// from shared memory -- and keeps the first k whose product equals the value.
// Results go back from registers with coalesced stores.
constexpr int RTHREADS = 256, RGK = 256;
constexpr size_t SMEM_RESOLVE = sizeof(float) * RGK * BN;  // 64 KiB

template <int SR>
__global__ void __launch_bounds__(RTHREADS, 2) k_argmax_resolve(TiledParams p)
{
    using O = Ops<SR>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float(*EB)[BN] = reinterpret_cast<float(*)[BN]>(smem_raw);
    const int tid = threadIdx.x;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int ngr = (p.K + RGK - 1) / RGK;
    // my outputs: rows rr + 16*r (r < 4), columns cc .. cc+3
    const int rr = tid / 16, cc = (tid % 16) * 4;
    for (uint32_t b = blockIdx.z; b < p.nbatch; b += gridDim.z) {
        int64_t oa, ob, oc, oi;
        batch_offsets(p.bt, b, oa, ob, oc, oi);
        const float* __restrict__ A = p.A + oa;
        const float* __restrict__ B = p.B + ob;
        float val[4][4];
        int code[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int m = m0 + rr + 16 * r, n = n0 + cc;
            const float* crow = p.C + oc + (int64_t)m * p.sCm;
            const int32_t* irow = p.I + oi + (int64_t)m * p.sIm;
            if (m < p.M && n + 3 < p.N && p.vecC && p.vecI) {
                const float4 c4 = *reinterpret_cast<const float4*>(crow + n);
                const int4 i4 = *reinterpret_cast<const int4*>(irow + n);
                val[r][0] = c4.x; val[r][1] = c4.y; val[r][2] = c4.z; val[r][3] = c4.w;
                code[r][0] = i4.x; code[r][1] = i4.y; code[r][2] = i4.z; code[r][3] = i4.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool in = m < p.M && n + j < p.N;
                    val[r][j] = in ? crow[(int64_t)(n + j) * p.sCn] : 0.0f;
                    code[r][j] = in ? irow[(int64_t)(n + j) * p.sIn] : 0;
                }
            }
        }
        int res[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int j = 0; j < 4; ++j) res[r][j] = 0;  // code 0: nothing beat the zero, argmax 0
        for (int g = 0; g < ngr; ++g) {
            const int k0 = g * RGK;
            const int kn = min(RGK, p.K - k0);
            bool any = false;
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int ch = code[r][j] - 1;
                    any |= ch >= 0 && ch * CH >= k0 && ch * CH < k0 + RGK;
                }
            if (!__syncthreads_or(any)) continue;
            // stage B rows k0 .. k0+kn of this tile's columns (zero outside the operand)
            for (int e = tid; e < kn * (BN / 4); e += RTHREADS) {
                const int kk = e / (BN / 4), nq = (e % (BN / 4)) * 4, gk = k0 + kk, gn = n0 + nq;
                float* dst = &EB[kk][nq];
                if (p.vecB) {
                    const int valid = max(0, min(4, p.N - gn));
                    cp_async16(dst, valid ? B + (int64_t)gk * p.sBk + gn : B, valid * 4);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[q] = (gn + q < p.N) ? __ldg(B + (int64_t)gk * p.sBk + gn + q) : 0.0f;
                }
            }
            cp_async_commit();
            cp_async_wait_all();
            __syncthreads();
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int m = m0 + rr + 16 * r;
                const float* arow = A + (int64_t)m * p.sAm;
                // the four columns' A segments: all loads in flight before any search
                float av[4][CH];
                int ka[4];
                bool live[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int ch = code[r][j] - 1;
                    live[j] = ch >= 0 && ch * CH >= k0 && ch * CH < k0 + RGK;
                    ka[j] = live[j] ? ch * CH : 0;
                    const float* src = live[j] ? arow + ka[j] : A;
                    const int kmax = live[j] ? min(CH, p.K - ka[j]) : 0;
                    if (p.vecA && kmax == CH) {
#pragma unroll
                        for (int kk = 0; kk < CH; kk += 4) {
                            const float4 x = __ldg(reinterpret_cast<const float4*>(src + kk));
                            av[j][kk] = x.x;
                            av[j][kk + 1] = x.y;
                            av[j][kk + 2] = x.z;
                            av[j][kk + 3] = x.w;
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < CH; ++kk) av[j][kk] = kk < kmax ? __ldg(src + kk) : 0.0f;
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (!live[j]) continue;
                    const int kl = ka[j] - k0, c = cc + j;
                    const int kmax = min(CH, p.K - ka[j]);
                    const float target = val[r][j];
                    int idx = 0;
#pragma unroll
                    for (int kk = CH - 1; kk >= 0; --kk)
                        if (kk < kmax && O::mul(av[j][kk], EB[kl + kk][c]) == target) idx = kk;
                    res[r][j] = ka[j] + idx;
                }
            }
            __syncthreads();  // before the next group overwrites the staged rows
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int m = m0 + rr + 16 * r, n = n0 + cc;
            if (m >= p.M) continue;
            int32_t* irow = p.I + oi + (int64_t)m * p.sIm;
            if (n + 3 < p.N && p.vecI) {
                *reinterpret_cast<int4*>(irow + n) = make_int4(res[r][0], res[r][1], res[r][2], res[r][3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (n + j < p.N) irow[(int64_t)(n + j) * p.sIn] = res[r][j];
            }
        }
    }
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
};

template <int SR, bool ARG, int VEC, int MAXM>
__global__ void __launch_bounds__(256) k_gemm_stream(StreamParams p)
{
    using O = Ops<SR>;
    for (uint32_t e = blockIdx.x * blockDim.x + threadIdx.x; e < p.total; e += gridDim.x * blockDim.x) {
        const uint32_t b = fdiv(e, p.div_nvec);
        const int n = (int)(e - b * p.nvec) * VEC;
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
                float4 x = __ldg(reinterpret_cast<const float4*>(Bb + (int64_t)k * p.sBk));
                bv[0] = x.x;
                bv[VEC > 1 ? 1 : 0] = x.y;
                bv[VEC > 2 ? 2 : 0] = x.z;
                bv[VEC > 3 ? 3 : 0] = x.w;
            } else {
#pragma unroll
                for (int v = 0; v < VEC; ++v) bv[v] = __ldg(Bb + (int64_t)k * p.sBk + (int64_t)v * p.sBn);
            }
#pragma unroll
            for (int m = 0; m < MAXM; ++m) {
                if (m < p.M) {
                    const float a = __ldg(Ab + (int64_t)m * p.sAm + (int64_t)k * p.sAk);
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
                    *reinterpret_cast<float4*>(cp) =
                        make_float4(best[m][0], best[m][VEC > 1 ? 1 : 0], best[m][VEC > 2 ? 2 : 0],
                                    best[m][VEC > 3 ? 3 : 0]);
                    if (ARG)
                        *reinterpret_cast<int4*>(ip) = make_int4(idx[m][0], idx[m][VEC > 1 ? 1 : 0],
                                                                 idx[m][VEC > 2 ? 2 : 0], idx[m][VEC > 3 ? 3 : 0]);
                } else {
#pragma unroll
                    for (int v = 0; v < VEC; ++v) {
                        cp[(int64_t)v * p.sCn] = best[m][v];
                        if (ARG) ip[(int64_t)v * p.sIn] = idx[m][v];
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
};

template <int SR, bool ARG>
__global__ void k_gemm_generic(GenericParams p)
{
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
            const float t = O::mul(__ldg(a + k * p.sAk), __ldg(b + k * p.sBk));
            if (O::better(t, best)) {
                best = t;
                idx = k;
            }
        }
        p.C[oc + m * p.sCm + n * p.sCn] = best;
        if (ARG) p.I[oi + m * p.sIm + n * p.sIn] = (int32_t)idx;
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

template <int SR, bool ARG>
int run_tiled(const GemmDesc& g, cudaStream_t s)
{
    TiledParams p{};
    p.M = (int)g.M;
    p.N = (int)g.N;
    p.K = (int)g.K;
    p.A = g.A;
    p.B = g.B;
    p.C = g.C;
    p.I = g.I;
    p.sAm = g.sAm;
    p.sBk = g.sBk;
    p.sCm = g.sCm;
    p.sCn = g.sCn;
    p.sIm = g.sIm;
    p.sIn = g.sIn;
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
    dim3 grid((unsigned)((g.N + BN - 1) / BN), (unsigned)((g.M + BM - 1) / BM),
              (unsigned)(nbatch < 65535 ? nbatch : 65535));
    k_gemm_tiled<SR, ARG><<<grid, TTHREADS, 0, s>>>(p);
    TROP_TRY(check_launch("k_gemm_tiled"));
    if (ARG) {
        k_argmax_resolve<SR><<<grid, RTHREADS, SMEM_RESOLVE, s>>>(p);
        TROP_TRY(check_launch("k_argmax_resolve"));
    }
    return TROP_OK;
}

template <int SR, bool ARG>
int run_stream(const GemmDesc& g, cudaStream_t s, const DeviceInfo* dev)
{
    StreamParams p{};
    p.M = (int)g.M;
    p.N = (int)g.N;
    p.K = (int)g.K;
    p.A = g.A;
    p.B = g.B;
    p.C = g.C;
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
    bool vec = g.N % 4 == 0 && g.sBn == 1 && g.sCn == 1 && (!ARG || g.sIn == 1) && ((uintptr_t)g.B % 16) == 0 &&
               ((uintptr_t)g.C % 16) == 0 && (!ARG || ((uintptr_t)g.I % 16) == 0) && g.sBk % 4 == 0 &&
               g.sCm % 4 == 0 && (!ARG || g.sIm % 4 == 0);
    for (int d = 0; d < p.bt.nb; ++d)
        vec = vec && p.bt.sB[d] % 4 == 0 && p.bt.sC[d] % 4 == 0 && (!ARG || p.bt.sI[d] % 4 == 0);
    const int VEC = vec ? 4 : 1;
    p.nvec = (uint32_t)(g.N / VEC);
    p.div_nvec = make_fastdiv(p.nvec);
    p.total = (uint32_t)(nbatch * p.nvec);
    int64_t blocks = ((int64_t)p.total + 255) / 256;
    int64_t cap = (int64_t)dev->sm_count * 16;
    int grid = (int)(blocks < cap ? (blocks < 1 ? 1 : blocks) : cap);
    // register arrays sized to the rows actually present keep occupancy high
    if (g.M <= 2) {
        if (vec) k_gemm_stream<SR, ARG, 4, 2><<<grid, 256, 0, s>>>(p);
        else k_gemm_stream<SR, ARG, 1, 2><<<grid, 256, 0, s>>>(p);
    } else if (g.M <= 4) {
        if (vec) k_gemm_stream<SR, ARG, 4, 4><<<grid, 256, 0, s>>>(p);
        else k_gemm_stream<SR, ARG, 1, 4><<<grid, 256, 0, s>>>(p);
    } else {
        if (vec) k_gemm_stream<SR, ARG, 4, MAXM_STREAM><<<grid, 256, 0, s>>>(p);
        else k_gemm_stream<SR, ARG, 1, MAXM_STREAM><<<grid, 256, 0, s>>>(p);
    }
    return check_launch("k_gemm_stream");
}

template <int SR, bool ARG>
int run_generic(const GemmDesc& g, cudaStream_t s, const DeviceInfo* dev)
{
    GenericParams p{};
    p.M = g.M;
    p.N = g.N;
    p.K = g.K;
    p.A = g.A;
    p.B = g.B;
    p.C = g.C;
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
    k_gemm_generic<SR, ARG><<<grid, 256, 0, s>>>(p);
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
    const bool grid_ok = (g.M + BM - 1) / BM <= 65535 && (g.N + BN - 1) / BN <= 65535;
    const bool grid_ok_t = (g.N + BM - 1) / BM <= 65535 && (g.M + BN - 1) / BN <= 65535;
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

template <int SR, bool ARG>
int run(const GemmDesc& g0, cudaStream_t s, const DeviceInfo* dev, const char** name)
{
    bool swap = false;
    Route r = choose(g0, swap);
    const GemmDesc g = swap ? swapped(g0) : g0;
    switch (r) {
    case R_TILED:
        if (name) *name = "k_gemm_tiled";
        return run_tiled<SR, ARG>(g, s);
    case R_STREAM:
        if (name) *name = "k_gemm_stream";
        return run_stream<SR, ARG>(g, s, dev);
    default:
        if (name) *name = "k_gemm_generic";
        return run_generic<SR, ARG>(g, s, dev);
    }
}

}  // namespace

int launch_gemm(const GemmDesc& g, cudaStream_t s, const char** kernel_name)
{
    const DeviceInfo* dev = nullptr;
    TROP_TRY(ensure_device(&dev));
    if (g.M == 0 || g.N == 0) return TROP_OK;
    for (int d = 0; d < g.nb; ++d)
        if (g.bsize[d] == 0) return TROP_OK;
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
        const void* kr[] = {(const void*)k_argmax_resolve<TROP_MAXPLUS>, (const void*)k_argmax_resolve<TROP_MINPLUS>,
                            (const void*)k_argmax_resolve<TROP_MAXTIMES>};
        for (const void* k : kr) {
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_RESOLVE);
            if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute (argmax resolve smem)");
        }
    }
    const void* ks[] = {
        (const void*)k_gemm_tiled<TROP_MAXPLUS, true>,  (const void*)k_gemm_tiled<TROP_MINPLUS, true>,
        (const void*)k_gemm_tiled<TROP_MAXTIMES, true>, (const void*)k_gemm_tiled<TROP_MAXPLUS, false>,
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
