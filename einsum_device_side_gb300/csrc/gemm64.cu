// gemm64.cu -- strided-batched tropical GEMM in binary64 (f64), with argmax.
//
// The operation is the one of gemm.cu, C[m,n] = (+)_k A[m,k] (x) B[k,n] with
// the (+) and (x) of the max-plus, min-plus and max-times semirings, here in
// binary64.  f64 operands: omeinsum-rs issue #52, "Resolved design for step 3"
// kernel (a) (the generic kernels serve f32 and f64 operands), and
// tropical-gemm PR #35, "Summary of latest fixes" (CPU dtype handling for f32
// and f64).  Each (x) is one correctly rounded double add or multiply, each
// (+) an exact comparison, argmax the smallest k that attains the optimum.
//
// GB300 runs binary64 arithmetic on a narrow pipe (about two operations per
// SM per clock, far below the FP32 lanes), so the one double operation a
// semiring step cannot avoid is the add or multiply.  Everything else stays
// off that pipe: the comparison uses the order-preserving integer image of the
// double (sign-magnitude folded into two's complement, so a signed 64-bit
// compare orders like the double for every non-NaN value), which the integer
// lanes evaluate.  With one double op per step and plenty of integer lanes
// the kernel's bound is the binary64 pipe; shared-memory and global traffic
// per step are a small fraction of what it could sustain.
//
// Tiles: 64 x 64 outputs per CTA, 256 threads, 4 x 4 outputs per thread
// (rows ty + 16i, columns tx + 16j, so the stores of a warp are contiguous
// along n), K in chunks of 16 staged through shared memory.  Tiles are walked
// by a grid-stride loop over (batch, tile row, tile column).
#include <cuda_runtime.h>
#include <math.h>

#define TROP_TU 3  // this file's id in a bounds-violation record
#include "internal.h"

namespace trop {
namespace {

constexpr int D_BM = 64, D_BN = 64, D_BK = 16, D_THREADS = 256;
constexpr int D_LD = D_BM + 1;  // padded row (doubles) of the staged tiles
// two CTAs per SM: sixteen warps to hide the shared-memory latency of the operand reads
#ifndef TROP_F64_MINB
#define TROP_F64_MINB 2
#endif

// order key: signed 64-bit integer that compares like the double (no NaN)
__device__ __forceinline__ long long okey(double x)
{
    const long long b = __double_as_longlong(x);
    return b ^ (long long)((unsigned long long)(b >> 63) >> 1);
}
__device__ __forceinline__ double from_okey(long long k)
{
    return __longlong_as_double(k ^ (long long)((unsigned long long)(k >> 63) >> 1));
}

template <int SR>
struct Ops64 {
    __device__ static double zero()
    {
        return SR == TROP_MAXPLUS ? -INFINITY : SR == TROP_MINPLUS ? INFINITY : 0.0;
    }
    __device__ static double mul(double a, double b) { return SR == TROP_MAXTIMES ? __dmul_rn(a, b) : __dadd_rn(a, b); }
    __device__ static bool better(long long t, long long best) { return SR == TROP_MINPLUS ? t < best : t > best; }
};

struct Gemm64Params {
    int64_t M, N, K;
    const double* A;
    const double* B;
    double* C;
    int32_t* I;
    int64_t sAm, sAk, sBk, sBn, sCm, sCn, sIm, sIn;
    int64_t tiles_m, tiles_n, total;
    int a_kfast, b_kfast;  // staging walks k fastest (that operand's k stride is 1)
    int nb;
    int64_t bsize[MAXB], sA[MAXB], sB[MAXB], sC[MAXB], sI[MAXB];
#if TROP_DEBUG_BOUNDS
    Span sp[4];  // A, B, C, I
#endif
};

template <int SR, bool ARG>
__global__ void __launch_bounds__(D_THREADS, TROP_F64_MINB) k_gemm_tiled_f64(Gemm64Params p)
{
    using O = Ops64<SR>;
    __shared__ double As[D_BK][D_LD];
    __shared__ double Bs[D_BK][D_LD];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const long long kzero = okey(O::zero());

    for (int64_t t = blockIdx.x; t < p.total; t += gridDim.x) {
        int64_t r = t;
        const int64_t tn = r % p.tiles_n;
        r /= p.tiles_n;
        const int64_t tm = r % p.tiles_m;
        r /= p.tiles_m;
        int64_t oa = 0, ob = 0, oc = 0, oi = 0;
        for (int d = p.nb - 1; d >= 0; --d) {
            const int64_t c = r % p.bsize[d];
            r /= p.bsize[d];
            oa += c * p.sA[d];
            ob += c * p.sB[d];
            oc += c * p.sC[d];
            oi += c * p.sI[d];
        }
        const int64_t m0 = tm * D_BM, n0 = tn * D_BN;
        const double* __restrict__ A = p.A + oa;
        const double* __restrict__ B = p.B + ob;

        long long best[4][4];
        int32_t idx[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                best[i][j] = kzero;
                idx[i][j] = 0;
            }

        for (int64_t k0 = 0; k0 < p.K; k0 += D_BK) {
            const int kc = (int)(p.K - k0 < D_BK ? p.K - k0 : D_BK);
            // stage A[m0.., k0..] as As[k][m] and B[k0.., n0..] as Bs[k][n]; 4 elements a thread each
#pragma unroll
            for (int q = 0; q < (D_BM * D_BK) / D_THREADS; ++q) {
                const int e = tid + q * D_THREADS;
                const int kk = p.a_kfast ? (e & (D_BK - 1)) : (e / D_BM);
                const int mm = p.a_kfast ? (e / D_BK) : (e & (D_BM - 1));
                const int64_t m = m0 + mm;
                double v = 0.0;
                if (kk < kc && m < p.M && TROP_IN(A + m * p.sAm + (k0 + kk) * p.sAk, sizeof(*A), p.sp[0]))
                    v = __ldg(A + m * p.sAm + (k0 + kk) * p.sAk);
                As[kk][mm] = v;
            }
#pragma unroll
            for (int q = 0; q < (D_BN * D_BK) / D_THREADS; ++q) {
                const int e = tid + q * D_THREADS;
                const int kk = p.b_kfast ? (e & (D_BK - 1)) : (e / D_BN);
                const int nn = p.b_kfast ? (e / D_BK) : (e & (D_BN - 1));
                const int64_t n = n0 + nn;
                double v = 0.0;
                if (kk < kc && n < p.N && TROP_IN(B + (k0 + kk) * p.sBk + n * p.sBn, sizeof(*B), p.sp[1]))
                    v = __ldg(B + (k0 + kk) * p.sBk + n * p.sBn);
                Bs[kk][nn] = v;
            }
            __syncthreads();
            auto step = [&](int kk) {
                double a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const long long v = okey(O::mul(a[i], b[j]));
                        if (O::better(v, best[i][j])) {
                            best[i][j] = v;
                            if (ARG) idx[i][j] = (int32_t)(k0 + kk);
                        }
                    }
            };
            if (kc == D_BK) {
#pragma unroll
                for (int kk = 0; kk < D_BK; ++kk) step(kk);
            } else {
                for (int kk = 0; kk < kc; ++kk) step(kk);
            }
            __syncthreads();
        }

#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t m = m0 + ty + 16 * i;
            if (m >= p.M) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t n = n0 + tx + 16 * j;
                if (n >= p.N) continue;
                if (TROP_IN(p.C + oc + m * p.sCm + n * p.sCn, sizeof(*p.C), p.sp[2]))
                    p.C[oc + m * p.sCm + n * p.sCn] = from_okey(best[i][j]);
                if (ARG && TROP_IN(p.I + oi + m * p.sIm + n * p.sIn, 4, p.sp[3])) p.I[oi + m * p.sIm + n * p.sIn] = idx[i][j];
            }
        }
    }
}

template <int SR, bool ARG>
int run_f64(const GemmDesc& g0, cudaStream_t s, const DeviceInfo* dev)
{
    // (x) commutes exactly, so C^T = B^T (x) A^T: take the orientation whose
    // output is contiguous along the tile's fast (n) direction
    GemmDesc g = g0;
    const bool arg = g0.I != nullptr;
    const bool swap = g0.sCn != 1 && g0.sCm == 1 && (!arg || g0.sIm == 1);
    if (swap) {
        g.M = g0.N;
        g.N = g0.M;
        g.A = g0.B;
        g.B = g0.A;
        g.sAm = g0.sBn;
        g.sAk = g0.sBk;
        g.sBk = g0.sAk;
        g.sBn = g0.sAm;
        g.sCm = g0.sCn;
        g.sCn = g0.sCm;
        g.sIm = g0.sIn;
        g.sIn = g0.sIm;
        for (int d = 0; d < g0.nb; ++d) {
            g.sAb[d] = g0.sBb[d];
            g.sBb[d] = g0.sAb[d];
        }
    }
    Gemm64Params p{};
#if TROP_DEBUG_BOUNDS
    gemm_spans(g, sizeof(*p.A), p.sp);
#endif
    p.M = g.M;
    p.N = g.N;
    p.K = g.K;
    p.A = static_cast<const double*>(g.A);
    p.B = static_cast<const double*>(g.B);
    p.C = static_cast<double*>(g.C);
    p.I = g.I;
    p.sAm = g.sAm;
    p.sAk = g.sAk;
    p.sBk = g.sBk;
    p.sBn = g.sBn;
    p.sCm = g.sCm;
    p.sCn = g.sCn;
    p.sIm = g.sIm;
    p.sIn = g.sIn;
    p.a_kfast = g.sAk == 1 && g.sAm != 1;
    p.b_kfast = g.sBk == 1 && g.sBn != 1;
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
    p.tiles_m = (g.M + D_BM - 1) / D_BM;
    p.tiles_n = (g.N + D_BN - 1) / D_BN;
    p.total = nbatch * p.tiles_m * p.tiles_n;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_gemm_tiled_f64<SR, ARG>, D_THREADS, 0);
    if (e != cudaSuccess) return cuda_error(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor (f64 gemm)");
    const int64_t cap = (int64_t)dev->sm_count * (per_sm > 0 ? per_sm : 1);
    const int grid = (int)(p.total < cap ? p.total : cap);
    k_gemm_tiled_f64<SR, ARG><<<grid, D_THREADS, 0, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "k_gemm_tiled_f64");
    count_launches(1);
    return TROP_OK;
}

}  // namespace

int launch_gemm_f64(const GemmDesc& g, cudaStream_t s)
{
    const DeviceInfo* dev = nullptr;
    TROP_TRY(ensure_device(&dev));
    if (g.M == 0 || g.N == 0) return TROP_OK;
    for (int d = 0; d < g.nb; ++d)
        if (g.bsize[d] == 0) return TROP_OK;
    const bool arg = g.I != nullptr;
    switch (g.semiring) {
    case TROP_MAXPLUS: return arg ? run_f64<TROP_MAXPLUS, true>(g, s, dev) : run_f64<TROP_MAXPLUS, false>(g, s, dev);
    case TROP_MINPLUS: return arg ? run_f64<TROP_MINPLUS, true>(g, s, dev) : run_f64<TROP_MINPLUS, false>(g, s, dev);
    case TROP_MAXTIMES: return arg ? run_f64<TROP_MAXTIMES, true>(g, s, dev) : run_f64<TROP_MAXTIMES, false>(g, s, dev);
    default: return set_error(TROP_ERR_INVALID_ARG, "unknown semiring %d", g.semiring);
    }
}

int register_gemm64_kernels()
{
    cudaFuncAttributes a;
    const void* ks[] = {
        (const void*)k_gemm_tiled_f64<TROP_MAXPLUS, true>,   (const void*)k_gemm_tiled_f64<TROP_MINPLUS, true>,
        (const void*)k_gemm_tiled_f64<TROP_MAXTIMES, true>,  (const void*)k_gemm_tiled_f64<TROP_MAXPLUS, false>,
        (const void*)k_gemm_tiled_f64<TROP_MINPLUS, false>,  (const void*)k_gemm_tiled_f64<TROP_MAXTIMES, false>,
    };
    for (const void* k : ks) {
        cudaError_t e = cudaFuncGetAttributes(&a, k);
        if (e != cudaSuccess) return cuda_error(e, "cudaFuncGetAttributes (f64 gemm kernels)");
    }
    return TROP_OK;
}

}  // namespace trop
