// gemm_int.cu -- strided-batched tropical GEMM on integer operands (i32, i64), with argmax.
//
// C[m,n] = (+)_k A[m,k] (x) B[k,n] with the (+) and (x) of the max-plus, min-plus and
// max-times semirings on exact integers.  Integer operands: omeinsum-rs issue #52, "Resolved
// design for step 3" kernel (a) (integer types in the permute/gather) and tropical-gemm PR #35,
// "Summary of latest fixes" (dtype handling beyond f32).  The pages fix no overflow policy for
// an integer contraction; the library's reading is that every product formed must fit the
// operand type (a + b, or a * b for max-times), so the results are exact.  Products are
// formed in unsigned arithmetic (wrapping, never undefined), which equals the exact integer
// whenever the precondition holds.  The zero is the type's min / max / 0 and only starts the
// running (+); argmax is the smallest k reaching the result (strict compare), 0 when nothing
// beats the zero.
//
// Tiles: 64 x 64 outputs per CTA, 256 threads, 4 x 4 outputs per thread (rows ty + 16i,
// columns tx + 16j, so a warp's stores are contiguous along n), K in chunks of 16 staged
// through shared memory; any strides (the staging walks k fastest for an operand whose k
// stride is 1).  Rows and columns past M and N are staged as 0 and never stored; a partial
// last chunk of K is walked only up to K.  Tiles are taken by a grid-stride loop.
#include <cuda_runtime.h>

#include <climits>
#include <type_traits>

#define TROP_TU 4  // this file's id in a bounds-violation record
#include "internal.h"

namespace trop {
namespace {

constexpr int I_BM = 64, I_BN = 64, I_BK = 16, I_THREADS = 256;
constexpr int I_LD = I_BM + 1;  // padded row of the staged tiles

template <int SR, typename T>
struct IOps {
    using U = typename std::make_unsigned<T>::type;
    __device__ static T zero()
    {
        if (SR == TROP_MAXTIMES) return T(0);
        if (std::is_same<T, int32_t>::value) return SR == TROP_MAXPLUS ? T(INT32_MIN) : T(INT32_MAX);
        return SR == TROP_MAXPLUS ? T(LLONG_MIN) : T(LLONG_MAX);
    }
    // exact when the product fits T (the precondition); wraps instead of overflowing otherwise
    __device__ static T mul(T a, T b) { return SR == TROP_MAXTIMES ? T(U(a) * U(b)) : T(U(a) + U(b)); }
    __device__ static bool better(T t, T best) { return SR == TROP_MINPLUS ? t < best : t > best; }
};

template <typename T>
struct GemmIntParams {
    int64_t M, N, K;
    const T* A;
    const T* B;
    T* C;
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

template <int SR, typename T, bool ARG>
__global__ void __launch_bounds__(I_THREADS) k_gemm_int(GemmIntParams<T> p)
{
    using O = IOps<SR, T>;
    pdl_wait();
    pdl_signal();
    __shared__ T As[I_BK][I_LD];
    __shared__ T Bs[I_BK][I_LD];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const T zero = O::zero();

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
        const int64_t m0 = tm * I_BM, n0 = tn * I_BN;
        const T* __restrict__ A = p.A + oa;
        const T* __restrict__ B = p.B + ob;

        T best[4][4];
        int32_t idx[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                best[i][j] = zero;
                idx[i][j] = 0;
            }

        for (int64_t k0 = 0; k0 < p.K; k0 += I_BK) {
            const int kc = (int)(p.K - k0 < I_BK ? p.K - k0 : I_BK);
#pragma unroll
            for (int q = 0; q < (I_BM * I_BK) / I_THREADS; ++q) {
                const int e = tid + q * I_THREADS;
                const int kk = p.a_kfast ? (e & (I_BK - 1)) : (e / I_BM);
                const int mm = p.a_kfast ? (e / I_BK) : (e & (I_BM - 1));
                const int64_t m = m0 + mm;
                T v = T(0);
                if (kk < kc && m < p.M && TROP_IN(A + m * p.sAm + (k0 + kk) * p.sAk, sizeof(*A), p.sp[0]))
                    v = __ldg(A + m * p.sAm + (k0 + kk) * p.sAk);
                As[kk][mm] = v;
            }
#pragma unroll
            for (int q = 0; q < (I_BN * I_BK) / I_THREADS; ++q) {
                const int e = tid + q * I_THREADS;
                const int kk = p.b_kfast ? (e & (I_BK - 1)) : (e / I_BN);
                const int nn = p.b_kfast ? (e / I_BK) : (e & (I_BN - 1));
                const int64_t n = n0 + nn;
                T v = T(0);
                if (kk < kc && n < p.N && TROP_IN(B + (k0 + kk) * p.sBk + n * p.sBn, sizeof(*B), p.sp[1]))
                    v = __ldg(B + (k0 + kk) * p.sBk + n * p.sBn);
                Bs[kk][nn] = v;
            }
            __syncthreads();
            auto step = [&](int kk) {
                T a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const T v = O::mul(a[i], b[j]);
                        if (O::better(v, best[i][j])) {
                            best[i][j] = v;
                            if (ARG) idx[i][j] = (int32_t)(k0 + kk);
                        }
                    }
            };
            if (kc == I_BK) {
#pragma unroll
                for (int kk = 0; kk < I_BK; ++kk) step(kk);
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
                    p.C[oc + m * p.sCm + n * p.sCn] = best[i][j];
                if (ARG && TROP_IN(p.I + oi + m * p.sIm + n * p.sIn, 4, p.sp[3])) p.I[oi + m * p.sIm + n * p.sIn] = idx[i][j];
            }
        }
    }
}

template <int SR, typename T, bool ARG>
int run_int(const GemmDesc& g0, cudaStream_t s, const DeviceInfo* dev)
{
    // (x) commutes exactly, so C^T = B^T (x) A^T: take the orientation whose output is
    // contiguous along the tile's fast (n) direction
    GemmDesc g = g0;
    const bool swap = g0.sCn != 1 && g0.sCm == 1 && (!ARG || g0.sIm == 1);
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
    GemmIntParams<T> p{};
#if TROP_DEBUG_BOUNDS
    gemm_spans(g, sizeof(*p.A), p.sp);
#endif
    p.M = g.M;
    p.N = g.N;
    p.K = g.K;
    p.A = static_cast<const T*>(g.A);
    p.B = static_cast<const T*>(g.B);
    p.C = static_cast<T*>(g.C);
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
    p.tiles_m = (g.M + I_BM - 1) / I_BM;
    p.tiles_n = (g.N + I_BN - 1) / I_BN;
    p.total = nbatch * p.tiles_m * p.tiles_n;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_gemm_int<SR, T, ARG>, I_THREADS, 0);
    if (e != cudaSuccess) return cuda_error(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor (integer gemm)");
    const int64_t cap = (int64_t)dev->sm_count * (per_sm > 0 ? per_sm : 1);
    const int grid = (int)(p.total < cap ? p.total : cap);
    (void)launch_pdl(k_gemm_int<SR, T, ARG>, dim3(grid), dim3(I_THREADS), 0, s, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "k_gemm_int");
    count_launches(1);
    return TROP_OK;
}

template <typename T>
int dispatch(const GemmDesc& g, cudaStream_t s, const DeviceInfo* dev)
{
    const bool arg = g.I != nullptr;
    switch (g.semiring) {
    case TROP_MAXPLUS: return arg ? run_int<TROP_MAXPLUS, T, true>(g, s, dev) : run_int<TROP_MAXPLUS, T, false>(g, s, dev);
    case TROP_MINPLUS: return arg ? run_int<TROP_MINPLUS, T, true>(g, s, dev) : run_int<TROP_MINPLUS, T, false>(g, s, dev);
    case TROP_MAXTIMES:
        return arg ? run_int<TROP_MAXTIMES, T, true>(g, s, dev) : run_int<TROP_MAXTIMES, T, false>(g, s, dev);
    default: return set_error(TROP_ERR_INVALID_ARG, "unknown semiring %d", g.semiring);
    }
}

}  // namespace

int launch_gemm_int(const GemmDesc& g, cudaStream_t s)
{
    const DeviceInfo* dev = nullptr;
    TROP_TRY(ensure_device(&dev));
    if (g.M == 0 || g.N == 0) return TROP_OK;
    for (int d = 0; d < g.nb; ++d)
        if (g.bsize[d] == 0) return TROP_OK;
    if (g.dtype == TROP_I32) return dispatch<int32_t>(g, s, dev);
    if (g.dtype == TROP_I64) return dispatch<int64_t>(g, s, dev);
    return set_error(TROP_ERR_DTYPE, "integer tropical GEMM: unsupported dtype %d", g.dtype);
}

int register_gemm_int_kernels()
{
    cudaFuncAttributes a;
    const void* ks[] = {
        (const void*)k_gemm_int<TROP_MAXPLUS, int32_t, true>, (const void*)k_gemm_int<TROP_MINPLUS, int32_t, true>,
        (const void*)k_gemm_int<TROP_MAXTIMES, int32_t, true>, (const void*)k_gemm_int<TROP_MAXPLUS, int64_t, true>,
        (const void*)k_gemm_int<TROP_MINPLUS, int64_t, true>, (const void*)k_gemm_int<TROP_MAXTIMES, int64_t, true>,
    };
    for (const void* k : ks) {
        cudaError_t e = cudaFuncGetAttributes(&a, k);
        if (e != cudaSuccess) return cuda_error(e, "cudaFuncGetAttributes (integer gemm kernels)");
    }
    return TROP_OK;
}

}  // namespace trop
