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
constexpr int APAD = 2;                          // float2 pad per A row (keeps 16-byte alignment)

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
};

template <int SR, bool ARG>
__global__ void __launch_bounds__(TTHREADS) k_gemm_tiled(TiledParams p)
{
    using O = Ops<SR>;
    __shared__ __align__(16) float2 As[2][BK][BM + APAD];
    __shared__ __align__(16) float Bs[2][BK][BN];
    __shared__ int32_t sid[ARG ? TM * TN : 1][ARG ? TTHREADS : 1];

    const int tid = threadIdx.x;
    const int tm = tid / (BN / TN), tn = tid % (BN / TN);
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int nkt = (p.K + BK - 1) / BK;

    for (uint32_t b = blockIdx.z; b < p.nbatch; b += gridDim.z) {
        int64_t oa, ob, oc, oi;
        batch_offsets(p.bt, b, oa, ob, oc, oi);
        const float* __restrict__ A = p.A + oa;
        const float* __restrict__ B = p.B + ob;

        // loader roles: A: rows tid/4 + 16*r, k quad (tid%4)*4;  B: rows tid/16 + 4*r, n quad (tid%16)*4
        const int la_m = tid / 4, la_k = (tid % 4) * 4;
        const int lb_k = tid / 16, lb_n = (tid % 16) * 4;

        float4 ra[4], rb[4];
        auto load_tile = [&](int kt) {
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
                    for (int q = 0; q < 4; ++q) v[q] = (m < p.M && k + q < p.K) ? __ldg(src + q) : O::zero();
                    ra[r] = make_float4(v[0], v[1], v[2], v[3]);
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int k = k0 + lb_k + 4 * r, n = n0 + lb_n;
                const float* src = B + (int64_t)k * p.sBk + n;
                if (k < p.K && n + 3 < p.N && p.vecB) {
                    rb[r] = __ldg(reinterpret_cast<const float4*>(src));
                } else {
                    float v[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) v[q] = (k < p.K && n + q < p.N) ? __ldg(src + q) : O::bpad();
                    rb[r] = make_float4(v[0], v[1], v[2], v[3]);
                }
            }
        };
        auto store_tile = [&](int buf) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int m = la_m + 16 * r;
                As[buf][la_k + 0][m] = make_float2(ra[r].x, ra[r].x);
                As[buf][la_k + 1][m] = make_float2(ra[r].y, ra[r].y);
                As[buf][la_k + 2][m] = make_float2(ra[r].z, ra[r].z);
                As[buf][la_k + 3][m] = make_float2(ra[r].w, ra[r].w);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) *reinterpret_cast<float4*>(&Bs[buf][lb_k + 4 * r][lb_n]) = rb[r];
        };

        float best[TM][TN];
        float snap[ARG ? TM : 1][ARG ? TN : 1];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) best[i][j] = O::zero();
        if (ARG) {
#pragma unroll
            for (int q = 0; q < TM * TN; ++q) sid[q][tid] = 0;
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) snap[ARG ? i : 0][ARG ? j : 0] = O::zero();
        }

        load_tile(0);
        store_tile(0);
        __syncthreads();
        for (int kt = 0; kt < nkt; ++kt) {
            const int buf = kt & 1;
            if (kt + 1 < nkt) load_tile(kt + 1);
#pragma unroll
            for (int kk = 0; kk < BK; kk += 2) {
                float2 a0[TM], a1[TM];
                float2 b0[TN / 2], b1[TN / 2];
                {
                    const float4* pa0 = reinterpret_cast<const float4*>(&As[buf][kk][tm * 4]);
                    const float4* pa0h = reinterpret_cast<const float4*>(&As[buf][kk][BM / 2 + tm * 4]);
                    const float4* pa1 = reinterpret_cast<const float4*>(&As[buf][kk + 1][tm * 4]);
                    const float4* pa1h = reinterpret_cast<const float4*>(&As[buf][kk + 1][BM / 2 + tm * 4]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float4 x = pa0[h], y = pa0h[h], z = pa1[h], w = pa1h[h];
                        a0[2 * h] = make_float2(x.x, x.y);
                        a0[2 * h + 1] = make_float2(x.z, x.w);
                        a0[4 + 2 * h] = make_float2(y.x, y.y);
                        a0[4 + 2 * h + 1] = make_float2(y.z, y.w);
                        a1[2 * h] = make_float2(z.x, z.y);
                        a1[2 * h + 1] = make_float2(z.z, z.w);
                        a1[4 + 2 * h] = make_float2(w.x, w.y);
                        a1[4 + 2 * h + 1] = make_float2(w.z, w.w);
                    }
                    float4 u = *reinterpret_cast<const float4*>(&Bs[buf][kk][tn * 4]);
                    float4 v = *reinterpret_cast<const float4*>(&Bs[buf][kk][BN / 2 + tn * 4]);
                    float4 s = *reinterpret_cast<const float4*>(&Bs[buf][kk + 1][tn * 4]);
                    float4 t = *reinterpret_cast<const float4*>(&Bs[buf][kk + 1][BN / 2 + tn * 4]);
                    b0[0] = make_float2(u.x, u.y);
                    b0[1] = make_float2(u.z, u.w);
                    b0[2] = make_float2(v.x, v.y);
                    b0[3] = make_float2(v.z, v.w);
                    b1[0] = make_float2(s.x, s.y);
                    b1[1] = make_float2(s.z, s.w);
                    b1[2] = make_float2(t.x, t.y);
                    b1[3] = make_float2(t.z, t.w);
                }
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int jp = 0; jp < TN / 2; ++jp) {
                        float2 t0 = O::mul2(a0[i], b0[jp]);
                        float2 t1 = O::mul2(a1[i], b1[jp]);
                        best[i][2 * jp] = O::fold3(best[i][2 * jp], t0.x, t1.x);
                        best[i][2 * jp + 1] = O::fold3(best[i][2 * jp + 1], t0.y, t1.y);
                    }
            }
            if (ARG) {
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) {
                        if (O::better(best[i][j], snap[ARG ? i : 0][ARG ? j : 0])) sid[i * TN + j][tid] = kt;
                        snap[ARG ? i : 0][ARG ? j : 0] = best[i][j];
                    }
            }
            if (kt + 1 < nkt) {
                __syncthreads();
                store_tile(buf ^ 1);
                __syncthreads();
            }
        }

        // ---------------- epilogue: resolve argmax inside the winning chunk, store
        const float zero = O::zero();
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int m = m0 + (i < 4 ? tm * 4 + i : BM / 2 + tm * 4 + (i - 4));
            if (m >= p.M) continue;
            float* crow = p.C + oc + (int64_t)m * p.sCm;
            int32_t* irow = ARG ? p.I + oi + (int64_t)m * p.sIm : nullptr;
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const int n = n0 + (j < 4 ? tn * 4 + j : BN / 2 + tn * 4 + (j - 4));
                if (n >= p.N) continue;
                const float v = best[i][j];
                crow[(int64_t)n * p.sCn] = v;
                if (ARG) {
                    int32_t idx = 0;
                    if (v != zero) {
                        const int k0 = sid[i * TN + j][tid] * BK;
                        const int k1 = min(k0 + BK, p.K);
                        const float* arow = A + (int64_t)m * p.sAm;
                        const float* bcol = B + n;
                        idx = k0;
                        for (int k = k0; k < k1; ++k) {
                            if (O::mul(__ldg(arow + k), __ldg(bcol + (int64_t)k * p.sBk)) == v) {
                                idx = k;
                                break;
                            }
                        }
                    }
                    irow[(int64_t)n * p.sIn] = idx;
                }
            }
        }
        __syncthreads();
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

template <int SR, bool ARG, int VEC>
__global__ void __launch_bounds__(256) k_gemm_stream(StreamParams p)
{
    using O = Ops<SR>;
    for (uint32_t e = blockIdx.x * blockDim.x + threadIdx.x; e < p.total; e += gridDim.x * blockDim.x) {
        const uint32_t b = fdiv(e, p.div_nvec);
        const int n = (int)(e - b * p.nvec) * VEC;
        int64_t oa, ob, oc, oi;
        batch_offsets(p.bt, b, oa, ob, oc, oi);
        float best[MAXM_STREAM][VEC];
        int32_t idx[MAXM_STREAM][VEC];
#pragma unroll
        for (int m = 0; m < MAXM_STREAM; ++m)
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
            for (int m = 0; m < MAXM_STREAM; ++m) {
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
        for (int m = 0; m < MAXM_STREAM; ++m) {
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
    for (int d = 0; d < p.bt.nb; ++d) {
        va = va && p.bt.sA[d] % 4 == 0;
        vb = vb && p.bt.sB[d] % 4 == 0;
    }
    p.vecA = va;
    p.vecB = vb;
    dim3 grid((unsigned)((g.N + BN - 1) / BN), (unsigned)((g.M + BM - 1) / BM),
              (unsigned)(nbatch < 65535 ? nbatch : 65535));
    k_gemm_tiled<SR, ARG><<<grid, TTHREADS, 0, s>>>(p);
    return check_launch("k_gemm_tiled");
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
    if (vec) k_gemm_stream<SR, ARG, 4><<<grid, 256, 0, s>>>(p);
    else k_gemm_stream<SR, ARG, 1><<<grid, 256, 0, s>>>(p);
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
    const bool big = g.M >= 16 && g.N >= 16 && g.K >= 8;
    if (fits32 && big) {
        if (g.sAk == 1 && g.sBn == 1) return R_TILED;
        if (g.sBk == 1 && g.sAm == 1) {
            swap = true;
            return R_TILED;
        }
    }
    if (fits32 && g.K <= 64) {
        if (g.M <= MAXM_STREAM && nbatch * ((g.N + 3) / 4) < (int64_t(1) << 31) && g.M <= g.N) return R_STREAM;
        if (g.N <= MAXM_STREAM && nbatch * ((g.M + 3) / 4) < (int64_t(1) << 31)) {
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
    const void* ks[] = {
        (const void*)k_gemm_tiled<TROP_MAXPLUS, true>,  (const void*)k_gemm_tiled<TROP_MINPLUS, true>,
        (const void*)k_gemm_tiled<TROP_MAXTIMES, true>, (const void*)k_gemm_tiled<TROP_MAXPLUS, false>,
        (const void*)k_gemm_stream<TROP_MAXPLUS, true, 4>, (const void*)k_gemm_stream<TROP_MAXPLUS, true, 1>,
        (const void*)k_gemm_generic<TROP_MAXPLUS, true>,
    };
    for (const void* k : ks) {
        cudaError_t e = cudaFuncGetAttributes(&a, k);
        if (e != cudaSuccess) return cuda_error(e, "cudaFuncGetAttributes (gemm kernels)");
    }
    return TROP_OK;
}

}  // namespace trop
