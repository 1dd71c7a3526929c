/*
 * oracle.c -- plain, slow, obviously-correct CPU definitions of the tropical
 * einsum hot path.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the bench's
 * CPU-baseline leg load this code; the library under test never does.  It
 * shares no source, header, table or helper with the CUDA path.
 *
 * What is defined here, and where the definition comes from:
 *
 *  - oracle_einsum: the tropical einsum of one or two strided operands.
 *      * tropical-gemm PR #35 "batched GPU ops with DLPack zero-copy output",
 *        Summary / key changes: batched f32 max-plus, min-plus and max-times
 *        (maxmul) kernels that also return an argmax.
 *      * omeinsum-rs issue #52 "GPU tropical path: keep tensors
 *        device-resident + device-side permute", section "Resolved design for
 *        step 3": kernel (a), the N-d permute / strided gather, and kernel
 *        (b), the diagonal/trace gather fused with the tropical max/min
 *        reduce (repeated labels, labels absent from the output).
 *    The definition is the direct one: for every output element, walk the
 *    contracted assignments in row-major order (labels ordered by first
 *    appearance in the first operand) and keep the running result with a
 *    STRICT comparison, so the argmax is the smallest contracted linear
 *    index that reaches the result.  Each tropical product rounds once in
 *    IEEE binary32 (the pages' kernels are the _f32 ones); max/min are exact.
 *    Semiring table (the pages name the three semirings but not their
 *    neutral elements; the usual tropical definitions are taken):
 *        max-plus : (+) = max, (x) = +, zero = -inf
 *        min-plus : (+) = min, (x) = +, zero = +inf
 *        max-times: (+) = max, (x) = *, zero = 0   (nonnegative domain)
 *    Integer operands (i32 / i64) take the same definition in exact integer
 *    arithmetic: each tropical product a + b (or a * b) is the exact integer,
 *    computed here in a wider type, and the inputs must make every product
 *    that is formed fit the operand type -- the pages fix no overflow policy
 *    for integer contractions, and this precondition is the reading taken (a
 *    product outside the type makes the oracle refuse the input with
 *    E_OVERFLOW instead of guessing).  The zero is the type's min / max / 0;
 *    it is only ever the start of the running (+), never an operand value.
 *    f64 (unary and pairwise) is the same definition in binary64: the
 *    tropical-gemm PR #35 "CPU Dtype Handling" commit supports f32 and f64
 *    ("no more silent precision loss"); each product rounds once in binary64.
 *
 *  - oracle_gemm_backward: the gradient of the batched tropical GEMM with
 *    respect to A and B, given dC and the forward argmax ("winner routing").
 *      * omeinsum-rs issue #52, "Acceptance criteria": forward, backward and
 *        argmax must stay consistent with the CPU path.
 *      * tropical-gemm PR #35, review of python/tropical_gemm/pytorch.py: the
 *        batched autograd functions route the gradient through the argmax
 *        with scatter_add.
 *      * rustytorch commit "ops::index": scatter-add walks the adjoint of the
 *        selection, deterministic with duplicate indices.
 *    Each output (b,m,n) sends dC[b,m,n] to k = I[b,m,n]:
 *        dA[b,m,k] += dC[b,m,n]            dB[b,k,n] += dC[b,m,n]
 *    for max-plus / min-plus, where d(a+b)/da = d(a+b)/db = 1, and
 *        dA[b,m,k] += dC[b,m,n] * B[b,k,n] dB[b,k,n] += dC[b,m,n] * A[b,m,k]
 *    for max-times.  Every output routes to its argmax, including the
 *    convention 0 when nothing beat the zero; an index outside [0,K) routes
 *    nowhere.  The sums run in increasing n (dA) and increasing m (dB), each
 *    product and each addition rounding once in binary32.
 *
 *  - oracle_ising_ground / oracle_ising_brute / oracle_ising_energy: the
 *    spin-glass workload that the contraction-tree executor is measured on.
 *    The pages do not describe it; the elimination order (row-major, one
 *    site at a time, max over the spin that leaves the frontier) and the tie
 *    rule (smallest index) are the readings the library is built to.
 *
 * Parallelism: output elements are independent, so an OpenMP loop over them
 * (or over the states of one elimination step) changes nothing in how any
 * single result is computed.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math [-fopenmp] -shared -fPIC.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { SR_MAXPLUS = 0, SR_MINPLUS = 1, SR_MAXTIMES = 2 };
enum { DT_F32 = 0, DT_I32 = 1, DT_I64 = 2, DT_F64 = 3 };
enum { OK = 0, E_ARG = -1, E_SHAPE = -2, E_DTYPE = -3, E_NOMEM = -4, E_OVERFLOW = -5 };

#define MAXLAB 64

/* ------------------------------------------------------------------------ */
/* semiring scalars                                                          */

static float f32_zero(int sr)
{
    if (sr == SR_MAXPLUS) return -INFINITY;
    if (sr == SR_MINPLUS) return INFINITY;
    return 0.0f;
}

static float f32_otimes(int sr, float a, float b)
{
    /* one binary32 operation: built with -ffp-contract=off, no fast-math */
    return sr == SR_MAXTIMES ? a * b : a + b;
}

static int f32_better(int sr, float t, float best)
{
    return sr == SR_MINPLUS ? (t < best) : (t > best);
}

static double f64_zero(int sr)
{
    if (sr == SR_MAXPLUS) return -INFINITY;
    if (sr == SR_MINPLUS) return INFINITY;
    return 0.0;
}

static double f64_otimes(int sr, double a, double b)
{
    /* one binary64 operation */
    return sr == SR_MAXTIMES ? a * b : a + b;
}

static int f64_better(int sr, double t, double best)
{
    return sr == SR_MINPLUS ? (t < best) : (t > best);
}

static int64_t i64_zero(int sr, int dtype)
{
    if (sr == SR_MAXTIMES) return 0;
    if (dtype == DT_I32) return sr == SR_MAXPLUS ? (int64_t)INT32_MIN : (int64_t)INT32_MAX;
    return sr == SR_MAXPLUS ? INT64_MIN : INT64_MAX;
}

static int i64_better(int sr, int64_t t, int64_t best)
{
    return sr == SR_MINPLUS ? (t < best) : (t > best);
}

/* exact integer tropical product; *fits = 0 when it lies outside the operand type */
static int64_t int_otimes(int sr, int dtype, int64_t a, int64_t b, int* fits)
{
    const __int128 p = sr == SR_MAXTIMES ? (__int128)a * (__int128)b : (__int128)a + (__int128)b;
    const __int128 lo = dtype == DT_I32 ? (__int128)INT32_MIN : (__int128)INT64_MIN;
    const __int128 hi = dtype == DT_I32 ? (__int128)INT32_MAX : (__int128)INT64_MAX;
    *fits = p >= lo && p <= hi;
    return (int64_t)p;
}

static int64_t int_load(int dtype, const void* base, int64_t off)
{
    return dtype == DT_I32 ? (int64_t)((const int32_t*)base)[off] : ((const int64_t*)base)[off];
}

/* ------------------------------------------------------------------------ */
/* label bookkeeping                                                         */

typedef struct {
    int n;                      /* number of distinct labels */
    int32_t name[3 * MAXLAB];
    int64_t size[3 * MAXLAB];
} labels_t;

static int label_id(labels_t* t, int32_t name, int64_t size, int add)
{
    for (int i = 0; i < t->n; ++i)
        if (t->name[i] == name) {
            if (size >= 0 && t->size[i] != size) return E_SHAPE;
            return i;
        }
    if (!add) return E_ARG;
    t->name[t->n] = name;
    t->size[t->n] = size;
    return t->n++;
}

/* advance an odometer over labels ids[0..n-1] (last fastest); 0 when done */
static int odometer_next(const int* ids, int n, const int64_t* size, int64_t* val)
{
    for (int i = n - 1; i >= 0; --i) {
        if (++val[ids[i]] < size[ids[i]]) return 1;
        val[ids[i]] = 0;
    }
    return 0;
}

static int64_t count_of(const int* ids, int n, const int64_t* size)
{
    int64_t c = 1;
    for (int i = 0; i < n; ++i) c *= size[ids[i]];
    return c;
}

static int64_t offset_of(int n, const int* ids, const int64_t* stride, const int64_t* val)
{
    int64_t off = 0;
    for (int i = 0; i < n; ++i) off += val[ids[i]] * stride[i];
    return off;
}

/*
 * oracle_einsum
 *   sr         semiring
 *   dtype      element type of A, B and out (f32, i32, i64 or f64)
 *   nA, labA, shA, stA, A   first operand: rank, label per axis, extents,
 *                           strides in elements, base pointer
 *   nB < 0  -> unary (B ignored); otherwise the second operand likewise
 *   nO, labO   output labels; out is contiguous row-major in that order
 *   argmax     nullable; int32 per output element
 *   samples    nullable; if given, only the output linear indices samples[s]
 *              are computed, and written to out[s] / argmax[s]
 *   nthreads   OpenMP threads (<= 0: library default)
 *
 * Pairwise:  out[o] = (+) over all assignments of the non-output labels of
 *            A[..] (x) B[..].  Contracted labels (in A and B, not in out)
 *            ordered by first appearance in A give the argmax index k; labels
 *            in only one operand and not in out are folded into v_k first.
 * Unary:     out[o] = (+) over the labels absent from out (order of first
 *            appearance in A), argmax = that linear index.  No such label ->
 *            a permute / diagonal gather.
 */
int oracle_einsum(int sr, int dtype,
                  int nA, const int32_t* labA, const int64_t* shA, const int64_t* stA, const void* A,
                  int nB, const int32_t* labB, const int64_t* shB, const int64_t* stB, const void* B,
                  int nO, const int32_t* labO, void* out, int32_t* argmax,
                  const int64_t* samples, int64_t nsamples, int nthreads)
{
    if (sr < 0 || sr > 2 || nA < 0 || nA > MAXLAB || nO < 0 || nO > MAXLAB || nB > MAXLAB) return E_ARG;
    if (dtype < 0 || dtype > 3) return E_DTYPE;
    const int pairwise = nB >= 0;

    labels_t t;
    t.n = 0;
    int idA[MAXLAB], idB[MAXLAB], idO[MAXLAB];
    for (int i = 0; i < nA; ++i) {
        if (shA[i] < 0) return E_SHAPE;
        if ((idA[i] = label_id(&t, labA[i], shA[i], 1)) < 0) return idA[i];
    }
    for (int i = 0; pairwise && i < nB; ++i) {
        if (shB[i] < 0) return E_SHAPE;
        if ((idB[i] = label_id(&t, labB[i], shB[i], 1)) < 0) return idB[i];
    }
    for (int i = 0; i < nO; ++i) {
        if ((idO[i] = label_id(&t, labO[i], -1, 0)) < 0) return E_ARG; /* output label unknown */
        for (int j = 0; j < i; ++j)
            if (idO[j] == idO[i]) return E_ARG;                          /* repeated output label */
    }

    int inA[3 * MAXLAB] = {0}, inB[3 * MAXLAB] = {0}, inO[3 * MAXLAB] = {0};
    for (int i = 0; i < nA; ++i) inA[idA[i]] = 1;
    for (int i = 0; pairwise && i < nB; ++i) inB[idB[i]] = 1;
    for (int i = 0; i < nO; ++i) inO[idO[i]] = 1;

    /* argmax labels K (first appearance in A) and the one-operand labels R */
    int K[3 * MAXLAB], nK = 0, R[3 * MAXLAB], nR = 0;
    int seen[3 * MAXLAB] = {0};
    for (int i = 0; i < nA; ++i) {
        int l = idA[i];
        if (seen[l] || inO[l]) continue;
        seen[l] = 1;
        if (!pairwise || inB[l]) K[nK++] = l; else R[nR++] = l;
    }
    for (int i = 0; pairwise && i < nB; ++i) {
        int l = idB[i];
        if (seen[l] || inO[l]) continue;
        seen[l] = 1;
        R[nR++] = l; /* in B only */
    }

    const int64_t total = count_of(idO, nO, t.size);
    const int64_t nwork = samples ? nsamples : total;
    const int64_t nK_assign = count_of(K, nK, t.size);
    const int64_t nR_assign = count_of(R, nR, t.size);
    for (int64_t s = 0; samples && s < nsamples; ++s)
        if (samples[s] < 0 || samples[s] >= total) return E_ARG;
    int overflow = 0; /* an integer product outside the operand type was formed */

#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 256)
#endif
    for (int64_t w = 0; w < nwork; ++w) {
        int64_t val[3 * MAXLAB] = {0};
        int64_t o = samples ? samples[w] : w;
        for (int i = nO - 1; i >= 0; --i) {
            int64_t sz = t.size[idO[i]];
            val[idO[i]] = o % sz;
            o /= sz;
        }
        int32_t idx = 0;
        if (dtype == DT_F32) {
            float best = f32_zero(sr);
            int64_t k = 0;
            if (nK_assign > 0) {
                for (int i = 0; i < nK; ++i) val[K[i]] = 0;
                do {
                    float v;
                    if (!pairwise) {
                        v = ((const float*)A)[offset_of(nA, idA, stA, val)];
                    } else {
                        v = f32_zero(sr);
                        if (nR_assign > 0) {
                            for (int i = 0; i < nR; ++i) val[R[i]] = 0;
                            do {
                                float a = ((const float*)A)[offset_of(nA, idA, stA, val)];
                                float b = ((const float*)B)[offset_of(nB, idB, stB, val)];
                                float p = f32_otimes(sr, a, b);
                                if (f32_better(sr, p, v)) v = p;
                            } while (odometer_next(R, nR, t.size, val));
                        }
                    }
                    if (f32_better(sr, v, best)) { best = v; idx = (int32_t)k; }
                    ++k;
                } while (odometer_next(K, nK, t.size, val));
            }
            ((float*)out)[w] = best;
        } else if (dtype == DT_F64) {
            double best = f64_zero(sr);
            int64_t k = 0;
            if (nK_assign > 0) {
                for (int i = 0; i < nK; ++i) val[K[i]] = 0;
                do {
                    double v;
                    if (!pairwise) {
                        v = ((const double*)A)[offset_of(nA, idA, stA, val)];
                    } else {
                        v = f64_zero(sr);
                        if (nR_assign > 0) {
                            for (int i = 0; i < nR; ++i) val[R[i]] = 0;
                            do {
                                double a = ((const double*)A)[offset_of(nA, idA, stA, val)];
                                double b = ((const double*)B)[offset_of(nB, idB, stB, val)];
                                double p = f64_otimes(sr, a, b);
                                if (f64_better(sr, p, v)) v = p;
                            } while (odometer_next(R, nR, t.size, val));
                        }
                    }
                    if (f64_better(sr, v, best)) { best = v; idx = (int32_t)k; }
                    ++k;
                } while (odometer_next(K, nK, t.size, val));
            }
            ((double*)out)[w] = best;
        } else {
            int64_t best = i64_zero(sr, dtype);
            int64_t k = 0;
            if (nK_assign > 0) {
                for (int i = 0; i < nK; ++i) val[K[i]] = 0;
                do {
                    int64_t v;
                    if (!pairwise) {
                        v = int_load(dtype, A, offset_of(nA, idA, stA, val));
                    } else {
                        v = i64_zero(sr, dtype);
                        if (nR_assign > 0) {
                            for (int i = 0; i < nR; ++i) val[R[i]] = 0;
                            do {
                                const int64_t a = int_load(dtype, A, offset_of(nA, idA, stA, val));
                                const int64_t b = int_load(dtype, B, offset_of(nB, idB, stB, val));
                                int fits;
                                const int64_t p = int_otimes(sr, dtype, a, b, &fits);
                                if (!fits) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                                    overflow = 1;
                                }
                                if (i64_better(sr, p, v)) v = p;
                            } while (odometer_next(R, nR, t.size, val));
                        }
                    }
                    if (i64_better(sr, v, best)) { best = v; idx = (int32_t)k; }
                    ++k;
                } while (odometer_next(K, nK, t.size, val));
            }
            if (dtype == DT_I32) ((int32_t*)out)[w] = (int32_t)best;
            else ((int64_t*)out)[w] = best;
        }
        if (argmax) argmax[w] = idx;
    }
    return overflow ? E_OVERFLOW : OK;
}

/* ------------------------------------------------------------------------ */
/* 2-D Edwards-Anderson spin glass, open boundary, zero field.
 * Spin x in {0,1} <-> s = 2x - 1.  Jh[r*(C-1)+c] couples (r,c)-(r,c+1),
 * Jv[r*C+c] couples (r,c)-(r+1,c).  W = max over spins of sum J s_i s_j;
 * the ground energy of H = -sum J s_i s_j is E0 = -W.                       */

/* Gradient of C = A (x) B (batched tropical GEMM) with respect to A and B
 * given dC and the forward argmax I (see the file header).  Strides in
 * elements; dA / dB may be NULL (not wanted); A / B are read only for
 * max-times.  Returns 0. */
int oracle_gemm_backward(int sr, int64_t batch, int64_t M, int64_t N, int64_t K,
                         const float* A, int64_t sAb, int64_t sAm, int64_t sAk,
                         const float* B, int64_t sBb, int64_t sBk, int64_t sBn,
                         const float* dC, int64_t sCb, int64_t sCm, int64_t sCn,
                         const int32_t* I, int64_t sIb, int64_t sIm, int64_t sIn,
                         float* dA, int64_t sdAb, int64_t sdAm, int64_t sdAk,
                         float* dB, int64_t sdBb, int64_t sdBk, int64_t sdBn)
{
    if (dA) {
        for (int64_t b = 0; b < batch; ++b)
            for (int64_t m = 0; m < M; ++m) {
                for (int64_t k = 0; k < K; ++k) dA[b * sdAb + m * sdAm + k * sdAk] = 0.0f;
                for (int64_t n = 0; n < N; ++n) {
                    int64_t k = I[b * sIb + m * sIm + n * sIn];
                    if (k < 0 || k >= K) continue;
                    float g = dC[b * sCb + m * sCm + n * sCn];
                    if (sr == SR_MAXTIMES) g = g * B[b * sBb + k * sBk + n * sBn];
                    float* t = &dA[b * sdAb + m * sdAm + k * sdAk];
                    *t = *t + g;
                }
            }
    }
    if (dB) {
        for (int64_t b = 0; b < batch; ++b)
            for (int64_t n = 0; n < N; ++n) {
                for (int64_t k = 0; k < K; ++k) dB[b * sdBb + k * sdBk + n * sdBn] = 0.0f;
                for (int64_t m = 0; m < M; ++m) {
                    int64_t k = I[b * sIb + m * sIm + n * sIn];
                    if (k < 0 || k >= K) continue;
                    float g = dC[b * sCb + m * sCm + n * sCn];
                    if (sr == SR_MAXTIMES) g = g * A[b * sAb + m * sAm + k * sAk];
                    float* t = &dB[b * sdBb + k * sdBk + n * sdBn];
                    *t = *t + g;
                }
            }
    }
    return 0;
}

static int spin_of(int x) { return 2 * x - 1; }

/* H(s) for spins given as +-1, row-major */
int64_t oracle_ising_energy(int R, int C, const int8_t* Jh, const int8_t* Jv, const int8_t* s)
{
    int64_t w = 0;
    for (int r = 0; r < R; ++r)
        for (int c = 0; c + 1 < C; ++c) w += (int64_t)Jh[r * (C - 1) + c] * s[r * C + c] * s[r * C + c + 1];
    for (int r = 0; r + 1 < R; ++r)
        for (int c = 0; c < C; ++c) w += (int64_t)Jv[r * C + c] * s[r * C + c] * s[(r + 1) * C + c];
    return -w;
}

/* exhaustive maximum over all 2^(R*C) configurations (R*C <= 30) */
int oracle_ising_brute(int R, int C, const int8_t* Jh, const int8_t* Jv, int64_t* W, int8_t* spins)
{
    const int n = R * C;
    if (R < 1 || C < 1 || n > 30) return E_ARG;
    int8_t* s = (int8_t*)malloc((size_t)n);
    if (!s) return E_NOMEM;
    int64_t best = INT64_MIN;
    for (int64_t cfg = 0; cfg < ((int64_t)1 << n); ++cfg) {
        for (int i = 0; i < n; ++i) s[i] = (int8_t)spin_of((int)((cfg >> i) & 1));
        int64_t w = -oracle_ising_energy(R, C, Jh, Jv, s);
        if (w > best) { best = w; memcpy(spins, s, (size_t)n); }
    }
    free(s);
    *W = best;
    return OK;
}

/*
 * Site-by-site max-plus elimination (row-major).  The frontier holds one spin
 * per column; column j is bit (C-1-j) of the state index (column 0 most
 * significant), i.e. the row-major linear index of the frontier tensor.
 *
 * Row 0 grows the frontier: the first state is the bond (0,0)-(0,1); each
 * further site of row 0 appends its spin and adds the bond to its left
 * neighbour.  Each site (r,c), r >= 1, replaces the spin u = (r-1,c) in
 * column c by n = (r,c):
 *     S'[.., n, ..] = max_u S[.., u, ..] + Jv s_u s_n + Jh s_l s_n
 * (the left term only for c >= 1, l = (r,c-1)), keeping the smallest u that
 * reaches the maximum as a 1-bit back-pointer.  The end is the maximum over
 * the last frontier, at its smallest maximising index.  Back-tracking walks
 * the back-pointers in reverse.
 */
int oracle_ising_ground(int R, int C, const int8_t* Jh, const int8_t* Jv,
                        int64_t* W, int8_t* spins, int nthreads)
{
    if (R < 2 || C < 2 || C > 30) return E_ARG;
    const int64_t NS = (int64_t)1 << C;
    int32_t* S = (int32_t*)malloc(sizeof(int32_t) * (size_t)NS);
    int32_t* T = (int32_t*)malloc(sizeof(int32_t) * (size_t)NS);
    const int64_t nsteps = (int64_t)(R - 1) * C;
    const int64_t bp_bytes = (NS + 7) / 8;
    uint8_t* bp = (uint8_t*)calloc((size_t)(nsteps * bp_bytes), 1);
    if (!S || !T || !bp) { free(S); free(T); free(bp); return E_NOMEM; }
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
    (void)nthreads;
#endif

    /* row 0 */
    for (int64_t i = 0; i < 4; ++i)
        S[i] = Jh[0] * spin_of((int)(i >> 1)) * spin_of((int)(i & 1));
    for (int c = 2; c < C; ++c) {
        const int64_t n_old = (int64_t)1 << c;
        const int J = Jh[c - 1];
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads) schedule(static)
#endif
        for (int64_t i = 0; i < n_old; ++i)
            for (int n = 0; n < 2; ++n)
                T[2 * i + n] = S[i] + J * spin_of((int)(i & 1)) * spin_of(n);
        int32_t* tmp = S; S = T; T = tmp;
    }

    /* rows 1 .. R-1 */
    for (int r = 1; r < R; ++r) {
        for (int c = 0; c < C; ++c) {
            const int bit = C - 1 - c;
            const int Jup = Jv[(r - 1) * C + c];
            const int Jleft = c >= 1 ? Jh[r * (C - 1) + c - 1] : 0;
            uint8_t* b = bp + ((int64_t)(r - 1) * C + c) * bp_bytes;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads) schedule(static)
#endif
            for (int64_t j8 = 0; j8 < NS; j8 += 8) {   /* 8 states per back-pointer byte */
                uint8_t byte = 0;
                for (int64_t i = j8; i < j8 + 8 && i < NS; ++i) {
                    const int n = (int)((i >> bit) & 1);
                    const int l = c >= 1 ? (int)((i >> (bit + 1)) & 1) : 0;
                    int32_t best = 0;
                    int arg = 0;
                    for (int u = 0; u < 2; ++u) {
                        const int64_t src = (i & ~((int64_t)1 << bit)) | ((int64_t)u << bit);
                        int32_t v = S[src] + Jup * spin_of(u) * spin_of(n);
                        if (c >= 1) v += Jleft * spin_of(l) * spin_of(n);
                        if (u == 0 || v > best) { best = v; arg = u; }
                    }
                    T[i] = best;
                    if (arg) byte |= (uint8_t)(1u << (i - j8));
                }
                b[j8 / 8] = byte;
            }
            int32_t* tmp = S; S = T; T = tmp;
        }
    }

    /* final maximum, smallest index */
    int64_t arg = 0;
    int32_t best = S[0];
    for (int64_t i = 1; i < NS; ++i)
        if (S[i] > best) { best = S[i]; arg = i; }
    *W = best;

    /* back-track */
    int64_t i = arg;
    for (int c = 0; c < C; ++c) spins[(R - 1) * C + c] = (int8_t)spin_of((int)((i >> (C - 1 - c)) & 1));
    for (int r = R - 1; r >= 1; --r) {
        for (int c = C - 1; c >= 0; --c) {
            const int bit = C - 1 - c;
            const uint8_t* b = bp + ((int64_t)(r - 1) * C + c) * bp_bytes;
            const int u = (b[i / 8] >> (i % 8)) & 1;
            spins[(r - 1) * C + c] = (int8_t)spin_of(u);
            i = (i & ~((int64_t)1 << bit)) | ((int64_t)u << bit);
        }
    }
    free(S); free(T); free(bp);
    return OK;
}

int oracle_abi_version(void) { return 1; }
