// backward.cu -- gradient of the strided-batched tropical GEMM, routed through
// the forward argmax ("winner routing").
//
// dA[b,m,k] = sum over n (increasing) with I[b,m,n] == k of g,
// dB[b,k,n] = sum over m (increasing) with I[b,m,n] == k of g,
// g = dC (max-plus, min-plus) or dC times the other operand (max-times).
// (omeinsum-rs issue #52 "Acceptance criteria": forward, backward and argmax
// consistent with the CPU path; tropical-gemm PR #35: the batched autograd
// functions send the gradient through the argmax with a scatter-add; the
// rustytorch commit's ops::index: a scatter-add over the adjoint of the
// selection, deterministic with duplicate indices and free of atomics.)
//
// The adjoint needs no sort: each output line (a row of dA, a column of dB) is
// walked in increasing step order, and every bin of it has one writer adding in
// that order, so every sum is the sequential one, bit for bit.
//   k_route_lane   max-plus and min-plus, both gradients in one launch
//                  (blockIdx.y): one lane per line with all of the line's bins
//                  in shared memory; rows of dA by 16-byte vector loads along
//                  the line, columns of dB by one load per step (consecutive
//                  lanes, consecutive columns: 128 contiguous bytes a step).
//                  Also max-times dB when dA is not wanted, the other
//                  operand's factors gathered a ring turn ahead.
//   k_route_match  max-times: a warp per line, the lanes of one bin applied in
//                  step order, which keeps the gathers of the other operand in
//                  flight across a whole warp; dA and dB in two launches that
//                  overlap.
// Longer contractions repeat the walk per 256-bin span.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <type_traits>

#define TROP_TU 5  // this file's id in a bounds-violation record
#include "internal.h"

namespace trop {
namespace {

// One gradient: owners (b, x), x < X, each walking s < S.
//   index and dC of (b, x, s):     I[b*sIb + x*sIx + s*sIs], G[b*sGb + x*sGx + s*sGs]
//   other operand of (b, k, s):    P[b*sPb + k*sPk + s*sPs]        (max-times)
//   gradient element (b, x, k):    O[b*sOb + x*sOx + k*sOk]
struct RouteJob {
    int64_t X, S;
    const int32_t* I;
    int64_t sIb, sIx, sIs;
    const float* G;
    int64_t sGb, sGx, sGs;
    const float* P;
    int64_t sPb, sPk, sPs;
    float* O;
    int64_t sOb, sOx, sOk;
    int vec;  // k_route_lane: the line's steps are contiguous and 16-byte aligned (vector loads)
#if TROP_DEBUG_BOUNDS
    Span sp[4];  // I, G, P, O
#endif
};

// checked global accesses of job j (plain accesses in the normal build): tensor k of
// RouteJob::sp must hold `bytes` at ptr
#define R_IN(ptr, bytes, k) TROP_IN(ptr, bytes, j.sp[k])

struct RouteParams {
    int64_t nbatch, K;
    RouteJob job[2];
    int njobs;
    // 0: wait for the grid before this one at the start (it may have signalled before its own
    // results were complete); 1: the grid before is the other gradient's k_route_match of the
    // same call, which signals only after its own wait, so the inputs are complete -- wait at the
    // end instead, so that this grid completes only after that one
    int late_wait;
};


// One lane per output line with all of the line's bins in shared memory, [bin][lane] (no bank
// conflicts whatever the bins); both gradients in one launch, the job picked by blockIdx.y.  A
// lane reads its own line 8 steps at a time through a ring of RT_RING register sets (the loads
// of the next three chunks in flight while a chunk is applied): when the line's steps are
// contiguous and 16-byte aligned (RouteJob::vec, the rows of dA) by 16-byte vectors, one full
// 32-byte sector per array, otherwise one load per step through the step strides (the columns
// of dB: consecutive lanes are consecutive columns, so a warp reads 128 contiguous bytes a
// step).  Steps are applied four at a time: the four bins are read together, and a step whose
// bin an earlier step of the group also hit continues from that step's new value, so every bin
// still adds its terms in increasing step order.  The term is dC itself (max-plus, min-plus) or,
// with MUL (max-times), dC times the other operand's entry at the step's winner, rounded once;
// those factors are gathered for the next chunk while a chunk is applied.
constexpr int RT_SPAN = 256;  // bins a lane holds per walk (longer contractions: one walk per span)
constexpr int RT_STEP = 8;    // steps per chunk
constexpr int RT_RING = 4;    // chunks in registers: one applied, three in flight
// [span][32] bins, rounded up to whole 32-row blocks, plus one row: the transposed copy of the
// last block (33-float rows) reaches one row past it
size_t lane_smem(int64_t K)
{
    const size_t rows = ((size_t)std::min<int64_t>(K, RT_SPAN) + 31) / 32 * 32 + 1;
    return sizeof(float) * rows * 32;
}
// lines k_route_lane reads by vectors: unit step stride and 16-byte aligned lines
bool lane_ok(const RouteJob& j)
{
    return j.sIs == 1 && j.sGs == 1 && j.sIx % 4 == 0 && j.sGx % 4 == 0 && j.sIb % 4 == 0 && j.sGb % 4 == 0 &&
           ((uintptr_t)j.I % 16) == 0 && ((uintptr_t)j.G % 16) == 0;
}

template <bool MUL>
__global__ void __launch_bounds__(32) k_route_lane(RouteParams p)
{
    extern __shared__ __align__(16) float bins[];  // [span][32]: bin k of lane l at k * 32 + l
    if (!p.late_wait) pdl_wait();
    pdl_signal();
    if ((int)blockIdx.y >= p.njobs) {
        if (p.late_wait) pdl_wait();
        return;
    }
    // the job's fields in registers (the job is picked by blockIdx.y)
    const RouteJob& jr = p.job[blockIdx.y];
    const int vec = jr.vec;
    const int64_t S = jr.S, X = jr.X, K = p.K;
    const int64_t sIs = jr.sIs, sGs = jr.sGs, sOk = jr.sOk;
    const int32_t* const I0 = jr.I;
    const float* const G0 = jr.G;
    const float* const P0 = jr.P;
    const int64_t sPb = jr.sPb, sPk = jr.sPk, sPs = jr.sPs;
    float* const O0 = jr.O;
    const int64_t sIb = jr.sIb, sIx = jr.sIx, sGb = jr.sGb, sGx = jr.sGx, sOb = jr.sOb, sOx = jr.sOx;
#if TROP_DEBUG_BOUNDS
    const RouteJob& j = jr;  // the spans the checks read
#endif
    const int l = threadIdx.x;
    const int64_t lines = p.nbatch * X;
    for (int64_t base = (int64_t)blockIdx.x * 32; base < lines; base += (int64_t)gridDim.x * 32) {
        const int64_t o = base + l;
        const bool valid = o < lines;
        const int64_t b = valid ? o / X : 0, x = valid ? o - b * X : 0;
        const int32_t* Il = I0 + b * sIb + x * sIx;
        const float* Gl = G0 + b * sGb + x * sGx;
        const float* Pl = MUL ? P0 + b * sPb : nullptr;  // the other operand of this line's batch
        float* Ol = O0 + b * sOb + x * sOx;
        for (int64_t kc = 0; kc < K; kc += RT_SPAN) {
            const int kn = (int)min((int64_t)RT_SPAN, K - kc);
            for (int k = 0; k < kn; ++k) bins[k * 32 + l] = 0.0f;
            const int64_t nch = (S + RT_STEP - 1) / RT_STEP;
            int kr[RT_RING][RT_STEP];
            float gr[RT_RING][RT_STEP];
            float pr[2][RT_STEP];  // max-times: the factors of the chunk applied now and of the next
            auto load = [&](auto slot, int64_t c) {
                constexpr int R = decltype(slot)::value;
                const int64_t s0 = c * RT_STEP;
                if (vec && valid && s0 + RT_STEP <= S) {
                    const int4 kz = make_int4(-1, -1, -1, -1);
                    const float4 gz = make_float4(0.f, 0.f, 0.f, 0.f);
                    const int4 k0 = R_IN(Il + s0, 16, 0) ? __ldg(reinterpret_cast<const int4*>(Il + s0)) : kz;
                    const int4 k1 = R_IN(Il + s0 + 4, 16, 0) ? __ldg(reinterpret_cast<const int4*>(Il + s0 + 4)) : kz;
                    const float4 g0 = R_IN(Gl + s0, 16, 1) ? __ldg(reinterpret_cast<const float4*>(Gl + s0)) : gz;
                    const float4 g1 = R_IN(Gl + s0 + 4, 16, 1) ? __ldg(reinterpret_cast<const float4*>(Gl + s0 + 4)) : gz;
                    kr[R][0] = k0.x; kr[R][1] = k0.y; kr[R][2] = k0.z; kr[R][3] = k0.w;
                    kr[R][4] = k1.x; kr[R][5] = k1.y; kr[R][6] = k1.z; kr[R][7] = k1.w;
                    gr[R][0] = g0.x; gr[R][1] = g0.y; gr[R][2] = g0.z; gr[R][3] = g0.w;
                    gr[R][4] = g1.x; gr[R][5] = g1.y; gr[R][6] = g1.z; gr[R][7] = g1.w;
                } else {
                    // one load per step through the step strides (consecutive lines are consecutive
                    // lanes: the columns of dB read 128 contiguous bytes a step)
                    const int32_t* ip = Il + s0 * sIs;
                    const float* gp = Gl + s0 * sGs;
#pragma unroll
                    for (int t = 0; t < RT_STEP; ++t) {
                        const bool in = valid && c < nch && s0 + t < S;
                        kr[R][t] = in && R_IN(ip, 4, 0) ? __ldg(ip) : -1;
                        gr[R][t] = in && R_IN(gp, 4, 1) ? __ldg(gp) : 0.0f;
                        ip += sIs;
                        gp += sGs;
                    }
                }
            };
            // bin of a step relative to the span, -1 when it routes nowhere in this span (K < 2^31:
            // an index below the span, or negative, wraps to a large unsigned value)
            const unsigned kc32 = (unsigned)kc;
            auto rel = [&](int k) {
                const unsigned d = (unsigned)k - kc32;
                return d < (unsigned)kn ? (int)d : -1;
            };
            // max-times: the other operand's entry at each step's winner for chunk c (indices in ring
            // slot KS) into factor slot PS, issued a turn before the chunk is applied; a step that
            // routes nowhere in this span loads nothing
            auto gather = [&](auto kslot, auto pslot, int64_t c) {
                constexpr int KS = decltype(kslot)::value, PS = decltype(pslot)::value;
                const int64_t s0 = c * RT_STEP;
#pragma unroll
                for (int t = 0; t < RT_STEP; ++t) {
                    const int k = kr[KS][t];
                    const float* pp = Pl + (int64_t)k * sPk + (s0 + t) * sPs;
                    pr[PS][t] = rel(k) >= 0 && R_IN(pp, 4, 2) ? __ldg(pp) : 0.0f;
                }
            };
            auto apply = [&](auto slot, auto pslot) {
                constexpr int R = decltype(slot)::value, PS = decltype(pslot)::value;
                (void)PS;
#pragma unroll
                for (int q = 0; q < RT_STEP; q += 4) {
                    int d[4];
                    float g[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        d[t] = rel(kr[R][q + t]);
                        // max-times: the term is dC times the factor, rounded once before the add
                        g[t] = MUL ? __fmul_rn(gr[R][q + t], pr[PS][q + t]) : gr[R][q + t];
                    }
                    const float x0 = d[0] >= 0 ? bins[d[0] * 32 + l] : 0.0f;
                    const float x1 = d[1] >= 0 ? bins[d[1] * 32 + l] : 0.0f;
                    const float x2 = d[2] >= 0 ? bins[d[2] * 32 + l] : 0.0f;
                    const float x3 = d[3] >= 0 ? bins[d[3] * 32 + l] : 0.0f;
                    // each step continues from the latest earlier step of the group on its bin
                    const float y0 = __fadd_rn(x0, g[0]);
                    const float y1 = __fadd_rn(d[1] == d[0] ? y0 : x1, g[1]);
                    const float y2 = __fadd_rn(d[2] == d[1] ? y1 : d[2] == d[0] ? y0 : x2, g[2]);
                    const float y3 = __fadd_rn(d[3] == d[2] ? y2 : d[3] == d[1] ? y1 : d[3] == d[0] ? y0 : x3, g[3]);
                    if (d[0] >= 0) bins[d[0] * 32 + l] = y0;
                    if (d[1] >= 0) bins[d[1] * 32 + l] = y1;
                    if (d[2] >= 0) bins[d[2] * 32 + l] = y2;
                    if (d[3] >= 0) bins[d[3] * 32 + l] = y3;
                }
            };
            using I0 = std::integral_constant<int, 0>;
            using I1 = std::integral_constant<int, 1>;
            using I2 = std::integral_constant<int, 2>;
            using I3 = std::integral_constant<int, 3>;
            static_assert(RT_RING == 4, "the ring is unrolled for four slots");
            load(I0{}, 0);
            load(I1{}, 1);
            load(I2{}, 2);
            if constexpr (MUL) gather(I0{}, I0{}, 0);
            // one ring turn: chunk c in slot R (c = R mod 4, so its factors sit in slot R mod 2)
            auto turn = [&](auto slot, int64_t c) {
                constexpr int R = decltype(slot)::value;
                load(std::integral_constant<int, (R + 3) % 4>{}, c + 3);
                if constexpr (MUL)
                    gather(std::integral_constant<int, (R + 1) % 4>{}, std::integral_constant<int, (R + 1) % 2>{}, c + 1);
                apply(slot, std::integral_constant<int, R % 2>{});
            };
            for (int64_t c = 0; c < nch; c += 4) {
                turn(I0{}, c);
                if (c + 1 >= nch) break;
                turn(I1{}, c + 1);
                if (c + 2 >= nch) break;
                turn(I2{}, c + 2);
                if (c + 3 >= nch) break;
                turn(I3{}, c + 3);
            }
            __syncwarp();
            if (sOk == 1) {
                // bins contiguous in the gradient: 32 x 32 blocks transposed through a padded
                // copy so that each store writes 32 consecutive bins of one line; blocks go last
                // to first, so the copy's extra row lies in a block already written
                for (int kb = ((kn - 1) / 32) * 32; kb >= 0; kb -= 32) {
                    float r[32];
#pragma unroll
                    for (int t = 0; t < 32; ++t) r[t] = kb + t < kn ? bins[(kb + t) * 32 + l] : 0.0f;
                    __syncwarp();
                    float* tb = bins + kb * 32;  // [line][33]
#pragma unroll
                    for (int t = 0; t < 32; ++t) tb[l * 33 + t] = r[t];
                    __syncwarp();
                    for (int rr = 0; rr < 32; ++rr) {
                        float* Or = reinterpret_cast<float*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(Ol), rr));
                        if (base + rr < lines && kb + l < kn && R_IN(Or + kc + kb + l, 4, 3)) Or[kc + kb + l] = tb[rr * 33 + l];
                    }
                    __syncwarp();
                }
            } else if (valid) {
                float* op = Ol + kc * sOk;
                for (int k = 0; k < kn; ++k, op += sOk)
                    if (R_IN(op, 4, 3)) *op = bins[k * 32 + l];
            }
            __syncwarp();
        }
    }
}

// One warp per output line, RM_WARPS lines per CTA, each line's RM_SPAN bins in shared memory
// ([line][bin], rows padded to RM_LD).  A line's steps are taken RM_CHUNK at a time, every load
// of a chunk issued before any of it is used (a warp keeps 2 KB in flight, which the HBM latency
// needs): read directly into registers when a line's steps are contiguous (the rows of dA: lane
// i holds steps i, i + 32, ...), otherwise staged by the CTA through shared memory, loaded
// coalesced along the lines (the columns of dB).  Lane i of warp w then takes step s0 + i of
// line w, 32 steps at a time.  Lanes whose steps hit the same bin find each other with
// __match_any_sync; a lane's rank in its group (the lanes below it) is its place in step order,
// and the group's adds are applied rank by rank, so every bin still adds its terms in increasing
// step order with one rounding each -- the sequential sum, bit for bit, with 1 KB of bins per
// line.  Max-times multiplies each term by the other operand's entry at the winner first (a
// gather, issued for the whole chunk before the first term is applied).
#ifndef TROP_RM_WARPS
#define TROP_RM_WARPS 16
#endif
constexpr int RM_WARPS = TROP_RM_WARPS, RM_THREADS = RM_WARPS * 32;
constexpr int RM_SPAN = 256;                 // bins per line and walk
constexpr int RM_LD = RM_SPAN + 1;           // [line][bin] rows: the column-wise output read is conflict-free
constexpr int RM_CHUNK = 256;                // steps of a line loaded together
constexpr int RM_NB = RM_CHUNK / 32;         // batches per chunk
constexpr int RM_CLD = RM_CHUNK + 1;         // staged [line][step] rows
constexpr int RM_PER = RM_CHUNK / 32;        // staged elements per thread and array (RM_CHUNK x RM_WARPS / RM_THREADS)
constexpr size_t RM_SMEM =
    sizeof(float) * ((size_t)RM_WARPS * RM_LD + 2 * (size_t)RM_WARPS * RM_CLD) + 2 * RM_WARPS * sizeof(int64_t);
static_assert(RM_WARPS == 8 || RM_WARPS == 16 || RM_WARPS == 32, "lines per CTA");

template <bool MUL>
__global__ void __launch_bounds__(RM_THREADS) k_route_match(RouteParams p)
{
    extern __shared__ __align__(16) float sm_match[];
    if (!p.late_wait) pdl_wait();
    pdl_signal();
    if ((int)blockIdx.y >= p.njobs) {
        if (p.late_wait) pdl_wait();
        return;
    }
    // the job's fields in registers once (indexing the parameter block by blockIdx.y would
    // reload them from the constant bank at every use)
    const RouteJob j = blockIdx.y == 0 ? p.job[0] : p.job[1];
    const int64_t K = p.K, S = j.S, X = j.X;
    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    float* bins = sm_match;                                                        // [RM_WARPS][RM_LD]
    int* ck = reinterpret_cast<int*>(sm_match + RM_WARPS * RM_LD);                 // [RM_WARPS][RM_CLD]
    float* cg = sm_match + RM_WARPS * RM_LD + RM_WARPS * RM_CLD;                   // [RM_WARPS][RM_CLD]
    int64_t* line_i = reinterpret_cast<int64_t*>(sm_match + RM_WARPS * RM_LD + 2 * RM_WARPS * RM_CLD);
    int64_t* line_p = line_i + RM_WARPS;
    const int64_t lines = p.nbatch * X;
    const bool direct = j.sIs == 1 && j.sGs == 1;  // a line's steps are contiguous
    const unsigned lanes_below = (1u << l) - 1u;
    float* mybins = bins + w * RM_LD;
    for (int64_t base = (int64_t)blockIdx.x * RM_WARPS; base < lines; base += (int64_t)gridDim.x * RM_WARPS) {
        __syncthreads();  // the previous group's readers of the tables, stages and bins are done
        if (tid < RM_WARPS) {
            const int64_t o = base + tid;
            const int64_t b = o < lines ? o / X : 0, x = o < lines ? o - b * X : 0;
            line_i[tid] = o < lines ? b * j.sIb + x * j.sIx : -1;
            line_p[tid] = b * j.sPb;
        }
        __syncthreads();
        const int64_t my_off = line_i[w];
        const bool my_valid = my_off >= 0;
        const float* Pl = MUL ? j.P + line_p[w] : nullptr;
        for (int64_t kc = 0; kc < K; kc += RM_SPAN) {
            const int kn = (int)min((int64_t)RM_SPAN, K - kc);
            const int kc32 = (int)kc;
            __syncthreads();  // the previous span's output reads of the bins are done
            for (int k = l; k < RM_SPAN; k += 32) mybins[k] = 0.0f;
            __syncwarp();
            for (int64_t c0 = 0; c0 < S; c0 += RM_CHUNK) {
                // ---- the chunk's steps: this lane's RM_NB steps c0 + 32 t + l
                int rk[RM_NB];
                float rg[RM_NB];
                if (direct) {
                    const int32_t* ip = j.I + (my_valid ? my_off : 0) + c0 + l;
                    const float* gp = j.G + (my_valid ? my_off : 0) + c0 + l;
#pragma unroll
                    for (int t = 0; t < RM_NB; ++t) {
                        const bool in = my_valid && c0 + 32 * t + l < S;
                        rk[t] = in && R_IN(ip + 32 * t, 4, 0) ? __ldg(ip + 32 * t) : -1;
                        rg[t] = in && R_IN(gp + 32 * t, 4, 1) ? __ldg(gp + 32 * t) : 0.0f;
                    }
                } else {
                    // staged: element e of the [RM_WARPS][RM_CHUNK] block, lines fastest
                    int sk[RM_PER];
                    float sg[RM_PER];
#pragma unroll
                    for (int u = 0; u < RM_PER; ++u) {
                        const int e = tid + u * RM_THREADS, r = e % RM_WARPS, t = e / RM_WARPS;
                        const int64_t off = line_i[r], st = c0 + t;
                        const bool in = off >= 0 && st < S;
                        sk[u] = in && R_IN(j.I + off + st * j.sIs, 4, 0) ? __ldg(j.I + off + st * j.sIs) : -1;
                        sg[u] = in && R_IN(j.G + off + st * j.sGs, 4, 1) ? __ldg(j.G + off + st * j.sGs) : 0.0f;
                    }
                    __syncthreads();  // the previous chunk's readers of the stage are done
#pragma unroll
                    for (int u = 0; u < RM_PER; ++u) {
                        const int e = tid + u * RM_THREADS, r = e % RM_WARPS, t = e / RM_WARPS;
                        ck[r * RM_CLD + t] = sk[u];
                        cg[r * RM_CLD + t] = sg[u];
                    }
                    __syncthreads();
#pragma unroll
                    for (int t = 0; t < RM_NB; ++t) {
                        rk[t] = ck[w * RM_CLD + 32 * t + l];
                        rg[t] = cg[w * RM_CLD + 32 * t + l];
                    }
                }
                // ---- max-times: the other operand at each step's winner, all gathers in flight together
                if (MUL) {
#pragma unroll
                    for (int t = 0; t < RM_NB; ++t) {
                        const int d = rk[t] - kc32;
                        if (rk[t] >= 0 && (unsigned)d < (unsigned)kn) {
                            const float* pp = Pl + (int64_t)rk[t] * j.sPk + (c0 + 32 * t + l) * j.sPs;
                            rg[t] = __fmul_rn(rg[t], R_IN(pp, 4, 2) ? __ldg(pp) : 0.0f);
                        }
                    }
                }
                // ---- the batches in step order
#pragma unroll
                for (int t = 0; t < RM_NB; ++t) {
                    const int d = rk[t] - kc32;
                    const bool in = rk[t] >= 0 && (unsigned)d < (unsigned)kn;
                    // lanes of one bin group together; distinct negative keys keep the others apart
                    const unsigned grp = __match_any_sync(0xffffffffu, in ? d : -1 - l);
                    const int rank = __popc(grp & lanes_below);
                    if (in && rank == 0) mybins[d] = __fadd_rn(mybins[d], rg[t]);
                    unsigned more = __ballot_sync(0xffffffffu, in && rank > 0);
                    for (int rr = 1; more; ++rr) {
                        __syncwarp();
                        if (in && rank == rr) mybins[d] = __fadd_rn(mybins[d], rg[t]);
                        more = __ballot_sync(0xffffffffu, in && rank > rr);
                    }
                    __syncwarp();
                }
            }
            __syncthreads();  // every line's bins are final
            if (j.sOk == 1) {
                // bins contiguous in the gradient: warp w writes line w, lanes along k
                const int64_t o = base + w;
                if (o < lines) {
                    const int64_t b = o / X, x = o - b * X;
                    float* Or = j.O + b * j.sOb + x * j.sOx + kc;
                    for (int kk = l; kk < kn; kk += 32)
                        if (R_IN(Or + kk, 4, 3)) Or[kk] = mybins[kk];
                }
            } else {
                // lines fastest (consecutive x when sOx == 1): thread (bin, line) of RM_WARPS lines
                const int r = tid % RM_WARPS;
                const int64_t o = base + r;
                if (o < lines) {
                    const int64_t b = o / X, x = o - b * X;
                    float* Or = j.O + b * j.sOb + x * j.sOx + kc * j.sOk;
                    for (int kk = tid / RM_WARPS; kk < kn; kk += RM_THREADS / RM_WARPS)
                        if (R_IN(Or + (int64_t)kk * j.sOk, 4, 3)) Or[(int64_t)kk * j.sOk] = bins[r * RM_LD + kk];
                }
            }
        }
    }
    if (p.late_wait) pdl_wait();
}

}  // namespace

int launch_gemm_backward(int semiring, int64_t batch, int64_t M, int64_t N, int64_t K, const float* A,
                         const int64_t* sA, const float* B, const int64_t* sB, const float* dC, const int64_t* sC,
                         const int32_t* I, float* dA, const int64_t* sdA, float* dB, const int64_t* sdB,
                         cudaStream_t s)
{
    const DeviceInfo* dev = nullptr;
    TROP_TRY(ensure_device(&dev));
    RouteParams p{};
    p.nbatch = batch;
    p.K = K;
    if (dA) {
        // owners: rows (b, m); walk n; other operand B[b,k,n]
        RouteJob& j = p.job[p.njobs++];
        j.X = M;
        j.S = N;
        j.I = I;
        j.sIb = sC[0], j.sIx = sC[1], j.sIs = sC[2];
        j.G = dC;
        j.sGb = sC[0], j.sGx = sC[1], j.sGs = sC[2];
        j.P = B;
        j.sPb = sB[0], j.sPk = sB[1], j.sPs = sB[2];
        j.O = dA;
        j.sOb = sdA[0], j.sOx = sdA[1], j.sOk = sdA[2];
    }
    if (dB) {
        // owners: columns (b, n); walk m; other operand A[b,m,k]
        RouteJob& j = p.job[p.njobs++];
        j.X = N;
        j.S = M;
        j.I = I;
        j.sIb = sC[0], j.sIx = sC[2], j.sIs = sC[1];
        j.G = dC;
        j.sGb = sC[0], j.sGx = sC[2], j.sGs = sC[1];
        j.P = A;
        j.sPb = sA[0], j.sPk = sA[2], j.sPs = sA[1];
        j.O = dB;
        j.sOb = sdB[0], j.sOx = sdB[2], j.sOk = sdB[1];
    }
    if (p.njobs == 0 || batch == 0 || K == 0) return TROP_OK;
    const bool mul = semiring == TROP_MAXTIMES;
#if TROP_DEBUG_BOUNDS
    for (int i = 0; i < p.njobs; ++i) {
        RouteJob& j = p.job[i];
        const int64_t xs[3] = {batch, j.X, j.S}, ks[3] = {batch, K, j.S}, os[3] = {batch, j.X, K};
        const int64_t si[3] = {j.sIb, j.sIx, j.sIs}, sg[3] = {j.sGb, j.sGx, j.sGs};
        const int64_t sp_[3] = {j.sPb, j.sPk, j.sPs}, so[3] = {j.sOb, j.sOx, j.sOk};
        j.sp[0] = span_of(j.I, 4, 3, xs, si);
        j.sp[1] = span_of(j.G, 4, 3, xs, sg);
        j.sp[2] = span_of(mul ? j.P : nullptr, 4, 3, ks, sp_);
        j.sp[3] = span_of(j.O, 4, 3, os, so);
    }
#endif
    auto launch_match = [&](RouteParams& q) -> int {
        int64_t ctas = 1;
        for (int i = 0; i < q.njobs; ++i) ctas = std::max(ctas, (batch * q.job[i].X + RM_WARPS - 1) / RM_WARPS);
        const unsigned gx = (unsigned)std::max<int64_t>(1, std::min<int64_t>(ctas, (int64_t)dev->sm_count * 16));
        const dim3 grid(gx, (unsigned)q.njobs);
        if (mul) (void)launch_pdl(k_route_match<true>, grid, dim3(RM_THREADS), RM_SMEM, s, q);
        else (void)launch_pdl(k_route_match<false>, grid, dim3(RM_THREADS), RM_SMEM, s, q);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_error(e, "k_route_match");
        count_launches(1);
        return TROP_OK;
    };
    // one launch of the lane-per-line kernel for the jobs of q
    auto launch_lane = [&](RouteParams& q) -> int {
        int64_t groups = 1;
        for (int i = 0; i < q.njobs; ++i) {
            q.job[i].vec = lane_ok(q.job[i]) ? 1 : 0;
            groups = std::max(groups, (batch * q.job[i].X + 31) / 32);
        }
        const unsigned gx = (unsigned)std::max<int64_t>(1, std::min<int64_t>(groups, (int64_t)dev->sm_count * 16));
        if (mul) (void)launch_pdl(k_route_lane<true>, dim3(gx, (unsigned)q.njobs), dim3(32), lane_smem(K), s, q);
        else (void)launch_pdl(k_route_lane<false>, dim3(gx, (unsigned)q.njobs), dim3(32), lane_smem(K), s, q);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_error(e, "k_route_lane");
        count_launches(1);
        return TROP_OK;
    };
    if (mul && dA) {
        // max-times with dA: each gradient in a launch of the match-rank kernel of its own, whose
        // factor gathers (B[b, k, n] across B's rows for dA) are in flight for a whole warp at
        // once; the second (dB) starts at once and waits at its end (RouteParams::late_wait), so
        // the two overlap (batch-64 256^3: 64 us; the lane walk for dB beside it, 72 us)
        if (p.njobs == 1) return launch_match(p);
        RouteParams pa = p;
        pa.njobs = 1;
        TROP_TRY(launch_match(pa));
        p.job[0] = p.job[1];
        p.njobs = 1;
        p.late_wait = 1;
        return launch_match(p);
    }
    // max-plus and min-plus: both jobs in one launch of the lane-per-line kernel (measured on the
    // batch-64 256^3 gradient: 28 us, against 42 us for the rows there and the columns in a
    // bin-split kernel staging 32 x 32 blocks); max-times dB alone: the lane walk too, its factor
    // gathers (A[b, m, k], one row of A per step and warp) hidden by its ring (28 us against 35 us
    // for the match kernel)
    return launch_lane(p);
}

int register_backward_kernels()
{
    const void* km[] = {(const void*)k_route_match<true>, (const void*)k_route_match<false>};
    for (const void* k : km) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RM_SMEM);
        if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute (match route smem)");
    }
    const void* kl[] = {(const void*)k_route_lane<true>, (const void*)k_route_lane<false>};
    for (const void* k : kl) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lane_smem(RT_SPAN));
        if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute (lane route smem)");
    }
    return TROP_OK;
}

}  // namespace trop
