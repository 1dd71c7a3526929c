// api.cpp -- validation, einsum planning and the extern "C" entry points.
//
// The lowering follows the shape of omeinsum-rs issue #52 ("GPU tropical
// path: keep tensors device-resident + device-side permute"): diagonals and
// traces are a unary pre-pass (section "Resolved design for step 3", kernel
// (b), and "Structural lessons from OMEinsum"), after which the GEMM sees
// clean batch x rows x contraction operands; operands are permuted on the
// device only when their strides cannot feed the GEMM, and the GEMM writes
// value and argmax through the output's own strides, which is how "GEMM
// transpose flags avoid one permute" is realised here.  Everything stays in
// device memory; the host only plans and launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <list>
#include <memory>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "internal.h"

namespace trop {

int register_unary_kernels();
int register_gemm_kernels();
int register_backward_kernels();
int register_gemm64_kernels();
int register_gemm_int_kernels();
int register_backtrack_kernels();
int launch_fill_i32(int32_t* p, int64_t n, int32_t value, cudaStream_t s);

int register_kernels_for_device()
{
    TROP_TRY(register_unary_kernels());
    TROP_TRY(register_gemm_kernels());
    TROP_TRY(register_backward_kernels());
    TROP_TRY(register_gemm64_kernels());
    TROP_TRY(register_gemm_int_kernels());
    TROP_TRY(register_backtrack_kernels());
    return TROP_OK;
}

namespace {

// ------------------------------------------------------------------ views
struct View {
    const void* data;
    int dtype;
    int rank;
    int32_t lab[MAXR];
    int64_t size[MAXR];
    int64_t stride[MAXR];
};

int find_label(const View& v, int32_t l)
{
    for (int i = 0; i < v.rank; ++i)
        if (v.lab[i] == l) return i;
    return -1;
}

int64_t numel(const View& v)
{
    int64_t n = 1;
    for (int i = 0; i < v.rank; ++i) n *= v.size[i];
    return n;
}

// repeated labels -> one axis whose stride is the sum (a diagonal view);
// labels in first-appearance order
int unique_view(const View& in, View& out)
{
    out = View{};
    out.data = in.data;
    out.dtype = in.dtype;
    for (int i = 0; i < in.rank; ++i) {
        int j = find_label(out, in.lab[i]);
        if (j >= 0) {
            if (out.size[j] != in.size[i])
                return set_error(TROP_ERR_SHAPE, "label %d repeated with extents %lld and %lld", in.lab[i],
                                 (long long)out.size[j], (long long)in.size[i]);
            out.stride[j] += in.stride[i];
            continue;
        }
        int k = out.rank++;
        out.lab[k] = in.lab[i];
        out.size[k] = in.size[i];
        out.stride[k] = in.stride[i];
    }
    return TROP_OK;
}

// ------------------------------------------------------------------ spec parsing
int parse_letters(const char* s, int n, int32_t* lab, int& rank)
{
    rank = 0;
    for (int i = 0; i < n; ++i) {
        char c = s[i];
        if (c == ' ') continue;
        if (!((c >= 'a' && c <= 'z') || (c >= 'A' && c <= 'Z')))
            return set_error(TROP_ERR_SPEC, "spec character '%c' is not a letter", c);
        if (rank >= MAXR) return set_error(TROP_ERR_SPEC, "spec operand has more than %d labels", MAXR);
        lab[rank++] = (int32_t)c;
    }
    return TROP_OK;
}

// "ab,bc->ac" or "aab->b"; nops = 1 or 2
int parse_spec(const char* spec, int& nops, int32_t la[MAXR], int& ra, int32_t lb[MAXR], int& rb,
               int32_t lo[MAXR], int& ro)
{
    if (!spec) return set_error(TROP_ERR_INVALID_ARG, "spec is NULL");
    const char* arrow = strstr(spec, "->");
    if (!arrow) return set_error(TROP_ERR_SPEC, "spec '%s' has no '->'", spec);
    const char* comma = (const char*)memchr(spec, ',', (size_t)(arrow - spec));
    if (comma) {
        nops = 2;
        TROP_TRY(parse_letters(spec, (int)(comma - spec), la, ra));
        TROP_TRY(parse_letters(comma + 1, (int)(arrow - comma - 1), lb, rb));
        if (memchr(comma + 1, ',', (size_t)(arrow - comma - 1)))
            return set_error(TROP_ERR_SPEC, "spec '%s' has more than two operands", spec);
    } else {
        nops = 1;
        TROP_TRY(parse_letters(spec, (int)(arrow - spec), la, ra));
        rb = 0;
    }
    TROP_TRY(parse_letters(arrow + 2, (int)strlen(arrow + 2), lo, ro));
    return TROP_OK;
}

// ------------------------------------------------------------------ tensor checks
int check_tensor(const trop_tensor* t, const char* name, bool need_data)
{
    if (!t) return set_error(TROP_ERR_INVALID_ARG, "%s is NULL", name);
    if (t->rank < 0 || t->rank > MAXR) return set_error(TROP_ERR_INVALID_ARG, "%s rank %d out of range", name, t->rank);
    if (dtype_bytes(t->dtype) == 0) return set_error(TROP_ERR_DTYPE, "%s has unknown dtype %d", name, t->dtype);
    int64_t n = 1;
    for (int i = 0; i < t->rank; ++i) {
        if (t->shape[i] < 0) return set_error(TROP_ERR_SHAPE, "%s has a negative extent", name);
        n *= t->shape[i];
    }
    if (n > 0 && need_data) TROP_TRY(check_device_pointer(t->data, name));
    return TROP_OK;
}

View view_of(const trop_tensor* t, const int32_t* lab)
{
    View v{};
    v.data = t->data;
    v.dtype = t->dtype;
    v.rank = t->rank;
    for (int i = 0; i < t->rank; ++i) {
        v.lab[i] = lab[i];
        v.size[i] = t->shape[i];
        v.stride[i] = t->stride[i];
    }
    return v;
}

// contiguous row-major strides for `n` extents
void contiguous_strides(int n, const int64_t* size, int64_t* stride)
{
    int64_t s = 1;
    for (int i = n - 1; i >= 0; --i) {
        stride[i] = s;
        s *= size[i];
    }
}

// ------------------------------------------------------------------ unary
struct UnaryPlan {
    View u;            // unique view of the input
    int n_red;
    int red_ax[MAXR];  // axes of u reduced, in u order
    int out_ax[MAXR];  // axis of u for each output label
};

int plan_unary(const View& in, const int32_t* lo, int ro, UnaryPlan& p)
{
    TROP_TRY(unique_view(in, p.u));
    bool used[MAXR] = {false};
    for (int i = 0; i < ro; ++i) {
        int j = find_label(p.u, lo[i]);
        if (j < 0) return set_error(TROP_ERR_SPEC, "output label %d does not appear in the input", lo[i]);
        if (used[j]) return set_error(TROP_ERR_SPEC, "output label %d is repeated", lo[i]);
        used[j] = true;
        p.out_ax[i] = j;
    }
    p.n_red = 0;
    for (int j = 0; j < p.u.rank; ++j)
        if (!used[j]) p.red_ax[p.n_red++] = j;
    return TROP_OK;
}

// run a planned unary op: out (strided) and argmax (contiguous in out shape, nullable); a
// split reduction keeps its partials in `fixed` when given, else in pool workspace
int exec_unary(int sr, const UnaryPlan& p, int ro, void* out, const int64_t* ostride, int32_t* argmax,
               cudaStream_t s, const ReduceScratch* fixed = nullptr)
{
    int64_t osize[MAXR], astride[MAXR];
    int64_t n_out = 1;
    for (int i = 0; i < ro; ++i) {
        osize[i] = p.u.size[p.out_ax[i]];
        n_out *= osize[i];
    }
    contiguous_strides(ro, osize, astride);
    if (n_out == 0) return TROP_OK;
    int64_t R = 1;
    for (int i = 0; i < p.n_red; ++i) R *= p.u.size[p.red_ax[i]];
    if (p.n_red == 0) {
        GatherDesc d{};
        d.rank = ro;
        for (int i = 0; i < ro; ++i) {
            d.size[i] = osize[i];
            d.s_in[i] = p.u.stride[p.out_ax[i]];
            d.s_out[i] = ostride[i];
        }
        TROP_TRY(launch_gather(p.u.data, out, (int)dtype_bytes(p.u.dtype), nullptr, nullptr, d, s));
        if (argmax) TROP_TRY(launch_fill_i32(argmax, n_out, 0, s));
        return TROP_OK;
    }
    if (argmax && R - 1 > INT32_MAX)
        return set_error(TROP_ERR_OVERFLOW, "reduced extent %lld does not fit an int32 argmax", (long long)R);
    ReduceDesc d{};
    d.out_rank = ro;
    for (int i = 0; i < ro; ++i) {
        d.out_size[i] = osize[i];
        d.out_s_in[i] = p.u.stride[p.out_ax[i]];
        d.out_s_out[i] = ostride[i];
        d.out_s_arg[i] = astride[i];
    }
    d.red_rank = p.n_red;
    for (int i = 0; i < p.n_red; ++i) {
        d.red_size[i] = p.u.size[p.red_ax[i]];
        d.red_s_in[i] = p.u.stride[p.red_ax[i]];
    }
    return launch_reduce(sr, p.u.dtype, p.u.data, out, argmax, d, fixed, s);
}

// ------------------------------------------------------------------ pairwise planning
enum Cls { C_BATCH, C_LEFT, C_RIGHT, C_K, C_RA, C_RB };

struct LabelInfo {
    int32_t lab;
    int64_t size;
    int cls;
    int64_t sA, sB, sO, sI;  // strides (0 where absent)
    int posO;                // position in the output (-1)
};

struct PairPlan {
    // pre-pass work
    bool reduceA, reduceB, permA, permB;
    // final GEMM layout (strides relative to the operand the GEMM reads)
    GemmDesc g;
    std::string text;
};

struct Workspace {
    std::vector<void*> blocks;
    cudaStream_t s;
    int alloc(size_t bytes, void** p)
    {
        int rc = pool_alloc(bytes, s, p);
        if (rc == TROP_OK) blocks.push_back(*p);
        return rc;
    }
    ~Workspace()
    {
        for (void* b : blocks) pool_retire(b, s);
    }
};

// One pre-pass of an operand recorded by the lowering: a (+)-reduction of its one-operand
// labels (reduce) or a permute, into a contiguous workspace tensor of `bytes`.  At run time its
// input is the operand's current buffer (the caller's, or the previous pre-pass's workspace).
struct PrePass {
    int operand;  // 0: A, 1: B
    bool reduce;
    UnaryPlan up;  // reduce: up.u is the input view (its data pointer is filled at run time)
    int ro;
    int64_t ostride[MAXR];
    GatherDesc gd;  // permute
    int elem_bytes;
    size_t bytes;
};

// A pairwise einsum lowered for one layout (labels, extents, strides, dtype, semiring): the
// pre-passes, then the GEMM.  Nothing in it depends on the data pointers, which run_lowered
// fills in: the GEMM reads each operand from the caller's buffer or from the workspace of that
// operand's last pre-pass.
struct LoweredPair {
    bool empty = false;  // no output element: nothing runs
    int npre = 0;
    PrePass pre[4];
    int last_pre[2] = {-1, -1};
    GemmDesc g{};  // A, B, C and I are filled at run time
    std::string text;
};

// reduce the one-operand labels of `v` (not in `keep`) into a contiguous workspace tensor
// holding the kept labels in v's order
void prereduce(const View& v, const std::vector<bool>& keep_mask, int operand, LoweredPair& L, View& out)
{
    out = View{};
    out.dtype = v.dtype;
    PrePass& P = L.pre[L.npre];
    P = PrePass{};
    P.operand = operand;
    P.reduce = true;
    P.up.u = v;
    int ro = 0;
    int32_t lo[MAXR];
    P.up.n_red = 0;
    for (int i = 0; i < v.rank; ++i) {
        if (keep_mask[i]) {
            P.up.out_ax[ro] = i;
            lo[ro++] = v.lab[i];
        } else {
            P.up.red_ax[P.up.n_red++] = i;
        }
    }
    P.ro = ro;
    out.rank = ro;
    for (int i = 0; i < ro; ++i) {
        out.lab[i] = lo[i];
        out.size[i] = v.size[P.up.out_ax[i]];
    }
    contiguous_strides(ro, out.size, out.stride);
    std::copy(out.stride, out.stride + ro, P.ostride);
    P.elem_bytes = (int)dtype_bytes(v.dtype);
    P.bytes = (size_t)std::max<int64_t>(numel(out), 1) * dtype_bytes(v.dtype);
    L.last_pre[operand] = L.npre++;
}

// permute v into a contiguous workspace tensor with labels in `order`
void permute_to(const View& v, const std::vector<int32_t>& order, int operand, LoweredPair& L, View& out)
{
    out = View{};
    out.dtype = v.dtype;
    out.rank = (int)order.size();
    for (int i = 0; i < out.rank; ++i) {
        int j = find_label(v, order[i]);
        out.lab[i] = order[i];
        out.size[i] = v.size[j];
    }
    contiguous_strides(out.rank, out.size, out.stride);
    PrePass& P = L.pre[L.npre];
    P = PrePass{};
    P.operand = operand;
    P.reduce = false;
    P.gd.rank = out.rank;
    for (int i = 0; i < out.rank; ++i) {
        int j = find_label(v, order[i]);
        P.gd.size[i] = v.size[j];
        P.gd.s_in[i] = v.stride[j];
        P.gd.s_out[i] = out.stride[i];
    }
    P.elem_bytes = (int)dtype_bytes(v.dtype);
    P.bytes = (size_t)std::max<int64_t>(numel(out), 1) * dtype_bytes(v.dtype);
    L.last_pre[operand] = L.npre++;
}

bool chain_merges(const std::vector<int32_t>& labs, const View& v)
{
    for (size_t i = 0; i + 1 < labs.size(); ++i) {
        int a = find_label(v, labs[i]), b = find_label(v, labs[i + 1]);
        if (v.stride[a] != v.stride[b] * v.size[b]) return false;
    }
    return true;
}

int64_t chain_stride(const std::vector<int32_t>& labs, const View& v)
{
    if (labs.empty()) return 0;
    return v.stride[find_label(v, labs.back())];
}

// pick a group of `cands` (labels of one operand that are free in the output)
// that merges into one axis in the operand, the output and the argmax layout
std::vector<int32_t> pick_group(const std::vector<int32_t>& cands, const View& v, const int32_t* lo, int ro,
                                const int64_t* ostride, const int64_t* osize)
{
    std::vector<int32_t> g;
    if (cands.empty()) return g;
    int32_t first = cands[0];
    for (int32_t l : cands) {
        int a = find_label(v, l), b = find_label(v, first);
        if (std::llabs(v.stride[a]) < std::llabs(v.stride[b])) first = l;
    }
    g.push_back(first);
    auto posO = [&](int32_t l) {
        for (int i = 0; i < ro; ++i)
            if (lo[i] == l) return i;
        return -1;
    };
    for (;;) {
        int32_t head = g.front();
        int hv = find_label(v, head), ho = posO(head);
        int32_t next = -1;
        for (int32_t l : cands) {
            if (std::find(g.begin(), g.end(), l) != g.end()) continue;
            int lv = find_label(v, l), lp = posO(l);
            if (lp != ho - 1) continue;
            if (v.stride[lv] != v.stride[hv] * v.size[hv]) continue;
            if (ostride[lp] != ostride[ho] * osize[ho]) continue;
            next = l;
            break;
        }
        if (next < 0) break;
        g.insert(g.begin(), next);
    }
    return g;
}

// The lowering of a pairwise einsum: label classes, unit labels dropped, groups of labels that
// merge into one GEMM axis, permutes only where strides cannot feed the GEMM.
// has_argmax: whether an argmax is written (decides the int32 range check and its layout).
int lower_pairwise(int sr, const View& A0, const View& B0, const int32_t* lo, int ro, const int64_t* ostride,
                   bool has_argmax, LoweredPair& L)
{
    if (dtype_bytes(A0.dtype) == 0 || B0.dtype != A0.dtype)
        return set_error(TROP_ERR_DTYPE, "pairwise tropical einsum needs two operands of one dtype (f32, f64, i32, i64)");
    View A, B;
    TROP_TRY(unique_view(A0, A));
    TROP_TRY(unique_view(B0, B));
    // output labels
    int64_t osize[MAXR];
    for (int i = 0; i < ro; ++i) {
        for (int j = 0; j < i; ++j)
            if (lo[j] == lo[i]) return set_error(TROP_ERR_SPEC, "output label %d is repeated", lo[i]);
        int a = find_label(A, lo[i]), b = find_label(B, lo[i]);
        if (a < 0 && b < 0) return set_error(TROP_ERR_SPEC, "output label %d appears in no operand", lo[i]);
        osize[i] = a >= 0 ? A.size[a] : B.size[b];
    }
    for (int i = 0; i < A.rank; ++i) {
        int b = find_label(B, A.lab[i]);
        if (b >= 0 && B.size[b] != A.size[i])
            return set_error(TROP_ERR_SHAPE, "label %d has extent %lld in A and %lld in B", A.lab[i],
                             (long long)A.size[i], (long long)B.size[b]);
    }
    int64_t astride[MAXR];
    contiguous_strides(ro, osize, astride);
    int64_t n_out = 1;
    for (int i = 0; i < ro; ++i) n_out *= osize[i];
    auto inO = [&](int32_t l) {
        for (int i = 0; i < ro; ++i)
            if (lo[i] == l) return i;
        return -1;
    };

    std::string desc;

    // one-operand labels absent from the output: (+)-reduce first
    {
        std::vector<bool> keepA(A.rank), keepB(B.rank);
        bool ra = false, rb = false;
        for (int i = 0; i < A.rank; ++i) {
            keepA[i] = inO(A.lab[i]) >= 0 || find_label(B, A.lab[i]) >= 0;
            ra = ra || !keepA[i];
        }
        for (int i = 0; i < B.rank; ++i) {
            keepB[i] = inO(B.lab[i]) >= 0 || find_label(A, B.lab[i]) >= 0;
            rb = rb || !keepB[i];
        }
        if (n_out > 0 && ra) {
            View t;
            prereduce(A, keepA, 0, L, t);
            A = t;
            desc += "reduceA ";
        }
        if (n_out > 0 && rb) {
            View t;
            prereduce(B, keepB, 1, L, t);
            B = t;
            desc += "reduceB ";
        }
    }
    if (n_out == 0) {
        L.empty = true;
        L.text = "empty output";
        return TROP_OK;
    }

    // classify
    std::vector<int32_t> Lk, Lb, Lm, Ln;
    for (int i = 0; i < A.rank; ++i) {
        int32_t l = A.lab[i];
        bool b = find_label(B, l) >= 0, o = inO(l) >= 0;
        if (b && o) Lb.push_back(l);
        else if (b) Lk.push_back(l);
        else Lm.push_back(l);
    }
    for (int i = 0; i < B.rank; ++i)
        if (find_label(A, B.lab[i]) < 0) Ln.push_back(B.lab[i]);
    int64_t K = 1;
    for (int32_t l : Lk) K *= A.size[find_label(A, l)];
    if (has_argmax && K - 1 > INT32_MAX)
        return set_error(TROP_ERR_OVERFLOW, "contracted extent %lld does not fit an int32 argmax", (long long)K);
    // size-1 contracted labels do not change the linear index
    {
        std::vector<int32_t> t;
        for (int32_t l : Lk)
            if (A.size[find_label(A, l)] != 1) t.push_back(l);
        Lk.swap(t);
    }

    auto group_sizes = [&](const std::vector<int32_t>& g, const View& v) {
        int64_t n = 1;
        for (int32_t l : g) n *= v.size[find_label(v, l)];
        return n;
    };
    auto drop_unit = [&](std::vector<int32_t>& g, const View& v) {
        std::vector<int32_t> t;
        for (int32_t l : g)
            if (v.size[find_label(v, l)] != 1) t.push_back(l);
        g.swap(t);
    };
    drop_unit(Lm, A);
    drop_unit(Ln, B);
    drop_unit(Lb, A);

    // the contraction must be one axis in both operands
    bool kA = chain_merges(Lk, A), kB = chain_merges(Lk, B);
    std::vector<int32_t> Gm = pick_group(Lm, A, lo, ro, ostride, osize);
    std::vector<int32_t> Gn = pick_group(Ln, B, lo, ro, ostride, osize);
    // also require the argmax layout (contiguous in output order) to merge: it
    // does whenever the output strides do for a contiguous output; otherwise
    // shrink the group to its fastest label
    auto argmax_ok = [&](const std::vector<int32_t>& g) {
        for (size_t i = 0; i + 1 < g.size(); ++i) {
            int a = inO(g[i]), b = inO(g[i + 1]);
            if (astride[a] != astride[b] * osize[b]) return false;
        }
        return true;
    };
    if (!argmax_ok(Gm)) Gm.erase(Gm.begin(), Gm.end() - 1);
    if (!argmax_ok(Gn)) Gn.erase(Gn.begin(), Gn.end() - 1);
    const int64_t M = group_sizes(Gm, A), N = group_sizes(Gn, B);
    const bool big = M >= 64 && N >= 64 && K >= 16;
    int64_t sAk = Lk.empty() ? 0 : chain_stride(Lk, A), sBk = Lk.empty() ? 0 : chain_stride(Lk, B);
    int64_t sAm = Gm.empty() ? 0 : chain_stride(Gm, A), sBn = Gn.empty() ? 0 : chain_stride(Gn, B);
    const bool nn = (Lk.empty() || sAk == 1) && (Gn.empty() || sBn == 1);
    const bool tt = (Lk.empty() || sBk == 1) && (Gm.empty() || sAm == 1);
    bool permA = !kA || (big && !nn && !tt && !(Lk.empty() || sAk == 1));
    bool permB = !kB || (big && !nn && !tt && !(Gn.empty() || sBn == 1));
    if (permA) {
        // [batch, free (A order), contracted]
        std::vector<int32_t> order;
        for (int32_t l : Lb) order.push_back(l);
        for (int i = 0; i < A.rank; ++i)
            if (std::find(Lm.begin(), Lm.end(), A.lab[i]) != Lm.end()) order.push_back(A.lab[i]);
        for (int32_t l : Lk) order.push_back(l);
        // unit labels ride along (size 1): keep every label of A
        for (int i = 0; i < A.rank; ++i)
            if (std::find(order.begin(), order.end(), A.lab[i]) == order.end()) order.insert(order.begin(), A.lab[i]);
        View t;
        permute_to(A, order, 0, L, t);
        A = t;
        desc += "permA ";
    }
    if (permB) {
        std::vector<int32_t> order;
        for (int32_t l : Lb) order.push_back(l);
        for (int32_t l : Lk) order.push_back(l);
        for (int i = 0; i < B.rank; ++i)
            if (std::find(Ln.begin(), Ln.end(), B.lab[i]) != Ln.end()) order.push_back(B.lab[i]);
        for (int i = 0; i < B.rank; ++i)
            if (std::find(order.begin(), order.end(), B.lab[i]) == order.end()) order.insert(order.begin(), B.lab[i]);
        View t;
        permute_to(B, order, 1, L, t);
        B = t;
        desc += "permB ";
    }
    if (permA || permB) {
        Gm = pick_group(Lm, A, lo, ro, ostride, osize);
        Gn = pick_group(Ln, B, lo, ro, ostride, osize);
        if (!argmax_ok(Gm)) Gm.erase(Gm.begin(), Gm.end() - 1);
        if (!argmax_ok(Gn)) Gn.erase(Gn.begin(), Gn.end() - 1);
        sAk = Lk.empty() ? 0 : chain_stride(Lk, A);
        sBk = Lk.empty() ? 0 : chain_stride(Lk, B);
    }

    GemmDesc& g = L.g;
    g = GemmDesc{};
    g.semiring = sr;
    g.dtype = A0.dtype;
    g.M = group_sizes(Gm, A);
    g.N = group_sizes(Gn, B);
    g.K = group_sizes(Lk, A);
    // the data pointers are the run's; a description takes every pointer as 256-byte aligned
    g.A = g.B = g.C = nullptr;
    g.I = has_argmax ? reinterpret_cast<int32_t*>(uintptr_t(256)) : nullptr;
    g.sAk = sAk;
    g.sBk = sBk;
    if (!Gm.empty()) {
        g.sAm = chain_stride(Gm, A);
        g.sCm = ostride[inO(Gm.back())];
        g.sIm = astride[inO(Gm.back())];
    }
    if (!Gn.empty()) {
        g.sBn = chain_stride(Gn, B);
        g.sCn = ostride[inO(Gn.back())];
        g.sIn = astride[inO(Gn.back())];
    }
    // batch: shared labels, then free labels outside the groups (stride 0 in the other operand)
    g.nb = 0;
    auto add_batch = [&](int32_t l) -> int {
        if (g.nb >= MAXB) return set_error(TROP_ERR_UNSUPPORTED, "more than %d batch axes after lowering", MAXB);
        int a = find_label(A, l), b = find_label(B, l), o = inO(l);
        int d = g.nb++;
        g.bsize[d] = a >= 0 ? A.size[a] : B.size[b];
        g.sAb[d] = a >= 0 ? A.stride[a] : 0;
        g.sBb[d] = b >= 0 ? B.stride[b] : 0;
        g.sCb[d] = ostride[o];
        g.sIb[d] = astride[o];
        return TROP_OK;
    };
    for (int i = 0; i < ro; ++i) {
        int32_t l = lo[i];
        bool inGm = std::find(Gm.begin(), Gm.end(), l) != Gm.end();
        bool inGn = std::find(Gn.begin(), Gn.end(), l) != Gn.end();
        if (inGm || inGn || osize[i] == 1) continue;
        // merge with the previous batch axis when every tensor's strides chain
        if (g.nb > 0) {
            int q = g.nb - 1;
            int a = find_label(A, l), b = find_label(B, l), o = inO(l);
            int64_t sz = a >= 0 ? A.size[a] : B.size[b];
            int64_t sa = a >= 0 ? A.stride[a] : 0, sb = b >= 0 ? B.stride[b] : 0;
            if (g.sAb[q] == sa * sz && g.sBb[q] == sb * sz && g.sCb[q] == ostride[o] * sz &&
                g.sIb[q] == astride[o] * sz) {
                g.bsize[q] *= sz;
                g.sAb[q] = sa;
                g.sBb[q] = sb;
                g.sCb[q] = ostride[o];
                g.sIb[q] = astride[o];
                continue;
            }
        }
        TROP_TRY(add_batch(l));
    }
    char buf[512];
    char route[128];
    describe_gemm(g, route, sizeof route);
    snprintf(buf, sizeof buf, "%sgemm M=%lld N=%lld K=%lld batch_axes=%d sAm=%lld sAk=%lld sBk=%lld sBn=%lld sCm=%lld sCn=%lld%s",
             desc.c_str(), (long long)g.M, (long long)g.N, (long long)g.K, g.nb, (long long)g.sAm,
             (long long)g.sAk, (long long)g.sBk, (long long)g.sBn, (long long)g.sCm, (long long)g.sCn, route);
    L.text = buf;
    return TROP_OK;
}

// Run a lowered pairwise einsum on actual buffers: each pre-pass into pool workspace (retired
// through the stream's event when the call ends), then the GEMM.
int run_lowered(int sr, const LoweredPair& L, const void* a_data, const void* b_data, void* out, int32_t* argmax,
                cudaStream_t s)
{
    if (L.empty) return TROP_OK;
    Workspace ws;
    ws.s = s;
    const void* cur[2] = {a_data, b_data};
    for (int i = 0; i < L.npre; ++i) {
        const PrePass& P = L.pre[i];
        void* p = nullptr;
        TROP_TRY(ws.alloc(P.bytes, &p));
        if (P.reduce) {
            UnaryPlan up = P.up;
            up.u.data = const_cast<void*>(cur[P.operand]);
            TROP_TRY(exec_unary(sr, up, P.ro, p, P.ostride, nullptr, s));
        } else {
            TROP_TRY(launch_gather(cur[P.operand], p, P.elem_bytes, nullptr, nullptr, P.gd, s));
        }
        cur[P.operand] = p;
    }
    GemmDesc g = L.g;
    g.A = cur[0];
    g.B = cur[1];
    g.C = out;
    g.I = argmax;
    return launch_gemm(g, s, nullptr);
}

// ------------------------------------------------------------------ plan cache
// Lowered pairwise einsums kept per layout, so that a repeated call (the same spec on tensors
// of the same shapes, strides, dtype and 16-byte alignment, the same semiring, with or without
// argmax) skips the lowering -- the analogue of the plan cache the tenferro-rs note keeps per
// contraction ("Problem").  Least recently used entries go first beyond the bound (64 by
// default, TROP_PLAN_CACHE from the environment at load; 0 disables it).
struct PlanCache {
    std::mutex mu;
    size_t capacity;
    std::list<std::pair<std::string, std::shared_ptr<const LoweredPair>>> lru;  // front: most recent
    std::unordered_map<std::string, decltype(lru)::iterator> map;
    PlanCache()
    {
        const char* e = std::getenv("TROP_PLAN_CACHE");
        capacity = e ? (size_t)std::max(0L, std::strtol(e, nullptr, 10)) : 64;
    }
};
PlanCache& plan_cache()
{
    static PlanCache c;
    return c;
}
void key_put(std::string& k, const void* p, size_t n) { k.append(static_cast<const char*>(p), n); }
void key_view(std::string& k, const View& v)
{
    key_put(k, &v.rank, sizeof v.rank);
    key_put(k, &v.dtype, sizeof v.dtype);
    key_put(k, v.lab, sizeof(int32_t) * v.rank);
    key_put(k, v.size, sizeof(int64_t) * v.rank);
    key_put(k, v.stride, sizeof(int64_t) * v.rank);
}

int plan_and_run_pairwise(int sr, const View& A0, const View& B0, const int32_t* lo, int ro, void* out,
                          const int64_t* ostride, int32_t* argmax, cudaStream_t s)
{
    PlanCache& C = plan_cache();
    size_t capacity;
    {
        std::lock_guard<std::mutex> lk(C.mu);
        capacity = C.capacity;
    }
    if (capacity == 0) {
        LoweredPair L;
        TROP_TRY(lower_pairwise(sr, A0, B0, lo, ro, ostride, argmax != nullptr, L));
        return run_lowered(sr, L, A0.data, B0.data, out, argmax, s);
    }
    std::string key;
    key.reserve(1024);
    const uint8_t head[2] = {(uint8_t)sr, (uint8_t)(argmax != nullptr)};
    key_put(key, head, sizeof head);
    // 16-byte alignment of every buffer (kernel choices below the lowering depend on it)
    const uint8_t align[4] = {(uint8_t)((uintptr_t)A0.data & 15), (uint8_t)((uintptr_t)B0.data & 15),
                              (uint8_t)((uintptr_t)out & 15), (uint8_t)((uintptr_t)argmax & 15)};
    key_put(key, align, sizeof align);
    key_view(key, A0);
    key_view(key, B0);
    key_put(key, &ro, sizeof ro);
    key_put(key, lo, sizeof(int32_t) * ro);
    key_put(key, ostride, sizeof(int64_t) * ro);
    std::shared_ptr<const LoweredPair> L;
    {
        std::lock_guard<std::mutex> lk(C.mu);
        auto it = C.map.find(key);
        if (it != C.map.end()) {
            C.lru.splice(C.lru.begin(), C.lru, it->second);
            L = it->second->second;
        }
    }
    count_plan(L != nullptr);
    if (!L) {
        auto fresh = std::make_shared<LoweredPair>();
        TROP_TRY(lower_pairwise(sr, A0, B0, lo, ro, ostride, argmax != nullptr, *fresh));
        L = fresh;
        std::lock_guard<std::mutex> lk(C.mu);
        if (C.map.find(key) == C.map.end()) {
            C.lru.emplace_front(key, L);
            C.map[key] = C.lru.begin();
            while (C.map.size() > C.capacity) {
                C.map.erase(C.lru.back().first);
                C.lru.pop_back();
            }
        }
    }
    return run_lowered(sr, *L, A0.data, B0.data, out, argmax, s);
}

int tensor_labels_check(const trop_tensor* t, int rank, const char* name)
{
    if (t->rank != rank)
        return set_error(TROP_ERR_SPEC, "%s has rank %d but the spec gives it %d labels", name, t->rank, rank);
    return TROP_OK;
}

}  // namespace
}  // namespace trop

using namespace trop;

// ====================================================================== entry points

namespace {

// tropical_permute_trace and its allocation-free twin: validation and lowering are shared;
// only where a split reduction keeps its partial results differs (no_alloc: the fixed scratch)
int permute_trace_impl(const trop_tensor* in, const char* spec, int semiring, const trop_tensor* out,
                       int32_t* argmax, cudaStream_t stream, bool no_alloc)
{
    if (semiring < 0 || semiring > 2) return set_error(TROP_ERR_INVALID_ARG, "unknown semiring %d", semiring);
    int nops, ra, rb, ro;
    int32_t la[MAXR], lb[MAXR], lo[MAXR];
    TROP_TRY(parse_spec(spec, nops, la, ra, lb, rb, lo, ro));
    if (nops != 1) return set_error(TROP_ERR_SPEC, "permute/trace takes one operand");
    TROP_TRY(check_tensor(in, "in", true));
    TROP_TRY(check_tensor(out, "out", true));
    TROP_TRY(tensor_labels_check(in, ra, "in"));
    TROP_TRY(tensor_labels_check(out, ro, "out"));
    if (in->dtype != out->dtype) return set_error(TROP_ERR_DTYPE, "in and out dtypes differ");
    TROP_TRY(ensure_device(nullptr));
    ReduceScratch fixed{};
    if (no_alloc) TROP_TRY(noalloc_scratch(&fixed.ptr, &fixed.bytes));
    UnaryPlan p{};
    TROP_TRY(plan_unary(view_of(in, la), lo, ro, p));
    int64_t n_out = 1;
    for (int i = 0; i < ro; ++i) {
        if (out->shape[i] != p.u.size[p.out_ax[i]])
            return set_error(TROP_ERR_SHAPE, "out extent %d is %lld, spec implies %lld", i, (long long)out->shape[i],
                             (long long)p.u.size[p.out_ax[i]]);
        n_out *= out->shape[i];
    }
    if (argmax && n_out > 0) TROP_TRY(check_device_pointer(argmax, "argmax"));
    return exec_unary(semiring, p, ro, out->data, out->stride, argmax, stream, no_alloc ? &fixed : nullptr);
}

}  // namespace

extern "C" int tropical_permute_trace(const trop_tensor* in, const char* spec, int semiring, const trop_tensor* out,
                                      int32_t* argmax, void* stream)
{
    clear_error();
    return permute_trace_impl(in, spec, semiring, out, argmax, (cudaStream_t)stream, false);
}

// Allocation-free twin of tropical_permute_trace for callers that must not
// allocate device memory: split reductions keep their partial results in the
// library's fixed scratch (noalloc.cu) instead of pool workspace.
extern "C" int tropical_permute_trace_noalloc(const trop_tensor* in, const char* spec, int semiring,
                                              const trop_tensor* out, int32_t* argmax, void* stream)
{
    clear_error();
    NoAllocScope no_alloc;  // every launcher below allocates nothing on this thread
    return permute_trace_impl(in, spec, semiring, out, argmax, (cudaStream_t)stream, true);
}

extern "C" int tropical_permute_pair(const trop_tensor* val_in, const trop_tensor* arg_in, const char* spec,
                                     const trop_tensor* val_out, const trop_tensor* arg_out, void* stream)
{
    clear_error();
    int nops, ra, rb, ro;
    int32_t la[MAXR], lb[MAXR], lo[MAXR];
    TROP_TRY(parse_spec(spec, nops, la, ra, lb, rb, lo, ro));
    if (nops != 1) return set_error(TROP_ERR_SPEC, "permute_pair takes one operand");
    TROP_TRY(check_tensor(val_in, "val_in", true));
    TROP_TRY(check_tensor(arg_in, "arg_in", true));
    TROP_TRY(check_tensor(val_out, "val_out", true));
    TROP_TRY(check_tensor(arg_out, "arg_out", true));
    TROP_TRY(tensor_labels_check(val_in, ra, "val_in"));
    TROP_TRY(tensor_labels_check(val_out, ro, "val_out"));
    if (arg_in->dtype != TROP_I32 || arg_out->dtype != TROP_I32)
        return set_error(TROP_ERR_DTYPE, "argmax tensors must be int32");
    if (val_in->dtype != val_out->dtype) return set_error(TROP_ERR_DTYPE, "value dtypes differ");
    if (arg_in->rank != val_in->rank || arg_out->rank != val_out->rank)
        return set_error(TROP_ERR_SHAPE, "argmax ranks differ from the value ranks");
    for (int i = 0; i < val_in->rank; ++i)
        if (arg_in->shape[i] != val_in->shape[i]) return set_error(TROP_ERR_SHAPE, "arg_in shape differs from val_in");
    for (int i = 0; i < val_out->rank; ++i)
        if (arg_out->shape[i] != val_out->shape[i]) return set_error(TROP_ERR_SHAPE, "arg_out shape differs from val_out");
    if (ra != ro) return set_error(TROP_ERR_SPEC, "permute_pair spec must be a permutation");
    for (int i = 0; i < ra; ++i)
        for (int j = 0; j < i; ++j)
            if (la[i] == la[j]) return set_error(TROP_ERR_SPEC, "permute_pair spec repeats a label");
    TROP_TRY(ensure_device(nullptr));
    GatherDesc d{};
    d.rank = ro;
    for (int i = 0; i < ro; ++i) {
        int j = -1;
        for (int k = 0; k < ra; ++k)
            if (la[k] == lo[i]) j = k;
        if (j < 0) return set_error(TROP_ERR_SPEC, "permute_pair output label %c missing from input", (char)lo[i]);
        if (val_out->shape[i] != val_in->shape[j]) return set_error(TROP_ERR_SHAPE, "val_out extent %d mismatch", i);
        d.size[i] = val_out->shape[i];
        d.s_in[i] = val_in->stride[j];
        d.s_out[i] = val_out->stride[i];
        d.s_in2[i] = arg_in->stride[j];
        d.s_out2[i] = arg_out->stride[i];
    }
    return launch_gather(val_in->data, val_out->data, (int)dtype_bytes(val_in->dtype),
                         static_cast<const int32_t*>(arg_in->data), static_cast<int32_t*>(arg_out->data), d,
                         (cudaStream_t)stream);
}

extern "C" int tropical_gemm_strided_batched_argmax(int semiring, int dtype, int64_t batch, int64_t M, int64_t N,
                                                    int64_t K, const void* A, int64_t sAb, int64_t sAm, int64_t sAk,
                                                    const void* B, int64_t sBb, int64_t sBk, int64_t sBn, void* C,
                                                    int64_t sCb, int64_t sCm, int64_t sCn, int32_t* argmax,
                                                    void* stream)
{
    clear_error();
    if (semiring < 0 || semiring > 2) return set_error(TROP_ERR_INVALID_ARG, "unknown semiring %d", semiring);
    if (dtype_bytes(dtype) == 0) return set_error(TROP_ERR_DTYPE, "tropical GEMM: unknown dtype %d", dtype);
    if (batch < 0 || M < 0 || N < 0 || K < 0) return set_error(TROP_ERR_INVALID_ARG, "negative extent");
    if (argmax && K - 1 > INT32_MAX)
        return set_error(TROP_ERR_OVERFLOW, "K = %lld does not fit an int32 argmax", (long long)K);
    if (batch == 0 || M == 0 || N == 0) return TROP_OK;
    TROP_TRY(ensure_device(nullptr));
    if (K > 0) {
        TROP_TRY(check_device_pointer(A, "A"));
        TROP_TRY(check_device_pointer(B, "B"));
    }
    TROP_TRY(check_device_pointer(C, "C"));
    if (argmax) TROP_TRY(check_device_pointer(argmax, "argmax"));
    GemmDesc g{};
    g.semiring = semiring;
    g.dtype = dtype;
    g.M = M;
    g.N = N;
    g.K = K;
    g.A = A;
    g.B = B;
    g.C = C;
    g.I = argmax;
    g.sAm = sAm;
    g.sAk = sAk;
    g.sBk = sBk;
    g.sBn = sBn;
    g.sCm = sCm;
    g.sCn = sCn;
    g.sIm = sCm;
    g.sIn = sCn;
    g.nb = 1;
    g.bsize[0] = batch;
    g.sAb[0] = sAb;
    g.sBb[0] = sBb;
    g.sCb[0] = sCb;
    g.sIb[0] = sCb;
    if (K == 0) {
        g.sAk = g.sBk = 0;
    }
    return launch_gemm(g, (cudaStream_t)stream, nullptr);
}

extern "C" int tropical_gemm_backward(int semiring, int64_t batch, int64_t M, int64_t N, int64_t K, const float* A,
                                      int64_t sAb, int64_t sAm, int64_t sAk, const float* B, int64_t sBb, int64_t sBk,
                                      int64_t sBn, const float* dC, int64_t sCb, int64_t sCm, int64_t sCn,
                                      const int32_t* argmax, float* dA, int64_t sdAb, int64_t sdAm, int64_t sdAk,
                                      float* dB, int64_t sdBb, int64_t sdBk, int64_t sdBn, void* stream)
{
    clear_error();
    if (semiring < 0 || semiring > 2) return set_error(TROP_ERR_INVALID_ARG, "unknown semiring %d", semiring);
    if (batch < 0 || M < 0 || N < 0 || K < 0) return set_error(TROP_ERR_INVALID_ARG, "negative extent");
    if (K > INT32_MAX) return set_error(TROP_ERR_OVERFLOW, "K = %lld exceeds the int32 argmax range", (long long)K);
    const bool wantA = dA && M > 0 && K > 0, wantB = dB && N > 0 && K > 0;
    if (batch == 0 || (!wantA && !wantB)) return TROP_OK;
    TROP_TRY(ensure_device(nullptr));
    if (wantA) TROP_TRY(check_device_pointer(dA, "dA"));
    if (wantB) TROP_TRY(check_device_pointer(dB, "dB"));
    const bool walks = (wantA && N > 0) || (wantB && M > 0);  // anything routes at all
    if (walks) {
        TROP_TRY(check_device_pointer(dC, "dC"));
        TROP_TRY(check_device_pointer(argmax, "argmax"));
        if (semiring == TROP_MAXTIMES) {
            if (wantA) TROP_TRY(check_device_pointer(B, "B"));
            if (wantB) TROP_TRY(check_device_pointer(A, "A"));
        }
    }
    const int64_t sA[3] = {sAb, sAm, sAk}, sB[3] = {sBb, sBk, sBn}, sC[3] = {sCb, sCm, sCn};
    const int64_t sdA[3] = {sdAb, sdAm, sdAk}, sdB[3] = {sdBb, sdBk, sdBn};
    return launch_gemm_backward(semiring, batch, M, N, K, A, sA, B, sB, dC, sC, argmax, wantA ? dA : nullptr, sdA,
                                wantB ? dB : nullptr, sdB, (cudaStream_t)stream);
}

extern "C" int tropical_einsum_pairwise(const char* spec, const trop_tensor* A, const trop_tensor* B, int semiring,
                                        const trop_tensor* out, int32_t* argmax, void* stream)
{
    clear_error();
    if (semiring < 0 || semiring > 2) return set_error(TROP_ERR_INVALID_ARG, "unknown semiring %d", semiring);
    int nops, ra, rb, ro;
    int32_t la[MAXR], lb[MAXR], lo[MAXR];
    TROP_TRY(parse_spec(spec, nops, la, ra, lb, rb, lo, ro));
    if (nops != 2) return set_error(TROP_ERR_SPEC, "pairwise einsum takes two operands");
    TROP_TRY(check_tensor(A, "A", true));
    TROP_TRY(check_tensor(B, "B", true));
    TROP_TRY(check_tensor(out, "out", true));
    TROP_TRY(tensor_labels_check(A, ra, "A"));
    TROP_TRY(tensor_labels_check(B, rb, "B"));
    TROP_TRY(tensor_labels_check(out, ro, "out"));
    if (dtype_bytes(out->dtype) == 0) return set_error(TROP_ERR_DTYPE, "out has an unknown dtype %d", out->dtype);
    if (A->dtype != out->dtype || B->dtype != out->dtype)
        return set_error(TROP_ERR_DTYPE, "A, B and out must share one dtype");
    TROP_TRY(ensure_device(nullptr));
    // output extents must match the operands
    View vA = view_of(A, la), vB = view_of(B, lb);
    int64_t n_out = 1;
    for (int i = 0; i < ro; ++i) {
        int64_t sz = -1;
        for (int j = 0; j < ra; ++j)
            if (la[j] == lo[i]) sz = A->shape[j];
        for (int j = 0; j < rb && sz < 0; ++j)
            if (lb[j] == lo[i]) sz = B->shape[j];
        if (sz >= 0 && out->shape[i] != sz)
            return set_error(TROP_ERR_SHAPE, "out extent %d is %lld, spec implies %lld", i, (long long)out->shape[i],
                             (long long)sz);
        n_out *= out->shape[i];
    }
    if (argmax && n_out > 0) TROP_TRY(check_device_pointer(argmax, "argmax"));
    return plan_and_run_pairwise(semiring, vA, vB, lo, ro, out->data, out->stride, argmax, (cudaStream_t)stream);
}

extern "C" void tropical_set_plan_cache_capacity(int capacity)
{
    PlanCache& C = plan_cache();
    std::lock_guard<std::mutex> lk(C.mu);
    C.capacity = capacity < 0 ? 0 : (size_t)capacity;
    while (C.map.size() > C.capacity) {
        C.map.erase(C.lru.back().first);
        C.lru.pop_back();
    }
}

extern "C" int tropical_plan_describe(const char* spec, int rank_a, const int64_t* shape_a, const int64_t* stride_a,
                                      int rank_b, const int64_t* shape_b, const int64_t* stride_b, char* buf,
                                      int buflen)
{
    clear_error();
    if (!buf || buflen <= 0 || !shape_a || !stride_a || !shape_b || !stride_b)
        return set_error(TROP_ERR_INVALID_ARG, "NULL argument");
    int nops, ra, rb, ro;
    int32_t la[MAXR], lb[MAXR], lo[MAXR];
    TROP_TRY(parse_spec(spec, nops, la, ra, lb, rb, lo, ro));
    if (nops != 2 || ra != rank_a || rb != rank_b) return set_error(TROP_ERR_SPEC, "spec does not match the ranks");
    View A{}, B{};
    A.dtype = B.dtype = TROP_F32;
    A.rank = ra;
    B.rank = rb;
    for (int i = 0; i < ra; ++i) {
        A.lab[i] = la[i];
        A.size[i] = shape_a[i];
        A.stride[i] = stride_a[i];
    }
    for (int i = 0; i < rb; ++i) {
        B.lab[i] = lb[i];
        B.size[i] = shape_b[i];
        B.stride[i] = stride_b[i];
    }
    int64_t osize[MAXR], ostride[MAXR];
    for (int i = 0; i < ro; ++i) {
        osize[i] = -1;
        for (int j = 0; j < ra; ++j)
            if (la[j] == lo[i]) osize[i] = shape_a[j];
        for (int j = 0; j < rb && osize[i] < 0; ++j)
            if (lb[j] == lo[i]) osize[i] = shape_b[j];
        if (osize[i] < 0) return set_error(TROP_ERR_SPEC, "output label appears in no operand");
    }
    contiguous_strides(ro, osize, ostride);
    std::string text;
    LoweredPair L;
    TROP_TRY(lower_pairwise(TROP_MAXPLUS, A, B, lo, ro, ostride, true, L));
    snprintf(buf, (size_t)buflen, "%s", L.text.c_str());
    return TROP_OK;
}

// ---------------------------------------------------------------------- trees
namespace {

struct NodeShape {
    int rank;
    int32_t lab[MAXR];
    int64_t size[MAXR];
};

int node_operand(int id, int n_inputs, const trop_tensor* inputs, const std::vector<NodeShape>& shapes,
                 const std::vector<void*>& inter, int nlab, const int32_t* labs, int dtype, View& v,
                 const char* name)
{
    if (id < n_inputs) {
        const trop_tensor* t = &inputs[id];
        if (t->rank != nlab)
            return set_error(TROP_ERR_SPEC, "%s: input %d has rank %d, node gives %d labels", name, id, t->rank, nlab);
        v = view_of(t, labs);
    } else {
        const NodeShape& sh = shapes[id - n_inputs];
        if (sh.rank != nlab)
            return set_error(TROP_ERR_SPEC, "%s: intermediate %d has rank %d, node gives %d labels", name, id, sh.rank,
                             nlab);
        v = View{};
        v.data = inter[id - n_inputs];
        v.dtype = dtype;
        v.rank = nlab;
        for (int i = 0; i < nlab; ++i) {
            v.lab[i] = labs[i];
            v.size[i] = sh.size[i];
        }
        contiguous_strides(nlab, v.size, v.stride);
    }
    return TROP_OK;
}

// shapes of every node output, validating labels; no device work
int tree_shapes(int n_inputs, const trop_tensor* inputs, int n_nodes, const trop_node* nodes,
                std::vector<NodeShape>& shapes, std::vector<int>& last_use, int dtype)
{
    shapes.assign(n_nodes, NodeShape{});
    last_use.assign(n_nodes, -1);
    for (int j = 0; j < n_nodes; ++j) {
        const trop_node& nd = nodes[j];
        const int ids[2] = {nd.lhs, nd.rhs};
        const int nl[2] = {nd.n_lhs, nd.n_rhs};
        const int32_t* ls[2] = {nd.lhs_labels, nd.rhs_labels};
        const int nops = nd.rhs < 0 ? 1 : 2;
        if (nd.n_out < 0 || nd.n_out > MAXR || (nd.n_out > 0 && !nd.out_labels))
            return set_error(TROP_ERR_INVALID_ARG, "node %d: bad output labels", j);
        if (nops == 2 && dtype_bytes(dtype) == 0)
            return set_error(TROP_ERR_DTYPE, "node %d: unknown dtype %d", j, dtype);
        int32_t all_lab[2 * MAXR];
        int64_t all_size[2 * MAXR];
        int nall = 0;
        for (int o = 0; o < nops; ++o) {
            int id = ids[o];
            if (id < 0 || id >= n_inputs + j)
                return set_error(TROP_ERR_INVALID_ARG, "node %d: operand id %d out of range", j, id);
            if (nl[o] < 0 || nl[o] > MAXR || (nl[o] > 0 && !ls[o]))
                return set_error(TROP_ERR_INVALID_ARG, "node %d: bad operand labels", j);
            const int64_t* sz;
            int rk;
            if (id < n_inputs) {
                if (inputs[id].dtype != dtype) return set_error(TROP_ERR_DTYPE, "input %d dtype differs from out", id);
                sz = inputs[id].shape;
                rk = inputs[id].rank;
            } else {
                sz = shapes[id - n_inputs].size;
                rk = shapes[id - n_inputs].rank;
                last_use[id - n_inputs] = j;
            }
            if (rk != nl[o]) return set_error(TROP_ERR_SPEC, "node %d: operand %d rank %d vs %d labels", j, id, rk, nl[o]);
            for (int i = 0; i < rk; ++i) {
                int32_t l = ls[o][i];
                if (l < 0 || l > 65535) return set_error(TROP_ERR_INVALID_ARG, "node %d: label %d out of range", j, l);
                int f = -1;
                for (int q = 0; q < nall; ++q)
                    if (all_lab[q] == l) f = q;
                if (f >= 0 && all_size[f] != sz[i])
                    return set_error(TROP_ERR_SHAPE, "node %d: label %d has extents %lld and %lld", j, l,
                                     (long long)all_size[f], (long long)sz[i]);
                if (f < 0) {
                    all_lab[nall] = l;
                    all_size[nall++] = sz[i];
                }
            }
        }
        NodeShape& sh = shapes[j];
        sh.rank = nd.n_out;
        for (int i = 0; i < nd.n_out; ++i) {
            int32_t l = nd.out_labels[i];
            int f = -1;
            for (int q = 0; q < nall; ++q)
                if (all_lab[q] == l) f = q;
            if (f < 0) return set_error(TROP_ERR_SPEC, "node %d: output label %d appears in no operand", j, l);
            for (int q = 0; q < i; ++q)
                if (nd.out_labels[q] == l) return set_error(TROP_ERR_SPEC, "node %d: output label %d repeated", j, l);
            sh.lab[i] = l;
            sh.size[i] = all_size[f];
        }
    }
    return TROP_OK;
}

}  // namespace

namespace {

int run_tree(int n_inputs, const trop_tensor* inputs, int n_nodes, const trop_node* nodes, int semiring,
             const trop_tensor* out, int32_t* const* node_argmax, cudaStream_t s)
{
    if (semiring < 0 || semiring > 2) return set_error(TROP_ERR_INVALID_ARG, "unknown semiring %d", semiring);
    if (n_inputs < 0 || n_nodes < 1 || (n_inputs > 0 && !inputs) || !nodes)
        return set_error(TROP_ERR_INVALID_ARG, "empty tree or NULL arrays");
    TROP_TRY(check_tensor(out, "out", true));
    for (int i = 0; i < n_inputs; ++i) {
        char nm[32];
        snprintf(nm, sizeof nm, "inputs[%d]", i);
        TROP_TRY(check_tensor(&inputs[i], nm, true));
    }
    TROP_TRY(ensure_device(nullptr));
    std::vector<NodeShape> shapes;
    std::vector<int> last_use;
    TROP_TRY(tree_shapes(n_inputs, inputs, n_nodes, nodes, shapes, last_use, out->dtype));
    const NodeShape& root = shapes[n_nodes - 1];
    if (out->rank != root.rank) return set_error(TROP_ERR_SHAPE, "out rank %d, root node rank %d", out->rank, root.rank);
    for (int i = 0; i < root.rank; ++i)
        if (out->shape[i] != root.size[i]) return set_error(TROP_ERR_SHAPE, "out extent %d mismatch with the root node", i);
    if (node_argmax)
        for (int j = 0; j < n_nodes; ++j) {
            int64_t n = 1;
            for (int i = 0; i < shapes[j].rank; ++i) n *= shapes[j].size[i];
            if (node_argmax[j] && n > 0) TROP_TRY(check_device_pointer(node_argmax[j], "node_argmax"));
        }
    std::vector<void*> inter(n_nodes, nullptr);
    int rc = TROP_OK;
    for (int j = 0; j < n_nodes && rc == TROP_OK; ++j) {
        const trop_node& nd = nodes[j];
        const bool root_node = j == n_nodes - 1;
        const NodeShape& sh = shapes[j];
        int64_t ostride[MAXR];
        void* dst;
        if (root_node) {
            dst = out->data;
            for (int i = 0; i < sh.rank; ++i) ostride[i] = out->stride[i];
        } else {
            int64_t n = 1;
            for (int i = 0; i < sh.rank; ++i) n *= sh.size[i];
            rc = pool_alloc((size_t)std::max<int64_t>(n, 1) * dtype_bytes(out->dtype), s, &inter[j]);
            if (rc != TROP_OK) break;
            dst = inter[j];
            contiguous_strides(sh.rank, sh.size, ostride);
        }
        int32_t* am = node_argmax ? node_argmax[j] : nullptr;
        View a{}, b{};
        rc = node_operand(nd.lhs, n_inputs, inputs, shapes, inter, nd.n_lhs, nd.lhs_labels, out->dtype, a, "lhs");
        if (rc == TROP_OK && nd.rhs >= 0)
            rc = node_operand(nd.rhs, n_inputs, inputs, shapes, inter, nd.n_rhs, nd.rhs_labels, out->dtype, b, "rhs");
        if (rc != TROP_OK) break;
        if (nd.rhs < 0) {
            a.dtype = out->dtype;
            UnaryPlan up{};
            rc = plan_unary(a, nd.out_labels, nd.n_out, up);
            if (rc == TROP_OK) rc = exec_unary(semiring, up, nd.n_out, dst, ostride, am, s);
        } else {
            rc = plan_and_run_pairwise(semiring, a, b, nd.out_labels, nd.n_out, dst, ostride, am, s);
        }
        // retire intermediates whose last consumer is this node
        const int ids[2] = {nd.lhs, nd.rhs};
        for (int o = 0; o < 2; ++o) {
            int id = ids[o];
            if (id >= n_inputs && last_use[id - n_inputs] == j && inter[id - n_inputs]) {
                pool_retire(inter[id - n_inputs], s);
                inter[id - n_inputs] = nullptr;
            }
        }
    }
    // intermediates nobody consumed (or left over after an error)
    for (int j = 0; j < n_nodes; ++j)
        if (inter[j]) pool_retire(inter[j], s);
    return rc;
}

// Capture run_tree's launches on `ps` into a graph with `arena` serving every workspace request.
int capture_tree(CaptureArena* arena, cudaStream_t ps, int n_inputs, const trop_tensor* inputs, int n_nodes,
                 const trop_node* nodes, int semiring, const trop_tensor* out, int32_t* const* node_argmax,
                 cudaGraph_t* graph)
{
    *graph = nullptr;
    cudaError_t e = cudaStreamBeginCapture(ps, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_error(e, "cudaStreamBeginCapture");
    set_capture_arena(arena);
    int rc = run_tree(n_inputs, inputs, n_nodes, nodes, semiring, out, node_argmax, ps);
    set_capture_arena(nullptr);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(ps, &g);
    if (rc != TROP_OK) {
        if (g) cudaGraphDestroy(g);
        cudaGetLastError();
        return rc;
    }
    if (e != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        return cuda_error(e, "cudaStreamEndCapture");
    }
    *graph = g;
    return TROP_OK;
}

}  // namespace

struct trop_tree_plan_s {
    int device;
    cudaGraphExec_t exec;
    void* arena;
    size_t arena_bytes;
    int64_t launches;
};

extern "C" int tropical_contract_tree(int n_inputs, const trop_tensor* inputs, int n_nodes, const trop_node* nodes,
                                      int semiring, const trop_tensor* out, int32_t* const* node_argmax, void* stream)
{
    clear_error();
    return run_tree(n_inputs, inputs, n_nodes, nodes, semiring, out, node_argmax, (cudaStream_t)stream);
}

extern "C" int tropical_tree_plan_create(int n_inputs, const trop_tensor* inputs, int n_nodes, const trop_node* nodes,
                                         int semiring, const trop_tensor* out, int32_t* const* node_argmax,
                                         trop_tree_plan* plan)
{
    clear_error();
    if (!plan) return set_error(TROP_ERR_INVALID_ARG, "NULL plan");
    *plan = nullptr;
    TROP_TRY(ensure_device(nullptr));  // module set-up stays outside the capture
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    cudaStream_t ps = nullptr;
    e = cudaStreamCreateWithFlags(&ps, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_error(e, "cudaStreamCreateWithFlags");
    // pass 1: the same lowering over a fake, aligned base measures the workspace high-water mark
    CaptureArena measure;
    measure.base = uintptr_t(1) << 40;
    measure.measuring = true;
    cudaGraph_t g = nullptr;
    int rc = capture_tree(&measure, ps, n_inputs, inputs, n_nodes, nodes, semiring, out, node_argmax, &g);
    if (g) cudaGraphDestroy(g);
    g = nullptr;
    void* mem = nullptr;
    const size_t bytes = std::max<size_t>(measure.high, 256);
    if (rc == TROP_OK) {
        e = cudaMalloc(&mem, bytes);
        if (e != cudaSuccess) {
            cudaGetLastError();
            rc = set_error(TROP_ERR_OOM, "plan workspace of %zu bytes: %s", bytes, cudaGetErrorString(e));
        }
    }
    // pass 2: real memory of that size; every block lands at the offset it had in pass 1
    CaptureArena real;
    real.base = reinterpret_cast<uintptr_t>(mem);
    real.capacity = bytes;
    if (rc == TROP_OK) rc = capture_tree(&real, ps, n_inputs, inputs, n_nodes, nodes, semiring, out, node_argmax, &g);
    cudaGraphExec_t exec = nullptr;
    if (rc == TROP_OK) {
        e = cudaGraphInstantiate(&exec, g, 0);
        if (e != cudaSuccess) rc = cuda_error(e, "cudaGraphInstantiate");
    }
    if (g) cudaGraphDestroy(g);
    cudaStreamDestroy(ps);
    if (rc != TROP_OK) {
        if (mem) cudaFree(mem);
        return rc;
    }
    *plan = new trop_tree_plan_s{dev, exec, mem, bytes, real.launches};
    return TROP_OK;
}

extern "C" int tropical_tree_plan_run(trop_tree_plan plan, void* stream)
{
    clear_error();
    if (!plan) return set_error(TROP_ERR_INVALID_ARG, "NULL plan");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (dev != plan->device)
        return set_error(TROP_ERR_DEVICE_MISMATCH, "plan belongs to device %d, current device is %d", plan->device, dev);
    note_stream_op();  // a graph launch: the next kernel waits for the whole graph
    e = cudaGraphLaunch(plan->exec, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_error(e, "cudaGraphLaunch");
    count_launches(plan->launches);
    return TROP_OK;
}

extern "C" int tropical_tree_plan_info(trop_tree_plan plan, int64_t* kernels, size_t* workspace_bytes)
{
    clear_error();
    if (!plan) return set_error(TROP_ERR_INVALID_ARG, "NULL plan");
    if (kernels) *kernels = plan->launches;
    if (workspace_bytes) *workspace_bytes = plan->arena_bytes;
    return TROP_OK;
}

extern "C" int tropical_tree_plan_destroy(trop_tree_plan plan)
{
    clear_error();
    if (!plan) return TROP_OK;
    int rc = TROP_OK;
    cudaError_t e = cudaGraphExecDestroy(plan->exec);
    if (e != cudaSuccess) rc = cuda_error(e, "cudaGraphExecDestroy");
    e = cudaFree(plan->arena);
    if (e != cudaSuccess && rc == TROP_OK) rc = cuda_error(e, "cudaFree (plan workspace)");
    delete plan;
    return rc;
}

extern "C" int tropical_tree_backtrack(int n_inputs, const trop_tensor* inputs, int n_nodes, const trop_node* nodes,
                                       int32_t* const* node_argmax, int64_t root_index, int n_labels,
                                       int32_t* assignment, void* stream)
{
    clear_error();
    if (n_inputs < 0 || n_nodes < 1 || (n_inputs > 0 && !inputs) || !nodes || !node_argmax || n_labels < 1)
        return set_error(TROP_ERR_INVALID_ARG, "NULL arrays or empty tree");
    TROP_TRY(ensure_device(nullptr));
    TROP_TRY(check_device_pointer(assignment, "assignment"));
    std::vector<NodeShape> shapes;
    std::vector<int> last_use;
    const int dtype = n_inputs > 0 ? inputs[0].dtype : TROP_F32;
    TROP_TRY(tree_shapes(n_inputs, inputs, n_nodes, nodes, shapes, last_use, dtype));
    int64_t root_n = 1;
    for (int i = 0; i < shapes[n_nodes - 1].rank; ++i) root_n *= shapes[n_nodes - 1].size[i];
    if (root_index < 0 || root_index >= root_n) return set_error(TROP_ERR_INVALID_ARG, "root_index out of range");
    // label table: per node, output labels then argmax labels
    std::vector<BtNode> bt(n_nodes);
    std::vector<int32_t> labs;
    std::vector<int64_t> sizes(n_labels, 1);
    for (int j = 0; j < n_nodes; ++j) {
        const trop_node& nd = nodes[j];
        const NodeShape& sh = shapes[j];
        bt[j].argmax = node_argmax[j];
        bt[j].lab_off = (int)labs.size();
        bt[j].n_out = sh.rank;
        for (int i = 0; i < sh.rank; ++i) {
            if (sh.lab[i] >= n_labels) return set_error(TROP_ERR_INVALID_ARG, "label %d >= n_labels", sh.lab[i]);
            labs.push_back(sh.lab[i]);
            sizes[sh.lab[i]] = sh.size[i];
        }
        // argmax labels: unary -> labels absent from out (first appearance in lhs);
        // binary -> labels in both operands absent from out (first appearance in lhs)
        std::vector<int32_t> kl;
        auto in_out = [&](int32_t l) {
            for (int i = 0; i < sh.rank; ++i)
                if (sh.lab[i] == l) return true;
            return false;
        };
        auto in_rhs = [&](int32_t l) {
            for (int i = 0; i < nd.n_rhs; ++i)
                if (nd.rhs_labels[i] == l) return true;
            return false;
        };
        const int64_t* lsz = nd.lhs < n_inputs ? inputs[nd.lhs].shape : shapes[nd.lhs - n_inputs].size;
        for (int i = 0; i < nd.n_lhs; ++i) {
            int32_t l = nd.lhs_labels[i];
            if (in_out(l) || std::find(kl.begin(), kl.end(), l) != kl.end()) continue;
            if (nd.rhs >= 0 && !in_rhs(l)) continue;
            if (l >= n_labels) return set_error(TROP_ERR_INVALID_ARG, "label %d >= n_labels", l);
            kl.push_back(l);
            sizes[l] = lsz[i];
        }
        // (extent-1 labels contribute digit 0 to the row-major index either way)
        bt[j].n_k = 0;
        for (int32_t l : kl) {
            labs.push_back(l);
            ++bt[j].n_k;
        }
    }
    // upload the tables through one workspace block
    const size_t nb_nodes = sizeof(BtNode) * bt.size();
    const size_t nb_labs = sizeof(int32_t) * std::max<size_t>(labs.size(), 1);
    const size_t nb_sizes = sizeof(int64_t) * sizes.size();
    const size_t off_labs = (nb_nodes + 255) / 256 * 256;
    const size_t off_sizes = off_labs + (nb_labs + 255) / 256 * 256;
    const size_t total = off_sizes + nb_sizes;
    std::vector<char> host(total, 0);
    memcpy(host.data(), bt.data(), nb_nodes);
    if (!labs.empty()) memcpy(host.data() + off_labs, labs.data(), sizeof(int32_t) * labs.size());
    memcpy(host.data() + off_sizes, sizes.data(), nb_sizes);
    cudaStream_t s = (cudaStream_t)stream;
    void* dev = nullptr;
    TROP_TRY(pool_alloc(total, s, &dev));
    // pageable source: the copy is staged by the driver before this call returns
    cudaError_t e = cudaMemcpyAsync(dev, host.data(), total, cudaMemcpyHostToDevice, s);
    int rc = e == cudaSuccess ? TROP_OK : cuda_error(e, "cudaMemcpyAsync (backtrack tables)");
    if (rc == TROP_OK)
        rc = launch_backtrack(static_cast<const BtNode*>(dev), n_nodes,
                              reinterpret_cast<const int32_t*>(static_cast<char*>(dev) + off_labs), (int)labs.size(),
                              reinterpret_cast<const int64_t*>(static_cast<char*>(dev) + off_sizes), root_index,
                              n_labels, assignment, s);
    pool_retire(dev, s);
    return rc;
}
