// backtrack.cu -- argmax back-tracking through a contraction tree, and a
// small fill kernel.
//
// Back-tracking: every node's argmax holds, per output element, the winning
// assignment of the labels it eliminated (row-major linear index).  Walking
// the nodes from the root backwards, each node's output labels are already
// known (its consumers come later in the node order), so one read of its
// argmax fixes the labels it eliminated.  The walk is inherently sequential;
// it runs on the device (one warp, or one thread for trees whose tables do not
// fit in shared memory) so that no argmax ever leaves device memory.
#include <cuda_runtime.h>

#include <cstdint>

#define TROP_TU 6  // this file's id in a bounds-violation record
#include "internal.h"

namespace trop {

namespace {

// In the bounds-checked build the walks take the violation record as one more argument and check
// each argmax read against its node's table (the product of its output extents) and each label
// against the assignment; in the normal build neither exists.
#if TROP_DEBUG_BOUNDS
#define BT_REC_PARAM , unsigned* rec
#define BT_REC_ARG , bounds_record()
#define BT_SPAN(base, n) (Span{reinterpret_cast<const char*>(base), reinterpret_cast<const char*>((base) + (n)), rec})
#else
#define BT_REC_PARAM
#define BT_REC_ARG
#endif

__global__ void k_backtrack(const BtNode* __restrict__ nodes, int n_nodes, const int32_t* __restrict__ labs,
                            const int64_t* __restrict__ sizes, int64_t root_index, int n_labels,
                            int32_t* __restrict__ assign BT_REC_PARAM)
{
    if (blockIdx.x != 0) return;
    for (int l = threadIdx.x; l < n_labels; l += blockDim.x) assign[l] = -1;
    __syncthreads();
    if (threadIdx.x != 0) return;
    // root output labels from root_index (row-major, last fastest)
    {
        const BtNode& r = nodes[n_nodes - 1];
        int64_t rem = root_index;
        for (int i = r.n_out - 1; i >= 0; --i) {
            const int32_t l = labs[r.lab_off + i];
            const int64_t sz = sizes[l];
            assign[l] = (int32_t)(rem % sz);
            rem /= sz;
        }
    }
    for (int j = n_nodes - 1; j >= 0; --j) {
        const BtNode nd = nodes[j];
        if (!nd.argmax || nd.n_k == 0) continue;
        int64_t o = 0;
        bool known = true;
#if TROP_DEBUG_BOUNDS
        int64_t total = 1;
#endif
        for (int i = 0; i < nd.n_out; ++i) {
            const int32_t l = labs[nd.lab_off + i];
            const int32_t v = assign[l];
            if (v < 0) known = false;
            o = o * sizes[l] + (v < 0 ? 0 : v);
#if TROP_DEBUG_BOUNDS
            total *= sizes[l];
#endif
        }
        if (!known) continue;
        int64_t a = TROP_IN(nd.argmax + o, 4, BT_SPAN(nd.argmax, total)) ? nd.argmax[o] : 0;
        for (int i = nd.n_k - 1; i >= 0; --i) {
            const int32_t l = labs[nd.lab_off + nd.n_out + i];
            const int64_t sz = sizes[l];
            if (TROP_IN(assign + l, 4, BT_SPAN(assign, n_labels))) assign[l] = (int32_t)(a % sz);
            a /= sz;
        }
    }
}

// The same walk with the node, label and extent tables and the assignment in shared memory (the
// tables of a tree fit there when the tree has up to a few thousand nodes).  One warp walks:
// lane i takes output label i of a node, a warp scan turns the extents into row-major strides
// and a warp sum gives the node's argmax offset, so a node costs one read of its argmax.
constexpr size_t BT_SMEM_MAX = 200 * 1024;
__host__ __device__ constexpr size_t bt_align(size_t n) { return (n + 15) / 16 * 16; }
__host__ __device__ inline size_t bt_smem_bytes(int n_nodes, int n_labs, int n_labels)
{
    return bt_align(sizeof(BtNode) * (size_t)n_nodes) + bt_align(sizeof(int64_t) * (size_t)n_labels) +
           bt_align(sizeof(int32_t) * (size_t)n_labs) + sizeof(int32_t) * (size_t)n_labels;
}

__global__ void __launch_bounds__(256) k_backtrack_smem(const BtNode* __restrict__ nodes_g, int n_nodes,
                                                        const int32_t* __restrict__ labs_g, int n_labs,
                                                        const int64_t* __restrict__ sizes_g, int64_t root_index,
                                                        int n_labels, int32_t* __restrict__ assign_g BT_REC_PARAM)
{
    extern __shared__ __align__(16) unsigned char bsm[];
    BtNode* nodes = reinterpret_cast<BtNode*>(bsm);
    int64_t* sizes = reinterpret_cast<int64_t*>(bsm + bt_align(sizeof(BtNode) * (size_t)n_nodes));
    int32_t* labs = reinterpret_cast<int32_t*>(reinterpret_cast<unsigned char*>(sizes) +
                                               bt_align(sizeof(int64_t) * (size_t)n_labels));
    int32_t* assign = reinterpret_cast<int32_t*>(reinterpret_cast<unsigned char*>(labs) +
                                                 bt_align(sizeof(int32_t) * (size_t)n_labs));
    const int tid = threadIdx.x;
    for (int i = tid; i < n_nodes; i += blockDim.x) nodes[i] = nodes_g[i];
    for (int i = tid; i < n_labels; i += blockDim.x) {
        sizes[i] = sizes_g[i];
        assign[i] = -1;
    }
    for (int i = tid; i < n_labs; i += blockDim.x) labs[i] = labs_g[i];
    __syncthreads();
    if (tid >= 32) return;
    const int lane = tid;
    const unsigned full = 0xffffffffu;
    if (lane == 0) {
        // root output labels from root_index (row-major, last fastest)
        const BtNode r = nodes[n_nodes - 1];
        int64_t rem = root_index;
        for (int i = r.n_out - 1; i >= 0; --i) {
            const int32_t l = labs[r.lab_off + i];
            const int64_t sz = sizes[l];
            assign[l] = (int32_t)(rem % sz);
            rem /= sz;
        }
    }
    __syncwarp();
    for (int j = n_nodes - 1; j >= 0; --j) {
        const BtNode nd = nodes[j];
        if (!nd.argmax || nd.n_k == 0) continue;
        int64_t sz = 1;
        int32_t v = 0;
        if (lane < nd.n_out) {
            const int32_t l = labs[nd.lab_off + lane];
            sz = sizes[l];
            v = assign[l];
        }
        if (__any_sync(full, v < 0)) continue;  // an output label no later node fixed
        // inclusive suffix product of the extents, then shifted: the row-major stride of lane i
        int64_t st = sz;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t t = __shfl_down_sync(full, st, d);
            if (lane + d < 32) st *= t;
        }
        int64_t stride = __shfl_down_sync(full, st, 1);
        if (lane == 31) stride = 1;
        int64_t o = lane < nd.n_out ? (int64_t)v * stride : 0;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) o += __shfl_xor_sync(full, o, d);
        if (lane == 0) {
            // (st of lane 0: the product of the node's output extents, its table's size)
            int64_t a = TROP_IN(nd.argmax + o, 4, BT_SPAN(nd.argmax, st)) ? nd.argmax[o] : 0;
            for (int i = nd.n_k - 1; i >= 0; --i) {
                const int32_t l = labs[nd.lab_off + nd.n_out + i];
                const int64_t s = sizes[l];
                if (TROP_IN(assign + l, 4, BT_SPAN(assign, n_labels))) assign[l] = (int32_t)(a % s);
                a /= s;
            }
        }
        __syncwarp();
    }
    for (int l = lane; l < n_labels; l += 32) assign_g[l] = assign[l];
}

__global__ void k_fill_i32(int32_t* __restrict__ p, int64_t n, int32_t v)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        p[i] = v;
}

}  // namespace

int launch_backtrack(const BtNode* nodes_dev, int n_nodes, const int32_t* labels_dev, int n_labs,
                     const int64_t* sizes_dev, int64_t root_index, int n_labels, int32_t* assignment, cudaStream_t s)
{
    const size_t smem = bt_smem_bytes(n_nodes, n_labs, n_labels);
    if (smem <= BT_SMEM_MAX)
        k_backtrack_smem<<<1, 256, smem, s>>>(nodes_dev, n_nodes, labels_dev, n_labs, sizes_dev, root_index, n_labels,
                                              assignment BT_REC_ARG);
    else
        k_backtrack<<<1, 256, 0, s>>>(nodes_dev, n_nodes, labels_dev, sizes_dev, root_index, n_labels,
                                      assignment BT_REC_ARG);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "k_backtrack");
    count_launches(1);
    return TROP_OK;
}

int launch_fill_i32(int32_t* p, int64_t n, int32_t value, cudaStream_t s)
{
    if (n <= 0) return TROP_OK;
    const DeviceInfo* dev = nullptr;
    TROP_TRY(ensure_device(&dev));
    int64_t blocks = (n + 255) / 256, cap = (int64_t)dev->sm_count * 8;
    k_fill_i32<<<(int)(blocks < cap ? blocks : cap), 256, 0, s>>>(p, n, value);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "k_fill_i32");
    count_launches(1);
    return TROP_OK;
}

int register_backtrack_kernels()
{
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncSetAttribute((const void*)k_backtrack_smem, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)BT_SMEM_MAX);
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute (backtrack smem)");
    e = cudaFuncGetAttributes(&a, (const void*)k_backtrack);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, (const void*)k_fill_i32);
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncGetAttributes (backtrack kernels)");
    return TROP_OK;
}

}  // namespace trop
