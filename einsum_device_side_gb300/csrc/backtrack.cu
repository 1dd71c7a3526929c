// backtrack.cu -- argmax back-tracking through a contraction tree, and a
// small fill kernel.
//
// Back-tracking: every node's argmax holds, per output element, the winning
// assignment of the labels it eliminated (row-major linear index).  Walking
// the nodes from the root backwards, each node's output labels are already
// known (its consumers come later in the node order), so one read of its
// argmax fixes the labels it eliminated.  The walk is inherently sequential;
// one device thread does it so that no argmax ever leaves device memory.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace trop {

namespace {

__global__ void k_backtrack(const BtNode* __restrict__ nodes, int n_nodes, const int32_t* __restrict__ labs,
                            const int64_t* __restrict__ sizes, int64_t root_index, int n_labels,
                            int32_t* __restrict__ assign)
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
        for (int i = 0; i < nd.n_out; ++i) {
            const int32_t l = labs[nd.lab_off + i];
            const int32_t v = assign[l];
            if (v < 0) known = false;
            o = o * sizes[l] + (v < 0 ? 0 : v);
        }
        if (!known) continue;
        int64_t a = nd.argmax[o];
        for (int i = nd.n_k - 1; i >= 0; --i) {
            const int32_t l = labs[nd.lab_off + nd.n_out + i];
            const int64_t sz = sizes[l];
            assign[l] = (int32_t)(a % sz);
            a /= sz;
        }
    }
}

__global__ void k_fill_i32(int32_t* __restrict__ p, int64_t n, int32_t v)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        p[i] = v;
}

}  // namespace

int launch_backtrack(const BtNode* nodes_dev, int n_nodes, const int32_t* labels_dev, const int64_t* sizes_dev,
                     int64_t root_index, int n_labels, int32_t* assignment, cudaStream_t s)
{
    k_backtrack<<<1, 256, 0, s>>>(nodes_dev, n_nodes, labels_dev, sizes_dev, root_index, n_labels, assignment);
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
    cudaError_t e = cudaFuncGetAttributes(&a, (const void*)k_backtrack);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, (const void*)k_fill_i32);
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncGetAttributes (backtrack kernels)");
    return TROP_OK;
}

}  // namespace trop
