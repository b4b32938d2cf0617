// host_io.cu -- token rows moved between host memory and the device by a kernel.
//
// A decode step carries one token's hidden state through every layer ("One Token Through
// Qwen3.6", One Complete Decode Step). A caller that keeps the token rows in host memory hands
// the layer a few rows and takes a few rows back per step, and for so few rows a copy-engine
// transfer costs more than its bytes: the copy's own latency, and the layer's launch exposed
// behind it. When the host buffer is pinned and mapped into the device address space,
// k_copy_rows moves the rows with plain 16-byte loads and stores over the host link instead,
// so the layer's launch follows a kernel on the same stream. (One token at the one-token
// kernel's shape needs neither: that kernel reads and writes the mapped host rows itself.)
#include "launch.h"

namespace moe {

// dst[i] = src[i] for n 16-byte units; one side is mapped host memory. A layer kernel launched
// with programmatic serialization may start at once (its weight-only copies overlap the trip
// over the host link): it waits for this grid to complete before it reads the rows.
__global__ void __launch_bounds__(256) k_copy_rows(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n) {
    grid_dep_launch();
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) dst[i] = __ldcg(src + i);
}

cudaError_t launch_copy_rows(const void* src, void* dst, size_t bytes, int num_sms, cudaStream_t s) {
    const size_t n = bytes / 16;
    if (n == 0) return cudaSuccess;
    const size_t blocks = (n + 255) / 256;
    const int grid = (int)(blocks < (size_t)4 * num_sms ? blocks : (size_t)4 * num_sms);
    MOE_LAUNCH(MOE_KERNEL_COPY_ROWS, s,
               (k_copy_rows<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), n)));
    return cudaGetLastError();
}

}  // namespace moe
