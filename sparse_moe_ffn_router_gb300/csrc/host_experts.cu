// host_experts.cu -- routed experts resident in host memory.
//
// The pages give the model a storage hierarchy (checkpoint on disk, system RAM, GPU memory,
// kernels; "One Token Through Qwen3.6", Where the Weights Live) and note that the routing
// decides which expert weights a layer actually needs ("One Token Through Qwen3.6", One
// Complete Decode Step). On a Grace-Blackwell node the routed experts can therefore stay in
// the host's memory, pinned and mapped into the device address space, with only the router
// and the shared expert in HBM: after the routing, k_fetch_experts copies the gate_up and down
// rows of the experts this call touches over the host link into a device shadow laid out like
// the full [E, 2I, H] and [E, H, I] tensors, and the expert kernels run from the shadow
// unchanged. The copy uses plain 16-byte loads of the mapped host memory (eight per thread in
// flight, each warp on one 4 KB stretch at a time), the ordinary way a kernel reads mapped
// pinned memory.
#include "launch.h"

namespace moe {

constexpr int kFetchUnroll = 8;

__global__ void __launch_bounds__(256) k_fetch_experts(LayerArgs a, const uint4* hgu, const uint4* hdn, uint4* sgu,
                                                       uint4* sdn) {
    const int n = a.hdr->n_act;  // experts with pairs, from the routing kernels
    const size_t gu = (size_t)2 * a.I * a.H / 8, dn = (size_t)a.H * a.I / 8, per = gu + dn;  // 16-byte units
    // warp w copies runs of 32 * kFetchUnroll consecutive units (4 KB), runs w, w + warps, ...:
    // each load instruction reads 512 contiguous bytes and a warp's loads in flight share
    // one 4 KB stretch of host memory. No run spans experts or the gate_up / down boundary:
    // with H % 128 == 0 and I % 64 == 0 (checked on the host), gu = H*I/4 and dn = H*I/8 are
    // multiples of 1024 units, so both are multiples of the run.
    constexpr size_t kRun = 32 * kFetchUnroll;
    const int lane = threadIdx.x & 31;
    const size_t warps = (size_t)gridDim.x * (blockDim.x >> 5);
    const size_t runs = (size_t)n * per / kRun;
    for (size_t q = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); q < runs; q += warps) {
        const size_t i0 = q * kRun, j = i0 / per, r0 = i0 - j * per;
        const size_t e = (size_t)a.act[j];
        const uint4* src = r0 < gu ? hgu + e * gu + r0 : hdn + e * dn + (r0 - gu);
        uint4* dst = r0 < gu ? sgu + e * gu + r0 : sdn + e * dn + (r0 - gu);
        uint4 v[kFetchUnroll];
#pragma unroll
        for (int u = 0; u < kFetchUnroll; ++u) v[u] = __ldcg(src + u * 32 + lane);
#pragma unroll
        for (int u = 0; u < kFetchUnroll; ++u) dst[u * 32 + lane] = v[u];
    }
}

cudaError_t launch_fetch_experts(const LayerArgs& a, const bf16* host_gate_up, const bf16* host_down, bf16* shadow_gate_up,
                                 bf16* shadow_down, cudaStream_t s) {
    MOE_LAUNCH(MOE_KERNEL_FETCH_EXPERTS, s,
               (k_fetch_experts<<<4 * a.num_sms, 256, 0, s>>>(
                   a, reinterpret_cast<const uint4*>(host_gate_up), reinterpret_cast<const uint4*>(host_down),
                   reinterpret_cast<uint4*>(shadow_gate_up), reinterpret_cast<uint4*>(shadow_down))));
    return cudaGetLastError();
}

}  // namespace moe
