// launch.h -- internal interface between the C-ABI entry points and the kernels.
#pragma once

#include "common.cuh"

namespace moe {

// Everything one call of the layer touches. Routing outputs (ids .. perm) point either into
// the caller's buffers (moe_route) or into the workspace (moe_forward).
struct LayerArgs {
    const bf16* x;
    const bf16* router_w;
    const bf16* router_b;
    const bf16* gate_up;
    const bf16* down;
    const bf16* sgu;  // shared gate_up [2Is, H]
    const bf16* sd;   // shared down [H, Is]
    const bf16* sg;   // shared gate [1, H]
    const bf16* residual;
    bf16* out;
    float* logits;    // [T, ldl] fp32: E router scores, then the shared-gate score at column E
    int32_t* ids;
    float* topw;
    float* sgate;
    int32_t* counts;
    int32_t* offsets;
    int32_t* perm;
    int32_t* inv;
    int32_t* lr;      // rank of each pair among its expert's pairs within its token block
    int32_t* cntb;    // [nb, E] pairs per expert per token block
    int32_t* base;    // [nb, E] first perm position of each (block, expert)
    int32_t* act;     // experts with pairs, ascending; count in hdr->n_act
    bf16* h;          // [P + T, Imax] gated activations
    float* Y;         // [T, K+1, H] weighted expert outputs, slot K = shared expert (fp32 path)
    bf16* Yb;         // the same in bf16 (tensor-core path)
    GemmGroup* up_groups;
    GemmGroup* dn_groups;
    int32_t* up_tiles;  // [n_groups + 1] first tile of each gate_up group
    int32_t* dn_tiles;
    int32_t* n_groups;
    UpRec* uprec;     // routed gate_up records (few-token path), nullptr when not produced
    uint64_t* dlog;   // [T, E+1] router scores tagged with their call (fused few-token kernel)
    uint64_t* dh;     // [P+T, Imax/2] gated activation pairs tagged with their call (same kernel)
    uint64_t* dx;     // [H/2] the token row's 32-bit words tagged with their call (T = 1, host rows)
    WsHeader* hdr;
    uint64_t wait_ns;   // time limit of the bounded waits of the one-token and streaming kernels
    int test_suppress;  // MOE_TEST_SUPPRESS_* (testing aid; 0 in normal use)
    bool gemm;
    bool x_host;      // x is pinned host memory mapped into the device (one-token kernel only)
    int flags;        // moe_dims.flags (MOE_FLAG_BF16_SCORES)
    int T, H, E, K, I, Is, Imax, ldl, nb;
    int64_t P;
    int num_sms;
};

// Bookkeeping around every kernel launch: the process-wide launch counter and the optional
// CUDA-event trace of moe_set_trace. Call before/after each <<<...>>>.
void trace_begin(int kernel, cudaStream_t s);
void trace_end(int kernel, cudaStream_t s);

#define MOE_LAUNCH(kernel_id, stream, launch_expr) \
    do {                                           \
        trace_begin(kernel_id, stream);            \
        launch_expr;                               \
        trace_end(kernel_id, stream);              \
    } while (0)

// Grouped-GEMM description consumed by the tensor-core kernel. With dense_rows > 0 there is a
// single group of dense_rows rows (the router) and the tables are not read.
// N tiles of the grouped GEMMs: gate_up takes FH gate rows and the FH matching up rows
// (FH = 128, else 64), down takes 256 output rows (else 128).
inline int gemm_up_half(const LayerArgs& a) { return (a.I % 128 == 0 && a.Is % 128 == 0) ? 128 : 64; }
inline int gemm_down_bn(const LayerArgs& a) { return (a.H % 256 == 0) ? 256 : 128; }

// Launch as a programmatic dependent of the previous kernel on the stream: the kernel may
// start while that one runs and must execute grid_dep_wait before touching its outputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct GemmPlan {
    const GemmGroup* groups;
    const int32_t* tile_start;
    const int32_t* n_groups;
    int dense_rows, dense_tiles;
    int k_routed, k_shared;       // reduction length of routed / shared groups
    int up_off_routed, up_off_shared;  // row offset of the up half in a merged gate_up block
    uint32_t* err;
};

cudaError_t launch_router(const LayerArgs& a, cudaStream_t s);
cudaError_t launch_route_fused(const LayerArgs& a, cudaStream_t s);
bool route_small_supported(const LayerArgs& a);
cudaError_t launch_fetch_experts(const LayerArgs& a, const bf16* host_gate_up, const bf16* host_down,
                                 bf16* shadow_gate_up, bf16* shadow_down, cudaStream_t s);
// dst = src, bytes a multiple of 16; one side pinned host memory mapped into the device.
cudaError_t launch_copy_rows(const void* src, void* dst, size_t bytes, int num_sms, cudaStream_t s);
cudaError_t launch_router_stats(const LayerArgs& a, float* P, float* f, float* loss, cudaStream_t s);
cudaError_t launch_route_small(const LayerArgs& a, cudaStream_t s);
bool route_cluster_supported(const LayerArgs& a);
cudaError_t launch_route_cluster(const LayerArgs& a, cudaStream_t s);
cudaError_t launch_router_gemm(const LayerArgs& a, cudaStream_t s);
cudaError_t launch_expert_gemms(const LayerArgs& a, cudaStream_t s);
cudaError_t launch_combine(const LayerArgs& a, cudaStream_t s);
cudaError_t launch_combine_pdl(const LayerArgs& a, cudaStream_t s);
bool stream_supported(const LayerArgs& a);
bool decode_fused_supported(const LayerArgs& a);
cudaError_t launch_decode_fused(const LayerArgs& a, cudaStream_t s);
cudaError_t launch_stream_experts(const LayerArgs& a, cudaStream_t s);
cudaError_t launch_dispatch(const LayerArgs& a, cudaStream_t s);
cudaError_t launch_experts(const LayerArgs& a, cudaStream_t s);
cudaError_t launch_rmsnorm(const bf16* x, const bf16* gamma, float eps, bf16* xn, int T, int H, cudaStream_t s);

}  // namespace moe
