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
    float* Y;         // [T, K+1, H] weighted expert outputs, slot K = shared expert
    WsHeader* hdr;
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

cudaError_t launch_router(const LayerArgs& a, cudaStream_t s);
cudaError_t launch_dispatch(const LayerArgs& a, cudaStream_t s);
cudaError_t launch_experts(const LayerArgs& a, cudaStream_t s);
cudaError_t launch_rmsnorm(const bf16* x, const bf16* gamma, float eps, bf16* xn, int T, int H, cudaStream_t s);

}  // namespace moe
