/*
 * moe.h -- C ABI of the GB300 (sm_103a) sparse Mixture-of-Experts feed-forward layer.
 *
 * The layer (per token t, "Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256 Experts):
 *   l      = x[t] . Wr^T (+ br)                        router scores, fp32 accumulate
 *   p      = softmax(l)                                 over the E experts
 *   ids    = the K experts of highest p, slot 0 first; equal scores go to the lower index
 *   w_k    = p[ids_k] / sum_j p[ids_j]                  renormalised to sum to 1
 *   y      = sigmoid(x[t] . ws) * S(x[t]) + sum_k w_k * X_{ids_k}(x[t])
 *   out[t] = residual[t] + y                            (residual optional)
 * where every expert is a SwiGLU network X(x) = (SiLU(x . Wg^T) * (x . Wu^T)) . Wd^T
 * (same page, Experts and Shared Expert; "Qwen3.6 35B-A3B", Blocks: SparseMoe, SwiGlu).
 *
 * Data types and layouts (bf16 = IEEE bfloat16 bit patterns; all row-major, [Out, In]
 * like `Linear` in "Qwen3.6 35B-A3B", Blocks: Linear):
 *   x, residual, out  [T, H]        bf16
 *   router_w          [E, H]        bf16       router_b [E] bf16, optional
 *   gate_up           [E, 2I, H]    bf16       rows [0,I) of each expert = gate, [I,2I) = up
 *   down              [E, H, I]     bf16
 *   shared_gate_up    [2Is, H]      bf16       same split as gate_up
 *   shared_down       [H, Is]       bf16
 *   shared_gate       [1, H]        bf16       (no bias)
 *
 * Ownership and execution. The caller owns every buffer; all pointers are device pointers
 * (16-byte aligned) unless stated otherwise. The library allocates nothing on the call
 * path: scratch lives in a caller-provided device workspace of moe_workspace_size() bytes,
 * zero-filled once before its first use (moe_workspace_init does that); the library leaves
 * it ready for the next call. Calls are asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream). Argument errors are detected on the host and returned before
 * anything is launched. A workspace must not be used by two calls that may overlap in time.
 * Weights are only read. A call may start reading them (never x, residual, out or the
 * workspace) while the kernel before it on `stream` is still finishing (programmatic
 * dependent launch), so that kernel must not be one that writes the weights: after writing
 * weights on `stream`, run any other work there, or synchronize, before the call.
 * One token at the pages' layer shape (H = 2048, I = Is = 512, T = 1) runs as one grid of one
 * CTA per SM whose CTAs exchange values with one another, so it needs every SM at once:
 * kernels on other streams that hold SMs longer than the wait limit (about 1 s) make the
 * call end with MOE_ERR_TIMEOUT in the workspace's error word rather than wait for them.
 * Results are deterministic: the same inputs give bit-identical outputs on every call.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Runtime dimensions: T tokens (B*S flattened; "Qwen3.6 35B-A3B", SparseMoe.forward takes
 * [B, S, H]), H hidden width, E routed experts, K experts per token, I routed inner width,
 * Is shared inner width. Supported: T >= 0, 128 <= H <= 8192 with H % 128 == 0,
 * 1 <= K <= 8, K <= E <= 256, 64 <= I, Is <= 2048 with I % 64 == 0 and Is % 64 == 0,
 * T * (K + 1) < 2^31. T == 0 is a valid no-op.
 * flags: 0, or MOE_FLAG_BF16_SCORES; any other bit is rejected with MOE_ERR_INVALID_ARG
 * before anything runs (moe_workspace_size ignores flags). */
typedef struct {
    int32_t T, H, E, K, I, Is;
    int32_t flags;
} moe_dims;

/* bf16-typed router outputs ("Qwen3.6 35B-A3B", Blocks: SparseMoe types `gate:
 * Linear<H, Experts, T>`, `shared_expert_gate: Linear<H, 1, T>` and `ranks(logits: Tensor[R,
 * Experts; T])` with T = bf16): each router score and the shared-gate score, accumulated in
 * fp32 with the bias added, is rounded to the nearest bf16 (ties to even) before the softmax,
 * the ranking and the sigmoid. Equal rounded scores rank the lower expert index first.
 * Without the flag the fp32 scores are used unrounded. */
#define MOE_FLAG_BF16_SCORES 1

/* Pointers to one layer's weights, in device memory (moe_forward_host_experts takes gate_up
 * and down in mapped host memory instead); router_b may be NULL. */
typedef struct {
    const void* router_w;
    const void* router_b;
    const void* gate_up;
    const void* down;
    const void* shared_gate_up;
    const void* shared_down;
    const void* shared_gate;
} moe_weights;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,         /* NULL pointer or negative size                       */
    MOE_ERR_UNSUPPORTED_SHAPE = 2,   /* dims outside the supported range above              */
    MOE_ERR_MISALIGNED = 3,          /* a pointer is not 16-byte aligned                    */
    MOE_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes < moe_workspace_size(d)                    */
    MOE_ERR_CUDA = 5,                /* a CUDA launch or runtime call failed                */
    MOE_ERR_TIMEOUT = 6,             /* a bounded device-side wait gave up                  */
    MOE_ERR_DEVICE = 7               /* a kernel flagged bad data (e.g. a non-finite score) */
} moe_status;

/* Bytes of device workspace that moe_route / moe_forward need for dims d (0 if d is
 * unsupported). Host-only; never fails otherwise. */
size_t moe_workspace_size(const moe_dims* d);

/* Zero-fill a workspace on `stream` (cudaMemsetAsync). Needed once after allocation. */
moe_status moe_workspace_init(void* workspace, size_t ws_bytes, void* stream);

/* Routing only: router scores, softmax, top-K, renormalisation, and the dispatch of the
 * (token, slot) pairs to experts ("Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256
 * Experts, Router; "One Token Through Qwen3.6", The Router).
 *   x        [T, H] bf16 in
 *   ids      [T, K] int32 out: expert of each slot, slot 0 = highest score
 *   topk_w   [T, K] fp32  out: renormalised routing weights (sum to 1 per token)
 *   counts   [E]    int32 out: pairs routed to each expert
 *   offsets  [E+1]  int32 out: exclusive prefix sum of counts, offsets[E] = T*K
 *   perm     [T*K]  int32 out: values t*K+k grouped by expert (ascending), tokens
 *                              ascending within an expert
 * Integer outputs are exact and reproducible; topk_w is fp32. */
moe_status moe_route(const moe_dims* d, const void* x, const moe_weights* w, int32_t* ids, float* topk_w,
                     int32_t* counts, int32_t* offsets, int32_t* perm, void* workspace, size_t ws_bytes,
                     void* stream);

/* The whole layer: out = residual + MoE(x), or MoE(x) when residual is NULL. out must not
 * overlap x; it may be the same buffer as residual. Routed and shared expert outputs are
 * summed per token in a fixed order (residual, shared, slot 0 .. K-1) in fp32 and rounded
 * to bf16 once. */
moe_status moe_forward(const moe_dims* d, const void* x, const moe_weights* w, const void* residual, void* out,
                       void* workspace, size_t ws_bytes, void* stream);

/* The layer with its token rows in HOST memory (the decode loop's view: a token's hidden
 * state arrives from the host and the layer's output goes back to it). On `stream`, in this
 * order: host_x is copied into dev_x, host_residual (when not NULL) into dev_out, moe_forward
 * runs on (dev_x, dev_out as residual or none, dev_out), and dev_out is copied into host_out.
 * Up to 1 MB of rows (T*H*2 bytes) in pinned host memory mapped into the device move by a
 * small copy kernel (MOE_KERNEL_COPY_ROWS) over the host link; pageable or larger buffers by
 * cudaMemcpyAsync (pageable ones work, but the driver stages them and may block the calling
 * thread). One token at the shape moe_forward runs in its one-token kernel, with host_x,
 * host_out and host_residual (when given) all pinned, mapped and 16-byte aligned, takes one
 * launch and no copy: that kernel reads x and the residual and writes out on the host rows
 * themselves, and dev_x / dev_out are left as they were. host_out holds the result once
 * `stream` has passed the call.
 *   host_x, host_residual, host_out  [T, H] bf16, host memory (pinned or pageable);
 *                                    host_out may be the same buffer as host_x or host_residual
 *   dev_x, dev_out                   [T, H] bf16, device memory, 16-byte aligned, disjoint
 * Errors: MOE_ERR_INVALID_ARG when host_x or host_out is NULL, a host buffer is device memory
 * or dev_x / dev_out is not device memory (cudaPointerGetAttributes, before any copy);
 * otherwise as moe_forward with x = dev_x and out = dev_out. */
moe_status moe_forward_host_io(const moe_dims* d, const void* host_x, const moe_weights* w, const void* host_residual,
                               void* host_out, void* dev_x, void* dev_out, void* workspace, size_t ws_bytes,
                               void* stream);

/* Routed experts resident in host memory ("One Token Through Qwen3.6", Where the Weights
 * Live: checkpoint on disk, system RAM, GPU memory, kernels; the routing decides which expert
 * weights a layer needs). Same layer as moe_forward, but w->gate_up and w->down point to HOST
 * memory that is pinned and mapped into the device address space (cudaHostAlloc, or
 * cudaHostRegister with mapping); every other weight, x, out, residual and the workspace are
 * device memory as for moe_forward. After the routing, one kernel copies the gate_up and down
 * rows of the experts this call touches over the host link into `shadow`, device memory of
 * moe_expert_shadow_size(d) bytes laid out like [E, 2I, H] followed by [E, H, I] bf16 (only
 * the touched experts' rows are written; the rest is left as it was), and the experts run
 * from there. One shadow can serve every layer of a model in turn.
 * Errors: MOE_ERR_INVALID_ARG when gate_up or down is not registered host memory mapped into
 * the device (checked with cudaPointerGetAttributes before any launch), when the registered
 * allocation holding gate_up or down ends before the whole [E, 2I, H] or [E, H, I] tensor
 * (checked where the driver reports the allocation's range), or shadow is NULL,
 * MOE_ERR_MISALIGNED when shadow is not 16-byte aligned, MOE_ERR_WORKSPACE_TOO_SMALL when
 * shadow_bytes < moe_expert_shadow_size(d); otherwise as moe_forward. */
size_t moe_expert_shadow_size(const moe_dims* d);
moe_status moe_forward_host_experts(const moe_dims* d, const void* x, const moe_weights* w, const void* residual,
                                    void* out, void* shadow, size_t shadow_bytes, void* workspace, size_t ws_bytes,
                                    void* stream);

/* RMSNorm of the pre-MoE norm ("RMSNorm -> MoE FFN -> +residual", "Qwen3.6-35B-A3B --
 * Architecture Overview", Stage 2; "Qwen3.6 35B-A3B", Blocks: RmsNorm):
 *   xn[t,h] = bf16( x[t,h] / sqrt(mean_h x[t,h]^2 + eps) * gamma[h] )   (fp32 arithmetic)
 * Uses d->T and d->H only. gamma [H] bf16 may be NULL (all ones). xn must not overlap x. */
moe_status moe_rmsnorm(const moe_dims* d, const void* x, const void* gamma, float eps, void* xn, void* stream);

/* Synchronise `stream`, then read and clear the device error word kept in `workspace`:
 * MOE_OK, MOE_ERR_DEVICE (a kernel saw a non-finite router score) or MOE_ERR_TIMEOUT. */
moe_status moe_last_device_error(void* workspace, void* stream);

/* Where an intermediate lives in the workspace after moe_forward (for inspection):
 *   tap 0  h      [T*K + T, max(I,Is)] bf16: gated activations, routed rows in perm order
 *                                             then the T shared-expert rows in token order
 *   tap 1  Y      [T, K+1, H] weighted expert outputs per slot, slot K = shared; fp32
 *                 when T < 256 (weight-streaming path), bf16 from T >= 256 (tensor-core
 *                 path): bytes / (T*(K+1)*H) tells which
 *   tap 2  sgate  [T] fp32: sigmoid(x . ws)
 *   tap 3  ids    [T, K] int32      tap 4  topk_w [T, K] fp32
 * Row strides are the widths given. Returns MOE_ERR_INVALID_ARG for an unknown tap. */
moe_status moe_workspace_tap(const moe_dims* d, int tap, size_t* offset, size_t* bytes);

/* Load-balancing statistics of one routing call ("Qwen3.6-35B-A3B -- Architecture Overview",
 * MoE FFN: 256 Experts, Load Balancing: an auxiliary loss, coefficient 0.001, penalises uneven
 * expert utilisation across the batch). The page gives no formula; this computes, for the T
 * tokens of x, the quantities such a loss is built from and the product form that is
 * smallest under uniform routing:
 *   P[e] = (1/T) sum_t softmax(router scores of token t)[e]   (full softmax over the E scores)
 *   f[e] = (tokens routed to expert e) / (T*K)
 *   loss = 0.001 * E * sum_e f[e] * P[e]
 * P, f: [E] fp32; loss: one fp32; all device pointers (P and f 16-byte aligned), owned by the
 * caller. The routing is the same as moe_route's (and it leaves the same results in the
 * workspace). Every sum runs in a fixed order, so repeated calls give identical bits.
 * T = 0 writes zeros. Errors as moe_route. */
moe_status moe_router_stats(const moe_dims* d, const void* x, const moe_weights* w, float* P, float* f, float* loss,
                            void* workspace, size_t ws_bytes, void* stream);

/* Kernels of the layer, for moe_set_trace. */
enum {
    MOE_KERNEL_ROUTER_SCORES = 0,   /* router + shared-gate scores                 */
    MOE_KERNEL_ROUTER_TOPK = 1,     /* softmax, top-K, renormalisation             */
    MOE_KERNEL_DISPATCH_LOCAL = 2,  /* per-block expert counts and ranks           */
    MOE_KERNEL_DISPATCH_SCAN = 3,   /* offsets and block bases                     */
    MOE_KERNEL_DISPATCH_SCATTER = 4,/* dispatch permutation                        */
    MOE_KERNEL_GATE_UP = 5,         /* gate/up projections + SwiGLU, all groups    */
    MOE_KERNEL_DOWN = 6,            /* down projection + routing-weight scale      */
    /* (from T >= 256 the router scores, gate_up and down run as tensor-core GEMMs) */
    MOE_KERNEL_COMBINE = 7,         /* fixed-order sum into the residual           */
    MOE_KERNEL_RMSNORM = 8,
    MOE_KERNEL_SHARED_GATE = 9,     /* not launched: the top-K kernel scores the shared gate */
    MOE_KERNEL_GATHER = 10,         /* not launched: the gate_up GEMM gathers the token rows from x */
    MOE_KERNEL_GEMM_PLAN = 11,      /* not launched: the dispatch scan writes the GEMM tables */
    MOE_KERNEL_DECODE_FUSED = 12,   /* whole layer in one persistent kernel (T = 1) */
    MOE_KERNEL_ROUTER_STATS = 13,   /* load-balancing statistics (moe_router_stats) */
    MOE_KERNEL_FETCH_EXPERTS = 14,  /* touched experts copied from host memory (moe_forward_host_experts) */
    MOE_KERNEL_COPY_ROWS = 15,      /* token rows to or from mapped host memory (moe_forward_host_io) */
    MOE_KERNEL_COUNT = 16
};

/* Benchmarking aid. While set, every launch of `kernel` made by this library records
 * start_events[i] on its stream just before the launch and stop_events[i] just after it,
 * i = 0, 1, ... cycling modulo n_events (cudaEvent_t handles owned by the caller), so the
 * caller can read that kernel's duration with cudaEventElapsedTime. n_events = 0 clears it.
 * Process-wide state, not thread-safe; no effect on results. */
moe_status moe_set_trace(int kernel, void* const* start_events, void* const* stop_events, int n_events);

/* Number of kernels this library has launched in this process so far. */
uint64_t moe_launch_count(void);

/* Testing aid for the bounded-wait path (the paper has no counterpart). Every wait of the
 * one-token kernel (moe_forward with T = 1 at the page's layer shape) and of the streaming
 * expert kernels (2 <= T < 256) gives up after a time limit, sets MOE_ERR_TIMEOUT in the
 * workspace's error word and lets the kernel run to its end with in-range indices; the calls
 * after a timeout need moe_workspace_init on that workspace. This sets, process-wide and for
 * the calls made after it returns:
 *   wait_ns   the time limit of those waits in nanoseconds; 0 restores the default (~1 s);
 *             at most 10 s;
 *   suppress  0 in normal use, or one signal to hold back so that a wait runs out:
 *             MOE_TEST_SUPPRESS_SCORE  CTA 1 of the one-token kernel does not publish its
 *                                      router scores (every CTA's wait for the scores runs out);
 *             MOE_TEST_SUPPRESS_STAGE  CTA 0 of the streaming gate_up kernel (9 <= T < 256)
 *                                      never loads its first ring stage (its consumers' wait
 *                                      on the stage's mbarrier runs out).
 * Results of calls made while a signal is held back are meaningless; no call faults, traps or
 * hangs. Returns MOE_ERR_INVALID_ARG for another suppress value or wait_ns above 10 s. Not
 * thread-safe with concurrent calls of the library. */
#define MOE_TEST_SUPPRESS_SCORE 1
#define MOE_TEST_SUPPRESS_STAGE 2
moe_status moe_test_set_wait(uint64_t wait_ns, int suppress);

/* Routing without any device allocation by the caller (the paper has no counterpart: this is
 * for callers of this library that cannot call cudaMalloc, such as a plugin whose host
 * framework owns every device allocation, an engine that reserved all of HBM up front, or a
 * latency-critical path that cannot take an allocation's synchronisation or its failure).
 * Same inputs, outputs and results as moe_route, but no workspace: its scratch is a fixed
 * 80 KiB array inside the library, held by every GPU that loads the library until the
 * process exits. Limits: T <= 64 and the scratch layout must fit (any E <= 256, K <= 8 fit);
 * larger sizes return MOE_ERR_UNSUPPORTED_SHAPE before anything is launched.
 * The first call on a device looks up the array's device address on the current device
 * (cudaGetSymbolAddress); make that first call before any stream capture. The address is
 * kept per device and context: the first call after a reset of the device looks it up again. Every call shares
 * the one array: calls that may overlap on the GPU (different streams, or devices sharing it)
 * race and must be ordered by the caller. Each call clears the part that must start at zero.
 * A non-finite router score is not reported (there is no workspace error word). */
moe_status moe_route_noalloc(const moe_dims* d, const void* x, const moe_weights* w, int32_t* ids, float* topk_w,
                             int32_t* counts, int32_t* offsets, int32_t* perm, void* stream);

/* Human-readable name of a status. Never NULL. */
const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
