// noalloc.cu -- moe_route_noalloc: few-token routing whose scratch lives in a fixed device
// array compiled into the library, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all (and so cannot provide the workspace that
// moe_route takes): a plugin inside a host framework that owns every device allocation, a
// serving engine that reserved all of HBM up front for weights and caches, or a latency-
// critical path where an allocation's implicit synchronisation or failure under memory
// pressure is not acceptable. For them this entry point runs the same fused routing kernel
// as moe_route (scores, top-K, renormalisation, dispatch) with its scratch in the static
// array below. The array is part of the library image: every GPU that loads the library holds
// its kRouteScratchBytes until the process exits.
#include <stdint.h>
#include <string.h>

#include <mutex>

#include <cuda.h>

#include "launch.h"

namespace moe {

// Scratch of one call: header, scores [T, E+1 rounded to 4] fp32, shared-gate values [T],
// per-pair ranks and inverse positions [T*K], the list of used experts [E+1].
constexpr size_t kRouteScratchBytes = 80 * 1024;

static __device__ __align__(256) uint8_t g_route_scratch[kRouteScratchBytes];

namespace {

struct ScratchLayout {
    size_t hdr, logits, sgate, lr, inv, act, total;
};

ScratchLayout scratch_layout(const moe_dims& d) {
    ScratchLayout s;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t r = o; o = align256(o + bytes); return r; };
    const size_t T = (size_t)d.T, P = (size_t)d.T * d.K, ldl = (size_t)((d.E + 1 + 3) & ~3);
    s.hdr = take(sizeof(WsHeader));
    s.logits = take(T * ldl * 4);
    s.sgate = take(T * 4);
    s.lr = take(P * 4);
    s.inv = take(P * 4);
    s.act = take((size_t)(d.E + 1) * 4);
    s.total = o;
    return s;
}

// The current CUDA context (the driver's handle), or nullptr when it cannot be read.
CUcontext current_context() {
    typedef CUresult (*GetCurrent)(CUcontext*);
    static GetCurrent fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (GetCurrent)p;
    });
    CUcontext ctx = nullptr;
    if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
    return ctx;
}

// Device address of the scratch array on the current device, looked up with that device
// current and cached per device together with the context it belongs to: after a reset of
// the device (a new primary context, where the library image and the array may have moved)
// the address is looked up again.
void* scratch_address(int dev, cudaError_t* err) {
    static std::mutex mu;
    static void* addr[128] = {};
    static CUcontext owner[128] = {};
    if (dev < 0 || dev >= 128) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    const CUcontext ctx = current_context();
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] || !ctx || owner[dev] != ctx) {
        void* p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_route_scratch);
        if (*err != cudaSuccess) return nullptr;
        addr[dev] = p;
        owner[dev] = current_context();
    }
    *err = cudaSuccess;
    return addr[dev];
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_route_noalloc(const moe_dims* d, const void* x, const moe_weights* w, int32_t* ids,
                                        float* topk_w, int32_t* counts, int32_t* offsets, int32_t* perm,
                                        void* stream) {
    if (!d || (d->flags & ~MOE_FLAG_BF16_SCORES)) return MOE_ERR_INVALID_ARG;
    Plan p;
    if (!make_plan(*d, &p)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (d->T > kFusedRouteTokens) return MOE_ERR_UNSUPPORTED_SHAPE;
    const ScratchLayout L = scratch_layout(*d);
    if (L.total > kRouteScratchBytes) return MOE_ERR_UNSUPPORTED_SHAPE;
    cudaStream_t s = (cudaStream_t)stream;
    if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
    if (d->T == 0) {
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * d->E, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (d->E + 1), s);
        return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    if (!x || !w || !w->router_w || !w->shared_gate || !ids || !topk_w || !perm) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w->router_w) || !aligned16(w->shared_gate) ||
        (w->router_b && !aligned16(w->router_b)) || !aligned16(ids) || !aligned16(topk_w) || !aligned16(counts) ||
        !aligned16(offsets) || !aligned16(perm))
        return MOE_ERR_MISALIGNED;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    char* base = (char*)scratch_address(dev, &e);
    if (!base) return MOE_ERR_CUDA;
    LayerArgs a;
    memset(&a, 0, sizeof a);
    a.x = (const bf16*)x;
    a.router_w = (const bf16*)w->router_w;
    a.router_b = (const bf16*)w->router_b;
    a.sg = (const bf16*)w->shared_gate;
    a.hdr = (WsHeader*)(base + L.hdr);
    a.logits = (float*)(base + L.logits);
    a.sgate = (float*)(base + L.sgate);
    a.lr = (int32_t*)(base + L.lr);
    a.inv = (int32_t*)(base + L.inv);
    a.act = (int32_t*)(base + L.act);
    a.ids = ids;
    a.topw = topk_w;
    a.counts = counts;
    a.offsets = offsets;
    a.perm = perm;
    a.flags = d->flags;
    a.T = p.T; a.H = p.H; a.E = p.E; a.K = p.K; a.I = p.I; a.Is = p.Is;
    a.Imax = p.Imax; a.ldl = p.ldl; a.nb = p.nb; a.P = p.P;
    // the array keeps the previous call's contents: the header (completion ticket, error word)
    // must start at zero
    e = cudaMemsetAsync(a.hdr, 0, sizeof(WsHeader), s);
    if (e == cudaSuccess) e = launch_route_fused(a, s);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
