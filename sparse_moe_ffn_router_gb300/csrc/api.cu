// api.cu -- the C-ABI entry points declared in include/moe.h: host-side validation, the
// workspace plan, and the stream-ordered launch sequence of the layer.
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include <cuda.h>
#include <vector>

#include "launch.h"

namespace moe {

static std::atomic<uint64_t> g_launches{0};

// Testing aid (moe_test_set_wait): time limit of the bounded device waits and the signal held back.
static std::atomic<uint64_t> g_wait_ns{kWaitNs};
static std::atomic<int> g_suppress{0};

struct TraceSlot {
    int n = 0;
    int i = 0;
    std::vector<void*> start, stop;
};
static TraceSlot g_trace[MOE_KERNEL_COUNT];

// Inside a stream capture an event record must be "external" to become an event node of the
// graph (a plain record only orders the capture); outside a capture only a plain record is valid.
static void trace_record(void* ev, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(s, &cs);
    if (cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags((cudaEvent_t)ev, s, cudaEventRecordExternal);
    else
        cudaEventRecord((cudaEvent_t)ev, s);
}

void trace_begin(int kernel, cudaStream_t s) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    TraceSlot& t = g_trace[kernel];
    if (t.n) trace_record(t.start[t.i % t.n], s);
}

void trace_end(int kernel, cudaStream_t s) {
    TraceSlot& t = g_trace[kernel];
    if (t.n) {
        trace_record(t.stop[t.i % t.n], s);
        ++t.i;
    }
}

}  // namespace moe

using namespace moe;

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

int sm_count() {
    static int cache[128];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 148;
    }
    return cache[dev];
}

// Common validation of moe_route / moe_forward. On success fills the plan and the
// workspace-backed fields of the argument block.
moe_status prepare(const moe_dims* d, const void* x, const moe_weights* w, void* ws, size_t ws_bytes, Plan* p,
                   LayerArgs* a) {
    if (!d || (d->flags & ~MOE_FLAG_BF16_SCORES)) return MOE_ERR_INVALID_ARG;
    if (!make_plan(*d, p)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (d->T == 0) return MOE_OK;
    if (!x || !w || !ws || !w->router_w || !w->gate_up || !w->down || !w->shared_gate_up || !w->shared_down ||
        !w->shared_gate)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(ws) || !aligned16(w->router_w) || !aligned16(w->gate_up) ||
        !aligned16(w->down) || !aligned16(w->shared_gate_up) || !aligned16(w->shared_down) ||
        !aligned16(w->shared_gate) || (w->router_b && !aligned16(w->router_b)))
        return MOE_ERR_MISALIGNED;
    if (ws_bytes < p->total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    memset(a, 0, sizeof *a);
    char* base = (char*)ws;
    a->flags = d->flags;
    a->x = (const bf16*)x;
    a->router_w = (const bf16*)w->router_w;
    a->router_b = (const bf16*)w->router_b;
    a->gate_up = (const bf16*)w->gate_up;
    a->down = (const bf16*)w->down;
    a->sgu = (const bf16*)w->shared_gate_up;
    a->sd = (const bf16*)w->shared_down;
    a->sg = (const bf16*)w->shared_gate;
    a->hdr = (WsHeader*)(base + p->o_hdr);
    a->logits = (float*)(base + p->o_logits);
    a->ids = (int32_t*)(base + p->o_ids);
    a->topw = (float*)(base + p->o_topw);
    a->sgate = (float*)(base + p->o_sgate);
    a->counts = (int32_t*)(base + p->o_counts);
    a->offsets = (int32_t*)(base + p->o_offsets);
    a->perm = (int32_t*)(base + p->o_perm);
    a->inv = (int32_t*)(base + p->o_inv);
    a->lr = (int32_t*)(base + p->o_lr);
    a->cntb = (int32_t*)(base + p->o_cntb);
    a->base = (int32_t*)(base + p->o_base);
    a->act = (int32_t*)(base + p->o_act);
    a->h = (bf16*)(base + p->o_h);
    a->Y = (float*)(base + p->o_y);
    a->Yb = (bf16*)(base + p->o_y);
    a->up_groups = (GemmGroup*)(base + p->o_upg);
    a->dn_groups = (GemmGroup*)(base + p->o_dng);
    a->up_tiles = (int32_t*)(base + p->o_upt);
    a->dn_tiles = (int32_t*)(base + p->o_dnt);
    a->n_groups = &a->hdr->n_groups;
    a->uprec = p->T <= kRecTokens ? (UpRec*)(base + p->o_uprec) : nullptr;
    a->dlog = p->T <= kRecTokens ? (uint64_t*)(base + p->o_dlog) : nullptr;
    a->dh = p->T <= kRecTokens ? (uint64_t*)(base + p->o_dh) : nullptr;
    a->dx = p->T == 1 ? (uint64_t*)(base + p->o_dx) : nullptr;
    a->gemm = p->gemm;
    a->x_host = false;
    a->T = p->T; a->H = p->H; a->E = p->E; a->K = p->K; a->I = p->I; a->Is = p->Is;
    a->Imax = p->Imax; a->ldl = p->ldl; a->nb = p->nb; a->P = p->P;
    a->num_sms = sm_count();
    a->wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    a->test_suppress = g_suppress.load(std::memory_order_relaxed);
    return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Router scores, top-K and dispatch: one fused launch for few tokens, else separate kernels.
// Routing: up to 8 tokens on one thread-block cluster (16 CTAs where the device allows, else
// 8); 9..255 tokens in two kernels (tensor-
// pipe scores, then top-K and the whole dispatch in one CTA); from 256 tokens the scores as a
// tcgen05 GEMM, top-K one warp per token and the three block-parallel dispatch kernels. (The
// single-kernel routing of up to 64 tokens is used only by the fixed-scratch entry point.)
constexpr int kFusedMaxTokens = 1;  // largest T that moe_forward runs in the fused decode kernel
constexpr size_t kKernelCopyBytes = 1 << 20;  // largest host-row transfer moe_forward_host_io gives k_copy_rows

// The output buffers of a layer call: out given, 16-byte aligned, not overlapping x, and
// either equal to the residual or apart from it.
moe_status check_output(const moe_dims* d, const void* x, const void* residual, const void* out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(out) || (residual && !aligned16(residual))) return MOE_ERR_MISALIGNED;
    const size_t act_bytes = (size_t)d->T * d->H * 2;
    if (overlap(out, act_bytes, x, act_bytes)) return MOE_ERR_INVALID_ARG;
    if (residual && residual != out && overlap(out, act_bytes, residual, act_bytes)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// Host memory that is pinned and mapped into the device address space; dev receives the
// address kernels use.
bool host_mapped(const void* p, const void** dev) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // clear the error this query left
        return false;
    }
    if (at.type != cudaMemoryTypeHost || !at.devicePointer) return false;
    *dev = at.devicePointer;
    return true;
}

// Whether the pinned allocation that holds p extends at least `bytes` past p. The driver's
// record of the allocation's range is read through cuPointerGetAttribute (looked up once); when
// the driver cannot report a range, the check passes and the caller's sizes are trusted.
bool host_range_covers(const void* p, size_t bytes) {
    typedef CUresult (*GetAttr)(void*, CUpointer_attribute, CUdeviceptr);
    static GetAttr fn = nullptr;
    static bool looked = false;
    if (!looked) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (GetAttr)f;
        looked = true;
    }
    if (!fn) return true;
    CUdeviceptr start = 0;
    size_t size = 0;
    if (fn(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, (CUdeviceptr)(uintptr_t)p) != CUDA_SUCCESS ||
        fn(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, (CUdeviceptr)(uintptr_t)p) != CUDA_SUCCESS || size == 0)
        return true;
    return (uintptr_t)p + bytes <= (uintptr_t)start + size;
}

// The kind of memory p points to (cudaMemoryTypeUnregistered for pageable host memory), or
// -1 when the query fails.
int memory_type(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // clear the error this query left
        return -1;
    }
    return (int)at.type;
}

// Host memory, pinned or pageable: what the host-side token rows may live in.
bool host_side(const void* p) {
    const int t = memory_type(p);
    return t == cudaMemoryTypeHost || t == cudaMemoryTypeUnregistered;
}

// Routing: scores, top-K and the dispatch tables.
cudaError_t launch_routing(const LayerArgs& a, cudaStream_t s) {
    if (route_cluster_supported(a)) return launch_route_cluster(a, s);
    if (route_small_supported(a)) return launch_route_small(a, s);
    cudaError_t e = launch_router(a, s);
    if (e == cudaSuccess) e = launch_dispatch(a, s);
    return e;
}

// The experts and the combine, once the routing tables are in the workspace.
cudaError_t launch_after_routing(const LayerArgs& a, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    if (a.gemm) {
        e = launch_expert_gemms(a, s);
        if (e == cudaSuccess) e = launch_combine(a, s);
    } else if (stream_supported(a)) {
        e = launch_stream_experts(a, s);  // the combine runs as its programmatic dependent
    } else {
        e = launch_experts(a, s);
        if (e == cudaSuccess) e = launch_combine(a, s);
    }
    return e;
}

// The whole layer, once its arguments are checked. One token: one persistent launch. From two
// tokens on the fused kernel's shared memory holds a smaller ring (the token rows and h rows
// grow with T) and the router kernel + streaming expert kernels are faster (measured per
// layer: T=2 37.7 vs 44.7 us, T=4 55.8 vs 85.7 us, T=8 84.8 vs 168.3 us).
cudaError_t launch_layer(const LayerArgs& a, cudaStream_t s) {
    if (a.T <= kFusedMaxTokens && decode_fused_supported(a)) return launch_decode_fused(a, s);
    cudaError_t e = launch_routing(a, s);
    if (e == cudaSuccess) e = launch_after_routing(a, s);
    return e;
}

}  // namespace

extern "C" size_t moe_workspace_size(const moe_dims* d) {
    Plan p;
    if (!d || !make_plan(*d, &p)) return 0;
    return p.total;
}

extern "C" moe_status moe_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
    if (!workspace) return MOE_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(workspace, 0, ws_bytes, (cudaStream_t)stream));
}

extern "C" moe_status moe_route(const moe_dims* d, const void* x, const moe_weights* w, int32_t* ids,
                                float* topk_w, int32_t* counts, int32_t* offsets, int32_t* perm, void* workspace,
                                size_t ws_bytes, void* stream) {
    Plan p;
    LayerArgs a;
    moe_status st = prepare(d, x, w, workspace, ws_bytes, &p, &a);
    if (st != MOE_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
    if (d->T == 0) {
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * d->E, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (d->E + 1), s);
        return cuda_status(e);
    }
    if (!ids || !topk_w || !perm) return MOE_ERR_INVALID_ARG;
    if (!aligned16(ids) || !aligned16(topk_w) || !aligned16(counts) || !aligned16(offsets) || !aligned16(perm))
        return MOE_ERR_MISALIGNED;
    a.ids = ids;
    a.topw = topk_w;
    a.counts = counts;
    a.offsets = offsets;
    a.perm = perm;
    return cuda_status(launch_routing(a, s));
}

extern "C" moe_status moe_router_stats(const moe_dims* d, const void* x, const moe_weights* w, float* P, float* f,
                                       float* loss, void* workspace, size_t ws_bytes, void* stream) {
    Plan p;
    LayerArgs a;
    moe_status st = prepare(d, x, w, workspace, ws_bytes, &p, &a);
    if (st != MOE_OK) return st;
    if (!P || !f || !loss) return MOE_ERR_INVALID_ARG;
    if (!aligned16(P) || !aligned16(f) || ((uintptr_t)loss & 3u)) return MOE_ERR_MISALIGNED;
    cudaStream_t s = (cudaStream_t)stream;
    if (d->T == 0) {
        cudaError_t e = cudaMemsetAsync(P, 0, sizeof(float) * d->E, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(f, 0, sizeof(float) * d->E, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(loss, 0, sizeof(float), s);
        return cuda_status(e);
    }
    // every score column must be in the workspace: below 256 tokens the tensor-pipe score
    // kernel and the one-CTA routing, from 256 the score GEMM and the top-K kernel
    cudaError_t e = route_small_supported(a) ? launch_route_small(a, s) : launch_router(a, s);
    if (e == cudaSuccess) e = launch_router_stats(a, P, f, loss, s);
    return cuda_status(e);
}

extern "C" moe_status moe_forward(const moe_dims* d, const void* x, const moe_weights* w, const void* residual,
                                  void* out, void* workspace, size_t ws_bytes, void* stream) {
    Plan p;
    LayerArgs a;
    moe_status st = prepare(d, x, w, workspace, ws_bytes, &p, &a);
    if (st != MOE_OK || d->T == 0) return st;
    st = check_output(d, x, residual, out);
    if (st != MOE_OK) return st;
    a.residual = (const bf16*)residual;
    a.out = (bf16*)out;
    return cuda_status(launch_layer(a, (cudaStream_t)stream));
}

extern "C" moe_status moe_forward_host_io(const moe_dims* d, const void* host_x, const moe_weights* w,
                                          const void* host_residual, void* host_out, void* dev_x, void* dev_out,
                                          void* workspace, size_t ws_bytes, void* stream) {
    Plan p;
    LayerArgs a;
    moe_status st = prepare(d, dev_x, w, workspace, ws_bytes, &p, &a);
    if (st != MOE_OK || d->T == 0) return st;
    st = check_output(d, dev_x, host_residual ? dev_out : nullptr, dev_out);
    if (st != MOE_OK) return st;
    if (!host_x || !host_out) return MOE_ERR_INVALID_ARG;
    if (!host_side(host_x) || !host_side(host_out) || (host_residual && !host_side(host_residual)) ||
        memory_type(dev_x) != cudaMemoryTypeDevice || memory_type(dev_out) != cudaMemoryTypeDevice)
        return MOE_ERR_INVALID_ARG;
    a.residual = host_residual ? (const bf16*)dev_out : nullptr;
    a.out = (bf16*)dev_out;
    const size_t act_bytes = (size_t)d->T * d->H * 2;
    cudaStream_t s = (cudaStream_t)stream;
    // Up to kKernelCopyBytes, rows in pinned mapped host memory move by k_copy_rows (a copy-engine
    // transfer would expose its own latency and the layer's launch behind it); pageable or
    // larger buffers by cudaMemcpyAsync.
    auto mapped = [&](const void* host, const void** dev) {
        return act_bytes <= kKernelCopyBytes && aligned16(host) && host_mapped(host, dev);
    };
    const void* m = nullptr;
    // One token on the one-token kernel: it reads the token row, the residual and writes the
    // output on the pinned mapped host rows themselves, so the rows cross the host link inside
    // the layer's own kernel (no copy launch before it and none after it). The row crosses the
    // link once (each CTA reads a share and passes it to the others through L2), each CTA reads
    // only the residual elements of the output rows it owns, before it writes them, and every
    // CTA has read the row before any CTA writes (the router scores, which need all of it, must
    // reach every CTA first), so the output may replace the host x or residual.
    {
        const void *mx = nullptr, *mr = nullptr, *mo = nullptr;
        if (a.T <= kFusedMaxTokens && a.dx && decode_fused_supported(a) && mapped(host_x, &mx) && mapped(host_out, &mo) &&
            (!host_residual || mapped(host_residual, &mr))) {
            a.x = (const bf16*)mx;
            a.x_host = true;
            a.residual = (const bf16*)mr;
            a.out = (bf16*)mo;
            return cuda_status(launch_decode_fused(a, s));
        }
    }
    cudaError_t e = mapped(host_x, &m) ? launch_copy_rows(m, dev_x, act_bytes, a.num_sms, s)
                                       : cudaMemcpyAsync(dev_x, host_x, act_bytes, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && host_residual)
        e = mapped(host_residual, &m) ? launch_copy_rows(m, dev_out, act_bytes, a.num_sms, s)
                                      : cudaMemcpyAsync(dev_out, host_residual, act_bytes, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = launch_layer(a, s);
    if (e == cudaSuccess)
        e = mapped(host_out, &m) ? launch_copy_rows(dev_out, const_cast<void*>(m), act_bytes, a.num_sms, s)
                                 : cudaMemcpyAsync(host_out, dev_out, act_bytes, cudaMemcpyDeviceToHost, s);
    return cuda_status(e);
}

extern "C" size_t moe_expert_shadow_size(const moe_dims* d) {
    Plan p;
    if (!d || !make_plan(*d, &p)) return 0;
    return ((size_t)d->E * 2 * d->I * d->H + (size_t)d->E * d->H * d->I) * 2;
}

extern "C" moe_status moe_forward_host_experts(const moe_dims* d, const void* x, const moe_weights* w,
                                               const void* residual, void* out, void* shadow, size_t shadow_bytes,
                                               void* workspace, size_t ws_bytes, void* stream) {
    Plan p;
    LayerArgs a;
    moe_status st = prepare(d, x, w, workspace, ws_bytes, &p, &a);
    if (st != MOE_OK || d->T == 0) return st;
    st = check_output(d, x, residual, out);
    if (st != MOE_OK) return st;
    if (!shadow) return MOE_ERR_INVALID_ARG;
    if (!aligned16(shadow)) return MOE_ERR_MISALIGNED;
    if (shadow_bytes < moe_expert_shadow_size(d)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    const void* hgu = nullptr;
    const void* hdn = nullptr;
    if (!host_mapped(w->gate_up, &hgu) || !host_mapped(w->down, &hdn)) return MOE_ERR_INVALID_ARG;
    // the fetch kernel reads any touched expert's rows: both whole tensors must be mapped
    if (!host_range_covers(w->gate_up, (size_t)d->E * 2 * d->I * d->H * 2) ||
        !host_range_covers(w->down, (size_t)d->E * d->H * d->I * 2))
        return MOE_ERR_INVALID_ARG;
    a.residual = (const bf16*)residual;
    a.out = (bf16*)out;
    bf16* sgu = (bf16*)shadow;
    bf16* sdn = sgu + (size_t)d->E * 2 * d->I * d->H;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_routing(a, s);
    if (e == cudaSuccess) e = launch_fetch_experts(a, (const bf16*)hgu, (const bf16*)hdn, sgu, sdn, s);
    a.gate_up = sgu;
    a.down = sdn;
    if (e == cudaSuccess) e = launch_after_routing(a, s);
    return cuda_status(e);
}

extern "C" moe_status moe_rmsnorm(const moe_dims* d, const void* x, const void* gamma, float eps, void* xn,
                                  void* stream) {
    if (!d) return MOE_ERR_INVALID_ARG;
    if (d->T < 0 || d->H < 128 || d->H > 8192 || d->H % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (d->T == 0) return MOE_OK;
    if (!x || !xn || !(eps >= 0.f)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xn) || (gamma && !aligned16(gamma))) return MOE_ERR_MISALIGNED;
    const size_t nbytes = (size_t)d->T * d->H * 2;
    if (overlap(x, nbytes, xn, nbytes)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_rmsnorm((const bf16*)x, (const bf16*)gamma, eps, (bf16*)xn, d->T, d->H,
                                      (cudaStream_t)stream));
}

extern "C" moe_status moe_last_device_error(void* workspace, void* stream) {
    if (!workspace) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t err = 0;
    WsHeader* hdr = (WsHeader*)workspace;
    cudaError_t e = cudaMemcpyAsync(&err, &hdr->err, sizeof err, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (err == 0) return MOE_OK;
    e = cudaMemsetAsync(&hdr->err, 0, sizeof err, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    return (err & ERR_TIMEOUT) ? MOE_ERR_TIMEOUT : MOE_ERR_DEVICE;
}

extern "C" moe_status moe_workspace_tap(const moe_dims* d, int tap, size_t* offset, size_t* bytes) {
    Plan p;
    if (!d || !offset || !bytes) return MOE_ERR_INVALID_ARG;
    if (!make_plan(*d, &p)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const size_t T = (size_t)d->T, P = (size_t)p.P;
    switch (tap) {
        case 0: *offset = p.o_h; *bytes = (P + T) * p.Imax * 2; return MOE_OK;
        case 1: *offset = p.o_y; *bytes = T * (d->K + 1) * d->H * (p.gemm ? 2 : 4); return MOE_OK;
        case 2: *offset = p.o_sgate; *bytes = T * 4; return MOE_OK;
        case 3: *offset = p.o_ids; *bytes = P * 4; return MOE_OK;
        case 4: *offset = p.o_topw; *bytes = P * 4; return MOE_OK;
        default: return MOE_ERR_INVALID_ARG;
    }
}

extern "C" moe_status moe_set_trace(int kernel, void* const* start_events, void* const* stop_events, int n_events) {
    if (kernel < 0 || kernel >= MOE_KERNEL_COUNT || n_events < 0 || n_events > (1 << 20)) return MOE_ERR_INVALID_ARG;
    if (n_events > 0 && (!start_events || !stop_events)) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < n_events; ++i)
        if (!start_events[i] || !stop_events[i]) return MOE_ERR_INVALID_ARG;
    TraceSlot& t = g_trace[kernel];
    t.n = 0;
    t.start.assign(start_events, start_events + n_events);
    t.stop.assign(stop_events, stop_events + n_events);
    t.n = n_events;
    t.i = 0;
    return MOE_OK;
}

extern "C" uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" moe_status moe_test_set_wait(uint64_t wait_ns, int suppress) {
    if (wait_ns > 10ull * kWaitNs ||
        (suppress != 0 && suppress != MOE_TEST_SUPPRESS_SCORE && suppress != MOE_TEST_SUPPRESS_STAGE))
        return MOE_ERR_INVALID_ARG;
    g_wait_ns.store(wait_ns ? wait_ns : kWaitNs, std::memory_order_relaxed);
    g_suppress.store(suppress, std::memory_order_relaxed);
    return MOE_OK;
}

extern "C" const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: a required pointer is NULL, buffers overlap, or an argument is out of range";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE: dims outside the supported range";
        case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED: a pointer is not 16-byte aligned";
        case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL: workspace smaller than moe_workspace_size()";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA launch or runtime call failed";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded device-side wait gave up";
        case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE: a kernel flagged a non-finite router score";
        default: return "unknown moe_status";
    }
}
