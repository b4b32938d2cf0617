// stream.cu -- the few-token (decode) regime of the experts: weight streaming.
//
// With few tokens every expert the router picked has only a handful of rows, so the layer is
// bound by reading the touched experts' weights from HBM once (4 MiB gate_up + 2 MiB down per
// expert at the full shape, "Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256 Experts).
// Both kernels are persistent (one CTA per SM) and stream weight rows through a 4-stage
// shared-memory ring filled by 1-D TMA bulk copies (cp.async.bulk) from a dedicated producer
// warp, with mbarrier full/empty handshakes, so each SM keeps up to 128 KB of loads in flight.
// Eight consumer warps take dot products of the staged rows with the group's token rows
// (warp w owns rows w, w+8, ...; lanes split the row into 16-byte chunks; fp32 FMA in a fixed
// order, then a butterfly sum).
//
// k_stream_up:   h = bf16(SiLU(x . Wg^T) * (x . Wu^T)), item = FPI gate rows + the FPI matching
//                up rows of one group; shared-expert items come first: they do not depend on
//                routing and run while the routing kernel finishes (programmatic dependent
//                launch; routed items wait with griddepcontrol.wait).
// k_stream_down: Y[t, slot] = scale * (h . Wd^T), item = 64 output rows of one group; items are
//                ordered by output block, and the CTA that completes the last item of a block
//                (ticket after a fence) sums that block for every token in the fixed order
//                residual, shared, slot 0..K-1 and writes out (no CTA waits on another).
#include "launch.h"
#include "sm100.cuh"

namespace moe {

constexpr int kStreamStages = 4;
constexpr int kStageBytes = 32768;
constexpr int kConsumers = 256;           // 8 consumer warps
constexpr int kStreamThreads = kConsumers + 32;
constexpr int kCombineRows = 64;          // output rows per down item / combine block

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

// Barrier of the consumer warps that also ANDs a predicate over them, so that all consumers
// take the same branch after a bounded wait (none is left behind in a named barrier).
__device__ __forceinline__ bool consumers_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok), "n"(kConsumers)
        : "memory");
    return r != 0;
}

// Rows of one stage for rows of length L: a power of two <= 64 with rows * L * 2 <= 32 KB.
__host__ __device__ __forceinline__ int stage_rows(int L) {
    int r = 64;
    while (r > 1 && r * L * 2 > kStageBytes) r >>= 1;
    return r;
}

// Tokens per shared-memory tile of activations of length L (<= 32 KB).
__host__ __device__ __forceinline__ int token_tile(int L) {
    int t = 8;
    while (t > 1 && t * L * 2 > 32768) t >>= 1;
    return t;
}

struct StreamSmem {
    uint8_t* ring;
    bf16* xs;        // [tile tokens, L] activations of the current token tile
    uint64_t* full;
    uint64_t* empty;
    int* flag;       // [0] = abort, [1] = combine ticket
};

__device__ __forceinline__ StreamSmem carve(uint8_t* raw, int T) {
    const uint32_t base = smem_u32(raw);
    uint8_t* p = raw + (((base + 127u) & ~127u) - base);
    StreamSmem s;
    s.ring = p;
    p += kStreamStages * kStageBytes;
    s.xs = reinterpret_cast<bf16*>(p);
    p += 32768;
    s.full = reinterpret_cast<uint64_t*>(p);
    s.empty = s.full + kStreamStages;
    s.flag = reinterpret_cast<int*>(s.empty + kStreamStages);
    return s;
}

constexpr int kStreamSmemBytes = 128 + kStreamStages * kStageBytes + 32768 + 2 * kStreamStages * 8 + 16;

__device__ __forceinline__ void stream_init(StreamSmem& s) {
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStreamStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], kConsumers / 32);
        }
        s.flag[0] = 0;
        fence_mbar_init();
    }
    __syncthreads();
}

// Producer side of one stage: wait until consumers freed it, then start the copy.
__device__ __forceinline__ bool produce(StreamSmem& s, int& it, const void* src, uint32_t bytes, uint32_t* err) {
    const int st = it % kStreamStages;
    const uint32_t ph = (uint32_t)(it / kStreamStages) & 1u;
    if (!mbar_wait(&s.empty[st], ph ^ 1u)) {
        atomicOr(err, ERR_TIMEOUT);
        *(volatile int*)&s.flag[0] = 1;
        return false;
    }
    mbar_arrive_expect_tx(&s.full[st], bytes);
    bulk_load(s.ring + (size_t)st * kStageBytes, src, bytes, &s.full[st]);
    ++it;
    return true;
}

// Consumer side: wait for stage `it`; returns its buffer or nullptr on timeout.
__device__ __forceinline__ const bf16* consume(StreamSmem& s, int it, uint32_t* err) {
    const int st = it % kStreamStages;
    const uint32_t ph = (uint32_t)(it / kStreamStages) & 1u;
    if (!mbar_wait(&s.full[st], ph)) {
        atomicOr(err, ERR_TIMEOUT);
        *(volatile int*)&s.flag[0] = 1;
        return nullptr;
    }
    return reinterpret_cast<const bf16*>(s.ring + (size_t)st * kStageBytes);
}

__device__ __forceinline__ void release(StreamSmem& s, int it) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&s.empty[it % kStreamStages]);
}

// Copy `mt` activation rows of length L into xs (row tt from src_row(tt)).
template <typename RowFn>
__device__ __forceinline__ void stage_rows_to_smem(bf16* xs, int L, int mt, RowFn src_row) {
    const int chunks = L / 8;
    for (int i = threadIdx.x; i < mt * chunks; i += kConsumers) {
        const int tt = i / chunks, c = i - tt * chunks;
        reinterpret_cast<uint4*>(xs + (size_t)tt * L)[c] = ld_ro(src_row(tt) + (size_t)c * 8);
    }
}

// Dot products of one staged row (length L) with mt staged activation rows; every lane gets
// the sums. Chunk order per lane and the butterfly are fixed, so results are reproducible.
template <int TT>
__device__ __forceinline__ void row_dots(const bf16* wrow, const bf16* xs, int L, int mt, int lane, float* out) {
    float acc[TT];
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) acc[tt] = 0.f;
    for (int c = lane; c < L / 8; c += 32) {
        const uint4 w = *reinterpret_cast<const uint4*>(wrow + (size_t)c * 8);
#pragma unroll
        for (int tt = 0; tt < TT; ++tt) {
            if (tt < mt) {
                float xf[8];
                unpack8(*reinterpret_cast<const uint4*>(xs + (size_t)tt * L + (size_t)c * 8), xf);
                acc[tt] = dot8(w, xf, acc[tt]);
            }
        }
    }
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) out[tt] = tt < mt ? warp_sum(acc[tt]) : 0.f;
}

// ---------------------------------------------------------------------------------------

struct UpItem {
    const bf16* W;
    int inner, row0, rows, f0;
    bool shared;
};

__device__ __forceinline__ UpItem up_item(const LayerArgs& a, int it, int n_shared_items, int fpi) {
    UpItem u;
    if (it < n_shared_items) {
        u = UpItem{a.sgu, a.Is, (int)a.P, a.T, it * fpi, true};
    } else {
        const int ipr = a.I / fpi;
        const int k = it - n_shared_items;
        const int g = k / ipr;
        const int e = a.act[g];
        u.W = a.gate_up + (size_t)e * 2 * a.I * a.H;
        u.inner = a.I;
        u.row0 = a.offsets[e];
        u.rows = a.offsets[e + 1] - u.row0;
        u.f0 = (k - g * ipr) * fpi;
        u.shared = false;
    }
    return u;
}

__global__ void __launch_bounds__(kStreamThreads, 1) k_stream_up(LayerArgs a) {
    extern __shared__ uint8_t smem_raw[];
    StreamSmem s = carve(smem_raw, a.T);
    stream_init(s);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int fpi = stage_rows(a.H);
    const int n_shared = a.Is / fpi;
    uint32_t* err = &a.hdr->err;
    // routed items need the routing: everything below `n_shared` can start at once
    int n_items = -1;

    if (warp == kConsumers / 32) {
        if (lane == 0) {
            int it = 0;
            bool waited = false;
            for (int i = blockIdx.x;; i += gridDim.x) {
                if (i >= n_shared && !waited) {
                    grid_dep_wait();
                    waited = true;
                    n_items = n_shared + a.hdr->n_act * (a.I / fpi);
                }
                if (n_items >= 0 && i >= n_items) break;
                if (*(volatile int*)&s.flag[0]) break;
                const UpItem u = up_item(a, i, n_shared, fpi);
                const uint32_t bytes = (uint32_t)(fpi * a.H * 2);
                if (!produce(s, it, u.W + (size_t)u.f0 * a.H, bytes, err)) break;
                if (!produce(s, it, u.W + (size_t)(u.inner + u.f0) * a.H, bytes, err)) break;
            }
            // every copy issued must land before the CTA's shared memory is released
            for (int k = 0; k < kStreamStages && it - 1 - k >= 0; ++k) {
                const int j = it - 1 - k;
                if (!mbar_wait(&s.full[j % kStreamStages], (uint32_t)(j / kStreamStages) & 1u)) atomicOr(err, ERR_TIMEOUT);
            }
        }
        return;
    }

    // consumers
    const int TT = token_tile(a.H);
    int it = 0;
    bool waited = false;
    for (int i = blockIdx.x;; i += gridDim.x) {
        if (i >= n_shared && !waited) {
            grid_dep_wait();
            waited = true;
            n_items = n_shared + a.hdr->n_act * (a.I / fpi);
        }
        if (n_items >= 0 && i >= n_items) break;
        const UpItem u = up_item(a, i, n_shared, fpi);
        const bf16* wgs = consume(s, it, err);
        const bf16* wus = wgs ? consume(s, it + 1, err) : nullptr;
        if (!consumers_all(wus != nullptr)) break;
        for (int r0 = 0; r0 < u.rows; r0 += TT) {
            const int mt = min(TT, u.rows - r0);
            stage_rows_to_smem(s.xs, a.H, mt, [&](int tt) {
                const int j = u.row0 + r0 + tt;
                const int t = u.shared ? j - (int)a.P : a.perm[j] / a.K;
                return a.x + (size_t)t * a.H;
            });
            consumers_sync();
            for (int f = warp; f < fpi; f += kConsumers / 32) {
                float g[8], uu[8];
                row_dots<8>(wgs + (size_t)f * a.H, s.xs, a.H, mt, lane, g);
                row_dots<8>(wus + (size_t)f * a.H, s.xs, a.H, mt, lane, uu);
#pragma unroll
                for (int tt = 0; tt < 8; ++tt)
                    if (lane == tt && tt < mt)
                        a.h[(size_t)(u.row0 + r0 + tt) * a.Imax + u.f0 + f] = __float2bfloat16_rn(silu(g[tt]) * uu[tt]);
            }
            consumers_sync();
        }
        release(s, it);
        release(s, it + 1);
        it += 2;
    }
    grid_dep_launch();
}

// ---------------------------------------------------------------------------------------

struct DownItem {
    const bf16* W;
    int inner, row0, rows, o0;
    bool shared;
};

__device__ __forceinline__ DownItem down_item(const LayerArgs& a, int it, int n_groups) {
    const int ob = it / n_groups, g = it - ob * n_groups;
    DownItem d;
    d.o0 = ob * kCombineRows;
    if (g == n_groups - 1) {
        d.W = a.sd;
        d.inner = a.Is;
        d.row0 = (int)a.P;
        d.rows = a.T;
        d.shared = true;
    } else {
        const int e = a.act[g];
        d.W = a.down + (size_t)e * a.H * a.I;
        d.inner = a.I;
        d.row0 = a.offsets[e];
        d.rows = a.offsets[e + 1] - d.row0;
        d.shared = false;
    }
    return d;
}

__global__ void __launch_bounds__(kStreamThreads, 1) k_stream_down(LayerArgs a) {
    extern __shared__ uint8_t smem_raw[];
    StreamSmem s = carve(smem_raw, a.T);
    stream_init(s);
    grid_dep_wait();  // h comes from k_stream_up; the routing from before it
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_groups = a.hdr->n_act + 1;
    const int n_items = n_groups * (a.H / kCombineRows);
    uint32_t* err = &a.hdr->err;

    if (warp == kConsumers / 32) {
        if (lane == 0) {
            int it = 0;
            for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
                if (*(volatile int*)&s.flag[0]) break;
                const DownItem d = down_item(a, i, n_groups);
                const int rps = stage_rows(d.inner);
                bool ok = true;
                for (int r = 0; r < kCombineRows && ok; r += rps)
                    ok = produce(s, it, d.W + (size_t)(d.o0 + r) * d.inner, (uint32_t)(rps * d.inner * 2), err);
                if (!ok) break;
            }
            for (int k = 0; k < kStreamStages && it - 1 - k >= 0; ++k) {
                const int j = it - 1 - k;
                if (!mbar_wait(&s.full[j % kStreamStages], (uint32_t)(j / kStreamStages) & 1u)) atomicOr(err, ERR_TIMEOUT);
            }
        }
        return;
    }

    int it = 0;
    for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
        const DownItem d = down_item(a, i, n_groups);
        const int rps = stage_rows(d.inner);
        const int TT = token_tile(d.inner);
        bool ok = true;
        for (int r = 0; r < kCombineRows && ok; r += rps, ++it) {
            const bf16* ws = consume(s, it, err);
            if (!consumers_all(ws != nullptr)) {
                ok = false;
                break;
            }
            for (int r0 = 0; r0 < d.rows; r0 += TT) {
                const int mt = min(TT, d.rows - r0);
                stage_rows_to_smem(s.xs, d.inner, mt, [&](int tt) { return a.h + (size_t)(d.row0 + r0 + tt) * a.Imax; });
                consumers_sync();
                int tok[8], slot[8];
                float sc[8];
#pragma unroll
                for (int tt = 0; tt < 8; ++tt) {
                    tok[tt] = 0;
                    slot[tt] = 0;
                    sc[tt] = 0.f;
                    if (tt < mt) {
                        const int j = d.row0 + r0 + tt;
                        if (d.shared) {
                            tok[tt] = j - (int)a.P;
                            slot[tt] = a.K;
                            sc[tt] = a.sgate[tok[tt]];
                        } else {
                            const int pv = a.perm[j];
                            tok[tt] = pv / a.K;
                            slot[tt] = pv - tok[tt] * a.K;
                            sc[tt] = a.topw[pv];
                        }
                    }
                }
                for (int rr = warp; rr < rps; rr += kConsumers / 32) {
                    float y[8];
                    row_dots<8>(ws + (size_t)rr * d.inner, s.xs, d.inner, mt, lane, y);
                    const int o = d.o0 + r + rr;
#pragma unroll
                    for (int tt = 0; tt < 8; ++tt)
                        if (lane == tt && tt < mt) a.Y[((size_t)tok[tt] * (a.K + 1) + slot[tt]) * a.H + o] = sc[tt] * y[tt];
                }
                consumers_sync();
            }
            release(s, it);
        }
        if (!ok) break;
        // fixed-order combine of this output block once every group has written it
        __threadfence();
        consumers_sync();
        if (threadIdx.x == 0) s.flag[1] = (int)atomicAdd(&a.comb_ticket[d.o0 / kCombineRows], 1u);
        consumers_sync();
        if (s.flag[1] == n_groups - 1) {
            __threadfence();
            for (int idx = threadIdx.x; idx < a.T * kCombineRows; idx += kConsumers) {
                const int t = idx / kCombineRows, o = d.o0 + (idx - t * kCombineRows);
                const float* yt = a.Y + (size_t)t * (a.K + 1) * a.H + o;
                float acc = a.residual ? __bfloat162float(a.residual[(size_t)t * a.H + o]) : 0.f;
                acc += __ldcg(yt + (size_t)a.K * a.H);
                for (int k = 0; k < a.K; ++k) acc += __ldcg(yt + (size_t)k * a.H);
                a.out[(size_t)t * a.H + o] = __float2bfloat16_rn(acc);
            }
            if (threadIdx.x == 0) a.comb_ticket[d.o0 / kCombineRows] = 0;  // re-arm
        }
    }
}

// ---------------------------------------------------------------------------------------

namespace {

template <typename K>
cudaError_t launch_pdl(K kernel, int grid, int smem, cudaStream_t s, const LayerArgs& a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kStreamThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace

bool stream_supported(const LayerArgs& a) {
    // the shared-memory ring holds at least one row, the activation tile at least one token,
    // and the gate results of an up item fit the [64, 256] buffer
    return a.H * 2 <= kStageBytes && a.Imax * 2 <= kStageBytes && a.T <= 256 && stage_rows(a.H) <= 64;
}

cudaError_t launch_stream_experts(const LayerArgs& a, cudaStream_t s) {
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_stream_up, cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_stream_down, cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamSmemBytes);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    cudaError_t e;
    MOE_LAUNCH(MOE_KERNEL_GATE_UP, s, (e = launch_pdl(k_stream_up, a.num_sms, kStreamSmemBytes, s, a)));
    if (e != cudaSuccess) return e;
    MOE_LAUNCH(MOE_KERNEL_DOWN, s, (e = launch_pdl(k_stream_down, a.num_sms, kStreamSmemBytes, s, a)));
    return e;
}

}  // namespace moe
