// decode.cu -- the whole MoE layer for one token (decode) in one persistent kernel.
//
// At decode a layer streams ~55 MB of weights per token ("Qwen3.6-35B-A3B -- Architecture
// Overview", MoE FFN: 256 Experts: router 2048 -> 256 plus the shared-expert gate, 8 routed
// SwiGLU experts with merged gate_up [1024 x 2048] and down [2048 x 512], one always-on
// shared expert of the same shape; "One Token Through Qwen3.6", The Router), and only the
// router and the shared expert (7 MB) are known before the routing. So the kernel's job is
// to start the routed stream as early as possible and then keep HBM busy until the end.
// It is built for that layer shape (H = 2048, expert widths 512); other shapes and more
// tokens take the routing and streaming kernels.
//
// One CTA per SM (G CTAs). CTA c owns:
//   - router rows c, c+G, ... (row E is the shared-expert gate);
//   - shared-expert features [c*Is/G, (c+1)*Is/G) and routed (slot, feature) pairs
//     P = c, c+G, ... of the F = K*I (P = slot * I + feature): the gate row and the up row of
//     each, giving h. Strided rather than a contiguous run: every CTA then works through the
//     slots in the same order, all of them on the same expert's rows at a time (measured
//     16.64 us per layer against 17.03 us for contiguous runs, alternating on one box);
//   - output rows [c*H/G, (c+1)*H/G) of the shared and of every routed expert's down
//     projection, and their fixed-order combine (residual + gated shared + slots 0..K-1).
// Its work is a fixed sequence of items, one per 8 KB ring slot: router rows, shared
// features, routed features, then down rows (shared first, then slots 0..K-1, 8 rows per
// item). Three producer warps (lane 0 of warp q issues items q, q+3, ...) copy items into the
// ring with 1-D TMA bulk copies: the router rows and shared features first, before the kernel
// waits for the previous one on the stream (programmatic launch), then the token row, and the
// rest as soon as the routing is known and a slot is free. (Issuing the shared expert's down
// rows before the routing too was measured slower: they compete with the token row and the
// router rows on the critical path.) Consumer warp w takes items w, w+9, ... in order, so the
// warps never wait for one another; a warp's dot products read the weights from shared memory
// with x held in registers, bf16 by bf16 (one token: an MMA would use one column of eight).
//
// Exchanges between CTAs carry a tag of the call instead of a flag: router scores are 64-bit
// words (tag, fp32 score), h values 32-bit words (16-bit tag, bf16 h), and, when the token row
// is in host memory, the row's 32-bit words as 64-bit words (tag, word), each CTA reading its
// share of the row over the host link (moe_forward_host_io); all are published with atomic
// exchanges (carried out at L2, where the other SMs' polls see them within about a
// microsecond; a plain store would need a fence, which stalls the SM's other warps). A
// reader polls the words it needs until all carry this call's tag; a word not yet rewritten
// by this call carries an earlier call's tag. Warp 0 of every CTA
// ranks the E scores itself (top-K with ties to the lower index, renormalised weights, the
// shared gate) right after its own router row and releases the producers as soon as the
// experts are known. Down items come last and wait only for the h words of their own expert
// slot.
//
// Every wait is bounded (~1 s): a timeout sets MOE_ERR_TIMEOUT in the workspace and the
// kernel still runs to its end with in-range indices. Each CTA counts itself in when it
// starts; CTA 0 moves the call's tag on at its end once all are in.
#include <atomic>
#include "launch.h"
#include "ring.cuh"

namespace moe {

// In-kernel timeline (a build with MOE_TIMELINE only): the global timer at fixed points of each
// CTA's call, read back with moe_timeline_read. Event e of CTA c is g_moe_tl[c * kTlEvents + e]:
//   0 CTA start                          5 warp 0: every CTA's router scores seen
//   1 producer 0: weight-only items out  6 warp 0: routing known, producer released
//   2 producer 0: previous kernel done   7 producer 0: every item issued
//   3 consumers: token row in registers  8 consumers: every item done (combine starts)
//   4 a router score published          9 combine done
constexpr int kTlEvents = 10, kTlCtas = 256;
#ifdef MOE_TIMELINE
__device__ unsigned long long g_moe_tl[kTlCtas * kTlEvents];
#define MOE_TL(ev)                                                                     \
    do {                                                                               \
        if (blockIdx.x < kTlCtas) g_moe_tl[blockIdx.x * kTlEvents + (ev)] = global_ns(); \
    } while (0)
#else
#define MOE_TL(ev) \
    do {           \
    } while (0)
#endif

constexpr int kOWarps = 9;                     // consumer warps
constexpr int kOProducers = 3;                 // producer warps (lane 0 of each issues copies)
constexpr int kOThreads = (kOWarps + kOProducers) * 32;
constexpr int kOH = 2048;                      // hidden width (the page's layer shape)
constexpr int kOI = 512;                       // routed and shared expert widths
constexpr int kONch = kOH / 256;               // 16-byte chunks of an H-long row per lane
constexpr int kOIch = kOI / 256;               // 16-byte chunks of an I-long row per lane
constexpr int kOMaxK = 8;                      // experts per token
constexpr int kOSlot = 8192;                   // ring slot: one feature's gate and up rows
constexpr int kOMaxSlots = 27;                 // ring slots at most (the count used: a multiple of kOWarps)
static_assert(kOMaxSlots <= 32, "one producer lane per slot in the exit drain");
static_assert(kOWarps % kOProducers == 0, "slot counts that are multiples of the consumer warps suit the producers");
constexpr int kOMaxItems = 64;
constexpr int kOMaxRo = kOSlot / (kOI * 2);    // down rows per item
constexpr int kOMaxOut = 16;                   // output rows per CTA

enum : int { kOkRouter = 0, kOkSharedUp = 1, kOkSharedDown = 2, kOkUp = 3, kOkDown = 4 };

// What one ring slot holds (written by the producer before the slot's copies).
struct OMeta {
    int kind;
    int k;  // expert slot 0..K-1, or K for the shared expert
    int a;  // router row / feature / first output row
    int n;  // rows (down items)
};

// The routing of the token as every CTA derives it, and the routed experts' weight blocks.
struct ORoute {
    const bf16* gu[kOMaxK];
    const bf16* dn[kOMaxK];
    int ids[kOMaxK];
    float w[kOMaxK];
    int inv[kOMaxK];
    float sg;
};

// Per-CTA share of the work; identical in every thread (32-bit arithmetic only).
struct OPlan {
    int nr;        // router rows: c, c + G, ...
    int fs0, nsf;  // shared features
    int o0, ro;    // output rows
    int dpk;       // down items per expert (kOMaxRo rows each)
    int nf;        // routed (slot, feature) pairs: P = c, c + G, ... of the K*I
    int n;         // items
};

struct OGeom {
    int nslot;
    int o_slot, o_meta, o_bar, o_ys, o_rt, o_iss, o_x, smem;
};

// Item j of a CTA's sequence: router rows, shared features, routed features, then down rows
// (the shared expert's first, then slots 0..K-1, kOMaxRo rows per item); the copies that load
// it and what its consumer does with it.
struct OItem {
    OMeta m;
    const void* src0;
    const void* src1;
    uint32_t b0, b1;
};

__device__ __forceinline__ OPlan oplan(const LayerArgs& a, int c, int G) {
    OPlan p;
    p.nr = c < a.E + 1 ? (a.E + 1 - c + G - 1) / G : 0;
    p.fs0 = c * kOI / G;
    p.nsf = (c + 1) * kOI / G - p.fs0;
    p.o0 = c * kOH / G;
    p.ro = (c + 1) * kOH / G - p.o0;
    const int F = a.K * kOI;
    p.nf = c < F ? (F - c + G - 1) / G : 0;
    p.dpk = (p.ro + kOMaxRo - 1) / kOMaxRo;
    p.n = p.nr + p.nsf + p.nf + (a.K + 1) * p.dpk;
    return p;
}

__device__ __forceinline__ OItem item_at(const LayerArgs& a, const OPlan& p, const ORoute& rt, int c, int G, int j) {
    OItem it;
    it.src1 = nullptr;
    it.b1 = 0;
    if (j < p.nr) {
        const int row = c + j * G;
        it.m = OMeta{kOkRouter, a.K, row, 1};
        it.src0 = row < a.E ? a.router_w + (size_t)row * kOH : a.sg;
        it.b0 = kOH * 2;
        return it;
    }
    j -= p.nr;
    if (j < p.nsf) {
        const int f = p.fs0 + j;
        it.m = OMeta{kOkSharedUp, a.K, f, 1};
        it.src0 = a.sgu + (size_t)f * kOH;
        it.src1 = a.sgu + (size_t)(kOI + f) * kOH;
        it.b0 = it.b1 = kOH * 2;
        return it;
    }
    j -= p.nsf;
    if (j < p.nf) {
        const int fi = c + j * G, k = fi / kOI, f = fi - k * kOI;  // (slot, feature) pair
        it.m = OMeta{kOkUp, k, f, 1};
        it.src0 = rt.gu[k] + (size_t)f * kOH;
        it.src1 = rt.gu[k] + (size_t)(kOI + f) * kOH;
        it.b0 = it.b1 = kOH * 2;
        return it;
    }
    j -= p.nf;
    const int kk = j / p.dpk, r0 = p.o0 + (j - kk * p.dpk) * kOMaxRo, n = min(kOMaxRo, p.o0 + p.ro - r0);
    it.m = OMeta{kk == 0 ? kOkSharedDown : kOkDown, kk == 0 ? a.K : kk - 1, r0, n};
    it.src0 = (kk == 0 ? a.sd : rt.dn[kk - 1]) + (size_t)r0 * kOI;
    it.b0 = (uint32_t)(n * kOI * 2);
    return it;
}

// Publishing a tagged word to the other CTAs: an atomic exchange is carried out at L2, where
// the other SMs' polls find it within about a microsecond; a plain relaxed store can stay
// buffered for several microseconds unless a fence follows it, and a fence holds up the
// memory instructions of the SM's other warps too. (The old value is not used.)
__device__ __forceinline__ void publish_u64(uint64_t* p, uint64_t v) {
    uint64_t old;
    asm volatile("atom.exch.relaxed.gpu.global.b64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void publish_u32(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.exch.relaxed.gpu.global.b32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint4 ld_relaxed_v4(const uint32_t* p) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
// 16 bytes from shared memory at a shared-window address (an explicit shared load; a generic
// load through a pointer into dynamic shared memory is several times slower here).
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// Lane 0 waits for a barrier phase (bounded); the warp shares the verdict.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int lane, uint64_t limit) {
    bool ok = lane == 0 ? mbar_wait(bar, parity, limit) : true;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok;
}

// Poll until *p - base >= n (unsigned, acquire); false after `limit` ns.
__device__ __forceinline__ bool wait_count(const uint32_t* p, uint32_t base, uint32_t n, uint64_t limit) {
    const uint64_t t0 = global_ns();
    for (;;) {
        if (ld_acquire(p) - base >= n) return true;
        if (global_ns() - t0 > limit) return false;
        __nanosleep(64);
    }
}

// Dot products of x (this lane's chunks in registers) with R H-long bf16 rows in shared
// memory; lane l takes the 16-byte chunks l, l+32, ... into two partial sums per row (short
// dependency chains), added in a fixed order, then the warp sums in a fixed order.
template <int R>
__device__ __forceinline__ void dot_rows(const uint32_t (&rows)[R], const uint4 (&xr)[kONch], int lane,
                                         float (&out)[R]) {
    float acc[R][2];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r][0] = acc[r][1] = 0.f;
    // loads run two chunks ahead of the multiplies (shared-memory loads wait behind the ring's
    // incoming copies)
    uint4 w[3][R];
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int r = 0; r < R; ++r) w[q][r] = lds128(rows[r] + 16u * (lane + 32 * q));
#pragma unroll
    for (int q = 0; q < kONch; ++q) {
        if (q + 2 < kONch)
#pragma unroll
            for (int r = 0; r < R; ++r) w[(q + 2) % 3][r] = lds128(rows[r] + 16u * (lane + 32 * (q + 2)));
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r][q & 1] = dot8_bf16(w[q % 3][r], xr[q], acc[r][q & 1]);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) out[r] = warp_sum(acc[r][0] + acc[r][1]);
}

// The tagged h words of expert slot k that this lane multiplies (chunks lane, lane+32, ... of
// the inner width: 8 words each, the bf16 h in each low half), polled until all carry `tag16`.
// False after `limit` ns (the words are then taken as they are).
__device__ bool poll_h(const uint32_t* words, uint32_t tag16, uint32_t (&hv)[kOIch][8], int lane, uint64_t limit) {
    uint32_t need = (1u << kOIch) - 1u;
    const uint64_t t0 = global_ns();
    bool ok = true;
    for (;;) {
        const bool give_up = !ok;
#pragma unroll
        for (int q = 0; q < kOIch; ++q)
            if ((need >> q) & 1u) {
                const uint32_t* p = words + 8 * (lane + 32 * q);
                const uint4 v0 = ld_relaxed_v4(p), v1 = ld_relaxed_v4(p + 4);
                const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                bool fresh = true;
#pragma unroll
                for (int i = 0; i < 8; ++i) fresh &= (w[i] >> 16) == tag16;
                if (fresh || give_up) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) hv[q][i] = w[i];
                    need &= ~(1u << q);
                }
            }
        if (!__any_sync(0xffffffffu, need != 0)) return ok;
        if (global_ns() - t0 > limit) ok = false;
    }
}

// Top-K of the token by warp 0 from the E + 1 tagged scores (expert scores, then the shared
// gate): lane l polls experts l, l+32, ... (lane 0 also the gate) until all carry this call's
// tag; each of K rounds takes the largest remaining key and, among equal keys, the lowest
// expert ("Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256 Experts, Router). The
// weights are the softmax over the kept scores (the full softmax renormalised over them).
// Arrives on `routed` once the experts, their weight blocks and dispatch positions are in rt.
__device__ void route_one(const LayerArgs& a, ORoute& rt, uint32_t tag, int lane, uint64_t* routed) {
    const uint64_t* l = a.dlog;
    uint32_t val[9];
    uint32_t need = 0;
#pragma unroll
    for (int j = 0; j < 9; ++j) {
        val[j] = 0u;  // a score of 0 if the wait times out
        const int e = j < 8 ? lane + 32 * j : a.E;
        if ((j < 8 && e < a.E) || (j == 8 && lane == 0)) need |= 1u << j;
    }
    const uint64_t t0 = global_ns();
    bool timed_out = false;
    for (;;) {
        uint64_t w[9];
#pragma unroll
        for (int j = 0; j < 9; ++j) w[j] = ((need >> j) & 1u) ? ld_relaxed_u64(l + (j < 8 ? lane + 32 * j : a.E)) : 0ull;
        uint32_t still = need;
#pragma unroll
        for (int j = 0; j < 9; ++j)
            if (((need >> j) & 1u) && (uint32_t)(w[j] >> 32) == tag) {
                val[j] = (uint32_t)w[j];
                still &= ~(1u << j);
            }
        need = still;
        if (!__any_sync(0xffffffffu, need != 0)) {
            if (lane == 0) MOE_TL(5);
            break;
        }
        if (global_ns() - t0 > a.wait_ns) {
            timed_out = true;
            break;
        }
    }
    bool bad = false;
    uint32_t key[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        key[j] = 0u;  // below every score: never taken while a real expert remains
        if (lane + 32 * j < a.E) {
            float v = router_score(__uint_as_float(val[j]), a.flags);
            if (!isfinite(v)) {
                bad = true;
                v = -INFINITY;
            }
            key[j] = score_key(v);
        }
    }
    float v0, myv;
    int mye;
    warp_topk(key, a.K, lane, v0, myv, mye);
    // dispatch position of slot `lane`: the slots whose expert is lower (the K experts differ)
    int pos = 0;
    for (int j = 0; j < a.K; ++j) pos += __shfl_sync(0xffffffffu, mye, j) < mye;
    if (lane < a.K) {
        rt.ids[lane] = mye;
        rt.inv[lane] = pos;
        rt.gu[lane] = a.gate_up + (size_t)mye * 2 * kOI * kOH;
        rt.dn[lane] = a.down + (size_t)mye * kOH * kOI;
    }
    // the producer may issue the routed items now; the weights and the shared gate are read
    // only after the consumers' barrier before the combine (and by this warp)
    __syncwarp();
    if (lane == 0) {
        MOE_TL(6);
        mbar_arrive(routed);
    }
    const float ex = lane < a.K ? expf(myv - v0) : 0.f;
    const float s = warp_sum(ex);
    if (lane < a.K) rt.w[lane] = ex / s;
    if (lane == 0) {
        const float z = router_score(__uint_as_float(val[8]), a.flags);
        if (!isfinite(z)) bad = true;
        rt.sg = 1.0f / (1.0f + expf(-z));
        if (timed_out) atomicOr(&a.hdr->err, ERR_TIMEOUT);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&a.hdr->err, ERR_NONFINITE_SCORE);
    __syncwarp();
}

// The routing results of the call in the workspace (ids, weights, counts, offsets, dispatch
// permutation, used experts, shared gate), written by warp 0 of CTA 0.
__device__ void write_routing(const LayerArgs& a, const ORoute& rt, int lane) {
    const int K = a.K;
    if (lane < K) {
        a.ids[lane] = rt.ids[lane];
        a.topw[lane] = rt.w[lane];
        a.perm[rt.inv[lane]] = lane;
        a.inv[lane] = rt.inv[lane];
        a.act[rt.inv[lane]] = rt.ids[lane];
    }
    for (int e = lane; e <= a.E; e += 32) {
        int less = 0, cnt = 0;
        for (int j = 0; j < K; ++j) {
            less += rt.ids[j] < e;
            cnt += rt.ids[j] == e;
        }
        a.offsets[e] = less;
        if (e < a.E) a.counts[e] = cnt;
    }
    if (lane == 0) {
        a.sgate[0] = rt.sg;
        a.hdr->n_act = K;
    }
}

__global__ void __launch_bounds__(kOThreads, 1) k_decode_fused(LayerArgs a, OGeom g) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* slots = base + g.o_slot;
    OMeta* meta = reinterpret_cast<OMeta*>(base + g.o_meta);
    uint64_t* full = reinterpret_cast<uint64_t*>(base + g.o_bar);
    uint64_t* empty = full + kOMaxSlots;
    uint64_t* routed = empty + kOMaxSlots;
    float* ys = reinterpret_cast<float*>(base + g.o_ys);  // [K + 1][kOMaxOut] down outputs, unscaled
    ORoute& rt = *reinterpret_cast<ORoute*>(base + g.o_rt);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int K = a.K, nslot = g.nslot;
    if (threadIdx.x == 0) MOE_TL(0);
    uint32_t* err = &a.hdr->err;
    // the kernel parameters the first steps read, fetched together: each first read of a
    // parameter line misses the constant cache, and in the order of use the misses would come
    // one after another
    asm volatile("" ::"l"(a.router_w), "l"(a.sg), "l"(a.sgu), "l"(a.x), "l"(a.hdr), "l"(a.gate_up), "l"(a.down),
                 "l"(a.dlog), "l"(a.dh), "r"(a.E), "r"(a.K), "r"(a.flags), "r"(g.nslot), "l"(a.wait_ns));
    const OPlan p = oplan(a, c, G);
    grid_dep_launch();  // the next kernel may be scheduled as this one's CTAs finish

    // ---- producers: warp kOWarps + q issues items q, q + kOProducers, ... (a slot is always
    // refilled by the same producer warp: kOProducers divides the slot count)
    const int pw = warp - kOWarps;
    uint8_t* issued = base + g.o_iss;  // items whose copies went out
    bool pok = true;
    int pj = pw, ps = pw;  // this producer's next item and its slot
    uint32_t pround = 0;
    // lane 0 of a producer warp: the next item of its share, once its slot is free (and, for
    // the routed items, once the routing is known)
    auto issue_next = [&](bool routed_known) -> bool {
        if (!routed_known && pj >= p.nr + p.nsf) return false;
        if (pround > 0 && !mbar_wait(&empty[ps], (pround - 1u) & 1u, a.wait_ns)) {
            pok = false;
            return false;
        }
        const OItem it = item_at(a, p, rt, c, G, pj);
        meta[ps] = it.m;
        uint8_t* dst = slots + (size_t)ps * kOSlot;
        mbar_arrive_expect_tx(&full[ps], it.b0 + it.b1);
        bulk_load(dst, it.src0, it.b0, &full[ps]);
        if (it.b1) bulk_load(dst + it.b0, it.src1, it.b1, &full[ps]);
        issued[pj] = 1;
        pj += kOProducers;
        ps += kOProducers;
        if (ps >= nslot) {
            ps -= nslot;
            ++pround;
        }
        return true;
    };
    if (pw >= 0) {
        for (int i = pw * 32 + lane; i < 2 * nslot + 1; i += kOProducers * 32)
            mbar_init(i < nslot ? &full[i] : i < 2 * nslot ? &empty[i - nslot] : routed, 1);
        for (int j = pw * 32 + lane; j < kOMaxItems; j += kOProducers * 32) issued[j] = 0;
        fence_mbar_init();
        __syncwarp();
        asm volatile("bar.sync 2, %0;" ::"n"(kOProducers * 32) : "memory");
        if (lane == 0) {
            // the router rows, then the shared expert's features: weights only, so they go out
            // before the wait for the previous kernel below
            while (pok && issue_next(false)) {
            }
            if (pw == 0) MOE_TL(1);
        }
    }
    // Launched with programmatic serialization, the kernel may start while the previous one on
    // the stream (the layer before, say, whose output is this token row) is still running:
    // everything from here on waits for it to complete and for its memory to be visible.
    grid_dep_wait();
    if (pw == 0 && lane == 0) MOE_TL(2);
    // the residual of this CTA's output rows, read now: at the combine its latency would come
    // last on the critical path (thread o < ro adds row o0 + o)
    const float resid = (threadIdx.x < p.ro && a.residual) ? __bfloat162float(a.residual[p.o0 + threadIdx.x]) : 0.f;
    // this call's tags and the CTA starts of earlier calls (both advanced by CTA 0 of the
    // previous call)
    const uint32_t epoch = *(volatile uint32_t*)&a.hdr->dec_epoch;
    const uint32_t sbase = *(volatile uint32_t*)&a.hdr->dec_start_base;
    __syncthreads();  // barriers initialised; every thread has read the tags before the count below
    if (threadIdx.x == 0) red_release_add(&a.hdr->dec_start, 1u);
    const uint32_t tag = epoch + 1u;
    const uint32_t tag16 = (tag - 1u) % 65535u + 1u;
    uint32_t* hw = reinterpret_cast<uint32_t*>(a.dh);  // [K + 1][I] tagged h words

    if (pw >= 0) {
        // ================= producers: the routed items once the routing is known
        if (lane == 0) {
            if (pok && pj < p.n && !mbar_wait(routed, 0, a.wait_ns)) pok = false;
            while (pok && pj < p.n && issue_next(true)) {
            }
            if (!pok) atomicOr(err, ERR_TIMEOUT);
            if (pw == 0) MOE_TL(7);
        }
        // every copy issued must land before the CTA can exit: the latest item of each slot
        __syncwarp();
        asm volatile("bar.sync 2, %0;" ::"n"(kOProducers * 32) : "memory");
        // (lane l of producer 0 takes slot l: a shared-memory operation waits behind the
        // consumers' loads, so one pass over the slots, not one per item)
        if (pw == 0) {
            bool ok = true;
            if (lane < nslot && lane < p.n) {
                int j = lane + nslot * ((p.n - 1 - lane) / nslot);  // the slot's last item
                while (j >= 0 && !issued[j]) j -= nslot;
                if (j >= 0) ok = mbar_poll(&full[lane], ((uint32_t)(j / nslot)) & 1u, a.wait_ns);
            }
            if (!ok) atomicOr(err, ERR_TIMEOUT);
        }
        return;
    }

    // ================= consumers: warp w takes items w, w + kOWarps, ...
    // this lane's chunks of x (packed bf16), straight from global memory into registers (after
    // the wait for the previous kernel above): one memory round trip, no copy through shared
    // memory and no barrier hand-off. A row in host memory crosses the host link once per call
    // instead: CTA c reads its share of the row's 32-bit words and publishes them as tagged
    // words (as the router scores), and each CTA's consumer threads gather all the words from
    // L2 into shared memory, where each warp takes its chunks (every CTA reading the whole row
    // over the link took 4 KB per CTA, 608 KB per call, at ~200 GB/s).
    uint4 xr[kONch];
    if (a.x_host) {
        constexpr int W = kOH / 2;                                 // 32-bit words of the row
        constexpr int kPer = (W + kOWarps * 32 - 1) / (kOWarps * 32);  // words per gathering thread
        const int per = (W + G - 1) / G;
        if (threadIdx.x < per && c * per + (int)threadIdx.x < W) {
            const int i = c * per + threadIdx.x;
            const uint32_t v = __ldcg(reinterpret_cast<const unsigned int*>(a.x) + i);
            publish_u64(a.dx + i, ((uint64_t)tag << 32) | v);
        }
        uint32_t* xs = reinterpret_cast<uint32_t*>(base + g.o_x);
        uint32_t need = 0;
#pragma unroll
        for (int q = 0; q < kPer; ++q)
            if ((int)threadIdx.x + q * kOWarps * 32 < W) need |= 1u << q;
        const uint64_t t0 = global_ns();
        while (need) {
            uint64_t w[kPer];
#pragma unroll
            for (int q = 0; q < kPer; ++q)
                w[q] = ((need >> q) & 1u) ? ld_relaxed_u64(a.dx + threadIdx.x + q * kOWarps * 32) : 0ull;
#pragma unroll
            for (int q = 0; q < kPer; ++q)
                if (((need >> q) & 1u) && (uint32_t)(w[q] >> 32) == tag) {
                    xs[threadIdx.x + q * kOWarps * 32] = (uint32_t)w[q];
                    need &= ~(1u << q);
                }
            if (need && global_ns() - t0 > a.wait_ns) {
                atomicOr(err, ERR_TIMEOUT);
                break;
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kOWarps * 32) : "memory");
#pragma unroll
        for (int q = 0; q < kONch; ++q) xr[q] = reinterpret_cast<const uint4*>(xs)[lane + 32 * q];
    } else {
#pragma unroll
        for (int q = 0; q < kONch; ++q) xr[q] = ld_ro(a.x + 8 * (lane + 32 * q));
    }
#ifdef MOE_TIMELINE
    if (warp == 0 && lane == 0 && xr[kONch - 1].w != 0xffffffffu) MOE_TL(3);  // the compare waits for the loads
#endif
    int s = warp % nslot;
    uint32_t round = warp / nslot;
    for (int j = warp; j < p.n; j += kOWarps) {
        if (!warp_wait(&full[s], round & 1u, lane, a.wait_ns)) {
            if (lane == 0) atomicOr(err, ERR_TIMEOUT);
            break;
        }
        const OMeta m = meta[s];
        const uint32_t d = smem_u32(slots) + (uint32_t)(s * kOSlot);
        if (m.kind == kOkRouter) {
            const uint32_t rows[1] = {d};
            float v[1];
            dot_rows<1>(rows, xr, lane, v);
            // (the testing aid MOE_TEST_SUPPRESS_SCORE keeps CTA 1's scores back, so that every
            // CTA's wait for the scores runs out)
            if (lane == 0 && !(a.test_suppress == MOE_TEST_SUPPRESS_SCORE && c == 1)) {
                float sc = v[0];
                if (m.a < a.E && a.router_b) sc += __bfloat162float(a.router_b[m.a]);
                publish_u64(a.dlog + m.a, ((uint64_t)tag << 32) | (uint64_t)__float_as_uint(sc));
                MOE_TL(4);
            }
        } else if (m.kind == kOkSharedUp || m.kind == kOkUp) {
            // feature a: its gate row, then its up row
            const uint32_t rows[2] = {d, d + kOH * 2};
            float v[2];
            dot_rows<2>(rows, xr, lane, v);
            if (lane == 0) {
                const bf16 h = __float2bfloat16_rn(silu(v[0]) * v[1]);
                const int row = m.kind == kOkSharedUp ? K : rt.inv[m.k];  // h tap: routed rows in dispatch order, then the shared row
                a.h[(size_t)row * kOI + m.a] = h;
                publish_u32(hw + (size_t)m.k * kOI + m.a, (tag16 << 16) | (uint32_t)__bfloat16_as_ushort(h));
            }
        } else {
            uint32_t hv[kOIch][8];  // tagged h words: the bf16 h in the low half
            if (!poll_h(hw + (size_t)m.k * kOI, tag16, hv, lane, a.wait_ns) && lane == 0) atomicOr(err, ERR_TIMEOUT);
            float acc[kOMaxRo];
#pragma unroll
            for (int r0 = 0; r0 < kOMaxRo; r0 += 4) {
                // four rows' loads in flight before their multiplies
                uint4 w[4][kOIch];
#pragma unroll
                for (int r = r0; r < r0 + 4; ++r)
#pragma unroll
                    for (int q = 0; q < kOIch; ++q)
                        w[r - r0][q] = lds128(d + (uint32_t)(min(r, m.n - 1) * kOI * 2) + 16u * (lane + 32 * q));
#pragma unroll
                for (int r = r0; r < r0 + 4; ++r) {
                    acc[r] = 0.f;
#pragma unroll
                    for (int q = 0; q < kOIch; ++q) acc[r] = dot8_bf16_lo(w[r - r0][q], hv[q], acc[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < kOMaxRo; ++r) {
                const float v = warp_sum(acc[r]);
                if (lane == r && r < m.n) ys[m.k * kOMaxOut + (m.a - p.o0) + r] = v;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (j == 0) {
            // warp 0 after its first item: the routing, then the producer may issue the
            // routed items
            route_one(a, rt, tag, lane, routed);
            if (c == 0) write_routing(a, rt, lane);
        }
        s += kOWarps;
        if (s >= nslot) {
            s -= nslot;
            ++round;
        }
    }
    if (warp == 0 && p.n == 0) {  // no item at all: still route, so the producer is released
        route_one(a, rt, tag, lane, routed);
        if (c == 0) write_routing(a, rt, lane);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kOWarps * 32) : "memory");  // every item's down outputs are in ys
    if (threadIdx.x == 0) MOE_TL(8);
    // residual + gated shared output + weighted slots 0..K-1, in that order
    const int tid = threadIdx.x;
    if (tid < p.ro) {
        const int o = p.o0 + tid;
        float acc = resid;
        const float sh = rt.sg * ys[K * kOMaxOut + tid];
        a.Y[(size_t)K * kOH + o] = sh;
        acc += sh;
        for (int k = 0; k < K; ++k) {
            const float v = rt.w[k] * ys[k * kOMaxOut + tid];
            a.Y[(size_t)k * kOH + o] = v;
            acc += v;
        }
        a.out[o] = __float2bfloat16_rn(acc);
    }
    if (tid == 0) MOE_TL(9);
    if (c == 0 && tid == 0) {
        // every CTA has read this call's tag once all have counted themselves in: move the
        // tag and the base on for the next call
        if (!wait_count(&a.hdr->dec_start, sbase, (uint32_t)G, a.wait_ns)) atomicOr(err, ERR_TIMEOUT);
        a.hdr->dec_epoch = tag == 0xffffffffu ? 0u : tag;
        a.hdr->dec_start_base = sbase + (uint32_t)G;
    }
}

#ifdef MOE_TIMELINE
// Copies the timeline of the last one-token call: kTlCtas * kTlEvents global-timer values (ns).
extern "C" int moe_timeline_read(unsigned long long* dst) {
    return (int)cudaMemcpyFromSymbol(dst, g_moe_tl, sizeof(g_moe_tl));
}
extern "C" int moe_timeline_shape(int* ctas, int* events) {
    *ctas = kTlCtas;
    *events = kTlEvents;
    return 0;
}
#endif

static bool decode_geom(int cap, OGeom* g) {
    int o = 0;
    g->o_rt = o; o += ((int)sizeof(ORoute) + 127) & ~127;
    g->o_ys = o; o += (kOMaxK + 1) * kOMaxOut * 4;
    g->o_bar = o; o += (2 * kOMaxSlots + 1) * 8;
    g->o_meta = o; o += kOMaxSlots * (int)sizeof(OMeta);
    g->o_iss = o; o += kOMaxItems;
    o = (o + 15) & ~15;
    g->o_x = o; o += kOH * 2;  // the token row, when it is read from host memory
    o = (o + 1023) & ~1023;
    g->o_slot = o;
    const int room = cap - 1024 - o;  // 1024: alignment of the dynamic base
    g->nslot = room / kOSlot < kOMaxSlots ? room / kOSlot : kOMaxSlots;
    // A multiple of the consumer warps: warp w consumes items w, w + kOWarps, ..., so the items
    // of one slot (j, j + nslot, ...) are all consumed by the same warp, in order. That is what
    // makes a parity wait on the slot's barrier exact: a warp never asks for a slot's next
    // phase before it has consumed the previous one, so the barrier cannot still be a phase
    // behind (where the parity test would take the phase before that for the one asked for).
    // kOWarps is a multiple of kOProducers, so each slot also keeps one producer.
    g->nslot -= g->nslot % kOWarps;
    g->smem = 1024 + o + g->nslot * kOSlot;
    return g->nslot >= kOWarps;
}

// Dynamic shared memory one CTA of the kernel may use on the current device (0 on failure).
static int dynamic_smem_cap() {
    static int cap[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!cap[dev]) {
        int optin = 0;
        cudaFuncAttributes fa;
        if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaFuncGetAttributes(&fa, k_decode_fused) != cudaSuccess)
            return 0;
        const int c = optin - (int)fa.sharedSizeBytes;
        if (c <= 0 ||
            cudaFuncSetAttribute(k_decode_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, c) != cudaSuccess)
            return 0;
        cap[dev] = c;
    }
    return cap[dev];
}

// The CTAs wait on one another, so the grid (one CTA per SM) must fit on the device at once:
// at least one CTA of this size per SM (checked once per device; the kernel is launched as an
// ordinary programmatic launch, see launch_decode_fused).
static bool one_cta_per_sm(const OGeom& g) {
    static int fits[64] = {};  // 0 unknown, 1 yes, 2 no
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!fits[dev]) {
        int n = 0;
        const bool ok = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_decode_fused, kOThreads, (size_t)g.smem) ==
                            cudaSuccess &&
                        n >= 1;
        (void)cudaGetLastError();
        fits[dev] = ok ? 1 : 2;
    }
    return fits[dev] == 1;
}

// The kernel is built for the pages' layer shape (H = 2048, expert widths 512) and one token;
// other shapes take the routing and streaming kernels.
bool decode_fused_supported(const LayerArgs& a) {
    if (!(a.T == 1 && a.H == kOH && a.I == kOI && a.Is == kOI && a.K <= kOMaxK && a.E <= 256 && a.num_sms >= 1 &&
          a.dlog && a.dh))
        return false;
    // output rows per CTA within one down item; the items issued before the ring is shared
    // (router rows, shared features) within the ring
    const int G = a.num_sms;
    const int ro = (kOH + G - 1) / G;
    if (ro > kOMaxOut || (a.E + G) / G + (kOI + G - 1) / G > kOWarps) return false;
    if ((a.E + G) / G + (kOI + G - 1) / G + (a.K * kOI + G - 1) / G + (a.K + 1) * ((ro + kOMaxRo - 1) / kOMaxRo) >
        kOMaxItems)
        return false;
    OGeom g;
    return decode_geom(dynamic_smem_cap(), &g) && one_cta_per_sm(g);
}

cudaError_t launch_decode_fused(const LayerArgs& a, cudaStream_t s) {
    OGeom g;
    if (!decode_geom(dynamic_smem_cap(), &g)) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.num_sms);
    cfg.blockDim = dim3(kOThreads);
    cfg.dynamicSmemBytes = (size_t)g.smem;
    cfg.stream = s;
    // Programmatic serialization: the launch and each CTA's set-up overlap the end of the
    // previous kernel (the kernel waits for it before it reads anything that kernel may write).
    // The CTAs wait on one another, which needs all of them resident at once: one CTA per SM
    // fits (decode_fused_supported checks it), and each CTA waits for the previous grid to
    // complete before its first wait on another CTA, so by then every SM is free for this
    // grid's CTAs. Not a cooperative launch: measured, that holds each launch back until the
    // previous kernel has left the GPU (18.98 us per layer launched one by one, against 16.37 us
    // without it; 16.40 against 16.13 us in a CUDA graph). Work on other streams that holds SMs
    // for longer than the wait limit makes the call end with MOE_ERR_TIMEOUT. A driver that
    // refuses the programmatic launch gets a plain launch from then on.
    static std::atomic<int> pdl_refused{0};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_refused.load() ? 0 : 1;
    cudaError_t e;
    MOE_LAUNCH(MOE_KERNEL_DECODE_FUSED, s, (e = cudaLaunchKernelEx(&cfg, k_decode_fused, a, g)));
    if (e != cudaSuccess && cfg.numAttrs == 1 && e != cudaErrorStreamCaptureInvalidated &&
        e != cudaErrorStreamCaptureUnsupported) {
        (void)cudaGetLastError();
        pdl_refused.store(1);
        cfg.numAttrs = 0;
        MOE_LAUNCH(MOE_KERNEL_DECODE_FUSED, s, (e = cudaLaunchKernelEx(&cfg, k_decode_fused, a, g)));
    }
    return e;
}

}  // namespace moe
