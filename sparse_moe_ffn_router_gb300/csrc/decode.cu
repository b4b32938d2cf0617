// decode.cu -- the whole MoE layer for a few tokens (T <= 8) in one persistent kernel;
// moe_forward runs it for a single token (from two tokens on the router and streaming expert
// kernels, with their larger ring, are faster).
//
// At decode the layer streams ~55 MB of weights per token ("Qwen3.6-35B-A3B -- Architecture
// Overview", MoE FFN: router 2048 -> 256 plus the shared-expert gate, 8 routed SwiGLU experts
// with merged gate_up [1024 x 2048] and down [2048 x 512], one always-on shared expert of the
// same shape), and every step depends on the one before. One CTA per SM runs the whole layer
// with two grid-wide exchanges:
//
//   1. router rows: CTA c scores its ceil((E+1)/G) rows of the router (the shared-gate row is
//      row E) for every token and stores each score as one 64-bit word together with the tag
//      of this call, so a reader recognises fresh scores by their tag (no flag, no fence);
//   2. shared gate_up: CTA c's even share of the shared expert's features (no routing needed),
//      computed while the other CTAs' scores arrive;
//   3. routing: EVERY CTA reads the T x (E+1) tagged scores and computes top-K, the
//      renormalised weights, the shared gate and the dispatch (counts, offsets, permutation)
//      itself. All CTAs derive the same tables, so no second exchange is needed for them;
//   4. routed gate_up: CTA c's even share of the n_act x I (expert, feature) pairs. Like the
//      scores, its h values are stored as tagged 64-bit words (two bf16 values and the tag);
//   5. down + combine: CTA c owns output rows [c*H/G, (c+1)*H/G) of every expert, shared and
//      routed. The shared expert's block comes right after step 3 (its h values were written in
//      step 2), the routed blocks stream in behind step 4; the CTA gathers the tagged h rows
//      into shared memory as soon as they carry this call's tag, multiplies, and sums residual
//      + gated shared output + weighted slots 0..K-1 of its rows in that fixed order.
//
// Roles: a producer warp streams each stage's rows into a ring of shared-memory stages with 1-D
// TMA bulk copies (one per row; rows 16 bytes apart modulo 128 so ldmatrix is conflict-free);
// 8 consumer warps compute (router rows as warp dot products; gate_up and down with warp-level
// bf16 MMAs, m16n8k16, fp32 accumulate, partial sums added in a fixed order), the routing and
// the gathers. No exchange needs a flag or a fence: a word is fresh when it carries this
// call's tag. Every wait is bounded (~1 s): a timeout sets MOE_ERR_TIMEOUT and the kernel still
// runs to its end with in-range indices. Each CTA counts itself in when it starts; CTA 0 moves
// the tag on at its end once all are in, so nothing has to be re-armed between calls.
#include "launch.h"
#include "ring.cuh"

namespace moe {

constexpr int kDTT = 8;                     // max tokens
constexpr int kDMaxH = 2048, kDMaxI = 512;  // largest hidden size / expert width
constexpr int kDMaxP = kDTT * 8;            // max (token, slot) pairs
constexpr int kDBlk = 4;                    // max down blocks per ring stage
constexpr int kDThreads = kConsumers + 32;  // 8 consumer warps and the producer
constexpr int kProducerWarp = kWarps;
constexpr uint32_t kPollNs = 128;           // longest sleep between two polls

enum { kStRoute = 0, kStUp = 1, kStTopK = 2, kStDown = 3, kStEnd = 4 };

// What one ring stage holds (written by the producer before the stage's barrier completes).
struct DMeta {
    int type;
    int n;           // route: rows; up: features; down: blocks
    int row0;        // route: first router row; up: first h row
    int f0;          // up: first feature
    int mt;          // up: tokens
    uint32_t toks;   // up: token of each of its mt h rows, 4 bits each
    int blk[kDBlk];  // down: expert slot of each block (0: shared expert, j >= 1: act[j - 1]);
                     // a stage holds the shared block alone or routed blocks only
};

// Shared-memory geometry of one launch, fixed on the host.
struct DGeom {
    int sf;     // features per gate_up stage (8 or 4); a stage holds 2 * sf rows of H
    int nst;    // ring stages
    int xp;     // pitch of x rows and H-long weight rows (2H + 16 bytes)
    int dp;     // pitch of h rows and down rows (2 Imax + 16 bytes)
    int rr;     // router rows per CTA
    int ro;     // output rows per CTA (at most)
    int nbs;    // down blocks per ring stage (1, 2 or 4); a block holds ro rows
    int stage;  // stage bytes
    int o_xs, o_hs, o_ys, o_red, o_st, o_meta, o_bar, smem;
};

// Routing tables, identical in every CTA.
struct DRoute {
    int sid[kDMaxP];    // expert of pair p = t*K + k
    float sw[kDMaxP];   // renormalised weight of pair p
    int less[kDMaxP];   // pairs whose expert is lower than pair p's
    int rank[kDMaxP];   // earlier pairs with pair p's expert
    int pcnt[kDMaxP];   // pairs with pair p's expert
    int perm[kDMaxP];   // pair at each dispatch position
    int inv[kDMaxP];    // dispatch position of each pair
    int act[kDMaxP];    // used experts, ascending
    int aoff[kDMaxP];   // first dispatch position of act[j]
    int acnt[kDMaxP];   // pairs of act[j]
    float sgate[kDTT];
    int n_act;
};

inline int round_up128(int b) { return (b + 127) & ~127; }

// Geometry for sf features per stage and nst stages; false if the layer does not fit it.
inline bool decode_geom(const LayerArgs& a, int G, int sf, int nst, DGeom* g) {
    g->sf = sf;
    g->nst = nst;
    g->xp = 2 * a.H + 16;
    g->dp = 2 * a.Imax + 16;
    g->rr = (a.E + 1 + G - 1) / G;
    g->ro = (a.H + G - 1) / G;
    g->stage = 2 * sf * g->xp;
    const int nb = g->stage / (g->ro * g->dp);
    g->nbs = nb >= 4 ? 4 : nb >= 2 ? 2 : nb;
    if (g->rr > 2 * sf || g->ro > 16 || g->nbs < 1 || (a.I | a.Is) & 1) return false;
    const int P = a.T * a.K;
    int o = 0;
    g->o_xs = o; o += round_up128(a.T * g->xp);
    g->o_hs = o; o += round_up128((P + a.T) * g->dp);
    g->o_ys = o; o += round_up128((P + a.T) * 16 * 4);
    g->o_red = o; o += 2 * kWarps * 32 * 16;
    g->o_st = o; o += nst * g->stage;
    g->o_meta = o; o += round_up128(nst * (int)sizeof(DMeta));
    g->o_bar = o; o += round_up128((2 * nst + 2) * 8);
    g->smem = o + 128;  // room to align the dynamic base to 128 bytes
    return true;
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Poll until *p - base >= n (unsigned, acquire), sleeping up to kPollNs between polls; false
// after ~1 s.
__device__ __forceinline__ bool wait_count(const uint32_t* p, uint32_t base, uint32_t n) {
    if (ld_acquire(p) - base >= n) return true;
    const uint64_t t0 = global_ns();
    uint32_t ns = 32;
    for (;;) {
        __nanosleep(ns);
        if (ld_acquire(p) - base >= n) return true;
        if (ns < kPollNs) ns <<= 1;
        if (global_ns() - t0 > 1000000000ull) return false;
    }
}

// Lane 0 waits for a barrier phase (bounded); the warp shares the outcome and, through the
// warp barrier, the visibility of what completed the phase.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int lane) {
    bool ok = lane == 0 ? mbar_wait(bar, parity) : true;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok;
}

// Barrier of the consumer warps that also counts the threads whose predicate is true.
__device__ __forceinline__ int consumers_count(bool p) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.popc.u32 %0, 1, %2, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)p), "n"(kConsumers)
        : "memory");
    return (int)r;
}

// D[16 x 8] += A[16 x 16 ksteps] B for this lane's A row (a_row: byte address of the row the
// lane feeds to ldmatrix, i.e. tile row lane % 16) and B row (token row of lane % 8), K range
// starting at element k0. Even and odd K steps go to two accumulators (two short dependency
// chains), added at the end.
__device__ __forceinline__ void mma_rows(float (&d)[4], uint32_t a_row, uint32_t b_row, int k0, int ksteps, int lane) {
    const uint32_t a = a_row + (uint32_t)((k0 + 8 * (lane >> 4)) * 2);
    const uint32_t b = b_row + (uint32_t)((k0 + 8 * ((lane >> 3) & 1)) * 2);
    float e[4] = {0.f, 0.f, 0.f, 0.f};
    int k = 0;
#pragma unroll 2
    for (; k + 1 < ksteps; k += 2) {
        uint32_t a0, a1, a2, a3, b0, b1, c0, c1, c2, c3, f0, f1;
        ldsm_x4(a + k * 32, a0, a1, a2, a3);
        ldsm_x2(b + k * 32, b0, b1);
        ldsm_x4(a + k * 32 + 32, c0, c1, c2, c3);
        ldsm_x2(b + k * 32 + 32, f0, f1);
        mma16816(d, a0, a1, a2, a3, b0, b1);
        mma16816(e, c0, c1, c2, c3, f0, f1);
    }
    if (k < ksteps) {
        uint32_t a0, a1, a2, a3, b0, b1;
        ldsm_x4(a + k * 32, a0, a1, a2, a3);
        ldsm_x2(b + k * 32, b0, b1);
        mma16816(d, a0, a1, a2, a3, b0, b1);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] += e[i];
}

// ---------------------------------------------------------------------------------------
// Routing ("Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: softmax over the 256 router
// scores, the 8 highest kept and renormalised; ties go to the lower expert index).

// Top-K of token t by one warp. Lane l polls the tagged scores of experts l, l+32, ... (lane 0
// also the shared-gate score) until all carry this call's tag; each of K rounds then takes the
// largest remaining key (warp max) and, among equal keys, the lowest expert index (warp min).
// The weights are the softmax over the kept scores, which equals the full softmax renormalised
// over them; lane k holds slot k.
__device__ void route_token(const LayerArgs& a, DRoute& rt, int t, int lane, uint32_t tag) {
    const uint64_t* l = a.dlog + (size_t)t * (a.E + 1);
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
        // all pending words are requested before any is examined (one round trip per poll)
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
        if (!__any_sync(0xffffffffu, need != 0)) break;
        if (global_ns() - t0 > 1000000000ull) {
            timed_out = true;
            break;
        }
        __nanosleep(64);
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
    const float ex = lane < a.K ? expf(myv - v0) : 0.f;
    const float s = warp_sum(ex);
    if (lane < a.K) {
        rt.sid[t * a.K + lane] = mye;
        rt.sw[t * a.K + lane] = ex / s;
    }
    if (lane == 0) {
        const float z = router_score(__uint_as_float(val[8]), a.flags);
        if (!isfinite(z)) bad = true;
        rt.sgate[t] = 1.0f / (1.0f + expf(-z));
        if (timed_out) atomicOr(&a.hdr->err, ERR_TIMEOUT);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&a.hdr->err, ERR_NONFINITE_SCORE);
}

// Dispatch of the P pairs by the consumer threads (thread p takes pair p): a stable counting
// sort by expert -- pair p goes to position #{pairs with a lower expert} + #{earlier pairs with
// its expert} -- and the ascending list of used experts with their first position and count.
// Starts and ends with a barrier of the consumers.
__device__ void route_dispatch(DRoute& rt, int P, int tid) {
    if (tid < P) {
        const int e = rt.sid[tid];
        int less = 0, cnt = 0, rank = 0;
        for (int q = 0; q < P; ++q) {
            const int eq = rt.sid[q];
            less += eq < e;
            cnt += eq == e;
            rank += (eq == e) & (q < tid);
        }
        rt.less[tid] = less;
        rt.rank[tid] = rank;
        rt.pcnt[tid] = cnt;
    }
    consumers_count(false);  // barrier: pass 1 complete
    int first = 0;
    if (tid < P) {
        const int e = rt.sid[tid], pos = rt.less[tid] + rt.rank[tid];
        rt.perm[pos] = tid;
        rt.inv[tid] = pos;
        if (rt.rank[tid] == 0) {
            first = 1;
            int j = 0;
            for (int q = 0; q < P; ++q) j += (rt.rank[q] == 0) & (rt.sid[q] < e);
            rt.act[j] = e;
            rt.aoff[j] = rt.less[tid];
            rt.acnt[j] = rt.pcnt[tid];
        }
    }
    const int na = consumers_count(first != 0);  // barrier: tables complete
    if (tid == 0) rt.n_act = na;
    consumers_sync();
}

// Even split of n items over G CTAs, boundaries rounded down to even (h values travel in pairs).
__device__ __forceinline__ int even_split(int n, int c, int G) { return (int)((long long)c * n / G) & ~1; }

// Copies h rows r0 .. r0+nr-1 (features 0 .. inner-1) of this call from their tagged words into
// shared memory (pitch dp), each consumer thread polling its words until they carry `tag`.
// False after ~1 s; the words not yet fresh are then copied as they are.
__device__ bool gather_h(const LayerArgs& a, uint8_t* hs, int dp, int r0, int nr, int inner, uint32_t tag, int tid) {
    constexpr int kB = 16;  // words in flight per thread
    const int wpr = inner / 2, ldw = a.Imax / 2, n = nr * wpr;
    const uint64_t t0 = global_ns();
    bool ok = true;
    for (int base = 0; base < n; base += kConsumers * kB) {
        uint32_t need = 0;
#pragma unroll
        for (int q = 0; q < kB; ++q)
            if (base + q * kConsumers + tid < n) need |= 1u << q;
        while (need) {
            uint64_t w[kB];
#pragma unroll
            for (int q = 0; q < kB; ++q) {
                const int idx = base + q * kConsumers + tid, r = idx / wpr;
                w[q] = ((need >> q) & 1u) ? ld_relaxed_u64(a.dh + (size_t)(r0 + r) * ldw + (idx - r * wpr)) : 0ull;
            }
            const bool give_up = !ok || global_ns() - t0 > 1000000000ull;
            uint32_t still = need;
#pragma unroll
            for (int q = 0; q < kB; ++q)
                if (((need >> q) & 1u) && ((uint32_t)(w[q] >> 32) == tag || give_up)) {
                    const int idx = base + q * kConsumers + tid, r = idx / wpr;
                    *reinterpret_cast<uint32_t*>(hs + (size_t)(r0 + r) * dp + (idx - r * wpr) * 4) = (uint32_t)w[q];
                    still &= ~(1u << q);
                }
            if (give_up) ok = false;
            need = still;
            if (need) __nanosleep(64);
        }
    }
    return ok;
}

// ---------------------------------------------------------------------------------------

__global__ void __launch_bounds__(kDThreads, 1) k_decode_fused(LayerArgs a, DGeom g) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ DRoute rt;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* base = smem_raw + (((raw + 127u) & ~127u) - raw);
    uint8_t* xs = base + g.o_xs;
    uint8_t* hs = base + g.o_hs;
    float* Ys = reinterpret_cast<float*>(base + g.o_ys);  // [P + T][16] unscaled down outputs
    float* red = reinterpret_cast<float*>(base + g.o_red);
    uint8_t* stg = base + g.o_st;
    DMeta* meta = reinterpret_cast<DMeta*>(base + g.o_meta);
    uint64_t* full = reinterpret_cast<uint64_t*>(base + g.o_bar);
    uint64_t* empty = full + g.nst;
    uint64_t* xbar = empty + g.nst;
    uint64_t* routed = xbar + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int T = a.T, H = a.H, E = a.E, K = a.K, P = T * K;
    uint32_t* err = &a.hdr->err;
    // this call's tag and the CTA starts of earlier calls (both advanced by CTA 0 of the
    // previous call)
    const uint32_t epoch = *(volatile uint32_t*)&a.hdr->dec_epoch;
    const uint32_t tag = epoch + 1u;
    const uint32_t sbase = *(volatile uint32_t*)&a.hdr->dec_start_base;
    const int o0 = c * H / G, ro = (c + 1) * H / G - o0;  // this CTA's output rows

    if (threadIdx.x == 0) {
        for (int s = 0; s < g.nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        mbar_init(xbar, 1);
        mbar_init(routed, 1);
        fence_mbar_init();
    }
    __syncthreads();  // also orders every thread's reads of the tag before the count below
    if (threadIdx.x == 0) red_release_add(&a.hdr->dec_start, 1u);

    if (warp == kProducerWarp) {
        // ================= producer: fills the stages in the order the consumers take them
        if (lane == 0) mbar_arrive_expect_tx(xbar, (uint32_t)(T * H * 2));
        __syncwarp();
        if (lane < T) bulk_load(xs + (size_t)lane * g.xp, a.x + (size_t)lane * H, H * 2, xbar);
        int it = 0;
        bool ok = true;
        auto claim = [&]() -> int {  // next stage, once the consumers have released it
            const int s = it % g.nst;
            if (!warp_wait(&empty[s], (((uint32_t)(it / g.nst)) & 1u) ^ 1u, lane)) ok = false;
            return s;
        };
        auto post = [&](int type) {  // a stage without copies
            const int s = claim();
            if (!ok) return;
            if (lane == 0) {
                meta[s].type = type;
                mbar_arrive(&full[s]);
            }
            __syncwarp();
            ++it;
        };
        // gate rows f0.. to stage rows 0.., up rows (inner + f0).. to stage rows sf..
        auto issue_up = [&](const bf16* W, int inner, int f0, int n, int row0, int mt, uint32_t toks) {
            const int s = claim();
            if (!ok) return;
            uint8_t* st = stg + (size_t)s * g.stage;
            if (lane == 0) {
                DMeta& m = meta[s];
                m.type = kStUp;
                m.n = n;
                m.row0 = row0;
                m.f0 = f0;
                m.mt = mt;
                m.toks = toks;
                mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * n * H * 2));
            }
            __syncwarp();
            if (lane < n)
                bulk_load(st + (size_t)lane * g.xp, W + (size_t)(f0 + lane) * H, H * 2, &full[s]);
            else if (lane >= 16 && lane < 16 + n)
                bulk_load(st + (size_t)(g.sf + lane - 16) * g.xp, W + (size_t)(inner + f0 + lane - 16) * H, H * 2,
                          &full[s]);
            ++it;
        };

        // 1. router rows (row E is the shared-expert gate)
        const int r0 = c * g.rr, nrr = max(0, min(E + 1, r0 + g.rr) - r0);
        if (nrr > 0) {
            const int s = claim();
            if (ok) {
                uint8_t* st = stg + (size_t)s * g.stage;
                if (lane == 0) {
                    meta[s].type = kStRoute;
                    meta[s].n = nrr;
                    meta[s].row0 = r0;
                    mbar_arrive_expect_tx(&full[s], (uint32_t)(nrr * H * 2));
                }
                __syncwarp();
                if (lane < nrr) {
                    const int row = r0 + lane;
                    bulk_load(st + (size_t)lane * g.xp, row < E ? a.router_w + (size_t)row * H : a.sg, H * 2,
                              &full[s]);
                }
                ++it;
            }
        }
        // down rows o0..o0+ro-1 of block j0.. (nb blocks) into the next stage
        auto issue_down = [&](int j0, int nb) {
            const int s = claim();
            if (!ok) return;
            uint8_t* st = stg + (size_t)s * g.stage;
            if (lane == 0) {
                uint32_t bytes = 0;
                DMeta& m = meta[s];
                m.type = kStDown;
                m.n = nb;
                for (int b = 0; b < nb; ++b) {
                    m.blk[b] = j0 + b;
                    bytes += (uint32_t)(ro * (j0 + b == 0 ? a.Is : a.I) * 2);
                }
                mbar_arrive_expect_tx(&full[s], bytes);
            }
            __syncwarp();
            for (int idx = lane; idx < nb * ro; idx += 32) {
                const int b = idx / ro, r = idx - b * ro, j = j0 + b;
                const int inner = j == 0 ? a.Is : a.I;
                const bf16* W = j == 0 ? a.sd : a.down + (size_t)rt.act[j - 1] * H * a.I;
                bulk_load(st + (size_t)(b * g.ro + r) * g.dp, W + (size_t)(o0 + r) * inner, inner * 2, &full[s]);
            }
            ++it;
        };
        // 2. shared gate_up: features [c*Is/G, (c+1)*Is/G), all tokens, h rows P..P+T-1
        //    (computed while the other CTAs' scores arrive)
        const int fs0 = even_split(a.Is, c, G), fs1 = even_split(a.Is, c + 1, G);
        for (int f = fs0; f < fs1 && ok; f += g.sf)
            issue_up(a.sgu, a.Is, f, min(g.sf, fs1 - f), P, T, 0x76543210u);
        // 3. the consumers compute the routing and hand the tables over through `routed`; the
        //    shared expert's down rows (output rows o0..o0+ro-1, slot 0) stream in meanwhile and
        //    are multiplied while the first routed weights are in flight
        if (ok) post(kStTopK);
        if (ok && ro > 0) issue_down(0, 1);
        if (ok && !warp_wait(routed, 0, lane)) ok = false;
        // 4. routed gate_up: (expert, feature) pairs [c*F/G, (c+1)*F/G) of the F = n_act * I
        const int n_act = ok ? rt.n_act : 0;
        const int F = n_act * a.I;
        const int g1 = even_split(F, c + 1, G);
        for (int gi = even_split(F, c, G); gi < g1 && ok;) {
            const int j = gi / a.I, f = gi - j * a.I;
            const int n = min(g.sf, min(g1 - gi, a.I - f));
            const int e = rt.act[j];
            const int row0 = rt.aoff[j], mt = rt.acnt[j];
            uint32_t toks = 0;
            for (int q = 0; q < mt; ++q) toks |= (uint32_t)(rt.perm[row0 + q] / K) << (4 * q);
            issue_up(a.gate_up + (size_t)e * 2 * a.I * H, a.I, f, n, row0, mt, toks);
            gi += n;
        }
        // 5. down rows o0..o0+ro-1 of each used expert (slots 1..n_act)
        for (int j0 = 1; ro > 0 && j0 <= n_act && ok; j0 += g.nbs) issue_down(j0, min(g.nbs, n_act + 1 - j0));
        if (!ok && lane == 0) atomicOr(err, ERR_TIMEOUT);
        // every copy issued must land before the CTA can exit
        if (lane == 0) {
            for (int k = 0; k < g.nst && it - 1 - k >= 0; ++k) {
                const int j = it - 1 - k;
                if (!mbar_wait(&full[j % g.nst], ((uint32_t)(j / g.nst)) & 1u)) atomicOr(err, ERR_TIMEOUT);
            }
            if (!mbar_wait(xbar, 0)) atomicOr(err, ERR_TIMEOUT);
        }
        __syncwarp();
        if (ok) post(kStEnd);
        return;
    }

    // ================= consumers
    const int tid = threadIdx.x;
    // router bias of the router row whose slices this warp sums (router stage with up to 8
    // rows, see there), requested before the first wait
    float bias = 0.f;
    {
        const int nrr = max(0, min(E + 1, c * g.rr + g.rr) - c * g.rr);
        const int wpr = nrr <= 1 ? 8 : nrr <= 2 ? 4 : nrr <= 4 ? 2 : 1;
        const int row = c * g.rr + warp / wpr;
        if (warp / wpr < nrr && row < E && a.router_b) bias = __bfloat162float(a.router_b[row]);
    }
    if (!consumers_all(warp_wait(xbar, 0, lane)) && tid == 0) atomicOr(err, ERR_TIMEOUT);
    int rb = 0;  // reduction buffer in use (alternates between the stages that reduce)
    bool have_sh = false, have_rh = false;  // shared / routed h rows gathered
    const uint32_t xs_a = smem_u32(xs), hs_a = smem_u32(hs);
    for (int it = 0;; ++it) {
        const int s = it % g.nst;
        if (!consumers_all(warp_wait(&full[s], ((uint32_t)(it / g.nst)) & 1u, lane))) {
            if (tid == 0) atomicOr(err, ERR_TIMEOUT);
            break;
        }
        const DMeta m = meta[s];
        const uint8_t* stp = stg + (size_t)s * g.stage;
        const uint32_t sa = smem_u32(stp);
        float* rbuf = red + rb * kWarps * 32 * 4;
        auto release = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        };

        if (m.type == kStEnd) {
            consumers_sync();  // every block's Ys rows are written
            // residual + gated shared output + weighted slots 0..K-1, in that order
            for (int idx = tid; idx < T * ro; idx += kConsumers) {
                const int t = idx / ro, r = idx - t * ro, o = o0 + r;
                float acc = a.residual ? __bfloat162float(a.residual[(size_t)t * H + o]) : 0.f;
                float* yt = a.Y + (size_t)t * (K + 1) * H + o;
                const float sh = rt.sgate[t] * Ys[(P + t) * 16 + r];
                yt[(size_t)K * H] = sh;
                acc += sh;
                for (int k = 0; k < K; ++k) {
                    const int p = t * K + k;
                    const float v = rt.sw[p] * Ys[p * 16 + r];
                    yt[(size_t)k * H] = v;
                    acc += v;
                }
                a.out[(size_t)t * H + o] = __float2bfloat16_rn(acc);
            }
            if (c == 0 && tid == 0) {
                // every CTA has read this call's tag once all have counted themselves in: move
                // the tag and the base on for the next call
                if (!wait_count(&a.hdr->dec_start, sbase, (uint32_t)G)) atomicOr(err, ERR_TIMEOUT);
                a.hdr->dec_epoch = tag == 0xffffffffu ? 0u : tag;
                a.hdr->dec_start_base = sbase + (uint32_t)G;
            }
            break;
        }

        if (m.type == kStTopK) {
            release();
            if (warp < T) route_token(a, rt, warp, lane, tag);
            consumers_sync();
            route_dispatch(rt, P, tid);
            if (tid == 0) mbar_arrive(routed);
            if (c == 0) {
                // the routing results of this call, for the caller and the workspace taps
                for (int p = tid; p < P; p += kConsumers) {
                    a.ids[p] = rt.sid[p];
                    a.topw[p] = rt.sw[p];
                    a.perm[p] = rt.perm[p];
                    a.inv[p] = rt.inv[p];
                }
                for (int e = tid; e <= E; e += kConsumers) {
                    int less = 0, cnt = 0;
                    for (int q = 0; q < P; ++q) {
                        less += rt.sid[q] < e;
                        cnt += rt.sid[q] == e;
                    }
                    a.offsets[e] = less;
                    if (e < E) a.counts[e] = cnt;
                }
                for (int j = tid; j < rt.n_act; j += kConsumers) a.act[j] = rt.act[j];
                if (tid < T) a.sgate[tid] = rt.sgate[tid];
                if (tid == 0) a.hdr->n_act = rt.n_act;
            }
            continue;
        }

        if (m.type == kStRoute) {
            // rows row0 .. row0+n-1 for every token: wpr warps per row, each a K slice of H/wpr
            // (lane l takes elements 8l + 256i of it); the slices' sums are added in a fixed
            // order by the row's first warp. Beyond 8 rows, warps loop over rows.
            const int wpr = m.n <= 1 ? 8 : m.n <= 2 ? 4 : m.n <= 4 ? 2 : 1;
            const int kl = H / wpr, q = warp % wpr;
            float* part = rbuf;  // [warp][kDTT] slice sums
            for (int rl = warp / wpr; rl < m.n; rl += kWarps / wpr) {
                const uint8_t* wr = stp + (size_t)rl * g.xp;
                float acc[kDTT];
#pragma unroll
                for (int t = 0; t < kDTT; ++t) acc[t] = 0.f;
                for (int k = q * kl + lane * 8; k < (q + 1) * kl; k += 256) {
                    const uint4 wv = *reinterpret_cast<const uint4*>(wr + k * 2);
#pragma unroll
                    for (int t = 0; t < kDTT; ++t)
                        if (t < T) {
                            float xf[8];
                            unpack8(*reinterpret_cast<const uint4*>(xs + (size_t)t * g.xp + k * 2), xf);
                            acc[t] = dot8(wv, xf, acc[t]);
                        }
                }
                float mine = 0.f;
#pragma unroll
                for (int t = 0; t < kDTT; ++t)
                    if (t < T) {
                        const float v = warp_sum(acc[t]);
                        if (lane == t) mine = v;
                    }
                if (wpr == 1) {
                    if (lane < T) {
                        const int row = m.row0 + rl;
                        const float b = (row < E && a.router_b) ? __bfloat162float(a.router_b[row]) : 0.f;
                        st_relaxed_u64(a.dlog + (size_t)lane * (E + 1) + row,
                                       ((uint64_t)tag << 32) | (uint64_t)__float_as_uint(mine + b));
                    }
                } else if (lane < T) {
                    part[warp * kDTT + lane] = mine;
                }
            }
            release();
            if (wpr > 1) {
                consumers_sync();
                rb ^= 1;
                if (q == 0 && warp / wpr < m.n && lane < T) {
                    float v = 0.f;
                    for (int w = warp; w < warp + wpr; ++w) v += part[w * kDTT + lane];
                    const int row = m.row0 + warp / wpr;
                    st_relaxed_u64(a.dlog + (size_t)lane * (E + 1) + row,
                                   ((uint64_t)tag << 32) | (uint64_t)__float_as_uint(v + bias));
                }
            }
            continue;
        }

        float d[4] = {0.f, 0.f, 0.f, 0.f};
        if (m.type == kStUp) {
            const int r = lane & 15, gi = r & 7;  // tile rows 0-7: gate of feature f0+gi, 8-15: its up row
            const int srow = gi < m.n ? (r >> 3) * g.sf + gi : 0;
            const int tt = lane & 7;
            const int tok = tt < m.mt ? (int)((m.toks >> (4 * tt)) & 15u) : 0;
            mma_rows(d, sa + (uint32_t)(srow * g.xp), xs_a + (uint32_t)(tok * g.xp), warp * (H / kWarps),
                     H / kWarps / 16, lane);
            release();
            *reinterpret_cast<float4*>(rbuf + (warp * 32 + lane) * 4) = make_float4(d[0], d[1], d[2], d[3]);
            consumers_sync();
            rb ^= 1;
            if (warp == 0) {
                float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float4 q4 = *reinterpret_cast<const float4*>(rbuf + (w * 32 + lane) * 4);
                    v[0] += q4.x; v[1] += q4.y; v[2] += q4.z; v[3] += q4.w;
                }
                // feature f0+rl for tokens t, t+1: the plain bf16 h (workspace tap) and, from the
                // lanes of even features, tagged pairs (f, f+1) for the other CTAs
                const int rl = lane >> 2, t = 2 * (lane & 3);
                const bf16 h0 = __float2bfloat16_rn(silu(v[0]) * v[2]);
                const bf16 h1 = __float2bfloat16_rn(silu(v[1]) * v[3]);
                const uint32_t u0 = __bfloat16_as_ushort(h0), u1 = __bfloat16_as_ushort(h1);
                const uint32_t n0 = __shfl_down_sync(0xffffffffu, u0, 4), n1 = __shfl_down_sync(0xffffffffu, u1, 4);
                if (rl < m.n) {
                    bf16* hrow = a.h + (size_t)(m.row0 + t) * a.Imax + m.f0 + rl;
                    if (t < m.mt) hrow[0] = h0;
                    if (t + 1 < m.mt) hrow[a.Imax] = h1;
                    if (!(rl & 1)) {
                        uint64_t* w = a.dh + (size_t)(m.row0 + t) * (a.Imax / 2) + (m.f0 + rl) / 2;
                        const uint64_t hi = (uint64_t)tag << 32;
                        if (t < m.mt) st_relaxed_u64(w, hi | (n0 << 16) | u0);
                        if (t + 1 < m.mt) st_relaxed_u64(w + a.Imax / 2, hi | (n1 << 16) | u1);
                    }
                }
            }
            continue;
        }

        // kStDown: block b of this stage by warps b*wpb .. b*wpb+wpb-1, each one K slice; the h
        // rows it needs are gathered first (all consumers)
        if (meta[s].blk[0] == 0 ? !have_sh : !have_rh) {
            const bool sh = meta[s].blk[0] == 0;
            const bool got = sh ? gather_h(a, hs, g.dp, P, T, a.Is, tag, tid) : gather_h(a, hs, g.dp, 0, P, a.I, tag, tid);
            if (!consumers_all(got) && tid == 0) atomicOr(err, ERR_TIMEOUT);
            (sh ? have_sh : have_rh) = true;
        }
        const int wpb = min(4, kWarps / g.nbs);
        const int b = warp / wpb, kq = warp - b * wpb;
        int j = 0, mt = 0, hrow0 = 0;
        if (b < m.n) {
            j = meta[s].blk[b];
            const int inner = j == 0 ? a.Is : a.I;
            hrow0 = j == 0 ? P : rt.aoff[j - 1];
            mt = j == 0 ? T : rt.acnt[j - 1];
            const int r = lane & 15, tt = lane & 7;
            const uint32_t a_row = sa + (uint32_t)((b * g.ro + (r < ro ? r : 0)) * g.dp);
            const uint32_t b_row = hs_a + (uint32_t)((hrow0 + (tt < mt ? tt : 0)) * g.dp);
            const int kl = inner / wpb;
            mma_rows(d, a_row, b_row, kq * kl, kl / 16, lane);
        }
        release();
        *reinterpret_cast<float4*>(rbuf + (warp * 32 + lane) * 4) = make_float4(d[0], d[1], d[2], d[3]);
        consumers_sync();
        rb ^= 1;
        if (b < m.n && kq == 0) {
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            for (int q = 0; q < wpb; ++q) {
                const float4 q4 = *reinterpret_cast<const float4*>(rbuf + ((b * wpb + q) * 32 + lane) * 4);
                v[0] += q4.x; v[1] += q4.y; v[2] += q4.z; v[3] += q4.w;
            }
            const int rl = lane >> 2, i0 = 2 * (lane & 3);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int r = rl + (q >= 2 ? 8 : 0), i = i0 + (q & 1);
                if (r < ro && i < mt) Ys[(j == 0 ? P + i : rt.perm[hrow0 + i]) * 16 + r] = v[q];
            }
        }
    }
}

// Geometry for this layer: the most bytes in flight that fit the shared memory of one CTA.
static bool pick_geom(const LayerArgs& a, int cap, DGeom* g) {
    static const int cfg[][2] = {{8, 3}, {4, 6}, {4, 5}, {4, 4}, {4, 3}, {8, 2}, {4, 2}};
    for (const auto& c : cfg)
        if (decode_geom(a, a.num_sms, c[0], c[1], g) && g->smem <= cap) return true;
    return false;
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
        const int c = optin - (int)fa.sharedSizeBytes - 1024;
        if (c <= 0 ||
            cudaFuncSetAttribute(k_decode_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, c) != cudaSuccess)
            return 0;
        cap[dev] = c;
    }
    return cap[dev];
}

bool decode_fused_supported(const LayerArgs& a) {
    if (!(a.T >= 1 && a.T <= kDTT && a.K <= 8 && a.H <= kDMaxH && a.H % 128 == 0 && a.Imax <= kDMaxI &&
          a.I % 64 == 0 && a.Is % 64 == 0 && a.E <= 256 && a.num_sms >= 1 && a.dlog && a.dh))
        return false;
    DGeom g;
    return pick_geom(a, dynamic_smem_cap(), &g);
}

cudaError_t launch_decode_fused(const LayerArgs& a, cudaStream_t s) {
    DGeom g;
    if (!pick_geom(a, dynamic_smem_cap(), &g)) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.num_sms);
    cfg.blockDim = dim3(kDThreads);
    cfg.dynamicSmemBytes = (size_t)g.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    MOE_LAUNCH(MOE_KERNEL_DECODE_FUSED, s, (e = cudaLaunchKernelEx(&cfg, k_decode_fused, a, g)));
    return e;
}

}  // namespace moe
