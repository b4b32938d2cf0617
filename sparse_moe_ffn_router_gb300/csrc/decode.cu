// decode.cu -- the whole MoE layer for a few tokens (T <= 8) in one persistent kernel.
//
// At decode the layer reads ~58 MB of weights per token ("Qwen3.6-35B-A3B -- Architecture
// Overview", MoE FFN: 256 Experts: router 2048 -> 256, 8 SwiGLU experts of 3 x 512 x 2048, the
// shared expert), and every step depends on the one before: scores -> top-K -> gate_up -> down
// -> sum. Separate kernels would drain and refill the GPU at every step. Here one CTA per SM
// walks one global, ordered list of work items:
//
//   [24 router items] [shared gate_up] [shared down] [routed gate_up] [routed down]
//
// (item i belongs to CTA i mod gridDim), so the whole shared expert streams while the router
// runs. Each CTA has three roles:
//  * a producer warp streams each item's weight rows into a ring of shared-memory stages with
//    1-D TMA bulk copies (one per row, 16 bytes apart modulo 128 so ldmatrix is conflict-free),
//    and the item's activation rows when they are ready;
//  * 8 consumer warps multiply a stage with warp-level bf16 MMAs (m16n8k16, fp32 accumulate;
//    weight rows x up to 8 tokens, K split over the warps and summed in a fixed order), write the
//    results, and hand the finished item to the signaller through a shared-memory queue;
//  * a signaller warp does every cross-CTA step off the compute path: gpu-scope release counts,
//    tickets, the routing (top-K, dispatch, work records, then a release flag) when it holds the
//    last router ticket, and the fixed-order combine of an output block (residual, shared,
//    slot 0..K-1) when it holds that block's last ticket.
// Dependencies point only to lower-numbered items, every wait is bounded (~1 s, then
// MOE_ERR_TIMEOUT), and the launch is cooperative (all CTAs resident). Routed gate_up items wait
// for the routing flag; a down item streams its weights at once and copies its h rows only when
// its expert's gate_up count is complete (acquire, then an async-proxy fence). The last CTA to
// finish re-arms the counters for the next call on the same workspace.
#include "launch.h"
#include "ring.cuh"

namespace moe {

constexpr int kDTT = 8;                         // max tokens
constexpr int kDMaxH = 2048, kDMaxI = 512;
constexpr int kDPitchH = 2 * kDMaxH + 16;
constexpr int kDStage = 16 * kDPitchH;          // largest stage: 16 rows of H
constexpr int kRouteItems = 24;
constexpr int kDnRows = 32;                     // down rows per item = combine block
constexpr int kDMaxSt = 3;
static_assert(kDnRows * (2 * kDMaxI + 16) + kDTT * (2 * kDMaxI + 16) <= kDStage, "down stage must fit");

enum { kItemRoute = 0, kItemUp = 1, kItemDown = 2, kItemEnd = 3 };
constexpr int kDThreads = kConsumers + 64;  // 8 consumer warps, the producer, the signaller
constexpr int kProducerWarp = kWarps, kSignalWarp = kWarps + 1;
constexpr int kQ = 4;                       // signaller queue entries

struct Event {
    int type, grp, blk, need;
};

struct DMeta {
    int type;
    int mt;        // tokens (up, down); rows (route)
    int row0;      // up: first h row; route: first router row
    int f0;        // up: first feature; down: first output row
    int inner;     // down: row length of Wd (I or Is)
    int grp;       // up: counter slot (expert id, E = shared)
    int block;     // down: output block
    int nact;      // down: experts with rows (a block is complete after nact + 1 items)
    uint32_t toks; // up: token of each of its mt rows, 4 bits each
    int tok[kDTT], slot[kDTT];
    float sc[kDTT];
};

struct DSmem {
    uint8_t* xs;
    uint8_t* st[kDMaxSt];
    float* red;
    DMeta* meta;
    Event* ev;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* xbar;
    uint64_t* evfull;
    uint64_t* evempty;
};

__host__ __device__ inline size_t decode_smem_bytes(int T, int nst) {
    return 1024 + (size_t)((T * kDPitchH + 127) & ~127) + (size_t)nst * kDStage + (size_t)nst * kWarps * 128 * 4 +
           (size_t)nst * sizeof(DMeta) + kQ * sizeof(Event) + (2 * nst + 1 + 2 * kQ) * 8 + 64;
}

__device__ __forceinline__ DSmem decode_carve(uint8_t* raw, int T, int nst) {
    const uint32_t base = smem_u32(raw);
    uint8_t* p = raw + (((base + 127u) & ~127u) - base);
    DSmem r;
    r.xs = p;
    p += (size_t)((T * kDPitchH + 127) & ~127);
    for (int s = 0; s < kDMaxSt; ++s) {
        r.st[s] = p;
        if (s < nst) p += kDStage;
    }
    r.red = reinterpret_cast<float*>(p);
    p += (size_t)nst * kWarps * 128 * 4;
    r.meta = reinterpret_cast<DMeta*>(p);
    p += (size_t)nst * sizeof(DMeta);
    r.ev = reinterpret_cast<Event*>(p);
    p += kQ * sizeof(Event);
    p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 7) & ~(uintptr_t)7);
    r.full = reinterpret_cast<uint64_t*>(p);
    r.empty = r.full + nst;
    r.xbar = r.empty + nst;
    r.evfull = r.xbar + 1;
    r.evempty = r.evfull + kQ;
    return r;
}

// Counters of the fused kernel (in the workspace): routing flag and ticket in the header,
// per-expert gate_up completion [E+1], per-block combine tickets [H/kDnRows], final ticket.
struct DFlags {
    uint32_t* route_flag;
    uint32_t* route_ticket;
    uint32_t* epoch;
    uint32_t* final_ticket;
    uint32_t* up_done;
    uint32_t* comb;
};

__device__ __forceinline__ DFlags decode_flags(const LayerArgs& a) {
    DFlags f;
    f.route_flag = &a.hdr->dec_flag;
    f.route_ticket = &a.hdr->route_ticket;
    f.epoch = &a.hdr->dec_epoch;
    f.final_ticket = &a.hdr->dec_final;
    f.up_done = a.dflags;
    f.comb = a.dflags + (a.E + 1);
    return f;
}

// MMA of one stage: D[16 x 8] for 16 A rows at `a_rows` (rows past `nrows` read row 0) and the
// B rows given per lane (token row of lane % 8), K range [k0, k0 + 16 * ksteps).
__device__ __forceinline__ void stage_mma(float (&d)[4], uint32_t a_rows, int nrows, uint32_t b_row, int pitch, int k0,
                                          int ksteps, int lane) {
    int ra = lane & 15;
    ra = ra < nrows ? ra : 0;
    const uint32_t a = a_rows + (uint32_t)(ra * pitch + (k0 + 8 * (lane >> 4)) * 2);
    const uint32_t b = b_row + (uint32_t)((k0 + 8 * ((lane >> 3) & 1)) * 2);
#pragma unroll 4
    for (int k = 0; k < ksteps; ++k) {
        uint32_t a0, a1, a2, a3, b0, b1;
        ldsm_x4(a + k * 32, a0, a1, a2, a3);
        ldsm_x2(b + k * 32, b0, b1);
        mma16816(d, a0, a1, a2, a3, b0, b1);
    }
}

// ---------------------------------------------------------------------------------------
// Routing in one warp (the signaller of the CTA that finished the last router item): top-K of
// every token from the scores in L2, renormalised weights, shared gate, dispatch, work records.

struct RouteScratch {
    int cnt[256];
    int off[257];
    int sids[kDTT * 8];
    int slr[kDTT * 8];
    int sperm[kDTT * 8];
    int sact[256];
};

__device__ void signal_route(const LayerArgs& a, RouteScratch& rs, int lane) {
    for (int t = 0; t < a.T; ++t) {
        const float* l = a.logits + (size_t)t * a.ldl;
        float v[8];
        bool bad = false;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane + 32 * j;
            v[j] = -INFINITY;
            if (e < a.E) {
                v[j] = __ldcg(l + e);
                if (!isfinite(v[j])) {
                    bad = true;
                    v[j] = -INFINITY;
                }
            }
        }
        uint32_t taken = 0;
        float sel_v[8];
        int sel_e[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k < a.K) {
                float bv = -INFINITY;
                int be = 0x7fffffff;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int e = lane + 32 * j;
                    if (e < a.E && !((taken >> j) & 1u) && (v[j] > bv || (v[j] == bv && e < be))) {
                        bv = v[j];
                        be = e;
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                    if (ov > bv || (ov == bv && oe < be)) {
                        bv = ov;
                        be = oe;
                    }
                }
                if ((be & 31) == lane) taken |= 1u << (be >> 5);
                sel_v[k] = bv;
                sel_e[k] = be;
            }
        }
        if (lane == 0) {
            float ex[8], s = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (k < a.K) {
                    ex[k] = expf(sel_v[k] - sel_v[0]);
                    s += ex[k];
                }
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (k < a.K) {
                    rs.sids[t * a.K + k] = sel_e[k];
                    a.ids[(size_t)t * a.K + k] = sel_e[k];
                    a.topw[(size_t)t * a.K + k] = ex[k] / s;
                }
            const float z = __ldcg(l + a.E);
            if (!isfinite(z)) bad = true;
            a.sgate[t] = 1.0f / (1.0f + expf(-z));
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&a.hdr->err, ERR_NONFINITE_SCORE);
    }
    for (int e = lane; e < a.E; e += 32) rs.cnt[e] = 0;
    __syncwarp();
    const int P = (int)a.P;
    for (int b0 = 0; b0 < P; b0 += 32) {
        const int i = b0 + lane;
        const bool valid = i < P;
        const int e = valid ? rs.sids[i] : -1;
        const unsigned m = __match_any_sync(0xffffffffu, e);
        const int rank_in = __popc(m & ((1u << lane) - 1u));
        const int cc = valid ? rs.cnt[e] : 0;
        __syncwarp();
        if (valid) {
            rs.slr[i] = cc + rank_in;
            if (rank_in == 0) rs.cnt[e] = cc + __popc(m);
        }
        __syncwarp();
    }
    int loc[8], run = 0, nz = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e = lane * 8 + j;
        loc[j] = e < a.E ? rs.cnt[e] : 0;
        run += loc[j];
        nz += loc[j] > 0;
    }
    int incl = run, inz = nz;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        const int z = __shfl_up_sync(0xffffffffu, inz, o);
        if (lane >= o) {
            incl += y;
            inz += z;
        }
    }
    int pos = incl - run, apos = inz - nz;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e = lane * 8 + j;
        if (e < a.E) {
            rs.off[e] = pos;
            if (loc[j] > 0) {
                rs.sact[apos] = e;
                a.act[apos++] = e;
            }
        }
        pos += loc[j];
    }
    const int n_act = __shfl_sync(0xffffffffu, inz, 31);
    if (lane == 31) rs.off[a.E] = incl;
    __syncwarp();
    for (int e = lane; e <= a.E; e += 32) {
        a.offsets[e] = rs.off[e];
        if (e < a.E) a.counts[e] = rs.cnt[e];
    }
    for (int i = lane; i < P; i += 32) {
        const int j = rs.off[rs.sids[i]] + rs.slr[i];
        a.perm[j] = i;
        a.inv[i] = j;
        rs.sperm[j] = i;
    }
    __syncwarp();
    const int fbs = a.I / 8;
    for (int idx = lane; idx < n_act * fbs; idx += 32) {
        const int g = idx / fbs, fb = idx - g * fbs;
        const int e = rs.sact[g];
        uint32_t toks = 0;
        for (int j = 0; j < rs.cnt[e]; ++j) toks |= (uint32_t)(rs.sperm[rs.off[e] + j] / a.K) << (4 * j);
        UpRec rec;
        rec.e = e;
        rec.row0 = rs.off[e];
        rec.f0 = (int16_t)(fb * 8);
        rec.mt = (int16_t)rs.cnt[e];
        rec.toks = toks;
        a.uprec[idx] = rec;
    }
    if (lane == 0) {
        a.hdr->n_act = n_act;
        a.hdr->n_uprec = n_act * fbs;
    }
    __syncwarp();
}

// Fixed-order sum of one output block of 32 rows for every token, by one warp. The shared
// expert's slot holds its unscaled output; its gate is applied (and stored back) here.
__device__ void signal_combine_block(const LayerArgs& a, int blk, int lane) {
    for (int idx = lane; idx < a.T * kDnRows; idx += 32) {
        const int t = idx / kDnRows, o = blk * kDnRows + (idx - t * kDnRows);
        float* yt = a.Y + (size_t)t * (a.K + 1) * a.H + o;
        float acc = a.residual ? __bfloat162float(a.residual[(size_t)t * a.H + o]) : 0.f;
        const float shared = a.sgate[t] * __ldcg(yt + (size_t)a.K * a.H);
        yt[(size_t)a.K * a.H] = shared;
        acc += shared;
        for (int k = 0; k < a.K; ++k) acc += __ldcg(yt + (size_t)k * a.H);
        a.out[(size_t)t * a.H + o] = __float2bfloat16_rn(acc);
    }
}

// ---------------------------------------------------------------------------------------

__global__ void __launch_bounds__(kDThreads, 1) k_decode_fused(LayerArgs a, int nst) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ RouteScratch rs;
    DSmem r = decode_carve(smem_raw, a.T, nst);
    const DFlags fl = decode_flags(a);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t* err = &a.hdr->err;
    const int pitch = 2 * a.H + 16;
    const uint32_t epoch = *(volatile uint32_t*)fl.epoch;
    const int R = (a.E + 1 + kRouteItems - 1) / kRouteItems;  // router rows per item
    const int n_sup = a.Is / 8;          // shared gate_up items (8 features each)
    const int n_blocks = a.H / kDnRows;  // shared down items (one per output block)
    const int base_u = kRouteItems + n_sup + n_blocks;
    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&r.full[s], 1);
            mbar_init(&r.empty[s], kWarps);
        }
        mbar_init(r.xbar, 1);
        for (int q = 0; q < kQ; ++q) {
            mbar_init(&r.evfull[q], 1);
            mbar_init(&r.evempty[q], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kProducerWarp) {
        // ================= producer
        if (lane == 0) mbar_arrive_expect_tx(r.xbar, (uint32_t)(a.T * a.H * 2));
        __syncwarp();
        if (lane < a.T) bulk_load(r.xs + (size_t)lane * pitch, a.x + (size_t)lane * a.H, a.H * 2, r.xbar);
        int it = 0, n_items = -1, n_u = 0, n_act = 0;
        bool fail = false;
        for (int i = blockIdx.x;; i += gridDim.x) {
            if (i >= base_u && n_items < 0) {
                bool ok = lane == 0 ? wait_at_least(fl.route_flag, epoch + 1) : true;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                __syncwarp();  // orders the other lanes' reads after lane 0's acquire
                if (!ok) {
                    fail = true;
                    break;
                }
                n_u = *(volatile int*)&a.hdr->n_uprec;
                n_act = *(volatile int*)&a.hdr->n_act;
                n_items = base_u + n_u + n_act * n_blocks;
            }
            if (n_items >= 0 && i >= n_items) break;
            const int s = it % nst;
            bool ok = lane == 0 ? mbar_wait(&r.empty[s], (((uint32_t)(it / nst)) & 1u) ^ 1u) : true;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                fail = true;
                break;
            }
            DMeta& m = r.meta[s];
            uint8_t* st = r.st[s];
            const bool up = (i >= kRouteItems && i < kRouteItems + n_sup) || (i >= base_u && i < base_u + n_u);
            if (i < kRouteItems) {
                const int r0 = i * R, nr = max(0, min(a.E + 1, r0 + R) - r0);
                if (lane == 0) {
                    m.type = kItemRoute;
                    m.mt = nr;
                    m.row0 = r0;
                    mbar_arrive_expect_tx(&r.full[s], (uint32_t)(nr * a.H * 2));
                }
                __syncwarp();
                if (lane < nr) {
                    const int row = r0 + lane;
                    bulk_load(st + (size_t)lane * pitch, row < a.E ? a.router_w + (size_t)row * a.H : a.sg, a.H * 2,
                              &r.full[s]);
                }
            } else if (up) {
                const bf16* W;
                int inner, row0, f0, mt, grp;
                uint32_t toks;
                if (i < kRouteItems + n_sup) {
                    W = a.sgu;
                    inner = a.Is;
                    row0 = (int)a.P;
                    f0 = (i - kRouteItems) * 8;
                    mt = a.T;
                    toks = 0x76543210u;
                    grp = a.E;
                } else {
                    const UpRec rec = a.uprec[i - base_u];
                    W = a.gate_up + (size_t)rec.e * 2 * a.I * a.H;
                    inner = a.I;
                    row0 = rec.row0;
                    f0 = rec.f0;
                    mt = rec.mt;
                    toks = rec.toks;
                    grp = rec.e;
                }
                if (lane == 0) {
                    m.type = kItemUp;
                    m.mt = mt;
                    m.row0 = row0;
                    m.f0 = f0;
                    m.grp = grp;
                    m.toks = toks;
                    mbar_arrive_expect_tx(&r.full[s], (uint32_t)(16 * a.H * 2));
                }
                __syncwarp();
                if (lane < 8)
                    bulk_load(st + (size_t)lane * pitch, W + (size_t)(f0 + lane) * a.H, a.H * 2, &r.full[s]);
                else if (lane < 16)
                    bulk_load(st + (size_t)lane * pitch, W + (size_t)(inner + f0 + lane - 8) * a.H, a.H * 2, &r.full[s]);
            } else {
                // down item: the shared expert's blocks first (no routing needed), then routed
                const bool shared = i < base_u;
                int blk, e;
                if (shared) {
                    blk = i - kRouteItems - n_sup;
                    e = a.E;
                } else {
                    const int d = i - base_u - n_u;
                    blk = d / n_act;
                    e = a.act[d - blk * n_act];
                }
                const int inner = shared ? a.Is : a.I;
                const bf16* W = shared ? a.sd : a.down + (size_t)e * a.H * a.I;
                const int hrow0 = shared ? (int)a.P : a.offsets[e];
                const int mt = shared ? a.T : a.offsets[e + 1] - hrow0;
                const int dp = 2 * inner + 16;
                if (lane < mt) {
                    if (shared) {
                        m.tok[lane] = lane;
                        m.slot[lane] = a.K;
                        m.sc[lane] = 1.f;  // the gate is applied in the combine
                    } else {
                        const int pv = a.perm[hrow0 + lane];
                        m.tok[lane] = pv / a.K;
                        m.slot[lane] = pv - (pv / a.K) * a.K;
                        m.sc[lane] = a.topw[pv];
                    }
                }
                if (lane == 0) {
                    m.type = kItemDown;
                    m.mt = mt;
                    m.f0 = blk * kDnRows;
                    m.inner = inner;
                    m.block = blk;
                    m.nact = -1;  // filled by the signaller from the routing
                    mbar_arrive_expect_tx(&r.full[s], (uint32_t)((kDnRows + mt) * inner * 2));
                }
                __syncwarp();
                bulk_load(st + (size_t)lane * dp, W + (size_t)(blk * kDnRows + lane) * inner, inner * 2, &r.full[s]);
                // h rows only once this expert's gate_up items are all done
                bool hok = lane == 0 ? wait_at_least(&fl.up_done[e], (uint32_t)(inner / 8)) : true;
                hok = __shfl_sync(0xffffffffu, hok, 0);
                __syncwarp();
                if (!hok) {
                    fail = true;
                    break;
                }
                fence_proxy_async_global();
                if (lane < mt)
                    bulk_load(st + (size_t)(kDnRows + lane) * dp, a.h + (size_t)(hrow0 + lane) * a.Imax, inner * 2,
                              &r.full[s]);
            }
            ++it;
        }
        if (fail && lane == 0) atomicOr(err, ERR_TIMEOUT);
        if (lane == 0) {
            // every copy issued must land before the CTA releases its shared memory (checked
            // before the end marker below reuses a stage slot)
            for (int k = 0; k < nst && it - 1 - k >= 0; ++k) {
                const int j = it - 1 - k;
                if (!mbar_wait(&r.full[j % nst], ((uint32_t)(j / nst)) & 1u)) atomicOr(err, ERR_TIMEOUT);
            }
            if (!mbar_wait(r.xbar, 0)) atomicOr(err, ERR_TIMEOUT);
            const int s = it % nst;
            if (mbar_wait(&r.empty[s], (((uint32_t)(it / nst)) & 1u) ^ 1u)) {
                r.meta[s].type = kItemEnd;
                mbar_arrive(&r.full[s]);
            } else {
                atomicOr(err, ERR_TIMEOUT);
            }
        }
        return;
    }

    if (warp == kSignalWarp) {
        // ================= signaller: cross-CTA counts, tickets, routing and combines
        bool live = true, routed = false;
        int n_act_sig = 0;
        for (int q_it = 0; live; ++q_it) {
            const int q = q_it % kQ;
            bool ok = lane == 0 ? mbar_wait(&r.evfull[q], ((uint32_t)(q_it / kQ)) & 1u) : true;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            if (!ok) {
                if (lane == 0) atomicOr(err, ERR_TIMEOUT);
                break;
            }
            const Event ev = r.ev[q];
            __syncwarp();
            if (lane == 0) mbar_arrive(&r.evempty[q]);
            if (ev.type == kItemRoute) {
                uint32_t old = 0;
                if (lane == 0) old = atom_acq_rel_add(fl.route_ticket, 1u);
                old = __shfl_sync(0xffffffffu, old, 0);
                __syncwarp();
                if (old == kRouteItems - 1) {
                    signal_route(a, rs, lane);
                    if (lane == 0) st_release(fl.route_flag, epoch + 1);
                }
            } else if (ev.type == kItemUp) {
                if (lane == 0) red_release_add(&fl.up_done[ev.grp], 1u);
            } else if (ev.type == kItemDown) {
                // a block is complete after the shared item and one item per routed expert; the
                // expert count comes from the routing (a shared item can finish before it)
                if (!routed) {
                    bool ok2 = lane == 0 ? wait_at_least(fl.route_flag, epoch + 1) : true;
                    ok2 = __shfl_sync(0xffffffffu, ok2, 0);
                    __syncwarp();
                    if (!ok2) {
                        if (lane == 0) atomicOr(err, ERR_TIMEOUT);
                        break;
                    }
                    n_act_sig = *(volatile int*)&a.hdr->n_act;
                    routed = true;
                }
                uint32_t old = 0;
                if (lane == 0) {
                    old = atom_release_add(&fl.comb[ev.blk], 1u);
                    if (old == (uint32_t)n_act_sig) __threadfence();
                }
                old = __shfl_sync(0xffffffffu, old, 0);
                __syncwarp();
                if (old == (uint32_t)n_act_sig) signal_combine_block(a, ev.blk, lane);
            } else {
                live = false;
            }
        }
        // the last CTA to finish re-arms the counters for the next call on this workspace
        uint32_t fin = 0;
        if (lane == 0) fin = atom_acq_rel_add(fl.final_ticket, 1u);
        fin = __shfl_sync(0xffffffffu, fin, 0);
        if (fin == gridDim.x - 1) {
            for (int e = lane; e <= a.E; e += 32) fl.up_done[e] = 0;
            for (int b = lane; b < n_blocks; b += 32) fl.comb[b] = 0;
            __syncwarp();
            if (lane == 0) {
                *fl.route_ticket = 0;
                *fl.final_ticket = 0;
                *fl.epoch = epoch + 1;
            }
        }
        return;
    }

    // ================= consumers
    bool xok = lane == 0 ? mbar_wait(r.xbar, 0) : true;
    xok = __shfl_sync(0xffffffffu, xok, 0);
    xok = consumers_all(xok);
    int q_it = 0;
    // hand a finished item to the signaller (warp 0, lane 0; after the item's writes)
    auto push = [&](int type, int grp, int blk) {
        if (threadIdx.x == 0) {
            const int q = q_it % kQ;
            if (!mbar_wait(&r.evempty[q], (((uint32_t)(q_it / kQ)) & 1u) ^ 1u)) atomicOr(err, ERR_TIMEOUT);
            r.ev[q] = Event{type, grp, blk, 0};
            mbar_arrive(&r.evfull[q]);
        }
        ++q_it;
    };
    for (int it = 0;; ++it) {
        const int s = it % nst;
        bool ok = xok && (lane == 0 ? mbar_wait(&r.full[s], ((uint32_t)(it / nst)) & 1u) : true);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!consumers_all(ok)) {
            if (threadIdx.x == 0) atomicOr(err, ERR_TIMEOUT);
            push(kItemEnd, 0, 0);
            break;
        }
        const DMeta& m = r.meta[s];
        const int type = m.type, mt = m.mt;
        if (type == kItemEnd) {
            push(kItemEnd, 0, 0);
            break;
        }
        const uint32_t sa = smem_u32(r.st[s]);
        float* red = r.red + (size_t)s * kWarps * 128;
        if (type == kItemRoute) {
            const int row0 = m.row0;
            const int tt = lane & 7;
            const uint32_t b_row = smem_u32(r.xs) + (uint32_t)((tt < a.T ? tt : 0) * pitch);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            stage_mma(d, sa, mt, b_row, pitch, warp * (a.H / kWarps), a.H / kWarps / 16, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&r.empty[s]);
            *reinterpret_cast<float4*>(red + (warp * 32 + lane) * 4) = make_float4(d[0], d[1], d[2], d[3]);
            consumers_sync();
            if (warp == 0) {
                float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float4 q4 = *reinterpret_cast<const float4*>(red + (w * 32 + lane) * 4);
                    v[0] += q4.x; v[1] += q4.y; v[2] += q4.z; v[3] += q4.w;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int rl = (lane >> 2) + (q >= 2 ? 8 : 0), t = 2 * (lane & 3) + (q & 1);
                    if (rl < mt && t < a.T) {
                        const int row = row0 + rl;
                        const float bias = (row < a.E && a.router_b) ? __bfloat162float(a.router_b[row]) : 0.f;
                        a.logits[(size_t)t * a.ldl + row] = v[q] + bias;
                    }
                }
                __syncwarp();
            }
            push(kItemRoute, 0, 0);
        } else if (type == kItemUp) {
            const int row0 = m.row0, f0 = m.f0, grp = m.grp;
            const uint32_t toks = m.toks;
            const int tt = lane & 7;
            const int tok = tt < mt ? (int)((toks >> (4 * tt)) & 15u) : 0;
            const uint32_t b_row = smem_u32(r.xs) + (uint32_t)(tok * pitch);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            stage_mma(d, sa, 16, b_row, pitch, warp * (a.H / kWarps), a.H / kWarps / 16, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&r.empty[s]);
            *reinterpret_cast<float4*>(red + (warp * 32 + lane) * 4) = make_float4(d[0], d[1], d[2], d[3]);
            consumers_sync();
            if (warp == 0) {
                float g0 = 0.f, g1 = 0.f, u0 = 0.f, u1 = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float4 q4 = *reinterpret_cast<const float4*>(red + (w * 32 + lane) * 4);
                    g0 += q4.x; g1 += q4.y; u0 += q4.z; u1 += q4.w;
                }
                const int f = lane >> 2, t = 2 * (lane & 3);
                if (t < mt) a.h[(size_t)(row0 + t) * a.Imax + f0 + f] = __float2bfloat16_rn(silu(g0) * u0);
                if (t + 1 < mt) a.h[(size_t)(row0 + t + 1) * a.Imax + f0 + f] = __float2bfloat16_rn(silu(g1) * u1);
                __syncwarp();
            }
            push(kItemUp, grp, 0);
        } else {
            const int inner = m.inner, f0 = m.f0, blk = m.block;
            const int dp = 2 * inner + 16;
            const int mtile = warp & 1, kq = warp >> 1;  // 2 row tiles x 4 K quarters
            const int kqlen = inner / 4;
            const int tt = lane & 7;
            const uint32_t b_row = sa + (uint32_t)((kDnRows + (tt < mt ? tt : 0)) * dp);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            stage_mma(d, sa + (uint32_t)(mtile * 16 * dp), 16, b_row, dp, kq * kqlen, kqlen / 16, lane);
            const int t0 = 2 * (lane & 3);
            size_t y0 = 0, y1 = 0;
            float s0 = 0.f, s1 = 0.f;
            if (t0 < mt) {
                y0 = ((size_t)m.tok[t0] * (a.K + 1) + m.slot[t0]) * a.H + f0;
                s0 = m.sc[t0];
            }
            if (t0 + 1 < mt) {
                y1 = ((size_t)m.tok[t0 + 1] * (a.K + 1) + m.slot[t0 + 1]) * a.H + f0;
                s1 = m.sc[t0 + 1];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&r.empty[s]);
            *reinterpret_cast<float4*>(red + (warp * 32 + lane) * 4) = make_float4(d[0], d[1], d[2], d[3]);
            consumers_sync();
            if (kq == 0) {
                float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 w4 = *reinterpret_cast<const float4*>(red + ((q * 2 + mtile) * 32 + lane) * 4);
                    v[0] += w4.x; v[1] += w4.y; v[2] += w4.z; v[3] += w4.w;
                }
                const int row = mtile * 16 + (lane >> 2);
                if (t0 < mt) {
                    a.Y[y0 + row] = s0 * v[0];
                    a.Y[y0 + row + 8] = s0 * v[2];
                }
                if (t0 + 1 < mt) {
                    a.Y[y1 + row] = s1 * v[1];
                    a.Y[y1 + row + 8] = s1 * v[3];
                }
            }
            consumers_sync();  // warp 1's rows are written before warp 0 hands the item over
            push(kItemDown, 0, blk);
        }
    }
}

bool decode_fused_supported(const LayerArgs& a) {
    return a.T >= 1 && a.T <= kDTT && a.uprec && a.dflags && a.H <= kDMaxH && a.H % 128 == 0 &&
           a.Imax <= kDMaxI && a.I % 32 == 0 && a.Is % 32 == 0 && a.E <= 256 &&
           (a.E + 1 + kRouteItems - 1) / kRouteItems <= 16;
}

cudaError_t launch_decode_fused(const LayerArgs& a, cudaStream_t s) {
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    const int cap = 220 * 1024;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_decode_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, cap);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int nst = decode_smem_bytes(a.T, 3) <= (size_t)cap ? 3 : 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.num_sms);
    cfg.blockDim = dim3(kDThreads);
    cfg.dynamicSmemBytes = decode_smem_bytes(a.T, nst);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    MOE_LAUNCH(MOE_KERNEL_GATE_UP, s, (e = cudaLaunchKernelEx(&cfg, k_decode_fused, a, nst)));
    return e;
}

}  // namespace moe
