// stream.cu -- the few-token (decode) regime of the experts: weight streaming.
//
// With few tokens every expert the router picked has only a handful of rows, so the layer is
// bound by reading the touched experts' weights from HBM once (4 MiB gate_up + 2 MiB down per
// expert at the full shape, "Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256 Experts).
//
// Both kernels are persistent (one CTA per SM). A producer warp walks the CTA's work items and,
// for each, fills one stage of a 3-stage shared-memory ring with the item's weight rows only,
// by 1-D TMA bulk copies (cp.async.bulk; gate/up one per 4 KB row, down one per group of 4
// consecutive 1 KB rows, with 16 bytes of padding per row or group so ldmatrix is free of bank
// conflicts), and writes the item's metadata into the stage before arming its mbarrier. The
// ring is sized for bytes in flight: at the full-GPU HBM rate a loaded SM needs close to
// 200 KB of copies outstanding, so the activation rows (x for gate_up, h for down) are kept
// out of it. Eight consumer warps multiply the staged rows with warp-level bf16 MMAs
// (m16n8k16, fp32 accumulate: 16 weight rows by the item's tokens, padded to 8), each warp over
// a fixed K range whose token-row fragments it holds in registers, loaded from L2 when the
// item's token set changes; the warps' partial results are summed in a fixed order. A stage
// is 16 (gate/up) or 64 (down) weight rows, too few rows for the 64/128-row tcgen05 MMA without
// four times larger stages; the tensor-core work is small either way, the kernels are bound by
// HBM.
//
// k_stream_up:   h = bf16(SiLU(x . Wg^T) * (x . Wu^T)); a stage holds 8 gate rows and the 8
//                matching up rows of one group, so the 16 x 8 MMA tile gives g and u of the same
//                features in the same lane. Shared-expert items come first: they need no
//                routing and run while the routing kernel finishes (programmatic dependent
//                launch); routed items start after griddepcontrol.wait.
// k_stream_down: Y[t, slot] = scale * (h . Wd^T); a stage holds 64 output rows of Wd of one
//                group. The fixed-order combine runs next as its own kernel (launched as a
//                programmatic dependent, so its launch overlaps this kernel's tail).
#include "launch.h"
#include "ring.cuh"
#include "sm100.cuh"

namespace moe {

constexpr int kSt = 3;                  // ring stages
constexpr int kTT = 8;                  // tokens per item (the MMA's N)
constexpr int kFps = 8;                 // up: features per stage (16 rows: 8 gate + 8 up)
constexpr int kRows = 64;               // down: output rows per stage (= combine block)
constexpr int kPad = 16;                // row padding: rows start 16 B apart modulo 128 B
constexpr int kMaxH = 2048, kMaxInner = 512;
constexpr int kPitchH = 2 * kMaxH + kPad;
constexpr int kMaxSteps = 16;           // MMA k-steps of one consumer warp per stage, at most
// A stage holds weight rows only: 16 gate/up rows of up to 2048 elements, or 16 groups of 4
// down rows of up to 512 -- the same 65,792 bytes.
constexpr int kStageBytes = 2 * kFps * kPitchH;
static_assert((kRows / 4) * (8 * kMaxInner + kPad) <= kStageBytes, "down stage must fit");
static_assert(kMaxH / kWarps / 16 <= kMaxSteps && kMaxInner / 2 / 16 <= kMaxSteps, "k-steps per warp");

// Down stage layout: kRows/4 groups of 4 consecutive Wd rows, each group one 1-D bulk copy
// (4 KB at inner = 512: copies of 1 KB rows stream markedly slower than 4 KB ones), groups
// 8*inner + 16 bytes apart so any 8 consecutive groups start in 8 different 16-byte bank
// slots. An MMA tile of 16 rows takes rows j and j+1 of 8 consecutive groups, so each 8x8
// ldmatrix fetch reads 8 different bank slots.
__host__ __device__ constexpr int dn_gpitch(int inner) { return 8 * inner + kPad; }

struct StageMeta {
    int mt;          // tokens in this item
    int row0;        // h row of the item's token 0 (up: written, down: read)
    int f0;          // up: first feature / down: first output row
    int inner;       // down: length of a weight row (I or Is)
    int key;         // the item's token set: consecutive items with one key use the same rows
    int tok[kTT], slot[kTT];
    float sc[kTT];
};

struct Ring {
    uint8_t* st0;    // stage s at st0 + s * kStageBytes
    StageMeta* meta;
    float* red;      // [kSt][kWarps][32][4] per-warp partial accumulators
    uint64_t* full;
    uint64_t* empty;
    int* misc;       // [0] abort, [1] combine verdict, [4..] group prefix table (producer)
};

constexpr int kMiscInts = 4 + 2 * 257;
constexpr int kRedBytes = kSt * kWarps * 32 * 4 * 4;
constexpr int kStreamSmemBytes =
    1024 + kSt * kStageBytes + kRedBytes + kSt * (int)sizeof(StageMeta) + 2 * kSt * 8 + kMiscInts * 4 + 64;

__device__ __forceinline__ Ring carve(uint8_t* raw) {
    const uint32_t base = smem_u32(raw);
    uint8_t* p = raw + (((base + 127u) & ~127u) - base);
    Ring r;
    r.st0 = p;
    p += kSt * kStageBytes;
    r.red = reinterpret_cast<float*>(p);
    p += kRedBytes;
    r.meta = reinterpret_cast<StageMeta*>(p);
    p += kSt * sizeof(StageMeta);
    p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 7) & ~(uintptr_t)7);
    r.full = reinterpret_cast<uint64_t*>(p);
    r.empty = r.full + kSt;
    r.misc = reinterpret_cast<int*>(r.empty + kSt);
    return r;
}

// ---------------------------------------------------------------------------------------

__device__ __forceinline__ void ring_init(Ring& r) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSt; ++s) {
            mbar_init(&r.full[s], 1);
            mbar_init(&r.empty[s], kWarps);
        }
        r.misc[0] = 0;
        fence_mbar_init();
    }
    __syncthreads();
}

// Producer warp: wait for stage `it` to be free; lane 0 polls, the warp follows its verdict.
__device__ __forceinline__ bool acquire_stage(Ring& r, int it, uint32_t* err, uint64_t limit) {
    const int lane = threadIdx.x & 31;
    bool ok = lane == 0 ? mbar_wait(&r.empty[it % kSt], (((uint32_t)(it / kSt)) & 1u) ^ 1u, limit) : true;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok && lane == 0) {
        atomicOr(err, ERR_TIMEOUT);
        *(volatile int*)&r.misc[0] = 1;
    }
    __syncwarp();
    return ok;
}

// Consumer warp: wait for stage `it`; lane 0 polls, the warp follows its verdict.
__device__ __forceinline__ bool wait_stage(Ring& r, int it, uint32_t* err, uint64_t limit) {
    const int lane = threadIdx.x & 31;
    bool ok = lane == 0 ? mbar_wait(&r.full[it % kSt], ((uint32_t)(it / kSt)) & 1u, limit) : true;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok && lane == 0) {
        atomicOr(err, ERR_TIMEOUT);
        *(volatile int*)&r.misc[0] = 1;
    }
    __syncwarp();
    return ok;
}

__device__ __forceinline__ void release_stage(Ring& r, int it) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&r.empty[it % kSt]);
}

// Producer drain: every copy issued must land before the CTA releases its shared memory.
__device__ __forceinline__ void drain(Ring& r, int issued, uint32_t* err, uint64_t limit) {
    for (int k = 0; k < kSt && issued - 1 - k >= 0; ++k) {
        const int j = issued - 1 - k;
        if (!mbar_wait(&r.full[j % kSt], ((uint32_t)(j / kSt)) & 1u, limit)) atomicOr(err, ERR_TIMEOUT);
    }
}

// Group prefix table built by the producer warp: tiles[g] = first item of routed group g
// (in items of `per_tile` per token tile), n_act + 1 entries.
__device__ void build_tiles(const LayerArgs& a, int* tiles, int per_tile) {
    const int lane = threadIdx.x & 31;
    const int n = a.hdr->n_act;
    int run = 0;
    for (int base = 0; base < n; base += 32) {
        const int g = base + lane;
        int v = 0;
        if (g < n) {
            const int e = a.act[g];
            v = ((a.offsets[e + 1] - a.offsets[e] + kTT - 1) / kTT) * per_tile;
        }
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (g < n) tiles[g] = run + incl - v;
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tiles[n] = run;
    __syncwarp();
}

// Routed token tiles over all groups (computed by each consumer warp).
__device__ __forceinline__ int routed_tiles(const LayerArgs& a, int lane) {
    int tot = 0;
    const int n = a.hdr->n_act;
    for (int g = lane; g < n; g += 32) {
        const int e = a.act[g];
        tot += (a.offsets[e + 1] - a.offsets[e] + kTT - 1) / kTT;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    return tot;
}

// Work of CTA c of G: shared-expert items [c*S/G, (c+1)*S/G) (they need no routing), then
// routed items [c*R/G, (c+1)*R/G) -- contiguous runs, so consecutive items mostly share their
// token tile (and expert): the producer looks the routing up, and the consumers load the token
// rows, once per change.
__device__ __forceinline__ int routed_split(int R, int c, int G) { return (int)((long long)c * R / G); }

// Largest g with tiles[g] <= i (tiles ascending, tiles[0] = 0).
__device__ __forceinline__ int find_group(const int* tiles, int n, int i) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tiles[mid] <= i) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Producer warp: copy `nrows` rows of `rowbytes` from src (rows `src_pitch` elements apart) to
// dst rows kPad-padded, lanes in parallel.
__device__ __forceinline__ void copy_rows(uint8_t* dst, int dst_pitch, const bf16* src, size_t src_pitch, int nrows,
                                          uint32_t rowbytes, uint64_t* bar, int lane) {
    for (int i = lane; i < nrows; i += 32) bulk_load(dst + (size_t)i * dst_pitch, src + (size_t)i * src_pitch, rowbytes, bar);
}

// ---------------------------------------------------------------------------------------
// Stage layout, up:   rows 0..7 gate features f0..f0+7, rows 8..15 the matching up rows
//                     (pitch 2H + 16).
//           down:     kRows/4 groups of 4 Wd rows (one copy each, see dn_gpitch).
// The activation rows (x for up, h for down) are not staged: each consumer warp holds its K
// range of the item's token rows as MMA operand fragments in registers and reloads them from
// L2 only when the token set changes (the items of one expert and token tile are consecutive),
// so the ring's shared memory carries weight bytes alone.

// B operand fragments of one consumer warp: token row `row` (lane l takes row l/4 of the tile)
// from element 0 over `ksteps` k-steps, in the m16n8k16 layout -- lane l holds elements
// 16s + 2(l%4) + {0, 1} and 16s + 8 + 2(l%4) + {0, 1} of k-step s. L2 loads (the rows were
// written by an earlier kernel).
__device__ __forceinline__ void load_bfrag(uint32_t (&b)[kMaxSteps][2], const bf16* row, int ksteps, int lane) {
    const unsigned int* p = reinterpret_cast<const unsigned int*>(row + 2 * (lane & 3));
#pragma unroll
    for (int k = 0; k < kMaxSteps; ++k)
        if (k < ksteps) {
            b[k][0] = __ldcg(p + 8 * k);
            b[k][1] = __ldcg(p + 8 * k + 4);
        }
}

__global__ void __launch_bounds__(kStreamThreads, 1) k_stream_up(LayerArgs a) {
    extern __shared__ uint8_t smem_raw[];
    Ring r = carve(smem_raw);
    ring_init(r);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t* err = &a.hdr->err;
    const int fb_s = a.Is / kFps, fb_r = a.I / kFps;          // feature blocks per group
    const int n_shared = fb_s * ((a.T + kTT - 1) / kTT);       // shared items first
    const int pitch = 2 * a.H + kPad;
    const int G = gridDim.x, c = blockIdx.x;
    // this CTA's shared items: a contiguous run in (token tile, feature block) order
    const int s0 = routed_split(n_shared, c, G), my_shared = routed_split(n_shared, c + 1, G) - s0;

    if (warp == kWarps) {
        // ---------------- producer
        int* tiles = r.misc + 4;
        int it = 0;
        // stage it: 8 gate rows f0.. and the matching up rows of W; lane < kTT holds the x row
        // of token lane of the item (a valid row for lanes past mt)
        auto issue = [&](const bf16* W, int inner, int f0, int hrow, int mt, int key, int tok) -> bool {
            if (__shfl_sync(0xffffffffu, *(volatile int*)&r.misc[0], 0)) return false;  // consumers gave up
            const int s = it % kSt;
            if (!acquire_stage(r, it, err, a.wait_ns)) return false;
            if (a.test_suppress == MOE_TEST_SUPPRESS_STAGE && blockIdx.x == 0 && it == 0) {
                // testing aid: CTA 0's first stage is never loaded, so its consumers' wait runs out
                ++it;
                return true;
            }
            StageMeta& m = r.meta[s];
            if (lane < kTT) m.tok[lane] = tok;
            if (lane == 0) {
                m.mt = mt;
                m.row0 = hrow;
                m.f0 = f0;
                m.key = key;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&r.full[s], (uint32_t)(2 * kFps * a.H * 2));
            __syncwarp();
            uint8_t* st = r.st0 + (size_t)s * kStageBytes;
            copy_rows(st, pitch, W + (size_t)f0 * a.H, a.H, kFps, a.H * 2, &r.full[s], lane);
            copy_rows(st + kFps * pitch, pitch, W + (size_t)(inner + f0) * a.H, a.H, kFps, a.H * 2, &r.full[s], lane);
            ++it;
            return true;
        };
        bool ok = true;
        for (int k = 0; k < my_shared && ok; ++k) {
            const int i = s0 + k, tile = i / fb_s, fb = i - tile * fb_s, t0 = tile * kTT;
            const int mt = min(kTT, a.T - t0);
            ok = issue(a.sgu, a.Is, fb * kFps, (int)a.P + t0, mt, -1 - t0, t0 + (lane < mt ? lane : 0));
        }
        grid_dep_wait();
        grid_dep_launch();  // the routing is complete: the down kernel may start (see below)
        const int n_act = a.hdr->n_act;
        build_tiles(a, tiles, fb_r);
        const int q1 = routed_split(tiles[n_act], c + 1, G);
        int g = -1, e = 0, off = 0, cnt = 0, ctile = -1, mt = 0, tok = 0;
        for (int q = routed_split(tiles[n_act], c, G); q < q1 && ok; ++q) {
            if (g < 0 || q >= tiles[g + 1]) {
                g = find_group(tiles, n_act, q);
                e = a.act[g];
                off = a.offsets[e];
                cnt = a.offsets[e + 1] - off;
                ctile = -1;
            }
            const int local = q - tiles[g], tile = local / fb_r, fb = local - tile * fb_r;
            if (tile != ctile) {
                ctile = tile;
                mt = min(kTT, cnt - tile * kTT);
                tok = lane < mt ? a.perm[off + tile * kTT + lane] / a.K : 0;
            }
            const int hrow = off + tile * kTT;
            ok = issue(a.gate_up + (size_t)e * 2 * a.I * a.H, a.I, fb * kFps, hrow, mt, hrow, tok);
        }
        if (lane == 0) drain(r, it, err, a.wait_ns);
        return;
    }

    // ---------------- consumers: warp w takes K range [w*H/8, (w+1)*H/8) of all 16 rows
    const int kw = a.H / kWarps, ksteps = kw / 16;
    int n_items = -1, ckey = 0x7fffffff;  // no item has this key
    uint32_t bfr[kMaxSteps][2];
    for (int it = 0;; ++it) {
        if (it == my_shared && n_items < 0) {
            grid_dep_wait();
            // The routing is complete, so the down kernel may launch: it reads the routing
            // before it waits for this grid, and it waits for this grid before it reads h. Its
            // CTAs take the SMs this kernel's CTAs leave and stream down weights while the
            // last gate_up items finish elsewhere.
            grid_dep_launch();
            const int R = routed_tiles(a, lane) * fb_r;
            n_items = my_shared + routed_split(R, c + 1, G) - routed_split(R, c, G);
        }
        if (n_items >= 0 && it >= n_items) break;
        const bool ok = wait_stage(r, it, err, a.wait_ns);
        if (!consumers_all(ok)) break;
        const int s = it % kSt;
        const StageMeta& m = r.meta[s];  // read in place: rewritten only after the stage is released
        const int mt = m.mt, row0 = m.row0, f0 = m.f0, key = m.key;
        if (key != ckey) {
            ckey = key;
            load_bfrag(bfr, a.x + (size_t)m.tok[lane >> 2] * a.H + warp * kw, ksteps, lane);
        }
        const uint32_t a_lane =
            smem_u32(r.st0 + (size_t)s * kStageBytes) + (uint32_t)((lane & 15) * pitch + (warp * kw + 8 * (lane >> 4)) * 2);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < kMaxSteps; ++k)
            if (k < ksteps) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(a_lane + k * 32, a0, a1, a2, a3);
                mma16816(d, a0, a1, a2, a3, bfr[k][0], bfr[k][1]);
            }
        release_stage(r, it);
        // fixed-order sum of the 8 warps' K ranges: lane l holds gate (d0, d1) and up (d2, d3)
        // of feature l/4 for tokens 2*(l%4) and 2*(l%4)+1
        float* red = r.red + (size_t)s * kWarps * 128;
        *reinterpret_cast<float4*>(red + (warp * 32 + lane) * 4) = make_float4(d[0], d[1], d[2], d[3]);
        consumers_sync();
        if (warp == 0) {
            float g0 = 0.f, g1 = 0.f, u0 = 0.f, u1 = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float4 v = *reinterpret_cast<const float4*>(red + (w * 32 + lane) * 4);
                g0 += v.x; g1 += v.y; u0 += v.z; u1 += v.w;
            }
            const int f = lane >> 2, t = 2 * (lane & 3);
            if (t < mt) a.h[(size_t)(row0 + t) * a.Imax + f0 + f] = __float2bfloat16_rn(silu(g0) * u0);
            if (t + 1 < mt) a.h[(size_t)(row0 + t + 1) * a.Imax + f0 + f] = __float2bfloat16_rn(silu(g1) * u1);
        }
    }
    grid_dep_launch();
}

// ---------------------------------------------------------------------------------------

// Few tokens (T <= 8, routing from the cluster router): the token rows are staged once per
// CTA, a stage holds only the 16 weight rows, and up to 3 stages are in flight. Routed items
// come from the router's work records (one 16-byte load each).
constexpr int kMaxSt = 3;
constexpr int kUpStage = 2 * kFps * kPitchH;

struct RingSmall {
    uint8_t* xs;
    uint8_t* st[kMaxSt];
    float* red;
    StageMeta* meta;
    uint32_t* toks;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* xbar;
};

constexpr int kSmallSmemCap = 220 * 1024;

__host__ __device__ inline size_t small_smem_bytes(int T, int nst) {
    return 1024 + (size_t)T * kPitchH + (size_t)nst * kUpStage + (size_t)nst * kWarps * 128 * 4 +
           (size_t)nst * (sizeof(StageMeta) + 4) + (2 * nst + 1) * 8 + 64;
}

__device__ __forceinline__ RingSmall carve_small(uint8_t* raw, int T, int nst) {
    const uint32_t base = smem_u32(raw);
    uint8_t* p = raw + (((base + 127u) & ~127u) - base);
    RingSmall r;
    r.xs = p;
    p += (size_t)((T * kPitchH + 127) & ~127);
    for (int s = 0; s < kMaxSt; ++s) {
        r.st[s] = p;
        if (s < nst) p += kUpStage;
    }
    r.red = reinterpret_cast<float*>(p);
    p += (size_t)nst * kWarps * 128 * 4;
    r.meta = reinterpret_cast<StageMeta*>(p);
    p += (size_t)nst * sizeof(StageMeta);
    r.toks = reinterpret_cast<uint32_t*>(p);
    p += (size_t)nst * 4;
    p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 7) & ~(uintptr_t)7);
    r.full = reinterpret_cast<uint64_t*>(p);
    r.empty = r.full + nst;
    r.xbar = r.empty + nst;
    return r;
}

__global__ void __launch_bounds__(kStreamThreads, 1) k_stream_up_small(LayerArgs a, int nst) {
    extern __shared__ uint8_t smem_raw[];
    RingSmall r = carve_small(smem_raw, a.T, nst);
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t* err = &a.hdr->err;
    const int pitch = 2 * a.H + kPad;
    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&r.full[s], 1);
            mbar_init(&r.empty[s], kWarps);
        }
        mbar_init(r.xbar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int n_shared = a.Is / kFps;  // one token tile: all T tokens

    if (warp == kWarps) {
        // ---------------- producer: the token rows once, then 16 weight rows per item
        if (lane == 0) mbar_arrive_expect_tx(r.xbar, (uint32_t)(a.T * a.H * 2));
        __syncwarp();
        if (lane < a.T) bulk_load(r.xs + (size_t)lane * pitch, a.x + (size_t)lane * a.H, a.H * 2, r.xbar);
        int it = 0, n_items = -1;
        for (int i = blockIdx.x;; i += gridDim.x) {
            if (i >= n_shared && n_items < 0) {
                grid_dep_wait();
                grid_dep_launch();  // the routing is complete: the down kernel may start
                n_items = n_shared + *(volatile int*)&a.hdr->n_uprec;
            }
            if (n_items >= 0 && i >= n_items) break;
            if (__shfl_sync(0xffffffffu, *(volatile int*)&abort_flag, 0)) break;
            const bf16* W;
            int inner, row0, f0, mt;
            uint32_t toks;
            if (i < n_shared) {
                W = a.sgu;
                inner = a.Is;
                row0 = (int)a.P;
                f0 = i * kFps;
                mt = a.T;
                toks = 0x76543210u;
            } else {
                const UpRec rec = a.uprec[i - n_shared];
                W = a.gate_up + (size_t)rec.e * 2 * a.I * a.H;
                inner = a.I;
                row0 = rec.row0;
                f0 = rec.f0;
                mt = rec.mt;
                toks = rec.toks;
            }
            const int s = it % nst;
            bool ok = lane == 0 ? mbar_wait(&r.empty[s], (((uint32_t)(it / nst)) & 1u) ^ 1u, a.wait_ns) : true;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    atomicOr(err, ERR_TIMEOUT);
                    abort_flag = 1;
                }
                break;
            }
            if (lane == 0) {
                StageMeta& m = r.meta[s];
                m.mt = mt;
                m.row0 = row0;
                m.f0 = f0;
                r.toks[s] = toks;
                mbar_arrive_expect_tx(&r.full[s], (uint32_t)(2 * kFps * a.H * 2));
            }
            __syncwarp();
            copy_rows(r.st[s], pitch, W + (size_t)f0 * a.H, a.H, kFps, a.H * 2, &r.full[s], lane);
            copy_rows(r.st[s] + kFps * pitch, pitch, W + (size_t)(inner + f0) * a.H, a.H, kFps, a.H * 2, &r.full[s],
                      lane);
            ++it;
        }
        if (lane == 0) {
            for (int k = 0; k < nst && it - 1 - k >= 0; ++k) {
                const int j = it - 1 - k;
                if (!mbar_wait(&r.full[j % nst], ((uint32_t)(j / nst)) & 1u, a.wait_ns)) atomicOr(err, ERR_TIMEOUT);
            }
            if (!mbar_wait(r.xbar, 0, a.wait_ns)) atomicOr(err, ERR_TIMEOUT);
        }
        return;
    }

    // ---------------- consumers: warp w takes K range [w*H/8, (w+1)*H/8) of all 16 rows
    bool xok = lane == 0 ? mbar_wait(r.xbar, 0, a.wait_ns) : true;
    xok = __shfl_sync(0xffffffffu, xok, 0);
    if (!consumers_all(xok)) {
        if (threadIdx.x == 0) atomicOr(err, ERR_TIMEOUT);
        grid_dep_launch();
        return;
    }
    const int kw = a.H / kWarps;
    int it = 0, n_items = -1;
    for (int i = blockIdx.x;; i += gridDim.x, ++it) {
        if (i >= n_shared && n_items < 0) {
            grid_dep_wait();
            // the routing is complete: the down kernel may launch (as in k_stream_up)
            grid_dep_launch();
            n_items = n_shared + *(volatile int*)&a.hdr->n_uprec;
        }
        if (n_items >= 0 && i >= n_items) break;
        const int s = it % nst;
        bool ok = lane == 0 ? mbar_wait(&r.full[s], ((uint32_t)(it / nst)) & 1u, a.wait_ns) : true;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!consumers_all(ok)) {
            if (threadIdx.x == 0) atomicOr(err, ERR_TIMEOUT);
            break;
        }
        const int mt = r.meta[s].mt, row0 = r.meta[s].row0, f0 = r.meta[s].f0;
        const uint32_t toks = r.toks[s];
        // B operand: lane l addresses token row (l % 8) of this item (rows past mt read row 0)
        const int tt = lane & 7;
        const int tok = tt < mt ? (int)((toks >> (4 * tt)) & 15u) : 0;
        const uint32_t sa = smem_u32(r.st[s]);
        const uint32_t b_lane = smem_u32(r.xs) + (uint32_t)(tok * pitch + (warp * kw + 8 * ((lane >> 3) & 1)) * 2);
        const uint32_t a_lane = sa + (uint32_t)((lane & 15) * pitch + (warp * kw + 8 * (lane >> 4)) * 2);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int k = 0; k < kw / 16; ++k) {
            uint32_t a0, a1, a2, a3, b0, b1;
            ldsm_x4(a_lane + k * 32, a0, a1, a2, a3);
            ldsm_x2(b_lane + k * 32, b0, b1);
            mma16816(d, a0, a1, a2, a3, b0, b1);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&r.empty[s]);
        float* red = r.red + (size_t)s * kWarps * 128;
        *reinterpret_cast<float4*>(red + (warp * 32 + lane) * 4) = make_float4(d[0], d[1], d[2], d[3]);
        consumers_sync();
        if (warp == 0) {
            float g0 = 0.f, g1 = 0.f, u0 = 0.f, u1 = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float4 v = *reinterpret_cast<const float4*>(red + (w * 32 + lane) * 4);
                g0 += v.x; g1 += v.y; u0 += v.z; u1 += v.w;
            }
            const int f = lane >> 2, t = 2 * (lane & 3);
            if (t < mt) a.h[(size_t)(row0 + t) * a.Imax + f0 + f] = __float2bfloat16_rn(silu(g0) * u0);
            if (t + 1 < mt) a.h[(size_t)(row0 + t + 1) * a.Imax + f0 + f] = __float2bfloat16_rn(silu(g1) * u1);
        }
    }
    grid_dep_launch();
}

// ---------------------------------------------------------------------------------------

__global__ void __launch_bounds__(kStreamThreads, 1) k_stream_down(LayerArgs a) {
    extern __shared__ uint8_t smem_raw[];
    Ring r = carve(smem_raw);
    ring_init(r);
    // The routing is complete (the gate_up kernel waited for it before it let this kernel
    // launch); only the h rows come from the gate_up kernel. The producer streams weights from
    // the start; the consumers wait for that kernel before they load any h row.
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t* err = &a.hdr->err;
    const int n_act = a.hdr->n_act;
    const int tiles_s = (a.T + kTT - 1) / kTT;
    const int n_blocks = a.H / kRows;
    const int G = gridDim.x, c = blockIdx.x;
    // this CTA's shared items: a contiguous run in (token tile, output block) order
    const int s0 = routed_split(n_blocks * tiles_s, c, G), my_shared = routed_split(n_blocks * tiles_s, c + 1, G) - s0;

    if (warp == kWarps) {
        // ---------------- producer: the shared items, then this CTA's run of routed items
        // (group, token tile, block)
        int* tiles = r.misc + 4;
        build_tiles(a, tiles, n_blocks);
        const int q0 = routed_split(tiles[n_act], c, G), q1 = routed_split(tiles[n_act], c + 1, G);
        const int n_mine = my_shared + q1 - q0;
        int it = 0;
        int g = -1, e = 0, off = 0, cnt = 0, ctile = -1;
        int tok = 0, slot = 0;
        float sc = 0.f;
        for (int k = 0; k < n_mine; ++k) {
            if (__shfl_sync(0xffffffffu, *(volatile int*)&r.misc[0], 0)) break;
            const bf16* W;
            int inner, hrow0, mt, blk;
            if (k < my_shared) {
                const int i = s0 + k, tile = i / n_blocks, t0 = tile * kTT;
                blk = i - tile * n_blocks;
                W = a.sd;
                inner = a.Is;
                hrow0 = (int)a.P + t0;
                mt = min(kTT, a.T - t0);
                if (lane < mt) {
                    tok = t0 + lane;
                    slot = a.K;
                    sc = a.sgate[t0 + lane];
                }
                ctile = -1;  // the routed token cache no longer matches
            } else {
                const int q = q0 + (k - my_shared);
                if (g < 0 || q >= tiles[g + 1]) {
                    g = find_group(tiles, n_act, q);
                    e = a.act[g];
                    off = a.offsets[e];
                    cnt = a.offsets[e + 1] - off;
                    ctile = -1;
                }
                const int local = q - tiles[g], tile = local / n_blocks;
                blk = local - tile * n_blocks;
                W = a.down + (size_t)e * a.H * a.I;
                inner = a.I;
                hrow0 = off + tile * kTT;
                mt = min(kTT, cnt - tile * kTT);
                if (tile != ctile) {
                    ctile = tile;
                    if (lane < mt) {
                        const int pv = a.perm[hrow0 + lane];
                        tok = pv / a.K;
                        slot = pv - tok * a.K;
                        sc = a.topw[pv];
                    }
                }
            }
            const int s = it % kSt;
            if (!acquire_stage(r, it, err, a.wait_ns)) break;
            StageMeta& m = r.meta[s];
            if (lane < mt) {
                m.tok[lane] = tok;
                m.slot[lane] = slot;
                m.sc[lane] = sc;
            }
            if (lane == 0) {
                m.mt = mt;
                m.row0 = hrow0;
                m.f0 = blk * kRows;
                m.inner = inner;
                m.key = hrow0;  // the h rows of the item
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&r.full[s], (uint32_t)(kRows * inner * 2));
            __syncwarp();
            copy_rows(r.st0 + (size_t)s * kStageBytes, dn_gpitch(inner), W + (size_t)blk * kRows * inner, 4 * (size_t)inner, kRows / 4,
                      inner * 8, &r.full[s], lane);
            ++it;
        }
        if (lane == 0) drain(r, it, err, a.wait_ns);
        return;
    }

    // ---------------- consumers: warp w takes M tile (w % 4) and K half (w / 4)
    const int R = routed_tiles(a, lane) * n_blocks;
    const int n_items = my_shared + routed_split(R, c + 1, G) - routed_split(R, c, G);
    const int mtile = warp & 3, khalf = warp >> 2;
    int ckey = -1;  // h rows are never negative
    uint32_t bfr[kMaxSteps][2];
    grid_dep_wait();  // the h rows of the gate_up kernel
    // every CTA of this grid is resident by now: the combine kernel may launch (it waits for
    // this grid before it reads Y), so its launch is done by the time the last item is
    grid_dep_launch();
    for (int it = 0; it < n_items; ++it) {
        const bool ok = wait_stage(r, it, err, a.wait_ns);
        if (!consumers_all(ok)) break;
        const int s = it % kSt;
        const StageMeta& m = r.meta[s];  // read in place: rewritten only after the stage is released
        const int mt = m.mt, inner = m.inner, f0 = m.f0, key = m.key;
        const int kh = inner / 2, ksteps = kh / 16;
        if (key != ckey) {
            ckey = key;
            const int n = lane >> 2;
            load_bfrag(bfr, a.h + (size_t)(m.row0 + (n < mt ? n : 0)) * a.Imax + khalf * kh, ksteps, lane);
        }
        const uint32_t sa = smem_u32(r.st0 + (size_t)s * kStageBytes);
        // M tile mtile: rows j, j+1 (j = 2*(mtile & 1)) of groups 8*(mtile >> 1) .. +7
        const int gbase = 8 * (mtile >> 1), jbase = 2 * (mtile & 1);
        const int tr = lane & 15;
        const uint32_t a_lane = sa + (uint32_t)((gbase + (tr & 7)) * dn_gpitch(inner) + (jbase + (tr >> 3)) * inner * 2 +
                                                (khalf * kh + 8 * (lane >> 4)) * 2);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < kMaxSteps; ++k)
            if (k < ksteps) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(a_lane + k * 32, a0, a1, a2, a3);
                mma16816(d, a0, a1, a2, a3, bfr[k][0], bfr[k][1]);
            }
        // tokens of this lane's accumulator columns
        const int t0 = 2 * (lane & 3);
        size_t y0 = 0, y1 = 0;
        float s0v = 0.f, s1v = 0.f;
        if (t0 < mt) {
            y0 = ((size_t)m.tok[t0] * (a.K + 1) + m.slot[t0]) * a.H + f0;
            s0v = m.sc[t0];
        }
        if (t0 + 1 < mt) {
            y1 = ((size_t)m.tok[t0 + 1] * (a.K + 1) + m.slot[t0 + 1]) * a.H + f0;
            s1v = m.sc[t0 + 1];
        }
        release_stage(r, it);
        // fixed-order sum of the two K halves, then scale and store: lane l holds tile rows l/4
        // and l/4 + 8 (Wd rows 4*(gbase + l/4) + jbase and the next one) for tokens t0, t0 + 1
        float* red = r.red + (size_t)s * kWarps * 128;
        if (khalf == 1) *reinterpret_cast<float4*>(red + (mtile * 32 + lane) * 4) = make_float4(d[0], d[1], d[2], d[3]);
        consumers_sync();
        if (khalf == 0) {
            const float4 v = *reinterpret_cast<const float4*>(red + (mtile * 32 + lane) * 4);
            const int row = 4 * (gbase + (lane >> 2)) + jbase;
            // rows row and row + 1 are adjacent in Y (row is even): one 8-byte store per token
            if (t0 < mt) *reinterpret_cast<float2*>(a.Y + y0 + row) = make_float2(s0v * (d[0] + v.x), s0v * (d[2] + v.z));
            if (t0 + 1 < mt)
                *reinterpret_cast<float2*>(a.Y + y1 + row) = make_float2(s1v * (d[1] + v.y), s1v * (d[3] + v.w));
        }
    }
    grid_dep_launch();
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
    // stages are laid out for rows of at most 2048 (gate/up) and 512 (down) elements; the K
    // range of each consumer warp must be a whole number of 16-element MMA steps
    return a.T >= 1 && a.T < kGemmMinTokens && a.H <= kMaxH && a.Imax <= kMaxInner && a.H % (kWarps * 16) == 0 &&
           a.I % 32 == 0 && a.Is % 32 == 0;
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
    if (a.uprec && a.T <= kRecTokens && route_cluster_supported(a)) {
        // 3 stages in flight while they fit next to the token rows (T <= 2), else 2
        const int nst = small_smem_bytes(a.T, 3) <= kSmallSmemCap ? 3 : 2;
        const int bytes = (int)small_smem_bytes(a.T, nst);
        static bool conf_small[64] = {};
        if (!conf_small[dev]) {
            e = cudaFuncSetAttribute(k_stream_up_small, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmallSmemCap);
            if (e != cudaSuccess) return e;
            conf_small[dev] = true;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(a.num_sms);
        cfg.blockDim = dim3(kStreamThreads);
        cfg.dynamicSmemBytes = bytes;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        MOE_LAUNCH(MOE_KERNEL_GATE_UP, s, (e = cudaLaunchKernelEx(&cfg, k_stream_up_small, a, nst)));
    } else {
        MOE_LAUNCH(MOE_KERNEL_GATE_UP, s, (e = launch_pdl(k_stream_up, a.num_sms, kStreamSmemBytes, s, a)));
    }
    if (e != cudaSuccess) return e;
    MOE_LAUNCH(MOE_KERNEL_DOWN, s, (e = launch_pdl(k_stream_down, a.num_sms, kStreamSmemBytes, s, a)));
    if (e != cudaSuccess) return e;
    return launch_combine_pdl(a, s);
}

}  // namespace moe
