// common.cuh -- device helpers and the workspace plan shared by the kernels of the MoE layer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

typedef __nv_bfloat16 bf16;

// Default time limit of a bounded device wait (~1 s of global time).
constexpr uint64_t kWaitNs = 1000000000ull;

// Bits of the device error word (first word of the workspace header).
enum : uint32_t { ERR_NONFINITE_SCORE = 1u, ERR_TIMEOUT = 2u, ERR_BAD_ROUTE = 4u };

// Workspace header: a device error word and small counters, zero-filled once by the caller.
struct WsHeader {
    uint32_t err;      // OR of ERR_* bits, cleared by moe_last_device_error
    int32_t n_act;     // experts with at least one routed pair (written by the dispatch scan)
    int32_t n_groups;  // GEMM groups: n_act routed experts + the shared expert
    uint32_t route_ticket;  // CTAs of the fused routing kernel that finished (re-armed to 0)
    int32_t n_uprec;        // routed gate_up work records written by the few-token router
    // Fused few-token kernel. Its router scores and gate_up outputs carry the tag epoch + 1 of
    // the call that wrote them. Every CTA of a call counts itself in on dec_start (which only
    // grows); CTA 0 advances the epoch and the base once all of them are in.
    uint32_t dec_epoch;       // calls completed on this workspace
    uint32_t dec_start_base;  // CTA starts of all earlier calls
    uint32_t pad0[25];
    uint32_t dec_start;       // CTAs started (own 128-byte line)
    uint32_t pad1[63];
};
static_assert(sizeof(WsHeader) == 384, "header layout");

// One routed gate_up work item of the few-token path (T <= 8), written by the router: expert,
// first h row of its tokens, first of its 8 features, token count, and the tokens themselves
// (4 bits each, in h-row order).
struct UpRec {
    int32_t e;
    int32_t row0;
    int16_t f0;
    int16_t mt;
    uint32_t toks;
};

// Tokens up to which the router writes UpRec records (and x rows are staged once per CTA).
constexpr int kRecTokens = 8;

// One group of the grouped GEMM: A rows [a_row0, a_row0 + rows) of the activation tensor,
// B block starting at weight row b_row0, output rows from out_row0; src selects the routed
// (0) or the shared-expert (1) tensor maps.
struct GemmGroup {
    int a_row0, rows, b_row0, out_row0, src;
};

// Tokens from which the layer runs its GEMMs on the tensor cores (below: weight streaming).
constexpr int kGemmMinTokens = 256;
// Tokens up to which routing runs as one fused launch (scores, top-K and dispatch).
constexpr int kFusedRouteTokens = 64;

// Byte offsets of every buffer inside the caller's workspace (256-byte aligned).
struct Plan {
    int T, H, E, K, I, Is, Imax;
    int64_t P;       // T*K routed pairs
    int ldl;         // row stride of the score matrix (E + 1 scores: E routed + the shared gate)
    int nb;          // token blocks of the dispatch
    bool gemm;       // many-token path (tensor-core GEMMs, bf16 Y) instead of weight streaming
    size_t o_hdr, o_logits, o_ids, o_topw, o_sgate, o_counts, o_offsets, o_perm, o_inv, o_lr, o_cntb, o_base,
        o_act, o_h, o_y, o_upg, o_dng, o_upt, o_dnt, o_uprec, o_dlog, o_dh, o_dx, total;
};

constexpr int kStatsTokens = 32;     // tokens per block of the load-balancing statistics
constexpr int kDispatchTokens = 64;  // tokens per block of the dispatch (counting-sort) kernels

inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Returns false for dims outside the supported range (see moe.h).
inline bool make_plan(const moe_dims& d, Plan* p) {
    if (d.T < 0 || d.H < 128 || d.H > 8192 || d.H % 128 || d.K < 1 || d.K > 8 || d.E < d.K || d.E > 256 ||
        d.I < 64 || d.I > 2048 || d.I % 64 || d.Is < 64 || d.Is > 2048 || d.Is % 64)
        return false;
    if ((int64_t)d.T * (d.K + 1) >= (int64_t)1 << 31) return false;
    p->T = d.T; p->H = d.H; p->E = d.E; p->K = d.K; p->I = d.I; p->Is = d.Is;
    p->Imax = d.I > d.Is ? d.I : d.Is;
    p->P = (int64_t)d.T * d.K;
    p->ldl = (d.E + 1 + 3) & ~3;
    p->nb = (d.T + kDispatchTokens - 1) / kDispatchTokens;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t r = o; o = align256(o + bytes); return r; };
    const size_t T = (size_t)d.T, P = (size_t)p->P;
    p->o_hdr = take(sizeof(WsHeader));
    p->o_logits = take(T * p->ldl * 4);
    p->o_ids = take(P * 4);
    p->o_topw = take(P * 4);
    p->o_sgate = take(T * 4);
    p->o_counts = take((size_t)d.E * 4);
    p->o_offsets = take((size_t)(d.E + 1) * 4);
    p->o_perm = take(P * 4);
    p->o_inv = take(P * 4);
    p->o_lr = take(P * 4);
    p->o_cntb = take((size_t)p->nb * d.E * 4);
    p->o_base = take((size_t)p->nb * d.E * 4);
    p->o_act = take((size_t)(d.E + 1) * 4);
    p->o_h = take((P + T) * p->Imax * 2);
    p->gemm = d.T >= kGemmMinTokens;
    // Y, which a statistics call borrows for its per-block partial sums (fp32 + int per expert)
    const size_t ybytes = T * (d.K + 1) * d.H * (p->gemm ? 2 : 4);
    const size_t sbytes = (size_t)((d.T + kStatsTokens - 1) / kStatsTokens) * d.E * 8;
    p->o_y = take(ybytes > sbytes ? ybytes : sbytes);
    p->o_upg = take((size_t)(d.E + 1) * sizeof(GemmGroup));
    p->o_dng = take((size_t)(d.E + 1) * sizeof(GemmGroup));
    p->o_upt = take((size_t)(d.E + 2) * 4);
    p->o_dnt = take((size_t)(d.E + 2) * 4);
    p->o_uprec = take(d.T <= kRecTokens ? P * (size_t)(d.I / 8) * sizeof(UpRec) : 0);
    p->o_dlog = take(d.T <= kRecTokens ? T * (size_t)(d.E + 1) * 8 : 0);
    p->o_dh = take(d.T <= kRecTokens ? (P + T) * (size_t)(p->Imax / 2) * 8 : 0);
    p->o_dx = take(d.T == 1 ? (size_t)(d.H / 2) * 8 : 0);  // the token row as tagged words (host rows)
    p->total = o;
    return true;
}

#ifdef __CUDACC__
// Streaming 16-byte load for data read once (weights): bypasses L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Ordinary read-only 16-byte load (activations, reused across warps).
__device__ __forceinline__ uint4 ld_ro(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// Two bf16 packed in one 32-bit word -> two floats (exact).
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z); f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

// acc + sum_i w[i] * x[i], in order i = 0..7 (fixed rounding order).
__device__ __forceinline__ float dot8(const uint4& w, const float* x, float acc) {
    acc = fmaf(bf_lo(w.x), x[0], acc); acc = fmaf(bf_hi(w.x), x[1], acc);
    acc = fmaf(bf_lo(w.y), x[2], acc); acc = fmaf(bf_hi(w.y), x[3], acc);
    acc = fmaf(bf_lo(w.z), x[4], acc); acc = fmaf(bf_hi(w.z), x[5], acc);
    acc = fmaf(bf_lo(w.w), x[6], acc); acc = fmaf(bf_hi(w.w), x[7], acc);
    return acc;
}

// The same sums with both operands left as bf16: fma.rn.f32.bf16 multiplies two bf16 (the
// product is exact in fp32) and adds in fp32 with one rounding, so the result is bit for bit
// dot8's, without the unpacking. x holds 8 packed bf16.
__device__ __forceinline__ float fma_bf16x2(uint32_t a, uint32_t b, float acc) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}
__device__ __forceinline__ float dot8_bf16(const uint4& w, const uint4& x, float acc) {
    acc = fma_bf16x2(w.x, x.x, acc);
    acc = fma_bf16x2(w.y, x.y, acc);
    acc = fma_bf16x2(w.z, x.z, acc);
    acc = fma_bf16x2(w.w, x.w, acc);
    return acc;
}
// acc + sum_i w[i] * h[i], i = 0..7, where h[i] is the low half (a bf16) of the 32-bit word
// hw[i]: the same order and roundings as dot8.
__device__ __forceinline__ float dot8_bf16_lo(const uint4& w, const uint32_t* hw, float acc) {
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm("{\n\t.reg .b16 al, ah, h0, h1, u0, u1;\n\t"
            "mov.b32 {al, ah}, %1;\n\tmov.b32 {h0, u0}, %2;\n\tmov.b32 {h1, u1}, %3;\n\t"
            "fma.rn.f32.bf16 %0, al, h0, %0;\n\t"
            "fma.rn.f32.bf16 %0, ah, h1, %0;\n\t}"
            : "+f"(acc)
            : "r"(wv[i]), "r"(hw[2 * i]), "r"(hw[2 * i + 1]));
    return acc;
}

// Butterfly sum over the warp; every lane ends with the same, order-fixed value.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// A router or shared-gate score as the routing uses it: the fp32 value, or that value rounded
// to the nearest bf16 under MOE_FLAG_BF16_SCORES.
__device__ __forceinline__ float router_score(float v, int flags) {
    return (flags & MOE_FLAG_BF16_SCORES) ? __bfloat162float(__float2bfloat16_rn(v)) : v;
}

// Order-preserving unsigned key of a router score: larger score, larger key; -0 is taken as
// +0. Key 0 lies below every score (an empty candidate).
__device__ __forceinline__ uint32_t score_key(float v) {
    if (v == 0.f) v = 0.f;
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-K of one token by a warp ("Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256
// Experts, Router: the 8 highest scores; ties go to the lower expert index). Lane l holds the
// keys of experts l + 32j in key[j]. Each lane first sorts its eight (key, j) pairs, larger key
// first and, among equal keys, lower j first (Batcher's odd-even merge network, 19 compare-
// exchanges); then each of K rounds takes the largest head key by a warp max and, among equal
// heads, the lowest expert by a warp min, and the winning lane drops its head. A lane's head is
// its lowest expert of its largest remaining key, so every round picks what a scan of all
// remaining keys would. Lane k < K receives slot k: its score (myv) and expert (mye); every
// lane receives the slot-0 score (v0).
__device__ __forceinline__ void topk_cas(uint32_t (&k)[8], uint32_t (&j)[8], int a, int b) {
    const bool sw = k[b] > k[a] || (k[b] == k[a] && j[b] < j[a]);
    const uint32_t ka = k[a], ja = j[a];
    k[a] = sw ? k[b] : ka;
    j[a] = sw ? j[b] : ja;
    k[b] = sw ? ka : k[b];
    j[b] = sw ? ja : j[b];
}
__device__ __forceinline__ void warp_topk(const uint32_t (&key)[8], int K, int lane, float& v0, float& myv, int& mye) {
    uint32_t k[8], j[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        k[i] = key[i];
        j[i] = (uint32_t)i;
    }
    topk_cas(k, j, 0, 1); topk_cas(k, j, 2, 3); topk_cas(k, j, 4, 5); topk_cas(k, j, 6, 7);
    topk_cas(k, j, 0, 2); topk_cas(k, j, 1, 3); topk_cas(k, j, 4, 6); topk_cas(k, j, 5, 7);
    topk_cas(k, j, 1, 2); topk_cas(k, j, 5, 6);
    topk_cas(k, j, 0, 4); topk_cas(k, j, 1, 5); topk_cas(k, j, 2, 6); topk_cas(k, j, 3, 7);
    topk_cas(k, j, 2, 4); topk_cas(k, j, 3, 5);
    topk_cas(k, j, 1, 2); topk_cas(k, j, 3, 4); topk_cas(k, j, 5, 6);
    v0 = 0.f;
    myv = 0.f;
    mye = 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        if (r < K) {
            const uint32_t m = __reduce_max_sync(0xffffffffu, k[0]);
            const uint32_t win = __reduce_min_sync(0xffffffffu, k[0] == m ? (uint32_t)lane + 32u * j[0] : 0xffffffffu);
            if ((int)(win & 31u) == lane) {
#pragma unroll
                for (int i = 0; i < 7; ++i) {
                    k[i] = k[i + 1];
                    j[i] = j[i + 1];
                }
                k[7] = 0u;
            }
            if (r == 0) v0 = key_score(m);
            if (r == lane) {
                myv = key_score(m);
                mye = (int)win;
            }
        }
    }
}

// Programmatic dependent launch: wait until the previous kernel on the stream has completed
// and its memory is visible (a no-op for a kernel launched without the attribute), and let
// the next kernel on the stream launch early (it waits the same way before reading ours).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}
#endif

}  // namespace moe
