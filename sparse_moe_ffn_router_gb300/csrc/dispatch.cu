// dispatch.cu -- exact, reproducible dispatch of (token, slot) pairs to experts.
//
// The pages say only that the router "determines which experts should receive this token"
// ("One Token Through Qwen3.6", The Router). The layout here is a stable counting sort of
// the pairs p = t*K + k by expert: counts, exclusive offsets, and perm (tokens ascending
// within an expert), in three integer passes:
//   1. per block of 64 tokens (one warp): per-expert counts and each pair's rank among the
//      block's pairs of the same expert, in token order (match_any + popc, no atomics);
//   2. one CTA: per-expert totals, the exclusive scan, each (block, expert) base, and the
//      list of experts that received pairs;
//   3. scatter: perm[base[block, e] + rank] = p, inv[p] = that position.
#include "launch.h"

namespace moe {

__global__ void __launch_bounds__(32) k_dispatch_local(LayerArgs a) {
    __shared__ int cnt[256];
    const int lane = threadIdx.x, b = blockIdx.x;
    for (int e = lane; e < a.E; e += 32) cnt[e] = 0;
    __syncwarp();
    const int64_t p0 = (int64_t)b * kDispatchTokens * a.K;
    const int64_t p1 = (int64_t)min((b + 1) * kDispatchTokens, a.T) * a.K;
    for (int64_t base = p0; base < p1; base += 32) {
        const int64_t i = base + lane;
        const bool valid = i < p1;
        const int e = valid ? a.ids[i] : -1;
        const unsigned m = __match_any_sync(0xffffffffu, e);
        const int rank_in = __popc(m & ((1u << lane) - 1u));
        const int c = valid ? cnt[e] : 0;
        __syncwarp();
        if (valid) {
            a.lr[i] = c + rank_in;
            if (rank_in == 0) cnt[e] = c + __popc(m);
        }
        __syncwarp();
    }
    for (int e = lane; e < a.E; e += 32) a.cntb[(size_t)b * a.E + e] = cnt[e];
}

__global__ void __launch_bounds__(256) k_dispatch_scan(LayerArgs a) {
    __shared__ int tot[256];
    __shared__ int off[257];
    const int e = threadIdx.x;
    if (e < a.E) {
        int s = 0;
        for (int b = 0; b < a.nb; ++b) s += a.cntb[(size_t)b * a.E + e];
        tot[e] = s;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0, na = 0;
        for (int j = 0; j < a.E; ++j) {
            off[j] = run;
            run += tot[j];
            if (tot[j] > 0) a.act[na++] = j;
        }
        off[a.E] = run;
        a.hdr->n_act = na;
    }
    __syncthreads();
    if (e < a.E) {
        a.counts[e] = tot[e];
        a.offsets[e] = off[e];
        int run = off[e];
        for (int b = 0; b < a.nb; ++b) {
            a.base[(size_t)b * a.E + e] = run;
            run += a.cntb[(size_t)b * a.E + e];
        }
    }
    if (e == 0) a.offsets[a.E] = off[a.E];
}

__global__ void __launch_bounds__(256) k_dispatch_scatter(LayerArgs a) {
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i >= a.P) return;
    const int t = (int)(i / a.K);
    const int b = t / kDispatchTokens;
    const int e = a.ids[i];
    const int j = a.base[(size_t)b * a.E + e] + a.lr[i];
    a.perm[j] = (int)i;
    a.inv[i] = j;
}

// Tables of the grouped tensor-core GEMMs: one group per expert that received pairs (in
// expert order), then the shared expert over all T tokens; each group's first tile.
__global__ void k_gemm_plan(LayerArgs a, int fh, int bn_dn) {
    // one warp: each group's tile counts, then a warp-wide running prefix over the groups
    const int lane = threadIdx.x & 31;
    if (threadIdx.x >= 32) return;
    const int n = a.hdr->n_act;
    int tu = 0, td = 0;
    for (int base = 0; base <= n; base += 32) {
        const int g = base + lane;
        int cu = 0, cd = 0;
        GemmGroup up{}, dn{};
        if (g < n) {
            const int e = a.act[g];
            const int r0 = a.offsets[e];
            const int rows = a.offsets[e + 1] - r0;
            up = GemmGroup{r0, rows, e * 2 * a.I, r0, 0};
            dn = GemmGroup{r0, rows, e * a.H, 0, 0};
            const int mt = (rows + 127) / 128;
            cu = mt * (a.I / fh);
            cd = mt * (a.H / bn_dn);
        } else if (g == n) {
            up = GemmGroup{0, a.T, 0, (int)a.P, 1};
            dn = GemmGroup{(int)a.P, a.T, 0, 0, 1};
            const int mt = (a.T + 127) / 128;
            cu = mt * (a.Is / fh);
            cd = mt * (a.H / bn_dn);
        }
        int iu = cu, id = cd;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int yu = __shfl_up_sync(0xffffffffu, iu, o);
            const int yd = __shfl_up_sync(0xffffffffu, id, o);
            if (lane >= o) {
                iu += yu;
                id += yd;
            }
        }
        if (g <= n) {
            a.up_groups[g] = up;
            a.dn_groups[g] = dn;
            a.up_tiles[g] = tu + iu - cu;
            a.dn_tiles[g] = td + id - cd;
        }
        tu += __shfl_sync(0xffffffffu, iu, 31);
        td += __shfl_sync(0xffffffffu, id, 31);
    }
    if (lane == 0) {
        a.up_tiles[n + 1] = tu;
        a.dn_tiles[n + 1] = td;
        *a.n_groups = n + 1;
    }
}

// xperm[j] = x[perm[j] / K]: the token rows in dispatch order, the A operand of gate_up.
__global__ void __launch_bounds__(256) k_gather_rows(LayerArgs a) {
    const int64_t j = blockIdx.x;
    const int t = a.perm[j] / a.K;
    const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)t * a.H);
    uint4* dst = reinterpret_cast<uint4*>(a.xperm + (size_t)j * a.H);
    for (int c = threadIdx.x; c < a.H / 8; c += 256) dst[c] = src[c];
}

cudaError_t launch_gemm_prep(const LayerArgs& a, cudaStream_t s) {
    const int fh = (a.I % 128 == 0 && a.Is % 128 == 0) ? 128 : 64;
    const int bn_dn = (a.H % 256 == 0) ? 256 : 128;
    MOE_LAUNCH(MOE_KERNEL_GEMM_PLAN, s, (k_gemm_plan<<<1, 32, 0, s>>>(a, fh, bn_dn)));
    MOE_LAUNCH(MOE_KERNEL_GATHER, s, (k_gather_rows<<<(unsigned)a.P, 256, 0, s>>>(a)));
    return cudaGetLastError();
}

cudaError_t launch_dispatch(const LayerArgs& a, cudaStream_t s) {
    MOE_LAUNCH(MOE_KERNEL_DISPATCH_LOCAL, s, (k_dispatch_local<<<a.nb, 32, 0, s>>>(a)));
    MOE_LAUNCH(MOE_KERNEL_DISPATCH_SCAN, s, (k_dispatch_scan<<<1, 256, 0, s>>>(a)));
    MOE_LAUNCH(MOE_KERNEL_DISPATCH_SCATTER, s, (k_dispatch_scatter<<<(unsigned)((a.P + 255) / 256), 256, 0, s>>>(a)));
    return cudaGetLastError();
}

}  // namespace moe
