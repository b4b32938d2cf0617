// dispatch.cu -- exact, reproducible dispatch of (token, slot) pairs to experts.
//
// The pages say only that the router "determines which experts should receive this token"
// ("One Token Through Qwen3.6", The Router). The layout here is a stable counting sort of
// the pairs p = t*K + k by expert: counts, exclusive offsets, and perm (tokens ascending
// within an expert), in three integer passes:
//   1. per block of 64 tokens (one warp): per-expert counts and each pair's rank among the
//      block's pairs of the same expert, in token order (match_any + popc, no atomics); the
//      block's expert ids are loaded up front, so the ranking loop waits on no memory;
//   2. one CTA: per-expert totals, the exclusive scan (one warp, shuffles), each (block,
//      expert) base, the list of experts that received pairs and, on the tensor-core path,
//      the grouped GEMMs' group and tile tables;
//   3. scatter: perm[base[block, e] + rank] = p, inv[p] = that position (the grouped gate_up
//      GEMM gathers its A rows from x through perm).
#include "launch.h"

namespace moe {

constexpr int kLocalIds = kDispatchTokens * 8 / 32;  // expert ids per lane of a block, at most

__global__ void __launch_bounds__(32) k_dispatch_local(LayerArgs a) {
    __shared__ int cnt[256];
    grid_dep_wait();  // the top-K's expert ids
    grid_dep_launch();
    const int lane = threadIdx.x, b = blockIdx.x;
    for (int e = lane; e < a.E; e += 32) cnt[e] = 0;
    const int64_t p0 = (int64_t)b * kDispatchTokens * a.K;
    const int64_t p1 = (int64_t)min((b + 1) * kDispatchTokens, a.T) * a.K;
    int ev[kLocalIds];
#pragma unroll
    for (int j = 0; j < kLocalIds; ++j) {
        const int64_t i = p0 + 32 * j + lane;
        ev[j] = i < p1 ? a.ids[i] : -1;
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < kLocalIds; ++j) {
        if (p0 + 32 * j >= p1) break;
        const int64_t i = p0 + 32 * j + lane;
        const int e = ev[j];
        const unsigned m = __match_any_sync(0xffffffffu, e);
        const int rank_in = __popc(m & ((1u << lane) - 1u));
        const int c = e >= 0 ? cnt[e] : 0;
        __syncwarp();
        if (e >= 0) {
            a.lr[i] = c + rank_in;
            if (rank_in == 0) cnt[e] = c + __popc(m);
        }
        __syncwarp();
    }
    for (int e = lane; e < a.E; e += 32) a.cntb[(size_t)b * a.E + e] = cnt[e];
}

// Tables of the grouped tensor-core GEMMs from the dispatch (one warp): one group per expert
// that received pairs (in expert order), then the shared expert over all T tokens; each
// group's first tile. act/off/tot: the expert list, offsets and counts in shared memory.
__device__ void gemm_plan_warp(const LayerArgs& a, const int* act, int n, const int* off, const int* tot, int fh,
                               int bn_dn) {
    const int lane = threadIdx.x & 31;
    int tu = 0, td = 0;
    for (int base = 0; base <= n; base += 32) {
        const int g = base + lane;
        int cu = 0, cd = 0;
        GemmGroup up{}, dn{};
        if (g < n) {
            const int e = act[g];
            const int r0 = off[e], rows = tot[e];
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

constexpr int kScanParts = 4, kScanRegs = 16;  // threads per expert, block counts kept in registers

__global__ void __launch_bounds__(256 * kScanParts) k_dispatch_scan(LayerArgs a, int fh, int bn_dn) {
    __shared__ int part[kScanParts][256];
    __shared__ int tot[256];
    __shared__ int off[257];
    __shared__ int sact[256];
    __shared__ int n_act_s;
    grid_dep_wait();  // the block counts of the local pass
    grid_dep_launch();
    // thread (q, e) takes blocks [q*nb/4, (q+1)*nb/4) of expert e: its counts in one round of
    // loads (up to kScanRegs of them kept for the bases), then their sum
    const int e = threadIdx.x & 255, q = threadIdx.x >> 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b0 = q * a.nb / kScanParts, b1 = (q + 1) * a.nb / kScanParts;
    int c[kScanRegs];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < kScanRegs; ++i) {
        c[i] = (e < a.E && b0 + i < b1) ? a.cntb[(size_t)(b0 + i) * a.E + e] : 0;
        sum += c[i];
    }
    if (e < a.E)
        for (int b = b0 + kScanRegs; b < b1; ++b) sum += a.cntb[(size_t)b * a.E + e];
    part[q][e] = sum;
    __syncthreads();
    if (q == 0) tot[e] = part[0][e] + part[1][e] + part[2][e] + part[3][e];
    __syncthreads();
    if (warp == 0) {
        // exclusive scan of the counts and the ascending list of experts with pairs: lane
        // owns experts 8*lane .. 8*lane + 7
        int loc[8], run = 0, nz = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            loc[j] = tot[lane * 8 + j];
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
            const int x = lane * 8 + j;
            if (x < a.E) {
                off[x] = pos;
                if (loc[j] > 0) {
                    sact[apos] = x;
                    a.act[apos] = x;
                    ++apos;
                }
            }
            pos += loc[j];
        }
        if (lane == 31) {
            off[a.E] = incl;
            n_act_s = inz;
            a.hdr->n_act = inz;
        }
    }
    __syncthreads();
    if (e < a.E) {
        if (q == 0) {
            a.counts[e] = tot[e];
            a.offsets[e] = off[e];
        }
        int run = off[e];
        for (int p = 0; p < q; ++p) run += part[p][e];
#pragma unroll
        for (int i = 0; i < kScanRegs; ++i)
            if (b0 + i < b1) {
                a.base[(size_t)(b0 + i) * a.E + e] = run;
                run += c[i];
            }
        for (int b = b0 + kScanRegs; b < b1; ++b) {
            a.base[(size_t)b * a.E + e] = run;
            run += a.cntb[(size_t)b * a.E + e];
        }
    }
    if (threadIdx.x == 0) a.offsets[a.E] = off[a.E];
    if (a.gemm && warp == 1) gemm_plan_warp(a, sact, n_act_s, off, tot, fh, bn_dn);
}

__global__ void __launch_bounds__(256) k_dispatch_scatter(LayerArgs a) {
    grid_dep_wait();  // the bases of the scan
    grid_dep_launch();
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i >= a.P) return;
    const int t = (int)(i / a.K);
    const int b = t / kDispatchTokens;
    const int e = a.ids[i];
    const int j = a.base[(size_t)b * a.E + e] + a.lr[i];
    a.perm[j] = (int)i;
    a.inv[i] = j;
}

cudaError_t launch_dispatch(const LayerArgs& a, cudaStream_t s) {
    const int fh = gemm_up_half(a), bn_dn = gemm_down_bn(a);
    cudaError_t e;
    MOE_LAUNCH(MOE_KERNEL_DISPATCH_LOCAL, s, (e = launch_pdl(k_dispatch_local, dim3(a.nb), dim3(32), 0, s, a)));
    if (e != cudaSuccess) return e;
    MOE_LAUNCH(MOE_KERNEL_DISPATCH_SCAN, s,
               (e = launch_pdl(k_dispatch_scan, dim3(1), dim3(256 * kScanParts), 0, s, a, fh, bn_dn)));
    if (e != cudaSuccess) return e;
    MOE_LAUNCH(MOE_KERNEL_DISPATCH_SCATTER, s,
               (e = launch_pdl(k_dispatch_scatter, dim3((unsigned)((a.P + 255) / 256)), dim3(256), 0, s, a)));
    return e;
}

}  // namespace moe
