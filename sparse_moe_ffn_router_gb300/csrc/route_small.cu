// route_small.cu -- routing of 9..255 tokens in two kernels.
//
// Router ("Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256 Experts, Router: a linear
// map H -> E, softmax, the 8 highest kept and renormalised; the shared-expert gate
// sigmoid(Linear(x, 1)) is scored as one more row, column E).
//
// k_router_mma: scores[t, r] = x[t] . W[r] (+ br[r]) on the tensor pipe. A cluster of S CTAs
//   takes 16 score rows and up to 64 tokens; CTA s of the cluster multiplies K slice s (H/S
//   columns) with warp-level bf16 MMAs (m16n8k16, fp32 accumulate, K in order; warp w takes
//   tokens 8w..8w+7). Its operand rows come in with 16-byte loads, sixteen per thread in flight,
//   into rows 16 bytes apart modulo 128 so ldmatrix is conflict-free. The S partial 16 x 64
//   tiles are then added in slice order through distributed shared memory, so a score does not
//   depend on which CTA finished first. S (1..8) is the smallest count that fits shared memory,
//   doubled while the grid stays within one wave of the SMs: a few dozen kilobytes per CTA
//   arrive in about one memory latency, where a few CTAs streaming the whole matrix were held
//   to the per-SM copy rate.
// k_route_small: ceil(T/8) CTAs of 1024 threads. Warp w of CTA c takes token 8c + w: top-K
//   (warp_topk: each lane sorts its order-preserving score keys, then K rounds of a warp max
//   over the lanes' largest remaining keys and, among equal keys, a warp min over expert
//   indices), the renormalised weights and the shared gate. The last
//   CTA to finish (a ticket counter in the workspace header, re-armed by that CTA) runs the
//   dispatch: one stable counting sort of the T*K (token, slot) pairs in chunks of 1024;
//   within a warp, pairs of one expert are ranked by lane (match_any), across the warps of a
//   chunk by a prefix of per-warp counts, across chunks by running counts.
// Both launch early (programmatic dependent launch): k_route_small waits for the scores
// (griddepcontrol.wait) and at once lets the expert kernel after it start the shared expert's
// work, which needs no routing; that kernel waits for the routing before its routed work.
#include <math.h>

#include "launch.h"
#include "ring.cuh"

namespace moe {

constexpr int kRmRows = 16, kRmTok = 64;  // score rows and tokens per cluster
constexpr int kRmMaxSplit = 8;            // K slices, one CTA each
constexpr int kRmSmemMax = 200 * 1024;    // dynamic shared memory of one CTA, at most
constexpr int kRmBatch = 16;              // 16-byte loads per thread in flight
constexpr int kRsThreads = 1024, kRsWarps = kRsThreads / 32;
constexpr int kRsTok = 8;  // tokens per routing CTA, one per warp
constexpr int kRsMaxP = 255 * 8;

__host__ __device__ constexpr int rm_pitch(int ks) { return 2 * ks + 16; }
static int rm_smem(int H, int S) { return (kRmRows + kRmTok) * rm_pitch(H / S); }

// K slices of one launch: the fewest that fit shared memory, doubled while the grid stays
// within the SMs (H is a multiple of 128, so every slice is a multiple of 16 columns).
static int rm_split(const LayerArgs& a) {
    const int clusters = ((a.E + 1 + kRmRows - 1) / kRmRows) * ((a.T + kRmTok - 1) / kRmTok);
    int S = 1;
    while (S < kRmMaxSplit && rm_smem(a.H, S) > kRmSmemMax) S *= 2;
    while (S < kRmMaxSplit && clusters * S * 2 <= a.num_sms) S *= 2;
    return S;
}

__device__ __forceinline__ void rm_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float rm_ld_cluster(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

__global__ void __launch_bounds__(256) k_router_mma(LayerArgs a, int S) {
    extern __shared__ __align__(16) uint8_t rm_smem_raw[];
    __shared__ float part[kRmRows * kRmTok];  // this slice's partial tile, [row][token]
    grid_dep_launch();  // the routing kernel may launch; it waits for this grid's scores
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.x;  // K slice == rank in the cluster (cluster S x 1 x 1)
    const int row0 = blockIdx.y * kRmRows, t0 = blockIdx.z * kRmTok;
    const int nr = min(kRmRows, a.E + 1 - row0), nt = min(kRmTok, a.T - t0);
    const int ks = a.H / S, k0 = s * ks, cpr = ks / 8, pitch = rm_pitch(ks);
    const int total = (nr + nt) * cpr;  // 16-byte pieces of this slice's operand rows

    // 1. the nr score rows, then the nt token rows, of K slice s into shared memory
    for (int b = tid; b < total; b += kRmBatch * 256) {
        uint4 v[kRmBatch];
#pragma unroll
        for (int u = 0; u < kRmBatch; ++u) {
            const int i = b + u * 256;
            v[u] = make_uint4(0u, 0u, 0u, 0u);
            if (i < total) {
                const int row = i / cpr, c = i - row * cpr;
                const bf16* src;
                if (row < nr) {
                    const int r = row0 + row;
                    src = r < a.E ? a.router_w + (size_t)r * a.H : a.sg;
                } else {
                    src = a.x + (size_t)(t0 + row - nr) * a.H;
                }
                v[u] = ld_ro(src + k0 + 8 * c);
            }
        }
#pragma unroll
        for (int u = 0; u < kRmBatch; ++u) {
            const int i = b + u * 256;
            if (i < total) {
                const int row = i / cpr, c = i - row * cpr;
                const int slot = row < nr ? row : kRmRows + row - nr;
                *reinterpret_cast<uint4*>(rm_smem_raw + (size_t)slot * pitch + 16 * c) = v[u];
            }
        }
    }
    __syncthreads();

    // 2. the 16 x 64 partial tile of this slice, K in order
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    if (8 * warp < nt) {
        const int ra = lane & 15, tb = lane & 7;
        const int arow = ra < nr ? ra : 0;
        const int brow = 8 * warp + tb < nt ? 8 * warp + tb : 0;
        const uint32_t sb = smem_u32(rm_smem_raw);
        const uint32_t pa = sb + (uint32_t)(arow * pitch + 16 * (lane >> 4));
        const uint32_t pb = sb + (uint32_t)((kRmRows + brow) * pitch + 16 * ((lane >> 3) & 1));
        for (int k = 0; k < ks / 16; ++k) {
            uint32_t a0, a1, a2, a3, b0, b1;
            ldsm_x4(pa + k * 32, a0, a1, a2, a3);
            ldsm_x2(pb + k * 32, b0, b1);
            mma16816(d, a0, a1, a2, a3, b0, b1);
        }
    }
    // lane holds rows lane/4 and lane/4 + 8 for tokens 8w + 2(lane%4) and the next one
#pragma unroll
    for (int q = 0; q < 4; ++q)
        part[((lane >> 2) + (q >= 2 ? 8 : 0)) * kRmTok + 8 * warp + 2 * (lane & 3) + (q & 1)] = d[q];
    rm_cluster_sync();  // every slice's partial tile is written

    // 3. CTA s adds its share of the tile over the slices 0..S-1, in that order
    const uint32_t pbase = smem_u32(part);
    const int per = kRmRows * kRmTok / S;
    for (int i = tid; i < per; i += 256) {
        const int e = s * per + i, rl = e / kRmTok, tl = e % kRmTok;
        if (rl < nr && tl < nt) {
            float p[kRmMaxSplit];
#pragma unroll
            for (int q = 0; q < kRmMaxSplit; ++q)
                p[q] = q < S ? rm_ld_cluster(pbase + 4u * (uint32_t)e, (uint32_t)q) : 0.f;
            float v = p[0];
#pragma unroll
            for (int q = 1; q < kRmMaxSplit; ++q)
                if (q < S) v += p[q];
            const int r = row0 + rl;
            const float bias = (r < a.E && a.router_b) ? __bfloat162float(a.router_b[r]) : 0.f;
            a.logits[(size_t)(t0 + tl) * a.ldl + r] = v + bias;
        }
    }
    rm_cluster_sync();  // the other slices read this CTA's tile up to here
}

// Top-K of token t by one warp: ids in slot order, renormalised weights, shared gate.
__device__ __forceinline__ void rs_topk_token(const LayerArgs& a, int t, int lane) {
    const float* l = a.logits + (size_t)t * a.ldl;
    const int E = a.E, K = a.K;
    bool bad = false;
    uint32_t key[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        key[j] = 0u;  // below every score: never taken while a real expert remains
        if (lane + 32 * j < E) {
            float v = router_score(l[lane + 32 * j], a.flags);
            if (!isfinite(v)) {
                bad = true;
                v = -INFINITY;
            }
            key[j] = score_key(v);
        }
    }
    float v0, myv;
    int mye;
    warp_topk(key, K, lane, v0, myv, mye);
    const float ex = lane < K ? expf(myv - v0) : 0.f;
    const float s = warp_sum(ex);
    if (lane < K) {
        a.ids[(size_t)t * K + lane] = mye;
        a.topw[(size_t)t * K + lane] = ex / s;
    }
    if (lane == 0) {
        const float z = router_score(l[E], a.flags);
        if (!isfinite(z)) bad = true;
        a.sgate[t] = 1.0f / (1.0f + expf(-z));
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&a.hdr->err, ERR_NONFINITE_SCORE);
}

__global__ void __launch_bounds__(kRsThreads, 1) k_route_small(LayerArgs a) {
    __shared__ int sid[kRsMaxP];
    __shared__ int srank[kRsMaxP];
    __shared__ uint16_t wcnt[kRsWarps][256];  // per-warp pair counts of each expert, then their prefix
    __shared__ int running[256], total[256], off[257];
    __shared__ int n_act_s;
    __shared__ uint32_t ticket;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T, E = a.E, K = a.K, P = T * K;
    grid_dep_wait();    // the scores of k_router_mma
    grid_dep_launch();  // the expert kernel may start its shared-expert work

    // 1. top-K, weights and shared gate of this CTA's tokens
    const int t = blockIdx.x * kRsTok + warp;
    if (warp < kRsTok && t < T) rs_topk_token(a, t, lane);

    // 2. the last CTA to get here sorts the pairs of every token: thread 0 counts the CTA in
    //    with one acquire-release atomic after the CTA barrier (the release covers the ids
    //    the CTA's warps wrote, the acquire the other CTAs' ids)
    __syncthreads();
    if (tid == 0) ticket = atom_acq_rel_add(&a.hdr->route_ticket, 1u);
    __syncthreads();
    if (ticket != gridDim.x - 1) return;
    for (int p = tid; p < P; p += kRsThreads) sid[p] = __ldcg(a.ids + p);
    for (int e = tid; e < 256; e += kRsThreads) running[e] = 0;
    __syncthreads();

    // stable counting sort of the pairs by expert, 1024 pairs at a time
    for (int b0 = 0; b0 < P; b0 += kRsThreads) {
        for (int i = tid; i < kRsWarps * 256; i += kRsThreads) (&wcnt[0][0])[i] = 0;
        __syncthreads();
        const int p = b0 + tid;
        const int e = p < P ? sid[p] : -1;
        const unsigned m = __match_any_sync(0xffffffffu, e);
        const int rw = __popc(m & ((1u << lane) - 1u));
        if (e >= 0 && rw == 0) wcnt[warp][e] = (uint16_t)__popc(m);
        __syncthreads();
        if (tid < E) {
            int run = 0;
            for (int w = 0; w < kRsWarps; ++w) {
                const int cnt = wcnt[w][tid];
                wcnt[w][tid] = (uint16_t)run;
                run += cnt;
            }
            total[tid] = run;
        }
        __syncthreads();
        if (e >= 0) srank[p] = running[e] + wcnt[warp][e] + rw;
        __syncthreads();
        if (tid < E) running[tid] += total[tid];
        __syncthreads();
    }
    // offsets (exclusive scan of the counts) and the ascending list of used experts, one warp
    if (warp == 0) {
        int loc[8], run = 0, nz = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane * 8 + j;
            loc[j] = e < E ? running[e] : 0;
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
            if (e < E) {
                off[e] = pos;
                if (loc[j] > 0) a.act[apos++] = e;
            }
            pos += loc[j];
        }
        if (lane == 31) {
            off[E] = incl;
            n_act_s = inz;
        }
    }
    __syncthreads();
    for (int e = tid; e <= E; e += kRsThreads) {
        a.offsets[e] = off[e];
        if (e < E) a.counts[e] = running[e];
    }
    if (tid == 0) {
        a.hdr->n_act = n_act_s;
        a.hdr->route_ticket = 0;  // re-arm for the next call on this workspace
    }
    for (int p = tid; p < P; p += kRsThreads) {
        const int j = off[sid[p]] + srank[p];
        a.perm[j] = p;
        a.inv[p] = j;
    }
}

bool route_small_supported(const LayerArgs& a) {
    return a.T >= 1 && a.T < kGemmMinTokens && (size_t)a.T * a.K <= (size_t)kRsMaxP && a.E <= 256 && a.K <= 8 &&
           a.H % 128 == 0 && rm_smem(a.H, kRmMaxSplit) <= kRmSmemMax;
}

cudaError_t launch_route_small(const LayerArgs& a, cudaStream_t s) {
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!configured[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(k_router_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, kRmSmemMax);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int S = rm_split(a);
    cudaError_t e = cudaSuccess;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(S, (a.E + 1 + kRmRows - 1) / kRmRows, (a.T + kRmTok - 1) / kRmTok);
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = rm_smem(a.H, S);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = S;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        MOE_LAUNCH(MOE_KERNEL_ROUTER_SCORES, s, (e = cudaLaunchKernelEx(&cfg, k_router_mma, a, S)));
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.T + kRsTok - 1) / kRsTok);
    cfg.blockDim = dim3(kRsThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    MOE_LAUNCH(MOE_KERNEL_ROUTER_TOPK, s, (e = cudaLaunchKernelEx(&cfg, k_route_small, a)));
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
