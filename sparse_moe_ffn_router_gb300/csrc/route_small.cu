// route_small.cu -- routing of 9..255 tokens in two kernels.
//
// Router ("Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256 Experts, Router: a linear
// map H -> E, softmax, the 8 highest kept and renormalised; the shared-expert gate
// sigmoid(Linear(x, 1)) is scored as one more row, column E).
//
// k_router_mma: scores[t, r] = x[t] . W[r] (+ br[r]) on the tensor pipe. A CTA takes 16 score
//   rows and 64 tokens; K streams through two shared-memory buffers in chunks of 512 with 1-D
//   TMA bulk copies (one per row, rows 16 bytes apart modulo 128 so ldmatrix is
//   conflict-free); warp w multiplies the 16 rows by tokens 8w..8w+7 with warp-level bf16 MMAs
//   (m16n8k16, fp32 accumulate, K in order).
// k_route_small: one CTA of 1024 threads. Top-K of every token (a warp per token: each of K
//   rounds takes the largest remaining order-preserving score key by a warp max and, among
//   equal keys, the lowest expert index by a warp min), the renormalised weights and the
//   shared gate; then the dispatch as one stable counting sort of the T*K (token, slot) pairs in
//   chunks of 1024: within a warp, pairs of one expert are ranked by lane (match_any), across
//   the warps of a chunk by a prefix of per-warp counts, across chunks by running counts.
// Both launch early (programmatic dependent launch): k_route_small waits for the scores
// (griddepcontrol.wait) and at once lets the expert kernel after it start the shared expert's
// work, which needs no routing; that kernel waits for the routing before its routed work.
#include <math.h>

#include "launch.h"
#include "ring.cuh"

namespace moe {

constexpr int kRmRows = 16, kRmTok = 64, kRmKc = 512;   // rows and tokens per CTA, K chunk
constexpr int kRmPitch = 2 * kRmKc + 16;                // bytes per staged row
constexpr int kRmBuf = (kRmRows + kRmTok) * kRmPitch;   // one K chunk of A and B rows
constexpr int kRmSmem = 2 * kRmBuf + 128;
constexpr int kRsThreads = 1024, kRsWarps = kRsThreads / 32;
constexpr int kRsMaxP = 255 * 8;

__global__ void __launch_bounds__(256) k_router_mma(LayerArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[2];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* base = smem_raw + (((raw + 127u) & ~127u) - raw);
    grid_dep_launch();  // the routing kernel may launch; it waits for this grid's scores
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * kRmRows, t0 = blockIdx.y * kRmTok;
    const int nr = min(kRmRows, a.E + 1 - row0), nt = min(kRmTok, a.T - t0);
    const int nc = (a.H + kRmKc - 1) / kRmKc;
    if (threadIdx.x == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // chunk c of the nr score rows and nt token rows into buffer c % 2 (warp 0)
    auto issue = [&](int c) {
        const int k0 = c * kRmKc, kl = min(kRmKc, a.H - k0);
        uint8_t* buf = base + (size_t)(c & 1) * kRmBuf;
        if (lane == 0) mbar_arrive_expect_tx(&full[c & 1], (uint32_t)((nr + nt) * kl * 2));
        __syncwarp();
        for (int i = lane; i < nr + nt; i += 32) {
            const bf16* src;
            if (i < nr) {
                const int r = row0 + i;
                src = (r < a.E ? a.router_w + (size_t)r * a.H : a.sg) + k0;
            } else {
                src = a.x + (size_t)(t0 + i - nr) * a.H + k0;
            }
            bulk_load(buf + (size_t)(i < nr ? i : kRmRows + i - nr) * kRmPitch, src, kl * 2, &full[c & 1]);
        }
    };
    if (warp == 0) {
        issue(0);
        if (nc > 1) issue(1);
    }
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    const int ra = lane & 15, tb = lane & 7;
    const int arow = ra < nr ? ra : 0;
    const int brow = 8 * warp + tb < nt ? 8 * warp + tb : 0;
    bool ok = true;
    for (int c = 0; c < nc; ++c) {
        const int kl = min(kRmKc, a.H - c * kRmKc);
        const bool w = lane == 0 ? mbar_wait(&full[c & 1], (uint32_t)((c >> 1) & 1)) : true;
        ok = __shfl_sync(0xffffffffu, w, 0) && ok;
        __syncwarp();
        const uint32_t buf = smem_u32(base + (size_t)(c & 1) * kRmBuf);
        if (8 * warp < nt) {
            const uint32_t pa = buf + (uint32_t)(arow * kRmPitch + 16 * (lane >> 4));
            const uint32_t pb = buf + (uint32_t)((kRmRows + brow) * kRmPitch + 16 * ((lane >> 3) & 1));
            for (int k = 0; k < kl / 16; ++k) {
                uint32_t a0, a1, a2, a3, b0, b1;
                ldsm_x4(pa + k * 32, a0, a1, a2, a3);
                ldsm_x2(pb + k * 32, b0, b1);
                mma16816(d, a0, a1, a2, a3, b0, b1);
            }
        }
        __syncthreads();  // every warp is done with this buffer
        if (warp == 0 && c + 2 < nc) issue(c + 2);
    }
    if (!ok && threadIdx.x == 0) atomicOr(&a.hdr->err, ERR_TIMEOUT);
    // lane holds rows lane/4 and lane/4 + 8 for tokens 8w + 2(lane%4) and the next one
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int rl = (lane >> 2) + (q >= 2 ? 8 : 0), tl = 8 * warp + 2 * (lane & 3) + (q & 1);
        if (rl < nr && tl < nt) {
            const int r = row0 + rl;
            const float b = (r < a.E && a.router_b) ? __bfloat162float(a.router_b[r]) : 0.f;
            a.logits[(size_t)(t0 + tl) * a.ldl + r] = d[q] + b;
        }
    }
}

// Order-preserving unsigned key of a score: larger score, larger key; -0 is taken as +0.
__device__ __forceinline__ uint32_t rs_key(float v) {
    if (v == 0.f) v = 0.f;
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float rs_score(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__global__ void __launch_bounds__(kRsThreads, 1) k_route_small(LayerArgs a) {
    __shared__ int sid[kRsMaxP];
    __shared__ int srank[kRsMaxP];
    __shared__ uint16_t wcnt[kRsWarps][256];  // per-warp pair counts of each expert, then their prefix
    __shared__ int running[256], total[256], off[257];
    __shared__ int n_act_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T, E = a.E, K = a.K, P = T * K;
    grid_dep_wait();    // the scores of k_router_mma
    grid_dep_launch();  // the expert kernel may start its shared-expert work

    // 1. top-K, weights and shared gate of every token
    for (int t = warp; t < T; t += kRsWarps) {
        const float* l = a.logits + (size_t)t * a.ldl;
        bool bad = false;
        uint32_t key[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            key[j] = 0u;  // below every score: never taken while a real expert remains
            if (lane + 32 * j < E) {
                float v = l[lane + 32 * j];
                if (!isfinite(v)) {
                    bad = true;
                    v = -INFINITY;
                }
                key[j] = rs_key(v);
            }
        }
        uint32_t taken = 0;
        float v0 = 0.f, myv = 0.f;
        int mye = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k < K) {
                uint32_t bk = 0;
                int bj = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (!((taken >> j) & 1u) && key[j] > bk) {
                        bk = key[j];
                        bj = j;
                    }
                const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
                const uint32_t win =
                    __reduce_min_sync(0xffffffffu, bk == m ? (uint32_t)(lane + 32 * bj) : 0xffffffffu);
                if ((int)(win & 31u) == lane) taken |= 1u << (win >> 5);
                if (k == 0) v0 = rs_score(m);
                if (k == lane) {
                    myv = rs_score(m);
                    mye = (int)win;
                }
            }
        }
        const float ex = lane < K ? expf(myv - v0) : 0.f;
        const float s = warp_sum(ex);
        if (lane < K) {
            sid[t * K + lane] = mye;
            a.ids[(size_t)t * K + lane] = mye;
            a.topw[(size_t)t * K + lane] = ex / s;
        }
        if (lane == 0) {
            const float z = l[E];
            if (!isfinite(z)) bad = true;
            a.sgate[t] = 1.0f / (1.0f + expf(-z));
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&a.hdr->err, ERR_NONFINITE_SCORE);
    }
    for (int e = tid; e < 256; e += kRsThreads) running[e] = 0;
    __syncthreads();

    // 2. stable counting sort of the pairs by expert, 1024 pairs at a time
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
    if (tid == 0) a.hdr->n_act = n_act_s;
    for (int p = tid; p < P; p += kRsThreads) {
        const int j = off[sid[p]] + srank[p];
        a.perm[j] = p;
        a.inv[p] = j;
    }
}

bool route_small_supported(const LayerArgs& a) {
    return a.T >= 1 && a.T < kGemmMinTokens && (size_t)a.T * a.K <= (size_t)kRsMaxP && a.E <= 256 && a.K <= 8 &&
           a.H % 128 == 0;
}

cudaError_t launch_route_small(const LayerArgs& a, cudaStream_t s) {
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!configured[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(k_router_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, kRmSmem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const dim3 g1((a.E + 1 + kRmRows - 1) / kRmRows, (a.T + kRmTok - 1) / kRmTok);
    MOE_LAUNCH(MOE_KERNEL_ROUTER_SCORES, s, (k_router_mma<<<g1, 256, kRmSmem, s>>>(a)));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kRsThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaSuccess;
    MOE_LAUNCH(MOE_KERNEL_ROUTER_TOPK, s, (e = cudaLaunchKernelEx(&cfg, k_route_small, a)));
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
