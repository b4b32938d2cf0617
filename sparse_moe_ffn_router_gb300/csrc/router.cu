// router.cu -- router scores, softmax/top-K/renormalisation, and RMSNorm.
//
// Router ("Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256 Experts, Router): a
// linear map H -> E scores every expert, softmax, the top K are kept and their weights
// renormalised to sum to 1. The shared-expert gate sigmoid(Linear(x, 1)) (same page, Shared
// Expert) is one more dot product of the same token, so it is scored here as column E.
#include <math.h>

#include <atomic>

#include "launch.h"
#include "sm100.cuh"

namespace moe {

constexpr int kRouterTokens = 8;  // tokens per warp in the fused routing kernel's scoring loop

// One warp per token: top-K of the E scores under the total order (score descending, index
// ascending), renormalised weights, and the shared-expert gate.
// Softmax is monotone, so selecting on scores selects on probabilities; the renormalised
// weight p_k / sum_sel p_j equals exp(l_k - l_0) / sum_sel exp(l_j - l_0) (the full
// softmax denominator cancels), which is what is computed.
__global__ void __launch_bounds__(256) k_router_topk(LayerArgs a) {
    grid_dep_wait();  // the scores of the router GEMM
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= a.T) return;
    const float* l = a.logits + (size_t)t * a.ldl;
    uint32_t key[8];
    bool bad = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        key[j] = 0u;
        if (lane + 32 * j < a.E) {
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
    warp_topk(key, a.K, lane, v0, myv, mye);
    // shared-expert gate score: the E router columns came from the tensor-core GEMM, the gate
    // is one more dot product x[t] . ws here (kept in column E for the workspace taps)
    float acc = 0.f;
    for (int c = lane; c < a.H / 8; c += 32) {
        float xf[8];
        unpack8(ld_ro(a.x + (size_t)t * a.H + (size_t)c * 8), xf);
        acc = dot8(ld_ro(a.sg + (size_t)c * 8), xf, acc);
    }
    float z = warp_sum(acc);
    if (lane == 0) a.logits[(size_t)t * a.ldl + a.E] = z;
    z = router_score(z, a.flags);
    const float ex = lane < a.K ? expf(myv - v0) : 0.f;
    const float s = warp_sum(ex);
    if (lane < a.K) {
        a.ids[(size_t)t * a.K + lane] = mye;
        a.topw[(size_t)t * a.K + lane] = ex / s;
    }
    if (lane == 0) {
        if (!isfinite(z)) bad = true;
        a.sgate[t] = 1.0f / (1.0f + expf(-z));
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&a.hdr->err, ERR_NONFINITE_SCORE);
}

// Routing of T >= 256 tokens: router GEMM on the tensor cores, then top-K (fewer tokens are
// routed by the one-cluster or the split router, which cover every supported shape).
cudaError_t launch_router(const LayerArgs& a, cudaStream_t s) {
    if (!a.gemm) return cudaErrorNotSupported;
    cudaError_t e = launch_router_gemm(a, s);
    if (e != cudaSuccess) return e;
    MOE_LAUNCH(MOE_KERNEL_ROUTER_TOPK, s, (e = launch_pdl(k_router_topk, dim3((a.T + 7) / 8), dim3(256), 0, s, a)));
    return e;
}

// RMSNorm, one CTA per token row: fp32 sum of squares in a fixed order, 1/sqrt, scale, bf16.
__global__ void __launch_bounds__(256) k_rmsnorm(const bf16* x, const bf16* gamma, float eps, bf16* xn, int H) {
    __shared__ float wsum[8];
    const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bf16* xr = x + (size_t)t * H;
    float ss = 0.f;
    for (int c = threadIdx.x; c < H / 8; c += 256) {
        float f[8];
        unpack8(ld_ro(xr + (size_t)c * 8), f);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) wsum[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += wsum[w];
    const float r = 1.0f / sqrtf(tot / (float)H + eps);
    for (int c = threadIdx.x; c < H / 8; c += 256) {
        float f[8], g[8];
        unpack8(ld_ro(xr + (size_t)c * 8), f);
        if (gamma) {
            unpack8(ld_ro(gamma + (size_t)c * 8), g);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) g[i] = 1.f;
        }
        uint4 o;
        o.x = pack_bf16x2(f[0] * r * g[0], f[1] * r * g[1]);
        o.y = pack_bf16x2(f[2] * r * g[2], f[3] * r * g[3]);
        o.z = pack_bf16x2(f[4] * r * g[4], f[5] * r * g[5]);
        o.w = pack_bf16x2(f[6] * r * g[6], f[7] * r * g[7]);
        *reinterpret_cast<uint4*>(xn + (size_t)t * H + (size_t)c * 8) = o;
    }
}

cudaError_t launch_rmsnorm(const bf16* x, const bf16* gamma, float eps, bf16* xn, int T, int H, cudaStream_t s) {
    MOE_LAUNCH(MOE_KERNEL_RMSNORM, s, (k_rmsnorm<<<T, 256, 0, s>>>(x, gamma, eps, xn, H)));
    return cudaGetLastError();
}

}  // namespace moe

namespace moe {

// ---------------------------------------------------------------------------------------
// Few-token routing in one launch (T <= kFusedRouteTokens): every CTA scores 8 rows of
// [Wr; ws] for all tokens; the CTA that finishes last (atomic ticket after a fence, so it sees
// every score) runs top-K for all tokens and the dispatch of the T*K pairs, then re-arms the
// ticket. No CTA ever waits on another.

__device__ void topk_one_token(const LayerArgs& a, const float* l, int t, int lane) {
    uint32_t key[8];
    bool bad = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        key[j] = 0u;
        if (lane + 32 * j < a.E) {
            float v = router_score(__ldcg(l + lane + 32 * j), a.flags);
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
        a.ids[(size_t)t * a.K + lane] = mye;
        a.topw[(size_t)t * a.K + lane] = ex / s;
    }
    if (lane == 0) {
        const float z = router_score(__ldcg(l + a.E), a.flags);
        if (!isfinite(z)) bad = true;
        a.sgate[t] = 1.0f / (1.0f + expf(-z));
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&a.hdr->err, ERR_NONFINITE_SCORE);
}

__global__ void __launch_bounds__(256) k_route_fused(LayerArgs a) {
    __shared__ int cnt[256];
    __shared__ int off[257];
    __shared__ int sids[kFusedRouteTokens * 8];
    __shared__ int slr[kFusedRouteTokens * 8];
    __shared__ unsigned ticket;
    // let the expert kernel start its shared-expert work now; its routed work waits for this
    // grid's completion (griddepcontrol.wait)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 1. scores of row r for all tokens
    const int r = blockIdx.x * 8 + warp;
    if (r <= a.E) {
        const bf16* wrow = r < a.E ? a.router_w + (size_t)r * a.H : a.sg;
        const float bias = (r < a.E && a.router_b) ? __bfloat162float(a.router_b[r]) : 0.f;
        for (int t0 = 0; t0 < a.T; t0 += kRouterTokens) {
            const int mt = min(kRouterTokens, a.T - t0);
            float acc[kRouterTokens];
#pragma unroll
            for (int i = 0; i < kRouterTokens; ++i) acc[i] = 0.f;
#pragma unroll 8
            for (int c = lane; c < a.H / 8; c += 32) {
                const uint4 wv = ld_ro(wrow + (size_t)c * 8);
#pragma unroll
                for (int tt = 0; tt < kRouterTokens; ++tt) {
                    if (tt < mt) {
                        float xf[8];
                        unpack8(ld_ro(a.x + (size_t)(t0 + tt) * a.H + (size_t)c * 8), xf);
                        acc[tt] = dot8(wv, xf, acc[tt]);
                    }
                }
            }
#pragma unroll
            for (int tt = 0; tt < kRouterTokens; ++tt) {
                if (tt < mt) {
                    const float s = warp_sum(acc[tt]);
                    if (lane == 0) a.logits[(size_t)(t0 + tt) * a.ldl + r] = s + bias;
                }
            }
        }
    }
    // 2. the last CTA to finish routes every token
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) ticket = atomicAdd(&a.hdr->route_ticket, 1u);
    __syncthreads();
    if (ticket != gridDim.x - 1) return;
    __threadfence();
    for (int t = warp; t < a.T; t += 8) topk_one_token(a, a.logits + (size_t)t * a.ldl, t, lane);
    for (int e = threadIdx.x; e < a.E; e += 256) cnt[e] = 0;
    __syncthreads();
    const int P = (int)a.P;
    for (int i = threadIdx.x; i < P; i += 256) sids[i] = a.ids[i];  // written above by this CTA
    __syncthreads();
    // 3. dispatch: per-expert ranks in token order (one warp, no atomics)
    if (warp == 0) {
        for (int base = 0; base < P; base += 32) {
            const int i = base + lane;
            const bool valid = i < P;
            const int e = valid ? sids[i] : -1;
            const unsigned m = __match_any_sync(0xffffffffu, e);
            const int rank_in = __popc(m & ((1u << lane) - 1u));
            const int c = valid ? cnt[e] : 0;
            __syncwarp();
            if (valid) {
                slr[i] = c + rank_in;
                if (rank_in == 0) cnt[e] = c + __popc(m);
            }
            __syncwarp();
        }
        // exclusive scan of the counts and the list of experts with pairs: lane owns 8 experts
        int loc[8], run = 0, nz = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane * 8 + j;
            loc[j] = e < a.E ? cnt[e] : 0;
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
                off[e] = pos;
                if (loc[j] > 0) a.act[apos++] = e;
            }
            pos += loc[j];
        }
        if (lane == 31) {
            off[a.E] = incl;
            a.hdr->n_act = inz;
            a.hdr->route_ticket = 0;  // re-arm for the next call on this workspace
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e <= a.E; e += 256) {
        a.offsets[e] = off[e];
        if (e < a.E) a.counts[e] = cnt[e];
    }
    for (int i = threadIdx.x; i < P; i += 256) {
        const int j = off[sids[i]] + slr[i];
        a.perm[j] = i;
        a.inv[i] = j;
    }
}

cudaError_t launch_route_fused(const LayerArgs& a, cudaStream_t s) {
    MOE_LAUNCH(MOE_KERNEL_ROUTER_SCORES, s, (k_route_fused<<<(a.E + 1 + 7) / 8, 256, 0, s>>>(a)));
    return cudaGetLastError();
}

}  // namespace moe

namespace moe {

// ---------------------------------------------------------------------------------------
// Few-token routing on one thread-block cluster of NC CTAs, the whole grid (16 where the device
// allows that non-portable size, else 8; T <= 8, H <= 2048, E <= 256).
// CTA c bulk-copies its ~(E+1)/NC rows of [Wr; ws] and the token rows into shared memory (one
// copy per row, rows 16 bytes apart modulo 128 so ldmatrix is conflict-free), scores them with
// warp-level bf16 MMAs (m16n8k16, fp32 accumulate; 16 rows by the tokens, K split over the 8
// warps and summed in a fixed order), and stores the scores straight into CTA 0's shared memory
// (distributed shared memory). After one cluster barrier CTA 0 runs top-K for all tokens and
// the dispatch from its own shared memory and writes the routing to global memory.

constexpr int kRouteCluster = 16;        // cluster size tried first (non-portable)
constexpr int kRouteClusterPortable = 8; // fallback
constexpr int kRouteMaxT = 8;
constexpr int kRoutePad = 16;

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_cluster_f32(uint32_t local_addr, int rank, float v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src), "r"(bytes), "r"((uint32_t)__cvta_generic_to_shared(bar))
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_r(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_r(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void mma16816_r(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

struct RouteSmem {
    __host__ __device__ static int rows(int E, int nc) { return (E + 1 + nc - 1) / nc; }
    __host__ __device__ static int mtiles(int E, int nc) { return (rows(E, nc) + 15) / 16; }
    static size_t bytes(int T, int H, int E, int ldl, int nc) {
        const size_t pitch = (size_t)H * 2 + kRoutePad;
        return 128 + (size_t)(rows(E, nc) + kRouteMaxT) * pitch + (size_t)T * ldl * 4 +
               (size_t)8 * mtiles(E, nc) * 128 * 4 + 64;
    }
};

__global__ void __launch_bounds__(256, 1) k_route_cluster(LayerArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ int cnt[256];
    __shared__ int off[257];
    __shared__ int sids[kRouteMaxT * 8];
    __shared__ int slr[kRouteMaxT * 8];
    __shared__ int sperm[kRouteMaxT * 8];
    __shared__ int sact[256];
    __shared__ uint32_t stoks[256];
    __shared__ int s_nact;
    __shared__ uint64_t bar;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;  // == rank in the (single) cluster
    const int NC = gridDim.x;
    const int R = RouteSmem::rows(a.E, NC), MT = RouteSmem::mtiles(a.E, NC);
    const int r0 = c * R, r1 = min(a.E + 1, r0 + R), nr = max(r1 - r0, 0);
    const int pitch = a.H * 2 + kRoutePad;
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(smem_raw);
    uint8_t* p = smem_raw + (((base + 127u) & ~127u) - base);
    uint8_t* wsm = p;                                   // [R rows][pitch]
    uint8_t* xsm = p + (size_t)R * pitch;               // [kRouteMaxT rows][pitch]
    float* lg = reinterpret_cast<float*>(xsm + (size_t)kRouteMaxT * pitch);  // [T, ldl] (CTA 0)
    float* red = lg + (size_t)a.T * a.ldl;              // [8 warps][MT][32 lanes][4]

    // 1. one bulk copy per row: this CTA's rows of [Wr; ws] (row E is the shared gate), then
    // the token rows. Launched with programmatic serialization, the kernel may start while the
    // previous kernel on the stream is still running: the weight rows go out at once, the
    // token rows (and every workspace access) only after the wait for that kernel.
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bar, (uint32_t)((nr + a.T) * a.H * 2));
    }
    __syncthreads();
    if (warp == 0) {
        for (int i = lane; i < nr; i += 32) {
            const int r = r0 + i;
            bulk_g2s(wsm + (size_t)i * pitch, r < a.E ? a.router_w + (size_t)r * a.H : a.sg, (uint32_t)(a.H * 2), &bar);
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // only now may the next kernel start: it reads x before it waits for this one
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (warp == 0 && lane < a.T)
        bulk_g2s(xsm + (size_t)lane * pitch, a.x + (size_t)lane * a.H, (uint32_t)(a.H * 2), &bar);
    bool ok = mbar_wait(&bar, 0);
    if (!ok) atomicOr(&a.hdr->err, ERR_TIMEOUT);

    // 2. scores: warp w sums K range [w*H/8, (w+1)*H/8) for every 16-row tile and the tokens
    if (ok) {
        const int kw = a.H / 8, k0 = warp * kw;
        const uint32_t wbase = (uint32_t)__cvta_generic_to_shared(wsm);
        const uint32_t xbase = (uint32_t)__cvta_generic_to_shared(xsm);
        const uint32_t b_lane = xbase + (uint32_t)((lane & 7) * pitch + (k0 + 8 * ((lane >> 3) & 1)) * 2);
        for (int mt = 0; mt < MT; ++mt) {
            int row = mt * 16 + (lane & 15);
            row = row < nr ? row : 0;  // rows past this CTA's share read row 0; their results are dropped
            const uint32_t a_lane = wbase + (uint32_t)(row * pitch + (k0 + 8 * (lane >> 4)) * 2);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int k = 0; k < kw / 16; ++k) {
                uint32_t a0, a1, a2, a3, b0, b1;
                ldsm_x4_r(a_lane + k * 32, a0, a1, a2, a3);
                ldsm_x2_r(b_lane + k * 32, b0, b1);
                mma16816_r(d, a0, a1, a2, a3, b0, b1);
            }
            *reinterpret_cast<float4*>(red + ((size_t)(warp * MT + mt) * 32 + lane) * 4) = make_float4(d[0], d[1], d[2], d[3]);
        }
    }
    __syncthreads();
    // fixed-order sum over the 8 warps; lane l of tile mt holds rows mt*16 + l/4 (+8), tokens
    // 2*(l%4) (+1); the score goes to CTA 0's shared memory
    if (ok) {
        for (int idx = threadIdx.x; idx < MT * 32; idx += 256) {
            const int mt = idx >> 5, l = idx & 31;
            float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int w = 0; w < 8; ++w) {
                const float4 v = *reinterpret_cast<const float4*>(red + ((size_t)(w * MT + mt) * 32 + l) * 4);
                s4.x += v.x; s4.y += v.y; s4.z += v.z; s4.w += v.w;
            }
            const float vals[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int rl = mt * 16 + (l >> 2) + (q >= 2 ? 8 : 0);
                const int t = 2 * (l & 3) + (q & 1);
                if (rl < nr && t < a.T) {
                    const int r = r0 + rl;
                    const float bias = (r < a.E && a.router_b) ? __bfloat162float(a.router_b[r]) : 0.f;
                    st_cluster_f32((uint32_t)__cvta_generic_to_shared(lg + (size_t)t * a.ldl + r), 0, vals[q] + bias);
                }
            }
        }
    }
    cluster_sync_all();
    if (c != 0) return;

    // 3. CTA 0: top-K of every token from shared memory, then the dispatch
    for (int t = warp; t < a.T; t += 8) {
        const float* l = lg + (size_t)t * a.ldl;
        uint32_t key[8];
        bool bad = false;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            key[j] = 0u;
            if (lane + 32 * j < a.E) {
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
        warp_topk(key, a.K, lane, v0, myv, mye);
        const float ex = lane < a.K ? expf(myv - v0) : 0.f;
        const float s = warp_sum(ex);
        if (lane < a.K) {
            sids[t * a.K + lane] = mye;
            a.ids[(size_t)t * a.K + lane] = mye;
            a.topw[(size_t)t * a.K + lane] = ex / s;
        }
        if (lane == 0) {
            const float z = router_score(l[a.E], a.flags);
            if (!isfinite(z)) bad = true;
            a.sgate[t] = 1.0f / (1.0f + expf(-z));
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&a.hdr->err, ERR_NONFINITE_SCORE);
    }
    for (int e = threadIdx.x; e < a.E; e += 256) cnt[e] = 0;
    __syncthreads();
    const int P = (int)a.P;
    if (warp == 0) {
        for (int b0 = 0; b0 < P; b0 += 32) {
            const int i = b0 + lane;
            const bool valid = i < P;
            const int e = valid ? sids[i] : -1;
            const unsigned m = __match_any_sync(0xffffffffu, e);
            const int rank_in = __popc(m & ((1u << lane) - 1u));
            const int cc = valid ? cnt[e] : 0;
            __syncwarp();
            if (valid) {
                slr[i] = cc + rank_in;
                if (rank_in == 0) cnt[e] = cc + __popc(m);
            }
            __syncwarp();
        }
        int loc[8], run = 0, nz = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane * 8 + j;
            loc[j] = e < a.E ? cnt[e] : 0;
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
                off[e] = pos;
                if (loc[j] > 0) {
                    sact[apos] = e;
                    a.act[apos++] = e;
                }
            }
            pos += loc[j];
        }
        if (lane == 31) {
            off[a.E] = incl;
            a.hdr->n_act = inz;
            s_nact = inz;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e <= a.E; e += 256) {
        a.offsets[e] = off[e];
        if (e < a.E) a.counts[e] = cnt[e];
    }
    for (int i = threadIdx.x; i < P; i += 256) {
        const int j = off[sids[i]] + slr[i];
        a.perm[j] = i;
        a.inv[i] = j;
        sperm[j] = i;
    }
    if (!a.uprec) return;
    __syncthreads();
    // gate_up work records of the routed experts: expert, first h row, 8 features, tokens.
    // The token list of each used expert once (its pairs' tokens in dispatch order, 4 bits
    // each; T <= 8), then warp w writes the records of experts w, w + 8, ..., lane l those of
    // feature blocks l, l + 32, ...
    const int fbs = a.I / 8, n = s_nact;
    for (int g = threadIdx.x; g < n; g += 256) {
        const int e = sact[g];
        uint32_t toks = 0;
        for (int j = 0; j < cnt[e]; ++j) toks |= (uint32_t)(sperm[off[e] + j] / a.K) << (4 * j);
        stoks[g] = toks;
    }
    __syncthreads();
    for (int g = warp; g < n; g += 8) {
        const int e = sact[g];
        UpRec rec;
        rec.e = e;
        rec.row0 = off[e];
        rec.mt = (int16_t)cnt[e];
        rec.toks = stoks[g];
        for (int fb = lane; fb < fbs; fb += 32) {
            rec.f0 = (int16_t)(fb * 8);
            a.uprec[(size_t)g * fbs + fb] = rec;
        }
    }
    if (threadIdx.x == 0) a.hdr->n_uprec = n * fbs;
}

bool route_cluster_supported(const LayerArgs& a) {
    return a.T >= 1 && a.T <= kRouteMaxT && a.E <= 256 && a.H % 128 == 0 &&
           RouteSmem::bytes(a.T, a.H, a.E, a.ldl, kRouteClusterPortable) <= 200 * 1024;
}

cudaError_t launch_route_cluster(const LayerArgs& a, cudaStream_t s) {
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    // the cluster size this device takes: 16 CTAs (half the rows each) when a cluster of that
    // non-portable size can be resident, else 8
    static int nc_dev[64] = {};
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_route_cluster, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        nc_dev[dev] = kRouteClusterPortable;
        if (cudaFuncSetAttribute(k_route_cluster, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(kRouteCluster);
            q.blockDim = dim3(256);
            q.dynamicSmemBytes = 200 * 1024;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = kRouteCluster;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            q.attrs = qa;
            q.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, k_route_cluster, &q) == cudaSuccess && clusters >= 1)
                nc_dev[dev] = kRouteCluster;
        }
        (void)cudaGetLastError();  // a refused query leaves no error behind
        configured[dev] = true;
    }
    const int nc = nc_dev[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nc);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = RouteSmem::bytes(a.T, a.H, a.E, a.ldl, nc);
    cfg.stream = s;
    // programmatic serialization: the launch and the weight-row copies overlap the end of the
    // previous kernel (the kernel waits for it before it reads x or the workspace). A driver
    // that refuses it together with the cluster gets the cluster launch alone from then on.
    static std::atomic<int> pdl_refused{0};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = nc;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_refused.load() ? 1 : 2;
    cudaError_t e;
    MOE_LAUNCH(MOE_KERNEL_ROUTER_SCORES, s, (e = cudaLaunchKernelEx(&cfg, k_route_cluster, a)));
    if (e != cudaSuccess && cfg.numAttrs == 2 && e != cudaErrorStreamCaptureInvalidated &&
        e != cudaErrorStreamCaptureUnsupported) {
        (void)cudaGetLastError();
        pdl_refused.store(1);
        cfg.numAttrs = 1;
        MOE_LAUNCH(MOE_KERNEL_ROUTER_SCORES, s, (e = cudaLaunchKernelEx(&cfg, k_route_cluster, a)));
    }
    return e;
}

}  // namespace moe
