// experts.cu -- SwiGLU experts over dispatched rows, and the fixed-order combine.
//
// expert_e(x) = SiLU(x . W_gate_e) * (x . W_up_e) . W_down_e ("Qwen3.6-35B-A3B -- Architecture
// Overview", MoE FFN: 256 Experts, Experts), with gate and up merged into one [2I, H] tensor
// per expert (rows [0,I) gate, [I,2I) up). The shared expert has the same structure and is
// treated as one more group whose rows are all T tokens in order (same page, Shared Expert).
//
// Groups: g < n_act is the g-th expert that received pairs (rows offsets[e] .. offsets[e+1]
// of the dispatch order, token = perm[j] / K); g = n_act is the shared expert (rows P .. P+T).
// Only experts that received pairs are read: each expert's weights stream from HBM once per
// 8-token tile (once in total when it has at most 8 rows).
#include "launch.h"

namespace moe {

constexpr int kTile = 8;        // rows (tokens) per register tile
constexpr int kUpFpw = 4;       // gate_up: features per warp (4 gate rows + 4 up rows)
constexpr int kUpFeat = 8 * kUpFpw;
constexpr int kDnRpw = 8;       // down: output rows per warp
constexpr int kDnRows = 8 * kDnRpw;

struct Group {
    const bf16* W;
    int inner, row0, rows;
    bool shared;
};

__device__ __forceinline__ Group routed_group(const LayerArgs& a, int g, const bf16* wbase, size_t wstride) {
    const int e = a.act[g];
    Group G;
    G.W = wbase + (size_t)e * wstride;
    G.inner = a.I;
    G.row0 = a.offsets[e];
    G.rows = a.offsets[e + 1] - G.row0;
    G.shared = false;
    return G;
}

// h[j, f] = bf16( SiLU(x_j . Wg[f]) * (x_j . Wu[f]) ) for the rows j of a group.
// Work item = (group, 32 features); each warp owns 4 features and streams their 8 weight
// rows once per 8-row tile, with every lane taking 16-byte chunks of H.
__global__ void __launch_bounds__(256) k_gate_up(LayerArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_act = a.hdr->n_act;
    const int ipr = a.I / kUpFeat, ips = a.Is / kUpFeat;
    const int items = n_act * ipr + ips;
    const int nchunk = a.H / 8;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        Group G;
        int fb;
        if (it >= n_act * ipr) {
            fb = it - n_act * ipr;
            G = {a.sgu, a.Is, (int)a.P, a.T, true};
        } else {
            const int g = it / ipr;
            fb = it - g * ipr;
            G = routed_group(a, g, a.gate_up, (size_t)2 * a.I * a.H);
        }
        const int f0 = fb * kUpFeat + warp * kUpFpw;
        const bf16* wg = G.W + (size_t)f0 * a.H;
        const bf16* wu = G.W + (size_t)(G.inner + f0) * a.H;
        for (int r0 = 0; r0 < G.rows; r0 += kTile) {
            const int mt = min(kTile, G.rows - r0);
            const bf16* xr[kTile];
#pragma unroll
            for (int tt = 0; tt < kTile; ++tt) {
                const int j = G.row0 + r0 + min(tt, mt - 1);
                const int t = G.shared ? j - (int)a.P : a.perm[j] / a.K;
                xr[tt] = a.x + (size_t)t * a.H;
            }
            float acc[2 * kUpFpw][kTile];
#pragma unroll
            for (int r = 0; r < 2 * kUpFpw; ++r)
#pragma unroll
                for (int tt = 0; tt < kTile; ++tt) acc[r][tt] = 0.f;
            for (int c = lane; c < nchunk; c += 32) {
                uint4 w[2 * kUpFpw];
#pragma unroll
                for (int r = 0; r < kUpFpw; ++r) {
                    w[r] = ld_stream(wg + (size_t)r * a.H + (size_t)c * 8);
                    w[kUpFpw + r] = ld_stream(wu + (size_t)r * a.H + (size_t)c * 8);
                }
#pragma unroll
                for (int tt = 0; tt < kTile; ++tt) {
                    if (tt < mt) {
                        float xf[8];
                        unpack8(ld_ro(xr[tt] + (size_t)c * 8), xf);
#pragma unroll
                        for (int r = 0; r < 2 * kUpFpw; ++r) acc[r][tt] = dot8(w[r], xf, acc[r][tt]);
                    }
                }
            }
#pragma unroll
            for (int tt = 0; tt < kTile; ++tt)
                if (tt < mt)
#pragma unroll
                    for (int r = 0; r < 2 * kUpFpw; ++r) acc[r][tt] = warp_sum(acc[r][tt]);
            // lane = f * 8 + tt writes one activation
#pragma unroll
            for (int f = 0; f < kUpFpw; ++f)
#pragma unroll
                for (int tt = 0; tt < kTile; ++tt)
                    if (lane == f * kTile + tt && tt < mt) {
                        const float hv = silu(acc[f][tt]) * acc[kUpFpw + f][tt];
                        a.h[(size_t)(G.row0 + r0 + tt) * a.Imax + f0 + f] = __float2bfloat16_rn(hv);
                    }
        }
    }
}

// Y[t, slot, o] = scale * (h_j . Wd[o]) for the rows j of a group: scale = topw[t, slot]
// for a routed pair, sigmoid gate sgate[t] with slot K for the shared expert. Work item =
// (group, 64 output rows); each warp owns 8 rows of Wd.
__global__ void __launch_bounds__(256) k_down(LayerArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_act = a.hdr->n_act;
    const int nob = a.H / kDnRows;
    const int items = (n_act + 1) * nob;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const int g = it / nob, ob = it - g * nob;
        Group G;
        if (g == n_act)
            G = {a.sd, a.Is, (int)a.P, a.T, true};
        else
            G = routed_group(a, g, a.down, (size_t)a.H * a.I);
        const int o0 = ob * kDnRows + warp * kDnRpw;
        const bf16* wr = G.W + (size_t)o0 * G.inner;
        const int nch = G.inner / 8;
        for (int r0 = 0; r0 < G.rows; r0 += kTile) {
            const int mt = min(kTile, G.rows - r0);
            int tok[kTile], slot[kTile];
            float sc[kTile];
#pragma unroll
            for (int tt = 0; tt < kTile; ++tt) {
                const int j = G.row0 + r0 + min(tt, mt - 1);
                if (G.shared) {
                    tok[tt] = j - (int)a.P;
                    slot[tt] = a.K;
                    sc[tt] = a.sgate[tok[tt]];
                } else {
                    const int pv = a.perm[j];
                    tok[tt] = pv / a.K;
                    slot[tt] = pv - tok[tt] * a.K;
                    sc[tt] = a.topw[pv];
                }
            }
            float acc[kDnRpw][kTile];
#pragma unroll
            for (int r = 0; r < kDnRpw; ++r)
#pragma unroll
                for (int tt = 0; tt < kTile; ++tt) acc[r][tt] = 0.f;
            for (int c = lane; c < nch; c += 32) {
                uint4 w[kDnRpw];
#pragma unroll
                for (int r = 0; r < kDnRpw; ++r) w[r] = ld_stream(wr + (size_t)r * G.inner + (size_t)c * 8);
#pragma unroll
                for (int tt = 0; tt < kTile; ++tt) {
                    if (tt < mt) {
                        float hf[8];
                        unpack8(ld_ro(a.h + (size_t)(G.row0 + r0 + tt) * a.Imax + (size_t)c * 8), hf);
#pragma unroll
                        for (int r = 0; r < kDnRpw; ++r) acc[r][tt] = dot8(w[r], hf, acc[r][tt]);
                    }
                }
            }
#pragma unroll
            for (int tt = 0; tt < kTile; ++tt)
                if (tt < mt)
#pragma unroll
                    for (int r = 0; r < kDnRpw; ++r) acc[r][tt] = warp_sum(acc[r][tt]);
#pragma unroll
            for (int r = 0; r < kDnRpw; ++r)
#pragma unroll
                for (int tt = 0; tt < kTile; ++tt)
                    if (lane == ((r * kTile + tt) & 31) && tt < mt)
                        a.Y[((size_t)tok[tt] * (a.K + 1) + slot[tt]) * a.H + o0 + r] = sc[tt] * acc[r][tt];
        }
    }
}

// out[t, o] = bf16( residual[t, o] + Y[t, K, o] + Y[t, 0, o] + ... + Y[t, K-1, o] ), summed in
// fp32 in exactly this order ("RMSNorm -> MoE FFN -> +residual", "Qwen3.6-35B-A3B --
// Architecture Overview", Stage 2).
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const bf16* p) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    return make_float4(bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y));
}

constexpr int kMaxCombineK = 8;  // slots per token the 8-wide combine keeps in registers

template <typename YT>
__global__ void __launch_bounds__(256) k_combine(LayerArgs a, const YT* Y) {
    // no-op unless launched as a programmatic dependent: then wait for the producer of Y
    grid_dep_wait();
    grid_dep_launch();
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    const int q = a.H / 4;
    if (i >= (int64_t)a.T * q) return;
    const int t = (int)(i / q), o = (int)(i - (int64_t)t * q) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.residual) acc = load4(a.residual + (size_t)t * a.H + o);
    const YT* yt = Y + (size_t)t * (a.K + 1) * a.H + o;
    float4 v = load4(yt + (size_t)a.K * a.H);
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    for (int k = 0; k < a.K; ++k) {
        v = load4(yt + (size_t)k * a.H);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    uint2 ov;
    ov.x = pack_bf16x2(acc.x, acc.y);
    ov.y = pack_bf16x2(acc.z, acc.w);
    *reinterpret_cast<uint2*>(a.out + (size_t)t * a.H + o) = ov;
}

// The bf16-Y combine with 8 outputs per thread: 16-byte loads of each of the K + 1 slot rows
// (twice the bytes in flight per thread), the same per-element order of additions.
__global__ void __launch_bounds__(256) k_combine_bf16x8(LayerArgs a, const bf16* Y) {
    grid_dep_wait();
    grid_dep_launch();
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    const int q = a.H / 8;
    if (i >= (int64_t)a.T * q) return;
    const int t = (int)(i / q), o = (int)(i - (int64_t)t * q) * 8;
    float acc[8];
    if (a.residual) {
        unpack8(ld_ro(a.residual + (size_t)t * a.H + o), acc);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    }
    const bf16* yt = Y + (size_t)t * (a.K + 1) * a.H + o;
    uint4 w[kMaxCombineK + 1];
    const int nk = a.K + 1;
#pragma unroll
    for (int k = 0; k < kMaxCombineK + 1; ++k)
        if (k < nk) w[k] = ld_ro(yt + (size_t)(k == 0 ? a.K : k - 1) * a.H);  // the shared slot first
#pragma unroll
    for (int k = 0; k < kMaxCombineK + 1; ++k)
        if (k < nk) {
            float v[8];
            unpack8(w[k], v);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] += v[e];
        }
    uint4 ov;
    ov.x = pack_bf16x2(acc[0], acc[1]);
    ov.y = pack_bf16x2(acc[2], acc[3]);
    ov.z = pack_bf16x2(acc[4], acc[5]);
    ov.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(a.out + (size_t)t * a.H + o) = ov;
}

cudaError_t launch_experts(const LayerArgs& a, cudaStream_t s) {
    const int up_items = a.E * (a.I / kUpFeat) + a.Is / kUpFeat;
    const int dn_items = (a.E + 1) * (a.H / kDnRows);
    const int cap = 4 * a.num_sms;
    MOE_LAUNCH(MOE_KERNEL_GATE_UP, s, (k_gate_up<<<min(up_items, cap), 256, 0, s>>>(a)));
    MOE_LAUNCH(MOE_KERNEL_DOWN, s, (k_down<<<min(dn_items, cap), 256, 0, s>>>(a)));
    return cudaGetLastError();
}

// The combine as a programmatic dependent launch of the preceding kernel (fp32 Y).
cudaError_t launch_combine_pdl(const LayerArgs& a, cudaStream_t s) {
    const int64_t nq = (int64_t)a.T * (a.H / 4);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((nq + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    const float* Y = a.Y;
    MOE_LAUNCH(MOE_KERNEL_COMBINE, s, (e = cudaLaunchKernelEx(&cfg, k_combine<float>, a, Y)));
    return e;
}

cudaError_t launch_combine(const LayerArgs& a, cudaStream_t s) {
    const int64_t nq = (int64_t)a.T * (a.H / 4);
    const unsigned grid = (unsigned)((nq + 255) / 256);
    cudaError_t e;
    if (a.gemm && a.H % 8 == 0 && a.K <= kMaxCombineK) {
        const bf16* Y = a.Yb;
        const unsigned grid8 = (unsigned)(((int64_t)a.T * (a.H / 8) + 255) / 256);
        MOE_LAUNCH(MOE_KERNEL_COMBINE, s, (e = launch_pdl(k_combine_bf16x8, dim3(grid8), dim3(256), 0, s, a, Y)));
    } else if (a.gemm) {
        const bf16* Y = a.Yb;
        MOE_LAUNCH(MOE_KERNEL_COMBINE, s, (e = launch_pdl(k_combine<bf16>, dim3(grid), dim3(256), 0, s, a, Y)));
    } else {
        MOE_LAUNCH(MOE_KERNEL_COMBINE, s, (k_combine<float><<<grid, 256, 0, s>>>(a, a.Y)));
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace moe
