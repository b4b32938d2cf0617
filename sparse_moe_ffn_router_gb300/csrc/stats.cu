// stats.cu -- load-balancing statistics of the routing ("Qwen3.6-35B-A3B -- Architecture
// Overview", MoE FFN: 256 Experts, Load Balancing: an auxiliary loss with coefficient 0.001
// penalises uneven expert utilisation across the batch). The page gives no formula; these
// kernels compute the two per-expert quantities such a loss is built from and the product
// form that is smallest under uniform routing:
//   P_e  = (1/T) sum_t softmax(l_t)_e     mean router probability (full softmax of E scores)
//   f_e  = count_e / (T K)                share of the T*K (token, slot) assignments
//   loss = 0.001 * E * sum_e f_e P_e
// k_stats_partial: one CTA per block of 64 tokens. Warp w takes tokens t0+w, t0+w+8, ... in
//   order and adds each token's softmax row into its registers (experts l, l+32, ... in lane
//   l); the CTA adds its warps' sums in warp order and counts its tokens' assignments.
// k_stats_final: one CTA adds the blocks' partial sums in block order, divides, and sums the
//   loss terms in a fixed tree order. Every sum has a fixed order, so repeated calls agree bit
//   for bit.
#include <math.h>

#include "launch.h"

namespace moe {

constexpr int kStTok = 64;  // tokens per partial block

__global__ void __launch_bounds__(256) k_stats_partial(LayerArgs a, float* part_p, int* part_c) {
    __shared__ float wsum[8][256];
    __shared__ int cnt[256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * kStTok, t1 = min(a.T, t0 + kStTok);
    for (int e = threadIdx.x; e < 256; e += 256) cnt[e] = 0;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    for (int t = t0 + warp; t < t1; t += 8) {
        const float* l = a.logits + (size_t)t * a.ldl;
        float v[8], m = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane + 32 * j;
            v[j] = -INFINITY;
            if (e < a.E) {
                const float s = router_score(l[e], a.flags);
                v[j] = isfinite(s) ? s : -INFINITY;
            }
            m = fmaxf(m, v[j]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float ex[8], s = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            ex[j] = lane + 32 * j < a.E ? expf(v[j] - m) : 0.f;
            s += ex[j];
        }
        s = warp_sum(s);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] += ex[j] / s;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) wsum[warp][lane + 32 * j] = acc[j];
    __syncthreads();
    for (int p = t0 * a.K + threadIdx.x; p < t1 * a.K; p += 256) atomicAdd(&cnt[a.ids[p]], 1);
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += 256) {
        float s = 0.f;
        for (int w = 0; w < 8; ++w) s += wsum[w][e];
        part_p[(size_t)blockIdx.x * a.E + e] = s;
        part_c[(size_t)blockIdx.x * a.E + e] = cnt[e];
    }
}

__global__ void __launch_bounds__(256) k_stats_final(LayerArgs a, const float* part_p, const int* part_c, int nb,
                                                     float* P, float* f, float* loss) {
    __shared__ float term[256];
    const int e = threadIdx.x;
    float t = 0.f;
    if (e < a.E) {
        float sp = 0.f;
        int c = 0;
        for (int b = 0; b < nb; ++b) {
            sp += part_p[(size_t)b * a.E + e];
            c += part_c[(size_t)b * a.E + e];
        }
        const float pe = sp / (float)a.T;
        const float fe = (float)c / (float)((long long)a.T * a.K);
        P[e] = pe;
        f[e] = fe;
        t = fe * pe;
    }
    term[e] = t;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (e < o) term[e] += term[e + o];
        __syncthreads();
    }
    if (e == 0) *loss = 0.001f * (float)a.E * term[0];
}

// Scratch: the slot-output region of the workspace (unused by a statistics call) holds the
// per-block partial sums and counts.
cudaError_t launch_router_stats(const LayerArgs& a, float* P, float* f, float* loss, cudaStream_t s) {
    const int nb = (a.T + kStTok - 1) / kStTok;
    float* part_p = reinterpret_cast<float*>(a.Y);
    int* part_c = reinterpret_cast<int*>(part_p + (size_t)nb * a.E);
    MOE_LAUNCH(MOE_KERNEL_ROUTER_STATS, s, (k_stats_partial<<<nb, 256, 0, s>>>(a, part_p, part_c)));
    MOE_LAUNCH(MOE_KERNEL_ROUTER_STATS, s, (k_stats_final<<<1, 256, 0, s>>>(a, part_p, part_c, nb, P, f, loss)));
    return cudaGetLastError();
}

}  // namespace moe
