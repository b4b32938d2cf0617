// stats.cu -- load-balancing statistics of the routing ("Qwen3.6-35B-A3B -- Architecture
// Overview", MoE FFN: 256 Experts, Load Balancing: an auxiliary loss with coefficient 0.001
// penalises uneven expert utilisation across the batch). The page gives no formula; these
// kernels compute the two per-expert quantities such a loss is built from and the product
// form that is smallest under uniform routing:
//   P_e  = (1/T) sum_t softmax(l_t)_e     mean router probability (full softmax of E scores)
//   f_e  = count_e / (T K)                share of the T*K (token, slot) assignments
//   loss = 0.001 * E * sum_e f_e P_e
// k_stats_partial: one CTA of 1024 threads per block of 32 tokens, one token per warp: the warp
//   turns its token's E scores into the full softmax row (experts l, l+32, ... in lane l) and
//   leaves it in shared memory; thread e then adds the 32 rows of expert e in token order, and
//   the CTA counts its tokens' assignments.
// k_stats_final: 4 threads per expert add the blocks' partial sums, each a contiguous quarter
//   of the blocks in block order, then the quarters in order; P = sum / T, f = count / (T K),
//   and the loss terms are summed in a fixed tree order. Every sum has a fixed order, so
//   repeated calls agree bit for bit.
#include <math.h>

#include "launch.h"

namespace moe {

constexpr int kStTok = kStatsTokens;  // tokens per partial block, one per warp
constexpr int kStThreads = 1024;
constexpr int kStParts = 4;     // threads per expert in the final sum

__global__ void __launch_bounds__(kStThreads) k_stats_partial(LayerArgs a, float* part_p, int* part_c) {
    __shared__ float prob[kStTok][256];
    __shared__ int cnt[256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * kStTok, t = t0 + warp;
    if (threadIdx.x < 256) cnt[threadIdx.x] = 0;
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = -INFINITY;
    if (t < a.T) {
        const float* l = a.logits + (size_t)t * a.ldl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane + 32 * j;
            if (e < a.E) {
                const float s = router_score(l[e], a.flags);
                v[j] = isfinite(s) ? s : -INFINITY;
            }
        }
    }
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, v[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float ex[8], s = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        ex[j] = (t < a.T && lane + 32 * j < a.E) ? expf(v[j] - m) : 0.f;
        s += ex[j];
    }
    s = warp_sum(s);
#pragma unroll
    for (int j = 0; j < 8; ++j) prob[warp][lane + 32 * j] = t < a.T ? ex[j] / s : 0.f;
    __syncthreads();
    const int t1 = min(a.T, t0 + kStTok);
    for (int p = t0 * a.K + threadIdx.x; p < t1 * a.K; p += kStThreads) atomicAdd(&cnt[a.ids[p]], 1);
    float sum = 0.f;
    if (threadIdx.x < a.E)
        for (int w = 0; w < kStTok; ++w) sum += prob[w][threadIdx.x];
    __syncthreads();
    if (threadIdx.x < a.E) {
        part_p[(size_t)blockIdx.x * a.E + threadIdx.x] = sum;
        part_c[(size_t)blockIdx.x * a.E + threadIdx.x] = cnt[threadIdx.x];
    }
}

__global__ void __launch_bounds__(256 * kStParts) k_stats_final(LayerArgs a, const float* part_p, const int* part_c,
                                                                int nb, float* P, float* f, float* loss) {
    __shared__ float qp[kStParts][256];
    __shared__ int qc[kStParts][256];
    __shared__ float term[256];
    const int e = threadIdx.x & 255, q = threadIdx.x >> 8;
    const int b0 = q * nb / kStParts, b1 = (q + 1) * nb / kStParts;
    float sp = 0.f;
    int c = 0;
    if (e < a.E) {
#pragma unroll 8
        for (int b = b0; b < b1; ++b) {
            sp += part_p[(size_t)b * a.E + e];
            c += part_c[(size_t)b * a.E + e];
        }
    }
    qp[q][e] = sp;
    qc[q][e] = c;
    __syncthreads();
    if (q == 0) {
        float t = 0.f;
        if (e < a.E) {
            float tp = 0.f;
            int tc = 0;
            for (int r = 0; r < kStParts; ++r) {
                tp += qp[r][e];
                tc += qc[r][e];
            }
            const float pe = tp / (float)a.T;
            const float fe = (float)tc / (float)((long long)a.T * a.K);
            P[e] = pe;
            f[e] = fe;
            t = fe * pe;
        }
        term[e] = t;
    }
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) term[threadIdx.x] += term[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) *loss = 0.001f * (float)a.E * term[0];
}

// Scratch: the slot-output region of the workspace (unused by a statistics call, and sized
// by the workspace plan for these partial sums too) holds the per-block sums and counts.
cudaError_t launch_router_stats(const LayerArgs& a, float* P, float* f, float* loss, cudaStream_t s) {
    const int nb = (a.T + kStTok - 1) / kStTok;
    float* part_p = reinterpret_cast<float*>(a.Y);
    int* part_c = reinterpret_cast<int*>(part_p + (size_t)nb * a.E);
    MOE_LAUNCH(MOE_KERNEL_ROUTER_STATS, s, (k_stats_partial<<<nb, kStThreads, 0, s>>>(a, part_p, part_c)));
    MOE_LAUNCH(MOE_KERNEL_ROUTER_STATS, s,
               (k_stats_final<<<1, 256 * kStParts, 0, s>>>(a, part_p, part_c, nb, P, f, loss)));
    return cudaGetLastError();
}

}  // namespace moe
