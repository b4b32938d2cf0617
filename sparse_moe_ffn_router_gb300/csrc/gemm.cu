// gemm.cu -- grouped bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA) for
// the many-token regime of the MoE layer.
//
// D[rows of a group, N tile] = A[rows, K] . B[N tile, K]^T, A = token rows (activations),
// B = weight rows ([Out, In] storage, "Qwen3.6 35B-A3B", Blocks: Linear), both K-major.
// Three uses, each with its own epilogue on the fp32 accumulator in TMEM:
//   kLogits  router scores, x . Wr^T (+ br), stored fp32 ("Qwen3.6-35B-A3B -- Architecture
//            Overview", MoE FFN: 256 Experts, Router);
//   kSwiGLU  expert gate/up: the B tile holds FH gate rows then the FH matching up rows of
//            the merged [2I, H] tensor, so one accumulator row holds g and u of the same
//            features and h = SiLU(g) * u is formed in registers (same page, Experts);
//   kScaleY  expert down: y = h . Wd^T scaled by the pair's routing weight (or the shared
//            expert's sigmoid gate) and written to the pair's slot of Y for the fixed-order
//            combine.
//
// One persistent CTA per SM walks the tile list (group-major, then N tile, then M tile, so
// the M tiles that share a weight tile run back to back and reuse it from L2). Roles:
//   warp 0    TMA producer (one lane): A and B tiles into a 4-stage shared-memory ring;
//   warp 1    TMEM owner and MMA issuer (one lane): 128 x BN x 16 tcgen05.mma steps into one
//             of two TMEM accumulators, tcgen05.commit frees ring stages / publishes tiles;
//   warps 2-5 epilogue: tcgen05.ld of the accumulator (warp w reads lanes 32*(w%4)..+31;
//             down has eight epilogue warps, 2-9, two per lane quadrant, each half the columns);
//   warps 6-13 (gate_up only) A gatherers: a routed expert's A rows are token rows of x, row
//             perm[j] / K for dispatch position j. Each k-block's 128-byte segment of a row is
//             copied by 8 lanes, 16 bytes each with cp.async (a warp instruction moves 4 rows;
//             eight warps keep enough of these row loads in flight: with two the GEMM ran
//             ~8 us longer per prefill layer),
//             straight from x into the A stage, in the 128-byte swizzled layout the tensor map
//             would give (16-byte chunk c of row r at r * 128 + (c ^ (r % 8)) * 16); rows past
//             the group's end are zero-filled. x rows are kept in L2 (evict-last) across the K
//             experts that read them, and no dispatched copy of x is written or read. The
//             shared expert's A rows are x itself, loaded by TMA.
#include "launch.h"
#include "sm100.cuh"

namespace moe {

constexpr int kBM = 128, kBK = 64;
constexpr int kGatherWarps = 8;
// epilogue warps: the down GEMM's short mainloop (K = I) leaves less time to write a tile out,
// so it has two per TMEM lane quadrant, each taking half of the tile's columns
template <int EPI>
constexpr int epi_warps() { return EPI == 2 ? 8 : 4; }
template <int EPI>
constexpr int gemm_threads() { return 64 + 32 * epi_warps<EPI>() + (EPI == 1 ? 32 * kGatherWarps : 0); }
constexpr uint32_t kAStage = kBM * kBK * 2;

enum { kLogits = 0, kSwiGLU = 1, kScaleY = 2 };

// Ring stages: as many as keep about 192 KB of A and B tiles in flight per SM.
template <int BN>
struct GemmSmem {
    static constexpr uint32_t kBStage = BN * kBK * 2;
    static constexpr int kStages = (int)((192u * 1024u) / (kAStage + kBStage));
    static constexpr uint32_t kTiles = kStages * (kAStage + kBStage);
    static constexpr uint32_t kScratch = 8 * 2048;  // epilogue: per warp 32 rows x 64 bytes
    static constexpr uint32_t kBytes = 1024 + kTiles + 256 + kScratch;  // alignment slack + tiles + barriers
    // full, empty and gathered-A barriers per stage, two accumulators' full and empty, the
    // MMA-done barrier, the TMEM address and the abort flag
    static_assert((3 * kStages + 5) * 8 + 8 <= 256, "barrier area");
};

__device__ __forceinline__ void flag_timeout(uint32_t* err, volatile int* abort_flag) {
    atomicOr(err, ERR_TIMEOUT);
    *abort_flag = 1;
}

struct TileInfo {
    int g, m0, n_idx, rows, a_row, src, kb;
};

// Locate tile t (tiles are visited in increasing order, so the group cursor only advances).
__device__ __forceinline__ bool find_tile(const GemmPlan& p, int t, int& g, TileInfo& ti) {
    const int ng = p.dense_rows > 0 ? 1 : *p.n_groups;
    if (p.dense_rows > 0) {
        g = 0;
    } else {
        while (g < ng && t >= p.tile_start[g + 1]) ++g;
        if (g >= ng) return false;
    }
    const GemmGroup G = p.dense_rows > 0 ? GemmGroup{0, p.dense_rows, 0, 0, 0} : p.groups[g];
    const int start = p.dense_rows > 0 ? 0 : p.tile_start[g];
    const int mt = (G.rows + kBM - 1) / kBM;
    const int local = t - start;
    ti.g = g;
    ti.n_idx = local / mt;
    ti.m0 = (local - ti.n_idx * mt) * kBM;
    ti.rows = G.rows;
    ti.a_row = G.a_row0;
    ti.src = G.src;
    ti.kb = (G.src ? p.k_shared : p.k_routed) / kBK;
    return true;
}

template <int EPI, int BN>
__global__ void __launch_bounds__(gemm_threads<EPI>(), 1)
    k_gemm(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
           const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1, const GemmPlan p,
           const LayerArgs a) {
    constexpr int kStages = GemmSmem<BN>::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * kAStage;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + GemmSmem<BN>::kTiles);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* accf = bars + 2 * kStages;
    uint64_t* acce = accf + 2;
    uint64_t* mma_done = acce + 2;
    uint64_t* fullA = mma_done + 1;  // gathered A stages (gate_up)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fullA + kStages);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint8_t* epi_scratch = smem + GemmSmem<BN>::kTiles + 256;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], epi_warps<EPI>());
        }
        mbar_init(mma_done, 1);
        if (EPI == kSwiGLU)
            for (int s = 0; s < kStages; ++s) mbar_init(&fullA[s], 32 * kGatherWarps);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA0);
        tma_prefetch_desc(&tmA1);
        tma_prefetch_desc(&tmB0);
        tma_prefetch_desc(&tmB1);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 2 * BN <= 256 ? 256 : 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the set-up above overlaps the previous kernel's tail; the tables, token rows and h it
    // reads are that kernel's (or an earlier one's) outputs
    grid_dep_wait();
    grid_dep_launch();
    const int total = p.dense_rows > 0 ? p.dense_tiles : p.tile_start[*p.n_groups];

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        int g = 0, it = 0;
        uint32_t last_par[kStages];
        bool issued[kStages];
        for (int s = 0; s < kStages; ++s) issued[s] = false;
        for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
            TileInfo ti;
            if (!find_tile(p, t, g, ti)) break;
            const CUtensorMap* mA = ti.src ? &tmA1 : &tmA0;
            const CUtensorMap* mB = ti.src ? &tmB1 : &tmB0;
            const GemmGroup G = p.dense_rows > 0 ? GemmGroup{0, p.dense_rows, 0, 0, 0} : p.groups[ti.g];
            for (int kb = 0; kb < ti.kb; ++kb, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                if (!mbar_wait(&empty[s], ph ^ 1u)) {
                    flag_timeout(p.err, abort_flag);
                    break;
                }
                const bool gathered = EPI == kSwiGLU && !ti.src;  // A comes from the gatherers
                mbar_arrive_expect_tx(&full[s], (gathered ? 0u : kAStage) + GemmSmem<BN>::kBStage);
                if (!gathered) tma_load_2d(sA + s * kAStage, mA, &full[s], kb * kBK, ti.a_row + ti.m0);
                if (EPI == kSwiGLU) {
                    const int fh = BN / 2;
                    const int half = ti.src ? p.up_off_shared : p.up_off_routed;
                    tma_load_2d(sB + s * GemmSmem<BN>::kBStage, mB, &full[s], kb * kBK, G.b_row0 + ti.n_idx * fh);
                    tma_load_2d(sB + s * GemmSmem<BN>::kBStage + fh * kBK * 2, mB, &full[s], kb * kBK,
                                G.b_row0 + half + ti.n_idx * fh);
                } else {
                    tma_load_2d(sB + s * GemmSmem<BN>::kBStage, mB, &full[s], kb * kBK, G.b_row0 + ti.n_idx * BN);
                }
                issued[s] = true;
                last_par[s] = ph;
            }
        }
        // every copy this CTA issued must land before shared memory is released
        for (int s = 0; s < kStages; ++s)
            if (issued[s] && !mbar_wait(&full[s], last_par[s])) flag_timeout(p.err, abort_flag);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
        int g = 0, it = 0, local = 0;
        for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x, ++local) {
            TileInfo ti;
            if (!find_tile(p, t, g, ti)) break;
            const int b = local & 1;
            const uint32_t use = (uint32_t)(local >> 1) & 1u;
            if (!mbar_wait(&acce[b], use ^ 1u)) {
                flag_timeout(p.err, abort_flag);
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(b * BN);
            bool ok = true;
            for (int kb = 0; kb < ti.kb; ++kb, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                if (!mbar_wait(&full[s], ph) || (EPI == kSwiGLU && !mbar_wait(&fullA[s], ph))) {
                    flag_timeout(p.err, abort_flag);
                    ok = false;
                    break;
                }
                // the gathered rows were written through the generic proxy; the tensor cores
                // read them through the async proxy
                if (EPI == kSwiGLU) fence_proxy_async_smem();
                tc_fence_after();
                const uint32_t a_addr = smem_u32(sA + s * kAStage);
                const uint32_t b_addr = smem_u32(sB + s * GemmSmem<BN>::kBStage);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    mma_bf16(d, sdesc_kmajor_sw128(a_addr + kk * 32), sdesc_kmajor_sw128(b_addr + kk * 32), idesc,
                             (kb | kk) != 0);
                mma_commit(&empty[s]);
            }
            if (!ok) break;
            mma_commit(&accf[b]);
        }
        mma_commit(mma_done);
        if (!mbar_wait(mma_done, 0)) flag_timeout(p.err, abort_flag);
    } else if (EPI == kSwiGLU && warp >= 2 + epi_warps<EPI>()) {
        // ---------------- A gatherers: gatherer warp w takes rows (128 / kGatherWarps) w +
        // lane / 8 + 4 i, i < kRows, chunk lane % 8 of each
        constexpr int kRows = kBM / (4 * kGatherWarps);  // rows per lane
        const int r0 = (warp - 2 - epi_warps<EPI>()) * (kBM / kGatherWarps) + (lane >> 3);
        const uint32_t c = (uint32_t)(lane & 7);
        const uint64_t pol_a = l2_evict_last();  // each token row is read by K experts
        int g = 0, it = 0;
        for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
            TileInfo ti;
            if (!find_tile(p, t, g, ti)) break;
            const bf16* src[kRows];
            uint32_t live = 0;
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
                const int m = ti.m0 + r0 + 4 * i;
                src[i] = a.x + c * 8;
                if (!ti.src && m < ti.rows) {
                    src[i] += (size_t)(a.perm[ti.a_row + m] / a.K) * a.H;
                    live |= 1u << i;
                }
            }
            bool ok = true;
            for (int kb = 0; kb < ti.kb; ++kb, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                // lane 0 waits for the stage to be free, the warp follows its verdict
                bool fr = lane == 0 ? mbar_wait(&empty[s], ph ^ 1u) : true;
                fr = __shfl_sync(0xffffffffu, fr, 0);
                if (!fr) {
                    if (lane == 0) flag_timeout(p.err, abort_flag);
                    ok = false;
                    break;
                }
                if (!ti.src) {
                    const uint32_t st = smem_u32(sA + s * kAStage);
#pragma unroll
                    for (int i = 0; i < kRows; ++i) {
                        const uint32_t r = (uint32_t)(r0 + 4 * i);
                        cp_async16(st + r * 128u + ((c ^ (r & 7u)) << 4), src[i] + kb * kBK, ((live >> i) & 1u) * 16u,
                                   pol_a);
                    }
                    cp_async_arrive(&fullA[s]);
                } else {
                    mbar_arrive(&fullA[s]);  // the shared expert's A stage comes by TMA
                }
            }
            if (!ok) break;
        }
        cp_async_wait_all();  // no copy of this CTA may still be in flight when it exits
    } else if (warp >= 2 && warp < 2 + epi_warps<EPI>()) {
        // ---------------- epilogue: TMEM lanes 32*(warp%4) .. +31, one accumulator row each
        const int q = warp & 3;
        const int r = q * 32 + lane;
        int g = 0, local = 0;
        for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x, ++local) {
            TileInfo ti;
            if (!find_tile(p, t, g, ti)) break;
            const int b = local & 1;
            const uint32_t use = (uint32_t)(local >> 1) & 1u;
            const int m = ti.m0 + r;  // row inside the group
            const bool live = m < ti.rows;
            // down: the row's token, slot and scale, read before the accumulator wait so that
            // their latency hides behind it
            int tok = 0, slot = 0;
            float sc = 0.f;
            if (EPI == kScaleY && live) {
                if (ti.src) {
                    tok = m;
                    slot = a.K;
                    sc = a.sgate[tok];
                } else {
                    const int pv = a.perm[ti.a_row + m];
                    tok = pv / a.K;
                    slot = pv - tok * a.K;
                    sc = a.topw[pv];
                }
            }
            // lane 0 waits, the warp follows its verdict (tcgen05.ld needs the whole warp)
            bool ready = lane == 0 ? mbar_wait(&accf[b], use) : true;
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready) {
                if (lane == 0) flag_timeout(p.err, abort_flag);
                break;
            }
            __syncwarp();
            tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN);
            if (EPI == kLogits) {
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tbase + c * 32, v);
                    tmem_ld_wait();
                    const int col0 = ti.n_idx * BN + c * 32;
                    if (live) {
                        float* dst = a.logits + (size_t)(ti.a_row + m) * a.ldl + col0;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int col = col0 + j;
                            if (col < a.E) {
                                float s = __uint_as_float(v[j]);
                                if (a.router_b) s += __bfloat162float(a.router_b[col]);
                                dst[j] = s;
                            }
                        }
                    }
                }
            } else if (EPI == kSwiGLU) {
                constexpr int FH = BN / 2;
                const GemmGroup G = p.groups[ti.g];
#pragma unroll 1
                for (int c = 0; c < FH / 32; ++c) {
                    uint32_t gv[32], uv[32];
                    tmem_ld32(tbase + c * 32, gv);
                    tmem_ld32(tbase + FH + c * 32, uv);
                    tmem_ld_wait();
                    if (live) {
                        uint4* dst = reinterpret_cast<uint4*>(a.h + (size_t)(G.out_row0 + m) * a.Imax + ti.n_idx * FH + c * 32);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint4 o;
                            uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int k = j * 8 + i * 2;
                                const float h0 = silu(__uint_as_float(gv[k])) * __uint_as_float(uv[k]);
                                const float h1 = silu(__uint_as_float(gv[k + 1])) * __uint_as_float(uv[k + 1]);
                                ow[i] = pack_bf16x2(h0, h1);
                            }
                            dst[j] = o;
                        }
                    }
                }
            } else {  // kScaleY
                // Each 32-column chunk of the warp's 32 rows (in its half of the columns) goes
                // through shared memory so that a
                // store instruction writes 8 rows x 64 contiguous bytes (whole sectors) instead of
                // 32 scattered 16-byte pieces. Lane l stores its row at l * 64 with its four
                // 16-byte pieces swizzled by (l / 2) % 4 (conflict-free both ways); in round i
                // lane l writes piece l % 4 of row l / 4 + 8 i.
                const uint32_t scr = smem_u32(epi_scratch) + (uint32_t)(warp - 2) * 2048u;
                const int hc = (warp - 2) >> 2;  // the half of the columns this warp writes
                const bf16* yrow = a.Yb + ((size_t)tok * (a.K + 1) + slot) * a.H + ti.n_idx * BN;
                const bf16* orow[4];
                bool olive[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int rr = (lane >> 2) + 8 * i;
                    orow[i] = reinterpret_cast<const bf16*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(yrow), rr));
                    olive[i] = __shfl_sync(0xffffffffu, live, rr);
                }
                const uint32_t pc = (uint32_t)(lane & 3);
#pragma unroll 1
                for (int c = hc * (BN / 64); c < (hc + 1) * (BN / 64); ++c) {
                    uint32_t v[32];
                    tmem_ld32(tbase + c * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t ow[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int k = j * 8 + i * 2;
                            ow[i] = pack_bf16x2(sc * __uint_as_float(v[k]), sc * __uint_as_float(v[k + 1]));
                        }
                        sts128(scr + (uint32_t)lane * 64u + (((uint32_t)j ^ (((uint32_t)lane >> 1) & 3u)) << 4), ow);
                    }
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t rr = (uint32_t)(lane >> 2) + 8u * i;
                        const uint4 o = lds128_smem(scr + rr * 64u + ((pc ^ ((rr >> 1) & 3u)) << 4));
                        if (olive[i])
                            *reinterpret_cast<uint4*>(const_cast<bf16*>(orow[i]) + c * 32 + pc * 8) = o;
                    }
                    __syncwarp();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * BN <= 256 ? 256 : 512);
    }
}

// ---------------------------------------------------------------------------------------
// host side: tensor maps and launches

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// 2D K-major bf16 tensor [rows, cols] (row pitch `pitch` elements), box {64, box_rows}, 128B swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t pitch, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {pitch * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPI, int BN>
cudaError_t launch_gemm(const CUtensorMap& A0, const CUtensorMap& A1, const CUtensorMap& B0, const CUtensorMap& B1,
                        const GemmPlan& p, const LayerArgs& a, int grid, cudaStream_t s) {
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm<EPI, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)GemmSmem<BN>::kBytes);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    return launch_pdl(k_gemm<EPI, BN>, dim3(grid), dim3(gemm_threads<EPI>()), (size_t)GemmSmem<BN>::kBytes, s, A0,
                      A1, B0, B1, p, a);
}

}  // namespace

// Router scores of all T tokens on the tensor cores: logits[:, 0:E] = x . Wr^T (+ br).
cudaError_t launch_router_gemm(const LayerArgs& a, cudaStream_t s) {
    // 64-wide N tiles: the E <= 256 score columns of T/128 token tiles would otherwise give
    // only T/128 tiles for 152 SMs
    constexpr int kBNr = 64;
    CUtensorMap mx, mw;
    if (!make_map(&mx, a.x, a.T, a.H, a.H, kBM) || !make_map(&mw, a.router_w, a.E, a.H, a.H, kBNr))
        return cudaErrorInvalidValue;
    GemmPlan p{};
    p.dense_rows = a.T;
    p.dense_tiles = ((a.T + kBM - 1) / kBM) * ((a.E + kBNr - 1) / kBNr);
    p.k_routed = p.k_shared = a.H;
    p.err = &a.hdr->err;
    const int grid = min(p.dense_tiles, a.num_sms);
    cudaError_t e;
    MOE_LAUNCH(MOE_KERNEL_ROUTER_SCORES, s, (e = launch_gemm<kLogits, kBNr>(mx, mx, mw, mw, p, a, grid, s)));
    return e;
}

// Expert GEMMs over the dispatched groups (routed experts + the shared expert).
cudaError_t launch_expert_gemms(const LayerArgs& a, cudaStream_t s) {
    const int fh = gemm_up_half(a);
    CUtensorMap mx, mgu, msgu, mh, mdn, msd;
    bool ok = make_map(&mx, a.x, a.T, a.H, a.H, kBM) &&
              make_map(&mgu, a.gate_up, (uint64_t)a.E * 2 * a.I, a.H, a.H, fh) &&
              make_map(&msgu, a.sgu, (uint64_t)2 * a.Is, a.H, a.H, fh) &&
              make_map(&mh, a.h, a.P + a.T, a.Imax, a.Imax, kBM);
    const int bn_dn = gemm_down_bn(a);
    ok = ok && make_map(&mdn, a.down, (uint64_t)a.E * a.H, a.I, a.I, bn_dn) &&
         make_map(&msd, a.sd, a.H, a.Is, a.Is, bn_dn);
    if (!ok) return cudaErrorInvalidValue;
    const int grid = a.num_sms;
    GemmPlan pu{};
    pu.groups = a.up_groups;
    pu.tile_start = a.up_tiles;
    pu.n_groups = a.n_groups;
    pu.k_routed = pu.k_shared = a.H;
    pu.up_off_routed = a.I;
    pu.up_off_shared = a.Is;
    pu.err = &a.hdr->err;
    cudaError_t e;
    if (fh == 128)
        MOE_LAUNCH(MOE_KERNEL_GATE_UP, s, (e = launch_gemm<kSwiGLU, 256>(mx, mx, mgu, msgu, pu, a, grid, s)));
    else
        MOE_LAUNCH(MOE_KERNEL_GATE_UP, s, (e = launch_gemm<kSwiGLU, 128>(mx, mx, mgu, msgu, pu, a, grid, s)));
    if (e != cudaSuccess) return e;
    GemmPlan pd{};
    pd.groups = a.dn_groups;
    pd.tile_start = a.dn_tiles;
    pd.n_groups = a.n_groups;
    pd.k_routed = a.I;
    pd.k_shared = a.Is;
    pd.err = &a.hdr->err;
    if (bn_dn == 256)
        MOE_LAUNCH(MOE_KERNEL_DOWN, s, (e = launch_gemm<kScaleY, 256>(mh, mh, mdn, msd, pd, a, grid, s)));
    else
        MOE_LAUNCH(MOE_KERNEL_DOWN, s, (e = launch_gemm<kScaleY, 128>(mh, mh, mdn, msd, pd, a, grid, s)));
    return e;
}

}  // namespace moe
