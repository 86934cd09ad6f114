// mg_attn_pair.cuh -- the fused kernel in its two-Q-tile form, for head dim 64 and the graph as
// written (Mirage documentation, tutorials/group-query-attention, "Define GQA Computation Graph":
// A = matmul(Q,K); E = exp(A); S = reduction(E,2); D = div(E,S); O = matmul(D,V)).
//
// One CTA per (batch b, pair of 128-row Q tiles, split j of the N axis): the split's K/V tiles are
// streamed once and feed both Q tiles, and softmax group g owns Q tile g outright: its S buffer,
// its P buffer and its accumulator O_g in tensor memory, and its rows' sums. Per K/V tile t:
//     S_g  = Q_g . K_t              tcgen05 MMA (S warp), fp32 in tensor memory, g = 0, 1
//     P_g  = exp(S_g) (0 beyond N)  group g, fp32; l += rowsum(P_g); fp16 P_g to tensor memory
//     O_g += fp16(P_g) . V_t        tcgen05 MMA with A read from tensor memory (P.V warp)
// No row data passes between the groups, so neither waits on the other: while one group's warps
// wait on tensor memory or a barrier, the other's keep the MUFU unit busy, and the tensor pipe
// takes S and P.V products of both tiles in turn. Compared with the one-tile kernel (two groups on
// alternate K/V tiles of the same rows), a K/V tile also costs half the shared-memory and L2 reads
// per unit of work.
//
// The division by the row sum and the split partials follow the one-tile kernel (mg_attn_kernels.cuh):
// one split writes fp16 O by TMA store; 2..16 splits of one wave combine in a cluster through L2
// (below); more go to the second kernel. The barrier protocol is restated on the CPU by
// tests/pipeline_model.py (PairSim), which a change here must follow.
//
// Tensor memory (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,320), O_1 [320,384), P_0
// [384,448), P_1 [448,512) (fp16 pairs: 128 columns of P in 64).
#pragma once

#include "mg_attn_kernels.cuh"

namespace mg {

constexpr int kPairD = 64;                                      // head dim of the two-tile kernel
constexpr uint32_t kPairQBytes = kBlockM * kPairD * 2;          // one Q tile
constexpr uint32_t kPairStageBytes = 2u * kPairD * kBlockN * 2; // K + V tile
constexpr uint32_t kPairTmemO = 256;                            // O_g at kPairTmemO + 64 g
constexpr uint32_t kPairTmemP = 384;                            // P_g at kPairTmemP + 64 g

// Shared-memory bytes of the two-tile kernel: alignment slack, two Q tiles, the K/V ring, the
// (unused) exchange area kept for layout symmetry with the one-tile kernel, and the barriers.
__host__ __device__ constexpr uint32_t pair_smem_bytes(int stages)
{
    return 1024u + 2u * kPairQBytes + static_cast<uint32_t>(stages) * kPairStageBytes + 2u * 128 * 4 + 512u;
}

// The cluster combine of the two-tile kernel moves the split partials through L2: each CTA stores
// its fp32 numerators and row sums, one cluster barrier publishes them, and each rank combines its
// rows from L2. (The one-tile kernel exchanges them on chip instead.)

// Index of the (split j, batch b, row tile mt) tile among the cluster combine's partial tiles.
__device__ __forceinline__ size_t cluster_tile(const FwdParams &p, int j, int b, int mt)
{
    return (static_cast<size_t>(j) * p.B + b) * p.m_tiles_per_b + mt;
}

// Rows per partial tile of the cluster combine: 128, or M when a batch has fewer rows.
__device__ __forceinline__ int cluster_tile_rows(const FwdParams &p) { return p.M < kBlockM ? p.M : kBlockM; }

// The reading side of the cluster combine, for CTA rank j and the row tiles (b, mt_first) ..
// (b, mt_first + ntiles - 1) of its CTA: rows [128 j / n, 128 (j+1) / n) of each tile as
// (sum_r w_r O_r) / (sum_r w_r l_r) over the n ranks, w_r = 1 (exp(m_r - max_r m_r) when SAFE),
// written as fp16 O. Partial tiles are tile-major (float4 column group outermost, the tile's
// cluster_tile_rows rows innermost). An element is (column group, row); the two lanes of a pair take the same elements,
// lane h the ranks [h RPL, h RPL + RPL), and a pair takes 8 / RPL elements at a time, so that each
// thread has its 8 loads in flight together. The pair then adds its two sums in a fixed order
// (lower ranks first) and each lane writes two of the element's four columns: the result does not
// depend on timing. (One call loops over the tiles: a call site per tile costs registers.)
template <int D, bool SAFE, int RPL>
__device__ __forceinline__ void cluster_combine_rows(const FwdParams &p, int b, int mt_first, int ntiles, int j,
                                                     int tid)
{
    constexpr int G = D / 4;          // float4 column groups per row
    constexpr int EPP = 8 / RPL;      // elements per pair per batch of loads
    constexpr int kPairs = kSoftmaxThreads / 2;
    const int n = p.n_split;
    const int pair = tid >> 1;
    const int h = tid & 1;
    const unsigned pair_mask = 3u << (tid & 30);
    const size_t tiles_per_rank = static_cast<size_t>(p.B) * p.m_tiles_per_b;
    const int TR = cluster_tile_rows(p);
    const float4 *ws4 = reinterpret_cast<const float4 *>(p.ws_o);
#pragma unroll 1
    for (int mt = mt_first; mt < mt_first + ntiles; ++mt) {
        const int m0 = mt * kBlockM;
        const int lo = j * kBlockM / n;
        // Rows this rank combines: its share of the tile, cut at M (rows past M hold no partials).
        const int R = max(0, min((j + 1) * kBlockM / n, p.M - m0) - lo);
        const int E = R * G;
        const size_t tile0 = static_cast<size_t>(b) * p.m_tiles_per_b + mt;
        for (int base = pair; base < E; base += kPairs * EPP) {
            // All loads first (L1 is bypassed: the partials were written by other SMs).
            float4 v[8];
            float lv[8], mr[8];
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const int e = base + (s / RPL) * kPairs;
                const int r = h * RPL + s % RPL;
                if (e < E && r < n) {
                    const size_t t = r * tiles_per_rank + tile0;
                    const int rr = lo + e % R;
                    v[s] = __ldcg(ws4 + (t * G + e / R) * TR + rr);
                    lv[s] = __ldcg(p.ws_l + t * TR + rr);
                    if (SAFE)
                        mr[s] = __ldcg(p.ws_m + t * TR + rr);
                }
            }
#pragma unroll
            for (int k = 0; k < EPP; ++k) {
                const int e = base + k * kPairs;  // the same on both lanes of the pair
                if (e >= E)
                    break;
                float mmax = 0.f;
                if (SAFE) {
                    mmax = -INFINITY;
#pragma unroll
                    for (int q = 0; q < RPL; ++q)
                        if (h * RPL + q < n)
                            mmax = fmaxf(mmax, mr[k * RPL + q]);
                    mmax = fmaxf(mmax, __shfl_xor_sync(pair_mask, mmax, 1));
                }
                float a[4] = {0.f, 0.f, 0.f, 0.f};
                float lsum = 0.f;
#pragma unroll
                for (int q = 0; q < RPL; ++q) {
                    if (h * RPL + q < n) {
                        const int s = k * RPL + q;
                        const float w = SAFE ? ptx::ex2_approx((mr[s] - mmax) * ptx::kLog2e) : 1.f;
                        a[0] = fmaf(w, v[s].x, a[0]);
                        a[1] = fmaf(w, v[s].y, a[1]);
                        a[2] = fmaf(w, v[s].z, a[2]);
                        a[3] = fmaf(w, v[s].w, a[3]);
                        lsum = fmaf(w, lv[s], lsum);
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float other = __shfl_xor_sync(pair_mask, a[c], 1);
                    a[c] = h == 0 ? a[c] + other : other + a[c];
                }
                const float lother = __shfl_xor_sync(pair_mask, lsum, 1);
                lsum = h == 0 ? lsum + lother : lother + lsum;
                const int rr = lo + e % R;
                const float inv = __frcp_rn(lsum);
                const uint32_t o = ptx::pack_half2(a[2 * h] * inv, a[2 * h + 1] * inv);
                *reinterpret_cast<uint32_t *>(p.O + (static_cast<size_t>(b) * p.M + m0 + rr) * D + (e / R) * 4 +
                                              2 * h) = o;
            }
        }
    }
}

template <int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    mg_attn_fwd_pair(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                     const __grid_constant__ CUtensorMap tmW, const FwdParams p)
{
    constexpr int D = kPairD;
    using BI = Bars<STAGES, 2>;
    static_assert(pair_smem_bytes(STAGES) <= 232448u, "tile configuration exceeds 227 KB");
    static_assert(STAGES >= 2, "the fp32 output staging takes two K/V stages");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sQ = ptx::smem_u32(smem);  // Q tile g at sQ + g * kPairQBytes
    const uint32_t sStage0 = sQ + 2 * kPairQBytes;
    float *l_xchg = reinterpret_cast<float *>(smem + 2 * kPairQBytes + STAGES * kPairStageBytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(l_xchg + 2 * kBlockM);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + BI::kCount);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    auto bar = [&](int i) { return ptx::smem_u32(bars + i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // CTA -> (b, row pair mp, split j); as in the one-tile kernel, the n_split CTAs of a row pair
    // are consecutive (one cluster) with the cluster combine.
    const int pairs_per_b = (p.m_tiles_per_b + 1) / 2;
    const int cta = blockIdx.x;
    const int mp = p.cluster_reduce ? (cta / p.n_split) % pairs_per_b : cta % pairs_per_b;
    const int j = p.cluster_reduce ? cta % p.n_split : (cta / pairs_per_b) % p.n_split;
    const int b = cta / (pairs_per_b * p.n_split);
    const int m0 = mp * 2 * kBlockM;  // first row of Q tile 0; Q tile g starts at m0 + 128 g
    const int T = (p.n_tiles - j + p.n_split - 1) / p.n_split;  // >= 1: n_split <= n_tiles
    auto tile_of = [&](int t) { return j + t * p.n_split; };

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(BI::kQFull), 1);
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar(BI::kKFull + s), 1);
            ptx::mbar_init(bar(BI::kVFull + s), 1);
            ptx::mbar_init(bar(BI::kKvEmpty + s), 1);
        }
        for (int g = 0; g < 2; ++g) {
            ptx::mbar_init(bar(BI::kSFull + g), 1);
            ptx::mbar_init(bar(BI::kSEmpty + g), kGroupWarps);
            ptx::mbar_init(bar(BI::kPFull + g), kGroupWarps);
            ptx::mbar_init(bar(BI::kPEmpty + g), 1);
        }
        ptx::mbar_init(bar(BI::kOFull), 1);
        ptx::mbar_init(bar(BI::kDrain), 1);
        ptx::mbar_init(bar(BI::kDrainPv), 1);
        ptx::mbar_init(bar(BI::kNever), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmQ);
        ptx::prefetch_tensormap(&tmK);
        ptx::prefetch_tensormap(&tmV);
        if (p.n_split == 1)
            ptx::prefetch_tensormap(&tmO);
        else if (!p.cluster_reduce)
            ptx::prefetch_tensormap(&tmW);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_holder), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    // Everything above touched only on-chip state; global memory waits for the previous grid.
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();

    const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            bool q_armed = false;
            int armed[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s)
                armed[s] = 0;
            bool ok = true;
            if (p.inject_timeout)
                ok = wait_bounded(wc, bar(BI::kNever), 0, BI::kNever);
            if (ok) {
                // Both Q tiles on one barrier; rows past M are zero-filled, computed and never
                // stored (plans take this kernel only for an even number of row tiles per batch).
                ptx::mbar_arrive_expect_tx(bar(BI::kQFull), 2 * kPairQBytes);
                q_armed = true;
                ptx::tma_load_3d(sQ, &tmQ, bar(BI::kQFull), 0, m0, b);
                ptx::tma_load_3d(sQ + kPairQBytes, &tmQ, bar(BI::kQFull), 0, m0 + kBlockM, b);
            }
            for (int t = 0; ok && t < T; ++t) {
                const int s = t % STAGES;
                const uint32_t round = static_cast<uint32_t>(t / STAGES);
                if (t >= STAGES && !wait_bounded(wc, bar(BI::kKvEmpty + s), (round & 1u) ^ 1u, BI::kKvEmpty + s)) {
                    ok = false;
                    break;
                }
                const int n0 = tile_of(t) * kBlockN;
                const uint32_t sK = sStage0 + s * kPairStageBytes;
                const uint32_t sV = sK + D * kBlockN * 2;
                ptx::mbar_arrive_expect_tx(bar(BI::kKFull + s), D * kBlockN * 2);
                ptx::mbar_arrive_expect_tx(bar(BI::kVFull + s), kBlockN * D * 2);
                ++armed[s];
                ptx::tma_load_3d(sK, &tmK, bar(BI::kKFull + s), n0, 0, b);
                ptx::tma_load_3d(sK + D * 128, &tmK, bar(BI::kKFull + s), n0 + 64, 0, b);
                ptx::tma_load_3d(sV, &tmV, bar(BI::kVFull + s), 0, n0, b);
            }
            if (ok) {
                // Tail: the commits that release the last stages must land before the CTA exits.
                for (int u = T - STAGES > 0 ? T - STAGES : 0; ok && u < T; ++u)
                    ok = wait_bounded(wc, bar(BI::kKvEmpty + u % STAGES), static_cast<uint32_t>(u / STAGES) & 1u,
                                      BI::kKvEmpty + u % STAGES);
            }
            if (*abort_flag) {
                // Unwind: every copy issued must land before the CTA's shared memory goes away.
                if (q_armed)
                    wait_drain(bar(BI::kQFull), 0, p.timeout_ns);
#pragma unroll
                for (int s = 0; s < STAGES; ++s)
                    if (armed[s] > 0) {
                        wait_drain(bar(BI::kKFull + s), static_cast<uint32_t>(armed[s] - 1) & 1u, p.timeout_ns);
                        wait_drain(bar(BI::kVFull + s), static_cast<uint32_t>(armed[s] - 1) & 1u, p.timeout_ns);
                    }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- S_g = Q_g . K issuer
        // Warp-wide waits (the decision to go on is a vote); the elect.sync lane issues.
        constexpr uint32_t idesc_s = ptx::idesc_f16_f32(kBlockM, kBlockN, false, true);
        auto warp_wait = [&](uint32_t b_, uint32_t parity, int where) -> bool {
            return __all_sync(0xffffffffu, wait_bounded(wc, b_, parity, where));
        };
        bool ok = warp_wait(bar(BI::kQFull), 0, BI::kQFull);
        for (int t = 0; ok && t < T; ++t) {
            const int s = t % STAGES;
            if (!warp_wait(bar(BI::kKFull + s), static_cast<uint32_t>(t / STAGES) & 1u, BI::kKFull + s)) {
                ok = false;
                break;
            }
            // B = K: N-major; 16 d-rows (2048 B) per k-step; the two 64-column halves D*128 B apart.
            const uint64_t k_desc = ptx::sdesc_sw128(sStage0 + s * kPairStageBytes, D * 128, 1024);
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                // S buffer g is free once group g has read S_g of the previous tile.
                if (t >= 1 && !warp_wait(bar(BI::kSEmpty + g), static_cast<uint32_t>(t - 1) & 1u, BI::kSEmpty + g)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                if (ptx::elect_one()) {
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        // A = Q_g: K-major; 16-column steps advance 32 B inside the swizzle row.
                        const uint64_t a_desc = ptx::sdesc_sw128(sQ + g * kPairQBytes + k * 32, 16, 1024);
                        ptx::mma_f16_ss(tmem + g * kBlockN, a_desc, k_desc + static_cast<uint64_t>(k * (2048 >> 4)),
                                        idesc_s, k > 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(bar(BI::kSFull + g));
                }
                __syncwarp();
            }
        }
        // Every S product issued completes before tensor memory is freed (see the one-tile kernel).
        if (ptx::elect_one()) {
            ptx::mma_commit(bar(BI::kDrain));
            wait_drain(bar(BI::kDrain), 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ---------------------------------------------------------------- O_g += P_g . V issuer
        constexpr uint32_t idesc_o = ptx::idesc_f16_f32(kBlockM, D, false, true);
        auto warp_wait = [&](uint32_t b_, uint32_t parity, int where) -> bool {
            return __all_sync(0xffffffffu, wait_bounded(wc, b_, parity, where));
        };
        bool ok = true;
        for (int t = 0; ok && t < T; ++t) {
            const int s = t % STAGES;
            // V first: every V phase completes on a copy this warp waits for in order.
            if (!warp_wait(bar(BI::kVFull + s), static_cast<uint32_t>(t / STAGES) & 1u, BI::kVFull + s)) {
                ok = false;
                break;
            }
            // B = V: d-major, 16 rows (2048 B) per k-step.
            const uint64_t v_desc = ptx::sdesc_sw128(sStage0 + s * kPairStageBytes + D * kBlockN * 2,
                                                     TileCfg<D>::kChunkRows128, 1024);
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                if (!warp_wait(bar(BI::kPFull + g), static_cast<uint32_t>(t) & 1u, BI::kPFull + g)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t tP = tmem + kPairTmemP + g * 64;
                if (ptx::elect_one()) {
#pragma unroll
                    for (int k = 0; k < kBlockN / 16; ++k)  // 16 K-columns per step = 8 tensor-memory columns
                        ptx::mma_f16_ts(tmem + kPairTmemO + g * D, tP + k * 8,
                                        v_desc + static_cast<uint64_t>(k * (2048 >> 4)), idesc_o,
                                        (t > 0 || k > 0) ? 1u : 0u);
                    ptx::mma_commit(bar(BI::kPEmpty + g));
                    if (g == 1) {
                        // Both products of the tile are behind this commit: the stage is free.
                        ptx::mma_commit(bar(BI::kKvEmpty + s));
                        if (t == T - 1)
                            ptx::mma_commit(bar(BI::kOFull));
                    }
                }
                __syncwarp();
            }
        }
        if (ok) {
            // Tail: the commits that release the last P buffers must land before the CTA exits.
            for (int g = 0; ok && g < 2; ++g)
                ok = warp_wait(bar(BI::kPEmpty + g), static_cast<uint32_t>(T - 1) & 1u, BI::kPEmpty + g);
        }
        if (!ok) {
            if (ptx::elect_one()) {
                ptx::mma_commit(bar(BI::kDrainPv));
                wait_drain(bar(BI::kDrainPv), 0, p.timeout_ns);
            }
            __syncwarp();
        }
    } else {
        // ---------------------------------------------------------------- softmax + epilogue
        const int sw = warp - 2;                 // 0..7
        const int q4 = warp & 3;                 // tensor-memory lane quarter this warp may access
        const int g = sw >> 2;                   // Q tile of this group
        const int row = q4 * 32 + lane;          // row inside Q tile g
        const int mg0 = m0 + g * kBlockM;        // first row of Q tile g
        const bool warp_rows = (mg0 + q4 * 32) < p.M;
        const uint32_t lane_addr = static_cast<uint32_t>(q4 * 32) << 16;
        auto warp_wait = [&](uint32_t b_, uint32_t parity, int where) -> bool {
            const bool r = wait_bounded(wc, b_, parity, where);
            return __all_sync(0xffffffffu, r);
        };
        uint64_t acc[2] = {0, 0};  // packed fp32 partial row sums
        const ptx::ExpPairConsts ek = ptx::exp_pair_consts();
        bool ok = true;
        for (int t = 0; ok && t < T; ++t) {
            if (!warp_wait(bar(BI::kSFull + g), static_cast<uint32_t>(t) & 1u, BI::kSFull + g)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const int n_valid = p.N - tile_of(t) * kBlockN;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t r0[32], r1[32];
                if (warp_rows) {
                    const uint32_t s_addr = tmem + lane_addr + g * kBlockN + half * 64;
                    ptx::tmem_ld_32x32b_x32(s_addr, r0);
                    ptx::tmem_ld_32x32b_x32(s_addr + 32, r1);
                    ptx::tmem_ld_wait(r0);
                    ptx::tmem_ld_wait(r1);
                }
                if (half == 1) {
                    // All of S_g is in registers: the buffer can take the next tile's product.
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        ptx::mbar_arrive(bar(BI::kSEmpty + g));
                }
                // The exponentials go to registers first; only their store into P_g waits for the
                // previous tile's P.V product to have read the buffer, so that product's latency
                // hides behind them.
                uint32_t w[32];
                if (warp_rows) {
                    const int nv = n_valid - half * 64;
                    if (nv >= 64) {
                        exp_slice<false>(r0, 0, nv, w, acc, ek, 0);
                        exp_slice<false>(r1, 32, nv, w + 16, acc, ek, 0);
                    } else {
                        exp_slice<true>(r0, 0, nv, w, acc, ek, 0);
                        exp_slice<true>(r1, 32, nv, w + 16, acc, ek, 0);
                    }
                }
                if (half == 0 && t >= 1 &&
                    !warp_wait(bar(BI::kPEmpty + g), static_cast<uint32_t>(t - 1) & 1u, BI::kPEmpty + g)) {
                    ok = false;
                    break;
                }
                if (warp_rows) {
                    ptx::tmem_st_32x32b_x32(tmem + lane_addr + kPairTmemP + g * 64 + half * 32, w);
                    ptx::tmem_st_wait();
                }
            }
            if (!ok)
                break;
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(bar(BI::kPFull + g));
        }

        // ------------------------------------------------------------ epilogue
        const float l = (__uint_as_float(static_cast<uint32_t>(acc[0])) +
                         __uint_as_float(static_cast<uint32_t>(acc[0] >> 32))) +
                        (__uint_as_float(static_cast<uint32_t>(acc[1])) +
                         __uint_as_float(static_cast<uint32_t>(acc[1] >> 32)));
        // "O is ready" is a decision all eight softmax warps share (a warp that unwound votes no),
        // so the barrier inside the branch below is reached by all of them or by none.
        const bool o_ready = ptx::named_barrier_and(kSoftmaxBarrier, kSoftmaxThreads,
                                                    ok && warp_wait(bar(BI::kOFull), 0, BI::kOFull));
        const int mt = 2 * mp + g;                   // row tile of this group
        if (o_ready) {
            ptx::tc_fence_after();
            // One split: fp16 O/l staged in stage 0 (tile g at +16 KB g) for a TMA store. Second
            // kernel: fp32 partials staged in stages 0-1 (tile g at +32 KB g). Cluster combine: fp32
            // partials stored from registers to the tile-major workspace.
            const uint32_t stage = sStage0;
            if (warp_rows) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    const int col = c * 32;
                    ptx::tmem_ld_32x32b_x32(tmem + lane_addr + kPairTmemO + g * D + col, r);
                    ptx::tmem_ld_wait(r);
                    if (p.cluster_reduce) {
                        // M >= 256 here, so partial tiles have 128 rows.
                        float4 *dst = reinterpret_cast<float4 *>(p.ws_o) +
                                      (cluster_tile(p, j, b, mt) * (D / 4) + col / 4) * kBlockM + row;
                        if (mg0 + row < p.M) {
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                dst[q * kBlockM] =
                                    make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                                __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
                        }
                    } else if (p.n_split == 1) {
                        const uint32_t chunk = stage + g * (kBlockM * D * 2);
                        const uint32_t u0 = static_cast<uint32_t>(col / 8);
                        const float inv = __frcp_rn(l);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            ptx::st_shared_v4(chunk + sw128_offset(row, u0 + q),
                                              ptx::pack_half2(__uint_as_float(r[8 * q + 0]) * inv,
                                                              __uint_as_float(r[8 * q + 1]) * inv),
                                              ptx::pack_half2(__uint_as_float(r[8 * q + 2]) * inv,
                                                              __uint_as_float(r[8 * q + 3]) * inv),
                                              ptx::pack_half2(__uint_as_float(r[8 * q + 4]) * inv,
                                                              __uint_as_float(r[8 * q + 5]) * inv),
                                              ptx::pack_half2(__uint_as_float(r[8 * q + 6]) * inv,
                                                              __uint_as_float(r[8 * q + 7]) * inv));
                    } else {
                        // fp32 partial: {32, 128} fp32 boxes; tile g's two boxes follow each other.
                        const uint32_t chunk = stage + g * (kBlockM * D * 4) + c * TileCfg<D>::kChunkRows128;
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            ptx::st_shared_v4(chunk + sw128_offset(row, q), r[4 * q + 0], r[4 * q + 1], r[4 * q + 2],
                                              r[4 * q + 3]);
                    }
                }
            }
            if (p.n_split > 1 && mg0 + row < p.M) {
                const size_t r = p.cluster_reduce ? cluster_tile(p, j, b, mt) * kBlockM + row
                                                  : (static_cast<size_t>(j) * p.B + b) * p.M + mg0 + row;
                p.ws_l[r] = l;
            }
            if (!p.cluster_reduce) {
                ptx::fence_proxy_async_smem();
                ptx::named_barrier(kSoftmaxBarrier, kSoftmaxThreads);
                if (sw == 0 && lane == 0) {
#pragma unroll
                    for (int gg = 0; gg < 2; ++gg) {
                        const int mr = m0 + gg * kBlockM;
                        if (mr >= p.M)
                            continue;  // tile 1 of an odd last pair: nothing to store
                        if (p.n_split == 1) {
                            ptx::tma_store_3d(&tmO, stage + gg * (kBlockM * D * 2), 0, mr, b);
                        } else {
#pragma unroll
                            for (int c = 0; c < D / 32; ++c)
                                ptx::tma_store_3d(&tmW, stage + gg * (kBlockM * D * 4) + c * TileCfg<D>::kChunkRows128,
                                                  c * 32, mr, j * p.B + b);
                        }
                    }
                    ptx::bulk_commit_group();
                    ptx::bulk_wait_group_read0();
                }
            }
        }
    }

    // Cluster combine, as in the one-tile kernel: one barrier publishes every CTA's partials (in
    // L2), then CTA rank j combines rows [128 j / n, 128 (j+1) / n) of each of the pair's row tiles.
    __syncwarp();
    if (p.cluster_reduce) {
        ptx::cluster_sync();
        if (warp >= 2 && warp < 2 + kSoftmaxWarps) {
            const int tid = threadIdx.x - 64;
            const int n = p.n_split;
            // Both row tiles of the pair in one call (the plan keeps pairs whole).
            if (n <= 2)
                cluster_combine_rows<D, false, 1>(p, b, 2 * mp, 2, j, tid);
            else if (n <= 4)
                cluster_combine_rows<D, false, 2>(p, b, 2 * mp, 2, j, tid);
            else if (n <= 8)
                cluster_combine_rows<D, false, 4>(p, b, 2 * mp, 2, j, tid);
            else
                cluster_combine_rows<D, false, 8>(p, b, 2 * mp, 2, j, tid);
        }
    }

    // Teardown: every tensor-memory access of the CTA is ordered before the free.
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace mg
