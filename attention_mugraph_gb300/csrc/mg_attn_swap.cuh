// mg_attn_swap.cuh -- the fused kernel specialised for few query rows (at most 16 per batch, head
// dim 128, the graph as written; Mirage documentation, tutorials/group-query-attention, "Define
// GQA Computation Graph", and its launch example "Launch Mirage-Generated GQA Kernel" with one query
// row per head).
//
// The one-tile kernel puts the query rows on the MMA's 128-row M axis, so a decode batch of 8 rows
// leaves 120 of them zero. Here the operands swap roles ("swap-AB"): per K/V tile of 128 keys,
//     S^T = K^T . Q^T     M = 128 keys, N = 16 query rows, K = d      (tcgen05, fp32 in tensor memory)
//     P^T = exp(S^T)      fp32; l[q] += sum over the tile's keys; fp16 P^T to shared memory
//     O^T += V^T . P^T    M = d = 128, N = 16 query rows, K = 128 keys
// so every MMA row is a key (or an output column) and nothing is padded but the N axis (16 columns
// for up to 16 rows). K and V serve as A operands in the layouts their TMA tiles already have (keys,
// resp. d, contiguous), Q^T and P^T as K-major B operands. S^T and O^T take 16 tensor-memory
// columns each; the row sum of query q is a sum over keys, i.e. over tensor-memory lanes, so each
// thread keeps one per query for its keys and the CTA reduces them once at the end.
//
// Roles, ring, bounded waits and unwinding are the one-tile kernel's (mg_attn_kernels.cuh): a TMA
// producer warp, an S-issuing warp, a P.V-issuing warp and two groups of four softmax warps that take
// alternate tiles, with the same barrier protocol (tests/pipeline_model.py, Sim, graph as written);
// P lives in shared memory, written by the softmax warps and read by the tensor core after a proxy
// fence. Split partials (fp32 O^T columns and row sums) are combined on chip when the n_split CTAs
// of a batch run as one thread-block cluster, else by the second kernel.
//
// ONLINE: the max-subtracted evaluation in one pass over K and V (each query row's maximum is not
// known before the last tile, so it is kept running). Each softmax group keeps its own running
// maximum m[q] and its own O^T accumulator (tensor-memory columns 32 and 48). Per tile the group
// finds the tile's maximum of every query over its 128 keys (a warp reduction, then the four warps'
// results through shared memory and a group barrier). Where some query's tile maximum exceeds m[q]
// by more than kSwapRescaleSlack, it raises every m[q] to its tile maximum (if larger) and scales
// its partial sums by alpha[q] = exp(m_old - m_new), and also its O^T accumulator, in tensor memory,
// once the tensor core has finished the group's previous P.V (its P buffer released) and before it
// publishes the new P^T. It writes P^T = exp(S^T - m); the CPU model of this
// protocol is tests/pipeline_model.py's ONLINE variant. The epilogue merges the two groups (weights
// exp(m_g - max m)); split partials carry their maximum to the combine, which weights them the same
// way. The result equals the graph as written, exp(S) / rowsum(exp(S)) . V, up to rounding.
//
// QK-norm (Mirage documentation, tutorials/attention-with-kv-norm: Q and K rms-normalised over d
// before the graph) runs on the ONLINE form with the scores scaled in fp32, S^T[n, q] a_q c_n:
// the query scales a_q = 1/rms(Q[q, :]) once per CTA from Q^T in shared memory (all softmax
// warps, one barrier), and per tile each thread's key scale c_n = 1/rms(K[:, n]) from the K tile
// in shared memory (a lane sums one 16-byte unit of every eighth d-row, then a reduce-scatter over
// the eight lanes of a unit), while the tensor core computes S^T. K is read once.
#pragma once

#include "mg_attn_kernels.cuh"

namespace mg {

constexpr int kSwapD = 128;
constexpr int kSwapNQ = 16;                                      // query rows per tile (MMA N)
constexpr uint32_t kSwapQBytes = kSwapNQ * kSwapD * 2;           // two 64-column chunks of 16 rows
constexpr uint32_t kSwapChunk = kSwapNQ * 128;                   // one such chunk (2 KB)
constexpr uint32_t kSwapStageBytes = 2u * kSwapD * kBlockN * 2;  // K + V tile
constexpr uint32_t kSwapPBytes = kSwapNQ * kBlockN * 2;          // P^T: two 64-key chunks of 16 rows
constexpr int kSwapPBuffers = 3;
// A stage's K tile is free once its S^T product completes (in the QK-norm form also once the
// four warps of the tile's group have read it for the key scales), and the load warp issues K
// tile t + kSwapKLead before V tile t: the K stream runs ahead of the V stream, whose stages are
// held until P.V.
constexpr int kSwapKLead = 2;
constexpr uint32_t kSwapTmemCols = 64;                           // S^T buffers at 0 and 16, O^T at 32 (and 48)
constexpr uint32_t kSwapTmemO = 32;
// Forms of the few-row kernel: the graph as written; ONLINE (max-subtracted, one pass); ONLINE
// with QK-norm scales.
constexpr int kSwapPlainForm = 0;
constexpr int kSwapOnlineForm = 1;
constexpr int kSwapQkNormForm = 2;
// ONLINE: per group, two buffers of the four warps' tile maxima; group 1's final maxima; the
// query scales (QK-norm).
constexpr uint32_t kSwapOnlineBytes = (2 * 2 * kGroupWarps * kSwapNQ + 2 * kSwapNQ) * 4;
// ONLINE: a group keeps the maximum it subtracts until some query's tile maximum exceeds it by
// more than this; any per-row shift cancels in the normalisation, and the scores stay at most 8
// above the subtracted value, so P <= e^8 ~ 2981 (fp16 keeps its relative precision up to 65504).
// The rescale then runs on a group's first tiles and on jumps, not on every small rise.
constexpr float kSwapRescaleSlack = 8.0f;

// Shared-memory bytes: alignment slack, Q^T, the P^T ring, the K/V ring, the per-warp row sums,
// (ONLINE) the maxima exchanged between warps, and the barriers.
__host__ __device__ constexpr uint32_t swap_smem_bytes(int stages, bool online = false)
{
    return 1024u + kSwapQBytes + kSwapPBuffers * kSwapPBytes + static_cast<uint32_t>(stages) * kSwapStageBytes +
           kSoftmaxWarps * kSwapNQ * 4 + (online ? kSwapOnlineBytes : 0u) + 512u;
}

// Warp-collective: lane i writes tensor-memory lane (taddr.lane + i), 16 consecutive 32-bit
// columns starting at taddr.col. Complete (and the registers reusable) after tmem_st_wait().
__device__ __forceinline__ void swap_tmem_st_x16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

// The maximum over the warp's 32 lanes of each of 16 values v[0..15], in 16 shuffles: at each step
// a lane keeps the half of its values that its lane bit selects and takes the maximum with the
// partner lane's copy of that half (the other half is what it sends). Lane L returns the maximum
// of value (L >> 1) & 15. v is overwritten.
__device__ __forceinline__ float warp_max16(float (&v)[16], int lane)
{
#pragma unroll
    for (int w = 8, bit = 16; w >= 1; w >>= 1, bit >>= 1) {
        const bool hi = (lane & bit) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float send = hi ? v[i] : v[i + w];
            const float keep = hi ? v[i + w] : v[i];
            v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, bit));
        }
    }
    return fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
}

template <int STAGES, int FORM = kSwapPlainForm>
__global__ void __launch_bounds__(kThreads, 1)
    mg_attn_fwd_swap(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                     const __grid_constant__ CUtensorMap tmW, const FwdParams p)
{
    constexpr int D = kSwapD;
    constexpr bool ONLINE = FORM != kSwapPlainForm;
    constexpr bool QKN = FORM == kSwapQkNormForm;
    using BI = Bars<STAGES, kSwapPBuffers>;
    static_assert(swap_smem_bytes(STAGES, ONLINE) <= 232448u, "tile configuration exceeds 227 KB");
    (void)tmO;
    (void)tmW;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sQ = ptx::smem_u32(smem);
    const uint32_t sP0 = sQ + kSwapQBytes;                        // P^T buffer pb at sP0 + pb * kSwapPBytes
    const uint32_t sStage0 = sP0 + kSwapPBuffers * kSwapPBytes;   // 1024-aligned: 4 KB steps so far
    float *l_red = reinterpret_cast<float *>(smem + kSwapQBytes + kSwapPBuffers * kSwapPBytes + STAGES * kSwapStageBytes);
    float *m_red = l_red + kSoftmaxWarps * kSwapNQ;           // ONLINE: [group][buffer][warp][query]
    float *m_fin = m_red + 2 * 2 * kGroupWarps * kSwapNQ;     // ONLINE: group 1's final maxima
    float *a_sc = m_fin + kSwapNQ;                            // QK-norm: the query scales
    uint64_t *bars = reinterpret_cast<uint64_t *>(ONLINE ? a_sc + kSwapNQ : m_red);
    // After the common barriers: the K halves of the stages released on their own (kKvEmpty then
    // releases the V halves).
    constexpr int kKEmpty = BI::kCount;
    static_assert((kKEmpty + STAGES) * 8 + 8 <= 512, "barrier area overflow");
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + kKEmpty + STAGES);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    auto bar = [&](int i) { return ptx::smem_u32(bars + i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // CTA -> (b, split j): one row tile per batch (M <= 16); split j takes the column tiles j,
    // j + n_split, ... as in the one-tile kernel.
    const int cta = blockIdx.x;
    const int j = cta % p.n_split;
    const int b = cta / p.n_split;
    const int T = (p.n_tiles - j + p.n_split - 1) / p.n_split;  // >= 1
    auto tile_of = [&](int t) { return j + t * p.n_split; };

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(BI::kQFull), 1);
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar(BI::kKFull + s), 1);
            ptx::mbar_init(bar(BI::kVFull + s), 1);
            ptx::mbar_init(bar(BI::kKvEmpty + s), 1);
            ptx::mbar_init(bar(kKEmpty + s), QKN ? 1 + kGroupWarps : 1);
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(bar(BI::kSFull + s), 1);
            ptx::mbar_init(bar(BI::kSEmpty + s), kGroupWarps);
        }
        for (int s = 0; s < kSwapPBuffers; ++s) {
            ptx::mbar_init(bar(BI::kPFull + s), kGroupWarps);
            ptx::mbar_init(bar(BI::kPEmpty + s), 1);
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
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_holder), kSwapTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    // Global memory waits for the previous grid as in the one-tile kernel: early == 1, the load
    // warp's first copies before its wait; early == 2, the dependents released now and only the
    // global writes after the wait.
    if (p.early == 2) {
        ptx::griddep_launch_dependents();
    } else if (!(warp == 0 && p.early == 1)) {
        ptx::griddep_wait();
        ptx::griddep_launch_dependents();
    }

    const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        // Lane 0 issues every copy; early loads as in the one-tile kernel (Q and the first STAGES
        // tiles before the warp's wait for the previous grid, which the other lanes take only
        // once lane 0 has issued them: the warp meets at a __syncwarp from both paths).
        if (lane != 0) {
            if (p.early == 1) {
                __syncwarp();
                ptx::griddep_wait();
                ptx::griddep_launch_dependents();
            }
        } else {
            bool q_armed = false;
            int armed_k[STAGES], armed_v[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s)
                armed_k[s] = armed_v[s] = 0;
            bool ok = true;
            auto issue_k = [&](int t) {
                const int s = t % STAGES;
                const uint32_t sK = sStage0 + s * kSwapStageBytes;
                const int n0 = tile_of(t) * kBlockN;
                ptx::mbar_arrive_expect_tx(bar(BI::kKFull + s), D * kBlockN * 2);
                ++armed_k[s];
                ptx::tma_load_3d(sK, &tmK, bar(BI::kKFull + s), n0, 0, b);
                ptx::tma_load_3d(sK + D * 128, &tmK, bar(BI::kKFull + s), n0 + 64, 0, b);
            };
            auto issue_v = [&](int t) {
                const int s = t % STAGES;
                const uint32_t sV = sStage0 + s * kSwapStageBytes + D * kBlockN * 2;
                const int n0 = tile_of(t) * kBlockN;
                ptx::mbar_arrive_expect_tx(bar(BI::kVFull + s), kBlockN * D * 2);
                ++armed_v[s];
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    ptx::tma_load_3d(sV + c * TileCfg<D>::kChunkRows128, &tmV, bar(BI::kVFull + s), c * 64, n0, b);
            };
            if (p.inject_timeout)
                ok = wait_bounded(wc, bar(BI::kNever), 0, BI::kNever);
            int tk = 0, tv = 0;  // the next K and V tiles to issue
            if (ok) {
                // Q[b, 0:16, 64c:64c+64] (the tensor map's box is 16 rows; rows past M read as zero).
                ptx::mbar_arrive_expect_tx(bar(BI::kQFull), kSwapQBytes);
                q_armed = true;
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    ptx::tma_load_3d(sQ + c * kSwapChunk, &tmQ, bar(BI::kQFull), c * 64, 0, b);
                if (p.early == 1)
                    for (; tk < T && tk < STAGES; ++tk) {  // the stages are free: no wait
                        issue_k(tk);
                        issue_v(tk);
                    }
                tv = tk;
            }
            if (p.early == 1) {
                __syncwarp();
                ptx::griddep_wait();
                ptx::griddep_launch_dependents();
            }
            // K tile tk once its stage's previous K is consumed, up to kSwapKLead tiles ahead of
            // the V stream; otherwise V tile tv once its stage's previous V is.
            while (ok && tv < T) {
                if (tk < T && tk <= tv + kSwapKLead) {
                    const int s = tk % STAGES;
                    if (tk >= STAGES && !wait_bounded(wc, bar(kKEmpty + s), ((tk / STAGES) & 1u) ^ 1u, kKEmpty + s))
                        ok = false;
                    else
                        issue_k(tk++);
                } else {
                    const int s = tv % STAGES;
                    if (tv >= STAGES &&
                        !wait_bounded(wc, bar(BI::kKvEmpty + s), ((tv / STAGES) & 1u) ^ 1u, BI::kKvEmpty + s))
                        ok = false;
                    else
                        issue_v(tv++);
                }
            }
            // The releases of the last stages land before the CTA exits.
            for (int u = T - STAGES > 0 ? T - STAGES : 0; ok && u < T; ++u) {
                const uint32_t ph = static_cast<uint32_t>(u / STAGES) & 1u;
                ok = wait_bounded(wc, bar(kKEmpty + u % STAGES), ph, kKEmpty + u % STAGES) &&
                     wait_bounded(wc, bar(BI::kKvEmpty + u % STAGES), ph, BI::kKvEmpty + u % STAGES);
            }
            if (*abort_flag) {
                if (q_armed)
                    wait_drain(bar(BI::kQFull), 0, p.timeout_ns);
#pragma unroll
                for (int s = 0; s < STAGES; ++s) {
                    if (armed_k[s] > 0)
                        wait_drain(bar(BI::kKFull + s), static_cast<uint32_t>(armed_k[s] - 1) & 1u, p.timeout_ns);
                    if (armed_v[s] > 0)
                        wait_drain(bar(BI::kVFull + s), static_cast<uint32_t>(armed_v[s] - 1) & 1u, p.timeout_ns);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- S^T = K^T . Q^T issuer
        // A = K^T: M-major (keys contiguous), the two 64-key halves D*128 B apart, 8-row groups
        // along d 1024 B apart, 16 d-rows (2048 B) per k-step. B = Q^T: K-major (d contiguous), 16
        // query rows, 64-column chunks kSwapChunk apart, 16-column steps 32 B inside a swizzle row.
        constexpr uint32_t idesc_s = ptx::idesc_f16_f32(kBlockN, kSwapNQ, true, false);
        uint64_t b_q[D / 16];
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
            b_q[k] = ptx::sdesc_sw128(sQ + (k >> 2) * kSwapChunk + (k & 3) * 32, 16, 1024);
        auto warp_wait = [&](uint32_t b_, uint32_t parity, int where) -> bool {
            return __all_sync(0xffffffffu, wait_bounded(wc, b_, parity, where));
        };
        bool ok = warp_wait(bar(BI::kQFull), 0, BI::kQFull);
        for (int u = 0; ok && u < T; ++u) {
            const int s = u % STAGES;
            const int sb = u & 1;
            if (!warp_wait(bar(BI::kKFull + s), static_cast<uint32_t>(u / STAGES) & 1u, BI::kKFull + s) ||
                (u >= 2 &&
                 !warp_wait(bar(BI::kSEmpty + sb), (static_cast<uint32_t>(u >> 1) & 1u) ^ 1u, BI::kSEmpty + sb))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint64_t a_k = ptx::sdesc_sw128(sStage0 + s * kSwapStageBytes, D * 128, 1024);
            if (ptx::elect_one()) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    ptx::mma_f16_ss(tmem + sb * kSwapNQ, a_k + static_cast<uint64_t>(k * (2048 >> 4)), b_q[k], idesc_s,
                                    k > 0 ? 1u : 0u);
                ptx::mma_commit(bar(BI::kSFull + sb));
                ptx::mma_commit(bar(kKEmpty + s));
            }
            __syncwarp();
        }
        if (ptx::elect_one()) {
            ptx::mma_commit(bar(BI::kDrain));
            wait_drain(bar(BI::kDrain), 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ---------------------------------------------------------------- O^T += V^T . P^T issuer
        // A = V^T: M-major (d contiguous), the two 64-column halves 128 rows x 128 B apart, 16 keys
        // (2048 B) per k-step. B = P^T: K-major (keys contiguous), 16 query rows, 64-key chunks
        // kSwapChunk apart.
        constexpr uint32_t idesc_o = ptx::idesc_f16_f32(D, kSwapNQ, true, false);
        auto warp_wait = [&](uint32_t b_, uint32_t parity, int where) -> bool {
            return __all_sync(0xffffffffu, wait_bounded(wc, b_, parity, where));
        };
        bool ok = true;
        for (int v = 0; ok && v < T; ++v) {
            const int pb = v % kSwapPBuffers;
            const int s = v % STAGES;
            if (!(warp_wait(bar(BI::kVFull + s), static_cast<uint32_t>(v / STAGES) & 1u, BI::kVFull + s) &&
                  warp_wait(bar(BI::kPFull + pb), static_cast<uint32_t>(v / kSwapPBuffers) & 1u, BI::kPFull + pb))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint64_t a_v =
                ptx::sdesc_sw128(sStage0 + s * kSwapStageBytes + D * kBlockN * 2, TileCfg<D>::kChunkRows128, 1024);
            const uint32_t sP = sP0 + pb * kSwapPBytes;
            // ONLINE: tile v accumulates into its group's O^T (columns 32 + 16 (v mod 2)), from its
            // group's first tile on.
            const uint32_t o_col = ONLINE ? kSwapTmemO + (v & 1) * kSwapNQ : kSwapTmemO;
            const int first = ONLINE ? 2 : 1;
            if (ptx::elect_one()) {
#pragma unroll
                for (int k = 0; k < kBlockN / 16; ++k)
                    ptx::mma_f16_ss(tmem + o_col, a_v + static_cast<uint64_t>(k * (2048 >> 4)),
                                    ptx::sdesc_sw128(sP + (k >> 2) * kSwapChunk + (k & 3) * 32, 16, 1024), idesc_o,
                                    (v >= first || k > 0) ? 1u : 0u);
                ptx::mma_commit(bar(BI::kKvEmpty + s));
                ptx::mma_commit(bar(BI::kPEmpty + pb));
                if (v == T - 1)
                    ptx::mma_commit(bar(BI::kOFull));
            }
            __syncwarp();
        }
        if (ok) {
            for (int u = T - kSwapPBuffers > 0 ? T - kSwapPBuffers : 0; ok && u < T; ++u)
                ok = warp_wait(bar(BI::kPEmpty + u % kSwapPBuffers), static_cast<uint32_t>(u / kSwapPBuffers) & 1u,
                               BI::kPEmpty + u % kSwapPBuffers);
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
        const int sw = warp - 2;
        const int q4 = warp & 3;
        const int g = sw >> 2;
        const int key = q4 * 32 + lane;  // this thread's key (tensor-memory lane) within a tile
        const uint32_t lane_addr = static_cast<uint32_t>(q4 * 32) << 16;
        auto warp_wait = [&](uint32_t b_, uint32_t parity, int where) -> bool {
            return __all_sync(0xffffffffu, wait_bounded(wc, b_, parity, where));
        };
        const ptx::ExpPairConsts ek = ptx::exp_pair_consts();
        float lq[kSwapNQ];  // this thread's part of each query row's sum (its keys, fp32)
#pragma unroll
        for (int q = 0; q < kSwapNQ; ++q)
            lq[q] = 0.f;
        // P^T element (query q, key) in its buffer: 64-key chunk, row q, the 128-byte swizzle.
        const uint32_t p_off = (key / 64) * kSwapChunk + (((static_cast<uint32_t>(key % 64) / 8) << 4) | ((key % 8) * 2));
        bool ok = true;
        float mrun[kSwapNQ];  // ONLINE: the group's running maximum of each query row
#pragma unroll
        for (int q = 0; q < kSwapNQ; ++q)
            mrun[q] = -INFINITY;
        if constexpr (ONLINE) {
            const int wq = sw & 3;  // warp within the group
            float *m_red_g = m_red + g * 2 * kGroupWarps * kSwapNQ;
            // Barrier ids stay compile-time constants (one branch per group).
            auto group_barrier_and = [&](bool pred) {
                return g == 0 ? ptx::named_barrier_and(kGroupBarrier0, kGroupWarps * 32, pred)
                              : ptx::named_barrier_and(kGroupBarrier0 + 1, kGroupWarps * 32, pred);
            };
            auto group_barrier_or = [&](bool pred) {
                return g == 0 ? ptx::named_barrier_or(kGroupBarrier0, kGroupWarps * 32, pred)
                              : ptx::named_barrier_or(kGroupBarrier0 + 1, kGroupWarps * 32, pred);
            };
            // exp(s - m) for queries q and q + 1 as one packed multiply-add: -m log2(e) in each half.
            uint64_t shift[kSwapNQ / 2];
#pragma unroll
            for (int q = 0; q < kSwapNQ / 2; ++q)
                shift[q] = 0;
            // QK-norm: the query scales a_q = 1/rms(Q[q, :]), 16 threads of the softmax warps per
            // query row, one 16-byte unit (8 columns) each, a 4-step sum over those 16 lanes; one
            // barrier of all softmax warps publishes them in shared memory (and ANDs the wait for
            // Q), where each tile reads them again (fewer registers live in the loop).
            // QK-norm, key scales: this lane's unit (8 keys) of the warp's 32 and its d-rows kr,
            // kr + 8, ... (kr alternates between the swizzle pattern's halves, so a quarter-warp's
            // eight loads hit eight distinct bank groups); after the reduce-scatter a lane holds
            // key 8 (lane & 3) + 4 bit4 + 2 bit3 + bit2 of the warp's, and one shuffle brings each
            // lane its own key's (key q4 * 32 + lane).
            const int kr = (((lane >> 2) & 1) << 2) | (lane >> 3);
            const uint32_t unit_phys = (static_cast<uint32_t>(((q4 & 1) << 2) | (lane & 3))) ^ static_cast<uint32_t>(kr);
            const int c_src = (lane >> 3) | ((lane & 1) << 2) | (((lane >> 1) & 1) << 3) | (((lane >> 2) & 1) << 4);
            if constexpr (QKN) {
                const int i = threadIdx.x - 64;  // 0 .. 255
                const int qr = i >> 4, part = i & 15;
                bool q_ok = warp_wait(bar(BI::kQFull), 0, BI::kQFull);
                float ss[2] = {0.f, 0.f};
                if (q_ok)
                    sum_sq_unit(*reinterpret_cast<const uint4 *>(smem + (part >> 3) * kSwapChunk + qr * 128 +
                                                                 (((part & 7) ^ (qr & 7)) << 4)),
                                ss);
                float t = ss[0] + ss[1];
#pragma unroll
                for (int o = 8; o >= 1; o >>= 1)
                    t += __shfl_xor_sync(0xffffffffu, t, o);
                if (part == 0)
                    a_sc[qr] = __frsqrt_rn(t * (1.f / D) + kQkNormEps);
                if (!ptx::named_barrier_and(kSoftmaxBarrier, kSoftmaxThreads, q_ok))
                    ok = false;
            }
            // Every warp of the group takes the same group barriers per tile, so all run the same
            // iterations: a failed wait clears `ok`, and the next barriers (or the epilogue's) stop
            // the others too.
            for (int u = g; u < T; u += 2) {
                const int pb = u % kSwapPBuffers;
                const int mb = (u >> 1) & 1;  // buffer of the tile maxima
                const bool valid = tile_of(u) * kBlockN + key < p.N;  // keys past N weigh 0
                uint32_t r[kSwapNQ];
                bool w_ok = ok;
                float cn = 1.f;  // QK-norm: this thread's key scale c_n = 1/rms(K[:, n])
                if constexpr (QKN) {
                    // From the K tile in shared memory, while the tensor core computes S^T; each
                    // warp's read is one of the arrivals that release the tile's K half.
                    const int st = u % STAGES;
                    w_ok = w_ok && warp_wait(bar(BI::kKFull + st), static_cast<uint32_t>(u / STAGES) & 1u, BI::kKFull + st);
                    if (w_ok) {
                        const uint8_t *kp = smem + (sStage0 - sQ) + st * kSwapStageBytes + (q4 >> 1) * (D * 128) +
                                            kr * 128 + (unit_phys << 4);
                        float sq[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int k = 0; k < D / 8; ++k)  // d-row kr + 8k
                            sum_sq_cols(*reinterpret_cast<const uint4 *>(kp + k * 1024), sq);
                        const float c = __frsqrt_rn(reduce_scatter8(sq, lane) * (1.f / D) + kQkNormEps);
                        cn = __shfl_sync(0xffffffffu, c, c_src);
                        if (lane == 0)  // every lane's loads are in c (the shuffles above)
                            ptx::mbar_arrive(bar(kKEmpty + st));
                    }
                }
                w_ok = w_ok && warp_wait(bar(BI::kSFull + g), static_cast<uint32_t>(u >> 1) & 1u, BI::kSFull + g);
                bool over = false;  // a score of this warp past its row's maximum by more than the slack
                if (w_ok) {
                    ptx::tc_fence_after();
                    ptx::tmem_ld_32x32b_x16(tmem + lane_addr + g * kSwapNQ, r);
                    ptx::tmem_ld_wait16(r);
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        ptx::mbar_arrive(bar(BI::kSEmpty + g));
                    if constexpr (QKN) {
#pragma unroll
                        for (int k = 0; k < kSwapNQ / 4; ++k) {  // the normalised scores, a_q c_n S^T[n, q]
                            const float4 a = reinterpret_cast<const float4 *>(a_sc)[k];
                            r[4 * k + 0] = __float_as_uint(__uint_as_float(r[4 * k + 0]) * (cn * a.x));
                            r[4 * k + 1] = __float_as_uint(__uint_as_float(r[4 * k + 1]) * (cn * a.y));
                            r[4 * k + 2] = __float_as_uint(__uint_as_float(r[4 * k + 2]) * (cn * a.z));
                            r[4 * k + 3] = __float_as_uint(__uint_as_float(r[4 * k + 3]) * (cn * a.w));
                        }
                    }
#pragma unroll
                    for (int q = 0; q < kSwapNQ; ++q)
                        over |= valid && __uint_as_float(r[q]) > mrun[q] + kSwapRescaleSlack;
                    over = __any_sync(0xffffffffu, over);
                }
                // One group barrier per tile tells every warp whether some warp failed a wait or
                // must raise the maximum (always on the group's first tile: m = -inf). Only then
                // do the tile's maxima go through shared memory, behind a second barrier.
                float alpha[kSwapNQ];
                bool changed = false;
                if (group_barrier_or(!w_ok || over)) {
                    if (w_ok) {
                        float t[kSwapNQ];
#pragma unroll
                        for (int q = 0; q < kSwapNQ; ++q)
                            t[q] = valid ? __uint_as_float(r[q]) : -INFINITY;
                        const float wmax = warp_max16(t, lane);
                        if ((lane & 1) == 0)
                            m_red_g[(mb * kGroupWarps + wq) * kSwapNQ + (lane >> 1)] = wmax;
                    }
                    if (!group_barrier_and(w_ok)) {
                        ok = false;
                        break;
                    }
                    // The tile's maximum of every query over the group's 128 keys (at least one key
                    // of a tile is below N, so it is finite), and the new maxima.
#pragma unroll
                    for (int q = 0; q < kSwapNQ; ++q)
                        alpha[q] = -INFINITY;
#pragma unroll
                    for (int w = 0; w < kGroupWarps; ++w) {
                        const float4 *row =
                            reinterpret_cast<const float4 *>(m_red_g + (mb * kGroupWarps + w) * kSwapNQ);
#pragma unroll
                        for (int k = 0; k < kSwapNQ / 4; ++k) {
                            const float4 x = row[k];
                            alpha[4 * k + 0] = fmaxf(alpha[4 * k + 0], x.x);
                            alpha[4 * k + 1] = fmaxf(alpha[4 * k + 1], x.y);
                            alpha[4 * k + 2] = fmaxf(alpha[4 * k + 2], x.z);
                            alpha[4 * k + 3] = fmaxf(alpha[4 * k + 3], x.w);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < kSwapNQ; ++q)
                        changed |= alpha[q] > mrun[q] + kSwapRescaleSlack;
                    if (changed) {  // the same on every thread of the group
#pragma unroll
                        for (int q = 0; q < kSwapNQ; ++q) {
                            const float mn = fmaxf(mrun[q], alpha[q]);
                            alpha[q] = ptx::ex2_approx((mrun[q] - mn) * ptx::kLog2e);  // 0 on the first tile
                            lq[q] *= alpha[q];
                            mrun[q] = mn;
                        }
#pragma unroll
                        for (int q = 0; q < kSwapNQ; q += 2)
                            shift[q / 2] = (static_cast<uint64_t>(__float_as_uint(-mrun[q + 1] * ptx::kLog2e)) << 32) |
                                           __float_as_uint(-mrun[q] * ptx::kLog2e);
                    }
                }
                if (u >= kSwapPBuffers &&
                    !warp_wait(bar(BI::kPEmpty + pb), (static_cast<uint32_t>(u / kSwapPBuffers) & 1u) ^ 1u,
                               BI::kPEmpty + pb))
                    ok = false;
                if (ok) {
                    uint8_t *pt = smem + kSwapQBytes + pb * kSwapPBytes;
#pragma unroll
                    for (int q = 0; q < kSwapNQ; q += 2) {
                        uint32_t e0, e1;
                        ptx::exp_pair_mufu(r[q], r[q + 1], ek, shift[q / 2], e0, e1);
                        e0 = valid ? e0 : 0u;
                        e1 = valid ? e1 : 0u;
                        lq[q] += __uint_as_float(e0);
                        lq[q + 1] += __uint_as_float(e1);
                        *reinterpret_cast<__half *>(pt + (p_off ^ ((q & 7) << 4)) + q * 128) =
                            __float2half_rn(__uint_as_float(e0));
                        *reinterpret_cast<__half *>(pt + (p_off ^ (((q + 1) & 7) << 4)) + (q + 1) * 128) =
                            __float2half_rn(__uint_as_float(e1));
                    }
                }
                // Rescale the group's O^T (its lanes = output columns, its columns = queries) once
                // the tensor core has finished the group's previous P.V, before this tile's P.V.
                if (ok && changed && u >= 2) {
                    const int q2 = u - 2;
                    if (warp_wait(bar(BI::kPEmpty + q2 % kSwapPBuffers),
                                  static_cast<uint32_t>(q2 / kSwapPBuffers) & 1u, BI::kPEmpty + q2 % kSwapPBuffers)) {
                        ptx::tc_fence_after();
                        uint32_t o[kSwapNQ];
                        const uint32_t taddr = tmem + lane_addr + kSwapTmemO + g * kSwapNQ;
                        ptx::tmem_ld_32x32b_x16(taddr, o);
                        ptx::tmem_ld_wait16(o);
#pragma unroll
                        for (int q = 0; q < kSwapNQ; ++q)
                            o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha[q]);
                        swap_tmem_st_x16(taddr, o);
                        ptx::tmem_st_wait();
                    } else {
                        ok = false;
                    }
                }
                if (ok) {
                    ptx::fence_proxy_async_smem();  // the tensor core reads P^T through the async proxy
                    ptx::tc_fence_before();         // and the rescaled O^T after the arrival
                    __syncwarp();
                    if (lane == 0)
                        ptx::mbar_arrive(bar(BI::kPFull + pb));
                }
            }
        } else {
        for (int u = g; ok && u < T; u += 2) {
            const int pb = u % kSwapPBuffers;
            if (!warp_wait(bar(BI::kSFull + g), static_cast<uint32_t>(u >> 1) & 1u, BI::kSFull + g)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            uint32_t r[kSwapNQ];
            ptx::tmem_ld_32x32b_x16(tmem + lane_addr + g * kSwapNQ, r);
            ptx::tmem_ld_wait16(r);
            // S^T is in registers: the buffer can take this group's next tile.
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(bar(BI::kSEmpty + g));
            if (u >= kSwapPBuffers &&
                !warp_wait(bar(BI::kPEmpty + pb), (static_cast<uint32_t>(u / kSwapPBuffers) & 1u) ^ 1u, BI::kPEmpty + pb)) {
                ok = false;
                break;
            }
            const bool valid = tile_of(u) * kBlockN + key < p.N;  // keys past N weigh 0
            uint8_t *pt = smem + kSwapQBytes + pb * kSwapPBytes;
#pragma unroll
            for (int q = 0; q < kSwapNQ; q += 2) {
                uint32_t e0, e1;
                ptx::exp_pair_mufu(r[q], r[q + 1], ek, 0, e0, e1);
                e0 = valid ? e0 : 0u;
                e1 = valid ? e1 : 0u;
                lq[q] += __uint_as_float(e0);
                lq[q + 1] += __uint_as_float(e1);
                // Rows q and q + 1 of the 128-byte swizzle: unit index XOR row mod 8.
                *reinterpret_cast<__half *>(pt + (p_off ^ ((q & 7) << 4)) + q * 128) = __float2half_rn(__uint_as_float(e0));
                *reinterpret_cast<__half *>(pt + (p_off ^ (((q + 1) & 7) << 4)) + (q + 1) * 128) =
                    __float2half_rn(__uint_as_float(e1));
            }
            ptx::fence_proxy_async_smem();  // the tensor core reads P^T through the async proxy
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(bar(BI::kPFull + pb));
        }
        }

        // ------------------------------------------------------------ epilogue
        // Row sums: each warp adds its 32 keys' parts (the same butterfly order on every lane), the
        // eight warps' sums meet in shared memory and add in warp order.
#pragma unroll
        for (int q = 0; q < kSwapNQ; ++q) {
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                lq[q] += __shfl_xor_sync(0xffffffffu, lq[q], o);
        }
        if (lane == 0) {
#pragma unroll
            for (int q = 0; q < kSwapNQ; ++q)
                l_red[sw * kSwapNQ + q] = lq[q];
            if (ONLINE && sw == kGroupWarps) {  // group 1's maxima, for group 0's merge
#pragma unroll
                for (int q = 0; q < kSwapNQ; ++q)
                    m_fin[q] = mrun[q];
            }
        }
        const bool o_ready = ptx::named_barrier_and(kSoftmaxBarrier, kSoftmaxThreads,
                                                    ok && warp_wait(bar(BI::kOFull), 0, BI::kOFull));
        float *stage_o = reinterpret_cast<float *>(smem + (sStage0 - sQ));  // [16][128]
        float *stage_l = stage_o + kSwapNQ * D;                                // [16]
        float *stage_m = stage_l + kSwapNQ;                                    // [16] (ONLINE)
        if (o_ready && g == 0) {
            // O^T lanes are output columns: the four warps of group 0 cover all 128.
            ptx::tc_fence_after();
            uint32_t o[kSwapNQ];
            ptx::tmem_ld_32x32b_x16(tmem + lane_addr + kSwapTmemO, o);
            ptx::tmem_ld_wait16(o);
            // ONLINE: group 1's accumulator (written only when the CTA has a second tile).
            const bool two = ONLINE && T >= 2;
            uint32_t o1[kSwapNQ];
            if (two) {
                ptx::tmem_ld_32x32b_x16(tmem + lane_addr + kSwapTmemO + kSwapNQ, o1);
                ptx::tmem_ld_wait16(o1);
            }
            const int c = q4 * 32 + lane;  // output column
            const int mq = p.M < kSwapNQ ? p.M : kSwapNQ;
            if (p.early == 2 && !p.cluster_reduce)
                ptx::griddep_wait();  // O or the partials are written below
#pragma unroll
            for (int q = 0; q < kSwapNQ; ++q) {
                if (q < mq) {
                    float l = 0.f;
                    float ov = __uint_as_float(o[q]);
                    float m = 0.f;
                    if constexpr (ONLINE) {
                        // Both groups' parts relative to the larger of their maxima.
                        float l0 = 0.f, l1 = 0.f;
#pragma unroll
                        for (int w = 0; w < kGroupWarps; ++w) {
                            l0 += l_red[w * kSwapNQ + q];
                            l1 += l_red[(kGroupWarps + w) * kSwapNQ + q];
                        }
                        m = two ? fmaxf(mrun[q], m_fin[q]) : mrun[q];
                        const float w0 = ptx::ex2_approx((mrun[q] - m) * ptx::kLog2e);
                        l = l0 * w0;
                        ov *= w0;
                        if (two) {
                            const float w1 = ptx::ex2_approx((m_fin[q] - m) * ptx::kLog2e);
                            l = fmaf(l1, w1, l);
                            ov = fmaf(__uint_as_float(o1[q]), w1, ov);
                        }
                    } else {
#pragma unroll
                        for (int w = 0; w < kSoftmaxWarps; ++w)
                            l += l_red[w * kSwapNQ + q];
                    }
                    if (p.n_split == 1) {
                        p.O[(static_cast<size_t>(b) * p.M + q) * D + c] = __float2half_rn(ov * __frcp_rn(l));
                    } else if (p.cluster_reduce) {
                        // Staged for the cluster's owners (the K/V ring is idle): O^T column c of
                        // query q, fp32, the row sum of q and (ONLINE) the maximum they are relative to.
                        stage_o[q * D + c] = ov;
                        if (c == 0) {
                            stage_l[q] = l;
                            if (ONLINE)
                                stage_m[q] = m;
                        }
                    } else {
                        const size_t r = (static_cast<size_t>(j) * p.B + b) * p.M + q;
                        p.ws_o[r * D + c] = ov;
                        if (c == 0) {
                            p.ws_l[r] = l;
                            if (ONLINE)
                                p.ws_m[r] = m;
                        }
                    }
                }
            }
        }
    }

    // On-chip combine (the n_split CTAs of a batch in one thread-block cluster, rank j): after a
    // cluster barrier every CTA's staged fp32 O^T and row sums are visible; rank j forms columns
    // [128 j / n, 128 (j + 1) / n) of every query row as sum_r O_r / sum_r l_r over the ranks in
    // rank order and writes fp16 O; a second barrier keeps each CTA's shared memory alive until
    // the others have read it. Every thread of every CTA reaches both barriers, on the unwinding
    // path too (a CTA that unwound staged nothing: O is then undefined, as the status says).
    __syncwarp();
    if (p.cluster_reduce) {
        ptx::cluster_sync();
        if (warp >= 2 && warp < 2 + kSoftmaxWarps) {
            const int n = p.n_split;
            const int c_lo = j * D / n;
            const int cols = (j + 1) * D / n - c_lo;
            const int mq = p.M < kSwapNQ ? p.M : kSwapNQ;
            const uint32_t so = ptx::smem_u32(smem) + (sStage0 - sQ);
            const uint32_t sl = so + kSwapNQ * D * 4;
            const uint32_t sm = sl + kSwapNQ * 4;
            for (int it = threadIdx.x - 64; it < mq * cols; it += kSoftmaxThreads) {
                const int q = it / cols;
                const int c = c_lo + it % cols;
                // ONLINE: rank r's partial is relative to its maximum m_r; weights exp(m_r - max m).
                float wt[kMaxClusterRanks];
#pragma unroll
                for (int r = 0; r < kMaxClusterRanks; ++r)
                    wt[r] = 1.f;
                if constexpr (ONLINE) {
                    float mmax = -INFINITY;
#pragma unroll
                    for (int r = 0; r < kMaxClusterRanks; ++r) {
                        if (r < n) {
                            wt[r] = ptx::ld_cluster_f32(ptx::map_to_rank(sm + static_cast<uint32_t>(q) * 4, r));
                            mmax = fmaxf(mmax, wt[r]);
                        }
                    }
#pragma unroll
                    for (int r = 0; r < kMaxClusterRanks; ++r)
                        if (r < n)
                            wt[r] = ptx::ex2_approx((wt[r] - mmax) * ptx::kLog2e);
                }
                float ov[kMaxClusterRanks], lv[kMaxClusterRanks];
#pragma unroll
                for (int r = 0; r < kMaxClusterRanks; ++r) {  // every load in flight before the sums
                    if (r < n) {
                        ov[r] = ptx::ld_cluster_f32(ptx::map_to_rank(so + static_cast<uint32_t>(q * D + c) * 4, r));
                        lv[r] = ptx::ld_cluster_f32(ptx::map_to_rank(sl + static_cast<uint32_t>(q) * 4, r));
                    }
                }
                float os = 0.f, ls = 0.f;
#pragma unroll
                for (int r = 0; r < kMaxClusterRanks; ++r) {
                    if (r < n) {
                        if constexpr (ONLINE) {
                            os = fmaf(ov[r], wt[r], os);
                            ls = fmaf(lv[r], wt[r], ls);
                        } else {
                            os += ov[r];
                            ls += lv[r];
                        }
                    }
                }
                if (p.early == 2)
                    ptx::griddep_wait();
                p.O[(static_cast<size_t>(b) * p.M + q) * D + c] = __float2half_rn(os * __frcp_rn(ls));
            }
        }
        ptx::cluster_sync_relaxed();
    }

    // Teardown: every tensor-memory access of the CTA is ordered before the free.
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kSwapTmemCols);
    }
}

}  // namespace mg
