// mg_attn_kernels.cuh -- the fused device kernel of the exp-normalised GQA graph.
//
// Graph (Mirage documentation, tutorials/group-query-attention, "Define GQA Computation
// Graph"): A = matmul(Q,K); E = exp(A); S = reduction(E,2); D = div(E,S); O = matmul(D,V).
//
// Kernel 1, mg_attn_fwd_partial: one CTA per (batch b, 128-row tile of Q, split j of the N
// axis). Split j owns the 128-column tiles j, j + n_split, j + 2 n_split, ... of K/V and loops
// over them, as the threadblock for-loop over N with a row-sum accumulator does in Mirage's attention
// search space (blog "Reading Mirage's muGraph search and backend generation through the
// GQA example", sections 4.2-4.3: forloop dims and the REDTOX_LD_SUM accumulator). Per tile:
//     S  = Q . K_tile                    tcgen05 MMA, fp32 in tensor memory
//     P  = exp(S) (0 beyond N)           fp32; l += rowsum(P) in fp32; fp16 P to tensor memory
//     O += fp16(P) . V_tile              tcgen05 MMA with A read from tensor memory
// The divide by the row sum commutes with the second product, so it is deferred.
// With one split the CTA divides and writes fp16 O (TMA store). With 2..16 splits that fit one
// wave, the splits of a row tile form a thread-block cluster and combine on chip (distributed
// shared memory, fixed rank order). Otherwise each writes the fp32 partial numerator O_j and row
// sum l_j to the workspace (TMA store) for kernel 2.
//
// Kernel 2 (mg_combine.cuh): O = (sum_j O_j) / (sum_j l_j) -> fp16, the second threadblock
// graph of the "attention" search configuration (blog, section 4.3). No max-subtraction
// means the partials combine by plain sums (weights exp(m_j - max m) in the max-subtracted
// variant).
//
// Variants (template parameter VAR): the graph as written, under the split schedule or under the
// stream-K schedule (CTAs share the (batch, column tile) units in equal runs; see kStreamK);
// max-subtracted (a first pass over the split's K tiles finds each row's maximum score m, then
// P = exp(S - m)); QK-norm (scores scaled by query-row and key-vector scales 1/rms,
// max-subtracted; the softmax warps compute the key-vector scales in the first pass from the K
// tiles it streams, and the query-row scales from the Q tile).
//
// Warp roles of kernel 1 (352 threads):
//   warp 0       TMA producer: Q once, then K/V tiles through a STAGES-deep mbarrier ring
//   warp 1       tensor-memory allocator; issues S = Q.K (elected lane)
//   warp 10      issues O += P.V (elected lane); two issuing warps keep an S from waiting
//                behind a P.V and the reverse
//   warps 2..9   softmax + epilogue, two groups of four: group g = (w-2)/4 takes the tiles
//                t with t % 2 == g, in S buffer g, all 128 columns of its rows; warp w reads
//                tensor-memory lanes 32*(w%4).. (its rows). In the epilogue group g takes
//                O columns [g d/2, (g+1) d/2).
// Tensor memory (512 columns): S buffers at columns [0,128) (group 0) and [128,256) (group 1),
// O at [256, 256 + d), then the fp16 P buffers (64 columns each, two fp16 per column): three
// for d = 64, two for d = 128, so the softmax warps can run ahead of the P.V products.
// Keeping P in tensor memory spares shared memory 64 KB of traffic per tile (P written by the
// softmax warps and read back by the MMA).
//
// Exponentials: ex2.approx on the MUFU unit after one two-wide fp32 fused multiply-add
// s*log2(e) - m*log2(e) per pair of columns (m = 0 for the graph as written). A polynomial path on the FMA pipe (exp_pair_fma, same fp32 accuracy) can take
// kPolyOf8 of every 8 columns; measured on GB300 (mg_diag_exp_rate), this sequence runs 32
// exponentials per clock per SM on MUFU and 13 on the FMA pipe, so the split is 0.
//
// Every wait is bounded by a global-timer deadline. A wait that runs out records
// MG_ERR_TIMEOUT in the status word, raises a CTA-wide abort flag, and every role then
// stops, drains the copies/MMAs it issued (again bounded), frees tensor memory and returns.
#pragma once

#include <cmath>
#include <cstdint>
#include <type_traits>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace mg {

constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kSoftmaxWarps = 8;
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kGroupWarps = kSoftmaxWarps / 2;  // softmax warps per group (one tile each)
constexpr int kThreads = 96 + kSoftmaxThreads;  // load warp, S warp, 8 softmax warps, P.V warp
constexpr int kPvWarp = kThreads / 32 - 1;
constexpr uint32_t kTmemCols = 512;
constexpr int kPolyOf8 = 0;        // columns (of every 8, even) whose exp runs on the FMA pipe
constexpr uint32_t kTmemO = 256;   // tensor-memory column of O; P buffers follow it
constexpr int kStatusTimeout = 7;  // MG_ERR_TIMEOUT
constexpr uint32_t kSoftmaxBarrier = 1;  // named barrier id of the softmax warps
constexpr int kMaxClusterRanks = 16;     // largest cluster of the on-chip combine
constexpr float kQkNormEps = 1e-6f;      // rms_norm epsilon of the QK-norm variant
constexpr uint32_t kGroupBarrier0 = 2;   // named barrier ids 2, 3: the four warps of softmax group 0, 1
// On-chip combine: a normalised partial value |x| below this is exchanged as fp16 alone (its rounding,
// at most 2^-10 here, is half the 2e-3 error bound); for a 32-column slice of a row with any larger
// value the reader also adds each value's fp16 remainder x - fp16(x), which restores close to fp32
// precision.
constexpr float kHiOnlyBelow = 4.0f;

template <int D>
struct TileCfg {
    static_assert(D == 64 || D == 128, "head dim must be 64 or 128");
    static constexpr int kChunks = D / 64;                  // 128-byte column chunks of a d-wide fp16 row
    static constexpr uint32_t kQBytes = kBlockM * D * 2;    // Q tile, K-major
    static constexpr uint32_t kKBytes = D * kBlockN * 2;    // K tile, N contiguous
    static constexpr uint32_t kVBytes = kBlockN * D * 2;    // V tile, d contiguous
    static constexpr uint32_t kStageBytes = kKBytes + kVBytes;
    static constexpr uint32_t kChunkRows128 = 128 * 128;        // one 128-row x 128-byte chunk
    static constexpr int kHalfCols = D / 2;                     // O columns per epilogue thread
    static constexpr uint32_t kTmemP = kTmemO + D;              // P buffer b at kTmemP + 64 b
    // P buffers: as many as tensor memory holds after S (2 x 128 columns) and O (d columns).
    static constexpr int kPBuffers = D == 64 ? 3 : 2;
    static_assert(kTmemP + 64 * kPBuffers <= kTmemCols, "tensor memory overflow");
    // On-chip combine staging, per row: fp16 x = O_j / l_j and its remainders (d + 8 halves each,
    // the pad keeping 8 consecutive rows on distinct banks), then kLmw floats: the row sum once per
    // 32-column slice (its sign bit says whether that slice's remainders are staged), the row
    // maximum, padding to 16 bytes.
    static constexpr int kRowHalves = D + 8;
    static constexpr int kLmw = D == 64 ? 4 : 8;
    // Receive area of the pushed exchange: a slot of ceil(128 / n) rows for each of the n ranks
    // (at most 140 rows in all for n <= 16), each row as staged.
    static constexpr uint32_t kRecvRows = 144;
    static constexpr uint32_t kRecvBytes = kRecvRows * (2u * kRowHalves * 2 + kLmw * 4);
};

// Shared-memory bytes of kernel 1 for a head dim and pipeline depth: alignment slack, Q, the
// K/V ring (its first stages are reused as the output staging area), the receive area of the
// pushed exchange (only with it), the row-sum exchange of the two softmax groups and the barriers.
__host__ __device__ constexpr uint32_t fwd_smem_bytes(int d, int stages, bool push = false)
{
    return 1024u + static_cast<uint32_t>(128 * d * 2) + static_cast<uint32_t>(stages) * (2u * d * 128 * 2) +
           (push ? (d == 64 ? TileCfg<64>::kRecvBytes : TileCfg<128>::kRecvBytes) : 0u) + 2u * 128 * 4 + 512u;
}

struct FwdParams {
    int B, M, N;
    int m_tiles_per_b;       // ceil(M / 128)
    int n_tiles;             // ceil(N / 128)
    int n_split;
    int cluster_reduce;      // the n_split CTAs of a row tile form a cluster and combine on chip
    __half *O;               // (B, M, d) fp16 output (written directly by the cluster reduction)
    float *ws_o;             // (n_split, B, M, d) partial numerators (the cluster combine's plain stores)
    float *ws_l;             // (n_split, B, M) partial row sums
    float *ws_m;             // (n_split, B, M) partial row maxima (max-subtracted variant only)
    float *col_scale;        // QK-norm: (B, N) key-vector scales 1/rms, written by the row-maximum
                             // pass and read by the main pass (+128 readable floats past the end)
    int *status;             // [0] sticky status, [1] which wait ran out
    unsigned long long timeout_ns;
    int inject_timeout;
    int early;               // what runs before the wait for the previous grid (the host found that no
                             // kernel that may still run writes Q, K or V): 0 nothing; 1 the load
                             // warp's Q and first STAGES K/V copies; 2 everything but the global
                             // writes, with the dependents released at the start (not with QK-norm's
                             // key scales in global memory or the stream-K schedule, which write
                             // global memory midway)
    int cs_tiles;            // QK-norm: the CTA's key-vector scales kept in shared memory, this many
                             // tiles of 128 after the fixed layout (0: in col_scale, global memory)
    long long sk_units;      // stream-K: B * n_tiles units (row tile, column tile)
    int sk_ctas;             // stream-K: G, the grid
    int sk_slots;            // stream-K: partial slots per row tile (the second kernel's split count)
};

// Barrier indices inside the CTA's barrier array.
template <int STAGES, int kPBuffers>
struct Bars {
    static constexpr int kQFull = 0;
    static constexpr int kKFull = 1;                // K tile of a stage landed (the S warp waits)
    static constexpr int kVFull = kKFull + STAGES;  // V tile of a stage landed (the P.V warp waits)
    static constexpr int kKvEmpty = kVFull + STAGES;
    static constexpr int kSFull = kKvEmpty + STAGES;
    static constexpr int kSEmpty = kSFull + 2;
    static constexpr int kPFull = kSEmpty + 2;
    static constexpr int kPEmpty = kPFull + kPBuffers;
    static constexpr int kOFull = kPEmpty + kPBuffers;
    static constexpr int kDrain = kOFull + 1;      // unwinding: the S warp's MMAs
    static constexpr int kDrainPv = kDrain + 1;    // unwinding: the P.V warp's MMAs
    static constexpr int kNever = kDrainPv + 1;
    static constexpr int kXRecv = kNever + 1;      // pushed exchange: every rank's rows have landed here
    static constexpr int kCount = kXRecv + 1;
    // + the tensor-memory address and the abort flag
    static_assert(kCount * 8 + 8 <= 512, "barrier area overflow");
};

struct WaitCtx {
    volatile int *abort_flag;
    int *status;
    unsigned long long timeout_ns;
};

// Bounded parity wait. Returns false (and the caller unwinds) if the CTA is aborting or
// the deadline passes; the first waiter to time out records where.
__device__ __forceinline__ bool wait_bounded(const WaitCtx &w, uint32_t bar, uint32_t parity, int where)
{
    // Fast path: a phase that has already completed is seen by a plain test, without the
    // potentially-suspending try_wait.
    if (ptx::mbar_test_wait(bar, parity))
        return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
        // try_wait may suspend the thread for a hardware-chosen time while the phase is
        // incomplete, so waiting warps leave the issue slots to working ones. Measured on GB300
        // (µs per call): 1-2 % faster than with a 100 µs suspend-time hint (gqa 6.65 against
        // 6.77), and a test_wait spin is slower than both (it competes for issue slots).
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        if (*w.abort_flag)
            return false;
        if (ptx::globaltimer_ns() - t0 > w.timeout_ns) {
            *w.abort_flag = 1;
            ptx::griddep_wait();  // (early start, or an early load warp) global memory only after
                                  // the previous grid
            if (atomicCAS(w.status, 0, kStatusTimeout) == 0)
                atomicExch(w.status + 1, where);
            return false;
        }
    }
}

// Bounded wait used only while unwinding: ignores the abort flag.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, unsigned long long timeout_ns)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > timeout_ns)
            return;
    }
}

// Byte offset of 16-byte unit `unit` of row `row` inside a 128-row x 128-byte chunk written in
// the TMA/UMMA 128-byte swizzle (unit index XOR row mod 8).
__device__ __forceinline__ uint32_t sw128_offset(int row, uint32_t unit)
{
    return static_cast<uint32_t>(row) * 128u + ((unit ^ static_cast<uint32_t>(row & 7)) << 4);
}

// The exponentials of one 32-column slice of a score row, packed as fp16 pairs into w[16]:
// exp(s[i] - m) for columns below n_valid, 0 past N (MASK: only the last tile needs the test);
// `shift` holds -m*log2(e) twice (+0 for the graph as written, where m = 0). Pairs of columns go
// through the f32x2 pipe: the first kPolyOf8 of every 8 by the polynomial, the rest by MUFU.
// The fp32 values add into two packed partial row sums (fixed order).
template <bool MASK>
__device__ __forceinline__ void exp_slice(const uint32_t (&r)[32], int col0, int n_valid, uint32_t *w,
                                          uint64_t (&acc)[2], const ptx::ExpPairConsts &k, uint64_t shift)
{
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        uint32_t e0, e1;
        if ((i & 7) < kPolyOf8)
            ptx::exp_pair_fma(r[i], r[i + 1], k, e0, e1);
        else
            ptx::exp_pair_mufu(r[i], r[i + 1], k, shift, e0, e1);
        if (MASK) {
            e0 = (col0 + i < n_valid) ? e0 : 0u;
            e1 = (col0 + i + 1 < n_valid) ? e1 : 0u;
        }
        acc[(i >> 1) & 1] = ptx::add_pair(acc[(i >> 1) & 1], e0, e1);
        w[i / 2] = ptx::pack_half2(__uint_as_float(e0), __uint_as_float(e1));
    }
}

// Running maximum of the valid columns of a 32-column slice (MASK: columns at or past n_valid
// are left out).
template <bool MASK>
__device__ __forceinline__ float max_slice(const uint32_t (&r)[32], int col0, int n_valid, float m)
{
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float v = __uint_as_float(r[i]);
        m = (!MASK || col0 + i < n_valid) ? fmaxf(m, v) : m;
    }
    return m;
}

// QK-norm variant: as exp_slice and max_slice for the scores s * c_col * a, where `cs` holds the
// slice's 32 key-vector scales c (16-byte aligned, the same for every row) and `arow` is
// a*log2(e) twice (this row's query scale; for the maximum the caller applies a afterwards).
template <bool MASK>
__device__ __forceinline__ void exp_slice_scaled(const uint32_t (&r)[32], int col0, int n_valid, uint32_t *w,
                                                 uint64_t (&acc)[2], const float *cs, uint64_t arow, uint64_t shift)
{
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const float4 c4 = *reinterpret_cast<const float4 *>(cs + (i & ~3));
        const float2 c = (i & 2) ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y);
        uint32_t e0, e1;
        ptx::exp_pair_mufu_scaled(r[i], r[i + 1], c.x, c.y, arow, shift, e0, e1);
        if (MASK) {
            e0 = (col0 + i < n_valid) ? e0 : 0u;
            e1 = (col0 + i + 1 < n_valid) ? e1 : 0u;
        }
        acc[(i >> 1) & 1] = ptx::add_pair(acc[(i >> 1) & 1], e0, e1);
        w[i / 2] = ptx::pack_half2(__uint_as_float(e0), __uint_as_float(e1));
    }
}

template <bool MASK>
__device__ __forceinline__ float max_slice_scaled(const uint32_t (&r)[32], int col0, int n_valid, float m,
                                                  const float *cs)
{
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        const float4 c = *reinterpret_cast<const float4 *>(cs + i);
        const float cc[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float v = __uint_as_float(r[i + q]) * cc[q];
            m = (!MASK || col0 + i + q < n_valid) ? fmaxf(m, v) : m;
        }
    }
    return m;
}

// QK-norm sums of squares (fp32) of eight fp16 values, one 16-byte unit of shared memory: into
// two running sums (a Q row), or column by column (eight key vectors, one d-row of each).
__device__ __forceinline__ void sum_sq_unit(const uint4 &w, float (&ss)[2])
{
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&words[h]));
        ss[0] = fmaf(f.x, f.x, ss[0]);
        ss[1] = fmaf(f.y, f.y, ss[1]);
    }
}

__device__ __forceinline__ void sum_sq_cols(const uint4 &w, float (&sq)[8])
{
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&words[h]));
        sq[2 * h] = fmaf(f.x, f.x, sq[2 * h]);
        sq[2 * h + 1] = fmaf(f.y, f.y, sq[2 * h + 1]);
    }
}

// Sums a[e] over the eight lanes that share lane % 4 (lane bits 2..4) and leaves element
// e = 4 bit4 + 2 bit3 + bit2 of the total on each lane: a reduce-scatter in three exchange steps
// (7 shuffles instead of 24 for eight full reductions), in a fixed order.
__device__ __forceinline__ float reduce_scatter8(const float (&a)[8], int lane)
{
    float b4[4], b2[2];
    const bool h4 = (lane & 16) != 0, h3 = (lane & 8) != 0, h2 = (lane & 4) != 0;
#pragma unroll
    for (int e = 0; e < 4; ++e)
        b4[e] = (h4 ? a[e + 4] : a[e]) + __shfl_xor_sync(0xffffffffu, h4 ? a[e] : a[e + 4], 16);
#pragma unroll
    for (int e = 0; e < 2; ++e)
        b2[e] = (h3 ? b4[e + 2] : b4[e]) + __shfl_xor_sync(0xffffffffu, h3 ? b4[e] : b4[e + 2], 8);
    return (h2 ? b2[1] : b2[0]) + __shfl_xor_sync(0xffffffffu, h2 ? b2[0] : b2[1], 4);
}

// Evaluation variants of kernel 1, compiled separately so that each carries only its own code.
enum Variant : int {
    kPlain = 0,    // the graph as written
    kSafe = 1,     // each row's maximum subtracted before exp (a first pass over K finds it)
    kQkNorm = 2,   // QK-norm: scores scaled by 1/rms of the query row and of the key vector; safe
    kStreamK = 3,  // the graph as written under a stream-K schedule (batches of at most 16 rows)
    kPush = 4,     // the graph as written, split partials pushed into each owner's receive area
};

// Stream-K schedule: the B row tiles x n_tiles column tiles form one sequence of units u = r n_tiles
// + column tile; CTA c takes units [c U / G, (c+1) U / G) (U units, G CTAs), which span at most
// kMaxSegments row tiles ("segments"). Each segment's partial goes to slot c - c_first(r) of its row
// tile r, c_first(r) being the CTA that holds the row tile's first unit.
constexpr int kMaxSegments = 2;
constexpr int kSkQRows = 16;  // Q rows loaded per segment (batches of at most 16 rows)

// The CTA holding unit u: the largest c with floor(c U / G) <= u.
__host__ __device__ __forceinline__ long long sk_cta_of(long long u, long long U, long long G)
{
    return ((u + 1) * G - 1) / U;
}

// Pushed exchange: the 32-row quarters of a row tile (one softmax warp per group each) that hold
// rows inside M and of CTA rank j's share [128 j / n, 128 (j + 1) / n). Every rank's warps of
// those quarters arrive once each on rank j's receive barrier.
__device__ __forceinline__ int push_quarters(const FwdParams &p, int m0, int j)
{
    const int n = p.n_split;
    const int lo = j * kBlockM / n, hi = (j + 1) * kBlockM / n;
    int quarters = 0;
    for (int q = 0; q < 4; ++q)
        if (m0 + 32 * q < p.M && 32 * q < hi && lo < 32 * q + 32)
            ++quarters;
    return quarters;
}

template <int D, int STAGES, int VAR>
__global__ void __launch_bounds__(kThreads, 1)
    mg_attn_fwd_partial(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                        const __grid_constant__ CUtensorMap tmW, const FwdParams p)
{
    using C = TileCfg<D>;
    constexpr bool kSafeMax = VAR == kSafe || VAR == kQkNorm;  // the row-maximum pass runs
    constexpr bool kQk = VAR == kQkNorm;
    constexpr bool kPushX = VAR == kPush;  // the pushed on-chip combine (its receive area after the ring)
    // The pushed variant always combines on chip and carries no code for the other epilogues (one
    // split's TMA store of O, the second kernel's partials). (A plain variant cut down the same
    // way measured no faster on GB300: GQA 6.64 against 6.60 us per call.)
    constexpr bool kClusterOnly = VAR == kPush;
    const bool cluster = kClusterOnly || p.cluster_reduce != 0;
    constexpr int kPBuffers = C::kPBuffers;
    using BI = Bars<STAGES, kPBuffers>;
    static_assert(fwd_smem_bytes(D, STAGES, VAR == kPush) <= 232448u, "tile configuration exceeds 227 KB");
    static_assert(128 * D * 4 <= C::kStageBytes, "output staging must fit in one K/V stage");
    static_assert(2 * 128 * C::kRowHalves * 2 + 128 * C::kLmw * 4 <= STAGES * C::kStageBytes,
                  "on-chip combine staging must fit in the K/V ring");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sQ = ptx::smem_u32(smem);
    const uint32_t sStage0 = sQ + C::kQBytes;
    uint8_t *recv = smem + C::kQBytes + STAGES * C::kStageBytes;
    float *l_xchg = reinterpret_cast<float *>(recv + (kPushX ? C::kRecvBytes : 0u));
    uint64_t *bars = reinterpret_cast<uint64_t *>(l_xchg + 2 * kBlockM);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + BI::kCount);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    // QK-norm with p.cs_tiles: the key-vector scales of this CTA's tiles, past the fixed layout.
    float *cs_smem = reinterpret_cast<float *>(smem + (fwd_smem_bytes(D, STAGES, kPushX) - 1024u));
    auto bar = [&](int i) { return ptx::smem_u32(bars + i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // CTA -> (b, split j, row tile mt). With the on-chip combine, the n_split CTAs of a row tile
    // are consecutive (one cluster, rank j); otherwise consecutive CTAs share (b, j) and so read
    // the same K/V tiles close together in time.
    const int cta = blockIdx.x;
    constexpr bool kSK = VAR == kStreamK;
    const int mt = kSK ? 0 : cluster ? (cta / p.n_split) % p.m_tiles_per_b : cta % p.m_tiles_per_b;
    const int j = kSK ? 0 : cluster ? cta % p.n_split : (cta / p.m_tiles_per_b) % p.n_split;
    const int b = kSK ? 0 : cta / (p.m_tiles_per_b * p.n_split);
    const int m0 = mt * kBlockM;
    // Stream-K: this CTA's units [u0, u1) and their segments (one per row tile touched; a batch is
    // one row tile here). Segment 1, when there is one, starts at step t1.
    const long long u0 = kSK ? static_cast<long long>(cta) * p.sk_units / p.sk_ctas : 0;
    const long long u1 = kSK ? static_cast<long long>(cta + 1) * p.sk_units / p.sk_ctas : 0;
    const int r0 = kSK ? static_cast<int>(u0 / p.n_tiles) : 0;
    const int nseg = kSK ? static_cast<int>((u1 - 1) / p.n_tiles) - r0 + 1 : 1;  // <= kMaxSegments (plan)
    const int t1 = kSK ? static_cast<int>(static_cast<long long>(r0 + 1) * p.n_tiles - u0) : 0;
    // Split j takes every n_split-th column tile, starting at tile j: the splits of a row tile
    // then read neighbouring K/V tiles at the same time, each row of K in one run of DRAM rather
    // than n_split runs far apart (measured on GB300 against contiguous runs of tiles: long_kv
    // 15.0 against 15.6 us per call, gqa 6.75 against 6.88, decode unchanged).
    const int T = kSK ? static_cast<int>(u1 - u0) : (p.n_tiles - j + p.n_split - 1) / p.n_split;  // >= 1
    auto tile_of = [&](int t) {  // column tile of step t
        return kSK ? static_cast<int>((u0 + t) % p.n_tiles) : j + t * p.n_split;
    };
    auto batch_of = [&](int t) { return kSK ? static_cast<int>((u0 + t) / p.n_tiles) : b; };
    auto seg_of = [&](int t) { return kSK && t >= t1 ? 1 : 0; };
    // Steps of the K/V ring: with the max-subtracted variant, T steps that stream K alone (the
    // row-maximum pass), then the T steps of the main pass.
    const int T1 = kSafeMax ? T : 0;
    const int U = T1 + T;

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(BI::kQFull), 1);
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar(BI::kKFull + s), 1);
            ptx::mbar_init(bar(BI::kVFull + s), 1);
            ptx::mbar_init(bar(BI::kKvEmpty + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(bar(BI::kSFull + s), 1);
            ptx::mbar_init(bar(BI::kSEmpty + s), kGroupWarps);
        }
        for (int s = 0; s < kPBuffers; ++s) {
            ptx::mbar_init(bar(BI::kPFull + s), kGroupWarps);
            ptx::mbar_init(bar(BI::kPEmpty + s), 1);
        }
        ptx::mbar_init(bar(BI::kOFull), 1);
        ptx::mbar_init(bar(BI::kDrain), 1);
        ptx::mbar_init(bar(BI::kDrainPv), 1);
        ptx::mbar_init(bar(BI::kNever), 1);
        // Pushed exchange: one arrival (the bytes it sends) per rank and per softmax warp with rows
        // of this CTA's share and inside M; a CTA whose share lies past M gets nothing and waits
        // for nothing.
        const int pq = kPushX ? push_quarters(p, m0, j) : 0;
        ptx::mbar_init(bar(BI::kXRecv), pq > 0 ? static_cast<uint32_t>(p.n_split * 2 * pq) : 1u);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmQ);
        ptx::prefetch_tensormap(&tmK);
        ptx::prefetch_tensormap(&tmV);
        if (p.n_split == 1)
            ptx::prefetch_tensormap(&tmO);
        else if (!cluster)
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
    // Pushed exchange: the first half of a cluster barrier whose wait, just before the first copy
    // to another CTA, says that every CTA's receive barrier is initialised.
    if (kPushX && cluster)
        ptx::cluster_arrive_release();

    // Everything above touched only on-chip state; global memory waits for the previous grid.
    // early == 1: the load warp's first copies go out before its wait (below); every thread
    // releases the dependents after its own wait, so a grid launched after this one never starts
    // before the one before this one has completed. early == 2: the dependents are released now,
    // every role runs without the wait, and each global write waits for the previous grid first
    // (the reads of Q, K and V may then overlap kernels further back; the host checks its recent
    // outputs for that). The release comes after this CTA's tensor-memory allocation: a CTA of a
    // later grid that shares the SM could otherwise hold the columns this one still has to
    // allocate while it waits for this grid to complete.
    if (p.early == 2) {
        ptx::griddep_launch_dependents();
    } else if (!(warp == 0 && p.early == 1)) {
        ptx::griddep_wait();
        ptx::griddep_launch_dependents();
    }

    const WaitCtx wc{abort_flag, p.status, p.timeout_ns};
    bool staged_ok = false;  // softmax warps: this CTA staged its output (its O was complete)

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        // Lane 0 issues every copy. Early loads: Q and the first STAGES steps' tiles go out before
        // the wait for the previous grid (the host allows it only when that grid writes none of
        // Q, K and V), so their DRAM latency overlaps the previous call's end. The other lanes
        // take the wait only once lane 0 has issued them (a lane blocked in the wait would hold
        // lane 0 back): the warp meets at a __syncwarp from both paths.
        if (lane != 0) {
            if (p.early == 1) {
                __syncwarp();
                ptx::griddep_wait();
                ptx::griddep_launch_dependents();
            }
        } else {
            bool q_armed = false;
            int armed[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s)
                armed[s] = 0;
            bool ok = true;
            // One step's copies into stage t % STAGES, once that stage is free.
            auto issue = [&](int t) {
                const int s = t % STAGES;
                const int n0 = tile_of(t < T1 ? t : t - T1) * kBlockN;
                const int bt = batch_of(t < T1 ? t : t - T1);
                const uint32_t sK = sStage0 + s * C::kStageBytes;
                const uint32_t sV = sK + C::kKBytes;
                // K and V land on separate barriers: S = Q.K need not wait for V. A step of the
                // row-maximum pass loads no V; its V barrier phase completes on a plain arrival,
                // so every step advances every barrier of its stage by one phase.
                ptx::mbar_arrive_expect_tx(bar(BI::kKFull + s), C::kKBytes);
                if (t < T1)
                    ptx::mbar_arrive(bar(BI::kVFull + s));
                else
                    ptx::mbar_arrive_expect_tx(bar(BI::kVFull + s), C::kVBytes);
                ++armed[s];
                // K[b, 0:d, n0:n0+64] and K[b, 0:d, n0+64:n0+128]: d rows of 128 bytes each.
                ptx::tma_load_3d(sK, &tmK, bar(BI::kKFull + s), n0, 0, bt);
                ptx::tma_load_3d(sK + D * 128, &tmK, bar(BI::kKFull + s), n0 + 64, 0, bt);
                // V[b, n0:n0+128, 64c:64c+64]: 128 rows of 128 bytes each.
                if (t >= T1) {
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        ptx::tma_load_3d(sV + c * C::kChunkRows128, &tmV, bar(BI::kVFull + s), c * 64, n0, bt);
                }
            };
            if (p.inject_timeout)
                ok = wait_bounded(wc, bar(BI::kNever), 0, BI::kNever);
            int t = 0;  // the next step to issue
            if (ok) {
                if constexpr (kSK) {
                    // One compact Q tile per segment (kSkQRows rows of 128-byte chunks: the tensor
                    // map's box is kSkQRows high), all on one barrier.
                    ptx::mbar_arrive_expect_tx(bar(BI::kQFull), nseg * C::kChunks * kSkQRows * 128);
                    q_armed = true;
                    for (int k = 0; k < nseg; ++k)
#pragma unroll
                        for (int c = 0; c < C::kChunks; ++c)  // Q[r0 + k, 0:16, 64c:64c+64]
                            ptx::tma_load_3d(sQ + (k * C::kChunks + c) * kSkQRows * 128, &tmQ, bar(BI::kQFull),
                                             c * 64, 0, r0 + k);
                } else {
                    ptx::mbar_arrive_expect_tx(bar(BI::kQFull), C::kQBytes);
                    q_armed = true;
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)  // Q[b, m0:m0+128, 64c:64c+64]
                        ptx::tma_load_3d(sQ + c * C::kChunkRows128, &tmQ, bar(BI::kQFull), c * 64, m0, b);
                }
                if (p.early == 1)
                    for (; t < U && t < STAGES; ++t)  // the stages are free: no wait
                        issue(t);
            }
            if (p.early == 1) {
                __syncwarp();
                ptx::griddep_wait();
                ptx::griddep_launch_dependents();
            }
            for (; ok && t < U; ++t) {
                const int s = t % STAGES;
                const uint32_t round = static_cast<uint32_t>(t / STAGES);
                if (t >= STAGES && !wait_bounded(wc, bar(BI::kKvEmpty + s), (round & 1u) ^ 1u, BI::kKvEmpty + s)) {
                    ok = false;
                    break;
                }
                issue(t);
            }
            if (ok) {
                // Tail: the commits that release the last stages must land before the CTA exits.
                for (int u = U - STAGES > 0 ? U - STAGES : 0; ok && u < U; ++u)
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
        // ---------------------------------------------------------------- S = Q.K issuer
        // The whole warp runs the loop and takes every wait together (the decision to go on is a
        // warp vote); the lane elect.sync picks issues each tile's MMAs and their commit. Measured
        // on GB300, an M=128, N=64 MMA issued this way occupies the tensor pipe 32 cycles (its
        // arithmetic), against 45 from a lone thread looping on its own and 57 from "lane == 0"
        // of a converged warp.
        constexpr uint32_t idesc_s = ptx::idesc_f16_f32(kBlockM, kBlockN, false, true);
        // A = Q: K-major; 16-column steps advance 32 B in a swizzle row; 8-row groups 1024 B apart.
        // A stream-K segment's compact Q tile has its 64-column chunks kSkQRows rows apart: the
        // product reads 128 rows from there, and rows past the tile's (past M here) are never
        // stored, whatever they hold.
        const uint32_t q_chunk = kSK ? kSkQRows * 128 : C::kChunkRows128;
        uint64_t a_q[D / 16];
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
            a_q[k] = ptx::sdesc_sw128(sQ + (k >> 2) * q_chunk + (k & 3) * 32, 16, 1024);
        // Segment 1's Q tile follows segment 0's: the same descriptors, start address moved on.
        const uint64_t q_seg_step = static_cast<uint64_t>((C::kChunks * kSkQRows * 128) >> 4);
        auto warp_wait = [&](uint32_t b_, uint32_t parity, int where) -> bool {
            return __all_sync(0xffffffffu, wait_bounded(wc, b_, parity, where));
        };
        bool ok = warp_wait(bar(BI::kQFull), 0, BI::kQFull);
        // S_u = Q . K_u into S buffer u % 2 (softmax group u % 2), as soon as K tile u is in its
        // stage and, for u >= 2, that group has read S_{u-2} out of the buffer (which it does in
        // the first half of tile u-2). The P.V products run from another warp, so an S never
        // waits behind a P.V.
        // With the max-subtracted variant the first T1 steps compute S for the row-maximum pass;
        // their completion also frees the K stage (no P.V reads it), except with QK-norm, where
        // the softmax group also reads the K tile (the key-vector scales) and frees the stage.
        for (int u = 0; ok && u < U; ++u) {
            const int s = u % STAGES;
            const int sb = u & 1;
            if (!warp_wait(bar(BI::kKFull + s), static_cast<uint32_t>(u / STAGES) & 1u, BI::kKFull + s) ||
                (u >= 2 &&
                 !warp_wait(bar(BI::kSEmpty + sb), (static_cast<uint32_t>(u >> 1) & 1u) ^ 1u, BI::kSEmpty + sb))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            // B = K: N-major; 16 d-rows (2048 B) per k-step; the two 64-column halves D*128 B apart.
            const uint64_t k_desc = ptx::sdesc_sw128(sStage0 + s * C::kStageBytes, D * 128, 1024);
            if (ptx::elect_one()) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    ptx::mma_f16_ss(tmem + sb * kBlockN, a_q[k] + (kSK ? seg_of(u) * q_seg_step : 0),
                                    k_desc + static_cast<uint64_t>(k * (2048 >> 4)), idesc_s, k > 0 ? 1u : 0u);
                ptx::mma_commit(bar(BI::kSFull + sb));
                if (!kQk && u < T1)
                    ptx::mma_commit(bar(BI::kKvEmpty + s));
            }
            __syncwarp();
        }
        // Every S product issued completes before tensor memory is freed, on the unwinding path
        // and also when another role aborts after this loop has ended (then nobody else may wait
        // for the last S buffers). elect.sync picks the same lane of the full warp every time.
        if (ptx::elect_one()) {
            ptx::mma_commit(bar(BI::kDrain));
            wait_drain(bar(BI::kDrain), 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ---------------------------------------------------------------- O += P.V issuer
        // Same pattern as the S issuer: warp-wide waits, the elected lane issues.
        constexpr uint32_t idesc_o = ptx::idesc_f16_f32(kBlockM, D, false, true);
        const uint32_t tmem_o = tmem + kTmemO;
        auto warp_wait = [&](uint32_t b_, uint32_t parity, int where) -> bool {
            return __all_sync(0xffffffffu, wait_bounded(wc, b_, parity, where));
        };
        bool ok = true;
        // O += P_u . V_u once the softmax warps have written P_u and V tile u has landed (K
        // tile u, which S_u needed, shares its stage). The completion releases K/V stage u and
        // P buffer u % kPBuffers.
        for (int v = 0; ok && v < T; ++v) {
            const int u = T1 + v;  // step of the K/V ring
            const int pb = v % kPBuffers;
            const int s = u % STAGES;
            // The graph as written waits for V first: it has usually landed long before P, and
            // its test then costs nothing after P's. In the two-pass variants the V barrier of a
            // stage also completes phases for the row-maximum steps, on the producer's plain
            // arrival when it issues them. A wait for V before P could test the barrier while
            // the phase before the awaited one is still open, and a parity wait would then pass
            // early. There P comes first: P of step u exists only once K of step u has landed, so
            // every earlier phase of that V barrier has completed.
            bool waited;
            if constexpr (!kSafeMax)
                waited = warp_wait(bar(BI::kVFull + s), static_cast<uint32_t>(u / STAGES) & 1u, BI::kVFull + s) &&
                         warp_wait(bar(BI::kPFull + pb), static_cast<uint32_t>(v / kPBuffers) & 1u, BI::kPFull + pb);
            else
                waited = warp_wait(bar(BI::kPFull + pb), static_cast<uint32_t>(v / kPBuffers) & 1u, BI::kPFull + pb) &&
                         warp_wait(bar(BI::kVFull + s), static_cast<uint32_t>(u / STAGES) & 1u, BI::kVFull + s);
            if (!waited) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t tP = tmem + C::kTmemP + pb * 64;
            // B = V: N(=d)-major, 16 rows (2048 B) per k-step; d-chunks 128 rows x 128 B apart.
            const uint64_t v_desc = ptx::sdesc_sw128(sStage0 + s * C::kStageBytes + C::kKBytes, C::kChunkRows128, 1024);
            // A stream-K segment's first product starts O afresh. It cannot overtake the previous
            // segment's epilogue, which reads O: it needs P of its tile, and the softmax group writes
            // that only after the epilogue's closing barrier.
            const bool fresh = v == 0 || (kSK && v == t1);
            if (ptx::elect_one()) {
                // A = P in tensor memory: 16 K-columns per step are 8 tensor-memory columns.
                ptx::mma_f16_ts(tmem_o, tP, v_desc, idesc_o, fresh ? 0u : 1u);
#pragma unroll
                for (int k = 1; k < kBlockN / 16; ++k)
                    ptx::mma_f16_ts(tmem_o, tP + k * 8, v_desc + static_cast<uint64_t>(k * (2048 >> 4)), idesc_o, 1u);
                ptx::mma_commit(bar(BI::kKvEmpty + s));
                ptx::mma_commit(bar(BI::kPEmpty + pb));
                // Committed by the thread that issued every P.V: O of the last step (of each
                // stream-K segment) is complete, one OFull phase per segment.
                if (v == T - 1 || (kSK && v == t1 - 1))
                    ptx::mma_commit(bar(BI::kOFull));
            }
            __syncwarp();
        }
        if (ok) {
            // Tail: the commits that release the last P buffers must land before the CTA exits.
            for (int u = T - kPBuffers > 0 ? T - kPBuffers : 0; ok && u < T; ++u)
                ok = warp_wait(bar(BI::kPEmpty + u % kPBuffers), static_cast<uint32_t>(u / kPBuffers) & 1u,
                               BI::kPEmpty + u % kPBuffers);
        }
        if (!ok) {
            // Unwinding, from the loop or from the tail: the P.V products issued complete before
            // tensor memory is freed.
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
        const int g = sw >> 2;                   // warp group: takes the tiles t with t % 2 == g
        const int row = q4 * 32 + lane;          // row inside the 128-row tile
        const bool warp_rows = (m0 + q4 * 32) < p.M;  // warp-uniform: any valid row in this warp
        const uint32_t lane_addr = static_cast<uint32_t>(q4 * 32) << 16;
        // The decision to go on is taken by the whole warp, so that no lane reaches a
        // warp-collective tcgen05.ld without the others.
        auto warp_wait = [&](uint32_t b_, uint32_t parity, int where) -> bool {
            const bool r = wait_bounded(wc, b_, parity, where);
            return __all_sync(0xffffffffu, r);
        };
        uint64_t acc[2] = {0, 0};  // packed fp32 partial row sums (+0.0 bit patterns)
        const ptx::ExpPairConsts ek = ptx::exp_pair_consts();
        bool ok = true;
        // QK-norm variant: a is this row's query scale, 1/rms of the Q tile's row (read from shared
        // memory once; rows past M take 1, their scores are 0 anyway); the key-vector scales c of
        // the split's columns are computed by the row-maximum pass below and kept for the main
        // pass in shared memory (p.cs_tiles; then the call may start early) or else in global
        // memory (L2).
        float a_row = 1.f;
        float *col_scale = nullptr;
        if constexpr (kQk) {
            col_scale = p.col_scale + static_cast<size_t>(b) * p.N;
            ok = warp_wait(bar(BI::kQFull), 0, BI::kQFull);
            if (ok && m0 + row < p.M) {
                // The row's 16-byte units in swizzled order (a permutation of the row: the sum is
                // the same), so the eight lanes of a quarter-warp hit eight distinct bank groups.
                float ss[2] = {0.f, 0.f};
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c)
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        sum_sq_unit(*reinterpret_cast<const uint4 *>(
                                        smem + c * C::kChunkRows128 + row * 128 + ((k ^ (row & 7)) << 4)),
                                    ss);
                a_row = __frsqrt_rn((ss[0] + ss[1]) * (1.f / D) + kQkNormEps);
            }
        }
        const uint32_t a_log2e = __float_as_uint(a_row * ptx::kLog2e);
        const uint64_t arow = ptx::pair_of(a_log2e);
        // Max-subtracted variant, first pass: each thread's running maximum of its row over the
        // valid columns of its group's steps (S only; the buffer is released once read).
        float m_row = -INFINITY;
        int u = g;
        if constexpr (kQk) {
            // Each tile's 128 key-vector scales first, from the K tile in shared memory: warp gw of
            // the group sums the squares of columns [32 gw, 32 gw + 32), a lane taking one 16-byte
            // unit (8 columns) of every eighth d-row (rows kr, kr + 8, ...; kr alternates between
            // the two halves of the swizzle pattern so that a quarter-warp's eight loads hit eight
            // distinct bank groups); a reduce-scatter over the eight lanes of a unit then leaves one
            // column's sum per lane. The scales meet in this group's half of l_xchg (free until the
            // maxima are exchanged); the group's two barriers per tile publish them and keep the
            // next tile's from overwriting them early. All four warps of the group run every
            // iteration and vote at the first barrier, so an abort leaves them together.
            const int gw = sw & 3;
            const int rs = lane >> 2;
            const int kr = ((rs & 1) << 2) | (rs >> 1);
            const uint32_t unit_phys = (static_cast<uint32_t>(((gw & 1) << 2) | (lane & 3))) ^ static_cast<uint32_t>(kr);
            const int my_col = 32 * gw + 8 * (lane & 3) + ((((lane >> 4) & 1) << 2) | (((lane >> 3) & 1) << 1) | ((lane >> 2) & 1));
            float *cs_tile = l_xchg + g * kBlockM;
            // Barrier ids stay compile-time constants (one branch per group).
            auto group_barrier_and = [&](bool pred) {
                return g == 0 ? ptx::named_barrier_and(kGroupBarrier0, kGroupWarps * 32, pred)
                              : ptx::named_barrier_and(kGroupBarrier0 + 1, kGroupWarps * 32, pred);
            };
            for (; u < T1; u += 2) {
                const int s = u % STAGES;
                // The sums need only the K tile; they run while the tensor core computes S.
                bool w_ok = ok && warp_wait(bar(BI::kKFull + s), static_cast<uint32_t>(u / STAGES) & 1u, BI::kKFull + s);
                if (w_ok) {
                    const uint8_t *kp = smem + C::kQBytes + s * C::kStageBytes + (gw >> 1) * (D * 128) + kr * 128 +
                                        (unit_phys << 4);
                    float sq[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int k = 0; k < D / 8; ++k)  // d-row kr + 8k
                        sum_sq_cols(*reinterpret_cast<const uint4 *>(kp + k * 1024), sq);
                    const float c = __frsqrt_rn(reduce_scatter8(sq, lane) * (1.f / D) + kQkNormEps);
                    cs_tile[my_col] = c;
                    if (p.cs_tiles) {
                        cs_smem[u * kBlockN + my_col] = c;  // u < T <= p.cs_tiles
                    } else {
                        if (p.early == 2)  // (the host starts this form early only with p.cs_tiles)
                            ptx::griddep_wait();
                        if (tile_of(u) * kBlockN + my_col < p.N)
                            col_scale[static_cast<size_t>(tile_of(u)) * kBlockN + my_col] = c;
                    }
                }
                w_ok = w_ok && warp_wait(bar(BI::kSFull + g), static_cast<uint32_t>(u >> 1) & 1u, BI::kSFull + g);
                w_ok = group_barrier_and(w_ok);
                if (!w_ok) {
                    ok = false;
                    break;
                }
                // The group is done with the K tile (the S product that read it has completed).
                if (gw == 0 && lane == 0)
                    ptx::mbar_arrive(bar(BI::kKvEmpty + s));
                ptx::tc_fence_after();
                const int n_valid = p.N - tile_of(u) * kBlockN;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    if (warp_rows) {
                        uint32_t r0[32], r1[32];
                        const uint32_t s_addr = tmem + lane_addr + g * kBlockN + half * 64;
                        ptx::tmem_ld_32x32b_x32(s_addr, r0);
                        ptx::tmem_ld_32x32b_x32(s_addr + 32, r1);
                        ptx::tmem_ld_wait(r0);
                        ptx::tmem_ld_wait(r1);
                        const int nv = n_valid - half * 64;
                        const float *cs = cs_tile + half * 64;
                        if (nv >= 64) {
                            m_row = max_slice_scaled<false>(r0, 0, nv, m_row, cs);
                            m_row = max_slice_scaled<false>(r1, 32, nv, m_row, cs + 32);
                        } else {
                            m_row = max_slice_scaled<true>(r0, 0, nv, m_row, cs);
                            m_row = max_slice_scaled<true>(r1, 32, nv, m_row, cs + 32);
                        }
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(bar(BI::kSEmpty + g));
                group_barrier_and(true);
            }
        } else {
            for (; ok && u < T1; u += 2) {
                if (!warp_wait(bar(BI::kSFull + g), static_cast<uint32_t>(u >> 1) & 1u, BI::kSFull + g)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const int n_valid = p.N - tile_of(u) * kBlockN;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    if (warp_rows) {
                        uint32_t r0[32], r1[32];
                        const uint32_t s_addr = tmem + lane_addr + g * kBlockN + half * 64;
                        ptx::tmem_ld_32x32b_x32(s_addr, r0);
                        ptx::tmem_ld_32x32b_x32(s_addr + 32, r1);
                        ptx::tmem_ld_wait(r0);
                        ptx::tmem_ld_wait(r1);
                        const int nv = n_valid - half * 64;
                        if (nv >= 64) {
                            m_row = max_slice<false>(r0, 0, nv, m_row);
                            m_row = max_slice<false>(r1, 32, nv, m_row);
                        } else {
                            m_row = max_slice<true>(r0, 0, nv, m_row);
                            m_row = max_slice<true>(r1, 32, nv, m_row);
                        }
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(bar(BI::kSEmpty + g));
            }
        }
        // The two groups' maxima meet in shared memory (both reach both barriers, on the
        // unwinding path too): m is the row's maximum over the split, and every exponential of
        // the main pass is exp(s - m) <= 1. The second barrier keeps the exchange slots from
        // being reused (by the row sums below) before every thread has read them.
        uint64_t shift = 0;  // +0.0 twice: exp(s) unshifted, as the graph is written
        float m = 0.f;
        if constexpr (kSafeMax) {
            l_xchg[g * kBlockM + row] = m_row * a_row;  // a_row > 0 (1 without QK-norm)
            ptx::named_barrier(kSoftmaxBarrier, kSoftmaxThreads);
            m = fmaxf(l_xchg[row], l_xchg[kBlockM + row]);
            ptx::named_barrier(kSoftmaxBarrier, kSoftmaxThreads);
            const uint32_t nm = __float_as_uint(-m * ptx::kLog2e);
            shift = ptx::pair_of(nm);
        }
        // The two groups alternate tiles, each with its own S buffer (g): while one group's warps
        // wait on tensor memory or a barrier, the other group's warps on the same scheduler keep
        // the MUFU unit busy. A thread covers its row's 128 columns of a tile in two 64-column
        // halves (64 fp32 registers at a time). Step u of the ring is tile t = u - T1.
        // Stream-K: each segment's steps, then that segment's epilogue; otherwise one segment.
        for (int k = 0; k < nseg; ++k) {
        const int t_beg = k == 0 ? 0 : t1;
        const int t_end = k + 1 < nseg ? t1 : T;
        for (u = T1 + t_beg + ((T1 + t_beg) % 2 == g ? 0 : 1); ok && u < T1 + t_end; u += 2) {
            const int t = u - T1;
            const int pb = t % kPBuffers;
            if (!warp_wait(bar(BI::kSFull + g), static_cast<uint32_t>(u >> 1) & 1u, BI::kSFull + g)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const int n_valid = p.N - tile_of(t) * kBlockN;  // columns of this tile inside N
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
                    // All of S is in registers: the buffer can take this group's next tile. One
                    // arrival per warp (after a warp barrier) rather than per thread.
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        ptx::mbar_arrive(bar(BI::kSEmpty + g));
                } else if (t >= kPBuffers &&
                           !warp_wait(bar(BI::kPEmpty + pb), (static_cast<uint32_t>(t / kPBuffers) & 1u) ^ 1u,
                                      BI::kPEmpty + pb)) {
                    ok = false;
                    break;
                }
                if (warp_rows) {
                    // Columns [64 half, 64 half + 64) of P are tensor-memory columns
                    // [32 half, 32 half + 32) of buffer pb (two fp16 per column).
                    const int nv = n_valid - half * 64;
                    uint32_t w[32];
                    if constexpr (kQk) {
                        const float *cs = (p.cs_tiles ? cs_smem + t * kBlockN
                                                      : col_scale + static_cast<size_t>(tile_of(t)) * kBlockN) +
                                          half * 64;
                        if (nv >= 64) {
                            exp_slice_scaled<false>(r0, 0, nv, w, acc, cs, arow, shift);
                            exp_slice_scaled<false>(r1, 32, nv, w + 16, acc, cs + 32, arow, shift);
                        } else {
                            exp_slice_scaled<true>(r0, 0, nv, w, acc, cs, arow, shift);
                            exp_slice_scaled<true>(r1, 32, nv, w + 16, acc, cs + 32, arow, shift);
                        }
                    } else if (nv >= 64) {
                        exp_slice<false>(r0, 0, nv, w, acc, ek, shift);
                        exp_slice<false>(r1, 32, nv, w + 16, acc, ek, shift);
                    } else {
                        exp_slice<true>(r0, 0, nv, w, acc, ek, shift);
                        exp_slice<true>(r1, 32, nv, w + 16, acc, ek, shift);
                    }
                    ptx::tmem_st_32x32b_x32(tmem + lane_addr + C::kTmemP + pb * 64 + half * 32, w);
                    ptx::tmem_st_wait();
                }
            }
            if (!ok)
                break;
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(bar(BI::kPFull + pb));
        }
        if constexpr (kSK) {
            // -------------------------------------------------------- stream-K segment epilogue
            // The segment's partial (fp32 numerators and the row sum, rows < M) goes to slot
            // c - c_first(r) of its row tile r = r0 + k (a batch: one row tile each), for the second
            // kernel; the row tile's last contributor also zeroes its unused slots, so each call
            // leaves every slot the second kernel reads defined. A barrier of all eight softmax
            // warps closes the epilogue: O and the row-sum exchange are free again after it.
            const float lg = (__uint_as_float(static_cast<uint32_t>(acc[0])) +
                              __uint_as_float(static_cast<uint32_t>(acc[0] >> 32))) +
                             (__uint_as_float(static_cast<uint32_t>(acc[1])) +
                              __uint_as_float(static_cast<uint32_t>(acc[1] >> 32)));
            acc[0] = 0;
            acc[1] = 0;
            l_xchg[g * kBlockM + row] = lg;
            const bool seg_ready = ptx::named_barrier_and(
                kSoftmaxBarrier, kSoftmaxThreads,
                ok && warp_wait(bar(BI::kOFull), static_cast<uint32_t>(k) & 1u, BI::kOFull));
            const float ls = l_xchg[row] + l_xchg[kBlockM + row];
            if (!seg_ready) {
                ok = false;
            } else {
                ptx::tc_fence_after();
                if (p.early == 2)  // (the host does not start this schedule early; kept safe)
                    ptx::griddep_wait();
                const int r = r0 + k;
                const int c_first = static_cast<int>(sk_cta_of(static_cast<long long>(r) * p.n_tiles, p.sk_units, p.sk_ctas));
                const int c_last = static_cast<int>(
                    sk_cta_of(static_cast<long long>(r + 1) * p.n_tiles - 1, p.sk_units, p.sk_ctas));
                const int slot = cta - c_first;
                const int zero_from = cta == c_last ? c_last - c_first + 1 : p.sk_slots;
                const bool mine = row < p.M;
                if (warp_rows) {
#pragma unroll
                    for (int c = 0; c < C::kHalfCols / 32; ++c) {
                        uint32_t rv[32];
                        const int col = g * C::kHalfCols + c * 32;
                        ptx::tmem_ld_32x32b_x32(tmem + lane_addr + kTmemO + col, rv);
                        ptx::tmem_ld_wait(rv);
                        if (mine) {
                            float4 *dst = reinterpret_cast<float4 *>(
                                p.ws_o + ((static_cast<size_t>(slot) * p.B + r) * p.M + row) * D + col);
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                dst[q] = make_float4(__uint_as_float(rv[4 * q]), __uint_as_float(rv[4 * q + 1]),
                                                     __uint_as_float(rv[4 * q + 2]), __uint_as_float(rv[4 * q + 3]));
                            for (int z = zero_from; z < p.sk_slots; ++z) {
                                float4 *zd = reinterpret_cast<float4 *>(
                                    p.ws_o + ((static_cast<size_t>(z) * p.B + r) * p.M + row) * D + col);
#pragma unroll
                                for (int q = 0; q < 8; ++q)
                                    zd[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                        }
                    }
                }
                if (g == 0 && mine) {
                    p.ws_l[(static_cast<size_t>(slot) * p.B + r) * p.M + row] = ls;
                    for (int z = zero_from; z < p.sk_slots; ++z)
                        p.ws_l[(static_cast<size_t>(z) * p.B + r) * p.M + row] = 0.f;
                }
                ptx::tc_fence_before();
                ptx::named_barrier(kSoftmaxBarrier, kSoftmaxThreads);
            }
        }
        }  // segments

        if constexpr (!kSK) {
        // ------------------------------------------------------------ epilogue
        // Row sum: this thread's tiles, then the two groups' sums added in a fixed order.
        const float l_group = (__uint_as_float(static_cast<uint32_t>(acc[0])) +
                               __uint_as_float(static_cast<uint32_t>(acc[0] >> 32))) +
                              (__uint_as_float(static_cast<uint32_t>(acc[1])) +
                               __uint_as_float(static_cast<uint32_t>(acc[1] >> 32)));
        l_xchg[g * kBlockM + row] = l_group;
        // One barrier publishes the half sums and makes "O is ready" a decision all eight softmax
        // warps share (a warp that unwound from an abort votes no), so the barrier inside the
        // branch below is reached by all of them or by none.
        const bool o_ready = ptx::named_barrier_and(kSoftmaxBarrier, kSoftmaxThreads,
                                                    ok && warp_wait(bar(BI::kOFull), 0, BI::kOFull));
        const float l = l_xchg[row] + l_xchg[kBlockM + row];
        staged_ok = o_ready;
        uint32_t push_bytes = 0;  // pushed exchange: bytes this thread sent its rows' owner
        if constexpr (kPushX)
            ptx::cluster_wait_acquire();  // every CTA's receive barrier is initialised
        if (o_ready) {
            ptx::tc_fence_after();
            // The K/V ring is idle (every PV has completed): stage this CTA's output there. For the
            // on-chip combine: the normalised partial x = O_j / l_j as fp16 rows of d + 8 halves
            // (the pad keeps 8 consecutive rows on distinct banks); for a 32-column slice of a row
            // with any |x| >= kHiOnlyBelow also the remainders x - fp16(x), in the same layout;
            // then the fp32 row sum l_j once per slice (each copy carries, in its sign bit, whether
            // that slice's remainders are staged; l_j >= 0) and the row maximum m_j, kLmw floats per
            // row, read by the cluster's CTAs after the cluster barrier (the pushed variant stores
            // the same values straight into their owners' receive areas instead). Otherwise the
            // 128-byte-swizzled layout the output tensor maps expect, then a TMA store.
            const uint32_t stage = sStage0;
            __half *stage_hi = reinterpret_cast<__half *>(smem + C::kQBytes);
            __half *stage_lo = stage_hi + kBlockM * C::kRowHalves;
            float *stage_lm = reinterpret_cast<float *>(stage_lo + kBlockM * C::kRowHalves);  // [128][kLmw]
            if (warp_rows) {
#pragma unroll
                for (int c = 0; c < C::kHalfCols / 32; ++c) {
                    uint32_t r[32];
                    const int col = g * C::kHalfCols + c * 32;  // first O column of this slice
                    ptx::tmem_ld_32x32b_x32(tmem + lane_addr + kTmemO + col, r);
                    ptx::tmem_ld_wait(r);
                    if (cluster) {
                        // One correctly rounded reciprocal, then products (l = 0 only if every
                        // exponential of the split underflowed; its partial is then 0).
                        const float inv = l > 0.f ? __frcp_rn(l) : 0.f;
                        uint4 *dhi = reinterpret_cast<uint4 *>(stage_hi + row * C::kRowHalves + col);
                        uint4 *dlo = reinterpret_cast<uint4 *>(stage_lo + row * C::kRowHalves + col);
                        // Pushed exchange: this row's slot in its owner's receive area (rank o holds
                        // rows [128 o / n, 128 (o + 1) / n); sender j's rows start at row j * R).
                        const int po = (row * p.n_split + p.n_split - 1) / kBlockM;
                        const uint32_t prow = static_cast<uint32_t>(j * ((kBlockM + p.n_split - 1) / p.n_split) + row -
                                                                    po * kBlockM / p.n_split);
                        const uint32_t pbar = kPushX ? ptx::map_to_rank(bar(BI::kXRecv), po) : 0u;
                        const uint32_t precv = ptx::smem_u32(recv);
                        bool wide = false;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t h4[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                const float x0 = __uint_as_float(r[8 * q + 2 * h]) * inv;
                                const float x1 = __uint_as_float(r[8 * q + 2 * h + 1]) * inv;
                                h4[h] = ptx::pack_half2(x0, x1);
                                wide = wide || fabsf(x0) >= kHiOnlyBelow || fabsf(x1) >= kHiOnlyBelow;
                            }
                            if constexpr (kPushX)
                                ptx::st_async_v4(ptx::map_to_rank(precv + (prow * C::kRowHalves + col) * 2 + q * 16, po),
                                                 h4[0], h4[1], h4[2], h4[3], pbar);
                            else
                                dhi[q] = make_uint4(h4[0], h4[1], h4[2], h4[3]);
                        }
                        if (wide) {
                            // Second pass, only for a slice that needs it: the same products again,
                            // minus their fp16 roundings (exact differences).
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint32_t l4[4];
#pragma unroll
                                for (int h = 0; h < 4; ++h) {
                                    const float x0 = __uint_as_float(r[8 * q + 2 * h]) * inv;
                                    const float x1 = __uint_as_float(r[8 * q + 2 * h + 1]) * inv;
                                    const uint32_t hw = ptx::pack_half2(x0, x1);
                                    const float2 hf = __half22float2(*reinterpret_cast<const __half2 *>(&hw));
                                    l4[h] = ptx::pack_half2(x0 - hf.x, x1 - hf.y);
                                }
                                if constexpr (kPushX)
                                    ptx::st_async_v4(
                                        ptx::map_to_rank(precv + (C::kRecvRows + prow) * C::kRowHalves * 2 + col * 2 + q * 16, po),
                                        l4[0], l4[1], l4[2], l4[3], pbar);
                                else
                                    dlo[q] = make_uint4(l4[0], l4[1], l4[2], l4[3]);
                            }
                        }
                        if constexpr (kPushX) {
                            ptx::st_async_b32(ptx::map_to_rank(precv + 2 * C::kRecvRows * C::kRowHalves * 2 +
                                                                   (prow * C::kLmw + col / 32) * 4, po),
                                              __float_as_uint(wide ? -l : l), pbar);
                            push_bytes += 64u + 4u + (wide ? 64u : 0u);
                        } else {
                            stage_lm[row * C::kLmw + col / 32] = wide ? -l : l;  // -0.0 when l = 0
                        }
                    } else if (p.n_split == 1) {
                        // fp16 O/l: chunk col/64 of a {64, 128} fp16 box; this slice is units (col%64)/8 .. +3.
                        // One correctly rounded reciprocal, then products: within 1.5 fp32 ulps of
                        // the quotient, far below the fp16 rounding that follows (0 and inf give
                        // the quotient's NaN / 0 as well). Measured on GB300: 32 IEEE divisions per
                        // thread took ~1 us of a one-tile call's epilogue.
                        const float inv = __frcp_rn(l);
                        const uint32_t chunk = stage + (col / 64) * C::kChunkRows128;
                        const uint32_t u0 = static_cast<uint32_t>((col % 64) / 8);
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
                        // fp32 partial: chunk col/32 of {32, 128} fp32 boxes; this slice fills units 0..7.
                        const uint32_t chunk = stage + (col / 32) * C::kChunkRows128;
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            ptx::st_shared_v4(chunk + sw128_offset(row, q), r[4 * q + 0], r[4 * q + 1], r[4 * q + 2],
                                              r[4 * q + 3]);
                    }
                }
            }
            if (cluster) {
                if (g == 0)
                    stage_lm[row * C::kLmw + D / 32] = m;
            } else {
                if (p.early == 2)
                    ptx::griddep_wait();  // the global writes below (and the TMA store) come after it
                if (p.n_split > 1 && g == 0 && m0 + row < p.M) {
                    const size_t r = (static_cast<size_t>(j) * p.B + b) * p.M + m0 + row;
                    p.ws_l[r] = l;
                    if (kSafeMax)
                        p.ws_m[r] = m;
                }
            }
            if (!cluster) {
                ptx::fence_proxy_async_smem();
                ptx::named_barrier(kSoftmaxBarrier, kSoftmaxThreads);
                if (sw == 0 && lane == 0) {
                    if (p.n_split == 1) {
#pragma unroll
                        for (int c = 0; c < D / 64; ++c)  // O[b, m0:m0+128, 64c:64c+64]
                            ptx::tma_store_3d(&tmO, stage + c * C::kChunkRows128, c * 64, m0, b);
                    } else {
#pragma unroll
                        for (int c = 0; c < D / 32; ++c)  // ws_o[j, b, m0:m0+128, 32c:32c+32]
                            ptx::tma_store_3d(&tmW, stage + c * C::kChunkRows128, c * 32, m0, j * p.B + b);
                    }
                    ptx::bulk_commit_group();
                    ptx::bulk_wait_group_read0();
                }
            }
        }
        if constexpr (kPushX) {
            // Pushed exchange: one arrival per warp and owner, with the bytes its lanes sent that
            // owner (0 from a CTA that unwound and sent nothing). An arrival and the stores it
            // counts may land in either order.
            if (cluster && warp_rows) {
                const int po = (row * p.n_split + p.n_split - 1) / kBlockM;
                const unsigned peers = __match_any_sync(0xffffffffu, po);
                const unsigned total = __reduce_add_sync(peers, push_bytes);
                if (lane == __ffs(peers) - 1)
                    ptx::mbar_arrive_expect_tx_cluster(ptx::map_to_rank(bar(BI::kXRecv), po), total);
            }
        }
        }  // !kSK
    }

    // On-chip combine of the split partials. CTA rank j forms rows [128 j / n, 128 (j+1) / n) of
    // its row tile as sum_r c_r x_r / sum_r c_r with c_r = l_r (times exp(m_r - max m) in the
    // max-subtracted variant), x_r = the fp16 value plus, where rank r flagged the slice, its fp16
    // remainder, over all n ranks in rank order (reproducible), and writes fp16 O. The staged rows
    // reach their owner in one of two ways:
    //  * pulled: after a cluster barrier every owner reads its rows out of the n CTAs' staging
    //    (distributed shared memory), and a second barrier keeps each CTA's shared memory alive
    //    until the others have read it;
    //  * pushed (on request): as each thread forms its row's values it stores them, from
    //    registers, into the row owner's receive area (st.async, each store counted on the owner's
    //    receive barrier, with one arrival per warp and owner), so an owner waits for its own rows
    //    only, not for a cluster-wide barrier, and reads them locally. A closing cluster barrier,
    //    which each CTA reaches only once the stores into it have landed (or, unwinding, after a
    //    bounded drain), keeps every receive area alive until nothing more can land in it.
    //    Measured on GB300 the pulled form is faster (0.5-1.4 us per call): a CTA-to-CTA store
    //    takes longer to land than an owner's load takes to return, and the early start does not
    //    make up for it; bulk copies of the staged rows instead of stores did no better.
    // Every thread of every CTA reaches every cluster barrier, on the unwinding path too.
    __syncwarp();
    if (cluster) {
        const bool softmax_warp = warp >= 2 && warp < 2 + kSoftmaxWarps;
        const int n = p.n_split;
        const int lo_row = j * kBlockM / n;
        const int hi_row = (j + 1) * kBlockM / n;
        const int R = (kBlockM + n - 1) / n;  // rows of a receive slot
        const uint32_t sh = ptx::smem_u32(smem + C::kQBytes);  // staged x: [128][kRowHalves] fp16
        const uint32_t sl = sh + kBlockM * C::kRowHalves * 2;  // staged remainders, same layout
        const uint32_t slm = sl + kBlockM * C::kRowHalves * 2; // staged row sums, maxima: [128][kLmw]
        const uint32_t rh = ptx::smem_u32(recv);                  // received x: [kRecvRows][kRowHalves]
        const uint32_t rl = rh + C::kRecvRows * C::kRowHalves * 2;  // received remainders
        const uint32_t rlm = rl + C::kRecvRows * C::kRowHalves * 2; // received [kRecvRows][kLmw]

        // One owner's rows from every rank; kPush: out of the receive area (slot r, row i at
        // r * R + i), else out of each rank's staging.
        auto combine = [&](auto push_tag) {
            constexpr bool kPush = decltype(push_tag)::value;
            constexpr int G = D / 8;  // 16-byte groups (8 fp16 columns) per row
            auto ld4 = [&](uint32_t local, int r) {
                return kPush ? ptx::ld_shared_v4(local) : ptx::ld_cluster_v4(ptx::map_to_rank(local, r));
            };
            auto ld1 = [&](uint32_t local, int r) {
                return kPush ? ptx::ld_shared_f32(local) : ptx::ld_cluster_f32(ptx::map_to_rank(local, r));
            };
            for (int it = threadIdx.x - 64; it < (hi_row - lo_row) * G; it += kSoftmaxThreads) {
                const int rr = lo_row + it / G;
                const int gq = it % G;
                if (m0 + rr >= p.M)
                    continue;
                // Rank r's copy of row rr: its index in the staging (pulled) or the receive area.
                auto row_of = [&](int r) { return static_cast<uint32_t>(kPush ? r * R + (rr - lo_row) : rr); };
                const uint32_t xh = kPush ? rh : sh;
                const uint32_t xl = kPush ? rl : sl;
                const uint32_t xlm = kPush ? rlm : slm;
                const uint32_t col_off = static_cast<uint32_t>(gq * 8 * 2);
                const uint32_t slice = static_cast<uint32_t>((gq * 8) / 32);
                // Max-subtracted variant: every rank's row maximum first, then the weights
                // exp(m_r - max m) (measured faster than requesting them with the values: fewer
                // registers live at once).
                float wt[kMaxClusterRanks];
#pragma unroll
                for (int r = 0; r < kMaxClusterRanks; ++r)
                    wt[r] = 1.f;
                if (kSafeMax) {
                    float mr[kMaxClusterRanks];
                    float mmax = -INFINITY;
#pragma unroll
                    for (int r = 0; r < kMaxClusterRanks; ++r) {
                        if (r < n) {
                            mr[r] = ld1(xlm + (row_of(r) * C::kLmw + D / 32) * 4, r);
                            mmax = fmaxf(mmax, mr[r]);
                        }
                    }
#pragma unroll
                    for (int r = 0; r < kMaxClusterRanks; ++r)
                        if (r < n)
                            wt[r] = ptx::ex2_approx((mr[r] - mmax) * ptx::kLog2e);
                }
                // Every rank's values and row sums are requested before the first is used: the
                // loads are in flight together rather than one round trip after another.
                float4 v[kMaxClusterRanks];
                float c[kMaxClusterRanks];
#pragma unroll
                for (int r = 0; r < kMaxClusterRanks; ++r) {
                    if (r < n) {
                        v[r] = ld4(xh + row_of(r) * C::kRowHalves * 2 + col_off, r);
                        c[r] = ld1(xlm + (row_of(r) * C::kLmw + slice) * 4, r);
                    }
                }
                uint32_t flags = 0;  // ranks that staged remainders for this slice of the row
#pragma unroll
                for (int r = 0; r < kMaxClusterRanks; ++r) {
                    if (r < n) {
                        flags |= (signbit(c[r]) ? 1u : 0u) << r;
                        c[r] = fabsf(c[r]) * wt[r];
                    }
                }
                float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                float lsum = 0.f;
                auto add_halves = [&](const float4 &w, float cr) {
                    const uint32_t words[4] = {__float_as_uint(w.x), __float_as_uint(w.y), __float_as_uint(w.z),
                                               __float_as_uint(w.w)};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&words[h]));
                        a[2 * h] = fmaf(cr, f.x, a[2 * h]);
                        a[2 * h + 1] = fmaf(cr, f.y, a[2 * h + 1]);
                    }
                };
#pragma unroll
                for (int r = 0; r < kMaxClusterRanks; ++r) {
                    if (r < n) {
                        add_halves(v[r], c[r]);
                        lsum += c[r];
                    }
                }
                if (flags) {
                    // Remainders of the flagged ranks: one more round of loads, all in flight.
#pragma unroll
                    for (int r = 0; r < kMaxClusterRanks; ++r)
                        if (r < n && ((flags >> r) & 1u))
                            v[r] = ld4(xl + row_of(r) * C::kRowHalves * 2 + col_off, r);
#pragma unroll
                    for (int r = 0; r < kMaxClusterRanks; ++r)
                        if (r < n && ((flags >> r) & 1u))
                            add_halves(v[r], c[r]);
                }
                const float inv = __frcp_rn(lsum);  // reciprocal, then products (as in the staging)
                uint4 w;
                w.x = ptx::pack_half2(a[0] * inv, a[1] * inv);
                w.y = ptx::pack_half2(a[2] * inv, a[3] * inv);
                w.z = ptx::pack_half2(a[4] * inv, a[5] * inv);
                w.w = ptx::pack_half2(a[6] * inv, a[7] * inv);
                if (p.early == 2)
                    ptx::griddep_wait();
                *reinterpret_cast<uint4 *>(p.O + (static_cast<size_t>(b) * p.M + m0 + rr) * D + gq * 8) = w;
            }
        };

        // The pushed form is a kernel variant of its own (the graph as written), so that the
        // default kernels carry neither its code nor its receive area.
        if constexpr (kPushX) {
            // (The softmax warps passed the first barrier's wait before their first store.)
            if (!softmax_warp)
                ptx::cluster_wait_acquire();
            if (softmax_warp && push_quarters(p, m0, j) > 0) {
                // (A CTA that is unwinding does not wait here; wait_bounded returns at once.)
                if (wait_bounded(wc, bar(BI::kXRecv), 0, BI::kXRecv)) {
                    combine(std::true_type{});
                } else {
                    // Even so, the stores on their way in land before this CTA passes the closing
                    // barrier and releases its shared memory: every rank has issued its stores
                    // and arrivals before any wait of its own.
                    wait_drain(bar(BI::kXRecv), 0, p.timeout_ns);
                }
            }
            ptx::cluster_sync_relaxed();
        } else {
            ptx::cluster_sync();  // every CTA's staging is visible
            if (softmax_warp)
                combine(std::false_type{});
            // Only "every CTA has finished reading the others' shared memory" is needed here; a
            // release would also hold each CTA until its output stores had drained.
            ptx::cluster_sync_relaxed();
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
