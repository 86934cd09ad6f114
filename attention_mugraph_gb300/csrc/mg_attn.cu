// mg_attn.cu -- host side of the C ABI declared in include/mg_attn.h: shape validation and
// planning, the plan's device workspace, TMA tensor-map encoding, kernel launches (with
// programmatic dependent launch), the host-buffer variant and the sticky status word.
#include "mg_attn.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>

#include "mg_attn_kernels.cuh"
#include "mg_attn_pair.cuh"
#include "mg_attn_swap.cuh"
#include "mg_combine.cuh"

namespace {

thread_local char g_last_error[512] = "";

void set_error(const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
}

mg_status fail(mg_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return s;
}

mg_status cuda_fail(cudaError_t e, const char *what)
{
    set_error("%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    return MG_ERR_CUDA;
}

constexpr int64_t kMaxDim = int64_t(1) << 30;
constexpr int64_t kMaxRows = (int64_t(1) << 31) - 1;
constexpr unsigned long long kDefaultTimeoutNs = 1000000000ull;
constexpr int64_t kMaxCluster = mg::kMaxClusterRanks;  // largest thread-block cluster (non-portable size)
// Deepest d = 64 K/V ring beside the pushed combine's receive area (227 KB of shared memory).
constexpr int kPushMaxStages = 5;
static_assert(mg::fwd_smem_bytes(64, kPushMaxStages, true) <= 232448u, "pushed combine exceeds shared memory");

// The driver's tensor-map encoder, fetched through the runtime so that no libcuda link is needed.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// The deepest K/V ring that fits.
int auto_stages(int64_t d) { return d == 64 ? 6 : 3; }

// The window of recent calls whose outputs an early read is compared with (see recent_outputs).
constexpr int kWindow = 16;

// The smallest grid (CTAs of one per SM) that may start early at level 2 (FwdParams::early) on a
// device with `sms` SMs: fewer than kWindow such grids fit the device at once (10 on 152 SMs).
int early_min_ctas(int sms) { return sms / kWindow + 1; }

using FwdKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                           const CUtensorMap, const mg::FwdParams);

template <int VAR>
FwdKernel fwd_kernel_variant(int64_t d, int stages)
{
    if (d == 64) {
        switch (stages) {
        case 2: return mg::mg_attn_fwd_partial<64, 2, VAR>;
        case 3: return mg::mg_attn_fwd_partial<64, 3, VAR>;
        case 4: return mg::mg_attn_fwd_partial<64, 4, VAR>;
        case 5: return mg::mg_attn_fwd_partial<64, 5, VAR>;
        case 6: return mg::mg_attn_fwd_partial<64, 6, VAR>;
        default: return nullptr;
        }
    }
    if (d == 128) {
        switch (stages) {
        case 2: return mg::mg_attn_fwd_partial<128, 2, VAR>;
        case 3: return mg::mg_attn_fwd_partial<128, 3, VAR>;
        default: return nullptr;
        }
    }
    return nullptr;
}

// The two-Q-tile kernel (head dim 64, the graph as written) for a pipeline depth.
FwdKernel pair_kernel(int stages)
{
    switch (stages) {
    case 2: return mg::mg_attn_fwd_pair<2>;
    case 3: return mg::mg_attn_fwd_pair<3>;
    case 4: return mg::mg_attn_fwd_pair<4>;
    case 5: return mg::mg_attn_fwd_pair<5>;
    case 6: return mg::mg_attn_fwd_pair<6>;
    default: return nullptr;
    }
}

// The few-row specialisation (head dim 128, transposed products) for a pipeline depth and form
// (the graph as written, its one-pass max-subtracted evaluation, QK-norm on that).
template <int STAGES>
FwdKernel swap_kernel_form(int form)
{
    return form == mg::kSwapQkNormForm   ? mg::mg_attn_fwd_swap<STAGES, mg::kSwapQkNormForm>
           : form == mg::kSwapOnlineForm ? mg::mg_attn_fwd_swap<STAGES, mg::kSwapOnlineForm>
                                         : mg::mg_attn_fwd_swap<STAGES, mg::kSwapPlainForm>;
}

FwdKernel swap_kernel(int stages, int flags)
{
    const int form = (flags & MG_FLAG_QK_NORM)        ? mg::kSwapQkNormForm
                     : (flags & MG_FLAG_SAFE_SOFTMAX) ? mg::kSwapOnlineForm
                                                      : mg::kSwapPlainForm;
    switch (stages) {
    case 2: return swap_kernel_form<2>(form);
    case 3: return swap_kernel_form<3>(form);
    default: return nullptr;
    }
}

// The one-tile kernel under the stream-K schedule (the graph as written).
FwdKernel sk_kernel(int64_t d, int stages) { return fwd_kernel_variant<mg::kStreamK>(d, stages); }

// The pushed on-chip combine: head dim 64, at most kPushMaxStages stages.
FwdKernel push_kernel(int stages)
{
    switch (stages) {
    case 2: return mg::mg_attn_fwd_partial<64, 2, mg::kPush>;
    case 3: return mg::mg_attn_fwd_partial<64, 3, mg::kPush>;
    case 4: return mg::mg_attn_fwd_partial<64, 4, mg::kPush>;
    case 5: return mg::mg_attn_fwd_partial<64, 5, mg::kPush>;
    default: return nullptr;
    }
}

// The fused kernel for a head dim, pipeline depth and the MG_FLAG_* evaluation flags.
FwdKernel fwd_kernel(int64_t d, int stages, int flags)
{
    if (flags & MG_FLAG_QK_NORM)
        return fwd_kernel_variant<mg::kQkNorm>(d, stages);
    if (flags & MG_FLAG_SAFE_SOFTMAX)
        return fwd_kernel_variant<mg::kSafe>(d, stages);
    return fwd_kernel_variant<mg::kPlain>(d, stages);
}

using CombineKernel = void (*)(const float *, const float *, const float *, __half *, int, int, int);

template <int D>
CombineKernel combine_kernel_d(int n_split)
{
    if (n_split <= mg::CombineCfg<D>::kMaxSplits)
        return mg::mg_attn_combine<D>;
    return mg::WideCombineCfg<D>::batch(n_split) == 4 ? mg::mg_attn_combine_wide<D, 4> : mg::mg_attn_combine_wide<D, 8>;
}

template <int D>
int combine_rows_per_cta(int n_split)
{
    return n_split <= mg::CombineCfg<D>::kMaxSplits ? mg::CombineCfg<D>::kRows : mg::WideCombineCfg<D>::kRows;
}

// The second kernel for a head dim and split count (its load batch depends on the split count).
CombineKernel combine_kernel(int64_t d, int n_split)
{
    return d == 64 ? combine_kernel_d<64>(n_split) : combine_kernel_d<128>(n_split);
}

// Stream-K partial slots per row tile: the most CTAs whose runs touch one row tile.
int64_t sk_slots(int64_t rows, int64_t n_tiles, int64_t G)
{
    const int64_t U = rows * n_tiles;
    int64_t most = 1;
    for (int64_t r = 0; r < rows; ++r)
        most = std::max<int64_t>(most, mg::sk_cta_of((r + 1) * n_tiles - 1, U, G) - mg::sk_cta_of(r * n_tiles, U, G) + 1);
    return most;
}

// Rows of partials per split: B*M for the second kernel; for the cluster combine, whole tiles of
// min(M, 128) rows.
int64_t partial_rows(int64_t B, int64_t M, bool cluster)
{
    const int64_t tile_rows = M < mg::kBlockM ? M : mg::kBlockM;
    return cluster ? B * ((M + mg::kBlockM - 1) / mg::kBlockM) * tile_rows : B * M;
}

// Validation and tiling decisions; touches no GPU.
mg_status decide(int64_t B, int64_t M, int64_t N, int64_t d, const mg_attn_options *opts, int32_t num_sms,
                 int32_t max_smem, mg_attn_plan_info *info, unsigned long long *timeout_ns, int *flags)
{
    if (!info)
        return fail(MG_ERR_INVALID_ARG, "info is NULL");
    if (B <= 0 || M <= 0 || N <= 0 || d <= 0)
        return fail(MG_ERR_INVALID_ARG, "dimensions must be positive (B=%lld M=%lld N=%lld d=%lld)", (long long)B,
                    (long long)M, (long long)N, (long long)d);
    if (B > kMaxDim || M > kMaxDim || N > kMaxDim || B * M > kMaxRows)
        return fail(MG_ERR_INVALID_ARG, "dimensions too large (B, M, N <= 2^30 and B*M < 2^31)");
    if (d != 64 && d != 128)
        return fail(MG_ERR_UNSUPPORTED, "head dim d=%lld not supported (64 or 128)", (long long)d);
    if (N % 8 != 0)
        return fail(MG_ERR_LAYOUT, "N=%lld must be a multiple of 8 (16-byte row stride of K for TMA)",
                    (long long)N);
    if (num_sms <= 0)
        return fail(MG_ERR_INVALID_ARG, "num_sms must be positive");
    mg_attn_options o{};
    if (opts)
        o = *opts;
    if (o.reserved != 0 ||
        (o.flags & ~(MG_FLAG_NO_PDL | MG_FLAG_INJECT_TIMEOUT | MG_FLAG_NO_CLUSTER | MG_FLAG_SAFE_SOFTMAX |
                     MG_FLAG_QK_NORM | MG_FLAG_Q_PAIRS | MG_FLAG_NO_Q_PAIRS | MG_FLAG_STREAM_K |
                     MG_FLAG_NO_STREAM_K | MG_FLAG_SWAP_AB | MG_FLAG_NO_SWAP_AB | MG_FLAG_PUSH_COMBINE |
                     MG_FLAG_NO_EARLY_LOADS | MG_FLAG_ISOLATED)) != 0)
        return fail(MG_ERR_CONFIG, "unknown option bits");
    if (o.timeout_ns != 0 && (o.timeout_ns < 1000 || o.timeout_ns > 60000000000LL))
        return fail(MG_ERR_CONFIG, "timeout_ns out of range [1e3, 6e10]");

    const int64_t m_tiles_per_b = (M + mg::kBlockM - 1) / mg::kBlockM;
    const int64_t m_tiles = B * m_tiles_per_b;
    const int64_t n_tiles = (N + mg::kBlockN - 1) / mg::kBlockN;
    if ((o.flags & MG_FLAG_Q_PAIRS) && (o.flags & MG_FLAG_NO_Q_PAIRS))
        return fail(MG_ERR_CONFIG, "MG_FLAG_Q_PAIRS and MG_FLAG_NO_Q_PAIRS together");
    if ((o.flags & MG_FLAG_STREAM_K) && (o.flags & MG_FLAG_NO_STREAM_K))
        return fail(MG_ERR_CONFIG, "MG_FLAG_STREAM_K and MG_FLAG_NO_STREAM_K together");
    if ((o.flags & MG_FLAG_SWAP_AB) && (o.flags & MG_FLAG_NO_SWAP_AB))
        return fail(MG_ERR_CONFIG, "MG_FLAG_SWAP_AB and MG_FLAG_NO_SWAP_AB together");

    // One wave: as many splits per unit (a row tile, or a pair of them) as keep every SM busy,
    // never fewer than one column tile per split.
    auto one_wave = [&](int64_t units) {
        int64_t n = units >= num_sms ? 1 : num_sms / units;
        return n > n_tiles ? n_tiles : (n < 1 ? 1 : n);
    };
    // The two-Q-tile kernel applies to head dim 64, the graph as written and an even number of
    // row tiles per batch, and only on request: measured on GB300 it is slower than the one-tile
    // kernel on every workload (its per-tile loop is no faster, and it needs twice the splits for
    // one wave).
    const bool pair_applies = d == 64 && !(o.flags & (MG_FLAG_SAFE_SOFTMAX | MG_FLAG_QK_NORM)) &&
                              m_tiles_per_b % 2 == 0;
    const bool pair = pair_applies && (o.flags & MG_FLAG_Q_PAIRS);
    const int64_t units = pair ? m_tiles / 2 : m_tiles;  // CTAs per split

    int64_t n_split = o.n_split;
    if (n_split < 0 || n_split > n_tiles)
        return fail(MG_ERR_CONFIG, "n_split=%lld out of range [0, %lld]", (long long)n_split, (long long)n_tiles);
    if (n_split == 0) {
        n_split = one_wave(units);
        // Few query rows per batch (at most 64, so a tile's arithmetic per byte of K/V is low and
        // HBM bounds the call): every split streams its tiles at the device's shared bandwidth, and
        // the call lasts as long as the longest split. Among the split counts down to 4/5 of one
        // wave, take the one that leaves the fewest idle tile slots, n * ceil(n_tiles / n) - n_tiles
        // (the largest on a tie). Measured on GB300 for (16, 8, 32768, 128): 8 splits of 32 tiles,
        // 48.3 us per call, against 9 splits of 28 or 29 tiles, 49.1 us.
        if (M <= 64 && n_split > 1) {
            int64_t best = n_split, best_waste = n_split * ((n_tiles + n_split - 1) / n_split) - n_tiles;
            for (int64_t n = n_split - 1; n >= 1 && 5 * n >= 4 * one_wave(units); --n) {
                const int64_t waste = n * ((n_tiles + n - 1) / n) - n_tiles;
                if (waste < best_waste) {
                    best = n;
                    best_waste = waste;
                }
            }
            n_split = best;
        }
        // Small problems: rather than more than 16 splits and a second kernel, take the largest
        // cluster (16) when that leaves at most 4 column tiles per CTA.
        if (n_split > kMaxCluster && !(o.flags & MG_FLAG_NO_CLUSTER) &&
            (n_tiles + kMaxCluster - 1) / kMaxCluster <= 4)
            n_split = kMaxCluster;
    }
    // Stream-K applies to the graph as written with at most 16 query rows per batch (one compact
    // Q tile per segment, a batch being one row tile), no explicit split, and runs of at most
    // n_tiles units (so a CTA touches at most two batches), and only on request: measured on
    // GB300 it is not faster on the decode shapes, which are bound by DRAM throughput (both
    // schedules stream ~5.4 TB/s there) rather than by uneven CTAs, and its contiguous runs give
    // concurrent CTAs K rows far apart where the split schedule's interleaved tiles keep them in
    // neighbouring DRAM locations; (16, 8, 32768, 128): 49.3 against 48.3 us per call,
    // (64, 1, 4096, 128): 28.2 against 26.7 (there also the second kernel against the cluster).
    bool stream_k = false;
    int64_t sk_ctas = 0;
    if (!pair && M <= mg::kSkQRows && o.n_split == 0 && !(o.flags & (MG_FLAG_SAFE_SOFTMAX | MG_FLAG_QK_NORM)) &&
        !(o.flags & MG_FLAG_NO_STREAM_K)) {
        const int64_t U = m_tiles * n_tiles;
        sk_ctas = U < num_sms ? U : num_sms;
        const int64_t run = (U + sk_ctas - 1) / sk_ctas;
        const int64_t split_run = (n_tiles + n_split - 1) / n_split;
        stream_k = run <= n_tiles && sk_ctas >= 2 && (o.flags & MG_FLAG_STREAM_K) && run <= split_run;
    }
    if (stream_k) {
        n_split = sk_slots(m_tiles, n_tiles, sk_ctas);
        if (n_split < 2)  // every run within one batch and every batch in one run: nothing to combine
            stream_k = false, n_split = one_wave(units);
    }
    // The few-row specialisation: head dim 128, at most 16 query rows per batch, the graph as
    // written, its max-subtracted evaluation or QK-norm (both in one pass there), under the split
    // schedule; the default there (measured on GB300, us per call against the one-tile kernel:
    // (16, 8, 32768, 128) 45.8 against 48.2, (64, 1, 4096, 128) 25.2 against 26.9).
    const bool swap = !pair && !stream_k && d == 128 && M <= mg::kSwapNQ && !(o.flags & MG_FLAG_NO_SWAP_AB);
    const bool safe = (o.flags & (MG_FLAG_SAFE_SOFTMAX | MG_FLAG_QK_NORM)) != 0;
    // The few-row kernel combines on chip too (fp32 partials; measured on GB300 for (64, 1, 4096,
    // 128), 2 splits: 24.3 us per call against 25.1 with the second kernel).
    const bool cluster =
        !stream_k && !(o.flags & MG_FLAG_NO_CLUSTER) && n_split >= 2 && n_split <= kMaxCluster;
    if (!stream_k && units * n_split > 0x7fffffffLL)
        return fail(MG_ERR_INVALID_ARG, "grid too large");

    const bool qk_norm = (o.flags & MG_FLAG_QK_NORM) != 0;
    int stages = o.stages == 0 ? auto_stages(d) : o.stages;
    if (stages < 2 || stages > 6)
        return fail(MG_ERR_CONFIG, "stages=%d out of range [2, 6]", stages);
    // The pushed on-chip combine applies to the graph as written at head dim 64 (its receive area
    // takes the place of one K/V stage; d = 128 has no room for it) unless an explicit depth leaves
    // no room, and only on request: measured on GB300 it is slower than the pulled form, us per
    // call (2, 256, 4096, 64) 7.55 against 6.56, (2, 64, 1024, 64) 5.79 against 5.28,
    // (16, 256, 4096, 64) 11.40 against 10.00 (the pulled form at 5 stages: 6.60, 5.29, 10.22).
    bool push = cluster && !pair && d == 64 && !(o.flags & (MG_FLAG_SAFE_SOFTMAX | MG_FLAG_QK_NORM)) &&
                (o.flags & MG_FLAG_PUSH_COMBINE);
    if (push && stages > kPushMaxStages) {
        if (o.stages == 0)
            stages = kPushMaxStages;
        else
            push = false;
    }
    uint32_t smem = pair   ? mg::pair_smem_bytes(stages)
                    : swap ? mg::swap_smem_bytes(stages, safe)
                           : mg::fwd_smem_bytes(static_cast<int>(d), stages, push);
    // QK-norm in the one-tile kernel under the split schedule: the CTA's key-vector scales (128
    // floats per column tile) in shared memory after the fixed layout, where they fit beside the
    // ring, so that no global memory is written before the epilogue (the call may start early).
    if (qk_norm && !pair && !swap && !stream_k) {
        const int64_t per_cta = (n_tiles + n_split - 1) / n_split;
        if (static_cast<int64_t>(smem) + per_cta * mg::kBlockN * 4 <= max_smem)
            smem += static_cast<uint32_t>(per_cta * mg::kBlockN * 4);
    }
    if (static_cast<int64_t>(smem) > max_smem ||
        !(pair ? pair_kernel(stages)
               : swap ? swap_kernel(stages, o.flags)
                      : stream_k ? sk_kernel(d, stages) : push ? push_kernel(stages) : fwd_kernel(d, stages, o.flags)))
        return fail(MG_ERR_INSUFFICIENT_SMEM, "d=%lld with %d stages needs %u bytes of shared memory (limit %d)",
                    (long long)d, stages, smem, max_smem);

    std::memset(info, 0, sizeof(*info));
    info->B = B;
    info->M = M;
    info->N = N;
    info->d = d;
    info->block_m = mg::kBlockM;
    info->block_n = mg::kBlockN;
    info->m_tiles = static_cast<int32_t>(m_tiles);
    info->n_tiles = static_cast<int32_t>(n_tiles);
    info->n_split = static_cast<int32_t>(n_split);
    info->stages = stages;
    info->threads = mg::kThreads;
    info->grid_ctas = static_cast<int32_t>(stream_k ? sk_ctas : units * n_split);
    info->smem_bytes = static_cast<int32_t>(smem);
    info->tmem_cols = static_cast<int32_t>(mg::kTmemCols);
    // The fused kernel writes O itself unless split partials go through the second kernel.
    info->kernels_per_run = (n_split > 1 && !cluster) ? 2 : 1;
    info->num_sms = num_sms;
    // Split partials in the workspace: numerators, row sums and (max-subtracted variant) row maxima,
    // for every split and row, for the second kernel and for the two-Q-tile kernel's cluster
    // combine (which keeps whole row tiles); the one-tile kernel's cluster combine exchanges them
    // on chip.
    const int64_t row_words = (o.flags & (MG_FLAG_SAFE_SOFTMAX | MG_FLAG_QK_NORM)) ? 2 : 1;
    const bool ws_partials = n_split > 1 && (!cluster || pair);
    const int64_t partial_bytes =
        ws_partials ? n_split * partial_rows(B, M, cluster && pair) * (d + row_words) * 4 : 0;
    // QK-norm: key-vector scales (B*N floats, then 128 more that reads of a last tile past N may
    // touch), from a 256-byte boundary.
    const int64_t scale_bytes = qk_norm ? 256 + (B * N + 128) * 4 : 0;
    info->workspace_bytes = 256 + partial_bytes + scale_bytes;
    info->cluster_ctas = cluster ? static_cast<int32_t>(n_split) : 0;
    info->q_tiles_per_cta = pair ? 2 : 1;
    info->schedule = stream_k ? 1 : 0;
    info->swap_ab = swap ? 1 : 0;
    info->xchg_push = push ? 1 : 0;
    if (timeout_ns)
        *timeout_ns = o.timeout_ns ? static_cast<unsigned long long>(o.timeout_ns) : kDefaultTimeoutNs;
    if (flags)
        *flags = o.flags;
    g_last_error[0] = '\0';
    return MG_OK;
}

// The fused kernel a plan's decisions call for.
FwdKernel plan_kernel(const mg_attn_plan_info &info, int flags)
{
    if (info.swap_ab == 1)
        return swap_kernel(info.stages, flags);
    if (info.schedule == 1)
        return sk_kernel(info.d, info.stages);
    if (info.xchg_push == 1)
        return push_kernel(info.stages);
    return info.q_tiles_per_cta == 2 ? pair_kernel(info.stages) : fwd_kernel(info.d, info.stages, flags);
}


// Host-buffer entry point: copies between the caller's pinned host buffers (read and written
// through their device-mapped addresses over the CPU-GPU link) and the plan's device staging, in
// 16-byte units. Up to three (src, dst, units) jobs per launch, walked as one index space with a
// grid stride. With `early`, each thread loads its first kEarlyUnits units before it waits for
// the previous grid on the stream, and stores them after: the loads of a call's inputs cross the
// link while the previous call's kernels still run (they only wait to be stored into staging that
// those kernels may still read).
constexpr int kEarlyUnits = 4;
struct CopyJobs {
    const uint4 *src[3];
    uint4 *dst[3];
    unsigned long long units[3];
    int early;  // the sources are final before the previous grid ends (host inputs)
};

__global__ void __launch_bounds__(512) mg_copy_units(const CopyJobs jobs)
{
    const unsigned long long n0 = jobs.units[0], n01 = n0 + jobs.units[1], n = n01 + jobs.units[2];
    const unsigned long long stride = static_cast<unsigned long long>(gridDim.x) * blockDim.x;
    const unsigned long long first = static_cast<unsigned long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    auto src_of = [&](unsigned long long u) {
        return u < n0 ? jobs.src[0] + u : u < n01 ? jobs.src[1] + (u - n0) : jobs.src[2] + (u - n01);
    };
    auto dst_of = [&](unsigned long long u) {
        return u < n0 ? jobs.dst[0] + u : u < n01 ? jobs.dst[1] + (u - n0) : jobs.dst[2] + (u - n01);
    };
    unsigned long long u = first;
    if (jobs.early) {
        uint4 v[kEarlyUnits];
#pragma unroll
        for (int k = 0; k < kEarlyUnits; ++k) {
            const unsigned long long e = first + k * stride;
            if (e < n)
                v[k] = *src_of(e);
        }
        mg::ptx::griddep_wait();  // the staging buffers may still be read by the previous call's kernels
        mg::ptx::griddep_launch_dependents();
#pragma unroll
        for (int k = 0; k < kEarlyUnits; ++k) {
            const unsigned long long e = first + k * stride;
            if (e < n)
                *dst_of(e) = v[k];
        }
        u = first + kEarlyUnits * stride;
    } else {
        mg::ptx::griddep_wait();  // the sources may be written by the previous kernels
        mg::ptx::griddep_launch_dependents();
    }
    for (; u + 3 * stride < n; u += 4 * stride) {
        const uint4 a = *src_of(u), b = *src_of(u + stride), c = *src_of(u + 2 * stride), d = *src_of(u + 3 * stride);
        *dst_of(u) = a;
        *dst_of(u + stride) = b;
        *dst_of(u + 2 * stride) = c;
        *dst_of(u + 3 * stride) = d;
    }
    for (; u < n; u += stride)
        *dst_of(u) = *src_of(u);
}

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// Whether a host pointer is page-locked host memory the device can address (its device address in
// *dev); false for pageable memory or on any query error (which is cleared).
bool device_mapped(const void *p, void **dev)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr || misaligned(a.devicePointer))
        return false;
    *dev = a.devicePointer;
    return true;
}

// One launch of the 16-byte copy kernel, PDL when allowed: two CTAs of 512 threads per SM, or
// with early loads just enough CTAs that every unit is among a thread's first kEarlyUnits (so a
// small copy fits beside the previous call's kernels and all of it is loaded before the wait).
cudaError_t launch_copy(const CopyJobs &jobs, int num_sms, bool pdl, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    unsigned long long grid = 2ull * static_cast<unsigned long long>(num_sms);
    if (jobs.early) {
        const unsigned long long units = jobs.units[0] + jobs.units[1] + jobs.units[2];
        const unsigned long long need = (units + 512ull * kEarlyUnits - 1) / (512ull * kEarlyUnits);
        grid = need < 1 ? 1 : (need < grid ? need : grid);
    }
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(512, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, mg_copy_units, jobs);
}

// Whether the current device can hold all ctas / n clusters of n CTAs of the fused kernel at
// once (one wave: a cluster left for a second wave would double the time). Sizes above 8 need
// the non-portable opt-in. Clears any error it provokes.
// How many clusters of n CTAs of `fwd` (with `smem` bytes of dynamic shared memory each) the
// device holds at once; -1 if the query fails.
int max_active_clusters(FwdKernel fwd, int n, int ctas, int smem)
{
    if (n > 8 && cudaFuncSetAttribute(reinterpret_cast<const void *>(fwd),
                                      cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(mg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeClusterDimension;
    a.val.clusterDim.x = static_cast<unsigned>(n);
    a.val.clusterDim.y = 1;
    a.val.clusterDim.z = 1;
    cfg.attrs = &a;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, reinterpret_cast<const void *>(fwd), &cfg) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return clusters;
}

// QK-norm in the one-tile kernel: how many column tiles of key-vector scales the plan keeps in
// shared memory (the bytes decide() added past the fixed layout), 0 when they go through global
// memory.
int qk_cs_tiles(const mg_attn_plan_info &in, int flags)
{
    if (!(flags & MG_FLAG_QK_NORM) || in.swap_ab != 0 || in.q_tiles_per_cta != 1 || in.schedule != 0)
        return 0;
    const int fixed = static_cast<int>(mg::fwd_smem_bytes(static_cast<int>(in.d), in.stages, in.xchg_push != 0));
    return (in.smem_bytes - fixed) / (mg::kBlockN * 4);
}

// The kernel's dynamic shared-memory limit raised to the plan's (before any occupancy query: at
// the default 48 KB limit the query would refuse the launch).
cudaError_t raise_smem_limit(FwdKernel fwd, int smem)
{
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(fwd), cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

// Places the on-chip combine's clusters on the device (the plan's kernel limit already raised).
// Back to back, a call's CTAs start while the previous call runs (programmatic dependent launch)
// and load early, but a cluster starts only where the device has room for it beside the previous
// call's clusters; the device holds fewer clusters of 13-16 CTAs than of 11-12 (GB300: 7 and 8).
// Without an explicit n_split, when two calls' clusters do not fit side by side, a smaller
// cluster with at most one more column tile per CTA that lets them is taken; failing that, when
// even one call's clusters do not fit, a smaller cluster that fits with at most two more, and
// failing that the second-kernel combine. Measured on GB300 (us per call, back to back):
// (2, 256, 4096, 64) 5.80 with 12 splits against 6.21 with 16 (of which 7 clusters fit at once,
// not the 8 of two calls); (4, 256, 4096, 64) 7.22 with 12 against 8.41 with 16 through the
// second kernel; (8, 256, 4096, 64) 8.11 with 6 against 9.66 with 9 through the second kernel.
mg_status fit_clusters(int64_t B, int64_t M, int64_t N, int64_t d, const mg_attn_options *opts, int sms,
                       int smem_optin, mg_attn_plan_info *info, unsigned long long *timeout_ns, int *flags,
                       FwdKernel *fwd)
{
    if (info->cluster_ctas == 0)
        return MG_OK;
    const int n = info->cluster_ctas;
    const int units = info->grid_ctas / n;
    const int act = max_active_clusters(*fwd, n, info->grid_ctas, info->smem_bytes);
    if (act >= 2 * units)
        return MG_OK;
    mg_attn_options o{};
    if (opts)
        o = *opts;
    // The one-tile kernel's two-pass variants stream each tile twice: one more tile per CTA costs
    // them more than the overlap gains (QK-norm on (2, 256, 4096, 64): 10.58 us with 12 splits
    // against 9.59 with 16), so they change the cluster only when it does not fit.
    const bool two_pass = (*flags & (MG_FLAG_SAFE_SOFTMAX | MG_FLAG_QK_NORM)) && info->swap_ab == 0;
    if (o.n_split == 0) {
        const int t = (info->n_tiles + n - 1) / n;
        for (int pass = two_pass ? 1 : 0; pass < 2; ++pass) {
            if (pass == 1 && act >= units)
                break;
            for (int c = n - 1; c >= 2 && (info->n_tiles + c - 1) / c <= t + 1 + pass; --c) {
                mg_attn_options oc = o;
                oc.n_split = c;
                mg_attn_plan_info ic;
                unsigned long long to = 0;
                int fl = 0;
                if (decide(B, M, N, d, &oc, sms, smem_optin, &ic, &to, &fl) != MG_OK || ic.cluster_ctas != c)
                    continue;
                FwdKernel f = plan_kernel(ic, fl);
                if (raise_smem_limit(f, ic.smem_bytes) != cudaSuccess) {
                    cudaGetLastError();
                    continue;
                }
                const int u = ic.grid_ctas / c;
                if (max_active_clusters(f, c, ic.grid_ctas, ic.smem_bytes) >= (pass == 0 ? 2 * u : u)) {
                    *info = ic;
                    *timeout_ns = to;
                    *flags = fl;
                    *fwd = f;
                    return MG_OK;
                }
            }
        }
    }
    if (act >= units)
        return MG_OK;
    // The device cannot place the clusters: plan again with the second-kernel combine (whose
    // kernel carries that epilogue: its limit is raised as well).
    o.flags |= MG_FLAG_NO_CLUSTER;
    mg_status st = decide(B, M, N, d, &o, sms, smem_optin, info, timeout_ns, flags);
    if (st != MG_OK)
        return st;
    *fwd = plan_kernel(*info, *flags);
    const cudaError_t e = raise_smem_limit(*fwd, info->smem_bytes);
    return e == cudaSuccess ? MG_OK : cuda_fail(e, "cudaFuncSetAttribute");
}

// Split count for back-to-back calls that start early (level 2, FwdParams::early): such calls
// overlap as far as the device holds their clusters, so a call's cost is its latency divided by
// the number of calls in flight, not its latency. A smaller split count puts more column tiles on
// each CTA (a longer call) but lets more calls be resident together. Without an explicit n_split,
// for a cluster plan that may start early, the split count from the one placed down to 2 that
// keeps at most max(8, the placed count's) column tiles per CTA (twice the placed count's when
// that lets no second call in) and a grid of at least early_min_ctas CTAs, and that maximises
// min(4, clusters the device holds / clusters per call, SMs / grid) is taken (the larger on a
// tie). Measured on GB300 (us per call, back to back at
// level 2; isolated, each call between events of its own): (2, 256, 4096, 64) 6 splits 1.83 and
// 12.64 against 12 splits 3.67 and 12.45; 8 splits 2.36 and 12.48; 4 splits 1.81 and 14.5;
// (4, 256, 4096, 64) 4 splits 2.40 against 6 splits 3.48 and 12 splits 7.32; (2, 256, 4096, 128)
// 6 splits 2.44 against 12 splits 4.51.
mg_status pipeline_splits(int64_t B, int64_t M, int64_t N, int64_t d, const mg_attn_options *opts, int sms,
                          int smem_optin, mg_attn_plan_info *info, unsigned long long *timeout_ns, int *flags,
                          FwdKernel *fwd)
{
    // (QK-norm in the one-tile kernel starts early only with its key scales in shared memory.)
    const bool qk_one_tile = (*flags & MG_FLAG_QK_NORM) && info->swap_ab == 0;
    if (info->cluster_ctas < 2 || (opts && opts->n_split != 0) || info->schedule != 0 || info->q_tiles_per_cta != 1 ||
        (qk_one_tile && qk_cs_tiles(*info, *flags) == 0) || (*flags & MG_FLAG_ISOLATED))
        return MG_OK;
    const int n = info->cluster_ctas;
    const int units = info->grid_ctas / n;
    auto tiles = [&](int c) { return (info->n_tiles + c - 1) / c; };
    auto in_flight = [&](FwdKernel f, int c, int grid, int smem) {
        const int a = max_active_clusters(f, c, grid, smem) / units;
        const int by_sms = sms / grid;
        const int m = a < by_sms ? a : by_sms;
        return m < 4 ? m : 4;
    };
    int best = in_flight(*fwd, n, info->grid_ctas, info->smem_bytes);
    // A placed count that lets no second call in takes up to twice its tiles per CTA, except in
    // the one-tile kernel's two-pass variants, whose calls alone would lose more than their
    // overlap gains (measured on GB300, (16, 256, 4096, 64), 4 against 2 splits, back to back /
    // alone in us: plain 9.13 / 14.6 against 6.93 / 18.7; max-subtracted 12.2 / 18.6 against
    // 9.55 / 24.9; QK-norm 16.5 / 22.8 against 13.4 / 34.9).
    const bool two_pass = (*flags & (MG_FLAG_SAFE_SOFTMAX | MG_FLAG_QK_NORM)) && info->swap_ab == 0;
    const int base = best >= 2 || two_pass ? tiles(n) : 2 * tiles(n);
    const int bound = base > 8 ? base : 8;
    mg_attn_options o{};
    if (opts)
        o = *opts;
    for (int c = n - 1; c >= 2 && tiles(c) <= bound && units * c >= early_min_ctas(sms); --c) {
        mg_attn_options oc = o;
        oc.n_split = c;
        mg_attn_plan_info ic;
        unsigned long long to = 0;
        int fl = 0;
        if (decide(B, M, N, d, &oc, sms, smem_optin, &ic, &to, &fl) != MG_OK || ic.cluster_ctas != c ||
            (qk_one_tile && qk_cs_tiles(ic, fl) == 0))
            continue;
        FwdKernel f = plan_kernel(ic, fl);
        if (raise_smem_limit(f, ic.smem_bytes) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        const int k = in_flight(f, c, ic.grid_ctas, ic.smem_bytes);
        if (k > best) {
            best = k;
            *info = ic;
            *timeout_ns = to;
            *flags = fl;
            *fwd = f;
        }
    }
    return MG_OK;
}

// Cluster placement, then the split count for calls that start early.
mg_status place_clusters(int64_t B, int64_t M, int64_t N, int64_t d, const mg_attn_options *opts, int sms,
                         int smem_optin, mg_attn_plan_info *info, unsigned long long *timeout_ns, int *flags,
                         FwdKernel *fwd)
{
    const mg_status st = fit_clusters(B, M, N, d, opts, sms, smem_optin, info, timeout_ns, flags, fwd);
    return st == MG_OK ? pipeline_splits(B, M, N, d, opts, sms, smem_optin, info, timeout_ns, flags, fwd) : st;
}

// Launch attributes of the fused kernel: programmatic dependent launch and the cluster shape.
int fused_launch_attrs(cudaLaunchAttribute (&attr)[2], bool pdl, int cluster_ctas)
{
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_ctas > 0) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_ctas);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    return n;
}

// 3-D tensor map over a contiguous (d2, d1, d0) array (d0 innermost) of fp16 (elem = 2) or fp32
// (elem = 4) with a box of box0 x box1 x 1 elements and 128-byte swizzle; out-of-range elements
// read as zero and are not written.
mg_status encode_3d(CUtensorMap *map, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                    uint32_t box1, uint32_t elem = 2)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc)
        return fail(MG_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * elem, d0 * d1 * elem};
    cuuint32_t box[3] = {box0, box1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = elem == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = enc(map, dt, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MG_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult %d", static_cast<int>(r));
    return MG_OK;
}

}  // namespace

struct mg_attn_plan {
    int device = -1;
    mg_attn_plan_info info{};
    int flags = 0;
    unsigned long long timeout_ns = kDefaultTimeoutNs;
    void *workspace = nullptr;  // [status words | ws_o | ws_l | ws_m (max-subtracted variant)]
    int *status = nullptr;
    float *ws_o = nullptr;
    float *ws_l = nullptr;
    float *ws_m = nullptr;
    float *col_scale = nullptr;  // QK-norm: (B, N) key-vector scales, then 128 spare floats
    FwdKernel fwd = nullptr;
    CombineKernel combine = nullptr;
    // Tensor maps Q, K, V, O (re-encoded when a pointer changes) and the fp32 partial workspace
    // (encoded once; zero when the plan has one split and no workspace).
    const void *map_ptr[4] = {nullptr, nullptr, nullptr, nullptr};
    CUtensorMap maps[5];
    // Device staging for mg_attn_run_host, allocated by its first call.
    void *staging = nullptr;
    // Optional events recorded around the fused kernel (mg_attn_set_timing_events).
    cudaEvent_t ev_begin = nullptr;
    cudaEvent_t ev_end = nullptr;
};

extern "C" {

int32_t mg_attn_version(void) { return 10000; }

const char *mg_attn_status_string(mg_status s)
{
    switch (s) {
    case MG_OK: return "success";
    case MG_ERR_INSUFFICIENT_SMEM: return "insufficient shared memory for the tile configuration";
    case MG_ERR_LAYOUT: return "layout error (alignment or N % 8)";
    case MG_ERR_CONFIG: return "configuration error (option out of range)";
    case MG_ERR_INVALID_ARG: return "invalid argument";
    case MG_ERR_UNSUPPORTED: return "unsupported head dim or device";
    case MG_ERR_CUDA: return "CUDA error";
    case MG_ERR_TIMEOUT: return "in-kernel wait timed out";
    }
    return "unknown status";
}

const char *mg_attn_last_error(void) { return g_last_error; }

mg_status mg_attn_query(int64_t B, int64_t M, int64_t N, int64_t d, const mg_attn_options *opts, int32_t num_sms,
                        int32_t max_smem_optin, mg_attn_plan_info *info)
{
    return decide(B, M, N, d, opts, num_sms, max_smem_optin, info, nullptr, nullptr);
}

mg_status mg_attn_plan_ex(int64_t B, int64_t M, int64_t N, int64_t d, const mg_attn_options *opts,
                          mg_attn_plan_t *out)
{
    if (!out)
        return fail(MG_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    int major = 0, minor = 0, sms = 0, smem_optin = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3)
        return fail(MG_ERR_UNSUPPORTED, "device %d has compute capability %d.%d; this library is built for 10.3", dev,
                    major, minor);

    mg_attn_plan_info info;
    unsigned long long timeout_ns = 0;
    int flags = 0;
    mg_status st = decide(B, M, N, d, opts, sms, smem_optin, &info, &timeout_ns, &flags);
    if (st != MG_OK)
        return st;

    FwdKernel fwd = plan_kernel(info, flags);
    e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fwd), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             info.smem_bytes);
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
        return fail(MG_ERR_UNSUPPORTED, "no sm_103a kernel image for device %d", dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute");
    if ((st = place_clusters(B, M, N, d, opts, sms, smem_optin, &info, &timeout_ns, &flags, &fwd)) != MG_OK)
        return st;

    struct mg_attn_plan *p = new (std::nothrow) struct mg_attn_plan();
    if (!p)
        return fail(MG_ERR_CUDA, "out of host memory");
    p->device = dev;
    p->info = info;
    p->flags = flags;
    p->timeout_ns = timeout_ns;
    p->fwd = fwd;
    p->combine = combine_kernel(d, info.n_split);
    e = cudaMalloc(&p->workspace, static_cast<size_t>(info.workspace_bytes));
    if (e != cudaSuccess) {
        delete p;
        return cuda_fail(e, "cudaMalloc(workspace)");
    }
    uint8_t *ws = static_cast<uint8_t *>(p->workspace);
    p->status = reinterpret_cast<int *>(ws);
    std::memset(p->maps, 0, sizeof(p->maps));
    const bool l2_cluster = info.cluster_ctas > 0 && info.q_tiles_per_cta == 2;
    if (info.n_split > 1 && (info.cluster_ctas == 0 || l2_cluster)) {
        const size_t rows = static_cast<size_t>(info.n_split) * partial_rows(B, M, l2_cluster);
        p->ws_o = reinterpret_cast<float *>(ws + 256);
        p->ws_l = p->ws_o + rows * d;
        if (flags & (MG_FLAG_SAFE_SOFTMAX | MG_FLAG_QK_NORM))
            p->ws_m = p->ws_l + rows;
    }
    if (info.n_split > 1 && info.cluster_ctas == 0) {
        // ws_o as (n_split*B, M, d) fp32, stored in {32, 128} boxes by the TMA.
        st = encode_3d(&p->maps[4], p->ws_o, d, M, static_cast<uint64_t>(info.n_split) * B, 32u, 128u, 4);
        if (st != MG_OK) {
            cudaFree(p->workspace);
            delete p;
            return st;
        }
    }
    if (flags & MG_FLAG_QK_NORM) {
        const size_t scale_floats = static_cast<size_t>(B) * N + 128;
        const uintptr_t at = reinterpret_cast<uintptr_t>(ws + info.workspace_bytes - scale_floats * 4 - 256);
        p->col_scale = reinterpret_cast<float *>((at + 255) & ~uintptr_t(255));
        e = cudaMemset(p->col_scale, 0, scale_floats * 4);
        if (e != cudaSuccess) {
            cudaFree(p->workspace);
            delete p;
            return cuda_fail(e, "cudaMemset(scales)");
        }
    }
    e = cudaMemset(p->workspace, 0, 256);
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(p->workspace);
        delete p;
        return cuda_fail(e, "cudaMemset(status)");
    }
    *out = p;
    return MG_OK;
}

mg_status mg_attn_plan(int64_t B, int64_t M, int64_t N, int64_t d, mg_attn_plan_t *out)
{
    return mg_attn_plan_ex(B, M, N, d, nullptr, out);
}

mg_status mg_attn_set_timing_events(mg_attn_plan_t plan, void *ev_begin, void *ev_end)
{
    if (!plan || (ev_begin == nullptr) != (ev_end == nullptr))
        return fail(MG_ERR_INVALID_ARG, "NULL plan, or only one of the two events");
    plan->ev_begin = static_cast<cudaEvent_t>(ev_begin);
    plan->ev_end = static_cast<cudaEvent_t>(ev_end);
    return MG_OK;
}

mg_status mg_attn_get_info(mg_attn_plan_t plan, mg_attn_plan_info *info)
{
    if (!plan || !info)
        return fail(MG_ERR_INVALID_ARG, "NULL plan or info");
    *info = plan->info;
    return MG_OK;
}

// The output ranges of the last kWindow calls enqueued on each stream (O as passed to
// mg_attn_run; hO and its device address for mg_attn_run_host). A call's first kernel (the
// host-buffer call's copy kernel, or the fused kernel) may read its inputs before the previous
// grid on its stream has completed. Which earlier kernels can still run then:
// * A kernel that releases its dependents after its own wait (every kernel of this library but
//   the fused kernel started at level 2, and a kernel of another origin, which releases them when
//   it completes unless it triggers early itself) has every kernel before it completed by the
//   time the next one can start.
// * A fused kernel at level 2 releases them at its start. A kernel cannot complete before the one
//   before it, so when kernel i still runs every later kernel does too, all their CTAs resident
//   (none can exit before its wait). Level 2 is used only for grids of at least
//   early_min_ctas(SMs) CTAs of one per SM, so fewer than kWindow such kernels fit the device
//   together.
// So the reads are early only when the previous call on the stream is known and no input shares
// bytes with the outputs of the last kWindow calls or with the call's own output. The first call
// on a stream, or one whose records were displaced by kStreamSlots newer streams, is not known,
// and nor is the first call of a stream capture. Calls enqueued under capture are recorded apart
// from the stream's eager calls, keyed by the capture's id, since the captured kernels run later
// as one graph.
struct OutRanges {
    cudaStream_t stream = nullptr;
    unsigned long long capture = 0;                     // the capture's id, 0 for eager calls
    uintptr_t lo[kWindow][2] = {}, hi[kWindow][2] = {};  // [lo, hi) ranges; empty when lo == hi
    int calls = 0;                                       // calls recorded (the newest at (calls-1) % kWindow)
    unsigned long long age = 0;
    bool used = false;
};
constexpr int kStreamSlots = 64;
std::mutex g_out_mu;
OutRanges g_out[kStreamSlots];
unsigned long long g_out_clock = 0;

// The id of the capture in progress on `stream`, 0 if none; ~0 if the query failed.
unsigned long long capture_of(cudaStream_t stream)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    unsigned long long id = 0;
    if (cudaStreamGetCaptureInfo(stream, &cs, &id) != cudaSuccess) {
        (void)cudaGetLastError();
        return ~0ull;
    }
    return cs == cudaStreamCaptureStatusActive ? id : 0;
}

OutRanges *find_slot(cudaStream_t stream, unsigned long long capture, bool claim)
{
    OutRanges *oldest = &g_out[0];
    for (auto &r : g_out) {
        if (r.used && r.stream == stream && r.capture == capture)
            return &r;
        if (!r.used || (oldest->used && r.age < oldest->age))
            oldest = &r;
    }
    if (claim) {
        *oldest = OutRanges{};
        return oldest;
    }
    return nullptr;
}

// The output ranges of the recent calls enqueued on `stream` under the same capture (or none);
// `used` is false when the previous call is unknown.
OutRanges recent_outputs(cudaStream_t stream)
{
    const unsigned long long capture = capture_of(stream);
    if (capture == ~0ull)
        return OutRanges{};
    std::lock_guard<std::mutex> lock(g_out_mu);
    const OutRanges *r = find_slot(stream, capture, false);
    return r ? *r : OutRanges{};
}

// Records the output ranges of the call just enqueued on `stream`.
void record_outputs(cudaStream_t stream, const void *a, size_t na, const void *b, size_t nb)
{
    const unsigned long long capture = capture_of(stream);
    std::lock_guard<std::mutex> lock(g_out_mu);
    OutRanges *slot = find_slot(stream, capture, true);
    slot->used = true;
    slot->stream = stream;
    slot->capture = capture;
    slot->age = ++g_out_clock;
    const int k = slot->calls % kWindow;
    slot->lo[k][0] = reinterpret_cast<uintptr_t>(a);
    slot->hi[k][0] = slot->lo[k][0] + (a ? na : 0);
    slot->lo[k][1] = reinterpret_cast<uintptr_t>(b);
    slot->hi[k][1] = slot->lo[k][1] + (b ? nb : 0);
    ++slot->calls;
}

bool overlaps_range(const void *p, size_t n, uintptr_t lo, uintptr_t hi)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(p);
    return lo < hi && x < hi && lo < x + n;
}

// Whether a call's first kernel may read its inputs before the previous grid on `stream` has
// completed: the previous call is known and no input (n[i] bytes at p[i], host or device address)
// shares bytes with the outputs of the last kWindow calls or with this call's own output
// [o, o + no).
bool may_load_early(cudaStream_t stream, const void *const *p, const size_t *n, int count, const void *o, size_t no)
{
    const OutRanges prev = recent_outputs(stream);
    if (!prev.used || prev.calls == 0)
        return false;
    const uintptr_t ol = reinterpret_cast<uintptr_t>(o);
    const int recorded = prev.calls < kWindow ? prev.calls : kWindow;
    for (int i = 0; i < count; ++i) {
        if (!p[i])
            continue;
        if (overlaps_range(p[i], n[i], ol, ol + no))
            return false;
        for (int k = 0; k < recorded; ++k)
            for (int r = 0; r < 2; ++r)
                if (overlaps_range(p[i], n[i], prev.lo[k][r], prev.hi[k][r]))
                    return false;
    }
    return true;
}

// How much of the fused kernel may run before the previous grid on the stream completes
// (FwdParams::early): 1, its first copies, where may_load_early allows; 2, everything but its
// global writes, with its dependents released at its start, for the one-tile and few-row kernels
// under the split schedule with grids of at least early_min_ctas CTAs, but not the one-tile
// kernel's QK-norm (its key scales go through global memory). Measured on GB300 (us per call,
// back to back): level 1 against 0, gqa 6.17 against 6.50, tiny 4.56 against 5.44, gqa_b8 9.86
// against 10.03, long_kv 14.52 against 14.82, decode 46.0 against 46.7, decode_m1 24.6 against
// 25.0; level 2, gqa 3.59 against 5.81 (two calls' clusters resident together, their work
// overlapping), tiny 1.66 against 4.47, (1, 256, 4096, 64) 2.15 against 5.61.
int early_level(const mg_attn_plan_info &in, int flags, cudaStream_t stream, const void *Q, const void *K,
                const void *V, const void *O)
{
    if (in.q_tiles_per_cta != 1)
        return 0;
    const size_t bq = static_cast<size_t>(in.B * in.M * in.d) * 2, bk = static_cast<size_t>(in.B * in.d * in.N) * 2;
    const void *inp[3] = {Q, K, V};
    const size_t nb[3] = {bq, bk, bk};
    if (!may_load_early(stream, inp, nb, 3, O, bq))
        return 0;
    const bool qk_global = (flags & MG_FLAG_QK_NORM) && in.swap_ab == 0 && qk_cs_tiles(in, flags) == 0;
    return in.schedule == 0 && !qk_global && in.grid_ctas >= early_min_ctas(in.num_sms) ? 2 : 1;
}

// mg_attn_run's work; `allow_early`: the fused kernel may load Q, K and V before the previous
// grid on the stream completes, where may_load_early allows it (the host-buffer entry point's
// staged inputs are written by the copy kernel just before: never).
static mg_status run_fused(mg_attn_plan_t plan, const void *Q, const void *K, const void *V, void *O,
                           mg_stream_t stream, bool allow_early)
{
    if (!plan || !Q || !K || !V || !O)
        return fail(MG_ERR_INVALID_ARG, "NULL plan or tensor pointer");
    if (misaligned(Q) || misaligned(K) || misaligned(V) || misaligned(O))
        return fail(MG_ERR_LAYOUT, "Q, K, V and O must be 16-byte aligned");
    const mg_attn_plan_info &in = plan->info;
    const uint64_t B = in.B, M = in.M, N = in.N, d = in.d;

    // Q (B, M, d): box 64 x 128 rows; K (B, d, N): box 64 columns x d rows; V (B, N, d): box 64 x 128
    // rows; O (B, M, d): box 64 x 128 rows.
    const void *ptrs[4] = {Q, K, V, O};
    const uint64_t dims[4][3] = {{d, M, B}, {N, d, B}, {d, N, B}, {d, M, B}};
    // Under the stream-K schedule the Q box is kSkQRows rows high (a compact tile per segment).
    const uint32_t qrows = in.schedule == 1 || in.swap_ab == 1 ? static_cast<uint32_t>(mg::kSkQRows) : 128u;
    const uint32_t box1[4] = {qrows, static_cast<uint32_t>(d), 128u, 128u};
    for (int i = 0; i < 4; ++i) {
        if (plan->map_ptr[i] != ptrs[i]) {
            plan->map_ptr[i] = nullptr;
            mg_status st = encode_3d(&plan->maps[i], ptrs[i], dims[i][0], dims[i][1], dims[i][2], 64u, box1[i]);
            if (st != MG_OK)
                return st;
            plan->map_ptr[i] = ptrs[i];
        }
    }

    mg::FwdParams prm;
    prm.B = static_cast<int>(B);
    prm.M = static_cast<int>(M);
    prm.N = static_cast<int>(N);
    prm.m_tiles_per_b = static_cast<int>((M + mg::kBlockM - 1) / mg::kBlockM);
    prm.n_tiles = in.n_tiles;
    prm.n_split = in.n_split;
    prm.cluster_reduce = in.cluster_ctas > 0 ? 1 : 0;
    prm.O = static_cast<__half *>(O);
    prm.ws_o = plan->ws_o;
    prm.ws_l = plan->ws_l;
    prm.ws_m = plan->ws_m;
    prm.col_scale = plan->col_scale;
    prm.status = plan->status;
    prm.timeout_ns = plan->timeout_ns;
    prm.inject_timeout = (plan->flags & MG_FLAG_INJECT_TIMEOUT) ? 1 : 0;
    prm.sk_units = static_cast<long long>(in.m_tiles) * in.n_tiles;
    prm.sk_ctas = in.grid_ctas;
    prm.sk_slots = in.n_split;

    cudaLaunchAttribute attr[2];
    const bool pdl = (plan->flags & MG_FLAG_NO_PDL) == 0;
    prm.cs_tiles = qk_cs_tiles(in, plan->flags);
    prm.early = allow_early && pdl && !(plan->flags & MG_FLAG_NO_EARLY_LOADS)
                    ? early_level(in, plan->flags, reinterpret_cast<cudaStream_t>(stream), Q, K, V, O)
                    : 0;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(in.grid_ctas), 1, 1);
    cfg.blockDim = dim3(mg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(in.smem_bytes);
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(fused_launch_attrs(attr, pdl, in.cluster_ctas));
    void *fwd_args[6] = {&plan->maps[0], &plan->maps[1], &plan->maps[2], &plan->maps[3], &plan->maps[4], &prm};
    cudaError_t e;
    if (plan->ev_begin && (e = cudaEventRecord(plan->ev_begin, cfg.stream)) != cudaSuccess)
        return cuda_fail(e, "cudaEventRecord(begin)");
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(plan->fwd), fwd_args);
    if (e != cudaSuccess)
        return cuda_fail(e, "launch mg_attn_fwd_partial");
    if (plan->ev_end && (e = cudaEventRecord(plan->ev_end, cfg.stream)) != cudaSuccess)
        return cuda_fail(e, "cudaEventRecord(end)");

    if (in.n_split > 1 && in.cluster_ctas == 0) {
        int rows = static_cast<int>(B * M);
        int n_split = in.n_split;
        const float *wo = plan->ws_o;
        const float *wl = plan->ws_l;
        const float *wm = plan->ws_m;
        __half *out = static_cast<__half *>(O);
        const int rows_per_cta = d == 64 ? combine_rows_per_cta<64>(n_split) : combine_rows_per_cta<128>(n_split);
        cudaLaunchConfig_t cc = cfg;
        cc.gridDim = dim3(static_cast<unsigned>((rows + rows_per_cta - 1) / rows_per_cta), 1, 1);
        cc.blockDim = dim3(256, 1, 1);
        cc.dynamicSmemBytes = 0;
        cc.numAttrs = static_cast<unsigned>(fused_launch_attrs(attr, pdl, 0));
        int early = prm.early == 2 ? 1 : 0;
        void *cargs[7] = {&wo, &wl, &wm, &out, &rows, &n_split, &early};
        e = cudaLaunchKernelExC(&cc, reinterpret_cast<const void *>(plan->combine), cargs);
        if (e != cudaSuccess)
            return cuda_fail(e, "launch mg_attn_combine");
    }
    record_outputs(cfg.stream, O, static_cast<size_t>(B * M * d) * 2, nullptr, 0);
    return MG_OK;
}

mg_status mg_attn_run(mg_attn_plan_t plan, const void *Q, const void *K, const void *V, void *O,
                      mg_stream_t stream)
{
    return run_fused(plan, Q, K, V, O, stream, true);
}

mg_status mg_attn_run_host(mg_attn_plan_t plan, const void *hQ, const void *hK, const void *hV, void *hO,
                           mg_stream_t stream)
{
    if (!plan || !hQ || !hK || !hV || !hO)
        return fail(MG_ERR_INVALID_ARG, "NULL plan or host pointer");
    const mg_attn_plan_info &in = plan->info;
    const size_t bq = static_cast<size_t>(in.B * in.M * in.d) * 2;
    const size_t bk = static_cast<size_t>(in.B * in.d * in.N) * 2;
    const size_t bv = bk;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t oq = 0, ok = up(bq), ov = ok + up(bk), oo = ov + up(bv), total = oo + up(bq);
    cudaError_t e;
    if (!plan->staging) {
        e = cudaMalloc(&plan->staging, total);
        if (e != cudaSuccess) {
            plan->staging = nullptr;
            return cuda_fail(e, "cudaMalloc(staging)");
        }
    }
    uint8_t *s = static_cast<uint8_t *>(plan->staging);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    // Pinned (page-locked, device-mapped) 16-byte-aligned host buffers are read by a copy kernel
    // through their device addresses, chained to the attention kernels with PDL, and O is written
    // back the same way (or directly, below); any other host memory goes through the copy engines.
    void *dQ = nullptr, *dK = nullptr, *dV = nullptr, *dO = nullptr;
    bool direct = device_mapped(hQ, &dQ) && device_mapped(hK, &dK) && device_mapped(hV, &dV) && device_mapped(hO, &dO);
    const bool pdl = (plan->flags & MG_FLAG_NO_PDL) == 0;
    if (direct) {
        CopyJobs in_jobs{};
        const void *src[3] = {dQ, dK, dV};
        const size_t off[3] = {oq, ok, ov};
        const size_t bytes[3] = {bq, bk, bv};
        for (int i = 0; i < 3; ++i) {
            in_jobs.src[i] = static_cast<const uint4 *>(src[i]);
            in_jobs.dst[i] = reinterpret_cast<uint4 *>(s + off[i]);
            in_jobs.units[i] = bytes[i] / 16;
        }
        // The inputs are loaded as soon as the copy kernel starts, possibly while the previous
        // kernel on this stream still runs (only that one: each of this library's kernels releases
        // its dependents after its own wait). So the loads wait as well when an input shares bytes
        // with what that kernel may still be writing: the previous call's output on this stream
        // (a chain of calls), or this call's own output (which a call before it on this plan may
        // be writing). Measured on GB300 (GQA graph, back-to-back calls): 13.5 us per call, against
        // 19.3 with every load after the wait (the link's transfer then overlaps the previous
        // call's attention kernel).
        const void *inp[6] = {hQ, hK, hV, dQ, dK, dV};
        const size_t nb[6] = {bq, bk, bv, bq, bk, bv};
        in_jobs.early = may_load_early(st, inp, nb, 6, hO, bq) ? 1 : 0;
        if ((e = launch_copy(in_jobs, plan->info.num_sms, pdl, st)) != cudaSuccess)
            return cuda_fail(e, "launch mg_copy_units (host to device)");
    } else if ((e = cudaMemcpyAsync(s + oq, hQ, bq, cudaMemcpyHostToDevice, st)) != cudaSuccess ||
               (e = cudaMemcpyAsync(s + ok, hK, bk, cudaMemcpyHostToDevice, st)) != cudaSuccess ||
               (e = cudaMemcpyAsync(s + ov, hV, bv, cudaMemcpyHostToDevice, st)) != cudaSuccess) {
        return cuda_fail(e, "cudaMemcpyAsync(host to device)");
    }
    // With split partials (the on-chip combine or the second kernel) O is written by plain stores,
    // which reach the pinned host buffer through its device address directly: no staging of O
    // and no copy back. One split writes O with a TMA store, which takes the staging path.
    const bool o_direct = direct && in.n_split > 1;
    mg_status r = run_fused(plan, s + oq, s + ok, s + ov, o_direct ? dO : s + oo, stream, false);
    if (r != MG_OK)
        return r;
    if (!o_direct) {
        if (direct) {
            CopyJobs out_jobs{};
            out_jobs.src[0] = reinterpret_cast<const uint4 *>(s + oo);
            out_jobs.dst[0] = static_cast<uint4 *>(dO);
            out_jobs.units[0] = bq / 16;
            if ((e = launch_copy(out_jobs, plan->info.num_sms, pdl, st)) != cudaSuccess)
                return cuda_fail(e, "launch mg_copy_units (device to host)");
        } else if ((e = cudaMemcpyAsync(hO, s + oo, bq, cudaMemcpyDeviceToHost, st)) != cudaSuccess) {
            return cuda_fail(e, "cudaMemcpyAsync(device to host)");
        }
    }
    // What the next call on this stream must not load early: hO, by its host and device addresses.
    record_outputs(st, hO, bq, direct ? dO : nullptr, bq);
    return MG_OK;
}

// ------------------------------------------------------------------ allocation-free entry point
}  // extern "C"

namespace {

// Scratch of mg_attn_run_noalloc: 256 bytes of status words, then the fp32 split partials
// (numerators, then row sums). A file-scope device array: no allocation call ever creates it.
__device__ __align__(256) unsigned char g_static_scratch[MG_ATTN_STATIC_SCRATCH_BYTES];

struct StaticDevice {
    bool ready = false;
    unsigned char *scratch = nullptr;  // device address of g_static_scratch on this device
    int sms = 0, smem_optin = 0;
};

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
StaticDevice g_static_dev[kMaxDevices];

// One-time, per-device set-up with that device current: check the device, look up the array's
// device address (its host-side name is only a stand-in) and clear the status words.
mg_status static_setup(StaticDevice **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(MG_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_static_mu);
    StaticDevice &sd = g_static_dev[dev];
    if (!sd.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sd.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sd.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
                cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (major != 10 || minor != 3)
            return fail(MG_ERR_UNSUPPORTED, "device %d has compute capability %d.%d; this library is built for 10.3",
                        dev, major, minor);
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        e = cudaMemset(ptr, 0, 256);
        if (e == cudaSuccess)
            e = cudaDeviceSynchronize();
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMemset(static scratch status)");
        sd.scratch = static_cast<unsigned char *>(ptr);
        sd.ready = true;
    }
    *out = &sd;
    return MG_OK;
}

}  // namespace

extern "C" {

mg_status mg_attn_run_noalloc(int64_t B, int64_t M, int64_t N, int64_t d, const void *Q, const void *K,
                              const void *V, void *O, mg_stream_t stream)
{
    if (!Q || !K || !V || !O)
        return fail(MG_ERR_INVALID_ARG, "NULL tensor pointer");
    if (misaligned(Q) || misaligned(K) || misaligned(V) || misaligned(O))
        return fail(MG_ERR_LAYOUT, "Q, K, V and O must be 16-byte aligned");
    StaticDevice *sd = nullptr;
    mg_status st = static_setup(&sd);
    if (st != MG_OK)
        return st;
    mg_attn_plan_info in;
    unsigned long long timeout_ns = 0;
    int flags = 0;
    st = decide(B, M, N, d, nullptr, sd->sms, sd->smem_optin, &in, &timeout_ns, &flags);
    if (st != MG_OK)
        return st;
    // The kernel's shared-memory limit is raised before the cluster occupancy query, as
    // mg_attn_plan_ex does: at the default 48 KB limit the query would refuse the cluster, and a
    // first call in a process would then take another combine than later calls.
    FwdKernel fwd = plan_kernel(in, 0);
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fwd),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, in.smem_bytes);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute");
    if ((st = place_clusters(B, M, N, d, nullptr, sd->sms, sd->smem_optin, &in, &timeout_ns, &flags, &fwd)) != MG_OK)
        return st;
    if (in.workspace_bytes > static_cast<int64_t>(MG_ATTN_STATIC_SCRATCH_BYTES))
        return fail(MG_ERR_INVALID_ARG,
                    "shape needs %lld bytes of split scratch; the static scratch holds %u bytes "
                    "(use mg_attn_plan / mg_attn_run)",
                    (long long)in.workspace_bytes, MG_ATTN_STATIC_SCRATCH_BYTES);

    CUtensorMap maps[5];
    std::memset(maps, 0, sizeof(maps));
    const void *ptrs[4] = {Q, K, V, O};
    const uint64_t uB = B, uM = M, uN = N, ud = d;
    const uint64_t dims[4][3] = {{ud, uM, uB}, {uN, ud, uB}, {ud, uN, uB}, {ud, uM, uB}};
    const uint32_t qrows = in.schedule == 1 || in.swap_ab == 1 ? static_cast<uint32_t>(mg::kSkQRows) : 128u;
    const uint32_t box1[4] = {qrows, static_cast<uint32_t>(d), 128u, 128u};
    for (int i = 0; i < 4; ++i)
        if ((st = encode_3d(&maps[i], ptrs[i], dims[i][0], dims[i][1], dims[i][2], 64u, box1[i])) != MG_OK)
            return st;
    const bool l2_cluster = in.cluster_ctas > 0 && in.q_tiles_per_cta == 2;
    float *ws_o =
        in.n_split > 1 && (in.cluster_ctas == 0 || l2_cluster) ? reinterpret_cast<float *>(sd->scratch + 256) : nullptr;
    if (ws_o && in.cluster_ctas == 0 &&
        (st = encode_3d(&maps[4], ws_o, ud, uM, static_cast<uint64_t>(in.n_split) * uB, 32u, 128u, 4)) != MG_OK)
        return st;

    mg::FwdParams prm;
    prm.B = static_cast<int>(B);
    prm.M = static_cast<int>(M);
    prm.N = static_cast<int>(N);
    prm.m_tiles_per_b = static_cast<int>((M + mg::kBlockM - 1) / mg::kBlockM);
    prm.n_tiles = in.n_tiles;
    prm.n_split = in.n_split;
    prm.cluster_reduce = in.cluster_ctas > 0 ? 1 : 0;
    prm.O = static_cast<__half *>(O);
    prm.status = reinterpret_cast<int *>(sd->scratch);
    prm.ws_o = ws_o;
    prm.ws_l = ws_o ? ws_o + static_cast<size_t>(in.n_split) * partial_rows(B, M, l2_cluster) * d : nullptr;
    prm.ws_m = nullptr;
    prm.col_scale = nullptr;
    prm.timeout_ns = timeout_ns;
    prm.inject_timeout = 0;
    prm.cs_tiles = qk_cs_tiles(in, flags);
    prm.early = early_level(in, flags, reinterpret_cast<cudaStream_t>(stream), Q, K, V, O);
    prm.sk_units = static_cast<long long>(in.m_tiles) * in.n_tiles;
    prm.sk_ctas = in.grid_ctas;
    prm.sk_slots = in.n_split;

    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(in.grid_ctas), 1, 1);
    cfg.blockDim = dim3(mg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(in.smem_bytes);
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(fused_launch_attrs(attr, true, in.cluster_ctas));
    void *fwd_args[6] = {&maps[0], &maps[1], &maps[2], &maps[3], &maps[4], &prm};
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(fwd), fwd_args);
    if (e != cudaSuccess)
        return cuda_fail(e, "launch mg_attn_fwd_partial");
    if (in.n_split > 1 && in.cluster_ctas == 0) {
        int rows = static_cast<int>(B * M);
        int n_split = in.n_split;
        const float *wo = ws_o;
        const float *wl = prm.ws_l;
        __half *out = static_cast<__half *>(O);
        const int rows_per_cta = d == 64 ? combine_rows_per_cta<64>(n_split) : combine_rows_per_cta<128>(n_split);
        cudaLaunchConfig_t cc = cfg;
        cc.gridDim = dim3(static_cast<unsigned>((rows + rows_per_cta - 1) / rows_per_cta), 1, 1);
        cc.blockDim = dim3(256, 1, 1);
        cc.dynamicSmemBytes = 0;
        cc.numAttrs = static_cast<unsigned>(fused_launch_attrs(attr, true, 0));
        const float *wm = nullptr;
        int early = prm.early == 2 ? 1 : 0;
        void *cargs[7] = {&wo, &wl, &wm, &out, &rows, &n_split, &early};
        e = cudaLaunchKernelExC(&cc, reinterpret_cast<const void *>(combine_kernel(d, n_split)), cargs);
        if (e != cudaSuccess)
            return cuda_fail(e, "launch mg_attn_combine");
    }
    record_outputs(cfg.stream, O, static_cast<size_t>(B * M * d) * 2, nullptr, 0);
    return MG_OK;
}

mg_status mg_attn_get_status(mg_attn_plan_t plan)
{
    if (!plan)
        return fail(MG_ERR_INVALID_ARG, "NULL plan");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaDeviceSynchronize");
    int words[2] = {0, 0};
    e = cudaMemcpy(words, plan->status, sizeof(words), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy(status)");
    if (words[0] == MG_ERR_TIMEOUT)
        return fail(MG_ERR_TIMEOUT, "in-kernel wait on barrier %d ran out", words[1]);
    if (words[0] != 0)
        return fail(MG_ERR_CUDA, "unexpected device status %d", words[0]);
    return MG_OK;
}

mg_status mg_attn_destroy(mg_attn_plan_t plan)
{
    if (!plan)
        return fail(MG_ERR_INVALID_ARG, "NULL plan");
    cudaError_t e = cudaDeviceSynchronize();
    cudaFree(plan->workspace);
    if (plan->staging)
        cudaFree(plan->staging);
    delete plan;
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaDeviceSynchronize");
    return MG_OK;
}

}  // extern "C"
