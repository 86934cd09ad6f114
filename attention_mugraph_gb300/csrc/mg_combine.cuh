// mg_combine.cuh -- kernel 2 of the exp-normalised GQA graph: the combine of split partials.
//
// Graph (Mirage documentation, tutorials/group-query-attention, "Define GQA Computation
// Graph"): A = matmul(Q,K); E = exp(A); S = reduction(E,2); D = div(E,S); O = matmul(D,V).
// When kernel 1 (mg_attn_fwd_partial) splits the N axis over more CTAs than a thread-block
// cluster combines on chip, each split j leaves its fp32 partial numerator O_j and row sum l_j
// (and, max-subtracted, its row maximum m_j) in the workspace, and this kernel forms
// O = (sum_j w_j O_j) / (sum_j w_j l_j) -> fp16, the second threadblock graph of the
// "attention" search configuration (blog "Reading Mirage's muGraph search and backend
// generation through the GQA example", section 4.3). Without max-subtraction every w_j = 1;
// with it, w_j = exp(m_j - max_j m_j).
#pragma once

#include <cmath>
#include <cstdint>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace mg {

// O[r, c] = (sum_j ws_o[j, r, c]) / (sum_j ws_l[j, r]) -> fp16, r = b*M + m, for up to
// kMaxSplits splits (mg_attn_combine_wide takes more). A CTA of 256 threads covers kRows rows. Thread (row, part, g) sums float4 column group g of its
// row over the splits j = part, part + kParts, ... (independent loads, all in flight together);
// the kParts partial sums then meet in shared memory in a fixed order, so the result is
// reproducible run to run.
template <int D>
struct CombineCfg {
    static constexpr int kGroups = D / 4;                  // float4 groups per row
    static constexpr int kParts = 4;                       // split-index residues per row
    static constexpr int kRows = 256 / (kGroups * kParts); // rows per CTA: 4 (d=64) or 2 (d=128)
    static constexpr int kMaxSplits = 16;                  // at most 4 partials per thread
};

template <int D>
__global__ void __launch_bounds__(256)
    mg_attn_combine(const float *__restrict__ ws_o, const float *__restrict__ ws_l, const float *__restrict__ ws_m,
                    __half *__restrict__ O, int rows, int n_split, int early)
{
    using CC = CombineCfg<D>;
    __shared__ float4 part_o[CC::kParts][CC::kRows][CC::kGroups];
    __shared__ float part_l[CC::kParts][CC::kRows];

    // Everything here waits for the fused kernel. early: that kernel started early (its
    // dependents released at its start), so this one releases the next call's fused kernel
    // before its wait too, and the next call overlaps this call's end.
    if (early) {
        ptx::griddep_launch_dependents();
        ptx::griddep_wait();
    } else {
        ptx::griddep_wait();
        ptx::griddep_launch_dependents();
    }

    const int g = threadIdx.x % CC::kGroups;
    const int part = (threadIdx.x / CC::kGroups) % CC::kParts;
    const int rl = threadIdx.x / (CC::kGroups * CC::kParts);
    const int r = blockIdx.x * CC::kRows + rl;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float l = 0.f;
    if (r < rows) {
        // Max-subtracted variant (ws_m given): split j's partial is relative to its row maximum
        // m_j and enters with weight exp(m_j - max_j m_j); otherwise every weight is 1.
        float mmax = 0.f;
        if (ws_m) {
            mmax = -INFINITY;
            for (int j = 0; j < n_split; ++j)
                mmax = fmaxf(mmax, ws_m[static_cast<size_t>(j) * rows + r]);
        }
        const float4 *src = reinterpret_cast<const float4 *>(ws_o) + static_cast<size_t>(r) * CC::kGroups + g;
        const size_t split_stride = static_cast<size_t>(rows) * CC::kGroups;
#pragma unroll 4
        for (int j = part; j < n_split; j += CC::kParts) {
            const float4 a = src[static_cast<size_t>(j) * split_stride];
            const float wt = ws_m ? ptx::ex2_approx((ws_m[static_cast<size_t>(j) * rows + r] - mmax) * ptx::kLog2e)
                                  : 1.f;
            acc.x += wt * a.x;
            acc.y += wt * a.y;
            acc.z += wt * a.z;
            acc.w += wt * a.w;
            if (g == 0)
                l += wt * ws_l[static_cast<size_t>(j) * rows + r];
        }
    }
    part_o[part][rl][g] = acc;
    if (g == 0)
        part_l[part][rl] = l;
    __syncthreads();
    if (part == 0 && r < rows) {
        float4 s = part_o[0][rl][g];
        float ls = part_l[0][rl];
#pragma unroll
        for (int q = 1; q < CC::kParts; ++q) {
            const float4 t = part_o[q][rl][g];
            s.x += t.x;
            s.y += t.y;
            s.z += t.z;
            s.w += t.w;
            ls += part_l[q][rl];
        }
        const float inv = __frcp_rn(ls);  // one reciprocal, then products
        uint2 w;
        w.x = ptx::pack_half2(s.x * inv, s.y * inv);
        w.y = ptx::pack_half2(s.z * inv, s.w * inv);
        *reinterpret_cast<uint2 *>(O + static_cast<size_t>(r) * D + g * 4) = w;
    }
}

// The same combine for more than CombineCfg::kMaxSplits splits (the long KV axis): eight parts
// per row, and each thread loads BATCH of its splits (4 or 8, WideCombineCfg::batch) before using
// the first, so that a thread's partials cost one round trip to L2 rather than one per four.
// Measured on GB300 for 38 splits of 512 rows: 16.0 against 19.0 us per call for the whole
// path; for 4 to 9 splits the deeper batch only adds registers, and mg_attn_combine stays.
// Max-subtracted variant (ws_m given): a part weights its splits by exp(m_j - mp) with mp the
// largest m_j among them, and the parts meet with weights exp(mp - max mp): in all, exp(m_j - max m).
template <int D>
struct WideCombineCfg {
    static constexpr int kGroups = D / 4;                  // float4 groups per row
    static constexpr int kParts = 8;                       // split-index residues per row
    static constexpr int kRows = 256 / (kGroups * kParts); // rows per CTA: 2 (d=64) or 1 (d=128)
    __host__ __device__ static constexpr int batch(int n_split) { return n_split <= 4 * kParts ? 4 : 8; }
};

template <int D, int BATCH>
__global__ void __launch_bounds__(256, BATCH == 4 ? 4 : 3)
    mg_attn_combine_wide(const float *__restrict__ ws_o, const float *__restrict__ ws_l,
                         const float *__restrict__ ws_m, __half *__restrict__ O, int rows, int n_split,
                         int early)
{
    using CC = WideCombineCfg<D>;
    __shared__ float4 part_o[CC::kParts][CC::kRows][CC::kGroups];
    __shared__ float part_l[CC::kParts][CC::kRows];
    __shared__ float part_m[CC::kParts][CC::kRows];

    // Everything here waits for the fused kernel. early: that kernel started early (its
    // dependents released at its start), so this one releases the next call's fused kernel
    // before its wait too, and the next call overlaps this call's end.
    if (early) {
        ptx::griddep_launch_dependents();
        ptx::griddep_wait();
    } else {
        ptx::griddep_wait();
        ptx::griddep_launch_dependents();
    }

    const int g = threadIdx.x % CC::kGroups;
    const int part = (threadIdx.x / CC::kGroups) % CC::kParts;
    const int rl = threadIdx.x / (CC::kGroups * CC::kParts);
    const int r = blockIdx.x * CC::kRows + rl;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float l = 0.f;
    float mp = ws_m ? -INFINITY : 0.f;
    if (r < rows) {
        if (ws_m) {
            for (int j = part; j < n_split; j += CC::kParts)
                mp = fmaxf(mp, ws_m[static_cast<size_t>(j) * rows + r]);
        }
        const float4 *src = reinterpret_cast<const float4 *>(ws_o) + static_cast<size_t>(r) * CC::kGroups + g;
        const size_t split_stride = static_cast<size_t>(rows) * CC::kGroups;
        for (int j0 = part; j0 < n_split; j0 += CC::kParts * BATCH) {
            float4 a[BATCH];
            float lw[BATCH], mw[BATCH];
#pragma unroll
            for (int q = 0; q < BATCH; ++q) {
                const int j = j0 + q * CC::kParts;
                if (j < n_split) {
                    a[q] = src[static_cast<size_t>(j) * split_stride];
                    lw[q] = g == 0 ? ws_l[static_cast<size_t>(j) * rows + r] : 0.f;
                    mw[q] = ws_m ? ws_m[static_cast<size_t>(j) * rows + r] : 0.f;
                }
            }
#pragma unroll
            for (int q = 0; q < BATCH; ++q) {
                if (j0 + q * CC::kParts < n_split) {
                    const float wt = ws_m ? ptx::ex2_approx((mw[q] - mp) * ptx::kLog2e) : 1.f;
                    acc.x += wt * a[q].x;
                    acc.y += wt * a[q].y;
                    acc.z += wt * a[q].z;
                    acc.w += wt * a[q].w;
                    l += wt * lw[q];
                }
            }
        }
    }
    part_o[part][rl][g] = acc;
    if (g == 0) {
        part_l[part][rl] = l;
        part_m[part][rl] = mp;
    }
    __syncthreads();
    if (part == 0 && r < rows) {
        float mmax = 0.f;
        if (ws_m) {
            mmax = -INFINITY;
#pragma unroll
            for (int q = 0; q < CC::kParts; ++q)
                mmax = fmaxf(mmax, part_m[q][rl]);
        }
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        float ls = 0.f;
#pragma unroll
        for (int q = 0; q < CC::kParts; ++q) {
            const float wq = ws_m ? ptx::ex2_approx((part_m[q][rl] - mmax) * ptx::kLog2e) : 1.f;
            const float4 t = part_o[q][rl][g];
            s.x += wq * t.x;
            s.y += wq * t.y;
            s.z += wq * t.z;
            s.w += wq * t.w;
            ls += wq * part_l[q][rl];
        }
        const float inv = __frcp_rn(ls);  // one reciprocal, then products
        uint2 w;
        w.x = ptx::pack_half2(s.x * inv, s.y * inv);
        w.y = ptx::pack_half2(s.z * inv, s.w * inv);
        *reinterpret_cast<uint2 *>(O + static_cast<size_t>(r) * D + g * 4) = w;
    }
}

}  // namespace mg
