// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers, TMA tensor copies,
// tcgen05 (tensor-memory allocation, MMA, commit, loads, fences), programmatic dependent
// launch and the global timer. Written from the public PTX ISA; no library headers.
#pragma once

#include <cstdint>
#include <cuda.h>  // CUtensorMap (type only)

namespace mg {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier.init visible to the async proxy (TMA, tcgen05.commit) and other threads.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// True once the phase with the given parity has completed; while it is incomplete the thread may
// be suspended for a hardware-chosen time before the call returns false.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase with the given parity (no suspension, returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// One lane of a converged warp returns true (elect.sync over the full mask).
__device__ __forceinline__ bool elect_one()
{
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, e;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled copy global -> shared; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int32_t c0,
                                            int32_t c1, int32_t c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// 3-D tiled copy shared -> global (rows past the tensor's extent are not written), tracked by
// the issuing thread's bulk-async group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int32_t c0, int32_t c1, int32_t c2)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until every committed bulk store of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Named barrier over `count` threads (a multiple of 32), id 1..15 (0 is __syncthreads).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ANDs a predicate over its participants: every thread gets the same
// answer, so a decision taken after it is uniform across them.
__device__ __forceinline__ bool named_barrier_and(uint32_t id, uint32_t count, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Named barrier that also ORs a predicate over its participants (the same answer on every thread).
__device__ __forceinline__ bool named_barrier_or(uint32_t id, uint32_t count, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy reads
// (the tensor core reading an operand that threads wrote with st.shared).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float4 ld_shared_v4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// ------------------------------------------------------------------ thread-block clusters

// Cluster-wide barrier (every thread of every CTA of the cluster, warps converged). The
// release/acquire pair orders each CTA's shared-memory writes before the others' reads of them.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Cluster-wide barrier without release semantics: it says only that every thread of the cluster
// has got here. A CTA's earlier loads from other CTAs' shared memory have returned by then (their
// values were used), and its global stores need not drain first, which a release would make it
// wait for.
__device__ __forceinline__ void cluster_sync_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}

// The two halves of a cluster-wide barrier, for an arrival made long before the wait (every
// thread of every CTA, warps converged, arrive and wait alternating). The release orders this
// thread's earlier writes (and, after fence_mbar_init, the CTA's barrier initialisations) before
// whatever the other CTAs do once their wait returns.
__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// One arrival, with `bytes` more expected, on an mbarrier in the shared memory of a CTA of this
// cluster (a shared::cluster address from map_to_rank).
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t cluster_bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_bar),
                 "r"(bytes)
                 : "memory");
}

// Asynchronous stores into the shared memory of a CTA of this cluster (shared::cluster addresses
// from map_to_rank), each counting its bytes on that CTA's mbarrier `cluster_bar` when it lands.
// The data leaves from registers: nothing of the sender's has to stay alive for it.
__device__ __forceinline__ void st_async_v4(uint32_t dst_cluster, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t cluster_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     dst_cluster),
                 "r"(a), "r"(b), "r"(c), "r"(d), "r"(cluster_bar)
                 : "memory");
}

__device__ __forceinline__ void st_async_b32(uint32_t dst_cluster, uint32_t v, uint32_t cluster_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(dst_cluster), "r"(v),
                 "r"(cluster_bar)
                 : "memory");
}

// The shared::cluster address of the same shared-memory location in the cluster's CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank)
{
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
    return d;
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// ------------------------------------------------------------------ tcgen05

// Whole warp: allocate `ncols` tensor-memory columns; the base address is written to
// shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], fp16 inputs, fp32 accumulate (kind::f16).
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc], fp16 inputs, fp32 accumulate (kind::f16). A is M x K with
// row i in tensor-memory lane i and two consecutive K elements per 32-bit column.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Warp-collective: lane i reads tensor-memory lane (taddr.lane + i), 32 consecutive 32-bit
// columns starting at taddr.col. Values are valid only after tmem_ld_wait().
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// As tmem_ld_32x32b_x32 for 16 consecutive columns.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait16(uint32_t (&r)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        asm volatile("" : "+r"(r[i]));
}

// Waits for this thread's outstanding tcgen05.ld and pins the registers after the wait, so
// the compiler cannot hoist their uses above it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        asm volatile("" : "+r"(r[i]));
}

// Warp-collective: lane i writes tensor-memory lane (taddr.lane + i), 32 consecutive 32-bit
// columns starting at taddr.col. Complete (and the registers reusable) after tmem_st_wait().
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ descriptors

// tcgen05 shared-memory matrix descriptor for a 128-byte-swizzled operand tile:
// start address (>>4) in bits 0-13, leading byte offset (>>4) in 16-29, stride byte offset
// (>>4) in 32-45, descriptor version 1 in bits 46-47, base offset 0 (tiles are 1024-byte
// aligned), swizzle mode 2 (128B) in bits 61-63.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor for kind::f16 with fp16 A and B and an fp32 accumulator:
// D format bits 4-5 (1 = f32), A/B formats bits 7-9 / 10-12 (0 = f16), A/B major bits 15/16
// (0 = K-major, 1 = MN-major), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n, bool a_mn_major, bool b_mn_major)
{
    return (1u << 4) | (0u << 7) | (0u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// ------------------------------------------------------------------ math / packing

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Degree-5 polynomial for 2^f on f in [-1/2, 1/2], coefficients chosen to minimise the maximum
// relative error (Remez exchange, csrc/exp2_poly_fit.py), highest degree first. Evaluated in
// fp32 with fused multiply-adds after the range reduction below, its relative error is <= 2.2e-7.
constexpr float kExp2C5 = 0x1.5c08e6p-10f;
constexpr float kExp2C4 = 0x1.3d0c52p-7f;
constexpr float kExp2C3 = 0x1.c6b6e4p-5f;
constexpr float kExp2C2 = 0x1.ebf918p-3f;
constexpr float kExp2C1 = 0x1.62e428p-1f;
constexpr float kExp2C0 = 0x1.000002p+0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kShifter = 12582912.0f;  // 1.5 * 2^23: x + shifter rounds x to an integer in the low bits

// 2^x on the FMA pipe, for offloading part of the exponentials from the MUFU unit.
// Range reduction x = r + f with r = round-to-nearest(x), taken with the shifter (exact for
// |x| < 2^22), and f in [-1/2, 1/2]; 2^f by the polynomial above; r is added to the exponent
// field. Inputs below -125 are clamped (a result near 2^-125, negligible next to any row sum).
__device__ __forceinline__ float exp2_fma(float x)
{
    x = fmaxf(x, -125.0f);
    const float t = x + kShifter;
    const float r = t - kShifter;
    const float f = x - r;
    float p = kExp2C5;
    p = fmaf(p, f, kExp2C4);
    p = fmaf(p, f, kExp2C3);
    p = fmaf(p, f, kExp2C2);
    p = fmaf(p, f, kExp2C1);
    p = fmaf(p, f, kExp2C0);
    return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

// exp(s) on the FMA pipe: exp2_fma with the log2(e) scale folded into the range reduction
// (t = s*log2e + shifter and f = s*log2e - r each take one fused multiply-add).
__device__ __forceinline__ float exp_fma(float s)
{
    s = fmaxf(s, -86.0f);  // s*log2e >= -124.07: the result stays a normal float
    const float t = fmaf(s, kLog2e, kShifter);
    const float r = t - kShifter;
    const float f = fmaf(s, kLog2e, -r);
    float p = kExp2C5;
    p = fmaf(p, f, kExp2C4);
    p = fmaf(p, f, kExp2C3);
    p = fmaf(p, f, kExp2C2);
    p = fmaf(p, f, kExp2C1);
    p = fmaf(p, f, kExp2C0);
    return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

// ------------------------------------------------------------------ packed pairs (f32x2)
// Blackwell's two-wide fp32 instructions process a pair of values per thread per instruction,
// halving the FMA-pipe issue cost of the exponentials.

__host__ __device__ constexpr uint64_t pair_of(uint32_t bits) { return (static_cast<uint64_t>(bits) << 32) | bits; }

// The constants of exp_fma, each duplicated into both halves of a 64-bit register.
struct ExpPairConsts {
    uint64_t log2e, shifter, c5, c4, c3, c2, c1, c0;
};

__device__ __forceinline__ ExpPairConsts exp_pair_consts()
{
    return ExpPairConsts{pair_of(__float_as_uint(kLog2e)), pair_of(__float_as_uint(kShifter)),
                         pair_of(__float_as_uint(kExp2C5)), pair_of(__float_as_uint(kExp2C4)),
                         pair_of(__float_as_uint(kExp2C3)), pair_of(__float_as_uint(kExp2C2)),
                         pair_of(__float_as_uint(kExp2C1)), pair_of(__float_as_uint(kExp2C0))};
}

// (exp(s0), exp(s1)) by exp_fma's steps on f32x2 pairs; bit-identical to exp_fma per element.
// The exponent add is one integer multiply-add per element: bits(p) + bits(t) * 2^23.
__device__ __forceinline__ void exp_pair_fma(uint32_t s0, uint32_t s1, const ExpPairConsts &k, uint32_t &e0,
                                             uint32_t &e1)
{
    asm("{\n\t.reg .b64 a, t, nr, f, p;\n\t.reg .f32 a0, a1;\n\t.reg .b32 t0, t1, p0, p1;\n\t"
        "max.f32 a0, %2, 0fC2AC0000;\n\t"  // -86.0
        "max.f32 a1, %3, 0fC2AC0000;\n\t"
        "mov.b64 a, {a0, a1};\n\t"
        "fma.rn.f32x2 t, a, %4, %5;\n\t"     // t = s*log2e + shifter
        "sub.rn.f32x2 nr, %5, t;\n\t"        // -r, exactly
        "fma.rn.f32x2 f, a, %4, nr;\n\t"     // f = s*log2e - r
        "fma.rn.f32x2 p, %6, f, %7;\n\t"
        "fma.rn.f32x2 p, p, f, %8;\n\t"
        "fma.rn.f32x2 p, p, f, %9;\n\t"
        "fma.rn.f32x2 p, p, f, %10;\n\t"
        "fma.rn.f32x2 p, p, f, %11;\n\t"
        "mov.b64 {t0, t1}, t;\n\t"
        "mov.b64 {p0, p1}, p;\n\t"
        "mad.lo.u32 %0, t0, 8388608, p0;\n\t"
        "mad.lo.u32 %1, t1, 8388608, p1;\n\t}"
        : "=r"(e0), "=r"(e1)
        : "f"(__uint_as_float(s0)), "f"(__uint_as_float(s1)), "l"(k.log2e), "l"(k.shifter), "l"(k.c5), "l"(k.c4),
          "l"(k.c3), "l"(k.c2), "l"(k.c1), "l"(k.c0));
}

// (exp(s0 - m), exp(s1 - m)) on the MUFU unit: one packed fused multiply-add s*log2(e) + shift
// with shift = -m*log2(e) in both halves (+0 gives exp(s) exactly as a plain multiply would),
// then ex2.approx each.
__device__ __forceinline__ void exp_pair_mufu(uint32_t s0, uint32_t s1, const ExpPairConsts &k, uint64_t shift,
                                              uint32_t &e0, uint32_t &e1)
{
    asm("{\n\t.reg .b64 a, x;\n\t.reg .f32 x0, x1;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "fma.rn.f32x2 x, a, %4, %5;\n\t"
        "mov.b64 {x0, x1}, x;\n\t"
        "ex2.approx.ftz.f32 x0, x0;\n\t"
        "ex2.approx.ftz.f32 x1, x1;\n\t"
        "mov.b32 %0, x0;\n\t"
        "mov.b32 %1, x1;\n\t}"
        : "=r"(e0), "=r"(e1)
        : "r"(s0), "r"(s1), "l"(k.log2e), "l"(shift));
}

// (exp(s0 c0 a - m), exp(s1 c1 a - m)) on the MUFU unit for scaled scores: one packed multiply
// by the column scales (c0, c1), one packed fused multiply-add by `arow` = a*log2(e) (twice) plus
// `shift` = -m*log2(e) (twice), then ex2.approx each.
__device__ __forceinline__ void exp_pair_mufu_scaled(uint32_t s0, uint32_t s1, float c0, float c1, uint64_t arow,
                                                     uint64_t shift, uint32_t &e0, uint32_t &e1)
{
    asm("{\n\t.reg .b64 a, c, t, x;\n\t.reg .f32 x0, x1;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 c, {%4, %5};\n\t"
        "mul.rn.f32x2 t, a, c;\n\t"
        "fma.rn.f32x2 x, t, %6, %7;\n\t"
        "mov.b64 {x0, x1}, x;\n\t"
        "ex2.approx.ftz.f32 x0, x0;\n\t"
        "ex2.approx.ftz.f32 x1, x1;\n\t"
        "mov.b32 %0, x0;\n\t"
        "mov.b32 %1, x1;\n\t}"
        : "=r"(e0), "=r"(e1)
        : "r"(s0), "r"(s1), "f"(c0), "f"(c1), "l"(arow), "l"(shift));
}

// acc + (e0, e1) on an f32x2 pair.
__device__ __forceinline__ uint64_t add_pair(uint64_t acc, uint32_t e0, uint32_t e1)
{
    uint64_t d;
    asm("{\n\t.reg .b64 x;\n\tmov.b64 x, {%2, %3};\n\tadd.rn.f32x2 %0, %1, x;\n\t}"
        : "=l"(d)
        : "l"(acc), "r"(e0), "r"(e1));
    return d;
}

// Two fp32 values to one fp16x2 word, round-to-nearest-even; `lo` lands at the lower address.
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ------------------------------------------------------------------ programmatic dependent launch

// Blocks until the grids this one depends on (the previous kernel in the stream, when
// launched with programmatic serialisation) have completed and their memory is visible.
// A no-op for a normal launch.
__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next grid in the stream start its prologue once every CTA of this grid has issued
// this or exited. It does not publish memory: the dependent still calls griddep_wait().
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace ptx
}  // namespace mg
