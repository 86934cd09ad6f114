// mg_diag.cu -- the two device measurements declared in include/mg_diag.h: the launch floor of
// the fused kernel's launch shape and the rate of its exponential.
#include "mg_diag.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <vector>

#include "mg_attn_kernels.cuh"

namespace {

thread_local char g_diag_error[512] = "";

mg_status diag_fail(mg_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_diag_error, sizeof(g_diag_error), fmt, ap);
    va_end(ap);
    return s;
}

mg_status diag_cuda(cudaError_t e, const char *what)
{
    return diag_fail(MG_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kFloorThreads = mg::kThreads;  // the fused kernel's block size
constexpr int kFloorMinSmem = 120 * 1024;
constexpr int kExpThreads = 512;
constexpr int kExpPairs = 8;  // independent pairs per thread and round

// The fused kernel's prologue and teardown and nothing else: tensor-memory allocation by warp 1,
// the dependent-launch handshake, one cluster barrier, the free.
// The tensor-memory address lives in the dynamic shared memory, like the fused kernel's, so the
// kernel accepts the same dynamic size (up to the opt-in limit, with no static shared memory).
__global__ void __launch_bounds__(kFloorThreads, 1) floor_kernel(int use_cluster)
{
    extern __shared__ uint32_t dyn_smem[];
    uint32_t &holder = dyn_smem[0];
    const int warp = threadIdx.x >> 5;
    if (warp == 1) {
        mg::ptx::tmem_alloc(mg::ptx::smem_u32(&holder), 512);
        mg::ptx::tmem_relinquish();
    }
    mg::ptx::tc_fence_before();
    __syncthreads();
    mg::ptx::tc_fence_after();
    mg::ptx::griddep_wait();
    mg::ptx::griddep_launch_dependents();
    if (use_cluster)
        mg::ptx::cluster_sync();
    mg::ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        mg::ptx::tc_fence_after();
        mg::ptx::tmem_dealloc(holder, 512);
    }
}

// Rounds of kExpPairs independent pairs per thread. Each result feeds the next round of its
// chain as exp(-x): the values stay in (0, 1], so no chain reaches inf or 0.
template <bool POLY>
__global__ void __launch_bounds__(kExpThreads, 1)
    exp_rate_kernel(int iters, unsigned long long *out, uint32_t *sink)
{
    mg::ptx::ExpPairConsts k = mg::ptx::exp_pair_consts();
    k.log2e = mg::ptx::pair_of(__float_as_uint(-mg::ptx::kLog2e));
    uint32_t x[2 * kExpPairs];
#pragma unroll
    for (int i = 0; i < 2 * kExpPairs; ++i)
        x[i] = __float_as_uint(0.25f + 0.01f * static_cast<float>(i + (threadIdx.x & 7)));
    __syncthreads();
    const long long c0 = clock64();
    const uint64_t g0 = mg::ptx::globaltimer_ns();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int p = 0; p < kExpPairs; ++p) {
            if (POLY)
                mg::ptx::exp_pair_fma(x[2 * p], x[2 * p + 1], k, x[2 * p], x[2 * p + 1]);
            else
                mg::ptx::exp_pair_mufu(x[2 * p], x[2 * p + 1], k, 0ull, x[2 * p], x[2 * p + 1]);
        }
    }
    __syncthreads();
    const long long c1 = clock64();
    const uint64_t g1 = mg::ptx::globaltimer_ns();
    if (threadIdx.x == 0) {
        out[2 * blockIdx.x] = static_cast<unsigned long long>(c1 - c0);
        out[2 * blockIdx.x + 1] = g1 - g0;
    }
    uint32_t acc = 0;
#pragma unroll
    for (int i = 0; i < 2 * kExpPairs; ++i)
        acc ^= x[i];
    if (acc == 0x7fc00001u)  // never true for values in (0, 1]; keeps the chains live
        sink[0] = acc;
}

double median(std::vector<double> v)
{
    std::sort(v.begin(), v.end());
    const size_t n = v.size();
    return n % 2 ? v[n / 2] : 0.5 * (v[n / 2 - 1] + v[n / 2]);
}

}  // namespace

extern "C" {

const char *mg_diag_last_error(void) { return g_diag_error; }

mg_status mg_diag_launch_floor(int32_t ctas, int32_t cluster, int32_t smem_bytes, int32_t pdl, int32_t launches,
                               float *us_per_launch)
{
    if (!us_per_launch)
        return diag_fail(MG_ERR_INVALID_ARG, "NULL output");
    if (ctas < 1 || ctas > 65535 || cluster < 1 || cluster > 16 || ctas % cluster != 0 || launches < 1 ||
        launches > 100000)
        return diag_fail(MG_ERR_INVALID_ARG, "ctas %d, cluster %d, launches %d out of range", ctas, cluster,
                         launches);
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess)
        return diag_cuda(e, "device query");
    if (smem_bytes < kFloorMinSmem || smem_bytes > optin)
        return diag_fail(MG_ERR_INVALID_ARG, "smem_bytes %d outside [%d, %d]", smem_bytes, kFloorMinSmem, optin);
    e = cudaFuncSetAttribute(floor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e == cudaSuccess && cluster > 8)
        e = cudaFuncSetAttribute(floor_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess)
        return diag_cuda(e, "cudaFuncSetAttribute");

    cudaStream_t s = nullptr;
    e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e != cudaSuccess)
        return diag_cuda(e, "cudaStreamCreate");
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(kFloorThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(na);

    mg_status st = MG_OK;
    cudaGraph_t g = nullptr;
    cudaGraphExec_t ge = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    const int use_cluster = cluster > 1 ? 1 : 0;
    if (cluster > 1) {
        int active = 0;
        e = cudaOccupancyMaxActiveClusters(&active, floor_kernel, &cfg);
        if (e != cudaSuccess)
            st = diag_cuda(e, "cudaOccupancyMaxActiveClusters");
        else if (active < 1)
            st = diag_fail(MG_ERR_CONFIG, "a cluster of %d CTAs with %d B of shared memory cannot be scheduled",
                           cluster, smem_bytes);
    }
    if (st == MG_OK) {
        e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
        for (int i = 0; e == cudaSuccess && i < launches; ++i)
            e = cudaLaunchKernelEx(&cfg, floor_kernel, use_cluster);
        const cudaError_t e_end = cudaStreamEndCapture(s, &g);
        if (e == cudaSuccess)
            e = e_end;
        if (e == cudaSuccess)
            e = cudaGraphInstantiate(&ge, g, 0);
        if (e == cudaSuccess)
            e = cudaGraphLaunch(ge, s);  // warm-up
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(s);
        if (e == cudaSuccess)
            e = cudaEventCreate(&e0);
        if (e == cudaSuccess)
            e = cudaEventCreate(&e1);
        if (e == cudaSuccess)
            e = cudaEventRecord(e0, s);
        if (e == cudaSuccess)
            e = cudaGraphLaunch(ge, s);
        if (e == cudaSuccess)
            e = cudaEventRecord(e1, s);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(s);
        float ms = 0.f;
        if (e == cudaSuccess)
            e = cudaEventElapsedTime(&ms, e0, e1);
        if (e != cudaSuccess)
            st = diag_cuda(e, "launch floor");
        else
            *us_per_launch = ms * 1000.f / static_cast<float>(launches);
    }
    if (e0)
        cudaEventDestroy(e0);
    if (e1)
        cudaEventDestroy(e1);
    if (ge)
        cudaGraphExecDestroy(ge);
    if (g)
        cudaGraphDestroy(g);
    cudaStreamDestroy(s);
    return st;
}

mg_status mg_diag_exp_rate(int32_t iters, int32_t poly, double *exp_per_clk_per_sm, double *exp_per_ns_per_sm)
{
    if (!exp_per_clk_per_sm || !exp_per_ns_per_sm)
        return diag_fail(MG_ERR_INVALID_ARG, "NULL output");
    if (iters < 1 || iters > 1000000)
        return diag_fail(MG_ERR_INVALID_ARG, "iters %d out of range", iters);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return diag_cuda(e, "device query");
    // More than half of an SM's shared memory per CTA: one CTA per SM.
    const int smem = kFloorMinSmem;
    auto kern = poly ? exp_rate_kernel<true> : exp_rate_kernel<false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return diag_cuda(e, "cudaFuncSetAttribute");
    cudaStream_t s = nullptr;
    e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e != cudaSuccess)
        return diag_cuda(e, "cudaStreamCreate");
    unsigned long long *d_out = nullptr;
    uint32_t *d_sink = nullptr;
    std::vector<unsigned long long> h(2 * static_cast<size_t>(sms));
    e = cudaMalloc(&d_out, h.size() * sizeof(unsigned long long));
    if (e == cudaSuccess)
        e = cudaMalloc(&d_sink, sizeof(uint32_t));
    for (int rep = 0; e == cudaSuccess && rep < 2; ++rep) {  // the first launch warms up
        kern<<<sms, kExpThreads, smem, s>>>(iters, d_out, d_sink);
        e = cudaGetLastError();
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(s);
    }
    if (e == cudaSuccess)
        e = cudaMemcpy(h.data(), d_out, h.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    mg_status st = MG_OK;
    if (e != cudaSuccess) {
        st = diag_cuda(e, "exp rate");
    } else {
        const double per_cta = static_cast<double>(iters) * kExpThreads * kExpPairs * 2;
        std::vector<double> clk, ns;
        for (int i = 0; i < sms; ++i) {
            clk.push_back(per_cta / static_cast<double>(std::max<unsigned long long>(h[2 * i], 1)));
            ns.push_back(per_cta / static_cast<double>(std::max<unsigned long long>(h[2 * i + 1], 1)));
        }
        *exp_per_clk_per_sm = median(clk);
        *exp_per_ns_per_sm = median(ns);
    }
    if (d_out)
        cudaFree(d_out);
    if (d_sink)
        cudaFree(d_sink);
    cudaStreamDestroy(s);
    return st;
}

}  // extern "C"
