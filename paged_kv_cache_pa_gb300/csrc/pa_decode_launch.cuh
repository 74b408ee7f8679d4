// pa_decode_launch.cuh -- host-side launch of one paged_decode_kernel
// instantiation: shared-memory attribute and occupancy (cached per device),
// persistent grid of min(items, SMs x resident CTAs), programmatic dependent
// launch after the plan kernel.
#pragma once

#include <atomic>

#include "pa_decode.cuh"
#include "pa_decode_mma.cuh"
#include "pa_launch.cuh"

namespace pa {

constexpr int kMaxDevices = 64;

template <int D, int GM, typename T, bool DIRECT>
pa_status_t launch_one_form(const DecodeParams &P, int grid_cap, cudaStream_t stream) {
    using Tn = Tuning<D, GM>;
    constexpr int R = Tn::kStages;
    constexpr int MINB = Tn::kMinBlocks;
    using L = Layout<D, GM, R>;
    auto kern = paged_decode_kernel<D, GM, T, R, MINB, DIRECT>;
    static std::atomic<int> occ_cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    int occ = occ_cache[dev].load(std::memory_order_relaxed);
    if (occ == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)L::bytes) != cudaSuccess)
            return PA_ERR_CUDA;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, L::bytes) !=
            cudaSuccess)
            return PA_ERR_CUDA;
        if (occ < 1) return PA_ERR_UNSUPPORTED;
        occ_cache[dev].store(occ, std::memory_order_relaxed);
    }
    long long grid = (long long)current_sm_count() * occ;
    if (grid > grid_cap) grid = grid_cap;
    if (grid < 1) grid = 1;

    if (launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), L::bytes, stream, P) != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}

// The kernel's planned or plan-free (DIRECT) form, as P.direct says.
template <int D, int GM, typename T>
pa_status_t launch_one(const DecodeParams &P, int grid_cap, cudaStream_t stream) {
    return P.direct ? launch_one_form<D, GM, T, true>(P, grid_cap, stream)
                    : launch_one_form<D, GM, T, false>(P, grid_cap, stream);
}

// Consumer warps per CTA of the tensor-core kernel.
constexpr int kMmaWarps = 4;

template <int D, typename T, bool DIRECT, int W = kMmaWarps>
pa_status_t launch_one_mma_form(const DecodeParams &P, int grid_cap, cudaStream_t stream) {
    using Tn = TuningMma<D, W>;
    constexpr int R = Tn::kStages;
    constexpr int MINB = Tn::kMinBlocks;
    using L = LayoutMma<D, R, W>;
    auto kern = paged_decode_mma_kernel<D, T, R, MINB, W, DIRECT>;
    static std::atomic<int> occ_cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    int occ = occ_cache[dev].load(std::memory_order_relaxed);
    if (occ == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)L::bytes) != cudaSuccess)
            return PA_ERR_CUDA;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads_mma<W>(), L::bytes) !=
            cudaSuccess)
            return PA_ERR_CUDA;
        if (occ < 1) return PA_ERR_UNSUPPORTED;
        occ_cache[dev].store(occ, std::memory_order_relaxed);
    }
    long long grid = (long long)current_sm_count() * occ;
    if (grid > grid_cap) grid = grid_cap;
    if (grid < 1) grid = 1;
    if (launch_pdl(kern, dim3((unsigned)grid), dim3(threads_mma<W>()), L::bytes, stream, P) !=
        cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}

template <int D, typename T>
pa_status_t launch_one_mma(const DecodeParams &P, int grid_cap, cudaStream_t stream) {
    return P.direct ? launch_one_mma_form<D, T, true>(P, grid_cap, stream)
                    : launch_one_mma_form<D, T, false>(P, grid_cap, stream);
}

template <int D, typename T>
pa_status_t dispatch_group(const DecodeParams &P, int grid_cap, cudaStream_t stream, int kernel) {
    const int G = P.G;
    if constexpr (D <= 128) {
        if (kernel == kKernelTensorCore && G <= 8) return launch_one_mma<D, T>(P, grid_cap, stream);
        if (G == 1) return launch_one<D, 1, T>(P, grid_cap, stream);
        if (G <= 8) return launch_one_mma<D, T>(P, grid_cap, stream);
    } else {
        if (G == 1) return launch_one<D, 1, T>(P, grid_cap, stream);
        if (G == 2) return launch_one<D, 2, T>(P, grid_cap, stream);
        if (G <= 4) return launch_one<D, 4, T>(P, grid_cap, stream);
        if (G <= 6) return launch_one<D, 6, T>(P, grid_cap, stream);
        if (G <= 8) return launch_one<D, 8, T>(P, grid_cap, stream);
    }
    return PA_ERR_UNSUPPORTED;
}

template <int D>
pa_status_t dispatch_dtype(const DecodeParams &P, pa_dtype_t dtype, int grid_cap,
                           cudaStream_t stream, int kernel) {
    if (dtype == PA_F16) return dispatch_group<D, __half>(P, grid_cap, stream, kernel);
    if (dtype == PA_BF16) return dispatch_group<D, __nv_bfloat16>(P, grid_cap, stream, kernel);
    return PA_ERR_INVALID_ARG;
}

}  // namespace pa
