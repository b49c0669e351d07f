// smem_limit.h -- a kernel's dynamic shared-memory limit, raised and never
// lowered.  Internal to libmoe_a2a.so.
//
// cudaFuncAttributeMaxDynamicSharedMemorySize is one value per kernel and
// context for the whole process, while each handle prepares the kernels for
// its own row size.  Setting it to a handle's own size would take it below
// what an earlier handle of a larger size launches with, and that handle's
// next launch would be refused.  So the limit only ever grows: the live
// value is read (correct also after the context was reset) and raised when
// it is below the size asked for, under one lock so that concurrent handles
// cannot lower each other's raise.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

namespace moe {

inline cudaError_t raise_smem_limit(const void *func, size_t bytes) {
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    cudaFuncAttributes fa;
    cudaError_t err = cudaFuncGetAttributes(&fa, func);
    if (err != cudaSuccess) return err;
    if ((size_t)fa.maxDynamicSharedSizeBytes >= bytes) return cudaSuccess;
    return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename Kernel>
inline cudaError_t raise_smem_limit(Kernel *func, size_t bytes) {
    return raise_smem_limit(reinterpret_cast<const void *>(func), bytes);
}

}  // namespace moe
