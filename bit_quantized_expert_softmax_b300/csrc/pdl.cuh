// Programmatic dependent launch for chains of kernels on one stream (the
// prefill layer's eight kernels, the decode-path router, expert and combine
// kernels, the output head's GEMV and sampler): a kernel launched with launch_pdl may be
// launched while the kernel before it in the stream is still finishing, so
// that its launch overlaps the end of that kernel instead of following it.
//
// Contract of a kernel launched this way: its first statement is
// griddep_wait(), which returns once the previous kernel has completed and its
// memory operations are visible; nothing before it touches memory. The
// kernels trigger their dependents only implicitly, as their CTAs exit
// (measured: an explicit trigger at the start of every CTA let the next
// kernel's CTAs take SM resources early and made the layer slower). Launched
// without the attribute, or with no kernel before it, griddep_wait() returns
// at once.
#pragma once

#include <cuda_runtime.h>

namespace flint {

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KP, typename... A>
cudaError_t launch_pdl(void (*kernel)(KP...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...);
}

}  // namespace flint
