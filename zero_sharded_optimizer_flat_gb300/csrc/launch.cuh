// Kernel launch with programmatic dependent launch (the Newton-Schulz kernels chain their
// launches this way).
#pragma once

#include <cuda_runtime.h>

#include <utility>

#include "internal.h"

namespace zopt {

// init() evaluated once per process, on the first call, and returned on every call: a
// function-local static of a template instantiated per lambda type, i.e. per call site, so
// concurrent first calls from several host threads are safe.
template <typename F>
auto once(F init) -> decltype(init()) {
  static const decltype(init()) value = init();
  return value;
}

// Launches `kernel` on `stream` with programmatic stream serialisation: it may start while
// the previous kernel finishes (every kernel here waits with griddepcontrol.wait before it
// touches global memory).
template <typename... KArgs, typename... Args>
zopt_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ZOPT_CUDA_TRY(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...));
  return ok();
}

}  // namespace zopt
