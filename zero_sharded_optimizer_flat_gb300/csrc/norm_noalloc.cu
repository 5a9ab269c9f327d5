// zopt_grad_norm_clip_noalloc: the gradient norm / clip reduction for callers that cannot
// allocate device memory.
//
// Some callers have no way to call cudaMalloc or a caching allocator at the point where the
// step runs: a plain-C host program or plugin that only receives device pointers from its
// framework, a real-time training loop that forbids allocation after start-up, or a process
// whose device memory is fully reserved by another runtime. zopt_grad_norm_clip needs a
// caller-provided workspace (block partial sums and an arrival counter); this variant keeps
// that scratch in a file-scope __device__ array instead, so the caller passes only the
// gradient and the stats struct.
//
// Limits: the array holds the arrival counter and kStaticPartials fp64 partial sums, 8,448
// bytes in all, and every GPU that loads the library keeps it until the process exits. A
// launch uses one partial per block. Its grid is the one zopt_grad_norm_clip takes (one wave
// of resident blocks: 304 for bf16 and 608 for fp32 gradients on a 152-SM GB300), capped at
// kStaticPartials blocks; the kernel walks the gradient grid-stride, so a capped grid covers
// every element too (it only changes the order of the fp64 partial sums). Under the cap the
// result is bit for bit zopt_grad_norm_clip's.
// All calls share the one array: calls that overlap on the GPU (different streams, or
// different host threads without ordering) race on it and give wrong results.
// The address cache below is per device index for the life of the process; after a
// cudaDeviceReset the module may load elsewhere, so this entry point must not be called
// again in a process that has reset a device it used.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "internal.h"
#include "norm_impl.cuh"

namespace zopt {
namespace {

constexpr int kStaticPartials = 1024;
constexpr size_t kStaticBytes = 256 + sizeof(double) * kStaticPartials;

// The scratch: a NormWorkspace header (arrival counter, 256 bytes) and the partials.
static __device__ __align__(256) unsigned char g_norm_scratch[kStaticBytes];

// The scratch's device address on each device. In host code `g_norm_scratch` names a host
// stand-in, not device memory, so the address is looked up once per device with that device
// current and cached here.
std::mutex g_mu;
std::vector<void*> g_scratch_addr;

zopt_status scratch_address(void** out) {
  int dev = 0;
  ZOPT_CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(g_mu);
  if (dev >= static_cast<int>(g_scratch_addr.size())) g_scratch_addr.resize(dev + 1, nullptr);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_norm_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(ZOPT_ECUDA, std::string("zopt_grad_norm_clip_noalloc: cudaGetSymbolAddress failed: ") +
                                  cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return ok();
}

}  // namespace
}  // namespace zopt

extern "C" zopt_status zopt_grad_norm_clip_noalloc(const void* grad, zopt_dtype dtype, int64_t n, float max_norm,
                                                   zopt_clip_stats* d_stats, zopt_stream stream) {
  using namespace zopt;
  zopt_status st = check_norm_args("zopt_grad_norm_clip_noalloc", grad, dtype, n, max_norm, d_stats);
  if (st != ZOPT_OK) return st;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != ZOPT_OK) return st;
  int blocks = norm_launch_blocks(n, dtype);
  if (blocks <= 0) return fail(ZOPT_ECUDA, "zopt_grad_norm_clip_noalloc: no CUDA device");
  if (blocks > kStaticPartials) blocks = kStaticPartials;  // grid-stride: fewer blocks still cover n
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the arrival counter must start at zero
  // (the partials are written before they are read).
  ZOPT_CUDA_TRY(cudaMemsetAsync(scratch, 0, sizeof(unsigned int), s));
  NormWorkspace* ws = static_cast<NormWorkspace*>(scratch);
  if (dtype == ZOPT_F32)
    norm_kernel<float><<<static_cast<unsigned>(blocks), kNormThreads, 0, s>>>(static_cast<const float*>(grad), n,
                                                                             max_norm, ws, d_stats);
  else
    norm_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), kNormThreads, 0, s>>>(
        static_cast<const __nv_bfloat16*>(grad), n, max_norm, ws, d_stats);
  ZOPT_CUDA_TRY(cudaGetLastError());
  return ok();
}
