// Internal helpers shared by libzopt's translation units (not part of the ABI).
#pragma once

#include <cstdint>
#include <cstdio>
#include <string>
#include <vector>

#include "zopt.h"

namespace zopt {

// Records `msg` as this host thread's last error and returns `st`.
zopt_status fail(zopt_status st, const std::string& msg);
// Clears the last error and returns ZOPT_OK.
zopt_status ok();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count of the current device (cached per device ordinal); 0 on error.
int sm_count();

}  // namespace zopt

// Host-side view of the layout object (owned by layout.cpp, read by the kernels' wrappers).
struct zopt_layout {
  int32_t world = 1, rank = 0;
  int64_t bucket = 0;  // effective bucket (multiple of world, >= world)
  int64_t numel = 0;   // N
  int64_t shard_len = 0;
  struct Bucket { int64_t start, end, padded, shard_offset; };
  std::vector<Bucket> buckets;
  std::vector<int32_t> seg_param;
  std::vector<int64_t> seg_param_off, seg_shard_off, seg_len;
  std::vector<int64_t> nodecay;  // flattened [begin, end) pairs
};

#define ZOPT_CUDA_TRY(expr)                                                             \
  do {                                                                                  \
    cudaError_t e_ = (expr);                                                            \
    if (e_ != cudaSuccess)                                                              \
      return ::zopt::fail(ZOPT_ECUDA, std::string(#expr ": ") + cudaGetErrorString(e_)); \
  } while (0)
