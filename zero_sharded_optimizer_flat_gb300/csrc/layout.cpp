// Flat bucketed shard layout (host only).
//
// deg/zero.py, ZeroMaster: parameters end to end in a flat vector of N elements; buckets of
// `bucket` elements after rounding the bucket down to a multiple of world (never below
// world); each bucket [s, e) padded to a multiple of world; rank r owns the r-th of world
// equal pieces of every bucket, concatenated in bucket order (class docstring, __init__,
// _pieces). Segments follow _segments: the parameter runs that cover a flat range.
#include <algorithm>
#include <new>

#include "internal.h"

namespace {

constexpr int64_t kMaxNumel = int64_t(1) << 62;

}  // namespace

extern "C" zopt_status zopt_shard_layout(const int64_t* numel, const uint8_t* decay, int32_t n_params,
                                         int64_t bucket, int32_t world, int32_t rank, zopt_layout** out) {
  if (out == nullptr) return zopt::fail(ZOPT_EINVAL, "zopt_shard_layout: out is NULL");
  *out = nullptr;
  if (n_params < 1 || numel == nullptr)
    return zopt::fail(ZOPT_EINVAL, "zopt_shard_layout: needs trainable parameters (n_params < 1)");
  if (world < 1) return zopt::fail(ZOPT_EINVAL, "zopt_shard_layout: world < 1");
  if (rank < 0 || rank >= world) return zopt::fail(ZOPT_EINVAL, "zopt_shard_layout: rank outside [0, world)");
  if (bucket < 1) return zopt::fail(ZOPT_EINVAL, "zopt_shard_layout: bucket < 1");

  std::vector<int64_t> offsets(static_cast<size_t>(n_params) + 1, 0);
  for (int32_t i = 0; i < n_params; ++i) {
    if (numel[i] < 0) return zopt::fail(ZOPT_EINVAL, "zopt_shard_layout: negative parameter size");
    if (numel[i] > kMaxNumel - offsets[i]) return zopt::fail(ZOPT_EINVAL, "zopt_shard_layout: total size >= 2^62");
    offsets[i + 1] = offsets[i] + numel[i];
  }
  const int64_t N = offsets[n_params];
  if (N < 1) return zopt::fail(ZOPT_EINVAL, "zopt_shard_layout: all parameters are empty");

  zopt_layout* L = new (std::nothrow) zopt_layout();
  if (L == nullptr) return zopt::fail(ZOPT_EINVAL, "zopt_shard_layout: out of host memory");
  L->world = world;
  L->rank = rank;
  L->numel = N;
  const int64_t w = world;
  L->bucket = std::max<int64_t>(w, bucket - bucket % w);

  // Buckets and this rank's piece of each.
  int64_t shard_off = 0;
  for (int64_t s = 0; s < N; s += L->bucket) {
    const int64_t e = std::min(N, s + L->bucket);
    const int64_t padded = (e - s + w - 1) / w * w;
    L->buckets.push_back({s, e, padded, shard_off});
    shard_off += padded / w;
  }
  L->shard_len = shard_off;

  // Segments of each piece, and the shard's decay flag runs (padding counts as no-decay).
  std::vector<std::pair<int64_t, int64_t>> nd;  // no-decay runs before merging
  auto add_nodecay = [&nd](int64_t a, int64_t b) {
    if (b <= a) return;
    if (!nd.empty() && nd.back().second == a)
      nd.back().second = b;
    else
      nd.emplace_back(a, b);
  };
  for (const auto& bk : L->buckets) {
    const int64_t piece = bk.padded / w;
    const int64_t a0 = bk.start + static_cast<int64_t>(rank) * piece;  // flat begin of the piece
    const int64_t b0 = std::min(bk.end, a0 + piece);                     // flat end of real data
    if (a0 < b0) {
      int32_t i = static_cast<int32_t>(std::upper_bound(offsets.begin(), offsets.end(), a0) - offsets.begin()) - 1;
      for (; i < n_params && offsets[i] < b0; ++i) {
        const int64_t a = std::max(a0, offsets[i]);
        const int64_t b = std::min(b0, offsets[i + 1]);
        if (b <= a) continue;
        const int64_t so = bk.shard_offset + (a - a0);
        L->seg_param.push_back(i);
        L->seg_param_off.push_back(a - offsets[i]);
        L->seg_shard_off.push_back(so);
        L->seg_len.push_back(b - a);
        const bool decays = decay == nullptr || decay[i] != 0;
        if (!decays) add_nodecay(so, so + (b - a));
      }
    }
    // padding slots of this piece: flat positions >= e
    const int64_t real = std::max<int64_t>(0, b0 - a0);
    add_nodecay(bk.shard_offset + real, bk.shard_offset + piece);
  }
  for (const auto& r : nd) {
    L->nodecay.push_back(r.first);
    L->nodecay.push_back(r.second);
  }
  *out = L;
  return zopt::ok();
}

extern "C" void zopt_layout_free(zopt_layout* layout) { delete layout; }

extern "C" int64_t zopt_layout_numel(const zopt_layout* L) { return L ? L->numel : -1; }
extern "C" int64_t zopt_layout_shard_len(const zopt_layout* L) { return L ? L->shard_len : -1; }

extern "C" int64_t zopt_layout_state_bytes(const zopt_layout* L, zopt_dtype grad_dtype) {
  if (L == nullptr || (grad_dtype != ZOPT_F32 && grad_dtype != ZOPT_BF16)) return -1;
  return L->shard_len * (12 + (grad_dtype == ZOPT_F32 ? 4 : 2));
}
extern "C" int32_t zopt_layout_world(const zopt_layout* L) { return L ? L->world : -1; }
extern "C" int32_t zopt_layout_rank(const zopt_layout* L) { return L ? L->rank : -1; }
extern "C" int32_t zopt_layout_num_buckets(const zopt_layout* L) {
  return L ? static_cast<int32_t>(L->buckets.size()) : -1;
}

extern "C" zopt_status zopt_layout_bucket(const zopt_layout* L, int32_t b, int64_t* start, int64_t* end,
                                          int64_t* padded, int64_t* shard_offset) {
  if (L == nullptr) return zopt::fail(ZOPT_EINVAL, "zopt_layout_bucket: layout is NULL");
  if (b < 0 || b >= static_cast<int32_t>(L->buckets.size()))
    return zopt::fail(ZOPT_EINVAL, "zopt_layout_bucket: bucket index out of range");
  const auto& bk = L->buckets[b];
  if (start) *start = bk.start;
  if (end) *end = bk.end;
  if (padded) *padded = bk.padded;
  if (shard_offset) *shard_offset = bk.shard_offset;
  return zopt::ok();
}

extern "C" int64_t zopt_layout_num_segments(const zopt_layout* L) {
  return L ? static_cast<int64_t>(L->seg_len.size()) : -1;
}

extern "C" zopt_status zopt_layout_segments(const zopt_layout* L, int32_t* param, int64_t* param_offset,
                                            int64_t* shard_offset, int64_t* length) {
  if (L == nullptr) return zopt::fail(ZOPT_EINVAL, "zopt_layout_segments: layout is NULL");
  const size_t n = L->seg_len.size();
  for (size_t i = 0; i < n; ++i) {
    if (param) param[i] = L->seg_param[i];
    if (param_offset) param_offset[i] = L->seg_param_off[i];
    if (shard_offset) shard_offset[i] = L->seg_shard_off[i];
    if (length) length[i] = L->seg_len[i];
  }
  return zopt::ok();
}

extern "C" int64_t zopt_layout_num_nodecay_runs(const zopt_layout* L) {
  return L ? static_cast<int64_t>(L->nodecay.size() / 2) : -1;
}

extern "C" zopt_status zopt_layout_nodecay_runs(const zopt_layout* L, int64_t* runs) {
  if (L == nullptr) return zopt::fail(ZOPT_EINVAL, "zopt_layout_nodecay_runs: layout is NULL");
  if (runs == nullptr && !L->nodecay.empty())
    return zopt::fail(ZOPT_EINVAL, "zopt_layout_nodecay_runs: runs is NULL");
  std::copy(L->nodecay.begin(), L->nodecay.end(), runs);
  return zopt::ok();
}
