// C ABI of the segmented top-k library: argument validation, launch planning
// and dispatch to the per-key-type kernels. See include/segtopk.h.
#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "../../include/segtopk.h"
#include "block_select.cuh"
#include "device_prep.h"
#include "dispatch.h"
#include "stream_topk.cuh"
#include "warp_topk.cuh"

namespace segtopk {
namespace {

thread_local int t_last_cuda_error = 0;
thread_local int t_last_launch_count = 0;

int cuda_fail(cudaError_t e)
{
  t_last_cuda_error = (int)e;
  return SEGTOPK_ERROR_CUDA;
}

const KeyOps* ops_for(int dtype)
{
  switch (dtype) {
  case SEGTOPK_F16: return &key_ops_f16();
  case SEGTOPK_BF16: return &key_ops_bf16();
  case SEGTOPK_F32: return &key_ops_f32();
  case SEGTOPK_F64: return &key_ops_f64();
  case SEGTOPK_U32: return &key_ops_u32();
  case SEGTOPK_I32: return &key_ops_i32();
  default: return nullptr;
  }
}

// Device facts, cached per device.
struct DeviceInfo {
  bool valid = false;
  int major = 0, minor = 0, sms = 0;
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

cudaError_t device_info(DeviceInfo* out)
{
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return e;
  if (dev < 0 || dev >= 64)
    return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.valid) {
    if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    d.valid = true;
  }
  *out = d;
  return cudaSuccess;
}

constexpr int64_t kMinSliceKeys = 16384; // a CTA of a multi-CTA cluster reads at least this many keys
constexpr int kThreads = kCtaThreads;

struct Plan {
  LaunchShape shape;
  uint32_t list_cap;
  uint32_t ring_bytes;
  int merge_gather;
  int64_t waves; // waves of resident CTAs (or clusters) over all segments
};

uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Largest C * k for which the cluster gathers whole candidate lists.
constexpr uint32_t kGatherListsMaxItems = 512;
// Largest C * k for which the cluster gathers local top-k lists into the leader.
constexpr uint32_t kGatherMaxItems = 2048;

// Candidate-list room beyond k: keys accepted after a selection before the
// list overflows and the next selection (over the list and the chunk being
// read) tightens the bound.
uint32_t list_slack(uint32_t k) { return std::max(1024u, k / 2); }

// Ring bytes of a kernel profile.
uint32_t profile_ring_bytes(int profile) { return profile == 0 ? ProfileLong::kRingBytes : ProfileMany::kRingBytes; }
uint32_t profile_cand_bytes(int profile) { return profile == 0 ? ProfileLong::kCandBytes : ProfileMany::kCandBytes; }

// Wait bound and copy-count offset handed to the kernels (changed only by the
// test hooks of the instrumented build).
long long g_wait_limit = kWaitLimitCycles;
uint32_t g_test_extra_tx = 0;

// Shared-memory sizing for a given k, cluster width and kernel profile. The
// ring doubles as sort scratch and, in a cluster leader, as gather space.
Plan size_plan(const KeyOps& ops, int32_t k, int cluster, int profile)
{
  Plan pl;
  const uint32_t kb = (uint32_t)ops.key_bytes;
  const uint32_t uk = (uint32_t)k;
  pl.list_cap = align_up(uk + list_slack(uk), 32);
  const uint32_t stream_ring = profile_ring_bytes(profile);
  const uint32_t sort_need = std::max(sort_scratch_bytes(uk, ops.rank_bits), finalize_scratch_bytes(kCountFinalMax));
  uint32_t need = sort_need;
  pl.merge_gather = 0;
  if (cluster > 1) {
    // 2: every CTA's whole list fits in the leader and C * k is small: no
    // local trims, one selection in the leader; 1: every CTA's local top-k
    // fits and the leader's selection over them stays short; 0: histogram
    // merge through DSMEM (measured faster than a gather of more than
    // kGatherMaxItems entries, whose serial selection and tie resolution in
    // the leader dominate)
    auto gather_need = [&](uint32_t cap) { return align16(cap * kb) + align16(cap * 4u) + sort_need; };
    if (gather_need((uint32_t)cluster * pl.list_cap) <= stream_ring && (uint32_t)cluster * uk <= kGatherListsMaxItems)
      pl.merge_gather = 2;
    else if (gather_need((uint32_t)cluster * uk) <= stream_ring && (uint32_t)cluster * uk <= kGatherMaxItems)
      pl.merge_gather = 1;
    need = pl.merge_gather ? gather_need((uint32_t)cluster * (pl.merge_gather == 2 ? pl.list_cap : uk))
                           : align16(uk * kb) + align16(uk * 4u) + sort_need;
  }
  pl.ring_bytes = align_up(std::max(stream_ring, need), 128);
  pl.shape.threads = kThreads;
  pl.shape.cluster = cluster;
  pl.shape.profile = profile;
  pl.shape.smem = kCtrlBytes + pl.ring_bytes + 2 * list_bytes(pl.list_cap, kb) + profile_cand_bytes(profile);
  return pl;
}

// Cluster width: fewest waves of resident clusters over all segments, ties
// toward the widest cluster ("Implement Segmented TopK using
// Thread-Block-Clusters", section 3.3 "Wave-aware cluster-size search"),
// using the occupancy the device reports for this kernel and its
// shared-memory size. A CTA of a multi-CTA cluster must get at least
// kMinSliceKeys keys of the longest segment.
cudaError_t choose_plan(const KeyOps& ops, int64_t num_segments, int64_t max_len, int32_t k, Plan* out)
{
  static const int widths[] = {1, 2, 3, 4, 6, 8, 12, 16};
  bool have = false;
  int64_t best_waves = 0;
  for (int c : widths) {
    if (c > 1 && max_len < (int64_t)c * kMinSliceKeys)
      break;
    Plan pl = size_plan(ops, k, c, 0);
    int resident = 0;
    cudaError_t e = ops.occupancy[0](pl.shape, &resident);
    if (e != cudaSuccess) {
      (void)cudaGetLastError(); // an unlaunchable width is skipped, not an error
      continue;
    }
    if (resident <= 0)
      continue;
    const int64_t waves = (num_segments + resident - 1) / resident;
    if (!have || waves <= best_waves) {
      have = true;
      best_waves = waves;
      pl.waves = waves;
      *out = pl;
    }
  }
  return have ? cudaSuccess : cudaErrorInvalidConfiguration;
}

// Plans are cached per (device, key type, num_segments, max_len, k, forced
// width): after the first call a call only validates and launches, so it can
// also be captured into a CUDA graph.
using PlanKey = std::tuple<int, int, int64_t, int64_t, int32_t, int>;
std::mutex g_plan_mu;
std::map<PlanKey, Plan> g_plans;

cudaError_t get_plan(int dtype, const KeyOps& ops, int64_t num_segments, int64_t max_len, int32_t k,
                     int forced_width, Plan* out, bool* unsupported)
{
  *unsupported = false;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return e;
  const PlanKey key(dev, dtype, num_segments, max_len, k, forced_width);
  {
    std::lock_guard<std::mutex> lk(g_plan_mu);
    auto it = g_plans.find(key);
    if (it != g_plans.end()) {
      *out = it->second;
      return cudaSuccess;
    }
  }
  Plan pl;
  if (forced_width > 0) {
    pl = size_plan(ops, k, forced_width, 0);
    int resident = 0;
    e = ops.occupancy[0](pl.shape, &resident);
    pl.waves = resident > 0 ? (num_segments + resident - 1) / resident : 0;
    if (e != cudaSuccess || resident <= 0) {
      (void)cudaGetLastError();
      *unsupported = true;
      return cudaSuccess;
    }
  } else {
    e = choose_plan(ops, num_segments, max_len, k, &pl);
    if (e != cudaSuccess)
      return e;
  }
  if (pl.shape.cluster == 1 && pl.waves > 1) {
    // several waves of single CTAs: the profile with more CTAs per SM, so
    // that one CTA's selections overlap the others' streams
    Plan pm = size_plan(ops, k, 1, 1);
    int resident = 0;
    e = ops.occupancy[1](pm.shape, &resident);
    if (e == cudaSuccess && resident > 0) {
      pm.waves = (num_segments + resident - 1) / resident;
      pl = pm;
    } else {
      (void)cudaGetLastError(); // keep the first profile
    }
  }
  std::lock_guard<std::mutex> lk(g_plan_mu);
  if (g_plans.size() > 4096)
    g_plans.clear();
  g_plans[key] = pl;
  *out = pl;
  return cudaSuccess;
}

int key_bytes_of(int dtype)
{
  switch (dtype) {
  case SEGTOPK_F16:
  case SEGTOPK_BF16: return 2;
  case SEGTOPK_F64: return 8;
  default: return 4;
  }
}

bool valid_pair(int det, int tie)
{
  if (tie == SEGTOPK_TIE_UNSPECIFIED)
    return true;
  return det == SEGTOPK_GPU_TO_GPU;
}

int validate(int dtype, const void* keys, const void* values, const int64_t* offsets,
             int64_t num_segments, int32_t k, int direction, int determinism, int tie_break,
             int ordering, const void* out_keys, const void* out_values, int64_t max_len,
             bool index_values = false)
{
  if (dtype < SEGTOPK_F16 || dtype > SEGTOPK_I32)
    return SEGTOPK_ERROR_INVALID_VALUE;
  if (direction != SEGTOPK_MAX && direction != SEGTOPK_MIN)
    return SEGTOPK_ERROR_INVALID_VALUE;
  if (determinism < SEGTOPK_NOT_GUARANTEED || determinism > SEGTOPK_GPU_TO_GPU)
    return SEGTOPK_ERROR_INVALID_VALUE;
  if (tie_break < SEGTOPK_TIE_UNSPECIFIED || tie_break > SEGTOPK_PREFER_LARGER_INDEX)
    return SEGTOPK_ERROR_INVALID_VALUE;
  if (ordering < SEGTOPK_UNSORTED || ordering > SEGTOPK_STABLE_SORTED)
    return SEGTOPK_ERROR_INVALID_VALUE;
  if (!valid_pair(determinism, tie_break))
    return SEGTOPK_ERROR_INVALID_COMBINATION;
  if (num_segments < 0 || k < 0)
    return SEGTOPK_ERROR_INVALID_VALUE;
  if (num_segments == 0 || k == 0)
    return SEGTOPK_SUCCESS;
  // out_values without values: only the host-buffer path's index mode
  if (!keys || !offsets || !out_keys || (values && !out_values) || (!values && out_values && !index_values))
    return SEGTOPK_ERROR_INVALID_VALUE;
  if (((uintptr_t)keys % (uintptr_t)key_bytes_of(dtype)) != 0)
    return SEGTOPK_ERROR_MISALIGNED;
  if (max_len > SEGTOPK_MAX_SEGMENT_LEN)
    return SEGTOPK_ERROR_NOT_SUPPORTED;
  if (k > SEGTOPK_MAX_K)
    return SEGTOPK_ERROR_NOT_SUPPORTED;
  if (num_segments > (int64_t)0x7fffffff / 16)
    return SEGTOPK_ERROR_NOT_SUPPORTED;
  return -1; // proceed
}

// The device-buffer call. With index_values, values may be null while
// out_values is not: out_values then receives each selected element's
// segment-local source index (the host-buffer path gathers the values
// itself).
int run_topk(segtopk_dtype key_dtype, const void* keys, const void* values, int value_bytes,
             const int64_t* segment_offsets, int64_t num_segments, int32_t k, segtopk_direction direction,
             segtopk_determinism determinism, segtopk_tie_break tie_break, segtopk_ordering ordering, void* out_keys,
             void* out_values, int64_t max_segment_len, const segtopk_options* options, void* stream,
             bool index_values)
{
  if (value_bytes != 4 && value_bytes != 8)
    return SEGTOPK_ERROR_INVALID_VALUE;
  t_last_launch_count = 0;
  int forced_width = 0;
  int32_t small_max = 0, team_max = 0;
  if (options) {
    for (int r : options->reserved)
      if (r != 0)
        return SEGTOPK_ERROR_INVALID_VALUE;
    if (options->cluster_width < 0 || options->cluster_width > 16)
      return SEGTOPK_ERROR_INVALID_VALUE;
    forced_width = options->cluster_width;
    small_max = options->small_segment_max_len;
    team_max = options->team_segment_max_len;
  }
  int v = validate(key_dtype, keys, values, segment_offsets, num_segments, k, direction, determinism,
                   tie_break, ordering, out_keys, out_values, max_segment_len, index_values);
  if (v >= 0)
    return v;
  DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess)
    return cuda_fail(e);
  if (dev.major != 10 || dev.minor != 3)
    return SEGTOPK_ERROR_DEVICE;
  cudaStream_t st = (cudaStream_t)stream;
  // Warp-select limits (k <= 32). With many segments, single warps for short
  // ones and the CTA path above (measured faster than teams there); with
  // fewer segments than SMs the latency of one segment sets the time, so
  // short segments take teams of eight warps and long ones the CTA path.
  const bool few = num_segments < (int64_t)dev.sms;
  if (small_max == 0)
    small_max = (forced_width > 0 || few) ? -1 : SEGTOPK_SMALL_SEGMENT_DEFAULT;
  if (team_max == 0)
    team_max = forced_width > 0 ? -1 : (few ? SEGTOPK_TEAM_SEGMENT_FEW : SEGTOPK_TEAM_SEGMENT_DEFAULT);
  if (k > kWarpPathMaxK)
    small_max = team_max = -1;
  const int64_t lim1 = small_max > 0 ? small_max : 0;                  // one warp: (0, lim1]
  const int64_t lim2 = team_max > 0 ? std::max<int64_t>(team_max, lim1) : lim1; // eight warps: (lim1, lim2]

  int64_t max_len = max_segment_len;
  if (max_len < 0) {
    // unknown bound: read the offsets back (synchronising)
    std::vector<int64_t> h((size_t)num_segments + 1);
    e = cudaMemcpyAsync(h.data(), segment_offsets, h.size() * sizeof(int64_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
      e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
      return cuda_fail(e);
    max_len = 0;
    for (int64_t s = 0; s < num_segments; ++s)
      max_len = std::max(max_len, h[(size_t)s + 1] - h[(size_t)s]);
    if (max_len > SEGTOPK_MAX_SEGMENT_LEN)
      return SEGTOPK_ERROR_NOT_SUPPORTED;
  }
  if (max_len <= 0)
    return SEGTOPK_SUCCESS;

  const KeyOps& ops = *ops_for(key_dtype);
  const uint64_t dirmask = (direction == SEGTOPK_MAX) ? ~0ull : 0ull;
  const uint64_t rank_mask = ops.rank_bits == 64 ? ~0ull : ((1ull << ops.rank_bits) - 1);
  // the CTA / cluster plan for segments beyond the warp-select limits, before
  // anything is launched (an unservable request launches nothing)
  const bool need_cta = max_len > lim2;
  Plan pl;
  if (need_cta) {
    bool unsupported = false;
    e = get_plan(key_dtype, ops, num_segments, max_len, k, forced_width, &pl, &unsupported);
    if (e != cudaSuccess)
      return cuda_fail(e);
    if (unsupported)
      return SEGTOPK_ERROR_NOT_SUPPORTED;
  }
  int launches = 0;
  for (int team = 0; team < 2; ++team) {
    // warp-select: segments in (lo, hi], one warp or eight warps each
    const int64_t lo = team ? lim1 : 0, hi = team ? lim2 : lim1;
    if (hi <= lo || max_len <= lo)
      continue;
    KernelParams w;
    std::memset(&w, 0, sizeof(w));
    w.keys = keys;
    w.values = values;
    w.offsets = segment_offsets;
    w.out_keys = out_keys;
    w.out_values = out_values;
    w.value_bytes = value_bytes;
    w.num_segments = num_segments;
    w.n_lo = lo;
    w.n_hi = std::min<int64_t>(hi, max_len);
    w.dirmask = dirmask & rank_mask;
    w.k = k;
    w.prefer_larger = (tie_break == SEGTOPK_PREFER_LARGER_INDEX) ? 1 : 0;
    w.sorted = (ordering != SEGTOPK_UNSORTED) ? 1 : 0;
    w.stable = (ordering == SEGTOPK_STABLE_SORTED) ? 1 : 0;
    w.tie_any = (determinism == SEGTOPK_NOT_GUARANTEED) ? 1 : 0;
    w.flag_overlong = max_len <= hi ? 1 : 0; // longer segments belong to a later launch
    e = ops.launch_warp[team](w, st);
    if (e != cudaSuccess)
      return cuda_fail(e);
    ++launches;
  }
  if (!need_cta) {
    t_last_launch_count = launches;
    return SEGTOPK_SUCCESS;
  }

  KernelParams p;
  std::memset(&p, 0, sizeof(p));
  p.keys = keys;
  p.values = values;
  p.offsets = segment_offsets;
  p.out_keys = out_keys;
  p.out_values = out_values;
  p.value_bytes = value_bytes;
  p.num_segments = num_segments;
  p.n_lo = lim2; // shorter segments took a warp-select path
  p.n_hi = max_len;
  p.dirmask = dirmask & rank_mask;
  p.k = k;
  p.list_cap = pl.list_cap;
  p.merge_gather = pl.merge_gather;
  // Speculative-bound sample: with one wave the slowest CTA sets the time, so
  // a larger sample (a steadier bound); with many waves the mean matters, so
  // a smaller one (less selection work per segment), except for 64-bit keys,
  // whose warp-minimum selection takes the larger sample at little extra
  // cost and keeps the candidate list about a fifth shorter.
  p.spec_keys = (pl.waves <= 1 || ops.rank_bits == 64) ? 2048u : 1024u;
  // Its margin, in standard deviations of the sample's share of the k best:
  // a slice whose bound proves too tight is read twice, which with one wave
  // sets the kernel's time (wide margin) and with many waves is averaged out
  // (narrower margin, shorter lists).
  // How: warp minimums (the exact target, cheap) with one wave and for 64-bit
  // ranks; digit passes that may stop with up to twice the target (suits
  // keys with many duplicates) for narrower keys over several waves. The
  // exact target wants the wider margin.
  p.spec_small = (pl.waves <= 1 || ops.rank_bits == 64) ? 1 : 0;
  p.spec_z = pl.waves <= 1 ? 4.0f : (p.spec_small ? 3.0f : 2.0f);
  p.spec_c = pl.waves <= 1 ? 3.0f : (p.spec_small ? 2.0f : 1.0f);
  p.ring_bytes = pl.ring_bytes;
  p.wait_limit = g_wait_limit;
  p.test_extra_tx = g_test_extra_tx;
  p.prefer_larger = (tie_break == SEGTOPK_PREFER_LARGER_INDEX) ? 1 : 0;
  p.sorted = (ordering != SEGTOPK_UNSORTED) ? 1 : 0;
  p.stable = (ordering == SEGTOPK_STABLE_SORTED) ? 1 : 0;
  p.tie_any = (determinism == SEGTOPK_NOT_GUARANTEED) ? 1 : 0;
  p.flag_overlong = 1;
  e = ops.launch[pl.shape.profile](p, pl.shape, st);
  if (e != cudaSuccess)
    return cuda_fail(e);
  t_last_launch_count = launches + 1;
  return SEGTOPK_SUCCESS;
}

} // namespace

// Records a failed CUDA call for segtopk_last_cuda_error on this thread (for
// the library's other translation units); returns SEGTOPK_ERROR_CUDA.
int record_cuda_error(cudaError_t e) { return cuda_fail(e); }

} // namespace segtopk

using namespace segtopk;

extern "C" int segtopk_batched_topk_ex(segtopk_dtype key_dtype, const void* keys, const int32_t* values,
                                       const int64_t* segment_offsets, int64_t num_segments, int32_t k,
                                       segtopk_direction direction, segtopk_determinism determinism,
                                       segtopk_tie_break tie_break, segtopk_ordering ordering,
                                       void* out_keys, int32_t* out_values, int64_t max_segment_len,
                                       const segtopk_options* options, void* stream)
{
  return run_topk(key_dtype, keys, values, 4, segment_offsets, num_segments, k, direction, determinism, tie_break,
                  ordering, out_keys, out_values, max_segment_len, options, stream, false);
}

extern "C" int segtopk_batched_topk_values(segtopk_dtype key_dtype, const void* keys, const void* values,
                                           int32_t value_bytes, const int64_t* segment_offsets,
                                           int64_t num_segments, int32_t k, segtopk_direction direction,
                                           segtopk_determinism determinism, segtopk_tie_break tie_break,
                                           segtopk_ordering ordering, void* out_keys, void* out_values,
                                           int64_t max_segment_len, const segtopk_options* options, void* stream)
{
  t_last_launch_count = 0;
  if (values && value_bytes != 4 && value_bytes != 8)
    return SEGTOPK_ERROR_INVALID_VALUE;
  return run_topk(key_dtype, keys, values, values ? value_bytes : 4, segment_offsets, num_segments, k, direction,
                  determinism, tie_break, ordering, out_keys, out_values, max_segment_len, options, stream, false);
}

extern "C" int segtopk_batched_topk(segtopk_dtype key_dtype, const void* keys, const int32_t* values,
                                    const int64_t* segment_offsets, int64_t num_segments, int32_t k,
                                    segtopk_direction direction, segtopk_determinism determinism,
                                    segtopk_tie_break tie_break, segtopk_ordering ordering,
                                    void* out_keys, int32_t* out_values, int64_t max_segment_len,
                                    void* stream)
{
  return segtopk_batched_topk_ex(key_dtype, keys, values, segment_offsets, num_segments, k, direction,
                                 determinism, tie_break, ordering, out_keys, out_values, max_segment_len,
                                 nullptr, stream);
}

namespace {
size_t ws_align(size_t x) { return (x + 255) & ~(size_t)255; }
} // namespace

namespace segtopk {
int host_offsets_scan(const int64_t* offsets, int64_t num_segments, int64_t* num_keys, int64_t* max_len)
{
  int64_t nk = 0, ml = 0;
  for (int64_t s = 0; s <= num_segments; ++s)
    if (offsets[s] < 0)
      return SEGTOPK_ERROR_INVALID_VALUE;
  for (int64_t s = 0; s < num_segments; ++s) {
    nk = std::max(nk, offsets[s + 1]);
    ml = std::max(ml, offsets[s + 1] - offsets[s]);
  }
  if ((uint64_t)nk > (uint64_t)(SIZE_MAX / 16))
    return SEGTOPK_ERROR_INVALID_VALUE;
  *num_keys = nk;
  *max_len = ml;
  return SEGTOPK_SUCCESS;
}
} // namespace segtopk

extern "C" size_t segtopk_host_workspace_bytes(segtopk_dtype key_dtype, int has_values, int64_t num_keys,
                                               int64_t num_segments, int32_t k)
{
  if (num_keys < 0 || num_segments < 0 || k < 0 || (uint64_t)num_keys > (uint64_t)(SIZE_MAX / 16) ||
      num_segments > (int64_t)0x7fffffff)
    return 0;
  const size_t kb = (size_t)key_bytes_of(key_dtype);
  // keys, offsets, output keys and, for pairs, the selected source indices
  size_t b = ws_align((size_t)num_keys * kb) + ws_align((size_t)(num_segments + 1) * 8) +
             ws_align((size_t)num_segments * (size_t)k * kb);
  if (has_values)
    b += ws_align((size_t)num_segments * (size_t)k * 4);
  return b;
}

extern "C" int segtopk_batched_topk_host(segtopk_dtype key_dtype, const void* keys, const int32_t* values,
                                         const int64_t* segment_offsets, int64_t num_segments, int32_t k,
                                         segtopk_direction direction, segtopk_determinism determinism,
                                         segtopk_tie_break tie_break, segtopk_ordering ordering,
                                         void* out_keys, int32_t* out_values, int64_t max_segment_len,
                                         void* device_workspace, size_t workspace_bytes, void* stream)
{
  t_last_launch_count = 0;
  (void)max_segment_len; // the host reads its own offsets: the true longest segment is known
  int v = validate(key_dtype, keys ? (const void*)16 : nullptr, values, segment_offsets, num_segments, k,
                   direction, determinism, tie_break, ordering, out_keys, out_values, -1);
  if (v >= 0)
    return v;
  if (!device_workspace)
    return SEGTOPK_ERROR_INVALID_VALUE;
  if (((uintptr_t)device_workspace & 255u) != 0)
    return SEGTOPK_ERROR_MISALIGNED;
  int64_t num_keys = 0, max_len = 0;
  v = host_offsets_scan(segment_offsets, num_segments, &num_keys, &max_len);
  if (v != SEGTOPK_SUCCESS)
    return v;
  if (max_len > SEGTOPK_MAX_SEGMENT_LEN)
    return SEGTOPK_ERROR_NOT_SUPPORTED;
  const size_t need = segtopk_host_workspace_bytes(key_dtype, values != nullptr, num_keys, num_segments, k);
  if (need == 0 || workspace_bytes < need)
    return SEGTOPK_ERROR_INVALID_VALUE;
  const size_t kb = (size_t)key_bytes_of(key_dtype);
  const size_t slots = (size_t)num_segments * (size_t)k;
  char* w = (char*)device_workspace;
  void* d_keys = w;
  w += ws_align((size_t)num_keys * kb);
  int64_t* d_offs = (int64_t*)w;
  w += ws_align((size_t)(num_segments + 1) * 8);
  void* d_out_keys = w;
  w += ws_align(slots * kb);
  int32_t* d_out_idx = values ? (int32_t*)w : nullptr;
  // Only keys and offsets travel to the device: the kernel writes each
  // selected element's segment-local source index, and the values are
  // gathered here from the caller's host array.
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(d_keys, keys, (size_t)num_keys * kb, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(d_offs, segment_offsets, (size_t)(num_segments + 1) * 8, cudaMemcpyHostToDevice, st);
  // slots past a short segment's length keep the caller's host contents
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(d_out_keys, out_keys, slots * kb, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess && values)
    e = cudaMemcpyAsync(d_out_idx, out_values, slots * 4, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess)
    return cuda_fail(e);
  int rc = run_topk(key_dtype, d_keys, nullptr, 4, d_offs, num_segments, k, direction, determinism, tie_break,
                    ordering, d_out_keys, d_out_idx, max_len, nullptr, stream, true);
  if (rc != SEGTOPK_SUCCESS)
    return rc;
  const int launches = t_last_launch_count;
  e = cudaMemcpyAsync(out_keys, d_out_keys, slots * kb, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && values)
    e = cudaMemcpyAsync(out_values, d_out_idx, slots * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaStreamSynchronize(st);
  if (e != cudaSuccess)
    return cuda_fail(e);
  if (values) {
    // written slots hold source indices: replace them by the values
    for (int64_t s = 0; s < num_segments; ++s) {
      const int64_t b = segment_offsets[s];
      const int64_t n = std::max<int64_t>(segment_offsets[s + 1] - b, 0);
      const int64_t m = std::min<int64_t>(n, k);
      int32_t* ov = out_values + (size_t)s * (size_t)k;
      for (int64_t j = 0; j < m; ++j) {
        const int64_t i = ov[j];
        if (i < 0 || i >= n)
          return SEGTOPK_ERROR_DEVICE; // cannot happen: the kernel writes indices of the segment
        ov[j] = values[b + i];
      }
    }
  }
  t_last_launch_count = launches;
  return SEGTOPK_SUCCESS;
}

extern "C" const char* segtopk_status_string(int status)
{
  switch (status) {
  case SEGTOPK_SUCCESS: return "success";
  case SEGTOPK_ERROR_INVALID_VALUE: return "invalid argument value";
  case SEGTOPK_ERROR_INVALID_COMBINATION: return "determinism / tie_break combination not allowed";
  case SEGTOPK_ERROR_NOT_SUPPORTED: return "request outside the supported limits";
  case SEGTOPK_ERROR_MISALIGNED: return "keys pointer is not aligned to its element size";
  case SEGTOPK_ERROR_CUDA: return "CUDA runtime error";
  case SEGTOPK_ERROR_DEVICE: return "unsupported device (needs sm_103)";
  default: return "unknown status";
  }
}

extern "C" int segtopk_last_cuda_error(void) { return t_last_cuda_error; }

extern "C" int segtopk_last_launch_count(void) { return t_last_launch_count; }

extern "C" int segtopk_read_device_error(uint32_t* error_word)
{
  if (!error_word)
    return SEGTOPK_ERROR_INVALID_VALUE;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess)
    return cuda_fail(e);
  uint32_t all = 0;
  const KeyOps* list[] = {&key_ops_f16(), &key_ops_bf16(), &key_ops_f32(),
                          &key_ops_f64(), &key_ops_u32(), &key_ops_i32()};
  for (const KeyOps* o : list) {
    uint32_t w = 0;
    e = o->read_error(&w);
    if (e != cudaSuccess)
      return cuda_fail(e);
    all |= w;
  }
  *error_word = all;
  return SEGTOPK_SUCCESS;
}

extern "C" int segtopk_read_stats(uint64_t* out, int n)
{
  if (!out || n < 0)
    return SEGTOPK_ERROR_INVALID_VALUE;
#ifndef SEGTOPK_STATS
  return SEGTOPK_ERROR_NOT_SUPPORTED;
#else
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess)
    return cuda_fail(e);
  unsigned long long sum[kStatCount] = {};
  const KeyOps* list[] = {&key_ops_f16(), &key_ops_bf16(), &key_ops_f32(),
                          &key_ops_f64(), &key_ops_u32(), &key_ops_i32()};
  for (const KeyOps* o : list) {
    e = o->read_stats(sum);
    if (e != cudaSuccess)
      return cuda_fail(e);
  }
  for (int i = 0; i < n; ++i)
    out[i] = i < kStatCount ? (uint64_t)sum[i] : 0u;
  return SEGTOPK_SUCCESS;
#endif
}

extern "C" int segtopk_set_test_hooks(long long wait_limit_cycles, uint32_t first_copy_extra_bytes)
{
#ifndef SEGTOPK_TEST_HOOKS
  (void)wait_limit_cycles;
  (void)first_copy_extra_bytes;
  return SEGTOPK_ERROR_NOT_SUPPORTED;
#else
  if (wait_limit_cycles <= 0 || (first_copy_extra_bytes & 15u) != 0 || first_copy_extra_bytes > 4096u)
    return SEGTOPK_ERROR_INVALID_VALUE;
  g_wait_limit = wait_limit_cycles;
  g_test_extra_tx = first_copy_extra_bytes;
  return SEGTOPK_SUCCESS;
#endif
}

extern "C" int segtopk_test_device_prep(int n, const int* devices, const uint32_t* smem_bytes,
                                        const int* cluster_widths, uint32_t* actions)
{
#ifndef SEGTOPK_TEST_HOOKS
  (void)n;
  (void)devices;
  (void)smem_bytes;
  (void)cluster_widths;
  (void)actions;
  return SEGTOPK_ERROR_NOT_SUPPORTED;
#else
  if (n < 0 || (n > 0 && (!devices || !smem_bytes || !cluster_widths || !actions)))
    return SEGTOPK_ERROR_INVALID_VALUE;
  // one fresh record per kernel kind, every attribute call taken to succeed
  DevicePrep stream_rec, warp_rec;
  for (int i = 0; i < n; ++i) {
    const int dev = devices[i];
    if (!DevicePrep::valid(dev)) {
      actions[i] = ~0u;
      continue;
    }
    if (cluster_widths[i] <= 0) { // a warp-kernel launch
      const uint32_t need = warp_rec.warp_needs(dev);
      if (need)
        warp_rec.warp_done(dev);
      actions[i] = need;
    } else {
      const uint32_t need = stream_rec.stream_needs(dev, smem_bytes[i], cluster_widths[i]);
      stream_rec.stream_done(dev, smem_bytes[i], need);
      actions[i] = need;
    }
  }
  return SEGTOPK_SUCCESS;
#endif
}

// ---------------------------------------------------------------------------
// Top-k over one array (no segments): two passes of the segmented selection.
// Pass 1 splits the array into `pieces` balanced contiguous pieces and
// writes each piece's k best, stably sorted, into the workspace; pass 2
// selects the k best of those pieces * k candidates. Every key of the array
// that is among its k best is among its piece's k best, so pass 2 sees all
// of them; and since each piece's candidates keep equal keys in source-index
// order and pieces follow one another in source order, a candidate's
// position orders equal keys as their array index does -- pass 2's tie-break
// and stable order are the array's.
// ---------------------------------------------------------------------------
namespace segtopk {
namespace topk_detail {
// Offsets of pass 1's balanced pieces and of pass 2's single segment.
__global__ void fill_piece_offsets(int64_t* offs, int64_t pieces, int64_t n, int64_t* offs2, int64_t candidates)
{
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t q = n / pieces, r = n % pieces;
  if (i <= pieces)
    offs[i] = i * q + (i < r ? i : r);
  if (i == 0) {
    offs2[0] = 0;
    offs2[1] = candidates;
  }
}
} // namespace topk_detail
} // namespace segtopk

namespace {

// Pieces of pass 1 for n keys: each at least max(65536, 16 k) keys, at most
// 304 of them (one wave of two CTAs on each of the 152 SMs).
int64_t topk_pieces(int64_t n, int32_t k)
{
  const int64_t min_piece = std::max<int64_t>(65536, 16 * (int64_t)k);
  return std::max<int64_t>(1, std::min<int64_t>(304, n / min_piece));
}

struct TopkLayout {
  int64_t pieces;
  size_t offs, offs2, ckeys, cvals, total;
};

TopkLayout topk_layout(int dtype, int32_t value_bytes, int64_t n, int32_t k)
{
  TopkLayout t;
  t.pieces = topk_pieces(n, k);
  const size_t cand = (size_t)t.pieces * (size_t)k;
  t.offs = 0;
  t.offs2 = ws_align((size_t)(t.pieces + 1) * 8);
  t.ckeys = t.offs2 + ws_align(16);
  t.cvals = t.ckeys + ws_align(cand * (size_t)key_bytes_of(dtype));
  t.total = t.cvals + (value_bytes ? ws_align(cand * (size_t)value_bytes) : 0);
  return t;
}

} // namespace

extern "C" size_t segtopk_topk_workspace_bytes(segtopk_dtype key_dtype, int32_t value_bytes, int64_t num_keys,
                                               int32_t k)
{
  if (num_keys < 0 || k < 0 || (value_bytes != 0 && value_bytes != 4 && value_bytes != 8) ||
      key_dtype < SEGTOPK_F16 || key_dtype > SEGTOPK_I32)
    return 0;
  return topk_layout(key_dtype, value_bytes, num_keys, k).total;
}

extern "C" int segtopk_topk(segtopk_dtype key_dtype, const void* keys, const void* values, int32_t value_bytes,
                            int64_t num_keys, int32_t k, segtopk_direction direction,
                            segtopk_determinism determinism, segtopk_tie_break tie_break,
                            segtopk_ordering ordering, void* out_keys, void* out_values, void* workspace,
                            size_t workspace_bytes, void* stream)
{
  t_last_launch_count = 0;
  if (num_keys < 0 || (values && value_bytes != 4 && value_bytes != 8) || (!values != !out_values))
    return SEGTOPK_ERROR_INVALID_VALUE;
  const int vb = values ? value_bytes : 4;
  // the rest of the argument checks are the segmented call's (one segment)
  int v = validate(key_dtype, keys, values, workspace ? (const int64_t*)workspace : nullptr, 1, k, direction,
                   determinism, tie_break, ordering, out_keys, out_values, 0);
  if (v >= 0)
    return v;
  if (num_keys == 0)
    return SEGTOPK_SUCCESS;
  if (((uintptr_t)workspace & 255u) != 0)
    return SEGTOPK_ERROR_MISALIGNED;
  const TopkLayout t = topk_layout(key_dtype, values ? value_bytes : 0, num_keys, k);
  if (workspace_bytes < t.total)
    return SEGTOPK_ERROR_INVALID_VALUE;
  if ((num_keys + t.pieces - 1) / t.pieces > SEGTOPK_MAX_SEGMENT_LEN)
    return SEGTOPK_ERROR_NOT_SUPPORTED;
  char* w = (char*)workspace;
  int64_t* offs = (int64_t*)(w + t.offs);
  int64_t* offs2 = (int64_t*)(w + t.offs2);
  void* ckeys = w + t.ckeys;
  void* cvals = values ? (void*)(w + t.cvals) : nullptr;
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t cand = t.pieces * (int64_t)k;
  segtopk::topk_detail::fill_piece_offsets<<<(unsigned)((t.pieces + 1 + 255) / 256), 256, 0, st>>>(offs, t.pieces, num_keys, offs2, cand);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return cuda_fail(e);
  if (t.pieces == 1) {
    const int rc = run_topk(key_dtype, keys, values, vb, offs, 1, k, direction, determinism, tie_break, ordering,
                            out_keys, out_values, num_keys, nullptr, stream, false);
    if (rc == SEGTOPK_SUCCESS)
      t_last_launch_count += 1;
    return rc;
  }
  // pass 1: every piece's k best, stably sorted (any order when any ties will do)
  const segtopk_ordering order1 = determinism == SEGTOPK_NOT_GUARANTEED ? SEGTOPK_UNSORTED : SEGTOPK_STABLE_SORTED;
  int rc = run_topk(key_dtype, keys, values, vb, offs, t.pieces, k, direction, determinism, tie_break, order1,
                    ckeys, cvals, (num_keys + t.pieces - 1) / t.pieces, nullptr, stream, false);
  if (rc != SEGTOPK_SUCCESS)
    return rc;
  const int launches1 = t_last_launch_count;
  // pass 2: the k best of the candidates
  rc = run_topk(key_dtype, ckeys, cvals, vb, offs2, 1, k, direction, determinism, tie_break, ordering, out_keys,
                out_values, cand, nullptr, stream, false);
  if (rc != SEGTOPK_SUCCESS)
    return rc;
  t_last_launch_count += launches1 + 1;
  return SEGTOPK_SUCCESS;
}
