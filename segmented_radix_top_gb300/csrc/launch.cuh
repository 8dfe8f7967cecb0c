// Launch helpers shared by the per-key-type translation units.
#pragma once

#include <mutex>

#include "device_prep.h"
#include "dispatch.h"
#include "stream_topk.cuh"
#include "warp_topk.cuh"

namespace segtopk {

template <KeyKind KK, int NT, class PR>
struct StreamLauncher {
  static cudaError_t prepare(uint32_t smem, int cluster)
  {
    // Raise the dynamic shared-memory opt-in lazily, only as far as needed,
    // on the current device.
    static DevicePrep st;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
      return e;
    if (!DevicePrep::valid(dev))
      return cudaErrorInvalidDevice;
    auto fn = stream_topk_kernel<KK, NT, PR>;
    std::lock_guard<std::mutex> lk(st.mu);
    const uint32_t need = st.stream_needs(dev, smem, cluster);
    if (need & DevicePrep::kRaiseSmem) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess)
        return e;
      st.stream_done(dev, smem, DevicePrep::kRaiseSmem);
    }
    if (need & DevicePrep::kNonPortable) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess)
        return e;
      st.stream_done(dev, smem, DevicePrep::kNonPortable);
    }
    return cudaSuccess;
  }

  static void config(const LaunchShape& s, int64_t num_segments, cudaLaunchConfig_t& cfg,
                     cudaLaunchAttribute* attr)
  {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = dim3((unsigned)(num_segments * s.cluster), 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = s.smem;
    cfg.numAttrs = 0;
    cfg.attrs = attr;
    if (s.cluster > 1) {
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)s.cluster;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.numAttrs = 1;
    }
  }

  static cudaError_t launch(const KernelParams& p, const LaunchShape& s, cudaStream_t stream)
  {
    cudaError_t e = prepare(s.smem, s.cluster);
    if (e != cudaSuccess)
      return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    config(s, p.num_segments, cfg, attr);
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, stream_topk_kernel<KK, NT, PR>, p);
  }

  static cudaError_t occupancy(const LaunchShape& s, int* resident)
  {
    cudaError_t e = prepare(s.smem, s.cluster);
    if (e != cudaSuccess)
      return e;
    if (s.cluster <= 1) {
      int per_sm = 0, dev = 0, sms = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stream_topk_kernel<KK, NT, PR>, NT, s.smem);
      if (e != cudaSuccess)
        return e;
      e = cudaGetDevice(&dev);
      if (e != cudaSuccess)
        return e;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      *resident = per_sm * sms;
      return e;
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    config(s, s.cluster, cfg, attr);
    return cudaOccupancyMaxActiveClusters(resident, stream_topk_kernel<KK, NT, PR>, &cfg);
  }
};

template <KeyKind KK, int W>
struct WarpLauncher {
  static cudaError_t launch(const KernelParams& p, cudaStream_t stream)
  {
    // Static shared memory only: ask for the largest shared-memory carveout,
    // so that the occupancy the launch bounds allow (32 one-warp CTAs, or four
    // eight-warp CTAs, per SM) is not cut by a small default carveout.
    static DevicePrep st;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
      return e;
    if (!DevicePrep::valid(dev))
      return cudaErrorInvalidDevice;
    {
      std::lock_guard<std::mutex> lk(st.mu);
      if (st.warp_needs(dev) & DevicePrep::kCarveout) {
        e = cudaFuncSetAttribute(warp_topk_kernel<KK, W>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
          return e;
        st.warp_done(dev);
      }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.num_segments, 1, 1); // one segment per CTA
    cfg.blockDim = dim3(32 * W, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, warp_topk_kernel<KK, W>, p);
  }
};

// Both readers below have internal linkage: each translation unit reads its
// own device words (an inline function would be merged across units).
static inline cudaError_t read_and_clear(uint32_t* word)
{
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(word, g_device_error, sizeof(uint32_t));
  if (e != cudaSuccess)
    return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(uint32_t));
}

// Adds this translation unit's statistics counters to out[0, kStatCount)
// and clears them (synchronous).
static inline cudaError_t read_and_clear_stats(unsigned long long* out)
{
  unsigned long long h[kStatCount] = {}, zero[kStatCount] = {};
  cudaError_t e = cudaMemcpyFromSymbol(h, g_stats, sizeof(h));
  if (e != cudaSuccess)
    return e;
  for (int i = 0; i < kStatCount; ++i)
    out[i] += h[i];
  return cudaMemcpyToSymbol(g_stats, zero, sizeof(zero));
}

} // namespace segtopk

#define SEGTOPK_DEFINE_KEY_OPS(NAME, KIND)                                                         \
  namespace segtopk {                                                                              \
  const KeyOps& key_ops_##NAME()                                                                   \
  {                                                                                                \
    static const KeyOps ops = {(int)sizeof(KeyTraits<KIND>::Raw),                                 \
                               KeyTraits<KIND>::kRankBits,                                         \
                               {&StreamLauncher<KIND, kCtaThreads, ProfileLong>::launch,           \
                                &StreamLauncher<KIND, kCtaThreads, ProfileMany>::launch},          \
                               {&WarpLauncher<KIND, 1>::launch, &WarpLauncher<KIND, kWarpTeam>::launch}, \
                               {&StreamLauncher<KIND, kCtaThreads, ProfileLong>::occupancy,        \
                                &StreamLauncher<KIND, kCtaThreads, ProfileMany>::occupancy},       \
                               &read_and_clear,                                                    \
                               &read_and_clear_stats};                                             \
    return ops;                                                                                    \
  }                                                                                                \
  }
