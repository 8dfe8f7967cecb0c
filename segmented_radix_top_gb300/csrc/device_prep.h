// Per-device launch preparation of one kernel (host code).
//
// Function attributes -- the dynamic shared-memory opt-in, the permission
// for non-portable cluster sizes, the shared-memory carveout -- belong to
// each device's copy of a kernel, so a process that drives several GPUs
// must set them once per device. This records, per device ordinal and under
// a lock held by the caller, which ones were set; the launchers ask what a
// launch still needs, make those CUDA calls, and record the ones that
// succeeded. The decisions are plain host logic, so the instrumented build
// exports a replay of them for host tests.
#pragma once

#include <cstdint>
#include <mutex>

namespace segtopk {

struct DevicePrep {
  static constexpr int kMaxDevices = 64;
  // actions a launch may need
  static constexpr uint32_t kRaiseSmem = 1u;   // raise the dynamic shared-memory opt-in
  static constexpr uint32_t kNonPortable = 2u; // allow clusters wider than 8
  static constexpr uint32_t kCarveout = 4u;    // prefer the largest shared-memory carveout

  std::mutex mu;
  uint32_t granted[kMaxDevices] = {};
  bool nonportable[kMaxDevices] = {};
  bool prepared[kMaxDevices] = {};

  static bool valid(int dev) { return dev >= 0 && dev < kMaxDevices; }

  // Segment kernel: what a launch with `smem` bytes of dynamic shared memory
  // and clusters of `cluster` CTAs still needs on device `dev`.
  uint32_t stream_needs(int dev, uint32_t smem, int cluster) const
  {
    uint32_t a = 0;
    if (smem > granted[dev])
      a |= kRaiseSmem;
    if (cluster > 8 && !nonportable[dev])
      a |= kNonPortable;
    return a;
  }
  void stream_done(int dev, uint32_t smem, uint32_t done)
  {
    if (done & kRaiseSmem)
      granted[dev] = smem;
    if (done & kNonPortable)
      nonportable[dev] = true;
  }

  // Warp kernel: the carveout, once per device.
  uint32_t warp_needs(int dev) const { return prepared[dev] ? 0u : kCarveout; }
  void warp_done(int dev) { prepared[dev] = true; }
};

} // namespace segtopk
