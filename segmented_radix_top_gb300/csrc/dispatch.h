// Host-side interface between the C ABI (api.cu) and the per-key-type kernel
// translation units (inst_*.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace segtopk {

struct KernelParams;

struct LaunchShape {
  int threads;        // CTA size
  int cluster;        // CTAs per segment (1 = plain launch)
  uint32_t smem;      // dynamic shared memory bytes
  int profile;        // kernel profile: 0 long segments, 1 many single-CTA segments
};

constexpr int kProfiles = 2;

// Entry points every key-type translation unit provides.
struct KeyOps {
  int key_bytes;
  int rank_bits;
  // Launch the segment kernel (profile s.profile) over all num_segments segments.
  cudaError_t (*launch[kProfiles])(const KernelParams& p, const LaunchShape& s, cudaStream_t stream);
  // Launch the warp-select kernel (k <= 32) over all num_segments segments,
  // one warp per segment ([0]) or a team of eight warps per segment ([1]); it
  // serves those with p.n_lo < n <= p.n_hi.
  cudaError_t (*launch_warp[2])(const KernelParams& p, cudaStream_t stream);
  // Resident clusters (cluster > 1) or resident CTAs (cluster == 1) per GPU.
  cudaError_t (*occupancy[kProfiles])(const LaunchShape& s, int* resident);
  // Read and clear this translation unit's device error word (synchronous).
  cudaError_t (*read_error)(uint32_t* word);
  // Add this translation unit's statistics counters to out[0, 16) and clear
  // them (synchronous; counted only by the statistics build).
  cudaError_t (*read_stats)(unsigned long long* out);
};

const KeyOps& key_ops_f16();
const KeyOps& key_ops_bf16();
const KeyOps& key_ops_f32();
const KeyOps& key_ops_f64();
const KeyOps& key_ops_u32();
const KeyOps& key_ops_i32();

// Records a failed CUDA call for segtopk_last_cuda_error; returns SEGTOPK_ERROR_CUDA.
int record_cuda_error(cudaError_t e);

// Host-side check of a host offsets array (host-buffer entry points): every
// offset non-negative and the addressed key count small enough for byte
// arithmetic. Gives the number of keys addressed (the largest segment end)
// and the longest segment. Returns a status code.
int host_offsets_scan(const int64_t* offsets, int64_t num_segments, int64_t* num_keys, int64_t* max_len);

} // namespace segtopk
