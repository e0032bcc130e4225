// Host-side launch interface between the C ABI (api.cu) and the two kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include "mfr_device.cuh"

namespace mfr {

constexpr int kStreamMaxThreads = 544;   // a routing warp + up to 16 compute warps
constexpr int kClusterMaxThreads = 512;  // R groups of SV threads
constexpr int kStreamSlots = 12;         // row slots in the stream kernel's shared-memory ring
constexpr int kStreamLists = 4;          // row lists (tokens) in its routing ring
constexpr int kStreamColumns = 2;        // 16-byte columns per compute thread per hidden pass

struct LaunchGeom {
  int grid;
  int block;
  int cluster;
  int smem;
  int smem_optin;  // the device's opt-in maximum of dynamic shared memory per block
};

cudaError_t launch_cluster_kernel(int act_dtype, const KParams& p, const LaunchGeom& g, cudaStream_t stream);
int cluster_kernel_max_active_clusters(int act_dtype, int K, const LaunchGeom& g);
cudaError_t launch_stream_kernel(int act_dtype, const KParams& p, const LaunchGeom& g, cudaStream_t stream);
int stream_kernel_blocks_per_sm(int act_dtype, const LaunchGeom& g);
cudaError_t read_and_reset_timeouts(unsigned int* count);

}  // namespace mfr
