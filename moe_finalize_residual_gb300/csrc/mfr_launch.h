// Host-side launch interface between the C ABI (api.cu) and the two kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include "mfr_device.cuh"

namespace mfr {

// Stream kernel shape (probe builds may override the defaults): a routing warp and kStreamGroups
// groups of compute warps, each group running its own stream of tokens.
#ifndef MFR_STREAM_GROUPS
#define MFR_STREAM_GROUPS 2
#endif
#ifndef MFR_STREAM_GROUP_WARPS
#define MFR_STREAM_GROUP_WARPS 7
#endif
#ifndef MFR_STREAM_COLUMNS
#define MFR_STREAM_COLUMNS 4
#endif
#ifndef MFR_STREAM_SLOTS
#define MFR_STREAM_SLOTS 6
#endif
constexpr int kStreamGroups = MFR_STREAM_GROUPS;
constexpr int kStreamGroupWarps = MFR_STREAM_GROUP_WARPS;
constexpr int kStreamMaxThreads = 32 * (1 + MFR_STREAM_GROUPS * MFR_STREAM_GROUP_WARPS);
constexpr int kStreamSlots = MFR_STREAM_SLOTS;      // row slots per group in shared memory
constexpr int kStreamLists = 4;                     // row lists (tokens) in the routing ring
constexpr int kStreamColumns = MFR_STREAM_COLUMNS;  // 16-byte columns per compute thread per hidden pass
static_assert(kStreamLists % kStreamGroups == 0, "a list slot must return to the group that used it");
static_assert(kStreamGroups == 1 || kStreamGroups == 2, "the stream kernel is built for one or two groups");
constexpr int kClusterMaxThreads = 512;             // R groups of SV threads
// Bulk-copy streaming kernel: a routing warp, a copy warp and 8 to kBulkMaxComputeWarps compute warps
// (the planner's choice per row width).
constexpr int kBulkMaxComputeWarps = 14;
constexpr int kBulkMaxColumns = 4;                  // 16-byte columns per compute thread per pass


struct LaunchGeom {
  int grid;
  int block;
  int cluster;
  int smem;
  int smem_optin;  // the device's opt-in maximum of dynamic shared memory per block
};

cudaError_t launch_cluster_kernel(int act_dtype, const KParams& p, const LaunchGeom& g, cudaStream_t stream);
// Cluster kernel forms: 8 routes in flight per thread with the register budget of two 512-thread CTAs
// per SM (plans that loop over chunks); 8 in flight with a wider register budget (one-chunk plans, whose
// CTAs are small); 16 in flight.
// The latency form is the one-chunk form with the route entries held in registers and branch-free
// predicated row loads, for grids that put at most 256 gathering threads on an SM.
// The split form (one chunk, top-k > 8) spreads each partial's routes over several thread groups.
enum ClusterForm {
  kClusterForm8 = 0,
  kClusterForm8OneChunk = 1,
  kClusterForm16 = 2,
  kClusterForm8Latency = 3,
  kClusterForm8Split = 4
};
int cluster_kernel_max_active_clusters(int act_dtype, int form, const LaunchGeom& g);
int cluster_kernel_blocks_per_sm(int act_dtype, int form, const LaunchGeom& g);
cudaError_t launch_stream_kernel(int act_dtype, const KParams& p, const LaunchGeom& g, cudaStream_t stream);
int stream_kernel_blocks_per_sm(int act_dtype, int groups, const LaunchGeom& g);
cudaError_t launch_bulk_kernel(int act_dtype, const KParams& p, const LaunchGeom& g, cudaStream_t stream);
int bulk_kernel_blocks_per_sm(int act_dtype, int cols_per_thread, const LaunchGeom& g);
cudaError_t read_and_reset_timeouts(unsigned int* count);
cudaError_t read_and_reset_bulk_timeouts(unsigned int* count);
cudaError_t read_and_reset_cluster_timeouts(unsigned int* count);

}  // namespace mfr
