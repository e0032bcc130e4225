// Small-batch fused finalize: one thread-block cluster per token, the hidden dimension split into
// equal slices, one slice per CTA of the cluster.
//
// Design (prior art: flashinfer PR #6546, finalizeKernelSmallBatch, Description -- one CTA per
// (token, hidden slice), 128-bit loads, top-K split over thread groups with a shared-memory combine,
// PDL trigger at kernel start; flashinfer PR #6631, Description -- load the indices and scales of
// the routes first, then all rows, so the row loads are in flight together):
//
//  1. trigger dependents; read every slot's route index and scale into shared memory (before the
//     dependency wait only when the caller says the routing is already complete);
//  2. wait for the preceding kernel (PDL), then issue EVERY gathered row slice of EVERY partial as
//     16-byte cp.async copies at once: all R*K routes and R shared rows of the token are in flight
//     together, spread over all threads (this is the top-K split over thread groups);
//  3. each thread owns 4 consecutive hidden elements and runs the FP32 fused multiply-add chain over
//     the staged rows in route order (the shared-memory combine; the order is the definition's, so
//     every partial's rounded row is bit-identical to a sequential evaluation);
//  4. rank sum, residual add, sum of squares; the sum of squares is reduced with warp shuffles, then
//     across warps in shared memory, then across the cluster's CTAs through distributed shared memory
//     in CTA-rank order, so every CTA gets the same deterministic total;
//  5. RMSNorm output and the quantisation epilogue.
//
// No CTA waits on a flag in global memory; the only cross-CTA synchronisation is the hardware
// cluster barrier, which every CTA reaches unconditionally.
#include "mfr_device.cuh"
#include "mfr_launch.h"

namespace mfr {

// Build this CTA's slot table for token t: the global source of every staged row, and the
// (offset, scale) table the arithmetic reads.  Slot s is staged at byte s * stride.
__device__ __forceinline__ void load_slots(const KParams& p, int t, int stride, const uint8_t** slot_src,
                                           int2* meta, int* sh_off, int tid, int nthreads) {
  for (int s = tid; s < p.nslots; s += nthreads) {
    const SlotSource o = slot_source(p, s, t);
    slot_src[s] = o.src;
    if (o.k >= 0)
      meta[o.r * p.K + o.k] = make_int2(o.src ? s * stride : -1, __float_as_int(o.scale));
    else
      sh_off[o.r] = s * stride;
  }
  for (int r = tid; r < p.R; r += nthreads)
    if (!((p.shared_mask >> r) & 1u)) sh_off[r] = -1;
}

template <typename A, int RMAX>
__global__ void __launch_bounds__(1024, 1) cluster_finalize_kernel(const __grid_constant__ KParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int nthreads = blockDim.x;
  const uint32_t C = cluster_nctarank();
  const uint32_t crank = cluster_ctarank();
  const int t = static_cast<int>(blockIdx.x / C);
  const int H = p.H;
  const int nvec_total = H >> 3;
  const int v0 = static_cast<int>(crank) * p.slice_vec;
  const int nv = max(0, min(nvec_total - v0, p.slice_vec));  // 16-byte vectors of this CTA's slice
  const int stride = p.slice_vec * 16;                       // bytes per staged row
  const int nslots = p.nslots;

  uint8_t* stage = smem;  // [nslots][slice] act
  uint8_t* zero_row = smem + p.off_zero;
  const uint8_t** slot_src = reinterpret_cast<const uint8_t**>(smem + p.off_src);
  int2* meta = reinterpret_cast<int2*>(smem + p.off_meta);
  int* sh_off = reinterpret_cast<int*>(smem + p.off_shoff);
  float* red = reinterpret_cast<float*>(smem + p.off_red);  // [32] warp sums, [32] CTA sum, [33] total

  for (int i = tid; i < p.slice_vec; i += nthreads) reinterpret_cast<uint4*>(zero_row)[i] = make_uint4(0, 0, 0, 0);
  if (p.pdl) pdl_launch_dependents();
  if (p.routing_early) load_slots(p, t, stride, slot_src, meta, sh_off, tid, nthreads);
  if (p.pdl) pdl_wait();
  if (!p.routing_early) load_slots(p, t, stride, slot_src, meta, sh_off, tid, nthreads);
  __syncthreads();

  // Gather: every valid (slot, 16-byte vector) pair of this slice, all in flight together.
  const int total = nslots * nv;
  const uint32_t stage_addr = smem_addr(stage);
  for (int i = tid; i < total; i += nthreads) {
    const int s = i / nv;
    const int v = i - s * nv;
    const uint8_t* src = slot_src[s];
    if (src != nullptr)
      cp_async16(stage_addr + static_cast<uint32_t>(s) * stride + v * 16, src + static_cast<int64_t>(v0 + v) * 16);
  }
  cp_async_commit();

  // This thread's 4 elements; residual and gamma load while the gather is in flight.
  const int el = tid * 4;
  const bool active = el < nv * 8;
  const int h = v0 * 8 + el;
  uint2 res_raw = make_uint2(0, 0), gam_raw = make_uint2(0, 0);
  if (active) {
    res_raw = ldg8(p.residual + (static_cast<int64_t>(t) * H + h) * 2);
    gam_raw = ldg8(p.gamma + static_cast<int64_t>(h) * 2);
  }
  cp_async_wait_all();
  __syncthreads();

  float S[4] = {0.f, 0.f, 0.f, 0.f}, x[4] = {0.f, 0.f, 0.f, 0.f};
  float ss = 0.0f;
  if (active) {
    finalize4<A, RMAX>(meta, sh_off, stage, zero_row, el * 2, p.R, p.K, p.rsf, S);
    const uint2 ro = residual_step<A>(S, res_raw, x, ss);
    if (p.residual_out != nullptr) stg8(p.residual_out + (static_cast<int64_t>(t) * H + h) * 2, ro);
  }

  // Sum of squares: warp shuffle, warps in order, then the cluster's CTAs in rank order.
  ss = warp_sum(ss);
  const int warp = tid >> 5, lane = tid & 31;
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (tid == 0) {
    float cta = 0.0f;
    for (int w = 0; w < (nthreads >> 5); ++w) cta = __fadd_rn(cta, red[w]);
    red[32] = cta;
  }
  if (C > 1) {
    cluster_arrive_release();
    cluster_wait_acquire();
    if (tid == 0) {
      float tot = 0.0f;
      for (uint32_t c = 0; c < C; ++c) tot = __fadd_rn(tot, dsmem_load_f32(&red[32], c));
      red[33] = tot;
    }
    cluster_arrive_release();  // this CTA's remote reads are done; matched by the wait at the end
  } else if (tid == 0) {
    red[33] = red[32];
  }
  __syncthreads();
  const float rstd = rms_rstd(red[33], H, p.eps);
  const float qscale = (p.quant != MFR_QUANT_NONE) ? *p.quant_scale : 1.0f;
  epilogue4<A>(p, t, h, active, x, gam_raw, rstd, qscale);
  if (C > 1) cluster_wait_acquire();  // no CTA leaves while a peer may still read its shared memory
}

template <typename A, int RMAX>
static cudaError_t launch_cluster(const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  auto kern = cluster_finalize_kernel<A, RMAX>;
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_optin);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.grid, 1, 1);
  cfg.blockDim = dim3(g.block, 1, 1);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = g.cluster;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (p.pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename A, int RMAX>
static int max_active_clusters(const LaunchGeom& g) {
  auto kern = cluster_finalize_kernel<A, RMAX>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_optin);
  cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.cluster, 1, 1);
  cfg.blockDim = dim3(g.block, 1, 1);
  cfg.dynamicSmemBytes = g.smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = g.cluster;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <typename A>
static cudaError_t launch_cluster_r(const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  if (p.R <= 1) return launch_cluster<A, 1>(p, g, stream);
  if (p.R <= 2) return launch_cluster<A, 2>(p, g, stream);
  if (p.R <= 4) return launch_cluster<A, 4>(p, g, stream);
  return launch_cluster<A, 8>(p, g, stream);
}

cudaError_t launch_cluster_kernel(int act_dtype, const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  return act_dtype == MFR_BF16 ? launch_cluster_r<__nv_bfloat16>(p, g, stream) : launch_cluster_r<__half>(p, g, stream);
}

// Occupancy of the cluster kernel; the R bound does not change its resources materially, so the
// widest instantiation answers for all.
int cluster_kernel_max_active_clusters(int act_dtype, const LaunchGeom& g) {
  return act_dtype == MFR_BF16 ? max_active_clusters<__nv_bfloat16, 8>(g) : max_active_clusters<__half, 8>(g);
}

}  // namespace mfr
