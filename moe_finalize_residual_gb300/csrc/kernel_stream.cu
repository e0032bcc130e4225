// Large-batch fused finalize: persistent CTAs (one per SM), each finalizing whole tokens in turn,
// with every gathered row streamed into a shared-memory ring by bulk asynchronous copies.
//
// Roles (warp specialisation inside one CTA):
//  - routing warp: for each of the CTA's tokens, reads the R*K route indices and scales, checks the
//    bound of every index, and writes the row addresses, scales and flags into a routing ring
//    (RDEPTH tokens ahead);
//  - producer warp: for each token and each hidden chunk, arms a stage's mbarrier with the exact byte
//    count and issues one cp.async.bulk per valid row (R*K routes, R shared rows, the residual row);
//    its lanes issue the copies of different rows in parallel.  Copies are per-CTA (no multicast);
//  - consumer warps: per stage, run the FP32 fused multiply-add chain over the staged rows in route
//    order for 4 elements per thread, round per partial, sum the ranks in order, add the residual,
//    write residual_out, keep x in shared memory and accumulate the sum of squares; at the end of a
//    token they reduce the sum of squares (shuffles, then the consumer warps in order) and write
//    norm_out and the quantised output from the kept x and a CTA-resident copy of gamma.
//
// Prior art: flashinfer PR #6546 (large-batch finalizeKernelVecLoad path); flashinfer PR #3385
// (RMSNorm inputs staged with TMA and mbarriers).  The arithmetic is that of flashinfer PR #6631,
// Description; it matches the cluster kernel operation for operation.
//
// Every wait on an mbarrier is bounded (about 2 s of device time).  A wait that runs out counts a
// timeout in device memory, tells the other roles to stop, and the producer waits (again bounded)
// for the copies it issued before the CTA exits.
#include "mfr_device.cuh"
#include "mfr_launch.h"

namespace mfr {

__device__ unsigned int g_wait_timeouts = 0;

constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kProducerWarp = 0;
constexpr int kRoutingWarp = 1;
constexpr int kFirstConsumerWarp = 2;

// Bounded wait.  Returns false if the CTA is aborting or the limit ran out (then it starts the abort).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             bool honour_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (honour_abort && *abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicAdd(&g_wait_timeouts, 1u);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// The same, with one decision for the whole warp: every lane waits, and the warp goes on only if all
// lanes saw the barrier complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, wait_bounded(bar, parity, abort_flag));
}

template <typename A, int RMAX>
__global__ void __launch_bounds__(kStreamMaxThreads, 1) stream_finalize_kernel(const __grid_constant__ KParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int ncw = static_cast<int>(blockDim.x >> 5) - kFirstConsumerWarp;  // consumer warps
  const int H = p.H, CH = p.chunk, NS = p.stages, D = p.rdepth, nslots = p.nslots;
  const int nch = (H + CH - 1) / CH;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  const uint32_t full0 = smem_addr(bars);          // NS: stage filled (1 arrival + transaction bytes)
  const uint32_t empty0 = full0 + 8u * NS;         // NS: stage consumed (one arrival per consumer warp)
  const uint32_t rfull0 = empty0 + 8u * NS;        // D: routing entry written (routing warp)
  const uint32_t rempty0 = rfull0 + 8u * D;        // D: routing entry released (producer + consumer warps)
  const uint32_t gbar = rempty0 + 8u * D;          // gamma resident
  const uint32_t cbar0 = gbar + 8u;                // 2: consumer warps done with a token (by parity)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * NS + 2 * D + 3);
  uint8_t* stage0 = smem + p.off_stage;
  uint8_t* ring0 = smem + p.off_ring;
  uint8_t* zero_row = smem + p.off_zero_s;
  uint8_t* gamma_s = smem + p.off_gamma;
  uint8_t* stash = smem + p.off_stash;
  float* sred = reinterpret_cast<float*>(smem + p.off_sred);  // [2][32]

  // Routing ring entry: row address [nslots] | (offset, scale) [R*K] | shared offset [8] | valid count.
  // Offsets are relative to a stage's base: slot s sits at s * CH * 2, the residual at nslots * CH * 2.
  const int ring_off_meta = nslots * 8;
  const int ring_off_shoff = ring_off_meta + p.R * p.K * 8;
  const int ring_off_count = ring_off_shoff + MFR_MAX_PARTIALS * 4;

  for (int i = tid; i < CH / 8; i += blockDim.x) reinterpret_cast<uint4*>(zero_row)[i] = make_uint4(0, 0, 0, 0);

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full0 + 8u * i, 1);
      mbar_init(empty0 + 8u * i, static_cast<uint32_t>(ncw));
    }
    for (int i = 0; i < D; ++i) {
      mbar_init(rfull0 + 8u * i, 1);
      mbar_init(rempty0 + 8u * i, 1u + static_cast<uint32_t>(ncw));
    }
    mbar_init(gbar, 1);
    mbar_init(cbar0, static_cast<uint32_t>(ncw));
    mbar_init(cbar0 + 8u, static_cast<uint32_t>(ncw));
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (p.pdl) {
    pdl_launch_dependents();
    pdl_wait();
  }

  const int ntok = (p.T - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);

  if (warp == kRoutingWarp) {
    for (int i = 0; i < ntok; ++i) {
      const int t = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
      const int slot = i % D;
      const uint32_t ph = static_cast<uint32_t>(i / D) & 1u;
      if (!warp_wait(rempty0 + 8u * slot, ph ^ 1u, abort_flag)) break;
      uint8_t* e = ring0 + slot * p.ring_bytes;
      int nvalid = 0;
      for (int s = lane; s < nslots; s += 32) {
        const SlotSource o = slot_source(p, s, t);
        reinterpret_cast<const uint8_t**>(e)[s] = o.src;
        if (o.k >= 0)
          reinterpret_cast<int2*>(e + ring_off_meta)[o.r * p.K + o.k] =
              make_int2(o.src ? s * CH * 2 : -1, __float_as_int(o.scale));
        else
          reinterpret_cast<int*>(e + ring_off_shoff)[o.r] = s * CH * 2;
        nvalid += o.src ? 1 : 0;
      }
      if (lane < p.R && !((p.shared_mask >> lane) & 1u)) reinterpret_cast<int*>(e + ring_off_shoff)[lane] = -1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) nvalid += __shfl_xor_sync(0xffffffffu, nvalid, o);
      if (lane == 0) *reinterpret_cast<int*>(e + ring_off_count) = nvalid;
      __syncwarp();
      if (lane == 0) mbar_arrive(rfull0 + 8u * slot);
    }
  } else if (warp == kProducerWarp) {
    if (lane == 0 && ntok > 0) {  // the consumers wait for gamma only if the CTA has a token
      mbar_arrive_expect_tx(gbar, static_cast<uint32_t>(H) * 2u);
      bulk_g2s(smem_addr(gamma_s), p.gamma, static_cast<uint32_t>(H) * 2u, gbar);
    }
    int st = 0;
    uint32_t sph = 0;
    int64_t armed = 0;  // stages armed so far
    bool ok = true;
    for (int i = 0; i < ntok && ok; ++i) {
      const int t = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
      const int slot = i % D;
      const uint32_t ph = static_cast<uint32_t>(i / D) & 1u;
      if (!warp_wait(rfull0 + 8u * slot, ph, abort_flag)) break;
      const uint8_t* e = ring0 + slot * p.ring_bytes;
      const int nvalid = *reinterpret_cast<const int*>(e + ring_off_count);
      for (int c = 0; c < nch; ++c) {
        const int h0 = c * CH;
        const uint32_t bytes = static_cast<uint32_t>(min(CH, H - h0)) * 2u;
        if (!warp_wait(empty0 + 8u * st, sph ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t sb = smem_addr(stage0 + st * p.stage_bytes);
        const uint32_t fb = full0 + 8u * st;
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, static_cast<uint32_t>(nvalid + 1) * bytes);
          bulk_g2s(sb + static_cast<uint32_t>(nslots) * CH * 2u,
                   p.residual + (static_cast<int64_t>(t) * H + h0) * 2, bytes, fb);
        }
        __syncwarp();
        for (int s = lane; s < nslots; s += 32) {
          const uint8_t* src = reinterpret_cast<const uint8_t* const*>(e)[s];
          if (src != nullptr) bulk_g2s(sb + static_cast<uint32_t>(s) * CH * 2u, src + static_cast<int64_t>(h0) * 2, bytes, fb);
        }
        ++armed;
        if (++st == NS) {
          st = 0;
          sph ^= 1u;
        }
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(rempty0 + 8u * slot);
    }
    // On an abort, wait (bounded, ignoring the abort flag) until the last copies of every stage have
    // landed, so none writes into shared memory after the CTA exits.
    if (*abort_flag) {
      for (int s = 0; s < NS && s < armed; ++s) {
        const int64_t last = armed - 1 - ((armed - 1 - s) % NS);  // last arm of stage s
        wait_bounded(full0 + 8u * s, static_cast<uint32_t>(last / NS) & 1u, abort_flag, false);
      }
      if (lane == 0) wait_bounded(gbar, 0, abort_flag, false);
    }
  } else {
    const int j = tid - kFirstConsumerWarp * 32;  // consumer thread index
    const int cw = warp - kFirstConsumerWarp;
    const float qscale = (p.quant != MFR_QUANT_NONE) ? *p.quant_scale : 1.0f;
    int st = 0;
    uint32_t sph = 0;
    bool gamma_ready = false;
    for (int i = 0; i < ntok; ++i) {
      const int t = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
      const int slot = i % D;
      const uint32_t ph = static_cast<uint32_t>(i / D) & 1u;
      if (!warp_wait(rfull0 + 8u * slot, ph, abort_flag)) break;
      const uint8_t* e = ring0 + slot * p.ring_bytes;
      const int2* meta = reinterpret_cast<const int2*>(e + ring_off_meta);
      const int* sh_off = reinterpret_cast<const int*>(e + ring_off_shoff);
      float ss = 0.0f;
      bool ok = true;
      for (int c = 0; c < nch; ++c) {
        const int h0 = c * CH;
        const int w = min(CH, H - h0);
        if (!warp_wait(full0 + 8u * st, sph, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* sb = stage0 + st * p.stage_bytes;
        const int el = j * 4;
        if (el < w) {
          float S[4] = {0.f, 0.f, 0.f, 0.f}, x[4];
          finalize4<A, RMAX>(meta, sh_off, sb, zero_row, el * 2, p.R, p.K, p.rsf, S);
          const uint2 res_raw = *reinterpret_cast<const uint2*>(sb + static_cast<int64_t>(nslots) * CH * 2 + el * 2);
          const uint2 ro = residual_step<A>(S, res_raw, x, ss);
          *reinterpret_cast<uint2*>(stash + static_cast<int64_t>(h0 + el) * 2) = ro;
          if (p.residual_out != nullptr) stg8(p.residual_out + (static_cast<int64_t>(t) * H + h0 + el) * 2, ro);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8u * st);
        if (++st == NS) {
          st = 0;
          sph ^= 1u;
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(rempty0 + 8u * slot);
      // Sum of squares over the consumer warps, in warp order (double-buffered by token parity).  The
      // consumer warps meet on an mbarrier so that this wait, like every other, is bounded.
      ss = warp_sum(ss);
      float* rb = sred + (i & 1) * 32;
      if (lane == 0) {
        rb[cw] = ss;
        mbar_arrive(cbar0 + 8u * (i & 1));
      }
      if (!warp_wait(cbar0 + 8u * (i & 1), static_cast<uint32_t>(i >> 1) & 1u, abort_flag)) break;
      float tot = 0.0f;
      for (int w2 = 0; w2 < ncw; ++w2) tot = __fadd_rn(tot, rb[w2]);
      const float rstd = rms_rstd(tot, H, p.eps);
      if (!gamma_ready) {
        if (!warp_wait(gbar, 0, abort_flag)) break;
        gamma_ready = true;
      }
      for (int c = 0; c < nch; ++c) {
        const int h0 = c * CH;
        const int el = j * 4;
        const bool active = el < min(CH, H - h0);
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        uint2 graw = make_uint2(0, 0);
        if (active) {
          unpack4<A>(*reinterpret_cast<const uint2*>(stash + static_cast<int64_t>(h0 + el) * 2), x);
          graw = *reinterpret_cast<const uint2*>(gamma_s + static_cast<int64_t>(h0 + el) * 2);
        }
        epilogue4<A>(p, t, h0 + el, active, x, graw, rstd, qscale);
      }
    }
  }
  __syncthreads();
}

template <typename A, int RMAX>
static cudaError_t launch_stream(const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  auto kern = stream_finalize_kernel<A, RMAX>;
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_optin);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.grid, 1, 1);
  cfg.blockDim = dim3(g.block, 1, 1);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (p.pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename A>
static cudaError_t launch_stream_r(const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  if (p.R <= 1) return launch_stream<A, 1>(p, g, stream);
  if (p.R <= 2) return launch_stream<A, 2>(p, g, stream);
  if (p.R <= 4) return launch_stream<A, 4>(p, g, stream);
  return launch_stream<A, 8>(p, g, stream);
}

cudaError_t launch_stream_kernel(int act_dtype, const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  return act_dtype == MFR_BF16 ? launch_stream_r<__nv_bfloat16>(p, g, stream) : launch_stream_r<__half>(p, g, stream);
}

template <typename A>
static int blocks_per_sm(const LaunchGeom& g) {
  auto kern = stream_finalize_kernel<A, 8>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_optin);
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, g.block, g.smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int stream_kernel_blocks_per_sm(int act_dtype, const LaunchGeom& g) {
  return act_dtype == MFR_BF16 ? blocks_per_sm<__nv_bfloat16>(g) : blocks_per_sm<__half>(g);
}

cudaError_t read_and_reset_timeouts(unsigned int* count) {
  cudaError_t e = cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(unsigned int));
}

}  // namespace mfr
