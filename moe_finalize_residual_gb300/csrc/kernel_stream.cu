// Large-batch fused finalize: persistent CTAs (one per SM), each finalizing whole tokens in turn,
// with every gathered row streamed into a shared-memory ring by asynchronous copies.
//
// Roles:
//  - routing warp: for each of the CTA's tokens, reads the R*K route indices and scales, checks the
//    bound of every index, and writes the token's list of rows -- valid routes in order, each
//    partial's shared row after its routes -- into a ring of lists (kLists tokens deep);
//  - compute warps: thread j owns 16-byte columns j, j + NCT, j + 2*NCT, ... of every row (8 elements
//    each; a hidden pass covers 8 * NCT * kQ elements).  Each thread copies ITS OWN columns of the
//    rows ahead with cp.async (16 bytes, through L2) into a ring of NB row slots, one commit group per
//    row, up to NB-1 rows ahead and across token boundaries, and later reads only what it copied: the
//    data needs no barrier, only cp.async.wait_group, which retires groups in issue order.  Every
//    compute thread issues copies, so the whole CTA keeps rows in flight.  For each row in list order
//    a thread applies the partial's FP32 fused multiply-add in route order; when the list moves to the
//    next partial it finishes the previous one (times the routed scaling factor, plus the shared row,
//    rounded once) into the FP32 rank sum; the residual row closes a pass (residual_out, kept in shared
//    memory, and the sum of squares).  After a token's last pass the compute warps reduce the sum of
//    squares and write norm_out and the quantised output from the kept values and gamma.
//
// Prior art: flashinfer PR #6546 (large-batch finalizeKernelVecLoad path); flashinfer PR #3385
// (RMSNorm inputs staged in shared memory).  The arithmetic is that of flashinfer PR #6631,
// Description, operation for operation the same as the cluster kernel's.
//
// A bulk-copy (cp.async.bulk) pipeline fed by a producer warp was measured first on this path and
// streamed at 15-30 GB/s per SM; per-thread 16-byte copies reach the HBM limit.
//
// Every wait on an mbarrier is bounded (about 2 s of device time).  A wait that runs out counts a
// timeout in device memory and tells the other warps to stop; every thread waits for its own copies
// before the CTA exits.
#include "mfr_device.cuh"
#include "mfr_launch.h"

namespace mfr {

__device__ unsigned int g_wait_timeouts = 0;

constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kRoutingWarp = 0;
constexpr int kFirstComputeWarp = 1;
constexpr int kQ = kStreamColumns;    // 16-byte columns per compute thread per pass
constexpr int kLists = kStreamLists;  // row lists in the ring (tokens)
constexpr uint32_t kRowShared = 0x100u;

// One listed row of a token: where it starts, its scale, its partial (and whether it is the
// partial's shared row).
struct RowEntry {
  const uint8_t* src;
  float scale;
  uint32_t tag;  // partial index | kRowShared
};

// Bounded wait.  Returns false if the CTA is aborting or the limit ran out (then it starts the abort).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicAdd(&g_wait_timeouts, 1u);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// The same, with one decision for the whole warp.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, wait_bounded(bar, parity, abort_flag));
}

// Finish partial rows into the rank sum: acc (times the factor unless the shared row already applied
// it), rounded once, added to S in FP32; acc restarts from +0.
template <typename A>
__device__ __forceinline__ void flush_partial(float acc[kQ * 8], float S[kQ * 8], bool shared_done, float rsf) {
#pragma unroll
  for (int i = 0; i < kQ * 8; ++i) {
    const float a = shared_done ? acc[i] : __fmul_rn(acc[i], rsf);
    S[i] = __fadd_rn(S[i], Act<A>::round(a));
    acc[i] = 0.0f;
  }
}

// Slot s of a token's row list, in list order: partial by partial, routes k = 0..K-1 then the
// partial's shared row (if it has one).  Returns the partial and k (-1 for the shared row).
__device__ __forceinline__ void slot_in_list_order(const KParams& p, int s, int& r, int& k) {
  int base = 0;
  for (r = 0; r < p.R - 1; ++r) {
    const int n = p.K + static_cast<int>((p.shared_mask >> r) & 1u);
    if (s < base + n) break;
    base += n;
  }
  k = s - base;
  if (k >= p.K) k = -1;
}

// The routing warp's list for token t (valid routes in order, then the partial's shared row), compacted
// with a warp ballot.  Returns the number of rows.
__device__ __forceinline__ int build_row_list(const KParams& p, int t, RowEntry* list, int lane) {
  int n = 0;
  for (int base = 0; base < p.nslots; base += 32) {
    const int s = base + lane;
    bool valid = false;
    RowEntry row;
    if (s < p.nslots) {
      int r, k;
      slot_in_list_order(p, s, r, k);
      const KPartial& P = p.part[r];
      if (k < 0) {
        row.src = P.shared + static_cast<int64_t>(t) * p.H * 2;
        row.scale = 1.0f;
        row.tag = static_cast<uint32_t>(r) | kRowShared;
        valid = true;
      } else {
        // flashinfer PR #6631, Test changes: -1 routes contribute nothing; one bound check per route.
        const int64_t ei = static_cast<int64_t>(t) * p.K + k;
        const int32_t idx = P.perm[ei];
        valid = idx >= 0 && static_cast<int64_t>(idx) < P.rows;
        if (valid) {
          row.src = P.gemm2 + static_cast<int64_t>(idx) * p.H * 2;
          row.scale = load_scale(P.scale, ei, p.scale_dtype);
          row.tag = static_cast<uint32_t>(r);
        }
      }
    }
    const uint32_t ballot = __ballot_sync(0xffffffffu, valid);
    if (valid) list[n + __popc(ballot & ((1u << lane) - 1u))] = row;
    n += __popc(ballot);
  }
  return n;
}

constexpr int kNB = kStreamSlots;     // row slots in the ring
constexpr int kLook = kNB - 1;        // rows in flight ahead of the one being read

template <typename A>
__global__ void __launch_bounds__(kStreamMaxThreads, 1) stream_finalize_kernel(const __grid_constant__ KParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int ncw = static_cast<int>(blockDim.x >> 5) - kFirstComputeWarp;  // compute warps
  const int nct = ncw * 32;
  const int H = p.H, W = p.chunk;
  const int npass = (H + W - 1) / W;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  const uint32_t rfull0 = smem_addr(bars);       // kLists: row list written (routing warp)
  const uint32_t rempty0 = rfull0 + 8u * kLists; // kLists: row list released (one arrival per compute warp)
  const uint32_t cbar0 = rempty0 + 8u * kLists;  // 2: compute warps done with a token (by parity)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kLists + 2);
  uint8_t* slots = smem + p.off_stage;           // kNB row slots of p.stage_bytes
  uint8_t* ring0 = smem + p.off_ring;
  uint8_t* gamma_s = smem + p.off_gamma;
  uint8_t* stash = smem + p.off_stash;
  float* sred = reinterpret_cast<float*>(smem + p.off_sred);  // [2][32]

  if (tid == 0) {
    for (int i = 0; i < kLists; ++i) {
      mbar_init(rfull0 + 8u * i, 1);
      mbar_init(rempty0 + 8u * i, static_cast<uint32_t>(ncw));
    }
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

  const int ntok =
      (p.T - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);

  if (warp == kRoutingWarp) {
    for (int i = 0; i < ntok; ++i) {
      const int t = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
      const int slot = i % kLists;
      if (!warp_wait(rempty0 + 8u * slot, (static_cast<uint32_t>(i / kLists) & 1u) ^ 1u, abort_flag)) break;
      uint8_t* e = ring0 + slot * p.ring_bytes;
      const int n = build_row_list(p, t, reinterpret_cast<RowEntry*>(e + 16), lane);
      if (lane == 0) *reinterpret_cast<int*>(e) = n;
      __syncwarp();
      if (lane == 0) mbar_arrive(rfull0 + 8u * slot);
    }
  } else {
    const int jt = tid - kFirstComputeWarp * 32;  // compute thread: owns 16-byte columns jt + nct*q
    const int cw = warp - kFirstComputeWarp;
    const float qscale = (p.quant != MFR_QUANT_NONE) ? *p.quant_scale : 1.0f;

    // This thread's columns of gamma (they travel with the first row's copies).
    for (int pass = 0; pass < npass; ++pass) {
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const int el = 8 * jt + 8 * nct * q, h = pass * W + el;
        if (el < W && h < H) cp_async16(smem_addr(gamma_s + static_cast<int64_t>(h) * 2), p.gamma + static_cast<int64_t>(h) * 2);
      }
    }

    // Issue cursor: token ii (local index), pass ip and row ij (0..n, n = the residual row) of it.
    int ii = 0, ip = 0, ij = 0, in_n = -1;
    const RowEntry* ilist = nullptr;
    uint32_t gi = 0;
    // Consume cursor (the same walk).
    int ci = 0, cp_ = 0, cj = 0, cn = -1;
    const RowEntry* clist = nullptr;
    uint32_t gc = 0;
    bool ok = true;

    // Issue this thread's columns of the next row (if there is one it may issue) and commit a group.
    auto issue_one = [&]() {
      if (ok && ii < ntok && ii < ci + kLists) {  // a list is reused only after its token is consumed
        if (in_n < 0) {
          const int slot = ii % kLists;
          if (warp_wait(rfull0 + 8u * slot, static_cast<uint32_t>(ii / kLists) & 1u, abort_flag)) {
            const uint8_t* e = ring0 + slot * p.ring_bytes;
            in_n = *reinterpret_cast<const int*>(e);
            ilist = reinterpret_cast<const RowEntry*>(e + 16);
          } else {
            ok = false;
          }
        }
        if (ok) {
          const int t = static_cast<int>(blockIdx.x) + ii * static_cast<int>(gridDim.x);
          const uint8_t* src = (ij < in_n) ? ilist[ij].src : p.residual + static_cast<int64_t>(t) * H * 2;
          const int h0 = ip * W;
          uint8_t* dst = slots + static_cast<size_t>(gi % kNB) * p.stage_bytes;
#pragma unroll
          for (int q = 0; q < kQ; ++q) {
            const int el = 8 * jt + 8 * nct * q;
            if (el < W && h0 + el < H)
              cp_async16(smem_addr(dst + el * 2), src + static_cast<int64_t>(h0 + el) * 2);
          }
          ++gi;
          if (++ij > in_n) {
            ij = 0;
            if (++ip == npass) {
              ip = 0;
              ++ii;
              in_n = -1;
            }
          }
        }
      }
      cp_async_commit();
    };

    for (int s = 0; s < kLook; ++s) issue_one();

    float acc[kQ * 8], S[kQ * 8];
#pragma unroll
    for (int i = 0; i < kQ * 8; ++i) acc[i] = S[i] = 0.0f;
    float ss = 0.0f;
    int cur = -1;
    bool shared_done = false;

    while (ok && ci < ntok) {
      issue_one();
      cp_async_wait_group<kLook>();  // this thread's columns of row gc have landed
      if (cn < 0) {  // the issue cursor already waited for this token's list
        const uint8_t* e = ring0 + (ci % kLists) * p.ring_bytes;
        cn = *reinterpret_cast<const int*>(e);
        clist = reinterpret_cast<const RowEntry*>(e + 16);
      }
      const int t = static_cast<int>(blockIdx.x) + ci * static_cast<int>(gridDim.x);
      const int jr = cj;
      const int h0 = cp_ * W;
      const uint8_t* row = slots + static_cast<size_t>(gc % kNB) * p.stage_bytes;
      if (jr < cn) {
        const RowEntry ent = clist[jr];
        const int r = static_cast<int>(ent.tag & 0xffu);
        if (r != cur) {  // the list moved to the next partial: finish the previous one
          if (cur >= 0) flush_partial<A>(acc, S, shared_done, p.rsf);
          cur = r;
          shared_done = false;
        }
        const bool is_shared = (ent.tag & kRowShared) != 0;  // the same for the whole CTA
        if (is_shared) {
#pragma unroll
          for (int q = 0; q < kQ; ++q) {
            const int el = 8 * jt + 8 * nct * q;
            if (el < W && h0 + el < H) {
              float v[8];
              unpack8<A>(*reinterpret_cast<const uint4*>(row + el * 2), v);
#pragma unroll
              for (int c = 0; c < 8; ++c) acc[8 * q + c] = __fadd_rn(__fmul_rn(acc[8 * q + c], p.rsf), v[c]);
            }
          }
        } else {
#pragma unroll
          for (int q = 0; q < kQ; ++q) {
            const int el = 8 * jt + 8 * nct * q;
            if (el < W && h0 + el < H) {
              float v[8];
              unpack8<A>(*reinterpret_cast<const uint4*>(row + el * 2), v);
#pragma unroll
              for (int c = 0; c < 8; ++c) acc[8 * q + c] = __fmaf_rn(ent.scale, v[c], acc[8 * q + c]);
            }
          }
        }
        shared_done = shared_done || is_shared;
      } else {  // the residual row closes the pass
        if (cur >= 0) flush_partial<A>(acc, S, shared_done, p.rsf);
        cur = -1;
        shared_done = false;
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
          const int el = 8 * jt + 8 * nct * q;
          if (el < W && h0 + el < H) {
            const uint4 res_raw = *reinterpret_cast<const uint4*>(row + el * 2);
            float x[8];
            const uint2 lo = residual_step<A>(&S[8 * q], make_uint2(res_raw.x, res_raw.y), x, ss);
            const uint2 hi = residual_step<A>(&S[8 * q + 4], make_uint2(res_raw.z, res_raw.w), x + 4, ss);
            const uint4 ro = make_uint4(lo.x, lo.y, hi.x, hi.y);
            *reinterpret_cast<uint4*>(stash + static_cast<int64_t>(h0 + el) * 2) = ro;
            if (p.residual_out != nullptr)
              *reinterpret_cast<uint4*>(p.residual_out + (static_cast<int64_t>(t) * H + h0 + el) * 2) = ro;
          }
        }
#pragma unroll
        for (int i = 0; i < kQ * 8; ++i) S[i] = 0.0f;
      }
      ++gc;
      if (++cj <= cn) continue;
      cj = 0;
      if (++cp_ < npass) continue;
      cp_ = 0;

      // Token done: release its list, reduce the sum of squares over the compute warps (in warp order,
      // double-buffered by token parity; the warps meet on an mbarrier so the wait is bounded), write
      // norm_out and the quantised output from the kept residual_out and gamma.
      __syncwarp();
      if (lane == 0) mbar_arrive(rempty0 + 8u * (ci % kLists));
      const float wsum = warp_sum(ss);
      float* rb = sred + (ci & 1) * 32;
      if (lane == 0) {
        rb[cw] = wsum;
        mbar_arrive(cbar0 + 8u * (ci & 1));
      }
      if (!warp_wait(cbar0 + 8u * (ci & 1), static_cast<uint32_t>(ci >> 1) & 1u, abort_flag)) {
        ok = false;
        break;
      }
      float tot = 0.0f;
      for (int w2 = 0; w2 < ncw; ++w2) tot = __fadd_rn(tot, rb[w2]);
      const float rstd = rms_rstd(tot, H, p.eps);
      for (int ps = 0; ps < npass; ++ps) {
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
          const int el = 8 * jt + 8 * nct * q;
          const int h = ps * W + el;
          const bool active = el < W && h < H;
          float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, g[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          if (active) {
            unpack8<A>(*reinterpret_cast<const uint4*>(stash + static_cast<int64_t>(h) * 2), x);
            unpack8<A>(*reinterpret_cast<const uint4*>(gamma_s + static_cast<int64_t>(h) * 2), g);
          }
          epilogue<A, 8>(p, t, h, active, x, g, rstd, qscale);
        }
      }
      ss = 0.0f;
      ++ci;
      cn = -1;
    }
    cp_async_wait_all();  // no copy of this thread may land after the CTA exits
  }
  __syncthreads();
}

template <typename A>
static cudaError_t launch_stream(const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  auto kern = stream_finalize_kernel<A>;
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

cudaError_t launch_stream_kernel(int act_dtype, const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  return act_dtype == MFR_BF16 ? launch_stream<__nv_bfloat16>(p, g, stream) : launch_stream<__half>(p, g, stream);
}

template <typename A>
static int blocks_per_sm(const LaunchGeom& g) {
  auto kern = stream_finalize_kernel<A>;
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
