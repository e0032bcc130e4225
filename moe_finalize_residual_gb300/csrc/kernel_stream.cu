// Large-batch fused finalize: persistent CTAs (one per SM), each finalizing whole tokens in turn,
// with every gathered row streamed into a shared-memory ring by asynchronous copies.
//
// Roles:
//  - routing warp: for each of the CTA's tokens, reads the R*K route indices and scales, checks the
//    bound of every index, and writes the token's list of rows into a ring of lists (kLists tokens
//    deep): valid routes in order, each partial's shared row after its routes, the residual row last;
//    each entry carries its partial and whether it is the partial's last row;
//  - compute warps, in G groups that run separate token streams (or, with at most one token per CTA,
//    split each token's hidden dimension between them): thread j of a group owns 16-byte columns
//    j, j + NCT, j + 2*NCT, ... of every row (8 elements each; a hidden pass covers 8 * NCT * kQ
//    elements).  Each thread copies ITS OWN columns of the rows ahead with cp.async (16 bytes, through
//    L2) into its group's ring of NB row slots, one commit group per row, up to NB-1 rows ahead and
//    across token boundaries, and later reads only what it copied: the data needs no barrier, only
//    cp.async.wait_group, which retires groups in issue order.  Per row a thread applies the partial's
//    FP32 fused multiply-add (or the shared-row step); after a partial's last row it rounds the
//    partial once into the FP32 rank sum; the residual row closes a pass (residual_out, kept in shared
//    memory, and the sum of squares).  After a token's last pass the group reduces the sum of squares
//    and writes norm_out and the quantised output from the kept values and gamma.
//
// The group shape is a compile-time constant, so a thread's column offsets are immediates and the
// per-row work is the copies, the arithmetic and a few cursor updates.
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
#include "mfr_rowlist.cuh"

#include <atomic>

namespace mfr {

__device__ unsigned int g_wait_timeouts = 0;

constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kRoutingWarp = 0;
constexpr int kFirstComputeWarp = 1;
constexpr int kQ = kStreamColumns;    // 16-byte columns per compute thread per pass
constexpr int kLists = kStreamLists;  // row lists in the ring (tokens)
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

// Round a finished partial into the rank sum: acc (times the factor unless the partial's shared row
// already applied it), rounded once, added to S in FP32; acc restarts from +0.  Element pairs use the
// packed FP32 operations, which round each lane like the scalar ones (the rounding to act between the
// multiply and the add keeps them from being contracted).
template <typename A>
__device__ __forceinline__ void flush_partial(float2 acc[kQ * 4], float2 S[kQ * 4], bool shared_done, float rsf) {
  const float2 f = make_float2(rsf, rsf);
#pragma unroll
  for (int i = 0; i < kQ * 4; ++i) {
    const float2 a = shared_done ? acc[i] : __fmul2_rn(acc[i], f);
    S[i] = __fadd2_rn(S[i], round_pair<A>(a));
    acc[i] = make_float2(0.0f, 0.0f);
  }
}

constexpr int kNB = kStreamSlots;  // row slots in a group's ring
constexpr int kLook = kNB - 1;     // rows in flight ahead of the one being read

// G groups of compute warps; G is a template parameter so that a thread's column offsets are
// immediates.
template <typename A, int G>
__global__ void __launch_bounds__(kStreamMaxThreads, 1) stream_finalize_kernel(const __grid_constant__ KParams p) {
  constexpr int NCW = kStreamGroups * kStreamGroupWarps / G;  // compute warps per group
  constexpr int NCT = 32 * NCW;                               // threads per group
  constexpr int QB = NCT * 16;                                // bytes between a thread's columns
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int H = p.H, W = p.chunk;
  const int npass = (H + W - 1) / W;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  const uint32_t rfull0 = smem_addr(bars);       // kLists: row list written (routing warp)
  const uint32_t rempty0 = rfull0 + 8u * kLists; // kLists: row list released (one arrival per compute warp)
  const uint32_t cbar0 = rempty0 + 8u * kLists;  // 2 per group: its warps done with a token (by parity)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kLists + 2 * kStreamGroups);
  uint8_t* ring0 = smem + p.off_ring;

  if (tid == 0) {
    for (int i = 0; i < kLists; ++i) {
      mbar_init(rfull0 + 8u * i, 1);
      mbar_init(rempty0 + 8u * i, static_cast<uint32_t>(p.split ? G * NCW : NCW));
    }
    // (the failure-detection test hook adds an arrival that never comes, so every wait on these runs out)
    if (p.split) {  // all groups work on every token: one reduction barrier pair for the CTA
      mbar_init(cbar0, static_cast<uint32_t>(G * NCW) + p.test_token_bar_extra);
      mbar_init(cbar0 + 8u, static_cast<uint32_t>(G * NCW) + p.test_token_bar_extra);
    } else {
      for (int i = 0; i < 2 * G; ++i) mbar_init(cbar0 + 8u * i, static_cast<uint32_t>(NCW) + p.test_token_bar_extra);
    }
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
    const int jall = tid - kFirstComputeWarp * 32;
    // Groups split the tokens (group g takes tokens g, g + G, ...; every pass) or, in split mode, each
    // token's hidden passes (group g takes pass g of every token).
    const int grp = jall / NCT;
    const int jt = jall - grp * NCT;  // owns 16-byte columns jt + NCT*q of every row
    const int cw = (jall >> 5) - grp * NCW;
    const int tok0 = p.split ? 0 : grp, tstride = p.split ? 1 : G;
    const int pass_lo = p.split ? grp : 0, pass_hi = p.split ? grp + 1 : npass;
    const int nred = p.split ? G * NCW : NCW, ridx = p.split ? grp * NCW + cw : cw;  // sum-of-squares slots
    const float qscale = (p.quant != MFR_QUANT_NONE) ? *p.quant_scale : 1.0f;
    const uint32_t slot0 =
        smem_addr(smem + p.off_stage + static_cast<size_t>(grp) * kNB * p.stage_bytes) + jt * 16;
    const uint32_t slot_end = slot0 + kNB * p.stage_bytes;
    uint8_t* stash = smem + p.off_stash + (p.split ? 0 : static_cast<size_t>(grp) * ((H * 2 + 15) & ~15));
    float* sred = reinterpret_cast<float*>(smem + p.off_sred) + (p.split ? 0 : grp * 64);  // [2][32]
    const uint32_t gcbar = p.split ? cbar0 : cbar0 + 16u * grp;
    // Columns of this thread that fall inside pass ps (bit q for column q).
    auto colmask = [&](int ps) -> uint32_t {
      const int lim = min(W, H - ps * W);
      uint32_t m = 0;
#pragma unroll
      for (int q = 0; q < kQ; ++q)
        if ((jt + q * NCT) * 8 < lim) m |= 1u << q;
      return m;
    };

    // Issue cursor: token ii (local index), pass ip and entry ij of its list (in_n entries).
    int ii = tok0, ip = pass_lo, ij = 0, in_n = -1;
    const RowEntry* ilist = nullptr;
    uint32_t idst = slot0, imask = colmask(pass_lo);
    int64_t ipoff = static_cast<int64_t>(pass_lo) * W * 2 + jt * 16;  // this thread's first column in a row
    int issued = 0;  // rows issued (one commit group each)
    // Consume cursor (the same walk).
    int ci = tok0, cpass = pass_lo, cj = 0, cn = -1;
    const RowEntry* clist = nullptr;
    uint32_t cdst = slot0, cmask = imask;
    int consumed = 0;
    bool ok = true;

    // Issue this thread's columns of the next row, if there is one it may issue: a list is reused only
    // after its token is consumed, so the cursor stays fewer than kLists tokens ahead.
    auto issue_one = [&]() {
      if (!(ok && ii < ntok && ii < ci + kLists)) return;
      if (in_n < 0) {
        const int slot = ii % kLists;
        if (!warp_wait(rfull0 + 8u * slot, static_cast<uint32_t>(ii / kLists) & 1u, abort_flag)) {
          ok = false;
          return;
        }
        const uint8_t* e = ring0 + slot * p.ring_bytes;
        in_n = *reinterpret_cast<const int*>(e);
        ilist = reinterpret_cast<const RowEntry*>(e + 16);
      }
      const uint8_t* row0 = ilist[ij].src;  // NULL: the closing entry of a finalize-only pass (no data)
      const uint32_t m = row0 != nullptr ? imask : 0u;  // (no copy is made from the placeholder address)
      const uint8_t* src = row0 != nullptr ? row0 + ipoff : reinterpret_cast<const uint8_t*>(p.part[0].perm);
#pragma unroll
      for (int q = 0; q < kQ; ++q) cp_async16_if(idst + q * QB, src + q * QB, (m >> q) & 1u);
      cp_async_commit();
      ++issued;
      idst += p.stage_bytes;
      if (idst == slot_end) idst = slot0;
      if (++ij == in_n) {
        ij = 0;
        if (++ip == pass_hi) {
          ip = pass_lo;
          ii += tstride;
          in_n = -1;
        }
        ipoff = static_cast<int64_t>(ip) * W * 2 + jt * 16;
        imask = colmask(ip);
      }
    };

    for (int s = 0; s < kLook; ++s) issue_one();

    float2 acc[kQ * 4], S[kQ * 4];
#pragma unroll
    for (int i = 0; i < kQ * 4; ++i) acc[i] = S[i] = make_float2(0.0f, 0.0f);
    float ss = 0.0f;

    while (ok && ci < ntok) {
      issue_one();
      // This thread's columns of row `consumed` are in the group issued `issued - consumed - 1` groups
      // before the newest; with fewer than kLook rows ahead, wait for all of them.
      if (issued - consumed > kLook) cp_async_wait_group<kLook>();
      else cp_async_wait_all();
      if (!ok) break;
      if (cn < 0) {  // the issue cursor already waited for this token's list
        const uint8_t* e = ring0 + (ci % kLists) * p.ring_bytes;
        cn = *reinterpret_cast<const int*>(e);
        clist = reinterpret_cast<const RowEntry*>(e + 16);
      }
      // The entry: source (unused here), scale and tag.
      const uint4 ent = lds16(smem_addr(clist + cj));
      const float scale = __uint_as_float(ent.z);
      const uint32_t tag = ent.w;
      // Columns outside the pass read as zeros and are never stored, so the arithmetic needs no branch.
      if (!(tag & (kTagShared | kTagResidual))) {  // a routed row: acc += scale * row, fused
        const float2 sc = make_float2(scale, scale);
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
          float2 v[4];
          unpack_pairs<A>(lds16_if(cdst + q * QB, (cmask >> q) & 1u), v);
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[4 * q + c] = __ffma2_rn(sc, v[c], acc[4 * q + c]);
        }
        if (tag & kTagLast) flush_partial<A>(acc, S, false, p.rsf);
      } else if (tag & kTagShared) {  // acc times the factor, rounded, plus the shared row (last)
        // Scalar operations here: a packed multiply followed by a packed add of its result may be
        // contracted into one packed FMA, which rounds once instead of twice.
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
          float2 v[4];
          unpack_pairs<A>(lds16_if(cdst + q * QB, (cmask >> q) & 1u), v);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float2& a = acc[4 * q + c];
            a = make_float2(__fadd_rn(__fmul_rn(a.x, p.rsf), v[c].x), __fadd_rn(__fmul_rn(a.y, p.rsf), v[c].y));
          }
        }
        flush_partial<A>(acc, S, true, p.rsf);
      } else {  // the residual row closes the pass: residual_out = round(round(S) + residual)
        const int t = static_cast<int>(blockIdx.x) + ci * static_cast<int>(gridDim.x);
        const int64_t hoff = static_cast<int64_t>(cpass) * W + jt * 8;  // element of column 0
        if (p.finalize_out != nullptr) {  // the finalized output S, rounded once
#pragma unroll
          for (int q = 0; q < kQ; ++q) {
            if (cmask & (1u << q)) {
              uint32_t w[4];
#pragma unroll
              for (int c = 0; c < 4; ++c) w[c] = Act<A>::pack(S[4 * q + c].x, S[4 * q + c].y);
              *reinterpret_cast<uint4*>(p.finalize_out + (static_cast<int64_t>(t) * H + hoff + q * NCT * 8) * 2) =
                  make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
          if (!p.fin_only && (cmask & (1u << q))) {
            float2 res[4];
            unpack_pairs<A>(lds16(cdst + q * QB), res);
            uint32_t w[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const float2 x = round_pair<A>(__fadd2_rn(round_pair<A>(S[4 * q + c]), res[c]));
              ss = __fmaf_rn(x.x, x.x, ss);  // the squares are exact for 16-bit values
              ss = __fmaf_rn(x.y, x.y, ss);
              w[c] = Act<A>::pack(x.x, x.y);
            }
            const uint4 ro = make_uint4(w[0], w[1], w[2], w[3]);
            const int64_t h = hoff + q * NCT * 8;
            *reinterpret_cast<uint4*>(stash + h * 2) = ro;
            if (p.residual_out != nullptr)
              *reinterpret_cast<uint4*>(p.residual_out + (static_cast<int64_t>(t) * H + h) * 2) = ro;
          }
        }
#pragma unroll
        for (int i = 0; i < kQ * 4; ++i) S[i] = make_float2(0.0f, 0.0f);
      }
      ++consumed;
      cdst += p.stage_bytes;
      if (cdst == slot_end) cdst = slot0;
      if (++cj < cn) continue;
      cj = 0;
      if (++cpass < pass_hi) {
        cmask = colmask(cpass);
        continue;
      }
      cpass = pass_lo;
      cmask = colmask(cpass);

      if (p.fin_only) {  // finalize-only: release the list; no RMSNorm
        __syncwarp();
        if (lane == 0) mbar_arrive(rempty0 + 8u * (ci % kLists));
        ci += tstride;
        cn = -1;
        continue;
      }
      // Token done: release its list, reduce the sum of squares over the group's warps (all compute
      // warps in split mode), in warp order, double-buffered by token parity (the warps meet on an
      // mbarrier so the wait is bounded), and write norm_out and the quantised output from the kept
      // residual_out and gamma.
      __syncwarp();
      if (lane == 0) mbar_arrive(rempty0 + 8u * (ci % kLists));
      const float wsum = warp_sum(ss);
      const int k = ci / tstride;  // the group's k-th token
      float* rb = sred + (k & 1) * 32;
      if (lane == 0) {
        rb[ridx] = wsum;
        mbar_arrive(gcbar + 8u * (k & 1));
      }
      if (!warp_wait(gcbar + 8u * (k & 1), static_cast<uint32_t>(k >> 1) & 1u, abort_flag)) {
        ok = false;
        break;
      }
      float tot = 0.0f;
      for (int w2 = 0; w2 < nred; ++w2) tot = __fadd_rn(tot, rb[w2]);
      const float rstd = rms_rstd(tot, H, p.eps);
      const int t = static_cast<int>(blockIdx.x) + ci * static_cast<int>(gridDim.x);
      for (int ps = pass_lo; ps < pass_hi; ++ps) {
        const uint32_t m = colmask(ps);
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
          const int h = ps * W + (jt + q * NCT) * 8;
          const bool active = (m >> q) & 1u;
          float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, g[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          if (active) {
            unpack8<A>(*reinterpret_cast<const uint4*>(stash + static_cast<int64_t>(h) * 2), x);
            unpack8<A>(ldg16(p.gamma + static_cast<int64_t>(h) * 2), g);
          }
          epilogue<A, 8>(p, t, h, active, x, g, rstd, qscale);
        }
      }
      ss = 0.0f;
      ci += tstride;
      cn = -1;
    }
    cp_async_wait_all();  // no copy of this thread may land after the CTA exits
  }
  __syncthreads();
}

template <typename A, int G>
static cudaError_t launch_stream(const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  auto kern = stream_finalize_kernel<A, G>;
  static std::atomic<int> configured[64] = {};  // per device: the attributes are set (once is enough)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_optin);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev].store(1, std::memory_order_release);
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
static cudaError_t launch_stream_groups(const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  return p.groups == 2 ? launch_stream<A, 2>(p, g, stream) : launch_stream<A, 1>(p, g, stream);
}

cudaError_t launch_stream_kernel(int act_dtype, const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  return act_dtype == MFR_BF16 ? launch_stream_groups<__nv_bfloat16>(p, g, stream)
                               : launch_stream_groups<__half>(p, g, stream);
}

template <typename A, int G>
static int blocks_per_sm(const LaunchGeom& g) {
  auto kern = stream_finalize_kernel<A, G>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_optin);
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, g.block, g.smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int stream_kernel_blocks_per_sm(int act_dtype, int groups, const LaunchGeom& g) {
  if (act_dtype == MFR_BF16)
    return groups == 2 ? blocks_per_sm<__nv_bfloat16, 2>(g) : blocks_per_sm<__nv_bfloat16, 1>(g);
  return groups == 2 ? blocks_per_sm<__half, 2>(g) : blocks_per_sm<__half, 1>(g);
}

cudaError_t read_and_reset_timeouts(unsigned int* count) {
  cudaError_t e = cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(unsigned int));
}

}  // namespace mfr
