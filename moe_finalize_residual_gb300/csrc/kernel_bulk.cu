// Large-batch fused finalize with bulk-copy staging: persistent CTAs (one per SM), each finalizing
// whole tokens in turn; every row the token reads is brought into shared memory by cp.async.bulk
// (non-multicast, from this GPU's own memory), so the compute warps run only the arithmetic.
//
// Roles:
//  - routing warp: for each of the CTA's tokens, up to kLists tokens ahead, it reads the R*K route
//    indices and scales, checks the bound of every index, and writes the token's row list (valid routes
//    in order, each partial's shared row after its routes, the residual row last; see mfr_rowlist.cuh)
//    into a ring of lists, so the index loads never hold up the copies;
//  - copy warp: pass by pass over the hidden dimension it copies the listed rows' slices of the pass
//    into a ring of stages, SR rows per stage: lane 0 posts the stage's byte count on the stage's
//    mbarrier and lanes 0..SR-1 each issue one row's bulk copy, all counted on that barrier.  One
//    barrier per stage, not per row: the barrier operations of one thread cost more than the copies
//    they guard.
//  - compute warps: thread j owns 16-byte columns j, j + NCT, ... of every row of a pass.  Per stage it
//    waits on the stage's barrier, runs the partial's FP32 fused multiply-adds on its columns (or the
//    shared-row step, the rounding of a finished partial into the rank sum, and the residual row that
//    closes the pass), and releases the stage.  After a token's last pass the warps meet on an
//    mbarrier to add their sums of squares in warp order.  The token's norm_out and quantised output
//    are then written from the kept residual_out (two buffers, by token parity) in slices between the
//    next token's stages, so the copy warp's ring keeps draining across the token boundary.
//
// The compute warps are 8 to 14, as the planner chooses for the row width (the row's 16-byte columns
// filling the threads evenly), so a thread's column offsets come from the launch parameters.
//
// Prior art: flashinfer PR #3385 (TMA / mbarrier staging of the RMSNorm inputs); flashinfer PR #6546
// (the large-batch finalizeKernelVecLoad path).  The arithmetic is that of flashinfer PR #6631,
// Description, operation for operation the same as the other kernels'.
//
// Every wait is bounded (about 2 s of device time).  A wait that runs out counts a timeout in device
// memory and raises the CTA's abort flag; the copy warp then waits (bounded) until its issued copies have
// landed before the CTA exits, so no copy writes into the shared memory of a CTA that has left.
#include "mfr_device.cuh"
#include "mfr_launch.h"
#include "mfr_rowlist.cuh"

#include <atomic>

namespace mfr {

__device__ unsigned int g_bulk_wait_timeouts = 0;

namespace {

constexpr uint64_t kLimitNs = 2000000000ull;
constexpr uint32_t kSleepHintNs = 20000;  // a waiting thread sleeps until the phase completes, or about 20 us
constexpr int kLists = 4;                // row lists (tokens) in the ring

// Bounded wait on an mbarrier phase.  Returns false if the CTA is aborting or the limit ran out (then it
// starts the abort).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if ((it & 7u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kLimitNs) {
        atomicAdd(&g_bulk_wait_timeouts, 1u);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool warp_wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag));
}

// One bulk copy global -> this CTA's shared memory, counted on `bar` (bytes and both addresses 16-byte
// aligned).
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Round a finished partial into the rank sum (see the stream kernel: the same operations).
template <typename A, int Q>
__device__ __forceinline__ void flush(float2 acc[Q * 4], float2 S[Q * 4], bool shared_done, float rsf) {
  const float2 f = make_float2(rsf, rsf);
#pragma unroll
  for (int i = 0; i < Q * 4; ++i) {
    const float2 a = shared_done ? acc[i] : __fmul2_rn(acc[i], f);
    S[i] = __fadd2_rn(S[i], round_pair<A>(a));
    acc[i] = make_float2(0.0f, 0.0f);
  }
}

}  // namespace

// Q: 16-byte columns per compute thread per pass (the pass covers 8 * NCT * Q elements at most, NCT the
// compute threads of the launch: p.compute_warps warps, chosen so the columns fill them evenly).
template <typename A, int Q>
__global__ void __launch_bounds__(32 * (2 + kBulkMaxComputeWarps), 1) bulk_finalize_kernel(const __grid_constant__ KParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int H = p.H, W = p.chunk;
  const int npass = (H + W - 1) / W;
  const int NST = p.stages, SR = p.stage_rows;
  const int kNCW = p.compute_warps;  // compute warps
  const int kNCT = 32 * kNCW;        // compute threads

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  const uint32_t full0 = smem_addr(bars);                 // NST: a stage's rows have landed
  const uint32_t empty0 = full0 + 8u * NST;               // NST: a stage is free (one arrival per compute warp)
  const uint32_t lfull0 = empty0 + 8u * NST;              // kLists: a row list is written
  const uint32_t lempty0 = lfull0 + 8u * kLists;          // kLists: a row list is released
  const uint32_t meet0 = lempty0 + 8u * kLists;           // 2: the compute warps' sums of squares (by parity)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * NST + 2 * kLists + 2);
  uint8_t* ring0 = smem + p.off_ring;
  const uint32_t stage0 = smem_addr(smem + p.off_stage);
  const int slot_bytes = p.stage_bytes;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, static_cast<uint32_t>(kNCW));
    }
    for (int i = 0; i < kLists; ++i) {
      mbar_init(lfull0 + 8u * i, 1);
      mbar_init(lempty0 + 8u * i, static_cast<uint32_t>(kNCW) + 1u);  // the compute warps and the copy warp
    }
    // (the failure-detection test hook adds an arrival that never comes, so every wait on these runs out)
    mbar_init(meet0, static_cast<uint32_t>(kNCW) + p.test_token_bar_extra);
    mbar_init(meet0 + 8u, static_cast<uint32_t>(kNCW) + p.test_token_bar_extra);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const int G = static_cast<int>(gridDim.x);
  const int ntok = (p.T - static_cast<int>(blockIdx.x) + G - 1) / G;
  // With the caller's leave to read the routing before the dependency wait, the first token's row list
  // is built before it.
  const bool early_list = p.routing_early && ntok > 0;
  if (p.pdl) pdl_launch_dependents();
  if (warp == 0 && early_list) {
    const int n = build_row_list(p, static_cast<int>(blockIdx.x), reinterpret_cast<RowEntry*>(smem + p.off_ring + 16),
                                 lane);
    if (lane == 0) *reinterpret_cast<int*>(smem + p.off_ring) = n;
    __syncwarp();
    if (lane == 0) mbar_arrive(lfull0);
  }
  if (p.pdl) pdl_wait();

  if (warp == 0) {
    // ---------------- routing warp ----------------
    for (int i = early_list ? 1 : 0; i < ntok; ++i) {
      const int slot = i % kLists;
      if (i >= kLists && !warp_wait_phase(lempty0 + 8u * slot, (static_cast<uint32_t>(i / kLists) & 1u) ^ 1u,
                                          abort_flag))
        break;
      uint8_t* e = ring0 + slot * p.ring_bytes;
      const int n = build_row_list(p, static_cast<int>(blockIdx.x) + i * G, reinterpret_cast<RowEntry*>(e + 16), lane);
      if (lane == 0) *reinterpret_cast<int*>(e) = n;
      __syncwarp();
      if (lane == 0) mbar_arrive(lfull0 + 8u * slot);
    }
  } else if (warp == 1) {
    // ---------------- copy warp ----------------
    uint32_t pc = 0;        // stages issued so far
    int ws = 0;             // the stage the next copies go to
    uint32_t wround = 0;    // how many times the ring has been filled before (for the free-stage wait)
    bool ok = true;
    for (int i = 0; i < ntok && ok; ++i) {
      const int slot = i % kLists;
      if (!warp_wait_phase(lfull0 + 8u * slot, static_cast<uint32_t>(i / kLists) & 1u, abort_flag)) break;
      const uint8_t* e = ring0 + slot * p.ring_bytes;
      const RowEntry* list = reinterpret_cast<const RowEntry*>(e + 16);
      const int n = *reinterpret_cast<const int*>(e);
      for (int ps = 0; ps < npass && ok; ++ps) {
        const int64_t off = static_cast<int64_t>(ps) * W * 2;
        const uint32_t bytes = static_cast<uint32_t>(min(W, H - ps * W)) * 2u;
        for (int j0 = 0; j0 < n; j0 += SR, ++pc) {
          const int s = ws;
          if (wround > 0 && !warp_wait_phase(empty0 + 8u * s, (wround & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          if (++ws == NST) {
            ws = 0;
            ++wround;
          }
          const int cnt = min(SR, n - j0);
          const uint8_t* src = (lane < cnt) ? list[j0 + lane].src : nullptr;  // NULL: a closing entry, no data
          const uint32_t with_data = __ballot_sync(0xffffffffu, src != nullptr);
          const uint32_t fb = full0 + 8u * s;
          if (lane == 0) mbar_arrive_expect_tx(fb, static_cast<uint32_t>(__popc(with_data)) * bytes);
          __syncwarp();
          if (src != nullptr)
            bulk_copy(stage0 + static_cast<uint32_t>((s * SR + lane) * slot_bytes), src + off, bytes, fb);
        }
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(lempty0 + 8u * slot);  // the copy warp no longer reads the list
    }
    // No copy may land after the CTA exits: wait (bounded, whatever the abort flag says) until the latest
    // phase of every stage issued has completed.
    if (lane == 0) {
      const uint32_t last = pc < static_cast<uint32_t>(NST) ? pc : static_cast<uint32_t>(NST);
      for (uint32_t q = 0; q < last; ++q) {
        const uint32_t c = pc - 1u - q;
        const uint32_t bar = full0 + 8u * (c % static_cast<uint32_t>(NST));
        const uint32_t par = (c / static_cast<uint32_t>(NST)) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar, par))
          if (global_timer_ns() - t0 > kLimitNs) {
            atomicAdd(&g_bulk_wait_timeouts, 1u);
            break;
          }
      }
    }
  } else {
    // ---------------- compute warps ----------------
    const int jt = tid - 64;                  // owns 16-byte columns jt + kNCT * q of a pass
    const int cw = warp - 2;
    const float qscale = (p.quant != MFR_QUANT_NONE) ? *p.quant_scale : 1.0f;
    uint8_t* stash0 = smem + p.off_stash;     // [2][H]: a token's residual_out, by token parity, for its epilogue
    float* sred = reinterpret_cast<float*>(smem + p.off_sred);  // [2][32] warp sums by token parity
    auto colmask = [&](int ps) -> uint32_t {
      const int lim = min(W, H - ps * W);
      uint32_t m = 0;
#pragma unroll
      for (int q = 0; q < Q; ++q)
        if ((jt + q * kNCT) * 8 < lim) m |= 1u << q;
      return m;
    };
    // A token's epilogue (norm_out and the quantised output) runs while the next token's rows stream in:
    // one slice (one column of one pass) after each stage the warp releases, the rest before that
    // token's own sums of squares meet.  Each thread reads back only the stash columns it wrote, and the
    // two stash buffers alternate by token, so the slices need no barrier.
    int pend_t = -1;           // token whose epilogue is pending, or -1
    int pend_i = 0;            // its place in this CTA's sequence (stash parity)
    int pend_k = 0;            // its next slice: pass pend_k / Q, column pend_k % Q
    float pend_rstd = 0.0f;
    const int nslices = npass * Q;
    auto epi_slice = [&]() {
      const int ps = pend_k / Q, q = pend_k - ps * Q;
      const int h = ps * W + (jt + q * kNCT) * 8;
      const bool active = (colmask(ps) >> q) & 1u;
      const uint8_t* st = stash0 + static_cast<int64_t>(pend_i & 1) * H * 2;
      float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, g[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (active) {
        unpack8<A>(*reinterpret_cast<const uint4*>(st + static_cast<int64_t>(h) * 2), x);
        unpack8<A>(ldg16(p.gamma + static_cast<int64_t>(h) * 2), g);
      }
      epilogue<A, 8>(p, pend_t, h, active, x, g, pend_rstd, qscale);  // all lanes (NVFP4 shuffles)
      ++pend_k;
    };
    float2 acc[Q * 4], S[Q * 4];
#pragma unroll
    for (int i = 0; i < Q * 4; ++i) acc[i] = S[i] = make_float2(0.0f, 0.0f);
    int cs = 0;          // the stage the next rows are in
    uint32_t cpar = 0;   // its barrier's phase parity
    bool ok = true;
    for (int i = 0; i < ntok && ok; ++i) {
      const int t = static_cast<int>(blockIdx.x) + i * G;
      const int slot = i % kLists;
      if (!warp_wait_phase(lfull0 + 8u * slot, static_cast<uint32_t>(i / kLists) & 1u, abort_flag)) break;
      const uint8_t* e = ring0 + slot * p.ring_bytes;
      const int n = *reinterpret_cast<const int*>(e);
      const RowEntry* list = reinterpret_cast<const RowEntry*>(e + 16);
      uint8_t* stash = stash0 + static_cast<int64_t>(i & 1) * H * 2;
      float ss = 0.0f;
      for (int ps = 0; ps < npass && ok; ++ps) {
        const uint32_t cmask = colmask(ps);
        // Byte offset of column q of this thread within a row slot.  Columns outside the pass read column
        // 0 of the row instead (inside the slot whatever its width): what they accumulate is never stored
        // or added to the sum of squares.
        uint32_t col_off[Q];
#pragma unroll
        for (int q = 0; q < Q; ++q)
          col_off[q] = ((cmask >> q) & 1u) ? static_cast<uint32_t>((jt + q * kNCT) * 16) : 0u;
        const uint32_t list_s = smem_addr(list);
        for (int j0 = 0; j0 < n; j0 += SR) {
          const int s = cs;
          if (!warp_wait_phase(full0 + 8u * s, cpar, abort_flag)) {
            ok = false;
            break;
          }
          const int cnt = min(SR, n - j0);
          uint32_t row = stage0 + static_cast<uint32_t>(s * SR * slot_bytes);  // the row's slot
          uint32_t ent_s = list_s + 16u * j0;
          for (int jj = 0; jj < cnt; ++jj, row += slot_bytes, ent_s += 16u) {
            const uint4 ent = lds16(ent_s);  // source (unused here), scale, tag
            const float scale = __uint_as_float(ent.z);
            const uint32_t tag = ent.w;
            if (!(tag & (kTagShared | kTagResidual))) {  // a routed row: acc += scale * row, fused
              const float2 sc = make_float2(scale, scale);
#pragma unroll
              for (int q = 0; q < Q; ++q) {
                float2 v[4];
                unpack_pairs<A>(lds16(row + col_off[q]), v);
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[4 * q + c] = __ffma2_rn(sc, v[c], acc[4 * q + c]);
              }
              if (tag & kTagLast) flush<A, Q>(acc, S, false, p.rsf);
            } else if (tag & kTagShared) {  // acc times the factor, then plus the shared row (scalar ops:
                                            // never contracted into one fused multiply-add)
#pragma unroll
              for (int q = 0; q < Q; ++q) {
                float2 v[4];
                unpack_pairs<A>(lds16(row + col_off[q]), v);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                  float2& a = acc[4 * q + c];
                  a = make_float2(__fadd_rn(__fmul_rn(a.x, p.rsf), v[c].x), __fadd_rn(__fmul_rn(a.y, p.rsf), v[c].y));
                }
              }
              flush<A, Q>(acc, S, true, p.rsf);
            } else {  // the residual row closes the pass: residual_out = round(round(S) + residual)
              const int64_t hoff = static_cast<int64_t>(ps) * W + jt * 8;
#pragma unroll
              for (int q = 0; q < Q; ++q) {
                if (!(cmask & (1u << q))) continue;
                const int64_t h = hoff + q * kNCT * 8;
                if (p.finalize_out != nullptr) {  // the finalized output S, rounded once
                  uint32_t w[4];
#pragma unroll
                  for (int c = 0; c < 4; ++c) w[c] = Act<A>::pack(S[4 * q + c].x, S[4 * q + c].y);
                  *reinterpret_cast<uint4*>(p.finalize_out + (static_cast<int64_t>(t) * H + h) * 2) =
                      make_uint4(w[0], w[1], w[2], w[3]);
                }
                if (p.fin_only) continue;  // (the closing entry of a finalize-only pass holds no data)
                float2 res[4];
                unpack_pairs<A>(lds16(row + col_off[q]), res);
                uint32_t w[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                  const float2 x = round_pair<A>(__fadd2_rn(round_pair<A>(S[4 * q + c]), res[c]));
                  ss = __fmaf_rn(x.x, x.x, ss);  // the squares are exact for 16-bit values
                  ss = __fmaf_rn(x.y, x.y, ss);
                  w[c] = Act<A>::pack(x.x, x.y);
                }
                const uint4 ro = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(stash + h * 2) = ro;
                if (p.residual_out != nullptr)
                  *reinterpret_cast<uint4*>(p.residual_out + (static_cast<int64_t>(t) * H + h) * 2) = ro;
              }
#pragma unroll
              for (int k = 0; k < Q * 4; ++k) S[k] = make_float2(0.0f, 0.0f);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(empty0 + 8u * s);
          if (++cs == NST) {
            cs = 0;
            cpar ^= 1u;
          }
          if (pend_t >= 0 && pend_k < nslices) epi_slice();  // the previous token's epilogue, a slice
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(lempty0 + 8u * slot);  // the list is no longer read
      while (pend_t >= 0 && pend_k < nslices) epi_slice();
      if (p.fin_only) continue;
      // Token done: add the warps' sums of squares in warp order (the warps meet on an mbarrier,
      // double-buffered by token parity, so the wait is bounded), then norm_out and the quantised output.
      const float wsum = warp_sum(ss);
      float* rb = sred + (i & 1) * 32;
      if (lane == 0) {
        rb[cw] = wsum;
        mbar_arrive(meet0 + 8u * (i & 1));
      }
      if (!warp_wait_phase(meet0 + 8u * (i & 1), static_cast<uint32_t>(i >> 1) & 1u, abort_flag)) {
        ok = false;
        break;
      }
      float tot = 0.0f;
      for (int w2 = 0; w2 < kNCW; ++w2) tot = __fadd_rn(tot, rb[w2]);
      pend_rstd = rms_rstd(tot, H, p.eps);
      pend_t = t;
      pend_i = i;
      pend_k = 0;
    }
    if (ok)  // the last token's epilogue
      while (pend_t >= 0 && pend_k < nslices) epi_slice();
  }
  __syncthreads();
}

namespace {

template <typename A, int Q>
cudaError_t launch_bulk(const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  auto kern = bulk_finalize_kernel<A, Q>;
  static std::atomic<int> configured[64] = {};  // per device: the attribute is set (once is enough)
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
cudaError_t launch_bulk_q(const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  switch (p.cols_per_thread) {
    case 1: return launch_bulk<A, 1>(p, g, stream);
    case 2: return launch_bulk<A, 2>(p, g, stream);
    case 3: return launch_bulk<A, 3>(p, g, stream);
    default: return launch_bulk<A, 4>(p, g, stream);
  }
}

template <typename A, int Q>
int blocks_per_sm_q(const LaunchGeom& g) {
  auto kern = bulk_finalize_kernel<A, Q>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_optin);
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, g.block, g.smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <typename A>
int blocks_per_sm_a(int q, const LaunchGeom& g) {
  switch (q) {
    case 1: return blocks_per_sm_q<A, 1>(g);
    case 2: return blocks_per_sm_q<A, 2>(g);
    case 3: return blocks_per_sm_q<A, 3>(g);
    default: return blocks_per_sm_q<A, 4>(g);
  }
}

}  // namespace

cudaError_t launch_bulk_kernel(int act_dtype, const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  return act_dtype == MFR_BF16 ? launch_bulk_q<__nv_bfloat16>(p, g, stream) : launch_bulk_q<__half>(p, g, stream);
}

int bulk_kernel_blocks_per_sm(int act_dtype, int cols_per_thread, const LaunchGeom& g) {
  return act_dtype == MFR_BF16 ? blocks_per_sm_a<__nv_bfloat16>(cols_per_thread, g)
                               : blocks_per_sm_a<__half>(cols_per_thread, g);
}

cudaError_t read_and_reset_bulk_timeouts(unsigned int* count) {
  cudaError_t e = cudaMemcpyFromSymbol(count, g_bulk_wait_timeouts, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_bulk_wait_timeouts, &zero, sizeof(unsigned int));
}

}  // namespace mfr
