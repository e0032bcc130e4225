// Small-batch fused finalize: one thread-block cluster per token, the hidden dimension split into
// equal slices, one slice per CTA of the cluster; a CTA covers its slice in one or more chunks.
//
// Design (prior art: flashinfer PR #6546, finalizeKernelSmallBatch, Description -- one CTA per
// (token, hidden slice), 128-bit loads, top-K work split over thread groups combined through shared
// memory, PDL trigger at kernel start (here after the gather, which measured faster); flashinfer PR
// #6631, Description -- load the indices and scales of the routes first, then all rows, so the row
// loads are in flight together):
//
//  * a CTA covers NCH chunks of SV 16-byte vectors of the token's hidden row; its threads form R groups
//    of SV, one group per partial: thread (r, v) owns vector v of each chunk of partial r.  With few
//    tokens a CTA holds one chunk and the row is spread over up to 16 CTAs; with more tokens fewer
//    CTAs per token loop over several chunks, so the grid stays about two CTAs per SM in one wave;
//  * each thread reads the route indices and scales of its partial (the same addresses for the whole
//    warp), then issues all its rows as 128-bit loads at once (up to KC in flight; K > KC repeats),
//    and runs the FP32 fused multiply-add chain over them in route order, then the factor and the
//    shared-expert row: every partial row is produced by one thread in the definition's order, so it
//    is bit-exact;
//  * the shared-expert, residual and gamma slices of every chunk are copied into shared memory (by
//    cp.async, before the row loads);
//    each group writes its rounded partial rows to shared memory (one buffer per chunk, so one barrier
//    serves all chunks); the (chunk, vector) items are then spread over all threads for the rank sum
//    in order (the shared-memory combine) and the residual add, residual_out kept in shared memory;
//  * the sum of squares is reduced with a warp butterfly, then a butterfly over the warp sums, then
//    across the cluster's CTAs: each CTA sends its sum into a slot of every peer's shared memory with
//    st.async, counted on the peer's mbarrier, and once its own mbarrier has all C sums every CTA adds
//    the slots by the same fixed butterfly, so all get the same deterministic total; then all threads
//    write residual_out, norm_out and the quantised output.
//
// No CTA waits on a flag in global memory.  Across CTAs there is the hardware cluster barrier at entry
// (every CTA reaches it unconditionally) and the exchange's mbarrier, whose wait is bounded.
#include "mfr_device.cuh"
#include "mfr_launch.h"

#include <atomic>

namespace mfr {

// The token's route table for partial P: entry k holds the row index of route k, or -1 for a route to
// skip (flashinfer PR #6631, Test changes: -1 routes contribute nothing; one bound check per route),
// and the bits of its scale.  Thread v of the partial's group fills entries v, v + SV, ...
__device__ __forceinline__ void fill_routes(const KParams& p, const KPartial& P, int t, int v, int SV, int2* rt) {
  for (int k = v; k < p.K; k += SV) {
    const int64_t e = static_cast<int64_t>(t) * p.K + k;
    const int32_t ix = P.perm[e];
    const float sc = load_scale(P.scale, e, p.scale_dtype);  // independent of the index: both loads in flight
    const bool ok = ix >= 0 && static_cast<int64_t>(ix) < P.rows;
    rt[k] = make_int2(ok ? ix : -1, ok ? __float_as_int(sc) : 0);
  }
}

// Routes k0..k0+KC-1 of the table, all KC rows in flight together, then the FMA chain over them in
// route order (rows of routes with index -1 are neither loaded nor added).  The one-chunk form (small
// batches, at most 256 gathering threads on an SM) keeps the KC table entries in registers and issues
// the row loads under predicates, with no branch between them; the other forms read a route's entry
// again for its FMA, so the indices and scales need no registers while the loads are in flight.
template <typename A, int KC>
__device__ __forceinline__ void gather_chain_regs(const KPartial& P, int H, int K, int vec, const int2* rt, int k0,
                                                  float2 acc[4]) {
  int2 e[KC];
#pragma unroll
  for (int j = 0; j < KC; ++j) e[j] = (k0 + j < K) ? rt[k0 + j] : make_int2(-1, 0);
  const uint8_t* base = P.gemm2 + static_cast<int64_t>(vec) * 16;
  const int64_t row_bytes = static_cast<int64_t>(H) * 2;
  uint4 d[KC];
#pragma unroll
  for (int j = 0; j < KC; ++j) d[j] = ldg16_if(base + static_cast<int64_t>(max(e[j].x, 0)) * row_bytes, e[j].x >= 0);
#pragma unroll
  for (int j = 0; j < KC; ++j) {
    if (e[j].x >= 0) {  // element pairs by the packed FMA, each lane rounded like fmaf
      float2 x[4];
      unpack_pairs<A>(d[j], x);
      const float2 sc = make_float2(__int_as_float(e[j].y), __int_as_float(e[j].y));
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = __ffma2_rn(sc, x[i], acc[i]);
    }
  }
}

template <typename A, int KC>
__device__ __forceinline__ void gather_chain(const KPartial& P, int H, int K, int vec, const int2* rt, int k0,
                                             float2 acc[4]) {
  uint4 d[KC];
#pragma unroll
  for (int j = 0; j < KC; ++j) {
    const int ix = (k0 + j < K) ? rt[k0 + j].x : -1;
    if (ix >= 0) d[j] = ldg16(P.gemm2 + (static_cast<int64_t>(ix) * H + vec * 8) * 2);
  }
  const uint32_t rt_s = smem_addr(rt + k0);
#pragma unroll
  for (int j = 0; j < KC; ++j) {
    if (k0 + j < K) {
      int ix, scb;
      asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(ix), "=r"(scb) : "r"(rt_s + 8u * j) : "memory");
      if (ix >= 0) {  // element pairs by the packed FMA, each lane rounded like fmaf
        float2 x[4];
        unpack_pairs<A>(d[j], x);
        const float2 sc = make_float2(__int_as_float(scb), __int_as_float(scb));
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = __ffma2_rn(sc, x[i], acc[i]);
      }
    }
  }
}

// Waits on the cluster exchange's mbarrier (phase 0) that end early: a wait is bounded at about 2 s of
// device time; one that runs out is counted here and the CTA goes on (its outputs are then wrong, which
// the count reports: moe_finalize_read_timeouts).
__device__ unsigned int g_cluster_wait_timeouts = 0;

__device__ __forceinline__ void cluster_exchange_wait(uint32_t bar) {
  if (mbar_try_wait(bar, 0)) return;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, 0)) return;
    if ((it & 31u) == 0 && global_timer_ns() - t0 > 2000000000ull) {
      if ((threadIdx.x & 31) == 0) atomicAdd(&g_cluster_wait_timeouts, 1u);
      return;
    }
  }
}

// Resident CTAs the compiler must allow for (it sets the register budget): two 512-thread CTAs per SM
// for the 8-routes-in-flight form that loops over chunks; one for the other forms (the one-chunk form
// runs small CTAs, which fit two to an SM all the same, and keeps more in registers).
#ifndef MFR_CLUSTER_MIN_BLOCKS
#define MFR_CLUSTER_MIN_BLOCKS 2
#endif

// SPLIT (one chunk, top-k > 8): each partial's routes are split over S = p.route_groups thread groups of
// SV threads, group s loading routes 8s .. 8s+7 of its vector, so every row is in flight in one round;
// groups s > 0 stage their raw rows in shared memory and group 0 runs the whole chain in route order.
template <typename A, int KC, int MINB, bool REGS, bool SPLIT = false>
__global__ void __launch_bounds__(kClusterMaxThreads, MINB) cluster_finalize_kernel(const __grid_constant__ KParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x;
  const int nthreads = blockDim.x;
  const int SV = p.slice_vec;
  const int NCH = p.nchunk;
  const uint32_t C = cluster_nctarank();
  const uint32_t crank = cluster_ctarank();
  const int t = static_cast<int>(blockIdx.x / C);
  const int H = p.H;
  const int nvec = H >> 3;
  const int S = SPLIT ? p.route_groups : 1;     // route groups per partial
  const int grp = tid / SV;                     // (partial, route group) of this thread
  const int r = SPLIT ? grp / S : grp;          // partial of this thread's group
  const int sg = SPLIT ? grp - r * S : 0;       // its route group: routes 8 * sg .. 8 * sg + 7
  const int v = tid - grp * SV;
  const int vec0 = static_cast<int>(crank) * NCH * SV + v;  // chunk ch holds vector vec0 + ch * SV
  const bool in_part = r < p.R;                 // loads rows of partial r
  const bool in_group = in_part && sg == 0;     // finishes partial r's vector v
  uint4* xch = reinterpret_cast<uint4*>(smem);                // [NCH][R][SV] shared rows, then partial rows
  uint4* res_s = xch + NCH * p.R * SV;                        // [NCH][SV] residual slices, then residual_out
  uint4* gam_s = res_s + NCH * SV;                            // [NCH][SV] gamma slices
  float* red = reinterpret_cast<float*>(smem + p.off_red);    // [0,32) warp sums, [32,34) unused,
                                                              // [34,50) the cluster's CTA sums by rank,
                                                              // [52,54) the exchange's mbarrier
  const KPartial& P = p.part[in_part ? r : 0];
  const bool has_shared = in_group && ((p.shared_mask >> r) & 1u);
  const bool lead_group = r == 0 && sg == 0;    // partial 0's group 0 copies the residual and gamma

  // Every CTA of the cluster arrives here on entry; the matching wait comes before the first write into
  // a peer's shared memory, so no CTA writes into one that has not started.
  // The cluster exchange's mbarrier: it completes once all C CTAs' sums (4 bytes each) have landed here.
  // It is set up before the entry arrive, so a peer that has passed the matching wait may write to it.
  const uint32_t xbar = smem_addr(red + 52);
  if (C > 1 && !p.fin_only && tid == 0) {
    mbar_init(xbar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(xbar, p.xch_tx_bytes);
  }
  if (C > 1 && !p.fin_only) cluster_arrive_relaxed();
  int2* rt = reinterpret_cast<int2*>(smem + p.off_routes) + (in_part ? r : 0) * p.K;  // this partial's routes
  if (p.routing_early && in_part) fill_routes(p, P, t, sg * SV + v, S * SV, rt);
  if (p.pdl) pdl_wait();
  if (!p.routing_early && in_part) fill_routes(p, P, t, sg * SV + v, S * SV, rt);

  // Rows that do not depend on the routing go out first, every chunk's, straight into shared memory.
  // A thread reads a shared row only after waiting for its own copies; the residual and gamma slices
  // are read by any thread, after the barrier that follows every thread's wait.
  for (int ch = 0; ch < NCH; ++ch) {
    const int vec = vec0 + ch * SV;
    if (!in_group || vec >= nvec) break;
    const int64_t off = (static_cast<int64_t>(t) * H + vec * 8) * 2;
    if (has_shared) cp_async16(smem_addr(&xch[(ch * p.R + r) * SV + v]), P.shared + off);
    if (lead_group && !p.fin_only) {
      cp_async16(smem_addr(&res_s[ch * SV + v]), p.residual + off);
      cp_async16(smem_addr(&gam_s[ch * SV + v]), p.gamma + static_cast<int64_t>(vec) * 16);
    }
  }
  cp_async_commit();
  __syncthreads();  // the route table is written

  // Each chunk: the partial's FMA chain over its routes, times the routed scaling factor, plus the
  // shared row, rounded once (the partial row p_r), into the chunk's exchange buffer.
  if constexpr (SPLIT) {
    // One chunk.  Every group loads its 8 routes at once; groups s > 0 stage the raw rows, group 0 adds its
    // own, then (after the barrier) the staged ones, in route order.
    uint4* stage = reinterpret_cast<uint4*>(smem + p.off_split);  // [R][S-1][8][SV]
    const bool live = in_part && vec0 < nvec;
    uint4 d[8];
    const uint8_t* base = P.gemm2 + static_cast<int64_t>(vec0) * 16;
    const int64_t row_bytes = static_cast<int64_t>(H) * 2;
    int2 e[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int k = 8 * sg + j;
      e[j] = (live && k < p.K) ? rt[k] : make_int2(-1, 0);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) d[j] = ldg16_if(base + static_cast<int64_t>(max(e[j].x, 0)) * row_bytes, e[j].x >= 0);
    if (sg > 0 && live) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (e[j].x >= 0) stage[((r * (S - 1) + sg - 1) * 8 + j) * SV + v] = d[j];
    }
    float2 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.0f, 0.0f);
    if (in_group && live) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (e[j].x >= 0) {
          float2 x[4];
          unpack_pairs<A>(d[j], x);
          const float2 sc = make_float2(__int_as_float(e[j].y), __int_as_float(e[j].y));
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i] = __ffma2_rn(sc, x[i], acc[i]);
        }
      }
    }
    __syncthreads();  // the staged rows are written
    if (in_group && live) {
      for (int k = 8; k < p.K; ++k) {
        const int2 ek = rt[k];
        if (ek.x >= 0) {
          float2 x[4];
          unpack_pairs<A>(stage[((r * (S - 1) + k / 8 - 1) * 8 + (k & 7)) * SV + v], x);
          const float2 sc = make_float2(__int_as_float(ek.y), __int_as_float(ek.y));
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i] = __ffma2_rn(sc, x[i], acc[i]);
        }
      }
      cp_async_wait_all();
      uint4* xr = &xch[r * SV + v];
      float shv[8];
      unpack8<A>(*xr, shv);
      float a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        a[i] = __fmul_rn((i & 1) ? acc[i >> 1].y : acc[i >> 1].x, p.rsf);
        if (has_shared) a[i] = __fadd_rn(a[i], shv[i]);
      }
      *xr = make_uint4(Act<A>::pack(a[0], a[1]), Act<A>::pack(a[2], a[3]), Act<A>::pack(a[4], a[5]),
                       Act<A>::pack(a[6], a[7]));
    }
  }
  // A chunk's partial row p_r from the FMA chain: times the routed scaling factor, plus the shared row,
  // rounded once, into the chunk's exchange buffer.
  auto finish_chunk = [&](int ch, float2 acc[4]) {
    uint4* xr = &xch[(ch * p.R + r) * SV + v];
    float shv[8];
    unpack8<A>(*xr, shv);
    // Scalar operations here: a packed multiply followed by a packed add of its result may be
    // contracted into one packed FMA, which rounds once instead of twice.
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      a[i] = __fmul_rn((i & 1) ? acc[i >> 1].y : acc[i >> 1].x, p.rsf);
      if (has_shared) a[i] = __fadd_rn(a[i], shv[i]);
    }
    *xr = make_uint4(Act<A>::pack(a[0], a[1]), Act<A>::pack(a[2], a[3]), Act<A>::pack(a[4], a[5]),
                     Act<A>::pack(a[6], a[7]));
  };
  // The (chunk, vector) items [it0, it1) of this CTA, spread over all its threads (item i to thread i mod
  // the block; consecutive threads take consecutive vectors): rank sum in order 0..R-1, residual add
  // (kept in place of the residual slice for the epilogue), sum of squares.
  const int nitems = NCH * SV;
  const int vbase = static_cast<int>(crank) * NCH * SV;  // the CTA's first vector
  float ss = 0.0f;
  auto items = [&](int it0, int it1) {
    for (int it = it0 + tid; it < it1; it += nthreads) {
      const int ch = it / SV, vv = it - ch * SV;
      if (vbase + it >= nvec) break;  // (vector vbase + it; later items are further along)
      float2 S[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) S[i] = make_float2(0.0f, 0.0f);
      for (int rr = 0; rr < p.R; ++rr) {
        float2 pr[4];
        unpack_pairs<A>(xch[(ch * p.R + rr) * SV + vv], pr);
#pragma unroll
        for (int i = 0; i < 4; ++i) S[i] = __fadd2_rn(S[i], pr[i]);
      }
      if (p.finalize_out != nullptr)  // the finalized output S, rounded once
        *reinterpret_cast<uint4*>(p.finalize_out + (static_cast<int64_t>(t) * H + (vbase + it) * 8) * 2) =
            make_uint4(Act<A>::pack(S[0].x, S[0].y), Act<A>::pack(S[1].x, S[1].y), Act<A>::pack(S[2].x, S[2].y),
                       Act<A>::pack(S[3].x, S[3].y));
      if (p.fin_only) continue;
      float2 res[4];
      unpack_pairs<A>(res_s[it], res);
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 x = round_pair<A>(__fadd2_rn(round_pair<A>(S[i]), res[i]));
        ss = __fmaf_rn(x.x, x.x, ss);  // x*x is exact for 16-bit x, so this equals ss + x*x
        ss = __fmaf_rn(x.y, x.y, ss);
        w[i] = Act<A>::pack(x.x, x.y);
      }
      // kept for the epilogue, which writes it out with norm_out after the cluster exchange (the stores
      // would otherwise sit between the items and the exchange on the critical path)
      res_s[it] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  };
  // The next kernel on the stream may launch once the gather is done (programmatic dependent launch).
  // Triggering after the gather rather than at kernel start measured faster at 16 tokens (4.66 against
  // 5.51 µs, L2-warm) and the same elsewhere: launched at start, the next launches' CTAs pile up on the
  // SMs while this one still gathers.
  if constexpr (SPLIT) {
    cp_async_wait_all();
    __syncthreads();
    if (p.pdl) pdl_launch_dependents();
    items(0, nitems);
  } else {
    for (int ch = 0; ch < NCH; ++ch) {
      const int vec = vec0 + ch * SV;
      if (!in_group || vec >= nvec) break;
      float2 acc[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.0f, 0.0f);
      if constexpr (REGS)
        for (int k0 = 0; k0 < p.K; k0 += KC) gather_chain_regs<A, KC>(P, H, p.K, vec, rt, k0, acc);
      else
        for (int k0 = 0; k0 < p.K; k0 += KC) gather_chain<A, KC>(P, H, p.K, vec, rt, k0, acc);
      if (ch == 0) cp_async_wait_all();
      finish_chunk(ch, acc);
    }
    cp_async_wait_all();
    __syncthreads();
    if (p.pdl) pdl_launch_dependents();
    items(0, nitems);
  }

  if (p.fin_only) return;  // finalize-only: no residual, RMSNorm or quantisation (the same for all threads)

  // Sum of squares: a warp butterfly, then one over the warp sums, then one over the cluster's CTA
  // sums.  Each butterfly has a fixed shape (lane i holds item i, zeros past the end), so the result is
  // the same on every lane and every run, and every warp of every CTA of a cluster adds the same slots
  // the same way: each warp computes the total itself, with no barrier after the exchange.
  ss = warp_sum(ss);
  const int warp = tid >> 5, lane = tid & 31;
  const int nw = nthreads >> 5;
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float tot;
  if (C > 1) {
    cluster_wait_acquire();  // all CTAs of the cluster have started (arrived on entry)
    // Lane c of warp 0 sends the CTA's sum to slot `crank` of CTA c (C <= 16), counted on CTA c's
    // exchange barrier; every warp then waits until its own CTA's barrier has all C sums and adds them.
    // A CTA leaves only after every peer's write into it has landed, and nothing is written into it
    // after that.
    if (warp == 0) {
      const float cta = warp_sum(lane < nw ? red[lane] : 0.0f);
      if (lane < static_cast<int>(C)) st_async_f32(&red[34 + crank], static_cast<uint32_t>(lane), cta, xbar);
    }
    cluster_exchange_wait(xbar);
    tot = warp_sum(lane < static_cast<int>(C) ? red[34 + lane] : 0.0f);
  } else {
    tot = warp_sum(lane < nw ? red[lane] : 0.0f);
  }
  const float rstd = rms_rstd(tot, H, p.eps);
  {
    const float qscale = (p.quant != MFR_QUANT_NONE) ? *p.quant_scale : 1.0f;
    for (int base = 0; base < nitems; base += nthreads) {  // the same trip count for every thread (NVFP4 shuffles)
      const int it = base + tid;
      const bool act = it < nitems && vbase + it < nvec;
      const int vec = vbase + it;
      const uint4 ro = act ? res_s[it] : make_uint4(0, 0, 0, 0);
      if (act && p.residual_out != nullptr)
        *reinterpret_cast<uint4*>(p.residual_out + (static_cast<int64_t>(t) * H + vec * 8) * 2) = ro;
      float x[8], g[8];
      unpack8<A>(ro, x);
      unpack8<A>(act ? gam_s[it] : make_uint4(0, 0, 0, 0), g);
      epilogue<A, 8>(p, t, vec * 8, act, x, g, rstd, qscale);
    }
  }
}

template <typename A, int KC, int MINB, bool REGS = false, bool SPLIT = false>
static cudaError_t launch_cluster(const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  auto kern = cluster_finalize_kernel<A, KC, MINB, REGS, SPLIT>;
  static std::atomic<int> configured[64] = {};  // per device: the attributes are set (once is enough)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_optin);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev].store(1, std::memory_order_release);
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

template <typename A, int KC, int MINB, bool REGS = false, bool SPLIT = false>
static int max_active_clusters(const LaunchGeom& g) {
  auto kern = cluster_finalize_kernel<A, KC, MINB, REGS, SPLIT>;
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

template <typename A, int KC, int MINB, bool REGS = false, bool SPLIT = false>
static int blocks_per_sm(const LaunchGeom& g) {
  auto kern = cluster_finalize_kernel<A, KC, MINB, REGS, SPLIT>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_optin);
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, g.block, g.smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// The plan's form: routes in flight per thread and register budget (see ClusterForm).
template <typename A>
static cudaError_t launch_form(const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  switch (p.cluster_form) {
    case kClusterForm8: return launch_cluster<A, 8, MFR_CLUSTER_MIN_BLOCKS>(p, g, stream);
    case kClusterForm8OneChunk: return launch_cluster<A, 8, 1>(p, g, stream);
    case kClusterForm8Latency: return launch_cluster<A, 8, 1, true>(p, g, stream);
    case kClusterForm8Split: return launch_cluster<A, 8, 1, false, true>(p, g, stream);
    default: return launch_cluster<A, 16, 1>(p, g, stream);
  }
}

cudaError_t launch_cluster_kernel(int act_dtype, const KParams& p, const LaunchGeom& g, cudaStream_t stream) {
  return act_dtype == MFR_BF16 ? launch_form<__nv_bfloat16>(p, g, stream) : launch_form<__half>(p, g, stream);
}

template <typename A>
static int blocks_per_sm_form(int form, const LaunchGeom& g) {
  switch (form) {
    case kClusterForm8: return blocks_per_sm<A, 8, MFR_CLUSTER_MIN_BLOCKS>(g);
    case kClusterForm8OneChunk: return blocks_per_sm<A, 8, 1>(g);
    case kClusterForm8Latency: return blocks_per_sm<A, 8, 1, true>(g);
    case kClusterForm8Split: return blocks_per_sm<A, 8, 1, false, true>(g);
    default: return blocks_per_sm<A, 16, 1>(g);
  }
}

int cluster_kernel_blocks_per_sm(int act_dtype, int form, const LaunchGeom& g) {
  return act_dtype == MFR_BF16 ? blocks_per_sm_form<__nv_bfloat16>(form, g) : blocks_per_sm_form<__half>(form, g);
}

template <typename A>
static int max_active_clusters_form(int form, const LaunchGeom& g) {
  switch (form) {
    case kClusterForm8: return max_active_clusters<A, 8, MFR_CLUSTER_MIN_BLOCKS>(g);
    case kClusterForm8OneChunk: return max_active_clusters<A, 8, 1>(g);
    case kClusterForm8Latency: return max_active_clusters<A, 8, 1, true>(g);
    case kClusterForm8Split: return max_active_clusters<A, 8, 1, false, true>(g);
    default: return max_active_clusters<A, 16, 1>(g);
  }
}

int cluster_kernel_max_active_clusters(int act_dtype, int form, const LaunchGeom& g) {
  return act_dtype == MFR_BF16 ? max_active_clusters_form<__nv_bfloat16>(form, g)
                               : max_active_clusters_form<__half>(form, g);
}

cudaError_t read_and_reset_cluster_timeouts(unsigned int* count) {
  cudaError_t e = cudaMemcpyFromSymbol(count, g_cluster_wait_timeouts, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_cluster_wait_timeouts, &zero, sizeof(unsigned int));
}

}  // namespace mfr
