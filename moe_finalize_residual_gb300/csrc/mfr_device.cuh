// Device-side pieces shared by the two finalize kernels: launch parameters, inline-PTX wrappers
// (cp.async, bulk copies, mbarriers, cluster barriers and DSMEM, programmatic dependent launch),
// activation-type traits, the per-slot routing metadata and the fused epilogue (RMSNorm output and
// FP8 / NVFP4 quantisation).
//
// Arithmetic follows the fused MoE finalize of flashinfer PR #6631 "perf(comm): gather MoE-finalize
// routes together and accumulate in FP32" (Description) and TensorRT-LLM PR #16778 (Fix): FP32
// fused multiply-add chain over the routes in order, times the routed scaling factor, plus the
// shared-expert row, one rounding per partial, FP32 rank sum in rank order, one rounding, residual
// add, RMSNorm on the rounded residual.  Every FP32 operation uses an explicitly rounded intrinsic
// (__fmaf_rn, __fmul_rn, __fadd_rn, __fdiv_rn, __fsqrt_rn) so the compiler cannot contract or
// reassociate it.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_finalize.h"

namespace mfr {

// ------------------------------------------------------------------------------------------------
// Launch parameters (passed by value as a __grid_constant__ kernel parameter)
// ------------------------------------------------------------------------------------------------

struct KPartial {
  const uint8_t* gemm2;   // [rows, H] act
  int64_t rows;
  const int32_t* perm;    // [T, K]
  const void* scale;      // [T, K] scale dtype, or nullptr
  const uint8_t* shared;  // [T, H] act, or nullptr
};

struct KParams {
  KPartial part[MFR_MAX_PARTIALS];
  const uint8_t* residual;
  const uint8_t* gamma;
  uint8_t* residual_out;
  uint8_t* norm_out;
  uint8_t* quant_out;
  uint8_t* sf_out;
  const float* quant_scale;
  int32_t T, H, K, R;
  int32_t scale_dtype;
  int32_t quant;
  int32_t sf_layout;
  uint32_t shared_mask;   // bit r set: partial r has a shared-expert row
  int32_t nslots;         // sum over r of (K + has_shared_r): every row a token may read
  int32_t pdl;            // launched with programmatic dependent launch
  int32_t routing_early;  // routing may be read before the dependency wait
  float rsf, eps;
  // cluster kernel
  int32_t slice_vec;      // 16-byte vectors of hidden per CTA (the last CTA may hold fewer)
  int32_t off_zero, off_src, off_meta, off_shoff, off_red;
  // stream kernel
  int32_t chunk;          // hidden elements per pipeline stage
  int32_t stages;         // pipeline depth
  int32_t rdepth;         // routing ring depth (tokens)
  int32_t stage_bytes;    // bytes of one stage: (nslots + 1 residual) * chunk * 2
  int32_t ring_bytes;     // bytes of one routing ring entry
  int32_t off_bar, off_stage, off_ring, off_zero_s, off_gamma, off_stash, off_sred;
};

// ------------------------------------------------------------------------------------------------
// PTX wrappers
// ------------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch (sm_90+): let the next kernel on the stream launch now / wait until
// the preceding kernel has completed and its memory is visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// 16-byte asynchronous global -> shared copy through L2 (bypassing L1).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bulk (non-tensor) global -> shared copy completing on an mbarrier.  Addresses 16-byte aligned,
// size a multiple of 16.  No multicast: the destination is this CTA's own shared memory.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Thread-block clusters.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Read a float from the shared memory of CTA `rank` of this cluster at the address that `local`
// has in this CTA.
__device__ __forceinline__ float dsmem_load_f32(const float* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint2 ldg8(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ void stg8(uint8_t* p, uint2 v) { *reinterpret_cast<uint2*>(p) = v; }

// Deterministic butterfly sum over the 32 lanes of a warp.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ------------------------------------------------------------------------------------------------
// Activation types (16-bit): unpack a pair, round-to-nearest-even back
// ------------------------------------------------------------------------------------------------

template <typename T>
struct Act;

template <>
struct Act<__nv_bfloat16> {
  static __device__ __forceinline__ float2 unpack(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
  }
  static __device__ __forceinline__ float round(float a) { return __bfloat162float(__float2bfloat16_rn(a)); }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};

template <>
struct Act<__half> {
  static __device__ __forceinline__ float2 unpack(uint32_t u) {
    return __half22float2(*reinterpret_cast<const __half2*>(&u));
  }
  static __device__ __forceinline__ float round(float a) { return __half2float(__float2half_rn(a)); }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};

template <typename A>
__device__ __forceinline__ void unpack4(uint2 raw, float v[4]) {
  float2 a = Act<A>::unpack(raw.x), b = Act<A>::unpack(raw.y);
  v[0] = a.x;
  v[1] = a.y;
  v[2] = b.x;
  v[3] = b.y;
}

__device__ __forceinline__ float load_scale(const void* base, int64_t i, int dtype) {
  if (base == nullptr) return 1.0f;  // absent expert scales read as 1.0
  if (dtype == MFR_FP32) return static_cast<const float*>(base)[i];
  const uint16_t b = static_cast<const uint16_t*>(base)[i];
  return dtype == MFR_BF16 ? __uint_as_float(static_cast<uint32_t>(b) << 16) : __half2float(__ushort_as_half(b));
}

// ------------------------------------------------------------------------------------------------
// Routing metadata.  Every row a token may read is a "slot": routes are slots r*K + k, the shared
// rows of the partials that have one follow as slots R*K + 0, 1, ...  A kernel stages slot s at byte
// offset s * stride of its stage and describes the token by a table:
//   meta[r*K + k] = {byte offset of the route's row in the stage, or -1 if the route is skipped;
//                    bits of its FP32 scale, or of -0.0f if skipped}
//   sh_off[r]     = byte offset of partial r's shared row, or -1.
// A skipped route reads a row of zeros with scale -0.0: fma(-0.0, +0.0, acc) == acc for every acc
// (including -0, infinities and NaN), so skipping costs no branch and changes no bit.
// ------------------------------------------------------------------------------------------------

__device__ __forceinline__ int shared_slot(const KParams& p, int r) {
  return p.R * p.K + __popc(p.shared_mask & ((1u << r) - 1u));
}

struct SlotSource {
  const uint8_t* src;  // row start in global memory (hidden index 0); nullptr if skipped
  float scale;
  int r, k;            // partial and route (k == -1 for a shared row)
};

// flashinfer PR #6631, Test changes: routes set to -1 contribute nothing; one bound check per route.
__device__ __forceinline__ SlotSource slot_source(const KParams& p, int s, int t) {
  SlotSource o;
  if (s < p.R * p.K) {
    o.r = s / p.K;
    o.k = s - o.r * p.K;
    const KPartial& P = p.part[o.r];
    const int64_t e = static_cast<int64_t>(t) * p.K + o.k;
    const int32_t idx = P.perm[e];
    const bool valid = idx >= 0 && static_cast<int64_t>(idx) < P.rows;
    o.src = valid ? P.gemm2 + static_cast<int64_t>(idx) * p.H * 2 : nullptr;
    o.scale = valid ? load_scale(P.scale, e, p.scale_dtype) : -0.0f;
  } else {
    int j = s - p.R * p.K;  // j-th partial with a shared row
    uint32_t m = p.shared_mask;
    for (; j > 0; --j) m &= m - 1u;
    o.r = __ffs(m) - 1;
    o.k = -1;
    o.src = p.part[o.r].shared + static_cast<int64_t>(t) * p.H * 2;
    o.scale = 1.0f;
  }
  return o;
}

// Finalize 4 consecutive elements (byte column `col` of every staged row): for each partial the FP32
// fused multiply-add chain over its routes in order k = 0..K-1 starting from +0, times the routed
// scaling factor, plus the shared row, rounded once to act; the rounded partials are added to S in
// rank order 0..R-1 (flashinfer PR #6631, Description; TensorRT-LLM PR #16778, Fix; flashinfer PR
// #3385, fixed rank order).  The R chains are independent until the rank sum, so they advance
// together, route by route, which gives each thread 4*R independent FMA chains.
template <typename A, int RMAX>
__device__ __forceinline__ void finalize4(const int2* __restrict__ meta, const int* __restrict__ sh_off,
                                          const uint8_t* stage, const uint8_t* zero_row, int col, int R, int K,
                                          float rsf, float S[4]) {
  float acc[RMAX][4];
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[r][i] = 0.0f;
  }
#pragma unroll 2
  for (int k = 0; k < K; ++k) {
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      if (r < R) {
        const int2 m = meta[r * K + k];
        const uint8_t* row = (m.x >= 0) ? stage + m.x : zero_row;
        float v[4];
        unpack4<A>(*reinterpret_cast<const uint2*>(row + col), v);
        const float sc = __int_as_float(m.y);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[r][i] = __fmaf_rn(sc, v[i], acc[r][i]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    if (r < R) {
      const int so = sh_off[r];
      float sh[4] = {0.f, 0.f, 0.f, 0.f};
      if (so >= 0) unpack4<A>(*reinterpret_cast<const uint2*>(stage + so + col), sh);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float a = __fmul_rn(acc[r][i], rsf);
        if (so >= 0) a = __fadd_rn(a, sh[i]);
        S[i] = __fadd_rn(S[i], Act<A>::round(a));  // p_r rounded once, summed in FP32 in rank order
      }
    }
  }
}

// residual_out = round(round(S) + residual); returns the 4 values and adds their squares to ss.
template <typename A>
__device__ __forceinline__ uint2 residual_step(const float S[4], uint2 res_raw, float x[4], float& ss) {
  float r[4];
  unpack4<A>(res_raw, r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[i] = Act<A>::round(__fadd_rn(Act<A>::round(S[i]), r[i]));
    ss = __fmaf_rn(x[i], x[i], ss);  // x*x is exact for 16-bit x, so this equals ss + x*x
  }
  return make_uint2(Act<A>::pack(x[0], x[1]), Act<A>::pack(x[2], x[3]));
}

// rstd = 1 / sqrt(sum/H + eps), each operation correctly rounded.
__device__ __forceinline__ float rms_rstd(float sum_sq, int H, float eps) {
  const float ms = __fdiv_rn(sum_sq, static_cast<float>(H));
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
}

// NVFP4 block-scale byte offset of (row m, 16-element block k) (flashinfer PR #3385: LINEAR and
// SWIZZLED_128x4 layouts; the 128x4 tile arrangement as in the public cuBLAS block-scaling layout).
__device__ __forceinline__ int64_t sf_offset(int64_t m, int64_t k, int H, int layout) {
  const int64_t cols = H / 16;
  if (layout == MFR_SF_ROW_MAJOR) return m * cols + k;
  const int64_t col_tiles = (cols + 3) / 4;
  const int64_t r = m & 127;
  return ((m >> 7) * col_tiles + (k >> 2)) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (k & 3);
}

// The epilogue for 4 consecutive hidden elements h..h+3 of token t held by one thread: norm_out
// = round((x * rstd) * gamma), then optional FP8 / NVFP4 quantisation of the rounded values.
// All 32 lanes of the warp must call it together (NVFP4 blocks span 4 adjacent lanes); lanes with
// active == false contribute nothing and write nothing.
template <typename A>
__device__ __forceinline__ void epilogue4(const KParams& p, int64_t t, int h, bool active, const float x[4],
                                          uint2 gamma_raw, float rstd, float qscale) {
  float g[4], y[4];
  unpack4<A>(gamma_raw, g);
#pragma unroll
  for (int i = 0; i < 4; ++i) y[i] = Act<A>::round(__fmul_rn(__fmul_rn(x[i], rstd), g[i]));
  const int64_t e = t * p.H + h;
  if (active && p.norm_out != nullptr)
    stg8(p.norm_out + e * 2, make_uint2(Act<A>::pack(y[0], y[1]), Act<A>::pack(y[2], y[3])));
  if (p.quant == MFR_QUANT_FP8_E4M3) {
    if (active) {
      uint32_t q = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        q |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fmul_rn(y[i], qscale), __NV_SATFINITE, __NV_E4M3))
             << (8 * i);
      *reinterpret_cast<uint32_t*>(p.quant_out + e) = q;
    }
  } else if (p.quant == MFR_QUANT_NVFP4) {
    float amax = 0.0f;
    if (active) {
#pragma unroll
      for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(y[i]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const __nv_fp8_storage_t sf =
        __nv_cvt_float_to_fp8(__fmul_rn(__fdiv_rn(amax, 6.0f), qscale), __NV_SATFINITE, __NV_E4M3);
    const float sf_val = __half2float(__half(__nv_cvt_fp8_to_halfraw(sf, __NV_E4M3)));
    const float es = (sf_val == 0.0f) ? 0.0f : __fdiv_rn(qscale, sf_val);
    if (active) {
      const uint32_t c01 = __nv_cvt_float2_to_fp4x2(make_float2(__fmul_rn(y[0], es), __fmul_rn(y[1], es)),
                                                    __NV_E2M1, cudaRoundNearest);
      const uint32_t c23 = __nv_cvt_float2_to_fp4x2(make_float2(__fmul_rn(y[2], es), __fmul_rn(y[3], es)),
                                                    __NV_E2M1, cudaRoundNearest);
      *reinterpret_cast<uint16_t*>(p.quant_out + e / 2) = static_cast<uint16_t>(c01 | (c23 << 8));
      if ((h & 15) == 0) p.sf_out[sf_offset(t, h >> 4, p.H, p.sf_layout)] = sf;
    }
  }
}

}  // namespace mfr
