// Device-side pieces shared by the two finalize kernels: launch parameters, inline-PTX wrappers
// (cp.async, mbarriers, cluster barriers, st.async into a peer's shared memory, programmatic dependent
// launch), activation-type traits, the residual step and the fused epilogue (RMSNorm output and FP8 /
// NVFP4 quantisation).
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
  uint8_t* finalize_out;  // the rounded rank sum S, or NULL
  int32_t fin_only;       // finalize_out is the only output: no residual, RMSNorm or quantisation
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
  int32_t slice_vec;      // cluster kernel: 16-byte vectors per CTA per chunk (the last CTA may hold fewer)
  int32_t nchunk;         // cluster kernel: chunks of slice_vec vectors per CTA
  int32_t route_batch;    // cluster kernel: routes in flight per thread (8 or 16; larger top-k in rounds)
  int32_t cluster_form;   // cluster kernel: the compiled form to launch (ClusterForm)
  int32_t off_routes;     // cluster kernel: shared-memory route table [R][K] (row index or -1, scale)
  int32_t route_groups;   // cluster kernel, split form: thread groups per partial (8 routes each)
  int32_t off_split;      // cluster kernel, split form: staged rows [R][route_groups-1][8][slice_vec]
  int32_t off_red;
  uint32_t xch_tx_bytes;  // cluster kernel: bytes the exchange barrier expects (4 per CTA of the cluster)
  // stream kernel
  int32_t chunk;          // hidden elements per pass
  int32_t stages;         // row buffers in the ring
  int32_t stage_bytes;    // bytes of one row buffer
  int32_t groups;         // stream kernel: groups of compute warps per CTA
  int32_t split;          // stream kernel: groups split each token's hidden passes (else the tokens)
  int32_t ring_bytes;     // bytes of one row-list entry
  int32_t off_bar, off_stage, off_ring, off_stash, off_sred;
  uint32_t test_token_bar_extra;  // stream kernels: arrivals the end-of-token barrier expects beyond their
                                  // warps' (1 only under the failure-detection test hook)
  // bulk-copy kernel (also chunk = pass width, stages, stage_bytes = one row slot, ring_bytes, offsets)
  int32_t stage_rows;       // rows per stage (one mbarrier per stage)
  int32_t cols_per_thread;  // 16-byte columns per compute thread per pass (template parameter)
  int32_t compute_warps;    // bulk-copy kernel: compute warps of the launch
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
// The same copy under a predicate (no branch): nothing is copied when `on` is false.
__device__ __forceinline__ void cp_async16_if(uint32_t dst, const void* src, bool on) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %2, 0;\n @p cp.async.cg.shared.global [%0], [%1], 16;\n}\n" ::"r"(dst),
      "l"(src), "r"(static_cast<int>(on))
      : "memory");
}
// 16-byte shared-memory load under a predicate (zeros when `on` is false).
__device__ __forceinline__ uint4 lds16_if(uint32_t addr, bool on) {
  uint4 v;
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %5, 0;\n mov.b32 %0, 0;\n mov.b32 %1, 0;\n mov.b32 %2, 0;\n"
      " mov.b32 %3, 0;\n @p ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n}\n"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "r"(addr), "r"(static_cast<int>(on))
      : "memory");
  return v;
}
__device__ __forceinline__ uint4 lds16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Wait until at most N of this thread's committed groups are still in flight (groups retire in order).
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

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

// The same test, but the thread may sleep (up to about `hint_ns`) until the phase completes instead of
// returning at once: waiting warps then take no issue slots from the working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
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
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Write a float into the shared memory of CTA `rank` of this cluster, at the address that `local` has
// in this CTA, and count its 4 bytes on that CTA's mbarrier (at the address `local_bar` has here): the
// receiver may read the value once that barrier's phase completes.
__device__ __forceinline__ void st_async_f32(const float* local, uint32_t rank, float v, uint32_t local_bar) {
  uint32_t ra, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_addr(local)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(local_bar), "r"(rank));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(ra),
               "r"(__float_as_uint(v)), "r"(rb)
               : "memory");
}

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

// 8 act values as 4 FP32 pairs, for the packed FP32 operations of sm_100 and later (__ffma2_rn and
// friends round each lane exactly like the scalar operation).
template <typename A>
__device__ __forceinline__ void unpack_pairs(uint4 raw, float2 v[4]) {
  v[0] = Act<A>::unpack(raw.x);
  v[1] = Act<A>::unpack(raw.y);
  v[2] = Act<A>::unpack(raw.z);
  v[3] = Act<A>::unpack(raw.w);
}

// Round both lanes to act and back to FP32.
template <typename A>
__device__ __forceinline__ float2 round_pair(float2 a) {
  return Act<A>::unpack(Act<A>::pack(a.x, a.y));
}

template <typename A>
__device__ __forceinline__ void unpack8(uint4 raw, float v[8]) {
  unpack4<A>(make_uint2(raw.x, raw.y), v);
  unpack4<A>(make_uint2(raw.z, raw.w), v + 4);
}

__device__ __forceinline__ uint4 ldg16(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
// 16-byte read-only global load under a predicate, with no branch (zeros when `on` is false; the address
// is then not read).  Volatile, so it stays after the dependency wait, but with no memory clobber, so the
// loads of a round issue back to back.
__device__ __forceinline__ uint4 ldg16_if(const uint8_t* p, bool on) {
  uint4 v;
  asm volatile(
      "{\n .reg .pred q;\n setp.ne.b32 q, %5, 0;\n mov.b32 %0, 0;\n mov.b32 %1, 0;\n mov.b32 %2, 0;\n"
      " mov.b32 %3, 0;\n @q ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\n}\n"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p), "r"(static_cast<int>(on)));
  return v;
}

__device__ __forceinline__ float load_scale(const void* base, int64_t i, int dtype) {
  if (base == nullptr) return 1.0f;  // absent expert scales read as 1.0
  if (dtype == MFR_FP32) return static_cast<const float*>(base)[i];
  const uint16_t b = static_cast<const uint16_t*>(base)[i];
  return dtype == MFR_BF16 ? __uint_as_float(static_cast<uint32_t>(b) << 16) : __half2float(__ushort_as_half(b));
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

// The epilogue for N (4 or 8) consecutive hidden elements h..h+N-1 of token t held by one thread:
// norm_out = round((x * rstd) * gamma), then optional FP8 / NVFP4 quantisation of the rounded values.
// All 32 lanes of the warp must call it together (an NVFP4 block spans 16/N adjacent lanes); lanes
// with active == false contribute nothing and write nothing.
template <typename A, int N>
__device__ __forceinline__ void epilogue(const KParams& p, int64_t t, int h, bool active, const float x[N],
                                         const float g[N], float rstd, float qscale) {
  static_assert(N == 4 || N == 8, "4 or 8 elements per thread");
  // (x * rstd) * gamma by packed FP32 multiplies (each lane rounded like __fmul_rn; two multiplies are
  // never contracted).  Packing to act rounds each value to nearest-even, as rounding first would.
  float y[N];
  const float2 r2 = make_float2(rstd, rstd);
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    const float2 v = __fmul2_rn(__fmul2_rn(make_float2(x[2 * i], x[2 * i + 1]), r2), make_float2(g[2 * i], g[2 * i + 1]));
    y[2 * i] = v.x;
    y[2 * i + 1] = v.y;
  }
  const int64_t e = t * p.H + h;
  if (active && p.norm_out != nullptr) {
    uint32_t w[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) w[i] = Act<A>::pack(y[2 * i], y[2 * i + 1]);
    if constexpr (N == 8)
      *reinterpret_cast<uint4*>(p.norm_out + e * 2) = make_uint4(w[0], w[1], w[2], w[3]);
    else
      *reinterpret_cast<uint2*>(p.norm_out + e * 2) = make_uint2(w[0], w[1]);
  }
  if (p.quant == MFR_QUANT_NONE) return;
  // The quantisers read the rounded norm_out values.
#pragma unroll
  for (int i = 0; i < N; ++i) y[i] = Act<A>::round(y[i]);
  if (p.quant == MFR_QUANT_FP8_E4M3) {
    if (active) {
      uint32_t q[N / 4];
#pragma unroll
      for (int j = 0; j < N / 4; ++j) {
        q[j] = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          q[j] |= static_cast<uint32_t>(
                      __nv_cvt_float_to_fp8(__fmul_rn(y[4 * j + i], qscale), __NV_SATFINITE, __NV_E4M3))
                  << (8 * i);
      }
      if constexpr (N == 8)  // one 8-byte store (e is a multiple of 8)
        *reinterpret_cast<uint2*>(p.quant_out + e) = make_uint2(q[0], q[1]);
      else
        *reinterpret_cast<uint32_t*>(p.quant_out + e) = q[0];
    }
  } else if (p.quant == MFR_QUANT_NVFP4) {
    float amax = 0.0f;
    if (active) {
#pragma unroll
      for (int i = 0; i < N; ++i) amax = fmaxf(amax, fabsf(y[i]));
    }
#pragma unroll
    for (int o = 1; o < 16 / N; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const __nv_fp8_storage_t sf =
        __nv_cvt_float_to_fp8(__fmul_rn(__fdiv_rn(amax, 6.0f), qscale), __NV_SATFINITE, __NV_E4M3);
    const float sf_val = __half2float(__half(__nv_cvt_fp8_to_halfraw(sf, __NV_E4M3)));
    const float es = (sf_val == 0.0f) ? 0.0f : __fdiv_rn(qscale, sf_val);
    if (active) {
      uint32_t codes = 0;  // N / 2 bytes, even element in the low nibble
#pragma unroll
      for (int j = 0; j < N / 2; ++j)
        codes |= static_cast<uint32_t>(__nv_cvt_float2_to_fp4x2(
                     make_float2(__fmul_rn(y[2 * j], es), __fmul_rn(y[2 * j + 1], es)), __NV_E2M1, cudaRoundNearest))
                 << (8 * j);
      if constexpr (N == 8)  // one 4-byte store (e / 2 is a multiple of 4)
        *reinterpret_cast<uint32_t*>(p.quant_out + e / 2) = codes;
      else
        *reinterpret_cast<uint16_t*>(p.quant_out + e / 2) = static_cast<uint16_t>(codes);
      if ((h & 15) == 0) p.sf_out[sf_offset(t, h >> 4, p.H, p.sf_layout)] = sf;
    }
  }
}

}  // namespace mfr
