// C ABI of the fused MoE finalize: argument validation (nothing is enqueued on error), launch
// planning for the two kernels, dispatch, size queries and status strings.
//
// Validation follows the guards named on the pages: the hidden size must be a multiple of the
// 128-bit vector width, since no tail is read or written partially (flashinfer PR #3385, review of
// the one-shot dispatch: reject token_dim not divisible by 16 / sizeof(T)); only the LINEAR and
// SWIZZLED_128x4 scale layouts are accepted (same review, layout whitelist); optional outputs may
// be NULL (same review: guard the prenormed output); 4 < topK <= 64 bounds the small-batch kernel
// of flashinfer PR #6546 (here any 1 <= K <= 64 is accepted).
#include <algorithm>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <map>
#include <tuple>

#include "mfr_launch.h"
#include "moe_finalize.h"

namespace mfr {
namespace {

thread_local char g_last_error[512] = "";

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return status;
}

struct DeviceInfo {
  int sms = 0;
  int smem_optin = 0;
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;
std::map<std::tuple<int, int, int, int, int>, int> g_cluster_ok;  // (dev, act, C, block, smem) -> clusters
std::map<std::tuple<int, int, int, int, int>, int> g_stream_bps;  // (dev, act, groups, block, smem) -> blocks/SM
std::map<std::tuple<int, int, int, int, int>, int> g_bulk_bps;    // (dev, act, columns, block, smem) -> blocks/SM

int device_info(DeviceInfo* out, int* dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MFR_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_devices.find(dev);
  if (it == g_devices.end()) {
    DeviceInfo d;
    int major = 0;
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return fail(MFR_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    if (major < 10) return fail(MFR_ERR_UNSUPPORTED, "device %d has compute capability %d.x; built for sm_103a", dev, major);
    it = g_devices.emplace(dev, d).first;
  }
  *out = it->second;
  *dev_out = dev;
  return MFR_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int validate(const mfr_args* a) {
  if (a == nullptr) return fail(MFR_ERR_INVALID_ARG, "args is NULL");
  if (a->T < 0) return fail(MFR_ERR_INVALID_ARG, "T = %d < 0", a->T);
  if (a->H < 8 || a->H > MFR_MAX_HIDDEN || a->H % 8 != 0)
    return fail(MFR_ERR_INVALID_ARG, "H = %d must be a multiple of 8 in [8, %d]", a->H, MFR_MAX_HIDDEN);
  if (a->K < 1 || a->K > MFR_MAX_TOP_K) return fail(MFR_ERR_INVALID_ARG, "K = %d outside [1, %d]", a->K, MFR_MAX_TOP_K);
  if (a->R < 1 || a->R > MFR_MAX_PARTIALS)
    return fail(MFR_ERR_INVALID_ARG, "R = %d outside [1, %d]", a->R, MFR_MAX_PARTIALS);
  if (a->act_dtype != MFR_BF16 && a->act_dtype != MFR_FP16)
    return fail(MFR_ERR_UNSUPPORTED, "act_dtype %d: only MFR_BF16 and MFR_FP16", a->act_dtype);
  if (a->scale_dtype != MFR_FP32 && a->scale_dtype != MFR_BF16 && a->scale_dtype != MFR_FP16)
    return fail(MFR_ERR_UNSUPPORTED, "scale_dtype %d unknown", a->scale_dtype);
  if (a->quant_mode < MFR_QUANT_NONE || a->quant_mode > MFR_QUANT_NVFP4)
    return fail(MFR_ERR_UNSUPPORTED, "quant_mode %d unknown", a->quant_mode);
  if (a->quant_mode == MFR_QUANT_NVFP4) {
    if (a->sf_layout != MFR_SF_ROW_MAJOR && a->sf_layout != MFR_SF_SWIZZLED_128x4)
      return fail(MFR_ERR_UNSUPPORTED, "sf_layout %d: only ROW_MAJOR and SWIZZLED_128x4", a->sf_layout);
    if (a->H % 16 != 0) return fail(MFR_ERR_INVALID_ARG, "NVFP4 needs H %% 16 == 0 (H = %d)", a->H);
  }
  if (a->flags & ~static_cast<uint32_t>(MFR_FLAG_PDL | MFR_FLAG_ROUTING_READY | MFR_FLAG_TEST_EXCHANGE_TIMEOUT |
                                        MFR_FLAG_TEST_STREAM_TIMEOUT))
    return fail(MFR_ERR_INVALID_ARG, "unknown flag bits 0x%x", a->flags);
  if (a->kernel < MFR_KERNEL_AUTO || a->kernel > MFR_KERNEL_BULK)
    return fail(MFR_ERR_INVALID_ARG, "kernel %d unknown", a->kernel);
  if (a->T == 0) return MFR_OK;  // nothing to read or write
  if (a->partials == nullptr) return fail(MFR_ERR_INVALID_ARG, "partials is NULL");
  const uintptr_t sdt_align = a->scale_dtype == MFR_FP32 ? 4 : 2;
  for (int r = 0; r < a->R; ++r) {
    const mfr_partial& P = a->partials[r];
    if (P.perm_idx == nullptr) return fail(MFR_ERR_INVALID_ARG, "partials[%d].perm_idx is NULL", r);
    if (P.num_rows < 0) return fail(MFR_ERR_INVALID_ARG, "partials[%d].num_rows < 0", r);
    if (P.num_rows > 0 && P.gemm2_out == nullptr)
      return fail(MFR_ERR_INVALID_ARG, "partials[%d].gemm2_out is NULL", r);
    if (P.num_rows > (int64_t{1} << 40) / a->H) return fail(MFR_ERR_INVALID_ARG, "partials[%d].num_rows too large", r);
    if (!aligned(P.gemm2_out, 16)) return fail(MFR_ERR_INVALID_ARG, "partials[%d].gemm2_out not 16-byte aligned", r);
    if (!aligned(P.perm_idx, 4)) return fail(MFR_ERR_INVALID_ARG, "partials[%d].perm_idx not 4-byte aligned", r);
    if (!aligned(P.expert_scale, sdt_align))
      return fail(MFR_ERR_INVALID_ARG, "partials[%d].expert_scale misaligned", r);
    if (!aligned(P.shared_out, 16)) return fail(MFR_ERR_INVALID_ARG, "partials[%d].shared_out not 16-byte aligned", r);
  }
  const bool fin_only = a->finalize_out != nullptr && a->residual_out == nullptr && a->norm_out == nullptr &&
                        a->quant_mode == MFR_QUANT_NONE;
  if (!fin_only && (a->residual == nullptr || a->gamma == nullptr))
    return fail(MFR_ERR_INVALID_ARG, "residual and gamma are required (unless finalize_out is the only output)");
  if (!aligned(a->residual, 16) || !aligned(a->gamma, 16) || !aligned(a->residual_out, 16) ||
      !aligned(a->norm_out, 16) || !aligned(a->finalize_out, 16))
    return fail(MFR_ERR_INVALID_ARG, "residual, gamma, residual_out, norm_out and finalize_out must be 16-byte aligned");
  if (a->quant_mode != MFR_QUANT_NONE) {
    if (a->quant_out == nullptr || a->quant_scale == nullptr)
      return fail(MFR_ERR_INVALID_ARG, "quantisation needs quant_out and quant_scale");
    if (a->quant_mode == MFR_QUANT_NVFP4 && a->sf_out == nullptr)
      return fail(MFR_ERR_INVALID_ARG, "NVFP4 needs sf_out (moe_finalize_sf_bytes bytes)");
    // the epilogue writes 8 FP8 bytes or 4 NVFP4 bytes per thread in one store
    if (!aligned(a->quant_scale, 4) || !aligned(a->quant_out, a->quant_mode == MFR_QUANT_FP8_E4M3 ? 8 : 4))
      return fail(MFR_ERR_INVALID_ARG, "quant_scale (4 bytes) or quant_out (8 bytes FP8, 4 bytes NVFP4) misaligned");
  }
  if (a->residual_out == nullptr && a->norm_out == nullptr && a->quant_mode == MFR_QUANT_NONE &&
      a->finalize_out == nullptr)
    return fail(MFR_ERR_INVALID_ARG, "no output requested");
  return MFR_OK;
}

void fill_params(const mfr_args* a, KParams* p) {
  std::memset(p, 0, sizeof(*p));
  p->T = a->T;
  p->H = a->H;
  p->K = a->K;
  p->R = a->R;
  uint32_t mask = 0;
  for (int r = 0; r < a->R; ++r) {
    const mfr_partial& P = a->partials[r];
    p->part[r].gemm2 = static_cast<const uint8_t*>(P.gemm2_out);
    p->part[r].rows = P.gemm2_out ? P.num_rows : 0;
    p->part[r].perm = P.perm_idx;
    p->part[r].scale = P.expert_scale;
    p->part[r].shared = static_cast<const uint8_t*>(P.shared_out);
    if (P.shared_out) mask |= 1u << r;
  }
  p->shared_mask = mask;
  p->nslots = a->R * a->K + __builtin_popcount(mask);
  p->residual = static_cast<const uint8_t*>(a->residual);
  p->gamma = static_cast<const uint8_t*>(a->gamma);
  p->residual_out = static_cast<uint8_t*>(a->residual_out);
  p->norm_out = static_cast<uint8_t*>(a->norm_out);
  p->finalize_out = static_cast<uint8_t*>(a->finalize_out);
  p->fin_only = (a->finalize_out != nullptr && a->residual_out == nullptr && a->norm_out == nullptr &&
                 a->quant_mode == MFR_QUANT_NONE) ? 1 : 0;
  p->quant_out = static_cast<uint8_t*>(a->quant_out);
  p->sf_out = static_cast<uint8_t*>(a->sf_out);
  p->quant_scale = a->quant_scale;
  p->scale_dtype = a->scale_dtype;
  p->quant = a->quant_mode;
  p->sf_layout = a->sf_layout;
  p->pdl = (a->flags & MFR_FLAG_PDL) ? 1 : 0;
  p->routing_early = (p->pdl && (a->flags & MFR_FLAG_ROUTING_READY)) ? 1 : 0;
  p->rsf = a->routed_scaling_factor;
  p->eps = a->eps;
  p->test_token_bar_extra = (a->flags & MFR_FLAG_TEST_STREAM_TIMEOUT) ? 1u : 0u;
}

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }
int ceil_div(int a, int b) { return (a + b - 1) / b; }
// Automatic choice (measured on GB300, L2-cold): the bulk-copy kernel once every SM streams at least
// kBulkMinTokensPerSm whole tokens and a row is at least kBulkMinHidden elements (bulk copies of 8 KB
// and more), else the cluster kernel.  Decode rows (H=6144, top-8, R=4, shared rows): cluster ahead up
// to 768 tokens (67.6 against 72.1 us), bulk from 1024 (84.4 against 87.0).  Bandwidth rows (H=7168, no
// shared rows): bulk from 768 (72.8 against 74.0; T=1024 87.3 against 94.1).  H=2048: cluster ahead at
// every size measured (T=2048: 61.2 against 87.4), the per-row work of 4 KB rows being too small for a
// compute warp.  The cluster planner's targets follow (probe builds may override them).
#ifndef MFR_BULK_MIN_TOKENS_PER_SM
#define MFR_BULK_MIN_TOKENS_PER_SM 6
#endif
#ifndef MFR_BULK_MIN_HIDDEN
#define MFR_BULK_MIN_HIDDEN 4096
#endif
#ifndef MFR_CLUSTER_BLOCK
#define MFR_CLUSTER_BLOCK 512
#endif
#ifndef MFR_CLUSTER_ALT_BLOCK
#define MFR_CLUSTER_ALT_BLOCK 384  // the smaller CTA size tried for multi-chunk plans (0: none)
#endif
#ifndef MFR_CLUSTER_CTAS_PER_SM
#define MFR_CLUSTER_CTAS_PER_SM 2
#endif
#ifndef MFR_CLUSTER_MAX_SIZE
#define MFR_CLUSTER_MAX_SIZE 16
#endif
constexpr int kBulkMinTokensPerSm = MFR_BULK_MIN_TOKENS_PER_SM;
constexpr int kBulkMinHidden = MFR_BULK_MIN_HIDDEN;
constexpr int kMaxCluster = MFR_CLUSTER_MAX_SIZE;

// Cluster kernel: C CTAs per token, each covering NCH chunks of SV 16-byte vectors of the hidden row
// for all R partials (R*SV threads).  C comes from the parallelism target (about two CTAs per SM over
// the batch), SV is capped by the preferred CTA size, and NCH covers the rest of the row; C <= 16 and
// R*SV <= kClusterMaxThreads.
// This plans one form of the kernel (kc routes in flight per thread) and reports how many waves of
// resident clusters its grid takes.
bool plan_cluster_form(const mfr_args* a, const DeviceInfo& d, int dev, int kc, int split, KParams* p, LaunchGeom* g,
                       int64_t* waves_out, int block_pref = MFR_CLUSTER_BLOCK) {
  const int nvec = a->H / 8;
  const int unit = (a->H % 16 == 0) ? 2 : 1;  // slices start on 16-element blocks when H allows
  const int R = a->R;
  const int RS = R * split;                   // thread groups: partials x route groups (split form)
  const int sv_max = (kClusterMaxThreads / RS) / unit * unit;
  if (sv_max < unit) return false;
  const int sv_soft = std::min(sv_max, std::max(unit, (block_pref / RS) / unit * unit));
  // About two CTAs per SM in all: c_goal CTAs per token, each covering nchunk chunks of sv vectors.
  // Few tokens: one chunk, the row spread over up to kMaxCluster CTAs.  More tokens: fewer CTAs per
  // token, each looping over several chunks.  More CTAs per token when shared memory is short.
  // Cluster sizes of 5-7 and 9-15 CTAs measured slower than the next smaller size in {1, 2, 3, 4, 8, 16}.
  const int c_raw = std::max(1, std::min(kMaxCluster, (MFR_CLUSTER_CTAS_PER_SM * d.sms) / std::max(1, a->T)));
  int c_goal = c_raw >= 16 ? 16 : c_raw >= 8 ? 8 : c_raw >= 4 ? 4 : c_raw;
  // One-chunk plans whose grid would put two CTAs on most SMs and one on the rest take half the cluster
  // when that still covers the slice in one chunk with at most one CTA per SM: every SM then moves the
  // same bytes (L2-warm: decode T=16 4.11 us with 8-CTA clusters against 4.22 with 16; top-22 H=2048
  // T=16 5.12 against 5.34).  Not with fewer doubled SMs (decode T=12: 3.90 against 3.80), nor for top-k
  // 9..16, whose wider block would take two rounds of loads (top-10 R=4 T=16: 5.25 against 4.73).
  if (c_goal >= 4 && 2 * static_cast<int64_t>(a->T) * c_goal > 3 * static_cast<int64_t>(d.sms) &&
      static_cast<int64_t>(a->T) * (c_goal / 2) <= d.sms && ceil_div(nvec, c_goal / 2) <= sv_max &&
      (a->K <= 8 || a->K > 16))
    c_goal /= 2;
  // Candidates in order of preference: c_goal, larger counts (when shared memory is short), then smaller
  // ones.  The first whose grid runs in one wave of resident clusters wins, else the one with the fewest
  // waves.  (The 16-routes-in-flight form takes about 120 registers a thread, so only one 448- or
  // 512-thread CTA fits on an SM, and c_goal's grid would take two waves.)
  int cands[kMaxCluster + 8];
  int ncand = 0;
  for (int cg = c_goal; cg <= kMaxCluster; ++cg) cands[ncand++] = cg;
  for (int cg : {8, 4, 3, 2, 1})
    if (cg < c_goal) cands[ncand++] = cg;
  bool found = false;
  int64_t best_waves = 0;
  for (int i = 0; i < ncand; ++i) {
    const int cg = cands[i];
    const int sv = std::min(sv_soft, align_up(ceil_div(nvec, cg), unit));
    const int nch = ceil_div(nvec, cg * sv);
    const int C = ceil_div(nvec, nch * sv);
    if (C > kMaxCluster || static_cast<int64_t>(a->T) * C > INT32_MAX) continue;  // grid.x is an int
    if (split > 1 && nch != 1) continue;  // the split form covers its slice in one chunk
    const int sv_fit = align_up(ceil_div(nvec, C * nch), unit);  // even slices
    const int block = align_up(sv_fit * RS, 32);
    const int off_red = align_up((R + 2) * nch * sv_fit * 16, 16);
    const int off_routes = align_up(off_red + 56 * 4, 16);  // 50 floats, then the exchange mbarrier
    const int off_split = align_up(off_routes + R * a->K * 8, 16);
    const int smem = align_up(off_split + (split > 1 ? R * (split - 1) * 8 * sv_fit * 16 : 0), 16);
    if (smem > d.smem_optin) continue;
    LaunchGeom geo{a->T * C, block, C, smem, d.smem_optin};
    // clusters (of C CTAs; single CTAs when C = 1) the GPU holds at once, for a form
    auto resident = [&](int f) {
      const auto key = std::make_tuple(dev, a->act_dtype * 4 + f, C, block, smem);
      int n;
      {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_cluster_ok.find(key);
        n = (it == g_cluster_ok.end()) ? -1 : it->second;
      }
      if (n < 0) {
        n = C > 1 ? cluster_kernel_max_active_clusters(a->act_dtype, f, geo)
                  : d.sms * cluster_kernel_blocks_per_sm(a->act_dtype, f, geo);
        std::lock_guard<std::mutex> lock(g_mu);
        g_cluster_ok[key] = n;
      }
      return n;
    };
    // One chunk: the wider register budget when it still runs in one wave, else the narrower one.  With
    // at most 256 gathering threads on any SM, the latency form (route entries in registers, branch-free
    // predicated loads): decode T=1 3.09 us against 3.41, T=8 3.50 against 3.72 (L2-warm); with more
    // threads per SM it is slower (T=12, two CTAs on some SMs: 4.12 against 3.81; T=16, one 384-thread
    // CTA per SM: 4.44 against 4.24).
    int form = split > 1 ? kClusterForm8Split : kc == 16 ? kClusterForm16 : nch == 1 ? kClusterForm8OneChunk : kClusterForm8;
    if (form == kClusterForm8OneChunk && a->K <= 8 &&
        static_cast<int64_t>(block) * ceil_div(a->T * C, d.sms) <= 256)
      form = kClusterForm8Latency;
    int n = resident(form);
    if ((form == kClusterForm8OneChunk || form == kClusterForm8Latency) && n < a->T) {
      form = kClusterForm8;
      n = resident(form);
    }
    if (n < 1) continue;
    const int64_t waves = (static_cast<int64_t>(a->T) + n - 1) / n;
    if (found && waves >= best_waves) continue;
    found = true;
    best_waves = waves;
    p->slice_vec = sv_fit;
    p->nchunk = nch;
    p->route_batch = kc;
    p->cluster_form = form;
    p->off_red = off_red;
    // 4 bytes from every CTA of the cluster (and 4 that never come under the timeout test hook)
    p->xch_tx_bytes = 4u * C + ((a->flags & MFR_FLAG_TEST_EXCHANGE_TIMEOUT) ? 4u : 0u);
    p->off_routes = off_routes;
    p->route_groups = split;
    p->off_split = off_split;
    *g = geo;
    *waves_out = waves;
    if (waves == 1) break;
  }
  return found;
}

// Top-k up to 8: eight routes in flight per thread.  Top-k 9..16: sixteen in flight (one round), unless
// that form's plan holds only one CTA per SM (a block of 384 or more threads at about 120 registers a
// thread) or takes more than one wave; then eight in flight over two rounds, with two CTAs per SM,
// measured faster (top-10, R=4, H=7168: T=128 14.2 against 15.6 µs, T=16 6.1 against 6.3; top-16,
// R=4, T=64: 10.6 against 12.9), while small blocks keep the single round (top-16, R=1, H=3584,
// T=128: 5.4 against 7.3).  Larger top-k: sixteen in flight.
// Row loads on the busiest SM for a one-wave plan: its CTAs x chunks x threads (each thread one 16-byte
// vector of one route per chunk).
int64_t busiest_sm_loads(const mfr_args* a, const DeviceInfo& d, const KParams& p, const LaunchGeom& g) {
  const int64_t per_sm = (static_cast<int64_t>(g.grid) + d.sms - 1) / d.sms;
  return per_sm * p.nchunk * static_cast<int64_t>(p.slice_vec) * a->R;
}

bool plan_cluster(const mfr_args* a, const DeviceInfo& d, int dev, KParams* p, LaunchGeom* g) {
  int64_t waves = 0;
  if (a->K <= 8) {
    if (!plan_cluster_form(a, d, dev, 8, 1, p, g, &waves)) return false;
    // Several chunks per CTA: smaller CTAs may spread the same rows over more SMs.  Take the 384-thread
    // plan when its busiest SM issues fewer row loads in one wave (decode T=64: C=4 x 384 threads
    // against C=3 x 512, 6.59 against 7.70 us L2-warm, 9.11 against 9.44 L2-cold); on a tie keep the
    // larger CTAs, which take fewer chunk rounds (T=128: 14.37 against 13.79 us L2-cold).
    if (MFR_CLUSTER_ALT_BLOCK > 0 && p->nchunk > 1 && waves == 1) {
      KParams p2 = *p;
      LaunchGeom g2{};
      int64_t w2 = 0;
      if (plan_cluster_form(a, d, dev, 8, 1, &p2, &g2, &w2, MFR_CLUSTER_ALT_BLOCK) && w2 == 1 &&
          busiest_sm_loads(a, d, p2, g2) < busiest_sm_loads(a, d, *p, *g)) {
        *p = p2;
        *g = g2;
      }
    }
    return true;
  }
  // Top-k > 8: the routes of a partial split over thread groups, when that plans one chunk in one wave.
  // L2-warm, same box: top-32 H=4096 T=1 5.77 -> 4.35 us; top-22 H=2048 T=1 5.11 -> 3.71; top-16 H=3584
  // T=1 4.10 -> 3.40, T=64 4.52 -> 4.12; top-10 R=2 T=1 3.63 -> 3.30 (never slower where it applies).
  if (a->K > 8) {
    KParams ps = *p;
    LaunchGeom gs{};
    if (plan_cluster_form(a, d, dev, 8, ceil_div(a->K, 8), &ps, &gs, &waves) && waves == 1) {
      *p = ps;
      *g = gs;
      return true;
    }
  }
  const bool ok16 = plan_cluster_form(a, d, dev, 16, 1, p, g, &waves);
  if (a->K > 16 || (ok16 && g->block < 384 && waves == 1)) return ok16;
  KParams p8 = *p;
  LaunchGeom g8{};
  if (plan_cluster_form(a, d, dev, 8, 1, &p8, &g8, &waves)) {
    *p = p8;
    *g = g8;
    return true;
  }
  return ok16;
}

// Stream kernel: persistent CTAs (one per SM) of a routing warp and kStreamGroups groups of compute
// warps, each group streaming its own tokens.  A compute thread copies its own 16-byte columns of the
// rows ahead into its group's ring of kStreamSlots row slots; a hidden pass covers 8 elements x
// kStreamColumns x the group's threads.
bool plan_stream(const mfr_args* a, const DeviceInfo& d, int dev, KParams* p, LaunchGeom* g) {
  const int block = 32 * (1 + kStreamGroups * kStreamGroupWarps);
  const int ring_bytes = align_up(16 + (p->nslots + 1) * 16, 16);  // the count, then the entries and the residual row
  const int bar_bytes = 8 * (2 * kStreamLists + 2 * kStreamGroups) + 8;
  const int off_stage = align_up(bar_bytes, 128);
  // With at most one token per CTA (T <= SMs) the groups split each token's hidden dimension (split
  // mode, pass width H / G); otherwise they split the tokens.  Widest pass first, two groups before
  // one; narrower passes when shared memory is short.
  const bool one_token_per_cta = a->T <= d.sms;
  for (int mode = one_token_per_cta ? 0 : 1; mode < 2; ++mode) {
  for (int G = kStreamGroups; G >= 1; --G) {
    if ((kStreamGroups * kStreamGroupWarps) % G != 0 || kStreamLists % G != 0) continue;
    const bool split = mode == 0;
    if (split && G < 2) continue;
    const int step = 8 * 32 * (kStreamGroups * kStreamGroupWarps / G);  // 8 elements x the group's threads
    const int w_split = align_up(ceil_div(a->H, G), 16);
    if (split && w_split > step * kStreamColumns) continue;
    for (int W = split ? w_split : step * kStreamColumns; W >= (split ? w_split : step); W -= step) {
      const int slot_bytes = std::min(W, a->H) * 2;
      const int off_ring = off_stage + G * kStreamSlots * slot_bytes;
      const int off_stash = align_up(off_ring + kStreamLists * ring_bytes, 16);
      const int off_sred = off_stash + G * align_up(a->H * 2, 16);
      const int smem = align_up(off_sred + kStreamGroups * 2 * 32 * 4, 128);
      if (smem > d.smem_optin) continue;
      LaunchGeom geo{0, block, 1, smem, d.smem_optin};
      const auto key = std::make_tuple(dev, a->act_dtype, G, block, smem);
      int bps;
      {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_stream_bps.find(key);
        bps = (it == g_stream_bps.end()) ? -1 : it->second;
      }
      if (bps < 0) {
        bps = stream_kernel_blocks_per_sm(a->act_dtype, G, geo);
        std::lock_guard<std::mutex> lock(g_mu);
        g_stream_bps[key] = bps;
      }
      if (bps < 1) continue;
      geo.grid = std::min(a->T, d.sms * bps);
      p->chunk = W;
      p->stages = kStreamSlots;
      p->stage_bytes = slot_bytes;
      p->groups = G;
      p->split = split ? 1 : 0;
      p->ring_bytes = ring_bytes;
      p->off_bar = 0;
      p->off_stage = off_stage;
      p->off_ring = off_ring;
      p->off_stash = off_stash;
      p->off_sred = off_sred;
      *g = geo;
      return true;
    }
  }
  }
  return false;
}

// Bulk-copy kernel: persistent CTAs (one per SM) of a routing warp, a copy warp and 8 to 14 compute
// warps (as many as fill their columns most evenly: the row's 16-byte columns over the threads, whole
// columns per thread; ties to more warps), 
// each CTA finalizing whole tokens in turn.  A pass covers the whole row when the compute threads can
// hold it in kBulkMaxColumns 16-byte columns each, else the row is cut into equal passes (multiples of
// 16 elements).  The ring takes stages of SR row slots: four stages, each with as many rows as shared
// memory allows (at least one, at most 8), fewer stages only when even one row per stage does not fit.
bool plan_bulk(const mfr_args* a, const DeviceInfo& d, int dev, KParams* p, LaunchGeom* g) {
  // Compute warps: decode H=6144 (768 columns) 12 warps, two columns each, 80.3 us at T=1024 against
  // 81.8 with 14; H=7168 (896 columns) 14 warps, 84.6 us against 86.7 with 12 (L2-cold).
  int ncw = kBulkMaxComputeWarps;
  {
    double best = -1.0;
    for (int w = 8; w <= kBulkMaxComputeWarps; w += 2) {
      const int nt = 32 * w;
      const int np = ceil_div(a->H, 8 * nt * kBulkMaxColumns);
      const int wp = np == 1 ? a->H : align_up(ceil_div(a->H, np), 16);
      const int q = ceil_div(ceil_div(wp, 8), nt);
      const double use = static_cast<double>(ceil_div(wp, 8)) / (static_cast<double>(q) * nt);
      if (use >= best) {
        best = use;
        ncw = w;
      }
    }
  }
  const int nct = 32 * ncw;
  const int block = 64 + nct;  // a routing warp, a copy warp and the compute warps
  const int max_pass = 8 * nct * kBulkMaxColumns;
  const int npass = ceil_div(a->H, max_pass);
  const int W = npass == 1 ? a->H : align_up(ceil_div(a->H, npass), 16);
  const int Q = ceil_div(ceil_div(W, 8), nct);
  const int slot_bytes = W * 2;
  const int ring_bytes = align_up(16 + (p->nslots + 1) * 16, 16);  // the count, then the entries and the residual row
  for (int nst = 4; nst >= 2; --nst) {
    const int off_bar = 0;
    const int bar_bytes = 8 * (2 * nst + 2 * 4 + 2) + 8;  // stages, lists, the token meeting; abort flag
    const int off_ring = align_up(off_bar + bar_bytes, 16);
    const int off_stash = align_up(off_ring + 4 * ring_bytes, 16);
    const int off_sred = align_up(off_stash + 2 * a->H * 2, 16);  // two stash buffers (by token parity)
    const int off_stage = align_up(off_sred + 2 * 32 * 4, 128);
    const int room = d.smem_optin - off_stage;
    const int sr = std::min(8, room / (nst * slot_bytes));
    if (sr < 1) continue;
    const int smem = off_stage + nst * sr * slot_bytes;
    LaunchGeom geo{0, block, 1, smem, d.smem_optin};
    const auto key = std::make_tuple(dev, a->act_dtype, Q, block, smem);
    int bps;
    {
      std::lock_guard<std::mutex> lock(g_mu);
      auto it = g_bulk_bps.find(key);
      bps = (it == g_bulk_bps.end()) ? -1 : it->second;
    }
    if (bps < 0) {
      bps = bulk_kernel_blocks_per_sm(a->act_dtype, Q, geo);
      std::lock_guard<std::mutex> lock(g_mu);
      g_bulk_bps[key] = bps;
    }
    if (bps < 1) continue;
    geo.grid = std::min(a->T, d.sms * bps);
    p->chunk = W;
    p->stages = nst;
    p->stage_rows = sr;
    p->stage_bytes = slot_bytes;
    p->cols_per_thread = Q;
    p->compute_warps = ncw;
    p->ring_bytes = ring_bytes;
    p->off_bar = off_bar;
    p->off_stage = off_stage;
    p->off_ring = off_ring;
    p->off_stash = off_stash;
    p->off_sred = off_sred;
    *g = geo;
    return true;
  }
  return false;
}

int make_plan(const mfr_args* a, KParams* p, LaunchGeom* g, int* kernel) {
  int st = validate(a);
  if (st != MFR_OK) return st;
  if (a->T == 0) {
    *kernel = MFR_KERNEL_AUTO;
    return MFR_OK;
  }
  DeviceInfo d;
  int dev = 0;
  if ((st = device_info(&d, &dev)) != MFR_OK) return st;
  fill_params(a, p);
  const bool auto_bulk = static_cast<int64_t>(a->T) >= static_cast<int64_t>(kBulkMinTokensPerSm) * d.sms &&
                         a->H >= kBulkMinHidden;
  const int first = a->kernel != MFR_KERNEL_AUTO ? a->kernel : auto_bulk ? MFR_KERNEL_BULK : MFR_KERNEL_CLUSTER;
  if (first == MFR_KERNEL_BULK && plan_bulk(a, d, dev, p, g)) {
    *kernel = MFR_KERNEL_BULK;
    return MFR_OK;
  }
  if (first == MFR_KERNEL_CLUSTER && plan_cluster(a, d, dev, p, g)) {
    *kernel = MFR_KERNEL_CLUSTER;
    return MFR_OK;
  }
  if (first == MFR_KERNEL_STREAM && plan_stream(a, d, dev, p, g)) {
    *kernel = MFR_KERNEL_STREAM;
    return MFR_OK;
  }
  if (a->kernel == MFR_KERNEL_AUTO) {  // the other kernels, when the first choice does not fit
    if (first != MFR_KERNEL_CLUSTER && plan_cluster(a, d, dev, p, g)) {
      *kernel = MFR_KERNEL_CLUSTER;
      return MFR_OK;
    }
    if (first != MFR_KERNEL_BULK && plan_bulk(a, d, dev, p, g)) {
      *kernel = MFR_KERNEL_BULK;
      return MFR_OK;
    }
    if (plan_stream(a, d, dev, p, g)) {
      *kernel = MFR_KERNEL_STREAM;
      return MFR_OK;
    }
  }
  return fail(MFR_ERR_UNSUPPORTED, "no kernel fits T=%d H=%d K=%d R=%d in shared memory (kernel %d)", a->T, a->H,
              a->K, a->R, a->kernel);
}

__global__ void empty_kernel(int pdl) {
  if (pdl) {
    pdl_launch_dependents();
    pdl_wait();
  }
}

// The dependent chain every finalize starts with, alone: read a route index, then 16 bytes per lane of
// the row it names, then write them.
__global__ void gather_floor_kernel(const int32_t* idx, const uint8_t* rows, int64_t nrows, int64_t row_bytes,
                                    uint8_t* out, int pdl) {
  if (pdl) {
    pdl_launch_dependents();
    pdl_wait();
  }
  const int32_t i = idx[0];
  const int64_t off = static_cast<int64_t>(threadIdx.x) * 16;
  if (i >= 0 && i < nrows && off + 16 <= row_bytes)
    *reinterpret_cast<uint4*>(out + off) = *reinterpret_cast<const uint4*>(rows + i * row_bytes + off);
}

}  // namespace
}  // namespace mfr

using namespace mfr;

extern "C" {

int moe_finalize_fused(const mfr_args* args, struct CUstream_st* stream) {
  KParams p;
  LaunchGeom g{};
  int kernel = 0;
  int st = make_plan(args, &p, &g, &kernel);
  if (st != MFR_OK || args->T == 0) return st;
  cudaError_t e = (kernel == MFR_KERNEL_CLUSTER) ? launch_cluster_kernel(args->act_dtype, p, g, stream)
                  : (kernel == MFR_KERNEL_BULK)  ? launch_bulk_kernel(args->act_dtype, p, g, stream)
                                                 : launch_stream_kernel(args->act_dtype, p, g, stream);
  if (e != cudaSuccess) return fail(MFR_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
  return MFR_OK;
}

int moe_finalize_plan(const mfr_args* args, mfr_plan* plan) {
  if (plan == nullptr) return fail(MFR_ERR_INVALID_ARG, "plan is NULL");
  KParams p;
  LaunchGeom g{};
  int kernel = 0;
  int st = make_plan(args, &p, &g, &kernel);
  if (st != MFR_OK) return st;
  plan->kernel = kernel;
  plan->grid = g.grid;
  plan->cluster = g.cluster;
  plan->block = g.block;
  plan->smem_bytes = g.smem;
  plan->chunk = kernel == MFR_KERNEL_CLUSTER ? p.slice_vec * 8 : p.chunk;  // cluster: hidden elements per chunk
  plan->stages = kernel == MFR_KERNEL_CLUSTER ? p.nchunk : p.stages;       // cluster: chunks per CTA
  return MFR_OK;
}

int64_t moe_finalize_sf_bytes(int32_t T, int32_t H, int32_t sf_layout) {
  if (T < 0 || H <= 0 || H % 16 != 0) return fail(MFR_ERR_INVALID_ARG, "T >= 0 and H a positive multiple of 16");
  const int64_t cols = H / 16;
  if (sf_layout == MFR_SF_ROW_MAJOR) return static_cast<int64_t>(T) * cols;
  if (sf_layout == MFR_SF_SWIZZLED_128x4) return ((static_cast<int64_t>(T) + 127) / 128) * 128 * ((cols + 3) / 4) * 4;
  return fail(MFR_ERR_UNSUPPORTED, "sf_layout %d unknown", sf_layout);
}

int64_t moe_finalize_quant_bytes(int32_t T, int32_t H, int32_t quant_mode) {
  if (T < 0 || H <= 0) return fail(MFR_ERR_INVALID_ARG, "T >= 0 and H > 0");
  switch (quant_mode) {
    case MFR_QUANT_NONE: return 0;
    case MFR_QUANT_FP8_E4M3: return static_cast<int64_t>(T) * H;
    case MFR_QUANT_NVFP4:
      if (H % 16 != 0) return fail(MFR_ERR_INVALID_ARG, "NVFP4 needs H %% 16 == 0");
      return static_cast<int64_t>(T) * H / 2;
    default: return fail(MFR_ERR_UNSUPPORTED, "quant_mode %d unknown", quant_mode);
  }
}

const char* moe_finalize_status_string(int status) {
  switch (status) {
    case MFR_OK: return "MFR_OK";
    case MFR_ERR_INVALID_ARG: return "MFR_ERR_INVALID_ARG: invalid argument";
    case MFR_ERR_UNSUPPORTED: return "MFR_ERR_UNSUPPORTED: unsupported combination";
    case MFR_ERR_CUDA: return "MFR_ERR_CUDA: CUDA runtime error";
    default: return "unknown status";
  }
}

const char* moe_finalize_last_error(void) { return g_last_error; }

int moe_finalize_empty_launch(struct CUstream_st* stream, uint32_t flags) {
  const int pdl = (flags & MFR_FLAG_PDL) ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, empty_kernel, pdl);
  if (e != cudaSuccess) return fail(MFR_ERR_CUDA, "empty launch: %s", cudaGetErrorString(e));
  return MFR_OK;
}

int moe_finalize_gather_floor_launch(const int32_t* idx, const void* rows, int64_t nrows, int64_t row_bytes,
                                     void* out, struct CUstream_st* stream, uint32_t flags) {
  if (idx == nullptr || rows == nullptr || out == nullptr || nrows <= 0 || row_bytes < 512 ||
      (reinterpret_cast<uintptr_t>(rows) | reinterpret_cast<uintptr_t>(out) | static_cast<uintptr_t>(row_bytes)) % 16)
    return fail(MFR_ERR_INVALID_ARG, "gather floor: non-null 16-byte aligned buffers, rows of at least 512 bytes");
  const int pdl = (flags & MFR_FLAG_PDL) ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gather_floor_kernel, idx, static_cast<const uint8_t*>(rows), nrows,
                                     row_bytes, static_cast<uint8_t*>(out), pdl);
  if (e != cudaSuccess) return fail(MFR_ERR_CUDA, "gather floor launch: %s", cudaGetErrorString(e));
  return MFR_OK;
}

int moe_finalize_read_timeouts(uint32_t* count) {
  if (count == nullptr) return fail(MFR_ERR_INVALID_ARG, "count is NULL");
  unsigned int c = 0, cc = 0, cb = 0;
  cudaError_t e = read_and_reset_timeouts(&c);
  if (e == cudaSuccess) e = read_and_reset_cluster_timeouts(&cc);
  if (e == cudaSuccess) e = read_and_reset_bulk_timeouts(&cb);
  if (e != cudaSuccess) return fail(MFR_ERR_CUDA, "reading the timeout counters: %s", cudaGetErrorString(e));
  *count = c + cc + cb;
  return MFR_OK;
}

int moe_finalize_abi_version(void) { return MFR_ABI_VERSION; }

}  // extern "C"
