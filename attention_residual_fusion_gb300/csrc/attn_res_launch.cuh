// attn_res_launch.cuh -- host-side launch of one kernel specialisation and
// the table that maps (num_blocks, split, delta?, output norm?) to it.
#pragma once

#include <atomic>
#include <cstdint>

#include "attn_res_kernel.cuh"
#include "attn_res_row.cuh"
#include "attn_res_stream.cuh"
#include "attn_res_generic.cuh"
#include "attn_res_tp.cuh"

namespace attn_res_host {

using attn_res_dev::Params;

// Enqueue one specialisation: T token rows, optional PDL, on `stream`.
using LaunchFn = cudaError_t (*)(const Params&, int64_t T, bool pdl,
                                 cudaStream_t stream, int device, int kc);

// Supported splits (CTAs per token row), in table order; launcher index
// kNumSplits is the any-width form (K = 0, kc = H / 1024 CTAs per row).
constexpr int kSplits[] = {4, 7, 8, 14, 16};
constexpr int kNumSplits = sizeof(kSplits) / sizeof(kSplits[0]);
constexpr int kAnyWidthSplitIndex = kNumSplits;

inline int split_index(int k) {
  for (int i = 0; i < kNumSplits; ++i)
    if (kSplits[i] == k) return i;
  return -1;
}

template <int S, bool D, bool O, int K>
cudaError_t launch_split(const Params& p, int64_t T, bool pdl,
                         cudaStream_t stream, int device, int kc) {
  using C = attn_res_dev::SplitCfg<S, D, O, K>;
  void (*kern)(Params) = attn_res_dev::attn_res_split_kernel<S, D, O, K>;
  if (K != 0) kc = K;
  if (kc < 1 || kc > (K ? 16 : attn_res_dev::kSplitRtMaxK)) return cudaErrorInvalidValue;
  if (C::COMM && kc > 8) {
    // clusters above 8 CTAs are opt-in, per function and device
    static std::atomic<uint64_t> enabled{0};
    const uint64_t bit = 1ull << (device & 63);
    if (!(enabled.load(std::memory_order_acquire) & bit)) {
      cudaError_t e = cudaFuncSetAttribute(
          kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      enabled.fetch_or(bit, std::memory_order_acq_rel);
    }
  }
  cudaLaunchAttribute attrs[2];
  unsigned n = 0;
  if (C::COMM) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = kc;
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(T * kc), 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// Shapes the persistent stream kernel is built for: CTAs per token row (K),
// 16-byte vectors per thread and per row (VPT), ring depth (STAGES).  Staged
// shapes (prefix and delta in the ring too) give CTAs per SM in place of the
// depth; their depth follows from the rows of a stage (staged_depth).
struct StreamShape {
  int k, vpt, stages;
  bool grouped;  // built for B > 1 token rows per bank row
  bool staged;   // prefix and delta staged in the ring; `stages` = CTAs per SM
};
// The next-to-last entry is the one shape built for shared bank rows (B > 1);
// the last (k = 0) serves any width H that is a multiple of 1024: H / 1024
// CTAs per token row, each with the per-CTA layout of (7,2,2), shared bank
// rows allowed.
constexpr StreamShape kStreamShapes[] = {
    {7, 1, 2, false, false}, {7, 2, 2, false, false}, {7, 2, 3, false, false},
    {7, 4, 2, false, false}, {4, 2, 2, false, false}, {4, 2, 3, false, false},
    {2, 4, 2, false, false}, {14, 2, 2, false, false}, {2, 8, 2, false, false},
    {4, 4, 5, false, true},  {7, 4, 7, false, true},  {4, 4, 4, false, true},
    {7, 2, 2, true, false},  {0, 2, 2, true, false}};
constexpr int kNumStreamShapes = sizeof(kStreamShapes) / sizeof(kStreamShapes[0]);
constexpr int kGroupedStreamShape = kNumStreamShapes - 2;
constexpr int kAnyWidthStreamShape = kNumStreamShapes - 1;

inline int stream_shape_index(int k, int vpt, int stages, bool grouped, bool staged) {
  for (int i = 0; i < kNumStreamShapes; ++i)
    if (kStreamShapes[i].k == k && kStreamShapes[i].vpt == vpt &&
        kStreamShapes[i].stages == stages && kStreamShapes[i].grouped == grouped &&
        kStreamShapes[i].staged == staged)
      return i;
  return -1;
}

// Ring depth of staged shape `sh` for num_blocks bank rows (with or without
// delta); < 2 means the shape does not exist for them.
constexpr int staged_stages(const StreamShape& sh, int num_blocks, bool has_delta) {
  const int vpc = attn_res_dev::kNV / sh.k;
  const int nw = (vpc / sh.vpt + 31) / 32;
  return attn_res_dev::staged_depth(num_blocks + (has_delta ? 2 : 1), (uint32_t)vpc * 16u,
                                    sh.stages,
                                    attn_res_dev::stream_static_bytes(num_blocks, sh.k, nw));
}

// Enqueue the persistent kernel: as many clusters as fit on the device at
// once (at most T), each streaming every ncl-th token.
using StreamLaunchFn = cudaError_t (*)(const Params&, int64_t T, bool pdl,
                                       cudaStream_t stream, int device, int kc);

template <int S, bool D, bool O, int K, int VPT, int STAGES, bool G, bool STAGED = false>
cudaError_t launch_stream(const Params& p, int64_t T, bool pdl, cudaStream_t stream,
                          int device, int kc) {
  using C = attn_res_dev::StreamCfg<S, D, O, K, VPT, STAGES, STAGED>;
  void (*kern)(Params, int64_t) =
      attn_res_dev::attn_res_stream_kernel<S, D, O, K, VPT, STAGES, G, STAGED>;
  // any width not a multiple of 1024: the entry point with a short last slice
  int ragged = 0;
  if constexpr (K == 0) {
    if (p.width % attn_res_dev::kRtCols != 0) {
      kern = attn_res_dev::attn_res_stream_ragged_kernel<S, D, O, VPT, STAGES, G>;
      ragged = 1;
    }
  }
  // CTAs per token row: K, or (K = 0, any width) kc = ceil(H / 1024) from the caller
  if (K != 0) kc = K;
  if (device < 0 || device >= 64 || kc < 1 || kc > attn_res_dev::kRtMaxK)
    return cudaErrorInvalidValue;
  // per device, split and entry point: attributes set and the number of
  // co-resident clusters
  static std::atomic<int> clusters_per_device[64][attn_res_dev::kRtMaxK + 1][2];
  int ncl_max = clusters_per_device[device][kc][ragged].load(std::memory_order_acquire);
  if (ncl_max == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (C::COMM && kc > 8) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    if (C::COMM) {
      cudaLaunchAttribute a;
      a.id = cudaLaunchAttributeClusterDimension;
      a.val.clusterDim.x = kc;
      a.val.clusterDim.y = 1;
      a.val.clusterDim.z = 1;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(kc * 1024, 1, 1);
      cfg.blockDim = dim3(C::THREADS, 1, 1);
      cfg.dynamicSmemBytes = C::SMEM_BYTES;
      cfg.attrs = &a;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&ncl_max, kern, &cfg);
      if (e != cudaSuccess) return e;
    } else {
      int per_sm = 0, sms = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::THREADS, C::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
      if (e != cudaSuccess) return e;
      ncl_max = per_sm * sms / kc;
    }
    if (ncl_max < 1) return cudaErrorInvalidConfiguration;
    clusters_per_device[device][kc][ragged].store(ncl_max, std::memory_order_release);
  }
  const int64_t ncl = T < ncl_max ? T : ncl_max;
  cudaLaunchAttribute attrs[2];
  unsigned n = 0;
  if (C::COMM) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = kc;
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ncl * kc), 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, p, T);
}

// The row kernel: one CTA per token row (the whole row), VPT vectors per
// thread, built for up to kRowMaxBlocks bank rows (its rows live in
// registers; more rows leave one CTA per SM or spill).  Supported VPT
// values, in table order.
constexpr int kRowMaxBlocks = 2;
constexpr int kRowVpts[] = {4, 7};
constexpr int kNumRowVpts = sizeof(kRowVpts) / sizeof(kRowVpts[0]);

inline int row_vpt_index(int vpt) {
  for (int i = 0; i < kNumRowVpts; ++i)
    if (kRowVpts[i] == vpt) return i;
  return -1;
}

using RowLaunchFn = cudaError_t (*)(const Params&, int64_t T, bool pdl, cudaStream_t stream);

template <int S, bool D, bool O, int VPT>
cudaError_t launch_row(const Params& p, int64_t T, bool pdl, cudaStream_t stream) {
  using C = attn_res_dev::RowCfg<S, D, O, VPT>;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(T), 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_res_dev::attn_res_row_kernel<S, D, O, VPT>, p);
}

// The row kernel with its rows in shared memory: built for kRowSmemMinBlocks
// .. kRowSmemMaxBlocks bank rows (two CTAs of up to 7 rows fit an SM, one
// CTA of up to 10 rows).
constexpr int kRowSmemMinBlocks = 1;
constexpr int kRowSmemMaxBlocks = 8;

template <int S, bool D, bool O, int VPT>
cudaError_t launch_row_smem(const Params& p, int64_t T, bool pdl, cudaStream_t stream) {
  using C = attn_res_dev::RowCfg<S, D, O, VPT>;
  void (*kern)(Params) = attn_res_dev::attn_res_row_smem_kernel<S, D, O, VPT>;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 0 || device >= 64) return cudaErrorInvalidValue;
  // the dynamic shared memory above 48 KB is opt-in, per function and device
  static std::atomic<uint64_t> enabled{0};
  const uint64_t bit = 1ull << device;
  if (!(enabled.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    enabled.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(T), 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// The general kernel: one CTA per token row, any H that is a multiple of 8.
using GenericLaunchFn = cudaError_t (*)(const Params&, int64_t T, int64_t H, bool pdl,
                                        cudaStream_t stream);

template <int S, bool D, bool O>
cudaError_t launch_generic(const Params& p, int64_t T, int64_t H, bool pdl, cudaStream_t stream) {
  void (*kern)(Params, int64_t) = attn_res_dev::attn_res_generic_kernel<S, D, O>;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(T), 1, 1);
  cfg.blockDim = dim3(attn_res_dev::kGenericThreads, 1, 1);
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p, H);
}

// Hidden-sharded phases: one CTA per token row, `threads` (32..256) wide.
using attn_res_dev::TpArgs;
using TpLaunchFn = cudaError_t (*)(const Params&, const TpArgs&, int64_t T, int threads, bool pdl,
                                   cudaStream_t stream);

template <class Kern>
cudaError_t launch_tp(Kern kern, const Params& p, const TpArgs& a, int64_t T, int threads,
                      bool pdl, cudaStream_t stream) {
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(T), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p, a);
}
template <int S, bool D, bool G>
cudaError_t launch_tp_sums(const Params& p, const TpArgs& a, int64_t T, int th, bool pdl,
                           cudaStream_t s) {
  return launch_tp(attn_res_dev::attn_res_tp_sums_kernel<S, D, G>, p, a, T, th, pdl, s);
}
template <int S, bool D>
cudaError_t launch_tp_sq(const Params& p, const TpArgs& a, int64_t T, int th, bool pdl,
                         cudaStream_t s) {
  return launch_tp(attn_res_dev::attn_res_tp_sq_kernel<S, D>, p, a, T, th, pdl, s);
}
template <int S, bool D, bool O, bool G>
cudaError_t launch_tp_finish(const Params& p, const TpArgs& a, int64_t T, int th, bool pdl,
                             cudaStream_t s) {
  return launch_tp(attn_res_dev::attn_res_tp_finish_kernel<S, D, O, G>, p, a, T, th, pdl, s);
}

// Hidden-sharded phases, persistent ring form: CTAs per SM x SMs CTAs (at
// most T), each with a `stages`-deep ring of its tokens' rows in dynamic
// shared memory.
using TpRingLaunchFn = cudaError_t (*)(const Params&, const TpArgs&, int64_t T, int threads,
                                       int stages, bool pdl, cudaStream_t stream, int device);

// bytes of one CTA's dynamic shared memory, at most (the kernel's static
// shared memory stays under 2 KB: within the 227 KB a CTA may have)
constexpr int kTpRingMaxSmem = 220 * 1024;

template <int S, bool D, int PH, bool O, bool G>
cudaError_t launch_tp_ring(const Params& p, const TpArgs& a, int64_t T, int threads, int stages,
                           bool pdl, cudaStream_t stream, int device) {
  using C = attn_res_dev::TpRingCfg<S, D, PH, O, G>;
  void (*kern)(Params, TpArgs, int) = attn_res_dev::attn_res_tp_ring_kernel<S, D, PH, O, G>;
  if (device < 0 || device >= 64 || stages < 2 || stages > attn_res_dev::kTpRingMaxStages ||
      threads < 32 || threads > C::THREADS_MAX || threads % 32)
    return cudaErrorInvalidValue;
  const int64_t smem = attn_res_dev::tp_ring_smem_bytes(C::ROWS, a.Hs, stages, PH == 0 && G, threads);
  if (smem > kTpRingMaxSmem) return cudaErrorInvalidValue;
  // per device: the attribute set once, and the last (shared memory,
  // threads) -> CTAs per SM x SMs answer, packed as key << 20 | CTAs
  static std::atomic<bool> attr_set[64];
  static std::atomic<uint64_t> resident[64];
  if (!attr_set[device].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kTpRingMaxSmem);
    if (e != cudaSuccess) return e;
    attr_set[device].store(true, std::memory_order_release);
  }
  const uint64_t key = ((uint64_t)smem << 10) | (uint64_t)threads;
  uint64_t r = resident[device].load(std::memory_order_acquire);
  int64_t ctas = (r >> 20) == key ? (int64_t)(r & 0xfffffu) : 0;
  if (ctas == 0) {
    int per_sm = 0, sms = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, (size_t)smem);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    ctas = (int64_t)per_sm * sms;
    if (ctas < 1 || ctas > 0xfffff) return cudaErrorInvalidConfiguration;
    resident[device].store((key << 20) | (uint64_t)ctas, std::memory_order_release);
  }
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(T < ctas ? T : ctas), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p, a, stages);
}

// One row of the table per num_blocks, defined in attn_res_inst.cu (compiled
// once per S).  Returns nullptr for an unknown split index.
LaunchFn launcher_s0(int split_idx, bool has_delta, bool has_onorm);
LaunchFn launcher_s1(int split_idx, bool has_delta, bool has_onorm);
LaunchFn launcher_s2(int split_idx, bool has_delta, bool has_onorm);
LaunchFn launcher_s3(int split_idx, bool has_delta, bool has_onorm);
LaunchFn launcher_s4(int split_idx, bool has_delta, bool has_onorm);
LaunchFn launcher_s5(int split_idx, bool has_delta, bool has_onorm);
LaunchFn launcher_s6(int split_idx, bool has_delta, bool has_onorm);
LaunchFn launcher_s7(int split_idx, bool has_delta, bool has_onorm);
LaunchFn launcher_s8(int split_idx, bool has_delta, bool has_onorm);

StreamLaunchFn stream_launcher_s0(int shape_idx, bool d, bool o);
StreamLaunchFn stream_launcher_s1(int shape_idx, bool d, bool o);
StreamLaunchFn stream_launcher_s2(int shape_idx, bool d, bool o);
StreamLaunchFn stream_launcher_s3(int shape_idx, bool d, bool o);
StreamLaunchFn stream_launcher_s4(int shape_idx, bool d, bool o);
StreamLaunchFn stream_launcher_s5(int shape_idx, bool d, bool o);
StreamLaunchFn stream_launcher_s6(int shape_idx, bool d, bool o);
StreamLaunchFn stream_launcher_s7(int shape_idx, bool d, bool o);
StreamLaunchFn stream_launcher_s8(int shape_idx, bool d, bool o);

RowLaunchFn row_smem_launcher_s0(int vpt_idx, bool d, bool o);
RowLaunchFn row_smem_launcher_s1(int vpt_idx, bool d, bool o);
RowLaunchFn row_smem_launcher_s2(int vpt_idx, bool d, bool o);
RowLaunchFn row_smem_launcher_s3(int vpt_idx, bool d, bool o);
RowLaunchFn row_smem_launcher_s4(int vpt_idx, bool d, bool o);
RowLaunchFn row_smem_launcher_s5(int vpt_idx, bool d, bool o);
RowLaunchFn row_smem_launcher_s6(int vpt_idx, bool d, bool o);
RowLaunchFn row_smem_launcher_s7(int vpt_idx, bool d, bool o);
RowLaunchFn row_smem_launcher_s8(int vpt_idx, bool d, bool o);
RowLaunchFn row_launcher_s0(int vpt_idx, bool d, bool o);
RowLaunchFn row_launcher_s1(int vpt_idx, bool d, bool o);
RowLaunchFn row_launcher_s2(int vpt_idx, bool d, bool o);
RowLaunchFn row_launcher_s3(int vpt_idx, bool d, bool o);
RowLaunchFn row_launcher_s4(int vpt_idx, bool d, bool o);
RowLaunchFn row_launcher_s5(int vpt_idx, bool d, bool o);
RowLaunchFn row_launcher_s6(int vpt_idx, bool d, bool o);
RowLaunchFn row_launcher_s7(int vpt_idx, bool d, bool o);
RowLaunchFn row_launcher_s8(int vpt_idx, bool d, bool o);

GenericLaunchFn generic_launcher_s0(bool d, bool o);
GenericLaunchFn generic_launcher_s1(bool d, bool o);
GenericLaunchFn generic_launcher_s2(bool d, bool o);
GenericLaunchFn generic_launcher_s3(bool d, bool o);
GenericLaunchFn generic_launcher_s4(bool d, bool o);
GenericLaunchFn generic_launcher_s5(bool d, bool o);
GenericLaunchFn generic_launcher_s6(bool d, bool o);
GenericLaunchFn generic_launcher_s7(bool d, bool o);
GenericLaunchFn generic_launcher_s8(bool d, bool o);

// phase 0: sums, 1: sum of squares, 2: finish
TpLaunchFn tp_launcher_s0(int phase, bool d, bool o, bool g);
TpLaunchFn tp_launcher_s1(int phase, bool d, bool o, bool g);
TpLaunchFn tp_launcher_s2(int phase, bool d, bool o, bool g);
TpLaunchFn tp_launcher_s3(int phase, bool d, bool o, bool g);
TpLaunchFn tp_launcher_s4(int phase, bool d, bool o, bool g);
TpLaunchFn tp_launcher_s5(int phase, bool d, bool o, bool g);
TpLaunchFn tp_launcher_s6(int phase, bool d, bool o, bool g);
TpLaunchFn tp_launcher_s7(int phase, bool d, bool o, bool g);
TpLaunchFn tp_launcher_s8(int phase, bool d, bool o, bool g);
TpRingLaunchFn tp_ring_launcher_s0(int phase, bool d, bool o, bool g);
TpRingLaunchFn tp_ring_launcher_s1(int phase, bool d, bool o, bool g);
TpRingLaunchFn tp_ring_launcher_s2(int phase, bool d, bool o, bool g);
TpRingLaunchFn tp_ring_launcher_s3(int phase, bool d, bool o, bool g);
TpRingLaunchFn tp_ring_launcher_s4(int phase, bool d, bool o, bool g);
TpRingLaunchFn tp_ring_launcher_s5(int phase, bool d, bool o, bool g);
TpRingLaunchFn tp_ring_launcher_s6(int phase, bool d, bool o, bool g);
TpRingLaunchFn tp_ring_launcher_s7(int phase, bool d, bool o, bool g);
TpRingLaunchFn tp_ring_launcher_s8(int phase, bool d, bool o, bool g);

}  // namespace attn_res_host
