// attn_res_launch.cuh -- host-side launch of one kernel specialisation and
// the table that maps (num_blocks, split, delta?, output norm?) to it.
#pragma once

#include <atomic>
#include <cstdint>

#include "attn_res_kernel.cuh"

namespace attn_res_host {

using attn_res_dev::Params;

// Enqueue one specialisation: T token rows, optional PDL, on `stream`.
using LaunchFn = cudaError_t (*)(const Params&, int64_t T, bool pdl,
                                 cudaStream_t stream, int device);

// Supported splits (CTAs per token row), in table order.
constexpr int kSplits[] = {4, 7, 8, 14, 16};
constexpr int kNumSplits = sizeof(kSplits) / sizeof(kSplits[0]);

inline int split_index(int k) {
  for (int i = 0; i < kNumSplits; ++i)
    if (kSplits[i] == k) return i;
  return -1;
}

template <int S, bool D, bool O, int K>
cudaError_t launch_split(const Params& p, int64_t T, bool pdl,
                         cudaStream_t stream, int device) {
  using C = attn_res_dev::SplitCfg<S, D, O, K>;
  void (*kern)(Params) = attn_res_dev::attn_res_split_kernel<S, D, O, K>;
  if (C::COMM && K > 8) {
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
    attrs[n].val.clusterDim.x = K;
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
  cfg.gridDim = dim3(static_cast<unsigned>(T * K), 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, p);
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

}  // namespace attn_res_host
