// attn_res_api.cu -- the C ABI declared in include/attn_res.h.
//
// Host side of the path: argument validation (the dispatch gate of vllm PR
// #54261 -- hidden size 7168, 0 <= num_blocks <= 8, num_blocks <= capacity,
// -1 <= block_write_idx < capacity -- turned into error returns, plus the
// alignment, stride and overlap checks a raw-pointer interface needs), the
// device check, the launch-shape policy and the launch itself.  Nothing is
// launched and nothing is written unless every check passes.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "attn_res.h"
#include "attn_res_launch.cuh"

namespace {

using attn_res_dev::kH;
using attn_res_dev::Params;
using namespace attn_res_host;

constexpr int64_t kMaxStride = int64_t(1) << 40;

// Split of a token row over CTAs.  Few tokens: many small CTAs per token, so
// one token's latency chain (load, reduce, exchange) runs on many SMs.  Many
// tokens: 7 CTAs of 128 threads, all threads active.
int auto_split(int64_t T) { return T <= 32 ? 8 : 7; }

attn_res_status_t resolve_split(int64_t T, uint32_t flags, int* k_out) {
  int k = static_cast<int>((flags >> 8) & 0xffu);
  if (k == 0) k = auto_split(T);
  if (split_index(k) < 0) return ATTN_RES_EINVAL;
  *k_out = k;
  return ATTN_RES_OK;
}

int threads_for_split(int k) {
  const int vpc = attn_res_dev::kNV / k;
  return (vpc + 31) / 32 * 32;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Region {
  uintptr_t lo, hi;  // [lo, hi) in bytes
  bool used;
  bool written;
};

Region rows_region(const void* p, int64_t T, int64_t row, bool used, bool written) {
  Region r{0, 0, used && p != nullptr, written};
  if (r.used) {
    const int64_t elems = (T - 1) * row + kH;
    r.lo = reinterpret_cast<uintptr_t>(p);
    r.hi = r.lo + static_cast<uintptr_t>(elems) * 2u;
  }
  return r;
}

bool overlaps(const Region& a, const Region& b) {
  return a.used && b.used && a.lo < b.hi && b.lo < a.hi;
}

// Per-device result of the compute-capability check: 0 unknown, 1 ok, 2 not ok.
std::atomic<int> g_device_state[64];

attn_res_status_t check_device(int* dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver)
               ? ATTN_RES_EDEVICE
               : ATTN_RES_ECUDA;
  }
  *dev_out = dev;
  if (dev < 0 || dev >= 64) return ATTN_RES_EDEVICE;
  int st = g_device_state[dev].load(std::memory_order_acquire);
  if (st == 0) {
    int major = 0, minor = 0, cluster = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&cluster, cudaDevAttrClusterLaunch, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      return ATTN_RES_ECUDA;
    }
    st = (major == 10 && minor == 3 && cluster) ? 1 : 2;
    g_device_state[dev].store(st, std::memory_order_release);
  }
  return st == 1 ? ATTN_RES_OK : ATTN_RES_EDEVICE;
}

LaunchFn lookup(int S, int split_idx, bool d, bool o) {
  switch (S) {
    case 0: return launcher_s0(split_idx, d, o);
    case 1: return launcher_s1(split_idx, d, o);
    case 2: return launcher_s2(split_idx, d, o);
    case 3: return launcher_s3(split_idx, d, o);
    case 4: return launcher_s4(split_idx, d, o);
    case 5: return launcher_s5(split_idx, d, o);
    case 6: return launcher_s6(split_idx, d, o);
    case 7: return launcher_s7(split_idx, d, o);
    case 8: return launcher_s8(split_idx, d, o);
    default: return nullptr;
  }
}

}  // namespace

extern "C" {

const char* attn_res_status_string(attn_res_status_t s) {
  switch (s) {
    case ATTN_RES_OK: return "ok";
    case ATTN_RES_EINVAL: return "invalid argument (size, index, stride, eps or required pointer)";
    case ATTN_RES_EALIGN: return "misaligned pointer (16 bytes) or stride (8 elements)";
    case ATTN_RES_EALIAS: return "a written tensor overlaps another argument";
    case ATTN_RES_ECUDA: return "CUDA runtime error";
    case ATTN_RES_EDEVICE: return "current device is not a compute capability 10.3 GPU";
  }
  return "unknown status";
}

int attn_res_hidden_size(void) { return ATTN_RES_HIDDEN; }
int attn_res_max_blocks(void) { return ATTN_RES_MAX_BLOCKS; }

attn_res_status_t attn_res_launch_shape(int64_t T, int num_blocks,
                                        int has_out_norm, uint32_t flags,
                                        int* split, int* threads_per_cta,
                                        int64_t* ctas, int* cluster) {
  if (T < 0 || num_blocks < 0 || num_blocks > ATTN_RES_MAX_BLOCKS) return ATTN_RES_EINVAL;
  int k = 0;
  attn_res_status_t st = resolve_split(T, flags, &k);
  if (st != ATTN_RES_OK) return st;
  const bool comm = num_blocks > 0 || has_out_norm;
  if (split) *split = k;
  if (threads_per_cta) *threads_per_cta = threads_for_split(k);
  if (ctas) *ctas = T * k;
  if (cluster) *cluster = comm ? k : 1;
  return ATTN_RES_OK;
}

attn_res_status_t attn_res(attn_res_bf16_t* prefix, const attn_res_bf16_t* delta,
                           attn_res_bf16_t* blocks, int num_blocks,
                           int block_write_idx, const attn_res_bf16_t* res_w,
                           const attn_res_bf16_t* rms_w,
                           const attn_res_bf16_t* out_norm_w, float eps,
                           float out_eps, attn_res_bf16_t* out, int64_t T,
                           const attn_res_layout_t* layout, void* stream) {
  // ---- arguments (pure host checks, no CUDA call) ----
  if (layout == nullptr || T < 0) return ATTN_RES_EINVAL;
  const int cap = layout->blocks_capacity;
  if (num_blocks < 0 || num_blocks > ATTN_RES_MAX_BLOCKS || cap < 0 || num_blocks > cap)
    return ATTN_RES_EINVAL;
  if (block_write_idx < -1 || block_write_idx >= cap) return ATTN_RES_EINVAL;
  if (!std::isfinite(eps) || eps < 0.f || !std::isfinite(out_eps) || out_eps < 0.f)
    return ATTN_RES_EINVAL;
  int split = 0;
  if (resolve_split(T, layout->flags, &split) != ATTN_RES_OK) return ATTN_RES_EINVAL;
  if ((layout->flags & ~(ATTN_RES_FLAG_PDL | ATTN_RES_FLAG_SPLIT(0xff))) != 0) return ATTN_RES_EINVAL;
  if (T * split > INT32_MAX) return ATTN_RES_EINVAL;
  // no rows: nothing is read or written, so pointers and strides do not matter
  if (T == 0) return ATTN_RES_OK;

  const bool has_delta = delta != nullptr;
  const bool has_onorm = out_norm_w != nullptr;
  const bool uses_bank = num_blocks > 0 || block_write_idx >= 0;
  if (!prefix || !res_w || !rms_w || !out || (uses_bank && !blocks)) return ATTN_RES_EINVAL;

  const int64_t pr = layout->prefix_row, dr = layout->delta_row, bt = layout->blocks_token,
                bs = layout->blocks_slot, orow = layout->out_row;
  auto bad_row_stride = [](int64_t s) { return s < kH || s > kMaxStride; };
  if (bad_row_stride(pr) || bad_row_stride(orow) || (has_delta && bad_row_stride(dr)))
    return ATTN_RES_EINVAL;
  if (uses_bank) {
    if (bad_row_stride(bs)) return ATTN_RES_EINVAL;
    if (T > 1 && (bt < (int64_t)(cap - 1) * bs + kH || bt > kMaxStride)) return ATTN_RES_EINVAL;
  }
  if (!aligned16(prefix) || !aligned16(res_w) || !aligned16(rms_w) || !aligned16(out) ||
      (has_delta && !aligned16(delta)) || (has_onorm && !aligned16(out_norm_w)) ||
      (uses_bank && !aligned16(blocks)))
    return ATTN_RES_EALIGN;
  if ((pr % 8) || (orow % 8) || (has_delta && (dr % 8)) || (uses_bank && ((bs % 8) || (bt % 8))))
    return ATTN_RES_EALIGN;

  {
    const int64_t bank_elems = (T - 1) * (T > 1 ? bt : 0) + (int64_t)(cap > 0 ? cap - 1 : 0) * bs + kH;
    Region regs[7] = {
        rows_region(prefix, T, pr, true, has_delta),
        rows_region(delta, T, dr, has_delta, false),
        Region{reinterpret_cast<uintptr_t>(blocks),
               reinterpret_cast<uintptr_t>(blocks) + static_cast<uintptr_t>(bank_elems) * 2u,
               uses_bank, block_write_idx >= 0},
        rows_region(res_w, 1, kH, true, false),
        rows_region(rms_w, 1, kH, true, false),
        rows_region(out_norm_w, 1, kH, has_onorm, false),
        rows_region(out, T, orow, true, true),
    };
    for (int i = 0; i < 7; ++i)
      for (int j = 0; j < 7; ++j)
        if (i != j && regs[i].written && overlaps(regs[i], regs[j])) return ATTN_RES_EALIAS;
  }

  // ---- device and launch ----
  int dev = 0;
  attn_res_status_t st = check_device(&dev);
  if (st != ATTN_RES_OK) return st;
  LaunchFn fn = lookup(num_blocks, split_index(split), has_delta, has_onorm);
  if (fn == nullptr) return ATTN_RES_EINVAL;

  Params p;
  p.prefix = prefix;
  p.delta = delta;
  p.blocks = blocks;
  p.res_w = res_w;
  p.rms_w = rms_w;
  p.onw = out_norm_w;
  p.out = out;
  p.prefix_row = pr;
  p.delta_row = has_delta ? dr : 0;
  p.blocks_token = uses_bank ? bt : 0;
  p.blocks_slot = uses_bank ? bs : 0;
  p.out_row = orow;
  p.write_idx = block_write_idx;
  p.eps = eps;
  p.out_eps = out_eps;
  const bool pdl = (layout->flags & ATTN_RES_FLAG_PDL) != 0;
  cudaError_t e = fn(p, T, pdl, static_cast<cudaStream_t>(stream), dev);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return ATTN_RES_ECUDA;
  }
  return ATTN_RES_OK;
}

}  // extern "C"
