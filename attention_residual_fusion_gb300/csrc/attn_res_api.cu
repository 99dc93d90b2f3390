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

constexpr uint32_t kKnownFlags = ATTN_RES_FLAG_PDL | ATTN_RES_FLAG_SPLIT(0xff) |
                                 ATTN_RES_FLAG_KERNEL(0xf) | ATTN_RES_FLAG_STAGES(0xf) |
                                 ATTN_RES_FLAG_VPT(0xf);

// From this many tokens on, the persistent stream kernel is used.
constexpr int64_t kStreamMinTokens = 80;
// From this many tokens on, the wider automatic choices below apply (measured
// at 256 and 1024 tokens; the switch point between them is not tuned).
constexpr int64_t kManyTokens = 512;

struct Plan {
  int kernel;  // ATTN_RES_KERNEL_*
  int split;   // CTAs per token row
  int stages;  // stream kernel: ring depth; staged form: CTAs per SM; 0 otherwise
  int vpt;     // 16-byte vectors per thread and row
  int shape;   // index into the stream kernel's shape table
};

// Automatic choice, from sweeps on GB300 of graph-replayed calls over input
// copies larger than 3x L2 (num_blocks 0..6 x output norm x T = 256, 1024,
// 2048, 4096, with delta; decode, prefill and long-prefill workloads):
//  * few tokens (T < 80: split 5.2 µs vs stream 6.0 µs at T = 64, 8.7 vs 7.6
//    µs at T = 96, 8 bank rows), or no exchange at all (no bank rows and no
//    output norm) below 512 tokens: the split kernel, 7 CTAs x 128 threads per
//    token, all threads active, so a token's latency chain runs on 7 SMs at
//    once;
//  * few bank rows: a row kernel, one CTA per token holding the whole row --
//    no cluster, and the block scheduler spreads the last rows over every SM
//    (T = 1024, no bank rows, output norm: 12.0 -> 11.1 µs; one bank row,
//    T = 256: 7.6 -> 6.4 µs), its rows in registers (up to two bank rows;
//    7 vectors per thread, or 4 where that fits more CTAs per SM) or, for
//    more rows or more tokens, in shared memory (7 vectors per thread, two
//    CTAs per SM, one from 6 bank rows; 4 bank rows, T = 256: 10.1 -> 9.4
//    µs; one bank row, T = 4096: 52.8 -> 47.5 µs);
//  * with an output norm, 3..5 bank rows and at least 512 tokens: the staged
//    form of the stream kernel (prefix and delta also in the ring) in the
//    shape of the tuned register form, (4,4) at 5 CTAs per SM for 3 bank
//    rows, (7,4) at 7 for 4, (4,4) at 4 for 5 (T = 1024, 4 bank rows:
//    23.9 -> 23.0 µs); without the norm, 3 bank rows below 512 tokens: (4,4)
//    at 5;
//  * otherwise the stream kernel, persistent clusters with a 2-deep TMA ring,
//    shape (CTAs per token, vectors per thread, stages):
//      (7,4,2) with 1..5 bank rows and an output norm, and 3..6 bank rows
//              from 512 token rows: one warp per CTA, so fewer warps share
//              the reduction and exchange work of a token;
//      (2,8,2) with no bank rows (output norm only): 2 CTAs of 2 warps per
//              token, so a token's short exchange spans only two CTAs, and
//              four such CTAs fit an SM;
//      (7,2,2) otherwise (6..8 bank rows, or no output norm): two warps per
//              CTA, more warps per SM to cover the longer per-token work.
//  * with shared bank rows (B > 1) the stream kernel has one shape, (7,2,2),
//    and neither a row kernel nor the staged form is chosen.
void auto_plan(int64_t T, int S, bool has_onorm, bool grouped, Plan* pl) {
  const bool exchange = S > 0 || has_onorm;
  const bool many = T >= kManyTokens;
  pl->kernel = ATTN_RES_KERNEL_SPLIT;
  if (T < kStreamMinTokens || grouped) {
    if (T >= kStreamMinTokens && exchange) pl->kernel = ATTN_RES_KERNEL_STREAM;
    return;
  }
  auto row = [&](int kernel, int vpt) {
    pl->kernel = kernel;
    pl->split = 1;
    pl->vpt = vpt;
  };
  auto staged = [&](int k, int ctas_per_sm) {
    pl->kernel = ATTN_RES_KERNEL_STAGED;
    pl->split = k;
    pl->vpt = 4;
    pl->stages = ctas_per_sm;
  };
  constexpr int REG = ATTN_RES_KERNEL_ROW, SMEM = ATTN_RES_KERNEL_ROW_SMEM;
  if (has_onorm) {
    switch (S) {
      case 0: return row(REG, many ? 7 : 4);
      case 1: return many ? row(SMEM, 7) : row(REG, 4);
      case 2: return T >= 4096 ? row(SMEM, 7) : row(REG, 7);
      case 3: return many ? staged(4, 5) : row(SMEM, 7);
      case 4: return many ? staged(7, 7) : row(SMEM, 7);
      case 5: return many ? staged(4, 4) : row(SMEM, 7);
      case 6: if (!many) return row(SMEM, 7); break;
      default: break;
    }
  } else if (!many) {
    switch (S) {
      case 0: return;  // the split kernel
      case 1:
      case 2: return row(REG, 4);
      case 3: return staged(4, 5);
      case 4:
      case 5: return row(SMEM, 7);
      default: break;
    }
  } else if (S <= 1) {
    return row(REG, 7);
  }
  pl->kernel = ATTN_RES_KERNEL_STREAM;
}

attn_res_status_t make_plan(int64_t T, int num_blocks, bool has_onorm, uint32_t flags, bool grouped,
                            Plan* out) {
  Plan pl;
  pl.kernel = static_cast<int>((flags >> 16) & 0xfu);
  pl.split = static_cast<int>((flags >> 8) & 0xffu);
  pl.stages = static_cast<int>((flags >> 20) & 0xfu);
  pl.vpt = static_cast<int>((flags >> 24) & 0xfu);
  pl.shape = -1;
  if (pl.kernel == 0) {
    // the automatic kernel; shape overrides given with it still apply below
    Plan a{0, 0, 0, 0, -1};
    auto_plan(T, num_blocks, has_onorm, grouped, &a);
    const bool overrides = pl.split != 0 || pl.stages != 0 || pl.vpt != 0;
    pl.kernel = a.kernel;
    if (!overrides) {
      pl.split = a.split;
      pl.stages = a.stages;
      pl.vpt = a.vpt;
    } else if (a.kernel == ATTN_RES_KERNEL_ROW || a.kernel == ATTN_RES_KERNEL_STAGED) {
      // shape overrides name a split or stream shape: keep their kernel family
      const bool exchange = num_blocks > 0 || has_onorm;
      pl.kernel = (T >= kStreamMinTokens && exchange) ? ATTN_RES_KERNEL_STREAM : ATTN_RES_KERNEL_SPLIT;
    }
  }
  if (pl.kernel == ATTN_RES_KERNEL_SPLIT) {
    if (pl.split == 0) pl.split = 7;
    if (pl.vpt == 0) pl.vpt = 1;
    if (split_index(pl.split) < 0 || pl.stages != 0 || pl.vpt != 1) return ATTN_RES_EINVAL;
  } else if (pl.kernel == ATTN_RES_KERNEL_GENERIC) {
    if (pl.split != 0 || pl.stages != 0 || pl.vpt != 0) return ATTN_RES_EINVAL;
    pl.split = 1;
  } else if (pl.kernel == ATTN_RES_KERNEL_STREAM) {
    const bool no_bank = !grouped && num_blocks == 0;
    if (pl.split == 0) {
      pl.split = 7;
      if (no_bank && (pl.vpt == 0 || pl.vpt == 4 || pl.vpt == 8)) pl.split = 2;
      if (no_bank && pl.vpt == 2) pl.split = 4;
    }
    if (pl.stages == 0) pl.stages = 2;
    if (pl.vpt == 0) {
      // one warp per CTA: 1..5 bank rows with an output norm, and 3..6 bank
      // rows from 512 token rows with or without it (measured 1.5-2 % faster
      // than two warps there once the ring's start is staggered)
      const bool one_warp = pl.split == 7 && ((num_blocks >= 1 && num_blocks <= 5 && has_onorm) ||
                                              (num_blocks >= 3 && num_blocks <= 6 && T >= kManyTokens));
      if (!grouped && pl.split == 2)
        pl.vpt = no_bank ? 8 : 4;  // (2,8,2): measured 2-5 % faster than (2,4,2) without bank rows
      else
        pl.vpt = (!grouped && one_warp) ? 4 : 2;
    }
    pl.shape = stream_shape_index(pl.split, pl.vpt, pl.stages, grouped, false);
    if (pl.shape < 0) return ATTN_RES_EINVAL;
  } else if (pl.kernel == ATTN_RES_KERNEL_ROW) {
    if (pl.split == 0) pl.split = 1;
    if (pl.vpt == 0) pl.vpt = 7;
    if (pl.split != 1 || pl.stages != 0 || row_vpt_index(pl.vpt) < 0 ||
        num_blocks > kRowMaxBlocks)
      return ATTN_RES_EINVAL;
  } else if (pl.kernel == ATTN_RES_KERNEL_ROW_SMEM) {
    if (pl.split == 0) pl.split = 1;
    if (pl.vpt == 0) pl.vpt = 4;
    if (pl.split != 1 || pl.stages != 0 || row_vpt_index(pl.vpt) < 0 ||
        num_blocks < kRowSmemMinBlocks || num_blocks > kRowSmemMaxBlocks)
      return ATTN_RES_EINVAL;
  } else if (pl.kernel == ATTN_RES_KERNEL_STAGED) {
    if (grouped) return ATTN_RES_EINVAL;
    if (pl.split == 0 && pl.vpt == 0 && pl.stages == 0) {
      pl.split = num_blocks == 4 ? 7 : 4;
      pl.vpt = 4;
      pl.stages = num_blocks == 4 ? 7 : (num_blocks == 5 ? 4 : 5);
    }
    pl.shape = stream_shape_index(pl.split, pl.vpt, pl.stages, false, true);
    if (pl.shape < 0) return ATTN_RES_EINVAL;
  } else {
    return ATTN_RES_EINVAL;
  }
  *out = pl;
  return ATTN_RES_OK;
}

int threads_for(int k, int vpt) {
  const int vpc = attn_res_dev::kNV / k;
  return (vpc / vpt + 31) / 32 * 32;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Region {
  uintptr_t lo, hi;  // [lo, hi) in bytes
  bool used;
  bool written;
};

Region rows_region(const void* p, int64_t T, int64_t row, int64_t H, bool used, bool written) {
  Region r{0, 0, used && p != nullptr, written};
  if (r.used) {
    const int64_t elems = (T - 1) * row + H;
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

// Device status word: error bits a kernel records instead of hanging (a
// stage wait that timed out).  One per device, for the life of the process.
__device__ unsigned int g_status_word;
std::atomic<uintptr_t> g_status_addr[64];

cudaError_t status_word(int dev, unsigned** out) {
  uintptr_t a = g_status_addr[dev].load(std::memory_order_acquire);
  if (a == 0) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_status_word);
    if (e != cudaSuccess) return e;
    a = reinterpret_cast<uintptr_t>(ptr);
    g_status_addr[dev].store(a, std::memory_order_release);
  }
  *out = reinterpret_cast<unsigned*>(a);
  return cudaSuccess;
}

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

RowLaunchFn lookup_row_smem(int S, int vpt_idx, bool d, bool o) {
  switch (S) {
    case 0: return row_smem_launcher_s0(vpt_idx, d, o);
    case 1: return row_smem_launcher_s1(vpt_idx, d, o);
    case 2: return row_smem_launcher_s2(vpt_idx, d, o);
    case 3: return row_smem_launcher_s3(vpt_idx, d, o);
    case 4: return row_smem_launcher_s4(vpt_idx, d, o);
    case 5: return row_smem_launcher_s5(vpt_idx, d, o);
    case 6: return row_smem_launcher_s6(vpt_idx, d, o);
    case 7: return row_smem_launcher_s7(vpt_idx, d, o);
    case 8: return row_smem_launcher_s8(vpt_idx, d, o);
    default: return nullptr;
  }
}

RowLaunchFn lookup_row(int S, int vpt_idx, bool d, bool o) {
  switch (S) {
    case 0: return row_launcher_s0(vpt_idx, d, o);
    case 1: return row_launcher_s1(vpt_idx, d, o);
    case 2: return row_launcher_s2(vpt_idx, d, o);
    case 3: return row_launcher_s3(vpt_idx, d, o);
    case 4: return row_launcher_s4(vpt_idx, d, o);
    case 5: return row_launcher_s5(vpt_idx, d, o);
    case 6: return row_launcher_s6(vpt_idx, d, o);
    case 7: return row_launcher_s7(vpt_idx, d, o);
    case 8: return row_launcher_s8(vpt_idx, d, o);
    default: return nullptr;
  }
}

GenericLaunchFn lookup_generic(int S, bool d, bool o) {
  switch (S) {
    case 0: return generic_launcher_s0(d, o);
    case 1: return generic_launcher_s1(d, o);
    case 2: return generic_launcher_s2(d, o);
    case 3: return generic_launcher_s3(d, o);
    case 4: return generic_launcher_s4(d, o);
    case 5: return generic_launcher_s5(d, o);
    case 6: return generic_launcher_s6(d, o);
    case 7: return generic_launcher_s7(d, o);
    case 8: return generic_launcher_s8(d, o);
    default: return nullptr;
  }
}

TpLaunchFn lookup_tp(int S, int phase, bool d, bool o, bool g) {
  switch (S) {
    case 0: return tp_launcher_s0(phase, d, o, g);
    case 1: return tp_launcher_s1(phase, d, o, g);
    case 2: return tp_launcher_s2(phase, d, o, g);
    case 3: return tp_launcher_s3(phase, d, o, g);
    case 4: return tp_launcher_s4(phase, d, o, g);
    case 5: return tp_launcher_s5(phase, d, o, g);
    case 6: return tp_launcher_s6(phase, d, o, g);
    case 7: return tp_launcher_s7(phase, d, o, g);
    case 8: return tp_launcher_s8(phase, d, o, g);
    default: return nullptr;
  }
}

TpRingLaunchFn lookup_tp_ring(int S, int phase, bool d, bool o, bool g) {
  switch (S) {
    case 0: return tp_ring_launcher_s0(phase, d, o, g);
    case 1: return tp_ring_launcher_s1(phase, d, o, g);
    case 2: return tp_ring_launcher_s2(phase, d, o, g);
    case 3: return tp_ring_launcher_s3(phase, d, o, g);
    case 4: return tp_ring_launcher_s4(phase, d, o, g);
    case 5: return tp_ring_launcher_s5(phase, d, o, g);
    case 6: return tp_ring_launcher_s6(phase, d, o, g);
    case 7: return tp_ring_launcher_s7(phase, d, o, g);
    case 8: return tp_ring_launcher_s8(phase, d, o, g);
    default: return nullptr;
  }
}

StreamLaunchFn lookup_stream(int S, int shape, bool d, bool o) {
  switch (S) {
    case 0: return stream_launcher_s0(shape, d, o);
    case 1: return stream_launcher_s1(shape, d, o);
    case 2: return stream_launcher_s2(shape, d, o);
    case 3: return stream_launcher_s3(shape, d, o);
    case 4: return stream_launcher_s4(shape, d, o);
    case 5: return stream_launcher_s5(shape, d, o);
    case 6: return stream_launcher_s6(shape, d, o);
    case 7: return stream_launcher_s7(shape, d, o);
    case 8: return stream_launcher_s8(shape, d, o);
    default: return nullptr;
  }
}

// Self-test of the bounded waits: one warp waits, with the same code the
// mixture kernels use, on an mbarrier that nothing ever arrives at; the wait
// must give up after limit_ns and record the stage time-out bit.
__global__ void attn_res_selftest_wait_kernel(unsigned* err, uint64_t limit_ns) {
  __shared__ __align__(8) unsigned long long bar;
  if (threadIdx.x == 0) {
    attn_res_dev::mbar_init(attn_res_dev::smem_addr(&bar), 1);
    attn_res_dev::fence_mbar_init();
  }
  __syncthreads();
  if (!attn_res_dev::mbar_wait_bounded(attn_res_dev::smem_addr(&bar), 0u, limit_ns) &&
      threadIdx.x == 0)
    atomicOr(err, attn_res_dev::kErrStageTimeout);
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

// The tensor arguments of one call, checked together.
struct RowArgs {
  int64_t H = 0;  // width of the rows this call touches
  int64_t T = 0;
  const attn_res_layout_t* layout = nullptr;
  attn_res_bf16_t* prefix = nullptr;
  const attn_res_bf16_t* delta = nullptr;
  attn_res_bf16_t* blocks = nullptr;
  int num_blocks = 0;
  int write_idx = -1;
  const attn_res_bf16_t* res_w = nullptr;
  const attn_res_bf16_t* rms_w = nullptr;
  const attn_res_bf16_t* onw = nullptr;
  attn_res_bf16_t* out = nullptr;
  bool need_weights = true;  // res_w and rms_w are read
  bool writes = true;        // out, prefix (with delta) and the bank slot are written
  Region extra[2] = {};      // float buffers of the hidden-sharded calls
  bool extra_spans_ok = true;  // and their extents checked by the caller
};

// (rows - 1) * stride below 2^61 elements.
bool span_ok(int64_t rows, int64_t stride) {
  return rows <= 1 || stride <= (int64_t(1) << 61) / (rows - 1);
}

// Token rows per bank row (B); 0 in the layout means 1.
int64_t bank_group(const attn_res_layout_t* L) {
  return L->blocks_group > 1 ? L->blocks_group : 1;
}

// Pointers, strides, alignment and overlaps (pure host checks), then the
// kernel parameters.  Scalars (num_blocks, write_idx, eps, flags, T >= 0) are
// checked by the caller first; T must be > 0 here.
attn_res_status_t check_rows(const RowArgs& a, Params* p) {
  const int64_t H = a.H, T = a.T;
  const attn_res_layout_t* L = a.layout;
  const int cap = L->blocks_capacity;
  const int64_t group = bank_group(L);
  const int64_t TB = (T + group - 1) / group;  // bank rows the call touches
  const bool has_delta = a.delta != nullptr;
  const bool has_onorm = a.onw != nullptr;
  const bool uses_bank = a.num_blocks > 0 || (a.writes && a.write_idx >= 0);
  if (!a.prefix || (a.need_weights && (!a.res_w || !a.rms_w)) || (a.writes && !a.out) ||
      (uses_bank && !a.blocks))
    return ATTN_RES_EINVAL;

  const int64_t pr = L->prefix_row, dr = L->delta_row, bt = L->blocks_token,
                bs = L->blocks_slot, orow = L->out_row;
  auto bad_row_stride = [H](int64_t s) { return s < H || s > kMaxStride; };
  if (bad_row_stride(pr) || (a.writes && bad_row_stride(orow)) || (has_delta && bad_row_stride(dr)))
    return ATTN_RES_EINVAL;
  if (uses_bank) {
    if (bad_row_stride(bs)) return ATTN_RES_EINVAL;
    if (TB > 1 && (bt < (int64_t)(cap - 1) * bs + H || bt > kMaxStride)) return ATTN_RES_EINVAL;
  }
  // every extent (rows - 1) * stride must stay far from int64 overflow
  if (!span_ok(T, pr) || (has_delta && !span_ok(T, dr)) || (a.writes && !span_ok(T, orow)) ||
      (uses_bank && !span_ok(TB, bt)) || !a.extra_spans_ok)
    return ATTN_RES_EINVAL;
  if (!aligned16(a.prefix) || (a.need_weights && (!aligned16(a.res_w) || !aligned16(a.rms_w))) ||
      (a.writes && !aligned16(a.out)) || (has_delta && !aligned16(a.delta)) ||
      (has_onorm && !aligned16(a.onw)) || (uses_bank && !aligned16(a.blocks)))
    return ATTN_RES_EALIGN;
  if ((pr % 8) || (a.writes && (orow % 8)) || (has_delta && (dr % 8)) ||
      (uses_bank && ((bs % 8) || (bt % 8))))
    return ATTN_RES_EALIGN;

  {
    const int64_t bank_elems = (TB - 1) * (TB > 1 ? bt : 0) + (int64_t)(cap > 0 ? cap - 1 : 0) * bs + H;
    Region regs[9] = {
        rows_region(a.prefix, T, pr, H, true, a.writes && has_delta),
        rows_region(a.delta, T, dr, H, has_delta, false),
        Region{reinterpret_cast<uintptr_t>(a.blocks),
               reinterpret_cast<uintptr_t>(a.blocks) + static_cast<uintptr_t>(bank_elems) * 2u,
               uses_bank, a.writes && a.write_idx >= 0},
        rows_region(a.res_w, 1, H, H, a.need_weights, false),
        rows_region(a.rms_w, 1, H, H, a.need_weights, false),
        rows_region(a.onw, 1, H, H, has_onorm, false),
        rows_region(a.out, T, orow, H, a.writes, a.writes),
        a.extra[0],
        a.extra[1],
    };
    for (int i = 0; i < 9; ++i)
      for (int j = 0; j < 9; ++j)
        if (i != j && regs[i].written && overlaps(regs[i], regs[j])) return ATTN_RES_EALIAS;
  }

  p->prefix = a.prefix;
  p->delta = a.delta;
  p->blocks = a.blocks;
  p->res_w = a.res_w;
  p->rms_w = a.rms_w;
  p->onw = a.onw;
  p->out = a.out;
  p->prefix_row = pr;
  p->delta_row = has_delta ? dr : 0;
  p->blocks_token = uses_bank ? bt : 0;
  p->blocks_slot = uses_bank ? bs : 0;
  p->out_row = a.writes ? orow : 0;
  p->write_idx = a.writes ? a.write_idx : -1;
  p->bank_group = group;
  p->tokens = T;
  p->inv_h = 1.0f / static_cast<float>(H);
  p->width = H;
  p->err = nullptr;
  return ATTN_RES_OK;
}

// Scalars every entry point checks the same way.
attn_res_status_t check_scalars(int64_t T, int64_t H, int num_blocks, int write_idx, float eps,
                                float out_eps, const attn_res_layout_t* layout,
                                uint32_t known = kKnownFlags) {
  if (layout == nullptr || T < 0) return ATTN_RES_EINVAL;
  if (H <= 0 || H % 8 != 0 || H > kMaxStride) return ATTN_RES_EINVAL;
  const int cap = layout->blocks_capacity;
  if (num_blocks < 0 || num_blocks > ATTN_RES_MAX_BLOCKS || cap < 0 || num_blocks > cap)
    return ATTN_RES_EINVAL;
  if (write_idx < -1 || write_idx >= cap) return ATTN_RES_EINVAL;
  if (layout->blocks_group < 0) return ATTN_RES_EINVAL;
  // rows sharing a bank row may not both read and write one of its slots
  if (bank_group(layout) > 1 && write_idx >= 0 && write_idx < num_blocks) return ATTN_RES_EINVAL;
  if (!std::isfinite(eps) || eps < 0.f || !std::isfinite(out_eps) || out_eps < 0.f)
    return ATTN_RES_EINVAL;
  if ((layout->flags & ~known) != 0) return ATTN_RES_EINVAL;
  return ATTN_RES_OK;
}

attn_res_status_t run(int64_t H, attn_res_bf16_t* prefix, const attn_res_bf16_t* delta,
                      attn_res_bf16_t* blocks, int num_blocks, int block_write_idx,
                      const attn_res_bf16_t* res_w, const attn_res_bf16_t* rms_w,
                      const attn_res_bf16_t* out_norm_w, float eps, float out_eps,
                      attn_res_bf16_t* out, int64_t T, const attn_res_layout_t* layout,
                      void* stream) {
  // ---- arguments (pure host checks, no CUDA call) ----
  attn_res_status_t st =
      check_scalars(T, H, num_blocks, block_write_idx, eps, out_eps, layout);
  if (st != ATTN_RES_OK) return st;
  Plan plan;
  if (make_plan(T, num_blocks, out_norm_w != nullptr, layout->flags, bank_group(layout) > 1,
                &plan) != ATTN_RES_OK)
    return ATTN_RES_EINVAL;
  // other widths up to 16384 whose CTAs of a row exchange sums: the
  // any-width forms, ceil(H / 1024) CTAs per row (the last one owning the
  // remainder) -- the split kernel below 80 tokens (up to 8 CTAs per row),
  // else the stream kernel (up to 16); otherwise the general kernel; no
  // shape overrides
  if (H != kH) {
    const uint32_t f = layout->flags;
    const int forced = static_cast<int>((f >> 16) & 0xfu);
    const bool overrides = ((f >> 8) & 0xffu) != 0 || ((f >> 20) & 0xffu) != 0;
    const int64_t kcols = (H + attn_res_dev::kRtCols - 1) / attn_res_dev::kRtCols;
    const bool any_width = kcols <= attn_res_dev::kRtMaxK;
    const bool exchange = num_blocks > 0 || out_norm_w != nullptr;
    if ((forced == ATTN_RES_KERNEL_STREAM && (!any_width || overrides || !exchange)) ||
        forced == ATTN_RES_KERNEL_STAGED || forced == ATTN_RES_KERNEL_ROW ||
        forced == ATTN_RES_KERNEL_ROW_SMEM)
      return ATTN_RES_EINVAL;
    const int kc = static_cast<int>(kcols);
    const bool split_ok = any_width && exchange && kc <= attn_res_dev::kSplitRtMaxK;
    if (forced == ATTN_RES_KERNEL_SPLIT && (!split_ok || overrides)) return ATTN_RES_EINVAL;
    const bool auto_fast = forced == 0 && !overrides && any_width && exchange;
    if (forced == ATTN_RES_KERNEL_SPLIT ||
        (auto_fast && split_ok && T < kStreamMinTokens)) {
      plan.kernel = ATTN_RES_KERNEL_SPLIT;
      plan.split = kc;
    } else if (forced == ATTN_RES_KERNEL_STREAM || auto_fast) {
      plan.kernel = ATTN_RES_KERNEL_STREAM;
      plan.shape = kAnyWidthStreamShape;
      plan.split = kc;
    } else {
      plan.kernel = ATTN_RES_KERNEL_GENERIC;
    }
  }
  if (plan.kernel == ATTN_RES_KERNEL_GENERIC) plan.split = 1;
  if (T * plan.split > INT32_MAX) return ATTN_RES_EINVAL;
  // no rows: nothing is read or written, so pointers and strides do not matter
  if (T == 0) return ATTN_RES_OK;

  RowArgs a;
  a.H = H;
  a.T = T;
  a.layout = layout;
  a.prefix = prefix;
  a.delta = delta;
  a.blocks = blocks;
  a.num_blocks = num_blocks;
  a.write_idx = block_write_idx;
  a.res_w = res_w;
  a.rms_w = rms_w;
  a.onw = out_norm_w;
  a.out = out;
  Params p;
  st = check_rows(a, &p);
  if (st != ATTN_RES_OK) return st;
  const bool has_delta = delta != nullptr;
  const bool has_onorm = out_norm_w != nullptr;
  p.eps = eps;
  p.out_eps = out_eps;

  // ---- device and launch ----
  int dev = 0;
  st = check_device(&dev);
  if (st != ATTN_RES_OK) return st;
  const bool pdl = (layout->flags & ATTN_RES_FLAG_PDL) != 0;
  cudaError_t e = status_word(dev, &p.err);
  if (e == cudaSuccess) {
    if (plan.kernel == ATTN_RES_KERNEL_GENERIC) {
      GenericLaunchFn fn = lookup_generic(num_blocks, has_delta, has_onorm);
      if (fn == nullptr) return ATTN_RES_EINVAL;
      e = fn(p, T, H, pdl, static_cast<cudaStream_t>(stream));
    } else if (plan.kernel == ATTN_RES_KERNEL_ROW || plan.kernel == ATTN_RES_KERNEL_ROW_SMEM) {
      RowLaunchFn fn = (plan.kernel == ATTN_RES_KERNEL_ROW ? lookup_row : lookup_row_smem)(
          num_blocks, row_vpt_index(plan.vpt), has_delta, has_onorm);
      if (fn == nullptr) return ATTN_RES_EINVAL;
      e = fn(p, T, pdl, static_cast<cudaStream_t>(stream));
    } else if (plan.kernel == ATTN_RES_KERNEL_SPLIT) {
      const int idx = H == kH ? split_index(plan.split) : kAnyWidthSplitIndex;
      LaunchFn fn = lookup(num_blocks, idx, has_delta, has_onorm);
      if (fn == nullptr) return ATTN_RES_EINVAL;
      e = fn(p, T, pdl, static_cast<cudaStream_t>(stream), dev, plan.split);
    } else {
      StreamLaunchFn fn = lookup_stream(num_blocks, plan.shape, has_delta, has_onorm);
      if (fn == nullptr) return ATTN_RES_EINVAL;
      e = fn(p, T, pdl, static_cast<cudaStream_t>(stream), dev, plan.split);
    }
  }
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return ATTN_RES_ECUDA;
  }
  return ATTN_RES_OK;
}

Region floats_region(const void* p, int64_t T, int64_t row, int64_t width, bool written) {
  Region r{0, 0, p != nullptr, written};
  if (r.used) {
    r.lo = reinterpret_cast<uintptr_t>(p);
    r.hi = r.lo + static_cast<uintptr_t>((T - 1) * row + width) * 4u;
  }
  return r;
}

// Threads per CTA of the sharded kernels: one 16-byte vector per thread where
// the shard fits in 256 threads, in whole warps.
int tp_threads(int64_t Hs, int cap) {
  const int64_t nv = Hs / 8;
  return static_cast<int>(nv >= cap ? cap : ((nv + 31) / 32) * 32);
}

// Form of the hidden-sharded kernels: the persistent ring when `stages`
// stages of a token's rows (and, for the sums, the query rows) fit in
// kTpRingMaxSmem bytes and there are at least
// kTpRingMinTokens rows (or when forced with ATTN_RES_KERNEL_STREAM), else
// one CTA per row (forced with ATTN_RES_KERNEL_GENERIC).  Ring depth 2 (a
// deeper ring fits fewer CTAs per SM and measured slower at every size);
// ATTN_RES_FLAG_STAGES(2..4) overrides it when the ring runs, and is an
// error together with ATTN_RES_KERNEL_GENERIC.  *stages = -1
// for an override that cannot be met (ATTN_RES_EINVAL).
// below ~1024 rows the ring's CTAs get one or two tokens each and its setup
// costs more than it saves (measured on TP8 shards of 896 columns)
constexpr int64_t kTpRingMinTokens = 1024;
bool tp_ring_plan(int phase, bool gram, int64_t T, int64_t Hs, int num_blocks, bool has_delta,
                  uint32_t flags, int threads, int* stages) {
  const int forced = static_cast<int>((flags >> 16) & 0xfu);
  const int want = static_cast<int>((flags >> 20) & 0xfu);
  const int rows = num_blocks + 1 + (has_delta ? 1 : 0);
  auto fits = [&](int st) {
    return attn_res_dev::tp_ring_smem_bytes(rows, Hs, st, phase == 0 && gram, threads) <= kTpRingMaxSmem;
  };
  *stages = 0;
  if ((forced != 0 && forced != ATTN_RES_KERNEL_STREAM && forced != ATTN_RES_KERNEL_GENERIC) ||
      (want != 0 && (want < 2 || want > attn_res_dev::kTpRingMaxStages))) {
    *stages = -1;
    return false;
  }
  bool ring = forced == ATTN_RES_KERNEL_STREAM ||
              (forced == 0 && T >= kTpRingMinTokens && fits(want ? want : 2));
  if (!ring) {
    if (want != 0 && forced == ATTN_RES_KERNEL_GENERIC) *stages = -1;  // a depth without the ring
    return false;
  }
  *stages = want ? want : 2;
  if (!fits(*stages)) *stages = -1;
  return *stages > 0;
}

// One phase of the hidden-sharded mixture: shared checks and launch.
// phase 0 reads the rows and weights and writes sums; phase 1 reads the rows
// and sums and writes sq; phase 2 reads the rows, sums and (with an output
// norm) sq, and writes out and the write-backs of c.
attn_res_status_t run_tp(int phase, int64_t Hs, int64_t H, attn_res_bf16_t* prefix,
                         const attn_res_bf16_t* delta, attn_res_bf16_t* blocks, int num_blocks,
                         int block_write_idx, const attn_res_bf16_t* res_w,
                         const attn_res_bf16_t* rms_w, bool onorm,
                         const attn_res_bf16_t* out_norm_w, float eps, float out_eps, float* sums,
                         int64_t sums_row, float* sq, attn_res_bf16_t* out, int64_t T,
                         const attn_res_layout_t* layout, void* stream) {
  // PDL, TP_GRAM, and the kernel form and ring depth overrides apply
  attn_res_status_t st = check_scalars(T, Hs, num_blocks, block_write_idx, eps, out_eps, layout,
                                       ATTN_RES_FLAG_PDL | ATTN_RES_FLAG_TP_GRAM |
                                           ATTN_RES_FLAG_KERNEL(0xf) | ATTN_RES_FLAG_STAGES(0xf));
  if (st != ATTN_RES_OK) return st;
  const bool gram = (layout->flags & ATTN_RES_FLAG_TP_GRAM) != 0;
  if (phase == 1 && gram) return ATTN_RES_EINVAL;  // the Gram form has no sq phase
  const int threads = tp_threads(Hs, (phase == 0 && gram) ? attn_res_dev::kTpGramThreads
                                                          : attn_res_dev::kTpMaxThreads);
  int stages = 0;
  const bool ring =
      tp_ring_plan(phase, gram, T, Hs, num_blocks, delta != nullptr, layout->flags, threads, &stages);
  if (stages < 0) return ATTN_RES_EINVAL;
  const int nr = attn_res_tp_sums_width(num_blocks, gram ? 1 : 0);
  if (H < Hs || H > kMaxStride || sums_row < nr || sums_row > kMaxStride) return ATTN_RES_EINVAL;
  if (T > INT32_MAX) return ATTN_RES_EINVAL;
  if (T == 0) return ATTN_RES_OK;
  const bool uses_sq = phase >= 1 && onorm && !gram;
  if (sums == nullptr || (uses_sq && sq == nullptr)) return ATTN_RES_EINVAL;
  if ((reinterpret_cast<uintptr_t>(sums) & 3u) || (uses_sq && (reinterpret_cast<uintptr_t>(sq) & 3u)))
    return ATTN_RES_EALIGN;

  RowArgs a;
  a.H = Hs;
  a.T = T;
  a.layout = layout;
  a.prefix = prefix;
  a.delta = delta;
  a.blocks = blocks;
  a.num_blocks = num_blocks;
  a.write_idx = block_write_idx;
  a.res_w = res_w;
  a.rms_w = rms_w;
  a.onw = phase == 2 ? out_norm_w : nullptr;
  a.out = out;
  a.need_weights = phase == 0;
  a.writes = phase == 2;
  a.extra_spans_ok = span_ok(T, sums_row);
  a.extra[0] = floats_region(sums, T, sums_row, nr, phase == 0);
  a.extra[1] = floats_region(uses_sq ? sq : nullptr, T, 1, 1, phase == 1);
  Params p;
  st = check_rows(a, &p);
  if (st != ATTN_RES_OK) return st;
  p.eps = eps;
  p.out_eps = out_eps;
  int dev = 0;
  st = check_device(&dev);
  if (st != ATTN_RES_OK) return st;
  TpArgs ta;
  ta.Hs = Hs;
  ta.inv_h = 1.0f / static_cast<float>(H);
  ta.sums = sums;
  ta.sums_row = sums_row;
  ta.sq = uses_sq ? sq : nullptr;
  const bool pdl = (layout->flags & ATTN_RES_FLAG_PDL) != 0;
  cudaError_t e = status_word(dev, &p.err);
  if (e == cudaSuccess) {
    if (ring) {
      TpRingLaunchFn fn = lookup_tp_ring(num_blocks, phase, delta != nullptr, onorm, gram);
      if (fn == nullptr) return ATTN_RES_EINVAL;
      e = fn(p, ta, T, threads, stages, pdl, static_cast<cudaStream_t>(stream), dev);
    } else {
      TpLaunchFn fn = lookup_tp(num_blocks, phase, delta != nullptr, onorm, gram);
      if (fn == nullptr) return ATTN_RES_EINVAL;
      e = fn(p, ta, T, threads, pdl, static_cast<cudaStream_t>(stream));
    }
  }
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return ATTN_RES_ECUDA;
  }
  return ATTN_RES_OK;
}

}  // namespace

extern "C" {

attn_res_status_t attn_res_tp_sums(int64_t Hs, const attn_res_bf16_t* prefix,
                                   const attn_res_bf16_t* delta, const attn_res_bf16_t* blocks,
                                   int num_blocks, const attn_res_bf16_t* res_w,
                                   const attn_res_bf16_t* rms_w, float* sums, int64_t sums_row,
                                   int64_t T, const attn_res_layout_t* layout, void* stream) {
  return run_tp(0, Hs, Hs, const_cast<attn_res_bf16_t*>(prefix), delta,
                const_cast<attn_res_bf16_t*>(blocks), num_blocks, -1, res_w, rms_w, false,
                nullptr, 0.f, 0.f, sums, sums_row, nullptr, nullptr, T, layout, stream);
}

attn_res_status_t attn_res_tp_sq(int64_t Hs, int64_t H, const attn_res_bf16_t* prefix,
                                 const attn_res_bf16_t* delta, const attn_res_bf16_t* blocks,
                                 int num_blocks, float eps, const float* sums, int64_t sums_row,
                                 float* sq, int64_t T, const attn_res_layout_t* layout,
                                 void* stream) {
  return run_tp(1, Hs, H, const_cast<attn_res_bf16_t*>(prefix), delta,
                const_cast<attn_res_bf16_t*>(blocks), num_blocks, -1, nullptr, nullptr, true,
                nullptr, eps, 0.f, const_cast<float*>(sums), sums_row, sq, nullptr, T, layout,
                stream);
}

attn_res_status_t attn_res_tp_finish(int64_t Hs, int64_t H, attn_res_bf16_t* prefix,
                                     const attn_res_bf16_t* delta, attn_res_bf16_t* blocks,
                                     int num_blocks, int block_write_idx,
                                     const attn_res_bf16_t* out_norm_w, float eps, float out_eps,
                                     const float* sums, int64_t sums_row, const float* sq,
                                     attn_res_bf16_t* out, int64_t T,
                                     const attn_res_layout_t* layout, void* stream) {
  return run_tp(2, Hs, H, prefix, delta, blocks, num_blocks, block_write_idx, nullptr, nullptr,
                out_norm_w != nullptr, out_norm_w, eps, out_eps, const_cast<float*>(sums),
                sums_row, const_cast<float*>(sq), out, T, layout, stream);
}

int attn_res_tp_sums_width(int num_blocks, int gram) {
  if (num_blocks < 0 || num_blocks > ATTN_RES_MAX_BLOCKS) return -1;
  const int n = num_blocks + 1;
  return 2 * n + (gram ? n * (n - 1) / 2 : 0);
}

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

attn_res_status_t attn_res_launch_shape(int64_t T, int num_blocks, int has_delta,
                                        int has_out_norm, uint32_t flags,
                                        int* kernel, int* split, int* stages,
                                        int* threads_per_cta, int64_t* ctas,
                                        int* cluster) {
  if (T < 0 || num_blocks < 0 || num_blocks > ATTN_RES_MAX_BLOCKS) return ATTN_RES_EINVAL;
  if ((flags & ~kKnownFlags) != 0) return ATTN_RES_EINVAL;
  Plan pl;
  attn_res_status_t st = make_plan(T, num_blocks, has_out_norm != 0, flags, false, &pl);
  if (st != ATTN_RES_OK) return st;
  const bool comm = num_blocks > 0 || has_out_norm;
  int th = 0, depth = 0, cl = 1;
  int64_t grid = 0;
  switch (pl.kernel) {
    case ATTN_RES_KERNEL_GENERIC:
      th = attn_res_dev::kGenericThreads, grid = T;
      break;
    case ATTN_RES_KERNEL_ROW:
    case ATTN_RES_KERNEL_ROW_SMEM:
      th = attn_res_dev::kNV / pl.vpt, grid = T;
      break;
    case ATTN_RES_KERNEL_SPLIT:
      th = threads_for(pl.split, pl.vpt), grid = T * pl.split, cl = comm ? pl.split : 1;
      break;
    case ATTN_RES_KERNEL_STAGED:
      depth = staged_stages(kStreamShapes[pl.shape], num_blocks, has_delta != 0);
      if (depth < 2) return ATTN_RES_EINVAL;
      th = threads_for(pl.split, pl.vpt), cl = comm ? pl.split : 1;
      break;
    default:  // the stream kernel
      th = threads_for(pl.split, pl.vpt), depth = pl.stages, cl = comm ? pl.split : 1;
      break;
  }
  if (kernel) *kernel = pl.kernel;
  if (split) *split = pl.split;
  if (stages) *stages = depth;
  if (threads_per_cta) *threads_per_cta = th;
  if (ctas) *ctas = grid;
  if (cluster) *cluster = cl;
  return ATTN_RES_OK;
}

attn_res_status_t attn_res_selftest_wait_timeout(unsigned int limit_us, unsigned int* bits) {
  if (bits == nullptr || limit_us == 0 || limit_us > 1000000u) return ATTN_RES_EINVAL;
  int dev = 0;
  attn_res_status_t st = check_device(&dev);
  if (st != ATTN_RES_OK) return st;
  unsigned* w = nullptr;
  cudaStream_t s = nullptr;
  cudaError_t e = status_word(dev, &w);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e == cudaSuccess) {
    attn_res_selftest_wait_kernel<<<1, 32, 0, s>>>(w, (uint64_t)limit_us * 1000u);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemcpy(bits, w, sizeof(unsigned), cudaMemcpyDeviceToHost);
  }
  if (s != nullptr) (void)cudaStreamDestroy(s);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return ATTN_RES_ECUDA;
  }
  return ATTN_RES_OK;
}

attn_res_status_t attn_res_device_status(unsigned int* bits, int clear) {
  if (bits == nullptr) return ATTN_RES_EINVAL;
  int dev = 0;
  attn_res_status_t st = check_device(&dev);
  if (st != ATTN_RES_OK) return st;
  unsigned* w = nullptr;
  if (status_word(dev, &w) != cudaSuccess ||
      cudaMemcpy(bits, w, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess) {
    (void)cudaGetLastError();
    return ATTN_RES_ECUDA;
  }
  if (clear && cudaMemset(w, 0, sizeof(unsigned)) != cudaSuccess) {
    (void)cudaGetLastError();
    return ATTN_RES_ECUDA;
  }
  return ATTN_RES_OK;
}

attn_res_status_t attn_res(attn_res_bf16_t* prefix, const attn_res_bf16_t* delta,
                           attn_res_bf16_t* blocks, int num_blocks,
                           int block_write_idx, const attn_res_bf16_t* res_w,
                           const attn_res_bf16_t* rms_w,
                           const attn_res_bf16_t* out_norm_w, float eps,
                           float out_eps, attn_res_bf16_t* out, int64_t T,
                           const attn_res_layout_t* layout, void* stream) {
  return run(kH, prefix, delta, blocks, num_blocks, block_write_idx, res_w, rms_w, out_norm_w,
             eps, out_eps, out, T, layout, stream);
}

attn_res_status_t attn_res_h(int64_t H, attn_res_bf16_t* prefix, const attn_res_bf16_t* delta,
                             attn_res_bf16_t* blocks, int num_blocks, int block_write_idx,
                             const attn_res_bf16_t* res_w, const attn_res_bf16_t* rms_w,
                             const attn_res_bf16_t* out_norm_w, float eps, float out_eps,
                             attn_res_bf16_t* out, int64_t T, const attn_res_layout_t* layout,
                             void* stream) {
  return run(H, prefix, delta, blocks, num_blocks, block_write_idx, res_w, rms_w, out_norm_w,
             eps, out_eps, out, T, layout, stream);
}

}  // extern "C"
