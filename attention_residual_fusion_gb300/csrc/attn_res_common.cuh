// attn_res_common.cuh -- PTX helpers, bf16 helpers and launch parameters
// shared by the AttnRes kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn_res_dev {

constexpr int kH = 7168;        // hidden size
constexpr int kVec = 8;         // bf16 per 16-byte vector
constexpr int kNV = kH / kVec;  // 896 vectors per row
constexpr float kInvH = 1.0f / kH;  // mean over the row as a product

struct Params {
  uint16_t* prefix;
  const uint16_t* delta;
  uint16_t* blocks;
  const uint16_t* res_w;
  const uint16_t* rms_w;
  const uint16_t* onw;
  uint16_t* out;
  int64_t prefix_row, delta_row, blocks_token, blocks_slot, out_row;
  int64_t bank_group;  // B: token rows per bank row (>= 1)
  float inv_h;         // 1 / H (the kernels built for H = 7168 use a constant)
  int64_t width;       // H (the any-width kernels: the last CTA's slice may be short)
  int64_t tokens;      // T
  int write_idx;
  float eps, out_eps;
  unsigned* err;  // device status word (error bits)
};

// Bank row of token row t: t / B, the row index the attn_res_kernel.cu
// excerpt of vllm PR #54261 gives block_res (tb / B).  T < 2^31.
// GROUPED = false: the caller guarantees B == 1 (no test in a token loop).
template <bool GROUPED = true>
__device__ __forceinline__ const uint16_t* bank_of(const Params& p, int64_t t) {
  if constexpr (!GROUPED) return p.blocks + t * p.blocks_token;
  const int64_t r = p.bank_group == 1 ? t : (int64_t)((uint32_t)t / (uint32_t)p.bank_group);
  return p.blocks + r * p.blocks_token;
}
// Whether token row t writes its c into the bank slot.  With B > 1 the rows
// of a group share the slot and the group's last row writes it (the value
// the slot would hold had the rows written in order); the slot is then never
// a source, so no row of the group reads it.
template <bool GROUPED = true>
__device__ __forceinline__ bool writes_slot(const Params& p, int64_t t) {
  if (p.write_idx < 0) return false;
  if (!GROUPED || p.bank_group == 1) return true;
  return ((uint32_t)t % (uint32_t)p.bank_group) == (uint32_t)(p.bank_group - 1) || t == p.tokens - 1;
}

// Error bits recorded in the device status word.
constexpr unsigned kErrStageTimeout = 1u;     // a shared-memory stage never filled
constexpr unsigned kErrExchangeTimeout = 2u;  // partial sums of a peer CTA never arrived
// Time-out of one bounded wait.  Everything waited on lands within
// microseconds; the limit only turns a lost completion into an error bit
// instead of a hang.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ---- global memory -----------------------------------------------------------------

// Row data is used once: no L1 allocation.  Coherent (not .nc) because prefix
// and one bank slot are rewritten by the kernel.
__device__ __forceinline__ uint4 ld_row(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
// Weights are read-only for the whole kernel and shared by all CTAs of an SM.
__device__ __forceinline__ uint4 ld_weight(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_row(uint16_t* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// ---- programmatic dependent launch -------------------------------------------------

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- clusters, shared memory, mbarriers ---------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// Arrival without release semantics: pairs with fence_mbar_init() in the
// thread that initialised the barriers peers will use (the release of those
// initialisations at cluster scope, per the PTX ISA's fence.mbarrier_init),
// so the arrival itself orders nothing.  The release form measured ~0.43 µs
// between a CTA's start and its first bulk copy.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase of parity `parity` of an mbarrier of this CTA, at most
// about limit_ns.  Returns false on time-out.  The clock is read once at the
// first miss and then every 1024 tries.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 1023u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}
// Waits unless an earlier wait of this thread already failed; records the
// failure once in the device status word.
__device__ __forceinline__ void wait_or_flag(uint32_t bar, uint32_t parity, bool& failed,
                                             unsigned* err, unsigned bit) {
  if (failed) return;
  if (!mbar_wait_bounded(bar, parity)) {
    failed = true;
    atomicOr(err, bit);
  }
}

// Bulk copy (TMA, one-dimensional) global -> this CTA's shared memory,
// completing `bytes` on the mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Store one 32-bit value into another CTA's shared memory; the store
// completes 4 bytes of transaction count on that CTA's mbarrier.
__device__ __forceinline__ void st_async_f32(uint32_t remote_addr, float v, uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(remote_addr),
      "r"(__float_as_uint(v)), "r"(remote_bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Order this thread's earlier shared-memory accesses (and those it observed
// through barriers) before its later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- packed fp32 pairs (f32x2 arithmetic) ---------------------------------------------

typedef unsigned long long f32x2;  // two fp32 lanes in one 64-bit register pair

__device__ __forceinline__ f32x2 f2_make(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2_lo(f32x2 a) { return __uint_as_float((uint32_t)a); }
__device__ __forceinline__ float f2_hi(f32x2 a) { return __uint_as_float((uint32_t)(a >> 32)); }
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// A bf16 pair (low half = even column) widened to an fp32 pair, exactly.
__device__ __forceinline__ f32x2 bf2_widen(uint32_t w) {
  f32x2 r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "r"(w << 16), "r"(w & 0xffff0000u));
  return r;
}

// ---- bf16 ------------------------------------------------------------------------------

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
  uint32_t u;
  memcpy(&u, &h, sizeof u);
  return u;
}
// Packed bf16 add, round to nearest even: the correctly rounded bf16 sum of
// each pair (the same value as an fp32 add followed by RNE to bf16, since
// 24 >= 2*8+2 bits makes that double rounding innocuous).
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint4 add_bf16x8(const uint4& a, const uint4& b) {
  return make_uint4(add_bf16x2(a.x, b.x), add_bf16x2(a.y, b.y), add_bf16x2(a.z, b.z),
                    add_bf16x2(a.w, b.w));
}
__device__ __forceinline__ uint32_t vword(const uint4& v, int k) {
  return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}

// ---- warp reductions ---------------------------------------------------------------------

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__host__ __device__ constexpr int pow2_at_least(int n) { return n <= 1 ? 1 : 2 * pow2_at_least((n + 1) / 2); }
__host__ __device__ constexpr int log2_exact(int n) { return n <= 1 ? 0 : 1 + log2_exact(n / 2); }

// Reduce P values (P a power of two, <= 32) across the warp, one sum per
// value: each butterfly step halves the values a lane carries, exchanging the
// half it gives up (P-1 shuffles in all, plus 5 - log2 P full steps).  On
// return v[0] of lane l holds the warp total of value l >> (5 - log2 P).
template <int P>
__device__ __forceinline__ float reduce_scatter(float (&v)[P], int lane) {
#pragma unroll
  for (int k = 0; k < 5; ++k) {
    const int o = 16 >> k;
    const int m = (P >> k) > 1 ? (P >> k) : 1;
    if (m > 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < m / 2; ++i) {
        const float give = upper ? v[i] : v[i + m / 2];
        const float keep = upper ? v[i + m / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, give, o);
      }
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
  return v[0];
}

}  // namespace attn_res_dev
