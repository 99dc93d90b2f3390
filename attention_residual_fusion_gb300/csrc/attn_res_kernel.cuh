// attn_res_kernel.cuh -- sm_103a kernel for the Kimi-K3 AttnRes mixture.
//
// One token row of H = 7168 bf16 is split over K CTAs of one thread-block
// cluster; CTA r owns the contiguous column slice [r*H/K, (r+1)*H/K) of every
// source row of that token, one 16-byte vector (8 bf16) per thread.  Each
// thread issues all of its row loads at once (up to 8 bank rows, the prefix
// row and the delta row: <= 160 B in flight per thread) and keeps them in
// registers, so every byte is read from HBM exactly once:
//
//   bank rows, weights      -> loaded before the grid-dependency wait
//   griddepcontrol.wait     -> prefix (and delta) are produced upstream
//   griddepcontrol.launch_dependents
//   c = bf16_rn(prefix + delta)
//   per source: sum of squares and dot with q = rms_w*res_w (fp32)
//   warp shuffle -> CTA shared memory -> cluster DSMEM exchange of 2N sums
//   logits, softmax (warp 0), weights broadcast through shared memory
//   acc = sum_i w_i x_i over the raw rows (fp32)
//   [output norm: second exchange of sum(acc^2)]
//   stores: out, then the write-backs of c (prefix, bank slot)
//
// Sources of the method: implementation walkthrough of vllm-ascend PR #14840
// (candidates, RMS normalisation, score, softmax, raw-row mix) and key source
// excerpts of the prhub summary of vllm PR #54261 (delta add and packing,
// block-bank write-back, output norm, PDL discipline).  The pages' kernel
// stages rows through a shared-memory ring with TMA and an online softmax per
// chunk; here the whole column slice of a token fits in registers, so the
// softmax is taken once over all logits after a single reduction.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn_res_dev {

constexpr int kH = 7168;          // hidden size
constexpr int kVec = 8;           // bf16 per 16-byte vector
constexpr int kNV = kH / kVec;    // 896 vectors per row

struct Params {
  uint16_t* prefix;
  const uint16_t* delta;
  uint16_t* blocks;
  const uint16_t* res_w;
  const uint16_t* rms_w;
  const uint16_t* onw;
  uint16_t* out;
  int64_t prefix_row, delta_row, blocks_token, blocks_slot, out_row;
  int write_idx;
  float eps, out_eps;
};

// ---- PTX helpers -----------------------------------------------------------

// Row data is used once: bypass L1 allocation.  Coherent (not .nc) because
// prefix and one bank slot are rewritten by this kernel.
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
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Store one float into the same shared-memory variable of CTA `rank` of this
// cluster (distributed shared memory).
__device__ __forceinline__ void st_dsmem_f32(uint32_t local, uint32_t rank,
                                             float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(local), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v)
               : "memory");
}

// ---- bf16 helpers ------------------------------------------------------------

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
  uint32_t u;
  memcpy(&u, &h, sizeof u);
  return u;
}
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
  // fp32 add of two bf16 values, then round to nearest even: equal to the
  // correctly rounded bf16 sum (24 >= 2*8+2 bits, double rounding innocuous).
  return pack_bf16x2(bf_lo(a) + bf_lo(b), bf_hi(a) + bf_hi(b));
}
__device__ __forceinline__ uint32_t vword(const uint4& v, int k) {
  return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}

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

// ---- configuration -----------------------------------------------------------

template <int S, bool HAS_DELTA, bool HAS_ONORM, int K>
struct SplitCfg {
  static constexpr int N = S + 1;                       // sources
  static constexpr int NR = 2 * N;                      // sums per token: ss_i, dt_i
  static constexpr int VPC = kNV / K;                   // vectors per CTA
  static constexpr int THREADS = (VPC + 31) / 32 * 32;  // one vector per thread
  static constexpr int NW = THREADS / 32;
  static constexpr bool FULL = (THREADS == VPC);        // no idle threads
  // CTAs of one token exchange partial sums only when there is a softmax
  // (S > 0) or an output norm; otherwise they run as independent CTAs.
  static constexpr bool COMM = (S > 0) || HAS_ONORM;
  static_assert(kNV % K == 0, "split must divide the 896 row vectors");
  static_assert(THREADS <= 1024, "split too small");
};

// ---- the kernel ------------------------------------------------------------------

template <int S, bool HAS_DELTA, bool HAS_ONORM, int K>
__global__ void __launch_bounds__(SplitCfg<S, HAS_DELTA, HAS_ONORM, K>::THREADS)
    attn_res_split_kernel(const Params p) {
  using C = SplitCfg<S, HAS_DELTA, HAS_ONORM, K>;
  constexpr int N = C::N;
  constexpr int NR = C::NR;
  constexpr int NW = C::NW;
  constexpr bool COMM = C::COMM;

  __shared__ float s_warp[NW][NR];  // per-warp partial sums
  __shared__ float s_cta[K][NR];    // per-CTA partial sums of every CTA of the cluster
  __shared__ float s_wt[N];         // softmax weights
  __shared__ float s_warp2[NW];     // output norm: per-warp sum(acc^2)
  __shared__ float s_cta2[K];       // output norm: per-CTA sum(acc^2)

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  // Without a cluster the K CTAs of a token are ordinary neighbours in x.
  const uint32_t rank = COMM ? cluster_ctarank() : (blockIdx.x % K);
  const int64_t t = blockIdx.x / K;
  const bool active = C::FULL || tid < C::VPC;
  const int64_t col = (int64_t)(rank * C::VPC + tid) * kVec;

  // Phase 0 of the cluster barrier: announce that this CTA runs.  Its wait,
  // just before the first DSMEM store, guarantees every peer has started.
  if (COMM) cluster_arrive_relaxed();

  // 1. bank rows: independent of the preceding kernel
  uint4 xb[S > 0 ? S : 1];
#pragma unroll
  for (int i = 0; i < (S > 0 ? S : 1); ++i) xb[i] = make_uint4(0, 0, 0, 0);
  uint4 rw = make_uint4(0, 0, 0, 0), qw = rw, ow = rw, pv = rw, dv = rw;
  if (active) {
    const uint16_t* bp = p.blocks + t * p.blocks_token + col;
#pragma unroll
    for (int i = 0; i < S; ++i) xb[i] = ld_row(bp + (int64_t)i * p.blocks_slot);
    // 2. weights
    rw = ld_weight(p.rms_w + col);
    qw = ld_weight(p.res_w + col);
    if (HAS_ONORM) ow = ld_weight(p.onw + col);
  }
  // 3. prefix and delta come from the preceding kernel (no-op without PDL)
  grid_dep_wait();
  if (active) {
    pv = ld_row(p.prefix + t * p.prefix_row + col);
    if (HAS_DELTA) dv = ld_row(p.delta + t * p.delta_row + col);
  }
  grid_dep_launch_dependents();

  // 4. current-layer row c
  uint4 cv = pv;
  if (HAS_DELTA) {
    cv.x = add_bf16x2(pv.x, dv.x);
    cv.y = add_bf16x2(pv.y, dv.y);
    cv.z = add_bf16x2(pv.z, dv.z);
    cv.w = add_bf16x2(pv.w, dv.w);
  }

  float acc[kVec];
  if constexpr (S == 0) {
    // one source: its softmax weight is exactly 1
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc[2 * k] = bf_lo(vword(cv, k));
      acc[2 * k + 1] = bf_hi(vword(cv, k));
    }
  } else {
    // 5. per-source sum of squares and dot with q
    float q[kVec];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      q[2 * k] = bf_lo(vword(rw, k)) * bf_lo(vword(qw, k));
      q[2 * k + 1] = bf_hi(vword(rw, k)) * bf_hi(vword(qw, k));
    }
    float part[NR];
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const uint4 x = (i < S) ? xb[i < S ? i : 0] : cv;
      float ss = 0.f, dt = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float a = bf_lo(vword(x, k)), b = bf_hi(vword(x, k));
        ss = fmaf(a, a, ss);
        ss = fmaf(b, b, ss);
        dt = fmaf(a, q[2 * k], dt);
        dt = fmaf(b, q[2 * k + 1], dt);
      }
      part[i] = ss;
      part[N + i] = dt;
    }
    // 6. reduce: warp, CTA, cluster
#pragma unroll
    for (int r = 0; r < NR; ++r) part[r] = warp_sum(part[r]);
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < NR; ++r) s_warp[warp][r] = part[r];
    }
    __syncthreads();
    cluster_wait_acquire();  // phase 0: all peers are running
    if (tid < NR) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) s += s_warp[w][tid];
      const uint32_t a = smem_addr(&s_cta[rank][tid]);
#pragma unroll
      for (int r = 0; r < K; ++r) st_dsmem_f32(a, r, s);
    }
    cluster_arrive_release();
    cluster_wait_acquire();  // phase 1: every CTA's sums are in s_cta
    // 7. logits and softmax in warp 0; every CTA sums the same values in the
    // same order, so all CTAs of the token get bit-identical weights.
    if (warp == 0) {
      float tot = 0.f;
      if (lane < NR) {
#pragma unroll
        for (int r = 0; r < K; ++r) tot += s_cta[r][lane];
      }
      const float dtv = __shfl_sync(0xffffffffu, tot, (lane + N) & 31);
      float logit = __int_as_float(0xff800000u);  // -inf
      if (lane < N) logit = dtv / sqrtf(tot / (float)kH + p.eps);
      const float m = warp_max(logit);
      const float e = (lane < N) ? expf(logit - m) : 0.f;
      const float z = warp_sum(e);
      if (lane < N) s_wt[lane] = e / z;
    }
    __syncthreads();
    // 8. mix the raw rows
#pragma unroll
    for (int j = 0; j < kVec; ++j) acc[j] = 0.f;
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float w = s_wt[i];
      const uint4 x = (i < S) ? xb[i < S ? i : 0] : cv;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[2 * k] = fmaf(w, bf_lo(vword(x, k)), acc[2 * k]);
        acc[2 * k + 1] = fmaf(w, bf_hi(vword(x, k)), acc[2 * k + 1]);
      }
    }
  }

  // 9. output RMSNorm on the fp32 accumulator
  float y[kVec];
  if constexpr (HAS_ONORM) {
    float sq = 0.f;
#pragma unroll
    for (int j = 0; j < kVec; ++j) sq = fmaf(acc[j], acc[j], sq);
    sq = warp_sum(sq);
    if (lane == 0) s_warp2[warp] = sq;
    __syncthreads();
    if constexpr (S == 0) cluster_wait_acquire();  // phase 0 not yet waited on
    if (tid == 0) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) s += s_warp2[w];
      const uint32_t a = smem_addr(&s_cta2[rank]);
#pragma unroll
      for (int r = 0; r < K; ++r) st_dsmem_f32(a, r, s);
    }
    cluster_arrive_release();
    cluster_wait_acquire();
    float tot = 0.f;
#pragma unroll
    for (int r = 0; r < K; ++r) tot += s_cta2[r];
    const float ro = 1.0f / sqrtf(tot / (float)kH + p.out_eps);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      y[2 * k] = acc[2 * k] * ro * bf_lo(vword(ow, k));
      y[2 * k + 1] = acc[2 * k + 1] * ro * bf_hi(vword(ow, k));
    }
  } else {
#pragma unroll
    for (int j = 0; j < kVec; ++j) y[j] = acc[j];
  }

  // 10. stores; the write-backs follow every read of this column slice
  if (active) {
    uint4 o;
    o.x = pack_bf16x2(y[0], y[1]);
    o.y = pack_bf16x2(y[2], y[3]);
    o.z = pack_bf16x2(y[4], y[5]);
    o.w = pack_bf16x2(y[6], y[7]);
    st_row(p.out + t * p.out_row + col, o);
    if (HAS_DELTA) st_row(p.prefix + t * p.prefix_row + col, cv);
    if (p.write_idx >= 0)
      st_row(p.blocks + t * p.blocks_token + (int64_t)p.write_idx * p.blocks_slot + col, cv);
  }
}

}  // namespace attn_res_dev
