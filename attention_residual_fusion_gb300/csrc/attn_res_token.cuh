// attn_res_token.cuh -- the mixture for one token, as seen by one thread
// that owns VPT 16-byte vectors (8 columns each) of every source row; shared
// by the split and the stream kernels.
//
// Per token (implementation walkthrough of vllm-ascend PR #14840; delta
// packing and output norm from the key source excerpts of vllm PR #54261):
//   c = bf16_rn(prefix + delta); per source i: ss_i = sum x^2, dt_i = <x, q>;
//   l_i = dt_i / sqrt(ss_i / H + eps); w = softmax(l); acc = sum_i w_i x_i;
//   optional out = acc / sqrt(mean(acc^2) + out_eps) * w_out.
//
// The full-row sums cross the K CTAs of the cluster through mailboxes in
// shared memory: every warp reduces its partial sums (reduce-scatter), and
// the lanes holding them store each one into the mailbox of every CTA of the
// cluster with st.async, which completes transaction bytes on the receiver's
// mbarrier.  A warp waits on its own CTA's mbarrier until all K x NW partial
// vectors have landed, then sums them in a fixed order -- so every warp of
// every CTA of the token computes bit-identical logits and weights, with no
// CTA barrier, no cluster barrier and no memory fence on the way.
// Elementwise products use packed fp32 pairs (fma.rn.f32x2).
#pragma once

#include "attn_res_common.cuh"

namespace attn_res_dev {

// Mailboxes of one CTA, double-buffered by token parity (a peer may run one
// token ahead; it cannot run two ahead, since it needs this CTA's sums of the
// token in between).
template <int K, int NW, int NR>
struct Mailbox {
  float sums[2][K * NW][NR];  // per source CTA and warp: ss_0..ss_S, dt_0..dt_S
  float sq[2][K * NW];        // per source CTA and warp: sum of acc^2
  unsigned long long bar_sums[2];
  unsigned long long bar_sq[2];
};

// The 2N per-source sums of a token (sum(x_i^2), then <x_i, q>) as a warp
// reduces them: one power-of-two butterfly of P values, plus a second one of
// P2 values when NR is just above a power of two (NR = 18 for S = 8 reduces
// as 16 + 2 instead of a padded 32).
template <int S>
struct SumsCfg {
  static constexpr int N = S + 1;              // sources
  static constexpr int NR = 2 * N;             // partial sums per token
  static constexpr int P_FULL = pow2_at_least(NR);
  static constexpr int P = (NR > 16) ? 16 : P_FULL;
  static constexpr int NR2 = NR - P > 0 ? NR - P : 0;  // values in the second butterfly
  static constexpr int P2 = NR2 > 0 ? pow2_at_least(NR2) : 1;
  static constexpr int SHIFT = 5 - log2_exact(P);
  static constexpr int SHIFT2 = 5 - log2_exact(P2);
  static_assert(NR2 <= 16, "second butterfly too large");
  static_assert(NR <= 32, "one lane per sum");
};

template <int S, bool HAS_DELTA, bool HAS_ONORM, int K, int NW>
struct TokenCfg : SumsCfg<S> {
  using Sums = SumsCfg<S>;
  using Sums::N;
  using Sums::NR;
  using Sums::P;
  using Sums::NR2;
  using Sums::P2;
  using Sums::SHIFT;
  using Sums::SHIFT2;
  static constexpr int ROWS = N + (HAS_DELTA ? 1 : 0);
  static constexpr uint32_t SUMS_BYTES = K * NW * NR * 4;  // expected per token
  static constexpr uint32_t SQ_BYTES = K * NW * 4;
  static constexpr bool COMM = (S > 0) || HAS_ONORM;
  static constexpr int NWARPS = NW;
  using Box = Mailbox<K, NW, NR>;  // sized for up to K CTAs
  static_assert(K * NW <= 32, "one lane per mailbox slot");
};

// Initialise the mailbox barriers (thread 0 of the CTA).
template <class Box>
__device__ __forceinline__ void mailbox_init(Box& mb) {
  for (int b = 0; b < 2; ++b) {
    mbar_init(smem_addr(&mb.bar_sums[b]), 1);
    mbar_init(smem_addr(&mb.bar_sq[b]), 1);
  }
}

// The row split: kc CTAs per token row (<= the K the mailboxes are sized
// for) and 1 / H for the means.  Kernels built for one width pass constants.
struct Split {
  int kc;
  float inv_h;
};

// Thread 0, once per token before waiting: the one arrival of this phase,
// with the byte count the peers' stores will complete.
template <class Cfg>
__device__ __forceinline__ void mailbox_expect(typename Cfg::Box& mb, int b, bool has_onorm,
                                               Split sp) {
  const uint32_t senders = (uint32_t)(sp.kc * Cfg::NWARPS);
  if (Cfg::N > 1) mbar_arrive_expect_tx(smem_addr(&mb.bar_sums[b]), senders * Cfg::NR * 4u);
  if (has_onorm) mbar_arrive_expect_tx(smem_addr(&mb.bar_sq[b]), senders * 4u);
}

// Time-out path only (a thread whose wait gave up, at exit): wait, bounded,
// for the last phase armed on each mailbox buffer -- token `last` and the one
// before it -- so that no peer's partial sums still land in this CTA's shared
// memory after it exits.  A phase that already completed returns at once;
// several threads may wait on one phase.
template <class Cfg>
__device__ __forceinline__ void mailbox_drain(typename Cfg::Box& mb, int64_t last, bool has_onorm) {
  for (int64_t j = last; j >= 0 && j >= last - 1; --j) {
    const int b = (int)(j & 1);
    const uint32_t parity = (uint32_t)((j >> 1) & 1);
    if (Cfg::N > 1) (void)mbar_wait_bounded(smem_addr(&mb.bar_sums[b]), parity);
    if (has_onorm) (void)mbar_wait_bounded(smem_addr(&mb.bar_sq[b]), parity);
  }
}

// q = rms_w * res_w for the thread's columns, as fp32 pairs.
template <int VPT>
__device__ __forceinline__ void make_query(const uint4 (&rw)[VPT], const uint4 (&qw)[VPT],
                                           f32x2 (&q)[VPT][4]) {
#pragma unroll
  for (int v = 0; v < VPT; ++v)
#pragma unroll
    for (int k = 0; k < 4; ++k)
      q[v][k] = f2_mul(bf2_widen(vword(rw[v], k)), bf2_widen(vword(qw[v], k)));
}

// The token runs in three phases so that a persistent kernel can overlap one
// token's exchanges with the next token's work:
//   A  token_sums:   current-layer row c, partial sums, send them to every CTA
//   B  token_mix:    wait for all sums, softmax, mix, release the row data,
//                    send sum(acc^2) (output norm)
//   C  token_finish: wait for all sum(acc^2), scale, pack the output
// Rows are zeros for idle threads.  b / parity: mailbox buffer of this token
// and its phase parity.

// Current-layer row from this thread's prefix and delta vectors.
template <bool HAS_DELTA, int VPT>
__device__ __forceinline__ void current_row(const uint4 (&pre)[VPT], const uint4 (&del)[VPT],
                                            uint4 (&c)[VPT]) {
#pragma unroll
  for (int v = 0; v < VPT; ++v) c[v] = HAS_DELTA ? add_bf16x8(pre[v], del[v]) : pre[v];
}

// ---- per-token building blocks (any transport of the sums) ----------------------
// row(i, v): vector v of bank row i < S; c: the current-layer row (the last
// source).

// The thread's partial sums over its VPT vectors of every source, reduced
// over the warp.  On return lane l holds in `lo` the warp total of sum
// l >> SHIFT (meaningful where lo_holder(l)) and in `hi` the total of sum
// P + (l >> SHIFT2) (where hi_holder(l)).
template <int S, int VPT, class Row>
__device__ __forceinline__ void warp_sums(Row row, const uint4 (&c)[VPT], const f32x2 (&q)[VPT][4],
                                          int lane, float& lo, float& hi) {
  using C = SumsCfg<S>;
  constexpr int N = C::N;
  constexpr int P = C::P;
  constexpr int P2 = C::P2;
  float part[P + P2];
#pragma unroll
  for (int r = 0; r < P + P2; ++r) part[r] = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    f32x2 ss = 0ull, dt = 0ull;  // +0.0f pairs
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const uint4 xi = (i < S) ? row(i < S ? i : 0, v) : c[v];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const f32x2 x2 = bf2_widen(vword(xi, k));
        ss = f2_fma(x2, x2, ss);
        dt = f2_fma(x2, q[v][k], dt);
      }
    }
    part[i] = f2_lo(ss) + f2_hi(ss);
    part[N + i] = f2_lo(dt) + f2_hi(dt);
  }
  float a[P];
#pragma unroll
  for (int r = 0; r < P; ++r) a[r] = part[r];
  lo = reduce_scatter<P>(a, lane);
  hi = 0.f;
  if constexpr (C::NR2 > 0) {
    float b[P2];
#pragma unroll
    for (int r = 0; r < P2; ++r) b[r] = part[P + r];
    hi = reduce_scatter<P2>(b, lane);
  }
}
// Which lanes hold a sum after warp_sums, and its index.
template <int S>
__device__ __forceinline__ bool lo_holder(int lane) {
  using C = SumsCfg<S>;
  return (lane & ((1 << C::SHIFT) - 1)) == 0 && (lane >> C::SHIFT) < (C::NR < C::P ? C::NR : C::P);
}
template <int S>
__device__ __forceinline__ int lo_index(int lane) { return lane >> SumsCfg<S>::SHIFT; }
template <int S>
__device__ __forceinline__ bool hi_holder(int lane) {
  using C = SumsCfg<S>;
  return C::NR2 > 0 && (lane & ((1 << C::SHIFT2) - 1)) == 0 && (lane >> C::SHIFT2) < C::NR2;
}
template <int S>
__device__ __forceinline__ int hi_index(int lane) { return SumsCfg<S>::P + (lane >> SumsCfg<S>::SHIFT2); }

// Logits and softmax from the token totals (lane l < NR holds sum l); lane
// i < N returns w_i.  Reciprocal square root and a fast quotient (z in
// [1, N]): a few ulp of fp32 on the weights, far below the bf16 output's
// resolution, and the same instructions in every warp, so the weights are
// bit-identical wherever they are computed from the same totals.
template <int S>
__device__ __forceinline__ float softmax_weight(float tot, int lane, float eps, float inv_h) {
  constexpr int N = S + 1;
  const float dtv = __shfl_sync(0xffffffffu, tot, (lane + N) & 31);
  float logit = __int_as_float(0xff800000u);  // -inf
  if (lane < N) logit = dtv * rsqrtf(fmaf(tot, inv_h, eps));
  const float m = warp_max(logit);
  const float e = (lane < N) ? expf(logit - m) : 0.f;
  const float z = warp_sum(e);
  return __fdividef(e, z);
}

// acc = sum_i w_i x_i over the raw rows; lane i holds w_i in `wl`.
template <int S, int VPT, class Row>
__device__ __forceinline__ void mix_rows(Row row, const uint4 (&c)[VPT], float wl,
                                         f32x2 (&acc)[VPT][4]) {
  constexpr int N = S + 1;
#pragma unroll
  for (int v = 0; v < VPT; ++v)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[v][k] = 0ull;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float w = __shfl_sync(0xffffffffu, wl, i);
    const f32x2 w2 = f2_make(w, w);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const uint4 xi = (i < S) ? row(i < S ? i : 0, v) : c[v];
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[v][k] = f2_fma(w2, bf2_widen(vword(xi, k)), acc[v][k]);
    }
  }
}

// The warp's sum of acc^2 over its columns (every lane gets it).
template <int VPT>
__device__ __forceinline__ float warp_sq(const f32x2 (&acc)[VPT][4]) {
  f32x2 sq2 = 0ull;
#pragma unroll
  for (int v = 0; v < VPT; ++v)
#pragma unroll
    for (int k = 0; k < 4; ++k) sq2 = f2_fma(acc[v][k], acc[v][k], sq2);
  return warp_sum(f2_lo(sq2) + f2_hi(sq2));
}

// Output vectors: acc scaled by ro and the norm weights (output norm), or acc
// itself, rounded to bf16.
template <bool HAS_ONORM, int VPT>
__device__ __forceinline__ void pack_out(f32x2 (&acc)[VPT][4], const uint4 (&ow)[VPT], float ro,
                                         uint4 (&out)[VPT]) {
  if constexpr (HAS_ONORM) {
    const f32x2 ro2 = f2_make(ro, ro);
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[v][k] = f2_mul(f2_mul(acc[v][k], ro2), bf2_widen(vword(ow[v], k)));
  }
#pragma unroll
  for (int v = 0; v < VPT; ++v)
    out[v] = make_uint4(pack_bf16x2(f2_lo(acc[v][0]), f2_hi(acc[v][0])),
                        pack_bf16x2(f2_lo(acc[v][1]), f2_hi(acc[v][1])),
                        pack_bf16x2(f2_lo(acc[v][2]), f2_hi(acc[v][2])),
                        pack_bf16x2(f2_lo(acc[v][3]), f2_hi(acc[v][3])));
}

// ---- the three phases over the cluster's mailboxes -----------------------------

template <int S, bool HAS_DELTA, bool HAS_ONORM, int K, int NW, int VPT, class Row>
__device__ __forceinline__ void token_sums(Row row, const uint4 (&c)[VPT],
                                           const f32x2 (&q)[VPT][4],
                                           typename TokenCfg<S, HAS_DELTA, HAS_ONORM, K, NW>::Box& mb,
                                           int b, uint32_t rank, int warp, int lane, Split sp) {
  if constexpr (S > 0) {
    // warp totals, then into every CTA's mailbox
    float tv, tv2;
    warp_sums<S, VPT>(row, c, q, lane, tv, tv2);
    const int src = (int)rank * NW + warp;
    const uint32_t bar = smem_addr(&mb.bar_sums[b]);
    if (lo_holder<S>(lane)) {
      const uint32_t a = smem_addr(&mb.sums[b][src][lo_index<S>(lane)]);
#pragma unroll
      for (int r = 0; r < sp.kc; ++r) st_async_f32(map_rank(a, r), tv, map_rank(bar, r));
    }
    if (hi_holder<S>(lane)) {
      const uint32_t a = smem_addr(&mb.sums[b][src][hi_index<S>(lane)]);
#pragma unroll
      for (int r = 0; r < sp.kc; ++r) st_async_f32(map_rank(a, r), tv2, map_rank(bar, r));
    }
  }
}

// after_mix(): called once the thread no longer needs any row data.
template <int S, bool HAS_DELTA, bool HAS_ONORM, int K, int NW, int VPT, class Row,
          class AfterMix>
__device__ __forceinline__ void token_mix(Row row,
                                          typename TokenCfg<S, HAS_DELTA, HAS_ONORM, K, NW>::Box& mb,
                                          int b, uint32_t parity, uint32_t rank, int warp,
                                          int lane, float eps, bool& failed, unsigned* err,
                                          AfterMix after_mix, const uint4 (&c)[VPT],
                                          f32x2 (&acc)[VPT][4], Split sp) {
  using C = TokenCfg<S, HAS_DELTA, HAS_ONORM, K, NW>;
  constexpr int NR = C::NR;
  if constexpr (S == 0) {
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[v][k] = bf2_widen(vword(c[v], k));
    after_mix();
  } else {
    wait_or_flag(smem_addr(&mb.bar_sums[b]), parity, failed, err, kErrExchangeTimeout);
    // token totals in a fixed order, logits and softmax (every warp)
    float tot = 0.f;
    if (lane < NR) {
#pragma unroll 4
      for (int s = 0; s < sp.kc * NW; ++s) tot += mb.sums[b][s][lane];
    }
    const float wl = softmax_weight<S>(tot, lane, eps, sp.inv_h);
    mix_rows<S, VPT>(row, c, wl, acc);
    after_mix();
  }
  if constexpr (HAS_ONORM) {
    const float sq = warp_sq<VPT>(acc);
    if (lane < sp.kc)
      st_async_f32(map_rank(smem_addr(&mb.sq[b][(int)rank * NW + warp]), lane), sq,
                   map_rank(smem_addr(&mb.bar_sq[b]), lane));
  }
}

template <int S, bool HAS_DELTA, bool HAS_ONORM, int K, int NW, int VPT>
__device__ __forceinline__ void token_finish(typename TokenCfg<S, HAS_DELTA, HAS_ONORM, K, NW>::Box& mb,
                                             int b, uint32_t parity, int lane, float out_eps,
                                             bool& failed, unsigned* err, const uint4 (&ow)[VPT],
                                             f32x2 (&acc)[VPT][4], uint4 (&out)[VPT], Split sp) {
  float ro = 1.f;
  if constexpr (HAS_ONORM) {
    wait_or_flag(smem_addr(&mb.bar_sq[b]), parity, failed, err, kErrExchangeTimeout);
    const float tot = warp_sum(lane < sp.kc * NW ? mb.sq[b][lane] : 0.f);
    ro = rsqrtf(fmaf(tot, sp.inv_h, out_eps));
  }
  pack_out<HAS_ONORM, VPT>(acc, ow, ro, out);
}

// The three phases back to back (one token, no overlap); c must hold the
// current-layer row.
template <int S, bool HAS_DELTA, bool HAS_ONORM, int K, int NW, int VPT, class Row,
          class AfterMix>
__device__ __forceinline__ void mix_token(Row row, const f32x2 (&q)[VPT][4],
                                          const uint4 (&ow)[VPT],
                                          typename TokenCfg<S, HAS_DELTA, HAS_ONORM, K, NW>::Box& mb,
                                          int b, uint32_t parity, uint32_t rank, int warp,
                                          int lane, float eps, float out_eps, bool& failed,
                                          unsigned* err, AfterMix after_mix, const uint4 (&c)[VPT],
                                          uint4 (&out)[VPT], Split sp) {
  f32x2 acc[VPT][4];
  token_sums<S, HAS_DELTA, HAS_ONORM, K, NW, VPT>(row, c, q, mb, b, rank, warp, lane, sp);
  token_mix<S, HAS_DELTA, HAS_ONORM, K, NW, VPT>(row, mb, b, parity, rank, warp, lane, eps, failed,
                                                 err, after_mix, c, acc, sp);
  token_finish<S, HAS_DELTA, HAS_ONORM, K, NW, VPT>(mb, b, parity, lane, out_eps, failed, err, ow,
                                                    acc, out, sp);
}

}  // namespace attn_res_dev
