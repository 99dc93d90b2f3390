// attn_res_kernel.cuh -- the split kernel: one thread-block cluster per token.
//
// A token row of H = 7168 bf16 is split over the K CTAs of one cluster; CTA r
// owns the contiguous column slice [r*H/K, (r+1)*H/K) of every source row,
// one 16-byte vector (8 bf16) per thread.  Each thread issues all of its row
// loads at once (up to 8 bank rows, the prefix row and the delta row: 160 B
// in flight per thread) and keeps them in registers, so every byte is read
// from HBM exactly once:
//
//   bank rows, weights      -> loaded before the grid-dependency wait
//   griddepcontrol.wait     -> prefix (and delta) are produced upstream
//   griddepcontrol.launch_dependents
//   mix_token: c, partial sums, DSMEM mailbox exchange, softmax, mix,
//              output norm (see attn_res_token.cuh)
//   stores: out, then the write-backs of c (prefix, bank slot)
//
// This is the latency path for few tokens.  The pages' SM100 kernel (prhub
// summaries of vllm PR #54261 and #50185) streams rows through a shared-memory
// ring with an online softmax per source chunk; here a token's column slice
// sits in registers and the softmax is taken once, after one exchange.
#pragma once

#include "attn_res_token.cuh"

namespace attn_res_dev {

// K = 0: any width H (a multiple of 8) up to 8192 -- ceil(H / 1024) CTAs per
// token row (read from the cluster shape), 1024 columns each, the last CTA
// the remainder.
constexpr int kSplitRtMaxK = 8;

template <int S, bool HAS_DELTA, bool HAS_ONORM, int K>
struct SplitCfg {
  static constexpr int VPC = K ? kNV / K : 1024 / kVec;  // vectors per CTA
  static constexpr int THREADS = (VPC + 31) / 32 * 32;  // one vector per thread
  static constexpr int NW = THREADS / 32;
  static constexpr bool FULL = (THREADS == VPC);        // no idle threads
  using Tok = TokenCfg<S, HAS_DELTA, HAS_ONORM, K ? K : kSplitRtMaxK, NW>;
  // CTAs of one token exchange partial sums only when there is a softmax
  // (S > 0) or an output norm; otherwise they run as independent CTAs.
  static constexpr bool COMM = Tok::COMM;
  static_assert(kNV % (K ? K : 1) == 0, "split must divide the 896 row vectors");
  static_assert(THREADS <= 1024, "split too small");
  static_assert(K * NW <= 32, "one lane per mailbox slot");
};

template <int S, bool HAS_DELTA, bool HAS_ONORM, int K>
__global__ void __launch_bounds__(SplitCfg<S, HAS_DELTA, HAS_ONORM, K>::THREADS)
    attn_res_split_kernel(const Params p) {
  using C = SplitCfg<S, HAS_DELTA, HAS_ONORM, K>;
  using Tok = typename C::Tok;
  constexpr int ROWS = Tok::ROWS;
  constexpr bool COMM = C::COMM;

  __shared__ typename Tok::Box mb;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  // CTAs per token row and 1 / H: constants, or from the cluster shape
  const Split sp{K ? K : (int)cluster_nctarank(), K ? kInvH : p.inv_h};
  // Without a cluster the CTAs of a token are ordinary neighbours in x.
  const uint32_t rank = COMM ? cluster_ctarank() : (blockIdx.x % sp.kc);
  const int64_t t = blockIdx.x / sp.kc;
  const int64_t col = (int64_t)(rank * C::VPC + tid) * kVec;
  // the last CTA of an any-width row may own fewer than 1024 columns
  const bool active = (C::FULL || tid < C::VPC) && (K != 0 || col < p.width);

  if (COMM) {
    if (tid == 0) {
      mailbox_init(mb);
      fence_mbar_init();
      mailbox_expect<Tok>(mb, 0, HAS_ONORM, sp);
    }
    // Announce this CTA (its mailboxes initialised and released by the fence
    // above) to the cluster; the matching wait, just before the first remote
    // store, guarantees every peer is running and ready to receive.
    cluster_arrive_relaxed();
  }

  // 1. bank rows: independent of the preceding kernel
  uint4 x[ROWS];
#pragma unroll
  for (int i = 0; i < ROWS; ++i) x[i] = make_uint4(0, 0, 0, 0);
  uint4 rw = make_uint4(0, 0, 0, 0), qw = rw, ow = rw;
  if (active) {
    const uint16_t* bp = bank_of(p, t) + col;
#pragma unroll
    for (int i = 0; i < S; ++i) x[i] = ld_row(bp + (int64_t)i * p.blocks_slot);
    // 2. weights
    rw = ld_weight(p.rms_w + col);
    qw = ld_weight(p.res_w + col);
    if (HAS_ONORM) ow = ld_weight(p.onw + col);
  }
  // 3. prefix and delta come from the preceding kernel (no-op without PDL)
  grid_dep_wait();
  if (active) {
    x[S] = ld_row(p.prefix + t * p.prefix_row + col);
    if (HAS_DELTA) x[S + 1] = ld_row(p.delta + t * p.delta_row + col);
  }
  grid_dep_launch_dependents();

  uint4 rwv[1] = {rw}, qwv[1] = {qw}, owv[1] = {ow};
  f32x2 q[1][4];
  make_query<1>(rwv, qwv, q);
  if (COMM) cluster_wait_acquire();

  bool failed = false;
  uint4 c[1], o[1];
  {
    const uint4 pre[1] = {x[S]}, del[1] = {x[ROWS - 1]};
    current_row<HAS_DELTA, 1>(pre, del, c);
  }
  mix_token<S, HAS_DELTA, HAS_ONORM, (K ? K : kSplitRtMaxK), C::NW, 1>(
      [&](int i, int) { return x[i]; }, q, owv, mb, 0, 0u, rank, warp, lane, p.eps, p.out_eps,
      failed, p.err, [] {}, c, o, sp);

  // 4. stores; the write-backs follow every read of this column slice
  if (active) {
    st_row(p.out + t * p.out_row + col, o[0]);
    if (HAS_DELTA) st_row(p.prefix + t * p.prefix_row + col, c[0]);
    if (writes_slot(p, t))
      st_row(const_cast<uint16_t*>(bank_of(p, t)) + (int64_t)p.write_idx * p.blocks_slot + col,
             c[0]);
  }
  // No drain of the mailboxes on the time-out path here (the stream kernel
  // has one): on this latency path even an untaken branch to it at the end
  // measured 0.1 µs per call (T = 1, 4 bank rows: 2.88 -> 2.99 µs).
}

}  // namespace attn_res_dev
