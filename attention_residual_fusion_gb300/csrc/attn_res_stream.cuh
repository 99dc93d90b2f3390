// attn_res_stream.cuh -- persistent, TMA-fed kernel for many tokens.
//
// Same column split and per-token arithmetic as the split kernel (one cluster
// of K CTAs per token row, CTA r owning a contiguous 1/K of every row, see
// attn_res_token.cuh), but each cluster loops over many tokens and keeps the
// HBM stream going while it computes:
//
//   * the lanes of warp 0 of each CTA issue bulk copies (cp.async.bulk, the
//     TMA engine's one-dimensional form; one lane per bank row) of the CTA's
//     slice of the token's bank rows into one stage of a STAGES-deep
//     shared-memory ring; the copies complete on the stage's `full` mbarrier
//     (expect-tx of the stage bytes);
//   * each thread loads its vectors of the token's prefix and delta rows
//     straight into registers one token ahead, so the ring holds bank rows
//     only -- shared memory, not registers, is what limits how many CTAs
//     (and so how many tokens) an SM keeps in flight;
//   * every thread waits on `full` (bounded: on time-out the kernel records an
//     error bit, stops issuing copies and runs to completion) and reads its
//     vectors straight from the stage, once for the partial sums and once for
//     the mix;
//   * after its last read of the stage each warp arrives on the stage's
//     `empty` mbarrier; thread 0 waits on it, the issuing lanes fence the
//     generic-proxy reads against the async proxy and refill the stage with
//     the token STAGES ahead;
//   * the first token's rows are requested first -- right after the barrier
//     set-up, before the cluster arrival -- and the other stages once they
//     have landed (a staggered start, so the first token's work overlaps the
//     next token's loads);
//   * dependents of a PDL launch are released only when this CTA has run
//     out of tokens (the grid holds every SM until then);
//   * the token phases run software-pipelined: B(j) (softmax, mix), refill,
//     A(j+1) (partial sums of the next token), C(j) (output norm, stores), so
//     one token's exchanges overlap the next token's work.
//
// Staging rows in shared memory with TMA and mbarriers follows the design of
// the kernel excerpted in the prhub summaries of vllm PR #54261 and #50185;
// the pages chunk sources with an online softmax, here a stage holds all bank
// rows of one token slice and the softmax is taken once.
#pragma once

#include "attn_res_token.cuh"

namespace attn_res_dev {

// K = 0: any width H (a multiple of 8) up to kRtMaxK * kRtCols --
// ceil(H / kRtCols) CTAs per token row (read at run time from the cluster
// shape), each owning kRtCols columns and the last one the remainder;
// otherwise K CTAs split the 7168 columns.
constexpr int kRtCols = 1024;
constexpr int kRtMaxK = 16;

// Ring depth of the staged form (STAGED below): as many stages of `rows` row
// slices of `slice_bytes` each as fit when `ctas_per_sm` CTAs share an SM's
// 228 KB of shared memory, each also holding `static_bytes` of static shared
// memory (mailboxes, barriers) and the 1 KB the system reserves, and within
// the 227 KB one CTA may have; at most kStagedMaxStages.  Below 2 the form
// does not exist for that row count.
constexpr int kStagedMaxStages = 8;
__host__ __device__ constexpr int staged_depth(int rows, uint32_t slice_bytes, int ctas_per_sm,
                                               uint32_t static_bytes) {
  const uint32_t per_cta = 233472u / (uint32_t)ctas_per_sm - 1024u - static_bytes;
  const uint32_t cap = 232448u - static_bytes;
  const int n = (int)((per_cta < cap ? per_cta : cap) / ((uint32_t)rows * slice_bytes));
  return n < kStagedMaxStages ? n : kStagedMaxStages;
}
// Static shared memory of a stream CTA: the mailboxes of K CTAs x NW warps
// for S bank rows, and a full and an empty barrier per stage (at most
// kStagedMaxStages).
__host__ __device__ constexpr uint32_t stream_static_bytes(int S, int K, int NW) {
  return (uint32_t)(2 * K * NW * 2 * (S + 1) * 4 + 2 * K * NW * 4 + 32) + 16u * kStagedMaxStages;
}

// STAGED: the ring holds the token's prefix and delta slices as well as its
// bank rows (one stage = S bank rows, prefix, delta), all brought in by bulk
// copies, so no row data waits in registers and the depth is limited by
// shared memory alone.  Without it the ring holds bank rows only and each
// thread loads its prefix and delta vectors into registers one token ahead.
template <int S, bool HAS_DELTA, bool HAS_ONORM, int K, int VPT, int STAGES, bool STAGED = false>
struct StreamCfg {
  static constexpr int VPC = K ? kNV / K : kRtCols / kVec;  // vectors per CTA per row
  static constexpr int THREADS = (VPC / VPT + 31) / 32 * 32;
  static constexpr int NW = THREADS / 32;
  using Tok = TokenCfg<S, HAS_DELTA, HAS_ONORM, K ? K : kRtMaxK, NW>;
  static constexpr bool COMM = Tok::COMM;
  static constexpr uint32_t SLICE_BYTES = VPC * 16;  // one row's slice, multiple of 16
  // row slices per stage: bank rows, then (staged) prefix and delta
  static constexpr int RING_ROWS = S + (STAGED ? (HAS_DELTA ? 2 : 1) : 0);
  static constexpr int PREFIX_ROW = S;       // staged: ring row of the prefix slice
  static constexpr int DELTA_ROW = S + 1;    // staged with delta: ring row of the delta slice
  static constexpr uint32_t STAGE_BYTES = RING_ROWS * SLICE_BYTES;
  static constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES;
  // CTAs per SM that shared memory allows (ring, mailboxes, barriers and the
  // 1 KB the system reserves per CTA, out of 228 KB), but never so many that
  // a thread gets fewer registers than its VPT vectors need (64 + 48 per
  // vector, at most 255): passed to __launch_bounds__ so the register budget
  // matches the occupancy shared memory permits.
  static constexpr uint32_t SMEM_PER_CTA =
      SMEM_BYTES + sizeof(typename Tok::Box) + 16 * STAGES + 1024;
  static constexpr int BY_SMEM = (int)(233472u / SMEM_PER_CTA);
  static constexpr int REG_FLOOR = (64 + (STAGED ? 40 : 48) * VPT) < 255
                                       ? (64 + (STAGED ? 40 : 48) * VPT) : 255;
  static constexpr int BY_REGS = 65536 / (THREADS * REG_FLOOR);
  static constexpr int MIN_BLOCKS_RAW = BY_SMEM < BY_REGS ? BY_SMEM : BY_REGS;
  static constexpr int MIN_BLOCKS = MIN_BLOCKS_RAW < 1 ? 1 : MIN_BLOCKS_RAW;
  static_assert(K == 0 || kNV % K == 0, "split must divide the 896 row vectors");
  static_assert(VPC % VPT == 0, "vectors per thread must divide the slice");
  static_assert(STAGES >= 2 && STAGES <= (STAGED ? kStagedMaxStages : 4), "ring depth");
  static_assert(sizeof(typename Tok::Box) + 16 * STAGES <= stream_static_bytes(S, K ? K : kRtMaxK, NW),
                "static shared memory above the staged-depth estimate");
  static_assert(!STAGED || K != 0, "the staged form is built for the 7168 split only");
  static_assert(RING_ROWS <= 32, "one issuing lane per ring row");
};

// GROUPED: B token rows per bank row with B > 1 possible (else B == 1 and the
// token loop carries no test for it).  RAGGED (K = 0 only): the last CTA of a
// row may own fewer than kRtCols columns (H not a multiple of kRtCols); its
// loads and stores past H are predicated off, its bank-row copies shortened,
// and the tail of its stage slots zeroed.  Without RAGGED every vector of a
// slice is in the row, as the tuned shapes need.
template <int S, bool HAS_DELTA, bool HAS_ONORM, int K, int VPT, int STAGES, bool GROUPED,
          bool RAGGED, bool STAGED>
__device__ __forceinline__ void stream_body(const Params& p, const int64_t T) {
  static_assert(K == 0 || !RAGGED, "only the any-width form has a short last slice");
  using C = StreamCfg<S, HAS_DELTA, HAS_ONORM, K, VPT, STAGES, STAGED>;
  using Tok = typename C::Tok;
  constexpr int VPC = C::VPC;
  constexpr int THREADS = C::THREADS;
  constexpr int NW = C::NW;
  constexpr bool COMM = C::COMM;

  extern __shared__ __align__(128) uint4 ring[];  // [STAGES][RING_ROWS][VPC]
  __shared__ __align__(8) unsigned long long full_bar[STAGES];
  __shared__ __align__(8) unsigned long long empty_bar[STAGES];
  __shared__ typename Tok::Box mb;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  // CTAs per token row and 1 / H: constants, or from the cluster shape
  const Split sp{K ? K : (int)cluster_nctarank(), K ? kInvH : p.inv_h};
  const uint32_t rank = COMM ? cluster_ctarank() : (blockIdx.x % sp.kc);
  const int64_t cid = blockIdx.x / sp.kc;  // cluster (token group) index
  const int64_t ncl = gridDim.x / sp.kc;   // clusters in the grid
  const int64_t ntok = (T > cid) ? (T - cid + ncl - 1) / ncl : 0;
  const int64_t slice0 = (int64_t)rank * VPC * kVec;  // first column of this CTA
  const uint32_t ring_addr = smem_addr(ring);
  // vector v of this thread: index tid + v * THREADS within the CTA's slice
  bool active[VPT];
  int64_t col[VPT];
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    col[v] = slice0 + (int64_t)(tid + v * THREADS) * kVec;
    active[v] = (((v + 1) * THREADS <= VPC) || (tid + v * THREADS < VPC)) &&
                (!RAGGED || col[v] < p.width);
  }
  // bytes of one row's slice of this CTA: fixed, or (ragged) what is left of
  // the row, a multiple of 16
  const uint32_t slice_bytes =
      !RAGGED ? C::SLICE_BYTES
              : (uint32_t)((p.width - slice0 < (int64_t)VPC * kVec ? p.width - slice0
                                                                  : (int64_t)VPC * kVec) * 2);

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), NW);
    }
    if (COMM) mailbox_init(mb);
    fence_mbar_init();
  }
  // ragged: the stage slots are read in full without a predicate; past a
  // short last slice (which the copies do not reach) they hold zeros, so the
  // sums and the mix see zero columns there
  if (RAGGED && slice_bytes < C::SLICE_BYTES) {
    const int tail = (int)(C::SLICE_BYTES - slice_bytes) / 16;
    for (int e = tid; e < STAGES * C::RING_ROWS * tail; e += THREADS)
      ring[(e / tail) * VPC + (int)(slice_bytes / 16) + e % tail] = make_uint4(0, 0, 0, 0);
  }
  // producer side (every lane of warp 0): the bank rows of one token into one
  // stage -- lane 0 arms the stage's barrier with the byte count of the whole
  // stage, then lane i < S issues the copy of bank row i, so the S copies go
  // out as one warp instruction; staged, lanes S and S + 1 copy the prefix
  // and delta slices (issue_current), after the grid-dependency wait
  auto issue_bank = [&](int64_t t, int s) {
    const uint32_t bar = smem_addr(&full_bar[s]);
    if (lane == 0) mbar_arrive_expect_tx(bar, RAGGED ? C::RING_ROWS * slice_bytes : C::STAGE_BYTES);
    __syncwarp();
    if (lane < S)
      bulk_load(ring_addr + (uint32_t)(s * C::RING_ROWS + lane) * C::SLICE_BYTES,
                bank_of<GROUPED>(p, t) + slice0 + (int64_t)lane * p.blocks_slot,
                RAGGED ? slice_bytes : C::SLICE_BYTES, bar);
  };
  auto issue_current = [&](int64_t t, int s) {
    if constexpr (STAGED) {
      const uint32_t bar = smem_addr(&full_bar[s]);
      const uint16_t* src = nullptr;
      if (lane == C::PREFIX_ROW) src = p.prefix + t * p.prefix_row + slice0;
      if (HAS_DELTA && lane == C::DELTA_ROW) src = p.delta + t * p.delta_row + slice0;
      if (src != nullptr)
        bulk_load(ring_addr + (uint32_t)(s * C::RING_ROWS + lane) * C::SLICE_BYTES, src,
                  RAGGED ? slice_bytes : C::SLICE_BYTES, bar);
    }
  };
  // every thread: its vectors of the token's prefix and delta rows
  auto load_current = [&](int64_t t, uint4 (&pre)[VPT], uint4 (&del)[VPT]) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      pre[v] = del[v] = make_uint4(0, 0, 0, 0);
      if (active[v]) {
        pre[v] = ld_row(p.prefix + t * p.prefix_row + col[v]);
        if (HAS_DELTA) del[v] = ld_row(p.delta + t * p.delta_row + col[v]);
      }
    }
  };

  // prologue: the first token's bank rows before the grid-dependency wait;
  // prefix and delta (produced upstream) after it.  The ring's other stages
  // are requested only once the first token's rows have landed (phase A): a
  // staggered start.  Requesting every stage of every CTA at once made the
  // DRAM interleave them all, so the first token's rows landed only at the
  // end of the whole burst and its work could not overlap the next token's
  // loads (measured: decode T = 256 13.9 -> 12.7 µs, T = 1024 with 4 bank
  // rows 23.4 -> 21.9 µs).  Thread 0 also tracks the stages whose last issued
  // copies it has not yet seen complete, and that issue's parity.
  // The first copies go out before the cluster arrival: thread 0 initialised
  // the stage barrier (released by its fence above) and arms it, and the
  // warp barrier in issue_bank orders that before the other lanes' copies.
  uint32_t pending = 0, pending_parity = 0;
  if (warp == 0 && ntok > 0) {
    issue_bank(cid, 0);
    pending = 1u;  // first use of a stage: parity 0 (tracked by thread 0)
  }
  if (COMM) {
    // matched by the wait before the first remote store; the mailbox
    // barriers were released by thread 0's fence, the ragged zero fill needs
    // the release of the arrival itself
    if constexpr (RAGGED) {
      cluster_arrive_release();
    } else {
      cluster_arrive_relaxed();
    }
  } else {
    __syncthreads();
  }
  // weights: read-only, independent of the preceding kernel
  uint4 rw[VPT], qw[VPT], ow[VPT];
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    rw[v] = qw[v] = ow[v] = make_uint4(0, 0, 0, 0);
    if (active[v]) {
      if (S > 0) {  // the query only enters the logits
        rw[v] = ld_weight(p.rms_w + col[v]);
        qw[v] = ld_weight(p.res_w + col[v]);
      }
      if (HAS_ONORM) ow[v] = ld_weight(p.onw + col[v]);
    }
  }
  grid_dep_wait();  // every thread: also orders our stores after the producer's work
  uint4 pre[VPT], del[VPT];  // prefix and delta of the next token to start
  if constexpr (STAGED) {
    if (warp == 0 && ntok > 0) issue_current(cid, 0);
  } else {
    if (ntok > 0) load_current(cid, pre, del);
  }

  f32x2 q[VPT][4];
  make_query<VPT>(rw, qw, q);
  if (COMM) cluster_wait_acquire();

  // Software pipeline over this cluster's tokens: B(j), refill, A(j+1), C(j)
  // (phases in attn_res_token.cuh).  A peer runs at most one token ahead,
  // which the double-buffered mailboxes allow.
  bool failed = false;
  auto stage_of = [&](int64_t j) { return ring + (int)(j % STAGES) * C::RING_ROWS * VPC + tid; };
  // A(j): current row; then, its prefix/delta registers free, the next
  // token's prefix/delta loads go out; then the partial sums.
  auto phase_a = [&](int64_t j, uint4 (&cc)[VPT]) {
    const int s = (int)(j % STAGES);
    const int b = (int)(j & 1);
    if (COMM && tid == 0) mailbox_expect<Tok>(mb, b, HAS_ONORM, sp);
    if constexpr (!STAGED) {
      current_row<HAS_DELTA, VPT>(pre, del, cc);
      if (j + 1 < ntok) load_current(cid + (j + 1) * ncl, pre, del);
    }
    const bool was_failed = failed;
    wait_or_flag(smem_addr(&full_bar[s]), (uint32_t)((j / STAGES) & 1), failed, p.err,
                 kErrStageTimeout);
    if (tid == 0 && !was_failed && !failed) pending &= ~(1u << s);
    // staggered start: token j + 1's rows go out once token j's have landed,
    // until every stage has been used once (first use: parity 0)
    if (warp == 0 && j + 1 < STAGES && j + 1 < ntok &&
        !__any_sync(0xffffffffu, failed)) {
      const int s1 = (int)(j + 1);
      issue_bank(cid + (j + 1) * ncl, s1);
      issue_current(cid + (j + 1) * ncl, s1);
      pending |= 1u << s1;
    }
    const uint4* stage = stage_of(j);
    if constexpr (STAGED) {
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const bool on = RAGGED || active[v];
        pre[v] = on ? stage[C::PREFIX_ROW * VPC + v * THREADS] : make_uint4(0, 0, 0, 0);
        del[v] = (on && HAS_DELTA) ? stage[C::DELTA_ROW * VPC + v * THREADS] : make_uint4(0, 0, 0, 0);
      }
      current_row<HAS_DELTA, VPT>(pre, del, cc);
    }
    token_sums<S, HAS_DELTA, HAS_ONORM, (K ? K : kRtMaxK), NW, VPT>(
        [&](int i, int v) { return (RAGGED || active[v]) ? stage[i * VPC + v * THREADS] : make_uint4(0, 0, 0, 0); },
        cc, q, mb, b, rank, warp, lane, sp);
  };

  uint4 c_cur[VPT];
  if (ntok > 0) phase_a(0, c_cur);
  for (int64_t j = 0; j < ntok; ++j) {
    const int s = (int)(j % STAGES);
    const uint32_t sparity = (uint32_t)((j / STAGES) & 1);
    const int b = (int)(j & 1);                         // mailbox buffer
    const uint32_t bparity = (uint32_t)((j >> 1) & 1);  // its phase parity
    const int64_t t = cid + j * ncl;
    const uint4* stage = stage_of(j);

    // B(j): softmax and mix; each warp releases the stage after its last read
    f32x2 acc[VPT][4];
    token_mix<S, HAS_DELTA, HAS_ONORM, (K ? K : kRtMaxK), NW, VPT>(
        [&](int i, int v) { return (RAGGED || active[v]) ? stage[i * VPC + v * THREADS] : make_uint4(0, 0, 0, 0); },
        mb, b, bparity, rank, warp, lane, p.eps, failed, p.err,
        [&]() {
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&empty_bar[s]));
        },
        c_cur, acc, sp);

    // refill stage s with the token STAGES ahead once every local warp is
    // done: thread 0 waits and decides for warp 0; each issuing lane orders
    // the warps' reads of the stage before its copy with a proxy fence
    if (warp == 0 && j + STAGES < ntok) {
      bool go = false;
      if (lane == 0 && !failed) {
        wait_or_flag(smem_addr(&empty_bar[s]), sparity, failed, p.err, kErrStageTimeout);
        go = !failed;
      }
      go = __shfl_sync(0xffffffffu, go, 0);
      __syncwarp();
      if (go) {
        fence_proxy_async_smem();
        issue_bank(cid + (j + STAGES) * ncl, s);
        issue_current(cid + (j + STAGES) * ncl, s);
        pending |= 1u << s;
        pending_parity = (pending_parity & ~(1u << s)) | ((sparity ^ 1u) << s);
      }
    }

    // A(j+1): next token's partial sums go out while this token's norm
    // exchange is in flight
    uint4 c_next[VPT];
    if (j + 1 < ntok) phase_a(j + 1, c_next);

    // C(j): output norm and stores
    const bool slot_write = writes_slot<GROUPED>(p, t);
    uint16_t* const slot = slot_write ? const_cast<uint16_t*>(bank_of<GROUPED>(p, t)) +
                                            (int64_t)p.write_idx * p.blocks_slot
                                      : nullptr;
    uint4 o[VPT];
    token_finish<S, HAS_DELTA, HAS_ONORM, (K ? K : kRtMaxK), NW, VPT>(
        mb, b, bparity, lane, p.out_eps, failed, p.err, ow, acc, o, sp);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      if (active[v]) {
        st_row(p.out + t * p.out_row + col[v], o[v]);
        if (HAS_DELTA) st_row(p.prefix + t * p.prefix_row + col[v], c_cur[v]);
        if (slot_write) st_row(slot + col[v], c_cur[v]);
      }
      c_cur[v] = c_next[v];
    }
  }

  // This grid occupies every SM until its clusters run out of tokens: let a
  // dependent grid launch only now, so its prologue overlaps our tail instead
  // of taking SM slots from clusters still streaming.
  grid_dep_launch_dependents();

  // After a time-out, do not leave with copies or a peer's partial sums still
  // landing in shared memory: thread 0 (the only one that issues copies, and
  // only while it has not failed) waits, bounded, for the copies it has not
  // seen complete; any thread whose wait timed out waits for the last armed
  // mailbox phases.  The CTA stays resident until its threads are done.
  if (tid == 0 && failed) {
    for (int s = 0; s < STAGES; ++s)
      if (pending & (1u << s))
        (void)mbar_wait_bounded(smem_addr(&full_bar[s]), (pending_parity >> s) & 1u);
  }
  if (COMM && failed) mailbox_drain<Tok>(mb, ntok - 1, HAS_ONORM);
}

template <int S, bool HAS_DELTA, bool HAS_ONORM, int K, int VPT, int STAGES, bool GROUPED,
          bool STAGED>
__global__ void __launch_bounds__(StreamCfg<S, HAS_DELTA, HAS_ONORM, K, VPT, STAGES, STAGED>::THREADS,
                                  StreamCfg<S, HAS_DELTA, HAS_ONORM, K, VPT, STAGES, STAGED>::MIN_BLOCKS)
    attn_res_stream_kernel(const Params p, const int64_t T) {
  stream_body<S, HAS_DELTA, HAS_ONORM, K, VPT, STAGES, GROUPED, false, STAGED>(p, T);
}

// Any width H that is not a multiple of kRtCols (the last CTA's slice short).
template <int S, bool HAS_DELTA, bool HAS_ONORM, int VPT, int STAGES, bool GROUPED>
__global__ void __launch_bounds__(StreamCfg<S, HAS_DELTA, HAS_ONORM, 0, VPT, STAGES>::THREADS,
                                  StreamCfg<S, HAS_DELTA, HAS_ONORM, 0, VPT, STAGES>::MIN_BLOCKS)
    attn_res_stream_ragged_kernel(const Params p, const int64_t T) {
  stream_body<S, HAS_DELTA, HAS_ONORM, 0, VPT, STAGES, GROUPED, true, false>(p, T);
}

}  // namespace attn_res_dev
