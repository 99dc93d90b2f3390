// attn_res_inst.cu -- every specialisation for one num_blocks value.
// Compiled once per S in 0..8 with -DATTN_RES_S=<S>, so the 9 translation
// units build in parallel.
#include <utility>

#include "attn_res_launch.cuh"

#ifndef ATTN_RES_S
#error "compile with -DATTN_RES_S=<num_blocks>"
#endif

#define ATTN_RES_CAT2(a, b) a##b
#define ATTN_RES_CAT(a, b) ATTN_RES_CAT2(a, b)

namespace attn_res_host {

namespace {
template <int K>
LaunchFn pick(bool d, bool o) {
  constexpr int S = ATTN_RES_S;
  if (d) return o ? &launch_split<S, true, true, K> : &launch_split<S, true, false, K>;
  return o ? &launch_split<S, false, true, K> : &launch_split<S, false, false, K>;
}
}  // namespace

LaunchFn ATTN_RES_CAT(launcher_s, ATTN_RES_S)(int split_idx, bool d, bool o) {
  switch (split_idx) {
    case 0: return pick<kSplits[0]>(d, o);
    case 1: return pick<kSplits[1]>(d, o);
    case 2: return pick<kSplits[2]>(d, o);
    case 3: return pick<kSplits[3]>(d, o);
    case 4: return pick<kSplits[4]>(d, o);
    case kAnyWidthSplitIndex: return pick<0>(d, o);
    default: return nullptr;
  }
}

namespace {
// A staged shape exists for this S and delta only if two stages fit.
template <int SH, bool D>
StreamLaunchFn pick_staged(bool o) {
  constexpr int S = ATTN_RES_S;
  constexpr StreamShape sh = kStreamShapes[SH];
  constexpr int ST = staged_stages(sh, S, D);
  if constexpr (ST < 2) {
    return nullptr;
  } else {
    return o ? &launch_stream<S, D, true, sh.k, sh.vpt, ST, sh.grouped, true>
             : &launch_stream<S, D, false, sh.k, sh.vpt, ST, sh.grouped, true>;
  }
}

template <int SH>
StreamLaunchFn pick_stream(bool d, bool o) {
  constexpr int S = ATTN_RES_S;
  constexpr int K = kStreamShapes[SH].k;
  constexpr int V = kStreamShapes[SH].vpt;
  constexpr int ST = kStreamShapes[SH].stages;
  constexpr bool G = kStreamShapes[SH].grouped;
  if constexpr (kStreamShapes[SH].staged) {
    return d ? pick_staged<SH, true>(o) : pick_staged<SH, false>(o);
  } else {
    if (d) return o ? &launch_stream<S, true, true, K, V, ST, G> : &launch_stream<S, true, false, K, V, ST, G>;
    return o ? &launch_stream<S, false, true, K, V, ST, G> : &launch_stream<S, false, false, K, V, ST, G>;
  }
}

template <int... I>
StreamLaunchFn pick_stream_at(int shape_idx, bool d, bool o, std::integer_sequence<int, I...>) {
  StreamLaunchFn fn = nullptr;
  ((shape_idx == I ? (fn = pick_stream<I>(d, o), 0) : 0), ...);
  return fn;
}
}  // namespace

StreamLaunchFn ATTN_RES_CAT(stream_launcher_s, ATTN_RES_S)(int shape_idx, bool d, bool o) {
  return pick_stream_at(shape_idx, d, o, std::make_integer_sequence<int, kNumStreamShapes>{});
}

namespace {
template <int V>
RowLaunchFn pick_row(bool d, bool o) {
  constexpr int S = ATTN_RES_S;
  if (d) return o ? &launch_row<S, true, true, V> : &launch_row<S, true, false, V>;
  return o ? &launch_row<S, false, true, V> : &launch_row<S, false, false, V>;
}
}  // namespace

RowLaunchFn ATTN_RES_CAT(row_launcher_s, ATTN_RES_S)(int vpt_idx, bool d, bool o) {
  static_assert(kNumRowVpts == 2, "update the switch below");
  if constexpr (ATTN_RES_S > kRowMaxBlocks) {
    return nullptr;
  } else {
    switch (vpt_idx) {
      case 0: return pick_row<kRowVpts[0]>(d, o);
      case 1: return pick_row<kRowVpts[1]>(d, o);
      default: return nullptr;
    }
  }
}

namespace {
template <int V>
RowLaunchFn pick_row_smem(bool d, bool o) {
  constexpr int S = ATTN_RES_S;
  if (d) return o ? &launch_row_smem<S, true, true, V> : &launch_row_smem<S, true, false, V>;
  return o ? &launch_row_smem<S, false, true, V> : &launch_row_smem<S, false, false, V>;
}
}  // namespace

RowLaunchFn ATTN_RES_CAT(row_smem_launcher_s, ATTN_RES_S)(int vpt_idx, bool d, bool o) {
  if constexpr (ATTN_RES_S < kRowSmemMinBlocks || ATTN_RES_S > kRowSmemMaxBlocks) {
    return nullptr;
  } else {
    switch (vpt_idx) {
      case 0: return pick_row_smem<kRowVpts[0]>(d, o);
      case 1: return pick_row_smem<kRowVpts[1]>(d, o);
      default: return nullptr;
    }
  }
}

GenericLaunchFn ATTN_RES_CAT(generic_launcher_s, ATTN_RES_S)(bool d, bool o) {
  constexpr int S = ATTN_RES_S;
  if (d) return o ? &launch_generic<S, true, true> : &launch_generic<S, true, false>;
  return o ? &launch_generic<S, false, true> : &launch_generic<S, false, false>;
}

template <int S, bool D>
TpLaunchFn tp_finish_fn(bool o, bool g) {
  if (o) return g ? &launch_tp_finish<S, D, true, true> : &launch_tp_finish<S, D, true, false>;
  return &launch_tp_finish<S, D, false, false>;  // without an output norm GRAM changes nothing
}

TpLaunchFn ATTN_RES_CAT(tp_launcher_s, ATTN_RES_S)(int phase, bool d, bool o, bool g) {
  constexpr int S = ATTN_RES_S;
  switch (phase) {
    case 0:
      if (d) return g ? &launch_tp_sums<S, true, true> : &launch_tp_sums<S, true, false>;
      return g ? &launch_tp_sums<S, false, true> : &launch_tp_sums<S, false, false>;
    case 1: return d ? &launch_tp_sq<S, true> : &launch_tp_sq<S, false>;
    case 2: return d ? tp_finish_fn<S, true>(o, g) : tp_finish_fn<S, false>(o, g);
    default: return nullptr;
  }
}

template <int S, bool D>
TpRingLaunchFn tp_ring_fn(int phase, bool o, bool g) {
  switch (phase) {
    case 0: return g ? &launch_tp_ring<S, D, 0, false, true> : &launch_tp_ring<S, D, 0, false, false>;
    case 1: return &launch_tp_ring<S, D, 1, true, false>;
    case 2:
      if (o) return g ? &launch_tp_ring<S, D, 2, true, true> : &launch_tp_ring<S, D, 2, true, false>;
      return &launch_tp_ring<S, D, 2, false, false>;  // without an output norm GRAM changes nothing
    default: return nullptr;
  }
}

TpRingLaunchFn ATTN_RES_CAT(tp_ring_launcher_s, ATTN_RES_S)(int phase, bool d, bool o, bool g) {
  constexpr int S = ATTN_RES_S;
  return d ? tp_ring_fn<S, true>(phase, o, g) : tp_ring_fn<S, false>(phase, o, g);
}

}  // namespace attn_res_host
