// attn_res_inst.cu -- every specialisation for one num_blocks value.
// Compiled once per S in 0..8 with -DATTN_RES_S=<S>, so the 9 translation
// units build in parallel.
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
template <int SH>
StreamLaunchFn pick_stream(bool d, bool o) {
  constexpr int S = ATTN_RES_S;
  constexpr int K = kStreamShapes[SH].k;
  constexpr int V = kStreamShapes[SH].vpt;
  constexpr int ST = kStreamShapes[SH].stages;
  constexpr bool G = kStreamShapes[SH].grouped;
  if (d) return o ? &launch_stream<S, true, true, K, V, ST, G> : &launch_stream<S, true, false, K, V, ST, G>;
  return o ? &launch_stream<S, false, true, K, V, ST, G> : &launch_stream<S, false, false, K, V, ST, G>;
}
}  // namespace

StreamLaunchFn ATTN_RES_CAT(stream_launcher_s, ATTN_RES_S)(int shape_idx, bool d, bool o) {
  static_assert(kNumStreamShapes == 11, "update the switch below");
  switch (shape_idx) {
    case 0: return pick_stream<0>(d, o);
    case 1: return pick_stream<1>(d, o);
    case 2: return pick_stream<2>(d, o);
    case 3: return pick_stream<3>(d, o);
    case 4: return pick_stream<4>(d, o);
    case 5: return pick_stream<5>(d, o);
    case 6: return pick_stream<6>(d, o);
    case 7: return pick_stream<7>(d, o);
    case 8: return pick_stream<8>(d, o);
    case 9: return pick_stream<9>(d, o);
    case 10: return pick_stream<10>(d, o);
    default: return nullptr;
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
