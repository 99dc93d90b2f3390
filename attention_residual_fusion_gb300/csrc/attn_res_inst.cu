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
    default: return nullptr;
  }
}

}  // namespace attn_res_host
