// attn_res_generic.cuh -- the mixture for any hidden size H (a multiple of 8).
//
// One CTA of 256 threads per token row; thread `tid` owns the 16-byte
// vectors tid, tid + 256, ... of every row, so any H works.  The CTA makes
// three passes over the token's rows (the second and third mostly hit L2):
//   1. current row c, per-source sum of squares and dot with q; CTA-wide
//      reduction, logits and softmax (implementation walkthrough of
//      vllm-ascend PR #14840);
//   2. with an output norm only: sum of acc^2 over the row;
//   3. acc = sum_i w_i x_i, output (normalised when asked), and the
//      write-backs of c -- each thread writes only vectors it alone reads, so
//      no barrier is needed between its reads and its writes.
// This is the functional path for widths that are not multiples of 1024 and
// for checking the GPU arithmetic at tiny H; H = 7168 uses the split and
// stream kernels, other multiples of 1024 the stream kernel's any-width form.
#pragma once

#include "attn_res_common.cuh"

namespace attn_res_dev {

constexpr int kGenericThreads = 256;
constexpr int kGenericWarps = kGenericThreads / 32;

template <int S, bool HAS_DELTA, bool HAS_ONORM>
__global__ void __launch_bounds__(kGenericThreads)
    attn_res_generic_kernel(const Params p, const int64_t H) {
  constexpr int N = S + 1;
  constexpr int NR = 2 * N;
  __shared__ float s_part[kGenericWarps][NR];
  __shared__ float s_wt[N];
  __shared__ float s_sq[kGenericWarps];
  __shared__ float s_ro;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int64_t t = blockIdx.x;
  const int64_t nv = H / kVec;

  grid_dep_wait();  // no loads before the producer of prefix / delta is done
  uint16_t* const bank_row = const_cast<uint16_t*>(bank_of(p, t));
  const bool slot_write = writes_slot(p, t);

  auto current = [&](int64_t col) -> uint4 {
    const uint4 pv = ld_row(p.prefix + t * p.prefix_row + col);
    return HAS_DELTA ? add_bf16x8(pv, ld_row(p.delta + t * p.delta_row + col)) : pv;
  };
  auto bank = [&](int i, int64_t col) -> uint4 {
    return ld_row(bank_row + (int64_t)i * p.blocks_slot + col);
  };

  // pass 1: partial sums
  float part[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) part[r] = 0.f;
  if constexpr (S > 0) {
    for (int64_t v = tid; v < nv; v += kGenericThreads) {
      const int64_t col = v * kVec;
      const uint4 rw = ld_weight(p.rms_w + col), qw = ld_weight(p.res_w + col);
      float q[kVec];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        q[2 * k] = bf_lo(vword(rw, k)) * bf_lo(vword(qw, k));
        q[2 * k + 1] = bf_hi(vword(rw, k)) * bf_hi(vword(qw, k));
      }
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const uint4 x = (i < S) ? bank(i < S ? i : 0, col) : current(col);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float a = bf_lo(vword(x, k)), b = bf_hi(vword(x, k));
          part[i] = fmaf(a, a, part[i]);
          part[i] = fmaf(b, b, part[i]);
          part[N + i] = fmaf(a, q[2 * k], part[N + i]);
          part[N + i] = fmaf(b, q[2 * k + 1], part[N + i]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) part[r] = warp_sum(part[r]);
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < NR; ++r) s_part[warp][r] = part[r];
    }
    __syncthreads();
    if (warp == 0) {
      float tot = 0.f;
      if (lane < NR) {
#pragma unroll
        for (int w = 0; w < kGenericWarps; ++w) tot += s_part[w][lane];
      }
      const float dtv = __shfl_sync(0xffffffffu, tot, (lane + N) & 31);
      float logit = __int_as_float(0xff800000u);  // -inf
      if (lane < N) logit = dtv / sqrtf(tot / (float)H + p.eps);
      const float m = warp_max(logit);
      const float e = (lane < N) ? expf(logit - m) : 0.f;
      const float z = warp_sum(e);
      if (lane < N) s_wt[lane] = e / z;
    }
    __syncthreads();
  } else {
    if (tid == 0) s_wt[0] = 1.f;
    __syncthreads();
  }

  auto mix = [&](int64_t col, uint4& c, float (&acc)[kVec]) {
    c = current(col);
#pragma unroll
    for (int k = 0; k < kVec; ++k) acc[k] = 0.f;
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float w = s_wt[i];
      const uint4 x = (i < S) ? bank(i < S ? i : 0, col) : c;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[2 * k] = fmaf(w, bf_lo(vword(x, k)), acc[2 * k]);
        acc[2 * k + 1] = fmaf(w, bf_hi(vword(x, k)), acc[2 * k + 1]);
      }
    }
  };

  // pass 2: output-norm sum of squares
  float ro = 1.f;
  if constexpr (HAS_ONORM) {
    float sq = 0.f;
    for (int64_t v = tid; v < nv; v += kGenericThreads) {
      uint4 c;
      float acc[kVec];
      mix(v * kVec, c, acc);
#pragma unroll
      for (int k = 0; k < kVec; ++k) sq = fmaf(acc[k], acc[k], sq);
    }
    sq = warp_sum(sq);
    if (lane == 0) s_sq[warp] = sq;
    __syncthreads();
    if (tid == 0) {
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < kGenericWarps; ++w) tot += s_sq[w];
      s_ro = 1.0f / sqrtf(tot / (float)H + p.out_eps);
    }
    __syncthreads();
    ro = s_ro;
  }

  // pass 3: output and write-backs
  for (int64_t v = tid; v < nv; v += kGenericThreads) {
    const int64_t col = v * kVec;
    uint4 c;
    float acc[kVec];
    mix(col, c, acc);
    if constexpr (HAS_ONORM) {
      const uint4 ow = ld_weight(p.onw + col);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[2 * k] = acc[2 * k] * ro * bf_lo(vword(ow, k));
        acc[2 * k + 1] = acc[2 * k + 1] * ro * bf_hi(vword(ow, k));
      }
    }
    st_row(p.out + t * p.out_row + col,
           make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                      pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
    if (HAS_DELTA) st_row(p.prefix + t * p.prefix_row + col, c);
    if (slot_write) st_row(bank_row + (int64_t)p.write_idx * p.blocks_slot + col, c);
  }
  grid_dep_launch_dependents();
}

}  // namespace attn_res_dev
