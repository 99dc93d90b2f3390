// attn_res_tp.cuh -- the mixture with the hidden dimension sharded across
// ranks (tensor parallel).
//
// Each rank holds a contiguous column shard of width Hs of every row (prefix,
// delta, bank rows, weights, output).  The logits need full-row sums and the
// output norm a full-row sum of squares of the mix, so the mixture splits at
// those points, with an all-reduce (sum) over the ranks between the kernels:
//
//   tp_sums    per token: ss_i = sum x_i^2 and dt_i = <x_i, q> over the shard,
//              written to sums[t, 0..2N)                    -> all-reduce(sums)
//   tp_sq      (output norm only) softmax from the reduced sums, acc = mix of
//              the shard, sq[t] = sum acc^2 over the shard  -> all-reduce(sq)
//   tp_finish  softmax from the reduced sums, mix again, output (normalised
//              with the reduced sq) and the write-backs of c
//
// Single-exchange form (GRAM): tp_sums also writes the off-diagonal Gram
// entries g_ij = <x_i, x_j> (i < j) after the 2N sums, and tp_finish takes
//   sum_h acc_h^2 = sum_i w_i^2 ss_i + 2 sum_{i<j} w_i w_j g_ij
// from the reduced entries: one all-reduce and two passes over the rows
// instead of two and three.  The identity is exact; in fp32 it loses relative
// accuracy only where the weighted rows cancel (|acc| much smaller than
// sum_i w_i |x_i|).
//
// H in the logits and the norm is the full width, passed in as 1/H.  The
// per-element arithmetic is that of the other kernels.  One CTA per token
// row, 32..256 threads (enough to give each thread one 16-byte vector of the
// shard where it fits).  The mix is recomputed in tp_finish rather than kept
// between calls, so the only data between calls are the floats per token the
// caller reduces.
#pragma once

#include "attn_res_common.cuh"

namespace attn_res_dev {

constexpr int kTpMaxThreads = 256;
constexpr int kTpMaxWarps = kTpMaxThreads / 32;

struct TpArgs {
  int64_t Hs;        // shard width (multiple of 8)
  float inv_h;       // 1 / full hidden size
  float* sums;       // [T, sums_row] (written by tp_sums, read by tp_sq / tp_finish)
  int64_t sums_row;  // floats between token rows of sums
  float* sq;         // [T] (written by tp_sq, read by tp_finish); null when unused
};

template <int S>
struct TpCfg {
  static constexpr int N = S + 1;
  static constexpr int NR = 2 * N;            // ss_i, dt_i
  static constexpr int NG = N * (N - 1) / 2;  // g_ij, i < j
};

// Sum NR per-thread values over the CTA.  The CTA totals end in
// scratch[0][r], readable by any thread after the call.
template <int NR>
__device__ __forceinline__ void cta_sum(const float (&v)[NR], float (*scratch)[NR]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const float s = warp_sum(v[r]);
    if (lane == 0) scratch[warp][r] = s;
  }
  __syncthreads();
  for (int r = threadIdx.x; r < NR; r += blockDim.x) {
    float s = scratch[0][r];
    for (int w = 1; w < nw; ++w) s += scratch[w][r];
    scratch[0][r] = s;  // only thread r touches column r here
  }
  __syncthreads();
}

template <bool HAS_DELTA>
__device__ __forceinline__ uint4 tp_current(const Params& p, int64_t t, int64_t col) {
  const uint4 pv = ld_row(p.prefix + t * p.prefix_row + col);
  return HAS_DELTA ? add_bf16x8(pv, ld_row(p.delta + t * p.delta_row + col)) : pv;
}

__device__ __forceinline__ uint4 tp_bank(const Params& p, int64_t t, int i, int64_t col) {
  return ld_row(p.blocks + t * p.blocks_token + (int64_t)i * p.blocks_slot + col);
}

// x_i = bank row i (i < S) or the current row c (i == S), widened to fp32.
template <int S, bool HAS_DELTA>
__device__ __forceinline__ void tp_sources(const Params& p, int64_t t, int64_t col,
                                           float (&x)[S + 1][kVec]) {
#pragma unroll
  for (int i = 0; i <= S; ++i) {
    const uint4 v = (i < S) ? tp_bank(p, t, i < S ? i : 0, col) : tp_current<HAS_DELTA>(p, t, col);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[i][2 * k] = bf_lo(vword(v, k));
      x[i][2 * k + 1] = bf_hi(vword(v, k));
    }
  }
}

template <int S, bool HAS_DELTA, bool GRAM>
__global__ void __launch_bounds__(kTpMaxThreads) attn_res_tp_sums_kernel(const Params p, const TpArgs a) {
  using C = TpCfg<S>;
  constexpr int N = C::N, NR = C::NR, NT = NR + (GRAM ? C::NG : 0);
  __shared__ float scratch[kTpMaxWarps][NT];
  const int64_t t = blockIdx.x;
  const int64_t nv = a.Hs / kVec;
  grid_dep_wait();
  float part[NT];
#pragma unroll
  for (int r = 0; r < NT; ++r) part[r] = 0.f;
  for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) {
    const int64_t col = v * kVec;
    const uint4 rw = ld_weight(p.rms_w + col), qw = ld_weight(p.res_w + col);
    float q[kVec];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      q[2 * k] = bf_lo(vword(rw, k)) * bf_lo(vword(qw, k));
      q[2 * k + 1] = bf_hi(vword(rw, k)) * bf_hi(vword(qw, k));
    }
    float x[N][kVec];
    tp_sources<S, HAS_DELTA>(p, t, col, x);
#pragma unroll
    for (int i = 0; i < N; ++i) {
#pragma unroll
      for (int k = 0; k < kVec; ++k) {
        part[i] = fmaf(x[i][k], x[i][k], part[i]);
        part[N + i] = fmaf(x[i][k], q[k], part[N + i]);
      }
    }
    if constexpr (GRAM) {
      int g = NR;
#pragma unroll
      for (int i = 0; i < N; ++i) {
#pragma unroll
        for (int j = i + 1; j < N; ++j, ++g) {
#pragma unroll
          for (int k = 0; k < kVec; ++k) part[g] = fmaf(x[i][k], x[j][k], part[g]);
        }
      }
    }
  }
  cta_sum<NT>(part, scratch);
  for (int r = threadIdx.x; r < NT; r += blockDim.x) a.sums[t * a.sums_row + r] = scratch[0][r];
  grid_dep_launch_dependents();
}

// Softmax weights of token t from the reduced sums (every thread).
template <int S>
__device__ __forceinline__ void tp_weights(const TpArgs& a, float eps, int64_t t, float (&w)[S + 1]) {
  constexpr int N = S + 1;
  if constexpr (S == 0) {
    w[0] = 1.f;  // a single source takes all the weight
    return;
  }
  const float* s = a.sums + t * a.sums_row;
  float logit[N];
  float m = __int_as_float(0xff800000u);
#pragma unroll
  for (int i = 0; i < N; ++i) {
    logit[i] = s[N + i] / sqrtf(s[i] * a.inv_h + eps);
    m = fmaxf(m, logit[i]);
  }
  float z = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    w[i] = expf(logit[i] - m);
    z += w[i];
  }
#pragma unroll
  for (int i = 0; i < N; ++i) w[i] = w[i] / z;
}

template <int S, bool HAS_DELTA>
__device__ __forceinline__ void tp_mix(const Params& p, int64_t t, int64_t col, const float (&w)[S + 1],
                                       uint4& c, float (&acc)[kVec]) {
  constexpr int N = S + 1;
  c = tp_current<HAS_DELTA>(p, t, col);
#pragma unroll
  for (int k = 0; k < kVec; ++k) acc[k] = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const uint4 x = (i < S) ? tp_bank(p, t, i < S ? i : 0, col) : c;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc[2 * k] = fmaf(w[i], bf_lo(vword(x, k)), acc[2 * k]);
      acc[2 * k + 1] = fmaf(w[i], bf_hi(vword(x, k)), acc[2 * k + 1]);
    }
  }
}

template <int S, bool HAS_DELTA>
__global__ void __launch_bounds__(kTpMaxThreads) attn_res_tp_sq_kernel(const Params p, const TpArgs a) {
  __shared__ float scratch[kTpMaxWarps][1];
  const int64_t t = blockIdx.x;
  const int64_t nv = a.Hs / kVec;
  grid_dep_wait();
  float w[S + 1];
  tp_weights<S>(a, p.eps, t, w);
  float sq[1] = {0.f};
  for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) {
    uint4 c;
    float acc[kVec];
    tp_mix<S, HAS_DELTA>(p, t, v * kVec, w, c, acc);
#pragma unroll
    for (int k = 0; k < kVec; ++k) sq[0] = fmaf(acc[k], acc[k], sq[0]);
  }
  cta_sum<1>(sq, scratch);
  if (threadIdx.x == 0) a.sq[t] = scratch[0][0];
  grid_dep_launch_dependents();
}

// sum_h acc_h^2 from the reduced sums and Gram entries, clamped at 0 (the
// fp32 sum of the terms can come out slightly negative where rows cancel).
template <int S>
__device__ __forceinline__ float tp_gram_sq(const TpArgs& a, int64_t t, const float (&w)[S + 1]) {
  constexpr int N = S + 1;
  const float* s = a.sums + t * a.sums_row;
  float diag = 0.f, off = 0.f;
  int g = 2 * N;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    diag = fmaf(w[i] * w[i], s[i], diag);
#pragma unroll
    for (int j = i + 1; j < N; ++j, ++g) off = fmaf(w[i] * w[j], s[g], off);
  }
  return fmaxf(fmaf(2.f, off, diag), 0.f);
}

template <int S, bool HAS_DELTA, bool HAS_ONORM, bool GRAM>
__global__ void __launch_bounds__(kTpMaxThreads) attn_res_tp_finish_kernel(const Params p, const TpArgs a) {
  const int64_t t = blockIdx.x;
  const int64_t nv = a.Hs / kVec;
  grid_dep_wait();
  float w[S + 1];
  tp_weights<S>(a, p.eps, t, w);
  float ro = 1.f;
  if constexpr (HAS_ONORM) {
    const float sq = GRAM ? tp_gram_sq<S>(a, t, w) : a.sq[t];
    ro = 1.0f / sqrtf(sq * a.inv_h + p.out_eps);
  }
  // each thread writes only the vectors it alone reads: no barrier needed
  for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) {
    const int64_t col = v * kVec;
    uint4 c;
    float acc[kVec];
    tp_mix<S, HAS_DELTA>(p, t, col, w, c, acc);
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
    if (p.write_idx >= 0)
      st_row(p.blocks + t * p.blocks_token + (int64_t)p.write_idx * p.blocks_slot + col, c);
  }
  grid_dep_launch_dependents();
}

}  // namespace attn_res_dev
