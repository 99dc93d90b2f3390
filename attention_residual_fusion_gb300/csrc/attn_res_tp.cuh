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
// The Gram form of tp_sums keeps ~130 values live per thread: at most 128
// threads per CTA, so the register budget is not capped below that.
constexpr int kTpGramThreads = 128;

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

// Warp totals of values [B, B + P) of v (zero beyond NR) into scratch[warp]:
// one reduce-scatter butterfly, after which lane l holds the total of value
// l >> (5 - log2 P).
template <int NR, int B, int P>
__device__ __forceinline__ void warp_totals(const float (&v)[NR], float (*scratch)[NR], int warp,
                                            int lane) {
  float a[P];
#pragma unroll
  for (int r = 0; r < P; ++r) a[r] = (B + r < NR) ? v[B + r < NR ? B + r : 0] : 0.f;
  const float tot = reduce_scatter<P>(a, lane);
  constexpr int SH = 5 - log2_exact(P);
  const int idx = lane >> SH;
  if ((lane & ((1 << SH) - 1)) == 0 && B + idx < NR) scratch[warp][B + idx] = tot;
}

// Warp totals of all NR values, in butterflies of at most 16 values (a wider
// one keeps more values live at once than the registers hold).
template <int NR, int B>
__device__ __forceinline__ void warp_groups(const float (&v)[NR], float (*scratch)[NR], int warp,
                                            int lane) {
  if constexpr (B < NR) {
    constexpr int P = (NR - B) >= 16 ? 16 : pow2_at_least(NR - B);
    warp_totals<NR, B, P>(v, scratch, warp, lane);
    warp_groups<NR, B + P>(v, scratch, warp, lane);
  }
}

// Sum NR per-thread values over the CTA.  The CTA totals end in
// scratch[0][r], readable by any thread after the call.
template <int NR>
__device__ __forceinline__ void cta_sum(const float (&v)[NR], float (*scratch)[NR]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  warp_groups<NR, 0>(v, scratch, warp, lane);
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
  return ld_row(bank_of(p, t) + (int64_t)i * p.blocks_slot + col);
}

// x_i = bank row i (i < S) or the current row c (i == S), widened to fp32
// pairs.
template <int S, bool HAS_DELTA>
__device__ __forceinline__ void tp_sources(const Params& p, int64_t t, int64_t col,
                                           f32x2 (&x)[S + 1][4]) {
#pragma unroll
  for (int i = 0; i <= S; ++i) {
    const uint4 v = (i < S) ? tp_bank(p, t, i < S ? i : 0, col) : tp_current<HAS_DELTA>(p, t, col);
#pragma unroll
    for (int k = 0; k < 4; ++k) x[i][k] = bf2_widen(vword(v, k));
  }
}

template <int S, bool HAS_DELTA, bool GRAM>
__global__ void __launch_bounds__(GRAM ? kTpGramThreads : kTpMaxThreads)
    attn_res_tp_sums_kernel(const Params p, const TpArgs a) {
  using C = TpCfg<S>;
  constexpr int N = C::N, NR = C::NR, NT = NR + (GRAM ? C::NG : 0);
  __shared__ float scratch[kTpMaxWarps][NT];
  const int64_t t = blockIdx.x;
  const int64_t nv = a.Hs / kVec;
  grid_dep_wait();
  // Without Gram entries the 2N sums accumulate as fp32 pairs; with them every
  // accumulator is a scalar, which keeps the register count (and so the
  // number of resident CTAs) within reach of the plain form.
  float part[NT];
#pragma unroll
  for (int r = 0; r < NT; ++r) part[r] = 0.f;
  f32x2 ss[GRAM ? 1 : N], dt[GRAM ? 1 : N];
#pragma unroll
  for (int i = 0; i < (GRAM ? 1 : N); ++i) ss[i] = dt[i] = 0ull;  // +0.0f pairs
  for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) {
    const int64_t col = v * kVec;
    const uint4 rw = ld_weight(p.rms_w + col), qw = ld_weight(p.res_w + col);
    f32x2 q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) q[k] = f2_mul(bf2_widen(vword(rw, k)), bf2_widen(vword(qw, k)));
    f32x2 x[N][4];
    tp_sources<S, HAS_DELTA>(p, t, col, x);
    if constexpr (!GRAM) {
#pragma unroll
      for (int i = 0; i < N; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ss[i] = f2_fma(x[i][k], x[i][k], ss[i]);
          dt[i] = f2_fma(x[i][k], q[k], dt[i]);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < N; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float lo = f2_lo(x[i][k]), hi = f2_hi(x[i][k]);
          part[i] = fmaf(hi, hi, fmaf(lo, lo, part[i]));
          part[N + i] = fmaf(hi, f2_hi(q[k]), fmaf(lo, f2_lo(q[k]), part[N + i]));
        }
      }
#pragma unroll
      for (int i = 0; i < N; ++i) {
#pragma unroll
        for (int j = 0; j < N; ++j) {
          if (j > i) {
            const int g = NR + i * N - i * (i + 1) / 2 + (j - i - 1);  // row-major over i < j
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              part[g] = fmaf(f2_lo(x[i][k]), f2_lo(x[j][k]), part[g]);
              part[g] = fmaf(f2_hi(x[i][k]), f2_hi(x[j][k]), part[g]);
            }
          }
        }
      }
    }
  }
  if constexpr (!GRAM) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      part[i] = f2_lo(ss[i]) + f2_hi(ss[i]);
      part[N + i] = f2_lo(dt[i]) + f2_hi(dt[i]);
    }
  }
  cta_sum<NT>(part, scratch);
  for (int r = threadIdx.x; r < NT; r += blockDim.x) a.sums[t * a.sums_row + r] = scratch[0][r];
  grid_dep_launch_dependents();
}

// Softmax weights of token t from the reduced sums: lane i < N of every warp
// takes logit i, the warp reduces, and the weights are broadcast to all lanes
// (every thread of the warp must call).  Same instructions as the unsharded
// kernels' softmax, so every warp gets bit-identical weights.
template <int S>
__device__ __forceinline__ void tp_weights(const TpArgs& a, float eps, int64_t t, float (&w)[S + 1]) {
  constexpr int N = S + 1;
  if constexpr (S == 0) {
    w[0] = 1.f;  // a single source takes all the weight
    return;
  }
  const int lane = threadIdx.x & 31;
  const float* s = a.sums + t * a.sums_row;
  float logit = __int_as_float(0xff800000u);  // -inf
  if (lane < N) logit = s[N + lane] * rsqrtf(fmaf(s[lane], a.inv_h, eps));
  const float m = warp_max(logit);
  const float e = (lane < N) ? expf(logit - m) : 0.f;
  const float z = warp_sum(e);
  const float wl = __fdividef(e, z);
#pragma unroll
  for (int i = 0; i < N; ++i) w[i] = __shfl_sync(0xffffffffu, wl, i);
}

template <int S, bool HAS_DELTA>
__device__ __forceinline__ void tp_mix(const Params& p, int64_t t, int64_t col, const float (&w)[S + 1],
                                       uint4& c, f32x2 (&acc)[4]) {
  constexpr int N = S + 1;
  c = tp_current<HAS_DELTA>(p, t, col);
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = 0ull;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const uint4 x = (i < S) ? tp_bank(p, t, i < S ? i : 0, col) : c;
    const f32x2 w2 = f2_make(w[i], w[i]);
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = f2_fma(w2, bf2_widen(vword(x, k)), acc[k]);
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
  f32x2 sq2 = 0ull;
  for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) {
    uint4 c;
    f32x2 acc[4];
    tp_mix<S, HAS_DELTA>(p, t, v * kVec, w, c, acc);
#pragma unroll
    for (int k = 0; k < 4; ++k) sq2 = f2_fma(acc[k], acc[k], sq2);
  }
  const float sq[1] = {f2_lo(sq2) + f2_hi(sq2)};
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
    ro = rsqrtf(fmaf(sq, a.inv_h, p.out_eps));
  }
  // each thread writes only the vectors it alone reads: no barrier needed
  const f32x2 ro2 = f2_make(ro, ro);
  const bool slot_write = writes_slot(p, t);
  for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) {
    const int64_t col = v * kVec;
    uint4 c;
    f32x2 acc[4];
    tp_mix<S, HAS_DELTA>(p, t, col, w, c, acc);
    if constexpr (HAS_ONORM) {
      const uint4 ow = ld_weight(p.onw + col);
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] = f2_mul(f2_mul(acc[k], ro2), bf2_widen(vword(ow, k)));
    }
    st_row(p.out + t * p.out_row + col,
           make_uint4(pack_bf16x2(f2_lo(acc[0]), f2_hi(acc[0])), pack_bf16x2(f2_lo(acc[1]), f2_hi(acc[1])),
                      pack_bf16x2(f2_lo(acc[2]), f2_hi(acc[2])), pack_bf16x2(f2_lo(acc[3]), f2_hi(acc[3]))));
    if (HAS_DELTA) st_row(p.prefix + t * p.prefix_row + col, c);
    if (slot_write)
      st_row(const_cast<uint16_t*>(bank_of(p, t)) + (int64_t)p.write_idx * p.blocks_slot + col, c);
  }
  grid_dep_launch_dependents();
}

}  // namespace attn_res_dev
