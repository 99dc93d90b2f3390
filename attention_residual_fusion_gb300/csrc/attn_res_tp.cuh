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
// per-element arithmetic is that of the other kernels.  Two forms of each
// phase: one CTA per token row, 32..256 threads (enough to give each thread
// one 16-byte vector of the shard where it fits), and a persistent ring form
// (below) for many token rows.  The mix is recomputed in tp_finish rather
// than kept between calls, so the only data between calls are the floats per
// token the caller reduces.
#pragma once

#include "attn_res_common.cuh"

namespace attn_res_dev {

// Warp-level tensor-core tiles (the Gram sums of the ring form).

// Four 8x8 b16 matrices from shared memory: lane l gives the address of row
// l % 8 of matrix l / 8 (16 bytes each); r[j] is this lane's part of matrix j.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
// d += A (16x16 bf16, row-major) x B (16x8 bf16, column-major), fp32.
__device__ __forceinline__ void mma_bf16_16x8x16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                 uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

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

// Sum NR per-thread values over the CTA with one barrier: the warps' totals
// go to scratch, and thread r (r < NR, then r + blockDim.x, ...) adds column
// r over the warps in warp order and hands it to store(r, total).  scratch
// must not be written again before every thread has passed a later barrier
// (double-buffer it across tokens).
template <int NR, class Store>
__device__ __forceinline__ void cta_sum_store(const float (&v)[NR], float (*scratch)[NR], Store store) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  warp_groups<NR, 0>(v, scratch, warp, lane);
  __syncthreads();
  for (int r = threadIdx.x; r < NR; r += blockDim.x) {
    float s = scratch[0][r];
    for (int w = 1; w < nw; ++w) s += scratch[w][r];
    store(r, s);
  }
}

template <bool HAS_DELTA>
__device__ __forceinline__ uint4 tp_current(const Params& p, int64_t t, int64_t col) {
  const uint4 pv = ld_row(p.prefix + t * p.prefix_row + col);
  return HAS_DELTA ? add_bf16x8(pv, ld_row(p.delta + t * p.delta_row + col)) : pv;
}

__device__ __forceinline__ uint4 tp_bank(const Params& p, int64_t t, int i, int64_t col) {
  return ld_row(bank_of(p, t) + (int64_t)i * p.blocks_slot + col);
}

// q = rms_w * res_w over one 16-byte vector of columns (exact in fp32).
__device__ __forceinline__ void tp_query(const Params& p, int64_t col, f32x2 (&q)[4]) {
  const uint4 rw = ld_weight(p.rms_w + col), qw = ld_weight(p.res_w + col);
#pragma unroll
  for (int k = 0; k < 4; ++k) q[k] = f2_mul(bf2_widen(vword(rw, k)), bf2_widen(vword(qw, k)));
}

// The sources' vectors: bank row i (i < S) from src(i), the current row c
// (i == S).
template <int S, class Src>
__device__ __forceinline__ void tp_gather(Src src, const uint4& c, uint4 (&x)[S + 1]) {
#pragma unroll
  for (int i = 0; i <= S; ++i) x[i] = (i < S) ? src(i < S ? i : 0) : c;
}

// One vector's contribution to a token's per-thread sums.  The sources are
// widened one 32-bit word (a column pair) at a time, so only one word of
// each is live in fp32; every accumulator still takes its terms in column
// order.  Without Gram entries the 2N sums accumulate as fp32 pairs in ss /
// dt; with them every accumulator is a scalar in part[] (packed pairs for
// the Gram entries too would need about 230 registers and halve the CTAs an
// SM holds, which costs more than the halved FMA count saves).
template <int S, bool GRAM, int NT>
__device__ __forceinline__ void tp_accumulate(const uint4 (&x)[S + 1], const f32x2 (&q)[4],
                                              f32x2 (&ss)[GRAM ? 1 : S + 1],
                                              f32x2 (&dt)[GRAM ? 1 : S + 1], float (&part)[NT]) {
  constexpr int N = S + 1, NR = 2 * N;
  if constexpr (!GRAM) {
    // few accumulators: every source widened up front schedules best
    f32x2 xw[N][4];
#pragma unroll
    for (int i = 0; i < N; ++i) {
#pragma unroll
      for (int k = 0; k < 4; ++k) xw[i][k] = bf2_widen(vword(x[i], k));
    }
#pragma unroll
    for (int i = 0; i < N; ++i) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        ss[i] = f2_fma(xw[i][k], xw[i][k], ss[i]);
        dt[i] = f2_fma(xw[i][k], q[k], dt[i]);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f32x2 xk[N];
#pragma unroll
      for (int i = 0; i < N; ++i) xk[i] = bf2_widen(vword(x[i], k));
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const float lo = f2_lo(xk[i]), hi = f2_hi(xk[i]);
        part[i] = fmaf(hi, hi, fmaf(lo, lo, part[i]));
        part[N + i] = fmaf(hi, f2_hi(q[k]), fmaf(lo, f2_lo(q[k]), part[N + i]));
      }
#pragma unroll
      for (int i = 0; i < N; ++i) {
#pragma unroll
        for (int j = 0; j < N; ++j) {
          if (j > i) {
            const int g = NR + i * N - i * (i + 1) / 2 + (j - i - 1);  // row-major over i < j
            part[g] = fmaf(f2_lo(xk[i]), f2_lo(xk[j]), part[g]);
            part[g] = fmaf(f2_hi(xk[i]), f2_hi(xk[j]), part[g]);
          }
        }
      }
    }
  }
}

// Zeroed accumulators of tp_accumulate.
template <int S, bool GRAM, int NT>
__device__ __forceinline__ void tp_clear(f32x2 (&ss)[GRAM ? 1 : S + 1], f32x2 (&dt)[GRAM ? 1 : S + 1],
                                         float (&part)[NT]) {
#pragma unroll
  for (int r = 0; r < NT; ++r) part[r] = 0.f;
#pragma unroll
  for (int i = 0; i < (GRAM ? 1 : S + 1); ++i) ss[i] = dt[i] = 0ull;  // +0.0f pairs
}

// The pair accumulators folded into part[0 .. 2N).
template <int S, bool GRAM, int NT>
__device__ __forceinline__ void tp_fold(const f32x2 (&ss)[GRAM ? 1 : S + 1],
                                        const f32x2 (&dt)[GRAM ? 1 : S + 1], float (&part)[NT]) {
  if constexpr (!GRAM) {
#pragma unroll
    for (int i = 0; i <= S; ++i) {
      part[i] = f2_lo(ss[i]) + f2_hi(ss[i]);
      part[S + 1 + i] = f2_lo(dt[i]) + f2_hi(dt[i]);
    }
  }
}

template <int S, bool HAS_DELTA, bool GRAM>
__global__ void __launch_bounds__(GRAM ? kTpGramThreads : kTpMaxThreads)
    attn_res_tp_sums_kernel(const Params p, const TpArgs a) {
  using C = TpCfg<S>;
  constexpr int NT = C::NR + (GRAM ? C::NG : 0);
  __shared__ float scratch[kTpMaxWarps][NT];
  const int64_t t = blockIdx.x;
  const int64_t nv = a.Hs / kVec;
  grid_dep_wait();
  float part[NT];
  f32x2 ss[GRAM ? 1 : C::N], dt[GRAM ? 1 : C::N];
  tp_clear<S, GRAM>(ss, dt, part);
  for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) {
    const int64_t col = v * kVec;
    f32x2 q[4];
    tp_query(p, col, q);
    uint4 x[C::N];
    tp_gather<S>([&](int i) { return tp_bank(p, t, i, col); }, tp_current<HAS_DELTA>(p, t, col), x);
    tp_accumulate<S, GRAM>(x, q, ss, dt, part);
  }
  tp_fold<S, GRAM>(ss, dt, part);
  cta_sum<NT>(part, scratch);
  for (int r = threadIdx.x; r < NT; r += blockDim.x) a.sums[t * a.sums_row + r] = scratch[0][r];
  grid_dep_launch_dependents();
}

// Softmax weights from a token's reduced sums s[0 .. 2N): lane i < N of every
// warp takes logit i, the warp reduces, and the weights are broadcast to all
// lanes (every thread of the warp must call).  Same instructions as the
// unsharded kernels' softmax, so every warp gets bit-identical weights.
template <int S>
__device__ __forceinline__ void tp_weights(const float* s, float inv_h, float eps, float (&w)[S + 1]) {
  constexpr int N = S + 1;
  if constexpr (S == 0) {
    w[0] = 1.f;  // a single source takes all the weight
    return;
  }
  const int lane = threadIdx.x & 31;
  float logit = __int_as_float(0xff800000u);  // -inf
  if (lane < N) logit = s[N + lane] * rsqrtf(fmaf(s[lane], inv_h, eps));
  const float m = warp_max(logit);
  const float e = (lane < N) ? expf(logit - m) : 0.f;
  const float z = warp_sum(e);
  const float wl = __fdividef(e, z);
#pragma unroll
  for (int i = 0; i < N; ++i) w[i] = __shfl_sync(0xffffffffu, wl, i);
}

// acc = sum_i w_i x_i over one vector of columns: src(i) gives bank row i's
// vector, c the current row's.
template <int S, class Src>
__device__ __forceinline__ void tp_mix(Src src, const uint4& c, const float (&w)[S + 1],
                                       f32x2 (&acc)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = 0ull;
#pragma unroll
  for (int i = 0; i <= S; ++i) {
    const uint4 x = (i < S) ? src(i < S ? i : 0) : c;
    const f32x2 w2 = f2_make(w[i], w[i]);
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = f2_fma(w2, bf2_widen(vword(x, k)), acc[k]);
  }
}

// sum_h acc_h^2 from the reduced sums and Gram entries s[2N ..], clamped at 0
// (the fp32 sum of the terms can come out slightly negative where rows
// cancel).
template <int S>
__device__ __forceinline__ float tp_gram_sq(const float* s, const float (&w)[S + 1]) {
  constexpr int N = S + 1;
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

// The output vector: acc (normalised by ro and scaled by the output-norm
// weights when HAS_ONORM), rounded to bf16.
template <bool HAS_ONORM>
__device__ __forceinline__ uint4 tp_output(const Params& p, int64_t col, f32x2 (&acc)[4], float ro) {
  if constexpr (HAS_ONORM) {
    const uint4 ow = ld_weight(p.onw + col);
    const f32x2 ro2 = f2_make(ro, ro);
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = f2_mul(f2_mul(acc[k], ro2), bf2_widen(vword(ow, k)));
  }
  return make_uint4(pack_bf16x2(f2_lo(acc[0]), f2_hi(acc[0])), pack_bf16x2(f2_lo(acc[1]), f2_hi(acc[1])),
                    pack_bf16x2(f2_lo(acc[2]), f2_hi(acc[2])), pack_bf16x2(f2_lo(acc[3]), f2_hi(acc[3])));
}

template <int S, bool HAS_DELTA>
__global__ void __launch_bounds__(kTpMaxThreads) attn_res_tp_sq_kernel(const Params p, const TpArgs a) {
  __shared__ float scratch[kTpMaxWarps][1];
  const int64_t t = blockIdx.x;
  const int64_t nv = a.Hs / kVec;
  grid_dep_wait();
  float w[S + 1];
  tp_weights<S>(a.sums + t * a.sums_row, a.inv_h, p.eps, w);
  f32x2 sq2 = 0ull;
  for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) {
    const int64_t col = v * kVec;
    f32x2 acc[4];
    tp_mix<S>([&](int i) { return tp_bank(p, t, i, col); }, tp_current<HAS_DELTA>(p, t, col), w, acc);
#pragma unroll
    for (int k = 0; k < 4; ++k) sq2 = f2_fma(acc[k], acc[k], sq2);
  }
  const float sq[1] = {f2_lo(sq2) + f2_hi(sq2)};
  cta_sum<1>(sq, scratch);
  if (threadIdx.x == 0) a.sq[t] = scratch[0][0];
  grid_dep_launch_dependents();
}

template <int S, bool HAS_DELTA, bool HAS_ONORM, bool GRAM>
__global__ void __launch_bounds__(kTpMaxThreads) attn_res_tp_finish_kernel(const Params p, const TpArgs a) {
  const int64_t t = blockIdx.x;
  const int64_t nv = a.Hs / kVec;
  grid_dep_wait();
  const float* s = a.sums + t * a.sums_row;
  float w[S + 1];
  tp_weights<S>(s, a.inv_h, p.eps, w);
  float ro = 1.f;
  if constexpr (HAS_ONORM) {
    const float sq = GRAM ? tp_gram_sq<S>(s, w) : a.sq[t];
    ro = rsqrtf(fmaf(sq, a.inv_h, p.out_eps));
  }
  // each thread writes only the vectors it alone reads: no barrier needed
  const bool slot_write = writes_slot(p, t);
  for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) {
    const int64_t col = v * kVec;
    const uint4 c = tp_current<HAS_DELTA>(p, t, col);
    f32x2 acc[4];
    tp_mix<S>([&](int i) { return tp_bank(p, t, i, col); }, c, w, acc);
    st_row(p.out + t * p.out_row + col, tp_output<HAS_ONORM>(p, col, acc, ro));
    if (HAS_DELTA) st_row(p.prefix + t * p.prefix_row + col, c);
    if (slot_write)
      st_row(const_cast<uint16_t*>(bank_of(p, t)) + (int64_t)p.write_idx * p.blocks_slot + col, c);
  }
  grid_dep_launch_dependents();
}

// ---- persistent form: a token's rows staged through a shared-memory ring -------------
//
// A CTA of the kernels above holds one token's rows only while it lives: its
// launch, its one load round trip and its reduction tail overlap nothing of
// its own, which leaves the narrow rows of a shard (1.8 KB at H_s = 896)
// short of the bytes in flight the memory system needs.  The ring form keeps
// G = CTAs per SM x SMs CTAs resident; CTA b takes the token rows b, b + G,
// b + 2G, ...  The rows of a token (bank rows 0..S-1, prefix, delta) arrive by
// one-dimensional bulk copies (TMA) in one stage of a `stages`-deep ring in
// shared memory: the lanes of warp 0 issue one row each, `stages` tokens
// ahead, completing on the stage's mbarrier.  Every thread reads its vectors
// from the stage; after the CTA barrier that ends a token (inside the
// reduction, or an explicit one in the finish phase) warp 0 refills the
// stage.  The reduced sums a token needs (and sq) are loaded one token ahead
// into a double-buffered array in shared memory, and the softmax weights are
// taken from them while the token's rows are still arriving.  Waits are
// bounded as in the stream kernel.  The arithmetic per element is that of the
// kernels above, except that the Gram sums (45 dot products of 9 rows per
// token at S = 8: a small dense contraction) run on mma.sync tiles: per step
// of 16 columns one 16 x 16 tile X holds the stage's rows (plus the query
// split into two exact bf16 rows), read once with ldmatrix, and X X^T takes
// two m16n8k16 mma whose B operands are A's own registers; the warps'
// 16 x 16 tiles are summed in warp order.  (tcgen05
// wants tiles of at least 64 rows in its core-matrix layout; a token has 9
// rows, stored row-major.)
//
// PHASE 0: sums; 1: sum of squares of the mix; 2: finish.

constexpr int kTpRingMaxStages = 4;

template <int S, bool HAS_DELTA, int PHASE, bool HAS_ONORM, bool GRAM>
struct TpRingCfg {
  static constexpr int N = S + 1, NR = 2 * N, NG = N * (N - 1) / 2;
  static constexpr int ROWS = N + (HAS_DELTA ? 1 : 0);  // rows per token in a stage
  static constexpr int NT = PHASE == 0 ? NR + (GRAM ? NG : 0) : 1;  // values a token reduces
  // floats of the reduced input a token reads: the 2N sums, the Gram
  // entries (finish, GRAM) or sq (finish, output norm, two exchanges) at 2N
  static constexpr bool SQ = PHASE == 2 && HAS_ONORM && !GRAM;
  static constexpr int NS = PHASE == 0 ? 0 : (PHASE == 2 && GRAM) ? NR + NG : NR + (SQ ? 1 : 0);
  static constexpr int THREADS_MAX = kTpMaxThreads;
  static constexpr int MIN_BLOCKS = 2;  // CTAs of THREADS_MAX threads per SM (the register cap)
  static constexpr int NWARPS_MAX = THREADS_MAX / 32;
  static_assert(NS <= 64 && ROWS <= 32, "two floats per thread of a 32-thread CTA, one lane per row");
  static_assert(N + 2 <= 16, "sources and the two query rows fit one 16-row tile");
};

// Bytes of dynamic shared memory of a ring kernel of `threads` threads:
// `stages` stages of ROWS rows at a pitch of row bytes + 16 (so the rows of
// an 8x8 ldmatrix tile fall in distinct banks), then, for the Gram sums
// (mma), the q_hi and q_lo rows, 16 zero bytes and two 16 x 16 fp32 tiles
// per warp.
__host__ __device__ constexpr int64_t tp_ring_smem_bytes(int rows, int64_t Hs, int stages, bool mma,
                                                         int threads) {
  return (int64_t)stages * rows * (Hs * 2 + 16) +
         (mma ? 2 * Hs * 2 + 16 + (int64_t)2 * (threads / 32) * 16 * 16 * 4 : 0);
}

// (The register cap comes from MIN_BLOCKS: without a minimum the register
// heuristic settles below what the phases keep live, and spills.)
template <int S, bool HAS_DELTA, int PHASE, bool HAS_ONORM, bool GRAM>
__global__ void __launch_bounds__(TpRingCfg<S, HAS_DELTA, PHASE, HAS_ONORM, GRAM>::THREADS_MAX,
                                  TpRingCfg<S, HAS_DELTA, PHASE, HAS_ONORM, GRAM>::MIN_BLOCKS)
    attn_res_tp_ring_kernel(const Params p, const TpArgs a, const int stages) {
  using C = TpRingCfg<S, HAS_DELTA, PHASE, HAS_ONORM, GRAM>;
  constexpr int N = C::N, NR = C::NR, ROWS = C::ROWS, NT = C::NT, NS = C::NS;
  // the Gram sums on tensor-core tiles; the plain 2N sums per thread
  constexpr bool MMA = PHASE == 0 && GRAM;
  // [stages][ROWS][pitch]; MMA: q_hi, q_lo, 16 zero bytes, tiles [2][warps][16][16]
  extern __shared__ __align__(128) uint4 ring[];
  __shared__ __align__(8) unsigned long long full_bar[kTpRingMaxStages];
  __shared__ float scratch[MMA ? 1 : 2][MMA ? 1 : kTpMaxWarps][MMA ? 1 : NT];
  __shared__ float sv[2][NS > 0 ? NS : 1];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x, nw = nthr >> 5;
  const int64_t nv = a.Hs / kVec;
  const uint32_t row_bytes = (uint32_t)nv * 16u;
  const uint32_t pitch = row_bytes + 16u;  // bytes between the rows of a stage
  const int64_t pv = nv + 1;              // the same in 16-byte vectors
  const uint32_t stage_bytes = (uint32_t)ROWS * pitch;
  // T < 2^31: token counts in 32 bits (no 64-bit division)
  const int64_t G = gridDim.x;
  const uint32_t T32 = (uint32_t)p.tokens;
  const int64_t ntok = T32 > blockIdx.x ? (int64_t)((T32 - blockIdx.x + gridDim.x - 1) / gridDim.x) : 0;
  const uint32_t ring_addr = smem_addr(ring);
  // MMA: the query split into two bf16 rows (q = q_hi + q_lo exactly) and a
  // zero row, after the ring
  uint4* const qhi = ring + (int64_t)stages * ROWS * pv;
  uint4* const qlo = qhi + nv;
  const uint32_t qhi_addr = smem_addr(qhi), qlo_addr = smem_addr(qlo);
  const uint32_t zero_addr = smem_addr(qlo + nv);
  // MMA: each warp's 16 x 16 tile of <row_m, row_n> (double-buffered)
  float(*const tiles)[16][16] = reinterpret_cast<float(*)[16][16]>(qlo + nv + 1);
  auto tile = [&](int b, int w) { return tiles[b * nw + w]; };

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(smem_addr(&full_bar[s]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  grid_dep_wait();

  // warp 0: the rows of local token j into stage s (lane 0 arms the stage's
  // barrier with the byte count, lane i < ROWS copies row i)
  auto issue = [&](int64_t j, int s) {
    const int64_t t = blockIdx.x + j * G;
    const uint32_t bar = smem_addr(&full_bar[s]);
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)ROWS * row_bytes);
    __syncwarp();
    if (lane < ROWS) {
      const uint16_t* src = lane < S    ? bank_of(p, t) + (int64_t)lane * p.blocks_slot
                            : lane == S ? p.prefix + t * p.prefix_row
                                        : p.delta + t * p.delta_row;
      bulk_load(ring_addr + (uint32_t)s * stage_bytes + (uint32_t)lane * pitch, src, row_bytes, bar);
    }
  };
  // floats r = tid and tid + nthr (< NS) of the reduced input of local token
  // j, into next[0..1]
  auto load_reduced = [&](int64_t j, float (&next)[2]) {
    const int64_t t = blockIdx.x + j * G;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int r = tid + k * nthr;
      if (r < NS) next[k] = (C::SQ && r == NR) ? a.sq[t] : a.sums[t * a.sums_row + r];
    }
  };
  auto store_reduced = [&](float* dst, const float (&next)[2]) {
#pragma unroll
    for (int k = 0; k < 2; ++k)
      if (tid + k * nthr < NS) dst[tid + k * nthr] = next[k];
  };

  // thread 0 tracks the stages whose last issued copies it has not yet seen
  // complete, and that issue's parity.  Staggered start: only the first
  // token's rows now; the other stages once they have landed (in the loop),
  // so the first token's work overlaps the next token's loads instead of
  // every CTA's whole ring arriving at once at the end of one burst.
  uint32_t pending = 0, pending_parity = 0;
  if (warp == 0 && ntok > 0) {
    issue(0, 0);
    pending = 1u;
  }
  if (NS > 0) {
    float first[2] = {0.f, 0.f};
    if (ntok > 0) load_reduced(0, first);
    store_reduced(sv[0], first);
  }
  // MMA: lane l addresses row l % 8 of 8x8 matrix l / 8 of the 16 x 16 tile
  // X of a step (rows: the sources, q_hi, q_lo, zeros; stored
  // [row][column]): matrices 0..3 = (rows 0-7 | 8-15) x (columns 0-7 | 8-15)
  // in the order of the A operand's registers.  The products wanted are
  // X X^T, and the B operand of X^T (16 x 8, column-major) for rows 0-7 of X
  // is A's registers 0 and 2, for rows 8-15 registers 1 and 3: one ldmatrix
  // per step serves both operands.
  int am = 0, ak = 0;
  if constexpr (MMA) {
    const int mj = lane >> 3, mr = lane & 7;
    am = (mj & 1) * 8 + mr;
    ak = (mj >> 1) * 8;
    for (int64_t v = tid; v < nv; v += nthr) {
      f32x2 q[4];
      tp_query(p, v * kVec, q);
      uint32_t h[4], l[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        h[k] = pack_bf16x2(f2_lo(q[k]), f2_hi(q[k]));
        // the remainder: exact for finite q (at most 8 significant bits); 0
        // where q is not finite, so that q_hi alone carries it
        float rl = f2_lo(q[k]) - bf_lo(h[k]), rh = f2_hi(q[k]) - bf_hi(h[k]);
        rl = rl == rl ? rl : 0.f;
        rh = rh == rh ? rh : 0.f;
        l[k] = pack_bf16x2(rl, rh);
      }
      qhi[v] = make_uint4(h[0], h[1], h[2], h[3]);
      qlo[v] = make_uint4(l[0], l[1], l[2], l[3]);
    }
    if (tid == 0) qlo[nv] = make_uint4(0, 0, 0, 0);
  }
  if (NS > 0 || MMA) __syncthreads();

  // plain sums with at most one vector per thread (the shard fits the CTA):
  // the thread's query vector once, not per token
  const bool one_vec = nv <= nthr;
  f32x2 q_own[4] = {};
  if constexpr (PHASE == 0 && !GRAM) {
    if (one_vec && tid < nv) tp_query(p, tid * kVec, q_own);
  }

  bool failed = false;
  int s = 0;            // stage of local token j: j % stages
  uint32_t parity = 0;  // its phase parity: (j / stages) & 1
  for (int64_t j = 0; j < ntok; ++j) {
    const int64_t t = blockIdx.x + j * G;
    const int b = (int)(j & 1);
    float next[2] = {0.f, 0.f};  // reduced input of the next token, in flight meanwhile
    if (NS > 0 && j + 1 < ntok) load_reduced(j + 1, next);
    // the weights (and the output norm's scale) need only the reduced sums:
    // take them while the token's rows are still arriving
    float w[N];
    float ro = 1.f;
    if constexpr (PHASE != 0) {
      tp_weights<S>(sv[b], a.inv_h, p.eps, w);
      if constexpr (PHASE == 2 && HAS_ONORM)
        ro = rsqrtf(fmaf(GRAM ? tp_gram_sq<S>(sv[b], w) : sv[b][NR], a.inv_h, p.out_eps));
    }
    const bool was_failed = failed;
    wait_or_flag(smem_addr(&full_bar[s]), parity, failed, p.err, kErrStageTimeout);
    if (tid == 0 && !was_failed && !failed) pending &= ~(1u << s);
    // staggered start: token j + 1 into its first (unused) stage
    if (warp == 0 && j + 1 < stages && j + 1 < ntok && !__any_sync(0xffffffffu, failed)) {
      issue(j + 1, (int)(j + 1));
      pending |= 1u << (int)(j + 1);
    }
    uint4* const st = ring + (int64_t)s * ROWS * pv;
    auto src = [&](int i, int64_t v) { return st[i * pv + v]; };
    auto cur = [&](int64_t v) {
      return HAS_DELTA ? add_bf16x8(st[S * pv + v], st[(S + 1) * pv + v]) : st[S * pv + v];
    };

    if constexpr (PHASE == 0 && !GRAM) {
      float part[NT];
      f32x2 ss[N], dt[N];
      tp_clear<S, false>(ss, dt, part);
      for (int64_t v = tid; v < nv; v += nthr) {
        f32x2 q[4];
        if (one_vec) {
#pragma unroll
          for (int k = 0; k < 4; ++k) q[k] = q_own[k];
        } else {
          tp_query(p, v * kVec, q);
        }
        uint4 x[N];
        tp_gather<S>([&](int i) { return src(i, v); }, cur(v), x);
        tp_accumulate<S, false>(x, q, ss, dt, part);
      }
      tp_fold<S, false>(ss, dt, part);
      cta_sum_store<NT>(part, scratch[b], [&](int r, float v) { a.sums[t * a.sums_row + r] = v; });
    } else if constexpr (MMA) {
      const int k16 = (int)((nv + 1) >> 1);  // 16-column steps (the last may be half)
      // c into the stage's prefix row, so that rows 0..S are the sources --
      // each warp for the two vectors of each 16-column step it multiplies
      // below (steps warp, warp + nw, ...), so a warp barrier suffices
      if constexpr (HAS_DELTA) {
        const int nsteps = warp < k16 ? (k16 - 1 - warp) / nw + 1 : 0;
        for (int e = lane; e < 2 * nsteps; e += 32) {
          const int64_t v = 2 * (int64_t)(warp + (e >> 1) * nw) + (e & 1);
          if (v < nv) st[S * pv + v] = cur(v);
        }
        __syncwarp();
      }
      const uint32_t sb = ring_addr + (uint32_t)s * stage_bytes;
      const uint32_t arow = am < N ? sb + (uint32_t)am * pitch : am == N ? qhi_addr : qlo_addr;
      const bool avalid = am < N + 2;
      // two accumulator sets (even and odd steps of this warp) halve the
      // chain of dependent mma; the tiles of the next two steps are read
      // while the current two multiply (steps past the row read the zero
      // bytes and add nothing)
      float d[2][2][4] = {};
      auto load = [&](int ks, uint32_t(&av)[4]) {
        const uint32_t ca = (uint32_t)ks * 16u + ak;
        ldsm_x4(avalid && ks < k16 && ca < a.Hs ? arow + ca * 2u : zero_addr, av);
      };
      auto mul = [&](const uint32_t(&av)[4], float(&e)[2][4]) {
        mma_bf16_16x8x16(e[0], av, av[0], av[2]);
        mma_bf16_16x8x16(e[1], av, av[1], av[3]);
      };
      uint32_t x0[4], x1[4];
      load(warp, x0);
      load(warp + nw, x1);
      for (int ks = warp; ks < k16; ks += 2 * nw) {
        uint32_t y0[4], y1[4];
        load(ks + 2 * nw, y0);
        load(ks + 3 * nw, y1);
        mul(x0, d[0]);
        mul(x1, d[1]);
#pragma unroll
        for (int e = 0; e < 4; ++e) x0[e] = y0[e], x1[e] = y1[e];
      }
      float d0[4], d1[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        d0[e] = d[0][0][e] + d[1][0][e];
        d1[e] = d[0][1][e] + d[1][1][e];
      }
      {
        const int r = lane >> 2, c2 = (lane & 3) * 2;
        float(*tw)[16] = tile(b, warp);
        *reinterpret_cast<float2*>(&tw[r][c2]) = make_float2(d0[0], d0[1]);
        *reinterpret_cast<float2*>(&tw[r + 8][c2]) = make_float2(d0[2], d0[3]);
        *reinterpret_cast<float2*>(&tw[r][8 + c2]) = make_float2(d1[0], d1[1]);
        *reinterpret_cast<float2*>(&tw[r + 8][8 + c2]) = make_float2(d1[2], d1[3]);
      }
      __syncthreads();  // every read of the stage is done; the tiles are complete
      // value r: ss_i = <x_i, x_i> (r < N), dt_i = <x_i, q_hi> + <x_i, q_lo>
      // (r < 2N), else g_ij = <x_i, x_j> (row-major over i < j); the warps'
      // tiles summed in warp order
      for (int r = tid; r < NT; r += nthr) {
        int vi = r, vj = r, vk = -1;
        if (r >= NR) {
          int g = r - NR;
          vi = 0;
          while (g >= N - 1 - vi) g -= N - 1 - vi++;
          vj = vi + 1 + g;
        } else if (r >= N) {
          vi = r - N;
          vj = N;
          vk = N + 1;
        }
        float v1 = 0.f;
        for (int w = 0; w < nw; ++w) v1 += tile(b, w)[vi][vj];
        if (vk >= 0) {
          float v2 = 0.f;
          for (int w = 0; w < nw; ++w) v2 += tile(b, w)[vi][vk];
          v1 += v2;
        }
        a.sums[t * a.sums_row + r] = v1;
      }
    } else {
      if constexpr (PHASE == 1) {
        f32x2 sq2 = 0ull;
        for (int64_t v = tid; v < nv; v += nthr) {
          f32x2 acc[4];
          tp_mix<S>([&](int i) { return src(i, v); }, cur(v), w, acc);
#pragma unroll
          for (int k = 0; k < 4; ++k) sq2 = f2_fma(acc[k], acc[k], sq2);
        }
        store_reduced(sv[b ^ 1], next);
        const float sq[1] = {f2_lo(sq2) + f2_hi(sq2)};
        cta_sum_store<1>(sq, scratch[b], [&](int, float v) { a.sq[t] = v; });
      } else {
        const bool slot_write = writes_slot(p, t);
        uint16_t* const slot = slot_write ? const_cast<uint16_t*>(bank_of(p, t)) +
                                                (int64_t)p.write_idx * p.blocks_slot
                                          : nullptr;
        for (int64_t v = tid; v < nv; v += nthr) {
          const int64_t col = v * kVec;
          const uint4 c = cur(v);
          f32x2 acc[4];
          tp_mix<S>([&](int i) { return src(i, v); }, c, w, acc);
          st_row(p.out + t * p.out_row + col, tp_output<HAS_ONORM>(p, col, acc, ro));
          if (HAS_DELTA) st_row(p.prefix + t * p.prefix_row + col, c);
          if (slot_write) st_row(slot + col, c);
        }
        store_reduced(sv[b ^ 1], next);
        __syncthreads();  // every read of the stage (and of sv[b]) is done
      }
    }

    // refill stage s with the token `stages` ahead: every thread is past its
    // last access to the stage (the barrier above); the issuing lanes order
    // those generic-proxy accesses before their copies with a proxy fence
    if (warp == 0 && j + stages < ntok) {
      if (!__any_sync(0xffffffffu, failed)) {
        fence_proxy_async_smem();
        issue(j + stages, s);
        if (tid == 0) {
          pending |= 1u << s;
          pending_parity = (pending_parity & ~(1u << s)) | ((parity ^ 1u) << s);
        }
      }
    }
    if (++s == stages) {
      s = 0;
      parity ^= 1u;
    }
  }

  grid_dep_launch_dependents();

  // After a time-out, do not leave with copies still landing in shared memory.
  if (tid == 0 && failed) {
    for (int s = 0; s < stages; ++s)
      if (pending & (1u << s))
        (void)mbar_wait_bounded(smem_addr(&full_bar[s]), (pending_parity >> s) & 1u);
  }
}

}  // namespace attn_res_dev
