/*
 * attn_res.h -- C ABI of the GB300-native Kimi-K3 attention-residual
 * (AttnRes) mixture.
 *
 * The operation (implementation walkthrough of vllm-ascend PR #14840 "Add
 * Kimi K3 attention residual fusion"; key source excerpts of the prhub summary
 * of vllm PR #54261 "SM100 Kimi-K3 AttnRes defaults to native CUDA"): for each
 * token row t of width H = 7168,
 *
 *   c      = bf16_rn(prefix[t] + delta[t])      (c = prefix[t] if no delta)
 *   x_i    = blocks[t, i]  for i < num_blocks,  x_S = c        (S = num_blocks)
 *   q      = rms_w * res_w
 *   l_i    = <x_i, q> / sqrt(mean(x_i^2) + eps)
 *   w      = softmax(l_0 .. l_S)
 *   acc    = sum_i w_i x_i                      (raw rows, fp32)
 *   out[t] = bf16_rn(acc * out_norm_w / sqrt(mean(acc^2) + out_eps))
 *            or bf16_rn(acc) when out_norm_w == NULL
 *   prefix[t] = c                  when delta != NULL          (in place)
 *   blocks[t, block_write_idx] = c when block_write_idx >= 0   (in place)
 *
 * All reads of a token see the values from before the call, so a write-back
 * slot may also be one of the sources (block_write_idx < num_blocks).
 *
 * Element type: every tensor is bf16, passed as a pointer to its 16-bit
 * patterns (uint16_t).  Strides are in elements.  All tensor pointers are
 * DEVICE pointers of the current CUDA device; the caller owns every buffer.
 * The library allocates no memory, keeps no per-call state and is
 * re-entrant.
 */
#ifndef ATTN_RES_H_
#define ATTN_RES_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Hidden size the kernels are built for (the Kimi-K3 width named in the
 * dispatch gate of vllm PR #54261). */
#define ATTN_RES_HIDDEN 7168
/* Largest num_blocks (same gate: 0 <= num_blocks <= 8). */
#define ATTN_RES_MAX_BLOCKS 8

typedef uint16_t attn_res_bf16_t; /* bf16 bit pattern */

typedef enum {
  ATTN_RES_OK = 0,
  ATTN_RES_EINVAL = 1,  /* a size, index, stride, eps or required pointer is invalid */
  ATTN_RES_EALIGN = 2,  /* a pointer is not 16-byte aligned or a stride is not a multiple of 8 */
  ATTN_RES_EALIAS = 3,  /* a written region overlaps another argument's region */
  ATTN_RES_ECUDA = 4,   /* the CUDA runtime reported an error (query, attribute or launch) */
  ATTN_RES_EDEVICE = 5  /* the current device is not a compute capability 10.3 GPU */
} attn_res_status_t;

/* Launch options, in attn_res_layout_t.flags. */

/* Programmatic dependent launch: the kernel may start while the previous
 * kernel of the stream is still running.  It loads the bank rows and the
 * weights first, then waits for that kernel (griddepcontrol.wait) before
 * reading prefix and delta, and lets its own dependents launch once those
 * loads are issued (the stream kernel and its staged form: once it has run
 * out of tokens).  Contract: no grid that may still be running when this
 * call's grid starts may write the bank rows it reads or the weights.  That
 * is the preceding kernel of the stream, and also any earlier one that the
 * preceding kernel lets run on -- a kernel that releases its dependents
 * before its own grid-dependency wait.  The kernels here wait before they
 * release, so in a chain of these calls only the immediately preceding
 * call counts: between a call that writes a bank slot and a later PDL call
 * that reads it, put a kernel launched without PDL (or any fully
 * stream-ordered operation), or make the reading call without the flag.
 * Placement of the wait: PDL discipline in the key source excerpts of vllm
 * PR #54261. */
#define ATTN_RES_FLAG_PDL 0x1u

/* Hidden-sharded calls only (attn_res_tp_*; attn_res and attn_res_h reject
 * it): the single-exchange form, see attn_res_tp_sums below. */
#define ATTN_RES_FLAG_TP_GRAM 0x2u

/* Tuning overrides (0 = automatic).  Results do not depend on them beyond
 * fp32 summation order.
 *   KERNEL(k): ATTN_RES_KERNEL_SPLIT -- one cluster per token row, rows held
 *              in registers (latency path for few tokens);
 *              ATTN_RES_KERNEL_STREAM -- persistent clusters that stream many
 *              tokens through a TMA-filled shared-memory ring of bank rows,
 *              prefix and delta loaded into registers one token ahead;
 *              ATTN_RES_KERNEL_STAGED -- the stream kernel with prefix and
 *              delta also in the ring, as deep as shared memory allows;
 *              ATTN_RES_KERNEL_ROW -- one CTA per token row holding the whole
 *              row in registers, no cluster (up to 2 bank rows);
 *              ATTN_RES_KERNEL_ROW_SMEM -- the same with the rows in shared
 *              memory, brought in by bulk copies (1..8 bank rows).
 *   SPLIT(k):  CTAs (one thread-block cluster) a token row is split over;
 *              split kernel 4, 7, 8, 14 or 16; stream kernel see below; the
 *              row kernels 1.
 *   STAGES(n): ring depth of the stream kernel; CTAs per SM the staged
 *              form's ring is sized for.
 *   VPT(n):    16-byte vectors per thread and row (split kernel: 1; row
 *              kernels: 4 or 7).
 * Stream kernel shapes (split, vpt, stages): (7,1,2) (7,2,2) (7,2,3) (7,4,2)
 * (4,2,2) (4,2,3) (2,4,2) (14,2,2) (2,8,2).  Unset fields default to:
 * split 2 with no bank rows (4 if VPT 2 is given, 7 for VPT 1), else 7;
 * stages 2; VPT 8 with split 2 and no bank rows, 4 with split 2 and bank
 * rows, or with split 7 and 1..5 bank rows and an output norm or 3..6 bank
 * rows from 512 token rows, else 2 -- so (7,4,2) there, (2,8,2) with no
 * bank rows, and (7,2,2) otherwise.
 * Staged shapes (split, vpt, CTAs per SM): (4,4,5) (7,4,7) (4,4,4); the
 * ring holds as many stages of the S + 1 (+1 with delta) row slices as fit,
 * and a shape whose ring cannot hold two is ATTN_RES_EINVAL for that S.
 * Without overrides: (4,4,5) for 3 bank rows, (7,4,7) for 4, (4,4,4) for 5.
 * Automatic choice (shape overrides without KERNEL keep to the split and
 * stream kernels), measured per case on GB300:
 *   T < 80, or shared bank rows below 80: the split kernel;
 *   shared bank rows (B > 1) from 80 rows: the stream kernel;
 *   otherwise, with an output norm: no bank row, the row kernel; 1 bank row,
 *   the row kernel below 512 rows and the shared-memory row kernel from
 *   512; 2, the row kernel below 4096 rows and the shared-memory one from
 *   4096; 3..5, the shared-memory row kernel below 512 rows and the staged
 *   form from 512; 6, the shared-memory row kernel below 512 rows and the
 *   stream kernel from 512; 7..8, the stream kernel;
 *   without an output norm, below 512 rows: no bank row, the split kernel;
 *   1..2, the row kernel; 3, the staged form; 4..5, the shared-memory row
 *   kernel; 6..8, the stream kernel; from 512 rows: 0..1 bank rows, the row
 *   kernel, else the stream kernel.
 * (The exact table is attn_res_launch_shape's answer.) */
#define ATTN_RES_FLAG_SPLIT(k) (((uint32_t)(k) & 0xffu) << 8)
#define ATTN_RES_FLAG_KERNEL(k) (((uint32_t)(k) & 0xfu) << 16)
#define ATTN_RES_FLAG_STAGES(n) (((uint32_t)(n) & 0xfu) << 20)
#define ATTN_RES_FLAG_VPT(n) (((uint32_t)(n) & 0xfu) << 24)
#define ATTN_RES_KERNEL_SPLIT 1
#define ATTN_RES_KERNEL_STREAM 2
#define ATTN_RES_KERNEL_GENERIC 3 /* one CTA per row, any H (see attn_res_h) */
#define ATTN_RES_KERNEL_STAGED 4  /* stream kernel with prefix and delta staged in the ring */
#define ATTN_RES_KERNEL_ROW 5     /* one CTA per token row, the whole row */
#define ATTN_RES_KERNEL_ROW_SMEM 6 /* the same with the rows in shared memory */

/* Memory layout of the tensors, in elements.  A row is H contiguous
 * elements; columns H .. stride-1 are padding that is never read or
 * written. */
typedef struct {
  int64_t prefix_row;      /* between token rows of prefix (>= H) */
  int64_t delta_row;       /* between token rows of delta (>= H; ignored if delta == NULL) */
  int64_t blocks_token;    /* between token rows of the bank (>= (capacity-1)*blocks_slot + H
                              when the call touches more than one bank row) */
  int64_t blocks_slot;     /* between slots of one token (>= H) */
  int64_t out_row;         /* between token rows of out (>= H) */
  int32_t blocks_capacity; /* slots allocated per token (blocks.shape[1]); >= num_blocks */
  uint32_t flags;          /* ATTN_RES_FLAG_* */
  int32_t blocks_group;    /* B: token rows per bank row (0 or 1: one bank row per
                              token); see "Shared bank rows" below */
} attn_res_layout_t;

/* Shared bank rows (B = layout.blocks_group > 1).  The attn_res_kernel.cu
 * excerpt of vllm PR #54261 addresses the bank at row tb / B for token row
 * tb; the pages never say what B stands for.  Here: token row t reads bank
 * row t / B (integer division), so the bank holds ceil(T / B) token rows of
 * blocks_token elements.  Several rows then share one write-back slot; it
 * ends holding c of the last row of each group (the value sequential writes
 * in token order would leave), and only that row writes it.  Because the
 * other rows of the group would read a slot that is being written,
 * 0 <= block_write_idx < num_blocks is ATTN_RES_EINVAL when B > 1; a
 * negative blocks_group is ATTN_RES_EINVAL too.  With B > 1 the stream
 * kernel is built in one shape, (7,2,2); other stream overrides are
 * ATTN_RES_EINVAL. */

/*
 * attn_res -- enqueue the AttnRes mixture for T token rows on `stream`.
 *
 *   prefix          [T, H] at prefix_row.  Read; overwritten with c when
 *                   delta != NULL.
 *   delta           [T, H] at delta_row, or NULL.
 *   blocks          bank [T, capacity, H] at (blocks_token, blocks_slot)
 *                   ([ceil(T / B), capacity, H] with shared bank rows).
 *                   Slots 0 .. num_blocks-1 are read; slot block_write_idx
 *                   (if >= 0) is overwritten with c; nothing else is touched.
 *                   May be NULL only when num_blocks == 0 and
 *                   block_write_idx == -1.
 *   num_blocks      valid bank slots S, 0 <= S <= min(8, capacity).
 *   block_write_idx -1 (no write-back) or 0 <= idx < capacity.
 *   res_w, rms_w    [H] weights (the reference's proj / qk weight and norm
 *                   weight); q = rms_w * res_w.
 *   out_norm_w      [H] output RMSNorm weight, or NULL for no output norm.
 *   eps, out_eps    finite, >= 0.
 *   out             [T, H] at out_row.
 *   T               token rows, >= 0.  T == 0 checks the scalar arguments
 *                   and returns OK; pointers and strides are not examined.
 *   layout          strides, capacity and flags (see above).  Not NULL.
 *   stream          a cudaStream_t of the current device (NULL = legacy
 *                   default stream).
 *
 * Requirements: all pointers 16-byte aligned; all strides multiples of 8;
 * the address range [ptr, ptr + extent) of each written tensor (out always,
 * prefix when delta != NULL, blocks when block_write_idx >= 0) does not
 * overlap the range of any other argument.
 *
 * Returns ATTN_RES_OK once the work is enqueued (the call is asynchronous).
 * Any other status is returned before anything is launched, and nothing is
 * written.  Faults during execution surface from later CUDA calls on the
 * stream, as for any kernel.
 */
attn_res_status_t attn_res(attn_res_bf16_t* prefix, const attn_res_bf16_t* delta,
                           attn_res_bf16_t* blocks, int num_blocks,
                           int block_write_idx, const attn_res_bf16_t* res_w,
                           const attn_res_bf16_t* rms_w,
                           const attn_res_bf16_t* out_norm_w, float eps,
                           float out_eps, attn_res_bf16_t* out, int64_t T,
                           const attn_res_layout_t* layout, void* stream);

/*
 * attn_res_h -- the same operation for any hidden size H > 0 that is a
 * multiple of 8 (one 16-byte vector); every [H]- and row-sized argument above
 * is then H elements wide and strides must be >= H.  H == ATTN_RES_HIDDEN
 * behaves exactly like attn_res.  Other widths:
 *   - H at most 16384, with bank rows or an output norm: any-width forms of
 *     the fast kernels with ceil(H / 1024) CTAs per token row (one cluster)
 *     of 1024 columns each, the last CTA owning the remainder -- below 80
 *     token rows and up to H = 8192 the split kernel (one vector per
 *     thread), else the stream kernel (the per-CTA layout of the (7,2,2)
 *     shape); KERNEL(SPLIT) or KERNEL(STREAM) force one of them; shape
 *     overrides are ATTN_RES_EINVAL;
 *   - otherwise (wider rows, or neither bank rows nor an output norm) a
 *     general kernel (one CTA of 256 threads per token row, same fp32
 *     arithmetic, the rows read three times through L2), a functional
 *     path.  ATTN_RES_FLAG_KERNEL(ATTN_RES_KERNEL_GENERIC) forces it, also at
 *     H == ATTN_RES_HIDDEN.  Forcing a fast kernel where no form of it fits
 *     the width (or the row has no exchange) is ATTN_RES_EINVAL; the row
 *     kernels and the staged form are built for H == ATTN_RES_HIDDEN only
 *     (forced at another width: ATTN_RES_EINVAL).
 * Returns ATTN_RES_EINVAL for a bad H.  (No counterpart on the pages, whose
 * kernel is built for H = 7168 only.)
 */
attn_res_status_t attn_res_h(int64_t H, attn_res_bf16_t* prefix,
                             const attn_res_bf16_t* delta, attn_res_bf16_t* blocks,
                             int num_blocks, int block_write_idx,
                             const attn_res_bf16_t* res_w, const attn_res_bf16_t* rms_w,
                             const attn_res_bf16_t* out_norm_w, float eps, float out_eps,
                             attn_res_bf16_t* out, int64_t T,
                             const attn_res_layout_t* layout, void* stream);

/*
 * Hidden-sharded (tensor-parallel) mixture.  The Kimi-K3 deployments the
 * prhub summary of vllm PR #54261 evaluates (impact section: TP8, TEP8,
 * DEP16, ...) may hold a column shard of each row per rank.  The logits need
 * full-row sums and the output norm a full-row sum of squares, so the
 * operation above splits at those two points; the caller all-reduces (sums)
 * the small float buffers between the calls:
 *
 *   attn_res_tp_sums   -> all-reduce sums [T, 2N]   (N = num_blocks + 1)
 *   attn_res_tp_sq     -> all-reduce sq [T]         (output norm only)
 *   attn_res_tp_finish
 *
 * Each rank passes its own shard: every row-sized argument (prefix, delta,
 * blocks rows, res_w, rms_w, out_norm_w, out) is the Hs columns that rank
 * owns, with the strides and layout rules of attn_res_h for width Hs (a
 * multiple of 8); H is the full hidden size (the sum of the shard widths),
 * used in mean(x^2) and mean(acc^2).  With one rank (Hs == H) the three calls
 * compute the same result as attn_res_h.  Float buffers are fp32 device
 * memory owned by the caller, 4-byte aligned; sums has sums_row >=
 * attn_res_tp_sums_width(num_blocks, gram) floats between token rows:
 * entries 0..N-1 are sum(x_i^2), N..2N-1 are <x_i, q> over the shard
 * (x_S = c).  layout->flags accepts ATTN_RES_FLAG_PDL, ATTN_RES_FLAG_TP_GRAM,
 * ATTN_RES_FLAG_KERNEL and ATTN_RES_FLAG_STAGES.  Two kernel forms, the same
 * results up to fp32 summation order:
 *   ring (ATTN_RES_KERNEL_STREAM) -- persistent CTAs (as many as fit on the
 *     device, at most T) each streaming every G-th token row's rows through
 *     a shared-memory ring filled by bulk copies (TMA), ATTN_RES_FLAG_STAGES
 *     2..4 deep (default 2); the Gram sums on warp-level tensor-core tiles;
 *   one CTA of 32..256 threads per token row (ATTN_RES_KERNEL_GENERIC).
 * Automatic: the ring from 1024 token rows when it fits in 220 KB of shared
 * memory (2 stages of num_blocks + 1 (+1 with delta) rows of Hs columns, plus
 * 4*Hs bytes and the warps' tiles for the Gram sums), else one CTA per row.
 * A forced ring that does not fit, another KERNEL value, or STAGES with
 * ATTN_RES_KERNEL_GENERIC is ATTN_RES_EINVAL; with the automatic form
 * STAGES applies only when the ring runs.  Errors as for attn_res (nothing
 * is launched unless ATTN_RES_OK is returned); a written float buffer that
 * overlaps any other argument is ATTN_RES_EALIAS.
 *
 * Single exchange (ATTN_RES_FLAG_TP_GRAM set on attn_res_tp_sums and
 * attn_res_tp_finish): attn_res_tp_sums also writes g_ij = <x_i, x_j> over
 * the shard for i < j (entries 2N.., row-major over i), and
 * attn_res_tp_finish takes sum(acc^2) = sum_i w_i^2 ss_i + 2 sum_{i<j} w_i
 * w_j g_ij from the reduced entries: one all-reduce and no attn_res_tp_sq
 * call (which rejects the flag).  Exact in real arithmetic; in fp32 the
 * output norm loses relative accuracy where the weighted rows cancel
 * (|acc| << sum_i w_i |x_i|), so the default is the two-exchange form.
 * The ring form computes the Gram products on warp-level tensor-core tiles
 * (mma.sync m16n8k16, bf16 in, fp32 accumulate; q split exactly into two
 * bf16 rows): the one dense contraction in this library, confined to this
 * opt-in form -- the mixture itself, like the pages' kernels, uses no tensor
 * cores (a bandwidth-bound mix of a few rows per token).
 */

/* Floats per token row of `sums`: 2N, plus N(N-1)/2 with gram != 0
 * (N = num_blocks + 1); -1 for num_blocks outside 0..8. */
int attn_res_tp_sums_width(int num_blocks, int gram);

/* Per-shard sums; reads prefix, delta, blocks[t, 0..num_blocks), res_w,
 * rms_w; writes sums[t, 0..attn_res_tp_sums_width(num_blocks, gram)). */
attn_res_status_t attn_res_tp_sums(int64_t Hs, const attn_res_bf16_t* prefix,
                                   const attn_res_bf16_t* delta, const attn_res_bf16_t* blocks,
                                   int num_blocks, const attn_res_bf16_t* res_w,
                                   const attn_res_bf16_t* rms_w, float* sums, int64_t sums_row,
                                   int64_t T, const attn_res_layout_t* layout, void* stream);

/* Output-norm partial: softmax from the reduced sums, acc over the shard,
 * sq[t] = sum(acc^2) over the shard.  Reads prefix, delta, blocks, sums;
 * writes sq[0..T).  sq must not be NULL. */
attn_res_status_t attn_res_tp_sq(int64_t Hs, int64_t H, const attn_res_bf16_t* prefix,
                                 const attn_res_bf16_t* delta, const attn_res_bf16_t* blocks,
                                 int num_blocks, float eps, const float* sums, int64_t sums_row,
                                 float* sq, int64_t T, const attn_res_layout_t* layout,
                                 void* stream);

/* Output and write-backs of the shard: softmax from the reduced sums, acc,
 * out (normalised with the reduced sq, or with the Gram entries under
 * ATTN_RES_FLAG_TP_GRAM, when out_norm_w != NULL; sq may be NULL otherwise),
 * prefix[t] = c when delta != NULL, blocks[t, block_write_idx] = c when
 * block_write_idx >= 0. */
attn_res_status_t attn_res_tp_finish(int64_t Hs, int64_t H, attn_res_bf16_t* prefix,
                                     const attn_res_bf16_t* delta, attn_res_bf16_t* blocks,
                                     int num_blocks, int block_write_idx,
                                     const attn_res_bf16_t* out_norm_w, float eps, float out_eps,
                                     const float* sums, int64_t sums_row, const float* sq,
                                     attn_res_bf16_t* out, int64_t T,
                                     const attn_res_layout_t* layout, void* stream);

/* Static text for a status code. */
const char* attn_res_status_string(attn_res_status_t status);

/* ATTN_RES_HIDDEN, for callers that load the library dynamically. */
int attn_res_hidden_size(void);

/* ATTN_RES_MAX_BLOCKS. */
int attn_res_max_blocks(void);

/*
 * attn_res_launch_shape -- the launch attn_res would make for T rows with
 * num_blocks sources, a delta row or not, output norm on/off and the given
 * flags: the kernel (ATTN_RES_KERNEL_*), CTAs per token row (`split`), ring
 * depth (`stages`: the stream kernel's STAGES; the staged form's depth,
 * which follows from the rows of a stage; 0 for the other kernels), threads
 * per CTA, CTAs in the grid (0 for the persistent stream kernel and its
 * staged form, whose grid is as many clusters as fit on the device, at most
 * T) and the thread-block cluster size (1 when the CTAs of a row never
 * exchange sums -- no bank rows and no output norm -- and for the row and
 * general kernels, which hold a row in one CTA).  Any output pointer may be
 * NULL.  Pure host computation, no CUDA call.  Returns ATTN_RES_EINVAL for
 * T < 0, num_blocks outside 0..8 or an unsupported override.
 */
attn_res_status_t attn_res_launch_shape(int64_t T, int num_blocks, int has_delta,
                                        int has_out_norm, uint32_t flags,
                                        int* kernel, int* split, int* stages,
                                        int* threads_per_cta, int64_t* ctas,
                                        int* cluster);

/*
 * attn_res_device_status -- error bits the kernels recorded on the current
 * device since the last clear (0 = none).  Bit 0: a wait for a shared-memory
 * stage of row data timed out; bit 1: a wait for the partial sums of another
 * CTA of the cluster timed out.  The kernel then finished without waiting
 * further and that call's outputs are not valid.  With `clear` != 0 the word is reset.  Synchronous
 * (cudaMemcpy); a diagnostic, not for the hot path.
 */
attn_res_status_t attn_res_device_status(unsigned int* bits, int clear);

/*
 * attn_res_selftest_wait_timeout -- exercise the kernels' time-out path on
 * the current device: one warp waits, with the same bounded-wait code the
 * mixture kernels use, on an mbarrier that nothing ever completes; after
 * about `limit_us` microseconds (1 .. 1 000 000) the wait gives up and bit 0
 * of the device status word is set.  Synchronous: returns after the kernel
 * finished, with the status word (not cleared) in *bits.  A diagnostic for
 * tests; it does not touch any caller buffer.
 */
attn_res_status_t attn_res_selftest_wait_timeout(unsigned int limit_us, unsigned int* bits);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_RES_H_ */
