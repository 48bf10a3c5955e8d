/*
 * verify_splitkv.h -- C ABI of the GB300 (sm_103a) split-KV verify attention.
 *
 * The operation (sglang "verify_splitkv.py" page: module docstring,
 * "_verify_prefix_stage1", "_verify_combine_stage2", "verify_splitkv_fwd"):
 * EAGLE speculative target-verify at topk = 1.  Sequence b owns l_ext draft
 * query rows q[qo_indptr[b] + i] (i < l_ext) and a prefix of
 * P_b = kv_indptr[b+1] - kv_indptr[b] tokens whose K/V rows live in a token
 * pool, addressed through kv_indices[kv_indptr[b] + j].  Query head h reads
 * KV head h / (h_q / h_kv).  Every draft row attends, under one softmax, over
 *   - all P_b prefix keys: score sm_scale * k_scale * <q, K_pool[loc]>,
 *     value v_scale * V_pool[loc];
 *   - the drafts t <= i of its own sequence: score sm_scale * <q, k_ext[t]>,
 *     value v_ext[t] (no k_scale / v_scale).
 * The library computes this with split-KV (flash-decode) partial softmaxes
 * over the prefix, merged by log-sum-exp with the causal draft block, and
 * writes o[qo_indptr[b] + i, h, :] in bf16.  An empty prefix (P_b = 0) yields
 * causal attention over the drafts alone.
 *
 * Threading and streams: every entry point may be called from any host
 * thread.  verify_splitkv_fwd enqueues one kernel on the given stream (two
 * for the small and mid-size shapes served by a prefix stream and a combine
 * kernel; vsk_launches_per_call tells which) and returns without
 * synchronising and without reading device memory.
 *
 * Memory: all tensor pointers are DEVICE pointers owned by the caller.  The
 * library never frees or retains them past the call.
 */
#ifndef VERIFY_SPLITKV_H
#define VERIFY_SPLITKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types of a vsk_tensor. */
enum {
  VSK_DTYPE_BF16 = 0,     /* bfloat16                                   */
  VSK_DTYPE_FP8E4M3 = 1,  /* float8 e4m3 "fn" (no infinities)           */
  VSK_DTYPE_I32 = 2,      /* int32                                      */
  VSK_DTYPE_I64 = 3,      /* int64                                      */
  VSK_DTYPE_U8 = 4        /* uint8 (also used for bool masks)           */
};

/* A strided view of device memory.  Strides and shape are in ELEMENTS.  For
 * 3-d tensors the last dimension must be contiguous (stride[2] == 1); 1-d
 * tensors must be contiguous.  Unused trailing entries are ignored. */
typedef struct vsk_tensor {
  const void* data;  /* device pointer (may be NULL only when the tensor is empty) */
  int32_t dtype;     /* one of VSK_DTYPE_*                                          */
  int32_t ndim;      /* 1 or 3                                                      */
  int64_t shape[3];
  int64_t stride[3];
} vsk_tensor;

/* Gate: returns 1 when verify_splitkv_fwd can serve this problem exactly,
 * 0 otherwise (the caller then falls back to its prefill/extend kernel).
 * Mirrors "can_handle" on the "verify_splitkv.py" page and adds this build's
 * own limits.  It inspects shapes, dtypes, strides, pointer alignment and the
 * scalar flags only: it never reads tensor VALUES.
 *
 *   q_extend   [B*l_ext, h_q, D]    bf16
 *   k_extend   [B*l_ext, h_kv, D]   bf16   (draft keys)
 *   v_extend   [B*l_ext, h_kv, Dv]  bf16   (draft values)
 *   k_buffer   [pool, h_kv, D]      bf16 or fp8 e4m3 (prefix key pool)
 *   v_buffer   [pool, h_kv, Dv]     same dtype as k_buffer
 *   qo_indptr  [B+1] int32, kv_indptr [B+1] int32, kv_indices [n] int32|int64
 *   is_causal  must be nonzero; max_len_extend (= l_ext) must be >= 1 and
 *              q_extend must hold exactly B * max_len_extend rows.
 *   sliding_window_size > 0, has_sinks != 0, logit_cap > 0 and
 *   xai_temperature_len > 0 are features this kernel does not implement:
 *   any of them makes the gate return 0.
 * Build limits: D and Dv in {64, 128, 256} (D != Dv is served by the
 * one-launch kernel); (h_q/h_kv) * l_ext <= 128 (<= 64 when D or Dv is 256);
 * pool rows 16-byte aligned (data pointer and the byte strides of both
 * leading dimensions); q/k_extend/v_extend 4-byte aligned with even strides.
 * On 0, vsk_last_error() names the first failed check. */
int vsk_can_handle(const vsk_tensor* q_extend, const vsk_tensor* k_extend,
                   const vsk_tensor* v_extend, const vsk_tensor* k_buffer,
                   const vsk_tensor* v_buffer, const vsk_tensor* qo_indptr,
                   const vsk_tensor* kv_indptr, const vsk_tensor* kv_indices,
                   int is_causal, int64_t max_len_extend,
                   int64_t sliding_window_size, int has_sinks, float logit_cap,
                   int64_t xai_temperature_len);

/* Split-KV verify attention ("verify_splitkv_fwd" on the "verify_splitkv.py"
 * page, same tensor roles).  Returns 1 after enqueueing the work on `stream`
 * (a cudaStream_t; NULL is the legacy default stream), or 0 having enqueued
 * NOTHING: the gate failed, o_extend is not a bf16 [B*l_ext, h_q, Dv] tensor
 * with a contiguous last dimension and even strides, the workspace is too
 * small, or a CUDA call failed.  vsk_last_error() says which.
 *
 *   o_extend    output, written only at rows [0, B*l_ext) and all h_q heads.
 *   k_scale, v_scale  dequantisation multipliers of the prefix pool (1.0 for
 *               a bf16 pool); they do not apply to k_extend / v_extend.
 *   sm_scale    softmax scale; a value <= 0 or NaN selects 1/sqrt(D).
 *   workspace   device scratch of workspace_bytes bytes, 256-byte aligned,
 *               zero-filled before its first use (cudaMemset or
 *               vsk_workspace_init) and then reused unchanged.  The call's
 *               counters (tickets) sit at the END of the buffer: the last
 *               64 KiB, which every call leaves at zero, or for very large
 *               batches (more than 16,384 tickets) a larger region, whose
 *               part beyond those 64 KiB the call clears on `stream` before
 *               its kernel (one cudaMemsetAsync).  So one buffer serves calls
 *               of any shapes that fit it.  The needed size is at most
 *               vsk_workspace_size(max_bs, ...) for any B <= max_bs on the
 *               same device.
 *               workspace == NULL selects a library-owned per-device buffer
 *               that grows on demand; growth allocates and synchronises the
 *               device, so make the first such call outside graph capture.
 *               Calls whose kernels may overlap on the GPU (different
 *               streams) must each have their own workspace.
 * Device-side checks: kv_indices values outside [0, pool) and inconsistent
 * indptr entries are never dereferenced; they set a bit in the workspace
 * error word (see vsk_read_error_flags) and the affected rows are computed
 * without those keys. */
int verify_splitkv_fwd(const vsk_tensor* q_extend, const vsk_tensor* k_extend,
                       const vsk_tensor* v_extend, const vsk_tensor* o_extend,
                       const vsk_tensor* k_buffer, const vsk_tensor* v_buffer,
                       const vsk_tensor* qo_indptr, const vsk_tensor* kv_indptr,
                       const vsk_tensor* kv_indices, int is_causal,
                       int64_t max_len_extend, float k_scale, float v_scale,
                       float sm_scale, void* workspace, size_t workspace_bytes,
                       void* stream);

/* Tree verify (speculative topk > 1): verify_splitkv_fwd with the draft
 * block under a custom mask instead of the causal rule (the case the
 * "verify_splitkv.py" page leaves to its fallback).  The mask layout is the
 * target-verify one of the "aiter_backend.py" page: for sequence b an
 * l_ext x (P_b + l_ext) uint8 matrix, row-major from custom_mask[mask_indptr[b]]
 * (row i = draft query i; columns = the P_b prefix keys, then the l_ext draft
 * keys; nonzero = visible).  Only the draft columns are read: every prefix
 * key stays visible (skip_prefix_custom_mask = True, the verify default).
 * A row with no visible key at all (empty prefix, no visible draft) gets 0.
 *   custom_mask  [n] uint8 (bool bytes accepted), device memory
 *   mask_indptr  [B+1] int32 or int64, device memory
 * Everything else, the return value and the workspace rules are those of
 * verify_splitkv_fwd (is_causal is implied).  mask_indptr entries whose rows
 * would fall outside custom_mask are not dereferenced: that sequence's
 * drafts fall back to the causal rule and error bit 16 is set. */
int verify_splitkv_tree_fwd(const vsk_tensor* q_extend, const vsk_tensor* k_extend,
                            const vsk_tensor* v_extend, const vsk_tensor* o_extend,
                            const vsk_tensor* k_buffer, const vsk_tensor* v_buffer,
                            const vsk_tensor* qo_indptr, const vsk_tensor* kv_indptr,
                            const vsk_tensor* kv_indices, const vsk_tensor* custom_mask,
                            const vsk_tensor* mask_indptr, int64_t max_len_extend,
                            float k_scale, float v_scale, float sm_scale,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Verify with the drafts already written to a paged KV cache (the unified
 * target-verify path of the "aiter_backend.py" page: the drafts' K/V are
 * stored before attention runs, the block table maps cache positions to
 * pages, and the key length of sequence b is seq_lens[b] + l_ext).  Cache
 * position t of sequence b lives in pool row
 *     block_table[b][t / page_size] * page_size + t % page_size;
 * positions [0, seq_lens[b]) are the prefix and [seq_lens[b], seq_lens[b] +
 * l_ext) the drafts, which see the whole prefix and, causally, the drafts up
 * to themselves.  k_scale / v_scale multiply EVERY cached key and value,
 * drafts included (they come from the same cache).  With l_ext = 1 this is
 * the plain paged decode step.
 *   q            [B*l_ext, h_q, D] bf16, sequence b's drafts at rows b*l_ext ..
 *   o            [B*l_ext, h_q, Dv] bf16 output (written, never read)
 *   k_cache, v_cache  [n_pages*page_size, h_kv, D] and [.., h_kv, Dv], bf16
 *                or fp8 e4m3 (same dtype), rows 16-byte aligned
 *   block_table  [B, max_blocks] int32 page ids, rows contiguous; only the
 *                columns covering positions < seq_lens[b] + l_ext are read
 *   seq_lens     [B] int32 cached tokens before the drafts
 *   page_size    tokens per page (>= 1); max_blocks*page_size must cover l_ext
 * D, Dv in {64, 128, 256}; (h_q/h_kv)*l_ext within the limits of
 * verify_splitkv_fwd, whose workspace rules, workspace size and return value
 * apply unchanged.  Device-side checks: a page id whose rows fall outside the
 * cache sets error bit 1 and those keys are left out; seq_lens[b] < 0 or
 * seq_lens[b] + l_ext beyond max_blocks*page_size sets bit 2 and sequence b
 * is computed with an empty prefix. */
int verify_splitkv_paged_fwd(const vsk_tensor* q, const vsk_tensor* o,
                             const vsk_tensor* k_cache, const vsk_tensor* v_cache,
                             const vsk_tensor* block_table, const vsk_tensor* seq_lens,
                             int64_t page_size, int64_t max_len_extend, float k_scale,
                             float v_scale, float sm_scale, void* workspace,
                             size_t workspace_bytes, void* stream);

/* verify_splitkv_fwd that also stores the new draft K/V into the cache in
 * the same launch (the draft K/V store that precedes attention on the
 * "aiter_backend.py" page, where the bf16 -> fp8 cast and the cache write are
 * one kernel).  Row t of sequence b (k_extend / v_extend row s_b + t) is
 * written to pool row out_cache_loc[s_b + t] of k_buffer / v_buffer as the
 * cache dtype's round-to-nearest-even of x / k_scale (x / v_scale for V) in
 * binary32, e4m3 saturating to +-448.  The attention itself is exactly that
 * of verify_splitkv_fwd: the drafts enter it as the fresh bf16 k_extend /
 * v_extend rows, without scales.
 *   out_cache_loc  [B*l_ext] int32 or int64 device array, one pool row per
 *                  q_extend row; those rows must not be prefix rows of any
 *                  sequence of the batch (they are written while the prefix
 *                  is being read).  A value outside [0, pool) is not written
 *                  and sets error bit 1.
 *   k_scale, v_scale  must be > 0 (they divide).
 * k_buffer / v_buffer are written through their (const-qualified) views.
 * Everything else as verify_splitkv_fwd (is_causal is implied). */
int verify_splitkv_write_fwd(const vsk_tensor* q_extend, const vsk_tensor* k_extend,
                             const vsk_tensor* v_extend, const vsk_tensor* o_extend,
                             const vsk_tensor* k_buffer, const vsk_tensor* v_buffer,
                             const vsk_tensor* qo_indptr, const vsk_tensor* kv_indptr,
                             const vsk_tensor* kv_indices, const vsk_tensor* out_cache_loc,
                             int64_t max_len_extend, float k_scale, float v_scale,
                             float sm_scale, void* workspace, size_t workspace_bytes,
                             void* stream);

/* verify_splitkv_paged_fwd with the drafts' K/V stored by the same launch:
 * k_new / v_new row b*l_ext + t ([B*l_ext, h_kv, D] / [B*l_ext, h_kv, Dv]
 * bf16) goes to cache position seq_lens[b] + t of k_cache / v_cache (block-
 * table addressing as in verify_splitkv_paged_fwd), stored as the cache
 * dtype's round-to-nearest-even of x / k_scale (x / v_scale) in binary32,
 * e4m3 saturating to +-448.  The attention then equals
 * verify_splitkv_paged_fwd run after that store: the drafts enter it as
 * stored (dequantised with k_scale / v_scale).  The draft positions must not
 * be prefix positions of any sequence of the batch; a draft position whose
 * page id is outside the cache is neither written nor attended and sets
 * error bit 1.  k_scale, v_scale must be > 0. */
int verify_splitkv_paged_write_fwd(const vsk_tensor* q, const vsk_tensor* k_new,
                                   const vsk_tensor* v_new, const vsk_tensor* o,
                                   const vsk_tensor* k_cache, const vsk_tensor* v_cache,
                                   const vsk_tensor* block_table, const vsk_tensor* seq_lens,
                                   int64_t page_size, int64_t max_len_extend, float k_scale,
                                   float v_scale, float sm_scale, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* Upper bound, in bytes, of the workspace verify_splitkv_fwd needs for any
 * batch of up to max_bs sequences with these head counts and sizes on the
 * CURRENT CUDA device (its SM count sets the number of persistent CTAs).
 * Returns 0 when the shapes are unsupported or no device is present. */
size_t vsk_workspace_size(int64_t max_bs, int64_t h_q, int64_t h_kv,
                          int64_t head_dim, int64_t v_head_dim,
                          int64_t max_len_extend);

/* Same bound for an explicit SM count (no CUDA call; usable without a GPU). */
size_t vsk_workspace_size_for_sms(int num_sms, int64_t max_bs, int64_t h_q,
                                  int64_t h_kv, int64_t head_dim,
                                  int64_t v_head_dim, int64_t max_len_extend);

/* Zero-fills `bytes` bytes of a workspace on `stream` (asynchronous).
 * Returns 1 on success, 0 on a CUDA error. */
int vsk_workspace_init(void* workspace, size_t bytes, void* stream);

/* Synchronises `stream`, then copies the device error word of `workspace`
 * into *flags and clears it.  workspace == NULL selects the library-owned
 * workspace of the current device, workspace == VSK_NOALLOC_SCRATCH the
 * built-in scratch of verify_splitkv_fwd_noalloc on the current device (its
 * word holds the flags of the most recent such call there).  Bits: 1 = a kv_indices value outside [0, pool); 2 = kv_indptr
 * not non-decreasing or beyond kv_indices; 4 = qo_indptr inconsistent with
 * l_ext; 8 = a pipeline wait that gave up after one second (only the
 * tensor-memory forms of the stream, selected by vsk_set_tuning_tc(1 or 2), have
 * such waits: the CTA then stops streaming, frees its tensor memory and
 * exits, and that call's output is not valid; the default kernel has no
 * waits that can time out); 16 = a mask_indptr entry of
 * verify_splitkv_tree_fwd outside custom_mask.  Returns 1 on success, 0 on a
 * CUDA error.
 * Intended for tests and debugging: it blocks the host. */
int vsk_read_error_flags(void* workspace, void* stream, uint32_t* flags);

/* Tuning override for tests and sweeps: number of persistent CTAs (0 = the
 * device's SM count times the CTAs that fit per SM) and the minimum prefix
 * tokens per CTA (0 = default: at least 64 tokens and at least the mean
 * prefix length / 24 from static shapes (kv_indices entries per sequence, or
 * the block table's capacity), which bounds the pieces a segment's finisher
 * merges; a nonzero value is used alone).  Affects the split of the prefix across
 * CTAs, never the definition of the result.  Process-wide; not thread-safe. */
void vsk_set_tuning(int num_ctas, int min_tokens_per_cta);

/* Tuning override of the CTA shape, for sweeps: at most `max_ring_stages`
 * 16-token stages in the shared-memory ring (>= 2; 0 = as many as fit) and at
 * most `max_kv_heads_per_cta` KV heads served by one CTA (a power of two;
 * 0 = up to 8).  Fewer heads per CTA means more, smaller CTAs per SM.  Never
 * changes the result beyond rounding order.  Process-wide; not thread-safe. */
void vsk_set_tuning_shape(int max_ring_stages, int max_kv_heads_per_cta);

/* Tuning override, for sweeps and tests: 16-row query tiles per consumer warp
 * (1 or 2; 0 = default: 2 at head_dim <= 128 when a KV head has more than 16
 * packed rows and the call's prefix holds at least 65,536 tokens (from static
 * shapes), else 1).  Affects the CTA shape, never the definition of the
 * result.  Process-wide; not thread-safe. */
void vsk_set_tuning_tiles(int tiles_per_warp);

/* Tuning switch over head_dim 256 calls with at most 32 packed query rows
 * per KV head ((h_q / h_kv) * max_len_extend <= 32): the tensor-memory forms
 * of the prefix stream (tcgen05.mma with accumulators in TMEM, one launch),
 * each followed by the combine kernel (a second launch on the same stream: it
 * folds the per-piece partials, adds the draft block and writes o).
 * vtr_kernel puts the packed query rows on the MMAs' M side (for an e4m3 pool
 * the queries split exactly into two e4m3 terms, so the scores come straight
 * from the e4m3 K rows); vtc_kernel puts the keys there.  Mode 3 (the
 * default) takes vtr_kernel where it measured faster on GB300: e4m3 pools with
 * 17-32 packed rows, or up to 16 rows below 1,048,576 prefix tokens x h_kv;
 * bf16 pools with up to 16 rows, or 17-32 rows below 786,432; never past
 * 8,388,608 (the one-launch kernel there).  Mode 2 takes vtr_kernel wherever
 * it applies, mode 1 vtc_kernel, mode 0 neither (the mma.sync forms only);
 * other values select mode 3.  All forms compute the same result up to
 * rounding order.  Process-wide; not thread-safe. */
void vsk_set_tuning_tc(int mode);

/* Tuning switch, for A/B runs and tests, over head_dim 256 calls with at most
 * 32 packed query rows per KV head.  Such a call can stream its prefix with
 * the column-split form of the mma.sync kernel (two warps share each 16-row
 * query tile, each holding half of the head dimension: half the accumulator
 * registers, so three CTAs of 2 to 4 warps fit an SM) and fold the partials in
 * a second launch on the same stream (the combine kernel: one CTA per
 * segment, 16-row tile and 32-column slice).  Mode 1 (the default) takes that
 * form when the call's prefix tokens (kv_indices entries, or block-table
 * capacity for the paged entry points) times h_kv are below 262,144 (bf16
 * pools) or 131,072 (e4m3), where it is the faster one on GB300 (from there
 * the stream-only kernel of vsk_set_tuning_split_launch takes over); mode 2
 * always takes it; mode 0 never does.  The tensor-memory streams of
 * vsk_set_tuning_tc take precedence (by default the rows-on-M one takes most
 * such calls).  All forms compute the same result up to rounding order.
 * Process-wide; not thread-safe. */
void vsk_set_tuning_colsplit(int mode);

/* Tuning switch, for A/B runs and tests, over head_dim 256 calls with 17 to 32
 * packed query rows per KV head: the column-split stream with both 16-row
 * tiles in each warp (one warp pair per KV head, each warp half of the head
 * dimension for both tiles, so every K / V element is loaded and, for an
 * e4m3 pool, converted once per head), then the combine kernel in a second
 * launch.  Mode 2 takes it wherever it applies, any pool and size; modes 0
 * and 1 (the default) never do: it beat the one-tile split on mid-size e4m3
 * calls, but the stream-only kernel of vsk_set_tuning_split_launch measured
 * faster still there.  All forms compute the same result up to rounding
 * order.  Process-wide; not thread-safe. */
void vsk_set_tuning_colsplit2(int mode);

/* Tuning switch, for A/B runs and tests, over calls with at most 32 draft
 * rows per sequence (head_dim == v_head_dim): the prefix is streamed by a
 * stream-only instance of the mma.sync kernel and the per-piece partials are
 * folded, the draft block added and o written by the combine kernel in a
 * second launch on the same stream (instead of the one-launch kernel's
 * ticketed tail).  Mode 1 (the default) takes that form where it measured
 * faster on GB300: at head_dim 64 / 128 when the call's prefix tokens times
 * h_kv are at most 4,194,304 (8,388,608 when (h_q / h_kv) * max_len_extend <=
 * 16); at head_dim 256 with at most 32 packed rows per KV head from where the
 * column split stops (262,144 bf16, 131,072 e4m3; any size with the column
 * split off) up to 8,388,608.  Mode 2 always takes it; mode 0
 * never does.  All forms compute the same result up to rounding order.
 * Process-wide; not thread-safe. */
void vsk_set_tuning_split_launch(int mode);

/* Tuning switch, for A/B runs and tests: the cluster form.  One
 * thread-block cluster of up to 16 CTAs per (sequence, KV head) segment
 * streams that segment's prefix, then, after a cluster barrier, the
 * cluster's CTAs fold the segment's partials, add the draft block and write
 * o: one launch, no tickets, no second kernel.  It serves head_dim ==
 * v_head_dim, at most 32 draft rows per sequence and at most 512 segments.
 * Mode 0 (the default) never takes it: the stream-only kernel with the
 * combine kernel launched as a programmatic dependent measured faster on
 * GB300 at every size (the tiny case 18.3 -> 16.3 us, warm).  Mode 1 takes
 * it when the call's prefix tokens (kv_indices entries, or block-table
 * capacity for the paged entry points) times h_kv are fewer than 2,048, where
 * it beat the one-launch kernel before that; mode 2 wherever it applies.
 * The tensor-memory streams of vsk_set_tuning_tc take precedence.  All forms
 * compute the same result up to rounding order.  Process-wide; not thread-safe. */
void vsk_set_tuning_cluster(int mode);

/* Tuning switch, for A/B runs: how the combine kernel of the two-launch forms
 * follows the prefix stream.  As a programmatic dependent
 * (cudaLaunchAttributeProgrammaticStreamSerialization) its CTAs may start
 * while the stream runs, read the call's lengths, qo_indptr and draft-row
 * locations, and wait for the stream grid before reading anything else;
 * otherwise it starts after the stream in plain stream order.  Mode 1 (the
 * default) takes the programmatic form for calls of at most 65,536 prefix
 * tokens x KV heads (about 2 us faster there on GB300; neutral to slower on
 * mid-size calls), mode 2 always, mode 0 never.  The result is the same
 * either way.  Process-wide; not thread-safe. */
void vsk_set_tuning_pdl(int mode);

/* Tuning switch, for A/B runs: mode 1 (the default) runs the head_dim 256
 * one-launch kernel over fp8 e4m3 pools (ring of at least three stages) with
 * software-pipelined stages (the softmax and PV products of a 16-token stage
 * are computed after the QK products of the next stage are issued, so each
 * warp interleaves two stages' work); mode 0 runs one stage after the other.
 * bf16 pools always run one stage after the other (pipelining measured no
 * faster there).  The result is the same either way.  Process-wide; not
 * thread-safe. */
void vsk_set_tuning_pipe(int mode);

/* Kernel launches a call of these static shapes makes on its stream under the
 * current tuning switches: 1 (the one-launch kernel) or 2 (a prefix stream,
 * then the combine kernel); 0 for shapes no entry point accepts.
 * `prefix_tokens` is what the entry point sees: the length of kv_indices for
 * the flat entry points, batch x block-table columns x page_size for the paged
 * ones.  For head_dim == v_head_dim; a call with v_head_dim != head_dim makes
 * one launch.  The count does not depend on the pool dtype (the pool-dependent
 * cut-overs all lie between two-launch forms).  Host only (no device call);
 * for CUDA-graph bookkeeping and launch counts. */
int vsk_launches_per_call(int64_t batch, int64_t h_q, int64_t h_kv, int64_t head_dim, int64_t max_len_extend,
                          int64_t prefix_tokens);

/* The form a call of these static shapes takes under the current tuning
 * switches, as a static string: "one_launch" (the persistent kernel, tickets
 * for the merge), "cluster" (one launch of thread-block clusters),
 * "column_split", "column_split_two_tiles", "stream_only",
 * "tensor_memory_rows" (vtr_kernel) or "tensor_memory" (vtc_kernel) (each a
 * prefix stream, then the combine kernel), or "" for shapes no entry point
 * accepts.  fp8_pool: nonzero for an e4m3 K/V pool (some cut-overs
 * depend on it).  prefix_tokens as for vsk_launches_per_call.  Host only. */
const char* vsk_call_form(int64_t batch, int64_t h_q, int64_t h_kv, int64_t head_dim, int64_t v_head_dim,
                          int64_t max_len_extend, int64_t prefix_tokens, int fp8_pool);

/* Size, in bytes, of the scratch array built into the library for
 * verify_splitkv_fwd_noalloc (32 MiB). */
#define VSK_NOALLOC_SCRATCH_BYTES (32 * 1024 * 1024)

/* Passed as the `workspace` argument of vsk_read_error_flags: selects the
 * built-in scratch of verify_splitkv_fwd_noalloc (a selector, never
 * dereferenced). */
#define VSK_NOALLOC_SCRATCH ((void*)1)

/* verify_splitkv_fwd for callers that must not allocate device memory.  The
 * source pages have no counterpart: it is a deployment convenience of this
 * library.  Some callers cannot call cudaMalloc: serving engines that give
 * all free HBM to their own pool allocator up front (a stray allocation can
 * fail, fragment that pool or stall the device while memory is mapped), and
 * plugin hosts whose interface passes only input and output pointers.  This
 * entry point takes the same tensors as verify_splitkv_fwd but no workspace:
 * its scratch is a VSK_NOALLOC_SCRATCH_BYTES array in the library's device
 * image, which every GPU that loads the library holds until the process
 * exits.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) and caches it; make that first call before any
 *     stream capture on that device.
 *   - The call plans exactly as verify_splitkv_fwd does (the same form: one
 *     launch, or a prefix stream then the combine kernel) and checks that
 *     plan's scratch against the array.  It then clears the array's error
 *     word and its ticket region on `stream` (cudaMemsetAsync) and enqueues
 *     the kernels.  vsk_read_error_flags(VSK_NOALLOC_SCRATCH, ...) reads
 *     (and clears) the error word of the most recent call on the device.
 *   - Every call shares the one array: calls whose kernels may overlap on the
 *     GPU (different streams, or different host threads) race and corrupt
 *     each other's results.  Serialise them on one stream.
 *   - A problem whose scratch exceeds VSK_NOALLOC_SCRATCH_BYTES (roughly, more
 *     than a few hundred sequence x KV-head-group segments at head_dim 128)
 *     is rejected: returns 0, nothing enqueued, and vsk_last_error() says so.
 * Returns 1 once enqueued, 0 otherwise (see verify_splitkv_fwd). */
int verify_splitkv_fwd_noalloc(const vsk_tensor* q_extend, const vsk_tensor* k_extend,
                               const vsk_tensor* v_extend, const vsk_tensor* o_extend,
                               const vsk_tensor* k_buffer, const vsk_tensor* v_buffer,
                               const vsk_tensor* qo_indptr, const vsk_tensor* kv_indptr,
                               const vsk_tensor* kv_indices, int is_causal,
                               int64_t max_len_extend, float k_scale, float v_scale,
                               float sm_scale, void* stream);

/* Message of the most recent 0 return on this host thread ("" if none). */
const char* vsk_last_error(void);

/* Library version string. */
const char* vsk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_SPLITKV_H */
