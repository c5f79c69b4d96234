/*
 * svkv.h -- C ABI of the KV-cache steps around verification, in the same
 * library as specverify.h (libspecverify.so): committing the verified
 * entries to a sink + ring KV cache, listing its valid slots, and windowing
 * the draft model's block table.
 *
 * Sources (page title and section):
 *   deferred speculative decoding page (lqnn.cn): "环形上下文与注意力沉淀机制"
 *     (S persistent sink slots, a ring of W slots, Slot(pos) = pos for
 *     pos < S, else S + ((pos - S) mod W)) and "C++ 环形 KV 缓存管理内核实现"
 *     (a preallocated pool per layer and head; append at Slot(pos), step pos;
 *     roll back after a failed speculation; the valid slots in logical order);
 *   vllm-ascend draft KV sliding-window page (cf-1.com): "窗口数学"
 *     (start = floor(max(seq + K - W, 0) / b) * b, windowed_len = seq - start,
 *     needed = ceil(windowed_len / b)), "block table 的裁剪方式" (the
 *     zero-padded clone of the block table's columns start / b + j) and
 *     "两条贯穿始终的不变量" (every length windowed by the same arithmetic,
 *     writes never windowed).
 *
 * Conventions as in specverify.h: caller-owned device buffers, calls
 * enqueued on `stream` (a cudaStream_t, NULL = legacy default stream),
 * host-detectable errors returned (SV_ERR_* codes of specverify.h), data
 * errors OR-ed into *dev_status (may be NULL) per request, nothing traps.
 */
#ifndef SVKV_H
#define SVKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* device status bit (besides the SV_ST_* bits of specverify.h) */
#define SV_ST_BAD_LENGTH 0x40 /* a negative position / sequence length, or an accepted
                                 count past the staged entries */

/*
 * Commit the verified entries of one speculation step to a sink + ring KV
 * cache, per request b:
 *   the step staged the KV of R = gamma + 1 inputs (the last emitted token and
 *   the gamma drafts) for logical positions pos[b] .. pos[b] + R - 1;
 *   with k = num_accepted[b] (spec_verify's out_num_accepted) the entries
 *   j = 0..k are valid: entry j is copied to ring slot Slot(pos[b] + j) of
 *   every layer/head row, and pos[b] advances by k + 1.  The other entries
 *   (rejected drafts) are dropped: the cache keeps its older entries, which
 *   an in-place append followed by a position rollback would overwrite.
 *   k < 0: nothing is committed (a dropped request).  k >= R or pos[b] < 0:
 *   nothing is committed and SV_ST_BAD_LENGTH is reported.
 * Layouts (bytes, row-major):
 *   k_pool, v_pool [B][LH][sink + window][row_bytes]   (LH = layers * kv heads)
 *   k_new, v_new   [B][LH][R][row_bytes]
 *   num_accepted [B] int32; pos [B] int32, updated in place.
 * Requires row_bytes a positive multiple of 16, all four KV buffers 16-byte
 * aligned, window >= R (a commit never laps the ring), sink >= 0, LH >= 1,
 * R <= 64, row_bytes <= 8192, LH * R * row_bytes <= 2^34 and B <= 65535;
 * positions stay below 2^31 - R
 * (a larger one is reported as SV_ST_BAD_LENGTH).
 * Two kernels: the copy, then the position update.
 */
int sv_kv_commit(void* k_pool, void* v_pool, const void* k_new, const void* v_new,
                 const int32_t* num_accepted, int32_t* pos, int B, int LH, int R,
                 int row_bytes, int sink, int window, int32_t* dev_status, void* stream);

/*
 * The valid physical slots of every request in logical order:
 *   pos[b] <= sink + window: slots 0 .. pos[b] - 1;
 *   otherwise the sinks 0 .. sink - 1, then Slot(p) for the last `window`
 *   positions p = pos[b] - window .. pos[b] - 1.
 * out_slots [B][sink + window] int32 (-1 past out_len[b]), out_len [B] int32.
 * pos[b] < 0 gives length 0 and SV_ST_BAD_LENGTH.
 */
int sv_kv_valid_slots(const int32_t* pos, int B, int sink, int window, int32_t* out_slots,
                      int32_t* out_len, int32_t* dev_status, void* stream);

/*
 * Width of the draft block-table clone for window W and block size b:
 * max(W / b + 1, ceil((W + b - 1) / b)).  The page's bound W / b + 1 holds
 * when b divides W; otherwise a window of up to W + b - 1 tokens can need
 * one column more.  Returns -1 for W < 1 or b < 1.
 */
int sv_window_cols(int window, int block_size);

/*
 * Draft KV sliding window (device), per request b with s = seq_lens[b]:
 *   start = floor(max(s + K - W, 0) / b) * b, out_seq_lens[b] = s - start,
 *   out_start_block[b] = start / b (may be NULL),
 *   out_block_table[b][j] = block_table[b][start / b + j] for
 *     j < ceil((s - start) / b) and start / b + j < full_cols, else 0,
 *   for j < sv_window_cols(W, b).
 * Layouts: seq_lens [B], block_table [B][full_cols], out_block_table
 * [B][sv_window_cols(W, b)], all int32.  K (future_offset) >= 0.
 * A negative seq_lens[b] gives 0 everywhere for b and SV_ST_BAD_LENGTH.
 */
int sv_window_block_table(const int32_t* seq_lens, const int32_t* block_table, int B,
                          int full_cols, int window, int block_size, int future_offset,
                          int32_t* out_seq_lens, int32_t* out_block_table,
                          int32_t* out_start_block, int32_t* dev_status, void* stream);

/*
 * The same windowing of sequence lengths on the host, for host-side mirrors
 * of the lengths (every copy of a length must be windowed alike): n lengths
 * from `seq_lens` to `out` (may alias).  Negative lengths give 0.  Returns
 * SV_OK, or SV_ERR_INVALID_ARG for bad W, b, K or NULL pointers with n > 0.
 */
int sv_window_seq_lens_host(const int32_t* seq_lens, int n, int window, int block_size,
                            int future_offset, int32_t* out);

#ifdef __cplusplus
}
#endif

#endif /* SVKV_H */
