/*
 * kv_oracle.c -- plain CPU oracle for the KV-cache steps around verification.
 * TEST INFRASTRUCTURE ONLY, like sv_oracle.c (the two are built into one
 * library): loaded by the tests, the smoke check and the benchmark's
 * CPU-baseline leg, never by the product path, and sharing no code with the
 * CUDA library.
 *
 * Sources (page title and section):
 *   [Deferred-SD] deferred speculative decoding page (lqnn.cn):
 *       "环形上下文与注意力沉淀机制" -- the cache holds S persistent sink slots
 *           and a ring of W slots; Slot(pos) = pos for pos < S, else
 *           S + ((pos - S) mod W);
 *       "C++ 环形 KV 缓存管理内核实现" -- a preallocated pool
 *           [layers][heads][S + W][dim]; appending writes the entry of the
 *           current logical position to Slot(pos) and steps pos; the valid
 *           slots are 0..pos-1 while pos <= S + W, else the sinks followed by
 *           the ring slots of the last W positions, oldest first.
 *   [Draft-window] vllm-ascend draft KV sliding-window page (cf-1.com):
 *       "窗口数学" -- start = floor(max(seq + K - W, 0) / b) * b,
 *           windowed_len = seq - start, start_block = start / b,
 *           needed = ceil(windowed_len / b) <= W / b + 1;
 *       "block table 的裁剪方式" -- the clone [reqs][max_window_blocks] takes columns
 *           start_block + j of the full table (the gather index clamped to the
 *           last column), zero in columns j >= needed and where
 *           start_block + j is past the full table's width;
 *       "两条贯穿始终的不变量" -- every length input is windowed by the same
 *           arithmetic; the slot mapping (writes) is never windowed.
 *
 * Readings taken where the page leaves a step open:
 *   K1  what is committed: the verification step ran the target over R =
 *       gamma + 1 inputs (the last emitted token and the gamma drafts) at
 *       logical positions pos .. pos + gamma and staged their KV; with k drafts
 *       accepted, entries 0..k are valid and are appended in order (the
 *       emitted token k is not yet in the cache: it is the next step's first
 *       input).  pos advances by k + 1.  The page's Rollback(accepted) -- it
 *       SUBTRACTS its argument from pos -- is read as dropping the gamma - k
 *       rejected entries; staging them and appending only the accepted ones
 *       reaches the same pos without writing rejected entries over live ring
 *       slots.  k < 0 commits nothing (a dropped request); k > gamma is
 *       invalid (flagged, nothing written).
 *   K2  a commit of more than W entries would overwrite its own entries;
 *       callers keep W >= R (the library rejects W < R).
 *   K3  the block-table clone's gather reads column min(start_block + j,
 *       full_cols - 1), and the value is then zeroed where j >= needed or
 *       start_block + j >= full_cols: the clamp only keeps the gather in
 *       bounds.  Negative sequence lengths are invalid (flagged; outputs 0).
 *   K4  the clone's width: the page bounds `needed` by W / b + 1, which holds
 *       when b divides W; otherwise windowed_len <= W + b - 1 can need one
 *       column more (W = 100, b = 16, K = 0, seq = 113: start 0, 8 blocks,
 *       W / b + 1 = 7).  The clone here has max(W / b + 1,
 *       ceil((W + b - 1) / b)) columns: the page's width, one more when
 *       W mod b >= 2.
 *
 * Every loop below is the definition written out.
 */
#include <stdint.h>
#include <string.h>

#ifndef SVO_MUTANT
#define SVO_MUTANT 0
#endif

#define KVO_INVALID 1

/* [Deferred-SD] "环形上下文与注意力沉淀机制": the slot formula. */
static int64_t kvo_slot(int64_t pos, int64_t sink, int64_t window) {
  if (pos < sink) return pos;
#if SVO_MUTANT == 12
  return (pos - sink) % window; /* planted: the ring offset by the sinks is lost */
#else
  return sink + (pos - sink) % window;
#endif
}

int64_t kvo_slot_of(int64_t pos, int sink, int window) { return kvo_slot(pos, sink, window); }

/* KV commit after verification (reading K1), request by request, entry by
 * entry, as the page's cache manager appends: write the entry of position
 * pos to Slot(pos), step pos.
 *   k_pool, v_pool [B][LH][sink + window][row_bytes]   (bytes)
 *   k_new, v_new   [B][LH][R][row_bytes]               (entry j: position pos + j)
 *   num_accepted   [B]; pos [B] in/out; out_flags [B] (KVO_INVALID) */
int kvo_commit(unsigned char* k_pool, unsigned char* v_pool, const unsigned char* k_new,
               const unsigned char* v_new, const int32_t* num_accepted, int32_t* pos, int B,
               int LH, int R, int row_bytes, int sink, int window, int32_t* out_flags) {
  if (B < 0 || LH < 0 || R < 1 || row_bytes < 0 || sink < 0 || window < 1) return -1;
  const size_t C = (size_t)sink + (size_t)window;
  for (int b = 0; b < B; ++b) {
    out_flags[b] = 0;
    const int k = num_accepted[b];
    if (k >= R || pos[b] < 0) { out_flags[b] = KVO_INVALID; continue; }
    if (k < 0) continue;
#if SVO_MUTANT == 13
    const int count = k; /* planted: the entry of the last emitted token is not committed */
#else
    const int count = k + 1;
#endif
    for (int j = 0; j < count; ++j) {
      const int64_t p = (int64_t)pos[b] + j;
      const size_t slot = (size_t)kvo_slot(p, sink, window);
      for (int lh = 0; lh < LH; ++lh) {
        const size_t dst = (((size_t)b * LH + lh) * C + slot) * (size_t)row_bytes;
        const size_t src = (((size_t)b * LH + lh) * (size_t)R + (size_t)j) * (size_t)row_bytes;
        memcpy(k_pool + dst, k_new + src, (size_t)row_bytes);
        memcpy(v_pool + dst, v_new + src, (size_t)row_bytes);
      }
    }
    pos[b] += count;
  }
  return 0;
}

/* The valid slots of every request in logical order ([Deferred-SD] cache
 * manager): out_slots [B][sink + window] (-1 past out_len[b]). */
int kvo_valid_slots(const int32_t* pos, int B, int sink, int window, int32_t* out_slots,
                    int32_t* out_len) {
  if (B < 0 || sink < 0 || window < 1) return -1;
  const int64_t C = (int64_t)sink + window;
  for (int b = 0; b < B; ++b) {
    int32_t* o = out_slots + (size_t)b * (size_t)C;
    for (int64_t j = 0; j < C; ++j) o[j] = -1;
    const int64_t p = pos[b];
    if (p < 0) { out_len[b] = 0; continue; }
    int64_t n = 0;
    if (p <= C) {
      for (int64_t i = 0; i < p; ++i) o[n++] = (int32_t)i;
    } else {
      for (int64_t i = 0; i < sink; ++i) o[n++] = (int32_t)i;
      const int64_t first = p - window; /* oldest position still in the ring */
      for (int64_t i = 0; i < window; ++i) o[n++] = (int32_t)kvo_slot(first + i, sink, window);
    }
    out_len[b] = (int32_t)n;
  }
  return 0;
}

/* Width of the block-table clone (reading K4). */
int kvo_window_cols(int W, int blk) {
  if (W < 1 || blk < 1) return -1;
  const int64_t page = (int64_t)W / blk + 1;
  const int64_t bound = ((int64_t)W + blk - 1 + blk - 1) / blk; /* ceil((W + b - 1) / b) */
  return (int)(page > bound ? page : bound);
}

/* [Draft-window] "窗口数学" and "block table 的裁剪方式" (readings K3, K4).
 *   seq_lens [B], table [B][full_cols]; outputs out_seq [B],
 *   out_table [B][max_cols] (max_cols = kvo_window_cols(W, blk)),
 *   out_start_block [B], out_needed [B], out_flags [B]. */
int kvo_window_block_table(const int32_t* seq_lens, const int32_t* table, int B, int full_cols,
                           int W, int blk, int K, int max_cols, int32_t* out_seq,
                           int32_t* out_table, int32_t* out_start_block, int32_t* out_needed,
                           int32_t* out_flags) {
  if (B < 0 || full_cols < 1 || W < 1 || blk < 1 || K < 0 || max_cols != kvo_window_cols(W, blk))
    return -1;
  for (int b = 0; b < B; ++b) {
    int32_t* ot = out_table + (size_t)b * (size_t)max_cols;
    for (int j = 0; j < max_cols; ++j) ot[j] = 0;
    out_flags[b] = 0;
    const int64_t seq = seq_lens[b];
    if (seq < 0) {
      out_flags[b] = KVO_INVALID;
      out_seq[b] = 0;
      out_start_block[b] = 0;
      out_needed[b] = 0;
      continue;
    }
    int64_t lo = seq + (int64_t)K - (int64_t)W;
    if (lo < 0) lo = 0;
#if SVO_MUTANT == 14
    const int64_t start = lo; /* planted: the start is not aligned down to a block */
#else
    const int64_t start = (lo / blk) * blk;
#endif
    const int64_t windowed = seq - start;
    const int64_t start_block = start / blk;
    const int64_t needed = (windowed + blk - 1) / blk;
    out_seq[b] = (int32_t)windowed;
    out_start_block[b] = (int32_t)start_block;
    out_needed[b] = (int32_t)needed;
    for (int j = 0; j < max_cols; ++j) {
      int64_t col = start_block + j;
      const int in_table = col < full_cols;
      if (col > full_cols - 1) col = full_cols - 1;
      const int32_t v = table[(size_t)b * (size_t)full_cols + (size_t)col];
#if SVO_MUTANT == 15
      ot[j] = in_table ? v : 0; /* planted: columns past `needed` are not zeroed */
#else
      ot[j] = (j < needed && in_table) ? v : 0;
#endif
    }
  }
  return 0;
}
