/*
 * svtree.h -- C ABI of token-tree (multi-branch) verification, in the same
 * library as specverify.h (libspecverify.so).
 *
 * Sources (page title and section):
 *   deferred speculative decoding page (lqnn.cn), opening section: the draft
 *     model emits a candidate token tree into the proposal queue that the
 *     accept / reject kernel evaluates;
 *   猜想解码 (Speculative Decoding) 全景, 考点3 (tree attention verifies
 *     several branches in one forward pass) and 考点2 (acceptance
 *     min(1, P_t / P_d), residual max(0, P_t - P_d) normalised, lossless).
 * The pages give no rule for sibling drafts; this call takes the multi-draft
 * form of the 考点2 rule (readings of the library's design notes):
 *
 *   the walk starts at the root, r = P_t[root];
 *   at node n, the children c of n are tested in index order with x =
 *   tokens[c] and Q = P_d[n]: accept iff u_accept[c] <= min(1, r(x) / Q(x))
 *   (Q(x) == 0 accepts); an accepted child is emitted and the walk moves to
 *   it with r = P_t[c]; a rejected one replaces r by
 *   max(0, r - Q) / sum_v max(0, r - Q);
 *   when no child is accepted (or n is a leaf) one token is drawn from r by
 *   the index-order inverse CDF with u_residual[n] (the smallest v whose
 *   running sum exceeds u * sum) and the walk ends.
 *   The result is distributed as P_t along the walk when the siblings were
 *   drawn independently from their parent's draft distribution.
 *   P = softmax(logits / T) per row, T = temperature[b].
 *
 * Layouts (row-major; dtype SV_F32 or SV_BF16 as in specverify.h):
 *   target_logits [B][N][V]: row n = the target distribution after the
 *                            path to node n (the tree-attention output)
 *   draft_logits  [B][N][V]: row n = the distribution n's children were drawn
 *                            from (rows of leaves are never read; may be NULL
 *                            when N == 1)
 *   parent        [B][N] int32: parent[b][0] == -1, 0 <= parent[b][n] < n
 *   tokens        [B][N] int32: token of node n (entry 0 unused)
 *   u_accept      [B][N] float: entry n used when node n is tested (entry 0
 *                            unused; may be NULL when N == 1)
 *   u_residual    [B][N] float: entry n used when the walk ends at node n
 *   temperature   [B] float
 *   out_tokens    [B][N] int32: tokens of the accepted nodes, then the drawn
 *                            token, then -1
 *   out_num_accepted [B] int32: accepted nodes (0 for an invalid request)
 *   out_nodes     [B][N] int32: the accepted nodes in order, then -1 (may be
 *                            NULL)
 * Only the rows on the walk are read: the target row of each visited node
 * and the draft row of each visited node that has children.  Validity
 * (bits OR-ed into *dev_status, which may be NULL; the request's outputs are
 * then -1 / 0):
 *   SV_ST_NONFINITE  a row the walk reads holds NaN / +inf or is all -inf
 *   SV_ST_BAD_TOKEN  a malformed parent array or a token outside [0, V)
 *   SV_ST_BAD_TEMP   temperature not finite or below 2^-126
 *   SV_ST_DEGENERATE (informational) a residual summed to 0 and P_t[n] was
 *                    used in its place
 * Requires 1 <= N <= SV_TREE_MAX_N, V >= 1, B >= 0, logit pointers aligned to
 * their element size.  All buffers are caller-owned device memory; the call
 * is one kernel launch on `stream` (a cudaStream_t, NULL = legacy default)
 * and needs no workspace.  Returns SV_OK or an SV_ERR_* code of
 * specverify.h.
 */
#ifndef SVTREE_H
#define SVTREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SV_TREE_MAX_N 256

int sv_tree_verify(int dtype, const void* target_logits, const void* draft_logits,
                   const int32_t* parent, const int32_t* tokens, const float* u_accept,
                   const float* u_residual, const float* temperature, int B, int N, int V,
                   int32_t* out_tokens, int32_t* out_num_accepted, int32_t* out_nodes,
                   int32_t* dev_status, void* stream);

/*
 * CTAs per request for sv_tree_verify (tuning and test aid): 0 (the
 * default) picks min(8, max(1, k * SMs / B)) with k = 2 for CTAs of 8 warps
 * and 1 for CTAs of 16 (sv_tree_set_warps); 1..8 forces that size.
 * Returns SV_OK or SV_ERR_INVALID_ARG.
 */
int sv_tree_set_cluster(int ctas);

/*
 * Warps per CTA for sv_tree_verify (tuning and test aid): 0 (the default)
 * takes 8 (two CTAs per SM) when 5 * B <= 4 * SMs and 16 (one CTA per SM)
 * otherwise; 8 or 16 forces that width.  The results are those of the
 * oracle either way (the rows' segment split, and so the rounding of the
 * masses, differs).  Returns SV_OK or SV_ERR_INVALID_ARG.
 */
int sv_tree_set_warps(int warps);

#ifdef __cplusplus
}
#endif

#endif /* SVTREE_H */
