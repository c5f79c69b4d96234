/*
 * specverify.h -- C ABI of the GB300 (sm_103a) speculative-decoding
 * verification library (libspecverify.so).
 *
 * The operation (Speculative Decoding overview page, "猜想解码 (Speculative
 * Decoding) 全景", sections 考点2, 第二章 and 第三章; the deferred-speculation
 * page's scheduler section "动态推迟投机验证调度器设计"):
 *
 *   for every request b, with temperature T_b, target rows i = 0..gamma and
 *   draft rows i = 0..gamma-1 over a vocabulary of V entries:
 *     P_t[i] = softmax(Lt[b][i] / T_b),  P_d[i] = softmax(Ld[b][i] / T_b)
 *     r_i    = min(1, P_t[i][x_i] / P_d[i][x_i])      (r_i = 1 when P_d[i][x_i] = 0)
 *     accept x_i iff u_accept[b][i] <= r_i; k = first i that is not accepted,
 *     or gamma when all are
 *     k < gamma: w = max(0, P_t[k] - P_d[k])  (residual distribution)
 *     k = gamma: w = P_t[gamma]              (bonus token)
 *     token k = smallest v with sum_{j<=v} w_j > u_resample[b][k] * sum_j w_j
 *   outputs: out_tokens[b] = (x_0 .. x_{k-1}, token k, -1 ...), out_num_accepted[b] = k.
 *
 * Layouts (all row-major, contiguous):
 *   target_logits  [B][gamma+1][V]   dtype (SV_F32: float, SV_BF16: bfloat16 bits)
 *   draft_logits   [B][gamma][V]     dtype
 *   draft_tokens   [B][gamma]        int32, expected in [0, V)
 *   u_accept       [B][gamma]        float, in [0, 1)
 *   u_resample     [B][gamma+1]      float, in [0, 1); only entry k is used
 *   temperature    [B]               float, finite and >= 2^-126
 *   out_tokens     [B][gamma+1]      int32, -1 padded
 *   out_num_accepted [B]             int32, in [0, gamma]
 *
 * Conventions:
 *   - Every pointer is a DEVICE pointer owned by the caller (logit pointers
 *     aligned to their element size, all others to 4 bytes); the library
 *     allocates nothing.  Calls are enqueued on `stream` (a cudaStream_t;
 *     NULL = legacy default stream) and return before the work finishes.
 *   - The return value reports only what the host can see: a bad argument, a
 *     too small workspace, or a failed launch.  Data errors are reported per
 *     request on the device: that request gets out_num_accepted = 0 and
 *     out_tokens all -1, and the matching SV_ST_* bit is OR-ed into
 *     *dev_status (when dev_status is not NULL).  Nothing traps.
 *   - -inf logits are legal (probability 0).  NaN or +inf anywhere in a
 *     request's rows, an all -inf row, a draft token outside [0, V) or a bad
 *     temperature invalidate that request only.
 *   - workspace: sv_workspace_bytes() bytes of device memory, 256-byte
 *     aligned, zeroed ONCE before its first use (sv_workspace_init); every
 *     call leaves it ready for the next one.  Calls that may overlap on the
 *     GPU (different streams) need separate workspaces.
 *   - The library is thread-safe apart from sv_set_tuning().
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* logit storage types */
enum { SV_F32 = 0, SV_BF16 = 1 };

/* host return codes */
enum {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1, /* NULL pointer, B < 0, gamma outside [0, SV_MAX_GAMMA], V < 1, misalignment */
  SV_ERR_DTYPE = 2,       /* dtype is neither SV_F32 nor SV_BF16 */
  SV_ERR_CUDA = 3,        /* a CUDA runtime call or the launch failed */
  SV_ERR_WORKSPACE = 4    /* workspace NULL, unaligned or smaller than sv_workspace_bytes() */
};

/* device status bits, OR-ed into *dev_status */
#define SV_ST_NONFINITE 0x1   /* NaN / +inf logit, or an all -inf row, in a request */
#define SV_ST_BAD_TOKEN 0x2   /* a draft token outside [0, V) */
#define SV_ST_BAD_TEMP 0x4    /* temperature not finite or below 2^-126 */
#define SV_ST_TIMEOUT 0x8     /* an internal wait gave up (results of the call are void) */
#define SV_ST_WORKSPACE 0x10  /* the workspace's control block was not in its ready state
                                 (another call's work overlapped, or it was overwritten);
                                 the call that reports this leaves it ready again */
#define SV_ST_DEGENERATE 0x20 /* informational: a residual summed to 0 and the target row
                                 was sampled instead */

#define SV_MAX_GAMMA 32

/* Bytes of workspace needed for any call with these sizes (any dtype). */
size_t sv_workspace_bytes(int B, int gamma, int V);

/* Zero a workspace on `stream` (a cudaMemsetAsync).  Call once after
 * allocating it. */
int sv_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Sampling verification (T > 0) for B requests -- the operation above.
 * dev_status may be NULL.  For gamma == 0, draft_logits, draft_tokens and
 * u_accept may be NULL: token 0 is then sampled from target row 0.
 */
int spec_verify(const void* target_logits, const void* draft_logits,
                const int32_t* draft_tokens, const float* u_accept,
                const float* u_resample, const float* temperature, int B, int gamma,
                int V, int dtype, int32_t* out_tokens, int32_t* out_num_accepted,
                void* workspace, size_t workspace_bytes, int32_t* dev_status,
                void* stream);

/*
 * spec_verify plus diagnostics (either may be NULL):
 *   out_p [B][gamma][2] float: (P_t[i][x_i], P_d[i][x_i]) for every i < gamma
 *   out_Z [B] float: the mass the final token was drawn from (sum of the
 *         residual after a rejection, sum of P_t[gamma] for the bonus)
 */
int spec_verify_diag(const void* target_logits, const void* draft_logits,
                     const int32_t* draft_tokens, const float* u_accept,
                     const float* u_resample, const float* temperature, int B,
                     int gamma, int V, int dtype, int32_t* out_tokens,
                     int32_t* out_num_accepted, float* out_p, float* out_Z,
                     void* workspace, size_t workspace_bytes, int32_t* dev_status,
                     void* stream);

/*
 * Greedy verification (temperature 0): a_i = argmax_v target_logits[b][i][v]
 * over the stored values, lowest index on ties; k = first i < gamma with
 * draft_tokens[b][i] != a_i, else gamma; out_tokens[b] = (a_0 .. a_k, -1 ...),
 * out_num_accepted[b] = k.  This is the temperature -> 0 limit of the
 * sampling rule (the pages give no greedy rule of their own).
 */
int spec_verify_greedy(const void* target_logits, const int32_t* draft_tokens, int B,
                       int gamma, int V, int dtype, int32_t* out_tokens,
                       int32_t* out_num_accepted, void* workspace, size_t workspace_bytes,
                       int32_t* dev_status, void* stream);

/*
 * Draft-side sampling: the step before verification.  The token x_i that
 * verification tests is one the draft model sampled from its own distribution
 * (Speculative Decoding overview page, 考点2 and the NumPy operator of
 * 第三章).  For every request b and row i < n of
 *   draft_logits [B][n][V]  dtype (one or more draft positions per request):
 *     P = softmax(draft_logits[b][i] / T_b)
 *     token = smallest v with sum_{j<=v} P_j > u_draft[b][i]   (index-order inverse CDF,
 *             the rule of the bonus token)
 *     m = max_v draft_logits[b][i][v] (the stored value), S = sum_v exp((l_v - m) / T_b)
 *   written to out_tokens[b * ncols + col + i] (int32) and
 *   out_stats[(b * ncols + col + i) * 2 + {0, 1}] = (m, S) (float).
 * col/ncols let a draft loop write position i of a [B][gamma] token array
 * one draft step at a time (n = 1, col = i, ncols = gamma) or all positions
 * at once (n = gamma, col = 0, ncols = gamma).  out_stats so written is the
 * draft_stats input of spec_verify_cached.
 *   u_draft [B][n] float in [0, 1); temperature [B] as for spec_verify.
 *   Requires 1 <= n <= SV_MAX_GAMMA, 0 <= col, col + n <= ncols.
 *   workspace: sv_draft_workspace_bytes(B, n, V) bytes, prepared as for
 *   spec_verify (the same workspace may serve both, if large enough for each,
 *   on one stream).
 *   A row with NaN / +inf, only -inf, or a bad temperature gets token -1 and
 *   stats (NaN, NaN); SV_ST_NONFINITE or SV_ST_BAD_TEMP is OR-ed into
 *   *dev_status.
 */
size_t sv_draft_workspace_bytes(int B, int n, int V);
int sv_draft_sample(const void* draft_logits, const float* u_draft, const float* temperature,
                    int B, int n, int V, int dtype, int col, int ncols, int32_t* out_tokens,
                    float* out_stats, void* workspace, size_t workspace_bytes,
                    int32_t* dev_status, void* stream);

/*
 * spec_verify with the draft rows' normalisers given: draft_stats
 * [B][gamma][2] float (8-byte aligned), (m, S) of every draft row as
 * sv_draft_sample reports them.  The result is spec_verify's; the draft rows
 * are then read only where needed (the logit of x_i, and row k after a
 * rejection), so the streaming pass reads (gamma + 1) * V logits per request
 * instead of (2 * gamma + 1) * V.  Stats that are not finite (or S <= 0)
 * invalidate the request like a non-finite logit (SV_ST_NONFINITE).  The
 * stats must belong to these draft rows at this temperature; the library
 * cannot check that.  out_p and out_Z as for spec_verify_diag (either may be
 * NULL); gamma == 0 needs no draft_stats.
 */
int spec_verify_cached(const void* target_logits, const void* draft_logits,
                       const int32_t* draft_tokens, const float* draft_stats,
                       const float* u_accept, const float* u_resample, const float* temperature,
                       int B, int gamma, int V, int dtype, int32_t* out_tokens,
                       int32_t* out_num_accepted, float* out_p, float* out_Z, void* workspace,
                       size_t workspace_bytes, int32_t* dev_status, void* stream);

/* Size of the built-in scratch of spec_verify_noalloc: 16 MiB.  Every GPU that
 * loads this library holds this much device memory until the process exits. */
#define SV_NOALLOC_MAX_WORKSPACE (16u << 20)

/*
 * spec_verify for callers that cannot allocate device memory.  (The pages
 * have no counterpart: this is a service of the library, not part of the
 * method.)  Some callers run where allocating is not allowed or not
 * possible: a plugin inside a host framework that owns all device memory
 * and hands out no allocator, or a latency-critical loop that must not pay
 * for cudaMalloc's implicit device synchronisation.  This entry point takes
 * the same inputs and outputs as spec_verify but no workspace: it uses a
 * scratch array built into the library (SV_NOALLOC_MAX_WORKSPACE bytes per
 * device) and calls no allocating routine.
 *   - Sizes whose sv_workspace_bytes(B, gamma, V) exceeds
 *     SV_NOALLOC_MAX_WORKSPACE return SV_ERR_WORKSPACE; nothing is launched.
 *   - Every call looks up the scratch array's device address
 *     (cudaGetSymbolAddress) with the calling thread's device current; the
 *     address is not cached, so a context created anew after
 *     cudaDeviceReset is served correctly.  The first call on a device also
 *     loads the library's kernels into that context: make it before any
 *     stream capture.
 *   - Each call resets the scratch's 64-byte control block on `stream`
 *     before its launches; every other byte of the scratch that a call reads
 *     is written earlier in the same call.
 *   - All calls on a device share the one array: calls that may overlap on
 *     the GPU (different streams, or different host threads) race and must
 *     be serialised by the caller.
 */
int spec_verify_noalloc(const void* target_logits, const void* draft_logits,
                        const int32_t* draft_tokens, const float* u_accept,
                        const float* u_resample, const float* temperature, int B,
                        int gamma, int V, int dtype, int32_t* out_tokens,
                        int32_t* out_num_accepted, int32_t* dev_status, void* stream);

/*
 * Process-wide tuning override for benchmarking sweeps (0 = automatic):
 * elements per phase-1 chunk (rounded up to a multiple of 64, capped at half
 * a reduce slot of logits).  Not thread-safe; set it before issuing calls.
 * Returns SV_OK.
 */
int sv_set_tuning(int chunk_elems);

/*
 * Process-wide choice of the kernels that follow the reduce in a sampling
 * call (spec_verify, spec_verify_diag, spec_verify_cached, spec_verify_noalloc),
 * for tests and benchmarking: 0 (the default) picks the fused tail when the
 * batch leaves at least two SMs per request (B * 2 <= SMs) and the
 * decide / residual / draw kernels otherwise; 1 forces the three kernels;
 * 2 forces the fused tail (one kernel, one cluster of up to 8 CTAs per
 * request); 3 runs the whole call as one kernel: one cluster per request
 * streams the request's rows, then decides and draws like the fused tail,
 * its second pass reading the rows the cluster has just streamed (mode 3
 * also runs greedy calls, spec_verify_greedy, as one kernel; the other
 * modes leave them as they are).  All compute the same decision and draw
 * the token by the same rule.  Not thread-safe, like sv_set_tuning().
 * Returns SV_OK, or SV_ERR_INVALID_ARG for a mode outside [0, 3].
 */
int sv_set_tail(int mode);

/*
 * Profiling aid: the next calls record the caller's CUDA events (cudaEvent_t
 * handles, created on the device the calls run on) on their stream: events[0]
 * before the first kernel and events[j] after the j-th (sampling runs four
 * kernels: reduce, decide, residual, draw, or two with the fused tail: reduce
 * and the fused kernel; greedy runs two), for j < n.
 * n = 0 turns it off.  n outside [0, 5] or a NULL handle: SV_ERR_INVALID_ARG.
 * Not thread-safe, like sv_set_tuning().
 */
int sv_set_stage_events(void* const* events, int n);

/*
 * Failure-handling test aid: while enabled, the next calls' streaming kernel
 * withholds one of its shared-memory slots (block 0 never fills its first
 * slot), so the waits on that slot run out after their one-second limit: the
 * call reports SV_ST_TIMEOUT in *dev_status, its results are void, and the
 * context stays usable for the calls after it.  No fault, trap or endless
 * wait is involved.  Not thread-safe, like sv_set_tuning().  Returns SV_OK.
 */
int sv_test_withhold_slot(int enable);

/* Human-readable name of a host return code. */
const char* sv_error_string(int code);

/* Library version, major * 100 + minor. */
int sv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
