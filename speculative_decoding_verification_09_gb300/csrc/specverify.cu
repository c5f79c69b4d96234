// specverify.cu -- sm_103a kernels and C ABI for the speculative-decoding
// verification step (see include/specverify.h for the operation, layouts and
// error behaviour).
//
// Method (Speculative Decoding overview page, "猜想解码 (Speculative Decoding)
// 全景": 考点2 acceptance probability and residual distribution, 第二章 the
// acceptance formula, 第三章 the NumPy operator; deferred-speculation page,
// scheduler section "动态推迟投机验证调度器设计": tempered softmax, accept in
// draft order, stop at the first rejection, index-order inverse CDF).
//
// GPU structure: four kernels in stream order per call, each launched with
// programmatic stream serialisation (its CTAs are placed early and wait on
// the device for the previous kernel's memory):
//   reduce   one CTA per SM, each streaming a contiguous range of row chunks
//            (chunk c of target row i and draft row i of request b; or two
//            target chunks when no draft rows are streamed), then units of
//            the last requests' chunks claimed from a counter, from HBM into a
//            ring of shared-memory slots with TMA bulk copies (cp.async.bulk,
//            completion counted on an mbarrier) issued by one producer lane;
//            consumer warps reduce each slot from registers and publish one
//            partial per warp: (max, sum of 2^((l - max) * log2e / T)) of the
//            target and draft shares, or (max, lowest index, NaN seen) for
//            greedy verification.
//   decide   one CTA per request: every row's partials combined (maxima, sums
//            as float pairs), then per position the acceptance test in
//            float-pair arithmetic, the first rejection k, all outputs but
//            token k, and a decision record (row k's normalisers) for the draw.
//   residual one CTA per SM over the phase-2 chunks of the rows token k is
//            drawn from (residual of row k, or target row gamma for the
//            bonus): the mass of each warp's contiguous sub-range.
//   draw     one CTA per request: the sub-range where the running mass
//            crosses u * Z, scanned in index order: token k.
// Batches that leave at least two SMs per request replace decide, residual
// and draw by one kernel, finish, with a cluster of CTAs per request (the
// decision in every CTA, segment masses shared through distributed shared
// memory, the token found by the CTA owning the crossing segment).
// Greedy verification runs reduce (chunk argmax) and decide only; draft
// sampling runs reduce (contiguous warp shares) and sample (one CTA per draft
// row: the crossing partial's span, scanned in index order).  On request
// (sv_set_tail(3)) a sampling or greedy call runs as one kernel, onecall:
// each request's cluster streams the request's rows through the reduce's
// ring, then decides (and draws, like finish) from rows still in L2.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "specverify.h"

namespace {

// ------------------------------------------------------------ constants

// Streaming kernels: 15 warps, the producer (warp 0) and NCW consumer warps in
// NGRP groups that take the ring's slots in turn (slot sequence number mod
// NGRP), so the groups' phases (loading, exponentials, reductions) need not
// coincide.  Warp w runs on SM sub-partition w % 4; both groups have warps on
// every sub-partition.
constexpr int NCW = 14;
constexpr int NTHR = 32 * (NCW + 1);
// Ring geometry of a streaming kernel: NG consumer groups of GW warps, NS
// slots (NS / NG per group), HALF bytes per row chunk (a slot holds a target
// and a draft chunk).
template <int NG_, int NS_, int HALF_>
struct Geo {
  static constexpr int NG = NG_;
  static constexpr int GW = NCW / NG_;
  static constexpr int NS = NS_;
  static constexpr int HALF = HALF_;
  static constexpr int SLOT = 2 * HALF_;
  // body vectors of a row chunk per consumer thread: vector j belongs to
  // thread j mod (GW * 32) of the group
  static constexpr int MAXV = (HALF_ / 16 + GW * 32 - 1) / (GW * 32);
  // a warp's contiguous run of a segment's vectors fits its registers
  static_assert(32 * MAXV >= (HALF_ / 16 + GW - 1) / GW, "warp run");
  // Every use of a slot must be consumed by the same group: a group waits
  // for use u of a slot only after consuming use u - 1, which is what makes
  // the mbarrier's phase parity unambiguous.
  static_assert(NCW % NG_ == 0 && NS_ % NG_ == 0, "groups");
};
using GeoReduce = Geo<2, 4, 24576>;    // phase 1: two groups of 7 warps, 4 slots of 48 KB
using GeoResidual = Geo<1, 2, 49152>;  // phase 2: one group of 14 warps, 2 slots of 96 KB
constexpr int CH1_MIN = 1024;          // smallest phase-1 chunk (elements)
constexpr int CH2_F32 = GeoResidual::HALF / 4;  // phase-2 chunk for fp32 (the workspace bound)
constexpr unsigned SUSPEND_HINT_NS = 1000000u;  // a waiting warp sleeps until the phase completes
constexpr int SMS_CAP = 256;           // the chunk heuristic assumes at most this many SMs
constexpr int MAXR = SV_MAX_GAMMA + 1;
constexpr int DECIDE_WARPS = 16;       // decide: warps per request
constexpr int DECIDE_WARPS_SMALL = 4;  // ... when R <= 4: a warp for every row, more CTAs per SM
constexpr int DRAW_WARPS = 4;          // draw: warps per request
constexpr int SAMPLE_WARPS = 4;        // draft sampling: warps per draft row
constexpr float LOG2E_F = 1.4426950408889634f;
constexpr double LOG2E_D = 1.4426950408889634;
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;  // one second

// ------------------------------------------------------------ workspace

struct Ctrl {                 // 64 bytes at the start of the workspace
  // both 0 between calls (the ready state); state is 1 while a call runs,
  // claims counts the reduce's claims of pool units (reset by the call's last kernel)
  unsigned long long state, claims;
  unsigned long long pad[6];  // pad[0]: the residual kernel's chunk-claim counter;
                              // pad[1]: pool units the reduce's CTAs took (0 between calls);
                              // pad[2]: CTAs of the one-kernel path done (0 between calls)
};
struct Partial {              // per (request, position, chunk, consumer warp)
  float a, b, c, d;           // sampling: m_t, s_t, m_d, s_d; greedy: value, index, nan, 0
};
// Decision record of a request (written by decide, read by residual and draw).
enum { MODE_INVALID = 0, MODE_REJECT = 1, MODE_BONUS = 2, MODE_TARGET = 3 };
struct Record {               // per request, 48 bytes
  int k, mode;
  float mt, kf;               // max logit of target row k; log2(e)/T in fp32
  float ist_hi, ist_lo;       // 1/S_t of row k as an unevaluated float pair
  float c0_hi, c0_lo;         // log2(P_d/P_t) = (l_d - l_t) * kf + c0 on row k, c0 as a pair
  int pad[4];
};
struct Mass {                 // per (request, phase-2 chunk, consumer warp)
  float hi, lo;               // the sub-range's mass as an unevaluated float pair
};
// A row's decision inputs, in shared memory of the decide kernel.
struct RowStat {
  float mt, md;               // row maxima
  float St_h, St_l, Sd_h, Sd_l;  // sum of 2^((l - max) * kf) over the row, float pairs
  int bad, amax;              // SV_ST_* bits, greedy argmax
};
static_assert(sizeof(Ctrl) == 64 && sizeof(Partial) == 16 && sizeof(Record) == 48 &&
                  sizeof(Mass) == 8,
              "layout");

struct Layout {
  size_t ctrl, part, rec, mass, total;
  int nch1_max, nch2_max;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

Layout make_layout(int B, int gamma, int V) {
  Layout L;
  const size_t R = size_t(gamma) + 1;
  // the chunk heuristic below never uses more chunks than this (it assumes
  // at most SMS_CAP SMs)
  const long long units = (long long)B * (long long)R;
  const long long by_bytes = (V + GeoReduce::HALF / 4 - 1) / (GeoReduce::HALF / 4);
  const long long by_tasks = units > 0 ? (8LL * SMS_CAP + units - 1) / units : 1;
  L.nch1_max = int(min((long long)(V + CH1_MIN - 1) / CH1_MIN, max(by_bytes, by_tasks)));
  L.nch2_max = (V + CH2_F32 - 1) / CH2_F32;
  L.ctrl = 0;
  L.part = align256(sizeof(Ctrl));
  L.rec = L.part + align256(size_t(B) * R * L.nch1_max * GeoReduce::GW * sizeof(Partial));
  L.mass = L.rec + align256(size_t(B) * sizeof(Record));
  L.total = L.mass + align256(size_t(B) * L.nch2_max * GeoResidual::GW * sizeof(Mass));
  return L;
}

// --------------------------------------------------------- kernel params

struct Params {
  const unsigned char* Lt;
  const unsigned char* Ld;
  const int32_t* x;
  const float* u_acc;
  const float* u_res;
  const float* temp;
  int B, gamma, V, R;
  int gs;                     // draft rows streamed by the reduce per request: gamma, or 0
                              // when the draft rows' normalisers are given (dstats)
  const float* dstats;        // cached draft normalisers [B][gamma][2] (m, S), or null
  int ch1, nch1, ch2, nch2, sub;
  int np1;                    // phase-1 partials per row: one per (chunk, consumer warp)
  long long tasks;            // phase-1 chunks, B * R * nch1
  int32_t* out_tokens;
  int32_t* out_n;
  float* out_p;
  float* out_Z;
  float* out_stats;           // draft sampling: row normalisers (m, S)
  int withhold_slot;          // failure-handling test: CTA 0 never fills its first reduce slot
  int reduce_grid;            // CTAs of the call's reduce kernel
  int col, ncols;             // draft sampling: row i of request b goes to column col + i of ncols
  int32_t* status;
  Ctrl* ctrl;
  Partial* part;
  Record* rec;
  Mass* mass;
};

// -------------------------------------------------------- device helpers

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed pairs of fp32 (one 64-bit register pair), for the f32x2 instructions.
__device__ __forceinline__ unsigned long long pk2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long sub2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
// warp-wide maximum, NaN if any lane holds NaN
__device__ __forceinline__ float warp_max_nan(float v) {
  float r;
  asm volatile("redux.sync.max.NaN.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
// warp-wide maximum of the lanes' non-NaN values (-inf if there are none)
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ uint32_t bmax_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------- mbarrier and TMA

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(unsigned long long* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(SUSPEND_HINT_NS)
      : "memory");
  return ok != 0;
}
// One-dimensional bulk copy global -> shared, completion counted on `bar`.
// Source, destination and size must be multiples of 16 bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes,
                                         unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Programmatic dependent launch: the next kernel of the call may be launched
// (and run what does not read this kernel's outputs) before this one ends;
// it waits for this kernel's completion, with its memory visible, before
// reading any of it.
__device__ __forceinline__ void allow_next_kernel() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_previous_kernel() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void set_status(const Params& P, int bits) {
  if (bits && P.status) atomicOr(P.status, bits);
}

// Units of the reduce's claimed pool (see reduce_split).
__device__ long long reduce_pool_units(const Params& P, long long nb);

// The control block's ready state, written by the last kernel of a call
// (the reduce of this call has completed; the next call's reduce reads it
// only after this kernel has completed).  The pool units the reduce's CTAs
// took must add up to the pool: a claim counter that did not start the call
// at 0 would have skipped units, and is reported like a workspace that was
// not in its ready state.
__device__ __forceinline__ void ready_for_next_call(const Params& P) {
  if (P.ctrl->pad[1] != (unsigned long long)reduce_pool_units(P, P.reduce_grid))
    set_status(P, SV_ST_WORKSPACE);
  P.ctrl->pad[1] = 0ull;
  P.ctrl->state = 0ull;
  P.ctrl->claims = 0ull;
}

// Bounded wait for phase `parity` of an mbarrier (the reduce kernel's waits are
// all within one CTA): false once the CTA gave up, or after one second, which
// records SV_ST_TIMEOUT and makes the CTA's other waiters give up too.
__device__ bool mbar_wait(unsigned long long* bar, unsigned parity, const Params& P,
                          volatile int* cta_abort) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (;;) {
    if (mbar_try(bar, parity)) return true;
    if (*cta_abort) return false;
    if (globaltimer() - t0 > WAIT_LIMIT_NS) {
      *cta_abort = 1;
      set_status(P, SV_ST_TIMEOUT);
      return false;
    }
  }
}

// ------------------------------------------------- element access

template <int DT>
struct Elem;
template <>
struct Elem<SV_F32> {
  static constexpr int ES = 4, VEC = 4;
  __device__ static float load(const unsigned char* base, long long idx) {
    return __ldg(reinterpret_cast<const float*>(base) + idx);
  }
  __device__ static float lds(const unsigned char* base, int idx) {
    return reinterpret_cast<const float*>(base)[idx];
  }
  __device__ static void sts(unsigned char* base, int idx, float v) {
    reinterpret_cast<float*>(base)[idx] = v;
  }
  // the VEC elements from element p of a shared-memory body, p >= 0 (any
  // alignment), as a vector
  __device__ static uint4 gather_shifted(const unsigned char* body, int p) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(body) + p;
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  // running max over vectors; packed state is the float's bits
  static constexpr uint32_t MAX_INIT = 0xff800000u;
  __device__ static uint32_t vmax_acc(uint32_t acc, const uint4& v) {
    float m = fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                       fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
    return __float_as_uint(fmax_nan(__uint_as_float(acc), m));
  }
  __device__ static float vmax_final(uint32_t acc) { return __uint_as_float(acc); }
  __device__ static uint32_t wmax(uint32_t a, uint32_t b) {
    return __float_as_uint(fmax_nan(__uint_as_float(a), __uint_as_float(b)));
  }
  __device__ static float vmax(const uint4& v) {
    return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                    fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
  static constexpr uint32_t NEG_INF_WORD = 0xff800000u;
  static constexpr int PAIRS = 2;  // fp32 pairs in a 16-byte vector
  __device__ static unsigned long long pair(const uint4& v, int q) {
    return q == 0 ? pk2(__uint_as_float(v.x), __uint_as_float(v.y))
                  : pk2(__uint_as_float(v.z), __uint_as_float(v.w));
  }
};
template <>
struct Elem<SV_BF16> {
  static constexpr int ES = 2, VEC = 8;
  __device__ static float load(const unsigned char* base, long long idx) {
    return __uint_as_float(uint32_t(__ldg(reinterpret_cast<const unsigned short*>(base) + idx))
                           << 16);
  }
  __device__ static float lds(const unsigned char* base, int idx) {
    return __uint_as_float(uint32_t(reinterpret_cast<const unsigned short*>(base)[idx]) << 16);
  }
  __device__ static void sts(unsigned char* base, int idx, float v) {  // v holds a bf16 value
    reinterpret_cast<unsigned short*>(base)[idx] = (unsigned short)(__float_as_uint(v) >> 16);
  }
  // the VEC elements from element p of a shared-memory body, p >= 0 (any
  // alignment), as a vector: four words at an even p, else five words
  // (elements p - 1 .. p + 8, the last one unused) funnel-shifted by 16 bits
  __device__ static uint4 gather_shifted(const unsigned char* body, int p) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(body) + (p >> 1);
    if ((p & 1) == 0) return make_uint4(w[0], w[1], w[2], w[3]);
    const uint32_t* v = w;  // word p >> 1 holds elements p - 1 and p
    return make_uint4(__funnelshift_r(v[0], v[1], 16), __funnelshift_r(v[1], v[2], 16),
                      __funnelshift_r(v[2], v[3], 16), __funnelshift_r(v[3], v[4], 16));
  }
  __device__ static void unpack(const uint4& v, float* f) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z); f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
  }
  // running max over vectors as a packed bf16 pair (both halves -inf at start)
  static constexpr uint32_t MAX_INIT = 0xff80ff80u;
  __device__ static uint32_t vmax_acc(uint32_t acc, const uint4& v) {
    return bmax_nan(acc, bmax_nan(bmax_nan(v.x, v.y), bmax_nan(v.z, v.w)));
  }
  __device__ static float vmax_final(uint32_t acc) { return fmax_nan(bf_lo(acc), bf_hi(acc)); }
  __device__ static uint32_t wmax(uint32_t a, uint32_t b) { return bmax_nan(a, b); }
  __device__ static float vmax(const uint4& v) {
    return vmax_final(bmax_nan(bmax_nan(v.x, v.y), bmax_nan(v.z, v.w)));
  }
  static constexpr uint32_t NEG_INF_WORD = 0xff80ff80u;
  static constexpr int PAIRS = 4;
  __device__ static unsigned long long pair(const uint4& v, int q) {
    const uint32_t w = q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
    return pk2(bf_lo(w), bf_hi(w));
  }
};

// ------------------------------------------------- reductions and merges

// Argmax triples (value, lowest index, NaN seen).
__device__ __forceinline__ void am_merge(float& best, int& bi, int& nan, float b2, int i2, int n2) {
  if (b2 > best || (b2 == best && i2 < bi)) { best = b2; bi = i2; }
  nan |= n2;
}
// Error-free sum of two floats (Knuth's two-sum): s + err == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& err) {
  s = a + b;
  const float bb = s - a;
  err = (a - (s - bb)) + (b - bb);
}
// Running sum as an unevaluated float pair (hi, lo): add x and renormalise.
__device__ __forceinline__ void ff_add(float& hi, float& lo, float x) {
  float s, e;
  two_sum(hi, x, s, e);
  const float t = lo + e;
  hi = s + t;
  lo = t - (hi - s);
}
// Sum of two float pairs.
__device__ __forceinline__ void ff_add2(float& hi, float& lo, float h2, float l2) {
  float s, e;
  two_sum(hi, h2, s, e);
  const float t = lo + l2 + e;
  hi = s + t;
  lo = t - (hi - s);
}
// Warp-wide sum of float pairs (about 48 significant bits), valid in every lane.
__device__ __forceinline__ void warp_sum_ff(float& hi, float& lo) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
    ff_add2(hi, lo, h2, l2);
  }
}
// Inclusive warp prefix sum of float pairs, lane order.
__device__ __forceinline__ void warp_scan_ff(float& hi, float& lo, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float h2 = __shfl_up_sync(0xffffffffu, hi, o);
    const float l2 = __shfl_up_sync(0xffffffffu, lo, o);
    if (lane >= o) ff_add2(hi, lo, h2, l2);
  }
}
__device__ __forceinline__ double ff_val(float hi, float lo) { return double(hi) + double(lo); }

// Float pairs (hi, lo), hi + lo the value: comparisons and the product with a
// float, in fp32 arithmetic (the fp64 units are slow on this part).
struct FF {
  float h, l;
};
__device__ __forceinline__ FF ff(float h, float l = 0.f) { return FF{h, l}; }
__device__ __forceinline__ FF operator+(FF a, FF b) {
  ff_add2(a.h, a.l, b.h, b.l);
  return a;
}
__device__ __forceinline__ FF operator-(FF a, FF b) {
  ff_add2(a.h, a.l, -b.h, -b.l);
  return a;
}
__device__ __forceinline__ bool ff_gt(FF a, FF b) {  // a > b
  const FF d = a - b;
  return d.h > 0.f || (d.h == 0.f && d.l > 0.f);
}
__device__ __forceinline__ bool ff_pos(FF a) { return a.h > 0.f || (a.h == 0.f && a.l > 0.f); }
__device__ __forceinline__ FF ff_mul(float u, FF z) {  // u * z
  const float p = u * z.h;
  const float e = fmaf(u, z.h, -p);  // the product's rounding error, exactly
  const float t = e + u * z.l;
  FF r;
  r.h = p + t;
  r.l = t - (r.h - p);
  return r;
}
__device__ __forceinline__ FF ff_shfl(FF a, int src) {
  return FF{__shfl_sync(0xffffffffu, a.h, src), __shfl_sync(0xffffffffu, a.l, src)};
}

// a - b exactly, as a float pair
__device__ __forceinline__ FF ff_diff(float a, float b) {
  FF r;
  two_sum(a, -b, r.h, r.l);
  return r;
}
// a * b for a float pair a and a float b, as a float pair (fma gives the
// rounding error of the leading product exactly)
__device__ __forceinline__ FF ff_mulf(FF a, float b) {
  const float p = a.h * b;
  const float e = fmaf(a.h, b, -p) + a.l * b;
  FF r;
  two_sum(p, e, r.h, r.l);
  return r;
}
// a * b for float pairs
__device__ __forceinline__ FF ff_mul2(FF a, FF b) {
  const float p = a.h * b.h;
  const float e = fmaf(a.h, b.h, -p) + (a.h * b.l + a.l * b.h);
  FF r;
  two_sum(p, e, r.h, r.l);
  return r;
}
// a / b for float pairs (one correction step of the float quotient)
__device__ __forceinline__ FF ff_div(FF a, FF b) {
  const float q = __fdiv_rn(a.h, b.h);
  const float rem = fmaf(-q, b.h, a.h) + (a.l - q * b.l);
  FF r;
  two_sum(q, __fdiv_rn(rem, b.h), r.h, r.l);
  return r;
}
// log2(e) / T as a float pair (log2(e) split into a float and its remainder)
__device__ __forceinline__ FF ff_log2e_over(float T) {
  constexpr float L_HI = 1.44269502162933349609375f;        // log2(e) rounded to a float
  constexpr float L_LO = 1.925963033500011e-08f;            // log2(e) - L_HI
  const float q = __fdiv_rn(L_HI, T);
  const float rem = fmaf(-q, T, L_HI) + L_LO;
  FF r;
  two_sum(q, __fdiv_rn(rem, T), r.h, r.l);
  return r;
}
// 2^e for a float pair e: 2^n * exp2f(f) with n = rint(e), f = e - n
// (|f| <= 1/2 + tiny), the scaling saturating to 0 or +inf like the exact value
__device__ __forceinline__ float ff_exp2(FF e) {
  if (!(e.h == e.h)) return e.h;
  if (e.h > 300.f) return INFINITY;
  if (e.h < -300.f) return 0.f;
  const float n = rintf(e.h);
  return ldexpf(exp2f((e.h - n) + e.l), int(n));
}


// 2^x in fp64 (used only for the rare P_d underflow case of the acceptance
// test, where the oracle's fp64 rounding decides): x = n + f with n = rint(x) and
// |f| <= 1/2, e^(f ln 2) by its Taylor series to degree 11 (truncation below
// 1e-14 relative), scaled by 2^n built in the exponent field in two factors.
// Out-of-range x saturate to 0 or +inf; NaN stays NaN.
__device__ __forceinline__ double exp2_d(double x) {
  if (!(x > -1075.0)) return x != x ? x : 0.0;
  if (x > 1024.0) return INFINITY;
  const double n = rint(x);
  const double t = (x - n) * 0.69314718055994530942;
  double p = 1.0 / 39916800.0;                    // 1/11!
  p = fma(p, t, 1.0 / 3628800.0);
  p = fma(p, t, 1.0 / 362880.0);
  p = fma(p, t, 1.0 / 40320.0);
  p = fma(p, t, 1.0 / 5040.0);
  p = fma(p, t, 1.0 / 720.0);
  p = fma(p, t, 1.0 / 120.0);
  p = fma(p, t, 1.0 / 24.0);
  p = fma(p, t, 1.0 / 6.0);
  p = fma(p, t, 0.5);
  p = fma(p, t, 1.0);
  p = fma(p, t, 1.0);
  const int ni = int(n);
  const int n1 = ni / 2, n2 = ni - n1;
  return p * __longlong_as_double((long long)(n1 + 1023) << 52) *
         __longlong_as_double((long long)(n2 + 1023) << 52);
}

__device__ __forceinline__ bool row_ok(float m, double S) {
  return (m > -INFINITY) && (m < INFINITY) && (S > 0.0) && (S < INFINITY);
}
__device__ __forceinline__ bool row_ok_ff(float m, float S_hi) {
  return (m > -INFINITY) && (m < INFINITY) && (S_hi > 0.f) && (S_hi < INFINITY);
}

// ------------------------------------------------ reduce: slots

// One slot's chunk, written by the producer.
struct alignas(16) Desc {
  int end;                    // 1: no more chunks for this CTA
  int b, i, c;                // request, row position, chunk
  int e0, n;                  // element range of the chunk within the row
  int head_t, nb_t;           // target: leading single elements, aligned body elements in smem
  int head_d, nb_d;           // draft likewise (or the second chunk of a pair)
  float kf;                   // sampling: log2(e) / T of the request
  float kf2;                  // pair: log2(e) / T of the second chunk's request
  int pair;                   // reduce without draft rows: the slot's second half holds
                              // the next target chunk (not a draft chunk)
  int n2;                     // pair: elements of the second chunk
  int pad[2];
  Record rec;                 // residual: the request's decision record (bulk-copied)
};
static_assert(offsetof(Desc, rec) % 16 == 0 && sizeof(Record) % 16 == 0, "record copy");
// Shared-memory control block of the streaming kernels (after the slots).
template <class G>
struct SmemCtl {
  unsigned long long full[G::NS], empty[G::NS];
  Desc desc[G::NS];
  int abort;
};
template <class G>
constexpr size_t smem_bytes() {
  return size_t(G::NS) * G::SLOT + sizeof(SmemCtl<G>);
}
static_assert(smem_bytes<GeoReduce>() <= 227 * 1024 && smem_bytes<GeoResidual>() <= 227 * 1024,
              "shared memory budget");


// ------------------------------------------------ phase 1: consumer reductions

// Group of consumer warp w (1..NCW) and its index in the group.  With two
// groups: group 0 is warps 1-3 and 8-11, group 1 warps 4-7 and 12-14, so
// both have warps on every SM sub-partition.
template <class G>
__device__ __forceinline__ void consumer_role(int w, int& grp, int& wg) {
  if (G::NG == 1) {
    grp = 0;
    wg = w - 1;
  } else {
    static_assert(G::NG <= 2, "role map");
    grp = (w >> 2) & 1;
    wg = grp == 0 ? (w < 4 ? w - 1 : w - 5) : (w < 8 ? w - 4 : w - 8);
  }
}

// sum over pairs of 2^((f - m) * kf), with packed fp32x2 arithmetic
template <int DT>
__device__ __forceinline__ float vec_expsum(const uint4& v, unsigned long long mm,
                                            unsigned long long kk) {
  using E = Elem<DT>;
  unsigned long long acc = pk2(0.f, 0.f);
#pragma unroll
  for (int q = 0; q < E::PAIRS; ++q) {
    float a, b;
    upk2(mul2(sub2(E::pair(v, q), mm), kk), a, b);
    acc = add2(acc, pk2(ex2(a), ex2(b)));
  }
  float a, b;
  upk2(acc, a, b);
  return a + b;
}

// A consumer warp's share of one slot, in one of two maps of a segment's nv
// body vectors to the group's threads:
//   interleaved (CONTIG false): vector j to thread j mod (GW * 32); warp 0
//     also takes the unaligned head and tail elements;
//   contiguous (CONTIG true): warp wg takes the run [wg * pw, (wg + 1) * pw)
//     with pw = ceil(nv / GW) (lane l its vectors l, l + 32, ...), so every
//     warp's partial is the sum over a contiguous span of the row, which the
//     draft sampler searches directly; warp 0 takes the head, warp GW - 1
//     the tail.
// The vectors are loaded from shared memory into registers (MAXV per segment
// per thread), plus the chunk fields the reduction needs.  Both segments
// (target and draft, or a pair of target chunks) are loaded together.
template <int MAXV>
struct Share {
  uint4 t[MAXV], d[MAXV];
  int b, i, c, e0, n, head_t, nb_t, head_d, nb_d;
  float kf, kf2;
  int pair, n2;
};
template <int DT, class G, bool CONTIG, bool PAIRS>
__device__ __forceinline__ void load_share(const Desc& d, const unsigned char* slot, bool has_d,
                                           int wg, int lane, Share<G::MAXV>& sh) {
  using E = Elem<DT>;
  constexpr int MAXV = G::MAXV, HALF = G::HALF, GW = G::GW;
  const int nvt = d.nb_t / E::VEC, nvd = has_d ? d.nb_d / E::VEC : 0;
  const uint4 neg = make_uint4(E::NEG_INF_WORD, E::NEG_INF_WORD, E::NEG_INF_WORD, E::NEG_INF_WORD);
  if (CONTIG) {
    const int pwt = (nvt + GW - 1) / GW, pwd = (nvd + GW - 1) / GW;
    const int jt0 = wg * pwt, jt1 = min(nvt, jt0 + pwt);
    const int jd0 = wg * pwd, jd1 = min(nvd, jd0 + pwd);
#pragma unroll
    for (int u = 0; u < MAXV; ++u) {
      const int jt = jt0 + lane + 32 * u, jd = jd0 + lane + 32 * u;
      sh.t[u] = jt < jt1 ? reinterpret_cast<const uint4*>(slot)[jt] : neg;
      sh.d[u] = jd < jd1 ? reinterpret_cast<const uint4*>(slot + HALF)[jd] : neg;
    }
  } else {
    const int tid = wg * 32 + lane;
#pragma unroll
    for (int u = 0; u < MAXV; ++u) {
      const int j = tid + u * GW * 32;
      sh.t[u] = j < nvt ? reinterpret_cast<const uint4*>(slot)[j] : neg;
      sh.d[u] = j < nvd ? reinterpret_cast<const uint4*>(slot + HALF)[j] : neg;
    }
  }
  sh.b = d.b; sh.i = d.i; sh.c = d.c; sh.e0 = d.e0; sh.n = d.n;
  sh.head_t = d.head_t; sh.nb_t = d.nb_t; sh.head_d = d.head_d; sh.nb_d = d.nb_d;
  sh.kf = d.kf;
  if (PAIRS) {
    sh.kf2 = d.kf2;
    sh.pair = d.pair;
    sh.n2 = d.n2;
  }
}

// The chunk after chunk c of row (b, i) in the reduce's task order.
__device__ __forceinline__ void next_chunk(const Params& P, int& b, int& i, int& c) {
  if (++c == P.nch1) {
    c = 0;
    if (++i == P.R) { i = 0; ++b; }
  }
}

// This warp's (max, sum 2^((l-max)*kf)) over its share of the slot's two
// segments: the target chunk (b, i, c), and the second segment: the draft
// chunk of the same span (PAIRS false, rows i < gs), or the next target
// chunk (PAIRS true, when the slot holds a pair), with its own element count
// and temperature.  The body vectors are in `sh`; consumer warp 0 also takes
// the few unaligned head elements, and the tail elements go to warp GW - 1
// (contiguous map) or warp 0 (interleaved map), from global memory.  Each
// lane sums relative to its own maximum; the lanes' sums are rescaled to the
// warp's.
template <int DT, int MAXV, int GW, bool PAIRS, bool CONTIG>
__device__ float4 reduce_share_ms(const Params& P, const Share<MAXV>& sh, int wg, int lane) {
  using E = Elem<DT>;
  const bool has_d = PAIRS ? sh.pair != 0 : sh.i < P.gs;
  const float kf_t = sh.kf, kf_d = PAIRS ? sh.kf2 : sh.kf;
  float ht = -INFINITY, tt = -INFINITY, hd = -INFINITY, td = -INFINITY;
  if (wg == 0 || wg == (CONTIG ? GW - 1 : 0)) {
    const int n_t = sh.n, n_d = PAIRS ? sh.n2 : sh.n;
    const unsigned char* gt =
        P.Lt + ((size_t(sh.b) * P.R + sh.i) * size_t(P.V) + sh.e0) * E::ES;
    const unsigned char* gd = nullptr;
    if (has_d) {
      if (PAIRS) {
        int b2 = sh.b, i2 = sh.i, c2 = sh.c;
        next_chunk(P, b2, i2, c2);
        gd = P.Lt + ((size_t(b2) * P.R + i2) * size_t(P.V) + size_t(c2) * P.ch1) * E::ES;
      } else {
        gd = P.Ld + ((size_t(sh.b) * P.gamma + sh.i) * size_t(P.V) + sh.e0) * E::ES;
      }
    }
    if (wg == 0) {
      if (lane < sh.head_t) ht = E::load(gt, lane);
      if (has_d && lane < sh.head_d) hd = E::load(gd, lane);
    }
    if (wg == (CONTIG ? GW - 1 : 0)) {
      if (lane < n_t - sh.head_t - sh.nb_t) tt = E::load(gt, sh.head_t + sh.nb_t + lane);
      if (has_d && lane < n_d - sh.head_d - sh.nb_d) td = E::load(gd, sh.head_d + sh.nb_d + lane);
    }
  }
  // lane maxima: balanced trees over the vectors
  uint32_t wt[MAXV], wd[MAXV];
#pragma unroll
  for (int u = 0; u < MAXV; ++u) {
    wt[u] = E::vmax_acc(E::MAX_INIT, sh.t[u]);
    wd[u] = E::vmax_acc(E::MAX_INIT, sh.d[u]);
  }
#pragma unroll
  for (int w = 1; w < MAXV; w *= 2)
#pragma unroll
    for (int u = 0; u + w < MAXV; u += 2 * w) {
      wt[u] = E::wmax(wt[u], wt[u + w]);
      wd[u] = E::wmax(wd[u], wd[u + w]);
    }
  const float mt = fmax_nan(E::vmax_final(wt[0]), fmax_nan(ht, tt));
  const float md = fmax_nan(E::vmax_final(wd[0]), fmax_nan(hd, td));
  // a NaN max makes the sum NaN; an all -inf share sums to 0
  const bool lt = mt > -INFINITY, ld = md > -INFINITY;
  const unsigned long long kkt = pk2(kf_t, kf_t), kkd = pk2(kf_d, kf_d);
  const unsigned long long mmt = pk2(mt, mt), mmd = pk2(md, md);
  float s_t = 0.f, s_d = 0.f;
#pragma unroll
  for (int u = 0; u < MAXV; ++u) {
    if (lt) s_t += vec_expsum<DT>(sh.t[u], mmt, kkt);
    if (ld) s_d += vec_expsum<DT>(sh.d[u], mmd, kkd);
  }
  if (lt) s_t += ex2((ht - mt) * kf_t) + ex2((tt - mt) * kf_t);
  if (ld) s_d += ex2((hd - md) * kf_d) + ex2((td - md) * kf_d);
  if (mt != mt) s_t = NAN;
  if (md != md) s_d = NAN;
  // rescale every lane's sum to the warp maximum and add them up
  const float Mt = warp_max_nan(mt), Md = warp_max_nan(md);
  if (lt && Mt > mt) s_t *= ex2((mt - Mt) * kf_t);
  if (ld && Md > md) s_d *= ex2((md - Md) * kf_d);
  if (Mt != Mt) s_t = NAN;
  if (Md != Md) s_d = NAN;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s_t += __shfl_xor_sync(0xffffffffu, s_t, o);
    s_d += __shfl_xor_sync(0xffffffffu, s_d, o);
  }
  return make_float4(Mt, s_t, Md, s_d);
}

// This warp's (largest value, lowest index among its occurrences, NaN seen)
// over its share of one target row chunk: body vectors `vec` (the slot's
// first or second segment, mapped to the threads as load_share maps it), the
// chunk at `gseg` starting at element e0 of its row with `head` single
// leading elements, nb body elements, n in all; indices are within the row.
template <int DT, class G, bool CONTIG>
__device__ float4 reduce_share_argmax(const uint4 (&vec)[G::MAXV], const unsigned char* gseg,
                                      int e0, int head, int nb, int n, int wg, int lane) {
  using E = Elem<DT>;
  constexpr int MAXV = G::MAXV;
  const int pw = (nb / E::VEC + G::GW - 1) / G::GW;
  float best = -INFINITY;
  int bi = INT_MAX, nan = 0;
  if (wg == 0 && lane < head) {
    const float l = E::load(gseg, lane);
    if (l != l) nan = 1;
    else if (l > best) { best = l; bi = e0 + lane; }
  }
#pragma unroll
  for (int u = 0; u < MAXV; ++u) {
    const int j = CONTIG ? wg * pw + lane + 32 * u : (wg * 32 + lane) + u * G::GW * 32;
    const uint4 v = vec[u];
    const float vm = E::vmax(v);
    if (vm != vm) {
      nan = 1;
    } else if (vm > best) {
      float f[E::VEC];
      E::unpack(v, f);
      int first = E::VEC - 1;
#pragma unroll
      for (int e = E::VEC - 1; e >= 0; --e)
        if (f[e] == vm) first = e;
      best = vm;
      bi = e0 + head + j * E::VEC + first;
    }
  }
  if (wg == (CONTIG ? G::GW - 1 : 0)) {
    const int t0 = head + nb;
    if (lane < n - t0) {
      const float l = E::load(gseg, t0 + lane);
      if (l != l) nan = 1;
      else if (l > best) { best = l; bi = e0 + t0 + lane; }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    const int n2 = __shfl_xor_sync(0xffffffffu, nan, o);
    am_merge(best, bi, nan, b2, i2, n2);
  }
  return make_float4(best, __int_as_float(bi), __int_as_float(nan), 0.f);
}

// Weight of one element of the final draw, up to the row's factor 1/S_t
// (applied once to the masses): e = 2^((l_t - m_t) * kf), the unnormalised
// P_t; after a rejection the residual max(0, P_t - P_d) = P_t * (1 - 2^delta)
// with delta = log2(P_d / P_t) = (l_d - l_t) * kf + c0, which keeps its
// relative precision where the rows nearly agree (no cancellation).  delta is
// clamped to <= 0 (weight 0, also for NaN); 1 - 2^delta is 1 - ex2(delta)
// where that loses little (delta < -1/2: ex2's relative error 2^-22 grows by
// at most 2^delta / (1 - 2^delta) < 2.5), else delta * p(delta) with p the
// degree-4 minimax fit (Remez exchange, relative error) of (1 - 2^delta) /
// delta on [-1/2, 0]: 1.3e-8 relative in exact arithmetic, 1.3e-7 as
// evaluated here in fp32 (fit_one_minus_exp2.py recomputes both).
// The exponent (l_t - m_t) * kf is formed as one fma with -m_t * kf rounded
// once per row: a common factor of all the row's weights.  weight() and
// vec_weights() perform the same fp32 operations per element.
constexpr float OMC1 = -0.69314717173667928f, OMC2 = -0.24022564279246794f,
                OMC3 = -0.055490406445877882f, OMC4 = -0.0095412810839257713f,
                OMC5 = -0.0011544522739422426f;
__device__ __forceinline__ float one_minus_exp2(float delta) {
  float p = OMC5;
  p = fmaf(p, delta, OMC4);
  p = fmaf(p, delta, OMC3);
  p = fmaf(p, delta, OMC2);
  p = fmaf(p, delta, OMC1);
  const float series = p * delta;
  const float alt = 1.f - ex2(delta);
  return delta < -0.5f ? alt : series;
}

__device__ __forceinline__ float weight(const Record& r, float lt, float ld) {
  const float et = ex2(fmaf(lt, r.kf, -(r.mt * r.kf)));
  if (r.mode == MODE_REJECT) {
    const float delta = fminf(fmaf(ld - lt, r.kf, r.c0_hi) + r.c0_lo, 0.f);  // log2(P_d / P_t)
    return et * one_minus_exp2(delta);
  }
  return et;
}

__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Weights of one 16-byte vector of target values `t` and draft values `dv`
// (TWO: after a rejection), added to the packed pair sum `acc`; the same
// operations as weight() on packed fp32 pairs.
template <int DT, bool TWO>
__device__ __forceinline__ void vec_weights_acc(const Record& r, const uint4& t, const uint4& dv,
                                                unsigned long long& acc) {
  using E = Elem<DT>;
  const float c1 = -(r.mt * r.kf);
  const unsigned long long cc = pk2(c1, c1), kk = pk2(r.kf, r.kf);
#pragma unroll
  for (int q = 0; q < E::PAIRS; ++q) {
    const unsigned long long lt = E::pair(t, q);
    float a, b;
    upk2(fma2(lt, kk, cc), a, b);
    const unsigned long long et = pk2(ex2(a), ex2(b));
    if (TWO) {
      const unsigned long long ch = pk2(r.c0_hi, r.c0_hi), cl = pk2(r.c0_lo, r.c0_lo);
      float d0, d1;
      upk2(add2(fma2(sub2(E::pair(dv, q), lt), kk, ch), cl), d0, d1);
      d0 = fminf(d0, 0.f);
      d1 = fminf(d1, 0.f);
      const unsigned long long dd = pk2(d0, d1);
      unsigned long long p = pk2(OMC5, OMC5);
      p = fma2(p, dd, pk2(OMC4, OMC4));
      p = fma2(p, dd, pk2(OMC3, OMC3));
      p = fma2(p, dd, pk2(OMC2, OMC2));
      p = fma2(p, dd, pk2(OMC1, OMC1));
      float s0, s1;
      upk2(mul2(p, dd), s0, s1);
      const float f0 = d0 < -0.5f ? 1.f - ex2(d0) : s0;
      const float f1 = d1 < -0.5f ? 1.f - ex2(d1) : s1;
      acc = add2(acc, mul2(et, pk2(f0, f1)));
    } else {
      acc = add2(acc, et);
    }
  }
}
// The same, summed on their own.
template <int DT>
__device__ __forceinline__ float vec_weights(const Record& r, const uint4& t, const uint4& dv,
                                             bool two) {
  unsigned long long acc = pk2(0.f, 0.f);
  if (two)
    vec_weights_acc<DT, true>(r, t, dv, acc);
  else
    vec_weights_acc<DT, false>(r, t, dv, acc);
  float a, b;
  upk2(acc, a, b);
  return a + b;
}

// ------------------------------------------------------------ reduce

// Split a chunk at `p` of d.n elements into single leading elements (up to the
// first 16-byte boundary) and an aligned body of whole vectors.
template <int DT>
__device__ __forceinline__ void split(const unsigned char* p, int n, int& head, int& nb) {
  using E = Elem<DT>;
  const int h = int(((16u - unsigned(reinterpret_cast<uintptr_t>(p) & 15u)) & 15u) / E::ES);
  head = h < n ? h : n;
  nb = ((n - head) / E::VEC) * E::VEC;
}

// The end marker for every consumer group, in slots seq .. seq + NGRP - 1.
template <class G>
__device__ void end_markers(const Params& P, SmemCtl<G>& C, long long seq) {
  for (int g = 0; g < G::NG; ++g, ++seq) {
    const int s = int(seq % G::NS);
    const unsigned use = unsigned(seq / G::NS);
    if (use > 0 && !mbar_wait(&C.empty[s], (use - 1) & 1u, P, &C.abort)) return;
    C.desc[s].end = 1;
    mbar_arrive(&C.full[s]);
  }
}

// Task weights: a chunk of a row that also streams its draft row weighs 2,
// a target-only chunk 1, so weight counts streamed bytes.  A request's tasks
// weigh w_req = nch1 * (R + gs): its first gs rows 2 * nch1 each, the rest
// nch1.  The smallest task whose weight before it reaches w, in closed form.
__device__ __forceinline__ long long task_at_weight(const Params& P, long long w) {
  const long long per_req = (long long)P.R * P.nch1;
  const long long w_req = (long long)P.nch1 * (P.R + P.gs);
  const long long w2 = 2LL * P.gs * P.nch1;  // weight of a request's two-row chunks
  const long long b = w / w_req, rem = w - b * w_req;
  const long long t_in = rem <= w2 ? (rem + 1) / 2 : P.gs * (long long)P.nch1 + (rem - w2);
  return b * per_req + t_in;
}

// Work split of the reduce.  The first (POOL_DIV - 1) / POOL_DIV of the
// weight is split statically: CTA x of nb streams the contiguous tasks from
// task_at_weight(ceil(Ws x / nb)) on, so every CTA starts with the same
// bytes.  The rest, tasks [ts, tasks) (the last requests' rows), is a pool
// of units of `unit` consecutive tasks that the CTAs claim one at a time
// from a counter in the control block once their static range is nearly
// done; CTAs whose copies are served faster take more units, so the grid
// ends together (a static split alone left the last CTA 2-18 us behind the
// median on the sampling workloads).
constexpr int POOL_DIV = 8;
struct Split {
  long long t0, t1;    // this CTA's static range
  long long ts;        // first pool task
  long long unit, nunits;
};
__device__ __forceinline__ Split reduce_split(const Params& P, long long x, long long nb) {
  const long long W = (long long)P.nch1 * (P.R + P.gs) * P.B;
  const long long Ws = W - W / POOL_DIV;
  Split sp;
  sp.t0 = task_at_weight(P, (Ws * x + nb - 1) / nb);
  sp.t1 = task_at_weight(P, (Ws * (x + 1) + nb - 1) / nb);
  sp.ts = task_at_weight(P, Ws);
  const long long pool = P.tasks - sp.ts;
  sp.unit = max(1LL, (pool + 4 * nb - 1) / (4 * nb));  // about four units per CTA
  sp.nunits = (pool + sp.unit - 1) / sp.unit;
  return sp;
}
__device__ long long reduce_pool_units(const Params& P, long long nb) {
  return reduce_split(P, 0, nb).nunits;
}

// Producer (one lane): the static range of chunks of its split, then the
// pool units it claims from *pool_ctr (the reduce: a counter in the control
// block, the count of units taken added to *taken_ctr; the one-kernel path:
// a counter in its cluster's first CTA), each in order, into the slot ring.  Chunk t is chunk
// t % nch1 of row t / nch1 (row = b * R + i).  A slot holds a target chunk
// and the same span of the draft row; where no draft rows are streamed
// (greedy verification, given draft normalisers, draft sampling) it holds
// two consecutive target chunks of one range instead (a pair), so every
// slot still carries up to two half-slots of logits.
template <int DT, bool GREEDY, bool PAIRS>
__device__ void producer(const Params& P, SmemCtl<GeoReduce>& C, unsigned char* slots,
                         const Split sp, unsigned long long* pool_ctr,
                         unsigned long long* taken_ctr) {
  using E = Elem<DT>;
  using G = GeoReduce;
  constexpr int NS = G::NS, SLOT = G::SLOT, HALF = G::HALF;
  long long t = sp.t0, tend = sp.t1;  // the range being streamed
  unsigned long long taken = 0;       // pool units this CTA took
  auto report = [&]() {
    if (taken && taken_ctr) atomicAdd(taken_ctr, taken);
  };
  // a claim is issued while the current range still has NS tasks to go, so
  // its round trip is hidden behind the slots in flight
  long long claimed = 0;
  bool pending = false;
  auto claim = [&]() {
    if (sp.nunits > 0) {
      claimed = (long long)atomicAdd(pool_ctr, 1ull);
      pending = true;
    }
  };
  int c = 0, b = 0, i = 0;
  float T = 1.f, T_next = 1.f;
  const unsigned char* trow = nullptr;
  const unsigned char* drow = nullptr;
  auto seek = [&](long long tt) {  // to chunk tt
    const long long row = tt / P.nch1;
    c = int(tt - row * P.nch1);
    b = int(row / P.R);
    i = int(row - (long long)b * P.R);
    T = (!GREEDY && b < P.B) ? __ldg(P.temp + b) : 1.f;  // b == B: an empty range at the end
    T_next = (!GREEDY && b + 1 < P.B) ? __ldg(P.temp + b + 1) : 1.f;
    trow = P.Lt + (size_t(b) * P.R + i) * size_t(P.V) * E::ES;
    drow = (!GREEDY && i < P.gs) ? P.Ld + (size_t(b) * P.gamma + i) * size_t(P.V) * E::ES
                                 : nullptr;
  };
  seek(t);
  auto advance = [&]() {  // to the next chunk
    if (++c == P.nch1) {
      c = 0;
      if (++i == P.R) {
        i = 0;
        ++b;
        T = T_next;
        if (!GREEDY && b + 1 < P.B) T_next = __ldg(P.temp + b + 1);
      }
      trow = P.Lt + (size_t(b) * P.R + i) * size_t(P.V) * E::ES;
      drow = (!GREEDY && i < P.gs) ? P.Ld + (size_t(b) * P.gamma + i) * size_t(P.V) * E::ES
                                   : nullptr;
    }
  };
  for (long long seq = 0;; ++seq) {
    const int s = int(seq % NS);
    const unsigned use = unsigned(seq / NS);
    if (!pending && tend - t <= NS) claim();
    if (t == tend) {  // on to the claimed unit, if the pool has one left
      if (pending && claimed < sp.nunits) {
        t = sp.ts + claimed * sp.unit;
        tend = min(t + sp.unit, P.tasks);
        pending = false;
        ++taken;
        seek(t);
      } else {
        report();
        end_markers(P, C, seq);
        return;
      }
    }
    if (C.abort) {
      report();
      end_markers(P, C, seq);
      return;
    }
    if (use > 0 && !mbar_wait(&C.empty[s], (use - 1) & 1u, P, &C.abort)) {
      report();
      return;
    }
    Desc& d = C.desc[s];
    d.end = 0;
    d.b = b; d.i = i; d.c = c;
    d.e0 = c * P.ch1;
    d.n = min(P.ch1, P.V - d.e0);
    d.kf = LOG2E_F / T;
    if (PAIRS) {
      d.kf2 = d.kf;
      d.pair = 0;
      d.n2 = 0;
    }
    const unsigned char* tseg = trow + size_t(d.e0) * E::ES;
    const unsigned char* dseg = drow ? drow + size_t(d.e0) * E::ES : nullptr;
    split<DT>(tseg, d.n, d.head_t, d.nb_t);
    ++t;
    if (PAIRS && t < tend) {  // the next target chunk of the range into the second half
      advance();
      const int e0b = c * P.ch1;
      d.pair = 1;
      d.n2 = min(P.ch1, P.V - e0b);
      d.kf2 = LOG2E_F / T;
      dseg = trow + size_t(e0b) * E::ES;
      split<DT>(dseg, d.n2, d.head_d, d.nb_d);
      ++t;
    } else if (dseg) {
      split<DT>(dseg, d.n, d.head_d, d.nb_d);
    } else {
      d.head_d = d.nb_d = 0;
    }
    const unsigned bt = unsigned(d.nb_t) * E::ES, bd = unsigned(d.nb_d) * E::ES;
    if (P.withhold_slot && blockIdx.x == 0 && seq == 0) {
      // failure-handling test: the first slot of CTA 0 is never filled, so its
      // consumers' bounded wait runs out (SV_ST_TIMEOUT) and the CTA gives up
    } else if (bt + bd == 0u) {
      mbar_arrive(&C.full[s]);
    } else {
      mbar_arrive_tx(&C.full[s], bt + bd);
      if (bt) bulk_g2s(slots + size_t(s) * SLOT, tseg + size_t(d.head_t) * E::ES, bt, &C.full[s]);
      if (bd)
        bulk_g2s(slots + size_t(s) * SLOT + HALF, dseg + size_t(d.head_d) * E::ES, bd,
                 &C.full[s]);
    }
    advance();  // after the copies are on their way (it may load a temperature)
  }
}

// Consumers: every warp loads its share of a slot into registers and hands
// the slot back at once (so the producer can refill it while the share is
// reduced), then publishes its own partial (two for a pair of target chunks).
template <int DT, bool GREEDY, bool PAIRS, bool CONTIG>
__device__ void consumer(const Params& P, SmemCtl<GeoReduce>& C, const unsigned char* slots) {
  using E = Elem<DT>;
  using G = GeoReduce;
  constexpr int NS = G::NS, SLOT = G::SLOT, GW = G::GW;
  const int lane = threadIdx.x & 31;
  int grp, wg;
  consumer_role<G>(int(threadIdx.x >> 5), grp, wg);
  // wait for slot `seq`, load this warp's share and release the slot; false
  // at the end marker or when the CTA gave up
  auto acquire = [&](long long seq, Share<G::MAXV>& sh) {
    const int s = int(seq % NS);
    const unsigned use = unsigned(seq / NS);
    if (!mbar_wait(&C.full[s], use & 1u, P, &C.abort)) return false;
    const Desc& d = C.desc[s];
    if (d.end) return false;
    const bool second = PAIRS ? d.pair != 0 : d.i < P.gs;
    load_share<DT, G, CONTIG, PAIRS>(d, slots + size_t(s) * SLOT, second, wg, lane, sh);
    __syncwarp();
    if (lane == 0) mbar_arrive(&C.empty[s]);
    return true;
  };
  auto process = [&](const Share<G::MAXV>& sh) {
    float4 out, out2 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (GREEDY) {
      const unsigned char* gt =
          P.Lt + ((size_t(sh.b) * P.R + sh.i) * size_t(P.V) + sh.e0) * E::ES;
      out = reduce_share_argmax<DT, G, CONTIG>(sh.t, gt, sh.e0, sh.head_t, sh.nb_t, sh.n, wg,
                                               lane);
      if (sh.pair) {
        int b2 = sh.b, i2 = sh.i, c2 = sh.c;
        next_chunk(P, b2, i2, c2);
        const unsigned char* g2 =
            P.Lt + ((size_t(b2) * P.R + i2) * size_t(P.V) + size_t(c2) * P.ch1) * E::ES;
        out2 = reduce_share_argmax<DT, G, CONTIG>(sh.d, g2, c2 * P.ch1, sh.head_d, sh.nb_d,
                                                  sh.n2, wg, lane);
      }
    } else if (PAIRS) {
      const float4 r = reduce_share_ms<DT, G::MAXV, GW, true, CONTIG>(P, sh, wg, lane);
      out = make_float4(r.x, r.y, -INFINITY, 0.f);
      out2 = make_float4(r.z, r.w, -INFINITY, 0.f);
    } else {
      out = reduce_share_ms<DT, G::MAXV, GW, false, CONTIG>(P, sh, wg, lane);
    }
    if (lane == 0) {
      Partial* dst = P.part + ((size_t(sh.b) * P.R + sh.i) * P.nch1 + sh.c) * GW + wg;
      *reinterpret_cast<float4*>(dst) = out;
      if (PAIRS && sh.pair) {
        int b2 = sh.b, i2 = sh.i, c2 = sh.c;
        next_chunk(P, b2, i2, c2);
        Partial* dst2 = P.part + ((size_t(b2) * P.R + i2) * P.nch1 + c2) * GW + wg;
        *reinterpret_cast<float4*>(dst2) = out2;
      }
    }
  };
  Share<G::MAXV> sh;
  for (long long seq = grp;; seq += G::NG) {
    if (!acquire(seq, sh)) return;
    process(sh);
  }
}

// GREEDY: chunk argmax instead of (max, sum); PAIRS: no draft rows are
// streamed and a slot carries two target chunks (greedy verification, given
// draft normalisers, draft sampling); CONTIG: the warps' shares are
// contiguous spans of the row (draft sampling searches them).
template <int DT, bool GREEDY, bool PAIRS, bool CONTIG>
__global__ void __launch_bounds__(NTHR, 1) sv_reduce(const Params P) {
  using G = GeoReduce;
  // every CTA of this grid is resident from the start (one per SM), so the
  // decide kernel's CTAs may take the SMs' spare room at once
  allow_next_kernel();
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* slots = smem;
  SmemCtl<G>& C = *reinterpret_cast<SmemCtl<G>*>(smem + size_t(G::NS) * G::SLOT);
  if (threadIdx.x == 0) {
    C.abort = 0;
    for (int s = 0; s < G::NS; ++s) {
      mbar_init(&C.full[s], 1);
      mbar_init(&C.empty[s], G::GW);
    }
  }
  // launched programmatically after the previous kernel in the stream (the
  // last kernel of an earlier call, or whatever wrote the logits): nothing
  // it wrote is read before it has completed
  wait_previous_kernel();
  if (threadIdx.x == 0) {
    // the workspace is in its ready state between calls; mark this call.
    // Only the state word is tested: the other CTAs of this grid may already
    // be claiming pool units, so the claim counter can be non-zero here.
    if (blockIdx.x == 0) {
      if (P.ctrl->state != 0ull) set_status(P, SV_ST_WORKSPACE);
      P.ctrl->state = 1ull;
      P.ctrl->pad[0] = 0ull;  // the residual kernel's chunk claims
    }
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    if (threadIdx.x == 0)
      producer<DT, GREEDY, PAIRS>(P, C, slots, reduce_split(P, blockIdx.x, gridDim.x),
                                  &P.ctrl->claims, &P.ctrl->pad[1]);
  } else {
    consumer<DT, GREEDY, PAIRS, CONTIG>(P, C, slots);
  }
}

// ------------------------------------------------------------ decide

// Combine of row i of request b (one warp): the maximum m of the partials'
// maxima and S = sum s_c * 2^((m_c - m) * kf), accumulated as float pairs.
// Target in fields (a, b), draft in (c, d).  Result valid in every lane.
// NC: the partials were written by an earlier kernel (read-only cache path);
// otherwise by this kernel's cluster, read with plain loads.
template <bool NC = true>
__device__ __forceinline__ float4 load_partial(const Partial* p) {
  return NC ? __ldg(reinterpret_cast<const float4*>(p)) : *reinterpret_cast<const float4*>(p);
}
template <bool NC = true>
__device__ void row_combine(const Partial* pp, int np, float kf, bool draft, float& mt,
                            FF& St, float& md, FF& Sd) {
  const int lane = threadIdx.x & 31;
  mt = -INFINITY;
  md = -INFINITY;
  for (int c = lane; c < np; c += 32) {
    const float4 v = load_partial<NC>(pp + c);
    mt = fmaxf(mt, v.x);
    md = fmaxf(md, v.z);
  }
  mt = warp_max(mt);
  md = warp_max(md);
  float th = 0.f, tl = 0.f, dh = 0.f, dl = 0.f;
  for (int c = lane; c < np; c += 32) {
    const float4 v = load_partial<NC>(pp + c);
    ff_add(th, tl, (mt == -INFINITY) ? v.y : v.y * ex2((v.x - mt) * kf));
    if (draft) ff_add(dh, dl, (md == -INFINITY) ? v.w : v.w * ex2((v.z - md) * kf));
  }
  warp_sum_ff(th, tl);
  St = ff(th, tl);
  if (draft) {
    warp_sum_ff(dh, dl);
    Sd = ff(dh, dl);
  } else {
    md = 0.f;
    Sd = ff(1.f);
  }
}

// Argmax of row i of request b (one warp) over its partials.
template <bool NC = true>
__device__ void row_argmax(const Partial* pp, int np, float& best, int& bi, int& nan) {
  const int lane = threadIdx.x & 31;
  best = -INFINITY;
  bi = INT_MAX;
  nan = 0;
  for (int c = lane; c < np; c += 32) {
    const float4 v = load_partial<NC>(pp + c);
    am_merge(best, bi, nan, v.x, __float_as_int(v.y), __float_as_int(v.z));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    const int n2 = __shfl_xor_sync(0xffffffffu, nan, o);
    am_merge(best, bi, nan, b2, i2, n2);
  }
}

// The draw's normalisers of every row i (one warp, lane i), whichever row
// turns out to be the first rejection: 1/S_t and, for i < gamma,
// c0 = (m_t - m_d) * kf + log2(S_t / S_d), each as an unevaluated float pair,
// in fp32 arithmetic: (m_t - m_d) * kf exactly (kf is the factor the row
// sums were formed with), log2 of the ratio as its binary exponent plus
// log2f of the mantissa in [1/2, 1) (absolute error about 1e-7) plus the
// ratio's low part.
struct Cand {
  float ist_hi, ist_lo, c0_hi, c0_lo;
};
__device__ void record_candidates(const Params& P, int b, const RowStat* rows, Cand* cand) {
  const int g = P.gamma, R = P.R;
  const int lane = threadIdx.x & 31;
  const float kf = LOG2E_F / __ldg(P.temp + b);
  for (int i = lane; i < R; i += 32) {
    const RowStat& rk = rows[i];
    Cand c{0.f, 0.f, 0.f, 0.f};
    if (rk.bad == 0) {
      const FF St = ff(rk.St_h, rk.St_l);
      const FF ist = ff_div(ff(1.f), St);
      c.ist_hi = ist.h;
      c.ist_lo = ist.l;
      if (i < g) {
        // log2(P_d[v] / P_t[v]) = (l_d[v] - l_t[v]) * kf + (m_t - m_d) * kf + log2(S_t / S_d)
        const FF q = ff_div(St, ff(rk.Sd_h, rk.Sd_l));
        int e = 0;
        const float mant = frexpf(q.h, &e);
        const float lg = log2f(mant) + q.l / (q.h * 0.69314718055994531f);
        FF c0 = ff_mulf(ff_diff(rk.mt, rk.md), kf);
        c0 = c0 + ff(float(e)) + ff(lg);
        c.c0_hi = c0.h;
        c.c0_lo = c0.l;
      }
    }
    cand[i] = c;
  }
}

// Sampling decision of request b (warp 0 of the CTA, rows in `rows`): lane
// i < gamma tests position i, accept iff u <= min(1, P_t / P_d) with
// P_t / P_d = 2^E * S_d / S_t, E = ((l_t - l_d) - (m_t - m_d)) * log2(e) / T,
// E formed in float pairs (exact differences, log2(e) / T as a pair) and
// 2^E by exp2f: the ratio carries a relative error of a few 1e-7, below the
// 1e-6 window in which the oracle flags a decision as a near-tie.  P_d = 0 in
// fp64 (l_d = -inf, or (l_d - m_d) / T so far below m_d that the oracle's
// fp64 underflows) accepts: the rare second case is settled in fp64 as the
// oracle does.  Then the first rejection k and the outputs but token k.
// Returns the record's mode and k (in lane 0).
template <int DT>
__device__ int2 decide_sample(const Params& P, int b, const RowStat* rows, float lt, float ld,
                              float u, bool tok_ok, int xi) {
  const int g = P.gamma, R = P.R;
  const int lane = threadIdx.x & 31;
  const float T = __ldg(P.temp + b);
  const bool t_ok = isfinite(T) && T >= 0x1p-126f;
  const FF k2 = ff_log2e_over(T);
  int bad = 0, acc = 1;
  float pt = NAN, pd = NAN;
  for (int i = lane; i < R; i += 32) bad |= rows[i].bad;
  if (lane < g) {
    const RowStat& r = rows[lane];
    if (!tok_ok) {
      bad |= SV_ST_BAD_TOKEN;
    } else if (bad == 0 && t_ok) {
      const FF St = ff(r.St_h, r.St_l), Sd = ff(r.Sd_h, r.Sd_l);
      const FF et = ff_mul2(ff_diff(lt, r.mt), k2);  // log2(P_t * S_t)
      const FF ed = ff_mul2(ff_diff(ld, r.md), k2);  // log2(P_d * S_d)
      bool pd_zero = ld == -INFINITY;
      if (!pd_zero && ed.h < -1000.f) {  // rare: does the oracle's fp64 P_d underflow?
        const double e64 = (double(ld) - double(r.md)) * (LOG2E_D / double(T));
        pd_zero = exp2_d(e64) / (double(r.Sd_h) + double(r.Sd_l)) == 0.0;
      }
      float ratio = 1.f;
      if (!pd_zero) {
        if (lt == -INFINITY) {  // P_t = 0
          ratio = 0.f;
        } else {
          const float p2 = ff_exp2(et - ed);
          const FF q = ff_div(Sd, St);
          ratio = fminf(1.f, p2 * q.h + p2 * q.l);
        }
      }
      acc = u <= ratio;
      if (P.out_p) {
        pt = lt == -INFINITY ? 0.f : ff_exp2(et) * ff_div(ff(1.f), St).h;
        pd = ld == -INFINITY ? 0.f : ff_exp2(ed) * ff_div(ff(1.f), Sd).h;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) bad |= __shfl_xor_sync(0xffffffffu, bad, o);
  if (!t_ok) bad |= SV_ST_BAD_TEMP;
  const bool valid = (bad == 0);
  const unsigned rej = __ballot_sync(0xffffffffu, lane < g && !acc);
  const int k = rej ? __ffs(rej) - 1 : g;
  // lane i < gamma holds x_i (no shuffle: lanes i >= R skip this loop)
  for (int i = lane; i < R; i += 32) {
    const int tok = i < g ? xi : -1;
    if (!valid || i != k) P.out_tokens[size_t(b) * R + i] = (valid && i < k) ? tok : -1;
  }
  if (P.out_p && lane < g) {
    P.out_p[(size_t(b) * g + lane) * 2] = valid ? pt : NAN;
    P.out_p[(size_t(b) * g + lane) * 2 + 1] = valid ? pd : NAN;
  }
  if (lane == 0) {
    P.out_n[b] = valid ? k : 0;
    if (!valid && P.out_Z) P.out_Z[b] = NAN;
    set_status(P, bad);
  }
  return make_int2(!valid ? MODE_INVALID : (k < g ? MODE_REJECT : MODE_BONUS), k);
}

// The decision record of request b (one thread): the draw's row k and its
// normalisers, read by the residual and draw kernels.
__device__ Record make_record(const Params& P, int b, int mode, int k, const RowStat* rows,
                              const Cand* cand) {
  Record r;
  r.k = k;
  r.mode = mode;
  r.kf = LOG2E_F / __ldg(P.temp + b);
  r.mt = 0.f;
  r.ist_hi = r.ist_lo = r.c0_hi = r.c0_lo = 0.f;
  r.pad[0] = r.pad[1] = r.pad[2] = r.pad[3] = 0;
  if (mode != MODE_INVALID) {
    r.mt = rows[k].mt;
    r.ist_hi = cand[k].ist_hi;
    r.ist_lo = cand[k].ist_lo;
    if (mode == MODE_REJECT) {
      r.c0_hi = cand[k].c0_hi;
      r.c0_lo = cand[k].c0_lo;
    }
  }
  return r;
}
__device__ void write_record(const Params& P, int b, int mode, int k, const RowStat* rows,
                             const Cand* cand) {
  const Record r = make_record(P, b, mode, k, rows, cand);
  int4* d = reinterpret_cast<int4*>(P.rec + b);
  const int4* src = reinterpret_cast<const int4*>(&r);
  d[0] = src[0]; d[1] = src[1]; d[2] = src[2];
}

// Greedy decision of request b (warp 0, rows in `rows`).
__device__ void decide_greedy(const Params& P, int b, const RowStat* rows) {
  const int g = P.gamma, R = P.R;
  const int lane = threadIdx.x & 31;
  int bad = 0;
  int am[2] = {-1, -1};
  for (int i = lane, q = 0; i < R; i += 32, ++q) {
    bad |= rows[i].bad;
    am[q] = rows[i].amax;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) bad |= __shfl_xor_sync(0xffffffffu, bad, o);
  int xi = -1;
  if (lane < g) {
    xi = __ldg(P.x + size_t(b) * g + lane);
    if (xi < 0 || xi >= P.V) bad |= SV_ST_BAD_TOKEN;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) bad |= __shfl_xor_sync(0xffffffffu, bad, o);
  const bool valid = (bad == 0);
  const unsigned mis = __ballot_sync(0xffffffffu, lane < g && xi != am[0]);
  const int k = mis ? __ffs(mis) - 1 : g;
  for (int i = lane, q = 0; i < R; i += 32, ++q)
    P.out_tokens[size_t(b) * R + i] = (valid && i <= k) ? am[q] : -1;
  if (lane == 0) {
    P.out_n[b] = valid ? k : 0;
    set_status(P, bad);
  }
}

// The decision's per-position inputs of request b (warp 0, lane i < gamma
// takes position i): draft token, accept uniform, and the target and draft
// logits at the token.  They are the call's inputs, so they are loaded before
// the wait for the partials.
template <int DT>
__device__ __forceinline__ void load_decision_inputs(const Params& P, int b, float& lt, float& ld,
                                                     float& u, bool& tok_ok, int& xi) {
  using E = Elem<DT>;
  const int g = P.gamma, R = P.R, V = P.V;
  const int lane = threadIdx.x & 31;
  lt = ld = u = 0.f;
  tok_ok = true;
  xi = -1;
  if ((threadIdx.x >> 5) == 0 && lane < g) {
    xi = __ldg(P.x + size_t(b) * g + lane);
    u = __ldg(P.u_acc + size_t(b) * g + lane);
    tok_ok = xi >= 0 && xi < V;
    if (tok_ok) {
      lt = E::load(P.Lt, (long long)(size_t(b) * R + lane) * V + xi);
      ld = E::load(P.Ld, (long long)(size_t(b) * g + lane) * V + xi);
    }
  }
}

// Every row's statistics of request b for the sampling decision, the warps of
// the CTA taking rows in turn: the partials combined (row_combine), or the
// draft row's normaliser as given (dst_sh, cached verification).
template <int NWARPS, bool NC = true>
__device__ void combine_rows(const Params& P, int b, float kf, const float2* dst_sh,
                             RowStat* rows) {
  const int warp = int(threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int g = P.gamma, R = P.R;
  const bool cached = P.dstats != nullptr;
  for (int i = warp; i < R; i += NWARPS) {
    const Partial* pp = P.part + (size_t(b) * R + i) * size_t(P.np1);
    float mt, md;
    FF St, Sd;
    row_combine<NC>(pp, P.np1, kf, i < P.gs, mt, St, md, Sd);
    if (cached && i < g) {  // the draft row's normaliser, as given
      md = dst_sh[i].x;
      Sd = ff(dst_sh[i].y);
    }
    if (lane == 0) {
      RowStat r;
      r.mt = mt; r.md = md;
      r.St_h = St.h; r.St_l = St.l; r.Sd_h = Sd.h; r.Sd_l = Sd.l;
      r.bad = (!row_ok_ff(mt, St.h) || (i < g && !row_ok_ff(md, Sd.h))) ? SV_ST_NONFINITE : 0;
      r.amax = -1;
      rows[i] = r;
    }
  }
}

// One CTA per request: NW warps combine the rows (row i by warp i % NW), then
// warp 0 decides.  The draft tokens, their logits and
// the uniforms are loaded by warp 0 before its rows; given draft normalisers
// (dstats) replace the draft rows' combine.
template <int DT, bool GREEDY, int NW>
__global__ void __launch_bounds__(32 * NW) sv_decide(const Params P, bool last) {
  __shared__ RowStat rows[MAXR];
  __shared__ Cand cand[MAXR];
  __shared__ float2 dst_sh[MAXR];
  __shared__ int2 mode_k;
  const int b = blockIdx.x, warp = int(threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int g = P.gamma, R = P.R;
  float lt = 0.f, ld = 0.f, u = 0.f;
  bool tok_ok = true;
  int xi = -1;
  if (!GREEDY) load_decision_inputs<DT>(P, b, lt, ld, u, tok_ok, xi);
  const float kf = GREEDY ? 0.f : LOG2E_F / __ldg(P.temp + b);
  const bool cached = !GREEDY && P.dstats != nullptr;
  if (cached && int(threadIdx.x) < g)
    dst_sh[threadIdx.x] = __ldg(reinterpret_cast<const float2*>(P.dstats) + size_t(b) * g +
                                threadIdx.x);
  // the loads above read only the call's inputs; the partials come from the
  // reduce kernel
  wait_previous_kernel();
  if (cached) __syncthreads();
  if (GREEDY) {
    for (int i = warp; i < R; i += NW) {
      const Partial* pp = P.part + (size_t(b) * R + i) * size_t(P.np1);
      float best;
      int bi, nan;
      row_argmax(pp, P.np1, best, bi, nan);
      if (lane == 0) {
        RowStat r;
        r.mt = best; r.md = 0.f; r.St_h = r.St_l = r.Sd_h = r.Sd_l = 0.f;
        r.bad = (nan || bi == INT_MAX || best == INFINITY) ? SV_ST_NONFINITE : 0;
        r.amax = bi;
        rows[i] = r;
      }
    }
  } else {
    combine_rows<NW>(P, b, kf, dst_sh, rows);
  }
  __syncthreads();
  if (GREEDY) {
    if (warp == 0) decide_greedy(P, b, rows);
  } else {
    // the record's normalisers for every row, beside the acceptance tests
    if (warp == 1) record_candidates(P, b, rows, cand);
    if (warp == 0) {
      const int2 mk = decide_sample<DT>(P, b, rows, lt, ld, u, tok_ok, xi);
      if (lane == 0) mode_k = mk;
    }
    __syncthreads();
    if (threadIdx.x == 0) write_record(P, b, mode_k.x, mode_k.y, rows, cand);
  }
  // greedy verification ends here: the workspace is ready for the next call
  if (last && b == 0 && threadIdx.x == 0) ready_for_next_call(P);
  // only now: the residual kernel's CTAs need whole SMs, which this grid's
  // CTAs still waiting to be placed must not lose to them
  allow_next_kernel();
}

// ------------------------------------------------------------ residual

// Weights of vectors [0, nv) of a target span `tv` (and draft span `dv` when
// TWO) read from global memory, PV per lane in flight, summed in packed pairs.
template <int DT, int PV, bool TWO>
__device__ __forceinline__ float global_vectors_mass(const Record& r, const uint4* tv,
                                                  const uint4* dv, int nv, int lane) {
  using E = Elem<DT>;
  const uint4 neg = make_uint4(E::NEG_INF_WORD, E::NEG_INF_WORD, E::NEG_INF_WORD, E::NEG_INF_WORD);
  unsigned long long acc = pk2(0.f, 0.f);
  for (int v0 = 0; v0 < nv; v0 += 32 * PV) {
    uint4 vt[PV], vd[TWO ? PV : 1];
#pragma unroll
    for (int u = 0; u < PV; ++u) {
      const int j = v0 + lane + 32 * u;
      vt[u] = j < nv ? __ldg(tv + j) : neg;
      if (TWO) vd[u] = j < nv ? __ldg(dv + j) : neg;
    }
#pragma unroll
    for (int u = 0; u < PV; ++u) vec_weights_acc<DT, TWO>(r, vt[u], TWO ? vd[u] : vt[u], acc);
  }
  float a, b;
  upk2(acc, a, b);
  return a + b;
}

// Mass of elements [lo, hi) of the row token k is drawn from: target row
// `trow` and (after a rejection) draft row `drow`; one warp, fp32 weights,
// lane sums added as float pairs.  Aligned spans are read as 16-byte vectors,
// PV per lane in flight.  TARGET_ONLY: the caller passes no draft row.
template <int DT, bool TARGET_ONLY = false>
__device__ void span_mass(const Record& r, const unsigned char* trow, const unsigned char* drow,
                          int lo, int hi, float& mh, float& ml) {
  using E = Elem<DT>;
  const int lane = threadIdx.x & 31;
  const bool two = !TARGET_ONLY && (r.mode == MODE_REJECT);
  float acc = 0.f;
  int e_tail = lo;
  const unsigned char* t0 = trow + size_t(lo) * E::ES;
  const unsigned char* d0 = two ? drow + size_t(lo) * E::ES : t0;
  if (((reinterpret_cast<uintptr_t>(t0) | reinterpret_cast<uintptr_t>(d0)) & 15u) == 0) {
    constexpr int PV = 4;  // vectors per lane in flight
    const int nv = (hi - lo) / E::VEC;
    const uint4* tv = reinterpret_cast<const uint4*>(t0);
    const uint4* dv = reinterpret_cast<const uint4*>(d0);
    acc = two ? global_vectors_mass<DT, PV, true>(r, tv, dv, nv, lane)
              : global_vectors_mass<DT, PV, false>(r, tv, dv, nv, lane);
    e_tail = lo + nv * E::VEC;
  }
  for (int e = e_tail + lane; e < hi; e += 32)
    acc += weight(r, E::load(trow, e), two ? E::load(drow, e) : 0.f);
  mh = acc;
  ml = 0.f;
  warp_sum_ff(mh, ml);
}

// Residual producer (one lane): phase-2 chunks claimed one at a time from a
// counter the whole grid shares (reset by the reduce kernel), so CTAs that
// finish their chunks early take more: the work spreads by bytes, whatever
// the mix of rejections (a target and a draft chunk) and bonus draws (a
// target chunk); a static cyclic split left the busiest CTA about 20 %
// above the mean.  Chunks are numbered chunk-major, t = c * B + b, so the
// short last chunks of the rows are claimed last; chunks of invalid requests
// are skipped.  Each slot gets the chunk of target row k (gamma for the
// bonus), the draft row k chunk after a rejection, and the request's record.
// Every CTA starts with chunk x of its own; claims run two chunks ahead and a
// chunk's (k, mode) is loaded one chunk ahead, so neither round trip is
// waited for.
template <int DT>
__device__ void producer_res(const Params& P, SmemCtl<GeoResidual>& C, unsigned char* slots) {
  using E = Elem<DT>;
  using G = GeoResidual;
  constexpr int NS = G::NS, SLOT = G::SLOT, HALF = G::HALF;
  const long long T = (long long)P.B * P.nch2;
  unsigned long long* claims = &P.ctrl->pad[0];
  // chunk x first (no claim to wait for), then chunks G, G + 1, ... by claim
  auto claim = [&]() { return (long long)gridDim.x + (long long)atomicAdd(claims, 1ull); };
  auto km_of = [&](long long tt) {
    return tt < T ? __ldg(reinterpret_cast<const int2*>(P.rec + tt % P.B)) : make_int2(0, 0);
  };
  long long t = blockIdx.x, t_next = claim();
  int2 km = km_of(t);
  long long seq = 0;
  while (t < T) {
    const int2 km_next = km_of(t_next);  // used in the next iteration
    const long long t_next2 = claim();
    const int c = int(t / P.B), b = int(t - (long long)c * P.B);
    if (km.y == MODE_REJECT || km.y == MODE_BONUS) {
      const int s = int(seq % NS);
      const unsigned use = unsigned(seq / NS);
      ++seq;
      if (use > 0 && !mbar_wait(&C.empty[s], (use - 1) & 1u, P, &C.abort)) return;
      if (C.abort) break;
      Desc& d = C.desc[s];
      const bool two = km.y == MODE_REJECT;
      const int rowk = two ? km.x : P.gamma;
      d.end = 0;
      d.b = b; d.i = rowk; d.c = c;
      d.e0 = c * P.ch2;
      d.n = min(P.ch2, P.V - d.e0);
      const unsigned char* tseg = P.Lt + ((size_t(b) * P.R + rowk) * size_t(P.V) + d.e0) * E::ES;
      const unsigned char* dseg =
          two ? P.Ld + ((size_t(b) * P.gamma + km.x) * size_t(P.V) + d.e0) * E::ES : nullptr;
      split<DT>(tseg, d.n, d.head_t, d.nb_t);
      d.head_d = d.nb_d = 0;
      if (dseg) split<DT>(dseg, d.n, d.head_d, d.nb_d);
      const unsigned bt = unsigned(d.nb_t) * E::ES, bd = unsigned(d.nb_d) * E::ES;
      mbar_arrive_tx(&C.full[s], bt + bd + unsigned(sizeof(Record)));
      if (bt) bulk_g2s(slots + size_t(s) * SLOT, tseg + size_t(d.head_t) * E::ES, bt, &C.full[s]);
      if (bd)
        bulk_g2s(slots + size_t(s) * SLOT + HALF, dseg + size_t(d.head_d) * E::ES, bd,
                 &C.full[s]);
      bulk_g2s(&d.rec, P.rec + b, unsigned(sizeof(Record)), &C.full[s]);
    }
    t = t_next;
    km = km_next;
    t_next = t_next2;
  }
  end_markers(P, C, seq);
}

// Weights of this warp's whole vectors [j0, vhi) of a slot (target body at
// tv, draft body at dv when TWO), summed in packed pairs: PV vectors per lane
// are copied into registers and the slot handed back (`release`) before the
// arithmetic.  The first PV - 1 rounds are read without a bounds test when
// every lane has a vector in each of them (all but the rows' last chunks);
// vectors past vhi read as -inf (weight 0).
template <int DT, int PV, bool TWO, typename Release>
__device__ __forceinline__ float slot_vectors_mass(const Record& r, const uint4* tv,
                                                   const uint4* dv, int j0, int vhi, int lane,
                                                   Release release) {
  using E = Elem<DT>;
  const uint4 neg = make_uint4(E::NEG_INF_WORD, E::NEG_INF_WORD, E::NEG_INF_WORD, E::NEG_INF_WORD);
  uint4 vt[PV], vd[TWO ? PV : 1];
  if (vhi - j0 >= 32 * (PV - 1)) {
#pragma unroll
    for (int u = 0; u < PV - 1; ++u) {
      const int j = j0 + lane + 32 * u;
      vt[u] = tv[j];
      if (TWO) vd[u] = dv[j];
    }
  } else {
#pragma unroll
    for (int u = 0; u < PV - 1; ++u) {
      const int j = j0 + lane + 32 * u;
      vt[u] = j < vhi ? tv[j] : neg;
      if (TWO) vd[u] = j < vhi ? dv[j] : neg;
    }
  }
  {
    const int j = j0 + lane + 32 * (PV - 1);
    vt[PV - 1] = j < vhi ? tv[j] : neg;
    if (TWO) vd[PV - 1] = j < vhi ? dv[j] : neg;
  }
  unsigned long long acc = pk2(0.f, 0.f);
  for (int j = j0 + lane + 32 * PV; j < vhi; j += 32)  // only if sub exceeds 32*PV vectors
    vec_weights_acc<DT, TWO>(r, tv[j], TWO ? dv[j] : tv[j], acc);
  release();
#pragma unroll
  for (int u = 0; u < PV; ++u) vec_weights_acc<DT, TWO>(r, vt[u], TWO ? vd[u] : vt[u], acc);
  float a, b;
  upk2(acc, a, b);
  return a + b;
}

// Mass of this warp's contiguous sub-range [cw*sub, (cw+1)*sub) of a
// phase-2 chunk held in a slot (target body at +0, draft body at +HALF),
// returned as a float pair (hi, lo) valid in every lane.  ALIGNED: every row
// of the call starts on a 16-byte boundary (the unaligned path is not
// compiled in).
template <int DT, bool ALIGNED, typename Release>
__device__ float2 warp_slot_mass(const Params& P, const Desc& d, const Record& r,
                                 const unsigned char* slot, int wg, int lane, Release release) {
  using E = Elem<DT>;
  using G = GeoResidual;
  constexpr int HALF = G::HALF;
  const bool two = (r.mode == MODE_REJECT);
  const int lo = wg * P.sub;
  const int hi = min(lo + P.sub, d.n);
  float acc = 0.f;
  if (lo >= hi) {
    release();
  } else {
    const unsigned char* trow = P.Lt + ((size_t(d.b) * P.R + d.i) * size_t(P.V) + d.e0) * E::ES;
    const unsigned char* drow =
        two ? P.Ld + ((size_t(d.b) * P.gamma + r.k) * size_t(P.V) + d.e0) * E::ES : nullptr;
    if (ALIGNED || (d.head_t == 0 && (!two || d.head_d == 0))) {
      // aligned: whole 16-byte vectors from shared memory, held in registers
      constexpr int PV = G::MAXV;  // a sub-range has at most 32 * PV vectors
      const uint4* tv = reinterpret_cast<const uint4*>(slot);
      const uint4* dv = reinterpret_cast<const uint4*>(slot + HALF);
      const int j0 = lo / E::VEC, vhi = min(hi, d.nb_t) / E::VEC;
      acc = two ? slot_vectors_mass<DT, PV, true>(r, tv, dv, j0, vhi, lane, release)
                : slot_vectors_mass<DT, PV, false>(r, tv, dv, j0, vhi, lane, release);
      for (int e = max(lo, d.nb_t) + lane; e < hi; e += 32)
        acc += weight(r, E::load(trow, e), two ? E::load(drow, e) : 0.f);
    } else if constexpr (!ALIGNED) {
      // rows not on 16-byte boundaries: the target body's whole vectors in
      // this warp's range, each paired with the draft elements of the same
      // indices, read from the draft body at a shift of delta = head_t -
      // head_d elements with narrower loads; the few other elements of the
      // range one by one (from shared memory before the slot is handed back,
      // from global memory after)
      constexpr int PV = G::MAXV;
      const int hd = two ? d.head_d : d.head_t;
      const int delta = d.head_t - hd;  // draft body index of target body index t: t + delta
      const int nvt = d.nb_t / E::VEC;
      auto cdiv = [](int x) { return x >= 0 ? (x + E::VEC - 1) / E::VEC : -((-x) / E::VEC); };
      auto fdiv = [](int x) { return x >= 0 ? x / E::VEC : -((-x + E::VEC - 1) / E::VEC); };
      int va = max(0, cdiv(lo - d.head_t)), vb = min(nvt, fdiv(hi - d.head_t));
      if (two) {
        va = max(va, cdiv(-delta));
        vb = min(vb, fdiv(d.nb_d - delta));
      }
      vb = max(va, vb);
      const uint4* tv = reinterpret_cast<const uint4*>(slot);
      const unsigned char* dbody = slot + HALF;
      const uint4 neg =
          make_uint4(E::NEG_INF_WORD, E::NEG_INF_WORD, E::NEG_INF_WORD, E::NEG_INF_WORD);
      uint4 vt[PV], vd[PV];
#pragma unroll
      for (int u = 0; u < PV; ++u) {
        const int j = va + lane + 32 * u;
        vt[u] = neg;
        vd[u] = neg;
        if (j < vb) {
          vt[u] = tv[j];
          vd[u] = two ? E::gather_shifted(dbody, j * E::VEC + delta) : vt[u];
        }
      }
      // elements outside those vectors: [lo, s1) and [s2, hi)
      const int s1 = min(hi, d.head_t + va * E::VEC);
      const int s2 = max(s1, d.head_t + vb * E::VEC);
      auto in_t = [&](int e) { return e - d.head_t >= 0 && e - d.head_t < d.nb_t; };
      auto in_d = [&](int e) { return !two || (e - hd >= 0 && e - hd < d.nb_d); };
      // from_smem: the elements both of whose values are in the slot, read
      // before it is handed back; otherwise the rest, both values read from
      // global memory (the slot may already hold the next chunk)
      auto scalar = [&](bool from_smem) {
        auto one = [&](int e) {
          if ((in_t(e) && in_d(e)) != from_smem) return;
          const float lt = from_smem ? E::lds(slot, e - d.head_t) : E::load(trow, e);
          const float ld = !two ? 0.f : from_smem ? E::lds(dbody, e - hd) : E::load(drow, e);
          acc += weight(r, lt, ld);
        };
        for (int e = lo + lane; e < s1; e += 32) one(e);
        for (int e = s2 + lane; e < hi; e += 32) one(e);
      };
      scalar(true);
      release();
      scalar(false);
#pragma unroll
      for (int u = 0; u < PV; ++u) acc += vec_weights<DT>(r, vt[u], vd[u], two);
    }
  }
  float2 m = make_float2(acc, 0.f);
  warp_sum_ff(m.x, m.y);
  return m;
}

template <int DT, bool ALIGNED>
__device__ void consumer_res(const Params& P, SmemCtl<GeoResidual>& C,
                             const unsigned char* slots) {
  using G = GeoResidual;
  constexpr int NS = G::NS, SLOT = G::SLOT, GW = G::GW;
  const int lane = threadIdx.x & 31;
  int grp, wg;
  consumer_role<G>(int(threadIdx.x >> 5), grp, wg);
  for (long long seq = grp;; seq += G::NG) {
    const int s = int(seq % NS);
    const unsigned use = unsigned(seq / NS);
    if (!mbar_wait(&C.full[s], use & 1u, P, &C.abort)) return;
    const Desc d = C.desc[s];
    if (d.end) return;
    auto release = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&C.empty[s]);
    };
    const float2 m =
        warp_slot_mass<DT, ALIGNED>(P, d, d.rec, slots + size_t(s) * SLOT, wg, lane, release);
    if (lane == 0) P.mass[(size_t(d.b) * P.nch2 + d.c) * GW + wg] = Mass{m.x, m.y};
  }
}

// ALIGNED: every target and draft row of the call starts on a 16-byte
// boundary (so does every phase-2 chunk); the kernel for other calls also
// pairs unaligned rows.
template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(NTHR, 1) sv_residual(const Params P) {
  using G = GeoResidual;
  allow_next_kernel();  // one CTA per SM: every CTA of this grid is resident
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* slots = smem;
  SmemCtl<G>& C = *reinterpret_cast<SmemCtl<G>*>(smem + size_t(G::NS) * G::SLOT);
  if (threadIdx.x == 0) {
    C.abort = 0;
    for (int s = 0; s < G::NS; ++s) {
      mbar_init(&C.full[s], 1);
      mbar_init(&C.empty[s], G::GW);
    }
  }
  __syncthreads();
  wait_previous_kernel();  // the decision records
  if (threadIdx.x < 32) {
    if (threadIdx.x == 0) producer_res<DT>(P, C, slots);
  } else {
    consumer_res<DT, ALIGNED>(P, C, slots);
  }
}

// ------------------------------------------------------------ draw

// Token k of request b, one CTA of DRAW_WARPS warps:
//   1. every warp takes a contiguous run of sub-ranges, loads their masses
//      (published by the residual kernel) and sums them; a block prefix over
//      the warps gives Z and the warp whose run crosses tau = u * Z;
//   2. that warp finds the crossing sub-range within its run (lane prefix);
//   3. the sub-range's elements are split over the warps, each warp sums its
//      slice's weights; a block prefix finds the crossing slice, whose warp
//      scans it in index order.
// When the residual summed to 0 (degenerate), the masses of target row k are
// recomputed in step 1 instead.  Running sums and tau are float pairs.
constexpr int DRAW_RUN = 4;  // sub-ranges per lane in step 1 (run of 128 per warp)

template <int DT>
__global__ void __launch_bounds__(32 * DRAW_WARPS) sv_draw(const Params P) {
  using E = Elem<DT>;
  constexpr int GW = GeoResidual::GW;
  __shared__ FF wsum[DRAW_WARPS];
  __shared__ FF sh_rest, sh_before;
  __shared__ int sh_q, sh_wsel;
  const int b = int(blockIdx.x), warp = int(threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int R = P.R, V = P.V;
  // every uniform of the request (only entry k is used): an input, loaded
  // before the wait
  const float u_lane = lane < R ? __ldg(P.u_res + size_t(b) * R + lane) : 0.f;
  // the next call's reduce may be placed as SMs free up: it waits for this
  // grid's completion before it reads anything
  allow_next_kernel();
  wait_previous_kernel();  // the masses (and, before them, the records)
  Record r;
  {
    const int4* src = reinterpret_cast<const int4*>(P.rec + b);
    int4* dst = reinterpret_cast<int4*>(&r);
    dst[0] = __ldg(src); dst[1] = __ldg(src + 1); dst[2] = __ldg(src + 2);
  }
  const bool last_cta = blockIdx.x == 0;
  const int nq = P.nch2 * GW;
  const Mass* ms = P.mass + size_t(b) * P.nch2 * GW;
  // 1a. the masses of this warp's run, loaded beside the record
  const int run = (nq + DRAW_WARPS - 1) / DRAW_WARPS;
  const int qa = min(nq, warp * run), qb = min(nq, qa + run);
  FF mq[DRAW_RUN];  // this lane's masses q = qa + lane + 32 j
#pragma unroll
  for (int j = 0; j < DRAW_RUN; ++j) {
    const int q = qa + lane + 32 * j;
    mq[j] = ff(0.f);
    if (q < qb) {
      const Mass m = ms[q];
      mq[j] = ff(m.hi, m.lo);
    }
  }
  if (r.mode == MODE_INVALID) {
    if (last_cta && threadIdx.x == 0) ready_for_next_call(P);
    return;
  }
  // k is the same in every thread; k = 32 (gamma = 32, all accepted) is past the lanes
  const float u = r.k < 32 ? __shfl_sync(0xffffffffu, u_lane, r.k)
                           : __ldg(P.u_res + size_t(b) * R + r.k);
  const int rowk = (r.mode == MODE_BONUS) ? P.gamma : r.k;
  const unsigned char* trow = P.Lt + (size_t(b) * R + rowk) * size_t(V) * E::ES;
  bool two = (r.mode == MODE_REJECT);
  const unsigned char* drow =
      two ? P.Ld + (size_t(b) * P.gamma + r.k) * size_t(V) * E::ES : nullptr;
  auto sub_lo = [&](int q) { return (q / GW) * P.ch2 + (q % GW) * P.sub; };
  auto sub_hi = [&](int q) { return min(sub_lo(q) + P.sub, min(V, (q / GW + 1) * P.ch2)); };
  // block-wide prefix of the warps' sums in wsum: the warp where the running
  // sum crosses tau (the last warp with mass if none) and the mass before it,
  // into sh_wsel / sh_before (thread 0)
  auto pick_warp = [&](FF tau) {
    if (threadIdx.x == 0) {
      FF base = ff(0.f), before = ff(0.f), before_last = ff(0.f);
      int sel = -1, last = -1;
      for (int w = 0; w < DRAW_WARPS; ++w) {
        const FF z = wsum[w];
        if (ff_pos(z)) {
          last = w;
          before_last = base;
          if (sel < 0 && ff_gt(base + z, tau)) { sel = w; before = base; }
        }
        base = base + z;
      }
      if (sel < 0) { sel = last < 0 ? 0 : last; before = before_last; }
      sh_wsel = sel;
      sh_before = before;
    }
    __syncthreads();
  };

  // 1. runs of sub-ranges: warp w takes [w * run, (w + 1) * run)
  bool degenerate = false;
  FF tot = ff(0.f);
  auto load_masses = [&]() {  // the rest of the run, and the run's sum
    tot = ff(0.f);
#pragma unroll
    for (int j = 0; j < DRAW_RUN; ++j) tot = tot + mq[j];
    for (int q = qa + lane + 32 * DRAW_RUN; q < qb; q += 32) {  // runs beyond 32 * DRAW_RUN
      const Mass m = ms[q];
      tot = tot + ff(m.hi, m.lo);
    }
  };
  auto target_masses = [&]() {  // degenerate case: masses of target row k, recomputed
    tot = ff(0.f);
    for (int j = 0; j < DRAW_RUN; ++j) mq[j] = ff(0.f);
    for (int q = qa; q < qb; ++q) {
      float h = 0.f, l = 0.f;
      if (sub_lo(q) < sub_hi(q)) span_mass<DT, true>(r, trow, nullptr, sub_lo(q), sub_hi(q), h, l);
      const int j = (q - qa) >> 5;
      if (lane == ((q - qa) & 31) && j < DRAW_RUN) mq[j] = ff(h, l);
      if (lane == 0) tot = tot + ff(h, l);
    }
  };
  auto block_total = [&]() {
    FF w = tot;
    warp_sum_ff(w.h, w.l);
    if (lane == 0) wsum[warp] = w;
    __syncthreads();
    FF z = ff(0.f);
    for (int k = 0; k < DRAW_WARPS; ++k) z = z + wsum[k];
    return z;
  };
  load_masses();
  FF Z = block_total();
  if (!ff_pos(Z)) {
    // the residual vanished in fp32: sample target row k instead (reading of
    // the Z = 0 case)
    degenerate = true;
    two = false;
    r.mode = MODE_TARGET;
    __syncthreads();
    target_masses();
    Z = block_total();
  }
  const FF tau = ff_mul(u, Z);
  pick_warp(tau);

  // 2. the crossing sub-range within the selected warp's run
  if (warp == sh_wsel) {
    const FF tau_w = tau - sh_before;
    FF base = ff(0.f), before = ff(0.f), before_last = ff(0.f);
    int qs = -1, qlast = qa;
    const int nj = run > 32 * DRAW_RUN ? (run + 31) / 32 : DRAW_RUN;
    for (int j = 0; j < nj && qs < 0; ++j) {
      const int q = qa + lane + 32 * j;
      FF z = ff(0.f);
      if (j < DRAW_RUN) {
#pragma unroll
        for (int jj = 0; jj < DRAW_RUN; ++jj)
          if (jj == j) z = mq[jj];
      } else if (!degenerate) {
        if (q < qb) {
          const Mass m = ms[q];
          z = ff(m.hi, m.lo);
        }
      } else {  // long runs, degenerate: recompute, one sub-range at a time
        for (int L = 0; L < 32; ++L) {
          const int qq = qa + L + 32 * j;
          float hh = 0.f, hl = 0.f;
          if (qq < qb && sub_lo(qq) < sub_hi(qq))
            span_mass<DT, true>(r, trow, nullptr, sub_lo(qq), sub_hi(qq), hh, hl);
          if (lane == L) z = ff(hh, hl);
        }
      }
      if (q >= qb) z = ff(0.f);
      FF incl = z;
      warp_scan_ff(incl.h, incl.l, lane);
      const bool posz = q < qb && ff_pos(z);
      const unsigned pos = __ballot_sync(0xffffffffu, posz);
      if (pos) {
        const int lp = 31 - __clz(pos);
        qlast = qa + 32 * j + lp;
        before_last = base + ff_shfl(incl - z, lp);
      }
      const unsigned hit = __ballot_sync(0xffffffffu, posz && ff_gt(base + incl, tau_w));
      if (hit) {
        const int l0 = __ffs(hit) - 1;
        qs = qa + 32 * j + l0;
        before = base + ff_shfl(incl - z, l0);
      }
      base = base + ff_shfl(incl, 31);
    }
    if (qs < 0) { qs = qlast; before = before_last; }
    if (lane == 0) {
      sh_q = qs;
      sh_rest = tau_w - before;  // what remains to cross inside the sub-range
    }
  }
  __syncthreads();

  // 3. the sub-range's elements in DRAW_WARPS slices of whole 8-element runs
  const int q = sh_q;
  const int lo = sub_lo(q), hi = sub_hi(q);
  const FF tau_q = sh_rest;
  const int nrun = (hi - lo + 7) / 8;                          // runs of 8 elements
  const int per_warp = (nrun + DRAW_WARPS - 1) / DRAW_WARPS;   // runs per warp
  const int ra = min(nrun, warp * per_warp), rb = min(nrun, ra + per_warp);
  constexpr int RUNS = 2;  // runs per lane held (slices of up to 64 runs = 512 elements)
  static_assert((GeoResidual::HALF / 2 + GW - 1) / GW + 8 <= DRAW_WARPS * 32 * RUNS * 8,
                "slice size");
  float w[RUNS][8];
  tot = ff(0.f);
#pragma unroll
  for (int j = 0; j < RUNS; ++j) {
    const int rr = ra + lane + 32 * j;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int el = lo + rr * 8 + e;
      w[j][e] = (rr < rb && el < hi)
                    ? weight(r, E::load(trow, el), two ? E::load(drow, el) : 0.f)
                    : 0.f;
      ff_add(tot.h, tot.l, w[j][e]);
    }
  }
  __syncthreads();  // wsum is reused
  block_total();
  pick_warp(tau_q);
  if (warp == sh_wsel) {
    const FF tau_s = tau_q - sh_before;
    FF base = ff(0.f);
    int tok = -1, last_pos = -1;
    for (int j = 0; j < RUNS && tok < 0; ++j) {
      const int rr = ra + lane + 32 * j;
      FF rs = ff(0.f);
      for (int e = 0; e < 8; ++e) {
        ff_add(rs.h, rs.l, w[j][e]);
        if (w[j][e] > 0.f) last_pos = lo + rr * 8 + e;
      }
      FF incl = rs;
      warp_scan_ff(incl.h, incl.l, lane);
      const unsigned hit =
          __ballot_sync(0xffffffffu, rr < rb && ff_pos(rs) && ff_gt(base + incl, tau_s));
      if (hit) {
        const int l0 = __ffs(hit) - 1;
        if (lane == l0) {
          FF acc = base + (incl - rs);
          int v = -1, lp = -1;
          for (int e = 0; e < 8; ++e) {
            ff_add(acc.h, acc.l, w[j][e]);
            if (w[j][e] > 0.f) lp = lo + rr * 8 + e;
            if (ff_gt(acc, tau_s)) { v = lo + rr * 8 + e; break; }
          }
          tok = (v >= 0) ? v : lp;
        }
        tok = __shfl_sync(0xffffffffu, tok, l0);
      }
      base = base + ff_shfl(incl, 31);
    }
    if (tok < 0) {  // rounding: the last element with mass in the slice
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        last_pos = max(last_pos, __shfl_xor_sync(0xffffffffu, last_pos, o));
      tok = last_pos < 0 ? lo : last_pos;
    }
    if (lane == 0) {
      P.out_tokens[size_t(b) * R + r.k] = tok;
      // the masses leave out the row's 1/S_t (a common factor)
      if (P.out_Z) P.out_Z[b] = float((double(Z.h) + double(Z.l)) *
                                      (double(r.ist_hi) + double(r.ist_lo)));
      if (degenerate) set_status(P, SV_ST_DEGENERATE);
    }
  }
  // the last kernel of a sampling call: the workspace is ready for the next one
  if (last_cta && threadIdx.x == 0) ready_for_next_call(P);
}

// ------------------------------------------- decide + residual + draw, fused

// The decision, the residual mass and the draw of one request in one kernel,
// for batches small enough that each request can have a cluster of CTAs:
// at a few dozen requests the three kernels above cost more in launches and
// hand-offs than in streaming the row pair.  One cluster of c CTAs per request:
//   1. every CTA combines the request's partials and takes the decision (the
//      same values in the same order in every CTA, so the same decision; the
//      outputs other than token k are written by each, with equal values);
//   2. the row token k is drawn from (with the draft row after a rejection)
//      is split into FIN_WARPS * c contiguous segments of whole 8-element
//      runs, one per warp of the cluster, each warp the mass of its segment
//      (the residual kernel's arithmetic), into shared memory;
//   3. after a cluster barrier every CTA reads all segment masses through
//      distributed shared memory in index order: Z, the segment where the
//      running mass crosses tau = u * Z (the last with mass if none), and what
//      remains of tau inside it;
//   4. the CTA owning that segment splits it over its warps, finds the
//      crossing slice by a block prefix, and that slice's warp scans it in
//      index order.
// A residual that sums to 0 is replaced by target row k (steps 2 and 3 again,
// SV_ST_DEGENERATE).
constexpr int FIN_WARPS = 16;
constexpr int FIN_MAXC = 8;  // CTAs per cluster (the portable limit)
// automatic choice for batches of at least two SMs per request: the whole call
// in one kernel (sv_onecall) rather than the reduce and the fused tail
constexpr bool ONECALL_AUTO = false;
// the same for greedy calls (the argmax reduce and the decision in one kernel)
constexpr bool ONECALL_GREEDY_AUTO = false;

// Bulk prefetch of [p, p + bytes) into L2 (p and bytes multiples of 16).
__device__ __forceinline__ void prefetch_l2(const void* p, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Steps 1-4 for request b of this CTA's cluster, the request's partials in
// P.part (NC: written by an earlier kernel; else by this cluster, visible
// after a cluster barrier).  The decision inputs and the given draft
// normalisers (dst_sh) were loaded by the caller.
template <int DT, bool NC>
__device__ void finish_request(const Params& P, const float2* dst_sh, float lt, float ld, float u,
                               bool tok_ok, int xi) {
  using E = Elem<DT>;
  __shared__ RowStat rows[MAXR];
  __shared__ Cand cand[MAXR];
  __shared__ int2 mode_k;
  __shared__ Record rec;
  __shared__ FF seg_mass[2][FIN_WARPS];  // [pass][warp]: read by every CTA of the cluster
  __shared__ FF wsum[FIN_WARPS];
  __shared__ FF sh_rest, sh_before, sh_Z;
  __shared__ int sh_seg, sh_wsel, sh_degen;
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int c = int(cluster.num_blocks()), q = int(cluster.block_rank());
  const int b = int(blockIdx.x) / c;
  const int warp = int(threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int g = P.gamma, R = P.R, V = P.V;
  const int nseg = FIN_WARPS * c;
  const float kf = LOG2E_F / __ldg(P.temp + b);

  // 1. rows and decision
  combine_rows<FIN_WARPS, NC>(P, b, kf, dst_sh, rows);
  __syncthreads();
  if (warp == 1) record_candidates(P, b, rows, cand);
  if (warp == 0) {
    const int2 mk = decide_sample<DT>(P, b, rows, lt, ld, u, tok_ok, xi);
    if (lane == 0) mode_k = mk;
  }
  __syncthreads();
  if (threadIdx.x == 0) rec = make_record(P, b, mode_k.x, mode_k.y, rows, cand);
  __syncthreads();
  Record r = rec;
  if (r.mode == MODE_INVALID) return;  // the same in every CTA: none reaches a cluster barrier

  const float ur = __ldg(P.u_res + size_t(b) * R + r.k);
  const int rowk = (r.mode == MODE_BONUS) ? g : r.k;
  const unsigned char* trow = P.Lt + (size_t(b) * R + rowk) * size_t(V) * E::ES;
  const unsigned char* drow =
      (r.mode == MODE_REJECT) ? P.Ld + (size_t(b) * g + r.k) * size_t(V) * E::ES : nullptr;
  const long long nrun = (V + 7) / 8;
  auto seg_lo = [&](int s) { return int(min((long long)V, nrun * s / nseg * 8)); };

  // 2 and 3 (twice if the residual vanished)
  bool degenerate = false;
  for (int pass = 0; pass < 2; ++pass) {
    {
      const int s = q * FIN_WARPS + warp;
      const int lo = seg_lo(s), hi = seg_lo(s + 1);
      // the segment into L2 at once, so that the warp's later load batches hit it
      const unsigned pf = unsigned(hi - lo) * E::ES & ~15u;
      if (pass == 0 && lane == 0 && pf > 0) {
        const unsigned char* pt = trow + size_t(lo) * E::ES;
        if ((reinterpret_cast<uintptr_t>(pt) & 15u) == 0) prefetch_l2(pt, pf);
        if (drow) {
          const unsigned char* pd = drow + size_t(lo) * E::ES;
          if ((reinterpret_cast<uintptr_t>(pd) & 15u) == 0) prefetch_l2(pd, pf);
        }
      }
      float h = 0.f, l = 0.f;
      if (lo < hi) span_mass<DT>(r, trow, drow, lo, hi, h, l);
      if (lane == 0) seg_mass[pass][warp] = ff(h, l);
    }
    cluster.sync();
    if (warp == 0) {
      // lane j holds segments 4 j .. 4 j + 3 (nseg <= 4 * 32)
      FF t[4], run = ff(0.f);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int s = 4 * lane + j;
        t[j] = ff(0.f);
        if (s < nseg) {
          const FF* src = cluster.map_shared_rank(&seg_mass[pass][0], s / FIN_WARPS);
          t[j] = src[s % FIN_WARPS];
        }
        run = run + t[j];
      }
      FF incl = run;
      warp_scan_ff(incl.h, incl.l, lane);
      const FF Z = ff_shfl(incl, 31);
      const bool degen = !ff_pos(Z);
      const FF tau = ff_mul(ur, Z);
      // the first segment with mass whose running total exceeds tau, else
      // the last segment with mass
      FF before = incl - run;  // mass of the segments before this lane's four
      int hit = INT_MAX, lastpos = -1;
      FF hit_before = ff(0.f), last_before = ff(0.f);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int s = 4 * lane + j;
        if (s < nseg && ff_pos(t[j])) {
          if (hit == INT_MAX && ff_gt(before + t[j], tau)) {
            hit = s;
            hit_before = before;
          }
          lastpos = s;
          last_before = before;
        }
        before = before + t[j];
      }
      const unsigned hits = __ballot_sync(0xffffffffu, hit != INT_MAX);
      const unsigned poss = __ballot_sync(0xffffffffu, lastpos >= 0);
      const int src_lane = hits ? __ffs(hits) - 1 : (poss ? 31 - __clz(poss) : 0);
      const int seg = __shfl_sync(0xffffffffu, hits ? hit : (lastpos >= 0 ? lastpos : 0), src_lane);
      const FF bef = ff_shfl(hits ? hit_before : last_before, src_lane);
      if (lane == 0) {
        sh_degen = degen && pass == 0;
        sh_seg = seg;
        sh_Z = Z;
        // past the last segment's total: aim at its last element with mass
        sh_rest = hits ? tau - bef : ff(INFINITY);
      }
    }
    __syncthreads();
    if (!sh_degen) break;
    // the residual vanished in fp32: draw from target row k instead
    degenerate = true;
    r.mode = MODE_TARGET;
    drow = nullptr;
  }
  // no CTA leaves while a peer may still read its segment masses
  cluster_arrive();

  // 4. the owner of the crossing segment finds the token
  const int sg = sh_seg;
  if (q == sg / FIN_WARPS) {
    const int lo = seg_lo(sg), hi = seg_lo(sg + 1);
    const int nr = (hi - lo + 7) / 8;
    const int per = (nr + FIN_WARPS - 1) / FIN_WARPS;
    const int a = min(hi, lo + min(nr, warp * per) * 8);
    const int e = min(hi, lo + min(nr, warp * per + per) * 8);
    // the slice's weights in batches of 32 * 8 elements (element i0 + lane +
    // 32 j in w[j]); the first batch stays in registers for the scan below
    FF s = ff(0.f);
    float w0[8];
    for (int i0 = a; i0 < e; i0 += 32 * 8) {
      float w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // the batch's loads first
        const int i = i0 + lane + 32 * j;
        w[j] = i < e ? weight(r, E::load(trow, i), drow ? E::load(drow, i) : 0.f) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        ff_add(s.h, s.l, w[j]);
        if (i0 == a) w0[j] = w[j];
      }
    }
    warp_sum_ff(s.h, s.l);
    if (lane == 0) wsum[warp] = s;
    __syncthreads();
    const FF rest = sh_rest;
    if (threadIdx.x == 0) {
      FF base = ff(0.f), before = ff(0.f), before_last = ff(0.f);
      int sel = -1, last = -1;
      for (int w = 0; w < FIN_WARPS; ++w) {
        const FF z = wsum[w];
        if (ff_pos(z)) {
          last = w;
          before_last = base;
          if (sel < 0 && ff_gt(base + z, rest)) { sel = w; before = base; }
        }
        base = base + z;
      }
      if (sel < 0) { sel = last < 0 ? 0 : last; before = before_last; }
      sh_wsel = sel;
      sh_before = before;
    }
    __syncthreads();
    if (warp == sh_wsel) {
      const FF tau_s = rest - sh_before;
      FF base = ff(0.f);
      int tok = -1, last_pos = -1;
      // tiles of 32 elements in index order: the first eight from registers
      auto tile = [&](int i0, float w) {
        FF incl = ff(w);
        warp_scan_ff(incl.h, incl.l, lane);
        incl = base + incl;
        const unsigned h = __ballot_sync(0xffffffffu, w > 0.f && ff_gt(incl, tau_s));
        const unsigned pv = __ballot_sync(0xffffffffu, w > 0.f);
        if (h) tok = i0 + __ffs(h) - 1;
        if (pv) last_pos = i0 + 31 - __clz(pv);
        base = ff_shfl(incl, 31);
      };
      if (a < e) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (tok < 0) tile(a + 32 * j, w0[j]);
      }
      for (int i0 = a + 32 * 8; i0 < e && tok < 0; i0 += 32) {  // slices past 256 elements
        const int i = i0 + lane;
        tile(i0, i < e ? weight(r, E::load(trow, i), drow ? E::load(drow, i) : 0.f) : 0.f);
      }
      if (tok < 0) tok = last_pos < 0 ? lo : last_pos;  // rounding: the last element with mass
      if (lane == 0) {
        P.out_tokens[size_t(b) * R + r.k] = tok;
        // the masses leave out the row's 1/S_t (a common factor)
        const FF Z = sh_Z;
        if (P.out_Z) P.out_Z[b] = float((double(Z.h) + double(Z.l)) *
                                        (double(r.ist_hi) + double(r.ist_lo)));
        if (degenerate) set_status(P, SV_ST_DEGENERATE);
      }
    }
  }
  cluster_wait();
}

template <int DT>
__global__ void __launch_bounds__(32 * FIN_WARPS, 1) sv_finish(const Params P) {
  __shared__ float2 dst_sh[MAXR];
  const int b = int(blockIdx.x) / int(cooperative_groups::this_cluster().num_blocks());
  const int g = P.gamma;
  // the call's inputs, before the wait
  float lt, ld, u;
  bool tok_ok;
  int xi;
  load_decision_inputs<DT>(P, b, lt, ld, u, tok_ok, xi);
  if (P.dstats != nullptr && int(threadIdx.x) < g)
    dst_sh[threadIdx.x] = __ldg(reinterpret_cast<const float2*>(P.dstats) + size_t(b) * g +
                                threadIdx.x);
  // the next call's reduce may be placed as SMs free up: it waits for this
  // grid's completion before it reads anything
  allow_next_kernel();
  wait_previous_kernel();  // the partials
  // the reduce has completed: the control block is ready for the next call
  if (blockIdx.x == 0 && threadIdx.x == 0) ready_for_next_call(P);
  __syncthreads();
  finish_request<DT, true>(P, dst_sh, lt, ld, u, tok_ok, xi);
}

// CTA q of c's share of request b's chunks, when the request's cluster
// streams it: like the reduce's split over the whole grid, equal parts of
// the first (POOL_DIV - 1) / POOL_DIV of the request's weight, the rest a
// pool of units the cluster's CTAs claim once their part is nearly done.
__device__ __forceinline__ Split request_split(const Params& P, int b, int q, int c) {
  const long long w_req = (long long)P.nch1 * (P.R + P.gs);
  const long long w0 = (long long)b * w_req;
  const long long Ws = w_req - w_req / POOL_DIV;
  Split sp;
  sp.t0 = task_at_weight(P, w0 + (Ws * q + c - 1) / c);
  sp.t1 = task_at_weight(P, w0 + (Ws * (q + 1) + c - 1) / c);
  sp.ts = task_at_weight(P, w0 + Ws);
  const long long pool = (long long)(b + 1) * P.R * P.nch1 - sp.ts;
  sp.unit = max(1LL, (pool + 2LL * c - 1) / (2LL * c));  // about two units per CTA
  sp.nunits = (pool + sp.unit - 1) / sp.unit;
  return sp;
}

// The whole call in one kernel, for batches that leave at least two SMs per
// request: one cluster of c CTAs per request streams the request's rows
// (this CTA's share of its chunks through the reduce's ring: producer lane,
// consumer warps 1..NCW, per-warp partials into P.part), then, after a
// cluster barrier, takes the decision, the residual mass and the draw as the
// fused tail does.  The rows token k is drawn from were streamed by the same
// cluster moments before, so that second pass reads them from L2.  The last
// CTA to finish (counted in the control block's pad[2]) puts the workspace
// back in its ready state.
template <int DT, bool GREEDY, bool PAIRS>
__global__ void __launch_bounds__(32 * FIN_WARPS, 1) sv_onecall(const Params P) {
  using G = GeoReduce;
  static_assert(FIN_WARPS >= NCW + 1, "a producer warp and the consumer warps");
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* slots = smem;
  SmemCtl<G>& C = *reinterpret_cast<SmemCtl<G>*>(smem + size_t(G::NS) * G::SLOT);
  __shared__ float2 dst_sh[MAXR];
  cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
  const int c = int(cluster.num_blocks()), q = int(cluster.block_rank());
  const int b = int(blockIdx.x) / c;
  const int warp = int(threadIdx.x >> 5), g = P.gamma;
  __shared__ unsigned long long pool_ctr;  // rank 0's counts the cluster's pool claims
  if (threadIdx.x == 0) {
    C.abort = 0;
    for (int s = 0; s < G::NS; ++s) {
      mbar_init(&C.full[s], 1);
      mbar_init(&C.empty[s], G::GW);
    }
    pool_ctr = 0ull;
  }
  // the counter is zero in every CTA before any CTA of the cluster claims
  // (the barrier completes below, after the wait for the previous kernel)
  cluster_arrive();
  // the next call's first kernel waits for this grid's completion
  allow_next_kernel();
  // launched programmatically after the previous kernel in the stream
  // (whatever wrote the logits, or an earlier call): nothing it wrote is
  // read before it has completed, the call's inputs included
  wait_previous_kernel();
  // the control block's ready state (only the state word is tested here; the
  // counters are checked by the last CTA to finish).  A workspace found busy
  // also gets its finish count cleared: no CTA of this grid can have counted
  // itself before block 0 starts, as each counts only after its request.
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (P.ctrl->state != 0ull) {
      set_status(P, SV_ST_WORKSPACE);
      P.ctrl->pad[2] = 0ull;
    }
    P.ctrl->state = 1ull;
  }
  // the decision's inputs: loaded now, used after the stream
  float lt, ld, u;
  bool tok_ok;
  int xi;
  lt = ld = u = 0.f;
  tok_ok = true;
  xi = -1;
  if (!GREEDY) load_decision_inputs<DT>(P, b, lt, ld, u, tok_ok, xi);
  if (!GREEDY && P.dstats != nullptr && int(threadIdx.x) < g)
    dst_sh[threadIdx.x] = __ldg(reinterpret_cast<const float2*>(P.dstats) + size_t(b) * g +
                                threadIdx.x);
  cluster_wait();
  __syncthreads();
  if (warp == 0) {
    if (threadIdx.x == 0)
      producer<DT, GREEDY, PAIRS>(P, C, slots, request_split(P, b, q, c),
                                  cluster.map_shared_rank(&pool_ctr, 0), nullptr);
  } else if (warp <= NCW) {
    consumer<DT, GREEDY, PAIRS, false>(P, C, slots);
  }
  __syncthreads();
  cluster.sync();  // every CTA's partials of the request are written
  if (GREEDY) {
    // the rows' argmaxes over the cluster's partials and the decision, by
    // the cluster's first CTA (as the decide kernel takes them)
    __shared__ RowStat rows[MAXR];
    if (q == 0) {
      const int lane = threadIdx.x & 31;
      for (int i = warp; i < P.R; i += FIN_WARPS) {
        const Partial* pp = P.part + (size_t(b) * P.R + i) * size_t(P.np1);
        float best;
        int bi, nan;
        row_argmax<false>(pp, P.np1, best, bi, nan);
        if (lane == 0) {
          RowStat r;
          r.mt = best; r.md = 0.f; r.St_h = r.St_l = r.Sd_h = r.Sd_l = 0.f;
          r.bad = (nan || bi == INT_MAX || best == INFINITY) ? SV_ST_NONFINITE : 0;
          r.amax = bi;
          rows[i] = r;
        }
      }
      __syncthreads();
      if (warp == 0) decide_greedy(P, b, rows);
    }
  } else {
    finish_request<DT, false>(P, dst_sh, lt, ld, u, tok_ok, xi);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&P.ctrl->pad[2], 1ull) == (unsigned long long)gridDim.x - 1ull) {
      __threadfence();
      // this path takes no pool units and no chunk claims: counters left
      // non-zero by another call's work mean the workspace was not ready
      if (P.ctrl->claims != 0ull || P.ctrl->pad[1] != 0ull) set_status(P, SV_ST_WORKSPACE);
      P.ctrl->claims = 0ull;
      P.ctrl->pad[0] = 0ull;
      P.ctrl->pad[1] = 0ull;
      P.ctrl->pad[2] = 0ull;
      P.ctrl->state = 0ull;
    }
  }
}

// ---------------------------------------------------------- draft sampling

// Block-wide inclusive prefix of float pairs in thread order (all threads of
// the CTA take part); `total` gets the CTA's sum.  wsum holds one entry per
// warp; the CTA synchronises twice.
template <int NW>
__device__ FF block_scan_ff(FF v, FF* wsum, FF& total) {
  const int warp = int(threadIdx.x >> 5), lane = threadIdx.x & 31;
  FF incl = v;
  warp_scan_ff(incl.h, incl.l, lane);
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  FF off = ff(0.f), tot = ff(0.f);
  for (int w = 0; w < NW; ++w) {
    if (w < warp) off = off + wsum[w];
    tot = tot + wsum[w];
  }
  __syncthreads();
  total = tot;
  return off + incl;
}

// Mass of the reduce's partial q of a row (a consumer warp's sum over its
// span) relative to the row maximum m, as a float.
__device__ __forceinline__ float partial_mass(const Partial* pp, int q, float m, float kf) {
  const float4 v = __ldg(reinterpret_cast<const float4*>(pp + q));
  return (m == -INFINITY) ? v.y : v.y * ex2((v.x - m) * kf);
}

// Element span [lo, hi) of a row that the reduce's partial q covers (chunk
// q / GW, consumer warp q % GW), as load_share assigns it: the warp's run of
// the chunk's aligned body, with the unaligned head on warp 0 and the tail on
// warp GW - 1.
template <int DT>
__device__ __forceinline__ void partial_span(const Params& P, const unsigned char* row, int q,
                                             int& lo, int& hi) {
  using E = Elem<DT>;
  constexpr int GW = GeoReduce::GW;
  const int c = q / GW, w = q - c * GW;
  const int e0 = c * P.ch1, n = min(P.ch1, P.V - e0);
  int head, nb;
  split<DT>(row + size_t(e0) * E::ES, n, head, nb);
  const int nv = nb / E::VEC, pw = (nv + GW - 1) / GW;
  const int v0 = min(nv, w * pw), v1 = min(nv, (w + 1) * pw);
  lo = (w == 0) ? e0 : e0 + head + v0 * E::VEC;
  hi = (w == GW - 1) ? e0 + n : e0 + head + v1 * E::VEC;
}

// a partial's span: a warp's run of at most ceil(HALF / 16 / GW) vectors plus
// a head or tail shorter than a vector, and a vector of margin
constexpr int SAMPLE_STAGE =
    ((GeoReduce::HALF / 16 + GeoReduce::GW - 1) / GeoReduce::GW) * 16 + 48;
constexpr int SAMPLE_KV = (SAMPLE_STAGE / 16 + 32 * SAMPLE_WARPS - 1) / (32 * SAMPLE_WARPS);

// Draft-token sampling, one CTA per draft row (row r = b * R + i of the
// reduce's rows): the row's maximum and normaliser S from the reduce's
// partials, the partial (a contiguous span of the row) where the running mass
// crosses tau = u * S, scanned over the partials in index order, then that
// span's elements, staged in shared memory: each thread sums a contiguous
// run of weights, a block prefix finds the crossing run, whose thread scans
// it in index order.  Writes the token and the row's (max, S) to column
// col + i of request b.
template <int DT>
__global__ void __launch_bounds__(32 * SAMPLE_WARPS) sv_sample(const Params P) {
  using E = Elem<DT>;
  constexpr int NW = SAMPLE_WARPS, NT = 32 * NW;
  __shared__ FF wsum[NW];
  __shared__ float wmax[NW];
  __shared__ FF sh_rest, sh_rest_last;
  __shared__ int sh_hit, sh_last, sh_tok_hit, sh_tok_last;
  __shared__ __align__(16) unsigned char stage[SAMPLE_STAGE];
  const int r = int(blockIdx.x), tid = int(threadIdx.x);
  const int warp = tid >> 5, lane = tid & 31;
  const int b = r / P.R, i = r - b * P.R;
  const size_t o = size_t(b) * P.ncols + P.col + i;
  // inputs, loaded before the wait for the partials
  const float u = __ldg(P.u_res + r);
  const float T = __ldg(P.temp + b);
  const bool t_ok = isfinite(T) && T >= 0x1p-126f;
  const float kf = LOG2E_F / T;
  if (tid == 0) {
    sh_hit = INT_MAX;
    sh_last = -1;
    sh_tok_hit = INT_MAX;
    sh_tok_last = -1;
  }
  allow_next_kernel();  // the next call's reduce waits for this grid's completion
  wait_previous_kernel();
  const Partial* pp = P.part + size_t(r) * P.np1;
  const int np = P.np1;
  // at most one partial per thread (the usual case): each thread loads its
  // partial once, and the scan that gives S below is also the scan of the
  // partials in index order that step 3 needs
  const bool one_round = np <= NT;
  float4 pv = make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
  if (one_round && tid < np) pv = __ldg(reinterpret_cast<const float4*>(pp + tid));
  // 1. the row maximum over the partials' maxima (NaN shows in the sums)
  float m = -INFINITY;
  if (one_round)
    m = fmaxf(m, pv.x);
  else
    for (int q = tid; q < np; q += NT) m = fmaxf(m, __ldg(&pp[q].a));
  m = warp_max(m);
  if (lane == 0) wmax[warp] = m;
  __syncthreads();
  m = wmax[0];
  for (int w = 1; w < NW; ++w) m = fmaxf(m, wmax[w]);
  // 2. the normaliser S, the sum of the partials' masses
  FF part = ff(0.f);
  if (one_round) {
    if (tid < np) ff_add(part.h, part.l, (m == -INFINITY) ? pv.y : pv.y * ex2((pv.x - m) * kf));
  } else {
    for (int q = tid; q < np; q += NT) ff_add(part.h, part.l, partial_mass(pp, q, m, kf));
  }
  FF S;
  const FF incl_part = block_scan_ff<NW>(part, wsum, S);
  const double Sd = ff_val(S.h, S.l);
  const bool ok = t_ok && row_ok(m, Sd);  // the same in every thread
  if (!ok) {
    if (tid == 0) {
      P.out_tokens[o] = -1;
      P.out_stats[2 * o] = NAN;
      P.out_stats[2 * o + 1] = NAN;
      set_status(P, t_ok ? SV_ST_NONFINITE : SV_ST_BAD_TEMP);
      if (r == 0) ready_for_next_call(P);
    }
    return;
  }
  // 3. the crossing partial, in rounds of NT partials (with one round, from
  // the scan of step 2: thread q holds partial q alone)
  const FF tau = ff_mul(u, S);
  FF base = ff(0.f);
  if (one_round) {
    const int q = tid;
    const FF z = part;
    const bool pos = q < np && ff_pos(z);
    if (pos && ff_gt(base + incl_part, tau)) atomicMin(&sh_hit, q);
    if (pos) atomicMax(&sh_last, q);
    __syncthreads();
    if (q == sh_hit) sh_rest = tau - (base + (incl_part - z));
    if (q == sh_last) sh_rest_last = z;
  }
  for (int q0 = 0; !one_round && q0 < np; q0 += NT) {
    const int q = q0 + tid;
    const FF z = ff(q < np ? partial_mass(pp, q, m, kf) : 0.f);
    FF rtot;
    const FF incl = block_scan_ff<NW>(z, wsum, rtot);
    const bool pos = q < np && ff_pos(z);
    if (pos && ff_gt(base + incl, tau)) atomicMin(&sh_hit, q);
    if (pos) atomicMax(&sh_last, q);
    __syncthreads();
    if (q == sh_hit) sh_rest = tau - (base + (incl - z));
    if (q == sh_last) sh_rest_last = z;  // the span's whole mass: its last element
    if (sh_hit != INT_MAX) break;        // the same in every thread
    base = base + rtot;
    __syncthreads();                     // sh_last is read above before the next round's updates
  }
  __syncthreads();
  const bool hit = sh_hit != INT_MAX;
  const int qs = hit ? sh_hit : sh_last;
  const FF rest = hit ? sh_rest : sh_rest_last;
  // 4. the span's elements, staged in shared memory: the body with 16-byte
  // loads, an unaligned head and tail element by element; element e sits at
  // stage index VEC + (e - a), a the span's first element on a 16-byte
  // boundary
  Record rr;
  rr.k = 0; rr.mode = MODE_BONUS; rr.mt = m; rr.kf = kf;
  rr.ist_hi = rr.ist_lo = rr.c0_hi = rr.c0_lo = 0.f;
  const unsigned char* row = P.Lt + size_t(r) * size_t(P.V) * E::ES;
  int lo, hi;
  partial_span<DT>(P, row, qs, lo, hi);
  int head, nbody;
  split<DT>(row + size_t(lo) * E::ES, hi - lo, head, nbody);
  const int a = lo + head, nvec = nbody / E::VEC;
  {
    const uint4* gv = reinterpret_cast<const uint4*>(row + size_t(a) * E::ES);
    uint4* sv = reinterpret_cast<uint4*>(stage);
    uint4 buf[SAMPLE_KV];
#pragma unroll
    for (int k = 0; k < SAMPLE_KV; ++k) {
      const int j = tid + k * NT;
      if (j < nvec) buf[k] = __ldg(gv + j);
    }
#pragma unroll
    for (int k = 0; k < SAMPLE_KV; ++k) {
      const int j = tid + k * NT;
      if (j < nvec) sv[1 + j] = buf[k];
    }
    for (int e = lo + tid; e < a; e += NT) E::sts(stage, E::VEC + (e - a), E::load(row, e));
    for (int e = a + nbody + tid; e < hi; e += NT)
      E::sts(stage, E::VEC + (e - a), E::load(row, e));
  }
  __syncthreads();
  // a contiguous run of the span per thread
  const int per = (hi - lo + NT - 1) / NT;
  const int a0 = min(hi, lo + tid * per), a1 = min(hi, a0 + per);
  FF run = ff(0.f);
  int lastpos = -1;
  for (int e = a0; e < a1; ++e) {
    const float w = weight(rr, E::lds(stage, E::VEC + (e - a)), 0.f);
    ff_add(run.h, run.l, w);
    if (w > 0.f) lastpos = e;
  }
  FF rtot;
  const FF incl = block_scan_ff<NW>(run, wsum, rtot);
  if (a0 < a1 && ff_pos(run) && ff_gt(incl, rest)) atomicMin(&sh_tok_hit, tid);
  if (lastpos >= 0) atomicMax(&sh_tok_last, lastpos);
  __syncthreads();
  if (tid == sh_tok_hit) {
    FF acc = incl - run;
    int tok = lastpos;
    for (int e = a0; e < a1; ++e) {
      const float w = weight(rr, E::lds(stage, E::VEC + (e - a)), 0.f);
      ff_add(acc.h, acc.l, w);
      if (ff_gt(acc, rest)) { tok = e; break; }
    }
    P.out_tokens[o] = tok;
  } else if (sh_tok_hit == INT_MAX && tid == 0) {  // rounding: the span's last element with mass
    P.out_tokens[o] = sh_tok_last < 0 ? lo : sh_tok_last;
  }
  if (tid == 0) {
    P.out_stats[2 * o] = m;
    P.out_stats[2 * o + 1] = float(Sd);
    if (r == 0) ready_for_next_call(P);
  }
}

// ---------------------------------------------------------------- host

struct Tuning {
  int chunk = 0;
  int tail = 0;  // 0: automatic, 1: decide/residual/draw, 2: fused tail, 3: one kernel (sv_set_tail)
  int withhold_slot = 0;         // failure-handling test (sv_test_withhold_slot)
  cudaEvent_t stage_ev[5] = {};  // profiling: events recorded around the kernels
  int stage_n = 0;
};
Tuning g_tune;

struct DevCache {
  bool init = false;
  int sms = 0;
};
std::mutex g_mu;
DevCache g_dev[64];

template <int DT>
bool prepare_kernel() {
  const int r = int(smem_bytes<GeoReduce>());
  if (cudaFuncSetAttribute(sv_onecall<DT, false, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, r) != cudaSuccess ||
      cudaFuncSetAttribute(sv_onecall<DT, false, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, r) != cudaSuccess ||
      cudaFuncSetAttribute(sv_onecall<DT, true, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, r) != cudaSuccess)
    return false;
  return cudaFuncSetAttribute(sv_residual<DT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(smem_bytes<GeoResidual>())) == cudaSuccess &&
         cudaFuncSetAttribute(sv_residual<DT, false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(smem_bytes<GeoResidual>())) == cudaSuccess &&
         cudaFuncSetAttribute(sv_reduce<DT, false, false, false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, r) == cudaSuccess &&
         cudaFuncSetAttribute(sv_reduce<DT, false, true, false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, r) == cudaSuccess &&
         cudaFuncSetAttribute(sv_reduce<DT, false, true, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, r) == cudaSuccess &&
         cudaFuncSetAttribute(sv_reduce<DT, true, true, false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, r) == cudaSuccess;
}

int device_info(int& sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DevCache& d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SV_ERR_CUDA;
    if (!prepare_kernel<SV_F32>() || !prepare_kernel<SV_BF16>())
      return SV_ERR_CUDA;
    d.init = true;
  }
  sms = d.sms;
  return SV_OK;
}

int round_up(long long x, int m) { return int(((x + m - 1) / m) * m); }

// Launch a kernel that follows another of the same call with programmatic
// stream serialisation: it may start before its predecessor ends and waits
// for it on the device (wait_previous_kernel).
template <typename... KArgs, typename... Args>
cudaError_t launch_after(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                         cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}
// The same, in clusters of `cluster` CTAs along x.
template <typename K>
cudaError_t launch_after_cluster(K kern, unsigned grid, unsigned block, unsigned cluster,
                                 cudaStream_t st, const Params& P, size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = cluster;
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

// One library call: which path, and its arguments as the C ABI gives them.
enum CallKind { CALL_SAMPLE = 0, CALL_GREEDY = 1, CALL_CACHED = 2, CALL_DRAFT = 3 };
struct Call {
  int kind = CALL_SAMPLE;
  const void* Lt = nullptr;   // target logits; the draft logits for CALL_DRAFT
  const void* Ld = nullptr;
  const int32_t* x = nullptr;
  const float* u_acc = nullptr;
  const float* u_res = nullptr;  // u_resample; u_draft for CALL_DRAFT
  const float* temp = nullptr;
  const float* dstats = nullptr;
  int B = 0, gamma = 0, V = 0, dtype = SV_F32;
  int n = 0;                  // CALL_DRAFT: rows per request
  int32_t* out_tokens = nullptr;
  int32_t* out_n = nullptr;
  float* out_p = nullptr;
  float* out_Z = nullptr;
  float* out_stats = nullptr;
  int col = 0, ncols = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  int32_t* status = nullptr;
  void* stream = nullptr;
};

int launch(const Call& a) {
  const bool greedy = a.kind == CALL_GREEDY, draft = a.kind == CALL_DRAFT;
  if (a.dtype != SV_F32 && a.dtype != SV_BF16) return SV_ERR_DTYPE;
  if (a.B < 0 || a.V < 1) return SV_ERR_INVALID_ARG;
  if (draft) {
    if (a.n < 1 || a.n > SV_MAX_GAMMA || a.col < 0 || a.ncols < a.col + a.n)
      return SV_ERR_INVALID_ARG;
  } else if (a.gamma < 0 || a.gamma > SV_MAX_GAMMA) {
    return SV_ERR_INVALID_ARG;
  }
  if (a.B == 0) return SV_OK;  // nothing to do; empty buffers may be NULL
  const int ES = a.dtype == SV_F32 ? 4 : 2;
  const int gamma = draft ? 0 : a.gamma;
  const int R = draft ? a.n : gamma + 1;
  if (!a.Lt || !a.out_tokens) return SV_ERR_INVALID_ARG;
  if (draft) {
    if (!a.u_res || !a.temp || !a.out_stats) return SV_ERR_INVALID_ARG;
  } else {
    if (!a.out_n || (!a.x && gamma > 0)) return SV_ERR_INVALID_ARG;
    if (!greedy && (!a.u_res || !a.temp || (gamma > 0 && (!a.Ld || !a.u_acc))))
      return SV_ERR_INVALID_ARG;
    if (a.kind == CALL_CACHED && gamma > 0 && !a.dstats) return SV_ERR_INVALID_ARG;
  }
  auto mis = [](const void* p, int al) {
    return p && (reinterpret_cast<uintptr_t>(p) % al) != 0;
  };
  if (mis(a.Lt, ES) || mis(a.Ld, ES) || mis(a.x, 4) || mis(a.u_acc, 4) || mis(a.u_res, 4) ||
      mis(a.temp, 4) || mis(a.dstats, 8) || mis(a.out_tokens, 4) || mis(a.out_n, 4) ||
      mis(a.out_p, 4) || mis(a.out_Z, 4) || mis(a.out_stats, 4) || mis(a.status, 4))
    return SV_ERR_INVALID_ARG;
  const int B = a.B, V = a.V;
  const Layout L = make_layout(B, R - 1, V);
  if (!a.ws || (reinterpret_cast<uintptr_t>(a.ws) & 255u) || a.ws_bytes < L.total)
    return SV_ERR_WORKSPACE;

  int sms = 0;
  int rc = device_info(sms);
  if (rc != SV_OK) return rc;
  const long long units = (long long)B * R;
  const int chmax = GeoReduce::HALF / ES;     // a phase-1 chunk fits half a slot
  const int chmax2 = GeoResidual::HALF / ES;  // phase 2 likewise

  // the tail after the reduce: for batches that leave at least two SMs per
  // request, one fused kernel with a cluster of fc CTAs per request
  int fc = 0;
  bool one = false;  // the whole call in one kernel (sv_onecall) with clusters of fc CTAs
  if (!greedy && !draft) {
    const int per = min(FIN_MAXC, sms / B);
    if (g_tune.tail == 2 || g_tune.tail == 3 || (g_tune.tail == 0 && per >= 2)) fc = max(1, per);
    one = fc > 0 && (g_tune.tail == 3 || (g_tune.tail == 0 && ONECALL_AUTO));
  } else if (greedy) {
    const int per = min(FIN_MAXC, sms / B);
    one = g_tune.tail == 3 || (g_tune.tail == 0 && ONECALL_GREEDY_AUTO && per >= 2);
    if (one) fc = max(1, per);
  }

  // phase-1 chunk: at most half a slot, at least CH1_MIN (or the whole row),
  // and small enough that every SM gets several tasks (in one-kernel calls:
  // that every CTA of a request's cluster gets two)
  int ch1;
  if (g_tune.chunk > 0) {
    ch1 = round_up(g_tune.chunk, 64);
  } else {
    const long long by_bytes = (V + chmax - 1) / chmax;
    const long long by_tasks = one ? (2LL * fc + R - 1) / R
                                   : (8LL * min(sms, SMS_CAP) + units - 1) / units;
    const long long want = max(1LL, max(by_bytes, by_tasks));
    ch1 = round_up((V + want - 1) / want, 64);
  }
  ch1 = min(chmax, max(ch1, min(CH1_MIN, round_up(V, 64))));
  if ((V + ch1 - 1) / ch1 > L.nch1_max)  // a tuning override asked for more chunks than fit
    ch1 = min(chmax, round_up((V + L.nch1_max - 1) / L.nch1_max, 64));
  const int nch1 = (V + ch1 - 1) / ch1;
  if (nch1 > L.nch1_max) return SV_ERR_INVALID_ARG;

  Params P;
  P.Lt = static_cast<const unsigned char*>(a.Lt);
  P.Ld = static_cast<const unsigned char*>(a.Ld);
  P.x = a.x; P.u_acc = a.u_acc; P.u_res = a.u_res; P.temp = a.temp;
  P.B = B; P.gamma = gamma; P.V = V; P.R = R;
  P.gs = (a.kind == CALL_SAMPLE) ? gamma : 0;  // draft rows the reduce streams
  P.dstats = (a.kind == CALL_CACHED && gamma > 0) ? a.dstats : nullptr;
  P.ch1 = ch1; P.nch1 = nch1;
  P.np1 = nch1 * GeoReduce::GW;
  P.tasks = (long long)B * R * nch1;
  P.ch2 = chmax2;
  P.nch2 = (V + chmax2 - 1) / chmax2;
  // each residual warp takes a contiguous sub-range of a phase-2 chunk, a
  // whole number of 16-byte vectors long (the last one may be shorter)
  P.sub = round_up((chmax2 + GeoResidual::GW - 1) / GeoResidual::GW, 8);
  P.out_tokens = a.out_tokens; P.out_n = a.out_n; P.out_p = a.out_p; P.out_Z = a.out_Z;
  P.out_stats = a.out_stats; P.col = a.col; P.ncols = a.ncols;
  P.withhold_slot = g_tune.withhold_slot;
  P.reduce_grid = int(min((long long)sms, P.tasks));
  P.status = a.status;
  unsigned char* w = static_cast<unsigned char*>(a.ws);
  P.ctrl = reinterpret_cast<Ctrl*>(w + L.ctrl);
  P.part = reinterpret_cast<Partial*>(w + L.part);
  P.rec = reinterpret_cast<Record*>(w + L.rec);
  P.mass = reinterpret_cast<Mass*>(w + L.mass);
  if ((long long)B * P.nch2 > 0x7fffffffLL || units > 0x7fffffffLL) return SV_ERR_INVALID_ARG;

  cudaStream_t st = static_cast<cudaStream_t>(a.stream);
  const unsigned grid = unsigned(min((long long)sms, P.tasks));
  const unsigned gres = unsigned(min((long long)sms, (long long)B * P.nch2));
  // profiling aid: event j after the j-th kernel (event 0 before the first)
  const Tuning& tu = g_tune;
  auto mark = [&](int j) {
    if (j < tu.stage_n) cudaEventRecord(tu.stage_ev[j], st);
  };
  mark(0);
  cudaError_t e = cudaSuccess;
  auto run = [&](auto reduce_k, auto decide_k, auto decide_small_k, auto residual_k, auto draw_k,
                 auto sample_k, auto finish_k, auto onecall_k) {
    if (one) {
      e = launch_after_cluster(onecall_k, unsigned(B) * unsigned(fc), 32 * FIN_WARPS,
                               unsigned(fc), st, P, smem_bytes<GeoReduce>());
      mark(1);
      return;
    }
    // programmatic launch: the reduce's CTAs may be placed while the previous
    // kernel in the stream finishes; it waits for that kernel on the device
    e = launch_after(reduce_k, grid, NTHR, smem_bytes<GeoReduce>(), st, P);
    mark(1);
    if (draft) {
      if (e == cudaSuccess)
        e = launch_after(sample_k, unsigned(units), 32 * SAMPLE_WARPS, 0, st, P);
      mark(2);
      return;
    }
    if (fc > 0) {
      if (e == cudaSuccess)
        e = launch_after_cluster(finish_k, unsigned(B) * unsigned(fc), 32 * FIN_WARPS,
                                 unsigned(fc), st, P, size_t(0));
      mark(2);
      return;
    }
    // one CTA per request; with at most four rows, four warps (a row each):
    // smaller CTAs, more of them resident at large batches
    if (e == cudaSuccess)
      e = R <= DECIDE_WARPS_SMALL
              ? launch_after(decide_small_k, unsigned(B), 32 * DECIDE_WARPS_SMALL, 0, st, P, greedy)
              : launch_after(decide_k, unsigned(B), 32 * DECIDE_WARPS, 0, st, P, greedy);
    mark(2);
    if (greedy) return;
    if (e == cudaSuccess) e = launch_after(residual_k, gres, NTHR, smem_bytes<GeoResidual>(), st, P);
    mark(3);
    if (e == cudaSuccess) e = launch_after(draw_k, unsigned(B), 32 * DRAW_WARPS, 0, st, P);
    mark(4);
  };
  // the reduce streams draft rows only for CALL_SAMPLE; the other paths pair
  // target chunks in its slots, and draft sampling needs contiguous shares
  // rows on 16-byte boundaries throughout: the residual kernel without the
  // unaligned-row path
  const bool aligned_rows = (uintptr_t(a.Lt) % 16 == 0) && (!a.Ld || uintptr_t(a.Ld) % 16 == 0) &&
                            (size_t(V) * ES) % 16 == 0;
  auto dispatch = [&](auto dt) {
    constexpr int D = decltype(dt)::value;
    auto go = [&](auto reduce_k, auto greedy_c, auto pairs_c) {
      constexpr bool GR = decltype(greedy_c)::value;
      constexpr bool PR = decltype(pairs_c)::value;  // the one-kernel path's slots: target pairs
      auto dk = sv_decide<D, GR, DECIDE_WARPS>;
      auto dks = sv_decide<D, GR, DECIDE_WARPS_SMALL>;
      auto ok = sv_onecall<D, GR, PR>;
      if (aligned_rows)
        run(reduce_k, dk, dks, sv_residual<D, true>, sv_draw<D>, sv_sample<D>, sv_finish<D>, ok);
      else
        run(reduce_k, dk, dks, sv_residual<D, false>, sv_draw<D>, sv_sample<D>, sv_finish<D>, ok);
    };
    if (greedy)
      go(sv_reduce<D, true, true, false>, std::true_type(), std::true_type());
    else if (draft)
      go(sv_reduce<D, false, true, true>, std::false_type(), std::true_type());
    else if (a.kind == CALL_CACHED)
      go(sv_reduce<D, false, true, false>, std::false_type(), std::true_type());
    else
      go(sv_reduce<D, false, false, false>, std::false_type(), std::false_type());
  };
  if (a.dtype == SV_F32)
    dispatch(std::integral_constant<int, SV_F32>());
  else
    dispatch(std::integral_constant<int, SV_BF16>());
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

Call sampling_call(const void* target_logits, const void* draft_logits,
                   const int32_t* draft_tokens, const float* u_accept, const float* u_resample,
                   const float* temperature, int B, int gamma, int V, int dtype,
                   int32_t* out_tokens, int32_t* out_num_accepted, void* workspace,
                   size_t workspace_bytes, int32_t* dev_status, void* stream) {
  Call c;
  c.kind = CALL_SAMPLE;
  c.Lt = target_logits; c.Ld = draft_logits; c.x = draft_tokens;
  c.u_acc = u_accept; c.u_res = u_resample; c.temp = temperature;
  c.B = B; c.gamma = gamma; c.V = V; c.dtype = dtype;
  c.out_tokens = out_tokens; c.out_n = out_num_accepted;
  c.ws = workspace; c.ws_bytes = workspace_bytes;
  c.status = dev_status; c.stream = stream;
  return c;
}

}  // namespace

extern "C" {

size_t sv_workspace_bytes(int B, int gamma, int V) {
  if (B < 0 || gamma < 0 || gamma > SV_MAX_GAMMA || V < 1) return 0;
  return make_layout(B, gamma, V).total;
}

int sv_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace) return SV_ERR_WORKSPACE;
  return cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? SV_OK
             : SV_ERR_CUDA;
}


int spec_verify_diag(const void* target_logits, const void* draft_logits,
                     const int32_t* draft_tokens, const float* u_accept,
                     const float* u_resample, const float* temperature, int B, int gamma,
                     int V, int dtype, int32_t* out_tokens, int32_t* out_num_accepted,
                     float* out_p, float* out_Z, void* workspace, size_t workspace_bytes,
                     int32_t* dev_status, void* stream) {
  Call c = sampling_call(target_logits, draft_logits, draft_tokens, u_accept, u_resample,
                         temperature, B, gamma, V, dtype, out_tokens, out_num_accepted,
                         workspace, workspace_bytes, dev_status, stream);
  c.out_p = out_p;
  c.out_Z = out_Z;
  return launch(c);
}

int spec_verify(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                const float* u_accept, const float* u_resample, const float* temperature, int B,
                int gamma, int V, int dtype, int32_t* out_tokens, int32_t* out_num_accepted,
                void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return launch(sampling_call(target_logits, draft_logits, draft_tokens, u_accept, u_resample,
                              temperature, B, gamma, V, dtype, out_tokens, out_num_accepted,
                              workspace, workspace_bytes, dev_status, stream));
}

int spec_verify_cached(const void* target_logits, const void* draft_logits,
                       const int32_t* draft_tokens, const float* draft_stats,
                       const float* u_accept, const float* u_resample, const float* temperature,
                       int B, int gamma, int V, int dtype, int32_t* out_tokens,
                       int32_t* out_num_accepted, float* out_p, float* out_Z, void* workspace,
                       size_t workspace_bytes, int32_t* dev_status, void* stream) {
  Call c = sampling_call(target_logits, draft_logits, draft_tokens, u_accept, u_resample,
                         temperature, B, gamma, V, dtype, out_tokens, out_num_accepted,
                         workspace, workspace_bytes, dev_status, stream);
  c.kind = CALL_CACHED;
  c.dstats = draft_stats;
  c.out_p = out_p;
  c.out_Z = out_Z;
  return launch(c);
}

int spec_verify_greedy(const void* target_logits, const int32_t* draft_tokens, int B, int gamma,
                       int V, int dtype, int32_t* out_tokens, int32_t* out_num_accepted,
                       void* workspace, size_t workspace_bytes, int32_t* dev_status,
                       void* stream) {
  Call c;
  c.kind = CALL_GREEDY;
  c.Lt = target_logits; c.x = draft_tokens;
  c.B = B; c.gamma = gamma; c.V = V; c.dtype = dtype;
  c.out_tokens = out_tokens; c.out_n = out_num_accepted;
  c.ws = workspace; c.ws_bytes = workspace_bytes;
  c.status = dev_status; c.stream = stream;
  return launch(c);
}

size_t sv_draft_workspace_bytes(int B, int n, int V) {
  if (B < 0 || n < 1 || n > SV_MAX_GAMMA || V < 1) return 0;
  return make_layout(B, n - 1, V).total;
}

int sv_draft_sample(const void* draft_logits, const float* u_draft, const float* temperature,
                    int B, int n, int V, int dtype, int col, int ncols, int32_t* out_tokens,
                    float* out_stats, void* workspace, size_t workspace_bytes,
                    int32_t* dev_status, void* stream) {
  Call c;
  c.kind = CALL_DRAFT;
  c.Lt = draft_logits; c.u_res = u_draft; c.temp = temperature;
  c.B = B; c.n = n; c.V = V; c.dtype = dtype; c.col = col; c.ncols = ncols;
  c.out_tokens = out_tokens; c.out_stats = out_stats;
  c.ws = workspace; c.ws_bytes = workspace_bytes;
  c.status = dev_status; c.stream = stream;
  return launch(c);
}

}  // extern "C"

// ------------------------------------------------- no-allocation entry point
// Scratch for spec_verify_noalloc, in the library's own device memory.  Host
// code may not use this name as a device address (on the host it names a
// stand-in object): the address is looked up per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SV_NOALLOC_MAX_WORKSPACE];

namespace {
// Device address of the scratch in the current context, looked up on every
// call with the calling thread's device current.  The lookup allocates
// nothing and enqueues nothing; it is not cached, because a context that is
// destroyed and created again (cudaDeviceReset) loads the module anew and
// the array may then sit at another address.
int noalloc_scratch(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SV_ERR_CUDA;
  *out = p;
  return SV_OK;
}
}  // namespace

extern "C" {

int spec_verify_noalloc(const void* target_logits, const void* draft_logits,
                        const int32_t* draft_tokens, const float* u_accept,
                        const float* u_resample, const float* temperature, int B, int gamma,
                        int V, int dtype, int32_t* out_tokens, int32_t* out_num_accepted,
                        int32_t* dev_status, void* stream) {
  if (B > 0 && gamma >= 0 && gamma <= SV_MAX_GAMMA && V >= 1 &&
      sv_workspace_bytes(B, gamma, V) > size_t(SV_NOALLOC_MAX_WORKSPACE))
    return SV_ERR_WORKSPACE;  // too large for the built-in scratch
  if (B <= 0 || (dtype != SV_F32 && dtype != SV_BF16) || gamma < 0 || gamma > SV_MAX_GAMMA ||
      V < 1)  // argument errors and the empty batch: no scratch needed
    return launch(sampling_call(target_logits, draft_logits, draft_tokens, u_accept,
                                u_resample, temperature, B, gamma, V, dtype, out_tokens,
                                out_num_accepted, nullptr, 0, dev_status, stream));
  void* scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc != SV_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the control block starts every call in its ready state (calls that may
  // overlap are the caller's to serialise)
  if (cudaMemsetAsync(scratch, 0, sizeof(Ctrl), st) != cudaSuccess) return SV_ERR_CUDA;
  return launch(sampling_call(target_logits, draft_logits, draft_tokens, u_accept, u_resample,
                              temperature, B, gamma, V, dtype, out_tokens, out_num_accepted,
                              scratch, SV_NOALLOC_MAX_WORKSPACE, dev_status, stream));
}

int sv_set_tuning(int chunk_elems) {
  g_tune.chunk = chunk_elems > 0 ? chunk_elems : 0;
  return SV_OK;
}

int sv_set_tail(int mode) {
  if (mode < 0 || mode > 3) return SV_ERR_INVALID_ARG;
  g_tune.tail = mode;
  return SV_OK;
}

int sv_test_withhold_slot(int enable) {
  g_tune.withhold_slot = enable ? 1 : 0;
  return SV_OK;
}

int sv_set_stage_events(void* const* events, int n) {
  if (n < 0 || n > 5 || (n > 0 && !events)) return SV_ERR_INVALID_ARG;
  for (int j = 0; j < n; ++j) {
    if (!events[j]) return SV_ERR_INVALID_ARG;
    g_tune.stage_ev[j] = static_cast<cudaEvent_t>(events[j]);
  }
  g_tune.stage_n = n;
  return SV_OK;
}

const char* sv_error_string(int code) {
  switch (code) {
    case SV_OK: return "SV_OK";
    case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG";
    case SV_ERR_DTYPE: return "SV_ERR_DTYPE";
    case SV_ERR_CUDA: return "SV_ERR_CUDA";
    case SV_ERR_WORKSPACE: return "SV_ERR_WORKSPACE";
    default: return "SV_ERR_UNKNOWN";
  }
}

int sv_version(void) { return 400; }

}  // extern "C"
