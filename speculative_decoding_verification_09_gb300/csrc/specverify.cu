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
// GPU structure: ONE persistent launch per call, one CTA per SM, warp
// specialised:
//   producer  (warp 0, one lane) claims task ids from an atomic counter (two
//             claims in flight) in a fixed global order and streams each
//             task's row chunks from HBM into a ring of shared-memory slots
//             with TMA bulk copies (cp.async.bulk, completion counted on an
//             mbarrier);
//   consumers (NCW warps) reduce each slot from shared memory and stage one
//             partial per warp; the warp of index (slot sequence mod NCW)
//             books the slot: it combines the staged partials, frees the
//             slot and publishes the result.
// Published values are 64-bit words whose high half is the launch epoch, so
// a reader knows a value is this launch's without any fence or counter; the
// per-task path has no atomics besides the task claim.
// Tasks, in a global order where every request's tasks follow each other at
// a distance of `lag` requests:
//   P1(b, i, c)  chunk c of target row i and draft row i of request b:
//                per-warp max (packed bf16 max) then sum 2^((l-max)*log2e/T);
//                the row chunk's (max, sum) pair is published.
//   D(b)         the decision: every consumer warp combines rows of b in fp64
//                (P_t(x_i), P_d(x_i), accept bit); the booking warp takes the
//                first rejection k, writes all outputs but token k and
//                publishes a decision record (release of the launch epoch).
//   P2(b, c)     chunk c of the row the last token is drawn from (residual of
//                row k, or target row gamma for the bonus), re-read from L2:
//                the mass of each warp's contiguous sub-range.
//   T3(b)        finds the sub-range where the running mass crosses u * Z and
//                scans it in index order with warp prefix sums: token k.
// A task only ever waits for tasks claimed before it (D for b's P1 chunks, P2
// for D's record, T3 for P2's masses), and nothing waits for a later task,
// so every wait ends; each wait still gives up after one second
// (SV_ST_TIMEOUT) instead of hanging.
// Greedy verification runs P1 (chunk argmax) and D only.
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "specverify.h"

namespace {

constexpr int NCW = 14;                // consumer warps (16 warps in all: 4 per SM sub-partition)
constexpr int NTHR = 32 * (NCW + 2);   // plus the producer warp and the booking warp
constexpr int NSTAGE = 8;              // staging ring depth (how far booking may lag)
constexpr int NSLOT = 3;               // shared-memory ring depth
constexpr int HALF = 32768;            // bytes of one row chunk in a slot
constexpr int SLOT = 2 * HALF;         // target chunk + draft chunk
constexpr int CH1_MIN = 1024;          // smallest phase-1 chunk (elements)
constexpr int CH2_F32 = HALF / 4;      // phase-2 chunk for fp32 (the workspace bound)
constexpr unsigned SUSPEND_HINT_NS = 1000000u;  // a waiting warp sleeps until the phase completes
constexpr int SMS_CAP = 256;           // the chunk heuristic assumes at most this many SMs
constexpr int KF_CAP = 2048;           // requests whose log2(e)/T is kept in shared memory
constexpr int MAXR = SV_MAX_GAMMA + 1;
constexpr float LOG2E_F = 1.4426950408889634f;
constexpr double LOG2E_D = 1.4426950408889634;
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;  // one second

enum : int { MODE_INVALID = 0, MODE_REJECT = 1, MODE_BONUS = 2, MODE_TARGET = 3 };
enum : int { K_END = 0, K_P1 = 1, K_D = 2, K_P2 = 3, K_T3 = 4, K_SKIP = 5 };

// ------------------------------------------------------------ workspace

struct Ctrl {                 // 64 bytes at the start of the workspace
  unsigned long long task;    // next task id
  unsigned exit_count;        // CTAs that finished
  unsigned epoch_counter;     // launch epoch = epoch_counter + 1
  int abort;                  // set when a wait gave up
  int pad[11];
};
struct ReqCtl {               // per request, 16 bytes
  unsigned flag;              // epoch of the published decision record
  unsigned pad[3];
};
struct Record {               // per request, 48 bytes
  int k, mode;
  float mt, kf;               // max logit of target row k; log2(e)/T in fp32
  unsigned epoch;
  float ist_hi, ist_lo;       // 1/S_t of row k as an unevaluated float pair (fp64 precision)
  float c0_hi, c0_lo;         // log2(P_d/P_t) = (l_d - l_t) * kf + c0 on row k, c0 as a pair
  int pad[3];
};
// Published values: (epoch << 32) | 32-bit payload, written with aligned
// 8-byte stores (single-copy atomic), so each word is either this launch's
// or visibly not.
struct Partial {              // per (request, position, chunk, consumer warp), 32 bytes
  unsigned long long w[4];    // sampling: m_t, s_t, m_d, s_d; greedy: value, index, nan, 0
};
struct ZPart {                // per (request, phase-2 chunk), 128 bytes
  unsigned long long w[2 * NCW];  // each sub-range's fp64 mass as (lo, hi) halves
};
// A row's decision inputs, staged in shared memory by the D task's warps.
struct RowStat {
  float mt, md;               // row maxima
  double St, Sd;              // sum of 2^((l - max) * kf) over the row, fp64
  float pt, pd;               // P_t(x_i), P_d(x_i)
  int acc, bad, amax, pad;    // accept bit, SV_ST_* bits, greedy argmax
};

static_assert(sizeof(Ctrl) == 64 && sizeof(ReqCtl) == 16 && sizeof(Record) == 48 &&
                  sizeof(Partial) == 32 && sizeof(ZPart) == 16 * NCW && sizeof(RowStat) == 48,
              "workspace record sizes");

struct Layout {
  size_t ctrl, req, rec, part, z2, total;
  int nch1_max, nch2_max;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

Layout make_layout(int B, int gamma, int V) {
  Layout L;
  const size_t R = size_t(gamma) + 1;
  // the chunk heuristic below never uses more chunks than this (it assumes
  // at most SMS_CAP SMs)
  const long long units = (long long)B * (long long)R;
  const long long by_bytes = (V + CH2_F32 - 1) / CH2_F32;
  const long long by_tasks = units > 0 ? (8LL * SMS_CAP + units - 1) / units : 1;
  L.nch1_max = int(min((long long)(V + CH1_MIN - 1) / CH1_MIN, max(by_bytes, by_tasks)));
  L.nch2_max = (V + CH2_F32 - 1) / CH2_F32;
  L.ctrl = 0;
  L.req = align256(sizeof(Ctrl));
  L.rec = L.req + align256(size_t(B) * sizeof(ReqCtl));
  L.part = L.rec + align256(size_t(B) * sizeof(Record));
  L.z2 = L.part + align256(size_t(B) * R * L.nch1_max * NCW * sizeof(Partial));
  L.total = L.z2 + align256(size_t(B) * L.nch2_max * sizeof(ZPart));
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
  int ch1, nch1, ch2, nch2, sub, lag;
  int np1;                    // phase-1 partials per row: one per (chunk, consumer warp)
  long long n1, n2, total;
  bool draw;                  // sampling: the task order has P2 and T3 tasks
  // the task order as regions of blocks of constant composition: region r
  // covers blocks [rj[r], rj[r+1]) of rsz[r] tasks each, starting at task rc[r]
  int nreg;
  long long rj[9], rc[9];
  int rsz[8];
  int32_t* out_tokens;
  int32_t* out_n;
  float* out_p;
  float* out_Z;
  int32_t* status;
  Ctrl* ctrl;
  ReqCtl* req;
  Record* rec;
  Partial* part;
  ZPart* z2;
};

// Shared-memory control block (after the slots).
struct Desc {                 // one slot's task, written by the producer, 96 bytes
  int kind, b, i, c;          // i: row position (P1) or the drawn row (P2); c: chunk
  int e0, n;                  // element range of the chunk within the row
  int head_t, nb_t;           // target: leading single elements, aligned body elements in smem
  int head_d, nb_d;           // draft likewise
  float kf;                   // sampling: log2(e) / T of the request
  int pad;
  Record rec;                 // P2: the request's decision record
};
struct SmemCtl {
  unsigned long long full[NSLOT], empty[NSLOT];      // data ring: producer <-> consumers
  unsigned long long staged[NSTAGE], freed[NSTAGE];  // staging ring: consumers <-> booking warp
  Desc desc[NSLOT];
  Desc sdesc[NSTAGE];                                // the task of each staging entry
  RowStat rows[NSTAGE][MAXR];
  int defer[16];                                     // T3 requests held back by the booking warp
  float kf_tab[2048];                                // log2(e)/T of the first 2048 requests
  unsigned epoch;
  int abort;
};
constexpr size_t SMEM_BYTES = size_t(NSLOT) * SLOT + sizeof(SmemCtl);
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

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

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A decision record as stored by another CTA (read through L2).
__device__ __forceinline__ Record load_record(const Record* p) {
  Record r;
  const int4 a = __ldcg(reinterpret_cast<const int4*>(p));
  const int4 b = __ldcg(reinterpret_cast<const int4*>(p) + 1);
  const int4 c = __ldcg(reinterpret_cast<const int4*>(p) + 2);
  r.k = a.x; r.mode = a.y; r.mt = __int_as_float(a.z); r.kf = __int_as_float(a.w);
  r.epoch = unsigned(b.x); r.ist_hi = __int_as_float(b.y); r.ist_lo = __int_as_float(b.z);
  r.c0_hi = __int_as_float(b.w);
  r.c0_lo = __int_as_float(c.x);
  r.pad[0] = r.pad[1] = r.pad[2] = 0;
  return r;
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

__device__ __forceinline__ void set_status(const Params& P, int bits) {
  if (bits && P.status) atomicOr(P.status, bits);
}
// Evidence that the workspace did not hold what this launch wrote (a record
// or partial with another epoch): the call's results are void.
__device__ __forceinline__ void mark_dirty(const Params& P) { set_status(P, SV_ST_WORKSPACE); }

__device__ __forceinline__ void give_up(const Params& P, SmemCtl& C) {
  atomicExch(&P.ctrl->abort, 1);
  set_status(P, SV_ST_TIMEOUT);
  *reinterpret_cast<volatile int*>(&C.abort) = 1;
}

// Wait for phase `parity` of an mbarrier; false after one second or when the
// launch was aborted.
__device__ bool mbar_wait(unsigned long long* bar, unsigned parity, const Params& P, SmemCtl& C) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (unsigned it = 1;; ++it) {
    if (mbar_try(bar, parity)) return true;
    if ((it & 3u) == 0u) {
      if (*reinterpret_cast<volatile int*>(&C.abort)) return false;
      if (globaltimer() - t0 > WAIT_LIMIT_NS) {
        give_up(P, C);
        return false;
      }
    }
  }
}

// Published words: (epoch << 32) | payload.
__device__ __forceinline__ unsigned long long tagged(unsigned epoch, uint32_t v) {
  return ((unsigned long long)epoch << 32) | v;
}
__device__ __forceinline__ void st_pair(void* p, unsigned long long a, unsigned long long b) {
  asm volatile("st.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void ld_pair(const void* p, unsigned long long& a, unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ bool is_mine(unsigned long long w, unsigned epoch) {
  return unsigned(w >> 32) == epoch;
}
__device__ __forceinline__ float payload_f(unsigned long long w) {
  return __uint_as_float(unsigned(w & 0xffffffffull));
}

// ------------------------------------------------------- element types

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
// (m, s) pairs: s = sum of 2^((l - m) * kf).  NaN sticks in s; an all -inf
// set keeps m = -inf, s = 0.  Argmax triples (value, lowest index, NaN seen):
__device__ __forceinline__ void am_merge(float& best, int& bi, int& nan, float b2, int i2, int n2) {
  if (b2 > best || (b2 == best && i2 < bi)) { best = b2; bi = i2; }
  nan |= n2;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_incl_scan_d(double v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// ------------------------------------------------ P1: consumer reductions

// Vectors of one row chunk a consumer thread owns: body vector j belongs to
// consumer thread j mod (NCW*32); a 16 KB chunk gives each thread at most
// MAXV vectors, held in registers.
constexpr int MAXV = (HALF / 16 + NCW * 32 - 1) / (NCW * 32);
static_assert(MAXV * 16 * NCW * 32 >= HALF, "chunk split");

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

// This warp's (max, sum 2^((l-max)*kf)) over its share of one row chunk: the
// aligned body in shared memory plus, for consumer warp 0, the few unaligned
// head/tail elements read from global memory.  Target and draft chunks are
// reduced together, every lane's vectors in registers; each lane sums
// relative to its own maximum and the lanes' sums are rescaled to the warp's.
template <int DT, typename Release>
__device__ void warp_ms2(const unsigned char* st, const unsigned char* sd, const Desc& d,
                         const unsigned char* gt, const unsigned char* gd, bool has_d, float kf,
                         int cw, int lane, float4& out, Release release) {
  using E = Elem<DT>;
  constexpr int NCT = NCW * 32;
  const int tid = cw * 32 + lane;
  const int nvt = d.nb_t / E::VEC, nvd = has_d ? d.nb_d / E::VEC : 0;
  const uint4 neg = make_uint4(E::NEG_INF_WORD, E::NEG_INF_WORD, E::NEG_INF_WORD, E::NEG_INF_WORD);
  uint4 vt[MAXV], vd[MAXV];
#pragma unroll
  for (int u = 0; u < MAXV; ++u) {
    const int j = tid + u * NCT;
    vt[u] = j < nvt ? reinterpret_cast<const uint4*>(st)[j] : neg;
    vd[u] = j < nvd ? reinterpret_cast<const uint4*>(sd)[j] : neg;
  }
  release();  // the chunk is in registers: the slot can be refilled
  float ht = -INFINITY, tt = -INFINITY, hd = -INFINITY, td = -INFINITY;
  if (cw == 0) {
    if (lane < d.head_t) ht = E::load(gt, lane);
    if (lane < d.n - d.head_t - d.nb_t) tt = E::load(gt, d.head_t + d.nb_t + lane);
    if (has_d) {
      if (lane < d.head_d) hd = E::load(gd, lane);
      if (lane < d.n - d.head_d - d.nb_d) td = E::load(gd, d.head_d + d.nb_d + lane);
    }
  }
  // lane maxima: balanced trees over the vectors
  uint32_t wt[MAXV], wd[MAXV];
#pragma unroll
  for (int u = 0; u < MAXV; ++u) {
    wt[u] = E::vmax_acc(E::MAX_INIT, vt[u]);
    wd[u] = E::vmax_acc(E::MAX_INIT, vd[u]);
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
  const unsigned long long kk = pk2(kf, kf);
  const unsigned long long mmt = pk2(mt, mt), mmd = pk2(md, md);
  float s_t = 0.f, s_d = 0.f;
#pragma unroll
  for (int u = 0; u < MAXV; ++u) {
    if (lt) s_t += vec_expsum<DT>(vt[u], mmt, kk);
    if (ld) s_d += vec_expsum<DT>(vd[u], mmd, kk);
  }
  if (lt) s_t += ex2((ht - mt) * kf) + ex2((tt - mt) * kf);
  if (ld) s_d += ex2((hd - md) * kf) + ex2((td - md) * kf);
  if (mt != mt) s_t = NAN;
  if (md != md) s_d = NAN;
  // rescale every lane's sum to the warp maximum and add them up
  const float Mt = warp_max_nan(mt), Md = warp_max_nan(md);
  if (lt && Mt > mt) s_t *= ex2((mt - Mt) * kf);
  if (ld && Md > md) s_d *= ex2((md - Md) * kf);
  if (Mt != Mt) s_t = NAN;
  if (Md != Md) s_d = NAN;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s_t += __shfl_xor_sync(0xffffffffu, s_t, o);
    s_d += __shfl_xor_sync(0xffffffffu, s_d, o);
  }
  out = make_float4(Mt, s_t, Md, s_d);
}

// This warp's (largest value, lowest index among its occurrences, NaN seen)
// over its share of one row chunk; indices are within the row.
template <int DT, typename Release>
__device__ void warp_argmax(const unsigned char* sbody, int nb, const unsigned char* gseg,
                            int head, int n, int e0, int cw, int lane, float& best_out,
                            int& bi_out, int& nan_out, Release release) {
  using E = Elem<DT>;
  const int nv = nb / E::VEC;
  const int tid = cw * 32 + lane;
  constexpr int NCT = NCW * 32;
  const uint4* sv = reinterpret_cast<const uint4*>(sbody);
  float best = -INFINITY;
  int bi = INT_MAX, nan = 0;
  if (cw == 0 && lane < head) {
    const float l = E::load(gseg, lane);
    if (l != l) nan = 1;
    else if (l > best) { best = l; bi = e0 + lane; }
  }
  uint4 vr[MAXV];
#pragma unroll
  for (int u = 0; u < MAXV; ++u) {
    const int j = tid + u * NCT;
    vr[u] = j < nv ? sv[j] : make_uint4(E::NEG_INF_WORD, E::NEG_INF_WORD, E::NEG_INF_WORD,
                                        E::NEG_INF_WORD);
  }
  release();
#pragma unroll
  for (int u = 0; u < MAXV; ++u) {
    const int j = tid + u * NCT;
    const uint4 v = vr[u];
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
  if (cw == 0) {
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
  best_out = best;
  bi_out = bi;
  nan_out = nan;
}

// ---------------------------------------------- P2 / P3: residual weights

// Weight of one element of the final draw (fp32, identical in P2 and P3).
// Residual max(0, P_t - P_d) formed as P_t * (1 - 2^delta) with
// delta = log2(P_d / P_t), so it keeps its relative precision where the two
// rows nearly agree (no cancellation); the normaliser is applied as hi + lo.
// 1 - 2^delta for delta <= 0, to fp32 relative precision: 1 - ex2(delta)
// where that loses nothing (delta < -1/2), else -expm1(y), y = delta*ln2 in
// [-0.347, 0], by its Taylor series to y^7 (truncation below 2e-8 relative).
__device__ __forceinline__ float one_minus_exp2(float delta) {
  const float y = delta * 0.69314718055994531f;
  float p = 1.f / 5040.f;
  p = fmaf(p, y, 1.f / 720.f);
  p = fmaf(p, y, 1.f / 120.f);
  p = fmaf(p, y, 1.f / 24.f);
  p = fmaf(p, y, 1.f / 6.f);
  p = fmaf(p, y, 0.5f);
  p = fmaf(p, y, 1.f);
  const float series = -y * p;
  return delta < -0.5f ? 1.f - ex2(delta) : series;
}

__device__ __forceinline__ float weight(const Record& r, float lt, float ld) {
  const float et = ex2((lt - r.mt) * r.kf);
  const float pt = fmaf(et, r.ist_hi, et * r.ist_lo);
  if (r.mode == MODE_REJECT) {
    const float delta = fmaf(ld - lt, r.kf, r.c0_hi) + r.c0_lo;  // log2(P_d / P_t)
    return (et > 0.f && delta < 0.f) ? pt * one_minus_exp2(delta) : 0.f;
  }
  return pt;
}

// Residual (or bonus) weights of one 16-byte vector of target values `t`
// and draft values `dv`, summed; packed fp32x2 arithmetic, the same formula
// as weight() element by element.
template <int DT>
__device__ __forceinline__ float vec_weights(const Record& r, const uint4& t, const uint4& dv,
                                             bool two) {
  using E = Elem<DT>;
  const unsigned long long mm = pk2(r.mt, r.mt), kk = pk2(r.kf, r.kf);
  const unsigned long long hh = pk2(r.ist_hi, r.ist_hi), ll = pk2(r.ist_lo, r.ist_lo);
  unsigned long long acc = pk2(0.f, 0.f);
#pragma unroll
  for (int q = 0; q < E::PAIRS; ++q) {
    const unsigned long long lt = E::pair(t, q);
    float a, b;
    upk2(mul2(sub2(lt, mm), kk), a, b);
    const unsigned long long et = pk2(ex2(a), ex2(b));
    unsigned long long pt;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(pt) : "l"(et), "l"(hh), "l"(mul2(et, ll)));
    if (two) {
      // delta = log2(P_d / P_t) = (l_d - l_t) * kf + c0
      unsigned long long dl;
      const unsigned long long ch = pk2(r.c0_hi, r.c0_hi), cl = pk2(r.c0_lo, r.c0_lo);
      asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(dl) : "l"(sub2(E::pair(dv, q), lt)), "l"(kk),
          "l"(ch));
      dl = add2(dl, cl);
      float d0, d1, e0, e1, p0, p1;
      upk2(dl, d0, d1);
      upk2(et, e0, e1);
      upk2(pt, p0, p1);
      const float w0 = (e0 > 0.f && d0 < 0.f) ? p0 * one_minus_exp2(d0) : 0.f;
      const float w1 = (e1 > 0.f && d1 < 0.f) ? p1 * one_minus_exp2(d1) : 0.f;
      acc = add2(acc, pk2(w0, w1));
    } else {
      acc = add2(acc, pt);
    }
  }
  float a, b;
  upk2(acc, a, b);
  return a + b;
}

// Mass of this warp's contiguous sub-range [cw*sub, (cw+1)*sub) of a P2
// chunk held in a slot (target body at +0, draft body at +HALF).
template <int DT, typename Release>
__device__ double warp_p2_mass(const Params& P, const Desc& d, const unsigned char* slot,
                               int cw, int lane, Release release) {
  using E = Elem<DT>;
  const Record& r = d.rec;
  const bool two = (r.mode == MODE_REJECT);
  const int lo = cw * P.sub;
  const int hi = min(lo + P.sub, d.n);
  if (lo >= hi) {
    release();
    return 0.0;
  }
  const unsigned char* trow =
      P.Lt + ((size_t(d.b) * P.R + d.i) * size_t(P.V) + d.e0) * E::ES;
  const unsigned char* drow =
      two ? P.Ld + ((size_t(d.b) * P.gamma + r.k) * size_t(P.V) + d.e0) * E::ES : nullptr;
  float acc = 0.f;
  if (d.head_t == 0 && (!two || d.head_d == 0)) {
    // aligned: whole 16-byte vectors from shared memory, held in registers
    constexpr int PV = 5;  // vectors per lane held in registers (a sub-range has <= 32*PV)
    const uint4* tv = reinterpret_cast<const uint4*>(slot);
    const uint4* dv = reinterpret_cast<const uint4*>(slot + HALF);
    const int j0 = lo / E::VEC, vhi = min(hi, d.nb_t) / E::VEC;
    uint4 vt[PV], vd[PV];
#pragma unroll
    for (int u = 0; u < PV; ++u) {
      const int j = j0 + lane + 32 * u;
      vt[u] = j < vhi ? tv[j] : make_uint4(E::NEG_INF_WORD, E::NEG_INF_WORD, E::NEG_INF_WORD,
                                           E::NEG_INF_WORD);
      vd[u] = (two && j < vhi) ? dv[j] : vt[u];
    }
    for (int j = j0 + lane + 32 * PV; j < vhi; j += 32)  // only if sub exceeds 32*PV vectors
      acc += vec_weights<DT>(r, tv[j], two ? dv[j] : tv[j], two);
    release();
#pragma unroll
    for (int u = 0; u < PV; ++u) acc += vec_weights<DT>(r, vt[u], vd[u], two);
    for (int e = max(lo, d.nb_t) + lane; e < hi; e += 32)
      acc += weight(r, E::load(trow, e), two ? E::load(drow, e) : 0.f);
  } else {
    // unaligned rows: element by element, from shared memory where held
    for (int e = lo + lane; e < hi; e += 32) {
      const int et = e - d.head_t, ed = e - d.head_d;
      const float lt = (et >= 0 && et < d.nb_t) ? E::lds(slot, et) : E::load(trow, e);
      float ld = 0.f;
      if (two) ld = (ed >= 0 && ed < d.nb_d) ? E::lds(slot + HALF, ed) : E::load(drow, e);
      acc += weight(r, lt, ld);
    }
    release();
  }
  return warp_sum_d(double(acc));
}

// ------------------------------------------------------------ waiting

// Poll until every lane's `ready` is true (re-evaluated by `probe`), for at
// most one second; false on timeout or abort.
template <typename Probe>
__device__ bool warp_poll(const Params& P, SmemCtl& C, Probe probe) {
  if (__all_sync(0xffffffffu, probe())) return true;
  const unsigned long long t0 = globaltimer();
  unsigned ns = 64;
  for (;;) {
    __nanosleep(ns);
    ns = ns < 2048 ? 2 * ns : ns;
    if (__all_sync(0xffffffffu, probe())) return true;
    const bool stop = *reinterpret_cast<volatile int*>(&P.ctrl->abort) ||
                      *reinterpret_cast<volatile int*>(&C.abort);
    if (__any_sync(0xffffffffu, stop)) return false;
    if (globaltimer() - t0 > WAIT_LIMIT_NS) {
      if ((threadIdx.x & 31) == 0) give_up(P, C);
      __syncwarp();
      return false;
    }
  }
}

// ------------------------------------------------------------ decisions

__device__ __forceinline__ bool row_ok(float m, double S) {
  return (m > -INFINITY) && (m < INFINITY) && (S > 0.0) && (S < INFINITY);
}

// A row's published partials: one per (chunk, consumer warp), row-major.
__device__ __forceinline__ const Partial* row_partials(const Params& P, int b, int i) {
  return P.part + (size_t(b) * P.R + i) * size_t(P.np1);
}

// Wait until all chunk partials of one row carry this launch's epoch.
__device__ bool wait_partials(const Params& P, SmemCtl& C, const Partial* pp) {
  const unsigned epoch = C.epoch;
  const int lane = threadIdx.x & 31;
  return warp_poll(P, C, [&]() {
    bool ok = true;
    for (int c = lane; c < P.np1; c += 32) {
      unsigned long long a, b, c2, d;
      ld_pair(&pp[c].w[0], a, b);
      ld_pair(&pp[c].w[2], c2, d);
      ok = ok && is_mine(a, epoch) && is_mine(b, epoch) && is_mine(c2, epoch) && is_mine(d, epoch);
    }
    return ok;
  });
}

// Combine of one row's partials (m_c, s_c) held in words (0, 1)
// or (2, 3); one warp, result valid in every lane.
__device__ void warp_row_combine(const Partial* pp, int nch, int f, float kf, float& m_out,
                                 double& S_out) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  for (int c = lane; c < nch; c += 32) {
    unsigned long long a, b;
    ld_pair(&pp[c].w[f], a, b);
    m = fmaxf(m, payload_f(a));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  double S = 0.0;
  for (int c = lane; c < nch; c += 32) {
    unsigned long long a, b;
    ld_pair(&pp[c].w[f], a, b);
    const float mc = payload_f(a), sc = payload_f(b);
    S += (m == -INFINITY) ? double(sc) : double(sc) * double(ex2((mc - m) * kf));
  }
  m_out = m;
  S_out = warp_sum_d(S);
}

// Row i of request b for the D task (one warp): lane 0 fills `out`.  The
// loads that do not depend on the partials (the draft token, its logits, the
// uniform) are issued first; the row's chunk partials are read into
// registers as soon as all carry this launch's epoch, the row maximum taken,
// and the sum rescaled in fp64 (one exponential per chunk).
constexpr int PCAP = 5;  // partials per lane held in registers (rows of <= 160 partials)

template <int DT>
__device__ void row_decide_sample(const Params& P, SmemCtl& C, int b, int i, float kf,
                                  RowStat& out) {
  using E = Elem<DT>;
  const int g = P.gamma, R = P.R, V = P.V;
  const int lane = threadIdx.x & 31;
  const unsigned epoch = C.epoch;
  const float T = __ldg(P.temp + b);
  const bool t_ok = isfinite(T) && T >= 0x1p-126f;
  const double k64 = LOG2E_D / double(T);
  int xi = 0;
  float lt = 0.f, ld = 0.f, u = 0.f;
  bool tok_ok = true;
  if (lane == 0 && i < g) {
    xi = __ldg(P.x + size_t(b) * g + i);
    u = __ldg(P.u_acc + size_t(b) * g + i);
    tok_ok = xi >= 0 && xi < V;
    if (tok_ok) {
      lt = E::load(P.Lt, (long long)(size_t(b) * R + i) * V + xi);
      ld = E::load(P.Ld, (long long)(size_t(b) * g + i) * V + xi);
    }
  }
  const Partial* pp = row_partials(P, b, i);
  float mt = -INFINITY, md = -INFINITY;
  double St = 0.0, Sd = 0.0;
  bool ready;
  if (P.np1 <= 32 * PCAP) {
    unsigned long long w[PCAP][4];
    ready = warp_poll(P, C, [&]() {
      bool ok = true;
#pragma unroll
      for (int q = 0; q < PCAP; ++q) {
        const int c = lane + 32 * q;
        if (c < P.np1) {
          ld_pair(&pp[c].w[0], w[q][0], w[q][1]);
          ld_pair(&pp[c].w[2], w[q][2], w[q][3]);
          ok = ok && is_mine(w[q][0], epoch) && is_mine(w[q][1], epoch) &&
               is_mine(w[q][2], epoch) && is_mine(w[q][3], epoch);
        }
      }
      return ok;
    });
    if (ready) {
#pragma unroll
      for (int q = 0; q < PCAP; ++q)
        if (lane + 32 * q < P.np1) {
          mt = fmaxf(mt, payload_f(w[q][0]));
          md = fmaxf(md, payload_f(w[q][2]));
        }
      mt = warp_max(mt);
      md = warp_max(md);
#pragma unroll
      for (int q = 0; q < PCAP; ++q)
        if (lane + 32 * q < P.np1) {
          const float m0 = payload_f(w[q][0]), s0 = payload_f(w[q][1]);
          const float m1 = payload_f(w[q][2]), s1 = payload_f(w[q][3]);
          St += (mt == -INFINITY) ? double(s0) : double(s0) * double(ex2((m0 - mt) * kf));
          Sd += (md == -INFINITY) ? double(s1) : double(s1) * double(ex2((m1 - md) * kf));
        }
      St = warp_sum_d(St);
      Sd = warp_sum_d(Sd);
    }
  } else {  // very long rows: poll, then two passes over the partials
    ready = wait_partials(P, C, pp);
    if (ready) {
      warp_row_combine(pp, P.np1, 0, kf, mt, St);
      warp_row_combine(pp, P.np1, 2, kf, md, Sd);
    }
  }
  if (i >= g) { md = 0.f; Sd = 1.0; }
  if (lane == 0) {
    int bad = ready ? 0 : SV_ST_TIMEOUT;
    if (!row_ok(mt, St) || (i < g && !row_ok(md, Sd))) bad |= SV_ST_NONFINITE;
    float pt = NAN, pd = NAN;
    int acc = 1;
    if (i < g) {
      if (!tok_ok) {
        bad |= SV_ST_BAD_TOKEN;
      } else if (bad == 0 && t_ok) {
        const double dpt = exp2((double(lt) - double(mt)) * k64) / St;
        const double dpd = exp2((double(ld) - double(md)) * k64) / Sd;
        const double r = dpd > 0.0 ? fmin(1.0, dpt / dpd) : 1.0;
        acc = double(u) <= r;
        pt = float(dpt);
        pd = float(dpd);
      }
    }
    out.mt = mt; out.md = md; out.St = St; out.Sd = Sd; out.pt = pt; out.pd = pd;
    out.acc = acc; out.bad = bad; out.amax = -1; out.pad = 0;
  }
}

template <int DT>
__device__ void row_decide_greedy(const Params& P, SmemCtl& C, int b, int i, RowStat& out) {
  const int g = P.gamma, V = P.V;
  const int lane = threadIdx.x & 31;
  const unsigned epoch = C.epoch;
  const Partial* pp = row_partials(P, b, i);
  const int np = P.np1;
  float best = -INFINITY;
  int bi = INT_MAX, nan = 0;
  const bool ready = warp_poll(P, C, [&]() {
    best = -INFINITY; bi = INT_MAX; nan = 0;
    bool ok = true;
    for (int q = lane; q < np; q += 32) {
      unsigned long long a, bb, cc, dd;
      ld_pair(&pp[q].w[0], a, bb);
      ld_pair(&pp[q].w[2], cc, dd);
      ok = ok && is_mine(a, epoch) && is_mine(bb, epoch) && is_mine(cc, epoch) &&
           is_mine(dd, epoch);
      am_merge(best, bi, nan, payload_f(a), int(bb & 0xffffffffull), int(cc & 0xffffffffull));
    }
    return ok;
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    const int n2 = __shfl_xor_sync(0xffffffffu, nan, o);
    am_merge(best, bi, nan, b2, i2, n2);
  }
  if (lane == 0) {
    int bad = ready ? 0 : SV_ST_TIMEOUT;
    if (nan || bi == INT_MAX || best == INFINITY) bad |= SV_ST_NONFINITE;
    if (i < g) {
      const int xi = __ldg(P.x + size_t(b) * g + i);
      if (xi < 0 || xi >= V) bad |= SV_ST_BAD_TOKEN;
    }
    out.mt = best; out.md = 0.f; out.St = out.Sd = 0.0; out.pt = out.pd = 0.f;
    out.acc = 0; out.bad = bad; out.amax = bi; out.pad = 0;
  }
}

// Request decision of the D task, by the booking warp, from the rows staged
// in shared memory: first rejection k, every output but token k, and the
// decision record.  The slot is freed as soon as the rows are in registers.
template <int DT>
__device__ void request_decide_sample(const Params& P, SmemCtl& C, int e, int b) {
  const int g = P.gamma, R = P.R;
  const int lane = threadIdx.x & 31;
  const unsigned epoch = C.epoch;
  const float T = __ldg(P.temp + b);
  const bool t_ok = isfinite(T) && T >= 0x1p-126f;
  const float kf = LOG2E_F / T;
  int bad = 0, acc = 1;
  float pt = NAN, pd = NAN;
  for (int i = lane; i < R; i += 32) {
    const RowStat& r = C.rows[e][i];
    bad |= r.bad;
    if (i == lane) { acc = r.acc; pt = r.pt; pd = r.pd; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) bad |= __shfl_xor_sync(0xffffffffu, bad, o);
  if (!t_ok) bad |= SV_ST_BAD_TEMP;
  const bool valid = (bad == 0);
  const unsigned rej = __ballot_sync(0xffffffffu, lane < g && !acc);
  const int k = rej ? __ffs(rej) - 1 : g;
  const RowStat rk = C.rows[e][k];
  __syncwarp();
  if (lane == 0) mbar_arrive(&C.freed[e]);  // the staging entry may be reused now
  for (int i = lane; i < R; i += 32) {
    int tok = -1;
    if (valid && i < k) tok = __ldg(P.x + size_t(b) * g + i);
    if (!valid || i != k) P.out_tokens[size_t(b) * R + i] = tok;
  }
  if (P.out_p && lane < g) {
    P.out_p[(size_t(b) * g + lane) * 2] = valid ? pt : NAN;
    P.out_p[(size_t(b) * g + lane) * 2 + 1] = valid ? pd : NAN;
  }
  if (lane == 0) {
    P.out_n[b] = valid ? k : 0;
    if (!valid && P.out_Z) P.out_Z[b] = NAN;
    set_status(P, bad);
    Record r;
    r.k = k;
    r.mode = !valid ? MODE_INVALID : (k < g ? MODE_REJECT : MODE_BONUS);
    r.kf = kf;
    r.epoch = epoch;
    r.mt = 0.f; r.ist_hi = r.ist_lo = r.c0_hi = r.c0_lo = 0.f;
    r.pad[0] = r.pad[1] = r.pad[2] = 0;
    if (valid) {
      r.mt = rk.mt;
      const double ist = 1.0 / rk.St;
      r.ist_hi = float(ist);
      r.ist_lo = float(ist - double(r.ist_hi));
      // log2(P_d[v] / P_t[v]) = (l_d[v] - l_t[v]) * kf + (m_t - m_d) * kf + log2(S_t / S_d)
      const double c0 =
          k < g ? (double(rk.mt) - double(rk.md)) * double(kf) + log2(rk.St / rk.Sd) : 0.0;
      r.c0_hi = float(c0);
      r.c0_lo = float(c0 - double(r.c0_hi));
    }
    int4* d = reinterpret_cast<int4*>(P.rec + b);
    const int4* src = reinterpret_cast<const int4*>(&r);
    d[0] = src[0]; d[1] = src[1]; d[2] = src[2];
    __threadfence();
    if (atomicExch(&P.req[b].flag, epoch) == epoch) mark_dirty(P);
  }
}

__device__ void request_decide_greedy(const Params& P, SmemCtl& C, int e, int b) {
  const int g = P.gamma, R = P.R;
  const int lane = threadIdx.x & 31;
  int bad = 0;
  int am[2] = {-1, -1};
  for (int i = lane, q = 0; i < R; i += 32, ++q) {
    bad |= C.rows[e][i].bad;
    am[q] = C.rows[e][i].amax;
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&C.freed[e]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) bad |= __shfl_xor_sync(0xffffffffu, bad, o);
  const bool valid = (bad == 0);
  const unsigned mis =
      __ballot_sync(0xffffffffu, lane < g && __ldg(P.x + size_t(b) * g + lane) != am[0]);
  const int k = mis ? __ffs(mis) - 1 : g;
  for (int i = lane, q = 0; i < R; i += 32, ++q)
    P.out_tokens[size_t(b) * R + i] = (valid && i <= k) ? am[q] : -1;
  if (lane == 0) {
    P.out_n[b] = valid ? k : 0;
    set_status(P, bad);
  }
}

// ------------------------------------------------------------------ T3

// Token k of request b (one warp): wait for the sub-range masses of every
// phase-2 chunk, find the sub-range where the running mass crosses u * Z and
// scan it in index order.
template <int DT>
__device__ void task_t3(const Params& P, SmemCtl& C, int b) {
  using E = Elem<DT>;
  const int lane = threadIdx.x & 31;
  const unsigned epoch = C.epoch;
  // the decision record: D(b) was claimed before this task but may still be running
  const bool decided =
      warp_poll(P, C, [&]() { return lane != 0 || ld_acquire(&P.req[b].flag) == epoch; });
  if (!decided) return;  // only after a timeout, which the status reports
  Record r = load_record(P.rec + b);
  if (r.mode == MODE_INVALID) return;
  const int R = P.R, V = P.V;
  const int nq = P.nch2 * NCW;
  ZPart* zp = P.z2 + size_t(b) * P.nch2;
  auto zword = [&](int q, unsigned long long& lo, unsigned long long& hi) {
    ld_pair(&zp[q / NCW].w[2 * (q % NCW)], lo, hi);
  };
  auto zval = [&](int q) {
    unsigned long long lo, hi;
    zword(q, lo, hi);
    return __hiloint2double(int(hi & 0xffffffffull), int(lo & 0xffffffffull));
  };
  const bool ready = warp_poll(P, C, [&]() {
    bool ok = true;
    for (int q = lane; q < nq; q += 32) {
      unsigned long long lo, hi;
      zword(q, lo, hi);
      ok = ok && is_mine(lo, epoch) && is_mine(hi, epoch);
    }
    return ok;
  });
  if (!ready) return;
  const float u = __ldg(P.u_res + size_t(b) * R + r.k);
  const int rowk = (r.mode == MODE_BONUS) ? P.gamma : r.k;
  const unsigned char* trow = P.Lt + (size_t(b) * R + rowk) * size_t(V) * E::ES;
  const bool two = (r.mode == MODE_REJECT);
  const unsigned char* drow =
      two ? P.Ld + (size_t(b) * P.gamma + r.k) * size_t(V) * E::ES : nullptr;

  // Z over all sub-ranges, in (chunk, sub-range) order, 32 at a time
  double Z = 0.0;
  for (int q0 = 0; q0 < nq; q0 += 32) {
    const int q = q0 + lane;
    const double z = q < nq ? zval(q) : 0.0;
    Z += __shfl_sync(0xffffffffu, warp_incl_scan_d(z, lane), 31);
  }
  bool degenerate = false;
  if (!(Z > 0.0)) {
    // the residual vanished in fp32: sample target row k instead (reading of
    // the Z = 0 case); recompute every sub-range mass for that distribution
    degenerate = true;
    r.mode = MODE_TARGET;
    Z = 0.0;
    for (int q = 0; q < nq; ++q) {
      const int lo = (q / NCW) * P.ch2 + (q % NCW) * P.sub;
      const int hi = min(lo + P.sub, min(V, (q / NCW + 1) * P.ch2));
      float acc = 0.f;
      for (int e = lo + lane; e < hi; e += 32) acc += weight(r, E::load(trow, e), 0.f);
      const double zq = warp_sum_d(double(acc));
      if (lane == 0) {
        unsigned long long wlo = tagged(epoch, unsigned(__double2loint(zq)));
        unsigned long long whi = tagged(epoch, unsigned(__double2hiint(zq)));
        st_pair(&zp[q / NCW].w[2 * (q % NCW)], wlo, whi);
      }
      Z += zq;
    }
    __threadfence();
    __syncwarp();
  }
  const double tau = double(u) * Z;
  // the (chunk, sub-range) where the running mass crosses tau
  double base = 0.0, before = 0.0;
  int qstar = -1, qlast = 0;
  for (int q0 = 0; q0 < nq && qstar < 0; q0 += 32) {
    const int q = q0 + lane;
    const double z = (q < nq) ? zval(q) : 0.0;
    const double incl = warp_incl_scan_d(z, lane);
    const unsigned pos = __ballot_sync(0xffffffffu, q < nq && z > 0.0);
    if (pos) qlast = q0 + 31 - __clz(pos);
    const unsigned hit = __ballot_sync(0xffffffffu, q < nq && z > 0.0 && base + incl > tau);
    if (hit) {
      const int l = __ffs(hit) - 1;
      qstar = q0 + l;
      before = base + __shfl_sync(0xffffffffu, incl - z, l);
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (qstar < 0) {  // rounding: take the last sub-range with mass
    qstar = qlast;
    before = 0.0;
    for (int q0 = 0; q0 < qstar; q0 += 32) {
      const int q = q0 + lane;
      const double z = (q < qstar) ? zval(q) : 0.0;
      before += __shfl_sync(0xffffffffu, warp_incl_scan_d(z, lane), 31);
    }
  }
  // scan the sub-range in index order
  const int lo = (qstar / NCW) * P.ch2 + (qstar % NCW) * P.sub;
  const int hi = min(lo + P.sub, min(V, (qstar / NCW + 1) * P.ch2));
  const double tau2 = tau - before;
  double run = 0.0;
  int tok = -1, last_pos = -1;
  // One round: lane l holds `cnt` consecutive weights w[] starting at element
  // e0 (the lanes' runs are consecutive); finds the crossing, if any.
  auto round = [&](const float* w, int cnt, int e0) {
    float tot = 0.f;
    for (int q = 0; q < cnt; ++q) {
      tot += w[q];
      if (w[q] > 0.f) last_pos = e0 + q;
    }
    const double incl = warp_incl_scan_d(double(tot), lane);
    const unsigned hit = __ballot_sync(0xffffffffu, tot > 0.f && run + incl > tau2);
    if (hit) {
      const int l = __ffs(hit) - 1;
      if (lane == l) {
        double acc = run + incl - double(tot);
        int v = -1, lp = -1;
        for (int q = 0; q < cnt; ++q) {
          acc += double(w[q]);
          if (w[q] > 0.f) lp = e0 + q;
          if (acc > tau2) { v = e0 + q; break; }
        }
        tok = (v >= 0) ? v : lp;
      }
      tok = __shfl_sync(0xffffffffu, tok, l);
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  };
  const unsigned char* tsub = trow + size_t(lo) * E::ES;
  const unsigned char* dsub = two ? drow + size_t(lo) * E::ES : nullptr;
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(tsub) & 15u) == 0) &&
                      (!two || (reinterpret_cast<uintptr_t>(dsub) & 15u) == 0);
  int done_e = lo;  // elements before done_e have been scanned
  if (vec_ok) {
    // whole 16-byte vectors: loaded UMAX per lane at a time (one round trip),
    // then scanned in rounds of 32 consecutive vectors
    constexpr int UMAX = 5;
    const int nv = (hi - lo) / E::VEC;
    const uint4* tv = reinterpret_cast<const uint4*>(tsub);
    const uint4* dvp = reinterpret_cast<const uint4*>(two ? dsub : tsub);
    for (int v0 = 0; v0 < nv && tok < 0; v0 += 32 * UMAX) {
      uint4 vt[UMAX], vd[UMAX];
#pragma unroll
      for (int u = 0; u < UMAX; ++u) {
        const int j = v0 + 32 * u + lane;
        vt[u] = j < nv ? __ldg(tv + j) : make_uint4(0u, 0u, 0u, 0u);
        vd[u] = (two && j < nv) ? __ldg(dvp + j) : vt[u];
      }
#pragma unroll
      for (int u = 0; u < UMAX; ++u) {
        if (tok >= 0 || v0 + 32 * u >= nv) break;
        const int j = v0 + 32 * u + lane;
        float ft[E::VEC], fd[E::VEC], w[E::VEC];
        E::unpack(vt[u], ft);
        E::unpack(vd[u], fd);
#pragma unroll
        for (int q = 0; q < E::VEC; ++q) w[q] = j < nv ? weight(r, ft[q], two ? fd[q] : 0.f) : 0.f;
        round(w, E::VEC, lo + j * E::VEC);
      }
    }
    done_e = lo + nv * E::VEC;
  }
  // the rest (all of it for unaligned rows): rounds of 32 lanes x 8 elements
  for (int r0 = done_e; r0 < hi && tok < 0; r0 += 256) {
    const int e0 = r0 + lane * 8;
    float w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = e0 + q;
      w[q] = (e < hi) ? weight(r, E::load(trow, e), two ? E::load(drow, e) : 0.f) : 0.f;
    }
    round(w, 8, e0);
  }
  if (tok < 0) {  // rounding: the last element with mass in the sub-range
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      last_pos = max(last_pos, __shfl_xor_sync(0xffffffffu, last_pos, o));
    tok = last_pos < 0 ? lo : last_pos;
  }
  if (lane == 0) {
    P.out_tokens[size_t(b) * R + r.k] = tok;
    if (P.out_Z) P.out_Z[b] = float(Z);
    if (degenerate) set_status(P, SV_ST_DEGENERATE);
  }
}

// ------------------------------------------------------------ producer

// The global task order is a sequence of blocks j = 0, 1, ...: block j holds
// P1 of request j, then D of request j - L, then P2 of request j - 2L, then
// T3 of request j - 3L (each where that request exists; greedy has P1 and D
// only).  tasks_before(j) counts the tasks of blocks 0..j-1.
__device__ void decode(const Params& P, long long t, int& kind, int& b, int& sub) {
  const long long B = P.B, L = P.lag;
  int r = 0;
  while (r + 1 < P.nreg && t >= P.rc[r + 1]) ++r;
  const unsigned off = unsigned(t - P.rc[r]);
  const unsigned sz = unsigned(P.rsz[r]);
  const long long j = P.rj[r] + off / sz;
  long long rem = off % sz;
  sub = 0;
  if (j < B) {
    if (rem < P.n1) { kind = K_P1; b = int(j); sub = int(rem); return; }
    rem -= P.n1;
  }
  if (j >= L && j < B + L) {
    if (rem < 1) { kind = K_D; b = int(j - L); return; }
    rem -= 1;
  }
  if (P.draw && j >= 2 * L && j < B + 2 * L) {
    if (rem < P.n2) { kind = K_P2; b = int(j - 2 * L); sub = int(rem); return; }
    rem -= P.n2;
  }
  kind = K_T3;
  b = int(j - 3 * L);
}

// Bulk-copy the aligned bodies of a target (and draft) row chunk into slot s.
template <int DT>
__device__ void issue(SmemCtl& C, int s, unsigned char* slot, Desc& d, const unsigned char* tseg,
                      const unsigned char* dseg) {
  using E = Elem<DT>;
  auto split = [&](const unsigned char* p, int& head, int& nb) {
    int h = int(((16u - unsigned(reinterpret_cast<uintptr_t>(p) & 15u)) & 15u) / E::ES);
    head = h < d.n ? h : d.n;
    nb = ((d.n - head) / E::VEC) * E::VEC;
  };
  split(tseg, d.head_t, d.nb_t);
  d.head_d = d.nb_d = 0;
  if (dseg) split(dseg, d.head_d, d.nb_d);
  const unsigned bt = unsigned(d.nb_t) * E::ES, bd = unsigned(d.nb_d) * E::ES;
  if (bt + bd == 0u) {
    mbar_arrive(&C.full[s]);
    return;
  }
  mbar_arrive_tx(&C.full[s], bt + bd);
  if (bt) bulk_g2s(slot, tseg + size_t(d.head_t) * E::ES, bt, &C.full[s]);
  if (bd) bulk_g2s(slot + HALF, dseg + size_t(d.head_d) * E::ES, bd, &C.full[s]);
}

// Wait (bounded) for request b's decision record of this launch.
__device__ bool wait_flag(const Params& P, SmemCtl& C, int b, unsigned epoch) {
  const unsigned* flag = &P.req[b].flag;
  if (ld_acquire(flag) == epoch) return true;
  const unsigned long long t0 = globaltimer();
  unsigned ns = 64;
  for (;;) {
    if (ld_acquire(flag) == epoch) return true;
    if (*reinterpret_cast<volatile int*>(&P.ctrl->abort) ||
        *reinterpret_cast<volatile int*>(&C.abort))
      return false;
    if (globaltimer() - t0 > WAIT_LIMIT_NS) {
      give_up(P, C);
      return false;
    }
    __nanosleep(ns);
    ns = ns < 2048 ? ns * 2 : ns;
  }
}

// Claims are kept two deep so the claim latency overlaps the copies; every
// CTA therefore ends holding exactly two claims at or beyond `total`.
template <int DT, bool GREEDY>
__device__ void producer(const Params& P, SmemCtl& C, unsigned char* slots) {
  using E = Elem<DT>;
  const unsigned epoch = C.epoch;
  unsigned long long q0 = atomicAdd(&P.ctrl->task, 1ull);
  unsigned long long q1 = atomicAdd(&P.ctrl->task, 1ull);
  for (long long seq = 0;; ++seq) {
    const int s = int(seq % NSLOT);
    const unsigned use = unsigned(seq / NSLOT);
    Desc& d = C.desc[s];
    unsigned char* slot = slots + size_t(s) * SLOT;
    const long long t = (long long)q0;
    q0 = q1;
    if (t >= P.total || *reinterpret_cast<volatile int*>(&C.abort)) {
      if (use > 0 && !mbar_wait(&C.empty[s], (use - 1) & 1u, P, C)) return;
      d.kind = K_END;
      mbar_arrive(&C.full[s]);
      return;
    }
    q1 = atomicAdd(&P.ctrl->task, 1ull);
    int kind, b, sub;
    decode(P, t, kind, b, sub);
    const float kf = GREEDY ? 0.f : (b < KF_CAP ? C.kf_tab[b] : LOG2E_F / __ldg(P.temp + b));
    if (use > 0 && !mbar_wait(&C.empty[s], (use - 1) & 1u, P, C)) return;
    d.b = b;
    d.kind = kind;
    d.kf = kf;
    if (kind == K_P1) {
      const int i = sub / P.nch1, c = sub - i * P.nch1;
      d.i = i; d.c = c;
      d.e0 = c * P.ch1;
      d.n = min(P.ch1, P.V - d.e0);
      const unsigned char* tseg =
          P.Lt + ((size_t(b) * P.R + i) * size_t(P.V) + d.e0) * E::ES;
      // greedy verification reads target rows only (it has no draft logits)
      const unsigned char* dseg =
          (!GREEDY && i < P.gamma && P.Ld)
              ? P.Ld + ((size_t(b) * P.gamma + i) * size_t(P.V) + d.e0) * E::ES
              : nullptr;
      issue<DT>(C, s, slot, d, tseg, dseg);
    } else if (kind == K_P2) {
      d.c = sub;
      Record r;
      const bool ok = wait_flag(P, C, b, epoch);
      if (ok) r = load_record(&P.rec[b]);
      else r.mode = MODE_INVALID;
      d.rec = r;
      if (r.mode == MODE_INVALID) {
        d.kind = K_SKIP;
        mbar_arrive(&C.full[s]);
        continue;
      }
      d.i = (r.mode == MODE_BONUS) ? P.gamma : r.k;
      d.e0 = sub * P.ch2;
      d.n = min(P.ch2, P.V - d.e0);
      const unsigned char* tseg =
          P.Lt + ((size_t(b) * P.R + d.i) * size_t(P.V) + d.e0) * E::ES;
      const unsigned char* dseg =
          r.mode == MODE_REJECT
              ? P.Ld + ((size_t(b) * P.gamma + r.k) * size_t(P.V) + d.e0) * E::ES
              : nullptr;
      issue<DT>(C, s, slot, d, tseg, dseg);
    } else {  // D and T3 carry no data
      mbar_arrive(&C.full[s]);
    }
  }
}

// --------------------------------------------------- consumers and books

// Staging entry e for a consumer warp: wait until the booking warp freed its
// previous use.
__device__ __forceinline__ bool stage_wait(const Params& P, SmemCtl& C, int e, unsigned use) {
  return use == 0 || mbar_wait(&C.freed[e], (use - 1) & 1u, P, C);
}

// Consumers: every warp reduces its share of each slot and publishes its own
// result (P1: the warp's (max, sum) pairs; P2: its sub-range mass) as
// epoch-tagged words; only D, T3 and the end marker go on to the booking
// warp through the staging ring (counted by dseq).
template <int DT, bool GREEDY>
__device__ void consumer(const Params& P, SmemCtl& C, const unsigned char* slots) {
  using E = Elem<DT>;
  const int cw = int(threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
  const unsigned epoch = C.epoch;
  long long dseq = 0;
  for (long long seq = 0;; ++seq) {
    const int s = int(seq % NSLOT);
    const unsigned use = unsigned(seq / NSLOT);
    if (!mbar_wait(&C.full[s], use & 1u, P, C)) return;
    const Desc d = C.desc[s];
    const unsigned char* slot = slots + size_t(s) * SLOT;
    // each warp hands the slot back as soon as it holds its share elsewhere
    bool released = false;
    auto release = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&C.empty[s]);
      released = true;
    };
    if (d.kind == K_P1) {
      const unsigned char* tseg =
          P.Lt + ((size_t(d.b) * P.R + d.i) * size_t(P.V) + d.e0) * E::ES;
      float4 out;
      if (GREEDY) {
        float best;
        int bi, nan;
        warp_argmax<DT>(slot, d.nb_t, tseg, d.head_t, d.n, d.e0, cw, lane, best, bi, nan, release);
        out = make_float4(best, __int_as_float(bi), __int_as_float(nan), 0.f);
      } else {
        const bool has_d = d.i < P.gamma;
        const unsigned char* dseg =
            has_d ? P.Ld + ((size_t(d.b) * P.gamma + d.i) * size_t(P.V) + d.e0) * E::ES
                  : nullptr;
        warp_ms2<DT>(slot, slot + HALF, d, tseg, dseg, has_d, d.kf, cw, lane, out, release);
      }
      // every warp publishes its own partial; the D task combines them
      if (lane == 0) {
        Partial* dst = P.part + ((size_t(d.b) * P.R + d.i) * P.nch1 + d.c) * NCW + cw;
        st_pair(&dst->w[0], tagged(epoch, __float_as_uint(out.x)), tagged(epoch, __float_as_uint(out.y)));
        st_pair(&dst->w[2], tagged(epoch, __float_as_uint(out.z)), tagged(epoch, __float_as_uint(out.w)));
      }
    } else if (!GREEDY && (d.kind == K_P2 || d.kind == K_SKIP)) {
      const double z = d.kind == K_P2 ? warp_p2_mass<DT>(P, d, slot, cw, lane, release) : 0.0;
      if (lane == 0) {
        ZPart* zp = P.z2 + size_t(d.b) * P.nch2 + d.c;
        st_pair(&zp->w[2 * cw], tagged(epoch, unsigned(__double2loint(z))),
                tagged(epoch, unsigned(__double2hiint(z))));
      }
    }
    if (!released) release();
    if (d.kind == K_D || d.kind == K_T3 || d.kind == K_END) {
      const int e = int(dseq % NSTAGE);
      const unsigned euse = unsigned(dseq / NSTAGE);
      ++dseq;
      if (!stage_wait(P, C, e, euse)) return;
      if (d.kind == K_D)
        for (int i = cw; i < P.R; i += NCW) {
          RowStat r;
          if (GREEDY) row_decide_greedy<DT>(P, C, d.b, i, r);
          else row_decide_sample<DT>(P, C, d.b, i, d.kf, r);
          if (lane == 0) C.rows[e][i] = r;
        }
      if (lane == 0) {
        if (cw == 0) C.sdesc[e] = d;
        mbar_arrive(&C.staged[e]);
      }
      if (d.kind == K_END) return;
    }
  }
}

__device__ __forceinline__ bool mbar_test(unsigned long long* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Are request b's decision and every phase-2 sub-range mass published?
__device__ bool t3_ready(const Params& P, SmemCtl& C, int b) {
  const int lane = threadIdx.x & 31;
  const unsigned epoch = C.epoch;
  int ok = 1;
  if (lane == 0) ok = ld_acquire(&P.req[b].flag) == epoch;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok) return false;
  const ZPart* zp = P.z2 + size_t(b) * P.nch2;
  bool all = true;
  for (int q = lane; q < P.nch2 * NCW; q += 32) {
    unsigned long long lo, hi;
    ld_pair(&zp[q / NCW].w[2 * (q % NCW)], lo, hi);
    all = all && is_mine(lo, epoch) && is_mine(hi, epoch);
  }
  return __all_sync(0xffffffffu, all);
}

constexpr int DEFCAP = 16;  // T3 tasks the booking warp may hold back

// The booking warp: request decisions of D tasks, and T3 draws, which it
// holds back (up to DEFCAP) while their inputs are not yet published and
// re-probes when idle, so that a slow request never delays another's decision.
template <int DT, bool GREEDY>
__device__ void booking(const Params& P, SmemCtl& C) {
  const int lane = threadIdx.x & 31;
  int* defer = C.defer;
  int ndef = 0;
  unsigned long long last_probe = 0, last_progress = globaltimer();
  for (long long dseq = 0;;) {
    const int e = int(dseq % NSTAGE);
    const unsigned euse = unsigned(dseq / NSTAGE);
    if (mbar_test(&C.staged[e], euse & 1u)) {
      const Desc d = C.sdesc[e];
      ++dseq;
      last_progress = globaltimer();
      if (d.kind == K_END) break;
      if (d.kind == K_D) {  // frees the entry itself once the rows are read
        if (GREEDY) request_decide_greedy(P, C, e, d.b);
        else request_decide_sample<DT>(P, C, e, d.b);
        continue;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&C.freed[e]);
      if (GREEDY) continue;
      if (ndef == 0 && t3_ready(P, C, d.b)) {
        task_t3<DT>(P, C, d.b);
      } else {
        if (ndef == DEFCAP) {  // full: finish the oldest (bounded wait)
          task_t3<DT>(P, C, defer[0]);
          if (lane == 0)
            for (int k = 1; k < ndef; ++k) defer[k - 1] = defer[k];
          __syncwarp();
          --ndef;
        }
        if (lane == 0) defer[ndef] = d.b;
        __syncwarp();
        ++ndef;
      }
      continue;
    }
    const unsigned long long now = globaltimer();
    const bool stop = *reinterpret_cast<volatile int*>(&P.ctrl->abort) ||
                      *reinterpret_cast<volatile int*>(&C.abort);
    if (__any_sync(0xffffffffu, stop)) break;
    if (now - last_progress > WAIT_LIMIT_NS) {
      if (lane == 0) give_up(P, C);
      __syncwarp();
      break;
    }
    if (ndef > 0) {
      if (now - last_probe > 1500) {
        last_probe = now;
        if (t3_ready(P, C, defer[0])) {
          task_t3<DT>(P, C, defer[0]);
          if (lane == 0)
            for (int k = 1; k < ndef; ++k) defer[k - 1] = defer[k];
          __syncwarp();
          --ndef;
          last_progress = globaltimer();
        }
      } else {
        __nanosleep(200);
      }
    } else if (!mbar_wait(&C.staged[e], euse & 1u, P, C)) {
      break;
    }
  }
  for (int k = 0; k < ndef; ++k) task_t3<DT>(P, C, defer[k]);  // the rest (bounded waits)
}

// --------------------------------------------------------- the kernel

template <int DT, bool GREEDY>
__global__ void __launch_bounds__(NTHR, 1) sv_kernel(const Params P) {
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* slots = smem;
  SmemCtl& C = *reinterpret_cast<SmemCtl*>(smem + size_t(NSLOT) * SLOT);
  if (threadIdx.x == 0) {
    C.epoch = __ldcg(&P.ctrl->epoch_counter) + 1u;
    C.abort = 0;
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&C.full[s], 1);
      mbar_init(&C.empty[s], NCW);
    }
    for (int e = 0; e < NSTAGE; ++e) {
      mbar_init(&C.staged[e], NCW);
      mbar_init(&C.freed[e], 1);
    }
  }
  if (!GREEDY)
    for (int b = threadIdx.x; b < min(P.B, KF_CAP); b += NTHR) C.kf_tab[b] = LOG2E_F / __ldg(P.temp + b);
  __syncthreads();
  const int warp = int(threadIdx.x >> 5);
  if (warp == 0) {
    if (threadIdx.x == 0) producer<DT, GREEDY>(P, C, slots);
  } else if (warp <= NCW) {
    consumer<DT, GREEDY>(P, C, slots);
  } else {
    booking<DT, GREEDY>(P, C);
  }
  __syncthreads();
  // exit: the last CTA out checks and resets the control block
  if (threadIdx.x == 0) {
    const unsigned old = atomicAdd(&P.ctrl->exit_count, 1u);
    if (old == gridDim.x - 1) {
      __threadfence();
      const unsigned long long tc = __ldcg(&P.ctrl->task);
      if (tc != (unsigned long long)P.total + 2ull * gridDim.x) set_status(P, SV_ST_WORKSPACE);
      P.ctrl->task = 0ull;
      P.ctrl->exit_count = 0u;
      P.ctrl->abort = 0;
      const unsigned e = P.ctrl->epoch_counter;
      P.ctrl->epoch_counter = (e + 1u) % 0xFFFFFFFFu;
    }
  }
}

// ---------------------------------------------------------------- host

struct Tuning {
  int chunk = 0, lag = 0;
};
Tuning g_tune;

struct DevCache {
  bool init = false;
  int sms = 0;
};
std::mutex g_mu;
DevCache g_dev[64];

template <int DT, bool G>
bool prepare_kernel() {
  return cudaFuncSetAttribute(sv_kernel<DT, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(SMEM_BYTES)) == cudaSuccess;
}

int device_info(int& sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DevCache& d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SV_ERR_CUDA;
    if (!prepare_kernel<SV_F32, false>() || !prepare_kernel<SV_F32, true>() ||
        !prepare_kernel<SV_BF16, false>() || !prepare_kernel<SV_BF16, true>())
      return SV_ERR_CUDA;
    d.init = true;
  }
  sms = d.sms;
  return SV_OK;
}

int round_up(long long x, int m) { return int(((x + m - 1) / m) * m); }

int launch(bool greedy, const void* Lt, const void* Ld, const int32_t* x, const float* u_acc,
           const float* u_res, const float* temp, int B, int gamma, int V, int dtype,
           int32_t* out_tokens, int32_t* out_n, float* out_p, float* out_Z, void* ws,
           size_t ws_bytes, int32_t* status, void* stream) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (B < 0 || gamma < 0 || gamma > SV_MAX_GAMMA || V < 1) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;  // nothing to do; empty buffers may be NULL
  const int ES = dtype == SV_F32 ? 4 : 2;
  if (!Lt || (!x && gamma > 0) || !out_tokens || !out_n) return SV_ERR_INVALID_ARG;
  if (!greedy && (!u_res || !temp || (gamma > 0 && (!Ld || !u_acc)))) return SV_ERR_INVALID_ARG;
  auto mis = [](const void* p, int a) { return p && (reinterpret_cast<uintptr_t>(p) % a) != 0; };
  if (mis(Lt, ES) || mis(Ld, ES) || mis(x, 4) || mis(u_acc, 4) || mis(u_res, 4) || mis(temp, 4) ||
      mis(out_tokens, 4) || mis(out_n, 4) || mis(out_p, 4) || mis(out_Z, 4) || mis(status, 4))
    return SV_ERR_INVALID_ARG;
  const Layout L = make_layout(B, gamma, V);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < L.total) return SV_ERR_WORKSPACE;

  int sms = 0;
  int rc = device_info(sms);
  if (rc != SV_OK) return rc;
  const int R = gamma + 1;
  const long long units = (long long)B * R;
  const int chmax = HALF / ES;  // a row chunk must fit half a slot

  // phase-1 chunk: at most half a slot, at least CH1_MIN (or the whole row),
  // and small enough that every SM gets several tasks
  int ch1;
  if (g_tune.chunk > 0) {
    ch1 = round_up(g_tune.chunk, 64);
  } else {
    const long long by_bytes = (V + chmax - 1) / chmax;
    const long long by_tasks = (8LL * min(sms, SMS_CAP) + units - 1) / units;
    const long long want = max(1LL, max(by_bytes, by_tasks));
    ch1 = round_up((V + want - 1) / want, 64);
  }
  ch1 = min(chmax, max(ch1, min(CH1_MIN, round_up(V, 64))));
  if ((V + ch1 - 1) / ch1 > L.nch1_max)  // a tuning override asked for more chunks than fit
    ch1 = min(chmax, round_up((V + L.nch1_max - 1) / L.nch1_max, 64));
  const int nch1 = (V + ch1 - 1) / ch1;
  if (nch1 > L.nch1_max) return SV_ERR_INVALID_ARG;

  Params P;
  P.Lt = static_cast<const unsigned char*>(Lt);
  P.Ld = static_cast<const unsigned char*>(Ld);
  P.x = x; P.u_acc = u_acc; P.u_res = u_res; P.temp = temp;
  P.B = B; P.gamma = gamma; P.V = V; P.R = R;
  P.ch1 = ch1; P.nch1 = nch1;
  P.np1 = nch1 * NCW;
  P.ch2 = chmax;
  P.nch2 = (V + chmax - 1) / chmax;
  // each consumer warp takes a contiguous sub-range of a phase-2 chunk, a
  // whole number of 16-byte vectors long (the last one may be shorter)
  P.sub = round_up((chmax + NCW - 1) / NCW, 8);
  P.n1 = (long long)R * nch1;
  P.n2 = greedy ? 0 : P.nch2;
  P.draw = !greedy;
  // per request: its P1 chunks, one D task, and (sampling) its P2 chunks and one T3 task
  const long long per_req = P.n1 + 1 + (greedy ? 0 : P.n2 + 1);
  P.total = (long long)B * per_req;
  const long long grid = min((long long)sms, P.total);
  // a request's D, P2 and T3 tasks each come `lag` requests after the stage
  // before them: enough tasks in between to cover everything in flight
  // (every CTA's slot ring and claims, 1.5 times)
  if (g_tune.lag > 0) P.lag = g_tune.lag;
  else P.lag = int(max(1LL, (3 * grid * (NSLOT + 2) / 2 + per_req - 1) / per_req));
  {
    // regions of constant block composition between the block indices where a
    // stage starts or ends (see decode)
    const long long Lg = P.lag, Bl = B;
    auto block_size = [&](long long j) {
      long long z = 0;
      if (j < Bl) z += P.n1;
      if (j >= Lg && j < Bl + Lg) z += 1;
      if (P.draw && j >= 2 * Lg && j < Bl + 2 * Lg) z += P.n2;
      if (P.draw && j >= 3 * Lg && j < Bl + 3 * Lg) z += 1;
      return z;
    };
    const long long J = Bl + (P.draw ? 3 : 1) * Lg;
    long long cuts[9] = {0, Lg, Bl, Bl + Lg, 2 * Lg, Bl + 2 * Lg, 3 * Lg, Bl + 3 * Lg, J};
    std::sort(cuts, cuts + 9);
    P.nreg = 0;
    long long c = 0;
    for (int q = 0; q < 9; ++q) {
      const long long ja = cuts[q], jb = (q + 1 < 9) ? cuts[q + 1] : J;
      if (ja >= J || jb <= ja) continue;
      const long long sz = block_size(ja);
      if (sz > 0) {
        P.rj[P.nreg] = ja;
        P.rc[P.nreg] = c;
        P.rsz[P.nreg] = int(sz);
        ++P.nreg;
      }
      c += sz * (min(jb, J) - ja);
    }
    P.rj[P.nreg] = J;
    P.rc[P.nreg] = c;
    if (c != P.total || P.total >= (1LL << 31)) return SV_ERR_INVALID_ARG;
  }
  P.out_tokens = out_tokens; P.out_n = out_n; P.out_p = out_p; P.out_Z = out_Z;
  P.status = status;
  unsigned char* w = static_cast<unsigned char*>(ws);
  P.ctrl = reinterpret_cast<Ctrl*>(w + L.ctrl);
  P.req = reinterpret_cast<ReqCtl*>(w + L.req);
  P.rec = reinterpret_cast<Record*>(w + L.rec);
  P.part = reinterpret_cast<Partial*>(w + L.part);
  P.z2 = reinterpret_cast<ZPart*>(w + L.z2);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dim3 g{unsigned(grid)}, blk{unsigned(NTHR)};
  if (dtype == SV_F32) {
    if (greedy) sv_kernel<SV_F32, true><<<g, blk, SMEM_BYTES, st>>>(P);
    else sv_kernel<SV_F32, false><<<g, blk, SMEM_BYTES, st>>>(P);
  } else {
    if (greedy) sv_kernel<SV_BF16, true><<<g, blk, SMEM_BYTES, st>>>(P);
    else sv_kernel<SV_BF16, false><<<g, blk, SMEM_BYTES, st>>>(P);
  }
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
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
  return launch(false, target_logits, draft_logits, draft_tokens, u_accept, u_resample,
                temperature, B, gamma, V, dtype, out_tokens, out_num_accepted, out_p, out_Z,
                workspace, workspace_bytes, dev_status, stream);
}

int spec_verify(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                const float* u_accept, const float* u_resample, const float* temperature, int B,
                int gamma, int V, int dtype, int32_t* out_tokens, int32_t* out_num_accepted,
                void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return launch(false, target_logits, draft_logits, draft_tokens, u_accept, u_resample,
                temperature, B, gamma, V, dtype, out_tokens, out_num_accepted, nullptr, nullptr,
                workspace, workspace_bytes, dev_status, stream);
}

int spec_verify_greedy(const void* target_logits, const int32_t* draft_tokens, int B, int gamma,
                       int V, int dtype, int32_t* out_tokens, int32_t* out_num_accepted,
                       void* workspace, size_t workspace_bytes, int32_t* dev_status,
                       void* stream) {
  return launch(true, target_logits, nullptr, draft_tokens, nullptr, nullptr, nullptr, B, gamma,
                V, dtype, out_tokens, out_num_accepted, nullptr, nullptr, workspace,
                workspace_bytes, dev_status, stream);
}

}  // extern "C"

// ------------------------------------------------- no-allocation entry point
// Scratch for spec_verify_noalloc, in the library's own device memory.  Host
// code may not use this name as a device address (on the host it names a
// stand-in object): the address is looked up per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SV_NOALLOC_MAX_WORKSPACE];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};  // device address of g_noalloc_scratch, per device

// Device address of the scratch on the current device; the lookup runs once
// per device, with that device current.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SV_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
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
    return launch(false, target_logits, draft_logits, draft_tokens, u_accept, u_resample,
                  temperature, B, gamma, V, dtype, out_tokens, out_num_accepted, nullptr,
                  nullptr, nullptr, 0, dev_status, stream);
  void* scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc != SV_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the task counter and the exit counter must start at zero; the launch
  // epoch after them must survive from call to call
  if (cudaMemsetAsync(scratch, 0, offsetof(Ctrl, epoch_counter), st) != cudaSuccess ||
      cudaMemsetAsync(static_cast<unsigned char*>(scratch) + offsetof(Ctrl, abort), 0,
                      sizeof(int), st) != cudaSuccess)
    return SV_ERR_CUDA;
  return launch(false, target_logits, draft_logits, draft_tokens, u_accept, u_resample,
                temperature, B, gamma, V, dtype, out_tokens, out_num_accepted, nullptr, nullptr,
                scratch, SV_NOALLOC_MAX_WORKSPACE, dev_status, stream);
}

int sv_set_tuning(int chunk_elems, int ctas_per_sm, int lag_requests) {
  (void)ctas_per_sm;  // the kernel always runs one CTA per SM
  g_tune.chunk = chunk_elems > 0 ? chunk_elems : 0;
  g_tune.lag = lag_requests > 0 ? lag_requests : 0;
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

int sv_version(void) { return 200; }

}  // extern "C"
