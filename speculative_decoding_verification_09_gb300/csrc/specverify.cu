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
// GPU structure: ONE persistent launch per call.  CTAs pull task ids from an
// atomic counter in a fixed global order:
//   P1(b, i, c)  chunk c of target row i and draft row i of request b: one
//                streaming pass with an online (max, sum 2^((l-max)*log2e/T))
//                per row, written as a partial.  The CTA that finishes the last
//                P1 task of b (atomic ticket) combines the partials in fp64,
//                computes P_t(x_i), P_d(x_i), the accept bits, the first
//                rejection k, writes every output except token k and publishes
//                a decision record (release store of the launch epoch).
//   P2(b, c)     chunk c of the row pair the last token is drawn from (residual
//                max(0, P_t - P_d) of row k, or P_t of row gamma for the bonus):
//                its mass.  P2 tasks of b sit `lag` requests after P1 of b in
//                the order, so they normally find the record ready; otherwise
//                they wait (bounded) for it.  The row pair was streamed moments
//                before, so this pass reads L2, not HBM.
//   P3(b)        run by the CTA finishing the last P2 task of b: picks the chunk
//                where the running mass crosses u * Z and scans it in index
//                order (block prefix sums) to emit token k.
// A waiting task only waits on tasks claimed earlier from the counter, and
// those never wait on later ones, so every wait ends; each wait still gives
// up after one second (SV_ST_TIMEOUT) instead of hanging.
// The greedy kernel runs P1 tasks (chunk argmax) and a decider only.
#include <cuda_runtime.h>
#include <limits.h>
#include <stddef.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "specverify.h"

namespace {

constexpr int NT = 256;           // threads per CTA
constexpr int NW = NT / 32;       // warps per CTA
constexpr int CH1_MIN = 512;      // smallest phase-1 chunk (elements)
constexpr int CH2 = 8192;         // phase-2 chunk (elements), a multiple of 64
constexpr int MAXR = SV_MAX_GAMMA + 1;
constexpr float LOG2E_F = 1.4426950408889634f;
constexpr double LOG2E_D = 1.4426950408889634;
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;  // one second

enum : int { MODE_INVALID = 0, MODE_REJECT = 1, MODE_BONUS = 2, MODE_TARGET = 3 };

// ------------------------------------------------------------ workspace

struct Ctrl {                 // 64 bytes at the start of the workspace
  unsigned long long task;    // next task id
  unsigned exit_count;        // CTAs that finished
  unsigned epoch_counter;     // launch epoch = epoch_counter + 1
  int abort;                  // set when a wait gave up
  int pad[11];
};
// Arrival counters carry the launch epoch in their high 32 bits; a counter
// holding another launch's epoch (or anything else) counts as zero, so no
// per-request word is ever reset and workspaces can be shared by calls of
// any shape that fits.
struct ReqCtl {               // per request, 32 bytes
  unsigned long long p1;      // (epoch << 32) | P1 arrivals
  unsigned long long p2;      // (epoch << 32) | P2 arrivals
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
struct Partial {              // per (request, position, chunk), 32 bytes
  float a, b, c, d;           // sampling: m_t, s_t, m_d, s_d; greedy: value, index bits, nan
  unsigned epoch;
  int pad[3];
};
struct ZPart {                // per (request, phase-2 chunk), 16 bytes
  double z;
  unsigned epoch;
  int pad;
};

static_assert(sizeof(Ctrl) == 64 && sizeof(ReqCtl) == 32 && sizeof(Record) == 48 &&
                  sizeof(Partial) == 32 && sizeof(ZPart) == 16,
              "workspace record sizes");

struct Layout {
  size_t ctrl, req, rec, part, z2, total;
  int nch1_max, nch2;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

Layout make_layout(int B, int gamma, int V) {
  Layout L;
  const size_t R = size_t(gamma) + 1;
  L.nch1_max = (V + CH1_MIN - 1) / CH1_MIN;
  L.nch2 = (V + CH2 - 1) / CH2;
  L.ctrl = 0;
  L.req = align256(sizeof(Ctrl));
  L.rec = L.req + align256(size_t(B) * sizeof(ReqCtl));
  L.part = L.rec + align256(size_t(B) * sizeof(Record));
  L.z2 = L.part + align256(size_t(B) * R * L.nch1_max * sizeof(Partial));
  L.total = L.z2 + align256(size_t(B) * L.nch2 * sizeof(ZPart));
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
  int ch1, nch1, ch2, nch2, lag;
  long long n1, n2, total;
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

// -------------------------------------------------------- device helpers

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint32_t bmax_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// A decision record as stored by another CTA (read through L2).
__device__ __forceinline__ Record load_record(const Record* p) {
  Record r;
  const int4 a = __ldcg(reinterpret_cast<const int4*>(p));
  const int4 b = __ldcg(reinterpret_cast<const int4*>(p) + 1);
  r.k = a.x; r.mode = a.y; r.mt = __int_as_float(a.z); r.kf = __int_as_float(a.w);
  r.epoch = unsigned(b.x); r.ist_hi = __int_as_float(b.y); r.ist_lo = __int_as_float(b.z);
  r.c0_hi = __int_as_float(b.w);
  const int4 c = __ldcg(reinterpret_cast<const int4*>(p) + 2);
  r.c0_lo = __int_as_float(c.x);
  return r;
}
// One arrival on an epoch-tagged counter; returns this launch's count after
// the arrival (1 for the first), or 0 if the update kept failing.
__device__ __forceinline__ unsigned arrive(unsigned long long* w, unsigned epoch) {
  const unsigned long long tag = (unsigned long long)epoch << 32;
  unsigned long long cur = __ldcg(w);
  for (int it = 0; it < (1 << 20); ++it) {
    const unsigned long long nxt = ((cur >> 32) == epoch) ? cur + 1 : (tag | 1ull);
    const unsigned long long prev = atomicCAS(w, cur, nxt);
    if (prev == cur) return unsigned(nxt & 0xffffffffull);
    cur = prev;
  }
  return 0u;
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

template <int DT>
struct Elem;
template <>
struct Elem<SV_F32> {
  static constexpr int ES = 4, VEC = 4;
  __device__ static float load(const unsigned char* base, long long idx) {
    return __ldg(reinterpret_cast<const float*>(base) + idx);
  }
  __device__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  __device__ static float vmax(const uint4& v) {
    return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                    fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
};
template <>
struct Elem<SV_BF16> {
  static constexpr int ES = 2, VEC = 8;
  __device__ static float load(const unsigned char* base, long long idx) {
    return __uint_as_float(uint32_t(__ldg(reinterpret_cast<const unsigned short*>(base) + idx))
                           << 16);
  }
  __device__ static void unpack(const uint4& v, float* f) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z); f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
  }
  __device__ static float vmax(const uint4& v) {
    uint32_t m = bmax_nan(bmax_nan(v.x, v.y), bmax_nan(v.z, v.w));
    return fmax_nan(bf_lo(m), bf_hi(m));
  }
};

// Row segment [e0, e0+n) split at 16-byte boundaries: `head` single elements,
// `nvec` aligned 16-byte vectors, then single tail elements.
struct Seg {
  const unsigned char* p0;
  int n, head, nvec, tail0;
};
template <int DT>
__device__ __forceinline__ Seg make_seg(const unsigned char* row, int e0, int n) {
  using E = Elem<DT>;
  Seg s;
  s.p0 = row + size_t(e0) * E::ES;
  s.n = n;
  int h = int(((16u - unsigned(reinterpret_cast<uintptr_t>(s.p0) & 15u)) & 15u) / E::ES);
  s.head = h < n ? h : n;
  s.nvec = (n - s.head) / E::VEC;
  s.tail0 = s.head + s.nvec * E::VEC;
  return s;
}

// ------------------------------------------------- online max / sum-exp
// State (m, s): s = sum over seen elements of 2^((l - m) * kf).  NaN sticks in
// s; +inf turns s into NaN; an all -inf stream keeps m = -inf, s = 0.

__device__ __forceinline__ void ms_raise(float& m, float& s, float vm, float kf) {
  if (!(vm <= m)) {
    s *= ex2((m - vm) * kf);
    m = vm;
  }
}
template <int DT>
__device__ __forceinline__ void ms_vec(const uint4& v, float& m, float& s, float kf) {
  using E = Elem<DT>;
  ms_raise(m, s, E::vmax(v), kf);
  if (m > -INFINITY) {
    float f[E::VEC];
    E::unpack(v, f);
#pragma unroll
    for (int e = 0; e < E::VEC; ++e) f[e] = ex2((f[e] - m) * kf);
#pragma unroll
    for (int w = 1; w < E::VEC; w *= 2)
#pragma unroll
      for (int e = 0; e < E::VEC; e += 2 * w) f[e] += f[e + w];
    s += f[0];
  }
}
__device__ __forceinline__ void ms_one(float l, float& m, float& s, float kf) {
  ms_raise(m, s, l, kf);
  if (m > -INFINITY) s += ex2((l - m) * kf);
}
__device__ __forceinline__ void ms_merge(float& m, float& s, float m2, float s2, float kf) {
  float mm = fmaxf(m, m2);
  if (mm == -INFINITY) {
    s = s + s2;
  } else {
    s = s * ex2((m - mm) * kf) + s2 * ex2((m2 - mm) * kf);
  }
  m = mm;
}

template <int DT>
__device__ void row_ms(const unsigned char* row, int e0, int n, float kf, float& m, float& s) {
  using E = Elem<DT>;
  const Seg g = make_seg<DT>(row, e0, n);
  const int tid = threadIdx.x;
  if (tid < g.head) ms_one(E::load(g.p0, tid), m, s, kf);
  const uint4* vp = reinterpret_cast<const uint4*>(g.p0 + size_t(g.head) * E::ES);
  int j = tid;
  for (; j + 3 * NT < g.nvec; j += 4 * NT) {
    uint4 a = ld_stream(vp + j), b = ld_stream(vp + j + NT);
    uint4 c = ld_stream(vp + j + 2 * NT), d = ld_stream(vp + j + 3 * NT);
    ms_vec<DT>(a, m, s, kf);
    ms_vec<DT>(b, m, s, kf);
    ms_vec<DT>(c, m, s, kf);
    ms_vec<DT>(d, m, s, kf);
  }
  for (; j < g.nvec; j += NT) ms_vec<DT>(ld_stream(vp + j), m, s, kf);
  if (tid < g.n - g.tail0) ms_one(E::load(g.p0, g.tail0 + tid), m, s, kf);
}

// -------------------------------------------------- greedy argmax state
// (best, idx): largest value, lowest index among its occurrences; idx stays
// INT_MAX while only -inf was seen.  nan records any NaN.

__device__ __forceinline__ void am_one(float l, int idx, float& best, int& bi, int& nan) {
  if (l != l) nan = 1;
  else if (l > best) { best = l; bi = idx; }
}
template <int DT>
__device__ __forceinline__ void am_vec(const uint4& v, int idx0, float& best, int& bi, int& nan) {
  using E = Elem<DT>;
  float vm = E::vmax(v);
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
    bi = idx0 + first;
  }
}
__device__ __forceinline__ void am_merge(float& best, int& bi, int& nan, float b2, int i2, int n2) {
  if (b2 > best || (b2 == best && i2 < bi)) { best = b2; bi = i2; }
  nan |= n2;
}

template <int DT>
__device__ void row_argmax(const unsigned char* row, int e0, int n, float& best, int& bi,
                           int& nan) {
  using E = Elem<DT>;
  const Seg g = make_seg<DT>(row, e0, n);
  const int tid = threadIdx.x;
  if (tid < g.head) am_one(E::load(g.p0, tid), e0 + tid, best, bi, nan);
  const uint4* vp = reinterpret_cast<const uint4*>(g.p0 + size_t(g.head) * E::ES);
  const int base = e0 + g.head;
  int j = tid;
  for (; j + 3 * NT < g.nvec; j += 4 * NT) {
    uint4 a = ld_stream(vp + j), b = ld_stream(vp + j + NT);
    uint4 c = ld_stream(vp + j + 2 * NT), d = ld_stream(vp + j + 3 * NT);
    am_vec<DT>(a, base + j * E::VEC, best, bi, nan);
    am_vec<DT>(b, base + (j + NT) * E::VEC, best, bi, nan);
    am_vec<DT>(c, base + (j + 2 * NT) * E::VEC, best, bi, nan);
    am_vec<DT>(d, base + (j + 3 * NT) * E::VEC, best, bi, nan);
  }
  for (; j < g.nvec; j += NT) am_vec<DT>(ld_stream(vp + j), base + j * E::VEC, best, bi, nan);
  if (tid < g.n - g.tail0) am_one(E::load(g.p0, g.tail0 + tid), e0 + g.tail0 + tid, best, bi, nan);
}

// ------------------------------------------------------ shared memory

struct SMem {
  unsigned long long task;
  unsigned epoch;
  int flag;
  int ok;
  float rf[4][NW];
  int ri[2][NW];
  double rd[NW];
  double incl[NT];
  // decider
  float pt[MAXR], pd[MAXR], mt[MAXR], md[MAXR];
  double St[MAXR], Sd[MAXR];
  int acc[MAXR], amax[MAXR];
  int bad;
  Record rec;
  // P3
  int hit_t, hit_v, last_v;
};

__device__ __forceinline__ void set_status(const Params& P, int bits) {
  if (bits && P.status) atomicOr(P.status, bits);
}
// Evidence that the workspace did not hold what this launch wrote (a record
// or partial with another epoch): the call's results are void.
__device__ __forceinline__ void mark_dirty(const Params& P) { set_status(P, SV_ST_WORKSPACE); }

// Block reduction of two (m, s) pairs; the result is valid in every thread.
__device__ void block_ms2(float& m1, float& s1, float& m2, float& s2, float kf, SMem& sm) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float a = __shfl_xor_sync(0xffffffffu, m1, o), b = __shfl_xor_sync(0xffffffffu, s1, o);
    float c = __shfl_xor_sync(0xffffffffu, m2, o), d = __shfl_xor_sync(0xffffffffu, s2, o);
    ms_merge(m1, s1, a, b, kf);
    ms_merge(m2, s2, c, d, kf);
  }
  if (lane == 0) { sm.rf[0][w] = m1; sm.rf[1][w] = s1; sm.rf[2][w] = m2; sm.rf[3][w] = s2; }
  __syncthreads();
  m1 = sm.rf[0][0]; s1 = sm.rf[1][0]; m2 = sm.rf[2][0]; s2 = sm.rf[3][0];
  for (int i = 1; i < NW; ++i) {
    ms_merge(m1, s1, sm.rf[0][i], sm.rf[1][i], kf);
    ms_merge(m2, s2, sm.rf[2][i], sm.rf[3][i], kf);
  }
  __syncthreads();
}

__device__ void block_argmax(float& best, int& bi, int& nan, SMem& sm) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float b2 = __shfl_xor_sync(0xffffffffu, best, o);
    int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    int n2 = __shfl_xor_sync(0xffffffffu, nan, o);
    am_merge(best, bi, nan, b2, i2, n2);
  }
  if (lane == 0) { sm.rf[0][w] = best; sm.ri[0][w] = bi; sm.ri[1][w] = nan; }
  __syncthreads();
  best = sm.rf[0][0]; bi = sm.ri[0][0]; nan = sm.ri[1][0];
  for (int i = 1; i < NW; ++i) am_merge(best, bi, nan, sm.rf[0][i], sm.ri[0][i], sm.ri[1][i]);
  __syncthreads();
}

__device__ double block_sum_d(double v, SMem& sm) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sm.rd[w] = v;
  __syncthreads();
  double t = 0.0;
  for (int i = 0; i < NW; ++i) t += sm.rd[i];
  __syncthreads();
  return t;
}

// Inclusive prefix sum over the CTA in thread order; also leaves every
// thread's inclusive value in sm.incl.
__device__ double block_incl_scan(double v, SMem& sm) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    double n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) sm.rd[w] = v;
  __syncthreads();
  double off = 0.0;
  for (int i = 0; i < w; ++i) off += sm.rd[i];
  v += off;
  sm.incl[threadIdx.x] = v;
  __syncthreads();
  return v;
}

// ------------------------------------------------------------- decider

// fp64 combine of one row's chunk partials (m_c, s_c) held in fields
// (a, b) or (c, d); executed by one warp, result valid in every lane.
__device__ void warp_row_combine(const Partial* pp, int nch, bool draft, float kf,
                                 unsigned epoch, float& m_out, double& S_out, int& stale) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  for (int c = lane; c < nch; c += 32) {
    float4 v = __ldcg(reinterpret_cast<const float4*>(pp + c));
    unsigned ep = __ldcg(&pp[c].epoch);
    if (ep != epoch) stale = 1;
    m = fmaxf(m, draft ? v.z : v.x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  double S = 0.0;
  for (int c = lane; c < nch; c += 32) {
    float4 v = __ldcg(reinterpret_cast<const float4*>(pp + c));
    float mc = draft ? v.z : v.x, sc = draft ? v.w : v.y;
    if (m == -INFINITY) S += double(sc);
    else S += double(sc) * exp2((double(mc) - double(m)) * double(kf));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
  stale = __any_sync(0xffffffffu, stale);
  m_out = m;
  S_out = S;
}

__device__ __forceinline__ bool row_ok(float m, double S) {
  return (m > -INFINITY) && (m < INFINITY) && (S > 0.0) && (S < INFINITY);
}

template <int DT>
__device__ void decide_sample(const Params& P, int b, SMem& sm) {
  using E = Elem<DT>;
  const int g = P.gamma, R = P.R, V = P.V;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const unsigned epoch = sm.epoch;
  const float T = __ldg(P.temp + b);
  const bool t_ok = isfinite(T) && T >= 0x1p-126f;
  const float kf = LOG2E_F / T;
  const double k64 = LOG2E_D / double(T);
  if (threadIdx.x == 0) sm.bad = 0;
  __syncthreads();
  int stale = 0;
  for (int i = w; i < R; i += NW) {
    const Partial* pp = P.part + (size_t(b) * R + i) * P.nch1;
    float mt, md = 0.f;
    double St, Sd = 1.0;
    warp_row_combine(pp, P.nch1, false, kf, epoch, mt, St, stale);
    if (i < g) warp_row_combine(pp, P.nch1, true, kf, epoch, md, Sd, stale);
    if (lane == 0) {
      int bad = 0;
      if (!row_ok(mt, St) || (i < g && !row_ok(md, Sd))) bad |= SV_ST_NONFINITE;
      float pt = NAN, pd = NAN;
      int acc = 1;
      if (i < g) {
        const int xi = __ldg(P.x + size_t(b) * g + i);
        if (xi < 0 || xi >= V) {
          bad |= SV_ST_BAD_TOKEN;
        } else if (!bad && t_ok) {
          const float lt = E::load(P.Lt, (long long)(size_t(b) * R + i) * V + xi);
          const float ld = E::load(P.Ld, (long long)(size_t(b) * g + i) * V + xi);
          const double dpt = exp2((double(lt) - double(mt)) * k64) / St;
          const double dpd = exp2((double(ld) - double(md)) * k64) / Sd;
          const double r = dpd > 0.0 ? fmin(1.0, dpt / dpd) : 1.0;
          acc = double(__ldg(P.u_acc + size_t(b) * g + i)) <= r;
          pt = float(dpt);
          pd = float(dpd);
        }
      }
      sm.pt[i] = pt; sm.pd[i] = pd; sm.acc[i] = acc;
      sm.mt[i] = mt; sm.md[i] = md;
      sm.St[i] = St;
      sm.Sd[i] = Sd;
      if (bad) atomicOr(&sm.bad, bad);
    }
  }
  if (stale && lane == 0) atomicOr(&sm.bad, 0x100);
  __syncthreads();
  if (w == 0) {
    int bad = sm.bad;
    if (!t_ok) bad |= SV_ST_BAD_TEMP;
    if (bad & 0x100) { mark_dirty(P); bad &= ~0x100; }
    const bool valid = (bad == 0);
    const unsigned rej = __ballot_sync(0xffffffffu, lane < g && !sm.acc[lane]);
    const int k = rej ? __ffs(rej) - 1 : g;
    for (int i = lane; i < R; i += 32) {
      int tok = -1;
      if (valid && i < k) tok = __ldg(P.x + size_t(b) * g + i);
      if (!valid || i != k) P.out_tokens[size_t(b) * R + i] = tok;
    }
    if (P.out_p)
      for (int i = lane; i < g; i += 32) {
        P.out_p[(size_t(b) * g + i) * 2] = valid ? sm.pt[i] : NAN;
        P.out_p[(size_t(b) * g + i) * 2 + 1] = valid ? sm.pd[i] : NAN;
      }
    if (lane == 0) {
      P.out_n[b] = valid ? k : 0;
      if (!valid && P.out_Z) P.out_Z[b] = NAN;
      set_status(P, bad);
      Record r;
      r.k = k;
      r.mode = !valid ? MODE_INVALID : (k < g ? MODE_REJECT : MODE_BONUS);
      r.mt = sm.mt[k];
      r.kf = kf;
      r.epoch = epoch;
      const double ist = 1.0 / sm.St[k];
      r.ist_hi = float(ist);
      r.ist_lo = float(ist - double(r.ist_hi));
      // log2(P_d[v] / P_t[v]) = (l_d[v] - l_t[v]) * kf + (m_t - m_d) * kf + log2(S_t / S_d)
      const double c0 = k < g ? (double(sm.mt[k]) - double(sm.md[k])) * double(kf) +
                                    log2(sm.St[k] / sm.Sd[k])
                              : 0.0;
      r.c0_hi = float(c0);
      r.c0_lo = float(c0 - double(r.c0_hi));
      r.pad[0] = r.pad[1] = r.pad[2] = 0;
      P.rec[b] = r;
      __threadfence();
      const unsigned old = atomicExch(&P.req[b].flag, epoch);
      if (old == epoch) mark_dirty(P);
    }
  }
}

template <int DT>
__device__ void decide_greedy(const Params& P, int b, SMem& sm) {
  const int g = P.gamma, R = P.R, V = P.V;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const unsigned epoch = sm.epoch;
  if (threadIdx.x == 0) sm.bad = 0;
  __syncthreads();
  for (int i = w; i < R; i += NW) {
    const Partial* pp = P.part + (size_t(b) * R + i) * P.nch1;
    float best = -INFINITY;
    int bi = INT_MAX, nan = 0, stale = 0;
    for (int c = lane; c < P.nch1; c += 32) {
      float4 v = __ldcg(reinterpret_cast<const float4*>(pp + c));
      if (__ldcg(&pp[c].epoch) != epoch) stale = 1;
      am_merge(best, bi, nan, v.x, __float_as_int(v.y), __float_as_int(v.z));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float b2 = __shfl_xor_sync(0xffffffffu, best, o);
      int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      int n2 = __shfl_xor_sync(0xffffffffu, nan, o);
      am_merge(best, bi, nan, b2, i2, n2);
    }
    stale = __any_sync(0xffffffffu, stale);
    if (lane == 0) {
      int bad = 0;
      if (nan || bi == INT_MAX || best == INFINITY) bad |= SV_ST_NONFINITE;
      if (stale) bad |= 0x100;
      if (i < g) {
        const int xi = __ldg(P.x + size_t(b) * g + i);
        if (xi < 0 || xi >= V) bad |= SV_ST_BAD_TOKEN;
      }
      sm.amax[i] = bi;
      if (bad) atomicOr(&sm.bad, bad);
    }
  }
  __syncthreads();
  if (w == 0) {
    int bad = sm.bad;
    if (bad & 0x100) { mark_dirty(P); bad &= ~0x100; }
    const bool valid = (bad == 0);
    const unsigned mis =
        __ballot_sync(0xffffffffu, lane < g && __ldg(P.x + size_t(b) * g + lane) != sm.amax[lane]);
    const int k = mis ? __ffs(mis) - 1 : g;
    for (int i = lane; i < R; i += 32)
      P.out_tokens[size_t(b) * R + i] = (valid && i <= k) ? sm.amax[i] : -1;
    if (lane == 0) {
      P.out_n[b] = valid ? k : 0;
      set_status(P, bad);
    }
  }
}

// ------------------------------------------------------------ P1 tasks

template <int DT, bool GREEDY>
__device__ void task_p1(const Params& P, int b, int sub, SMem& sm) {
  using E = Elem<DT>;
  const int i = sub / P.nch1, c = sub - i * P.nch1;
  const int e0 = c * P.ch1;
  const int n = min(P.ch1, P.V - e0);
  const unsigned char* trow = P.Lt + (size_t(b) * P.R + i) * size_t(P.V) * E::ES;
  Partial out;
  if (GREEDY) {
    float best = -INFINITY;
    int bi = INT_MAX, nan = 0;
    row_argmax<DT>(trow, e0, n, best, bi, nan);
    block_argmax(best, bi, nan, sm);
    out.a = best; out.b = __int_as_float(bi); out.c = __int_as_float(nan); out.d = 0.f;
  } else {
    const float kf = LOG2E_F / __ldg(P.temp + b);
    float mt = -INFINITY, st = 0.f, md = -INFINITY, sd = 0.f;
    row_ms<DT>(trow, e0, n, kf, mt, st);
    if (i < P.gamma) {
      const unsigned char* drow = P.Ld + (size_t(b) * P.gamma + i) * size_t(P.V) * E::ES;
      row_ms<DT>(drow, e0, n, kf, md, sd);
    }
    block_ms2(mt, st, md, sd, kf, sm);
    out.a = mt; out.b = st; out.c = md; out.d = sd;
  }
  if (threadIdx.x == 0) {
    Partial* dst = P.part + (size_t(b) * P.R + i) * P.nch1 + c;
    *reinterpret_cast<float4*>(dst) = make_float4(out.a, out.b, out.c, out.d);
    dst->epoch = sm.epoch;
    __threadfence();
    const unsigned cnt = arrive(&P.req[b].p1, sm.epoch);
    if (cnt == 0u) {
      atomicExch(&P.ctrl->abort, 1);
      set_status(P, SV_ST_TIMEOUT);
    }
    sm.flag = (cnt == (unsigned)P.n1);
    if (sm.flag) __threadfence();
  }
  __syncthreads();
  if (sm.flag) {
    if (GREEDY) decide_greedy<DT>(P, b, sm);
    else decide_sample<DT>(P, b, sm);
  }
}

// ------------------------------------------------------- P2 / P3 tasks

// Weight of one element of the final draw (fp32, identical in P2 and P3).
// Residual max(0, P_t - P_d) formed as P_t * (1 - 2^delta) with
// delta = log2(P_d / P_t), so it keeps its relative precision where the two
// rows nearly agree (no cancellation); the normaliser is applied as hi + lo.
__device__ __forceinline__ float weight(const Record& r, float lt, float ld) {
  const float et = ex2((lt - r.mt) * r.kf);
  const float pt = fmaf(et, r.ist_hi, et * r.ist_lo);
  if (r.mode == MODE_REJECT) {
    if (et == 0.f) return 0.f;
    const float delta = fmaf(ld - lt, r.kf, r.c0_hi) + r.c0_lo;
    return fmaxf(-pt * expm1f(delta * 0.69314718055994531f), 0.f);
  }
  return pt;
}

// Weights of the element group a thread owns in one "round" of a segment:
// round -1 = head (one element per thread < head), rounds 0.. = aligned
// vectors (thread t owns vector r*NT + t), round nrounds = tail.  Returns the
// number of elements written to w[] and their first element index (relative
// to the segment start) in *first.
template <int DT>
__device__ __forceinline__ int group_weights(const Record& r, const Seg& st,
                                             const unsigned char* drow_seg, bool same_align,
                                             int kind, int j, float* w, int* first) {
  using E = Elem<DT>;
  const bool two = (r.mode == MODE_REJECT);
  if (kind != 1) {  // single element
    const int e = (kind == 0) ? j : st.tail0 + j;
    *first = e;
    const float lt = E::load(st.p0, e);
    const float ld = two ? E::load(drow_seg, e) : 0.f;
    w[0] = weight(r, lt, ld);
    return 1;
  }
  const int e = st.head + j * E::VEC;
  *first = e;
  float ft[E::VEC], fd[E::VEC];
  E::unpack(ld_stream(reinterpret_cast<const uint4*>(st.p0 + size_t(e) * E::ES)), ft);
  if (two) {
    if (same_align) {
      E::unpack(ld_stream(reinterpret_cast<const uint4*>(drow_seg + size_t(e) * E::ES)), fd);
    } else {
#pragma unroll
      for (int q = 0; q < E::VEC; ++q) fd[q] = E::load(drow_seg, e + q);
    }
  }
#pragma unroll
  for (int q = 0; q < E::VEC; ++q) w[q] = weight(r, ft[q], two ? fd[q] : 0.f);
  return E::VEC;
}

template <int DT>
__device__ __forceinline__ void p2_segments(const Params& P, int b, const Record& r, int c2,
                                            Seg& st, const unsigned char*& dseg, bool& same) {
  using E = Elem<DT>;
  const int e0 = c2 * P.ch2;
  const int n = min(P.ch2, P.V - e0);
  const int rowk = (r.mode == MODE_BONUS) ? P.gamma : r.k;
  const unsigned char* trow = P.Lt + (size_t(b) * P.R + rowk) * size_t(P.V) * E::ES;
  st = make_seg<DT>(trow, e0, n);
  dseg = st.p0;
  same = true;
  if (r.mode == MODE_REJECT) {
    const unsigned char* drow = P.Ld + (size_t(b) * P.gamma + r.k) * size_t(P.V) * E::ES;
    dseg = drow + size_t(e0) * E::ES;
    same = ((reinterpret_cast<uintptr_t>(dseg) ^ reinterpret_cast<uintptr_t>(st.p0)) & 15u) == 0;
  }
}

// Mass of phase-2 chunk c2 (all threads return it).
template <int DT>
__device__ double chunk_mass(const Params& P, int b, const Record& r, int c2, SMem& sm) {
  using E = Elem<DT>;
  Seg st;
  const unsigned char* dseg;
  bool same;
  p2_segments<DT>(P, b, r, c2, st, dseg, same);
  float acc = 0.f, w[E::VEC];
  int first;
  const int tid = threadIdx.x;
  if (tid < st.head) {
    group_weights<DT>(r, st, dseg, same, 0, tid, w, &first);
    acc += w[0];
  }
  for (int j = tid; j < st.nvec; j += NT) {
    group_weights<DT>(r, st, dseg, same, 1, j, w, &first);
    float t = 0.f;
#pragma unroll
    for (int q = 0; q < E::VEC; ++q) t += w[q];
    acc += t;
  }
  if (tid < st.n - st.tail0) {
    group_weights<DT>(r, st, dseg, same, 2, tid, w, &first);
    acc += w[0];
  }
  return block_sum_d(double(acc), sm);
}

// Index (within the row) of the smallest element of chunk c2 whose running
// mass exceeds tau (tau relative to the chunk start); the last element with
// mass when rounding leaves tau at or beyond the chunk's total.
template <int DT>
__device__ int chunk_search(const Params& P, int b, const Record& r, int c2, double tau,
                            SMem& sm) {
  using E = Elem<DT>;
  Seg st;
  const unsigned char* dseg;
  bool same;
  p2_segments<DT>(P, b, r, c2, st, dseg, same);
  const int tid = threadIdx.x;
  const int nbody = (st.nvec + NT - 1) / NT;
  if (tid == 0) { sm.hit_v = -1; sm.last_v = -1; }
  __syncthreads();
  double base = 0.0;
  int last_mine = -1;
  for (int round = -1; round <= nbody; ++round) {
    const int kind = (round < 0) ? 0 : (round == nbody ? 2 : 1);
    const int j = (kind == 1) ? round * NT + tid : tid;
    const bool have = (kind == 0) ? (tid < st.head)
                                  : (kind == 2 ? (tid < st.n - st.tail0) : (j < st.nvec));
    float w[E::VEC];
    int first = 0, cnt = 0;
    float tot = 0.f;
    if (have) {
      cnt = group_weights<DT>(r, st, dseg, same, kind, j, w, &first);
      for (int q = 0; q < cnt; ++q) {
        tot += w[q];
        if (w[q] > 0.f) last_mine = first + q;
      }
    }
    const double incl = block_incl_scan(double(tot), sm);
    const double rtotal = sm.incl[NT - 1];
    if (tid == 0) sm.hit_t = NT;
    __syncthreads();
    if (cnt > 0 && base + incl > tau) atomicMin(&sm.hit_t, tid);
    __syncthreads();
    const int ht = sm.hit_t;
    if (ht < NT) {
      if (tid == ht) {
        double run = base + (tid > 0 ? sm.incl[tid - 1] : 0.0);
        int v = -1, lastpos = -1;
        for (int q = 0; q < cnt; ++q) {
          run += double(w[q]);
          if (w[q] > 0.f) lastpos = first + q;
          if (run > tau) { v = first + q; break; }
        }
        sm.hit_v = (v >= 0) ? v : lastpos;
      }
      __syncthreads();
      break;
    }
    base += rtotal;
  }
  int hit = sm.hit_v;
  if (hit < 0) {  // no crossing: the last element with mass in the chunk
    atomicMax(&sm.last_v, last_mine);
    __syncthreads();
    hit = sm.last_v;
  }
  __syncthreads();
  return (hit < 0 ? 0 : hit) + c2 * P.ch2;
}

template <int DT>
__device__ void task_p3(const Params& P, int b, SMem& sm) {
  const unsigned epoch = sm.epoch;
  if (threadIdx.x == 0) {
    sm.ok = (ld_acquire(&P.req[b].flag) == epoch);
    if (sm.ok) sm.rec = load_record(&P.rec[b]);
  }
  __syncthreads();
  Record r = sm.rec;
  if (sm.ok && r.mode != MODE_INVALID) {
    const int R = P.R;
    const float u = __ldg(P.u_res + size_t(b) * R + r.k);
    double Z = 0.0;
    int stale = 0;
    if (threadIdx.x == 0) {
      for (int c = 0; c < P.nch2; ++c) {
        if (__ldcg(&P.z2[size_t(b) * P.nch2 + c].epoch) != epoch) stale = 1;
        Z += __ldcg(&P.z2[size_t(b) * P.nch2 + c].z);
      }
      if (stale) mark_dirty(P);
      sm.rd[0] = Z;
    }
    __syncthreads();
    Z = sm.rd[0];
    __syncthreads();
    const bool degenerate = !(Z > 0.0);
    if (degenerate) {  // residual vanished: sample the target row k instead
      r.mode = MODE_TARGET;
      Z = 0.0;
      for (int c = 0; c < P.nch2; ++c) {
        const double zc = chunk_mass<DT>(P, b, r, c, sm);
        if (threadIdx.x == 0) P.z2[size_t(b) * P.nch2 + c].z = zc;
        Z += zc;
      }
      __syncthreads();
    }
    const double tau = double(u) * Z;
    int cstar = -1;
    double before = 0.0;
    if (threadIdx.x == 0) {
      double C = 0.0;
      int lastpos = 0;
      for (int c = 0; c < P.nch2; ++c) {
        const double zc = __ldcg(&P.z2[size_t(b) * P.nch2 + c].z);
        if (zc > 0.0) lastpos = c;
        if (C + zc > tau) { cstar = c; before = C; break; }
        C += zc;
      }
      if (cstar < 0) {  // rounding: take the last chunk with mass
        cstar = lastpos;
        before = 0.0;
        for (int c = 0; c < cstar; ++c) before += __ldcg(&P.z2[size_t(b) * P.nch2 + c].z);
      }
      sm.hit_t = cstar;
      sm.rd[0] = before;
    }
    __syncthreads();
    cstar = sm.hit_t;
    before = sm.rd[0];
    __syncthreads();
    const int tok = chunk_search<DT>(P, b, r, cstar, tau - before, sm);
    if (threadIdx.x == 0) {
      P.out_tokens[size_t(b) * R + r.k] = tok;
      if (P.out_Z) P.out_Z[b] = float(Z);
      if (degenerate) set_status(P, SV_ST_DEGENERATE);
    }
  }
}

template <int DT>
__device__ void task_p2(const Params& P, int b, int c2, SMem& sm) {
  const unsigned epoch = sm.epoch;
  if (threadIdx.x == 0) {
    int ok = 0;
    const unsigned* flag = &P.req[b].flag;
    if (ld_acquire(flag) == epoch) {
      ok = 1;
    } else {
      const unsigned long long t0 = globaltimer();
      unsigned ns = 64;
      for (;;) {
        if (ld_acquire(flag) == epoch) { ok = 1; break; }
        if (*reinterpret_cast<volatile int*>(&P.ctrl->abort)) break;
        if (globaltimer() - t0 > WAIT_LIMIT_NS) {
          atomicExch(&P.ctrl->abort, 1);
          set_status(P, SV_ST_TIMEOUT);
          break;
        }
        __nanosleep(ns);
        ns = ns < 2048 ? ns * 2 : ns;
      }
    }
    sm.ok = ok;
    if (ok) sm.rec = load_record(&P.rec[b]);
  }
  __syncthreads();
  const Record r = sm.rec;
  double z = 0.0;
  if (sm.ok && r.mode != MODE_INVALID) z = chunk_mass<DT>(P, b, r, c2, sm);
  if (threadIdx.x == 0) {
    ZPart* dst = P.z2 + size_t(b) * P.nch2 + c2;
    dst->z = z;
    dst->epoch = epoch;
    __threadfence();
    const unsigned cnt = arrive(&P.req[b].p2, epoch);
    if (cnt == 0u) {
      atomicExch(&P.ctrl->abort, 1);
      set_status(P, SV_ST_TIMEOUT);
    }
    sm.flag = (cnt == (unsigned)P.n2);
    if (sm.flag) __threadfence();
  }
  __syncthreads();
  if (sm.flag) task_p3<DT>(P, b, sm);
}

// --------------------------------------------------------- the kernel

// Global task order: P1 of requests 0..Lc-1, then for j = Lc..B-1 the P1
// tasks of j followed by the P2 tasks of j-Lc, then P2 of the last Lc.
__device__ __forceinline__ void decode(const Params& P, long long t, int& kind, int& b, int& sub) {
  const long long n1 = P.n1, n2 = P.n2;
  const long long Lc = n2 ? min((long long)P.lag, (long long)P.B) : (long long)P.B;
  const long long A = Lc * n1;
  if (t < A) { kind = 1; b = int(t / n1); sub = int(t - b * n1); return; }
  t -= A;
  const long long mid = (P.B - Lc) * (n1 + n2);
  if (t < mid) {
    const long long j = Lc + t / (n1 + n2);
    const long long r = t % (n1 + n2);
    if (r < n1) { kind = 1; b = int(j); sub = int(r); }
    else { kind = 2; b = int(j - Lc); sub = int(r - n1); }
    return;
  }
  t -= mid;
  kind = 2;
  b = int(P.B - Lc + t / n2);
  sub = int(t % n2);
}

template <int DT, bool GREEDY>
__global__ void __launch_bounds__(NT) sv_kernel(const Params P) {
  __shared__ SMem sm;
  if (threadIdx.x == 0) sm.epoch = __ldcg(&P.ctrl->epoch_counter) + 1u;
  for (;;) {
    if (threadIdx.x == 0) sm.task = atomicAdd(&P.ctrl->task, 1ull);
    __syncthreads();
    const long long t = (long long)sm.task;
    if (t >= P.total) break;
    int kind, b, sub;
    decode(P, t, kind, b, sub);
    if (kind == 1) task_p1<DT, GREEDY>(P, b, sub, sm);
    else if (!GREEDY) task_p2<DT>(P, b, sub, sm);
    __syncthreads();
  }
  // exit: the last CTA out checks and resets the control block
  if (threadIdx.x == 0) {
    const unsigned old = atomicAdd(&P.ctrl->exit_count, 1u);
    sm.flag = (old == gridDim.x - 1);
    if (sm.flag) {
      __threadfence();
      const unsigned long long tc = __ldcg(&P.ctrl->task);
      if (tc != (unsigned long long)P.total + gridDim.x) set_status(P, SV_ST_WORKSPACE);
    }
  }
  __syncthreads();
  if (sm.flag) {
    if (threadIdx.x == 0) {
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
  int chunk = 0, ctas = 0, lag = 0;
};
Tuning g_tune;

struct DevCache {
  bool init = false;
  int sms = 0;
  int occ[2][2] = {{0, 0}, {0, 0}};  // [dtype][greedy]
};
std::mutex g_mu;
DevCache g_dev[64];

template <int DT, bool G>
int occupancy() {
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sv_kernel<DT, G>, NT, 0) != cudaSuccess)
    return 0;
  return occ;
}

int device_info(int& sms, int& occ, int dtype, bool greedy) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DevCache& d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SV_ERR_CUDA;
    d.occ[0][0] = occupancy<SV_F32, false>();
    d.occ[0][1] = occupancy<SV_F32, true>();
    d.occ[1][0] = occupancy<SV_BF16, false>();
    d.occ[1][1] = occupancy<SV_BF16, true>();
    for (auto& a : d.occ)
      for (int v : a)
        if (v <= 0) return SV_ERR_CUDA;
    d.init = true;
  }
  sms = d.sms;
  occ = d.occ[dtype][greedy ? 1 : 0];
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

  int sms = 0, occ = 0;
  int rc = device_info(sms, occ, dtype, greedy);
  if (rc != SV_OK) return rc;
  const int per_sm = g_tune.ctas > 0 ? min(g_tune.ctas, occ) : occ;
  const long long grid_max = (long long)sms * per_sm;
  const int R = gamma + 1;
  const long long units = (long long)B * R;

  int nch1;
  int ch1;
  if (g_tune.chunk > 0) {
    ch1 = max(round_up(g_tune.chunk, 64), CH1_MIN);
  } else {
    const long long by_bytes = ((long long)V * ES + 32767) / 32768;
    const long long by_tasks = (8 * grid_max + units - 1) / units;
    const long long want = max(1ll, max(by_bytes, by_tasks));
    ch1 = max(round_up((V + want - 1) / want, 64), CH1_MIN);
  }
  nch1 = (V + ch1 - 1) / ch1;
  if (nch1 > L.nch1_max) return SV_ERR_INVALID_ARG;  // cannot happen: ch1 >= CH1_MIN

  Params P;
  P.Lt = static_cast<const unsigned char*>(Lt);
  P.Ld = static_cast<const unsigned char*>(Ld);
  P.x = x; P.u_acc = u_acc; P.u_res = u_res; P.temp = temp;
  P.B = B; P.gamma = gamma; P.V = V; P.R = R;
  P.ch1 = ch1; P.nch1 = nch1;
  P.ch2 = CH2; P.nch2 = L.nch2;
  P.n1 = (long long)R * nch1;
  P.n2 = greedy ? 0 : L.nch2;
  P.total = (long long)B * (P.n1 + P.n2);
  const long long grid = min(grid_max, P.total);
  if (g_tune.lag > 0) P.lag = g_tune.lag;
  else P.lag = int(max(1ll, (3 * grid / 2 + P.n1 + P.n2 - 1) / (P.n1 + P.n2)));
  P.out_tokens = out_tokens; P.out_n = out_n; P.out_p = out_p; P.out_Z = out_Z;
  P.status = status;
  unsigned char* w = static_cast<unsigned char*>(ws);
  P.ctrl = reinterpret_cast<Ctrl*>(w + L.ctrl);
  P.req = reinterpret_cast<ReqCtl*>(w + L.req);
  P.rec = reinterpret_cast<Record*>(w + L.rec);
  P.part = reinterpret_cast<Partial*>(w + L.part);
  P.z2 = reinterpret_cast<ZPart*>(w + L.z2);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == SV_F32) {
    if (greedy) sv_kernel<SV_F32, true><<<unsigned(grid), NT, 0, st>>>(P);
    else sv_kernel<SV_F32, false><<<unsigned(grid), NT, 0, st>>>(P);
  } else {
    if (greedy) sv_kernel<SV_BF16, true><<<unsigned(grid), NT, 0, st>>>(P);
    else sv_kernel<SV_BF16, false><<<unsigned(grid), NT, 0, st>>>(P);
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
  g_tune.chunk = chunk_elems > 0 ? chunk_elems : 0;
  g_tune.ctas = ctas_per_sm > 0 ? ctas_per_sm : 0;
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

int sv_version(void) { return 100; }

}  // extern "C"
