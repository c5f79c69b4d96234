// tree.cu -- sm_103a kernel and C ABI of token-tree verification (see
// include/svtree.h for the operation, layouts and error behaviour).
//
// The rule is the multi-draft form of the acceptance test and residual of
// 猜想解码 (Speculative Decoding) 全景, 考点2, applied along a candidate token
// tree (deferred speculative decoding page, opening section; the same
// overview page, 考点3).  With C_0 = 0, S_0 = 1, the residual after j rejected
// siblings at a node is
//     r_j = max(0, P_t - C_j P_d) / S_j,  C_{j+1} = C_j + S_j,
//     S_{j+1} = sum_v max(0, P_t - C_{j+1} P_d),
// which is max(0, r_j - P_d) normalised, so every rejection costs one pass
// over the node's two rows and one scalar.
//
// Design: one cluster of c CTAs (c <= 8) walks one request's tree.  A node's
// rows are split into 16 c contiguous segments, one per warp of the cluster;
// every pass (the rows' max and exp-sum, or the residual's mass) leaves one
// partial per warp in shared memory, and after a cluster barrier every CTA
// combines all partials through distributed shared memory in the same fixed
// order, so all CTAs take the same decisions without further exchange.  The
// final draw finds the segment holding u * Z from the segment totals, and the
// CTA owning it rescans only that segment.  Only rows on the walk are read
// (a visited node's target row, and its draft row when it has children);
// a rejection's residual pass re-reads rows that the node's first pass has
// just brought into L2.

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "specverify.h"
#include "svtree.h"

namespace cg = cooperative_groups;

namespace {

// Warps per CTA: 16 (one CTA per SM), or 8 (two per SM) where the batch
// leaves room for two CTAs per SM (the kernel is a template on the width).
constexpr int TW_MAX = 16, TW_MIN = 8;
constexpr int TMAXC = 8;          // CTAs per cluster (the portable limit)
static_assert(SV_TREE_MAX_N <= 32 * TW_MIN, "one child per thread at every node");
constexpr int TU = 4;             // 16-byte vectors per lane and row in a batch
constexpr int NS = 3;             // ring slots per warp
constexpr int CHV = 32 * TU;      // 16-byte vectors of one row in a slot
constexpr int CHB = CHV * 16;     // bytes of one row in a slot
// dynamic shared memory of a CTA of tw warps: 192 KB per SM at either width
constexpr size_t ring_bytes(int tw) { return size_t(tw) * NS * 2 * CHB; }
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;  // one second
constexpr int RB = 8;             // elements per lane loaded together in the final rescan
constexpr double LOG2E_D = 1.4426950408889634;

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
__device__ __forceinline__ float warp_max_nan(float v) {
  float r;
  asm volatile("redux.sync.max.NaN.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ uint32_t bmax_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// Packed fp32 pairs (one 64-bit register pair) for the f32x2 instructions.
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
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ void prefetch_l2(const void* p, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
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
      : "r"(smem_addr(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}
// One-dimensional bulk copy global -> this CTA's shared memory, completion
// counted on `bar`; addresses and size multiples of 16 bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes,
                                         unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Float pairs (h + l): sums with about 48 significant bits.
struct FF {
  float h, l;
};
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}
__device__ __forceinline__ FF ff_add(FF a, FF b) {
  float s, e;
  two_sum(a.h, b.h, s, e);
  const float t = a.l + b.l + e;
  FF r;
  r.h = s + t;
  r.l = t - (r.h - s);
  return r;
}
__device__ __forceinline__ FF ff_addf(FF a, float x) {  // a + x
  float s, e;
  two_sum(a.h, x, s, e);
  const float t = a.l + e;
  FF r;
  r.h = s + t;
  r.l = t - (r.h - s);
  return r;
}
__device__ __forceinline__ FF ff_neg(FF a) { return FF{-a.h, -a.l}; }
__device__ __forceinline__ bool ff_gt(FF a, FF b) {
  const FF d = ff_add(a, ff_neg(b));
  return d.h > 0.f || (d.h == 0.f && d.l > 0.f);
}
__device__ __forceinline__ FF ff_scale(FF a, float s) {  // a * s
  const float p = a.h * s;
  const float e = fmaf(a.h, s, -p) + a.l * s;
  FF r;
  two_sum(p, e, r.h, r.l);
  return r;
}
__device__ __forceinline__ FF ff_shfl_xor(FF a, int o) {
  return FF{__shfl_xor_sync(0xffffffffu, a.h, o), __shfl_xor_sync(0xffffffffu, a.l, o)};
}
__device__ __forceinline__ FF ff_shfl_up(FF a, int o) {
  return FF{__shfl_up_sync(0xffffffffu, a.h, o), __shfl_up_sync(0xffffffffu, a.l, o)};
}
__device__ __forceinline__ FF ff_shfl(FF a, int src) {
  return FF{__shfl_sync(0xffffffffu, a.h, src), __shfl_sync(0xffffffffu, a.l, src)};
}
__device__ __forceinline__ FF warp_sum(FF a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = ff_add(a, ff_shfl_xor(a, o));
  return a;
}
__device__ __forceinline__ FF warp_scan(FF a, int lane) {  // inclusive, lane order
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const FF b = ff_shfl_up(a, o);
    if (lane >= o) a = ff_add(a, b);
  }
  return a;
}
__device__ __forceinline__ double ff_d(FF a) { return double(a.h) + double(a.l); }

template <int DT>
struct TE;
template <>
struct TE<SV_F32> {
  static constexpr int ES = 4, VEC = 4, PAIRS = 2;
  __device__ static float at(const unsigned char* row, long long i) {
    return __ldg(reinterpret_cast<const float*>(row) + i);
  }
  __device__ static unsigned long long pair(const uint4& v, int q) {
    return q == 0 ? pk2(__uint_as_float(v.x), __uint_as_float(v.y))
                  : pk2(__uint_as_float(v.z), __uint_as_float(v.w));
  }
  __device__ static float vmax(const uint4& v) {  // NaN if any element is NaN
    return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                    fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
};
template <>
struct TE<SV_BF16> {
  static constexpr int ES = 2, VEC = 8, PAIRS = 4;
  __device__ static float at(const unsigned char* row, long long i) {
    return __uint_as_float(uint32_t(__ldg(reinterpret_cast<const unsigned short*>(row) + i))
                           << 16);
  }
  __device__ static unsigned long long pair(const uint4& v, int q) {
    const uint32_t w = q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
    return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  __device__ static float vmax(const uint4& v) {
    const uint32_t m = bmax_nan(bmax_nan(v.x, v.y), bmax_nan(v.z, v.w));
    return fmax_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
  }
};

struct TreeParams {
  const unsigned char* Lt;
  const unsigned char* Ld;
  const int32_t* parent;
  const int32_t* tokens;
  const float* u_acc;
  const float* u_res;
  const float* temp;
  int32_t* out_tokens;
  int32_t* out_n;
  int32_t* out_nodes;
  int32_t* status;
  int B, N, V;
  int same_align;  // Lt and Ld rows share their 16-byte alignment
};

struct Part {  // one warp's share of a pass
  float m;     // row max (statistics pass)
  float h, l;  // exp-sum relative to m, or residual mass (float pair)
  float pad;
};

// Entries of the segment arrays: the combines give lane l segments 4 l ..
// 4 l + 3 of the at most TW_MAX * TMAXC segments, and write all 4 * 32.
constexpr int SEG_SLOTS = 4 * 32;
static_assert(TW_MAX * TMAXC <= SEG_SLOTS, "every segment has an entry");

struct TreeSmem {
  int32_t parent[SV_TREE_MAX_N];
  int32_t token[SV_TREE_MAX_N];
  int32_t path_tok[SV_TREE_MAX_N];
  int32_t path_node[SV_TREE_MAX_N];
  float xl_t[SV_TREE_MAX_N];  // target / draft logit of each child's token at the current node
  float xl_d[SV_TREE_MAX_N];
  float ua[SV_TREE_MAX_N];    // accept uniform of each child of the current node
  float ur;                   // residual uniform of the current node
  Part part[2][2][TW_MAX];  // [buffer][target, draft][warp], alternating per pass
  // running mass after each segment (index order), and each segment's mass;
  // the combines write 4 entries per lane of a warp, whatever the segment count
  FF seg_incl[SEG_SLOTS];
  FF seg_tot[SEG_SLOTS];
  FF piece[TW_MAX];
  float mt, md;
  FF St, Sd, Z;
  float K;
  int accept, seg_pick, degenerate;
  int abort;                      // a ring wait gave up (the call's results are void)
  unsigned long long bar[TW_MAX][NS];  // per-warp ring slots: bytes arrived
};

// Element range of segment g of a row split into nseg contiguous segments.
__device__ __forceinline__ void seg_range(long long V, int g, int nseg, long long& a,
                                          long long& e) {
  a = V * g / nseg;
  e = V * (g + 1) / nseg;
}

// Head / body / tail split of [a, e) of a row so that the body starts on a
// 16-byte boundary.
template <int DT>
__device__ __forceinline__ void split16(const unsigned char* row, long long a, long long e,
                                        long long& head_end, long long& nvec) {
  using E = TE<DT>;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row) + uintptr_t(a) * E::ES;
  long long h = (long long)(((16 - (addr & 15)) & 15) / E::ES);
  if (h > e - a) h = e - a;
  head_end = a + h;
  nvec = (e - head_end) / E::VEC;
}

__device__ __forceinline__ void set_status(int32_t* status, int bits) {
  if (status && bits) atomicOr(status, bits);
}

// A warp's ring: NS slots of CHB bytes of the target row and CHB of the
// draft row, filled by bulk copies that lane 0 issues, each slot's arrival
// counted on its mbarrier.  Fill f (counted over the kernel) goes to slot
// f % NS and completes phase (f / NS) & 1 of its barrier.
struct Ring {
  unsigned char* base;
  unsigned long long* bar;
  unsigned seq;     // fills consumed
  unsigned issued;  // fills issued
};

// Bounded wait for a ring slot: false after one second (recording
// SV_ST_TIMEOUT and the CTA's abort flag) or once another warp gave up.
__device__ bool ring_wait(unsigned long long* bar, unsigned parity, TreeSmem& sm,
                          int32_t* status) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (;;) {
    if (mbar_try(bar, parity)) return true;
    if (*(volatile int*)&sm.abort) return false;
    if (globaltimer() - t0 > WAIT_LIMIT_NS) {
      *(volatile int*)&sm.abort = 1;
      set_status(status, SV_ST_TIMEOUT);
      return false;
    }
  }
}

// Stream nvec 16-byte vectors of a row body (and of the draft body when bd
// is not null) through the warp's ring; consume(ct, cd, nv) sees each slot's
// nv <= CHV vectors in order.
template <class F>
__device__ __forceinline__ void stream_body(Ring& R, TreeSmem& sm, int32_t* status,
                                            const unsigned char* bt, const unsigned char* bd,
                                            long long nvec, int lane, F&& consume) {
  if (*(volatile int*)&sm.abort) return;
  const long long nch = (nvec + CHV - 1) / CHV;
  const unsigned base = R.seq;
  auto issue = [&](long long k) {
    const int sl = int((base + unsigned(k)) % NS);
    const unsigned nb = unsigned(min((long long)CHV, nvec - k * CHV)) * 16u;
    unsigned char* dst = R.base + size_t(sl) * 2 * CHB;
    mbar_arrive_tx(&R.bar[sl], bd ? 2 * nb : nb);
    bulk_g2s(dst, bt + k * CHB, nb, &R.bar[sl]);
    if (bd) bulk_g2s(dst + CHB, bd + k * CHB, nb, &R.bar[sl]);
  };
  if (lane == 0)
    for (long long k = 0; k < nch && k < NS; ++k) issue(k);
  R.issued = base + unsigned(min(nch, (long long)NS));
  for (long long k = 0; k < nch; ++k) {
    const unsigned f = base + unsigned(k);
    const int sl = int(f % NS);
    if (!ring_wait(&R.bar[sl], (f / NS) & 1u, sm, status)) {
      R.seq = f;  // fills f .. issued - 1 may still be in flight
      return;
    }
    const uint4* ct = reinterpret_cast<const uint4*>(R.base + size_t(sl) * 2 * CHB);
    consume(ct, ct + CHV, int(min((long long)CHV, nvec - k * CHV)));
    __syncwarp();
    if (k + NS < nch) {
      if (lane == 0) issue(k + NS);
      R.issued = base + unsigned(k + NS + 1);
    }
  }
  R.seq = base + unsigned(nch);
}

// Statistics of one warp's segment: running max m and exp-sum s relative to
// it per lane, then the warp's (max, sum).  Each batch of TU vectors per lane
// first moves the running max (rescaling the sum once), then adds its terms
// 2^((x - m) kf), computed on packed pairs and summed in fp32, to a float
// pair.  NaN propagates through the max; an all -inf segment gives (-inf, 0).
struct MS {
  float m;
  FF s;
};
__device__ __forceinline__ void ms_rescale(MS& a, float vm, float kf) {
  const float mn = fmax_nan(a.m, vm);
  if (mn != a.m) {
    a.s = ff_scale(a.s, ex2((a.m - mn) * kf));
    a.m = mn;
  }
}
__device__ __forceinline__ void ms_add1(MS& a, float x, float kf) {
  ms_rescale(a, x, kf);
  if (a.m > -INFINITY) a.s = ff_addf(a.s, ex2((x - a.m) * kf));
}
__device__ __forceinline__ Part ms_warp(MS a, float kf) {
  const float M = warp_max_nan(a.m);
  FF s{0.f, 0.f};
  if (M > -INFINITY && M < INFINITY && a.m > -INFINITY) s = ff_scale(a.s, ex2((a.m - M) * kf));
  if (!(M == M)) s.h = M;
  s = warp_sum(s);
  return Part{M, s.h, s.l, 0.f};
}
// sum over a vector of 2^((x - m) kf), the subtraction and product on pairs
template <int DT>
__device__ __forceinline__ unsigned long long vec_exp(const uint4& v, unsigned long long mm,
                                                      unsigned long long kk,
                                                      unsigned long long acc) {
#pragma unroll
  for (int q = 0; q < TE<DT>::PAIRS; ++q) {
    float x, y;
    upk2(mul2(sub2(TE<DT>::pair(v, q), mm), kk), x, y);
    acc = add2(acc, pk2(ex2(x), ex2(y)));
  }
  return acc;
}
__device__ __forceinline__ float sum2(unsigned long long acc) {
  float x, y;
  upk2(acc, x, y);
  return x + y;
}

template <int DT>
__device__ void stats_pass(const TreeParams& P, TreeSmem& sm, Ring& R, const unsigned char* rt,
                           const unsigned char* rd, bool with_draft, long long a, long long e,
                           float kf, int lane, Part& pt, Part& pd) {
  using E = TE<DT>;
  MS st{-INFINITY, {0.f, 0.f}}, sd{-INFINITY, {0.f, 0.f}};
  const bool vec = !with_draft || P.same_align;
  long long hend = e, nvec = 0;
  if (vec) split16<DT>(rt, a, e, hend, nvec);
  if (lane == 0 && nvec > CHV * NS) {  // the body past the ring's first fills, into L2
    const long long off = (long long)CHV * NS * 16;
    prefetch_l2(rt + hend * E::ES + off, unsigned(nvec * 16 - off));
    if (with_draft) prefetch_l2(rd + hend * E::ES + off, unsigned(nvec * 16 - off));
  }
  // scalar head (or the whole segment when the rows' alignments differ)
  for (long long i = a + lane; i < hend; i += 32) {
    ms_add1(st, E::at(rt, i), kf);
    if (with_draft) ms_add1(sd, E::at(rd, i), kf);
  }
  const unsigned long long kk = pk2(kf, kf);
  stream_body(R, sm, P.status, rt + hend * E::ES, with_draft ? rd + hend * E::ES : nullptr, nvec,
              lane, [&](const uint4* ct, const uint4* cd, int nv) {
                uint4 xt[TU], xd[TU];
                float bt = -INFINITY, bd = -INFINITY;
#pragma unroll
                for (int u = 0; u < TU; ++u) {
                  if (lane + 32 * u < nv) {
                    xt[u] = ct[lane + 32 * u];
                    bt = fmax_nan(bt, E::vmax(xt[u]));
                    if (with_draft) {
                      xd[u] = cd[lane + 32 * u];
                      bd = fmax_nan(bd, E::vmax(xd[u]));
                    }
                  }
                }
                ms_rescale(st, bt, kf);
                if (st.m > -INFINITY) {
                  const unsigned long long mm = pk2(st.m, st.m);
                  unsigned long long acc = 0ull;
#pragma unroll
                  for (int u = 0; u < TU; ++u)
                    if (lane + 32 * u < nv) acc = vec_exp<DT>(xt[u], mm, kk, acc);
                  st.s = ff_addf(st.s, sum2(acc));
                }
                if (with_draft) {
                  ms_rescale(sd, bd, kf);
                  if (sd.m > -INFINITY) {
                    const unsigned long long mm = pk2(sd.m, sd.m);
                    unsigned long long acc = 0ull;
#pragma unroll
                    for (int u = 0; u < TU; ++u)
                      if (lane + 32 * u < nv) acc = vec_exp<DT>(xd[u], mm, kk, acc);
                    sd.s = ff_addf(sd.s, sum2(acc));
                  }
                }
              });
  for (long long i = hend + nvec * E::VEC + lane; i < e; i += 32) {
    ms_add1(st, E::at(rt, i), kf);
    if (with_draft) ms_add1(sd, E::at(rd, i), kf);
  }
  pt = ms_warp(st, kf);
  pd = with_draft ? ms_warp(sd, kf) : Part{-INFINITY, 0.f, 0.f, 0.f};
}

// Residual weight of one element: max(0, e_t - K e_d) with e = 2^((l - m) kf),
// or e_t alone when K == 0 (a draw from the target row).  The packed path
// below performs the same operations, so both give the same values.
__device__ __forceinline__ float weight(float lt, float ld, float mt, float md, float kf,
                                        float K) {
  const float et = ex2((lt - mt) * kf);
  if (K == 0.f) return et;
  return fmaxf(0.f, fmaf(-K, ex2((ld - md) * kf), et));
}

// Lane sum of the residual weights over [a, e) (lanes interleaved; each
// batch of vectors summed in fp32 on pairs and added to a float pair).
template <int DT>
__device__ FF mass_lane(const TreeParams& P, TreeSmem& sm, Ring& R, const unsigned char* rt,
                        const unsigned char* rd, long long a, long long e, float mt, float md,
                        float kf, float K, int lane) {
  using E = TE<DT>;
  const bool with_draft = K != 0.f;
  const bool vec = !with_draft || P.same_align;
  long long hend = e, nvec = 0;
  if (vec) split16<DT>(rt, a, e, hend, nvec);
  FF s{0.f, 0.f};
  for (long long i = a + lane; i < hend; i += 32)
    s = ff_addf(s, weight(E::at(rt, i), with_draft ? E::at(rd, i) : 0.f, mt, md, kf, K));
  const unsigned long long kk = pk2(kf, kf), mmt = pk2(mt, mt), mmd = pk2(md, md),
                           nk = pk2(-K, -K);
  stream_body(R, sm, P.status, rt + hend * E::ES, with_draft ? rd + hend * E::ES : nullptr, nvec,
              lane, [&](const uint4* ct, const uint4* cd, int nv) {
                unsigned long long acc = 0ull;
#pragma unroll
                for (int u = 0; u < TU; ++u) {
                  if (lane + 32 * u < nv) {
                    const uint4 xt = ct[lane + 32 * u];
                    if (!with_draft) {
                      acc = vec_exp<DT>(xt, mmt, kk, acc);
                    } else {
                      const uint4 xd = cd[lane + 32 * u];
#pragma unroll
                      for (int q = 0; q < E::PAIRS; ++q) {
                        float t0, t1, d0, d1;
                        upk2(mul2(sub2(E::pair(xt, q), mmt), kk), t0, t1);
                        upk2(mul2(sub2(E::pair(xd, q), mmd), kk), d0, d1);
                        // e_t - K e_d on the pair (one rounding each, as fmaf)
                        upk2(fma2(pk2(ex2(d0), ex2(d1)), nk, pk2(ex2(t0), ex2(t1))), t0, t1);
                        acc = add2(acc, pk2(fmaxf(0.f, t0), fmaxf(0.f, t1)));
                      }
                    }
                  }
                }
                s = ff_addf(s, sum2(acc));
              });
  for (long long i = hend + nvec * E::VEC + lane; i < e; i += 32)
    s = ff_addf(s, weight(E::at(rt, i), with_draft ? E::at(rd, i) : 0.f, mt, md, kf, K));
  return s;
}

// Combine of a mass pass (warp 0): the partials of all TW c segments, read
// from every CTA of the cluster in index order (lane l holds segments
// 4 l .. 4 l + 3), into the segment totals, their running sums and the total.
template <int TW>
__device__ void combine_mass(cg::cluster_group& cluster, TreeSmem& sm, int buf, int nseg,
                             int lane) {
  FF t[4], run{0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int g = 4 * lane + j;
    t[j] = FF{0.f, 0.f};
    if (g < nseg) {
      const Part* src = cluster.map_shared_rank(&sm.part[buf][0][0], g / TW);
      const Part p = src[g % TW];
      t[j] = FF{p.h, p.l};
    }
    run = ff_add(run, t[j]);
  }
  const FF incl = warp_scan(run, lane);
  FF before = ff_shfl_up(incl, 1);
  if (lane == 0) before = FF{0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    before = ff_add(before, t[j]);
    sm.seg_tot[4 * lane + j] = t[j];
    sm.seg_incl[4 * lane + j] = before;
  }
  const FF Z = ff_shfl(incl, 31);
  if (lane == 0) sm.Z = Z;
}

// The walk of one request by one cluster.  Every CTA of the cluster runs the
// same control flow: decisions are taken from values that each CTA combines
// from the same partials in the same order.
template <int DT, int TW>
__global__ void __launch_bounds__(32 * TW, TW_MAX / TW) sv_tree_walk(const TreeParams P) {
  using E = TE<DT>;
  constexpr int TTHR = 32 * TW;
  __shared__ TreeSmem sm;
  extern __shared__ __align__(128) unsigned char ring_mem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int c = int(cluster.num_blocks());
  const int q = int(cluster.block_rank());
  const int b = int(blockIdx.x) / c;
  const int tid = int(threadIdx.x), warp = tid >> 5, lane = tid & 31;
  const int N = P.N;
  const long long V = P.V;
  const int nseg = TW * c;

  if (lane == 0)
    for (int sl = 0; sl < NS; ++sl) mbar_init(&sm.bar[warp][sl], 1);
  if (tid == 0) sm.abort = 0;
  Ring R{ring_mem + size_t(warp) * NS * 2 * CHB, sm.bar[warp], 0u, 0u};

  // tree structure and its validity (every node, before any row is read)
  int bad = 0;
  for (int i = tid; i < N; i += TTHR) {
    const int p = P.parent[(long long)b * N + i];
    const int t = i ? P.tokens[(long long)b * N + i] : 0;
    sm.parent[i] = p;
    sm.token[i] = t;
    bad |= (i == 0) ? (p != -1) : (p < 0 || p >= i || t < 0 || t >= V);
  }
  const float T = P.temp[b];
  const bool bad_temp = !(T == T && T < INFINITY && T >= 0x1p-126f);
  bad = __syncthreads_or(bad);
  int32_t* otok = P.out_tokens + (long long)b * N;
  int32_t* onode = P.out_nodes ? P.out_nodes + (long long)b * N : nullptr;
  if (bad || bad_temp) {
    if (q == 0) {
      for (int i = tid; i < N; i += TTHR) {
        otok[i] = -1;
        if (onode) onode[i] = -1;
      }
      if (tid == 0) {
        P.out_n[b] = 0;
        set_status(P.status, (bad ? SV_ST_BAD_TOKEN : 0) | (bad_temp ? SV_ST_BAD_TEMP : 0));
      }
    }
    return;  // no pass ran: no peer reads this CTA's shared memory
  }
  const float kf = float(LOG2E_D / double(T));
  const size_t row_bytes = size_t(V) * E::ES;

  int n = 0, k = 0, buf = 0;
  bool invalid = false;
  float Kseg = 0.f;  // K of the residual whose segment totals are in sm.seg_*
  // scalar state of the walk (thread 0): r = max(0, P_t - C P_d) / S
  float C = 0.f, S = 1.f;
  int status_bits = 0;

  for (;;) {
    int hc = 0;
    for (int i = n + 1 + tid; i < N; i += TTHR) hc |= (sm.parent[i] == n);
    const bool has_child = __syncthreads_or(hc) != 0;
    const unsigned char* rt = P.Lt + ((long long)b * N + n) * row_bytes;
    const unsigned char* rd = has_child ? P.Ld + ((long long)b * N + n) * row_bytes : nullptr;
    // the children's logits at their tokens and uniforms, for the accept
    // tests: loaded into registers now and stored after the pass, so that no
    // warp waits for them before it starts streaming (child ci of thread tid
    // is node n + 1 + tid: N <= TTHR)
    const int ci = n + 1 + tid;
    const bool mine = ci < N && sm.parent[ci] == n;
    float cxt = 0.f, cxd = 0.f, cua = 0.f, cur = 0.f;
    if (mine) {
      cxt = E::at(rt, sm.token[ci]);
      cxd = E::at(rd, sm.token[ci]);
      cua = P.u_acc[(long long)b * N + ci];
    }
    if (tid == TTHR - 1) cur = P.u_res[(long long)b * N + n];

    // pass 1: the rows' max and exp-sum
    {
      long long a, e;
      seg_range(V, q * TW + warp, nseg, a, e);
      Part pt, pd;
      stats_pass<DT>(P, sm, R, rt, rd, has_child, a, e, kf, lane, pt, pd);
      if (lane == 0) {
        sm.part[buf][0][warp] = pt;
        sm.part[buf][1][warp] = pd;
      }
    }
    if (mine) {
      sm.xl_t[ci] = cxt;
      sm.xl_d[ci] = cxd;
      sm.ua[ci] = cua;
    }
    if (tid == TTHR - 1) sm.ur = cur;
    cluster.sync();
    // warp 0 combines the target row's partials, warp 1 the draft row's
    if (warp < (has_child ? 2 : 1)) {
      {
        const int r = warp;
        Part p[4];
        float M = -INFINITY;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int g = 4 * lane + j;
          p[j] = Part{-INFINITY, 0.f, 0.f, 0.f};
          if (g < nseg) {
            const Part* src = cluster.map_shared_rank(&sm.part[buf][r][0], g / TW);
            p[j] = src[g % TW];
          }
          M = fmax_nan(M, p[j].m);
        }
        M = warp_max_nan(M);
        const bool fin = M > -INFINITY && M < INFINITY;
        FF t[4], run{0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          t[j] = FF{0.f, 0.f};
          if (fin && p[j].m > -INFINITY) t[j] = ff_scale(FF{p[j].h, p[j].l}, ex2((p[j].m - M) * kf));
          run = ff_add(run, t[j]);
        }
        if (r == 0 && !has_child && fin) {
          // a leaf: its draw is from P_t, whose segment totals are these
          const FF incl = warp_scan(run, lane);
          FF before = ff_shfl_up(incl, 1);
          if (lane == 0) before = FF{0.f, 0.f};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            before = ff_add(before, t[j]);
            sm.seg_tot[4 * lane + j] = t[j];
            sm.seg_incl[4 * lane + j] = before;
          }
          const FF Z = ff_shfl(incl, 31);
          if (lane == 0) sm.Z = Z;
        }
        const FF tot = warp_sum(run);
        if (lane == 0) {
          if (r == 0) {
            sm.mt = M;
            sm.St = tot;
          } else {
            sm.md = M;
            sm.Sd = tot;
          }
        }
      }
    }
    buf ^= 1;
    __syncthreads();
    const float mt = sm.mt, md = has_child ? sm.md : 0.f;
    const FF St = sm.St, Sd = has_child ? sm.Sd : FF{1.f, 0.f};
    const bool ok_t = mt > -INFINITY && mt < INFINITY && St.h > 0.f && St.h < INFINITY;
    const bool ok_d = !has_child || (md > -INFINITY && md < INFINITY && Sd.h > 0.f &&
                                     Sd.h < INFINITY);
    if (!ok_t || !ok_d) {
      invalid = true;
      break;
    }
    if (tid == 0) {
      C = 0.f;
      S = 1.f;
    }
    bool seg_ready = !has_child;  // a leaf's segment totals came with pass 1
    Kseg = 0.f;
    int next = -1;
    for (int cc = n + 1; cc < N; ++cc) {
      if (sm.parent[cc] != n) continue;
      if (tid == 0) {
        // r(x) / P_d(x) with P = 2^((l - m) kf) / S_row, the same terms the
        // passes summed; where a term underflows fp32 it is taken in fp64
        const float et = ex2((sm.xl_t[cc] - mt) * kf);
        const float ed = ex2((sm.xl_d[cc] - md) * kf);
        float ratio = 1.f;
        if (et > 0.f && ed > 0.f) {
          const float pt = et / St.h, pq = ed / Sd.h;
          ratio = fminf(1.f, fmaxf(0.f, pt - C * pq) / (S * pq));
        } else {
          const double kd = double(kf);
          const double pt = exp2((double(sm.xl_t[cc]) - double(mt)) * kd) / ff_d(St);
          const double pq = exp2((double(sm.xl_d[cc]) - double(md)) * kd) / ff_d(Sd);
          if (pq > 0.0)
            ratio = float(fmin(1.0, fmax(0.0, pt - double(C) * pq) / (double(S) * pq)));
        }
        const int acc = sm.ua[cc] <= ratio;
        sm.accept = acc;
        if (!acc) {
          C += S;
          sm.K = C * (St.h / Sd.h);
        }
      }
      __syncthreads();
      if (sm.accept) {
        next = cc;
        break;
      }
      // a rejection: the mass of the next residual
      const float K = sm.K;
      {
        long long a, e;
        seg_range(V, q * TW + warp, nseg, a, e);
        const FF s = warp_sum(mass_lane<DT>(P, sm, R, rt, rd, a, e, mt, md, kf, K, lane));
        if (lane == 0) sm.part[buf][0][warp] = Part{0.f, s.h, s.l, 0.f};
      }
      cluster.sync();
      if (warp == 0) combine_mass<TW>(cluster, sm, buf, nseg, lane);
      buf ^= 1;
      __syncthreads();
      if (tid == 0) {
        const float Snew = (sm.Z.h + sm.Z.l) / St.h;
        sm.degenerate = !(Snew > 0.f);
        if (Snew > 0.f) {
          S = Snew;
        } else {  // the residual vanished: continue from P_t[n]
          C = 0.f;
          S = 1.f;
          status_bits |= SV_ST_DEGENERATE;
        }
      }
      __syncthreads();
      seg_ready = !sm.degenerate;
      Kseg = K;
    }
    if (next >= 0) {
      if (tid == 0) {
        sm.path_tok[k] = sm.token[next];
        sm.path_node[k] = next;
      }
      ++k;
      n = next;
      continue;
    }
    // the draw from the current residual (or from P_t[n])
    if (!seg_ready) {
      Kseg = 0.f;
      long long a, e;
      seg_range(V, q * TW + warp, nseg, a, e);
      const FF s = warp_sum(mass_lane<DT>(P, sm, R, rt, rd, a, e, mt, md, kf, 0.f, lane));
      if (lane == 0) sm.part[buf][0][warp] = Part{0.f, s.h, s.l, 0.f};
      cluster.sync();
      if (warp == 0) combine_mass<TW>(cluster, sm, buf, nseg, lane);
      buf ^= 1;
      __syncthreads();
    }
    // the segment holding tau = u * Z: the first with positive mass whose
    // running total exceeds tau (else the last with positive mass)
    if (warp == 0) {
      const float u = sm.ur;
      const FF Z = sm.Z;
      const float p = u * Z.h;
      FF tau;
      two_sum(p, fmaf(u, Z.h, -p) + u * Z.l, tau.h, tau.l);
      int hit = nseg, last = -1;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int g = 4 * lane + j;
        if (g < nseg && sm.seg_tot[g].h > 0.f) {
          last = g;
          if (hit == nseg && ff_gt(sm.seg_incl[g], tau)) hit = g;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        hit = min(hit, __shfl_xor_sync(0xffffffffu, hit, o));
        last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
      }
      // a valid row has positive mass, so `last` >= 0; clamp all the same
      const int g = hit < nseg ? hit : (last >= 0 ? last : 0);
      if (lane == 0) {
        sm.seg_pick = g;
        const FF prev = g > 0 ? sm.seg_incl[g - 1] : FF{0.f, 0.f};
        // past the last segment's total: aim at its last positive element
        sm.piece[0] = hit < nseg ? ff_add(tau, ff_neg(prev)) : FF{INFINITY, 0.f};
      }
    }
    __syncthreads();
    break;
  }
  const int gpick = invalid ? 0 : sm.seg_pick;
  const FF tau_seg = sm.piece[0];
  // after a ring wait gave up, wait (bounded) for this warp's copies still in
  // flight before the shared memory they target is released
  if (*(volatile int*)&sm.abort) {
    const unsigned long long t0 = globaltimer();
    for (unsigned f = R.seq; f < R.issued; ++f)
      while (!mbar_try(&R.bar[f % NS], (f / NS) & 1u) && globaltimer() - t0 < WAIT_LIMIT_NS) {
      }
  }
  // no CTA leaves while a peer may still read its partials
  cluster.sync();

  if (invalid) {
    if (q == 0) {
      for (int i = tid; i < N; i += TTHR) {
        otok[i] = -1;
        if (onode) onode[i] = -1;
      }
      if (tid == 0) {
        P.out_n[b] = 0;
        set_status(P.status, SV_ST_NONFINITE | status_bits);
      }
    }
    return;
  }
  if (q != gpick / TW) return;

  // rescan the picked segment: TW pieces, one per warp, then one warp scans
  // the piece holding the remaining tau element by element
  const unsigned char* rt = P.Lt + ((long long)b * N + n) * row_bytes;
  const unsigned char* rd = Kseg != 0.f ? P.Ld + ((long long)b * N + n) * row_bytes : nullptr;
  const float mt = sm.mt, md = Kseg != 0.f ? sm.md : 0.f;
  long long sa, se;
  seg_range(V, gpick, nseg, sa, se);
  {
    long long a, e;
    seg_range(se - sa, warp, TW, a, e);
    FF s{0.f, 0.f};
    for (long long i0 = sa + a; i0 < sa + e; i0 += 32 * RB) {
      float lt[RB], ld[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) {  // all of the batch's loads first
        const long long i = i0 + 32 * r + lane;
        lt[r] = i < sa + e ? E::at(rt, i) : -INFINITY;
        ld[r] = (rd && i < sa + e) ? E::at(rd, i) : 0.f;
      }
      float v = 0.f;
#pragma unroll
      for (int r = 0; r < RB; ++r)
        if (i0 + 32 * r + lane < sa + e) v += weight(lt[r], ld[r], mt, md, kf, Kseg);
      s = ff_addf(s, v);
    }
    const FF t = warp_sum(s);
    if (lane == 0) sm.piece[warp] = t;  // every thread read sm.piece[0] before the cluster barrier
  }
  __syncthreads();
  int drawn = 0;
  if (warp == 0) {
    const FF t = lane < TW ? sm.piece[lane] : FF{0.f, 0.f};
    const FF incl = warp_scan(t, lane);
    const bool pos = t.h > 0.f;
    const unsigned hits = __ballot_sync(0xffffffffu, pos && ff_gt(incl, tau_seg));
    const unsigned poss = __ballot_sync(0xffffffffu, pos);
    const int j = hits ? __ffs(hits) - 1 : (poss ? 31 - __clz(poss) : 0);
    FF before = ff_shfl_up(incl, 1);
    if (lane == 0) before = FF{0.f, 0.f};
    before = ff_shfl(before, j);
    const FF tau = hits ? ff_add(tau_seg, ff_neg(before)) : FF{INFINITY, 0.f};
    long long a, e;
    seg_range(se - sa, j, TW, a, e);
    FF run{0.f, 0.f};
    long long found = -1, lastpos = -1;
    for (long long i0 = sa + a; i0 < sa + e && found < 0; i0 += 32 * RB) {
      float w[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) {  // the batch's loads first, then its tiles in order
        const long long i = i0 + 32 * r + lane;
        w[r] = i < sa + e ? weight(E::at(rt, i), rd ? E::at(rd, i) : 0.f, mt, md, kf, Kseg) : 0.f;
      }
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        if (found < 0) {
          const long long t0 = i0 + 32 * r;
          const FF inc = ff_add(run, warp_scan(FF{w[r], 0.f}, lane));
          const unsigned h = __ballot_sync(0xffffffffu, w[r] > 0.f && ff_gt(inc, tau));
          const unsigned pv = __ballot_sync(0xffffffffu, w[r] > 0.f);
          if (h) found = t0 + __ffs(h) - 1;
          if (pv) lastpos = t0 + 31 - __clz(pv);
          run = ff_shfl(inc, 31);
        }
      }
    }
    drawn = int(found >= 0 ? found : (lastpos >= 0 ? lastpos : sa));
    if (lane == 0) sm.seg_pick = drawn;
  }
  __syncthreads();
  drawn = sm.seg_pick;
  // outputs: the accepted path, the drawn token, -1 after
  for (int i = tid; i < N; i += TTHR) {
    otok[i] = i < k ? sm.path_tok[i] : (i == k ? drawn : -1);
    if (onode) onode[i] = i < k ? sm.path_node[i] : -1;
  }
  if (tid == 0) {
    P.out_n[b] = k;
    set_status(P.status, status_bits);
  }
}

int g_cluster = 0;
int g_warps = 0;
std::mutex g_tree_mu;
int g_sms[64] = {};

template <int TW>
bool set_ring_smem() {
  return cudaFuncSetAttribute(sv_tree_walk<SV_F32, TW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(ring_bytes(TW))) == cudaSuccess &&
         cudaFuncSetAttribute(sv_tree_walk<SV_BF16, TW>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(ring_bytes(TW))) == cudaSuccess;
}

int sms_of_device(int& sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_tree_mu);
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        !set_ring_smem<TW_MAX>() || !set_ring_smem<TW_MIN>())
      return SV_ERR_CUDA;
    g_sms[dev] = n;
  }
  sms = g_sms[dev];
  return SV_OK;
}

}  // namespace

extern "C" int sv_tree_set_cluster(int ctas) {
  if (ctas < 0 || ctas > TMAXC) return SV_ERR_INVALID_ARG;
  g_cluster = ctas;
  return SV_OK;
}

extern "C" int sv_tree_set_warps(int warps) {
  if (warps != 0 && warps != TW_MIN && warps != TW_MAX) return SV_ERR_INVALID_ARG;
  g_warps = warps;
  return SV_OK;
}

extern "C" int sv_tree_verify(int dtype, const void* target_logits, const void* draft_logits,
                              const int32_t* parent, const int32_t* tokens,
                              const float* u_accept, const float* u_residual,
                              const float* temperature, int B, int N, int V,
                              int32_t* out_tokens, int32_t* out_num_accepted,
                              int32_t* out_nodes, int32_t* dev_status, void* stream) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (B < 0 || N < 1 || N > SV_TREE_MAX_N || V < 1) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  const int es = dtype == SV_F32 ? 4 : 2;
  if (!target_logits || !parent || !tokens || !u_residual || !temperature || !out_tokens ||
      !out_num_accepted)
    return SV_ERR_INVALID_ARG;
  if (N > 1 && (!draft_logits || !u_accept)) return SV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(target_logits) % es ||
      reinterpret_cast<uintptr_t>(draft_logits) % es)
    return SV_ERR_INVALID_ARG;
  int sms = 0;
  if (int rc = sms_of_device(sms)) return rc;
  // CTA width: two CTAs of 8 warps per SM up to a batch of 0.8 requests per
  // SM (a second CTA runs while one waits at a barrier, and small batches
  // get their rows in more segments), one of 16 above (measured crossover
  // between 112 and 128 requests on 152 SMs)
  const int tw = g_warps ? g_warps : (5 * (long long)B <= 4LL * sms ? TW_MIN : TW_MAX);
  int c = g_cluster;
  if (c == 0) {
    c = int((long long)sms * (TW_MAX / tw) / B);
    c = c < 1 ? 1 : (c > TMAXC ? TMAXC : c);
  }
  if ((long long)B * c > 0x7fffffffLL) return SV_ERR_INVALID_ARG;
  TreeParams P;
  P.Lt = static_cast<const unsigned char*>(target_logits);
  P.Ld = static_cast<const unsigned char*>(draft_logits);
  P.parent = parent;
  P.tokens = tokens;
  P.u_acc = u_accept;
  P.u_res = u_residual;
  P.temp = temperature;
  P.out_tokens = out_tokens;
  P.out_n = out_num_accepted;
  P.out_nodes = out_nodes;
  P.status = dev_status;
  P.B = B;
  P.N = N;
  P.V = V;
  P.same_align = ((reinterpret_cast<uintptr_t>(target_logits) ^
                   reinterpret_cast<uintptr_t>(draft_logits)) & 15) == 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(B) * unsigned(c));
  cfg.blockDim = dim3(unsigned(32 * tw));
  cfg.dynamicSmemBytes = ring_bytes(tw);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = unsigned(c);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t err;
  if (tw == TW_MIN)
    err = dtype == SV_F32 ? cudaLaunchKernelEx(&cfg, sv_tree_walk<SV_F32, TW_MIN>, P)
                          : cudaLaunchKernelEx(&cfg, sv_tree_walk<SV_BF16, TW_MIN>, P);
  else
    err = dtype == SV_F32 ? cudaLaunchKernelEx(&cfg, sv_tree_walk<SV_F32, TW_MAX>, P)
                          : cudaLaunchKernelEx(&cfg, sv_tree_walk<SV_BF16, TW_MAX>, P);
  return err == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
