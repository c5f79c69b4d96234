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

constexpr int TW = 16;            // warps per CTA
constexpr int TTHR = 32 * TW;
constexpr int TMAXC = 8;          // CTAs per cluster (the portable limit)
constexpr int TU = 4;             // 16-byte vectors in flight per lane and row
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
  static constexpr int ES = 4, VEC = 4;
  __device__ static float at(const unsigned char* row, long long i) {
    return __ldg(reinterpret_cast<const float*>(row) + i);
  }
  __device__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};
template <>
struct TE<SV_BF16> {
  static constexpr int ES = 2, VEC = 8;
  __device__ static float at(const unsigned char* row, long long i) {
    return __uint_as_float(uint32_t(__ldg(reinterpret_cast<const unsigned short*>(row) + i))
                           << 16);
  }
  __device__ static void unpack(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      f[2 * q] = __uint_as_float(w[q] << 16);
      f[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
    }
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

struct TreeSmem {
  int32_t parent[SV_TREE_MAX_N];
  int32_t token[SV_TREE_MAX_N];
  int32_t path_tok[SV_TREE_MAX_N];
  int32_t path_node[SV_TREE_MAX_N];
  Part part[2][2][TW];    // [buffer][target, draft][warp], alternating per pass
  FF seg_incl[TW * TMAXC];  // running mass after each segment (index order)
  FF seg_tot[TW * TMAXC];
  FF piece[TW];
  float mt, md;
  FF St, Sd, Z;
  float K;
  int accept, seg_pick, degenerate;
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

// Statistics of one warp's segment: running max m and exp-sum s relative to
// it per lane (the sum is rescaled when the max grows; each vector's terms are
// summed in fp32 and added to a float pair), then the warp's (max, sum).  NaN
// propagates through the max; an all -inf segment gives (-inf, 0).
struct MS {
  float m;
  FF s;
};
__device__ __forceinline__ void ms_add(MS& a, float vm, const float* f, int n, float kf) {
  const float mn = fmax_nan(a.m, vm);
  if (mn != a.m) {
    a.s = ff_scale(a.s, ex2((a.m - mn) * kf));
    a.m = mn;
  }
  if (a.m > -INFINITY) {
    float v = 0.f;
    for (int i = 0; i < n; ++i) v += ex2((f[i] - a.m) * kf);
    a.s = ff_addf(a.s, v);
  }
}
__device__ __forceinline__ Part ms_warp(MS a, float kf) {
  const float M = warp_max_nan(a.m);
  FF s{0.f, 0.f};
  if (M > -INFINITY && M < INFINITY && a.m > -INFINITY) s = ff_scale(a.s, ex2((a.m - M) * kf));
  if (!(M == M)) s.h = M;
  s = warp_sum(s);
  return Part{M, s.h, s.l, 0.f};
}

template <int DT>
__device__ void stats_pass(const TreeParams& P, const unsigned char* rt, const unsigned char* rd,
                           bool with_draft, long long a, long long e, float kf, int lane,
                           Part& pt, Part& pd) {
  using E = TE<DT>;
  MS st{-INFINITY, {0.f, 0.f}}, sd{-INFINITY, {0.f, 0.f}};
  const bool vec = !with_draft || P.same_align;
  long long hend = e, nvec = 0;
  if (vec) split16<DT>(rt, a, e, hend, nvec);
  // scalar head (or the whole segment when the rows' alignments differ)
  for (long long i = a + lane; i < hend; i += 32) {
    float f = E::at(rt, i);
    ms_add(st, f, &f, 1, kf);
    if (with_draft) {
      float d = E::at(rd, i);
      ms_add(sd, d, &d, 1, kf);
    }
  }
  const uint4* vt = reinterpret_cast<const uint4*>(rt + hend * E::ES);
  const uint4* vd = reinterpret_cast<const uint4*>(rd + hend * E::ES);
  for (long long j0 = 0; j0 < nvec; j0 += 32 * TU) {
    uint4 xt[TU], xd[TU];
#pragma unroll
    for (int u = 0; u < TU; ++u) {
      const long long j = j0 + lane + 32 * u;
      if (j < nvec) {
        xt[u] = __ldg(vt + j);
        if (with_draft) xd[u] = __ldg(vd + j);
      }
    }
#pragma unroll
    for (int u = 0; u < TU; ++u) {
      if (j0 + lane + 32 * u < nvec) {
        float f[E::VEC];
        E::unpack(xt[u], f);
        float vm = f[0];
#pragma unroll
        for (int i = 1; i < E::VEC; ++i) vm = fmax_nan(vm, f[i]);
        ms_add(st, vm, f, E::VEC, kf);
        if (with_draft) {
          E::unpack(xd[u], f);
          vm = f[0];
#pragma unroll
          for (int i = 1; i < E::VEC; ++i) vm = fmax_nan(vm, f[i]);
          ms_add(sd, vm, f, E::VEC, kf);
        }
      }
    }
  }
  for (long long i = hend + nvec * E::VEC + lane; i < e; i += 32) {
    float f = E::at(rt, i);
    ms_add(st, f, &f, 1, kf);
    if (with_draft) {
      float d = E::at(rd, i);
      ms_add(sd, d, &d, 1, kf);
    }
  }
  pt = ms_warp(st, kf);
  pd = with_draft ? ms_warp(sd, kf) : Part{-INFINITY, 0.f, 0.f, 0.f};
}

// Residual weight of one element: max(0, e_t - K e_d) with e = 2^((l - m) kf),
// or e_t alone when K == 0 (a draw from the target row).
__device__ __forceinline__ float weight(float lt, float ld, float mt, float md, float kf,
                                        float K) {
  const float et = ex2((lt - mt) * kf);
  if (K == 0.f) return et;
  return fmaxf(0.f, fmaf(-K, ex2((ld - md) * kf), et));
}

// Lane sum of the residual weights over [a, e) (lanes interleaved; each
// vector's weights summed in fp32 and added to a float pair).
template <int DT>
__device__ FF mass_lane(const TreeParams& P, const unsigned char* rt, const unsigned char* rd,
                        long long a, long long e, float mt, float md, float kf, float K,
                        int lane) {
  using E = TE<DT>;
  const bool with_draft = K != 0.f;
  const bool vec = !with_draft || P.same_align;
  long long hend = e, nvec = 0;
  if (vec) split16<DT>(rt, a, e, hend, nvec);
  FF s{0.f, 0.f};
  for (long long i = a + lane; i < hend; i += 32)
    s = ff_addf(s, weight(E::at(rt, i), with_draft ? E::at(rd, i) : 0.f, mt, md, kf, K));
  const uint4* vt = reinterpret_cast<const uint4*>(rt + hend * E::ES);
  const uint4* vd = reinterpret_cast<const uint4*>(rd + hend * E::ES);
  for (long long j0 = 0; j0 < nvec; j0 += 32 * TU) {
    uint4 xt[TU], xd[TU];
#pragma unroll
    for (int u = 0; u < TU; ++u) {
      const long long j = j0 + lane + 32 * u;
      if (j < nvec) {
        xt[u] = __ldg(vt + j);
        if (with_draft) xd[u] = __ldg(vd + j);
      }
    }
#pragma unroll
    for (int u = 0; u < TU; ++u) {
      if (j0 + lane + 32 * u < nvec) {
        float f[E::VEC], d[E::VEC];
        E::unpack(xt[u], f);
        if (with_draft) {
          E::unpack(xd[u], d);
        } else {
#pragma unroll
          for (int i = 0; i < E::VEC; ++i) d[i] = 0.f;
        }
        float v = 0.f;
#pragma unroll
        for (int i = 0; i < E::VEC; ++i) v += weight(f[i], d[i], mt, md, kf, K);
        s = ff_addf(s, v);
      }
    }
  }
  for (long long i = hend + nvec * E::VEC + lane; i < e; i += 32)
    s = ff_addf(s, weight(E::at(rt, i), with_draft ? E::at(rd, i) : 0.f, mt, md, kf, K));
  return s;
}

__device__ __forceinline__ void set_status(const TreeParams& P, int bits) {
  if (P.status && bits) atomicOr(P.status, bits);
}

// The walk of one request by one cluster.  Every CTA of the cluster runs the
// same control flow: decisions are taken from values that each CTA combines
// from the same partials in the same order.
template <int DT>
__global__ void __launch_bounds__(TTHR, 1) sv_tree_walk(const TreeParams P) {
  using E = TE<DT>;
  __shared__ TreeSmem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int c = int(cluster.num_blocks());
  const int q = int(cluster.block_rank());
  const int b = int(blockIdx.x) / c;
  const int tid = int(threadIdx.x), warp = tid >> 5, lane = tid & 31;
  const int N = P.N;
  const long long V = P.V;
  const int nseg = TW * c;

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
        set_status(P, (bad ? SV_ST_BAD_TOKEN : 0) | (bad_temp ? SV_ST_BAD_TEMP : 0));
      }
    }
    return;  // no pass ran: no peer reads this CTA's shared memory
  }
  const float kf = float(LOG2E_D / double(T));
  const double kd = double(kf);
  const size_t row_bytes = size_t(V) * E::ES;

  int n = 0, k = 0, buf = 0;
  bool invalid = false;
  int drawn = -1;
  int owner = -1;       // rank of the CTA that rescans the drawn segment
  FF tau_seg{0.f, 0.f};  // u * Z less the mass before that segment
  int gpick = 0;
  float Kdraw = 0.f;
  // scalar state of the walk, thread 0 only
  double C = 0.0, S = 1.0;
  int status_bits = 0;

  for (;;) {
    int hc = 0;
    for (int i = n + 1 + tid; i < N; i += TTHR) hc |= (sm.parent[i] == n);
    const bool has_child = __syncthreads_or(hc) != 0;
    const unsigned char* rt = P.Lt + ((long long)b * N + n) * row_bytes;
    const unsigned char* rd = has_child ? P.Ld + ((long long)b * N + n) * row_bytes : nullptr;

    // pass 1: the rows' max and exp-sum
    {
      long long a, e;
      seg_range(V, q * TW + warp, nseg, a, e);
      Part pt, pd;
      stats_pass<DT>(P, rt, rd, has_child, a, e, kf, lane, pt, pd);
      if (lane == 0) {
        sm.part[buf][0][warp] = pt;
        sm.part[buf][1][warp] = pd;
      }
    }
    cluster.sync();
    if (warp == 0) {
      for (int r = 0; r < (has_child ? 2 : 1); ++r) {
        Part p[4];
        float M = -INFINITY;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int g = lane + 32 * j;
          p[j] = Part{-INFINITY, 0.f, 0.f, 0.f};
          if (g < nseg) {
            const Part* src = cluster.map_shared_rank(&sm.part[buf][r][0], g / TW);
            p[j] = src[g % TW];
          }
          M = fmax_nan(M, p[j].m);
        }
        M = warp_max_nan(M);
        FF s{0.f, 0.f};
        if (M > -INFINITY && M < INFINITY) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (p[j].m > -INFINITY) s = ff_add(s, ff_scale(FF{p[j].h, p[j].l}, ex2((p[j].m - M) * kf)));
        }
        s = warp_sum(s);
        if (lane == 0) {
          if (r == 0) {
            sm.mt = M;
            sm.St = s;
          } else {
            sm.md = M;
            sm.Sd = s;
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
      C = 0.0;
      S = 1.0;
    }
    bool mass_current = false;  // the last mass pass matches the current residual
    int next = -1;
    for (int cc = n + 1; cc < N; ++cc) {
      if (sm.parent[cc] != n) continue;
      if (tid == 0) {
        const int x = sm.token[cc];
        const double pt = exp2((double(E::at(rt, x)) - double(mt)) * kd) / ff_d(St);
        const double pq = exp2((double(E::at(rd, x)) - double(md)) * kd) / ff_d(Sd);
        double ratio = 1.0;
        if (pq > 0.0) ratio = fmin(1.0, fmax(0.0, pt - C * pq) / (S * pq));
        const int acc = double(P.u_acc[(long long)b * N + cc]) <= ratio;
        sm.accept = acc;
        if (!acc) {
          C += S;
          sm.K = float(C * ff_d(St) / ff_d(Sd));
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
        const FF s = warp_sum(mass_lane<DT>(P, rt, rd, a, e, mt, md, kf, K, lane));
        if (lane == 0) sm.part[buf][0][warp] = Part{0.f, s.h, s.l, 0.f};
      }
      cluster.sync();
      if (warp == 0) {
        // segment totals in index order: lane holds segments 4 lane .. 4 lane + 3
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
          const int g = 4 * lane + j;
          before = ff_add(before, t[j]);
          if (g < TW * TMAXC) {
            sm.seg_tot[g] = t[j];
            sm.seg_incl[g] = before;
          }
        }
        const FF Z = ff_shfl(incl, 31);
        if (lane == 0) sm.Z = Z;
      }
      buf ^= 1;
      __syncthreads();
      if (tid == 0) {
        const double Snew = ff_d(sm.Z) / ff_d(St);
        sm.degenerate = !(Snew > 0.0);
        if (Snew > 0.0) {
          S = Snew;
        } else {  // the residual vanished: continue from P_t[n]
          C = 0.0;
          S = 1.0;
          status_bits |= SV_ST_DEGENERATE;
        }
      }
      __syncthreads();
      mass_current = !sm.degenerate;
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
    Kdraw = mass_current ? sm.K : 0.f;
    if (!mass_current) {
      long long a, e;
      seg_range(V, q * TW + warp, nseg, a, e);
      const FF s = warp_sum(mass_lane<DT>(P, rt, rd, a, e, mt, md, kf, 0.f, lane));
      if (lane == 0) sm.part[buf][0][warp] = Part{0.f, s.h, s.l, 0.f};
      cluster.sync();
      if (warp == 0) {
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
          const int g = 4 * lane + j;
          before = ff_add(before, t[j]);
          if (g < TW * TMAXC) {
            sm.seg_tot[g] = t[j];
            sm.seg_incl[g] = before;
          }
        }
        const FF Z = ff_shfl(incl, 31);
        if (lane == 0) sm.Z = Z;
      }
      buf ^= 1;
      __syncthreads();
    }
    // the segment holding tau = u * Z: the first with positive mass whose
    // running total exceeds tau (else the last with positive mass)
    if (warp == 0) {
      const float u = P.u_res[(long long)b * N + n];
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
    gpick = sm.seg_pick;
    tau_seg = sm.piece[0];
    owner = gpick / TW;
    break;
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
        set_status(P, SV_ST_NONFINITE | status_bits);
      }
    }
    return;
  }
  if (q != owner) return;

  // rescan the picked segment: 16 pieces, one per warp, then one warp scans
  // the piece holding the remaining tau element by element
  const unsigned char* rt = P.Lt + ((long long)b * N + n) * row_bytes;
  const unsigned char* rd = P.Ld ? P.Ld + ((long long)b * N + n) * row_bytes : nullptr;
  const float mt = sm.mt, md = Kdraw != 0.f ? sm.md : 0.f;
  long long sa, se;
  seg_range(V, gpick, nseg, sa, se);
  {
    long long a, e;
    seg_range(se - sa, warp, TW, a, e);
    FF s{0.f, 0.f};
    for (long long i = sa + a + lane; i < sa + e; i += 32)
      s = ff_addf(s, weight(E::at(rt, i), Kdraw != 0.f ? E::at(rd, i) : 0.f, mt, md, kf, Kdraw));
    const FF t = warp_sum(s);
    __syncthreads();  // sm.piece[0] was read by every thread above
    if (lane == 0) sm.piece[warp] = t;
  }
  __syncthreads();
  if (warp == 0) {
    FF t = lane < TW ? sm.piece[lane] : FF{0.f, 0.f};
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
    for (long long i0 = sa + a; i0 < sa + e && found < 0; i0 += 32) {
      const long long i = i0 + lane;
      const float w = i < sa + e ? weight(E::at(rt, i), Kdraw != 0.f ? E::at(rd, i) : 0.f, mt, md,
                                          kf, Kdraw)
                                 : 0.f;
      const FF inc = ff_add(run, warp_scan(FF{w, 0.f}, lane));
      const unsigned h = __ballot_sync(0xffffffffu, w > 0.f && ff_gt(inc, tau));
      const unsigned pv = __ballot_sync(0xffffffffu, w > 0.f);
      if (h) found = i0 + __ffs(h) - 1;
      if (pv) lastpos = i0 + 31 - __clz(pv);
      run = ff_shfl(inc, 31);
    }
    drawn = int(found >= 0 ? found : (lastpos >= 0 ? lastpos : sa));
  }
  // outputs: the accepted path, the drawn token, -1 after
  if (warp == 0) drawn = __shfl_sync(0xffffffffu, drawn, 0);
  __syncthreads();
  if (warp == 0 && lane == 0) sm.seg_pick = drawn;
  __syncthreads();
  drawn = sm.seg_pick;
  for (int i = tid; i < N; i += TTHR) {
    otok[i] = i < k ? sm.path_tok[i] : (i == k ? drawn : -1);
    if (onode) onode[i] = i < k ? sm.path_node[i] : -1;
  }
  if (tid == 0) {
    P.out_n[b] = k;
    set_status(P, status_bits);
  }
}

int g_cluster = 0;
std::mutex g_tree_mu;
int g_sms[64] = {};

int sms_of_device(int& sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_tree_mu);
  if (!g_sms[dev] &&
      cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SV_ERR_CUDA;
  sms = g_sms[dev];
  return SV_OK;
}

}  // namespace

extern "C" int sv_tree_set_cluster(int ctas) {
  if (ctas < 0 || ctas > TMAXC) return SV_ERR_INVALID_ARG;
  g_cluster = ctas;
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
  int c = g_cluster;
  if (c == 0) {
    c = sms / B;
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
  cfg.blockDim = dim3(TTHR);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = unsigned(c);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t err = dtype == SV_F32 ? cudaLaunchKernelEx(&cfg, sv_tree_walk<SV_F32>, P)
                                          : cudaLaunchKernelEx(&cfg, sv_tree_walk<SV_BF16>, P);
  return err == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
