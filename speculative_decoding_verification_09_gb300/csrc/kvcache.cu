// kvcache.cu -- sm_103a kernels and C ABI of the KV-cache steps around
// verification (see include/svkv.h for the operations, layouts and error
// behaviour):
//
//   sv_kv_commit           copy kernel (one 2-D grid: request x span of the
//                          request's staged vectors) + position update
//   sv_kv_valid_slots      one thread per (request, slot index)
//   sv_window_block_table  one thread per (request, clone column)
//
// The ring slot formula and the valid-slot order follow the deferred
// speculative decoding page, sections "环形上下文与注意力沉淀机制" and
// "C++ 环形 KV 缓存管理内核实现"; the window arithmetic follows the vllm-ascend
// draft KV sliding-window page, sections "窗口数学" and "block table 的裁剪方式".
//
// All three are memory-bound gathers and scatters of whole 16-byte vectors
// (the commit) or of int32 words (the maps); the commit moves only the
// accepted entries: rejected drafts are never written.

#include <cuda_runtime.h>
#include <stdint.h>

#include "specverify.h"
#include "svkv.h"

namespace {

constexpr int KV_THREADS = 256;
constexpr int KV_UNROLL = 4;     // 16-byte vectors in flight per thread
constexpr int KV_MAX_R = 64;     // staged entries per request
constexpr int KV_MAX_NVEC = 512; // 16-byte vectors per KV row (8 KB rows)
constexpr int MAP_THREADS = 128;

// n / d for 0 <= n < 2^31 and 1 <= d <= 512 as (n * ceil(2^40 / d)) >> 40: the
// multiplier's excess over 2^40 / d is below 1, so the product's excess over
// n * 2^40 / d stays below 2^31 / 2^40 <= 1 / d, less than the distance from
// n / d to the next integer.
unsigned long long div_magic(int d) { return ((1ull << 40) + unsigned(d) - 1) / unsigned(d); }
__device__ __forceinline__ int div_by(int n, unsigned long long m) {
  return int((unsigned long long)(unsigned)n * m >> 40);
}

__device__ __forceinline__ void allow_next_kernel() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_previous_kernel() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void set_status(int32_t* status, int bits) {
  if (status && bits) atomicOr(status, bits);
}

// Slot(pos) of a cache with `sink` persistent slots and a ring of `window`.
__device__ __host__ __forceinline__ long long ring_slot(long long pos, int sink, int window) {
  return pos < sink ? pos : sink + (pos - sink) % window;
}

struct KvParams {
  unsigned char* k_pool;
  unsigned char* v_pool;
  const unsigned char* k_new;
  const unsigned char* v_new;
  const int32_t* num_accepted;
  int32_t* pos;
  int32_t* status;
  int B, LH, R, nvec, sink, window;  // nvec: 16-byte vectors per row
  int per_req;                       // LH * R * nvec, staged vectors per request
  unsigned long long m_nvec, m_R;    // division multipliers (div_magic)
};

// Copy of the accepted entries.  Request b = blockIdx.y; the CTAs of a
// request stride over its staged vectors f = (lh * R + j) * nvec + q, which
// are contiguous in k_new / v_new; entry j <= k goes to row (b, lh) of the
// pools at slot Slot(pos + j).  KV_UNROLL vectors of K and of V per thread
// are loaded before any is stored.
__global__ void __launch_bounds__(KV_THREADS) sv_kv_copy(const KvParams K) {
  __shared__ int slot_of[KV_MAX_R];  // Slot(pos + j) of the committed entries
  allow_next_kernel();  // the position update waits for this grid's completion
  const int b = int(blockIdx.y);
  const int k = __ldg(K.num_accepted + b);
  const int p = __ldg(K.pos + b);
  if (k < 0 || k >= K.R || p < 0 || p > 0x7fffffff - K.R) return;  // dropped or invalid
  if (int(threadIdx.x) <= k)
    slot_of[threadIdx.x] = int(ring_slot((long long)p + threadIdx.x, K.sink, K.window));
  __syncthreads();
  const int C = K.sink + K.window;
  const uint4* kn = reinterpret_cast<const uint4*>(K.k_new) + size_t(b) * K.per_req;
  const uint4* vn = reinterpret_cast<const uint4*>(K.v_new) + size_t(b) * K.per_req;
  uint4* kp = reinterpret_cast<uint4*>(K.k_pool);
  uint4* vp = reinterpret_cast<uint4*>(K.v_pool);
  const int stride = int(gridDim.x) * KV_THREADS;
  for (int f0 = int(blockIdx.x) * KV_THREADS + int(threadIdx.x); f0 < K.per_req;
       f0 += stride * KV_UNROLL) {
    uint4 kv[KV_UNROLL], vv[KV_UNROLL];
    size_t dst[KV_UNROLL];
    bool use[KV_UNROLL];
#pragma unroll
    for (int u = 0; u < KV_UNROLL; ++u) {
      const int f = f0 + u * stride;
      const int row = div_by(f, K.m_nvec), q = f - row * K.nvec;
      const int lh = div_by(row, K.m_R), j = row - lh * K.R;
      use[u] = f < K.per_req && j <= k;
      dst[u] = use[u] ? ((size_t(b) * K.LH + lh) * C + size_t(slot_of[j])) * K.nvec + q : 0;
      if (use[u]) {
        kv[u] = __ldg(kn + f);
        vv[u] = __ldg(vn + f);
      }
    }
#pragma unroll
    for (int u = 0; u < KV_UNROLL; ++u) {
      if (use[u]) {
        kp[dst[u]] = kv[u];
        vp[dst[u]] = vv[u];
      }
    }
  }
}

// Position update after the copy: pos[b] += k + 1 for a committed request.
__global__ void __launch_bounds__(KV_THREADS) sv_kv_advance(const KvParams K) {
  const int b = int(blockIdx.x) * KV_THREADS + int(threadIdx.x);
  int k = 0, p = 0;
  if (b < K.B) {  // inputs of this call, read before the wait
    k = __ldg(K.num_accepted + b);
  }
  wait_previous_kernel();  // the copy kernel has read every position
  if (b >= K.B) return;
  p = K.pos[b];
  if (k >= K.R || p < 0 || p > 0x7fffffff - K.R) {  // the position would overflow
    set_status(K.status, SV_ST_BAD_LENGTH);
    return;
  }
  if (k >= 0) K.pos[b] = p + k + 1;
}

// Valid slots of request blockIdx.y, entries j = blockIdx.x * MAP_THREADS + tid.
__global__ void __launch_bounds__(MAP_THREADS) sv_kv_slots(const int32_t* pos, int sink,
                                                           int window, int32_t* out_slots,
                                                           int32_t* out_len, int32_t* status) {
  const int b = int(blockIdx.y);
  const int C = sink + window;
  const int j = int(blockIdx.x) * MAP_THREADS + int(threadIdx.x);
  const long long p = __ldg(pos + b);
  const long long n = p < 0 ? 0 : (p < C ? p : C);
  if (j < C) {
    long long slot = -1;
    if (j < n) {
      if (p <= C) slot = j;
      else if (j < sink) slot = j;
      else slot = ring_slot(p - window + (j - sink), sink, window);
    }
    out_slots[size_t(b) * C + j] = int32_t(slot);
  }
  if (j == 0) {
    out_len[b] = int32_t(n);
    if (p < 0) set_status(status, SV_ST_BAD_LENGTH);
  }
}

// The window arithmetic of one sequence length: start block and the number
// of blocks the windowed length needs; false for a negative length.
__device__ __host__ __forceinline__ bool window_of(long long s, int W, int blk, int K,
                                                  long long& start, long long& needed) {
  if (s < 0) return false;
  long long lo = s + K - W;
  if (lo < 0) lo = 0;
  start = (lo / blk) * blk;
  needed = (s - start + blk - 1) / blk;
  return true;
}

// Clone column j = blockIdx.x * MAP_THREADS + tid of request blockIdx.y.
__global__ void __launch_bounds__(MAP_THREADS) sv_window_table(
    const int32_t* seq_lens, const int32_t* table, int full_cols, int W, int blk, int K,
    int cols, int32_t* out_seq, int32_t* out_table, int32_t* out_start_block, int32_t* status) {
  const int b = int(blockIdx.y);
  const int j = int(blockIdx.x) * MAP_THREADS + int(threadIdx.x);
  const long long s = __ldg(seq_lens + b);
  long long start = 0, needed = 0;
  const bool ok = window_of(s, W, blk, K, start, needed);
  const long long sb = start / blk;
  if (j < cols) {
    int32_t v = 0;
    const long long col = sb + j;
    if (ok && j < needed && col < full_cols) v = __ldg(table + size_t(b) * full_cols + col);
    out_table[size_t(b) * cols + j] = v;
  }
  if (j == 0) {
    out_seq[b] = ok ? int32_t(s - start) : 0;
    if (out_start_block) out_start_block[b] = ok ? int32_t(sb) : 0;
    if (!ok) set_status(status, SV_ST_BAD_LENGTH);
  }
}

int window_cols(int W, int blk) {
  if (W < 1 || blk < 1) return -1;
  const long long page = (long long)W / blk + 1;
  const long long bound = ((long long)W + 2LL * blk - 2) / blk;  // ceil((W + b - 1) / b)
  const long long c = page > bound ? page : bound;
  return c > 0x7fffffffLL ? -1 : int(c);
}

bool misaligned(const void* p, unsigned a) {
  return (reinterpret_cast<uintptr_t>(p) % a) != 0;
}

}  // namespace

extern "C" {

int sv_kv_commit(void* k_pool, void* v_pool, const void* k_new, const void* v_new,
                 const int32_t* num_accepted, int32_t* pos, int B, int LH, int R, int row_bytes,
                 int sink, int window, int32_t* dev_status, void* stream) {
  if (B < 0 || LH < 1 || R < 1 || R > KV_MAX_R || row_bytes < 16 || (row_bytes % 16) != 0 ||
      row_bytes / 16 > KV_MAX_NVEC || sink < 0 || window < R ||
      (long long)sink + window > 0x7fffffffLL)
    return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!k_pool || !v_pool || !k_new || !v_new || !num_accepted || !pos) return SV_ERR_INVALID_ARG;
  if (misaligned(k_pool, 16) || misaligned(v_pool, 16) || misaligned(k_new, 16) ||
      misaligned(v_new, 16) || misaligned(num_accepted, 4) || misaligned(pos, 4) ||
      (dev_status && misaligned(dev_status, 4)))
    return SV_ERR_INVALID_ARG;
  const long long per_req = (long long)LH * R * (row_bytes / 16);
  if (per_req > (1LL << 30) || B > 65535) return SV_ERR_INVALID_ARG;  // int indexing inside
  KvParams K;
  K.k_pool = static_cast<unsigned char*>(k_pool);
  K.v_pool = static_cast<unsigned char*>(v_pool);
  K.k_new = static_cast<const unsigned char*>(k_new);
  K.v_new = static_cast<const unsigned char*>(v_new);
  K.num_accepted = num_accepted;
  K.pos = pos;
  K.status = dev_status;
  K.B = B; K.LH = LH; K.R = R; K.nvec = row_bytes / 16;
  K.sink = sink; K.window = window;
  K.per_req = int(per_req);
  K.m_nvec = div_magic(K.nvec);
  K.m_R = div_magic(R);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // CTAs per request: enough for KV_UNROLL vectors per thread per pass
  const long long per_cta = (long long)KV_THREADS * KV_UNROLL;
  const unsigned gx = unsigned((per_req + per_cta - 1) / per_cta);
  sv_kv_copy<<<dim3(gx, unsigned(B)), KV_THREADS, 0, st>>>(K);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((B + KV_THREADS - 1) / KV_THREADS));
  cfg.blockDim = dim3(KV_THREADS);
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, sv_kv_advance, K) != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

int sv_kv_valid_slots(const int32_t* pos, int B, int sink, int window, int32_t* out_slots,
                      int32_t* out_len, int32_t* dev_status, void* stream) {
  if (B < 0 || sink < 0 || window < 1 || (long long)sink + window > 0x7fffffffLL)
    return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!pos || !out_slots || !out_len || B > 65535) return SV_ERR_INVALID_ARG;
  if (misaligned(pos, 4) || misaligned(out_slots, 4) || misaligned(out_len, 4) ||
      (dev_status && misaligned(dev_status, 4)))
    return SV_ERR_INVALID_ARG;
  const int C = sink + window;
  sv_kv_slots<<<dim3(unsigned((C + MAP_THREADS - 1) / MAP_THREADS), unsigned(B)), MAP_THREADS,
                 0, static_cast<cudaStream_t>(stream)>>>(pos, sink, window, out_slots, out_len,
                                                         dev_status);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

int sv_window_cols(int window, int block_size) { return window_cols(window, block_size); }

int sv_window_block_table(const int32_t* seq_lens, const int32_t* block_table, int B,
                          int full_cols, int window, int block_size, int future_offset,
                          int32_t* out_seq_lens, int32_t* out_block_table,
                          int32_t* out_start_block, int32_t* dev_status, void* stream) {
  const int cols = window_cols(window, block_size);
  if (B < 0 || full_cols < 1 || cols < 1 || future_offset < 0) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!seq_lens || !block_table || !out_seq_lens || !out_block_table || B > 65535)
    return SV_ERR_INVALID_ARG;
  if (misaligned(seq_lens, 4) || misaligned(block_table, 4) || misaligned(out_seq_lens, 4) ||
      misaligned(out_block_table, 4) || (out_start_block && misaligned(out_start_block, 4)) ||
      (dev_status && misaligned(dev_status, 4)))
    return SV_ERR_INVALID_ARG;
  sv_window_table<<<dim3(unsigned((cols + MAP_THREADS - 1) / MAP_THREADS), unsigned(B)),
                    MAP_THREADS, 0, static_cast<cudaStream_t>(stream)>>>(
      seq_lens, block_table, full_cols, window, block_size, future_offset, cols, out_seq_lens,
      out_block_table, out_start_block, dev_status);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

int sv_window_seq_lens_host(const int32_t* seq_lens, int n, int window, int block_size,
                            int future_offset, int32_t* out) {
  if (n < 0 || window < 1 || block_size < 1 || future_offset < 0) return SV_ERR_INVALID_ARG;
  if (n > 0 && (!seq_lens || !out)) return SV_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    long long start = 0, needed = 0;
    const long long s = seq_lens[i];
    out[i] = window_of(s, window, block_size, future_offset, start, needed) ? int32_t(s - start)
                                                                            : 0;
  }
  return SV_OK;
}

}  // extern "C"
