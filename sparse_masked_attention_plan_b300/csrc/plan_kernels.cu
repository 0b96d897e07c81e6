// plan_kernels.cu -- the plan builder on the GPU.
//
// * Column flags and compaction: C = sorted(strided columns U global columns),
//   the keys every query may read ("Attention variants", sreshtalluri.github.io,
//   section 4: local_strided and with_global; ai360xpert "Sparse Attention",
//   sections on strided and global attention).  Also a 128-bit mask per key
//   block marking its columns in C, used by the forward kernels' predicate.
// * Tile classification: for every (query block, key block) tile of the 128 x 128
//   grid, the exact number of allowed pairs, from a per-row closed form (interval
//   intersection for the local rule, arithmetic-progression counts for strided
//   columns, binary search for global columns, per-block additions for BigBird's
//   random blocks), then empty / full / partial.  The
//   block-level skipping of "Attention variants", section "Use the library"
//   (create_block_mask; "never loading zero blocks") rests on this classification;
//   the per-tile counts sum to the glossary's edge count E ("Sparse attention",
//   glossary.selfmadequant.com, section "When the cost is linear").
#include <cuda_runtime.h>

#include "internal.h"

namespace spattn {
namespace {

__device__ __forceinline__ int floordiv(int n, int s) {  // s > 0
  return n >= 0 ? n / s : -((-n + s - 1) / s);
}

// #{j in [x, y] : j % stride == offset}
__device__ __forceinline__ int ap_count(const MaskDev& m, int x, int y) {
  if (m.stride <= 0 || y < x) return 0;
  return floordiv(y - m.offset, m.stride) - floordiv(x - 1 - m.offset, m.stride);
}

__device__ __forceinline__ int lower_bound(const int32_t* a, int n, int v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] < v) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// #{g in G', x <= g <= y}: global columns that are not strided columns
__device__ __forceinline__ int gns_count(const MaskDev& m, int x, int y) {
  if (m.n_gns == 0 || y < x) return 0;
  return lower_bound(m.gpos_ns, m.n_gns, y + 1) - lower_bound(m.gpos_ns, m.n_gns, x);
}

// #{j in [x, y] : j % d == r}  (0 <= r < d)
__device__ __forceinline__ int mod_count(int x, int y, int r, int d) {
  if (y < x) return 0;
  return floordiv(y - r, d) - floordiv(x - 1 - r, d);
}

// Inverse of a modulo m (gcd(a, m) == 1, m >= 1), by the extended Euclidean algorithm.
__device__ long long inv_mod(long long a, long long m) {
  long long g = m, x = 0, x1 = 1, a1 = ((a % m) + m) % m;
  while (a1 != 0) {
    const long long q = g / a1;
    long long t = g - q * a1;
    g = a1;
    a1 = t;
    t = x - q * x1;
    x = x1;
    x1 = t;
  }
  return ((x % m) + m) % m;
}

__device__ __forceinline__ long long floordiv64(long long u, long long v) {  // v > 0
  return u >= 0 ? u / v : -((-u + v - 1) / v);
}

// #{j in [x, y] : j % m1 == r1 and j % m2 == r2}, by the Chinese remainder theorem.
__device__ int crt_count(int x, int y, int r1, int m1, int r2, int m2) {
  if (y < x) return 0;
  long long a = m1, b = m2;
  while (b) {
    const long long t = a % b;
    a = b;
    b = t;
  }
  const long long g = a;
  if (((static_cast<long long>(r2) - r1) % g + g) % g != 0) return 0;
  const long long mg = m2 / g;  // solve m1 t == r2 - r1 (mod m2)
  const long long rhs = (((static_cast<long long>(r2) - r1) / g) % mg + mg) % mg;
  const long long t = mg == 1 ? 0 : (rhs * inv_mod((m1 / g) % mg, mg)) % mg;
  const long long L = static_cast<long long>(m1) / g * m2;
  const long long j0 = r1 + static_cast<long long>(m1) * t;  // the residue modulo L
  return static_cast<int>(floordiv64(y - j0, L) - floordiv64(x - 1 - j0, L));
}

// Non-strided global columns in [x, y] on the dilation grid (j % d == r).
__device__ int gns_count_grid(const MaskDev& m, int x, int y, int r, int d) {
  if (m.n_gns == 0 || y < x) return 0;
  int c = 0;
  for (int k = lower_bound(m.gpos_ns, m.n_gns, x); k < m.n_gns && m.gpos_ns[k] <= y; ++k)
    c += (m.gpos_ns[k] % d) == r;
  return c;
}

// Keys j in [a, b] allowed by the local, strided and global rules for query row i
// (closed form; a <= b inside [0, T)).  The local keys are the j of the local span
// with (i - j) % dilation == 0.
__device__ int row_count_base(const MaskDev& m, int i, int a, int b) {
  const int jmax = m.causal ? i : m.T - 1;
  if (b > jmax) b = jmax;
  if (b < a) return 0;
  if (m.rowglobal[i]) return b - a + 1;  // a global row reads every permitted key
  const int d = m.dilation;
  int lo, hi;
  if (m.causal) {
    lo = m.window ? i - (m.window - 1) * d : 0;
    hi = i;
  } else {
    lo = m.radius >= 0 ? i - m.radius * d : 0;
    hi = m.radius >= 0 ? i + m.radius * d : m.T - 1;
  }
  const int la = max(a, lo), lb = min(b, hi);
  if (d == 1) {
    const int nl = lb >= la ? lb - la + 1 : 0;
    const int ns = ap_count(m, a, b) - (nl ? ap_count(m, la, lb) : 0);
    const int ng = gns_count(m, a, b) - (nl ? gns_count(m, la, lb) : 0);
    return nl + ns + ng;
  }
  const int res = i % d;
  const int nl = mod_count(la, lb, res, d);
  const int ns = ap_count(m, a, b) -
                 (nl && m.stride > 0 ? crt_count(la, lb, m.offset, m.stride, res, d) : 0);
  const int ng = gns_count(m, a, b) - (nl ? gns_count_grid(m, la, lb, res, d) : 0);
  return nl + ns + ng;
}

// Allowed keys j in [a, b] for query row i: the rules above plus the random blocks of
// i's query block, each adding its permitted keys that no other rule allows (the
// blocks of one row are disjoint, so the additions do not overlap).
__device__ int row_count(const MaskDev& m, int i, int a, int b) {
  int c = row_count_base(m, i, a, b);
  if (m.rand_block == 0 || m.rowglobal[i]) return c;
  const int jmax = m.causal ? i : m.T - 1;
  const int q = i / m.rand_block;
  for (int x = m.r_off[q]; x < m.r_off[q + 1]; ++x) {
    const int c0 = max(a, m.r_kb[x] * m.rand_block);
    const int c1 = min(min(b, jmax), m.r_kb[x] * m.rand_block + m.rand_block - 1);
    if (c0 <= c1) c += (c1 - c0 + 1) - row_count_base(m, i, c0, c1);
  }
  return c;
}

// Does a random block of a query row in [q0, q1] reach a key in [k0, k1]?
__device__ bool rand_meets(const MaskDev& m, int q0, int q1, int k0, int k1) {
  if (m.rand_block == 0) return false;
  for (int q = q0 / m.rand_block; q <= q1 / m.rand_block; ++q)
    for (int x = m.r_off[q]; x < m.r_off[q + 1]; ++x) {
      const int c0 = m.r_kb[x] * m.rand_block;
      if (c0 <= k1 && c0 + m.rand_block - 1 >= k0) return true;
    }
  return false;
}

// Can any (i in [q0,q1], j in [k0,k1]) be allowed by the local rule?  Conservative
// (the local span only, ignoring the dilation grid): it only gates a fast skip.
__device__ __forceinline__ bool local_meets(const MaskDev& m, int q0, int q1, int k0, int k1) {
  if (m.causal) {
    if (k0 > q1) return false;
    return m.window == 0 || max(0, q0 - k1) <= (m.window - 1) * m.dilation;
  }
  if (m.radius < 0) return true;
  return max(0, max(k0 - q1, q0 - k1)) <= m.radius * m.dilation;
}

__global__ void k_strided_flags(MaskDev m, uint8_t* flags, uint8_t* rowglobal) {
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < m.T; j += gridDim.x * blockDim.x) {
    flags[j] = (m.stride > 0 && j % m.stride == m.offset) ? 1 : 0;
    rowglobal[j] = 0;
  }
}

__global__ void k_global_flags(MaskDev m, uint8_t* flags, uint8_t* rowglobal) {
  for (int a = blockIdx.x * blockDim.x + threadIdx.x; a < m.n_global; a += gridDim.x * blockDim.x) {
    flags[m.gpos[a]] = 1;
    rowglobal[m.gpos[a]] = 1;
  }
}

// One block: stream compaction of the flagged columns in ascending order.
__global__ void __launch_bounds__(1024) k_compact(const uint8_t* flags, int T, int32_t* cols,
                                                  int32_t* n_cols) {
  __shared__ int warp_sums[32];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int chunk = (T + nt - 1) / nt;
  const int b = min(T, tid * chunk), e = min(T, b + chunk);
  int cnt = 0;
  for (int j = b; j < e; ++j) cnt += flags[j];
  // block exclusive scan of cnt
  const int lane = tid & 31, wid = tid >> 5;
  int x = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = lane < (nt >> 5) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  int pos = x - cnt + (wid > 0 ? warp_sums[wid - 1] : 0);
  for (int j = b; j < e; ++j)
    if (flags[j]) cols[pos++] = j;
  if (tid == nt - 1) *n_cols = pos;
}

__global__ void k_colmask(const uint8_t* flags, int T, int nkb, uint32_t* colmask) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= nkb * 4) return;
  const int base = t * 32;
  uint32_t w = 0;
  for (int b = 0; b < 32; ++b)
    if (base + b < T && flags[base + b]) w |= 1u << b;
  colmask[t] = w;
}

// Exact allowed-pair count of tile (qb, kb).  `grow_in_qb`: the query block holds
// a global row.
__device__ int tile_count(const MaskDev& m, const uint32_t* colmask, int qb, int kb,
                          bool grow_in_qb) {
  const int q0 = qb * kTile, q1 = min(q0 + kTile, m.T) - 1;
  const int k0 = kb * kTile, k1 = min(k0 + kTile, m.T) - 1;
  if (m.causal && k0 > q1) return 0;  // every key of the tile is in the future
  if (!grow_in_qb && !local_meets(m, q0, q1, k0, k1) && !rand_meets(m, q0, q1, k0, k1)) {
    const uint32_t any = colmask[kb * 4] | colmask[kb * 4 + 1] | colmask[kb * 4 + 2] |
                         colmask[kb * 4 + 3];
    if (!any) return 0;  // no local pair, no strided or global column, no global row
  }
  int c = 0;
  for (int i = q0; i <= q1; ++i) c += row_count(m, i, k0, k1);
  return c;
}

__device__ bool block_has_global_row(const MaskDev& m, int qb) {
  __shared__ int any;
  if (threadIdx.x == 0) any = 0;
  __syncthreads();
  const int i = qb * kTile + threadIdx.x;
  if (threadIdx.x < kTile && i < m.T && m.rowglobal[i]) any = 1;
  __syncthreads();
  return any != 0;
}

__global__ void __launch_bounds__(256) k_tile_count(MaskDev m, const uint32_t* colmask, int nkb,
                                                     int32_t* q_nonempty, int32_t* q_full,
                                                     long long* q_pairs) {
  __shared__ int s_nonempty, s_full;
  __shared__ unsigned long long s_pairs;
  const int qb = blockIdx.x;
  const bool grow = block_has_global_row(m, qb);
  if (threadIdx.x == 0) { s_nonempty = 0; s_full = 0; s_pairs = 0ull; }
  __syncthreads();
  const int rows = min(kTile, m.T - qb * kTile);
  int ne = 0, fu = 0;
  unsigned long long pr = 0;
  for (int kb = threadIdx.x; kb < nkb; kb += blockDim.x) {
    const int c = tile_count(m, colmask, qb, kb, grow);
    const int cols = min(kTile, m.T - kb * kTile);
    ne += c > 0;
    fu += c == rows * cols;
    pr += static_cast<unsigned long long>(c);
  }
  atomicAdd(&s_nonempty, ne);
  atomicAdd(&s_full, fu);
  atomicAdd(&s_pairs, pr);
  __syncthreads();
  if (threadIdx.x == 0) {
    q_nonempty[qb] = s_nonempty;
    q_full[qb] = s_full;
    q_pairs[qb] = static_cast<long long>(s_pairs);
  }
}

__global__ void __launch_bounds__(256) k_tile_fill(MaskDev m, const uint32_t* colmask, int nkb,
                                                    const int32_t* q_offset, int32_t* tile_qb,
                                                    int32_t* tile_kb, int32_t* tile_cnt,
                                                    uint8_t* tile_cls) {
  __shared__ int warp_cnt[8];
  const int qb = blockIdx.x;
  const bool grow = block_has_global_row(m, qb);
  const int rows = min(kTile, m.T - qb * kTile);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int base = q_offset[qb];
  for (int kb0 = 0; kb0 < nkb; kb0 += blockDim.x) {
    const int kb = kb0 + threadIdx.x;
    const int c = kb < nkb ? tile_count(m, colmask, qb, kb, grow) : 0;
    const unsigned bal = __ballot_sync(0xffffffffu, c > 0);
    if (lane == 0) warp_cnt[wid] = __popc(bal);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < 8; ++w) {
      before += w < wid ? warp_cnt[w] : 0;
      total += warp_cnt[w];
    }
    if (c > 0) {
      const int pos = base + before + __popc(bal & ((1u << lane) - 1u));
      const int cols = min(kTile, m.T - kb * kTile);
      tile_qb[pos] = qb;
      tile_kb[pos] = kb;
      tile_cnt[pos] = c;
      tile_cls[pos] = (c == rows * cols) ? 1 : 2;
    }
    base += total;
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_column_flags(const MaskDev& m, uint8_t* flags, uint8_t* rowglobal,
                                cudaStream_t st) {
  const int blocks = min(4096, (m.T + 255) / 256);
  k_strided_flags<<<blocks, 256, 0, st>>>(m, flags, rowglobal);
  if (m.n_global > 0) k_global_flags<<<(m.n_global + 255) / 256, 256, 0, st>>>(m, flags, rowglobal);
  return cudaGetLastError();
}

cudaError_t launch_compact_columns(const uint8_t* flags, int32_t T, int32_t* cols,
                                   int32_t* n_cols, cudaStream_t st) {
  k_compact<<<1, 1024, 0, st>>>(flags, T, cols, n_cols);
  return cudaGetLastError();
}

cudaError_t launch_colmask(const uint8_t* flags, int32_t T, int32_t nkb, uint32_t* colmask,
                           cudaStream_t st) {
  k_colmask<<<(nkb * 4 + 255) / 256, 256, 0, st>>>(flags, T, nkb, colmask);
  return cudaGetLastError();
}

cudaError_t launch_tile_count(const MaskDev& m, const uint32_t* colmask, int32_t nqb,
                              int32_t nkb, int32_t* q_nonempty, int32_t* q_full,
                              long long* q_pairs, cudaStream_t st) {
  k_tile_count<<<nqb, 256, 0, st>>>(m, colmask, nkb, q_nonempty, q_full, q_pairs);
  return cudaGetLastError();
}

cudaError_t launch_tile_fill(const MaskDev& m, const uint32_t* colmask, int32_t nqb,
                             int32_t nkb, const int32_t* q_offset, int32_t* tile_qb,
                             int32_t* tile_kb, int32_t* tile_cnt, uint8_t* tile_cls,
                             cudaStream_t st) {
  k_tile_fill<<<nqb, 256, 0, st>>>(m, colmask, nkb, q_offset, tile_qb, tile_kb, tile_cnt,
                                   tile_cls);
  return cudaGetLastError();
}

}  // namespace spattn
