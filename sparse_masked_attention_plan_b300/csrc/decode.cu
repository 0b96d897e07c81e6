// decode.cu -- one generation step of sliding-window attention against a capped
// ring-buffer KV cache.
//
// The token at position t reads positions max(0, t-w+1) .. t, the w most recent
// tokens including itself ("Sparse and sliding-window attention", section "Sliding
// window attention"), so the cache keeps only the last cap >= w tokens and never
// grows ("Attention variants", section 1, the sliding-window KV cache): position p
// lives in slot p % cap.  Query heads are grouped over key/value heads (GQA: query
// head h reads key/value head h / G, G = Hq / Hkv), which is how the pages size the
// cache (per key/value head).
//
// The step is HBM-bound: every cached key and value row is read once per step and
// used by the G query heads of its group.  The slot range [0, cap) of each (batch,
// key/value head) is split across CTAs; a CTA streams 64-slot sub-chunks of K and V
// into shared memory with bulk asynchronous copies (two stages, an mbarrier per
// stage), runs an online softmax over them for the G query heads, and leaves (max,
// sum, unnormalised output) per head; a second kernel merges the splits.  The valid
// slots of a step are one circular interval of slot space (up to two linear ones), so
// a CTA copies only valid rows and needs no per-element mask.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace spattn {
namespace {

constexpr int kThreads = 256;
constexpr int kSub = 64;      // slots per sub-chunk
constexpr int kMaxGroup = 8;  // query heads per key/value head
constexpr uint64_t kWaitBudget = 8000000000ull;

template <typename In, int D>
struct DecCfg {
  static constexpr int kRowBytes = D * sizeof(In);
  static constexpr int kStageBytes = kSub * kRowBytes;  // K or V of one sub-chunk
  static constexpr int kVecPerRow = kRowBytes / 16;     // uint4 per row
  static constexpr int kVecPerLane = kVecPerRow / 8;    // 8 lanes per row
  static constexpr int kElemsPerVec = 16 / sizeof(In);
  // shared layout: K[2], V[2] stages | q [8][D] | s [8][kSub] | m, l, corr [8] | red | bars
  static constexpr int kOffQ = 4 * kStageBytes;
  static constexpr int kOffS = kOffQ + kMaxGroup * D * 4;
  static constexpr int kOffStats = kOffS + kMaxGroup * kSub * 4;
  static constexpr int kOffRed = kOffStats + 3 * kMaxGroup * 4;
  static constexpr int kOffBar = kOffRed + kThreads * 4 * 4;
  static constexpr int kSmemBytes = kOffBar + 16;
};

__device__ __forceinline__ void to_float(const uint4& v, float* out, const float*) {
  const float* f = reinterpret_cast<const float*>(&v);
  out[0] = f[0];
  out[1] = f[1];
  out[2] = f[2];
  out[3] = f[3];
}
__device__ __forceinline__ void to_float(const uint4& v, float* out, const __nv_bfloat16*) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __bfloat1622float2(h[k]);
    out[2 * k] = f.x;
    out[2 * k + 1] = f.y;
  }
}
__device__ __forceinline__ float2 ld2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 ld2(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ float ld1(const float* p) { return *p; }
__device__ __forceinline__ float ld1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st1(float* p, float v) { *p = v; }
__device__ __forceinline__ void st1(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

struct DecParams {
  const void* q;    // [B][Hq][D]
  const void* Kc;   // [B][Hkv][cap][D]
  const void* Vc;
  const int64_t* pos;  // [B]
  void* out;        // [B][Hq][D]
  float* lse;       // [B][Hq] or null
  float* part;      // [B*Hq][nsplit][D + 2]: unnormalised output, max, sum
  int* err;
  int32_t B, Hq, Hkv, G, nsplit;
  int64_t cap, window, span;
  float scale;
};

// The valid slots of the step intersected with [lo, hi): up to two intervals.
struct Ranges {
  int64_t a[2], b[2];
  int n;
};

__device__ __forceinline__ Ranges valid_ranges(int64_t t, int64_t cap, int64_t w, int64_t lo,
                                               int64_t hi) {
  Ranges r;
  r.n = 0;
  if (t < 0) return r;
  const int64_t n = min(w, t + 1);
  const int64_t start = (t - n + 1) % cap;
  int64_t ia[2], ib[2], ni = 1;
  ia[0] = start;
  ib[0] = min(cap, start + n);
  if (start + n > cap) {
    ia[1] = 0;
    ib[1] = start + n - cap;
    ni = 2;
  }
  for (int k = 0; k < ni; ++k) {
    const int64_t a = max(ia[k], lo), b = min(ib[k], hi);
    if (a < b) {
      r.a[r.n] = a;
      r.b[r.n] = b;
      ++r.n;
    }
  }
  return r;
}

// Sub-chunk `o` of the ranges: first slot and row count.
__device__ __forceinline__ void sub_chunk(const Ranges& r, int o, int64_t& s0, int& rows) {
  const int64_t n0 = (r.b[0] - r.a[0] + kSub - 1) / kSub;
  const int k = o < n0 ? 0 : 1;
  const int64_t oo = o < n0 ? o : o - n0;
  s0 = r.a[k] + oo * kSub;
  rows = static_cast<int>(min(static_cast<int64_t>(kSub), r.b[k] - s0));
}

template <typename In, int D>
__global__ void __launch_bounds__(kThreads) decode_kernel(const DecParams p) {
  using Cfg = DecCfg<In, D>;
  extern __shared__ __align__(128) uint8_t smem[];
  In* sK = reinterpret_cast<In*>(smem);                       // [2][kSub][D]
  In* sV = reinterpret_cast<In*>(smem + 2 * Cfg::kStageBytes);  // [2][kSub][D]
  float* sq = reinterpret_cast<float*>(smem + Cfg::kOffQ);    // [8][D]
  float* ss = reinterpret_cast<float*>(smem + Cfg::kOffS);    // [8][kSub]
  float* sm_ = reinterpret_cast<float*>(smem + Cfg::kOffStats);
  float* sl = sm_ + kMaxGroup;
  float* scorr = sl + kMaxGroup;
  float* sred = reinterpret_cast<float*>(smem + Cfg::kOffRed);
  const uint32_t bar0 = smem_addr(smem + Cfg::kOffBar);

  const int split = blockIdx.x % p.nsplit;
  const int bk = blockIdx.x / p.nsplit;  // b * Hkv + kv head
  const int b = bk / p.Hkv, hk = bk % p.Hkv;
  const int G = p.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t t = p.pos[b];
  const int64_t lo = static_cast<int64_t>(split) * p.span;
  const Ranges rg = valid_ranges(t, p.cap, p.window, lo, min(p.cap, lo + p.span));
  int n_sub = 0;
  for (int k = 0; k < rg.n; ++k) n_sub += static_cast<int>((rg.b[k] - rg.a[k] + kSub - 1) / kSub);
  const In* Kbase = static_cast<const In*>(p.Kc) + static_cast<int64_t>(bk) * p.cap * D;
  const In* Vbase = static_cast<const In*>(p.Vc) + static_cast<int64_t>(bk) * p.cap * D;

  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    fence_barrier_init();
  }
  // the G query rows of this group, fp32
  const In* qb = static_cast<const In*>(p.q) + (static_cast<int64_t>(b) * p.Hq + hk * G) * D;
  for (int x = tid; x < G * D; x += kThreads) sq[x] = ld1(qb + x);
  if (tid < kMaxGroup) {
    sm_[tid] = -INFINITY;
    sl[tid] = 0.f;
  }
  __syncthreads();

  auto issue = [&](int o) {
    int64_t s0;
    int rows;
    sub_chunk(rg, o, s0, rows);
    const uint32_t bytes = static_cast<uint32_t>(rows) * Cfg::kRowBytes;
    const uint32_t bar = bar0 + 8 * (o & 1);
    mbar_arrive_expect_tx(bar, 2 * bytes);
    bulk_load(smem_addr(sK + (o & 1) * kSub * D), Kbase + s0 * D, bytes, bar);
    bulk_load(smem_addr(sV + (o & 1) * kSub * D), Vbase + s0 * D, bytes, bar);
  };
  int issued = 0;
  if (tid == 0) {
    for (; issued < 2 && issued < n_sub; ++issued) issue(issued);
  }

  // PV mapping: pairs of output columns (g, 2c .. 2c+1); with fewer pairs than
  // threads the keys of a sub-chunk are split over `ks` groups of threads.
  const int npairs = G * D / 2;
  const int nact = min(npairs, kThreads);
  const int ks = kThreads / nact;
  const int kg = tid / nact, pi0 = tid % nact;
  const int ppt = (npairs + kThreads - 1) / kThreads;  // 1 or 2
  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};

  for (int o = 0; o < n_sub; ++o) {
    const int st = o & 1;
    bool ok = mbar_wait(bar0 + 8 * st, (o >> 1) & 1, kWaitBudget, p.err, kErrTimeout);
    ok = __syncthreads_and(ok);
    if (!ok) {
      // drain this CTA's copies still in flight (bounded), then leave
      if (tid == 0)
        for (int x = o; x < issued; ++x)
          mbar_wait(bar0 + 8 * (x & 1), (x >> 1) & 1, kWaitBudget, p.err, kErrTimeout);
      __syncthreads();
      return;
    }
    int64_t s0;
    int rows;
    sub_chunk(rg, o, s0, rows);
    const In* K = sK + st * kSub * D;
    const In* V = sV + st * kSub * D;
    // scores: 8 lanes per row, 4 rows per warp, 32 rows per pass
    {
      const int gi = lane >> 3, li = lane & 7;
#pragma unroll
      for (int pass = 0; pass < kSub / 32; ++pass) {
        const int r = pass * 32 + warp * 4 + gi;
        float kv[Cfg::kVecPerLane * Cfg::kElemsPerVec];
#pragma unroll
        for (int u = 0; u < Cfg::kVecPerLane; ++u) {
          const uint4 v = reinterpret_cast<const uint4*>(K + r * D)[li + 8 * u];
          to_float(v, kv + u * Cfg::kElemsPerVec, static_cast<const In*>(nullptr));
        }
        for (int g = 0; g < G; ++g) {
          float dot = 0.f;
#pragma unroll
          for (int u = 0; u < Cfg::kVecPerLane; ++u)
#pragma unroll
            for (int e = 0; e < Cfg::kElemsPerVec; ++e)
              dot = fmaf(sq[g * D + (li + 8 * u) * Cfg::kElemsPerVec + e],
                         kv[u * Cfg::kElemsPerVec + e], dot);
          dot += __shfl_xor_sync(0xffffffffu, dot, 1);
          dot += __shfl_xor_sync(0xffffffffu, dot, 2);
          dot += __shfl_xor_sync(0xffffffffu, dot, 4);
          if (li == 0) ss[g * kSub + r] = r < rows ? dot * p.scale : -INFINITY;
        }
      }
    }
    __syncthreads();
    // online softmax statistics: warp g owns query head g
    if (warp < G) {
      const float s_a = ss[warp * kSub + lane], s_b = ss[warp * kSub + lane + 32];
      float mx = fmaxf(s_a, s_b);
#pragma unroll
      for (int k = 16; k > 0; k >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, k));
      const float m_old = sm_[warp];
      const float m_new = fmaxf(m_old, mx);  // finite: row 0 of a sub-chunk is valid
      const float pa = expf(s_a - m_new), pb = expf(s_b - m_new);
      float sum = pa + pb;
#pragma unroll
      for (int k = 16; k > 0; k >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, k);
      ss[warp * kSub + lane] = pa;
      ss[warp * kSub + lane + 32] = pb;
      __syncwarp();
      if (lane == 0) {
        const float corr = expf(m_old - m_new);  // 0 on the first sub-chunk
        scorr[warp] = corr;
        sl[warp] = sl[warp] * corr + sum;
        sm_[warp] = m_new;
      }
    }
    __syncthreads();
    // weighted values
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (k >= ppt) break;
      const int pi = pi0 + k * kThreads;
      if (pi >= npairs) break;
      const int g = pi / (D / 2), c = 2 * (pi % (D / 2));
      const float corr = scorr[g];
      float a0 = acc[k][0] * corr, a1 = acc[k][1] * corr;
      for (int j = kg; j < rows; j += ks) {
        const float pj = ss[g * kSub + j];
        const float2 v = ld2(V + j * D + c);
        a0 = fmaf(pj, v.x, a0);
        a1 = fmaf(pj, v.y, a1);
      }
      acc[k][0] = a0;
      acc[k][1] = a1;
    }
    __syncthreads();  // stage st is free again
    if (tid == 0 && issued < n_sub) issue(issued++);
  }

  // combine the key groups and write this split's partial result
  float* out = p.part + (static_cast<int64_t>(b) * p.Hq + hk * G) * p.nsplit * (D + 2);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    if (k >= ppt) break;
    const int pi = pi0 + k * kThreads;
    if (pi >= npairs) break;
    if (ks > 1) {
      sred[(kg * nact + pi0) * 2] = acc[k][0];
      sred[(kg * nact + pi0) * 2 + 1] = acc[k][1];
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    if (k >= ppt) break;
    const int pi = pi0 + k * kThreads;
    if (pi >= npairs || kg != 0) break;
    float a0 = acc[k][0], a1 = acc[k][1];
    if (ks > 1) {
      a0 = a1 = 0.f;
      for (int x = 0; x < ks; ++x) {
        a0 += sred[(x * nact + pi0) * 2];
        a1 += sred[(x * nact + pi0) * 2 + 1];
      }
    }
    const int g = pi / (D / 2), c = 2 * (pi % (D / 2));
    float* row = out + (static_cast<int64_t>(g) * p.nsplit + split) * (D + 2);
    row[c] = a0;
    row[c + 1] = a1;
  }
  if (tid < G) {
    float* row = out + (static_cast<int64_t>(tid) * p.nsplit + split) * (D + 2);
    row[D] = sm_[tid];
    row[D + 1] = sl[tid];
  }
}

// Merge the splits of every (batch, query head): one warp each.
template <typename In, int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecParams p) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<int64_t>(p.B) * p.Hq) return;
  const float* part = p.part + row * p.nsplit * (D + 2);
  float M = -INFINITY;
  for (int c = 0; c < p.nsplit; ++c)
    if (part[c * (D + 2) + D + 1] > 0.f) M = fmaxf(M, part[c * (D + 2) + D]);
  float L = 0.f, acc[D / 32];
#pragma unroll
  for (int x = 0; x < D / 32; ++x) acc[x] = 0.f;
  if (M > -INFINITY) {
    for (int c = 0; c < p.nsplit; ++c) {
      const float* r = part + c * (D + 2);
      const float l = r[D + 1];
      if (!(l > 0.f)) continue;
      const float w = expf(r[D] - M);
      L = fmaf(l, w, L);
#pragma unroll
      for (int x = 0; x < D / 32; ++x) acc[x] = fmaf(r[x * 32 + lane], w, acc[x]);
    }
  }
  In* o = static_cast<In*>(p.out) + row * D;
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int x = 0; x < D / 32; ++x) st1(o + x * 32 + lane, acc[x] * inv);
  if (lane == 0 && p.lse) p.lse[row] = L > 0.f ? M + logf(L) : -INFINITY;
}

// Ring-buffer append: slot pos[b] % cap of every (b, kv head) gets the new row.
template <typename In>
__global__ void kv_append_kernel(In* Kc, In* Vc, const In* kn, const In* vn, const int64_t* pos,
                                 int32_t Hkv, int64_t cap, int32_t D) {
  const int bk = blockIdx.x;
  const int64_t t = pos[bk / Hkv];
  if (t < 0) return;
  const int64_t dst = (static_cast<int64_t>(bk) * cap + t % cap) * D;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    Kc[dst + c] = kn[static_cast<int64_t>(bk) * D + c];
    Vc[dst + c] = vn[static_cast<int64_t>(bk) * D + c];
  }
}

template <typename In, int D>
cudaError_t launch_decode_typed(const DecParams& p, cudaStream_t st) {
  using Cfg = DecCfg<In, D>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(decode_kernel<In, D>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t ctas = static_cast<int64_t>(p.B) * p.Hkv * p.nsplit;
  decode_kernel<In, D><<<static_cast<unsigned>(ctas), kThreads, Cfg::kSmemBytes, st>>>(p);
  const int64_t rows = static_cast<int64_t>(p.B) * p.Hq;
  decode_combine_kernel<In, D><<<static_cast<unsigned>((rows + 3) / 4), 128, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

int decode_splits(int64_t B, int64_t Hkv, int64_t cap) {
  // enough CTAs for ~6 per SM (3 resident x 2 waves), each at least one sub-chunk
  const int64_t target = 148 * 6;
  const int64_t per = (target + B * Hkv - 1) / (B * Hkv);
  const int64_t max_split = (cap + kSub - 1) / kSub;
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(per, std::min<int64_t>(max_split, 64))));
}

int64_t decode_span(int64_t cap, int nsplit) {
  const int64_t span = (cap + nsplit - 1) / nsplit;
  return (span + kSub - 1) / kSub * kSub;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  DecParams p;
  p.q = a.q;
  p.Kc = a.Kc;
  p.Vc = a.Vc;
  p.pos = a.pos;
  p.out = a.out;
  p.lse = a.lse;
  p.part = a.part;
  p.err = a.err;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.Hq / a.Hkv;
  p.nsplit = a.nsplit;
  p.cap = a.cap;
  p.window = a.window;
  p.span = decode_span(a.cap, a.nsplit);
  p.scale = a.scale;
  if (a.bf16) {
    if (a.d == 64) return launch_decode_typed<__nv_bfloat16, 64>(p, st);
    if (a.d == 128) return launch_decode_typed<__nv_bfloat16, 128>(p, st);
  } else {
    if (a.d == 64) return launch_decode_typed<float, 64>(p, st);
    if (a.d == 128) return launch_decode_typed<float, 128>(p, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_kv_append(bool bf16, void* Kc, void* Vc, const void* kn, const void* vn,
                             const int64_t* pos, int32_t B, int32_t Hkv, int64_t cap, int32_t d,
                             cudaStream_t st) {
  const unsigned grid = static_cast<unsigned>(int64_t(B) * Hkv);
  if (bf16)
    kv_append_kernel<__nv_bfloat16><<<grid, 128, 0, st>>>(
        static_cast<__nv_bfloat16*>(Kc), static_cast<__nv_bfloat16*>(Vc),
        static_cast<const __nv_bfloat16*>(kn), static_cast<const __nv_bfloat16*>(vn), pos, Hkv,
        cap, d);
  else
    kv_append_kernel<float><<<grid, 128, 0, st>>>(static_cast<float*>(Kc), static_cast<float*>(Vc),
                                                  static_cast<const float*>(kn),
                                                  static_cast<const float*>(vn), pos, Hkv, cap, d);
  return cudaGetLastError();
}

}  // namespace spattn
