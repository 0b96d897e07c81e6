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
// into shared memory through a ring of stages with an mbarrier per stage (TMA boxes
// for bf16, bulk copies of the valid rows for fp32), runs an online softmax over them
// for the G query heads, and leaves (max, sum, unnormalised output) per head; a second
// kernel merges the splits.  The valid slots of a step are one circular interval of
// slot space (up to two linear ones), so a sub-chunk is a run of consecutive slots and
// only its ragged end needs a mask.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace spattn {
namespace {

constexpr int kThreads = 256;
constexpr int kSub = 64;      // slots per sub-chunk
constexpr int kMaxGroup = 8;  // query heads per key/value head
constexpr int kStages = 2;    // sub-chunks (K and V rows) in flight per CTA
constexpr uint64_t kWaitBudget = 8000000000ull;

template <typename In, int D, int G>
struct DecCfg {
  static constexpr int kRowBytes = D * sizeof(In);
  static constexpr int kStageBytes = kSub * kRowBytes;  // K or V rows of one sub-chunk
  static constexpr int kVecPerRow = kRowBytes / 16;     // uint4 per row
  static constexpr int kVecPerLane = kVecPerRow / 8;    // 8 lanes per row
  static constexpr int kElemsPerVec = 16 / sizeof(In);
  static constexpr int kFrag = kVecPerLane * kElemsPerVec;  // = D / 8 elements per lane
  static constexpr int kPairs = D / 2;                      // column pairs of one head
  static constexpr int kKeyGroups = kThreads / kPairs;      // PV threads per column pair
  // shared layout: K [kStages], V [kStages] | scores [G][kSub] | weights [kSub][G] |
  // m, l, corr [8] | barriers
  static constexpr int kOffS = 2 * kStages * kStageBytes;
  static constexpr int kOffP = kOffS + G * kSub * 4;
  static constexpr int kOffStats = kOffP + G * kSub * 4;
  static constexpr int kOffBar = kOffStats + 3 * kMaxGroup * 4;
  static constexpr int kSmemBytes = kOffBar + 8 * kStages;
  static_assert(kKeyGroups * G * D * 4 <= 2 * kStages * kStageBytes, "reduction fits the stages");
};

// 16 bytes of In as kElemsPerVec floats, packed in pairs.
__device__ __forceinline__ void unpack(const uint4& v, uint64_t* out, const float*) {
  out[0] = (static_cast<uint64_t>(v.y) << 32) | v.x;
  out[1] = (static_cast<uint64_t>(v.w) << 32) | v.z;
}
__device__ __forceinline__ uint64_t ld2p(const float* p) {
  return *reinterpret_cast<const uint64_t*>(p);
}
__device__ __forceinline__ float ld1(const float* p) { return *p; }
__device__ __forceinline__ void st1(float* p, float v) { *p = v; }
__device__ __forceinline__ void st1(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

struct DecParams {
  const void* q;    // [B][Hq][D]
  const void* Kc;   // [B][Hkv][cap][D]
  const void* Vc;
  const int64_t* pos;  // [B]
  void* out;        // [B][Hq][D]
  float* lse;       // [B][Hq] or null
  float* part;      // [B*Hq][nsplit][D + 2]: unnormalised output, max (log2 units), sum
  int* err;
  const void* kn;   // [B][Hkv][D] the step's own key/value rows to append first, or null
  const void* vn;
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

// fp32 decode on the FP32 FMA units (the bf16 kernel is decode_mma_kernel below).
// Online softmax over the CTA's slots, one 64-slot sub-chunk (its K and V rows, one
// copy each) at a time through a ring of kStages buffers.  Scores run in log2 units:
// q is pre-multiplied by scale * log2(e), the weights are exp2 of the differences,
// and the combine step converts the result back.
template <typename In, int D, int G>
__global__ void __launch_bounds__(kThreads) decode_kernel(const DecParams p) {
  using Cfg = DecCfg<In, D, G>;
  constexpr int F2 = Cfg::kFrag / 2;
  extern __shared__ __align__(128) uint8_t smem[];
  In* sK = reinterpret_cast<In*>(smem);                                // [kStages][kSub][D]
  In* sV = reinterpret_cast<In*>(smem + kStages * Cfg::kStageBytes);  // [kStages][kSub][D]
  float* ss = reinterpret_cast<float*>(smem + Cfg::kOffS);             // [G][kSub] scores
  float* sp = reinterpret_cast<float*>(smem + Cfg::kOffP);             // [kSub][G] weights
  float* sm_ = reinterpret_cast<float*>(smem + Cfg::kOffStats);
  float* sl = sm_ + kMaxGroup;
  float* scorr = sl + kMaxGroup;
  const uint32_t bar0 = smem_addr(smem + Cfg::kOffBar);

  const int split = blockIdx.x % p.nsplit;
  const int bk = blockIdx.x / p.nsplit;  // b * Hkv + kv head
  const int b = bk / p.Hkv, hk = bk % p.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gi = lane >> 3, li = lane & 7;
  const int64_t t = p.pos[b];
  const int64_t lo = static_cast<int64_t>(split) * p.span;
  const Ranges rg = valid_ranges(t, p.cap, p.window, lo, min(p.cap, lo + p.span));
  int n_sub = 0;
  for (int k = 0; k < rg.n; ++k) n_sub += static_cast<int>((rg.b[k] - rg.a[k] + kSub - 1) / kSub);
  const In* Kbase = static_cast<const In*>(p.Kc) + static_cast<int64_t>(bk) * p.cap * D;
  const In* Vbase = static_cast<const In*>(p.Vc) + static_cast<int64_t>(bk) * p.cap * D;

  auto issue = [&](int o) {
    int64_t s0;
    int rows;
    sub_chunk(rg, o, s0, rows);
    const uint32_t bytes = static_cast<uint32_t>(rows) * Cfg::kRowBytes;
    const int st = o % kStages;
    const uint32_t bar = bar0 + 8 * st;
    mbar_arrive_expect_tx(bar, 2 * bytes);
    bulk_load(smem_addr(sK + st * kSub * D), Kbase + s0 * D, bytes, bar);
    bulk_load(smem_addr(sV + st * kSub * D), Vbase + s0 * D, bytes, bar);
  };
  int issued = 0;
  if (tid == 0) {  // the first copies start before anything else
    for (int k = 0; k < kStages; ++k) mbar_init(bar0 + 8 * k, 1);
    fence_barrier_init();
    for (; issued < kStages && issued < n_sub; ++issued) issue(issued);
  }
  if (tid < kMaxGroup) {
    sm_[tid] = -INFINITY;
    sl[tid] = 0.f;
  }
  // this lane's slice of the G query rows, scaled into log2 units
  uint64_t qf[G][F2];
  {
    const In* qb = static_cast<const In*>(p.q) + (static_cast<int64_t>(b) * p.Hq + hk * G) * D;
    const float qs = p.scale * 1.4426950408889634f;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int u = 0; u < Cfg::kVecPerLane; ++u)
#pragma unroll
        for (int e = 0; e < Cfg::kElemsPerVec; e += 2) {
          const In* src = qb + g * D + (li + 8 * u) * Cfg::kElemsPerVec + e;
          qf[g][(u * Cfg::kElemsPerVec + e) / 2] = f32x2(ld1(src) * qs, ld1(src + 1) * qs);
        }
  }
  __syncthreads();

  // weighted values: thread owns column pair cp of every head, for the keys
  // kg, kg + kKeyGroups, ... of each sub-chunk
  const int cp = tid % Cfg::kPairs, kg = tid / Cfg::kPairs;
  uint64_t acc[G];
#pragma unroll
  for (int g = 0; g < G; ++g) acc[g] = 0ull;

  for (int o = 0; o < n_sub; ++o) {
    const int st = o % kStages;
    bool ok = mbar_wait(bar0 + 8 * st, (o / kStages) & 1, kWaitBudget, p.err, kErrTimeout);
    ok = __syncthreads_and(ok);
    if (!ok) {
      // drain this CTA's copies still in flight (bounded), then leave
      if (tid == 0)
        for (int x = o; x < issued; ++x)
          mbar_wait(bar0 + 8 * (x % kStages), (x / kStages) & 1, kWaitBudget, p.err,
                    kErrTimeout);
      __syncthreads();
      return;
    }
    int64_t s0;
    int rows;
    sub_chunk(rg, o, s0, rows);
    const In* K = sK + st * kSub * D;
    const In* V = sV + st * kSub * D;
    // scores: 8 lanes per key row, 4 rows per warp, 32 rows per pass
#pragma unroll
    for (int pass = 0; pass < kSub / 32; ++pass) {
      const int r = pass * 32 + warp * 4 + gi;
      uint64_t kf[F2];
#pragma unroll
      for (int u = 0; u < Cfg::kVecPerLane; ++u)
        unpack(reinterpret_cast<const uint4*>(K + r * D)[li + 8 * u],
               kf + u * Cfg::kElemsPerVec / 2, static_cast<const In*>(nullptr));
#pragma unroll
      for (int g = 0; g < G; ++g) {
        uint64_t a2 = 0ull;
#pragma unroll
        for (int x = 0; x < F2; ++x) a2 = fma_f32x2(qf[g][x], kf[x], a2);
        float lo2, hi2;
        f32x2_split(a2, lo2, hi2);
        float dot = lo2 + hi2;
        dot += __shfl_xor_sync(0xffffffffu, dot, 1);
        dot += __shfl_xor_sync(0xffffffffu, dot, 2);
        dot += __shfl_xor_sync(0xffffffffu, dot, 4);
        if (li == 0) ss[g * kSub + r] = r < rows ? dot : -INFINITY;
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
      const float pa = exp2f(s_a - m_new), pb = exp2f(s_b - m_new);
      float sum = pa + pb;
#pragma unroll
      for (int k = 16; k > 0; k >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, k);
      sp[lane * G + warp] = pa;
      sp[(lane + 32) * G + warp] = pb;
      if (lane == 0) {
        const float corr = exp2f(m_old - m_new);  // 0 on the first sub-chunk
        scorr[warp] = corr;
        sl[warp] = sl[warp] * corr + sum;
        sm_[warp] = m_new;
      }
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float c = scorr[g];
      acc[g] = fma_f32x2(acc[g], f32x2(c, c), 0ull);
    }
    for (int j = kg; j < rows; j += Cfg::kKeyGroups) {
      const uint64_t v2 = ld2p(V + j * D + 2 * cp);
      float pw[G];
      if constexpr (G % 4 == 0) {
#pragma unroll
        for (int g = 0; g < G; g += 4) {
          const float4 x = *reinterpret_cast<const float4*>(sp + j * G + g);
          pw[g] = x.x;
          pw[g + 1] = x.y;
          pw[g + 2] = x.z;
          pw[g + 3] = x.w;
        }
      } else {
#pragma unroll
        for (int g = 0; g < G; ++g) pw[g] = sp[j * G + g];
      }
#pragma unroll
      for (int g = 0; g < G; ++g) acc[g] = fma_f32x2(f32x2(pw[g], pw[g]), v2, acc[g]);
    }
    __syncthreads();  // stage st is free again
    if (tid == 0 && issued < n_sub) issue(issued++);
  }

  // sum the key groups (in the now idle stage buffers) and write this split's partial
  float* red = reinterpret_cast<float*>(smem);  // [kKeyGroups][G][D]
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float a0, a1;
    f32x2_split(acc[g], a0, a1);
    red[(kg * G + g) * D + 2 * cp] = a0;
    red[(kg * G + g) * D + 2 * cp + 1] = a1;
  }
  __syncthreads();
  float* out = p.part + (static_cast<int64_t>(b) * p.Hq + hk * G) * p.nsplit * (D + 2);
  for (int x = tid; x < G * D; x += kThreads) {
    const int g = x / D, c = x % D;
    float a = 0.f;
#pragma unroll
    for (int k = 0; k < Cfg::kKeyGroups; ++k) a += red[(k * G + g) * D + c];
    out[(static_cast<int64_t>(g) * p.nsplit + split) * (D + 2) + c] = a;
  }
  if (tid < G) {
    float* row = out + (static_cast<int64_t>(tid) * p.nsplit + split) * (D + 2);
    row[D] = sm_[tid];
    row[D + 1] = sl[tid];
  }
}

// bf16 decode with the dot products on the warp-level tensor cores.  The scores of a
// group's G query heads against a sub-chunk of keys are S^T = K q^T (an m16n8k16 MMA:
// 16 slots x 8 heads, the heads past G zero), and the output is O^T += V^T P^T (16 value
// columns x 8 heads per MMA).  That takes the dot products off the FP32 and issue paths,
// which bound the plain version, so the step is left to the memory system.  Each of the
// 4 warps owns 16 slots of every 64-slot sub-chunk and keeps its own running max, sum
// and output (in the MMA fragment layout a lane holds heads 2 (l % 4) and 2 (l % 4) + 1
// in S^T and O^T alike, so its running max rescales its own outputs); the warps merge
// once at the end.  A sub-chunk's K and V rows arrive as TMA boxes of 64 rows x 64
// columns with the 128-byte swizzle (16-byte chunk c of row r stored at chunk c ^ (r % 8)),
// which keeps the eight rows of every 8 x 8 matrix load in distinct banks.
constexpr int kMmaWarps = 4;
constexpr int kMmaThreads = 32 * kMmaWarps;
// three sub-chunks in flight (96 KB at d = 128, still two CTAs per SM): with few heads a
// CTA's share of the bandwidth needs the third stage to cover the memory latency
constexpr int kMmaStages = 3;

template <int D>
struct MmaCfg {
  static constexpr int kBoxBytes = kSub * 128;           // 64 rows x 64 bf16 columns
  static constexpr int kBoxes = D / 64;                   // boxes per row block
  static constexpr int kTensorBytes = kBoxes * kBoxBytes;  // K or V rows of one sub-chunk
  static constexpr int kStageBytes = 2 * kTensorBytes;    // K then V
  static constexpr int kSteps = D / 16;                   // 16-wide steps over d (k or m tiles)
  // shared layout (1024-byte aligned): stages [kMmaStages] of K, V | per-warp max and
  // sum [2][warps][8] | barriers full [kMmaStages], empty [kMmaStages]
  static constexpr int kOffStats = kMmaStages * kStageBytes;
  static constexpr int kOffBar = kOffStats + 2 * kMmaWarps * 8 * 4;
  static constexpr int kSmemBytes = kOffBar + 16 * kMmaStages + 1024;
  static_assert(kSub == 16 * kMmaWarps, "16 slots per warp");
  static_assert(kMmaWarps * 8 * D * 4 <= kMmaStages * kStageBytes, "warp partials fit");
  static_assert(kOffBar % 8 == 0, "alignment");
};

// Shared address of 16-byte chunk c (8 columns) of row r in a swizzled row block.
__device__ __forceinline__ uint32_t swz(uint32_t block, int r, int c) {
  return block + (c >> 3) * (kSub * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

template <int D, int G>
__global__ void __launch_bounds__(kMmaThreads)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const DecParams p) {
  using Cfg = MmaCfg<D>;
  constexpr float kRescale = 8.0f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s0addr = smem_addr(smem);                      // stage st at + st * kStageBytes
  float* wm = reinterpret_cast<float*>(smem + Cfg::kOffStats);  // [warps][8] max
  float* wl = wm + kMmaWarps * 8;                               // [warps][8] sum
  const uint32_t full0 = smem_addr(smem + Cfg::kOffBar);
  const uint32_t empty0 = full0 + 8 * kMmaStages;

  const int split = blockIdx.x % p.nsplit;
  const int bk = blockIdx.x / p.nsplit;  // b * Hkv + kv head
  const int b = bk / p.Hkv, hk = bk % p.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = lane >> 2, tig = lane & 3;
  const int64_t t = p.pos[b];
  const int64_t lo = static_cast<int64_t>(split) * p.span;
  const Ranges rg = valid_ranges(t, p.cap, p.window, lo, min(p.cap, lo + p.span));
  int n_sub = 0;
  for (int k = 0; k < rg.n; ++k) n_sub += static_cast<int>((rg.b[k] - rg.a[k] + kSub - 1) / kSub);
  // With the step's own rows given (spattn_decode_append), the CTA whose slot range
  // holds slot t % cap appends them: it writes them to the cache for later steps and
  // puts them into its shared tile of that slot after the copy has landed, so this step
  // reads them without waiting for the global write.  No other CTA reads that slot.
  const int64_t s_new = (p.kn && t >= 0) ? t % p.cap : -1;
  const bool owner = s_new >= lo && s_new < min(p.cap, lo + p.span);
  const uint4* kn_row = owner ? reinterpret_cast<const uint4*>(
                                    static_cast<const __nv_bfloat16*>(p.kn) + static_cast<int64_t>(bk) * D)
                              : nullptr;
  const uint4* vn_row = owner ? reinterpret_cast<const uint4*>(
                                    static_cast<const __nv_bfloat16*>(p.vn) + static_cast<int64_t>(bk) * D)
                              : nullptr;
  if (owner && threadIdx.x >= 64 && threadIdx.x < 64 + 2 * (D / 8)) {  // warps 2-3: global rows
    const int c = threadIdx.x - 64;  // 16-byte chunk c % (D / 8) of K (c < D / 8) or V
    const int64_t off = (static_cast<int64_t>(bk) * p.cap + s_new) * D;
    uint4* dst = reinterpret_cast<uint4*>(
        const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(c < D / 8 ? p.Kc : p.Vc)) + off);
    dst[c % (D / 8)] = (c < D / 8 ? kn_row : vn_row)[c % (D / 8)];
  }

  // thread 0 copies sub-chunk o: 64 rows from its first slot, K then V, one box per 64
  // columns (rows past the slot range are read too, and masked; past cap they are zero)
  auto issue = [&](int o) {
    int64_t s0;
    int rows;
    sub_chunk(rg, o, s0, rows);
    const int st = o % kMmaStages;
    const uint32_t bar = full0 + 8 * st, dst = s0addr + st * Cfg::kStageBytes;
    mbar_arrive_expect_tx(bar, Cfg::kStageBytes);
#pragma unroll
    for (int c = 0; c < Cfg::kBoxes; ++c) {
      tma_load_4d(dst + c * Cfg::kBoxBytes, &tmK, bar, 64 * c, 0, static_cast<int>(s0), bk);
      tma_load_4d(dst + Cfg::kTensorBytes + c * Cfg::kBoxBytes, &tmV, bar, 64 * c, 0,
                  static_cast<int>(s0), bk);
    }
  };
  int issued = 0;  // copies issued so far: counted alike by every lane of warp 0
  if (warp == 0) {  // the first copies start before anything else
    if (lane == 0) {
      for (int k = 0; k < kMmaStages; ++k) {
        mbar_init(full0 + 8 * k, 1);
        mbar_init(empty0 + 8 * k, kMmaWarps);
      }
      fence_barrier_init();
    }
    for (; issued < kMmaStages && issued < n_sub; ++issued)
      if (lane == 0) issue(issued);
    __syncwarp();
  }
  // q as the B operand of S^T = K q^T: lane holds elements 16 kk + 2 tig (+1) and
  // (+8) of head grp; heads past G are zero
  uint32_t qb[Cfg::kSteps][2];
  {
    const __nv_bfloat16* qg =
        static_cast<const __nv_bfloat16*>(p.q) + (static_cast<int64_t>(b) * p.Hq + hk * G) * D;
#pragma unroll
    for (int kk = 0; kk < Cfg::kSteps; ++kk) {
      qb[kk][0] = 0u;
      qb[kk][1] = 0u;
      if (grp < G) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(qg + grp * D + 16 * kk + 2 * tig);
        qb[kk][0] = src[0];
        qb[kk][1] = src[4];
      }
    }
  }
  __syncthreads();  // barrier initialisation is visible

  const float c2 = p.scale * 1.4426950408889634f;  // scores in log2 units
  float m[2] = {-INFINITY, -INFINITY}, lp[2] = {0.f, 0.f};  // heads 2 tig, 2 tig + 1
  float o[Cfg::kSteps][4];  // O^T: value column 16 mt + grp (+8), heads 2 tig (+1)
#pragma unroll
  for (int mt = 0; mt < Cfg::kSteps; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
  // this lane's rows in the 8 x 8 matrix loads: K as the A operand of S^T, V as the
  // (transposed) A operand of O^T
  const int k0 = warp * 16;  // this warp's slots [k0, k0 + 16) of every sub-chunk
  const int rk = k0 + (lane & 7) + 8 * ((lane >> 3) & 1), ck = lane >> 4;
  const int rv = k0 + (lane & 7) + 8 * ((lane >> 4) & 1), cv = (lane >> 3) & 1;
  bool ok = true;
  for (int sc = 0; sc < n_sub; ++sc) {
    const int st = sc % kMmaStages;
    if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * st, (sc / kMmaStages) & 1, kWaitBudget,
                                           p.err, kErrTimeout))) {
      ok = false;
      break;
    }
    int64_t s0;
    int rows;
    sub_chunk(rg, sc, s0, rows);
    if (owner && s_new >= s0 && s_new < s0 + rows && (s_new - s0) / 16 == warp) {
      // this warp's rows hold the appended slot: the step's own K and V rows replace
      // whatever the copy read there (lane l: 16-byte chunk l % (D / 8) of K or V)
      const int r = static_cast<int>(s_new - s0);
      uint8_t* blk = smem + st * Cfg::kStageBytes;
      for (int x = lane; x < 2 * (D / 8); x += 32) {
        const int c = x % (D / 8);
        uint8_t* tile = blk + (x < D / 8 ? 0 : Cfg::kTensorBytes);
        *reinterpret_cast<uint4*>(tile + (c >> 3) * Cfg::kBoxBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4)) =
            (x < D / 8 ? kn_row : vn_row)[c];
      }
      fence_proxy_async_smem();  // ordered before the copies that later refill the stage
      __syncwarp();
    }
    if (k0 < rows) {  // (slot k0 valid: every max below is finite)
      const uint32_t kst = s0addr + st * Cfg::kStageBytes, vst = kst + Cfg::kTensorBytes;
      if (k0 + 16 > rows) {
        // rows past the slot range hold other slots' values; zero them so that
        // 0-weight slots add exact zeros (whatever those rows hold)
        uint8_t* vblk = smem + st * Cfg::kStageBytes + Cfg::kTensorBytes;
        for (int x = lane; x < (k0 + 16 - rows) * Cfg::kBoxes * 8; x += 32) {
          const int r = rows + x / (Cfg::kBoxes * 8), c = x % (Cfg::kBoxes * 8);
          *reinterpret_cast<uint4*>(vblk + (c >> 3) * Cfg::kBoxBytes + r * 128 + 16 * (c & 7)) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // ordered before the copies that later refill the stage
        __syncwarp();
      }
      // S^T (16 slots x 8 heads) = K q^T, over d in 16-wide steps
      float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < Cfg::kSteps; ++kk) {
        uint32_t a[4];
        ldmatrix_x4(swz(kst, rk, 2 * kk + ck), a);
        mma_16816_bf16(s, a, qb[kk][0], qb[kk][1]);
      }
      // lane: slots k0 + grp (s[0], s[1]) and k0 + grp + 8 (s[2], s[3]), heads 2 tig (+1)
      const bool va = k0 + grp < rows, vb = k0 + grp + 8 < rows;
      const float x[4] = {va ? s[0] * c2 : -INFINITY, va ? s[1] * c2 : -INFINITY,
                          vb ? s[2] * c2 : -INFINITY, vb ? s[3] * c2 : -INFINITY};
      // per head, the max over the warp's 16 slots (the 8 lanes sharing tig); the
      // running max moves (and the outputs rescale) only when it grows by more than 2^8
      float corr[2];
      bool need = false;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float mx = fmaxf(x[j], x[2 + j]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        corr[j] = 1.f;
        if (mx > m[j] + kRescale) {
          corr[j] = exp2f(m[j] - mx);  // 0 while m[j] is -inf
          lp[j] *= corr[j];
          m[j] = mx;
          need = true;
        }
      }
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int mt = 0; mt < Cfg::kSteps; ++mt) {
          o[mt][0] *= corr[0];
          o[mt][1] *= corr[1];
          o[mt][2] *= corr[0];
          o[mt][3] *= corr[1];
        }
      }
      float pw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) pw[e] = exp2f(x[e] - m[e & 1]);  // 0 for slots past the rows
      lp[0] += pw[0] + pw[2];
      lp[1] += pw[1] + pw[3];
      // P^T as the B operand: the transposes of P's two 8 x 8 blocks (slots x heads)
      const uint32_t b0 = movmatrix_trans(pack_bf16x2(pw[0], pw[1]));
      const uint32_t b1 = movmatrix_trans(pack_bf16x2(pw[2], pw[3]));
      // O^T (d x heads) += V^T (d x slots) P^T (slots x heads), 16 value columns a step
#pragma unroll
      for (int mt = 0; mt < Cfg::kSteps; ++mt) {
        uint32_t a[4];
        ldmatrix_x4_trans(swz(vst, rv, 2 * mt + cv), a);
        mma_16816_bf16(o[mt], a, b0, b1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);  // this warp has left the stage
    if (warp == 0 && issued < n_sub) {            // refill it once every warp has left
      if (__all_sync(0xffffffffu, mbar_wait(empty0 + 8 * st, (sc / kMmaStages) & 1, kWaitBudget,
                                            p.err, kErrTimeout))) {
        if (lane == 0) issue(issued);
        ++issued;
      } else {
        ok = false;
      }
      __syncwarp();
    }
  }
  // drain: the last copies issued into each stage have landed (at once when consumed)
  if (tid == 0)
    for (int x = max(0, issued - kMmaStages); x < issued; ++x)
      mbar_wait(full0 + 8 * (x % kMmaStages), (x / kMmaStages) & 1, kWaitBudget, p.err,
                kErrTimeout);
  if (!__syncthreads_and(ok)) return;

  // merge the warps (in the now idle stage buffers) and write this split's partial
  float* red = reinterpret_cast<float*>(smem);  // [warps][8][D]
#pragma unroll
  for (int j = 0; j < 2; ++j) {  // the warp's sum: the 8 lanes sharing tig
    lp[j] += __shfl_xor_sync(0xffffffffu, lp[j], 4);
    lp[j] += __shfl_xor_sync(0xffffffffu, lp[j], 8);
    lp[j] += __shfl_xor_sync(0xffffffffu, lp[j], 16);
  }
#pragma unroll
  for (int mt = 0; mt < Cfg::kSteps; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      red[(warp * 8 + 2 * tig + (e & 1)) * D + 16 * mt + grp + 8 * (e >> 1)] = o[mt][e];
  if (grp == 0) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      wm[warp * 8 + 2 * tig + j] = m[j];
      wl[warp * 8 + 2 * tig + j] = lp[j];
    }
  }
  __syncthreads();
  float* out = p.part + (static_cast<int64_t>(b) * p.Hq + hk * G) * p.nsplit * (D + 2);
  for (int x = tid; x < G * D; x += kMmaThreads) {
    const int g = x / D, c = x % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w) M = fmaxf(M, wm[w * 8 + g]);
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w)
      if (wm[w * 8 + g] > -INFINITY) a = fmaf(red[(w * 8 + g) * D + c], exp2f(wm[w * 8 + g] - M), a);
    out[(static_cast<int64_t>(g) * p.nsplit + split) * (D + 2) + c] = a;
  }
  if (tid < G) {
    float M = -INFINITY, L = 0.f;
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w) M = fmaxf(M, wm[w * 8 + tid]);
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w)
      if (wm[w * 8 + tid] > -INFINITY) L = fmaf(wl[w * 8 + tid], exp2f(wm[w * 8 + tid] - M), L);
    float* row = out + (static_cast<int64_t>(tid) * p.nsplit + split) * (D + 2);
    row[D] = M;
    row[D + 1] = L;
  }
}

// Merge the splits of every (batch, query head): one warp each.  Maxima are in log2
// units; LSE is returned in natural-log units.
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
      const float w = exp2f(r[D] - M);
      L = fmaf(l, w, L);
#pragma unroll
      for (int x = 0; x < D / 32; ++x) acc[x] = fmaf(r[x * 32 + lane], w, acc[x]);
    }
  }
  In* o = static_cast<In*>(p.out) + row * D;
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int x = 0; x < D / 32; ++x) st1(o + x * 32 + lane, acc[x] * inv);
  if (lane == 0 && p.lse) p.lse[row] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
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

// bf16 runs on the warp-level tensor cores; fp32 (products that must stay within 1e-5)
// on the FP32 FMA units.
template <typename In, int D, int G>
cudaError_t launch_decode_g(const DecParams& p, cudaStream_t st) {
  constexpr bool kMma = std::is_same<In, __nv_bfloat16>::value;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    if constexpr (kMma)
      attr_err = cudaFuncSetAttribute(decode_mma_kernel<D, G>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      MmaCfg<D>::kSmemBytes);
    else
      attr_err = cudaFuncSetAttribute(decode_kernel<In, D, G>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      DecCfg<In, D, G>::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const unsigned ctas = static_cast<unsigned>(static_cast<int64_t>(p.B) * p.Hkv * p.nsplit);
  if constexpr (kMma) {
    CUtensorMap mK, mV;  // the caches as [B * Hkv][cap][D], boxes of 64 slots x 64 columns
    const long long bh = static_cast<long long>(p.B) * p.Hkv;
    if (!make_map(&mK, p.Kc, D, p.cap, bh, 1, kSub) || !make_map(&mV, p.Vc, D, p.cap, bh, 1, kSub))
      return cudaErrorInvalidValue;
    decode_mma_kernel<D, G><<<ctas, kMmaThreads, MmaCfg<D>::kSmemBytes, st>>>(mK, mV, p);
  } else
    decode_kernel<In, D, G><<<ctas, kThreads, DecCfg<In, D, G>::kSmemBytes, st>>>(p);
  const int64_t rows = static_cast<int64_t>(p.B) * p.Hq;
  decode_combine_kernel<In, D><<<static_cast<unsigned>((rows + 3) / 4), 128, 0, st>>>(p);
  return cudaGetLastError();
}

template <typename In, int D>
cudaError_t launch_decode_typed(const DecParams& p, cudaStream_t st) {
  switch (p.G) {
    case 1: return launch_decode_g<In, D, 1>(p, st);
    case 2: return launch_decode_g<In, D, 2>(p, st);
    case 4: return launch_decode_g<In, D, 4>(p, st);
    case 8: return launch_decode_g<In, D, 8>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int decode_splits(int64_t B, int64_t Hkv, int64_t cap) {
  // At most 2 x 148 CTAs in all (the bf16 kernel keeps two per SM resident, so this
  // is a single wave): few, long CTAs amortise each CTA's start-up and final merge over
  // many sub-chunks.  Measured on the bf16 kernel (graph-replayed steps): B = 8 (64 kv
  // heads) 31.7 us at 4 splits against 34.1 at 6 and 38.0 at 2; B = 32 (256 kv heads)
  // 88.7 us at 1 split against 93.6 at 3.
  constexpr int64_t kResidentCtas = 2 * 148;
  const int64_t per = kResidentCtas / (B * Hkv);
  const int64_t most = (cap + kSub - 1) / kSub;
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(per, std::min<int64_t>(most, 64))));
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
  p.kn = a.kn;
  p.vn = a.vn;
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
