// fwd_simt.cu -- fp32 forward pass of block-sparse masked attention on the FP32
// FMA units (no TF32: its 10-bit mantissa cannot hold 1e-5 absolute error).
//
// Same definition and the same schedule walk as the tensor-core kernel (masked
// softmax normalised over S_i only: "Sparse attention" glossary, section "Choose
// the available reads"), at the granularity of 64-row query groups.  One CTA =
// one work item of 64 query rows of one (batch, head); 8 warps own 8 rows each.
// Keys are staged 32 at a time in shared memory; lane l scores key l, the row
// maximum and row sum are warp-shuffle reductions, and each lane accumulates
// d/32 output columns of every row it owns, with an online (rescaled) softmax in
// fp32 using expf.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "predicate.cuh"

namespace spattn {
namespace {

constexpr int kRows = 64;     // query rows per CTA
constexpr int kSub = 32;      // keys staged per step
constexpr int kWarps = 8;
constexpr int kRowsPerWarp = kRows / kWarps;

struct SParams {
  const float* Q;
  const float* K;
  const float* V;
  const float* Kc;
  const float* Vc;
  const float* Qg;
  float* O;
  float* LSE;
  float scale;
  int n_cols;
  const uint32_t* colmask;
  MaskDev mask;
  const int4* items;
  const int4* entries;
  unsigned long long* walk;
};

template <int D>
struct SimtCfg {
  static constexpr int kSmemFloats = kRows * D + kSub * (D + 1) + kSub * D;
  static constexpr int kSmemBytes = kSmemFloats * 4;
};

template <int D>
__global__ void __launch_bounds__(256) fwd_simt_kernel(const SParams p) {
  extern __shared__ float sm[];
  float* sq = sm;                       // [kRows][D]
  float* sk = sq + kRows * D;           // [kSub][D+1] (padded: lane l reads row l)
  float* sv = sk + kSub * (D + 1);      // [kSub][D]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int4 item = p.items[blockIdx.x];
  const int bh = blockIdx.y;
  const MaskDev& m = p.mask;
  const bool gathered = (item.w & kItemGathered) != 0;
  const long long T = m.T;

  // Q rows of this group (gathered global rows or consecutive rows), zero padded.
  for (int t = threadIdx.x; t < kRows * D; t += blockDim.x) {
    const int r = t / D, c = t % D;
    const int a = item.x + r;
    float v = 0.f;
    if (gathered) {
      if (a < m.n_global) v = p.Qg[(static_cast<long long>(bh) * m.n_global + a) * D + c];
    } else if (a < T) {
      v = p.Q[(static_cast<long long>(bh) * T + a) * D + c];
    }
    sq[t] = v;
  }

  int rows_i[kRowsPerWarp];
  bool rows_valid[kRowsPerWarp];
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int a = item.x + warp * kRowsPerWarp + k;
    if (gathered) {
      rows_valid[k] = a < m.n_global;
      rows_i[k] = rows_valid[k] ? m.gpos[a] : 0;
    } else {
      rows_valid[k] = a < T;
      rows_i[k] = a;
    }
  }
  float mrow[kRowsPerWarp], lrow[kRowsPerWarp], acc[kRowsPerWarp][D / 32];
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    mrow[k] = -INFINITY;
    lrow[k] = 0.f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) acc[k][c] = 0.f;
  }
  unsigned long long walked = 0;

  for (int n = 0; n < item.z; ++n) {
    const int4 e = p.entries[item.y + n];
    if (!(e.y & kActive0)) continue;
    ++walked;
    const int kind = (e.y >> kKindShift) & 3;
    const bool packed = kind == kKindPacked;
    const bool full = (e.y & kFull0) != 0;
    const float* Ks = packed ? p.Kc : p.K;
    const float* Vs = packed ? p.Vc : p.V;
    const long long src_rows = packed ? p.n_cols : T;

    for (int sb = 0; sb < kTile / kSub; ++sb) {
      __syncthreads();
      for (int t = threadIdx.x; t < kSub * D; t += blockDim.x) {
        const int r = t / D, c = t % D;
        const long long row = static_cast<long long>(e.x) + sb * kSub + r;
        float kv = 0.f, vv = 0.f;
        if (row < src_rows) {
          const long long off = (static_cast<long long>(bh) * src_rows + row) * D + c;
          kv = Ks[off];
          vv = Vs[off];
        }
        sk[r * (D + 1) + c] = kv;
        sv[r * D + c] = vv;
      }
      __syncthreads();
      const int cidx = sb * kSub + lane;  // column within the 128-key tile
#pragma unroll
      for (int k = 0; k < kRowsPerWarp; ++k) {
        const float* q = sq + (warp * kRowsPerWarp + k) * D;
        const float* kr = sk + lane * (D + 1);
        float dot = 0.f;
#pragma unroll 16
        for (int c = 0; c < D; ++c) dot = fmaf(q[c], kr[c], dot);
        // the row's predicate, rebuilt here rather than held for all rows (registers)
        const bool ok = full || pred_allowed(make_predicate(m, p.colmask, e, rows_i[k]), cidx);
        const float s = ok ? dot * p.scale : -INFINITY;
        float mx = s;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float mnew = fmaxf(mrow[k], mx);
        if (mnew == -INFINITY) continue;  // nothing allowed yet for this row (warp-uniform)
        const float corr = (mrow[k] == -INFINITY) ? 0.f : expf(mrow[k] - mnew);
        const float pj = ok ? expf(s - mnew) : 0.f;
        float sum = pj;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        lrow[k] = lrow[k] * corr + sum;
        mrow[k] = mnew;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float a = acc[k][c] * corr;
#pragma unroll 8
          for (int j = 0; j < kSub; ++j)
            a = fmaf(__shfl_sync(0xffffffffu, pj, j), sv[j * D + c * 32 + lane], a);
          acc[k][c] = a;
        }
      }
    }
  }

#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int i = rows_i[k];
    const bool write = rows_valid[k] && (gathered || !m.rowglobal[i]);
    if (!write) continue;
    const long long row = static_cast<long long>(bh) * T + i;
    const float inv = lrow[k] > 0.f ? 1.f / lrow[k] : 0.f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) p.O[row * D + c * 32 + lane] = acc[k][c] * inv;
    if (lane == 0 && p.LSE) p.LSE[row] = mrow[k] + logf(lrow[k]);
  }
  if (threadIdx.x == 0 && p.walk && walked) atomicAdd(p.walk, walked);
}

template <int D>
cudaError_t launch_d(const TcArgs& a, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(fwd_simt_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    SimtCfg<D>::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  SParams sp;
  sp.Q = static_cast<const float*>(a.Q);
  sp.K = static_cast<const float*>(a.K);
  sp.V = static_cast<const float*>(a.V);
  sp.Kc = static_cast<const float*>(a.Kc);
  sp.Vc = static_cast<const float*>(a.Vc);
  sp.Qg = static_cast<const float*>(a.Qg);
  sp.O = static_cast<float*>(a.O);
  sp.LSE = a.LSE;
  sp.scale = a.scale;
  sp.n_cols = a.n_cols;
  sp.colmask = a.colmask;
  sp.mask = a.mask;
  sp.items = a.items;
  sp.entries = a.entries;
  sp.walk = a.walk;
  dim3 grid(a.n_items, a.BH);
  fwd_simt_kernel<D><<<grid, 256, SimtCfg<D>::kSmemBytes, st>>>(sp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(int d, const TcArgs& a, cudaStream_t st) {
  if (a.n_items == 0) return cudaSuccess;
  if (d == 64) return launch_d<64>(a, st);
  if (d == 128) return launch_d<128>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace spattn
