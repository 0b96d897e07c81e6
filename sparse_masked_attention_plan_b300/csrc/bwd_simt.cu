// bwd_simt.cu -- gradients of block-sparse masked attention on the FP32 FMA units
// (fp32 inputs; bf16 inputs use this file's row-dot kernel and the tensor-core
// kernels of bwd_tc.cu).
//
// For y_i = sum_{j in S_i} alpha_ij v_j with alpha_ij = softmax over S_i of
// s_ij = scale q_i . k_j ("Sparse attention" glossary, section "Choose the
// available reads"), the chain rule through the softmax over S_i gives, with
// D_i = dO_i . y_i and alpha_ij = exp(s_ij - LSE_i) recomputed from the saved LSE:
//   dp_ij = dO_i . v_j,   ds_ij = alpha_ij (dp_ij - D_i),
//   dQ_i = scale sum_j ds_ij k_j,  dK_j = scale sum_i ds_ij q_i,  dV_j = sum_i alpha_ij dO_i.
// Three kernels:
//   * rowdot: D_i for every row (one warp per row);
//   * dq: query-major, the fp32 forward schedule (64-row groups) and predicate, so
//     every row's dQ is summed inside one CTA;
//   * dkdv: key-major, 64-key units of the backward schedule (the same split of each
//     row's allowed set into band keys, packed sparse columns and dense walks of
//     global rows, listed per key), so every key's dK and dV are summed inside one
//     CTA.  Units of packed columns run first and leave fp32 partial sums that the
//     natural unit of the same key adds before the single rounding to the output.
// No atomics: the result does not depend on the launch order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "predicate.cuh"

namespace spattn {
namespace {

constexpr int kThreads = 256;

template <typename In>
__device__ __forceinline__ float ld(const In* p, long long i);
template <>
__device__ __forceinline__ float ld<float>(const float* p, long long i) {
  return p[i];
}
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p, long long i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st(float* p, long long i, float v) { p[i] = v; }
__device__ __forceinline__ void st(__nv_bfloat16* p, long long i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

// ---- D_i = dO_i . O_i ---------------------------------------------------------------

template <typename In, int D>
__global__ void __launch_bounds__(kThreads) rowdot_kernel(const In* __restrict__ O,
                                                          const In* __restrict__ dO,
                                                          float* __restrict__ Dvec,
                                                          long long rows) {
  const long long r = static_cast<long long>(blockIdx.x) * (kThreads / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float acc = 0.f;
#pragma unroll
  for (int c = lane; c < D; c += 32) acc = fmaf(ld(O, r * D + c), ld(dO, r * D + c), acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) Dvec[r] = acc;
}

// ---- dQ: query-major ------------------------------------------------------------------

constexpr int kQRows = 64, kSub = 32, kWarps = kThreads / 32, kRowsPerWarp = kQRows / kWarps;

template <int D>
struct DqCfg {
  static constexpr int kSmemBytes = (2 * kQRows * D + 2 * kSub * (D + 1)) * 4;
};

template <typename In, int D>
__global__ void __launch_bounds__(kThreads) dq_kernel(const BwdArgs p) {
  extern __shared__ float sm[];
  float* sq = sm;                     // [kQRows][D]
  float* sdo = sq + kQRows * D;       // [kQRows][D]
  float* sk = sdo + kQRows * D;       // [kSub][D+1]
  float* sv = sk + kSub * (D + 1);    // [kSub][D+1]
  const In* Q = static_cast<const In*>(p.Q);
  const In* K = static_cast<const In*>(p.K);
  const In* V = static_cast<const In*>(p.V);
  const In* dO = static_cast<const In*>(p.dO);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int4 item = p.q_items[blockIdx.x];
  const int bh = blockIdx.y;
  const MaskDev& m = p.mask;
  const bool gathered = (item.w & kItemGathered) != 0;
  const long long T = m.T;
  const long long head = static_cast<long long>(bh) * T;

  for (int t = threadIdx.x; t < kQRows * D; t += blockDim.x) {
    const int r = t / D, c = t % D;
    const int a = item.x + r;
    long long i = -1;
    if (gathered) {
      if (a < m.n_global) i = m.gpos[a];
    } else if (a < T) {
      i = a;
    }
    sq[t] = i >= 0 ? ld(Q, (head + i) * D + c) : 0.f;
    sdo[t] = i >= 0 ? ld(dO, (head + i) * D + c) : 0.f;
  }
  int rows_i[kRowsPerWarp];
  bool rows_valid[kRowsPerWarp];
  float lse[kRowsPerWarp], dv[kRowsPerWarp], acc[kRowsPerWarp][D / 32];
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int a = item.x + warp * kRowsPerWarp + k;
    rows_valid[k] = gathered ? a < m.n_global : a < T;
    rows_i[k] = rows_valid[k] ? (gathered ? m.gpos[a] : a) : 0;
    lse[k] = rows_valid[k] ? p.LSE[head + rows_i[k]] : 0.f;
    dv[k] = rows_valid[k] ? p.Dvec[head + rows_i[k]] : 0.f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) acc[k][c] = 0.f;
  }

  for (int n = 0; n < item.z; ++n) {
    const int4 e = p.q_entries[item.y + n];
    if (!(e.y & kActive0)) continue;
    const int kind = (e.y >> kKindShift) & 3;
    const bool packed = kind == kKindPacked;
    const bool full = (e.y & kFull0) != 0;
    const long long src_rows = packed ? p.n_cols : T;
    for (int sb = 0; sb < kTile / kSub; ++sb) {
      __syncthreads();
      for (int t = threadIdx.x; t < kSub * D; t += blockDim.x) {
        const int r = t / D, c = t % D;
        const long long row = static_cast<long long>(e.x) + sb * kSub + r;
        float kv = 0.f, vv = 0.f;
        if (row < src_rows) {
          const long long j = packed ? p.cols[row] : row;
          kv = ld(K, (head + j) * D + c);
          vv = ld(V, (head + j) * D + c);
        }
        sk[r * (D + 1) + c] = kv;
        sv[r * (D + 1) + c] = vv;
      }
      __syncthreads();
      const int cidx = sb * kSub + lane;
#pragma unroll 1
      for (int k = 0; k < kRowsPerWarp; ++k) {
        if (!rows_valid[k]) continue;  // warp-uniform
        const float* q = sq + (warp * kRowsPerWarp + k) * D;
        const float* g = sdo + (warp * kRowsPerWarp + k) * D;
        const float* kr = sk + lane * (D + 1);
        const float* vr = sv + lane * (D + 1);
        float s = 0.f, dp = 0.f;
#pragma unroll 16
        for (int c = 0; c < D; ++c) {
          s = fmaf(q[c], kr[c], s);
          dp = fmaf(g[c], vr[c], dp);
        }
        const bool ok = full || pred_allowed(make_predicate(m, p.colmask, e, rows_i[k]), cidx);
        const float pij = ok ? expf(s * p.scale - lse[k]) : 0.f;
        const float ds = pij * (dp - dv[k]);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float a = acc[k][c];
#pragma unroll 8
          for (int j = 0; j < kSub; ++j)
            a = fmaf(__shfl_sync(0xffffffffu, ds, j), sk[j * (D + 1) + c * 32 + lane], a);
          acc[k][c] = a;
        }
      }
    }
  }

  In* dQ = static_cast<In*>(p.dQ);
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int i = rows_i[k];
    if (!rows_valid[k] || !(gathered || !m.rowglobal[i])) continue;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) st(dQ, (head + i) * D + c * 32 + lane, acc[k][c] * p.scale);
  }
}

// ---- dK, dV: key-major ----------------------------------------------------------------
//
// Thread t owns key t / 4 of the unit and the quarter g = t % 4 of the head
// dimension; a row's dot products are reduced over the four quarter lanes.  Shared
// rows are stored as four chunks of D/4 values each skewed by 4 floats, so the
// four quarters of one row start in different banks.

template <int D>
struct KvCfg {
  static constexpr int kChunk = D / 4;
  static constexpr int kRowStride = 4 * (kChunk + 4);
  static constexpr int kSmemBytes = (2 * kBwdRows * kRowStride + 2 * kBwdRows) * 4 + kBwdRows * 4;
};

__device__ __forceinline__ bool in_random(const MaskDev& m, long long i, long long j) {
  if (m.rand_block == 0) return false;
  const int q = static_cast<int>(i / m.rand_block), k = static_cast<int>(j / m.rand_block);
  for (int x = m.r_off[q]; x < m.r_off[q + 1]; ++x)
    if (m.r_kb[x] == k) return true;
  return false;
}

__device__ __forceinline__ bool band_allowed(const MaskDev& m, const uint32_t* colmask,
                                             long long i, long long j) {
  const long long gap = i - j;
  bool local;
  if (m.causal) {
    local = gap >= 0 && (m.window == 0 || gap < static_cast<long long>(m.window) * m.dilation);
  } else {
    const long long a = gap < 0 ? -gap : gap;
    local = m.radius < 0 || a <= static_cast<long long>(m.radius) * m.dilation;
  }
  if (local && m.dilation > 1) local = ((gap % m.dilation) + m.dilation) % m.dilation == 0;
  if (local) return true;
  const uint32_t w = colmask[(j / kTile) * 4 + (j % kTile) / 32];
  return (((w >> (j & 31)) & 1u) || in_random(m, i, j)) && (!m.causal || j <= i);
}

// A key tile reached only by random blocks: the random keys that are not strided or
// global columns (the packed entries cover those).
__device__ __forceinline__ bool random_allowed(const MaskDev& m, const uint32_t* colmask,
                                               long long i, long long j) {
  const uint32_t w = colmask[(j / kTile) * 4 + (j % kTile) / 32];
  return !((w >> (j & 31)) & 1u) && in_random(m, i, j) && (!m.causal || j <= i);
}

template <typename In, int D>
__global__ void __launch_bounds__(kThreads) dkdv_kernel(const BwdArgs p, int unit0) {
  using Cfg = KvCfg<D>;
  constexpr int C = Cfg::kChunk;
  extern __shared__ float sm[];
  float* sq = sm;                                  // [64][kRowStride]
  float* sdo = sq + kBwdRows * Cfg::kRowStride;    // [64][kRowStride]
  float* slse = sdo + kBwdRows * Cfg::kRowStride;  // [64]
  float* sdv = slse + kBwdRows;                    // [64]
  int* srow = reinterpret_cast<int*>(sdv + kBwdRows);  // [64] row index, -1 = skip
  const In* Q = static_cast<const In*>(p.Q);
  const In* K = static_cast<const In*>(p.K);
  const In* V = static_cast<const In*>(p.V);
  const In* dO = static_cast<const In*>(p.dO);
  const MaskDev& m = p.mask;
  const long long T = m.T;
  const int4 unit = p.units[unit0 + blockIdx.x];
  const bool packed_unit = (unit.w & kUnitPacked) != 0;
  const int bh = blockIdx.y;
  const long long head = static_cast<long long>(bh) * T;
  const int kk = threadIdx.x >> 2, g = threadIdx.x & 3;
  const int key = unit.x + kk;  // key row, or packed column index
  const bool key_valid = packed_unit ? key < p.n_cols : key < T;
  const long long j = key_valid ? (packed_unit ? p.cols[key] : key) : 0;

  float kr[C], vr[C], dk[C], dvv[C];
#pragma unroll
  for (int x = 0; x < C; ++x) {
    kr[x] = key_valid ? ld(K, (head + j) * D + g * C + x) : 0.f;
    vr[x] = key_valid ? ld(V, (head + j) * D + g * C + x) : 0.f;
    dk[x] = 0.f;
    dvv[x] = 0.f;
  }

  for (int n = 0; n < unit.z; ++n) {
    const int4 e = p.u_entries[unit.y + n];
    const bool gathered = (e.y & kEntryGathered) != 0;
    const int kind = (e.y >> kKindShift) & 3;
    __syncthreads();
    for (int t = threadIdx.x; t < kBwdRows * D; t += blockDim.x) {
      const int r = t / D, c = t % D;
      const int a = e.x + r;
      long long i = -1;
      if (gathered) {
        if (a < m.n_global) i = m.gpos[a];
      } else if (a < T && !m.rowglobal[a]) {
        i = a;  // global rows are summed by their dense walk only
      }
      const int s = r * Cfg::kRowStride + (c / C) * (C + 4) + c % C;
      sq[s] = i >= 0 ? ld(Q, (head + i) * D + c) : 0.f;
      sdo[s] = i >= 0 ? ld(dO, (head + i) * D + c) : 0.f;
      if (c == 0) {
        srow[r] = static_cast<int>(i);
        slse[r] = i >= 0 ? p.LSE[head + i] : 0.f;
        sdv[r] = i >= 0 ? p.Dvec[head + i] : 0.f;
      }
    }
    __syncthreads();
#pragma unroll 1
    for (int r = 0; r < kBwdRows; ++r) {
      const int i = srow[r];
      if (i < 0) continue;  // block-uniform
      const float* q = sq + r * Cfg::kRowStride + g * (C + 4);
      const float* go = sdo + r * Cfg::kRowStride + g * (C + 4);
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int x = 0; x < C; ++x) {
        s = fmaf(q[x], kr[x], s);
        dp = fmaf(go[x], vr[x], dp);
      }
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      dp += __shfl_xor_sync(0xffffffffu, dp, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      dp += __shfl_xor_sync(0xffffffffu, dp, 2);
      bool ok = key_valid;
      if (ok) {
        if (kind == kKindPacked) ok = key >= e.z && key < e.w;
        else if (kind == kKindDense) ok = !m.causal || j <= i;
        else if (kind == kKindRandom) ok = random_allowed(m, p.colmask, i, j);
        else ok = band_allowed(m, p.colmask, i, j);
      }
      const float pij = ok ? expf(s * p.scale - slse[r]) : 0.f;
      const float ds = pij * (dp - sdv[r]);
#pragma unroll
      for (int x = 0; x < C; ++x) {
        dvv[x] = fmaf(pij, go[x], dvv[x]);
        dk[x] = fmaf(ds, q[x], dk[x]);
      }
    }
  }

  if (!key_valid) return;
  if (packed_unit) {
    const long long o = (static_cast<long long>(bh) * p.n_cols + key) * D + g * C;
#pragma unroll
    for (int x = 0; x < C; ++x) {
      p.dKc[o + x] = dk[x];
      p.dVc[o + x] = dvv[x];
    }
    return;
  }
  const int c = p.n_cols ? p.colidx[j] : -1;
  if (c >= 0) {
    const long long o = (static_cast<long long>(bh) * p.n_cols + c) * D + g * C;
#pragma unroll
    for (int x = 0; x < C; ++x) {
      dk[x] += p.dKc[o + x];
      dvv[x] += p.dVc[o + x];
    }
  }
  In* dK = static_cast<In*>(p.dK);
  In* dV = static_cast<In*>(p.dV);
#pragma unroll
  for (int x = 0; x < C; ++x) {
    st(dK, (head + j) * D + g * C + x, dk[x] * p.scale);
    st(dV, (head + j) * D + g * C + x, dvv[x]);
  }
}

template <typename In, int D>
cudaError_t launch_typed(const BwdArgs& a, cudaStream_t st, bool with_dq, bool with_dkdv) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(dq_kernel<In, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    DqCfg<D>::kSmemBytes);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(dkdv_kernel<In, D>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      KvCfg<D>::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const long long rows = static_cast<long long>(a.BH) * a.mask.T;
  const long long rb = (rows + kWarps - 1) / kWarps;
  rowdot_kernel<In, D><<<static_cast<unsigned>(rb), kThreads, 0, st>>>(
      static_cast<const In*>(a.O), static_cast<const In*>(a.dO), a.Dvec, rows);
  if (with_dq && a.n_q_items > 0)
    dq_kernel<In, D><<<dim3(a.n_q_items, a.BH), kThreads, DqCfg<D>::kSmemBytes, st>>>(a);
  if (!with_dkdv) return cudaGetLastError();
  if (a.n_packed_units > 0)
    dkdv_kernel<In, D><<<dim3(a.n_packed_units, a.BH), kThreads, KvCfg<D>::kSmemBytes, st>>>(a, 0);
  const int nat = a.n_units - a.n_packed_units;
  if (nat > 0)
    dkdv_kernel<In, D><<<dim3(nat, a.BH), kThreads, KvCfg<D>::kSmemBytes, st>>>(a, a.n_packed_units);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_simt(int d, const BwdArgs& a, cudaStream_t st, bool with_dq,
                            bool with_dkdv) {
  if (a.bf16) {
    if (d == 64) return launch_typed<__nv_bfloat16, 64>(a, st, with_dq, with_dkdv);
    if (d == 128) return launch_typed<__nv_bfloat16, 128>(a, st, with_dq, with_dkdv);
  } else {
    if (d == 64) return launch_typed<float, 64>(a, st, with_dq, with_dkdv);
    if (d == 128) return launch_typed<float, 128>(a, st, with_dq, with_dkdv);
  }
  return cudaErrorInvalidValue;
}

}  // namespace spattn
