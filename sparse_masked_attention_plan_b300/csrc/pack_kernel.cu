// pack_kernel.cu -- gathers the rows the compacted tiles need into dense buffers.
//
// Strided and global key columns outside a query group's band are read through
// packed copies Kc[bh][p] = K[bh][C[p]], Vc[bh][p] = V[bh][C[p]], so that the
// forward kernel can stream them with TMA like any other key tile.  Global query
// rows (which read every key: "Attention variants", sreshtalluri.github.io,
// section 4, with_global) are gathered into Qg[bh][a] = Q[bh][G[a]].  Pure data
// movement: 16-byte vector loads and stores, grid-stride over all rows.
#include <cuda_runtime.h>

#include "internal.h"

namespace spattn {
namespace {

__global__ void __launch_bounds__(256) k_pack(const uint4* __restrict__ Q,
                                              const uint4* __restrict__ K,
                                              const uint4* __restrict__ V, uint4* __restrict__ Kc,
                                              uint4* __restrict__ Vc, uint4* __restrict__ Qg,
                                              const int32_t* __restrict__ cols, int n_cols,
                                              const int32_t* __restrict__ gpos, int n_global,
                                              long long BH, long long T, int vec_per_row) {
  const long long rows_per_bh = 2LL * n_cols + n_global;
  const long long total = BH * rows_per_bh * vec_per_row;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const int v = static_cast<int>(t % vec_per_row);
    const long long r = t / vec_per_row;
    const long long bh = r / rows_per_bh;
    const int k = static_cast<int>(r % rows_per_bh);
    if (k < n_cols) {
      const long long src = (bh * T + cols[k]) * vec_per_row + v;
      Kc[(bh * n_cols + k) * vec_per_row + v] = K[src];
    } else if (k < 2 * n_cols) {
      const int p = k - n_cols;
      const long long src = (bh * T + cols[p]) * vec_per_row + v;
      Vc[(bh * n_cols + p) * vec_per_row + v] = V[src];
    } else {
      const int a = k - 2 * n_cols;
      const long long src = (bh * T + gpos[a]) * vec_per_row + v;
      Qg[(bh * n_global + a) * vec_per_row + v] = Q[src];
    }
  }
}

}  // namespace

cudaError_t launch_pack(const void* Q, const void* K, const void* V, void* Kc, void* Vc,
                        void* Qg, const int32_t* cols, int32_t n_cols, const int32_t* gpos,
                        int32_t n_global, int64_t BH, int64_t T, int32_t row_bytes,
                        cudaStream_t st) {
  const int vec = row_bytes / 16;
  const long long total = BH * (2LL * n_cols + n_global) * vec;
  if (total == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (total + 255) / 256;
  if (blocks > 8LL * sms) blocks = 8LL * sms;
  k_pack<<<static_cast<int>(blocks), 256, 0, st>>>(
      static_cast<const uint4*>(Q), static_cast<const uint4*>(K), static_cast<const uint4*>(V),
      static_cast<uint4*>(Kc), static_cast<uint4*>(Vc), static_cast<uint4*>(Qg), cols, n_cols,
      gpos, n_global, BH, T, vec);
  return cudaGetLastError();
}

}  // namespace spattn
