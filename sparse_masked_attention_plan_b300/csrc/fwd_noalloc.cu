// fwd_noalloc.cu -- the forward pass for callers that cannot allocate device memory.
//
// spattn_fwd packs the strided / global key columns (and the global query rows)
// into scratch that the plan allocates with cudaMalloc on first use.  Some callers
// cannot allow that: a process whose device memory is entirely owned by another
// allocator (a framework's caching allocator that has already reserved the GPU), or
// a latency-critical loop where a cudaMalloc -- which may synchronise the device or
// fail under memory pressure -- must never happen after start-up.  This entry point
// runs the same kernels but takes its packing scratch from one fixed array in the
// library's own device memory, so it allocates nothing.
//
// The array is a file-scope __device__ object of kStaticScratchBytes.  Every GPU
// that loads the library holds it until the process exits.  In host code its name
// is only a stand-in for the symbol, not a device address: the first call on each
// device looks the address up with cudaGetSymbolAddress (with that device current)
// and caches it with the context it belongs to (a call in a new context on that device
// looks it up again); that first call should therefore come before any stream capture.
// All calls share the one array and it keeps the last call's contents; nothing in
// it has to start at zero, because the packing kernel overwrites every byte the
// forward kernel reads.  Two calls whose work overlaps on the GPU (different
// streams, no ordering between them) race on the array and give wrong results.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "spattn.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// The array's device address per device, remembered together with the CUDA context
// it was looked up in: a new context on the device (after cudaDeviceReset, or when the
// primary context was released and made again) loads the module afresh, and the
// array may then sit at another address, so the lookup is repeated.
struct AddrCache {
  CUcontext ctx;
  void* addr;
};
std::mutex g_addr_mu;
AddrCache g_addr[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
  });
  return fn;
}

// Device address of g_static_scratch on `dev` (the current device) in the current
// context, looked up once per (device, context).
cudaError_t static_scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_addr_mu);
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CUcontext ctx = nullptr;
  CtxGetCurrentFn get = ctx_get_current();
  if (!get || get(&ctx) != CUDA_SUCCESS) return cudaErrorInitializationError;
  if (!g_addr[dev].addr || g_addr[dev].ctx != ctx) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = {ctx, p};
  }
  *out = g_addr[dev].addr;
  return cudaSuccess;
}

spattn_status err(spattn_status s, const char* msg) {
  spattn::set_last_error(msg);
  return s;
}

}  // namespace

extern "C" spattn_status spattn_fwd_static_scratch(const spattn_plan* p, int32_t B, int32_t H,
                                                   spattn_dtype dtype, const void* Q,
                                                   const void* K, const void* V, float scale,
                                                   void* O, float* LSE, void* cuda_stream) {
  if (!p) return err(SPATTN_ERR_NULL, "plan is NULL");
  if (!Q || !K || !V || !O) return err(SPATTN_ERR_NULL, "Q, K, V or O is NULL");
  for (const void* x : {Q, K, V, static_cast<const void*>(O)})
    if (reinterpret_cast<uintptr_t>(x) % 16 != 0)
      return err(SPATTN_ERR_ALIGN, "Q, K, V and O must be 16-byte aligned");
  if (LSE && reinterpret_cast<uintptr_t>(LSE) % 4) return err(SPATTN_ERR_ALIGN, "LSE misaligned");
  if (B < 1 || H < 1) return err(SPATTN_ERR_SHAPE, "B and H must be >= 1");
  const int64_t BH = int64_t(B) * H;
  if (BH > 65535) return err(SPATTN_ERR_SHAPE, "B*H exceeds 65535");
  if (dtype != SPATTN_BF16 && dtype != SPATTN_FP32) return err(SPATTN_ERR_DTYPE, "unknown dtype");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return err(SPATTN_ERR_INVALID_SPEC, "scale must be positive and finite");
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  const int esize = dtype == SPATTN_BF16 ? 2 : 4;
  const int64_t ng = static_cast<int64_t>(p->gpos.size());
  const size_t row_bytes = size_t(p->d) * esize;
  const size_t kc_bytes = size_t(BH) * p->n_cols * row_bytes;
  const size_t qg_bytes = size_t(BH) * ng * row_bytes;
  const size_t need = 2 * kc_bytes + qg_bytes;
  if (need > kStaticScratchBytes)
    return err(SPATTN_ERR_SHAPE,
               "packing scratch for this plan and B*H exceeds the 16 MiB static array; "
               "use spattn_fwd (which allocates) or a smaller B*H per call");
  uint8_t* base = nullptr;
  if (need) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = static_scratch_address(dev, reinterpret_cast<void**>(&base));
    if (e != cudaSuccess) return err(SPATTN_ERR_CUDA, cudaGetErrorString(e));
    e = spattn::launch_pack(Q, K, V, base, base + kc_bytes, base + 2 * kc_bytes, p->d_cols,
                            p->n_cols, p->d_gpos, static_cast<int32_t>(ng), BH, p->T,
                            static_cast<int32_t>(row_bytes), stream);
    if (e != cudaSuccess) return err(SPATTN_ERR_CUDA, cudaGetErrorString(e));
  }
  // the same launch arguments as spattn_fwd (test hooks and wait budget included),
  // with the packing scratch in the static array
  spattn::TcArgs a;
  spattn::fill_fwd_args(p, dtype == SPATTN_BF16, BH, Q, K, V, base, base ? base + kc_bytes : nullptr,
                        base ? base + 2 * kc_bytes : nullptr, O, LSE, scale, &a);
  cudaError_t e;
  if (dtype == SPATTN_BF16) {
    const char* why = "";
    e = spattn::launch_fwd_tc(p->d, a, stream, &why);
  } else {
    e = spattn::launch_fwd_simt(p->d, a, stream);
  }
  if (e != cudaSuccess) return err(SPATTN_ERR_CUDA, cudaGetErrorString(e));
  return SPATTN_OK;
}
