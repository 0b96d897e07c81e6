// internal.h -- library-internal types shared by the host API and the kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

namespace spattn {

constexpr int kTile = 128;  // BM = BN of the natural grid

// Entry flag layout (see spattn_plan_copy_schedule in spattn.h).
constexpr int kActive0 = 1, kActive1 = 2, kFull0 = 4, kFull1 = 8;
constexpr int kKindShift = 4;
constexpr int kKindBand = 0, kKindPacked = 1, kKindDense = 2, kKindRandom = 3;
constexpr int kItemGathered = 1;
// A gathered item whose global rows fit in one query tile: both query tiles hold the
// same rows and walk alternate key tiles (entry n is active for tile n % 2 only); the
// two partial softmax states are merged at the end.
constexpr int kItemSplit = 2;

// Key-major (backward) schedule: a unit is 64 consecutive keys, either natural key
// rows (k0 .. k0+63) or packed sparse columns (C[c0] .. C[c0+63]); its entries are
// 64-row query groups {q0, flags, a, b} with the entry kind in the same bits as above
// and kEntryGathered set when q0 indexes the global rows.  Packed entries read packed
// columns [a, b) of the unit.
constexpr int kBwdRows = 64, kBwdKeys = 64;
constexpr int kUnitPacked = 1;
constexpr int kEntryGathered = 1;
// Set on band entries whose local window alone allows every (row, key) pair of the
// group's rows and the unit's keys: the kernels skip the per-key mask words.
constexpr int kEntryFull = 2;

// Device error word bits.
constexpr int kErrTimeout = 1;

// Normalised mask, as the kernels see it.  T <= 2^30, so rows and columns fit int32.
struct MaskDev {
  int32_t T;
  int32_t causal;
  int32_t window;  // causal local width, 0 = none
  int32_t radius;  // bidirectional radius, -1 = none
  int32_t dilation;  // local keys every dilation-th position (1 = contiguous)
  int32_t stride;  // 0 = none
  int32_t offset;
  int32_t n_global;
  int32_t n_gns;               // globals that are not strided columns
  const int32_t* gpos;         // sorted distinct global positions [n_global]
  const int32_t* gpos_ns;      // sorted globals that are not strided [n_gns]
  const uint8_t* rowglobal;    // [T] 1 where the row is a global token
  int32_t rand_block;          // random-block size b (0: no random blocks)
  const int32_t* r_off;        // [ceil(T/b) + 1] random key blocks of query block q:
  const int32_t* r_kb;         //   r_kb[r_off[q] .. r_off[q+1]), ascending
};

struct Schedule {
  int32_t group_rows = 0;  // query rows per work item
  int32_t qtile_rows = 0;  // rows per query tile
  int32_t n_qtiles = 0;    // query tiles per work item
  std::vector<int32_t> items;    // 4 per item, launch order
  std::vector<int32_t> entries;  // 4 per entry
  int4* d_items = nullptr;
  int4* d_entries = nullptr;
  int64_t tile_products = 0;  // (query tile x key tile) products per (batch, head)
  int32_t n_major = 0;        // leading items (>= 1.5x the median length) launched first
  int32_t n_packed_units = 0;  // key-major schedule: packed units come first
  // forward at d = 64: fewer than 80 % of the (entry, query tile) slots are products
  // (entries that one query tile skips, e.g. random blocks): the kernel with one
  // MMA-issuing warp per query tile is then faster than the one-warp issue order
  int32_t mma_per_tile = 0;
};

}  // namespace spattn

struct spattn_plan {
  // normalised spec
  int32_t causal = 1;
  int64_t window = 0, radius = -1, stride = 0, offset = 0, dilation = 1;
  int64_t T = 0;
  int32_t d = 0;
  int device = 0;
  std::vector<int32_t> gpos;     // sorted distinct
  std::vector<int32_t> gpos_ns;  // globals that are not strided columns
  // random blocks (BigBird): block size and, per query block, its key blocks (CSR)
  int32_t rand_block = 0;
  std::vector<int32_t> r_off, r_kb;
  int32_t* d_roff = nullptr;
  int32_t* d_rkb = nullptr;
  // natural grid
  int32_t nqb = 0, nkb = 0;
  int64_t pairs = 0, n_full = 0, n_partial = 0, n_empty = 0, n_nonempty = 0;
  int32_t* d_tile_qb = nullptr;
  int32_t* d_tile_kb = nullptr;
  int32_t* d_tile_cnt = nullptr;
  uint8_t* d_tile_cls = nullptr;
  // sparse columns
  int32_t n_cols = 0;
  std::vector<int32_t> cols;  // host copy of the compacted columns
  int32_t* d_cols = nullptr;
  uint32_t* d_colmask = nullptr;  // [nkb][4] bit c: column kb*128+c is strided or global
  uint8_t* d_rowglobal = nullptr;
  int32_t* d_gpos = nullptr;
  int32_t* d_gpos_ns = nullptr;
  // execution schedules: [0] tensor-core bf16 kernel, [1] fp32 kernel, [2] the
  // tensor-core kernel on the residue classes of a dilated window (when dview > 1)
  spattn::Schedule sched[3];
  // Dilated view: with dilation d > 1, no strided or global columns and d | T, the
  // window is d independent contiguous windows, one per residue class r of the rows
  // (positions r, r + d, ...); the bf16 kernel then walks sched[2] over T / d rows.
  int32_t dview = 1;
  uint32_t* d_colmask_res = nullptr;  // all zero: no strided / global columns
  uint8_t* d_rowzero = nullptr;       // no global rows
  // key-major schedule of the backward pass and the packed index of every key
  // (-1 where the key is not a sparse column)
  spattn::Schedule bsched;     // 64-key units, 64-row groups (FP32-unit kernels)
  spattn::Schedule bsched_tc;  // 128-key units, 128-row groups (tensor-core kernel)
  spattn::Schedule bsched_res;  // the same over the residue classes of a dilated view
  int32_t* d_colidx = nullptr;
  // random blocks transposed (key block -> query blocks), for the key-major kernels
  std::vector<int32_t> rt_off, rt_qb;
  int32_t* d_rtoff = nullptr;
  int32_t* d_rtqb = nullptr;
  // packing scratch (packed K, V of the sparse columns and gathered global-row Q)
  void* d_scratch = nullptr;
  size_t scratch_bytes = 0;
  // backward scratch: row dots D_i [BH][T] and packed-column dK, dV [BH][|C|][d], fp32
  void* d_bscratch = nullptr;
  size_t bscratch_bytes = 0;
  // debug walk counter and device error word
  unsigned long long* d_walk = nullptr;
  int32_t walk_enabled = 0;
  int* d_err = nullptr;
  uint64_t wait_budget_cycles = 8000000000ull;  // ~4 s at the maximum SM clock
  int32_t inject_timeout = 0;                     // test hook, see spattn_plan_test_wait_timeout
  // spattn_fwd_host: a copy-in and a copy-out stream and the per-chunk events of its
  // pipeline (host -> device of chunk k+1, forward of chunk k, device -> host of chunk
  // k-1), created on first use on the plan's device
  static constexpr int kHostChunks = 16;
  cudaStream_t host_in = nullptr, host_out = nullptr;
  cudaEvent_t host_ev[2 * kHostChunks + 2] = {};

  spattn::MaskDev mask_dev() const {
    spattn::MaskDev m;
    m.T = static_cast<int32_t>(T);
    m.causal = causal;
    m.window = static_cast<int32_t>(window);
    m.radius = static_cast<int32_t>(radius);
    m.dilation = static_cast<int32_t>(dilation);
    m.stride = static_cast<int32_t>(stride);
    m.offset = static_cast<int32_t>(offset);
    m.n_global = static_cast<int32_t>(gpos.size());
    m.n_gns = static_cast<int32_t>(gpos_ns.size());
    m.gpos = d_gpos;
    m.gpos_ns = d_gpos_ns;
    m.rowglobal = d_rowglobal;
    m.rand_block = rand_block;
    m.r_off = d_roff;
    m.r_kb = d_rkb;
    return m;
  }

  // The mask as the bf16 kernel sees it in the dilated view: T / d rows, contiguous.
  spattn::MaskDev mask_dev_res() const {
    spattn::MaskDev m = mask_dev();
    m.T = static_cast<int32_t>(T / dview);
    m.dilation = 1;
    m.rowglobal = d_rowzero;
    return m;
  }
};

// ---- launchers implemented in the .cu files (host side, return cudaError_t) ----
namespace spattn {

// plan_kernels.cu
cudaError_t launch_column_flags(const MaskDev& m, uint8_t* flags, uint8_t* rowglobal,
                                cudaStream_t st);
cudaError_t launch_compact_columns(const uint8_t* flags, int32_t T, int32_t* cols,
                                   int32_t* n_cols, cudaStream_t st);
cudaError_t launch_colmask(const uint8_t* flags, int32_t T, int32_t nkb, uint32_t* colmask,
                           cudaStream_t st);
cudaError_t launch_tile_count(const MaskDev& m, const uint32_t* colmask, int32_t nqb,
                              int32_t nkb, int32_t* q_nonempty, int32_t* q_full,
                              long long* q_pairs, cudaStream_t st);
cudaError_t launch_tile_fill(const MaskDev& m, const uint32_t* colmask, int32_t nqb,
                             int32_t nkb, const int32_t* q_offset, int32_t* tile_qb,
                             int32_t* tile_kb, int32_t* tile_cnt, uint8_t* tile_cls,
                             cudaStream_t st);

// pack_kernel.cu: gathers rows of K and V at `cols` and rows of Q at `gpos`.
cudaError_t launch_pack(const void* Q, const void* K, const void* V, void* Kc, void* Vc,
                        void* Qg, const int32_t* cols, int32_t n_cols, const int32_t* gpos,
                        int32_t n_global, int64_t BH, int64_t T, int32_t row_bytes,
                        cudaStream_t st);

// fwd_tc.cu (bf16 tensor-core forward)
struct TcArgs {
  const void* Q;
  const void* K;
  const void* V;
  const void* Kc;
  const void* Vc;
  const void* Qg;
  void* O;
  float* LSE;
  int32_t BH;
  int32_t n_cols;
  float scale;
  const uint32_t* colmask;
  MaskDev mask;
  const int4* items;
  const int4* entries;
  int32_t n_items;
  unsigned long long* walk;
  int* err;
  uint64_t wait_budget_cycles;
  int32_t inject_timeout = 0;
  int32_t n_major = 0;
  int32_t dview = 1;  // residue classes of a dilated view (mask.T is then T / dview)
  int32_t mma_per_tile = 0;  // see Schedule::mma_per_tile
};
cudaError_t launch_fwd_tc(int d, const TcArgs& a, cudaStream_t st, const char** why);

// fwd_simt.cu (fp32 forward)
cudaError_t launch_fwd_simt(int d, const TcArgs& a, cudaStream_t st);

// bwd_simt.cu (backward on the FP32 FMA units, bf16 or fp32 inputs)
struct BwdArgs {
  const void* Q;
  const void* K;
  const void* V;
  const void* O;
  const float* LSE;
  const void* dO;
  void* dQ;
  void* dK;
  void* dV;
  float* Dvec;    // [BH][T] scratch
  float* dKc;     // [BH][n_cols][d] scratch
  float* dVc;
  int32_t BH;
  int32_t n_cols;
  float scale;
  int32_t bf16;
  const int32_t* cols;
  const int32_t* colidx;
  const uint32_t* colmask;
  MaskDev mask;
  // query-major walk (dQ): the fp32 forward schedule
  const int4* q_items;
  const int4* q_entries;
  int32_t n_q_items;
  // key-major walk (dK, dV)
  const int4* units;
  const int4* u_entries;
  int32_t n_packed_units;
  int32_t n_units;
};
// The row dots D_i always; dQ and dK/dV unless the tensor-core kernels take them.
cudaError_t launch_bwd_simt(int d, const BwdArgs& a, cudaStream_t st, bool with_dq = true,
                            bool with_dkdv = true);

// bwd_tc.cu (bf16 dQ on the tensor cores; walks the tensor-core forward schedule)
struct BwdTcArgs {
  const void* Q;
  const void* K;
  const void* V;
  const void* dO;
  const void* Kc;   // packed sparse-column K, V rows [BH][n_cols][d]
  const void* Vc;
  const void* Qg;   // gathered global-row Q, dO rows [BH][n_global][d]
  const void* dOg;
  void* dQ;
  const float* LSE;
  const float* Dvec;
  int32_t BH;
  int32_t n_cols;
  float scale;
  const uint32_t* colmask;
  MaskDev mask;
  const int4* items;
  const int4* entries;
  int32_t n_items;
  int* err;
  uint64_t wait_budget_cycles;
  // key-major dK / dV
  void* dK;
  void* dV;
  float* dKc;
  float* dVc;
  const int32_t* cols;
  const int32_t* colidx;
  const int32_t* rt_off;
  const int32_t* rt_qb;
  const int4* units;
  const int4* u_entries;
  int32_t n_packed_units;
  int32_t n_units;
  int32_t dview = 1;  // residue classes of a dilated view (mask.T is then T / dview)
};
cudaError_t launch_bwd_dq_tc(int d, const BwdTcArgs& a, cudaStream_t st, const char** why);
cudaError_t launch_bwd_dkdv_tc(int d, const BwdTcArgs& a, cudaStream_t st, const char** why);

// decode.cu (one generation step against a ring-buffer KV cache)
struct DecodeArgs {
  const void* q;
  const void* Kc;
  const void* Vc;
  const int64_t* pos;
  void* out;
  float* lse;
  float* part;  // [B*Hq][nsplit][d + 2] scratch
  int* err;
  int32_t B, Hq, Hkv, d, nsplit, bf16;
  int64_t cap, window;
  float scale;
  const void* kn = nullptr;  // bf16 only: the step's own rows, appended by the kernel
  const void* vn = nullptr;
};
int decode_splits(int64_t B, int64_t Hkv, int64_t cap);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_kv_append(bool bf16, void* Kc, void* Vc, const void* kn, const void* vn,
                             const int64_t* pos, int32_t B, int32_t Hkv, int64_t cap, int32_t d,
                             cudaStream_t st);

// spattn_api.cu: schedule, mask view and column data a forward launch of `dtype` uses.
void select_schedule(const spattn_plan* p, bool bf16, TcArgs* a);

// spattn_api.cu: every field of a forward launch's arguments from the plan, the
// caller's buffers and the packing scratch (Kc, Vc, Qg; NULL when nothing is packed),
// the schedule included.  Both forward entry points fill their launches with it.
void fill_fwd_args(const spattn_plan* p, bool bf16, int64_t BH, const void* Q, const void* K,
                   const void* V, void* Kc, void* Vc, void* Qg, void* O, float* LSE, float scale,
                   TcArgs* a);

// spattn_api.cu: set the calling thread's spattn_last_error() message.
void set_last_error(const char* msg);

}  // namespace spattn
