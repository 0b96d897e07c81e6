// fwd_tc.cu -- bf16 forward pass of block-sparse masked attention on the fifth-
// generation tensor cores (tcgen05) of sm_103a.
//
// What it computes, per (batch, head) and query row i with allowed set S_i:
//     y_i = sum_{j in S_i} softmax_j(scale q_i.k_j) v_j,  LSE_i = ln sum exp(...)
// with the softmax normalised over S_i only ("Sparse attention" glossary,
// glossary.selfmadequant.com, section "Choose the available reads", the displayed
// equation).  Only the schedule's tiles are computed: band tiles of the natural
// 128 x 128 grid and packed tiles of strided / global columns; empty tiles are never
// loaded ("Attention variants", sreshtalluri.github.io, section "Use the library":
// block-level skipping; "Sparse attention" glossary, "When the cost is linear":
// block computation that skips excluded regions).
//
// One CTA = one work item = two 128-row query tiles of one (batch, head) sharing a
// stream of key/value tiles.  Warp roles (320 threads):
//   warps 0-3  softmax + correction + epilogue for query tile 0 (TMEM lanes 0-127)
//   warps 4-7  the same for query tile 1
//   warp 8     TMA producer: Q tiles once, then K and V tiles into a ring of slots
//   warp 9     MMA issuer (one thread): S_t = Q_t K^T and O_t += P_t V, tcgen05
//              (d = 64 schedules whose entries are often read by one query tile only:
//              warps 9 and 10, one per query tile, 352 threads)
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+d), O1 [256+d,256+2d);
// P_t (bf16) overwrites the first 64 columns of S_t and feeds the PV product directly
// from TMEM.  The MMA issue order
//     S0(n), PV1(n-1), S1(n), PV0(n)
// lets the softmax of one query tile overlap the other tile's two products.
// Online softmax in fp32 with the exp2 form and a conditional rescale: the running
// maximum moves (and O is rescaled) only when a row maximum grows by more than
// 2^8; the final O / l and LSE use the same stale maximum, so the result is exact.
// One thread owns one query row (its TMEM lane), so row max and row sum need no
// cross-thread reduction.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "predicate.cuh"
#include "ptx.cuh"
#include "tmap.h"

namespace spattn {
namespace {

constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;  // with two MMA warps: warps 9 and 10 for query tile 0, 1
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D, int MW = 1>
struct TcCfg {
  static constexpr int kChunkBytes = kTile * 64 * 2;  // 128 rows x 64 bf16, one swizzle span
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStages = D == 128 ? 4 : 8;
  static constexpr int kSmemQ = 2 * kTileBytes;
  static constexpr int kSmemKV = kStages * kTileBytes;
  // barriers: full[S], empty[S], q_full, s_full[2], p_full[2], o_final, and one that
  // nothing ever arrives on (the wait-timeout test waits on it)
  static constexpr int kBarFull = 0, kBarEmpty = kStages, kBarQ = 2 * kStages,
                       kBarS = 2 * kStages + 1, kBarP = 2 * kStages + 3,
                       kBarO = 2 * kStages + 5, kBarNever = 2 * kStages + 6,
                       kNumBars = 2 * kStages + 7;
  // split items: the two query tiles' row maxima and sums, [tile][2][row] fp32
  static constexpr int kSmemX = 2 * 2 * kTile * 4;
  static constexpr int kSmemBytes = kSmemQ + kSmemKV + kSmemX + kNumBars * 8 + 16 + 1024;
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 0, 1);
  // TMEM: S_t [128t, 128t+128), P_t (bf16) over the first 64 columns of S_t, O_t at
  // 256 + d t.  (At d = 64 a layout with P_t in columns of its own, so that the next S_t
  // could be computed while the softmax works, was measured slower on the 16K-token
  // workload: 0.219 against 0.213 ms.)
  static constexpr uint32_t kColS0 = 0, kColS1 = 128;  // S of query tile 0, 1
  static constexpr uint32_t kColP0 = kColS0, kColP1 = kColS1;
  static constexpr uint32_t kColO0 = 256, kColO1 = 256 + D;
  // MW = 2 (d = 64, for schedules in which many entries are read by one query tile
  // only): one MMA-issuing warp per query tile, each running its tile's chain (S, then
  // PV once P is in TMEM) without waiting on the other tile's hand-offs; K/V slots are
  // released by both warps.  With one warp the fixed order S0(n), PV1(n-1), S1(n), PV0(n)
  // staggers the tiles, which is faster when both read every entry.
  static constexpr int kMmaWarps = MW;
  static constexpr int kThreads = 32 * (kMmaWarp + MW);
};

struct KParams {
  __nv_bfloat16* O;
  float* LSE;
  float scale_log2;
  const uint32_t* colmask;
  MaskDev mask;
  const int4* items;
  const int4* entries;
  unsigned long long* walk;
  int* err;
  uint64_t budget;
  int inject_timeout;  // test hook: the MMA warp first waits on a barrier nobody signals
  int BH;        // work units along the head axis: (batch, head) x residue classes
  int n_items;
  int n_major;  // leading (longest) items launched for every head before the rest
  int dview;    // residue classes of a dilated view (1: rows are the sequence itself)
  int T_out;    // sequence length of O and LSE (the mask's T times dview)
};

// Descriptors are built once per operand base; a k-step only adds its byte offset
// / 16 to the start-address field (bits 0-13), which cannot carry out because
// shared-memory addresses stay below 2^18.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
  using C = TcCfg<D>;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off16 = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
    mma_ss(d_tmem, q_desc + off16, k_desc + off16, C::kIdescQK, kk > 0 ? 1u : 0u);
  }
}

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc,
                                         bool accumulate) {
  using C = TcCfg<D>;
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk)
    mma_ts(d_tmem, p_tmem + kk * 8, v_desc + ((kk * 16 * 128) >> 4), C::kIdescPV,
           (accumulate || kk > 0) ? 1u : 0u);
}

template <int D, int MW>
__global__ void __launch_bounds__(TcCfg<D, MW>::kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmQg,
                  const __grid_constant__ CUtensorMap tmKc, const __grid_constant__ CUtensorMap tmVc,
                  const KParams p) {
  using C = TcCfg<D, MW>;
  static_assert(C::kIdescQK == TcCfg<D>::kIdescQK && C::kIdescPV == TcCfg<D>::kIdescPV,
                "the issue helpers use the one-warp configuration's shapes");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_addr(smem);
  const uint32_t sKV = sQ + C::kSmemQ;
  float* xch = reinterpret_cast<float*>(smem + C::kSmemQ + C::kSmemKV);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kSmemQ + C::kSmemKV + C::kSmemX);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  const uint32_t bar0 = smem_addr(bars);
#define BAR(k) (bar0 + 8u * static_cast<uint32_t>(k))

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Launch order: the n_major longest items for every (batch, head) first (rank-major,
  // longest first), then the rest head by head (neighbouring query groups of one head
  // share K/V tiles in L2).
  int rank, bh;
  {
    const int u = blockIdx.x, nm = p.n_major * p.BH;
    if (u < nm) {
      rank = u / p.BH;
      bh = u % p.BH;
    } else {
      const int rest = p.n_items - p.n_major;
      bh = (u - nm) / rest;
      rank = p.n_major + (u - nm) % rest;
    }
  }
  // a unit along the head axis is a (batch, head) and, in a dilated view, a residue
  // class r: its query / key row q is sequence position q * dview + r
  const int res = bh % p.dview;
  bh /= p.dview;
  const int4 item = p.items[rank];
  const int n_ent = item.z;
  const int4* ents = p.entries + item.y;
  const bool gathered = (item.w & kItemGathered) != 0;
  const bool split = (item.w & kItemSplit) != 0;  // both tiles hold the same rows
  const MaskDev& m = p.mask;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(BAR(C::kBarFull + s), 1);
      // one arrival per MMA-issuing warp: a commit after its products read the slot, or a
      // plain arrival (after the slot's copy landed) when its query tile skips the entry
      mbar_init(BAR(C::kBarEmpty + s), C::kMmaWarps);
    }
    mbar_init(BAR(C::kBarQ), 1);
    mbar_init(BAR(C::kBarS + 0), 1);
    mbar_init(BAR(C::kBarS + 1), 1);
    // p_full and s_free: one arrival per softmax warp (a single arrive per warp keeps the
    // hand-off off the critical path: 128 arrivals on one barrier word serialise)
    mbar_init(BAR(C::kBarP + 0), 4);
    mbar_init(BAR(C::kBarP + 1), 4);
    mbar_init(BAR(C::kBarO), C::kMmaWarps);
    mbar_init(BAR(C::kBarNever), 1);
    fence_barrier_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(gathered ? &tmQg : &tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the loop (its values stay warp-uniform); one lane issues.
    const void* mapQ = gathered ? static_cast<const void*>(&tmQg) : static_cast<const void*>(&tmQ);
    if (elect_one()) {
      mbar_arrive_expect_tx(BAR(C::kBarQ), 2 * C::kTileBytes);
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(sQ + t * C::kTileBytes + c * C::kChunkBytes, mapQ, BAR(C::kBarQ), c * 64,
                      res, item.x + (split ? 0 : t * kTile), bh);
    }
    __syncwarp();
    int issued = 0;
    bool ok = true;
    int4 e_next = ents[0];
    for (int n = 0; n < n_ent && ok; ++n) {
      const int4 e = e_next;
      if (n + 1 < n_ent) e_next = ents[n + 1];
      const bool packed = ((e.y >> kKindShift) & 3) == kKindPacked;
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        const int it = 2 * n + kv;
        const int s = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(BAR(C::kBarEmpty + s), ph ^ 1u, p.budget, p.err, kErrTimeout))) {
          ok = false;
          break;
        }
        const void* map = kv ? (packed ? static_cast<const void*>(&tmVc) : static_cast<const void*>(&tmV))
                             : (packed ? static_cast<const void*>(&tmKc) : static_cast<const void*>(&tmK));
        if (elect_one()) {
          mbar_arrive_expect_tx(BAR(C::kBarFull + s), C::kTileBytes);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d(sKV + s * C::kTileBytes + c * C::kChunkBytes, map, BAR(C::kBarFull + s),
                        c * 64, packed ? 0 : res, e.x, bh);
        }
        __syncwarp();
        ++issued;
      }
    }
    // Drain: wait until the last load issued into each slot has landed, so no
    // copy is still writing this CTA's shared memory when it exits.
    for (int it = issued - 1; it >= 0 && it >= issued - C::kStages; --it)
      mbar_wait(BAR(C::kBarFull + it % C::kStages), (it / C::kStages) & 1, p.budget, p.err,
                kErrTimeout);
    mbar_wait(BAR(C::kBarQ), 0, p.budget, p.err, kErrTimeout);  // the Q tiles too
    __syncwarp();
  } else if (warp == kMmaWarp || (C::kMmaWarps == 2 && warp == kMmaWarp + 1)) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and waits; one elected lane (always lane 0 of the
    // converged warp, so commits track its own products) issues MMAs and commits.
    unsigned long long walked = 0;
    const uint64_t q0_desc = smem_desc_sw128(sQ, 16, 1024);
    const uint64_t q1_desc = smem_desc_sw128(sQ + C::kTileBytes, 16, 1024);
    const uint64_t kv_kdesc = smem_desc_sw128(sKV, 16, 1024);  // slot 0 as a K operand
    const uint64_t kv_vdesc = smem_desc_sw128(sKV, C::kChunkBytes, 1024);  // slot 0 as V
    constexpr uint32_t kSlot16 = C::kTileBytes >> 4;
    bool ok = __all_sync(0xffffffffu, !p.inject_timeout ||
                                          mbar_wait(BAR(C::kBarNever), 0, p.budget, p.err, kErrTimeout));
    ok = ok && __all_sync(0xffffffffu, mbar_wait(BAR(C::kBarQ), 0, p.budget, p.err, kErrTimeout));
    if (ok && C::kMmaWarps == 2) {
      // query tile t = warp - 9: S_t(n), then PV_t(n) once P_t(n) is in TMEM (the next
      // S_t overwrites P_t, so it follows in issue order)
      tc_fence_after();
      const int t = warp - kMmaWarp;
      const uint64_t q_desc = t ? q1_desc : q0_desc;
      const uint32_t colS = t ? C::kColS1 : C::kColS0, colO = t ? C::kColO1 : C::kColO0;
      uint32_t pph = 0u;
      bool oinit = false;
      auto wait_full = [&](int it) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(BAR(C::kBarFull + it % C::kStages),
                                                 (it / C::kStages) & 1, p.budget, p.err,
                                                 kErrTimeout));
      };
      auto release = [&](int it, bool used) {  // this warp's arrival on the slot of `it`
        if (elect_one()) {
          if (used) mma_commit(BAR(C::kBarEmpty + it % C::kStages));
          else mbar_arrive(BAR(C::kBarEmpty + it % C::kStages));
        }
        __syncwarp();
      };
      // Each entry's K is checked one entry early, while this tile's softmax runs (it was
      // loaded long before, as a rule): a wait costs the warp a few hundred cycles even
      // when its phase is complete, and between PV(n) and S(n+1) it would lengthen
      // the tile's chain.
      int4 e_next = ents[0];
      if (n_ent > 0 && !wait_full(0)) ok = false;
      for (int n = 0; n < n_ent && ok; ++n) {
        const int4 e = e_next;
        if (n + 1 < n_ent) e_next = ents[n + 1];  // load ahead: global latency off the issue path
        const bool a = (e.y & (kActive0 << t)) != 0;
        const int kit = 2 * n, vit = 2 * n + 1;
        tc_fence_after();
        if (a) {
          if (elect_one()) {
            issue_qk<D>(tmem + colS, q_desc, kv_kdesc + (kit % C::kStages) * kSlot16);
            mma_commit(BAR(C::kBarS + t));
          }
          __syncwarp();
          ++walked;
        }
        release(kit, a);
        if (!wait_full(vit)) { ok = false; break; }
        if (n + 1 < n_ent && !wait_full(kit + 2)) { ok = false; break; }
        tc_fence_after();
        if (a) {
          if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::kBarP + t), pph, p.budget, p.err,
                                                 kErrTimeout))) { ok = false; break; }
          pph ^= 1u;
          tc_fence_after();
          if (elect_one())
            issue_pv<D>(tmem + colO, tmem + colS, kv_vdesc + (vit % C::kStages) * kSlot16, oinit);
          __syncwarp();
          oinit = true;
        }
        release(vit, a);
      }
    } else if (ok) {
      tc_fence_after();
      int pend1 = -1;
      uint32_t pend_vs = 0;
      uint32_t pph[2] = {0u, 0u};
      bool oinit[2] = {false, false};
      // At d = 64 each entry's K is checked one entry early, while tile 0's softmax
      // runs (with eight slots it was loaded long before): a wait costs the warp a few
      // hundred cycles even when its phase is complete, and between PV0(n) and S0(n+1)
      // it lengthens both tiles' chains (16K tokens 1 % faster).  At d = 128 the check
      // stays at the top of the entry (the early one was not faster there).
      constexpr bool kEarlyK = D == 64;
      auto wait_k = [&](int it) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(BAR(C::kBarFull + it % C::kStages),
                                                 (it / C::kStages) & 1, p.budget, p.err,
                                                 kErrTimeout));
      };
      int4 e_next = ents[0];
      if (kEarlyK && n_ent > 0 && !wait_k(0)) ok = false;
      for (int n = 0; ok && n < n_ent; ++n) {
        const int4 e = e_next;
        if (n + 1 < n_ent) e_next = ents[n + 1];  // load ahead: global latency off the issue path
        const bool a0 = (e.y & kActive0) != 0, a1 = (e.y & kActive1) != 0;
        const int kit = 2 * n, vit = 2 * n + 1;
        const uint32_t ks = kit % C::kStages, vs = vit % C::kStages;
        if (!kEarlyK && !wait_k(kit)) { ok = false; break; }
        tc_fence_after();
        const uint64_t k_desc = kv_kdesc + ks * kSlot16;
        if (a0) {
          if (elect_one()) {
            issue_qk<D>(tmem + C::kColS0, q0_desc, k_desc);
            mma_commit(BAR(C::kBarS + 0));
          }
          __syncwarp();
          ++walked;
        }
        if (pend1 >= 0) {
          if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::kBarP + 1), pph[1], p.budget, p.err,
                                                 kErrTimeout))) { ok = false; break; }
          pph[1] ^= 1u;
          tc_fence_after();
          if (elect_one()) {
            issue_pv<D>(tmem + C::kColO1, tmem + C::kColS1, kv_vdesc + pend_vs * kSlot16, oinit[1]);
            mma_commit(BAR(C::kBarEmpty + pend_vs));
          }
          __syncwarp();
          oinit[1] = true;
          pend1 = -1;
        }
        if (a1) {
          if (elect_one()) {
            issue_qk<D>(tmem + C::kColS1, q1_desc, k_desc);
            mma_commit(BAR(C::kBarS + 1));
          }
          __syncwarp();
          ++walked;
        }
        if (elect_one()) mma_commit(BAR(C::kBarEmpty + ks));
        __syncwarp();
        if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::kBarFull + vs), (vit / C::kStages) & 1,
                                               p.budget, p.err, kErrTimeout))) { ok = false; break; }
        if (kEarlyK && n + 1 < n_ent && !wait_k(kit + 2)) { ok = false; break; }
        tc_fence_after();
        if (a0) {
          if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::kBarP + 0), pph[0], p.budget, p.err,
                                                 kErrTimeout))) { ok = false; break; }
          pph[0] ^= 1u;
          tc_fence_after();
          if (elect_one()) issue_pv<D>(tmem + C::kColO0, tmem + C::kColS0, kv_vdesc + vs * kSlot16, oinit[0]);
          __syncwarp();
          oinit[0] = true;
        }
        if (a1) {
          pend1 = n;
          pend_vs = vs;
        } else {
          if (elect_one()) mma_commit(BAR(C::kBarEmpty + vs));
          __syncwarp();
        }
      }
      if (ok && pend1 >= 0) {
        if (__all_sync(0xffffffffu, mbar_wait(BAR(C::kBarP + 1), pph[1], p.budget, p.err, kErrTimeout))) {
          tc_fence_after();
          if (elect_one()) {
            issue_pv<D>(tmem + C::kColO1, tmem + C::kColS1, kv_vdesc + pend_vs * kSlot16, oinit[1]);
            mma_commit(BAR(C::kBarEmpty + pend_vs));
          }
          __syncwarp();
        }
      }
    }
    // Arrives when every product issued above has completed; the epilogue reads
    // O after it, and waiting here keeps TMEM allocated until no product runs.
    if (elect_one()) mma_commit(BAR(C::kBarO));
    __syncwarp();
    mbar_wait(BAR(C::kBarO), 0, p.budget, p.err, kErrTimeout);
    if (lane == 0 && p.walk && walked) atomicAdd(p.walk, walked);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps
    const int wg = warp >> 2;
    const int r = ((warp & 3) << 5) | lane;
    const uint32_t lane_base = tmem + ((static_cast<uint32_t>(warp & 3) * 32u) << 16);
    const uint32_t colS = wg ? C::kColS1 : C::kColS0, colO = wg ? C::kColO1 : C::kColO0;
    const uint32_t colP = wg ? C::kColP1 : C::kColP0;
    const int local = (split ? 0 : wg * kTile) + r;
    int i;
    bool valid;
    if (gathered) {
      const int a = item.x + local;
      valid = a < m.n_global;
      i = valid ? m.gpos[a] : 0;
    } else {
      i = item.x + local;
      valid = i < m.T;
    }
    const float c2 = p.scale_log2;
    float mrow = -INFINITY, lrow = 0.f;
    uint32_t sph = 0;
    int n_done = 0;
    int4 e_next = ents[0];
    for (int n = 0; n < n_ent; ++n) {
      const int4 e = e_next;
      if (n + 1 < n_ent) e_next = ents[n + 1];
      if (!(e.y & (kActive0 << wg))) continue;
      // the row's allowed columns, computed before the wait (they do not depend on S, and
      // the column-mask load overlaps the product)
      const bool partial = !(e.y & (kFull0 << wg));
      uint32_t w[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
      if (partial) row_mask(make_predicate(m, p.colmask, e, i), w);
      const bool got = mbar_wait(BAR(C::kBarS + wg), sph, p.budget, p.err, kErrTimeout);
      if (!__all_sync(0xffffffffu, got)) break;
      sph ^= 1u;
      tc_fence_after();
      // the whole S row of this thread (one TMEM load), masked where not allowed
      uint32_t sr[kTile];
      tmem_ld128(lane_base + colS, sr);
      if (partial) {
#pragma unroll
        for (int c = 0; c < kTile; ++c)
          if (!((w[c >> 5] >> (c & 31)) & 1u)) sr[c] = 0xff800000u;  // -inf
      }
      float mx8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) mx8[j] = __uint_as_float(sr[j]);
#pragma unroll
      for (int c = 8; c + 16 <= kTile; c += 16)  // columns 8..119, two per instruction
#pragma unroll
        for (int j = 0; j < 8; ++j)
          mx8[j] = fmax3(mx8[j], __uint_as_float(sr[c + j]), __uint_as_float(sr[c + 8 + j]));
#pragma unroll
      for (int j = 0; j < 8; ++j) mx8[j] = fmaxf(mx8[j], __uint_as_float(sr[kTile - 8 + j]));
      const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                             fmaxf(mx8[6], mx8[7]));
      const float mcand = fmaxf(mrow, mx * c2);
      const bool need = mcand > mrow + kRescaleThreshold;
      float corr = 1.f;
      if (need) {
        corr = fast_exp2(mrow - mcand);
        mrow = mcand;
        lrow *= corr;
      }
      const float msub = (mrow == -INFINITY) ? 0.f : mrow;
      // P = 2^(s * scale * log2 e - m), stored as bf16 over the first half of S;
      // the scale-and-shift and the row sum run two columns per instruction
      const uint64_t c2x2 = f32x2(c2, c2), nmx2 = f32x2(-msub, -msub);
      uint64_t acc2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int b = 0; b < 16; ++b) {
          const int c0 = 32 * q + 2 * b;
          float x0, x1;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(sr[c0]), __uint_as_float(sr[c0 + 1])), c2x2,
                                nmx2),
                      x0, x1);
          const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          acc2[b & 1] = add_f32x2(acc2[b & 1], f32x2(p0, p1));
          pk[b] = pack_bf16x2(p0, p1);
        }
        tmem_st16(lane_base + colP + 16 * q, pk);
      }
      float s0, s1, s2, s3;
      f32x2_split(acc2[0], s0, s1);
      f32x2_split(acc2[1], s2, s3);
      const float sum = (s0 + s1) + (s2 + s3);
      lrow += sum;
      if (n_done > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(lane_base + colO + 32 * q, o);
#pragma unroll
          for (int b = 0; b < 32; ++b) o[b] = __float_as_uint(__uint_as_float(o[b]) * corr);
          tmem_st32(lane_base + colO + 32 * q, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();  // every lane's P and O stores are complete before lane 0 arrives
      if (lane == 0) mbar_arrive(BAR(C::kBarP + wg));
      ++n_done;
    }
    // ---------------------------------------------------------- epilogue
    if (split) {
      // both tiles walked alternate key tiles for the same rows: merge the two partial
      // states, m = max(m0, m1), l = l0 2^(m0 - m) + l1 2^(m1 - m), O likewise; tile t's
      // thread of row r writes columns t d / 2 .. of the row (both O_t are in its lanes)
      xch[wg * 2 * kTile + r] = mrow;
      xch[wg * 2 * kTile + kTile + r] = lrow;
      bar_sync(1, 256);
      const float m0 = xch[r], l0 = xch[kTile + r];
      const float m1 = xch[2 * kTile + r], l1 = xch[3 * kTile + r];
      const float mm = fmaxf(m0, m1);
      const float a0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - mm);
      const float a1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - mm);
      const float lsum = l0 * a0 + l1 * a1;
      const bool got = mbar_wait(BAR(C::kBarO), 0, p.budget, p.err, kErrTimeout);
      if (__all_sync(0xffffffffu, got)) {
        tc_fence_after();
        const bool write = valid;
        const float inv = (write && lsum > 0.f) ? 1.f / lsum : 0.f;
        const float w0 = a0 * inv, w1 = a1 * inv;
        const size_t row = static_cast<size_t>(bh) * p.T_out + static_cast<size_t>(i) * p.dview + res;
        uint4* dst = reinterpret_cast<uint4*>(p.O + row * D + wg * (D / 2));
#pragma unroll
        for (int q = 0; q < D / 64; ++q) {
          const uint32_t c = wg * (D / 2) + 32 * q;
          uint32_t o0[32], o1[32];
          tmem_ld32(lane_base + C::kColO0 + c, o0);
          tmem_ld32(lane_base + C::kColO1 + c, o1);
          if (write) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              float f[8];
#pragma unroll
              for (int k = 0; k < 8; ++k)
                f[k] = __uint_as_float(o0[8 * v4 + k]) * w0 + __uint_as_float(o1[8 * v4 + k]) * w1;
              uint4 w;
              w.x = pack_bf16x2(f[0], f[1]);
              w.y = pack_bf16x2(f[2], f[3]);
              w.z = pack_bf16x2(f[4], f[5]);
              w.w = pack_bf16x2(f[6], f[7]);
              dst[4 * q + v4] = w;
            }
          }
        }
        if (write && wg == 0 && p.LSE) p.LSE[row] = (mm + log2f(lsum)) * 0.69314718055994531f;
      }
    } else if (n_done > 0) {
      const bool got = mbar_wait(BAR(C::kBarO), 0, p.budget, p.err, kErrTimeout);
      if (__all_sync(0xffffffffu, got)) {
        tc_fence_after();
        const bool write = valid && (gathered || !m.rowglobal[i]);
        const float inv = (write && lrow > 0.f) ? 1.f / lrow : 0.f;
        const size_t row = static_cast<size_t>(bh) * p.T_out + static_cast<size_t>(i) * p.dview + res;
        uint4* dst = reinterpret_cast<uint4*>(p.O + row * D);
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(lane_base + colO + 32 * q, o);
          if (write) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(o[8 * v4 + 0]) * inv, __uint_as_float(o[8 * v4 + 1]) * inv);
              w.y = pack_bf16x2(__uint_as_float(o[8 * v4 + 2]) * inv, __uint_as_float(o[8 * v4 + 3]) * inv);
              w.z = pack_bf16x2(__uint_as_float(o[8 * v4 + 4]) * inv, __uint_as_float(o[8 * v4 + 5]) * inv);
              w.w = pack_bf16x2(__uint_as_float(o[8 * v4 + 6]) * inv, __uint_as_float(o[8 * v4 + 7]) * inv);
              dst[4 * q + v4] = w;
            }
          }
        }
        if (write && p.LSE) p.LSE[row] = (mrow + log2f(lrow)) * 0.69314718055994531f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
#undef BAR
}

// ---------------------------------------------------------------- host side

template <int D, int MW>
cudaError_t launch_d(const TcArgs& a, cudaStream_t st, const char** why) {
  using C = TcCfg<D, MW>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(fwd_tc_kernel<D, MW>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const long long T = a.mask.T;  // rows per residue class
  const long long dv = a.dview;
  CUtensorMap mQ, mK, mV, mQg, mKc, mVc;
  bool ok = make_map(&mQ, a.Q, D, T, a.BH, dv) && make_map(&mK, a.K, D, T, a.BH, dv) &&
            make_map(&mV, a.V, D, T, a.BH, dv);
  ok = ok && (a.n_cols > 0 ? make_map(&mKc, a.Kc, D, a.n_cols, a.BH) && make_map(&mVc, a.Vc, D, a.n_cols, a.BH)
                           : (mKc = mK, mVc = mV, true));
  ok = ok && (a.mask.n_global > 0 ? make_map(&mQg, a.Qg, D, a.mask.n_global, a.BH) : (mQg = mQ, true));
  if (!ok) {
    *why = "cuTensorMapEncodeTiled failed";
    return cudaErrorInvalidValue;
  }
  KParams kp;
  kp.O = static_cast<__nv_bfloat16*>(a.O);
  kp.LSE = a.LSE;
  kp.scale_log2 = a.scale * 1.4426950408889634f;
  kp.colmask = a.colmask;
  kp.mask = a.mask;
  kp.items = a.items;
  kp.entries = a.entries;
  kp.walk = a.walk;
  kp.err = a.err;
  kp.budget = a.wait_budget_cycles;
  kp.inject_timeout = a.inject_timeout;
  kp.n_items = a.n_items;
  kp.n_major = a.n_major;
  kp.dview = static_cast<int>(dv);
  kp.T_out = static_cast<int>(T * dv);
  kp.BH = a.BH * static_cast<int>(dv);
  const long long ctas = static_cast<long long>(a.n_items) * a.BH * dv;
  if (ctas > 0x7fffffffLL) {
    *why = "too many work items";
    return cudaErrorInvalidValue;
  }
  fwd_tc_kernel<D, MW><<<static_cast<unsigned>(ctas), C::kThreads, C::kSmemBytes, st>>>(
      mQ, mK, mV, mQg, mKc, mVc, kp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(int d, const TcArgs& a, cudaStream_t st, const char** why) {
  if (a.n_items == 0) return cudaSuccess;
  if (d == 64) return a.mma_per_tile ? launch_d<64, 2>(a, st, why) : launch_d<64, 1>(a, st, why);
  if (d == 128) return launch_d<128, 1>(a, st, why);
  *why = "head dim must be 64 or 128";
  return cudaErrorInvalidValue;
}

}  // namespace spattn
