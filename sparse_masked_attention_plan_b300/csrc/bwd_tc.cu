// bwd_tc.cu -- bf16 backward pass on the tcgen05 tensor cores: dQ (query-major) and
// dK, dV (key-major).
//
// For a query row i with allowed set S_i, the saved log-sum-exp LSE_i and the row
// dot D_i = dO_i . O_i, the chain rule through the softmax over S_i ("Sparse
// attention" glossary, section "Choose the available reads", differentiated) gives
//     P_ij = exp(scale q_i.k_j - LSE_i),  dS_ij = P_ij (dO_i.v_j - D_i)   (j in S_i),
//     dQ_i = scale sum_j dS_ij k_j.
// A CTA owns one 128-row query tile of one (batch, head) and walks the key tiles the
// forward schedule gives that tile (band tiles, packed sparse columns, dense walks of
// global rows), with the forward's per-row predicate inside partial tiles.
// Warp roles (576 threads):
//   warps 0-15 elementwise: P and dS of one query row per thread (its TMEM lane), in
//              four warpgroups that own key columns 32c .. 32c+31 (four warps per
//              sub-partition hide each other's latency)
//   warp 16    TMA producer: Q and dO tiles once, then K and V tiles into a ring
//   warp 17    MMA issuer: S = Q K^T and dP = dO V^T (both operands K-major from shared
//              memory), then dQ += dS K with dS (bf16) from TMEM and the same K tile
//              read as an MN-major operand
// TMEM: S of the key tile at 0 and dP at 128 (whole 128-key products), dQ at 256, and
// two dS buffers (bf16, 64 columns each) after it, used by alternate key tiles.  The
// next tile's S is issued once every elementwise warp has read this tile's S, so it
// runs while P is computed; the warps compute P from S while dP is still being
// computed.  P needs no running maximum: the forward's LSE already normalises it.
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

template <int D>
struct DqCfg {
  static constexpr int kChunkBytes = kTile * 64 * 2;  // 128 rows x 64 bf16, one swizzle span
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStages = D == 128 ? 4 : 8;
  // a tile's K and V take consecutive slots and complete the (even) K slot's barrier
  static_assert(kStages % 2 == 0, "K slots are the even slots");
  static constexpr int kSmemQ = 2 * kTileBytes;  // Q and dO
  static constexpr int kSmemKV = kStages * kTileBytes;
  // four elementwise warpgroups (warpgroup c owns keys 32c .. 32c+31 of every key tile),
  // then the TMA warp and the MMA warp (18 warps: up to 5 on one SM sub-partition, whose
  // 16K registers leave 96 per thread)
  static constexpr int kLoadWarp = 16, kMmaWarp = 17, kThreads = 32 * (kMmaWarp + 1);
  // kBarS + 0 / + 1: S / dP of the key tile are in TMEM
  // kBarP: every elementwise warp has written its rows of dS (one arrival per warp)
  // kBarSfree: every elementwise warp has read its columns of S
  static constexpr int kBarFull = 0, kBarEmpty = kStages, kBarQ = 2 * kStages,
                       kBarS = 2 * kStages + 1, kBarP = 2 * kStages + 3,
                       kBarDone = 2 * kStages + 4, kBarSfree = 2 * kStages + 5,
                       kNumBars = 2 * kStages + 6;
  static constexpr int kSmemBytes = kSmemQ + kSmemKV + kNumBars * 8 + 16 + 1024;
  static constexpr uint32_t kIdescFull = idesc_bf16_f32(128, 128, 0, 0);
  static constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, D, 0, 1);
  // Whole-tile products: S = Q K^T (TMEM 0) and dP = dO V^T (TMEM 128) of all 128 keys
  // as two N = 128 products with a barrier each (64-key halves would run at two thirds
  // of the tensor rate: with both operands in shared memory a 128x64x16 product takes
  // 48 cycles against 64 for 128x128x16).  dQ accumulates at 256; dS (bf16, 64 columns)
  // goes to one of two buffers after dQ (tile k uses buffer k % 2, chunk q at +16q), so
  // S of the next tile is computed as soon as every warp has read S (kBarSfree), while
  // the elementwise warps work on this tile; dP of the next tile follows this tile's dQ
  // products.  A dS buffer is rewritten two tiles later, after the dP product issued
  // behind that tile's dQ products has completed.
  static constexpr uint32_t kColDQ = 256;
  static constexpr uint32_t kColDS = 256 + D;
};

struct DqParams {
  __nv_bfloat16* dQ;
  const float* LSE;
  const float* Dvec;
  float scale;
  float scale_log2;
  const uint32_t* colmask;
  MaskDev mask;
  const int4* items;
  const int4* entries;
  int* err;
  uint64_t budget;
  int BH;     // work units along the head axis: (batch, head) x residue classes
  int dview;  // residue classes of a dilated view (1: rows are the sequence itself)
  int T_out;  // sequence length (the mask's T times dview)
};

// A (128 rows) x B^T (128 rows), both K-major over d: a whole-tile S or dP product.
template <int D>
__device__ __forceinline__ void issue_tile(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
  using C = DqCfg<D>;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off16 = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
    mma_ss(d_tmem, a_desc + off16, b_desc + off16, C::kIdescFull, kk > 0 ? 1u : 0u);
  }
}


// k-steps 2 chunk, 2 chunk + 1 of an accumulating product over the 128-wide tile
// dimension: the 32 columns one elementwise chunk has just written to TMEM (A, at
// a_chunk) against rows 32 chunk .. of the MN-major shared-memory operand (B).
template <int D>
__device__ __forceinline__ void issue_acc_chunk(uint32_t d_tmem, uint32_t a_chunk, uint64_t b_mn_desc,
                                                int chunk, bool accumulate) {
  using C = DqCfg<D>;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int kk = 2 * chunk + k;
    mma_ts(d_tmem, a_chunk + k * 8, b_mn_desc + ((kk * 16 * 128) >> 4), C::kIdescDQ,
           (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <int D>
__global__ void __launch_bounds__(DqCfg<D>::kThreads, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                     const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmQg, const __grid_constant__ CUtensorMap tmdOg,
                     const __grid_constant__ CUtensorMap tmKc, const __grid_constant__ CUtensorMap tmVc,
                     const DqParams p) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_addr(smem);
  const uint32_t sdO = sQ + C::kTileBytes;
  const uint32_t sKV = sQ + C::kSmemQ;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kSmemQ + C::kSmemKV);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  const uint32_t bar0 = smem_addr(bars);
#define BAR(k) (bar0 + 8u * static_cast<uint32_t>(k))

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA = (work item, query tile t, (batch, head)); heads vary fastest so neighbouring
  // CTAs of one item share nothing but the items of one head share K/V tiles in L2
  // a unit along the head axis is a (batch, head) and, in a dilated view, a residue
  // class r: its row q is sequence position q * dview + r
  const int res = (blockIdx.x % p.BH) % p.dview, bh = (blockIdx.x % p.BH) / p.dview;
  const int rank = (blockIdx.x / p.BH) >> 1;
  const int t = (blockIdx.x / p.BH) & 1;
  const int4 item = p.items[rank];
  // a split item of the forward schedule (both query tiles hold the same global rows,
  // alternate key tiles): the tile-0 CTA takes every entry of it, the tile-1 CTA nothing
  const bool split = (item.w & kItemSplit) != 0;
  const bool idle = split && t == 1;
  const int n_ent = idle ? 0 : item.z;
  const int4* ents = p.entries + item.y;
  const bool gathered = (item.w & kItemGathered) != 0;
  const MaskDev& m = p.mask;
  const int qrow0 = item.x + (split ? 0 : t * kTile);  // first row (or gathered index) of the tile
  const int active_bit = split ? (kActive0 | kActive1) : kActive0 << t;
  const int full_bit = split ? (kFull0 | kFull1) : kFull0 << t;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(BAR(C::kBarFull + s), 1);
      mbar_init(BAR(C::kBarEmpty + s), 1);
    }
    mbar_init(BAR(C::kBarQ), 1);
    mbar_init(BAR(C::kBarS + 0), 1);
    mbar_init(BAR(C::kBarS + 1), 1);
    // dS hand-off and S read: one arrival per elementwise warp (one per thread would
    // serialise on the barrier word, on the critical path)
    mbar_init(BAR(C::kBarP), 16);
    mbar_init(BAR(C::kBarDone), 1);
    mbar_init(BAR(C::kBarSfree), 16);
    fence_barrier_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::kLoadWarp) {
    // ------------------------------------------------------------ TMA producer
    const void* mapQ = gathered ? static_cast<const void*>(&tmQg) : static_cast<const void*>(&tmQ);
    const void* mapdO = gathered ? static_cast<const void*>(&tmdOg) : static_cast<const void*>(&tmdO);
    if (elect_one()) {
      mbar_arrive_expect_tx(BAR(C::kBarQ), 2 * C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_4d(sQ + c * C::kChunkBytes, mapQ, BAR(C::kBarQ), c * 64, gathered ? 0 : res, qrow0, bh);
        tma_load_4d(sdO + c * C::kChunkBytes, mapdO, BAR(C::kBarQ), c * 64, gathered ? 0 : res, qrow0,
                    bh);
      }
    }
    __syncwarp();
    // Tile t's K takes slot 2t and its V slot 2t + 1 (mod the ring); both complete the
    // K slot's barrier, so the MMA warp waits once per tile.  V is issued first: its
    // slot frees after dP, K's only after the dQ products, so at that point only K's
    // copy is still to come.
    int tiles = 0;     // tiles whose K and V were both issued
    bool v_only = false;  // the loop left between a tile's V and its K
    int4 e_next = n_ent ? ents[0] : make_int4(0, 0, 0, 0);
    for (int n = 0; n < n_ent; ++n) {
      const int4 e = e_next;
      if (n + 1 < n_ent) e_next = ents[n + 1];  // load ahead: latency off the issue path
      if (!(e.y & active_bit)) continue;
      const bool packed = ((e.y >> kKindShift) & 3) == kKindPacked;
      const int itk = 2 * tiles, itv = itk + 1;
      const int sk = itk % C::kStages, sv = itv % C::kStages;
      const void* mapk = packed ? static_cast<const void*>(&tmKc) : static_cast<const void*>(&tmK);
      const void* mapv = packed ? static_cast<const void*>(&tmVc) : static_cast<const void*>(&tmV);
      if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::kBarEmpty + sv), ((itv / C::kStages) & 1) ^ 1u,
                                             p.budget, p.err, kErrTimeout)))
        break;
      if (elect_one()) {
        mbar_expect_tx(BAR(C::kBarFull + sk), C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(sKV + sv * C::kTileBytes + c * C::kChunkBytes, mapv, BAR(C::kBarFull + sk),
                      c * 64, packed ? 0 : res, e.x, bh);
      }
      __syncwarp();
      v_only = true;
      if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::kBarEmpty + sk), ((itk / C::kStages) & 1) ^ 1u,
                                             p.budget, p.err, kErrTimeout)))
        break;
      if (elect_one()) {
        mbar_arrive_expect_tx(BAR(C::kBarFull + sk), C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(sKV + sk * C::kTileBytes + c * C::kChunkBytes, mapk, BAR(C::kBarFull + sk),
                      c * 64, packed ? 0 : res, e.x, bh);
      }
      __syncwarp();
      v_only = false;
      ++tiles;
    }
    // no copy is left in flight when the CTA exits: a V whose K was never issued (the
    // loop left on a timed-out wait) gets the missing arrival, so that its barrier
    // completes when V lands
    const int pending = tiles + (v_only ? 1 : 0);
    if (v_only && elect_one()) mbar_arrive(BAR(C::kBarFull + (2 * tiles) % C::kStages));
    __syncwarp();
    for (int t2 = pending - 1; t2 >= 0 && t2 >= pending - C::kStages / 2; --t2)
      mbar_wait(BAR(C::kBarFull + (2 * t2) % C::kStages), ((2 * t2) / C::kStages) & 1, p.budget,
                p.err, kErrTimeout);
    mbar_wait(BAR(C::kBarQ), 0, p.budget, p.err, kErrTimeout);
    __syncwarp();
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    const uint64_t q_desc = smem_desc_sw128(sQ, 16, 1024);
    const uint64_t do_desc = smem_desc_sw128(sdO, 16, 1024);
    const uint64_t kv_kdesc = smem_desc_sw128(sKV, 16, 1024);             // slot 0, K-major
    const uint64_t kv_mndesc = smem_desc_sw128(sKV, C::kChunkBytes, 1024);  // slot 0, MN-major
    constexpr uint32_t kSlot16 = C::kTileBytes >> 4;
    bool ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::kBarQ), 0, p.budget, p.err, kErrTimeout));
    if (ok) {
      tc_fence_after();
      // Per key tile: S of the next tile once every warp has read this tile's S, the dQ
      // products chunk by chunk as dS arrives, then dP of the next tile.
      auto next_active = [&](int x) {
        while (x < n_ent && !(ents[x].y & active_bit)) ++x;
        return x;
      };
      auto wait_kv = [&](int it) -> bool {  // K (slot it) and V (slot it + 1) of a tile
        return __all_sync(0xffffffffu, mbar_wait(BAR(C::kBarFull + it % C::kStages),
                                                 (it / C::kStages) & 1, p.budget, p.err,
                                                 kErrTimeout));
      };
      // S and dP of the tile whose K and V copies are at `it`
      auto issue_s = [&](int it) {
        if (elect_one()) {
          issue_tile<D>(tmem, q_desc, kv_kdesc + (it % C::kStages) * kSlot16);
          mma_commit(BAR(C::kBarS + 0));
        }
        __syncwarp();
      };
      auto issue_dp = [&](int it) {
        const uint32_t vs = (it + 1) % C::kStages;
        if (elect_one()) {
          issue_tile<D>(tmem + 128, do_desc, kv_kdesc + vs * kSlot16);
          mma_commit(BAR(C::kBarS + 1));
          mma_commit(BAR(C::kBarEmpty + vs));  // V is no longer needed
        }
        __syncwarp();
      };
      int it = 0, done = 0;
      int n = next_active(0);
      if (n < n_ent) {
        if (!wait_kv(0)) ok = false;
        if (ok) {
          tc_fence_after();
          issue_s(0);
          issue_dp(0);
        }
      }
      while (ok && n < n_ent) {
        const int n1 = next_active(n + 1);
        const uint32_t ks = it % C::kStages;
        const uint32_t par = done & 1;
        if (n1 < n_ent) {  // S of the next tile once every warp has read this tile's S
          if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::kBarSfree), par, p.budget, p.err,
                                                 kErrTimeout)) ||
              !wait_kv(it + 2)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(it + 2);
        }
        const uint32_t dsb = C::kColDS + 64 * (done & 1);
        // dQ += dS K once every warpgroup has written its 32 keys of dS
        if (!__all_sync(0xffffffffu,
                        mbar_wait(BAR(C::kBarP), par, p.budget, p.err, kErrTimeout))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            issue_acc_chunk<D>(tmem + C::kColDQ, tmem + dsb + 16 * q, kv_mndesc + ks * kSlot16, q,
                               done > 0);
        }
        __syncwarp();
        if (elect_one()) mma_commit(BAR(C::kBarEmpty + ks));
        __syncwarp();
        if (n1 < n_ent) issue_dp(it + 2);  // every chunk has read this tile's dP
        it += 2;
        ++done;
        n = n1;
      }
    }
    if (elect_one()) mma_commit(BAR(C::kBarDone));
    __syncwarp();
    mbar_wait(BAR(C::kBarDone), 0, p.budget, p.err, kErrTimeout);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ elementwise warps
    const int wg = warp >> 2;  // keys 32 wg .. 32 wg + 31 of every key tile
    const int r = ((warp & 3) << 5) | lane;
    const uint32_t lane_base = tmem + ((static_cast<uint32_t>(warp & 3) * 32u) << 16);
    int i;
    bool valid;
    if (gathered) {
      const int a = qrow0 + r;
      valid = a < m.n_global;
      i = valid ? m.gpos[a] : 0;
    } else {
      i = qrow0 + r;
      valid = i < m.T;
    }
    const size_t row = static_cast<size_t>(bh) * p.T_out +
                       (gathered ? static_cast<size_t>(i) : static_cast<size_t>(i) * p.dview + res);
    const float lse2 = valid ? p.LSE[row] * 1.4426950408889634f : 0.f;
    const float dsc = p.scale;
    const float dterm = valid ? -p.Dvec[row] * dsc : 0.f;
    const float c2 = p.scale_log2;
    const uint64_t c2x2 = f32x2(c2, c2), nl2x2 = f32x2(-lse2, -lse2);
    const uint64_t dsc2 = f32x2(dsc, dsc), dterm2 = f32x2(dterm, dterm);
    uint32_t sph = 0;
    int n_done = 0;
    // entries two ahead and the tile's column-mask words one ahead, so that no global
    // load's latency sits between one tile's hand-off and the next tile's mask
    int4 e_next = n_ent ? ents[0] : make_int4(0, 0, 0, 0);
    int4 e_next2 = n_ent > 1 ? ents[1] : make_int4(0, 0, 0, 0);
    uint4 cm_next = n_ent ? colmask_words(p.colmask, e_next) : make_uint4(0u, 0u, 0u, 0u);
    for (int n = 0; n < n_ent; ++n) {
      const int4 e = e_next;
      const uint4 cm = cm_next;
      e_next = e_next2;
      if (n + 2 < n_ent) e_next2 = ents[n + 2];
      if (n + 1 < n_ent) cm_next = colmask_words(p.colmask, e_next);
      if (!(e.y & active_bit)) continue;
      // the row's mask word for this warpgroup's 32 keys, computed before the wait so
      // that it overlaps the products
      uint32_t wq = 0xffffffffu;
      if (!(e.y & full_bit)) wq = row_word(make_predicate(m, cm, e, i), wg);
      // P of this warpgroup's 32 keys from S (while dP is still being computed), then
      // dS = scale P (dP - D) as dP arrives
      if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::kBarS + 0), sph, p.budget, p.err, kErrTimeout)))
        break;
      tc_fence_after();
      if (!valid) wq = 0u;
      float pr[32];
      {
        uint32_t sv[32];
        tmem_ld32(lane_base + 32 * wg, sv);
        tc_fence_before();
        __syncwarp();  // every lane has read S before lane 0 arrives for the warp
        if (lane == 0) mbar_arrive(BAR(C::kBarSfree));
#pragma unroll
        for (int b = 0; b < 16; ++b) {
          const int c0 = 2 * b;
          float x0, x1;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(sv[c0]), __uint_as_float(sv[c0 + 1])), c2x2,
                                nl2x2), x0, x1);
          pr[c0] = ((wq >> c0) & 1u) ? fast_exp2(x0) : 0.f;
          pr[c0 + 1] = ((wq >> (c0 + 1)) & 1u) ? fast_exp2(x1) : 0.f;
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::kBarS + 1), sph, p.budget, p.err, kErrTimeout)))
        break;
      sph ^= 1u;
      tc_fence_after();
      // dS of the 32 keys, 16 at a time, into this tile's dS buffer (keys 32 wg .. at
      // column 16 wg as bf16 pairs)
      const uint32_t dsc_col = lane_base + C::kColDS + 64 * (n_done & 1) + 16 * wg;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t dv[16], pk[8];
        tmem_ld16(lane_base + 128 + 32 * wg + 16 * hf, dv);
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const int c0 = 2 * b;
          const uint64_t t2 = fma_f32x2(f32x2(__uint_as_float(dv[c0]), __uint_as_float(dv[c0 + 1])),
                                        dsc2, dterm2);
          float g0, g1;
          f32x2_split(mul_f32x2(f32x2(pr[16 * hf + c0], pr[16 * hf + c0 + 1]), t2), g0, g1);
          pk[b] = pack_bf16x2(g0, g1);
        }
        tmem_st8(dsc_col + 8 * hf, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();  // every lane's dS is stored before lane 0 arrives for the warp
      if (lane == 0) mbar_arrive(BAR(C::kBarP));
      ++n_done;
    }
    // ---------------------------------------------------------- epilogue
    const bool write = !idle && valid && (gathered || !m.rowglobal[i]);
    bool have = false;
    if (n_done > 0) {
      have = __all_sync(0xffffffffu, mbar_wait(BAR(C::kBarDone), 0, p.budget, p.err, kErrTimeout));
      if (have) tc_fence_after();
    }
    // this warpgroup's quarter of the d columns (32 at d = 128, 16 at d = 64)
    constexpr int kQc = D / 4;
    uint4* dst = reinterpret_cast<uint4*>(p.dQ + row * D + kQc * wg);
    uint32_t o[32];
    if (have) {
      if constexpr (kQc == 32) {
        tmem_ld32(lane_base + C::kColDQ + 32 * wg, o);
      } else {
        uint32_t h[16];
        tmem_ld16(lane_base + C::kColDQ + 16 * wg, h);
#pragma unroll
        for (int b = 0; b < 16; ++b) o[b] = h[b];
      }
    } else {
#pragma unroll
      for (int b = 0; b < kQc; ++b) o[b] = 0u;
    }
    if (write) {
#pragma unroll
      for (int v4 = 0; v4 < kQc / 8; ++v4) {
        uint4 x;
        x.x = pack_bf16x2(__uint_as_float(o[8 * v4 + 0]), __uint_as_float(o[8 * v4 + 1]));
        x.y = pack_bf16x2(__uint_as_float(o[8 * v4 + 2]), __uint_as_float(o[8 * v4 + 3]));
        x.z = pack_bf16x2(__uint_as_float(o[8 * v4 + 4]), __uint_as_float(o[8 * v4 + 5]));
        x.w = pack_bf16x2(__uint_as_float(o[8 * v4 + 6]), __uint_as_float(o[8 * v4 + 7]));
        dst[v4] = x;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
#undef BAR
}

// ---------------------------------------------------------------- dK, dV (key-major)
//
//     dV_j = sum_i P_ij dO_i,   dK_j = scale sum_i dS_ij q_i   (i with j in S_i)
// Warp roles as in the dQ kernel (warps 0-15 elementwise in four warpgroups, each
// owning 32 query columns; 16 producer; 17 MMA).
// A CTA owns one 128-key unit (natural keys, or packed sparse columns) of one (batch,
// head): its K and V tiles stay in shared memory while the 128-row query tiles that
// read it stream through a ring (Q and dO per stage).  Per query tile:
//   S^T = K Q^T and dP^T = V dO^T (tensor cores, TMEM lanes = keys, columns = queries);
//   elementwise (thread = key): P^T = 2^(S^T scale log2 e - LSE log2 e) under the
//   key's mask, dS^T = scale P^T (dP^T - D), both to TMEM as bf16 pairs over the
//   first 16 of each warpgroup's own 32 columns;
//   dV += P^T dO and dK += dS^T Q (A from TMEM; dO and Q read as MN-major operands).
// Each warp loads the LSE and D of its 32 queries itself, one tile ahead; a query that
// is not a row of this tile (past the end, or a global row summed by its own dense walk)
// gets LSE = +inf, which makes its weight 0 without a mask.  The key-side mask (the
// warpgroup's one 32-row word) is a few spans per thread: the key's local window seen
// from the key (the rows whose window holds it), all later rows for a strided or global
// column, the query blocks that list the key's block as random (transposed lists), a
// range of packed columns, or the suffix of gathered global rows at or after the key;
// entries whose rows and keys all lie inside the local window skip it (host flag).
// TMEM: S^T of the whole query tile at 0, dP^T at 128, dV at 256, dK at 256 + d.

template <int D>
struct KvCfg {
  static constexpr int kChunkBytes = kTile * 64 * 2;
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStages = D == 128 ? 2 : 4;  // one stage = the Q and dO tiles
  static constexpr int kSmemKV = 2 * kTileBytes;
  static constexpr int kSmemRing = kStages * 2 * kTileBytes;
  // four elementwise warpgroups (warpgroup q owns query chunk q of every tile), then the
  // TMA warp and the MMA warp
  // (18 warps: up to 5 on one SM sub-partition, whose 16K registers leave 96 per thread)
  static constexpr int kLoadWarp = 16, kMmaWarp = 17, kThreads = 32 * (kMmaWarp + 1);
  // LSE and D of each elementwise warp's 32 query columns: [warp][2][32]
  static constexpr int kSmemVec = 16 * 2 * 32 * 4;
  // kBarS + 0 / + 1: S^T / dP^T of the query tile are in TMEM; kBarP / kBarDS: every
  // elementwise warp has written its rows of P^T / dS^T (one arrival per warp)
  // a stage's Q and dO complete one barrier (kBarFull); each has its own slot-free
  // barrier: dO's slot is free once dV has read it, Q's only once dK has
  static constexpr int kBarKV = 0, kBarFull = 1, kBarEmptyQ = 1 + kStages,
                       kBarEmptyDO = 1 + 2 * kStages, kBarS = 1 + 3 * kStages,
                       kBarP = 3 + 3 * kStages, kBarDS = 4 + 3 * kStages,
                       kBarDone = 5 + 3 * kStages, kNumBars = 6 + 3 * kStages;
  static constexpr int kSmemBytes = kSmemKV + kSmemRing + kSmemVec + kNumBars * 8 + 16 + 1024;
  // products use the dQ kernel's issue helpers (128 x 128 tiles and 128 x d chunks).
  // TMEM: S^T of the whole query tile at 0 (query q in column q), dP^T at 128; chunk c
  // (queries 32c .. 32c+31) writes its P^T and dS^T (bf16 pairs) over the first 16 of
  // its own 32 columns of each; dV, dK after them
  static constexpr uint32_t kColDV = 256, kColDK = 256 + D;
};

struct KvParams {
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  float* dKc;  // packed-column partial sums [BH][n_cols][d] (fp32)
  float* dVc;
  const float* LSE;
  const float* Dvec;
  float scale;
  float scale_log2;
  const uint32_t* colmask;
  MaskDev mask;
  const int32_t* cols;
  const int32_t* colidx;
  const int32_t* rt_off;
  const int32_t* rt_qb;
  const int4* units;
  const int4* entries;
  int unit0;
  int n_cols;
  int* err;
  uint64_t budget;
  int BH;     // work units along the head axis: (batch, head) x residue classes
  int dview;  // residue classes of a dilated view (1: rows are the sequence itself)
  int T_out;  // sequence length (the mask's T times dview)
};

// Bits of [a, b] (tile columns) in the four 32-bit words.
__device__ __forceinline__ void add_span(int a, int b, uint32_t (&w)[4]) {
  a = max(a, 0);
  b = min(b, kTile - 1);
  if (a > b) return;
#pragma unroll
  for (int k = 0; k < 4; ++k) w[k] |= span_bits(a, b, 32 * k);
}

// What the mask says about key j whatever the query tile: whether it is a strided or
// global column, and its range in the transposed random-block list.  Loaded once per
// CTA, so no global load sits on the per-tile path.
struct KeyInfo {
  bool colbit;
  int rt_lo, rt_hi;
};

__device__ __forceinline__ KeyInfo key_info(const KvParams& p, int j) {
  const MaskDev& m = p.mask;
  KeyInfo k;
  const uint32_t cw = p.colmask[(j / kTile) * 4 + (j % kTile) / 32];
  k.colbit = (cw >> (j & 31)) & 1u;
  k.rt_lo = k.rt_hi = 0;
  if (m.rand_block) {
    const int kb = j / m.rand_block;
    k.rt_lo = p.rt_off[kb];
    k.rt_hi = p.rt_off[kb + 1];
  }
  return k;
}

// Word k (rows 32k .. 32k+31) of the query rows of the tile at row q0 that may read key
// j (packed index c_pk for packed units), for an entry of `kind`; rows that are not rows
// of the tile are removed separately (LSE = +inf).  The band tile with a contiguous
// window and no random blocks is one span; other band and random tiles build all four
// words and return word k.
__device__ __forceinline__ uint32_t key_word(const KvParams& p, int kind, int4 e, int q0, int j,
                                             int c_pk, const KeyInfo& ki, int k) {
  const MaskDev& m = p.mask;
  const int base = 32 * k;
  if (kind == kKindPacked) return (c_pk >= e.z && c_pk < e.w) ? 0xffffffffu : 0u;
  if (kind == kKindDense) {  // gathered global rows q0 .. : every key j <= their position
    const int nr = min(kTile, m.n_global - q0);
    int r0 = 0;
    if (m.causal) {
      int lo = 0, hi = nr;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (m.gpos[q0 + mid] < j) lo = mid + 1; else hi = mid;
      }
      r0 = lo;
    }
    return span_bits(r0, nr - 1, base);
  }
  const int jc = j - q0;  // the key's own column
  const bool colbit = ki.colbit;
  if (kind == kKindBand && m.dilation == 1 && !m.rand_block) {
    // causal: the window [jc, jc + w - 1] or, for a strided or global key, every later
    // row [jc, 127] (which contains it); bidirectional: [jc - r, jc + r] or every row
    int lo = 0, hi = kTile - 1;
    if (m.causal) {
      lo = jc;
      if (!colbit && m.window) hi = jc + static_cast<int>(m.window) - 1;
    } else if (!colbit && m.radius >= 0) {
      lo = jc - static_cast<int>(m.radius);
      hi = jc + static_cast<int>(m.radius);
    }
    return span_bits(lo, hi, base);
  }
  uint32_t w[4];
  const int cut = m.causal ? jc : 0;
  uint32_t extra[4] = {0u, 0u, 0u, 0u};
  if (m.rand_block && !(kind == kKindRandom && colbit)) {
    for (int x = ki.rt_lo; x < ki.rt_hi; ++x) {
      const int r0 = p.rt_qb[x] * m.rand_block - q0;
      add_span(max(r0, cut), r0 + m.rand_block - 1, extra);
    }
  }
  if (kind == kKindRandom) {
#pragma unroll
    for (int x = 0; x < 4; ++x) w[x] = extra[x];
  } else {
    if (colbit) add_span(cut, kTile - 1, extra);
    RowPredicate pr;
    const int d = m.dilation;
    if (m.causal) {
      pr.lo = jc;
      pr.hi = m.window ? jc + (m.window - 1) * d : m.T - 1 - q0;
    } else {
      pr.lo = m.radius >= 0 ? jc - m.radius * d : 0;
      pr.hi = m.radius >= 0 ? jc + m.radius * d : kTile - 1;
    }
    pr.hi = min(pr.hi, kTile - 1);
    pr.hb = kTile - 1;
    pr.dil = d;
    pr.res = d == 1 ? 0 : ((jc % d) + d) % d;  // no division when d = 1
#pragma unroll
    for (int x = 0; x < 4; ++x) pr.bits[x] = extra[x];
    row_mask(pr, w);
  }
  // word k by value: w stays in registers
  return k == 0 ? w[0] : (k == 1 ? w[1] : (k == 2 ? w[2] : w[3]));
}

template <int D>
__global__ void __launch_bounds__(KvCfg<D>::kThreads, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                       const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmQg, const __grid_constant__ CUtensorMap tmdOg,
                       const __grid_constant__ CUtensorMap tmKc, const __grid_constant__ CUtensorMap tmVc,
                       const KvParams p) {
  using C = KvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sK = smem_addr(smem);
  const uint32_t sV = sK + C::kTileBytes;
  const uint32_t sRing = sK + C::kSmemKV;  // stage s: Q at +0, dO at +kTileBytes
  float* s_vec = reinterpret_cast<float*>(smem + C::kSmemKV + C::kSmemRing);  // [warp][LSE, D][32]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kSmemKV + C::kSmemRing + C::kSmemVec);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  const uint32_t bar0 = smem_addr(bars);
#define BAR(k) (bar0 + 8u * static_cast<uint32_t>(k))

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int res = (blockIdx.x % p.BH) % p.dview, bh = (blockIdx.x % p.BH) / p.dview;
  const int4 unit = p.units[p.unit0 + blockIdx.x / p.BH];
  const bool packed_unit = (unit.w & kUnitPacked) != 0;
  const int n_ent = unit.z;
  const int4* ents = p.entries + unit.y;
  const MaskDev& m = p.mask;

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::kBarKV), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(BAR(C::kBarFull + s), 1);
      mbar_init(BAR(C::kBarEmptyQ + s), 1);
      mbar_init(BAR(C::kBarEmptyDO + s), 1);
    }
    mbar_init(BAR(C::kBarS + 0), 1);
    mbar_init(BAR(C::kBarS + 1), 1);
    // one arrival per elementwise warp on the P^T and dS^T hand-offs
    mbar_init(BAR(C::kBarP), 16);
    mbar_init(BAR(C::kBarDS), 16);
    mbar_init(BAR(C::kBarDone), 1);
    fence_barrier_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::kLoadWarp) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      const void* mk = packed_unit ? static_cast<const void*>(&tmKc) : static_cast<const void*>(&tmK);
      const void* mv = packed_unit ? static_cast<const void*>(&tmVc) : static_cast<const void*>(&tmV);
      mbar_arrive_expect_tx(BAR(C::kBarKV), 2 * C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_4d(sK + c * C::kChunkBytes, mk, BAR(C::kBarKV), c * 64, packed_unit ? 0 : res,
                    unit.x, bh);
        tma_load_4d(sV + c * C::kChunkBytes, mv, BAR(C::kBarKV), c * 64, packed_unit ? 0 : res,
                    unit.x, bh);
      }
    }
    __syncwarp();
    // per query tile: dO first, then Q; both complete the stage's one barrier, dO raising
    // its expected bytes, Q arriving.  With two stages (d = 128) dO is issued as soon as
    // its slot is free (after dV), so that when Q's frees (after dK) only Q is still to
    // come; with more, the stage is taken whole once Q's slot is free
    constexpr bool kSplitFree = C::kStages == 2;
    int issued = 0;
    bool do_only = false;  // the loop left between a tile's dO and its Q
    int4 e_next = n_ent ? ents[0] : make_int4(0, 0, 0, 0);
    for (int n = 0; n < n_ent; ++n) {
      const int4 e = e_next;
      if (n + 1 < n_ent) e_next = ents[n + 1];
      const bool gathered = (e.y & kEntryGathered) != 0;
      const int s = n % C::kStages;
      const uint32_t ph = (n / C::kStages) & 1;
      const int r4 = gathered ? 0 : res;
      const void* mq = gathered ? static_cast<const void*>(&tmQg) : static_cast<const void*>(&tmQ);
      const void* md = gathered ? static_cast<const void*>(&tmdOg) : static_cast<const void*>(&tmdO);
      const uint32_t dst = sRing + s * 2 * C::kTileBytes;
      if (!__all_sync(0xffffffffu, mbar_wait(BAR((kSplitFree ? C::kBarEmptyDO : C::kBarEmptyQ) + s),
                                             ph ^ 1u, p.budget, p.err, kErrTimeout)))
        break;
      if (elect_one()) {
        mbar_expect_tx(BAR(C::kBarFull + s), C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(dst + C::kTileBytes + c * C::kChunkBytes, md, BAR(C::kBarFull + s), c * 64, r4,
                      e.x, bh);
      }
      __syncwarp();
      do_only = true;
      if (kSplitFree && !__all_sync(0xffffffffu, mbar_wait(BAR(C::kBarEmptyQ + s), ph ^ 1u,
                                                           p.budget, p.err, kErrTimeout)))
        break;
      if (elect_one()) {
        mbar_arrive_expect_tx(BAR(C::kBarFull + s), C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(dst + c * C::kChunkBytes, mq, BAR(C::kBarFull + s), c * 64, r4, e.x, bh);
      }
      __syncwarp();
      do_only = false;
      ++issued;
    }
    // no copy is left in flight when the CTA exits: a dO whose Q was never issued (the
    // loop left on a timed-out wait) gets the missing arrival, so that its barrier
    // completes when dO lands
    const int pending = issued + (do_only ? 1 : 0);
    if (do_only && elect_one()) mbar_arrive(BAR(C::kBarFull + issued % C::kStages));
    __syncwarp();
    for (int it = pending - 1; it >= 0 && it >= pending - C::kStages; --it)
      mbar_wait(BAR(C::kBarFull + it % C::kStages), (it / C::kStages) & 1, p.budget, p.err,
                kErrTimeout);
    mbar_wait(BAR(C::kBarKV), 0, p.budget, p.err, kErrTimeout);
    __syncwarp();
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    const uint64_t k_desc = smem_desc_sw128(sK, 16, 1024);
    const uint64_t v_desc = smem_desc_sw128(sV, 16, 1024);
    const uint64_t ring_k = smem_desc_sw128(sRing, 16, 1024);              // stage 0 Q, K-major
    const uint64_t ring_mn = smem_desc_sw128(sRing, C::kChunkBytes, 1024);  // stage 0 Q, MN-major
    constexpr uint32_t kStage16 = (2 * C::kTileBytes) >> 4, kDo16 = C::kTileBytes >> 4;
    bool ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::kBarKV), 0, p.budget, p.err, kErrTimeout));
    if (ok) {
      tc_fence_after();
      // Whole-tile products (128 x 128 x 16 runs at the full tensor rate; a 64-query
      // half would take 48 cycles for half the work).  Issue order per query tile n:
      //   S^T(n), dP^T(n), [P^T(n) written] dV(n), S^T(n+1), [dS^T(n) written] dK(n),
      //   dP^T(n+1), ...
      // dV needs only P, so it runs while the warps compute dS; S^T(n+1) overwrites the
      // P^T(n) columns only after dV(n) (the products execute in issue order), and
      // dP^T(n+1) the dS^T(n) columns only after dK(n), so the warps compute P of the
      // next tile while dK and dP run.
      auto wait_q = [&](int n) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(BAR(C::kBarFull + n % C::kStages),
                                                 (n / C::kStages) & 1, p.budget, p.err,
                                                 kErrTimeout));
      };
      auto issue_s = [&](int n) {
        if (elect_one()) {
          issue_tile<D>(tmem, k_desc, ring_k + (n % C::kStages) * kStage16);
          mma_commit(BAR(C::kBarS + 0));
        }
        __syncwarp();
      };
      auto issue_dp = [&](int n) {
        if (elect_one()) {
          issue_tile<D>(tmem + 128, v_desc, ring_k + (n % C::kStages) * kStage16 + kDo16);
          mma_commit(BAR(C::kBarS + 1));
        }
        __syncwarp();
      };
      if (n_ent > 0) {
        if (!wait_q(0)) ok = false;
        if (ok) {
          tc_fence_after();
          issue_s(0);
          issue_dp(0);
        }
      }
      for (int n = 0; ok && n < n_ent; ++n) {
        const uint32_t s = n % C::kStages;
        const uint32_t par = n & 1;
        // With more than two stages the next tile's Q and dO are long since loaded, as a
        // rule, and are checked while the warps still compute P, so that S^T(n+1) follows
        // dV(n) at once; with two (d = 128) Q's slot is refilled only after dK(n-1), and
        // the wait is left as late as possible
        constexpr bool kEarlyQ = C::kStages > 2;
        if (kEarlyQ && n + 1 < n_ent && !wait_q(n + 1)) break;
        // dV += P^T dO over the tile's four 32-query chunks
        if (!__all_sync(0xffffffffu,
                        mbar_wait(BAR(C::kBarP), par, p.budget, p.err, kErrTimeout)))
          break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            issue_acc_chunk<D>(tmem + C::kColDV, tmem + 32 * c, ring_mn + s * kStage16 + kDo16, c,
                               n > 0);
          if (C::kStages == 2) mma_commit(BAR(C::kBarEmptyDO + s));  // dV has read dO
        }
        __syncwarp();
        if (n + 1 < n_ent) {
          if (!kEarlyQ && !wait_q(n + 1)) break;
          tc_fence_after();
          issue_s(n + 1);
        }
        // dK += dS^T Q, then Q's slot is free
        if (!__all_sync(0xffffffffu,
                        mbar_wait(BAR(C::kBarDS), par, p.budget, p.err, kErrTimeout)))
          break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            issue_acc_chunk<D>(tmem + C::kColDK, tmem + 128 + 32 * c, ring_mn + s * kStage16, c,
                               n > 0);
          mma_commit(BAR(C::kBarEmptyQ + s));  // dK has read Q
        }
        __syncwarp();
        if (n + 1 < n_ent) issue_dp(n + 1);
      }
    }
    if (elect_one()) mma_commit(BAR(C::kBarDone));
    __syncwarp();
    mbar_wait(BAR(C::kBarDone), 0, p.budget, p.err, kErrTimeout);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ elementwise warps
    // warpgroup wg: query chunk wg of every tile and, in the epilogue, half of the
    // columns of dV (wg < 2) or dK
    const int wg = warp >> 2;
    const int hh = wg >> 1, qc = wg & 1;
    const int kk = ((warp & 3) << 5) | lane;  // key row of the unit = TMEM lane
    const uint32_t lane_base = tmem + ((static_cast<uint32_t>(warp & 3) * 32u) << 16);
    const int key = unit.x + kk;
    const bool key_valid = packed_unit ? key < p.n_cols : key < m.T;
    const int j = key_valid ? (packed_unit ? p.cols[key] : key) : 0;
    const float c2 = p.scale_log2, dsc = p.scale;
    const uint64_t c2x2 = f32x2(c2, c2), dsc2 = f32x2(dsc, dsc);
    const size_t head = static_cast<size_t>(bh) * p.T_out;
    // sequence position of view row x (gathered global rows are positions already)
    auto seq = [&](int x) { return static_cast<size_t>(x) * p.dview + res; };
    uint32_t sph = 0;
    int n_done = 0;
    const KeyInfo ki = key_info(p, j);
    // LSE and D of query column 32 wg + lane of an entry (every warp loads its
    // chunk's 32 columns itself), one entry ahead so the global loads overlap the
    // previous tile's work.  The loads are issued unconditionally (a row outside the
    // sequence reads row 0) and whether the column is a row of the tile (inside the
    // sequence and not a global row, whose gradient comes from its gathered tile) is
    // decided when the values are used (`in_seq` and the loaded `is_global` flag), so
    // nothing waits for the loads here
    auto column_values = [&](const int4& e, float& lse_v, float& dd_v, uint32_t& in_seq,
                             uint32_t& is_global) {
      const int a = e.x + 32 * wg + lane;
      size_t at;
      if (e.y & kEntryGathered) {  // the row's position comes from the global list
        const int i = a < m.n_global ? m.gpos[a] : -1;
        in_seq = i >= 0;
        is_global = 0u;
        at = head + static_cast<size_t>(max(i, 0));
      } else {
        const int i = a < m.T ? a : 0;
        in_seq = a < m.T;
        is_global = m.rowglobal[i];
        at = head + seq(i);
      }
      lse_v = p.LSE[at];
      dd_v = p.Dvec[at];
    };
    // this warp's LSE and D: lane l writes column l, every lane reads all 32
    float* s_lse = s_vec + warp * 64;
    float* s_dd = s_lse + 32;
    // entries two ahead, so the next entry's row index is there when its values load
    int4 e_next = n_ent ? ents[0] : make_int4(0, 0, 0, 0);
    int4 e_next2 = n_ent > 1 ? ents[1] : make_int4(0, 0, 0, 0);
    float lse_next = 0.f, dd_next = 0.f;
    uint32_t in_next = 0u, glob_next = 0u;
    if (n_ent) column_values(e_next, lse_next, dd_next, in_next, glob_next);
    for (int n = 0; n < n_ent; ++n) {
      const int4 e = e_next;
      const bool keep_next = in_next && !glob_next;
      const float lse_cur = keep_next ? lse_next * 1.4426950408889634f : INFINITY;
      const float dd_cur = keep_next ? dd_next * dsc : 0.f;
      e_next = e_next2;
      if (n + 2 < n_ent) e_next2 = ents[n + 2];
      const int kind = (e.y >> kKindShift) & 3;
      __syncwarp();  // every lane has read the previous tile's values
      s_lse[lane] = lse_cur;
      s_dd[lane] = dd_cur;
      __syncwarp();
      if (n + 1 < n_ent) column_values(e_next, lse_next, dd_next, in_next, glob_next);
      // this chunk's word of the key's mask (rows 32 wg .. 32 wg + 31 of the tile)
      uint32_t wq = (e.y & kEntryFull) ? 0xffffffffu : key_word(p, kind, e, e.x, j, key, ki, wg);
      if (!key_valid) wq = 0u;
      if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::kBarS + 0), sph, p.budget, p.err, kErrTimeout)))
        break;
      tc_fence_after();
      // S^T of the chunk's 32 queries -> P (kept in fp32 for dS), P^T (bf16 pairs) over
      // the first 16 of those columns, which only this warpgroup reads
      const uint32_t cs = lane_base + 32 * wg;
      const bool all = wq == 0xffffffffu;
      float pf[32];
      {
        uint32_t sv[32];
        tmem_ld32(cs, sv);
        uint32_t pp[16];
#pragma unroll
        for (int b = 0; b < 16; b += 2) {  // four columns per step: one vector load
          const float4 l4 = *reinterpret_cast<const float4*>(s_lse + 2 * b);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int x = 2 * (b + h);  // column within the chunk
            const float la = h ? l4.z : l4.x, lb = h ? l4.w : l4.y;
            float x0, x1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1])), c2x2,
                                  f32x2(-la, -lb)), x0, x1);
            float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
            if (!all) {
              if (!((wq >> x) & 1u)) p0 = 0.f;
              if (!((wq >> (x + 1)) & 1u)) p1 = 0.f;
            }
            pf[x] = p0;
            pf[x + 1] = p1;
            pp[b + h] = pack_bf16x2(p0, p1);
          }
        }
        tmem_st16(cs, pp);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();  // every lane's P^T is stored before lane 0 arrives for the warp
      if (lane == 0) mbar_arrive(BAR(C::kBarP));
      if (!__all_sync(0xffffffffu, mbar_wait(BAR(C::kBarS + 1), sph, p.budget, p.err, kErrTimeout)))
        break;
      sph ^= 1u;
      tc_fence_after();
      // dP^T -> dS = P (dP - D) scale, 16 columns at a time, dS^T over the first 16 of
      // the chunk's dP^T columns (each half's words over columns already read)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t dv[16];
        tmem_ld16(cs + 128 + 16 * hf, dv);
        uint32_t pg[8];
#pragma unroll
        for (int b = 0; b < 8; b += 2) {
          const float4 d4 = *reinterpret_cast<const float4*>(s_dd + 16 * hf + 2 * b);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int x = 2 * (b + h);  // column within the half
            const int xc = 16 * hf + x;  // column within the chunk
            const float da = h ? d4.z : d4.x, db = h ? d4.w : d4.y;
            const uint64_t t2 = fma_f32x2(f32x2(__uint_as_float(dv[x]), __uint_as_float(dv[x + 1])),
                                          dsc2, f32x2(-da, -db));
            float g0, g1;
            f32x2_split(mul_f32x2(f32x2(pf[xc], pf[xc + 1]), t2), g0, g1);
            pg[b + h] = pack_bf16x2(g0, g1);
          }
        }
        tmem_st8(cs + 128 + 8 * hf, pg);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();  // every lane's dS^T is stored before lane 0 arrives for the warp
      if (lane == 0) mbar_arrive(BAR(C::kBarDS));
      ++n_done;
    }
    // ---------------------------------------------------------- epilogue
    bool have = false;
    if (n_done > 0) {
      have = __all_sync(0xffffffffu, mbar_wait(BAR(C::kBarDone), 0, p.budget, p.err, kErrTimeout));
      if (have) tc_fence_after();
    }
    const int cpk = (!packed_unit && key_valid && p.n_cols) ? p.colidx[j] : -1;
    {
      const int half = hh;  // warpgroups 0, 1 write dV, warpgroups 2, 3 dK
      const uint32_t col = half ? C::kColDK : C::kColDV;
#pragma unroll
      for (int qi = 0; qi < D / 64; ++qi) {
        const int q = qc * (D / 64) + qi;  // this warpgroup's half of the 32-column chunks
        uint32_t o[32];
        if (have) {
          tmem_ld32(lane_base + col + 32 * q, o);
        } else {
#pragma unroll
          for (int b = 0; b < 32; ++b) o[b] = 0u;
        }
        if (!key_valid) continue;
        if (packed_unit) {
          float* dst = (half ? p.dKc : p.dVc) + (static_cast<size_t>(bh) * p.n_cols + key) * D + 32 * q;
#pragma unroll
          for (int b = 0; b < 32; b += 4)
            *reinterpret_cast<float4*>(dst + b) =
                make_float4(__uint_as_float(o[b]), __uint_as_float(o[b + 1]),
                            __uint_as_float(o[b + 2]), __uint_as_float(o[b + 3]));
          continue;
        }
        float f[32];
#pragma unroll
        for (int b = 0; b < 32; ++b) f[b] = __uint_as_float(o[b]);
        if (cpk >= 0) {
          const float* src = (half ? p.dKc : p.dVc) + (static_cast<size_t>(bh) * p.n_cols + cpk) * D + 32 * q;
#pragma unroll
          for (int b = 0; b < 32; b += 4) {
            const float4 x = *reinterpret_cast<const float4*>(src + b);
            f[b] += x.x;
            f[b + 1] += x.y;
            f[b + 2] += x.z;
            f[b + 3] += x.w;
          }
        }
        uint4* dst = reinterpret_cast<uint4*>((half ? p.dK : p.dV) + (head + seq(j)) * D + 32 * q);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          uint4 x;
          x.x = pack_bf16x2(f[8 * v4 + 0], f[8 * v4 + 1]);
          x.y = pack_bf16x2(f[8 * v4 + 2], f[8 * v4 + 3]);
          x.z = pack_bf16x2(f[8 * v4 + 4], f[8 * v4 + 5]);
          x.w = pack_bf16x2(f[8 * v4 + 6], f[8 * v4 + 7]);
          dst[v4] = x;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
#undef BAR
}

template <int D>
cudaError_t launch_kv_d(const BwdTcArgs& a, cudaStream_t st, const char** why) {
  using C = KvCfg<D>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(bwd_dkdv_tc_kernel<D>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const long long T = a.mask.T;  // rows per residue class
  const long long dv = a.dview;
  CUtensorMap mQ, mdO, mK, mV, mQg, mdOg, mKc, mVc;
  bool ok = make_map(&mQ, a.Q, D, T, a.BH, dv) && make_map(&mdO, a.dO, D, T, a.BH, dv) &&
            make_map(&mK, a.K, D, T, a.BH, dv) && make_map(&mV, a.V, D, T, a.BH, dv);
  ok = ok && (a.n_cols > 0 ? make_map(&mKc, a.Kc, D, a.n_cols, a.BH) && make_map(&mVc, a.Vc, D, a.n_cols, a.BH)
                           : (mKc = mK, mVc = mV, true));
  ok = ok && (a.mask.n_global > 0 ? make_map(&mQg, a.Qg, D, a.mask.n_global, a.BH) &&
                                        make_map(&mdOg, a.dOg, D, a.mask.n_global, a.BH)
                                  : (mQg = mQ, mdOg = mdO, true));
  if (!ok) {
    *why = "cuTensorMapEncodeTiled failed";
    return cudaErrorInvalidValue;
  }
  KvParams kp;
  kp.dK = static_cast<__nv_bfloat16*>(a.dK);
  kp.dV = static_cast<__nv_bfloat16*>(a.dV);
  kp.dKc = a.dKc;
  kp.dVc = a.dVc;
  kp.LSE = a.LSE;
  kp.Dvec = a.Dvec;
  kp.scale = a.scale;
  kp.scale_log2 = a.scale * 1.4426950408889634f;
  kp.colmask = a.colmask;
  kp.mask = a.mask;
  kp.cols = a.cols;
  kp.colidx = a.colidx;
  kp.rt_off = a.rt_off;
  kp.rt_qb = a.rt_qb;
  kp.units = a.units;
  kp.entries = a.u_entries;
  kp.n_cols = a.n_cols;
  kp.err = a.err;
  kp.budget = a.wait_budget_cycles;
  kp.BH = a.BH * static_cast<int>(dv);
  kp.dview = static_cast<int>(dv);
  kp.T_out = static_cast<int>(T * dv);
  // packed units first: their partial sums are added by the natural units
  const int parts[2][2] = {{0, a.n_packed_units}, {a.n_packed_units, a.n_units}};
  for (const auto& pr : parts) {
    const long long ctas = static_cast<long long>(pr[1] - pr[0]) * a.BH * dv;
    if (ctas <= 0) continue;
    if (ctas > 0x7fffffffLL) {
      *why = "too many key units";
      return cudaErrorInvalidValue;
    }
    kp.unit0 = pr[0];
    bwd_dkdv_tc_kernel<D><<<static_cast<unsigned>(ctas), C::kThreads, C::kSmemBytes, st>>>(
        mQ, mdO, mK, mV, mQg, mdOg, mKc, mVc, kp);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int D>
cudaError_t launch_dq_d(const BwdTcArgs& a, cudaStream_t st, const char** why) {
  using C = DqCfg<D>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(bwd_dq_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const long long T = a.mask.T;  // rows per residue class
  const long long dv = a.dview;
  CUtensorMap mQ, mdO, mK, mV, mQg, mdOg, mKc, mVc;
  bool ok = make_map(&mQ, a.Q, D, T, a.BH, dv) && make_map(&mdO, a.dO, D, T, a.BH, dv) &&
            make_map(&mK, a.K, D, T, a.BH, dv) && make_map(&mV, a.V, D, T, a.BH, dv);
  ok = ok && (a.n_cols > 0 ? make_map(&mKc, a.Kc, D, a.n_cols, a.BH) && make_map(&mVc, a.Vc, D, a.n_cols, a.BH)
                           : (mKc = mK, mVc = mV, true));
  ok = ok && (a.mask.n_global > 0 ? make_map(&mQg, a.Qg, D, a.mask.n_global, a.BH) &&
                                        make_map(&mdOg, a.dOg, D, a.mask.n_global, a.BH)
                                  : (mQg = mQ, mdOg = mdO, true));
  if (!ok) {
    *why = "cuTensorMapEncodeTiled failed";
    return cudaErrorInvalidValue;
  }
  DqParams kp;
  kp.dQ = static_cast<__nv_bfloat16*>(a.dQ);
  kp.LSE = a.LSE;
  kp.Dvec = a.Dvec;
  kp.scale = a.scale;
  kp.scale_log2 = a.scale * 1.4426950408889634f;
  kp.colmask = a.colmask;
  kp.mask = a.mask;
  kp.items = a.items;
  kp.entries = a.entries;
  kp.err = a.err;
  kp.budget = a.wait_budget_cycles;
  kp.BH = a.BH * static_cast<int>(dv);
  kp.dview = static_cast<int>(dv);
  kp.T_out = static_cast<int>(T * dv);
  const long long ctas = static_cast<long long>(a.n_items) * 2 * a.BH * dv;
  if (ctas > 0x7fffffffLL) {
    *why = "too many work items";
    return cudaErrorInvalidValue;
  }
  bwd_dq_tc_kernel<D><<<static_cast<unsigned>(ctas), C::kThreads, C::kSmemBytes, st>>>(
      mQ, mdO, mK, mV, mQg, mdOg, mKc, mVc, kp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv_tc(int d, const BwdTcArgs& a, cudaStream_t st, const char** why) {
  if (d == 64) return launch_kv_d<64>(a, st, why);
  if (d == 128) return launch_kv_d<128>(a, st, why);
  *why = "head dim must be 64 or 128";
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dq_tc(int d, const BwdTcArgs& a, cudaStream_t st, const char** why) {
  if (a.n_items == 0) return cudaSuccess;
  if (d == 64) return launch_dq_d<64>(a, st, why);
  if (d == 128) return launch_dq_d<128>(a, st, why);
  *why = "head dim must be 64 or 128";
  return cudaErrorInvalidValue;
}

}  // namespace spattn
