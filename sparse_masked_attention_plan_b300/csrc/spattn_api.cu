// spattn_api.cu -- the C ABI (include/spattn.h): spec validation, plan building
// (GPU kernels + host scheduler), forward dispatch, errors.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "internal.h"
#include "spattn.h"

using spattn::kTile;

namespace {

thread_local std::string g_last_error;

spattn_status fail(spattn_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

#define CUDA_TRY(expr)                                                                  \
  do {                                                                                  \
    cudaError_t e_ = (expr);                                                            \
    if (e_ != cudaSuccess)                                                              \
      return fail(SPATTN_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_));     \
  } while (0)

constexpr int64_t kMaxT = int64_t(1) << 30;

template <typename T>
cudaError_t dev_alloc(T** p, size_t n) {
  return cudaMalloc(reinterpret_cast<void**>(p), std::max<size_t>(n, 1) * sizeof(T));
}

void free_plan_memory(spattn_plan* p) {
  void* ptrs[] = {p->d_tile_qb, p->d_tile_kb, p->d_tile_cnt, p->d_tile_cls, p->d_cols,
                  p->d_colmask, p->d_rowglobal, p->d_gpos, p->d_gpos_ns, p->d_scratch,
                  p->d_walk, p->d_err, p->sched[0].d_items, p->sched[0].d_entries,
                  p->sched[1].d_items, p->sched[1].d_entries, p->sched[2].d_items,
                  p->sched[2].d_entries, p->d_colmask_res, p->d_rowzero,
                  p->bsched.d_items, p->bsched.d_entries, p->d_colidx, p->d_bscratch,
                  p->d_roff, p->d_rkb, p->bsched_tc.d_items, p->bsched_tc.d_entries,
                  p->d_rtoff, p->d_rtqb, p->bsched_res.d_items, p->bsched_res.d_entries};
  for (void* q : ptrs)
    if (q) cudaFree(q);
  for (cudaEvent_t e : p->host_ev)
    if (e) cudaEventDestroy(e);
  if (p->host_in) cudaStreamDestroy(p->host_in);
  if (p->host_out) cudaStreamDestroy(p->host_out);
}

// ---- host scheduler ---------------------------------------------------------------
//
// A work item is a group of `group_rows` query rows split into `n_qtiles` query
// tiles of `qtile_rows`.  Its entries are (1) the band key tiles of the natural grid
// that the local rule of its rows reaches, and (2) chunks of up to 128 packed sparse
// columns that lie outside that band.  Each entry records which query tiles have at
// least one allowed pair in it (the others skip it) and which need no predicate.
// Global rows get their own items that walk every key tile their causality permits.

struct Sched {
  const spattn_plan* p;
  int64_t lower(int64_t v) const {  // #C < v
    return std::lower_bound(p->cols.begin(), p->cols.end(), static_cast<int32_t>(
                                std::min<int64_t>(v, INT32_MAX))) - p->cols.begin();
  }
  int64_t upper(int64_t v) const {  // #C <= v
    return std::upper_bound(p->cols.begin(), p->cols.end(), static_cast<int32_t>(
                                std::min<int64_t>(v, INT32_MAX))) - p->cols.begin();
  }
  static int64_t floor_div(int64_t x, int64_t d) { return x >= 0 ? x / d : -((-x + d - 1) / d); }
  // Is a multiple of the dilation inside [lo, hi]?
  bool grid_in(int64_t lo, int64_t hi) const {
    if (lo > hi) return false;
    const int64_t d = p->dilation;
    return (floor_div(lo + d - 1, d)) * d <= hi;
  }
  // Any (i in [a,b], j in [k0,k1]) allowed by the local rule?  (The distances i - j
  // of such pairs fill [a - k1, b - k0]; the rule wants one on the dilation grid.)
  bool local_meets(int64_t a, int64_t b, int64_t k0, int64_t k1) const {
    const int64_t d = p->dilation;
    if (p->causal) {
      const int64_t hi = p->window ? std::min(b - k0, (p->window - 1) * d) : b - k0;
      return grid_in(std::max<int64_t>(0, a - k1), hi);
    }
    int64_t lo = a - k1, hi = b - k0;
    if (p->radius >= 0) {
      lo = std::max(lo, -p->radius * d);
      hi = std::min(hi, p->radius * d);
    }
    return grid_in(lo, hi);
  }
  // Every (i in [a,b], j in [k0,k1]) allowed by the local rule?  (never with a dilation)
  bool local_covers(int64_t a, int64_t b, int64_t k0, int64_t k1) const {
    if (p->dilation > 1) return false;
    if (p->causal) return k1 <= a && (p->window == 0 || b - k0 < p->window);
    if (p->radius < 0) return true;
    return b - k0 <= p->radius && k1 - a <= p->radius;
  }
  bool cols_in(int64_t x, int64_t y) const { return y >= x && upper(y) - lower(x) > 0; }
  // Does a random block of the rows [a, b] reach a key in [k0, k1] (causal: k <= b)?
  bool rand_in(int64_t a, int64_t b, int64_t k0, int64_t k1) const {
    if (p->r_kb.empty() || a > b) return false;
    if (p->causal) k1 = std::min(k1, b);
    if (k0 > k1) return false;
    const int64_t rb = p->rand_block;
    for (int64_t q = a / rb; q <= b / rb; ++q)
      for (int32_t x = p->r_off[q]; x < p->r_off[q + 1]; ++x) {
        const int64_t c0 = int64_t(p->r_kb[x]) * rb, c1 = c0 + rb - 1;
        if (c0 <= k1 && c1 >= k0) return true;
      }
    return false;
  }
  // The natural key tiles (of `tile` keys) that random blocks of rows [a, b] reach.
  void rand_tiles(int64_t a, int64_t b, int64_t tile, std::vector<int64_t>* out) const {
    if (p->r_kb.empty()) return;
    const int64_t rb = p->rand_block;
    for (int64_t q = a / rb; q <= b / rb; ++q)
      for (int32_t x = p->r_off[q]; x < p->r_off[q + 1]; ++x)
        out->push_back(int64_t(p->r_kb[x]) * rb / tile);
  }
};

void build_schedule(const spattn_plan* p, spattn::Schedule* s, int group_rows, int qtile_rows,
                    int n_qtiles, bool longest_first) {
  using namespace spattn;
  Sched h{p};
  const int64_t T = p->T;
  const int64_t nc = p->n_cols;
  s->group_rows = group_rows;
  s->qtile_rows = qtile_rows;
  s->n_qtiles = n_qtiles;
  s->items.clear();
  s->entries.clear();
  s->tile_products = 0;
  struct Item { int32_t q0, off, cnt, flags; };
  std::vector<Item> items;
  auto push = [&](int32_t src, int32_t flags, int32_t kb, int32_t lim) {
    s->entries.insert(s->entries.end(), {src, flags, kb, lim});
    s->tile_products += ((flags & kActive0) ? 1 : 0) + ((flags & kActive1) ? 1 : 0);
  };
  const int64_t n_groups = (T + group_rows - 1) / group_rows;
  for (int64_t g = 0; g < n_groups; ++g) {
    const int64_t r0 = g * group_rows, r1 = std::min<int64_t>(r0 + group_rows, T) - 1;
    int64_t jlo, jhi;
    const int64_t d = p->dilation;
    if (p->causal) {
      jlo = p->window ? std::max<int64_t>(0, r0 - (p->window - 1) * d) : 0;
      jhi = r1;
    } else {
      jlo = p->radius >= 0 ? std::max<int64_t>(0, r0 - p->radius * d) : 0;
      jhi = p->radius >= 0 ? std::min<int64_t>(T - 1, r1 + p->radius * d) : T - 1;
    }
    const int64_t kb_lo = jlo / kTile, kb_hi = jhi / kTile;
    const int32_t off = static_cast<int32_t>(s->entries.size() / 4);
    for (int64_t kb = kb_lo; kb <= kb_hi; ++kb) {
      const int64_t k0 = kb * kTile, k1 = std::min<int64_t>(k0 + kTile, T) - 1;
      const bool ragged = k0 + kTile > T;
      int32_t flags = kKindBand << kKindShift;
      for (int t = 0; t < n_qtiles; ++t) {
        const int64_t a = r0 + int64_t(t) * qtile_rows;
        if (a >= T) continue;
        const int64_t b = std::min<int64_t>(a + qtile_rows, T) - 1;
        const bool active = h.local_meets(a, b, k0, k1) ||
                            h.cols_in(k0, p->causal ? std::min(k1, b) : k1) ||
                            h.rand_in(a, b, k0, k1);
        if (!active) continue;
        flags |= kActive0 << t;
        if (!ragged && h.local_covers(a, b, k0, k1)) flags |= kFull0 << t;
      }
      if (flags & (kActive0 | kActive1)) push(static_cast<int32_t>(k0), flags, static_cast<int32_t>(kb), 0);
    }
    {  // key tiles outside the band that random blocks of the group's rows reach
      std::vector<int64_t> rt;
      h.rand_tiles(r0, r1, kTile, &rt);
      std::sort(rt.begin(), rt.end());
      rt.erase(std::unique(rt.begin(), rt.end()), rt.end());
      for (int64_t kb : rt) {
        if (kb >= kb_lo && kb <= kb_hi) continue;
        const int64_t k0 = kb * kTile, k1 = std::min<int64_t>(k0 + kTile, T) - 1;
        int32_t flags = kKindRandom << kKindShift;
        for (int t = 0; t < n_qtiles; ++t) {
          const int64_t a = r0 + int64_t(t) * qtile_rows;
          if (a >= T) continue;
          const int64_t b = std::min<int64_t>(a + qtile_rows, T) - 1;
          if (h.rand_in(a, b, k0, k1)) flags |= kActive0 << t;
        }
        if (flags & (kActive0 | kActive1)) push(static_cast<int32_t>(k0), flags, static_cast<int32_t>(kb), 0);
      }
    }
    if (nc > 0) {
      const int64_t a_idx = h.lower(kb_lo * kTile), b_idx = h.lower((kb_hi + 1) * kTile);
      const int64_t e_idx = p->causal ? h.upper(r1) : nc;
      const int64_t ranges[2][2] = {{0, std::min(a_idx, e_idx)}, {b_idx, e_idx}};
      for (auto& rg : ranges) {
        for (int64_t s0 = rg[0]; s0 < rg[1]; s0 += kTile) {
          const int64_t lim = rg[1];
          int32_t flags = kKindPacked << kKindShift;
          for (int t = 0; t < n_qtiles; ++t) {
            const int64_t a = r0 + int64_t(t) * qtile_rows;
            if (a >= T) continue;
            const int64_t b = std::min<int64_t>(a + qtile_rows, T) - 1;
            // causal: packed columns precede the band, so every row reads them
            if (p->causal && p->cols[s0] > b) continue;
            flags |= kActive0 << t;
            const bool whole = s0 + kTile <= lim &&
                               (!p->causal || p->cols[s0 + kTile - 1] <= a);
            if (whole) flags |= kFull0 << t;
          }
          if (flags & (kActive0 | kActive1))
            push(static_cast<int32_t>(s0), flags, -1, static_cast<int32_t>(lim));
        }
      }
    }
    const int32_t cnt = static_cast<int32_t>(s->entries.size() / 4) - off;
    if (cnt > 0) items.push_back({static_cast<int32_t>(r0), off, cnt, 0});
  }
  // global rows: every key that causality permits.  A group whose rows fit in one
  // query tile is split (d = 64 only, where it was measured faster): both tiles hold its
  // rows and take alternate key tiles, so the dense walk that every global row needs
  // runs at two tiles per entry pair.
  const int64_t ng = static_cast<int64_t>(p->gpos.size());
  for (int64_t q0 = 0; q0 < ng; q0 += group_rows) {
    const int32_t off = static_cast<int32_t>(s->entries.size() / 4);
    const int64_t last = p->gpos[std::min<int64_t>(q0 + group_rows, ng) - 1];
    const int64_t kb_hi = (p->causal ? last : T - 1) / kTile;
    const bool split = n_qtiles == 2 && p->d == 64 && ng - q0 <= qtile_rows && kb_hi >= 1;
    for (int64_t kb = 0; kb <= kb_hi; ++kb) {
      const int64_t k0 = kb * kTile, k1 = std::min<int64_t>(k0 + kTile, T) - 1;
      const bool ragged = k0 + kTile > T;
      int32_t flags = kKindDense << kKindShift;
      for (int t = 0; t < n_qtiles; ++t) {
        const int64_t a = q0 + (split ? 0 : int64_t(t) * qtile_rows);
        if (a >= ng) continue;
        if (split && t != (kb & 1)) continue;
        const int64_t b = std::min<int64_t>(a + qtile_rows, ng) - 1;
        const int64_t rmin = p->gpos[a], rmax = p->gpos[b];
        if (p->causal && k0 > rmax) continue;
        flags |= kActive0 << t;
        if (!ragged && (!p->causal || k1 <= rmin)) flags |= kFull0 << t;
      }
      if (flags & (kActive0 | kActive1)) push(static_cast<int32_t>(k0), flags, static_cast<int32_t>(kb), 0);
    }
    const int32_t cnt = static_cast<int32_t>(s->entries.size() / 4) - off;
    if (cnt > 0)
      items.push_back({static_cast<int32_t>(q0), off, cnt, kItemGathered | (split ? kItemSplit : 0)});
  }
  {
    const int64_t n_ent = static_cast<int64_t>(s->entries.size() / 4);
    s->mma_per_tile = (p->d == 64 && n_qtiles == 2 && 5 * s->tile_products < 8 * n_ent) ? 1 : 0;
  }
  if (longest_first)
    std::stable_sort(items.begin(), items.end(),
                     [](const Item& x, const Item& y) { return x.cnt > y.cnt; });
  for (const Item& it : items) s->items.insert(s->items.end(), {it.q0, it.off, it.cnt, it.flags});
  // items much longer than the median (e.g. gathered global rows that read every key)
  // are launched first for every head, so they do not end up in the last wave
  s->n_major = 0;
  if (longest_first && !items.empty()) {
    const int32_t median = items[items.size() / 2].cnt;
    while (s->n_major < static_cast<int32_t>(items.size()) &&
           2 * items[s->n_major].cnt >= 3 * median && items[s->n_major].cnt > median)
      ++s->n_major;
  }
}

// Key-major schedule of the backward pass: the same decomposition of every row's
// allowed set as the forward schedule (band keys of the natural grid inside the
// group's band range, packed sparse columns outside it, random-block tiles, dense
// walks for global rows), with groups of kRows query rows listed per unit of kKeys
// keys instead of per query group, so that the gradient of every key is summed inside
// one CTA.  kKeys divides the 128-key tile; kRows is 64 or 128.
void build_bwd_schedule(const spattn_plan* p, spattn::Schedule* s, int64_t kRows,
                        int64_t kKeys) {
  using namespace spattn;
  Sched h{p};
  const int64_t T = p->T;
  const int64_t nc = p->n_cols;
  const int64_t nu_nat = (T + kKeys - 1) / kKeys, nu_pk = (nc + kKeys - 1) / kKeys;
  std::vector<std::vector<int32_t>> nat(nu_nat), pk(nu_pk);
  auto add = [](std::vector<int32_t>& v, int64_t q0, int32_t flags, int64_t a, int64_t b) {
    v.insert(v.end(), {static_cast<int32_t>(q0), flags, static_cast<int32_t>(a),
                       static_cast<int32_t>(b)});
  };
  const int64_t d = p->dilation;
  for (int64_t r0 = 0; r0 < T; r0 += kRows) {
    const int64_t r1 = std::min<int64_t>(r0 + kRows, T) - 1;
    int64_t jlo, jhi;
    if (p->causal) {
      jlo = p->window ? std::max<int64_t>(0, r0 - (p->window - 1) * d) : 0;
      jhi = r1;
    } else {
      jlo = p->radius >= 0 ? std::max<int64_t>(0, r0 - p->radius * d) : 0;
      jhi = p->radius >= 0 ? std::min<int64_t>(T - 1, r1 + p->radius * d) : T - 1;
    }
    const int64_t kb_lo = jlo / kTile, kb_hi = jhi / kTile;
    const int64_t u_hi = std::min<int64_t>(nu_nat - 1, (kb_hi + 1) * (kTile / kKeys) - 1);
    for (int64_t u = kb_lo * (kTile / kKeys); u <= u_hi; ++u) {
      const int64_t k0 = u * kKeys, k1 = std::min<int64_t>(k0 + kKeys, T) - 1;
      if (h.local_meets(r0, r1, k0, k1) || h.cols_in(k0, p->causal ? std::min(k1, r1) : k1) ||
          h.rand_in(r0, r1, k0, k1)) {
        // every pair inside the local window: causal 0 <= i - j < window, else
        // |i - j| <= radius (contiguous windows only)
        bool full = d == 1;
        if (p->causal)
          full = full && k1 <= r0 && (p->window == 0 || r1 - k0 < p->window);
        else
          full = full && (p->radius < 0 || (r1 - k0 <= p->radius && k1 - r0 <= p->radius));
        add(nat[u], r0, (kKindBand << kKindShift) | (full ? kEntryFull : 0), 0, 0);
      }
    }
    {  // units outside the band range that random blocks of the group's rows reach
      std::vector<int64_t> ru;
      h.rand_tiles(r0, r1, kKeys, &ru);
      std::vector<int64_t> all;
      for (int64_t u0 : ru)  // a random block of b keys spans b / 64 units (or part of one)
        for (int64_t u = u0; u < u0 + std::max<int64_t>(1, p->rand_block / kKeys); ++u)
          all.push_back(u);
      std::sort(all.begin(), all.end());
      all.erase(std::unique(all.begin(), all.end()), all.end());
      const int64_t band_u0 = kb_lo * (kTile / kKeys);
      for (int64_t u : all) {
        if (u >= nu_nat || (u >= band_u0 && u <= u_hi)) continue;
        const int64_t k0 = u * kKeys, k1 = std::min<int64_t>(k0 + kKeys, T) - 1;
        if (h.rand_in(r0, r1, k0, k1)) add(nat[u], r0, kKindRandom << kKindShift, 0, 0);
      }
    }
    if (nc > 0) {
      const int64_t a_idx = h.lower(kb_lo * kTile), b_idx = h.lower((kb_hi + 1) * kTile);
      const int64_t e_idx = p->causal ? h.upper(r1) : nc;
      const int64_t ranges[2][2] = {{0, std::min(a_idx, e_idx)}, {b_idx, e_idx}};
      for (auto& rg : ranges)
        for (int64_t u = rg[0] / kKeys; rg[0] < rg[1] && u <= (rg[1] - 1) / kKeys; ++u)
          add(pk[u], r0, kKindPacked << kKindShift, std::max(rg[0], u * kKeys),
              std::min(rg[1], (u + 1) * kKeys));
    }
  }
  const int64_t ng = static_cast<int64_t>(p->gpos.size());
  for (int64_t q0 = 0; q0 < ng; q0 += kRows) {
    const int64_t last = p->gpos[std::min<int64_t>(q0 + kRows, ng) - 1];
    const int64_t u_hi = (p->causal ? last : T - 1) / kKeys;
    for (int64_t u = 0; u <= u_hi; ++u)
      add(nat[u], q0, (kKindDense << kKindShift) | kEntryGathered, 0, 0);
  }
  s->group_rows = kRows;
  s->qtile_rows = kRows;
  s->n_qtiles = 1;
  s->items.clear();
  s->entries.clear();
  s->tile_products = 0;
  s->n_major = 0;
  s->n_packed_units = static_cast<int32_t>(nu_pk);
  auto emit = [&](std::vector<int32_t>& v, int64_t key0, int32_t flags) {
    const int32_t off = static_cast<int32_t>(s->entries.size() / 4);
    const int32_t cnt = static_cast<int32_t>(v.size() / 4);
    s->items.insert(s->items.end(), {static_cast<int32_t>(key0), off, cnt, flags});
    s->entries.insert(s->entries.end(), v.begin(), v.end());
    s->tile_products += cnt;
  };
  for (int64_t u = 0; u < nu_pk; ++u) emit(pk[u], u * kKeys, kUnitPacked);
  for (int64_t u = 0; u < nu_nat; ++u) emit(nat[u], u * kKeys, 0);
}

spattn_status upload_schedule(spattn::Schedule* s) {
  const size_t ni = s->items.size() / 4, ne = s->entries.size() / 4;
  CUDA_TRY(dev_alloc(&s->d_items, ni));
  CUDA_TRY(dev_alloc(&s->d_entries, ne));
  if (ni) CUDA_TRY(cudaMemcpy(s->d_items, s->items.data(), ni * sizeof(int4), cudaMemcpyHostToDevice));
  if (ne)
    CUDA_TRY(cudaMemcpy(s->d_entries, s->entries.data(), ne * sizeof(int4), cudaMemcpyHostToDevice));
  return SPATTN_OK;
}

spattn_status check_ptr(const void* p, const char* name) {
  if (!p) return fail(SPATTN_ERR_NULL, "%s is NULL", name);
  if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
    return fail(SPATTN_ERR_ALIGN, "%s is not 16-byte aligned", name);
  return SPATTN_OK;
}

}  // namespace

void spattn::set_last_error(const char* msg) { g_last_error = msg; }

void spattn::select_schedule(const spattn_plan* p, bool bf16, TcArgs* a) {
  const bool view = bf16 && p->dview > 1;
  const spattn::Schedule& s = p->sched[view ? 2 : (bf16 ? 0 : 1)];
  a->items = s.d_items;
  a->entries = s.d_entries;
  a->n_items = static_cast<int32_t>(s.items.size() / 4);
  a->n_major = s.n_major;
  a->mask = view ? p->mask_dev_res() : p->mask_dev();
  a->colmask = view ? p->d_colmask_res : p->d_colmask;
  a->n_cols = view ? 0 : p->n_cols;
  a->dview = view ? p->dview : 1;
  a->mma_per_tile = s.mma_per_tile;
}

void spattn::fill_fwd_args(const spattn_plan* p, bool bf16, int64_t BH, const void* Q,
                           const void* K, const void* V, void* Kc, void* Vc, void* Qg, void* O,
                           float* LSE, float scale, TcArgs* a) {
  a->Q = Q;
  a->K = K;
  a->V = V;
  a->Kc = Kc ? Kc : K;
  a->Vc = Vc ? Vc : V;
  a->Qg = Qg ? Qg : Q;
  a->O = O;
  a->LSE = LSE;
  a->BH = static_cast<int32_t>(BH);
  a->n_cols = p->n_cols;
  a->scale = scale;
  a->walk = p->walk_enabled ? p->d_walk : nullptr;
  a->err = p->d_err;
  a->wait_budget_cycles = p->wait_budget_cycles;
  a->inject_timeout = p->inject_timeout;
  select_schedule(p, bf16, a);
}

extern "C" {

const char* spattn_last_error(void) { return g_last_error.c_str(); }

const char* spattn_version(void) { return "spattn 0.1 (sm_103a tcgen05)"; }

spattn_status spattn_mask_validate(const spattn_mask_spec* spec, int64_t T) {
  if (!spec) return fail(SPATTN_ERR_NULL, "spec is NULL");
  if (T < 1 || T > kMaxT) return fail(SPATTN_ERR_SHAPE, "T=%lld outside [1, 2^30]", (long long)T);
  if (spec->causal != 0 && spec->causal != 1)
    return fail(SPATTN_ERR_INVALID_SPEC, "causal must be 0 or 1");
  if (spec->causal) {
    if (spec->window < 0) return fail(SPATTN_ERR_INVALID_SPEC, "window must be >= 0");
    if (spec->radius != -1) return fail(SPATTN_ERR_INVALID_SPEC, "causal mask takes radius = -1");
  } else {
    if (spec->radius < -1) return fail(SPATTN_ERR_INVALID_SPEC, "radius must be >= -1");
    if (spec->window != 0) return fail(SPATTN_ERR_INVALID_SPEC, "bidirectional mask takes window = 0");
  }
  if (spec->dilation < 0 || spec->dilation > (int64_t(1) << 31))
    return fail(SPATTN_ERR_INVALID_SPEC, "dilation must lie in [0, 2^31]");
  if (spec->dilation > 1 && (spec->window > (int64_t(1) << 31) || spec->radius > (int64_t(1) << 31)))
    return fail(SPATTN_ERR_INVALID_SPEC, "with a dilation, window and radius must be <= 2^31");
  if (spec->stride < 0) return fail(SPATTN_ERR_INVALID_SPEC, "stride must be >= 0");
  if (spec->stride == 0 && spec->stride_offset != 0)
    return fail(SPATTN_ERR_INVALID_SPEC, "stride_offset must be 0 without a stride");
  if (spec->stride > 0 && (spec->stride_offset < 0 || spec->stride_offset >= spec->stride))
    return fail(SPATTN_ERR_INVALID_SPEC, "stride_offset must lie in [0, stride)");
  if (spec->n_global < 0 || spec->n_global > T)
    return fail(SPATTN_ERR_INVALID_SPEC, "n_global must lie in [0, T]");
  if (spec->n_global > 0) {
    if (!spec->global_pos) return fail(SPATTN_ERR_NULL, "global_pos is NULL");
    std::vector<int32_t> g(spec->global_pos, spec->global_pos + spec->n_global);
    for (int32_t x : g)
      if (x < 0 || x >= T) return fail(SPATTN_ERR_INVALID_SPEC, "global position %d outside [0, T)", x);
    std::sort(g.begin(), g.end());
    for (size_t a = 1; a < g.size(); ++a)
      if (g[a] == g[a - 1]) return fail(SPATTN_ERR_INVALID_SPEC, "duplicate global position %d", g[a]);
  }
  if (spec->n_rand < 0) return fail(SPATTN_ERR_INVALID_SPEC, "n_rand must be >= 0");
  if (spec->n_rand > 0) {
    const int64_t b = spec->rand_block;
    if (b != 16 && b != 32 && b != 64 && b != 128)
      return fail(SPATTN_ERR_INVALID_SPEC, "rand_block must be 16, 32, 64 or 128");
    if (!spec->rand_pairs) return fail(SPATTN_ERR_NULL, "rand_pairs is NULL");
    const int64_t nb = (T + b - 1) / b;
    if (spec->n_rand > nb * nb) return fail(SPATTN_ERR_INVALID_SPEC, "more random pairs than blocks");
    std::vector<int64_t> keys(static_cast<size_t>(spec->n_rand));
    for (int64_t a = 0; a < spec->n_rand; ++a) {
      const int64_t q = spec->rand_pairs[2 * a], k = spec->rand_pairs[2 * a + 1];
      if (q < 0 || q >= nb || k < 0 || k >= nb)
        return fail(SPATTN_ERR_INVALID_SPEC, "random pair (%lld, %lld) outside [0, %lld)",
                    (long long)q, (long long)k, (long long)nb);
      keys[a] = q * nb + k;
    }
    std::sort(keys.begin(), keys.end());
    for (size_t a = 1; a < keys.size(); ++a)
      if (keys[a] == keys[a - 1]) return fail(SPATTN_ERR_INVALID_SPEC, "duplicate random pair");
  }
  return SPATTN_OK;
}

spattn_status spattn_plan_create(const spattn_mask_spec* spec, int64_t T, int32_t head_dim,
                                 void* cuda_stream, spattn_plan** out) {
  if (!out) return fail(SPATTN_ERR_NULL, "out is NULL");
  *out = nullptr;
  spattn_status st = spattn_mask_validate(spec, T);
  if (st != SPATTN_OK) return st;
  if (head_dim != 64 && head_dim != 128)
    return fail(SPATTN_ERR_SHAPE, "head_dim %d not supported (64 or 128)", head_dim);
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);

  spattn_plan* p = new spattn_plan();
  auto bail = [&](spattn_status s) {
    free_plan_memory(p);
    delete p;
    return s;
  };
  // normalise: widths beyond T describe the same set as T
  p->T = T;
  p->d = head_dim;
  p->causal = spec->causal;
  p->window = std::min<int64_t>(spec->window, T);
  p->radius = spec->radius < 0 ? -1 : std::min<int64_t>(spec->radius, T);
  p->dilation = spec->dilation < 1 ? 1 : spec->dilation;
  if (p->dilation >= T) {  // only distance 0 is a multiple of d below T: each row reads itself
    if (p->causal) p->window = 1; else p->radius = 0;
    p->dilation = 1;
  }
  if (p->dilation > 1) {  // spans reaching past the sequence are the unbounded window
    if (p->causal && p->window > 0 && (p->window - 1) * p->dilation >= T) p->window = 0;
    if (!p->causal && p->radius >= 0 && p->radius * p->dilation >= T) p->radius = -1;
  }
  p->stride = spec->stride;
  p->offset = spec->stride_offset;
  if (p->stride > T) {  // at most one strided column, j == offset
    if (p->offset < T) p->stride = T; else { p->stride = 0; p->offset = 0; }
  }
  if (spec->n_rand > 0) {  // random blocks as CSR: query block -> ascending key blocks
    const int64_t b = spec->rand_block, nb = (T + b - 1) / b;
    std::vector<std::pair<int32_t, int32_t>> pr;
    for (int64_t a = 0; a < spec->n_rand; ++a)
      pr.emplace_back(spec->rand_pairs[2 * a], spec->rand_pairs[2 * a + 1]);
    std::sort(pr.begin(), pr.end());
    p->rand_block = static_cast<int32_t>(b);
    p->r_off.assign(static_cast<size_t>(nb) + 1, 0);
    for (auto& x : pr) {
      ++p->r_off[x.first + 1];
      p->r_kb.push_back(x.second);
    }
    for (int64_t q = 0; q < nb; ++q) p->r_off[q + 1] += p->r_off[q];
  }
  p->gpos.assign(spec->global_pos, spec->global_pos + spec->n_global);
  std::sort(p->gpos.begin(), p->gpos.end());
  for (int32_t x : p->gpos)
    if (!(p->stride > 0 && x % p->stride == p->offset)) p->gpos_ns.push_back(x);
  if (cudaGetDevice(&p->device) != cudaSuccess)
    return bail(fail(SPATTN_ERR_CUDA, "no CUDA device"));

  p->nqb = static_cast<int32_t>((T + kTile - 1) / kTile);
  p->nkb = p->nqb;
  const int32_t Ti = static_cast<int32_t>(T);
  uint8_t* d_flags = nullptr;
  int32_t* d_ncols = nullptr;
  int32_t *d_qne = nullptr, *d_qfull = nullptr, *d_qoff = nullptr;
  long long* d_qpairs = nullptr;
  auto cleanup_tmp = [&] {
    cudaFree(d_flags);
    cudaFree(d_ncols);
    cudaFree(d_qne);
    cudaFree(d_qfull);
    cudaFree(d_qoff);
    cudaFree(d_qpairs);
  };
#define PLAN_TRY(expr)                                                                 \
  do {                                                                                 \
    cudaError_t e_ = (expr);                                                           \
    if (e_ != cudaSuccess) {                                                           \
      cleanup_tmp();                                                                   \
      return bail(fail(SPATTN_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_))); \
    }                                                                                  \
  } while (0)

  PLAN_TRY(dev_alloc(&p->d_roff, p->r_off.size()));
  PLAN_TRY(dev_alloc(&p->d_rkb, p->r_kb.size()));
  if (!p->r_kb.empty()) {
    PLAN_TRY(cudaMemcpy(p->d_roff, p->r_off.data(), p->r_off.size() * 4, cudaMemcpyHostToDevice));
    PLAN_TRY(cudaMemcpy(p->d_rkb, p->r_kb.data(), p->r_kb.size() * 4, cudaMemcpyHostToDevice));
  }
  PLAN_TRY(dev_alloc(&p->d_gpos, p->gpos.size()));
  PLAN_TRY(dev_alloc(&p->d_gpos_ns, p->gpos_ns.size()));
  if (!p->gpos.empty())
    PLAN_TRY(cudaMemcpy(p->d_gpos, p->gpos.data(), p->gpos.size() * 4, cudaMemcpyHostToDevice));
  if (!p->gpos_ns.empty())
    PLAN_TRY(cudaMemcpy(p->d_gpos_ns, p->gpos_ns.data(), p->gpos_ns.size() * 4, cudaMemcpyHostToDevice));
  PLAN_TRY(dev_alloc(&p->d_rowglobal, T));
  PLAN_TRY(dev_alloc(&p->d_colmask, size_t(p->nkb) * 4));
  PLAN_TRY(dev_alloc(&p->d_cols, T));
  PLAN_TRY(dev_alloc(&d_flags, T));
  PLAN_TRY(dev_alloc(&d_ncols, 1));
  PLAN_TRY(dev_alloc(&p->d_walk, 1));
  PLAN_TRY(dev_alloc(&p->d_err, 1));
  PLAN_TRY(cudaMemsetAsync(p->d_walk, 0, sizeof(unsigned long long), stream));
  PLAN_TRY(cudaMemsetAsync(p->d_err, 0, sizeof(int), stream));
  const spattn::MaskDev m = p->mask_dev();

  // sparse columns: flags -> compacted list -> per-key-block bit masks
  PLAN_TRY(spattn::launch_column_flags(m, d_flags, p->d_rowglobal, stream));
  PLAN_TRY(spattn::launch_compact_columns(d_flags, Ti, p->d_cols, d_ncols, stream));
  PLAN_TRY(spattn::launch_colmask(d_flags, Ti, p->nkb, p->d_colmask, stream));
  int32_t ncols = 0;
  PLAN_TRY(cudaMemcpyAsync(&ncols, d_ncols, 4, cudaMemcpyDeviceToHost, stream));
  PLAN_TRY(cudaStreamSynchronize(stream));
  p->n_cols = ncols;
  p->cols.resize(ncols);
  if (ncols) PLAN_TRY(cudaMemcpy(p->cols.data(), p->d_cols, size_t(ncols) * 4, cudaMemcpyDeviceToHost));

  // natural-grid classification: count pass, offsets, fill pass
  PLAN_TRY(dev_alloc(&d_qne, p->nqb));
  PLAN_TRY(dev_alloc(&d_qfull, p->nqb));
  PLAN_TRY(dev_alloc(&d_qoff, p->nqb));
  PLAN_TRY(dev_alloc(&d_qpairs, p->nqb));
  PLAN_TRY(spattn::launch_tile_count(m, p->d_colmask, p->nqb, p->nkb, d_qne, d_qfull, d_qpairs, stream));
  std::vector<int32_t> qne(p->nqb), qfull(p->nqb), qoff(p->nqb);
  std::vector<long long> qpairs(p->nqb);
  PLAN_TRY(cudaMemcpyAsync(qne.data(), d_qne, size_t(p->nqb) * 4, cudaMemcpyDeviceToHost, stream));
  PLAN_TRY(cudaMemcpyAsync(qfull.data(), d_qfull, size_t(p->nqb) * 4, cudaMemcpyDeviceToHost, stream));
  PLAN_TRY(cudaMemcpyAsync(qpairs.data(), d_qpairs, size_t(p->nqb) * 8, cudaMemcpyDeviceToHost, stream));
  PLAN_TRY(cudaStreamSynchronize(stream));
  int64_t total = 0;
  for (int32_t q = 0; q < p->nqb; ++q) {
    qoff[q] = static_cast<int32_t>(total);
    total += qne[q];
    p->n_full += qfull[q];
    p->pairs += qpairs[q];
  }
  p->n_nonempty = total;
  p->n_partial = total - p->n_full;
  p->n_empty = int64_t(p->nqb) * p->nkb - total;
  PLAN_TRY(dev_alloc(&p->d_tile_qb, total));
  PLAN_TRY(dev_alloc(&p->d_tile_kb, total));
  PLAN_TRY(dev_alloc(&p->d_tile_cnt, total));
  PLAN_TRY(dev_alloc(&p->d_tile_cls, total));
  PLAN_TRY(cudaMemcpyAsync(d_qoff, qoff.data(), size_t(p->nqb) * 4, cudaMemcpyHostToDevice, stream));
  PLAN_TRY(spattn::launch_tile_fill(m, p->d_colmask, p->nqb, p->nkb, d_qoff, p->d_tile_qb,
                                    p->d_tile_kb, p->d_tile_cnt, p->d_tile_cls, stream));
  PLAN_TRY(cudaStreamSynchronize(stream));
  cleanup_tmp();
#undef PLAN_TRY

  // execution schedules
  build_schedule(p, &p->sched[0], 2 * kTile, kTile, 2, true);
  build_schedule(p, &p->sched[1], 64, 64, 1, true);
  if (p->dilation > 1 && p->stride == 0 && p->gpos.empty() && p->r_kb.empty() &&
      T % p->dilation == 0) {
    // dilated view: residue class r holds rows r, r + d, ...; there the dilated
    // window is a contiguous window of the same width over T / d rows
    spattn_plan v;
    v.T = T / p->dilation;
    v.causal = p->causal;
    v.window = p->window;
    v.radius = p->radius;
    v.dilation = 1;
    build_schedule(&v, &p->sched[2], 2 * kTile, kTile, 2, true);
    build_bwd_schedule(&v, &p->bsched_res, kTile, kTile);
    p->dview = static_cast<int32_t>(p->dilation);
    const int64_t nkb_res = (v.T + kTile - 1) / kTile;
    cudaError_t e = dev_alloc(&p->d_colmask_res, size_t(nkb_res) * 4);
    if (e == cudaSuccess) e = dev_alloc(&p->d_rowzero, v.T);
    if (e == cudaSuccess) e = cudaMemset(p->d_colmask_res, 0, size_t(nkb_res) * 16);
    if (e == cudaSuccess) e = cudaMemset(p->d_rowzero, 0, size_t(v.T));
    if (e != cudaSuccess) return bail(fail(SPATTN_ERR_CUDA, "plan: %s", cudaGetErrorString(e)));
  }
  build_bwd_schedule(p, &p->bsched, spattn::kBwdRows, spattn::kBwdKeys);
  build_bwd_schedule(p, &p->bsched_tc, spattn::kTile, spattn::kTile);
  {  // random blocks transposed: key block -> the query blocks that list it
    if (!p->r_kb.empty()) {
      const int64_t nb = static_cast<int64_t>(p->r_off.size()) - 1;
      p->rt_off.assign(static_cast<size_t>(nb) + 1, 0);
      for (int32_t k : p->r_kb) ++p->rt_off[k + 1];
      for (int64_t q = 0; q < nb; ++q) p->rt_off[q + 1] += p->rt_off[q];
      p->rt_qb.assign(p->r_kb.size(), 0);
      std::vector<int32_t> fill(p->rt_off.begin(), p->rt_off.end() - 1);
      for (int64_t q = 0; q < nb; ++q)
        for (int32_t x = p->r_off[q]; x < p->r_off[q + 1]; ++x) p->rt_qb[fill[p->r_kb[x]]++] = static_cast<int32_t>(q);
    }
    cudaError_t e = dev_alloc(&p->d_rtoff, p->rt_off.size());
    if (e == cudaSuccess) e = dev_alloc(&p->d_rtqb, p->rt_qb.size());
    if (e == cudaSuccess && !p->rt_qb.empty())
      e = cudaMemcpy(p->d_rtoff, p->rt_off.data(), p->rt_off.size() * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !p->rt_qb.empty())
      e = cudaMemcpy(p->d_rtqb, p->rt_qb.data(), p->rt_qb.size() * 4, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return bail(fail(SPATTN_ERR_CUDA, "plan: %s", cudaGetErrorString(e)));
  }
  for (auto& s : p->sched) {
    spattn_status us = upload_schedule(&s);
    if (us != SPATTN_OK) return bail(us);
  }
  {
    spattn_status us = upload_schedule(&p->bsched);
    if (us == SPATTN_OK) us = upload_schedule(&p->bsched_tc);
    if (us == SPATTN_OK) us = upload_schedule(&p->bsched_res);
    if (us != SPATTN_OK) return bail(us);
    std::vector<int32_t> colidx(size_t(T), -1);
    for (int32_t c = 0; c < p->n_cols; ++c) colidx[p->cols[c]] = c;
    cudaError_t e = dev_alloc(&p->d_colidx, size_t(T));
    if (e == cudaSuccess)
      e = cudaMemcpy(p->d_colidx, colidx.data(), size_t(T) * 4, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return bail(fail(SPATTN_ERR_CUDA, "plan: %s", cudaGetErrorString(e)));
  }
  *out = p;
  return SPATTN_OK;
}

spattn_status spattn_plan_info(const spattn_plan* p, int64_t* pairs, int64_t* n_full,
                               int64_t* n_partial, int64_t* n_empty, int32_t* bm, int32_t* bn) {
  if (!p) return fail(SPATTN_ERR_NULL, "plan is NULL");
  if (pairs) *pairs = p->pairs;
  if (n_full) *n_full = p->n_full;
  if (n_partial) *n_partial = p->n_partial;
  if (n_empty) *n_empty = p->n_empty;
  if (bm) *bm = kTile;
  if (bn) *bn = kTile;
  return SPATTN_OK;
}

spattn_status spattn_plan_copy_tiles(const spattn_plan* p, int32_t* qb, int32_t* kb, int32_t* cnt,
                                     uint8_t* cls, int64_t cap, int64_t* n) {
  if (!p) return fail(SPATTN_ERR_NULL, "plan is NULL");
  if (n) *n = p->n_nonempty;
  const int64_t k = std::min(cap, p->n_nonempty);
  if (k > 0) {
    if (qb) CUDA_TRY(cudaMemcpy(qb, p->d_tile_qb, size_t(k) * 4, cudaMemcpyDeviceToHost));
    if (kb) CUDA_TRY(cudaMemcpy(kb, p->d_tile_kb, size_t(k) * 4, cudaMemcpyDeviceToHost));
    if (cnt) CUDA_TRY(cudaMemcpy(cnt, p->d_tile_cnt, size_t(k) * 4, cudaMemcpyDeviceToHost));
    if (cls) CUDA_TRY(cudaMemcpy(cls, p->d_tile_cls, size_t(k), cudaMemcpyDeviceToHost));
  }
  if (cap < p->n_nonempty) return fail(SPATTN_ERR_SHAPE, "capacity %lld < %lld tiles", (long long)cap,
                                       (long long)p->n_nonempty);
  return SPATTN_OK;
}

spattn_status spattn_plan_copy_columns(const spattn_plan* p, int32_t* cols, int64_t cap, int64_t* n) {
  if (!p) return fail(SPATTN_ERR_NULL, "plan is NULL");
  if (n) *n = p->n_cols;
  const int64_t k = std::min<int64_t>(cap, p->n_cols);
  if (cols && k > 0) std::memcpy(cols, p->cols.data(), size_t(k) * 4);
  if (cap < p->n_cols) return fail(SPATTN_ERR_SHAPE, "capacity %lld < %d columns", (long long)cap, p->n_cols);
  return SPATTN_OK;
}

spattn_status spattn_plan_copy_schedule(const spattn_plan* p, int32_t which, int32_t* items,
                                        int64_t item_cap, int64_t* n_items, int32_t* entries,
                                        int64_t entry_cap, int64_t* n_entries,
                                        int64_t* tile_products) {
  if (!p) return fail(SPATTN_ERR_NULL, "plan is NULL");
  if (which < 0 || which > 4) return fail(SPATTN_ERR_SHAPE, "which must be 0 .. 4");
  const spattn::Schedule& s = which == 4 ? p->bsched_tc : which == 3 ? p->bsched : p->sched[which];
  const int64_t ni = s.items.size() / 4, ne = s.entries.size() / 4;
  if (n_items) *n_items = ni;
  if (n_entries) *n_entries = ne;
  if (tile_products) *tile_products = s.tile_products * (which == 2 ? p->dview : 1);
  if ((items && item_cap < ni) || (entries && entry_cap < ne))
    return fail(SPATTN_ERR_SHAPE, "schedule arrays too small");
  if (items && ni) std::memcpy(items, s.items.data(), size_t(ni) * 16);
  if (entries && ne) std::memcpy(entries, s.entries.data(), size_t(ne) * 16);
  return SPATTN_OK;
}

spattn_status spattn_plan_set_walk_counter(spattn_plan* p, int32_t enable) {
  if (!p) return fail(SPATTN_ERR_NULL, "plan is NULL");
  p->walk_enabled = enable ? 1 : 0;
  CUDA_TRY(cudaMemset(p->d_walk, 0, sizeof(unsigned long long)));
  return SPATTN_OK;
}

spattn_status spattn_plan_walk_count(const spattn_plan* p, int64_t* count) {
  if (!p || !count) return fail(SPATTN_ERR_NULL, "plan or count is NULL");
  CUDA_TRY(cudaDeviceSynchronize());
  unsigned long long v = 0;
  CUDA_TRY(cudaMemcpy(&v, p->d_walk, sizeof v, cudaMemcpyDeviceToHost));
  *count = static_cast<int64_t>(v);
  return SPATTN_OK;
}

spattn_status spattn_fwd(const spattn_plan* cp, int32_t B, int32_t H, spattn_dtype dtype,
                         const void* Q, const void* K, const void* V, float scale, void* O,
                         float* LSE, void* cuda_stream) {
  if (!cp) return fail(SPATTN_ERR_NULL, "plan is NULL");
  spattn_plan* p = const_cast<spattn_plan*>(cp);  // owns mutable scratch
  spattn_status st;
  if ((st = check_ptr(Q, "Q")) || (st = check_ptr(K, "K")) || (st = check_ptr(V, "V")) ||
      (st = check_ptr(O, "O")))
    return st;
  if (LSE && reinterpret_cast<uintptr_t>(LSE) % 4) return fail(SPATTN_ERR_ALIGN, "LSE misaligned");
  if (B < 1 || H < 1) return fail(SPATTN_ERR_SHAPE, "B and H must be >= 1");
  const int64_t BH = int64_t(B) * H;
  if (BH > 65535) return fail(SPATTN_ERR_SHAPE, "B*H = %lld exceeds 65535", (long long)BH);
  if (dtype != SPATTN_BF16 && dtype != SPATTN_FP32) return fail(SPATTN_ERR_DTYPE, "unknown dtype");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(SPATTN_ERR_INVALID_SPEC, "scale must be positive and finite");
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  const int esize = dtype == SPATTN_BF16 ? 2 : 4;
  const int64_t ng = static_cast<int64_t>(p->gpos.size());
  const size_t row_bytes = size_t(p->d) * esize;
  const size_t kc_bytes = size_t(BH) * p->n_cols * row_bytes;
  const size_t qg_bytes = size_t(BH) * ng * row_bytes;
  const size_t need = 2 * kc_bytes + qg_bytes;
  if (need > p->scratch_bytes) {
    if (p->d_scratch) {
      CUDA_TRY(cudaStreamSynchronize(stream));
      CUDA_TRY(cudaFree(p->d_scratch));
      p->d_scratch = nullptr;
      p->scratch_bytes = 0;
    }
    CUDA_TRY(cudaMalloc(&p->d_scratch, need));
    p->scratch_bytes = need;
  }
  uint8_t* base = static_cast<uint8_t*>(p->d_scratch);
  void* Kc = need ? base : nullptr;
  void* Vc = need ? base + kc_bytes : nullptr;
  void* Qg = need ? base + 2 * kc_bytes : nullptr;
  if (need)
    CUDA_TRY(spattn::launch_pack(Q, K, V, Kc, Vc, Qg, p->d_cols, p->n_cols, p->d_gpos,
                                 static_cast<int32_t>(ng), BH, p->T, static_cast<int32_t>(row_bytes),
                                 stream));
  spattn::TcArgs a;
  spattn::fill_fwd_args(p, dtype == SPATTN_BF16, BH, Q, K, V, Kc, Vc, Qg, O, LSE, scale, &a);
  if (dtype == SPATTN_BF16) {
    const char* why = "";
    cudaError_t e = spattn::launch_fwd_tc(p->d, a, stream, &why);
    if (e != cudaSuccess)
      return fail(SPATTN_ERR_CUDA, "tensor-core forward launch: %s (%s)", cudaGetErrorString(e), why);
  } else {
    cudaError_t e = spattn::launch_fwd_simt(p->d, a, stream);
    if (e != cudaSuccess) return fail(SPATTN_ERR_CUDA, "fp32 forward launch: %s", cudaGetErrorString(e));
  }
  return SPATTN_OK;
}

spattn_status spattn_bwd(const spattn_plan* cp, int32_t B, int32_t H, spattn_dtype dtype,
                         const void* Q, const void* K, const void* V, const void* O,
                         const float* LSE, const void* dO, float scale, void* dQ, void* dK,
                         void* dV, void* cuda_stream) {
  if (!cp) return fail(SPATTN_ERR_NULL, "plan is NULL");
  spattn_plan* p = const_cast<spattn_plan*>(cp);  // owns mutable scratch
  spattn_status st;
  if ((st = check_ptr(Q, "Q")) || (st = check_ptr(K, "K")) || (st = check_ptr(V, "V")) ||
      (st = check_ptr(O, "O")) || (st = check_ptr(LSE, "LSE")) || (st = check_ptr(dO, "dO")) ||
      (st = check_ptr(dQ, "dQ")) || (st = check_ptr(dK, "dK")) || (st = check_ptr(dV, "dV")))
    return st;
  if (B < 1 || H < 1) return fail(SPATTN_ERR_SHAPE, "B and H must be >= 1");
  const int64_t BH = int64_t(B) * H;
  if (BH > 65535) return fail(SPATTN_ERR_SHAPE, "B*H = %lld exceeds 65535", (long long)BH);
  if (dtype != SPATTN_BF16 && dtype != SPATTN_FP32) return fail(SPATTN_ERR_DTYPE, "unknown dtype");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(SPATTN_ERR_INVALID_SPEC, "scale must be positive and finite");
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  const bool tc = dtype == SPATTN_BF16;
  const size_t dvec_bytes = (size_t(BH) * p->T * 4 + 255) / 256 * 256;
  const size_t kc_bytes = size_t(BH) * p->n_cols * p->d * 4;
  // bf16: packed K/V of the sparse columns and gathered Q/dO of the global rows for
  // the tensor-core dQ kernel
  const int64_t ng = static_cast<int64_t>(p->gpos.size());
  const size_t row_b = size_t(p->d) * 2;
  const size_t pk_bytes = tc ? (size_t(BH) * p->n_cols * row_b + 255) / 256 * 256 : 0;
  const size_t pg_bytes = tc ? (size_t(BH) * ng * row_b + 255) / 256 * 256 : 0;
  const size_t need = dvec_bytes + 2 * kc_bytes + 2 * pk_bytes + 2 * pg_bytes;
  if (need > p->bscratch_bytes) {
    if (p->d_bscratch) {
      CUDA_TRY(cudaStreamSynchronize(stream));
      CUDA_TRY(cudaFree(p->d_bscratch));
      p->d_bscratch = nullptr;
      p->bscratch_bytes = 0;
    }
    CUDA_TRY(cudaMalloc(&p->d_bscratch, need));
    p->bscratch_bytes = need;
  }
  uint8_t* base = static_cast<uint8_t*>(p->d_bscratch);
  spattn::BwdArgs a;
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.O = O;
  a.LSE = LSE;
  a.dO = dO;
  a.dQ = dQ;
  a.dK = dK;
  a.dV = dV;
  a.Dvec = reinterpret_cast<float*>(base);
  a.dKc = reinterpret_cast<float*>(base + dvec_bytes);
  a.dVc = reinterpret_cast<float*>(base + dvec_bytes + kc_bytes);
  a.BH = static_cast<int32_t>(BH);
  a.n_cols = p->n_cols;
  a.scale = scale;
  a.bf16 = dtype == SPATTN_BF16;
  a.cols = p->d_cols;
  a.colidx = p->d_colidx;
  a.colmask = p->d_colmask;
  a.mask = p->mask_dev();
  a.q_items = p->sched[1].d_items;
  a.q_entries = p->sched[1].d_entries;
  a.n_q_items = static_cast<int32_t>(p->sched[1].items.size() / 4);
  a.units = p->bsched.d_items;
  a.u_entries = p->bsched.d_entries;
  a.n_packed_units = p->bsched.n_packed_units;
  a.n_units = static_cast<int32_t>(p->bsched.items.size() / 4);
  cudaError_t e = spattn::launch_bwd_simt(p->d, a, stream, !tc, !tc);
  if (e != cudaSuccess) return fail(SPATTN_ERR_CUDA, "backward launch: %s", cudaGetErrorString(e));
  if (tc) {
    uint8_t* pk = base + dvec_bytes + 2 * kc_bytes;
    void* Kc = pk;
    void* Vc = pk + pk_bytes;
    void* Qg = pk + 2 * pk_bytes;
    void* dOg = pk + 2 * pk_bytes + pg_bytes;
    if (p->n_cols > 0 || ng > 0) {
      CUDA_TRY(spattn::launch_pack(Q, K, V, Kc, Vc, Qg, p->d_cols, p->n_cols, p->d_gpos,
                                   static_cast<int32_t>(ng), BH, p->T, static_cast<int32_t>(row_b),
                                   stream));
      if (ng > 0)  // the same gather of the global rows, of dO
        CUDA_TRY(spattn::launch_pack(dO, K, V, nullptr, nullptr, dOg, p->d_cols, 0, p->d_gpos,
                                     static_cast<int32_t>(ng), BH, p->T,
                                     static_cast<int32_t>(row_b), stream));
    }
    spattn::BwdTcArgs t;
    t.Q = Q;
    t.K = K;
    t.V = V;
    t.dO = dO;
    t.Kc = p->n_cols ? Kc : K;
    t.Vc = p->n_cols ? Vc : V;
    t.Qg = ng ? Qg : Q;
    t.dOg = ng ? dOg : dO;
    t.dQ = dQ;
    t.LSE = LSE;
    t.Dvec = a.Dvec;
    t.BH = static_cast<int32_t>(BH);
    t.n_cols = p->n_cols;
    t.scale = scale;
    t.colmask = p->d_colmask;
    t.mask = p->mask_dev();
    t.items = p->sched[0].d_items;
    t.entries = p->sched[0].d_entries;
    t.n_items = static_cast<int32_t>(p->sched[0].items.size() / 4);
    t.err = p->d_err;
    t.wait_budget_cycles = p->wait_budget_cycles;
    t.dK = dK;
    t.dV = dV;
    t.dKc = a.dKc;
    t.dVc = a.dVc;
    t.cols = p->d_cols;
    t.colidx = p->d_colidx;
    t.rt_off = p->d_rtoff;
    t.rt_qb = p->d_rtqb;
    t.units = p->bsched_tc.d_items;
    t.u_entries = p->bsched_tc.d_entries;
    t.n_packed_units = p->bsched_tc.n_packed_units;
    t.n_units = static_cast<int32_t>(p->bsched_tc.items.size() / 4);
    if (p->dview > 1) {  // a dilated window on its residue classes, as the forward walks it
      t.mask = p->mask_dev_res();
      t.colmask = p->d_colmask_res;
      t.n_cols = 0;
      t.items = p->sched[2].d_items;
      t.entries = p->sched[2].d_entries;
      t.n_items = static_cast<int32_t>(p->sched[2].items.size() / 4);
      t.units = p->bsched_res.d_items;
      t.u_entries = p->bsched_res.d_entries;
      t.n_packed_units = 0;
      t.n_units = static_cast<int32_t>(p->bsched_res.items.size() / 4);
      t.dview = p->dview;
    }
    const char* why = "";
    e = spattn::launch_bwd_dq_tc(p->d, t, stream, &why);
    if (e != cudaSuccess)
      return fail(SPATTN_ERR_CUDA, "tensor-core dQ launch: %s (%s)", cudaGetErrorString(e), why);
    e = spattn::launch_bwd_dkdv_tc(p->d, t, stream, &why);
    if (e != cudaSuccess)
      return fail(SPATTN_ERR_CUDA, "tensor-core dK/dV launch: %s (%s)", cudaGetErrorString(e), why);
  }
  return SPATTN_OK;
}

// ---- decode ------------------------------------------------------------------------

namespace {
spattn_status decode_shape(int32_t B, int32_t Hq, int32_t Hkv, int64_t cap, int64_t window,
                           int32_t d, spattn_dtype dtype) {
  if (B < 1 || Hq < 1 || Hkv < 1) return fail(SPATTN_ERR_SHAPE, "B, Hq and Hkv must be >= 1");
  if (Hq % Hkv != 0 || (Hq / Hkv != 1 && Hq / Hkv != 2 && Hq / Hkv != 4 && Hq / Hkv != 8))
    return fail(SPATTN_ERR_SHAPE, "Hq / Hkv must be 1, 2, 4 or 8");
  if (int64_t(B) * Hkv > (int64_t(1) << 24)) return fail(SPATTN_ERR_SHAPE, "B * Hkv too large");
  if (cap < 1 || cap > (int64_t(1) << 30)) return fail(SPATTN_ERR_SHAPE, "cap must be in [1, 2^30]");
  if (window < 0 || window > cap)
    return fail(SPATTN_ERR_INVALID_SPEC, "window must be in [0, cap] (0 = cap)");
  if (d != 64 && d != 128) return fail(SPATTN_ERR_SHAPE, "head_dim must be 64 or 128");
  if (dtype != SPATTN_BF16 && dtype != SPATTN_FP32) return fail(SPATTN_ERR_DTYPE, "unknown dtype");
  return SPATTN_OK;
}
constexpr size_t kDecodeHeader = 256;  // error word, padded
}  // namespace

spattn_status spattn_decode_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int64_t cap,
                                            int32_t head_dim, size_t* bytes) {
  if (!bytes) return fail(SPATTN_ERR_NULL, "bytes is NULL");
  spattn_status st = decode_shape(B, Hq, Hkv, cap, 0, head_dim, SPATTN_BF16);
  if (st != SPATTN_OK) return st;
  const int ns = spattn::decode_splits(B, Hkv, cap);
  *bytes = kDecodeHeader + size_t(B) * Hq * ns * (head_dim + 2) * 4;
  return SPATTN_OK;
}

spattn_status spattn_kv_append(int32_t B, int32_t Hkv, int64_t cap, int32_t head_dim,
                               spattn_dtype dtype, void* Kc, void* Vc, const void* k_new,
                               const void* v_new, const int64_t* pos, void* cuda_stream) {
  spattn_status st = decode_shape(B, Hkv, Hkv, cap, 0, head_dim, dtype);
  if (st != SPATTN_OK) return st;
  if ((st = check_ptr(Kc, "K_cache")) || (st = check_ptr(Vc, "V_cache")) ||
      (st = check_ptr(k_new, "k_new")) || (st = check_ptr(v_new, "v_new")))
    return st;
  if (!pos) return fail(SPATTN_ERR_NULL, "pos is NULL");
  if (reinterpret_cast<uintptr_t>(pos) % 8) return fail(SPATTN_ERR_ALIGN, "pos misaligned");
  CUDA_TRY(spattn::launch_kv_append(dtype == SPATTN_BF16, Kc, Vc, k_new, v_new, pos, B, Hkv, cap,
                                    head_dim, static_cast<cudaStream_t>(cuda_stream)));
  return SPATTN_OK;
}

spattn_status spattn_decode(int32_t B, int32_t Hq, int32_t Hkv, int64_t cap, int64_t window,
                            int32_t head_dim, spattn_dtype dtype, const void* q, const void* Kc,
                            const void* Vc, const int64_t* pos, float scale, void* out,
                            float* lse, void* workspace, size_t workspace_bytes,
                            void* cuda_stream) {
  spattn_status st = decode_shape(B, Hq, Hkv, cap, window, head_dim, dtype);
  if (st != SPATTN_OK) return st;
  if ((st = check_ptr(q, "q")) || (st = check_ptr(Kc, "K_cache")) ||
      (st = check_ptr(Vc, "V_cache")) || (st = check_ptr(out, "out")) ||
      (st = check_ptr(workspace, "workspace")))
    return st;
  if (!pos) return fail(SPATTN_ERR_NULL, "pos is NULL");
  if (reinterpret_cast<uintptr_t>(pos) % 8) return fail(SPATTN_ERR_ALIGN, "pos misaligned");
  if (lse && reinterpret_cast<uintptr_t>(lse) % 4) return fail(SPATTN_ERR_ALIGN, "lse misaligned");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(SPATTN_ERR_INVALID_SPEC, "scale must be positive and finite");
  size_t need = 0;
  spattn_decode_workspace_bytes(B, Hq, Hkv, cap, head_dim, &need);
  if (workspace_bytes < need)
    return fail(SPATTN_ERR_SHAPE, "workspace of %zu bytes < %zu needed", workspace_bytes, need);
  spattn::DecodeArgs a;
  a.q = q;
  a.Kc = Kc;
  a.Vc = Vc;
  a.pos = pos;
  a.out = out;
  a.lse = lse;
  a.err = static_cast<int*>(workspace);
  a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kDecodeHeader);
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = head_dim;
  a.nsplit = spattn::decode_splits(B, Hkv, cap);
  a.bf16 = dtype == SPATTN_BF16;
  a.cap = cap;
  a.window = window ? window : cap;
  a.scale = scale;
  cudaError_t e = spattn::launch_decode(a, static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return fail(SPATTN_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return SPATTN_OK;
}

spattn_status spattn_decode_append(int32_t B, int32_t Hq, int32_t Hkv, int64_t cap,
                                   int64_t window, int32_t head_dim, spattn_dtype dtype,
                                   const void* q, void* Kc, void* Vc, const void* k_new,
                                   const void* v_new, const int64_t* pos, float scale, void* out,
                                   float* lse, void* workspace, size_t workspace_bytes,
                                   void* cuda_stream) {
  spattn_status st = decode_shape(B, Hq, Hkv, cap, window, head_dim, dtype);
  if (st != SPATTN_OK) return st;
  if ((st = check_ptr(q, "q")) || (st = check_ptr(Kc, "K_cache")) ||
      (st = check_ptr(Vc, "V_cache")) || (st = check_ptr(out, "out")) ||
      (st = check_ptr(workspace, "workspace")) || (st = check_ptr(k_new, "k_new")) ||
      (st = check_ptr(v_new, "v_new")))
    return st;
  if (!pos) return fail(SPATTN_ERR_NULL, "pos is NULL");
  if (reinterpret_cast<uintptr_t>(pos) % 8) return fail(SPATTN_ERR_ALIGN, "pos misaligned");
  if (lse && reinterpret_cast<uintptr_t>(lse) % 4) return fail(SPATTN_ERR_ALIGN, "lse misaligned");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(SPATTN_ERR_INVALID_SPEC, "scale must be positive and finite");
  size_t need = 0;
  spattn_decode_workspace_bytes(B, Hq, Hkv, cap, head_dim, &need);
  if (workspace_bytes < need)
    return fail(SPATTN_ERR_SHAPE, "workspace of %zu bytes < %zu needed", workspace_bytes, need);
  spattn::DecodeArgs a;
  a.q = q;
  a.Kc = Kc;
  a.Vc = Vc;
  a.pos = pos;
  a.out = out;
  a.lse = lse;
  a.err = static_cast<int*>(workspace);
  a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kDecodeHeader);
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = head_dim;
  a.nsplit = spattn::decode_splits(B, Hkv, cap);
  a.bf16 = dtype == SPATTN_BF16;
  a.cap = cap;
  a.window = window ? window : cap;
  a.scale = scale;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e = cudaSuccess;
  if (a.bf16) {  // the decode kernel appends the rows itself
    a.kn = k_new;
    a.vn = v_new;
  } else {  // fp32: the append kernel first, as spattn_kv_append
    e = spattn::launch_kv_append(false, Kc, Vc, k_new, v_new, pos, B, Hkv, cap, head_dim, stream);
    if (e != cudaSuccess) return fail(SPATTN_ERR_CUDA, "append launch: %s", cudaGetErrorString(e));
  }
  e = spattn::launch_decode(a, stream);
  if (e != cudaSuccess) return fail(SPATTN_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return SPATTN_OK;
}

spattn_status spattn_decode_check(void* workspace, void* cuda_stream) {
  if (!workspace) return fail(SPATTN_ERR_NULL, "workspace is NULL");
  CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)));
  int e = 0;
  CUDA_TRY(cudaMemcpy(&e, workspace, sizeof e, cudaMemcpyDeviceToHost));
  CUDA_TRY(cudaMemset(workspace, 0, sizeof(int)));
  if (e & spattn::kErrTimeout)
    return fail(SPATTN_ERR_TIMEOUT, "a device-side wait of the decode kernel ran out of time");
  return SPATTN_OK;
}

spattn_status spattn_fwd_host(const spattn_plan* p, int32_t B, int32_t H, spattn_dtype dtype,
                              const void* Qh, const void* Kh, const void* Vh, float scale, void* Oh,
                              float* LSEh, void* Qd, void* Kd, void* Vd, void* Od, float* LSEd,
                              void* cuda_stream) {
  if (!p) return fail(SPATTN_ERR_NULL, "plan is NULL");
  if (!Qh || !Kh || !Vh || !Oh) return fail(SPATTN_ERR_NULL, "a host buffer is NULL");
  if ((LSEh == nullptr) != (LSEd == nullptr))
    return fail(SPATTN_ERR_NULL, "LSE_host and LSE_dev must both be set or both be NULL");
  if (B < 1 || H < 1) return fail(SPATTN_ERR_SHAPE, "B and H must be >= 1");
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  const size_t esize = dtype == SPATTN_BF16 ? 2 : 4;
  spattn_status st;
  if ((st = check_ptr(Qd, "Q_dev")) || (st = check_ptr(Kd, "K_dev")) || (st = check_ptr(Vd, "V_dev")) ||
      (st = check_ptr(Od, "O_dev")))
    return st;
  spattn_plan* mp = const_cast<spattn_plan*>(p);  // owns the pipeline's streams and events
  if (!mp->host_in) {
    CUDA_TRY(cudaStreamCreateWithFlags(&mp->host_in, cudaStreamNonBlocking));
    CUDA_TRY(cudaStreamCreateWithFlags(&mp->host_out, cudaStreamNonBlocking));
    for (cudaEvent_t& e : mp->host_ev) CUDA_TRY(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
  }
  // Chunks of consecutive (batch, head) units ([B][H][T][d] keeps each chunk contiguous):
  // the copy-in stream brings chunk k+1 while `stream` computes chunk k and the
  // copy-out stream returns chunk k-1; every unit is computed independently, so the
  // results equal one spattn_fwd over all units.
  const int64_t BH = int64_t(B) * H;
  const int64_t n_chunks = std::min<int64_t>(BH, spattn_plan::kHostChunks);
  const int64_t per = (BH + n_chunks - 1) / n_chunks;
  const size_t unit = size_t(p->T) * p->d * esize;
  cudaEvent_t* ev = mp->host_ev;
  cudaEvent_t ev_start = ev[2 * spattn_plan::kHostChunks], ev_done = ev[2 * spattn_plan::kHostChunks + 1];
  // earlier work on `stream` may still use the device buffers
  CUDA_TRY(cudaEventRecord(ev_start, stream));
  CUDA_TRY(cudaStreamWaitEvent(mp->host_in, ev_start, 0));
  for (int64_t c = 0; c * per < BH; ++c) {
    const int64_t u0 = c * per, cnt = std::min(per, BH - u0);
    const size_t off = size_t(u0) * unit, len = size_t(cnt) * unit;
    auto at = [off](const void* b) { return static_cast<const char*>(b) + off; };
    auto atw = [off](void* b) { return static_cast<char*>(b) + off; };
    CUDA_TRY(cudaMemcpyAsync(atw(Qd), at(Qh), len, cudaMemcpyHostToDevice, mp->host_in));
    CUDA_TRY(cudaMemcpyAsync(atw(Kd), at(Kh), len, cudaMemcpyHostToDevice, mp->host_in));
    CUDA_TRY(cudaMemcpyAsync(atw(Vd), at(Vh), len, cudaMemcpyHostToDevice, mp->host_in));
    CUDA_TRY(cudaEventRecord(ev[2 * c], mp->host_in));
    CUDA_TRY(cudaStreamWaitEvent(stream, ev[2 * c], 0));
    float* lse_d = LSEd ? LSEd + size_t(u0) * p->T : nullptr;
    st = spattn_fwd(p, 1, static_cast<int32_t>(cnt), dtype, atw(Qd), atw(Kd), atw(Vd), scale,
                    atw(Od), lse_d, cuda_stream);
    if (st != SPATTN_OK) {
      cudaStreamSynchronize(mp->host_in);
      return st;
    }
    CUDA_TRY(cudaEventRecord(ev[2 * c + 1], stream));
    CUDA_TRY(cudaStreamWaitEvent(mp->host_out, ev[2 * c + 1], 0));
    CUDA_TRY(cudaMemcpyAsync(atw(Oh), at(Od), len, cudaMemcpyDeviceToHost, mp->host_out));
    if (LSEh)
      CUDA_TRY(cudaMemcpyAsync(LSEh + size_t(u0) * p->T, lse_d, size_t(cnt) * p->T * 4,
                               cudaMemcpyDeviceToHost, mp->host_out));
  }
  CUDA_TRY(cudaEventRecord(ev_done, mp->host_out));
  CUDA_TRY(cudaStreamWaitEvent(stream, ev_done, 0));
  CUDA_TRY(cudaStreamSynchronize(stream));
  return SPATTN_OK;
}

spattn_status spattn_plan_set_wait_budget(spattn_plan* p, uint64_t cycles) {
  if (!p) return fail(SPATTN_ERR_NULL, "plan is NULL");
  if (cycles == 0) return fail(SPATTN_ERR_SHAPE, "the wait budget must be positive");
  p->wait_budget_cycles = cycles;
  return SPATTN_OK;
}

spattn_status spattn_plan_test_wait_timeout(spattn_plan* p, int32_t enable) {
  if (!p) return fail(SPATTN_ERR_NULL, "plan is NULL");
  p->inject_timeout = enable ? 1 : 0;
  return SPATTN_OK;
}

spattn_status spattn_plan_check_device(const spattn_plan* p, void* cuda_stream) {
  if (!p) return fail(SPATTN_ERR_NULL, "plan is NULL");
  CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)));
  int e = 0;
  CUDA_TRY(cudaMemcpy(&e, p->d_err, sizeof e, cudaMemcpyDeviceToHost));
  CUDA_TRY(cudaMemset(p->d_err, 0, sizeof(int)));
  if (e & spattn::kErrTimeout)
    return fail(SPATTN_ERR_TIMEOUT, "a device-side wait ran out of its time budget");
  return SPATTN_OK;
}

void spattn_plan_destroy(spattn_plan* p) {
  if (!p) return;
  cudaDeviceSynchronize();
  free_plan_memory(p);
  delete p;
}

}  // extern "C"
