// predicate.cuh -- the per-element mask predicate the forward kernels apply inside
// tiles that are not entirely allowed.
//
// For query row i and a key tile whose column c maps to key j, every schedule
// entry kind reduces to one test:
//     allowed(c) = (lo <= c <= hi)  or  (bit c of the tile's column mask and c <= hb)
// * band tile of the natural grid (keys k0..k0+127): [lo, hi] is the local window
//   of row i (causal: i-w+1 .. i, "Sparse attention" glossary, section "Choose the
//   available reads"; bidirectional: i-r .. i+r, "Attention variants" section 3),
//   the column mask marks strided and global columns, readable up to hb (= i in a
//   causal mask, octlm "Sparse attention", "One mask function for every pattern").
// * packed sparse columns [src, lim): every packed column is a strided or global
//   column that lies before the group's band (causal) or anywhere (bidirectional),
//   so only c < lim - src is tested.
// * dense walk of a global row: every key j <= i (causal) or every key
//   ("Attention variants", section 4, with_global).
// * random blocks (BigBird's random connections, "Sparse and sliding-window
//   attention", section "Block-sparse attention: BigBird"): inside a band tile the
//   columns of row i's random key blocks join the column mask (they are cut at hb
//   like the strided ones); a key tile outside the band reached only by random blocks
//   (kind "random") has no local span, and its mask is the random columns minus the
//   strided and global ones, which the packed entries already cover.
// Keys at or past T (ragged last tile) fall outside [lo, hi] and past hb.
#pragma once

#include <cstdint>

#include "internal.h"

namespace spattn {

// Bits c of the 128-key tile at k0 that lie in a random key block of row i.
__device__ __forceinline__ void random_bits(const MaskDev& m, int i, int k0, uint32_t (&w)[4]) {
  w[0] = w[1] = w[2] = w[3] = 0u;
  if (m.rand_block == 0 || i >= m.T) return;
  const int q = i / m.rand_block;
  for (int x = m.r_off[q]; x < m.r_off[q + 1]; ++x) {
    const int c0 = m.r_kb[x] * m.rand_block - k0;
    if (c0 < 0 || c0 >= kTile) continue;  // block sizes divide the tile: wholly in or out
    const int c1 = c0 + m.rand_block - 1;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int a = max(c0 - 32 * k, 0), b = min(c1 - 32 * k, 31);
      if (a <= b) w[k] |= ((2u << b) - 1u) & (0xffffffffu << a);
    }
  }
}

struct RowPredicate {
  int lo, hi, hb;
  int dil, res;  // band columns also need c % dil == res (a dilated local window)
  uint32_t bits[4];
};

// The column-mask words of an entry's key tile (band and random entries; zero for the
// other kinds, which do not read them).  Loaded apart from make_predicate so that a
// kernel can fetch them one entry ahead.
__device__ __forceinline__ uint4 colmask_words(const uint32_t* colmask, int4 e) {
  const int kind = (e.y >> kKindShift) & 3;
  if (kind == kKindBand || kind == kKindRandom)
    return *reinterpret_cast<const uint4*>(colmask + 4 * e.z);
  return make_uint4(0u, 0u, 0u, 0u);
}

// The predicate of row i in the entry's tile, with the tile's column-mask words `w`.
__device__ __forceinline__ RowPredicate make_predicate(const MaskDev& m, uint4 w, int4 e, int i) {
  RowPredicate p;
  const int kind = (e.y >> kKindShift) & 3;
  const int k0 = e.x;
  p.bits[0] = p.bits[1] = p.bits[2] = p.bits[3] = 0u;
  p.hb = -1;
  p.dil = 1;
  p.res = 0;
  if (kind == kKindBand) {
    int lo, hi, hb;
    const int d = m.dilation;
    if (m.causal) {
      lo = m.window ? i - (m.window - 1) * d : 0;
      hi = i;
      hb = i;
    } else {
      lo = m.radius >= 0 ? i - m.radius * d : 0;
      hi = m.radius >= 0 ? i + m.radius * d : m.T - 1;
      hb = m.T - 1;
    }
    p.dil = d;
    p.res = ((i - k0) % d + d) % d;  // column c = key k0 + c is on the grid iff c % d == res
    hi = min(hi, m.T - 1);
    hb = min(hb, m.T - 1);
    p.lo = lo - k0;
    p.hi = hi - k0;
    p.hb = hb - k0;
    p.bits[0] = w.x;
    p.bits[1] = w.y;
    p.bits[2] = w.z;
    p.bits[3] = w.w;
    if (m.rand_block) {
      uint32_t r[4];
      random_bits(m, i, k0, r);
#pragma unroll
      for (int k = 0; k < 4; ++k) p.bits[k] |= r[k];
    }
  } else if (kind == kKindRandom) {
    p.lo = 1;  // no local span
    p.hi = 0;
    p.hb = (m.causal ? min(i, m.T - 1) : m.T - 1) - k0;
    uint32_t r[4];
    random_bits(m, i, k0, r);
    p.bits[0] = r[0] & ~w.x;
    p.bits[1] = r[1] & ~w.y;
    p.bits[2] = r[2] & ~w.z;
    p.bits[3] = r[3] & ~w.w;
  } else if (kind == kKindPacked) {
    p.lo = 0;
    p.hi = e.w - e.x - 1;
  } else {
    p.lo = 0;
    p.hi = (m.causal ? min(i, m.T - 1) : m.T - 1) - k0;
  }
  return p;
}

__device__ __forceinline__ RowPredicate make_predicate(const MaskDev& m, const uint32_t* colmask,
                                                       int4 e, int i) {
  return make_predicate(m, colmask_words(colmask, e), e, i);
}

// Bits b of a 32-bit word with lo <= base + b <= hi.
__device__ __forceinline__ uint32_t span_bits(int lo, int hi, int base) {
  int a = lo - base, b = hi - base;
  if (b < 0 || a > 31 || b < a) return 0u;
  a = max(a, 0);
  b = min(b, 31);
  return ((2u << b) - 1u) & (0xffffffffu << a);
}

// The allowed columns of a 128-key tile as four 32-bit words (bit c of word c/32).
__device__ __forceinline__ void row_mask(const RowPredicate& p, uint32_t (&w)[4]) {
  if (p.dil == 1) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      w[k] = span_bits(p.lo, p.hi, 32 * k) | (p.bits[k] & span_bits(0, p.hb, 32 * k));
    return;
  }
  // dilated window: every dil-th column of [lo, hi] starting on the row's residue
#pragma unroll
  for (int k = 0; k < 4; ++k) w[k] = p.bits[k] & span_bits(0, p.hb, 32 * k);
  int c = max(p.lo, 0);
  c += ((p.res - c) % p.dil + p.dil) % p.dil;
  const int last = min(p.hi, kTile - 1);
  for (; c <= last; c += p.dil) {  // word selected by value: w stays in registers
    const uint32_t bit = 1u << (c & 31);
    const int k = c >> 5;
    w[0] |= k == 0 ? bit : 0u;
    w[1] |= k == 1 ? bit : 0u;
    w[2] |= k == 2 ? bit : 0u;
    w[3] |= k == 3 ? bit : 0u;
  }
}

// Word k (columns 32k .. 32k+31) of row_mask, selected by value so that nothing is
// indexed at run time; a contiguous window builds only that word.
__device__ __forceinline__ uint32_t row_word(const RowPredicate& p, int k) {
  const uint32_t bits = k == 0 ? p.bits[0] : (k == 1 ? p.bits[1] : (k == 2 ? p.bits[2] : p.bits[3]));
  if (p.dil == 1) return span_bits(p.lo, p.hi, 32 * k) | (bits & span_bits(0, p.hb, 32 * k));
  uint32_t w[4];
  row_mask(p, w);
  return k == 0 ? w[0] : (k == 1 ? w[1] : (k == 2 ? w[2] : w[3]));
}

__device__ __forceinline__ bool pred_allowed(const RowPredicate& p, int c) {
  const bool in_band = c >= p.lo && c <= p.hi && (p.dil == 1 || c % p.dil == p.res);
  const bool in_cols = ((p.bits[c >> 5] >> (c & 31)) & 1u) && c <= p.hb;
  return in_band || in_cols;
}

}  // namespace spattn
