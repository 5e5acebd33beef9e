// Block-sparse mask metadata as the kernels read it: for each mask head (one
// shared head, or K*G query heads) and each block of 128 query positions x 128
// keys, a class (EMPTY, FULL, PARTIAL) and, for PARTIAL blocks, an index into a
// pool of 128 x 128 bitmasks (row-major, 4 words of 32 keys per query row,
// bit i of word w is key 32*w + i).  The mask is never expanded to T x S.
#pragma once
#include <cstdint>
#include "kernels.h"

namespace fa {

enum : int { BM_EMPTY = 0, BM_FULL = 1, BM_PARTIAL = 2 };

// Conjunction of two tile classes: empty if either is, partial if either is.
__device__ __forceinline__ int class_and(int a, int b) {
  if (a == BM_EMPTY || b == BM_EMPTY) return BM_EMPTY;
  return (a == BM_PARTIAL || b == BM_PARTIAL) ? BM_PARTIAL : BM_FULL;
}

// Class of mask block (qb, kb) for a packed Q tile of kv head kh: the G query
// heads share the tile, so their classes are merged (all empty -> EMPTY, all
// full -> FULL, else PARTIAL).
__device__ __forceinline__ int bm_tile_class(const BlockMask& m, int kh, int G, int qb, int kb) {
  if (m.cls == nullptr) return BM_FULL;
  if (m.heads == 1) return m.cls[(long)qb * m.nkb + kb];
  bool any_empty = false, any_full = false, any_partial = false;
  for (int g = 0; g < G; ++g) {
    const int c = m.cls[((long)(kh * G + g) * m.nqb + qb) * m.nkb + kb];
    any_empty |= c == BM_EMPTY;
    any_full |= c == BM_FULL;
    any_partial |= c == BM_PARTIAL;
  }
  if (!any_full && !any_partial) return BM_EMPTY;
  if (!any_empty && !any_partial) return BM_FULL;
  return BM_PARTIAL;
}

// 32 keys [32*word, 32*word + 32) of block (qb, kb) for query position t of
// query head (kh, g): bit i set = key kept.
__device__ __forceinline__ uint32_t bm_row_word(const BlockMask& m, int kh, int G, int g, int t, int kb,
                                                int word) {
  const int h = m.heads == 1 ? 0 : kh * G + g;
  const int qb = t >> 7;
  const long blk = ((long)h * m.nqb + qb) * m.nkb + kb;
  const int c = m.cls[blk];
  if (c == BM_FULL) return 0xffffffffu;
  if (c == BM_EMPTY) return 0u;
  return __ldg(m.bits + ((long)m.idx[blk] * 128 + (t & 127)) * 4 + word);
}

}  // namespace fa
