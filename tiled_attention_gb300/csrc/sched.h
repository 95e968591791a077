// sched.h — mask-aware tile scheduling shared by the host planner and the kernels.
//
// Every mask kind gives each query row i a contiguous visible key interval
// [vis_lo(i), vis_hi(i)], and both ends are nondecreasing in i. So for a tile of rows
// [r0, r1] and keys [k0, k1]:
//   * some pair is visible  <=>  k0 <= vis_hi(r1) and k1 >= vis_lo(r0);
//   * every pair is visible <=>  vis_lo(r1) <= k0 and k1 <= vis_hi(r0).
// Tiles of the first kind that are not of the second are the boundary tiles, the only ones
// that need an element mask ("Optimizing Triton Kernels for Custom Attention Patterns on
// H100", Pattern B: mask only the first and last key tile; Pattern A: skip the boundary check
// inside a document). Key tiles holding no visible pair are never loaded or computed. The
// same page names prefix-LM among the masks with this kind of structure; causal, both window
// forms, both document forms and prefix-LM all give monotone intervals.
#pragma once

#if defined(__CUDACC__)
#define TA_HD __host__ __device__ __forceinline__
#else
#define TA_HD inline
#endif

namespace ta {

enum MaskKind { kMaskNone = 0, kMaskCausal = 1, kMaskSliding = 2, kMaskDocument = 3,
                kMaskPaged = 4, kMaskDecode = 5, kMaskSlidingBidir = 6, kMaskDocumentBidir = 7,
                kMaskPrefixLM = 8, kMaskPagedPrefill = 9 };

// Kinds whose query rows are packed segments described by cu_seqlens. For PAGED_PREFILL a
// segment is one sequence's query chunk; its keys (the sequence's context, held in a paged
// pool) are numbered so that key j sits at index k_org + j with k_org = chunk start -
// (context length - chunk length). The chunk's last row then lines up with the context's
// last key, and the causal rule j <= i of that shared index space is the chunked-prefill
// mask: chunk row t sees the context's keys up to position (context - chunk) + t.
TA_HD constexpr bool is_packed(int mask) {
  return mask == kMaskDocument || mask == kMaskDocumentBidir || mask == kMaskPagedPrefill;
}

enum TileKind { kTileEmpty = 0, kTileFull = 1, kTileBoundary = 2 };

TA_HD int imin(int a, int b) { return a < b ? a : b; }
TA_HD int imax(int a, int b) { return a > b ? a : b; }

// First visible key of query row i; keys are numbered in the same space as rows, and the keys
// a tile schedule may touch start at k_org (0, or the start of the query's document segment).
//   SLIDING        i - W < j        (causal window of W keys, the query included)
//   SLIDING_BIDIR  i - W <= j       (W keys on each side of the query)
TA_HD int vis_lo(int mask, int window, int k_org, int i) {
  if (mask == kMaskSliding) return imax(k_org, i - window + 1);
  if (mask == kMaskSlidingBidir) return imax(k_org, i - window);
  return k_org;
}

// Last visible key of query row i; keys end before k_end. `window` is the two-sided window
// (SLIDING_BIDIR) or the prefix length P (PREFIX_LM: rows below P see the whole prefix).
TA_HD int vis_hi(int mask, int window, int k_end, int i) {
  if (mask == kMaskNone || mask == kMaskDocumentBidir) return k_end - 1;
  if (mask == kMaskSlidingBidir)  // i + W without overflow for any W >= 0
    return i > k_end - 1 - window ? k_end - 1 : i + window;
  if (mask == kMaskPrefixLM) return imin(imax(i, window - 1), k_end - 1);
  return imin(i, k_end - 1);
}

TA_HD bool pair_visible(int mask, int window, int k_org, int k_end, int i, int j) {
  return j >= vis_lo(mask, window, k_org, i) && j <= vis_hi(mask, window, k_end, i);
}

struct KvRange {
  int lo, hi;  // key tiles [lo, hi), numbered from k_org; empty when hi <= lo
};

// Key tiles holding at least one visible pair for the valid query rows
// [r0, min(r0 + bm, row_end)).
TA_HD KvRange kv_tile_range(int mask, int window, int r0, int bm, int row_end, int k_org,
                            int k_end, int bn) {
  KvRange r{0, 0};
  const int r1 = imin(r0 + bm, row_end) - 1;
  if (r1 < r0) return r;
  const int a = vis_lo(mask, window, k_org, r0);
  const int b = vis_hi(mask, window, k_end, r1);
  if (b < a) return r;
  r.lo = (a - k_org) / bn;
  r.hi = (b - k_org) / bn + 1;
  return r;
}

TA_HD int tile_kind(int mask, int window, int r0, int bm, int row_end, int k_org, int k_end,
                    int bn, int t) {
  const int r1 = imin(r0 + bm, row_end) - 1;
  if (r1 < r0) return kTileEmpty;
  const int k0 = k_org + t * bn;
  const int k1 = k0 + bn - 1;
  if (k0 > vis_hi(mask, window, k_end, r1) || k1 < vis_lo(mask, window, k_org, r0))
    return kTileEmpty;
  if (vis_lo(mask, window, k_org, r1) <= k0 && k1 <= vis_hi(mask, window, k_end, r0))
    return kTileFull;
  return kTileBoundary;
}

// Query rows handled by one prefill work unit: two 128-row tiles.
constexpr int kUnitRows = 256;

TA_HD int pairs_for_rows(int rows) { return (rows + kUnitRows - 1) / kUnitRows; }
// 128-row (query or key) tiles covering `rows` rows.
TA_HD int tiles_for_rows(int rows) { return (rows + kUnitRows / 2 - 1) / (kUnitRows / 2); }
// DOCUMENT_BIDIR work list: the pairs of a segment of `len` rows that cost c key tiles. Every
// pair costs 2 n (n = tiles_for_rows(len)) except the last pair of an odd n, which costs n.
TA_HD int pairs_of_cost(int len, int c) {
  const int n = tiles_for_rows(len), np = pairs_for_rows(len);
  const int full = (n & 1) ? np - 1 : np;
  return (n > 0 && 2 * n == c ? full : 0) + ((n & 1) && n == c ? 1 : 0);
}
// The largest cost below `below` that a segment of `len` rows has pairs of; -1 if none.
TA_HD int cost_below(int len, int below) {
  const int n = tiles_for_rows(len), np = pairs_for_rows(len);
  int c = -1;
  if (n > 0 && ((n & 1) ? np - 1 : np) > 0 && 2 * n < below) c = 2 * n;
  if ((n & 1) && n < below) c = imax(c, n);
  return c;
}

}  // namespace ta
