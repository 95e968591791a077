// prefill.cuh — fused tiled attention forward for sm_103a (no mask, causal, sliding window
// one- and two-sided, document segments causal and non-causal, prefix-LM, and chunked prefill
// over a paged KV cache).
//
// Work unit: two 128-row query tiles of one (batch or segment, query head). The kernel is
// persistent, one CTA per SM: CTA b of G takes units b, 2G-1-b, 2G+b, 4G-1-b, ... of the
// longest-first unit list (a snake over rounds, which evens out the per-SM sums; the list is
// ordered by pair level, or by unit cost for non-causal documents: see decode_unit). The K/V
// ring, three rotating Q buffers and every barrier phase run on across units, so the next
// unit's loads and first S MMAs overlap the current unit's last tiles and epilogue. Within a
// unit the key tiles are visited in ascending order; at d = 64 tile 1's extra tiles come first
// (kRot, see geometry).
//
// The tiled computation with a running row max m and row sum l, rescaling the output
// accumulator by exp(m - m_new) when the max grows, is the one described in "Flash MSA
// Attention Kernel Implementation Tutorial" ("Understanding Flash MSA Core Mechanics"); the
// producer / consumer split with arrive / wait barriers around a double-use shared-memory
// ring follows "FlashAttention-3: Warp Specialization and the 75% FLOPS Barrier on Hopper"
// ("Warp Specialization on Hopper", "The Tensor Memory Accelerator"), re-targeted to
// Blackwell: tcgen05 MMAs with accumulators in tensor memory instead of register WGMMA.
//
// Roles (384 threads):
//   warp 0      TMA producer: per unit, the two Q tiles into the next free Q buffers, then
//               K_j, V_j into a STAGES-deep smem ring.
//   warp 1      MMA issuer (one elected lane) and TMEM owner: S_i = Q_i K_j^T (SS MMA) and
//               O_i += P_i V_j (P read from TMEM, V from smem). At d = 64 (96-key tiles, two
//               S buffers per query tile) warp 1 issues query tile 0's MMAs and warp 2 tile
//               1's.
//   warp 3      paged prefill with pages under 64 tokens only: issues the V_j entries of the
//               ring (warp 0 then issues the Q tiles and the K_j entries).
//   warps 4-7   softmax warpgroup for query tile 0; warps 8-11 for query tile 1. One thread
//               owns one query row (TMEM lane): it reads its S row, applies the element mask
//               on boundary tiles only, updates m and l with exp2, writes P (bf16) back into
//               TMEM over S, rescales its O row only when the max grew by more than 2^8, and
//               finally writes O / l (bf16) and the LSE.
// TMEM columns at d = 128: S_0/P_0 [0,128), S_1/P_1 [128,256), O_0 [256,384), O_1 [384,512).
// At d = 64: S/P buffer b of query tile i at [(2i + b) * 96, (2i + b + 1) * 96), O_0 and O_1 in
// the 128 columns after the four buffers.
//
// Issue order per key tile j at d = 128: PV_0(j-1), S_0(j), PV_1(j-1), S_1(j). tcgen05 MMAs of one
// thread complete in order, so S_i(j) overwrites P_i(j-1) only after PV_i(j-1) has read it,
// and "S_i(j) complete" implies "PV_i(j-1) complete": the softmax may rescale O_i right after
// it sees S_i(j). While warpgroup 0 works on S_0(j), the tensor core runs PV_1 / S_1 and the
// other way round.
#pragma once

#include <cuda_bf16.h>

#include <cfloat>

#include "ptx.cuh"
#include "sched.h"

namespace ta {

struct PrefillParams {
  void* o;                  // bf16 [planes, N, D]
  float* lse;               // fp32 [planes, N]
  const int* cu_seqlens;    // packed kinds: [B+1] segment / query-chunk starts
  const int* seqlens_k;     // PAGED_PREFILL: [B] context lengths (each chunk included)
  const int* table;         // PAGED_PREFILL: [B, max_pages] block table
  int max_pages, page_size, page_shift, num_pages;  // PAGED_PREFILL (page_size = 1 << shift)
  int B, Hq, Hkv, N, group; // N: rows per (batch, head) plane (T for DOCUMENT)
  int num_units;            // work units; DOCUMENT: an upper bound (surplus ones decode invalid)
  int window;               // SLIDING / SLIDING_BIDIR window, PREFIX_LM prefix length
  float scale_log2;         // scale * log2(e)
  const float* q_scales;    // FP8: [B*Hq, nbq] per-128-row-tile scales of Q
  const float* k_scales;    // FP8: [B*Hkv, nbk] per-128-row-tile scales of K
  int nbq, nbk;             // FP8: tiles per plane (ceil(N / 128))
  int* status;
  unsigned long long timeout_ns;
};

// Key-tile width. 128 in general. At d = 64 (but for the paged kind, whose page boxes must
// tile the key tile) 96: each query tile then holds two S buffers in TMEM (4 x 96 + 2 x 64 =
// 512 columns), so S of the next key tile is computed while the softmax works on this one.
__host__ __device__ constexpr int prefill_key_tile(int d, int mask) {
  return d == 64 && mask != kMaskPagedPrefill ? 96 : 128;
}

template <int D, int BN_ = 128>
struct PrefillCfg {
  static constexpr int BM = 128;
  static constexpr int BN = BN_;
  // Two S buffers per query tile (see prefill_key_tile).
  static constexpr bool kDoubleS = BN == 96;
  static constexpr int kThreads = 384;
  static constexpr int kChunkBytes = BM * 128;        // one 64-column, 128-row swizzle panel
  static constexpr int kPanels = D / 64;
  static constexpr int kQBytes = BM * D * 2;
  static constexpr int kKVBytes = BN * D * 2;
  static constexpr int kSmemLimit = 232448;           // 227 KB opt-in maximum per block
  static constexpr int kCtrlBytes = 1024;
  // Three Q buffers for two query tiles: the next unit's tile loads into a buffer released a
  // key tile or more earlier, so its latency hides behind the current unit's last tiles.
  static constexpr int kQBufs = 3;
  static constexpr int kStagesFit =
      (kSmemLimit - 1024 - kCtrlBytes - kQBufs * kQBytes) / kKVBytes;
  static constexpr int kMaxStages = kDoubleS ? 12 : 8;
  static constexpr int kStages = kStagesFit > kMaxStages ? kMaxStages : kStagesFit;
  static constexpr int kSmemBytes = 1024 + kQBufs * kQBytes + kStages * kKVBytes + kCtrlBytes;
  static constexpr int kTmemCols = 512;
  // Launch: 384 threads x 168 registers = 64512. Warpgroup 0 (producer, MMA, two idle warps)
  // drops to 88, the two softmax warpgroups rise to 208: 128*88 + 256*208 = 64512.
  static constexpr uint32_t kRegsControl = 88;
  static constexpr uint32_t kRegsSoftmax = 208;
  static constexpr uint32_t kIdescS = idesc_bf16(BM, BN, false, false);  // Q, K both K-major
  static constexpr uint32_t kIdescO = idesc_bf16(BM, D, false, true);    // V is MN-major
};

template <int ST>
struct PrefillCtrl {
  uint64_t q_full[3];
  uint64_t q_empty[3];  // the epilogue that staged O in the buffer has finished with it
  uint64_t kv_full[ST];
  uint64_t kv_empty[ST];
  uint64_t s_ready[2];
  uint64_t p_ready[2];
  uint64_t o_done[2];
  uint64_t drain[2];  // [1]: the second issuing warp (two S buffers)
  uint32_t tmem_base;
  int abort_flag;
  // Two S buffers per query tile: S ready, P ready and P.V done per (query tile, buffer).
  // One barrier per buffer keeps every parity wait unambiguous: a buffer's next phase needs
  // the consumer of its current one to have moved on.
  uint64_t s_ready2[2][2];
  uint64_t p_ready2[2][2];
  uint64_t pv_done[2][2];
};

struct Unit {
  int valid, bh, kvh, q_row0, k_org, k_end, seq;
};

// Position of one role in the packed unit list. Every role of a CTA visits its units in
// increasing order (round k takes unit kG + b or kG + G-1-b), so each keeps a cursor: the level
// it stands on, the number of units on the levels above it, and the number of segments on it.
// A unit then costs one scan over the segments, plus one more per level passed.
struct UnitCursor {
  int started;  // the segment lengths have been checked and tmax found
  int t;        // current level (tmax before the first one)
  int base;     // units on the levels above t
  int cnt;      // segments holding level t (0 before the first level)
};

// Work unit u in launch order: levels from the deepest (most key tiles) down, then batch /
// segment, then head (heads sharing a kv head are adjacent). The level of a unit is its pair
// index inside its segment, plus, for PAGED_PREFILL, the pairs of context that precede the
// chunk ((context - chunk) / 256), so long contexts start first. For DOCUMENT_BIDIR, where
// every query row of a segment sees the whole segment, a unit costs 2 n key tiles (n = the
// segment's tile count) or n (the last pair of an odd n, whose second tile is empty); its
// level is that cost, a level holds every such pair of every segment (segment, then pair,
// then head), and the list is sorted by cost. Units must be asked for in increasing order
// with the same cursor; warp-collective.
template <int MASK>
__device__ __forceinline__ Unit decode_unit(int u, const PrefillParams& p, UnitCursor& cur) {
  Unit r{0, 0, 0, 0, 0, 0, 0};
  const int lane = static_cast<int>(lane_id());
  if (!is_packed(MASK)) {
    const int per_level = p.B * p.Hq;
    const int npairs = pairs_for_rows(p.N);
    if (u >= per_level * npairs) return r;
    const int level = npairs - 1 - u / per_level;
    const int bh = u % per_level;
    r.valid = 1;
    r.bh = bh;
    r.kvh = (bh / p.Hq) * p.Hkv + (bh % p.Hq) / p.group;
    r.q_row0 = level * kUnitRows;
    r.k_org = 0;
    r.k_end = p.N;
    return r;
  }
  // Packed kinds: the warp scans the segments 32 at a time.
  const int* cu = p.cu_seqlens;
  constexpr bool kCostLevels = MASK == kMaskDocumentBidir;
  // First level of segment s.
  auto level0 = [&](int s) {
    return MASK == kMaskPagedPrefill ? (p.seqlens_k[s] - (cu[s + 1] - cu[s])) / kUnitRows : 0;
  };
  if (!cur.started) {
    int tmax = 0;
    bool bad = false;
    for (int s0 = 0; s0 < p.B; s0 += 32) {
      const int s = s0 + lane;
      if (s < p.B) {
        const int len = cu[s + 1] - cu[s];
        bad |= len < 0;
        if (MASK == kMaskPagedPrefill) {
          const int lk = p.seqlens_k[s];
          bad |= lk < len || lk > p.max_pages * p.page_size;
        }
        if (!bad)
          tmax = imax(tmax, kCostLevels ? 2 * tiles_for_rows(len) + 1
                                        : level0(s) + pairs_for_rows(len));
      }
    }
    for (int off = 16; off; off >>= 1)
      tmax = imax(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    bad = __any_sync(0xffffffffu, bad) || cu[0] != 0 || cu[p.B] != p.N;
    if (bad) {
      if (u == 0 && lane == 0) report_status(p.status, -7);
      cur.t = -1;  // no level: every unit decodes invalid
    } else {
      cur.t = tmax;
    }
    cur.started = 1;
    cur.base = 0;
    cur.cnt = 0;
  }
  // Segment s has a unit at level t iff level0(s) <= t < level0(s) + its pair count.
  auto has_level = [&](int s, int t) {
    const int l0 = level0(s);
    return t >= l0 && t < l0 + pairs_for_rows(cu[s + 1] - cu[s]);
  };
  // Step down to the level holding u, visiting only levels some segment has (for
  // PAGED_PREFILL a long context puts its chunk's units far above level 0).
  while (u >= cur.base + cur.cnt * p.Hq) {
    if (cur.t <= 0) return r;
    int next = -1;  // the highest level below cur.t that some segment has
    for (int s0 = 0; s0 < p.B; s0 += 32) {
      const int s = s0 + lane;
      if (s < p.B) {
        if (kCostLevels) {
          next = imax(next, cost_below(cu[s + 1] - cu[s], cur.t));
        } else {
          const int l0 = level0(s);
          const int c = imin(cur.t - 1, l0 + pairs_for_rows(cu[s + 1] - cu[s]) - 1);
          if (c >= l0) next = imax(next, c);
        }
      }
    }
    for (int off = 16; off; off >>= 1)
      next = imax(next, __shfl_xor_sync(0xffffffffu, next, off));
    cur.base += cur.cnt * p.Hq;
    cur.cnt = 0;
    cur.t = next;
    if (next < 0) return r;
    for (int s0 = 0; s0 < p.B; s0 += 32) {
      const int s = s0 + lane;
      if (kCostLevels) {
        int c = s < p.B ? pairs_of_cost(cu[s + 1] - cu[s], next) : 0;
        for (int off = 16; off; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
        cur.cnt += c;
      } else {
        cur.cnt += __popc(__ballot_sync(0xffffffffu, s < p.B && has_level(s, next)));
      }
    }
  }
  const int t = cur.t;
  const int idx = (u - cur.base) / p.Hq;
  const int h = (u - cur.base) % p.Hq;
  int seen = 0, seg = -1;
  int pair = 0;
  if (kCostLevels) {
    // The idx-th pair on this cost level: an inclusive prefix sum of the segments' counts.
    for (int s0 = 0; s0 < p.B && seg < 0; s0 += 32) {
      const int s = s0 + lane;
      const int len = s < p.B ? cu[s + 1] - cu[s] : 0;
      const int c = s < p.B ? pairs_of_cost(len, t) : 0;
      int incl = c;
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      const unsigned m = __ballot_sync(0xffffffffu, idx < seen + incl);
      if (m) {
        const int src = __ffs(m) - 1;
        const int k = idx - seen - (__shfl_sync(0xffffffffu, incl, src) -
                                    __shfl_sync(0xffffffffu, c, src));
        seg = s0 + src;
        // Pairs of the full cost come first; the odd last pair is on a level of its own.
        pair = 2 * tiles_for_rows(cu[seg + 1] - cu[seg]) == t
                   ? k
                   : pairs_for_rows(cu[seg + 1] - cu[seg]) - 1;
      }
      seen += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (seg < 0) return r;
    r.valid = 1;
    r.bh = h;
    r.kvh = h / p.group;
    r.seq = seg;
    r.k_end = cu[seg + 1];
    r.q_row0 = cu[seg] + pair * kUnitRows;
    r.k_org = cu[seg];
    return r;
  }
  for (int s0 = 0; s0 < p.B && seg < 0; s0 += 32) {
    const int s = s0 + lane;
    unsigned m = __ballot_sync(0xffffffffu, s < p.B && has_level(s, t));
    const int c = __popc(m);
    if (idx < seen + c) {
      for (int z = 0; z < idx - seen; ++z) m &= m - 1;
      seg = s0 + __ffs(m) - 1;
    }
    seen += c;
  }
  r.valid = 1;
  r.bh = h;
  r.kvh = h / p.group;
  r.seq = seg;
  r.k_end = cu[seg + 1];
  r.q_row0 = cu[seg] + (t - level0(seg)) * kUnitRows;
  r.k_org = MASK == kMaskPagedPrefill ? cu[seg] - (p.seqlens_k[seg] - (cu[seg + 1] - cu[seg]))
                                      : cu[seg];
  return r;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Visibility word of one 32-column chunk: bit t is set when column t lies in [lo, hi] (any
// integers; no bit when hi < lo).
__device__ __forceinline__ uint32_t vis_bits32(int lo, int hi) {
  const int a = imax(lo, 0), b = imin(hi, 31);
  return a <= b ? (0xffffffffu >> (31 - (b - a))) << a : 0u;
}

// 32 scores -> 16 packed bf16x2 probabilities exp2(c*s - m); partial sums in sa / sb.
__device__ __forceinline__ void exp2_pack_32(const float* f, float2 cc, float2 mm, float2& sa,
                                             float2& sb, uint32_t* pk) {
#pragma unroll
  for (int t = 0; t < 16; t += 2) {
    const float2 x0 = __ffma2_rn(make_float2(f[2 * t], f[2 * t + 1]), cc, mm);
    const float2 x1 = __ffma2_rn(make_float2(f[2 * t + 2], f[2 * t + 3]), cc, mm);
    const float2 p0 = make_float2(fast_exp2(x0.x), fast_exp2(x0.y));
    const float2 p1 = make_float2(fast_exp2(x1.x), fast_exp2(x1.y));
    sa = __fadd2_rn(sa, p0);
    sb = __fadd2_rn(sb, p1);
    pk[t] = pack_bf16x2(p0.x, p0.y);
    pk[t + 1] = pack_bf16x2(p1.x, p1.y);
  }
}

// FP8: Q and K are E4M3 with one fp32 scale per 128-row tile (the block quantization of the
// FlashAttention-3 page); S = Q K^T runs as tcgen05 kind::f8f6f4 and the two tile scales join
// the softmax's per-tile constant. V, P and O stay bf16. Dense kinds, D = 128 only.
template <int D, int MASK, bool FP8 = false>
__global__ void __launch_bounds__(384, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_o, const PrefillParams p) {
  using C = PrefillCfg<D, prefill_key_tile(D, MASK)>;
  constexpr int BM = C::BM, BN = C::BN, STAGES = C::kStages, QB = C::kQBufs;
  constexpr bool kDB = C::kDoubleS;
  static_assert(!kDB || (D == 64 && !FP8 && MASK != kMaskPagedPrefill), "double S: d = 64");
  // TMEM columns: S (or P) of query tile i, buffer b; the O accumulators after them.
  constexpr int kSBufs = kDB ? 2 : 1;
  constexpr int kOCol = 2 * kSBufs * BN;
  static_assert(kOCol + 2 * D <= C::kTmemCols, "TMEM columns");
  // Visit tile 1's extra key tiles first (see geometry below): at d = 64, for the kinds whose
  // two query tiles can end on different key tiles. Measured on GB300: 5.5 % faster for the
  // causal document workload at d = 64, where the softmax chain dominates; slower at d = 128,
  // where the next unit's tile-1 Q then lands in the buffer that tile 0's epilogue frees last.
  constexpr bool kRot = D == 64 && MASK != kMaskNone && MASK != kMaskDocumentBidir;
  // Boundary-tile mask as one bit test per score, skipping 32-column chunks the whole warp
  // sees (vis_bits32), for the kinds where it measured faster on GB300: the two window kinds
  // (boundary tiles at both edges of every row's range; sliding -4.8 %, two-sided -5.5 %)
  // and the document kinds at d = 64 (-4.3 %). The causal, prefix-LM and paged kinds keep
  // the compare-per-score form: with the other form their kernels compiled to a slower
  // softmax overall (causal N=8192 +6.9 %), though boundary tiles are 1.5 % of their tiles.
  constexpr bool kBitMask = MASK == kMaskSliding || MASK == kMaskSlidingBidir ||
                            (D == 64 && (MASK == kMaskDocument || MASK == kMaskDocumentBidir));
  static_assert(!FP8 || (D == 128 && !is_packed(MASK)), "FP8: dense kinds, D = 128");
  // Q and K tiles: 64 bf16 or 128 E4M3 columns per 128-byte swizzle panel. Q buffers keep
  // their bf16 size in both cases: the epilogue stages the bf16 O tile in them.
  constexpr int kQKPanels = FP8 ? D / 128 : C::kPanels;
  constexpr int kQKPanelCols = FP8 ? 128 : 64;
  constexpr uint32_t kQLoadBytes = BM * D * (FP8 ? 1 : 2);
  constexpr uint32_t kKLoadBytes = BN * D * (FP8 ? 1 : 2);
  constexpr int kSSteps = FP8 ? D / 32 : D / 16;  // 32-byte K steps of one S = Q K^T
  constexpr uint32_t kIdescS = FP8 ? idesc_e4m3(BM, BN) : C::kIdescS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* q_s = smem;                                  // [QB][kQBytes]
  uint8_t* kv_s = smem + QB * C::kQBytes;               // [STAGES][kKVBytes]
  using Ctrl = PrefillCtrl<C::kMaxStages>;
  Ctrl* ctl = reinterpret_cast<Ctrl*>(kv_s + STAGES * C::kKVBytes);
  static_assert(sizeof(Ctrl) <= C::kCtrlBytes, "control block");

  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(lane_id());

  if (warp == 0) {
    if (lane == 0) {
      ctl->abort_flag = 0;
      for (int q = 0; q < QB; ++q) {
        mbar_init(&ctl->q_full[q], 1);
        mbar_init(&ctl->q_empty[q], 4);  // one arrival per epilogue warp
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(&ctl->s_ready[i], 1);
        mbar_init(&ctl->p_ready[i], 128);
        mbar_init(&ctl->o_done[i], 1);
      }
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(&ctl->kv_full[s], 1);
        mbar_init(&ctl->kv_empty[s], kDB ? 2 : 1);  // one release per issuing warp
      }
      if constexpr (kDB) {
        for (int i = 0; i < 2; ++i)
          for (int bb = 0; bb < 2; ++bb) {
            mbar_init(&ctl->s_ready2[i][bb], 1);
            mbar_init(&ctl->p_ready2[i][bb], 128);
            mbar_init(&ctl->pv_done[i][bb], 1);
          }
      }
      mbar_init(&ctl->drain[0], 1);
      mbar_init(&ctl->drain[1], 1);
      fence_mbar_init();
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      prefetch_tensormap(&tm_o);
    }
  } else if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = ctl->tmem_base;
  const WaitCtl wc{p.timeout_ns, p.status, &ctl->abort_flag};
  const WaitCtl wc_drain{p.timeout_ns, p.status, nullptr};
  const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  // The unit of this CTA's k-th round: a snake over the longest-first list.
  auto unit_of = [&](int k) { return k * G + ((k & 1) ? G - 1 - b : b); };
  // Key-tile ranges of a unit's two query tiles and their union [lo, hi). The two ranges
  // overlap for every mask kind, so the union has no gap. Visible keys never move left as the
  // row grows, so tile 0's range starts at lo. Where tile 1's range runs past tile 0's by e1
  // tiles (the diagonal tile of a causal unit) and kRot is set, the unit visits those e1 tiles
  // first and then [lo, hi - e1) in order (kv_at): both query tiles end on the same key tile,
  // and the next unit's first S does not wait for tile 1's extra softmax. Otherwise e1 = 0
  // and the order is plain ascending.
  auto geometry = [&](const Unit& un, KvRange (&rng)[2], int& lo, int& hi) {
    lo = 0x7fffffff;
    hi = -1;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      rng[i] = kv_tile_range(MASK, p.window, un.q_row0 + i * BM, BM, un.k_end, un.k_org,
                             un.k_end, BN);
      if (rng[i].hi > rng[i].lo) {
        lo = imin(lo, rng[i].lo);
        hi = imax(hi, rng[i].hi);
      }
    }
  };
  auto extra_of = [](const KvRange (&rng)[2]) {
    const bool both = rng[0].hi > rng[0].lo && rng[1].hi > rng[1].lo;
    return (both && rng[1].lo >= rng[0].lo && rng[1].lo < rng[0].hi && rng[1].hi > rng[0].hi)
               ? rng[1].hi - rng[0].hi
               : 0;
  };
  // Key tile at position x of a unit's visiting order, and the index of key tile j in query
  // tile i's own sequence of tiles.
  auto kv_at = [](int x, int lo, int hi, int e1) {
    return kRot ? (x < e1 ? hi - e1 + x : lo + x - e1) : lo + x;
  };
  auto tile_index = [](int i, int j, const KvRange (&rng)[2], int hi, int e1) {
    if (kRot && i == 1) return j >= hi - e1 ? j - (hi - e1) : j - rng[1].lo + e1;
    return j - rng[i].lo;
  };
  // Every role walks the same unit sequence; a Q load is counted only for a query tile with
  // work, in tile order, so all roles agree on which buffer (count % QB) holds which tile.
  UnitCursor cur{0, 0, 0, 0};  // this role's place in the packed unit list

  // Register split between warpgroup 0 and the softmax warpgroups. The window and prefix-LM
  // kinds at d = 128 run faster with 96 / 200 (A/B on GB300: sliding window -1 %, two-sided
  // -2.1 %, prefix-LM -3 %; 128*96 + 256*200 = 63488 of the 64512 launched); the other kinds
  // keep 88 / 208 (causal N=8192 unchanged, document d=64 and chunked prefill slower with
  // 96 / 200).
  constexpr bool kWideControl = D == 128 && !FP8 &&
                                (MASK == kMaskSliding || MASK == kMaskSlidingBidir ||
                                 MASK == kMaskPrefixLM);
  constexpr uint32_t kRegsCtl = kWideControl ? 96 : C::kRegsControl;
  constexpr uint32_t kRegsSm = kWideControl ? 200 : C::kRegsSoftmax;
  static_assert(128 * kRegsCtl + 256 * kRegsSm <= 384 * 168, "register split above the launch");
  if (warp < 4) {
    regs_decrease<kRegsCtl>();
    // Paged prefill with pages of 16 or 32 tokens: a key tile is 8 or 4 page boxes per 64-column
    // panel, and one warp issues them more slowly than the tensor core consumes them (a clock64
    // trace put the producer at ~1350 cycles per ring entry against ~750 with 64-token pages). So
    // warp 3, idle otherwise, issues the V entries and warp 0 the Q loads and the K entries.
    // (Written as one comparison with the warp index: the plain "warp == 0 || ..." form, though
    // it reduces to "warp == 0" for the other kinds, changed ptxas's spills in their kernels.)
    const bool split_v = MASK == kMaskPagedPrefill && p.page_shift < 6;
    if (warp == (split_v && warp == 3 ? 3 : 0)) {
      // -------------------------------------------------------------- TMA producer
      int e = 0;   // K/V ring entries issued
      int qn = 0;  // Q loads issued
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int u = unit_of(k);
        if (u >= p.num_units) break;
        const Unit un = decode_unit<MASK>(u, p, cur);  // warp-collective
        if (!un.valid) break;
        KvRange rng[2];
        int lo, hi;
        geometry(un, rng, lo, hi);
        const int e1 = kRot ? extra_of(rng) : 0;
        if (lane == 0) {
          for (int i = 0; i < 2 && ok && (!split_v || warp == 0); ++i) {
            if (rng[i].hi <= rng[i].lo) continue;
            const int qb = qn % QB;
            ok = mbar_wait(&ctl->q_empty[qb], ((qn / QB) & 1) ^ 1, wc);
            if (!ok) break;
            ++qn;
            mbar_arrive_expect_tx(&ctl->q_full[qb], kQLoadBytes);
            for (int c = 0; c < kQKPanels; ++c)
              tma_load_3d(q_s + qb * C::kQBytes + c * C::kChunkBytes, &tm_q, &ctl->q_full[qb],
                          c * kQKPanelCols, un.q_row0 + i * BM, un.bh);
          }
          // Ring entry e holds K or V of the key tile at position x/2 (x = e - first entry of
          // the unit; K for even x).
          for (int x = 0; MASK != kMaskPagedPrefill && x < 2 * (hi - lo) && ok; ++x, ++e) {
            const int st = e % STAGES;
            ok = mbar_wait(&ctl->kv_empty[st], ((e / STAGES) & 1) ^ 1, wc);
            if (!ok) break;
            mbar_arrive_expect_tx(&ctl->kv_full[st], (x & 1) ? C::kKVBytes : kKLoadBytes);
            const CUtensorMap* m = (x & 1) ? &tm_v : &tm_k;
            uint8_t* dst = kv_s + st * C::kKVBytes;
            const int npan = (x & 1) ? C::kPanels : kQKPanels;
            const int pcols = (x & 1) ? 64 : kQKPanelCols;
            for (int c = 0; c < npan; ++c)
              tma_load_3d(dst + c * C::kChunkBytes, m, &ctl->kv_full[st], c * pcols,
                          un.k_org + (kRot ? kv_at(x / 2, lo, hi, e1) : lo + x / 2) * BN,
                          un.kvh);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (MASK == kMaskPagedPrefill) {
          // Key tile j of the sequence is BN / P pages, each its own box of P rows, and lane
          // sb < BN / P owns page sb of every tile: it reads that page's table entry (one tile
          // ahead, so the read overlaps the current tile's copies) and issues its boxes; the
          // table reads and the copies of a tile run in parallel across the lanes. A page past
          // the context, or whose entry is outside the pool (never addressed; the status word
          // reports it), is read from the plane just past the pool, which TMA fills with
          // zeros, so the stage always receives its full bytes.
          const int lp = p.page_shift;
          const int nb = BN >> lp;
          const int lk = un.k_end - un.k_org;
          const int* trow = p.table + static_cast<size_t>(un.seq) * p.max_pages;
          auto plane_of = [&](int j) {
            const int tok = j * BN + (lane << lp);
            int pl = p.num_pages * p.Hkv;
            if (lane < nb && tok < lk) {
              const int raw = __ldg(trow + (tok >> lp));
              if (raw < 0 || raw >= p.num_pages)
                report_status(p.status, -5);
              else
                pl = raw * p.Hkv + un.kvh;
            }
            return pl;
          };
          int pl_next = hi > lo ? plane_of(kv_at(0, lo, hi, e1)) : 0;
          int pl = 0;
          for (int x = 0; x < 2 * (hi - lo) && ok; ++x, ++e) {
            if (split_v && (x & 1) != (warp == 3 ? 1 : 0)) continue;  // the other warp's entry
            const int st = e % STAGES;
            if (lane == 0) ok = mbar_wait(&ctl->kv_empty[st], ((e / STAGES) & 1) ^ 1, wc);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane == 0) mbar_arrive_expect_tx(&ctl->kv_full[st], C::kKVBytes);
            __syncwarp();
            const CUtensorMap* m = (x & 1) ? &tm_v : &tm_k;
            uint8_t* dst = kv_s + st * C::kKVBytes;
            if (split_v || !(x & 1)) pl = pl_next;  // the first entry of its tile this warp issues
            if (lane < nb) {
              for (int c = 0; c < C::kPanels; ++c)
                tma_load_3d(dst + c * C::kChunkBytes + (lane << lp) * 128, m, &ctl->kv_full[st],
                            c * 64, 0, pl);
            }
            if ((split_v || !(x & 1)) && x / 2 + 1 < hi - lo)
              pl_next = plane_of(kv_at(x / 2 + 1, lo, hi, e1));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (lane == 0) {
        // Let copies still in flight land before the CTA can exit (no-op on the normal path).
        for (int x = imax(0, e - STAGES); x < e; ++x)
          mbar_wait(&ctl->kv_full[x % STAGES], (x / STAGES) & 1, wc_drain);
        for (int x = imax(0, qn - QB); x < qn; ++x)
          mbar_wait(&ctl->q_full[x % QB], (x / QB) & 1, wc_drain);
      }
    } else if (warp == 1 || (kDB && warp == 2)) {
      // -------------------------------------------------------------- MMA issuer
      // The whole warp runs this loop, so descriptors and loop state are warp-uniform; one
      // elected lane issues each tcgen05 instruction (see mma_ss). Waits are agreed on by the
      // whole warp so it never diverges.
      constexpr unsigned kFull = 0xffffffffu;
      if constexpr (kDB) {
        // Two S buffers per query tile and one issuing warp per query tile: warp 1 issues
        // tile 0's MMAs, warp 2 tile 1's (one warp for both spent most of each key tile on
        // barrier checks and bookkeeping, on a sub-partition shared with two softmax warps,
        // and fell behind the softmax). Position x of a unit is its x-th key tile in visiting
        // order (kv_at); its K is ring entry e + 2x, its V e + 2x + 1. The S of positions 0
        // and 1 go first; step x issues P.V of position x and then the S of position x + 2
        // into the buffer that P.V has just read (MMAs of one thread run in order), so the
        // tile's next S is computed while its softmax works on the current one. Every ring
        // entry takes one release from each issuer (kv_empty counts two), and each issuer
        // waits for an entry to land before releasing it, used or not, so neither can release
        // a slot ahead of its refill.
        const int i = warp - 1;  // this warp's query tile
        int e = 0;               // ring entry of the unit's first K
        int qc = 0;              // Q loads of both tiles before this unit
        int sn = 0;              // S tiles issued so far (buffer sn & 1)
        int pn = 0;              // P tiles consumed so far (buffer pn & 1)
        bool ok = true;
        for (int k = 0; ok; ++k) {
          const int u = unit_of(k);
          if (u >= p.num_units) break;
          const Unit un = decode_unit<MASK>(u, p, cur);  // warp-collective
          if (!un.valid) break;
          KvRange rng[2];
          int lo, hi;
          geometry(un, rng, lo, hi);
          const int e1 = kRot ? extra_of(rng) : 0;
          const int npos = hi - lo;
          const int n0 = rng[0].hi > rng[0].lo ? 1 : 0, n1 = rng[1].hi > rng[1].lo ? 1 : 0;
          const int qn = i == 0 ? qc : qc + n0;  // this tile's Q load
          const uint64_t q_desc = sw128_desc(smem_u32(q_s + (qn % QB) * C::kQBytes), 16, 1024);
          const int rlo = i ? rng[1].lo : rng[0].lo, rhi = i ? rng[1].hi : rng[0].hi;
          const int tlen = rhi - rlo;
          // Index of key tile j in this tile's own visiting order (see tile_index).
          auto my_index = [&](int j) {
            return (kRot && i == 1) ? (j >= hi - e1 ? j - (hi - e1) : j - rlo + e1) : j - rlo;
          };
          auto key_at = [&](int x) { return kRot ? kv_at(x, lo, hi, e1) : lo + x; };
          // Satisfied checks are tested once first and the bounded wait runs only when an
          // entry is not there yet (as in the d = 128 issuer below): these warps share their
          // sub-partitions with the softmax warps that bound d = 64. Measured on GB300: dense
          // causal -1.5 %, non-causal document -3 %, no mask and sliding window -1.9 %.
          auto wait_entry = [&](int en) {
            if (__all_sync(kFull, mbar_try_wait(&ctl->kv_full[en % STAGES], (en / STAGES) & 1)))
              return true;
            return __all_sync(kFull,
                              mbar_wait(&ctl->kv_full[en % STAGES], (en / STAGES) & 1, wc)) != 0;
          };
          // S of position x (if this tile sees that key tile), then release K of x.
          auto do_k = [&](int x) -> bool {
            const int en = e + 2 * x;
            if (!wait_entry(en)) return false;
            tc_fence_after();
            const int j = key_at(x);
            if (j >= rlo && j < rhi) {
              if (my_index(j) == 0) {  // the tile's first S: its Q
                if (!__all_sync(kFull, mbar_wait(&ctl->q_full[qn % QB], (qn / QB) & 1, wc)))
                  return false;
                tc_fence_after();
              }
              const int buf = sn & 1;
              const uint32_t d_s = tmem + (i * 2 + buf) * BN;
              const uint64_t k_desc =
                  sw128_desc(smem_u32(kv_s + (en % STAGES) * C::kKVBytes), 16, 1024);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off16 = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
                mma_ss(d_s, q_desc + off16, k_desc + off16, C::kIdescS, kk > 0 ? 1u : 0u);
              }
              mma_commit(&ctl->s_ready2[i][buf]);
              ++sn;
            }
            mma_commit(&ctl->kv_empty[en % STAGES]);
            return true;
          };
          // P.V of position x into O (the tile's first one overwrites it), then release V.
          auto do_v = [&](int x) -> bool {
            const int en = e + 2 * x + 1;
            if (!wait_entry(en)) return false;
            tc_fence_after();
            const int j = key_at(x);
            if (j >= rlo && j < rhi) {
              const int buf = pn & 1;
              if (!__all_sync(kFull, mbar_try_wait(&ctl->p_ready2[i][buf], (pn >> 1) & 1)) &&
                  !__all_sync(kFull, mbar_wait(&ctl->p_ready2[i][buf], (pn >> 1) & 1, wc)))
                return false;
              tc_fence_after();
              const int t = my_index(j);
              const uint32_t d_o = tmem + kOCol + i * D;
              const uint32_t a_p = tmem + (i * 2 + buf) * BN;
              const uint64_t v_desc =
                  sw128_desc(smem_u32(kv_s + (en % STAGES) * C::kKVBytes), C::kChunkBytes, 1024);
#pragma unroll
              for (int kk = 0; kk < BN / 16; ++kk)
                mma_ts(d_o, a_p + kk * 8, v_desc + kk * (2048 >> 4), C::kIdescO,
                       kk > 0 ? 1u : (t > 0 ? 1u : 0u));
              mma_commit(&ctl->pv_done[i][buf]);
              if (t + 1 == tlen) mma_commit(&ctl->o_done[i]);
              ++pn;
            }
            mma_commit(&ctl->kv_empty[en % STAGES]);
            return true;
          };
          bool okk = true;
          for (int x = 0; x < 2 && x < npos && okk; ++x) okk = do_k(x);
          for (int x = 0; x < npos && okk; ++x) {
            okk = do_v(x);
            if (okk && x + 2 < npos) okk = do_k(x + 2);
          }
          ok = okk;
          e += 2 * npos;
          qc += n0 + n1;
        }
      } else {
      int e = 0;              // ring entry of the next K
      int qc = 0;             // Q loads consumed before this unit
      int pb0 = 0, pb1 = 0;   // P tiles consumed before this unit, per query tile
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int u = unit_of(k);
        if (u >= p.num_units) break;
        const Unit un = decode_unit<MASK>(u, p, cur);  // warp-collective
        if (!un.valid) break;
        KvRange rng[2];
        int lo, hi;
        geometry(un, rng, lo, hi);
        const int e1 = kRot ? extra_of(rng) : 0;
        auto active = [&](int i, int j) { return j >= rng[i].lo && j < rng[i].hi; };
        const int qn0 = qc, qn1 = qc + (rng[0].hi > rng[0].lo ? 1 : 0);
        // Descriptors of the two Q tiles; a K step adds its byte offset / 16 to the start
        // field, which stays inside its 14 bits for any shared-memory address.
        const uint64_t q_desc0 = sw128_desc(smem_u32(q_s + (qn0 % QB) * C::kQBytes), 16, 1024);
        const uint64_t q_desc1 = sw128_desc(smem_u32(q_s + (qn1 % QB) * C::kQBytes), 16, 1024);
        // Step x = j - lo: the P.V of the key tile at position x - 1 and the S of the one at x.
        for (int j = lo; j <= hi && ok; ++j) {
          const bool have_v = j > lo;
          const bool have_k = j < hi;
          const int jv = kRot ? kv_at(j - 1 - lo, lo, hi, e1) : j - 1;
          const int jk = kRot ? kv_at(j - lo, lo, hi, e1) : j;
          const int ev = e - 1, ek = e;  // V of position x - 1 precedes K of x in the ring
          // This warp issues every MMA of the CTA, and a clock64 trace put it, not the softmax,
          // on the critical path at d = 128: its satisfied barrier checks cost ~430 cycles per
          // step done one after the other. So V's and K's entries are tested together first
          // (two independent try_waits, one vote); the bounded waits run only if one is not
          // ready. Measured on GB300: causal B2 Hq32 Hkv8 N8192 -3.5 %, sliding window -3.9 %,
          // causal B4 H16 N2048 -2.8 %.
          {
            const bool rv = !have_v || mbar_try_wait(&ctl->kv_full[ev % STAGES], (ev / STAGES) & 1);
            const bool rk = !have_k || mbar_try_wait(&ctl->kv_full[ek % STAGES], (ek / STAGES) & 1);
            if (!__all_sync(kFull, rv && rk)) {
              if (have_v)
                ok = __all_sync(kFull,
                                mbar_wait(&ctl->kv_full[ev % STAGES], (ev / STAGES) & 1, wc));
              if (have_k && ok)
                ok = __all_sync(kFull,
                                mbar_wait(&ctl->kv_full[ek % STAGES], (ek / STAGES) & 1, wc));
            }
          }
          if (!ok) break;
          tc_fence_after();
          // V panel: 128 keys x 64 columns; a K step of 16 keys is 2048 bytes; the next
          // 64-column panel (N direction) is kChunkBytes further (LBO), 8-key groups are 1024
          // bytes apart (SBO). K is K-major like Q.
          const uint64_t v_desc =
              sw128_desc(smem_u32(kv_s + (ev % STAGES) * C::kKVBytes), C::kChunkBytes, 1024);
          const uint64_t k_desc =
              sw128_desc(smem_u32(kv_s + (ek % STAGES) * C::kKVBytes), 16, 1024);
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (!ok) break;
            if (have_v && active(i, jv)) {
              // The unit's first P.V overwrites O_i. The previous unit's epilogue has read O_i
              // out by then: the softmax threads publish this P only after it.
              const int pv = kRot ? tile_index(i, jv, rng, hi, e1) : 0;
              const int pn = (i ? pb1 : pb0) + (kRot ? pv : j - 1 - rng[i].lo);
              if (!__all_sync(kFull, mbar_try_wait(&ctl->p_ready[i], pn & 1)))
                ok = __all_sync(kFull, mbar_wait(&ctl->p_ready[i], pn & 1, wc));
              if (!ok) break;
              tc_fence_after();
              const uint32_t d_o = tmem + 256 + i * D;
              const uint32_t a_p = tmem + i * 128;
              const uint32_t acc0 = (kRot ? pv > 0 : j - 1 > rng[i].lo) ? 1u : 0u;
              // The paged kind at d = 128 issues each chain of eight MMAs from one elected
              // block: 3 % faster there on GB300 with 16-token pages. The other kinds compiled
              // to a slower kernel with it (more spills in the softmax) and keep one call per
              // MMA.
              if constexpr (MASK == kMaskPagedPrefill && D == 128) {
                mma_ts_chain8(d_o, a_p, v_desc, C::kIdescO, acc0);
              } else {
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                  mma_ts(d_o, a_p + kk * 8, v_desc + kk * (2048 >> 4), C::kIdescO,
                         kk > 0 ? 1u : acc0);
              }
              if (kRot ? pv + 1 == rng[i].hi - rng[i].lo : j == rng[i].hi)
                mma_commit(&ctl->o_done[i]);
              // Release this V as soon as its last reader is issued.
              if (i == 1 || !active(1, jv)) mma_commit(&ctl->kv_empty[ev % STAGES]);
            }
            if (have_k && active(i, jk)) {
              if (kRot ? tile_index(i, jk, rng, hi, e1) == 0 : j == rng[i].lo) {
                const int qn = i ? qn1 : qn0;
                ok = __all_sync(kFull, mbar_wait(&ctl->q_full[qn % QB], (qn / QB) & 1, wc));
                if (!ok) break;
                tc_fence_after();
              }
              const uint32_t d_s = tmem + i * 128;
              const uint64_t q_desc = i ? q_desc1 : q_desc0;
              if constexpr (MASK == kMaskPagedPrefill && D == 128 && !FP8) {
                mma_ss_chain8<C::kChunkBytes / 16>(d_s, q_desc, k_desc, kIdescS);
              } else {
#pragma unroll
                for (int kk = 0; kk < kSSteps; ++kk) {
                  // K-major panels: a K step (16 bf16 or 32 E4M3 columns) is 32 bytes inside a
                  // 128-byte swizzle row; every 4 steps move to the next panel. 8-row groups:
                  // 1024 B.
                  const uint32_t off16 = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
                  if constexpr (FP8)
                    mma_ss_f8(d_s, q_desc + off16, k_desc + off16, kIdescS, kk > 0 ? 1u : 0u);
                  else
                    mma_ss(d_s, q_desc + off16, k_desc + off16, kIdescS, kk > 0 ? 1u : 0u);
                }
              }
              mma_commit(&ctl->s_ready[i]);
            }
          }
          if (!ok) break;
          if (have_k) {
            mma_commit(&ctl->kv_empty[ek % STAGES]);
            e += 2;  // K and V of position x; the last step only drains the last V
          }
        }
        qc = qn1 + (rng[1].hi > rng[1].lo ? 1 : 0);
        pb0 += imax(rng[0].hi - rng[0].lo, 0);
        pb1 += imax(rng[1].hi - rng[1].lo, 0);
      }
      }
      // Every MMA this warp issued has completed before TMEM can be released.
      mma_commit(&ctl->drain[warp - 1]);
      mbar_wait(&ctl->drain[warp - 1], 0, wc_drain);
    }
  } else {
    regs_increase<kRegsSm>();
    // ---------------------------------------------------------------- softmax warpgroups
    const int i = (warp - 4) >> 2;          // query tile
    const int quarter = warp & 3;           // TMEM lanes [32*quarter, 32*quarter + 32)
    const int r = quarter * 32 + lane;      // row inside the tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t s_col = lane_base + i * 128;
    const uint32_t o_col = lane_base + kOCol + i * D;
    const float c0 = p.scale_log2;
    int sc = 0, oc = 0;  // S tiles and finished units of this query tile consumed
    int pending_q = -1;  // tile 1: Q buffer whose O store may still be reading it
    auto release_pending = [&]() {
      if (pending_q >= 0) {
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->q_empty[pending_q]);
        pending_q = -1;
      }
    };
    int qc = 0;          // Q loads of all tiles before this unit
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = unit_of(k);
      if (u >= p.num_units) break;
      const Unit un = decode_unit<MASK>(u, p, cur);  // warp-collective
      if (!un.valid) break;
      KvRange rng[2];
      int lo_u, hi_u;
      geometry(un, rng, lo_u, hi_u);
      const int e1 = kRot ? extra_of(rng) : 0;
      const KvRange my = i ? rng[1] : rng[0];
      const int qn = qc + ((i == 1 && rng[0].hi > rng[0].lo) ? 1 : 0);  // this tile's Q load
      qc += (rng[0].hi > rng[0].lo ? 1 : 0) + (rng[1].hi > rng[1].lo ? 1 : 0);
      if (my.hi <= my.lo) {
        release_pending();  // no key tile here to release it after
        continue;
      }
      const int q_row0 = un.q_row0, k_org = un.k_org, k_end = un.k_end, bh = un.bh;
      const int row_end = k_end;  // query rows and keys share one index space
      const int row = q_row0 + i * BM + r;  // absolute query row
      float m_run = -INFINITY;  // running max in log2 units (may trail the true max by < 8)
      float l_run = 0.f;
      // FP8: this query tile's scale; each key tile's joins it below.
      const float cq = FP8 ? c0 * __ldg(p.q_scales + static_cast<size_t>(bh) * p.nbq +
                                        (q_row0 + i * BM) / BM)
                           : c0;
      // Tile 1 visits its e1 extra tiles first, then the rest in order (see geometry).
      const int ex = i ? e1 : 0;
      for (int j0 = my.lo; j0 < my.hi && ok; ++j0) {
        const int j = !kRot ? j0 : (j0 - my.lo < ex ? my.hi - ex + (j0 - my.lo) : j0 - ex);
        // Scale of the raw scores in log2 units. FP8: times the key tile's scale, kept
        // positive (a zero scale means an all-zero tile, whose raw scores are 0; a positive
        // floor keeps masked -inf scores at -inf instead of NaN).
        const float c =
            FP8 ? fmaxf(cq * __ldg(p.k_scales + static_cast<size_t>(un.kvh) * p.nbk + j),
                        FLT_MIN)
                : c0;
        if constexpr (kDB) {
          // Key tiles of 96: three 32-column chunks, S in buffer sc & 1 of this tile.
          const int sbuf = sc & 1;
          ok = __all_sync(0xffffffffu, mbar_wait(&ctl->s_ready2[i][sbuf], (sc >> 1) & 1, wc));
          if (!ok) break;
          tc_fence_after();
          const uint32_t sb_col = lane_base + (i * 2 + sbuf) * BN;
          uint32_t s0[32], s1[32], s2[32];
          tmem_ld_x32(sb_col + 0, s0);
          tmem_ld_x32(sb_col + 32, s1);
          tmem_ld_x32(sb_col + 64, s2);
          tmem_wait_ld_x32(s0);
          tmem_wait_ld_x32(s1);
          tmem_wait_ld_x32(s2);
          float* f0 = reinterpret_cast<float*>(s0);
          float* f1 = reinterpret_cast<float*>(s1);
          float* f2 = reinterpret_cast<float*>(s2);
          const int kind = tile_kind(MASK, p.window, q_row0 + i * BM, BM, row_end, k_org,
                                     k_end, BN, j);
          if (kind == kTileBoundary) {
            const int key0 = k_org + j * BN;
            const int lo_k = vis_lo(MASK, p.window, k_org, row) - key0;
            const int hi_k = vis_hi(MASK, p.window, k_end, row) - key0;
            if constexpr (kBitMask) {
              const uint32_t b0 = vis_bits32(lo_k, hi_k), b1 = vis_bits32(lo_k - 32, hi_k - 32);
              const uint32_t b2 = vis_bits32(lo_k - 64, hi_k - 64);
              if (!__all_sync(0xffffffffu, b0 == 0xffffffffu)) {
#pragma unroll
                for (int t = 0; t < 32; ++t)
                  if (!(b0 & (1u << t))) f0[t] = -INFINITY;
              }
              if (!__all_sync(0xffffffffu, b1 == 0xffffffffu)) {
#pragma unroll
                for (int t = 0; t < 32; ++t)
                  if (!(b1 & (1u << t))) f1[t] = -INFINITY;
              }
              if (!__all_sync(0xffffffffu, b2 == 0xffffffffu)) {
#pragma unroll
                for (int t = 0; t < 32; ++t)
                  if (!(b2 & (1u << t))) f2[t] = -INFINITY;
              }
            } else {
#pragma unroll
              for (int t = 0; t < 32; ++t) {
                if (t < lo_k || t > hi_k) f0[t] = -INFINITY;
                if (t + 32 < lo_k || t + 32 > hi_k) f1[t] = -INFINITY;
                if (t + 64 < lo_k || t + 64 > hi_k) f2[t] = -INFINITY;
              }
            }
          }
          // Row max: three independent chains of 3-input max over the 96 scores.
          float mx0 = fmax3(f0[0], f0[1], f0[2]), mx1 = fmax3(f1[0], f1[1], f1[2]);
          float mx2 = fmax3(f2[0], f2[1], f2[2]);
#pragma unroll
          for (int t = 3; t < 31; t += 2) {
            mx0 = fmax3(mx0, f0[t], f0[t + 1]);
            mx1 = fmax3(mx1, f1[t], f1[t + 1]);
            mx2 = fmax3(mx2, f2[t], f2[t + 1]);
          }
          mx0 = fmax3(mx0, f0[31], f1[31]);
          const float m_tile = fmax3(mx0, mx1, fmaxf(mx2, f2[31])) * c;
          float alpha = 1.f;
          if (m_tile > m_run + 8.f) {
            alpha = fast_exp2(m_run - m_tile);  // 0 when m_run is -inf
            m_run = m_tile;
          }
          if (j0 > my.lo && __any_sync(0xffffffffu, alpha < 1.f)) {
            // O holds this tile's previous P.V only once that MMA has finished: here S of
            // this key tile was issued before it, so wait for it explicitly.
            const int pv = sc - 1;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&ctl->pv_done[i][pv & 1], (pv >> 1) & 1, wc));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < D / 16; ++cc) {
              uint32_t ov[16];
              tmem_ld_x16(o_col + cc * 16, ov);
              tmem_wait_ld_x16(ov);
#pragma unroll
              for (int t = 0; t < 16; ++t)
                ov[t] = __float_as_uint(__uint_as_float(ov[t]) * alpha);
              tmem_st_x16(o_col + cc * 16, ov);
            }
          }
          const float msub = (m_run == -INFINITY) ? 0.f : m_run;
          const float2 cc2 = make_float2(c, c);
          const float2 mm = make_float2(-msub, -msub);
          float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
          uint32_t pk[16];
          exp2_pack_32(f0, cc2, mm, sa, sb, pk);
          tmem_st_x16(sb_col + 0, pk);
          exp2_pack_32(f1, cc2, mm, sa, sb, pk);
          tmem_st_x16(sb_col + 16, pk);
          exp2_pack_32(f2, cc2, mm, sa, sb, pk);
          tmem_st_x16(sb_col + 32, pk);
          l_run = l_run * alpha + ((sa.x + sa.y) + (sb.x + sb.y));
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&ctl->p_ready2[i][sbuf]);
          ++sc;
        } else {
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl->s_ready[i], (sc++) & 1, wc));
        if (!ok) break;
        tc_fence_after();
        uint32_t s0[32], s1[32], s2[32], s3[32];
        tmem_ld_x32(s_col + 0, s0);
        tmem_ld_x32(s_col + 32, s1);
        tmem_ld_x32(s_col + 64, s2);
        tmem_ld_x32(s_col + 96, s3);
        tmem_wait_ld_x32(s0);
        tmem_wait_ld_x32(s1);
        tmem_wait_ld_x32(s2);
        tmem_wait_ld_x32(s3);
        float* f0 = reinterpret_cast<float*>(s0);
        float* f1 = reinterpret_cast<float*>(s1);
        float* f2 = reinterpret_cast<float*>(s2);
        float* f3 = reinterpret_cast<float*>(s3);
        const int kind = tile_kind(MASK, p.window, q_row0 + i * BM, BM, row_end, k_org, k_end,
                                   BN, j);
        if (kind == kTileBoundary) {
          const int key0 = k_org + j * BN;
          const int lo_k = vis_lo(MASK, p.window, k_org, row) - key0;
          const int hi_k = vis_hi(MASK, p.window, k_end, row) - key0;
          if constexpr (kBitMask) {
            // One bit test per score; a chunk visible to all 32 rows of the warp is skipped.
            const uint32_t b0 = vis_bits32(lo_k, hi_k), b1 = vis_bits32(lo_k - 32, hi_k - 32);
            const uint32_t b2 = vis_bits32(lo_k - 64, hi_k - 64);
            const uint32_t b3 = vis_bits32(lo_k - 96, hi_k - 96);
            if (!__all_sync(0xffffffffu, b0 == 0xffffffffu)) {
#pragma unroll
              for (int t = 0; t < 32; ++t)
                if (!(b0 & (1u << t))) f0[t] = -INFINITY;
            }
            if (!__all_sync(0xffffffffu, b1 == 0xffffffffu)) {
#pragma unroll
              for (int t = 0; t < 32; ++t)
                if (!(b1 & (1u << t))) f1[t] = -INFINITY;
            }
            if (!__all_sync(0xffffffffu, b2 == 0xffffffffu)) {
#pragma unroll
              for (int t = 0; t < 32; ++t)
                if (!(b2 & (1u << t))) f2[t] = -INFINITY;
            }
            if (!__all_sync(0xffffffffu, b3 == 0xffffffffu)) {
#pragma unroll
              for (int t = 0; t < 32; ++t)
                if (!(b3 & (1u << t))) f3[t] = -INFINITY;
            }
          } else {
#pragma unroll
            for (int t = 0; t < 32; ++t) {
              if (t < lo_k || t > hi_k) f0[t] = -INFINITY;
              if (t + 32 < lo_k || t + 32 > hi_k) f1[t] = -INFINITY;
              if (t + 64 < lo_k || t + 64 > hi_k) f2[t] = -INFINITY;
              if (t + 96 < lo_k || t + 96 > hi_k) f3[t] = -INFINITY;
            }
          }
        }
        // Row max: four independent chains of 3-input max over the 128 scores.
        float mx0 = fmax3(f0[0], f0[1], f0[2]), mx1 = fmax3(f1[0], f1[1], f1[2]);
        float mx2 = fmax3(f2[0], f2[1], f2[2]), mx3 = fmax3(f3[0], f3[1], f3[2]);
#pragma unroll
        for (int t = 3; t < 31; t += 2) {
          mx0 = fmax3(mx0, f0[t], f0[t + 1]);
          mx1 = fmax3(mx1, f1[t], f1[t + 1]);
          mx2 = fmax3(mx2, f2[t], f2[t + 1]);
          mx3 = fmax3(mx3, f3[t], f3[t + 1]);
        }
        mx0 = fmax3(mx0, f0[31], f1[31]);
        mx2 = fmax3(mx2, f2[31], f3[31]);
        const float m_tile = fmax3(fmaxf(mx0, mx1), mx2, mx3) * c;
        float alpha = 1.f;
        // Conditional rescale: move the reference max only when the tile max exceeds it by
        // more than 8 (a factor 256 in exp2), so most tiles skip the O read-modify-write.
        if (m_tile > m_run + 8.f) {
          alpha = fast_exp2(m_run - m_tile);  // 0 when m_run is -inf
          m_run = m_tile;
        }
        if (j0 > my.lo && __any_sync(0xffffffffu, alpha < 1.f)) {
          // 16 columns at a time: the 128 scores are still live here.
#pragma unroll
          for (int cc = 0; cc < D / 16; ++cc) {
            uint32_t ov[16];
            tmem_ld_x16(o_col + cc * 16, ov);
            tmem_wait_ld_x16(ov);
#pragma unroll
            for (int t = 0; t < 16; ++t)
              ov[t] = __float_as_uint(__uint_as_float(ov[t]) * alpha);
            tmem_st_x16(o_col + cc * 16, ov);
          }
        }
        const float msub = (m_run == -INFINITY) ? 0.f : m_run;
        // p = exp2(c*s - m) two at a time: one packed FMA, two MUFU ex2, one packed add into
        // two independent partial sums, one bf16x2 pack.
        const float2 cc2 = make_float2(c, c);
        const float2 mm = make_float2(-msub, -msub);
        float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
        uint32_t pk[16];
        exp2_pack_32(f0, cc2, mm, sa, sb, pk);
        tmem_st_x16(s_col + 0, pk);
        exp2_pack_32(f1, cc2, mm, sa, sb, pk);
        tmem_st_x16(s_col + 16, pk);
        exp2_pack_32(f2, cc2, mm, sa, sb, pk);
        tmem_st_x16(s_col + 32, pk);
        exp2_pack_32(f3, cc2, mm, sa, sb, pk);
        tmem_st_x16(s_col + 48, pk);
        l_run = l_run * alpha + ((sa.x + sa.y) + (sb.x + sb.y));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&ctl->p_ready[i]);
        }
        release_pending();
      }
      if (!ok) break;
      // -------------------------------------------------------------- epilogue
      ok = __all_sync(0xffffffffu, mbar_wait(&ctl->o_done[i], (oc++) & 1, wc));
      if (!ok) break;
      tc_fence_after();
      const bool live = row < row_end;
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      // The warp's 32 rows go out through shared memory and one TMA store per 64-column
      // panel, staged in this tile's Q buffer (its last S MMA completed before o_done) in the
      // 128-byte-swizzled layout the store expects; the buffer goes back to the producer once
      // the stores have read it. Rows past the tensor's extent are clipped by the store; a
      // DOCUMENT warp whose rows run past its segment writes them one thread per row instead,
      // so the next segment's rows stay untouched.
      const int warp_row0 = q_row0 + i * BM + quarter * 32;
      const bool staged = !is_packed(MASK) || warp_row0 + 31 < row_end;
      uint8_t* stage = q_s + (qn % QB) * C::kQBytes;
      uint8_t* orow = static_cast<uint8_t*>(p.o) +
                      (static_cast<size_t>(bh) * p.N + static_cast<size_t>(row)) * D * 2;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t ov[32];
        tmem_ld_x32(o_col + cc * 32, ov);
        tmem_wait_ld_x32(ov);
        uint32_t w[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
          w[t] = pack_bf16x2(__uint_as_float(ov[2 * t]) * inv_l,
                             __uint_as_float(ov[2 * t + 1]) * inv_l);
        if (staged) {
          // 16-byte chunk k of row r sits at chunk k ^ (r % 8) of the row's 128 bytes.
          const uint32_t rbase = smem_u32(stage + (cc >> 1) * C::kChunkBytes + r * 128);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            st_shared_v4(rbase + ((((cc & 1) * 4 + v4) ^ (r & 7)) << 4), w[4 * v4],
                         w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
        } else if (live) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            st_global_v4(orow + cc * 64 + v4 * 16, w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2],
                         w[4 * v4 + 3]);
        }
      }
      if (staged && warp_row0 < row_end) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (int cp = 0; cp < C::kPanels; ++cp)
            tma_store_3d(&tm_o, stage + cp * C::kChunkBytes + quarter * 32 * 128, cp * 64,
                         warp_row0, bh);
          bulk_commit_group();
        }
      }
      // The buffer goes back to the producer only after the stores have read it. Tile 0's
      // buffer takes the next unit's tile-1 Q, so it is released now. Tile 1's takes a Q two
      // units on: for the causal kinds it is released after this warp's next key tile (or at
      // the end), so tile 1 starts its next unit without waiting for the store (measured: a
      // gain for causal, causal-document and paged prefill, a loss for the two-sided window).
      constexpr bool kDeferTile1 =
          MASK == kMaskCausal || MASK == kMaskDocument || MASK == kMaskPagedPrefill;
      if (i == 0 || !kDeferTile1) {
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->q_empty[qn % QB]);
      } else {
        pending_q = qn % QB;
      }
      if (live)
        p.lse[static_cast<size_t>(bh) * p.N + row] =
            l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994530942f : -INFINITY;
    }
    release_pending();  // the last unit's store, before shared memory goes away
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace ta
