// decode.cuh — paged-KV decode (one query token per sequence) with split-KV partials and a
// fused log-sum-exp-weighted combine.
//
// The KV cache is a pool of pages [num_pages, Hkv, P, D] (P = 16, 32, 64 or 128 tokens);
// sequence b's logical page p lives at physical page block_table[b][p] ("Optimizing Triton
// Kernels for Custom Attention Patterns on H100", Pattern C). Instead of first gathering pages
// into a dense buffer, the producer warp issues TMA boxes straight from the pool into a
// shared-memory ring of 64-token stages (64/P pages per stage, or half a 128-token page), so
// every K/V byte crosses HBM once. The same kernel also reads dense
// per-sequence caches [B, Hkv, L, D] (p.dense): the second stage of that page's two-stage
// path, which first gathers the pages into such a cache.
//
// Grid (split, kv head g, sequence b): a CTA handles `chunk_pages` 64-token stages of one
// (b, g) (32 when the batch has at least as many (b, g) groups as SMs, else 16; the host
// chooses) for all G = Hq/Hkv query heads of the group. Decode reads each K/V byte once and is HBM-bound;
// the arithmetic only has to stay off the critical path. It runs as warp-level bf16 MMAs
// (mma.sync m16n8k16, fp32 accumulate) with the G heads as the rows of a 16-row tile: an
// instruction-count choice, not a throughput one (scalar FMAs needed ~600 instructions per
// thread per page and made the consumers, not HBM, the bottleneck). Each of the four consumer
// warps owns a 16-token slice of every page and keeps its own running max, sum and O (the
// online softmax of "Flash MSA Attention Kernel Implementation Tutorial", "Understanding Flash
// MSA Core Mechanics", in exp2 form), so pages need no cross-warp synchronisation; the four
// partial results are merged once per chunk with the same rescaling identity.
//
// Combine: each split writes its unnormalised O, max m and sum l (log2 units) to the
// workspace; the last split to finish (atomic ticket per (b, g)) merges them in split order,
// each thread loading a batch of splits at once for four columns of one head:
//   M = max_c m_c,  L = sum_c l_c 2^(m_c - M),  O = sum_c O_c 2^(m_c - M) / L,
//   LSE = (M + log2 L) ln 2
// — the same rescaling identity as the online update, applied across splits. The order is
// fixed, so results are bit-reproducible.
#pragma once

#include "ptx.cuh"
#include "sched.h"

namespace ta {

struct DecodeParams {
  const uint4* q;        // bf16 [B, Hq, 1, D]
  const int* cu;         // [B+1] cumulative context lengths
  const int* table;      // [B, max_pages] (max_pages = ceil(longest context / page_size))
  void* o;               // bf16 [B, Hq, 1, D]
  float* lse;            // [B, Hq]
  float* part_o;         // [B*Hkv, max_splits, G, D]
  float* part_ml;        // [B*Hkv, max_splits, G, 2]
  int* counters;         // [B*Hkv], zero before the launch
  int B, Hq, Hkv, max_pages, num_pages, max_splits, chunk_pages;
  int group;             // query heads per kv head, Hq / Hkv (at most the kernel's tile rows)
  int page_shift;        // log2 of the tokens per pool page (paged: 4..7); a TMA box holds
                         // min(page_size, 64) rows
  int dense;             // 1: K/V are dense caches [B*Hkv, max_len, D], no block table
  int max_len;           // longest valid context (N: the cache rows, or the table's reach)
  float scale_log2;
  int* status;
  unsigned long long timeout_ns;
};

template <int D, int G>  // G: tile rows holding query heads
struct DecodeCfg {
  static constexpr int kPage = 64;  // tokens per ring stage
  static constexpr int kWarps = 4;  // consumer warp w owns tokens [16w, 16w + 16) of each page
  static constexpr int kConsumers = kWarps * 32;
  static constexpr int kThreads = kConsumers + 32;
  static constexpr int kPanels = D / 64;
  static constexpr int kPanelBytes = kPage * 128;           // 64 tokens x 64 columns
  static constexpr int kPageBytes = kPage * D * 2;          // one (page, kv-head) of K or V
  static constexpr int kStageBytes = 2 * kPageBytes;        // K and V
  static constexpr int kStages = (96 * 1024) / kStageBytes; // 3 (D=128), 6 (D=64)
  static constexpr int kKSteps = D / 16;                    // k-steps of S = Q K^T
  static constexpr int kNTiles = D / 8;                     // n-tiles of O += P V
  static constexpr bool kHi = G > 8;                        // rows 8..15 of the tile are heads
  static constexpr int kRingBytes = kStages * kStageBytes;
  // misc area: control 256 | per-warp row max [4][16] | per-warp row sum [4][16]
  static constexpr int kOffMax = 256, kOffSum = 512, kMiscBytes = 768;
  static constexpr int kSmemBytes = 1024 + kRingBytes + kMiscBytes;
  static_assert(G >= 1 && G <= 16, "query heads per kv head");
  static_assert(kWarps * G * D * 4 <= kRingBytes, "the warps' O rows reuse the ring");
};

struct DecodeCtrl {
  uint64_t full[8];
  uint64_t empty[8];
  int abort_flag;
  int is_last;
};

// D(16x8, fp32) += A(16x16, bf16, row-major) * B(16x8, bf16, column-major).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}

// Byte offset of the 16-byte chunk holding columns [d0, d0 + 8) of `token` in a page that TMA
// wrote with 128-byte swizzle (64-column panels of 64 rows x 128 bytes).
__device__ __forceinline__ uint32_t page_chunk(int token, int d0) {
  return static_cast<uint32_t>((d0 >> 6) * (64 * 128) + token * 128 +
                               ((((d0 & 63) >> 3) ^ (token & 7)) << 4));
}

// GT: rows of the MMA tile that hold query heads (1, 2, 4, 8 or 16); the group's G = Hq / Hkv
// heads (G <= GT) fill the first G, and the rest are computed on zero queries and dropped.
template <int D, int GT>
__global__ void __launch_bounds__(160, 2)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  using C = DecodeCfg<D, GT>;
  constexpr int S = C::kStages;
  const int G = p.group;  // query heads of the group, 1 <= G <= GT
  const int split = static_cast<int>(blockIdx.x);
  const int g = static_cast<int>(blockIdx.y);
  const int b = static_cast<int>(blockIdx.z);
  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5;
  const int lane = tid & 31;

  int L = p.cu[b + 1] - p.cu[b];
  if (L < 0 || L > p.max_len) {
    if (split == 0 && tid == 0) report_status(p.status, -7);
    L = 0;
  }
  const int npages = (L + C::kPage - 1) / C::kPage;
  const int nsplit = (npages + p.chunk_pages - 1) / p.chunk_pages;
  uint16_t* o16 = static_cast<uint16_t*>(p.o);
  if (L == 0) {
    // Empty context: O = 0, LSE = -inf.
    if (split == 0) {
      for (int idx = tid; idx < G * D; idx += C::kThreads)
        o16[(static_cast<size_t>(b) * p.Hq + g * G + idx / D) * D + idx % D] = 0;
      if (tid < G) p.lse[static_cast<size_t>(b) * p.Hq + g * G + tid] = -INFINITY;
    }
    return;
  }
  if (split >= nsplit) return;
  const int pg0 = split * p.chunk_pages;
  const int n = imin(npages - pg0, p.chunk_pages);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* misc = ring + C::kRingBytes;
  DecodeCtrl* ctl = reinterpret_cast<DecodeCtrl*>(misc);
  float* red_m = reinterpret_cast<float*>(misc + C::kOffMax);  // [4 warps][16 rows]
  float* red_l = reinterpret_cast<float*>(misc + C::kOffSum);  // [4 warps][16 rows]

  if (tid == C::kConsumers) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], C::kWarps);
    }
    ctl->abort_flag = 0;
    ctl->is_last = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl wc{p.timeout_ns, p.status, &ctl->abort_flag};
  const WaitCtl wc_drain{p.timeout_ns, p.status, nullptr};

  if (warp == C::kWarps) {
    // ---------------------------------------------------------------- TMA producer
    const int* row = p.dense ? nullptr : p.table + static_cast<size_t>(b) * p.max_pages;
    const int lp = p.page_shift;  // log2(page_size)
    int issued = 0;
    if (p.dense || lp >= 6) {
      if (lane == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        // One box per stage: 64 rows of the dense cache, or the whole (P = 64) or one half
        // (P = 128) of a page. A stage whose table entry is outside the pool (never addressed;
        // the status word reports it) is loaded from the plane just past the pool, which TMA
        // fills with zeros, so the stage always receives its full bytes.
        for (int k = 0; k < n; ++k) {
          const int st = k % S;
          if (!mbar_wait(&ctl->empty[st], ((k / S) & 1) ^ 1, wc)) break;
          ++issued;
          uint8_t* dst = ring + st * C::kStageBytes;
          const int tok = (pg0 + k) * C::kPage;
          int plane, row0;
          if (p.dense) {
            // Rows past the cache's end read as zeros; rows past L_b are masked by the
            // consumers.
            plane = b * p.Hkv + g;
            row0 = tok;
          } else {
            const int phys = row[tok >> lp];
            row0 = tok & ((1 << lp) - 1);
            plane = phys * p.Hkv + g;
            if (phys < 0 || phys >= p.num_pages) {
              report_status(p.status, -5);
              plane = p.num_pages * p.Hkv;
            }
          }
          mbar_arrive_expect_tx(&ctl->full[st], C::kStageBytes);
#pragma unroll
          for (int pn = 0; pn < C::kPanels; ++pn) {
            tma_load_3d(dst + pn * C::kPanelBytes, &tm_k, &ctl->full[st], pn * 64, row0, plane);
            tma_load_3d(dst + C::kPageBytes + pn * C::kPanelBytes, &tm_v, &ctl->full[st],
                        pn * 64, row0, plane);
          }
        }
      }
    } else {
      // Pages of 16 or 32 tokens: stage k is 64 >> lp whole pages, and lane sb < 64 >> lp
      // owns page sb of every stage: it reads that page's table entry one stage ahead (so the
      // read overlaps the current stage) and issues its boxes, in parallel with the other
      // lanes. A page past the context, or whose table entry is outside the pool, is loaded
      // from the zero-filled plane past the pool.
      if (lane == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
      }
      const int nb = C::kPage >> lp;  // boxes per stage (4 or 2)
      auto plane_of = [&](int k) {
        const int tok = (pg0 + k) * C::kPage + (lane << lp);
        int pl = p.num_pages * p.Hkv;
        if (lane < nb && tok < L) {
          const int raw = __ldg(row + (tok >> lp));
          if (raw < 0 || raw >= p.num_pages)
            report_status(p.status, -5);
          else
            pl = raw * p.Hkv + g;
        }
        return pl;
      };
      int pl_next = n > 0 ? plane_of(0) : 0;
      for (int k = 0; k < n; ++k) {
        const int st = k % S;
        bool okw = true;
        if (lane == 0) okw = mbar_wait(&ctl->empty[st], ((k / S) & 1) ^ 1, wc);
        if (!__shfl_sync(0xffffffffu, okw, 0)) break;
        ++issued;
        uint8_t* dst = ring + st * C::kStageBytes;
        const int pl = pl_next;
        if (lane == 0) mbar_arrive_expect_tx(&ctl->full[st], C::kStageBytes);
        __syncwarp();
        if (lane < nb) {
#pragma unroll
          for (int pn = 0; pn < C::kPanels; ++pn) {
            tma_load_3d(dst + pn * C::kPanelBytes + (lane << lp) * 128, &tm_k, &ctl->full[st],
                        pn * 64, 0, pl);
            tma_load_3d(dst + C::kPageBytes + pn * C::kPanelBytes + (lane << lp) * 128, &tm_v,
                        &ctl->full[st], pn * 64, 0, pl);
          }
        }
        if (k + 1 < n) pl_next = plane_of(k + 1);
      }
    }
    if (lane == 0) {
      for (int k = imax(0, issued - S); k < issued; ++k)
        mbar_wait(&ctl->full[k % S], (k / S) & 1, wc_drain);
    }
    return;  // the producer takes no part in the consumer barriers below
  }

  // ------------------------------------------------------------------ consumers
  const int r = lane >> 2;  // tile rows r and r + 8 (heads), fragment columns 2q, 2q + 1
  const int q = lane & 3;
  const size_t head0 = static_cast<size_t>(b) * p.Hq + static_cast<size_t>(g) * G;
  // Q as the A operand: rows = heads (zero past G), k = head dimension.
  uint32_t qa[C::kKSteps][4];
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(p.q);
#pragma unroll
    for (int kk = 0; kk < C::kKSteps; ++kk) {
      const bool lo = r < G, hi = C::kHi && r + 8 < G;
      qa[kk][0] = lo ? q32[(head0 + r) * (D / 2) + kk * 8 + q] : 0u;
      qa[kk][2] = lo ? q32[(head0 + r) * (D / 2) + kk * 8 + 4 + q] : 0u;
      qa[kk][1] = hi ? q32[(head0 + r + 8) * (D / 2) + kk * 8 + q] : 0u;
      qa[kk][3] = hi ? q32[(head0 + r + 8) * (D / 2) + kk * 8 + 4 + q] : 0u;
    }
  }
  float o[C::kNTiles][4];
#pragma unroll
  for (int nt = 0; nt < C::kNTiles; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY;  // running max (log2 units), trails by < 8
  float l_lo = 0.f, l_hi = 0.f;              // this thread's share of the running sums
  const float c = p.scale_log2;
  const uint32_t ring_u32 = smem_u32(ring);
  const int tok_w = warp * 16;
  // ldmatrix row addresses: lane -> (matrix, row); see the fragment maps below.
  const int mrow = lane & 7, msel = lane >> 3;
  const int k_token = tok_w + 8 * (msel >> 1) + mrow;  // K: matrices (n-tile, k half)
  const int k_half = (msel & 1) * 8;
  const int v_token = tok_w + 8 * (msel & 1) + mrow;   // V: matrices (n-tile, token half)
  const int v_sub = (msel >> 1) * 8;
  bool ok = true;

  for (int k = 0; k < n; ++k) {
    const int st = k % S;
    ok = __all_sync(0xffffffffu, mbar_wait(&ctl->full[st], (k / S) & 1, wc));
    if (ok) {
      const uint32_t kp = ring_u32 + st * C::kStageBytes;
      const uint32_t vp = kp + C::kPageBytes;
      // S = Q K^T for this warp's 16 tokens: two 8-token n-tiles.
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < C::kKSteps; ++kk) {
        uint32_t kb[4];
        ldmatrix_x4(kb, kp + page_chunk(k_token, kk * 16 + k_half));
        mma_bf16_16816(s0, qa[kk], kb[0], kb[1]);
        mma_bf16_16816(s1, qa[kk], kb[2], kb[3]);
      }
      // Scale, mask keys past the context, update the running max of rows r (and r + 8).
      const int tok = (pg0 + k) * C::kPage + tok_w + 2 * q;
      float x[2][4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int te = tok + (e & 1);
        x[0][e] = (te < L) ? s0[e] * c : -INFINITY;
        x[1][e] = (te + 8 < L) ? s1[e] * c : -INFINITY;
      }
      float mx_lo = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
      float mx_hi = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      float a_lo = 1.f, a_hi = 1.f;
      // Conditional rescale: move the reference max only when it grows by more than 8.
      if (mx_lo > m_lo + 8.f) {
        a_lo = fast_exp2(m_lo - mx_lo);
        m_lo = mx_lo;
      }
      if (C::kHi && mx_hi > m_hi + 8.f) {
        a_hi = fast_exp2(m_hi - mx_hi);
        m_hi = mx_hi;
      }
      if (__any_sync(0xffffffffu, a_lo < 1.f || a_hi < 1.f)) {
#pragma unroll
        for (int nt = 0; nt < C::kNTiles; ++nt) {
          o[nt][0] *= a_lo;
          o[nt][1] *= a_lo;
          o[nt][2] *= a_hi;
          o[nt][3] *= a_hi;
        }
        l_lo *= a_lo;
        l_hi *= a_hi;
      }
      const float sub_lo = (m_lo == -INFINITY) ? 0.f : m_lo;
      const float sub_hi = (m_hi == -INFINITY) ? 0.f : m_hi;
      const bool live_lo = r < G, live_hi = C::kHi && r + 8 < G;
      float pr[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        pr[nt][0] = live_lo ? fast_exp2(x[nt][0] - sub_lo) : 0.f;
        pr[nt][1] = live_lo ? fast_exp2(x[nt][1] - sub_lo) : 0.f;
        pr[nt][2] = live_hi ? fast_exp2(x[nt][2] - sub_hi) : 0.f;
        pr[nt][3] = live_hi ? fast_exp2(x[nt][3] - sub_hi) : 0.f;
      }
      l_lo += (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
      l_hi += (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
      // The S accumulators of the two n-tiles are, as bf16 pairs, the A fragment of P.
      const uint32_t pa[4] = {pack_bf16x2(pr[0][0], pr[0][1]), pack_bf16x2(pr[0][2], pr[0][3]),
                              pack_bf16x2(pr[1][0], pr[1][1]), pack_bf16x2(pr[1][2], pr[1][3])};
      // O += P V over this warp's 16 tokens, two 8-column n-tiles per ldmatrix.
#pragma unroll
      for (int pair = 0; pair < C::kNTiles / 2; ++pair) {
        uint32_t vb[4];
        ldmatrix_x4_trans(vb, vp + page_chunk(v_token, pair * 16 + v_sub));
        mma_bf16_16816(o[2 * pair], pa, vb[0], vb[1]);
        mma_bf16_16816(o[2 * pair + 1], pa, vb[2], vb[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->empty[st]);
  }

  // ------------------------------------------------------------------ merge the four warps
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
  named_barrier_sync(1, C::kConsumers);  // every consumer is past its last ring read
  if (q == 0) {
    red_m[warp * 16 + r] = m_lo;
    red_l[warp * 16 + r] = l_lo;
    red_m[warp * 16 + r + 8] = m_hi;
    red_l[warp * 16 + r + 8] = l_hi;
  }
  named_barrier_sync(1, C::kConsumers);
  float M_lo = red_m[r], M_hi = red_m[r + 8];
#pragma unroll
  for (int w = 1; w < C::kWarps; ++w) {
    M_lo = fmaxf(M_lo, red_m[w * 16 + r]);
    M_hi = fmaxf(M_hi, red_m[w * 16 + r + 8]);
  }
  {
    const float f_lo = (m_lo == -INFINITY) ? 0.f : fast_exp2(m_lo - M_lo);
    const float f_hi = (m_hi == -INFINITY) ? 0.f : fast_exp2(m_hi - M_hi);
#pragma unroll
    for (int nt = 0; nt < C::kNTiles; ++nt) {
      o[nt][0] *= f_lo;
      o[nt][1] *= f_lo;
      o[nt][2] *= f_hi;
      o[nt][3] *= f_hi;
    }
  }
  // Each warp's rescaled rows of the group's heads go to the idle ring, [warp][G][D] fp32.
  // After one barrier every consumer thread sums four columns of one head over the warps in a
  // fixed order, (w0 + w2) + (w1 + w3), and writes them out: the result is bit-reproducible,
  // and the partials leave as coalesced 16-byte stores from all four warps.
  float* buf = reinterpret_cast<float*>(ring);
#pragma unroll
  for (int nt = 0; nt < C::kNTiles; ++nt) {
    if (r < G)
      *reinterpret_cast<float2*>(buf + (warp * G + r) * D + nt * 8 + 2 * q) =
          make_float2(o[nt][0], o[nt][1]);
    if (C::kHi && r + 8 < G)
      *reinterpret_cast<float2*>(buf + (warp * G + r + 8) * D + nt * 8 + 2 * q) =
          make_float2(o[nt][2], o[nt][3]);
  }
  named_barrier_sync(1, C::kConsumers);

  const size_t bg = static_cast<size_t>(b) * p.Hkv + g;
  const bool single = nsplit == 1;
  constexpr int kQuads = D / 4;  // four-column groups of one head's row
  for (int idx = tid; idx < G * kQuads; idx += C::kConsumers) {
    const int hh = idx / kQuads, d0 = (idx % kQuads) * 4;
    float4 w[C::kWarps];
#pragma unroll
    for (int ww = 0; ww < C::kWarps; ++ww)
      w[ww] = *reinterpret_cast<const float4*>(buf + (ww * G + hh) * D + d0);
    const float4 s = make_float4((w[0].x + w[2].x) + (w[1].x + w[3].x),
                                 (w[0].y + w[2].y) + (w[1].y + w[3].y),
                                 (w[0].z + w[2].z) + (w[1].z + w[3].z),
                                 (w[0].w + w[2].w) + (w[1].w + w[3].w));
    // The head's max and sum over the warps (the same M that rescaled each warp's O above).
    float Mr = red_m[hh];
#pragma unroll
    for (int ww = 1; ww < C::kWarps; ++ww) Mr = fmaxf(Mr, red_m[ww * 16 + hh]);
    float Lr = 0.f;
#pragma unroll
    for (int ww = 0; ww < C::kWarps; ++ww) {
      const float mw = red_m[ww * 16 + hh];
      if (mw != -INFINITY) Lr += red_l[ww * 16 + hh] * fast_exp2(mw - Mr);
    }
    const size_t orow = head0 + hh;
    if (single) {
      const float inv = Lr > 0.f ? 1.f / Lr : 0.f;
      *reinterpret_cast<uint2*>(o16 + orow * D + d0) =
          make_uint2(pack_bf16x2(s.x * inv, s.y * inv), pack_bf16x2(s.z * inv, s.w * inv));
      if (d0 == 0)
        p.lse[orow] = Lr > 0.f ? (Mr + log2f(Lr)) * 0.69314718055994530942f : -INFINITY;
    } else {
      const size_t base = (bg * p.max_splits + split) * G + hh;
      *reinterpret_cast<float4*>(p.part_o + base * D + d0) = s;
      if (d0 == 0) {
        p.part_ml[2 * base] = Mr;
        p.part_ml[2 * base + 1] = Lr;
      }
    }
  }
  if (single) return;

  // Ticket: once every consumer has written its partials, thread 0 publishes them (a fence,
  // then the counter) and the split that draws the last ticket merges.
  named_barrier_sync(1, C::kConsumers);
  if (tid == 0) {
    __threadfence();
    const int ticket = atomicAdd(&p.counters[bg], 1);
    __threadfence();
    ctl->is_last = ticket == nsplit - 1;
  }
  named_barrier_sync(1, C::kConsumers);
  if (!ctl->is_last) return;
  __threadfence();
  // Last split of (b, g): merge the splits in split order,
  //   M = max_c m_c,  L = sum_c l_c 2^(m_c - M),  O = sum_c O_c 2^(m_c - M) / L,
  // summing in split order as a plain loop over the splits would. Each thread takes four
  // columns of one head and issues the loads of a whole batch of splits before it uses any,
  // so the merge costs a few L2 round trips instead of one or more per split.
  constexpr int kBatch = 16;
  const size_t base_bg = bg * p.max_splits * G;  // (b, g)'s first partial row
  for (int idx = tid; idx < G * kQuads; idx += C::kConsumers) {
    const int hh = idx / kQuads, d0 = (idx % kQuads) * 4;
    const float* ml = p.part_ml + 2 * (base_bg + hh);     // split c at + 2 c G
    const float* po = p.part_o + (base_bg + hh) * D + d0;  // split c at + c G D
    // M first, in its own pass, unless one batch holds every split.
    float M = -INFINITY;
    for (int c0 = 0; nsplit > kBatch && c0 < nsplit; c0 += kBatch) {
      float mv[kBatch];
#pragma unroll
      for (int t = 0; t < kBatch; ++t)
        mv[t] = c0 + t < nsplit ? __ldcg(ml + 2 * static_cast<size_t>(c0 + t) * G) : -INFINITY;
#pragma unroll
      for (int t = 0; t < kBatch; ++t) M = fmaxf(M, mv[t]);
    }
    float Ls = 0.f;
    float4 Os = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < nsplit; c0 += kBatch) {
      float2 mlv[kBatch];
      float4 ov[kBatch];
#pragma unroll
      for (int t = 0; t < kBatch; ++t) {
        const size_t c = static_cast<size_t>(imin(c0 + t, nsplit - 1));
        mlv[t] = __ldcg(reinterpret_cast<const float2*>(ml + 2 * c * G));
        ov[t] = __ldcg(reinterpret_cast<const float4*>(po + c * G * D));
      }
      if (nsplit <= kBatch) {
#pragma unroll
        for (int t = 0; t < kBatch; ++t)
          if (t < nsplit) M = fmaxf(M, mlv[t].x);
      }
#pragma unroll
      for (int t = 0; t < kBatch; ++t) {
        if (c0 + t < nsplit) {
          const float wt = exp2f(mlv[t].x - M);
          Ls += mlv[t].y * wt;
          Os.x += ov[t].x * wt;
          Os.y += ov[t].y * wt;
          Os.z += ov[t].z * wt;
          Os.w += ov[t].w * wt;
        }
      }
    }
    const size_t orow = head0 + hh;
    *reinterpret_cast<uint2*>(o16 + orow * D + d0) =
        make_uint2(pack_bf16x2(Os.x / Ls, Os.y / Ls), pack_bf16x2(Os.z / Ls, Os.w / Ls));
    if (d0 == 0) p.lse[orow] = (M + log2f(Ls)) * 0.69314718055994530942f;
  }
  if (tid == 0) p.counters[bg] = 0;
}

}  // namespace ta
