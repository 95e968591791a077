// decode.cuh — paged-KV decode (one query token per sequence) with split-KV partials and a
// fused log-sum-exp-weighted combine.
//
// The KV cache is a pool of pages [num_pages, Hkv, 64, D]; sequence b's logical page p lives
// at physical page block_table[b][p] ("Optimizing Triton Kernels for Custom Attention
// Patterns on H100", Pattern C). Instead of first gathering pages into a dense buffer, the
// producer warp issues one TMA box per (page, kv-head, 64 columns) straight from the pool into
// a shared-memory ring, so every K/V byte crosses HBM once.
//
// Grid (split, kv head g, sequence b): a CTA handles `chunk_pages` pages of one (b, g) for
// all G = Hq/Hkv query heads of the group. Decode reads each K/V byte once and does ~4 FLOP
// per byte, so it is HBM-bound and runs on the CUDA cores (mixed bf16 x bf16 + fp32 FMA), not
// the tensor cores. Per page: scores for (token, head) pairs, a per-head running max and sum
// (the online softmax of "Flash MSA Attention Kernel Implementation Tutorial", "Understanding
// Flash MSA Core Mechanics", in exp2 form), then P.V into per-thread fp32 accumulators.
//
// Combine: each split writes its unnormalised O, max m and sum l (log2 units) to the
// workspace; the last split to finish (atomic ticket per (b, g)) merges them in split order:
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
  const int* table;      // [B, max_pages]
  void* o;               // bf16 [B, Hq, 1, D]
  float* lse;            // [B, Hq]
  float* part_o;         // [B*Hkv, max_splits, G, D]
  float* part_ml;        // [B*Hkv, max_splits, G, 2]
  int* counters;         // [B*Hkv], zero before the launch
  int B, Hq, Hkv, max_pages, num_pages, max_splits, chunk_pages;
  float scale_log2;
  int* status;
  unsigned long long timeout_ns;
};

template <int D, int G>
struct DecodeCfg {
  static constexpr int kPage = 64;
  static constexpr int kConsumers = 256;
  static constexpr int kThreads = kConsumers + 32;
  static constexpr int kPanels = D / 64;
  static constexpr int kPanelBytes = kPage * 128;           // 64 tokens x 64 columns
  static constexpr int kPageBytes = kPage * D * 2;          // one (page, kv-head) of K or V
  static constexpr int kStageBytes = 2 * kPageBytes;        // K and V
  static constexpr int kStages = (96 * 1024) / kStageBytes; // 3 (D=128), 6 (D=64)
  static constexpr int kGP = G < 2 ? 2 : G;                 // heads per p row, padded to pairs
  static constexpr int kPairs = kPage * G;
  static constexpr int kPairsPerThread = (kPairs + kConsumers - 1) / kConsumers;
  static constexpr int kDPairs = D / 2;
  static constexpr int kTokenGroups = kConsumers / kDPairs;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kQPitch = D * 2 + 16;  // padded so the G query rows hit distinct banks
  static constexpr int kMiscBytes = 2048 + G * kQPitch;
  static constexpr int kSmemBytes = 1024 + kRingBytes + kMiscBytes;  // ring + ctrl/p/red/q
};

struct DecodeCtrl {
  uint64_t full[8];
  uint64_t empty[8];
  int abort_flag;
  int is_last;
};

// c + a.lo * b.lo + a.hi * b.hi (bf16 pairs, exact products, fp32 accumulation).
__device__ __forceinline__ float dot2_bf16(uint32_t a, uint32_t b, float c) {
  asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
      " fma.rn.f32.bf16 %0, al, bl, %0;\n fma.rn.f32.bf16 %0, ah, bh, %0;\n}"
      : "+f"(c)
      : "r"(a), "r"(b));
  return c;
}

// (c00, c01, c10, c11) += (p.lo * v.lo, p.lo * v.hi, p.hi * v.lo, p.hi * v.hi).
__device__ __forceinline__ void outer2_bf16(uint32_t p, uint32_t v, float& c00, float& c01,
                                            float& c10, float& c11) {
  asm("{\n .reg .b16 pl, ph, vl, vh;\n mov.b32 {pl, ph}, %4;\n mov.b32 {vl, vh}, %5;\n"
      " fma.rn.f32.bf16 %0, pl, vl, %0;\n fma.rn.f32.bf16 %1, pl, vh, %1;\n"
      " fma.rn.f32.bf16 %2, ph, vl, %2;\n fma.rn.f32.bf16 %3, ph, vh, %3;\n}"
      : "+f"(c00), "+f"(c01), "+f"(c10), "+f"(c11)
      : "r"(p), "r"(v));
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
  return static_cast<uint16_t>(pack_bf16x2(x, 0.f) & 0xFFFFu);
}

template <int D, int G>
__global__ void __launch_bounds__(288, 2)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  using C = DecodeCfg<D, G>;
  constexpr int S = C::kStages;
  const int split = static_cast<int>(blockIdx.x);
  const int g = static_cast<int>(blockIdx.y);
  const int b = static_cast<int>(blockIdx.z);
  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5;
  const int lane = tid & 31;

  int L = p.cu[b + 1] - p.cu[b];
  if (L < 0 || L > p.max_pages * C::kPage) {
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
  uint16_t* p_buf = reinterpret_cast<uint16_t*>(misc + 256);              // [64][kGP]
  float* red_max = reinterpret_cast<float*>(misc + 256 + 64 * 8 * 2);     // [G][8]
  float* red_l = red_max + 8 * 8;                                         // [G][8]
  uint8_t* q_s = misc + 2048;                                             // [G][kQPitch]

  if (tid == C::kConsumers) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 8);
    }
    ctl->abort_flag = 0;
    ctl->is_last = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl wc{p.timeout_ns, p.status, &ctl->abort_flag};
  const WaitCtl wc_drain{p.timeout_ns, p.status, nullptr};

  if (warp == 8) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      const int* row = p.table + static_cast<size_t>(b) * p.max_pages + pg0;
      int issued = 0;
      for (int k = 0; k < n; ++k) {
        const int st = k % S;
        if (!mbar_wait(&ctl->empty[st], ((k / S) & 1) ^ 1, wc)) break;
        const int phys = row[k];
        ++issued;
        if (phys < 0 || phys >= p.num_pages) {
          // Out-of-pool entry: never address it. The stage completes without data and the
          // status word tells the caller the result is invalid.
          report_status(p.status, -5);
          mbar_arrive(&ctl->full[st]);
          continue;
        }
        mbar_arrive_expect_tx(&ctl->full[st], C::kStageBytes);
        uint8_t* dst = ring + st * C::kStageBytes;
        const int plane = phys * p.Hkv + g;
#pragma unroll
        for (int pn = 0; pn < C::kPanels; ++pn) {
          tma_load_3d(dst + pn * C::kPanelBytes, &tm_k, &ctl->full[st], pn * 64, 0, plane);
          tma_load_3d(dst + C::kPageBytes + pn * C::kPanelBytes, &tm_v, &ctl->full[st], pn * 64,
                      0, plane);
        }
      }
      for (int k = imax(0, issued - S); k < issued; ++k)
        mbar_wait(&ctl->full[k % S], (k / S) & 1, wc_drain);
    }
    return;  // the producer takes no part in the consumer barriers below
  }

  // ------------------------------------------------------------------ consumers
  const int h_qk = tid % G;  // head of this thread's score pairs (256 % G == 0)
  const bool qk_live = tid < C::kPairs;
  for (int idx = tid; idx < G * (D / 8); idx += C::kConsumers) {
    const int hh = idx / (D / 8), ch = idx % (D / 8);
    *reinterpret_cast<uint4*>(q_s + hh * C::kQPitch + ch * 16) =
        p.q[(static_cast<size_t>(b) * p.Hq + g * G + hh) * (D / 8) + ch];
  }
  named_barrier_sync(1, C::kConsumers);
  const uint8_t* q_row = q_s + h_qk * C::kQPitch;
  const int dp = tid % C::kDPairs;
  const int tg = tid / C::kDPairs;
  const int v_off = (dp / 32) * C::kPanelBytes + (dp % 4) * 4;  // panel + bytes inside chunk
  const int v_chunk = (dp % 32) / 4;
  float acc[G][2];
  float m_run[G];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    acc[hh][0] = acc[hh][1] = 0.f;
    m_run[hh] = -INFINITY;
  }
  float l_part = 0.f;
  const float c = p.scale_log2;
  bool ok = true;

  for (int k = 0; k < n; ++k) {
    const int st = k % S;
    ok = __all_sync(0xffffffffu, mbar_wait(&ctl->full[st], (k / S) & 1, wc));
    // Every consumer warp must take the same number of named barriers: a warp that gave up
    // still walks the page loop, without touching the ring.
    const uint8_t* kp = ring + st * C::kStageBytes;
    const uint8_t* vp = kp + C::kPageBytes;
    const int tok0 = (pg0 + k) * C::kPage;

    float sc[C::kPairsPerThread];
    float mloc = -INFINITY;
#pragma unroll
    for (int u = 0; u < C::kPairsPerThread; ++u) {
      const int idx = tid + u * C::kConsumers;
      const int t = idx / G;
      float s = -INFINITY;
      if (idx < C::kPairs && ok && tok0 + t < L) {
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int pn = 0; pn < C::kPanels; ++pn) {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint4 kv = *reinterpret_cast<const uint4*>(
                kp + pn * C::kPanelBytes + t * 128 + ((ch ^ (t & 7)) << 4));
            const uint4 qv = *reinterpret_cast<const uint4*>(q_row + pn * 128 + ch * 16);
            a0 = dot2_bf16(qv.x, kv.x, a0);
            a1 = dot2_bf16(qv.y, kv.y, a1);
            a2 = dot2_bf16(qv.z, kv.z, a2);
            a3 = dot2_bf16(qv.w, kv.w, a3);
          }
        }
        s = ((a0 + a1) + (a2 + a3)) * c;
      }
      sc[u] = s;
      mloc = fmaxf(mloc, s);
    }
#pragma unroll
    for (int off = G; off < 32; off <<= 1)
      mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, off));
    if (lane < G) red_max[lane * 8 + warp] = mloc;
    named_barrier_sync(1, C::kConsumers);

    float alpha[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const float4 x = *reinterpret_cast<const float4*>(red_max + hh * 8);
      const float4 y = *reinterpret_cast<const float4*>(red_max + hh * 8 + 4);
      const float pm = fmaxf(fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)),
                             fmaxf(fmaxf(y.x, y.y), fmaxf(y.z, y.w)));
      const float mn = fmaxf(m_run[hh], pm);
      alpha[hh] = (mn == -INFINITY) ? 1.f : fast_exp2(m_run[hh] - mn);
      m_run[hh] = mn;
    }
    {
      float m_own = m_run[0], a_own = alpha[0];
#pragma unroll
      for (int hh = 1; hh < G; ++hh) {
        m_own = (hh == h_qk) ? m_run[hh] : m_own;
        a_own = (hh == h_qk) ? alpha[hh] : a_own;
      }
      const float msub = (m_own == -INFINITY) ? 0.f : m_own;
      l_part *= a_own;
#pragma unroll
      for (int u = 0; u < C::kPairsPerThread; ++u) {
        const int idx = tid + u * C::kConsumers;
        if (idx < C::kPairs) {
          const float pv = fast_exp2(sc[u] - msub);
          l_part += pv;
          p_buf[(idx / G) * C::kGP + h_qk] = bf16_bits(pv);
        }
      }
      if (G == 1 && qk_live) p_buf[(tid / G) * C::kGP + 1] = 0;
    }
    named_barrier_sync(1, C::kConsumers);

#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      acc[hh][0] *= alpha[hh];
      acc[hh][1] *= alpha[hh];
    }
    if (ok) {
#pragma unroll 4
      for (int t = tg; t < C::kPage; t += C::kTokenGroups) {
        const uint32_t vw =
            *reinterpret_cast<const uint32_t*>(vp + v_off + t * 128 + ((v_chunk ^ (t & 7)) << 4));
        const uint32_t* prow = reinterpret_cast<const uint32_t*>(p_buf + t * C::kGP);
#pragma unroll
        for (int w = 0; w < C::kGP / 2; ++w) {
          float dummy0 = 0.f, dummy1 = 0.f;
          float& c10 = (2 * w + 1 < G) ? acc[(2 * w + 1) % G][0] : dummy0;
          float& c11 = (2 * w + 1 < G) ? acc[(2 * w + 1) % G][1] : dummy1;
          outer2_bf16(prow[w], vw, acc[2 * w][0], acc[2 * w][1], c10, c11);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->empty[st]);
  }

  // ------------------------------------------------------------------ split result
  float* red_acc = reinterpret_cast<float*>(ring);  // [kTokenGroups][G][D]; ring is idle now
#pragma unroll
  for (int off = G; off < 32; off <<= 1) l_part += __shfl_xor_sync(0xffffffffu, l_part, off);
  named_barrier_sync(1, C::kConsumers);  // every consumer is past its last ring read
  if (lane < G) red_l[lane * 8 + warp] = l_part;
#pragma unroll
  for (int hh = 0; hh < G; ++hh)
    *reinterpret_cast<float2*>(red_acc + (tg * G + hh) * D + 2 * dp) =
        make_float2(acc[hh][0], acc[hh][1]);
  named_barrier_sync(1, C::kConsumers);

  const size_t bg = static_cast<size_t>(b) * p.Hkv + g;
  const bool single = nsplit == 1;
  for (int idx = tid; idx < G * D; idx += C::kConsumers) {
    const int hh = idx / D, d = idx % D;
    float ou = 0.f;
#pragma unroll
    for (int q = 0; q < C::kTokenGroups; ++q) ou += red_acc[(q * G + hh) * D + d];
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) l += red_l[hh * 8 + w];
    float mrun = m_run[0];
#pragma unroll
    for (int h2 = 1; h2 < G; ++h2) mrun = (h2 == hh) ? m_run[h2] : mrun;
    if (single) {
      o16[(static_cast<size_t>(b) * p.Hq + g * G + hh) * D + d] = bf16_bits(ou / l);
      if (d == 0)
        p.lse[static_cast<size_t>(b) * p.Hq + g * G + hh] =
            (mrun + log2f(l)) * 0.69314718055994530942f;
    } else {
      const size_t base = (bg * p.max_splits + split) * G + hh;
      p.part_o[base * D + d] = ou;
      if (d == 0) {
        p.part_ml[2 * base] = mrun;
        p.part_ml[2 * base + 1] = l;
      }
    }
  }
  if (single) return;

  __threadfence();
  named_barrier_sync(1, C::kConsumers);
  if (tid == 0) {
    const int ticket = atomicAdd(&p.counters[bg], 1);
    ctl->is_last = ticket == nsplit - 1;
  }
  named_barrier_sync(1, C::kConsumers);
  if (!ctl->is_last) return;
  __threadfence();
  for (int idx = tid; idx < G * D; idx += C::kConsumers) {
    const int hh = idx / D, d = idx % D;
    const size_t base0 = (bg * p.max_splits) * G + hh;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, __ldcg(p.part_ml + 2 * (base0 + s * G)));
    float Ls = 0.f, Os = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const size_t bs = base0 + static_cast<size_t>(s) * G;
      const float w = exp2f(__ldcg(p.part_ml + 2 * bs) - M);
      Ls += __ldcg(p.part_ml + 2 * bs + 1) * w;
      Os += __ldcg(p.part_o + bs * D + d) * w;
    }
    o16[(static_cast<size_t>(b) * p.Hq + g * G + hh) * D + d] = bf16_bits(Os / Ls);
    if (d == 0)
      p.lse[static_cast<size_t>(b) * p.Hq + g * G + hh] =
          (M + log2f(Ls)) * 0.69314718055994530942f;
  }
  if (tid == 0) p.counters[bg] = 0;
}

}  // namespace ta
