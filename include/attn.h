/*
 * attn.h — C ABI of the GB300 (sm_103a) tiled attention forward library (libtiled_attn.so).
 *
 * The library computes O = softmax(scale * Q K^T + mask) V without materialising the score
 * matrix: each query tile keeps a running row max m and row sum l and rescales its
 * accumulator by exp(m - m_new) when the max grows ("Flash MSA Attention Kernel
 * Implementation Tutorial", section "Understanding Flash MSA Core Mechanics"). It also returns
 * the natural-log log-sum-exp of the scaled, masked scores of every query row.
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller. The library never allocates,
 *    frees or retains them beyond the call. Elements are bf16 (raw 16-bit patterns) unless
 *    stated; LSE is fp32. Every tensor is contiguous and 16-byte aligned.
 *  - Calls are asynchronous on the given stream (a cudaStream_t; NULL = legacy default stream)
 *    and never synchronise the host, except attn_get_status().
 *  - Errors are returned, never thrown or printed: 0 on success, a negative ATTN_ERR_* code
 *    otherwise, with a message for attn_last_error(). An invalid call launches nothing.
 *  - Conditions only the device can see (a bad cu_seqlens entry, a block-table entry outside
 *    the pool, a pipeline wait that ran past its time limit) are written to a device status
 *    word that attn_get_status() reads and clears.
 *  - CUDA graphs: the first call on a device sets one-time kernel attributes and caches device
 *    addresses. From then on every compute entry point only enqueues memsets and kernel
 *    launches on the given stream, so it may be captured into a CUDA graph and replayed with
 *    new inputs written in place (attn_get_status(), which synchronises, may not be captured).
 */
#ifndef TILED_ATTN_H
#define TILED_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Which keys a query row i may attend to (j indexes keys):
 *  NONE          every key j < N.
 *  CAUSAL        j <= i.
 *  SLIDING       i - window < j <= i (causal window of `window` keys, the query included;
 *                "Optimizing Triton Kernels for Custom Attention Patterns on H100",
 *                Pattern B, read as a causal window).
 *  DOCUMENT      cu_seqlens[s] <= j <= i where segment s holds i (no attention across
 *                segments, causal inside one; same page, Pattern A).
 *  PAGED_DECODE  one query per sequence sees its whole context, read through a block table
 *                (same page, Pattern C).
 *  DECODE        one query per sequence sees its whole context, read from a dense
 *                per-sequence cache: the second stage of the two-stage paged path of the
 *                same page, Pattern C (an ordinary attention kernel run on pages that
 *                attn_gather_pages has gathered).
 *  SLIDING_BIDIR i - window <= j <= i + window: Pattern B's neighbourhood of W keys on
 *                both sides taken literally (window >= 0 keys on each side of the query).
 *  DOCUMENT_BIDIR cu_seqlens[s] <= j < cu_seqlens[s+1] where segment s holds i: Pattern A's
 *                kernel as printed (every key of the query's own segment, none outside it).
 *  PREFIX_LM     j <= i or j < window: a prefix of `window` tokens that see each other in
 *                both directions, then causal rows (the prefix-LM mask the same page lists
 *                among masks whose structure a kernel should exploit). */
enum attn_mask_kind {
    ATTN_MASK_NONE = 0,
    ATTN_MASK_CAUSAL = 1,
    ATTN_MASK_SLIDING = 2,
    ATTN_MASK_DOCUMENT = 3,
    ATTN_MASK_PAGED_DECODE = 4,
    ATTN_MASK_DECODE = 5,
    ATTN_MASK_SLIDING_BIDIR = 6,
    ATTN_MASK_DOCUMENT_BIDIR = 7,
    ATTN_MASK_PREFIX_LM = 8,
    /* Chunked prefill over a paged cache: only attn_fwd_paged_prefill takes it (attn_fwd
     * returns ATTN_ERR_INVALID); attn_plan_units plans it. */
    ATTN_MASK_PAGED_PREFILL = 9
};

enum attn_status {
    ATTN_OK = 0,
    ATTN_ERR_INVALID = -1,     /* an argument breaks the contract below */
    ATTN_ERR_UNSUPPORTED = -2, /* valid attention, but outside what the kernels implement */
    ATTN_ERR_CUDA = -3,        /* a CUDA runtime / driver call failed */
    ATTN_ERR_TIMEOUT = -4,     /* (status word) a pipeline wait gave up after its time limit */
    ATTN_ERR_BOUNDS = -5,      /* (status word) block-table entry outside [0, num_pages) */
    ATTN_ERR_WORKSPACE = -6,   /* workspace missing or smaller than attn_workspace_bytes() */
    ATTN_ERR_SEQLENS = -7      /* (status word) cu_seqlens not monotone / not ending at N */
};

/*
 * attn_fwd — fused tiled attention forward pass.
 *
 * The document kinds are DOCUMENT and DOCUMENT_BIDIR; the dense kinds are NONE, CAUSAL,
 * SLIDING, SLIDING_BIDIR and PREFIX_LM.
 * q, o      bf16. Dense kinds [B,Hq,N,d]; document kinds [1,Hq,N,d] with N = total packed
 *           tokens; PAGED_DECODE and DECODE [B,Hq,1,d].
 * k, v      bf16. Dense kinds [B,Hkv,N,d]; document kinds [1,Hkv,N,d]; PAGED_DECODE page pools
 *           [num_pages,Hkv,page_size,d] (one (page, kv-head) block is contiguous); DECODE
 *           dense caches [B,Hkv,N,d] (rows past a sequence's length are never read into the
 *           result).
 * lse       fp32, ln sum_j exp(scale * q_i . k_j) over the visible keys. [B,Hq,N]; document
 *           kinds [1,Hq,N]; PAGED_DECODE and DECODE [B,Hq].
 * B         batch (dense), number of segments (document kinds) or sequences (decode kinds).
 * Hq, Hkv   query / key-value heads; Hq % Hkv == 0; query head h reads kv head h/(Hq/Hkv).
 *           PAGED_DECODE and DECODE take at most 16 query heads per kv head (else
 *           ATTN_ERR_UNSUPPORTED): the group's heads are the rows of one 16-row MMA tile.
 * N         keys per sequence (dense), packed tokens (document kinds), the longest context
 *           (PAGED_DECODE: block_table has ceil(N/page_size) columns), or the rows of each
 *           dense cache (DECODE).
 * d         head dimension; 64 or 128 (else ATTN_ERR_UNSUPPORTED).
 * scale     multiplies q.k before the softmax (callers usually pass 1/sqrt(d)).
 * mask_kind enum attn_mask_kind.
 * window    SLIDING: number of keys visible to a query (>= 1). SLIDING_BIDIR: keys visible
 *           on each side of the query (>= 0). PREFIX_LM: prefix length (>= 0; 0 and 1 give
 *           the causal mask, >= N no mask). Ignored otherwise. Out of range:
 *           ATTN_ERR_INVALID.
 * cu_seqlens int32 device array [B+1], cu[0] = 0, nondecreasing. Document kinds: segment starts,
 *           cu[B] = N. PAGED_DECODE and DECODE: cumulative context lengths
 *           (L_b = cu[b+1] - cu[b], 0 <= L_b <= N). Checked on the device (status
 *           ATTN_ERR_SEQLENS). Unused otherwise.
 * block_table int32 device array [B, ceil(N/page_size)]: physical page of logical page p of
 *           sequence b; entries past a sequence's last page are ignored (-1 by convention).
 *           PAGED_DECODE only.
 * page_size tokens per page; PAGED_DECODE supports 16, 32, 64 and 128.
 * num_pages pages in the k / v pools (PAGED_DECODE; bounds-checked on the device).
 *           block_table, page_size and num_pages are ignored for DECODE.
 * workspace device scratch of at least attn_workspace_bytes(...) bytes (may be NULL when that
 *           is 0). Its contents need not be initialised; concurrent calls need separate ones.
 * stream    cudaStream_t to launch on.
 * A sequence with L_b = 0 gets O = 0 and LSE = -inf.
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
             int Hkv, int N, int d, float scale, int mask_kind, int window,
             const int32_t *cu_seqlens, const int32_t *block_table, int page_size,
             int num_pages, void *workspace, size_t workspace_bytes, void *stream);

/*
 * attn_fwd_paged_prefill — chunked prefill (or prefix reuse) over a paged KV cache.
 *
 * Sequence b holds a context of Lk_b = seqlens_k[b] tokens in a page pool; its last Lq_b
 * tokens are the new query chunk, whose own keys and values are already in the pool. Chunk row
 * t sits at position Lk_b - Lq_b + t and attends to the context keys j <= Lk_b - Lq_b + t:
 * causal attention aligned to the end of the context. This is the block-table indirection of
 * "Optimizing Triton Kernels for Custom Attention Patterns on H100", Pattern C (whose use
 * cases include prefix caching), with a query block longer than one token. Keys are gathered
 * page by page through the block table inside the kernel; no dense copy is made.
 *
 * q, o      bf16 [1, Hq, total_q, d]: the chunks packed back to back.
 * lse       fp32 [1, Hq, total_q] (natural log, as for attn_fwd).
 * k, v      bf16 page pools [num_pages, Hkv, page_size, d].
 * cu_seqlens_q int32 device array [B+1]: chunk starts, cu[0] = 0, nondecreasing,
 *           cu[B] = total_q.
 * seqlens_k int32 device array [B]: context lengths, Lq_b <= Lk_b <= max_pages * page_size.
 *           Checked on the device with cu_seqlens_q (status ATTN_ERR_SEQLENS, nothing computed).
 * block_table int32 device array [B, max_pages]: physical page of logical page p of sequence
 *           b. Only entries p < ceil(Lk_b / page_size) are read; an entry outside
 *           [0, num_pages) is never dereferenced (status ATTN_ERR_BOUNDS, that page reads as
 *           zeros).
 * page_size 16, 32, 64 or 128 (else ATTN_ERR_UNSUPPORTED).
 * d         64 or 128. Hq % Hkv == 0; query head h reads kv head h / (Hq / Hkv).
 * Pool slots of a sequence's last page past Lk_b must hold finite values (their
 * probabilities are exactly zero, and zero times a non-finite value is not zero).
 * No workspace; asynchronous on `stream`; the caller owns every buffer.
 */
int attn_fwd_paged_prefill(const void *q, const void *k, const void *v, void *o, float *lse,
                           int B, int Hq, int Hkv, int total_q, int d, float scale,
                           const int32_t *cu_seqlens_q, const int32_t *seqlens_k,
                           const int32_t *block_table, int max_pages, int page_size,
                           int num_pages, void *stream);

/*
 * attn_quantize_fp8 — FP8 E4M3 block quantization of a bf16 tensor x [planes, N, d].
 *
 * The block quantization of "FlashAttention-3: Warp Specialization and the 75% FLOPS Barrier on
 * Hopper" ("FP8 Block Quantization"), with one scale per 128-row tile of a plane (the page's
 * prose says per tile): for rows [128t, min(128t + 128, N)) of plane p,
 *   scales[p][t] = amax / 448                      (fp32, IEEE division; 0 if amax is 0)
 *   x8[p][r][c]  = E4M3(x[p][r][c] / scales[p][t]) (IEEE fp32 division, round to nearest even,
 *                                                   saturating; 0 when the scale is 0)
 * x     bf16 [planes, N, d], 16-byte aligned (device).
 * x8    E4M3 bytes [planes, N, d], 16-byte aligned (device, written).
 * scales fp32 [planes, ceil(N/128)] (device, written).
 * d 64 or 128; planes <= 65535. Asynchronous on `stream`.
 */
int attn_quantize_fp8(const void *x, void *x8, float *scales, int planes, int N, int d,
                      void *stream);

/*
 * attn_fwd_fp8 — attention forward with E4M3 Q and K (the FP8 path of the same page).
 *
 * Same result definition as attn_fwd, with Q and K replaced by their dequantized blocks:
 * q[b,h,i,:] = q8[b,h,i,:] * q_scales[b*Hq + h][i / 128] and likewise for k. S = Q K^T runs on
 * the FP8 tensor cores (fp32 accumulation); the two tile scales join the softmax's per-tile
 * scale, so the rescale after the matmul costs nothing per element. V, P and O stay bf16.
 * q8        E4M3 [B, Hq, N, 128]; k8 E4M3 [B, Hkv, N, 128]; v bf16 [B, Hkv, N, 128].
 * o, lse    as attn_fwd (bf16 [B, Hq, N, 128], fp32 [B, Hq, N]).
 * q_scales  fp32 [B*Hq, ceil(N/128)]; k_scales fp32 [B*Hkv, ceil(N/128)] (attn_quantize_fp8's
 *           layout). Finite and >= 0 (a 0 scale means an all-zero tile).
 * d         128 only (else ATTN_ERR_UNSUPPORTED).
 * mask_kind NONE, CAUSAL, SLIDING, SLIDING_BIDIR or PREFIX_LM (the document, paged and decode
 *           kinds return ATTN_ERR_UNSUPPORTED); window as for attn_fwd.
 * No workspace; asynchronous on `stream`.
 */
int attn_fwd_fp8(const void *q8, const void *k8, const void *v, void *o, float *lse,
                 const float *q_scales, const float *k_scales, int B, int Hq, int Hkv, int N,
                 int d, float scale, int mask_kind, int window, void *stream);

/* Bytes of workspace attn_fwd needs for these arguments (0 for the prefill kinds; DECODE
 * ignores page_size). */
size_t attn_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int mask_kind, int page_size);

/*
 * attn_gather_pages — copy paged K or V into a dense per-sequence layout.
 * pool [num_pages,Hkv,page_size,d] bf16 -> dst [B,Hkv,max_pages*page_size,d] bf16 where
 * dst[b,g,p*page_size + t] = pool[block_table[b,p], g, t]. Pages whose table entry is negative
 * are left untouched. Entries >= num_pages set ATTN_ERR_BOUNDS in the status word and are
 * skipped. This is the page-gather stage of the two-stage paged path of "Optimizing Triton
 * Kernels for Custom Attention Patterns on H100", Pattern C; the fused decode reads pages
 * in place instead.
 */
int attn_gather_pages(const void *pool, void *dst, const int32_t *block_table, int B,
                      int max_pages, int Hkv, int page_size, int d, int num_pages,
                      void *stream);

/*
 * attn_paged_decode_noalloc — paged decode for callers that cannot allocate device memory.
 * (No counterpart on the pages: this is a packaging of attn_fwd's PAGED_DECODE case.)
 *
 * Same arguments, layouts and results as attn_fwd with mask_kind = ATTN_MASK_PAGED_DECODE,
 * without the workspace: the split-KV scratch is a fixed 16 MiB (16777216-byte) array inside
 * the library, held by every GPU that loads it until the process exits. Meant for callers
 * that get no scratch buffer from their host framework (a custom-op interface, another
 * framework's memory pool) or must not let cudaMalloc / cudaFree synchronise the device on a
 * serving path. It allocates nothing.
 *  - Arguments are checked first as attn_fwd checks them (ATTN_ERR_INVALID or
 *    ATTN_ERR_UNSUPPORTED with the reason). Then it returns ATTN_ERR_UNSUPPORTED, with a
 *    message, when attn_workspace_bytes() of the request exceeds the array
 *    (attn_noalloc_scratch_bytes()); nothing is launched then.
 *  - The first call on each device looks up the array's device address (cudaGetSymbolAddress)
 *    with that device current; make that first call before any stream capture.
 *  - Every call shares the one array per device and it keeps the last call's contents. Its
 *    split tickets sit in a fixed region before the partials (one int per sequence x kv head,
 *    B * Hkv at most 65536): zero when the library loads, and left zero by every launch that
 *    runs to its end, so this entry point issues no memset. Calls whose kernels overlap on the
 *    GPU (different streams, or host threads without ordering) race on it: order them.
 */
int attn_paged_decode_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int Hq, int Hkv, int N, int d, float scale,
                              const int32_t *cu_seqlens, const int32_t *block_table,
                              int page_size, int num_pages, void *stream);

/* Size in bytes of attn_paged_decode_noalloc's scratch for partials (16 MiB; its 256 KiB of
 * tickets come on top): a request is served iff attn_workspace_bytes() of it, with mask_kind
 * PAGED_DECODE, is at most this. */
size_t attn_noalloc_scratch_bytes(void);

/* Synchronises `stream`, then returns and clears the device status word (ATTN_OK or one of
 * ATTN_ERR_TIMEOUT / ATTN_ERR_BOUNDS / ATTN_ERR_SEQLENS), or ATTN_ERR_CUDA if the stream
 * reported a CUDA error. */
int attn_get_status(void *stream);

/* Message for the last non-zero return on the calling thread ("" if none). Thread-local;
 * valid until the next call on that thread. */
const char *attn_last_error(void);

/* Failure-detection self-test: launches one thread that waits, through the same bounded
 * wait every kernel uses, on a barrier nothing arrives on. After timeout_ns (1 ns .. 10 s) it
 * gives up and the status word reads ATTN_ERR_TIMEOUT; the GPU context stays usable.
 * Asynchronous; read the outcome with attn_get_status(stream). */
int attn_selftest_wait_timeout(unsigned long long timeout_ns, void *stream);

/* Measurement helper: the exp2 throughput ceiling of this GPU's special-function (MUFU) units,
 * against which the softmax's exponentials per second are reported. Launches `blocks` CTAs of
 * 256 threads (1 .. 65535); every thread evaluates `iters` (1 .. 2^20) rounds of eight
 * independent chains x <- 2^(-x), with the same ex2.approx instruction the softmax uses, and
 * writes one float per thread to `out` (device, blocks * 256 floats, caller-owned) so the work
 * cannot be elided. Exponentials evaluated: blocks * 256 * 8 * iters. Asynchronous on
 * `stream`; the caller times it. Returns ATTN_OK, ATTN_ERR_INVALID or ATTN_ERR_CUDA. */
int attn_bench_ex2(float *out, int blocks, int iters, void *stream);

/* Forgets the library's cached device addresses on every device: the status word's and the
 * allocation-free decode's scratch array's. Call it around cudaDeviceReset (or anything else
 * that ends the context): the next call on a device looks both up again. Must not overlap
 * other calls into the library. */
void attn_release(void);

/* Which device addresses the library has cached for `device`: bit 0 the status word's, bit 1
 * the allocation-free decode's scratch array's (0 after attn_release). ATTN_ERR_INVALID for a
 * device index outside [0, 64). Host-only; makes no CUDA call. */
int attn_cached_device_state(int device);

/* Library version, (major << 16) | minor. */
int attn_version(void);

/*
 * Host-only planning helpers (no CUDA calls; usable without a GPU). They run the same
 * tile-classification code the kernels run, so tests can check the schedule exhaustively.
 *
 * attn_plan_kv_range: for query rows [r0, min(r0+bm, row_end)) and keys indexed from k_org
 * (valid keys [k_org, k_end)), the half-open range [*lo, *hi) of bn-wide key tiles (tile t
 * covers keys k_org + t*bn ... + bn-1) holding at least one visible pair. *hi <= *lo when
 * none does. Returns 0, or ATTN_ERR_INVALID (a decode kind, or a window out of range).
 *
 * attn_plan_tile_kind: 0 if tile t holds no visible pair for those rows, 1 if every (row,
 * key) pair in it is visible (no element mask needed), 2 if it is a boundary tile.
 */
int attn_plan_kv_range(int mask_kind, int window, int r0, int bm, int row_end, int k_org,
                       int k_end, int bn, int *lo, int *hi);
int attn_plan_tile_kind(int mask_kind, int window, int r0, int bm, int row_end, int k_org,
                        int k_end, int bn, int t);

/*
 * attn_plan_units: the prefill work list in launch order. One unit is a pair of bm-row query
 * tiles of one (batch or segment, query head); units are ordered longest-first (pair index
 * descending), then by batch/segment, then head, so the heaviest causal tiles start first and
 * heads sharing a kv head run side by side. cu_seqlens is a HOST array here (document kinds
 * only). For ATTN_MASK_PAGED_PREFILL it holds the B+1 chunk starts followed by the B context
 * lengths, the pair index counts within the chunk, and units are ordered by pair index plus
 * (context - chunk) / (2*bm) descending, so the chunks with the longest contexts start first.
 * Writes up to max_units records of 3 ints (segment or batch, head, pair index) to out and
 * returns the unit count (or a negative ATTN_ERR_*).
 */
int attn_plan_units(int mask_kind, int B, int Hq, int N, const int32_t *cu_seqlens_host,
                    int32_t *out, int max_units);

#ifdef __cplusplus
}
#endif

#endif /* TILED_ATTN_H */
