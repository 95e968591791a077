// api.cu — the C ABI of include/attn.h: argument validation, tensor-map encoding, work-list
// sizing, kernel dispatch, the device status word, the page-gather kernel and the host-side
// planning helpers.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/attn.h"
#include "launch.h"
#include "sched.h"

namespace ta {

// ------------------------------------------------------------------ errors
namespace {
thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}
}  // namespace

// ------------------------------------------------------------------ device status word
// One int per device (a __device__ variable exists once per device context).
__device__ int g_status_word;

namespace {
constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices];
std::mutex g_mu;

int g_num_sms[kMaxDevices];

// Split-KV scratch of attn_paged_decode_noalloc, for callers that cannot allocate: one fixed
// array per device, held from the library's load until the process exits. Its device address
// is looked up once per device (cudaGetSymbolAddress) and cached here; attn_release forgets it
// together with the status word's. The first kNoAllocTicketBytes hold the split tickets, one
// int per (sequence, kv head): zero when the library loads (device globals start zeroed), and
// every decode launch that runs to its end leaves them zero again, so this entry point needs
// no memset. 65536 tickets cover every request whose partials fit the 16 MiB after them (at
// least 268 bytes per group). The partials follow.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB of partials
constexpr size_t kNoAllocTicketBytes = size_t(256) << 10;   // 65536 tickets
static __device__ __align__(256) unsigned char
    g_noalloc_scratch[kNoAllocTicketBytes + kNoAllocScratchBytes];
void* g_noalloc_scratch_ptr[kMaxDevices];

int sm_count(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device %d", dev);
  if (!g_num_sms[dev]) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    g_num_sms[dev] = n;
  }
  *out = g_num_sms[dev];
  return ATTN_OK;
}

int status_ptr(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_status_ptr[dev];
  return ATTN_OK;
}

// ------------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p)
      return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  *fn = g_encode;
  return ATTN_OK;
}

// 3-D bf16 view [planes][rows][inner] with a 64-column x box_rows box, 128-byte swizzle.
int encode_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t planes,
              uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  int rc = get_encoder(&enc);
  if (rc) return rc;
  cuuint64_t dims[3] = {inner, rows, planes};
  cuuint64_t strides[2] = {inner * 2, inner * 2 * rows};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return ATTN_OK;
}

// 3-D E4M3 (byte) view [planes][rows][inner] with a 128-column x box_rows box, 128-byte
// swizzle: one box row is one 128-byte swizzle row, as for the bf16 maps' 64 columns.
int encode_3d_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                 uint64_t planes, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  int rc = get_encoder(&enc);
  if (rc) return rc;
  cuuint64_t dims[3] = {inner, rows, planes};
  cuuint64_t strides[2] = {inner, inner * rows};
  cuuint32_t box[3] = {128, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled (u8) failed (%d)", (int)r);
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Mask kinds served by the prefill kernel.
bool prefill_kind(int m) {
  return m == ATTN_MASK_NONE || m == ATTN_MASK_CAUSAL || m == ATTN_MASK_SLIDING ||
         m == ATTN_MASK_DOCUMENT || m == ATTN_MASK_SLIDING_BIDIR ||
         m == ATTN_MASK_DOCUMENT_BIDIR || m == ATTN_MASK_PREFIX_LM;
}

bool document_kind(int m) { return m == ATTN_MASK_DOCUMENT || m == ATTN_MASK_DOCUMENT_BIDIR; }

// Page sizes of the paged kinds: multiples of the 8-row swizzle atom that divide the
// 128-row prefill tile and either divide or are twice the 64-row decode stage.
bool page_size_ok(int p) { return p == 16 || p == 32 || p == 64 || p == 128; }

// log2 of a power of two (the page sizes page_size_ok accepts).
int log2_exact(int p) {
  int s = 0;
  while ((1 << s) < p) ++s;
  return s;
}

// The window argument: SLIDING needs >= 1 key, SLIDING_BIDIR >= 0 keys per side, PREFIX_LM a
// prefix of >= 0 tokens; the other kinds ignore it.
bool window_ok(int m, int window) {
  if (m == ATTN_MASK_SLIDING) return window >= 1;
  if (m == ATTN_MASK_SLIDING_BIDIR || m == ATTN_MASK_PREFIX_LM) return window >= 0;
  return true;
}

constexpr unsigned long long kTimeoutNs = 2000000000ull;  // 2 s per pipeline wait
constexpr int kDecodeStage = 64;       // tokens per decode ring stage
constexpr int kMaxDecodeGroup = 16;    // query heads per kv head: the rows of one MMA tile
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeLayout {
  size_t part_o, part_ml, counters, total;
  int max_pages, max_splits, chunk_pages;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Streaming multiprocessors of the current device, or 152 (GB300's count) when no device is
// visible, so that host-only callers size workspaces the same way. Sets no error message.
int sms_or_default() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return 152;
  }
  if (!g_num_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return 152;
    }
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

// 64-token stages per split-KV CTA. Longer CTAs spend less on start-up and on the combine,
// but need enough (sequence, kv head) groups to fill the GPU. Measured on GB300: with 32
// sequences x 8 kv heads of 1K-16K tokens, 32 stages run 3.5 % faster than 16 with 64-token
// pages and 3.9 % with 16-token pages (48 and 64 are slower); with one 16K-token sequence x 8
// kv heads, 16 stages take 25.6 us, 8 stages 27.6 us and 4 stages 33.8 us, and splits sized to
// cover all SMs (14 stages) change nothing. So: 32 once there are as many groups as SMs, else
// 16. The choice depends on B and Hkv only, so every decode of the same batch shape splits,
// and rounds, the same way.
int decode_chunk_pages(int B, int Hkv) {
  return static_cast<long long>(B) * Hkv >= sms_or_default() ? 32 : 16;
}

// Split-KV scratch: splits of decode_chunk_pages 64-token stages over contexts of up to N.
DecodeLayout decode_layout(int B, int Hq, int Hkv, int N, int d) {
  DecodeLayout L{};
  L.chunk_pages = decode_chunk_pages(B, Hkv);
  L.max_pages = (N + kDecodeStage - 1) / kDecodeStage;
  L.max_splits = (L.max_pages + L.chunk_pages - 1) / L.chunk_pages;
  const size_t groups = static_cast<size_t>(B) * Hkv;
  const size_t G = Hkv > 0 ? static_cast<size_t>(Hq / Hkv) : 0;
  L.part_o = 0;
  L.part_ml = align256(groups * L.max_splits * G * d * sizeof(float));
  L.counters = L.part_ml + align256(groups * L.max_splits * G * 2 * sizeof(float));
  L.total = L.counters + align256(groups * sizeof(int));
  return L;
}
}  // namespace

cudaError_t ensure_smem_attr(const void* func, int bytes, unsigned long long* done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) __atomic_fetch_or(done_mask, bit, __ATOMIC_RELEASE);
  return e;
}

// ------------------------------------------------------------------ page gather
__global__ void gather_pages_kernel(const uint4* __restrict__ pool, uint4* __restrict__ dst,
                                    const int* __restrict__ table, int max_pages, int Hkv,
                                    int page_vec, int num_pages, int* status) {
  const int p = static_cast<int>(blockIdx.x);
  const int b = static_cast<int>(blockIdx.y);
  const int phys = table[static_cast<size_t>(b) * max_pages + p];
  if (phys < 0) return;
  if (phys >= num_pages) {
    if (threadIdx.x == 0) report_status(status, ATTN_ERR_BOUNDS);
    return;
  }
  for (int g = 0; g < Hkv; ++g) {
    const uint4* src = pool + (static_cast<size_t>(phys) * Hkv + g) * page_vec;
    uint4* out = dst + ((static_cast<size_t>(b) * Hkv + g) * max_pages + p) * page_vec;
    for (int i = static_cast<int>(threadIdx.x); i < page_vec; i += blockDim.x) out[i] = src[i];
  }
}

// ------------------------------------------------------------------ FP8 block quantization
// One CTA per (128-row block, plane) of x [planes, N, d] (bf16): amax over the block's rows,
// scale = amax / 448 (IEEE fp32 division; 448 is the largest finite E4M3 value), codes =
// E4M3(x / scale) rounded to nearest even with saturation, the division again IEEE fp32. An
// all-zero block gets scale 0 and zero codes. This is the block quantization of the
// FlashAttention-3 page ("FP8 Block Quantization"), one scale per 128-row tile.
//
// Every element of a block is divided by the same scale s, so the correctly rounded quotient
// x / s comes from Markstein's correction step (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990; also
// Muller et al., "Handbook of Floating-Point Arithmetic", the division chapter): with
// y = RN(1/s) and q = RN(x * y) (within one ulp of x / s), the remainder r = x - q * s is exact
// in one FMA, and RN(q + r * y) is RN(x / s). That is one multiply and two FMAs per element
// instead of a full division. A zero quotient keeps the sign of q (x = -0 gives -0), and a
// block whose reciprocal is not finite (s below 2^-126) divides element by element.
constexpr int kFp8Block = 128;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> E4M3 codes in one 16-bit word, `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Persistent: CTA c takes blocks c, c + G, c + 2G, ... of the (plane, 128-row block) list. A
// block is contiguous in memory (rows x d bf16), so one thread brings it into shared memory
// with one bulk copy, and the next block's copy is in flight while this one is converted (two
// buffers): loads overlap the reduction and the conversion instead of following them.
constexpr int kQuantThreads = 256;
constexpr int kQuantBufBytes = kFp8Block * 128 * 2;  // one block: 128 rows x d <= 128 bf16
// Measured on GB300 (Q and K of the causal N=8192 workload, 251 MB): three CTAs per SM with
// two buffers each, 54 us; two CTAs with three buffers, 60 us; 512 threads per CTA, 58 us.
constexpr int kQuantBufs = 2;  // blocks in flight or in use per CTA
constexpr int kQuantCtasPerSm = 3;
constexpr int kQuantSmemBytes = kQuantBufs * kQuantBufBytes + 64;

__global__ void __launch_bounds__(kQuantThreads)
    quantize_fp8_kernel(const uint8_t* __restrict__ x, uint2* __restrict__ x8,
                        float* __restrict__ scales, int N, int d, int nb, int nblocks,
                        int* status, unsigned long long timeout_ns) {
  extern __shared__ __align__(128) uint8_t qsm[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(qsm + kQuantBufs * kQuantBufBytes);
  __shared__ float red[kQuantThreads / 32];
  __shared__ float s_scale;
  __shared__ int s_abort;
  const int tid = static_cast<int>(threadIdx.x);
  if (tid == 0) {
    for (int b = 0; b < kQuantBufs; ++b) mbar_init(&bar[b], 1);
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl wc{timeout_ns, status, &s_abort};
  const WaitCtl wc_drain{timeout_ns, status, nullptr};
  auto issue = [&](int t, int slot) {  // one thread
    const int pl = t / nb, r0 = (t % nb) * kFp8Block;
    const uint32_t bytes = static_cast<uint32_t>(imin(kFp8Block, N - r0) * d * 2);
    mbar_arrive_expect_tx(&bar[slot], bytes);
    bulk_load(qsm + slot * kQuantBufBytes, x + (static_cast<size_t>(pl) * N + r0) * d * 2, bytes,
              &bar[slot]);
  };
  const int G = static_cast<int>(gridDim.x);
  int t = static_cast<int>(blockIdx.x);
  int issued = 0;  // copies issued by thread 0
  if (tid == 0)
    for (int j = 0; j < kQuantBufs - 1 && t + j * G < nblocks; ++j) {
      issue(t + j * G, j);
      ++issued;
    }
  int k = 0;
  for (; t < nblocks; t += G, ++k) {
    const int slot = k % kQuantBufs;
    // The buffer of the block kQuantBufs - 1 ahead was last read in the previous iteration,
    // before its closing barrier.
    const int ta = t + (kQuantBufs - 1) * G;
    if (tid == 0 && ta < nblocks) {
      issue(ta, (k + kQuantBufs - 1) % kQuantBufs);
      ++issued;
    }
    const bool ok = mbar_wait(&bar[slot], (k / kQuantBufs) & 1, wc);
    if (!__syncthreads_and(ok)) break;
    const int pl = t / nb, bt = t % nb, r0 = bt * kFp8Block;
    const int nvec = imin(kFp8Block, N - r0) * d / 8;  // 8-element vectors of the block
    const uint4* v = reinterpret_cast<const uint4*>(qsm + slot * kQuantBufBytes);
    // Block maximum of |x| on packed bf16 pairs (abs and max are exact in bf16).
    __nv_bfloat162 amax2 = __floats2bfloat162_rn(0.f, 0.f);
    for (int i = tid; i < nvec; i += kQuantThreads) {
      const uint4 q = v[i];
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        amax2 = __hmax2(amax2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w[e])));
    }
    float amax = fmaxf(__low2float(amax2), __high2float(amax2));
    for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    if (tid == 0) {
      float m = red[0];
      for (int w = 1; w < kQuantThreads / 32; ++w) m = fmaxf(m, red[w]);
      const float sc = __fdiv_rn(m, 448.f);
      s_scale = sc;
      scales[static_cast<size_t>(pl) * nb + bt] = sc;
    }
    __syncthreads();
    const float sc = s_scale;
    uint2* out = x8 + (static_cast<size_t>(pl) * N + r0) * d / 8;
    const float rc = sc == 0.f ? 0.f : __frcp_rn(sc);
    if (sc == 0.f) {
      for (int i = tid; i < nvec; i += kQuantThreads) out[i] = make_uint2(0u, 0u);
    } else if (isfinite(rc)) {
      // Markstein's correction (see above) on pairs: one packed multiply and two packed
      // FMAs per two elements; a zero quotient keeps the sign of the product.
      const float2 rc2 = make_float2(rc, rc), nsc2 = make_float2(-sc, -sc);
      for (int i = tid; i < nvec; i += kQuantThreads) {
        const uint4 q = v[i];
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        uint32_t c[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 xv = make_float2(bf16_lo(w[e]), bf16_hi(w[e]));
          const float2 q0 = __fmul2_rn(xv, rc2);
          const float2 q1 = __ffma2_rn(__ffma2_rn(q0, nsc2, xv), rc2, q0);
          c[e] = e4m3x2(q1.x == 0.f ? q0.x : q1.x, q1.y == 0.f ? q0.y : q1.y);
        }
        out[i] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
      }
    } else {
      for (int i = tid; i < nvec; i += kQuantThreads) {
        const uint4 q = v[i];
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        uint32_t c[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          c[e] = e4m3x2(__fdiv_rn(bf16_lo(w[e]), sc), __fdiv_rn(bf16_hi(w[e]), sc));
        out[i] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
      }
    }
    __syncthreads();  // this buffer, red and s_scale are free again
  }
  // After a timeout, let copies still in flight land before the CTA exits.
  if (tid == 0)
    for (int j = k; j < issued; ++j)
      mbar_wait(&bar[j % kQuantBufs], (j / kQuantBufs) & 1, wc_drain);
}

// Self-test of the bounded pipeline wait: one thread waits on an mbarrier that nothing
// arrives on, with the same mbar_wait the kernels use, and must give up after timeout_ns,
// record ATTN_ERR_TIMEOUT and return.
__global__ void wait_timeout_selftest_kernel(unsigned long long timeout_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl wc{timeout_ns, status, &abort_flag};
    mbar_wait(&bar, 0, wc);
  }
}

// Exp2 throughput probe: per thread, eight independent chains x <- 2^(-x), one ex2.approx
// (the softmax's instruction) per chain and round. The chains settle at the fixed point of
// 2^(-x) (about 0.641), so no value leaves (0, 1]. One float per thread is stored so the
// work stays live.
__global__ void ex2_rate_kernel(float* out, int iters) {
  float x[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) x[k] = 0.1f * static_cast<float>(k) + 1e-3f * (threadIdx.x & 31);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = fast_exp2(-x[k]);
  }
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) s += x[k];
  out[static_cast<size_t>(blockIdx.x) * 256 + threadIdx.x] = s;
}

}  // namespace ta

using namespace ta;

extern "C" {

int attn_selftest_wait_timeout(unsigned long long timeout_ns, void* stream) {
  g_last_error.clear();
  if (timeout_ns == 0 || timeout_ns > 10000000000ull)
    return fail(ATTN_ERR_INVALID, "timeout_ns must be in (0, 1e10]");
  int* status = nullptr;
  int rc = status_ptr(&status);
  if (rc) return rc;
  wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(timeout_ns,
                                                                               status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return ATTN_OK;
}

int attn_bench_ex2(float* out, int blocks, int iters, void* stream) {
  g_last_error.clear();
  if (!out || blocks < 1 || blocks > 65535 || iters < 1 || iters > (1 << 20))
    return fail(ATTN_ERR_INVALID, "attn_bench_ex2: out, blocks in [1, 65535], iters in [1, 2^20]");
  ex2_rate_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(out, iters);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "ex2 rate launch");
  return ATTN_OK;
}

int attn_version(void) { return (0 << 16) | 1; }

const char* attn_last_error(void) { return g_last_error.c_str(); }

size_t attn_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int mask_kind,
                            int page_size) {
  if (mask_kind == ATTN_MASK_DECODE) page_size = kDecodeStage;
  if ((mask_kind != ATTN_MASK_PAGED_DECODE && mask_kind != ATTN_MASK_DECODE) || B <= 0 ||
      Hkv <= 0 || Hq <= 0 || N <= 0 || page_size <= 0 || d <= 0)
    return 0;
  return decode_layout(B, Hq, Hkv, N, d).total;
}

namespace ta {
namespace {
// The body of attn_fwd. `tickets`, when not null, is a ticket array that is already zero (the
// allocation-free scratch's): the decode then uses it instead of the workspace's and skips
// the memset that clears those.
int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int N, int d, float scale, int mask_kind, int window,
             const int32_t* cu_seqlens, const int32_t* block_table, int page_size,
             int num_pages, void* workspace, size_t workspace_bytes, int* tickets,
             void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (mask_kind < ATTN_MASK_NONE || mask_kind > ATTN_MASK_PREFIX_LM)
    return fail(ATTN_ERR_INVALID, "unknown mask_kind %d", mask_kind);
  const bool decode = mask_kind == ATTN_MASK_PAGED_DECODE || mask_kind == ATTN_MASK_DECODE;
  if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0)
    return fail(ATTN_ERR_INVALID, "need B >= 0, N >= 0, Hq > 0, Hkv > 0");
  if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID, "Hq (%d) %% Hkv (%d) != 0", Hq, Hkv);
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim %d (64 or 128)", d);
  if (!std::isfinite(scale)) return fail(ATTN_ERR_INVALID, "scale is not finite");
  if (!(scale > 0.f)) return fail(ATTN_ERR_UNSUPPORTED, "scale must be > 0");
  if (!window_ok(mask_kind, window))
    return fail(ATTN_ERR_INVALID, "window %d out of range for mask_kind %d", window, mask_kind);
  if ((document_kind(mask_kind) || decode) && !cu_seqlens)
    return fail(ATTN_ERR_INVALID, "cu_seqlens is required");
  if (B == 0 || N == 0) return ATTN_OK;  // nothing to compute
  if (!q || !k || !v || !o || !lse) return fail(ATTN_ERR_INVALID, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(ATTN_ERR_INVALID, "tensors must be 16-byte aligned");
  const int group = Hq / Hkv;
  DecodeLayout L{};
  if (decode) {
    if (mask_kind == ATTN_MASK_PAGED_DECODE) {
      if (!block_table) return fail(ATTN_ERR_INVALID, "block_table is required");
      if (!page_size_ok(page_size))
        return fail(ATTN_ERR_UNSUPPORTED, "page_size %d (16, 32, 64 or 128)", page_size);
      if (num_pages <= 0) return fail(ATTN_ERR_INVALID, "num_pages %d", num_pages);
      if (static_cast<long long>(num_pages) * Hkv >= (1ll << 31))
        return fail(ATTN_ERR_UNSUPPORTED, "page pool too large");
    } else if (static_cast<long long>(B) * Hkv >= (1ll << 31)) {
      return fail(ATTN_ERR_UNSUPPORTED, "B*Hkv too large");
    }
    if (group > kMaxDecodeGroup)
      return fail(ATTN_ERR_UNSUPPORTED, "query heads per kv head %d (at most %d)", group,
                  kMaxDecodeGroup);
    L = decode_layout(B, Hq, Hkv, N, d);
    if (L.max_splits > 65535 || Hkv > 65535 || B > 65535)
      return fail(ATTN_ERR_UNSUPPORTED, "decode grid too large");
    if (!workspace || workspace_bytes < L.total || !aligned16(workspace))
      return fail(ATTN_ERR_WORKSPACE, "workspace needs %zu bytes (16-byte aligned)", L.total);
  } else {
    if (static_cast<long long>(B) * Hq >= (1ll << 31))
      return fail(ATTN_ERR_UNSUPPORTED, "B*Hq too large");
    const long long units = document_kind(mask_kind)
                                ? static_cast<long long>(Hq) * (N / kUnitRows + B)
                                : static_cast<long long>(B) * Hq * pairs_for_rows(N);
    if (units >= (1ll << 31) - 1) return fail(ATTN_ERR_UNSUPPORTED, "too many work units");
  }
  int* status = nullptr;
  int rc = status_ptr(&status);
  if (rc) return rc;

  if (decode) {
    // PAGED_DECODE: the pools as [num_pages * Hkv][page_size][d], boxes of min(page_size, 64)
    // rows; DECODE: the dense caches as [B * Hkv][N][d], boxes of 64 rows.
    const bool dense = mask_kind == ATTN_MASK_DECODE;
    const uint64_t rows = dense ? static_cast<uint64_t>(N) : static_cast<uint64_t>(page_size);
    const uint64_t planes = dense ? static_cast<uint64_t>(B) * Hkv
                                  : static_cast<uint64_t>(num_pages) * Hkv;
    const uint32_t box = dense ? kDecodeStage : static_cast<uint32_t>(imin(page_size, kDecodeStage));
    CUtensorMap tk, tv;
    if ((rc = encode_3d(&tk, k, d, rows, planes, box))) return rc;
    if ((rc = encode_3d(&tv, v, d, rows, planes, box))) return rc;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    DecodeParams p{};
    p.q = static_cast<const uint4*>(q);
    p.cu = cu_seqlens;
    p.table = dense ? nullptr : block_table;
    p.dense = dense ? 1 : 0;
    p.o = o;
    p.lse = lse;
    p.part_o = reinterpret_cast<float*>(ws + L.part_o);
    p.part_ml = reinterpret_cast<float*>(ws + L.part_ml);
    p.counters = tickets ? tickets : reinterpret_cast<int*>(ws + L.counters);
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.max_pages = dense ? 0 : (N + page_size - 1) / page_size;
    p.num_pages = dense ? 0 : num_pages;
    p.page_shift = dense ? 6 : log2_exact(page_size);
    p.max_len = N;
    p.max_splits = L.max_splits;
    p.chunk_pages = L.chunk_pages;
    p.group = group;
    p.scale_log2 = scale * kLog2e;
    p.status = status;
    p.timeout_ns = kTimeoutNs;
    cudaError_t e = cudaSuccess;
    if (!tickets) {
      e = cudaMemsetAsync(p.counters, 0, sizeof(int) * static_cast<size_t>(B) * Hkv, stream);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(counters)");
    }
    e = launch_decode(d, group, tk, tv, p, dim3(L.max_splits, Hkv, B), stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return ATTN_OK;
  }

  // Prefill kinds. For DOCUMENT the unit count is an upper bound (the segment lengths live
  // on the device): units past the real end decode invalid and end a CTA's loop.
  const int planes_q = document_kind(mask_kind) ? Hq : B * Hq;
  const int planes_kv = document_kind(mask_kind) ? Hkv : B * Hkv;
  const long long units = document_kind(mask_kind)
                              ? static_cast<long long>(Hq) * (N / kUnitRows + B)
                              : static_cast<long long>(B) * Hq * pairs_for_rows(N);
  CUtensorMap tq, tk, tv, to;
  if ((rc = encode_3d(&tq, q, d, N, planes_q, 128))) return rc;
  if ((rc = encode_3d(&to, o, d, N, planes_q, 32))) return rc;
  const uint32_t kv_rows = static_cast<uint32_t>(prefill_key_tile(d, mask_kind));
  if ((rc = encode_3d(&tk, k, d, N, planes_kv, kv_rows))) return rc;
  if ((rc = encode_3d(&tv, v, d, N, planes_kv, kv_rows))) return rc;
  PrefillParams p{};
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = cu_seqlens;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.group = group;
  p.num_units = static_cast<int>(units);
  p.window = window;
  p.scale_log2 = scale * kLog2e;
  p.status = status;
  p.timeout_ns = kTimeoutNs;
  // Persistent: at most one CTA per SM (the kernel needs a whole SM's shared memory).
  int sms = 0;
  if ((rc = sm_count(&sms))) return rc;
  const int grid = p.num_units < sms ? p.num_units : sms;
  cudaError_t e = d == 64 ? launch_prefill_d64(mask_kind, tq, tk, tv, to, p, grid, stream)
                          : launch_prefill_d128(mask_kind, tq, tk, tv, to, p, grid, stream);
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return ATTN_OK;
}
}  // namespace
}  // namespace ta

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int N, int d, float scale, int mask_kind, int window,
             const int32_t* cu_seqlens, const int32_t* block_table, int page_size,
             int num_pages, void* workspace, size_t workspace_bytes, void* stream) {
  g_last_error.clear();
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, mask_kind, window, cu_seqlens,
                  block_table, page_size, num_pages, workspace, workspace_bytes, nullptr, stream);
}

int attn_fwd_paged_prefill(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int Hq, int Hkv, int total_q, int d, float scale,
                           const int32_t* cu_seqlens_q, const int32_t* seqlens_k,
                           const int32_t* block_table, int max_pages, int page_size,
                           int num_pages, void* stream) {
  g_last_error.clear();
  if (B < 0 || total_q < 0 || Hq <= 0 || Hkv <= 0)
    return fail(ATTN_ERR_INVALID, "need B >= 0, total_q >= 0, Hq > 0, Hkv > 0");
  if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID, "Hq (%d) %% Hkv (%d) != 0", Hq, Hkv);
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim %d (64 or 128)", d);
  if (!std::isfinite(scale)) return fail(ATTN_ERR_INVALID, "scale is not finite");
  if (!(scale > 0.f)) return fail(ATTN_ERR_UNSUPPORTED, "scale must be > 0");
  if (!page_size_ok(page_size))
    return fail(ATTN_ERR_UNSUPPORTED, "page_size %d (16, 32, 64 or 128)", page_size);
  if (B == 0 || total_q == 0) return ATTN_OK;  // no query rows
  if (!q || !k || !v || !o || !lse || !cu_seqlens_q || !seqlens_k || !block_table)
    return fail(ATTN_ERR_INVALID, "null pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(ATTN_ERR_INVALID, "tensors must be 16-byte aligned");
  if (max_pages <= 0 || num_pages <= 0)
    return fail(ATTN_ERR_INVALID, "max_pages %d, num_pages %d", max_pages, num_pages);
  if (static_cast<long long>(num_pages) * Hkv >= (1ll << 31) ||
      static_cast<long long>(max_pages) * page_size >= (1ll << 31))
    return fail(ATTN_ERR_UNSUPPORTED, "page pool or block table too large");
  const long long units = static_cast<long long>(Hq) * (total_q / kUnitRows + B);
  if (units >= (1ll << 31) - 1) return fail(ATTN_ERR_UNSUPPORTED, "too many work units");
  int* status = nullptr;
  int rc = status_ptr(&status);
  if (rc) return rc;
  // Q, O, LSE packed [1, Hq, total_q]; the pools as [num_pages * Hkv][page_size][d] with one
  // page per box.
  CUtensorMap tq, tk, tv, to;
  if ((rc = encode_3d(&tq, q, d, total_q, Hq, 128))) return rc;
  if ((rc = encode_3d(&to, o, d, total_q, Hq, 32))) return rc;
  const uint64_t planes = static_cast<uint64_t>(num_pages) * Hkv;
  if ((rc = encode_3d(&tk, k, d, page_size, planes, page_size))) return rc;
  if ((rc = encode_3d(&tv, v, d, page_size, planes, page_size))) return rc;
  PrefillParams p{};
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = cu_seqlens_q;
  p.seqlens_k = seqlens_k;
  p.table = block_table;
  p.max_pages = max_pages;
  p.page_size = page_size;
  p.page_shift = log2_exact(page_size);
  p.num_pages = num_pages;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = total_q;
  p.group = Hq / Hkv;
  p.num_units = static_cast<int>(units);
  p.window = 0;
  p.scale_log2 = scale * kLog2e;
  p.status = status;
  p.timeout_ns = kTimeoutNs;
  int sms = 0;
  if ((rc = sm_count(&sms))) return rc;
  const int grid = p.num_units < sms ? p.num_units : sms;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = d == 64 ? launch_prefill_d64(kMaskPagedPrefill, tq, tk, tv, to, p, grid, st)
                          : launch_prefill_d128(kMaskPagedPrefill, tq, tk, tv, to, p, grid, st);
  if (e != cudaSuccess) return cuda_fail(e, "paged prefill launch");
  return ATTN_OK;
}

int attn_quantize_fp8(const void* x, void* x8, float* scales, int planes, int N, int d,
                      void* stream) {
  g_last_error.clear();
  if (planes < 0 || N < 0) return fail(ATTN_ERR_INVALID, "planes %d, N %d", planes, N);
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim %d (64 or 128)", d);
  if (planes == 0 || N == 0) return ATTN_OK;
  if (!x || !x8 || !scales) return fail(ATTN_ERR_INVALID, "null pointer");
  if (!aligned16(x) || !aligned16(x8) || (reinterpret_cast<uintptr_t>(scales) & 3u))
    return fail(ATTN_ERR_INVALID, "x and x8 must be 16-byte aligned, scales 4-byte aligned");
  if (planes > 65535) return fail(ATTN_ERR_UNSUPPORTED, "planes %d > 65535", planes);
  const int nb = (N + kFp8Block - 1) / kFp8Block;
  if (static_cast<long long>(nb) * planes >= (1ll << 31) - (1ll << 20))
    return fail(ATTN_ERR_UNSUPPORTED, "too many 128-row blocks");
  const int nblocks = nb * planes;
  int* status = nullptr;
  int rc = status_ptr(&status);
  if (rc) return rc;
  int sms = 0;
  if ((rc = sm_count(&sms))) return rc;
  static unsigned long long done = 0;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(quantize_fp8_kernel),
                                   kQuantSmemBytes, &done);
  if (e != cudaSuccess) return cuda_fail(e, "quantize smem attribute");
  const int grid = nblocks < kQuantCtasPerSm * sms ? nblocks : kQuantCtasPerSm * sms;
  quantize_fp8_kernel<<<grid, kQuantThreads, kQuantSmemBytes, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t*>(x), static_cast<uint2*>(x8), scales, N, d, nb, nblocks, status,
      kTimeoutNs);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return ATTN_OK;
}

int attn_fwd_fp8(const void* q8, const void* k8, const void* v, void* o, float* lse,
                 const float* q_scales, const float* k_scales, int B, int Hq, int Hkv, int N,
                 int d, float scale, int mask_kind, int window, void* stream) {
  g_last_error.clear();
  if (mask_kind < ATTN_MASK_NONE || mask_kind > ATTN_MASK_PAGED_PREFILL)
    return fail(ATTN_ERR_INVALID, "unknown mask_kind %d", mask_kind);
  if (mask_kind != ATTN_MASK_NONE && mask_kind != ATTN_MASK_CAUSAL &&
      mask_kind != ATTN_MASK_SLIDING && mask_kind != ATTN_MASK_SLIDING_BIDIR &&
      mask_kind != ATTN_MASK_PREFIX_LM)
    return fail(ATTN_ERR_UNSUPPORTED, "FP8 takes the dense mask kinds (not %d)", mask_kind);
  if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0)
    return fail(ATTN_ERR_INVALID, "need B >= 0, N >= 0, Hq > 0, Hkv > 0");
  if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID, "Hq (%d) %% Hkv (%d) != 0", Hq, Hkv);
  if (d != 128) return fail(ATTN_ERR_UNSUPPORTED, "FP8 head dim %d (128)", d);
  if (!std::isfinite(scale)) return fail(ATTN_ERR_INVALID, "scale is not finite");
  if (!(scale > 0.f)) return fail(ATTN_ERR_UNSUPPORTED, "scale must be > 0");
  if (!window_ok(mask_kind, window))
    return fail(ATTN_ERR_INVALID, "window %d out of range for mask_kind %d", window, mask_kind);
  if (B == 0 || N == 0) return ATTN_OK;
  if (!q8 || !k8 || !v || !o || !lse || !q_scales || !k_scales)
    return fail(ATTN_ERR_INVALID, "null pointer");
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(ATTN_ERR_INVALID, "tensors must be 16-byte aligned");
  if (static_cast<long long>(B) * Hq >= (1ll << 31))
    return fail(ATTN_ERR_UNSUPPORTED, "B*Hq too large");
  const long long units = static_cast<long long>(B) * Hq * pairs_for_rows(N);
  if (units >= (1ll << 31) - 1) return fail(ATTN_ERR_UNSUPPORTED, "too many work units");
  int* status = nullptr;
  int rc = status_ptr(&status);
  if (rc) return rc;
  CUtensorMap tq, tk, tv, to;
  if ((rc = encode_3d_u8(&tq, q8, d, N, static_cast<uint64_t>(B) * Hq, 128))) return rc;
  if ((rc = encode_3d_u8(&tk, k8, d, N, static_cast<uint64_t>(B) * Hkv, 128))) return rc;
  if ((rc = encode_3d(&tv, v, d, N, static_cast<uint64_t>(B) * Hkv, 128))) return rc;
  if ((rc = encode_3d(&to, o, d, N, static_cast<uint64_t>(B) * Hq, 32))) return rc;
  PrefillParams p{};
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.group = Hq / Hkv;
  p.num_units = static_cast<int>(units);
  p.window = window;
  p.scale_log2 = scale * kLog2e;
  p.q_scales = q_scales;
  p.k_scales = k_scales;
  p.nbq = p.nbk = (N + kFp8Block - 1) / kFp8Block;
  p.status = status;
  p.timeout_ns = kTimeoutNs;
  int sms = 0;
  if ((rc = sm_count(&sms))) return rc;
  const int grid = p.num_units < sms ? p.num_units : sms;
  cudaError_t e =
      launch_prefill_fp8(mask_kind, tq, tk, tv, to, p, grid, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "FP8 prefill launch");
  return ATTN_OK;
}

int attn_gather_pages(const void* pool, void* dst, const int32_t* block_table, int B,
                      int max_pages, int Hkv, int page_size, int d, int num_pages,
                      void* stream) {
  g_last_error.clear();
  if (B < 0 || max_pages < 0 || Hkv <= 0 || page_size <= 0 || d <= 0 || num_pages < 0)
    return fail(ATTN_ERR_INVALID, "bad gather sizes");
  if (B == 0 || max_pages == 0) return ATTN_OK;
  if (!pool || !dst || !block_table) return fail(ATTN_ERR_INVALID, "null pointer");
  if (!aligned16(pool) || !aligned16(dst))
    return fail(ATTN_ERR_INVALID, "pool and dst must be 16-byte aligned");
  if ((static_cast<long long>(page_size) * d * 2) % 16 != 0)
    return fail(ATTN_ERR_UNSUPPORTED, "page_size * d * 2 must be a multiple of 16");
  if (max_pages > 2147483647 || B > 65535) return fail(ATTN_ERR_UNSUPPORTED, "grid too large");
  int* status = nullptr;
  int rc = status_ptr(&status);
  if (rc) return rc;
  const int page_vec = page_size * d * 2 / 16;
  gather_pages_kernel<<<dim3(max_pages, B), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(pool), static_cast<uint4*>(dst), block_table, max_pages, Hkv,
      page_vec, num_pages, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "gather launch");
  return ATTN_OK;
}

int attn_get_status(void* stream) {
  g_last_error.clear();
  int* status = nullptr;
  int rc = status_ptr(&status);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int value = 0;
  cudaError_t e = cudaMemcpyAsync(&value, status, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  if (value != 0) {
    const int zero = 0;
    e = cudaMemcpyAsync(status, &zero, sizeof(int), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    fail(value, "device status %d", value);
  }
  return value;
}

void attn_release(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < kMaxDevices; ++i) {
    g_status_ptr[i] = nullptr;
    g_noalloc_scratch_ptr[i] = nullptr;
  }
}

int attn_cached_device_state(int device) {
  if (device < 0 || device >= kMaxDevices) return ATTN_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  return (g_status_ptr[device] ? 1 : 0) | (g_noalloc_scratch_ptr[device] ? 2 : 0);
}

int attn_plan_kv_range(int mask_kind, int window, int r0, int bm, int row_end, int k_org,
                       int k_end, int bn, int* lo, int* hi) {
  if (!lo || !hi || bm <= 0 || bn <= 0 || !prefill_kind(mask_kind) ||
      !window_ok(mask_kind, window))
    return ATTN_ERR_INVALID;
  const KvRange r = kv_tile_range(mask_kind, window, r0, bm, row_end, k_org, k_end, bn);
  *lo = r.lo;
  *hi = r.hi;
  return ATTN_OK;
}

int attn_plan_tile_kind(int mask_kind, int window, int r0, int bm, int row_end, int k_org,
                        int k_end, int bn, int t) {
  if (bm <= 0 || bn <= 0 || !prefill_kind(mask_kind) || !window_ok(mask_kind, window))
    return ATTN_ERR_INVALID;
  return tile_kind(mask_kind, window, r0, bm, row_end, k_org, k_end, bn, t);
}

int attn_plan_units(int mask_kind, int B, int Hq, int N, const int32_t* cu, int32_t* out,
                    int max_units) {
  const bool paged = mask_kind == ATTN_MASK_PAGED_PREFILL;
  if (B < 0 || Hq <= 0 || N < 0 || !(prefill_kind(mask_kind) || paged))
    return ATTN_ERR_INVALID;
  std::vector<int32_t> units;
  if (paged) {
    // cu holds the chunk starts [B+1] followed by the context lengths [B]. A unit's level is
    // its pair index plus the pairs of context before its chunk.
    if (!cu) return ATTN_ERR_INVALID;
    const int32_t* lk = cu + B + 1;
    int tmax = 0;
    for (int s = 0; s < B; ++s) {
      const int len = cu[s + 1] - cu[s];
      if (len < 0 || lk[s] < len) return ATTN_ERR_SEQLENS;
      tmax = imax(tmax, (lk[s] - len) / kUnitRows + pairs_for_rows(len));
    }
    for (int t = tmax - 1; t >= 0; --t)
      for (int s = 0; s < B; ++s) {
        const int l0 = (lk[s] - (cu[s + 1] - cu[s])) / kUnitRows;
        if (t >= l0 && t < l0 + pairs_for_rows(cu[s + 1] - cu[s]))
          for (int h = 0; h < Hq; ++h) units.insert(units.end(), {s, h, t - l0});
      }
  } else if (!document_kind(mask_kind)) {
    const int npairs = pairs_for_rows(N);
    for (int level = npairs - 1; level >= 0; --level)
      for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hq; ++h) units.insert(units.end(), {b, h, level});
  } else if (mask_kind == ATTN_MASK_DOCUMENT_BIDIR) {
    // Sorted by cost: levels are key-tile counts, highest first; on a level, segments in
    // order, their pairs of that cost in order, then heads.
    if (!cu) return ATTN_ERR_INVALID;
    int cmax = 0;
    for (int s = 0; s < B; ++s) {
      const int len = cu[s + 1] - cu[s];
      if (len < 0) return ATTN_ERR_SEQLENS;
      cmax = imax(cmax, 2 * tiles_for_rows(len));
    }
    for (int c = cmax; c >= 1; --c)
      for (int s = 0; s < B; ++s) {
        const int len = cu[s + 1] - cu[s];
        const int k = pairs_of_cost(len, c);
        for (int x = 0; x < k; ++x) {
          const int pair = 2 * tiles_for_rows(len) == c ? x : pairs_for_rows(len) - 1;
          for (int h = 0; h < Hq; ++h) units.insert(units.end(), {s, h, pair});
        }
      }
  } else {
    if (!cu) return ATTN_ERR_INVALID;
    int tmax = 0;
    for (int s = 0; s < B; ++s) {
      const int len = cu[s + 1] - cu[s];
      if (len < 0) return ATTN_ERR_SEQLENS;
      tmax = imax(tmax, pairs_for_rows(len));
    }
    for (int t = tmax - 1; t >= 0; --t)
      for (int s = 0; s < B; ++s)
        if (pairs_for_rows(cu[s + 1] - cu[s]) > t)
          for (int h = 0; h < Hq; ++h) units.insert(units.end(), {s, h, t});
  }
  const int n = static_cast<int>(units.size() / 3);
  if (out)
    std::memcpy(out, units.data(), sizeof(int32_t) * 3 * static_cast<size_t>(imin(n, max_units)));
  return n;
}

}  // extern "C"

// ------------------------------------------------------------------ allocation-free decode
// Some callers cannot hand this library a workspace and cannot let it call cudaMalloc: code
// running inside another framework's device-memory pool or a custom-op interface that passes
// no scratch buffer, and serving loops where the implicit device synchronisation of
// cudaMalloc / cudaFree is not acceptable. attn_paged_decode_noalloc serves them: its
// split-KV partials and tickets live in g_noalloc_scratch (declared with the status word),
// which every GPU that loads this library holds until the process exits.
namespace ta {
namespace {
// Device address of the scratch array on the current device. In host code the array's name
// is only a host-side stand-in, so the address comes from cudaGetSymbolAddress, once per
// device, with that device current.
int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_noalloc_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(decode scratch)");
    g_noalloc_scratch_ptr[dev] = p;
  }
  *out = g_noalloc_scratch_ptr[dev];
  return ATTN_OK;
}
}  // namespace
}  // namespace ta

extern "C" size_t attn_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int attn_paged_decode_noalloc(const void* q, const void* k, const void* v, void* o,
                                         float* lse, int B, int Hq, int Hkv, int N, int d,
                                         float scale, const int32_t* cu_seqlens,
                                         const int32_t* block_table, int page_size,
                                         int num_pages, void* stream) {
  g_last_error.clear();
  // The cheap argument checks come first, so that an invalid request reports its own reason
  // rather than a scratch size computed from invalid arguments.
  if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0)
    return fail(ATTN_ERR_INVALID, "need B >= 0, N >= 0, Hq > 0, Hkv > 0");
  if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID, "Hq (%d) %% Hkv (%d) != 0", Hq, Hkv);
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim %d (64 or 128)", d);
  if (!page_size_ok(page_size))
    return fail(ATTN_ERR_UNSUPPORTED, "page_size %d (16, 32, 64 or 128)", page_size);
  if (Hq / Hkv > kMaxDecodeGroup)
    return fail(ATTN_ERR_UNSUPPORTED, "query heads per kv head %d (at most %d)", Hq / Hkv,
                kMaxDecodeGroup);
  const size_t need =
      attn_workspace_bytes(B, Hq, Hkv, N, d, ATTN_MASK_PAGED_DECODE, page_size);
  if (need > kNoAllocScratchBytes)
    return fail(ATTN_ERR_UNSUPPORTED,
                "this decode needs %zu bytes of split-KV scratch; the allocation-free entry "
                "point has %zu (fewer sequences, kv heads or a shorter longest context fit)",
                need, kNoAllocScratchBytes);
  if (static_cast<long long>(B) * Hkv > static_cast<long long>(kNoAllocTicketBytes / sizeof(int)))
    return fail(ATTN_ERR_UNSUPPORTED, "B * Hkv %lld above the %zu tickets of the scratch",
                static_cast<long long>(B) * Hkv, kNoAllocTicketBytes / sizeof(int));
  void* scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  // The tickets are the scratch's fixed, already-zero ones (no memset); the partials, written
  // before they are read, follow them.
  uint8_t* base = static_cast<uint8_t*>(scratch);
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, ATTN_MASK_PAGED_DECODE, 0,
                  cu_seqlens, block_table, page_size, num_pages, base + kNoAllocTicketBytes,
                  kNoAllocScratchBytes, reinterpret_cast<int*>(base), stream);
}
