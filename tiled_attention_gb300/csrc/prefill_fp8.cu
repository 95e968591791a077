// prefill_fp8.cu — instantiations of the prefill kernel with E4M3 Q / K (head dimension 128,
// the dense mask kinds).
#include "launch.h"

namespace ta {

namespace {
template <int MASK>
cudaError_t launch_one(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& o, const PrefillParams& p, int grid,
                       cudaStream_t stream) {
  static unsigned long long done = 0;
  auto kern = prefill_kernel<128, MASK, true>;
  constexpr int smem = PrefillCfg<128, prefill_key_tile(128, MASK)>::kSmemBytes;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem, &done);
  if (e != cudaSuccess) return e;
  using Cfg = PrefillCfg<128, prefill_key_tile(128, MASK)>;
  kern<<<grid, Cfg::kThreads, smem, stream>>>(q, k, v, o, p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_prefill_fp8(int mask, const CUtensorMap& q, const CUtensorMap& k,
                               const CUtensorMap& v, const CUtensorMap& o,
                               const PrefillParams& p, int grid, cudaStream_t stream) {
  switch (mask) {
    case kMaskNone: return launch_one<kMaskNone>(q, k, v, o, p, grid, stream);
    case kMaskCausal: return launch_one<kMaskCausal>(q, k, v, o, p, grid, stream);
    case kMaskSliding: return launch_one<kMaskSliding>(q, k, v, o, p, grid, stream);
    case kMaskSlidingBidir: return launch_one<kMaskSlidingBidir>(q, k, v, o, p, grid, stream);
    case kMaskPrefixLM: return launch_one<kMaskPrefixLM>(q, k, v, o, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ta
