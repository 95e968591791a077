// decode.cu — instantiations of the paged decode kernel (head dim 64 / 128, group 1 / 2 / 4 / 8).
#include "launch.h"

namespace ta {

namespace {
template <int D, int G>
cudaError_t launch_one(const CUtensorMap& k, const CUtensorMap& v, const DecodeParams& p,
                       dim3 grid, cudaStream_t stream) {
  static unsigned long long done = 0;
  auto kern = decode_kernel<D, G>;
  constexpr int smem = DecodeCfg<D, G>::kSmemBytes;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem, &done);
  if (e != cudaSuccess) return e;
  kern<<<grid, DecodeCfg<D, G>::kThreads, smem, stream>>>(k, v, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(int group, const CUtensorMap& k, const CUtensorMap& v,
                     const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_one<D, 1>(k, v, p, grid, stream);
    case 2: return launch_one<D, 2>(k, v, p, grid, stream);
    case 4: return launch_one<D, 4>(k, v, p, grid, stream);
    case 8: return launch_one<D, 8>(k, v, p, grid, stream);
    case 16: return launch_one<D, 16>(k, v, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t launch_decode(int d, int group, const CUtensorMap& k, const CUtensorMap& v,
                          const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  return d == 64 ? launch_d<64>(group, k, v, p, grid, stream)
                 : launch_d<128>(group, k, v, p, grid, stream);
}

}  // namespace ta
