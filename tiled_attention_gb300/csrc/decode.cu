// decode.cu — instantiations of the paged decode kernel: head dim 64 / 128, and 1, 2, 4, 8 or
// 16 tile rows of query heads (a group of G heads runs on the smallest that holds it).
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
  if (group < 1 || group > 16) return cudaErrorInvalidValue;
  if (group == 1) return launch_one<D, 1>(k, v, p, grid, stream);
  if (group == 2) return launch_one<D, 2>(k, v, p, grid, stream);
  if (group <= 4) return launch_one<D, 4>(k, v, p, grid, stream);
  if (group <= 8) return launch_one<D, 8>(k, v, p, grid, stream);
  return launch_one<D, 16>(k, v, p, grid, stream);
}
}  // namespace

cudaError_t launch_decode(int d, int group, const CUtensorMap& k, const CUtensorMap& v,
                          const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  return d == 64 ? launch_d<64>(group, k, v, p, grid, stream)
                 : launch_d<128>(group, k, v, p, grid, stream);
}

}  // namespace ta
