// launch.h — host-side launchers of the kernel instantiations (each defined in its own
// translation unit so the instantiations compile in parallel).
#pragma once

#include <cuda_runtime.h>

#include "decode.cuh"
#include "prefill.cuh"

namespace ta {

// Launch prefill_kernel<d, mask> with `grid` CTAs; returns the launch error. `o` maps the
// output with 32-row boxes (one softmax warp's rows).
cudaError_t launch_prefill_d64(int mask, const CUtensorMap& q, const CUtensorMap& k,
                               const CUtensorMap& v, const CUtensorMap& o,
                               const PrefillParams& p, int grid, cudaStream_t stream);
cudaError_t launch_prefill_d128(int mask, const CUtensorMap& q, const CUtensorMap& k,
                                const CUtensorMap& v, const CUtensorMap& o,
                                const PrefillParams& p, int grid, cudaStream_t stream);

// Launch prefill_kernel<128, mask, FP8 = true> (E4M3 Q / K; dense mask kinds).
cudaError_t launch_prefill_fp8(int mask, const CUtensorMap& q, const CUtensorMap& k,
                               const CUtensorMap& v, const CUtensorMap& o,
                               const PrefillParams& p, int grid, cudaStream_t stream);

// Launch decode_kernel<d, group> on grid (max_splits, Hkv, B).
cudaError_t launch_decode(int d, int group, const CUtensorMap& k, const CUtensorMap& v,
                          const DecodeParams& p, dim3 grid, cudaStream_t stream);

// Sets the dynamic shared-memory limit of `func` once per device.
cudaError_t ensure_smem_attr(const void* func, int bytes, unsigned long long* done_mask);

}  // namespace ta
