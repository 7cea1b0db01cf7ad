// attn_pm.cu -- instantiations of the position-major tcgen05 attention kernel
// (FP8 E4M3 caches, row tiles of 16 and 32).
#include "attn_pm.cuh"
#include "launch.h"

namespace trtv {

template <bool FP8, int NR>
static cudaError_t go_pm(const CUtensorMap& kv_map, const CUtensorMap& q_map, const AttnParams& p, int grid,
                         size_t smem, cudaStream_t st) {
  const void* fn = reinterpret_cast<const void*>(&attn_pm_kernel<FP8, NR>);
  cudaError_t e = ensure_smem_attr(fn, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_pm_kernel<FP8, NR>, dim3(grid), dim3(pm_threads(FP8, NR)), smem, st,
                    kv_map, q_map, p);
}

cudaError_t launch_attn_pm(bool fp8, int nr, const CUtensorMap& kv_map, const CUtensorMap& q_map,
                           const AttnParams& p, int grid, size_t smem, cudaStream_t st) {
  if (!fp8) return cudaErrorInvalidValue;  // bf16 tiles of at most 32 rows run on the mma.sync kernel
  if (nr == 16) return go_pm<true, 16>(kv_map, q_map, p, grid, smem, st);
  if (nr == 32) return go_pm<true, 32>(kv_map, q_map, p, grid, smem, st);
  return cudaErrorInvalidValue;
}

}  // namespace trtv
