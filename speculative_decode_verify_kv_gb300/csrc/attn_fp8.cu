// attn_fp8.cu -- instantiations of the attention kernels (mma.sync and tcgen05) for FP8 E4M3 KV caches.
#include "attn.cuh"
#include "attn_umma.cuh"
#include "launch.h"

namespace trtv {

template <int D, int MT>
static cudaError_t go_attn(const CUtensorMap& map, const AttnParams& p, int grid, size_t smem,
                        cudaStream_t st) {
  const void* fn = reinterpret_cast<const void*>(&attn_kernel<true, D, MT>);
  cudaError_t e = ensure_smem_attr(fn, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_kernel<true, D, MT>, dim3(grid), dim3(kThreads), smem, st, map, p);
}

cudaError_t launch_attn_fp8(int head_dim, int mt, const CUtensorMap& map, const AttnParams& p, int grid,
                        size_t smem, cudaStream_t st) {
  if (head_dim != 128) return cudaErrorInvalidValue;
  switch (mt) {
    case 1: return go_attn<128, 1>(map, p, grid, smem, st);
    case 2: return go_attn<128, 2>(map, p, grid, smem, st);
    case 4: return go_attn<128, 4>(map, p, grid, smem, st);
    case 8: return go_attn<128, 8>(map, p, grid, smem, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_umma_fp8(const CUtensorMap& kv_map, const CUtensorMap& q_map, const AttnParams& p,
                                 int grid, size_t smem, cudaStream_t st) {
  const void* fn = reinterpret_cast<const void*>(&attn_umma_kernel<128, true>);
  cudaError_t e = ensure_smem_attr(fn, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_umma_kernel<128, true>, dim3(grid), dim3(kUmmaAttnThreads), smem, st, kv_map, q_map, p);
}

}  // namespace trtv
