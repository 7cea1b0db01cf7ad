// attn_bf16.cu -- instantiations of the attention kernels (mma.sync and tcgen05) for bf16 KV caches.
#include "attn.cuh"
#include "attn_umma.cuh"
#include "launch.h"

namespace trtv {

template <int D, int MT>
static cudaError_t go_attn(const CUtensorMap& map, const AttnParams& p, int grid, size_t smem,
                        cudaStream_t st) {
  const void* fn = reinterpret_cast<const void*>(&attn_kernel<false, D, MT>);
  cudaError_t e = ensure_smem_attr(fn, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_kernel<false, D, MT>, dim3(grid), dim3(kThreads), smem, st, map, p);
}

cudaError_t launch_attn_bf16(int head_dim, int mt, const CUtensorMap& map, const AttnParams& p, int grid,
                        size_t smem, cudaStream_t st) {
  if (head_dim == 128) {
    switch (mt) {
      case 1: return go_attn<128, 1>(map, p, grid, smem, st);
      case 2: return go_attn<128, 2>(map, p, grid, smem, st);
      case 4: return go_attn<128, 4>(map, p, grid, smem, st);
      case 8: return go_attn<128, 8>(map, p, grid, smem, st);
    }
  } else if (head_dim == 64) {
    switch (mt) {
      case 1: return go_attn<64, 1>(map, p, grid, smem, st);
      case 2: return go_attn<64, 2>(map, p, grid, smem, st);
      case 4: return go_attn<64, 4>(map, p, grid, smem, st);
      case 8: return go_attn<64, 8>(map, p, grid, smem, st);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_umma(const CUtensorMap& kv_map, const CUtensorMap& q_map, const AttnParams& p,
                             int grid, size_t smem, cudaStream_t st) {
  // 64-row tiles: M = 64 UMMAs with 16 rows in every TMEM lane quadrant
  if (p.rows_pad == 64) {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(&attn_umma_kernel<128, false, true>), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_umma_kernel<128, false, true>, dim3(grid), dim3(kUmmaAttnThreads), smem, st, kv_map,
                      q_map, p);
  }
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(&attn_umma_kernel<128, false>), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_umma_kernel<128, false>, dim3(grid), dim3(kUmmaAttnThreads), smem, st, kv_map, q_map, p);
}

}  // namespace trtv
