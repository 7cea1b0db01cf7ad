// proxy_fp8.cu -- instantiations of the proxy kernel for FP8 E4M3 KV caches.
#include "proxy.cuh"
#include "launch.h"

namespace trtv {

template <int D, int MT>
static cudaError_t go_proxy(const CUtensorMap& map, const ProxyParams& p, int grid, size_t smem,
                        cudaStream_t st) {
  const void* fn = reinterpret_cast<const void*>(&proxy_kernel<true, D, MT>);
  cudaError_t e = ensure_smem_attr(fn, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(proxy_kernel<true, D, MT>, dim3(grid), dim3(kThreads), smem, st, map, p);
}

cudaError_t launch_proxy_fp8(int head_dim, int mt, const CUtensorMap& map, const ProxyParams& p, int grid,
                        size_t smem, cudaStream_t st) {
  if (head_dim != 128) return cudaErrorInvalidValue;
  switch (mt) {
    case 1: return go_proxy<128, 1>(map, p, grid, smem, st);
    case 2: return go_proxy<128, 2>(map, p, grid, smem, st);
    case 4: return go_proxy<128, 4>(map, p, grid, smem, st);
    case 8: return go_proxy<128, 8>(map, p, grid, smem, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace trtv
