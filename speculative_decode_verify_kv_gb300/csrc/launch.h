// launch.h -- host-side launchers of the kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace trtv {

struct AttnParams;
struct ProxyParams;
struct PlanOut;

// n int32 counters set to 0 on `st` (a kernel in the programmatic launch chain)
cudaError_t launch_zero(int32_t* c, int n, cudaStream_t st);

// attention: head_dim in {64, 128}; mt (row tiles of 16) in {1, 2, 4, 8}
cudaError_t launch_attn_bf16(int head_dim, int mt, const CUtensorMap& map, const AttnParams& p,
                             int grid, size_t smem, cudaStream_t st);
cudaError_t launch_attn_fp8(int head_dim, int mt, const CUtensorMap& map, const AttnParams& p,
                            int grid, size_t smem, cudaStream_t st);
cudaError_t launch_proxy_bf16(int head_dim, int mt, const CUtensorMap& map, const ProxyParams& p,
                              int grid, size_t smem, cudaStream_t st);
cudaError_t launch_proxy_fp8(int head_dim, int mt, const CUtensorMap& map, const ProxyParams& p,
                             int grid, size_t smem, cudaStream_t st);

// tcgen05 attention: bf16, head_dim 128, power-of-two group, group * qo_len <= 128
cudaError_t launch_attn_umma(const CUtensorMap& kv_map, const CUtensorMap& q_map, const AttnParams& p,
                             int grid, size_t smem, cudaStream_t st);

// tcgen05 attention over FP8 E4M3 caches: head_dim 128, power-of-two group,
// 32 < group * qo_len <= 64 (kind::f8f6f4 UMMAs; Q and P as two E4M3 terms)
cudaError_t launch_attn_umma_fp8(const CUtensorMap& kv_map, const CUtensorMap& q_map, const AttnParams& p,
                                 int grid, size_t smem, cudaStream_t st);

// position-major tcgen05 attention (positions on the UMMA's M, rows on N):
// FP8 caches, head_dim 128, power-of-two group, group * qo_len <= nr rows,
// nr in {16, 32}
cudaError_t launch_attn_pm(bool fp8, int nr, const CUtensorMap& kv_map, const CUtensorMap& q_map,
                           const AttnParams& p, int grid, size_t smem, cudaStream_t st);

// tcgen05 proxy: bf16, head_dim 128, power-of-two group <= 16, group * qo_len <= 128
cudaError_t launch_proxy_umma(const CUtensorMap& kv_map, const CUtensorMap& q_map, const ProxyParams& p,
                              int grid, size_t smem, cudaStream_t st);

cudaError_t launch_subpage_view(const int32_t* pt, const int32_t* lens, int32_t* k_sub,
                                int32_t* v_sub, int batch, int qo_len, int max_pages,
                                int num_slots, int stride, int* err, cudaStream_t st);
cudaError_t launch_sparse_plan(const int32_t* idx, const int32_t* lens, int batch, int qo_len,
                               int num_kv_heads, int max_pages, int topk, const PlanOut& out,
                               const int32_t* pt, int num_slots, int* err, cudaStream_t st);
cudaError_t launch_topk(const float* scores, const int32_t* lens, int batch, int qo_len,
                        int num_kv_heads, int max_pages, int topk, int32_t* out, int* err,
                        cudaStream_t st);

// KV slot staging of the qo_len verify tokens (k_new / v_new: bf16 [B*T, Hk, D]).
cudaError_t launch_stage_kv(const void* k_new, const void* v_new, void* pool, const int32_t* pt,
                            const int32_t* lens, int batch, int qo_len, int Hk, int D, int max_pages,
                            int num_slots, int stride, bool fp8, float k_scale, float v_scale, int* err,
                            cudaStream_t st);

// Flat (CSR) page table <-> padded table, row bases from the lengths:
// to_flat: src = padded table, dst = flat (indptr may be null);
// else:    src = flat, dst = padded table (indptr unused).
cudaError_t launch_flat_table(bool to_flat, const int32_t* src, const int32_t* lens, int batch,
                              int qo_len, int max_pages, int32_t* dst, int32_t* indptr, int* err,
                              cudaStream_t st);

// Split-KV combine of the cut sequences, launched right after an attention
// kernel with programmatic dependent launch (no-op for a single CTA).
cudaError_t launch_combine(int head_dim, const AttnParams& p, cudaStream_t st);

// Launch with programmatic dependent launch: the kernel may be scheduled while
// the previous kernel of the stream is still running (once that one has
// triggered), and every kernel of the library calls pdl_wait() before it reads
// or writes global memory that the previous kernel may touch.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Raise a kernel's dynamic shared-memory limit once per device.
cudaError_t ensure_smem_attr(const void* func, size_t bytes);

}  // namespace trtv
