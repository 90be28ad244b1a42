// bf16 instances of the decode-attention kernel (tensor-core GQA contraction).
#include "attend_impl.cuh"

namespace fastocr {

cudaError_t launch_bf16(int head_dim, int mode, const Params& p, cudaStream_t s) {
  switch (head_dim) {
    case 64: return dispatch_mode<__nv_bfloat16, 64>(mode, p, s);
    case 128: return dispatch_mode<__nv_bfloat16, 128>(mode, p, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t prepare_bf16() {
  cudaError_t e = prepare_all_modes<__nv_bfloat16, 64>();
  return e != cudaSuccess ? e : prepare_all_modes<__nv_bfloat16, 128>();
}

int max_cluster_bf16(int head_dim, int variant) {
  return head_dim == 64 ? max_cluster_of<__nv_bfloat16, 64>(variant) : max_cluster_of<__nv_bfloat16, 128>(variant);
}

int active_clusters_bf16(int head_dim, int cluster) {
  return head_dim == 64 ? active_clusters<__nv_bfloat16, 64>(cluster) : active_clusters<__nv_bfloat16, 128>(cluster);
}

}  // namespace fastocr
