// fp32 instances of the decode-attention kernel (CUDA-core arithmetic, no TF32).
#include "attend_impl.cuh"

namespace fastocr {

cudaError_t launch_f32(int head_dim, int mode, const Params& p, cudaStream_t s) {
  switch (head_dim) {
    case 64: return dispatch_mode<float, 64>(mode, p, s);
    case 128: return dispatch_mode<float, 128>(mode, p, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t prepare_f32() {
  cudaError_t e = prepare_all_modes<float, 64>();
  return e != cudaSuccess ? e : prepare_all_modes<float, 128>();
}

int max_cluster_f32(int head_dim, int variant) {
  return head_dim == 64 ? max_cluster_of<float, 64>(variant) : max_cluster_of<float, 128>(variant);
}

// The selection kernel does not depend on the cache dtype; this unit hosts
// its stand-alone launch.
cudaError_t launch_select(const Params& p, cudaStream_t s) { return launch_select_kernel(p, s); }

int active_clusters_f32(int head_dim, int cluster) {
  return head_dim == 64 ? active_clusters<float, 64>(cluster) : active_clusters<float, 128>(cluster);
}

}  // namespace fastocr
