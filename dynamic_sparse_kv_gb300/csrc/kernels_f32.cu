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

int smem_bytes_f32(int head_dim, int max_img) {
  return head_dim == 64 ? attend_smem_bytes<float, 64>(max_img)
                        : attend_smem_bytes<float, 128>(max_img);
}

cudaError_t prepare_f32() {
  cudaError_t e = prepare_all_modes<float, 64>();
  return e != cudaSuccess ? e : prepare_all_modes<float, 128>();
}

}  // namespace fastocr
