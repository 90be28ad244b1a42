// C ABI of libfastocr.so (declared in include/fastocr.h): argument checking,
// the workspace, split-K sizing and kernel dispatch. Host code only.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "attend_kernels.cuh"
#include "fastocr.h"

namespace fastocr {
cudaError_t launch_bf16(int head_dim, int mode, const Params& p, cudaStream_t s);
cudaError_t launch_f32(int head_dim, int mode, const Params& p, cudaStream_t s);
cudaError_t launch_select(const Params& p, cudaStream_t s);
cudaError_t prepare_bf16();
cudaError_t prepare_f32();
int max_cluster_bf16(int head_dim, int variant);
int max_cluster_f32(int head_dim, int variant);
int active_clusters_bf16(int head_dim, int cluster);
int active_clusters_f32(int head_dim, int cluster);
}  // namespace fastocr

using namespace fastocr;

struct fastocr_handle {
  fastocr_dims dims;
  int device;
  int num_sms;
  int log2_page;
  int split_override[3];
  int variant_override[3];      // 0: automatic, else Variant + 1
  int max_splits;   // largest thread-block cluster the device co-schedules (<= 16)
  int max_splits_v[kNumVariants];   // same per variant (0: the variant does not exist)
  int active[kMaxSplits + 1];   // clusters of each size the device holds at once
  long len_hint;    // caller's N_t of the coming calls (0: unknown), split choice only
  void* ws;
  size_t ws_bytes;
  float* logits;
  float* sigma_part;
  double* profile;
  int32_t* status;
};

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int ilog2_exact(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return (1 << l) == x ? l : -1;
}

int slot_of(int mode) { return mode == kSparse ? 1 : (mode == kRswa ? 2 : 0); }

// Kernel variant and split count of a launch whose attend lists hold about
// `len` entries per (sequence, KV head) unit; caller overrides win.
void plan_launch(const fastocr_handle* h, int mode, long len, Params& p) {
  const int slot = slot_of(mode);
  const long units = (long)h->dims.batch * h->dims.num_kv_heads;
  if (len < 1) len = 1;
  int v = h->variant_override[slot] - 1;   // -1: automatic
  int s = h->split_override[slot];         // 0: automatic
  if (s == 0) s = choose_splits(units, len, h->max_splits, h->active, h->num_sms);
  // grids that leave room for the next kernel's CTAs at one CTA per SM take
  // the deeper pipeline (more of each CTA's tiles staged before the wait)
  if (v < 0)
    v = (2L * s * units <= h->num_sms && s <= h->max_splits_v[kDeep]) ? kDeep : kGeneral;
  p.variant = v;
  p.splits = std::max(1, std::min(s, h->max_splits_v[v]));
  // small grids release the next kernel right away (its CTAs then prefetch
  // while this one runs); grids that need the whole GPU release it only
  // after their main loop, so its CTAs do not take slots from this grid
  p.pdl_early = (long)p.splits * units <= h->num_sms;
}

long max_tokens(const fastocr_handle* h) {
  return (long)h->dims.max_pages_per_seq << h->log2_page;
}

// cache length the split choice assumes: the caller's hint, else the capacity
long expected_tokens(const fastocr_handle* h) {
  return h->len_hint > 0 ? std::min(h->len_hint, max_tokens(h)) : max_tokens(h);
}

fastocr_status check_kv(const fastocr_handle* h, const fastocr_kv* kv) {
  if (!kv || !kv->k || !kv->v || !kv->block_table || !kv->seq_len) return FASTOCR_ERR_NULL;
  if (kv->num_pages < 1) return FASTOCR_ERR_INVALID;
  if (!aligned16(kv->k) || !aligned16(kv->v)) return FASTOCR_ERR_ALIGN;
  // cache rows are indexed with 32-bit integers inside the kernels
  if ((long long)kv->num_pages * h->dims.num_kv_heads * h->dims.page_size >= (1LL << 31))
    return FASTOCR_ERR_UNSUPPORTED;
  return FASTOCR_OK;
}

Params base_params(const fastocr_handle* h, const void* q, const fastocr_kv* kv, void* out) {
  Params p;
  memset(&p, 0, sizeof(p));
  const fastocr_dims& d = h->dims;
  p.q = q;
  p.out = out;
  p.k = kv->k;
  p.v = kv->v;
  p.block_table = kv->block_table;
  p.seq_len = kv->seq_len;
  p.num_pages = kv->num_pages;
  p.max_pages = d.max_pages_per_seq;
  p.log2_page = h->log2_page;
  p.B = d.batch;
  p.Hq = d.num_q_heads;
  p.Hkv = d.num_kv_heads;
  p.g = d.num_q_heads / d.num_kv_heads;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d.head_dim));
  p.logits = h->logits;
  p.sigma_part = h->sigma_part;
  p.sel_src = h->sigma_part;   // the selection sums the KV heads' score shares
  p.sel_heads = d.num_kv_heads;
  p.sel_head_stride = d.max_img_tokens;
  p.sel_batch_stride = (long)d.num_kv_heads * d.max_img_tokens;
  p.profile = h->profile;
  p.profile_layer = -1;
  p.status = h->status;
  p.max_img = d.max_img_tokens;
  return p;
}

fastocr_status launch(const fastocr_handle* h, int mode, long len, Params p,
                      fastocr_stream stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  plan_launch(h, mode, len, p);
  cudaError_t e = h->dims.dtype == FASTOCR_DTYPE_BF16 ? launch_bf16(h->dims.head_dim, mode, p, s)
                                                       : launch_f32(h->dims.head_dim, mode, p, s);
  return e == cudaSuccess ? FASTOCR_OK : FASTOCR_ERR_CUDA;
}

}  // namespace

extern "C" {

int32_t fastocr_abi_version(void) { return FASTOCR_ABI_VERSION; }

const char* fastocr_status_string(int32_t status) {
  switch (status) {
    case FASTOCR_OK: return "ok";
    case FASTOCR_ERR_NULL: return "a required pointer is NULL";
    case FASTOCR_ERR_INVALID: return "an argument is out of range";
    case FASTOCR_ERR_UNSUPPORTED: return "shape not supported by the kernels";
    case FASTOCR_ERR_CUDA: return "a CUDA runtime call failed";
    case FASTOCR_ERR_NO_DEVICE: return "no usable sm_103 CUDA device";
    case FASTOCR_ERR_ALIGN: return "a device pointer is not 16-byte aligned";
  }
  return "unknown status";
}

fastocr_status fastocr_create(const fastocr_dims* dims, fastocr_handle** out) {
  if (!dims || !out) return FASTOCR_ERR_NULL;
  const fastocr_dims d = *dims;
  if (d.batch < 1 || d.num_q_heads < 1 || d.num_kv_heads < 1 || d.max_pages_per_seq < 1 ||
      d.num_layers < 1 || d.max_img_tokens < 0 || d.page_size < 1 || d.page_size > 256)
    return FASTOCR_ERR_INVALID;
  if (d.num_q_heads % d.num_kv_heads != 0) return FASTOCR_ERR_INVALID;
  if (d.dtype != FASTOCR_DTYPE_F32 && d.dtype != FASTOCR_DTYPE_BF16) return FASTOCR_ERR_INVALID;
  const int log2_page = ilog2_exact(d.page_size);
  if (log2_page < 0) return FASTOCR_ERR_INVALID;
  if (d.num_q_heads / d.num_kv_heads > kSlots) return FASTOCR_ERR_UNSUPPORTED;
  if (d.head_dim != 64 && d.head_dim != 128) return FASTOCR_ERR_UNSUPPORTED;
  if (d.max_img_tokens > kMaxImg) return FASTOCR_ERR_UNSUPPORTED;
  if ((long long)d.max_pages_per_seq * d.page_size >= (1LL << 30)) return FASTOCR_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FASTOCR_ERR_NO_DEVICE;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return FASTOCR_ERR_NO_DEVICE;
  if (prop.major != 10 || prop.minor != 3) return FASTOCR_ERR_NO_DEVICE;
  if (prepare_bf16() != cudaSuccess || prepare_f32() != cudaSuccess) return FASTOCR_ERR_CUDA;

  const size_t units = (size_t)d.batch * d.num_kv_heads;
  const size_t img = (size_t)d.max_img_tokens;
  size_t off = 0;
  const size_t o_logits = off;
  off = align_up(off + units * img * kSlots * sizeof(float), 256);
  const size_t o_sigma = off;
  off = align_up(off + units * img * sizeof(float), 256);
  const size_t o_zero = off;  // profiler and status: zeroed once here
  const size_t o_profile = off;
  off = align_up(off + (size_t)d.num_layers * sizeof(double), 256);
  const size_t o_status = off;
  off = align_up(off + sizeof(int32_t), 256);

  fastocr_handle* h = static_cast<fastocr_handle*>(calloc(1, sizeof(fastocr_handle)));
  if (!h) return FASTOCR_ERR_CUDA;
  h->dims = d;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  h->log2_page = log2_page;
  for (int v = 0; v < kNumVariants; ++v)
    h->max_splits_v[v] = d.dtype == FASTOCR_DTYPE_BF16 ? max_cluster_bf16(d.head_dim, v)
                                                       : max_cluster_f32(d.head_dim, v);
  h->max_splits = h->max_splits_v[kGeneral];
  for (int c = 1; c <= h->max_splits; ++c)
    h->active[c] = d.dtype == FASTOCR_DTYPE_BF16 ? active_clusters_bf16(d.head_dim, c)
                                                 : active_clusters_f32(d.head_dim, c);
  h->ws_bytes = off;
  if (cudaMalloc(&h->ws, off) != cudaSuccess) {
    free(h);
    return FASTOCR_ERR_CUDA;
  }
  char* base = static_cast<char*>(h->ws);
  h->logits = reinterpret_cast<float*>(base + o_logits);
  h->sigma_part = reinterpret_cast<float*>(base + o_sigma);
  h->profile = reinterpret_cast<double*>(base + o_profile);
  h->status = reinterpret_cast<int32_t*>(base + o_status);
  if (cudaMemset(base + o_zero, 0, off - o_zero) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(h->ws);
    free(h);
    return FASTOCR_ERR_CUDA;
  }
  *out = h;
  return FASTOCR_OK;
}

fastocr_status fastocr_destroy(fastocr_handle* h) {
  if (!h) return FASTOCR_OK;
  cudaError_t e = cudaDeviceSynchronize();
  cudaError_t f = cudaFree(h->ws);
  free(h);
  return (e == cudaSuccess && f == cudaSuccess) ? FASTOCR_OK : FASTOCR_ERR_CUDA;
}

fastocr_status fastocr_full_attend(fastocr_handle* h, const void* q, const fastocr_kv* kv,
                                   void* out, fastocr_stream stream) {
  if (!h || !q || !out) return FASTOCR_ERR_NULL;
  fastocr_status st = check_kv(h, kv);
  if (st != FASTOCR_OK) return st;
  if (!aligned16(q) || !aligned16(out)) return FASTOCR_ERR_ALIGN;
  Params p = base_params(h, q, kv, out);
  return launch(h, kFull, expected_tokens(h), p, stream);
}

fastocr_status fastocr_focal_attend(fastocr_handle* h, const void* q, const fastocr_kv* kv,
                                    const int32_t* img_range, double tau, void* out,
                                    int32_t* idx, int32_t idx_stride, int32_t* k_out,
                                    int32_t profile_layer, fastocr_stream stream) {
  if (!h || !q || !out || !img_range || !idx || !k_out) return FASTOCR_ERR_NULL;
  fastocr_status st = check_kv(h, kv);
  if (st != FASTOCR_OK) return st;
  if (!aligned16(q) || !aligned16(out)) return FASTOCR_ERR_ALIGN;
  if (!(tau > 0.0 && tau <= 1.0)) return FASTOCR_ERR_INVALID;
  if (h->dims.max_img_tokens < 1) return FASTOCR_ERR_INVALID;
  if (idx_stride < keep_count(tau, h->dims.max_img_tokens)) return FASTOCR_ERR_INVALID;
  if (profile_layer < -1 || profile_layer >= h->dims.num_layers) return FASTOCR_ERR_INVALID;
  Params p = base_params(h, q, kv, out);
  p.img_range = img_range;
  p.tau = tau;
  p.idx_out = idx;
  p.idx_stride = idx_stride;
  p.k_out = k_out;
  p.profile_layer = profile_layer;
  return launch(h, kFocal, expected_tokens(h), p, stream);
}

fastocr_status fastocr_profile_attend(fastocr_handle* h, const void* q, const fastocr_kv* kv,
                                      const int32_t* img_range, void* out, int32_t profile_layer,
                                      fastocr_stream stream) {
  if (!h || !q || !out || !img_range) return FASTOCR_ERR_NULL;
  fastocr_status st = check_kv(h, kv);
  if (st != FASTOCR_OK) return st;
  if (!aligned16(q) || !aligned16(out)) return FASTOCR_ERR_ALIGN;
  if (profile_layer < 0 || profile_layer >= h->dims.num_layers) return FASTOCR_ERR_INVALID;
  Params p = base_params(h, q, kv, out);
  p.img_range = img_range;
  p.profile_layer = profile_layer;
  return launch(h, kProfile, expected_tokens(h), p, stream);
}

fastocr_status fastocr_focal_scores(fastocr_handle* h, const void* q, const fastocr_kv* kv,
                                    const int32_t* img_range, void* out, float* sigma,
                                    int32_t sigma_stride, fastocr_stream stream) {
  if (!h || !q || !out || !img_range || !sigma) return FASTOCR_ERR_NULL;
  fastocr_status st = check_kv(h, kv);
  if (st != FASTOCR_OK) return st;
  if (!aligned16(q) || !aligned16(out)) return FASTOCR_ERR_ALIGN;
  if (h->dims.max_img_tokens < 1 || sigma_stride < h->dims.max_img_tokens)
    return FASTOCR_ERR_INVALID;
  Params p = base_params(h, q, kv, out);
  p.img_range = img_range;
  p.tau = 1.0;
  p.sigma_out = sigma;
  p.sigma_stride = sigma_stride;
  return launch(h, kFocal, expected_tokens(h), p, stream);
}

fastocr_status fastocr_select(fastocr_handle* h, const fastocr_kv* kv, const int32_t* img_range,
                              const float* sigma, int32_t sigma_stride, double tau, int32_t* idx,
                              int32_t idx_stride, int32_t* k_out, fastocr_stream stream) {
  if (!h || !kv || !kv->seq_len || !img_range || !sigma || !idx || !k_out)
    return FASTOCR_ERR_NULL;
  if (!(tau > 0.0 && tau <= 1.0)) return FASTOCR_ERR_INVALID;
  if (h->dims.max_img_tokens < 1 || sigma_stride < h->dims.max_img_tokens)
    return FASTOCR_ERR_INVALID;
  if (idx_stride < keep_count(tau, h->dims.max_img_tokens)) return FASTOCR_ERR_INVALID;
  Params p;
  memset(&p, 0, sizeof(p));
  p.seq_len = kv->seq_len;
  p.max_pages = h->dims.max_pages_per_seq;
  p.log2_page = h->log2_page;
  p.B = h->dims.batch;
  p.img_range = img_range;
  p.tau = tau;
  p.idx_out = idx;
  p.idx_stride = idx_stride;
  p.k_out = k_out;
  p.sel_src = sigma;
  p.sel_heads = 1;
  p.sel_head_stride = 0;
  p.sel_batch_stride = sigma_stride;
  p.profile_layer = -1;
  p.status = h->status;
  p.max_img = h->dims.max_img_tokens;
  return launch_select(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FASTOCR_OK
                                                                            : FASTOCR_ERR_CUDA;
}

fastocr_status fastocr_sparse_attend_ex(fastocr_handle* h, const void* q, const fastocr_kv* kv,
                                        const int32_t* img_range, const int32_t* idx,
                                        int32_t idx_stride, const int32_t* k, void* out,
                                        uint32_t flags, fastocr_stream stream) {
  if (!h || !q || !out || !img_range || !idx || !k) return FASTOCR_ERR_NULL;
  fastocr_status st = check_kv(h, kv);
  if (st != FASTOCR_OK) return st;
  if (!aligned16(q) || !aligned16(out)) return FASTOCR_ERR_ALIGN;
  const uint32_t known = FASTOCR_SELECTION_FINAL | FASTOCR_SELECTION_PENDING;
  if (idx_stride < 1 || (flags & ~known) || (flags & known) == known) return FASTOCR_ERR_INVALID;
  Params p = base_params(h, q, kv, out);
  p.img_range = img_range;
  p.idx = idx;
  p.idx_stride = idx_stride;
  p.k_in = k;
  p.sel_final = (flags & FASTOCR_SELECTION_FINAL) ? 1 : 0;
  p.sel_pending = (flags & FASTOCR_SELECTION_PENDING) ? 1 : 0;
  // text tokens (cache minus the image) plus at most idx_stride selected ones
  const long text = std::max(0L, expected_tokens(h) - (long)h->dims.max_img_tokens);
  return launch(h, kSparse, std::min(expected_tokens(h), text + idx_stride), p, stream);
}

fastocr_status fastocr_sparse_attend(fastocr_handle* h, const void* q, const fastocr_kv* kv,
                                     const int32_t* img_range, const int32_t* idx,
                                     int32_t idx_stride, const int32_t* k, void* out,
                                     fastocr_stream stream) {
  return fastocr_sparse_attend_ex(h, q, kv, img_range, idx, idx_stride, k, out, 0u, stream);
}

fastocr_status fastocr_rswa_attend(fastocr_handle* h, const void* q, const fastocr_kv* kv,
                                   int32_t prefix_len, int32_t window, void* out,
                                   fastocr_stream stream) {
  if (!h || !q || !out) return FASTOCR_ERR_NULL;
  fastocr_status st = check_kv(h, kv);
  if (st != FASTOCR_OK) return st;
  if (!aligned16(q) || !aligned16(out)) return FASTOCR_ERR_ALIGN;
  if (prefix_len < 0 || window < 0) return FASTOCR_ERR_INVALID;
  Params p = base_params(h, q, kv, out);
  p.prefix_len = prefix_len;
  p.window = window;
  return launch(h, kRswa, std::min(expected_tokens(h), (long)prefix_len + window), p, stream);
}

fastocr_status fastocr_profiler_reset(fastocr_handle* h, fastocr_stream stream) {
  if (!h) return FASTOCR_ERR_NULL;
  cudaError_t e = cudaMemsetAsync(h->profile, 0, (size_t)h->dims.num_layers * sizeof(double),
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FASTOCR_OK : FASTOCR_ERR_CUDA;
}

fastocr_status fastocr_profiler_select(fastocr_handle* h, int32_t n_focal, int32_t* layers_out,
                                       double* ratio_out, fastocr_stream stream) {
  if (!h || !layers_out) return FASTOCR_ERR_NULL;
  const int L = h->dims.num_layers;
  if (n_focal < 1 || n_focal > L) return FASTOCR_ERR_INVALID;
  std::vector<double> mass(L);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(mass.data(), h->profile, L * sizeof(double), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FASTOCR_ERR_CUDA;
  std::vector<int> order(L);
  for (int l = 0; l < L; ++l) order[l] = l;
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return mass[a] > mass[b]; });  // ties keep lower id first
  std::vector<int> chosen(order.begin(), order.begin() + n_focal);
  std::sort(chosen.begin(), chosen.end());
  for (int i = 0; i < n_focal; ++i) layers_out[i] = chosen[i];
  if (ratio_out)
    for (int l = 0; l < L; ++l) ratio_out[l] = mass[l];
  return FASTOCR_OK;
}

fastocr_status fastocr_profiler_read(fastocr_handle* h, double* mass_out, fastocr_stream stream) {
  if (!h || !mass_out) return FASTOCR_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(mass_out, h->profile, (size_t)h->dims.num_layers * sizeof(double),
                      cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FASTOCR_ERR_CUDA;
  return FASTOCR_OK;
}

fastocr_status fastocr_profiler_load(fastocr_handle* h, const double* mass_in,
                                     fastocr_stream stream) {
  if (!h || !mass_in) return FASTOCR_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // synchronous on the stream: the caller's host array may go away on return
  if (cudaMemcpyAsync(h->profile, mass_in, (size_t)h->dims.num_layers * sizeof(double),
                      cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FASTOCR_ERR_CUDA;
  return FASTOCR_OK;
}

fastocr_status fastocr_device_status(fastocr_handle* h, int32_t* status, fastocr_stream stream) {
  if (!h || !status) return FASTOCR_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, h->status, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemsetAsync(h->status, 0, sizeof(int32_t), s) != cudaSuccess)
    return FASTOCR_ERR_CUDA;
  *status = v;
  return FASTOCR_OK;
}

fastocr_status fastocr_set_length_hint(fastocr_handle* h, int32_t n_t) {
  if (!h) return FASTOCR_ERR_NULL;
  if (n_t < 0) return FASTOCR_ERR_INVALID;
  h->len_hint = n_t;
  return FASTOCR_OK;
}

fastocr_status fastocr_set_splits(fastocr_handle* h, int32_t mode, int32_t splits) {
  if (!h) return FASTOCR_ERR_NULL;
  if (mode < 0 || mode > 2 || splits < 0) return FASTOCR_ERR_INVALID;
  h->split_override[mode] = splits == 0 ? 0 : std::min(std::max(splits, 1), kMaxSplits);
  return FASTOCR_OK;
}

fastocr_status fastocr_set_variant(fastocr_handle* h, int32_t mode, int32_t variant) {
  if (!h) return FASTOCR_ERR_NULL;
  if (mode < 0 || mode > 2 || variant < 0 || variant > kNumVariants) return FASTOCR_ERR_INVALID;
  if (variant > 0 && h->max_splits_v[variant - 1] == 0) return FASTOCR_ERR_UNSUPPORTED;
  h->variant_override[mode] = variant;
  return FASTOCR_OK;
}

}  // extern "C"
