// Allocation-free focal-layer entry point (fastocr_focal_attend_noalloc).
//
// Some callers cannot allocate device memory when they call into this
// library: code running inside another allocator's arena, plugins whose
// host forbids cudaMalloc after start-up, or real-time loops that must not
// take the driver's allocation locks. The regular focal call needs a handle
// whose workspace fastocr_create allocates; this variant instead keeps its
// scratch (image logits and per-KV-head scores) in a fixed-size array that
// is part of the library image, so the call itself allocates nothing.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "attend_kernels.cuh"
#include "fastocr.h"

namespace fastocr {
cudaError_t launch_bf16(int head_dim, int mode, const Params& p, cudaStream_t s);
cudaError_t launch_f32(int head_dim, int mode, const Params& p, cudaStream_t s);
cudaError_t prepare_bf16();
cudaError_t prepare_f32();
int max_cluster_bf16(int head_dim, int variant);
int max_cluster_f32(int head_dim, int variant);
int active_clusters_bf16(int head_dim, int cluster);
int active_clusters_f32(int head_dim, int cluster);
}  // namespace fastocr

using namespace fastocr;

namespace {

constexpr size_t kUnitsImg = FASTOCR_NOALLOC_MAX_UNITS_IMG;   // B * H_kv * max_img_tokens
constexpr size_t kScratchFloats = kUnitsImg * (kSlots + 1);   // logits [.., 8] + scores [..]

// Lives on every device that loads the library, until the process exits.
// Host code must not pass this name to a kernel (it is a host-side stand-in);
// the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) float g_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
struct DeviceState {
  bool ready;
  float* scratch;      // device address of g_scratch on this device
  int num_sms;
  int max_cluster[2][2];  // [dtype][head_dim == 128]
  int max_cluster_deep[2][2];
  int active[2][2][kMaxSplits + 1];  // clusters of each size held at once
};
DeviceState g_state[kMaxDevices];
std::mutex g_mutex;

// First call on a device: look up the scratch address and the launch limits.
fastocr_status device_setup(int dev, DeviceState** out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& s = g_state[dev];
  if (!s.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return FASTOCR_ERR_NO_DEVICE;
    if (prop.major != 10 || prop.minor != 3) return FASTOCR_ERR_NO_DEVICE;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || !ptr) return FASTOCR_ERR_CUDA;
    if (prepare_bf16() != cudaSuccess || prepare_f32() != cudaSuccess) return FASTOCR_ERR_CUDA;
    s.scratch = static_cast<float*>(ptr);
    s.num_sms = prop.multiProcessorCount;
    s.max_cluster[FASTOCR_DTYPE_F32][0] = max_cluster_f32(64, kGeneral);
    s.max_cluster[FASTOCR_DTYPE_F32][1] = max_cluster_f32(128, kGeneral);
    s.max_cluster[FASTOCR_DTYPE_BF16][0] = max_cluster_bf16(64, kGeneral);
    s.max_cluster[FASTOCR_DTYPE_BF16][1] = max_cluster_bf16(128, kGeneral);
    s.max_cluster_deep[FASTOCR_DTYPE_F32][0] = max_cluster_f32(64, kDeep);
    s.max_cluster_deep[FASTOCR_DTYPE_F32][1] = max_cluster_f32(128, kDeep);
    s.max_cluster_deep[FASTOCR_DTYPE_BF16][0] = max_cluster_bf16(64, kDeep);
    s.max_cluster_deep[FASTOCR_DTYPE_BF16][1] = max_cluster_bf16(128, kDeep);
    for (int dt = 0; dt < 2; ++dt)
      for (int wide = 0; wide < 2; ++wide)
        for (int c = 1; c <= s.max_cluster[dt][wide]; ++c)
          s.active[dt][wide][c] = dt == FASTOCR_DTYPE_BF16 ? active_clusters_bf16(wide ? 128 : 64, c)
                                                          : active_clusters_f32(wide ? 128 : 64, c);
    s.ready = true;
  }
  *out = &s;
  return FASTOCR_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" fastocr_status fastocr_focal_attend_noalloc(
    const fastocr_dims* dims, const void* q, const fastocr_kv* kv, const int32_t* img_range,
    double tau, void* out, int32_t* idx, int32_t idx_stride, int32_t* k_out, int32_t* status,
    fastocr_stream stream) {
  if (!dims || !q || !kv || !img_range || !out || !idx || !k_out || !status)
    return FASTOCR_ERR_NULL;
  if (!kv->k || !kv->v || !kv->block_table || !kv->seq_len) return FASTOCR_ERR_NULL;
  const fastocr_dims d = *dims;
  if (d.batch < 1 || d.num_q_heads < 1 || d.num_kv_heads < 1 || d.max_pages_per_seq < 1 ||
      d.max_img_tokens < 1 || d.page_size < 1 || d.page_size > 256 || kv->num_pages < 1)
    return FASTOCR_ERR_INVALID;
  if (d.num_q_heads % d.num_kv_heads != 0) return FASTOCR_ERR_INVALID;
  if (d.dtype != FASTOCR_DTYPE_F32 && d.dtype != FASTOCR_DTYPE_BF16) return FASTOCR_ERR_INVALID;
  int log2_page = 0;
  while ((1 << log2_page) < d.page_size) ++log2_page;
  if ((1 << log2_page) != d.page_size) return FASTOCR_ERR_INVALID;
  if (!(tau > 0.0 && tau <= 1.0)) return FASTOCR_ERR_INVALID;
  if (idx_stride < keep_count(tau, d.max_img_tokens)) return FASTOCR_ERR_INVALID;
  if (d.num_q_heads / d.num_kv_heads > kSlots) return FASTOCR_ERR_UNSUPPORTED;
  if (d.head_dim != 64 && d.head_dim != 128) return FASTOCR_ERR_UNSUPPORTED;
  if (d.max_img_tokens > kMaxImg) return FASTOCR_ERR_UNSUPPORTED;
  if ((long long)d.max_pages_per_seq * d.page_size >= (1LL << 30)) return FASTOCR_ERR_UNSUPPORTED;
  if ((long long)kv->num_pages * d.num_kv_heads * d.page_size >= (1LL << 31))
    return FASTOCR_ERR_UNSUPPORTED;
  // the fixed scratch bounds the problem size
  if ((unsigned long long)d.batch * d.num_kv_heads * d.max_img_tokens > kUnitsImg)
    return FASTOCR_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(out) || !aligned16(kv->k) || !aligned16(kv->v))
    return FASTOCR_ERR_ALIGN;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return FASTOCR_ERR_NO_DEVICE;
  DeviceState* st = nullptr;
  fastocr_status s = device_setup(dev, &st);
  if (s != FASTOCR_OK) return s;

  const size_t units_img = (size_t)d.batch * d.num_kv_heads * d.max_img_tokens;
  Params p;
  memset(&p, 0, sizeof(p));
  p.q = q;
  p.out = out;
  p.k = kv->k;
  p.v = kv->v;
  p.block_table = kv->block_table;
  p.seq_len = kv->seq_len;
  p.num_pages = kv->num_pages;
  p.max_pages = d.max_pages_per_seq;
  p.log2_page = log2_page;
  p.B = d.batch;
  p.Hq = d.num_q_heads;
  p.Hkv = d.num_kv_heads;
  p.g = d.num_q_heads / d.num_kv_heads;
  p.img_range = img_range;
  p.tau = tau;
  p.idx_out = idx;
  p.idx_stride = idx_stride;
  p.k_out = k_out;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d.head_dim));
  // every logit and score the kernels read is written earlier in the same
  // call, so the scratch needs no clearing between calls
  p.logits = st->scratch;
  p.sigma_part = st->scratch + units_img * kSlots;
  p.sel_src = p.sigma_part;   // the selection sums the KV heads' score shares
  p.sel_heads = d.num_kv_heads;
  p.sel_head_stride = d.max_img_tokens;
  p.sel_batch_stride = (long)d.num_kv_heads * d.max_img_tokens;
  p.profile = nullptr;
  p.profile_layer = -1;
  p.status = status;
  p.max_img = d.max_img_tokens;
  // same split rule as fastocr_focal_attend on a handle without a length hint
  const int wide = d.head_dim == 128 ? 1 : 0;
  p.splits = choose_splits((long)d.batch * d.num_kv_heads, (long)d.max_pages_per_seq << log2_page,
                           st->max_cluster[d.dtype][wide], st->active[d.dtype][wide],
                           st->num_sms);
  p.pdl_early = (long)p.splits * p.Hkv * p.B <= st->num_sms;
  p.variant = 2L * p.splits * p.Hkv * p.B <= st->num_sms &&
                      p.splits <= st->max_cluster_deep[d.dtype][wide]
                  ? kDeep
                  : kGeneral;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const cudaError_t e = d.dtype == FASTOCR_DTYPE_BF16 ? launch_bf16(d.head_dim, kFocal, p, cs)
                                                      : launch_f32(d.head_dim, kFocal, p, cs);
  return e == cudaSuccess ? FASTOCR_OK : FASTOCR_ERR_CUDA;
}
