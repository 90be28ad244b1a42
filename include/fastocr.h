/*
 * fastocr.h -- C ABI of libfastocr.so: decode attention of FastOCR
 * (focal layers with image-token selection, non-focal gather attention,
 * Cross-Step Fixation Reuse) and of R-SWA, over a paged, never-evicted
 * KV cache, on one NVIDIA GB300 (sm_103a).
 *
 * Sources:
 *  [FGP]   FastOCR: Dynamic Visual Fixation via KV Cache Pruning for Efficient
 *          Document Parsing -- technical summary (gist.science), section
 *          "Focal-Guided Pruning": focal layers attend to the full KV cache and
 *          pick the most-attended image tokens at keep ratio tau; the
 *          selection is propagated to every non-focal layer, which attends only
 *          to the pruned set. Focal layers are found by profiling each layer's
 *          image-attention ratio over a warm-up of w steps.
 *  [CSFR]  same page, section "Cross-Step Fixation Reuse": non-focal layers
 *          before the first focal layer start from F_last, the previous step's
 *          selection of the deepest focal layer.
 *  [RSWA]  Unlimited OCR summary (my-wiki-6fu.pages.dev), R-SWA paragraph:
 *          attention limited to a global prefix (visual + prompt tokens) and a
 *          causal sliding window of width n (default 128) over generated text.
 *  [ABS]   FastOCR abstract: the full cache is kept; which tokens are attended
 *          changes per step (no eviction).
 *
 * Conventions shared by every call
 * --------------------------------
 *  B sequences, H_q query heads, H_kv KV heads (H_q % H_kv == 0 and
 *  g = H_q / H_kv <= 8), head dimension d (64 or 128). Query head h reads
 *  KV head h / g. Softmax scale 1/sqrt(d).
 *  dtype: FASTOCR_DTYPE_BF16 (q, K, V, out in bf16; fp32 accumulation) or
 *         FASTOCR_DTYPE_F32 (all fp32, CUDA-core arithmetic, no TF32).
 *  q, out:        [B, H_q, d] contiguous, device memory, caller-owned.
 *  K, V caches:   [num_pages, H_kv, page_size, d] contiguous per layer, device.
 *  block_table:   [B, max_pages_per_seq] int32, device; page of token p of
 *                 sequence b is block_table[b][p / page_size], row p % page_size.
 *  seq_len:       [B] int32, device; N_t = tokens in the cache, the current
 *                 decode token included (its K/V already written).
 *  img_range:     [B, 2] int32, device; (start, N_img) of the image tokens.
 *                 Text prefix = [0, start); generated = [start + N_img, N_t).
 *  Image scores (focal layers) are the probabilities of the layer's softmax
 *  over the whole cache, summed over all H_q query heads; k = ceil(tau*N_img)
 *  (IEEE double, ceil(tau*N_img - 1e-9), clamped to [1, N_img]); ties go to
 *  the lower position; selections are absolute positions, ascending.
 *
 *  Every compute call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *  legacy default stream), allocates nothing and never synchronises, so a
 *  sequence of calls can be captured in a CUDA graph. Calls that share a
 *  handle must be ordered (one stream, or events): the handle's workspace is
 *  reused by every call.
 *
 *  Overlap with the preceding kernel: the kernels are launched with
 *  programmatic dependent launch, so they may start while the kernel before
 *  them on `stream` is still running. Until that kernel has completed they
 *  read only seq_len, block_table, img_range and the K/V rows (and their
 *  block-table entries) of positions below N_t - 1; q, the selection (idx,
 *  k) and the current token's K/V row are read after it completes. So the
 *  former must be written before the kernel preceding the call starts -- in
 *  a decode step they are set once before the first layer -- while q, the
 *  selection and the current token may come from the kernel right before.
 *  One exception: a gather (sparse) call stages the rows of the selection it
 *  expects before that kernel completes, so if img_range contains the
 *  current token N_t - 1 (the image normally ends before the generated
 *  text), that token's K/V must be written before the preceding kernel
 *  starts as well. fastocr_sparse_attend_ex's flags change when the
 *  selection is read: FASTOCR_SELECTION_FINAL reads it only before the wait,
 *  FASTOCR_SELECTION_PENDING (large grids) only after it.
 *
 *  Errors: argument errors are detected on the host and returned as a
 *  negative status before anything is launched. Faults in device data (page
 *  id out of range, seq_len above capacity, selection outside the image,
 *  bad image range) never trap: the kernel masks the offending token, ORs a
 *  FASTOCR_DEV_* bit into the handle's device status word and goes on;
 *  read and clear it with fastocr_device_status().
 */
#ifndef FASTOCR_H
#define FASTOCR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 2 adds fastocr_focal_scores, fastocr_select, fastocr_set_variant,
 * fastocr_read_probe, fastocr_copy, fastocr_profile_attend,
 * fastocr_profiler_read / fastocr_profiler_load and fastocr_sparse_attend_ex
 * to version 1; no call of version 1 changed. */
#define FASTOCR_ABI_VERSION 2

typedef struct fastocr_handle fastocr_handle;
typedef void* fastocr_stream; /* cudaStream_t */

typedef enum {
  FASTOCR_OK = 0,
  FASTOCR_ERR_NULL = -1,        /* a required pointer is NULL */
  FASTOCR_ERR_INVALID = -2,     /* a size / ratio / layer id is out of range */
  FASTOCR_ERR_UNSUPPORTED = -3, /* shape outside what the kernels implement */
  FASTOCR_ERR_CUDA = -4,        /* a CUDA runtime call failed */
  FASTOCR_ERR_NO_DEVICE = -5,   /* no usable sm_103 device */
  FASTOCR_ERR_ALIGN = -6        /* a device pointer is not 16-byte aligned */
} fastocr_status;

typedef enum { FASTOCR_DTYPE_F32 = 0, FASTOCR_DTYPE_BF16 = 1 } fastocr_dtype;

/* Device status bits (fastocr_device_status). */
#define FASTOCR_DEV_BAD_PAGE 1      /* block_table entry outside [0, num_pages) */
#define FASTOCR_DEV_BAD_SEQLEN 2    /* seq_len < 1 or above max_pages_per_seq*page_size */
#define FASTOCR_DEV_BAD_IMG 4       /* img_range outside [0, N_t) */
#define FASTOCR_DEV_BAD_SELECTION 8 /* selected position outside the image, or k > N_img */
#define FASTOCR_DEV_INTERNAL 16     /* a kernel-internal consistency check failed (a library bug) */

/* Shapes fixed for the life of a handle. */
typedef struct {
  int32_t batch;             /* B >= 1 */
  int32_t num_q_heads;       /* H_q */
  int32_t num_kv_heads;      /* H_kv; H_q % H_kv == 0, H_q / H_kv <= 8 */
  int32_t head_dim;          /* d: 64 or 128 */
  int32_t dtype;             /* fastocr_dtype */
  int32_t page_size;         /* tokens per page: power of two, 1..256 */
  int32_t max_pages_per_seq; /* columns of block_table */
  int32_t max_img_tokens;    /* upper bound of N_img (<= 16384); 0 if no focal calls */
  int32_t num_layers;        /* profiler slots (>= 1) */
} fastocr_dims;

/* One layer's KV cache (all pointers device memory, caller-owned). */
typedef struct {
  const void* k;              /* [num_pages, H_kv, page_size, d] */
  const void* v;              /* [num_pages, H_kv, page_size, d] */
  const int32_t* block_table; /* [B, max_pages_per_seq] */
  const int32_t* seq_len;     /* [B] */
  int32_t num_pages;          /* pages in k and v (bounds check) */
} fastocr_kv;

/* Library and ABI version; never fails, needs no GPU. */
int32_t fastocr_abi_version(void);

/* Human-readable text of a fastocr_status; never NULL, needs no GPU. */
const char* fastocr_status_string(int32_t status);

/* Create a handle for the current CUDA device: checks dims, allocates the
 * workspace (focal-layer image logits, per-KV-head image scores, profiler
 * accumulator, device status word) once; split partials never leave the
 * chip (they merge in distributed shared memory). *out is set only on FASTOCR_OK.
 * Synchronous. Errors: NULL, INVALID, UNSUPPORTED, NO_DEVICE, CUDA. */
fastocr_status fastocr_create(const fastocr_dims* dims, fastocr_handle** out);

/* Free the handle and its workspace (synchronises the device first).
 * NULL is accepted and ignored. */
fastocr_status fastocr_destroy(fastocr_handle* h);

/* Full decode attention over [0, N_t) for every sequence -- the dense / tau=1
 * baseline layer. [FGP] (what focal layers compute, without selection). */
fastocr_status fastocr_full_attend(fastocr_handle* h, const void* q, const fastocr_kv* kv,
                                   void* out, fastocr_stream stream);

/* Focal layer [FGP]: full decode attention over [0, N_t), image scores
 * (head-summed probabilities of image tokens), and the top
 * k_b = ceil(tau*N_img_b) image tokens of every sequence, written to
 * idx[b*idx_stride + 0 .. k_b-1] as ascending absolute positions, with k_b in
 * k_out[b]. Scoring and selection run on the device (no host round trip).
 * tau in (0, 1]; idx_stride >= ceil(tau*max_img_tokens). Two kernels run
 * back to back on `stream`: the attention (which also leaves each KV head's
 * share of the image scores in the workspace) and the selection.
 * profile_layer >= 0 (< num_layers) adds the image probability mass summed
 * over sequences and query heads to that layer's profiler slot (warm-up);
 * -1 disables profiling. */
fastocr_status fastocr_focal_attend(fastocr_handle* h, const void* q, const fastocr_kv* kv,
                                    const int32_t* img_range, double tau, void* out,
                                    int32_t* idx, int32_t idx_stride, int32_t* k_out,
                                    int32_t profile_layer, fastocr_stream stream);

/* Focal-layer profiling without a selection [FGP, focal layer selection]:
 * full decode attention over [0, N_t) (out as fastocr_full_attend), and the
 * image probability mass -- for every sequence and query head, the softmax
 * probability of the layer's full-cache attention summed over the image
 * tokens [start_b, start_b + N_img_b) -- summed into profiler slot
 * profile_layer (0 <= profile_layer < num_layers), the quantity
 * fastocr_focal_attend adds with profile_layer >= 0. One kernel: no image
 * logits, scores or top-k are made. For the warm-up steps whose selections
 * nothing reads (every step of a profiling window but its last, whose
 * selection of the deepest chosen layer becomes F_last). The mass is summed
 * per (sequence, KV head) group and split in double-precision atomics, so
 * its last bits depend on their order; img_range as fastocr_focal_attend
 * (max_img_tokens does not bound it). */
fastocr_status fastocr_profile_attend(fastocr_handle* h, const void* q, const fastocr_kv* kv,
                                      const int32_t* img_range, void* out, int32_t profile_layer,
                                      fastocr_stream stream);

/* Head-sharded focal layer, part 1 [FGP]: what fastocr_focal_attend computes
 * for this handle's heads, without the selection. A sequence's heads may be
 * split over several GPUs (tensor parallelism), each holding whole GQA
 * groups; the image score is a sum over all query heads, so each GPU's share
 * must be summed (an all-reduce) before the top-k, which fastocr_select then
 * takes. Writes out (this handle's H_q heads) and sigma[b*sigma_stride + i],
 * i < N_img_b: the image probabilities of token start_b + i summed over this
 * handle's query heads (fp32, device, caller-owned; sigma_stride >=
 * max_img_tokens). Entries at and beyond N_img_b are not written. */
fastocr_status fastocr_focal_scores(fastocr_handle* h, const void* q, const fastocr_kv* kv,
                                    const int32_t* img_range, void* out, float* sigma,
                                    int32_t sigma_stride, fastocr_stream stream);

/* Head-sharded focal layer, part 2 [FGP]: the top k_b = ceil(tau*N_img_b) of
 * the scores sigma[b*sigma_stride + i], i < N_img_b (any non-negative fp32
 * values, e.g. fastocr_focal_scores shares summed over all GPUs), ties to the
 * lower position, written like fastocr_focal_attend's selection to
 * idx[b*idx_stride ..] (ascending absolute positions) and k_out[b]. Reads
 * kv->seq_len and img_range only (other kv fields may be NULL). Every GPU
 * that passes the same scores gets the same selection. One kernel on stream;
 * tau in (0, 1]; idx_stride >= ceil(tau*max_img_tokens). */
fastocr_status fastocr_select(fastocr_handle* h, const fastocr_kv* kv, const int32_t* img_range,
                              const float* sigma, int32_t sigma_stride, double tau, int32_t* idx,
                              int32_t idx_stride, int32_t* k_out, fastocr_stream stream);

/* Non-focal layer [FGP, CSFR]: attention over the text prefix [0, start),
 * the k[b] selected image positions idx[b*idx_stride + 0 .. k[b]-1] (any
 * order, each inside the image range), and the generated tokens
 * [start + N_img, N_t). Passing F_last (the previous step's selection of the
 * deepest focal layer) here is Cross-Step Fixation Reuse. A k[b] outside
 * [0, min(N_img, idx_stride)] or a position outside the image range is
 * reported as FASTOCR_DEV_BAD_SELECTION and clamped / masked. */
fastocr_status fastocr_sparse_attend(fastocr_handle* h, const void* q, const fastocr_kv* kv,
                                     const int32_t* img_range, const int32_t* idx,
                                     int32_t idx_stride, const int32_t* k, void* out,
                                     fastocr_stream stream);

/* fastocr_sparse_attend with flags (0 = the call above). FASTOCR_SELECTION_FINAL:
 * the caller guarantees that idx and k were written before the kernel
 * preceding this call on `stream` began (e.g. a gather layer that is not the
 * first after the focal layer whose selection it uses: the selection kernel
 * is then two or more launches back, and programmatic dependent launch lets
 * a kernel start only once the one before its predecessor has completed).
 * The kernel then takes the selection it reads before the wait as final and
 * skips re-reading it after the wait (and the CTA barrier that check needs).
 * With the flag set and the guarantee broken, the layer may attend a stale
 * selection; nothing faults. FASTOCR_SELECTION_PENDING: a hint that the kernel
 * right before this call writes idx and k (e.g. the selection of the focal
 * layer just before): large grids then stage only the text before the wait
 * and lay the selection out after it, instead of staging the selection they
 * read early, which would be the previous one, and redoing it; small grids
 * (whole lists staged early) ignore it. Results do not depend on it. Both
 * flags, or any other bit: FASTOCR_ERR_INVALID. */
#define FASTOCR_SELECTION_FINAL 1u
#define FASTOCR_SELECTION_PENDING 2u
fastocr_status fastocr_sparse_attend_ex(fastocr_handle* h, const void* q, const fastocr_kv* kv,
                                        const int32_t* img_range, const int32_t* idx,
                                        int32_t idx_stride, const int32_t* k, void* out,
                                        uint32_t flags, fastocr_stream stream);

/* R-SWA layer [RSWA]: attention over [0, prefix_len) and the last `window`
 * tokens of [prefix_len, N_t), the current token included. prefix_len >= 0,
 * window >= 0. */
fastocr_status fastocr_rswa_attend(fastocr_handle* h, const void* q, const fastocr_kv* kv,
                                   int32_t prefix_len, int32_t window, void* out,
                                   fastocr_stream stream);

/* Zero the profiler accumulator of every layer (asynchronous on stream). */
fastocr_status fastocr_profiler_reset(fastocr_handle* h, fastocr_stream stream);

/* Focal layer selection [FGP]: read the accumulated image-attention mass of
 * every layer (synchronises `stream`), write the n_focal layers with the
 * largest mass (ties: lower layer id) in ascending order to layers_out
 * (host, n_focal entries) and, if ratio_out is not NULL, the mass of every
 * layer to ratio_out (host, num_layers entries). 1 <= n_focal <= num_layers. */
fastocr_status fastocr_profiler_select(fastocr_handle* h, int32_t n_focal, int32_t* layers_out,
                                       double* ratio_out, fastocr_stream stream);

/* Checkpoint and resume of the warm-up profile [FGP]: copy the accumulated
 * image-attention mass of every layer to mass_out (host, num_layers doubles;
 * synchronises `stream`), or load it from mass_in (host, num_layers doubles;
 * the copy is complete when the call returns). Together with the focal set C
 * and the F_last selection, which the caller owns, this is the whole state
 * the method carries between decode steps. */
fastocr_status fastocr_profiler_read(fastocr_handle* h, double* mass_out, fastocr_stream stream);
fastocr_status fastocr_profiler_load(fastocr_handle* h, const double* mass_in,
                                     fastocr_stream stream);

/* Read the device status word (FASTOCR_DEV_* bits, 0 = clean) into *status
 * (host) and clear it. Synchronises `stream`. */
fastocr_status fastocr_device_status(fastocr_handle* h, int32_t* status, fastocr_stream stream);

/* Tell the handle the cache length N_t (tokens per sequence, the largest in
 * the batch) that the coming calls will see; 0 clears the hint. Only the
 * choice of the split-K factor uses it (without a hint it assumes a full
 * cache of max_pages_per_seq*page_size tokens); results do not depend on it,
 * and a wrong hint only costs speed. A call captured in a CUDA graph keeps
 * the split factor chosen at capture. */
fastocr_status fastocr_set_length_hint(fastocr_handle* h, int32_t n_t);

/* Override the split-K factor of a mode (0 = full/focal, 1 = sparse,
 * 2 = R-SWA); 0 restores the automatic choice. Splits are clamped to
 * [1, 16] (the splits of one sequence and KV head form one thread-block
 * cluster) and to the largest cluster the device co-schedules. */
fastocr_status fastocr_set_splits(fastocr_handle* h, int32_t mode, int32_t splits);

/* Measurement utility, not a step of the method: read `bytes` (a multiple
 * of 16, >= 16) of device memory at `src` (16-byte aligned) exactly once with
 * streaming loads that bypass L1, in one kernel on `stream`, folding the data
 * into a value that may be ORed into *sink (device uint32, caller-owned; its
 * content is meaningless). Timed with events around it on a buffer much
 * larger than L2, it gives the read-only HBM bandwidth that bounds the attend
 * kernels, which only read the K/V cache. Asynchronous; allocates nothing.
 * Errors: NULL, INVALID (size), ALIGN, NO_DEVICE, CUDA. */
fastocr_status fastocr_read_probe(const void* src, int64_t bytes, uint32_t* sink,
                                  fastocr_stream stream);

/* Data-movement utility, not a step of the method: copy `bytes` (a multiple
 * of 16, >= 0) from src to dst (both 16-byte aligned, not overlapping) with
 * the SMs, in one kernel on `stream`. It is launched with programmatic
 * dependent launch: it waits for the kernel before it to complete before it
 * reads src or writes dst, and lets the next kernel start its pre-wait work
 * while it copies (the attend kernels read their q only after their wait).
 * Either pointer may be device memory, managed memory or page-locked host
 * memory (cudaHostAlloc or cudaHostRegister), which the SMs address through
 * unified addressing -- over NVLink-C2C on a Grace-Blackwell node, where this
 * moves a step's queries in faster than a copy engine and without the
 * launch gap a copy node leaves before the next kernel. Pageable host memory
 * is refused. The caller guarantees that [ptr, ptr + bytes) lies inside each
 * allocation. Asynchronous; allocates nothing.
 * Errors: NULL, INVALID (size, overlap, memory the device cannot address),
 * ALIGN, NO_DEVICE, CUDA. */
fastocr_status fastocr_copy(void* dst, const void* src, int64_t bytes, fastocr_stream stream);

/* Override the kernel variant of a mode (0 = full/focal, 1 = sparse,
 * 2 = R-SWA): 0 = automatic (default), 1 = general (6 warps of 2 stages, two
 * CTAs an SM), 2 = deep (4 warps of 6 stages, one CTA an SM). Results do not
 * depend on it (up to summation order); it exists for tuning and testing.
 * Returns UNSUPPORTED for a variant whose shared memory does not fit this
 * handle's dtype and head size. */
fastocr_status fastocr_set_variant(fastocr_handle* h, int32_t mode, int32_t variant);

/* Allocation-free focal layer. The pages describe no such call; it exists
 * for callers that may not allocate GPU memory at the point where they run
 * attention -- for example code living inside another framework's memory
 * pool, plugins whose host forbids cudaMalloc once started, or latency-
 * critical loops that must not take the driver's allocation locks. It needs
 * no handle: it computes exactly what fastocr_focal_attend computes (same
 * kernels, same split rule, profiling off) but keeps its scratch -- the image
 * logits and per-KV-head scores -- in one fixed array of
 * FASTOCR_NOALLOC_MAX_UNITS_IMG * 9 floats (about 2.4 MB) compiled into the
 * library, which every GPU that loads the library holds until the process
 * exits. It calls no cudaMalloc or cudaFree and no allocating library
 * routine.
 *
 * dims: shapes as for fastocr_create (num_layers is ignored); the problem
 * must satisfy batch * num_kv_heads * max_img_tokens <=
 * FASTOCR_NOALLOC_MAX_UNITS_IMG, otherwise the call returns
 * FASTOCR_ERR_UNSUPPORTED without launching anything. q, kv, img_range, tau,
 * out, idx, idx_stride, k_out: as for fastocr_focal_attend. status: device
 * int32 the kernels OR FASTOCR_DEV_* bits into (the caller clears it).
 *
 * The first call on a device sets that device up (looks up the device
 * address of the fixed array with cudaGetSymbolAddress, raises the kernels'
 * shared-memory limits, reads the SM count); make that first call outside
 * any stream capture. Every call on a device uses the same array and leaves
 * its contents behind; nothing in it needs clearing because each call writes
 * every value it later reads. Calls whose executions overlap on the GPU
 * (different streams, or several host threads) race on the array: order
 * them. */
#define FASTOCR_NOALLOC_MAX_UNITS_IMG 65536
fastocr_status fastocr_focal_attend_noalloc(const fastocr_dims* dims, const void* q,
                                            const fastocr_kv* kv, const int32_t* img_range,
                                            double tau, void* out, int32_t* idx,
                                            int32_t idx_stride, int32_t* k_out, int32_t* status,
                                            fastocr_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* FASTOCR_H */
