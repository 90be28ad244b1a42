// Decode-attention kernels of FastOCR (focal / sparse) and R-SWA for sm_103a.
//
// One kernel template covers every layer kind; they differ only in the
// attend list -- the ordered list of cache positions a query looks at:
//   full   : [0, N_t)                                       (dense / tau = 1)
//   focal  : [0, N_t), plus image-token logits for scoring  (FastOCR,
//            Focal-Guided Pruning: focal layers see the whole cache)
//   sparse : [0, start) ++ selected image positions ++ [start+N_img, N_t)
//            (FastOCR, cross-layer propagation / Cross-Step Fixation Reuse)
//   rswa   : [0, L_m) ++ [max(L_m, N_t - n), N_t)           (Unlimited OCR, R-SWA)
//
// Work decomposition (split-K flash-decode): grid = (splits, H_kv, B); the S
// splits of one (sequence, KV head) form a thread-block cluster. A CTA owns a
// contiguous slice of that KV head's attend list; its warps stream 16-token
// tiles of the slice independently through a cp.async pipeline (6 warps of 2
// stages; 4 warps of 6 stages for grids that leave every CTA an SM of its
// own), in 16-byte chunks into XOR-swizzled rows, so any gathered row is a
// coalesced 256-byte read and ldmatrix is conflict-free; the copies carry an
// L2 evict-first policy (each row is read once). For bf16 the GQA group (g <= 8 query
// heads) x 16 keys contraction and the P.V product run on the tensor cores
// (mma.sync m16n8k16, keys / head dims on M, query heads on N); fp32 runs on
// the CUDA cores. Softmax is online in the base-2 domain with a lazily moved
// running max. The CTAs of a cluster push their partials into each other's
// shared memory and merge after one cluster barrier (no global partials, no
// spin-waits); a single CTA merges its warps straight into the output. In focal mode every CTA also stores its image tokens' logits
// and, after the merge, turns them into its KV head's share of the head-summed
// probabilities; a separate one-CTA-per-sequence kernel, chained by
// programmatic dependent launch, sums the KV heads and radix-selects the top
// k (ties to the lower position) without a host round trip.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fastocr {

constexpr int kTile = 16;      // tokens per warp tile
constexpr int kSlots = 8;      // query-head slots per KV head (g <= 8)
// Kernel variants (warps per CTA x cp.async stages per warp):
//  kGeneral 6 x 2: two CTAs share an SM (one of them typically the next
//           layer's, staging its first tiles); with one CTA of a grid on an SM
//           a warp's tile loop is bound by its own instruction latency, so
//           more warps stream faster, and 12 stages still fit twice per SM.
//  kDeep    4 x 6: one CTA per SM, for grids at most half the SM count; a
//           batch-1 CTA stages its whole share before the wait.
enum Variant : int { kGeneral = 0, kDeep = 1, kNumVariants = 2 };
__host__ __device__ constexpr int stages_of(int v) { return v == kDeep ? 6 : 2; }
__host__ __device__ constexpr int warps_for(int v) { return v == kDeep ? 4 : 6; }
__host__ __device__ constexpr int ctas_per_sm(int v) { return v == kGeneral ? 2 : 1; }
constexpr float kLazyMax = 8.f; // running-max slack (log2 units) before a rescale
constexpr int kMaxSplits = 16;  // = the largest thread-block cluster used
constexpr int kMaxImg = 16384; // image tokens whose scores fit in shared memory

// kProfile: full attention that also adds the layer's image-attention mass
// to the profiler (a warm-up step whose selections are not kept): no logits,
// no scores, no selection kernel.
enum Mode : int { kFull = 0, kFocal = 1, kSparse = 2, kRswa = 3, kProfile = 4 };

// device status bits (same values as FASTOCR_DEV_* in fastocr.h)
constexpr int kDevBadPage = 1;
constexpr int kDevBadSeqLen = 2;
constexpr int kDevBadImg = 4;
constexpr int kDevBadSelection = 8;
constexpr int kDevInternal = 16;   // a cache row outside the cache reached a copy

struct Params {
  const void* q;
  void* out;
  const void* k;
  const void* v;
  const int32_t* block_table;
  const int32_t* seq_len;
  int num_pages, max_pages, log2_page;
  int B, Hq, Hkv, g;
  // index sets
  const int32_t* img_range;  // [B,2] focal / sparse
  const int32_t* idx;        // sparse: selected positions
  int idx_stride;
  const int32_t* k_in;       // sparse: [B]
  int sel_final;             // sparse: idx and k_in were final before the previous kernel began
  int sel_pending;           // sparse: the previous kernel writes idx and k_in (no early staging)
  int32_t* idx_out;          // focal: [B, idx_stride]
  int32_t* k_out;            // focal: [B]
  double tau;
  int prefix_len, window;    // rswa
  int splits;
  float scale_log2;          // log2(e) / sqrt(d)
  // workspace
  float* logits;             // [B, H_kv, max_img, kSlots]
  float* sigma_part;         // [B, H_kv, max_img]
  // selection kernel: the score of image token i of sequence b is
  // sum over c < sel_heads of sel_src[b*sel_batch_stride + c*sel_head_stride + i]
  // (the KV heads' shares in the workspace, or a caller's scores)
  const float* sel_src;
  int sel_heads;
  long sel_head_stride, sel_batch_stride;
  float* sigma_out;          // set: write the summed scores [B, sigma_stride] and select nothing
  int sigma_stride;
  double* profile;           // [num_layers]
  int profile_layer;
  int pdl_early;             // grid fits on the SMs next to the next one: trigger it at once
  int variant;               // host: which Variant to launch
  int32_t* status;
  int max_img;
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous copy global -> shared (zero-filled past src_bytes),
// with an L2 cache policy (from createpolicy).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes,
                                               uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;\n" ::"r"(dst),
               "l"(src), "r"(src_bytes), "l"(pol)
               : "memory");
}
// L2 policy for data read once: its lines are the first to be evicted, so
// the stream does not push out what is still to be read (a focal layer's
// image logits, the next layer's prefetched rows).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}
// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col). Register-only
// operations (this and movmatrix) are left free for the compiler to schedule;
// ldmatrix stays ordered after the cp.async waits.
__device__ __forceinline__ void mma_bf16(float c[4], const uint32_t a[4], uint32_t b0,
                                         uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
      "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Thread-block cluster: barrier (release/acquire) and distributed shared memory.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
}
// Store to the same shared-memory offset as `local` in CTA `rank` of the cluster.
__device__ __forceinline__ void st_dsmem_f32x2(float* local, uint32_t rank, float a, float b) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};\n" ::"r"(remote), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ void st_dsmem_f32x4(float* local, uint32_t rank, float4 v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(remote), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// Bring `bytes` (multiple of 16) at `p` into L2; never faults on a valid address.
__device__ __forceinline__ void prefetch_l2(const void* ptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(ptr), "r"(bytes) : "memory");
}
// 2^x on the special-function unit (x = -inf gives +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Keep count k = ceil(tau * n - 1e-9) in IEEE double, clamped to [1, n];
// explicit round-to-nearest intrinsics keep the compiler from fusing the
// multiply and subtract, so host, device and any IEEE double evaluation agree.
__host__ __device__ inline int keep_count(double tau, int n) {
  if (n <= 0) return 0;
#ifdef __CUDA_ARCH__
  double x = __dsub_rn(__dmul_rn(tau, (double)n), 1e-9);
#else
  volatile double prod = tau * (double)n;
  volatile double x = prod - 1e-9;
#endif
  double c = ceil(x);
  int k = c < 1.0 ? 1 : (c > (double)n ? n : (int)c);
  return k;
}

// ---------------------------------------------------------------- attend list

struct AttendList {
  int n_t;
  int n_pre;             // positions [0, n_pre)
  const int32_t* sel;    // then sel[0 .. n_sel)
  int n_sel;
  int tail_start;        // then tail_start + [0, n_att - n_pre - n_sel)
  int n_att;
  int img_start, n_img;  // image range (focal: logits; sparse: selection check)
};

// Lengths and image range of sequence b (validated and clamped; faults are
// ORed into `bad`). n_pre/n_att describe the full-cache list [0, N_t).
template <int MODE>
__device__ __forceinline__ AttendList make_list(const Params& p, int b, int& bad) {
  AttendList L;
  const int cap = p.max_pages << p.log2_page;
  int n_t = __ldcg(p.seq_len + b);
  if (n_t < 1 || n_t > cap) {
    bad |= kDevBadSeqLen;
    n_t = n_t < 0 ? 0 : (n_t > cap ? cap : n_t);
  }
  L.n_t = n_t;
  L.n_pre = n_t;
  L.n_att = n_t;
  L.sel = nullptr;
  L.n_sel = 0;
  L.tail_start = 0;
  L.img_start = 0;
  L.n_img = 0;
  if (MODE == kFocal || MODE == kSparse || MODE == kProfile) {
    int s = __ldcg(p.img_range + 2 * b), n = __ldcg(p.img_range + 2 * b + 1);
    if (s < 0 || n < 0 || s > n_t || n > n_t - s || (MODE == kFocal && n > p.max_img)) {
      bad |= kDevBadImg;
      s = s < 0 ? 0 : (s > n_t ? n_t : s);
      n = n < 0 ? 0 : (n > n_t - s ? n_t - s : n);
      if (MODE == kFocal && n > p.max_img) n = p.max_img;
    }
    L.img_start = s;
    L.n_img = n;
  }
  if (MODE == kSparse) L.sel = p.idx + (size_t)b * p.idx_stride;
  return L;
}

// ---------------------------------------------------------------- shared memory

// Work-list entries resolved to cache rows per round: a multiple of the CTA
// size (every thread resolves the same number).
__host__ __device__ constexpr int slice_for(int v) { return v == kDeep ? 1024 : 960; }

template <typename T, int D, int V = kGeneral>
struct Smem {
  static constexpr int ST = stages_of(V);
  static constexpr int kWarps = warps_for(V);
  static constexpr int kSliceMax = slice_for(V);
  static_assert(kSliceMax % (32 * kWarps) == 0 && kSliceMax % kTile == 0, "slice layout");
  static constexpr int kRowBytes = D * (int)sizeof(T);
  static constexpr int kStageBytes = 2 * kTile * kRowBytes;          // K rows then V rows
  static constexpr int kPipeBytes = kWarps * ST * kStageBytes;
  static constexpr int kRowOffset = kPipeBytes;                      // int row[kSliceMax]
  static constexpr int kPosOffset = kRowOffset + kSliceMax * 4;      // int pos[kSliceMax]
  // partials pushed here by the other CTAs of the cluster (never overlaps
  // the pipeline, which may still be in use when they arrive)
  static constexpr int kRecvMl = kPosOffset + kSliceMax * 4;         // f32 [kMaxSplits][8][2]
  static constexpr int kRecvAcc = kRecvMl + kMaxSplits * kSlots * 2 * 4;
  static constexpr int kRecvAccFloats = 4 * (kSlots * D / 4 + kMaxSplits);
  // the CTA's one reading of k before the wait (sparse), shared by its threads
  static constexpr int kSpecK = kRecvAcc + kRecvAccFloats * 4;
  static constexpr int kQOffset = kSpecK + 16;                       // f32 path: q[8][D]
  static constexpr int kMainBytes = kQOffset + (sizeof(T) == 4 ? kSlots * D * 4 : 0);
};

template <int D, int kWarps>
struct EpiSmem {
  // reuses the pipeline area once streaming is done: per-warp partials
  // wm[W][8], wl[W][8], wacc[W][8][D]; focal: the heads' max M[8], 1/sum invL[8];
  // profile: the per-warp image sums wil[W][8]
  static constexpr int kWm = 0;
  static constexpr int kWl = kWm + kWarps * kSlots * 4;
  static constexpr int kWacc = kWl + kWarps * kSlots * 4;
  static constexpr int kM = kWacc + kWarps * kSlots * D * 4;
  static constexpr int kInvL = kM + kSlots * 4;
  static constexpr int kWil = kInvL + kSlots * 4;
  static constexpr int kBytes = kWil + kWarps * kSlots * 4;
};

template <typename T, int D, int V = kGeneral>
inline int attend_smem_bytes() {
  static_assert(EpiSmem<D, warps_for(V)>::kBytes <= Smem<T, D, V>::kPipeBytes,
                "epilogue must fit the pipeline area");
  return Smem<T, D, V>::kMainBytes;
}

// A variant exists where its shared memory fits one CTA (the general one
// always does; bf16 fits it twice an SM).
template <typename T, int D, int V>
constexpr bool variant_fits() {
  return Smem<T, D, V>::kMainBytes <= 227 * 1024;
}

// Split-K factor S (= cluster size) for `units` (sequence, KV head) pairs and
// attend lists of about `len` tokens; active[s] = clusters of s CTAs the
// device holds at once, num_sms its SM count. Model: clusters run in waves of
// active[S]; a wave costs a fixed ~4 us (CTA start, pipeline fill, merge and
// cluster barrier) plus its CTAs' share of len/S tokens at ~8 ns per token,
// slowed down when the wave's CTAs together ask for more than HBM delivers
// (~30 GB/s per CTA under load); a partial last wave is charged for the CTAs
// it holds. Every doubling of the cluster adds ~0.25 us of merge latency; a
// grid of at most num_sms CTAs also lets the next kernel's CTAs stage their
// first tiles while it runs (programmatic dependent launch), worth ~3 us.
// Fitted to forced split counts of every layer kind on GB300 (graph-replayed
// layers, L2 flushed; 4 to 640 units of 525 to 18.5k tokens): the choice is
// within 3% of the fastest forced count on each (1 sequence: 16 splits for
// full layers, 12 for gather ones; 32 sequences: 2 and 1; 80 or more
// sequences: 1 for gather layers).
inline int choose_splits(long units, long len, int max_splits, const int* active, int num_sms) {
  const double ns_per_token = 8.0, cta_gbs = 30.0, hbm_gbs = 6500.0, wave_fixed_us = 4.0,
               us_per_doubling = 0.25, overlap_us = 3.0;
  if (len < 1) len = 1;
  int best = 1;
  double best_cost = 1e300;
  for (int s = 1; s <= max_splits; ++s) {
    const int act = active[s];
    if (act < 1) continue;
    const double chunk_us = ((len + s - 1) / s) * ns_per_token * 1e-3;
    // one wave of `clusters` clusters
    auto wave_us = [&](long clusters) {
      const double load = (double)clusters * s * cta_gbs / hbm_gbs;
      return wave_fixed_us + chunk_us * (load > 1.0 ? load : 1.0);
    };
    const long full = units / act, rest = units % act;
    double cost = full * wave_us(act) + (rest ? wave_us(rest) : 0.0) +
                  us_per_doubling * log2((double)s);
    if (units * s <= num_sms) cost -= overlap_us;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// ---------------------------------------------------------------- warp reductions

__device__ __forceinline__ float warp_max_gid(float x) {  // over lanes with equal lane%4
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 8));
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 16));
  return x;
}
__device__ __forceinline__ float warp_sum_gid(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  x += __shfl_xor_sync(0xffffffffu, x, 8);
  x += __shfl_xor_sync(0xffffffffu, x, 16);
  return x;
}

// ---------------------------------------------------------------- per-warp state

// bf16 tensor-core path: thread (gid = lane/4, tig = lane%4) owns query-head
// slots 2*tig, 2*tig+1; accumulator O^T[d][head] as m16n8 fragments.
template <int D>
struct WarpStateMma {
  float acc[D / 16][4];
  float m[2], l[2];
  float il[2];   // profile mode: the image tokens' share of l
  uint32_t qf[D / 16][2];
};

// fp32 CUDA-core path: lane owns head-dim columns lane + 32*j of every slot.
template <int D>
struct WarpStateF32 {
  float acc[kSlots][D / 32];
  float m[kSlots], l[kSlots];
  float il[kSlots];   // profile mode: the image tokens' share of l
};

}  // namespace fastocr
