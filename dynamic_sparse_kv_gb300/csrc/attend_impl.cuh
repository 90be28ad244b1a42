// Kernel body of the split-K decode attention (see attend_kernels.cuh for the
// design). Included by the per-dtype translation units, which instantiate it.
#pragma once

#include <math_constants.h>

#include "attend_kernels.cuh"

namespace fastocr {

// ---------------------------------------------------------------- top-k

constexpr int kSelectThreads = 1024;
constexpr int kSelSub = 4;   // sub-histograms per radix pass (warp w counts into w % 4)

// Shared memory of the selection kernel: keys[max_img] (fp32 bit patterns),
// then the histograms of the four radix passes [4][kSelSub][256] (zeroed
// before the kernel waits for its predecessor), then scratch.
struct SelectSmem {
  static constexpr int kNW = kSelectThreads / 32;
  __host__ __device__ static int hist_offset(int max_img) { return (max_img * 4 + 15) / 16 * 16; }
  __host__ __device__ static int scratch_offset(int max_img) { return hist_offset(max_img) + 4 * kSelSub * 256 * 4; }
  __host__ __device__ static int bytes(int max_img) { return scratch_offset(max_img) + (8 + 2 * kNW) * 4 + kNW * 8 + 16; }
};

// Selection kernel of a focal layer: one CTA of NT threads per sequence,
// launched right after the focal attend kernel, which left each KV head's
// share of the image scores in the workspace (or on its own, on scores a
// caller supplies). It sums the shares into keys in
// a fixed head order, adds the image mass to the profiler slot (warm-up only),
// then either writes the summed scores out (sigma_out) or
// selects the k largest keys (ties to the lower offset) with an 8-bit
// radix select over the fp32 bit patterns (scores are >= 0, so the unsigned
// order is the float order); the first pass is counted while the keys are
// summed, and the search stops as soon as every key sharing the decided prefix
// is kept. Plain shared-memory atomics into kSelSub sub-histograms measured
// faster than aggregating equal digits of a warp with __match_any_sync first.
// The selection is written in ascending position order.
template <int NT>
__global__ void __launch_bounds__(NT) select_kernel(const Params p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
  int* hist = reinterpret_cast<int*>(smem + SelectSmem::hist_offset(p.max_img));   // [4][kSelSub][256]
  int* scratch = reinterpret_cast<int*>(smem + SelectSmem::scratch_offset(p.max_img));
  double* dscr = reinterpret_cast<double*>(scratch + 8 + 2 * NW);
  for (int i = tid; i < 4 * kSelSub * 256; i += NT) hist[i] = 0;
  // lengths and image range are final before the attend kernel starts, so
  // the keep count (double arithmetic, one thread) is known before the wait
  int bad = 0;  // make_list flags: already reported by the attend kernel
  const AttendList L = make_list<kFocal>(p, b, bad);
  const int n = L.n_img;
  if (tid == NT - 1) scratch[2] = keep_count(p.tau, n);

  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  __syncthreads();   // histograms zeroed, keep count known

  // keys = sum of the KV heads' shares (fixed order); first-pass histogram
  const bool profiling = p.profile_layer >= 0;
  double local = 0.0;
  int* h0 = hist + (warp & (kSelSub - 1)) * 256;
  const float* sp_b = p.sel_src + (size_t)b * p.sel_batch_stride;
  float* so_b = p.sigma_out ? p.sigma_out + (size_t)b * p.sigma_stride : nullptr;
  for (int i0 = 0; i0 < n; i0 += 4 * NT) {
    float sv[4] = {0.f, 0.f, 0.f, 0.f};
    for (int hk0 = 0; hk0 < p.sel_heads; hk0 += 4) {   // 16 loads in flight, summed in head order
      float v[4][4];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * NT + tid;
          v[c][u] = (hk0 + c < p.sel_heads && i < n)
                        ? __ldcg(sp_b + (size_t)(hk0 + c) * p.sel_head_stride + i) : 0.f;
        }
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (hk0 + c < p.sel_heads) sv[u] += v[c][u];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * NT + tid;
      const bool act = i < n;
      // scores are >= 0, so the bit pattern without its (zero) sign bit keeps
      // their order; the first 8-bit digit is then the whole exponent
      const uint32_t key = __float_as_uint(sv[u]) << 1;
      if (act) {
        keys[i] = key;
        if (profiling) local += (double)sv[u];
        if (so_b) so_b[i] = sv[u];
      }
      if (act) atomicAdd(h0 + (key >> 24), 1);
    }
  }
  if (profiling) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
    if (lane == 0) dscr[warp] = local;
  }
  if (tid == 0 && !so_b) p.k_out[b] = scratch[2];
  __syncthreads();
  if (profiling && tid == 0) {
    double tot = 0.0;
    for (int w = 0; w < NW; ++w) tot += dscr[w];
    atomicAdd(p.profile + p.profile_layer, tot);
  }
  if (so_b) return;   // scores only: the caller selects (e.g. after summing head shards)
  const int k = scratch[2];
  if (k == 0) return;

  // --- radix select of the k-th largest key
  uint32_t prefix = 0, mask = 0;
  int krem = k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    int* hp = hist + pass * kSelSub * 256;
    if (pass > 0) {
      int* my = hp + (warp & (kSelSub - 1)) * 256;
      for (int base = warp * 32; base < n; base += NT) {
        const int i = base + lane;
        const uint32_t key = i < n ? keys[i] : 0u;
        if (i < n && (key & mask) == prefix) atomicAdd(my + ((key >> shift) & 255u), 1);
      }
      __syncthreads();
    }
    if (warp == 0) {
      // lane L scans bins 255-8L .. 248-8L (descending), summing the sub-histograms
      int cnt[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int bin = 255 - 8 * lane - j;
        int c = 0;
#pragma unroll
        for (int sb = 0; sb < kSelSub; ++sb) c += hp[sb * 256 + bin];
        cnt[j] = c;
        tot += c;
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - tot;
      if (excl < krem && krem <= incl) {
        int c = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (c + cnt[j] >= krem) {
            scratch[0] = 255 - 8 * lane - j;
            scratch[1] = c;
            scratch[3] = cnt[j];
            break;
          }
          c += cnt[j];
        }
      }
    }
    __syncthreads();
    prefix |= (uint32_t)scratch[0] << shift;
    mask |= 255u << shift;
    krem -= scratch[1];
    if (krem == scratch[3]) break;   // every key with this prefix is kept
  }
  // keep: (key & mask) > prefix, or == prefix for the first krem such keys
  const uint32_t thr = prefix;

  // --- stable compaction: thread t owns the keys [t*per, t*per + per), per a
  // multiple of 4 read as 16-byte vectors. An exclusive block scan of the
  // packed (greater, equal) counts gives each thread its output offset: the
  // kept keys before it are every greater key before it plus the first krem
  // equal keys of the whole row.
  const int per = ((n + NT - 1) / NT + 3) & ~3;
  const int lo = tid * per, hi = min(n, lo + per);
  int gt = 0, eq = 0;
  for (int i0 = lo; i0 < hi; i0 += 4) {
    const uint4 kv = *reinterpret_cast<const uint4*>(keys + i0);
    const uint32_t kk[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool ok = i0 + u < hi;
      const uint32_t key = kk[u] & mask;
      gt += ok && key > thr;
      eq += ok && key == thr;
    }
  }
  int* s_warp = scratch + 8;           // [NW]: packed warp totals, then their exclusive prefix
  const int packed = (gt << 16) | eq;  // both counts <= kMaxImg < 2^15
  int incl = packed;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int t = lane < NW ? s_warp[lane] : 0;
    int v = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane < NW) s_warp[lane] = v - t;
  }
  __syncthreads();
  const int before = s_warp[warp] + incl - packed;
  int eq_run = before & 0xffff;
  int out = (before >> 16) + min(eq_run, krem);
  int32_t* dst = p.idx_out + (size_t)b * p.idx_stride;
  for (int i0 = lo; i0 < hi; i0 += 4) {
    const uint4 kv = *reinterpret_cast<const uint4*>(keys + i0);
    const uint32_t kk[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (i0 + u >= hi) break;
      const uint32_t key = kk[u] & mask;
      bool take = key > thr;
      if (key == thr) {
        take = eq_run < krem;
        ++eq_run;
      }
      if (take) {
        if (out < k)   // never false for a consistent selection; guards the store anyway
          dst[out] = L.img_start + i0 + u;
        else
          bad |= kDevInternal;
        ++out;
      }
    }
  }
  if (bad & kDevInternal) atomicOr(p.status, kDevInternal);
}

inline int select_smem_bytes(int max_img) { return SelectSmem::bytes(max_img); }


inline cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, int smem, cudaStream_t stream,
                                     cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// ---------------------------------------------------------------- main kernel

//
// Work list of one CTA. The mode's attend set minus the current token N_t-1
// is the "text" list (at most two contiguous position ranges); the S CTAs of a
// (sequence, KV head) take equal contiguous shares of it, in sparse mode every
// CTA also takes an equal share of the selection, and the last CTA takes the
// current token. Text entries -- cache rows of earlier tokens, their pages,
// the lengths -- are final before the previous kernel on the stream starts,
// so they are resolved and their first tiles staged into shared memory before
// griddepcontrol.wait. So is the current token's row, but its K/V only after
// the wait. The selection (k and idx) may be written by the previous kernel:
// it is resolved and staged speculatively before the wait and checked after
// it; q is read only after it.
struct CtaList {
  int n_t;
  int a1, len1, a2, len2;   // text ranges [a1, a1+len1) and [a2, a2+len2)
  int txt_lo, n_txt;        // this CTA's text entries
  int has_cur, cur_pos;     // this CTA attends the current token
  const int32_t* sel;       // sparse: selected positions of this sequence
  int sel_lo, n_sel;        // this CTA's selection entries
  int img_start, n_img;
};

template <int MODE>
__device__ __forceinline__ CtaList make_cta_list(const Params& p, int b, int split, int& bad) {
  CtaList c;
  const AttendList L = make_list<MODE>(p, b, bad);   // lengths and image range (not k)
  const int n_t = L.n_t;
  c.n_t = n_t;
  c.img_start = L.img_start;
  c.n_img = L.n_img;
  c.sel = L.sel;
  c.sel_lo = 0;
  c.n_sel = 0;
  const int cur = n_t - 1;
  int a1 = 0, len1 = 0, a2 = 0, len2 = 0, in_set = 0;
  if (n_t >= 1) {
    if (MODE == kFull || MODE == kFocal || MODE == kProfile) {
      len1 = n_t - 1;
      in_set = 1;
    } else if (MODE == kRswa) {
      const int pre = min(p.prefix_len, n_t);
      if (cur < p.prefix_len) {
        len1 = cur;
        in_set = 1;
      } else {
        len1 = pre;
        a2 = max(p.prefix_len, n_t - p.window);
        len2 = max(0, cur - a2);
        in_set = p.window >= 1;
      }
    } else {  // kSparse: prefix [0, start) and generated [start + N_img, N_t)
      const int tail = L.img_start + L.n_img;
      if (cur >= tail) {
        len1 = L.img_start;
        a2 = tail;
        len2 = cur - tail;
        in_set = 1;
      } else if (cur < L.img_start) {
        len1 = cur;
        in_set = 1;
      } else {
        len1 = L.img_start;
      }
    }
  }
  c.a1 = a1;
  c.len1 = len1;
  c.a2 = a2;
  c.len2 = len2;
  const int n_text = len1 + len2;
  const int per = (n_text + p.splits - 1) / p.splits;
  c.txt_lo = split * per;
  c.n_txt = max(0, min(per, n_text - c.txt_lo));
  c.has_cur = in_set && split == p.splits - 1;
  c.cur_pos = cur;
  return c;
}

// Selection share of this CTA (sparse) for k selected positions.
__device__ __forceinline__ void add_selection(const Params& p, int k, int split, CtaList& c,
                                              int& bad) {
  const int k_cap = min(c.n_img, p.idx_stride);
  if (k < 0 || k > k_cap) {
    bad |= kDevBadSelection;
    k = k < 0 ? 0 : k_cap;
  }
  const int per = (k + p.splits - 1) / p.splits;
  c.sel_lo = split * per;
  c.n_sel = max(0, min(per, k - c.sel_lo));
}

// V: the kernel variant (warps per CTA and cp.async stages per warp).
template <typename T, int D, int MODE, int V>
__global__ void __launch_bounds__(32 * warps_for(V), ctas_per_sm(V)) attend_kernel(const Params p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  using SM = Smem<T, D, V>;
  constexpr int ST = stages_of(V);
  constexpr int kWarps = warps_for(V);
  constexpr int kThreads = 32 * kWarps;
  constexpr int kSliceMax = slice_for(V);
  using E = EpiSmem<D, kWarps>;
  constexpr bool kMma = sizeof(T) == 2;
  constexpr int ROWB = SM::kRowBytes;
  constexpr int CH = ROWB / 16;                 // 16-byte chunks per row
  const float kNegInf = -CUDART_INF_F;

  const int split = blockIdx.x, hkv = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const T* __restrict__ kg = static_cast<const T*>(p.k);
  const T* __restrict__ vg = static_cast<const T*>(p.v);
  const int32_t* __restrict__ bt = p.block_table + (size_t)b * p.max_pages;
  const int page_mask = (1 << p.log2_page) - 1;
  unsigned char* pipe = smem + warp * ST * SM::kStageBytes;
  int* srow = reinterpret_cast<int*>(smem + SM::kRowOffset);
  int* spos = reinterpret_cast<int*>(smem + SM::kPosOffset);

  // announce this CTA to its cluster (the partial exchange waits for it);
  // a single split has no partner and skips every cluster barrier
  if (p.splits > 1) cluster_arrive_relaxed();

  int bad = 0;
  // A selection that the previous kernel is still writing is not read before
  // the wait: only the text is staged, and the selection is laid out after
  // it. Only the general variant does so: its pipeline holds a few of a
  // CTA's tiles, so a stale guess costs a drain and a full restart, while the
  // deep variant's small grids stage whole lists and measured faster guessing.
  const bool sel_pending = MODE == kSparse && V == kGeneral && p.sel_pending;
  // Otherwise k and this CTA's share of the selection are read before the
  // wait (checked after it unless the caller declared them final), issued
  // together with the lengths' loads. The share is guessed from the keep
  // capacity (k = idx_stride, the usual case); a wrong guess costs one more
  // round of loads below.
  constexpr int kPer = kSliceMax / kThreads;   // entries a thread resolves
  int spec_raw[kPer];   // selection entry v = tid + j*kThreads of the share
#pragma unroll
  for (int j = 0; j < kPer; ++j) spec_raw[j] = -1;
  int k_ld = 0, lo_g = 0, n_g = 0;
  if (MODE == kSparse && !sel_pending) {
    const int per_g = (p.idx_stride + p.splits - 1) / p.splits;
    lo_g = split * per_g;
    n_g = max(0, min(per_g, p.idx_stride - lo_g));
    const int32_t* sel_b = p.idx + (size_t)b * p.idx_stride;
    if (tid == 0) k_ld = __ldcg(p.k_in + b);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int v = tid + j * kThreads;
      spec_raw[j] = v < n_g ? __ldcg(sel_b + lo_g + v) : -1;
    }
  }
  CtaList c = make_cta_list<MODE>(p, b, split, bad);

  // Work list of this CTA: [text, padded to whole tiles][selection, padded to
  // whole tiles (sparse)][current token]. Padding entries are masked. A tile
  // therefore never mixes entries of different kinds: text tiles and (in
  // sparse mode, speculatively) selection tiles can be staged before the
  // wait, and the current token, whose K/V the previous kernel may still be
  // writing, sits alone in the last tile.
  const int n_txt_pad = (c.n_txt + kTile - 1) / kTile * kTile;
  int n_sel_pad = 0;
  // cache position of work-list entry u (-1: masked)
  auto pos_of = [&](int u) -> int {
    if (u < n_txt_pad) {
      if (u >= c.n_txt) return -1;
      const int t = c.txt_lo + u;
      return t < c.len1 ? c.a1 + t : c.a2 + (t - c.len1);
    }
    u -= n_txt_pad;
    if (u >= n_sel_pad) return c.cur_pos;   // u == n_sel_pad, only with has_cur
    if (u >= c.n_sel) return -1;
    const int pos = __ldcg(c.sel + c.sel_lo + u);
    if (pos < c.img_start || pos >= c.img_start + c.n_img) {
      bad |= kDevBadSelection;
      return -1;
    }
    return pos;
  };

  // Resolve entries [u0, u1) of the round starting at entry rb into cache rows
  // (page*H_kv + hkv)*page_size + slot (-1: masked) and positions; every
  // lookup of a thread is issued before any is used.
  auto resolve = [&](int rb, int u0, int u1) {
    int pos[kPer], page[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int u = u0 + tid + j * kThreads;
      pos[j] = u < u1 ? pos_of(u) : -1;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) page[j] = pos[j] >= 0 ? __ldcg(bt + (pos[j] >> p.log2_page)) : -1;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int u = u0 + tid + j * kThreads;
      if (u >= u1) continue;
      int row = -1, ps = pos[j];
      if (ps >= 0) {
        if (page[j] < 0 || page[j] >= p.num_pages) {
          bad |= kDevBadPage;
          ps = -1;
        } else {
          row = ((page[j] * p.Hkv + hkv) << p.log2_page) | (ps & page_mask);
        }
      }
      srow[u - rb] = row;
      spos[u - rb] = ps;
    }
  };

  // Stage tile j of this warp in the current round: 16 K rows and 16 V rows
  // in 16-byte chunks. One instruction covers 32/CH whole rows; a lane takes
  // chunk `lane % CH` of rows `lane / CH`, `lane / CH + 32/CH`, ..., and reads
  // each row index once for both K and V. Masked rows are zero-filled.
  static_assert(CH <= 32 && 32 % CH == 0, "a row must fit one warp instruction");
  const int n_rows = (p.num_pages * p.Hkv) << p.log2_page;   // < 2^31, checked on the host
  constexpr int kRowsPerInst = 32 / CH;
  constexpr int kIss = kTile / kRowsPerInst;   // instructions per 16 rows
  const int ch_lane = lane % CH, row_lane = lane / CH;
  // lane constants of the copies: this lane's chunk of K and V rows, and its
  // swizzled destination offset in each of its kIss rows of a stage
  const char* kg_lane = reinterpret_cast<const char*>(kg) + ch_lane * 16;
  const char* vg_lane = reinterpret_cast<const char*>(vg) + ch_lane * 16;
  uint32_t doff[kIss];
#pragma unroll
  for (int i = 0; i < kIss; ++i) {
    const int r = i * kRowsPerInst + row_lane;
    doff[i] = r * ROWB + ((ch_lane ^ (r & 7)) << 4);
  }
  const uint64_t pol_stream = l2_policy_evict_first();   // K/V rows are read once
  auto issue = [&](int j, int n_round) {
    const int stage = j % ST;
    const int base = (warp + j * kWarps) * kTile;
    const uint32_t sb = smem_u32(pipe + stage * SM::kStageBytes);
    int rows[kIss];
#pragma unroll
    for (int i = 0; i < kIss; ++i) {
      const int r = i * kRowsPerInst + row_lane;
      rows[i] = base + r < n_round ? srow[base + r] : -1;
      if (rows[i] >= n_rows) {   // never true for a resolved row; guards the copy anyway
        bad |= kDevInternal;
        rows[i] = -1;
      }
    }
#pragma unroll
    for (int i = 0; i < kIss; ++i) {
      const size_t off = (size_t)max(rows[i], 0) * ROWB;
      const int bytes = rows[i] >= 0 ? 16 : 0;
      cp_async16(sb + doff[i], kg_lane + off, bytes, pol_stream);
      cp_async16(sb + doff[i] + kTile * ROWB, vg_lane + off, bytes, pol_stream);
    }
  };

  // ---------------- before the previous kernel completes
  // Rows of round 0: the text, the selection (sparse; read before the wait)
  // and the current token (its row is final now, its K/V may not be), with
  // all their page lookups in one round. Then every whole tile of this warp
  // that the pipeline holds, up to but excluding the current token's.
  const int n_txt0 = min(n_txt_pad, kSliceMax);
  int pre_issued = 0;   // leading tiles of this warp already staged
  int spec_u1 = n_txt_pad;   // selection entries read before the wait: [n_txt_pad, spec_u1)
  if (MODE == kSparse && !sel_pending) {
    // One thread's reading of k is shared by the CTA: the previous kernel
    // may be writing k, and threads that saw different values would lay out
    // (and stage) the list differently.
    int* s_spec_k = reinterpret_cast<int*>(smem + SM::kSpecK);
    if (tid == 0) *s_spec_k = k_ld;
    __syncthreads();
    const int k_cap = min(c.n_img, p.idx_stride);
    const int spec_k = min(max(*s_spec_k, 0), k_cap);
    const int per = (spec_k + p.splits - 1) / p.splits;
    c.sel_lo = split * per;
    c.n_sel = max(0, min(per, spec_k - c.sel_lo));
    if (c.sel_lo != lo_g || c.n_sel > n_g) {   // CTA-uniform: the guessed share missed
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int v = tid + j * kThreads;
        spec_raw[j] = v < c.n_sel ? __ldcg(c.sel + c.sel_lo + v) : -1;
      }
    }
    n_sel_pad = (c.n_sel + kTile - 1) / kTile * kTile;
    spec_u1 = min(kSliceMax, n_txt_pad + c.n_sel);
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if (n_txt_pad + tid + j * kThreads >= spec_u1) spec_raw[j] = -1;
  }
  const int n_pre = min(kSliceMax, n_txt_pad + n_sel_pad);   // entries before the current token
  {
    const int u_staged = kWarps * ST * kTile;   // entries the pre-wait tiles can cover
    int tpos[kPer], tpage[kPer], sps[kPer], spage[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int u = tid + j * kThreads;
      tpos[j] = u < n_txt0 ? pos_of(u) : -1;   // text entries: no memory reads
      const int r = spec_raw[j];
      sps[j] = (MODE == kSparse && r >= c.img_start && r < c.img_start + c.n_img) ? r : -1;
    }
    const bool cur_here = c.has_cur && tid == 0 && n_pre < kSliceMax;
#pragma unroll
    for (int j = 0; j < kPer; ++j) tpage[j] = tpos[j] >= 0 ? __ldcg(bt + (tpos[j] >> p.log2_page)) : -1;
#pragma unroll
    for (int j = 0; j < kPer; ++j) spage[j] = sps[j] >= 0 ? __ldcg(bt + (sps[j] >> p.log2_page)) : -1;
    const int cpage = cur_here ? __ldcg(bt + (c.cur_pos >> p.log2_page)) : -1;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {   // text
      const int u = tid + j * kThreads;
      if (u >= n_txt0) continue;
      int row = -1, ps = tpos[j];
      if (ps >= 0) {
        if (tpage[j] < 0 || tpage[j] >= p.num_pages) {
          bad |= kDevBadPage;
          ps = -1;
        } else {
          row = ((tpage[j] * p.Hkv + hkv) << p.log2_page) | (ps & page_mask);
        }
      }
      srow[u] = row;
      spos[u] = ps;
    }
    if (MODE == kSparse && !sel_pending) {
#pragma unroll
      for (int j = 0; j < kPer; ++j) {   // selection
        const int u = n_txt_pad + tid + j * kThreads;
        if (u >= n_pre) continue;
        int row = -1, ps = sps[j];
        if (ps >= 0 && spage[j] >= 0 && spage[j] < p.num_pages) {
          row = ((spage[j] * p.Hkv + hkv) << p.log2_page) | (ps & page_mask);
          // beyond the staged tiles: pull into L2 for later. Only the general
          // variant (large grids) does: there it shortens the post-wait stream,
          // while the deep variant's small grids measured faster without the
          // extra traffic next to the running layer.
          if constexpr (V == kGeneral) {
            if (u >= u_staged) {
              prefetch_l2(kg + (size_t)row * D, ROWB);
              prefetch_l2(vg + (size_t)row * D, ROWB);
            }
          }
        } else {
          ps = -1;
        }
        srow[u] = row;
        spos[u] = ps;
      }
    }
    if (cur_here) {
      int row = -1, ps = c.cur_pos;
      if (cpage >= 0 && cpage < p.num_pages) {
        row = ((cpage * p.Hkv + hkv) << p.log2_page) | (ps & page_mask);
        prefetch_l2(kg + (size_t)row * D, ROWB);
        prefetch_l2(vg + (size_t)row * D, ROWB);
      } else {
        bad |= kDevBadPage;
        ps = -1;
      }
      srow[n_pre] = row;
      spos[n_pre] = ps;
    }
  }
  // q and the current token's K/V may still be written by the previous
  // kernel, so they are read only after the wait; pulling their lines into L2
  // now is safe (L2 is where those writes land) and shortens that read.
  if (tid == 0)
    prefetch_l2(static_cast<const T*>(p.q) + ((size_t)b * p.Hq + (size_t)hkv * p.g) * D,
                p.g * D * (uint32_t)sizeof(T));
  __syncthreads();
#pragma unroll 1
  for (int j = 0; j < ST; ++j) {
    const int end = (warp + j * kWarps + 1) * kTile;
    if (pre_issued == j && end <= n_pre) {
      issue(j, n_pre);
      cp_async_commit();
      ++pre_issued;
    }
  }

  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if (p.pdl_early) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  // ---------------- after it: the current token's tile, q and the final
  // selection, all in flight together. The tile follows the staged ones in
  // its warp's order (sparse: under the speculative layout, redone below if
  // the speculation fails).
  if (c.has_cur && n_pre < kSliceMax && !sel_pending) {
    const int t_cur = n_pre / kTile;   // n_pre is a multiple of kTile here
    if (warp == t_cur % kWarps && pre_issued == t_cur / kWarps && pre_issued < ST) {
      issue(pre_issued, n_pre + 1);
      cp_async_commit();
      ++pre_issued;
    }
  }
  WarpStateMma<D> sm_;
  WarpStateF32<D> sf_;
  const int gid = lane >> 2, tig = lane & 3;
  if constexpr (kMma) {
    const bool have = gid < p.g;
    const T* qrow = static_cast<const T*>(p.q) + ((size_t)b * p.Hq + hkv * p.g + (have ? gid : 0)) * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      sm_.qf[ks][0] = have ? __ldcg(reinterpret_cast<const unsigned int*>(qrow + 16 * ks + 2 * tig)) : 0u;
      sm_.qf[ks][1] = have ? __ldcg(reinterpret_cast<const unsigned int*>(qrow + 16 * ks + 8 + 2 * tig)) : 0u;
    }
  }
  bool relaid = false;   // the selection's rows were resolved again (CTA-uniform)
  if (sel_pending) {
    // the selection is final now: lay it out behind the text and resolve its
    // rows (and the current token's, which moves behind it); the text tiles
    // staged before the wait stay where they are
    const int k = __ldcg(p.k_in + b);
    add_selection(p, k, split, c, bad);
    n_sel_pad = (c.n_sel + kTile - 1) / kTile * kTile;
    resolve(0, n_txt_pad, min(n_txt_pad + n_sel_pad + c.has_cur, kSliceMax));
    relaid = true;
  } else if (MODE == kSparse && p.sel_final) {
    // the caller guarantees that k and idx were written before the previous
    // kernel began, so the reading before the wait is the real selection:
    // only report its faulty entries (each thread its own, no barrier)
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int u = n_txt_pad + tid + j * kThreads;
      if (u >= spec_u1) continue;
      if (spec_raw[j] < c.img_start || spec_raw[j] >= c.img_start + c.n_img)
        bad |= kDevBadSelection;
      else if (spos[u] < 0)
        bad |= kDevBadPage;
    }
    const int k_read = *reinterpret_cast<const int*>(smem + SM::kSpecK);   // clamped before use
    if (tid == 0 && (k_read < 0 || k_read > min(c.n_img, p.idx_stride))) bad |= kDevBadSelection;
  } else if (MODE == kSparse) {
    // keep the speculative entries only if this CTA's share is unchanged
    const int k = __ldcg(p.k_in + b);
    int raw2[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int u = n_txt_pad + tid + j * kThreads;
      raw2[j] = u < spec_u1 ? __ldcg(c.sel + c.sel_lo + (u - n_txt_pad)) : -1;
    }
    const int spec_lo = c.sel_lo, spec_n = c.n_sel;
    add_selection(p, k, split, c, bad);
    int ok = c.sel_lo == spec_lo && c.n_sel == spec_n;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int u = n_txt_pad + tid + j * kThreads;
      if (u < spec_u1 && raw2[j] != spec_raw[j]) ok = 0;
    }
    if (__syncthreads_and(ok)) {   // the speculative entries are the real ones: report faulty ones
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int u = n_txt_pad + tid + j * kThreads;
        if (u >= spec_u1) continue;
        if (raw2[j] < c.img_start || raw2[j] >= c.img_start + c.n_img)
          bad |= kDevBadSelection;
        else if (spos[u] < 0)
          bad |= kDevBadPage;
      }
    } else {   // drop the staged tiles and lay out the selection and current token again
      cp_async_wait<0>();
      pre_issued = 0;
      n_sel_pad = (c.n_sel + kTile - 1) / kTile * kTile;
      resolve(0, n_txt_pad, min(n_txt_pad + n_sel_pad + c.has_cur, kSliceMax));
      relaid = true;
    }
  }
  const int n_cta = n_txt_pad + n_sel_pad + c.has_cur;

  float* logit_base = nullptr;
  if (MODE == kFocal)
    logit_base = p.logits + ((size_t)b * p.Hkv + hkv) * (size_t)p.max_img * kSlots;

  if constexpr (kMma) {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sm_.acc[mt][e] = 0.f;
    sm_.m[0] = sm_.m[1] = kNegInf;
    sm_.l[0] = sm_.l[1] = 0.f;
    sm_.il[0] = sm_.il[1] = 0.f;
  } else {
    float* qs = reinterpret_cast<float*>(smem + SM::kQOffset);
    for (int e = tid; e < kSlots * D; e += kThreads) {
      const int h = e / D, d = e % D;
      qs[e] = h < p.g ? __ldcg(static_cast<const float*>(p.q) + ((size_t)b * p.Hq + hkv * p.g + h) * D + d) : 0.f;
    }
#pragma unroll
    for (int h = 0; h < kSlots; ++h) {
      sf_.m[h] = kNegInf;
      sf_.l[h] = 0.f;
      sf_.il[h] = 0.f;
#pragma unroll
      for (int j = 0; j < D / 32; ++j) sf_.acc[h][j] = 0.f;
    }
  }
  // the fp32 path's q and rows resolved again after the wait are read by
  // every warp; otherwise each warp starts as soon as its own q has arrived
  if (!kMma || relaid) __syncthreads();

  // lane constants of the ldmatrix addresses within a stage (bf16): K reads
  // row `lane & 15`, chunk 2ks + (lane >> 4); V reads row
  // (lane & 7) + 8 (lane >> 4), chunk 2mt + ((lane >> 3) & 1). Chunk bit 3
  // (ks, mt >= 4) is untouched by the swizzle: 128 bytes added per 4 steps.
  uint32_t koff[4], voff[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int kr = (lane & 7) + (lane & 8), kc = 2 * q + (lane >> 4);
    koff[q] = kr * ROWB + ((kc ^ (kr & 7)) << 4);
    const int vr = (lane & 7) + ((lane >> 4) << 3), vc = 2 * q + ((lane >> 3) & 1);
    voff[q] = vr * ROWB + ((vc ^ (vr & 7)) << 4);
  }

  // Tensor-core tile body, in two parts so that the next tile's QK^T can be
  // issued before this tile's softmax and PV (software pipelining).
  // (1) S^T of the tile whose K rows start at shared address kA.
  auto tile_qk = [&](uint32_t kA, float cfr[4]) {
    // S^T[16 keys x 8 heads] = K[16 x D] . Q^T[D x 8] in kChains independent
    // accumulation chains (16-wide slices of d taken round robin) to cut
    // the dependent MMA latency
    constexpr int kChains = D / 16 >= 4 ? 4 : D / 16;
    float cc[kChains][4];
#pragma unroll
    for (int q = 0; q < kChains; ++q) cc[q][0] = cc[q][1] = cc[q][2] = cc[q][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      // chunk 2ks + (lane >> 4) of row `lane & 15`, swizzled: a lane
      // constant for ks % 4 plus 8 chunks per 4 ks
      uint32_t a[4];
      ldmatrix_x4(a, kA + koff[ks & 3] + (ks >> 2) * 128);
      mma_bf16(cc[ks % kChains], a, sm_.qf[ks][0], sm_.qf[ks][1]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float s = cc[0][e];
#pragma unroll
      for (int q = 1; q < kChains; ++q) s += cc[q][e];
      cfr[e] = s;
    }
  };
  // (2) masks, logits (focal), online softmax and O^T += V^T P^T for the tile
  // of work-list entries [tbase, tbase + 16) whose V rows start at vA.
  auto tile_rest = [&](const float cfr[4], uint32_t vA, int tbase, int n_round) {
    // cache positions of keys gid and gid+8 (-1: masked or past the end)
    const int posA = tbase + gid < n_round ? spos[tbase + gid] : -1;
    const int posB = tbase + gid + 8 < n_round ? spos[tbase + gid + 8] : -1;
    const float s0 = posA >= 0 ? cfr[0] * p.scale_log2 : kNegInf;
    const float s1 = posA >= 0 ? cfr[1] * p.scale_log2 : kNegInf;
    const float s2 = posB >= 0 ? cfr[2] * p.scale_log2 : kNegInf;
    const float s3 = posB >= 0 ? cfr[3] * p.scale_log2 : kNegInf;
    if (MODE == kFocal) {
      if (posA >= c.img_start && posA < c.img_start + c.n_img)
        *reinterpret_cast<float2*>(logit_base + (size_t)(posA - c.img_start) * kSlots + 2 * tig) =
            make_float2(s0, s1);
      if (posB >= c.img_start && posB < c.img_start + c.n_img)
        *reinterpret_cast<float2*>(logit_base + (size_t)(posB - c.img_start) * kSlots + 2 * tig) =
            make_float2(s2, s3);
    }
    // Online softmax with a lazily moved running max (base-2 logits): the
    // max and the output scale are updated only when a score exceeds the
    // running max by more than kLazyMax, so most tiles need neither the
    // cross-lane max nor a rescale; probabilities stay below 2^kLazyMax.
    if (__any_sync(0xffffffffu, s0 > sm_.m[0] + kLazyMax || s2 > sm_.m[0] + kLazyMax ||
                                    s1 > sm_.m[1] + kLazyMax || s3 > sm_.m[1] + kLazyMax)) {
      const float mx0 = warp_max_gid(fmaxf(s0, s2));
      const float mx1 = warp_max_gid(fmaxf(s1, s3));
      const float mn0 = fmaxf(sm_.m[0], mx0), mn1 = fmaxf(sm_.m[1], mx1);
      const float al0 = fast_exp2(sm_.m[0] - (mn0 == kNegInf ? 0.f : mn0));
      const float al1 = fast_exp2(sm_.m[1] - (mn1 == kNegInf ? 0.f : mn1));
      sm_.l[0] *= al0;
      sm_.l[1] *= al1;
      if constexpr (MODE == kProfile) {
        sm_.il[0] *= al0;
        sm_.il[1] *= al1;
      }
      sm_.m[0] = mn0;
      sm_.m[1] = mn1;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        sm_.acc[mt][0] *= al0;
        sm_.acc[mt][1] *= al1;
        sm_.acc[mt][2] *= al0;
        sm_.acc[mt][3] *= al1;
      }
    }
    const float b0f = sm_.m[0] == kNegInf ? 0.f : sm_.m[0];
    const float b1f = sm_.m[1] == kNegInf ? 0.f : sm_.m[1];
    const float p0 = fast_exp2(s0 - b0f), p2 = fast_exp2(s2 - b0f);
    const float p1 = fast_exp2(s1 - b1f), p3 = fast_exp2(s3 - b1f);
    // The P.V product takes the probabilities rounded to bf16. Outside focal
    // layers the softmax sum adds those same rounded values, so the weights
    // that multiply V sum to exactly 1 after normalisation (rounding moves a
    // weight by at most 2^-9 relative, never the total). A focal layer's sum
    // also turns its logits into the image scores, which must be the
    // probabilities themselves, so there it adds the unrounded values; so does
    // a profiling layer, whose image mass is a ratio of such sums.
    const uint32_t pk01 = pack_bf16(p0, p1), pk23 = pack_bf16(p2, p3);
    if (MODE == kFocal || MODE == kProfile) {
      sm_.l[0] += p0 + p2;
      sm_.l[1] += p1 + p3;
      if constexpr (MODE == kProfile) {
        const bool iA = posA >= c.img_start && posA < c.img_start + c.n_img;
        const bool iB = posB >= c.img_start && posB < c.img_start + c.n_img;
        sm_.il[0] += (iA ? p0 : 0.f) + (iB ? p2 : 0.f);
        sm_.il[1] += (iA ? p1 : 0.f) + (iB ? p3 : 0.f);
      }
    } else {
      sm_.l[0] += __uint_as_float(pk01 << 16) + __uint_as_float(pk23 << 16);
      sm_.l[1] += __uint_as_float(pk01 & 0xffff0000u) + __uint_as_float(pk23 & 0xffff0000u);
    }
    // P^T[16 keys x 8 heads] as the B operand: transpose the two 8x8 blocks
    const uint32_t bb0 = movmatrix_trans(pk01);
    const uint32_t bb1 = movmatrix_trans(pk23);
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      uint32_t a[4];
      ldmatrix_x4_trans(a, vA + voff[mt & 3] + (mt >> 2) * 128);
      // O^T[16 dims x 8 heads] += V^T[16 dims x 16 keys] . P^T[16 keys x 8 heads]
      mma_bf16(sm_.acc[mt], a, bb0, bb1);
    }
  };

  // ---------------- stream the work list in rounds of kSliceMax entries
  for (int rb = 0; rb < n_cta; rb += kSliceMax) {
    const int n_round = min(n_cta - rb, kSliceMax);
    int first = 0;            // tiles of this warp already staged for this round
    if (rb > 0) {
      resolve(rb, rb, rb + n_round);
      __syncthreads();
    } else {
      first = pre_issued;
    }
    const int n_tiles = (n_round + kTile - 1) / kTile;
    const int my_tiles = n_tiles > warp ? (n_tiles - warp + kWarps - 1) / kWarps : 0;
#pragma unroll 1
    for (int j = 0; j < ST - 1; ++j) {
      if (j < first) continue;
      if (j < my_tiles) issue(j, n_round);
      cp_async_commit();
    }
    if constexpr (kMma && ST >= 4) {
      // Software pipelined (deep variant): the next tile's QK^T is issued
      // before this tile's softmax and PV, keeping ST-2 tiles in flight.
      // Tile j of this warp sits in stage j % ST and in commit group j, or
      // j + 1 once all ST stages were staged before the wait (`first` == ST,
      // an empty group follows them): wait<ST-2> covers the next tile in both.
      float cfr_n[4];
      if (my_tiles > 0) {
        cp_async_wait<ST - 2>();
        __syncwarp();
        tile_qk(smem_u32(pipe), cfr_n);
      }
      for (int it = 0; it < my_tiles; ++it) {
        const int jn = it + ST - 1;   // tiles below `first` were staged already
        if (jn >= first && jn < my_tiles) issue(jn, n_round);
        cp_async_commit();
        const float cfr[4] = {cfr_n[0], cfr_n[1], cfr_n[2], cfr_n[3]};
        cp_async_wait<ST - 2>();
        __syncwarp();
        // past the last tile this reads a stage no copy is writing; unused
        tile_qk(smem_u32(pipe + ((it + 1) % ST) * SM::kStageBytes), cfr_n);
        tile_rest(cfr, smem_u32(pipe + (it % ST) * SM::kStageBytes + kTile * ROWB),
                  (warp + it * kWarps) * kTile, n_round);
        __syncwarp();
      }
    } else {
    for (int it = 0; it < my_tiles; ++it) {
      const int jn = it + ST - 1;   // tiles below `first` were staged already
      if (jn >= first && jn < my_tiles) issue(jn, n_round);
      cp_async_commit();
      cp_async_wait<ST - 1>();
      __syncwarp();
      const int stage = it % ST;
      unsigned char* kS = pipe + stage * SM::kStageBytes;
      unsigned char* vS = kS + kTile * ROWB;
      const int tbase = (warp + it * kWarps) * kTile;   // tile start within the round

      if constexpr (kMma) {
        float cfr[4];
        tile_qk(smem_u32(kS), cfr);
        tile_rest(cfr, smem_u32(vS), tbase, n_round);
      } else {
        const float* qs = reinterpret_cast<const float*>(smem + SM::kQOffset);
        const int r = lane & 15, half = lane >> 4;
        float s[kSlots];
#pragma unroll
        for (int h = 0; h < kSlots; ++h) s[h] = 0.f;
#pragma unroll
        for (int cc = 0; cc < CH / 2; ++cc) {
          const int ch = half * (CH / 2) + cc;
          const float4 kv = *reinterpret_cast<const float4*>(kS + r * ROWB + ((ch ^ (r & 7)) << 4));
#pragma unroll
          for (int h = 0; h < kSlots; ++h) {
            const float4 qv = *reinterpret_cast<const float4*>(qs + h * D + ch * 4);
            s[h] = fmaf(kv.x, qv.x, s[h]);
            s[h] = fmaf(kv.y, qv.y, s[h]);
            s[h] = fmaf(kv.z, qv.z, s[h]);
            s[h] = fmaf(kv.w, qv.w, s[h]);
          }
        }
        const int pos = tbase + r < n_round ? spos[tbase + r] : -1;
#pragma unroll
        for (int h = 0; h < kSlots; ++h) {
          s[h] += __shfl_xor_sync(0xffffffffu, s[h], 16);
          s[h] = pos >= 0 ? s[h] * p.scale_log2 : kNegInf;
        }
        if (MODE == kFocal) {
          if (half == 0 && pos >= c.img_start && pos < c.img_start + c.n_img) {
            float* dst = logit_base + (size_t)(pos - c.img_start) * kSlots;
            *reinterpret_cast<float4*>(dst) = make_float4(s[0], s[1], s[2], s[3]);
            *reinterpret_cast<float4*>(dst + 4) = make_float4(s[4], s[5], s[6], s[7]);
          }
        }
        float pr[kSlots];
#pragma unroll
        for (int h = 0; h < kSlots; ++h) {
          float mx = s[h];
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          const float mn = fmaxf(sf_.m[h], mx);
          const float base = mn == kNegInf ? 0.f : mn;
          const float al = fast_exp2(sf_.m[h] - base);
          pr[h] = fast_exp2(s[h] - base);
          sf_.l[h] = sf_.l[h] * al + (half == 0 ? pr[h] : 0.f);
          if constexpr (MODE == kProfile)
            sf_.il[h] = sf_.il[h] * al +
                        (half == 0 && pos >= c.img_start && pos < c.img_start + c.n_img ? pr[h] : 0.f);
          sf_.m[h] = mn;
#pragma unroll
          for (int j = 0; j < D / 32; ++j) sf_.acc[h][j] *= al;
        }
#pragma unroll 4
        for (int tok = 0; tok < kTile; ++tok) {
          float ph[kSlots];
#pragma unroll
          for (int h = 0; h < kSlots; ++h) ph[h] = __shfl_sync(0xffffffffu, pr[h], tok);
#pragma unroll
          for (int j = 0; j < D / 32; ++j) {
            const int d = lane + 32 * j;
            const float v =
                *reinterpret_cast<const float*>(vS + tok * ROWB + ((((d >> 2) ^ (tok & 7))) << 4) + (d & 3) * 4);
#pragma unroll
            for (int h = 0; h < kSlots; ++h) sf_.acc[h][j] = fmaf(ph[h], v, sf_.acc[h][j]);
          }
        }
      }
      __syncwarp();
    }
    }
    cp_async_wait<0>();
    __syncthreads();   // before the next round overwrites the row list
  }
  cp_async_wait<0>();
  // the next kernel may now be scheduled; it waits for this grid to finish
  if (!p.pdl_early) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  __syncthreads();

  // ---------------- per-warp partials -> shared memory
  float* wm = reinterpret_cast<float*>(smem + E::kWm);
  float* wl = reinterpret_cast<float*>(smem + E::kWl);
  float* wacc = reinterpret_cast<float*>(smem + E::kWacc);
  float* wil = reinterpret_cast<float*>(smem + E::kWil);   // profile mode
  if constexpr (kMma) {
    const float l0 = warp_sum_gid(sm_.l[0]), l1 = warp_sum_gid(sm_.l[1]);
    const int h0 = warp * kSlots + 2 * tig, h1 = h0 + 1;
    if (gid == 0) {
      wm[h0] = sm_.m[0];
      wm[h1] = sm_.m[1];
      wl[h0] = l0;
      wl[h1] = l1;
    }
    if constexpr (MODE == kProfile) {
      const float il0 = warp_sum_gid(sm_.il[0]), il1 = warp_sum_gid(sm_.il[1]);
      if (gid == 0) {
        wil[h0] = il0;
        wil[h1] = il1;
      }
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      wacc[h0 * D + 16 * mt + gid] = sm_.acc[mt][0];
      wacc[h1 * D + 16 * mt + gid] = sm_.acc[mt][1];
      wacc[h0 * D + 16 * mt + 8 + gid] = sm_.acc[mt][2];
      wacc[h1 * D + 16 * mt + 8 + gid] = sm_.acc[mt][3];
    }
  } else {
#pragma unroll
    for (int h = 0; h < kSlots; ++h) {
      float l = sf_.l[h];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (lane == 0) {
        wm[warp * kSlots + h] = sf_.m[h];
        wl[warp * kSlots + h] = l;
      }
      if constexpr (MODE == kProfile) {
        float il = sf_.il[h];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) il += __shfl_xor_sync(0xffffffffu, il, o);
        if (lane == 0) wil[warp * kSlots + h] = il;
      }
#pragma unroll
      for (int j = 0; j < D / 32; ++j) wacc[(warp * kSlots + h) * D + lane + 32 * j] = sf_.acc[h][j];
    }
  }
  if (bad) atomicOr(p.status, bad);
  __syncthreads();

  // focal: this CTA's image tokens and the logits of its first kSgU*kThreads
  // of them, loaded now so that the load latency hides behind the merge
  constexpr int kSgU = 8;   // image tokens a thread scores per round (16 loads in flight)
  const int img_end = c.img_start + c.n_img;
  // a focal text list is [0, N_t - 1): text index = position
  const int sg_lo = max(c.txt_lo, c.img_start) - c.img_start;
  const int sg_hi = min(c.txt_lo + c.n_txt, img_end) - c.img_start;
  float4 sgx[kSgU][2];
  if constexpr (MODE == kFocal) {
#pragma unroll
    for (int u = 0; u < kSgU; ++u) {
      const int i = sg_lo + u * kThreads + tid;
      const float4* src4 = reinterpret_cast<const float4*>(logit_base + (size_t)i * kSlots);
      sgx[u][0] = i < sg_hi ? __ldcg(src4) : make_float4(0.f, 0.f, 0.f, 0.f);
      sgx[u][1] = i < sg_hi ? __ldcg(src4 + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  const int S = p.splits;
  constexpr int C4 = D / 4;
  const int n_pairs = p.g * C4;
  auto warp_scales = [&](int h, float sc[kWarps]) -> float {   // CTA max of head h
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * kSlots + h]);
    const float base = M == kNegInf ? 0.f : M;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) sc[w] = fast_exp2(wm[w * kSlots + h] - base);
    return M;
  };
  T* outp = static_cast<T*>(p.out) + ((size_t)b * p.Hq + (size_t)hkv * p.g) * D;
  auto store_pair = [&](int e, float4 acc) {   // output dims 4*(e % C4).. of head e / C4
    T* o = outp + (e / C4) * D + 4 * (e % C4);
    if constexpr (kMma) {
      uint2 w;
      w.x = pack_bf16(acc.x, acc.y);
      w.y = pack_bf16(acc.z, acc.w);
      *reinterpret_cast<uint2*>(o) = w;
    } else {
      *reinterpret_cast<float4*>(o) = acc;
    }
  };
  float* sM = reinterpret_cast<float*>(smem + E::kM);        // focal: heads' max
  float* sInvL = reinterpret_cast<float*>(smem + E::kInvL);  // focal: heads' 1/sum

  if (S == 1) {
    // ---------------- one CTA holds the whole list: its warps' partials
    // merge straight into the output, in one pass after one barrier
    for (int e = tid; e < n_pairs; e += kThreads) {
      const int h = e / C4, c4 = e % C4;
      float sc[kWarps];
      warp_scales(h, sc);
      float L = 0.f;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        L = fmaf(wl[w * kSlots + h], sc[w], L);
        const float4 v = *reinterpret_cast<const float4*>(wacc + (w * kSlots + h) * D + 4 * c4);
        a.x = fmaf(v.x, sc[w], a.x);
        a.y = fmaf(v.y, sc[w], a.y);
        a.z = fmaf(v.z, sc[w], a.z);
        a.w = fmaf(v.w, sc[w], a.w);
      }
      const float inv = L > 0.f ? __frcp_rn(L) : 0.f;
      store_pair(e, make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv));
    }
    if (MODE == kFocal && tid < kSlots) {
      float sc[kWarps];
      const float M = warp_scales(tid, sc);
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) L = fmaf(wl[w * kSlots + tid], sc[w], L);
      sM[tid] = M == kNegInf ? 0.f : M;
      sInvL[tid] = L > 0.f ? __frcp_rn(L) : 0.f;
    }
    if constexpr (MODE == kProfile) {
      // the unit's image mass: sum over its heads of (image share of the
      // softmax sum) / (softmax sum), added to the layer's profiler slot
      if (warp == 0) {
        double mass = 0.0;
        if (lane < p.g) {
          float sc[kWarps];
          warp_scales(lane, sc);
          float L = 0.f, IL = 0.f;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) {
            L = fmaf(wl[w * kSlots + lane], sc[w], L);
            IL = fmaf(wil[w * kSlots + lane], sc[w], IL);
          }
          mass = L > 0.f ? (double)IL / (double)L : 0.0;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mass += __shfl_xor_sync(0xffffffffu, mass, o);
        if (lane == 0) atomicAdd(p.profile + p.profile_layer, mass);
      }
    }
  } else {
    // ---------------- push the CTA partial to the CTAs of the cluster
    // CTA `r` of the S splits owns output pairs [r*per, (r+1)*per) of the
    // (head, 4 dims) pairs; every CTA writes its share of each owner's pairs,
    // and its per-head (max, sum), straight into the owner's shared memory.
    // The CTA partial (its W warps merged) is formed by the pushing threads
    // themselves: a thread needs only its head's W (max, sum) pairs.
    const uint32_t rank = cluster_ctarank();
    const int per = (n_pairs + S - 1) / S;
    float* rml = reinterpret_cast<float*>(smem + SM::kRecvMl);     // [S][8][2]
    float* racc = reinterpret_cast<float*>(smem + SM::kRecvAcc);   // [S][per][4]
    cluster_wait();   // every CTA of the cluster has started (its receive area exists)
    for (int e = tid; e < S * kSlots; e += kThreads) {
      const int r = e / kSlots, h = e % kSlots;
      float sc[kWarps];
      const float M = warp_scales(h, sc);
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) L = fmaf(wl[w * kSlots + h], sc[w], L);
      st_dsmem_f32x2(rml + (rank * kSlots + h) * 2, r, M, L);
    }
    for (int e = tid; e < n_pairs; e += kThreads) {
      const int h = e / C4, c4 = e % C4;
      float sc[kWarps];
      warp_scales(h, sc);
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float4 v = *reinterpret_cast<const float4*>(wacc + (w * kSlots + h) * D + 4 * c4);
        a.x = fmaf(v.x, sc[w], a.x);
        a.y = fmaf(v.y, sc[w], a.y);
        a.z = fmaf(v.z, sc[w], a.z);
        a.w = fmaf(v.w, sc[w], a.w);
      }
      const int r = e / per;
      st_dsmem_f32x4(racc + ((size_t)rank * per + (e - r * per)) * 4, r, a);
    }
    cluster_sync();   // release the pushes, acquire everyone else's

    // ---------------- owner: merge the S partials of its pairs (local memory only)
    // Each thread forms its head's max and 1/sum over the S partials itself
    // (broadcast reads), so the merge needs no further barrier.
    auto head_stats = [&](int h, float& base, float& inv) {
      float ms[kMaxSplits], ls[kMaxSplits];   // all reads issued together
#pragma unroll
      for (int s = 0; s < kMaxSplits; ++s) {
        ms[s] = s < S ? rml[(s * kSlots + h) * 2] : kNegInf;
        ls[s] = s < S ? rml[(s * kSlots + h) * 2 + 1] : 0.f;
      }
      float M = kNegInf;
#pragma unroll
      for (int s = 0; s < kMaxSplits; ++s) M = fmaxf(M, ms[s]);
      base = M == kNegInf ? 0.f : M;
      float L = 0.f;
#pragma unroll
      for (int s = 0; s < kMaxSplits; ++s) L = fmaf(ls[s], fast_exp2(ms[s] - base), L);
      inv = L > 0.f ? __frcp_rn(L) : 0.f;
    };
    // G adjacent lanes share one output pair, each summing every G-th partial
    const int e_lo = (int)rank * per, e_hi = min(n_pairs, e_lo + per);
    const int n_mine = max(0, e_hi - e_lo);
    int G = 1;
    while (G * 2 <= S && G * 2 * n_mine <= kThreads && G < 16) G *= 2;
    const int sub = tid % G;
    for (int e = e_lo + tid / G; e < e_lo + ((n_mine + (kThreads / G) - 1) / (kThreads / G)) * (kThreads / G);
         e += kThreads / G) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      const bool ok = e < e_hi;
      const int h = ok ? e / C4 : 0;
      if (ok) {
        float base, inv;
        head_stats(h, base, inv);
        for (int s = sub; s < S; s += G) {
          const float4 v = *reinterpret_cast<const float4*>(racc + ((size_t)s * per + (e - e_lo)) * 4);
          const float sc = fast_exp2(rml[(s * kSlots + h) * 2] - base) * inv;
          acc.x = fmaf(v.x, sc, acc.x);
          acc.y = fmaf(v.y, sc, acc.y);
          acc.z = fmaf(v.z, sc, acc.z);
          acc.w = fmaf(v.w, sc, acc.w);
        }
      }
      for (int o = 1; o < G; o <<= 1) {
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
      }
      if (ok && sub == 0) store_pair(e, acc);
    }
    if (MODE == kFocal && tid < kSlots) head_stats(tid, sM[tid], sInvL[tid]);
    if constexpr (MODE == kProfile) {
      // this CTA's share of the unit's image mass: its image sums rescaled to
      // the heads' max over the cluster, over the heads' sum over the cluster
      // (the S shares add up to the unit's mass in the profiler slot)
      if (warp == 0) {
        double mass = 0.0;
        if (lane < p.g) {
          float base, inv, sc[kWarps];
          head_stats(lane, base, inv);
          const float Mc = warp_scales(lane, sc);
          float IL = 0.f;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) IL = fmaf(wil[w * kSlots + lane], sc[w], IL);
          const float bc = Mc == kNegInf ? 0.f : Mc;
          mass = IL > 0.f ? (double)(IL * fast_exp2(bc - base)) * (double)inv : 0.0;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mass += __shfl_xor_sync(0xffffffffu, mass, o);
        if (lane == 0) atomicAdd(p.profile + p.profile_layer, mass);
      }
    }
  }

  // ---------------- focal: scores of the image tokens this CTA streamed
  // (its text share; the last CTA also the current token) from the logits it
  // wrote itself and the heads' final max and sum: no other CTA's writes read
  if constexpr (MODE == kFocal) {
    __syncthreads();
    float Mh[kSlots], iL[kSlots];
#pragma unroll
    for (int h = 0; h < kSlots; ++h) {
      Mh[h] = h < p.g ? sM[h] : 0.f;
      iL[h] = h < p.g ? sInvL[h] : 0.f;
    }
    auto score = [&](float4 x0, float4 x1) -> float {
      const float xv[kSlots] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      float sg = 0.f;
#pragma unroll
      for (int h = 0; h < kSlots; ++h)
        if (h < p.g) sg = fmaf(fast_exp2(xv[h] - Mh[h]), iL[h], sg);
      return sg;
    };
    const size_t unit = (size_t)b * p.Hkv + hkv;
    float* sp = p.sigma_part + unit * p.max_img;
    for (int i0 = sg_lo; i0 < sg_hi; i0 += kSgU * kThreads) {
      if (i0 > sg_lo) {   // later blocks of kSgU*kThreads tokens
#pragma unroll
        for (int u = 0; u < kSgU; ++u) {
          const int i = i0 + u * kThreads + tid;
          const float4* src4 = reinterpret_cast<const float4*>(logit_base + (size_t)i * kSlots);
          sgx[u][0] = i < sg_hi ? __ldcg(src4) : make_float4(0.f, 0.f, 0.f, 0.f);
          sgx[u][1] = i < sg_hi ? __ldcg(src4 + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < kSgU; ++u) {
        const int i = i0 + u * kThreads + tid;
        const float sg = score(sgx[u][0], sgx[u][1]);
        if (i < sg_hi) sp[i] = sg;
      }
    }
    if (c.has_cur && tid == 0 && c.cur_pos >= c.img_start && c.cur_pos < img_end) {
      const int i = c.cur_pos - c.img_start;
      const float4* src4 = reinterpret_cast<const float4*>(logit_base + (size_t)i * kSlots);
      sp[i] = score(__ldcg(src4), __ldcg(src4 + 1));
    }
  }
}

// Launch with programmatic dependent launch: the grid may be scheduled while
// the previous kernel on the stream is still running. Before its
// griddepcontrol.wait it reads only what the previous kernel cannot be
// writing (lengths, block table, image range, K/V rows of earlier tokens)
// and, speculatively, the selection; q, the selection it keeps and the
// current token's K/V are read after the wait.
// A focal layer is two launches: the attend kernel, then the selection kernel.
template <typename T, int D, int MODE, int V>
cudaError_t launch_attend(const Params& p, cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pdl_config(dim3(p.splits, p.Hkv, p.B), dim3(32 * warps_for(V), 1, 1),
                                      attend_smem_bytes<T, D, V>(), stream, attr);
  attr[1].id = cudaLaunchAttributeClusterDimension;   // the splits of one (b, hkv)
  attr[1].val.clusterDim.x = p.splits;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attend_kernel<T, D, MODE, V>, p);
  if (e != cudaSuccess || MODE != kFocal) return e;
  cudaLaunchAttribute attr2[1];
  cudaLaunchConfig_t cfg2 = pdl_config(dim3(p.B, 1, 1), dim3(kSelectThreads, 1, 1),
                                       select_smem_bytes(p.max_img), stream, attr2);
  return cudaLaunchKernelEx(&cfg2, select_kernel<kSelectThreads>, p);
}

// The selection kernel on its own, on the scores p.sel_src describes.
inline cudaError_t launch_select_kernel(const Params& p, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(p.B, 1, 1), dim3(kSelectThreads, 1, 1),
                                      select_smem_bytes(p.max_img), stream, attr);
  return cudaLaunchKernelEx(&cfg, select_kernel<kSelectThreads>, p);
}

// Raise the dynamic shared-memory limits once per device, before any launch
// (so never inside a stream capture).
// Every kernel of the library asks for the largest shared-memory carveout, so
// that an SM never has to drain to change its shared-memory/L1 split between
// two of them (the kernels keep no data in L1).
template <typename Kern>
cudaError_t prepare_attend(Kern k, int bytes) {
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <typename T, int D, int V>
cudaError_t prepare_modes() {
  const int bytes = attend_smem_bytes<T, D, V>();
  cudaError_t e;
  if ((e = prepare_attend(attend_kernel<T, D, kFull, V>, bytes))) return e;
  if ((e = prepare_attend(attend_kernel<T, D, kFocal, V>, bytes))) return e;
  if ((e = prepare_attend(attend_kernel<T, D, kSparse, V>, bytes))) return e;
  if ((e = prepare_attend(attend_kernel<T, D, kProfile, V>, bytes))) return e;
  return prepare_attend(attend_kernel<T, D, kRswa, V>, bytes);
}

template <typename T, int D>
cudaError_t prepare_all_modes() {
  cudaError_t e;
  if ((e = prepare_modes<T, D, kGeneral>())) return e;
  if constexpr (variant_fits<T, D, kDeep>())
    if ((e = prepare_modes<T, D, kDeep>())) return e;
  if ((e = cudaFuncSetAttribute(select_kernel<kSelectThreads>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                select_smem_bytes(kMaxImg))))
    return e;
  return cudaFuncSetAttribute(select_kernel<kSelectThreads>,
                              cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

// How many clusters of `c` CTAs of the general variant the device holds at
// once (0 if a cluster of that size cannot be scheduled).
template <typename T, int D>
int active_clusters(int c) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c, 1, 1);
  cfg.blockDim = dim3(32 * warps_for(kGeneral), 1, 1);
  cfg.dynamicSmemBytes = attend_smem_bytes<T, D>();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = c;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, attend_kernel<T, D, kFull, kGeneral>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// Largest cluster (<= kMaxSplits) of variant V that the device can
// co-schedule (0: the variant does not exist for this dtype and head size).
template <typename T, int D, int V>
int max_cluster_size() {
  if constexpr (!variant_fits<T, D, V>()) {
    return 0;
  } else {
    for (int c = kMaxSplits; c > 1; c >>= 1) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(c, 1, 1);
      cfg.blockDim = dim3(32 * warps_for(V), 1, 1);
      cfg.dynamicSmemBytes = attend_smem_bytes<T, D, V>();
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = c;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, attend_kernel<T, D, kFull, V>, &cfg) == cudaSuccess && n > 0)
        return c;
      cudaGetLastError();
    }
    return 1;
  }
}

template <typename T, int D>
int max_cluster_of(int variant) {
  switch (variant) {
    case kGeneral: return max_cluster_size<T, D, kGeneral>();
    case kDeep: return max_cluster_size<T, D, kDeep>();
  }
  return 0;
}

template <typename T, int D, int V>
cudaError_t dispatch_variant(int mode, const Params& p, cudaStream_t s) {
  switch (mode) {
    case kFull: return launch_attend<T, D, kFull, V>(p, s);
    case kFocal: return launch_attend<T, D, kFocal, V>(p, s);
    case kSparse: return launch_attend<T, D, kSparse, V>(p, s);
    case kRswa: return launch_attend<T, D, kRswa, V>(p, s);
    case kProfile: return launch_attend<T, D, kProfile, V>(p, s);
  }
  return cudaErrorInvalidValue;
}

template <typename T, int D>
cudaError_t dispatch_mode(int mode, const Params& p, cudaStream_t s) {
  if constexpr (variant_fits<T, D, kDeep>())
    if (p.variant == kDeep) return dispatch_variant<T, D, kDeep>(mode, p, s);
  if (p.variant != kGeneral) return cudaErrorInvalidValue;
  return dispatch_variant<T, D, kGeneral>(mode, p, s);
}

}  // namespace fastocr
