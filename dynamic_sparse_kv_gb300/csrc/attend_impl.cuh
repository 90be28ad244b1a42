// Kernel body of the split-K decode attention (see attend_kernels.cuh for the
// design). Included by the per-dtype translation units, which instantiate it.
#pragma once

#include <math_constants.h>

#include "attend_kernels.cuh"

namespace fastocr {

// ---------------------------------------------------------------- top-k

// Image scores and selection of sequence b, run by one CTA of NT threads:
// sum the per-KV-head partial scores into keys (shared memory) in head order,
// add the image mass to the profiler, and select the k largest keys (ties to
// the lower offset) with a 4-pass 8-bit radix select over the fp32 bit
// patterns (scores are >= 0, so the unsigned order is the float order). The
// selection is written in ascending position order.
template <int NT>
__device__ __forceinline__ void score_and_select(const Params& p, int b, const AttendList& L,
                                                 unsigned char* smem) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = L.n_img;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
  int* hist = reinterpret_cast<int*>(smem + TopkSmem::hist_offset(p.max_img));
  int* scratch = hist + 256;                                   // 2*NW + 2 ints
  double* dscr = reinterpret_cast<double*>(scratch + 2 * NW + 2 + ((2 * NW + 2) & 1));

  double local = 0.0;
  const float* sp_b = p.sigma_part + (size_t)b * p.Hkv * p.max_img;
  for (int i0 = 0; i0 < n; i0 += 4 * NT) {
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    for (int hk0 = 0; hk0 < p.Hkv; hk0 += 4) {   // 16 loads in flight, summed in head order
      float v[4][4];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * NT + tid;
          v[c][u] = (hk0 + c < p.Hkv && i < n) ? __ldcg(sp_b + (size_t)(hk0 + c) * p.max_img + i) : 0.f;
        }
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (hk0 + c < p.Hkv) s[u] += v[c][u];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * NT + tid;
      if (i < n) {
        keys[i] = __float_as_uint(s[u]);
        local += (double)s[u];
      }
    }
  }
  if (p.profile_layer >= 0) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
    if (lane == 0) dscr[warp] = local;
    __syncthreads();
    if (tid == 0) {
      double tot = 0.0;
      for (int w = 0; w < NW; ++w) tot += dscr[w];
      atomicAdd(p.profile + p.profile_layer, tot);
    }
  }
  const int k = keep_count(p.tau, n);
  if (tid == 0) p.k_out[b] = k;
  __syncthreads();
  if (k == 0) return;

  // --- radix select of the k-th largest key
  uint32_t prefix = 0, mask = 0;
  int krem = k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += NT) hist[i] = 0;
    __syncthreads();
    for (int base = warp * 32; base < n; base += NT) {
      const int i = base + lane;
      const uint32_t key = i < n ? keys[i] : 0u;
      const bool act = i < n && (key & mask) == prefix;
      const uint32_t dig = act ? ((key >> shift) & 255u) : 256u;
      const uint32_t same = __match_any_sync(0xffffffffu, dig);
      if (act && lane == __ffs(same) - 1) atomicAdd(hist + dig, __popc(same));
    }
    __syncthreads();
    if (warp == 0) {
      // lane L scans bins 255-8L .. 248-8L (descending)
      int cnt[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = hist[255 - 8 * lane - j];
        tot += cnt[j];
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
    __syncthreads();
  }
  const uint32_t thr = prefix;  // the k-th largest key; krem of its copies are kept

  // --- stable compaction: warp w owns offsets [w*per, (w+1)*per), read 32 at a time
  const int per = ((n + NW - 1) / NW + 31) / 32 * 32;
  const int lo = warp * per, hi = min(n, lo + per);
  const uint32_t lt_mask = (1u << lane) - 1u;
  int gt = 0, eq = 0;
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const bool ok = i < hi;
    const uint32_t key = ok ? keys[i] : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, ok && key > thr));
    eq += __popc(__ballot_sync(0xffffffffu, ok && key == thr));
  }
  if (lane == 0) {
    scratch[2 + warp] = gt;
    scratch[2 + NW + warp] = eq;
  }
  __syncthreads();
  int eq_before = 0, out_before = 0;
  {
    int eb = 0;
    for (int w = 0; w < NW; ++w) {
      const int g_w = scratch[2 + w], e_w = scratch[2 + NW + w];
      int take = krem - eb;
      take = take < 0 ? 0 : (take > e_w ? e_w : take);
      if (w < warp) out_before += g_w + take;
      if (w == warp) eq_before = eb;
      eb += e_w;
    }
  }
  int32_t* dst = p.idx_out + (size_t)b * p.idx_stride;
  int eq_run = eq_before, out_run = out_before;
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const bool ok = i < hi;
    const uint32_t key = ok ? keys[i] : 0u;
    const bool is_gt = ok && key > thr, is_eq = ok && key == thr;
    const uint32_t eq_b = __ballot_sync(0xffffffffu, is_eq);
    const int my_eq_rank = eq_run + __popc(eq_b & lt_mask);
    const bool take = is_gt || (is_eq && my_eq_rank < krem);
    const uint32_t take_b = __ballot_sync(0xffffffffu, take);
    if (take) dst[out_run + __popc(take_b & lt_mask)] = L.img_start + i;
    eq_run += __popc(eq_b);
    out_run += __popc(take_b);
  }
}

constexpr int kSelectThreads = 1024;

// Selection kernel of a focal layer: one CTA of 1024 threads per sequence,
// launched right after the focal attend kernel (which left the per-KV-head
// partial scores in the workspace).
template <int NT>
__global__ void __launch_bounds__(NT) select_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem[];
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  int bad = 0;  // already reported by the attend kernel
  const AttendList L = make_list<kFocal>(p, blockIdx.x, bad);
  score_and_select<NT>(p, blockIdx.x, L, smem);
}

inline int select_smem_bytes(int max_img) {
  return TopkSmem::hist_offset(max_img) + 256 * 4 + (2 * (kSelectThreads / 32) + 4) * 4 +
         (kSelectThreads / 32) * 8 + 16;
}

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

template <typename T, int D, int MODE>
__global__ void __launch_bounds__(kThreads, 2) attend_kernel(const Params p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  using SM = Smem<T, D>;
  using E = EpiSmem<D>;
  constexpr bool kMma = sizeof(T) == 2;
  constexpr int ROWB = SM::kRowBytes;
  constexpr int CH = ROWB / 16;                 // 16-byte chunks per row
  constexpr int kElemPerChunk = 16 / (int)sizeof(T);
  const float kNegInf = -CUDART_INF_F;

  const int split = blockIdx.x, hkv = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const T* __restrict__ kg = static_cast<const T*>(p.k);
  const T* __restrict__ vg = static_cast<const T*>(p.v);
  const int32_t* __restrict__ bt = p.block_table + (size_t)b * p.max_pages;
  const int page_mask = (1 << p.log2_page) - 1;

  // While the previous kernel on the stream may still run (programmatic
  // dependent launch), warm L2 with this CTA's K/V rows, computed from a
  // speculative read of the lengths, block table and selection. These reads
  // only choose prefetch addresses (validated, never used for results), and
  // every global read below bypasses L1, so stale values cannot leak in.
  {
    int ignore = 0;
    const AttendList Ls = make_list<MODE>(p, b, ignore);
    int ch = (Ls.n_att + p.splits - 1) / p.splits;
    ch = (ch + kTile - 1) / kTile * kTile;
    const int lo = split * ch, hi = min(Ls.n_att, lo + ch);
    const uint32_t page_bytes = (uint32_t)(D * sizeof(T)) << p.log2_page;
    auto prefetch_positions = [&](int pos_lo, int pos_hi) {
      if (pos_hi <= pos_lo) return;
      const int pg1 = (pos_hi - 1) >> p.log2_page;
      for (int j = (pos_lo >> p.log2_page) + tid; j <= pg1; j += kThreads) {
        const int page = __ldcg(bt + j);
        if (page >= 0 && page < p.num_pages) {
          const size_t off = ((size_t)page * p.Hkv + hkv) * ((size_t)D << p.log2_page);
          prefetch_l2(kg + off, page_bytes);
          prefetch_l2(vg + off, page_bytes);
        }
      }
    };
    prefetch_positions(lo, min(hi, Ls.n_pre));
    const int sel_end = Ls.n_pre + Ls.n_sel;
    if (MODE == kSparse) {
      for (int v = max(lo, Ls.n_pre) + tid; v < min(hi, sel_end); v += kThreads) {
        const int pos = __ldcg(Ls.sel + (v - Ls.n_pre));
        if (pos < Ls.img_start || pos >= Ls.img_start + Ls.n_img) continue;
        const int page = __ldcg(bt + (pos >> p.log2_page));
        if (page < 0 || page >= p.num_pages) continue;
        const size_t off =
            ((((size_t)page * p.Hkv + hkv) << p.log2_page) | (size_t)(pos & page_mask)) * D;
        prefetch_l2(kg + off, D * sizeof(T));
        prefetch_l2(vg + off, D * sizeof(T));
      }
    }
    const int t_lo = max(lo, sel_end), t_hi = hi;
    if (t_hi > t_lo)
      prefetch_positions(Ls.tail_start + (t_lo - sel_end), Ls.tail_start + (t_hi - sel_end));
  }

  // wait until the previous kernel on the stream has completed and its
  // writes are visible (no-op when launched without the PDL attribute)
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if (p.pdl_early) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  int bad = 0;
  const AttendList L = make_list<MODE>(p, b, bad);

  // this CTA's slice [r_lo, r_hi) of the attend list
  int chunk = (L.n_att + p.splits - 1) / p.splits;
  chunk = (chunk + kTile - 1) / kTile * kTile;
  const int r_lo = split * chunk;
  const int r_hi = min(L.n_att, r_lo + chunk);

  unsigned char* pipe = smem + warp * kStages * SM::kStageBytes;
  int* srow = reinterpret_cast<int*>(smem + SM::kRowOffset);

  // Resolve list entries [rlo, rhi) (at most kSliceMax) to cache rows
  // (page * H_kv + hkv) * page_size + slot, -1 if masked, into shared memory.
  // All lookups of a thread are issued before any is used, so a round costs
  // two memory latencies (selection, then block table) instead of two per tile.
  auto resolve = [&](int rlo, int rhi) {
    constexpr int kPer = kSliceMax / kThreads;
    int pos[kPer], page[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int v = rlo + tid + j * kThreads;
      pos[j] = v < rhi ? list_pos<MODE>(L, v, bad) : -1;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) page[j] = pos[j] >= 0 ? __ldcg(bt + (pos[j] >> p.log2_page)) : -1;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int v = rlo + tid + j * kThreads;
      if (v >= rhi) continue;
      int row = -1;
      if (pos[j] >= 0) {
        if (page[j] < 0 || page[j] >= p.num_pages)
          bad |= kDevBadPage;
        else
          row = ((page[j] * p.Hkv + hkv) << p.log2_page) | (pos[j] & page_mask);
      }
      srow[v - rlo] = row;
    }
  };

  // Stage tile j (of this warp, within the current round) into its pipeline
  // slot: 2 x 16 rows in 16-byte chunks, each instruction covering whole rows.
  auto issue = [&](int j, int n_round) {
    const int stage = j % kStages;
    const int base = (warp + j * kWarps) * kTile;
    long long rowoff = -1;
    if (lane < kTile && base + lane < n_round) {
      const int row = srow[base + lane];
      rowoff = row >= 0 ? (long long)row * D : -1;
    }
    const uint32_t sb = smem_u32(pipe + stage * SM::kStageBytes);
#pragma unroll
    for (int i = 0; i < 2 * kTile * CH / 32; ++i) {
      const int c = i * 32 + lane;
      const int kv = c / (kTile * CH);
      const int rem = c % (kTile * CH);
      const int row = rem / CH, ch = rem % CH;
      const long long ro = __shfl_sync(0xffffffffu, rowoff, row);
      const T* src = (kv == 0 ? kg : vg) + (ro < 0 ? 0 : ro) + ch * kElemPerChunk;
      const uint32_t dst = sb + kv * (kTile * ROWB) + row * ROWB + ((ch ^ (row & 7)) << 4);
      cp_async16(dst, src, ro < 0 ? 0 : 16);
    }
  };

  float* logit_base = nullptr;
  if (MODE == kFocal)
    logit_base = p.logits + ((size_t)b * p.Hkv + hkv) * (size_t)p.max_img * kSlots;

  // ---------------- per-warp streaming
  WarpStateMma<D> sm_;
  WarpStateF32<D> sf_;
  const int gid = lane >> 2, tig = lane & 3;
  if constexpr (kMma) {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sm_.acc[mt][e] = 0.f;
    sm_.m[0] = sm_.m[1] = kNegInf;
    sm_.l[0] = sm_.l[1] = 0.f;
    const bool have = gid < p.g;
    const T* qrow = static_cast<const T*>(p.q) + ((size_t)b * p.Hq + hkv * p.g + (have ? gid : 0)) * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      sm_.qf[ks][0] = have ? __ldcg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * tig)) : 0u;
      sm_.qf[ks][1] = have ? __ldcg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * tig)) : 0u;
    }
  } else {
    float* qs = reinterpret_cast<float*>(smem + SM::kQOffset);
    for (int e = tid; e < kSlots * D; e += kThreads) {
      const int h = e / D, d = e % D;
      qs[e] = h < p.g ? static_cast<const float*>(p.q)[((size_t)b * p.Hq + hkv * p.g + h) * D + d] : 0.f;
    }
#pragma unroll
    for (int h = 0; h < kSlots; ++h) {
      sf_.m[h] = kNegInf;
      sf_.l[h] = 0.f;
#pragma unroll
      for (int j = 0; j < D / 32; ++j) sf_.acc[h][j] = 0.f;
    }
    __syncthreads();
  }

  for (int rlo = r_lo; rlo < r_hi; rlo += kSliceMax) {
  const int n_round = min(r_hi - rlo, kSliceMax);
  resolve(rlo, rlo + n_round);
  __syncthreads();
  const int n_tiles = (n_round + kTile - 1) / kTile;
  const int my_tiles = n_tiles > warp ? (n_tiles - warp + kWarps - 1) / kWarps : 0;
#pragma unroll
  for (int j = 0; j < kStages - 1; ++j) {
    if (j < my_tiles) issue(j, n_round);
    cp_async_commit();
  }
  for (int it = 0; it < my_tiles; ++it) {
    if (it + kStages - 1 < my_tiles) issue(it + kStages - 1, n_round);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const int stage = it % kStages;
    unsigned char* kS = pipe + stage * SM::kStageBytes;
    unsigned char* vS = kS + kTile * ROWB;
    const int tbase = (warp + it * kWarps) * kTile;    // tile start within the round

    if constexpr (kMma) {
      // S^T[16 keys x 8 heads] = K[16 x D] . Q^T[D x 8]
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t kA = smem_u32(kS), vA = smem_u32(vS);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int row = (lane & 7) + (lane & 8);
        const int ch = 2 * ks + (lane >> 4);
        uint32_t a[4];
        ldmatrix_x4(a, kA + row * ROWB + ((ch ^ (row & 7)) << 4));
        mma_bf16(c, a, sm_.qf[ks][0], sm_.qf[ks][1]);
      }
      // list position of tokens gid / gid+8 (= cache position in focal mode), -1 if masked
      const int posA = (tbase + gid < n_round && srow[tbase + gid] >= 0) ? rlo + tbase + gid : -1;
      const int posB = (tbase + gid + 8 < n_round && srow[tbase + gid + 8] >= 0) ? rlo + tbase + gid + 8 : -1;
      const float s0 = posA >= 0 ? c[0] * p.scale_log2 : kNegInf;
      const float s1 = posA >= 0 ? c[1] * p.scale_log2 : kNegInf;
      const float s2 = posB >= 0 ? c[2] * p.scale_log2 : kNegInf;
      const float s3 = posB >= 0 ? c[3] * p.scale_log2 : kNegInf;
      if (MODE == kFocal) {
        if (posA >= L.img_start && posA < L.img_start + L.n_img)
          *reinterpret_cast<float2*>(logit_base + (size_t)(posA - L.img_start) * kSlots + 2 * tig) =
              make_float2(s0, s1);
        if (posB >= L.img_start && posB < L.img_start + L.n_img)
          *reinterpret_cast<float2*>(logit_base + (size_t)(posB - L.img_start) * kSlots + 2 * tig) =
              make_float2(s2, s3);
      }
      const float mx0 = warp_max_gid(fmaxf(s0, s2));
      const float mx1 = warp_max_gid(fmaxf(s1, s3));
      const float mn0 = fmaxf(sm_.m[0], mx0), mn1 = fmaxf(sm_.m[1], mx1);
      const float b0f = mn0 == kNegInf ? 0.f : mn0, b1f = mn1 == kNegInf ? 0.f : mn1;
      const float al0 = fast_exp2(sm_.m[0] - b0f), al1 = fast_exp2(sm_.m[1] - b1f);
      const float p0 = fast_exp2(s0 - b0f), p2 = fast_exp2(s2 - b0f);
      const float p1 = fast_exp2(s1 - b1f), p3 = fast_exp2(s3 - b1f);
      sm_.l[0] = sm_.l[0] * al0 + (p0 + p2);
      sm_.l[1] = sm_.l[1] * al1 + (p1 + p3);
      sm_.m[0] = mn0;
      sm_.m[1] = mn1;
      // P^T[16 keys x 8 heads] as the B operand: transpose the two 8x8 blocks
      const uint32_t bb0 = movmatrix_trans(pack_bf16(p0, p1));
      const uint32_t bb1 = movmatrix_trans(pack_bf16(p2, p3));
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        sm_.acc[mt][0] *= al0;
        sm_.acc[mt][1] *= al1;
        sm_.acc[mt][2] *= al0;
        sm_.acc[mt][3] *= al1;
        const int row = (lane & 7) + ((lane >> 4) << 3);
        const int ch = 2 * mt + ((lane >> 3) & 1);
        uint32_t a[4];
        ldmatrix_x4_trans(a, vA + row * ROWB + ((ch ^ (row & 7)) << 4));
        // O^T[16 dims x 8 heads] += V^T[16 dims x 16 keys] . P^T[16 keys x 8 heads]
        mma_bf16(sm_.acc[mt], a, bb0, bb1);
      }
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
      const int pos = (tbase + r < n_round && srow[tbase + r] >= 0) ? rlo + tbase + r : -1;
#pragma unroll
      for (int h = 0; h < kSlots; ++h) {
        s[h] += __shfl_xor_sync(0xffffffffu, s[h], 16);
        s[h] = pos >= 0 ? s[h] * p.scale_log2 : kNegInf;
      }
      if (MODE == kFocal) {
        if (half == 0 && pos >= L.img_start && pos < L.img_start + L.n_img) {
          float* dst = logit_base + (size_t)(pos - L.img_start) * kSlots;
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
  cp_async_wait<0>();
  __syncthreads();   // before the next round overwrites the row list
  }
  cp_async_wait<0>();
  // the next kernel may now be scheduled; it waits for this grid to finish
  if (!p.pdl_early) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  __syncthreads();

  // ---------------- CTA merge of the four warps -> split partial
  float* wm = reinterpret_cast<float*>(smem + E::kWm);
  float* wl = reinterpret_cast<float*>(smem + E::kWl);
  float* wacc = reinterpret_cast<float*>(smem + E::kWacc);
  if constexpr (kMma) {
    const float l0 = warp_sum_gid(sm_.l[0]), l1 = warp_sum_gid(sm_.l[1]);
    const int h0 = warp * kSlots + 2 * tig, h1 = h0 + 1;
    if (gid == 0) {
      wm[h0] = sm_.m[0];
      wm[h1] = sm_.m[1];
      wl[h0] = l0;
      wl[h1] = l1;
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
#pragma unroll
      for (int j = 0; j < D / 32; ++j) wacc[(warp * kSlots + h) * D + lane + 32 * j] = sf_.acc[h][j];
    }
  }
  __syncthreads();

  // ---------------- this CTA's partial (m, l, acc) of every head slot, in shared memory
  float* cm = reinterpret_cast<float*>(smem + E::kPartM);
  float* cl = reinterpret_cast<float*>(smem + E::kPartL);
  float* cacc = reinterpret_cast<float*>(smem + E::kPartAcc);
  for (int e = tid; e < kSlots * D; e += kThreads) {
    const int h = e / D, d = e % D;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * kSlots + h]);
    const float base = M == kNegInf ? 0.f : M;
    float A = 0.f, Ls = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float sc = fast_exp2(wm[w * kSlots + h] - base);
      A = fmaf(wacc[(w * kSlots + h) * D + d], sc, A);
      Ls = fmaf(wl[w * kSlots + h], sc, Ls);
    }
    cacc[e] = A;
    if (d == 0) {
      cm[h] = M;
      cl[h] = Ls;
    }
  }
  if (bad) atomicOr(p.status, bad);
  // The CTAs of one (sequence, KV head) form a thread-block cluster; the split
  // partials are merged through distributed shared memory. Global writes of
  // this CTA (focal logits) are fenced before the cluster barrier so that the
  // other CTAs of the cluster read them after it.
  if (MODE == kFocal) __threadfence();
  __syncthreads();
  cluster_sync();

  const int S = p.splits;               // == cluster size
  const uint32_t rank = cluster_ctarank();
  float* sM = reinterpret_cast<float*>(smem + E::kM);
  float* sInvL = reinterpret_cast<float*>(smem + E::kInvL);
  float* sScale = reinterpret_cast<float*>(smem + E::kScale);  // [S][8]
  float* rml = reinterpret_cast<float*>(smem + E::kRemoteMl);   // [S][8][2]
  for (int e = tid; e < S * kSlots; e += kThreads) {
    const int s = e / kSlots, h = e % kSlots;
    rml[2 * e] = ld_dsmem_f32(cm + h, s);
    rml[2 * e + 1] = ld_dsmem_f32(cl + h, s);
  }
  __syncthreads();
  if (tid < kSlots) {
    const int h = tid;
    float M = kNegInf;
    for (int s = 0; s < S; ++s) M = fmaxf(M, rml[2 * (s * kSlots + h)]);
    const float base = M == kNegInf ? 0.f : M;
    float Ls = 0.f;
    for (int s = 0; s < S; ++s)
      Ls = fmaf(rml[2 * (s * kSlots + h) + 1], fast_exp2(rml[2 * (s * kSlots + h)] - base), Ls);
    sM[h] = base;
    sInvL[h] = Ls > 0.f ? __frcp_rn(Ls) : 0.f;
  }
  __syncthreads();
  for (int e = tid; e < S * kSlots; e += kThreads) {
    const int h = e % kSlots;
    sScale[e] = fast_exp2(rml[2 * e] - sM[h]) * sInvL[h];
  }
  __syncthreads();

  // ---------------- outputs: CTA `rank` owns a slice of the (head, 4-dim) pairs
  {
    constexpr int C4 = D / 4;
    const int n_pairs = p.g * C4;
    const int per = (n_pairs + S - 1) / S;
    const int e_hi = min(n_pairs, (int)(rank + 1) * per);
    T* outp = static_cast<T*>(p.out) + ((size_t)b * p.Hq + (size_t)hkv * p.g) * D;
    for (int e = (int)rank * per + tid; e < e_hi; e += kThreads) {
      const int h = e / C4, c4 = e % C4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s0 = 0; s0 < S; s0 += 8) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          v[u] = s0 + u < S ? ld_dsmem_f32x4(cacc + h * D + 4 * c4, s0 + u)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float sc = s0 + u < S ? sScale[(s0 + u) * kSlots + h] : 0.f;
          acc.x = fmaf(v[u].x, sc, acc.x);
          acc.y = fmaf(v[u].y, sc, acc.y);
          acc.z = fmaf(v[u].z, sc, acc.z);
          acc.w = fmaf(v[u].w, sc, acc.w);
        }
      }
      T* o = outp + h * D + 4 * c4;
      if constexpr (kMma) {
        uint2 w;
        w.x = pack_bf16(acc.x, acc.y);
        w.y = pack_bf16(acc.z, acc.w);
        *reinterpret_cast<uint2*>(o) = w;
      } else {
        *reinterpret_cast<float4*>(o) = acc;
      }
    }
  }

  // ---------------- focal: this group's share of the image scores, split over the cluster
  if constexpr (MODE == kFocal) {
    float Mh[kSlots], iL[kSlots];
#pragma unroll
    for (int h = 0; h < kSlots; ++h) {
      Mh[h] = h < p.g ? sM[h] : 0.f;
      iL[h] = h < p.g ? sInvL[h] : 0.f;
    }
    const size_t unit = (size_t)b * p.Hkv + hkv;
    float* sp = p.sigma_part + unit * p.max_img;
    const int nper = (L.n_img + S - 1) / S;
    const int i_lo = (int)rank * nper, i_hi = min(L.n_img, i_lo + nper);
    for (int i0 = i_lo; i0 < i_hi; i0 += 4 * kThreads) {
      float4 x[4][2];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kThreads + tid;
        const float4* src4 = reinterpret_cast<const float4*>(logit_base + (size_t)i * kSlots);
        x[u][0] = i < i_hi ? __ldcg(src4) : make_float4(0.f, 0.f, 0.f, 0.f);
        x[u][1] = i < i_hi ? __ldcg(src4 + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kThreads + tid;
        const float xv[kSlots] = {x[u][0].x, x[u][0].y, x[u][0].z, x[u][0].w,
                                  x[u][1].x, x[u][1].y, x[u][1].z, x[u][1].w};
        float sg = 0.f;
#pragma unroll
        for (int h = 0; h < kSlots; ++h)
          if (h < p.g) sg = fmaf(fast_exp2(xv[h] - Mh[h]), iL[h], sg);
        if (i < i_hi) sp[i] = sg;
      }
    }
  }
  // no CTA may leave while another still reads its shared memory
  cluster_sync();
}

// Launch with programmatic dependent launch: the grid may be scheduled while
// the previous kernel on the stream finishes its epilogue; it waits for that
// kernel's completion (griddepcontrol.wait) before reading any global memory.
// A focal layer is two launches: the attend kernel, then the selection kernel.
template <typename T, int D, int MODE>
cudaError_t launch_attend(const Params& p, cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pdl_config(dim3(p.splits, p.Hkv, p.B), dim3(kThreads, 1, 1),
                                      attend_smem_bytes<T, D>(), stream, attr);
  attr[1].id = cudaLaunchAttributeClusterDimension;   // the splits of one (b, hkv)
  attr[1].val.clusterDim.x = p.splits;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attend_kernel<T, D, MODE>, p);
  if (e != cudaSuccess || MODE != kFocal) return e;
  cudaLaunchAttribute attr2[1];
  cudaLaunchConfig_t cfg2 = pdl_config(dim3(p.B, 1, 1), dim3(kSelectThreads, 1, 1),
                                       select_smem_bytes(p.max_img), stream, attr2);
  return cudaLaunchKernelEx(&cfg2, select_kernel<kSelectThreads>, p);
}

// Raise the dynamic shared-memory limits once per device, before any launch
// (so never inside a stream capture).
template <typename Kern>
cudaError_t prepare_attend(Kern k, int bytes) {
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <typename T, int D>
cudaError_t prepare_all_modes() {
  const int bytes = attend_smem_bytes<T, D>();
  cudaError_t e;
  if ((e = prepare_attend(attend_kernel<T, D, kFull>, bytes))) return e;
  if ((e = prepare_attend(attend_kernel<T, D, kFocal>, bytes))) return e;
  if ((e = prepare_attend(attend_kernel<T, D, kSparse>, bytes))) return e;
  if ((e = prepare_attend(attend_kernel<T, D, kRswa>, bytes))) return e;
  return cudaFuncSetAttribute(select_kernel<kSelectThreads>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              select_smem_bytes(kMaxImg));
}

// Largest cluster (<= kMaxSplits) of this kernel that the device can co-schedule.
template <typename T, int D>
int max_cluster_size() {
  for (int c = kMaxSplits; c > 1; c >>= 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = attend_smem_bytes<T, D>();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attend_kernel<T, D, kFull>, &cfg) == cudaSuccess && n > 0)
      return c;
    cudaGetLastError();
  }
  return 1;
}

template <typename T, int D>
cudaError_t dispatch_mode(int mode, const Params& p, cudaStream_t s) {
  switch (mode) {
    case kFull: return launch_attend<T, D, kFull>(p, s);
    case kFocal: return launch_attend<T, D, kFocal>(p, s);
    case kSparse: return launch_attend<T, D, kSparse>(p, s);
    case kRswa: return launch_attend<T, D, kRswa>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fastocr
