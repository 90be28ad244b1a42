// Kernel body of the split-K decode attention (see attend_kernels.cuh for the
// design). Included by the per-dtype translation units, which instantiate it.
#pragma once

#include <math_constants.h>

#include "attend_kernels.cuh"

namespace fastocr {

// ---------------------------------------------------------------- top-k

// Sum the per-KV-head partial scores of sequence b into keys (shared memory),
// add the image mass to the profiler, and select the k largest keys (ties to
// the lower offset) with a 4-pass 8-bit radix select over the fp32 bit
// patterns (scores are >= 0, so the unsigned order is the float order). The
// selection is written in ascending position order.
static __device__ __noinline__ void score_and_select(const Params& p, int b, const AttendList& L,
                                 unsigned char* smem) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = L.n_img;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
  int* hist = reinterpret_cast<int*>(smem + TopkSmem::hist_offset(p.max_img));
  int* scratch = hist + 256;  // 64 ints

  double local = 0.0;
  for (int i = tid; i < n; i += kThreads) {
    float s = 0.f;
    for (int hk = 0; hk < p.Hkv; ++hk)
      s += __ldcg(p.sigma_part + ((size_t)b * p.Hkv + hk) * p.max_img + i);
    keys[i] = __float_as_uint(s);
    local += (double)s;
  }
  if (p.profile_layer >= 0) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
    double* dscr = reinterpret_cast<double*>(scratch + 32);
    if (lane == 0) dscr[warp] = local;
    __syncthreads();
    if (tid == 0) {
      double tot = 0.0;
      for (int w = 0; w < kWarps; ++w) tot += dscr[w];
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
    for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t key = keys[i];
      if ((key & mask) == prefix) atomicAdd(hist + ((key >> shift) & 255u), 1);
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
  const int per = ((n + kWarps - 1) / kWarps + 31) / 32 * 32;
  const int lo = warp * per, hi = min(n, lo + per);
  const uint32_t lt_mask = (1u << lane) - 1u;
  int gt = 0, eq = 0;
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < hi ? keys[i] : 0u;
    const bool ok = i < hi;
    gt += __popc(__ballot_sync(0xffffffffu, ok && key > thr));
    eq += __popc(__ballot_sync(0xffffffffu, ok && key == thr));
  }
  if (lane == 0) {
    scratch[8 + warp] = gt;
    scratch[16 + warp] = eq;
  }
  __syncthreads();
  int eq_before = 0, out_before = 0;
  {
    int eb = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int g_w = scratch[8 + w], e_w = scratch[16 + w];
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
  int bad = 0;
  const AttendList L = make_list<MODE>(p, b, bad);

  // this CTA's slice [r_lo, r_hi) of the attend list, in 16-token tiles
  int chunk = (L.n_att + p.splits - 1) / p.splits;
  chunk = (chunk + kTile - 1) / kTile * kTile;
  const int r_lo = split * chunk;
  const int r_hi = min(L.n_att, r_lo + chunk);
  const int n_tiles = r_hi > r_lo ? (r_hi - r_lo + kTile - 1) / kTile : 0;
  const int my_tiles = n_tiles > warp ? (n_tiles - warp + kWarps - 1) / kWarps : 0;

  const T* __restrict__ kg = static_cast<const T*>(p.k);
  const T* __restrict__ vg = static_cast<const T*>(p.v);
  const int32_t* __restrict__ bt = p.block_table + (size_t)b * p.max_pages;
  const int page_mask = (1 << p.log2_page) - 1;
  unsigned char* pipe = smem + warp * kStages * SM::kStageBytes;
  int* spos = reinterpret_cast<int*>(smem + SM::kPosOffset) + warp * kStages * kTile;

  // Stage tile j of this warp: lanes 0..15 resolve the cache rows, then the
  // warp copies 2 x 16 rows in 16-byte chunks (each instruction = whole rows).
  auto issue = [&](int j) {
    const int stage = j % kStages;
    const int base = r_lo + (warp + j * kWarps) * kTile;
    long long rowoff = -1;
    if (lane < kTile) {
      int pos = -1;
      const int v = base + lane;
      if (v < r_hi) {
        pos = list_pos<MODE>(L, v, bad);
        if (pos >= 0) {
          const int page = __ldg(bt + (pos >> p.log2_page));
          if (page < 0 || page >= p.num_pages) {
            bad |= kDevBadPage;
            pos = -1;
          } else {
            rowoff = ((((long long)page * p.Hkv + hkv) << p.log2_page) | (pos & page_mask)) * D;
          }
        }
      }
      spos[stage * kTile + lane] = pos;
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
      sm_.qf[ks][0] = have ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * tig)) : 0u;
      sm_.qf[ks][1] = have ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * tig)) : 0u;
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

#pragma unroll
  for (int j = 0; j < kStages - 1; ++j) {
    if (j < my_tiles) issue(j);
    cp_async_commit();
  }
  for (int it = 0; it < my_tiles; ++it) {
    if (it + kStages - 1 < my_tiles) issue(it + kStages - 1);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const int stage = it % kStages;
    unsigned char* kS = pipe + stage * SM::kStageBytes;
    unsigned char* vS = kS + kTile * ROWB;
    const int* tpos = spos + stage * kTile;

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
      const int posA = tpos[gid], posB = tpos[gid + 8];
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
      const int pos = tpos[r];
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

  const size_t unit = (size_t)b * p.Hkv + hkv;
  {
    float* pacc = p.part_acc + ((unit * kMaxSplits + split) * kSlots) * D;
    float* pml = p.part_ml + ((unit * kMaxSplits + split) * kSlots) * 2;
    for (int e = tid; e < p.g * D; e += kThreads) {
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
      pacc[h * D + d] = A;
      if (d == 0) {
        pml[2 * h] = M;
        pml[2 * h + 1] = Ls;
      }
    }
  }
  if (bad) atomicOr(p.status, bad);
  __threadfence();
  __syncthreads();
  int* misc = reinterpret_cast<int*>(smem + E::kMisc);
  if (tid == 0) misc[0] = atomicAdd(p.cnt_head + unit, 1) == p.splits - 1;
  __syncthreads();
  if (!misc[0]) return;
  __threadfence();
  if (tid == 0) p.cnt_head[unit] = 0;  // ready for the next launch

  // ---------------- last CTA of (b, hkv): merge the splits
  const int S = p.splits;
  float* sM = reinterpret_cast<float*>(smem + E::kM);
  float* sInvL = reinterpret_cast<float*>(smem + E::kInvL);
  float* sScale = reinterpret_cast<float*>(smem + E::kScale);   // [S][8] then m,l staging
  float* sml = wacc;                                             // [S][8][2] staging
  const float* pml_u = p.part_ml + (unit * kMaxSplits) * kSlots * 2;
  for (int e = tid; e < S * kSlots * 2; e += kThreads) sml[e] = __ldcg(pml_u + e);
  __syncthreads();
  for (int h = warp; h < p.g; h += kWarps) {
    float M = kNegInf;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, sml[(s * kSlots + h) * 2]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float base = M == kNegInf ? 0.f : M;
    float Ls = 0.f;
    for (int s = lane; s < S; s += 32)
      Ls += sml[(s * kSlots + h) * 2 + 1] * fast_exp2(sml[(s * kSlots + h) * 2] - base);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
    if (lane == 0) {
      sM[h] = base;
      sInvL[h] = Ls > 0.f ? __frcp_rn(Ls) : 0.f;
    }
  }
  __syncthreads();
  for (int e = tid; e < S * kSlots; e += kThreads) {
    const int s = e / kSlots, h = e % kSlots;
    sScale[e] = h < p.g ? fast_exp2(sml[e * 2] - sM[h]) * sInvL[h] : 0.f;
  }
  __syncthreads();
  {
    const float* pacc_u = p.part_acc + (unit * kMaxSplits) * kSlots * D;
    T* outp = static_cast<T*>(p.out) + ((size_t)b * p.Hq + (size_t)hkv * p.g) * D;
    for (int e = tid; e < p.g * D; e += kThreads) {
      const int h = e / D, d = e % D;
      float A0 = 0.f, A1 = 0.f, A2 = 0.f, A3 = 0.f;
      int s = 0;
      for (; s + 4 <= S; s += 4) {
        A0 = fmaf(__ldcg(pacc_u + ((size_t)(s + 0) * kSlots + h) * D + d), sScale[(s + 0) * kSlots + h], A0);
        A1 = fmaf(__ldcg(pacc_u + ((size_t)(s + 1) * kSlots + h) * D + d), sScale[(s + 1) * kSlots + h], A1);
        A2 = fmaf(__ldcg(pacc_u + ((size_t)(s + 2) * kSlots + h) * D + d), sScale[(s + 2) * kSlots + h], A2);
        A3 = fmaf(__ldcg(pacc_u + ((size_t)(s + 3) * kSlots + h) * D + d), sScale[(s + 3) * kSlots + h], A3);
      }
      for (; s < S; ++s)
        A0 = fmaf(__ldcg(pacc_u + ((size_t)s * kSlots + h) * D + d), sScale[s * kSlots + h], A0);
      const float o = (A0 + A1) + (A2 + A3);
      if constexpr (kMma)
        outp[h * D + d] = __float2bfloat16_rn(o);
      else
        outp[h * D + d] = o;
    }
  }
  if constexpr (MODE == kFocal) {

    // ---------------- focal: this group's share of the image scores
    {
      float Mh[kSlots], iL[kSlots];
#pragma unroll
      for (int h = 0; h < kSlots; ++h) {
        Mh[h] = h < p.g ? sM[h] : 0.f;
        iL[h] = h < p.g ? sInvL[h] : 0.f;
      }
      float* sp = p.sigma_part + unit * p.max_img;
      for (int i = tid; i < L.n_img; i += kThreads) {
        const float4 x0 = __ldcg(reinterpret_cast<const float4*>(logit_base + (size_t)i * kSlots));
        const float4 x1 = __ldcg(reinterpret_cast<const float4*>(logit_base + (size_t)i * kSlots + 4));
        const float x[kSlots] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        float sg = 0.f;
#pragma unroll
        for (int h = 0; h < kSlots; ++h)
          if (h < p.g) sg = fmaf(fast_exp2(x[h] - Mh[h]), iL[h], sg);
        sp[i] = sg;
      }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) misc[1] = atomicAdd(p.cnt_seq + b, 1) == p.Hkv - 1;
    __syncthreads();
    if (!misc[1]) return;
    __threadfence();
    if (tid == 0) p.cnt_seq[b] = 0;
    score_and_select(p, b, L, smem);
  }
}

template <typename T, int D, int MODE>
cudaError_t launch_attend(const Params& p, cudaStream_t stream) {
  const int smem = attend_smem_bytes<T, D>(MODE == kFocal ? p.max_img : 0);
  dim3 grid(p.splits, p.Hkv, p.B);
  attend_kernel<T, D, MODE><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

// Raise the dynamic shared-memory limit of every mode of one (T, D) once per
// device, before any launch (so never inside a stream capture).
template <typename T, int D>
cudaError_t prepare_all_modes() {
  const int bytes = attend_smem_bytes<T, D>(kMaxImg);
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(attend_kernel<T, D, kFull>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes))) return e;
  if ((e = cudaFuncSetAttribute(attend_kernel<T, D, kFocal>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes))) return e;
  if ((e = cudaFuncSetAttribute(attend_kernel<T, D, kSparse>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes))) return e;
  return cudaFuncSetAttribute(attend_kernel<T, D, kRswa>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
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
