// moe_route.cu -- host C ABI (include/moe_route.h) and the routing,
// permutation, gather and output kernels of the fused MoE layer forward.
//
// Launch sequence of moe_forward on the caller's stream:
//   route_kernel    a-1 routing (warp per token, NaN -> -FLT_MAX in
//                   registers, k rounds of warp arg-max with ties to the
//                   lower expert index) + per-CTA expert histogram and the
//                   rank of each pick among equal ids in its CTA
//   scan_kernel     a-2/a-3: per-expert totals, exclusive scans, per-CTA
//                   bases and the token-tile work list (single CTA)
//   gather_kernel   a-2: slot of every pick, src/pos, permuted activation
//                   rows (FP8: quantised once per token, 128-column groups)
//   grouped GEMMs   a-4/a-5 gate+up with SiLU, a-6/a-7 down with the routing
//                   weight (grouped_gemm.cu): one launch when both GEMMs share
//                   a tile list, else one launch each
//   combine_kernel  a-7: out[t] = sum over j of the token's k weighted rows,
//                   in pick order (fp32 sum, deterministic)
// No atomics are used to count or place rows: a pick's rank is the number of
// equal ids before it in its routing CTA, the CTA's count of an expert is
// written once (by that expert's last pick there, as rank + 1), the scan
// adds the CTAs' counts in CTA order, and every slot follows from those.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/moe_route.h"
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kRouteThreads = 256;  // 8 warps
constexpr int kMaxK = 32;
constexpr int kMaxE = 1024;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per pipeline wait
constexpr int kTmMinEst = 32;  // FP8 plans from this estimate on run token-major
constexpr int kHotRows = 256;  // rows of an expert that select CTA pairs on the device

// ------------------------------------------------------------------ routing
__device__ __forceinline__ float sanitize_logit(float v) {
  // NaN -> -FLT_MAX (PR #39593, "Fix"); +-Inf -> +-FLT_MAX so weights stay finite
  if (isnan(v)) return -FLT_MAX;
  if (isinf(v)) return v > 0.0f ? FLT_MAX : -FLT_MAX;
  return v;
}

// Order-preserving unsigned key of a sanitised (finite) logit: a > b as
// floats exactly when key(a) > key(b), with -0 taken as +0 (they compare
// equal as floats).  Every finite value maps above 0, so 0 can stand for
// "no candidate".  Warp maxima and minima of these keys are single
// reduction instructions (redux.sync) instead of shuffle ladders.
__device__ __forceinline__ uint32_t logit_key(float v) {
  const uint32_t b = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

__device__ __forceinline__ float load_logit(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load_logit(const __nv_bfloat16* p) {
  return __bfloat162float(p[0]);
}

// Values per logits load in routing: as many of a lane's VPT values as fit
// 16 bytes (1: one logit per load)
template <int VPT, typename LT>
__host__ __device__ constexpr int vec_width() {
  return (16 / static_cast<int>(sizeof(LT))) < VPT ? 16 / static_cast<int>(sizeof(LT)) : VPT;
}

// W consecutive logits of row t from expert e0 (the address aligned to W
// elements), as floats
template <typename LT, int W>
__device__ __forceinline__ void load_logits(const LT* __restrict__ row, int e0, float (&out)[W]) {
  if constexpr (W == 1) {
    out[0] = load_logit(row + e0);
  } else if constexpr (sizeof(LT) == 4) {  // f32: W in {2, 4}
    if constexpr (W == 4) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(row + e0));
      out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
    } else {
      const float2 a = __ldg(reinterpret_cast<const float2*>(row + e0));
      out[0] = a.x; out[1] = a.y;
    }
  } else {  // bf16: W in {2, 4, 8}
    uint32_t raw[W / 2];
    if constexpr (W == 8) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(row + e0));
      raw[0] = a.x; raw[1] = a.y; raw[2] = a.z; raw[3] = a.w;
    } else if constexpr (W == 4) {
      const uint2 a = __ldg(reinterpret_cast<const uint2*>(row + e0));
      raw[0] = a.x; raw[1] = a.y;
    } else {
      raw[0] = __ldg(reinterpret_cast<const unsigned int*>(row + e0));
    }
#pragma unroll
    for (int j = 0; j < W / 2; ++j) {
      out[2 * j] = __uint_as_float(raw[j] << 16);              // low half: the lower expert
      out[2 * j + 1] = __uint_as_float(raw[j] & 0xffff0000u);  // high half
    }
  }
}

// One token's routing by one warp (a-1): sanitised logits of token t, an
// optional group mask, k rounds of warp arg-max (ties to the lower expert
// index), then softmax or sigmoid weights, renormalised when asked.  Lanes
// j < k end with pick j's expert (my_id) and weight (my_w).  Lane `lane`
// holds value i of expert (i / W) * 32W + lane * W + i % W: its experts
// ascend with i, and W consecutive experts come from one load.
template <int VPT, typename LT, int W>
__device__ __forceinline__ void route_token(const LT* __restrict__ logits, int t, int E, int k,
                                            int scoring, int renorm, int n_group, int topk_group,
                                            int lane, int& my_id, float& my_w) {
  auto expert = [&](int i) { return (i / W) * 32 * W + lane * W + i % W; };
  const LT* row = logits + static_cast<size_t>(t) * E;
  float v[VPT];
#pragma unroll
  for (int b = 0; b < VPT / W; ++b) {
    const int e0 = b * 32 * W + lane * W;
    float part[W];
    if (e0 < E) {  // with W > 1, E is a multiple of W: the whole load is in the row
      load_logits<LT, W>(row, e0, part);
    } else {
#pragma unroll
      for (int j = 0; j < W; ++j) part[j] = 0.0f;
    }
#pragma unroll
    for (int j = 0; j < W; ++j) v[b * W + j] = sanitize_logit(part[j]);
  }
  uint32_t vk[VPT];  // the logits' order keys (0: no expert in this slot)
#pragma unroll
  for (int i = 0; i < VPT; ++i) vk[i] = (expert(i) < E) ? logit_key(v[i]) : 0u;
  uint32_t taken = 0;
  if (n_group > 1) {
    // group-limited routing: lane g holds the key of the largest sanitised
    // logit of group g; keep the topk_group best groups (ties to the lower
    // group) and exclude the other groups' experts below
    const int gs = E / n_group;
    uint32_t my_gkey = 0;
    for (int g = 0; g < n_group; ++g) {
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int e = expert(i);
        if (e < E && e / gs == g) m = max(m, vk[i]);
      }
      m = __reduce_max_sync(0xffffffffu, m);
      if (lane == g) my_gkey = m;
    }
    uint32_t kept = 0;
    bool mine_kept = false;
    for (int r = 0; r < topk_group; ++r) {
      const uint32_t ck = (lane < n_group && !mine_kept) ? my_gkey : 0u;
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, ck);
      const uint32_t g = __reduce_min_sync(0xffffffffu, (ck == kmax) ? lane : 0xffffffffu);
      kept |= 1u << g;
      if (lane == static_cast<int>(g)) mine_kept = true;
    }
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int e = expert(i);
      if (e < E && !((kept >> (e / gs)) & 1u)) taken |= 1u << i;
    }
  }
  float my_v = 0.0f;
  for (int j = 0; j < k; ++j) {
    // this lane's best remaining expert (lane-local experts ascend with i,
    // so '>' keeps the lower index on ties), then the warp's: the largest
    // key, and among lanes holding it the lowest expert index
    uint32_t bk = 0;
    uint32_t bi = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      if (!((taken >> i) & 1u) && vk[i] > bk) {
        bk = vk[i];
        bi = static_cast<uint32_t>(expert(i));
      }
    }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t best = __reduce_min_sync(0xffffffffu, (bk == kmax) ? bi : 0xffffffffu);
    // the winner's lane and its slot in that lane
    const uint32_t wl = (best / W) % 32u, wi = (best / (32u * W)) * W + best % W;
    if (wl == static_cast<uint32_t>(lane)) taken |= 1u << wi;
    if (lane == j) {
      my_id = static_cast<int>(best);
      my_v = key_logit(kmax);
    }
  }
  // weights
  const float vmax = __shfl_sync(0xffffffffu, my_v, 0);  // pick 0 is the row maximum
  float score = 0.0f;
  if (scoring == 0) {
    if (renorm) {
      score = (lane < k) ? expf(my_v - vmax) : 0.0f;  // the full-row sum cancels
    } else {
      float z = 0.0f;
#pragma unroll
      for (int i = 0; i < VPT; ++i)
        if (expert(i) < E) z += expf(v[i] - vmax);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
      score = (lane < k) ? expf(my_v - vmax) / z : 0.0f;
    }
  } else {
    score = (lane < k) ? 1.0f / (1.0f + expf(-my_v)) : 0.0f;
  }
  if (renorm) {
    float den = score;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    my_w = (den > 0.0f && isfinite(den)) ? score / den : 1.0f / static_cast<float>(k);
  } else {
    my_w = score;
  }
}

// mode 0: routing only; 1: routing + histogram; 2: validate caller ids + histogram
template <int VPT, typename LT>
__global__ void __launch_bounds__(VPT <= 8 ? 1024 : kRouteThreads, 1)
    route_kernel(const LT* __restrict__ logits, int T, int E, int k, int scoring, int renorm,
                 int tpc, int mode, const int* __restrict__ ids_in, const float* __restrict__ w_in,
                 int* __restrict__ ids, float* __restrict__ w, int* __restrict__ chunk_counts,
                 int* __restrict__ lrank, unsigned* __restrict__ err, int e_base, int e_local,
                 int n_group, int topk_group) {
  extern __shared__ int sid[];  // [tpc * k] picks of this CTA's tokens, then [e_local] counts
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int t0 = blockIdx.x * tpc;
  const int ntok = min(tpc, T - t0);

  for (int tl = warp; tl < ntok; tl += nwarps) {
    const int t = t0 + tl;
    int my_id = -1;
    float my_w = 0.0f;
    if (mode != 2) {
      // logits read W to a load when the row length and the pointer allow
      // it (W consecutive experts per lane per load), else one per load;
      // the picks are the same either way
      constexpr int WV = vec_width<VPT, LT>();
      const bool vec = WV > 1 && E % WV == 0 &&
                       (reinterpret_cast<uintptr_t>(logits) % (WV * sizeof(LT))) == 0;
      if (vec)
        route_token<VPT, LT, WV>(logits, t, E, k, scoring, renorm, n_group, topk_group, lane,
                                 my_id, my_w);
      else
        route_token<VPT, LT, 1>(logits, t, E, k, scoring, renorm, n_group, topk_group, lane,
                                my_id, my_w);
    } else {
      // caller-supplied picks: an id outside [0, E) or repeated within the
      // token is reported and skipped rather than used as an index
      int id = (lane < k) ? ids_in[static_cast<size_t>(t) * k + lane] : -1;
      const float wt = (lane < k) ? w_in[static_cast<size_t>(t) * k + lane] : 0.0f;
      unsigned bad = 0;
      if (lane < k && (id < 0 || id >= E)) {
        bad |= 1u;
        id = -1;
      }
      for (int j = 0; j < kMaxK; ++j) {
        const int other = __shfl_sync(0xffffffffu, id, j);
        if (j < lane && lane < k && id >= 0 && other == id) {
          bad |= 2u;
          id = -1;
        }
      }
      if (bad) atomicOr(err, bad);
      my_id = id;
      my_w = wt;
    }
    if (lane < k) {
      ids[static_cast<size_t>(t) * k + lane] = my_id;
      w[static_cast<size_t>(t) * k + lane] = my_w;
      // histogram and permutation see this rank's experts only (local index);
      // picks of other expert-parallel ranks' experts are skipped (-1)
      if (mode != 0)
        sid[tl * k + lane] =
            (my_id >= e_base && my_id < e_base + e_local) ? my_id - e_base : -1;
    }
  }
  if (mode == 0) return;
  __syncthreads();

  // each pick's rank among the equal ids before it (a warp per pick, its
  // lanes splitting the CTA's picks), and this CTA's per-expert counts: the
  // last pick of an expert in the CTA (no equal id after it) is its only
  // writer, and stores rank + 1
  const int n = ntok * k;
  int* cnt = sid + tpc * k;
  for (int e = threadIdx.x; e < e_local; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  for (int f = warp; f < n; f += nwarps) {
    const int e = sid[f];
    int r = 0;
    bool later = false;
    for (int g = lane; g < n; g += 32) {
      const bool same = sid[g] == e;
      r += (g < f && same);
      later |= (g > f && same);
    }
    r = __reduce_add_sync(0xffffffffu, r);
    later = __any_sync(0xffffffffu, later);
    if (lane == 0) {
      lrank[static_cast<size_t>(t0) * k + f] = (e >= 0) ? r : -1;
      if (e >= 0 && !later) cnt[e] = r + 1;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < e_local; e += blockDim.x)
    chunk_counts[static_cast<size_t>(blockIdx.x) * e_local + e] = cnt[e];
}

// ------------------------------------------------------------------ scan
// Block-wide exclusive scan of one int per thread (blockDim = 1024).
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += y;
    }
    warp_sums[lane] = s;  // inclusive
    if (lane == 31) *total = s;
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  __syncthreads();
  return before;
}

// Token-tile width of an expert with `cnt` rows: the plan's tile (from the
// rows-per-expert estimate) is the floor; with per_expert set, an expert
// with more rows gets the smallest of 32 / 64 / 128 / 256 that covers them,
// capped at n_max (256 for prefill-sized plans, else 128), so hot experts
// of concentrated routing read each weight block once per n_max rows
// instead of once per `tile_n` rows.
__device__ __forceinline__ int expert_tile(int cnt, int tile_n, int per_expert, int n_max) {
  if (!per_expert) return tile_n;
  int n = cnt <= 16 ? 16 : cnt <= 32 ? 32 : cnt <= 64 ? 64 : cnt <= 128 ? 128 : 256;
  n = n > tile_n ? n : tile_n;
  return n < n_max ? n : n_max;
}

// Writes one token-tile list per grouped GEMM: list 1 with widths up to
// n_max1 (GEMM1), list 2 up to n_max2 (GEMM2); when the caps agree list 2
// is not written and GEMM2 reads list 1.
// With heavy_first, the experts that fill at least one whole tile come
// first (in expert order), then the rest: a grid-stride walk over the list
// then deals the long items out evenly before the short ones.
// An expert that needs several tiles has its rows split evenly over them
// (rounded up to 16; at most the width): a tile's MMAs take time in
// proportion to its rows above a floor (about N/2 cycles for N > 92 per
// 128-row MMA), so 288 rows as 144 + 144 finish well before 256 + 32 would,
// with the same weight traffic.
__device__ void write_tile_list(int e, int E, int cnt, int off, int ne, int max_tiles,
                               bool heavy_first, int* warp_sums, int* tot, int4* tiles,
                               int* ntiles, unsigned* err) {
  const int ntl = (cnt + ne - 1) / ne;
  const int step = ntl > 1 ? min(ne, (((cnt + ntl - 1) / ntl) + 15) & ~15) : ne;
  int tstart;
  if (heavy_first) {
    const bool heavy = cnt >= ne;
    __shared__ int tot_heavy;
    const int hs = block_exclusive_scan(heavy ? ntl : 0, warp_sums, &tot_heavy);
    const int ls = block_exclusive_scan(heavy ? 0 : ntl, warp_sums, tot);
    tstart = heavy ? hs : tot_heavy + ls;
    if (e == 0) *tot += tot_heavy;
    __syncthreads();
  } else {
    tstart = block_exclusive_scan(ntl, warp_sums, tot);
  }
  if (e == 0) {
    if (*tot > max_tiles) atomicOr(err, 8u);
    *ntiles = min(*tot, max_tiles);
  }
  if (e < E)
    for (int i = 0; i < ntl && tstart + i < max_tiles; ++i)
      tiles[tstart + i] = make_int4(e, off + i * step, min(step, cnt - i * step), ne);
}

__global__ void __launch_bounds__(1024)
    scan_kernel(const int* __restrict__ chunk_counts, int n_chunks, int E, int tile_n,
                int per_expert, int n_max1, int n_max2, int max_tiles,
                int* __restrict__ chunk_base, int* __restrict__ counts,
                int* __restrict__ offsets, int4* __restrict__ tiles1, int* __restrict__ ntiles1,
                int4* __restrict__ tiles2, int* __restrict__ ntiles2, int* __restrict__ dep,
                int heavy_first, unsigned* __restrict__ err, unsigned* __restrict__ hint,
                int hot_rows, unsigned* __restrict__ family) {
  __shared__ int warp_sums[32];
  pdl_trigger();
  pdl_wait();
  // fused-GEMM tile counters and the two work counters that follow them
  for (int i = threadIdx.x; i < max_tiles + 2; i += blockDim.x) dep[i] = 0;
  __shared__ int tot_rows, tot_tiles1, tot_tiles2;
  const int e = threadIdx.x;
  int cnt = 0;
  if (e < E) {
    for (int c = 0; c < n_chunks; ++c) {
      const size_t i = static_cast<size_t>(c) * E + e;
      chunk_base[i] = cnt;
      cnt += chunk_counts[i];
    }
    counts[e] = cnt;
  }
  const int off = block_exclusive_scan(cnt, warp_sums, &tot_rows);
  if (e < E) offsets[e] = off;
  if (e == 0) offsets[E] = tot_rows;
  // how many of the local experts this call routes to, for the next call's
  // GEMM (see GemmArgs::spec_hint), tagged so that stale workspace bytes
  // never read as a count
  const int tch = __syncthreads_count(e < E && cnt > 0);
  if (threadIdx.x == 0)
    st_relaxed_gpu(hint, kSpecHintTag | static_cast<unsigned>(min(tch, 0xffff)));
  // Plans that choose the GEMM kernel family here (hot_rows > 0): an expert
  // with at least hot_rows rows (a whole 256-row CTA-pair tile) selects the
  // CTA-pair kernels and their tile list (widths up to 256, heavy experts
  // first); otherwise the single-CTA list the host asked for.  Concentrated
  // routing (H20 article, paras. 4 and 6) is the case this serves.
  if (hot_rows > 0) {
    const bool hot = __syncthreads_or(e < E && cnt >= hot_rows) != 0;
    if (threadIdx.x == 0) *family = hot ? kFamilyPair : kFamilySingle;
    if (hot) {
      n_max1 = n_max2 = 256;
      heavy_first = 1;
    }
  }
  write_tile_list(e, E, cnt, off, expert_tile(cnt, tile_n, per_expert, n_max1), max_tiles,
                  heavy_first, warp_sums, &tot_tiles1, tiles1, ntiles1, err);
  if (n_max2 != n_max1)
    write_tile_list(e, E, cnt, off, expert_tile(cnt, tile_n, per_expert, n_max2), max_tiles,
                    heavy_first, warp_sums, &tot_tiles2, tiles2, ntiles2, err);
}

// ------------------------------------------------------------------ gather
// One warp per (token t, 256 columns): the slots of t's k picks (slot =
// offset[e] + chunk base + rank among equal ids in the routing CTA), src /
// pos, and t's activation columns copied (FP8: quantised once per token,
// 128-column groups = 16 lanes x 8 values) into each of the k permuted rows.
// QT: 0 copy f32, 1 copy bf16, 2 quantise bf16 -> e4m3
template <int QT>
__global__ void __launch_bounds__(256)
    gather_kernel(const void* __restrict__ x, const int* __restrict__ ids,
                  const int* __restrict__ lrank, const int* __restrict__ chunk_base,
                  const int* __restrict__ offsets, int T, int H, int k, int tpc, int e_base,
                  int e_local, int* __restrict__ src, int* __restrict__ pos,
                  void* __restrict__ xq, float* __restrict__ xs) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int chunks = (H + 255) / 256;
  const long long g = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (g >= static_cast<long long>(T) * chunks) return;
  const int t = static_cast<int>(g / chunks);
  const int c = static_cast<int>(g % chunks);

  int my_slot = -1;
  if (lane < k) {
    const size_t f = static_cast<size_t>(t) * k + lane;
    const int eg = ids[f];  // global id; -1 = skipped pick
    const int e = eg - e_base;
    if (eg >= 0 && e >= 0 && e < e_local)
      my_slot = offsets[e] + chunk_base[static_cast<size_t>(t / tpc) * e_local + e] + lrank[f];
    if (c == 0) {
      pos[f] = my_slot;
      if (my_slot >= 0) src[my_slot] = static_cast<int>(f);
    }
  }
  const int h0 = c * 256 + lane * 8;
  const bool active = h0 < H;
  if constexpr (QT == 0) {
    float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
    const float* xr = static_cast<const float*>(x) + static_cast<size_t>(t) * H + h0;
    if (active) {
      v0 = __ldg(reinterpret_cast<const float4*>(xr));
      v1 = __ldg(reinterpret_cast<const float4*>(xr) + 1);
    }
    for (int j = 0; j < k; ++j) {
      const int s = __shfl_sync(0xffffffffu, my_slot, j);
      if (s >= 0 && active) {
        float4* d = reinterpret_cast<float4*>(static_cast<float*>(xq) + static_cast<size_t>(s) * H + h0);
        d[0] = v0;
        d[1] = v1;
      }
    }
  } else if constexpr (QT == 1) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (active)
      v = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(x) +
                                               static_cast<size_t>(t) * H + h0));
    for (int j = 0; j < k; ++j) {
      const int s = __shfl_sync(0xffffffffu, my_slot, j);
      if (s >= 0 && active)
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(xq) + static_cast<size_t>(s) * H +
                                  h0) = v;
    }
  } else {
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (active) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(
          static_cast<const __nv_bfloat16*>(x) + static_cast<size_t>(t) * H + h0));
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = __low2float(b2[i]);
        v[2 * i + 1] = __high2float(b2[i]);
      }
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
#pragma unroll
    for (int off = 8; off > 0; off >>= 1)  // 16 lanes = one 128-column group
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float scale = __fdiv_rn(fmaxf(m, 1e-10f), 448.0f);
    uint2 packed = make_uint2(0u, 0u);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float q = __fdiv_rn(v[i], scale);
      q = fmaxf(fminf(q, 448.0f), -448.0f);
      const uint32_t code = __nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3);
      if (i < 4)
        packed.x |= code << (8 * i);
      else
        packed.y |= code << (8 * (i - 4));
    }
    const int groups = H / 128;
    for (int j = 0; j < k; ++j) {
      const int s = __shfl_sync(0xffffffffu, my_slot, j);
      if (s >= 0 && active) {
        *reinterpret_cast<uint2*>(static_cast<uint8_t*>(xq) + static_cast<size_t>(s) * H + h0) =
            packed;
        if ((lane & 15) == 0) xs[static_cast<size_t>(s) * groups + h0 / 128] = scale;
      }
    }
  }
}

// ------------------------------------------------------------------ output
// a-7: out[t, h] = sum over j = 0..k-1 of ybuf[pos[t*k + j], h], where the
// rows already carry the routing weight.  One warp per (token, 256 columns),
// 8 columns per lane, fp32 sum in pick order; skipped picks (pos < 0) add
// nothing.
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 r = __ldg(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __low2float(b[i]);
    v[2 * i + 1] = __high2float(b[i]);
  }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 r;
  __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) b[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = r;
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// RB rows' loads in flight per lane: 4 for small batches (too few warps to
// hide the load latency otherwise), 1 when the warps alone fill the GPU
// (measured: eight in flight at T=4096 took 61 us against 35 with one)
template <typename YT, int RB>
__global__ void __launch_bounds__(256)
    combine_kernel(const YT* __restrict__ ybuf, const int* __restrict__ pos, int T, int H, int k,
                   YT* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int chunks = (H + 255) / 256;
  const long long g = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (g >= static_cast<long long>(T) * chunks) return;
  const int t = static_cast<int>(g / chunks);
  const int h0 = static_cast<int>(g % chunks) * 256 + lane * 8;
  const bool active = h0 < H;
  // the token's k rows: positions read once per warp, then RB rows' loads
  // in flight at a time; the sum keeps pick order
  const int my_pos = lane < k ? __ldg(pos + static_cast<size_t>(t) * k + lane) : -1;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j0 = 0; j0 < k; j0 += RB) {
    float v[RB][8];
    bool use[RB];
#pragma unroll
    for (int u = 0; u < RB; ++u) {
      const int p = __shfl_sync(0xffffffffu, my_pos, (j0 + u) & 31);
      use[u] = active && j0 + u < k && p >= 0;
      if (use[u]) load8(ybuf + static_cast<size_t>(p) * H + h0, v[u]);
    }
#pragma unroll
    for (int u = 0; u < RB; ++u)
      if (use[u]) {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += v[u][i];
      }
  }
  if (active) store8(out + static_cast<size_t>(t) * H + h0, acc);
}

// ------------------------------------------------------------------ host helpers
static int vpt_for(int E) {
  const int v = (E + 31) / 32;
  if (v <= 1) return 1;
  if (v <= 2) return 2;
  if (v <= 4) return 4;
  if (v <= 8) return 8;
  if (v <= 16) return 16;
  return 32;
}

// threads of a routing CTA: one warp per token of the chunk while the
// logits of a row fit in 8 registers per lane (E <= 256), else 8 warps
static int route_threads(int vpt, int tpc) { return vpt <= 8 ? 32 * tpc : kRouteThreads; }

template <typename LT>
static void launch_route_t(int vpt, dim3 grid, size_t smem, cudaStream_t st, const LT* logits,
                           int T, int E, int k, int scoring, int renorm, int tpc, int mode,
                           const int* ids_in, const float* w_in, int* ids, float* w, int* cc,
                           int* lr, unsigned* err, int e_base, int e_local, int n_group = 1,
                           int topk_group = 1) {
#define MOE_ROUTE_CASE(V)                                                                      \
  case V:                                                                                      \
    launch_chained(route_kernel<V, LT>, grid, dim3(route_threads(V, tpc)), smem, st, logits, T, \
                   E, k, scoring, renorm, tpc, mode, ids_in, w_in, ids, w, cc, lr, err, e_base, \
                   e_local, n_group, topk_group);                                              \
    break;
  switch (vpt) {
    MOE_ROUTE_CASE(1)
    MOE_ROUTE_CASE(2)
    MOE_ROUTE_CASE(4)
    MOE_ROUTE_CASE(8)
    MOE_ROUTE_CASE(16)
    MOE_ROUTE_CASE(32)
  }
#undef MOE_ROUTE_CASE
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D K-major tensor map: inner = K elements, rows; box = 128 bytes x box_rows
static bool make_tmap(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize,
                      uint64_t inner, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * static_cast<uint64_t>(esize)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D K-major tensor map over w13 [E, 2I, H] seen as [2E planes, I rows, H]
// (plane 2e is expert e's gate rows, 2e+1 its up rows); box = 128 bytes x 128
// rows x 2 planes, so one copy brings a feature block's gate and up rows
static bool make_tmap_gate_up(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize,
                              uint64_t H, uint64_t I, uint64_t EL) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {H, I, 2 * EL};
  cuuint64_t strides[2] = {H * static_cast<uint64_t>(esize), I * H * static_cast<uint64_t>(esize)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esize), 128, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The TMA tensor maps of one forward: weights (w13, w2) and the permuted
// token rows (xq, act) at every box height, plus the half-height token maps
// of CTA-pair plans.  A map only encodes an address, a shape and a box, so
// an entry stays valid for as long as the caller passes the same pointers
// with the same shapes (also when a buffer is freed and another of the same
// shape is allocated at the same address).
struct MapKey {
  int dev, kind, H, I, EL, pair;
  long long R;
  const void *w13, *w2, *xq, *act;
  bool operator==(const MapKey& o) const {
    return dev == o.dev && kind == o.kind && H == o.H && I == o.I && EL == o.EL &&
           pair == o.pair && R == o.R && w13 == o.w13 && w2 == o.w2 && xq == o.xq &&
           act == o.act;
  }
};
struct MapSet {
  GemmMaps m1, m2, h1, h2;  // h1/h2: half-height token maps (CTA pairs)
  GemmMaps t1, t2;          // FP8 token-major: 256 weight rows per copy
};

static bool encode_maps(const MapKey& key, MapSet* s) {
  const int esize = key.kind == KIND_TF32 ? 4 : key.kind == KIND_BF16 ? 2 : 1;
  const CUtensorMapDataType dt = key.kind == KIND_TF32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : key.kind == KIND_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  bool ok = make_tmap(&s->m1.a, key.w13, dt, esize, key.H, static_cast<uint64_t>(key.EL) * 2 * key.I,
                      128) &&
            make_tmap(&s->m2.a, key.w2, dt, esize, key.I, static_cast<uint64_t>(key.EL) * key.H,
                      128);
  for (int i = 0; i < kTokMaps && ok; ++i) {  // token boxes 16 .. 256 rows
    const uint32_t rows = 16u << i;
    ok = make_tmap(&s->m1.b[i], key.xq, dt, esize, key.H, key.R, rows) &&
         make_tmap(&s->m2.b[i], key.act, dt, esize, key.I, key.R, rows);
  }
  s->h1 = s->m1;
  s->h2 = s->m2;
  for (int i = 0; i < kTokMaps && ok && key.pair; ++i) {  // half tiles 8 .. 128 rows
    const uint32_t rows = 8u << i;
    ok = make_tmap(&s->h1.b[i], key.xq, dt, esize, key.H, key.R, rows) &&
         make_tmap(&s->h2.b[i], key.act, dt, esize, key.I, key.R, rows);
  }
  s->t1 = s->m1;
  s->t2 = s->m2;
  if (ok && key.kind == KIND_E4M3)
    ok = make_tmap_gate_up(&s->t1.a, key.w13, dt, esize, key.H, key.I, key.EL) &&
         make_tmap(&s->t2.a, key.w2, dt, esize, key.I, static_cast<uint64_t>(key.EL) * key.H, 256);
  return ok;
}

// A small cache of encoded map sets, most recently used first; host threads
// may call concurrently.  The copy out is taken under the lock.
static bool cached_maps(const MapKey& key, MapSet* out) {
  constexpr int kEntries = 16;
  static MapKey keys[kEntries];
  static MapSet sets[kEntries];
  static int used = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i) {
    if (keys[i] == key) {
      *out = sets[i];
      if (i > 0) {  // move to the front
        const MapKey kk = keys[i];
        const MapSet ss = sets[i];
        for (int j = i; j > 0; --j) {
          keys[j] = keys[j - 1];
          sets[j] = sets[j - 1];
        }
        keys[0] = kk;
        sets[0] = ss;
      }
      return true;
    }
  }
  MapSet s;
  if (!encode_maps(key, &s)) return false;
  if (used < kEntries) ++used;
  for (int j = used - 1; j > 0; --j) {  // the least recently used entry drops out
    keys[j] = keys[j - 1];
    sets[j] = sets[j - 1];
  }
  keys[0] = key;
  sets[0] = s;
  *out = s;
  return true;
}

static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int max_stages(int na, int n_max, int kblocks, bool fp8) {
  const int budget = 227 * 1024 - gemm_extra_smem(n_max, kblocks, fp8);
  int s = budget / gemm_stage_bytes(na, n_max);
  return s > 8 ? 8 : s;
}

// TMEM accumulator slots: two per-tile accumulators (double buffer) for
// BF16/TF32, one when a tile's accumulators take all 512 columns; for FP8 one slot per 128-K block, as many as 512 columns hold
// (up to 16), so the MMAs can run ahead of the scale-folding epilogue.
static int slots_for(int na, int n_max, bool fp8) {
  int s = 512 / (na * n_max);
  if (!fp8) return s >= 2 ? 2 : 1;  // a 2 x 256-column G1 tile fills TMEM alone
  return s > 16 ? 16 : s;
}

static uint32_t tmem_cols_for(int need) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(need)) c <<= 1;
  return c;
}

static int plan_ok(const moe_plan_t* p) {
  return p && p->abi_version == MOE_ABI_VERSION && p->T >= 0 && p->E >= 1 && p->k >= 1 &&
         p->tile_n >= 16 && p->ep_size >= 1 && p->e_local >= 1 &&
         p->e_local * p->ep_size == p->E && p->ep_rank >= 0 && p->ep_rank < p->ep_size &&
         p->n_group >= 1 && p->topk_group >= 1;
}

// the common forward; ids_in/w_in non-null selects caller-supplied routing
static int forward_impl(const moe_plan_t* p, const void* x, const void* logits, const int* ids_in,
                        const float* w_in, const void* w13, const float* s13, const void* w2,
                        const float* s2, void* out, void* ws, size_t ws_bytes, void* stream,
                        void* const* events = nullptr, bool with_ids = false) {
  if (!plan_ok(p)) return MOE_ERR_INVALID_ARG;
  const bool fp8 = p->dtype == MOE_DTYPE_FP8_BLOCK128;
  if (p->T == 0) return MOE_OK;  // empty batch: nothing to read or write
  if (!x || !w13 || !w2 || !out || !ws) return MOE_ERR_INVALID_ARG;
  if (with_ids ? (!ids_in || !w_in) : !logits) return MOE_ERR_INVALID_ARG;
  if (fp8 != (s13 != nullptr) || fp8 != (s2 != nullptr)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w13) || !aligned16(w2) || !aligned16(out) || !aligned16(ws))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < p->workspace_bytes) return MOE_ERR_WORKSPACE;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  auto at = [&](uint64_t off) { return static_cast<void*>(wsb + off); };
  unsigned* err = static_cast<unsigned*>(at(p->off_err));
  int* ids = static_cast<int*>(at(p->off_ids));
  float* topw = static_cast<float*>(at(p->off_w));
  int* chunk_counts = static_cast<int*>(at(p->off_chunk_counts));
  int* lrank = static_cast<int*>(at(p->off_lrank));
  int* counts = static_cast<int*>(at(p->off_counts));
  int* offsets = static_cast<int*>(at(p->off_offsets));
  int* chunk_base = static_cast<int*>(at(p->off_chunk_base));
  int* src = static_cast<int*>(at(p->off_src));
  int* pos = static_cast<int*>(at(p->off_pos));
  int4* tiles = static_cast<int4*>(at(p->off_tiles));
  int* ntiles = static_cast<int*>(at(p->off_ntiles));
  int4* tiles2 = static_cast<int4*>(at(p->off_tiles2));
  int* ntiles2 = static_cast<int*>(at(p->off_ntiles2));
  int* dep = static_cast<int*>(at(p->off_dep));
  void* xq = at(p->off_xq);
  float* xs = static_cast<float*>(at(p->off_xs));
  void* act = at(p->off_act);
  float* as = static_cast<float*>(at(p->off_as));
  void* ybuf = at(p->off_y);

  const int T = p->T, H = p->H, I = p->I, E = p->E, k = p->k;
  const int EL = p->e_local, e_base = p->ep_rank * p->e_local;  // this rank's experts
  const long long R = static_cast<long long>(T) * k;
  auto mark = [&](int i) {
    if (events) cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st);
  };
  if (cudaMemsetAsync(err, 0, sizeof(unsigned), st) != cudaSuccess) return MOE_ERR_CUDA;
  mark(0);

  // a-1 routing (+ histogram)
  const size_t route_smem = static_cast<size_t>(p->route_tpc * k + EL) * sizeof(int);
  const int mode = with_ids ? 2 : 1;
  if (p->dtype == MOE_DTYPE_F32)
    launch_route_t<float>(vpt_for(E), dim3(p->n_chunks), route_smem, st,
                          static_cast<const float*>(logits), T, E, k, p->scoring, p->renorm,
                          p->route_tpc, mode, ids_in, w_in, ids, topw, chunk_counts, lrank, err,
                          e_base, EL, p->n_group, p->topk_group);
  else
    launch_route_t<__nv_bfloat16>(vpt_for(E), dim3(p->n_chunks), route_smem, st,
                                  static_cast<const __nv_bfloat16*>(logits), T, E, k, p->scoring,
                                  p->renorm, p->route_tpc, mode, ids_in, w_in, ids, topw,
                                  chunk_counts, lrank, err, e_base, EL, p->n_group, p->topk_group);
  mark(1);
  // a-2 / a-3 scan and tile list
  // FP8 kernels are specialised per tile width.  When experts average more
  // than half the plan's tile (est > tile_n / 2, so that many hold more
  // rows than the tile), the kernel is one size wider (at most 64) and each
  // expert's tile grows to the rows it holds: fewer tiles, each weight block
  // streamed once per expert instead of once per tile.
  // Token-major FP8 plans (gemm_tm) tile every expert's rows by 128: the
  // tokens sit on the MMA's M side.
  const bool tm = fp8 && p->gemm_tm != 0;
  const int fp8_nt = (fp8 && 2 * p->est > p->tile_n && p->tile_n < 64) ? 2 * p->tile_n : p->tile_n;
  const int per_expert = tm ? 0 : fp8 ? (fp8_nt > p->tile_n ? 1 : 0) : 1;
  const int scan_tile = tm ? 128 : p->tile_n;
  // the largest tile the device may choose per GEMM.  One CTA per tile:
  // GEMM1 keeps two 2 x n-column accumulators in TMEM, so 128 is its widest
  // double-buffered tile; GEMM2 (one accumulator) widens hot experts to 256
  // tokens in prefill-sized plans (est > 64).  CTA pairs: 256 for both
  // (each CTA holds half of the tile's rows).
  const bool pair_plan = p->gemm_pair != 0 && !fp8;
  const int NM1 = tm ? 128 : pair_plan ? 256 : fp8 ? fp8_nt : 128;
  const int NM2 = tm ? 128 : pair_plan ? 256 : fp8 ? fp8_nt : (p->tile_n >= 128 ? 256 : 128);
  // BF16/F32 plans that run one CTA per tile and one fused launch, with
  // enough tokens for an expert to fill a 256-row CTA-pair tile, choose the
  // kernel family on the device, from the rows the experts actually hold
  const bool dyn = p->gemm_dyn != 0 && !fp8 && !pair_plan && p->est <= 32 && NM1 == NM2;
  unsigned* family = err + 2;
  launch_chained(scan_kernel, dim3(1), dim3(1024), 0, st, chunk_counts, p->n_chunks, EL, scan_tile,
                 per_expert, NM1, NM2, p->max_tiles, chunk_base, counts, offsets, tiles, ntiles,
                 tiles2, ntiles2, dep, pair_plan ? 1 : 0, err, err + 1, dyn ? kHotRows : 0,
                 family);
  mark(2);
  // a-2 gather
  const long long gwarps = static_cast<long long>(T) * ((H + 255) / 256);
  const unsigned gblocks = static_cast<unsigned>((gwarps * 32 + 255) / 256);
  if (p->dtype == MOE_DTYPE_F32)
    launch_chained(gather_kernel<0>, dim3(gblocks), dim3(256), 0, st, x, ids, lrank, chunk_base,
                   offsets, T, H, k, p->route_tpc, e_base, EL, src, pos, xq, xs);
  else if (p->dtype == MOE_DTYPE_BF16)
    launch_chained(gather_kernel<1>, dim3(gblocks), dim3(256), 0, st, x, ids, lrank, chunk_base,
                   offsets, T, H, k, p->route_tpc, e_base, EL, src, pos, xq, xs);
  else
    launch_chained(gather_kernel<2>, dim3(gblocks), dim3(256), 0, st, x, ids, lrank, chunk_base,
                   offsets, T, H, k, p->route_tpc, e_base, EL, src, pos, xq, xs);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  mark(3);

  // a-4 .. a-7 grouped GEMMs
  const int kind = p->dtype == MOE_DTYPE_F32 ? KIND_TF32
                   : p->dtype == MOE_DTYPE_BF16 ? KIND_BF16 : KIND_E4M3;
  const int esize = kind == KIND_TF32 ? 4 : kind == KIND_BF16 ? 2 : 1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  const bool pair = pair_plan || dyn;  // the CTA-pair maps are needed
  MapSet ms;
  if (!cached_maps(MapKey{dev, kind, H, I, EL, pair ? 1 : 0, R, w13, w2, xq, act}, &ms))
    return MOE_ERR_CUDA;
  const GemmMaps& m1 = ms.m1;
  const GemmMaps& m2 = ms.m2;

  const int sms = sm_count();
  if (sms <= 0) return MOE_ERR_CUDA;
  const int kb1 = H / (128 / esize), kb2 = I / (128 / esize);
  const int kbmax = kb1 > kb2 ? kb1 : kb2;
  if (tm) {
    // token-major FP8: GEMM1 items are one 128-feature block (gate and up
    // rows) x one 128-row token tile; GEMM2 items 256 output rows x one tile
    GemmArgs g{};
    g.p[0] = GemmPhase{tiles, ntiles, 2, 128, I / 128, H / 128, 2 * I, I, I, s13, 2 * I / 128, xs};
    g.p[1] = GemmPhase{tiles, ntiles, 2, 256, (H + 255) / 256, I / 128, H, 128, H, s2, H / 128,
                       as};
    g.R = static_cast<int>(R);
    g.act = act;
    g.act_scale = as;
    g.I = I;
    g.src = src;
    g.topw = topw;
    g.ybuf = ybuf;
    g.H = H;
    g.err = err;
    g.limit_ns = kWaitLimitNs;
    for (int mode = 1; mode <= 2; ++mode) {
      const int st_max = (227 * 1024 - tm_smem_bytes(mode, 0)) / kTmStageBytes;
      g.stages = st_max > 8 ? 8 : st_max;
      const int smem = tm_smem_bytes(mode, g.stages);
      const long long items = static_cast<long long>(p->max_tiles) * g.p[mode - 1].mblocks;
      const int grid = static_cast<int>(items < sms ? items : sms);
      // GEMM1 reads x rows and stores act rows with TMA; GEMM2 reads act rows
      // (its y rows go out with plain stores)
      if (launch_grouped_gemm_tm(mode, g, mode == 1 ? ms.t1 : ms.t2, m2, grid, smem, st) !=
          cudaSuccess)
        return MOE_ERR_CUDA;
      mark(3 + mode);
    }
  } else {
    // CTA-pair launches (GEMM1 then GEMM2) and single-CTA launches (one
    // fused, or GEMM1 then GEMM2); `want` non-zero: the launch runs only if
    // this call's scan chose that family; `marks`: record the GEMM events
    auto run_pair = [&](unsigned want, bool marks) -> bool {
      // CTA pairs: half-height token maps, items of 256 weight rows, one
      // token tile list (widths up to 256) for both GEMMs
      const GemmMaps& h1 = ms.h1;
      const GemmMaps& h2 = ms.h2;
      GemmArgs g{};
      g.p[0] = GemmPhase{tiles, ntiles, 2, 256, (I + 255) / 256, kb1, 2 * I, I, I, nullptr, 0,
                         nullptr};
      g.p[1] = GemmPhase{tiles, ntiles, 1, 256, (H + 255) / 256, kb2, H, 128, H, nullptr, 0,
                         nullptr};
      g.R = static_cast<int>(R);
      g.act = act;
      g.I = I;
      g.src = src;
      g.topw = topw;
      g.ybuf = ybuf;
      g.H = H;
      g.err = err;
      g.limit_ns = kWaitLimitNs;
      g.family = want ? family : nullptr;
      g.family_want = want;
      g.n_max = 256;
      auto launch_pair = [&](int mode, const GemmMaps& maps) -> bool {
        const int na = mode == 1 ? 2 : 1;
        g.run1 = mode == 1;
        g.run2 = mode == 2;
        g.na_max = na;
        const int budget = 227 * 1024 - kPairExtraSmem;
        const int sb = gemm_pair_stage_bytes(na, g.n_max, mode == 1 ? 1 : 2);
        g.stages = budget / sb > 8 ? 8 : budget / sb;
        g.nslots = 512 / (na * g.n_max) >= 2 ? 2 : 1;
        g.tmem_cols = 512;
        const int smem = g.stages * sb + kPairExtraSmem;
        const long long items = static_cast<long long>(p->max_tiles) * g.p[mode - 1].mblocks;
        return launch_grouped_gemm_pair(kind, mode, g, maps, smem, items, st) == cudaSuccess;
      };
      if (!launch_pair(1, h1)) return false;
      if (marks) mark(4);
      if (!launch_pair(2, h2)) return false;
      if (marks) mark(5);
      return true;
    };
    auto run_single = [&](unsigned want, bool marks) -> bool {
      GemmArgs g{};
      g.p[0] = GemmPhase{tiles, ntiles, 2, 128, p->g1_mblocks, kb1, 2 * I, I, I, s13,
                         fp8 ? 2 * I / 128 : 0, xs};
      // one launch for both GEMMs when they share a tile list and experts hold
      // few rows (est <= 32): GEMM2 work then fills the tail of GEMM1's.  With
      // more rows per expert GEMM1's items are many and short relative to the
      // whole, and two launches with their own stage layouts run faster.
      const bool fused = NM1 == NM2 && p->est <= 32;
      // fused GEMM2 items take two 128-row weight tiles (256 output rows), so
      // that they stream as many weight bytes per stage as GEMM1 items; FP8
      // GEMM2 items do so as well, halving the per-item epilogue work (scale
      // staging, barriers) per output row
      const int na2 = ((fused || fp8) && H % 256 == 0) ? 2 : 1;
      const bool one_list = NM1 == NM2;  // the scan writes list 2 only when widths differ
      g.p[1] = GemmPhase{one_list ? tiles : tiles2, one_list ? ntiles : ntiles2, na2, 128 * na2,
                         (H + 128 * na2 - 1) / (128 * na2), kb2, H, 128, H, s2,
                         fp8 ? H / 128 : 0, as};
      g.dep = dep;
      // early L2 prefetch of GEMM1 weights, when the previous call on this
      // workspace routed to nearly every local expert (the tile list then has
      // about one tile per expert, in expert order)
      g.spec_experts = EL;
      g.spec_min = EL - EL / 16;
      g.spec_hint = err + 1;
      g.R = static_cast<int>(R);
      g.act = act;
      g.act_scale = as;
      g.I = I;
      g.src = src;
      g.topw = topw;
      g.ybuf = ybuf;
      g.H = H;
      g.err = err;
      g.limit_ns = kWaitLimitNs;
      g.family = want ? family : nullptr;
      g.family_want = want;
      const GemmMaps maps[2] = {m1, m2};
      auto launch = [&](int run1, int run2, int nm, int na) -> bool {
        g.work_counter = dep + p->max_tiles + (run1 ? 0 : 1);  // zeroed by the scan
        g.run1 = run1;
        g.run2 = run2;
        g.fused = run1 && run2;
        g.n_max = nm;
        g.na_max = na;
        g.stages = max_stages(na, nm, kbmax, fp8);
        g.nslots = slots_for(na, nm, fp8);
        g.tmem_cols = tmem_cols_for(g.nslots * na * nm);
        const long long work = static_cast<long long>(p->max_tiles) *
                               ((run1 ? g.p[0].mblocks : 0) + (run2 ? g.p[1].mblocks : 0));
        const int grid = static_cast<int>(work < sms ? work : sms);
        const int smem = g.stages * gemm_stage_bytes(na, nm) + gemm_extra_smem(nm, kbmax, fp8);
        return launch_grouped_gemm(kind, g, maps, grid, smem, st) == cudaSuccess;
      };
      if (fused) {
        if (!launch(1, 1, NM1, 2)) return false;
        if (marks) {
          mark(4);
          mark(5);
        }
      } else {
        if (!launch(1, 0, NM1, 2)) return false;
        if (marks) mark(4);
        if (!launch(0, 1, NM2, na2)) return false;
        if (marks) mark(5);
      }
      return true;
    };
    if (dyn) {
      // both families are enqueued; the launches of the one the scan did not
      // choose leave right after their dependent-launch wait.  The chain
      // still runs about 5 us longer than a plan that fixes the CTA-pair
      // family; leaving before the wait (the next launch then waiting for
      // the gather's CTAs itself), or setting up before it, measured no
      // faster.  Single-CTA first measured faster on uniform routing and the
      // same on concentrated routing.  Events: [4] after the single-CTA
      // launch, [5] after the CTA-pair launches
      if (!run_single(kFamilySingle, false)) return MOE_ERR_CUDA;
      mark(4);
      if (!run_pair(kFamilyPair, false)) return MOE_ERR_CUDA;
      mark(5);
    } else if (pair) {
      if (!run_pair(0, true)) return MOE_ERR_CUDA;
    } else {
      if (!run_single(0, true)) return MOE_ERR_CUDA;
    }
  }

  // a-7: sum of each token's k weighted rows
  const long long cwarps = static_cast<long long>(T) * ((H + 255) / 256);
  const unsigned cblocks = static_cast<unsigned>((cwarps * 32 + 255) / 256);
  if (p->dtype == MOE_DTYPE_F32)
    launch_chained(T <= 512 ? combine_kernel<float, 4> : combine_kernel<float, 1>, dim3(cblocks),
                   dim3(256), 0, st, static_cast<const float*>(ybuf), pos, T, H, k,
                   static_cast<float*>(out));
  else
    launch_chained(T <= 512 ? combine_kernel<__nv_bfloat16, 4> : combine_kernel<__nv_bfloat16, 1>,
                   dim3(cblocks), dim3(256), 0, st, static_cast<const __nv_bfloat16*>(ybuf), pos,
                   T, H, k, static_cast<__nv_bfloat16*>(out));
  mark(6);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

// ====================================================================== C ABI
using namespace moe;

extern "C" {

int moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape for this dtype";
    case MOE_ERR_WORKSPACE: return "workspace smaller than plan->workspace_bytes";
    case MOE_ERR_CUDA: return "CUDA runtime or launch error";
    case MOE_ERR_DEVICE: return "device error word set (bad or duplicate ids, capacity)";
    case MOE_ERR_TIMEOUT: return "a device pipeline wait timed out";
    default: return "unknown error";
  }
}

int moe_plan(int T, int H, int I, int E, int k, int dtype, int scoring, int renorm, int force_est,
             moe_plan_t* plan) {
  return moe_plan_ep(T, H, I, E, k, dtype, scoring, renorm, force_est, 1, 0, plan);
}

int moe_plan_ep(int T, int H, int I, int E, int k, int dtype, int scoring, int renorm,
                int force_est, int ep_size, int ep_rank, moe_plan_t* plan) {
  if (!plan) return MOE_ERR_INVALID_ARG;
  if (ep_size < 1 || ep_rank < 0 || ep_rank >= ep_size || E % ep_size != 0)
    return MOE_ERR_INVALID_ARG;
  if (T < 0 || H <= 0 || I <= 0 || E < 1 || E > kMaxE || k < 1 || k > E || k > kMaxK ||
      force_est < 0)
    return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_DTYPE_F32 && dtype != MOE_DTYPE_BF16 && dtype != MOE_DTYPE_FP8_BLOCK128)
    return MOE_ERR_INVALID_ARG;
  if (scoring != MOE_SCORING_SOFTMAX && scoring != MOE_SCORING_SIGMOID) return MOE_ERR_INVALID_ARG;
  const int kstep = dtype == MOE_DTYPE_F32 ? 32 : dtype == MOE_DTYPE_BF16 ? 64 : 128;
  if (H % kstep != 0 || I % kstep != 0) return MOE_ERR_UNSUPPORTED;
  const long long R = static_cast<long long>(T) * k;
  if (R > (1ll << 30) || static_cast<long long>(T) * H > (1ll << 40)) return MOE_ERR_INVALID_ARG;

  moe_plan_t p;
  std::memset(&p, 0, sizeof(p));
  p.abi_version = MOE_ABI_VERSION;
  p.T = T;
  p.H = H;
  p.I = I;
  p.E = E;
  p.k = k;
  p.dtype = dtype;
  p.scoring = scoring;
  p.renorm = renorm ? 1 : 0;
  p.force_est = force_est;
  p.route_tpc = T > 2048 ? 32 : 8;
  p.n_chunks = (T + p.route_tpc - 1) / p.route_tpc;
  p.ep_size = ep_size;
  p.ep_rank = ep_rank;
  p.n_group = 1;
  p.topk_group = 1;
  p.e_local = E / ep_size;
  const int EL = p.e_local;
  p.g1_mblocks = (I + 127) / 128;
  p.g2_mblocks = (H + 127) / 128;

  // 1) worst-case capacity, from (T, k, E, H, I, dtype) alone: the tile list
  //    is bounded with the smallest token tile (16), whatever est says
  const long long max_tiles = (R + 15) / 16 + (EL < R ? EL : R) + 1;
  p.max_tiles = static_cast<int32_t>(max_tiles);
  const int ex = dtype == MOE_DTYPE_F32 ? 4 : dtype == MOE_DTYPE_BF16 ? 2 : 1;
  uint64_t off = 0;
  auto take = [&](uint64_t bytes) {
    const uint64_t o = off;
    off += (bytes + 255) & ~static_cast<uint64_t>(255);
    return o;
  };
  p.off_err = take(16);
  p.off_ids = take(R * 4);
  p.off_w = take(R * 4);
  p.off_chunk_counts = take(static_cast<uint64_t>(p.n_chunks) * EL * 4);
  p.off_lrank = take(R * 4);
  p.off_counts = take(static_cast<uint64_t>(EL) * 4);
  p.off_offsets = take(static_cast<uint64_t>(EL + 1) * 4);
  p.off_chunk_base = take(static_cast<uint64_t>(p.n_chunks) * EL * 4);
  p.off_src = take(R * 4);
  p.off_pos = take(R * 4);
  p.off_tiles = take(static_cast<uint64_t>(max_tiles) * 16);
  p.off_ntiles = take(16);
  p.off_tiles2 = take(static_cast<uint64_t>(max_tiles) * 16);
  p.off_ntiles2 = take(16);
  p.off_dep = take(static_cast<uint64_t>(max_tiles + 2) * 4);
  p.off_xq = take(static_cast<uint64_t>(R) * H * ex);
  p.off_xs = take(dtype == MOE_DTYPE_FP8_BLOCK128 ? static_cast<uint64_t>(R) * (H / 128) * 4 : 0);
  p.off_act = take(static_cast<uint64_t>(R) * I * ex);
  p.off_as = take(dtype == MOE_DTYPE_FP8_BLOCK128 ? static_cast<uint64_t>(R) * (I / 128) * 4 : 0);
  p.off_y = take(static_cast<uint64_t>(R) * H * (dtype == MOE_DTYPE_F32 ? 4 : 2));
  p.workspace_bytes = off;

  // 2) then the estimate (H20 article, para. 3) and the tile it selects;
  //    the denominator is all physical experts, across expert-parallel ranks
  const long long est = force_est > 0 ? force_est : (R + E - 1) / E;
  p.est = static_cast<int32_t>(est < 1 ? 1 : est);
  p.tile_n = p.est <= 16 ? 16 : p.est <= 32 ? 32 : p.est <= 64 ? 64 : 128;
  // FP8: the scale-folding epilogue keeps gate and up sums of each token
  // column in registers, which caps its tiles at 64 tokens
  if (dtype == MOE_DTYPE_FP8_BLOCK128 && p.tile_n > 64) p.tile_n = 64;
  // experts with more than 32 rows on average: BF16/F32 GEMMs on CTA pairs
  p.gemm_pair = (dtype != MOE_DTYPE_FP8_BLOCK128 && p.est > 32) ? 1 : 0;
  // FP8 with 32 or more rows per expert on average: token-major GEMMs
  p.gemm_tm = (dtype == MOE_DTYPE_FP8_BLOCK128 && p.est >= kTmMinEst) ? 1 : 0;
  // one-CTA-per-tile BF16/F32 plans whose batch can hold a whole 256-row
  // CTA-pair tile for one expert: the device picks the family per call
  p.gemm_dyn = (dtype != MOE_DTYPE_FP8_BLOCK128 && !p.gemm_pair && T >= kHotRows) ? 1 : 0;
  *plan = p;
  return MOE_OK;
}

int moe_plan_describe(const moe_plan_t* p, char* buf, size_t n) {
  if (!plan_ok(p)) return MOE_ERR_INVALID_ARG;
  static const char* dn[] = {"f32", "bf16", "fp8_block128"};
  int len = std::snprintf(
      buf, buf ? n : 0,
      "moe_plan T=%d H=%d I=%d E=%d (ep %d/%d, %d local) k=%d dtype=%s scoring=%s renorm=%d "
      "est=%d%s tile_n=%d gemm=%s route_tpc=%d chunks=%d max_tiles=%d g1_blocks=%d "
      "g2_blocks=%d workspace=%llu B",
      p->T, p->H, p->I, p->E, p->ep_rank, p->ep_size, p->e_local, p->k, dn[p->dtype],
      p->scoring ? "sigmoid" : "softmax", p->renorm,
      p->est, p->force_est ? " (forced)" : "", p->tile_n,
      (p->dtype == MOE_DTYPE_FP8_BLOCK128 && p->gemm_tm) ? "token-major"
      : (p->dtype != MOE_DTYPE_FP8_BLOCK128 && p->gemm_pair) ? "cta-pair"
      : (p->dtype != MOE_DTYPE_FP8_BLOCK128 && p->gemm_dyn) ? "swap-ab|cta-pair (per call)"
                                                            : "swap-ab",
      p->route_tpc, p->n_chunks, p->max_tiles, p->g1_mblocks, p->g2_mblocks,
      static_cast<unsigned long long>(p->workspace_bytes));
  return len;
}

int moe_forward(const moe_plan_t* plan, const void* x, const void* logits, const void* w13,
                const float* s13, const void* w2, const float* s2, void* out, void* ws,
                size_t ws_bytes, void* stream) {
  return forward_impl(plan, x, logits, nullptr, nullptr, w13, s13, w2, s2, out, ws, ws_bytes,
                      stream);
}

int moe_forward_timed(const moe_plan_t* plan, const void* x, const void* logits, const void* w13,
                      const float* s13, const void* w2, const float* s2, void* out, void* ws,
                      size_t ws_bytes, void* stream, void* const* events, int n_events) {
  if (!events || n_events != 7) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 7; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  return forward_impl(plan, x, logits, nullptr, nullptr, w13, s13, w2, s2, out, ws, ws_bytes,
                      stream, events);
}

int moe_forward_with_ids(const moe_plan_t* plan, const void* x, const int32_t* ids,
                         const float* topk_w, const void* w13, const float* s13, const void* w2,
                         const float* s2, void* out, void* ws, size_t ws_bytes, void* stream) {
  return forward_impl(plan, x, nullptr, ids, topk_w, w13, s13, w2, s2, out, ws, ws_bytes, stream,
                      nullptr, true);
}

static bool groups_ok(int E, int k, int n_group, int topk_group) {
  return n_group >= 1 && n_group <= 32 && E % n_group == 0 && topk_group >= 1 &&
         topk_group <= n_group && k <= topk_group * (E / n_group);
}

int moe_plan_set_groups(moe_plan_t* plan, int n_group, int topk_group) {
  if (!plan_ok(plan) || !groups_ok(plan->E, plan->k, n_group, topk_group))
    return MOE_ERR_INVALID_ARG;
  plan->n_group = n_group;
  plan->topk_group = topk_group;
  return MOE_OK;
}

int moe_route_topk(const void* logits, int logits_dtype, int T, int E, int k, int scoring,
                   int renorm, int32_t* ids, float* w, void* stream) {
  return moe_route_grouped_topk(logits, logits_dtype, T, E, k, 1, 1, scoring, renorm, ids, w,
                                stream);
}

int moe_route_grouped_topk(const void* logits, int logits_dtype, int T, int E, int k,
                           int n_group, int topk_group, int scoring, int renorm, int32_t* ids,
                           float* w, void* stream) {
  if (T < 0 || E < 1 || E > kMaxE || k < 1 || k > E || k > kMaxK) return MOE_ERR_INVALID_ARG;
  if (!groups_ok(E, k, n_group, topk_group)) return MOE_ERR_INVALID_ARG;
  if (logits_dtype != MOE_LOGITS_F32 && logits_dtype != MOE_LOGITS_BF16) return MOE_ERR_INVALID_ARG;
  if (scoring != MOE_SCORING_SOFTMAX && scoring != MOE_SCORING_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;  // empty batch: null pointers allowed
  if (!logits || !ids || !w) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int tpc = 8;
  dim3 grid((T + tpc - 1) / tpc);
  if (logits_dtype == MOE_LOGITS_F32)
    launch_route_t<float>(vpt_for(E), grid, 0, st, static_cast<const float*>(logits), T, E, k,
                          scoring, renorm ? 1 : 0, tpc, 0, nullptr, nullptr, ids, w, nullptr,
                          nullptr, nullptr, 0, E, n_group, topk_group);
  else
    launch_route_t<__nv_bfloat16>(vpt_for(E), grid, 0, st,
                                  static_cast<const __nv_bfloat16*>(logits), T, E, k, scoring,
                                  renorm ? 1 : 0, tpc, 0, nullptr, nullptr, ids, w, nullptr,
                                  nullptr, nullptr, 0, E, n_group, topk_group);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_check(const moe_plan_t* plan, void* ws, uint32_t* bits, void* stream) {
  if (!plan_ok(plan) || !ws) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned word = 0;
  unsigned* err = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(ws) + plan->off_err);
  if (cudaMemcpyAsync(&word, err, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (word && cudaMemsetAsync(err, 0, sizeof(unsigned), st) != cudaSuccess) return MOE_ERR_CUDA;
  if (bits) *bits = word;
  if (word & MOE_DEVERR_TIMEOUT) return MOE_ERR_TIMEOUT;
  return word ? MOE_ERR_DEVICE : MOE_OK;
}

// ------------------------------------------------------------------ no-alloc entry
// Some callers cannot call cudaMalloc at all: code that runs inside a
// framework's allocator hook or a custom memory pool, plug-ins whose host
// forbids device allocation after start-up, and call sites that must stay
// free of allocation so they can be replayed in a fixed memory budget.
// moe_forward_noalloc serves them with a workspace that lives in this
// library's own device image: a file-scope array, reserved when the module
// is loaded on a device and held until the process exits.  Its size is the
// hard limit of this entry point.
static constexpr size_t kNoAllocWorkspaceBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoAllocWorkspaceBytes];

// The calling thread's current CUDA context (driver API, looked up through
// the runtime's entry-point query), or null.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
static CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of g_noalloc_workspace, looked up with that device current
// the first time a device (and context) calls.  In host code the array's
// name is only a host-side stand-in, never a device address, so it must not
// be passed to a kernel.  The address is remembered together with the
// context it was looked up in: after cudaDeviceReset, or when the primary
// context is torn down and created again, the module is loaded anew and the
// address is looked up again on the next call.
static void* noalloc_workspace_ptr() {
  constexpr int kMaxDevices = 64;
  static void* ptrs[kMaxDevices] = {};
  static CUcontext ctxs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev] || !ctx || ctxs[dev] != ctx) {
    // no context bound to this thread yet, a new device, or a new context:
    // the runtime query binds the device's context and loads the module
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || !p) return nullptr;
    ptrs[dev] = p;
    ctxs[dev] = current_context();
  }
  return ptrs[dev];
}

int moe_forward_noalloc(const moe_plan_t* plan, const void* x, const void* logits,
                        const void* w13, const float* s13, const void* w2, const float* s2,
                        void* out, void* stream) {
  if (!plan_ok(plan)) return MOE_ERR_INVALID_ARG;
  if (plan->workspace_bytes > kNoAllocWorkspaceBytes) return MOE_ERR_WORKSPACE;
  void* ws = noalloc_workspace_ptr();
  if (!ws) return MOE_ERR_CUDA;
  // the error word is the only region that must start from zero; the
  // forward clears it on the stream before its first kernel
  return forward_impl(plan, x, logits, nullptr, nullptr, w13, s13, w2, s2, out, ws,
                      kNoAllocWorkspaceBytes, stream);
}

int moe_check_noalloc(const moe_plan_t* plan, uint32_t* bits, void* stream) {
  if (!plan_ok(plan)) return MOE_ERR_INVALID_ARG;
  if (plan->workspace_bytes > kNoAllocWorkspaceBytes) return MOE_ERR_WORKSPACE;
  void* ws = noalloc_workspace_ptr();
  if (!ws) return MOE_ERR_CUDA;
  return moe_check(plan, ws, bits, stream);
}

}  // extern "C"
