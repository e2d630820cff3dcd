// grouped_gemm_tm.cu -- token-major grouped GEMMs for block-scaled FP8 e4m3
// (steps a-4 .. a-7 of the fused MoE layer), tcgen05/TMEM fed by TMA.
//
// Orientation: the MMA's M side is a tile of up to 128 permuted token rows of
// one expert, its N side 256 weight rows of that expert:
//   GEMM1 item: 128 gate rows and the matching 128 up rows of one 128-feature
//               block (two TMA boxes stacked into one 256-row operand), so a
//               single M=128, N=256 MMA per 32-byte K step covers both;
//   GEMM2 item: 256 output rows (two 128-row blocks of w2).
// An N=256 MMA runs at the tensor pipe's full rate; narrower ones do not.
//
// FP8 [128,128] block scales (Lab notes #6, "Method": fp8_w8a8, block
// [128,128]) with per-token 128-column activation groups: each 128-deep K
// block is accumulated into its own TMEM slot (two slots of 256 columns,
// double-buffered), and the epilogue folds it into fp32 registers.  With
// tokens on the M side every epilogue thread owns one token row, so the
// block's scale is a scalar per thread and weight block:
//   acc[n] += P_kb[row, n] * s_x[row, kb] * s_w[block(n), kb],
// which honours arbitrary fp32 scales exactly (the hardware block-scaled MMA
// takes only power-of-two scales per 32 elements).
//
//   warp 0       TMA producer: two 128-row weight boxes + one token box per
//                128-byte K block (the token box is only as high as the
//                tile's rows need; rows past it are never stored)
//   warp 1       TMEM allocation and the single-thread MMA issuer
//   warps 2, 3   idle (they complete warp group 0's register hand-back)
//   warps 4..19  epilogue: four warps per TMEM lane quadrant, each holding
//                32 columns of both 128-column halves of its rows
//                GEMM1: act = SiLU(gate) * up, then e4m3 per token and
//                       128-feature group (the group's amax meets across the
//                       four warps of a quadrant in shared memory), staged
//                       swizzled and written with TMA tensor stores
//                GEMM2: ybuf[row] = w[t,j] * y (the combine's weighting),
//                       each warp's rows turned around in its own shared
//                       memory and written 8 rows x 64 bytes per store
//
// Every wait is bounded; a timeout sets MOE_DEVERR_TIMEOUT, raises a CTA
// abort flag, drains in-flight copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <mutex>

#include "gemm_common.cuh"
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

// Warp group 0 (warps 0..3): TMA producer, MMA issuer and two idle warps;
// warp groups 1..4: the 16 epilogue warps.  Launched at 96 registers per
// thread (640 threads: 61,440), warp group 0 gives registers back down to 64
// and the epilogue takes them up to 104: 128 x 64 + 512 x 104 = 61,440, and
// every SM sub-partition holds one warp of group 0 and four epilogue warps,
// so the split balances there too (the epilogue's two 16-column TMEM loads
// and 64 accumulators fit in 104 without spilling).
constexpr int kTmRegsLaunch = 96;
constexpr int kTmRegsGroup0 = 64;
constexpr int kTmRegsEpilogue = 104;
constexpr int kTmEpiWarps = 16;
constexpr int kTmEpiWarp0 = 4;  // first epilogue warp
constexpr int kTmThreads = 32 * (kTmEpiWarp0 + kTmEpiWarps);
constexpr int kTmCols = 32;  // columns per epilogue thread in each 128-column half
static_assert(128 * kTmRegsGroup0 + 32 * kTmEpiWarps * kTmRegsEpilogue ==
                  kTmThreads * kTmRegsLaunch,
              "the register split must hand out exactly the launch's registers");

// the smallest token box (16, 32, 64 or 128 rows) that holds `rows`
__device__ __forceinline__ int tm_box_rows(int rows) {
  return rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : 128;
}

// SiLU(z) = z * sigmoid(z) with sigmoid(z) = (1 + tanh(z/2)) / 2: one
// hardware tanh approximation (relative error about 2^-11, far below the
// e4m3 step the result is quantised to) instead of an exponential and a
// reciprocal; large negative z give 0, large positive z give z
__device__ __forceinline__ float silu_tanh(float z) {
  const float h = 0.5f * z;
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
  return fmaf(h, t, h);
}

// Shared-memory byte offset of 16-byte chunk `c` of row `r` in a tile of
// 128-byte rows laid out with the 128-byte swizzle (the layout a TMA tensor
// map with CU_TENSOR_MAP_SWIZZLE_128B reads): the chunk index is XORed with
// the row's position in its 8-row (1024-byte) group.  Tiles start on
// 1024-byte boundaries.
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
  return static_cast<uint32_t>(r) * 128u + static_cast<uint32_t>((c ^ (r & 7)) << 4);
}

// TMA stores of rows [0, n16) of a staged tile (n16 a multiple of 16, at most
// 128) to rows row0.. of the tensor, column x: one box per set bit of n16
// (128 / 64 / 32 / 16 rows), so that no row past the tile's own is written.
__device__ __forceinline__ void store_rows16(const GemmMaps& out, uint32_t stg, int n16, int x,
                                             int row0) {
  int r0 = 0;
#pragma unroll
  for (int h = 128; h >= 16; h >>= 1) {
    if (n16 & h) {
      tma_store_2d(&out.b[tok_map_index(h)], stg + static_cast<uint32_t>(r0) * 128u, x, row0 + r0);
      r0 += h;
    }
  }
}

// eight values -> eight e4m3 codes (clamped to +-448 first), little-endian
__device__ __forceinline__ uint2 pack_e4m3x8(const float* v, float inv_scale) {
  uint2 out = make_uint2(0u, 0u);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float q = fmaxf(fminf(v[i] * inv_scale, 448.0f), -448.0f);
    const uint32_t code = __nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3);
    if (i < 4)
      out.x |= code << (8 * i);
    else
      out.y |= code << (8 * (i - 4));
  }
  return out;
}

template <int MODE>
__global__ void __launch_bounds__(kTmThreads, 1)
    moe_gemm_tm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ GemmMaps omaps,
                       const GemmArgs args) {
  constexpr int G = MODE - 1;  // which GEMM
  extern __shared__ uint8_t smem_raw[];

  const GemmPhase& P = args.p[G];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = args.stages;
  const uint64_t limit = args.limit_ns;
  const int kbs = P.kblocks;

  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // output staging: GEMM1 one 128-row x 128-byte act block (128-byte
  // swizzled, for the TMA stores), GEMM2 2 KB per epilogue warp
  uint8_t* stg = stages + static_cast<size_t>(S) * kTmStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(stg + tm_out_bytes(MODE));
  uint64_t* empty = full + S;
  uint64_t* accf = empty + S;  // [2] K-block slot written by the MMAs
  uint64_t* acce = accf + 2;   // [2] K-block slot folded by the epilogue
  uint64_t* done = acce + 2;   // all MMAs of this CTA complete
  uint64_t* epib = done + 1;   // epilogue-internal barrier
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epib + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // GEMM1: [2 items][4 parts][128 rows] partial amax per token row
  float* red = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 512);

  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&accf[b]), 1);
      mbar_init(smem_u32(&acce[b]), kTmEpiWarps);
    }
    mbar_init(smem_u32(done), 1);
    mbar_init(smem_u32(epib), kTmEpiWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.a);
    for (int j = 0; j < kTokMaps; ++j) {
      prefetch_tmap(&maps.b[j]);
      prefetch_tmap(&omaps.b[j]);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the tile list and token rows are the predecessor kernels' output

  const int nwork = (*P.ntiles) * P.mblocks;
  int never = 0;
  bool ok = true;

  if (warp < kTmEpiWarp0) {
    // warp group 0 hands registers back before its roles start
    setmaxnreg_dec<kTmRegsGroup0>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();  // weights: streamed
      const uint64_t pol_x = policy_evict_last();   // token rows: reused per block
      uint32_t it = 0;
      int4 next = static_cast<int>(blockIdx.x) < nwork ? P.tiles[blockIdx.x / P.mblocks]
                                                         : int4{0, 0, 0, 0};
      for (int w = blockIdx.x; w < nwork && ok; w += gridDim.x) {
        const int4 tile = next;
        if (w + static_cast<int>(gridDim.x) < nwork) next = P.tiles[(w + gridDim.x) / P.mblocks];
        const int mb = w % P.mblocks;
        const int box = tm_box_rows(tile.z);
        const CUtensorMap* tmx = &maps.b[tok_map_index(box)];
        const int b_row = tile.x * P.a_rows_per_e + mb * P.row_step;
        const uint32_t tx = 2u * 16384u + static_cast<uint32_t>(box) * 128u;
        for (int kb = 0; kb < kbs; ++kb, ++it) {
          const int s = static_cast<int>(it % S);
          if (!mbar_wait(smem_u32(&empty[s]), ((it / S) & 1u) ^ 1u, limit, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* st = stages + static_cast<size_t>(s) * kTmStageBytes;
          const uint32_t fb = smem_u32(&full[s]);
          mbar_arrive_expect_tx(fb, tx);
          const int kx = kb * 128;
          // the item's 256 weight rows in one copy: GEMM1's gate block and up
          // block as the two planes of a 3-D box, GEMM2's two output blocks
          // as one 256-row box
          if constexpr (G == 0)
            tma_load_3d(smem_u32(st), &maps.a, fb, kx, mb * 128, 2 * tile.x, pol_w);
          else
            tma_load_2d(smem_u32(st), &maps.a, fb, kx, b_row, pol_w);
          tma_load_2d(smem_u32(st + 32768), tmx, fb, kx, tile.y, pol_x);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(args.err, kDevErrTimeout);
      }
      // never leave with copies in flight: wait for the last S stages issued
      for (uint32_t j = (it > static_cast<uint32_t>(S) ? it - S : 0u); j < it; ++j)
        mbar_wait(smem_u32(&full[j % S]), (j / S) & 1u, limit, &never);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // M = 128 token rows, N = 256 weight rows, e4m3 x e4m3 -> f32
      const uint32_t idesc = idesc_make(KindTraits<KIND_E4M3>::fmt, 128, 256);
      uint32_t it = 0, kc = 0;
      for (int w = blockIdx.x; w < nwork && ok; w += gridDim.x) {
        for (int kb = 0; kb < kbs; ++kb, ++it, ++kc) {
          const uint32_t slot = kc & 1u;
          if (!mbar_wait(smem_u32(&acce[slot]), ((kc >> 1) & 1u) ^ 1u, limit, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int s = static_cast<int>(it % S);
          if (!mbar_wait(smem_u32(&full[s]), (it / S) & 1u, limit, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(stages + static_cast<size_t>(s) * kTmStageBytes);
          const uint64_t bd0 = sdesc_sw128(sa);          // 256 weight rows
          const uint64_t ad0 = sdesc_sw128(sa + 32768);  // 128 token rows
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_issue<KIND_E4M3>(tmem_base + slot * 256u, ad0 + 2u * ks, bd0 + 2u * ks, idesc,
                                 ks != 0);
          mma_commit(smem_u32(&empty[s]));    // frees the stage once read
          mma_commit(smem_u32(&accf[slot]));  // the K block's partial is in TMEM
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(args.err, kDevErrTimeout);
      }
      // never free TMEM under a running MMA
      mma_commit(smem_u32(done));
      mbar_wait(smem_u32(done), 0, limit, &never);
    }
    __syncwarp();
  }
  } else {
    // ------------------------------------------------------------ epilogue
    setmaxnreg_inc<kTmRegsEpilogue>();
    const int ew = warp - kTmEpiWarp0;
    const int q = warp & 3;    // TMEM lane quadrant this warp may read
    const int part = ew >> 2;  // which 32 columns of each 128-column half
    const int r = q * 32 + lane;  // this thread's token row within the tile
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t kc = 0, eb = 0, ib = 0;

    auto warp_arrive = [&](uint64_t* bar) {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(bar));
    };
    auto ep_barrier = [&]() -> bool {
      warp_arrive(epib);
      const bool got = mbar_wait(smem_u32(epib), eb & 1u, limit, abort_flag);
      ++eb;
      return __all_sync(0xffffffffu, got);
    };

    // Scale pointers of work item (tile, mb) for this thread's row:
    // activation scales of the row, one per K block, and weight scales of
    // the item's two 128-row blocks (GEMM1: the gate and the up block of the
    // feature block; GEMM2: two consecutive output blocks).  GEMM2's second
    // block lies past the expert's rows when H is not a multiple of 256 (its
    // outputs are not stored): the first block's scales stand in for it
    // rather than another expert's or those past the array.
    auto scale_ptrs = [&](const int4& tl, int mbi, const float*& sxp, const float*& sw0p,
                          const float*& sw1p) {
      const int gr = tl.y + (r < tl.z ? r : 0);  // a valid row for the loads
      sxp = P.b_scale + static_cast<size_t>(gr) * kbs;
      sw0p = P.w_scale + (static_cast<size_t>(tl.x) * P.w_scale_rows_per_e +
                          static_cast<size_t>(mbi) * (P.row_step / 128)) * kbs;
      const bool blk1 = G == 0 || mbi * P.row_step + 128 < P.m_valid;
      sw1p = blk1 ? sw0p + static_cast<size_t>(P.a_up_off / 128) * kbs : sw0p;
    };
    // the first item's tile and first K block's scales; later items' are
    // loaded one item ahead (the tile) and during the previous item's last
    // K block (the scales), off the path from one item to the next
    int4 tile = static_cast<int>(blockIdx.x) < nwork ? P.tiles[blockIdx.x / P.mblocks]
                                                     : int4{0, 0, 0, 0};
    float sx_n = 0.0f, sw0_n = 0.0f, sw1_n = 0.0f;
    if (static_cast<int>(blockIdx.x) < nwork) {
      const float *a, *b, *c;
      scale_ptrs(tile, blockIdx.x % P.mblocks, a, b, c);
      sx_n = __ldg(a);
      sw0_n = __ldg(b);
      sw1_n = __ldg(c);
    }

    for (int w = blockIdx.x; w < nwork && ok; w += gridDim.x, ++ib) {
      const int wn = w + static_cast<int>(gridDim.x);
      const int4 tile_next = wn < nwork ? P.tiles[wn / P.mblocks] : tile;
      const int mb = w % P.mblocks;
      const int row0 = tile.y, nrows = tile.z;
      const bool live = r < nrows;
      const int grow = row0 + (live ? r : 0);
      const float *sxp, *sw0p, *sw1p;
      scale_ptrs(tile, mb, sxp, sw0p, sw1p);
      tile = tile_next;
      float wt = 0.0f;  // GEMM2: the routing weight of this row's pick
      if (G == 1 && live) wt = __ldg(args.topw + __ldg(args.src + grow));

      // accumulators as pairs of columns: the fold is one packed two-lane
      // FMA (each lane rounded exactly like fmaf) per pair of columns
      float2 acc0[kTmCols / 2], acc1[kTmCols / 2];
#pragma unroll
      for (int c = 0; c < kTmCols / 2; ++c) {
        acc0[c] = make_float2(0.0f, 0.0f);
        acc1[c] = make_float2(0.0f, 0.0f);
      }
      for (int kb = 0; kb < kbs; ++kb, ++kc) {
        const float c0 = sx_n * sw0_n, c1 = sx_n * sw1_n;
        const float2 c02 = make_float2(c0, c0), c12 = make_float2(c1, c1);
        if (kb + 1 < kbs) {  // the next block's scales load under this block's fold
          sx_n = __ldg(sxp + kb + 1);
          sw0_n = __ldg(sw0p + kb + 1);
          sw1_n = __ldg(sw1p + kb + 1);
        } else if (wn < nwork) {  // and after the last block, the next item's first
          const float *a, *b, *c;
          scale_ptrs(tile_next, wn % P.mblocks, a, b, c);
          sx_n = __ldg(a);
          sw0_n = __ldg(b);
          sw1_n = __ldg(c);
        }
        const uint32_t slot = kc & 1u;
        const bool got = mbar_wait(smem_u32(&accf[slot]), (kc >> 1) & 1u, limit, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = lane_addr + slot * 256u + static_cast<uint32_t>(part * kTmCols);
        const uint32_t a1 = a0 + 128u;
        // rounds of FC columns of both halves, one TMEM round trip each (GEMM2
        // keeps more state live across the loop and takes narrower rounds)
        constexpr int FC = G == 0 ? 16 : 8;
#pragma unroll
        for (int c = 0; c < kTmCols; c += FC) {
          float p0[FC], p1[FC];
          tmem_ld<FC>(a0 + c, p0);
          tmem_ld<FC>(a1 + c, p1);
          tmem_wait_ld(p0, p1);
#pragma unroll
          for (int i = 0; i < FC / 2; ++i) {
            acc0[c / 2 + i] =
                __ffma2_rn(make_float2(p0[2 * i], p0[2 * i + 1]), c02, acc0[c / 2 + i]);
            acc1[c / 2 + i] =
                __ffma2_rn(make_float2(p1[2 * i], p1[2 * i + 1]), c12, acc1[c / 2 + i]);
          }
        }
        tc_fence_before();
        warp_arrive(&acce[slot]);
      }
      if (!ok) break;

      const bool elected = ew == 0 && lane == 0;  // issues the TMA stores
      const int n16 = nrows & ~15;  // rows stored by TMA; the rest by their threads
      if constexpr (G == 0) {
        // act = SiLU(gate) * up for this row's 32 features of the block,
        // then e4m3 over the block's 128 features with one scale per row
        float act[kTmCols];
        float m = 0.0f;
#pragma unroll
        for (int c = 0; c < kTmCols / 2; ++c) {
          act[2 * c] = silu_tanh(acc0[c].x) * acc1[c].x;
          act[2 * c + 1] = silu_tanh(acc0[c].y) * acc1[c].y;
          m = fmaxf(m, fmaxf(fabsf(act[2 * c]), fabsf(act[2 * c + 1])));
        }
        float* rb = red + (ib & 1u) * 512;
        rb[part * 128 + r] = m;
        if (elected) bulk_wait_read<0>();  // the previous item's store has read the staging
        if (!ep_barrier()) {
          ok = false;
          break;
        }
        const float amax = fmaxf(fmaxf(rb[r], rb[128 + r]), fmaxf(rb[256 + r], rb[384 + r]));
        const float scale = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
        // v / scale as v * (1 / scale): at most one fp32 ulp apart, far
        // below the e4m3 step
        const float inv = __frcp_rn(scale);
        uint4 v[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint2 lo = pack_e4m3x8(act + 16 * h, inv);
          const uint2 hi = pack_e4m3x8(act + 16 * h + 8, inv);
          v[h] = make_uint4(lo.x, lo.y, hi.x, hi.y);
          *reinterpret_cast<uint4*>(stg + sw128_offset(r, 2 * part + h)) = v[h];
        }
        if (live) {
          if (part == 0)
            args.act_scale[static_cast<size_t>(grow) * (args.I / 128) + mb] = scale;
          if (r >= n16) {  // the tile's last rows past a multiple of 16
            uint8_t* dst = static_cast<uint8_t*>(args.act) + static_cast<size_t>(grow) * args.I +
                           mb * 128 + part * kTmCols;
            reinterpret_cast<uint4*>(dst)[0] = v[0];
            reinterpret_cast<uint4*>(dst)[1] = v[1];
          }
        }
        fence_proxy_async_shared();
        if (!ep_barrier()) {
          ok = false;
          break;
        }
        if (elected && n16 > 0) {
          store_rows16(omaps, smem_u32(stg), n16, mb * 128, row0);
          bulk_commit();
        }
      } else {
        // weighted rows of the two output blocks, bf16.  Each warp turns its
        // 32 rows x 32 columns of a half around in its own 2 KB of shared
        // memory, so that every store instruction writes 8 rows x 64
        // contiguous bytes instead of 32 rows x 16 bytes; only __syncwarp
        // orders it.  16-byte chunk c of row l sits at chunk position
        // c ^ ((l >> 1) & 3): both the row-wise writes and the column-wise
        // reads then touch each bank group once per 8 lanes.
        uint8_t* wsl = stg + ew * 2048;  // this warp's slice
        auto store_half = [&](const float2(&a)[kTmCols / 2], int half) -> bool {
          const int h0 = mb * 256 + half * 128 + part * kTmCols;  // this warp's first column
          if (mb * 256 + half * 128 >= args.H) return true;      // uniform: the block past H
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 v;
            v.x = pack_bf16x2(wt * a[4 * i].x, wt * a[4 * i].y);
            v.y = pack_bf16x2(wt * a[4 * i + 1].x, wt * a[4 * i + 1].y);
            v.z = pack_bf16x2(wt * a[4 * i + 2].x, wt * a[4 * i + 2].y);
            v.w = pack_bf16x2(wt * a[4 * i + 3].x, wt * a[4 * i + 3].y);
            *reinterpret_cast<uint4*>(wsl + lane * 64 + ((i ^ ((lane >> 1) & 3)) << 4)) = v;
          }
          __syncwarp();
          const int c = lane & 3;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int rr = i * 8 + (lane >> 2);  // row within the warp's 32
            const uint4 v =
                *reinterpret_cast<const uint4*>(wsl + rr * 64 + ((c ^ ((rr >> 1) & 3)) << 4));
            const int rt = q * 32 + rr;  // row within the tile
            if (rt < nrows)
              *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.ybuf) +
                                        static_cast<size_t>(row0 + rt) * args.H + h0 + c * 8) = v;
          }
          __syncwarp();
          return true;
        };
        if (!store_half(acc0, 0) || !store_half(acc1, 1)) {
          ok = false;
          break;
        }
      }
    }
    // every store has landed before the CTA leaves
    if (ew == 0 && lane == 0) bulk_wait<0>();
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) atomicOr(args.err, kDevErrTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

template <int MODE>
static cudaError_t launch_tm_mode(const GemmArgs& args, const GemmMaps& maps,
                                  const GemmMaps& omaps, int grid, int smem, cudaStream_t stream) {
  auto kern = moe_gemm_tm_kernel<MODE>;
  // max dynamic smem is a per-function attribute, raised once per size (and
  // again after a switch of device); host threads may launch concurrently
  static std::mutex mu;
  static int configured = 0, conf_dev = -1;
  static bool regs_checked = false;
  {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (!regs_checked) {
      // the register split hands out exactly the registers of a launch at
      // kTmRegsLaunch per thread; with fewer, the epilogue's increase could
      // never be granted, so such a build is refused rather than launched
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != kTmRegsLaunch) return cudaErrorInvalidConfiguration;
      regs_checked = true;
    }
    if (dev != conf_dev || configured < smem) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      configured = dev != conf_dev ? smem : (configured > smem ? configured : smem);
      conf_dev = dev;
    }
  }
  return launch_chained(kern, dim3(grid), dim3(kTmThreads), static_cast<size_t>(smem), stream,
                        maps, omaps, args);
}

cudaError_t launch_grouped_gemm_tm(int mode, const GemmArgs& args, const GemmMaps& maps,
                                   const GemmMaps& omaps, int grid, int smem,
                                   cudaStream_t stream) {
  if (args.stages < 1 || grid < 1 || smem < tm_smem_bytes(mode, args.stages))
    return cudaErrorInvalidValue;
  return mode == 1 ? launch_tm_mode<1>(args, maps, omaps, grid, smem, stream)
                   : launch_tm_mode<2>(args, maps, omaps, grid, smem, stream);
}

}  // namespace moe
