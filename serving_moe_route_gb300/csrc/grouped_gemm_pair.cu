// grouped_gemm_pair.cu -- the grouped GEMMs of the fused MoE layer (steps
// a-4 .. a-7) on CTA pairs, for BF16/TF32 batches whose experts hold many
// rows (prefill-sized plans).
//
// A cluster of two CTAs runs one tcgen05.mma with cta_group::2 per K step:
// M = 256 weight rows (128 in each CTA's shared memory), N = up to 256 token
// rows of one expert (N/2 in each CTA).  Each SM thus streams half of the
// token tile and its own 128 weight rows, and the tensor cores of both SMs
// work on every byte either CTA loaded -- half the shared-memory operand
// traffic per multiply-add of a single-CTA 128 x N tile, which is what keeps
// the tensor pipe fed when every expert has hundreds of rows (H20 article,
// para. 3: the large-estimate tile; here still swap-AB, so the token side
// follows each expert's row count in steps of 16).
//
//   GEMM1 item: 256 features (gate rows and up rows, 128 of each per CTA)
//               x one token tile; two pair MMAs per K step (gate, up) into
//               the two halves of one TMEM slot (2 x N columns).
//   GEMM2 item: 256 output rows (128 per CTA) x one token tile; one pair MMA
//               per K step, two TMEM slots so the epilogue overlaps.
//
//   warp 0      TMA producer of this CTA's half of every stage; the copies
//               of both CTAs complete on the even CTA's `full` barrier
//   warp 1      TMEM allocation (both CTAs); MMA issue (even CTA only):
//               GEMM1's gate MMAs and all of GEMM2's
//   warp 18     GEMM1's up MMAs (even CTA only; a second issuer, since one
//               thread's issue cost exceeds a pair MMA's tensor time below
//               N = 256)
//   warps 2..17 epilogue of this CTA's 128 rows (four warps per TMEM lane
//               quadrant, each a quarter of the token columns); the
//               drained-slot signal goes to the even CTA's `acce` barrier
//
// Both CTAs walk the same item sequence (items c, c + clusters, ...).  Every
// wait is bounded; a CTA that gives up raises the timeout bit and both CTAs
// meet at the final cluster barrier before TMEM is freed.
#include <mutex>

#include "gemm_common.cuh"

namespace moe {

// token columns of a pair tile: its rows rounded up to 16 (each CTA then
// holds a multiple of 8 rows, whole 128-byte swizzle atoms), at most the
// tile width
__device__ __forceinline__ int pair_cols(const int4& tile) {
  const int r = (tile.z + 15) & ~15;
  return r < tile.w ? r : tile.w;
}

// the smallest half-tile map (8, 16, 32, 64 or 128 rows) that holds h rows
__device__ __forceinline__ int half_map_index(int h) {
  return h <= 8 ? 0 : h <= 16 ? 1 : h <= 32 ? 2 : h <= 64 ? 3 : 4;
}

// epilogue warps of a pair CTA: with a single GEMM1 accumulator slot the
// MMAs wait for the drain, so it is spread over more warps than in the
// single-CTA kernel
constexpr int kPairEpiWarps = 16;
// warp 0 producer, warp 1 first MMA issuer, warps 2 .. 17 epilogue, the last
// warp the second MMA issuer (GEMM1 up rows)
constexpr int kPairMmaWarp2 = 2 + kPairEpiWarps;
constexpr int kPairThreads = 96 + 32 * kPairEpiWarps;

template <int KIND, int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    moe_gemm_pair_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs args) {
  constexpr int G = MODE - 1;           // which GEMM
  constexpr int NA = MODE == 1 ? 2 : 1;  // 128-row weight tiles per CTA and K block
  // K blocks (128 bytes of K each) per pipeline stage: GEMM2 takes two, so
  // that every stage (and every commit) carries eight MMAs like GEMM1's
  constexpr int KS = MODE == 1 ? 1 : 2;
  constexpr int BKE = 128 / KindTraits<KIND>::esize;
  constexpr int EW = kPairEpiWarps;
  constexpr int EPI_THREADS = EW * 32;
  constexpr int CS = EW / 4;  // column parts per lane quadrant
  extern __shared__ uint8_t smem_raw[];

  const GemmPhase& P = args.p[G];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(cluster_count_x());
  const int S = args.stages;
  const int NS = args.nslots;
  const int NM = args.n_max;  // widest pair tile (both CTAs' token rows)
  const uint32_t sub_bytes = NA * 16384u + static_cast<uint32_t>(NM / 2) * 128u;  // one K block
  const uint32_t stage_bytes = KS * sub_bytes;
  const int nst = (P.kblocks + KS - 1) / KS;  // stages per item (a K block past the end reads zeros)
  const uint32_t slot_cols = static_cast<uint32_t>(NA * NM);
  const uint64_t limit = args.limit_ns;

  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + static_cast<size_t>(S) * stage_bytes);
  uint64_t* empty = full + S;  // [S] stage read by the pair MMAs (both CTAs)
  uint64_t* accf = empty + S;  // [NS] accumulator slot written (both CTAs)
  uint64_t* acce = accf + NS;  // [NS] slot drained by both epilogues (even CTA)
  uint64_t* done = acce + NS;
  uint64_t* epib = done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epib + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* cw = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 512);  // [NM]

  pdl_trigger();
  // A launch whose kernel family the scan picks on the device waits for its
  // predecessors first and leaves at once (both CTAs read the same word)
  // when the other family was picked, holding no TMEM and touching no
  // barrier.
  if (args.family) {
    pdl_wait();
    if (*args.family != args.family_want) return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);  // the even CTA's: its producer's arrival + bytes
      mbar_init(smem_u32(&empty[s]), 2);  // a commit from each MMA issuer
    }
    for (int b = 0; b < NS; ++b) {
      mbar_init(smem_u32(&accf[b]), 2);
      mbar_init(smem_u32(&acce[b]), 2 * EW);
    }
    mbar_init(smem_u32(done), 2);
    mbar_init(smem_u32(epib), EW);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.a);
    for (int j = 0; j < kTokMaps; ++j) prefetch_tmap(&maps.b[j]);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), args.tmem_cols);
    tmem_relinquish_pair();
  }
  // barriers of both CTAs initialised and TMEM allocated before any use
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (!args.family) pdl_wait();  // the tile list and token rows are the predecessors' output

  const int nwork = (*P.ntiles) * P.mblocks;
  int never = 0;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      const uint32_t full_even = mapa_shared(smem_u32(full), 0);
      uint32_t it = 0;
      // each role reads the next item's tile one item ahead, so that the
      // load's latency overlaps the current item
      int4 next = cid < nwork ? P.tiles[cid / P.mblocks] : int4{0, 0, 0, 0};
      for (int w = cid; w < nwork && ok; w += ncl) {
        const int4 tile = next;
        if (w + ncl < nwork) next = P.tiles[(w + ncl) / P.mblocks];
        const int mb = w % P.mblocks;
        const int h = pair_cols(tile) / 2;  // token rows of this CTA
        const int mi = half_map_index(h);
        const uint32_t tx = KS * (NA * 16384u + (8u << mi) * 128u);  // bytes this CTA loads
        const int a_row = tile.x * P.a_rows_per_e + mb * P.row_step + 128 * static_cast<int>(rank);
        const int t_row = tile.y + static_cast<int>(rank) * h;
        for (int kb = 0; kb < nst; ++kb, ++it) {
          const int s = static_cast<int>(it % S);
          if (!mbar_wait(smem_u32(&empty[s]), ((it / S) & 1u) ^ 1u, limit, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t st = smem_u32(stages + static_cast<size_t>(s) * stage_bytes);
          const uint32_t fb = full_even + 8u * static_cast<uint32_t>(s);
          // the even CTA expects both CTAs' bytes (equal boxes on both sides)
          if (leader) mbar_arrive_expect_tx(smem_u32(&full[s]), 2u * tx);
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            const uint32_t sk = st + kk * sub_bytes;
            const int kx = (kb * KS + kk) * BKE;
            tma_load_2d_pair(sk, &maps.a, fb, kx, a_row, pol_w);
            if (NA == 2)
              tma_load_2d_pair(sk + 16384u, &maps.a, fb, kx, a_row + P.a_up_off, pol_w);
            tma_load_2d_pair(sk + NA * 16384u, &maps.b[mi], fb, kx, t_row, pol_x);
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(args.err, kDevErrTimeout);
      }
      // never leave with copies in flight: the last S stages issued have
      // been read by the MMAs (so their bytes landed) once `empty` flips
      for (uint32_t j = (it > static_cast<uint32_t>(S) ? it - S : 0u); j < it; ++j)
        mbar_wait(smem_u32(&empty[j % S]), (j / S) & 1u, limit, &never);
    }
    __syncwarp();
  } else if (warp == 1 || warp == kPairMmaWarp2) {
    // ------------------------------------------------------------ MMA issuers (even CTA)
    // GEMM1's gate and up MMAs come from two threads in different warps
    // (separate accumulators): below N = 256 a pair MMA's issue cost on one
    // thread exceeds its tensor time.  GEMM2's MMAs all accumulate into one
    // slot and stay on the first issuer, so that their order (and rounding)
    // is fixed; the second issuer still commits to every barrier, each of
    // which takes two arrivals.
    const int my_a = warp == 1 ? 0 : 1;
    if (lane == 0 && leader) {
      uint32_t it = 0, tc = 0;
      int4 next = cid < nwork ? P.tiles[cid / P.mblocks] : int4{0, 0, 0, 0};
      for (int w = cid; w < nwork && ok; w += ncl) {
        const int4 tile = next;
        if (w + ncl < nwork) next = P.tiles[(w + ncl) / P.mblocks];
        const uint32_t idesc =
            idesc_make(KindTraits<KIND>::fmt, 256, static_cast<uint32_t>(pair_cols(tile)));
        const uint32_t buf = tc % NS;
        if (!mbar_wait_cluster(smem_u32(&acce[buf]), ((tc / NS) & 1u) ^ 1u, limit, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + buf * slot_cols;
        for (int kb = 0; kb < nst; ++kb, ++it) {
          const int s = static_cast<int>(it % S);
          if (!mbar_wait(smem_u32(&full[s]), (it / S) & 1u, limit, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(stages + static_cast<size_t>(s) * stage_bytes);
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            const uint32_t sk = sa + kk * sub_bytes;
            const uint64_t bd0 = sdesc_sw128(sk + NA * 16384u);
#pragma unroll
            for (int a = 0; a < NA; ++a) {
              if (a != my_a) continue;
              const uint64_t ad0 = sdesc_sw128(sk + a * 16384u);
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                mma_issue_pair<KIND>(d + a * NM, ad0 + 2u * ks, bd0 + 2u * ks, idesc,
                                     (kb | kk | ks) != 0);
            }
          }
          mma_commit_pair(smem_u32(&empty[s]), 3);  // frees the stage in both CTAs
        }
        if (!ok) break;
        mma_commit_pair(smem_u32(&accf[buf]), 3);
        ++tc;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(args.err, kDevErrTimeout);
      }
      // never free TMEM under a running MMA
      mma_commit_pair(smem_u32(done), 1);
      mbar_wait(smem_u32(done), 0, limit, &never);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int q = warp & 3;    // TMEM lane quadrant this warp may read
    const int part = ew >> 2;  // which quarter of the token columns
    const int r_in_tile = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t acce_even = mapa_shared(smem_u32(acce), 0);
    uint32_t tc = 0, eb = 0;
    auto ep_barrier = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(epib));
      const bool got = mbar_wait(smem_u32(epib), eb & 1u, limit, abort_flag);
      ++eb;
      return __all_sync(0xffffffffu, got);
    };
    int4 next = cid < nwork ? P.tiles[cid / P.mblocks] : int4{0, 0, 0, 0};
    for (int w = cid; w < nwork && ok; w += ncl) {
      const int4 tile = next;
      if (w + ncl < nwork) next = P.tiles[(w + ncl) / P.mblocks];
      const int mb = w % P.mblocks;
      const int row0 = tile.y, nrows = tile.z;
      const int n = pair_cols(tile);
      // this thread's output row: a feature of GEMM1 (gate and up share it)
      // or an output row of GEMM2
      const int row = mb * P.row_step + 128 * static_cast<int>(rank) + r_in_tile;
      const bool row_ok = row < P.m_valid;
      if (MODE == 2) {
        if (!ep_barrier()) {  // the previous item's readers of cw are done
          ok = false;
          break;
        }
        for (int j = ew * 32 + lane; j < n; j += EPI_THREADS)
          cw[j] = (j < nrows) ? __ldg(args.topw + __ldg(args.src + row0 + j)) : 0.0f;
        if (!ep_barrier()) {
          ok = false;
          break;
        }
      }
      const uint32_t buf = tc % NS;
      const bool got = mbar_wait(smem_u32(&accf[buf]), (tc / NS) & 1u, limit, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // this warp's share of the n columns, in whole 8-column groups
      const int ng = n >> 3;
      const int c_begin = ((part * ng) / CS) * 8;
      const int c_end = (((part + 1) * ng) / CS) * 8;
      const uint32_t taddr = lane_addr + buf * slot_cols;
      if constexpr (MODE == 1 && KIND == KIND_BF16) {
        // GEMM1 has a single accumulator slot, so the MMAs of the next item
        // wait for it: read every column of this warp (at most 64) and
        // reduce it to packed bf16 act first, free the slot, then store
        uint32_t pk[32];
        const int ncols = c_end - c_begin;
#pragma unroll
        for (int r = 0; r < 4; ++r) {  // 16 columns per round
          if (r * 16 < ncols) {        // warp-uniform
            const int c = c_begin + r * 16;
            float g0[8], u0[8], g1[8], u1[8];
            tmem_ld8(taddr + c, g0);
            tmem_ld8(taddr + NM + c, u0);
            const bool two = r * 16 + 8 < ncols;
            if (two) {
              tmem_ld8(taddr + c + 8, g1);
              tmem_ld8(taddr + NM + c + 8, u1);
            }
            tmem_wait_ld(g0, u0, g1, u1);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              pk[r * 8 + j] = pack_bf16x2(silu_f(g0[2 * j]) * u0[2 * j],
                                          silu_f(g0[2 * j + 1]) * u0[2 * j + 1]);
              pk[r * 8 + 4 + j] = pack_bf16x2(silu_f(g1[2 * j]) * u1[2 * j],
                                              silu_f(g1[2 * j + 1]) * u1[2 * j + 1]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acce_even + 8u * buf);
        if (row_ok) {
          __nv_bfloat16* act = static_cast<__nv_bfloat16*>(args.act);
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int cl = r * 16 + 2 * j;  // column within this warp's share
              const int col = c_begin + cl;
              if (cl < ncols && col < nrows) {
                act[static_cast<size_t>(row0 + col) * args.I + row] =
                    __ushort_as_bfloat16(static_cast<unsigned short>(pk[r * 8 + j] & 0xffffu));
                if (col + 1 < nrows)
                  act[static_cast<size_t>(row0 + col + 1) * args.I + row] =
                      __ushort_as_bfloat16(static_cast<unsigned short>(pk[r * 8 + j] >> 16));
              }
            }
        }
      } else {
        for (int c = c_begin; c < c_end;) {
          if (c_end - c >= 32) {
            epi_chunk<KIND, 32>(args, G, NA, taddr, NM, c, row0, nrows, row, row_ok, row, false,
                                cw);
            c += 32;
          } else {
            epi_chunk<KIND, 8>(args, G, NA, taddr, NM, c, row0, nrows, row, row_ok, row, false,
                               cw);
            c += 8;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acce_even + 8u * buf);
      }
      ++tc;
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) atomicOr(args.err, kDevErrTimeout);
    }
  }

  // neither CTA leaves (or frees TMEM) while the other may still touch its
  // shared memory, barriers or TMEM
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, args.tmem_cols);
}

template <int KIND, int MODE>
static cudaError_t launch_pair_mode(const GemmArgs& args, const GemmMaps& maps, int smem,
                                    long long max_items, cudaStream_t stream) {
  auto kern = moe_gemm_pair_kernel<KIND, MODE>;
  // max dynamic smem (a per-function attribute) and the co-resident cluster
  // count at that size, set up once per size and device; host threads may
  // launch concurrently
  static std::mutex mu;
  static int configured = 0, conf_dev = -1, clusters = 0;
  int dev = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return de;
  std::lock_guard<std::mutex> lock(mu);
  if (dev != conf_dev || configured != smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = smem;
    conf_dev = dev;
    clusters = 0;
  }
  if (clusters == 0) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kPairThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    clusters = n;
  }
  // a persistent grid: every cluster resident at once
  const long long ncl = max_items < clusters ? (max_items > 0 ? max_items : 1) : clusters;
  return launch_chained(kern, dim3(static_cast<unsigned>(2 * ncl)), dim3(kPairThreads),
                        static_cast<size_t>(smem), stream, maps, args);
}

cudaError_t launch_grouped_gemm_pair(int kind, int mode, const GemmArgs& args,
                                     const GemmMaps& maps, int smem, long long max_items,
                                     cudaStream_t stream) {
  if (args.nslots < 1 || args.nslots > 2 || args.n_max > 256 || (args.n_max & 15))
    return cudaErrorInvalidValue;
  if (kind == KIND_BF16)
    return mode == 1 ? launch_pair_mode<KIND_BF16, 1>(args, maps, smem, max_items, stream)
                     : launch_pair_mode<KIND_BF16, 2>(args, maps, smem, max_items, stream);
  if (kind == KIND_TF32)
    return mode == 1 ? launch_pair_mode<KIND_TF32, 1>(args, maps, smem, max_items, stream)
                     : launch_pair_mode<KIND_TF32, 2>(args, maps, smem, max_items, stream);
  return cudaErrorInvalidValue;
}

}  // namespace moe
