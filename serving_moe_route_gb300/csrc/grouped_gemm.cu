// grouped_gemm.cu -- tcgen05/TMEM grouped GEMMs of the fused MoE layer
// (steps a-4 .. a-7), fed by TMA, for TF32, BF16 and block-scaled FP8 e4m3.
//
// One persistent CTA per SM walks a device-built list of work items
// (token tile x 128-row weight block).  Swap-AB orientation: the MMA's M
// side is 128 rows of one expert's weight matrix, its N side a tile of n
// permuted token rows of that expert, n = 16 .. 256 set per expert from its
// row count with the rows-per-expert estimate as the floor (H20 article,
// para. 3), so a decode-sized expert with a handful of rows still fills the
// 128-wide M side with weights and a hot expert gets wide tiles.
//
// GEMM1 (gate+up, a-4/a-5) and GEMM2 (down, a-6/a-7) run as one launch when
// they share a tile list: GEMM2 items follow all GEMM1 items in the work
// list, and a GEMM2 item waits until every GEMM1 item of its token tile has
// written its activations (a per-tile counter released by the GEMM1
// epilogue), so CTAs that run out of GEMM1 work start GEMM2 work at once.
//
//   warp 0      TMA producer: weight tile(s) + token tile per 128-byte K step
//   warp 1      TMEM allocator; tcgen05.mma issuer of weight tile 0
//   warp 10     tcgen05.mma issuer of weight tile 1 (GEMM1 up rows, GEMM2's
//               second 128 output rows): at small N one thread's issue cost
//               sets the MMA rate, so the two tiles' MMAs come from two
//   warps 2..9  epilogue: tcgen05.ld from TMEM, then
//                 GEMM1: act = SiLU(gate) * up  (FP8: + per-token 128-group
//                        e4m3 quantisation, clamp with fminf/fmaxf as in
//                        PR #39593 "Purpose")
//                 GEMM2: ybuf[row] = w[t,j] * y  (the combine's weighting;
//                        the k rows of a token are summed by the combine
//                        kernel)
//
// FP8 [128,128] block scales (Lab notes #6, config file line): each 128-K
// block is accumulated into its own TMEM slot; the slots form groups (four
// once there are eight slots or more, else two) handed between the MMA
// warps and the epilogue as a unit, and the epilogue folds every block into fp32 registers with the
// product weight-scale x activation-scale, so arbitrary fp32 scales are
// honoured.  FP8 kernels are specialised per tile width (16/32/64; the
// gate and up register accumulators of a 128-wide tile would not fit).
//
// Every wait is bounded (see mbar_wait / wait_counter); a timeout sets
// MOE_DEVERR_TIMEOUT in the error word, raises a CTA-wide abort flag, drains
// in-flight copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <mutex>

#include "gemm_common.cuh"
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kMaxSlots = 16;
constexpr int kQueue = 8;  // work items handed from the producer to MMA + epilogue

// Work item w of a launch: GEMM g (0 or 1), token tile t of that GEMM's
// list, 128-row weight block mb.
struct Item {
  int g, t, mb;
  int4 tile;
};

// Token columns the MMAs of a tile compute: its rows rounded up to the MMA's
// 16-column step, at most the tile width.  The last tile of an expert is
// usually partly filled; computing only its rows keeps the tensor work of a
// skewed batch close to the rows routed (the columns beyond are never read).
template <int NT>
__device__ __forceinline__ int mma_cols(const int4& tile) {
  const int w = NT > 0 ? NT : tile.w;
  const int r = (tile.z + 15) & ~15;
  return r < w ? r : w;
}

__device__ __forceinline__ Item item_at(const GemmArgs& A, int w, int nwork1) {
  Item it;
  if (w < nwork1) {
    it.g = 0;
    it.t = w / A.p[0].mblocks;
    it.mb = w % A.p[0].mblocks;
  } else {
    const int v = w - nwork1;
    it.g = 1;
    it.t = v / A.p[1].mblocks;
    it.mb = v % A.p[1].mblocks;
  }
  it.tile = A.p[it.g].tiles[it.t];
  return it;
}

// NT = 0: runtime tile width per work item (BF16/TF32, per-expert widths);
// NT > 0: fixed width (FP8, the plan's tile).  MODE 1: GEMM1 items only,
// 2: GEMM2 items only, 3: both (fused); single-GEMM kernels carry only
// their own epilogue.
template <int KIND, int NT, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ GemmMaps maps1, const __grid_constant__ GemmMaps maps2,
                    const GemmArgs args) {
  constexpr bool FP8 = (KIND == KIND_E4M3);
  static_assert(!FP8 || NT > 0, "FP8 kernels are specialised per tile width");
  static_assert(NT <= 64, "FP8 register accumulators hold at most 2 x 32 columns");
  constexpr int BKE = 128 / KindTraits<KIND>::esize;  // elements per 128-byte K step
  constexpr int EPI_THREADS = kEpiWarps * 32;
  constexpr int CS = kEpiWarps / 4;          // column splits per lane quadrant
  constexpr int CPT = NT > 0 ? NT / CS : 8;  // FP8 columns per epilogue thread
  extern __shared__ uint8_t smem_raw[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = args.stages;
  const int NS = args.nslots;
  // FP8: the slots are handed between the MMAs and the epilogue in NG groups
  // of GS K blocks (four groups once there are 8 slots or more, so that the
  // epilogue frees slots often enough for the MMAs not to wait on it)
  const uint32_t ng_shift = (FP8 && NS >= 8) ? 2u : 1u;
  const uint32_t NG = 1u << ng_shift;
  const int GS = FP8 ? (NS >> ng_shift) : 1;  // FP8: K blocks per handed-over group
  const int NM = args.n_max;
  const int NAM = args.na_max;
  const uint32_t stage_bytes = NAM * 16384u + static_cast<uint32_t>(NM) * 128u;
  const uint32_t slot_cols = static_cast<uint32_t>(NAM * NM);
  const uint64_t limit = args.limit_ns;
  const int kb_max = args.p[0].kblocks > args.p[1].kblocks ? args.p[0].kblocks
                                                            : args.p[1].kblocks;

  // ---- shared memory carve-up (stage ring 1024-aligned for 128B swizzle)
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + static_cast<size_t>(S) * stage_bytes);
  uint64_t* empty = full + S;
  uint64_t* accf = empty + S;  // [NS] accumulator (group) written by the MMAs
  uint64_t* acce = accf + NS;  // [NS] accumulator (group) drained by the epilogue
  uint64_t* done = acce + NS;  // all MMAs of this CTA complete
  uint64_t* epib = done + 1;   // epilogue-internal barrier
  uint64_t* qfull = epib + 1;  // [kQueue] work-queue entry written
  uint64_t* qempty = qfull + kQueue;  // [kQueue] entry read by the MMA thread and the epilogue
  // [kQueue] work items (index w, -1 = end, and the item's tile) handed over
  Item* queue = reinterpret_cast<Item*>(
      (reinterpret_cast<uintptr_t>(qempty + kQueue) + 15) & ~static_cast<uintptr_t>(15));
  int* queue_w = reinterpret_cast<int*>(queue + kQueue);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(queue_w + kQueue);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* cs = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 1024);
  // FP8: [4][NM] per-column amax per lane quadrant and [NM] reciprocal
  // scales (GEMM1), column weights (GEMM2)
  float* red = cs + 2 * kb_max * NM;

  pdl_trigger();
  auto early_prefetch = [&]() {
    if (MODE == 2 || !args.spec_hint || warp != 0 || lane != 0) return;
    // The routing, scan and gather kernels are still running and HBM is
    // mostly idle.  With about one tile per expert in expert order (routing
    // that touches nearly every expert, judged by the previous call), this
    // CTA's first work item is likely item blockIdx.x: expert
    // blockIdx.x / mblocks.  The weights are an input, not a predecessor's
    // output, so its first K blocks can be brought into L2 now; a wrong
    // guess costs only idle bandwidth.
    const GemmPhase& P0 = args.p[0];
    const unsigned h = ld_relaxed_gpu(args.spec_hint);
    const bool wide = (h & 0xffff0000u) == kSpecHintTag &&
                      static_cast<int>(h & 0xffffu) >= args.spec_min;
    const int e = static_cast<int>(blockIdx.x) / P0.mblocks;
    if (wide && e < args.spec_experts) {
      const int a_row = e * P0.a_rows_per_e + (static_cast<int>(blockIdx.x) % P0.mblocks) * P0.row_step;
      const int nk = P0.kblocks < 16 ? P0.kblocks : 16;
      for (int kb = 0; kb < nk; ++kb) {
        tma_prefetch_2d(&maps1.a, kb * BKE, a_row);
        tma_prefetch_2d(&maps1.a, kb * BKE, a_row + P0.a_up_off);
      }
    }
  };
  // A launch whose kernel family the scan picks on the device waits for its
  // predecessors first and leaves at once when the other family was picked,
  // holding no TMEM and touching no barrier.
  if (args.family) {
    early_prefetch();
    pdl_wait();
    if (*args.family != args.family_want) return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 2);  // a commit from each MMA issuer
    }
    // epilogue-side barriers take one arrival per epilogue warp (lane 0,
    // after __syncwarp orders the warp's TMEM loads and shared stores)
    for (int b = 0; b < NS; ++b) {
      mbar_init(smem_u32(&accf[b]), 2);
      mbar_init(smem_u32(&acce[b]), kEpiWarps);
    }
    mbar_init(smem_u32(done), 2);
    mbar_init(smem_u32(epib), kEpiWarps);
    for (int i = 0; i < kQueue; ++i) {
      mbar_init(smem_u32(&qfull[i]), 1);
      mbar_init(smem_u32(&qempty[i]), 2 + kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < 2; ++i) {
      const GemmMaps& M = i ? maps2 : maps1;
      if (i ? args.run2 : args.run1) {
        prefetch_tmap(&M.a);
        for (int j = 0; j < kTokMaps; ++j) prefetch_tmap(&M.b[j]);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), args.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // everything above is local set-up; the tile lists and token rows are the
  // predecessor kernels' output
  if (!args.family) {
    early_prefetch();
    pdl_wait();
  }

  const int nwork1 = args.run1 ? (*args.p[0].ntiles) * args.p[0].mblocks : 0;
  const int nwork2 = args.run2 ? (*args.p[1].ntiles) * args.p[1].mblocks : 0;
  const int nwork = nwork1 + nwork2;
  int never = 0;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();  // weights: streamed once
      const uint64_t pol_x = policy_evict_last();   // token tiles: reused per block
      uint32_t it = 0, qi = 0;
      // Fused launches take items in list order from a global counter (CTAs
      // that finish early take more); the index after the current one is
      // taken one item ahead so the atomic's latency overlaps the loads.
      // Single-GEMM launches walk the list with a grid stride.
      int w_next = MODE == 3 ? atomicAdd(args.work_counter, 1) : static_cast<int>(blockIdx.x);
      Item nxt{};  // the next item's tile, loaded one item ahead
      if (w_next < nwork) nxt = item_at(args, w_next, nwork1);
      while (ok) {
        const int w = w_next < nwork ? w_next : -1;
        Item I = nxt;
        if constexpr (MODE == 3) {
          // hand the item to the MMA thread and the epilogue
          const int qs = static_cast<int>(qi % kQueue);
          if (!mbar_wait(smem_u32(&qempty[qs]), ((qi / kQueue) & 1u) ^ 1u, limit, abort_flag)) {
            ok = false;
            break;
          }
          queue[qs] = I;
          queue_w[qs] = w;
          mbar_arrive(smem_u32(&qfull[qs]));
          ++qi;
        }
        if (w < 0) break;
        w_next = MODE == 3 ? atomicAdd(args.work_counter, 1) : w + static_cast<int>(gridDim.x);
        if (w_next < nwork) nxt = item_at(args, w_next, nwork1);
        if constexpr (MODE != 3) I.g = MODE - 1;
        const GemmPhase& P = args.p[I.g];
        const GemmMaps& M = I.g ? maps2 : maps1;
        const int na = MODE == 1 ? 2 : (MODE == 2 && !FP8) ? 1 : P.na;  // single-GEMM launches: fixed
        // the box: the smallest map height that holds the tile's rows
        // rounded up to the MMA's 16-column step
        const int nbox = 16 << tok_map_index(mma_cols<NT>(I.tile));
        const int a_row = I.tile.x * P.a_rows_per_e + I.mb * P.row_step;
        const uint32_t tx = na * 16384u + static_cast<uint32_t>(nbox) * 128u;
        const CUtensorMap* tmb = &M.b[tok_map_index(nbox)];  // one box of nbox token rows
        if (MODE == 3 && I.g == 1) {
          // this tile's activations are written by GEMM1 items of other CTAs
          if (!wait_counter(args.dep + I.t, args.p[0].mblocks, limit, abort_flag)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
        }
        for (int kb = 0; kb < P.kblocks; ++kb, ++it) {
          const int s = static_cast<int>(it % S);
          if (!mbar_wait(smem_u32(&empty[s]), ((it / S) & 1u) ^ 1u, limit, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* st = stages + static_cast<size_t>(s) * stage_bytes;
          const uint32_t fb = smem_u32(&full[s]);
          mbar_arrive_expect_tx(fb, tx);
          const int kx = kb * BKE;
          tma_load_2d(smem_u32(st), &M.a, fb, kx, a_row, pol_w);
          if (na == 2) tma_load_2d(smem_u32(st + 16384), &M.a, fb, kx, a_row + P.a_up_off, pol_w);
          tma_load_2d(smem_u32(st + NAM * 16384), tmb, fb, kx, I.tile.y, pol_x);
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
  } else if (warp == 1 || warp == kMmaWarp2) {
    // ------------------------------------------------------------ MMA issuers
    // Two threads in different warps issue the MMAs of each K block: the
    // first those of weight tile 0 (GEMM1 gate rows), the second those of
    // tile 1 (up rows, or GEMM2's second 128 output rows).  At small N an
    // MMA's issue cost on one thread, not the tensor pipe, sets the pace
    // (about 110 cycles per MMA from one thread against 56 from two, for
    // M=128, N<=64), so two issuers double the K blocks a CTA can consume.
    // Both walk the same items and stages and both commit to every stage,
    // accumulator and final barrier (each of which takes two arrivals).
    const int my_a = warp == 1 ? 0 : 1;
    if (lane == 0) {
      uint32_t it = 0, tc = 0, gc = 0, qi = 0;
      int w_static = static_cast<int>(blockIdx.x);
      Item nxt{};
      if (MODE != 3 && w_static < nwork) nxt = item_at(args, w_static, nwork1);
      while (ok) {
        int w;
        Item I;
        if constexpr (MODE == 3) {
          const int qs = static_cast<int>(qi % kQueue);
          if (!mbar_wait(smem_u32(&qfull[qs]), (qi / kQueue) & 1u, limit, abort_flag)) {
            ok = false;
            break;
          }
          w = queue_w[qs];
          I = queue[qs];
          mbar_arrive(smem_u32(&qempty[qs]));
          ++qi;
        } else {
          w = w_static < nwork ? w_static : -1;
          I = nxt;
          w_static += gridDim.x;
          if (w >= 0 && w_static < nwork) nxt = item_at(args, w_static, nwork1);
          I.g = MODE - 1;
        }
        if (w < 0) break;
        const int na = MODE == 1 ? 2 : (MODE == 2 && !FP8) ? 1 : args.p[I.g].na;
        const int kbs = args.p[I.g].kblocks;
        const uint32_t idesc =
            idesc_make(KindTraits<KIND>::fmt, 128, static_cast<uint32_t>(mma_cols<NT>(I.tile)));
        uint32_t dbase = 0, buf = 0;
        if (!FP8) {
          buf = tc % NS;
          if (!mbar_wait(smem_u32(&acce[buf]), ((tc / NS) & 1u) ^ 1u, limit, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          dbase = buf * slot_cols;
        }
        for (int kb = 0; kb < kbs; ++kb, ++it) {
          const int s = static_cast<int>(it % S);
          if (FP8 && kb % GS == 0) {  // a new group of K blocks: its slots must be drained
            buf = gc & (NG - 1u);
            if (!mbar_wait(smem_u32(&acce[buf]), ((gc >> ng_shift) & 1u) ^ 1u, limit, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          if (!mbar_wait(smem_u32(&full[s]), (it / S) & 1u, limit, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (FP8) dbase = (buf * GS + static_cast<uint32_t>(kb % GS)) * slot_cols;
          const uint32_t sa = smem_u32(stages + static_cast<size_t>(s) * stage_bytes);
          // descriptors built once per stage; each 32-byte K step adds 2 to
          // the encoded start address (addresses stay below 256 KB)
          const uint64_t bd0 = sdesc_sw128(sa + NAM * 16384);
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            if (a < na && a == my_a) {
              const uint64_t ad0 = sdesc_sw128(sa + a * 16384);
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                const uint32_t accumulate = FP8 ? (ks != 0) : ((kb | ks) != 0);
                mma_issue<KIND>(tmem_base + dbase + a * NM, ad0 + 2u * ks, bd0 + 2u * ks, idesc,
                                accumulate);
              }
            }
          }
          mma_commit(smem_u32(&empty[s]));  // frees the stage once read
          if (FP8 && (kb % GS == GS - 1 || kb == kbs - 1)) {
            mma_commit(smem_u32(&accf[buf]));
            ++gc;
          }
        }
        if (!ok) break;
        if (!FP8) {
          mma_commit(smem_u32(&accf[buf]));
          ++tc;
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
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int q = warp & 3;    // TMEM lane quadrant this warp may read
    const int part = ew >> 2;  // which half of the token columns
    const int r_in_tile = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t tc = 0, gc = 0, eb = 0, qi = 0;

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

    int w_static = static_cast<int>(blockIdx.x);
    Item nxt{};
    if (MODE != 3 && w_static < nwork) nxt = item_at(args, w_static, nwork1);
    while (ok) {
      int w;
      Item I;
      if constexpr (MODE == 3) {
        const int qs = static_cast<int>(qi % kQueue);
        const bool gotq = mbar_wait(smem_u32(&qfull[qs]), (qi / kQueue) & 1u, limit, abort_flag);
        if (!__all_sync(0xffffffffu, gotq)) {
          ok = false;
          break;
        }
        w = queue_w[qs];
        I = queue[qs];
        warp_arrive(&qempty[qs]);
        ++qi;
      } else {
        w = w_static < nwork ? w_static : -1;
        I = nxt;
        w_static += gridDim.x;
        if (w >= 0 && w_static < nwork) nxt = item_at(args, w_static, nwork1);
        I.g = MODE - 1;
      }
      if (w < 0) break;
      const GemmPhase& P = args.p[I.g];
      const int na = MODE == 1 ? 2 : (MODE == 2 && !FP8) ? 1 : P.na;  // single-GEMM launches: fixed
      const int row0 = I.tile.y, nrows = I.tile.z;
      // output row of accumulator a: GEMM1 gate and up share a feature row;
      // GEMM2's second weight tile covers the next 128 output rows
      const int row = I.mb * P.row_step + r_in_tile;
      const int row_b = I.g ? row + 128 : row;
      const bool row_ok = row < P.m_valid;
      const bool row_b_ok = row_b < P.m_valid;

      if constexpr (!FP8) {
        const int n = mma_cols<NT>(I.tile);
        const int hc = n / CS;  // columns per thread (a multiple of 8)
        const int c_begin = part * hc;
        float* cw = cs;  // GEMM2: routing weight of each token column of this tile
        if (I.g == 1) {
          if (!ep_barrier()) {  // the previous tile's readers are done
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
        const uint32_t sl = tc % NS;
        const bool got = mbar_wait(smem_u32(&accf[sl]), (tc / NS) & 1u, limit, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dcol = sl * slot_cols;
        for (int c0 = 0; c0 < hc;) {  // 32-column chunks while they fit, then 8
          if (hc - c0 >= 32) {
            epi_chunk<KIND, 32>(args, I.g, na, lane_addr + dcol, NM, c_begin + c0, row0, nrows, row,
                                row_ok, row_b, row_b_ok, cw);
            c0 += 32;
          } else {
            epi_chunk<KIND, 8>(args, I.g, na, lane_addr + dcol, NM, c_begin + c0, row0, nrows, row,
                               row_ok, row_b, row_b_ok, cw);
            c0 += 8;
          }
        }
        tc_fence_before();
        warp_arrive(&acce[sl]);
        ++tc;
      } else {
        // -------- FP8: per-column scale products cs[a][kb][j] = s_w[a][kb] * s_x[j][kb]
        const int kbs = P.kblocks;
        const int c_begin = part * CPT;
        if (MODE == 3 && I.g == 1) {
          // the activation scales of this tile come from GEMM1 items of
          // other CTAs in this launch: acquire them (already released)
          const bool got = wait_counter(args.dep + I.t, args.p[0].mblocks, limit, abort_flag);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
        }
        if (!ep_barrier()) {
          ok = false;
          break;
        }
        const float* sw = P.w_scale + (static_cast<size_t>(I.tile.x) * P.w_scale_rows_per_e +
                                       I.mb * (P.row_step / 128)) * kbs;
        // eight products per thread and pass, their loads issued together
        const int ncs = na * kbs * NT;
        for (int i0 = ew * 32 + lane; i0 < ncs; i0 += 8 * EPI_THREADS) {
          float swv[8], bsv[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * EPI_THREADS;
            swv[u] = 0.0f;
            bsv[u] = 0.0f;
            if (i < ncs) {
              const int a = i / (kbs * NT);
              const int kb = (i / NT) % kbs;
              const int j = i % NT;
              if (j < nrows) {
                swv[u] = __ldg(sw + static_cast<size_t>(a) * (P.a_up_off / 128) * kbs + kb);
                const float* bs = P.b_scale + static_cast<size_t>(row0 + j) * kbs + kb;
                // fused: GEMM2's scales are written in this launch, so read
                // them through L2 (coherent) rather than the read-only path
                bsv[u] = MODE == 3 ? __ldcg(bs) : __ldg(bs);
              }
            }
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * EPI_THREADS;
            if (i < ncs) cs[i] = swv[u] * bsv[u];
          }
        }
        if (I.g == 1)  // GEMM2: the routing weight of each token column
          for (int j = ew * 32 + lane; j < NT; j += EPI_THREADS)
            red[j] = (j < nrows) ? __ldg(args.topw + __ldg(args.src + row0 + j)) : 0.0f;
        if (!ep_barrier()) {
          ok = false;
          break;
        }
        float acc0[CPT], acc1[CPT];  // acc1: up (GEMM1) or the second 128 rows (GEMM2)
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          acc0[c] = 0.0f;
          acc1[c] = 0.0f;
        }
        for (int kb0 = 0; kb0 < kbs; kb0 += GS, ++gc) {
          const uint32_t buf = gc & (NG - 1u);
          const bool got = mbar_wait(smem_u32(&accf[buf]), (gc >> ng_shift) & 1u, limit, abort_flag);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int kend = kb0 + GS < kbs ? kb0 + GS : kbs;
          for (int kb = kb0; kb < kend; ++kb) {
            const uint32_t dcol = (buf * GS + static_cast<uint32_t>(kb - kb0)) * slot_cols;
            const float* c0p = cs + kb * NT + c_begin;
            const float* c1p = cs + (kbs + kb) * NT + c_begin;
            // this thread's columns of the block in chunks of up to 16, one
            // wait per chunk
            constexpr int FC = CPT < 16 ? CPT : 16;
#pragma unroll
            for (int f0 = 0; f0 < CPT; f0 += FC) {
              float p0[FC], p1[FC];
              tmem_ld<FC>(lane_addr + dcol + c_begin + f0, p0);
              if (na == 2) {
                tmem_ld<FC>(lane_addr + dcol + NM + c_begin + f0, p1);
                tmem_wait_ld(p0, p1);
              } else {
                tmem_wait_ld(p0);
              }
#pragma unroll
              for (int c0 = 0; c0 < FC; c0 += 4) {
                const float4 s0 = *reinterpret_cast<const float4*>(c0p + f0 + c0);
                acc0[f0 + c0] = fmaf(p0[c0], s0.x, acc0[f0 + c0]);
                acc0[f0 + c0 + 1] = fmaf(p0[c0 + 1], s0.y, acc0[f0 + c0 + 1]);
                acc0[f0 + c0 + 2] = fmaf(p0[c0 + 2], s0.z, acc0[f0 + c0 + 2]);
                acc0[f0 + c0 + 3] = fmaf(p0[c0 + 3], s0.w, acc0[f0 + c0 + 3]);
              }
              if (na == 2) {
#pragma unroll
                for (int c0 = 0; c0 < FC; c0 += 4) {
                  const float4 s1 = *reinterpret_cast<const float4*>(c1p + f0 + c0);
                  acc1[f0 + c0] = fmaf(p1[c0], s1.x, acc1[f0 + c0]);
                  acc1[f0 + c0 + 1] = fmaf(p1[c0 + 1], s1.y, acc1[f0 + c0 + 1]);
                  acc1[f0 + c0 + 2] = fmaf(p1[c0 + 2], s1.z, acc1[f0 + c0 + 2]);
                  acc1[f0 + c0 + 3] = fmaf(p1[c0 + 3], s1.w, acc1[f0 + c0 + 3]);
                }
              }
            }
          }
          tc_fence_before();
          warp_arrive(&acce[buf]);
        }
        if (!ok) break;

        if (I.g == 0) {
          // act = SiLU(gate) * up, then e4m3 per token over this 128-row group
          float m[CPT];
#pragma unroll
          for (int c = 0; c < CPT; ++c) {
            acc0[c] = silu_f(acc0[c]) * acc1[c];
            m[c] = fabsf(acc0[c]);
          }
          // each lane ends with the maximum over this warp's 32 rows of one
          // of the warp's columns; the four lane quadrants meet in red[]
          const float wmax = col_max_transpose<CPT>(m, lane);
          if (lane < CPT) red[q * NT + c_begin + lane] = wmax;
          if (!ep_barrier()) {
            ok = false;
            break;
          }
          uint8_t* act_q = static_cast<uint8_t*>(args.act);
          const int groups = args.I / 128;
          float* inv_scale = red + 4 * NT;
          {  // one thread per token column: the group's scale (amax / 448) and its reciprocal
            const int j = ew * 32 + lane;
            if (j < NT) {
              const float amax =
                  fmaxf(fmaxf(red[j], red[NT + j]), fmaxf(red[2 * NT + j], red[3 * NT + j]));
              const float scale = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
              inv_scale[j] = __frcp_rn(scale);
              if (j < nrows) args.act_scale[static_cast<size_t>(row0 + j) * groups + I.mb] = scale;
            }
          }
          if (!ep_barrier()) {
            ok = false;
            break;
          }
#pragma unroll
          for (int c = 0; c < CPT; ++c) {
            const int j = c_begin + c;
            if (j < nrows) {
              // v / scale as v * (1 / scale): at most one fp32 ulp apart,
              // far below the e4m3 step
              float v = acc0[c] * inv_scale[j];
              v = fmaxf(fminf(v, 448.0f), -448.0f);
              act_q[static_cast<size_t>(row0 + j) * args.I + row] =
                  static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < CPT; ++c) {
            const int j = c_begin + c;
            if (j < nrows) {
              const float wt = red[j];
              if (row_ok)
                store_val<KIND_BF16>(args.ybuf, static_cast<size_t>(row0 + j) * args.H + row,
                                     wt * acc0[c]);
              if (na == 2 && row_b_ok)
                store_val<KIND_BF16>(args.ybuf, static_cast<size_t>(row0 + j) * args.H + row_b,
                                     wt * acc1[c]);
            }
          }
        }
      }

      if (MODE == 3 && I.g == 0) {
        // publish this GEMM1 item: all epilogue threads' activation stores
        // become visible (to generic and TMA readers) before the count moves.
        // Each thread orders its stores for the async proxy; the barrier
        // (mbarrier arrive/wait: release/acquire at CTA scope) orders them
        // before the publishing thread, whose GPU-scope fence is cumulative
        // over them -- one fence per item instead of one per thread.
        fence_proxy_async_global();
        if (!ep_barrier()) {
          ok = false;
          break;
        }
        if (ew == 0 && lane == 0) {
          __threadfence();
          atomicAdd(args.dep + I.t, 1);
        }
      }
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) atomicOr(args.err, kDevErrTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, args.tmem_cols);
}

template <int KIND, int NT, int MODE>
static cudaError_t launch_mode(const GemmArgs& args, const GemmMaps* maps, int grid, int smem,
                               cudaStream_t stream) {
  auto kern = moe_gemm_kernel<KIND, NT, MODE>;
  // max dynamic smem is a per-function attribute, raised once per size (and
  // again after a switch of device); host threads may launch concurrently
  static std::mutex mu;
  static int configured = 0, conf_dev = -1;
  {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (dev != conf_dev || configured < smem) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      configured = dev != conf_dev ? smem : (configured > smem ? configured : smem);
      conf_dev = dev;
    }
  }
  return launch_chained(kern, dim3(grid), dim3(kThreads), static_cast<size_t>(smem), stream,
                        maps[0], maps[1], args);
}

template <int KIND, int NT>
static cudaError_t launch_one(const GemmArgs& args, const GemmMaps* maps, int grid, int smem,
                              cudaStream_t stream) {
  if (args.run1 && args.run2) return launch_mode<KIND, NT, 3>(args, maps, grid, smem, stream);
  if (args.run1) return launch_mode<KIND, NT, 1>(args, maps, grid, smem, stream);
  return launch_mode<KIND, NT, 2>(args, maps, grid, smem, stream);
}

cudaError_t launch_grouped_gemm(int kind, const GemmArgs& args, const GemmMaps* maps, int grid,
                                int smem, cudaStream_t stream) {
  if (args.nslots < 1 || args.nslots > kMaxSlots) return cudaErrorInvalidValue;
  if (kind == KIND_TF32) return launch_one<KIND_TF32, 0>(args, maps, grid, smem, stream);
  if (kind == KIND_BF16) return launch_one<KIND_BF16, 0>(args, maps, grid, smem, stream);
  if (args.nslots < 2 || (args.nslots & 1)) return cudaErrorInvalidValue;
  switch (args.n_max) {
    case 16: return launch_one<KIND_E4M3, 16>(args, maps, grid, smem, stream);
    case 32: return launch_one<KIND_E4M3, 32>(args, maps, grid, smem, stream);
    case 64: return launch_one<KIND_E4M3, 64>(args, maps, grid, smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
