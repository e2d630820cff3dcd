// moe_internal.cuh -- declarations shared by the two translation units of
// the library (host API + routing/permutation kernels, grouped GEMMs).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

// operand element kinds of the grouped GEMMs
enum GemmKind : int { KIND_TF32 = 0, KIND_BF16 = 1, KIND_E4M3 = 2 };

// Tensor maps of one grouped GEMM: the weight operand (128-row boxes) and
// the permuted token rows with one map per tile height 16, 32, 64, 128, 256,
// so that every token tile is a single TMA box.
constexpr int kTokMaps = 5;
struct GemmMaps {
  CUtensorMap a;
  CUtensorMap b[kTokMaps];
};

// index into GemmMaps::b of a tile n rows high (n a power of two, 16..256)
__host__ __device__ inline int tok_map_index(int n) {
  return n <= 16 ? 0 : n <= 32 ? 1 : n <= 64 ? 2 : n <= 128 ? 3 : 4;
}

// One of the two grouped GEMMs of the layer.
struct GemmPhase {
  const int4* tiles;        // [max_tiles] {expert, first permuted row, rows, tile n}
  const int* ntiles;        // device count of valid tiles
  int na;                   // 128-row weight tiles per work item (1 or 2)
  int row_step;             // weight rows per item index step (G1: 128; G2: 128 * na)
  int mblocks;              // items per token tile (G1: ceil(I/128), G2: ceil(H/row_step))
  int kblocks;              // K / (128 bytes / element size)
  int a_rows_per_e;         // rows of one expert in the A view (G1: 2I, G2: H)
  int a_up_off;             // rows from the first to the second weight tile (G1: I, G2: 128)
  int m_valid;              // G1: I, G2: H -- weight rows at or beyond are masked
  const float* w_scale;     // FP8 weight block scales (s13 / s2)
  int w_scale_rows_per_e;   // G1: 2I/128, G2: H/128
  const float* b_scale;     // FP8 activation group scales [R, kblocks]
};

// Arguments of one grouped GEMM launch (swap-AB orientation: the MMA's M
// side is 128 weight rows of one expert, its N side a tile of up to n_max
// permuted token rows of that expert; each tile carries its own n).  A
// launch runs GEMM1 items, GEMM2 items, or both: fused, GEMM2 items follow
// GEMM1's in one work list and each waits until all GEMM1 items of its
// token tile have finished (dep counters); there CTAs take items in list
// order through a global counter, so faster CTAs take more items.
struct GemmArgs {
  GemmPhase p[2];      // [0] gate+up GEMM, [1] down GEMM
  int run1, run2;      // which GEMMs this launch runs
  int fused;           // both, sharing tile list p[0]; GEMM2 waits on dep
  int* dep;            // [max_tiles] finished GEMM1 items per tile (fused)
  int* work_counter;   // next work item of this launch (zeroed before the launch)
  int n_max;           // largest tile n (stage and TMEM slot size)
  int na_max;          // weight tiles per stage: 2 if GEMM1 runs, else 1
  int R;               // permuted rows (T*k)
  int stages;          // shared-memory pipeline depth
  int nslots;          // TMEM accumulator slots (per tile; FP8: per 128-K block)
  uint32_t tmem_cols;  // allocated TMEM columns (power of two)
  // GEMM1 output: act [R, I] (f32 / bf16 / e4m3), FP8 group scales [R, I/128]
  void* act;
  float* act_scale;
  int I;
  // GEMM2 output: ybuf[row, h] = w[src[row]] * y[row, h] (bf16, f32 for TF32)
  const int* src;
  const float* topw;
  void* ybuf;
  int H;
  unsigned* err;
  unsigned long long limit_ns;
  // GEMM1 weight prefetch before the predecessor kernels finish: when the
  // word at spec_hint (written by the previous call's scan on this
  // workspace: kSpecHintTag | experts routed to) says that call routed to at
  // least spec_min of the spec_experts local experts, CTA c assumes its
  // first work item is item c of a list with about one tile per expert in
  // expert order, and prefetches that item's first K blocks of weights into
  // L2 while it waits.  The word is read with a relaxed load (the current
  // call's scan may be writing it); it only steers a prefetch.
  int spec_experts;
  int spec_min;
  const unsigned* spec_hint;
  // Kernel family chosen on the device: when family is set, this launch
  // runs only if *family == family_want (written by this call's scan kernel,
  // read after the dependent-launch wait); otherwise it has no work.
  const unsigned* family;
  unsigned family_want;
};

// family words written by the scan kernel of plans that choose the GEMM
// kernel family on the device
constexpr unsigned kFamilySingle = 1u;  // one CTA per tile (moe_gemm_kernel)
constexpr unsigned kFamilyPair = 2u;    // CTA pairs (moe_gemm_pair_kernel)

constexpr unsigned kSpecHintTag = 0x5ec00000u;

// smem bytes for one pipeline stage: na weight tiles of 128 rows x 128 B
// and one token tile of n_max rows x 128 B
inline int gemm_stage_bytes(int na, int n_max) { return na * 16384 + n_max * 128; }

// bytes of shared memory outside the stage ring (FP8: column scale products
// of the longer K, the per-column amax exchange and reciprocal scales;
// otherwise GEMM2's per-column weights)
inline int gemm_extra_smem(int n_max, int kblocks_max, bool fp8) {
  return 1024 /* align slack */ + 1024 /* barriers, work queue, flags */ +
         (fp8 ? 2 * n_max * kblocks_max * 4 + 5 * n_max * 4 : n_max * 4);
}

// Launch a kernel that may overlap its predecessor's tail in the stream
// (programmatic dependent launch); the kernel calls pdl_wait() before it
// touches anything the predecessor writes or reads.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_chained(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Launch one grouped GEMM kernel (GEMM1, GEMM2 or both fused).
cudaError_t launch_grouped_gemm(int kind, const GemmArgs& args, const GemmMaps* maps, int grid,
                                int smem_bytes, cudaStream_t stream);

// CTA-pair grouped GEMMs (BF16/TF32): one stage of one CTA holds, for each
// of its ks K blocks, na 128-row weight tiles and half of an n_max-row token
// tile (GEMM1: na 2, ks 1; GEMM2: na 1, ks 2); the token maps of `maps` are
// 8, 16, 32, 64 and 128 rows high (half tiles).
inline int gemm_pair_stage_bytes(int na, int n_max, int ks) {
  return ks * (na * 16384 + (n_max / 2) * 128);
}
constexpr int kPairExtraSmem = 3072;  // align slack, barriers, GEMM2 column weights

// Launch GEMM1 (mode 1) or GEMM2 (mode 2) on CTA pairs; the grid is as many
// clusters as can be resident at once, at most max_items.
cudaError_t launch_grouped_gemm_pair(int kind, int mode, const GemmArgs& args,
                                     const GemmMaps& maps, int smem_bytes, long long max_items,
                                     cudaStream_t stream);

// Token-major FP8 grouped GEMMs (grouped_gemm_tm.cu): one stage holds two
// 128-row weight boxes and a token box of up to 128 rows (128 bytes of K
// each).  Outside the ring: output staging (GEMM1: a 128-row x 128-byte act
// block for its TMA stores; GEMM2: 2 KB per epilogue warp to turn its rows
// around), alignment slack, barriers and (GEMM1) the amax exchange.
constexpr int kTmStageBytes = 3 * 16384;
__host__ __device__ constexpr int tm_out_bytes(int mode) { return mode == 1 ? 16384 : 32768; }
__host__ __device__ constexpr int tm_smem_bytes(int mode, int stages) {
  return 1024 + stages * kTmStageBytes + tm_out_bytes(mode) + 512 + (mode == 1 ? 4096 : 0);
}

// Launch token-major GEMM1 (mode 1: gate+up with SiLU and e4m3 act) or
// GEMM2 (mode 2: down with the routing weight) over `grid` persistent CTAs.
// `maps`: the weights (a) and the input token rows (b, 16 .. 256 rows high);
// `omaps`: GEMM1's act rows for its TMA stores (b, 16 .. 256 rows high).
cudaError_t launch_grouped_gemm_tm(int mode, const GemmArgs& args, const GemmMaps& maps,
                                   const GemmMaps& omaps, int grid, int smem_bytes,
                                   cudaStream_t stream);

}  // namespace moe
