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

// Arguments of one grouped GEMM launch (swap-AB orientation: the MMA's M
// side is 128 weight rows of one expert, its N side a tile of up to
// n_max permuted token rows of that expert; each tile carries its own n).
struct GemmArgs {
  const int4* tiles;   // [max_tiles] {expert, first permuted row, rows, tile n}
  const int* ntiles;   // device count of valid tiles
  int mblocks;         // 128-row weight blocks per expert (G1: ceil(I/128))
  int kblocks;         // K / (128 bytes / element size)
  int n_max;           // largest tile n (stage and TMEM slot size)
  int a_rows_per_e;    // rows of one expert in the A view (G1: 2I, G2: H)
  int a_up_off;        // G1: I (first up row); G2: 0
  int m_valid;         // G1: I, G2: H -- weight rows at or beyond are masked
  int R;               // permuted rows (T*k)
  int stages;          // shared-memory pipeline depth
  int nslots;          // TMEM accumulator slots (per tile; FP8: per 128-K block)
  uint32_t tmem_cols;  // allocated TMEM columns (power of two)
  // G1 epilogue: act [R, I] (f32 / bf16 / e4m3) and FP8 group scales [R, I/128]
  void* act;
  float* act_scale;
  int I;
  // G2 epilogue: ybuf[row, h] = w[src[row]] * y[row, h] (bf16, f32 for TF32)
  const int* src;
  const float* topw;
  void* ybuf;
  int H;
  // FP8: weight block scales and activation group scales [R, kblocks]
  const float* w_scale;
  int w_scale_rows_per_e;  // G1: 2I/128, G2: H/128
  const float* b_scale;
  unsigned* err;
  unsigned long long limit_ns;
};

// smem bytes for one pipeline stage: NA weight tiles of 128 rows x 128 B
// and one token tile of n_max rows x 128 B
inline int gemm_stage_bytes(int na, int n_max) { return na * 16384 + n_max * 128; }

// bytes of shared memory outside the stage ring (FP8: column scale products
// and the per-column amax exchange; otherwise G2's per-column weights)
inline int gemm_extra_smem(int na, int n_max, int kblocks, bool fp8) {
  return 1024 /* align slack */ + 512 /* barriers, flags */ +
         (fp8 ? na * n_max * kblocks * 4 + 4 * n_max * 4 : n_max * 4 /* column weights */);
}

// Launch grouped GEMM `g` (1: gate+up with SiLU, 2: down with weighting).
cudaError_t launch_grouped_gemm(int kind, int g, const GemmArgs& args, const GemmMaps& maps,
                                int grid, int smem_bytes, cudaStream_t stream);

}  // namespace moe
