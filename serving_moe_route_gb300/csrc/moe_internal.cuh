// moe_internal.cuh -- declarations shared by the two translation units of
// the library (host API + routing/permutation kernels, grouped GEMMs).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

// operand element kinds of the grouped GEMMs
enum GemmKind : int { KIND_TF32 = 0, KIND_BF16 = 1, KIND_E4M3 = 2 };

// Arguments of one grouped GEMM launch (swap-AB orientation: the MMA's M
// side is 128 weight rows of one expert, its N side is a tile of up to
// tile_n permuted token rows of that expert).
struct GemmArgs {
  const int4* tiles;   // [max_tiles] {expert, first permuted row, rows, 0}
  const int* ntiles;   // device count of valid tiles
  int mblocks;         // 128-row weight blocks per expert (G1: ceil(I/128))
  int kblocks;         // K / (128 bytes / element size)
  int N;               // token tile = MMA N
  int a_rows_per_e;    // rows of one expert in the A view (G1: 2I, G2: H)
  int a_up_off;        // G1: I (first up row); G2: 0
  int m_valid;         // G1: I, G2: H -- weight rows at or beyond are masked
  int R;               // permuted rows (T*k)
  int stages;          // shared-memory pipeline depth
  uint32_t tmem_cols;  // allocated TMEM columns (power of two)
  // G1 epilogue: act [R, I] (f32 / bf16 / e4m3) and FP8 group scales [R, I/128]
  void* act;
  float* act_scale;
  int I;
  // G2 epilogue: out_acc[t, h] += w[f] * y for f = src[row], t = f / k
  const int* src;
  const float* topw;
  float* out_acc;
  int H, k;
  // FP8: weight block scales and activation group scales [R, kblocks]
  const float* w_scale;
  int w_scale_rows_per_e;  // G1: 2I/128, G2: H/128
  const float* b_scale;
  unsigned* err;
  unsigned long long limit_ns;
};

// smem bytes for one pipeline stage: NA weight tiles of 128 rows x 128 B
// and one token tile of N rows x 128 B
inline int gemm_stage_bytes(int na, int N) { return na * 16384 + N * 128; }

// bytes of shared memory outside the stage ring
inline int gemm_extra_smem(int N, int kblocks) {
  return 1024 /* align slack */ + 256 /* barriers, flags */ + N * kblocks * 4 + 4 * N * 4;
}

// Launch grouped GEMM `g` (1: gate+up with SiLU, 2: down with combine).
cudaError_t launch_grouped_gemm(int kind, int g, const GemmArgs& args, const CUtensorMap& ta,
                                const CUtensorMap& tb, int grid, int smem_bytes,
                                cudaStream_t stream);

}  // namespace moe
