// gemm_common.cuh -- device pieces shared by the single-CTA and CTA-pair
// grouped GEMM kernels: operand kinds, the thread layout of a CTA, and the
// BF16/TF32 epilogue (act = SiLU(gate) * up, or the weighted down rows).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

constexpr unsigned kDevErrTimeout = 4u;
constexpr int kEpiWarps = 8;  // two column halves per TMEM lane quadrant
// warp 0 producer, warp 1 first MMA issuer, warps 2 .. 1 + kEpiWarps
// epilogue, the last warp the second MMA issuer
constexpr int kMmaWarp2 = 2 + kEpiWarps;
constexpr int kThreads = 96 + 32 * kEpiWarps;

template <int KIND>
struct KindTraits;
template <>
struct KindTraits<KIND_TF32> {
  static constexpr uint32_t fmt = 2;
  static constexpr int esize = 4;
};
template <>
struct KindTraits<KIND_BF16> {
  static constexpr uint32_t fmt = 1;
  static constexpr int esize = 2;
};
template <>
struct KindTraits<KIND_E4M3> {
  static constexpr uint32_t fmt = 0;
  static constexpr int esize = 1;
};

// SiLU(z) = z / (1 + e^-z) with the fast exponential and fast division
// (relative error ~1e-6, far inside the layer's tolerance); for z below
// about -88 the denominator is +inf and the quotient 0, the limit of SiLU
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Column maxima of a warp's C x 32 block (C columns per lane, one row per
// lane) in 31 shuffles for C = 32: while the partner distance is at least C
// every column is reduced; below it each step keeps half of the remaining
// columns and trades the other half with the partner lane.  Lane l returns
// the maximum of column (l mod C).  m[] is overwritten.
template <int C>
__device__ __forceinline__ float col_max_transpose(float (&m)[C], int lane) {
#pragma unroll
  for (int off = 16; off >= C; off >>= 1)
#pragma unroll
    for (int i = 0; i < C; ++i) m[i] = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], off));
#pragma unroll
  for (int off = C / 2; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? m[i] : m[i + off];
      const float keep = upper ? m[i + off] : m[i];
      m[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, off));
    }
  }
  return m[0];
}

// two floats rounded to bf16 (nearest-even), lo in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// activation (GEMM1 output) and weighted expert output (GEMM2 output) stores
template <int KIND>
__device__ __forceinline__ void store_val(void* base, size_t idx, float v) {
  if constexpr (KIND == KIND_TF32)
    static_cast<float*>(base)[idx] = v;
  else
    static_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
}

// BF16/TF32 epilogue for C token columns starting at cc of one work item:
// both accumulators are loaded from TMEM before one wait.  GEMM1 writes
// act = SiLU(gate) * up; GEMM2 writes the weighted rows of one (na = 1) or
// two (na = 2: rows row and row_b) 128-row weight tiles.
template <int KIND, int C>
__device__ __forceinline__ void epi_chunk(const GemmArgs& A, int g, int na, uint32_t taddr, int NM,
                                          int cc, int row0, int nrows, int row, bool row_ok,
                                          int row_b, bool row_b_ok, const float* cw) {
  float v0[C], v1[C];
  tmem_ld<C>(taddr + cc, v0);
  if (g == 0 || na == 2) {
    tmem_ld<C>(taddr + NM + cc, v1);
    tmem_wait_ld(v0, v1);
  } else {
    tmem_wait_ld(v0);
  }
  if (g == 0) {
    if (row_ok) {
#pragma unroll
      for (int jj = 0; jj < C; ++jj)
        if (cc + jj < nrows)
          store_val<KIND>(A.act, static_cast<size_t>(row0 + cc + jj) * A.I + row,
                          silu_f(v0[jj]) * v1[jj]);
    }
  } else {
    if (row_ok) {
#pragma unroll
      for (int jj = 0; jj < C; ++jj)
        if (cc + jj < nrows)
          store_val<KIND>(A.ybuf, static_cast<size_t>(row0 + cc + jj) * A.H + row,
                          cw[cc + jj] * v0[jj]);
    }
    if (na == 2 && row_b_ok) {
#pragma unroll
      for (int jj = 0; jj < C; ++jj)
        if (cc + jj < nrows)
          store_val<KIND>(A.ybuf, static_cast<size_t>(row0 + cc + jj) * A.H + row_b,
                          cw[cc + jj] * v1[jj]);
    }
  }
}

}  // namespace moe
