// ep.cu -- the expert-parallel exchange's arithmetic around the local slice
// (H20 article, para. 2: the fused-MoE call takes the expert-parallel size
// and rank; para. 3: 400 expert slots over 8 GPUs).  A rank routes its own
// tokens over all E experts, sends each token once to every rank that owns
// one of its picks, runs its own experts on what it receives, and sums the
// partial rows that come back.  These kernels compute the send plan, pack
// the send rows and sum the returned partials; moving the rows between
// ranks is the caller's collective.
//
//   ep_dispatch_kernel  one CTA: for every rank d, the tokens with a pick
//                       owned by d (owner = id / e_local), in token order;
//                       groups in rank order.  Block scans, no atomics.
//   ep_pack_kernel      warp per send row: the token's activation row, its
//                       k ids and k weights copied to the send buffers
//   ep_combine_kernel   warp per (token, 256 columns): the token's partial
//                       rows summed in rank order (deterministic), fp32
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe_route.h"
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kEpThreads = 1024;
constexpr int kEpMaxRanks = 32;

// exclusive scan of one int per thread over the CTA (1024 threads); *total
// receives the sum.  Every thread calls it.
__device__ int ep_block_scan(int v, int* warp_sums, int* total) {
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
    warp_sums[lane] = s;
    if (lane == 31) *total = s;
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  __syncthreads();
  return before;
}

// bit d of the result: token t has a pick owned by rank d
__device__ __forceinline__ uint32_t ep_owner_mask(const int* ids, int t, int k, int e_local,
                                                  int ep_size) {
  uint32_t m = 0;
  for (int j = 0; j < k; ++j) {
    const int id = ids[static_cast<size_t>(t) * k + j];
    if (id < 0) continue;
    const int d = id / e_local;
    if (d < ep_size) m |= 1u << d;
  }
  return m;
}

__global__ void __launch_bounds__(kEpThreads)
    ep_dispatch_kernel(const int* __restrict__ ids, int T, int k, int e_local, int ep_size,
                       int* __restrict__ send_counts, int* __restrict__ send_tokens,
                       int* __restrict__ row_of) {
  __shared__ int warp_sums[32];
  __shared__ int total;
  __shared__ int count[kEpMaxRanks], start[kEpMaxRanks];
  // pass 1: tokens per rank
  if (threadIdx.x < kEpMaxRanks) count[threadIdx.x] = 0;
  __syncthreads();
  for (int d = 0; d < ep_size; ++d) {
    int run = 0;
    for (int t0 = 0; t0 < T; t0 += kEpThreads) {
      const int t = t0 + threadIdx.x;
      const int f = (t < T) ? static_cast<int>((ep_owner_mask(ids, t, k, e_local, ep_size) >> d) & 1u) : 0;
      ep_block_scan(f, warp_sums, &total);
      run += total;
    }
    if (threadIdx.x == 0) count[d] = run;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    int s = 0;
    for (int d = 0; d < ep_size; ++d) {
      start[d] = s;
      s += count[d];
    }
  }
  __syncthreads();
  if (threadIdx.x < ep_size) send_counts[threadIdx.x] = count[threadIdx.x];
  // pass 2: each (token, rank) pair's row in the send order
  for (int d = 0; d < ep_size; ++d) {
    int base = start[d];
    for (int t0 = 0; t0 < T; t0 += kEpThreads) {
      const int t = t0 + threadIdx.x;
      const int f = (t < T) ? static_cast<int>((ep_owner_mask(ids, t, k, e_local, ep_size) >> d) & 1u) : 0;
      const int pos = ep_block_scan(f, warp_sums, &total);
      if (t < T) {
        const int row = f ? base + pos : -1;
        row_of[static_cast<size_t>(t) * ep_size + d] = row;
        if (f) send_tokens[row] = t;
      }
      base += total;
    }
  }
}

// one warp per send row; rows at or past the total of send_counts are left
template <typename XT>
__global__ void __launch_bounds__(256)
    ep_pack_kernel(const XT* __restrict__ x, const int* __restrict__ ids,
                   const float* __restrict__ w, int T, int H, int k, int ep_size,
                   const int* __restrict__ send_counts, const int* __restrict__ send_tokens,
                   XT* __restrict__ x_send, int* __restrict__ ids_send,
                   float* __restrict__ w_send) {
  const int lane = threadIdx.x & 31;
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  int n = lane < ep_size ? send_counts[lane] : 0;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) n += __shfl_xor_sync(0xffffffffu, n, off);
  if (row >= n) return;
  const int t = send_tokens[row];
  const XT* src = x + static_cast<size_t>(t) * H;
  XT* dst = x_send + static_cast<size_t>(row) * H;
  // 16 bytes per lane and step when the rows allow it, else one element
  constexpr int VW = 16 / static_cast<int>(sizeof(XT));
  if (H % VW == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
      (reinterpret_cast<uintptr_t>(x_send) & 15) == 0) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (int h = lane; h < H / VW; h += 32) d4[h] = s4[h];
  } else {
    for (int h = lane; h < H; h += 32) dst[h] = src[h];
  }
  if (lane < k) {
    ids_send[static_cast<size_t>(row) * k + lane] = ids[static_cast<size_t>(t) * k + lane];
    w_send[static_cast<size_t>(row) * k + lane] = w[static_cast<size_t>(t) * k + lane];
  }
}

// out[t, h] = sum over d = 0 .. ep_size-1 (ascending) of back[row_of[t, d], h]
__global__ void __launch_bounds__(256)
    ep_combine_kernel(const float* __restrict__ back, const int* __restrict__ row_of, int T,
                      int H, int ep_size, float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int chunks = (H + 255) / 256;
  const long long g = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (g >= static_cast<long long>(T) * chunks) return;
  const int t = static_cast<int>(g / chunks);
  const int h0 = static_cast<int>(g % chunks) * 256 + lane * 8;
  const int my_row = lane < ep_size ? row_of[static_cast<size_t>(t) * ep_size + lane] : -1;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  // two 16-byte loads per row when this lane's 8 columns are whole and aligned
  const bool vec = h0 + 8 <= H && (H & 3) == 0 && (reinterpret_cast<uintptr_t>(back) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(out) & 15) == 0;
  for (int d = 0; d < ep_size; ++d) {
    const int r = __shfl_sync(0xffffffffu, my_row, d);
    if (r < 0) continue;
    const float* p = back + static_cast<size_t>(r) * H + h0;
    if (vec) {
      const float4 a = reinterpret_cast<const float4*>(p)[0];
      const float4 b = reinterpret_cast<const float4*>(p)[1];
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (h0 + i < H) acc[i] += p[i];
    }
  }
  if (vec) {
    float4* o = reinterpret_cast<float4*>(out + static_cast<size_t>(t) * H + h0);
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (h0 + i < H) out[static_cast<size_t>(t) * H + h0 + i] = acc[i];
  }
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_ep_dispatch(const int32_t* ids, int T, int k, int e_local, int ep_size,
                    int32_t* send_counts, int32_t* send_tokens, int32_t* row_of, void* stream) {
  if (T < 0 || k < 1 || k > 32 || e_local < 1 || ep_size < 1 || ep_size > kEpMaxRanks)
    return MOE_ERR_INVALID_ARG;
  if (!send_counts) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!ids || !send_tokens || !row_of)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ep_dispatch_kernel<<<1, kEpThreads, 0, st>>>(ids, T, k, e_local, ep_size, send_counts,
                                               send_tokens, row_of);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_ep_pack(const void* x, int x_dtype, const int32_t* ids, const float* w, int T, int H,
                int k, int ep_size, const int32_t* send_counts, const int32_t* send_tokens,
                void* x_send, int32_t* ids_send, float* w_send, void* stream) {
  if (T < 0 || H < 1 || k < 1 || k > 32 || ep_size < 1 || ep_size > kEpMaxRanks)
    return MOE_ERR_INVALID_ARG;
  if (x_dtype != MOE_DTYPE_F32 && x_dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !ids || !w || !send_counts || !send_tokens || !x_send || !ids_send || !w_send)
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long rows = static_cast<long long>(T) * ep_size;  // capacity of the send buffers
  const unsigned blocks = static_cast<unsigned>((rows * 32 + 255) / 256);
  if (x_dtype == MOE_DTYPE_F32)
    ep_pack_kernel<float><<<blocks, 256, 0, st>>>(
        static_cast<const float*>(x), ids, w, T, H, k, ep_size, send_counts, send_tokens,
        static_cast<float*>(x_send), ids_send, w_send);
  else
    ep_pack_kernel<uint16_t><<<blocks, 256, 0, st>>>(
        static_cast<const uint16_t*>(x), ids, w, T, H, k, ep_size, send_counts, send_tokens,
        static_cast<uint16_t*>(x_send), ids_send, w_send);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_ep_combine(const float* back, const int32_t* row_of, int T, int H, int ep_size,
                   float* out, void* stream) {
  if (T < 0 || H < 1 || ep_size < 1 || ep_size > kEpMaxRanks) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!back || !row_of || !out) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long warps = static_cast<long long>(T) * ((H + 255) / 256);
  ep_combine_kernel<<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, st>>>(
      back, row_of, T, H, ep_size, out);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
