// Packing between the padded [B, L, row] and the packed [T, row] layouts
// (DisentangledFlash 0.2.0 README, "Packed unpadded inference":
// pack_padded_with_info converts right-padded input to FlashAttention-style
// rows with cu_seqlens, and its metadata is reused by every encoder layer and
// by unpack_packed).
//
// The metadata of a mask [B, L] is built in three launches: a count per batch
// row (one block per row), one block that scans the counts into cu_seqlens and
// the totals, and a second pass per row that ranks the valid positions (warp
// ballots and a block scan) and writes the packed -> padded list and its
// inverse.  Moving rows is a pure gather over 16-byte vectors in both
// directions (pack reads through `indices`, unpack through `inverse`, which
// also yields the zero rows), so every store is coalesced; both are bound by
// HBM bandwidth.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "df_attn.h"

namespace dfa {
namespace {

constexpr int kScanThreads = 1024;

// Block-wide exclusive prefix of 0/1 flags (one per thread); returns the
// thread's prefix and sets *total to the block's count.  Uses `warp_sums`
// (32 ints of shared memory).
__device__ __forceinline__ int block_rank(bool flag, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned ballot = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(ballot & ((1u << lane) - 1u));
  if (lane == 0) warp_sums[warp] = __popc(ballot);
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int v = lane < nw ? warp_sums[lane] : 0;
    // inclusive scan over the warp sums
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane < nw) warp_sums[lane] = v;
  }
  __syncthreads();
  const int before = warp > 0 ? warp_sums[warp - 1] : 0;
  *total = warp_sums[(blockDim.x >> 5) - 1];
  __syncthreads();  // warp_sums is reused by the next call
  return before + in_warp;
}

// counts[b] = number of valid positions of batch row b (written to cu[b + 1])
__global__ void __launch_bounds__(kScanThreads) count_rows(const uint8_t* mask, int L, int32_t* cu) {
  __shared__ int warp_sums[32];
  const uint8_t* row = mask + (size_t)blockIdx.x * L;
  int count = 0;
  for (int i0 = 0; i0 < L; i0 += blockDim.x) {
    const int i = i0 + threadIdx.x;
    int chunk;
    block_rank(i < L && row[i] != 0, warp_sums, &chunk);
    count += chunk;
  }
  if (threadIdx.x == 0) cu[blockIdx.x + 1] = count;
}

// cu[0] = 0, cu[b + 1] = cu[b] + count[b]; stats = {T, max count}
__global__ void __launch_bounds__(kScanThreads) scan_counts(int B, int32_t* cu, int32_t* stats) {
  __shared__ int warp_sums[32];
  __shared__ int s_max[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int carry = 0, mx = 0;
  for (int b0 = 0; b0 < B; b0 += blockDim.x) {
    const int b = b0 + threadIdx.x;
    const int c = b < B ? cu[b + 1] : 0;
    mx = max(mx, c);
    // inclusive scan of c over the block
    int v = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += u;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int incl = v + (warp > 0 ? warp_sums[warp - 1] : 0) + carry;
    const int block_total = warp_sums[(blockDim.x >> 5) - 1];
    __syncthreads();
    if (b < B) cu[b + 1] = incl;
    carry += block_total;
  }
  // maximum count
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) s_max[warp] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    int m = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = max(m, s_max[w]);
    cu[0] = 0;
    stats[0] = carry;
    stats[1] = m;
  }
}

// indices[cu[b] + rank] = b L + i for each valid i; inverse[b L + i] = that
// packed row, or -1
__global__ void __launch_bounds__(kScanThreads) rank_rows(const uint8_t* mask, int L, const int32_t* cu,
                                                          int32_t* indices, int32_t* inverse) {
  __shared__ int warp_sums[32];
  const size_t base = (size_t)blockIdx.x * L;
  int next = cu[blockIdx.x];
  for (int i0 = 0; i0 < L; i0 += blockDim.x) {
    const int i = i0 + threadIdx.x;
    const bool valid = i < L && mask[base + i] != 0;
    int chunk;
    const int r = block_rank(valid, warp_sums, &chunk);
    if (i < L) {
      const int k = valid ? next + r : -1;
      inverse[base + i] = k;
      if (valid) indices[k] = (int32_t)(base + i);
    }
    next += chunk;
  }
}

__global__ void pack_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ indices,
                                 const int32_t* __restrict__ stats, int nv, uint4* __restrict__ tokens) {
  const size_t total = (size_t)stats[0] * nv;
  for (size_t f = (size_t)blockIdx.x * blockDim.x + threadIdx.x; f < total;
       f += (size_t)gridDim.x * blockDim.x) {
    const size_t k = f / nv, v = f - k * nv;
    tokens[f] = x[(size_t)indices[k] * nv + v];
  }
}

__global__ void unpack_rows_kernel(const uint4* __restrict__ tokens, const int32_t* __restrict__ inverse,
                                   size_t rows, int nv, uint4* __restrict__ out) {
  const size_t total = rows * nv;
  for (size_t f = (size_t)blockIdx.x * blockDim.x + threadIdx.x; f < total;
       f += (size_t)gridDim.x * blockDim.x) {
    const size_t r = f / nv, v = f - r * nv;
    const int k = inverse[r];
    out[f] = k >= 0 ? tokens[(size_t)k * nv + v] : make_uint4(0u, 0u, 0u, 0u);
  }
}

int copy_grid() {
  static int blocks = 0;
  if (!blocks) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    blocks = std::max(sms, 1) * 8;  // 8 resident blocks of 256 threads per SM
  }
  return blocks;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace dfa

using namespace dfa;

extern "C" df_status df_pack_info(const uint8_t* mask, int B, int L, int32_t* cu_seqlens,
                                  int32_t* indices, int32_t* inverse, int32_t* stats,
                                  df_stream_t stream) {
  if (!mask || !cu_seqlens || !indices || !inverse || !stats || B < 1 || L < 1 ||
      (long long)B * L > (1ll << 30))
    return DF_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  count_rows<<<B, kScanThreads, 0, s>>>(mask, L, cu_seqlens);
  scan_counts<<<1, kScanThreads, 0, s>>>(B, cu_seqlens, stats);
  rank_rows<<<B, kScanThreads, 0, s>>>(mask, L, cu_seqlens, indices, inverse);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

extern "C" df_status df_pack_rows(const void* x, const int32_t* indices, const int32_t* stats, int rows,
                                  size_t row_bytes, void* tokens, df_stream_t stream) {
  if (!x || !indices || !stats || !tokens || rows < 1 || row_bytes == 0 || row_bytes % 16 != 0 ||
      row_bytes / 16 > (size_t)INT32_MAX)
    return DF_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(tokens)) return DF_ERR_ALIGNMENT;
  pack_rows_kernel<<<copy_grid(), 256, 0, (cudaStream_t)stream>>>(
      static_cast<const uint4*>(x), indices, stats, (int)(row_bytes / 16), static_cast<uint4*>(tokens));
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

extern "C" df_status df_unpack_rows(const void* tokens, const int32_t* inverse, int rows,
                                    size_t row_bytes, void* out, df_stream_t stream) {
  if (!tokens || !inverse || !out || rows < 1 || row_bytes == 0 || row_bytes % 16 != 0 ||
      row_bytes / 16 > (size_t)INT32_MAX)
    return DF_ERR_INVALID_ARG;
  if (!aligned16(tokens) || !aligned16(out)) return DF_ERR_ALIGNMENT;
  unpack_rows_kernel<<<copy_grid(), 256, 0, (cudaStream_t)stream>>>(
      static_cast<const uint4*>(tokens), inverse, (size_t)rows, (int)(row_bytes / 16),
      static_cast<uint4*>(out));
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}
