// Head size 32 on the tensor-core path (bf16 / fp16): the heads are widened to
// 64 with zeros, the d = 64 kernels run on the widened copies with the scale of
// d = 32, and the first 32 columns of the output are copied back.  A zero
// column adds nothing to Q.K, Q.PK, K.PQ or to a column of O it does not
// produce, so the result is the d = 32 attention (the score scale
// 1 / sqrt(3 d) uses the true d).  Both copies are HBM-bound 16-byte moves.
#include "df_common.cuh"

#include <algorithm>

namespace dfa {
namespace {

struct PadArgs {
  const uint4* src[5];
  uint4* dst[5];
  long long rows[5];  // rows of 32 16-bit values (64 bytes)
};

// dst row = the 64-byte source row followed by 64 zero bytes
__global__ void pad32_kernel(const PadArgs a) {
  const int w = blockIdx.y;
  const uint4* __restrict__ src = a.src[w];
  uint4* __restrict__ dst = a.dst[w];
  const long long total = a.rows[w] * 8;
  for (long long f = (long long)blockIdx.x * blockDim.x + threadIdx.x; f < total;
       f += (long long)gridDim.x * blockDim.x) {
    const long long r = f >> 3;
    const int c = (int)(f & 7);
    dst[f] = c < 4 ? src[r * 4 + c] : make_uint4(0u, 0u, 0u, 0u);
  }
}

__global__ void unpad32_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, long long rows) {
  const long long total = rows * 4;
  for (long long f = (long long)blockIdx.x * blockDim.x + threadIdx.x; f < total;
       f += (long long)gridDim.x * blockDim.x)
    dst[f] = src[(f >> 2) * 8 + (f & 3)];
}

int copy_blocks(long long vectors) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  return (int)std::max<long long>(1, std::min<long long>((vectors + 255) / 256, (long long)sms * 8));
}

}  // namespace

cudaError_t launch_pad32(const void* const src[5], void* const dst[5], const long long rows[5],
                         cudaStream_t s) {
  PadArgs a;
  long long most = 0;
  for (int w = 0; w < 5; ++w) {
    a.src[w] = static_cast<const uint4*>(src[w]);
    a.dst[w] = static_cast<uint4*>(dst[w]);
    a.rows[w] = rows[w];
    most = std::max(most, rows[w] * 8);
  }
  if (most == 0) return cudaSuccess;
  pad32_kernel<<<dim3(copy_blocks(most), 5), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_unpad32(const void* src, void* dst, long long rows, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  unpad32_kernel<<<copy_blocks(rows * 4), 256, 0, s>>>(static_cast<const uint4*>(src),
                                                       static_cast<uint4*>(dst), rows);
  return cudaGetLastError();
}

}  // namespace dfa
