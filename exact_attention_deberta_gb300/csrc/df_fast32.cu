// Fast fp32 mode: fp32 q, k, v, pos_key, pos_query are rounded to fp16 (an
// 11-bit significand, as TF32 keeps), the fp16 tensor-core forward runs on the
// copies, and its fp16 output is widened back to fp32.  Both conversions are
// HBM-bound moves of 16 bytes (fp32 side) per thread and step.  A value fp16
// cannot hold (|x| > 65504, or not finite) is counted in a flag word that the
// output conversion turns into DF_ERR_INVALID_ARG in the device status word
// (the forward in between clears that word when it starts).
#include "df_common.cuh"

#include <cuda_fp16.h>

#include <algorithm>

namespace dfa {
namespace {

struct HalfArgs {
  const float4* src[5];
  uint2* dst[5];
  long long n4[5];  // groups of four values
  int* flag;
};

__device__ __forceinline__ uint32_t half2_bits(__half2 h) {
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void to_half_kernel(const HalfArgs a) {
  const int w = blockIdx.y;
  const float4* __restrict__ src = a.src[w];
  uint2* __restrict__ dst = a.dst[w];
  bool bad = false;
  for (long long f = (long long)blockIdx.x * blockDim.x + threadIdx.x; f < a.n4[w];
       f += (long long)gridDim.x * blockDim.x) {
    const float4 x = src[f];
    // !(|x| <= max) also catches NaN
    bad |= !(fabsf(x.x) <= 65504.f) || !(fabsf(x.y) <= 65504.f) || !(fabsf(x.z) <= 65504.f) ||
           !(fabsf(x.w) <= 65504.f);
    dst[f] = make_uint2(half2_bits(__floats2half2_rn(x.x, x.y)), half2_bits(__floats2half2_rn(x.z, x.w)));
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(a.flag, 1);
}

__global__ void to_float_kernel(const uint2* __restrict__ src, float4* __restrict__ dst, long long n4,
                                const int* flag, df_ws_header* hdr) {
  if (blockIdx.x == 0 && threadIdx.x == 0 && *flag != 0) raise_device_error(hdr, DF_ERR_INVALID_ARG, 700);
  for (long long f = (long long)blockIdx.x * blockDim.x + threadIdx.x; f < n4;
       f += (long long)gridDim.x * blockDim.x) {
    const uint2 v = src[f];
    const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
    const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
    dst[f] = make_float4(lo.x, lo.y, hi.x, hi.y);
  }
}

int convert_blocks(long long groups) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  return (int)std::max<long long>(1, std::min<long long>((groups + 255) / 256, (long long)sms * 8));
}

}  // namespace

cudaError_t launch_to_half(const float* const src[5], void* const dst[5], const long long n[5], int* flag,
                           cudaStream_t s) {
  HalfArgs a;
  long long most = 0;
  for (int w = 0; w < 5; ++w) {
    a.src[w] = reinterpret_cast<const float4*>(src[w]);
    a.dst[w] = static_cast<uint2*>(dst[w]);
    a.n4[w] = n[w] / 4;
    most = std::max(most, a.n4[w]);
  }
  a.flag = flag;
  cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(int), s);
  if (e != cudaSuccess || most == 0) return e;
  to_half_kernel<<<dim3(convert_blocks(most), 5), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_to_float(const void* src, float* dst, long long n, const int* flag, void* hdr,
                            cudaStream_t s) {
  const long long n4 = n / 4;
  to_float_kernel<<<convert_blocks(std::max(n4, 1LL)), 256, 0, s>>>(
      static_cast<const uint2*>(src), reinterpret_cast<float4*>(dst), n4, flag,
      static_cast<df_ws_header*>(hdr));
  return cudaGetLastError();
}

}  // namespace dfa
