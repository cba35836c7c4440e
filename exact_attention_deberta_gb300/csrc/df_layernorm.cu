// Residual add + LayerNorm of the encoder (bf16 / fp16 in and out, fp32
// statistics): out[m] = (y - mean y) / sqrt(var y + eps) * gamma + beta with
// y = x[m] + residual[m] (residual optional), the normalisation after the
// attention output and after the feed-forward block of a DeBERTa encoder layer,
// and of the relative embeddings.
//
// One warp per row: each lane holds N / 32 values (16-byte vector loads of 8
// values), the mean and then the variance of the deviations come from two warp
// reductions over registers (no second pass over memory), the row is written
// back with 16-byte stores.  HBM bound: a row is read once (twice with the
// residual) and written once.
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "df_common.cuh"

namespace dfa {
namespace {

template <typename T>
__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  const T* h = reinterpret_cast<const T*>(&v);
#pragma unroll
  for (int e = 0; e < 8; ++e) f[e] = IO<T>::to_f(h[e]);
}

template <typename T>
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 v;
  T* h = reinterpret_cast<T*>(&v);
#pragma unroll
  for (int e = 0; e < 8; ++e) h[e] = IO<T>::from_f(f[e]);
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// V vectors of 8 values per lane: N = 256 V
template <typename T, int V>
__global__ void __launch_bounds__(256) layernorm_kernel(const T* __restrict__ x, const T* __restrict__ res,
                                                        const T* __restrict__ gamma,
                                                        const T* __restrict__ beta, int M, float eps,
                                                        T* __restrict__ out) {
  constexpr int N = 256 * V;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= M) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)row * N);
  const uint4* rr = res ? reinterpret_cast<const uint4*>(res + (size_t)row * N) : nullptr;
  float y[V][8];
  float s = 0.f;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    unpack8<T>(xr[v * 32 + lane], y[v]);
    if (rr) {
      float r[8];
      unpack8<T>(rr[v * 32 + lane], r);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[v][e] += r[e];
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) s += y[v][e];
  }
  const float mean = warp_sum(s) * (1.f / N);
  float q = 0.f;
#pragma unroll
  for (int v = 0; v < V; ++v)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float dv = y[v][e] - mean;
      q += dv * dv;
    }
  const float rstd = rsqrtf(warp_sum(q) * (1.f / N) + eps);
  const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
  const uint4* b4 = reinterpret_cast<const uint4*>(beta);
  uint4* o4 = reinterpret_cast<uint4*>(out + (size_t)row * N);
#pragma unroll
  for (int v = 0; v < V; ++v) {
    float g[8], b[8], o[8];
    unpack8<T>(g4[v * 32 + lane], g);
    unpack8<T>(b4[v * 32 + lane], b);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = (y[v][e] - mean) * rstd * g[e] + b[e];
    o4[v * 32 + lane] = pack8<T>(o);
  }
}

template <typename T>
cudaError_t launch_ln(const void* x, const void* res, const void* g, const void* b, int M, int N, float eps,
                      void* out, cudaStream_t s) {
  const int blocks = (M + 7) / 8;  // 8 rows (warps) per block
  const T* xp = static_cast<const T*>(x);
  const T* rp = static_cast<const T*>(res);
  const T* gp = static_cast<const T*>(g);
  const T* bp = static_cast<const T*>(b);
  T* op = static_cast<T*>(out);
  switch (N / 256) {
    case 1: layernorm_kernel<T, 1><<<blocks, 256, 0, s>>>(xp, rp, gp, bp, M, eps, op); break;
    case 2: layernorm_kernel<T, 2><<<blocks, 256, 0, s>>>(xp, rp, gp, bp, M, eps, op); break;
    case 3: layernorm_kernel<T, 3><<<blocks, 256, 0, s>>>(xp, rp, gp, bp, M, eps, op); break;
    case 4: layernorm_kernel<T, 4><<<blocks, 256, 0, s>>>(xp, rp, gp, bp, M, eps, op); break;
    case 6: layernorm_kernel<T, 6><<<blocks, 256, 0, s>>>(xp, rp, gp, bp, M, eps, op); break;
    case 8: layernorm_kernel<T, 8><<<blocks, 256, 0, s>>>(xp, rp, gp, bp, M, eps, op); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace dfa

using namespace dfa;

extern "C" df_status df_layernorm(const void* x, const void* residual, const void* gamma, const void* beta,
                                  int M, int N, float eps, void* out, df_dtype dtype, df_stream_t stream) {
  if (!x || !gamma || !beta || !out || M < 1 || N < 1 || !(eps > 0.f)) return DF_ERR_INVALID_ARG;
  if (dtype != DF_BF16 && dtype != DF_FP16) return DF_ERR_UNSUPPORTED;
  const int v = N / 256;
  if (N % 256 != 0 || !(v == 1 || v == 2 || v == 3 || v == 4 || v == 6 || v == 8)) return DF_ERR_UNSUPPORTED;
  if (!al16(x) || !al16(gamma) || !al16(beta) || !al16(out) || (residual && !al16(residual)))
    return DF_ERR_ALIGNMENT;
  const cudaError_t e =
      dtype == DF_BF16
          ? launch_ln<__nv_bfloat16>(x, residual, gamma, beta, M, N, eps, out, (cudaStream_t)stream)
          : launch_ln<__half>(x, residual, gamma, beta, M, N, eps, out, (cudaStream_t)stream);
  return e == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}
