// Projections that feed the attention (tcgen05 GEMM, bf16 / fp16 in and out,
// fp32 accumulation): y_i = x . W_i^T + b_i for up to three weight blocks W_i
// [N, K] that share the input x [M, K], each written to its own [M, N] output.
//
// DisentangledFlash 0.2.0 README, "Status": the fused QKV projection is always
// enabled (one pass over the hidden states gives Q, K and V, each in the
// [tokens, heads x head size] layout the attention reads); the same kernel
// gives the relative-position projections PK and PQ of the relative
// embeddings (two weight blocks, one input).
//
// One CTA per SM, persistent over 128 x 256 output tiles (row block outermost,
// so the 9 tiles of a row block of a QKV projection reuse its rows from L2):
//   warp 0     TMA producer: per 64-column K block, the 128 x 64 block of x and
//              the 256 x 64 block of W_i (128-byte swizzle) into a 4-stage ring;
//   warp 1     tcgen05.mma issuer (M = 128, N = 256, K = 16 per instruction)
//              into one of two TMEM accumulators (256 columns each), so the
//              epilogue of a tile overlaps the next tile's MMAs;
//   warps 2-5  epilogue: TMEM -> registers, + bias, rounded to the I/O type,
//              16-byte stores to the tile's output rows.
// Every wait is bounded; one that runs out records DF_ERR_DEVICE_TIMEOUT in the
// caller's status word (if given), the CTA stops issuing, drains its copies
// and MMAs in flight, frees its tensor memory and returns.
#include <cudaTypedefs.h>

#include <algorithm>
#include <type_traits>

#include "df_tc_common.cuh"

namespace dfa {
namespace {

using namespace ptx;

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kLinThreads = 192;
constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kBBytes = kBN * kBK * 2;  // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr unsigned long long kLinBudget = 1ull << 33;  // cycles (seconds at GB300 clocks)

struct LinSmem {
  static constexpr uint32_t stages = 0;                                // [S][A | B]
  static constexpr uint32_t bias = stages + kStages * kStageBytes;     // float [2][256]
  static constexpr uint32_t bars = bias + 2 * kBN * 4;
  // full[S], empty[S], acc_full[2], acc_empty[2], drain
  static constexpr int kBars = 2 * kStages + 4 + 1;
  static constexpr uint32_t misc = bars + kBars * 8;                   // abort flag, tmem slot
  static constexpr uint32_t bytes = misc + 16;
  static constexpr uint32_t alloc = bytes + 1024;
};

struct LinArgs {
  int M, K, N, n_out;
  int act;  // 0: none, 1: GELU (erf form)
  const void* bias[3];
  void* out[3];
  int32_t* status;
};

struct LinMaps {
  CUtensorMap a;
  CUtensorMap b[3];
};

__device__ __forceinline__ bool lin_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         int32_t* status) {
  if (*abort) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (*abort) return false;
    if ((unsigned long long)(clock64() - t0) > kLinBudget) {
      *abort = 1;
      if (status) atomicCAS(status, 0, (int32_t)DF_ERR_DEVICE_TIMEOUT);
      return false;
    }
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kLinThreads, 1)
    linear_kernel(const LinArgs args, const __grid_constant__ LinMaps maps) {
  using SL = LinSmem;
  constexpr uint32_t kIdesc = idesc_f16(kBM, kBN, BF16 ? 1 : 0, 0, 0);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  float* sBias = reinterpret_cast<float*>(sm + SL::bias);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SL::bars);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* acc_full = bars + 2 * kStages;
  uint64_t* acc_empty = acc_full + 2;  // the four epilogue warps read the accumulator
  uint64_t* drain = acc_empty + 2;
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + SL::misc);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SL::misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full + b, 1);
      mbar_init(acc_empty + b, 4);
    }
    mbar_init(drain, 1);
    *s_abort = 0;
    mbar_fence_init();
    tma_prefetch_desc(&maps.a);
    for (int i = 0; i < args.n_out; ++i) tma_prefetch_desc(&maps.b[i]);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  // two fp32 accumulators of kBN columns each: columns 0 .. 2 kBN - 1
  static_assert(tmem_region_fits(kBN, kBN, 512), "two accumulators in 512 columns");

  const int n_mb = (args.M + kBM - 1) / kBM, n_nb = args.N / kBN, nk = args.K / kBK;
  const int per_mb = args.n_out * n_nb;
  const int tiles = n_mb * per_mb;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t g = 0, g_issued = 0;
      for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int mb = tile / per_mb, rem = tile - mb * per_mb;
        const int i = rem / n_nb, nb = rem - i * n_nb;
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = g % kStages;
          if (!lin_wait(empty + s, ((g / kStages) & 1) ^ 1, s_abort, args.status)) continue;
          uint8_t* st = sm + SL::stages + s * kStageBytes;
          mbar_expect_tx(full + s, kStageBytes);
          tma_load_2d(st, &maps.a, kb * kBK, mb * kBM, full + s);
          tma_load_2d(st + kABytes, &maps.b[i], kb * kBK, nb * kBN, full + s);
          g_issued = g + 1;
        }
      }
      // no copy may still be landing when the CTA leaves
      for (uint32_t k = g_issued > (uint32_t)kStages ? g_issued - kStages : 0; k < g_issued; ++k)
        mbar_wait(full + k % kStages, (k / kStages) & 1, kLinBudget);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t g = 0, tc = 0;
      for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++tc) {
        const int buf = tc & 1;
        const uint32_t tacc = tmem + 256u * buf;
        // the epilogue has read this accumulator's previous tile
        bool ok = lin_wait(acc_empty + buf, ((tc >> 1) & 1) ^ 1, s_abort, args.status);
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = g % kStages;
          ok = lin_wait(full + s, (g / kStages) & 1, s_abort, args.status) && ok;
          if (!ok) continue;
          const uint8_t* st = sm + SL::stages + s * kStageBytes;
          const uint64_t da = sdesc_sw128(smem_u32(st), 16, 1024);
          const uint64_t db = sdesc_sw128(smem_u32(st + kABytes), 16, 1024);
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_ss(tacc, da + 2 * k, db + 2 * k, kIdesc, (kb > 0 || k > 0) ? 1u : 0u);
          mma_commit(empty + s);
        }
        if (ok) mma_commit(acc_full + buf);
      }
      mma_commit(drain);
      mbar_wait(drain, 0, kLinBudget);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 64;        // 0..127
    const int quad = warp & 3;              // TMEM lane quadrant
    const int row = quad * 32 + lane;       // row inside the tile
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    uint32_t tc = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++tc) {
      const int mb = tile / per_mb, rem = tile - mb * per_mb;
      const int i = rem / n_nb, nb = rem - i * n_nb;
      const int buf = tc & 1;
      // this tile's 256 bias values (zero without a bias)
      const T* bias = static_cast<const T*>(args.bias[i]);
      float* sb = sBias + buf * kBN;
      for (int c = et; c < kBN; c += 128)
        sb[c] = bias ? IO<T>::to_f(bias[nb * kBN + c]) : 0.f;
      named_sync(1, 128);
      const bool ok = lin_wait(acc_full + buf, (tc >> 1) & 1, s_abort, args.status);
      tc_fence_after();
      const int grow = mb * kBM + row;
      const bool store = ok && grow < args.M && *s_abort == 0;
      T* dst = static_cast<T*>(args.out[i]) + (size_t)grow * args.N + nb * kBN;
      const uint32_t tacc = tmem + 256u * buf + lane_off;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tacc + 32 * c, r);
        tmem_ld_wait(r);
        if (store) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float a = __uint_as_float(r[2 * e]) + sb[32 * c + 2 * e];
            float b = __uint_as_float(r[2 * e + 1]) + sb[32 * c + 2 * e + 1];
            if (args.act == 1) {  // GELU: x (1 + erf(x / sqrt 2)) / 2
              a = 0.5f * a * (1.f + erff(a * 0.70710678118654752f));
              b = 0.5f * b * (1.f + erff(b * 0.70710678118654752f));
            }
            w[e] = BF16 ? pack_bf16x2(a, b) : pack_f16x2(a, b);
          }
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int e = 0; e < 4; ++e) d4[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
      // the accumulator is read: the MMA warp may refill it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + buf);
      // sb is rewritten two tiles later, after every epilogue thread is past here
      named_sync(1, 128);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 lin_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// Row-major [rows][cols] 16-bit matrix in 64 x box_rows boxes, 128-byte swizzle;
// rows past the end read as zeros.
bool encode_k_major(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows,
                    bool bf16) {
  auto enc = lin_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
             const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int lin_sm_count() {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  return sms;
}

bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

template <bool BF16>
cudaError_t launch_linear(const LinArgs& a, const LinMaps& maps, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(linear_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)LinSmem::alloc);
  if (e != cudaSuccess) return e;
  const int tiles = (a.M + kBM - 1) / kBM * a.n_out * (a.N / kBN);
  linear_kernel<BF16><<<std::min(tiles, lin_sm_count()), kLinThreads, LinSmem::alloc, s>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace
}  // namespace dfa

using namespace dfa;

extern "C" df_status df_linear(const void* x, int M, int K, int n_out, const void* const* w,
                               const void* const* bias, int N, void* const* out, int activation,
                               df_dtype dtype, int32_t* status, df_stream_t stream) {
  if (!x || !w || !out || M < 1 || K < 1 || N < 1 || n_out < 1 || n_out > 3) return DF_ERR_INVALID_ARG;
  if (activation != 0 && activation != 1) return DF_ERR_INVALID_ARG;
  if (dtype != DF_BF16 && dtype != DF_FP16) return DF_ERR_UNSUPPORTED;
  if (K % kBK != 0 || N % kBN != 0) return DF_ERR_UNSUPPORTED;
  if ((long long)M * K > (1ll << 40)) return DF_ERR_INVALID_ARG;
  if (!al16(x)) return DF_ERR_ALIGNMENT;
  LinArgs a;
  a.M = M;
  a.K = K;
  a.N = N;
  a.n_out = n_out;
  a.act = activation;
  a.status = status;
  LinMaps maps;
  const bool bf16 = dtype == DF_BF16;
  if (!encode_k_major(&maps.a, x, M, K, kBM, bf16)) return DF_ERR_CUDA;
  for (int i = 0; i < 3; ++i) {
    a.bias[i] = nullptr;
    a.out[i] = nullptr;
  }
  for (int i = 0; i < n_out; ++i) {
    if (!w[i] || !out[i]) return DF_ERR_INVALID_ARG;
    if (!al16(w[i]) || !al16(out[i]) || (bias && bias[i] && !al16(bias[i]))) return DF_ERR_ALIGNMENT;
    if (!encode_k_major(&maps.b[i], w[i], N, K, kBN, bf16)) return DF_ERR_CUDA;
    a.bias[i] = bias ? bias[i] : nullptr;
    a.out[i] = out[i];
  }
  const cudaError_t e = bf16 ? launch_linear<true>(a, maps, (cudaStream_t)stream)
                             : launch_linear<false>(a, maps, (cudaStream_t)stream);
  return e == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}
